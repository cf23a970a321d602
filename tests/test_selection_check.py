"""The GPU tests' exact-selection check (gpu_util.exact_selection_agrees),
run on hand-made planes on the CPU: it accepts the exact plane's ids, it
rejects other ids on a row whose Top16 cut the plane decides, and it skips a
row whose cut lies within the blocks' tolerances (there rounding may pick
either block)."""
import numpy as np
import pytest

import oracle

from gpu_util import exact_selection_agrees


def _plane():
    # one token, 4 heads, 40 columns; nvp 40, init 1, local 2 -> 13 free slots
    rng = np.random.default_rng(5)
    ex = np.round(rng.normal(0.0, 4.0, size=(1, 4, 40)), 3)
    ab = np.full_like(ex, 100.0)           # tolerance 1e-5 * 100 + 1e-7 ~ 1e-3
    nvp = np.array([40], np.int32)
    return ex, ab, nvp


def _ids(ex, nvp):
    _, ids = oracle.select(ex.astype(np.float32), nvp, init_blocks=1, local_blocks=2)
    return ids


def test_exact_ids_pass_and_rows_are_decided():
    ex, ab, nvp = _plane()
    checked, skipped = exact_selection_agrees(ex, ab, _ids(ex, nvp), nvp, 1, 2)
    assert (checked, skipped) == (4, 0)


def test_a_wrong_id_on_a_decided_row_fails():
    ex, ab, nvp = _plane()
    ids = _ids(ex, nvp).copy()
    free = [c for c in range(1, 38) if c not in ids[0, 0]]
    ids[0, 0, 5] = free[0]                 # swap in a block the exact plane rejects
    with pytest.raises(AssertionError):
        exact_selection_agrees(ex, ab, ids, nvp, 1, 2)


def test_a_cut_within_the_tolerance_is_skipped():
    ex, ab, nvp = _plane()
    ids = _ids(ex, nvp)
    # head 1: make the best rejected free block tie the last selected one
    # within the tolerances, and hand in the other choice
    h = 1
    sel = [c for c in ids[0, h] if 1 <= c < 38]
    rej = [c for c in range(1, 38) if c not in sel]
    last = min(sel, key=lambda c: (ex[0, h, c], -c))
    best_rej = max(rej, key=lambda c: (ex[0, h, c], -c))
    ex[0, h, best_rej] = ex[0, h, last] - 5e-4     # closer than the two tolerances
    ids = _ids(ex, nvp).copy()
    swapped = np.sort(np.where(ids[0, h] == last, best_rej, ids[0, h]))
    ids[0, h] = np.concatenate([swapped[swapped >= 0], swapped[swapped < 0]])
    checked, skipped = exact_selection_agrees(ex, ab, ids, nvp, 1, 2)
    assert (checked, skipped) == (3, 1)
