"""The oracle against the hand-derived cases in tests/golden/hand_cases.json."""
import json
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _f(x):
    return float("-inf") if x == "-inf" else float(x)


def _load():
    with open(GOLDEN) as f:
        return json.load(f)


def _fp8(v):
    return int(torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def test_golden_score_plane():
    g = _load()["score"]
    dql = g["decode_query_len"]
    T = len(g["seq_lens"]) * dql
    q = np.zeros((T, 4, 128), np.uint8)
    for h, a in enumerate(g["q_dim0_per_head"]):
        q[:, h, 0] = _fp8(a)
    k = np.zeros((g["pool_pages"], 128, 128), np.uint8)
    bt = np.array(g["block_table"], np.int32)
    for pos, dim, v in g["k_nonzero"]:
        k[bt[0, pos // 128], pos % 128, dim] = _fp8(v)
    plane, _ = oracle.score(q, k, bt, np.array(g["seq_lens"], np.int32), cols=g["cols"],
                            rank=g["rank"], world_size=g["world_size"],
                            page_size=g["page_size"], decode_query_len=dql)
    expected = np.array([[[_f(x) for x in row] for row in tok] for tok in g["expected"]])
    assert np.array_equal(plane, expected)


def test_golden_select_row():
    g = _load()["select"]
    sc = np.array([_f(x) for x in g["scores"]], np.float32)
    ids = np.arange(len(sc), dtype=np.int32)
    s, i = oracle.select_pairs(ids, sc, g["num_valid_pages"], g["init_blocks"],
                               g["local_blocks"])
    assert i.tolist() == g["expected_ids"]
    assert s.tolist() == [_f(x) for x in g["expected_scores"]]


def test_golden_recv_row():
    g = _load()["recv_row"]
    assert g["h"] // g["heads_per_rank"] == g["expected_owner"]
    assert oracle.recv_row(g["slot"], g["rank"], g["world_size"], g["heads_per_rank"], g["h"],
                           g["capacity"], g["t"]) == g["expected_row"]
