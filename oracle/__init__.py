"""CPU oracle for the decode-time ICP block indexer (test infrastructure).

This package is the slow, plain reference the CUDA library is checked
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the product package never does.  It shares
no code with the CUDA path: the arithmetic lives in ``icp_oracle.c`` (plain
C, fp64, exact dots), this module only marshals numpy arrays through ctypes.

What each function follows is stated in ``icp_oracle.c``; the page names are
the FlashInfer ``msa_ops`` API pages ``msa_icp_decode_index_score_sharded``
(scoring), ``msa_icp_topk_select_publish`` (Top16 select, receive rows) and
``prepare_msa_icp_indexer`` (forced blocks, the decode chain).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HEADS = 4
DIM = 128
TOPK = 16
ROW_WORDS = 33

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "icp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile icp_oracle.c into liboracle.so next to it (plain gcc, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int, ctypes.c_int64
    lib.icp_orc_e4m3.restype = ctypes.c_double
    lib.icp_orc_e4m3.argtypes = [ctypes.c_uint8]
    lib.icp_orc_columns_with_keys.argtypes = [i32, i32, i32]
    lib.icp_orc_columns_written.argtypes = [i32, i32, i32]
    lib.icp_orc_score.argtypes = [P, P, i64, P, i64, P, i32, i32, i32, i32, i32, i32, P, P]
    lib.icp_orc_select_pairs.argtypes = [i32, P, P, i32, i32, i32, P, P]
    lib.icp_orc_select.argtypes = [P, i32, i32, i32, P, i32, i32, i32, i32, P, P]
    lib.icp_orc_recv_row.restype = ctypes.c_int64
    lib.icp_orc_recv_row.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.icp_orc_publish.argtypes = [P, i32, i32, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32]
    lib.icp_orc_merge.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, i32, P, P]
    lib.icp_orc_publish_tagged.argtypes = [P, i32, i32, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                           i32, i32]
    lib.icp_orc_merge_tagged.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, P, P]
    lib.icp_orc_score_chunks.argtypes = [P, P, i64, P, i64, P, P, i32, i32, i32, i32, i32, P, P]
    lib.icp_orc_carrier.argtypes = [P, i32, i32, P, i32, i32, i32, i32, i32, i32, P]
    lib.icp_orc_merge_carrier.argtypes = [P, P, i32, i32, i32, i32, i32, P, P]
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def e4m3_value(code: int) -> float:
    """Value of one float8_e4m3fn code (NaN for 0x7F / 0xFF)."""
    return _load().icp_orc_e4m3(int(code))


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def columns_with_keys(seq_len: int, page_size: int, world_size: int) -> int:
    return _load().icp_orc_columns_with_keys(int(seq_len), int(page_size), int(world_size))


def columns_written(seq_len: int, page_size: int, world_size: int) -> int:
    return _load().icp_orc_columns_written(int(seq_len), int(page_size), int(world_size))


def score(index_q, index_k, block_table, seq_lens, *, cols, rank, world_size, page_size,
          decode_query_len, fill=np.nan):
    """Exact score plane (float64 [T, 4, cols]) and its |q.k| scale plane.

    index_q: uint8 [B*dql, 4, 128]; index_k: uint8 [pages, page_size/world_size, 128];
    block_table: int32 [B, W]; seq_lens: int32 [B].  Columns outside a
    request's written range keep ``fill``.
    """
    lib = _load()
    q = _c(index_q, np.uint8)
    k = _c(index_k, np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    B = sl.shape[0]
    T = B * decode_query_len
    assert q.shape == (T, HEADS, DIM), q.shape
    assert k.ndim == 3 and k.shape[1] == page_size // world_size and k.shape[2] == DIM
    plane = np.full((T, HEADS, cols), fill, dtype=np.float64)
    absplane = np.full((T, HEADS, cols), fill, dtype=np.float64)
    stride = bt.shape[1] if bt.ndim == 2 else 0
    rc = lib.icp_orc_score(_ptr(q), _ptr(k), k.shape[0], _ptr(bt), stride, _ptr(sl), B, cols,
                           rank, world_size, page_size, decode_query_len, _ptr(plane),
                           _ptr(absplane))
    if rc != 0:
        raise ValueError(f"icp_orc_score failed with {rc}")
    return plane, absplane


def select_pairs(ids, scores, nvp, init_blocks, local_blocks):
    lib = _load()
    ids = _c(ids, np.int32)
    sc = _c(scores, np.float32)
    out_s = np.empty(TOPK, np.float32)
    out_i = np.empty(TOPK, np.int32)
    n = lib.icp_orc_select_pairs(ids.shape[0], _ptr(ids), _ptr(sc), int(nvp), init_blocks,
                                 local_blocks, _ptr(out_s), _ptr(out_i))
    if n < 0:
        raise ValueError("icp_orc_select_pairs failed")
    return out_s, out_i


def select(scores, num_valid_pages, *, init_blocks, local_blocks, index_scale=1,
           index_offset=0):
    """Top16 per row of a float32 plane [T, H, K] -> (scores [T,H,16], ids [T,H,16])."""
    lib = _load()
    sc = _c(scores, np.float32)
    nvp = _c(num_valid_pages, np.int32)
    T, H, K = sc.shape
    out_s = np.empty((T, H, TOPK), np.float32)
    out_i = np.empty((T, H, TOPK), np.int32)
    rc = lib.icp_orc_select(_ptr(sc), T, H, K, _ptr(nvp), init_blocks, local_blocks,
                            index_scale, index_offset, _ptr(out_s), _ptr(out_i))
    if rc != 0:
        raise ValueError("icp_orc_select failed")
    return out_s, out_i


def recv_row(slot, rank, world_size, heads_per_rank, h, capacity, t) -> int:
    return _load().icp_orc_recv_row(slot, rank, world_size, heads_per_rank, h, capacity, t)


def recv_rows_per_owner(world_size, heads_per_rank, capacity) -> int:
    return 3 * world_size * heads_per_rank * capacity


def publish(scores, num_valid_pages, recv, *, slot, rank, world_size, heads_per_rank, capacity,
            force_begin_blocks, force_end_blocks, index_scale=1, index_offset=0) -> int:
    """Write legacy rows into ``recv`` (list of ws int32 arrays [rows, 33]); returns #busy rows."""
    lib = _load()
    sc = _c(scores, np.float32)
    nvp = _c(num_valid_pages, np.int32)
    T, H, K = sc.shape
    assert H == world_size * heads_per_rank
    for r in recv:
        assert r.dtype == np.int32 and r.flags.c_contiguous
    arr = (ctypes.c_void_p * world_size)(*[r.ctypes.data for r in recv])
    rc = lib.icp_orc_publish(_ptr(sc), T, K, _ptr(nvp), arr, slot, rank, world_size,
                             heads_per_rank, capacity, force_begin_blocks, force_end_blocks,
                             index_scale, index_offset)
    if rc < 0:
        raise ValueError("icp_orc_publish failed")
    return rc


def merge(recv, num_valid_pages, *, T, slot, owner, world_size, heads_per_rank, capacity,
          init_blocks, local_blocks):
    """Owner merge of its receive rows -> (scores [T,hpr,16], ids [T,hpr,16], #missing)."""
    lib = _load()
    assert recv.dtype == np.int32 and recv.flags.c_contiguous
    nvp = _c(num_valid_pages, np.int32)
    out_s = np.empty((T, heads_per_rank, TOPK), np.float32)
    out_i = np.empty((T, heads_per_rank, TOPK), np.int32)
    rc = lib.icp_orc_merge(_ptr(recv), _ptr(nvp), T, slot, owner, world_size, heads_per_rank,
                           capacity, init_blocks, local_blocks, _ptr(out_s), _ptr(out_i))
    if rc < 0:
        raise ValueError("icp_orc_merge failed")
    return out_s, out_i, rc


def publish_tagged(scores, num_valid_pages, recv, generations, *, slot, rank, world_size,
                   heads_per_rank, capacity, force_begin_blocks, force_end_blocks,
                   index_scale=1, index_offset=0):
    """Tagged publish into ``recv`` (ws int64 arrays [rows, 32]); advances
    ``generations`` (int32 [3, ws*hpr, capacity])."""
    lib = _load()
    sc = _c(scores, np.float32)
    nvp = _c(num_valid_pages, np.int32)
    T, H, K = sc.shape
    for r in recv:
        assert r.dtype == np.int64 and r.flags.c_contiguous
    assert generations.dtype == np.int32 and generations.flags.c_contiguous
    arr = (ctypes.c_void_p * world_size)(*[r.ctypes.data for r in recv])
    rc = lib.icp_orc_publish_tagged(_ptr(sc), T, K, _ptr(nvp), arr, _ptr(generations), slot, rank,
                                    world_size, heads_per_rank, capacity, force_begin_blocks,
                                    force_end_blocks, index_scale, index_offset)
    if rc < 0:
        raise ValueError("icp_orc_publish_tagged failed")


def merge_tagged(recv, expected, num_valid_pages, *, T, slot, world_size, heads_per_rank,
                 capacity, init_blocks, local_blocks):
    """Owner merge of tagged rows -> (scores, ids, #sources that had not arrived)."""
    lib = _load()
    assert recv.dtype == np.int64 and recv.flags.c_contiguous
    assert expected.dtype == np.int32 and expected.flags.c_contiguous
    nvp = _c(num_valid_pages, np.int32)
    out_s = np.empty((T, heads_per_rank, TOPK), np.float32)
    out_i = np.empty((T, heads_per_rank, TOPK), np.int32)
    rc = lib.icp_orc_merge_tagged(_ptr(recv), _ptr(expected), _ptr(nvp), T, slot, world_size,
                                  heads_per_rank, capacity, init_blocks, local_blocks,
                                  _ptr(out_s), _ptr(out_i))
    if rc < 0:
        raise ValueError("icp_orc_merge_tagged failed")
    return out_s, out_i, rc


def sharded_merge_equals_unsharded(index_q, index_k_full, block_table, seq_lens,
                                   num_valid_pages, *, world_size, page_size, decode_query_len,
                                   cols, init_blocks, local_blocks, slot=0):
    """Score every shard, publish, merge per owner, and compare with the
    unsharded Top16 of the fp32-rounded exact plane.  Returns
    (merged_scores [T,4,16], merged_ids, unsharded_scores, unsharded_ids);
    raises AssertionError if they differ in any bit.

    For P256 sharded layouts the shard plane has one column per local page
    and the global id of column c is 2c + rank*2//world_size.
    """
    ws = world_size
    hpr = HEADS // ws
    T = len(seq_lens) * decode_query_len
    k_full = np.asarray(index_k_full, np.uint8)
    # unsharded reference: P128 -> columns are B128 blocks; P256 unsharded uses
    # the B128-block extension, so both give one column per global block.
    full_cols = cols if page_size == 128 else 2 * cols
    full_plane, _ = score(index_q, k_full, block_table, seq_lens, cols=full_cols, rank=0,
                          world_size=1, page_size=page_size, decode_query_len=decode_query_len,
                          fill=-np.inf)
    ref_s, ref_i = select(full_plane.astype(np.float32), num_valid_pages,
                          init_blocks=init_blocks, local_blocks=local_blocks)
    capacity = T
    recv = [np.zeros((recv_rows_per_owner(ws, hpr, capacity), ROW_WORDS), np.int32)
            for _ in range(ws)]
    rp = page_size // ws
    for rank in range(ws):
        shard = np.ascontiguousarray(k_full[:, rank * rp:(rank + 1) * rp, :])
        plane, _ = score(index_q, shard, block_table, seq_lens, cols=cols, rank=rank,
                         world_size=ws, page_size=page_size, decode_query_len=decode_query_len,
                         fill=-np.inf)
        scale, offset = (1, 0) if page_size == 128 else (2, rank * 2 // ws)
        busy = publish(plane.astype(np.float32), num_valid_pages, recv, slot=slot, rank=rank,
                       world_size=ws, heads_per_rank=hpr, capacity=capacity,
                       force_begin_blocks=init_blocks, force_end_blocks=local_blocks,
                       index_scale=scale, index_offset=offset)
        assert busy == 0
    out_s = np.empty((T, HEADS, TOPK), np.float32)
    out_i = np.empty((T, HEADS, TOPK), np.int32)
    for owner in range(ws):
        s, i, missing = merge(recv[owner], num_valid_pages, T=T, slot=slot, owner=owner,
                              world_size=ws, heads_per_rank=hpr, capacity=capacity,
                              init_blocks=init_blocks, local_blocks=local_blocks)
        assert missing == 0
        out_s[:, owner * hpr:(owner + 1) * hpr] = s
        out_i[:, owner * hpr:(owner + 1) * hpr] = i
    assert np.array_equal(out_i, ref_i), "merged ids differ from the unsharded Top16"
    assert np.array_equal(out_s.view(np.int32), ref_s.view(np.int32)), \
        "merged scores differ from the unsharded Top16"
    return out_s, out_i, ref_s, ref_i


CARRIER_WORDS = 32


def score_chunks(index_q, index_k, block_table, seq_lens, qo_indptr, *, cols, rank, world_size,
                 page_size, fill=np.nan):
    """Exact score plane of a prefill window (float64 [T, 4, cols]) and its
    |q.k| scale plane.  Request b's tokens are rows qo_indptr[b] ..
    qo_indptr[b+1] - 1, the newest positions of its seq_len (the decode plane
    with a per-request query length; see icp_orc_score_chunks)."""
    lib = _load()
    q = _c(index_q, np.uint8)
    k = _c(index_k, np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    qo = _c(qo_indptr, np.int32)
    B = sl.shape[0]
    assert qo.shape == (B + 1,)
    T = int(qo[-1])
    assert q.shape[0] >= T and q.shape[1:] == (HEADS, DIM), q.shape
    assert k.ndim == 3 and k.shape[1] == page_size // world_size and k.shape[2] == DIM
    plane = np.full((T, HEADS, cols), fill, dtype=np.float64)
    absplane = np.full((T, HEADS, cols), fill, dtype=np.float64)
    stride = bt.shape[1] if bt.ndim == 2 else 0
    rc = lib.icp_orc_score_chunks(_ptr(q), _ptr(k), k.shape[0], _ptr(bt), stride, _ptr(sl),
                                  _ptr(qo), B, cols, rank, world_size, page_size, _ptr(plane),
                                  _ptr(absplane))
    if rc != 0:
        raise ValueError(f"icp_orc_score_chunks failed with {rc}")
    return plane, absplane


def carrier(scores, num_valid_pages, *, world_size, heads_per_rank, init_blocks, local_blocks,
            index_scale=1, index_offset=0):
    """One rank's carrier rows int32 [ws, T, hpr, 32] from its plane [T, ws*hpr, K]."""
    lib = _load()
    sc = _c(scores, np.float32)
    nvp = _c(num_valid_pages, np.int32)
    T, H, K = sc.shape
    assert H == world_size * heads_per_rank
    out = np.zeros((world_size, T, heads_per_rank, CARRIER_WORDS), np.int32)
    rc = lib.icp_orc_carrier(_ptr(sc), T, K, _ptr(nvp), world_size, heads_per_rank, init_blocks,
                             local_blocks, index_scale, index_offset, _ptr(out))
    if rc != 0:
        raise ValueError("icp_orc_carrier failed")
    return out


def merge_carrier(received, num_valid_pages, *, world_size, heads_per_rank, init_blocks,
                  local_blocks):
    """Owner merge of received carrier rows int32 [ws, T, hpr, 32] ->
    (scores [T,hpr,16], ids [T,hpr,16])."""
    lib = _load()
    rc_ = _c(received, np.int32)
    nvp = _c(num_valid_pages, np.int32)
    ws, T, hpr, w = rc_.shape
    assert ws == world_size and hpr == heads_per_rank and w == CARRIER_WORDS
    out_s = np.empty((T, hpr, TOPK), np.float32)
    out_i = np.empty((T, hpr, TOPK), np.int32)
    rc = lib.icp_orc_merge_carrier(_ptr(rc_), _ptr(nvp), T, world_size, heads_per_rank,
                                   init_blocks, local_blocks, _ptr(out_s), _ptr(out_i))
    if rc != 0:
        raise ValueError("icp_orc_merge_carrier failed")
    return out_s, out_i
