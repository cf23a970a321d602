"""ctypes binding to libicp.so: same names and argument order as include/icp.h.

Marshalling only: each function checks dtypes, shapes, devices and
contiguity of the torch tensors, then passes ``data_ptr()`` values and the
current CUDA stream to the C entry point.  Every step of the computation runs
in the library's CUDA kernels.  Importing this module fails loudly when the
library has not been built (``python -m sparse_attention_block_gb300.build``);
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# ICP_LIBRARY names another build of the same library (the timeline build)
LIB_PATH = os.environ.get("ICP_LIBRARY") or os.path.join(_HERE, "_lib", "libicp.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m sparse_attention_block_gb300.build`")

lib = ctypes.CDLL(LIB_PATH)

HEADS, DIM, TOPK, ROW_WORDS = 4, 128, 16, 33
MAX_COLS, MAX_K, MAX_BATCH = 8192, 12287, 4096
DEFAULT_SPIN_LIMIT = 67108864

OK, ERR_INVALID_ARG, ERR_CUDA, ERR_UNSUPPORTED, ERR_TIMEOUT = 0, 1, 2, 3, 4

_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t

lib.icp_status_string.restype = ctypes.c_char_p
lib.icp_status_string.argtypes = [_I32]
lib.icp_score_columns.restype = _I32
lib.icp_score_columns.argtypes = [_I32, _I32, _I32]
lib.icp_score.restype = _I32
lib.icp_score.argtypes = [_P, _P, _I64, _P, _I64, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                          _I32, _I32, _P, _P]
lib.icp_top16_select.restype = _I32
lib.icp_top16_select.argtypes = [_P, _I32, _I32, _P, _I32, _I32, _I32, _I32, _P, _P, _P]
lib.icp_publish_rows.restype = _I32
lib.icp_publish_rows.argtypes = [_P, _I32, _I32, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                                 _I32, _I64, _I32, _I32, _I32, _P]
lib.icp_score_select_workspace_bytes.restype = _SZ
lib.icp_score_select_workspace_bytes.argtypes = [_I32, _I32]
lib.icp_score_select.restype = _I32
lib.icp_score_select.argtypes = [_P, _P, _I64, _P, _I64, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                                 _I32, _P, _I32, _I32, _P, _SZ, _P, _P, _P, _P]
lib.icp_score_select_noalloc.restype = _I32
lib.icp_score_select_noalloc.argtypes = [_P, _P, _I64, _P, _I64, _P, _I32, _I32, _I32, _I32,
                                         _I32, _I32, _I32, _P, _I32, _I32, _P, _P, _P, _P]
lib.icp_publish_rows_tagged.restype = _I32
lib.icp_publish_rows_tagged.argtypes = [_P, _I32, _I32, _P, _P, _P, _I32, _I32, _I32, _I32,
                                        _I32, _I32, _I32, _I32, _I32, _I32, _P]
lib.icp_merge_tagged.restype = _I32
lib.icp_merge_tagged.argtypes = [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I64,
                                 _P, _P, _P, _I32, _P]
lib.icp_merge.restype = _I32
lib.icp_merge.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I64, _P, _P, _P,
                          _I32, _P]
lib.icp_prefill_plan_words.restype = _I64
lib.icp_prefill_plan_words.argtypes = [_I32, _I32]
lib.icp_prefill_plan.restype = _I32
lib.icp_prefill_plan.argtypes = [_P, _P, _I32, _I32, _P, _I64, _P, _P]
lib.icp_prefill_score.restype = _I32
lib.icp_prefill_score.argtypes = [_P, _P, _I64, _P, _I64, _P, _I64, _P, _I32, _I32, _I32, _I32,
                                  _I32, _P, _P]
lib.icp_prefill_select.restype = _I32
lib.icp_prefill_select.argtypes = [_P, _I32, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P,
                                   _P]
lib.icp_prefill_merge.restype = _I32
lib.icp_prefill_merge.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P]


class IcpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.icp_status_string(status).decode()} (status {status})")


def _check(status: int, where: str):
    if status != OK:
        raise IcpError(status, where)


def icp_check_errors(errors, where: str = "icp"):
    """Reads the `errors` counter (a device-to-host copy, so it waits for the
    work queued before it) and raises IcpError(ERR_TIMEOUT) when a bounded
    device wait ran out.  Not for the hot path: call it where the caller
    synchronizes anyway."""
    if int(errors.sum().item()) > 0:
        raise IcpError(ERR_TIMEOUT, where)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtypes, ndim=None, contiguous=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


_FP8 = (torch.uint8, torch.float8_e4m3fn)


def _on_current_device(*tensors):
    """The library launches on the current CUDA device: every tensor must live
    there (a tensor of another device would be read through a foreign
    pointer)."""
    cur = torch.cuda.current_device()
    for t in tensors:
        if t is not None and t.get_device() != cur:
            raise ValueError(f"a tensor is on {t.device}, the current device is cuda:{cur}")


def _rows_at_least(t, n: int, name: str):
    if t.shape[0] < n:
        raise ValueError(f"{name} has {t.shape[0]} rows, the call reads {n}")


def icp_score_columns(max_seq_len: int, page_size: int, world_size: int) -> int:
    cols = lib.icp_score_columns(int(max_seq_len), int(page_size), int(world_size))
    if cols < 0:
        raise ValueError("invalid arguments for icp_score_columns")
    return cols


def icp_score(index_q, index_k, block_table, seq_lens, score_out, *, rank: int, world_size: int,
              page_size: int, decode_query_len: int, max_decode_query_len: int,
              enable_pdl: bool = False, errors=None, stream=None):
    """Decode index scores into score_out [T, 4, cols] (msa_icp_decode_index_score_sharded).

    enable_pdl: start early under programmatic dependent launch (see include/icp.h)."""
    B = seq_lens.shape[0]
    T = B * decode_query_len
    qp = _dev(index_q, "index_q", _FP8, 3)
    kp = _dev(index_k, "index_k", _FP8, 3)
    if tuple(index_q.shape) != (T, HEADS, DIM):
        raise ValueError(f"index_q must be [{T}, 4, 128], got {tuple(index_q.shape)}")
    if tuple(index_k.shape[1:]) != (page_size // world_size, DIM):
        raise ValueError(f"index_k must be [pages, {page_size // world_size}, 128]")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be 2-D with unit last stride")
    btp = _dev(block_table, "block_table", (torch.int32,), 2, contiguous=False)
    slp = _dev(seq_lens, "seq_lens", (torch.int32,), 1)
    sop = _dev(score_out, "score_out", (torch.float32,), 3)
    if score_out.shape[0] != T or score_out.shape[1] != HEADS:
        raise ValueError(f"score_out must be [{T}, 4, cols]")
    ep = 0 if errors is None else _dev(errors, "errors", (torch.int32,), 1)
    _rows_at_least(block_table, B, "block_table")
    _on_current_device(index_q, index_k, block_table, seq_lens, score_out, errors)
    _check(lib.icp_score(qp, kp, index_k.shape[0], btp, block_table.stride(0), slp, sop, B,
                         score_out.shape[2], rank, world_size, page_size, decode_query_len,
                         max_decode_query_len, 1 if enable_pdl else 0, ep, _stream(stream)),
           "icp_score")


def icp_top16_select(scores, num_valid_pages, out_scores, out_ids, *, init_blocks: int,
                     local_blocks: int, index_scale: int = 1, index_offset: int = 0,
                     stream=None):
    """Top16 of every (token, head) row of scores [T, 4, K] into out_* [T, 4, 16]."""
    sp = _dev(scores, "scores", (torch.float32,), 3)
    T, H, K = scores.shape
    if H != HEADS:
        raise ValueError("scores must have 4 heads")
    np_ = _dev(num_valid_pages, "num_valid_pages", (torch.int32,), 1)
    if num_valid_pages.shape[0] != T:
        raise ValueError("num_valid_pages must be [T]")
    osp = _dev(out_scores, "out_scores", (torch.float32,), 3)
    oip = _dev(out_ids, "out_ids", (torch.int32,), 3)
    if tuple(out_scores.shape) != (T, HEADS, TOPK) or tuple(out_ids.shape) != (T, HEADS, TOPK):
        raise ValueError("out_scores / out_ids must be [T, 4, 16]")
    _on_current_device(scores, num_valid_pages, out_scores, out_ids)
    _check(lib.icp_top16_select(sp, T, K, np_, init_blocks, local_blocks, index_scale,
                                index_offset, osp, oip, _stream(stream)), "icp_top16_select")


def recv_rows(world_size: int, heads_per_rank: int, capacity: int) -> int:
    """Rows of one owner's legacy receive storage: [3][ws][hpr][capacity]."""
    return 3 * world_size * heads_per_rank * capacity


def icp_publish_rows(scores, num_valid_pages, recv_bases, errors, *, slot: int, rank: int,
                     world_size: int, heads_per_rank: int, capacity: int,
                     force_begin_blocks: int, force_end_blocks: int,
                     spin_limit: int = DEFAULT_SPIN_LIMIT, index_scale: int = 1,
                     index_offset: int = 0, enable_pdl: bool = False, stream=None):
    """Top16 select + publish into legacy receive rows (msa_icp_topk_select_publish).

    enable_pdl: launch with programmatic dependent launch (see include/icp.h)."""
    sp = _dev(scores, "scores", (torch.float32,), 3)
    T, H, K = scores.shape
    if H != world_size * heads_per_rank:
        raise ValueError("scores must have world_size * heads_per_rank heads")
    np_ = _dev(num_valid_pages, "num_valid_pages", (torch.int32,), 1)
    rbp = _dev(recv_bases, "recv_bases", (torch.int64,), 1)
    if recv_bases.shape[0] != world_size:
        raise ValueError("recv_bases must be [world_size]")
    ep = _dev(errors, "errors", (torch.int32,), 1)
    _rows_at_least(num_valid_pages, T, "num_valid_pages")
    _rows_at_least(errors, 1, "errors")
    _on_current_device(scores, num_valid_pages, recv_bases, errors)
    _check(lib.icp_publish_rows(sp, T, K, np_, rbp, ep, slot, rank, world_size, heads_per_rank,
                                capacity, force_begin_blocks, force_end_blocks, spin_limit,
                                index_scale, index_offset, 1 if enable_pdl else 0,
                                _stream(stream)), "icp_publish_rows")


def icp_merge(recv, num_valid_pages, out_scores, out_ids, errors, *, T: int, slot: int,
              world_size: int, heads_per_rank: int, capacity: int, init_blocks: int,
              local_blocks: int, spin_limit: int = DEFAULT_SPIN_LIMIT, enable_pdl: bool = False,
              stream=None):
    """Owner merge of this owner's receive rows into out_* [T, heads_per_rank, 16].

    enable_pdl: launch with programmatic dependent launch (see include/icp.h)."""
    rp = _dev(recv, "recv", (torch.int32,), None)
    if recv.numel() < recv_rows(world_size, heads_per_rank, capacity) * ROW_WORDS:
        raise ValueError("recv is smaller than [3][ws][hpr][capacity][33]")
    np_ = _dev(num_valid_pages, "num_valid_pages", (torch.int32,), 1)
    osp = _dev(out_scores, "out_scores", (torch.float32,), 3)
    oip = _dev(out_ids, "out_ids", (torch.int32,), 3)
    if tuple(out_scores.shape) != (T, heads_per_rank, TOPK) or \
            tuple(out_ids.shape) != (T, heads_per_rank, TOPK):
        raise ValueError("out_scores / out_ids must be [T, heads_per_rank, 16]")
    ep = _dev(errors, "errors", (torch.int32,), 1)
    _rows_at_least(num_valid_pages, T, "num_valid_pages")
    _rows_at_least(errors, 1, "errors")
    _on_current_device(recv, num_valid_pages, out_scores, out_ids, errors)
    _check(lib.icp_merge(rp, np_, T, slot, world_size, heads_per_rank, capacity, init_blocks,
                         local_blocks, spin_limit, ep, osp, oip, 1 if enable_pdl else 0,
                         _stream(stream)), "icp_merge")


def icp_score_select_workspace_bytes(batch: int, decode_query_len: int) -> int:
    n = lib.icp_score_select_workspace_bytes(int(batch), int(decode_query_len))
    if n == 0 and batch > 0:
        raise ValueError("invalid arguments for icp_score_select_workspace_bytes")
    return n


def icp_score_select(index_q, index_k, block_table, seq_lens, num_valid_pages, out_scores,
                     out_ids, workspace, *, cols: int, rank: int, world_size: int,
                     page_size: int, decode_query_len: int, max_decode_query_len: int,
                     init_blocks: int, local_blocks: int, errors=None, stream=None):
    """Fused scorer + Top16 select (no score plane) into out_* [T, 4, 16].

    ``workspace`` is a uint8 device tensor of at least
    icp_score_select_workspace_bytes(batch, decode_query_len) bytes (256-byte aligned).
    """
    B = seq_lens.shape[0]
    T = B * decode_query_len
    qp = _dev(index_q, "index_q", _FP8, 3)
    kp = _dev(index_k, "index_k", _FP8, 3)
    if tuple(index_q.shape) != (T, HEADS, DIM):
        raise ValueError(f"index_q must be [{T}, 4, 128], got {tuple(index_q.shape)}")
    if tuple(index_k.shape[1:]) != (page_size // world_size, DIM):
        raise ValueError(f"index_k must be [pages, {page_size // world_size}, 128]")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be 2-D with unit last stride")
    btp = _dev(block_table, "block_table", (torch.int32,), 2, contiguous=False)
    slp = _dev(seq_lens, "seq_lens", (torch.int32,), 1)
    np_ = _dev(num_valid_pages, "num_valid_pages", (torch.int32,), 1)
    osp = _dev(out_scores, "out_scores", (torch.float32,), 3)
    oip = _dev(out_ids, "out_ids", (torch.int32,), 3)
    if tuple(out_scores.shape) != (T, HEADS, TOPK) or tuple(out_ids.shape) != (T, HEADS, TOPK):
        raise ValueError("out_scores / out_ids must be [T, 4, 16]")
    wp = _dev(workspace, "workspace", (torch.uint8,), 1)
    ep = 0 if errors is None else _dev(errors, "errors", (torch.int32,), 1)
    _rows_at_least(block_table, B, "block_table")
    _rows_at_least(num_valid_pages, T, "num_valid_pages")
    _on_current_device(index_q, index_k, block_table, seq_lens, num_valid_pages, out_scores,
                       out_ids, workspace, errors)
    _check(lib.icp_score_select(qp, kp, index_k.shape[0], btp, block_table.stride(0), slp, B,
                                cols, rank, world_size, page_size, decode_query_len,
                                max_decode_query_len, np_, init_blocks, local_blocks, wp,
                                workspace.numel(), osp, oip, ep, _stream(stream)),
           "icp_score_select")


def icp_publish_rows_tagged(scores, num_valid_pages, recv_bases, generations, *, slot: int,
                            rank: int, world_size: int, heads_per_rank: int, capacity: int,
                            force_begin_blocks: int, force_end_blocks: int,
                            index_scale: int = 1, index_offset: int = 0,
                            enable_pdl: bool = False, stream=None):
    """Top16 select + publish into tagged receive rows (int64 generation << 32 | word)."""
    sp = _dev(scores, "scores", (torch.float32,), 3)
    T, H, K = scores.shape
    if H != world_size * heads_per_rank:
        raise ValueError("scores must have world_size * heads_per_rank heads")
    np_ = _dev(num_valid_pages, "num_valid_pages", (torch.int32,), 1)
    rbp = _dev(recv_bases, "recv_bases", (torch.int64,), 1)
    if recv_bases.shape[0] != world_size:
        raise ValueError("recv_bases must be [world_size]")
    gp = _dev(generations, "generations", (torch.int32,), 3)
    if tuple(generations.shape) != (3, world_size * heads_per_rank, capacity):
        raise ValueError("generations must be [3, world_size * heads_per_rank, capacity]")
    _rows_at_least(num_valid_pages, T, "num_valid_pages")
    _on_current_device(scores, num_valid_pages, recv_bases, generations)
    _check(lib.icp_publish_rows_tagged(sp, T, K, np_, rbp, gp, slot, rank, world_size,
                                       heads_per_rank, capacity, force_begin_blocks,
                                       force_end_blocks, index_scale, index_offset,
                                       1 if enable_pdl else 0, _stream(stream)),
           "icp_publish_rows_tagged")


def icp_merge_tagged(recv, expected, num_valid_pages, out_scores, out_ids, errors, *, T: int,
                     slot: int, world_size: int, heads_per_rank: int, capacity: int,
                     init_blocks: int, local_blocks: int, spin_limit: int = DEFAULT_SPIN_LIMIT,
                     enable_pdl: bool = False, stream=None):
    """Owner merge of tagged rows into out_* [T, heads_per_rank, 16]."""
    rp = _dev(recv, "recv", (torch.int64,), None)
    if recv.numel() < recv_rows(world_size, heads_per_rank, capacity) * 32:
        raise ValueError("recv is smaller than [3][ws][hpr][capacity][32]")
    ep_ = _dev(expected, "expected", (torch.int32,), None)
    if expected.numel() < recv_rows(world_size, heads_per_rank, capacity):
        raise ValueError("expected must hold [3][ws][hpr][capacity] counters")
    np_ = _dev(num_valid_pages, "num_valid_pages", (torch.int32,), 1)
    osp = _dev(out_scores, "out_scores", (torch.float32,), 3)
    oip = _dev(out_ids, "out_ids", (torch.int32,), 3)
    if tuple(out_scores.shape) != (T, heads_per_rank, TOPK) or \
            tuple(out_ids.shape) != (T, heads_per_rank, TOPK):
        raise ValueError("out_scores / out_ids must be [T, heads_per_rank, 16]")
    erp = _dev(errors, "errors", (torch.int32,), 1)
    _rows_at_least(num_valid_pages, T, "num_valid_pages")
    _rows_at_least(errors, 1, "errors")
    _on_current_device(recv, expected, num_valid_pages, out_scores, out_ids, errors)
    _check(lib.icp_merge_tagged(rp, ep_, np_, T, slot, world_size, heads_per_rank, capacity,
                                init_blocks, local_blocks, spin_limit, erp, osp, oip,
                                1 if enable_pdl else 0, _stream(stream)), "icp_merge_tagged")


NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024


def icp_score_select_noalloc(index_q, index_k, block_table, seq_lens, num_valid_pages,
                             out_scores, out_ids, *, cols: int, rank: int, world_size: int,
                             page_size: int, decode_query_len: int, max_decode_query_len: int,
                             init_blocks: int, local_blocks: int, errors=None, stream=None):
    """icp_score_select with the library's fixed scratch array instead of a
    workspace, for callers that cannot allocate device memory at call time.
    Raises IcpError (invalid argument) when the batch needs more scratch than
    NOALLOC_SCRATCH_BYTES."""
    B = seq_lens.shape[0]
    T = B * decode_query_len
    qp = _dev(index_q, "index_q", _FP8, 3)
    kp = _dev(index_k, "index_k", _FP8, 3)
    if tuple(index_q.shape) != (T, HEADS, DIM):
        raise ValueError(f"index_q must be [{T}, 4, 128], got {tuple(index_q.shape)}")
    if tuple(index_k.shape[1:]) != (page_size // world_size, DIM):
        raise ValueError(f"index_k must be [pages, {page_size // world_size}, 128]")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be 2-D with unit last stride")
    btp = _dev(block_table, "block_table", (torch.int32,), 2, contiguous=False)
    slp = _dev(seq_lens, "seq_lens", (torch.int32,), 1)
    np_ = _dev(num_valid_pages, "num_valid_pages", (torch.int32,), 1)
    osp = _dev(out_scores, "out_scores", (torch.float32,), 3)
    oip = _dev(out_ids, "out_ids", (torch.int32,), 3)
    if tuple(out_scores.shape) != (T, HEADS, TOPK) or tuple(out_ids.shape) != (T, HEADS, TOPK):
        raise ValueError("out_scores / out_ids must be [T, 4, 16]")
    ep = 0 if errors is None else _dev(errors, "errors", (torch.int32,), 1)
    _rows_at_least(block_table, B, "block_table")
    _rows_at_least(num_valid_pages, T, "num_valid_pages")
    _on_current_device(index_q, index_k, block_table, seq_lens, num_valid_pages, out_scores,
                       out_ids, errors)
    _check(lib.icp_score_select_noalloc(qp, kp, index_k.shape[0], btp, block_table.stride(0),
                                        slp, B, cols, rank, world_size, page_size,
                                        decode_query_len, max_decode_query_len, np_,
                                        init_blocks, local_blocks, osp, oip, ep,
                                        _stream(stream)), "icp_score_select_noalloc")


# ------------------------------------------------------------------ prefill
CARRIER_WORDS = 32


def icp_prefill_plan_words(batch: int, T: int) -> int:
    """int32 words of a prefill plan for a window of T tokens from batch requests."""
    n = lib.icp_prefill_plan_words(int(batch), int(T))
    if n < 0:
        raise ValueError("invalid arguments for icp_prefill_plan_words (too many records?)")
    return n


def icp_prefill_plan(qo_indptr, seq_lens, plan, *, T: int, errors=None, stream=None):
    """prefill_window_plan: every request's chunk as records of up to 64 tokens, into plan."""
    B = seq_lens.shape[0]
    qp = _dev(qo_indptr, "qo_indptr", (torch.int32,), 1)
    if qo_indptr.shape[0] != B + 1:
        raise ValueError("qo_indptr must be [batch + 1]")
    slp = _dev(seq_lens, "seq_lens", (torch.int32,), 1)
    pp = _dev(plan, "plan", (torch.int32,), 1)
    ep = 0 if errors is None else _dev(errors, "errors", (torch.int32,), 1)
    _on_current_device(qo_indptr, seq_lens, plan, errors)
    _check(lib.icp_prefill_plan(qp, slp, B, int(T), pp, plan.numel(), ep, _stream(stream)),
           "icp_prefill_plan")


def icp_prefill_score(index_q, index_k, block_table, plan, score_out, *, rank: int,
                      world_size: int, page_size: int, errors=None, stream=None):
    """prefill_local, scoring half: the window's plane score_out [T, 4, cols]."""
    T = index_q.shape[0]
    qp = _dev(index_q, "index_q", _FP8, 3)
    kp = _dev(index_k, "index_k", _FP8, 3)
    if tuple(index_q.shape[1:]) != (HEADS, DIM):
        raise ValueError("index_q must be [T, 4, 128]")
    if tuple(index_k.shape[1:]) != (page_size // world_size, DIM):
        raise ValueError(f"index_k must be [pages, {page_size // world_size}, 128]")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be 2-D with unit last stride")
    btp = _dev(block_table, "block_table", (torch.int32,), 2, contiguous=False)
    pp = _dev(plan, "plan", (torch.int32,), 1)
    sop = _dev(score_out, "score_out", (torch.float32,), 3)
    if score_out.shape[0] != T or score_out.shape[1] != HEADS:
        raise ValueError(f"score_out must be [{T}, 4, cols]")
    ep = 0 if errors is None else _dev(errors, "errors", (torch.int32,), 1)
    _on_current_device(index_q, index_k, block_table, plan, score_out, errors)
    _check(lib.icp_prefill_score(qp, kp, index_k.shape[0], btp, block_table.stride(0), pp,
                                 plan.numel(), sop, T, score_out.shape[2], rank, world_size,
                                 page_size, ep, _stream(stream)), "icp_prefill_score")


def icp_prefill_select(scores, num_valid_pages, carrier, *, world_size: int,
                       heads_per_rank: int, init_blocks: int, local_blocks: int,
                       index_scale: int = 1, index_offset: int = 0, stream=None):
    """prefill_local, list half: Top16 per row into carrier [ws, T, hpr, 32]."""
    sp = _dev(scores, "scores", (torch.float32,), 3)
    T, H, K = scores.shape
    if H != world_size * heads_per_rank:
        raise ValueError("scores must be [T, world_size * heads_per_rank, K]")
    np_ = _dev(num_valid_pages, "num_valid_pages", (torch.int32,), 1)
    cp = _dev(carrier, "carrier", (torch.int32,), 4)
    if tuple(carrier.shape) != (world_size, T, heads_per_rank, CARRIER_WORDS):
        raise ValueError("carrier must be [world_size, T, heads_per_rank, 32]")
    _rows_at_least(num_valid_pages, T, "num_valid_pages")
    _on_current_device(scores, num_valid_pages, carrier)
    _check(lib.icp_prefill_select(sp, T, K, np_, world_size, heads_per_rank, init_blocks,
                                  local_blocks, index_scale, index_offset, cp, _stream(stream)),
           "icp_prefill_select")


def icp_prefill_merge(received, num_valid_pages, out_scores, out_ids, *, world_size: int,
                      heads_per_rank: int, init_blocks: int, local_blocks: int, stream=None):
    """prefill_merge: received carrier rows [ws, T, hpr, 32] -> out_* [T, hpr, 16]."""
    rp = _dev(received, "received", (torch.int32,), 4)
    ws, T, hpr, w = received.shape
    if ws != world_size or hpr != heads_per_rank or w != CARRIER_WORDS:
        raise ValueError("received must be [world_size, T, heads_per_rank, 32]")
    np_ = _dev(num_valid_pages, "num_valid_pages", (torch.int32,), 1)
    osp = _dev(out_scores, "out_scores", (torch.float32,), 3)
    oip = _dev(out_ids, "out_ids", (torch.int32,), 3)
    if tuple(out_scores.shape) != (T, hpr, TOPK) or tuple(out_ids.shape) != (T, hpr, TOPK):
        raise ValueError("out_scores / out_ids must be [T, heads_per_rank, 16]")
    _rows_at_least(num_valid_pages, T, "num_valid_pages")
    _on_current_device(received, num_valid_pages, out_scores, out_ids)
    _check(lib.icp_prefill_merge(rp, np_, T, world_size, heads_per_rank, init_blocks,
                                 local_blocks, osp, oip, _stream(stream)), "icp_prefill_merge")
