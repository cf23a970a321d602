"""Seeded synthetic inputs for the decode-time ICP block indexer.

This module only draws random inputs; it holds none of the indexer's
arithmetic.  Both the CUDA path and the CPU oracle are fed from it.

Recipe (every workload uses one ``torch.Generator`` seeded with ``seed``, and
draws in the fixed order below):

1. ``seq_lens``: the listed values, or ``randint(lo, hi + 1)`` per request.
2. ``block_table``: request b needs ``ceil(seq_len_b / page_size)`` pages.  A
   random permutation of the page pool is dealt out in request order; unused
   table entries hold -1.  The pool is the sum of the pages needed unless a
   pool size is given (the tiny workload uses a 64-page pool).
3. ``u``: one random unit direction, ``N(0, I) / |N(0, I)|``.
4. planted blocks: every logical B128 block of every request is planted
   independently with probability ``planted`` (5 %, or 1 % for the
   long-context workload).
5. ``index_q``: ``float8_e4m3fn(0.5 * N(0, 1) + 1.5 * u)`` for every
   (token, head) row, shape [B * decode_query_len, 4, 128].
6. ``index_k``: ``float8_e4m3fn(0.5 * N(0, 1))`` for every row of every pool
   page, plus ``1.5 * u`` on the 128 rows of each planted block, shape
   [pool, page_size, 128]; a sharded workload hands rank r the contiguous rows
   ``[r * page_size / ws, (r + 1) * page_size / ws)`` of every page.
7. ``num_valid_pages[t]`` = ``ceil((seq_len - decode_query_len + j + 1) / 128)``,
   the number of B128 blocks holding at least one key visible to the token.

The standalone select plane is ``N(0, 1)`` float32 [T, 4, K] in which, per row,
2 % of the columns copy the value of another random column of the same row;
``num_valid_pages`` is ``randint(1, K + 1)`` per token.

fp8 tensors are returned as ``torch.uint8`` holding the e4m3fn bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

HEADS = 4
DIM = 128


@dataclass(frozen=True)
class DecodeSpec:
    name: str
    batch: int
    page_size: int
    world_size: int
    decode_query_len: int
    max_decode_query_len: int
    init_blocks: int
    local_blocks: int
    planted: float = 0.05
    seq_lens: tuple = ()          # explicit lengths, or
    seq_range: tuple = ()         # (lo, hi) inclusive
    pool_pages: int = 0           # 0: exactly the pages needed
    capacity: int = 0             # receive rows per (slot, source, head); 0 -> T
    description: str = ""

    @property
    def T(self) -> int:
        return self.batch * self.decode_query_len


# The five workloads: shapes, limits and distributions as stated for the
# decode indexer (4 index heads x 128 fp8 dims everywhere).
TINY = DecodeSpec(
    "tiny", batch=2, page_size=128, world_size=1, decode_query_len=1, max_decode_query_len=1,
    init_blocks=1, local_blocks=2, seq_lens=(1000, 2500), pool_pages=64,
    description="tiny decode, unsharded: B=2, seq_lens {1000, 2500}, P128, dql 1, "
                "64-page pool, init 1, local 2")
BATCHED = DecodeSpec(
    "batched", batch=64, page_size=128, world_size=1, decode_query_len=1,
    max_decode_query_len=1, init_blocks=1, local_blocks=4, seq_range=(4096, 32768),
    description="batched decode, unsharded: B=64, seq_len U[4096, 32768], P128, dql 1, "
                "init 1, local 4")
MULTITOKEN = DecodeSpec(
    "multitoken", batch=128, page_size=256, world_size=1, decode_query_len=4,
    max_decode_query_len=8, init_blocks=2, local_blocks=4, seq_range=(8192, 131072),
    description="multi-token decode: B=128, seq_len U[8192, 131072], P256, dql 4 "
                "(max 8), T=512, init 2, local 4")
SHARDED = DecodeSpec(
    "sharded", batch=32, page_size=128, world_size=4, decode_query_len=2,
    max_decode_query_len=2, init_blocks=1, local_blocks=3, seq_range=(65536, 262144),
    capacity=64,
    description="sharded layout on one GPU: world_size 4, P128 (32 K rows per page per "
                "shard), B=32, seq_len U[65536, 262144], dql 2, capacity 64, 3 slots, "
                "init 1, local 3")
LONGCTX = DecodeSpec(
    "longctx", batch=8, page_size=128, world_size=1, decode_query_len=8,
    max_decode_query_len=8, init_blocks=4, local_blocks=8, planted=0.01,
    seq_lens=(1_000_000,) * 8,
    description="long-context stress: B=8, seq_len 1,000,000 (7813 blocks, cols 7816), "
                "P128, dql 8 (T=64), 1 % planted, init 4, local 8")

DECODE_SPECS = {s.name: s for s in (TINY, BATCHED, MULTITOKEN, SHARDED, LONGCTX)}

# Prefill window: every request brings a chunk of decode_query_len new tokens
# (its newest positions), drawn with the same recipe.
PREFILL = DecodeSpec(
    "prefill", batch=4, page_size=128, world_size=1, decode_query_len=2048,
    max_decode_query_len=2048, init_blocks=1, local_blocks=4, seq_range=(4096, 32768),
    description="prefill window: B=4 requests, chunks of 2048 new tokens (T=8192), "
                "seq_len U[4096, 32768] after the chunk, P128, init 1, local 4")

# standalone Top16 select on a [T=256, 4, K=12284] plane
SELECT_T, SELECT_K, SELECT_INIT, SELECT_LOCAL, SELECT_DUP = 256, 12284, 4, 8, 0.02


@dataclass
class DecodeInputs:
    spec: DecodeSpec
    seq_lens: torch.Tensor          # int32 [B]
    block_table: torch.Tensor       # int32 [B, W]
    index_q: torch.Tensor           # uint8 [T, 4, 128]
    index_k: torch.Tensor           # uint8 [pool, page_size, 128] (all rows of every page)
    num_valid_pages: torch.Tensor   # int32 [T]
    planted: torch.Tensor           # bool [B, max B128 blocks]
    u: torch.Tensor                 # float32 [128]
    shards: list = field(default_factory=list)  # uint8 [pool, page_size/ws, 128] per rank

    @property
    def T(self) -> int:
        return int(self.seq_lens.numel()) * self.spec.decode_query_len


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _fp8_bits(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def make_decode_inputs(spec: DecodeSpec, *, seed: int = 0, device="cpu", batch: int = 0,
                       seq_lens=None, make_shards: bool = True,
                       page_chunk: int = 2048) -> DecodeInputs:
    """Draw one decode workload.  ``batch``/``seq_lens`` override the spec (smaller cases)."""
    device = torch.device(device)
    g = _gen(device, seed)
    B = batch or spec.batch
    ps = spec.page_size
    if seq_lens is not None:
        sl = torch.as_tensor(seq_lens, dtype=torch.int64, device=device)
        B = sl.numel()
    elif spec.seq_lens:
        sl = torch.tensor(list(spec.seq_lens)[:B], dtype=torch.int64, device=device)
        B = sl.numel()
    else:
        lo, hi = spec.seq_range
        sl = torch.randint(lo, hi + 1, (B,), generator=g, device=device, dtype=torch.int64)
    pages = (sl + ps - 1) // ps
    needed = int(pages.sum().item())
    pool = max(spec.pool_pages, needed) if spec.pool_pages else needed
    perm = torch.randperm(pool, generator=g, device=device).to(torch.int32)
    width = max(int(pages.max().item()), 1) if B > 0 else 1
    bt = torch.full((B, width), -1, dtype=torch.int32, device=device)
    starts = torch.cumsum(pages, 0) - pages
    cols_idx = torch.arange(width, device=device)
    mask = cols_idx[None, :] < pages[:, None]
    src = (starts[:, None] + cols_idx[None, :]).clamp(max=max(pool - 1, 0))
    bt[mask] = perm[src[mask]]

    u = torch.randn(DIM, generator=g, device=device, dtype=torch.float32)
    u = u / u.norm()

    blocks = (sl + 127) // 128
    maxblocks = max(int(blocks.max().item()), 1) if B > 0 else 1
    planted = torch.rand((B, maxblocks), generator=g, device=device) < spec.planted
    planted &= torch.arange(maxblocks, device=device)[None, :] < blocks[:, None]

    T = B * spec.decode_query_len
    qf = 0.5 * torch.randn((T, HEADS, DIM), generator=g, device=device) + 1.5 * u
    index_q = _fp8_bits(qf)
    del qf

    # planted flag per (pool page, B128 sub-block of the page)
    sub = ps // 128
    page_planted = torch.zeros((pool, sub), dtype=torch.bool, device=device)
    bidx = torch.arange(maxblocks, device=device)
    blk_page_slot = (bidx // sub)[None, :].expand(B, maxblocks)
    blk_sub = (bidx % sub)[None, :].expand(B, maxblocks)
    sel = planted
    if sel.any():
        pg = torch.gather(bt.to(torch.int64), 1,
                          blk_page_slot.clamp(max=width - 1).contiguous())[sel]
        page_planted[pg, blk_sub[sel]] = True

    index_k = torch.empty((pool, ps, DIM), dtype=torch.uint8, device=device)
    for p0 in range(0, pool, page_chunk):
        p1 = min(pool, p0 + page_chunk)
        kf = 0.5 * torch.randn((p1 - p0, ps, DIM), generator=g, device=device)
        add = page_planted[p0:p1].repeat_interleave(128, dim=1)  # [n, ps]
        kf += add[:, :, None].to(kf.dtype) * (1.5 * u)
        index_k[p0:p1] = _fp8_bits(kf)
        del kf

    j = torch.arange(spec.decode_query_len, device=device)
    pos = (sl[:, None] - spec.decode_query_len + j[None, :]).reshape(-1)
    nvp = torch.div(pos + 1 + 127, 128, rounding_mode="floor").clamp(min=0).to(torch.int32)

    inp = DecodeInputs(spec=spec, seq_lens=sl.to(torch.int32), block_table=bt, index_q=index_q,
                       index_k=index_k, num_valid_pages=nvp, planted=planted, u=u)
    if make_shards and spec.world_size > 1:
        rp = ps // spec.world_size
        inp.shards = [index_k[:, r * rp:(r + 1) * rp].contiguous()
                      for r in range(spec.world_size)]
    return inp


def make_select_plane(*, T: int = SELECT_T, K: int = SELECT_K, dup: float = SELECT_DUP,
                      seed: int = 0, device="cpu"):
    """N(0,1) plane [T, 4, K] with per-row duplicated columns, and num_valid_pages [T]."""
    device = torch.device(device)
    g = _gen(device, seed)
    plane = torch.randn((T, HEADS, K), generator=g, device=device, dtype=torch.float32)
    ndup = int(round(dup * K))
    if ndup > 0:
        rows = T * HEADS
        flat = plane.view(rows, K)
        dst = torch.rand((rows, K), generator=g, device=device).argsort(dim=1)[:, :ndup]
        srcc = torch.randint(0, K, (rows, ndup), generator=g, device=device)
        vals = torch.gather(flat, 1, srcc)
        flat.scatter_(1, dst, vals)
    nvp = torch.randint(1, K + 1, (T,), generator=g, device=device, dtype=torch.int32)
    return plane, nvp


def columns_for(spec: DecodeSpec, max_seq_len: int) -> int:
    """Plane width for a workload: one column per unit (B128 block, or local
    page for P256 sharded), padded to the next multiple of 4."""
    unit = 128 if (spec.page_size == 128 or spec.world_size == 1) else spec.page_size
    n = (max_seq_len + unit - 1) // unit
    return max(4, (n + 3) // 4 * 4)
