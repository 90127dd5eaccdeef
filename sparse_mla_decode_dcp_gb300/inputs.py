"""Seeded synthetic inputs for sparse MLA decode under decode-context-parallel.

This module only *creates* inputs. It holds none of the arithmetic the decode
path computes: it never maps a global token id to a slot, never dequantises a
cache row and never evaluates attention. Both the CUDA path and the float64
oracle consume what it builds.

What it builds, per workload:

* ``ctx[R]`` context lengths (the query tokens' own KV is already cached, as in
  an MTP/spec-decode step where the context counts every query token).
* ``topk[T, K]`` int32 *global* token positions per query row, -1 padded, in
  random order (the sparse indexer's contract: "FlashMLA sparse fp8 path + DCP
  + MTP", implementation breakdown step 2; global top-k merge from PR #46076).
* ``req_id[T]`` int32, row ``b*S + s`` belongs to request ``b`` (spec-decode
  row order, dense FlashMLA LSE flattening in the same page).
* For each of the D simulated shards: a paged pool of 656-byte ``fp8_ds_mla``
  rows and a block table ``[R, W_d]`` (-1 where unused).  A request with
  ``n`` tokens on a shard owns ``ceil(n / block_size)`` physical blocks drawn
  from a random permutation of the shard's blocks, plus ~10% spare blocks that
  nobody owns.  Which tokens a shard holds comes from the interleave rule
  (runs of I consecutive positions go to the shards in turn; I = 1: position
  p is held by shard p mod D); this module uses that rule only to count how
  many rows each request owns on each shard, the bookkeeping a KV block
  allocator does.
* ``q[T, H, 576]`` bf16 ~ N(0, 1).

Row byte layout (the plainest reading of "576 vs 656 layout": the parts in the
order 512 e4m3 latent values, 4 fp32 scales, 64 bf16 rope values):

    [0, 512)    e4m3 codes of latent dims 0..511
    [512, 528)  4 little-endian fp32 scales, scale g covers dims 128g..128g+127
    [528, 656)  64 little-endian bf16 rope values (key dims 512..575)

A live row is filled with nope ~ N(0,1) quantised per 128-dim group with
``scale = absmax / 448`` (divide, clamp to +-448, round-to-nearest-even to
e4m3 through torch's float8 cast) and rope ~ N(0,1) rounded to bf16.  Every
row no request owns (block tails, spare blocks) is poisoned with 0xFF bytes:
e4m3 NaN codes, NaN scales and NaN rope, so a stray read shows up as NaN.

Random draws: one ``numpy.random.default_rng(seed)`` drives all structure
(contexts, top-k, -1 placement, block permutations) in the order written in
``make_workload``; cache values and q come from a ``torch.Generator`` on the
target device seeded with ``seed``.  Consumers read the produced bytes, so the
two sides never need to reproduce each other's draws.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

ROW_BYTES = 656
NOPE_DIM = 512
ROPE_DIM = 64
QK_DIM = NOPE_DIM + ROPE_DIM  # 576
V_DIM = NOPE_DIM  # 512
GROUP = 128
N_GROUPS = NOPE_DIM // GROUP  # 4
CODES_END = NOPE_DIM  # 512
SCALES_END = CODES_END + 4 * N_GROUPS  # 528
E4M3_MAX = 448.0
POISON_BYTE = 0xFF


@dataclass
class WorkloadSpec:
    """Shape and distribution recipe of one synthetic decode batch."""

    name: str
    num_reqs: int
    tokens_per_req: int  # S, query tokens per request (2 = MTP step)
    heads: int  # H, gathered query heads
    topk: int  # K
    dcp: int  # D
    block_size: int
    ctx_kind: str  # "fixed" | "loguniform" | "uniform"
    ctx_lo: int = 0
    ctx_hi: int = 0
    ctx_fixed: Sequence[int] = ()
    tiny_ctx_reqs: int = 0  # requests forced to a context of 1..3 tokens
    neg_frac: float = 0.0  # fraction of K slots forced to -1 after padding
    spare_frac: float = 0.10
    sm_scale: float = 1.0 / math.sqrt(192.0)
    interleave: int = 1  # I: runs of I consecutive positions per shard

    @property
    def num_tokens(self) -> int:
        return self.num_reqs * self.tokens_per_req


# The five workloads of the sparse MLA DCP decode study, by what they are.
WORKLOADS = {
    "tiny": WorkloadSpec(
        name="tiny", num_reqs=2, tokens_per_req=1, heads=16, topk=64, dcp=2,
        block_size=16, ctx_kind="fixed", ctx_fixed=(200, 37), neg_frac=0.10),
    "single_shard": WorkloadSpec(
        name="single_shard", num_reqs=32, tokens_per_req=1, heads=64,
        topk=2048, dcp=1, block_size=64, ctx_kind="fixed",
        ctx_fixed=(4096,) * 32),
    "dcp4_long": WorkloadSpec(
        name="dcp4_long", num_reqs=64, tokens_per_req=1, heads=128, topk=2048,
        dcp=4, block_size=64, ctx_kind="loguniform", ctx_lo=4096,
        ctx_hi=65536, tiny_ctx_reqs=4),
    "mtp2": WorkloadSpec(
        name="mtp2", num_reqs=64, tokens_per_req=2, heads=128, topk=2048,
        dcp=2, block_size=64, ctx_kind="uniform", ctx_lo=8192, ctx_hi=32768),
    "serving_dcp8": WorkloadSpec(
        name="serving_dcp8", num_reqs=128, tokens_per_req=1, heads=128,
        topk=2048, dcp=8, block_size=64, ctx_kind="loguniform", ctx_lo=1024,
        ctx_hi=131072, neg_frac=0.05),
}
WORKLOAD_ORDER = ["tiny", "single_shard", "dcp4_long", "mtp2", "serving_dcp8"]


@dataclass
class Shard:
    """One simulated DCP rank: its paged pool and its block table."""

    pool: torch.Tensor  # uint8 [num_slots, 656]
    block_table: np.ndarray  # int32 [R, row_stride], -1 where unused
    width: int  # number of meaningful columns of block_table
    live_rows: int  # rows holding real cache entries


@dataclass
class Workload:
    spec: WorkloadSpec
    seed: int
    ctx: np.ndarray  # int64 [R]
    req_id: np.ndarray  # int32 [T]
    topk: np.ndarray  # int32 [T, K]
    q: torch.Tensor  # bf16 [T, H, 576]
    shards: List[Shard] = field(default_factory=list)

    @property
    def T(self) -> int:
        return int(self.topk.shape[0])

    @property
    def H(self) -> int:
        return self.spec.heads

    @property
    def K(self) -> int:
        return int(self.topk.shape[1])

    @property
    def D(self) -> int:
        return self.spec.dcp


def draw_contexts(spec: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    """Context lengths per request (draw 1 of the structure stream)."""
    R = spec.num_reqs
    if spec.ctx_kind == "fixed":
        ctx = np.asarray(spec.ctx_fixed, dtype=np.int64)
        assert ctx.shape == (R,)
    elif spec.ctx_kind == "loguniform":
        u = rng.uniform(math.log(spec.ctx_lo), math.log(spec.ctx_hi), size=R)
        ctx = np.clip(np.floor(np.exp(u)), spec.ctx_lo, spec.ctx_hi).astype(np.int64)
    elif spec.ctx_kind == "uniform":
        ctx = rng.integers(spec.ctx_lo, spec.ctx_hi + 1, size=R).astype(np.int64)
    else:
        raise ValueError(spec.ctx_kind)
    if spec.tiny_ctx_reqs:
        which = rng.choice(R, size=spec.tiny_ctx_reqs, replace=False)
        ctx[which] = rng.integers(1, 4, size=spec.tiny_ctx_reqs)
    ctx = np.maximum(ctx, spec.tokens_per_req)
    return ctx


def draw_topk_row(rng: np.random.Generator, n_cand: int, K: int,
                  neg_frac: float) -> np.ndarray:
    """K global positions drawn from [0, n_cand): min(K, n_cand) distinct
    uniform positions, -1 padding up to K, random order, then floor(neg_frac*K)
    uniformly chosen entries (without replacement) overwritten with -1."""
    n_valid = min(K, n_cand)
    ids = rng.choice(n_cand, size=n_valid, replace=False).astype(np.int64)
    row = np.full(K, -1, dtype=np.int64)
    row[:n_valid] = ids
    row = rng.permutation(row)
    n_neg = int(math.floor(neg_frac * K))
    if n_neg:
        row[rng.choice(K, size=n_neg, replace=False)] = -1
    return row.astype(np.int32)


def rows_on_shard(ctx: int, D: int, d: int, interleave: int = 1) -> int:
    """How many of a request's ctx cached positions shard d holds when runs
    of `interleave` consecutive positions go to the shards in turn
    (allocation bookkeeping only): whole rounds of I*D positions give I each,
    then the last partial round."""
    I = int(interleave)
    full, rem = divmod(int(ctx), I * D)
    return full * I + min(max(rem - d * I, 0), I)


def random_rows(n: int, gen: torch.Generator, device) -> torch.Tensor:
    """n live fp8_ds_mla rows (uint8 [n, 656]) with the documented recipe."""
    out = torch.empty((n, ROW_BYTES), dtype=torch.uint8, device=device)
    chunk = 1 << 16
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        nope = torch.randn((m, N_GROUPS, GROUP), generator=gen, device=device,
                           dtype=torch.float32)
        rope = torch.randn((m, ROPE_DIM), generator=gen, device=device,
                           dtype=torch.float32)
        absmax = nope.abs().amax(dim=2, keepdim=True)
        scale = absmax / E4M3_MAX  # fp32
        safe = torch.where(scale > 0, scale, torch.ones_like(scale))
        codes = (nope / safe).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
        codes = torch.where(scale > 0, codes.view(torch.uint8),
                            torch.zeros_like(codes.view(torch.uint8)))
        blk = out[s:s + m]
        blk[:, :CODES_END] = codes.reshape(m, NOPE_DIM)
        blk[:, CODES_END:SCALES_END] = (
            scale.reshape(m, N_GROUPS).contiguous().view(torch.uint8))
        blk[:, SCALES_END:] = rope.to(torch.bfloat16).contiguous().view(torch.uint8)
    return out


def build_shard(ctx: np.ndarray, D: int, d: int, block_size: int,
                spare_frac: float, rng: np.random.Generator,
                gen: torch.Generator, device, row_stride_pad: int = 0,
                interleave: int = 1) -> Shard:
    R = len(ctx)
    n = np.array([rows_on_shard(c, D, d, interleave) for c in ctx], dtype=np.int64)
    nblk = (n + block_size - 1) // block_size
    used = int(nblk.sum())
    spare = max(1, int(math.ceil(spare_frac * used)))
    total = used + spare
    perm = rng.permutation(total).astype(np.int64)
    width = max(1, int(nblk.max()) if R else 1)
    stride = width + row_stride_pad
    bt = np.full((R, stride), -1, dtype=np.int32)
    live_per_block = np.zeros(total, dtype=np.int64)
    cursor = 0
    for r in range(R):
        ids = perm[cursor:cursor + nblk[r]]
        cursor += nblk[r]
        bt[r, :nblk[r]] = ids
        if nblk[r]:
            live_per_block[ids[:-1]] = block_size
            live_per_block[ids[-1]] = n[r] - (nblk[r] - 1) * block_size
    pool = torch.full((total * block_size, ROW_BYTES), POISON_BYTE,
                      dtype=torch.uint8, device=device)
    live = (torch.arange(block_size).unsqueeze(0)
            < torch.from_numpy(live_per_block).unsqueeze(1)).reshape(-1)
    live = live.to(device)
    n_live = int(n.sum())
    if n_live:
        pool[live] = random_rows(n_live, gen, device)
    return Shard(pool=pool, block_table=bt, width=width, live_rows=n_live)


def draw_topk(spec: WorkloadSpec, ctx: np.ndarray, rng: np.random.Generator) -> np.ndarray:
    """The top-k rows of every query token, in row order (b * S + s): token s
    of request b sits at position ctx[b] - S + s and its ids are <= it."""
    S = spec.tokens_per_req
    topk = np.empty((spec.num_tokens, spec.topk), dtype=np.int32)
    for b in range(spec.num_reqs):
        for s in range(S):
            pos = int(ctx[b]) - S + s  # query position; top-k ids <= pos
            topk[b * S + s] = draw_topk_row(rng, pos + 1, spec.topk, spec.neg_frac)
    return topk


def make_workload(spec: WorkloadSpec | str, seed: int = 0, device="cpu",
                  row_stride_pad: int = 0, ctx_override: Optional[Sequence[int]] = None
                  ) -> Workload:
    """Build one workload.  Structure draws, in order: contexts, then top-k
    rows in row order, then per shard d = 0..D-1 its block permutation.
    Value draws (torch generator on ``device``): per shard its live rows, then q.
    """
    if isinstance(spec, str):
        spec = WORKLOADS[spec]
    rng = np.random.default_rng(seed)
    if ctx_override is not None:
        ctx = np.asarray(ctx_override, dtype=np.int64)
        assert ctx.shape == (spec.num_reqs,)
    else:
        ctx = draw_contexts(spec, rng)
    S = spec.tokens_per_req
    T = spec.num_tokens
    req_id = np.repeat(np.arange(spec.num_reqs, dtype=np.int32), S)
    topk = draw_topk(spec, ctx, rng)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shards = [build_shard(ctx, spec.dcp, d, spec.block_size, spec.spare_frac,
                          rng, gen, device, row_stride_pad, spec.interleave)
              for d in range(spec.dcp)]
    q = torch.randn((T, spec.heads, QK_DIM), generator=gen, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    return Workload(spec=spec, seed=seed, ctx=ctx, req_id=req_id, topk=topk,
                    q=q, shards=shards)
