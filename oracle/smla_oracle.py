"""Plain float64 definition of sparse MLA decode under decode-context-parallel.

TEST INFRASTRUCTURE: imported only by tests/, __graft_entry__.smoke() and the
CPU-baseline legs of bench.py.  It shares no code with the CUDA path.

Sources (page title, then section):
  [P1] "[eldritch] attention: support DCP in SM120 FlashInfer sparse MLA"
  [P2] "[Bugfix][Attention] Stabilize sparse-MLA DCP for GLM PCP evals"
  [P3] "FlashMLA sparse fp8 path + DCP + MTP" (vLLM PR #46514 summary)

Every function here is the plain definition of the result the decode path
reaches, written for a reader to check by eye: no blocking, no fusion, no
reordering beyond what the definition states.  Library primitives used as
steps: numpy matmul, exp, log, max.

Pins (tests/test_oracle.py), all independent of this file's arithmetic:
  e4m3_to_f64 ........ all 256 codes against torch.float8_e4m3fn, spec values
  bf16_bits_to_f64 ... every bit pattern class against torch.bfloat16
  parse_rows ......... rows packed by struct/torch encoders round-trip
  dcp_filter_convert_index ... a KV-append simulation (per-shard running
                       counters and block allocation) for interleave sizes
                       1..4, partition/inverse invariants, D=1 plain paged
                       mapping for any interleave size
  dcp_local_seq_len .. closed forms (whole rounds of I*D positions plus the
                       partial round) for interleave sizes 1..4
  topk_select ........ torch.topk on distinct scores, numpy argmax at K=1,
                       the all-equal closed form, short rows
  dcp_topk_merge ..... per-rank local top-k then merge equals the unsharded
                       selection, with and without ties
  dense_mla_decode ... paged, sharded over D ranks and merged, against torch
                       float64 SDPA with a causal mask over the logical token
                       sequence; spec-decode tokens equal single-token requests
  flatten_lse_bhs .... torch permute + reshape
  sparse_mla_decode .. torch float64 scaled_dot_product_attention + logsumexp
                       on dense cases, q=0 closed form, single-slot closed
                       form, order invariance, the pages' empty-row case
  lse_merge .......... sharded-then-merged equals unsharded, identity
                       element, all-empty rows
"""
from __future__ import annotations

import math

import numpy as np

NOPE_DIM = 512
ROPE_DIM = 64
GROUP = 128
ROW_BYTES = 656


# --------------------------------------------------------------------------
# fp8 e4m3 ("fn" variant of the OCP 8-bit floating point format): 1 sign
# bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, and the
# pattern S.1111.111 is NaN.  The fp8_ds_mla cache stores its 512 latent
# values this way [P1 Scope / Limitations; P3 features and motivation].
# --------------------------------------------------------------------------
def _e4m3_value(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:  # subnormal: m/8 * 2^(1-7)
        return sign * (man / 8.0) * 2.0 ** (-6)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode uint8 e4m3 codes to float64 (exact)."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns (uint16) to float64 (exact): a bf16 value
    is the top half of the fp32 value with the same bits."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):  # NaN patterns widen to NaN
        return u32.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Row parse.  The pages say only that a packed fp8_ds_mla row is 656 bytes
# for 576 logical dims [P3 related PRs, "576 vs 656 layout"].  Reading taken:
# the parts in the order the problem statement lists them --
#   bytes [0, 512)   512 e4m3 codes (latent dims 0..511)
#   bytes [512, 528) 4 little-endian fp32 scales; scale g covers 128g..128g+127
#   bytes [528, 656) 64 little-endian bf16 rope values (key dims 512..575)
# and a latent value is code * scale (multiplicative scale).
# --------------------------------------------------------------------------
def parse_rows(rows: np.ndarray):
    """uint8 [n, 656] -> (nope float64 [n, 512], rope float64 [n, 64])."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    assert rows.ndim == 2 and rows.shape[1] == ROW_BYTES
    codes = rows[:, :NOPE_DIM]
    scales = np.ascontiguousarray(rows[:, 512:528]).view("<f4").astype(np.float64)
    rope_bits = np.ascontiguousarray(rows[:, 528:656]).view("<u2")
    nope = e4m3_to_f64(codes) * np.repeat(scales, GROUP, axis=1)
    rope = bf16_bits_to_f64(rope_bits)
    return nope, rope


# --------------------------------------------------------------------------
# DCP filter + convert [P3 implementation breakdown step 2 and the
# _forward_fp8_kv_mixed_batch snippet; P1 Summary "convert global sparse
# top-k token ids to this DCP rank's local physical KV slots"].
# Interleave size I (the snippet passes cp_kv_cache_interleave_size; the
# pages validate only I = 1 [P3 implementation breakdown step 4]): groups of
# I consecutive positions go to the ranks in turn, so position t lives on
# rank (t div I) mod D at rank-local position (t div (I*D))*I + t mod I --
# for I = 1, rank t mod D at position t div D.  The rank-local position then
# goes through that rank's paged block table.  Entries that are negative or
# owned by another rank become -1 *in place* (compact_valid_to_front=False).
# With D=1 this is the plain request-index -> global-slot conversion of the
# non-DCP branch, whatever I is.
# --------------------------------------------------------------------------
def dcp_filter_convert_index(req_id, block_table, topk, D, rank, block_size, interleave=1):
    """Returns (local_slots int32 [T, K], valid_count int32 [T])."""
    topk = np.asarray(topk, dtype=np.int64)
    req_id = np.asarray(req_id, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    I = int(interleave)
    assert I >= 1
    T, K = topk.shape
    out = np.full((T, K), -1, dtype=np.int64)
    for i in range(T):
        r = req_id[i]
        t = topk[i]
        mine = (t >= 0) & ((t // I) % D == rank)
        tm = t[mine]
        lp = (tm // (I * D)) * I + tm % I  # rank-local position
        col = lp // block_size
        assert np.all(col < bt.shape[1]), "top-k id beyond the block table"
        phys = bt[r, col]
        assert np.all(phys >= 0), "top-k id in an unallocated block"
        out[i, mine] = phys * block_size + lp % block_size
    valid_count = (out >= 0).sum(axis=1)
    return out.astype(np.int32), valid_count.astype(np.int32)


def dcp_local_seq_len(ctx: int, D: int, rank: int, interleave: int = 1) -> int:
    """Number of a request's ctx positions that rank holds [P2 "DCP decode
    rank scalar", get_dcp_local_seq_lens], groups of `interleave` positions
    going to the ranks in turn."""
    I = int(interleave)
    return sum(1 for t in range(int(ctx)) if (t // I) % D == rank)


# --------------------------------------------------------------------------
# Global top-k of indexer scores, the step that produces this path's input
# [P1 Summary "global sparse top-k token ids"; P3 related PRs, the DCP
# sparse-indexer mechanism "global top-k merge, DCP index filtering"].  The
# pages do not spell the selection out.  Reading taken: a row keeps the K
# largest scores among its candidate positions 0..n-1 (n = the request's
# context, or the query's own position + 1 in spec decode), ranked by score
# descending and, among equal scores, by position ascending; with fewer than
# K candidates it keeps all of them and pads with -1.  The output lists the
# kept positions in that rank order, padding last.
# --------------------------------------------------------------------------
def topk_select(scores, n_cand, K):
    """scores float [T, L]; n_cand int [T] (positions >= n_cand[i] are not
    candidates); returns int32 [T, K] positions, -1 padded."""
    scores = np.asarray(scores, dtype=np.float64)
    T = scores.shape[0]
    out = np.full((T, K), -1, dtype=np.int64)
    for i in range(T):
        n = int(n_cand[i])
        pos = np.arange(n)
        # lexsort: the last key is the primary one
        order = np.lexsort((pos, -scores[i, :n]))
        keep = order[:K]
        out[i, :len(keep)] = pos[keep]
    return out.astype(np.int32)


# Under DCP each rank scores only the positions it holds and keeps its own
# top-k of them, as global ids; the global top-k is then the top-k of the
# union of the ranks' candidates, by the same rank order.
def dcp_topk_merge(cand_ids, cand_scores, K):
    """cand_ids: sequence over ranks of int [T, K_d] global positions (-1 =
    no candidate); cand_scores: the matching scores.  Returns int32 [T, K]."""
    ids = np.concatenate([np.asarray(c, dtype=np.int64) for c in cand_ids], axis=1)
    sc = np.concatenate([np.asarray(c, dtype=np.float64) for c in cand_scores], axis=1)
    T = ids.shape[0]
    out = np.full((T, K), -1, dtype=np.int64)
    for i in range(T):
        live = ids[i] >= 0
        pos, val = ids[i, live], sc[i, live]
        order = np.lexsort((pos, -val))
        keep = order[:K]
        out[i, :len(keep)] = pos[keep]
    return out.astype(np.int32)


# --------------------------------------------------------------------------
# Sparse MLA decode with LSE return [P1 Why; P3 implementation breakdown
# steps 1 and 3].  For query row i and head h, over the valid slots j of the
# row (negative entries skipped, each occurrence counted):
#     k_j = (nope_j || rope_j)                    576 dims
#     s_j = sm_scale * <q[i,h,:], k_j>
#     lse = log(sum_j exp(s_j))                   natural log, sm_scale included
#     out = sum_j exp(s_j - lse) * nope_j         values are the 512-d latent
# A row with no valid slot is the merge identity: out = 0, lse = -inf.
# --------------------------------------------------------------------------
def sparse_mla_decode_rows(q_row: np.ndarray, rows: np.ndarray, sm_scale: float):
    """One query row.  q_row float64 [H, 576]; rows uint8 [n, 656].
    Returns (out float64 [H, 512], lse float64 [H])."""
    H = q_row.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((H, NOPE_DIM)), np.full(H, -np.inf)
    nope, rope = parse_rows(rows)
    k = np.concatenate([nope, rope], axis=1)  # [n, 576]
    s = sm_scale * (q_row @ k.T)  # [H, n]
    m = s.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    p = np.exp(s - lse[:, None])
    return p @ nope, lse


def sparse_mla_decode(q_bits: np.ndarray, pool: np.ndarray,
                      local_slots: np.ndarray, sm_scale: float):
    """q_bits uint16 [T, H, 576] (bf16 bit patterns); pool uint8
    [num_slots, 656]; local_slots int [T, K].  Returns (out float64
    [T, H, 512], lse float64 [T, H]); LSE rows are tokens in input row order
    (b*S + s for spec decode) [P3 dense FlashMLA LSE flattening]."""
    q = bf16_bits_to_f64(q_bits)
    T, H, _ = q.shape
    out = np.zeros((T, H, NOPE_DIM))
    lse = np.full((T, H), -np.inf)
    slots = np.asarray(local_slots, dtype=np.int64)
    for i in range(T):
        valid = slots[i][slots[i] >= 0]
        assert np.all(valid < pool.shape[0]), "slot beyond the pool"
        out[i], lse[i] = sparse_mla_decode_rows(q[i], pool[valid], sm_scale)
    return out, lse


# --------------------------------------------------------------------------
# Dense MLA decode with LSE return [P3 key snippets, the dense FlashMLA
# decode path (vllm/v1/attention/backends/mla/flashmla.py): under DCP it
# returns the LSE, flattened from [batch, heads, seq_len] to
# [tokens, heads]].  Request b has S query tokens at positions
# ctx_b - S .. ctx_b - 1; token s attends every position up to and including
# its own.  Under DCP, rank d attends only the positions it holds, so its
# (out, lse) per token is a partial that the LSE merge combines.  Rows come
# out in token order b*S + s.
# --------------------------------------------------------------------------
def dense_mla_decode(q_bits, pool, block_table, ctx, S, D, rank, block_size, sm_scale,
                     interleave=1):
    """q_bits uint16 [B*S, H, 576] (row b*S + s); pool uint8 [num_slots, 656]
    and block_table int32 [B, W] of rank `rank`; ctx int [B].  Returns
    (out float64 [B*S, H, 512], lse float64 [B*S, H])."""
    ctx = np.asarray(ctx, dtype=np.int64)
    B = ctx.shape[0]
    T = B * S
    H = q_bits.shape[1]
    out = np.zeros((T, H, NOPE_DIM))
    lse = np.full((T, H), -np.inf)
    for b in range(B):
        for s_ in range(S):
            i = b * S + s_
            p = int(ctx[b]) - S + s_  # this token's position
            positions = np.arange(p + 1, dtype=np.int32)[None]
            slots, _ = dcp_filter_convert_index(np.array([b]), block_table, positions, D, rank,
                                                block_size, interleave)
            mine = slots[0][slots[0] >= 0]
            q = bf16_bits_to_f64(q_bits[i])
            out[i], lse[i] = sparse_mla_decode_rows(q, np.asarray(pool)[mine], sm_scale)
    return out, lse


def flatten_lse_bhs(lse_bhs):
    """[batch, heads, seq_len] -> [batch * seq_len, heads], row b*S + s."""
    lse_bhs = np.asarray(lse_bhs)
    B, H, S = lse_bhs.shape
    flat = np.empty((B * S, H), dtype=lse_bhs.dtype)
    for b in range(B):
        for s_ in range(S):
            flat[b * S + s_] = lse_bhs[b, :, s_]
    return flat


# --------------------------------------------------------------------------
# LSE-weighted merge of D partial results [P1 Why; P3 executive summary 1
# and implementation breakdown step 3].  With M = max_d lse_d:
#     lse = M + log(sum_d exp(lse_d - M)),  out = sum_d exp(lse_d - lse) out_d
# A (0, -inf) partial contributes nothing; if every partial is -inf the
# result is (0, -inf) with no NaN.
# --------------------------------------------------------------------------
def lse_merge(outs, lses):
    """outs: sequence of [T, H, 512]; lses: sequence of [T, H].
    Returns (out float64 [T, H, 512], lse float64 [T, H])."""
    L = np.stack([np.asarray(x, dtype=np.float64) for x in lses])  # [D,T,H]
    O = np.stack([np.asarray(x, dtype=np.float64) for x in outs])  # [D,T,H,V]
    M = L.max(axis=0)
    empty = np.isneginf(M)
    M_safe = np.where(empty, 0.0, M)
    w = np.exp(L - M_safe[None])  # exp(-inf) = 0
    total = w.sum(axis=0)
    lse = np.where(empty, -np.inf, M_safe + np.log(np.where(empty, 1.0, total)))
    weight = np.where(empty[None], 0.0, w / np.where(empty, 1.0, total)[None])
    out = (weight[..., None] * O).sum(axis=0)
    return out, lse
