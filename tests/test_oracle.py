"""Pins of the float64 oracle against facts independent of its own code.

Every check here compares the oracle with something it does not share code
with: torch's float8/bfloat16 casts, torch's float64 scaled-dot-product
attention and logsumexp, hand-worked fixtures under tests/golden/, a
simulation of a paged KV cache filled one token at a time, closed forms and
invariants the pages state.  Runs on CPU.
"""
import json
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_decode_dcp_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SM_SCALE = 1.0 / math.sqrt(192.0)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- fp8, bf16
def test_e4m3_table_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    nan_ref, nan_got = np.isnan(ref), np.isnan(got)
    assert np.array_equal(nan_ref, nan_got)
    assert nan_got.sum() == 2  # 0x7F and 0xFF only
    assert np.array_equal(ref[~nan_ref], got[~nan_got])
    # signed zeros decode with their sign
    assert np.array_equal(np.signbit(ref[~nan_ref]), np.signbit(got[~nan_got]))


def test_e4m3_spec_values():
    g = _golden("e4m3_spec_values.json")
    for code_hex, val in g["values"].items():
        got = oracle.e4m3_to_f64(np.array([int(code_hex, 16)], dtype=np.uint8))[0]
        if val == "nan":
            assert math.isnan(got), code_hex
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), code_hex


def test_bf16_widen_matches_torch():
    rng = np.random.default_rng(1)
    bits = np.concatenate([
        rng.integers(0, 1 << 16, size=20000, dtype=np.uint64).astype(np.uint16),
        np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x3F80,
                  0xBF80, 0x7F7F, 0xFF7F, 0x7F80, 0xFF80], dtype=np.uint16)])
    ref = (torch.from_numpy(bits.astype(np.int32)).to(torch.int16)
           .view(torch.bfloat16).to(torch.float64).numpy())
    got = oracle.bf16_bits_to_f64(bits)
    same = (ref == got) | (np.isnan(ref) & np.isnan(got))
    assert same.all()


# ----------------------------------------------------------------- row parse
def _pack_row(codes_u8, scales_f32, rope_bf16_bits):
    """Pack one row with struct (independent of the oracle's parser)."""
    b = bytes(codes_u8.tolist())
    b += struct.pack("<4f", *[float(s) for s in scales_f32])
    b += struct.pack("<64H", *[int(x) for x in rope_bf16_bits])
    assert len(b) == 656
    return np.frombuffer(b, dtype=np.uint8)


def test_parse_rows_roundtrip_known_values():
    rng = np.random.default_rng(2)
    vals = torch.from_numpy(rng.uniform(-448, 448, size=512)).to(torch.float8_e4m3fn)
    codes = vals.view(torch.uint8).numpy()
    scales = np.array([0.5, 3.0e-3, 7.25, 1.0], dtype=np.float32)
    rope = torch.from_numpy(rng.normal(size=64)).to(torch.bfloat16)
    rope_bits = rope.view(torch.int16).numpy().astype(np.uint16)
    row = _pack_row(codes, scales, rope_bits)
    nope, rope_got = oracle.parse_rows(row[None])
    expect_nope = vals.to(torch.float64).numpy() * np.repeat(
        scales.astype(np.float64), 128)
    assert np.array_equal(nope[0], expect_nope)
    assert np.array_equal(rope_got[0], rope.to(torch.float64).numpy())


def test_parse_rows_generator_rows_dequantise_close_to_source():
    """Rows made by the generator decode to within e4m3 precision of N(0,1)
    samples: |nope| <= absmax of its group, codes reach +-448 in each group."""
    gen = torch.Generator().manual_seed(3)
    rows = inputs.random_rows(64, gen, "cpu").numpy()
    nope, rope = oracle.parse_rows(rows)
    scales = rows[:, 512:528].copy().view("<f4").astype(np.float64)
    for g in range(4):
        grp = nope[:, 128 * g:128 * (g + 1)]
        # the group's largest magnitude is exactly 448 * scale (absmax / 448 scale)
        assert np.allclose(np.abs(grp).max(axis=1), 448.0 * scales[:, g], rtol=0, atol=0)
    assert np.all(np.isfinite(rope)) and 0.5 < rope.std() < 2.0


# ---------------------------------------------------------- filter + convert
def test_index_worked_examples():
    g = _golden("index_worked_example.json")
    for case in g["cases"]:
        slots, count = oracle.dcp_filter_convert_index(
            np.array(case["req_id"]), np.array(case["block_table"]),
            np.array(case["topk"]), case["D"], case["rank"], case["block_size"])
        assert slots.tolist() == case["local_slots"], case["note"]
        assert count.tolist() == case["valid_count"], case["note"]


def _simulate_paged_cache(ctx, D, bs, rng, interleave=1):
    """Fill a D-rank paged KV cache one token at a time, the way a cache
    manager appends: runs of `interleave` consecutive tokens go to the ranks
    in turn, each rank keeps a running row counter per request and takes a
    fresh random free block when the current one is full.  Returns per-rank
    block tables and where[(r, t)] = (rank, slot)."""
    R = len(ctx)
    tables = [[[] for _ in range(R)] for _ in range(D)]
    free = [list(rng.permutation(4 * sum(ctx) // bs + 8 * R + 8)) for _ in range(D)]
    counters = np.zeros((D, R), dtype=np.int64)
    where = {}
    for r in range(R):
        d, run = 0, 0  # the rank taking tokens now, and how many it has taken in a row
        for t in range(ctx[r]):
            if run == interleave:
                d, run = (d + 1) % D, 0
            run += 1
            c = counters[d, r]
            if c % bs == 0:
                tables[d][r].append(int(free[d].pop()))
            where[(r, t)] = (d, tables[d][r][-1] * bs + c % bs)
            counters[d, r] += 1
    bts = []
    for d in range(D):
        W = max(1, max(len(x) for x in tables[d]))
        bt = np.full((R, W + 1), -1, dtype=np.int32)
        for r in range(R):
            bt[r, :len(tables[d][r])] = tables[d][r]
        bts.append(bt)
    return bts, where, counters


@pytest.mark.parametrize("D,bs,ctx,interleave", [
    (1, 4, [13, 5], 1), (2, 4, [13, 1, 9], 1), (3, 2, [7, 2, 11], 1),
    (4, 16, [200, 3, 1, 64], 1), (8, 4, [50, 7], 1),
    (1, 4, [13, 5], 3), (2, 4, [13, 1, 9], 2), (3, 2, [7, 2, 11], 4),
    (4, 16, [200, 3, 1, 64], 2), (4, 4, [77, 30], 3), (8, 4, [50, 7], 4)])
def test_index_matches_append_simulation(D, bs, ctx, interleave):
    rng = np.random.default_rng(D * 100 + bs + 7 * interleave)
    bts, where, counters = _simulate_paged_cache(ctx, D, bs, rng, interleave)
    R = len(ctx)
    rows, req = [], []
    for r in range(R):
        for _ in range(3):
            K = 12
            row = rng.integers(-2, ctx[r], size=K)  # some negative ids too
            rows.append(row)
            req.append(r)
    topk = np.array(rows, dtype=np.int32)
    req_id = np.array(req, dtype=np.int32)
    owned = np.zeros(topk.shape, dtype=np.int64)
    for d in range(D):
        slots, count = oracle.dcp_filter_convert_index(req_id, bts[d], topk, D, d, bs,
                                                       interleave=interleave)
        for i in range(topk.shape[0]):
            for j in range(topk.shape[1]):
                t = int(topk[i, j])
                if t >= 0 and where[(int(req_id[i]), t)][0] == d:
                    assert slots[i, j] == where[(int(req_id[i]), t)][1]
                    owned[i, j] += 1
                else:
                    assert slots[i, j] == -1
        assert np.array_equal(count, (slots >= 0).sum(axis=1))
    # partition: every non-negative id is owned by exactly one rank
    assert np.array_equal(owned, (topk >= 0).astype(np.int64))
    # per-rank counts of a request equal the local sequence length helper
    for d in range(D):
        for r in range(R):
            assert counters[d, r] == oracle.dcp_local_seq_len(ctx[r], D, d, interleave)


def test_index_all_positions_counts_equal_local_seq_lens():
    rng = np.random.default_rng(5)
    ctx = [37, 200]
    for D in (1, 2, 4):
        bts, where, _ = _simulate_paged_cache(ctx, D, 16, rng)
        topk = np.full((2, 256), -1, dtype=np.int32)
        for r in range(2):
            topk[r, :ctx[r]] = rng.permutation(ctx[r])
        for d in range(D):
            _, count = oracle.dcp_filter_convert_index(
                np.arange(2), bts[d], topk, D, d, 16)
            assert count.tolist() == [oracle.dcp_local_seq_len(c, D, d) for c in ctx]


def test_local_seq_len_closed_form():
    # ceil((ctx - rank) / D) for ctx > rank, else 0
    for ctx in range(0, 40):
        for D in (1, 2, 3, 4, 8):
            for rank in range(D):
                want = max(0, -(-(ctx - rank) // D))
                assert oracle.dcp_local_seq_len(ctx, D, rank) == want


def test_local_seq_len_closed_form_interleaved():
    # whole rounds of I*D positions give each rank I; in the partial round the
    # rank's run starts at I*rank
    for ctx in range(0, 60):
        for D in (1, 2, 3, 4):
            for I in (1, 2, 3, 4):
                for rank in range(D):
                    rounds, rem = divmod(ctx, I * D)
                    want = rounds * I + min(max(rem - I * rank, 0), I)
                    assert oracle.dcp_local_seq_len(ctx, D, rank, I) == want


def test_index_interleave_is_a_bijection_onto_rank_local_positions():
    # per request, (rank, rank-local position) of the positions 0..ctx-1 are
    # distinct and each rank's local positions are exactly 0..count-1, so a
    # rank's identity block table (block b -> b) maps them to slots 0..count-1
    bs = 4
    for D in (1, 2, 3, 4):
        for I in (1, 2, 3, 5):
            ctx = 3 * I * D + 2
            t = np.arange(ctx, dtype=np.int32)[None]
            seen = set()
            for d in range(D):
                W = ctx // bs + 2
                ident = np.arange(W, dtype=np.int32)[None]
                slots, count = oracle.dcp_filter_convert_index(
                    np.zeros(1, np.int32), ident, t, D, d, bs, interleave=I)
                local = sorted(int(x) for x in slots[0] if x >= 0)
                assert local == list(range(int(count[0])))
                seen.update((d, x) for x in local)
            assert len(seen) == ctx


def test_index_single_rank_is_plain_paging_for_any_interleave():
    rng = np.random.default_rng(11)
    bt = rng.permutation(40).astype(np.int32).reshape(2, 20)
    topk = rng.integers(-1, 79, size=(2, 16)).astype(np.int32)
    for I in (1, 2, 7):
        slots, _ = oracle.dcp_filter_convert_index(np.array([0, 1], np.int32), bt, topk, 1, 0, 4,
                                                   interleave=I)
        for i in range(2):
            for j in range(16):
                t = int(topk[i, j])
                assert slots[i, j] == (-1 if t < 0 else bt[i, t // 4] * 4 + t % 4)


# ----------------------------------------------------------------- attention
def _dense_case(n, H, seed):
    gen = torch.Generator().manual_seed(seed)
    rows = inputs.random_rows(n, gen, "cpu")
    q = torch.randn((H, 576), generator=gen).to(torch.bfloat16)
    return rows, q


def _torch_dequant(rows: torch.Tensor):
    """K [n, 576] and V [n, 512] in float64 through torch's own casts."""
    codes = rows[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    scales = rows[:, 512:528].contiguous().view(torch.float32).to(torch.float64)
    nope = codes * scales.repeat_interleave(128, dim=1)
    rope = rows[:, 528:].contiguous().view(torch.bfloat16).to(torch.float64)
    return torch.cat([nope, rope], dim=1), nope


def _q_bits(q_bf16: torch.Tensor) -> np.ndarray:
    return q_bf16.contiguous().view(torch.int16).numpy().astype(np.uint16)


@pytest.mark.parametrize("n,H", [(1, 4), (7, 16), (64, 8), (300, 3)])
def test_attention_dense_matches_torch_sdpa(n, H):
    rows, q = _dense_case(n, H, seed=n)
    k, v = _torch_dequant(rows)
    qd = q.to(torch.float64)
    ref_out = torch.nn.functional.scaled_dot_product_attention(
        qd.unsqueeze(1), k.unsqueeze(0).expand(H, n, 576),
        v.unsqueeze(0).expand(H, n, 512), scale=SM_SCALE).squeeze(1)
    ref_lse = torch.logsumexp(SM_SCALE * (qd @ k.T), dim=1)
    # top-k = every position, in a random order, with -1s sprinkled in
    rng = np.random.default_rng(n)
    slots = np.concatenate([rng.permutation(n), -np.ones(5, dtype=np.int64)])
    slots = rng.permutation(slots)[None]
    out, lse = oracle.sparse_mla_decode(_q_bits(q)[None], rows.numpy(), slots, SM_SCALE)
    assert np.allclose(out[0], ref_out.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(lse[0], ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_attention_q_zero_closed_form():
    rows, _ = _dense_case(37, 2, seed=9)
    _, v = _torch_dequant(rows)
    q = torch.zeros((2, 576), dtype=torch.bfloat16)
    out, lse = oracle.sparse_mla_decode(_q_bits(q)[None], rows.numpy(),
                                        np.arange(37)[None], SM_SCALE)
    assert np.allclose(lse[0], math.log(37), rtol=0, atol=1e-14)
    assert np.allclose(out[0], v.mean(dim=0).numpy()[None], rtol=1e-13, atol=1e-14)


def test_attention_single_slot_closed_form():
    rows, q = _dense_case(5, 6, seed=10)
    k, v = _torch_dequant(rows)
    slots = np.array([[-1, 3, -1, -1]])
    out, lse = oracle.sparse_mla_decode(_q_bits(q)[None], rows.numpy(), slots, SM_SCALE)
    s = SM_SCALE * (q.to(torch.float64) @ k[3])
    assert np.allclose(lse[0], s.numpy(), rtol=1e-15, atol=1e-15)
    assert np.array_equal(out[0], np.broadcast_to(v[3].numpy(), (6, 512)))


def test_attention_order_invariance():
    rows, q = _dense_case(100, 4, seed=11)
    rng = np.random.default_rng(11)
    base = np.concatenate([rng.choice(100, 40, replace=False), -np.ones(8, np.int64)])
    a = oracle.sparse_mla_decode(_q_bits(q)[None], rows.numpy(), base[None], SM_SCALE)
    b = oracle.sparse_mla_decode(_q_bits(q)[None], rows.numpy(),
                                 rng.permutation(base)[None], SM_SCALE)
    assert np.allclose(a[0], b[0], rtol=0, atol=1e-12)
    assert np.allclose(a[1], b[1], rtol=0, atol=1e-12)


def test_attention_duplicate_slots_count_twice():
    """Reading taken: a slot listed twice is attended twice (the multiset)."""
    rows, q = _dense_case(3, 2, seed=12)
    k, v = _torch_dequant(rows)
    out, lse = oracle.sparse_mla_decode(_q_bits(q)[None], rows.numpy(),
                                        np.array([[0, 0, 2]]), SM_SCALE)
    kk = torch.stack([k[0], k[0], k[2]])
    vv = torch.stack([v[0], v[0], v[2]])
    s = SM_SCALE * (q.to(torch.float64) @ kk.T)
    assert np.allclose(lse[0], torch.logsumexp(s, 1).numpy(), atol=1e-13)
    assert np.allclose(out[0], (torch.softmax(s, 1) @ vv).numpy(), atol=1e-13)


def test_empty_row_case_from_pages():
    g = _golden("empty_row_case.json")
    T, H = g["num_tokens"], g["num_heads"]
    rows, _ = _dense_case(4, H, seed=13)
    q = torch.randn((T, H, 576), generator=torch.Generator().manual_seed(13))
    out, lse = oracle.sparse_mla_decode(_q_bits(q.to(torch.bfloat16)), rows.numpy(),
                                        np.array(g["local_indices"]), SM_SCALE)
    for r in g["empty_rows"]:
        assert np.array_equal(out[r], np.zeros_like(out[r]))
        assert np.all(np.isneginf(lse[r]))
    for r in g["nonempty_rows"]:
        assert np.all(np.isfinite(lse[r]))
    assert not np.isnan(out).any() and not np.isnan(lse).any()


# --------------------------------------------------------------------- merge
def _unsharded(wl, T_rows=None):
    """Attention over the union of every shard's rows for each query row:
    gather each valid global id's row from the shard the conversion puts it
    on, then one softmax over all of them."""
    pools = [s.pool.numpy() for s in wl.shards]
    q = _q_bits(wl.q)
    per_shard = [oracle.dcp_filter_convert_index(wl.req_id, s.block_table, wl.topk,
                                                 wl.D, d, wl.spec.block_size)[0]
                 for d, s in enumerate(wl.shards)]
    outs, lses = [], []
    for i in range(wl.T):
        rows = np.concatenate([pools[d][per_shard[d][i][per_shard[d][i] >= 0]]
                               for d in range(wl.D)])
        o, l = oracle.sparse_mla_decode_rows(oracle.bf16_bits_to_f64(q[i]), rows,
                                             wl.spec.sm_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def _sharded(wl):
    q = _q_bits(wl.q)
    outs, lses = [], []
    for d, s in enumerate(wl.shards):
        slots, _ = oracle.dcp_filter_convert_index(wl.req_id, s.block_table, wl.topk,
                                                   wl.D, d, wl.spec.block_size)
        o, l = oracle.sparse_mla_decode(q, s.pool.numpy(), slots, wl.spec.sm_scale)
        outs.append(o)
        lses.append(l)
    return outs, lses


def test_merge_of_shards_equals_unsharded_tiny():
    wl = inputs.make_workload("tiny", seed=0)
    outs, lses = _sharded(wl)
    out, lse = oracle.lse_merge(outs, lses)
    u_out, u_lse = _unsharded(wl)
    assert np.allclose(out, u_out, rtol=0, atol=1e-12)
    assert np.allclose(lse, u_lse, rtol=0, atol=1e-12)
    # every token reached the gathered rows through exactly one shard
    assert np.isfinite(lse).all()


def test_merge_of_shards_equals_unsharded_with_empty_shards():
    spec = inputs.WorkloadSpec(
        name="t", num_reqs=4, tokens_per_req=1, heads=4, topk=16, dcp=4,
        block_size=4, ctx_kind="fixed", ctx_fixed=(1, 2, 3, 40))
    wl = inputs.make_workload(spec, seed=4)
    outs, lses = _sharded(wl)
    # the ctx-1 request has nothing on ranks 1..3, ctx-2 nothing on 2..3
    assert np.isneginf(lses[1][0]).all() and np.isneginf(lses[3][1]).all()
    out, lse = oracle.lse_merge(outs, lses)
    u_out, u_lse = _unsharded(wl)
    assert np.allclose(out, u_out, rtol=0, atol=1e-12)
    assert np.allclose(lse, u_lse, rtol=0, atol=1e-12)


def test_merge_matches_torch_logsumexp():
    rng = np.random.default_rng(6)
    lses = [rng.normal(size=(3, 5)) * 4 for _ in range(4)]
    outs = [rng.normal(size=(3, 5, 512)) for _ in range(4)]
    out, lse = oracle.lse_merge(outs, lses)
    L = torch.from_numpy(np.stack(lses))
    ref_lse = torch.logsumexp(L, dim=0)
    w = torch.softmax(L, dim=0)
    ref_out = (w.unsqueeze(-1) * torch.from_numpy(np.stack(outs))).sum(0)
    assert np.allclose(lse, ref_lse.numpy(), atol=1e-13)
    assert np.allclose(out, ref_out.numpy(), atol=1e-13)


def test_merge_identity_changes_nothing_and_no_nan():
    rng = np.random.default_rng(7)
    o = rng.normal(size=(2, 3, 512))
    l = rng.normal(size=(2, 3))
    out, lse = oracle.lse_merge([o, np.zeros_like(o)], [l, np.full_like(l, -np.inf)])
    assert np.array_equal(out, o) and np.array_equal(lse, l)
    out, lse = oracle.lse_merge([np.zeros_like(o), o], [np.full_like(l, -np.inf), l])
    assert np.array_equal(out, o) and np.array_equal(lse, l)


def test_merge_all_empty_is_identity():
    z = np.zeros((2, 3, 512))
    ninf = np.full((2, 3), -np.inf)
    out, lse = oracle.lse_merge([z, z, z], [ninf, ninf, ninf])
    assert np.array_equal(out, z) and np.isneginf(lse).all()
    assert not np.isnan(out).any()


# --------------------------------------------------------------- spec decode
def test_spec_decode_rows_equal_per_token_results():
    spec = inputs.WorkloadSpec(
        name="mtp_small", num_reqs=3, tokens_per_req=2, heads=4, topk=32, dcp=2,
        block_size=8, ctx_kind="uniform", ctx_lo=20, ctx_hi=90)
    wl = inputs.make_workload(spec, seed=8)
    q = _q_bits(wl.q)
    for d, s in enumerate(wl.shards):
        slots, _ = oracle.dcp_filter_convert_index(wl.req_id, s.block_table, wl.topk,
                                                   wl.D, d, spec.block_size)
        out, lse = oracle.sparse_mla_decode(q, s.pool.numpy(), slots, spec.sm_scale)
        assert lse.shape == (6, 4)
        for b in range(3):
            for t in range(2):
                o1, l1 = oracle.sparse_mla_decode(q[b * 2 + t][None], s.pool.numpy(),
                                                  slots[b * 2 + t][None], spec.sm_scale)
                assert np.array_equal(lse[b * 2 + t], l1[0])
                assert np.array_equal(out[b * 2 + t], o1[0])
    # causality comes only from the indices: no id exceeds its own position
    for b in range(3):
        for t in range(2):
            pos = wl.ctx[b] - 2 + t
            assert wl.topk[b * 2 + t].max() <= pos


# ------------------------------------------------------- generator structure
def test_generator_structure_tiny():
    wl = inputs.make_workload("tiny", seed=0)
    assert wl.topk.shape == (2, 64) and wl.q.shape == (2, 16, 576)
    # ctx 37 row: 37 valid + 27 pad, then 6 random -1s (may overlap pads)
    for i, c in enumerate(wl.ctx):
        row = wl.topk[i]
        valid = row[row >= 0]
        assert len(set(valid.tolist())) == len(valid)
        assert valid.max() < c
        assert min(64, c) - 6 <= len(valid) <= min(64, c)
    for d, s in enumerate(wl.shards):
        assert s.live_rows == sum(oracle.dcp_local_seq_len(c, 2, d) for c in wl.ctx)
        poison = (s.pool.numpy() == 0xFF).all(axis=1)
        assert (~poison).sum() == s.live_rows


@pytest.mark.parametrize("interleave", [1, 2, 4, 64])
def test_generator_shard_sizes_follow_the_interleave_rule(interleave):
    """The generator sizes each shard's block allocation from its own count of
    the positions a shard holds; that count must equal the oracle's (pinned
    by the append simulation), and the oracle's conversion of every id must
    land inside the allocated blocks (it asserts otherwise)."""
    for ctx in list(range(0, 300)) + [4095, 4096, 65537]:
        for D in (1, 2, 3, 4, 8):
            for d in range(D):
                assert inputs.rows_on_shard(ctx, D, d, interleave) == \
                    oracle.dcp_local_seq_len(ctx, D, d, interleave), (ctx, D, d)
    spec = inputs.WorkloadSpec(name="il", num_reqs=3, tokens_per_req=1, heads=4, topk=256,
                               dcp=4, block_size=16, ctx_kind="uniform", ctx_lo=100,
                               ctx_hi=3000, interleave=interleave)
    wl = inputs.make_workload(spec, seed=interleave)
    for d, s in enumerate(wl.shards):
        assert s.live_rows == sum(oracle.dcp_local_seq_len(c, 4, d, interleave) for c in wl.ctx)
        sl, cnt = oracle.dcp_filter_convert_index(wl.req_id, s.block_table, wl.topk, 4, d, 16,
                                                  interleave)
        live = ~(s.pool.numpy()[sl[sl >= 0]] == 0xFF).all(axis=1)
        assert live.all()  # every converted id points at a filled row


# ------------------------------------------------------------- top-k select
def test_topk_select_matches_torch_topk_on_distinct_scores():
    rng = np.random.default_rng(21)
    for K in (1, 5, 64):
        T, L = 6, 150
        scores = rng.standard_normal((T, L))
        assert len(np.unique(scores)) == scores.size  # distinct: one right answer
        n_cand = rng.integers(0, L + 1, size=T)
        n_cand[0], n_cand[1] = L, 3
        got = oracle.topk_select(scores, n_cand, K)
        for i in range(T):
            n = int(n_cand[i])
            m = min(K, n)
            want = torch.topk(torch.from_numpy(scores[i, :n]), m, sorted=True).indices.numpy()
            assert got[i, :m].tolist() == want.tolist()
            assert np.all(got[i, m:] == -1)


def test_topk_select_k1_is_numpy_argmax_with_ties():
    rng = np.random.default_rng(22)
    scores = rng.integers(0, 4, size=(40, 30)).astype(np.float64)  # many ties
    got = oracle.topk_select(scores, np.full(40, 30), 1)
    assert got[:, 0].tolist() == np.argmax(scores, axis=1).tolist()  # first of equal maxima


def test_topk_select_all_equal_scores_keep_the_first_positions():
    for n in (0, 1, 7, 20):
        for K in (1, 7, 12):
            got = oracle.topk_select(np.zeros((1, 25)), [n], K)[0]
            m = min(K, n)
            assert got.tolist() == list(range(m)) + [-1] * (K - m)


def test_topk_select_short_rows_keep_every_candidate():
    rng = np.random.default_rng(23)
    scores = rng.standard_normal((3, 10))
    got = oracle.topk_select(scores, [0, 4, 10], 16)
    assert got[0].tolist() == [-1] * 16
    assert sorted(got[1, :4].tolist()) == [0, 1, 2, 3] and np.all(got[1, 4:] == -1)
    assert sorted(got[2, :10].tolist()) == list(range(10)) and np.all(got[2, 10:] == -1)


@pytest.mark.parametrize("D,K,decimals", [(1, 8, 6), (2, 16, 6), (4, 16, 1), (3, 40, 0)])
def test_dcp_topk_merge_of_rank_local_topk_equals_unsharded(D, K, decimals):
    # every global top-k entry is in its owner's local top-k under the same
    # order, so shard-then-merge selects exactly what one unsharded pass does
    rng = np.random.default_rng(D * 10 + K)
    T, L = 5, 97
    scores = np.round(rng.standard_normal((T, L)), decimals)  # decimals=0/1: heavy ties
    n_cand = rng.integers(1, L + 1, size=T)
    want = oracle.topk_select(scores, n_cand, K)
    cand_ids, cand_scores = [], []
    for d in range(D):
        local = scores[:, d::D]  # rank d holds positions d, d + D, ... (interleave 1)
        n_local = np.array([oracle.dcp_local_seq_len(int(n), D, d) for n in n_cand])
        lp = oracle.topk_select(local, n_local, K).astype(np.int64)
        ids = np.where(lp >= 0, lp * D + d, -1)
        cand_ids.append(ids)
        cand_scores.append(np.where(ids >= 0, np.take_along_axis(scores, np.maximum(ids, 0), 1),
                                    0.0))
    got = oracle.dcp_topk_merge(cand_ids, cand_scores, K)
    assert np.array_equal(got, want)


# ------------------------------------------------------------- dense decode
def _paged_dense_case(ctx, D, bs, S, H, seed, interleave=1):
    """Logical token rows per request, the D ranks' paged pools holding them
    (every row no token owns is NaN bytes), the ranks' block tables and q."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    bts, where, _ = _simulate_paged_cache(ctx, D, bs, rng, interleave)
    tokens = [inputs.random_rows(c, gen, "cpu").numpy() for c in ctx]
    n_slots = max(s for (_, s) in where.values()) + bs
    pools = [np.full((n_slots, 656), 0xFF, dtype=np.uint8) for _ in range(D)]
    for (r, t), (d, slot) in where.items():
        pools[d][slot] = tokens[r][t]
    q = torch.randn((len(ctx) * S, H, 576), generator=gen).to(torch.bfloat16)
    return tokens, pools, bts, q


@pytest.mark.parametrize("D,S,interleave", [(1, 1, 1), (1, 2, 1), (2, 2, 1), (4, 1, 1), (3, 2, 2)])
def test_dense_decode_sharded_and_merged_matches_torch_causal_sdpa(D, S, interleave):
    ctx, bs, H = [37, 9, 64], 8, 4
    tokens, pools, bts, q = _paged_dense_case(ctx, D, bs, S, H, seed=D * 10 + S, interleave=interleave)
    parts = [oracle.dense_mla_decode(_q_bits(q), pools[d], bts[d], ctx, S, D, d, bs, SM_SCALE,
                                     interleave) for d in range(D)]
    out, lse = oracle.lse_merge([p[0] for p in parts], [p[1] for p in parts])
    for b, c in enumerate(ctx):
        for s in range(S):
            i, p = b * S + s, c - S + s
            k, v = _torch_dequant(torch.from_numpy(tokens[b][: p + 1]))
            qd = q[i].to(torch.float64)
            n = p + 1
            ref = torch.nn.functional.scaled_dot_product_attention(
                qd.unsqueeze(1), k.unsqueeze(0).expand(H, n, 576),
                v.unsqueeze(0).expand(H, n, 512), scale=SM_SCALE).squeeze(1)
            ref_lse = torch.logsumexp(SM_SCALE * (qd @ k.T), dim=1)
            assert np.allclose(out[i], ref.numpy(), rtol=1e-12, atol=1e-12)
            assert np.allclose(lse[i], ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_dense_decode_spec_tokens_equal_single_token_requests():
    # a request's 2 query tokens at positions c-2, c-1 are the 1-token requests
    # with contexts c-1 and c over the same cache
    ctx, bs, H = [21, 40], 4, 3
    tokens, pools, bts, q = _paged_dense_case(ctx, 2, bs, 2, H, seed=9)
    single_ctx = [c - 1 + s for c in ctx for s in range(2)]
    single_bts = [np.repeat(bt[: len(ctx)], 2, axis=0) for bt in bts]
    for d in range(2):
        o2, l2 = oracle.dense_mla_decode(_q_bits(q), pools[d], bts[d], ctx, 2, 2, d, bs, SM_SCALE)
        o1, l1 = oracle.dense_mla_decode(_q_bits(q), pools[d], single_bts[d], single_ctx, 1, 2, d,
                                         bs, SM_SCALE)
        assert np.array_equal(o2, o1) and np.array_equal(l2, l1)


def test_flatten_lse_matches_torch_permute_reshape():
    x = torch.arange(2 * 3 * 4, dtype=torch.float64).reshape(2, 3, 4)  # [batch, heads, seq_len]
    want = x.permute(0, 2, 1).reshape(2 * 4, 3)
    assert np.array_equal(oracle.flatten_lse_bhs(x.numpy()), want.numpy())


@pytest.mark.parametrize("D,I", [(1, 1), (2, 1), (3, 2), (4, 4)])
def test_rank_local_position_to_global_id_is_the_inverse_conversion(D, I):
    """The global id the per-rank top-k reports for local position j of rank
    r, (j div I) I D + r I + j mod I, must be the position the conversion
    rule sends to rank r's local position j."""
    for r in range(D):
        for j in range(200):
            t = (j // I) * I * D + r * I + j % I
            assert (t // I) % D == r
            assert (t // (I * D)) * I + t % I == j
    # and the oracle's conversion agrees on a one-block-per-position table
    ctx = 300
    for r in range(D):
        n = oracle.dcp_local_seq_len(ctx, D, r, I)
        bt = np.arange(n, dtype=np.int32)[None]  # block j holds local position j (bs = 1)
        ids = np.array([[(j // I) * I * D + r * I + j % I for j in range(n)]], dtype=np.int32)
        slots, cnt = oracle.dcp_filter_convert_index(np.array([0]), bt, ids, D, r, 1, I)
        assert slots[0].tolist() == list(range(n)) and cnt[0] == n
