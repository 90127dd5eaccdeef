"""GPU parity: every step of the path through the C ABI against the float64
oracle on the same seeded inputs, for all five workloads at full size plus
edge cases.  Indices and valid counts must be bit-exact; out/lse follow the
tolerances in oracle/compare.py."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.compare import compare_out_lse
from sparse_mla_decode_dcp_gb300 import capi, inputs
from sparse_mla_decode_dcp_gb300.pipeline import DcpDecodeStep

pytestmark = pytest.mark.gpu


def _q_bits(q):
    return q.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)


class Run:
    """One workload on the GPU plus its oracle results (computed lazily)."""

    def __init__(self, name, dev):
        self.wl = inputs.make_workload(name, seed=0, device=dev)
        self.step = DcpDecodeStep(self.wl, device=dev)
        capi.load()
        capi.get_device_error(clear=True)
        self.out, self.lse = self.step.run()
        torch.cuda.synchronize()
        self.deverr = capi.get_device_error(clear=True)
        st = self.step
        self.f_out, self.f_lse = capi.dcp_sparse_mla_decode_fused(
            st.q, st.req_id, st.topk, st.pools, st.block_tables, self.wl.spec.block_size,
            self.wl.spec.sm_scale, bt_widths=st.bt_widths)
        torch.cuda.synchronize()
        self.f_deverr = capi.get_device_error(clear=True)
        self._ref = None

    def ref(self):
        if self._ref is None:
            wl = self.wl
            q = _q_bits(wl.q)
            slots, counts, outs, lses = [], [], [], []
            for d, s in enumerate(wl.shards):
                sl, c = oracle.dcp_filter_convert_index(wl.req_id, s.block_table, wl.topk,
                                                        wl.D, d, wl.spec.block_size)
                o, l = oracle.sparse_mla_decode(q, s.pool.cpu().numpy(), sl, wl.spec.sm_scale)
                slots.append(sl)
                counts.append(c)
                outs.append(o)
                lses.append(l)
            self._ref = (slots, counts, outs, lses)
        return self._ref


_RUNS = {}


@pytest.fixture(scope="module", params=inputs.WORKLOAD_ORDER)
def run(request, cuda_device):
    name = request.param
    if name not in _RUNS:
        _RUNS.clear()
        torch.cuda.empty_cache()
        _RUNS[name] = Run(name, cuda_device)
    return _RUNS[name]


def test_index_bit_exact(run):
    slots, counts, _, _ = run.ref()
    for d in range(run.wl.D):
        assert np.array_equal(run.step.local_slots[d].cpu().numpy(), slots[d]), f"shard {d}"
        assert np.array_equal(run.step.valid_count[d].cpu().numpy(), counts[d]), f"shard {d}"
    assert run.deverr == 0


def test_decode_matches_oracle_per_shard(run):
    _, _, outs, lses = run.ref()
    for d in range(run.wl.D):
        compare_out_lse(run.step.part_out[d], run.step.part_lse[d], outs[d], lses[d],
                        where=f"{run.wl.spec.name} shard {d}")


def test_merged_matches_oracle(run):
    _, _, outs, lses = run.ref()
    ref_out, ref_lse = oracle.lse_merge(outs, lses)
    compare_out_lse(run.out, run.lse, ref_out, ref_lse, where=f"{run.wl.spec.name} merged")


def test_fused_step_matches_oracle(run):
    """Conversion, decode and merge of all shards in one launch."""
    _, _, outs, lses = run.ref()
    ref_out, ref_lse = oracle.lse_merge(outs, lses)
    compare_out_lse(run.f_out, run.f_lse, ref_out, ref_lse, where=f"{run.wl.spec.name} fused")
    assert run.f_deverr == 0


def test_fused_step_agrees_with_pipeline(run):
    assert torch.equal(torch.isneginf(run.f_lse), torch.isneginf(run.lse))
    fin = torch.isfinite(run.lse)
    assert (run.f_lse[fin] - run.lse[fin]).abs().max().item() < 2e-3


def test_merge_kernel_alone_on_gpu_partials(run):
    """The oracle merge fed with the GPU's own bf16/fp32 partials isolates the
    merge kernel's error from the decode kernel's."""
    outs = [oracle.compare.to_f64(o) for o in run.step.part_out]
    lses = [oracle.compare.to_f64(l) for l in run.step.part_lse]
    ref_out, ref_lse = oracle.lse_merge(outs, lses)
    compare_out_lse(run.out, run.lse, ref_out, ref_lse, where="merge only")
    fin = np.isfinite(ref_lse)
    assert np.abs(run.lse.cpu().numpy()[fin] - ref_lse[fin]).max(initial=0) < 1e-5


def test_empty_shard_rows_are_identity(run):
    """Rows whose shard holds no candidate come out as exact (0, -inf)."""
    for d in range(run.wl.D):
        empty = run.step.valid_count[d].cpu().numpy() == 0
        if not empty.any():
            continue
        bits = run.step.part_out[d].cpu().view(torch.int16).numpy()[empty]
        assert np.all(bits == 0)
        assert torch.isneginf(run.step.part_lse[d].cpu()[torch.from_numpy(empty)]).all()


# --------------------------------------------------------------- edge cases
def _small_pool(n, dev, seed=1):
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    return inputs.random_rows(n, gen, dev)


def _decode_vs_oracle(q, pool, slots, sm_scale, where):
    out, lse = capi.sparse_mla_decode(q, pool, slots, sm_scale)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.sparse_mla_decode(_q_bits(q), pool.cpu().numpy(),
                                                slots.cpu().numpy(), sm_scale)
    compare_out_lse(out, lse, ref_out, ref_lse, where=where)
    return out, lse


def test_empty_row_case_from_pages(cuda_device):
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "empty_row_case.json")))
    pool = _small_pool(4, cuda_device)
    gen = torch.Generator(device=cuda_device).manual_seed(5)
    q = torch.randn((g["num_tokens"], g["num_heads"], 576), generator=gen,
                    device=cuda_device).to(torch.bfloat16)
    slots = torch.tensor(g["local_indices"], dtype=torch.int32, device=cuda_device)
    out, lse = _decode_vs_oracle(q, pool, slots, 1 / math.sqrt(192), "pages' case")
    for r in g["empty_rows"]:
        assert torch.all(out[r].view(torch.int16) == 0)
        assert torch.isneginf(lse[r]).all()
    for r in g["nonempty_rows"]:
        assert torch.isfinite(lse[r]).all()
    assert out.is_contiguous() and not out.isnan().any() and not lse.isnan().any()


@pytest.mark.parametrize("H", [1, 2, 16, 33, 64, 100, 127, 128])
def test_decode_head_counts(cuda_device, H):
    dev = cuda_device
    pool = _small_pool(300, dev, seed=H)
    g = torch.Generator(device=dev).manual_seed(1000 + H)  # independent of the pool
    T, K = 5, 96
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(H)
    s = np.stack([rng.permutation(np.concatenate([rng.choice(300, K - 10 * i, replace=False),
                                                  -np.ones(10 * i, np.int64)]))
                  for i in range(T)]).astype(np.int32)
    s[3] = -1  # one fully empty row
    slots = torch.from_numpy(s).to(dev)
    _decode_vs_oracle(q, pool, slots, 1 / math.sqrt(192), f"H={H}")


@pytest.mark.parametrize("K", [1, 3, 37, 64, 100, 128, 129, 192, 2048, 4096])
def test_decode_topk_sizes(cuda_device, K):
    """Rows of 1 to 64 key tiles (one row with every other entry -1): the
    MMA thread's QK^T(j) / PV(j - 2) order at its short-row edges (one, two
    and three tiles) and with split-K over long rows."""
    dev = cuda_device
    n = max(K, 8) + 50
    pool = _small_pool(n, dev, seed=K)
    g = torch.Generator(device=dev).manual_seed(1000 + K)  # independent of the pool
    T, H = 3, 128
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(K)
    s = np.stack([rng.choice(n, K, replace=False) for _ in range(T)]).astype(np.int32)
    s[1, ::2] = -1
    _decode_vs_oracle(q, pool, torch.from_numpy(s).to(dev), 1 / math.sqrt(192), f"K={K}")


def test_decode_single_valid_slot_lse_is_score(cuda_device):
    dev = cuda_device
    pool = _small_pool(10, dev, seed=3)
    g = torch.Generator(device=dev).manual_seed(1000 + 3)  # independent of the pool
    q = torch.randn((4, 128, 576), generator=g, device=dev).to(torch.bfloat16)
    s = torch.full((4, 64), -1, dtype=torch.int32, device=dev)
    for i in range(4):
        s[i, 7 * i] = i + 2
    _decode_vs_oracle(q, pool, s, 1 / math.sqrt(192), "single slot")


def test_decode_duplicate_slots(cuda_device):
    dev = cuda_device
    pool = _small_pool(20, dev, seed=4)
    g = torch.Generator(device=dev).manual_seed(1000 + 4)  # independent of the pool
    q = torch.randn((2, 64, 576), generator=g, device=dev).to(torch.bfloat16)
    s = torch.tensor([[0, 0, 5, 5, 5, -1, 7, 0], [3, -1, 3, 3, -1, -1, 19, 3]],
                     dtype=torch.int32, device=dev)
    _decode_vs_oracle(q, pool, s, 1 / math.sqrt(192), "duplicates")


def test_decode_order_invariance(cuda_device):
    dev = cuda_device
    pool = _small_pool(5000, dev, seed=6)
    g = torch.Generator(device=dev).manual_seed(1000 + 6)  # independent of the pool
    q = torch.randn((4, 128, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(6)
    s = np.stack([rng.choice(5000, 2048, replace=False) for _ in range(4)]).astype(np.int32)
    s[:, rng.choice(2048, 500, replace=False)] = -1
    perm = np.stack([rng.permutation(row) for row in s])
    o1, l1 = _decode_vs_oracle(q, pool, torch.from_numpy(s).to(dev), 0.072, "order a")
    o2, l2 = _decode_vs_oracle(q, pool, torch.from_numpy(perm).to(dev), 0.072, "order b")
    assert (l1 - l2).abs().max().item() < 2e-3


def test_decode_slot_out_of_range_is_masked_and_flagged(cuda_device):
    dev = cuda_device
    pool = _small_pool(16, dev, seed=7)
    g = torch.Generator(device=dev).manual_seed(1000 + 7)  # independent of the pool
    q = torch.randn((2, 16, 576), generator=g, device=dev).to(torch.bfloat16)
    bad = torch.tensor([[1, 2, 16, 3], [100000, -1, -1, -1]], dtype=torch.int32, device=dev)
    good = torch.tensor([[1, 2, -1, 3], [-1, -1, -1, -1]], dtype=torch.int32, device=dev)
    capi.get_device_error(clear=True)
    out_b, lse_b = capi.sparse_mla_decode(q, pool, bad, 0.07)
    torch.cuda.synchronize()
    assert capi.get_device_error(clear=True) & capi.DEVERR_SLOT_RANGE
    out_g, lse_g = capi.sparse_mla_decode(q, pool, good, 0.07)
    torch.cuda.synchronize()
    assert torch.equal(out_b, out_g) and torch.equal(lse_b, lse_g)
    assert torch.isneginf(lse_b[1]).all()


def test_zero_tokens_is_noop(cuda_device):
    dev = cuda_device
    pool = _small_pool(4, dev)
    q = torch.empty((0, 16, 576), dtype=torch.bfloat16, device=dev)
    s = torch.empty((0, 8), dtype=torch.int32, device=dev)
    out, lse = capi.sparse_mla_decode(q, pool, s, 0.07)
    assert out.shape == (0, 16, 512) and lse.shape == (0, 16)
    req = torch.empty((0,), dtype=torch.int32, device=dev)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    ls, cnt = capi.dcp_filter_convert_index(req, bt, s, 2, 0, 16)
    assert ls.shape == (0, 8)
    o, l = capi.dcp_lse_merge([out, out], [lse, lse])
    assert o.shape == (0, 16, 512)


def test_fused_bad_inputs_masked_and_flagged(cuda_device):
    """Ids past a block table, unallocated blocks and bad request ids drop
    out of the softmax and set device error bits; the rest matches the oracle."""
    dev = cuda_device
    D, bs = 2, 4
    pools = [_small_pool(32, dev, seed=20 + d) for d in range(D)]
    bts = [torch.tensor([[0, 1, -1], [2, 3, 4]], dtype=torch.int32, device=dev),
           torch.tensor([[5, -1, -1], [1, 6, 7]], dtype=torch.int32, device=dev)]
    req = torch.tensor([0, 9, 1], dtype=torch.int32, device=dev)
    topk = torch.tensor([[0, 1, 2, 3, 50, 17, -1, 6],
                         [0, 1, 2, 3, 4, 5, 6, 7],
                         [0, 1, 9, 10, 20, 21, -1, 8]], dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(21)
    q = torch.randn((3, 16, 576), generator=g, device=dev).to(torch.bfloat16)
    capi.get_device_error(clear=True)
    out, lse = capi.dcp_sparse_mla_decode_fused(q, req, topk, pools, bts, bs, 0.07)
    torch.cuda.synchronize()
    err = capi.get_device_error(clear=True)
    assert err & capi.DEVERR_BLOCK_TABLE and err & capi.DEVERR_REQ_ID
    assert torch.isneginf(lse[1]).all() and torch.all(out[1].view(torch.int16) == 0)
    # reference: drop the bad ids by hand (50 -> rank 0 local 25 -> column 6
    # past the width; 17 -> rank 1 local 8 -> column 2 = -1 for request 0)
    clean = torch.tensor([[0, 1, 2, 3, -1, -1, -1, 6], [-1] * 8,
                          [0, 1, 9, 10, 20, 21, -1, 8]], dtype=torch.int32, device=dev)
    q_bits = _q_bits(q)
    outs, lses = [], []
    for d in range(D):
        sl, _ = oracle.dcp_filter_convert_index(np.array([0, 0, 1]), bts[d].cpu().numpy(),
                                                clean.cpu().numpy(), D, d, bs)
        sl[1] = -1
        o, l = oracle.sparse_mla_decode(q_bits, pools[d].cpu().numpy(), sl, 0.07)
        outs.append(o)
        lses.append(l)
    ref_out, ref_lse = oracle.lse_merge(outs, lses)
    compare_out_lse(out, lse, ref_out, ref_lse, where="fused bad inputs")


@pytest.mark.parametrize("K", [64, 2048, 4096])
def test_fused_small_batches_split_k(cuda_device, K):
    """Few query rows: the fused step splits each row over several clusters
    and a second kernel combines the splits."""
    dev = cuda_device
    spec = inputs.WorkloadSpec(
        name="fused_small", num_reqs=3, tokens_per_req=1, heads=128, topk=K, dcp=4,
        block_size=64, ctx_kind="uniform", ctx_lo=K // 2, ctx_hi=3 * K)
    wl = inputs.make_workload(spec, seed=K, device=dev)
    step = DcpDecodeStep(wl, device=dev)
    out, lse = step.run()
    torch.cuda.synchronize()
    f_out, f_lse = capi.dcp_sparse_mla_decode_fused(
        step.q, step.req_id, step.topk, step.pools, step.block_tables, spec.block_size,
        spec.sm_scale, bt_widths=step.bt_widths)
    torch.cuda.synchronize()
    q_bits = _q_bits(wl.q)
    outs, lses = [], []
    for d, s in enumerate(wl.shards):
        sl, _ = oracle.dcp_filter_convert_index(wl.req_id, s.block_table, wl.topk, wl.D, d,
                                                spec.block_size)
        o, l = oracle.sparse_mla_decode(q_bits, s.pool.cpu().numpy(), sl, spec.sm_scale)
        outs.append(o)
        lses.append(l)
    ref_out, ref_lse = oracle.lse_merge(outs, lses)
    compare_out_lse(f_out, f_lse, ref_out, ref_lse, where=f"fused K={K}")
    compare_out_lse(out, lse, ref_out, ref_lse, where=f"pipeline K={K}")


@pytest.mark.parametrize("H,D,I", [(16, 3, 2), (100, 2, 1), (1, 5, 4)])
def test_fused_split_k_heads_shards_interleave(cuda_device, H, D, I):
    """The fused step with split-K (2 rows, 4 key ranges each, combined by
    the separate kernel) over head counts that leave an 8-head group part
    empty, odd shard counts and interleave sizes."""
    dev = cuda_device
    spec = inputs.WorkloadSpec(
        name=f"fused_sk_{H}_{D}_{I}", num_reqs=2, tokens_per_req=1, heads=H, topk=1024, dcp=D,
        block_size=16, ctx_kind="uniform", ctx_lo=700, ctx_hi=5000, interleave=I,
        neg_frac=0.1)
    wl = inputs.make_workload(spec, seed=H + 10 * D + I, device=dev)
    assert capi.decode_workspace_size(wl.T, H, wl.K) > 0
    step = DcpDecodeStep(wl, device=dev)
    capi.get_device_error(clear=True)
    f_out, f_lse = step.run_fused()
    torch.cuda.synchronize()
    assert capi.get_device_error(clear=True) == 0
    q_bits = _q_bits(wl.q)
    outs, lses = [], []
    for d, sh in enumerate(wl.shards):
        sl, _ = oracle.dcp_filter_convert_index(wl.req_id, sh.block_table, wl.topk, wl.D, d,
                                                spec.block_size, I)
        o, l = oracle.sparse_mla_decode(q_bits, sh.pool.cpu().numpy(), sl, spec.sm_scale)
        outs.append(o)
        lses.append(l)
    ref_out, ref_lse = oracle.lse_merge(outs, lses)
    compare_out_lse(f_out, f_lse, ref_out, ref_lse, where=f"fused split-K H={H} D={D} I={I}")


@pytest.mark.parametrize("interleave", [2, 4, 64])
def test_interleaved_step_matches_oracle(cuda_device, interleave):
    """Interleave size I > 1 (runs of I consecutive positions per shard) end
    to end: per-shard conversion bit-exact, the 2D+1 launch pipeline and the
    fused step both against the oracle's merge of its per-shard decodes."""
    dev = cuda_device
    spec = inputs.WorkloadSpec(
        name=f"interleave{interleave}", num_reqs=8, tokens_per_req=1, heads=128, topk=2048,
        dcp=4, block_size=64, ctx_kind="uniform", ctx_lo=2000, ctx_hi=20000,
        interleave=interleave)
    wl = inputs.make_workload(spec, seed=interleave, device=dev)
    step = DcpDecodeStep(wl, device=dev)
    capi.get_device_error(clear=True)
    out, lse = step.run()
    torch.cuda.synchronize()
    f_out, f_lse = step.run_fused()
    torch.cuda.synchronize()
    f_out, f_lse = f_out.clone(), f_lse.clone()
    assert capi.get_device_error(clear=True) == 0
    q_bits = _q_bits(wl.q)
    outs, lses = [], []
    for d, s in enumerate(wl.shards):
        sl, cnt = oracle.dcp_filter_convert_index(wl.req_id, s.block_table, wl.topk, wl.D, d,
                                                  spec.block_size, interleave)
        assert np.array_equal(step.local_slots[d].cpu().numpy(), sl), f"shard {d}"
        assert np.array_equal(step.valid_count[d].cpu().numpy(), cnt), f"shard {d}"
        o, l = oracle.sparse_mla_decode(q_bits, s.pool.cpu().numpy(), sl, spec.sm_scale)
        outs.append(o)
        lses.append(l)
    ref_out, ref_lse = oracle.lse_merge(outs, lses)
    compare_out_lse(out, lse, ref_out, ref_lse, where=f"pipeline I={interleave}")
    compare_out_lse(f_out, f_lse, ref_out, ref_lse, where=f"fused I={interleave}")


# ---------------------------------------------------------- index edge cases
def _convert_vs_oracle(req, bt, topk, D, rank, bs, dev, width=None, interleave=1):
    ls, cnt = capi.dcp_filter_convert_index(
        torch.from_numpy(req).to(dev), torch.from_numpy(bt).to(dev),
        torch.from_numpy(topk).to(dev), D, rank, bs, interleave=interleave, bt_width=width)
    torch.cuda.synchronize()
    ref_ls, ref_cnt = oracle.dcp_filter_convert_index(
        req, bt if width is None else bt[:, :width], topk, D, rank, bs, interleave)
    assert np.array_equal(ls.cpu().numpy(), ref_ls)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt)


def test_index_worked_examples_on_gpu(cuda_device):
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "index_worked_example.json")))
    for case in g["cases"]:
        ls, cnt = capi.dcp_filter_convert_index(
            torch.tensor(case["req_id"], dtype=torch.int32, device=cuda_device),
            torch.tensor(case["block_table"], dtype=torch.int32, device=cuda_device),
            torch.tensor(case["topk"], dtype=torch.int32, device=cuda_device),
            case["D"], case["rank"], case["block_size"])
        assert ls.cpu().tolist() == case["local_slots"], case["note"]
        assert cnt.cpu().tolist() == case["valid_count"], case["note"]


@pytest.mark.parametrize("K", [1, 5, 37, 64, 2048, 3001, 8192])
@pytest.mark.parametrize("D", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("interleave", [1, 2, 4, 64])
def test_index_random_shapes(cuda_device, K, D, interleave):
    """Random requests, ids and -1s against the oracle, bit-exact, for every
    rank; K spans one CTA per row and the four-CTA split (with a ragged last
    chunk at 3001 and several 16-byte groups per thread at 8192)."""
    rng = np.random.default_rng(K * 10 + D + 1000 * interleave)
    R, bs = 5, 16
    ctx = rng.integers(1, 5000, size=R)
    counts = [[inputs.rows_on_shard(int(c), D, d, interleave) for c in ctx] for d in range(D)]
    W = int(max(-(-n // bs) for row in counts for n in row)) + 1
    for rank in range(D):
        bt = np.full((R, W + 3), -1, dtype=np.int32)
        for r in range(R):
            nb = -(-counts[rank][r] // bs)
            bt[r, :nb] = rng.permutation(10000)[:nb]
        req = rng.integers(0, R, size=7).astype(np.int32)
        topk = np.stack([np.where(rng.random(K) < 0.1, -1,
                                  rng.integers(0, int(ctx[r]), size=K)) for r in req]).astype(np.int32)
        _convert_vs_oracle(req, bt, topk, D, rank, bs, cuda_device, interleave=interleave)


def test_index_bad_inputs_masked_and_flagged(cuda_device):
    dev = cuda_device
    bt = torch.tensor([[3, -1], [5, 6]], dtype=torch.int32, device=dev)
    req = torch.tensor([0, 7, 1], dtype=torch.int32, device=dev)  # 7: bad request
    # row 0: 40 -> local 20 -> block col 1 = -1 (unallocated); 100 -> col 3 past width
    topk = torch.tensor([[0, 40, 100, 2], [0, 2, 4, 6], [0, 20, 2, -5]],
                        dtype=torch.int32, device=dev)
    capi.get_device_error(clear=True)
    ls, cnt = capi.dcp_filter_convert_index(req, bt, topk, 2, 0, 16)
    torch.cuda.synchronize()
    err = capi.get_device_error(clear=True)
    assert err & capi.DEVERR_BLOCK_TABLE and err & capi.DEVERR_REQ_ID
    assert ls.cpu().tolist() == [[48, -1, -1, 49], [-1, -1, -1, -1], [80, 90, 81, -1]]
    assert cnt.cpu().tolist() == [2, 0, 3]


def test_index_row_stride_and_width(cuda_device):
    rng = np.random.default_rng(9)
    bt = np.full((3, 12), -1, dtype=np.int32)
    bt[:, :4] = rng.permutation(100)[:12].reshape(3, 4)
    req = np.array([2, 0, 1, 1], dtype=np.int32)
    topk = rng.integers(-1, 4 * 16 * 2, size=(4, 40)).astype(np.int32)
    _convert_vs_oracle(req, bt, topk, 2, 1, 16, cuda_device, width=4)


def test_index_permutation_equivariance(cuda_device):
    dev = cuda_device
    wl = inputs.make_workload("tiny", seed=3)
    perm = np.random.default_rng(3).permutation(wl.K)
    for d, s in enumerate(wl.shards):
        bt = torch.from_numpy(s.block_table).to(dev)
        req = torch.from_numpy(wl.req_id).to(dev)
        a, _ = capi.dcp_filter_convert_index(req, bt, torch.from_numpy(wl.topk).to(dev),
                                             wl.D, d, wl.spec.block_size)
        b, _ = capi.dcp_filter_convert_index(req, bt,
                                             torch.from_numpy(wl.topk[:, perm].copy()).to(dev),
                                             wl.D, d, wl.spec.block_size)
        assert torch.equal(a[:, torch.from_numpy(perm).to(dev)], b)


# ---------------------------------------------------------- merge edge cases
def test_merge_all_empty_and_identity(cuda_device):
    dev = cuda_device
    T, H = 3, 8
    g = torch.Generator(device=dev).manual_seed(11)
    o = torch.randn((T, H, 512), generator=g, device=dev).to(torch.bfloat16)
    l = torch.randn((T, H), generator=g, device=dev)
    z = torch.zeros_like(o)
    ninf = torch.full_like(l, -math.inf)
    out, lse = capi.dcp_lse_merge([z, o, z], [ninf, l, ninf])
    assert torch.equal(out, o)
    assert (lse - l).abs().max().item() < 1e-6
    out, lse = capi.dcp_lse_merge([z, z], [ninf, ninf])
    assert torch.all(out.view(torch.int16) == 0) and torch.isneginf(lse).all()


@pytest.mark.parametrize("D", [1, 2, 5, 16])
def test_merge_random_vs_oracle(cuda_device, D):
    dev = cuda_device
    T, H = 7, 33
    g = torch.Generator(device=dev).manual_seed(D)
    outs = [torch.randn((T, H, 512), generator=g, device=dev).to(torch.bfloat16)
            for _ in range(D)]
    lses = [torch.randn((T, H), generator=g, device=dev) * 5 for _ in range(D)]
    lses[0][2] = -math.inf
    out, lse = capi.dcp_lse_merge(outs, lses)
    ref_out, ref_lse = oracle.lse_merge([oracle.compare.to_f64(x) for x in outs],
                                        [oracle.compare.to_f64(x) for x in lses])
    compare_out_lse(out, lse, ref_out, ref_lse, where=f"merge D={D}")


@pytest.mark.parametrize("D,T", [(4, 40), (8, 20), (16, 10)])
def test_merge_more_rows_than_warps(cuda_device, D, T):
    """Thousands of (token, head) rows at D = 4, 8 and 16: every CTA of the
    merge grid, the last one partly filled, and an empty row at the end."""
    dev = cuda_device
    H = 128
    g = torch.Generator(device=dev).manual_seed(100 + D)
    outs = [torch.randn((T, H, 512), generator=g, device=dev).to(torch.bfloat16)
            for _ in range(D)]
    lses = [torch.randn((T, H), generator=g, device=dev) * 3 for _ in range(D)]
    lses[D - 1][T - 1] = -math.inf
    out, lse = capi.dcp_lse_merge(outs, lses)
    ref_out, ref_lse = oracle.lse_merge([oracle.compare.to_f64(x) for x in outs],
                                        [oracle.compare.to_f64(x) for x in lses])
    compare_out_lse(out, lse, ref_out, ref_lse, where=f"merge D={D} T={T}")


# ---------------------------------------------------------------- spec decode
def test_spec_decode_rows_equal_single_token_calls(cuda_device):
    """The MTP step's batched rows (b*2 + s) equal per-token calls."""
    dev = cuda_device
    spec = inputs.WorkloadSpec(
        name="mtp_small", num_reqs=6, tokens_per_req=2, heads=128, topk=512, dcp=2,
        block_size=64, ctx_kind="uniform", ctx_lo=600, ctx_hi=3000)
    wl = inputs.make_workload(spec, seed=12, device=dev)
    step = DcpDecodeStep(wl, device=dev)
    step.run()
    torch.cuda.synchronize()
    for d in range(wl.D):
        for i in range(wl.T):
            o, l = capi.sparse_mla_decode(step.q[i:i + 1], step.pools[d],
                                          step.local_slots[d][i:i + 1], spec.sm_scale)
            assert (o[0].float() - step.part_out[d][i].float()).abs().max().item() < 2e-2
            assert (l[0] - step.part_lse[d][i]).abs().max().item() < 2e-3


# ------------------------------------------------- fused step from host memory
def _pinned(t):
    return t.detach().cpu().contiguous().pin_memory()


@pytest.mark.parametrize("chunks", [1, 4, 8])
def test_fused_host_equals_device_step(cuda_device, chunks):
    """The host-buffer form (copies in, row groups decoded as their inputs
    land, copies back) gives the device form's results bit for bit: each row
    runs the same code whichever launch holds it (64 rows: no split-K either
    way)."""
    dev = cuda_device
    wl = inputs.make_workload("dcp4_long", seed=3, device=dev)
    step = DcpDecodeStep(wl, device=dev)
    ref_out, ref_lse = step.run_fused()
    torch.cuda.synchronize()
    ref_out, ref_lse = ref_out.cpu(), ref_lse.cpu()
    q_host, topk_host = _pinned(step.q), _pinned(step.topk)
    out_host = torch.full(tuple(ref_out.shape), 7, dtype=torch.bfloat16).pin_memory()
    lse_host = torch.full(tuple(ref_lse.shape), 7.0, dtype=torch.float32).pin_memory()
    step.q.zero_()
    step.topk.fill_(-1)
    step.out.zero_()
    for _ in range(2):
        step.run_fused_from_host(q_host, topk_host, out_host, lse_host, chunks=chunks)
        torch.cuda.synchronize()
        assert torch.equal(out_host, ref_out) and torch.equal(lse_host, ref_lse)
        out_host.fill_(7)
    # the staging buffers hold the step's device copies afterwards
    assert torch.equal(step.q.cpu(), q_host) and torch.equal(step.topk.cpu(), topk_host)


def test_fused_host_replays_in_cuda_graph(cuda_device):
    """The host-buffer step captured in a CUDA graph (its copy, group and
    copy-out streams join the capture through their events) replays to the
    device step's results, the host buffers refilled on every replay."""
    dev = cuda_device
    wl = inputs.make_workload("dcp4_long", seed=4, device=dev)
    step = DcpDecodeStep(wl, device=dev)
    ref_out, ref_lse = step.run_fused()
    torch.cuda.synchronize()
    ref_out, ref_lse = ref_out.cpu(), ref_lse.cpu()
    q_host, topk_host = _pinned(step.q), _pinned(step.topk)
    out_host = torch.empty(tuple(ref_out.shape), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty(tuple(ref_lse.shape), dtype=torch.float32).pin_memory()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    step.stream = s
    with torch.cuda.stream(s):
        step.run_fused_from_host(q_host, topk_host, out_host, lse_host, chunks=4)  # warm-up
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step.run_fused_from_host(q_host, topk_host, out_host, lse_host, chunks=4)
    for _ in range(2):
        out_host.fill_(7)
        lse_host.fill_(7.0)
        step.q.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_host, ref_out) and torch.equal(lse_host, ref_lse)


@pytest.mark.parametrize("chunks", [1, 3, 8])
def test_fused_host_ragged_groups_match_oracle(cuda_device, chunks):
    """5 rows in one group (then split-K over the workspace), in 3 groups
    (2, 2, 1) or in 8 asked for (one row per group), the groups decoded
    without split-K, against the oracle's per-shard decode and merge; one
    row's ids all -1."""
    dev = cuda_device
    spec = inputs.WorkloadSpec(
        name="host_ragged", num_reqs=5, tokens_per_req=1, heads=128, topk=2048, dcp=2,
        block_size=64, ctx_kind="uniform", ctx_lo=1500, ctx_hi=9000)
    wl = inputs.make_workload(spec, seed=17, device=dev)
    wl.topk[3] = -1
    step = DcpDecodeStep(wl, device=dev)
    q_host, topk_host = _pinned(wl.q), torch.from_numpy(wl.topk).contiguous().pin_memory()
    out_host = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty((wl.T, wl.H), dtype=torch.float32).pin_memory()
    capi.get_device_error(clear=True)
    step.run_fused_from_host(q_host, topk_host, out_host, lse_host, chunks=chunks)
    torch.cuda.synchronize()
    assert capi.get_device_error(clear=True) == 0
    q = _q_bits(wl.q)
    outs, lses = [], []
    for d, sh in enumerate(wl.shards):
        sl, _ = oracle.dcp_filter_convert_index(wl.req_id, sh.block_table, wl.topk, wl.D, d,
                                                spec.block_size)
        o, l = oracle.sparse_mla_decode(q, sh.pool.cpu().numpy(), sl, spec.sm_scale)
        outs.append(o)
        lses.append(l)
    ref_out, ref_lse = oracle.lse_merge(outs, lses)
    compare_out_lse(out_host, lse_host, ref_out, ref_lse, where=f"fused from host, chunks={chunks}")
    assert torch.all(out_host[3].view(torch.int16) == 0) and torch.isneginf(lse_host[3]).all()


# ------------------------------------------------------- workspace and graphs
@pytest.mark.parametrize("T,K", [(4, 2048), (40, 4096)])
def test_split_k_workspace_reused_across_calls(cuda_device, T, K):
    """Split-K arrival counters return to zero after every call, so one
    workspace serves any number of calls and results repeat bit for bit.
    4 rows x 8 key ranges fit one wave (the separate split combine); 40 rows
    x 2 ranges do not (the in-kernel combine, which counts arrivals)."""
    dev = cuda_device
    pool = _small_pool(5000, dev, seed=31)
    g = torch.Generator(device=dev).manual_seed(1000 + 31)  # independent of the pool
    H = 128
    assert capi.decode_workspace_size(T, H, K) > 0
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(31)
    s = torch.from_numpy(np.stack([rng.choice(5000, K, replace=False)
                                   for _ in range(T)]).astype(np.int32)).to(dev)
    ws = capi.alloc_decode_workspace(T, H, K, dev)
    first = capi.sparse_mla_decode(q, pool, s, 0.07, workspace=ws)
    first = (first[0].clone(), first[1].clone())
    for _ in range(3):
        o, l = capi.sparse_mla_decode(q, pool, s, 0.07, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(o, first[0]) and torch.equal(l, first[1])
    tick = ws[-256:]  # the counters sit in the last 256-byte block
    assert torch.count_nonzero(tick).item() == 0
    ref_out, ref_lse = oracle.sparse_mla_decode(_q_bits(q), pool.cpu().numpy(),
                                                s.cpu().numpy(), 0.07)
    compare_out_lse(first[0], first[1], ref_out, ref_lse, where=f"split-K T={T} K={K}")


@pytest.mark.parametrize("T,K", [(2, 1024), (40, 4096)])
@pytest.mark.parametrize("H", [1, 7, 33, 100])
def test_split_k_head_counts(cuda_device, H, T, K):
    """Split-K rows with head counts that leave the separate combine's last
    8-head group part-empty (2 rows x 4 key ranges) and the in-kernel
    combine's last columns unused (40 rows x 2 ranges)."""
    dev = cuda_device
    pool = _small_pool(5000, dev, seed=50 + H)
    g = torch.Generator(device=dev).manual_seed(2000 + H)
    assert capi.decode_workspace_size(T, H, K) > 0
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(50 + H)
    s = np.stack([rng.choice(5000, K, replace=False) for _ in range(T)]).astype(np.int32)
    s[1, 300:] = -1  # the later key ranges of row 1 hold nothing
    _decode_vs_oracle(q, pool, torch.from_numpy(s).to(dev), 0.07, f"split-K H={H} T={T}")


def test_split_k_combine_many_key_ranges(cuda_device):
    """300 key ranges of 2048 entries per row, mostly -1 (a grid of several
    waves: the in-kernel combine, which takes its per-range weights 288
    ranges at a time): row 0 has partials in both weight chunks, row 1 only
    past the first (one in its last range), and the all -1 row comes out as
    the merge identity."""
    dev = cuda_device
    n_pool = 4096
    pool = _small_pool(n_pool, dev, seed=41)
    g = torch.Generator(device=dev).manual_seed(1000 + 41)
    T, H, K = 3, 128, 300 * 2048
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(41)
    s = np.full((T, K), -1, dtype=np.int32)
    # row 0: a few keys in every 7th key range
    for sp in range(0, 300, 7):
        pos = sp * 2048 + rng.choice(2048, 5, replace=False)
        s[0, pos] = rng.choice(n_pool, 5, replace=False)
    # row 1: keys only in key ranges 288.. (the second chunk), one in the last range
    for sp in (288, 290, 299):
        pos = sp * 2048 + rng.choice(2048, 40, replace=False)
        s[1, pos] = rng.choice(n_pool, 40, replace=False)
    s[1, K - 1] = 17
    # row 2: no valid entry at all
    slots = torch.from_numpy(s).to(dev)
    out, lse = _decode_vs_oracle(q, pool, slots, 0.07, where="split combine over 300 key ranges")
    assert torch.count_nonzero(out[2]).item() == 0
    assert torch.isneginf(lse[2]).all()


def test_split_k_separate_combine_many_key_ranges(cuda_device):
    """One row over 76 key ranges (one wave of 152 CTAs: the separate split
    combine), mostly -1: the combine takes the ranges 32 per lane group
    (three groups, the last ragged) and the held ones 8 at a time."""
    dev = cuda_device
    n_pool = 4096
    pool = _small_pool(n_pool, dev, seed=43)
    g = torch.Generator(device=dev).manual_seed(1000 + 43)
    T, H, K = 1, 128, 40 * 2048
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(43)
    s = np.full((T, K), -1, dtype=np.int32)
    per = -(-K // 76)  # entries per key range
    held = [0, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 31, 32, 40, 63, 64, 70, 75]
    for sp in held:
        lo, hi = sp * per, min(K, (sp + 1) * per)
        pos = lo + rng.choice(hi - lo, 6, replace=False)
        s[0, pos] = rng.choice(n_pool, 6, replace=False)
    _decode_vs_oracle(q, pool, torch.from_numpy(s).to(dev), 0.07, where="separate combine, 76 ranges")


def test_split_k_decode_replays_in_cuda_graph(cuda_device):
    """A split-K call -- the decode kernel and the split combine launched
    programmatically dependent on it -- captured in a CUDA graph replays to
    the same bits as the call made directly."""
    dev = cuda_device
    pool = _small_pool(3000, dev, seed=61)
    g = torch.Generator(device=dev).manual_seed(1061)
    T, H, K = 2, 128, 2048
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(61)
    slots = torch.from_numpy(np.stack([rng.choice(3000, K, replace=False)
                                       for _ in range(T)]).astype(np.int32)).to(dev)
    ws = capi.alloc_decode_workspace(T, H, K, dev)
    assert ws is not None
    ref_out, ref_lse = capi.sparse_mla_decode(q, pool, slots, 0.07, workspace=ws)
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    out = torch.empty_like(ref_out)
    lse = torch.empty_like(ref_lse)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            capi.sparse_mla_decode(q, pool, slots, 0.07, out=out, lse=lse, workspace=ws)
    for _ in range(2):
        out.fill_(7)
        lse.fill_(7)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("path", ["fused", "pipeline"])
def test_step_replays_in_cuda_graph(cuda_device, path):
    dev = cuda_device
    wl = inputs.make_workload("tiny", seed=5, device=dev)
    step = DcpDecodeStep(wl, device=dev)
    fn = step.run_fused if path == "fused" else step.run
    fn()
    torch.cuda.synchronize()
    ref_out, ref_lse = step.out.clone(), step.lse.clone()
    step.out.zero_()
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            fn()
    for _ in range(2):
        step.out.fill_(7)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(step.out, ref_out) and torch.equal(step.lse, ref_lse)


def _p_rounding_bound_check(out, ref_out, ref_lse, q, pool, s):
    """P is rounded to fp16 (relative 2^-11 per weight) before the PV product,
    so out[h, c] may be off by up to 2^-11 * sum_j w_hj |v_jc| -- an absolute
    error that does not shrink when cancellation makes out small -- plus the
    final bf16 rounding.  A missed or doubled rescale is off by a factor of
    2^8 or more and fails this bound."""
    o = out.float().cpu().numpy().astype(np.float64)
    qf = oracle.bf16_bits_to_f64(_q_bits(q))
    sl = s.cpu().numpy()
    pool_np = pool.cpu().numpy()
    for t in range(sl.shape[0]):
        valid = sl[t][sl[t] >= 0]
        nope, rope = oracle.parse_rows(pool_np[valid])
        sc = (qf[t] @ np.concatenate([nope, rope], axis=1).T) / math.sqrt(192)
        w = np.exp(sc - ref_lse[t][:, None])
        p_round = 2.0 ** -11 * (w @ np.abs(nope))
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref_out[t]), 2.0 ** -126))) - 7)
        assert np.all(np.abs(o[t] - ref_out[t]) <= 1.5 * p_round + ulp + 1e-6), t


def _forced_rescale_inputs(dev, rope_boost, latent_scale_late):
    n = 512
    pool = _small_pool(n, dev, seed=41)
    scales = torch.full((n, 4), 2.0 ** -9, dtype=torch.float32, device=dev)
    scales[64:] = latent_scale_late  # rows past the first tile
    pool[:, 512:528] = scales.view(torch.uint8)
    if rope_boost != 1.0:
        rope = pool[64:, 528:656].contiguous().view(torch.bfloat16).float() * rope_boost
        pool[64:, 528:656] = rope.to(torch.bfloat16).view(torch.uint8)
    g = torch.Generator(device=dev).manual_seed(1041)
    T, H = 3, 128
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    s = torch.arange(n, dtype=torch.int32, device=dev).repeat(T, 1)  # tile 0 = small rows
    s[1] = torch.flip(s[1], dims=[0])  # large rows first: no rescale needed
    s[2, 100:300] = -1
    return pool, q, s


def test_decode_forced_rescale(cuda_device):
    """Later tiles carry 5x larger rope values, so their scores jump by more
    than 2^8 above the running maximum for most (but not all) head rows,
    exercising the O rescale (and rows of one warp disagreeing about it).
    Values (the latent) keep power-of-two scales and stay below 1, so every
    dequantised key is exact in fp16 and the contract's tolerances apply in
    full."""
    dev = cuda_device
    pool, q, s = _forced_rescale_inputs(dev, rope_boost=5.0, latent_scale_late=2.0 ** -9)
    capi.get_device_error(clear=True)
    out, lse = capi.sparse_mla_decode(q, pool, s, 1 / math.sqrt(192))
    torch.cuda.synchronize()
    assert capi.get_device_error(clear=True) == 0
    ref_out, ref_lse = oracle.sparse_mla_decode(_q_bits(q), pool.cpu().numpy(), s.cpu().numpy(),
                                                1 / math.sqrt(192))
    # the scores really do jump: the late rows' maximum exceeds the first
    # tile's by more than 8 in log2 units for most head rows of token 0
    qf = oracle.bf16_bits_to_f64(_q_bits(q))[0]
    nope, rope = oracle.parse_rows(pool.cpu().numpy())
    sc = (qf @ np.concatenate([nope, rope], axis=1).T) / math.sqrt(192) * 1.4426950408889634
    jump = sc[:, 64:].max(axis=1) - sc[:, :64].max(axis=1)
    assert (jump > 8).mean() > 0.5 and (jump <= 8).any()
    compare_out_lse(out, lse, ref_out, ref_lse, where="forced rescale")
    # exact keys: only fp32 accumulation, ex2 and the fp16 P remain
    assert np.abs(lse.cpu().numpy() - ref_lse).max() < 2e-4
    _p_rounding_bound_check(out, ref_out, ref_lse, q, pool, s)


def test_decode_forced_rescale_large_values(cuda_device):
    """The same jump driven by 16x larger latents, so the output itself
    reaches |out| ~ 14.  There a bf16 ulp is 2^-4 = 0.0625: a correctly
    rounded result can differ from the oracle's bf16 rounding by one ulp,
    above the absolute 2e-2 the contract states for the workloads' unit-scale
    outputs.  So this case is held to the contract's relative L2 and LSE
    tolerances and, per element, to the derived fp16-P bound (which a missed
    or doubled rescale fails by orders of magnitude)."""
    dev = cuda_device
    pool, q, s = _forced_rescale_inputs(dev, rope_boost=1.0, latent_scale_late=2.0 ** -5)
    capi.get_device_error(clear=True)
    out, lse = capi.sparse_mla_decode(q, pool, s, 1 / math.sqrt(192))
    torch.cuda.synchronize()
    assert capi.get_device_error(clear=True) == 0
    ref_out, ref_lse = oracle.sparse_mla_decode(_q_bits(q), pool.cpu().numpy(), s.cpu().numpy(),
                                                1 / math.sqrt(192))
    assert np.abs(ref_out).max() > 8
    assert np.abs(lse.cpu().numpy() - ref_lse).max() < 2e-4
    o = out.float().cpu().numpy().astype(np.float64)
    assert np.linalg.norm(o - ref_out) / np.linalg.norm(ref_out) < 1e-2
    _p_rounding_bound_check(out, ref_out, ref_lse, q, pool, s)


# ---------------------------------------------------------------- dense decode
def _dense_case(dev, B, S, D, I, lo, hi, seed):
    spec = inputs.WorkloadSpec(
        name=f"dense_{B}x{S}_D{D}_I{I}", num_reqs=B, tokens_per_req=S, heads=128, topk=64,
        dcp=D, block_size=64, ctx_kind="uniform", ctx_lo=lo, ctx_hi=hi, interleave=I)
    wl = inputs.make_workload(spec, seed=seed, device=dev)
    pools = [s.pool for s in wl.shards]
    bts = [torch.from_numpy(s.block_table).to(dev) for s in wl.shards]
    ctx = torch.from_numpy(wl.ctx.astype(np.int32)).to(dev)
    return wl, pools, bts, ctx, int(wl.ctx.max())


@pytest.mark.parametrize("D,S,I", [(1, 1, 1), (2, 1, 1), (2, 2, 1), (4, 1, 1), (4, 2, 1),
                                   (2, 2, 2), (4, 1, 4)])
def test_dense_decode_matches_oracle(cuda_device, D, S, I):
    """Every cached position of each request's causal context: one rank's
    partial (rank = d) against the oracle's dense decode of that rank, and the
    merged result (rank = -1, one launch over all pools) against the oracle's
    LSE merge of the ranks' partials; rows in token order b*S + s, i.e. the
    [batch, heads, seq_len] -> [tokens, heads] flattening of the LSE."""
    dev = cuda_device
    wl, pools, bts, ctx, max_ctx = _dense_case(dev, 5, S, D, I, 1, 4096, seed=10 * D + S + I)
    spec = wl.spec
    q_bits = _q_bits(wl.q)
    capi.get_device_error(clear=True)
    refs_o, refs_l = [], []
    for d in range(D):
        o, l = capi.dcp_dense_mla_decode(wl.q, ctx, max_ctx, S, pools, bts, spec.block_size,
                                         spec.sm_scale, rank=d, interleave=I)
        torch.cuda.synchronize()
        ro, rl = oracle.dense_mla_decode(q_bits, wl.shards[d].pool.cpu().numpy(),
                                         wl.shards[d].block_table, wl.ctx, S, D, d,
                                         spec.block_size, spec.sm_scale, I)
        compare_out_lse(o, l, ro, rl, where=f"dense rank {d}")
        refs_o.append(ro)
        refs_l.append(rl)
    ref_out, ref_lse = oracle.lse_merge(refs_o, refs_l)
    out, lse = capi.dcp_dense_mla_decode(wl.q, ctx, max_ctx, S, pools, bts, spec.block_size,
                                         spec.sm_scale, rank=-1, interleave=I)
    torch.cuda.synchronize()
    assert capi.get_device_error(clear=True) == 0
    compare_out_lse(out, lse, ref_out, ref_lse, where=f"dense merged D={D} S={S} I={I}")
    # the flattening: [B, H, S] read back in token order equals the kernel's rows
    B, H = len(wl.ctx), spec.heads
    lse_bhs = lse.cpu().numpy().reshape(B, S, H).transpose(0, 2, 1)
    assert np.array_equal(oracle.flatten_lse_bhs(lse_bhs), lse.cpu().numpy())


def test_dense_decode_skips_empty_key_ranges(cuda_device):
    """Dense grids of several waves (the in-kernel split combine) whose short
    rows leave key ranges -- for rank 1 of the shortest, every range --
    without a position: those splits skip the set-up and publish empty
    partials, and such a split may be its row's last arrival and combine it.
    Merged (4 ranges per row) and per rank (2 ranges per row)."""
    dev = cuda_device
    rng = np.random.default_rng(91)
    ctx_fixed = tuple(int(c) for c in np.concatenate(
        [[2, 2, 3, 4, 5, 1000, 2049, 2050, 2051, 4097, 4098, 8192], rng.integers(2, 8193, 28)]))
    spec = inputs.WorkloadSpec(
        name="dense_short_rows", num_reqs=40, tokens_per_req=2, heads=128, topk=64, dcp=2,
        block_size=64, ctx_kind="fixed", ctx_fixed=ctx_fixed, interleave=1)
    wl = inputs.make_workload(spec, seed=91, device=dev)
    pools = [sh.pool for sh in wl.shards]
    bts = [torch.from_numpy(sh.block_table).to(dev) for sh in wl.shards]
    ctx = torch.from_numpy(wl.ctx.astype(np.int32)).to(dev)
    max_ctx = int(wl.ctx.max())
    q_bits = _q_bits(wl.q)
    capi.get_device_error(clear=True)
    refs_o, refs_l = [], []
    for d in range(2):
        o, l = capi.dcp_dense_mla_decode(wl.q, ctx, max_ctx, 2, pools, bts, spec.block_size,
                                         spec.sm_scale, rank=d)
        torch.cuda.synchronize()
        ro, rl = oracle.dense_mla_decode(q_bits, wl.shards[d].pool.cpu().numpy(),
                                         wl.shards[d].block_table, wl.ctx, 2, 2, d,
                                         spec.block_size, spec.sm_scale)
        compare_out_lse(o, l, ro, rl, where=f"dense short rows rank {d}")
        empty = np.isneginf(rl).all(axis=1)
        if d == 1:
            assert empty.any()  # token 0 of a context of 2 has only position 0, on rank 0
        assert torch.all(o[torch.from_numpy(empty).to(dev)].view(torch.int16) == 0)
        refs_o.append(ro)
        refs_l.append(rl)
    out, lse = capi.dcp_dense_mla_decode(wl.q, ctx, max_ctx, 2, pools, bts, spec.block_size,
                                         spec.sm_scale)
    torch.cuda.synchronize()
    assert capi.get_device_error(clear=True) == 0
    ref_out, ref_lse = oracle.lse_merge(refs_o, refs_l)
    compare_out_lse(out, lse, ref_out, ref_lse, where="dense short rows merged")


def test_dense_decode_split_k_long_contexts(cuda_device):
    """Enough rows that the split count is set by the 2048-key list limit and
    contexts above it: several splits per row, combined by the split merge."""
    dev = cuda_device
    wl, pools, bts, ctx, max_ctx = _dense_case(dev, 40, 2, 2, 1, 2500, 4096, seed=77)
    spec = wl.spec
    assert capi.dense_decode_workspace_size(80, 128, max_ctx, 2, 1, -1) > 0
    out, lse = capi.dcp_dense_mla_decode(wl.q, ctx, max_ctx, 2, pools, bts, spec.block_size,
                                         spec.sm_scale)
    torch.cuda.synchronize()
    q_bits = _q_bits(wl.q)
    refs = [oracle.dense_mla_decode(q_bits, wl.shards[d].pool.cpu().numpy(),
                                    wl.shards[d].block_table, wl.ctx, 2, 2, d, spec.block_size,
                                    spec.sm_scale) for d in range(2)]
    ref_out, ref_lse = oracle.lse_merge([r[0] for r in refs], [r[1] for r in refs])
    compare_out_lse(out, lse, ref_out, ref_lse, where="dense split-K")


def test_dense_decode_context_out_of_range_is_flagged(cuda_device):
    """A context shorter than its request's query tokens (or past max_ctx) is
    an input error: those rows come out as (0, -inf) and the device error
    word says so; the other rows are unaffected."""
    dev = cuda_device
    wl, pools, bts, ctx, max_ctx = _dense_case(dev, 3, 2, 2, 1, 100, 600, seed=5)
    spec = wl.spec
    good_out, good_lse = capi.dcp_dense_mla_decode(wl.q, ctx, max_ctx, 2, pools, bts,
                                                   spec.block_size, spec.sm_scale)
    torch.cuda.synchronize()
    bad = ctx.clone()
    bad[1] = 1  # request 1 has 2 query tokens but a context of 1
    capi.get_device_error(clear=True)
    out, lse = capi.dcp_dense_mla_decode(wl.q, bad, max_ctx, 2, pools, bts, spec.block_size,
                                         spec.sm_scale)
    torch.cuda.synchronize()
    assert capi.get_device_error(clear=True) & capi.DEVERR_CONTEXT
    assert torch.isneginf(lse[2:4]).all() and torch.all(out[2:4].view(torch.int16) == 0)
    keep = torch.tensor([0, 1, 4, 5], device=dev)
    assert torch.equal(out[keep], good_out[keep]) and torch.equal(lse[keep], good_lse[keep])


# ------------------------------------------------------------ global top-k
def _topk_vs_oracle(dev, scores64, n_cand, K, where):
    """Both forms of the select: rows longer than a chunk cut into chunks
    (with a workspace) and one CTA per whole row (without)."""
    s32 = np.asarray(scores64, dtype=np.float32)
    want = oracle.topk_select(s32.astype(np.float64), n_cand, K)
    sc = torch.from_numpy(s32).to(dev)
    nc = torch.from_numpy(np.asarray(n_cand, dtype=np.int32)).to(dev)
    for ws in (True, None):
        got = capi.topk_select(sc, nc, K, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), want), (where, ws)


def test_topk_select_chunk_edges(cuda_device):
    """Few long rows cut into chunks (min(8, SMs / T) a row, of
    ceil(L / count) rounded up to 4 candidates): rows ending just before, at
    and just past a chunk's end, a row shorter than K and an empty one in a
    chunked call, one row of 2^21 candidates with and without ties, and 32
    rows (4 chunks each on a 152-SM GPU): the union of the chunks' K best
    holds the row's K best."""
    rng = np.random.default_rng(81)
    T, L = 8, 16 * 16384 + 5
    assert capi.topk_select_workspace_size(T, L, 2048) > 0
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    count = min(8, sms // T)
    chunk = ((L + count - 1) // count + 3) // 4 * 4
    scores = rng.standard_normal((T, L))
    n_cand = [chunk - 1, chunk, chunk + 1, 2 * chunk, 2 * chunk + 1, L, 100, 0]
    _topk_vs_oracle(cuda_device, scores, n_cand, 2048, "chunk edges")
    # the kept scores come back through the chunks' slabs: each is its id's
    # score, and the padding's is 0
    s32 = scores.astype(np.float32)
    ids, kept = capi.topk_select(torch.from_numpy(s32).to(cuda_device),
                                 torch.tensor(n_cand, dtype=torch.int32, device=cuda_device),
                                 2048, with_scores=True)
    ids, kept = ids.cpu().numpy(), kept.cpu().numpy()
    valid = ids >= 0
    rows = np.broadcast_to(np.arange(T)[:, None], ids.shape)
    assert np.array_equal(kept[valid], s32[rows[valid], ids[valid]])
    assert np.all(kept[~valid] == 0)
    big = rng.standard_normal((1, 1 << 21))
    _topk_vs_oracle(cuda_device, big, [(1 << 21) - 3], 2048, "one long row")
    _topk_vs_oracle(cuda_device, np.round(big, 1), [1 << 21], 4096, "one long row, ties")
    many = rng.standard_normal((32, 262144))
    _topk_vs_oracle(cuda_device, many, rng.integers(0, 262145, size=32), 2048, "32 rows")


@pytest.mark.parametrize("L,K", [(97, 16), (3000, 1000), (5000, 2048), (131072, 2048),
                                 (50000, 3001), (20000, 4096), (30000, 8192), (40000, 16384),
                                 (300000, 16384)])
def test_topk_select_matches_oracle(cuda_device, L, K):
    """Random rows up to 128k candidates, some shorter than K: bit-exact ids.
    K covers every sort the kernel picks by the padded size kp: the shared-
    memory network (kp 1024, 16384), warp runs and merges (kp 2048, 4096),
    the register network (kp 8192)."""
    rng = np.random.default_rng(L + K)
    T = 6
    scores = rng.standard_normal((T, L))
    n_cand = rng.integers(0, L + 1, size=T)
    n_cand[0], n_cand[1] = L, min(L, K // 2)  # full row, and fewer than K candidates
    _topk_vs_oracle(cuda_device, scores, n_cand, K, f"L={L} K={K}")


def test_topk_select_pair_and_many_rows(cuda_device):
    """Rows of 16384 or more positions take a cluster of two CTAs each
    while two CTAs a row fit on the GPU, the first walking ceil(n / 8) quads
    and the second the rest: rows whose second half is empty or short, NaN,
    signed zeros and infinities among the scores; then 100 such rows, more
    than half the SM count, which take one CTA each."""
    rng = np.random.default_rng(91)
    L = 20000
    scores = rng.standard_normal((12, L))
    scores[:, 1] = np.nan
    scores[:, 2] = -0.0
    scores[:, 6] = np.inf
    scores[:, 9] = -np.inf
    scores[5, :4000] = 0.0
    n_cand = [0, 1, 3, 4, 5, 7, 8, 9, 16383, 16384, L, 9999]
    for K in (4, 2048):
        _topk_vs_oracle(cuda_device, scores, n_cand, K, f"pairs K={K}")
    many = rng.standard_normal((100, L))
    _topk_vs_oracle(cuda_device, many, rng.integers(0, L + 1, size=100), 2048, "100 rows")


@pytest.mark.parametrize("decimals", [0, 1])
def test_topk_select_heavy_ties(cuda_device, decimals):
    """Scores rounded to few decimals: thousands of equal scores straddle the
    K-th place, and the ids among them must be the smallest positions."""
    rng = np.random.default_rng(50 + decimals)
    scores = np.round(rng.standard_normal((5, 30000)), decimals)
    _topk_vs_oracle(cuda_device, scores, np.full(5, 30000), 2048, f"ties {decimals}")
    _topk_vs_oracle(cuda_device, np.zeros((2, 5000)), [5000, 100], 2048, "all equal")


@pytest.mark.parametrize("L,K", [(60000, 2048), (40000, 16384)])
def test_topk_select_boundary_bin_past_shared_memory(cuda_device, L, K):
    """More equal scores at the K-th place than the kernel's shared-memory
    list holds (its radix select then reads the row again from global
    memory): still the smallest ids among the ties, in order."""
    rng = np.random.default_rng(L)
    scores = np.zeros((3, L))
    scores[2, rng.integers(0, L, 500)] = 1.0  # a few larger scores ahead of the ties
    _topk_vs_oracle(cuda_device, scores, [L, L // 2, L], K, f"ties past shared memory L={L}")


@pytest.mark.parametrize("L", [5, 6, 7, 19])
def test_topk_select_row_alignments(cuda_device, L):
    """Row strides that start rows at every offset within 16 bytes, and row
    lengths shorter than, equal to and past a few aligned quads: the scores
    before a row's first aligned quad and after its last one are read one by
    one, and every candidate is seen exactly once."""
    rng = np.random.default_rng(70 + L)
    T = 8
    scores = rng.standard_normal((T, L))
    n_cand = [min(L, x) for x in (0, 1, 2, 3, 4, 5, 7, L)]
    for K in (4, 16):
        _topk_vs_oracle(cuda_device, scores, n_cand, K, f"L={L} K={K}")


def test_topk_select_nan_and_signed_zero(cuda_device):
    """NaN ranks below every number (-inf included) and -0 ties with +0."""
    row = np.array([0.0, -0.0, np.nan, 1.5, -np.inf, np.nan, -0.0, 2.0, np.inf, -1.0], np.float64)
    scores = np.stack([row, row[::-1].copy()])
    for K in (1, 3, 6, 10, 12):
        _topk_vs_oracle(cuda_device, scores, [10, 10], K, f"special K={K}")


@pytest.mark.parametrize("D,I,decimals", [(2, 1, 6), (4, 1, 1), (4, 2, 6), (3, 64, 0)])
def test_dcp_topk_local_then_merge_equals_unsharded(cuda_device, D, I, decimals):
    """Per rank: the top-k of the positions it holds, as global ids (one
    launch per rank over its local score array); then the merge of the ranks'
    candidates: bit-exact equal to the oracle's unsharded top-k, and to the
    oracle's merge of the same candidates."""
    dev = cuda_device
    rng = np.random.default_rng(D * 100 + I + decimals)
    T, L, K = 4, 20000, 2048
    scores = np.round(rng.standard_normal((T, L)), decimals).astype(np.float32)
    n_cand = rng.integers(1, L + 1, size=T)
    n_cand[0] = 1500  # fewer candidates than K
    want = oracle.topk_select(scores.astype(np.float64), n_cand, K)
    ids, scs = [], []
    for r in range(D):
        n_loc = np.array([oracle.dcp_local_seq_len(int(n), D, r, I) for n in n_cand], np.int32)
        Lr = oracle.dcp_local_seq_len(L, D, r, I)
        gl = np.array([(j // I) * I * D + r * I + j % I for j in range(Lr)])
        local = np.ascontiguousarray(scores[:, gl])
        i_r, s_r = capi.topk_select(torch.from_numpy(local).to(dev),
                                    torch.from_numpy(n_loc).to(dev), K, D=D, rank=r,
                                    interleave=I, with_scores=True)
        ids.append(i_r)
        scs.append(s_r)
    cand_ids = torch.cat(ids, dim=1).contiguous()
    cand_sc = torch.cat(scs, dim=1).contiguous()
    got = capi.dcp_topk_merge(cand_ids, cand_sc, K)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want)
    ref = oracle.dcp_topk_merge([x.cpu().numpy() for x in ids],
                                [x.cpu().numpy().astype(np.float64) for x in scs], K)
    assert np.array_equal(got.cpu().numpy(), ref)


# --------------------------------------------------- precision envelope, range
def _envelope_case(dev, sigma):
    """q ~ N(0, sigma^2): the rows' largest |score| grows as ~7.9 sigma nats
    at sm_scale = 1/sqrt(192) over unit-variance latents."""
    gen = torch.Generator(device=dev).manual_seed(3)
    n = 6000
    pool = inputs.random_rows(n, gen, dev)
    rng = np.random.default_rng(3)
    T, H, K = 4, 128, 2048
    s = np.stack([rng.choice(n, K, replace=False) for _ in range(T)]).astype(np.int32)
    s[1, 100:] = -1  # a row of 100 keys
    s[2, 8:] = -1    # a row of 8 keys
    g = torch.Generator(device=dev).manual_seed(1003)
    q = (torch.randn((T, H, 576), generator=g, device=dev) * sigma).to(torch.bfloat16)
    out, lse = capi.sparse_mla_decode(q, pool, torch.from_numpy(s).to(dev), 1 / math.sqrt(192))
    torch.cuda.synchronize()
    qb = _q_bits(q)
    ref_out, ref_lse = oracle.sparse_mla_decode(qb, pool.cpu().numpy(), s, 1 / math.sqrt(192))
    qf = oracle.bf16_bits_to_f64(qb)
    smax = 0.0
    for t in range(T):
        nope, rope = oracle.parse_rows(pool.cpu().numpy()[s[t][s[t] >= 0]])
        smax = max(smax, float(np.abs(qf[t] @ np.concatenate([nope, rope], 1).T).max()
                               / math.sqrt(192)))
    return out, lse, ref_out, ref_lse, smax


@pytest.mark.parametrize("sigma", [1.0, 1.5])
def test_precision_envelope_scores_up_to_12_nats(cuda_device, sigma):
    """Keys are rounded once to fp16 (relative 2^-11) and q is bf16 on both
    sides, so a score carries an absolute error of ~1.8e-4 per nat of score;
    the LSE error follows the row's largest scores.  Rows whose scores reach
    8-12 nats (q with 1-1.5x the workloads' spread) meet every tolerance."""
    out, lse, ref_out, ref_lse, smax = _envelope_case(cuda_device, sigma)
    assert 7 <= smax <= 12.5
    compare_out_lse(out, lse, ref_out, ref_lse, where=f"envelope sigma={sigma}")


def test_precision_beyond_the_envelope(cuda_device):
    """With q at 4x the spread the largest scores reach ~31 nats: the LSE
    error still follows the error model (<= 2.5e-4 per nat of the row's
    largest |score|) but leaves the 2e-3 tolerance, which holds while those
    scores stay below ~15 nats; out stays within its tolerances (a weighted
    average of latents, it does not inherit the score offset)."""
    out, lse, ref_out, ref_lse, smax = _envelope_case(cuda_device, 4.0)
    err = np.abs(lse.cpu().numpy() - ref_lse).max()
    assert smax > 25
    assert 2e-3 < err <= 2.5e-4 * smax
    o = out.float().cpu().numpy()
    ob = oracle.compare.bf16_round(ref_out)
    assert np.linalg.norm(o - ob) / np.linalg.norm(ob) <= 1e-2 and np.abs(o - ob).max() <= 2e-2


def test_range_guard_flags_values_the_fp16_keys_cannot_carry(cuda_device):
    """A q or rope value past fp16's range, a group scale whose values would
    overflow fp16 and a nonzero scale below 2^-22 each set SMLA_DEVERR_RANGE;
    in-range inputs (scales up to 65504/448, zero scales) do not."""
    dev = cuda_device
    gen = torch.Generator(device=dev).manual_seed(8)
    pool = inputs.random_rows(64, gen, dev)
    g = torch.Generator(device=dev).manual_seed(1008)
    q = torch.randn((2, 16, 576), generator=g, device=dev).to(torch.bfloat16)
    slots = torch.arange(64, dtype=torch.int32, device=dev).reshape(2, 32)

    def flags(qq, pp):
        capi.get_device_error(clear=True)
        capi.sparse_mla_decode(qq, pp, slots, 0.07)
        torch.cuda.synchronize()
        return capi.get_device_error(clear=True)

    assert flags(q, pool) == 0
    ok = pool.clone()
    sc = ok[:, 512:528].contiguous().view(torch.float32)
    sc[3, 1] = 146.0   # largest values 448 x 146 = 65408: still fp16
    sc[5, 2] = 0.0     # an all-zero group
    ok[:, 512:528] = sc.view(torch.uint8)
    assert flags(q, ok) == 0
    big_q = q.clone()
    big_q[1, 3, 200] = 70000.0
    assert flags(big_q, pool) & capi.DEVERR_RANGE
    for row, col, val in ((7, 0, 150.0), (40, 3, 1e-8)):
        bad = pool.clone()
        sc = bad[:, 512:528].contiguous().view(torch.float32)
        sc[row, col] = val
        bad[:, 512:528] = sc.view(torch.uint8)
        assert flags(q, bad) & capi.DEVERR_RANGE, (row, col, val)
    rope = pool.clone()
    r = rope[:, 528:656].contiguous().view(torch.bfloat16)
    r[20, 5] = float("inf")
    rope[:, 528:656] = r.view(torch.uint8)
    assert flags(q, rope) & capi.DEVERR_RANGE
