"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory at call time -- code running
inside CUDA stream capture (where cudaMalloc is not allowed) or a host that
forbids device allocation after start-up -- so they cannot hand
smla_sparse_mla_decode the workspace it needs for its split-K partials.
smla_sparse_mla_decode_noalloc keeps that scratch in a device array the
library owns.  This file is collected last so that a failure here leaves
every other test already run."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.compare import LSE_ABS, OUT_MAX_ABS, OUT_REL_L2, compare_out_lse
from sparse_mla_decode_dcp_gb300 import capi, inputs


def _within_tolerance(out, lse, ref_out, ref_lse):
    assert torch.equal(torch.isneginf(lse), torch.isneginf(ref_lse))
    fin = torch.isfinite(ref_lse)
    assert (lse[fin] - ref_lse[fin]).abs().max().item() <= LSE_ABS
    o, r = out.double(), ref_out.double()
    assert ((o - r).norm() / r.norm()).item() <= OUT_REL_L2
    assert (o - r).abs().max().item() <= OUT_MAX_ABS


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_device):
    dev = cuda_device
    lib = capi.load()
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    n = 6000
    pool = inputs.random_rows(n, gen, dev)
    g = torch.Generator(device=dev).manual_seed(1077)
    T, H, K = 4, 128, 2048  # few rows: the split-K path, so the scratch is used
    need = capi.decode_workspace_size(T, H, K)
    assert 0 < need <= capi.NOALLOC_SCRATCH_BYTES
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(77)
    s = np.stack([rng.choice(n, K, replace=False) for _ in range(T)]).astype(np.int32)
    s[1, rng.choice(K, 700, replace=False)] = -1
    s[3] = -1  # an empty row: (0, -inf)
    slots = torch.from_numpy(s).to(dev)
    scale = 1.0 / math.sqrt(192.0)
    ref_out, ref_lse = capi.sparse_mla_decode(
        q, pool, slots, scale, workspace=torch.zeros(need, dtype=torch.uint8, device=dev))
    torch.cuda.synchronize()
    for _ in range(2):  # the second call reuses the scratch the first one left
        out = torch.full((T, H, 512), 7, dtype=torch.bfloat16, device=dev)
        lse = torch.full((T, H), 7.0, dtype=torch.float32, device=dev)
        st = lib.smla_sparse_mla_decode_noalloc(
            q.data_ptr(), pool.data_ptr(), n, slots.data_ptr(), T, H, K, ctypes.c_float(scale),
            out.data_ptr(), lse.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == capi.SMLA_OK, capi.status_string(st)
        torch.cuda.synchronize()
        _within_tolerance(out, lse, ref_out, ref_lse)
        # the same kernel on the same inputs, combining its split-K partials
        # in the same fixed order: the results agree bit for bit, so a scratch
        # layout mistake cannot hide inside the tolerance
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
        assert torch.all(out[3].view(torch.int16) == 0)


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_device):
    lib = capi.load()
    T, H, K = 200, 128, 4096
    assert capi.decode_workspace_size(T, H, K) > capi.NOALLOC_SCRATCH_BYTES
    fake = 0x10000  # never dereferenced: the size check comes first
    st = lib.smla_sparse_mla_decode_noalloc(fake, fake, 10, fake, T, H, K, ctypes.c_float(0.07),
                                            fake, fake, None)
    assert st == capi.SMLA_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_replays_in_cuda_graph(cuda_device):
    """The case the entry point exists for: the call captured in a CUDA graph
    (nothing allocated inside the capture; the reset of its scratch counters
    becomes a memset node), replayed for two different top-k draws written
    into the same input buffer: each replay bit-equal to the workspace entry
    point on that draw and within the oracle's tolerance."""
    dev = cuda_device
    lib = capi.load()
    gen = torch.Generator(device=dev)
    gen.manual_seed(78)
    n = 5000
    pool = inputs.random_rows(n, gen, dev)
    g = torch.Generator(device=dev).manual_seed(1078)
    T, H, K = 3, 128, 2048  # few rows: split-K through the library's scratch
    need = capi.decode_workspace_size(T, H, K)
    assert 0 < need <= capi.NOALLOC_SCRATCH_BYTES
    q = torch.randn((T, H, 576), generator=g, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(78)
    draws = [np.stack([rng.choice(n, K, replace=False) for _ in range(T)]).astype(np.int32)
             for _ in range(2)]
    draws[1][2, rng.choice(K, 1500, replace=False)] = -1
    slots = torch.from_numpy(draws[0]).to(dev)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(192.0)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))

    def call():
        st = lib.smla_sparse_mla_decode_noalloc(
            q.data_ptr(), pool.data_ptr(), n, slots.data_ptr(), T, H, K, ctypes.c_float(scale),
            out.data_ptr(), lse.data_ptr(), ctypes.c_void_p(s.cuda_stream))
        assert st == capi.SMLA_OK, capi.status_string(st)

    with torch.cuda.stream(s):
        call()  # warm-up: the scratch address and the kernel's attributes, outside the capture
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            call()
    torch.cuda.synchronize()
    q_bits = q.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)
    for d in draws:
        slots.copy_(torch.from_numpy(d).to(dev))
        out.fill_(7)
        lse.fill_(7.0)
        graph.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = capi.sparse_mla_decode(
            q, pool, slots, scale, workspace=torch.zeros(need, dtype=torch.uint8, device=dev))
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
        o, l = oracle.sparse_mla_decode(q_bits, pool.cpu().numpy(), d, scale)
        compare_out_lse(out, lse, o, l, where="noalloc graph replay")
