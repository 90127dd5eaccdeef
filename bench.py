"""Benchmark: sparse-MLA decode query-tokens/s under DCP on GB300.

One step = the whole hot path over one decode batch of the DCP=4 long-context
workload (64 requests x 1 query token, H=128 gathered heads, top-k 2048, four
simulated shards): per shard filter+convert and sparse MLA decode, then the
LSE merge of the four partials.  `--path fused` (default) runs the step as one
launch (conversion, decode and merge fused); `--path pipeline` as the 2D+1
launches of the three C-ABI calls.  Both are timed; the JSON line reports the
chosen one as `value` and both under `paths`.  Inputs are resident in HBM when the timed
region starts; L2 is flushed (a 256 MiB write) before every timed step, outside
the step's CUDA events.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle instead (the reference arm of this build), on the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA decode query-tokens/s and % roofline (H=128, topk=2048, DCP=4)"
UNIT = "query-tokens/s"
DEFAULT_WORKLOAD = "dcp4_long"
FLUSH_BYTES = 256 << 20
QK_DIM, V_DIM, ROW_BYTES = 576, 512, 656
HOST_CHUNKS = 4  # row groups of the host-buffer step (fastest of 1-8 on dcp4_long)
# hashed to decide whether a committed ncu traffic figure still applies
DECODE_SOURCES = ["sparse_mla_decode_dcp_gb300/csrc/smla_decode.cu",
                  "sparse_mla_decode_dcp_gb300/csrc/smla_sm100.cuh"]
KERNEL_SOURCES = {
    "smla_dcp_sparse_mla_decode_fused": DECODE_SOURCES,
    "smla_sparse_mla_decode": DECODE_SOURCES,
    "smla_dcp_dense_mla_decode": DECODE_SOURCES,
    "smla_dcp_filter_convert_index": ["sparse_mla_decode_dcp_gb300/csrc/smla_index.cu"],
    "smla_dcp_lse_merge": ["sparse_mla_decode_dcp_gb300/csrc/smla_merge.cu"],
    "smla_topk_select": ["sparse_mla_decode_dcp_gb300/csrc/smla_topk.cu"],
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--path", default="fused", choices=["fused", "pipeline"],
                   help="fused: one launch per step; pipeline: D x convert + D x decode + merge")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-aux", action="store_true",
                   help="time the chosen path only: no warm-up or timing of the other path, "
                        "per-launch decode times, e2e or CPU baseline (profiling runs)")
    p.add_argument("--cpu-sample-tokens", type=int, default=64)
    return p.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------ helpers
def algorithmic_units(step):
    """Valid (non -1) slots per shard: the units the decode roofline counts."""
    import torch
    step.run()
    torch.cuda.synchronize()
    return [int(v.sum().item()) for v in step.valid_count]


def source_sha256(sources=DECODE_SOURCES) -> str:
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, src), "rb") as g:
            h.update(g.read())
    return h.hexdigest()


def decode_source_sha256() -> str:
    return source_sha256(DECODE_SOURCES)


def profile_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    profiles/<kernel>_<workload>.md, if that summary was taken on the
    kernel's source as it is now (its `source_sha256:` line, the hash of
    KERNEL_SOURCES[kernel]); else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            m = re.match(r"^\s*-?\s*`?([a-z_0-9]+)`?\s*:\s*`?([^`\s]+)`?", line)
            if m:
                fields.setdefault(m.group(1), m.group(2))
    if kernel not in KERNEL_SOURCES or fields.get("source_sha256") != source_sha256(
            KERNEL_SOURCES[kernel]):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def blas_threads():
    """Threads the BLAS library numpy loaded will use (queried from the
    library itself), or None when it cannot be asked."""
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            libs = {line.split()[-1] for line in f if "openblas" in line.lower() and ".so" in line}
    except OSError:
        return None
    for path in sorted(libs):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for name in ("openblas_get_num_threads", "openblas_get_num_threads64_",
                     "scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads"):
            fn = getattr(lib, name, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    return None


def cpu_baseline(wl, sample_tokens: int, min_seconds: float = 10.0, max_passes: int = 200):
    """The float64 oracle as it stands, timed on this host on a bounded sample
    of the same workload: the first `sample_tokens` query rows, every shard's
    convert + decode, then the merge -- repeated until at least `min_seconds`
    of CPU work have been timed (one pass of the full workload takes well
    under a second)."""
    import oracle
    import torch
    n = min(sample_tokens, wl.T)
    q_bits = wl.q[:n].detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)
    pools = [s.pool.cpu().numpy() for s in wl.shards]
    passes = 0
    t0 = time.perf_counter()
    while True:
        outs, lses = [], []
        for d, s in enumerate(wl.shards):
            sl, _ = oracle.dcp_filter_convert_index(wl.req_id[:n], s.block_table, wl.topk[:n],
                                                    wl.D, d, wl.spec.block_size,
                                                    wl.spec.interleave)
            o, l = oracle.sparse_mla_decode(q_bits, pools[d], sl, wl.spec.sm_scale)
            outs.append(o)
            lses.append(l)
        oracle.lse_merge(outs, lses)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            break
    threads = blas_threads()
    return {"value": passes * n / dt, "unit": UNIT,
            "cores": threads if threads is not None else (os.cpu_count() or 1),
            "kind": "oracle", "host_cores": os.cpu_count(), "blas_threads": threads,
            "cpu_model": cpu_model(),
            "sample": f"first {n} of {wl.T} query rows of {wl.spec.name}, all {wl.D} shards "
                      f"(convert + decode) + merge, float64 numpy, {passes} passes; {dt:.2f} s"}


def cpu_baseline_single_thread(workload: str, seed: int, sample_tokens: int = 2,
                               min_seconds: float = 8.0):
    """The same oracle timing in a process of its own whose BLAS may use one
    thread only (OMP/OpenBLAS/MKL thread counts set to 1 before numpy loads).
    The child builds the workload on the CPU: the structure (contexts, top-k
    ids, block tables) comes from the same seeded draws, the values from the
    CPU generator -- the oracle's cost does not depend on them."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, bench\n"
            "from sparse_mla_decode_dcp_gb300 import inputs\n"
            f"wl = inputs.make_workload({workload!r}, seed={seed}, device='cpu')\n"
            f"print(json.dumps(bench.cpu_baseline(wl, {sample_tokens}, {min_seconds})))\n")
    try:
        p = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=600)
        return json.loads(p.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"unavailable": f"single-thread oracle run failed: {type(e).__name__}"}


def workload_config(wl, args, world: int) -> dict:
    """The `config` object both arms print for the same workload."""
    return {"workload": args.workload, "path": args.path, "T": wl.T, "H": wl.H, "K": wl.K,
            "D": wl.D, "interleave": wl.spec.interleave, "block_size": wl.spec.block_size,
            "requests": wl.spec.num_reqs, "cached_tokens": int(sum(int(c) for c in wl.ctx)),
            "l2": "flushed before every step (256 MiB write, outside the events)",
            "parallelism": f"replicas x{world}" if world > 1 else
                           "single GPU, D shards simulated as D pools"}


# ------------------------------------------------------------ multi-rank
def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank float over the default process group (identity when
    no group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(tokens_per_step: int, steps: int, total_ms_this_rank: float,
                         world: int, device=None):
    """Whole-job value: every rank processed `tokens_per_step * steps` query
    tokens; the job took the slowest rank's time.  Returns (value, ms_per_step)."""
    total_ms = max_over_ranks(total_ms_this_rank, device)
    return world * tokens_per_step * steps / (total_ms / 1e3), total_ms / steps


# ------------------------------------------------------------ GPU arm
def _timed_steps(fn, n, flush, stream):
    """Per-step device times (ms) of `fn`, L2 flushed before each step
    outside the step's CUDA events."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for i in range(n):
        flush.fill_(1)
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def _pipeline_launch_ms(step, wl, n, flush, stream):
    """Per-launch times of the three kernels inside the 2D+1 launch pipeline
    (events on the launching stream around each launch; L2 flushed before
    each step).  Returns (index [n, D], decode [n, D], merge [n]) in ms."""
    import torch

    from sparse_mla_decode_dcp_gb300 import capi
    D = wl.D
    idx, dec, mrg = [], [], []
    for _ in range(n):
        flush.fill_(1)
        ev_i, ev_d = [], []
        for d in range(D):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            capi.dcp_filter_convert_index(
                step.req_id, step.block_tables[d], step.topk, D, d, wl.spec.block_size,
                interleave=wl.spec.interleave, bt_width=step.bt_widths[d],
                local_slots=step.local_slots[d],
                valid_count=step.valid_count[d])
            ev[1].record(stream)
            capi.sparse_mla_decode(step.q, step.pools[d], step.local_slots[d], wl.spec.sm_scale,
                                   out=step.part_out[d], lse=step.part_lse[d],
                                   workspace=step.workspace)
            ev[2].record(stream)
            ev_i.append((ev[0], ev[1]))
            ev_d.append((ev[1], ev[2]))
        em = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        em[0].record(stream)
        capi.dcp_lse_merge(step.part_out, step.part_lse, out=step.out, lse=step.lse)
        em[1].record(stream)
        torch.cuda.synchronize()
        idx.append([a.elapsed_time(b) for a, b in ev_i])
        dec.append([a.elapsed_time(b) for a, b in ev_d])
        mrg.append(em[0].elapsed_time(em[1]))
    return np.array(idx), np.array(dec), np.array(mrg)


def _e2e_overlapped(step, wl, q_host, n, stream, sets=4):
    """End to end as a serving loop runs it: every step copies its q and
    top-k ids in from pinned host memory and its out + lse back, through the
    public API, with step k's input copies (one copy stream) and step k - 1's
    output copies (another) overlapping step k - 1's and step k's compute on
    two device buffer sets.  The steps cycle through `sets` different top-k
    draws of the workload's contexts, so a step's cache rows were last read
    `sets` steps earlier (sets x ~80 MB of rows, more than L2 holds); no L2
    flush inside the loop.  Returns (ms per step, h2d bytes, d2h bytes)."""
    import torch

    from sparse_mla_decode_dcp_gb300 import capi, inputs
    dev = step.q.device
    spec = wl.spec
    topk_hosts = [torch.from_numpy(inputs.draw_topk(spec, wl.ctx, np.random.default_rng(1000 + k)))
                  .pin_memory() for k in range(sets)]
    out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    lse_host = torch.empty(step.lse.shape, dtype=step.lse.dtype).pin_memory()
    bufs = [(step.q, step.topk, step.out, step.lse),
            (torch.empty_like(step.q), torch.empty_like(step.topk), torch.empty_like(step.out),
             torch.empty_like(step.lse))]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}

    def run(count):
        for k in range(count):
            j = k % 2
            q, topk, out, lse = bufs[j]
            if k >= 2:
                h2d_s.wait_event(ev["done"][j])  # step k - 2 has read this set
            with torch.cuda.stream(h2d_s):
                q.copy_(q_host, non_blocking=True)
                topk.copy_(topk_hosts[k % sets], non_blocking=True)
                ev["in"][j].record(h2d_s)
            stream.wait_event(ev["in"][j])
            if k >= 2:
                stream.wait_event(ev["out"][j])  # step k - 2's results are out
            capi.dcp_sparse_mla_decode_fused(
                q, step.req_id, topk, step.pools, step.block_tables, spec.block_size,
                spec.sm_scale, interleave=spec.interleave, bt_widths=step.bt_widths,
                out=out, lse=lse, workspace=step.workspace, stream=stream)
            ev["done"][j].record(stream)
            d2h_s.wait_event(ev["done"][j])
            with torch.cuda.stream(d2h_s):
                out_host.copy_(out, non_blocking=True)
                lse_host.copy_(lse, non_blocking=True)
                ev["out"][j].record(d2h_s)

    run(4)  # warm-up
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    h2d_s.wait_event(t0)
    d2h_s.wait_event(t0)
    run(n)
    # the end: every stream's work of the n steps
    d2h_s.wait_stream(stream)
    d2h_s.wait_stream(h2d_s)
    t1.record(d2h_s)
    torch.cuda.synchronize()
    h2d = q_host.numel() * q_host.element_size() + topk_hosts[0].numel() * 4
    d2h = out_host.numel() * out_host.element_size() + lse_host.numel() * 4
    return t0.elapsed_time(t1) / n, h2d, d2h


def _hbm_roofline(kernel, launch_ms, nbytes, peaks, unit_note, workload):
    """HBM roofline of a memory-bound kernel: algorithmic bytes per launch
    over its mean launch time, against the measured copy bandwidth."""
    achieved = nbytes / (launch_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": profile_traffic(kernel, workload),
            "kernel": kernel,
            "launch_us": launch_ms * 1e3, "algorithmic_bytes_per_launch": nbytes,
            "bytes": unit_note,
            "peak_source": f"{peaks['source']} MEASURED_PEAKS.json copy bandwidth"}


def _roofline(kernel, launch_ms, keys_per_launch, H, peaks, workload):
    flop_per_key = 2.0 * H * (QK_DIM + V_DIM)
    flops = flop_per_key * keys_per_launch
    nbytes = ROW_BYTES * keys_per_launch
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if flop_per_key / ROW_BYTES >= ridge:
        roof = {"bound": "tensor", "achieved": flops / (launch_ms * 1e-3) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": nbytes / (launch_ms * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profile_traffic(kernel, workload)
    roof.update({
        "kernel": kernel,
        "peak_source": f"{peaks['source']} MEASURED_PEAKS.json burst figure"
                       + ("; fp16 MMA nominal rate = bf16" if roof["bound"] == "tensor" else ""),
        "launch_us": launch_ms * 1e3,
        "algorithmic_flops_per_launch": flops,
        "algorithmic_bytes_per_launch": nbytes,
        "achieved_hbm_gbs": nbytes / (launch_ms * 1e-3) / 1e9,
    })
    return roof


def _dense_path(step, wl, n, flush, stream, peaks, workload):
    """The dense decode (every cached position of each row's causal context,
    merged over the D pools in one launch) on the same caches."""
    import torch

    from sparse_mla_decode_dcp_gb300 import capi
    dev = step.q.device
    S = wl.spec.tokens_per_req
    ctx = torch.from_numpy(wl.ctx.astype(np.int32)).to(dev)
    max_ctx = int(wl.ctx.max())
    n_ws = capi.dense_decode_workspace_size(wl.T, wl.H, max_ctx, wl.D, wl.spec.interleave, -1)
    ws = torch.zeros(n_ws, dtype=torch.uint8, device=dev) if n_ws else None
    out = torch.empty_like(step.out)
    lse = torch.empty_like(step.lse)

    def run():
        capi.dcp_dense_mla_decode(step.q, ctx, max_ctx, S, step.pools, step.block_tables,
                                  wl.spec.block_size, wl.spec.sm_scale,
                                  interleave=wl.spec.interleave, bt_widths=step.bt_widths,
                                  out=out, lse=lse, workspace=ws)
    run()
    ms = float(np.mean(_timed_steps(run, n, flush, stream)))
    keys = int(sum(int(c) - S + s + 1 for c in wl.ctx for s in range(S)))
    roof = _roofline("smla_dcp_dense_mla_decode", ms, keys, wl.H, peaks, workload)
    roof["keys_per_launch"] = keys
    del ws
    return {"ms_per_step": ms, "value": wl.T / (ms * 1e-3), "launches_per_step": 1,
            "roofline": roof}


def _topk_path(wl, n, flush, stream, peaks, dev, workload):
    """Global top-K of synthetic indexer scores: one fp32 score per cached
    position of each row (seeded normal draws), K = the workload's top-k."""
    import torch

    from sparse_mla_decode_dcp_gb300 import capi
    S = wl.spec.tokens_per_req
    L = int(wl.ctx.max())
    gen = torch.Generator(device=dev).manual_seed(12345)
    scores = torch.randn((wl.T, L), generator=gen, device=dev, dtype=torch.float32)
    n_cand_np = np.array([int(wl.ctx[t // S]) - S + t % S + 1 for t in range(wl.T)], np.int32)
    n_cand = torch.from_numpy(n_cand_np).to(dev)
    ids = torch.empty((wl.T, wl.K), dtype=torch.int32, device=dev)
    ws_bytes = capi.topk_select_workspace_size(wl.T, L, wl.K)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    def run():
        st = capi.load().smla_topk_select(scores.data_ptr(), scores.stride(0), L,
                                          n_cand.data_ptr(), wl.T, wl.K, 1, 0, 1, ids.data_ptr(),
                                          None, ws.data_ptr(), ws_bytes, int(stream.cuda_stream))
        assert st == capi.SMLA_OK, st
    run()
    ms = float(np.mean(_timed_steps(run, n, flush, stream)))
    nbytes = 4 * int(n_cand_np.sum()) + 4 * wl.T * wl.K
    # rows longer than a chunk: one launch over the chunks, one merging them
    return {"ms_per_step": ms, "launches_per_step": 2 if ws_bytes else 1,
            "roofline": _hbm_roofline("smla_topk_select", ms, nbytes, peaks,
                                      "4 B per candidate score read + 4 B per id written",
                                      workload)}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from sparse_mla_decode_dcp_gb300 import capi, inputs
    from sparse_mla_decode_dcp_gb300.pipeline import DcpDecodeStep

    rank, world, local_rank = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    capi.load()

    wl = inputs.make_workload(args.workload, seed=args.seed + rank, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = DcpDecodeStep(wl, device=dev)
    units = algorithmic_units(step)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    T, H, K, D = wl.T, wl.H, wl.K, wl.D
    paths = {"fused": (step.run_fused, 1), "pipeline": (step.run, step.launches_per_step)}
    main_fn, main_launches = paths[args.path]
    alt_name = "pipeline" if args.path == "fused" else "fused"
    alt_fn, _ = paths[alt_name]

    # The clock sampler starts first; the warm-up steps then run directly
    # before the timed region, since after a GPU idle period of a fraction of a
    # second the first launch takes two to three times a steady step.
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.25)
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        main_fn()
        if not args.no_aux:
            flush.fill_(1)
            alt_fn()
    torch.cuda.synchronize()

    # Timed region: exactly `steps` steps of the reported path.
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    step_ms = _timed_steps(main_fn, args.steps, flush, stream)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    value, ms_per_step = aggregate_throughput(T, args.steps, float(sum(step_ms)), world, dev)

    total_keys = sum(units)
    peaks = load_peaks()
    roofline_us = max(
        2.0 * H * (QK_DIM + V_DIM) * total_keys / (peaks["bf16_tflops"] * 1e12),
        ROW_BYTES * total_keys / (peaks["hbm_gbs"] * 1e9)) * 1e6
    if args.no_aux:
        # profiling run: the chosen path only, one reduced line
        roof = _roofline("smla_dcp_sparse_mla_decode_fused" if args.path == "fused" else
                         "smla_sparse_mla_decode", ms_per_step / (1 if args.path == "fused" else D),
                         total_keys / (1 if args.path == "fused" else D), H, peaks, args.workload)
        roof["roofline_us_per_step"] = roofline_us
        if rank == 0:
            print(json.dumps({
                "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
                "higher_is_better": True, "config": {"workload": args.workload, "path": args.path},
                "roofline": roof, "aux": "skipped (--no-aux)",
                "gpu_launches": args.steps * main_launches, "clocks": clocks}), flush=True)
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    # The other form of the same step, and per-launch decode times.
    n_aux = max(10, min(args.steps, 50))
    alt_ms = float(np.mean(_timed_steps(alt_fn, n_aux, flush, stream)))
    idx_ms, dec_ms, mrg_ms = _pipeline_launch_ms(step, wl, n_aux, flush, stream)
    if args.path == "fused":
        roof = _roofline("smla_dcp_sparse_mla_decode_fused", ms_per_step, total_keys, H, peaks,
                         args.workload)
        roof["launches_per_step"] = 1
    else:
        roof = _roofline("smla_sparse_mla_decode", float(dec_ms.mean()), total_keys / D, H, peaks,
                         args.workload)
        roof["launches_per_step"] = D
    roof["valid_slots_per_shard"] = units
    roof["roofline_us_per_step"] = roofline_us
    pipeline_ms = alt_ms if args.path == "fused" else ms_per_step
    fused_ms = ms_per_step if args.path == "fused" else alt_ms
    per_shard_roof = _roofline("smla_sparse_mla_decode", float(dec_ms.mean()), total_keys / D, H,
                               peaks, args.workload)
    dense_path = _dense_path(step, wl, max(3, min(n_aux, 10)), flush, stream, peaks,
                             args.workload)
    topk_path = _topk_path(wl, n_aux, flush, stream, peaks, dev, args.workload)
    # index: read the top-k ids and write the slots (4 B each per entry),
    # read the row's request id and write its valid count
    index_roof = _hbm_roofline("smla_dcp_filter_convert_index", float(idx_ms.mean()),
                               8 * T * K + 8 * T, peaks,
                               "8 B per top-k entry (id in, slot out) + 8 B per row",
                               args.workload)
    # merge: D partial rows of 512 bf16 + fp32 lse in, one merged row out
    merge_roof = _hbm_roofline("smla_dcp_lse_merge", float(mrg_ms.mean()),
                               (D + 1) * T * H * (2 * V_DIM + 4), peaks,
                               "(D + 1) x (1024 B out row + 4 B lse) per (token, head)",
                               args.workload)

    # End to end through the public API with host buffers: every step copies
    # q and the top-k ids from pinned host memory and reads out + lse back.
    q_host = wl.q.detach().cpu().pin_memory()
    topk_host = torch.from_numpy(wl.topk).pin_memory()
    out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    lse_host = torch.empty(step.lse.shape, dtype=step.lse.dtype).pin_memory()
    h2d = q_host.numel() * q_host.element_size() + topk_host.numel() * 4
    d2h = out_host.numel() * out_host.element_size() + lse_host.numel() * 4

    def serial_step():
        step.q.copy_(q_host, non_blocking=True)
        step.topk.copy_(topk_host, non_blocking=True)
        main_fn()
        out_host.copy_(step.out, non_blocking=True)
        lse_host.copy_(step.lse, non_blocking=True)

    if args.path == "fused":
        # the library's host-buffer entry point: row groups whose copies in,
        # decode and copies back overlap one another
        def e2e_step():
            step.run_fused_from_host(q_host, topk_host, out_host, lse_host, chunks=HOST_CHUNKS)
    else:
        e2e_step = serial_step
    n_e2e = max(3, min(args.steps, 100))
    for _ in range(3):  # warm after the host-side set-up above
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(float(np.mean(_timed_steps(e2e_step, n_e2e, flush, stream))), dev)
    for _ in range(3):
        serial_step()
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(float(np.mean(_timed_steps(serial_step, n_e2e, flush, stream))),
                               dev)
    ov_ms, ov_h2d, ov_d2h = _e2e_overlapped(step, wl, q_host, max(8, min(args.steps, 200)), stream)
    ov_ms = max_over_ranks(ov_ms, dev)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16xf16->f32 (MMA), f32 softmax", "data": "synthetic",
        "config": workload_config(wl, args, world),
        "roofline": roof,
        "paths": {
            "fused": {"ms_per_step": fused_ms, "value": world * T / (fused_ms * 1e-3),
                      "launches_per_step": 1},
            "pipeline": {"ms_per_step": pipeline_ms, "value": world * T / (pipeline_ms * 1e-3),
                         "launches_per_step": step.launches_per_step,
                         "decode_launch_us": [float(x) * 1e3 for x in dec_ms.mean(axis=0)],
                         "decode_roofline": per_shard_roof,
                         "index_launch_us": [float(x) * 1e3 for x in idx_ms.mean(axis=0)],
                         "index_roofline": index_roof,
                         "merge_launch_us": float(mrg_ms.mean()) * 1e3,
                         "merge_roofline": merge_roof},
            "dense": dense_path,
            "topk": topk_path,
        },
        "e2e": {"value": world * T / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": (f"smla_dcp_sparse_mla_decode_fused_host, {HOST_CHUNKS} row groups: "
                        "q and top-k ids in from pinned host memory, out and lse back"
                        if args.path == "fused" else
                        "copies in, the step's launches, copies back, in stream order")},
        "e2e_serial": {"value": world * T / (serial_ms * 1e-3), "unit": UNIT,
                       "ms_per_step": serial_ms,
                       "how": "the same copies and the step in stream order, nothing overlapped"},
        "e2e_overlapped": {"value": world * T / (ov_ms * 1e-3), "unit": UNIT,
                           "h2d_bytes_per_step": ov_h2d, "d2h_bytes_per_step": ov_d2h,
                           "ms_per_step": ov_ms,
                           "how": "fused path; step k's input copies and step k-1's output "
                                  "copies overlap compute on two buffer sets and two copy "
                                  "streams; steps cycle through 4 top-k draws (no L2 flush)"},
        "gpu_launches": args.steps * main_launches,
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, args.cpu_sample_tokens)
        result["cpu_baseline"]["single_thread"] = cpu_baseline_single_thread(args.workload,
                                                                             args.seed)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


# ------------------------------------------------------------ reference arm
def run_reference(args):
    """The reference arm of this build: the float64 CPU oracle, timed as it
    stands on this host's cores, on the same workload and metric.  Each step
    is a bounded sample of the workload's query rows (all D shards' convert +
    decode, then the merge), sized from a measured per-row time so that the
    whole --steps/--warmup run stays within about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from sparse_mla_decode_dcp_gb300 import inputs
    wl = inputs.make_workload(args.workload, seed=args.seed, device="cpu")
    probe = cpu_baseline(wl, 2)
    per_row_s = 1.0 / probe["value"]
    budget_s = 120.0
    n = int(budget_s / (max(1, args.steps + args.warmup) * per_row_s))
    n = max(1, min(wl.T, n))
    for _ in range(args.warmup):
        cpu_baseline(wl, n)
    times = []
    b = None
    for _ in range(args.steps):
        b = cpu_baseline(wl, n)
        times.append(n / b["value"])
    value = n * len(times) / sum(times)
    b["value"] = value
    b["sample"] = f"{n} query rows per step: " + b["sample"]
    result = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(wl, args, world),
        "cpu_baseline": b,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
