"""One DCP decode step over D simulated shards on one GPU.

Per shard d: filter + convert the global top-k to shard d's slots, then
sparse MLA decode over shard d's pool; finally the LSE-weighted merge of the
D partials (the single-GPU stand-in for the cross-rank LSE all-gather and
output reduce-scatter of "[eldritch] attention: support DCP in SM120
FlashInfer sparse MLA", Why / Scope).

Every buffer is allocated once in the constructor, so ``run`` launches
2*D + 1 kernels and allocates nothing.
"""
from __future__ import annotations

from typing import List, Optional

import torch

from . import capi
from .inputs import Workload


class DcpDecodeStep:
    def __init__(self, wl: Workload, device="cuda", stream: Optional[torch.cuda.Stream] = None):
        self.wl = wl
        self.device = torch.device(device)
        self.stream = stream
        T, H, K, D = wl.T, wl.H, wl.K, wl.D
        dev = self.device
        self.q = wl.q.to(dev).contiguous()
        self.req_id = torch.from_numpy(wl.req_id).to(dev)
        self.topk = torch.from_numpy(wl.topk).to(dev)
        self.pools: List[torch.Tensor] = [s.pool.to(dev) for s in wl.shards]
        self.block_tables = [torch.from_numpy(s.block_table).to(dev) for s in wl.shards]
        self.bt_widths = [s.width for s in wl.shards]
        self.local_slots = [torch.empty((T, K), dtype=torch.int32, device=dev) for _ in range(D)]
        self.valid_count = [torch.empty((T,), dtype=torch.int32, device=dev) for _ in range(D)]
        self.part_out = [torch.empty((T, H, capi.V_DIM), dtype=torch.bfloat16, device=dev)
                         for _ in range(D)]
        self.part_lse = [torch.empty((T, H), dtype=torch.float32, device=dev) for _ in range(D)]
        self.out = torch.empty((T, H, capi.V_DIM), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.workspace = capi.alloc_decode_workspace(T, H, K, dev)

    @property
    def launches_per_step(self) -> int:
        return 2 * self.wl.D + 1

    def run_shard(self, d: int):
        wl = self.wl
        capi.dcp_filter_convert_index(
            self.req_id, self.block_tables[d], self.topk, wl.D, d, wl.spec.block_size,
            interleave=wl.spec.interleave, bt_width=self.bt_widths[d],
            local_slots=self.local_slots[d],
            valid_count=self.valid_count[d], stream=self.stream)
        capi.sparse_mla_decode(
            self.q, self.pools[d], self.local_slots[d], wl.spec.sm_scale,
            out=self.part_out[d], lse=self.part_lse[d], workspace=self.workspace,
            stream=self.stream)

    def run_fused(self):
        """The same step in one launch (conversion, decode and merge fused)."""
        wl = self.wl
        return capi.dcp_sparse_mla_decode_fused(
            self.q, self.req_id, self.topk, self.pools, self.block_tables,
            wl.spec.block_size, wl.spec.sm_scale, interleave=wl.spec.interleave,
            bt_widths=self.bt_widths,
            out=self.out, lse=self.lse, workspace=self.workspace, stream=self.stream)

    def run_fused_from_host(self, q_host: torch.Tensor, topk_host: torch.Tensor,
                            out_host: torch.Tensor, lse_host: torch.Tensor, chunks: int = 4):
        """The fused step with q and the top-k ids in pinned host memory and
        out/lse returned there: the library copies them in and out through
        this step's device buffers, row groups pipelined."""
        wl = self.wl
        return capi.dcp_sparse_mla_decode_fused_host(
            q_host, topk_host, out_host, lse_host, self.req_id, self.pools, self.block_tables,
            wl.spec.block_size, wl.spec.sm_scale, interleave=wl.spec.interleave,
            bt_widths=self.bt_widths, q_dev=self.q, topk_dev=self.topk, out_dev=self.out,
            lse_dev=self.lse, workspace=self.workspace, chunks=chunks, stream=self.stream)

    def run(self):
        for d in range(self.wl.D):
            self.run_shard(d)
        capi.dcp_lse_merge(self.part_out, self.part_lse, out=self.out, lse=self.lse,
                           stream=self.stream)
        return self.out, self.lse
