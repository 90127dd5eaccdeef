"""Thin Python binding of ``include/smla.h`` (ctypes).

Argument marshalling only: it checks dtypes/devices/contiguity, allocates
outputs with torch when the caller passes none, and hands raw device
pointers plus the current CUDA stream to the C ABI.  Every step of the path
runs in the library's kernels.  Loading fails loudly when ``libsmla.so`` has
not been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple, Union

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsmla.so")

SMLA_OK = 0
SMLA_ERR_INVALID_ARG = 1
SMLA_ERR_UNSUPPORTED = 2
SMLA_ERR_WORKSPACE = 3
SMLA_ERR_CUDA = 4

DEVERR_BLOCK_TABLE = 1
DEVERR_REQ_ID = 2
DEVERR_SLOT_RANGE = 4
DEVERR_TIMEOUT = 8
DEVERR_CONTEXT = 16
DEVERR_RANGE = 32

MAX_HEADS = 128
MAX_DCP = 16
ROW_BYTES = 656
QK_DIM = 576
V_DIM = 512

_c_i32, _c_i64, _c_sz, _c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/smla.h
SIGNATURES = {
    "smla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "smla_get_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "smla_dcp_filter_convert_index": (ctypes.c_int, [
        _c_vp, _c_vp, _c_i64, _c_i32, _c_i32, _c_vp, _c_i32, _c_i32, _c_i32, _c_i32,
        _c_i32, _c_i32, _c_vp, _c_vp, _c_vp]),
    "smla_decode_workspace_size": (_c_sz, [_c_i32, _c_i32, _c_i32]),
    "smla_sparse_mla_decode": (ctypes.c_int, [
        _c_vp, _c_vp, _c_i64, _c_vp, _c_i32, _c_i32, _c_i32, ctypes.c_float, _c_vp,
        _c_vp, _c_vp, _c_sz, _c_vp]),
    "smla_sparse_mla_decode_noalloc": (ctypes.c_int, [
        _c_vp, _c_vp, _c_i64, _c_vp, _c_i32, _c_i32, _c_i32, ctypes.c_float, _c_vp, _c_vp,
        _c_vp]),
    "smla_dcp_sparse_mla_decode_fused": (ctypes.c_int, [
        _c_vp, _c_i32, _c_i32, _c_i32, ctypes.c_float, _c_vp, _c_vp, _c_i32, _c_i32, _c_i32,
        _c_i32, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]),
    "smla_dcp_sparse_mla_decode_fused_host": (ctypes.c_int, [
        _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i32, _c_i32, _c_i32,
        ctypes.c_float, _c_vp, _c_i32, _c_i32, _c_i32, _c_i32, _c_vp, _c_vp, _c_vp, _c_vp,
        _c_vp, _c_vp, _c_sz, _c_i32, _c_vp]),
    "smla_dense_decode_workspace_size": (_c_sz, [_c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                                 _c_i32]),
    "smla_dcp_dense_mla_decode": (ctypes.c_int, [
        _c_vp, _c_i32, _c_i32, _c_i32, ctypes.c_float, _c_vp, _c_i32, _c_i32, _c_i32, _c_i32,
        _c_i32, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz, _c_vp]),
    "smla_topk_select_workspace_size": (_c_sz, [_c_i32, _c_i32, _c_i32]),
    "smla_topk_select": (ctypes.c_int, [
        _c_vp, _c_i64, _c_i32, _c_vp, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_vp, _c_vp,
        _c_vp, _c_sz, _c_vp]),
    "smla_dcp_topk_merge": (ctypes.c_int, [
        _c_vp, _c_vp, _c_i64, _c_i32, _c_i32, _c_i32, _c_vp, _c_vp, _c_vp]),
    "smla_dcp_lse_merge": (ctypes.c_int, [
        _c_vp, _c_vp, _c_i32, _c_i32, _c_i32, _c_vp, _c_vp, _c_vp]),
}

_lib = None


class SmlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Load libsmla.so once (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().smla_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != SMLA_OK:
        raise SmlaError(fn, status)


def _stream_ptr(stream: Optional[torch.cuda.Stream], device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def get_device_error(clear: bool = True) -> int:
    """OR of DEVERR_* bits raised by kernels on the current device."""
    v = ctypes.c_uint32(0)
    _check("smla_get_device_error", load().smla_get_device_error(ctypes.byref(v), int(clear)))
    return int(v.value)


def dcp_filter_convert_index(req_id_per_token: torch.Tensor, block_table: torch.Tensor,
                             topk_global: torch.Tensor, D: int, rank: int,
                             block_size: int, *, interleave: int = 1,
                             bt_width: Optional[int] = None,
                             local_slots: Optional[torch.Tensor] = None,
                             valid_count: Optional[torch.Tensor] = None,
                             with_valid_count: bool = True,
                             stream: Optional[torch.cuda.Stream] = None
                             ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    dev = topk_global.device
    _need(req_id_per_token, "req_id_per_token", torch.int32, dev)
    _need(topk_global, "topk_global", torch.int32, dev)
    if block_table.dtype != torch.int32 or block_table.device != dev or block_table.dim() != 2:
        raise ValueError("block_table must be a 2-D int32 tensor on the top-k device")
    if block_table.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    T, K = topk_global.shape
    if local_slots is None:
        local_slots = torch.empty((T, K), dtype=torch.int32, device=dev)
    _need(local_slots, "local_slots", torch.int32, dev)
    if valid_count is None and with_valid_count:
        valid_count = torch.empty((T,), dtype=torch.int32, device=dev)
    if valid_count is not None:
        _need(valid_count, "valid_count", torch.int32, dev)
    width = block_table.shape[1] if bt_width is None else int(bt_width)
    st = load().smla_dcp_filter_convert_index(
        req_id_per_token.data_ptr(), block_table.data_ptr(), block_table.stride(0),
        width, block_table.shape[0], topk_global.data_ptr(), T, K, D, rank,
        block_size, int(interleave), local_slots.data_ptr(),
        valid_count.data_ptr() if valid_count is not None else None,
        _stream_ptr(stream, dev))
    _check("smla_dcp_filter_convert_index", st)
    return local_slots, valid_count


def decode_workspace_size(T: int, H: int, K: int) -> int:
    return int(load().smla_decode_workspace_size(T, H, K))


def alloc_decode_workspace(T: int, H: int, K: int, device) -> Optional[torch.Tensor]:
    """Zero-filled workspace for smla_sparse_mla_decode (None if none needed)."""
    n = decode_workspace_size(T, H, K)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def sparse_mla_decode(q: torch.Tensor, kv_cache: torch.Tensor, local_slots: torch.Tensor,
                      sm_scale: float, *, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None
                      ) -> Tuple[torch.Tensor, torch.Tensor]:
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(kv_cache, "kv_cache", torch.uint8, dev)
    _need(local_slots, "local_slots", torch.int32, dev)
    T, H, Dq = q.shape
    if Dq != QK_DIM:
        raise ValueError(f"q last dim must be {QK_DIM}")
    if kv_cache.dim() != 2 or kv_cache.shape[1] != ROW_BYTES:
        raise ValueError(f"kv_cache must be [num_slots, {ROW_BYTES}] uint8")
    K = local_slots.shape[1]
    if local_slots.shape[0] != T:
        raise ValueError("local_slots rows must equal q tokens")
    if out is None:
        out = torch.empty((T, H, V_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    if workspace is None:
        workspace = alloc_decode_workspace(T, H, K, dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().smla_sparse_mla_decode(
        q.data_ptr(), kv_cache.data_ptr(), kv_cache.shape[0], local_slots.data_ptr(),
        T, H, K, float(sm_scale), out.data_ptr(), lse.data_ptr(), ws_ptr, ws_bytes,
        _stream_ptr(stream, dev))
    _check("smla_sparse_mla_decode", st)
    return out, lse


NOALLOC_SCRATCH_BYTES = 32 << 20


def sparse_mla_decode_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, local_slots: torch.Tensor,
                              sm_scale: float, *, out: Optional[torch.Tensor] = None,
                              lse: Optional[torch.Tensor] = None,
                              stream: Optional[torch.cuda.Stream] = None
                              ) -> Tuple[torch.Tensor, torch.Tensor]:
    """smla_sparse_mla_decode without a workspace argument: the split-K scratch
    is the library's own device array, for callers that cannot allocate device
    memory (see include/smla.h).  Such callers pass `out` and `lse`; when
    omitted they are allocated here for convenience."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(kv_cache, "kv_cache", torch.uint8, dev)
    _need(local_slots, "local_slots", torch.int32, dev)
    T, H, Dq = q.shape
    K = local_slots.shape[1]
    if Dq != QK_DIM or local_slots.shape[0] != T:
        raise ValueError("q must be [T, H, 576] and local_slots [T, K]")
    if kv_cache.dim() != 2 or kv_cache.shape[1] != ROW_BYTES:
        raise ValueError(f"kv_cache must be [num_slots, {ROW_BYTES}] uint8")
    if out is None:
        out = torch.empty((T, H, V_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    st = load().smla_sparse_mla_decode_noalloc(
        q.data_ptr(), kv_cache.data_ptr(), kv_cache.shape[0], local_slots.data_ptr(),
        T, H, K, float(sm_scale), out.data_ptr(), lse.data_ptr(), _stream_ptr(stream, dev))
    _check("smla_sparse_mla_decode_noalloc", st)
    return out, lse


def dcp_sparse_mla_decode_fused(q: torch.Tensor, req_id_per_token: torch.Tensor,
                                topk_global: torch.Tensor, kv_caches: Sequence[torch.Tensor],
                                block_tables: Sequence[torch.Tensor], block_size: int,
                                sm_scale: float, *, interleave: int = 1,
                                bt_widths: Optional[Sequence[int]] = None,
                                out: Optional[torch.Tensor] = None,
                                lse: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None,
                                stream: Optional[torch.cuda.Stream] = None
                                ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Filter+convert, decode and merge of D shards in one launch; returns the
    merged (out, lse)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(req_id_per_token, "req_id_per_token", torch.int32, dev)
    _need(topk_global, "topk_global", torch.int32, dev)
    D = len(kv_caches)
    if D != len(block_tables) or D < 1:
        raise ValueError("need one block table per KV pool (>= 1)")
    T, H, Dq = q.shape
    K = topk_global.shape[1]
    if Dq != QK_DIM or topk_global.shape[0] != T:
        raise ValueError("q must be [T, H, 576] and topk [T, K]")
    num_reqs = None
    for kv, bt in zip(kv_caches, block_tables):
        _need(kv, "kv_caches[d]", torch.uint8, dev)
        if kv.dim() != 2 or kv.shape[1] != ROW_BYTES:
            raise ValueError(f"kv_caches[d] must be [num_slots, {ROW_BYTES}] uint8")
        if bt.dtype != torch.int32 or bt.device != dev or bt.dim() != 2 or bt.stride(1) != 1:
            raise ValueError("block_tables[d] must be 2-D int32 with contiguous rows")
        num_reqs = bt.shape[0] if num_reqs is None else min(num_reqs, bt.shape[0])
    if out is None:
        out = torch.empty((T, H, V_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    if workspace is None:
        workspace = alloc_decode_workspace(T, H, K, dev)
    widths = [bt.shape[1] for bt in block_tables] if bt_widths is None else list(bt_widths)
    pools = (ctypes.c_void_p * D)(*[kv.data_ptr() for kv in kv_caches])
    nslots = (ctypes.c_int64 * D)(*[kv.shape[0] for kv in kv_caches])
    bts = (ctypes.c_void_p * D)(*[bt.data_ptr() for bt in block_tables])
    strides = (ctypes.c_int64 * D)(*[bt.stride(0) for bt in block_tables])
    wids = (ctypes.c_int32 * D)(*widths)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().smla_dcp_sparse_mla_decode_fused(
        q.data_ptr(), T, H, K, float(sm_scale), req_id_per_token.data_ptr(),
        topk_global.data_ptr(), num_reqs, D, block_size, int(interleave), pools, nslots, bts,
        strides, wids,
        out.data_ptr(), lse.data_ptr(), ws_ptr, ws_bytes, _stream_ptr(stream, dev))
    _check("smla_dcp_sparse_mla_decode_fused", st)
    return out, lse


MAX_HOST_CHUNKS = 8


def _need_host(t: torch.Tensor, name: str, dtype, shape):
    if t.dtype != dtype or t.device.type != "cpu" or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} host tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def dcp_sparse_mla_decode_fused_host(q_host: torch.Tensor, topk_host: torch.Tensor,
                                     out_host: torch.Tensor, lse_host: torch.Tensor,
                                     req_id_per_token: torch.Tensor,
                                     kv_caches: Sequence[torch.Tensor],
                                     block_tables: Sequence[torch.Tensor], block_size: int,
                                     sm_scale: float, *, interleave: int = 1,
                                     bt_widths: Optional[Sequence[int]] = None,
                                     q_dev: Optional[torch.Tensor] = None,
                                     topk_dev: Optional[torch.Tensor] = None,
                                     out_dev: Optional[torch.Tensor] = None,
                                     lse_dev: Optional[torch.Tensor] = None,
                                     workspace: Optional[torch.Tensor] = None,
                                     chunks: int = 4,
                                     stream: Optional[torch.cuda.Stream] = None
                                     ) -> Tuple[torch.Tensor, torch.Tensor]:
    """The fused step from and to (pinned) host memory: q and the top-k ids
    are copied in and out/lse back by the library, row groups pipelined
    (smla_dcp_sparse_mla_decode_fused_host).  Returns (out_host, lse_host),
    which hold the results once `stream` has reached the end of the call."""
    dev = req_id_per_token.device
    _need(req_id_per_token, "req_id_per_token", torch.int32, dev)
    T, H, Dq = q_host.shape
    K = topk_host.shape[1]
    _need_host(q_host, "q_host", torch.bfloat16, (T, H, QK_DIM))
    _need_host(topk_host, "topk_host", torch.int32, (T, K))
    _need_host(out_host, "out_host", torch.bfloat16, (T, H, V_DIM))
    _need_host(lse_host, "lse_host", torch.float32, (T, H))
    D = len(kv_caches)
    if D != len(block_tables) or D < 1:
        raise ValueError("need one block table per KV pool (>= 1)")
    num_reqs = None
    for kv, bt in zip(kv_caches, block_tables):
        _need(kv, "kv_caches[d]", torch.uint8, dev)
        if kv.dim() != 2 or kv.shape[1] != ROW_BYTES:
            raise ValueError(f"kv_caches[d] must be [num_slots, {ROW_BYTES}] uint8")
        if bt.dtype != torch.int32 or bt.device != dev or bt.dim() != 2 or bt.stride(1) != 1:
            raise ValueError("block_tables[d] must be 2-D int32 with contiguous rows")
        num_reqs = bt.shape[0] if num_reqs is None else min(num_reqs, bt.shape[0])
    if q_dev is None:
        q_dev = torch.empty((T, H, QK_DIM), dtype=torch.bfloat16, device=dev)
    if topk_dev is None:
        topk_dev = torch.empty((T, K), dtype=torch.int32, device=dev)
    if out_dev is None:
        out_dev = torch.empty((T, H, V_DIM), dtype=torch.bfloat16, device=dev)
    if lse_dev is None:
        lse_dev = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(q_dev, "q_dev", torch.bfloat16, dev)
    _need(topk_dev, "topk_dev", torch.int32, dev)
    _need(out_dev, "out_dev", torch.bfloat16, dev)
    _need(lse_dev, "lse_dev", torch.float32, dev)
    if workspace is None and min(chunks, T) == 1:
        workspace = alloc_decode_workspace(T, H, K, dev)
    widths = [bt.shape[1] for bt in block_tables] if bt_widths is None else list(bt_widths)
    pools = (ctypes.c_void_p * D)(*[kv.data_ptr() for kv in kv_caches])
    nslots = (ctypes.c_int64 * D)(*[kv.shape[0] for kv in kv_caches])
    bts = (ctypes.c_void_p * D)(*[bt.data_ptr() for bt in block_tables])
    strides = (ctypes.c_int64 * D)(*[bt.stride(0) for bt in block_tables])
    wids = (ctypes.c_int32 * D)(*widths)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().smla_dcp_sparse_mla_decode_fused_host(
        q_host.data_ptr(), topk_host.data_ptr(), out_host.data_ptr(), lse_host.data_ptr(),
        q_dev.data_ptr(), topk_dev.data_ptr(), out_dev.data_ptr(), lse_dev.data_ptr(),
        T, H, K, float(sm_scale), req_id_per_token.data_ptr(), num_reqs, D, block_size,
        int(interleave), pools, nslots, bts, strides, wids, ws_ptr, ws_bytes, int(chunks),
        _stream_ptr(stream, dev))
    _check("smla_dcp_sparse_mla_decode_fused_host", st)
    return out_host, lse_host


def dense_decode_workspace_size(T: int, H: int, max_ctx: int, D: int, interleave: int = 1,
                                rank: int = -1) -> int:
    return int(load().smla_dense_decode_workspace_size(T, H, max_ctx, D, interleave, rank))


def dcp_dense_mla_decode(q: torch.Tensor, ctx_lens: torch.Tensor, max_ctx: int, S: int,
                         kv_caches: Sequence[Optional[torch.Tensor]],
                         block_tables: Sequence[Optional[torch.Tensor]], block_size: int,
                         sm_scale: float, *, rank: int = -1, interleave: int = 1,
                         bt_widths: Optional[Sequence[int]] = None,
                         out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None
                         ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Dense decode over each request's whole causal context: merged over the
    D pools (rank = -1) or one rank's partial (rank >= 0; only its pool and
    table are read).  q is [B*S, H, 576]; rows come out in token order b*S+s."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, dev)
    T, H, Dq = q.shape
    B = ctx_lens.shape[0]
    if Dq != QK_DIM or T != B * S:
        raise ValueError("q must be [B*S, H, 576] with B = len(ctx_lens)")
    D = len(kv_caches)
    if D != len(block_tables) or D < 1:
        raise ValueError("need one block table per KV pool (>= 1)")
    used = [d for d in range(D) if rank < 0 or d == rank]
    for d in used:
        kv, bt = kv_caches[d], block_tables[d]
        _need(kv, "kv_caches[d]", torch.uint8, dev)
        if kv.dim() != 2 or kv.shape[1] != ROW_BYTES:
            raise ValueError(f"kv_caches[d] must be [num_slots, {ROW_BYTES}] uint8")
        if bt.dtype != torch.int32 or bt.device != dev or bt.dim() != 2 or bt.stride(1) != 1:
            raise ValueError("block_tables[d] must be 2-D int32 with contiguous rows")
    if out is None:
        out = torch.empty((T, H, V_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    if workspace is None:
        n = dense_decode_workspace_size(T, H, max_ctx, D, interleave, rank)
        workspace = torch.zeros(n, dtype=torch.uint8, device=dev) if n else None
    widths = [0] * D
    for d in used:
        widths[d] = block_tables[d].shape[1] if bt_widths is None else int(bt_widths[d])
    ptr = lambda t: t.data_ptr() if t is not None else None
    pools = (ctypes.c_void_p * D)(*[ptr(kv_caches[d]) if d in used else None for d in range(D)])
    nslots = (ctypes.c_int64 * D)(*[kv_caches[d].shape[0] if d in used else 0 for d in range(D)])
    bts = (ctypes.c_void_p * D)(*[ptr(block_tables[d]) if d in used else None for d in range(D)])
    strides = (ctypes.c_int64 * D)(*[block_tables[d].stride(0) if d in used else 0
                                     for d in range(D)])
    wids = (ctypes.c_int32 * D)(*widths)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().smla_dcp_dense_mla_decode(
        q.data_ptr(), B, S, H, float(sm_scale), ctx_lens.data_ptr(), int(max_ctx), D, int(rank),
        int(block_size), int(interleave), pools, nslots, bts, strides, wids, out.data_ptr(),
        lse.data_ptr(), ws_ptr, ws_bytes, _stream_ptr(stream, dev))
    _check("smla_dcp_dense_mla_decode", st)
    return out, lse


MAX_TOPK = 16384


def topk_select_workspace_size(T: int, L: int, K: int) -> int:
    """Bytes of the optional workspace topk_select uses to cut long rows
    into chunks (0: no row of L candidates is cut)."""
    return int(load().smla_topk_select_workspace_size(T, L, K))


def topk_select(scores: torch.Tensor, n_cand: torch.Tensor, K: int, *, D: int = 1, rank: int = 0,
                interleave: int = 1, with_scores: bool = False,
                workspace: Union[torch.Tensor, None, bool] = True,
                stream: Optional[torch.cuda.Stream] = None):
    """Top-K of each row's first n_cand local positions of `rank` (score
    descending, id ascending), as global ids, -1 padded.  scores is
    [T, L] fp32 with contiguous rows.  workspace: a uint8 device tensor of
    at least topk_select_workspace_size(T, L, K) bytes, True (allocate one
    here when that size is not 0) or None (rows are never cut into chunks)."""
    dev = scores.device
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be a 2-D fp32 tensor with contiguous rows")
    _need(n_cand, "n_cand", torch.int32, dev)
    T, L = scores.shape
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    sc = torch.empty((T, K), dtype=torch.float32, device=dev) if with_scores else None
    if workspace is True:
        need = topk_select_workspace_size(T, L, K) if 1 <= K <= MAX_TOPK else 0
        workspace = torch.empty(need, dtype=torch.uint8, device=dev) if need else None
    elif workspace is False:
        workspace = None
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, dev)
    st = load().smla_topk_select(scores.data_ptr(), scores.stride(0), L, n_cand.data_ptr(), T, K,
                                 D, rank, interleave, ids.data_ptr(),
                                 sc.data_ptr() if sc is not None else None,
                                 workspace.data_ptr() if workspace is not None else None,
                                 workspace.numel() if workspace is not None else 0,
                                 _stream_ptr(stream, dev))
    _check("smla_topk_select", st)
    return (ids, sc) if with_scores else ids


def dcp_topk_merge(cand_ids: torch.Tensor, cand_scores: torch.Tensor, K: int, *,
                   with_scores: bool = False, stream: Optional[torch.cuda.Stream] = None):
    """Top-K of each row's candidates (ids >= 0) by the same rule."""
    dev = cand_ids.device
    _need(cand_ids, "cand_ids", torch.int32, dev)
    _need(cand_scores, "cand_scores", torch.float32, dev)
    if cand_ids.shape != cand_scores.shape or cand_ids.dim() != 2:
        raise ValueError("cand_ids and cand_scores must be [T, M]")
    T, M = cand_ids.shape
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    sc = torch.empty((T, K), dtype=torch.float32, device=dev) if with_scores else None
    st = load().smla_dcp_topk_merge(cand_ids.data_ptr(), cand_scores.data_ptr(), M, M, T, K,
                                    ids.data_ptr(), sc.data_ptr() if sc is not None else None,
                                    _stream_ptr(stream, dev))
    _check("smla_dcp_topk_merge", st)
    return (ids, sc) if with_scores else ids


def dcp_lse_merge(outs: Sequence[torch.Tensor], lses: Sequence[torch.Tensor], *,
                  out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None
                  ) -> Tuple[torch.Tensor, torch.Tensor]:
    D = len(outs)
    if D != len(lses) or D < 1:
        raise ValueError("need as many lse tensors as out tensors (>= 1)")
    dev = outs[0].device
    T, H, V = outs[0].shape
    for o, l in zip(outs, lses):
        _need(o, "outs[d]", torch.bfloat16, dev)
        _need(l, "lses[d]", torch.float32, dev)
        if tuple(o.shape) != (T, H, V) or tuple(l.shape) != (T, H):
            raise ValueError("all partials must share [T, H, 512] / [T, H]")
    if out is None:
        out = torch.empty((T, H, V_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    out_ptrs = (ctypes.c_void_p * D)(*[o.data_ptr() for o in outs])
    lse_ptrs = (ctypes.c_void_p * D)(*[l.data_ptr() for l in lses])
    st = load().smla_dcp_lse_merge(out_ptrs, lse_ptrs, D, T, H, out.data_ptr(),
                                   lse.data_ptr(), _stream_ptr(stream, dev))
    _check("smla_dcp_lse_merge", st)
    return out, lse
