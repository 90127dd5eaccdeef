"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/smla.h declares, and rejects bad
arguments with the documented status before touching the device."""
import ctypes
import os
import re

import pytest

from sparse_mla_decode_dcp_gb300 import build as smla_build
from sparse_mla_decode_dcp_gb300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smla.h")


@pytest.fixture(scope="module")
def lib():
    smla_build.build()
    return capi.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    src = re.sub(r"#define[^\n]*", "", src)
    return sorted(set(re.findall(r"\b(smla_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_three_path_calls():
    names = _declared_functions()
    for n in ("smla_dcp_filter_convert_index", "smla_sparse_mla_decode",
              "smla_dcp_lse_merge", "smla_decode_workspace_size",
              "smla_dcp_sparse_mla_decode_fused", "smla_dcp_sparse_mla_decode_fused_host",
              "smla_dcp_dense_mla_decode",
              "smla_dense_decode_workspace_size",
              "smla_status_string", "smla_get_device_error"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libsmla.so does not export {name}"
        assert name in capi.SIGNATURES, f"binding lacks a signature for {name}"


def test_status_strings(lib):
    assert capi.status_string(0) == "SMLA_OK"
    assert capi.status_string(1) == "SMLA_ERR_INVALID_ARG"
    assert capi.status_string(2) == "SMLA_ERR_UNSUPPORTED"
    assert capi.status_string(3) == "SMLA_ERR_WORKSPACE"
    assert capi.status_string(4) == "SMLA_ERR_CUDA"
    assert capi.status_string(99) == "SMLA_UNKNOWN_STATUS"


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced


def _convert(lib, **kw):
    a = dict(req=FAKE, bt=FAKE, stride=4, width=4, nreq=2, topk=FAKE, T=3, K=8,
             D=2, rank=0, bs=16, I=1, out=FAKE, cnt=None)
    a.update(kw)
    return lib.smla_dcp_filter_convert_index(
        a["req"], a["bt"], a["stride"], a["width"], a["nreq"], a["topk"], a["T"],
        a["K"], a["D"], a["rank"], a["bs"], a["I"], a["out"], a["cnt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), capi.SMLA_ERR_INVALID_ARG),
    (dict(K=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(D=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(rank=2), capi.SMLA_ERR_INVALID_ARG),
    (dict(rank=-1), capi.SMLA_ERR_INVALID_ARG),
    (dict(bs=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(I=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(I=-2), capi.SMLA_ERR_INVALID_ARG),
    (dict(nreq=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(width=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(stride=3), capi.SMLA_ERR_INVALID_ARG),
    (dict(req=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(bt=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(topk=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(out=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(out=FAKE + 2), capi.SMLA_ERR_INVALID_ARG),
    (dict(cnt=FAKE + 1), capi.SMLA_ERR_INVALID_ARG),
    (dict(T=0, req=None, topk=None, out=None), capi.SMLA_OK),
])
def test_convert_argument_checks(lib, kw, status):
    assert _convert(lib, **kw) == status


def _decode(lib, **kw):
    a = dict(q=FAKE, kv=FAKE, ns=100, slots=FAKE, T=2, H=16, K=64, scale=0.07,
             out=FAKE, lse=FAKE, ws=None, wsb=0)
    a.update(kw)
    if "ws_auto" in kw:
        need = lib.smla_decode_workspace_size(a["T"], a["H"], a["K"])
        a["ws"], a["wsb"] = (FAKE if need else None), need
    return lib.smla_sparse_mla_decode(
        a["q"], a["kv"], a["ns"], a["slots"], a["T"], a["H"], a["K"],
        ctypes.c_float(a["scale"]), a["out"], a["lse"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), capi.SMLA_ERR_INVALID_ARG),
    (dict(K=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(H=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(H=129), capi.SMLA_ERR_UNSUPPORTED),
    (dict(H=256), capi.SMLA_ERR_UNSUPPORTED),
    (dict(ns=-1), capi.SMLA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), capi.SMLA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), capi.SMLA_ERR_INVALID_ARG),
    (dict(scale=0.0), capi.SMLA_ERR_INVALID_ARG),
    (dict(scale=-0.07), capi.SMLA_ERR_INVALID_ARG),
    (dict(q=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(kv=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(slots=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(out=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(lse=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), capi.SMLA_ERR_INVALID_ARG),
    (dict(kv=FAKE + 4), capi.SMLA_ERR_INVALID_ARG),
    (dict(out=FAKE + 2), capi.SMLA_ERR_INVALID_ARG),
    (dict(T=0, q=None, kv=None, slots=None, out=None, lse=None), capi.SMLA_OK),
])
def test_decode_argument_checks(lib, kw, status):
    assert _decode(lib, **kw) == status


def test_decode_workspace_checks(lib):
    for T, H, K in [(64, 128, 2048), (32, 64, 2048), (2, 16, 64), (128, 128, 2048)]:
        need = capi.decode_workspace_size(T, H, K)
        if need == 0:
            continue
        assert _decode(lib, T=T, H=H, K=K, ws=None, wsb=0) == capi.SMLA_ERR_WORKSPACE
        assert _decode(lib, T=T, H=H, K=K, ws=FAKE, wsb=need - 1) == capi.SMLA_ERR_WORKSPACE
        assert _decode(lib, T=T, H=H, K=K, ws=FAKE + 16, wsb=need) == capi.SMLA_ERR_WORKSPACE


def test_workspace_size_shape_only(lib):
    assert capi.decode_workspace_size(-1, 16, 64) == 0
    assert capi.decode_workspace_size(2, 0, 64) == 0
    assert capi.decode_workspace_size(2, 129, 64) == 0
    assert capi.decode_workspace_size(2, 16, 0) == 0
    # pure function of the shape
    assert capi.decode_workspace_size(64, 128, 2048) == capi.decode_workspace_size(64, 128, 2048)
    # monotone in T
    assert capi.decode_workspace_size(128, 128, 2048) >= capi.decode_workspace_size(64, 128, 2048)


def _fused(lib, D=2, **kw):
    a = dict(q=FAKE, T=2, H=16, K=64, scale=0.07, req=FAKE, topk=FAKE, nreq=2, bs=16, I=1,
             pools=[FAKE] * D, nslots=[100] * D, bts=[FAKE] * D, strides=[4] * D,
             widths=[4] * D, out=FAKE, lse=FAKE, ws=None, wsb=0)
    a.update(kw)
    n = max(D, 1)
    arr = lambda typ, xs: (typ * n)(*(list(xs) + [0] * (n - len(xs)))[:n])
    return lib.smla_dcp_sparse_mla_decode_fused(
        a["q"], a["T"], a["H"], a["K"], ctypes.c_float(a["scale"]), a["req"], a["topk"],
        a["nreq"], D, a["bs"], a["I"], arr(ctypes.c_void_p, a["pools"]),
        arr(ctypes.c_int64, a["nslots"]),
        arr(ctypes.c_void_p, a["bts"]), arr(ctypes.c_int64, a["strides"]),
        arr(ctypes.c_int32, a["widths"]), a["out"], a["lse"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("D,kw,status", [
    (0, {}, capi.SMLA_ERR_INVALID_ARG),
    (17, {}, capi.SMLA_ERR_UNSUPPORTED),
    (2, dict(H=129), capi.SMLA_ERR_UNSUPPORTED),
    (2, dict(T=-1), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(K=0), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(bs=0), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(I=0), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(nreq=0), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(scale=float("nan")), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(scale=-1.0), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(q=None), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(topk=None), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(q=FAKE + 8), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(pools=[FAKE, None]), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(pools=[FAKE, FAKE + 4]), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(nslots=[100, -1]), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(bts=[None, FAKE]), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(widths=[0, 4]), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(strides=[4, 3]), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(T=0, q=None, topk=None, req=None, out=None, lse=None), capi.SMLA_OK),
])
def test_fused_argument_checks(lib, D, kw, status):
    assert _fused(lib, D=D, **kw) == status


def test_fused_workspace_checks(lib):
    need = capi.decode_workspace_size(3, 128, 2048)
    assert need > 0
    assert _fused(lib, T=3, H=128, K=2048) == capi.SMLA_ERR_WORKSPACE
    assert _fused(lib, T=3, H=128, K=2048, ws=FAKE, wsb=need - 1) == capi.SMLA_ERR_WORKSPACE


def _fused_host(lib, D=2, **kw):
    a = dict(qh=FAKE, th=FAKE, oh=FAKE, lh=FAKE, q=FAKE, topk=FAKE, out=FAKE, lse=FAKE, T=2,
             H=16, K=64, scale=0.07, req=FAKE, nreq=2, bs=16, I=1, pools=[FAKE] * D,
             nslots=[100] * D, bts=[FAKE] * D, strides=[4] * D, widths=[4] * D, ws=None, wsb=0,
             chunks=2)
    a.update(kw)
    arr = lambda typ, xs: (typ * D)(*xs)
    return lib.smla_dcp_sparse_mla_decode_fused_host(
        a["qh"], a["th"], a["oh"], a["lh"], a["q"], a["topk"], a["out"], a["lse"], a["T"],
        a["H"], a["K"], ctypes.c_float(a["scale"]), a["req"], a["nreq"], D, a["bs"], a["I"],
        arr(ctypes.c_void_p, a["pools"]), arr(ctypes.c_int64, a["nslots"]),
        arr(ctypes.c_void_p, a["bts"]), arr(ctypes.c_int64, a["strides"]),
        arr(ctypes.c_int32, a["widths"]), a["ws"], a["wsb"], a["chunks"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(chunks=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(chunks=capi.MAX_HOST_CHUNKS + 1), capi.SMLA_ERR_INVALID_ARG),
    (dict(qh=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(th=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(oh=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(lh=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), capi.SMLA_ERR_INVALID_ARG),    # staging buffers as the fused step's
    (dict(out=FAKE + 4), capi.SMLA_ERR_INVALID_ARG),
    (dict(topk=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(H=129), capi.SMLA_ERR_UNSUPPORTED),
    (dict(scale=0.0), capi.SMLA_ERR_INVALID_ARG),
    # row groups decode without split-K: one cluster's list holds 2048 keys
    (dict(K=2049), capi.SMLA_ERR_UNSUPPORTED),
    # one group (chunks = 1, or above T): the usual split-K policy and workspace
    (dict(T=3, H=128, K=2048, chunks=1), capi.SMLA_ERR_WORKSPACE),
    (dict(T=1, H=128, K=4096, chunks=4), capi.SMLA_ERR_WORKSPACE),
    (dict(T=0, qh=None, th=None, oh=None, lh=None, q=None, topk=None, out=None, lse=None,
          req=None), capi.SMLA_OK),
])
def test_fused_host_argument_checks(lib, kw, status):
    assert _fused_host(lib, **kw) == status


def _merge(lib, D=2, T=3, H=4, outs=None, lses=None, out=FAKE, lse=FAKE):
    if outs is None:
        outs = [FAKE] * max(D, 1)
    if lses is None:
        lses = [FAKE] * max(D, 1)
    op = (ctypes.c_void_p * len(outs))(*outs)
    lp = (ctypes.c_void_p * len(lses))(*lses)
    return lib.smla_dcp_lse_merge(op, lp, D, T, H, out, lse, None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(D=17), capi.SMLA_ERR_UNSUPPORTED),
    (dict(T=-1), capi.SMLA_ERR_INVALID_ARG),
    (dict(H=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(out=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(lse=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(out=FAKE + 8), capi.SMLA_ERR_INVALID_ARG),
    (dict(outs=[FAKE, None]), capi.SMLA_ERR_INVALID_ARG),
    (dict(outs=[FAKE, FAKE + 8]), capi.SMLA_ERR_INVALID_ARG),
    (dict(lses=[FAKE, FAKE + 2]), capi.SMLA_ERR_INVALID_ARG),
    (dict(T=0), capi.SMLA_OK),
])
def test_merge_argument_checks(lib, kw, status):
    assert _merge(lib, **kw) == status


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(capi, "_lib", None)
    monkeypatch.setattr(capi, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        capi.load()


def _dense(lib, D=2, **kw):
    a = dict(q=FAKE, B=2, S=1, H=16, scale=0.07, ctx=FAKE, maxc=100, rank=-1, bs=16, I=1,
             pools=[FAKE] * D, nslots=[100] * D, bts=[FAKE] * D, strides=[4] * D,
             widths=[4] * D, out=FAKE, lse=FAKE, ws=None, wsb=0)
    a.update(kw)
    n = max(D, 1)
    arr = lambda typ, xs: (typ * n)(*(list(xs) + [0] * (n - len(xs)))[:n])
    return lib.smla_dcp_dense_mla_decode(
        a["q"], a["B"], a["S"], a["H"], ctypes.c_float(a["scale"]), a["ctx"], a["maxc"], D,
        a["rank"], a["bs"], a["I"], arr(ctypes.c_void_p, a["pools"]),
        arr(ctypes.c_int64, a["nslots"]), arr(ctypes.c_void_p, a["bts"]),
        arr(ctypes.c_int64, a["strides"]), arr(ctypes.c_int32, a["widths"]), a["out"], a["lse"],
        a["ws"], a["wsb"], None)


@pytest.mark.parametrize("D,kw,status", [
    (0, {}, capi.SMLA_ERR_INVALID_ARG),
    (17, {}, capi.SMLA_ERR_UNSUPPORTED),
    (2, dict(H=129), capi.SMLA_ERR_UNSUPPORTED),
    (2, dict(B=-1), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(S=0), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(maxc=0), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(rank=2), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(rank=-2), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(bs=0), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(I=0), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(scale=float("inf")), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(ctx=None), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(q=FAKE + 8), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(pools=[FAKE, None]), capi.SMLA_ERR_INVALID_ARG),
    # rank >= 0 reads only its own pool and table: the others may be empty
    # (the call passes every argument check and stops at the missing workspace)
    (2, dict(rank=0, maxc=65536, pools=[FAKE, None], bts=[FAKE, None], widths=[4, 0]),
     capi.SMLA_ERR_WORKSPACE),
    (2, dict(rank=1, pools=[FAKE, None]), capi.SMLA_ERR_INVALID_ARG),
    (2, dict(B=0, q=None, ctx=None, out=None, lse=None), capi.SMLA_OK),
])
def test_dense_argument_checks(lib, D, kw, status):
    assert _dense(lib, D=D, **kw) == status


def test_dense_workspace_size_is_a_function_of_the_shape(lib):
    assert capi.dense_decode_workspace_size(2, 16, 0, 2) == 0
    assert capi.dense_decode_workspace_size(2, 16, 100, 2, 1, 2) == 0
    big = capi.dense_decode_workspace_size(8, 128, 65536, 4, 1, -1)
    one = capi.dense_decode_workspace_size(8, 128, 65536, 4, 1, 0)
    assert big > one > 0  # one rank holds a quarter of the positions
    assert big == capi.decode_workspace_size(8, 128, 65536)


def _topk_select(lib, **kw):
    a = dict(scores=FAKE, stride=100, L=100, n=FAKE, T=2, K=16, D=1, rank=0, I=1, out=FAKE,
             sc=None, ws=None, ws_bytes=0)
    a.update(kw)
    return lib.smla_topk_select(a["scores"], a["stride"], a["L"], a["n"], a["T"], a["K"], a["D"],
                                a["rank"], a["I"], a["out"], a["sc"], a["ws"], a["ws_bytes"],
                                None)


def _topk_merge(lib, **kw):
    a = dict(ids=FAKE, scores=FAKE, stride=64, M=64, T=2, K=16, out=FAKE, sc=None)
    a.update(kw)
    return lib.smla_dcp_topk_merge(a["ids"], a["scores"], a["stride"], a["M"], a["T"], a["K"],
                                   a["out"], a["sc"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), capi.SMLA_ERR_INVALID_ARG),
    (dict(L=-1), capi.SMLA_ERR_INVALID_ARG),
    (dict(stride=99), capi.SMLA_ERR_INVALID_ARG),
    (dict(D=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(D=2, rank=2), capi.SMLA_ERR_INVALID_ARG),
    (dict(I=0), capi.SMLA_ERR_INVALID_ARG),
    (dict(K=0), capi.SMLA_ERR_UNSUPPORTED),
    (dict(K=16385), capi.SMLA_ERR_UNSUPPORTED),
    (dict(scores=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(n=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(out=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(out=FAKE + 2), capi.SMLA_ERR_INVALID_ARG),
    (dict(T=0, scores=None, n=None, out=None), capi.SMLA_OK),
    # 300000 candidates, K = 16: up to 8 chunks a row, 2 x 8 x 16 x 8 = 2048 bytes
    (dict(L=300000, stride=300000, ws=FAKE, ws_bytes=2047), capi.SMLA_ERR_WORKSPACE),
    (dict(L=300000, stride=300000, ws=FAKE + 8, ws_bytes=4096), capi.SMLA_ERR_WORKSPACE),
    (dict(ws=FAKE + 8, ws_bytes=4096), capi.SMLA_ERR_WORKSPACE),
])
def test_topk_select_argument_checks(lib, kw, status):
    assert _topk_select(lib, **kw) == status


def test_topk_select_workspace_size_is_a_function_of_the_shape(lib):
    # rows are cut only for T <= 32 and L >= 16 x max(16384, 8 x the sort
    # size); the workspace then holds 8 chunks' K ids and scores a row
    assert capi.topk_select_workspace_size(8, 262143, 2048) == 0
    assert capi.topk_select_workspace_size(8, 262144, 2048) == 8 * 8 * 2048 * 8
    assert capi.topk_select_workspace_size(32, 1 << 20, 2048) == 32 * 8 * 2048 * 8
    assert capi.topk_select_workspace_size(33, 1 << 20, 2048) == 0  # many rows: whole
    assert capi.topk_select_workspace_size(64, 65536, 2048) == 0
    assert capi.topk_select_workspace_size(3, 300000, 16) == 3 * 8 * 16 * 8
    assert capi.topk_select_workspace_size(2, (1 << 21) - 1, 9000) == 0  # sort size 16384
    assert capi.topk_select_workspace_size(2, 1 << 21, 9000) == 2 * 8 * 9000 * 8
    assert capi.topk_select_workspace_size(0, 200000, 16) == 0
    assert capi.topk_select_workspace_size(2, 200000, 0) == 0
    assert capi.topk_select_workspace_size(2, 200000, 16385) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), capi.SMLA_ERR_INVALID_ARG),
    (dict(M=-1), capi.SMLA_ERR_INVALID_ARG),
    (dict(stride=63), capi.SMLA_ERR_INVALID_ARG),
    (dict(K=0), capi.SMLA_ERR_UNSUPPORTED),
    (dict(ids=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(scores=None), capi.SMLA_ERR_INVALID_ARG),
    (dict(sc=FAKE + 1), capi.SMLA_ERR_INVALID_ARG),
    (dict(T=0, ids=None, scores=None, out=None), capi.SMLA_OK),
])
def test_topk_merge_argument_checks(lib, kw, status):
    assert _topk_merge(lib, **kw) == status
