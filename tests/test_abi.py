"""CPU checks of the C ABI: the library loads, exports every function that
include/osattn.h declares, and rejects bad arguments on the host before any
CUDA call (so these run without a GPU; no call here reaches a kernel)."""
import ctypes
import glob
import os
import re

import pytest

from attention_forward_online_gb300 import osattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from attention_forward_online_gb300 import _build

    _build.build()
    return osattn.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"^[A-Za-z_][\w \*]*?\b(osattn_\w+)\s*\(", text, flags=re.M))
    return names


def test_every_declared_function_is_exported(L):
    names = declared_functions()
    assert {"osattn_fwd", "osattn_status_string", "osattn_get_device_status",
            "osattn_version"} <= names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    assert set(osattn.EXPORTS) == names


def test_version_and_status_strings(L):
    assert osattn.version() == 1
    for code, text in [(0, "ok"), (1, "invalid argument"), (2, "unsupported"),
                       (3, "CUDA error"), (4, "timed out"), (77, "unknown")]:
        assert text in osattn.status_string(code)


P = 0x10000  # a 16-byte aligned fake address; validation fails before it is used


def call(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=1, Nq=8, Nkv=8, d=64, scale=0.125,
             causal=0, key_len=None, dtype=osattn.BF16)
    a.update(kw)
    return osattn.fwd_raw(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"],
                          a["Nkv"], a["d"], a["scale"], a["causal"], a["key_len"], a["dtype"],
                          ctypes.c_void_p(None))


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), osattn.ERR_INVALID_ARG),
    (dict(k=None), osattn.ERR_INVALID_ARG),
    (dict(v=None), osattn.ERR_INVALID_ARG),
    (dict(o=None), osattn.ERR_INVALID_ARG),
    (dict(lse=None), osattn.ERR_INVALID_ARG),
    (dict(B=0), osattn.ERR_INVALID_ARG),
    (dict(H=-1), osattn.ERR_INVALID_ARG),
    (dict(Nq=0), osattn.ERR_INVALID_ARG),
    (dict(Nkv=0), osattn.ERR_INVALID_ARG),
    (dict(scale=float("nan")), osattn.ERR_INVALID_ARG),
    (dict(scale=float("inf")), osattn.ERR_INVALID_ARG),
    (dict(q=P + 8), osattn.ERR_INVALID_ARG),
    (dict(o=P + 2), osattn.ERR_INVALID_ARG),
    (dict(lse=P + 2), osattn.ERR_INVALID_ARG),
    (dict(key_len=P + 1), osattn.ERR_INVALID_ARG),
    (dict(d=96), osattn.ERR_UNSUPPORTED),
    (dict(d=256), osattn.ERR_UNSUPPORTED),
    (dict(dtype=7), osattn.ERR_UNSUPPORTED),
])
def test_host_validation_rejects_before_launch(L, kw, expect):
    assert call(**kw) == expect


def test_binding_rejects_cpu_tensors(L):
    import torch

    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        osattn.fwd(q, q, q)
    with pytest.raises(TypeError):
        osattn.fwd(q, q.float(), q)


def test_splitkv_workspace_size(L):
    # num_splits * B*H*Nq * (d + 1) fp32 values
    assert osattn.splitkv_workspace_bytes(1, 1, 4, 64, 2) == 2 * 4 * 65 * 4
    assert osattn.splitkv_workspace_bytes(2, 3, 100, 128, 7) == 7 * 600 * 129 * 4
    assert osattn.splitkv_workspace_bytes(0, 1, 4, 64, 2) == 0
    assert osattn.splitkv_workspace_bytes(1, 1, 4, 64, 0) == 0


def call_split(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=1, Nq=8, Nkv=8, d=64, scale=0.125, causal=0,
             key_len=None, dtype=osattn.BF16, splits=2, ws=P, ws_bytes=1 << 20)
    a.update(kw)
    return osattn.lib().osattn_fwd_splitkv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"],
                                           a["H"], a["Nq"], a["Nkv"], a["d"], a["scale"],
                                           a["causal"], a["key_len"], a["dtype"], a["splits"],
                                           a["ws"], a["ws_bytes"], ctypes.c_void_p(None))


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), osattn.ERR_INVALID_ARG),
    (dict(splits=0), osattn.ERR_INVALID_ARG),
    (dict(splits=129), osattn.ERR_INVALID_ARG),
    (dict(ws=None), osattn.ERR_INVALID_ARG),
    (dict(ws=P + 4), osattn.ERR_INVALID_ARG),
    (dict(ws_bytes=2 * 8 * 65 * 4 - 1), osattn.ERR_INVALID_ARG),
    (dict(dtype=osattn.FP32), osattn.ERR_UNSUPPORTED),
    (dict(d=96), osattn.ERR_UNSUPPORTED),
])
def test_splitkv_host_validation(L, kw, expect):
    assert call_split(**kw) == expect


def test_noalloc_rejects_problems_beyond_its_scratch(L):
    # 4 x 8 x 4096 rows x 129 floats x 4 splits > 32 MiB: rejected on the host
    need = osattn.splitkv_workspace_bytes(4, 8, 4096, 128, 4)
    assert need > osattn.NOALLOC_SCRATCH_BYTES
    rc = L.osattn_fwd_splitkv_noalloc(P, P, P, P, P, 4, 8, 4096, 4096, 128, 0.125, 0, None,
                                      osattn.BF16, 4, ctypes.c_void_p(None))
    assert rc == osattn.ERR_SCRATCH_LIMIT
    assert "scratch" in osattn.status_string(rc)


@pytest.mark.parametrize("kw,expect", [
    (dict(splits=129), osattn.ERR_INVALID_ARG),
    (dict(splits=0), osattn.ERR_INVALID_ARG),
    (dict(q=None), osattn.ERR_INVALID_ARG),
    (dict(o=P + 8), osattn.ERR_INVALID_ARG),
    (dict(dtype=osattn.FP32), osattn.ERR_UNSUPPORTED),
    (dict(d=96), osattn.ERR_UNSUPPORTED),
])
@pytest.mark.parametrize("large", [False, True], ids=["small", "beyond_scratch"])
def test_noalloc_checks_arguments_before_its_scratch_limit(L, kw, expect, large):
    # Invalid arguments get the statuses of osattn_fwd_splitkv whether or not
    # the problem would also exceed the built-in scratch array.
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=4 if large else 1, H=8 if large else 1,
             Nq=4096 if large else 8, Nkv=4096 if large else 8, d=128, dtype=osattn.BF16,
             splits=4)
    a.update(kw)
    rc = L.osattn_fwd_splitkv_noalloc(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                                      a["Nq"], a["Nkv"], a["d"], 0.125, 0, None, a["dtype"],
                                      a["splits"], ctypes.c_void_p(None))
    assert rc == expect


def test_softmax_rows_host_validation(L):
    f = L.osattn_softmax_rows
    nul = ctypes.c_void_p(None)
    assert f(None, P, None, 4, 8, osattn.BF16, nul) == osattn.ERR_INVALID_ARG
    assert f(P, P, None, 0, 8, osattn.BF16, nul) == osattn.ERR_INVALID_ARG
    assert f(P, P, None, 4, 0, osattn.BF16, nul) == osattn.ERR_INVALID_ARG
    assert f(P + 1, P, None, 4, 8, osattn.BF16, nul) == osattn.ERR_INVALID_ARG
    assert f(P, P + 2, None, 4, 8, osattn.FP32, nul) == osattn.ERR_INVALID_ARG
    assert f(P, P, P + 2, 4, 8, osattn.FP32, nul) == osattn.ERR_INVALID_ARG
    assert f(P, P, None, 4, 8, 9, nul) == osattn.ERR_UNSUPPORTED


def call_strided(strides=(None, None, None, None), **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=2, Nq=8, Nkv=8, d=64, scale=0.125, causal=0,
             key_len=None, dtype=osattn.BF16)
    a.update(kw)
    arrs = [None if s is None else (ctypes.c_int64 * 3)(*s) for s in strides]
    return osattn.lib().osattn_fwd_strided(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"],
                                           a["H"], a["Nq"], a["Nkv"], a["d"], *arrs, a["scale"],
                                           a["causal"], a["key_len"], a["dtype"],
                                           ctypes.c_void_p(None))


BNHD = (8 * 2 * 64, 64, 2 * 64)  # [B, N, H, d] storage seen as [B, H, N, d]


@pytest.mark.parametrize("strides,dtype", [
    ((BNHD, BNHD, BNHD, (0, 64, 128)), osattn.BF16),          # zero stride
    ((BNHD, (-64, 64, 128), BNHD, BNHD), osattn.BF16),         # negative stride
    (((1024, 64, 132), BNHD, BNHD, BNHD), osattn.BF16),        # row 264 B: not 16-B multiple
    ((BNHD, BNHD, (1024, 68, 128), BNHD), osattn.FP16),        # head 136 B
    ((BNHD, BNHD, BNHD, (1024, 64, 130)), osattn.FP32),        # fp32 row 520 B
    ((BNHD, BNHD, BNHD, (1 << 40, 64, 128)), osattn.BF16),     # >= 2^40 bytes
])
def test_strided_host_validation(L, strides, dtype):
    assert call_strided(strides, dtype=dtype) == osattn.ERR_INVALID_ARG


def test_strided_shares_osattn_fwd_checks(L):
    assert call_strided(q=None) == osattn.ERR_INVALID_ARG
    assert call_strided(d=96) == osattn.ERR_UNSUPPORTED
    assert call_strided(dtype=3) == osattn.ERR_UNSUPPORTED
    assert call_strided(o=P + 8) == osattn.ERR_INVALID_ARG


def test_fp16_dtype_passes_host_validation_like_bf16(L):
    # Same rejections for fp16 as for bf16 (the first failing check decides).
    assert call(dtype=osattn.FP16, d=96) == osattn.ERR_UNSUPPORTED
    assert call(dtype=osattn.FP16, q=P + 8) == osattn.ERR_INVALID_ARG
    assert call_split(dtype=osattn.FP16, splits=0) == osattn.ERR_INVALID_ARG
    f = L.osattn_softmax_rows
    assert f(P + 1, P, None, 4, 8, osattn.FP16, ctypes.c_void_p(None)) == osattn.ERR_INVALID_ARG


def test_binding_rejects_non_unit_inner_stride(L):
    import torch

    q = torch.zeros(1, 1, 64, 4, dtype=torch.bfloat16).transpose(2, 3)  # d axis strided
    with pytest.raises(ValueError):
        osattn._bhn_strides(q)


def call_bwd(**kw):
    a = dict(q=P, k=P, v=P, o=P, do=P, lse=P, dq=P, dk=P, dv=P, B=1, H=1, Nq=8, Nkv=8, d=64,
             scale=0.125, causal=0, key_len=None, dtype=osattn.BF16, ws=P, ws_bytes=1 << 20)
    a.update(kw)
    return osattn.lib().osattn_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"],
                                   a["dk"], a["dv"], a["B"], a["H"], a["Nq"], a["Nkv"], a["d"],
                                   a["scale"], a["causal"], a["key_len"], a["dtype"], a["ws"],
                                   a["ws_bytes"], ctypes.c_void_p(None))


def test_bwd_workspace_size(L):
    assert osattn.bwd_workspace_bytes(2, 3, 100) == 2 * 3 * 100 * 4
    assert osattn.bwd_workspace_bytes(0, 3, 100) == 0


@pytest.mark.parametrize("kw,expect", [
    (dict(do=None), osattn.ERR_INVALID_ARG),
    (dict(dq=None), osattn.ERR_INVALID_ARG),
    (dict(dk=P + 2), osattn.ERR_INVALID_ARG),
    (dict(dv=P + 8), osattn.ERR_INVALID_ARG),
    (dict(o=None), osattn.ERR_INVALID_ARG),
    (dict(lse=None), osattn.ERR_INVALID_ARG),
    (dict(ws=None), osattn.ERR_INVALID_ARG),
    (dict(ws_bytes=8 * 4 - 1), osattn.ERR_INVALID_ARG),
    (dict(Nq=0), osattn.ERR_INVALID_ARG),
    (dict(scale=float("nan")), osattn.ERR_INVALID_ARG),
    (dict(dtype=3), osattn.ERR_UNSUPPORTED),
    (dict(d=96), osattn.ERR_UNSUPPORTED),
    (dict(dtype=osattn.FP32, dv=P + 8), osattn.ERR_INVALID_ARG),
    (dict(dtype=osattn.FP32, ws_bytes=8 * 4 - 1), osattn.ERR_INVALID_ARG),
])
def test_bwd_host_validation(L, kw, expect):
    assert call_bwd(**kw) == expect


def call_bwd_strided(strides=(None,) * 8, **kw):
    a = dict(q=P, k=P, v=P, o=P, do=P, lse=P, dq=P, dk=P, dv=P, B=1, H=2, Nq=8, Nkv=8, d=64,
             scale=0.125, causal=0, key_len=None, dtype=osattn.BF16, ws=P, ws_bytes=1 << 20)
    a.update(kw)
    arrs = [None if s is None else (ctypes.c_int64 * 3)(*s) for s in strides]
    return osattn.lib().osattn_bwd_strided(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"],
                                           a["dq"], a["dk"], a["dv"], a["B"], a["H"], a["Nq"],
                                           a["Nkv"], a["d"], *arrs, a["scale"], a["causal"],
                                           a["key_len"], a["dtype"], a["ws"], a["ws_bytes"],
                                           ctypes.c_void_p(None))


@pytest.mark.parametrize("slot", range(8))
@pytest.mark.parametrize("bad", [(0, 64, 128), (1024, -64, 128), (1024, 64, 132), (1 << 40, 64, 128)])
def test_bwd_strided_host_validation(L, slot, bad):
    # Every one of the eight stride arrays (Q, K, V, O, dO, dQ, dK, dV) is
    # checked: zero, negative, not a 16-byte multiple, >= 2^40 bytes.
    strides = [BNHD] * 8
    strides[slot] = bad
    assert call_bwd_strided(strides) == osattn.ERR_INVALID_ARG


def test_bwd_strided_shares_osattn_bwd_checks(L):
    assert call_bwd_strided(do=None) == osattn.ERR_INVALID_ARG
    assert call_bwd_strided(ws_bytes=2 * 8 * 4 - 1) == osattn.ERR_INVALID_ARG
    assert call_bwd_strided(dtype=3) == osattn.ERR_UNSUPPORTED
    # fp32 strides: multiples of 4 elements (16 bytes)
    assert call_bwd_strided([(1024, 64, 66)] + [BNHD] * 7, dtype=osattn.FP32) == osattn.ERR_INVALID_ARG
    assert call_bwd_strided(d=96) == osattn.ERR_UNSUPPORTED
    assert call_bwd_strided((BNHD,) * 8, dv=P + 8) == osattn.ERR_INVALID_ARG


def call_offload(**kw):
    a = dict(qh=P, kh=P, vh=P, oh=P, lh=P, q=P, k=P, v=P, o=P, lse=P, B=1, H=2, Nq=8, Nkv=8, d=64,
             scale=0.125, causal=0, key_len=None, dtype=osattn.BF16, hpc=1)
    a.update(kw)
    return osattn.lib().osattn_fwd_offload(a["qh"], a["kh"], a["vh"], a["oh"], a["lh"], a["q"],
                                           a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                                           a["Nq"], a["Nkv"], a["d"], a["scale"], a["causal"],
                                           a["key_len"], a["dtype"], a["hpc"],
                                           ctypes.c_void_p(None))


@pytest.mark.parametrize("kw,expect", [
    (dict(qh=None), osattn.ERR_INVALID_ARG),
    (dict(lh=None), osattn.ERR_INVALID_ARG),
    (dict(o=None), osattn.ERR_INVALID_ARG),
    (dict(q=P + 8), osattn.ERR_INVALID_ARG),
    (dict(hpc=-1), osattn.ERR_INVALID_ARG),
    (dict(Nkv=0), osattn.ERR_INVALID_ARG),
    (dict(d=96), osattn.ERR_UNSUPPORTED),
    (dict(dtype=3), osattn.ERR_UNSUPPORTED),
])
def test_offload_host_validation(L, kw, expect):
    assert call_offload(**kw) == expect


def call_bwd_offload(**kw):
    a = dict(h=[P] * 9, d_=[P] * 9, B=1, H=2, Nq=8, Nkv=8, d=64, scale=0.125, causal=0,
             key_len=None, dtype=osattn.BF16, ws=P, ws_bytes=1 << 20, hpc=0)
    a.update(kw)
    return osattn.lib().osattn_bwd_offload(*a["h"], *a["d_"], a["B"], a["H"], a["Nq"], a["Nkv"],
                                           a["d"], a["scale"], a["causal"], a["key_len"],
                                           a["dtype"], a["ws"], a["ws_bytes"], a["hpc"],
                                           ctypes.c_void_p(None))


@pytest.mark.parametrize("kw,expect", [
    (dict(h=[P] * 8 + [None]), osattn.ERR_INVALID_ARG),          # dV_host
    (dict(h=[None] + [P] * 8), osattn.ERR_INVALID_ARG),          # Q_host
    (dict(d_=[P] * 4 + [None] + [P] * 4), osattn.ERR_INVALID_ARG),  # dO
    (dict(d_=[P] * 8 + [P + 8]), osattn.ERR_INVALID_ARG),         # dV misaligned
    (dict(ws=None), osattn.ERR_INVALID_ARG),
    (dict(ws_bytes=2 * 8 * 4 - 1), osattn.ERR_INVALID_ARG),
    (dict(hpc=-2), osattn.ERR_INVALID_ARG),
    (dict(d=96), osattn.ERR_UNSUPPORTED),
    (dict(dtype=3), osattn.ERR_UNSUPPORTED),
])
def test_bwd_offload_host_validation(L, kw, expect):
    assert call_bwd_offload(**kw) == expect


@pytest.mark.parametrize("args,expect", [
    ((None, P, P, P, P, P, 4, 8, osattn.BF16, 0), osattn.ERR_INVALID_ARG),   # in_host
    ((P, P, None, P, P, P, 4, 8, osattn.BF16, 0), osattn.ERR_INVALID_ARG),   # lse_host without lse
    ((P, P, P, P, P, None, 4, 8, osattn.BF16, 0), osattn.ERR_INVALID_ARG),   # lse without lse_host
    ((P, P, P, P, P, P, 0, 8, osattn.BF16, 0), osattn.ERR_INVALID_ARG),      # rows
    ((P, P, P, P, P, P, 4, 8, osattn.BF16, -1), osattn.ERR_INVALID_ARG),     # rows_per_chunk
    ((P, P, P, P + 1, P, P, 4, 8, osattn.BF16, 0), osattn.ERR_INVALID_ARG),  # misaligned in
    ((P, P, P, P, P, P, 4, 8, 7, 0), osattn.ERR_UNSUPPORTED),
])
def test_softmax_rows_offload_host_validation(L, args, expect):
    assert L.osattn_softmax_rows_offload(*args, ctypes.c_void_p(None)) == expect


def test_step_trace_hook_is_unsupported_in_the_product_build(L):
    # The per-step clock stamps exist only in the separate profiling build
    # (OSATTN_STEP_TRACE=1); the product library answers UNSUPPORTED without
    # touching the device, and still reports the buffer size a trace needs.
    need = ctypes.c_size_t(0)
    rc = L.osattn_step_trace_read(None, 0, ctypes.byref(need))
    assert rc == osattn.ERR_UNSUPPORTED
    assert need.value == (8 * 7 * 128 * 4 + 4096 * 6) * 8
