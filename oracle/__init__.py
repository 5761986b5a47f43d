"""fp64 CPU oracle for the attention forward pass and its gradients (test
infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline use this package.  The product library never imports it, and it
never imports the product.  The arithmetic lives in ``osattn_ref.cpp``
(plain C++17, double precision); this module compiles it with the host C++
compiler and wraps it with ctypes/numpy.

What each function computes, with the passage it restates, is documented in
``osattn_ref.cpp``.  Sources: chapter 6 "Softmax 与 Online Softmax" of the
"手写 FlashAttention v2" CUDA book (yangyitao.com) and the m.xxqk.cn article
on parallel softmax / FlashAttention (§1.1, §4.1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "osattn_ref.cpp")
_LIB = os.path.join(_HERE, "libosattn_ref.so")
_lock = threading.Lock()
_lib = None

DTYPE_BF16 = 0
DTYPE_FP32 = 1
DTYPE_FP64 = 2
DTYPE_FP16 = 3


def build(force: bool = False) -> str:
    """Compile ``osattn_ref.cpp`` into ``libosattn_ref.so`` (portable flags)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O3", "-std=c++17", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        vp = ctypes.c_void_p
        lib.osattn_ref_softmax_naive.argtypes = [dp, ctypes.c_int, dp]
        lib.osattn_ref_softmax_safe.argtypes = [dp, ctypes.c_int, dp, dp, dp]
        lib.osattn_ref_online_stats.argtypes = [dp, ctypes.c_int, dp, dp, dp]
        lib.osattn_ref_combine.argtypes = [ctypes.c_double] * 4 + [dp, dp]
        lib.osattn_ref_combine.restype = None
        lib.osattn_ref_lse.argtypes = [ctypes.c_double, ctypes.c_double]
        lib.osattn_ref_lse.restype = ctypes.c_double
        lib.osattn_ref_attention_fwd.argtypes = [
            vp, vp, vp, ctypes.c_int, dp, dp,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_int, vp, vp, ctypes.c_int64, ctypes.c_int]
        lib.osattn_ref_softmax_rows.argtypes = [vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                                dp, dp, ctypes.c_int]
        lib.osattn_ref_attention_bwd.argtypes = [
            vp, vp, vp, vp, ctypes.c_int, dp, dp, dp,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_int, vp, ctypes.c_int]
        lib.osattn_ref_attention_blocked.argtypes = [
            vp, vp, vp, ctypes.c_int, dp, dp,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_int, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        _lib = lib
        return lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _vec(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(-1))


def softmax_naive(x) -> np.ndarray:
    """Two-pass e^x / sum e^x with no max subtraction (ch. 6 §6.1)."""
    x = _vec(x)
    y = np.empty_like(x)
    if _load().osattn_ref_softmax_naive(_dptr(x), x.size, _dptr(y)):
        raise ValueError("invalid input")
    return y


def softmax_safe(x):
    """Three-pass safe softmax (ch. 6 §6.2).  Returns (y, m, l)."""
    x = _vec(x)
    y = np.empty_like(x)
    m = np.zeros(1)
    l = np.zeros(1)
    if _load().osattn_ref_softmax_safe(_dptr(x), x.size, _dptr(y), _dptr(m), _dptr(l)):
        raise ValueError("invalid input")
    return y, float(m[0]), float(l[0])


def online_stats(x):
    """Online (m, l) recurrence one element at a time (ch. 6 §6.3.1).

    Returns (m, l, trace) where trace[t] is l after element t."""
    x = _vec(x)
    m = np.zeros(1)
    l = np.zeros(1)
    trace = np.zeros(max(x.size, 1))
    if _load().osattn_ref_online_stats(_dptr(x), x.size, _dptr(m), _dptr(l), _dptr(trace)):
        raise ValueError("invalid input")
    return float(m[0]), float(l[0]), trace[: x.size]


def combine(a, b):
    """(m, l) combine of ch. 6 §6.4.1; a and b are (m, l) pairs."""
    m = ctypes.c_double()
    l = ctypes.c_double()
    _load().osattn_ref_combine(float(a[0]), float(a[1]), float(b[0]), float(b[1]),
                               ctypes.byref(m), ctypes.byref(l))
    return (m.value, l.value)


def lse(m: float, l: float) -> float:
    """LSE = m + log l (ch. 6 §6.5)."""
    return float(_load().osattn_ref_lse(float(m), float(l)))


def _as_raw(t):
    """Return (contiguous numpy array holding the exact bits, dtype code)."""
    import torch  # local import: numpy inputs need no torch

    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu").contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy(), DTYPE_BF16
        if t.dtype == torch.float16:
            return t.view(torch.int16).numpy(), DTYPE_FP16
        if t.dtype == torch.float32:
            return t.numpy(), DTYPE_FP32
        if t.dtype == torch.float64:
            return t.numpy(), DTYPE_FP64
        raise TypeError(f"unsupported dtype {t.dtype}")
    a = np.ascontiguousarray(t)
    if a.dtype == np.float16:
        return a.view(np.int16), DTYPE_FP16
    if a.dtype == np.float32:
        return a, DTYPE_FP32
    if a.dtype == np.float64:
        return a, DTYPE_FP64
    raise TypeError(f"unsupported dtype {a.dtype}")


def attention_fwd(Q, K, V, scale: float, causal: bool = False, key_len=None,
                  rows=None, nthreads: int = 0):
    """Attention forward by the definition (three-pass safe softmax per row).

    Q: [B,H,Nq,d]; K, V: [B,H,Nkv,d] (torch bf16/fp16/fp32/fp64 or numpy
    fp16/fp32/fp64, all of one dtype; any strides: the values are read).
    key_len: None or B ints.  rows: None for every row (returns O
    [B,H,Nq,d], LSE [B,H,Nq]) or a list of flat row indices (b*H+h)*Nq+i
    (returns O [n,d], LSE [n]).  Results are fp64."""
    q, dt = _as_raw(Q)
    k, dk = _as_raw(K)
    v, dv = _as_raw(V)
    if not (dt == dk == dv):
        raise TypeError("Q, K, V must share one dtype")
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    if k.shape != (B, H, Nkv, d) or v.shape != (B, H, Nkv, d):
        raise ValueError("shape mismatch")
    kl = None
    if key_len is not None:
        kl = np.ascontiguousarray(np.asarray(key_len, dtype=np.int32).reshape(-1))
        if kl.size != B:
            raise ValueError("key_len must have B entries")
    if rows is None:
        O = np.empty((B, H, Nq, d))
        L = np.empty((B, H, Nq))
        rp, n = None, 0
    else:
        ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        O = np.empty((ra.size, d))
        L = np.empty(ra.size)
        rp, n = ra.ctypes.data, ra.size
    rc = _load().osattn_ref_attention_fwd(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dt, _dptr(O), _dptr(L),
        B, H, Nq, Nkv, d, float(scale), int(bool(causal)),
        None if kl is None else kl.ctypes.data, rp, n, int(nthreads))
    if rc:
        raise ValueError("invalid arguments to the oracle")
    return O, L


def attention_bwd(Q, K, V, dO, scale: float, causal: bool = False, key_len=None,
                  nthreads: int = 0):
    """Gradients (dQ, dK, dV) of the attention forward for an upstream
    gradient dO shaped like O, by the chain rule on the definition (see
    osattn_ref.cpp).  Q, dO: [B,H,Nq,d]; K, V: [B,H,Nkv,d], one dtype (as for
    attention_fwd).  Results are fp64."""
    q, dt = _as_raw(Q)
    k, dk = _as_raw(K)
    v, dv = _as_raw(V)
    g, dg = _as_raw(dO)
    if not (dt == dk == dv == dg):
        raise TypeError("Q, K, V, dO must share one dtype")
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    if k.shape != (B, H, Nkv, d) or v.shape != (B, H, Nkv, d) or g.shape != q.shape:
        raise ValueError("shape mismatch")
    kl = None
    if key_len is not None:
        kl = np.ascontiguousarray(np.asarray(key_len, dtype=np.int32).reshape(-1))
        if kl.size != B:
            raise ValueError("key_len must have B entries")
    dQ = np.empty((B, H, Nq, d))
    dK = np.empty((B, H, Nkv, d))
    dV = np.empty((B, H, Nkv, d))
    rc = _load().osattn_ref_attention_bwd(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data, dt, _dptr(dQ), _dptr(dK),
        _dptr(dV), B, H, Nq, Nkv, d, float(scale), int(bool(causal)),
        None if kl is None else kl.ctypes.data, int(nthreads))
    if rc:
        raise ValueError("invalid arguments to the oracle")
    return dQ, dK, dV


def softmax_rows(X, nthreads: int = 0):
    """Row softmax of a [rows, N] tensor (torch bf16/fp16/fp32/fp64 or numpy
    fp16/fp32/fp64) by the three-pass safe softmax, row by row (ch. 6 §6.2); also
    returns the row LSE (§6.5).  All -inf rows give y = 0, LSE = -inf."""
    x, dt = _as_raw(X)
    if x.ndim != 2:
        raise ValueError("X must be [rows, N]")
    rows, N = x.shape
    Y = np.empty((rows, N))
    L = np.empty(rows)
    if _load().osattn_ref_softmax_rows(x.ctypes.data, dt, rows, N, _dptr(Y), _dptr(L),
                                       int(nthreads)):
        raise ValueError("invalid arguments to the oracle")
    return Y, L


def attention_blocked(Q, K, V, scale: float, causal: bool = False, key_len=None,
                      block: int = 16, form: int = 1, nthreads: int = 0):
    """Blocked online attention loop of ch. 6 §6.6 (form 0: block max + beta;
    form 1: exponentiate against the new running max).  All rows."""
    q, dt = _as_raw(Q)
    k, _ = _as_raw(K)
    v, _ = _as_raw(V)
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    kl = None
    if key_len is not None:
        kl = np.ascontiguousarray(np.asarray(key_len, dtype=np.int32).reshape(-1))
    O = np.empty((B, H, Nq, d))
    L = np.empty((B, H, Nq))
    rc = _load().osattn_ref_attention_blocked(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dt, _dptr(O), _dptr(L),
        B, H, Nq, Nkv, d, float(scale), int(bool(causal)),
        None if kl is None else kl.ctypes.data, int(block), int(form), int(nthreads))
    if rc:
        raise ValueError("invalid arguments to the oracle")
    return O, L
