"""ctypes binding for libosattn (argument marshalling only).

Every step of the forward pass, the backward pass and the row softmax runs
in the library's CUDA kernels, and the host-memory (offload) entry points
copy through the library's own streams; this module checks tensor shapes,
allocates outputs with torch (device and pinned host memory are torch's job
here), and passes raw pointers and the current stream through the C ABI
declared in include/osattn.h.  If libosattn.so is missing the calls raise:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libosattn.so")

BF16 = 0
FP32 = 1
FP16 = 2
OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_TIMEOUT = 4
ERR_SCRATCH_LIMIT = 5
NOALLOC_SCRATCH_BYTES = 32 << 20

EXPORTS = ("osattn_fwd", "osattn_fwd_strided", "osattn_fwd_splitkv",
           "osattn_splitkv_workspace_bytes", "osattn_fwd_splitkv_noalloc",
           "osattn_bwd", "osattn_bwd_strided", "osattn_bwd_workspace_bytes",
           "osattn_fwd_offload", "osattn_bwd_offload", "osattn_softmax_rows",
           "osattn_softmax_rows_offload",
           "osattn_status_string", "osattn_get_device_status",
           "osattn_version", "osattn_set_wait_limit_ns", "osattn_test_wait_timeout",
           "osattn_last_timeout_site", "osattn_step_trace_read")

_lock = threading.Lock()
_lib = None


class OsattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def lib():
    """Load libosattn.so (built in-tree by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; "
                    "g.build()\"` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32 = ctypes.c_void_p, ctypes.c_int
            L.osattn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                     ctypes.c_float, i32, vp, i32, vp]
            L.osattn_fwd.restype = i32
            i64p = ctypes.POINTER(ctypes.c_int64)
            L.osattn_fwd_strided.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                             i64p, i64p, i64p, i64p,
                                             ctypes.c_float, i32, vp, i32, vp]
            L.osattn_fwd_strided.restype = i32
            L.osattn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                             ctypes.c_float, i32, vp, i32, i32, vp,
                                             ctypes.c_size_t, vp]
            L.osattn_fwd_splitkv.restype = i32
            L.osattn_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                     ctypes.c_float, i32, vp, i32, i32, vp]
            L.osattn_fwd_splitkv_noalloc.restype = i32
            L.osattn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                     ctypes.c_float, i32, vp, i32, vp, ctypes.c_size_t, vp]
            L.osattn_bwd.restype = i32
            L.osattn_bwd_strided.argtypes = ([vp] * 9 + [i32] * 5 + [i64p] * 8 +
                                             [ctypes.c_float, i32, vp, i32, vp, ctypes.c_size_t, vp])
            L.osattn_bwd_strided.restype = i32
            L.osattn_fwd_offload.argtypes = ([vp] * 10 + [i32] * 5 + [ctypes.c_float, i32, vp, i32,
                                                                       i32, vp])
            L.osattn_fwd_offload.restype = i32
            L.osattn_bwd_offload.argtypes = ([vp] * 18 + [i32] * 5 + [ctypes.c_float, i32, vp, i32,
                                                                       vp, ctypes.c_size_t, i32, vp])
            L.osattn_bwd_offload.restype = i32
            L.osattn_softmax_rows_offload.argtypes = [vp] * 6 + [ctypes.c_int64, i32, i32,
                                                                 ctypes.c_int64, vp]
            L.osattn_softmax_rows_offload.restype = i32
            L.osattn_bwd_workspace_bytes.argtypes = [i32, i32, i32]
            L.osattn_bwd_workspace_bytes.restype = ctypes.c_size_t
            L.osattn_softmax_rows.argtypes = [vp, vp, vp, ctypes.c_int64, i32, i32, vp]
            L.osattn_softmax_rows.restype = i32
            L.osattn_splitkv_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            L.osattn_splitkv_workspace_bytes.restype = ctypes.c_size_t
            L.osattn_status_string.argtypes = [i32]
            L.osattn_status_string.restype = ctypes.c_char_p
            L.osattn_get_device_status.argtypes = [vp]
            L.osattn_get_device_status.restype = i32
            L.osattn_version.argtypes = []
            L.osattn_version.restype = i32
            L.osattn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.osattn_set_wait_limit_ns.restype = ctypes.c_uint64
            L.osattn_test_wait_timeout.argtypes = [vp]
            L.osattn_test_wait_timeout.restype = i32
            L.osattn_last_timeout_site.argtypes = []
            L.osattn_last_timeout_site.restype = i32
            L.osattn_step_trace_read.argtypes = [vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]
            L.osattn_step_trace_read.restype = i32
            _lib = L
        return _lib


def step_trace():
    """The clock stamps of a profiling build (OSATTN_STEP_TRACE=1; see
    include/osattn.h): (per-step stamps, a numpy int64 array [8, 7, 128, 4];
    per-CTA times, [4096, 6])."""
    import numpy as np

    need = ctypes.c_size_t(0)
    lib().osattn_step_trace_read(None, 0, ctypes.byref(need))
    buf = np.zeros(need.value // 8, dtype=np.int64)
    st = lib().osattn_step_trace_read(buf.ctypes.data, buf.nbytes, ctypes.byref(need))
    if st != OK:
        raise OsattnError(st, "osattn_step_trace_read")
    n = 8 * 7 * 128 * 4
    return buf[:n].reshape(8, 7, 128, 4), buf[n:].reshape(4096, 6)


def status_string(status: int) -> str:
    return lib().osattn_status_string(int(status)).decode()


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def fwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nkv, d, scale, causal,
            key_len_ptr, dtype, stream_handle) -> int:
    """Direct call of osattn_fwd with integer pointers; returns the status."""
    return lib().osattn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(Nq),
                            int(Nkv), int(d), float(scale), int(bool(causal)), key_len_ptr,
                            int(dtype), stream_handle)


def _dtype_code(t) -> int:
    import torch

    codes = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}
    if t.dtype not in codes:
        raise TypeError("q, k, v must all be bf16, all fp16 or all fp32")
    return codes[t.dtype]


def _shapes(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    if tuple(k.shape) != (B, H, Nkv, d) or tuple(v.shape) != (B, H, Nkv, d):
        raise ValueError("k and v must be [B, H, Nkv, d] matching q")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    for t in (q, k, v):
        if not t.is_cuda:
            raise ValueError("q, k, v must be CUDA tensors")
    return B, H, Nq, Nkv, d


def _key_len_ptr(key_len, B):
    import torch

    if key_len is None:
        return None, None
    if key_len.dtype != torch.int32 or not key_len.is_cuda or key_len.numel() != B:
        raise ValueError("key_len must be a CUDA int32 tensor with B entries")
    key_len = key_len.contiguous()
    return key_len, key_len.data_ptr()


def _bhn_strides(t):
    """(b, h, row) element strides of a [B, H, N, d] view whose d axis is
    contiguous, as a ctypes int64[3]."""
    if t.stride(3) != 1:
        raise ValueError("the last (d) axis must have stride 1")
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def fwd(q, k, v, scale: float | None = None, causal: bool = False, key_len=None,
        out=None, lse=None, stream=None):
    """O, LSE = attention forward of CUDA tensors q [B,H,Nq,d], k/v [B,H,Nkv,d].

    dtype bf16, fp16 or fp32 (all three alike).  q, k, v and `out` may be any
    views whose last axis is contiguous (e.g. transposes of [B, N, H, d]);
    contiguous tensors go through osattn_fwd, others through
    osattn_fwd_strided with their strides.  key_len: None or a CUDA int32
    tensor [B].  `out` (q's shape and dtype) and `lse` (contiguous fp32
    [B, H, Nq]) may be given preallocated.  Enqueued on `stream` (default:
    torch's current stream); raises OsattnError if the library rejects the
    call."""
    import torch

    B, H, Nq, Nkv, d = _shapes(q, k, v)
    dtype = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_cuda:
        raise ValueError("out must be a CUDA tensor matching q")
    if tuple(lse.shape) != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be fp32 [B, H, Nq]")
    kl, kl_ptr = _key_len_ptr(key_len, B)
    if all(t.is_contiguous() for t in (q, k, v, out)):
        st = fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                     B, H, Nq, Nkv, d, scale, causal, kl_ptr, dtype, _stream_handle(stream))
        what = "osattn_fwd"
    else:
        qs, ks, vs, os_ = (_bhn_strides(t) for t in (q, k, v, out))
        st = lib().osattn_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                      lse.data_ptr(), B, H, Nq, Nkv, d, qs, ks, vs, os_,
                                      float(scale), int(bool(causal)), kl_ptr, dtype,
                                      _stream_handle(stream))
        what = "osattn_fwd_strided"
    del kl
    if st != OK:
        raise OsattnError(st, what)
    return out, lse


MAX_SPLITS = 128


def splitkv_workspace_bytes(B: int, H: int, Nq: int, d: int, num_splits: int) -> int:
    return int(lib().osattn_splitkv_workspace_bytes(int(B), int(H), int(Nq), int(d),
                                                    int(num_splits)))


def _check_qkv(q, k, v):
    B, H, Nq, Nkv, d = _shapes(q, k, v)
    _dtype_code(q)
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    return B, H, Nq, Nkv, d


def fwd_offload(q_host, k_host, v_host, out_host=None, lse_host=None, q=None, k=None, v=None,
                out=None, lse=None, scale: float | None = None, causal: bool = False,
                key_len=None, heads_per_chunk: int = 0, stream=None):
    """Attention forward of host tensors through osattn_fwd_offload: q_host
    [B,H,Nq,d], k_host/v_host [B,H,Nkv,d] (contiguous CPU tensors, pinned for
    the copies to overlap the compute) are copied in chunks of heads to the
    device buffers q, k, v (allocated when not given), attended, and O/LSE are
    copied back into out_host/lse_host (pinned CPU tensors, allocated when not
    given).  Returns (out_host, lse_host); they are valid once `stream` has
    synchronised.  key_len is a CUDA int32 tensor with B entries or None;
    heads_per_chunk 0 lets the library size the chunks."""
    import torch

    for t in (q_host, k_host, v_host):
        if t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q_host, k_host, v_host must be contiguous 4-D CPU tensors")
    B, H, Nq, d = q_host.shape
    Nkv = k_host.shape[2]
    if tuple(k_host.shape) != (B, H, Nkv, d) or tuple(v_host.shape) != (B, H, Nkv, d):
        raise ValueError("k_host and v_host must be [B, H, Nkv, d] matching q_host")
    if k_host.dtype != q_host.dtype or v_host.dtype != q_host.dtype:
        raise TypeError("q_host, k_host, v_host must share one dtype")
    dtype = _dtype_code(q_host)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", torch.cuda.current_device())
    q = torch.empty(q_host.shape, dtype=q_host.dtype, device=dev) if q is None else q
    k = torch.empty(k_host.shape, dtype=k_host.dtype, device=dev) if k is None else k
    v = torch.empty(v_host.shape, dtype=v_host.dtype, device=dev) if v is None else v
    out = torch.empty(q_host.shape, dtype=q_host.dtype, device=dev) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev) if lse is None else lse
    if out_host is None:
        out_host = torch.empty(q_host.shape, dtype=q_host.dtype).pin_memory()
    if lse_host is None:
        lse_host = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
    for t, ref in ((q, q_host), (k, k_host), (v, v_host), (out, q_host), (out_host, q_host)):
        if tuple(t.shape) != tuple(ref.shape) or t.dtype != ref.dtype or not t.is_contiguous():
            raise ValueError("device buffers and out_host must be contiguous and match the inputs")
    for t in (lse, lse_host):
        if tuple(t.shape) != (B, H, Nq) or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("lse and lse_host must be contiguous fp32 [B, H, Nq]")
    if out_host.is_cuda or lse_host.is_cuda or not all(t.is_cuda for t in (q, k, v, out, lse)):
        raise ValueError("host tensors must be CPU tensors and staging buffers CUDA tensors")
    key_len, kl_ptr = _key_len_ptr(key_len, B)
    st = lib().osattn_fwd_offload(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(),
                                  out_host.data_ptr(), lse_host.data_ptr(), q.data_ptr(),
                                  k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H,
                                  Nq, Nkv, d, float(scale), int(bool(causal)), kl_ptr, dtype,
                                  int(heads_per_chunk), _stream_handle(stream))
    if st != OK:
        raise OsattnError(st, "osattn_fwd_offload")
    return out_host, lse_host


def fwd_splitkv(q, k, v, num_splits: int, scale: float | None = None, causal: bool = False,
                key_len=None, out=None, lse=None, workspace=None, stream=None):
    """Split-KV attention forward (bf16 or fp16): same result as fwd(), the key axis cut
    into num_splits ranges merged by the (m, l) combine.  `workspace` may be a
    preallocated CUDA uint8 tensor of at least splitkv_workspace_bytes(...)
    bytes; otherwise torch allocates one."""
    import torch

    B, H, Nq, Nkv, d = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    need = splitkv_workspace_bytes(B, H, Nq, d, max(int(num_splits), 1))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    key_len, kl_ptr = _key_len_ptr(key_len, B)
    dtype = _dtype_code(q)
    st = lib().osattn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), B, H, Nq, Nkv, d, float(scale),
                                  int(bool(causal)), kl_ptr, dtype, int(num_splits),
                                  workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream))
    if st != OK:
        raise OsattnError(st, "osattn_fwd_splitkv")
    return out, lse


def bwd_workspace_bytes(B: int, H: int, Nq: int) -> int:
    return int(lib().osattn_bwd_workspace_bytes(int(B), int(H), int(Nq)))


def bwd(q, k, v, o, lse, do, scale: float | None = None, causal: bool = False, key_len=None,
        dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of the attention forward for the upstream gradient `do`.

    q, k, v, o, do: CUDA bf16, fp16 or fp32 tensors ([B,H,Nq,d] for q, o, do;
    [B,H,Nkv,d] for k, v), any views whose last axis is contiguous; lse: the
    contiguous fp32 [B,H,Nq] LSE that fwd() returned for the same inputs.
    Contiguous tensors go through osattn_bwd, others through
    osattn_bwd_strided.  Outputs may be given preallocated (any such views);
    `workspace` (a CUDA uint8 tensor of at least bwd_workspace_bytes(B, H,
    Nq) bytes) too."""
    import torch

    B, H, Nq, Nkv, d = _shapes(q, k, v)
    dtype = _dtype_code(q)
    for t in (o, do):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_cuda:
            raise ValueError("o and do must be CUDA tensors shaped and typed like q")
    if tuple(lse.shape) != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be fp32 [B, H, Nq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, ref in ((dq, q), (dk, k), (dv, v)):
        if t.shape != ref.shape or t.dtype != ref.dtype or not t.is_cuda:
            raise ValueError("dq, dk, dv must be CUDA tensors shaped and typed like q, k, v")
    need = bwd_workspace_bytes(B, H, Nq)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    key_len, kl_ptr = _key_len_ptr(key_len, B)
    ts = (q, k, v, o, do, dq, dk, dv)
    ptrs = [t.data_ptr() for t in ts]
    tail = (float(scale), int(bool(causal)), kl_ptr, dtype, workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if all(t.is_contiguous() for t in ts):
        st = lib().osattn_bwd(*ptrs[:5], lse.data_ptr(), *ptrs[5:], B, H, Nq, Nkv, d, *tail)
        what = "osattn_bwd"
    else:
        strides = [_bhn_strides(t) for t in ts]
        st = lib().osattn_bwd_strided(*ptrs[:5], lse.data_ptr(), *ptrs[5:], B, H, Nq, Nkv, d,
                                      *strides, *tail)
        what = "osattn_bwd_strided"
    if st != OK:
        raise OsattnError(st, what)
    return dq, dk, dv


def bwd_offload(q_host, k_host, v_host, o_host, lse_host, do_host, scale: float | None = None,
                causal: bool = False, key_len=None, dq_host=None, dk_host=None, dv_host=None,
                device_buffers=None, workspace=None, heads_per_chunk: int = 0, stream=None):
    """Gradients of host tensors through osattn_bwd_offload: inputs as for
    bwd() but contiguous CPU tensors (pinned for the copies to overlap the
    compute); dq_host, dk_host, dv_host are allocated (pinned) when not given.
    device_buffers, if given, is a tuple of the nine contiguous CUDA staging
    tensors (q, k, v, o, do, dq, dk, dv, lse); otherwise they are allocated.
    Returns (dq_host, dk_host, dv_host), valid once `stream` has
    synchronised."""
    import torch

    ins = (q_host, k_host, v_host, o_host, do_host)
    for t in ins + (lse_host,):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host inputs must be contiguous CPU tensors")
    if q_host.dim() != 4:
        raise ValueError("q_host must be [B, H, Nq, d]")
    B, H, Nq, d = q_host.shape
    Nkv = k_host.shape[2]
    if tuple(k_host.shape) != (B, H, Nkv, d) or tuple(v_host.shape) != (B, H, Nkv, d):
        raise ValueError("k_host and v_host must be [B, H, Nkv, d] matching q_host")
    for t in (o_host, do_host):
        if tuple(t.shape) != tuple(q_host.shape):
            raise ValueError("o_host and do_host must be shaped like q_host")
    for t in ins[1:]:
        if t.dtype != q_host.dtype:
            raise TypeError("host inputs must share one dtype")
    if tuple(lse_host.shape) != (B, H, Nq) or lse_host.dtype != torch.float32:
        raise ValueError("lse_host must be fp32 [B, H, Nq]")
    dtype = _dtype_code(q_host)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", torch.cuda.current_device())
    if device_buffers is None:
        mk = lambda ref: torch.empty(ref.shape, dtype=ref.dtype, device=dev)  # noqa: E731
        device_buffers = (mk(q_host), mk(k_host), mk(v_host), mk(o_host), mk(do_host),
                          mk(q_host), mk(k_host), mk(v_host), mk(lse_host))
    qd, kd, vd, od, dod, dqd, dkd, dvd, lsed = device_buffers
    for t, ref in zip(device_buffers, (q_host, k_host, v_host, o_host, do_host, q_host, k_host,
                                       v_host, lse_host)):
        if (not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(ref.shape)
                or t.dtype != ref.dtype):
            raise ValueError("device buffers must be contiguous CUDA tensors matching the inputs")
    pin = lambda ref: torch.empty(ref.shape, dtype=ref.dtype).pin_memory()  # noqa: E731
    dq_host = pin(q_host) if dq_host is None else dq_host
    dk_host = pin(k_host) if dk_host is None else dk_host
    dv_host = pin(v_host) if dv_host is None else dv_host
    for t, ref in ((dq_host, q_host), (dk_host, k_host), (dv_host, v_host)):
        if t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(ref.shape) or t.dtype != ref.dtype:
            raise ValueError("dq_host, dk_host, dv_host must be contiguous CPU tensors matching the inputs")
    need = bwd_workspace_bytes(B, H, Nq)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    key_len, kl_ptr = _key_len_ptr(key_len, B)
    st = lib().osattn_bwd_offload(
        q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), o_host.data_ptr(),
        do_host.data_ptr(), lse_host.data_ptr(), dq_host.data_ptr(), dk_host.data_ptr(),
        dv_host.data_ptr(), qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(),
        dod.data_ptr(), lsed.data_ptr(), dqd.data_ptr(), dkd.data_ptr(), dvd.data_ptr(), B, H, Nq,
        Nkv, d, float(scale), int(bool(causal)), kl_ptr, dtype, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), int(heads_per_chunk), _stream_handle(stream))
    if st != OK:
        raise OsattnError(st, "osattn_bwd_offload")
    return dq_host, dk_host, dv_host


def softmax_rows(x, out=None, lse=None, want_lse: bool = True, stream=None):
    """Row softmax of a contiguous CUDA [rows, N] bf16/fp16/fp32 tensor (online (m, l)
    normaliser).  Returns (y, lse or None); `out` may be `x` (in place)."""
    import torch

    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA [rows, N] tensor")
    codes = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}
    if x.dtype not in codes:
        raise TypeError("x must be bf16, fp16 or fp32")
    rows, N = x.shape
    out = torch.empty_like(x) if out is None else out
    if want_lse and lse is None:
        lse = torch.empty(rows, dtype=torch.float32, device=x.device)
    dtype = codes[x.dtype]
    st = lib().osattn_softmax_rows(x.data_ptr(), out.data_ptr(),
                                   None if lse is None else lse.data_ptr(), rows, N, dtype,
                                   _stream_handle(stream))
    if st != OK:
        raise OsattnError(st, "osattn_softmax_rows")
    return out, lse


def softmax_rows_offload(x_host, out_host=None, lse_host=None, x=None, out=None, lse=None,
                         want_lse: bool = True, rows_per_chunk: int = 0, stream=None):
    """Row softmax of a contiguous CPU [rows, N] tensor (pinned for the copies
    to overlap) through osattn_softmax_rows_offload; x/out/lse are the device
    staging buffers (allocated when not given), out_host/lse_host the pinned
    results (allocated when not given).  Returns (out_host, lse_host or None),
    valid once `stream` has synchronised."""
    import torch

    if x_host.dim() != 2 or x_host.is_cuda or not x_host.is_contiguous():
        raise ValueError("x_host must be a contiguous CPU [rows, N] tensor")
    codes = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}
    if x_host.dtype not in codes:
        raise TypeError("x_host must be bf16, fp16 or fp32")
    rows, N = x_host.shape
    dev = torch.device("cuda", torch.cuda.current_device())
    x = torch.empty(x_host.shape, dtype=x_host.dtype, device=dev) if x is None else x
    out = torch.empty_like(x) if out is None else out
    out_host = torch.empty(x_host.shape, dtype=x_host.dtype).pin_memory() if out_host is None else out_host
    if want_lse:
        lse = torch.empty(rows, dtype=torch.float32, device=dev) if lse is None else lse
        lse_host = torch.empty(rows, dtype=torch.float32).pin_memory() if lse_host is None else lse_host
    else:
        lse = lse_host = None
    for t in (x, out):
        if not t.is_cuda or not t.is_contiguous() or t.shape != x_host.shape or t.dtype != x_host.dtype:
            raise ValueError("x and out must be contiguous CUDA tensors shaped like x_host")
    if out_host.is_cuda or not out_host.is_contiguous() or out_host.shape != x_host.shape:
        raise ValueError("out_host must be a contiguous CPU tensor shaped like x_host")
    st = lib().osattn_softmax_rows_offload(
        x_host.data_ptr(), out_host.data_ptr(), None if lse_host is None else lse_host.data_ptr(),
        x.data_ptr(), out.data_ptr(), None if lse is None else lse.data_ptr(), rows, N,
        codes[x_host.dtype], int(rows_per_chunk), _stream_handle(stream))
    if st != OK:
        raise OsattnError(st, "osattn_softmax_rows_offload")
    return out_host, lse_host


def get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return lib().osattn_get_device_status(_stream_handle(stream))


def version() -> int:
    return lib().osattn_version()
