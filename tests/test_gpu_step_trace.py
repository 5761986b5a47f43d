"""The profiling build's per-step clock stamps (osattn_step_trace_read).

Builds libosattn_trace.so (OSATTN_STEP_TRACE=1), runs one causal bf16
forward through it and checks the stamp layout the profiles rely on: per
traced CTA and K/V step, the phases of each role in order, one P stamp per
softmax warp, the correction warps' rescale flag 0 or 1.  The product
library is untouched (it answers OSATTN_ERR_UNSUPPORTED, tests/test_abi.py).
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")


@pytest.mark.gpu
def test_step_trace_stamps_follow_the_kernel_phases():
    from attention_forward_online_gb300 import _build, osattn
    from attention_forward_online_gb300.run_workload import print_cta_times, print_step_trace

    L = ctypes.CDLL(_build.build(step_trace=True))
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    L.osattn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                             vp, i32, vp]
    L.osattn_step_trace_read.argtypes = [vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]
    B, H, N, d = 1, 4, 4096, 128
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    for _ in range(2):
        rc = L.osattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H, N, N, d, d ** -0.5, 1, None, osattn.BF16, None)
        assert rc == osattn.OK
    torch.cuda.synchronize()
    need = ctypes.c_size_t(0)
    L.osattn_step_trace_read(None, 0, ctypes.byref(need))
    assert need.value == (8 * 7 * 128 * 4 + 4096 * 6) * 8
    buf = np.zeros(need.value // 8, dtype=np.int64)
    assert L.osattn_step_trace_read(buf.ctypes.data, buf.nbytes, ctypes.byref(need)) == osattn.OK
    tr = buf[:8 * 7 * 128 * 4].reshape(8, 7, 128, 4)
    ct = buf[8 * 7 * 128 * 4:].reshape(4096, 6)
    # the first CTAs run the longest causal units, one per head: CTAs 0-3 the
    # last 256 rows of heads 0-3 (31 and 32 K/V steps for tiles 0 and 1),
    # CTAs 4-7 the 256 rows before them (29 and 30)
    for cta in range(8):
        sm0, sm1, mma = tr[cta, 0], tr[cta, 1], tr[cta, 2]
        n0, n1 = int((sm0[:, 3] > 0).sum()), int((sm1[:, 3] > 0).sum())
        assert (n0, n1) == ((31, 32) if cta < 4 else (29, 30)), (cta, n0, n1)
        for sm, n in ((sm0, n0), (sm1, n1)):
            assert (np.diff(sm[:n], axis=1) >= 0).all()      # S seen <= in registers <= alpha <= P
            assert (np.diff(sm[:n, 0]) > 0).all()            # steps in order
        assert (np.diff(mma[1:n1, 0]) > 0).all()             # MMA iterations in order
        warps = tr[cta, 3][:n0]
        assert (warps > 0).all()                             # each softmax warp of tile 0 published P
        corr = tr[cta, 5][:n0]
        assert (corr[:, 0] > 0).all() and (corr[:, 2] >= corr[:, 0]).all()
        assert set(np.unique(corr[:, 3])) <= {0, 1}
        assert corr[0, 3] == 0                               # no O to rescale at the first step
    print_step_trace(tr[:2])
    # per-CTA times: the launch's 64 CTAs (4 heads x 16 query blocks), each
    # start <= setup done <= first S <= epilogue <= end, on a valid SM
    n = 4 * 16
    c = ct[:n]
    assert (np.diff(c[:, :5], axis=1) >= 0).all(), c[:4]
    assert ((c[:, 5] >= 0) & (c[:, 5] < 1024)).all()
    print_cta_times(ct, n)
