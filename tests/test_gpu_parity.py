"""GPU parity: libosattn (through the C ABI) against the fp64 oracle.

Small shapes are compared element by element on every output; the five
specified workloads run at full size in the launch configuration the bench
times, compared on sampled rows the oracle computes one by one (every
128-row tile edge of one head included) plus properties that hold at any
size.  Tolerances: see tests/_compare.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_online_gb300 import osattn
from attention_forward_online_gb300.inputs import WORKLOADS, make_inputs, make_qkv, sample_rows

from _compare import check

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run_gpu(q, k, v, scale, causal, key_len):
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    kl = None if key_len is None else torch.as_tensor(key_len, dtype=torch.int32).to(DEV)
    O = torch.full_like(qd, float("nan"))
    L = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=DEV)
    osattn.fwd(qd, kd, vd, scale=scale, causal=causal, key_len=kl, out=O, lse=L)
    st = osattn.get_device_status()
    assert st == osattn.OK, osattn.status_string(st)
    return O.double().cpu().numpy(), L.double().cpu().numpy()


KIND = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}


def kind_of(t):
    return KIND[t.dtype]


EDGE = [
    # B, H, Nq, Nkv, d, causal, key_len, q_std
    (1, 1, 1, 1, 64, False, None, 1.0),
    (1, 2, 1, 300, 128, False, None, 1.0),
    (2, 2, 200, 333, 64, False, [333, 150], 1.0),
    (1, 1, 333, 200, 128, True, None, 1.0),
    (1, 1, 130, 300, 64, True, None, 1.0),
    (3, 1, 257, 257, 128, True, [257, 129, 0], 1.0),
    (1, 1, 128, 128, 64, False, [127], 1.0),
    (1, 1, 256, 256, 64, False, [128], 1.0),
    (1, 1, 256, 256, 128, False, [129], 1.0),
    (2, 1, 50, 50, 64, True, [1, 50], 1.0),
    (1, 3, 384, 384, 128, True, None, 1.0),
    (1, 2, 300, 700, 128, False, [1000], 8.0),
    (2, 2, 512, 512, 64, True, [512, 3], 3.0),
    (1, 1, 640, 1000, 128, False, [0], 1.0),
]


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("case", EDGE, ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[5] else "") + f"kl{c[6]}")
def test_edge_shapes_full_parity(case, dtype):
    B, H, Nq, Nkv, d, causal, kl, q_std = case
    q, k, v = make_qkv(B, H, Nq, Nkv, d, dtype, seed=1000 + Nq + Nkv, q_std=q_std)
    scale = 1 / math.sqrt(d)
    O, L = run_gpu(q, k, v, scale, causal, kl)
    Oref, Lref = oracle.attention_fwd(q, k, v, scale, causal, kl)
    check(O, L, Oref, Lref, kind_of(q))


SCALES = [
    # B, H, Nq, Nkv, d, causal, key_len, scale
    (1, 2, 300, 700, 128, False, None, -1 / math.sqrt(128)),
    (2, 1, 384, 384, 64, True, [384, 200], -1 / math.sqrt(64)),
    (1, 1, 257, 513, 128, True, None, -2.0),
    (1, 2, 200, 333, 64, False, [333], 0.0),
    (1, 1, 300, 300, 128, True, None, 0.0),
    (1, 1, 256, 640, 64, False, None, 2.0),
]


# fp32 runs the cases with |scale| <= 1/sqrt(d) only: its 1e-5 gate is the
# stated fp32 tolerance for logits of std up to 8, and a scale of 2 at d = 128
# gives logits of std ~23, where rounding one 128-term fp32 dot product alone
# moves the LSE by ~1e-5.
SCALE_RUNS = [(c, dt) for c in SCALES for dt in KIND
              if dt is not torch.float32 or abs(c[7]) <= 1 / math.sqrt(c[4])]


@pytest.mark.parametrize(
    "case,dtype", SCALE_RUNS,
    ids=["x".join(map(str, c[:5])) + ("c" if c[5] else "") + f"s{c[7]:.3g}-{KIND[dt]}"
         for c, dt in SCALE_RUNS])
def test_negative_zero_and_large_scale_full_parity(case, dtype):
    """The scale enters the softmax as s * scale: for a negative scale the
    row max of s * scale is scale times the row MIN of s, which the bf16/fp16
    kernel takes from its tensor-memory loads (the min reduction) on unmasked
    tiles; zero gives uniform weights.  Every output against the oracle."""
    B, H, Nq, Nkv, d, causal, kl, scale = case
    q, k, v = make_qkv(B, H, Nq, Nkv, d, dtype, seed=2000 + Nq + Nkv, q_std=1.0)
    O, L = run_gpu(q, k, v, scale, causal, kl)
    Oref, Lref = oracle.attention_fwd(q, k, v, scale, causal, kl)
    check(O, L, Oref, Lref, kind_of(q))


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
def test_worked_example_through_kernel(dtype):
    # Logits (1, 5, 3) for one query (chapter 6 §6.3.2), V = identity on the
    # first three columns, so O[0:3] is the printed probability vector.
    d = 64
    q = torch.zeros(1, 1, 1, d)
    q[0, 0, 0, 0] = 1.0
    k = torch.zeros(1, 1, 3, d)
    k[0, 0, :, 0] = torch.tensor([1.0, 5.0, 3.0])
    v = torch.zeros(1, 1, 3, d)
    v[0, 0, 0, 0] = v[0, 0, 1, 1] = v[0, 0, 2, 2] = 1.0
    q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    O, L = run_gpu(q, k, v, 1.0, False, None)
    Oref, Lref = oracle.attention_fwd(q, k, v, 1.0)
    check(O, L, Oref, Lref, kind_of(q))
    np.testing.assert_allclose(O[0, 0, 0, :3], [0.0159, 0.8668, 0.1173], atol=1e-4 + 4e-3)
    assert abs(L[0, 0, 0] - (5 + math.log(1.1536))) < 1e-3


def test_config_fp32_b1_h1_n128_d64_full():
    w = WORKLOADS["fp32_b1_h1_n128_d64"]
    q, k, v, kl = make_inputs(w)
    O, L = run_gpu(q, k, v, w.scale, w.causal, kl)
    Oref, Lref = oracle.attention_fwd(q, k, v, w.scale, w.causal, kl)
    stats = check(O, L, Oref, Lref, "fp32")
    print(w.name, stats)


def test_config_bf16_b2_h4_n1024_keypad_full():
    w = WORKLOADS["bf16_b2_h4_n1024_d64_keypad"]
    q, k, v, kl = make_inputs(w)
    O, L = run_gpu(q, k, v, w.scale, w.causal, kl.tolist())
    Oref, Lref = oracle.attention_fwd(q, k, v, w.scale, w.causal, kl.tolist())
    print(w.name, check(O, L, Oref, Lref, "bf16"))


def test_fully_masked_row_call():
    # The extra row of the key-padding workload: one query whose keys are
    # all masked (key_len 0) -> O = 0, LSE = -inf, no NaN.
    q, k, v = make_qkv(1, 1, 1, 1024, 64, torch.bfloat16, seed=5)
    O, L = run_gpu(q, k, v, 0.125, False, [0])
    assert np.all(O == 0.0) and L[0, 0, 0] == -np.inf
    # and appended as a third batch entry of the workload itself
    q, k, v = make_qkv(3, 4, 1024, 1024, 64, torch.bfloat16, seed=1)
    O, L = run_gpu(q, k, v, 0.125, False, [1024, 724, 0])
    assert np.all(O[2] == 0.0) and np.all(L[2] == -np.inf)
    assert not np.isnan(O).any() and np.isfinite(L[:2]).all()


@pytest.mark.parametrize("name", ["bf16_causal_b4_h16_n4096_d64", "bf16_b8_h40_n2048_d128",
                                  "bf16_causal_b1_h32_n16384_d128_qstd3"])
def test_config_full_size_sampled(name):
    w = WORKLOADS[name]
    q, k, v, kl = make_inputs(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O = torch.full_like(qd, float("nan"))
    L = torch.full((w.B, w.H, w.Nq), float("nan"), dtype=torch.float32, device=DEV)
    osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal, out=O, lse=L)
    assert osattn.get_device_status() == osattn.OK
    # properties at full size: every element written and finite, and each
    # output a convex combination of V rows (bf16 rounding allowed for).
    assert not torch.isnan(O).any().item() and torch.isfinite(L).all().item()
    assert (O.float().abs().amax() <= v.float().abs().amax().to(DEV) * 1.01).item()
    rows = sample_rows(w.B, w.H, w.Nq, 200, seed=w.seed)
    Oref, Lref = oracle.attention_fwd(q, k, v, w.scale, w.causal, None, rows=rows)
    Og = O.reshape(-1, w.d)[torch.tensor(rows, device=DEV)].double().cpu().numpy()
    Lg = L.reshape(-1)[torch.tensor(rows, device=DEV)].double().cpu().numpy()
    print(name, len(rows), "rows", check(Og, Lg, Oref, Lref, "bf16"))


def test_deterministic_and_stream_ordered():
    q, k, v = make_qkv(2, 3, 700, 900, 128, torch.bfloat16, seed=77)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        O1, L1 = osattn.fwd(qd, kd, vd, causal=True)
        O2, L2 = osattn.fwd(qd, kd, vd, causal=True)
    s.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_output_guard_bands_untouched():
    B, H, N, d = 1, 2, 300, 64
    for dtype in (torch.bfloat16, torch.float32):
        q, k, v = make_qkv(B, H, N, N, d, dtype, seed=9)
        qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
        pad = 4096
        obuf = torch.full((pad + B * H * N * d + pad,), 7.0, dtype=dtype, device=DEV)
        lbuf = torch.full((pad + B * H * N + pad,), 7.0, dtype=torch.float32, device=DEV)
        O = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
        L = lbuf[pad:pad + B * H * N].view(B, H, N)
        osattn.fwd(qd, kd, vd, causal=True, out=O, lse=L)
        torch.cuda.synchronize()
        assert torch.all(obuf[:pad] == 7.0) and torch.all(obuf[-pad:] == 7.0)
        assert torch.all(lbuf[:pad] == 7.0) and torch.all(lbuf[-pad:] == 7.0)


def test_device_side_validation_errors():
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(osattn.OsattnError) as e:
        osattn.fwd(q, q, q, scale=float("nan"))
    assert e.value.status == osattn.ERR_INVALID_ARG
    # an output view that starts 2 bytes past a 16-byte boundary
    buf = torch.zeros(8 * 64 + 1, dtype=torch.bfloat16, device=DEV)
    O = buf[1:].view(1, 1, 8, 64)
    with pytest.raises(osattn.OsattnError) as e:
        osattn.fwd(q, q, q, out=O)
    assert e.value.status == osattn.ERR_INVALID_ARG
    q96 = torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(osattn.OsattnError) as e:
        osattn.fwd(q96, q96, q96)
    assert e.value.status == osattn.ERR_UNSUPPORTED


def test_wait_timeout_reports_status_and_recovers():
    # A kernel waits on an mbarrier nobody arrives on; the bounded wait gives
    # up after the (shortened) limit and reports OSATTN_ERR_TIMEOUT.  The
    # context stays usable: a forward call afterwards still matches.
    L = osattn.lib()
    assert osattn.get_device_status() == osattn.OK
    prev = L.osattn_set_wait_limit_ns(2_000_000)  # 2 ms
    try:
        assert L.osattn_test_wait_timeout(osattn._stream_handle(None)) == osattn.OK
        assert osattn.get_device_status() == osattn.ERR_TIMEOUT
        assert osattn.get_device_status() == osattn.OK  # cleared
    finally:
        L.osattn_set_wait_limit_ns(prev)
    q, k, v = make_qkv(1, 1, 130, 130, 64, torch.bfloat16, seed=3)
    O, Lg = run_gpu(q, k, v, 0.125, True, None)
    Oref, Lref = oracle.attention_fwd(q, k, v, 0.125, True)
    check(O, Lg, Oref, Lref, "bf16")


@pytest.mark.parametrize("name", ["bf16_causal_b4_h16_n4096_d64", "bf16_b8_h40_n2048_d128",
                                  "bf16_causal_b1_h32_n16384_d128_qstd3"])
def test_config_full_size_every_row(name):
    # The three large workloads at full size, every output row against the
    # oracle (about 3 TFLOP of fp64 work in all, multithreaded over rows),
    # in the launch configuration the bench times.
    w = WORKLOADS[name]
    q, k, v, kl = make_inputs(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O = torch.full_like(qd, float("nan"))
    L = torch.full((w.B, w.H, w.Nq), float("nan"), dtype=torch.float32, device=DEV)
    osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal, out=O, lse=L)
    assert osattn.get_device_status() == osattn.OK
    Og = O.double().cpu().numpy()
    Lg = L.double().cpu().numpy()
    del O, L
    Oref, Lref = oracle.attention_fwd(q, k, v, w.scale, w.causal, None)
    print(name, "every row", check(Og, Lg, Oref, Lref, "bf16"))


def test_causal_unit_groups_with_a_partial_last_group():
    # Causal units run longest first within groups of heads sized to 32 MB
    # of K/V: at N = 8192, d = 128 a group is 8 heads, so 12 heads make a
    # full group and a partial one.  Every unit must be computed (outputs
    # are NaN-prefilled) and sampled rows must match the oracle.
    B, H, N, d = 1, 12, 8192, 128
    q, k, v = make_qkv(B, H, N, N, d, torch.bfloat16, seed=123, q_std=2.0)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O = torch.full_like(qd, float("nan"))
    L = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=DEV)
    scale = 1 / math.sqrt(d)
    osattn.fwd(qd, kd, vd, scale=scale, causal=True, out=O, lse=L)
    assert osattn.get_device_status() == osattn.OK
    assert not torch.isnan(O).any().item() and torch.isfinite(L).all().item()
    rows = sample_rows(B, H, N, 600, seed=5)
    Oref, Lref = oracle.attention_fwd(q, k, v, scale, True, None, rows=rows)
    idx = torch.tensor(rows, device=DEV)
    check(O.reshape(-1, d)[idx].double().cpu().numpy(), L.reshape(-1)[idx].double().cpu().numpy(),
          Oref, Lref, "bf16")
    # the backward kernels order their causal CTAs the same way
    g = torch.Generator().manual_seed(124)
    dod = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).to(DEV)
    grads = [torch.full_like(t, float("nan")) for t in (qd, kd, vd)]
    osattn.bwd(qd, kd, vd, O, L, dod, scale=scale, causal=True, dq=grads[0], dk=grads[1],
               dv=grads[2])
    assert osattn.get_device_status() == osattn.OK
    for t in grads:
        assert torch.isfinite(t.float()).all().item()


@pytest.mark.parametrize("name,n_rows", [("bf16_causal_b4_h16_n4096_d64", 0),
                                         ("bf16_causal_b1_h32_n16384_d128_qstd3", 4000)])
def test_kernel_arithmetic_within_raw_1e2_before_output_rounding(name, n_rows):
    # The 1e-2 gate on O holds for the kernel's arithmetic itself; the half
    # bf16 ulp added by the gate only covers rounding the output.  The
    # split-KV entry point with one range runs the same kernel but writes
    # O / l in fp32 to the caller's workspace (before the combine rounds it
    # to bf16): that fp32 O must be within a raw 1e-2 of the oracle.
    w = WORKLOADS[name]
    q, k, v, _ = make_inputs(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    ws = torch.empty(osattn.splitkv_workspace_bytes(w.B, w.H, w.Nq, w.d, 1), dtype=torch.uint8,
                     device=DEV)
    osattn.fwd_splitkv(qd, kd, vd, 1, scale=w.scale, causal=w.causal, workspace=ws)
    assert osattn.get_device_status() == osattn.OK
    n_o = w.B * w.H * w.Nq * w.d
    o32 = ws[:4 * n_o].view(torch.float32).reshape(w.B * w.H * w.Nq, w.d)
    if n_rows:
        rows = sample_rows(w.B, w.H, w.Nq, n_rows, seed=w.seed + 11)
        Oref, _ = oracle.attention_fwd(q, k, v, w.scale, w.causal, None, rows=rows)
        got = o32[torch.tensor(rows, device=DEV)].double().cpu().numpy()
    else:
        Oref, _ = oracle.attention_fwd(q, k, v, w.scale, w.causal, None)
        Oref = Oref.reshape(-1, w.d)
        got = o32.double().cpu().numpy()
    err = float(np.abs(got - Oref).max())
    print(name, "fp32 O before output rounding: max-abs error", err)
    assert err <= 1e-2
