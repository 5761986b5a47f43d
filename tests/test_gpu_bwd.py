"""GPU parity of the backward pass (osattn_bwd: dQ, dK, dV) against the fp64
oracle's gradients, on the forward outputs (O, LSE) of the library itself.

Gate per gradient tensor g (reading c18):
    |g - g_ref| <= 2e-2 |g_ref| + t * rms(g_ref) + half an ulp of g_ref + 1e-5,
with t = 8e-2 for bf16 and 1.5e-2 for fp16.  fp32 (SIMT kernels, fp32
throughout) is gated by |g - g_ref| <= 1e-4 |g_ref| + 1e-4 rms(g_ref) + 1e-6:
its only departures from exact arithmetic are fp32 roundings, and the
largest of them, a d-term score dot product (relative error below
d * 2^-24 of sum |q_k k_k|, about 8e-5 in the exponent for d = 128 and the
inputs below), bounds the relative error of P and hence of each gradient.  The kernels round P and dS to
the input type before the MMAs (unit roundoff u = 2^-9 for bf16, 2^-12 for
fp16), read D from the 16-bit O of the forward pass, accumulate in fp32 and
round the result once more.  Each row of dS sums to zero, so dQ and dK are
cancellations whose rounding error is a fraction of the gradient's rms
rather than of the element: an fp64 model of exactly these roundings puts
the largest error at 5.3 % of rms for bf16 and 0.84 % for fp16 on the cases
below, and t is 1.5 times that.  The 1e-5 floor covers gradients that are
exactly zero (a single visible key): there dP and D are the same d-term dot
product summed in two different fp32 orders, whose difference (about
d * 2^-24 for unit-scale inputs) becomes a tiny nonzero dS.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_online_gb300 import osattn
from attention_forward_online_gb300.inputs import make_qkv

from _compare import half_ulp_bf16, half_ulp_fp16

pytestmark = pytest.mark.gpu
DEV = "cuda"
KIND = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}


T_RMS = {"bf16": 8e-2, "fp16": 1.5e-2, "fp32": 1e-4}


def check_grad(g, ref, kind, name):
    g = np.asarray(g, dtype=np.float64)
    assert not np.isnan(g).any(), f"NaN in {name}"
    rms = math.sqrt(float((ref ** 2).mean())) if ref.size else 0.0
    if kind == "fp32":
        gate = 1e-4 * np.abs(ref) + T_RMS[kind] * rms + 1e-6
    else:
        ulp = half_ulp_bf16(ref) if kind == "bf16" else half_ulp_fp16(ref)
        gate = 2e-2 * np.abs(ref) + T_RMS[kind] * rms + ulp + 1e-5
    err = np.abs(g - ref)
    bad = err > gate
    assert not bad.any(), (f"{name}: error {err.max():.3e} over gate at {np.argwhere(bad)[:4].tolist()} "
                           f"(ref {ref[bad][:4]}, got {g[bad][:4]}, rms {rms:.3e})")
    return float(err.max()), rms


def run_case(B, H, Nq, Nkv, d, causal, kl, dtype, seed):
    q, k, v = make_qkv(B, H, Nq, Nkv, d, dtype, seed=seed, q_std=1.5)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(B, H, Nq, d, generator=g).to(dtype)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    kld = None if kl is None else torch.tensor(kl, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(d)
    o, lse = osattn.fwd(qd, kd, vd, scale=scale, causal=causal, key_len=kld)
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    osattn.bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal, key_len=kld, dq=dq, dk=dk, dv=dv)
    assert osattn.get_device_status() == osattn.OK
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, scale, causal, kl)
    kind = KIND[dtype]
    stats = [check_grad(t.double().cpu().numpy(), r, kind, n)
             for t, r, n in ((dq, rq, "dQ"), (dk, rk, "dK"), (dv, rv, "dV"))]
    return stats, (dq, dk, dv)


CASES = [
    # B, H, Nq, Nkv, d, causal, key_len
    (1, 1, 128, 128, 64, False, None),
    (1, 2, 256, 256, 128, True, None),
    (2, 2, 200, 333, 64, False, [333, 100]),
    (1, 1, 130, 300, 128, True, None),
    (1, 1, 300, 130, 64, True, None),
    (1, 1, 1, 1, 64, False, None),
    (2, 1, 257, 257, 128, True, [257, 129]),
    (1, 2, 384, 512, 128, False, [400]),
]


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[5] else "") + f"kl{c[6]}")
def test_bwd_matches_oracle(case, dtype):
    B, H, Nq, Nkv, d, causal, kl = case
    stats, _ = run_case(B, H, Nq, Nkv, d, causal, kl, dtype, seed=4000 + Nq + Nkv + d)
    print(case, KIND[dtype], "max err / rms (dQ, dK, dV):", stats)


def test_bwd_fully_masked_batch_has_zero_gradients():
    B, H, N, d = 2, 2, 200, 64
    q, k, v = make_qkv(B, H, N, N, d, torch.bfloat16, seed=77)
    do = torch.randn(B, H, N, d).to(torch.bfloat16)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    kld = torch.tensor([N, 0], dtype=torch.int32, device=DEV)
    o, lse = osattn.fwd(qd, kd, vd, key_len=kld)
    dq, dk, dv = osattn.bwd(qd, kd, vd, o, lse, dod, key_len=kld)
    assert osattn.get_device_status() == osattn.OK
    for t in (dq, dk, dv):
        assert torch.all(t[1] == 0).item()
        assert torch.isfinite(t.float()).all().item()
    assert dq[0].abs().max().item() > 0


def test_bwd_deterministic():
    stats, (dq1, dk1, dv1) = run_case(1, 4, 512, 512, 128, True, None, torch.bfloat16, seed=91)
    q, k, v = make_qkv(1, 4, 512, 512, 128, torch.bfloat16, seed=91, q_std=1.5)
    g = torch.Generator().manual_seed(92)
    do = torch.randn(1, 4, 512, 128, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    o, lse = osattn.fwd(qd, kd, vd, causal=True)
    dq2, dk2, dv2 = osattn.bwd(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    for a, b in ((dq1, dq2), (dk1, dk2), (dv1, dv2)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bwd_full_size_workloads_sampled_heads():
    # The backward workloads at full size, in the launch configuration the
    # bench times: whole heads of the B8 H40 2048 d128 problem against the
    # oracle; for the causal 16K problem, dQ of the first 2048 query rows (a
    # causal row only depends on keys up to its own index, so a prefix of the
    # problem has the same dQ rows) and finiteness everywhere.
    from attention_forward_online_gb300.inputs import BWD_WORKLOADS, make_grad_out, make_inputs

    for name, heads, prefix in (("bwd_bf16_b8_h40_n2048_d128", 2, None),
                                ("bwd_bf16_causal_b1_h32_n16384_d128_qstd3", 2, 2048)):
        w = BWD_WORKLOADS[name]
        q, k, v, _ = make_inputs(w)
        do = make_grad_out(w)
        qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
        o, lse = osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal)
        dq, dk, dv = osattn.bwd(qd, kd, vd, o, lse, dod, scale=w.scale, causal=w.causal)
        assert osattn.get_device_status() == osattn.OK
        for t in (dq, dk, dv):
            assert torch.isfinite(t.float()).all().item()
        n = prefix or w.Nq
        sl = (slice(w.B - 1, w.B), slice(w.H - heads, w.H), slice(0, n))
        rq, rk, rv = oracle.attention_bwd(q[sl], k[sl], v[sl], do[sl], w.scale, w.causal)
        out = [check_grad(dq[sl].double().cpu().numpy(), rq, "bf16", "dQ")]
        if prefix is None:
            out.append(check_grad(dk[sl].double().cpu().numpy(), rk, "bf16", "dK"))
            out.append(check_grad(dv[sl].double().cpu().numpy(), rv, "bf16", "dV"))
        print(name, "max err / rms:", out)


def _bnhd(t):
    """The same values stored as [B, N, H, d], returned as a [B, H, N, d] view."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("case", [(2, 3, 300, 333, 64, False, [333, 100]), (1, 2, 257, 257, 128, True, None)],
                         ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[5] else ""))
def test_bwd_strided_matches_contiguous_bitwise(case, dtype):
    # Q, K, V, O, dO read and dQ, dK, dV written in the [B, N, H, d] layout
    # (osattn_bwd_strided) give the contiguous call's gradients bit for bit,
    # and therefore pass the oracle gate too.
    B, H, Nq, Nkv, d, causal, kl = case
    stats, (dq1, dk1, dv1) = run_case(B, H, Nq, Nkv, d, causal, kl, dtype, seed=4000 + Nq + Nkv + d)
    q, k, v = make_qkv(B, H, Nq, Nkv, d, dtype, seed=4000 + Nq + Nkv + d, q_std=1.5)
    g = torch.Generator().manual_seed(4000 + Nq + Nkv + d + 1)
    do = torch.randn(B, H, Nq, d, generator=g).to(dtype)
    qd, kd, vd, dod = (_bnhd(t.to(DEV)) for t in (q, k, v, do))
    assert not qd.is_contiguous()
    kld = None if kl is None else torch.tensor(kl, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(d)
    o, lse = osattn.fwd(qd, kd, vd, scale=scale, causal=causal, key_len=kld)
    o = _bnhd(o)
    outs = [torch.full((B, n, H, d), float("nan"), dtype=dtype, device=DEV).transpose(1, 2)
            for n in (Nq, Nkv, Nkv)]
    osattn.bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal, key_len=kld,
               dq=outs[0], dk=outs[1], dv=outs[2])
    assert osattn.get_device_status() == osattn.OK
    torch.cuda.synchronize()
    bits = torch.int32 if dtype == torch.float32 else torch.int16
    for a, b in zip((dq1, dk1, dv1), outs):
        assert torch.equal(a.view(bits), b.contiguous().view(bits))
