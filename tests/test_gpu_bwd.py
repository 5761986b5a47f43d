"""GPU parity of the backward pass (osattn_bwd: dQ, dK, dV) against the fp64
oracle's gradients, on the forward outputs (O, LSE) of the library itself.

16-bit gates per gradient tensor g (reading c18), from the rounding model in
tests/_bwd_model.py, which tests/test_bwd_rounding_model.py checks on the
CPU:
    elementwise  |g - g_ref| <= t_max rms(g_ref) + half an ulp of g_ref + 1e-5
    aggregate    rms(g - g_ref) <= t_rms rms(g_ref)
with (t_max, t_rms) per tensor 1.5 times what the model of the kernels'
roundings (P and dS to 16 bits, D from the stored 16-bit O, the forward's
16-bit P and O) predicts on the very cases below.  fp32 (SIMT kernels,
fp32 throughout) is gated by |g - g_ref| <= 1e-4 |g_ref| + 1e-4 rms(g_ref)
+ 1e-6: its only departures from exact arithmetic are fp32 roundings, and
the largest of them, a d-term score dot product (relative error below
d * 2^-24 of sum |q_k k_k|, about 8e-5 in the exponent for d = 128 and the
inputs below), bounds the relative error of P and hence of each gradient.
"""
import math

import numpy as np
import pytest
import torch

import _bwd_model as M
import oracle
from attention_forward_online_gb300 import osattn
from attention_forward_online_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda"
KIND = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}


def check_grad(g, ref, kind, name, gates=None):
    g = np.asarray(g, dtype=np.float64)
    if kind != "fp32":
        gates = gates or M.GATES["small"][kind]
        return M.check_grad_gate(g, ref, gates[name], kind, name)
    assert not np.isnan(g).any(), f"NaN in {name}"
    rms = math.sqrt(float((ref ** 2).mean())) if ref.size else 0.0
    gate = 1e-4 * np.abs(ref) + 1e-4 * rms + 1e-6
    err = np.abs(g - ref)
    bad = err > gate
    assert not bad.any(), (f"{name}: error {err.max():.3e} over gate at {np.argwhere(bad)[:4].tolist()} "
                           f"(ref {ref[bad][:4]}, got {g[bad][:4]}, rms {rms:.3e})")
    return float(err.max()), rms


def run_case(B, H, Nq, Nkv, d, causal, kl, dtype, seed):
    q, k, v, do = M.small_case_inputs((B, H, Nq, Nkv, d, causal, kl), dtype, seed)
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


CASES = M.SMALL_CASES  # B, H, Nq, Nkv, d, causal, key_len


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[5] else "") + f"kl{c[6]}")
def test_bwd_matches_oracle(case, dtype):
    B, H, Nq, Nkv, d, causal, kl = case
    stats, _ = run_case(B, H, Nq, Nkv, d, causal, kl, dtype, seed=M.small_case_seed(case))
    print(case, KIND[dtype], "(max err, rms err) / rms (dQ, dK, dV):", stats)


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
    B, H, Nq, Nkv, d, causal, kl = M.DETERMINISM_CASE
    stats, (dq1, dk1, dv1) = run_case(B, H, Nq, Nkv, d, causal, kl, torch.bfloat16, seed=91)
    q, k, v, do = M.small_case_inputs(M.DETERMINISM_CASE, torch.bfloat16, 91)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    o, lse = osattn.fwd(qd, kd, vd, causal=True)
    dq2, dk2, dv2 = osattn.bwd(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    for a, b in ((dq1, dq2), (dk1, dk2), (dv1, dv2)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name", M.FULL_SIZE)
def test_bwd_full_size_workloads_whole_heads(name):
    # The backward workloads at full size, in the launch configuration the
    # bench times; dQ, dK and dV of the whole last two heads against the
    # oracle (the causal 16K rows at full length), finiteness everywhere.
    from attention_forward_online_gb300.inputs import BWD_WORKLOADS, make_grad_out, make_inputs

    w = BWD_WORKLOADS[name]
    q, k, v, _ = make_inputs(w)
    do = make_grad_out(w)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), do.to(DEV)
    o, lse = osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal)
    dq, dk, dv = osattn.bwd(qd, kd, vd, o, lse, dod, scale=w.scale, causal=w.causal)
    assert osattn.get_device_status() == osattn.OK
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all().item()
    sl = (slice(w.B - 1, w.B), slice(w.H - M.FULL_SIZE_HEADS, w.H))
    ref = oracle.attention_bwd(q[sl], k[sl], v[sl], do[sl], w.scale, w.causal)
    out = [check_grad(t[sl].double().cpu().numpy(), r, "bf16", n, M.GATES[name]["bf16"])
           for t, r, n in zip((dq, dk, dv), ref, ("dQ", "dK", "dV"))]
    print(name, "(max err, rms err) / rms (dQ, dK, dV):", out)


def _bnhd(t):
    """The same values stored as [B, N, H, d], returned as a [B, H, N, d] view."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("case", M.STRIDED_CASES,
                         ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[5] else ""))
def test_bwd_strided_matches_contiguous_bitwise(case, dtype):
    # Q, K, V, O, dO read and dQ, dK, dV written in the [B, N, H, d] layout
    # (osattn_bwd_strided) give the contiguous call's gradients bit for bit,
    # and therefore pass the oracle gate too.
    B, H, Nq, Nkv, d, causal, kl = case
    stats, (dq1, dk1, dv1) = run_case(B, H, Nq, Nkv, d, causal, kl, dtype, seed=M.small_case_seed(case))
    q, k, v, do = M.small_case_inputs(case, dtype)
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
