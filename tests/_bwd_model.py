"""A model of the roundings the 16-bit backward kernels make, and the
gradient gates it justifies (test infrastructure, CPU only).

The backward pass has no tolerance of its own in the method's statement, so
its gates are derived here.  The model takes the exact gradients of the
attention definition (the chain rule: P = exp(s - LSE), D = rowsum(P dP),
dS = P (dP - D), dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K) and
inserts the roundings that the library's 16-bit path makes, and only those:

  forward   P rounded to the 16-bit type against the running row max of the
            128-key tiles seen so far, O = sum P V / l with the fp32 row
            sum of the unrounded P, O stored in the 16-bit type;
  D         = rowsum(dO * O) read from that stored O (not rowsum(P dP));
  dV        from P rounded to the 16-bit type;
  dK, dQ    from dS = P (dP - D) rounded to the 16-bit type (P itself kept
            at full precision, as the kernels keep it in fp32 registers);
  outputs   dQ, dK, dV stored in the 16-bit type.

Products are accumulated exactly (fp64 here, fp32 in the kernels: fp32 sums
over at most 16384 terms add ~1e-5 relative, far below the 16-bit steps).
Everything else is exact fp64.  The unrounded path of the same code equals
the fp64 oracle's gradients (checked in test_bwd_rounding_model.py).

Two gates per gradient tensor g against the oracle's g_ref, with
rms = rms(g_ref) and hu(x) half an ulp of x in the 16-bit type:
  elementwise  |g - g_ref| <= t_max * rms + hu(g_ref) + 1e-5
  aggregate    rms(g - g_ref) <= t_rms * rms
t_max and t_rms are 1.5 times the model's max (|error| - hu(g_ref)) / rms
and rms(error) / rms over the cases each gate is used on (the margin covers the
fp32 arithmetic and ex2 approximation the model leaves out; they move a
16-bit rounding only where a value lies within ~1e-6 of a rounding boundary).
The 1e-5 floor covers gradients that are exactly zero (a single visible
key), where the kernels' dP and D are one dot product summed in two fp32
orders.  The aggregate gate is the sharp one: a kernel error worth a
percent of the gradient's rms moves rms(error) far beyond 1.5 times the
rounding noise, which is ~0.2 % of rms.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from _compare import half_ulp_bf16, half_ulp_fp16

# Query rows per block of the model (bounds its memory at long sequences).
_ROWS = 1024
# Key tile of the forward kernel: its running row max advances per tile.
_KEY_TILE = 128


def round16(x, kind: str):
    """fp64 -> fp32 -> 16-bit (round to nearest even at each step) -> fp64:
    the kernels hold the values in fp32 and convert them with cvt.rn."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.float32)
    t = t.to(torch.bfloat16 if kind == "bf16" else torch.float16)
    return t.to(torch.float64).numpy()


def model_bwd(Q, K, V, dO, scale, causal=False, key_len=None, kind="bf16", rounded=True,
              round_ds=None, d_fn=None):
    """(dQ, dK, dV) in fp64 for [B,H,N,d] fp64 arrays holding the exact
    16-bit inputs.  rounded=False gives the exact gradients, rounded=True
    the model of the kernels' roundings described above.  round_ds replaces
    the rounding of dS and d_fn maps each block's D before use (the tests
    plant kernel mistakes through them)."""
    B, H, Nq, d = Q.shape
    Nkv = K.shape[2]
    dQ = np.zeros((B, H, Nq, d))
    dK = np.zeros((B, H, Nkv, d))
    dV = np.zeros((B, H, Nkv, d))
    keys = np.arange(Nkv)
    for b in range(B):
        nvis = Nkv if key_len is None else min(max(int(key_len[b]), 0), Nkv)
        for h in range(H):
            q, k, v, g = Q[b, h], K[b, h], V[b, h], dO[b, h]
            for r0 in range(0, Nq, _ROWS):
                r1 = min(Nq, r0 + _ROWS)
                kend = min(nvis, r1) if causal else nvis  # keys any row of the block sees
                if kend <= 0:
                    continue
                rows = np.arange(r0, r1)
                vis = np.broadcast_to(keys[None, :kend] < nvis, (r1 - r0, kend))
                if causal:
                    vis = vis & (keys[None, :kend] <= rows[:, None])
                s = np.where(vis, scale * (q[r0:r1] @ k[:kend].T), -np.inf)
                has = vis.any(axis=1)
                m = np.where(has, s.max(axis=1), 0.0)
                e = np.where(vis, np.exp(s - m[:, None]), 0.0)
                den = e.sum(axis=1)
                lse = np.where(has, m + np.log(np.where(has, den, 1.0)), 0.0)
                p = np.where(vis, np.exp(s - lse[:, None]), 0.0)
                dp = g[r0:r1] @ v[:kend].T
                if rounded:
                    # forward: P against the running max of the tiles so far
                    nt = (kend + _KEY_TILE - 1) // _KEY_TILE
                    tmax = np.full((r1 - r0, nt), -np.inf)
                    for t in range(nt):
                        blk = s[:, t * _KEY_TILE:(t + 1) * _KEY_TILE]
                        tmax[:, t] = blk.max(axis=1)
                    run = np.maximum.accumulate(tmax, axis=1)
                    run = np.where(np.isfinite(run), run, 0.0)
                    mrun = np.repeat(run, _KEY_TILE, axis=1)[:, :kend]
                    pf = np.where(vis, round16(np.where(vis, np.exp(s - mrun), 0.0), kind), 0.0)
                    w = pf * np.exp(mrun - m[:, None])  # the alpha rescales of O
                    inv = np.where(has, 1.0 / np.where(has, den, 1.0), 0.0)
                    o16 = round16((w @ v[:kend]) * inv[:, None], kind)
                    D = (g[r0:r1] * o16).sum(axis=1)
                    if d_fn is not None:
                        D = d_fn(D)
                    ds = p * (dp - D[:, None])
                    pm = round16(p, kind)
                    dsm = round16(ds, kind) if round_ds is None else round_ds(ds)
                else:
                    D = (p * dp).sum(axis=1)
                    ds = p * (dp - D[:, None])
                    pm, dsm = p, ds
                dV[b, h, :kend] += pm.T @ g[r0:r1]
                dK[b, h, :kend] += scale * (dsm.T @ q[r0:r1])
                dQ[b, h, r0:r1] = scale * (dsm @ k[:kend])
    if rounded:
        dQ, dK, dV = (round16(t, kind) for t in (dQ, dK, dV))
    return dQ, dK, dV


def half_ulp(x, kind: str):
    return half_ulp_bf16(x) if kind == "bf16" else half_ulp_fp16(x)


def error_stats(g, ref, kind: str):
    """(max (|g - ref| - hu(ref)) / rms(ref), rms(g - ref) / rms(ref))."""
    g = np.asarray(g, dtype=np.float64)
    rms = math.sqrt(float((ref ** 2).mean())) if ref.size else 0.0
    err = g - ref
    if rms == 0.0:
        return 0.0, 0.0
    over = np.maximum(np.abs(err) - half_ulp(ref, kind), 0.0)
    return float(over.max()) / rms, math.sqrt(float((err ** 2).mean())) / rms


# Cases of the GPU backward tests (shapes, key_len and seeds): the small
# parity cases (tests/test_gpu_bwd.py: CASES, the strided cases and the
# determinism case) and the two full-size workloads, whose whole last two
# heads are compared.
SMALL_CASES = [
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
STRIDED_CASES = [(2, 3, 300, 333, 64, False, [333, 100]), (1, 2, 257, 257, 128, True, None)]
DETERMINISM_CASE = (1, 4, 512, 512, 128, True, None)
FULL_SIZE = ("bwd_bf16_b8_h40_n2048_d128", "bwd_bf16_causal_b1_h32_n16384_d128_qstd3")
FULL_SIZE_HEADS = 2


def small_case_seed(case) -> int:
    _, _, Nq, Nkv, d, _, _ = case
    return 4000 + Nq + Nkv + d


def small_case_inputs(case, dtype, seed=None):
    """(q, k, v, dO) of a small GPU test case on the CPU: Q ~ N(0, 1.5^2),
    dO ~ N(0, 1) from seed + 1."""
    from attention_forward_online_gb300.inputs import make_qkv

    B, H, Nq, Nkv, d, _, _ = case
    seed = small_case_seed(case) if seed is None else seed
    q, k, v = make_qkv(B, H, Nq, Nkv, d, dtype, seed=seed, q_std=1.5)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(B, H, Nq, d, generator=g).to(dtype)
    return q, k, v, do


# (t_max, t_rms) per gradient tensor: 1.5 x the model's figures over the
# cases each entry gates (tests/test_bwd_rounding_model.py recomputes the
# model and checks these values against it).
GATES = {
    "small": {
        "bf16": {"dQ": (0.0798, 0.00404), "dK": (0.0647, 0.00394), "dV": (0.066, 0.00357)},
        "fp16": {"dQ": (0.0062, 0.00051), "dK": (0.00668, 0.0005), "dV": (0.00804, 0.000456)},
    },
    "bwd_bf16_b8_h40_n2048_d128": {
        "bf16": {"dQ": (0.0189, 0.00355), "dK": (0.0145, 0.00352), "dV": (0.0177, 0.00351)},
    },
    "bwd_bf16_causal_b1_h32_n16384_d128_qstd3": {
        "bf16": {"dQ": (0.0958, 0.00416), "dK": (0.0979, 0.00396), "dV": (0.0732, 0.00349)},
    },
}

FLOOR = 1e-5


def check_grad_gate(g, ref, gate, kind, name):
    """Applies one (t_max, t_rms) gate; returns (max err / rms, rms err / rms)."""
    g = np.asarray(g, dtype=np.float64)
    assert not np.isnan(g).any(), f"NaN in {name}"
    t_max, t_rms = gate
    rms = math.sqrt(float((ref ** 2).mean())) if ref.size else 0.0
    err = np.abs(g - ref)
    bad = err > t_max * rms + half_ulp(ref, kind) + FLOOR
    assert not bad.any(), (f"{name}: error {err.max():.3e} over {t_max} x rms {rms:.3e} at "
                           f"{np.argwhere(bad)[:4].tolist()} (ref {ref[bad][:4]}, got {g[bad][:4]})")
    rerr = math.sqrt(float((err ** 2).mean())) if err.size else 0.0
    assert rerr <= t_rms * rms + FLOOR, f"{name}: rms error {rerr:.3e} over {t_rms} x rms {rms:.3e}"
    return (float(err.max()) / rms, rerr / rms) if rms > 0 else (0.0, 0.0)
