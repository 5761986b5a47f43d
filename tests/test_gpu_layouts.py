"""GPU parity of the fp16 element type and of strided (non-contiguous)
Q, K, V and O, through osattn_fwd_strided, against the fp64 oracle.

The oracle reads the logical [B, H, N, d] values whatever the storage, so a
strided call must match it within the same gates as a contiguous one; and
since the kernels visit the same tiles in the same order, a strided call must
also reproduce the contiguous call bit for bit.  Tolerances: tests/_compare.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_online_gb300 import osattn
from attention_forward_online_gb300.inputs import WORKLOADS, make_qkv, sample_rows

from _compare import check

pytestmark = pytest.mark.gpu
DEV = "cuda"
KIND = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}


def bnhd(t):
    """The same values stored as [B, N, H, d], returned as a [B, H, N, d] view."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def nan_out_bnhd(B, H, N, d, dtype):
    return torch.full((B, N, H, d), float("nan"), dtype=dtype, device=DEV).transpose(1, 2)


def contiguous_call(q, k, v, scale, causal, kl):
    O, L = osattn.fwd(q.contiguous(), k.contiguous(), v.contiguous(), scale=scale,
                      causal=causal, key_len=kl)
    return O, L


CASES = [
    # B, H, Nq, Nkv, d, causal, key_len
    (2, 3, 300, 333, 64, False, [333, 100]),
    (1, 2, 257, 257, 128, True, None),
    (2, 2, 130, 700, 128, False, [700, 0]),
    (1, 4, 512, 512, 64, True, [400]),
]


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[5] else ""))
def test_bnhd_layout_matches_oracle_and_contiguous(case, dtype):
    B, H, Nq, Nkv, d, causal, kl = case
    q, k, v = make_qkv(B, H, Nq, Nkv, d, dtype, seed=3000 + Nq + d, q_std=2.0)
    scale = 1 / math.sqrt(d)
    qd, kd, vd = bnhd(q.to(DEV)), bnhd(k.to(DEV)), bnhd(v.to(DEV))
    assert not qd.is_contiguous()
    kld = None if kl is None else torch.tensor(kl, dtype=torch.int32, device=DEV)
    O = nan_out_bnhd(B, H, Nq, d, dtype)
    L = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=DEV)
    osattn.fwd(qd, kd, vd, scale=scale, causal=causal, key_len=kld, out=O, lse=L)
    assert osattn.get_device_status() == osattn.OK
    Oref, Lref = oracle.attention_fwd(q, k, v, scale, causal, kl)
    check(O.double().cpu().numpy(), L.double().cpu().numpy(), Oref, Lref, KIND[dtype])
    Oc, Lc = contiguous_call(qd, kd, vd, scale, causal, kld)
    torch.cuda.synchronize()
    assert torch.equal(O.contiguous().view(torch.int16 if dtype != torch.float32 else torch.int32),
                       Oc.view(torch.int16 if dtype != torch.float32 else torch.int32))
    assert torch.equal(L, Lc)


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
def test_packed_qkv_views_and_interleaved_output(dtype):
    # One [B, N, 3, H, d] tensor (a fused QKV projection's output); the
    # result goes into a [B, N, H, d] buffer, i.e. [B, N, H*d] for the next
    # projection.
    B, H, N, d = 2, 3, 400, 128
    q, k, v = make_qkv(B, H, N, N, d, dtype, seed=41)
    qkv = torch.stack([t.transpose(1, 2) for t in (q, k, v)], dim=2).to(DEV)  # [B,N,3,H,d]
    qv, kv, vv = (qkv[:, :, i].transpose(1, 2) for i in range(3))
    O = nan_out_bnhd(B, H, N, d, dtype)
    Ob, Lb = osattn.fwd(qv, kv, vv, causal=True, out=O)
    assert Ob is O and osattn.get_device_status() == osattn.OK
    Oref, Lref = oracle.attention_fwd(q, k, v, 1 / math.sqrt(d), True)
    check(O.double().cpu().numpy(), Lb.double().cpu().numpy(), Oref, Lref, KIND[dtype])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32],
                         ids=["bf16", "fp16", "fp32"])
def test_padded_rows_batch_gaps_and_guard_columns(dtype):
    # Row stride d + pad, a batch stride of two batches (every other batch of
    # a larger tensor), and O inside a padded buffer whose pad columns must
    # stay untouched.
    B, H, Nq, Nkv, d = 2, 2, 200, 333, 64
    pad = 8 if dtype != torch.float32 else 4
    q, k, v = make_qkv(B, H, Nq, Nkv, d, dtype, seed=43)
    big_q = torch.zeros(2 * B, H, Nq, d + pad, dtype=dtype, device=DEV)
    big_q[::2, :, :, :d] = q.to(DEV)
    qd = big_q[::2, :, :, :d]
    kbuf = torch.zeros(B, H, Nkv, d + pad, dtype=dtype, device=DEV)
    kbuf[..., :d] = k.to(DEV)
    kd = kbuf[..., :d]
    vd = bnhd(v.to(DEV))
    sentinel = 7.0
    obuf = torch.full((B, H, Nq, d + pad), sentinel, dtype=dtype, device=DEV)
    od = obuf[..., :d]
    _, L = osattn.fwd(qd, kd, vd, causal=False, out=od)
    assert osattn.get_device_status() == osattn.OK
    assert torch.all(obuf[..., d:] == sentinel).item()
    Oref, Lref = oracle.attention_fwd(q, k, v, 1 / math.sqrt(d), False)
    check(od.double().cpu().numpy(), L.double().cpu().numpy(), Oref, Lref, KIND[dtype])


@pytest.mark.parametrize("case", [
    # B, H, Nq, Nkv, d, causal, key_len, splits
    (1, 2, 256, 2000, 128, False, None, [1, 3, 16]),
    (2, 2, 257, 1100, 64, True, [1100, 300], [2, 9]),
], ids=["d128", "d64c"])
def test_splitkv_fp16_matches_oracle(case):
    B, H, Nq, Nkv, d, causal, kl, splits_list = case
    q, k, v = make_qkv(B, H, Nq, Nkv, d, torch.float16, seed=2100 + Nq, q_std=2.0)
    scale = 1 / math.sqrt(d)
    Oref, Lref = oracle.attention_fwd(q, k, v, scale, causal, kl)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    kld = None if kl is None else torch.tensor(kl, dtype=torch.int32, device=DEV)
    for splits in splits_list:
        O, L = osattn.fwd_splitkv(qd, kd, vd, splits, scale=scale, causal=causal, key_len=kld)
        assert osattn.get_device_status() == osattn.OK
        assert O.dtype == torch.float16
        check(O.double().cpu().numpy(), L.double().cpu().numpy(), Oref, Lref, "fp16")


@pytest.mark.parametrize("name,layout", [("bf16_b8_h40_n2048_d128", "bnhd"),
                                         ("bf16_causal_b1_h32_n16384_d128_qstd3", "contiguous")])
def test_fp16_full_size_sampled(name, layout):
    # The specified bf16 workload shapes, drawn in fp16 (same seeds), at full
    # size in the tensor-core kernel's launch configuration.
    w = WORKLOADS[name]
    q, k, v = make_qkv(w.B, w.H, w.Nq, w.Nkv, w.d, torch.float16, w.seed, w.q_std, w.kv_std)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    if layout == "bnhd":
        qd, kd, vd = bnhd(qd), bnhd(kd), bnhd(vd)
        O = nan_out_bnhd(w.B, w.H, w.Nq, w.d, torch.float16)
    else:
        O = torch.full_like(qd, float("nan"))
    L = torch.full((w.B, w.H, w.Nq), float("nan"), dtype=torch.float32, device=DEV)
    osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal, out=O, lse=L)
    assert osattn.get_device_status() == osattn.OK
    assert not torch.isnan(O).any().item() and torch.isfinite(L).all().item()
    rows = sample_rows(w.B, w.H, w.Nq, 200, seed=w.seed)
    Oref, Lref = oracle.attention_fwd(q, k, v, w.scale, w.causal, None, rows=rows)
    idx = torch.tensor(rows, device=DEV)
    Og = O.contiguous().reshape(-1, w.d)[idx].double().cpu().numpy()
    Lg = L.reshape(-1)[idx].double().cpu().numpy()
    print(name, layout, len(rows), "rows", check(Og, Lg, Oref, Lref, "fp16"))


def test_fp16_large_logits_do_not_overflow():
    # |s| up to a few hundred: e^s would overflow fp16 (max 65504) but the
    # kernel exponentiates s - m <= 0, so P stays in [0, 1].
    q, k, v = make_qkv(1, 2, 256, 300, 64, torch.float16, seed=47, q_std=8.0)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O, L = osattn.fwd(qd, kd, vd, scale=1.0)
    assert osattn.get_device_status() == osattn.OK
    Oref, Lref = oracle.attention_fwd(q, k, v, 1.0)
    assert np.abs(Lref).max() > 100
    check(O.double().cpu().numpy(), L.double().cpu().numpy(), Oref, Lref, "fp16")
