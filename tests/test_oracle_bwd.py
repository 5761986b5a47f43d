"""Pins for the oracle's gradients (osattn_ref_attention_bwd), against
things other than the gradient code itself: central finite differences of
the scalar loss sum(dO * O) computed with the oracle's forward pass, torch
autograd (fp64, CPU) on a plain softmax(QK^T) V composition, and closed
forms.  CPU only.
"""
import math

import numpy as np
import pytest
import torch


def _loss(ref, Q, K, V, dO, scale, causal, kl):
    O, _ = ref.attention_fwd(Q, K, V, scale, causal, kl)
    return float((O * dO).sum())


CASES = [
    # B, H, Nq, Nkv, d, causal, key_len
    (1, 2, 5, 7, 4, False, None),
    (2, 1, 6, 6, 3, True, None),
    (2, 2, 4, 9, 5, False, [9, 4]),
    (1, 1, 7, 5, 4, True, [3]),
    (3, 1, 3, 4, 2, True, [4, 0, 2]),
]


@pytest.mark.parametrize("case", CASES)
def test_gradients_match_finite_differences(ref, case):
    B, H, Nq, Nkv, d, causal, kl = case
    rng = np.random.default_rng(100 + Nq * Nkv)
    Q = rng.normal(size=(B, H, Nq, d)) * 1.5
    K = rng.normal(size=(B, H, Nkv, d))
    V = rng.normal(size=(B, H, Nkv, d))
    dO = rng.normal(size=(B, H, Nq, d))
    scale = 0.7
    dQ, dK, dV = ref.attention_bwd(Q, K, V, dO, scale, causal, kl)
    h = 1e-5
    for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        num = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            keep = X[idx]
            X[idx] = keep + h
            lp = _loss(ref, Q, K, V, dO, scale, causal, kl)
            X[idx] = keep - h
            lm = _loss(ref, Q, K, V, dO, scale, causal, kl)
            X[idx] = keep
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(G, num, atol=1e-7, rtol=0, err_msg=f"d{name}")


def _torch_grads(Q, K, V, dO, scale, causal, kl):
    q = torch.tensor(Q, dtype=torch.float64, requires_grad=True)
    k = torch.tensor(K, dtype=torch.float64, requires_grad=True)
    v = torch.tensor(V, dtype=torch.float64, requires_grad=True)
    B, H, Nq, d = Q.shape
    Nkv = K.shape[2]
    s = torch.matmul(q, k.transpose(-2, -1)) * scale
    vis = torch.ones(B, 1, Nq, Nkv, dtype=torch.bool)
    if kl is not None:
        for b in range(B):
            vis[b, :, :, max(0, min(kl[b], Nkv)):] = False
    if causal:
        vis &= torch.ones(Nq, Nkv, dtype=torch.bool).tril()
    s = s.masked_fill(~vis, float("-inf"))
    row_has = vis.any(-1, keepdim=True)
    p = torch.softmax(torch.where(row_has, s, torch.zeros_like(s)), dim=-1)
    p = torch.where(vis, p, torch.zeros_like(p))
    o = torch.matmul(p, v)
    o.backward(torch.tensor(dO, dtype=torch.float64))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("dtype", [torch.float64, torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("case", [(2, 3, 33, 47, 16, False, [47, 20]), (2, 2, 40, 40, 8, True, None),
                                  (1, 2, 17, 64, 32, True, [50])])
def test_gradients_match_torch_autograd(ref, case, dtype):
    B, H, Nq, Nkv, d, causal, kl = case
    g = torch.Generator().manual_seed(17)
    q = (torch.randn(B, H, Nq, d, generator=g) * 2).to(dtype)
    k = torch.randn(B, H, Nkv, d, generator=g).to(dtype)
    v = torch.randn(B, H, Nkv, d, generator=g).to(dtype)
    do = torch.randn(B, H, Nq, d, generator=g).to(dtype)
    scale = 1 / math.sqrt(d)
    dQ, dK, dV = ref.attention_bwd(q, k, v, do, scale, causal, kl)
    tq, tk, tv = _torch_grads(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                              do.double().numpy(), scale, causal, kl)
    np.testing.assert_allclose(dQ, tq, atol=1e-11, rtol=0)
    np.testing.assert_allclose(dK, tk, atol=1e-11, rtol=0)
    np.testing.assert_allclose(dV, tv, atol=1e-11, rtol=0)


def test_single_key_closed_form(ref):
    # One visible key: P = 1 whatever the logits, so dQ = dK = 0 and dV[0]
    # is the sum of the upstream gradients of the rows that see it.
    rng = np.random.default_rng(5)
    Q, K, V = rng.normal(size=(2, 2, 6, 4)), rng.normal(size=(2, 2, 1, 4)), rng.normal(size=(2, 2, 1, 4))
    dO = rng.normal(size=(2, 2, 6, 4))
    dQ, dK, dV = ref.attention_bwd(Q, K, V, dO, 0.5)
    assert np.abs(dQ).max() < 1e-14 and np.abs(dK).max() < 1e-14
    np.testing.assert_allclose(dV[:, :, 0], dO.sum(axis=2), atol=1e-13)


def test_masked_batch_has_zero_gradients(ref):
    rng = np.random.default_rng(6)
    Q, K, V, dO = (rng.normal(size=s) for s in [(2, 1, 5, 4), (2, 1, 6, 4), (2, 1, 6, 4), (2, 1, 5, 4)])
    dQ, dK, dV = ref.attention_bwd(Q, K, V, dO, 0.5, key_len=[6, 0])
    assert np.all(dQ[1] == 0) and np.all(dK[1] == 0) and np.all(dV[1] == 0)
    assert np.abs(dQ[0]).max() > 0 and np.abs(dK[0]).max() > 0


def test_dv_columns_sum_rule(ref):
    # sum_j dV_j = sum_i dO_i over rows that see at least one key (each row's
    # probabilities sum to one), for any mask.
    rng = np.random.default_rng(7)
    Q, K, V, dO = (rng.normal(size=s) for s in [(1, 2, 9, 4), (1, 2, 7, 4), (1, 2, 7, 4), (1, 2, 9, 4)])
    _, _, dV = ref.attention_bwd(Q, K, V, dO, 0.3, causal=True)
    np.testing.assert_allclose(dV.sum(axis=2), dO.sum(axis=2), atol=1e-12)


def test_bwd_rejects_bad_arguments(ref):
    q = np.zeros((1, 1, 2, 4))
    with pytest.raises(ValueError):
        ref.attention_bwd(q, q, q, np.zeros((1, 1, 3, 4)), 1.0)
    with pytest.raises(TypeError):
        ref.attention_bwd(q, q, q, q.astype(np.float32), 1.0)
