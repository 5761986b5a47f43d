"""Pins for the fp64 oracle, against things other than the oracle itself.

Every check here is fixed by the pages or by mathematics: the worked example
x = (1, 5, 3) of chapter 6 §6.3.2 (values as printed), closed forms, library
routines (scipy), invariants (rows sum to one, combine symmetry and
associativity, the (-inf, 0) identity), and the claim of §6.6 that the
blocked loop reproduces softmax(qK^T)V to ~1e-15.  CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_x153.json")


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------- worked example
def test_worked_example_online_trace(ref, golden):
    m, l, trace = ref.online_stats(golden["x"])
    assert m == golden["m"]
    np.testing.assert_allclose(trace, golden["l_trace"], atol=golden["tol"], rtol=0)


def test_worked_example_safe_softmax(ref, golden):
    y, m, l = ref.softmax_safe(golden["x"])
    assert m == golden["m"]
    assert abs(l - golden["l_trace"][-1]) <= golden["tol"]
    np.testing.assert_allclose(y, golden["y"], atol=golden["tol"], rtol=0)
    x = np.array(golden["x"])
    np.testing.assert_allclose(np.exp(x - m), golden["exp_terms"], atol=golden["tol"])


@pytest.mark.parametrize("dtype", [torch.float64, torch.float32, torch.bfloat16])
def test_worked_example_as_attention(ref, golden, dtype):
    # One query, three keys with logits (1, 5, 3) at scale 1; V = identity, so
    # the output row is the probability vector y itself.
    Q = torch.tensor([[[[1.0, 0.0, 0.0]]]], dtype=dtype)
    K = torch.tensor([[[[1.0, 0, 0], [5.0, 0, 0], [3.0, 0, 0]]]], dtype=dtype)
    V = torch.eye(3, dtype=dtype).reshape(1, 1, 3, 3)
    O, L = ref.attention_fwd(Q, K, V, scale=1.0)
    np.testing.assert_allclose(O[0, 0, 0], golden["y"], atol=golden["tol"], rtol=0)
    assert abs(L[0, 0, 0] - (golden["m"] + math.log(golden["l_trace"][-1]))) < 1e-4


# ---------------------------------------------------------------- scalar softmax
def _rows(rng, n_rows=50, max_len=40, lo=-20, hi=20):
    for _ in range(n_rows):
        n = int(rng.integers(1, max_len))
        yield rng.uniform(lo, hi, size=n)


def test_naive_matches_safe_on_tiny_rows(ref):
    rng = np.random.default_rng(0)
    for x in _rows(rng):
        np.testing.assert_allclose(ref.softmax_naive(x), ref.softmax_safe(x)[0],
                                   rtol=1e-13, atol=1e-300)


def test_safe_softmax_rows_sum_to_one(ref):
    rng = np.random.default_rng(1)
    for x in _rows(rng, lo=-800, hi=800):
        y = ref.softmax_safe(x)[0]
        assert np.all(np.isfinite(y)) and np.all(y >= 0)
        assert abs(y.sum() - 1.0) < 1e-12


def test_safe_softmax_matches_scipy(ref):
    rng = np.random.default_rng(2)
    for x in _rows(rng, lo=-1000, hi=1000):
        y, m, l = ref.softmax_safe(x)
        np.testing.assert_allclose(y, scipy.special.softmax(x), rtol=1e-12, atol=1e-300)
        assert abs(ref.lse(m, l) - scipy.special.logsumexp(x)) < 1e-12 * max(1, abs(m))


def test_naive_overflows_where_safe_does_not(ref):
    # Chapter 6 §6.2: e^1000 overflows double too; the naive form gives NaN.
    x = np.array([1000.0, 1000.0, 999.0])
    with np.errstate(all="ignore"):
        assert np.isnan(ref.softmax_naive(x)).all()
    y = ref.softmax_safe(x)[0]
    assert np.all(np.isfinite(y))
    np.testing.assert_allclose(y, scipy.special.softmax(x), rtol=1e-14)


# ---------------------------------------------------------------- online recurrence
def test_online_matches_safe_random(ref):
    rng = np.random.default_rng(3)
    for x in _rows(rng, n_rows=100, max_len=300, lo=-50, hi=50):
        m, l, _ = ref.online_stats(x)
        _, m3, l3 = ref.softmax_safe(x)
        assert m == m3
        assert abs(l - l3) <= 1e-12 * l3


def test_online_with_leading_neg_inf_run(ref):
    # Chapter 6 §6.4: rows whose first elements are -inf (masked) must not
    # produce NaN; the guarded update skips them.
    x = np.concatenate([np.full(300, -np.inf), np.random.default_rng(4).normal(size=100)])
    m, l, trace = ref.online_stats(x)
    assert np.all(trace[:300] == 0.0)
    assert np.all(np.isfinite(trace))
    assert abs(ref.lse(m, l) - scipy.special.logsumexp(x)) < 1e-12


def test_online_all_masked_is_identity(ref):
    m, l, trace = ref.online_stats(np.full(17, -np.inf))
    assert m == -np.inf and l == 0.0 and not np.isnan(trace).any()
    assert ref.lse(m, l) == -np.inf


# ---------------------------------------------------------------- combine monoid
def _chunk_states(ref, x, rng):
    cuts = np.sort(rng.choice(np.arange(1, len(x)), size=min(len(x) - 1, int(rng.integers(1, 8))),
                              replace=False)) if len(x) > 1 else np.array([], dtype=int)
    states = []
    for part in np.split(x, cuts):
        m, l, _ = ref.online_stats(part)
        states.append((m, l))
    return states


def test_combine_symmetric(ref):
    rng = np.random.default_rng(5)
    for _ in range(200):
        a = (rng.normal() * 10, rng.uniform(0.5, 100))
        b = (rng.normal() * 10, rng.uniform(0.5, 100))
        assert ref.combine(a, b)[0] == ref.combine(b, a)[0]
        assert abs(ref.combine(a, b)[1] - ref.combine(b, a)[1]) <= 1e-14 * ref.combine(a, b)[1]


def test_combine_associative_under_random_splits(ref):
    rng = np.random.default_rng(6)
    for x in _rows(rng, n_rows=60, max_len=200, lo=-30, hi=30):
        whole_m, whole_l, _ = ref.online_stats(x)
        states = _chunk_states(ref, x, rng)
        # left fold
        acc = (-np.inf, 0.0)
        for s in states:
            acc = ref.combine(acc, s)
        # random merge order (random tree)
        pool = list(states)
        while len(pool) > 1:
            i, j = sorted(rng.choice(len(pool), size=2, replace=False))
            merged = ref.combine(pool[j], pool[i])
            pool = [p for k, p in enumerate(pool) if k not in (i, j)] + [merged]
        for m, l in (acc, pool[0]):
            assert m == whole_m
            assert abs(l - whole_l) <= 1e-12 * whole_l


def test_combine_identity_and_empty(ref):
    a = (2.5, 3.75)
    assert ref.combine((-np.inf, 0.0), a) == a
    assert ref.combine(a, (-np.inf, 0.0)) == a
    e = ref.combine((-np.inf, 0.0), (-np.inf, 0.0))
    assert e[0] == -np.inf and e[1] == 0.0


def test_combine_equals_quantity_sum(ref):
    # Chapter 6 §6.4.1: a state (m, l) stands for l*e^m; combine adds them.
    rng = np.random.default_rng(7)
    for _ in range(100):
        a = (rng.uniform(-5, 5), rng.uniform(0.1, 10))
        b = (rng.uniform(-5, 5), rng.uniform(0.1, 10))
        m, l = ref.combine(a, b)
        assert abs(l * math.exp(m) - (a[1] * math.exp(a[0]) + b[1] * math.exp(b[0]))) < 1e-12 * l * math.exp(m)


# ---------------------------------------------------------------- attention
def _np_attention(q, k, v, scale, causal=False, key_len=None):
    """softmax(scale*QK^T + mask) V through numpy matmul and scipy's softmax /
    logsumexp (library routines), per (b, h)."""
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    O = np.zeros((B, H, Nq, d))
    L = np.full((B, H, Nq), -np.inf)
    for b in range(B):
        kl = Nkv if key_len is None else min(max(key_len[b], 0), Nkv)
        for h in range(H):
            s = scale * (q[b, h] @ k[b, h].T)
            mask = np.zeros_like(s, dtype=bool)
            mask[:, kl:] = True
            if causal:
                mask |= np.arange(Nkv)[None, :] > np.arange(Nq)[:, None]
            s = np.where(mask, -np.inf, s)
            live = ~mask.all(axis=1)
            if live.any():
                O[b, h, live] = scipy.special.softmax(s[live], axis=1) @ v[b, h]
                L[b, h, live] = scipy.special.logsumexp(s[live], axis=1)
    return O, L


CASES = [
    # B, H, Nq, Nkv, d, causal, key_len
    (1, 1, 5, 7, 4, False, None),
    (2, 3, 33, 47, 16, False, [47, 20]),
    (2, 2, 40, 40, 8, True, None),
    (3, 1, 29, 29, 8, True, [29, 0, 11]),
    (1, 2, 17, 64, 32, False, [70]),
    (2, 1, 20, 9, 8, True, [-3, 9]),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dtype", [torch.float64, torch.float32, torch.bfloat16, torch.float16])
def test_attention_matches_library_route(ref, case, dtype):
    B, H, Nq, Nkv, d, causal, kl = case
    g = torch.Generator().manual_seed(11)
    q = (torch.randn(B, H, Nq, d, generator=g) * 2).to(dtype)
    k = torch.randn(B, H, Nkv, d, generator=g).to(dtype)
    v = torch.randn(B, H, Nkv, d, generator=g).to(dtype)
    scale = 1 / math.sqrt(d)
    O, L = ref.attention_fwd(q, k, v, scale, causal, kl)
    O2, L2 = _np_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                           scale, causal, kl)
    assert not np.isnan(O).any() and not np.isnan(L).any()
    np.testing.assert_allclose(O, O2, atol=1e-12, rtol=0)
    fin = np.isfinite(L2)
    assert np.array_equal(np.isfinite(L), fin)
    np.testing.assert_allclose(L[fin], L2[fin], atol=1e-12, rtol=0)
    assert np.all(L[~fin] == -np.inf) and np.all(O[~np.isfinite(L)] == 0.0)


def test_attention_single_key_is_that_value(ref):
    rng = np.random.default_rng(8)
    q, k, v = rng.normal(size=(2, 2, 6, 8)), rng.normal(size=(2, 2, 1, 8)), rng.normal(size=(2, 2, 1, 8))
    O, L = ref.attention_fwd(q, k, v, scale=0.3)
    np.testing.assert_allclose(O, np.broadcast_to(v, O.shape), atol=1e-15)
    np.testing.assert_allclose(L, 0.3 * np.einsum("bhid,bhd->bhi", q, k[:, :, 0]), atol=1e-14)


def test_fp16_decoding_every_finite_bit_pattern(ref):
    # With one key the softmax weight is exactly 1, so O = V: the oracle's
    # IEEE binary16 decoder must agree with numpy's on all 63488 finite
    # patterns (zeros, subnormals, normals, both signs).
    bits = np.arange(1 << 16, dtype=np.uint16)
    h = bits.view(np.float16)
    h = h[np.isfinite(h)]
    assert h.size == 63488
    v = torch.from_numpy(h.copy()).reshape(1, h.size // 64, 1, 64)
    q = torch.zeros_like(v)
    O, L = ref.attention_fwd(q, q, v, scale=1.0)
    assert np.array_equal(O.reshape(-1), h.astype(np.float64))
    assert np.all(L == 0.0)


def test_attention_zero_query_averages_visible_values(ref):
    # All logits equal -> uniform weights over J; LSE = log|J|.
    rng = np.random.default_rng(9)
    B, H, N, d = 2, 2, 12, 4
    q = np.zeros((B, H, N, d))
    k, v = rng.normal(size=(B, H, N, d)), rng.normal(size=(B, H, N, d))
    kl = [12, 5]
    O, L = ref.attention_fwd(q, k, v, scale=1.0, causal=True, key_len=kl)
    for b in range(B):
        for i in range(N):
            n = min(kl[b], i + 1)
            np.testing.assert_allclose(O[b, :, i], v[b, :, :n].mean(axis=1), atol=1e-14)
            np.testing.assert_allclose(L[b, :, i], math.log(n), atol=1e-14)


def test_attention_one_hot_keys_closed_form(ref):
    # K = identity rows, Q[i] = a * e_{sigma(i)} with a non-symmetric sigma:
    # logit a*scale at key sigma(i), 0 elsewhere, so
    #   O[i] = (e^{a s} V[sigma(i)] + sum_{j != sigma(i)} V[j]) / (e^{a s} + n - 1).
    n, a, scale = 6, 4.0, 0.5
    sigma = [3, 0, 5, 1, 1, 2, 4]
    q = np.zeros((1, 1, len(sigma), n))
    for i, s in enumerate(sigma):
        q[0, 0, i, s] = a
    k = np.eye(n).reshape(1, 1, n, n)
    v = np.random.default_rng(10).normal(size=(1, 1, n, n))
    O, L = ref.attention_fwd(q, k, v, scale)
    w = math.exp(a * scale)
    for i, s in enumerate(sigma):
        expect = (w * v[0, 0, s] + v[0, 0].sum(axis=0) - v[0, 0, s]) / (w + n - 1)
        np.testing.assert_allclose(O[0, 0, i], expect, atol=1e-14)
        assert abs(L[0, 0, i] - math.log(w + n - 1)) < 1e-14


def test_attention_causal_first_row_is_first_value(ref):
    rng = np.random.default_rng(12)
    q, k, v = (rng.normal(size=(1, 3, 9, 8)) for _ in range(3))
    O, L = ref.attention_fwd(q, k, v, scale=0.25, causal=True)
    np.testing.assert_allclose(O[:, :, 0], v[:, :, 0], atol=1e-15)
    np.testing.assert_allclose(L[:, :, 0], 0.25 * (q[:, :, 0] * k[:, :, 0]).sum(-1), atol=1e-14)


def test_attention_fully_masked_rows_are_zero_not_nan(ref):
    rng = np.random.default_rng(13)
    q, k, v = (rng.normal(size=(3, 2, 5, 4)) for _ in range(3))
    O, L = ref.attention_fwd(q, k, v, scale=1.0, key_len=[5, 0, -7])
    assert not np.isnan(O).any() and not np.isnan(L).any()
    assert np.all(O[1:] == 0.0) and np.all(L[1:] == -np.inf)
    assert np.all(np.isfinite(L[0]))


def test_attention_key_len_full_equals_no_mask_and_clamps(ref):
    rng = np.random.default_rng(14)
    q, k, v = (rng.normal(size=(2, 2, 7, 4)) for _ in range(3))
    base = ref.attention_fwd(q, k, v, 0.5)
    for kl in ([7, 7], [100, 8]):
        got = ref.attention_fwd(q, k, v, 0.5, key_len=kl)
        np.testing.assert_array_equal(got[0], base[0])
        np.testing.assert_array_equal(got[1], base[1])
    one = ref.attention_fwd(q, k, v, 0.5, key_len=[1, 1])
    np.testing.assert_allclose(one[0], np.broadcast_to(v[:, :, :1], one[0].shape), atol=1e-15)


def test_attention_key_permutation_invariance(ref):
    rng = np.random.default_rng(15)
    q, k, v = (rng.normal(size=(1, 2, 6, 8)) for _ in range(3))
    perm = rng.permutation(6)
    O1, L1 = ref.attention_fwd(q, k, v, 0.7)
    O2, L2 = ref.attention_fwd(q, k[:, :, perm], v[:, :, perm], 0.7)
    np.testing.assert_allclose(O1, O2, atol=1e-14)
    np.testing.assert_allclose(L1, L2, atol=1e-14)


def test_attention_rows_subset_matches_full(ref):
    rng = np.random.default_rng(16)
    q, k, v = (rng.normal(size=(2, 3, 10, 8)) for _ in range(3))
    O, L = ref.attention_fwd(q, k, v, 0.4, causal=True, key_len=[10, 6])
    rows = [0, 7, 29, 30, 59]
    Os, Ls = ref.attention_fwd(q, k, v, 0.4, causal=True, key_len=[10, 6], rows=rows)
    np.testing.assert_array_equal(Os, O.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(Ls, L.reshape(-1)[rows])


@pytest.mark.parametrize("form", [0, 1])
@pytest.mark.parametrize("block", [1, 3, 16, 64])
def test_blocked_loop_matches_definition(ref, form, block):
    # Chapter 6 §6.6 reports the blocked loop equal to softmax(qK^T)V to
    # ~1e-15 in numpy; both forms of the loop, any block size, with masks
    # and large logits.
    g = torch.Generator().manual_seed(17)
    B, H, N, d = 2, 2, 70, 16
    q = torch.randn(B, H, N, d, generator=g, dtype=torch.float64) * 6
    k = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    for causal, kl in ((False, None), (True, [70, 31]), (False, [0, 5])):
        O, L = ref.attention_fwd(q, k, v, 0.25, causal, kl)
        Ob, Lb = ref.attention_blocked(q, k, v, 0.25, causal, kl, block=block, form=form)
        np.testing.assert_allclose(Ob, O, atol=1e-12, rtol=0)
        fin = np.isfinite(L)
        assert np.array_equal(fin, np.isfinite(Lb))
        np.testing.assert_allclose(Lb[fin], L[fin], atol=1e-12, rtol=0)


def test_oracle_rejects_bad_arguments(ref):
    q = np.zeros((1, 1, 2, 4))
    with pytest.raises(ValueError):
        ref.attention_fwd(q, q, q, 1.0, rows=[5])
    with pytest.raises(ValueError):
        ref.attention_fwd(q, np.zeros((1, 1, 2, 3)), q, 1.0)


# ---------------------------------------------------------------- batched row softmax
@pytest.mark.parametrize("dtype", [torch.float64, torch.float32, torch.bfloat16, torch.float16])
def test_softmax_rows_matches_scipy_and_worked_example(ref, golden, dtype):
    g = torch.Generator().manual_seed(21)
    X = (torch.randn(37, 301, generator=g, dtype=torch.float64) * 5).to(dtype)
    X[3, :50] = -float("inf")           # leading masked run
    X[7, :] = -float("inf")             # fully masked row
    X[9, 0] = golden["x"][0]
    Y, L = ref.softmax_rows(X)
    x = X.double().numpy()
    live = np.isfinite(x).any(axis=1)
    np.testing.assert_allclose(Y[live], scipy.special.softmax(x[live], axis=1), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(L[live], scipy.special.logsumexp(x[live], axis=1), atol=1e-12)
    assert np.all(Y[~live] == 0.0) and np.all(L[~live] == -np.inf)
    assert np.allclose(Y[live].sum(axis=1), 1.0, atol=1e-12)
    Yw, Lw = ref.softmax_rows(np.array([golden["x"]]))
    np.testing.assert_allclose(Yw[0], golden["y"], atol=golden["tol"])
