"""The rounding model behind the backward gates (tests/_bwd_model.py), on
the CPU: its exact path is the oracle's gradient, its rounded path sets
every gate at 1.5 times what it predicts, and the gates reject plausible
kernel mistakes that a looser tolerance would let through.
"""
import math

import numpy as np
import pytest
import torch

import _bwd_model as M
import oracle

KINDS = {"bf16": torch.bfloat16, "fp16": torch.float16}
NAMES = ("dQ", "dK", "dV")


def _np(*ts):
    return [t.double().numpy() for t in ts]


@pytest.mark.parametrize("kind", list(KINDS))
@pytest.mark.parametrize("case", M.SMALL_CASES[:5], ids=lambda c: "x".join(map(str, c[:5])))
def test_exact_path_is_the_oracle_gradient(case, kind):
    B, H, Nq, Nkv, d, causal, kl = case
    q, k, v, do = M.small_case_inputs(case, KINDS[kind])
    scale = 1 / math.sqrt(d)
    ex = M.model_bwd(*_np(q, k, v, do), scale, causal, kl, kind, rounded=False)
    ref = oracle.attention_bwd(q, k, v, do, scale, causal, kl)
    for a, b in zip(ex, ref):
        assert np.abs(a - b).max() <= 1e-10 * max(1.0, np.abs(b).max())


def _small_family_stats(kind):
    worst = {n: [0.0, 0.0] for n in NAMES}
    cases = [(c, None) for c in M.SMALL_CASES + M.STRIDED_CASES] + [(M.DETERMINISM_CASE, 91)]
    for case, seed in cases:
        B, H, Nq, Nkv, d, causal, kl = case
        arrs = _np(*M.small_case_inputs(case, KINDS[kind], seed))
        scale = 1 / math.sqrt(d)
        ex = M.model_bwd(*arrs, scale, causal, kl, kind, rounded=False)
        md = M.model_bwd(*arrs, scale, causal, kl, kind, rounded=True)
        for n, a, b in zip(NAMES, md, ex):
            st = M.error_stats(a, b, kind)
            worst[n] = [max(worst[n][0], st[0]), max(worst[n][1], st[1])]
    return worst


def _full_size_stats(name):
    from attention_forward_online_gb300.inputs import BWD_WORKLOADS, make_grad_out, make_inputs

    w = BWD_WORKLOADS[name]
    q, k, v, _ = make_inputs(w)
    do = make_grad_out(w)
    sl = (slice(w.B - 1, w.B), slice(w.H - M.FULL_SIZE_HEADS, w.H))
    arrs = _np(q[sl], k[sl], v[sl], do[sl])
    ex = M.model_bwd(*arrs, w.scale, w.causal, None, "bf16", rounded=False)
    md = M.model_bwd(*arrs, w.scale, w.causal, None, "bf16", rounded=True)
    return {n: M.error_stats(a, b, "bf16") for n, a, b in zip(NAMES, md, ex)}


def _assert_margin(gates, stats):
    for n in NAMES:
        for t, s, what in zip(gates[n], stats[n], ("t_max", "t_rms")):
            assert s > 0
            assert 1.5 <= t / s <= 1.52, f"{n} {what}: gate {t} vs model {s:.4g} (ratio {t / s:.3f})"


@pytest.mark.parametrize("kind", list(KINDS))
def test_small_case_gates_are_one_and_a_half_times_the_model(kind):
    _assert_margin(M.GATES["small"][kind], _small_family_stats(kind))


@pytest.mark.parametrize("name", M.FULL_SIZE)
def test_full_size_gates_are_one_and_a_half_times_the_model(name):
    # the whole last two heads of the workload, as the GPU test compares them
    _assert_margin(M.GATES[name]["bf16"], _full_size_stats(name))


def _round_bits5(x):
    """Round to nearest on a grid of 5 significant bits."""
    a = np.abs(x)
    step = 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-300))) - 4)
    return np.round(x / step) * step


def _planted(mistake):
    """Model gradients of one small bf16 case with one plausible kernel
    mistake, and the exact gradients."""
    case = (1, 2, 256, 256, 128, False, None)
    q, k, v, g = _np(*M.small_case_inputs(case, torch.bfloat16))
    scale = 1 / math.sqrt(128)
    ex = M.model_bwd(q, k, v, g, scale, kind="bf16", rounded=False)
    got = list(M.model_bwd(q, k, v, g, scale, kind="bf16", rounded=True))
    if mistake == "p_one_percent_high":
        # P = exp(s - LSE) against an LSE 0.01 too low: every P 1 % large
        got[2] = M.round16(ex[2] * math.exp(0.01), "bf16")
    elif mistake == "one_key_block_of_dk_missing":
        got[1][:, :, 16:32] = 0.0
    elif mistake == "dq_key_loop_one_short":
        got[0] = M.model_bwd(q, k[:, :, :-1], v[:, :, :-1], g, scale, kind="bf16")[0]
    elif mistake == "d_of_the_next_row":
        # D staged one row off: row i uses D of row i + 1
        got = list(M.model_bwd(q, k, v, g, scale, kind="bf16", d_fn=lambda D: np.roll(D, -1)))
    elif mistake == "ds_with_five_bits":
        # dS packed keeping 5 significant bits instead of bf16's 8
        got = list(M.model_bwd(q, k, v, g, scale, kind="bf16", round_ds=_round_bits5))
    return got, ex


@pytest.mark.parametrize("mistake", ["p_one_percent_high", "one_key_block_of_dk_missing",
                                     "dq_key_loop_one_short", "d_of_the_next_row", "ds_with_five_bits"])
def test_gates_reject_planted_kernel_mistakes(mistake):
    got, ex = _planted(mistake)
    gates = M.GATES["small"]["bf16"]
    failed = []
    for n, a, b in zip(NAMES, got, ex):
        try:
            M.check_grad_gate(a, b, gates[n], "bf16", n)
        except AssertionError:
            failed.append(n)
    assert failed, f"{mistake} passed every gate"


def test_unplanted_model_passes_its_gates():
    case = (1, 2, 256, 256, 128, False, None)
    arrs = _np(*M.small_case_inputs(case, torch.bfloat16))
    ex = M.model_bwd(*arrs, 1 / math.sqrt(128), False, None, "bf16", rounded=False)
    md = M.model_bwd(*arrs, 1 / math.sqrt(128), False, None, "bf16", rounded=True)
    for n, a, b in zip(NAMES, md, ex):
        M.check_grad_gate(a, b, M.GATES["small"]["bf16"][n], "bf16", n)
