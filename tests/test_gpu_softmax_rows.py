"""GPU parity of the standalone online row softmax (osattn_softmax_rows)
against the fp64 oracle's three-pass row softmax.  Tolerances as for the
attention outputs (tests/_compare.py): fp32 1e-5; bf16 and fp16 1e-2 + half
an ulp of the output, LSE 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_online_gb300 import osattn

from _compare import check

pytestmark = pytest.mark.gpu
DEV = "cuda"

SHAPES = [(7, 1), (5, 3), (33, 8), (9, 100), (4, 255), (16, 256), (3, 2048), (3, 2049),
          (40, 4096), (2, 5000), (3, 16384), (2, 16385), (3, 32768),
          # rows split across a cluster: parts in registers (2 to 16 CTAs) ...
          (3, 32769), (3, 40000), (3, 65536), (3, 100003), (3, 262144), (3, 524288),
          # ... and rows streamed twice by the cluster's CTAs
          (3, 524296), (3, 1048576), (3, 1048573)]


def make_rows(rows, N, dtype, seed, scale=3.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, N, generator=g) * scale
    if rows > 2:
        x[1, : max(1, N // 3)] = -float("inf")  # leading masked run
        x[2, :] = -float("inf")                 # fully masked row
    return x.to(dtype)


KIND = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_softmax_rows_matches_oracle(shape, dtype):
    rows, N = shape
    x = make_rows(rows, N, dtype, seed=rows * 1000 + N)
    xd = x.to(DEV)
    y = torch.full_like(xd, float("nan"))
    lse = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
    osattn.softmax_rows(xd, out=y, lse=lse)
    assert osattn.get_device_status() == osattn.OK
    Yref, Lref = oracle.softmax_rows(x)
    Y = y.double().cpu().numpy()
    check(Y, lse.double().cpu().numpy(), Yref, Lref, KIND[dtype])
    live = np.isfinite(Lref)
    assert np.allclose(Y[live].sum(axis=1), 1.0, atol=1e-5 if dtype == torch.float32 else 2e-2)


def test_softmax_rows_in_place_unaligned_and_without_lse():
    x = make_rows(6, 1001, torch.float32, seed=3)
    Yref, _ = oracle.softmax_rows(x)
    buf = torch.empty(6 * 1001 + 1, dtype=torch.float32, device=DEV)
    xd = buf[1:].view(6, 1001)  # 4-byte but not 16-byte aligned: scalar path
    xd.copy_(x.to(DEV))
    y, l = osattn.softmax_rows(xd, out=xd, want_lse=False)
    assert l is None
    torch.cuda.synchronize()
    np.testing.assert_allclose(xd.double().cpu().numpy(), Yref, atol=1e-5, rtol=0)


def test_softmax_rows_worked_example():
    # Chapter 6 §6.3.2: x = (1, 5, 3) -> y ~ (0.0159, 0.8668, 0.1173)
    x = torch.tensor([[1.0, 5.0, 3.0]], device=DEV)
    y, l = osattn.softmax_rows(x)
    torch.cuda.synchronize()
    np.testing.assert_allclose(y.cpu().numpy()[0], [0.0159, 0.8668, 0.1173], atol=1e-4)
    assert abs(l.item() - (5 + np.log(1.1536))) < 1e-4


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("N", [65536, 262144, 1048576])
def test_split_row_with_a_cluster_part_fully_masked(N, dtype):
    # Whole parts of a split row masked (-inf): their CTAs hold the empty
    # state (-inf, 0), which the guarded combine across the cluster must
    # absorb without NaN; one row masked everywhere but its last element.
    g = torch.Generator().manual_seed(N)
    x = torch.randn(3, N, generator=g) * 3.0
    x[0, N // 8: N // 2] = -float("inf")
    x[1, : N - 1] = -float("inf")
    x[2, N // 2:] = -float("inf")
    x = x.to(dtype)
    xd = x.to(DEV)
    y, lse = osattn.softmax_rows(xd)
    assert osattn.get_device_status() == osattn.OK
    Yref, Lref = oracle.softmax_rows(x)
    Y = y.double().cpu().numpy()
    check(Y, lse.double().cpu().numpy(), Yref, Lref, KIND[dtype])
    assert Y[1, -1] == 1.0 and np.all(Y[1, :-1] == 0.0)
