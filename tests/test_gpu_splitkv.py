"""GPU parity of the split-KV path (key axis cut into ranges, partials merged
by the (m, l) combine) against the fp64 oracle, and against the unsplit
kernel.  Tolerances: tests/_compare.py."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_online_gb300 import osattn
from attention_forward_online_gb300.inputs import SPLITKV_WORKLOADS, make_inputs, make_qkv, sample_rows

from _compare import check

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_split(q, k, v, scale, causal, key_len, splits):
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    kl = None if key_len is None else torch.as_tensor(key_len, dtype=torch.int32).to(DEV)
    O = torch.full_like(qd, float("nan"))
    L = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=DEV)
    osattn.fwd_splitkv(qd, kd, vd, splits, scale=scale, causal=causal, key_len=kl, out=O, lse=L)
    assert osattn.get_device_status() == osattn.OK
    return O.double().cpu().numpy(), L.double().cpu().numpy()


CASES = [
    # B, H, Nq, Nkv, d, causal, key_len, splits
    (1, 2, 256, 2000, 128, False, None, [1, 2, 3, 7, 16]),
    (1, 2, 700, 700, 64, True, None, [1, 3, 5]),
    (3, 1, 300, 1000, 128, False, [1000, 129, 0], [4]),
    (1, 1, 128, 256, 64, False, None, [16]),
    (2, 2, 257, 1100, 128, True, [1100, 300], [2, 9]),
    (1, 3, 1, 5000, 128, False, None, [40]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[5] else ""))
def test_splitkv_matches_oracle(case):
    B, H, Nq, Nkv, d, causal, kl, splits_list = case
    q, k, v = make_qkv(B, H, Nq, Nkv, d, torch.bfloat16, seed=2000 + Nq, q_std=2.0)
    scale = 1 / math.sqrt(d)
    Oref, Lref = oracle.attention_fwd(q, k, v, scale, causal, kl)
    for splits in splits_list:
        O, L = run_split(q, k, v, scale, causal, kl, splits)
        check(O, L, Oref, Lref, "bf16")


def test_splitkv_agrees_with_unsplit_kernel():
    q, k, v = make_qkv(2, 4, 512, 3000, 128, torch.bfloat16, seed=31)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O1, L1 = osattn.fwd(qd, kd, vd)
    O2, L2 = osattn.fwd_splitkv(qd, kd, vd, 6)
    torch.cuda.synchronize()
    assert (O1.float() - O2.float()).abs().max().item() <= 8e-3
    assert (L1 - L2).abs().max().item() <= 1e-4


def test_splitkv_workload_full_size_sampled():
    w = SPLITKV_WORKLOADS["bf16_b1_h8_q512_kv65536_d128"]
    q, k, v, kl = make_inputs(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O, L = osattn.fwd_splitkv(qd, kd, vd, w.splits, scale=w.scale, causal=w.causal)
    assert osattn.get_device_status() == osattn.OK
    assert not torch.isnan(O).any().item() and torch.isfinite(L).all().item()
    rows = sample_rows(w.B, w.H, w.Nq, 64, seed=5)
    Oref, Lref = oracle.attention_fwd(q, k, v, w.scale, w.causal, None, rows=rows)
    idx = torch.tensor(rows, device=DEV)
    print(w.name, check(O.reshape(-1, w.d)[idx].double().cpu().numpy(),
                        L.reshape(-1)[idx].double().cpu().numpy(), Oref, Lref, "bf16"))


def test_splitkv_rejects_small_workspace_and_fp32():
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(osattn.OsattnError) as e:
        osattn.fwd_splitkv(q, q, q, 2, workspace=ws)
    assert e.value.status == osattn.ERR_INVALID_ARG
    qf = q.float()
    with pytest.raises(osattn.OsattnError) as e:
        osattn.fwd_splitkv(qf, qf, qf, 2)
    assert e.value.status == osattn.ERR_UNSUPPORTED
