"""The allocation-free split-KV entry point against the workspace one.

osattn_fwd_splitkv_noalloc serves callers that cannot allocate device
memory (an application whose memory manager owns the device budget, or a
latency-critical path that cannot afford cudaMalloc): its partial results
live in a fixed array inside the library instead of a caller workspace.
This file is collected last so that a failure here leaves every other test
already run; it passes both alone in a fresh process and after the others.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from attention_forward_online_gb300 import osattn
from attention_forward_online_gb300.inputs import make_qkv

from _compare import check

pytestmark = pytest.mark.gpu
DEV = "cuda"


def noalloc_call(q, k, v, splits, causal=False, key_len=None):
    """Direct C-ABI call of osattn_fwd_splitkv_noalloc on torch's stream."""
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    O = torch.full_like(q, float("nan"))
    L = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=q.device)
    kl = None if key_len is None else key_len.data_ptr()
    rc = osattn.lib().osattn_fwd_splitkv_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), L.data_ptr(), B, H, Nq, Nkv, d,
        1.0 / math.sqrt(d), int(causal), kl, osattn.BF16, splits,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == osattn.OK, osattn.status_string(rc)
    return O, L


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    # Two different problems back to back: the second must not see anything
    # the first left in the shared scratch array.
    problems = [
        (2, 4, 512, 3000, 128, True, [3000, 1500], 7, 51),
        (1, 3, 300, 5000, 64, False, None, 5, 52),
    ]
    for B, H, Nq, Nkv, d, causal, kl, splits, seed in problems:
        q, k, v = (t.to(DEV) for t in make_qkv(B, H, Nq, Nkv, d, torch.bfloat16, seed=seed))
        klt = None if kl is None else torch.tensor(kl, dtype=torch.int32, device=DEV)
        O_ref, L_ref = osattn.fwd_splitkv(q, k, v, splits, causal=causal, key_len=klt)
        O, L = noalloc_call(q, k, v, splits, causal, klt)
        assert osattn.get_device_status() == osattn.OK
        check(O.double().cpu().numpy(), L.double().cpu().numpy(),
              O_ref.double().cpu().numpy(), L_ref.double().cpu().numpy(), "bf16")


def test_noalloc_rejects_a_problem_beyond_its_scratch():
    q = torch.zeros(4, 8, 4096, 128, dtype=torch.bfloat16, device=DEV)
    rc = osattn.lib().osattn_fwd_splitkv_noalloc(
        q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), 4, 8, 4096, 4096,
        128, 0.125, 0, None, osattn.BF16, 4, ctypes.c_void_p(None))
    assert rc == osattn.ERR_SCRATCH_LIMIT
