"""The allocation-free split-KV entry point against the workspace one.

osattn_fwd_splitkv_noalloc serves callers that cannot allocate device
memory (an application whose memory manager owns the device budget, or a
latency-critical path that cannot afford cudaMalloc): its partial results
live in a fixed array inside the library instead of a caller workspace.
Its results are compared with the workspace entry point's (bit for bit) and
with the fp64 oracle, after NaN was left in the shared array.  This file is collected last so that a failure here leaves every other test
already run; it passes both alone in a fresh process and after the others.
"""
import ctypes
import math

import pytest
import torch

import oracle
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


def poison_scratch():
    """Leaves NaN partials over almost all of the shared scratch array (31.7 MB
    of its 32 MiB): a call whose values are NaN, so every partial O is NaN."""
    q = torch.zeros(2, 4, 512, 128, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(2, 4, 1024, 128, dtype=torch.bfloat16, device=DEV)
    v = torch.full((2, 4, 1024, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    assert osattn.splitkv_workspace_bytes(2, 4, 512, 128, 15) > 0.9 * osattn.NOALLOC_SCRATCH_BYTES
    O, _ = noalloc_call(q, k, v, 15)
    torch.cuda.synchronize()
    assert torch.isnan(O.float()).any().item()


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    # Two different problems back to back, after a call that filled the
    # shared array with NaN: each must equal the workspace entry point bit
    # for bit (same kernels, same splits) and meet the oracle's gates, so
    # nothing left in the array by an earlier call reaches a result.
    problems = [
        (2, 4, 512, 3000, 128, True, [3000, 1500], 7, 51),
        (1, 3, 300, 5000, 64, False, None, 5, 52),
    ]
    poison_scratch()
    for B, H, Nq, Nkv, d, causal, kl, splits, seed in problems:
        qc, kc, vc = make_qkv(B, H, Nq, Nkv, d, torch.bfloat16, seed=seed)
        q, k, v = qc.to(DEV), kc.to(DEV), vc.to(DEV)
        klt = None if kl is None else torch.tensor(kl, dtype=torch.int32, device=DEV)
        O_ws, L_ws = osattn.fwd_splitkv(q, k, v, splits, causal=causal, key_len=klt)
        O, L = noalloc_call(q, k, v, splits, causal, klt)
        assert osattn.get_device_status() == osattn.OK
        assert torch.equal(O.view(torch.int16), O_ws.view(torch.int16))
        assert torch.equal(L.view(torch.int32), L_ws.view(torch.int32))
        O_ref, L_ref = oracle.attention_fwd(qc, kc, vc, 1.0 / math.sqrt(d), causal, kl)
        check(O.double().cpu().numpy(), L.double().cpu().numpy(), O_ref, L_ref, "bf16")


def test_noalloc_call_takes_no_device_memory():
    q, k, v = (t.to(DEV) for t in make_qkv(1, 2, 256, 2048, 128, torch.bfloat16, seed=53))
    noalloc_call(q, k, v, 4)  # warm-up: kernels loaded, scratch address looked up
    O = torch.empty_like(q)
    L = torch.empty(1, 2, 256, dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        rc = osattn.lib().osattn_fwd_splitkv_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), L.data_ptr(), 1, 2, 256, 2048,
            128, 1.0 / math.sqrt(128), 0, None, osattn.BF16, 4,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == osattn.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert osattn.get_device_status() == osattn.OK


def test_noalloc_rejects_a_problem_beyond_its_scratch():
    q = torch.zeros(4, 8, 4096, 128, dtype=torch.bfloat16, device=DEV)
    rc = osattn.lib().osattn_fwd_splitkv_noalloc(
        q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), 4, 8, 4096, 4096,
        128, 0.125, 0, None, osattn.BF16, 4, ctypes.c_void_p(None))
    assert rc == osattn.ERR_SCRATCH_LIMIT
