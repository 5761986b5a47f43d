"""GPU tests of osattn_fwd_offload: host inputs copied in chunks of heads,
attended and copied back, pipelined on three streams.  The kernels see the
same data as a device-resident osattn_fwd call, and each unit of work is
independent of the others, so the host results must equal that call's bit
for bit, whatever the chunking; and they must pass the oracle gate."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_online_gb300 import osattn
from attention_forward_online_gb300.inputs import make_qkv

from _compare import check

pytestmark = pytest.mark.gpu
KIND = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}


def _bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("case", [
    # B, H, Nq, Nkv, d, causal, key_len, heads_per_chunk
    (2, 5, 300, 300, 128, True, None, 2),
    (2, 3, 200, 333, 64, False, [333, 100], 1),
    (1, 4, 256, 512, 128, False, [400], 8),
    (3, 7, 129, 700, 64, True, [700, 1, 64], 0),
], ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[5] else "") + f"h{c[7]}")
def test_offload_matches_device_call(case, dtype):
    B, H, Nq, Nkv, d, causal, kl, hpc = case
    q, k, v = make_qkv(B, H, Nq, Nkv, d, dtype, seed=5000 + H + Nq, q_std=1.5)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    kld = None if kl is None else torch.tensor(kl, dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(d)
    Oh, Lh = osattn.fwd_offload(qh, kh, vh, scale=scale, causal=causal, key_len=kld,
                                heads_per_chunk=hpc)
    torch.cuda.synchronize()
    assert osattn.get_device_status() == osattn.OK
    Od, Ld = osattn.fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal, key_len=kld)
    torch.cuda.synchronize()
    assert torch.equal(_bits(Oh), _bits(Od.cpu()))
    assert torch.equal(Lh, Ld.cpu())
    Oref, Lref = oracle.attention_fwd(q, k, v, scale, causal, kl)
    check(Oh.double().numpy(), Lh.double().numpy(), Oref, Lref, KIND[dtype])


def test_offload_waits_for_earlier_work_on_the_stream():
    # A kernel still writing the staging buffer on `stream` must finish
    # before the copies overwrite it: fill the buffers on the stream first.
    B, H, N, d = 1, 8, 1024, 128
    q, k, v = make_qkv(B, H, N, N, d, torch.bfloat16, seed=61)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    s = torch.cuda.Stream()
    qd = torch.empty_like(q, device="cuda")
    kd, vd = torch.empty_like(qd), torch.empty_like(qd)
    with torch.cuda.stream(s):
        for t in (qd, kd, vd):
            t.fill_(float("nan"))
        Oh, Lh = osattn.fwd_offload(qh, kh, vh, q=qd, k=kd, v=vd, causal=True, heads_per_chunk=3,
                                    stream=s)
    s.synchronize()
    Od, Ld = osattn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(_bits(Oh), _bits(Od.cpu())) and torch.equal(Lh, Ld.cpu())


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("case", [
    # B, H, Nq, Nkv, d, causal, key_len, heads_per_chunk
    (2, 5, 300, 300, 128, True, None, 2),
    (2, 3, 200, 333, 64, False, [333, 100], 0),
    # Nq not a multiple of 4: the chunks run in order on one stream
    (1, 4, 301, 256, 64, True, None, 1),
], ids=lambda c: "x".join(map(str, c[:5])) + ("c" if c[5] else "") + f"h{c[7]}")
def test_bwd_offload_matches_device_call(case, dtype):
    B, H, Nq, Nkv, d, causal, kl, hpc = case
    q, k, v = make_qkv(B, H, Nq, Nkv, d, dtype, seed=6000 + H + Nq, q_std=1.5)
    g = torch.Generator().manual_seed(6001)
    do = torch.randn(B, H, Nq, d, generator=g).to(dtype)
    kld = None if kl is None else torch.tensor(kl, dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(d)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = osattn.fwd(qd, kd, vd, scale=scale, causal=causal, key_len=kld)
    ref = osattn.bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal, key_len=kld)
    torch.cuda.synchronize()
    host = [t.pin_memory() for t in (q, k, v, o.cpu(), lse.cpu(), do)]
    out = osattn.bwd_offload(*host, scale=scale, causal=causal, key_len=kld, heads_per_chunk=hpc)
    torch.cuda.synchronize()
    assert osattn.get_device_status() == osattn.OK
    for a, b in zip(out, ref):
        assert torch.equal(_bits(a), _bits(b.cpu()))


@pytest.mark.parametrize("dtype", list(KIND), ids=list(KIND.values()))
@pytest.mark.parametrize("shape,rpc", [((1000, 4096), 0), ((37, 50000), 5), ((300, 1000), 64)])
def test_softmax_rows_offload_matches_device_call(shape, rpc, dtype):
    g = torch.Generator().manual_seed(71)
    x = (torch.randn(*shape, generator=g) * 3).to(dtype)
    yh, lh = osattn.softmax_rows_offload(x.pin_memory(), rows_per_chunk=rpc)
    torch.cuda.synchronize()
    yd, ld = osattn.softmax_rows(x.cuda())
    torch.cuda.synchronize()
    assert torch.equal(_bits(yh), _bits(yd.cpu())) and torch.equal(lh, ld.cpu())
    yh2, none = osattn.softmax_rows_offload(x.pin_memory(), want_lse=False, rows_per_chunk=rpc)
    torch.cuda.synchronize()
    assert none is None and torch.equal(_bits(yh2), _bits(yd.cpu()))


def test_offload_fully_masked_batch_and_oversized_chunks():
    # A batch entry with key_len 0 (O = 0, LSE = -inf, no NaN) and
    # heads_per_chunk above H (one chunk per batch entry).
    B, H, N, d = 2, 3, 200, 64
    q, k, v = make_qkv(B, H, N, N, d, torch.bfloat16, seed=81)
    kld = torch.tensor([N, 0], dtype=torch.int32, device="cuda")
    Oh, Lh = osattn.fwd_offload(q.pin_memory(), k.pin_memory(), v.pin_memory(), key_len=kld,
                                heads_per_chunk=100)
    torch.cuda.synchronize()
    assert torch.all(Oh[1] == 0) and torch.all(torch.isneginf(Lh[1]))
    assert torch.isfinite(Oh.float()).all() and torch.isfinite(Lh[0]).all()
    Od, Ld = osattn.fwd(q.cuda(), k.cuda(), v.cuda(), key_len=kld)
    torch.cuda.synchronize()
    assert torch.equal(_bits(Oh), _bits(Od.cpu())) and torch.equal(Lh, Ld.cpu())


def test_offload_reuses_buffers_across_calls():
    # Two calls in a row on the same staging buffers and stream: the second
    # call's copies in must wait for the first call's copies out.
    B, H, N, d = 1, 6, 512, 128
    s = torch.cuda.Stream()
    bufs = None
    outs = []
    for seed in (91, 92):
        q, k, v = make_qkv(B, H, N, N, d, torch.bfloat16, seed=seed)
        if bufs is None:
            bufs = [torch.empty_like(t, device="cuda") for t in (q, k, v, q)] + [
                torch.empty((B, H, N), dtype=torch.float32, device="cuda")]
        Oh, Lh = osattn.fwd_offload(q.pin_memory(), k.pin_memory(), v.pin_memory(), q=bufs[0],
                                    k=bufs[1], v=bufs[2], out=bufs[3], lse=bufs[4], causal=True,
                                    heads_per_chunk=2, stream=s)
        outs.append((q, k, v, Oh, Lh))
    s.synchronize()
    for q, k, v, Oh, Lh in outs:
        Od, Ld = osattn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(_bits(Oh), _bits(Od.cpu())) and torch.equal(Lh, Ld.cpu())
