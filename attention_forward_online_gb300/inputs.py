"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random tensors; it holds none of the attention
arithmetic.  Both the CUDA path and the fp64 oracle are fed the same
quantised bytes produced here.

Recipe: a CPU ``torch.Generator`` seeded per workload draws, in this order,
Q, K and V as ``torch.randn`` in fp32, each multiplied by its standard
deviation, then rounded to the workload dtype (round-to-nearest-even).  The
pages use no dataset; the five workloads below reproduce the shapes and value
distributions the attention forward pass is specified on (the LLaMA-2-13B
head shape H=40, d=128 at batch 8 / sequence 2048 is the one the
"FlashAttention 2.0" article times on an A100).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import torch


TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "bf16", "fp16" or "fp32"
    B: int
    H: int
    Nq: int
    Nkv: int
    d: int
    causal: bool
    key_len: Optional[Tuple[int, ...]]
    seed: int
    q_std: float = 1.0
    kv_std: float = 1.0
    splits: int = 0  # > 0: measured through the split-KV entry point with this many ranges
    bwd: bool = False  # True: the backward pass (dQ, dK, dV) is measured

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Nominal forward FLOPs: 4*B*H*Nq*Nkv*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.Nq * self.Nkv * self.d
        return f / 2 if self.causal else f

    def torch_dtype(self):
        return TORCH_DTYPES[self.dtype]

    @property
    def bwd_flops(self) -> float:
        """Nominal backward FLOPs: the five products S, dP, dV, dK, dQ of
        2*N*N*d each per head, 2.5 times the forward count."""
        return 2.5 * self.flops


WORKLOADS = {
    w.name: w
    for w in [
        Workload("fp32_b1_h1_n128_d64", "fp32", 1, 1, 128, 128, 64, False, None, seed=0),
        Workload("bf16_b2_h4_n1024_d64_keypad", "bf16", 2, 4, 1024, 1024, 64, False,
                 (1024, 724), seed=1),
        Workload("bf16_causal_b4_h16_n4096_d64", "bf16", 4, 16, 4096, 4096, 64, True,
                 None, seed=2),
        Workload("bf16_b8_h40_n2048_d128", "bf16", 8, 40, 2048, 2048, 128, False, None,
                 seed=3),
        Workload("bf16_causal_b1_h32_n16384_d128_qstd3", "bf16", 1, 32, 16384, 16384, 128,
                 True, None, seed=4, q_std=3.0),
    ]
}

# Workloads for the split-KV path: few (b, h) rows with long key sequences,
# where one CTA per 256 query rows cannot fill 152 SMs (16 CTAs here); the
# key axis is cut into 9 ranges (144 CTAs).
SPLITKV_WORKLOADS = {
    w.name: w
    for w in [
        Workload("bf16_b1_h8_q512_kv65536_d128", "bf16", 1, 8, 512, 65536, 128, False, None,
                 seed=5, splits=9),
    ]
}

# Backward-pass workloads: the two largest forward shapes, with an upstream
# gradient dO ~ N(0, 1) drawn after Q, K and V from the workload's seed + 1000.
BWD_WORKLOADS = {
    w.name: w
    for w in [
        Workload("bwd_bf16_b8_h40_n2048_d128", "bf16", 8, 40, 2048, 2048, 128, False, None,
                 seed=3, bwd=True),
        Workload("bwd_bf16_causal_b1_h32_n16384_d128_qstd3", "bf16", 1, 32, 16384, 16384, 128,
                 True, None, seed=4, q_std=3.0, bwd=True),
    ]
}


def make_grad_out(w: Workload):
    """Upstream gradient dO [B,H,Nq,d] ~ N(0, 1) on the CPU, in the workload dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 1000)
    return torch.randn((w.B, w.H, w.Nq, w.d), generator=g, dtype=torch.float32).to(w.torch_dtype())


@dataclasses.dataclass(frozen=True)
class RowWorkload:
    """A [rows, N] matrix of logits for the standalone row softmax."""
    name: str
    dtype: str
    rows: int
    N: int
    seed: int
    std: float = 3.0

    def torch_dtype(self):
        return TORCH_DTYPES[self.dtype]

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "fp32" else 2

    @property
    def bytes_moved(self) -> int:
        """Read once + write once per element, plus the fp32 LSE per row."""
        return self.rows * self.N * self.elem_bytes * 2 + self.rows * 4


# The chapter's exercise is a whole-row softmax at N = 4096; 65536 such rows
# (512 MiB of bf16 each way) keep every SM streaming and exceed L2.
ROW_WORKLOADS = {
    w.name: w
    for w in [
        RowWorkload("softmax_rows_bf16_r65536_n4096", "bf16", 65536, 4096, seed=6),
        RowWorkload("softmax_rows_fp32_r32768_n4096", "fp32", 32768, 4096, seed=7),
        # the chapter's closing exercise: rows of 1M elements, each split
        # across the CTAs of a thread-block cluster
        RowWorkload("softmax_rows_bf16_r256_n1048576", "bf16", 256, 1 << 20, seed=8),
        RowWorkload("softmax_rows_fp32_r128_n1048576", "fp32", 128, 1 << 20, seed=9),
    ]
}


def make_rows(w: RowWorkload):
    """Logits [rows, N] ~ N(0, std^2) on the CPU, rounded to the dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    return (torch.randn((w.rows, w.N), generator=g, dtype=torch.float32) * w.std).to(w.torch_dtype())


# The workload the benchmark times by default: the largest bf16 one.
BENCH_WORKLOAD = "bf16_causal_b1_h32_n16384_d128_qstd3"


def make_qkv(B: int, H: int, Nq: int, Nkv: int, d: int, dtype, seed: int,
             q_std: float = 1.0, kv_std: float = 1.0):
    """Q [B,H,Nq,d], K and V [B,H,Nkv,d] on the CPU, drawn as described above."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, Nkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, Nkv, d), generator=g, dtype=torch.float32)
    if q_std != 1.0:
        q.mul_(q_std)
    if kv_std != 1.0:
        k.mul_(kv_std)
        v.mul_(kv_std)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def make_inputs(w: Workload):
    """(Q, K, V, key_len or None) for a workload, on the CPU."""
    q, k, v = make_qkv(w.B, w.H, w.Nq, w.Nkv, w.d, w.torch_dtype(), w.seed, w.q_std, w.kv_std)
    kl = None if w.key_len is None else torch.tensor(w.key_len, dtype=torch.int32)
    return q, k, v, kl


def sample_rows(B: int, H: int, Nq: int, n: int, seed: int, include_edges: bool = True):
    """A seeded list of flat row indices (b*H+h)*Nq+i for spot checks at full
    size; always includes the first and last row of the first and last
    (b, h) and the rows around every 128-row tile edge of one head."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    total = B * H * Nq
    picks = set(torch.randint(0, total, (n,), generator=g).tolist())
    if include_edges:
        last_bh = (B * H - 1) * Nq
        for base in (0, last_bh):
            picks.update({base, base + Nq - 1})
        bh = int(torch.randint(0, B * H, (1,), generator=g))
        for t in range(0, Nq, 128):
            for off in (t, t + 127):
                if off < Nq:
                    picks.add(bh * Nq + off)
    return sorted(picks)
