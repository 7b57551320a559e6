"""Seeded synthetic inputs shaped like the FlashAttention pages' workloads.

This module holds no attention arithmetic: it only draws random tensors and
names the workload shapes.  Both the CUDA path and the fp64 checker consume
the same bf16 tensors drawn here.

Recipe: entries are i.i.d. N(0, 1), drawn in fp32 on the CPU with a seeded
``torch.Generator`` and rounded once to bf16 (round to nearest even).  The
long-context workload multiplies every 64th query row by 10 before the
rounding, so that a row's running maximum jumps late in the sweep.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    backward: bool
    boost_every: int = 0   # every k-th query row scaled (0 = none)
    boost: float = 1.0

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d), rounded to fp32 as the kernels receive it."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    def fwd_flops(self) -> float:
        """Counted forward FLOPs: 4*B*H*N^2*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        """Counted backward FLOPs: 2.5x the forward count."""
        return 2.5 * self.fwd_flops()


# Shapes of the five workloads the method is measured on.
WORKLOADS = {
    "single_head_n256_d64": Workload("single_head_n256_d64", 1, 1, 256, 64, False, False),
    "memory_exercise_n4096_d64": Workload("memory_exercise_n4096_d64", 1, 1, 4096, 64, False, False),
    "memory_exercise_n4096_d64_causal": Workload("memory_exercise_n4096_d64_causal", 1, 1, 4096, 64, True, False),
    "throughput_b8_h16_n4096_d64": Workload("throughput_b8_h16_n4096_d64", 8, 16, 4096, 64, False, False),
    "throughput_b8_h16_n4096_d64_causal": Workload("throughput_b8_h16_n4096_d64_causal", 8, 16, 4096, 64, True, False),
    "training_b4_h16_n8192_d128_causal": Workload("training_b4_h16_n8192_d128_causal", 4, 16, 8192, 128, True, True),
    "long_context_b1_h32_n16384_d128_causal": Workload(
        "long_context_b1_h32_n16384_d128_causal", 1, 32, 16384, 128, True, True, boost_every=64, boost=10.0),
    "very_long_b1_h8_n65536_d128_causal": Workload("very_long_b1_h8_n65536_d128_causal", 1, 8, 65536, 128, True, False),
}


def randn_bf16(shape, seed: int) -> torch.Tensor:
    """Seeded N(0,1) draw in fp32 on the CPU, rounded to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)



@dataclass(frozen=True)
class DecodeWorkload:
    """One decoding step: Nq query rows per head against Nk cached keys and
    values (causal, aligned at the last key)."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool = True

    @property
    def scale(self) -> float:
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    def kv_bytes(self) -> int:
        """K and V read once: the compulsory HBM traffic that bounds the step."""
        return 2 * self.B * self.H * self.Nk * self.d * 2

    def hbm_bytes(self) -> int:
        """K, V and q read (bf16), O (fp32) and LSE (fp32) written."""
        rows = self.B * self.H * self.Nq
        return self.kv_bytes() + rows * self.d * 2 + rows * self.d * 4 + rows * 4

    def flops(self) -> float:
        """4*d FLOPs per (query, eligible key) pair."""
        pairs = sum(min(i + 1 + self.Nk - self.Nq, self.Nk) if self.causal else self.Nk for i in range(self.Nq))
        return 4.0 * self.B * self.H * pairs * self.d


# A decoding step of 8 sequences x 32 heads over a 32k-token cache: K and V
# are 4.3 GB, far larger than L2, and are read once.
DECODE_WORKLOADS = {
    "decode_b8_h32_nq1_nk32768_d128": DecodeWorkload("decode_b8_h32_nq1_nk32768_d128", 8, 32, 1, 32768, 128),
    # a quarter of the batch (1.07 GB of K/V, still far larger than L2): the
    # size on which multi-pass profiler captures are taken
    "decode_b2_h32_nq1_nk32768_d128": DecodeWorkload("decode_b2_h32_nq1_nk32768_d128", 2, 32, 1, 32768, 128),
}


def make_decode_inputs(B: int, H: int, Nq: int, Nk: int, d: int, seed: int = 0) -> dict:
    """CPU bf16 q [B, H, Nq, d] and k, v [B, H, Nk, d], successive N(0, 1)
    draws of one seeded generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = {}
    for name, n in (("q", Nq), ("k", Nk), ("v", Nk)):
        out[name] = torch.randn(B, H, n, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def make_inputs(B: int, H: int, N: int, d: int, seed: int = 0, with_grad: bool = False,
                boost_every: int = 0, boost: float = 1.0) -> dict:
    """Return CPU bf16 tensors q, k, v (and dO) of shape [B, H, N, d].

    Each tensor has its own derived seed so that q, k, v and dO are
    independent draws.  With ``boost_every`` = k > 0, query rows i with
    i % k == 0 are multiplied by ``boost`` in fp32 before the bf16 rounding.
    """
    shape = (B, H, N, d)
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = {}
    names = ["q", "k", "v"] + (["do"] if with_grad else [])
    for name in names:
        x = torch.randn(*shape, generator=g, dtype=torch.float32)
        if name == "q" and boost_every > 0:
            x[:, :, ::boost_every, :] *= boost
        out[name] = x.to(torch.bfloat16)
    return out


def make_fp8_inputs(B: int, H: int, N: int, d: int, seed: int = 0) -> dict:
    """Seeded N(0,1) q, k, v rounded to FP8 E4M3 by torch's float32 ->
    float8_e4m3fn cast, as uint8 bit patterns: q, k, v [B, H, N, d] and vt,
    v transposed to [B, H, d, N] (the layout the FP8 forward reads V in)."""
    g = torch.Generator().manual_seed(seed)
    q, k, v = (torch.randn((B, H, N, d), generator=g) for _ in range(3))
    q8, k8, v8 = (t.to(torch.float8_e4m3fn).view(torch.uint8) for t in (q, k, v))
    return {"q": q8, "k": k8, "v": v8, "vt": v8.transpose(-1, -2).contiguous()}


def fp8_values(t: torch.Tensor) -> torch.Tensor:
    """float32 values of E4M3 bit patterns held as uint8."""
    return t.view(torch.float8_e4m3fn).to(torch.float32)


def workload_inputs(w: Workload, seed: int = 0) -> dict:
    return make_inputs(w.B, w.H, w.N, w.d, seed=seed, with_grad=w.backward,
                       boost_every=w.boost_every, boost=w.boost)


def sample_rows(B: int, H: int, N: int, count: int, seed: int) -> list:
    """Seeded sample of distinct (b, h, i) query rows, always including the
    first and the last row of the first head."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7919)
    total = B * H * N
    picks = {(0, 0, 0), (0, 0, N - 1)}
    while len(picks) < min(count, total):
        flat = int(torch.randint(0, total, (1,), generator=g))
        bh, i = divmod(flat, N)
        picks.add((bh // H, bh % H, i))
    return sorted(picks)
