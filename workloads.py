"""Seeded synthetic workloads for the FlashAttention-2 forward pass.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It draws inputs and counts work; it holds none of the attention
arithmetic itself.

Workloads follow the shapes named for this path (all tensors [B, H, N, D],
Q/K/V i.i.d. normal, cast to the 16-bit type with round-to-nearest-even):

  tiny      B=1  H=1  N=128    D=64   fp16  non-causal   seed 0
  pages     B=1  H=8  N=8192   D=64   fp16  non-causal   seed 1
            (the shape of the RTX 4090 table on the "FlashAttention-2 MMA
            代码学习" page, performance table at the top of the page)
  causal128 B=4  H=16 N=4096   D=128  bf16  causal       seed 2
  ragged    B=2  H=12 N=1000   D=64   fp16  non-causal   seed 3, Q/K ~ N(0, 3^2)
  long      B=1  H=4  N=32768  D=128  bf16  causal       seed 4
  target    B=1  H=8  N=8192   D=128  bf16  non-causal   seed 5
            (the N=8192, D=128 non-causal case the throughput goal is stated on)
  target_f16  same shape as target in fp16, seed 5
  target_b4   B=4 H=16 N=8192 D=128 bf16 non-causal, seed 6 (supplementary: more
              units per SM, less wave-quantisation tail)
  pages_d32   B=1 H=8 N=8192 D=32 fp16 non-causal, seed 7 (the pages' shape at
              the smallest head dimension the tiling_qk page lists)
  target_d96  B=1 H=8 N=8192 D=96 bf16 non-causal, seed 8 (the target shape at
              head dimension 96)
  target_d256 B=1 H=8 N=8192 D=256 bf16 non-causal, seed 9 (the target shape at
              the first head dimension of the tiling_qk page's d-tiled range)
  target_d512, target_d1024  the same at head dimensions 512 (seed 10) and
              1024 (seed 11), the largest the tiling_qk page's launcher takes

Scale is 1/sqrt(D) everywhere. Draw order: Q, then K, then V, each
``torch.randn(shape, dtype=float32, generator=g) * sigma`` from a CPU
generator seeded with the workload's seed, then cast to the 16-bit dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str          # "f16" or "bf16"
    causal: bool
    seed: int
    sigma_qk: float = 1.0
    sigma_v: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float16 if self.dtype == "f16" else torch.bfloat16

    def describe(self) -> str:
        return (f"B{self.B}-H{self.H}-N{self.N}-D{self.D} {self.dtype} "
                f"{'causal' if self.causal else 'non-causal'}")


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 128, 64, "f16", False, 0),
    "pages": Workload("pages", 1, 8, 8192, 64, "f16", False, 1),
    "causal128": Workload("causal128", 4, 16, 4096, 128, "bf16", True, 2),
    "ragged": Workload("ragged", 2, 12, 1000, 64, "f16", False, 3, sigma_qk=3.0),
    "long": Workload("long", 1, 4, 32768, 128, "bf16", True, 4),
    "target": Workload("target", 1, 8, 8192, 128, "bf16", False, 5),
    "target_f16": Workload("target_f16", 1, 8, 8192, 128, "f16", False, 5),
    "target_b4": Workload("target_b4", 4, 16, 8192, 128, "bf16", False, 6),
    "pages_d32": Workload("pages_d32", 1, 8, 8192, 32, "f16", False, 7),
    "target_d96": Workload("target_d96", 1, 8, 8192, 96, "bf16", False, 8),
    "target_d256": Workload("target_d256", 1, 8, 8192, 256, "bf16", False, 9),
    "target_d512": Workload("target_d512", 1, 8, 8192, 512, "bf16", False, 10),
    "target_d1024": Workload("target_d1024", 1, 8, 8192, 1024, "bf16", False, 11),
}

# The five workloads the parity contract names, in their stated order.
CONTRACT = ("tiny", "pages", "causal128", "ragged", "long")


def custom(B: int, H: int, N: int, D: int, dtype: str = "bf16", causal: bool = False,
           seed: int = 0, sigma_qk: float = 1.0, sigma_v: float = 1.0) -> Workload:
    """A workload of arbitrary shape (used by edge-case tests and sweeps)."""
    return Workload(f"B{B}H{H}N{N}D{D}{dtype}{'c' if causal else ''}s{seed}",
                    B, H, N, D, dtype, causal, seed, sigma_qk, sigma_v)


def make_inputs(w: Workload):
    """Return (q, k, v) as contiguous CPU tensors of the workload's 16-bit dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.D)
    q = torch.randn(shape, dtype=torch.float32, generator=g) * w.sigma_qk
    k = torch.randn(shape, dtype=torch.float32, generator=g) * w.sigma_qk
    v = torch.randn(shape, dtype=torch.float32, generator=g) * w.sigma_v
    dt = w.torch_dtype
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()


def make_grad_output(w: Workload) -> torch.Tensor:
    """The upstream gradient dO for the backward pass: i.i.d. N(0, 1) of the
    workload's shape, drawn from a CPU generator seeded with seed + 1000 (so
    Q, K, V are the forward's inputs unchanged), cast to the 16-bit dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 1000)
    shape = (w.B, w.H, w.N, w.D)
    return (torch.randn(shape, dtype=torch.float32, generator=g)).to(w.torch_dtype).contiguous()


def flops(w: Workload) -> float:
    """Metric FLOPs of one forward: 4*B*H*N^2*D, halved under the causal mask."""
    f = 4.0 * w.B * w.H * float(w.N) * w.N * w.D
    return f / 2.0 if w.causal else f


def algorithmic_bytes(w: Workload) -> int:
    """Compulsory HBM bytes: read Q, K, V once, write O (16-bit) and LSE (fp32)."""
    elems = w.B * w.H * w.N * w.D
    return 4 * elems * 2 + w.B * w.H * w.N * 4


def with_seed(w: Workload, seed: int) -> Workload:
    return replace(w, seed=seed)


def bwd_flops(w: Workload) -> float:
    """Metric FLOPs of one backward: five N x N x D matrix products per head
    (S, dP, dV, dK, dQ), 10*B*H*N^2*D, halved under the causal mask
    (2.5 times the forward's)."""
    return 2.5 * flops(w)


def bwd_algorithmic_bytes(w: Workload) -> int:
    """Compulsory HBM bytes of one backward: read Q, K, V, O, dO (16-bit) and
    LSE (fp32) once, write dQ, dK, dV (16-bit)."""
    elems = w.B * w.H * w.N * w.D
    return 8 * elems * 2 + w.B * w.H * w.N * 4


# ------------------------------------------------------------ structured inputs
# Inputs shaped to reach the corners of the online softmax: the exponent base
# moving on many K/V tiles, every score far below zero, and one dominant key
# in a ragged last tile. They change only how Q, K, V are drawn (directions,
# magnitudes, signs); the attention arithmetic is elsewhere.
STRUCTURED_KINDS = ("rising", "negative", "dominant_last")

RISE_NATS_PER_TILE = 12.0   # "rising": growth of the scores per 128 keys (natural-log units)
NEGATIVE_NATS = 180.0       # "negative": typical magnitude of the (all negative) scores
DOMINANT_NATS = 25.0        # "dominant_last": the dominant key's score above the rest


def dominant_key(N: int) -> int:
    """The dominant key of the "dominant_last" inputs: four keys into the last
    128-key tile (the last key if that tile is shorter), so that under the
    causal mask the rows from it to N-1 see it."""
    start = 128 * ((N - 1) // 128)
    return min(start + 4, N - 1)


def make_structured_inputs(w: Workload, kind: str):
    """(q, k, v) of the workload's shape and dtype, drawn to reach one corner case.

    rising:        Q_i = sqrt(D) u + noise and K_j = c_j u + noise for a unit
                   direction u per head, c_j growing by RISE_NATS_PER_TILE per
                   128 keys, so that scale * <Q_i, K_j> is about c_j: every
                   row's maximum rises tile after tile.
    negative:      Q >= 0 and K <= -c elementwise, with c set so that the
                   scores are about -NEGATIVE_NATS: every score of every row
                   is far below zero.
    dominant_last: Q_i = sqrt(D) u + noise, K ~ N(0, 1) except the key
                   dominant_key(N) = DOMINANT_NATS u: one key, in the last
                   (ragged) K/V tile, outweighs all others by about
                   DOMINANT_NATS.
    V ~ N(0, sigma_v^2) in every case. Draw order from the seeded CPU
    generator: u, then the kind's noise terms, then V.
    """
    if kind not in STRUCTURED_KINDS:
        raise ValueError(f"unknown kind {kind!r}")
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    B, H, N, D = w.B, w.H, w.N, w.D
    shape = (B, H, N, D)
    u = torch.randn((B, H, 1, D), dtype=torch.float64, generator=g)
    u = u / u.norm(dim=-1, keepdim=True)
    rd = math.sqrt(D)
    if kind == "rising":
        c = (torch.arange(N, dtype=torch.float64) * (RISE_NATS_PER_TILE / 128.0)).view(1, 1, N, 1)
        q = rd * u + 0.5 * torch.randn(shape, dtype=torch.float64, generator=g)
        k = c * u + 0.5 * torch.randn(shape, dtype=torch.float64, generator=g)
    elif kind == "negative":
        # E|z| = sqrt(2/pi) for z ~ N(0, 1): scores ~ -(1/sqrt(D)) * D * E|z| * (c + E|z|)
        ez = math.sqrt(2.0 / math.pi)
        cneg = NEGATIVE_NATS / (rd * ez) - ez
        q = torch.randn(shape, dtype=torch.float64, generator=g).abs()
        k = -(cneg + torch.randn(shape, dtype=torch.float64, generator=g).abs())
    else:
        q = rd * u + 0.5 * torch.randn(shape, dtype=torch.float64, generator=g)
        k = torch.randn(shape, dtype=torch.float64, generator=g)
        k[:, :, dominant_key(N), :] = DOMINANT_NATS * u[:, :, 0, :]
    v = torch.randn(shape, dtype=torch.float64, generator=g) * w.sigma_v
    dt = w.torch_dtype
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()
