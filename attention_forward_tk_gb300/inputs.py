"""Seeded synthetic inputs for the attention forward workloads.

This module only draws random numbers and rounds them to bf16; it holds no
attention arithmetic, so the CUDA path and the CPU oracle can both be fed from
it without sharing any part of the method.

Workloads (the five problem shapes the library is measured and checked on):

  name            B   H   N      D    mask     values
  n256_d64        1   1   256    64   none     Q, K, V ~ N(0, 1)
  n1024_d64       16  16  1024   64   none     Q, K, V ~ N(0, 1)
  n4096_d128      16  16  4096   128  none     Q, K, V ~ N(0, 1)
  n8192_d128_c    8   16  8192   128  causal   Q, K, V ~ N(0, 1)
  n16384_d128_c   4   32  16384  128  causal   Q, K ~ 4 N(0, 1);
                                               V ~ Student-t(3), clipped to +-8

and three inference shapes, queries and keys of different lengths (timed
beside them, split over keys):

  prefill_q256_k32k_d128   B 1, H 32, Nq 256, Nk 32768, D 128, unmasked, N(0, 1)
  chunk_q1024_k16k_d128_c  B 1, H 32, Nq 1024, Nk 16384, D 128, causal (the queries
                           are the last 1024 positions), N(0, 1), seed 9
  decode_b8_q1_k16k_d128   B 8, H 32, Nq 1, Nk 16384, D 128, unmasked, N(0, 1), seed 10

the backward pass (tk_attn_bwd) on the shapes of n4096_d128 and n8192_d128_c,
with the output gradient dO ~ N(0, 1) drawn after Q, K, V by draw_grad(),

Based linear attention (tk_based_fwd) on B16 H16 N4096, causal, with 16-wide
feature rows q, k ~ N(0, 1) and 64-wide values v ~ N(0, 1) (draw_based),

and one dense GEMM shape for tk_gemm_bf16 (C = A B^T):

  gemm_8192   M = N = K = 8192, A and B ~ N(0, 1)

The scale is 1/sqrt(D) in every workload (the kernel examples on the pages use
1/sqrt(64) = 0.125 and 1/sqrt(128) ~= 0.08838834764).

Recipe: a CPU ``torch.Generator`` seeded with the workload's index (0..5) draws
Q, then K, then V, in float32, with the shape [B, H, N, D] (K and V [B, H, Nk,
D] for the inference shape); scaling (4 N(0,1))
and clipping happen in float32 before one round-to-nearest-even conversion to
bfloat16.  A Student-t(3) draw is z / sqrt((z1^2 + z2^2 + z3^2) / 3) with all
four normals from the same generator (z first, then a [..., 3] block).
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
    D: int
    causal: bool
    dist: str  # "normal" or "peaky_t3"
    seed: int
    Nk: int = 0  # keys per slice when it differs from N (inference shapes)

    @property
    def keys(self) -> int:
        return self.Nk or self.N

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def shape(self):
        return (self.B, self.H, self.N, self.D)

    @property
    def kv_shape(self):
        return (self.B, self.H, self.keys, self.D)

    @property
    def flops(self) -> float:
        """4*B*H*D times the (query, key) pairs: N*Nk unmasked; under the causal
        mask N^2/2 when Nk = N (the metric's halving), and the visible pairs
        Nq*Nk - Nq*(Nq-1)/2 when the Nq queries are the last positions of Nk."""
        if self.causal and self.Nk:
            pairs = self.N * self.Nk - self.N * (self.N - 1) / 2
        else:
            pairs = self.N * self.keys / (2 if self.causal else 1)
        return 4.0 * self.B * self.H * self.D * pairs

    @property
    def io_bytes(self) -> int:
        """Q, K, V read and O written in bf16, LSE written in fp32."""
        q_elems = self.B * self.H * self.N * self.D
        kv_elems = self.B * self.H * self.keys * self.D
        return (2 * q_elems + 2 * kv_elems) * 2 + self.B * self.H * self.N * 4


WORKLOADS = (
    Workload("n256_d64", 1, 1, 256, 64, False, "normal", 0),
    Workload("n1024_d64", 16, 16, 1024, 64, False, "normal", 1),
    Workload("n4096_d128", 16, 16, 4096, 128, False, "normal", 2),
    Workload("n8192_d128_c", 8, 16, 8192, 128, True, "normal", 3),
    Workload("n16384_d128_c", 4, 32, 16384, 128, True, "peaky_t3", 4),
)
# Inference shapes (tk_attn_fwd_qk, split over keys): queries against a
# longer run of cached keys.  Not among the five measured configurations;
# timed beside them (bench.py --all-workloads).
EXTRA_WORKLOADS = (
    Workload("prefill_q256_k32k_d128", 1, 32, 256, 128, False, "normal", 5, Nk=32768),
    # a causal prefill chunk: the last 1024 positions of a 16384-token sequence
    Workload("chunk_q1024_k16k_d128_c", 1, 32, 1024, 128, True, "normal", 9, Nk=16384),
    # a decode step: one query per sequence against 16384 cached keys, 8 sequences
    Workload("decode_b8_q1_k16k_d128", 8, 32, 1, 128, False, "normal", 10, Nk=16384),
)
BY_NAME = {w.name: w for w in WORKLOADS + EXTRA_WORKLOADS}


def _randn(g: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32, device=g.device)


def _student_t3(g: torch.Generator, shape) -> torch.Tensor:
    z = _randn(g, shape)
    w = _randn(g, tuple(shape) + (3,))
    chi2_over_nu = (w * w).sum(dim=-1) / 3.0
    return z / torch.sqrt(chi2_over_nu)


def draw(shape, seed: int, dist: str = "normal", device="cpu", kv_shape=None):
    """Q, K, V as bf16 tensors of `shape`, per the recipe above.

    With the default CPU generator the values are the ones every parity test
    and the oracle see.  `device="cuda"` draws the same distributions with
    the device's generator (other values, no host work): the benchmark uses
    it for full-size inputs it does not compare.
    """
    kvs = shape if kv_shape is None else kv_shape
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    if dist == "normal":
        q = _randn(g, shape)
        k = _randn(g, kvs)
        v = _randn(g, kvs)
    elif dist == "peaky_t3":
        q = 4.0 * _randn(g, shape)
        k = 4.0 * _randn(g, kvs)
        v = _student_t3(g, kvs).clamp_(-8.0, 8.0)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return (q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16))


def draw_grad(shape, seed: int, device="cpu"):
    """dO for the backward pass: N(0, 1) rounded to bf16, from a generator
    seeded with 1000 + seed (so it never repeats the draw of Q, K, V)."""
    g = torch.Generator(device=device)
    g.manual_seed(1000 + int(seed))
    return _randn(g, shape).to(torch.bfloat16)


# The backward pass is measured on the forward's D = 128 shapes.
BWD_WORKLOADS = tuple(w for w in WORKLOADS if w.name in ("n4096_d128", "n8192_d128_c"))


@dataclass(frozen=True)
class BasedWorkload:
    name: str
    B: int
    H: int
    N: int
    causal: bool
    seed: int
    Df: int = 16
    Dv: int = 64

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.Df)

    @property
    def flops(self) -> float:
        """Tensor-core FLOPs of the direct (quadratic) evaluation: per visible
        (query, key) pair 2 Df for the score and 2 Dv for the weighted value,
        N^2 pairs per slice (halved under the causal mask)."""
        pairs = self.N * self.N / (2 if self.causal else 1)
        return self.B * self.H * pairs * 2.0 * (self.Df + self.Dv)

    @property
    def linear_flops(self) -> float:
        """Tensor FLOPs the linear-time kernel (tk_based_fwd_linear) executes:
        per 128-position chunk Q K^T (K 16) and A V_ext (N 128: the 64 values,
        the ones column of z, padding); phi(Q) S (K 160) for every chunk but
        a slice's first, and the state update (N 160) for every chunk but its
        last."""
        nc = (self.N + 127) // 128
        per_chunk = 2.0 * 128 * 128 * (16 + 128)
        state = 2.0 * 128 * 128 * 160
        return self.B * self.H * (nc * per_chunk + 2 * (nc - 1) * state)


BASED_WORKLOADS = (BasedWorkload("based_n4096_c", 16, 16, 4096, True, 8),)
BASED_BY_NAME = {w.name: w for w in BASED_WORKLOADS}


def draw_based(B: int, H: int, N: int, seed: int, Df: int = 16, Dv: int = 64, device="cpu"):
    """q, k [B, H, N, Df] then v [B, H, N, Dv], N(0, 1) rounded to bf16, from
    one generator seeded with `seed`."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    q = _randn(g, (B, H, N, Df))
    k = _randn(g, (B, H, N, Df))
    v = _randn(g, (B, H, N, Dv))
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


@dataclass(frozen=True)
class GemmWorkload:
    name: str
    M: int
    N: int
    K: int
    seed: int

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def io_bytes(self) -> int:
        """A and B read, C written, bf16."""
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


# The square bf16 product the pages compare with cuBLAS, at the size the
# cuBLAS peak of this GPU is measured on.
GEMM_WORKLOADS = (GemmWorkload("gemm_8192", 8192, 8192, 8192, 6),)
GEMM_BY_NAME = {w.name: w for w in GEMM_WORKLOADS}


def draw_gemm(M: int, N: int, K: int, seed: int, device="cpu"):
    """A [M, K] then B [N, K], N(0, 1) rounded to bf16, from one generator
    seeded with `seed` (the same recipe as draw())."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    a = _randn(g, (M, K))
    b = _randn(g, (N, K))
    return a.to(torch.bfloat16), b.to(torch.bfloat16)


def workload_inputs(w: Workload, device="cpu"):
    return draw(w.shape, w.seed, w.dist, device=device, kv_shape=w.kv_shape)
