"""fp64 oracle for the bf16 GEMM C = A B^T (A [M, K], B [N, K], row-major).

TEST INFRASTRUCTURE ONLY (see the package docstring).  The plain definition
C_ij = sum_k a_ik b_jk with every bf16 input widened exactly to float64; the
library matrix product (numpy, float64) serves as the one step, as a plain
definition allows.  Also returns the per-element magnitude sum
sum_k |a_ik b_jk|, which bounds the rounding of any fp32 accumulation order.

Source: the GEMM the ThunderKittens paper summary benchmarks against cuBLAS
("ThunderKittens: Simple, Fast, and Adorable AI Kernels", shd-paper.top,
abstract and experimental highlights: GEMM on a par with cuBLAS); the pages
give no kernel for it, so the definition here is the textbook one.
"""
import numpy as np

from .brute import _bf16_bits


def _widen(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm_abt(a, b):
    """C = A B^T in float64 and sum_k |a_ik b_jk|; a, b bf16 (tensors or bits)."""
    A = _widen(np.ascontiguousarray(_bf16_bits(a)))
    B = _widen(np.ascontiguousarray(_bf16_bits(b)))
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("a must be [M, K] and b [N, K]")
    return A @ B.T, np.abs(A) @ np.abs(B).T
