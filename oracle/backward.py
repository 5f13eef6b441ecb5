"""fp64 oracle for the attention backward pass: dQ, dK, dV.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages give no formulas for the backward pass.  They report that the
library ships causal and non-causal FlashAttention backward kernels (the
comment thread of the Spanish news page, es.news.hada.io topic 14783) that
beat the strongest baselines by 10-40% (the paper summary "ThunderKittens:
Simple, Fast, and Adorable AI Kernels", shd-paper.top, abstract).  The
gradient is therefore the calculus of the forward definition the kernel
examples compute, O = softmax_row(S) V with S = scale Q K^T (masked entries
-inf), written out step by step for a loss L with dL/dO = dO:

  dV = P^T dO                                  (O is linear in V)
  dP = dO V^T                                  (O is linear in P)
  dS_ij = P_ij (dP_ij - sum_l P_il dP_il)      (Jacobian of one softmax row)
  dQ = scale dS K,   dK = scale dS^T Q         (S is bilinear in Q, K)

Masked entries have P = 0 and so dS = 0.  Every bf16 input is widened
exactly to float64; P comes from the row's exact log-sum-exp.

Besides the gradients the oracle returns per-element magnitude sums, the
quantities the rounding of a bf16/fp32 kernel is bounded by:

  mag_dV[j,d] = sum_i P_ij |dO_id|
  mag_dS[i,j] = P_ij (|dP_ij| + sum_d |dO_id O_id|)
  mag_dK[j,d] = scale sum_i mag_dS[i,j] |Q_id|
  mag_dQ[i,d] = scale sum_j mag_dS[i,j] |K_jd|

(sum_d |dO_id O_id| bounds the error of computing sum_l P_il dP_il as the
row sum of dO * O from an O rounded to bf16.)
"""
from __future__ import annotations

import numpy as np

from .brute import _bf16_bits


def _widen(x) -> np.ndarray:
    bits = np.ascontiguousarray(_bf16_bits(x))
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _slice_bwd(q, k, v, do, scale, causal):
    """One (batch, head) slice, all arrays float64 [N, D]."""
    n = q.shape[0]
    s = scale * (q @ k.T)
    if causal:
        s = np.where(np.tril(np.ones((n, n), dtype=bool)), s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    p = e / e.sum(axis=1, keepdims=True)
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    row = (p * dp).sum(axis=1, keepdims=True)
    ds = p * (dp - row)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    mag_dv = p.T @ np.abs(do)
    mag_ds = p * (np.abs(dp) + (np.abs(do) * np.abs(o)).sum(axis=1, keepdims=True))
    mag_dk = scale * (mag_ds.T @ np.abs(q))
    mag_dq = scale * (mag_ds @ np.abs(k))
    return dq, dk, dv, mag_dq, mag_dk, mag_dv


def attention_bwd(q, k, v, do, scale: float, causal: bool, slices=None):
    """Gradients of [B, H, N, D] attention with respect to Q, K, V.

    q, k, v, do: bf16 (torch tensors or uint16 bit arrays) of one shape.
    slices: optional list of flat (b*H + h) indices to compute (default all).
    Returns a dict of float64 arrays [S, N, D] over the chosen slices:
    dq, dk, dv, mag_dq, mag_dk, mag_dv.
    """
    Q, K, V, dO = (_widen(t) for t in (q, k, v, do))
    if not (Q.shape == K.shape == V.shape == dO.shape) or Q.ndim != 4:
        raise ValueError("q, k, v, do must be [B, H, N, D] of one shape")
    B, H, N, D = Q.shape
    flat = [x.reshape(B * H, N, D) for x in (Q, K, V, dO)]
    idx = range(B * H) if slices is None else list(slices)
    out = {name: [] for name in ("dq", "dk", "dv", "mag_dq", "mag_dk", "mag_dv")}
    for s in idx:
        res = _slice_bwd(flat[0][s], flat[1][s], flat[2][s], flat[3][s], float(scale),
                         bool(causal))
        for name, arr in zip(("dq", "dk", "dv", "mag_dq", "mag_dk", "mag_dv"), res):
            out[name].append(arr)
    return {name: np.stack(vals) for name, vals in out.items()}
