"""Tile-by-tile online-softmax attention in float64 (numpy).

TEST INFRASTRUCTURE ONLY (see the package docstring).

This restates the recurrence that the kernel examples in the ThunderKittens
news write-up (88811315.cn, post 77732) run over K/V tiles -- the "RTX 4090
flash attention" example and the "H100 FlashAttention-2 forward" example --
for one (batch, head) slice held as float64 arrays:

  per query block, keep a running row max m, a running normaliser l and an
  output accumulator; for each key block compute the scaled scores S, raise
  the running max to include rowmax(S), exponentiate S against the new max,
  shrink the old normaliser by exp(m_old - m_new) and add the new row sums.

Two ways of carrying the output are offered:

  mode="renormalize"  the pages' form: after each key block the weights are
                      divided by the updated normaliser, and the old output is
                      first multiplied by l_old * exp(m_old - m_new) / l_new,
                      so the output is a normalised average at every step;
  mode="deferred"     the output accumulates unnormalised weights times V,
                      rescaled by exp(m_old - m_new) per block, and is divided
                      by l once at the end.

Both return the log-sum-exp m + ln(l) of the scaled (masked) scores.  Tile
sizes are arguments so tests can use sizes that do not divide N.  Under the
causal mask (key j visible to query i iff j <= i) key blocks that start after
the last query of a block are skipped, as a causal kernel would.
"""
from __future__ import annotations

import numpy as np


def tiled_online_softmax(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                         scale: float, causal: bool, block_q: int,
                         block_k: int, mode: str = "deferred"):
    """q, k, v: float64 [N, D].  Returns (o [N, D], lse [N])."""
    if mode not in ("deferred", "renormalize"):
        raise ValueError("mode must be 'deferred' or 'renormalize'")
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    o = np.zeros((n, d))
    lse = np.zeros(n)
    for r0 in range(0, n, block_q):
        r1 = min(n, r0 + block_q)
        qi = q[r0:r1]
        rows = np.arange(r0, r1)
        m = np.full(r1 - r0, -np.inf)
        l = np.zeros(r1 - r0)
        acc = np.zeros((r1 - r0, d))
        for c0 in range(0, n, block_k):
            if causal and c0 > r1 - 1:
                break  # every key of this block is in the future of every query
            c1 = min(n, c0 + block_k)
            s = scale * (qi @ k[c0:c1].T)
            if causal:
                cols = np.arange(c0, c1)
                s = np.where(cols[None, :] > rows[:, None], -np.inf, s)
            m_new = np.maximum(m, s.max(axis=1))
            # m_new is finite: key 0 is visible to every query and lies in the
            # first key block, which is never skipped.
            p = np.exp(s - m_new[:, None])
            alpha = np.exp(m - m_new)
            if mode == "deferred":
                l = alpha * l + p.sum(axis=1)
                acc = alpha[:, None] * acc + p @ v[c0:c1]
            else:
                l_old = l
                l = alpha * l_old + p.sum(axis=1)
                p = p / l[:, None]
                keep = (l_old * alpha) / l
                acc = keep[:, None] * acc + p @ v[c0:c1]
            m = m_new
        o[r0:r1] = acc / l[:, None] if mode == "deferred" else acc
        lse[r0:r1] = m + np.log(l)
    return o, lse
