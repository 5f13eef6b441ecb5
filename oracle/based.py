"""fp64 oracle for Based linear attention (causal or not).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name a "Based linear attention" kernel and its throughput (215
TFLOPs on H100, over 300 counting the algorithm's recompute: the Chinese news
write-up, 88811315.cn post 77732, and the Spanish page, es.news.hada.io topic
14783) but define neither its feature map nor its normalisation.  The
reading taken here is the published Based form: linear attention whose
feature map is the second-order Taylor expansion of exp,

    phi(x) = [1, x, vec(x x^T) / sqrt(2)]   so   phi(q).phi(k) = T(q.k),
    T(s) = 1 + s + s^2 / 2,

with the dot product scaled (s = scale q.k) and the output normalised by
the kernel's row sum:

    y_i = sum_{j visible} T(s_ij) v_j  /  z_i,   z_i = sum_{j visible} T(s_ij)

(visible: j <= i under the causal mask, every j otherwise).  T(s) >= 1/2 for
every real s, so z_i > 0.  `based_quadratic` evaluates this definition
directly; `based_recurrent` evaluates the same output through the explicit
feature maps and a running state sum_j phi(k_j) v_j^T, which is the linear-
time algorithm linear attention is named for, so the two pin each other.
"""
from __future__ import annotations

import numpy as np

from .brute import _bf16_bits


def _widen(x) -> np.ndarray:
    bits = np.ascontiguousarray(_bf16_bits(x))
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def taylor2(s):
    """T(s) = 1 + s + s^2 / 2."""
    return 1.0 + s + 0.5 * s * s


def based_quadratic(q, k, v, scale: float, causal: bool):
    """y [B, H, N, Dv], z [B, H, N] and the magnitude sum_j T |v_j| / z.

    q, k: bf16 [B, H, N, Df]; v: bf16 [B, H, N, Dv] (tensors or bit arrays).
    """
    Q, K, V = _widen(q), _widen(k), _widen(v)
    if Q.shape != K.shape or Q.shape[:3] != V.shape[:3] or Q.ndim != 4:
        raise ValueError("q, k must be [B, H, N, Df] and v [B, H, N, Dv]")
    n = Q.shape[2]
    a = taylor2(scale * np.einsum("bhid,bhjd->bhij", Q, K))
    if causal:
        a = np.where(np.tril(np.ones((n, n), dtype=bool)), a, 0.0)
    z = a.sum(axis=-1)
    y = np.einsum("bhij,bhjd->bhid", a, V) / z[..., None]
    mag = np.einsum("bhij,bhjd->bhid", a, np.abs(V)) / z[..., None]
    return y, z, mag


def based_rows(q, k, v, scale: float, rows):
    """Causal y, z and the magnitude sum for chosen rows only, straight from
    the definition above: row i of slice b*H + h (flat index (b*H + h)*N + i)
    sums T(scale q_i.k_j) over its keys j <= i.  Memory and time grow with N
    per row, so long sequences can be checked on a sample.
    Returns y [R, Dv], z [R], mag [R, Dv]."""
    Q, K, V = _widen(q), _widen(k), _widen(v)
    if Q.shape != K.shape or Q.shape[:3] != V.shape[:3] or Q.ndim != 4:
        raise ValueError("q, k must be [B, H, N, Df] and v [B, H, N, Dv]")
    B, H, N, Df = Q.shape
    Dv = V.shape[-1]
    Qf, Kf, Vf = Q.reshape(B * H, N, Df), K.reshape(B * H, N, Df), V.reshape(B * H, N, Dv)
    rows = np.asarray(rows, dtype=np.int64)
    y = np.empty((rows.size, Dv))
    z = np.empty(rows.size)
    mag = np.empty((rows.size, Dv))
    for r, flat in enumerate(rows):
        bh, i = divmod(int(flat), N)
        a = taylor2(scale * (Kf[bh, : i + 1] @ Qf[bh, i]))
        z[r] = a.sum()
        y[r] = (a @ Vf[bh, : i + 1]) / z[r]
        mag[r] = (a @ np.abs(Vf[bh, : i + 1])) / z[r]
    return y, z, mag


def feature_map(x, scale: float):
    """phi(sqrt(scale) x) for rows x [..., Df]: [1, x', vec(x' x'^T)/sqrt(2)]."""
    x = np.sqrt(scale) * x
    outer = np.einsum("...i,...j->...ij", x, x).reshape(*x.shape[:-1], -1) / np.sqrt(2.0)
    ones = np.ones(x.shape[:-1] + (1,))
    return np.concatenate([ones, x, outer], axis=-1)


def based_recurrent(q, k, v, scale: float):
    """Causal y and z through explicit feature maps and a running state.

    State after key j: S_j = sum_{l <= j} phi(k_l) v_l^T, s_j = sum phi(k_l);
    y_i = phi(q_i) S_i / phi(q_i) s_i.  (scale is split as sqrt(scale) on q
    and on k, so phi(q).phi(k) = T(scale q.k).)
    """
    Q, K, V = _widen(q), _widen(k), _widen(v)
    fq, fk = feature_map(Q, scale), feature_map(K, scale)
    B, H, N, _ = Q.shape
    y = np.zeros(V.shape)
    z = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            state = np.zeros((fk.shape[-1], V.shape[-1]))
            norm = np.zeros(fk.shape[-1])
            for i in range(N):
                state += np.outer(fk[b, h, i], V[b, h, i])
                norm += fk[b, h, i]
                z[b, h, i] = fq[b, h, i] @ norm
                y[b, h, i] = (fq[b, h, i] @ state) / z[b, h, i]
    return y, z
