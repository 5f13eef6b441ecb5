"""Based linear attention (tk_based_fwd) through the C ABI against the fp64
oracle's based_quadratic, element by element.

Tolerance, from the arithmetic: the kernel forms T(s) in fp32 from an fp32
score, rounds it to bf16 as the A operand of T V (2^-9 relative per term),
sums z from the unrounded fp32 T, and rounds y to bf16 once.  So

    |y - y_exact| <= 2^-7 mag + 2^-8 |y_exact|,   mag = sum_j T |v_j| / z,
    |z - z_exact| <= 2^-12 z_exact  (fp32 sums of up to N positive terms),

and the relative RMS error of y must stay below 2^-6.
"""

import numpy as np
import pytest
import torch

from attention_forward_tk_gb300.inputs import BASED_BY_NAME, draw_based

pytestmark = pytest.mark.gpu


def run_based(tk_lib, q, k, v, scale, causal):
    dev = torch.device("cuda", 0)
    B, H, N, Df = q.shape
    Dv = v.shape[3]
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    y = torch.full((B, H, N, Dv), float("nan"), dtype=torch.bfloat16, device=dev)
    z = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = tk_lib.tk_based_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), y.data_ptr(),
                             z.data_ptr(), B, H, N, Df, Dv, scale, int(causal), stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    torch.cuda.synchronize()
    return y.float().cpu().double().numpy(), z.cpu().double().numpy()


def check(got_y, got_z, ref_y, ref_z, mag):
    assert np.isfinite(got_y).all() and np.isfinite(got_z).all()
    err = np.abs(got_y - ref_y)
    tol = 2.0 ** -7 * mag + 2.0 ** -8 * np.abs(ref_y)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert (err <= tol).all(), f"y {worst}: got {got_y[worst]}, exact {ref_y[worst]}"
    assert (np.abs(got_z - ref_z) <= 2.0 ** -12 * ref_z).all()
    rel = np.sqrt((err ** 2).sum() / (ref_y ** 2).sum())
    assert rel <= 2.0 ** -6, f"relative RMS error {rel:.3e}"


CASES = [
    # (B, H, N, causal, scale)
    (1, 1, 128, False, 0.25),
    (1, 2, 256, True, 0.25),
    (2, 1, 200, True, 0.25),    # ragged tail
    (2, 1, 200, False, 0.25),
    (1, 1, 1, True, 0.25),      # one key: y = v
    (4, 10, 512, False, 0.25),  # 160 units: several per CTA
    (2, 20, 512, True, 0.25),
    (2, 2, 1000, True, 1.0),    # larger scores (s up to ~16)
    (1, 3, 129, True, -0.5),    # negative scale: T still >= 1/2
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_based_parity(tk_lib, oracle_lib, case):
    B, H, N, causal, scale = case
    q, k, v = draw_based(B, H, N, seed=1100 + N + B + H)
    y, z = run_based(tk_lib, q, k, v, scale, causal)
    ry, rz, mag = oracle_lib.based_quadratic(q, k, v, scale, causal)
    check(y, z, ry, rz, mag)


def test_based_rejects_other_widths(tk_lib):
    dev = torch.device("cuda", 0)
    t = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device=dev)
    y = torch.full((1, 1, 128, 64), 2.0, dtype=torch.bfloat16, device=dev)
    z = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    st = tk_lib.tk_based_fwd(t.data_ptr(), t.data_ptr(), t.data_ptr(), y.data_ptr(),
                             z.data_ptr(), 1, 1, 128, 32, 64, 0.25, 1,
                             torch.cuda.current_stream().cuda_stream)
    assert st == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (y == 2.0).all()


def test_based_full_size_sampled_slices(tk_lib, oracle_lib):
    """based_n4096_c (B16 H16 N4096, causal), the whole launch on the GPU, two
    (batch, head) slices checked in full."""
    w = BASED_BY_NAME["based_n4096_c"]
    q, k, v = draw_based(w.B, w.H, w.N, w.seed)
    y, z = run_based(tk_lib, q, k, v, w.scale, w.causal)
    for s in (0, w.B * w.H - 1):
        b, h = divmod(s, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        ry, rz, mag = oracle_lib.based_quadratic(q[sl], k[sl], v[sl], w.scale, w.causal)
        check(y[sl], z[sl], ry, rz, mag)


# ---------------------------------------------------------------- linear-time form

def run_based_linear(tk_lib, q, k, v, scale):
    dev = torch.device("cuda", 0)
    B, H, N, Df = q.shape
    Dv = v.shape[3]
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    y = torch.full((B, H, N, Dv), float("nan"), dtype=torch.bfloat16, device=dev)
    z = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = tk_lib.tk_based_fwd_linear(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), y.data_ptr(),
                                    z.data_ptr(), B, H, N, Df, Dv, scale, stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    torch.cuda.synchronize()
    return y.float().cpu().double().numpy(), z.cpu().double().numpy()


def check_linear(got_y, got_z, ref_y, ref_z, mag):
    """tk_based_fwd_linear takes bf16 operands in every product: T inside a
    chunk (as the direct kernel), the feature maps phi(q), phi(k) and the
    bf16 copy of the fp32 state.  Each rounding is 2^-9 relative and
    independent of the others; the numerator and z share phi(q), phi(k) and
    T, and differ only in the state copy's rounding of their own rows.  So y
    keeps the direct kernel's bound (2^-7 mag + 2^-8 |y|), and z, a sum of
    bf16 products, is held to 2^-7 relative."""
    assert np.isfinite(got_y).all() and np.isfinite(got_z).all()
    err = np.abs(got_y - ref_y)
    tol = 2.0 ** -7 * mag + 2.0 ** -8 * np.abs(ref_y)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert (err <= tol).all(), f"y {worst}: got {got_y[worst]}, exact {ref_y[worst]}"
    zerr = np.abs(got_z - ref_z) / ref_z
    assert zerr.max() <= 2.0 ** -7, f"z relative error {zerr.max():.3e}"
    rel = np.sqrt((err ** 2).sum() / (ref_y ** 2).sum())
    assert rel <= 2.0 ** -6, f"relative RMS error {rel:.3e}"


LIN_CASES = [
    # (B, H, N, scale): always causal
    (1, 1, 1, 0.25),      # one position: y = v
    (1, 2, 128, 0.25),    # one chunk: no state
    (1, 2, 129, 0.25),    # a second chunk of one position
    (2, 1, 200, 0.25),    # ragged tail
    (1, 2, 256, 0.25),
    (2, 2, 1000, 1.0),    # larger scores (s up to ~16)
    (1, 2, 2048, 0.25),   # 16 chunks through the state
    (4, 40, 300, 0.25),   # 160 slices: two on some CTAs
    (1, 1, 640, 0.0),     # scale 0: T = 1, y is the running mean of v
]


@pytest.mark.parametrize("case", LIN_CASES, ids=lambda c: "x".join(map(str, c)))
def test_based_linear_parity(tk_lib, oracle_lib, case):
    B, H, N, scale = case
    q, k, v = draw_based(B, H, N, seed=1300 + N + B + H)
    y, z = run_based_linear(tk_lib, q, k, v, scale)
    ry, rz, mag = oracle_lib.based_quadratic(q, k, v, scale, True)
    check_linear(y, z, ry, rz, mag)


def test_based_linear_rejects_negative_scale(tk_lib):
    dev = torch.device("cuda", 0)
    q = torch.zeros((1, 1, 128, 16), dtype=torch.bfloat16, device=dev)
    v = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device=dev)
    y = torch.full((1, 1, 128, 64), 2.0, dtype=torch.bfloat16, device=dev)
    z = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    st = tk_lib.tk_based_fwd_linear(q.data_ptr(), q.data_ptr(), v.data_ptr(), y.data_ptr(),
                                    z.data_ptr(), 1, 1, 128, 16, 64, -0.25,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == tk_lib.TK_ATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (y == 2.0).all()


def test_based_linear_full_size_sampled_slices(tk_lib, oracle_lib):
    """based_n4096_c through the linear-time kernel: the whole launch on the
    GPU, two slices checked in full against the oracle, and every slice
    against the direct kernel (both within their bounds of the exact y)."""
    w = BASED_BY_NAME["based_n4096_c"]
    q, k, v = draw_based(w.B, w.H, w.N, w.seed)
    y, z = run_based_linear(tk_lib, q, k, v, w.scale)
    for s in (0, w.B * w.H - 1):
        b, h = divmod(s, w.H)
        sl = (slice(b, b + 1), slice(h, h + 1))
        ry, rz, mag = oracle_lib.based_quadratic(q[sl], k[sl], v[sl], w.scale, w.causal)
        check_linear(y[sl], z[sl], ry, rz, mag)
    yd, zd = run_based(tk_lib, q, k, v, w.scale, True)
    assert np.abs(y - yd).max() <= 2.0 ** -5
    assert (np.abs(z - zd) <= 2.0 ** -6 * zd).all()


def _long_rows(BH, N, seed):
    """Chunk and tile edges, the middle, the last rows and 30 random rows of
    every slice, as flat indices (b*H + h)*N + i."""
    rng = np.random.default_rng(seed)
    per = {0, 1, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1}
    rows = []
    for bh in range(BH):
        idx = sorted(per | set(rng.integers(0, N, 30).tolist()))
        rows.extend(bh * N + i for i in idx)
    return np.asarray(rows, dtype=np.int64)


@pytest.mark.parametrize("N", [65536, 65536 + 77])
def test_based_long_sequence_sampled_rows(tk_lib, oracle_lib, N):
    """Sequences 16x the timed one (512 chunks through the linear-time
    kernel's running state; rows of 512 key tiles in the direct kernel), both
    kernels, causal, on sampled rows against the oracle's per-row evaluation
    of the definition."""
    B, H, scale = 1, 4, 0.25
    q, k, v = draw_based(B, H, N, seed=1500 + N)
    rows = _long_rows(B * H, N, seed=N)
    ry, rz, mag = oracle_lib.based_rows(q, k, v, scale, rows)
    yl, zl = run_based_linear(tk_lib, q, k, v, scale)
    check_linear(yl.reshape(-1, 64)[rows], zl.reshape(-1)[rows], ry, rz, mag)
    yd, zd = run_based(tk_lib, q, k, v, scale, True)
    check(yd.reshape(-1, 64)[rows], zd.reshape(-1)[rows], ry, rz, mag)
