"""bf16 GEMM C = A B^T (tk_gemm_bf16) through the C ABI against the fp64
oracle's gemm_abt, element by element.

Tolerance, from the arithmetic: every product of two bf16 values is exact in
fp32, so the kernel's result differs from the exact sum by the fp32
accumulation error, at most a small multiple of 2^-24 * sum_k |a_ik b_jk| per
add, and then by one rounding to bf16, at most 2^-9 |C_ij|.  The test allows

    |C - C_exact| <= 2^-8 |C_exact| + 2^-14 sum_k |a_ik b_jk|

(twice the rounding bound, and 2^10 fp32 units of the magnitude sum for the
accumulation), and further asks that at least 90% of the entries equal the
exact sum rounded once to bf16: any dropped or repeated K block, transposed
operand or misplaced tile is off by far more than either allows.
"""
import numpy as np
import pytest
import torch

from attention_forward_tk_gb300.inputs import GEMM_BY_NAME, draw_gemm

pytestmark = pytest.mark.gpu


def run_gemm(tk_lib, a, b, fill=float("nan")):
    dev = torch.device("cuda", 0)
    M, K = a.shape
    N = b.shape[0]
    ad, bd = a.to(dev), b.to(dev)
    c = torch.full((M, N), fill, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = tk_lib.tk_gemm_bf16(ad.data_ptr(), bd.data_ptr(), c.data_ptr(), M, N, K, stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    torch.cuda.synchronize()
    return c.cpu()


def check(c, exact, mag, min_match=0.9):
    got = c.double().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - exact)
    tol = 2.0 ** -8 * np.abs(exact) + 2.0 ** -14 * mag
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert (err <= tol).all(), (
        f"entry {worst}: got {got[worst]}, exact {exact[worst]}, tol {tol[worst]}")
    rounded = torch.from_numpy(exact).to(torch.bfloat16).double().numpy()
    match = float((got == rounded).mean())
    assert match >= min_match, f"only {match:.3f} of the entries equal round_bf16(exact)"


CASES = [
    # (M, N, K)
    (128, 256, 64),     # one tile, one K block
    (1, 8, 8),          # one row, one 16-byte column group, K below one block
    (300, 520, 200),    # ragged M, N and K tails
    (1000, 1000, 1000),
    (4096, 4096, 256),  # 512 tiles: several per CTA, both accumulators, ring wrap-around
    (256, 512, 8192),   # 128 K blocks through the 4-stage ring
    (130, 264, 72),     # tails of one row, 8 columns and 8 K-columns past full tiles
    (2048, 2048, 512),  # 64 tiles: one wave more than half full, no tile split into halves
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_gemm_parity(tk_lib, oracle_lib, case):
    M, N, K = case
    a, b = draw_gemm(M, N, K, seed=700 + M + N + K)
    exact, mag = oracle_lib.gemm_abt(a, b)
    check(run_gemm(tk_lib, a, b), exact, mag)


def test_gemm_structured(tk_lib, oracle_lib):
    """A = I picks columns of B^T: C = B^T exactly (one nonzero product per
    entry, so no rounding anywhere)."""
    K = 192
    a = torch.eye(K, dtype=torch.bfloat16)
    _, b = draw_gemm(8, 264, K, seed=31)
    c = run_gemm(tk_lib, a, b)
    assert torch.equal(c, b.t().contiguous())


def test_gemm_empty(tk_lib):
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream().cuda_stream
    # K = 0: empty sums, C = 0 (the empty operands still need non-null bases)
    c = torch.full((64, 40), float("nan"), dtype=torch.bfloat16, device=dev)
    pa = torch.empty(16, dtype=torch.bfloat16, device=dev)
    st = tk_lib.tk_gemm_bf16(pa.data_ptr(), pa.data_ptr(), c.data_ptr(), 64, 40, 0, stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(c.cpu(), torch.zeros(64, 40, dtype=torch.bfloat16))
    # M = 0 (or N = 0): nothing is written
    c2 = torch.full((8, 8), 7.0, dtype=torch.bfloat16, device=dev)
    a2 = torch.randn(8, 64, device=dev).to(torch.bfloat16)
    st = tk_lib.tk_gemm_bf16(a2.data_ptr(), a2.data_ptr(), c2.data_ptr(), 0, 8, 64, stream)
    assert st == 0
    torch.cuda.synchronize()
    assert (c2 == 7.0).all()


def test_gemm_rejects(tk_lib):
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream().cuda_stream
    a = torch.zeros(64, 64, dtype=torch.bfloat16, device=dev)
    c = torch.full((64, 64), 3.0, dtype=torch.bfloat16, device=dev)
    # N not a multiple of 8, K not a multiple of 8, misaligned base, overlap
    assert tk_lib.tk_gemm_bf16(a.data_ptr(), a.data_ptr(), c.data_ptr(), 64, 60, 64, stream) == -2
    assert tk_lib.tk_gemm_bf16(a.data_ptr(), a.data_ptr(), c.data_ptr(), 64, 64, 60, stream) == -2
    assert tk_lib.tk_gemm_bf16(a.data_ptr() + 2, a.data_ptr(), c.data_ptr(), 8, 8, 8,
                               stream) == -2
    assert tk_lib.tk_gemm_bf16(a.data_ptr(), a.data_ptr(), a.data_ptr(), 64, 64, 64,
                               stream) == -1
    torch.cuda.synchronize()
    assert (c == 3.0).all()


def test_gemm_full_size_sampled(tk_lib, oracle_lib):
    """The 8192^3 product (the size the cuBLAS peak is measured on), in the
    launch the benchmark times, checked on 48 sampled rows in full."""
    w = GEMM_BY_NAME["gemm_8192"]
    a, b = draw_gemm(w.M, w.N, w.K, w.seed)
    c = run_gemm(tk_lib, a, b)
    rows = np.random.default_rng(5).choice(w.M, size=48, replace=False)
    rows[:2] = (0, w.M - 1)
    exact, mag = oracle_lib.gemm_abt(a[rows], b)
    check(c[rows], exact, mag)
