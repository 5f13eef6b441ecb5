"""The backward pass (tk_attn_bwd) through the C ABI against the fp64
oracle's attention_bwd, element by element.  The forward runs first on the
GPU (tk_attn_fwd), as in training, and its O and LSE feed the backward.

Tolerance, from the arithmetic: the kernel rounds P and dS to bf16 for the
gradient products (2^-9 relative each), forms delta = rowsum(dO * O) from the
bf16 O (error <= 2^-9 sum_d |dO O| plus fp32 rounding), and rounds each
gradient to bf16 once.  Every one of these errors is bounded by 2^-9 times
the oracle's magnitude sum for that element, so

    |g - g_exact| <= 2^-7 mag_g + 2^-8 |g_exact|

holds for correct code with room to spare; and since rounding errors add in
quadrature, the relative RMS error of each gradient tensor must stay below
2^-6, which a dropped tile, a wrong sign or a transposed operand exceeds by
far.
"""
import math

import numpy as np
import pytest
import torch

from attention_forward_tk_gb300.inputs import draw, draw_grad

pytestmark = pytest.mark.gpu


def run_fwd_bwd(tk_lib, q, k, v, do, scale, causal):
    dev = torch.device("cuda", 0)
    B, H, N, D = q.shape
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = tk_lib.tk_attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, N, D, scale, int(causal), stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    grads = [torch.full_like(qd, float("nan")) for _ in range(3)]
    need = tk_lib.tk_attn_bwd_workspace_bytes(B, H, N, D)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    st = tk_lib.tk_attn_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), dod.data_ptr(), grads[0].data_ptr(),
                            grads[1].data_ptr(), grads[2].data_ptr(), B, H, N, D, scale,
                            int(causal), ws.data_ptr(), need, stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    torch.cuda.synchronize()
    return [g.float().cpu().double().numpy().reshape(B * H, N, D) for g in grads]


def check(got, ref, slices=None):
    for name, g in zip(("dq", "dk", "dv"), got):
        if slices is not None:
            g = g[slices]
        exact, mag = ref[name], ref["mag_" + name]
        assert np.isfinite(g).all(), name
        err = np.abs(g - exact)
        tol = 2.0 ** -7 * mag + 2.0 ** -8 * np.abs(exact) + 1e-30
        worst = np.unravel_index(np.argmax(err - tol), err.shape)
        assert (err <= tol).all(), (
            f"{name} {worst}: got {g[worst]}, exact {exact[worst]}, tol {tol[worst]}")
        norm = np.sqrt((exact ** 2).sum())
        if norm > 0:
            rel = np.sqrt((err ** 2).sum()) / norm
            assert rel <= 2.0 ** -6, f"{name}: relative RMS error {rel:.3e}"


CASES = [
    # (B, H, N, D, causal)
    (1, 1, 128, 64, False),
    (1, 1, 128, 128, True),
    (1, 2, 256, 64, True),
    (2, 1, 200, 128, False),   # ragged tail
    (2, 1, 200, 64, True),
    (1, 3, 300, 128, True),
    (1, 1, 1, 64, False),      # one key: dV = dO, dQ = dK = 0 up to rounding
    (1, 1, 1, 128, True),
    (4, 10, 512, 64, False),   # 160 units: several per CTA
    (2, 20, 512, 128, True),   # 160 units, causal
    (1, 1, 1000, 128, True),
    (2, 2, 129, 64, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_bwd_parity(tk_lib, oracle_lib, case):
    B, H, N, D, causal = case
    seed = 900 + N + D + B * 7 + H
    q, k, v = draw((B, H, N, D), seed)
    do = draw_grad((B, H, N, D), seed)
    scale = 1.0 / math.sqrt(D)
    got = run_fwd_bwd(tk_lib, q, k, v, do, scale, causal)
    check(got, oracle_lib.attention_bwd(q, k, v, do, scale, causal))


def test_bwd_peaky_inputs(tk_lib, oracle_lib):
    # large scores (4 N(0,1) queries and keys): P is nearly one-hot per row
    q, k, v = draw((1, 2, 384, 128), 77, dist="peaky_t3")
    do = draw_grad((1, 2, 384, 128), 77)
    got = run_fwd_bwd(tk_lib, q, k, v, do, 0.3, True)
    check(got, oracle_lib.attention_bwd(q, k, v, do, 0.3, True))


def test_bwd_rejects_short_workspace(tk_lib):
    dev = torch.device("cuda", 0)
    t = [torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device=dev) for _ in range(8)]
    lse = torch.zeros((1, 1, 256), dtype=torch.float32, device=dev)
    need = tk_lib.tk_attn_bwd_workspace_bytes(1, 1, 256, 64)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    t[5].fill_(3.0)
    st = tk_lib.tk_attn_bwd(t[0].data_ptr(), t[1].data_ptr(), t[2].data_ptr(), t[3].data_ptr(),
                            lse.data_ptr(), t[4].data_ptr(), t[5].data_ptr(), t[6].data_ptr(),
                            t[7].data_ptr(), 1, 1, 256, 64, 0.125, 0, ws.data_ptr(), need - 4,
                            torch.cuda.current_stream().cuda_stream)
    assert st == tk_lib.TK_ATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (t[5] == 3.0).all()


@pytest.mark.parametrize("shape", [(16, 16, 4096, False), (8, 16, 4096, True),
                                   (8, 16, 8192, True)],
                         ids=["n4096", "n4096_causal", "n8192_causal"])
def test_bwd_full_size_sampled_slices(tk_lib, oracle_lib, shape):
    """The timed backward shapes (B16 H16 N4096 D128, and B8 H16 N8192 D128
    causal) and a causal N4096 one, the whole launch on the GPU, four (batch,
    head) slices spread over the launch checked in full."""
    B, H, N, causal = shape
    D = 128
    q, k, v = draw((B, H, N, D), 2)
    do = draw_grad((B, H, N, D), 2)
    scale = 1.0 / math.sqrt(D)
    got = run_fwd_bwd(tk_lib, q, k, v, do, scale, causal)
    slices = [0, B * H // 3, 2 * B * H // 3 + 1, B * H - 1]
    check(got, oracle_lib.attention_bwd(q, k, v, do, scale, causal, slices=slices), slices)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_autograd_attention(tk_lib, oracle_lib, causal):
    """attention() under torch autograd: the forward kernel, then the
    backward kernels on the saved O and LSE, give the oracle's gradients of
    sum(O * dO)."""
    from attention_forward_tk_gb300 import attention
    B, H, N, D = 2, 2, 300, 64
    q, k, v = draw((B, H, N, D), 21 + int(causal))
    do = draw_grad((B, H, N, D), 21)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (t.to(dev).requires_grad_() for t in (q, k, v))
    o = attention(qd, kd, vd, causal=causal)
    (o.float() * do.to(dev).float()).sum().backward()
    torch.cuda.synchronize()
    got = [t.grad.float().cpu().double().numpy().reshape(B * H, N, D) for t in (qd, kd, vd)]
    check(got, oracle_lib.attention_bwd(q, k, v, do, 1.0 / math.sqrt(D), causal))


def test_bwd_causal_beyond_the_unit_lists(tk_lib, oracle_lib):
    """More causal units (B2 H100 N8192: 200 slices x 64 tiles = 12,800) than
    the per-CTA unit lists hold: the kernels fall back to the stride order.
    Two slices checked in full."""
    B, H, N, D = 2, 100, 8192, 64
    q, k, v = draw((B, H, N, D), 5)
    do = draw_grad((B, H, N, D), 5)
    scale = 1.0 / math.sqrt(D)
    got = run_fwd_bwd(tk_lib, q, k, v, do, scale, True)
    slices = [7, B * H - 1]
    check(got, oracle_lib.attention_bwd(q, k, v, do, scale, True, slices=slices), slices)
