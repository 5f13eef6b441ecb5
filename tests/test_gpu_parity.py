"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small shapes that span several 128-row tiles and ragged tails, both masks,
both head dims; every output element is compared.  Tolerances (bf16 inputs,
fp32 accumulation, bf16 output): max |dO| <= 2e-2, mean |dO| <= 2e-3,
max |dLSE| <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

from attention_forward_tk_gb300.inputs import draw
from conftest import TOL_LSE_MAX, TOL_O_MAX, TOL_O_MEAN

pytestmark = pytest.mark.gpu


def run_gpu(tk_lib, q, k, v, scale, causal):
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    B, H, N, D = q.shape
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    st = tk_lib.tk_attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, N, D, scale, int(causal),
                            torch.cuda.current_stream().cuda_stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    assert tk_lib.tk_attn_last_device_error(torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def compare(o, lse, o_ref, lse_ref, tag=""):
    assert np.isfinite(o).all(), f"{tag}: non-finite O"
    assert np.isfinite(lse).all(), f"{tag}: non-finite LSE"
    do = np.abs(o - o_ref)
    dl = np.abs(lse - lse_ref)
    assert do.max() <= TOL_O_MAX, f"{tag}: max|dO| {do.max():.3e}"
    assert do.mean() <= TOL_O_MEAN, f"{tag}: mean|dO| {do.mean():.3e}"
    assert dl.max() <= TOL_LSE_MAX, f"{tag}: max|dLSE| {dl.max():.3e}"
    return do.max(), do.mean(), dl.max()


SHAPES = [
    # (B, H, N, D)
    (1, 1, 256, 64),     # the smallest measured workload, exactly
    (1, 1, 256, 128),
    (2, 3, 1000, 64),    # ragged tail, several units
    (1, 2, 1000, 128),
    (1, 1, 1, 64),       # one key
    (1, 1, 1, 128),
    (1, 1, 2, 128),
    (3, 1, 17, 64),
    (1, 1, 127, 128),
    (1, 1, 128, 64),
    (1, 1, 129, 128),
    (1, 1, 255, 64),
    (1, 1, 257, 128),
    (2, 2, 640, 128),    # 2.5 units per head
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_parity_small(tk_lib, oracle_lib, shape, causal):
    B, H, N, D = shape
    seed = 1000 + N * 7 + D + B * 3 + H + int(causal)
    q, k, v = draw(shape, seed=seed)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(tk_lib, q, k, v, scale, causal)
    o_ref, lse_ref = oracle_lib.attention(q, k, v, scale, causal)
    compare(o, lse, o_ref, lse_ref, f"{shape} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_parity_peaky_values(tk_lib, oracle_lib, causal):
    # Q, K = 4 N(0,1) and V = Student-t(3) clipped to +-8: peaky softmax with
    # frequent running-max jumps, the stress distribution of the longest workload.
    shape = (1, 2, 1536, 128)
    q, k, v = draw(shape, seed=77, dist="peaky_t3")
    scale = 1.0 / math.sqrt(128)
    o, lse = run_gpu(tk_lib, q, k, v, scale, causal)
    o_ref, lse_ref = oracle_lib.attention(q, k, v, scale, causal)
    compare(o, lse, o_ref, lse_ref, f"peaky causal={causal}")


@pytest.mark.parametrize("scale", [0.01, 0.3, 1.7])
def test_parity_non_default_scale(tk_lib, oracle_lib, scale):
    shape = (1, 1, 384, 64)
    q, k, v = draw(shape, seed=31)
    o, lse = run_gpu(tk_lib, q, k, v, scale, False)
    o_ref, lse_ref = oracle_lib.attention(q, k, v, scale, False)
    compare(o, lse, o_ref, lse_ref, f"scale={scale}")


def test_many_heads_more_units_than_sms(tk_lib, oracle_lib):
    # 2 * 160 * 1 = 320 units > 152 SMs: every CTA runs two or three units
    shape = (2, 160, 200, 64)
    q, k, v = draw(shape, seed=41)
    scale = 0.125
    for causal in (False, True):
        o, lse = run_gpu(tk_lib, q, k, v, scale, causal)
        o_ref, lse_ref = oracle_lib.attention(q, k, v, scale, causal)
        compare(o, lse, o_ref, lse_ref, f"many heads causal={causal}")


def test_outputs_beyond_n_untouched(tk_lib):
    # rows past N are never written: pad a buffer and check the pad survives
    dev = torch.device("cuda", 0)
    B, H, N, D = 1, 1, 200, 64
    q, k, v = draw((B, H, N, D), seed=5)
    big_o = torch.full((B * H * N * D + 4096,), 7.0, dtype=torch.bfloat16, device=dev)
    big_l = torch.full((B * H * N + 1024,), 7.0, dtype=torch.float32, device=dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    st = tk_lib.tk_attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), big_o.data_ptr(),
                            big_l.data_ptr(), B, H, N, D, 0.125, 1,
                            torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.all(big_o[B * H * N * D:] == 7.0)
    assert torch.all(big_l[B * H * N:] == 7.0)


def test_errors_leave_outputs_untouched(tk_lib):
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in draw((1, 1, 64, 64), seed=6))
    o = torch.full_like(q, 3.0)
    lse = torch.full((1, 1, 64), 3.0, device=dev)
    st = tk_lib.tk_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), 1, 1, 64, 96, 0.125, 0, 0)
    assert st == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(o == 3.0) and torch.all(lse == 3.0)


def test_torch_wrapper_matches_raw_call(tk_lib, oracle_lib):
    from attention_forward_tk_gb300 import attention_forward
    q, k, v = draw((1, 2, 300, 128), seed=8)
    dev = torch.device("cuda", 0)
    o, lse = attention_forward(q.to(dev), k.to(dev), v.to(dev), causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_lib.attention(q, k, v, 1 / math.sqrt(128), True)
    compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, "wrapper")


def test_host_buffer_path_matches(tk_lib, oracle_lib):
    from attention_forward_tk_gb300 import attention_forward_host
    q, k, v = draw((2, 2, 512, 64), seed=9)
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = attention_forward_host(q, k, v, causal=False)
    o_ref, lse_ref = oracle_lib.attention(q, k, v, 0.125, False)
    compare(o.float().double().numpy(), lse.double().numpy(), o_ref, lse_ref, "host path")


def test_host_buffer_pieces_match_one_piece(tk_lib):
    # the pipelined pieces of the batch give exactly the single-call result
    from attention_forward_tk_gb300 import attention_forward_host
    q, k, v = draw((5, 2, 384, 128), seed=10)
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o1, l1 = attention_forward_host(q, k, v, causal=True, chunks=1)
    o1, l1 = o1.clone(), l1.clone()
    o4, l4 = attention_forward_host(q, k, v, causal=True, chunks=4)
    assert torch.equal(o1, o4) and torch.equal(l1, l4)
    o1, l1 = o1.clone(), l1.clone()
    o7, l7 = attention_forward_host(q, k, v, causal=True, chunks=7)  # pieces cut inside batch entries
    assert torch.equal(o1, o7) and torch.equal(l1, l7)


@pytest.mark.parametrize("N", [301, 302])
def test_host_call_odd_lengths_equal_the_device_call(tk_lib, N):
    # LSE rows of an odd (or 2 mod 4) length start 16-byte aligned only every
    # 4 (or 2) slices: the pieces are cut there; the result is the device
    # call's, bit for bit, for every piece count
    from attention_forward_tk_gb300 import attention_forward, attention_forward_host
    q, k, v = draw((3, 3, N, 64), seed=12)
    dev = torch.device("cuda", 0)
    od, ld = attention_forward(q.to(dev), k.to(dev), v.to(dev), causal=True)
    torch.cuda.synchronize()
    od, ld = od.cpu(), ld.cpu()
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    for pieces in (1, 2, 3, 5, 9):
        o, l = attention_forward_host(q, k, v, causal=True, chunks=pieces)
        assert torch.equal(o, od) and torch.equal(l, ld), pieces


def test_host_call_pageable_buffers_and_a_side_stream(tk_lib, oracle_lib):
    # plain (pageable) host tensors through the raw C call on a non-default
    # stream: the outputs are valid once that stream is synchronised
    from attention_forward_tk_gb300.api import tk_attn_fwd_host_workspace_bytes
    B, H, N, D = 2, 3, 260, 128
    q, k, v = draw((B, H, N, D), seed=13)
    o = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32)
    dev = torch.device("cuda", 0)
    ws = torch.empty(tk_attn_fwd_host_workspace_bytes(B, H, N, D), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)
    st = tk_lib.tk_attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, N, D, 1 / math.sqrt(D), 0, 2,
                                 ws.data_ptr(), ws.numel(), s.cuda_stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    s.synchronize()
    assert tk_lib.tk_attn_last_device_error(s.cuda_stream) == 0
    o_ref, lse_ref = oracle_lib.attention(q, k, v, 1 / math.sqrt(D), False)
    compare(o.float().double().numpy(), lse.double().numpy(), o_ref, lse_ref, "pageable host call")


def test_host_call_from_two_threads(tk_lib):
    # two host threads, each with its own buffers, workspace and stream, call
    # the host-buffer entry point at once: the per-device copy streams and
    # events are shared, and each result is the device call's
    import threading

    from attention_forward_tk_gb300 import attention_forward
    from attention_forward_tk_gb300.api import tk_attn_fwd_host_workspace_bytes
    dev = torch.device("cuda", 0)
    B, H, N, D = 2, 4, 640, 128
    inputs = [draw((B, H, N, D), seed=30 + t) for t in range(2)]
    expect = []
    for q, k, v in inputs:
        o, l = attention_forward(q.to(dev), k.to(dev), v.to(dev), causal=True)
        torch.cuda.synchronize()
        expect.append((o.cpu(), l.cpu()))
    results, errors = [None, None], []

    def worker(t):
        try:
            q, k, v = (x.pin_memory() for x in inputs[t])
            o = torch.empty((B, H, N, D), dtype=torch.bfloat16, pin_memory=True)
            l = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
            ws = torch.empty(tk_attn_fwd_host_workspace_bytes(B, H, N, D), dtype=torch.uint8,
                             device=dev)
            s = torch.cuda.Stream(dev)
            for _ in range(5):
                st = tk_lib.tk_attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             o.data_ptr(), l.data_ptr(), B, H, N, D,
                                             1 / math.sqrt(D), 1, 3, ws.data_ptr(), ws.numel(),
                                             s.cuda_stream)
                assert st == 0, st
            s.synchronize()
            results[t] = (o.clone(), l.clone())
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t in range(2):
        assert torch.equal(results[t][0], expect[t][0]) and torch.equal(results[t][1], expect[t][1])
