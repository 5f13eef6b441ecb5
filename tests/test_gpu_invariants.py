"""Properties the definition fixes, checked on the CUDA path (through the C ABI),
plus the paths of the kernel that only unusual inputs reach: V values beyond
the fp16 range (per-tile power-of-two scaling of V), many short causal units
per CTA, and the device-side timeout status."""
import math

import numpy as np
import pytest
import torch

from attention_forward_tk_gb300.inputs import draw
from conftest import TOL_LSE_MAX, TOL_O_MAX, TOL_O_MEAN

pytestmark = pytest.mark.gpu


def run_gpu(tk_lib, q, k, v, scale, causal):
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev).contiguous(), k.to(dev).contiguous(), v.to(dev).contiguous()
    B, H, N, D = q.shape
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = tk_lib.tk_attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), B, H, N, D, scale, int(causal), stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def bf(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_constant_v_gives_constant_o(tk_lib, causal, D):
    q, k, v = draw((1, 2, 777, D), seed=201 + D)
    row = v[0, 0, 5].clone()
    vc = row.expand_as(v).contiguous()
    o, _ = run_gpu(tk_lib, q, k, vc, 1 / math.sqrt(D), causal)
    ref = np.broadcast_to(row.double().numpy(), o.shape)
    # the result is a bf16 rounding of the exact value v
    assert np.abs(o - ref).max() <= np.abs(ref).max() * 2 ** -8


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_is_uniform(tk_lib, causal):
    _, k, v = draw((1, 1, 600, 128), seed=202)
    q = torch.zeros_like(k)
    o, lse = run_gpu(tk_lib, q, k, v, 0.088, causal)
    vd = v.double().numpy()
    n = 600
    if causal:
        ref = np.cumsum(vd, axis=2) / np.arange(1, n + 1)[None, None, :, None]
        ref_lse = np.log(np.arange(1, n + 1))[None, None, :]
    else:
        ref = np.broadcast_to(vd.mean(axis=2, keepdims=True), vd.shape)
        ref_lse = np.full((1, 1, n), math.log(n))
    assert np.abs(o - ref).max() <= TOL_O_MAX
    assert np.abs(lse - ref_lse).max() <= TOL_LSE_MAX


def test_key_shift_moves_lse_only(tk_lib):
    # K + u (u a small integer vector, exact in bf16 for these inputs) adds
    # scale * q_i . u to every score of row i: O is unchanged and LSE moves
    # by exactly that amount.
    D, N = 64, 500
    q = bf(torch.randint(-2, 3, (1, 1, N, D)).float())
    k = bf(torch.randint(-2, 3, (1, 1, N, D)).float())
    _, _, v = draw((1, 1, N, D), seed=203)
    u = torch.randint(-3, 4, (D,)).float()
    k2 = bf(k.float() + u)
    assert torch.equal(k2.float(), k.float() + u)
    scale = 0.125
    o1, l1 = run_gpu(tk_lib, q, k, v, scale, False)
    o2, l2 = run_gpu(tk_lib, q, k2, v, scale, False)
    shift = scale * (q.double()[0, 0] @ u.double()).numpy()
    assert np.abs(o2 - o1).max() <= 2e-2
    assert np.abs((l2 - l1)[0, 0] - shift).max() <= 1e-3


def test_permuting_kv_rows_together(tk_lib):
    q, k, v = draw((2, 2, 384, 128), seed=204)
    perm = torch.randperm(384, generator=torch.Generator().manual_seed(3))
    o1, l1 = run_gpu(tk_lib, q, k, v, 0.09, False)
    o2, l2 = run_gpu(tk_lib, q, k[:, :, perm], v[:, :, perm], 0.09, False)
    assert np.abs(o2 - o1).max() <= TOL_O_MAX
    assert np.abs(l2 - l1).max() <= TOL_LSE_MAX


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("where", ["all", "late"])
def test_v_beyond_fp16_range(tk_lib, oracle_lib, causal, where):
    # V with magnitudes up to 2^20 (fp16 stops at 65504): "all" scales every
    # tile; "late" makes only keys >= 600 large, so the exponent drops in the
    # middle of a unit and O already accumulated must be rescaled to match.
    N, D = 1000, 128
    q, k, v = draw((1, 2, N, D), seed=205)
    big = torch.ones((1, 2, N, 1))
    if where == "all":
        big[:] = 2.0 ** 20
    else:
        big[:, :, 600:] = 2.0 ** 20
    v = bf(v.float() * big)
    scale = 1 / math.sqrt(D)
    o, lse = run_gpu(tk_lib, q, k, v, scale, causal)
    o_ref, lse_ref = oracle_lib.attention(q, k, v, scale, causal)
    assert np.isfinite(o).all()
    # compare in units of the V magnitude
    rel = np.abs(o - o_ref) / 2.0 ** 20
    assert rel.max() <= TOL_O_MAX and rel.mean() <= TOL_O_MEAN
    assert np.abs(lse - lse_ref).max() <= TOL_LSE_MAX


@pytest.mark.parametrize("D", [64, 128])
def test_many_single_step_causal_units(tk_lib, oracle_lib, D):
    # N = 256 causal: every unit's first tile takes one K/V step; 608 units
    # give each CTA four in a row (exercises the per-unit barrier phases).
    shape = (8, 76, 256, D)
    q, k, v = draw(shape, seed=206 + D)
    scale = 1 / math.sqrt(D)
    o, lse = run_gpu(tk_lib, q, k, v, scale, True)
    o_ref, lse_ref = oracle_lib.attention(q, k, v, scale, True)
    assert np.abs(o - o_ref).max() <= TOL_O_MAX
    assert np.abs(o - o_ref).mean() <= TOL_O_MEAN
    assert np.abs(lse - lse_ref).max() <= TOL_LSE_MAX


def test_device_timeout_is_reported_and_recoverable(tk_lib, oracle_lib):
    # The test hook makes the kernel skip one K load; the bounded wait for it
    # runs out, the kernel abandons its work and the status word says so.
    # The next call on the same context is correct.
    dev = torch.device("cuda", 0)
    q, k, v = draw((1, 2, 512, 64), seed=207)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((1, 2, 512), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    args = (qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
            1, 2, 512, 64, 0.125, 0, stream)
    tk_lib.tk_attn_debug_drop_load(1)
    try:
        assert tk_lib.tk_attn_fwd(*args) == 0
        assert tk_lib.tk_attn_last_device_error(stream) == tk_lib.TK_ATTN_ERR_DEVICE_TIMEOUT
    finally:
        tk_lib.tk_attn_debug_drop_load(0)
    # the status word was cleared by the read above
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    assert tk_lib.tk_attn_fwd(*args) == 0
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_lib.attention(q, k, v, 0.125, False)
    assert np.abs(o.float().cpu().double().numpy() - o_ref).max() <= TOL_O_MAX
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= TOL_LSE_MAX


def test_causal_unit_lists_mixed_lengths(tk_lib, oracle_lib):
    # 2 * 20 heads * 5 query blocks = 200 causal units of five lengths on 152
    # CTAs: the host-built unit lists give CTAs different unit counts.
    shape = (2, 20, 1280, 128)
    q, k, v = draw(shape, seed=208)
    scale = 1 / math.sqrt(128)
    o, lse = run_gpu(tk_lib, q, k, v, scale, True)
    o_ref, lse_ref = oracle_lib.attention(q, k, v, scale, True)
    assert np.abs(o - o_ref).max() <= TOL_O_MAX
    assert np.abs(o - o_ref).mean() <= TOL_O_MEAN
    assert np.abs(lse - lse_ref).max() <= TOL_LSE_MAX


def test_causal_more_units_than_the_list_holds(tk_lib, oracle_lib):
    # 1 * 12100 heads * 1 query block: more causal units than a launch's unit
    # lists hold, so the kernel takes them in stride order.  Checked on a few
    # heads spread over the range (N = 16: one ragged tile per head).
    B, H, N, D = 1, 12100, 16, 64
    q, k, v = draw((B, H, N, D), seed=209)
    scale = 0.125
    o, lse = run_gpu(tk_lib, q, k, v, scale, True)
    heads = [0, 1, 151, 152, 6049, 12098, 12099]
    sub = (q[:, heads], k[:, heads], v[:, heads])
    o_ref, lse_ref = oracle_lib.attention(*sub, scale, True)
    assert np.abs(o[:, heads] - o_ref).max() <= TOL_O_MAX
    assert np.abs(lse[:, heads] - lse_ref).max() <= TOL_LSE_MAX
