"""Queries and keys of different lengths with the keys split into ranges
(tk_attn_fwd_splitkv), through the C ABI, against the fp64 oracle's
attention_qk, element by element.  Tolerances as for the single-pass call:
max |dO| <= 2e-2, mean |dO| <= 2e-3, max |dLSE| <= 1e-3."""
import math

import numpy as np
import pytest
import torch

from conftest import TOL_LSE_MAX, TOL_O_MAX, TOL_O_MEAN

pytestmark = pytest.mark.gpu


def draw_qk(B, H, Nq, Nk, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, Nq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H, Nk, D), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, Nk, D), generator=g).to(torch.bfloat16)
    return q, k, v


def run_split(tk_lib, q, k, v, scale, splits, ws_extra=0, ws_bytes=None):
    dev = torch.device("cuda", 0)
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=dev)
    need = tk_lib.tk_attn_splitkv_workspace_bytes(B, H, Nq, Nk, D, splits)
    ws = torch.empty(max(need + ws_extra, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = tk_lib.tk_attn_fwd_splitkv(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), B, H, Nq, Nk, D, scale, splits,
                                    ws.data_ptr(), need if ws_bytes is None else ws_bytes, stream)
    if st != 0:
        torch.cuda.synchronize()
        return st, o, lse, need
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    torch.cuda.synchronize()
    return st, o.float().cpu().double().numpy(), lse.cpu().double().numpy(), need


CASES = [
    # (B, H, Nq, Nk, D, splits)
    (1, 4, 256, 4096, 128, 0),   # default split count (one 128-key tile per range here)
    (2, 3, 100, 3000, 64, 5),    # ragged query and key tails
    (1, 8, 1, 2048, 128, 0),     # one query row per slice (decode)
    (1, 2, 300, 1000, 64, 1),    # one range: the single-pass kernel with Nq != Nk
    (1, 1, 17, 129, 128, 7),     # 2 key tiles: clamped to 2 ranges
    (2, 2, 512, 256, 64, 0),     # more queries than keys
    (1, 2, 640, 5000, 128, 3),   # 3 query blocks x 3 ranges
    # at most 128 queries: the second Q tile of every unit is empty
    (1, 8, 1, 2048, 64, 1),      # decode, single pass, head dim 64
    (2, 4, 64, 1500, 128, 1),    # half of tile 0's warps hold no query
    (1, 2, 128, 777, 64, 2),     # tile 0 full, tile 1 empty, split
    (8, 32, 1, 4096, 128, 4),    # decode, several units per CTA (stage reuse across units)
    (8, 32, 3, 4096, 64, 8),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_splitkv_parity(tk_lib, oracle_lib, case):
    B, H, Nq, Nk, D, splits = case
    q, k, v = draw_qk(B, H, Nq, Nk, D, seed=500 + Nq + Nk + D + splits)
    scale = 1 / math.sqrt(D)
    st, o, lse, _ = run_split(tk_lib, q, k, v, scale, splits)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    o_ref, lse_ref = oracle_lib.attention_qk(q, k, v, scale, False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    do = np.abs(o - o_ref)
    assert do.max() <= TOL_O_MAX, do.max()
    assert do.mean() <= TOL_O_MEAN, do.mean()
    assert np.abs(lse - lse_ref).max() <= TOL_LSE_MAX


def test_splitkv_ranges_agree_with_one_range(tk_lib):
    # the combination over ranges against the single-pass result: both within
    # rounding of one another for every split count
    q, k, v = draw_qk(1, 4, 256, 2048, 64, seed=601)
    _, o1, l1, need1 = run_split(tk_lib, q, k, v, 0.125, 1)
    assert need1 == 0
    for s in (2, 3, 16):
        st, o, l, need = run_split(tk_lib, q, k, v, 0.125, s)
        assert st == 0 and need > 0
        assert np.abs(o - o1).max() <= 2e-2
        assert np.abs(l - l1).max() <= 1e-4


def test_splitkv_rejects_a_short_workspace(tk_lib):
    q, k, v = draw_qk(1, 2, 128, 1024, 128, seed=602)
    B, H, Nq, Nk, D = 1, 2, 128, 1024, 128
    need = tk_lib.tk_attn_splitkv_workspace_bytes(B, H, Nq, Nk, D, 4)
    assert need == 4 * B * H * Nq * (D + 1) * 4
    st, o, lse, _ = run_split(tk_lib, q, k, v, 0.1, 4, ws_bytes=need - 16)
    assert st == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert torch.isnan(o).all() and torch.isnan(lse).all()  # outputs untouched


@pytest.mark.parametrize("name", ["prefill_q256_k32k_d128", "chunk_q1024_k16k_d128_c",
                                  "decode_b8_q1_k16k_d128"])
def test_inference_workload_all_rows(tk_lib, oracle_lib, name):
    # the timed inference shapes at full size, the default split count,
    # every row against the oracle
    from attention_forward_tk_gb300.inputs import BY_NAME, workload_inputs
    w = BY_NAME[name]
    q, k, v = workload_inputs(w)
    st, o, lse = run_qk(tk_lib, q, k, v, w.scale, w.causal, 0)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    o_ref, lse_ref = oracle_lib.attention_qk(q, k, v, w.scale, w.causal)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    do = np.abs(o - o_ref)
    assert do.max() <= TOL_O_MAX, do.max()
    assert do.mean() <= TOL_O_MEAN, do.mean()
    assert np.abs(lse - lse_ref).max() <= TOL_LSE_MAX


def run_qk(tk_lib, q, k, v, scale, causal, splits):
    """tk_attn_fwd_qk (optionally causal, aligned to the last key)."""
    dev = torch.device("cuda", 0)
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=dev)
    need = tk_lib.tk_attn_splitkv_workspace_bytes(B, H, Nq, Nk, D, splits)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = tk_lib.tk_attn_fwd_qk(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, H, Nq, Nk, D, scale, int(causal), splits,
                               ws.data_ptr(), need, stream)
    if st == 0:
        assert tk_lib.tk_attn_last_device_error(stream) == 0
    torch.cuda.synchronize()
    return st, o.float().cpu().double().numpy(), lse.cpu().double().numpy()


CAUSAL_CASES = [
    # (B, H, Nq, Nk, D, splits): causal, queries are the last Nq positions
    (1, 4, 256, 4096, 128, 0),   # a prefill chunk at the end of 4096 keys, default split
    (2, 3, 100, 3000, 64, 5),    # ragged tails
    (1, 8, 1, 2048, 128, 0),     # decode: one query sees every key
    (1, 2, 300, 1000, 64, 1),    # one range: the single-pass kernel with an offset mask
    (1, 1, 17, 129, 128, 7),
    (1, 2, 640, 5000, 128, 3),   # blocks with different range counts
    (1, 2, 1000, 1000, 128, 4),  # Nq == Nk: tk_attn_fwd's causal mask, split over keys
    (1, 2, 256, 320, 128, 3),    # the first rows see no key of the last range
    (2, 1, 256, 320, 64, 3),
    (1, 3, 513, 2100, 64, 0),
    (2, 4, 64, 1500, 128, 1),    # at most 128 queries, single pass
    (1, 2, 128, 777, 64, 2),
    (1, 4, 33, 4000, 128, 0),
    (4, 40, 16, 3000, 128, 3),   # several units per CTA
]


@pytest.mark.parametrize("case", CAUSAL_CASES, ids=lambda c: "x".join(map(str, c)))
def test_qk_causal_parity(tk_lib, oracle_lib, case):
    B, H, Nq, Nk, D, splits = case
    q, k, v = draw_qk(B, H, Nq, Nk, D, seed=800 + Nq + Nk + D + splits)
    scale = 1 / math.sqrt(D)
    st, o, lse = run_qk(tk_lib, q, k, v, scale, True, splits)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    o_ref, lse_ref = oracle_lib.attention_qk(q, k, v, scale, True)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    do = np.abs(o - o_ref)
    assert do.max() <= TOL_O_MAX, do.max()
    assert do.mean() <= TOL_O_MEAN, do.mean()
    assert np.abs(lse - lse_ref).max() <= TOL_LSE_MAX


def test_qk_unmasked_is_the_split_call(tk_lib):
    # causal = 0 is tk_attn_fwd_splitkv exactly
    q, k, v = draw_qk(1, 2, 300, 2000, 128, seed=901)
    st1, o1, l1 = run_qk(tk_lib, q, k, v, 0.09, False, 3)
    st2, o2, l2, _ = run_split(tk_lib, q, k, v, 0.09, 3)
    assert st1 == 0 and st2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_qk_causal_rejects_more_queries_than_keys(tk_lib):
    q, k, v = draw_qk(1, 1, 300, 200, 64, seed=902)
    st, o, lse = run_qk(tk_lib, q, k, v, 0.125, True, 0)
    assert st == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert np.isnan(o).all() and np.isnan(lse).all()  # outputs untouched


@pytest.mark.parametrize("case", [(1, 8, 1, 262144 + 33, False), (1, 8, 5, 262144 + 33, True)],
                         ids=["decode_256k", "q5_256k_causal"])
def test_long_key_range_all_rows(tk_lib, oracle_lib, case):
    """A quarter million cached keys (16x the timed decode shape): the
    default split over keys, every query row against the oracle.  Peaky
    inputs (4 N(0,1) queries and keys, Student-t V), so that O is of order one
    rather than a near-zero average of 2.6*10^5 rows."""
    from attention_forward_tk_gb300.inputs import draw
    B, H, Nq, Nk, causal = case
    D = 128
    q, k, v = draw((B, H, Nq, D), 1700 + Nq, "peaky_t3", kv_shape=(B, H, Nk, D))
    scale = 1 / math.sqrt(D)
    st, o, lse = run_qk(tk_lib, q, k, v, scale, causal, 0)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    o_ref, lse_ref = oracle_lib.attention_qk(q, k, v, scale, causal)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    do = np.abs(o - o_ref)
    assert do.max() <= TOL_O_MAX, do.max()
    assert do.mean() <= TOL_O_MEAN, do.mean()
    assert np.abs(lse - lse_ref).max() <= TOL_LSE_MAX
