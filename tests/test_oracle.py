"""Pins for the fp64 oracle: closed forms, invariants, special cases.

Each test fixes a property that the definition O = softmax(scale Q K^T
[+ causal mask]) V, LSE = ln sum exp(scores) forces, chosen so that a plausible
slip in the oracle (a dropped term, a wrong sign or index, a transposed
operand, log base 2 instead of e, an off-by-one causal mask) fails at least
one of them.  No GPU needed.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from attention_forward_tk_gb300.inputs import draw

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def bits(x):
    """float array of bf16-exact values -> bf16 bit patterns (uint16)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.as_tensor(np.asarray(x, dtype=np.float32))), \
        "test inputs must be exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def widen(t):
    return t.double().numpy()


def run(oracle_lib, q, k, v, scale, causal, **kw):
    return oracle_lib.attention(q, k, v, scale, causal, **kw)


# --------------------------------------------------------------------------
# hand-derived golden cases


def test_golden_closed_forms(oracle_lib):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    assert len(cases) >= 4
    for c in cases:
        o, lse = run(oracle_lib, bits(c["q"]), bits(c["k"]), bits(c["v"]),
                     c["scale"], c["causal"])
        np.testing.assert_allclose(o, np.asarray(c["o"], float), rtol=0, atol=1e-12,
                                   err_msg=c["name"])
        np.testing.assert_allclose(lse, np.asarray(c["lse"], float), rtol=0,
                                   atol=1e-12, err_msg=c["name"])


# --------------------------------------------------------------------------
# invariants and closed forms on random bf16 inputs


@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(oracle_lib, causal):
    # V = 1 makes O_i = sum_j P_ij exactly.
    q, k, _ = draw((2, 3, 37, 16), seed=11)
    v = torch.ones_like(q)
    o, _ = run(oracle_lib, q, k, v, 0.25, causal)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(oracle_lib, causal):
    q, k, v = draw((1, 2, 29, 8), seed=12)
    row = v[0, 0, 0].clone()
    vc = row.expand_as(v).contiguous()
    o, _ = run(oracle_lib, q, k, vc, 0.3, causal)
    np.testing.assert_allclose(o, np.broadcast_to(widen(row), o.shape), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_row_shift_moves_lse_only(oracle_lib, causal):
    q, k, v = draw((1, 1, 40, 16), seed=13)
    rows = np.arange(40)
    shifts = np.linspace(-7.0, 11.0, 40)
    o0, l0, _ = oracle_lib.attention_rows(q, k, v, 0.25, causal, rows)
    o1, l1, _ = oracle_lib.attention_rows(q, k, v, 0.25, causal, rows, shifts)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1 - l0, shifts, rtol=0, atol=1e-12)


def test_single_key(oracle_lib):
    q, k, v = draw((2, 2, 1, 64), seed=14)
    o, lse = run(oracle_lib, q, k, v, 0.125, False)
    np.testing.assert_array_equal(o, widen(v))
    dot = (widen(q) * widen(k)).sum(-1)
    np.testing.assert_allclose(lse, 0.125 * dot, rtol=0, atol=1e-12)


def test_causal_row_zero_is_v0(oracle_lib):
    q, k, v = draw((1, 3, 50, 32), seed=15)
    o, lse = run(oracle_lib, q, k, v, 0.2, True)
    np.testing.assert_array_equal(o[:, :, 0, :], widen(v)[:, :, 0, :])
    dot = (widen(q)[:, :, 0] * widen(k)[:, :, 0]).sum(-1)
    np.testing.assert_allclose(lse[:, :, 0], 0.2 * dot, rtol=0, atol=1e-12)


def test_zero_query_is_uniform(oracle_lib):
    _, k, v = draw((1, 2, 33, 16), seed=16)
    q = torch.zeros_like(k)
    n = 33
    o, lse = run(oracle_lib, q, k, v, 0.5, False)
    np.testing.assert_allclose(o, np.broadcast_to(widen(v).mean(axis=2, keepdims=True), o.shape),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, math.log(n), rtol=0, atol=1e-12)
    o, lse = run(oracle_lib, q, k, v, 0.5, True)
    prefix_mean = np.cumsum(widen(v), axis=2) / np.arange(1, n + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix_mean, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.log(np.arange(1, n + 1))[None, None, :].repeat(2, 1),
                               rtol=0, atol=1e-12)


def test_two_keys_sigmoid(oracle_lib):
    q, k, v = draw((1, 1, 2, 16), seed=17)
    qd, kd, vd = widen(q)[0, 0], widen(k)[0, 0], widen(v)[0, 0]
    scale = 0.37
    o, lse = run(oracle_lib, q, k, v, scale, False)
    for i in range(2):
        s0, s1 = scale * qd[i] @ kd[0], scale * qd[i] @ kd[1]
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        np.testing.assert_allclose(o[0, 0, i], w0 * vd[0] + w1 * vd[1], rtol=0, atol=1e-12)
        hi = max(s0, s1)
        np.testing.assert_allclose(lse[0, 0, i], hi + math.log1p(math.exp(min(s0, s1) - hi)),
                                   rtol=0, atol=1e-12)


def test_permuting_kv_rows_together(oracle_lib):
    q, k, v = draw((1, 2, 45, 16), seed=18)
    perm = torch.randperm(45, generator=torch.Generator().manual_seed(5))
    o0, l0 = run(oracle_lib, q, k, v, 0.25, False)
    o1, l1 = run(oracle_lib, q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(),
                 0.25, False)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)
    # permuting K alone must change the result (V rows no longer match K rows)
    o2, _ = run(oracle_lib, q, k[:, :, perm].contiguous(), v, 0.25, False)
    assert np.abs(o2 - o0).max() > 1e-3
    # permuting Q rows permutes the outputs
    o3, l3 = run(oracle_lib, q[:, :, perm].contiguous(), k, v, 0.25, False)
    np.testing.assert_allclose(o3, o0[:, :, perm.numpy()], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l3, l0[:, :, perm.numpy()], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_v_power_of_two_homogeneity(oracle_lib, causal):
    q, k, v = draw((1, 1, 31, 8), seed=19)
    o0, _ = run(oracle_lib, q, k, v, 0.3, causal)
    o1, _ = run(oracle_lib, q, k, (v.float() * 8).to(torch.bfloat16), 0.3, causal)
    np.testing.assert_array_equal(o1, 8 * o0)


def test_causal_row_equals_full_prefix(oracle_lib):
    q, k, v = draw((1, 1, 24, 16), seed=20)
    oc, lc = run(oracle_lib, q, k, v, 0.25, True)
    for i in (0, 1, 7, 23):
        qs = q[:, :, : i + 1].contiguous()
        ks = k[:, :, : i + 1].contiguous()
        vs = v[:, :, : i + 1].contiguous()
        of, lf = run(oracle_lib, qs, ks, vs, 0.25, False)
        np.testing.assert_allclose(oc[0, 0, i], of[0, 0, i], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lc[0, 0, i], lf[0, 0, i], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_lse_bounds(oracle_lib, causal):
    q, k, v = draw((1, 1, 64, 32), seed=21, dist="peaky_t3")
    scale = 1 / math.sqrt(32)
    _, lse = run(oracle_lib, q, k, v, scale, causal)
    s = scale * widen(q)[0, 0] @ widen(k)[0, 0].T
    n = 64
    for i in range(n):
        vis = s[i, : i + 1] if causal else s[i]
        assert vis.max() - 1e-12 <= lse[0, 0, i] <= vis.max() + math.log(vis.size) + 1e-12


# --------------------------------------------------------------------------
# second routines: tiled online softmax and the library's attention


@pytest.mark.parametrize("mode", ["deferred", "renormalize"])
@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_matches_tiled_online_softmax(oracle_lib, mode, causal):
    from oracle import tiled_online_softmax
    for n, bq, bk in [(1, 1, 1), (5, 2, 3), (17, 4, 5), (33, 16, 16), (64, 7, 9), (64, 64, 16)]:
        q, k, v = draw((1, 1, n, 16), seed=100 + n, dist="peaky_t3")
        scale = 0.25
        o, lse = run(oracle_lib, q, k, v, scale, causal)
        ot, lt = tiled_online_softmax(widen(q)[0, 0], widen(k)[0, 0], widen(v)[0, 0],
                                      scale, causal, bq, bk, mode)
        np.testing.assert_allclose(ot, o[0, 0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lt, lse[0, 0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(oracle_lib, causal):
    q, k, v = draw((2, 2, 70, 64), seed=22)
    scale = 0.125
    o, lse = run(oracle_lib, q, k, v, scale, causal)
    qd, kd, vd = q.double(), k.double(), v.double()
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=causal,
                                                           scale=scale)
    s = scale * qd @ kd.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(70, 70, dtype=torch.bool).triu(1), float("-inf"))
    ref_lse = torch.logsumexp(s, dim=-1)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


def test_row_subset_matches_full(oracle_lib):
    q, k, v = draw((2, 3, 20, 16), seed=23)
    o, lse = run(oracle_lib, q, k, v, 0.25, True)
    rows = np.array([0, 19, 20, 59, 119, 77])
    os_, ls, used = oracle_lib.attention_rows(q, k, v, 0.25, True, rows)
    assert used >= 1
    np.testing.assert_array_equal(os_, o.reshape(-1, 16)[rows])
    np.testing.assert_array_equal(ls, lse.reshape(-1)[rows])


def test_rejects_bad_rows(oracle_lib):
    q, k, v = draw((1, 1, 4, 8), seed=24)
    with pytest.raises(ValueError):
        oracle_lib.attention_rows(q, k, v, 0.25, False, [4])


# --------------------------------------------------------------------------
# queries and keys of different lengths (inference shape)


def qk_inputs(seed, BH=2, Nq=5, Nk=23, D=64):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((1, BH, Nq, D), generator=g).to(torch.bfloat16)
    k = torch.randn((1, BH, Nk, D), generator=g).to(torch.bfloat16)
    v = torch.randn((1, BH, Nk, D), generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
def test_qk_zero_query_is_uniform(oracle_lib, causal):
    # Q = 0: every visible score is 0, so O is the mean of the visible V rows
    # and LSE = ln(#visible): all Nk keys, or Nk - Nq + 1 + i under the mask
    # aligned to the last key.
    _, k, v = qk_inputs(301)
    q = torch.zeros((1, 2, 5, 64), dtype=torch.bfloat16)
    o, lse = oracle_lib.attention_qk(q, k, v, 0.3, causal)
    vd = widen(v)[0]
    Nq, Nk = 5, 23
    for i in range(Nq):
        n = (Nk - Nq + 1 + i) if causal else Nk
        np.testing.assert_allclose(o[0, :, i], vd[:, :n].mean(axis=1), atol=1e-12)
        np.testing.assert_allclose(lse[0, :, i], math.log(n), atol=1e-12)


def test_qk_single_key(oracle_lib):
    q, k, v = qk_inputs(302, Nk=1)
    q = q[:, :, :1]
    o, lse = oracle_lib.attention_qk(q, k, v, 0.125, False)
    np.testing.assert_allclose(o, widen(v), atol=1e-12)
    ref = 0.125 * (widen(q)[0, :, 0] * widen(k)[0, :, 0]).sum(-1)
    np.testing.assert_allclose(lse[0, :, 0], ref, atol=1e-12)


def test_qk_causal_last_query_sees_every_key(oracle_lib):
    # under the mask aligned to the last key, the last query sees all Nk keys:
    # it must equal the unmasked result for that row
    q, k, v = qk_inputs(303)
    oc, lc = oracle_lib.attention_qk(q, k, v, 0.1, True)
    on, ln_ = oracle_lib.attention_qk(q, k, v, 0.1, False)
    np.testing.assert_allclose(oc[0, :, -1], on[0, :, -1], atol=1e-12)
    np.testing.assert_allclose(lc[0, :, -1], ln_[0, :, -1], atol=1e-12)
    # and the first query sees Nk - Nq + 1 keys: its LSE is below the full one
    assert np.all(lc[0, :, 0] < ln_[0, :, 0])


@pytest.mark.parametrize("causal", [False, True])
def test_qk_matches_torch_sdpa_float64(oracle_lib, causal):
    # special case that reduces to a library routine: float64 scaled-dot-
    # product attention with an explicit mask (key j <= i + Nk - Nq)
    q, k, v = qk_inputs(304, BH=3, Nq=7, Nk=40)
    Nq, Nk = 7, 40
    qd, kd, vd = (t.double() for t in (q, k, v))
    scale = 0.11
    mask = None
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        mask = j <= i + (Nk - Nq)
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask, scale=scale)
    s = scale * qd @ kd.transpose(-1, -2)
    if causal:
        s = s.masked_fill(~mask, float("-inf"))
    ref_lse = torch.logsumexp(s, dim=-1)
    o, lse = oracle_lib.attention_qk(q, k, v, scale, causal)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), atol=1e-12)


def test_qk_key_splits_combine_by_lse(oracle_lib):
    # the identity a split over keys relies on: with O_s, LSE_s the results on
    # disjoint key ranges, LSE = ln sum_s exp(LSE_s) and O = sum_s
    # exp(LSE_s - LSE) O_s reproduce the result over all keys
    q, k, v = qk_inputs(305, Nk=40)
    o, lse = oracle_lib.attention_qk(q, k, v, 0.125, False)
    bounds = [0, 13, 14, 40]
    parts = [oracle_lib.attention_qk(q, k[:, :, a:b], v[:, :, a:b], 0.125, False)
             for a, b in zip(bounds[:-1], bounds[1:])]
    lses = np.stack([pl for _, pl in parts])
    tot = np.log(np.exp(lses - lses.max(0)).sum(0)) + lses.max(0)
    comb = sum(np.exp(pl - tot)[..., None] * po for po, pl in parts)
    np.testing.assert_allclose(tot, lse, atol=1e-12)
    np.testing.assert_allclose(comb, o, atol=1e-12)


def test_qk_rejects_causal_with_more_queries_than_keys(oracle_lib):
    q, k, v = qk_inputs(306, Nq=5, Nk=3)
    with pytest.raises(ValueError):
        oracle_lib.attention_qk(q, k, v, 0.1, True)


# --------------------------------------------------------------------------
# the GEMM oracle (C = A B^T)


def test_gemm_brute_force_triple_loop(oracle_lib):
    g = torch.Generator().manual_seed(401)
    a = torch.randn((5, 7), generator=g).to(torch.bfloat16)
    b = torch.randn((3, 7), generator=g).to(torch.bfloat16)
    c, mag = oracle_lib.gemm_abt(a, b)
    A, B = widen(a), widen(b)
    for i in range(5):
        for j in range(3):
            ref = 0.0
            absref = 0.0
            for k in range(7):
                ref += A[i, k] * B[j, k]
                absref += abs(A[i, k] * B[j, k])
            assert abs(c[i, j] - ref) <= 1e-12
            assert abs(mag[i, j] - absref) <= 1e-12


def test_gemm_identity_and_transpose(oracle_lib):
    # B = I returns A; swapping the operands transposes the product
    g = torch.Generator().manual_seed(402)
    a = torch.randn((6, 6), generator=g).to(torch.bfloat16)
    b = torch.randn((4, 6), generator=g).to(torch.bfloat16)
    eye = torch.eye(6).to(torch.bfloat16)
    c, _ = oracle_lib.gemm_abt(a, eye)
    np.testing.assert_array_equal(c, widen(a))
    c1, _ = oracle_lib.gemm_abt(a, b)
    c2, _ = oracle_lib.gemm_abt(b, a)
    np.testing.assert_allclose(c1, c2.T, atol=1e-12)


def test_gemm_golden_small(oracle_lib):
    # hand-computed: rows of A against rows of B
    a = bits([[1.0, 2.0, 0.5], [-1.0, 0.0, 4.0]])
    b = bits([[2.0, -1.0, 8.0], [0.25, 0.5, -2.0]])
    c, mag = oracle_lib.gemm_abt(a, b)
    np.testing.assert_array_equal(c, [[2 - 2 + 4, 0.25 + 1 - 1], [-2 + 0 + 32, -0.25 + 0 - 8]])
    np.testing.assert_array_equal(mag, [[2 + 2 + 4, 0.25 + 1 + 1], [2 + 0 + 32, 0.25 + 0 + 8]])


# --------------------------------------------------------------------------
# the backward oracle (dQ, dK, dV)


def _fwd_loss64(Q, K, V, dO, scale, causal):
    """sum(dO * O) with O from float64 torch.softmax: an independent forward."""
    s = scale * (Q @ K.transpose(-1, -2))
    if causal:
        n = Q.shape[-2]
        s = s.masked_fill(~torch.ones(n, n, dtype=torch.bool).tril(), float("-inf"))
    return (dO * (torch.softmax(s, dim=-1) @ V)).sum()


def _bwd_inputs(seed, shape, dist=1.0):
    g = torch.Generator().manual_seed(seed)
    return tuple((dist * torch.randn(shape, generator=g)).to(torch.bfloat16) for _ in range(4))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_float64_autograd(oracle_lib, causal):
    q, k, v, do = _bwd_inputs(501 + causal, (2, 2, 37, 16))
    r = oracle_lib.attention_bwd(q, k, v, do, 0.3, causal)
    Q, K, V = (t.double().requires_grad_() for t in (q, k, v))
    _fwd_loss64(Q, K, V, do.double(), 0.3, causal).backward()
    for name, t in (("dq", Q), ("dk", K), ("dv", V)):
        np.testing.assert_allclose(r[name], t.grad.numpy().reshape(4, 37, 16), rtol=1e-10,
                                   atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_finite_differences(oracle_lib, causal):
    # central differences of sum(dO * O) at the bf16 point, in float64
    q, k, v, do = _bwd_inputs(511 + causal, (1, 1, 9, 4), dist=1.5)
    r = oracle_lib.attention_bwd(q, k, v, do, 0.7, causal)
    base = [t.double() for t in (q, k, v)]
    dO = do.double()
    h = 1e-6
    rng = np.random.default_rng(3)
    for which, name in enumerate(("dq", "dk", "dv")):
        for _ in range(6):
            i, d = int(rng.integers(9)), int(rng.integers(4))
            plus = [t.clone() for t in base]
            minus = [t.clone() for t in base]
            plus[which][0, 0, i, d] += h
            minus[which][0, 0, i, d] -= h
            fd = (_fwd_loss64(*plus, dO, 0.7, causal) - _fwd_loss64(*minus, dO, 0.7, causal)) / (2 * h)
            assert abs(float(fd) - r[name][0, i, d]) <= 1e-7 * (1 + abs(float(fd))), (name, i, d)


def test_bwd_single_key(oracle_lib):
    # one key: P = 1, so dV = dO and the softmax passes no gradient to S
    q, k, v, do = _bwd_inputs(521, (1, 2, 1, 8))
    r = oracle_lib.attention_bwd(q, k, v, do, 0.5, False)
    np.testing.assert_array_equal(r["dv"], widen(do).reshape(2, 1, 8))
    assert np.abs(r["dq"]).max() <= 1e-15 and np.abs(r["dk"]).max() <= 1e-15


def test_bwd_causal_first_row_and_last_key(oracle_lib):
    # causal: query 0 sees key 0 only (dQ_0 = 0); key N-1 is seen by query
    # N-1 only, so dV_{N-1} = P_{N-1,N-1} dO_{N-1}
    q, k, v, do = _bwd_inputs(531, (1, 1, 12, 8))
    r = oracle_lib.attention_bwd(q, k, v, do, 0.4, True)
    assert np.abs(r["dq"][0, 0]).max() <= 1e-15
    Q, K = widen(q)[0, 0], widen(k)[0, 0]
    s = 0.4 * Q[11] @ K.T
    p_last = math.exp(s[11] - s.max()) / np.exp(s - s.max()).sum()
    np.testing.assert_allclose(r["dv"][0, 11], p_last * widen(do)[0, 0, 11], rtol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_dk_sums_to_zero_over_keys(oracle_lib, causal):
    # every row of dS sums to zero (a softmax row is shift-invariant), so
    # sum_j dK_j = scale sum_i (sum_j dS_ij) q_i = 0
    q, k, v, do = _bwd_inputs(541 + causal, (1, 2, 40, 8))
    r = oracle_lib.attention_bwd(q, k, v, do, 0.25, causal)
    assert np.abs(r["dk"].sum(axis=1)).max() <= 1e-12 * (1 + np.abs(r["dk"]).max())


def test_bwd_key_shift_leaves_dq_and_dv(oracle_lib):
    # adding one vector c to every key shifts each score row by q_i . c,
    # which the softmax ignores: P, dS, dV and dQ are unchanged (dK moves)
    g = torch.Generator().manual_seed(551)
    ints = lambda shape: (torch.randint(-8, 9, shape, generator=g).float() / 8)
    q, k, v, do = (ints((1, 1, 10, 4)) for _ in range(4))
    c = ints((4,))
    r0 = oracle_lib.attention_bwd(*(bits(t.numpy()) for t in (q, k, v, do)), 0.5, False)
    r1 = oracle_lib.attention_bwd(*(bits(t.numpy()) for t in (q, k + c, v, do)), 0.5, False)
    np.testing.assert_allclose(r1["dq"], r0["dq"], atol=1e-12)
    np.testing.assert_allclose(r1["dv"], r0["dv"], atol=1e-12)


def test_bwd_slices_and_magnitudes(oracle_lib):
    q, k, v, do = _bwd_inputs(561, (2, 3, 20, 8))
    full = oracle_lib.attention_bwd(q, k, v, do, 0.3, True)
    part = oracle_lib.attention_bwd(q, k, v, do, 0.3, True, slices=[4, 1])
    for name in full:
        np.testing.assert_array_equal(part[name], full[name][[4, 1]])
    for g in ("dq", "dk", "dv"):
        assert (full["mag_" + g] >= np.abs(full[g]) - 1e-12).all()


# --------------------------------------------------------------------------
# the Based linear-attention oracle


def test_based_taylor_values(oracle_lib):
    from oracle.based import taylor2
    np.testing.assert_array_equal(taylor2(np.array([0.0, -1.0, 2.0, -2.0, 1.0])),
                                  [1.0, 0.5, 5.0, 1.0, 2.5])
    s = np.linspace(-6, 6, 1201)
    assert taylor2(s).min() == 0.5  # minimum 1/2 at s = -1: the normaliser is never zero


def test_based_golden_two_keys(oracle_lib):
    # Df = 1, scale 1: q1 = 1 against k = (1, -2): T = (2.5, 1) for query 1
    q = bits([[[[0.0], [1.0]]]])
    k = bits([[[[1.0], [-2.0]]]])
    v = bits([[[[2.0, 0.0], [-4.0, 8.0]]]])
    y, z, _ = oracle_lib.based_quadratic(q, k, v, 1.0, True)
    np.testing.assert_allclose(z[0, 0], [1.0, 3.5], rtol=1e-15)
    np.testing.assert_allclose(y[0, 0, 0], [2.0, 0.0], rtol=1e-15)
    np.testing.assert_allclose(y[0, 0, 1], [(2.5 * 2 - 4) / 3.5, 8 / 3.5], rtol=1e-15)


@pytest.mark.parametrize("scale", [0.25, 1.0])
def test_based_quadratic_equals_recurrent(oracle_lib, scale):
    # the definition evaluated directly and through explicit 1 + Df + Df^2
    # feature maps with a running state agree
    g = torch.Generator().manual_seed(601)
    q, k = (torch.randn((2, 2, 33, 4), generator=g).to(torch.bfloat16) for _ in range(2))
    v = torch.randn((2, 2, 33, 5), generator=g).to(torch.bfloat16)
    y1, z1, _ = oracle_lib.based_quadratic(q, k, v, scale, True)
    y2, z2 = oracle_lib.based_recurrent(q, k, v, scale)
    np.testing.assert_allclose(z1, z2, rtol=1e-12)
    np.testing.assert_allclose(y1, y2, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_based_zero_query_averages(oracle_lib, causal):
    # q = 0: every T is 1, so y is the (prefix) mean of v and z counts keys
    g = torch.Generator().manual_seed(611)
    q = torch.zeros((1, 1, 9, 4), dtype=torch.bfloat16)
    k = torch.randn((1, 1, 9, 4), generator=g).to(torch.bfloat16)
    v = torch.randn((1, 1, 9, 3), generator=g).to(torch.bfloat16)
    y, z, _ = oracle_lib.based_quadratic(q, k, v, 0.5, causal)
    V = widen(v)[0, 0]
    if causal:
        np.testing.assert_allclose(z[0, 0], np.arange(1, 10))
        np.testing.assert_allclose(y[0, 0], np.cumsum(V, axis=0) / np.arange(1, 10)[:, None],
                                   rtol=1e-12, atol=1e-15)
    else:
        np.testing.assert_allclose(z[0, 0], 9.0)
        np.testing.assert_allclose(y[0, 0], np.broadcast_to(V.mean(axis=0), (9, 3)), rtol=1e-12,
                                   atol=1e-15)


def test_based_causal_last_row_sees_everything(oracle_lib):
    g = torch.Generator().manual_seed(621)
    q, k = (torch.randn((1, 2, 17, 8), generator=g).to(torch.bfloat16) for _ in range(2))
    v = torch.randn((1, 2, 17, 6), generator=g).to(torch.bfloat16)
    yc, zc, mc = oracle_lib.based_quadratic(q, k, v, 0.3, True)
    yn, zn, _ = oracle_lib.based_quadratic(q, k, v, 0.3, False)
    np.testing.assert_allclose(yc[:, :, -1], yn[:, :, -1], rtol=1e-13)
    np.testing.assert_allclose(zc[:, :, -1], zn[:, :, -1], rtol=1e-13)
    assert (mc >= np.abs(yc) - 1e-12).all()


def test_based_rows_match_the_recurrent_form(oracle_lib):
    # the per-row evaluation against the running-state form (an independent
    # route through explicit feature maps), on rows of every slice
    g = torch.Generator().manual_seed(631)
    q, k = (torch.randn((2, 2, 40, 4), generator=g).to(torch.bfloat16) for _ in range(2))
    v = torch.randn((2, 2, 40, 3), generator=g).to(torch.bfloat16)
    rows = [0, 1, 39, 40, 77, 80 + 17, 159]
    y, z, mag = oracle_lib.based_rows(q, k, v, 0.4, rows)
    yr, zr = oracle_lib.based_recurrent(q, k, v, 0.4)
    np.testing.assert_allclose(z, zr.reshape(-1)[rows], rtol=1e-12)
    np.testing.assert_allclose(y, yr.reshape(-1, 3)[rows], rtol=1e-10, atol=1e-12)
    assert (mag >= np.abs(y) - 1e-12).all()
    # row 0 of a slice sees its own key alone: y = v_0
    np.testing.assert_array_equal(y[0], widen(v)[0, 0, 0])
