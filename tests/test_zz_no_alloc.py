"""The no-allocation entry point, tk_attn_fwd_splitkv_static, through the C
ABI: the split over keys with its partial results in the library's static
scratch instead of a caller workspace.  Checked on two calls in a row
against tk_attn_fwd_splitkv (the same computation with a torch-allocated
workspace: the outputs must be bit-identical) and against the fp64 oracle
within the parity tolerances (max |dO| <= 2e-2, mean |dO| <= 2e-3,
max |dLSE| <= 1e-3).  Warmed-up calls must leave the device's free memory
and torch's allocator statistics unchanged.  Also checked: its rejection of
a split whose partial results exceed the scratch.

This file is collected last, so a run that stops at the first failure has
already run every other test; it passes alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

from conftest import TOL_LSE_MAX, TOL_O_MAX, TOL_O_MEAN

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def inputs(B, H, Nq, Nk, D, seed):
    """Host (CPU) and device copies of q, k, v ~ N(0, 1), bf16."""
    g = torch.Generator().manual_seed(seed)
    dev = torch.device("cuda", 0)
    host = (torch.randn((B, H, Nq, D), generator=g).to(torch.bfloat16),
            torch.randn((B, H, Nk, D), generator=g).to(torch.bfloat16),
            torch.randn((B, H, Nk, D), generator=g).to(torch.bfloat16))
    return host, tuple(t.to(dev) for t in host)


def outputs(q):
    B, H, Nq, _ = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=q.device)
    return o, lse


@pytest.mark.parametrize("shape", [(1, 8, 256, 8192, 128, 0), (2, 3, 100, 3000, 64, 5)],
                         ids=["B1H8q256k8192d128", "B2H3q100k3000d64s5"])
def test_static_scratch_matches_workspace_call_twice(tk_lib, oracle_lib, shape):
    B, H, Nq, Nk, D, splits = shape
    scale = 0.1
    (qh, kh, vh), (q, k, v) = inputs(B, H, Nq, Nk, D, seed=700 + Nq)
    stream = torch.cuda.current_stream().cuda_stream
    need = tk_lib.tk_attn_splitkv_workspace_bytes(B, H, Nq, Nk, D, splits)
    assert 0 < need <= SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    o_ref, l_ref = outputs(q)
    st = tk_lib.tk_attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_ref.data_ptr(),
                                    l_ref.data_ptr(), B, H, Nq, Nk, D, scale, splits,
                                    ws.data_ptr(), need, stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    o_ora, l_ora = oracle_lib.attention_qk(qh, kh, vh, scale, False)
    results = [outputs(q) for _ in range(2)]
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved())
    for o, lse in results:  # two calls in a row share (and reuse) the scratch
        st = tk_lib.tk_attn_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, D,
                                               scale, splits, stream)
        assert st == 0, tk_lib.tk_attn_status_string(st)
        torch.cuda.synchronize()
    # the calls allocated nothing on the device, through torch or around it
    free1, _ = torch.cuda.mem_get_info()
    assert (torch.cuda.memory_allocated(), torch.cuda.memory_reserved()) == stats0
    assert free1 == free0
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    for call, (o, lse) in enumerate(results):
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        # the same kernels and the same split as the workspace call: identical bits
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), call
        do = np.abs(o.float().cpu().double().numpy() - o_ora)
        dl = np.abs(lse.cpu().double().numpy() - l_ora)
        assert do.max() <= TOL_O_MAX, (call, do.max())
        assert do.mean() <= TOL_O_MEAN, (call, do.mean())
        assert dl.max() <= TOL_LSE_MAX, (call, dl.max())


def test_static_scratch_rejects_a_split_beyond_it(tk_lib):
    # 8 ranges x 64 heads x 4096 queries x 129 floats = 1.08 GB of partial
    # results: more than the 64 MiB scratch.  Rejected before any launch
    # (real device buffers of the declared sizes, about 1.2 GB, never read).
    B, H, Nq, Nk, D, splits = 1, 64, 4096, 32768, 128, 8
    need = tk_lib.tk_attn_splitkv_workspace_bytes(B, H, Nq, Nk, D, splits)
    assert need > SCRATCH_BYTES
    dev = torch.device("cuda", 0)
    qb = B * H * Nq * D * 2
    kb = B * H * Nk * D * 2
    # disjoint device buffers of the declared sizes (contents irrelevant)
    q = torch.zeros(qb, dtype=torch.uint8, device=dev)
    o = torch.full((qb,), 0x7F, dtype=torch.uint8, device=dev)
    k = torch.zeros(kb, dtype=torch.uint8, device=dev)
    v = torch.zeros(kb, dtype=torch.uint8, device=dev)
    lse = torch.full((B * H * Nq,), 3.0, dtype=torch.float32, device=dev)
    st = tk_lib.tk_attn_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, D, 0.1,
                                           splits, torch.cuda.current_stream().cuda_stream)
    assert st == tk_lib.TK_ATTN_ERR_TOO_LARGE
    assert "static scratch" in tk_lib.tk_attn_status_string(st)
    torch.cuda.synchronize()
    assert torch.all(o == 0x7F) and torch.all(lse == 3.0)  # outputs untouched
