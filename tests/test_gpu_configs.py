"""The five measured workloads at full size, through the C ABI, in the launch
configuration the benchmark times.

The fp64 oracle checks a sample of rows one by one (every row for the
smallest workload): first and last rows of tiles and units, the ragged end,
and random rows, over several (batch, head) slices.  Tolerances as in the
small-shape parity tests.
"""
import numpy as np
import pytest
import torch

from attention_forward_tk_gb300.inputs import WORKLOADS, workload_inputs
from conftest import TOL_LSE_MAX, TOL_O_MAX, TOL_O_MEAN

pytestmark = pytest.mark.gpu


def sample_rows(BH, N, n_random, seed):
    """Flat row indices bh*N + i covering tile/unit edges and random rows."""
    rng = np.random.default_rng(seed)
    edges = sorted({i for i in (0, 1, 2, 63, 64, 126, 127, 128, 129, 255, 256, 257,
                                N // 2, N - 129, N - 128, N - 2, N - 1) if 0 <= i < N})
    heads = sorted({0, BH - 1, *rng.integers(0, BH, size=3).tolist()})
    rows = [bh * N + i for bh in heads for i in edges]
    rows += rng.integers(0, BH * N, size=n_random).tolist()
    return np.unique(np.asarray(rows, dtype=np.int64))


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_workload_parity(tk_lib, oracle_lib, w):
    q, k, v = workload_inputs(w)
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = tk_lib.tk_attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), w.B, w.H, w.N, w.D, w.scale, int(w.causal), stream)
    assert st == 0, tk_lib.tk_attn_status_string(st)
    assert tk_lib.tk_attn_last_device_error(stream) == 0
    torch.cuda.synchronize()
    # properties that hold at any size, on every row
    assert torch.isfinite(lse).all()
    assert torch.isfinite(o.float()).all()
    vmax = vd.float().abs().amax().item()
    assert o.float().abs().amax().item() <= vmax * (1 + 2 ** -8)  # O is a convex mix of V rows
    BH = w.B * w.H
    if BH * w.N <= 4096:
        rows = np.arange(BH * w.N)
    else:
        rows = sample_rows(BH, w.N, n_random=768, seed=w.seed)
    o_ref, lse_ref, _ = oracle_lib.attention_rows(q, k, v, w.scale, w.causal, rows)
    o_gpu = o.reshape(BH * w.N, w.D)[torch.as_tensor(rows, device=dev)].float().cpu().double().numpy()
    l_gpu = lse.reshape(-1)[torch.as_tensor(rows, device=dev)].cpu().double().numpy()
    do = np.abs(o_gpu - o_ref)
    dl = np.abs(l_gpu - lse_ref)
    msg = f"{w.name}: max|dO| {do.max():.3e} mean|dO| {do.mean():.3e} max|dLSE| {dl.max():.3e}"
    print(msg)
    assert do.max() <= TOL_O_MAX, msg
    assert do.mean() <= TOL_O_MEAN, msg
    assert dl.max() <= TOL_LSE_MAX, msg
