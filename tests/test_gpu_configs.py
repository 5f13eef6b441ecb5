"""The five measured workloads at full size, through the C ABI, in the launch
configuration the benchmark times, compared with the fp64 oracle on EVERY
output row.

The oracle runs on the host cores (fp64, OpenMP) in chunks of whole slices,
so host memory stays bounded; each chunk's rows are compared with the GPU's
as soon as they are computed.  The statistics are over all B*H*N rows:
max |dO| and mean |dO| over all B*H*N*D elements, max |dLSE| over all rows.
The oracle takes about 5 minutes for the four large workloads on 16 cores.
"""
import time

import numpy as np
import pytest
import torch

from attention_forward_tk_gb300.inputs import WORKLOADS, workload_inputs
from conftest import TOL_LSE_MAX, TOL_O_MAX, TOL_O_MEAN

pytestmark = pytest.mark.gpu

# rows of oracle work per chunk (whole slices): about 0.3 GB of fp64 output
CHUNK_ROWS = 1 << 18


def run_gpu(tk_lib, w, q, k, v):
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
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_workload_parity_all_rows(tk_lib, oracle_lib, w):
    q, k, v = workload_inputs(w)
    o_gpu, lse_gpu = run_gpu(tk_lib, w, q, k, v)
    BH, N, D = w.B * w.H, w.N, w.D
    qf, kf, vf = (t.reshape(BH, N, D) for t in (q, k, v))
    o_gpu = o_gpu.reshape(BH, N, D)
    lse_gpu = lse_gpu.reshape(BH, N)
    slices = max(1, CHUNK_ROWS // N)
    max_do = 0.0
    sum_do = 0.0
    max_dl = 0.0
    worst = None
    t0 = time.perf_counter()
    for b0 in range(0, BH, slices):
        b1 = min(BH, b0 + slices)
        o_ref, lse_ref = oracle_lib.attention(qf[b0:b1], kf[b0:b1], vf[b0:b1], w.scale, w.causal)
        do = np.abs(o_gpu[b0:b1].double().numpy() - o_ref)
        dl = np.abs(lse_gpu[b0:b1].double().numpy() - lse_ref)
        sum_do += float(do.sum())
        if do.max() > max_do:
            idx = np.unravel_index(int(do.argmax()), do.shape)
            worst = (b0 + int(idx[0]), int(idx[1]), int(idx[2]), float(o_ref[idx]))
            max_do = float(do.max())
        max_dl = max(max_dl, float(dl.max()))
    mean_do = sum_do / (BH * N * D)
    msg = (f"{w.name}: all {BH * N} rows: max|dO| {max_do:.3e} mean|dO| {mean_do:.3e} "
           f"max|dLSE| {max_dl:.3e}; worst (slice, row, col, O) {worst}; "
           f"oracle {time.perf_counter() - t0:.1f} s")
    print(msg)
    assert max_do <= TOL_O_MAX, msg
    assert mean_do <= TOL_O_MEAN, msg
    assert max_dl <= TOL_LSE_MAX, msg
