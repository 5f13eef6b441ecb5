"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol ``include/tk_attn.h`` declares, and its host-side argument checks
return the documented status codes.  No compute calls."""
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "tk_attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tk_(?:attn|gemm|based)_\w+)\s*\(", text)))


def test_header_declares_the_binding_names(tk_lib):
    assert declared_functions() == sorted(tk_lib.EXPORTED)


def test_library_exports_every_declared_symbol(tk_lib):
    lib = tk_lib.library()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(tk_lib):
    assert tk_lib.tk_attn_version() == 10600
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = tk_lib.tk_attn_status_string(code)
        assert s and s != "unknown status"
    assert tk_lib.tk_attn_status_string(12345) == "unknown status"


# Fake, never-dereferenced, 16-byte-aligned addresses far apart.
Q, K, V, O, L = (1 << 40), (2 << 40), (3 << 40), (4 << 40), (5 << 40)


def check(tk_lib, q=Q, k=K, v=V, o=O, lse=L, B=2, H=3, N=100, D=64, scale=0.125, causal=0):
    return tk_lib.tk_attn_check_args(q, k, v, o, lse, B, H, N, D, scale, causal)


def test_valid_arguments(tk_lib):
    assert check(tk_lib) == tk_lib.TK_ATTN_OK
    assert check(tk_lib, D=128, causal=1, N=1) == tk_lib.TK_ATTN_OK


@pytest.mark.parametrize("kw", [dict(q=0), dict(k=0), dict(v=0), dict(o=0), dict(lse=0),
                                dict(B=0), dict(H=-1), dict(N=0), dict(scale=0.0),
                                dict(scale=-1.0), dict(scale=float("inf")),
                                dict(scale=float("nan"))])
def test_invalid_arguments(tk_lib, kw):
    assert check(tk_lib, **kw) == tk_lib.TK_ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(D=32), dict(D=96), dict(D=256), dict(q=Q + 8),
                                dict(o=O + 2), dict(lse=L + 4),
                                dict(B=65536, H=65536, N=1)])
def test_unsupported_arguments(tk_lib, kw):
    assert check(tk_lib, **kw) == tk_lib.TK_ATTN_ERR_UNSUPPORTED


def test_overlapping_outputs_are_rejected(tk_lib):
    # O [2,3,100,64] bf16 = 76800 bytes; LSE inside it, or O on top of V
    assert check(tk_lib, lse=O + 1024) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert check(tk_lib, o=V + 16) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert check(tk_lib, lse=Q + 76800 - 16) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    # adjacent but not overlapping is fine
    assert check(tk_lib, lse=O + 76800) == tk_lib.TK_ATTN_OK


def test_fwd_rejects_bad_arguments_before_touching_cuda(tk_lib):
    # the same validation runs first inside tk_attn_fwd, so no GPU is needed
    assert tk_lib.tk_attn_fwd(0, K, V, O, L, 1, 1, 16, 64, 0.125, 0, 0) == \
        tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert tk_lib.tk_attn_fwd(Q, K, V, O, L, 1, 1, 16, 80, 0.125, 0, 0) == \
        tk_lib.TK_ATTN_ERR_UNSUPPORTED


def test_fwd_without_a_gpu_reports_arch(tk_lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert tk_lib.tk_attn_fwd(Q, K, V, O, L, 1, 1, 16, 64, 0.125, 0, 0) == \
        tk_lib.TK_ATTN_ERR_ARCH


def test_binding_raises_when_library_missing(monkeypatch):
    from attention_forward_tk_gb300 import api
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "LIB_PATH", "/nonexistent/libtk_attn.so")
    with pytest.raises(api.TkAttnError):
        api.library()


def test_splitkv_rejects_bad_arguments_before_touching_cuda(tk_lib):
    # the argument checks of the split-key call run before any CUDA call
    args = dict(B=1, H=2, Nq=16, Nk=300, D=64, scale=0.125, splits=0)

    def call(q=Q, k=K, v=V, o=O, lse=L, **kw):
        a = dict(args, **kw)
        return tk_lib.tk_attn_fwd_splitkv(q, k, v, o, lse, a["B"], a["H"], a["Nq"], a["Nk"],
                                          a["D"], a["scale"], a["splits"], 0, 0, 0)
    assert call(q=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert call(Nk=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert call(scale=-1.0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert call(D=96) == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    assert call(k=K + 8) == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    # O [1,2,16,64] bf16 = 4096 bytes: LSE inside it overlaps
    assert call(lse=O + 1024) == tk_lib.TK_ATTN_ERR_INVALID_ARG


def test_splitkv_workspace_query_without_a_gpu(tk_lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert tk_lib.tk_attn_splitkv_workspace_bytes(1, 2, 16, 300, 64, 4) == 0
    assert tk_lib.tk_attn_splitkv_workspace_bytes(1, 2, 16, 300, 96, 4) == 0


def test_gemm_rejects_bad_arguments_before_touching_cuda(tk_lib):
    A, B_, C = Q, K, O

    def chk(a=A, b=B_, c=C, M=256, N=512, K=128):
        return tk_lib.tk_gemm_bf16_check_args(a, b, c, M, N, K)
    assert chk() == tk_lib.TK_ATTN_OK
    assert chk(M=0) == tk_lib.TK_ATTN_OK and chk(K=0) == tk_lib.TK_ATTN_OK
    assert chk(a=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(M=-1) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(K=-8) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(N=500) == tk_lib.TK_ATTN_ERR_UNSUPPORTED   # row stride of C not 16 bytes
    assert chk(K=100) == tk_lib.TK_ATTN_ERR_UNSUPPORTED   # row stride of A, B not 16 bytes
    assert chk(b=B_ + 8) == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    # C [256, 512] bf16 = 256 KiB starting inside A (64 KiB) or B (128 KiB)
    assert chk(c=A + 4096) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(c=B_ - 4096) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    # A and B may alias (C = A A^T)
    assert chk(b=A, N=256) == tk_lib.TK_ATTN_OK
    # the full call checks first, so it needs no GPU to reject
    assert tk_lib.tk_gemm_bf16(A, B_, C, 256, 500, 128, 0) == tk_lib.TK_ATTN_ERR_UNSUPPORTED


def test_bwd_rejects_bad_arguments_before_touching_cuda(tk_lib):
    DO, DQ, DK, DV, WS = (6 << 40), (7 << 40), (8 << 40), (9 << 40), (10 << 40)
    need = tk_lib.tk_attn_bwd_workspace_bytes(2, 3, 100, 64)
    assert need == 2 * 6 * 128 * 4  # two fp32 rows per padded 128-row tile
    assert tk_lib.tk_attn_bwd_workspace_bytes(2, 3, 100, 96) == 0

    def chk(q=Q, k=K, v=V, o=O, lse=L, do=DO, dq=DQ, dk=DK, dv=DV, B=2, H=3, N=100, D=64,
            scale=0.125, ws=WS, wsb=need):
        return tk_lib.tk_attn_bwd_check_args(q, k, v, o, lse, do, dq, dk, dv, B, H, N, D, scale,
                                             ws, wsb)
    assert chk() == tk_lib.TK_ATTN_OK
    assert chk(do=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(ws=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(N=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(scale=float("nan")) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(wsb=need - 4) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(D=96) == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    assert chk(dk=DK + 8) == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    # dq inside q, dv inside dk, the workspace inside dv
    assert chk(dq=Q + 64) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(dv=DK + 64) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(ws=DV + 64) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    # the full call checks first, so it needs no GPU to reject
    assert tk_lib.tk_attn_bwd(Q, K, V, O, L, DO, DQ, DK, DV, 2, 3, 100, 96, 0.125, 0, WS, need,
                              0) == tk_lib.TK_ATTN_ERR_UNSUPPORTED


def test_based_rejects_bad_arguments_before_touching_cuda(tk_lib):
    def chk(q=Q, k=K, v=V, y=O, z=L, B=2, H=3, N=100, Df=16, Dv=64, scale=0.25):
        return tk_lib.tk_based_check_args(q, k, v, y, z, B, H, N, Df, Dv, scale)
    assert chk() == tk_lib.TK_ATTN_OK
    assert chk(scale=-0.5) == tk_lib.TK_ATTN_OK  # T(s) >= 1/2 for any real s
    assert chk(scale=float("inf")) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(v=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(H=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(Df=32) == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    assert chk(Dv=128) == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    assert chk(z=L + 4) == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    # y [2,3,100,64] bf16 = 76800 bytes: z inside it, or y over v
    assert chk(z=O + 1024) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert chk(y=V + 512) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert tk_lib.tk_based_fwd(Q, K, V, O, L, 2, 3, 100, 32, 64, 0.25, 1, 0) == \
        tk_lib.TK_ATTN_ERR_UNSUPPORTED


# ---------------------------------------------------------------- host-buffer call

W = 6 << 40  # fake device workspace, 256-byte aligned


def host_need(B=2, H=3, N=100, D=64):
    r = lambda x: (x + 255) // 256 * 256
    return 4 * r(B * H * N * D * 2) + r(B * H * N * 4)


def test_host_workspace_bytes(tk_lib):
    assert tk_lib.tk_attn_fwd_host_workspace_bytes(2, 3, 100, 64) == host_need()
    assert tk_lib.tk_attn_fwd_host_workspace_bytes(1, 1, 1, 128) == host_need(1, 1, 1, 128)
    for bad in ((0, 1, 1, 64), (1, 1, 0, 64), (1, 1, 16, 96)):
        assert tk_lib.tk_attn_fwd_host_workspace_bytes(*bad) == 0


def host_check(tk_lib, pieces=0, ws=W, ws_bytes=None, **kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, B=2, H=3, N=100, D=64, scale=0.125, causal=0)
    a.update(kw)
    need = host_need(a["B"], a["H"], a["N"], a["D"]) if ws_bytes is None else ws_bytes
    return tk_lib.tk_attn_fwd_host_check_args(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"],
                                              a["H"], a["N"], a["D"], a["scale"], a["causal"],
                                              pieces, ws, need)


def test_host_call_arguments(tk_lib):
    assert host_check(tk_lib) == tk_lib.TK_ATTN_OK
    assert host_check(tk_lib, pieces=64, causal=1) == tk_lib.TK_ATTN_OK
    # the tensor rules of tk_attn_fwd apply to the host buffers
    assert host_check(tk_lib, D=96) == tk_lib.TK_ATTN_ERR_UNSUPPORTED
    assert host_check(tk_lib, q=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert host_check(tk_lib, o=V + 16) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    # the pieces count and the workspace
    assert host_check(tk_lib, pieces=-1) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert host_check(tk_lib, ws=0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert host_check(tk_lib, ws=W + 16) == tk_lib.TK_ATTN_ERR_INVALID_ARG   # not 256-aligned
    assert host_check(tk_lib, ws_bytes=host_need() - 1) == tk_lib.TK_ATTN_ERR_INVALID_ARG
    assert host_check(tk_lib, ws=O - 256) == tk_lib.TK_ATTN_ERR_INVALID_ARG  # over the output


def test_host_call_rejects_before_touching_cuda(tk_lib):
    assert tk_lib.tk_attn_fwd_host(Q, K, V, O, L, 2, 3, 100, 64, 0.125, 0, -1, W, host_need(),
                                   0) == tk_lib.TK_ATTN_ERR_INVALID_ARG
