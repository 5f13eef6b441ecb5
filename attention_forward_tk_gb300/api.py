"""ctypes binding over the C ABI declared in ``include/tk_attn.h``.

Argument marshalling only: every step of the attention forward pass runs in
the CUDA kernels of ``libtk_attn.so``.  PyTorch supplies device memory and
streams.  The library is built in-tree (``attention_forward_tk_gb300/_build``)
by :func:`attention_forward_tk_gb300.build.build_library`; if it is missing or
fails to load, every call raises :class:`TkAttnError` -- there is no fallback.

The functions named ``tk_attn_*`` mirror the C entry points one for one and
take raw integers (device addresses, sizes, a stream handle).  The
``attention_forward*`` helpers wrap them for torch tensors.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtk_attn.so")

TK_ATTN_OK = 0
TK_ATTN_ERR_INVALID_ARG = -1
TK_ATTN_ERR_UNSUPPORTED = -2
TK_ATTN_ERR_ARCH = -3
TK_ATTN_ERR_LAUNCH = -4
TK_ATTN_ERR_DEVICE_TIMEOUT = -5
TK_ATTN_ERR_TOO_LARGE = -6

# every symbol include/tk_attn.h declares
EXPORTED = (
    "tk_attn_fwd",
    "tk_attn_fwd_host",
    "tk_attn_fwd_host_workspace_bytes",
    "tk_attn_fwd_host_check_args",
    "tk_attn_fwd_splitkv",
    "tk_attn_fwd_qk",
    "tk_attn_fwd_splitkv_static",
    "tk_attn_splitkv_workspace_bytes",
    "tk_attn_check_args",
    "tk_attn_status_string",
    "tk_attn_version",
    "tk_attn_last_device_error",
    "tk_attn_debug_drop_load",
    "tk_gemm_bf16",
    "tk_gemm_bf16_check_args",
    "tk_attn_bwd",
    "tk_attn_bwd_workspace_bytes",
    "tk_attn_bwd_check_args",
    "tk_based_fwd",
    "tk_based_fwd_linear",
    "tk_based_check_args",
)


class TkAttnError(RuntimeError):
    """A non-zero status from the library, or the library could not be loaded."""

    def __init__(self, msg: str, status: int | None = None):
        super().__init__(msg)
        self.status = status


_lock = threading.Lock()
_lib = None


def library() -> ctypes.CDLL:
    """Load libtk_attn.so once and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise TkAttnError(
                f"{LIB_PATH} is missing: build it with "
                "attention_forward_tk_gb300.build.build_library()")
        try:
            lib = ctypes.CDLL(LIB_PATH)
        except OSError as e:  # pragma: no cover - depends on the machine
            raise TkAttnError(f"cannot load {LIB_PATH}: {e}") from e
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.tk_attn_fwd.restype = i
        lib.tk_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        lib.tk_attn_fwd_host.restype = i
        lib.tk_attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp,
                                         ctypes.c_size_t, vp]
        lib.tk_attn_fwd_host_workspace_bytes.restype = ctypes.c_size_t
        lib.tk_attn_fwd_host_workspace_bytes.argtypes = [i, i, i, i]
        lib.tk_attn_fwd_host_check_args.restype = i
        lib.tk_attn_fwd_host_check_args.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp,
                                                    ctypes.c_size_t]
        lib.tk_attn_fwd_splitkv.restype = i
        lib.tk_attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp,
                                            ctypes.c_size_t, vp]
        lib.tk_attn_fwd_qk.restype = i
        lib.tk_attn_fwd_qk.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp,
                                       ctypes.c_size_t, vp]
        lib.tk_attn_fwd_splitkv_static.restype = i
        lib.tk_attn_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.tk_attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
        lib.tk_attn_splitkv_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.tk_attn_check_args.restype = i
        lib.tk_attn_check_args.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i]
        lib.tk_attn_status_string.restype = ctypes.c_char_p
        lib.tk_attn_status_string.argtypes = [i]
        lib.tk_attn_version.restype = i
        lib.tk_attn_version.argtypes = []
        lib.tk_attn_last_device_error.restype = i
        lib.tk_attn_last_device_error.argtypes = [vp]
        lib.tk_attn_debug_drop_load.restype = None
        lib.tk_attn_debug_drop_load.argtypes = [i]
        lib.tk_attn_bwd.restype = i
        lib.tk_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp,
                                    ctypes.c_size_t, vp]
        lib.tk_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.tk_attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.tk_attn_bwd_check_args.restype = i
        lib.tk_attn_bwd_check_args.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f,
                                               vp, ctypes.c_size_t]
        lib.tk_based_fwd.restype = i
        lib.tk_based_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.tk_based_fwd_linear.restype = i
        lib.tk_based_fwd_linear.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
        lib.tk_based_check_args.restype = i
        lib.tk_based_check_args.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f]
        lib.tk_gemm_bf16.restype = i
        lib.tk_gemm_bf16.argtypes = [vp, vp, vp, i, i, i, vp]
        lib.tk_gemm_bf16_check_args.restype = i
        lib.tk_gemm_bf16_check_args.argtypes = [vp, vp, vp, i, i, i]
        _lib = lib
        return _lib


# ----------------------------------------------------------------- raw C calls


def tk_attn_fwd(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int,
                D: int, scale: float, causal: int, stream: int) -> int:
    return int(library().tk_attn_fwd(q, k, v, o, lse, B, H, N, D, ctypes.c_float(scale),
                                     int(causal), stream))


def tk_attn_fwd_host(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int,
                     D: int, scale: float, causal: int, pieces: int, workspace: int,
                     workspace_bytes: int, stream: int) -> int:
    return int(library().tk_attn_fwd_host(q, k, v, o, lse, B, H, N, D, ctypes.c_float(scale),
                                          int(causal), int(pieces), workspace,
                                          int(workspace_bytes), stream))


def tk_attn_fwd_host_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return int(library().tk_attn_fwd_host_workspace_bytes(B, H, N, D))


def tk_attn_fwd_host_check_args(q: int, k: int, v: int, o: int, lse: int, B: int, H: int,
                                N: int, D: int, scale: float, causal: int, pieces: int,
                                workspace: int, workspace_bytes: int) -> int:
    return int(library().tk_attn_fwd_host_check_args(q, k, v, o, lse, B, H, N, D,
                                                     ctypes.c_float(scale), int(causal),
                                                     int(pieces), workspace,
                                                     int(workspace_bytes)))


def tk_attn_fwd_splitkv(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Nq: int,
                        Nk: int, D: int, scale: float, num_splits: int, workspace: int,
                        workspace_bytes: int, stream: int) -> int:
    return int(library().tk_attn_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, D,
                                             ctypes.c_float(scale), int(num_splits), workspace,
                                             int(workspace_bytes), stream))


def tk_attn_fwd_qk(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, Nq: int, Nk: int,
                   D: int, scale: float, causal: int, num_splits: int, workspace: int,
                   workspace_bytes: int, stream: int) -> int:
    return int(library().tk_attn_fwd_qk(q, k, v, o, lse, B, H, Nq, Nk, D, ctypes.c_float(scale),
                                        int(causal), int(num_splits), workspace,
                                        int(workspace_bytes), stream))


def tk_attn_fwd_splitkv_static(q: int, k: int, v: int, o: int, lse: int, B: int, H: int,
                               Nq: int, Nk: int, D: int, scale: float, num_splits: int,
                               stream: int) -> int:
    return int(library().tk_attn_fwd_splitkv_static(q, k, v, o, lse, B, H, Nq, Nk, D,
                                                    ctypes.c_float(scale), int(num_splits),
                                                    stream))


def tk_attn_splitkv_workspace_bytes(B: int, H: int, Nq: int, Nk: int, D: int,
                                    num_splits: int) -> int:
    return int(library().tk_attn_splitkv_workspace_bytes(B, H, Nq, Nk, D, int(num_splits)))


def tk_attn_check_args(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int,
                       D: int, scale: float, causal: int) -> int:
    return int(library().tk_attn_check_args(q, k, v, o, lse, B, H, N, D,
                                            ctypes.c_float(scale), int(causal)))


def tk_attn_status_string(status: int) -> str:
    return library().tk_attn_status_string(int(status)).decode()


def tk_attn_version() -> int:
    return int(library().tk_attn_version())


def tk_attn_last_device_error(stream: int) -> int:
    return int(library().tk_attn_last_device_error(stream))


def tk_attn_debug_drop_load(enable: int) -> None:
    library().tk_attn_debug_drop_load(int(enable))


def tk_attn_bwd(q: int, k: int, v: int, o: int, lse: int, dout: int, dq: int, dk: int,
                dv: int, B: int, H: int, N: int, D: int, scale: float, causal: int,
                workspace: int, workspace_bytes: int, stream: int) -> int:
    return int(library().tk_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, D,
                                     ctypes.c_float(scale), int(causal), workspace,
                                     int(workspace_bytes), stream))


def tk_attn_bwd_workspace_bytes(B: int, H: int, N: int, D: int) -> int:
    return int(library().tk_attn_bwd_workspace_bytes(B, H, N, D))


def tk_attn_bwd_check_args(q: int, k: int, v: int, o: int, lse: int, dout: int, dq: int,
                           dk: int, dv: int, B: int, H: int, N: int, D: int, scale: float,
                           workspace: int, workspace_bytes: int) -> int:
    return int(library().tk_attn_bwd_check_args(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, D,
                                                 ctypes.c_float(scale), workspace,
                                                 int(workspace_bytes)))


def tk_based_fwd(q: int, k: int, v: int, y: int, z: int, B: int, H: int, N: int, Df: int,
                 Dv: int, scale: float, causal: int, stream: int) -> int:
    return int(library().tk_based_fwd(q, k, v, y, z, B, H, N, Df, Dv, ctypes.c_float(scale),
                                      int(causal), stream))


def tk_based_fwd_linear(q: int, k: int, v: int, y: int, z: int, B: int, H: int, N: int,
                        Df: int, Dv: int, scale: float, stream: int) -> int:
    return int(library().tk_based_fwd_linear(q, k, v, y, z, B, H, N, Df, Dv,
                                             ctypes.c_float(scale), stream))


def tk_based_check_args(q: int, k: int, v: int, y: int, z: int, B: int, H: int, N: int, Df: int,
                        Dv: int, scale: float) -> int:
    return int(library().tk_based_check_args(q, k, v, y, z, B, H, N, Df, Dv,
                                             ctypes.c_float(scale)))


def tk_gemm_bf16(a: int, b: int, c: int, M: int, N: int, K: int, stream: int) -> int:
    return int(library().tk_gemm_bf16(a, b, c, M, N, K, stream))


def tk_gemm_bf16_check_args(a: int, b: int, c: int, M: int, N: int, K: int) -> int:
    return int(library().tk_gemm_bf16_check_args(a, b, c, M, N, K))


# short aliases
status_string = tk_attn_status_string
version = tk_attn_version


def last_device_error(stream=None) -> int:
    return tk_attn_last_device_error(_stream_handle(stream))


# ----------------------------------------------------------------- torch helpers


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int):
    if status != TK_ATTN_OK:
        raise TkAttnError(f"tk_attn_fwd: {tk_attn_status_string(status)} ({status})", status)


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None,
                      out=None, lse=None, stream=None):
    """O, LSE = attention forward of bf16 CUDA tensors [B, H, N, D].

    Enqueued on `stream` (default: torch's current stream); returns
    immediately.  `out` (bf16 [B,H,N,D]) and `lse` (fp32 [B,H,N]) are
    allocated by torch when not given.
    """
    import torch
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must be [B, H, N, D] tensors of one shape")
    B, H, N, D = (int(x) for x in q.shape)
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check(tk_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                       lse.data_ptr(), B, H, N, D, float(scale), int(bool(causal)),
                       _stream_handle(stream)))
    return out, lse


def attention_forward_splitkv(q, k, v, scale: float | None = None, num_splits: int = 0,
                              out=None, lse=None, workspace=None, stream=None,
                              causal: bool = False):
    """O, LSE for bf16 CUDA tensors q [B, H, Nq, D] against k, v [B, H, Nk, D],
    with the keys split into `num_splits` ranges (0: the library's default).
    causal: key j visible to query i iff j <= i + Nk - Nq (the queries are
    the sequence's last Nq positions; tk_attn_fwd_qk).  The workspace is
    allocated by torch when not given.  Enqueued on `stream`; returns
    immediately.
    """
    import torch
    if q.dim() != 4 or k.shape != v.shape or k.dim() != 4 or q.shape[:2] != k.shape[:2] or \
            q.shape[3] != k.shape[3]:
        raise ValueError("q must be [B, H, Nq, D] and k, v [B, H, Nk, D]")
    B, H, Nq, D = (int(x) for x in q.shape)
    Nk = int(k.shape[2])
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    need = tk_attn_splitkv_workspace_bytes(B, H, Nq, Nk, D, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(tk_attn_fwd_qk(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr(), B, H, Nq, Nk, D, float(scale), int(bool(causal)),
                          int(num_splits), ws_ptr, ws_bytes, _stream_handle(stream)))
    return out, lse


def attention_backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
                       dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV for bf16 CUDA tensors [B, H, N, D], given the forward's o and
    lse (from attention_forward on the same inputs) and the output gradient
    dout.  Enqueued on `stream`; returns immediately.  Outputs and the
    workspace are allocated by torch when not given.
    """
    import torch
    if q.dim() != 4 or any(t.shape != q.shape for t in (k, v, o, dout)):
        raise ValueError("q, k, v, o, dout must be [B, H, N, D] tensors of one shape")
    B, H, N, D = (int(x) for x in q.shape)
    for t in (q, k, v, o, dout):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, o, dout must be contiguous bf16 CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = tk_attn_bwd_workspace_bytes(B, H, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = tk_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, D,
                     float(scale), int(bool(causal)), workspace.data_ptr(),
                     workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if st != TK_ATTN_OK:
        raise TkAttnError(f"tk_attn_bwd: {tk_attn_status_string(st)} ({st})", st)
    return dq, dk, dv


_autograd_fn = None


def _attention_function():
    """The torch.autograd.Function behind attention(), made on first use (so
    that importing this module does not import torch)."""
    global _autograd_fn
    if _autograd_fn is None:
        import torch

        class _Attention(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, causal, scale):
                o, lse = attention_forward(q, k, v, causal, scale)
                ctx.save_for_backward(q, k, v, o, lse)
                ctx.causal, ctx.scale = causal, scale
                return o

            @staticmethod
            def backward(ctx, dout):
                q, k, v, o, lse = ctx.saved_tensors
                dq, dk, dv = attention_backward(q, k, v, o, lse, dout.contiguous(), ctx.causal,
                                                ctx.scale)
                return dq, dk, dv, None, None

        _autograd_fn = _Attention
    return _autograd_fn


def attention(q, k, v, causal: bool = False, scale: float | None = None):
    """Differentiable attention for contiguous bf16 CUDA tensors [B, H, N, D]
    (torch autograd): O from tk_attn_fwd, which also keeps the LSE; dQ, dK,
    dV from tk_attn_bwd on the saved O and LSE when the graph is
    differentiated.  Runs on torch's current stream."""
    return _attention_function().apply(q, k, v, bool(causal), scale)


def based_forward(q, k, v, causal: bool = True, scale: float | None = None, out=None, z=None,
                  stream=None, algorithm: str = "auto"):
    """Based linear attention: y, z for bf16 CUDA tensors q, k [B, H, N, 16] and
    v [B, H, N, 64] (scale defaults to 1/sqrt(16)).  Enqueued on `stream`.

    algorithm: "direct" (tk_based_fwd, every visible pair), "linear"
    (tk_based_fwd_linear, chunks and a running state; causal only) or "auto"
    (linear for causal calls longer than 256 positions, else direct)."""
    import torch
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k must be [B, H, N, Df] and v [B, H, N, Dv]")
    B, H, N, Df = (int(x) for x in q.shape)
    Dv = int(v.shape[3])
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(Df)
    out = torch.empty_like(v) if out is None else out
    z = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if z is None else z
    if algorithm not in ("auto", "direct", "linear"):
        raise ValueError(f"unknown algorithm {algorithm!r}")
    if algorithm == "linear" and not causal:
        raise ValueError("the linear-time Based kernel is causal only")
    if algorithm == "linear" or (algorithm == "auto" and causal and N > 256):
        st = tk_based_fwd_linear(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 z.data_ptr(), B, H, N, Df, Dv, float(scale),
                                 _stream_handle(stream))
        name = "tk_based_fwd_linear"
    else:
        st = tk_based_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), z.data_ptr(),
                          B, H, N, Df, Dv, float(scale), int(bool(causal)), _stream_handle(stream))
        name = "tk_based_fwd"
    if st != TK_ATTN_OK:
        raise TkAttnError(f"{name}: {tk_attn_status_string(st)} ({st})", st)
    return out, z


def gemm_bf16(a, b, out=None, stream=None):
    """C = A B^T for bf16 CUDA tensors a [M, K] and b [N, K] (fp32 accumulation,
    bf16 result [M, N]).  Enqueued on `stream`; returns immediately.
    """
    import torch
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[1]:
        raise ValueError("a must be [M, K] and b [N, K]")
    for t in (a, b):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("a, b must be contiguous bf16 CUDA tensors")
    M, K = (int(x) for x in a.shape)
    N = int(b.shape[0])
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    st = tk_gemm_bf16(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K,
                      _stream_handle(stream))
    if st != TK_ATTN_OK:
        raise TkAttnError(f"tk_gemm_bf16: {tk_attn_status_string(st)} ({st})", st)
    return out


def attention_forward_host(q, k, v, causal: bool = False, scale: float | None = None,
                           workspace=None, out=None, lse=None, stream=None,
                           chunks: int | None = None):
    """The same call for bf16 tensors in (preferably pinned) host memory,
    through tk_attn_fwd_host: the library copies q, k, v to the device, runs
    the forward pass and copies O and LSE back into host tensors `out` /
    `lse` (allocated pinned when not given), pipelined over `chunks` pieces
    of whole (batch, head) slices (None: the library's default); then this
    function waits for the stream.  `workspace` is a device uint8 tensor of at
    least tk_attn_fwd_host_workspace_bytes(B, H, N, D) bytes, reused between
    calls when given.  Returns (out, lse) on the host."""
    import torch
    B, H, N, D = (int(x) for x in q.shape)
    if not (q.shape == k.shape == v.shape) or q.dtype != torch.bfloat16 or q.is_cuda:
        raise ValueError("q, k, v must be bf16 host tensors of one [B, H, N, D] shape")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    dev = torch.device("cuda", torch.cuda.current_device())
    need = tk_attn_fwd_host_workspace_bytes(B, H, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    st = tk_attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr(), B, H, N, D, float(scale), int(bool(causal)),
                          0 if chunks is None else int(chunks), workspace.data_ptr(),
                          workspace.numel(), _stream_handle(s))
    if st != TK_ATTN_OK:
        raise TkAttnError(f"tk_attn_fwd_host: {tk_attn_status_string(st)} ({st})", st)
    s.synchronize()
    return out, lse
