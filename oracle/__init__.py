"""fp64 CPU oracle for the fused attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import, call or build anything in this
package.  The CUDA library never links or loads it, and the two share no code:
this package computes attention from its plain definition, in double
precision, so the GPU kernels have something independent to be checked against.

Contents
  attention_rows   plain definition (C, OpenMP, fp64) for chosen rows
  attention        the same for every row of a [B, H, N, D] problem
  attention_qk_rows, attention_qk
                   the same definition for Nq queries against Nk keys
                   (inference shape); causal aligned to the last key
  attention_bwd    dQ, dK, dV of the same definition for a given dO (numpy,
                   fp64), with the magnitude sums that bound kernel rounding
  based_quadratic, based_recurrent, based_rows
                   Based linear attention (Taylor-2 feature map): the
                   definition evaluated directly, through explicit feature
                   maps with a running state (causal), and directly for
                   chosen causal rows only
  gemm_abt         C = A B^T for bf16 A [M, K], B [N, K] in float64, with the
                   per-element magnitude sum that bounds fp32 accumulation
  tiled_online_softmax
                   numpy restatement of the tile-by-tile online-softmax
                   recurrence the kernel examples on the pages use, both in
                   the pages' per-step-renormalising form and in the
                   deferred-division form; tiny sizes only.
  build            compile the C part (called by the graft entry's build()).

Sources: the attention definition computed by the "RTX 4090 flash attention"
and "H100 FlashAttention-2 forward" examples in the ThunderKittens news
write-up (88811315.cn, post 77732); the causal mask and the log-sum-exp follow
the plainest reading of the requested interface (keys j <= i visible; natural
log over scaled, masked scores).
"""
from .brute import (attention, attention_qk, attention_qk_rows, attention_rows, build, lib_path,
                    max_threads)
from .backward import attention_bwd
from .based import based_quadratic, based_recurrent, based_rows
from .gemm import gemm_abt
from .tiled import tiled_online_softmax

__all__ = [
    "attention_bwd",
    "based_quadratic",
    "based_recurrent",
    "based_rows",
    "attention",
    "attention_qk",
    "attention_qk_rows",
    "attention_rows",
    "build",
    "gemm_abt",
    "lib_path",
    "max_threads",
    "tiled_online_softmax",
]
