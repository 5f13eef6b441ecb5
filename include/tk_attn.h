/*
 * tk_attn.h -- C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * Entry points: tk_attn_fwd (the forward pass, below), tk_attn_fwd_host (the
 * same from and to host memory, copies pipelined with the kernel), tk_attn_fwd_splitkv,
 * tk_attn_fwd_qk and tk_attn_fwd_splitkv_static (queries against a longer
 * key set, keys split into ranges; tk_attn_fwd_qk also causal), tk_attn_bwd
 * (dQ, dK, dV), tk_based_fwd and tk_based_fwd_linear (Based linear attention,
 * direct and linear-time) and tk_gemm_bf16 (C = A B^T), each with argument checks that
 * need no GPU, plus status, version and device-error queries.
 *
 * The operation (one call = one whole forward pass over B*H independent
 * (batch, head) slices):
 *
 *   O[b,h]   = softmax( scale * Q[b,h] K[b,h]^T  [+ causal mask] ) V[b,h]
 *   LSE[b,h,i] = ln sum_j exp( scale * q_i . k_j )   over the visible keys j
 *
 * This is the attention that the flash-attention kernel examples compute in
 * the ThunderKittens news write-up (88811315.cn, post 77732): the "RTX 4090
 * flash attention" example (head dim 64) and the "H100 FlashAttention-2
 * forward" example (head dims 64 and 128), which stream K/V in tiles with an
 * online softmax so the N x N score matrix never reaches memory.  Those
 * examples fold a fixed scale (0.125 = 1/sqrt(64), 0.08838834764 = 1/sqrt(128))
 * into Q; here the scale is an argument, applied in fp32 to the fp32 scores.
 * The causal mask (key j visible to query i iff j <= i, diagonal included)
 * and the LSE output are not in those examples; they follow the plainest
 * reading of this interface (natural log, over the scaled, masked scores).
 *
 * Conventions for every entry point:
 *   - Tensors are dense, row-major, in GPU device memory owned by the caller:
 *       q, k, v, o : bf16  [B, H, N, D]   (element (b,h,i,d) at ((b*H+h)*N+i)*D+d)
 *       lse        : fp32  [B, H, N]
 *     Base addresses must be 16-byte aligned.  o and lse must not overlap each
 *     other or any input.
 *   - The library allocates no device memory, never frees caller memory and
 *     never synchronises the stream (except tk_attn_last_device_error).  Work
 *     is enqueued on `stream` (0 = the legacy default stream) and runs
 *     asynchronously; results are valid once the stream reaches that point.
 *   - One exception, once per device: the first call of any entry point on a
 *     device sets that device up (kernel attributes, the address of the
 *     device error word, which it clears with cudaMemset) and ends with
 *     cudaDeviceSynchronize.  Make that first call before any stream
 *     capture; later calls never synchronise.
 *   - Return value: TK_ATTN_OK (0) or a negative TK_ATTN_ERR_* code.  On any
 *     error no work is enqueued and the outputs are left untouched.
 *   - Thread safety: calls may come from several host threads; cached host
 *     state (device properties, the driver entry point) is initialised once.
 *
 * `tk_attn_stream_t` is the CUDA runtime's stream handle type (cudaStream_t),
 * declared here without CUDA headers so plain C callers can include this file.
 */
#ifndef TK_ATTN_H_
#define TK_ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tk_attn_stream_t;

#define TK_ATTN_OK 0
#define TK_ATTN_ERR_INVALID_ARG (-1)   /* null pointer, B/H/N <= 0, bad scale, overlap */
#define TK_ATTN_ERR_UNSUPPORTED (-2)   /* D not 64 or 128, pointer not 16-byte aligned,
                                          or sizes beyond the 32-bit tensor-map ranges */
#define TK_ATTN_ERR_ARCH (-3)          /* current device is not a compute-capability
                                          10.3 (sm_103a) GPU, or no device */
#define TK_ATTN_ERR_LAUNCH (-4)        /* CUDA reported an error building tensor maps
                                          or launching the kernel */
#define TK_ATTN_ERR_DEVICE_TIMEOUT (-5) /* a kernel gave up waiting on an on-chip
                                           barrier (reported by
                                           tk_attn_last_device_error only) */
#define TK_ATTN_ERR_TOO_LARGE (-6)      /* tk_attn_fwd_splitkv_static: the ranges'
                                           partial results exceed its static scratch */

#define TK_ATTN_VERSION 10600 /* major*10000 + minor*100 + patch */

/*
 * tk_attn_fwd -- fused attention forward, asynchronous on `stream`.
 *
 *   q, k, v  [in]  device bf16 [B,H,N,D]
 *   o        [out] device bf16 [B,H,N,D]; o = bf16_rne(softmax(...) V)
 *   lse      [out] device fp32 [B,H,N]; natural-log log-sum-exp of the scaled,
 *                  masked scores of each row
 *   B, H, N  >= 1; any N (no multiple-of-tile requirement)
 *   D        64 or 128
 *   scale    finite and > 0 (usually 1/sqrt(D))
 *   causal   0: every key visible; nonzero: key j visible to query i iff j <= i
 *   stream   CUDA stream to enqueue on
 *
 * Limits (checked before any CUDA call, else TK_ATTN_ERR_UNSUPPORTED):
 * B*H < 2^31 and B*H*ceil(N/256) < 2^31 (work units); each of q, k, v and o
 * below 2^40 bytes (the tensor map's stride range).
 * Errors: TK_ATTN_ERR_INVALID_ARG, _UNSUPPORTED, _ARCH, _LAUNCH (see above).
 */
int tk_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                int B, int H, int N, int D, float scale, int causal,
                tk_attn_stream_t stream);

/*
 * tk_attn_check_args -- the host-side argument validation of tk_attn_fwd,
 * without touching the GPU.  Same arguments (minus the stream); returns the
 * code tk_attn_fwd would return before any CUDA call (TK_ATTN_OK,
 * _INVALID_ARG or _UNSUPPORTED).  Pointers are only compared, never read.
 */
int tk_attn_check_args(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, int B, int H, int N, int D, float scale,
                       int causal);

/*
 * tk_attn_fwd_host -- tk_attn_fwd with Q, K, V read from, and O, LSE
 * written to, HOST memory: the operation is the one above; this call adds
 * the movement between host and device.  Same shapes, layouts, scale and
 * mask as tk_attn_fwd; q, k, v, o, lse are host pointers (page-locked
 * memory, e.g. from cudaHostAlloc, lets the copies overlap the kernel;
 * pageable memory works, with copies the runtime may stage synchronously).
 *
 * The B*H independent (batch, head) slices are cut into `pieces` runs of
 * whole slices (0 = the default: up to 32 pieces of at least two waves of
 * 256-query units each on the device's SMs; clamped to [1, min(64, B*H)]).
 * Piece c's host-to-device copies run on a copy-in stream, its tk_attn_fwd
 * launch on `stream`, its device-to-host copies on a copy-out stream, so the
 * copies of neighbouring pieces overlap the kernel.  The library creates
 * the two side streams and their events once per device; calls on one
 * device enqueue their work one at a time.
 *
 * workspace / workspace_bytes: caller-owned DEVICE memory of at least
 * tk_attn_fwd_host_workspace_bytes(B, H, N, D) bytes, 256-byte aligned,
 * holding the device copies of Q, K, V, O and LSE.  It must not be in use
 * by other work while the call's work runs.
 *
 * Ordering: the call's work starts after the work enqueued on `stream`
 * before it, and `stream` reaches its next work only after the call's last
 * copy-out: O and LSE are valid on the host once the stream reaches that
 * point (synchronise the stream before reading them).
 *
 * Errors: those of tk_attn_check_args (before any CUDA call, nothing
 * enqueued, outputs untouched); TK_ATTN_ERR_INVALID_ARG also for pieces < 0
 * or a missing, misaligned, short or overlapping workspace; _ARCH, _LAUNCH.
 * A CUDA error after the first piece was enqueued returns _LAUNCH with
 * that piece's work still enqueued (and ordered before `stream`'s next work).
 */
int tk_attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int N, int D, float scale, int causal, int pieces,
                     void *workspace, size_t workspace_bytes, tk_attn_stream_t stream);

/* Device workspace tk_attn_fwd_host needs (0 for invalid sizes). */
size_t tk_attn_fwd_host_workspace_bytes(int B, int H, int N, int D);

/* The argument checks of tk_attn_fwd_host alone (no GPU needed). */
int tk_attn_fwd_host_check_args(const void *q, const void *k, const void *v, const void *o,
                                const float *lse, int B, int H, int N, int D, float scale,
                                int causal, int pieces, const void *workspace,
                                size_t workspace_bytes);

/*
 * tk_attn_fwd_splitkv -- the same attention for Nq query rows against Nk
 * keys per (batch, head) slice, unmasked, with the keys split into ranges
 * processed in parallel: the inference shape (a block of new queries against
 * a long run of cached keys), where (slice, 256-query block) pairs alone
 * would leave most SMs idle.  Every key is visible to every query.
 *
 * Definition: the attention definition of the flash-attention examples in
 * the ThunderKittens news write-up (88811315.cn, post 77732), with the query
 * and key counts apart.  The split is exact: range s yields O_s (normalised
 * by its own row sum) and LSE_s, and LSE = ln sum_s exp(LSE_s),
 * O = sum_s exp(LSE_s - LSE) O_s, the same deferred normalisation the
 * examples' per-tile loop applies between K/V tiles.  The pages give no
 * separate inference kernel; this is the plain reading of attention at
 * inference.
 *
 * Arguments (device pointers, contiguous, row-major, 16-byte aligned):
 *   q, o        bf16 [B, H, Nq, D];  k, v  bf16 [B, H, Nk, D];  lse  fp32 [B, H, Nq]
 *   num_splits  key ranges; <= 0 picks enough ranges that (slice, query block,
 *               range) units cover every SM.  Clamped to one range per
 *               128-key tile, and to a count that leaves no range empty.
 *   workspace   device memory the caller owns, at least
 *               tk_attn_splitkv_workspace_bytes(...) bytes (0 when the call
 *               uses one range; then workspace may be NULL); 16-byte aligned,
 *               disjoint from the tensors.  Holds per-range O_s (fp32) and
 *               LSE_s.  Calls that share a workspace must not overlap on the
 *               GPU.
 *   D, scale, stream as for tk_attn_fwd.
 * Two kernel launches on `stream` (ranges, then their combination), or one
 * when there is a single range.  Allocates nothing.
 * Returns TK_ATTN_OK, _INVALID_ARG (null or overlapping pointers, sizes <= 0,
 * bad scale, missing or short workspace), _UNSUPPORTED (head dim, alignment,
 * sizes), _ARCH or _LAUNCH; outputs are untouched on any error.
 */
int tk_attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                        int B, int H, int Nq, int Nk, int D, float scale, int num_splits,
                        void *workspace, size_t workspace_bytes, tk_attn_stream_t stream);

/*
 * tk_attn_splitkv_workspace_bytes -- workspace tk_attn_fwd_splitkv needs for
 * these sizes and split request on the current device (the default split
 * count depends on its SM count): S * B * H * Nq * (D + 1) * 4 bytes for S
 * ranges, 0 for one range or for invalid sizes.
 */
size_t tk_attn_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int D, int num_splits);

/*
 * tk_attn_fwd_qk -- tk_attn_fwd_splitkv with an optional causal mask aligned
 * to the end of the key sequence: the Nq queries are the last Nq positions
 * of a sequence of Nk (a prefill chunk, or a decode step, against the keys
 * cached before it), so key j is visible to query i iff j <= i + (Nk - Nq).
 * For Nq == Nk this is tk_attn_fwd's causal mask.
 *
 * Definition: the attention of the flash-attention examples in the
 * ThunderKittens news write-up (88811315.cn, post 77732); neither those
 * examples nor the rest of the pages fix how a causal mask aligns when
 * queries and keys differ in number, and this is the reading where the
 * queries come last.  causal = 0 is exactly tk_attn_fwd_splitkv.
 *
 * Arguments as for tk_attn_fwd_splitkv, plus causal (0 or nonzero); causal
 * requires Nq <= Nk (else TK_ATTN_ERR_INVALID_ARG).  Under the mask each
 * 256-query block splits only the keys it sees, into ranges of the same
 * length as the unmasked call would use; the workspace the unmasked call
 * needs (tk_attn_splitkv_workspace_bytes) is always enough.  Returns and
 * errors as for tk_attn_fwd_splitkv; outputs untouched on any error.
 */
int tk_attn_fwd_qk(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                   int H, int Nq, int Nk, int D, float scale, int causal, int num_splits,
                   void *workspace, size_t workspace_bytes, tk_attn_stream_t stream);

/*
 * tk_attn_fwd_splitkv_static -- tk_attn_fwd_splitkv for callers that cannot
 * allocate device memory: no workspace argument, and the call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).  The
 * per-range partial results go to a 64 MiB scratch array that is part of
 * the library (a static device array: every GPU that loads the library holds
 * it until the process exits).  The pages have no counterpart: this is an
 * interface variant, not a step of the method.
 *
 * Arguments, ranges and results as for tk_attn_fwd_splitkv.  Returns
 * TK_ATTN_ERR_TOO_LARGE, outputs untouched, when the ranges' partial results
 * (tk_attn_splitkv_workspace_bytes) exceed 64 MiB; fewer ranges
 * (num_splits) or the workspace call then serve.  Nothing in the scratch
 * needs to start at zero.  Every call shares the one array, so calls that
 * overlap on the GPU (other streams, or other threads) race: serialise them.
 * The first call of any tk_attn entry point on a device sets the device up
 * (kernel attributes, the scratch and error-word addresses); make that call
 * before any stream capture.
 */
int tk_attn_fwd_splitkv_static(const void *q, const void *k, const void *v, void *o,
                               float *lse, int B, int H, int Nq, int Nk, int D, float scale,
                               int num_splits, tk_attn_stream_t stream);

/*
 * tk_attn_bwd -- the backward pass of tk_attn_fwd: given dO = dL/dO for some
 * loss L, the gradients
 *
 *   dV = P^T dO,   dS = P o (dO V^T - delta),   dQ = scale dS K,
 *   dK = scale dS^T Q,   with P_ij = exp(scale q_i.k_j - LSE_i) (0 where
 *   masked) and delta_i = sum_d dO_id O_id,
 *
 * the chain rule through the forward definition.  The ThunderKittens pages
 * report causal and non-causal FlashAttention backward kernels (comment
 * thread of es.news.hada.io topic 14783; the paper summary "ThunderKittens:
 * Simple, Fast, and Adorable AI Kernels", shd-paper.top, abstract) but give
 * no formulas; these are the calculus of the forward operation above.
 *
 *   q, k, v, o, dout : bf16 [B, H, N, D]   (o and lse from tk_attn_fwd on
 *   lse              : fp32 [B, H, N]       the same q, k, v, scale, causal)
 *   dq, dk, dv       : bf16 [B, H, N, D]   outputs
 *   workspace        : device scratch of tk_attn_bwd_workspace_bytes(B, H, N,
 *                      D) bytes (fp32 delta and base-2 LSE per row, padded to
 *                      128-row tiles); overwritten, owned by the caller
 *
 * Same conventions as tk_attn_fwd (device memory owned by the caller,
 * 16-byte aligned bases, asynchronous on `stream`, no allocation).  The
 * outputs and the workspace must not overlap each other or any input
 * (TK_ATTN_ERR_INVALID_ARG), and workspace_bytes must cover the size above.
 * Three kernels run on the stream: the row sums, then dK/dV, then dQ.
 */
int tk_attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int D,
                float scale, int causal, void *workspace, size_t workspace_bytes,
                tk_attn_stream_t stream);

/* Workspace bytes tk_attn_bwd needs (0 for invalid sizes); no GPU needed. */
size_t tk_attn_bwd_workspace_bytes(int B, int H, int N, int D);

/* The argument checks of tk_attn_bwd alone (no GPU needed). */
int tk_attn_bwd_check_args(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, const void *dout, const void *dq, const void *dk,
                           const void *dv, int B, int H, int N, int D, float scale,
                           const void *workspace, size_t workspace_bytes);

/*
 * tk_based_fwd -- Based linear attention, forward:
 *
 *   y_i = sum_{j visible} T(s_ij) v_j / z_i,   z_i = sum_{j visible} T(s_ij),
 *   s_ij = scale q_i . k_j,   T(s) = 1 + s + s^2 / 2
 *
 * (visible: j <= i if causal, else every j).  T is the inner product of the
 * second-order Taylor feature maps of exp, phi(x) = [1, x, vec(x x^T)/sqrt 2].
 * The ThunderKittens pages name a Based linear-attention kernel and its
 * throughput (88811315.cn post 77732; es.news.hada.io topic 14783) without
 * defining it; this is the published Based form.  T(s) >= 1/2, so z > 0.
 *
 *   q, k : bf16 [B, H, N, Df]   feature rows, Df = 16
 *   v, y : bf16 [B, H, N, Dv]   Dv = 64
 *   z    : fp32 [B, H, N]       the normaliser
 *
 * Same conventions as tk_attn_fwd; scale may be any finite value.  Other
 * feature or value widths: TK_ATTN_ERR_UNSUPPORTED.
 */
int tk_based_fwd(const void *q, const void *k, const void *v, void *y, float *z, int B, int H,
                 int N, int Df, int Dv, float scale, int causal, tk_attn_stream_t stream);

/*
 * tk_based_fwd_linear -- the causal output of tk_based_fwd through the
 * linear-time algorithm the pages' Based figure refers to: chunks of 128
 * positions, the part of each sum inside a chunk evaluated as T(s_ij)
 * directly, the part before it as phi(q_i) S with the running state
 * S = sum_j phi(k_j) v_j^T (153 features: the distinct terms of phi) and its
 * row of sum_j phi(k_j) for z.  Work is linear in N: about 15 MFLOP of
 * tensor products per 128 positions of a slice, whatever N (the direct
 * evaluation takes 2 (16 + 64) FLOPs per visible pair).
 * Products take bf16 operands (phi and a bf16 copy of the fp32 state) with
 * fp32 accumulation.  Arguments, layouts and errors as tk_based_fwd (always
 * causal); scale must be >= 0 (the feature maps take sqrt(scale)), else
 * TK_ATTN_ERR_INVALID_ARG.  TK_ATTN_ERR_LAUNCH also when the kernel was built
 * with other than the 72 registers a thread its warp roles are split for
 * (checked once per device; the other entry points are unaffected).
 */
int tk_based_fwd_linear(const void *q, const void *k, const void *v, void *y, float *z, int B,
                        int H, int N, int Df, int Dv, float scale, tk_attn_stream_t stream);

/* The argument checks of tk_based_fwd alone (no GPU needed). */
int tk_based_check_args(const void *q, const void *k, const void *v, const void *y,
                        const float *z, int B, int H, int N, int Df, int Dv, float scale);

/*
 * tk_gemm_bf16 -- dense bf16 matrix product with fp32 accumulation:
 *
 *   C[i, j] = sum_k A[i, k] * B[j, k]      (C = A B^T), rounded once to bf16
 *
 * The ThunderKittens paper summary ("ThunderKittens: Simple, Fast, and
 * Adorable AI Kernels", shd-paper.top, abstract and results) reports GEMM
 * at cuBLAS speed as one of the library's kernels; the operation is the
 * textbook product, written here in the layout its tiles use (both operands
 * K-major, as a linear layer's weight is stored).
 *
 *   a : bf16 [M, K] row-major      b : bf16 [N, K] row-major
 *   c : bf16 [M, N] row-major      (device memory owned by the caller)
 *
 * M, N, K >= 0.  N and K must be multiples of 8 (16-byte row strides) and
 * the three base addresses 16-byte aligned, else TK_ATTN_ERR_UNSUPPORTED.
 * M == 0 or N == 0 enqueues nothing; K == 0 sets C to zero.  c must not
 * overlap a or b (TK_ATTN_ERR_INVALID_ARG).  Same stream, allocation and
 * error conventions as tk_attn_fwd; a barrier wait that runs out is reported
 * by tk_attn_last_device_error.
 */
int tk_gemm_bf16(const void *a, const void *b, void *c, int M, int N, int K,
                 tk_attn_stream_t stream);

/* The argument checks of tk_gemm_bf16 alone (no GPU needed). */
int tk_gemm_bf16_check_args(const void *a, const void *b, const void *c, int M, int N, int K);

/* Static, human-readable text for a status code (never NULL). */
const char *tk_attn_status_string(int status);

/* TK_ATTN_VERSION of the loaded library. */
int tk_attn_version(void);

/*
 * tk_attn_last_device_error -- synchronises `stream`, then returns and clears
 * the device-side error word of the current device: TK_ATTN_OK, or
 * TK_ATTN_ERR_DEVICE_TIMEOUT if a kernel abandoned a barrier wait (it then
 * stops its work early and its outputs are incomplete), or TK_ATTN_ERR_LAUNCH
 * if the synchronisation itself failed.  Meant for tests and diagnostics.
 */
int tk_attn_last_device_error(tk_attn_stream_t stream);

/*
 * tk_attn_debug_drop_load -- test hook for the device-side failure path.
 * While enabled (nonzero), every tk_attn_fwd launch skips one K/V load in its
 * first CTA; the MMA thread's bounded wait for that load runs out after about
 * a second, the kernel abandons its work (outputs incomplete) and
 * tk_attn_last_device_error then returns TK_ATTN_ERR_DEVICE_TIMEOUT.  Nothing
 * faults or hangs and the CUDA context stays usable.  Process-wide; off by
 * default.  Not part of the attention operation.
 */
void tk_attn_debug_drop_load(int enable);

#ifdef __cplusplus
}
#endif

#endif /* TK_ATTN_H_ */
