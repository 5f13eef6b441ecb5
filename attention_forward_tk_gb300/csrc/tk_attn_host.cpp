// tk_attn_host.cpp -- the forward pass from and to host memory: a pipeline of
// host-to-device copies, tk_attn_fwd launches and device-to-host copies over
// pieces of the B*H independent (batch, head) slices (tk_attn_fwd_host in
// include/tk_attn.h).  It uses the public C ABI and the CUDA runtime only.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "tk_attn.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxPieces = 64;

// Per device: the copy-in and copy-out streams and the events that order
// the pieces across them.  Created on the first call on the device; calls on
// one device enqueue their work one at a time (the mutex), so one call's
// event records never interleave with another's.
struct Pipe {
  std::mutex mu;
  bool ready = false;
  int num_sms = 0;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in_done[kMaxPieces] = {}, fwd_done[kMaxPieces] = {};
};
Pipe g_pipe[kMaxDevices];

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool setup(Pipe &pp, int dev) {
  if (pp.ready) return true;
  if (cudaDeviceGetAttribute(&pp.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  if (cudaStreamCreateWithFlags(&pp.s_in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&pp.s_out, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&pp.start, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&pp.end, cudaEventDisableTiming) != cudaSuccess)
    return false;
  for (int i = 0; i < kMaxPieces; ++i)
    if (cudaEventCreateWithFlags(&pp.in_done[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&pp.fwd_done[i], cudaEventDisableTiming) != cudaSuccess)
      return false;
  pp.ready = true;
  return true;
}

bool overlaps(uintptr_t a, size_t na, uintptr_t b, size_t nb) {
  return na && nb && a < b + nb && b < a + na;
}

}  // namespace

extern "C" size_t tk_attn_fwd_host_workspace_bytes(int B, int H, int N, int D) {
  if (B <= 0 || H <= 0 || N <= 0 || (D != 64 && D != 128)) return 0;
  const size_t tensor = round256((size_t)B * (size_t)H * (size_t)N * (size_t)D * 2u);
  return 4 * tensor + round256((size_t)B * (size_t)H * (size_t)N * 4u);
}

extern "C" int tk_attn_fwd_host_check_args(const void *q, const void *k, const void *v,
                                           const void *o, const float *lse, int B, int H, int N,
                                           int D, float scale, int causal, int pieces,
                                           const void *workspace, size_t workspace_bytes) {
  int st = tk_attn_check_args(q, k, v, o, lse, B, H, N, D, scale, causal);
  if (st) return st;
  if (pieces < 0) return TK_ATTN_ERR_INVALID_ARG;
  const size_t need = tk_attn_fwd_host_workspace_bytes(B, H, N, D);
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < need)
    return TK_ATTN_ERR_INVALID_ARG;
  const size_t tensor = (size_t)B * H * N * D * 2u, rows = (size_t)B * H * N * 4u;
  const uintptr_t w = (uintptr_t)workspace;
  const uintptr_t host[4] = {(uintptr_t)q, (uintptr_t)k, (uintptr_t)v, (uintptr_t)o};
  for (uintptr_t h : host)
    if (overlaps(w, need, h, tensor)) return TK_ATTN_ERR_INVALID_ARG;
  if (overlaps(w, need, (uintptr_t)lse, rows)) return TK_ATTN_ERR_INVALID_ARG;
  return TK_ATTN_OK;
}

extern "C" int tk_attn_fwd_host(const void *q, const void *k, const void *v, void *o,
                                float *lse, int B, int H, int N, int D, float scale, int causal,
                                int pieces, void *workspace, size_t workspace_bytes,
                                tk_attn_stream_t stream) {
  int st = tk_attn_fwd_host_check_args(q, k, v, o, lse, B, H, N, D, scale, causal, pieces,
                                       workspace, workspace_bytes);
  if (st) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return TK_ATTN_ERR_ARCH;
  }
  Pipe &pp = g_pipe[dev];
  std::lock_guard<std::mutex> lock(pp.mu);
  if (!setup(pp, dev)) {
    cudaGetLastError();
    return TK_ATTN_ERR_LAUNCH;
  }
  const long long BH = (long long)B * H;
  // Pieces: by default up to 32, each of at least two waves of 256-query
  // units on the device's SMs (fewer pieces leave more of the last piece's
  // kernel and copy-back unoverlapped; smaller ones run the kernel below a
  // full wave).
  long long np = pieces;
  if (np == 0) {
    np = BH * ((N + 255) / 256) / (2LL * pp.num_sms);
    if (np > 32) np = 32;
  }
  if (np < 1) np = 1;
  if (np > kMaxPieces) np = kMaxPieces;
  if (np > BH) np = BH;
  // A piece starts on a slice whose LSE row begins 16-byte aligned (the
  // kernel's alignment rule): a multiple of g slices.
  const long long g = (N % 4 == 0) ? 1 : (N % 2 == 0) ? 2 : 4;
  const size_t row = (size_t)N * D * 2u, lrow = (size_t)N * 4u;
  const size_t tensor = round256((size_t)BH * row);
  char *qd = static_cast<char *>(workspace), *kd = qd + tensor, *vd = kd + tensor,
       *od = vd + tensor, *ld = od + tensor;
  const char *qh = static_cast<const char *>(q), *kh = static_cast<const char *>(k),
             *vh = static_cast<const char *>(v);
  char *oh = static_cast<char *>(o), *lh = reinterpret_cast<char *>(lse);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bool ok = cudaEventRecord(pp.start, s) == cudaSuccess &&
            cudaStreamWaitEvent(pp.s_in, pp.start, 0) == cudaSuccess;
  long long b0 = 0;
  for (long long c = 0; c < np && ok; ++c) {
    long long b1 = c + 1 == np ? BH : BH * (c + 1) / np;
    b1 -= (c + 1 == np) ? 0 : b1 % g;
    if (b1 <= b0) continue;  // emptied by the rounding
    const size_t off = (size_t)b0 * row, bytes = (size_t)(b1 - b0) * row;
    const size_t loff = (size_t)b0 * lrow, lbytes = (size_t)(b1 - b0) * lrow;
    // copy-in stream: this piece's Q, K, V
    ok = cudaMemcpyAsync(qd + off, qh + off, bytes, cudaMemcpyDefault, pp.s_in) == cudaSuccess &&
         cudaMemcpyAsync(kd + off, kh + off, bytes, cudaMemcpyDefault, pp.s_in) == cudaSuccess &&
         cudaMemcpyAsync(vd + off, vh + off, bytes, cudaMemcpyDefault, pp.s_in) == cudaSuccess &&
         cudaEventRecord(pp.in_done[c], pp.s_in) == cudaSuccess &&
         cudaStreamWaitEvent(s, pp.in_done[c], 0) == cudaSuccess;
    if (!ok) break;
    // the caller's stream: the kernel on this piece, as a problem of b1 - b0 heads
    st = tk_attn_fwd(qd + off, kd + off, vd + off, od + off, reinterpret_cast<float *>(ld + loff),
                     1, (int)(b1 - b0), N, D, scale, causal, stream);
    if (st) break;
    // copy-out stream: this piece's O and LSE
    ok = cudaEventRecord(pp.fwd_done[c], s) == cudaSuccess &&
         cudaStreamWaitEvent(pp.s_out, pp.fwd_done[c], 0) == cudaSuccess &&
         cudaMemcpyAsync(oh + off, od + off, bytes, cudaMemcpyDefault, pp.s_out) == cudaSuccess &&
         cudaMemcpyAsync(lh + loff, ld + loff, lbytes, cudaMemcpyDefault, pp.s_out) ==
             cudaSuccess;
    b0 = b1;
  }
  // The caller's stream reaches its next work only after the last copy-out
  // (also after a failure part-way, so that work already enqueued stays
  // ordered before it).
  const bool joined = cudaEventRecord(pp.end, pp.s_out) == cudaSuccess &&
                      cudaStreamWaitEvent(s, pp.end, 0) == cudaSuccess;
  if (st) return st;
  if (!ok || !joined) {
    cudaGetLastError();
    return TK_ATTN_ERR_LAUNCH;
  }
  return TK_ATTN_OK;
}
