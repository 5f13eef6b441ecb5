// tk_attn_combine.cuh -- second kernel of the split-over-keys attention call.
//
// A query row's keys were cut into S ranges; range s left O_s (already divided
// by its own row sum, fp32) and LSE_s = ln sum_{j in s} exp(score_j).  Over
// all keys,
//   LSE = ln sum_s exp(LSE_s)
//   O   = sum_s exp(LSE_s - LSE) O_s
// because exp(LSE_s - LSE) is range s's share of the row's softmax mass.  The
// result is rounded to bf16; LSE stays fp32.  A range with no key visible to
// the row (causal) has LSE_s = -inf and O_s = 0 and weighs nothing.  This is the same deferred
// normalisation the single-pass kernel applies between K/V tiles, applied
// once more between key ranges.  Memory-bound: one warp per query row, the D
// columns spread over the lanes.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace tkattn {

constexpr int kCombineWarps = 8;  // query rows per block

struct CombineParams {
  int S;            // ranges in the partial results' layout [S, rows]
  long long rows;   // B * H * Nq
  int Nq;           // query rows per slice
  int causal;       // causal: block mb of a slice wrote only its own ranges
  int q_off;        // absolute position of query row 0 (causal)
  int split_tiles;  // 128-key tiles per range
  int nkv;          // 128-key tiles per slice
};

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
    tk_attn_combine_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part,
                           __nv_bfloat16 *__restrict__ o, float *__restrict__ lse,
                           const CombineParams cp) {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  constexpr int kPer = D / 32;  // columns per lane
  const long long row = (long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long rows = cp.rows;
  if (row >= rows) return;
  // Ranges this row's block wrote: all of them, or under the causal mask those
  // up to the block's first tile's last visible key (the key ranges of the
  // forward kernel's causal split).
  int S = cp.S;
  if (cp.causal) {
    const int mb = (int)(row % cp.Nq) / 256;
    const int last_row = min(mb * 256 + 127, cp.Nq - 1);
    const int v0 = min((last_row + cp.q_off) / 128 + 1, cp.nkv);
    S = max(1, (v0 + cp.split_tiles - 1) / cp.split_tiles);
  }
  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lse_part[(size_t)s * rows + row]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
  float z = 0.f;
  for (int s = lane; s < S; s += 32) z += expf(lse_part[(size_t)s * rows + row] - mx);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
  const float total = mx + logf(z);
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  for (int s = 0; s < S; ++s) {
    const float w = expf(lse_part[(size_t)s * rows + row] - total);
    const float *src = o_part + ((size_t)s * rows + row) * D + lane * kPer;
    if constexpr (kPer == 4) {
      const float4 x = *reinterpret_cast<const float4 *>(src);
      acc[0] += w * x.x;
      acc[1] += w * x.y;
      acc[2] += w * x.z;
      acc[3] += w * x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2 *>(src);
      acc[0] += w * x.x;
      acc[1] += w * x.y;
    }
  }
  __nv_bfloat16 *dst = o + row * D + lane * kPer;
  if constexpr (kPer == 4) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0], acc[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2], acc[3]);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t *>(&a);
    w.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(dst) = w;
  } else {
    *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(acc[0], acc[1]);
  }
  if (lane == 0) lse[row] = total;
}

}  // namespace tkattn
