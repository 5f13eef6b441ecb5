// tk_gemm.cuh -- bf16 GEMM C = A B^T on the same TMA / tcgen05 / mbarrier
// layers as the attention kernel (GB300, sm_103a).
//
//   A [M, K], B [N, K] bf16 row-major (both K-major), C [M, N] bf16,
//   fp32 accumulation in tensor memory.
//
// The paper summary "ThunderKittens: Simple, Fast, and Adorable AI Kernels"
// (shd-paper.top, abstract and results) reports that the tile primitives match
// cuBLAS on GEMM but prints no GEMM kernel; this one is written for Blackwell
// from the textbook definition C_ij = sum_k A_ik B_jk.
//
// One persistent CTA per SM, 192 threads:
//   warps 0-3  epilogue: tensor memory -> registers -> bf16 -> global
//              (thread = output row = TMEM lane)
//   warp 4     TMA producer (one thread): A and B tiles through a ring
//   warp 5     tcgen05 MMA issue (one thread) and TMEM allocation
// Output tiles of 128 x 256; K in steps of 64 (one 128-byte swizzle row):
// a stage holds A 128 x 64 (16 KB) and B 256 x 64 (32 KB).  Two 256-column
// fp32 accumulators in tensor memory let the epilogue drain one tile while
// the MMAs of the next fill the other.  Every mbarrier wait is bounded; a
// wait that runs out raises the CTA's abort flag and records an error code.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace tkattn {

// 2-D tiled load global -> shared with an L2 cache-policy hint; completion is
// counted on `bar` in bytes (the whole box, including zero-filled elements).
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map,
                                                 uint64_t *bar, int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

struct GemmParams {
  __nv_bfloat16 *c;  // [M, N]
  int *err;          // device error word
  int M, N, K;
  int tiles_m, tiles_n, num_tiles, k_blocks;
};

struct GemmCfg {
  static constexpr int kBM = 128, kBN = 256, kBK = 64;
  static constexpr int kStages = 4;
  static constexpr int kABytes = kBM * kBK * 2;     // 16 KB
  static constexpr int kBBytes = kBN * kBK * 2;     // 32 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kSmemAlloc = kStages * kStageBytes + 1024;
  static constexpr int kThreads = 192;
  static constexpr int kGroupM = 8;  // tile raster: groups of 8 M-tiles share B tiles in L2
};

struct GemmShared {
  uint64_t full[GemmCfg::kStages];   // TMA landed A and B of a stage   (1 + tx)
  uint64_t empty[GemmCfg::kStages];  // MMAs done reading a stage       (commit)
  uint64_t acc_full[2];              // accumulator b complete          (commit)
  uint64_t acc_empty[2];             // epilogue has read accumulator b (4 warps)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// Tile t -> (tm, tn): groups of kGroupM consecutive M-tiles walk all N-tiles,
// so the CTAs running at one time share B tiles (and A tiles) in L2.
__device__ __forceinline__ void gemm_tile(const GemmParams &p, int t, int &tm, int &tn) {
  const int per_group = GemmCfg::kGroupM * p.tiles_n;
  const int g = t / per_group;
  const int first_m = g * GemmCfg::kGroupM;
  const int gm = min(GemmCfg::kGroupM, p.tiles_m - first_m);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

__global__ void __launch_bounds__(GemmCfg::kThreads, 1)
    tk_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_b, const GemmParams p) {
  using C = GemmCfg;
  extern __shared__ uint8_t smem_raw[];
  __shared__ GemmShared sb;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = &sb.abort;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sb.full[s], 1);
      mbar_init(&sb.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sb.acc_full[b], 1);
      mbar_init(&sb.acc_empty[b], 4);
    }
    mbar_init(&sb.mma_done, 1);
    sb.abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&sb.tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sb.tmem_base;

  if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    const int row_in_tile = warp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    int tc = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++tc) {
      int tm, tn;
      gemm_tile(p, t, tm, tn);
      const int b = tc & 1;
      if (!mbar_wait(&sb.acc_full[b], (tc >> 1) & 1, abort_flag)) {
        sb.abort = 1;
        atomicCAS(p.err, 0, 1);
        break;
      }
      tc_fence_after_sync();
      const int row = tm * C::kBM + row_in_tile;
      const bool valid = row < p.M;
      __nv_bfloat16 *crow = p.c + (size_t)(valid ? row : 0) * p.N;
#pragma unroll 1
      for (int c0 = 0; c0 < C::kBN; c0 += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + lane_off + b * 256 + c0, r);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          reg_barrier(r[2 * i]);
          reg_barrier(r[2 * i + 1]);
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        }
        const int col = tn * C::kBN + c0;
        if (valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i)  // 8 columns per 16-byte store; N is a multiple of 8
            if (col + 8 * i < p.N)
              *reinterpret_cast<uint4 *>(crow + col + 8 * i) =
                  make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.acc_empty[b]);
    }
  } else if (warp == 4 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    uint32_t it = 0;  // k-blocks loaded so far (all tiles)
    const uint64_t pol = l2_policy_evict_last();
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int tm, tn;
      gemm_tile(p, t, tm, tn);
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const uint32_t s = it % C::kStages;
        if (it >= (uint32_t)C::kStages &&
            !mbar_wait(&sb.empty[s], ((it / C::kStages) - 1) & 1, abort_flag)) {
          sb.abort = 1;
          atomicCAS(p.err, 0, 1);
          goto producer_exit;
        }
        uint8_t *stage = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&sb.full[s], C::kStageBytes);
        tma_load_2d_hint(stage, &tm_a, &sb.full[s], kb * C::kBK, tm * C::kBM, pol);
        tma_load_2d_hint(stage + C::kABytes, &tm_b, &sb.full[s], kb * C::kBK, tn * C::kBN, pol);
      }
    }
  producer_exit:
    // wait for the copies still in flight before the CTA can exit
    {
      int never = 0;
      for (uint32_t s = 0; s < (uint32_t)C::kStages && s < it; ++s) {
        const uint32_t last = it - 1 - ((it - 1 - s) % C::kStages);
        mbar_wait(&sb.full[s], (last / C::kStages) & 1, &never);
      }
    }
  } else if (warp == 5 && lane == 0) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idesc = idesc_f32acc(true, C::kBM, C::kBN, false, false);
    const uint32_t hi = sdesc_sw128_hi(1024);
    const uint32_t base_lo = sdesc_sw128_lo(smem_addr(smem), 16);
    uint32_t it = 0;
    int tc = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++tc) {
      const int b = tc & 1;
      // the epilogue has drained this accumulator (used two tiles ago)
      if (tc >= 2 && !mbar_wait(&sb.acc_empty[b], ((tc >> 1) - 1) & 1, abort_flag)) {
        sb.abort = 1;
        atomicCAS(p.err, 0, 1);
        goto mma_exit;
      }
      tc_fence_after_sync();
      const uint32_t d = tmem + b * 256;
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const uint32_t s = it % C::kStages;
        if (!mbar_wait(&sb.full[s], (it / C::kStages) & 1, abort_flag)) {
          sb.abort = 1;
          atomicCAS(p.err, 0, 1);
          goto mma_exit;
        }
        tc_fence_after_sync();
        const uint32_t a_lo = base_lo + s * (C::kStageBytes >> 4);
        const uint32_t b_lo = a_lo + (C::kABytes >> 4);
        if (kb == 0)
          umma_ss_w<0>(d, a_lo, b_lo, hi, idesc);
        else
          umma_ss_w<1>(d, a_lo, b_lo, hi, idesc);
#pragma unroll
        for (int kk = 1; kk < 4; ++kk)  // 16 K-columns = 32 bytes of a swizzled row
          umma_ss_w<1>(d, a_lo + kk * 2, b_lo + kk * 2, hi, idesc);
        umma_commit(&sb.empty[s]);  // the stage is free once these MMAs have read it
      }
      umma_commit(&sb.acc_full[b]);
    }
  mma_exit:
    umma_commit(&sb.mma_done);
    {
      int never = 0;
      mbar_wait(&sb.mma_done, 0, &never);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace tkattn
