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
// Pairs of CTAs (a cluster of two, on the two SMs of one TPC) share one
// 256 x 256 output tile through tcgen05's two-CTA MMA (cta_group::2): each CTA
// loads 128 rows of A and 128 rows of B per 64-wide K step (32 KB), and the
// first CTA of the pair issues M256 N256 K16 MMAs that read the operands of
// both.  Per SM that is two thirds of the shared-memory fill and L2 traffic of
// a one-CTA 128 x 256 tile for the same tensor-core work.  Each CTA's tensor
// memory holds its 128 rows of the two 256-column fp32 accumulators, so one
// tile's epilogue overlaps the next tile's MMAs.  192 threads per CTA:
//   warps 0-3  epilogue: tensor memory -> registers -> bf16 -> global
//              (thread = output row = TMEM lane)
//   warp 4     TMA producer (one thread): this CTA's halves through a ring
//   warp 5     TMEM allocation; in the first CTA, one thread issues the MMAs
// Every mbarrier wait is bounded; a wait that runs out raises the abort flag
// of both CTAs and records an error code, and the kernel winds down.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace tkattn {

// ---------------------------------------------------------------- pair helpers

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Whole-cluster barrier (every thread of both CTAs).
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion (bytes) is
// counted on an mbarrier that may sit in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Two-CTA MMA from descriptor words (see umma_ss_w): A rows 0-127 and B rows
// 0-127 from this CTA's shared memory, rows 128-255 from the peer's at the
// same offsets; D rows 0-127 in this CTA's TMEM, 128-255 in the peer's.
template <uint32_t kAcc>
__device__ __forceinline__ void umma_pair_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                             uint32_t hi, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 a, b;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 a, {%1, %3};\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "n"(kAcc)
      : "memory");
}

// Arrive once on the mbarrier at `bar`'s offset in every CTA of `mask` when
// all tcgen05 operations this thread issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(mask)
      : "memory");
}

// ---------------------------------------------------------------- kernel

struct GemmParams {
  __nv_bfloat16 *c;  // [M, N]
  int *err;          // device error word
  int M, N, K;
  int tiles_m, tiles_n, num_tiles, k_blocks;
};

struct GemmCfg {
  static constexpr int kBM = 256, kBN = 256, kBK = 64;  // tile of a CTA pair
  static constexpr int kHalf = 128;                     // rows of A and of B per CTA
  static constexpr int kStages = 6;
  static constexpr int kABytes = kHalf * kBK * 2;  // 16 KB
  static constexpr int kBBytes = kHalf * kBK * 2;  // 16 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kSmemAlloc = kStages * kStageBytes + 1024;
  static constexpr int kThreads = 192;
  static constexpr int kGroupM = 8;  // tile raster: groups of 8 M-tiles share B tiles in L2
};

struct GemmShared {
  uint64_t full[GemmCfg::kStages];   // first CTA: both CTAs' halves landed (1 + tx)
  uint64_t empty[GemmCfg::kStages];  // MMAs done reading a stage (commit, both CTAs)
  uint64_t acc_full[2];              // accumulator b complete (commit, both CTAs)
  uint64_t acc_empty[2];             // first CTA: 8 epilogue warps have read accumulator b
  uint64_t mma_done;                 // every MMA complete (commit, both CTAs)
  uint32_t tmem_base;
  int abort;
};

// Tile t -> (tm, tn): groups of kGroupM consecutive M-tiles walk all N-tiles,
// so the pairs running at one time share B tiles (and A tiles) in L2.
__device__ __forceinline__ void gemm_tile(const GemmParams &p, int t, int &tm, int &tn) {
  const int per_group = GemmCfg::kGroupM * p.tiles_n;
  const int g = t / per_group;
  const int first_m = g * GemmCfg::kGroupM;
  const int gm = min(GemmCfg::kGroupM, p.tiles_m - first_m);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GemmCfg::kThreads, 1)
    tk_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_b, const GemmParams p) {
  using C = GemmCfg;
  extern __shared__ uint8_t smem_raw[];
  __shared__ GemmShared sb;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool first = rank == 0;
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
  volatile int *abort_flag = &sb.abort;
  auto raise_abort = [&]() {
    sb.abort = 1;
    st_cluster_u32(mapa_shared(smem_addr(&sb.abort), rank ^ 1u), 1u);
    atomicCAS(p.err, 0, 1);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sb.full[s], 1);
      mbar_init(&sb.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sb.acc_full[b], 1);
      mbar_init(&sb.acc_empty[b], 8);
    }
    mbar_init(&sb.mma_done, 1);
    sb.abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc_pair(&sb.tmem_base, 512);
    tmem_relinquish_pair();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  tc_fence_before_sync();
  cluster_sync();  // both CTAs' barriers initialised before any remote signal
  tc_fence_after_sync();
  const uint32_t tmem = sb.tmem_base;

  if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    const int row_in_tile = (int)rank * C::kHalf + warp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t acc_empty0 = mapa_shared(smem_addr(&sb.acc_empty[0]), 0);
    int tc = 0;
    for (int t = pair; t < p.num_tiles; t += num_pairs, ++tc) {
      int tm, tn;
      gemm_tile(p, t, tm, tn);
      const int b = tc & 1;
      if (!mbar_wait(&sb.acc_full[b], (tc >> 1) & 1, abort_flag)) {
        if (lane == 0) raise_abort();
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
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8u * b);
    }
  } else if (warp == 4 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    uint32_t it = 0;  // K steps loaded so far (all tiles)
    const uint64_t pol = l2_policy_evict_last();
    const uint32_t full0 = mapa_shared(smem_addr(&sb.full[0]), 0);
    bool ok = true;
    for (int t = pair; t < p.num_tiles && ok; t += num_pairs) {
      int tm, tn;
      gemm_tile(p, t, tm, tn);
      const int arow = tm * C::kBM + (int)rank * C::kHalf;
      const int brow = tn * C::kBN + (int)rank * C::kHalf;
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const uint32_t s = it % C::kStages;
        if (it >= (uint32_t)C::kStages &&
            !mbar_wait(&sb.empty[s], ((it / C::kStages) - 1) & 1, abort_flag)) {
          raise_abort();
          ok = false;
          break;
        }
        uint8_t *stage = smem + s * C::kStageBytes;
        if (first) mbar_arrive_expect_tx(&sb.full[s], 2 * C::kStageBytes);
        tma_load_2d_pair(stage, &tm_a, full0 + 8u * s, kb * C::kBK, arow, pol);
        tma_load_2d_pair(stage + C::kABytes, &tm_b, full0 + 8u * s, kb * C::kBK, brow, pol);
      }
    }
    if (ok) {
      // The MMAs' last commits on this CTA's stage barriers have landed once
      // each stage's final phase completes: nothing remote is left in flight.
      for (uint32_t s = 0; s < (uint32_t)C::kStages && s < it; ++s) {
        const uint32_t last = it - 1 - ((it - 1 - s) % C::kStages);
        if (!mbar_wait(&sb.empty[s], (last / C::kStages) & 1, abort_flag)) break;
      }
    } else {
      // let copies already issued land before the pair winds down (~100 us)
      for (int i = 0; i < 100; ++i) __nanosleep(1000);
    }
  } else if (warp == 5 && lane == 0 && first) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idesc = idesc_f32acc(true, C::kBM, C::kBN, false, false);
    const uint32_t hi = sdesc_sw128_hi(1024);
    const uint32_t base_lo = sdesc_sw128_lo(smem_addr(smem), 16);
    uint32_t it = 0;
    int tc = 0;
    bool ok = true;
    for (int t = pair; t < p.num_tiles && ok; t += num_pairs, ++tc) {
      const int b = tc & 1;
      // both CTAs' epilogues have drained this accumulator (used two tiles ago)
      if (tc >= 2 && !mbar_wait(&sb.acc_empty[b], ((tc >> 1) - 1) & 1, abort_flag)) {
        raise_abort();
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t d = tmem + b * 256;
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const uint32_t s = it % C::kStages;
        if (!mbar_wait(&sb.full[s], (it / C::kStages) & 1, abort_flag)) {
          raise_abort();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_lo = base_lo + s * (C::kStageBytes >> 4);
        const uint32_t b_lo = a_lo + (C::kABytes >> 4);
        if (kb == 0)
          umma_pair_ss<0>(d, a_lo, b_lo, hi, idesc);
        else
          umma_pair_ss<1>(d, a_lo, b_lo, hi, idesc);
#pragma unroll
        for (int kk = 1; kk < 4; ++kk)  // 16 K-columns = 32 bytes of a swizzled row
          umma_pair_ss<1>(d, a_lo + kk * 2, b_lo + kk * 2, hi, idesc);
        umma_commit_pair(&sb.empty[s], 0x3);  // the stage is free in both CTAs
      }
      if (ok) umma_commit_pair(&sb.acc_full[b], 0x3);
    }
    if (ok) {
      // both epilogues have read the last accumulators: their arrivals on
      // this CTA's barriers have landed
      for (int i = tc >= 2 ? tc - 2 : 0; i < tc; ++i)
        if (!mbar_wait(&sb.acc_empty[i & 1], (i >> 1) & 1, abort_flag)) break;
    }
    umma_commit_pair(&sb.mma_done, 0x3);
  }
  if (warp == 5) {
    if (lane == 0) {
      int never = 0;
      mbar_wait(&sb.mma_done, 0, &never);  // no MMA still writes this CTA's TMEM
    }
    __syncwarp();
  }
  tc_fence_before_sync();
  cluster_sync();
  if (warp == 5) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace tkattn
