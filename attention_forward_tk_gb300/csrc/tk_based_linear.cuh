// tk_based_linear.cuh -- Based linear attention, causal, through the
// linear-time chunked algorithm (GB300, sm_103a).
//
// The same output as tk_based_fwd's causal form,
//   y_i = sum_{j<=i} T(s_ij) v_j / z_i,   z_i = sum_{j<=i} T(s_ij),
//   s_ij = scale q_i.k_j,   T(s) = 1 + s + s^2 / 2,
// computed in chunks of 128 positions instead of over all (query, key)
// pairs.  T(s_ij) is the inner product of feature maps phi(q_i).phi(k_j):
//   phi(x) = [1, x', x'_a^2 / sqrt 2 (16 terms), x'_a x'_b for a < b (120)],
//   x' = sqrt(scale) x,
// 153 features, the distinct terms of the second-order Taylor map [1, x,
// vec(x x^T)/sqrt 2] (a pair a < b carries the weight of both its ordered
// terms), padded to 160.  This is the linear-time form the pages' Based
// figure refers to (the Based paragraph of the ThunderKittens news write-up,
// 88811315.cn post 77732; the performance section of es.news.hada.io topic
// 14783).  For chunk c, with V extended by a ones column so that every
// product also carries z:
//   y_c = [T(scale Q_c K_c^T), causal within the chunk] V_c + phi(Q_c) S_{c-1}
//   S_c = S_{c-1} + phi(K_c)^T V_c,          S_{-1} = 0.
//
// One CTA per slice, its chunks in order.  Tensor memory:
//   [0,128)   S_qk = Q_c K_c^T (fp32), then bf16 A = T(.) over its first 64 columns
//   [128,256) Y = A V_ext + phi(Q_c) S_ext (column 64: z)
//   [256,416) S^T (lanes: value columns 0..63, 64 = the ones column; fp32)
// Shared memory: a two-stage ring of (V_c, Q_c, K_c), the constant second
// half of V_ext, phi(Q_c), phi(K_c) and S_ext = bf16 copy of S^T, each
// 128 rows x 192 features in three 128-byte-swizzled 64-column chunks.
// Products per chunk (one MMA thread):
//   S_qk = Q K^T        M128 N128 K16        (32-byte-swizzled 16-wide rows)
//   Y  = A V_ext        M128 N128 K128  TS   (A from TMEM, V_ext MN-major)
//   Y += phi(Q) S_ext   M128 N128 K160  SS   (both K-major)
//   S^T += V_ext^T phi(K)  M128 N160 K128  SS (both MN-major)
// Warps: 0-3 apply T and write y / z, 4-7 build phi(Q_c) and phi(K_c),
// 8-11 copy S^T to S_ext in bf16, 12 issues MMAs, 13 loads tiles.
//
// Every wait is bounded; a wait that runs out raises the abort flag and the
// device error word, as in the attention kernels.
#pragma once

#include <utility>

#include "tk_based.cuh"

namespace tkattn {

struct BasedLinParams {
  const __nv_bfloat16 *q, *k;  // [BH, N, 16] (the feature warps read rows directly)
  __nv_bfloat16 *y;            // [BH, N, 64]
  float *z;                    // [BH, N]
  int *err;
  int BH, N, nc;               // nc = ceil(N / 128) chunks per slice
  float scale, sqrt_scale;
};

struct BasedLinCfg {
  static constexpr int kFeat = 153, kFeatPad = 160;  // features; MMA extent
  static constexpr int kChunkB = 128 * 128;           // one 64-column chunk: 128 rows x 128 B
  static constexpr int kPanelBytes = 3 * kChunkB;     // 128 rows x 192 bf16 features
  static constexpr int kVBytes = kChunkB;             // V_c: 128 keys x 64 values
  static constexpr int kQKBytes = 128 * 16 * 2;       // Q_c or K_c: 128 rows x 32 B
  static constexpr int kStageBytes = kVBytes + 2 * kQKBytes;  // 24 KB: V, Q, K
  static constexpr int kOffConst = 2 * kStageBytes;   // V_ext columns 64..127
  static constexpr int kOffPhiQ = kOffConst + kChunkB;
  static constexpr int kOffPhiK = kOffPhiQ + kPanelBytes;
  static constexpr int kOffSext = kOffPhiK + kPanelBytes;
  static constexpr int kSmemBytes = kOffSext + kPanelBytes;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static constexpr int kThreads = 448;
  static constexpr uint32_t kColS = 0, kColY = 128, kColSt = 256;
};

struct BasedLinShared {
  uint64_t in_full[2], in_empty[2];  // (V, Q, K) of a chunk landed / read     (tx / commit)
  uint64_t s_full;                   // S_qk complete                           (commit)
  uint64_t p_full;                   // bf16 A in TMEM                          (4 warps)
  uint64_t y_full, y_free;           // Y complete / read by the epilogue       (commit / 4 warps)
  uint64_t phi_full, phi_empty;      // phi(Q_c), phi(K_c) written / read       (4 warps / commit)
  uint64_t st_full, sx_full;         // S^T updated / copied to S_ext           (commit / 4 warps)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// The a < b pairs in order (0,1), (0,2), ..., (0,15), (1,2), ...: pair r.
__host__ __device__ constexpr int based_pair_a(int r) {
  int a = 0;
  while (r >= 15 - a) {
    r -= 15 - a;
    ++a;
  }
  return a;
}
__host__ __device__ constexpr int based_pair_b(int r) {
  int a = 0;
  while (r >= 15 - a) {
    r -= 15 - a;
    ++a;
  }
  return a + 1 + r;
}

// Feature F of phi(x') for x'[16].
template <int F>
__device__ __forceinline__ float based_feature(const float (&x)[16]) {
  if constexpr (F == 0) {
    return 1.f;
  } else if constexpr (F <= 16) {
    return x[F - 1];
  } else if constexpr (F <= 32) {
    return x[F - 17] * x[F - 17] * 0.70710678118654752f;
  } else if constexpr (F < BasedLinCfg::kFeat) {
    constexpr int a = based_pair_a(F - 33), b = based_pair_b(F - 33);
    return x[a] * x[b];
  } else {
    return 0.f;
  }
}

// Row r of a feature panel: 16-byte unit U (features 8U .. 8U+7) goes to
// chunk U / 8, swizzled position (U mod 8) ^ (r mod 8).
template <int U>
__device__ __forceinline__ void based_feature_unit(const float (&x)[16], uint8_t *panel, int r) {
  uint4 w;
  w.x = pack_bf16x2(based_feature<8 * U + 0>(x), based_feature<8 * U + 1>(x));
  w.y = pack_bf16x2(based_feature<8 * U + 2>(x), based_feature<8 * U + 3>(x));
  w.z = pack_bf16x2(based_feature<8 * U + 4>(x), based_feature<8 * U + 5>(x));
  w.w = pack_bf16x2(based_feature<8 * U + 6>(x), based_feature<8 * U + 7>(x));
  *reinterpret_cast<uint4 *>(panel + (U >> 3) * BasedLinCfg::kChunkB + r * 128 +
                             (((U & 7) ^ (r & 7)) << 4)) = w;
}

template <int... U>
__device__ __forceinline__ void based_feature_row(std::integer_sequence<int, U...>,
                                                  const float (&x)[16], uint8_t *panel, int r) {
  (based_feature_unit<U>(x, panel, r), ...);
}

// x' = sqrt(scale) x for row g of a [BH, N, 16] tensor (zeros past N).
__device__ __forceinline__ void based_load_row(const __nv_bfloat16 *t, int bh, int N, int g,
                                               float sq, float (&x)[16]) {
  uint4 a = make_uint4(0, 0, 0, 0), b = a;
  if (g < N) {
    const uint4 *src = reinterpret_cast<const uint4 *>(t + ((size_t)bh * N + g) * 16);
    a = src[0];
    b = src[1];
  }
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16) * sq;
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u) * sq;
  }
}

__global__ void __launch_bounds__(448, 1)
    tk_based_linear_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const BasedLinParams p) {
  using C = BasedLinCfg;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BasedLinShared sb;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *phiq = smem + C::kOffPhiQ, *phik = smem + C::kOffPhiK, *sext = smem + C::kOffSext;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = &sb.abort;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sb.in_full[s], 1);
      mbar_init(&sb.in_empty[s], 1);
    }
    mbar_init(&sb.s_full, 1);
    mbar_init(&sb.p_full, 4);
    mbar_init(&sb.y_full, 1);
    mbar_init(&sb.y_free, 4);
    mbar_init(&sb.phi_full, 4);
    mbar_init(&sb.phi_empty, 1);
    mbar_init(&sb.st_full, 1);
    mbar_init(&sb.sx_full, 4);
    mbar_init(&sb.mma_done, 1);
    sb.abort = 0;
    fence_mbar_init();
  }
  if (warp >= 8 && warp < 12) {
    // V_ext columns 64..127: a ones column (64) and zeros, in the 128-byte
    // swizzle (row r's 16-byte unit u at position u ^ (r mod 8)).
    const int r = threadIdx.x - 256;
#pragma unroll
    for (int pu = 0; pu < 8; ++pu) {
      const uint4 w = ((pu ^ (r & 7)) == 0) ? make_uint4(0x3f80u, 0, 0, 0) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(smem + C::kOffConst + r * 128 + pu * 16) = w;
    }
    fence_proxy_async_smem();
  }
  if (warp == 12) {
    tmem_alloc(&sb.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sb.tmem_base;
  auto fail = [&]() {
    sb.abort = 1;
    atomicCAS(p.err, 0, kDevErrTimeout);
  };
  auto stage_base = [&](uint32_t it) { return smem + (it & 1) * C::kStageBytes; };

  if (warp < 4) {
    // ---------------------------------------------------------- A = T(.), y / z
    const int r = warp * 32 + lane;  // row in the chunk = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint64_t c2 = f2_pack(p.scale, p.scale);
    const float hc = 0.5f * p.scale * p.scale;
    const uint64_t hcc2 = f2_pack(hc, hc);
    const uint64_t one2 = f2_pack(1.f, 1.f);
    uint32_t it = 0;
    bool ok = true;
    for (int bh = blockIdx.x; bh < p.BH && ok; bh += gridDim.x) {
      for (int c = 0; c < p.nc; ++c, ++it) {
        if (!mbar_wait(&sb.s_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int g = c * 128 + r;              // this row's position
        const int kmax = min(r, p.N - 1 - c * 128);  // last visible key of the chunk
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t sv[64];
          tmem_ld_32x32b_x32(tmem + lane_off + C::kColS + 64 * hf,
                             *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
          tmem_ld_32x32b_x32(tmem + lane_off + C::kColS + 64 * hf + 32,
                             *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
          tmem_wait_ld();
          uint32_t pk[32];
#pragma unroll
          for (int t = 0; t < 64; t += 2) {
            reg_barrier(sv[t]);
            reg_barrier(sv[t + 1]);
            const uint64_t x = f2_pack(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1]));
            float a0, a1;
            f2_unpack(f2_fma(x, f2_fma(x, hcc2, c2), one2), a0, a1);
            const int kk = 64 * hf + t;
            if (kk > kmax) a0 = 0.f;
            if (kk + 1 > kmax) a1 = 0.f;
            pk[t >> 1] = pack_bf16x2(a0, a1);
          }
          tmem_st_32x32b_x32(tmem + lane_off + C::kColS + 32 * hf, pk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.p_full);
        // ---- y = Y / z for this chunk's rows (< N), z
        if (!mbar_wait(&sb.y_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t yv[64], zv[16];
        tmem_ld_32x32b_x32(tmem + lane_off + C::kColY, *reinterpret_cast<uint32_t(*)[32]>(&yv[0]));
        tmem_ld_32x32b_x32(tmem + lane_off + C::kColY + 32,
                           *reinterpret_cast<uint32_t(*)[32]>(&yv[32]));
        tmem_ld_32x32b_x16(tmem + lane_off + C::kColY + 64, zv);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 64; ++t) reg_barrier(yv[t]);
        reg_barrier(zv[0]);
        const float z = __uint_as_float(zv[0]);
        const float inv = 1.f / z;
        if (g < p.N) {
          uint4 *dst = reinterpret_cast<uint4 *>(p.y + ((size_t)bh * p.N + g) * 64);
#pragma unroll
          for (int t = 0; t < 8; ++t)
            dst[t] = make_uint4(
                pack_bf16x2(__uint_as_float(yv[8 * t]) * inv, __uint_as_float(yv[8 * t + 1]) * inv),
                pack_bf16x2(__uint_as_float(yv[8 * t + 2]) * inv, __uint_as_float(yv[8 * t + 3]) * inv),
                pack_bf16x2(__uint_as_float(yv[8 * t + 4]) * inv, __uint_as_float(yv[8 * t + 5]) * inv),
                pack_bf16x2(__uint_as_float(yv[8 * t + 6]) * inv, __uint_as_float(yv[8 * t + 7]) * inv));
          p.z[(size_t)bh * p.N + g] = z;
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.y_free);
      }
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------- phi(Q_c), phi(K_c)
    const int r = (warp - 4) * 32 + lane;
    uint32_t it = 0;
    bool ok = true;
    for (int bh = blockIdx.x; bh < p.BH && ok; bh += gridDim.x) {
      for (int c = 0; c < p.nc; ++c, ++it) {
        float x[16];
        based_load_row(p.q, bh, p.N, c * 128 + r, p.sqrt_scale, x);
        // the previous chunk's products are done with both panels
        if (it > 0 && !mbar_wait(&sb.phi_empty, (it - 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        based_feature_row(std::make_integer_sequence<int, 20>{}, x, phiq, r);
        based_load_row(p.k, bh, p.N, c * 128 + r, p.sqrt_scale, x);
        based_feature_row(std::make_integer_sequence<int, 20>{}, x, phik, r);
        fence_proxy_async_smem();  // the generic writes become visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.phi_full);
      }
    }
  } else if (warp < 12) {
    // ---------------------------------------------------------- S^T -> S_ext (bf16)
    const int d = (warp - 8) * 32 + lane;  // value column of S = TMEM lane = S_ext row
    const uint32_t lane_off = (uint32_t)((warp - 8) * 32) << 16;
    uint32_t cv = 0;
    bool ok = true;
    for (int bh = blockIdx.x; bh < p.BH && ok; bh += gridDim.x) {
      for (int c = 0; c + 1 < p.nc; ++c, ++cv) {
        if (!mbar_wait(&sb.st_full, cv & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll 1
        for (int f0 = 0; f0 < C::kFeatPad; f0 += 32) {
          uint32_t sv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::kColSt + f0, sv);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 4; ++u) {  // 16-byte units of 8 features
            const int U = (f0 >> 3) + u;
            reg_barrier(sv[8 * u]);
            reg_barrier(sv[8 * u + 7]);
            const uint4 w = make_uint4(
                pack_bf16x2(__uint_as_float(sv[8 * u]), __uint_as_float(sv[8 * u + 1])),
                pack_bf16x2(__uint_as_float(sv[8 * u + 2]), __uint_as_float(sv[8 * u + 3])),
                pack_bf16x2(__uint_as_float(sv[8 * u + 4]), __uint_as_float(sv[8 * u + 5])),
                pack_bf16x2(__uint_as_float(sv[8 * u + 6]), __uint_as_float(sv[8 * u + 7])));
            *reinterpret_cast<uint4 *>(sext + (U >> 3) * C::kChunkB + d * 128 +
                                       (((U & 7) ^ (d & 7)) << 4)) = w;
          }
        }
        tc_fence_before_sync();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.sx_full);
      }
    }
  } else if (warp == 12 && lane == 0) {
    // ---------------------------------------------------------- MMA issue
    constexpr uint32_t idS = idesc_f32acc(true, 128, 128, false, false);   // Q K^T
    constexpr uint32_t idA = idesc_f32acc(true, 128, 128, false, true);    // A V_ext
    constexpr uint32_t idF = idesc_f32acc(true, 128, 128, false, false);   // phi(Q) S_ext
    constexpr uint32_t idU = idesc_f32acc(true, 128, C::kFeatPad, true, true);  // V_ext^T phi(K)
    const uint32_t dhi = sdesc_sw128_hi(1024);
    const uint32_t phiq_lo = sdesc_sw128_lo(smem_addr(phiq), 16);
    const uint32_t sext_lo = sdesc_sw128_lo(smem_addr(sext), 16);
    const uint32_t phik_lo = sdesc_sw128_lo(smem_addr(phik), C::kChunkB);
    uint32_t it = 0, cv = 0;
    bool ok = true;
    for (int bh = blockIdx.x; bh < p.BH && ok; bh += gridDim.x) {
      for (int c = 0; c < p.nc; ++c, ++it) {
        uint8_t *st = stage_base(it);
        // V_ext of this stage: its 64 values, then the constant block, LBO apart
        const uint32_t v_lo = sdesc_sw128_lo(smem_addr(st), (uint32_t)(smem + C::kOffConst - st));
        if (!mbar_wait(&sb.in_full[it & 1], (it >> 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        umma_bf16_ss(tmem + C::kColS, sdesc_sw32(smem_addr(st + C::kVBytes)),
                     sdesc_sw32(smem_addr(st + C::kVBytes + C::kQKBytes)), idS, 0);
        umma_commit(&sb.s_full);
        // Y = A V_ext once the previous chunk's y has been read and A written
        if ((it > 0 && !mbar_wait(&sb.y_free, (it - 1) & 1, abort_flag)) ||
            !mbar_wait(&sb.p_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_grad<1>(tmem + C::kColY, tmem + C::kColS, v_lo, dhi, idA, 0u);
        // Y += phi(Q_c) S_{c-1}, once the features and the state copy are in
        if (!mbar_wait(&sb.phi_full, it & 1, abort_flag) ||
            (c > 0 && !mbar_wait(&sb.sx_full, cv & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (c > 0) {
          ++cv;
#pragma unroll
          for (int kk = 0; kk < C::kFeatPad / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * C::kChunkB + (kk & 3) * 32) >> 4;
            umma_ss_w<1>(tmem + C::kColY, phiq_lo + off, sext_lo + off, dhi, idF);
          }
        }
        umma_commit(&sb.y_full);
        if (c + 1 < p.nc) {
          // S^T (+)= V_ext^T phi(K_c): 16 keys (2048 B of each operand) per MMA
          if (c > 0)
            umma_ss_w<1>(tmem + C::kColSt, v_lo, phik_lo, dhi, idU);
          else
            umma_ss_w<0>(tmem + C::kColSt, v_lo, phik_lo, dhi, idU);
#pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            umma_ss_w<1>(tmem + C::kColSt, v_lo + kk * (2048 >> 4), phik_lo + kk * (2048 >> 4), dhi,
                         idU);
          umma_commit(&sb.st_full);
        }
        umma_commit(&sb.phi_empty);
        umma_commit(&sb.in_empty[it & 1]);
      }
    }
    umma_commit(&sb.mma_done);
    int never = 0;
    mbar_wait(&sb.mma_done, 0, &never);
  } else if (warp == 13 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    uint32_t it = 0;
    bool ok = true;
    for (int bh = blockIdx.x; bh < p.BH && ok; bh += gridDim.x) {
      for (int c = 0; c < p.nc; ++c, ++it) {
        if (it >= 2 && !mbar_wait(&sb.in_empty[it & 1], ((it >> 1) - 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        uint8_t *st = stage_base(it);
        mbar_arrive_expect_tx(&sb.in_full[it & 1], C::kStageBytes);
        tma_load_3d(st, &tm_v, &sb.in_full[it & 1], 0, c * 128, bh);
        tma_load_3d(st + C::kVBytes, &tm_q, &sb.in_full[it & 1], 0, c * 128, bh);
        tma_load_3d(st + C::kVBytes + C::kQKBytes, &tm_k, &sb.in_full[it & 1], 0, c * 128, bh);
      }
    }
    if (ok) {
      // the last loads of both stages were consumed (their in_empty commits landed)
      for (uint32_t s = 0; s < 2 && s < it; ++s) {
        const uint32_t last = it - 1 - ((it - 1 - s) & 1);
        if (!mbar_wait(&sb.in_empty[s], (last >> 1) & 1, abort_flag)) break;
      }
    } else {
      for (int i = 0; i < 200; ++i) __nanosleep(1000);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace tkattn
