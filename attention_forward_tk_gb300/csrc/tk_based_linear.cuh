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
//   [0,128)   S_qk = Q_c K_c^T (fp32), then bf16 A = T(.): keys 0..63 in
//             columns [0,32), keys 64..127 in [64,96) (each key half over its own S)
//   [128,288) Y = A V_ext + phi(Q_c) S_ext in two 80-column buffers, chunk c
//             in buffer c mod 2 (column 64: z), so a chunk's products need not
//             wait for the previous chunk's y to be read
//   [288,448) S^T (lanes: value columns 0..63, 64 = the ones column; fp32)
// Shared memory: a two-stage ring of (V_c, Q_c, K_c), the constant second
// half of V_ext, phi(Q_c), phi(K_c) and S_ext = bf16 copy of S^T, each
// 128 rows x 192 features in three 128-byte-swizzled 64-column chunks.
// Products per chunk (one MMA thread), in issue order:
//   S_qk = Q K^T        M128 N128 K16        (32-byte-swizzled 16-wide rows)
//   S^T += V_ext^T phi(K)  M128 N160 K128  SS (both MN-major; not for a slice's last chunk)
//   Y  = A V_ext        M128 N80  K128  TS   (A from TMEM, V_ext MN-major)
//   Y += phi(Q) S_ext   M128 N80  K160  SS   (both K-major; not for a slice's first chunk)
// The state update runs first, so the copy of the new state starts while
// Y's products run: the copy warps load S^T from tensor memory into
// registers as soon as the update is done, and store it over S_ext once the
// phi(Q) S_ext product that still reads the old copy is done.
// Warps: 0-7 apply T and write y / z (two per TMEM lane quadrant, 64 keys
// and 32 output columns each), 8-11 build phi(K_c), 12-15 phi(Q_c), 16-23
// copy S^T to S_ext in bf16 (two per lane quadrant, 80 features each), 24
// issues MMAs, 25 loads tiles, 26-27 idle (the register split is by
// warpgroup: 72 registers a thread at launch; the two feature warpgroups
// give up 16 each and the two copy warpgroups take them, 2 x (72 + 56 + 88)
// + 72 = 504 a thread per warpgroup, x 128 = the 896 x 72 the block holds).
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
  static constexpr int kThreads = 896;  // 28 warps (the last two idle)
  // Y in two buffers of 80 columns (64 values, z, padding to a multiple of 16)
  static constexpr uint32_t kYCols = 80;
  static constexpr uint32_t kColS = 0, kColY = 128, kColSt = kColY + 2 * kYCols;
};

struct BasedLinShared {
  uint64_t in_full[2], in_empty[2];  // (V, Q, K) of a chunk landed / read     (tx / commit)
  uint64_t s_full;                   // S_qk complete                           (commit)
  uint64_t p_full;                   // bf16 A in TMEM                          (4 warps)
  uint64_t y_full[2], y_free[2];     // Y buffer complete / read by the epilogue (commit / 8 warps)
  uint64_t phik_full, phik_empty;    // phi(K_c) written / read                 (4 warps / commit)
  uint64_t phiq_full, phiq_empty;    // phi(Q_c) written / read                 (4 warps / commit)
  uint64_t st_full, st_read;         // S^T updated / loaded into registers     (commit / 4 warps)
  uint64_t sx_full, sext_free;       // S_ext stored / read by phi(Q) S_ext     (4 warps / commit)
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

__global__ void __launch_bounds__(896, 1)
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
    mbar_init(&sb.p_full, 8);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sb.y_full[b], 1);
      mbar_init(&sb.y_free[b], 8);
    }
    mbar_init(&sb.phik_full, 4);
    mbar_init(&sb.phik_empty, 1);
    mbar_init(&sb.phiq_full, 4);
    mbar_init(&sb.phiq_empty, 1);
    mbar_init(&sb.st_full, 1);
    mbar_init(&sb.st_read, 8);
    mbar_init(&sb.sx_full, 8);
    mbar_init(&sb.sext_free, 1);
    mbar_init(&sb.mma_done, 1);
    sb.abort = 0;
    fence_mbar_init();
  }
  if (warp >= 16 && warp < 20) {
    // V_ext columns 64..127: a ones column (64) and zeros, in the 128-byte
    // swizzle (row r's 16-byte unit u at position u ^ (r mod 8)).
    const int r = threadIdx.x - 512;
#pragma unroll
    for (int pu = 0; pu < 8; ++pu) {
      const uint4 w = ((pu ^ (r & 7)) == 0) ? make_uint4(0x3f80u, 0, 0, 0) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(smem + C::kOffConst + r * 128 + pu * 16) = w;
    }
    fence_proxy_async_smem();
  }
  if (warp == 24) {
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

  if (warp < 8) {
    // ---------------------------------------------------------- A = T(.), y / z
    const int hh = warp >> 2;              // key half (A) and output-column half (y)
    const int r = (warp & 3) * 32 + lane;  // row in the chunk = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint64_t c2 = f2_pack(p.scale, p.scale);
    const float hc = 0.5f * p.scale * p.scale;
    const uint64_t hcc2 = f2_pack(hc, hc);
    const uint64_t one2 = f2_pack(1.f, 1.f);
    // y = Y / z of chunk `ec` (global index `eit`) for its rows < N, and z
    auto epilogue = [&](int ebh, int ec, uint32_t eit) -> bool {
      const uint32_t yb = eit & 1;
      if (!mbar_wait(&sb.y_full[yb], (eit >> 1) & 1, abort_flag)) return false;
      tc_fence_after_sync();
      const uint32_t ycol = C::kColY + yb * C::kYCols;
      uint32_t yv[32], zv[16];
      tmem_ld_32x32b_x32(tmem + lane_off + ycol + 32 * hh, yv);
      tmem_ld_32x32b_x16(tmem + lane_off + ycol + 64, zv);
      tmem_wait_ld();
#pragma unroll
      for (int t = 0; t < 32; ++t) reg_barrier(yv[t]);
      reg_barrier(zv[0]);
      const float z = __uint_as_float(zv[0]);
      const float inv = 1.f / z;
      const int g = ec * 128 + r;
      if (g < p.N) {
        uint4 *dst = reinterpret_cast<uint4 *>(p.y + ((size_t)ebh * p.N + g) * 64 + 32 * hh);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          dst[t] = make_uint4(
              pack_bf16x2(__uint_as_float(yv[8 * t]) * inv, __uint_as_float(yv[8 * t + 1]) * inv),
              pack_bf16x2(__uint_as_float(yv[8 * t + 2]) * inv, __uint_as_float(yv[8 * t + 3]) * inv),
              pack_bf16x2(__uint_as_float(yv[8 * t + 4]) * inv, __uint_as_float(yv[8 * t + 5]) * inv),
              pack_bf16x2(__uint_as_float(yv[8 * t + 6]) * inv, __uint_as_float(yv[8 * t + 7]) * inv));
        if (hh == 0) p.z[(size_t)ebh * p.N + g] = z;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.y_free[yb]);
      return true;
    };
    uint32_t it = 0;
    int pend_bh = -1, pend_c = 0;  // the chunk whose y is still to be written
    uint32_t pend_it = 0;
    bool ok = true;
    for (int bh = blockIdx.x; bh < p.BH && ok; bh += gridDim.x) {
      for (int c = 0; c < p.nc; ++c, ++it) {
        if (!mbar_wait(&sb.s_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int kmax = min(r, p.N - 1 - c * 128);  // last visible key of the chunk
        // Keys 64 hh .. 64 hh + 63: their bf16 pairs go over the first 32 of
        // their own 64 S columns, which only this warp reads; each 32-key
        // quarter's 16 columns are written after the quarter is loaded, over
        // columns already loaded.
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
          uint32_t sv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::kColS + 64 * hh + 32 * q4, sv);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            reg_barrier(sv[t]);
            reg_barrier(sv[t + 1]);
            const uint64_t x = f2_pack(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1]));
            float a0, a1;
            f2_unpack(f2_fma(x, f2_fma(x, hcc2, c2), one2), a0, a1);
            const int kk = 64 * hh + 32 * q4 + t;
            if (kk > kmax) a0 = 0.f;
            if (kk + 1 > kmax) a1 = 0.f;
            pk[t >> 1] = pack_bf16x2(a0, a1);
          }
          tmem_st_32x32b_x16(tmem + lane_off + C::kColS + 64 * hh + 16 * q4, pk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.p_full);
        // the previous chunk's y, while this chunk's products run
        if (pend_bh >= 0 && !epilogue(pend_bh, pend_c, pend_it)) {
          fail();
          ok = false;
          break;
        }
        pend_bh = bh;
        pend_c = c;
        pend_it = it;
      }
    }
    if (ok && pend_bh >= 0 && !epilogue(pend_bh, pend_c, pend_it)) fail();
  } else if (warp < 16) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;\n" ::: "memory");
    // ---------------------------------------------------------- phi(K_c) (8-11), phi(Q_c) (12-15)
    const bool is_k = warp < 12;
    const int r = (warp & 3) * 32 + lane;
    const __nv_bfloat16 *src = is_k ? p.k : p.q;
    uint8_t *panel = is_k ? phik : phiq;
    uint64_t *empty = is_k ? &sb.phik_empty : &sb.phiq_empty;
    uint64_t *full = is_k ? &sb.phik_full : &sb.phiq_full;
    uint32_t it = 0;
    bool ok = true;
    for (int bh = blockIdx.x; bh < p.BH && ok; bh += gridDim.x) {
      for (int c = 0; c < p.nc; ++c, ++it) {
        float x[16];
        based_load_row(src, bh, p.N, c * 128 + r, p.sqrt_scale, x);
        // the previous chunk's product is done with the panel
        if (it > 0 && !mbar_wait(empty, (it - 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        based_feature_row(std::make_integer_sequence<int, 20>{}, x, panel, r);
        fence_proxy_async_smem();  // the generic writes become visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
      }
    }
  } else if (warp < 24) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 88;\n" ::: "memory");
    // ---------------------------------------------------------- S^T -> S_ext (bf16)
    const int fh = (warp - 16) >> 2;       // feature half: features 80 fh .. 80 fh + 79
    const int d = (warp & 3) * 32 + lane;  // value column of S = TMEM lane = S_ext row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // phi(Q) S_ext reads S_ext rows 0 .. 79 (N = 80): the lane quadrant of
    // rows 96 .. 127 keeps the barriers only, and rows 80 .. 95 are not stored
    const bool used = (warp & 3) * 32 < (int)C::kYCols;
    uint32_t cv = 0, dseen = 0;  // copies made; phi(Q) S_ext products of earlier slices
    bool ok = true;
    for (int bh = blockIdx.x; bh < p.BH && ok; bh += gridDim.x) {
      for (int c = 0; c + 1 < p.nc; ++c, ++cv) {
        if (!mbar_wait(&sb.st_full, cv & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint4 w[10];  // this warp's 80 features of the row in bf16, 16-byte units
        if (used) {
#pragma unroll
          for (int f0 = 0; f0 < 80; f0 += 16) {
            uint32_t sv[16];
            tmem_ld_32x32b_x16(tmem + lane_off + C::kColSt + 80 * fh + f0, sv);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              reg_barrier(sv[8 * u]);
              reg_barrier(sv[8 * u + 7]);
              w[(f0 >> 3) + u] = make_uint4(
                  pack_bf16x2(__uint_as_float(sv[8 * u]), __uint_as_float(sv[8 * u + 1])),
                  pack_bf16x2(__uint_as_float(sv[8 * u + 2]), __uint_as_float(sv[8 * u + 3])),
                  pack_bf16x2(__uint_as_float(sv[8 * u + 4]), __uint_as_float(sv[8 * u + 5])),
                  pack_bf16x2(__uint_as_float(sv[8 * u + 6]), __uint_as_float(sv[8 * u + 7])));
            }
          }
        }
        // S^T is in registers: the next update may accumulate into it
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.st_read);
        // S_ext may be overwritten once every phi(Q) S_ext product issued
        // before this copy is done: this slice's first c, and earlier slices'
        const uint32_t D = dseen + (uint32_t)c;
        if (D > 0 && !mbar_wait(&sb.sext_free, (D - 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        if (d < (int)C::kYCols) {
#pragma unroll
          for (int u = 0; u < 10; ++u) {
            const int U = 10 * fh + u;
            *reinterpret_cast<uint4 *>(sext + (U >> 3) * C::kChunkB + d * 128 +
                                       (((U & 7) ^ (d & 7)) << 4)) = w[u];
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.sx_full);
      }
      dseen += (uint32_t)(p.nc - 1);
    }
  } else if (warp == 24 && lane == 0) {
    // ---------------------------------------------------------- MMA issue
    constexpr uint32_t idS = idesc_f32acc(true, 128, 128, false, false);   // Q K^T
    constexpr uint32_t idA = idesc_f32acc(true, 128, C::kYCols, false, true);   // A V_ext
    constexpr uint32_t idF = idesc_f32acc(true, 128, C::kYCols, false, false);  // phi(Q) S_ext
    constexpr uint32_t idU = idesc_f32acc(true, 128, C::kFeatPad, true, true);  // V_ext^T phi(K)
    const uint32_t dhi = sdesc_sw128_hi(1024);
    const uint32_t phiq_lo = sdesc_sw128_lo(smem_addr(phiq), 16);
    const uint32_t sext_lo = sdesc_sw128_lo(smem_addr(sext), 16);
    const uint32_t phik_lo = sdesc_sw128_lo(smem_addr(phik), C::kChunkB);
    uint32_t it = 0, cv = 0;
    uint32_t ups = 0, upw = 0;  // state updates issued; st_read phases waited
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
        // S^T (+)= V_ext^T phi(K_c), before a slice's last chunk, once phi(K_c)
        // is written and the copy warps hold the previous state
        if (!mbar_wait(&sb.phik_full, it & 1, abort_flag) ||
            (c + 1 < p.nc && ups > upw && !mbar_wait(&sb.st_read, upw & 1, abort_flag))) {
          fail();
          ok = false;
          break;
        }
        if (c + 1 < p.nc && ups > upw) ++upw;
        tc_fence_after_sync();
        if (c + 1 < p.nc) {
          // 16 keys (2048 B of each operand) per MMA
          if (c > 0)
            umma_ss_w<1>(tmem + C::kColSt, v_lo, phik_lo, dhi, idU);
          else
            umma_ss_w<0>(tmem + C::kColSt, v_lo, phik_lo, dhi, idU);
#pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            umma_ss_w<1>(tmem + C::kColSt, v_lo + kk * (2048 >> 4), phik_lo + kk * (2048 >> 4), dhi,
                         idU);
          umma_commit(&sb.st_full);
          ++ups;
        }
        umma_commit(&sb.phik_empty);
        // Y_b = A V_ext (b = chunk mod 2) once A is written and the y of the
        // chunk two back, the buffer's previous use, has been read
        const uint32_t tY = tmem + C::kColY + (it & 1) * C::kYCols;
        if ((it >= 2 && !mbar_wait(&sb.y_free[it & 1], ((it >> 1) - 1) & 1, abort_flag)) ||
            !mbar_wait(&sb.p_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_grad<2>(tY, tmem + C::kColS, v_lo, dhi, idA, 0u);  // A in two column halves
        // Y += phi(Q_c) S_{c-1}, once phi(Q_c) and the state copy are in
        if (!mbar_wait(&sb.phiq_full, it & 1, abort_flag) ||
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
            umma_ss_w<1>(tY, phiq_lo + off, sext_lo + off, dhi, idF);
          }
          umma_commit(&sb.sext_free);
        }
        umma_commit(&sb.y_full[it & 1]);
        umma_commit(&sb.phiq_empty);
        umma_commit(&sb.in_empty[it & 1]);
      }
    }
    umma_commit(&sb.mma_done);
    int never = 0;
    mbar_wait(&sb.mma_done, 0, &never);
  } else if (warp == 25 && lane == 0) {
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
  if (warp == 24) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace tkattn
