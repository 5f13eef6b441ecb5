// tk_based.cuh -- Based linear attention, forward, on GB300 (sm_103a).
//
//   y_i = sum_{j visible} T(s_ij) v_j / z_i,   z_i = sum_{j visible} T(s_ij),
//   s_ij = scale q_i.k_j,   T(s) = 1 + s + s^2 / 2
//
// T is the second-order Taylor expansion of exp, i.e. the inner product of
// the Based feature maps phi(x) = [1, x, vec(x x^T)/sqrt(2)].  The pages name
// a Based linear-attention kernel and its speed (215 TFLOPs on H100: the
// Chinese news write-up, 88811315.cn post 77732; the Spanish page,
// es.news.hada.io topic 14783) without defining it; this is the published
// Based form with feature dimension 16 and value dimension 64.
//
// The kernel evaluates the causal sum tile by tile on the tensor cores, the
// attention kernel's structure with T in place of the exponential: no
// running maximum, since T > 0 needs no stabilising shift.  One unit = (slice,
// 128-query tile); K/V tiles stream through a ring.  Per key tile:
//   S = Q K^T       one M128 N128 K16 MMA (32-byte-swizzled 16-wide rows)
//   A = T(scale S)  sixteen elementwise warps (four per TMEM lane quadrant,
//                   32 key columns each), bf16 into S's TMEM columns
//   O += A V        TS MMAs (A from TMEM, V MN-major)
// S has three TMEM buffers, so the next tiles' S run while the warps work.
#pragma once

#include "tk_attn_bwd.cuh"

namespace tkattn {

struct BasedParams {
  __nv_bfloat16 *y;  // [BH, N, 64]
  float *z;          // [BH, N] normaliser
  int *err;
  int BH, N, nt, num_units;
  int head_group;  // causal order: slices per L2-sized section
  float scale;
};

struct BasedCfg {
  static constexpr int kDf = 16, kDv = 64;
  static constexpr int kQKBytes = 128 * kDf * 2;  // 4 KB: 128 rows x 32 B
  static constexpr int kVBytes = 128 * kDv * 2;   // 16 KB
  static constexpr int kStageBytes = kQKBytes + kVBytes;
  static constexpr int kStages = 8;
  static constexpr int kSmemAlloc = kQKBytes + kStages * kStageBytes + 1024;
  static constexpr int kThreads = 576;  // 16 elementwise warps, producer, MMA
  static constexpr int kSBufs = 3;  // S buffers in TMEM, 128 columns each
  static constexpr uint32_t kColO = 128 * kSBufs;
};

struct BasedShared {
  uint64_t fix_full, fix_empty;  // the unit's Q tile landed / released
  uint64_t kv_full[BasedCfg::kStages], kv_empty[BasedCfg::kStages];
  uint64_t s_full[BasedCfg::kSBufs];  // S into buffer b complete  (commit)
  uint64_t p_full[BasedCfg::kSBufs];  // bf16 A in buffer b        (16 warps)
  uint64_t lsum_bar;             // partial row sums written       (16 warps)
  uint64_t acc_full, acc_empty;  // O of a unit done / read        (commit / 16 warps)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  float lsum[2][4][128];         // [unit parity][column quarter][row] partial row sums
};

// Shared-memory descriptor, K-major, 32-byte swizzle: 8-row groups of 32-byte
// rows, 256 B apart; a 16-element K extent fits one swizzle row, so the
// leading offset is unused.
__device__ __forceinline__ uint64_t sdesc_sw32(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(256 >> 4) << 32) |
         (1ull << 46) | (6ull << 61);
}

// Causal: slices in sections of head_group whose K and V fit in about half
// the L2, longest query tiles first within a section (tile i meets i + 1 key
// tiles), so the CTAs running at one time share K/V out of L2.
template <bool kCausal>
__device__ __forceinline__ void based_unit(const BasedParams &p, int u, int &bh, int &i, int &n) {
  if (kCausal) {
    const int per = p.head_group * p.nt;
    const int g = u / per;
    const int r = u - g * per;
    const int hg = min(p.head_group, p.BH - g * p.head_group);
    const int t = r / hg;
    bh = g * p.head_group + (r - t * hg);
    i = p.nt - 1 - t;
    n = i + 1;
  } else {
    bh = u / p.nt;
    i = u - bh * p.nt;
    n = p.nt;
  }
}

template <bool kCausal>
__global__ void __launch_bounds__(576, 1)
    tk_based_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const BasedParams p) {
  using C = BasedCfg;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BasedShared sb;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem, *ring = smem + C::kQKBytes;  // stage: K (4 KB) then V (16 KB)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = &sb.abort;
  if (threadIdx.x == 0) {
    mbar_init(&sb.fix_full, 1);
    mbar_init(&sb.fix_empty, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&sb.kv_full[s], 1);
      mbar_init(&sb.kv_empty[s], 1);
    }
    for (int b = 0; b < C::kSBufs; ++b) {
      mbar_init(&sb.s_full[b], 1);
      mbar_init(&sb.p_full[b], 16);
    }
    mbar_init(&sb.lsum_bar, 16);
    mbar_init(&sb.acc_full, 1);
    mbar_init(&sb.acc_empty, 16);
    mbar_init(&sb.mma_done, 1);
    sb.abort = 0;
    fence_mbar_init();
  }
  if (warp == 17) {
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
  // Step t uses S buffer t % 3, with its own s_full and p_full barriers: the
  // next steps' S are already in flight when a step's A is published, so one
  // barrier per buffer keeps every barrier at most one phase ahead of its
  // waiter (a parity wait cannot tell phase t from phase t + 2).
  constexpr uint32_t NB = C::kSBufs;
  auto s_col = [](uint32_t step) { return 128u * (step % NB); };

  if (warp < 16) {
    // ---------------------------------------------------------- elementwise
    const int qd = warp & 3, h = warp >> 2;  // lane quadrant, column quarter
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const int r = qd * 32 + lane;  // query row within the tile = TMEM lane
    // T(scale x) = 1 + x (c + x c^2 / 2), c = scale: two packed FMAs per pair
    const uint64_t c2 = f2_pack(p.scale, p.scale);
    const float hc = 0.5f * p.scale * p.scale;
    const uint64_t hcc2 = f2_pack(hc, hc);
    const uint64_t one2 = f2_pack(1.f, 1.f);
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++uc) {
      int bh, i, n;
      based_unit<kCausal>(p, u, bh, i, n);
      const int qi = i * 128 + r;
      uint64_t la = f2_pack(0.f, 0.f), lb = la;
#pragma unroll 1
      for (int j = 0; j < n; ++j, ++it) {
        if (!mbar_wait(&sb.s_full[it % NB], (it / NB) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tS = tmem + lane_off + s_col(it);
        const bool edge = (kCausal && j == i) || (j * 128 + 128 > p.N);
        {
          const int col0 = 32 * h;
          uint32_t sv[32];
          tmem_ld_32x32b_x32(tS + col0, sv);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 32; t += 4) {
            reg_barrier(sv[t]);
            reg_barrier(sv[t + 1]);
            reg_barrier(sv[t + 2]);
            reg_barrier(sv[t + 3]);
            const uint64_t x0 = f2_pack(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1]));
            const uint64_t x1 = f2_pack(__uint_as_float(sv[t + 2]), __uint_as_float(sv[t + 3]));
            uint64_t t0 = f2_fma(x0, f2_fma(x0, hcc2, c2), one2);
            uint64_t t1 = f2_fma(x1, f2_fma(x1, hcc2, c2), one2);
            if (edge) {  // the diagonal tile or a ragged tail only
              float a0, a1, a2, a3;
              f2_unpack(t0, a0, a1);
              f2_unpack(t1, a2, a3);
              const int kj = j * 128 + col0 + t;
              if ((kCausal && kj > qi) || kj >= p.N) a0 = 0.f;
              if ((kCausal && kj + 1 > qi) || kj + 1 >= p.N) a1 = 0.f;
              if ((kCausal && kj + 2 > qi) || kj + 2 >= p.N) a2 = 0.f;
              if ((kCausal && kj + 3 > qi) || kj + 3 >= p.N) a3 = 0.f;
              t0 = f2_pack(a0, a1);
              t1 = f2_pack(a2, a3);
            }
            la = f2_add(la, t0);
            lb = f2_add(lb, t1);
            float a0, a1, a2, a3;
            f2_unpack(t0, a0, a1);
            f2_unpack(t1, a2, a3);
            pk[t >> 1] = pack_bf16x2(a0, a1);
            pk[(t >> 1) + 1] = pack_bf16x2(a2, a3);
          }
          tmem_st_32x32b_x16(tS + 32 * h, pk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.p_full[it % NB]);
      }
      if (!ok) break;
      // ---- epilogue: y = O / z for this query tile (rows < N), z
      float l0, l1, l2, l3;
      f2_unpack(la, l0, l1);
      f2_unpack(lb, l2, l3);
      sb.lsum[uc & 1][h][r] = (l0 + l1) + (l2 + l3);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.lsum_bar);
      if (!mbar_wait(&sb.lsum_bar, uc & 1, abort_flag)) {
        fail();
        break;
      }
      const float l = (sb.lsum[uc & 1][0][r] + sb.lsum[uc & 1][1][r]) +
                      (sb.lsum[uc & 1][2][r] + sb.lsum[uc & 1][3][r]);
      if (!mbar_wait(&sb.acc_full, uc & 1, abort_flag)) {
        fail();
        break;
      }
      tc_fence_after_sync();
      // quarter h of the 64 output columns: 16 each
      uint32_t rv[16];
      tmem_ld_32x32b_x16(tmem + lane_off + C::kColO + 16 * h, rv);
      tmem_wait_ld();
      const float inv = 1.f / l;
      uint32_t pk[8];
#pragma unroll
      for (int t = 0; t < 16; t += 2) {
        reg_barrier(rv[t]);
        reg_barrier(rv[t + 1]);
        pk[t >> 1] = pack_bf16x2(__uint_as_float(rv[t]) * inv, __uint_as_float(rv[t + 1]) * inv);
      }
      if (qi < p.N) {
        __nv_bfloat16 *dst = p.y + ((size_t)bh * p.N + qi) * C::kDv + 16 * h;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        if (h == 0) p.z[(size_t)bh * p.N + qi] = l;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.acc_empty);
    }
  } else if (warp == 16 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++uc) {
      int bh, i, n;
      based_unit<kCausal>(p, u, bh, i, n);
      if (uc > 0 && !mbar_wait(&sb.fix_empty, (uc - 1) & 1, abort_flag)) {
        fail();
        break;
      }
      mbar_arrive_expect_tx(&sb.fix_full, C::kQKBytes);
      tma_load_3d(sQ, &tm_q, &sb.fix_full, 0, i * 128, bh);
      for (int j = 0; j < n; ++j, ++it) {
        const uint32_t s = it % S;
        if (it >= (uint32_t)S && !mbar_wait(&sb.kv_empty[s], ((it / S) - 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        uint8_t *stage = ring + s * C::kStageBytes;
        mbar_arrive_expect_tx(&sb.kv_full[s], C::kStageBytes);
        tma_load_3d(stage, &tm_k, &sb.kv_full[s], 0, j * 128, bh);
        tma_load_3d(stage + C::kQKBytes, &tm_v, &sb.kv_full[s], 0, j * 128, bh);
      }
    }
    for (int i = 0; i < 200 && !ok; ++i) __nanosleep(1000);
  } else if (warp == 17 && lane == 0) {
    // ---------------------------------------------------------- MMA issue
    constexpr uint32_t idS = idesc_f32acc(true, 128, 128, false, false);
    constexpr uint32_t idO = idesc_f32acc(true, 128, C::kDv, false, true);
    const uint32_t dhi = sdesc_sw128_hi(1024);
    const uint64_t qdesc = sdesc_sw32(smem_addr(sQ));
    auto k_addr = [&](uint32_t t) { return smem_addr(ring + (t % S) * C::kStageBytes); };
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++uc) {
      int bh, i, n;
      based_unit<kCausal>(p, u, bh, i, n);
      // S of the first steps, one per buffer
      if (!mbar_wait(&sb.fix_full, uc & 1, abort_flag)) {
        fail();
        break;
      }
      for (int j = 0; j < (int)NB && j < n && ok; ++j) {
        if (!mbar_wait(&sb.kv_full[(it + j) % S], ((it + j) / S) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        umma_bf16_ss(tmem + s_col(it + j), qdesc, sdesc_sw32(k_addr(it + j)), idS, 0);
        umma_commit(&sb.s_full[(it + j) % NB]);
        if (j == n - 1) umma_commit(&sb.fix_empty);  // Q is read by the S products only
      }
      if (!ok) break;
      if (uc > 0 && !mbar_wait(&sb.acc_empty, (uc - 1) & 1, abort_flag)) {
        fail();
        break;
      }
      for (int j = 0; j < n; ++j, ++it) {
        if (!mbar_wait(&sb.p_full[it % NB], (it / NB) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        // O += A V (A from TMEM in four column quarters, V MN-major)
        issue_grad<4>(tmem + C::kColO, tmem + s_col(it),
                      sdesc_sw128_lo(k_addr(it) + C::kQKBytes, 16384), dhi, idO, j > 0 ? 1u : 0u);
        umma_commit(&sb.kv_empty[it % S]);
        if (j + (int)NB < n) {
          // S three steps ahead, into the buffer this step's A has just left
          if (!mbar_wait(&sb.kv_full[(it + NB) % S], ((it + NB) / S) & 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after_sync();
          umma_bf16_ss(tmem + s_col(it + NB), qdesc, sdesc_sw32(k_addr(it + NB)), idS, 0);
          umma_commit(&sb.s_full[(it + NB) % NB]);
          if (j + (int)NB + 1 == n) umma_commit(&sb.fix_empty);
        }
      }
      if (!ok) break;
      umma_commit(&sb.acc_full);
    }
    umma_commit(&sb.mma_done);
    int never = 0;
    mbar_wait(&sb.mma_done, 0, &never);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 17) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace tkattn
