// tk_attn_bwd.cuh -- the attention backward pass on GB300 (sm_103a): dQ, dK
// and dV of O = softmax(scale Q K^T [+ causal mask]) V for a given dO, from
// the forward's O and LSE.
//
// The pages report causal and non-causal FlashAttention backward kernels in
// ThunderKittens (the comment thread of the Spanish news page,
// es.news.hada.io topic 14783; the paper summary "ThunderKittens: Simple,
// Fast, and Adorable AI Kernels", shd-paper.top, abstract) but print none.
// The arithmetic is the chain rule through the forward definition:
//   P_ij  = exp(scale q_i.k_j - LSE_i)           (recomputed, masked -> 0)
//   dV_j  = sum_i P_ij dO_i
//   dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - delta_i),  delta_i = sum_d dO_id O_id
//   dK_j  = scale sum_i dS_ij q_i,   dQ_i = scale sum_j dS_ij k_j
//
// Three kernels, one stream, no atomics:
//   prep   -delta_i and -LSE_i log2(e) into a workspace padded to whole tiles
//   dkdv   one unit = (slice, 128-key tile j): K_j, V_j stay in shared memory
//          while every 128-query tile i streams through a ring.  S^T = K Q^T
//          and dP^T = V dO^T go to TMEM; eight elementwise warps turn them
//          into bf16 P^T and dS^T in place, and two tcgen05 MMAs with A read
//          from TMEM accumulate dV += P^T dO and dK += dS^T Q in TMEM.
//   dq     one unit = (slice, 128-query tile i): Q_i, dO_i stay while the
//          K/V tiles stream; S = Q K^T and dP = dO V^T in TMEM, bf16 dS in
//          place, dQ += dS K in TMEM.
// dkdv and dq each recompute S and dP, so the pass runs 7 tile products per
// (query tile, key tile) pair instead of the 5 an atomic dQ update needs; in
// exchange no fp32 dQ buffer and no reduction traffic.
//
// Tiles use the forward's layout (128 rows, 64-column chunks with the
// 128-byte swizzle, TMA from [B*H, N, D] tensor maps), so the forward's
// S-product issue helper serves S^T, dP^T, S and dP alike; the gradient
// products read their B operand (dO, Q or K) MN-major like the forward's V.
#pragma once

#include "tk_attn_fwd.cuh"

namespace tkattn {

struct BwdParams {
  __nv_bfloat16 *dq, *dk, *dv;  // [BH, N, D] outputs
  const float *lse2;            // [BH, Npad] -LSE * log2(e), zero past N
  const float *delta;           // [BH, Npad] -rowsum(dO * O), zero past N
  int *err;                     // device error word
  int BH, N, Npad, nt;          // nt = Npad / 128 tiles per slice
  int num_units;
  int head_group;               // causal order: slices per L2-sized section
  float scale, scale_log2;      // scale and scale * log2(e)
};

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 128;   // 128 rows x 128 B
  static constexpr int kStages = D == 128 ? 2 : 4;  // dkdv: ring depth in (Q, dO) pairs
  static constexpr int kSmemBytes = (2 + 2 * kStages) * kTileBytes;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  // dq: K and V rings of their own (K is needed one step earlier than V)
  static constexpr int kKStages = D == 128 ? 3 : 4, kVStages = D == 128 ? 2 : 4;
  static constexpr int kDqSmemAlloc = (2 + kKStages + kVStages) * kTileBytes + 1024;
  static constexpr int kDqThreads = 576;   // dq: 16 elementwise warps, producer, MMA
  static constexpr int kThreads = 576;            // dkdv: 16 elementwise warps, producer, MMA
  // TMEM columns: S (or S^T), dP (or dP^T), and the D-wide accumulators
  static constexpr uint32_t kColS = 0, kColdP = 128, kColA = 256, kColB = 256 + D;
};

template <int kStages>
struct BwdShared {
  uint64_t fix_full, fix_empty;  // the unit's resident pair landed / released
  uint64_t ring_full[kStages], ring_empty[kStages];
  uint64_t s_full;               // S (dkdv: S^T) of a step complete   (commit)
  uint64_t p_full;               // bf16 P^T of a step in TMEM         (8 warps)
  uint64_t dp_full;              // dkdv: dP^T of a step complete      (commit)
  uint64_t ds_full;              // dkdv: bf16 dS^T of a step in TMEM  (8 warps)
  uint64_t acc_full, acc_empty;  // unit's accumulators done / read    (commit / 8 warps)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  alignas(128) float vec[kStages][2][128];  // dkdv: -LSE log2(e), -delta of the ring's query tile
};

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// D (+)= A[tmem, bf16 pairs] B[smem, MN-major] over 128 rows of K: 16 per MMA.
// The elementwise warps leave the 128 K-columns' bf16 pairs in two halves,
// columns [0, 32) and [64, 96) of the A region.
// With kParts = 4 (sixteen elementwise warps) the pairs sit in four quarters,
// columns [0, 16), [32, 48), [64, 80) and [96, 112).
template <int kParts = 2>
__device__ __forceinline__ void issue_grad(uint32_t tD, uint32_t tA, uint32_t b_lo, uint32_t dhi,
                                           uint32_t idG, uint32_t acc) {
  constexpr int kPer = 8 / kParts;  // MMAs (16 K-columns each) per part
  umma_ts_w_rt(tD, tA, b_lo, dhi, idG, acc);
#pragma unroll
  for (int kk = 1; kk < 8; ++kk)
    umma_ts_w<1>(tD, tA + (128 / kParts) * (kk / kPer) + 8 * (kk % kPer),
                 b_lo + kk * (2048 >> 4), dhi, idG);
}

// ---------------------------------------------------------------- prep

constexpr int kPrepWarps = 8;

// -delta = -rowsum(dO * O) in fp32 and -LSE * log2(e), one warp per padded
// row (negated, so the elementwise passes use them as packed f32x2 addends);
// rows past N get zeros.
template <int D>
__global__ void __launch_bounds__(kPrepWarps * 32)
    tk_attn_bwd_prep_kernel(const __nv_bfloat16 *__restrict__ o,
                            const __nv_bfloat16 *__restrict__ dout,
                            const float *__restrict__ lse, float *__restrict__ lse2,
                            float *__restrict__ delta, int N, int Npad, long long rows) {
  const long long row = (long long)blockIdx.x * kPrepWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const long long bh = row / Npad;
  const int i = (int)(row - bh * Npad);
  float acc = 0.f, l2 = 0.f;
  if (i < N) {
    const size_t base = ((size_t)bh * N + i) * D + lane * (D / 32);
    if constexpr (D == 128) {
      const uint2 a = *reinterpret_cast<const uint2 *>(o + base);
      const uint2 b = *reinterpret_cast<const uint2 *>(dout + base);
      const uint32_t av[2] = {a.x, a.y}, bv[2] = {b.x, b.y};
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        acc = fmaf(__uint_as_float(av[t] << 16), __uint_as_float(bv[t] << 16), acc);
        acc = fmaf(__uint_as_float(av[t] & 0xffff0000u), __uint_as_float(bv[t] & 0xffff0000u),
                   acc);
      }
    } else {
      const uint32_t a = *reinterpret_cast<const uint32_t *>(o + base);
      const uint32_t b = *reinterpret_cast<const uint32_t *>(dout + base);
      acc = fmaf(__uint_as_float(a << 16), __uint_as_float(b << 16), acc);
      acc = fmaf(__uint_as_float(a & 0xffff0000u), __uint_as_float(b & 0xffff0000u), acc);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
    l2 = lse[bh * N + i] * 1.4426950408889634f;
  }
  if (lane == 0) {
    lse2[row] = -l2;
    delta[row] = -acc;
  }
}

// ---------------------------------------------------------------- shared parts

// Units.  dkdv: u -> (slice, key tile j); non-causal slice-major (a slice's
// key tiles share its Q/dO in L2), causal longest first (j ascending: tile j
// meets nt - j query tiles).  dq: u -> (slice, query tile i); causal longest
// first (i descending: tile i meets i + 1 key tiles).  Causal units go in
// sections of head_group slices whose streamed tiles (Q and dO, or K and V)
// fit in about 40 MB of L2, longest first within a section, so the CTAs
// running at one time share those tiles in L2 instead of each streaming
// another slice's from HBM.
__device__ __forceinline__ void causal_section(const BwdParams &p, int u, int &bh, int &r) {
  const int per_section = p.head_group * p.nt;
  const int section = u / per_section;
  const int rr = u - section * per_section;
  const int g = min(p.head_group, p.BH - section * p.head_group);  // slices in this section
  r = rr / g;  // rank by length within the section
  bh = section * p.head_group + rr % g;
}

// The uc-th unit of this CTA, or -1 when none is left: causal launches
// carry each CTA's list, built on the host greedily in the unit order (the
// next unit to the CTA with the fewest tile steps so far, as for the
// forward's SchedTable); otherwise, and when the list does not fit, the
// stride order.
template <bool kCausal>
__device__ __forceinline__ int bwd_unit_at(const SchedFor<kCausal> &tab, const BwdParams &p,
                                           int uc) {
  if constexpr (kCausal) {
    if (tab.n > 0) {
      const int i = tab.off[blockIdx.x] + uc;
      return i < tab.off[blockIdx.x + 1] ? (int)tab.units[i] : -1;
    }
  }
  const int u = blockIdx.x + uc * (int)gridDim.x;
  return u < p.num_units ? u : -1;
}

template <bool kCausal>
__device__ __forceinline__ void dkdv_unit(const BwdParams &p, int u, int &bh, int &j, int &i0,
                                          int &n) {
  if (kCausal) {
    causal_section(p, u, bh, j);
    i0 = j;
    n = p.nt - j;
  } else {
    bh = u / p.nt;
    j = u - bh * p.nt;
    i0 = 0;
    n = p.nt;
  }
}

template <bool kCausal>
__device__ __forceinline__ void dq_unit(const BwdParams &p, int u, int &bh, int &i, int &n) {
  if (kCausal) {
    int r;
    causal_section(p, u, bh, r);
    i = p.nt - 1 - r;
    n = i + 1;
  } else {
    bh = u / p.nt;
    i = u - bh * p.nt;
    n = p.nt;
  }
}

// ---------------------------------------------------------------- dK, dV

// One step (key tile j, query tile i) runs as two halves so that the tensor
// core keeps working while the elementwise warps do:
//   MMA:  S^T_i, dP^T_i | wait P_i: dV += P^T_i dO_i, S^T_{i+1} |
//         wait dS_i: dK += dS^T_i Q_i, dP^T_{i+1} | wait P_{i+1} ...
//   warps: wait S^T_i: P^T_i = exp2(S^T c - L) -> TMEM (bf16)  | signal P_i
//          wait dP^T_i: dS^T_i = P (dP^T - delta) -> TMEM      | signal dS_i
// S^T_{i+1} overwrites P^T_i and dP^T_{i+1} overwrites dS^T_i only after the
// MMAs that read them, because one thread issues all MMAs in order.
template <int D, bool kCausal>
__global__ void __launch_bounds__(576, 1)
    tk_attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_do, const BwdParams p,
                            const __grid_constant__ SchedFor<kCausal> tab) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdShared<C::kStages> sb;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sK = smem, *sV = smem + C::kTileBytes, *ring = smem + 2 * C::kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = &sb.abort;
  if (threadIdx.x == 0) {
    mbar_init(&sb.fix_full, 1);
    mbar_init(&sb.fix_empty, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sb.ring_full[s], 1);
      mbar_init(&sb.ring_empty[s], 1);
    }
    mbar_init(&sb.s_full, 1);
    mbar_init(&sb.p_full, 16);
    mbar_init(&sb.dp_full, 1);
    mbar_init(&sb.ds_full, 16);
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

  if (warp < 16) {
    // ---------------------------------------------------------- elementwise
    const int qd = warp & 3, h = warp >> 2;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const int r = qd * 32 + lane;  // key row within the tile = TMEM lane
    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int u = bwd_unit_at<kCausal>(tab, p, 0); u >= 0 && ok;
         u = bwd_unit_at<kCausal>(tab, p, (int)++uc)) {
      int bh, j, i0, n;
      dkdv_unit<kCausal>(p, u, bh, j, i0, n);
      const int kj = j * 128 + r;
#pragma unroll 1
      for (int st = 0; st < n; ++st, ++it) {
        const int i = i0 + st;
        const uint32_t s = it % C::kStages;
        if (!mbar_wait(&sb.s_full, it & 1, abort_flag) ||
            !mbar_wait(&sb.ring_full[s], (it / C::kStages) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const bool edge = (kCausal && i == j) || (i * 128 + 128 > p.N);
        // P^T = exp2(S^T scale log2(e) - LSE_i log2(e)), masked -> 0; kept in fp32.
        // Warp (qd, h) takes query columns 32 h .. 32 h + 31 of its lane quadrant.
        uint64_t pr[16];
        {
          const int c = 0;
          const int col0 = 32 * h;
          uint32_t sv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::kColS + col0, sv);
          tmem_wait_ld();
          const uint64_t *nL = reinterpret_cast<const uint64_t *>(sb.vec[s][0] + col0);
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            reg_barrier(sv[t]);
            reg_barrier(sv[t + 1]);
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1])), c2,
                             nL[t >> 1]),
                      a0, a1);
            float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            if (edge) {
              const int qi = i * 128 + col0 + t;
              if ((kCausal && qi < kj) || qi >= p.N) p0 = 0.f;
              if ((kCausal && qi + 1 < kj) || qi + 1 >= p.N) p1 = 0.f;
            }
            pr[16 * c + (t >> 1)] = f2_pack(p0, p1);
            pk[t >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st_32x32b_x16(tmem + lane_off + C::kColS + 32 * h, pk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.p_full);
        // dS^T = P^T (dP^T - delta_i)
        if (!mbar_wait(&sb.dp_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        {
          const int c = 0;
          const int col0 = 32 * h;
          uint32_t dv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::kColdP + col0, dv);
          tmem_wait_ld();
          const uint64_t *nD = reinterpret_cast<const uint64_t *>(sb.vec[s][1] + col0);
          uint32_t dk[16];
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            reg_barrier(dv[t]);
            reg_barrier(dv[t + 1]);
            float d0, d1;
            f2_unpack(f2_mul(pr[16 * c + (t >> 1)],
                             f2_add(f2_pack(__uint_as_float(dv[t]), __uint_as_float(dv[t + 1])),
                                    nD[t >> 1])),
                      d0, d1);
            dk[t >> 1] = pack_bf16x2(d0, d1);
          }
          tmem_st_32x32b_x16(tmem + lane_off + C::kColdP + 32 * h, dk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.ds_full);
      }
      if (!ok) break;
      // ---- epilogue: dV and scale * dK of this key tile, rows < N
      if (!mbar_wait(&sb.acc_full, uc & 1, abort_flag)) {
        fail();
        break;
      }
      tc_fence_after_sync();
      const bool valid = kj < p.N;
      const size_t row_off = ((size_t)bh * p.N + (valid ? kj : 0)) * D;
      {
        // warps h = 0, 1 write dV, h = 2, 3 write scale * dK, each half the columns
        const int g = h >> 1;
        const uint32_t col = g ? C::kColB : C::kColA;
        __nv_bfloat16 *dst = (g ? p.dk : p.dv) + row_off;
        const float mul = g ? p.scale : 1.f;
#pragma unroll 1
        for (int c0 = (h & 1) * (D / 2); c0 < ((h & 1) + 1) * (D / 2); c0 += 32) {
          uint32_t rv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + col + c0, rv);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            reg_barrier(rv[t]);
            reg_barrier(rv[t + 1]);
            pk[t >> 1] =
                pack_bf16x2(__uint_as_float(rv[t]) * mul, __uint_as_float(rv[t + 1]) * mul);
          }
          if (valid) {
#pragma unroll
            for (int t = 0; t < 4; ++t)
              *reinterpret_cast<uint4 *>(dst + c0 + 8 * t) =
                  make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.acc_empty);
    }
  } else if (warp == 16 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int u = bwd_unit_at<kCausal>(tab, p, 0); u >= 0 && ok;
         u = bwd_unit_at<kCausal>(tab, p, (int)++uc)) {
      int bh, j, i0, n;
      dkdv_unit<kCausal>(p, u, bh, j, i0, n);
      if (uc > 0 && !mbar_wait(&sb.fix_empty, (uc - 1) & 1, abort_flag)) {
        fail();
        break;
      }
      mbar_arrive_expect_tx(&sb.fix_full, 2 * C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(sK + c * C::kChunkBytes, &tm_k, &sb.fix_full, c * 64, j * 128, bh);
        tma_load_3d(sV + c * C::kChunkBytes, &tm_v, &sb.fix_full, c * 64, j * 128, bh);
      }
      for (int st = 0; st < n; ++st, ++it) {
        const int i = i0 + st;
        const uint32_t s = it % C::kStages;
        if (it >= (uint32_t)C::kStages &&
            !mbar_wait(&sb.ring_empty[s], ((it / C::kStages) - 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        uint8_t *sQ = ring + s * 2 * C::kTileBytes, *sdO = sQ + C::kTileBytes;
        mbar_arrive_expect_tx(&sb.ring_full[s], 2 * C::kTileBytes + 1024);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(sQ + c * C::kChunkBytes, &tm_q, &sb.ring_full[s], c * 64, i * 128, bh);
          tma_load_3d(sdO + c * C::kChunkBytes, &tm_do, &sb.ring_full[s], c * 64, i * 128, bh);
        }
        const size_t vo = (size_t)bh * p.Npad + (size_t)i * 128;
        bulk_load(sb.vec[s][0], p.lse2 + vo, 512, &sb.ring_full[s]);
        bulk_load(sb.vec[s][1], p.delta + vo, 512, &sb.ring_full[s]);
      }
    }
    // copies still in flight land before the CTA can exit
    for (int i = 0; i < 200 && !ok; ++i) __nanosleep(1000);
  } else if (warp == 17 && lane == 0) {
    // ---------------------------------------------------------- MMA issue
    constexpr uint32_t idS = idesc_f32acc(true, 128, 128, false, false);
    constexpr uint32_t idG = idesc_f32acc(true, 128, D, false, true);
    const uint32_t dhi = sdesc_sw128_hi(1024);
    const uint32_t k_lo = sdesc_sw128_lo(smem_addr(sK), 16);
    const uint32_t v_lo = sdesc_sw128_lo(smem_addr(sV), 16);
    uint32_t it = 0, uc = 0;
    bool ok = true;
    auto stage_q = [&](uint32_t t) { return smem_addr(ring + (t % C::kStages) * 2 * C::kTileBytes); };
    for (int u = bwd_unit_at<kCausal>(tab, p, 0); u >= 0 && ok;
         u = bwd_unit_at<kCausal>(tab, p, (int)++uc)) {
      int bh, j, i0, n;
      dkdv_unit<kCausal>(p, u, bh, j, i0, n);
      if (!mbar_wait(&sb.fix_full, uc & 1, abort_flag) ||
          !mbar_wait(&sb.ring_full[it % C::kStages], (it / C::kStages) & 1, abort_flag)) {
        fail();
        break;
      }
      tc_fence_after_sync();
      // step 0's S^T = K Q^T and dP^T = V dO^T (rows: keys; columns: queries)
      issue_s<D>(tmem + C::kColS, k_lo, sdesc_sw128_lo(stage_q(it), 16), dhi, idS);
      umma_commit(&sb.s_full);
      issue_s<D>(tmem + C::kColdP, v_lo, sdesc_sw128_lo(stage_q(it) + C::kTileBytes, 16), dhi,
                 idS);
      umma_commit(&sb.dp_full);
      // K_j and V_j are read by the S^T and dP^T products only: the last dP^T
      // releases them, so the next unit's pair loads during this unit's tail
      if (n == 1) umma_commit(&sb.fix_empty);
      // the epilogue has read the previous unit's accumulators
      if (uc > 0 && !mbar_wait(&sb.acc_empty, (uc - 1) & 1, abort_flag)) {
        fail();
        break;
      }
      for (int st = 0; st < n; ++st, ++it) {
        const uint32_t sq = stage_q(it), sdo = sq + C::kTileBytes;
        const uint32_t acc = st > 0 ? 1u : 0u;
        if (!mbar_wait(&sb.p_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        // dV += P^T dO (B operand MN-major), then the next step's S^T
        issue_grad<4>(tmem + C::kColA, tmem + C::kColS, sdesc_sw128_lo(sdo, C::kChunkBytes), dhi,
                   idG, acc);
        const bool more = st + 1 < n;
        if (more) {
          if (!mbar_wait(&sb.ring_full[(it + 1) % C::kStages], ((it + 1) / C::kStages) & 1,
                         abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_s<D>(tmem + C::kColS, k_lo, sdesc_sw128_lo(stage_q(it + 1), 16), dhi, idS);
          umma_commit(&sb.s_full);
        }
        if (!mbar_wait(&sb.ds_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        // dK += dS^T Q, then the next step's dP^T
        issue_grad<4>(tmem + C::kColB, tmem + C::kColdP, sdesc_sw128_lo(sq, C::kChunkBytes), dhi,
                   idG, acc);
        umma_commit(&sb.ring_empty[it % C::kStages]);
        if (more) {
          issue_s<D>(tmem + C::kColdP, v_lo, sdesc_sw128_lo(stage_q(it + 1) + C::kTileBytes, 16),
                     dhi, idS);
          umma_commit(&sb.dp_full);
          if (st + 2 == n) umma_commit(&sb.fix_empty);
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

// ---------------------------------------------------------------- dQ

template <int kKStages, int kVStages>
struct DqShared {
  uint64_t fix_full, fix_empty;  // the unit's Q_i, dO_i landed / released
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full;               // S_j complete                          (commit)
  uint64_t s_read;               // S_j read into registers               (16 warps)
  uint64_t dp_full;              // dP_j complete (over S_j)              (commit)
  uint64_t ds_full;              // bf16 dS_j in TMEM (over dP_j)         (16 warps)
  uint64_t acc_full, acc_empty;  // dQ done / read                        (commit / 16 warps)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// Sixteen elementwise warps, four per TMEM lane quadrant, each on 32 of the
// 128 key columns.  Step j (key tile j) lives in one of two 128-column
// buffers, b = j mod 2: S_j = Q K_j^T, then dP_j = dO V_j^T over it once the
// warps hold S_j in registers, then bf16 dS_j over dP_j, which dQ += dS_j K_j
// reads.  The MMA thread issues, per step,
//   wait S_j read: dP_j | S_{j+1} (other buffer) | wait dS_j: dQ += dS_j K_j
// so the tensor core computes dP_j and S_{j+1} while the warps compute P_j
// and then dS_j, and dP_{j+1} follows dQ_j as soon as S_{j+1} has been read.
// In-order issue keeps every buffer's products apart: S_{j+2} overwrites
// dS_j only after the dQ product that reads it.
template <int D, bool kCausal>
__global__ void __launch_bounds__(576, 1)
    tk_attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_do, const BwdParams p,
                          const __grid_constant__ SchedFor<kCausal> tab) {
  using C = BwdCfg<D>;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ DqShared<KS, VS> sb;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem, *sdO = smem + C::kTileBytes;
  uint8_t *kring = smem + 2 * C::kTileBytes, *vring = kring + KS * C::kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = &sb.abort;
  if (threadIdx.x == 0) {
    mbar_init(&sb.fix_full, 1);
    mbar_init(&sb.fix_empty, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(&sb.k_full[s], 1);
      mbar_init(&sb.k_empty[s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(&sb.v_full[s], 1);
      mbar_init(&sb.v_empty[s], 1);
    }
    mbar_init(&sb.s_full, 1);
    mbar_init(&sb.s_read, 16);
    mbar_init(&sb.dp_full, 1);
    mbar_init(&sb.ds_full, 16);
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
  auto s_col = [](uint32_t step) { return (step & 1) ? C::kColdP : C::kColS; };

  if (warp < 16) {
    // ---------------------------------------------------------- elementwise
    const int qd = warp & 3, h = warp >> 2;  // lane quadrant, column quarter
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const int r = qd * 32 + lane;  // query row within the tile = TMEM lane
    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int u = bwd_unit_at<kCausal>(tab, p, 0); u >= 0 && ok;
         u = bwd_unit_at<kCausal>(tab, p, (int)++uc)) {
      int bh, i, n;
      dq_unit<kCausal>(p, u, bh, i, n);
      const int qi = i * 128 + r;
      const size_t vo = (size_t)bh * p.Npad + qi;
      const uint64_t nl2 = f2_pack(p.lse2[vo], p.lse2[vo]);
      const uint64_t ndl = f2_pack(p.delta[vo], p.delta[vo]);
#pragma unroll 1
      for (int j = 0; j < n; ++j, ++it) {
        if (!mbar_wait(&sb.s_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tS = tmem + lane_off + s_col(it) + 32 * h;
        const bool edge = (kCausal && j == i) || (j * 128 + 128 > p.N);
        {
          const int col0 = 32 * h;
          uint32_t sv[32];
          tmem_ld_32x32b_x32(tS, sv);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) reg_barrier(sv[t]);
          // S_j is in registers: dP_j may overwrite it
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sb.s_read);
          uint64_t pp[16];  // P in fp32 pairs, held while dP_j is computed
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1])), c2, nl2),
                      a0, a1);
            float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            if (edge) {
              const int kj = j * 128 + col0 + t;
              if ((kCausal && kj > qi) || kj >= p.N) p0 = 0.f;
              if ((kCausal && kj + 1 > qi) || kj + 1 >= p.N) p1 = 0.f;
            }
            pp[t >> 1] = f2_pack(p0, p1);
          }
          if (!mbar_wait(&sb.dp_full, it & 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after_sync();
          uint32_t dv[32];
          tmem_ld_32x32b_x32(tS, dv);
          tmem_wait_ld();
          uint32_t dk[16];
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            reg_barrier(dv[t]);
            reg_barrier(dv[t + 1]);
            float d0, d1;
            f2_unpack(f2_mul(pp[t >> 1],
                             f2_add(f2_pack(__uint_as_float(dv[t]), __uint_as_float(dv[t + 1])),
                                    ndl)),
                      d0, d1);
            dk[t >> 1] = pack_bf16x2(d0, d1);
          }
          tmem_st_32x32b_x16(tS, dk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.ds_full);
      }
      if (!ok) break;
      // ---- epilogue: scale * dQ of this query tile, rows < N
      if (!mbar_wait(&sb.acc_full, uc & 1, abort_flag)) {
        fail();
        break;
      }
      tc_fence_after_sync();
      const bool valid = qi < p.N;
      __nv_bfloat16 *dst = p.dq + ((size_t)bh * p.N + (valid ? qi : 0)) * D;
      // quarter h of the 128 rows' dQ columns: 32 columns each (D = 64: two quarters)
      for (int c0 = 32 * h; c0 < D; c0 += 128) {
        uint32_t rv[32];
        tmem_ld_32x32b_x32(tmem + lane_off + C::kColA + c0, rv);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          reg_barrier(rv[t]);
          reg_barrier(rv[t + 1]);
          pk[t >> 1] = pack_bf16x2(__uint_as_float(rv[t]) * p.scale,
                                   __uint_as_float(rv[t + 1]) * p.scale);
        }
        if (valid) {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            *reinterpret_cast<uint4 *>(dst + c0 + 8 * t) =
                make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.acc_empty);
    }
  } else if (warp == 16 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int u = bwd_unit_at<kCausal>(tab, p, 0); u >= 0 && ok;
         u = bwd_unit_at<kCausal>(tab, p, (int)++uc)) {
      int bh, i, n;
      dq_unit<kCausal>(p, u, bh, i, n);
      if (uc > 0 && !mbar_wait(&sb.fix_empty, (uc - 1) & 1, abort_flag)) {
        fail();
        break;
      }
      mbar_arrive_expect_tx(&sb.fix_full, 2 * C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(sQ + c * C::kChunkBytes, &tm_q, &sb.fix_full, c * 64, i * 128, bh);
        tma_load_3d(sdO + c * C::kChunkBytes, &tm_do, &sb.fix_full, c * 64, i * 128, bh);
      }
      for (int j = 0; j < n; ++j, ++it) {
        const uint32_t ks = it % KS, vs = it % VS;
        if (it >= (uint32_t)KS && !mbar_wait(&sb.k_empty[ks], ((it / KS) - 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        uint8_t *sK = kring + ks * C::kTileBytes;
        mbar_arrive_expect_tx(&sb.k_full[ks], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sK + c * C::kChunkBytes, &tm_k, &sb.k_full[ks], c * 64, j * 128, bh);
        if (it >= (uint32_t)VS && !mbar_wait(&sb.v_empty[vs], ((it / VS) - 1) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        uint8_t *sV = vring + vs * C::kTileBytes;
        mbar_arrive_expect_tx(&sb.v_full[vs], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sV + c * C::kChunkBytes, &tm_v, &sb.v_full[vs], c * 64, j * 128, bh);
      }
    }
    for (int i = 0; i < 200 && !ok; ++i) __nanosleep(1000);
  } else if (warp == 17 && lane == 0) {
    // ---------------------------------------------------------- MMA issue
    constexpr uint32_t idS = idesc_f32acc(true, 128, 128, false, false);
    constexpr uint32_t idG = idesc_f32acc(true, 128, D, false, true);
    const uint32_t dhi = sdesc_sw128_hi(1024);
    const uint32_t q_lo = sdesc_sw128_lo(smem_addr(sQ), 16);
    const uint32_t do_lo = sdesc_sw128_lo(smem_addr(sdO), 16);
    auto k_addr = [&](uint32_t t) { return smem_addr(kring + (t % KS) * C::kTileBytes); };
    auto v_addr = [&](uint32_t t) { return smem_addr(vring + (t % VS) * C::kTileBytes); };
    uint32_t it = 0, uc = 0;
    bool ok = true;
    for (int u = bwd_unit_at<kCausal>(tab, p, 0); u >= 0 && ok;
         u = bwd_unit_at<kCausal>(tab, p, (int)++uc)) {
      int bh, i, n;
      dq_unit<kCausal>(p, u, bh, i, n);
      // S_0 = Q K_0^T (rows: queries; columns: keys)
      if (!mbar_wait(&sb.fix_full, uc & 1, abort_flag) ||
          !mbar_wait(&sb.k_full[it % KS], (it / KS) & 1, abort_flag)) {
        fail();
        break;
      }
      tc_fence_after_sync();
      issue_s<D>(tmem + s_col(it), q_lo, sdesc_sw128_lo(k_addr(it), 16), dhi, idS);
      umma_commit(&sb.s_full);
      for (int j = 0; j < n; ++j, ++it) {
        // dP_j = dO V_j^T over S_j, once the warps hold S_j
        if (!mbar_wait(&sb.s_read, it & 1, abort_flag) ||
            !mbar_wait(&sb.v_full[it % VS], (it / VS) & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_s<D>(tmem + s_col(it), do_lo, sdesc_sw128_lo(v_addr(it), 16), dhi, idS);
        umma_commit(&sb.dp_full);
        umma_commit(&sb.v_empty[it % VS]);
        // Q_i and dO_i are read by the S and dP products only: the last dP
        // releases them, so the next unit's pair loads during this unit's tail
        if (j + 1 == n) umma_commit(&sb.fix_empty);
        if (j + 1 < n) {
          // the next scores, into the other buffer, while the warps work
          if (!mbar_wait(&sb.k_full[(it + 1) % KS], ((it + 1) / KS) & 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_s<D>(tmem + s_col(it + 1), q_lo, sdesc_sw128_lo(k_addr(it + 1), 16), dhi, idS);
          umma_commit(&sb.s_full);
        }
        // dQ += dS_j K_j (B operand MN-major); the unit's first one overwrites
        // dQ, after the previous unit's epilogue has read it
        if ((j == 0 && uc > 0 && !mbar_wait(&sb.acc_empty, (uc - 1) & 1, abort_flag)) ||
            !mbar_wait(&sb.ds_full, it & 1, abort_flag)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_grad<4>(tmem + C::kColA, tmem + s_col(it),
                      sdesc_sw128_lo(k_addr(it), C::kChunkBytes), dhi, idG, j > 0 ? 1u : 0u);
        umma_commit(&sb.k_empty[it % KS]);
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
