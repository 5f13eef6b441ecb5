// tk_attn_fwd.cuh -- the fused attention forward kernel for GB300 (sm_103a).
//
// Computes, for every (batch, head) slice,
//   O   = softmax(scale * Q K^T [+ causal mask]) V          (bf16 out)
//   LSE = ln sum_j exp(scale * q_i . k_j)  over visible keys (fp32 out)
// streaming K/V in 128-key tiles with an online softmax, so the N x N score
// matrix never leaves the SM.  This is the computation of the flash-attention
// examples in the ThunderKittens news write-up (88811315.cn, post 77732): the
// "RTX 4090 flash attention" example and the "H100 FlashAttention-2 forward"
// example, whose per-tile loop keeps a running row max and row sum, rescales
// the output accumulator when the max grows and adds P V.  Those examples
// divide by the running sum every step; here the division is deferred to the
// end, which is the same quantity and yields the LSE directly.
//
// Blackwell mapping (one CTA per SM, persistent over work units):
//   work unit   = one (batch*head, 256-query block): two 128-row Q tiles that
//                 share every K/V tile they load.
//   warps 0-3   softmax for Q tile 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax for Q tile 1
//   warps 8-11  correction: rescale O in TMEM when the row max grows, and the
//               epilogue O / l -> bf16, LSE
//   warp 12     tcgen05 MMA issue (one thread) and TMEM allocation
//   warp 13     TMA producer (one thread): Q tiles, then a K/V ring
//   warps 14-15 idle (keep the register split warpgroup-aligned)
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128) S0 / P0    [128,256) S1 / P1    [256,256+D) O0    [256+D,256+2D) O1
//   P_t (bf16, two per column) overwrites the first 64 columns of S_t after
//   the softmax has read S_t; the next S_t MMA is issued after the P_t V MMA,
//   and the tensor core runs one thread's MMAs in issue order.
//
// Every wait on an mbarrier is bounded; a wait that runs out raises a shared
// abort flag (all roles then leave their loops), records an error code in a
// device word that the host reads, waits for its own copies and MMAs in
// flight, frees the tensor memory and returns.  Nothing traps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace tkattn {

// error codes written to the device error word (host maps them to statuses)
constexpr int kDevErrTimeout = 1;

struct FwdParams {
  __nv_bfloat16 *o;  // [BH, N, D]
  float *lse;        // [BH, N]
  int *err;          // device error word
  int BH;            // batch * heads
  int N;             // sequence length
  int num_mblocks;   // ceil(N / 256)
  int num_units;     // BH * num_mblocks
  float scale_log2;  // scale * log2(e)
};

template <int D>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int kBM = 128;                  // query rows per Q tile
  static constexpr int kBN = 128;                  // keys per K/V tile
  static constexpr int kUnitRows = 2 * kBM;        // query rows per work unit
  static constexpr int kTileBytes = kBM * D * 2;   // one Q, K or V tile (bf16)
  static constexpr int kChunks = D / 64;           // 128-byte swizzle column chunks
  static constexpr int kChunkBytes = kBM * 128;    // one chunk: 128 rows x 128 B
  static constexpr int kStages = D == 128 ? 4 : 8; // K/V ring depth (tiles)
  static constexpr int kSmemBytes = (2 + kStages) * kTileBytes;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;  // + alignment slack
  static constexpr int kThreads = 512;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
};

// Shared-memory bookkeeping that is not tile data.
struct FwdBarriers {
  uint64_t q_full[2];     // TMA Q tile landed              (count 1 + tx)
  uint64_t q_empty;       // all S MMAs of a unit done       (tcgen05.commit)
  uint64_t kv_full[8];    // TMA K or V tile landed          (count 1 + tx)
  uint64_t kv_empty[8];   // MMAs reading the stage done     (tcgen05.commit)
  uint64_t s_full[2];     // S_t = Q_t K^T complete          (tcgen05.commit)
  uint64_t p_full[2];     // P_t written to TMEM             (4 softmax warps)
  uint64_t stats_full[2]; // alpha_t written to shared       (4 softmax warps)
  uint64_t o_ready[2];    // O_t rescaled / drained          (4 correction warps)
  uint64_t o_full[2];     // last P_t V MMA of a unit done   (tcgen05.commit)
  uint64_t fin_full[2];   // final m, l of a unit written    (4 softmax warps)
  uint64_t mma_done;      // every MMA of the CTA complete   (tcgen05.commit)
  uint32_t tmem_base;
  int abort;
  float alpha[2][128];        // per-row rescale factor of the current step
  float m_fin[2][2][128];     // [unit parity][tile][row] final scaled-log2 max
  float l_fin[2][2][128];     // [unit parity][tile][row] final row sum of P
  float lt_fin[2][2][128];    // [unit parity][tile][row] same, of bf16-rounded P
};

__device__ __forceinline__ void raise_abort(FwdBarriers &sb, int *err, int code) {
  sb.abort = 1;
  atomicCAS(err, 0, code);
}

// Unit u -> (bh, mblock).  Non-causal: head-major, so CTAs running at the same
// time share a head's K/V in L2.  Causal: longest query blocks first.
__device__ __forceinline__ void unit_coords(const FwdParams &p, bool causal, int u, int &bh,
                                            int &mb) {
  if (causal) {
    mb = p.num_mblocks - 1 - u / p.BH;
    bh = u % p.BH;
  } else {
    bh = u / p.num_mblocks;
    mb = u % p.num_mblocks;
  }
}

// Number of 128-key tiles Q tile t of block mb visits.
__device__ __forceinline__ int kv_tiles(const FwdParams &p, bool causal, int mb, int t) {
  const int nkv = (p.N + 127) / 128;
  if (!causal) return nkv;
  const int last_row = min(mb * 256 + t * 128 + 127, p.N - 1);
  return last_row / 128 + 1;
}

template <int D, bool kCausal>
__global__ void __launch_bounds__(512, 1)
    tk_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdBarriers sb;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem;                        // 2 tiles
  uint8_t *sKV = smem + 2 * C::kTileBytes;   // kStages tiles

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int *abort_flag = &sb.abort;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sb.q_full[t], 1);
      mbar_init(&sb.s_full[t], 1);
      mbar_init(&sb.p_full[t], 4);
      mbar_init(&sb.stats_full[t], 4);
      mbar_init(&sb.o_ready[t], 4);
      mbar_init(&sb.o_full[t], 1);
      mbar_init(&sb.fin_full[t], 4);
    }
    mbar_init(&sb.q_empty, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sb.kv_full[s], 1);
      mbar_init(&sb.kv_empty[s], 1);
    }
    mbar_init(&sb.mma_done, 1);
    sb.abort = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(&sb.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 13 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sb.tmem_base;

  if (warp < 8) {
    // ------------------------------------------------------------ softmax
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;\n" ::: "memory");
    const int t = warp >> 2;                 // Q tile
    const int row = (warp & 3) * 32 + lane;  // row in tile == TMEM lane
    const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (t ? C::kColS1 : C::kColS0);
    const float c = p.scale_log2;
    uint32_t s_phase = 0;
    int uc = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++uc) {
      int bh, mb;
      unit_coords(p, kCausal, u, bh, mb);
      const int n_t = kv_tiles(p, kCausal, mb, t);
      const int qrow = mb * 256 + t * 128 + row;  // global query index
      float m_run = -INFINITY, l_run = 0.f, lt_run = 0.f;
      for (int j = 0; j < n_t; ++j) {
        if (!mbar_wait(&sb.s_full[t], s_phase, abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto done;
        }
        s_phase ^= 1;
        tc_fence_after_sync();
        uint32_t s[128];
        tmem_ld_32x32b_x32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld_32x32b_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld_32x32b_x32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
        tmem_ld_32x32b_x32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 128; ++i) reg_barrier(s[i]);
        // Mask keys beyond N, and keys after the query under the causal mask.
        const int k0 = j * 128;
        const bool need_mask = (k0 + 128 > p.N) || (kCausal && k0 + 127 > mb * 256 + t * 128);
        if (need_mask) {
          int lim = p.N - k0;
          if (kCausal) lim = min(lim, qrow - k0 + 1);
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) s[i] = __float_as_uint(-INFINITY);
        }
        // Row max of the raw scores; scale > 0 so max(s)*c = max(s*c).
        float mx0 = fmaxf(__uint_as_float(s[0]), __uint_as_float(s[1]));
        float mx1 = fmaxf(__uint_as_float(s[2]), __uint_as_float(s[3]));
#pragma unroll
        for (int i = 4; i < 128; i += 4) {
          mx0 = max3(mx0, __uint_as_float(s[i]), __uint_as_float(s[i + 1]));
          mx1 = max3(mx1, __uint_as_float(s[i + 2]), __uint_as_float(s[i + 3]));
        }
        const float m_new = fmaxf(m_run, fmaxf(mx0, mx1) * c);
        const float alpha = ex2_approx(m_run - m_new);  // 0 on the first tile
        sb.alpha[t][row] = alpha;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.stats_full[t]);
        // P = 2^(s*c - m_new).  Two row sums: of the fp32 P (for the LSE) and
        // of the bf16-rounded P the P V MMA consumes (for normalising O, so
        // the weights applied to V sum to one exactly as used).
        const uint64_t c2 = f2_pack(c, c);
        const uint64_t nm2 = f2_pack(-m_new, -m_new);
        uint64_t la = 0, lb = 0, lta = 0, ltb = 0;  // (+0.f, +0.f) pairs
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2,
                           nm2),
                    x0, x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * i + 2]), __uint_as_float(s[2 * i + 3])),
                           c2, nm2),
                    x2, x3);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
          pk[i] = pack_bf16x2(p0, p1);
          pk[i + 1] = pack_bf16x2(p2, p3);
          la = f2_add(la, f2_pack(p0, p1));
          lb = f2_add(lb, f2_pack(p2, p3));
          lta = f2_add(lta, bf16x2_widen(pk[i]));
          ltb = f2_add(ltb, bf16x2_widen(pk[i + 1]));
        }
        tmem_st_32x32b_x32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st_32x32b_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        {
          float a0, a1, b0, b1;
          f2_unpack(f2_add(la, lb), a0, a1);
          f2_unpack(f2_add(lta, ltb), b0, b1);
          l_run = l_run * alpha + (a0 + a1);
          lt_run = lt_run * alpha + (b0 + b1);
        }
        m_run = m_new;
        if (j == n_t - 1) {
          sb.m_fin[uc & 1][t][row] = m_run;
          sb.l_fin[uc & 1][t][row] = l_run;
          sb.lt_fin[uc & 1][t][row] = lt_run;
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sb.p_full[t]);
          if (j == n_t - 1) mbar_arrive(&sb.fin_full[t]);
        }
      }
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ correction + epilogue
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;\n" ::: "memory");
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t st_phase[2] = {0, 0};
    uint32_t ofull_phase[2] = {0, 0};
    int uc = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++uc) {
      int bh, mb;
      unit_coords(p, kCausal, u, bh, mb);
      const int n0 = kv_tiles(p, kCausal, mb, 0);
      const int n1 = kv_tiles(p, kCausal, mb, 1);
      for (int j = 0; j < n1; ++j) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (j >= (t ? n1 : n0)) continue;
          if (!mbar_wait(&sb.stats_full[t], st_phase[t], abort_flag)) {
            raise_abort(sb, p.err, kDevErrTimeout);
            goto done;
          }
          st_phase[t] ^= 1;
          if (j > 0) {
            const float alpha = sb.alpha[t][row];
            if (__any_sync(0xffffffffu, alpha != 1.0f)) {
              // S_t of this step is complete, and its commit covers the
              // previous P_t V MMA: O_t holds its accumulated value.
              tc_fence_after_sync();
              const uint32_t tO = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
#pragma unroll
              for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tO + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  reg_barrier(r[i]);
                  r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                }
                tmem_st_32x32b_x32(tO + c0, r);
              }
              tmem_wait_st();
            }
          }
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sb.o_ready[t]);
        }
      }
      // epilogue: O / l -> bf16, LSE = (m + log2 l) * ln 2
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!mbar_wait(&sb.fin_full[t], uc & 1, abort_flag) ||
            !mbar_wait(&sb.o_full[t], ofull_phase[t], abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto done;
        }
        ofull_phase[t] ^= 1;
        tc_fence_after_sync();
        const float m = sb.m_fin[uc & 1][t][row];
        const float l = sb.l_fin[uc & 1][t][row];
        const float inv_l = 1.0f / sb.lt_fin[uc & 1][t][row];
        const int qrow = mb * 256 + t * 128 + row;
        const bool valid = qrow < p.N;
        __nv_bfloat16 *orow = p.o + ((size_t)bh * p.N + (valid ? qrow : 0)) * D;
        const uint32_t tO = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tO + c0, r);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            reg_barrier(r[2 * i]);
            reg_barrier(r[2 * i + 1]);
            pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l,
                                __uint_as_float(r[2 * i + 1]) * inv_l);
          }
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        if (valid) p.lse[(size_t)bh * p.N + qrow] = (m + lg2_approx(l)) * 0.69314718055994531f;
        // O_t has been read out: the next unit may overwrite it.  (Its first
        // P_t V MMA also waits on the o_ready arrival of step 0 above.)
      }
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;\n" ::: "memory");
    if (warp == 12 && lane == 0) {
      // ---------------------------------------------------------- MMA issue
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
      const uint32_t sQ_addr = smem_addr(sQ);
      const uint32_t sKV_addr = smem_addr(sKV);
      uint32_t q_phase = 0, p_phase[2] = {0, 0}, or_phase[2] = {0, 0};
      uint32_t kv_idx = 0;  // loads consumed so far (K_0, V_0, K_1, ...)
      for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
        int bh, mb;
        unit_coords(p, kCausal, u, bh, mb);
        const int n0 = kv_tiles(p, kCausal, mb, 0);
        const int n1 = kv_tiles(p, kCausal, mb, 1);
        if (!mbar_wait(&sb.q_full[0], q_phase, abort_flag) ||
            !mbar_wait(&sb.q_full[1], q_phase, abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto mma_exit;
        }
        q_phase ^= 1;
        tc_fence_after_sync();
        uint32_t k_stage = 0, v_stage = 0;
        // Issue order per step j: P0 V_{j-1}, S0 = Q0 K_j^T, P1 V_{j-1},
        // S1 = Q1 K_j^T.  Each softmax then has the other tile's two MMAs
        // (about 1024 tensor-core clocks) to turn S into P.
        for (int j = 0; j <= n1; ++j) {
#pragma unroll 1
          for (int t = 0; t < 2; ++t) {
            const int n_t = t ? n1 : n0;
            if (j >= 1 && j <= n_t) {
              // O_t += P_t V_{j-1}
              if (!mbar_wait(&sb.p_full[t], p_phase[t], abort_flag) ||
                  !mbar_wait(&sb.o_ready[t], or_phase[t], abort_flag)) {
                raise_abort(sb, p.err, kDevErrTimeout);
                goto mma_exit;
              }
              p_phase[t] ^= 1;
              or_phase[t] ^= 1;
              tc_fence_after_sync();
              const uint32_t tP = tmem + (t ? C::kColS1 : C::kColS0);
              const uint32_t tO = tmem + (t ? C::kColO1 : C::kColO0);
              const uint32_t vbase = sKV_addr + v_stage * C::kTileBytes;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_bf16_ts(tO, tP + kk * 8,
                             sdesc_sw128(vbase + kk * 2048, C::kChunkBytes, 1024), idO,
                             (j > 1 || kk > 0) ? 1u : 0u);
              if (j == n_t) umma_commit(&sb.o_full[t]);
              if (t == 1) umma_commit(&sb.kv_empty[v_stage]);  // V_{j-1} fully used
            }
            if (j < n_t) {
              if (t == 0 || j >= n0) {
                // first user of K_j in this step waits for it
                k_stage = kv_idx % C::kStages;
                if (!mbar_wait(&sb.kv_full[k_stage], (kv_idx / C::kStages) & 1, abort_flag)) {
                  raise_abort(sb, p.err, kDevErrTimeout);
                  goto mma_exit;
                }
                ++kv_idx;
                tc_fence_after_sync();
              }
              // S_t = Q_t K_j^T
              const uint32_t qbase = sQ_addr + t * C::kTileBytes;
              const uint32_t kbase = sKV_addr + k_stage * C::kTileBytes;
              const uint32_t tS = tmem + (t ? C::kColS1 : C::kColS0);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                umma_bf16_ss(tS, sdesc_sw128(qbase + off, 16, 1024),
                             sdesc_sw128(kbase + off, 16, 1024), idS, kk > 0 ? 1u : 0u);
              }
              umma_commit(&sb.s_full[t]);
              if (t == 1) {
                umma_commit(&sb.kv_empty[k_stage]);  // K_j fully used
                if (j == n1 - 1) umma_commit(&sb.q_empty);
                // V_j, needed by the next step's P V MMAs
                v_stage = kv_idx % C::kStages;
                if (!mbar_wait(&sb.kv_full[v_stage], (kv_idx / C::kStages) & 1, abort_flag)) {
                  raise_abort(sb, p.err, kDevErrTimeout);
                  goto mma_exit;
                }
                ++kv_idx;
                tc_fence_after_sync();
              }
            }
          }
        }
      }
    mma_exit:
      // every MMA this thread issued must finish before the TMEM is freed
      umma_commit(&sb.mma_done);
      {
        int never = 0;
        mbar_wait(&sb.mma_done, 0, &never);
      }
    } else if (warp == 13 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      uint32_t kv_idx = 0;
      uint32_t q_loads = 0;  // Q tile pairs issued
      int uc = 0;
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++uc) {
        int bh, mb;
        unit_coords(p, kCausal, u, bh, mb);
        const int n1 = kv_tiles(p, kCausal, mb, 1);
        if (uc > 0 && !mbar_wait(&sb.q_empty, (uc - 1) & 1, abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto load_exit;
        }
        for (int t = 0; t < 2; ++t) {
          mbar_arrive_expect_tx(&sb.q_full[t], C::kTileBytes);
          for (int ch = 0; ch < C::kChunks; ++ch)
            tma_load_3d_hint(sQ + t * C::kTileBytes + ch * C::kChunkBytes, &tm_q, &sb.q_full[t],
                             ch * 64, mb * 256 + t * 128, bh, pol_q);
        }
        ++q_loads;
        for (int j = 0; j < n1; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t s = kv_idx % C::kStages;
            const uint32_t fill = kv_idx / C::kStages;
            if (fill > 0 && !mbar_wait(&sb.kv_empty[s], (fill - 1) & 1, abort_flag)) {
              raise_abort(sb, p.err, kDevErrTimeout);
              goto load_exit;
            }
            mbar_arrive_expect_tx(&sb.kv_full[s], C::kTileBytes);
            const CUtensorMap *tm = kv ? &tm_v : &tm_k;
            for (int ch = 0; ch < C::kChunks; ++ch)
              tma_load_3d_hint(sKV + s * C::kTileBytes + ch * C::kChunkBytes, tm, &sb.kv_full[s],
                               ch * 64, j * 128, bh, pol_kv);
            ++kv_idx;
          }
        }
      }
    load_exit:
      // wait for the copies still in flight (all consumed on the normal path)
      {
        int never = 0;
        for (uint32_t s = 0; s < (uint32_t)C::kStages && s < kv_idx; ++s) {
          const uint32_t last = kv_idx - 1 - ((kv_idx - 1 - s) % C::kStages);
          mbar_wait(&sb.kv_full[s], (last / C::kStages) & 1, &never);
        }
        if (q_loads > 0) {
          mbar_wait(&sb.q_full[0], (q_loads - 1) & 1, &never);
          mbar_wait(&sb.q_full[1], (q_loads - 1) & 1, &never);
        }
      }
    }
  }
done:
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 12) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace tkattn
