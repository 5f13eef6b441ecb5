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
//   warps 8-11  V converter (bf16 -> fp16 in shared memory) and epilogue
//   warp 12     tcgen05 MMA issue for Q tile 0 (one thread), TMEM allocation
//   warp 13     tcgen05 MMA issue for Q tile 1 (one thread)
//   warp 14     TMA producer (one thread): Q tiles, then a K/V ring
//   warp 15     idle (keeps the register split warpgroup-aligned)
// Per K/V step each issuing thread runs its tile's P V and S MMAs; while one
// softmax warpgroup works, the other tile's MMAs run.  The issue slots of an
// SM sub-partition are shared with two softmax warps, so each tile gets its
// own issuing thread on its own sub-partition.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128) S0 / P0    [128,256) S1 / P1    [256,256+D) O0    [256+D,256+2D) O1
//   P_t (fp16, two per column) overwrites the first 64 columns of S_t after
//   the softmax has read S_t; the next S_t MMA is issued after the P_t V MMA
//   by the same thread, and one thread's MMAs run in issue order.
//
// Precision: S = Q K^T in bf16 x bf16 -> fp32.  P is rounded to fp16
// (at most 2^-11 relative, eight times finer than bf16) and multiplied with
// V in fp16 x fp16 -> fp32; each V tile is converted exactly to fp16 in
// shared memory, scaled by a power of two 2^E when its magnitudes would
// overflow fp16 (E is non-increasing along a unit and O is rescaled to
// match, so the scaling is exact).  The running max is lazy: a row's
// reference max moves only when the tile max exceeds it by more than 2^8
// (log2 units), so P <= 256 and O needs rescaling rarely.  The row sum l is
// accumulated in fp32 from the unrounded P, and gives the LSE.  O is divided
// by l plus the fp16 rounding error of each tile's largest P: in a row that
// one key dominates, numerator and denominator then carry the same rounded
// weight, and the dominant value passes through without the 2^-11 error.
//
// Every wait on an mbarrier is bounded; a wait that runs out raises a shared
// abort flag (all roles then leave their loops), records an error code in a
// device word that the host reads, waits for its own copies and MMAs in
// flight, frees the tensor memory and returns.  Nothing traps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "sm103_ptx.cuh"

namespace tkattn {

// error codes written to the device error word (host maps them to statuses)
constexpr int kDevErrTimeout = 1;

struct FwdParams {
  __nv_bfloat16 *o;  // [BH, N, D]
  float *lse;        // [BH, N]
  int *err;          // device error word
  int BH;            // batch * heads
  int N;             // query rows per slice (Nq)
  int Nk;            // keys per slice (== N except for the queries-vs-keys calls)
  int q_off;         // causal: absolute position of query row 0 (Nk - Nq; key j is
                     // visible to query i iff j <= i + q_off)
  int num_mblocks;   // ceil(N / 256)
  int num_units;     // BH * num_mblocks
  float scale_log2;  // scale * log2(e)
  int test_drop_load;  // test hook: CTA 0 skips its first K load (0 = off)
  int head_group;      // causal unit order: heads per section (>= 1)
  // Split over keys (inference shape): every (slice, 256-query block) is cut
  // into ranges of split_tiles 128-key tiles; a unit writes its range's O / l
  // (fp32) and natural-log LSE to o_part [num_splits, BH, N, D] and lse_part
  // [num_splits, BH, N], which a second kernel combines.  Unmasked: every
  // block has num_splits ranges.  Causal: block mb has
  // ceil(kv_tiles(mb, 0) / split_tiles) ranges (at most num_splits), the last
  // of which also holds the key tiles only the block's second Q tile sees;
  // units_per_bh counts them over the blocks of one slice.
  int num_splits;
  int split_tiles;
  int units_per_bh;
  float *o_part;
  float *lse_part;
};

// Causal units differ in length (a query block visits only the keys up to
// it), so causal launches carry each CTA's list of units, assigned on the
// host greedily in the unit order: every unit goes to the CTA whose list is
// shortest so far, counted in K/V steps.  That is the order a dynamic queue
// would produce, with no claiming on the device.  Lists live in the kernel's
// parameter space; more units than fit fall back to the stride order.
constexpr int kSchedMaxGrid = 160;
constexpr int kSchedCap = 12032;
struct SchedTable {
  int n;                               // units listed; 0 = stride order
  uint16_t off[kSchedMaxGrid + 1];     // CTA b runs units[off[b] .. off[b+1])
  uint16_t units[kSchedCap];
};
struct NoSchedTable {};
template <bool kCausal>
using SchedFor = typename std::conditional<kCausal, SchedTable, NoSchedTable>::type;

template <int D, bool kHalf = false>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int kBM = 128;                  // query rows per Q tile
  static constexpr int kBN = 128;                  // keys per K/V tile
  static constexpr int kTileBytes = kBM * D * 2;   // one Q, K or V tile (16-bit)
  static constexpr int kChunks = D / 64;           // 128-byte swizzle column chunks
  static constexpr int kChunkBytes = kBM * 128;    // one chunk: 128 rows x 128 B
  static constexpr int kStages = D == 128 ? 4 : 8; // K/V ring depth (tiles; even)
  // Q tile pairs in shared memory: with D = 64 the next unit's pair loads
  // while the current one is in use; with D = 128 there is room for one.
  static constexpr int kQBufs = D == 64 ? 2 : 1;
  static constexpr int kSmemBytes = (2 * kQBufs + kStages) * kTileBytes;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;  // + alignment slack
  static constexpr int kThreads = 512;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  // With D = 64 the tensor memory has room for P next to S (columns
  // [384, 512)), so the next S MMA of a tile needs only the softmax to have
  // read S, not its whole pass: S and P are decoupled.  With D = 128 the 512
  // columns hold S and O alone and P overwrites S, except in launches of at
  // most 128 queries (kHalf): there every unit's second Q tile lies past the
  // last query and only keeps the barrier protocol, and tile 0's P takes the
  // second tile's S columns.
  static constexpr bool kSplitP = D == 64 || kHalf;
  static constexpr uint32_t kColP0 = !kSplitP ? kColS0 : D == 64 ? 384 : kColS1;
  static constexpr uint32_t kColP1 = !kSplitP ? kColS1 : D == 64 ? 448 : kColS1 + 64;
  // converter: 16-byte words of one V tile per converter thread
  static constexpr int kConvVec = kTileBytes / 16 / 128;
  static_assert(kStages % 2 == 0, "K tiles in even stages, V tiles in odd stages");
};

// Lazy-max threshold (log2 units): P stays <= 2^kTau.
constexpr float kTau = 8.0f;

// Shared-memory bookkeeping that is not tile data.
struct FwdShared {
  uint64_t q_full[2][2];  // [buffer][tile] TMA Q tile landed   (1 + tx)
  uint64_t q_empty[2];    // [buffer] S MMAs done with the pair (commit per issuer)
  uint64_t kv_full[8];    // TMA K or V tile landed             (1 + tx)
  uint64_t kv_empty[8];   // both tiles' MMAs done with stage   (commit per issuer)
  uint64_t v_ready[8];    // V tile converted to fp16           (4 converter warps)
  uint64_t s_full[2];     // S_t = Q_t K^T complete             (commit)
  uint64_t p_full[2];     // P_t in TMEM, O_t rescaled          (4 softmax warps)
  uint64_t fin_full[2][2]; // [unit parity][tile] final m, l in shared (4 softmax warps)
  uint64_t o_full[2];     // last P_t V MMA of a unit done      (commit)
  uint64_t o_free[2];     // epilogue has read O_t              (4 converter warps)
  uint64_t conv_bar;      // converter warps' tile-max exchange (4 converter warps)
  uint64_t mma_done[2];   // every MMA of issuing thread t done   (commit)
  uint32_t tmem_base;
  int abort;
  int v_exp[8];           // power-of-two exponent of each converted V stage
  uint32_t conv_max[2][4];
  float m_fin[2][2][128];  // [unit parity][tile][row] final reference max (scaled log2)
  float l_fin[2][2][128];  // [unit parity][tile][row] final row sum
  float lc_fin[2][2][128]; // [unit parity][tile][row] fp16 rounding of the tile maxima's P
  uint64_t s_free[2];     // softmax has read S_t (split P only) (4 softmax warps)
  uint64_t pv_done[2];    // P_t V MMA complete (split P only)  (commit)
  uint64_t exp_turn[2];   // split P: tile t may run its exponentials (4 warps of the other tile)
};

__device__ __forceinline__ void raise_abort(FwdShared &sb, int *err, int code) {
  sb.abort = 1;
  atomicCAS(err, 0, code);
}

// Unit u -> (bh, mblock).  Non-causal: head-major, so CTAs running at the same
// time share a head's K/V in L2.  Causal: heads are taken in sections of
// head_group (sized on the host so a section's K/V fits in L2), and within a
// section the longest query blocks come first.
__host__ __device__ __forceinline__ void unit_coords(const FwdParams &p, bool causal, int u,
                                                     int &bh, int &mb) {
  if (causal) {
    const int per_section = p.head_group * p.num_mblocks;
    const int section = u / per_section;
    const int r = u - section * per_section;
    const int g = min(p.head_group, p.BH - section * p.head_group);  // heads in this section
    mb = p.num_mblocks - 1 - r / g;
    bh = section * p.head_group + r % g;
  } else {
    bh = u / p.num_mblocks;
    mb = u % p.num_mblocks;
  }
}

// Number of 128-key tiles Q tile t of block mb visits.
__host__ __device__ __forceinline__ int kv_tiles(const FwdParams &p, bool causal, int mb, int t) {
  const int nkv = (p.Nk + 127) / 128;
  if (!causal) return nkv;
  const int last_row = min(mb * 256 + t * 128 + 127, p.N - 1);
  return min((last_row + p.q_off) / 128 + 1, nkv);
}

// Causal split: key ranges of query block mb.
__host__ __device__ __forceinline__ int causal_ranges(const FwdParams &p, int mb) {
  const int v0 = kv_tiles(p, true, mb, 0);
  return max(1, (v0 + p.split_tiles - 1) / p.split_tiles);
}

// The uc-th work unit of this CTA, or -1 when none is left.
template <bool kCausal>
__device__ __forceinline__ int unit_at(const SchedFor<kCausal> &tab, const FwdParams &p,
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

// Unit u -> slice, query block, key split and its key tiles: the first tile
// j0 and how many tiles Q tile 0 / Q tile 1 visit.
template <bool kCausal, bool kSplit>
__device__ __forceinline__ void unit_info(const FwdParams &p, int u, int &bh, int &mb, int &s,
                                          int &j0, int &n0, int &n1) {
  if constexpr (kSplit && kCausal) {
    // blocks have different range counts: walk them
    bh = u / p.units_per_bh;
    int r = u - bh * p.units_per_bh;
    int ranges = 1;
    for (mb = 0; mb < p.num_mblocks - 1; ++mb) {
      ranges = causal_ranges(p, mb);
      if (r < ranges) break;
      r -= ranges;
    }
    if (mb == p.num_mblocks - 1) ranges = causal_ranges(p, mb);
    s = r;
    j0 = s * p.split_tiles;
    if (s == ranges - 1) {  // the last range: up to each tile's last visible key
      n0 = kv_tiles(p, true, mb, 0) - j0;
      n1 = kv_tiles(p, true, mb, 1) - j0;
    } else {
      n0 = n1 = p.split_tiles;
    }
  } else if constexpr (kSplit) {
    const int per_bh = p.num_mblocks * p.num_splits;
    bh = u / per_bh;
    const int r = u - bh * per_bh;
    mb = r / p.num_splits;
    s = r - mb * p.num_splits;
    j0 = s * p.split_tiles;
    n0 = n1 = min(p.split_tiles, (p.Nk + 127) / 128 - j0);
  } else {
    unit_coords(p, kCausal, u, bh, mb);
    s = 0;
    j0 = 0;
    n0 = kv_tiles(p, kCausal, mb, 0);
    n1 = kv_tiles(p, kCausal, mb, 1);
  }
}

// S = Q K^T for one Q tile: 16 head-dim columns (32 B of a swizzled row) per MMA.
template <int D>
__device__ __forceinline__ void issue_s(uint32_t tS, uint32_t a_lo, uint32_t b_lo, uint32_t dhi,
                                        uint32_t idS) {
  umma_ss_w<0>(tS, a_lo, b_lo, dhi, idS);
#pragma unroll
  for (int kk = 1; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * FwdCfg<D>::kChunkBytes + (kk & 3) * 32) >> 4;
    umma_ss_w<1>(tS, a_lo + off, b_lo + off, dhi, idS);
  }
}

// O (+)= P V for one Q tile: 16 keys (8 P columns, 2048 B of V) per MMA.
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint32_t v_lo, uint32_t dhi,
                                         uint32_t idO, uint32_t acc) {
  umma_ts_w_rt(tO, tP, v_lo, dhi, idO, acc);
#pragma unroll
  for (int kk = 1; kk < 8; ++kk) umma_ts_w<1>(tO, tP + kk * 8, v_lo + kk * (2048 >> 4), dhi, idO);
}

template <int D, bool kCausal, bool kSplit, bool kHalf>
__global__ void __launch_bounds__(512, 1)
    tk_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const FwdParams p,
                       const __grid_constant__ SchedFor<kCausal> tab) {
  using C = FwdCfg<D, kHalf>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdShared sb;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem;                                 // kQBufs pairs of tiles
  uint8_t *sKV = smem + 2 * C::kQBufs * C::kTileBytes;  // kStages tiles

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int *abort_flag = &sb.abort;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sb.q_full[0][t], 1);
      mbar_init(&sb.q_full[1][t], 1);
      mbar_init(&sb.q_empty[t], C::kSplitP && !kHalf ? 2 : 1);  // one commit per issuer
      mbar_init(&sb.s_full[t], 1);
      mbar_init(&sb.s_free[t], 4);
      mbar_init(&sb.pv_done[t], 1);
      mbar_init(&sb.exp_turn[t], 4);
      mbar_init(&sb.p_full[t], 4);
      mbar_init(&sb.fin_full[0][t], 4);
      mbar_init(&sb.fin_full[1][t], 4);
      mbar_init(&sb.o_full[t], 1);
      mbar_init(&sb.o_free[t], 4);
      mbar_init(&sb.mma_done[t], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sb.kv_full[s], 1);
      mbar_init(&sb.kv_empty[s], C::kSplitP && !kHalf ? 2 : 1);
      mbar_init(&sb.v_ready[s], 4);
    }
    mbar_init(&sb.conv_bar, 4);
    // tile 0 takes the first exponential turn
    for (int i = 0; i < 4; ++i) mbar_arrive(&sb.exp_turn[0]);
    sb.abort = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(&sb.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 14 && lane == 0) {
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 176;\n" ::: "memory");
    const int t = warp >> 2;                 // Q tile
    const int row = (warp & 3) * 32 + lane;  // row in tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (t ? C::kColS1 : C::kColS0);
    const uint32_t tO = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
    const uint32_t tP = tmem + lane_off + (t ? C::kColP1 : C::kColP0);
    const float c = p.scale_log2;
    uint32_t s_phase = 0;
    uint32_t steps = 0;  // S tiles this warp has processed (all units): P V MMAs issued before
    uint32_t turns = 0;  // split P: exponential turns this tile has taken
    uint32_t kvb = 0;  // K/V load index of this unit's K_0
    for (int uc = 0;; ++uc) {
      const int u = unit_at<kCausal>(tab, p, uc);
      if (u < 0) break;
      int bh, mb, sp, j0, n0, n1;
      unit_info<kCausal, kSplit>(p, u, bh, mb, sp, j0, n0, n1);
      const int n_t = t ? n1 : n0;
      const int qrow = mb * 256 + t * 128 + row;  // global query index
      // With at most 128 queries, tile 1 and the warps of tile 0 whose 32 rows
      // all lie past the last query keep the barrier protocol and skip the
      // arithmetic; the two tiles then take no exponential turns.
      const bool idle = kHalf && (t == 1 || (warp & 3) * 32 >= p.N);
      float m_run = -INFINITY, l_run = 0.f;
      float lc_run = 0.f;  // sum of (fp16(P) - P) over each tile's largest P
      int e_cur = 0;  // V exponent O is accumulated at
      for (int j = 0; j < n_t; ++j) {
        if (!mbar_wait(&sb.s_full[t], s_phase, abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto done;
        }
        s_phase ^= 1;
        if (idle) {
          // split P here: S read, previous P V done, P written
          __syncwarp();
          if (lane == 0) mbar_arrive(&sb.s_free[t]);
          if (steps > 0 && !mbar_wait(&sb.pv_done[t], (steps - 1) & 1, abort_flag)) {
            raise_abort(sb, p.err, kDevErrTimeout);
            goto done;
          }
          ++steps;
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&sb.p_full[t]);
            if (j == n_t - 1) mbar_arrive(&sb.fin_full[uc & 1][t]);
          }
          continue;
        }
        tc_fence_after_sync();
        uint32_t s[128];
        tmem_ld_32x32b_x32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld_32x32b_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld_32x32b_x32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
        tmem_ld_32x32b_x32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 128; ++i) reg_barrier(s[i]);
        if constexpr (C::kSplitP) {
          // S_t is in registers: the MMA thread may overwrite it with the next S.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sb.s_free[t]);
        }
        // Mask keys beyond N, and keys after the query under the causal mask.
        const int k0 = (j0 + j) * 128;
        const bool need_mask =
            (k0 + 128 > p.Nk) || (kCausal && k0 + 127 > mb * 256 + t * 128 + p.q_off);
        if (need_mask) {
          int lim = p.Nk - k0;
          if (kCausal) lim = min(lim, qrow + p.q_off - k0 + 1);
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) s[i] = __float_as_uint(-INFINITY);
        }
        // Row max of the raw scores; scale > 0 so max(s)*c = max(s*c).
        float mx[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx[q] = fmaxf(__uint_as_float(s[2 * q]), __uint_as_float(s[2 * q + 1]));
#pragma unroll
        for (int i = 16; i < 128; i += 16) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            mx[q] = max3(mx[q], __uint_as_float(s[i + 2 * q]), __uint_as_float(s[i + 2 * q + 1]));
        }
        const float s_max =
            fmaxf(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], max3(mx[5], mx[6], mx[7])));
        const float m_cand = s_max * c;
        // Lazy max: move the reference only when the tile max exceeds it by
        // more than kTau (always on the first tile, where m_run = -inf).
        const bool grow = m_cand > m_run + kTau;
        const float m_new = grow ? m_cand : m_run;
        const float fac = grow ? ex2_approx(m_run - m_new) : 1.0f;  // 0 on the first tile
        m_run = m_new;
        // A causal key range can hold no key visible to a row yet (its first
        // tiles lie past the row): keep its P at 0 instead of 2^(-inf + inf).
        float m_use = m_run;
        if constexpr (kSplit && kCausal) m_use = m_run == -INFINITY ? 0.f : m_run;
        // The tile's largest P exactly as the loop below computes it, and the
        // error its fp16 rounding puts into the P V product.
        const float p_max = ex2_approx(fmaf(s_max, c, -m_use));
        const float p_max_err = round_to_f16(p_max) - p_max;
        // P = 2^(s*c - m_run) <= 2^kTau, rounded to fp16 for the P V MMA;
        // the row sum is taken over the fp32 P.
        const uint64_t c2 = f2_pack(c, c);
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        uint64_t la = 0, lb = 0;  // (+0.f, +0.f) pairs
        // Split P: the two tiles' softmax warps of an SM sub-partition take
        // turns at the exponentials (the special-function unit is the shared
        // bottleneck), so each one's other work overlaps the other's
        // exponentials.  Turns pair step j of tile 0 with step j of tile 1;
        // a causal unit's last tile-1 step has no partner and takes no turn.
        const bool take_turn = C::kSplitP && !kHalf && (t == 0 || j < n0);
        if (take_turn && !mbar_wait(&sb.exp_turn[t], turns & 1, abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto done;
        }
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
          pk[i] = pack_f16x2(p0, p1);
          pk[i + 1] = pack_f16x2(p2, p3);
          la = f2_add(la, f2_pack(p0, p1));
          lb = f2_add(lb, f2_pack(p2, p3));
        }
        if (take_turn) {
          ++turns;
          __syncwarp();
          if (lane == 0) mbar_arrive(&sb.exp_turn[t ^ 1]);
        }
        if constexpr (C::kSplitP) {
          // The previous P_t V MMA must be done reading P_t (and writing O_t,
          // which the rescale below touches).
          if (steps > 0 && !mbar_wait(&sb.pv_done[t], (steps - 1) & 1, abort_flag)) {
            raise_abort(sb, p.err, kDevErrTimeout);
            goto done;
          }
          tc_fence_after_sync();
          ++steps;
          tmem_st_32x32b_x32(tP + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          tmem_st_32x32b_x32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        } else {
          tmem_st_32x32b_x32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          tmem_st_32x32b_x32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        }
        // Exponent of the V tile this step multiplies (set by the converter;
        // waited here, after the P stores, to keep it off the exp path).
        const uint32_t vidx = kvb + 2 * j + 1;
        if (!mbar_wait(&sb.v_ready[vidx % C::kStages], (vidx / C::kStages) & 1, abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto done;
        }
        const int e_j = sb.v_exp[vidx % C::kStages];
        // O_t must be multiplied by this factor before the P_t V MMA of this
        // step: the reference max moved, or V_j was scaled by a smaller 2^e.
        const float ofac = (e_j == e_cur) ? fac : fac * exp2i(e_j - e_cur);
        e_cur = e_j;
        // Rescale this warp's O rows (after the scores are dead, to keep
        // register pressure down).  The previous P_t V MMA is complete (its
        // commit is covered by this step's S_t commit, or waited above when
        // P is split from S): O_t holds its accumulated value.
        if (j > 0 && __any_sync(0xffffffffu, ofac != 1.0f)) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tO + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              reg_barrier(r[i]);
              reg_barrier(r[i + 1]);
              float a, b;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                               f2_pack(ofac, ofac)),
                        a, b);
              r[i] = __float_as_uint(a);
              r[i + 1] = __float_as_uint(b);
            }
            tmem_st_32x32b_x32(tO + c0, r);
          }
        }
        {
          float a0, a1;
          f2_unpack(f2_add(la, lb), a0, a1);
          l_run = l_run * fac + (a0 + a1);
          lc_run = lc_run * fac + p_max_err;
        }
        if (j == n_t - 1) {
          sb.m_fin[uc & 1][t][row] = m_run;
          sb.l_fin[uc & 1][t][row] = l_run;
          sb.lc_fin[uc & 1][t][row] = lc_run;
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sb.p_full[t]);
          if (j == n_t - 1) mbar_arrive(&sb.fin_full[uc & 1][t]);
        }
      }
      kvb += 2 * n1;
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ V converter + epilogue
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;\n" ::: "memory");
    const int cw = warp - 8;                 // converter warp 0..3
    const int ct = threadIdx.x - 256;        // converter thread 0..127
    const int row = (warp & 3) * 32 + lane;  // epilogue: row == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t kvb = 0;
    uint32_t conv_count = 0;  // V tiles converted (conv_bar phases)
    // the unit whose epilogue is pending
    int pend_bh = -1, pend_mb = 0, pend_sp = 0, pend_uc = 0, pend_e[2] = {0, 0};
    for (int uc = 0;; ++uc) {
      const int u = unit_at<kCausal>(tab, p, uc);
      const bool have_unit = u >= 0;
      int bh = 0, mb = 0, sp = 0, j0 = 0, n0 = 0, n1 = 0;
      if (have_unit) unit_info<kCausal, kSplit>(p, u, bh, mb, sp, j0, n0, n1);
      int e_run = 0, e_t0 = 0, e_t1 = 0;
      for (int j = 0; j <= n1; ++j) {
        // The previous unit's epilogue runs after this unit's first V tile
        // is converted (so its P V MMAs can start), or at the very end.
        if (pend_bh >= 0 && (j == 1 || !have_unit)) {
#pragma unroll 1
          for (int t = 0; t < 2; ++t) {
            // fin_full is double-buffered by unit parity: a unit whose tile 0
            // takes a single K/V step can finish before this epilogue starts.
            if (!mbar_wait(&sb.fin_full[pend_uc & 1][t], (pend_uc >> 1) & 1, abort_flag) ||
                !mbar_wait(&sb.o_full[t], pend_uc & 1, abort_flag)) {
              raise_abort(sb, p.err, kDevErrTimeout);
              goto done;
            }
            tc_fence_after_sync();
            const float m = sb.m_fin[pend_uc & 1][t][row];
            const float l = sb.l_fin[pend_uc & 1][t][row];
            float oscale = exp2i(-pend_e[t]) / (l + sb.lc_fin[pend_uc & 1][t][row]);
            if constexpr (kSplit && kCausal) oscale = l > 0.f ? oscale : 0.f;  // no key in range
            const int qrow = pend_mb * 256 + t * 128 + row;
            const bool valid = qrow < p.N;
            const uint32_t tO = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
            if constexpr (kSplit) {
              // this key range's O / l in fp32, and its LSE, for the combine
              const size_t prow = ((size_t)pend_sp * p.BH + pend_bh) * p.N + (valid ? qrow : 0);
              float4 *orow = reinterpret_cast<float4 *>(p.o_part + prow * D);
#pragma unroll 1
              for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tO + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) reg_barrier(r[i]);
                if (valid) {
#pragma unroll
                  for (int i = 0; i < 8; ++i)
                    orow[c0 / 4 + i] = make_float4(__uint_as_float(r[4 * i]) * oscale,
                                                   __uint_as_float(r[4 * i + 1]) * oscale,
                                                   __uint_as_float(r[4 * i + 2]) * oscale,
                                                   __uint_as_float(r[4 * i + 3]) * oscale);
                }
              }
              if (valid) p.lse_part[prow] = (m + lg2_approx(l)) * 0.69314718055994531f;
            } else {
              __nv_bfloat16 *orow = p.o + ((size_t)pend_bh * p.N + (valid ? qrow : 0)) * D;
#pragma unroll 1
              for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tO + c0, r);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  reg_barrier(r[2 * i]);
                  reg_barrier(r[2 * i + 1]);
                  pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * oscale,
                                      __uint_as_float(r[2 * i + 1]) * oscale);
                }
                if (valid) {
                  uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
              }
              if (valid)
                p.lse[(size_t)pend_bh * p.N + qrow] = (m + lg2_approx(l)) * 0.69314718055994531f;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sb.o_free[t]);
          }
          pend_bh = -1;
        }
        if (j == n1) break;
        // Convert V_j (bf16 -> fp16, in place, scaled by 2^e_run).
        const uint32_t vidx = kvb + 2 * j + 1;
        const uint32_t st = vidx % C::kStages;
        if (!mbar_wait(&sb.kv_full[st], (vidx / C::kStages) & 1, abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto done;
        }
        uint4 *tile = reinterpret_cast<uint4 *>(sKV + st * C::kTileBytes);
        uint4 w[C::kConvVec];
#pragma unroll
        for (int i = 0; i < C::kConvVec; ++i) w[i] = tile[ct + 128 * i];
        // Convert at the unit's current exponent and store; fp16 holds every
        // bf16 value below 2^16 exactly, and a value at or above it becomes
        // inf, which the running |max| below detects.
        uint32_t hmax = 0;  // per-16-bit-lane max |fp16| of the results
        if (e_run == 0) {
#pragma unroll
          for (int i = 0; i < C::kConvVec; ++i) {
            const uint4 o = bf16x8_to_f16x8(w[i]);
            hmax = maxabs_f16x2(hmax, maxabs_f16x2(maxabs_f16x2(o.x, o.y), maxabs_f16x2(o.z, o.w)));
            tile[ct + 128 * i] = o;
          }
        } else {
          const float sc = exp2i(e_run);
#pragma unroll
          for (int i = 0; i < C::kConvVec; ++i) {
            const uint4 o = bf16x8_to_f16x8_scaled(w[i], sc);
            hmax = maxabs_f16x2(hmax, maxabs_f16x2(maxabs_f16x2(o.x, o.y), maxabs_f16x2(o.z, o.w)));
            tile[ct + 128 * i] = o;
          }
        }
        const bool ovf = __any_sync(0xffffffffu, ((hmax & 0x7fffu) >= 0x7c00u) ||
                                                     (((hmax >> 16) & 0x7fffu) >= 0x7c00u));
        // All four converter warps must agree before the tile is released.
        if (lane == 0) {
          sb.conv_max[conv_count & 1][cw] = ovf ? 1u : 0u;
          mbar_arrive(&sb.conv_bar);
        }
        if (!mbar_wait(&sb.conv_bar, conv_count & 1, abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto done;
        }
        const bool any_ovf = (sb.conv_max[conv_count & 1][0] | sb.conv_max[conv_count & 1][1] |
                              sb.conv_max[conv_count & 1][2] | sb.conv_max[conv_count & 1][3]) != 0;
        ++conv_count;
        if (any_ovf) {
          // Rare: magnitudes at or above 2^16 * 2^-e_run.  Find the tile's
          // largest |v| (bf16 bit patterns order like magnitudes), lower the
          // unit's exponent so it fits, and convert again.
          uint32_t amax2 = 0;
#pragma unroll
          for (int i = 0; i < C::kConvVec; ++i) {
            amax2 = max_u16x2(amax2, w[i].x & 0x7fff7fffu);
            amax2 = max_u16x2(amax2, w[i].y & 0x7fff7fffu);
            amax2 = max_u16x2(amax2, w[i].z & 0x7fff7fffu);
            amax2 = max_u16x2(amax2, w[i].w & 0x7fff7fffu);
          }
          const uint32_t wmax = __reduce_max_sync(0xffffffffu, max(amax2 & 0xffffu, amax2 >> 16));
          if (lane == 0) {
            sb.conv_max[conv_count & 1][cw] = wmax;
            mbar_arrive(&sb.conv_bar);
          }
          if (!mbar_wait(&sb.conv_bar, conv_count & 1, abort_flag)) {
            raise_abort(sb, p.err, kDevErrTimeout);
            goto done;
          }
          const uint32_t amax =
              max(max(sb.conv_max[conv_count & 1][0], sb.conv_max[conv_count & 1][1]),
                  max(sb.conv_max[conv_count & 1][2], sb.conv_max[conv_count & 1][3]));
          ++conv_count;
          // |v| < 2^(k+1) with k = biased exponent - 127; scale by 2^(15-k).
          // Non-finite inputs (exponent field 255) are passed through.
          const int kexp = (int)(amax >> 7) - 127;
          if (amax < 0x7f80u && kexp >= 16) e_run = min(e_run, 15 - kexp);
          const float sc = exp2i(e_run);
#pragma unroll
          for (int i = 0; i < C::kConvVec; ++i) tile[ct + 128 * i] = bf16x8_to_f16x8_scaled(w[i], sc);
        }
        fence_proxy_async_smem();  // the generic writes become visible to the tensor core
        if (ct == 0) sb.v_exp[st] = e_run;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb.v_ready[st]);
        if (j == n0 - 1) e_t0 = e_run;
        if (j == n1 - 1) e_t1 = e_run;
      }
      if (!have_unit) break;
      pend_bh = bh;
      pend_mb = mb;
      pend_sp = sp;
      pend_uc = uc;
      pend_e[0] = e_t0;
      pend_e[1] = e_t1;
      kvb += 2 * n1;
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;\n" ::: "memory");
    if constexpr (C::kSplitP) {
      if ((warp == 12 || warp == 13) && lane == 0) {
        // ---------------------------------------------------------- MMA issue
        // Split P (D = 64): one issuing thread per Q tile (warp 12: tile 0,
        // warp 13: tile 1), on two SM sub-partitions whose issue slots the
        // softmax warps contend for; each tile's MMAs touch only its own tensor
        // memory, and K/V stages and Q buffers are released by one commit from
        // each thread.  Step j issues S_t for K_j as soon as the softmax has read
        // the previous S_t, then P_t V_{j-1} when the softmax pass ends, so the
        // next scores are computed while the softmax of the current ones runs.
        const int t = warp - 12;
        constexpr uint32_t idS = idesc_f32acc(true, 128, 128, false, false);  // bf16 Q, K
        constexpr uint32_t idO = idesc_f32acc(false, 128, D, false, true);    // fp16 P, V
        // Descriptor words: the low word carries the address / 16, stepped by
        // adds; the high word (stride 1024 B, 128-byte swizzle) is shared.
        const uint32_t dhi = sdesc_sw128_hi(1024);
        const uint32_t a_lo0 = sdesc_sw128_lo(smem_addr(sQ), 16) + t * (C::kTileBytes >> 4);
        const uint32_t k_lo0 = sdesc_sw128_lo(smem_addr(sKV), 16);
        const uint32_t v_lo0 = sdesc_sw128_lo(smem_addr(sKV), C::kChunkBytes);
        const uint32_t tS = tmem + (t ? C::kColS1 : C::kColS0);
        const uint32_t tP = tmem + (t ? C::kColP1 : C::kColP0);
        const uint32_t tO = tmem + (t ? C::kColO1 : C::kColO0);
        uint32_t p_phase = 0;
        uint32_t s_cnt = 0;  // S MMAs issued (split P: s_free phases)
        uint32_t kvb = 0;
        for (int uc = 0;; ++uc) {
          const int u = unit_at<kCausal>(tab, p, uc);
          if (u < 0) break;
          int bh, mb, sp, j0, n0, n1;
          unit_info<kCausal, kSplit>(p, u, bh, mb, sp, j0, n0, n1);
          const int n_t = t ? n1 : n0;
          const int qb = uc % C::kQBufs;  // Q buffer of this unit
          // With at most 128 queries tile 1 has no row: its thread issues no
          // MMA and keeps only its own tile's barriers.  It neither waits for
          // nor releases K/V stages and Q tiles (tile 0's commits alone do):
          // a releaser that issues nothing could run a whole ring ahead and
          // complete a stage's release while tile 0 still reads it.
          const bool idle = kHalf && t == 1;
#pragma unroll 1
          for (int j = 0; j <= n1; ++j) {
            const uint32_t kidx = kvb + 2 * j, vidx = kidx - 1;  // K_j and V_{j-1}
            const uint32_t ks = kidx % C::kStages, vs = vidx % C::kStages;
            const bool do_s = j < n_t, do_pv = j >= 1 && j <= n_t;
            if (do_s) {
              // S_t = Q_t K_j^T once K_j has landed and the softmax has read
              // the previous S_t
              if ((!idle && !mbar_wait(&sb.kv_full[ks], (kidx / C::kStages) & 1, abort_flag)) ||
                  (j == 0 && !idle &&
                   !mbar_wait(&sb.q_full[qb][t], (uc / C::kQBufs) & 1, abort_flag)) ||
                  (s_cnt > 0 && !mbar_wait(&sb.s_free[t], (s_cnt - 1) & 1, abort_flag))) {
                raise_abort(sb, p.err, kDevErrTimeout);
                goto mma_exit_split;
              }
              ++s_cnt;
              tc_fence_after_sync();
              if (!idle)
                issue_s<D>(tS, a_lo0 + qb * (2 * C::kTileBytes >> 4),
                           k_lo0 + ks * (C::kTileBytes >> 4), dhi, idS);
              umma_commit(&sb.s_full[t]);
            }
            if (do_pv) {
              // O_t (+)= P_t V_{j-1} once the softmax has written P_t
              if ((j == 1 && uc > 0 && !mbar_wait(&sb.o_free[t], (uc - 1) & 1, abort_flag)) ||
                  !mbar_wait(&sb.p_full[t], p_phase, abort_flag)) {
                raise_abort(sb, p.err, kDevErrTimeout);
                goto mma_exit_split;
              }
              p_phase ^= 1;
              tc_fence_after_sync();
              if (!idle) issue_pv(tO, tP, v_lo0 + vs * (C::kTileBytes >> 4), dhi, idO, j > 1 ? 1u : 0u);
              umma_commit(&sb.pv_done[t]);
              if (j == n_t) umma_commit(&sb.o_full[t]);
            }
            // this tile is done with K_j, V_{j-1} (and, after the unit's last S,
            // with its Q tile); every stage gets one commit from each issuing
            // thread
            if (!idle) {
              if (j < n1) umma_commit(&sb.kv_empty[ks]);
              if (j >= 1) umma_commit(&sb.kv_empty[vs]);
              if (j == n1 - 1) umma_commit(&sb.q_empty[qb]);
            }
          }
          kvb += 2 * n1;
        }
      mma_exit_split:
        // every MMA this thread issued must finish before the TMEM is freed
        umma_commit(&sb.mma_done[t]);
        {
          int never = 0;
          mbar_wait(&sb.mma_done[t], 0, &never);
        }
      }
    } else if (warp == 12 && lane == 0) {
      // ---------------------------------------------------------- MMA issue
      // Shared S/P (D = 128): one issuing thread.  Step j issues P0 V_{j-1},
      // S0 = Q0 K_j^T, then P1 V_{j-1}, S1 = Q1 K_j^T, so each softmax
      // warpgroup works while the other tile's two MMAs run, and a tile's
      // scores complete as one group (two independent issuers would
      // interleave the tiles' MMAs and delay both).  The softmax signals P_t
      // only once V_{j-1} is converted; this thread checks that K_j has
      // landed (one probe per step, usually already complete).  Keeping that
      // check here rather than in the softmax shortens the softmax's step by
      // a barrier probe: +4% on the causal workloads.
      constexpr uint32_t idS = idesc_f32acc(true, 128, 128, false, false);  // bf16 Q, K
      constexpr uint32_t idO = idesc_f32acc(false, 128, D, false, true);    // fp16 P, V
      // Descriptor words: the low word carries the address / 16, stepped by
      // adds; the high word (stride 1024 B, 128-byte swizzle) is shared.
      const uint32_t dhi = sdesc_sw128_hi(1024);
      const uint32_t q_lo = sdesc_sw128_lo(smem_addr(sQ), 16);
      const uint32_t k_lo0 = sdesc_sw128_lo(smem_addr(sKV), 16);
      const uint32_t v_lo0 = sdesc_sw128_lo(smem_addr(sKV), C::kChunkBytes);
      uint32_t p_phase[2] = {0, 0};
      uint32_t kvb = 0;
      for (int uc = 0;; ++uc) {
        const int u = unit_at<kCausal>(tab, p, uc);
        if (u < 0) break;
        int bh, mb, sp, j0, n0, n1;
        unit_info<kCausal, kSplit>(p, u, bh, mb, sp, j0, n0, n1);
#pragma unroll 1
        for (int j = 0; j <= n1; ++j) {
          const uint32_t kidx = kvb + 2 * j, vidx = kidx - 1;  // K_j and V_{j-1}
          const uint32_t ks = kidx % C::kStages, vs = vidx % C::kStages;
          bool k_ready = false;
          // Unrolled, so the per-tile phases stay in registers: a local-memory
          // access after a commit would stall this thread until the pipe drains.
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int n_t = t ? n1 : n0;
            const bool do_pv = j >= 1 && j <= n_t;
            const bool do_s = j < n_t;
            const uint32_t tS = tmem + (t ? C::kColS1 : C::kColS0);
            const uint32_t tO = tmem + (t ? C::kColO1 : C::kColO0);
            // The softmax signals P_t only after V_{j-1} is converted; K_j and
            // (for a unit's first S) the Q tile are waited for here.
            if (do_pv) {
              if ((j == 1 && uc > 0 && !mbar_wait(&sb.o_free[t], (uc - 1) & 1, abort_flag)) ||
                  !mbar_wait(&sb.p_full[t], p_phase[t], abort_flag)) {
                raise_abort(sb, p.err, kDevErrTimeout);
                goto mma_exit;
              }
              p_phase[t] ^= 1;
            }
            if (do_s) {
              if ((j == 0 && !mbar_wait(&sb.q_full[0][t], uc & 1, abort_flag)) ||
                  (!k_ready && !mbar_wait(&sb.kv_full[ks], (kidx / C::kStages) & 1, abort_flag))) {
                raise_abort(sb, p.err, kDevErrTimeout);
                goto mma_exit;
              }
              k_ready = true;
            }
            tc_fence_after_sync();
            if (do_pv) {
              // O_t (+)= P_t V_{j-1}: 16 keys (8 P columns, 2048 B of V) per MMA
              const uint32_t v_lo = v_lo0 + vs * (C::kTileBytes >> 4);
              umma_ts_w_rt(tO, tS, v_lo, dhi, idO, j > 1 ? 1u : 0u);
#pragma unroll
              for (int kk = 1; kk < 8; ++kk)
                umma_ts_w<1>(tO, tS + kk * 8, v_lo + kk * (2048 >> 4), dhi, idO);
            }
            if (do_s) {
              // S_t = Q_t K_j^T: 16 head-dim columns (32 B of a swizzled row) per MMA
              const uint32_t a_lo = q_lo + t * (C::kTileBytes >> 4);
              const uint32_t b_lo = k_lo0 + ks * (C::kTileBytes >> 4);
              umma_ss_w<0>(tS, a_lo, b_lo, dhi, idS);
#pragma unroll
              for (int kk = 1; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
                umma_ss_w<1>(tS, a_lo + off, b_lo + off, dhi, idS);
              }
              umma_commit(&sb.s_full[t]);
            }
            if (do_pv && j == n_t) umma_commit(&sb.o_full[t]);
          }
          if (j < n1) umma_commit(&sb.kv_empty[ks]);   // both tiles are done with K_j
          if (j >= 1) umma_commit(&sb.kv_empty[vs]);   // ... and with V_{j-1}
          if (j == n1 - 1) umma_commit(&sb.q_empty[0]);  // and with both Q tiles
        }
        kvb += 2 * n1;
      }
    mma_exit:
      // every MMA this thread issued must finish before the TMEM is freed
      umma_commit(&sb.mma_done[0]);
      {
        int never = 0;
        mbar_wait(&sb.mma_done[0], 0, &never);
      }

    }
    if (warp == 14 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      uint32_t kv_idx = 0;
      uint32_t q_loads = 0;  // Q tile pairs issued
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      for (int uc = 0;; ++uc) {
        const int u = unit_at<kCausal>(tab, p, uc);
        if (u < 0) break;
        int bh, mb, sp, j0, n0, n1;
        unit_info<kCausal, kSplit>(p, u, bh, mb, sp, j0, n0, n1);
        // Q buffer qb was last used kQBufs units ago
        const int qb = uc % C::kQBufs;
        if (uc >= C::kQBufs && !mbar_wait(&sb.q_empty[qb], (uc / C::kQBufs - 1) & 1, abort_flag)) {
          raise_abort(sb, p.err, kDevErrTimeout);
          goto load_exit;
        }
        for (int t = 0; t < 2; ++t) {
          mbar_arrive_expect_tx(&sb.q_full[qb][t], C::kTileBytes);
          for (int ch = 0; ch < C::kChunks; ++ch)
            tma_load_3d_hint(sQ + (2 * qb + t) * C::kTileBytes + ch * C::kChunkBytes, &tm_q,
                             &sb.q_full[qb][t],
                             ch * 64, mb * 256 + t * 128, bh, pol_q);
        }
        ++q_loads;
        for (int j = 0; j < n1; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t s = kv_idx % C::kStages;
            const uint32_t fill = kv_idx / C::kStages;
            if (p.test_drop_load && blockIdx.x == 0 && uc == 0 && j == 0 && kv == 0) {
              // Test hook: this load is never issued, so the MMA thread's
              // bounded wait for it runs out and the kernel reports a timeout.
              ++kv_idx;
              continue;
            }
            if (fill > 0 && !mbar_wait(&sb.kv_empty[s], (fill - 1) & 1, abort_flag)) {
              raise_abort(sb, p.err, kDevErrTimeout);
              goto load_exit;
            }
            mbar_arrive_expect_tx(&sb.kv_full[s], C::kTileBytes);
            const CUtensorMap *tm = kv ? &tm_v : &tm_k;
            for (int ch = 0; ch < C::kChunks; ++ch)
              tma_load_3d_hint(sKV + s * C::kTileBytes + ch * C::kChunkBytes, tm, &sb.kv_full[s],
                               ch * 64, (j0 + j) * 128, bh, pol_kv);
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
          if (p.test_drop_load && blockIdx.x == 0 && last == 0) continue;  // never issued
          mbar_wait(&sb.kv_full[s], (last / C::kStages) & 1, &never);
        }
        // the last load of each Q buffer
        for (uint32_t b = 0; b < (uint32_t)C::kQBufs && b < q_loads; ++b) {
          const uint32_t last = q_loads - 1 - ((q_loads - 1 - b) % C::kQBufs);  // load index
          mbar_wait(&sb.q_full[b][0], (last / C::kQBufs) & 1, &never);
          mbar_wait(&sb.q_full[b][1], (last / C::kQBufs) & 1, &never);
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
