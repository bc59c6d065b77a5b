// Backward pass of chunk-aligned window softmax attention on sm_103a: dq, dk, dv of sum(out * dout).
//
// The kept relation is symmetric. A frame key of chunk c is kept by exactly the frame queries of the chunks
// within r of c (the clamped window of c itself) and by every global query; a global key is kept by every query
// (VDN-Minimax-H3 window-attention article, section 一: chunk window plus fully connected globals). So the
// forward's work list serves the whole backward:
//   * read query-major (item rows = queries, segments = their keys) it drives the dq kernel;
//   * read key-major (item rows = keys, segments = the queries that keep them) it drives the dk / dv kernel.
// Both kernels recompute the probabilities from the forward's row log-sum-exp, P = exp(s / sqrt(D) - lse), with the
// scores s from tcgen05 MMAs, so no probability matrix is ever stored. Per (b, h), with c = 1 / sqrt(D):
//   Dvec_i = dout_i . out_i,  dP_ij = dout_i . v_j,  dS_ij = P_ij (dP_ij - Dvec_i),
//   dq_i = c sum_j dS_ij k_j,  dk_j = c sum_i dS_ij q_i,  dv_j = sum_i P_ij dout_i.
// The global rows' dq (and the global keys' dk, dv) are split along the other operand like the forward's global
// leg: each split writes an fp32 partial and bwd_sum_kernel adds the splits in a fixed order (deterministic).
//
// Every wait is bounded; on expiry a kernel latches an error in the plan's error word and unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "wa_device.cuh"
#include "wa_internal.h"
#include "wa_ptx.cuh"

namespace wa {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  const Item* items;
  int n_items;
  const float* lse;   // [B*H][L] natural-log row log-sum-exp of the forward
  const float* dvec;  // [B*H][L] dout_i . out_i
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* ws_dq;       // [B*H][G][n_splits][D] fp32 partials of the global rows (dq) / global keys (dk, dv)
  float* ws_dk;
  float* ws_dv;
  int* err;
  int64_t sb, sl, sh;
  int H, G, g0, L, n_splits;
  float c_log2;       // log2(e) / sqrt(D): turns a raw score into log2 units of the scaled score
  float scale;        // 1 / sqrt(D)
  int debug_flags;
  int* item_counter;  // ItemFeed counter (two ints, zero at launch); nullptr: static striding
  int bh_count;       // B * H (index checks of a debug build)
};

// First row of the j-th 128-row tile of an item's segments, and how many of its rows belong to the segment.
__device__ __forceinline__ int step_row(const Item& it, int j, int nt0, int* valid) {
  const int lo = j < nt0 ? it.s0_lo + j * kTileRows : it.s1_lo + (j - nt0) * kTileRows;
  const int hi = j < nt0 ? it.s0_hi : it.s1_hi;
  *valid = min(kTileRows, hi - lo);
  return lo;
}

// One 128-row tile of a [B, L, H, D] bf16 tensor: D / 64 boxes of 128 rows x 128 bytes (128-byte swizzle).
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar, int h, int row, int b) {
#pragma unroll
  for (int hf = 0; hf < D / 64; ++hf) tma_load_4d(dst + hf * kTileRows * 128, map, bar, hf * 64, h, row, b);
}

// Columns [c_lo, c_lo + NC) of one accumulator row (fp32 in TMEM) times `mul`: bf16 into `dst`, or fp32 into `part`
// when that is set (both already offset to column c_lo).
template <int NC>
__device__ __forceinline__ void store_cols(uint32_t t_acc, float mul, bool row_ok, __nv_bfloat16* dst, float* part) {
#pragma unroll
  for (int c0 = 0; c0 < NC; c0 += 32) {
    uint32_t o[32];
    tmem_ld_x32(t_acc + c0, o);  // warp-collective: every lane loads, only rows that exist store
    if (!row_ok) continue;
    if (part != nullptr) {
      float4* d4 = reinterpret_cast<float4*>(part + c0);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        d4[c] = make_float4(__uint_as_float(o[4 * c]) * mul, __uint_as_float(o[4 * c + 1]) * mul,
                            __uint_as_float(o[4 * c + 2]) * mul, __uint_as_float(o[4 * c + 3]) * mul);
    } else {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        d4[c] = make_uint4(pack_bf16(__uint_as_float(o[8 * c]) * mul, __uint_as_float(o[8 * c + 1]) * mul),
                           pack_bf16(__uint_as_float(o[8 * c + 2]) * mul, __uint_as_float(o[8 * c + 3]) * mul),
                           pack_bf16(__uint_as_float(o[8 * c + 4]) * mul, __uint_as_float(o[8 * c + 5]) * mul),
                           pack_bf16(__uint_as_float(o[8 * c + 6]) * mul, __uint_as_float(o[8 * c + 7]) * mul));
    }
  }
}

struct Smem {
  uint8_t* p;
  uint32_t base;
};

// The dynamic shared-memory window rounded up to 1024 bytes (the 128-byte swizzle repeats every 1024 bytes).
__device__ __forceinline__ Smem align_smem(uint8_t* raw) {
  uint8_t* s = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  return Smem{s, smem_u32(s)};
}

// Every thread: wait for all roles, then warp 0 frees the tensor memory (and the CTA's item claims are over).
__device__ __forceinline__ void teardown(uint32_t tmem, int warp, const ItemFeed& feed) {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) feed.finish();
  if (warp == 0) {
    __syncwarp();  // tcgen05.dealloc is warp-collective: reconverge after the role branches
    tmem_dealloc(tmem, 512);
  }
}

// Elementwise warps and column groups. Warp w < 4 kCG works on TMEM lanes 32 (w % 4) .. +31 (one row of the tile
// per thread) and on the 128 / kCG columns of column group w / 4; so kCG warps share each sub-partition and hide
// one another's latency. A group packs its bf16 results (P, dS) into the first half of its own column range, so no
// group overwrites columns another group has yet to read; the MMAs that take them from TMEM address each 16-column
// block accordingly (tmem_a_block).
constexpr int kCG = 2;
constexpr int kCW = kTileRows / kCG;            // columns per group
constexpr int kEwWarps = 4 * kCG;
// Two MMA-issuing warps on different sub-partitions (the dq kernel uses both): an issuing warp shares its
// sub-partition with busy elementwise warps, which slows its stream of tcgen05.mma below the tensor core's rate, so
// the dq kernel splits its products between two warps. Each TMEM region is written and read by MMAs of one warp
// only, so their in-order execution covers every hazard.
constexpr int kMmaWarpX = kEwWarps, kMmaWarpY = kEwWarps + 1, kLoadWarp = kEwWarps + 2;
constexpr int kBwdThreads = 32 * (kEwWarps + 3);

// TMEM column offset of the bf16 A-operand block kk (16 rows of the reduction dimension: 8 packed columns) inside a
// 128-column region whose groups each packed their half.
__host__ __device__ constexpr uint32_t tmem_a_block(int kk) {
  return (uint32_t)((kk * 16) / kCW * kCW + (kk % (kCW / 16)) * 8);
}

// First column and count of a group's share of a D-column accumulator row in the epilogue (at least 32 columns).
template <int D>
struct EpiCols {
  static constexpr int kCols = D / kCG >= 32 ? D / kCG : 32;
};

// =====================================================================================================================
// dq kernel: query-major. Each work item's query tiles are processed one after the other ("sub-items"), each against
// the item's key segments, one 128-key tile per step.
//   warps 0 .. 4 kCG - 1  elementwise: P = 2^(s c' - lse'), dS = P (dP - Dvec) as bf16, one row and one column
//                          group per thread
//   warp 4 kCG            MMA issuer X (whole warp, one elected lane issues): S = Q K^T and dq += dS K
//   warp 4 kCG + 1        MMA issuer Y (whole warp, one elected lane issues): dP = dout V^T
//   warp 4 kCG + 2        TMA producer (whole warp; lane 0 claims items and issues the copies): Q and dout tiles of
//                          the sub-item, rings of key and value tiles; the lanes zero the rows of a segment's last key
//                          tile that lie past the segment's end before releasing it
// TMEM: R0, R1 [0,256) score buffers (step n's S in R[n % 2]; dS, packed bf16, overwrites the front of each group's
// columns and is the A operand of dS.K straight from TMEM), R2 [256,384) dP, R3 [384, 384+D) the dq accumulator.
// The next step's S and dP are issued before this step's dS.K, so the elementwise work of a step overlaps the
// tensor core's.
// =====================================================================================================================
template <int D>
struct DqCfg {
  static constexpr int kTileBytes = kTileRows * D * 2;
  static constexpr int kKSlots = 3, kVSlots = 2;
  static constexpr int kQOff = 0, kDOOff = kTileBytes;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKSlots * kTileBytes;
  static constexpr int kBarOff = kVOff + kVSlots * kTileBytes;
  // q_full, q_empty, s_full[2], p_full[2], dp_free, o_full, drain_x, drain_y, then the rings' full / empty barriers,
  // k_land (a segment's last key tile lands there and is cleaned before its full barrier is arrived), then the
  // work-item ring's (ItemFeed)
  static constexpr int kNumBars = 10 + 2 * kKSlots + 2 * kVSlots + 1 + 2 * kItemRingSlots;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM address, abort flag, 2 spare words, item ring
  static constexpr int kSmemBytes = kMiscOff + 16 + 4 * kItemRingSlots + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);  // both operands K-major
  static constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, D, 0, 1);   // dS from TMEM, key tile MN-major
};

// dS = P (dP - Dvec) for one thread's kCW columns of one row, packed to bf16 over the front of those columns.
// kMask: columns at or past `valid` (a segment's ragged last tile) get dS = 0.
template <bool kMask>
__device__ __forceinline__ void dq_row_step(uint32_t tS, const uint32_t (&dpr)[kCW / 32][32], float c_log2,
                                            float neg_lse2, float drow, int col0, int valid) {
#pragma unroll
  for (int ch = 0; ch < kCW / 32; ++ch) {
    uint32_t sr[32], pk[16];
    tmem_ld_x32(tS + 32 * ch, sr);
#pragma unroll
    for (int c = 0; c < 16; ++c) {  // packed pairs: one f32x2 instruction per two columns
      float x0, x1, t0, t1, d0, d1;
      fma2(x0, x1, __uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1]), c_log2, c_log2, neg_lse2, neg_lse2);
      const float p0 = ex2(x0);
      const float p1 = ex2(x1);
      add2(t0, t1, __uint_as_float(dpr[ch][2 * c]), __uint_as_float(dpr[ch][2 * c + 1]), -drow, -drow);
      mul2(d0, d1, p0, p1, t0, t1);
      if (kMask) {  // selected, not multiplied: dP there comes from value rows outside the segment (maybe not finite)
        const int col = col0 + 32 * ch + 2 * c;
        d0 = col < valid ? d0 : 0.f;
        d1 = col + 1 < valid ? d1 : 0.f;
      }
      pk[c] = pack_bf16(d0, d1);
    }
    tmem_st_x16(tS + 16 * ch, pk);
  }
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    wa_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const BwdParams prm) {
  using C = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem sm = align_smem(smem_raw);
  const uint32_t sQ = sm.base + C::kQOff, sDO = sm.base + C::kDOOff, sK = sm.base + C::kKOff, sV = sm.base + C::kVOff;
  const uint32_t bar = sm.base + C::kBarOff;
  const uint32_t b_qfull = bar, b_qempty = bar + 8, b_dpfree = bar + 48, b_ofull = bar + 56, b_drain_x = bar + 64,
                 b_drain_y = bar + 72;
  auto b_sfull = [&](uint32_t n) { return bar + 16 + 8 * (n & 1); };
  auto b_pfull = [&](uint32_t n) { return bar + 32 + 8 * (n & 1); };
  auto b_kfull = [&](uint32_t s) { return bar + 8 * (10 + s); };
  auto b_kempty = [&](uint32_t s) { return bar + 8 * (10 + C::kKSlots + s); };
  auto b_vfull = [&](uint32_t s) { return bar + 8 * (10 + 2 * C::kKSlots + s); };
  auto b_vempty = [&](uint32_t s) { return bar + 8 * (10 + 2 * C::kKSlots + C::kVSlots + s); };
  const uint32_t b_kland = bar + 8 * (10 + 2 * C::kKSlots + 2 * C::kVSlots);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm.p + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm.p + C::kMiscOff + 4);
  const ItemFeed feed{prm.item_counter, prm.n_items, reinterpret_cast<volatile int*>(sm.p + C::kMiscOff + 16),
                      bar + 8 * (C::kNumBars - 2 * kItemRingSlots)};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* err = prm.err;

  if (tid == 0) {
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 2);  // both issuers: the last S (reads Q) and the last dP (reads dout) of the sub-item
    for (uint32_t n = 0; n < 2; ++n) {
      mbar_init(b_sfull(n), 2);         // S from issuer X, dP from issuer Y
      mbar_init(b_pfull(n), kEwWarps);  // one arrival per elementwise warp
    }
    mbar_init(b_dpfree, kEwWarps);
    mbar_init(b_ofull, 1);
    mbar_init(b_drain_x, 1);
    mbar_init(b_drain_y, 1);
    feed.init(kEwWarps + 2);  // item consumers: issuers X and Y, the elementwise warps
    for (int s = 0; s < C::kKSlots; ++s) {
      mbar_init(b_kfull(s), 1);
      mbar_init(b_kempty(s), 1);
    }
    for (int s = 0; s < C::kVSlots; ++s) {
      mbar_init(b_vfull(s), 1);
      mbar_init(b_vempty(s), 1);
    }
    mbar_init(b_kland, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tR2 = tmem + 256, tR3 = tmem + 384;

  if (warp == kLoadWarp) {
    // ---------------------------------------------------------------------------------------- TMA producer
    // The whole warp runs the loop (waits are warp-wide); lane 0 claims the items and issues the copies. A
    // segment's last key tile lands on k_land: the 32 lanes zero its rows past the segment's end (keys outside the
    // rows' kept sets: their dS is 0, but 0 x Inf would be NaN in dS.K) before k_full is arrived.
    {
      const bool leader = lane == 0;
      uint32_t k_n = 0, v_n = 0, q_n = 0, kl_n = 0;  // kl_n: segment-final key tiles landed on k_land
      bool ok = true, dropped = false;
      for (uint32_t n = 0; ok; ++n) {
        const int idx = feed.claim_warp(n, abort_flag, err, ok);
        if (idx < 0) break;
        const Item it = load_item(prm.items, idx);
#ifdef WA_DEBUG
        if (!item_in_bounds(it, ItemBounds{prm.bh_count, prm.L, prm.g0, prm.G, prm.n_splits})) {
          if (leader) {
            atomicOr(err, kErrBounds);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
#endif
        const int b = it.bh / prm.H, h = it.bh % prm.H;
        const int ntq = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
        const int nt0 = seg_tiles(it.s0_lo, it.s0_hi);
        const int nt = nt0 + seg_tiles(it.s1_lo, it.s1_hi);
        for (int t = 0; t < ntq && ok; ++t) {
          ok = mbar_wait_warp(b_qempty, (q_n & 1) ^ 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          if (!ok) break;
          if (leader) {
            if ((prm.debug_flags & 2) && !dropped && blockIdx.x == 0) {
              dropped = true;  // fault injection for the watchdog test: this sub-item's query tiles never arrive
            } else {
              mbar_arrive_expect_tx(b_qfull, 2 * C::kTileBytes);
              load_tile<D>(sQ, &tm_q, b_qfull, h, it.q_lo + t * kTileRows, b);
              load_tile<D>(sDO, &tm_do, b_qfull, h, it.q_lo + t * kTileRows, b);
            }
          }
          q_n++;
          for (int j = 0; j < nt && ok; ++j) {
            int valid;
            const int row = step_row(it, j, nt0, &valid);
            const bool tail = valid < kTileRows;
            const uint32_t ks = k_n % C::kKSlots, vs = v_n % C::kVSlots;
            ok = mbar_wait_warp(b_kempty(ks), ((k_n / C::kKSlots) & 1) ^ 1, abort_flag, err, kErrTimeout,
                                kWaitLimitNs);
            if (!ok) break;
            if (leader) {
              const uint32_t kbar = tail ? b_kland : b_kfull(ks);
              mbar_arrive_expect_tx(kbar, C::kTileBytes);
              load_tile<D>(sK + ks * C::kTileBytes, &tm_k, kbar, h, row, b);
            }
            k_n++;
            ok = mbar_wait_warp(b_vempty(vs), ((v_n / C::kVSlots) & 1) ^ 1, abort_flag, err, kErrTimeout,
                                kWaitLimitNs);
            if (ok && leader) {
              mbar_arrive_expect_tx(b_vfull(vs), C::kTileBytes);
              load_tile<D>(sV + vs * C::kTileBytes, &tm_v, b_vfull(vs), h, row, b);
            }
            if (ok) v_n++;
            if (tail) {  // the value copy is already on its way; now clean the key tile and release it
              const bool landed = mbar_wait_warp(b_kland, kl_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
              kl_n++;
              if (landed) zero_tile_rows(sK + ks * C::kTileBytes, D / 64, valid, lane);
              if (leader) mbar_arrive(b_kfull(ks));  // in place of the copy's arrival (also when unwinding)
              ok = ok && landed;
            }
          }
        }
      }
      if (!ok && leader) {  // let the copies already issued land before the CTA's shared memory goes away
        for (uint32_t n = k_n > (uint32_t)C::kKSlots ? k_n - C::kKSlots : 0; n < k_n; ++n)
          mbar_wait_drain(b_kfull(n % C::kKSlots), (n / C::kKSlots) & 1, kDrainLimitNs);
        for (uint32_t n = v_n > (uint32_t)C::kVSlots ? v_n - C::kVSlots : 0; n < v_n; ++n)
          mbar_wait_drain(b_vfull(n % C::kVSlots), (n / C::kVSlots) & 1, kDrainLimitNs);
        if (kl_n) mbar_wait_drain(b_kland, (kl_n - 1) & 1, kDrainLimitNs);
        if (q_n) mbar_wait_drain(b_qfull, (q_n - 1) & 1, kDrainLimitNs);
      }
    }
  } else if (warp == kMmaWarpX || warp == kMmaWarpY) {
    // ---------------------------------------------------------------------------------------- MMA issuers
    // X: S(n) = Q K_n^T into R[n % 2] and dq += dS(n) K_n; in its order S(n+1) comes before dq(n) and S(n+2) after
    //    it, so the score buffer dq(n) reads is rewritten only behind it.
    // Y: dP(n) = dout V_n^T into R2, once the elementwise warps have read dP(n-1).
    const bool is_x = warp == kMmaWarpX;
    {  // the whole warp runs the issue loop; one elected lane issues (issue model in wa_ptx.cuh)
      uint32_t k_n = 0, v_n = 0, q_n = 0, gs = 0;  // gs: steps of all earlier sub-items
      bool ok = true;
      const uint64_t dq_ = sdesc_sw128(sQ, 16, 1024), ddo = sdesc_sw128(sDO, 16, 1024);
      const uint64_t dk_ = sdesc_sw128(sK, 16, 1024), dv_ = sdesc_sw128(sV, 16, 1024);
      const uint64_t dk_mn = sdesc_sw128(sK, kTileRows * 128, 1024);  // key tiles as the MN-major B of dS.K
      const uint32_t hi = (uint32_t)(dq_ >> 32);                      // common high word of every descriptor
      // acc[tmem] = A B^T over the head dimension, both K-major (S = Q K^T, dP = dout V^T)
      auto issue_nt = [&](uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * kTileRows * 128 + (kk % 4) * 32) >> 4;
          mma_ss(d_tmem, a_lo + off, b_lo + off, hi, C::kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      for (uint32_t n = 0; ok; ++n) {
        const int idx = feed.fetch(n, abort_flag, err, ok);
        if (idx < 0) break;
        const Item it = load_item(prm.items, idx);
        const int ntq = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
        const int nt = seg_tiles(it.s0_lo, it.s0_hi) + seg_tiles(it.s1_lo, it.s1_hi);
        for (int t = 0; t < ntq && ok; ++t) {
          ok = mbar_wait_warp(b_qfull, q_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          q_n++;
          if (!ok) break;
          if (is_x) {
            uint32_t kcur = k_n % C::kKSlots;
            ok = mbar_wait_warp(b_kfull(kcur), (k_n / C::kKSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
            k_n++;
            if (!ok) break;
            tc_fence_after();
            issue_nt(tmem + 128 * (gs & 1), (uint32_t)dq_, (uint32_t)dk_ + ((kcur * C::kTileBytes) >> 4));
            mma_commit(b_sfull(gs));
            if (nt == 1) mma_commit(b_qempty);
            for (int j = 0; j < nt && ok; ++j) {
              const uint32_t n = gs + j;
              uint32_t knext = 0;
              if (j + 1 < nt) {
                knext = k_n % C::kKSlots;
                ok = mbar_wait_warp(b_kfull(knext), (k_n / C::kKSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
                k_n++;
                if (!ok) break;
                tc_fence_after();
                issue_nt(tmem + 128 * ((n + 1) & 1), (uint32_t)dq_, (uint32_t)dk_ + ((knext * C::kTileBytes) >> 4));
                mma_commit(b_sfull(n + 1));
                if (j + 1 == nt - 1) mma_commit(b_qempty);  // every S of the sub-item has been issued
              }
              ok = mbar_wait_warp(b_pfull(n), (n >> 1) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);  // dS(n) ready
              if (!ok) break;
              tc_fence_after();
              // dq += dS(n) K_n: dS from TMEM (16 keys per MMA, from R[n % 2]), K_n MN-major
              const uint32_t kb = (uint32_t)dk_mn + ((kcur * C::kTileBytes) >> 4);
#pragma unroll
              for (int kk = 0; kk < kTileRows / 16; ++kk)
                mma_ts(tR3, tmem + 128 * (n & 1) + tmem_a_block(kk), kb + ((kk * 2048) >> 4), hi, C::kIdescDQ,
                       (j > 0 || kk > 0) ? 1u : 0u);
              mma_commit(b_kempty(kcur));
              kcur = knext;
            }
            if (!ok) break;
            mma_commit(b_ofull);
          } else {
            for (int j = 0; j < nt && ok; ++j) {
              const uint32_t n = gs + j;
              if (n > 0) {  // the elementwise warps have read dP(n-1) out of R2
                ok = mbar_wait_warp(b_dpfree, (n - 1) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
                if (!ok) break;
              }
              const uint32_t vs = v_n % C::kVSlots;
              ok = mbar_wait_warp(b_vfull(vs), (v_n / C::kVSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
              v_n++;
              if (!ok) break;
              tc_fence_after();
              issue_nt(tR2, (uint32_t)ddo, (uint32_t)dv_ + ((vs * C::kTileBytes) >> 4));
              mma_commit(b_sfull(n));
              mma_commit(b_vempty(vs));
              if (j == nt - 1) mma_commit(b_qempty);  // every dP of the sub-item has been issued
            }
          }
          gs += nt;
        }
      }
      const uint32_t drain = is_x ? b_drain_x : b_drain_y;
      mma_commit(drain);
      mbar_wait_drain(drain, 0, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else if (warp < kEwWarps) {
    // ---------------------------------------------------------------------------------------- elementwise
    const int r = 32 * (warp & 3) + lane;  // query row in the tile == TMEM lane
    const int col0 = kCW * (warp >> 2);   // this thread's key columns [col0, col0 + kCW)
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    uint32_t o_n = 0, gs = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int idx = feed.fetch(n, abort_flag, err, ok);
      if (idx < 0) break;
      const Item it = load_item(prm.items, idx);
      const int ntq = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
      const int nt0 = seg_tiles(it.s0_lo, it.s0_hi);
      const int nt = nt0 + seg_tiles(it.s1_lo, it.s1_hi);
      for (int t = 0; t < ntq && ok; ++t) {
        const int row = it.q_lo + t * kTileRows + r;
        const bool in_seq = row < prm.L;
        const float neg_lse2 = in_seq ? -__ldg(prm.lse + (int64_t)it.bh * prm.L + row) * kLog2e : 0.f;
        const float drow = in_seq ? __ldg(prm.dvec + (int64_t)it.bh * prm.L + row) : 0.f;
        for (int j = 0; j < nt; ++j) {
          const uint32_t n = gs + j;
          int valid;
          step_row(it, j, nt0, &valid);
          ok = mbar_wait(b_sfull(n), (n >> 1) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          uint32_t dpr[kCW / 32][32];
#pragma unroll
          tmem_ld_x64(tR2 + lane_base + col0, *reinterpret_cast<uint32_t(*)[kCW]>(&dpr[0][0]));  // one wait
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_dpfree);
          const uint32_t tS = tmem + lane_base + 128 * (n & 1) + col0;
          if (valid >= kTileRows)
            dq_row_step<false>(tS, dpr, prm.c_log2, neg_lse2, drow, col0, valid);
          else
            dq_row_step<true>(tS, dpr, prm.c_log2, neg_lse2, drow, col0, valid);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_pfull(n));
        }
        if (!ok) break;
        ok = mbar_wait(b_ofull, o_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        o_n++;
        if (!ok) break;
        tc_fence_after();
        constexpr int EC = EpiCols<D>::kCols;
        const int c_lo = EC * (warp >> 2);
        if (c_lo < D) {
          const bool row_ok = row < it.q_hi;
          const int b = it.bh / prm.H, h = it.bh % prm.H;
          if (it.split < 0) {
            store_cols<EC>(tR3 + lane_base + c_lo, prm.scale, row_ok,
                           prm.dq + (int64_t)b * prm.sb + (int64_t)row * prm.sl + (int64_t)h * prm.sh + c_lo, nullptr);
          } else {
            const int64_t slot = ((int64_t)it.bh * prm.G + (row - prm.g0)) * prm.n_splits + it.split;
            store_cols<EC>(tR3 + lane_base + c_lo, prm.scale, row_ok, nullptr, prm.ws_dq + slot * D + c_lo);
          }
        }
        tc_fence_before();
        gs += nt;
      }
    }
  }
  teardown(tmem, warp, feed);
}

// =====================================================================================================================
// dk / dv kernel: key-major. Item rows are read as keys (one 128-key tile per sub-item, resident for the sub-item)
// and the item's segments as the queries that keep them, streamed one 128-query tile per step.
//   warps 0 .. 4 kCG - 1  elementwise, one key (TMEM lane) and one group of query columns per thread.
//                          Phase A: P^T = 2^(s c' - lse'_col) -> bf16 into TMEM. Phase B: dS^T = P^T (dP^T - Dvec_col)
//                          -> bf16 into TMEM. P stays in fp32 registers between the phases.
//   warp 4 kCG            MMA issuer: S^T = K Q^T, dP^T = V dout^T, dv += P^T dout, dk += dS^T Q
//   warp 4 kCG + 1        query-tile loader (the dq kernel's second issuer; both kernels share one launch shape):
//                          lane 0 issues the TMA copies of the query tiles into their own ring; the lanes zero the
//                          rows of a segment's last tile that lie past the segment's end before releasing it
//   warp 4 kCG + 2        loads (all lanes): lane 0 issues the TMA copies (the key / value tiles of the sub-item and
//                          a ring of dout tiles); every lane then stages 4 query columns' values (log2-domain lse,
//                          Dvec, both negated) into the dout slot. Columns past the segment get -lse' = -inf and
//                          -Dvec = 0, and (as for the query tiles) the rows of a segment's last dout tile past the
//                          segment's end are zeroed before release, so their P and dS are exactly 0 and every
//                          product with them is 0, with no masking in the elementwise code.
// TMEM: S^T [0,128) (P^T packed over the front of each group's columns), dP^T [128,256) (dS^T likewise),
// dv [256, 256+D), dk [384, 384+D). Issue order per step n: dv(n) after P^T(n) is written, then S^T(n+1); dk(n)
// after dS^T(n), then dP^T(n+1). So the tensor core computes dv(n) and S^T(n+1) while the elementwise warps work on
// dS^T(n), and dk(n) and dP^T(n+1) while they start P^T(n+1).
// =====================================================================================================================
template <int D>
struct DkvCfg {
  static constexpr int kTileBytes = kTileRows * D * 2;
  // Two rings, each filled by its own loader warp: query tiles (read by S^T(j) and dk(j)) and dout tiles with the
  // per-column values (read by dP^T(j), dv(j) and the elementwise phases). A query tile's slot is free once dk of
  // the tile kQSlots steps back has completed, early enough for the copy to land before S^T needs it.
  static constexpr int kQSlots = D == 128 ? 3 : 4;
  static constexpr int kDSlots = D == 128 ? 2 : 3;
  static constexpr int kKOff = 0, kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;
  static constexpr int kDOOff = kQOff + kQSlots * kTileBytes;
  // per dout slot: -lse'[128] then -Dvec[128], fp32 (negated so that the elementwise warps add them with packed
  // f32x2 instructions)
  static constexpr int kColOff = kDOOff + kDSlots * kTileBytes;
  static constexpr int kColBytes = 64 * 16;
  static constexpr int kBarOff = kColOff + kDSlots * kColBytes;
  // kv_full, kv_empty, s_full, p_full, dp_full, ds_full, o_full, drain_x, q_full[], q_empty[], d_full[], d_empty[],
  // q_land, d_land (a segment's last query / dout tile lands there and is cleaned before its full barrier is
  // arrived), then the ItemFeed's 2 kItemRingSlots
  static constexpr int kNumBars = 8 + 2 * kQSlots + 2 * kDSlots + 2 + 2 * kItemRingSlots;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM address, abort flag, 2 spare words, item ring
  static constexpr int kUsed = kMiscOff + 16 + 4 * kItemRingSlots;
  // Room to realign the window to 1024 bytes (the 128-byte swizzle repeats every 1024 bytes): a full 1024 where it
  // fits, else what is left of the 227 KB (D = 128: 768 bytes, so any window on a 256-byte boundary still works).
  // A window further off than that is reported at launch (WA_ERR_DEVICE_BOUNDS) and nothing is computed.
  static constexpr int kSlack = kUsed + 1024 <= 232448 ? 1024 : (232448 - kUsed) / 16 * 16;
  static constexpr int kSmemBytes = kUsed + kSlack;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);  // both operands K-major
  static constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, 0, 1);  // A from TMEM, query-side tile MN-major
};

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    wa_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const BwdParams prm) {
  using C = DkvCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (((0u - smem_u32(smem_raw)) & 1023u) > (uint32_t)C::kSlack) {  // no room to realign: report, touch nothing
    if (threadIdx.x == 0) {
      atomicOr(prm.err, kErrBounds);
      ItemFeed{prm.item_counter, prm.n_items, nullptr, 0}.finish();  // keeps the claim counter rewound
    }
    return;
  }
  const Smem sm = align_smem(smem_raw);
  const uint32_t sK = sm.base + C::kKOff, sV = sm.base + C::kVOff, sQ = sm.base + C::kQOff, sDO = sm.base + C::kDOOff;
  const uint32_t sCol = sm.base + C::kColOff;
  const uint32_t bar = sm.base + C::kBarOff;
  const uint32_t b_kvfull = bar, b_kvempty = bar + 8, b_sfull = bar + 16, b_pfull = bar + 24, b_dpfull = bar + 32,
                 b_dsfull = bar + 40, b_ofull = bar + 48, b_drain_x = bar + 56;
  auto b_qfull = [&](uint32_t s) { return bar + 8 * (8 + s); };
  auto b_qempty = [&](uint32_t s) { return bar + 8 * (8 + C::kQSlots + s); };
  auto b_dfull = [&](uint32_t s) { return bar + 8 * (8 + 2 * C::kQSlots + s); };
  auto b_dempty = [&](uint32_t s) { return bar + 8 * (8 + 2 * C::kQSlots + C::kDSlots + s); };
  const uint32_t b_qland = bar + 8 * (8 + 2 * C::kQSlots + 2 * C::kDSlots);
  const uint32_t b_dland = b_qland + 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm.p + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm.p + C::kMiscOff + 4);
  const ItemFeed feed{prm.item_counter, prm.n_items, reinterpret_cast<volatile int*>(sm.p + C::kMiscOff + 16),
                      bar + 8 * (C::kNumBars - 2 * kItemRingSlots)};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* err = prm.err;

  if (tid == 0) {
    mbar_init(b_kvfull, 1);
    mbar_init(b_kvempty, 1);
    mbar_init(b_sfull, 1);
    mbar_init(b_pfull, kEwWarps);
    mbar_init(b_dpfull, 1);
    mbar_init(b_dsfull, kEwWarps);
    mbar_init(b_ofull, 1);
    mbar_init(b_drain_x, 1);
    for (int s = 0; s < C::kQSlots; ++s) {
      mbar_init(b_qfull(s), 1);   // the copy's expect-tx arrival
      mbar_init(b_qempty(s), 1);  // the MMA commit after dk(j)
    }
    for (int s = 0; s < C::kDSlots; ++s) {
      mbar_init(b_dfull(s), 1 + 32);         // the copy's expect-tx arrival + one per loader lane (column values)
      mbar_init(b_dempty(s), 1 + kEwWarps);  // the MMA commit after dv(j) + one per elementwise warp
    }
    mbar_init(b_qland, 1);
    mbar_init(b_dland, 1);
    feed.init(kEwWarps + 2);  // item consumers: the issuer, the query-tile loader, the elementwise warps
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;

  if (warp == kLoadWarp) {
    // ---------------------------------------------------------------- key/value, dout and column-value loader
    uint32_t kv_n = 0, d_n = 0, dl_n = 0;  // dl_n: segment-final dout tiles landed on d_land
    bool ok = true, dropped = false;
    for (uint32_t n = 0; ok; ++n) {
      const int idx = feed.claim_warp(n, abort_flag, err, ok);
      if (idx < 0) break;
      const Item it = load_item(prm.items, idx);
#ifdef WA_DEBUG
      if (!item_in_bounds(it, ItemBounds{prm.bh_count, prm.L, prm.g0, prm.G, prm.n_splits})) {
        if (lane == 0) {
          atomicOr(err, kErrBounds);
          *abort_flag = 1;
        }
        ok = false;
        break;
      }
#endif
      const int b = it.bh / prm.H, h = it.bh % prm.H;
      const int ntk = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
      const int nt0 = seg_tiles(it.s0_lo, it.s0_hi);
      const int nt = nt0 + seg_tiles(it.s1_lo, it.s1_hi);
      const float* lse_bh = prm.lse + (int64_t)it.bh * prm.L;
      const float* dv_bh = prm.dvec + (int64_t)it.bh * prm.L;
      for (int t = 0; t < ntk && ok; ++t) {
        ok = mbar_wait(b_kvempty, (kv_n & 1) ^ 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(b_kvfull, 2 * C::kTileBytes);
          load_tile<D>(sK, &tm_k, b_kvfull, h, it.q_lo + t * kTileRows, b);
          load_tile<D>(sV, &tm_v, b_kvfull, h, it.q_lo + t * kTileRows, b);
        }
        kv_n++;
        for (int j = 0; j < nt && ok; ++j) {
          int valid;
          const int row = step_row(it, j, nt0, &valid);
          // this lane's 4 query columns: loads issued before the wait so that their latency hides behind it
          float l4[4], d4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = 4 * lane + i;
            l4[i] = c < valid ? -__ldg(lse_bh + row + c) * kLog2e : -INFINITY;
            d4[i] = c < valid ? -__ldg(dv_bh + row + c) : 0.f;
          }
          const uint32_t ds = d_n % C::kDSlots;
          ok = mbar_wait(b_dempty(ds), ((d_n / C::kDSlots) & 1) ^ 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          // A segment's last tile lands on d_land: its rows past the segment's end (queries that do not keep these
          // keys) are zeroed before d_full is arrived, so every product with them is exactly 0 (their P and dS are
          // 0: -lse' = -inf and -Dvec = 0 below), whatever those rows hold.
          const bool tail = valid < kTileRows;
          if (lane == 0) {
            const uint32_t dbar = tail ? b_dland : b_dfull(ds);
            mbar_arrive_expect_tx(dbar, C::kTileBytes);
            if ((prm.debug_flags & 4) && !dropped && blockIdx.x == 0)
              dropped = true;  // fault injection for the watchdog test: bytes expected, no copy issued
            else
              load_tile<D>(sDO + ds * C::kTileBytes, &tm_do, dbar, h, row, b);
          }
          const uint32_t cb = sCol + ds * C::kColBytes + 16 * lane;
          sts_f4(cb, make_float4(l4[0], l4[1], l4[2], l4[3]));
          sts_f4(cb + 512, make_float4(d4[0], d4[1], d4[2], d4[3]));
          if (tail) {
            ok = mbar_wait(b_dland, dl_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
            ok = __all_sync(0xffffffffu, ok);
            dl_n++;
            if (ok) zero_tile_rows(sDO + ds * C::kTileBytes, D / 64, valid, lane);
            if (lane == 0) mbar_arrive(b_dfull(ds));  // in place of the copy's arrival
          }
          mbar_arrive(b_dfull(ds));  // release: the column values are visible to whoever waits on d_full
          d_n++;
        }
      }
    }
    if (!ok && lane == 0) {
      if (kv_n) mbar_wait_drain(b_kvfull, (kv_n - 1) & 1, kDrainLimitNs);
      if (dl_n) mbar_wait_drain(b_dland, (dl_n - 1) & 1, kDrainLimitNs);
      for (uint32_t n = d_n > (uint32_t)C::kDSlots ? d_n - C::kDSlots : 0; n < d_n; ++n)
        mbar_wait_drain(b_dfull(n % C::kDSlots), (n / C::kDSlots) & 1, kDrainLimitNs);
    }
  } else if (warp == kMmaWarpY) {
    // ------------------------------------------------------------------------------------- query-tile loader
    uint32_t q_n = 0, ql_n = 0;  // ql_n: segment-final query tiles landed on q_land
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int idx = feed.fetch(n, abort_flag, err, ok);
      if (idx < 0) break;
      const Item it = load_item(prm.items, idx);
      const int b = it.bh / prm.H, h = it.bh % prm.H;
      const int ntk = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
      const int nt0 = seg_tiles(it.s0_lo, it.s0_hi);
      const int nt = nt0 + seg_tiles(it.s1_lo, it.s1_hi);
      for (int t = 0; t < ntk && ok; ++t) {
        for (int j = 0; j < nt && ok; ++j) {
          int valid;
          const int row = step_row(it, j, nt0, &valid);
          const uint32_t qs = q_n % C::kQSlots;
          ok = mbar_wait(b_qempty(qs), ((q_n / C::kQSlots) & 1) ^ 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          // a segment's last tile: cleaned like the dout tiles (rows past the segment's end become zeros)
          const bool tail = valid < kTileRows;
          if (lane == 0) {
            const uint32_t qbar = tail ? b_qland : b_qfull(qs);
            mbar_arrive_expect_tx(qbar, C::kTileBytes);
            load_tile<D>(sQ + qs * C::kTileBytes, &tm_q, qbar, h, row, b);
          }
          q_n++;
          if (tail) {
            ok = mbar_wait(b_qland, ql_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
            ok = __all_sync(0xffffffffu, ok);
            ql_n++;
            if (ok) zero_tile_rows(sQ + qs * C::kTileBytes, D / 64, valid, lane);
            if (lane == 0) mbar_arrive(b_qfull(qs));  // in place of the copy's arrival
          }
        }
      }
    }
    if (!ok && lane == 0) {
      for (uint32_t n = q_n > (uint32_t)C::kQSlots ? q_n - C::kQSlots : 0; n < q_n; ++n)
        mbar_wait_drain(b_qfull(n % C::kQSlots), (n / C::kQSlots) & 1, kDrainLimitNs);
      if (ql_n) mbar_wait_drain(b_qland, (ql_n - 1) & 1, kDrainLimitNs);
    }
  } else if (warp == kMmaWarpX) {
    // ------------------------------------------------------------------------------------------ MMA issuer
    // One thread, in the order dv(j), S^T(j+1), dk(j), dP^T(j+1): the elementwise warps' next scores are queued
    // right behind the product that frees their region. (A second issuer thread was measured slower here: the
    // chain dv(j) -> S^T(j+1) -> phase A stays on one thread either way, and the other thread's products then
    // compete with it on the tensor core.)
    {  // the whole warp runs the issue loop; one elected lane issues (issue model in wa_ptx.cuh)
      uint32_t kv_n = 0, q_n = 0, d_n = 0, p_n = 0, ds_n = 0;
      bool ok = true;
      const uint64_t dk_ = sdesc_sw128(sK, 16, 1024), dv_ = sdesc_sw128(sV, 16, 1024);
      const uint64_t dq_k = sdesc_sw128(sQ, 16, 1024), dd_k = sdesc_sw128(sDO, 16, 1024);  // K-major B (S^T, dP^T)
      const uint64_t dq_mn = sdesc_sw128(sQ, kTileRows * 128, 1024);  // MN-major B (dk)
      const uint64_t dd_mn = sdesc_sw128(sDO, kTileRows * 128, 1024);  // MN-major B (dv)
      const uint32_t hi = (uint32_t)(dk_ >> 32);
      auto issue_nt = [&](uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk / 4) * kTileRows * 128 + (kk % 4) * 32) >> 4;
          mma_ss(d_tmem, a_lo + off, b_lo + off, hi, C::kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      // acc (+)= A[tmem: 128 keys x 128 queries, bf16] . B[smem: 128 queries x D], 16 queries per MMA
      auto issue_acc = [&](uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk)
          mma_ts(d_tmem, a_tmem + tmem_a_block(kk), b_lo + ((kk * 2048) >> 4), hi, C::kIdescAcc,
                 (acc || kk > 0) ? 1u : 0u);
      };
      auto tile_at = [&](uint64_t desc, uint32_t s) { return (uint32_t)desc + ((s * C::kTileBytes) >> 4); };
      for (uint32_t n = 0; ok; ++n) {
        const int idx = feed.fetch(n, abort_flag, err, ok);
        if (idx < 0) break;
        const Item it = load_item(prm.items, idx);
        const int ntk = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
        const int nt = seg_tiles(it.s0_lo, it.s0_hi) + seg_tiles(it.s1_lo, it.s1_hi);
        for (int t = 0; t < ntk && ok; ++t) {
          ok = mbar_wait_warp(b_kvfull, kv_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          kv_n++;
          uint32_t qs = q_n % C::kQSlots, ds = d_n % C::kDSlots;
          ok = ok && mbar_wait_warp(b_qfull(qs), (q_n / C::kQSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          q_n++;
          if (!ok) break;
          tc_fence_after();
          issue_nt(tS, (uint32_t)dk_, tile_at(dq_k, qs));  // S^T(0) = K Q_0^T
          mma_commit(b_sfull);
          ok = mbar_wait_warp(b_dfull(ds), (d_n / C::kDSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          d_n++;
          if (!ok) break;
          tc_fence_after();
          issue_nt(tDP, (uint32_t)dv_, tile_at(dd_k, ds));  // dP^T(0) = V dout_0^T
          mma_commit(b_dpfull);
          if (nt == 1) mma_commit(b_kvempty);
          for (int j = 0; j < nt && ok; ++j) {
            ok = mbar_wait_warp(b_pfull, p_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);  // P^T(j) in TMEM
            p_n++;
            if (!ok) break;
            tc_fence_after();
            issue_acc(tDV, tS, tile_at(dd_mn, ds), j > 0);  // dv += P^T(j) dout_j
            mma_commit(b_dempty(ds));  // dout_j is read for the last time (its column values: elementwise warps)
            uint32_t qn = 0, dn = 0;
            if (j + 1 < nt) {
              qn = q_n % C::kQSlots;
              ok = mbar_wait_warp(b_qfull(qn), (q_n / C::kQSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
              q_n++;
              if (!ok) break;
              tc_fence_after();
              issue_nt(tS, (uint32_t)dk_, tile_at(dq_k, qn));  // S^T(j+1)
              mma_commit(b_sfull);
            }
            ok = mbar_wait_warp(b_dsfull, ds_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);  // dS^T(j) in TMEM
            ds_n++;
            if (!ok) break;
            tc_fence_after();
            issue_acc(tDK, tDP, tile_at(dq_mn, qs), j > 0);  // dk += dS^T(j) Q_j
            mma_commit(b_qempty(qs));
            if (j + 1 < nt) {
              dn = d_n % C::kDSlots;
              ok = mbar_wait_warp(b_dfull(dn), (d_n / C::kDSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
              d_n++;
              if (!ok) break;
              tc_fence_after();
              issue_nt(tDP, (uint32_t)dv_, tile_at(dd_k, dn));  // dP^T(j+1)
              mma_commit(b_dpfull);
              if (j + 1 == nt - 1) mma_commit(b_kvempty);  // every MMA that reads the key / value tiles is issued
            }
            qs = qn;
            ds = dn;
          }
          if (!ok) break;
          mma_commit(b_ofull);
        }
      }
      mma_commit(b_drain_x);
      mbar_wait_drain(b_drain_x, 0, ok ? kWaitLimitNs : kDrainLimitNs);
    }
  } else if (warp < kEwWarps) {
    // ---------------------------------------------------------------------------------------- elementwise
    const int r = 32 * (warp & 3) + lane;  // key row in the tile == TMEM lane
    const int col0 = kCW * (warp >> 2);   // this thread's query columns [col0, col0 + kCW)
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    uint32_t d_n = 0, s_n = 0, o_n = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int idx = feed.fetch(n, abort_flag, err, ok);
      if (idx < 0) break;
      const Item it = load_item(prm.items, idx);
      const int ntk = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
      const int nt = seg_tiles(it.s0_lo, it.s0_hi) + seg_tiles(it.s1_lo, it.s1_hi);
      for (int t = 0; t < ntk && ok; ++t) {
        for (int j = 0; j < nt; ++j) {
          const uint32_t ds = d_n % C::kDSlots;
          ok = mbar_wait(b_dfull(ds), (d_n / C::kDSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          ok = ok && mbar_wait(b_sfull, s_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          ok = __all_sync(0xffffffffu, ok);
          d_n++;
          if (!ok) break;
          tc_fence_after();
          const uint32_t cb = sCol + ds * C::kColBytes + col0 * 4;  // -lse' of this thread's first column
          // Phase A: P^T = 2^(s c' - lse'_col) over this thread's query columns
          float p[kCW];
          uint32_t sr64[kCW];  // this thread's score columns in one TMEM load (one wait, not one per 32 columns)
          tmem_ld_x64(tS + lane_base + col0, sr64);
#pragma unroll
          for (int ch = 0; ch < kCW / 32; ++ch) {
            uint32_t pk[16];
            const uint32_t* sr = sr64 + 32 * ch;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 nl = lds_f4(cb + (32 * ch + 4 * c4) * 4);  // -lse' of 4 columns
              const int i = 32 * ch + 4 * c4;
              float x0, x1, x2, x3;
              fma2(x0, x1, __uint_as_float(sr[4 * c4]), __uint_as_float(sr[4 * c4 + 1]), prm.c_log2, prm.c_log2, nl.x,
                   nl.y);
              fma2(x2, x3, __uint_as_float(sr[4 * c4 + 2]), __uint_as_float(sr[4 * c4 + 3]), prm.c_log2, prm.c_log2,
                   nl.z, nl.w);
              p[i] = ex2(x0);
              p[i + 1] = ex2(x1);
              p[i + 2] = ex2(x2);
              p[i + 3] = ex2(x3);
              pk[2 * c4] = pack_bf16(p[i], p[i + 1]);
              pk[2 * c4 + 1] = pack_bf16(p[i + 2], p[i + 3]);
            }
            tmem_st_x16(tS + lane_base + col0 + 16 * ch, pk);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_pfull);
          // Phase B: dS^T = P^T (dP^T - Dvec_col)
          ok = mbar_wait(b_dpfull, s_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          ok = __all_sync(0xffffffffu, ok);
          s_n++;
          if (!ok) break;
          tc_fence_after();
          uint32_t dr64[kCW];  // this thread's dP^T columns in one TMEM load
          tmem_ld_x64(tDP + lane_base + col0, dr64);
#pragma unroll
          for (int ch = 0; ch < kCW / 32; ++ch) {
            uint32_t pk[16];
            const uint32_t* dr = dr64 + 32 * ch;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 nd = lds_f4(cb + 512 + (32 * ch + 4 * c4) * 4);  // -Dvec of 4 columns
              const int i = 32 * ch + 4 * c4;
              float t0, t1, t2, t3;
              add2(t0, t1, __uint_as_float(dr[4 * c4]), __uint_as_float(dr[4 * c4 + 1]), nd.x, nd.y);
              add2(t2, t3, __uint_as_float(dr[4 * c4 + 2]), __uint_as_float(dr[4 * c4 + 3]), nd.z, nd.w);
              mul2(t0, t1, t0, t1, p[i], p[i + 1]);
              mul2(t2, t3, t2, t3, p[i + 2], p[i + 3]);
              pk[2 * c4] = pack_bf16(t0, t1);
              pk[2 * c4 + 1] = pack_bf16(t2, t3);
            }
            tmem_st_x16(tDP + lane_base + col0 + 16 * ch, pk);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(b_dsfull);
            mbar_arrive(b_dempty(ds));  // this slot's column values are no longer needed
          }
        }
        if (!ok) break;
        ok = mbar_wait(b_ofull, o_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        o_n++;
        if (!ok) break;
        tc_fence_after();
        constexpr int EC = EpiCols<D>::kCols;
        const int c_lo = EC * (warp >> 2);
        if (c_lo < D) {
          const int key = it.q_lo + t * kTileRows + r;
          const bool row_ok = key < it.q_hi;
          const int b = it.bh / prm.H, h = it.bh % prm.H;
          if (it.split < 0) {
            const int64_t off = (int64_t)b * prm.sb + (int64_t)key * prm.sl + (int64_t)h * prm.sh + c_lo;
            store_cols<EC>(tDV + lane_base + c_lo, 1.f, row_ok, prm.dv + off, nullptr);
            store_cols<EC>(tDK + lane_base + c_lo, prm.scale, row_ok, prm.dk + off, nullptr);
          } else {
            const int64_t slot = (((int64_t)it.bh * prm.G + (key - prm.g0)) * prm.n_splits + it.split) * D + c_lo;
            store_cols<EC>(tDV + lane_base + c_lo, 1.f, row_ok, nullptr, prm.ws_dv + slot);
            store_cols<EC>(tDK + lane_base + c_lo, prm.scale, row_ok, nullptr, prm.ws_dk + slot);
          }
        }
        tc_fence_before();
      }
    }
  }
  teardown(tmem, warp, feed);
}

// Dvec_i = dout_i . out_i for every (b, i, h); fp32 into [B*H][L]. One warp per 8 consecutive rows of one (b, h):
// each row is read by a group of D/8 lanes with 16-byte loads (all of a warp's loads are issued before any is
// used), and the warp's 8 results land in one 32-byte sector of dvec.
template <int D>
__global__ void __launch_bounds__(256) bwd_dot_kernel(const __nv_bfloat16* __restrict__ out,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      float* __restrict__ dvec, int64_t units, int L, int H,
                                                      int64_t sb, int64_t sl, int64_t sh) {
  constexpr int kGroup = D / 8;             // lanes per row: 16 (D = 128) or 8 (D = 64)
  constexpr int kRowsPerLoad = 32 / kGroup;  // rows covered by one warp-wide load
  constexpr int kLoads = 8 / kRowsPerLoad;
  const int64_t u = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // unit: (b, h, block of 8 rows)
  const int lane = threadIdx.x & 31;
  if (u >= units) return;
  const int nlb = (L + 7) / 8;
  const int64_t bh = u / nlb;
  const int l0 = (int)(u % nlb) * 8;
  const int b = (int)(bh / H), h = (int)(bh % H);
  const int sub = lane % kGroup, grp = lane / kGroup;
  uint4 a[kLoads], g[kLoads];
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    const int l = l0 + i * kRowsPerLoad + grp;
    if (l < L) {
      const int64_t off = (int64_t)b * sb + (int64_t)l * sl + (int64_t)h * sh + sub * 8;
      a[i] = __ldg(reinterpret_cast<const uint4*>(out + off));
      g[i] = __ldg(reinterpret_cast<const uint4*>(dout + off));
    } else {
      a[i] = make_uint4(0u, 0u, 0u, 0u);
      g[i] = a[i];
    }
  }
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    const uint32_t av[4] = {a[i].x, a[i].y, a[i].z, a[i].w}, gv[4] = {g[i].x, g[i].y, g[i].z, g[i].w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[e]));
      acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
    }
#pragma unroll
    for (int o = kGroup / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    const int l = l0 + i * kRowsPerLoad + grp;
    if (sub == 0 && l < L) dvec[bh * L + l] = acc;
  }
}

// Sum the split partials of the global rows into bf16 rows: tensor blockIdx.y (0 dq, 1 dk, 2 dv), one warp per row,
// splits added in index order.
template <int D>
__global__ void __launch_bounds__(256) bwd_sum_kernel(const float* __restrict__ ws, int64_t part_elems,
                                                      __nv_bfloat16* dq, __nv_bfloat16* dk, __nv_bfloat16* dv,
                                                      int rows, int G, int H, int g0, int P, int64_t sb, int64_t sl,
                                                      int64_t sh) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int which = blockIdx.y;
  const float* src = ws + which * part_elems + (int64_t)r * P * D;
  __nv_bfloat16* dst = which == 0 ? dq : (which == 1 ? dk : dv);
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  for (int p = 0; p < P; ++p) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] += __ldg(src + (int64_t)p * D + lane + 32 * i);
  }
  const int bh = r / G, gr = r % G;
  const int b = bh / H, h = bh % H;
  __nv_bfloat16* d = dst + (int64_t)b * sb + (int64_t)(g0 + gr) * sl + (int64_t)h * sh;
#pragma unroll
  for (int i = 0; i < kPer; ++i) d[lane + 32 * i] = __float2bfloat16_rn(acc[i]);
}

template <int D>
int launch_backward_d(const BackwardArgs& a, cudaStream_t s, int num_sms, void* const* events) {
  if (int e = ensure_smem_attr(reinterpret_cast<const void*>(&wa_dq_kernel<D>), DqCfg<D>::kSmemBytes)) return e;
  if (int e = ensure_smem_attr(reinterpret_cast<const void*>(&wa_dkdv_kernel<D>), DkvCfg<D>::kSmemBytes)) return e;
  const Geometry& g = *a.geo;
  const wa_layout_t& l = g.layout;
  alignas(64) CUtensorMap mq, mk, mv, mdo;
  if (!make_tile_map(&mq, a.q, g, 2) || !make_tile_map(&mk, a.k, g, 2) || !make_tile_map(&mv, a.v, g, 2) ||
      !make_tile_map(&mdo, a.dout, g, 2))
    return (int)cudaErrorInvalidValue;
  auto rec = [&](int i) { return events ? cudaEventRecord((cudaEvent_t)events[i], s) : cudaSuccess; };
  cudaError_t e = rec(0);
  if (e != cudaSuccess) return (int)e;
  const int64_t units = (int64_t)l.B * l.H * ((g.L + 7) / 8);
  bwd_dot_kernel<D><<<(unsigned)((units + 7) / 8), 256, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(a.out), reinterpret_cast<const __nv_bfloat16*>(a.dout), a.dvec, units,
      (int)g.L, l.H, l.stride_b, l.stride_l, l.stride_h);
  if ((e = cudaGetLastError()) != cudaSuccess || (e = rec(1)) != cudaSuccess) return (int)e;
  BwdParams p;
  p.items = a.items;
  p.n_items = a.n_items;
  p.lse = a.lse;
  p.dvec = a.dvec;
  p.dq = reinterpret_cast<__nv_bfloat16*>(a.dq);
  p.dk = reinterpret_cast<__nv_bfloat16*>(a.dk);
  p.dv = reinterpret_cast<__nv_bfloat16*>(a.dv);
  p.ws_dq = a.ws;
  p.ws_dk = a.ws ? a.ws + a.part_elems : nullptr;
  p.ws_dv = a.ws ? a.ws + 2 * a.part_elems : nullptr;
  p.err = a.err;
  p.sb = l.stride_b;
  p.sl = l.stride_l;
  p.sh = l.stride_h;
  p.H = l.H;
  p.G = g.G;
  p.g0 = (int)g.g0;
  p.L = (int)g.L;
  p.n_splits = a.n_splits;
  p.c_log2 = (float)(1.4426950408889634 / sqrt((double)D));
  p.scale = (float)(1.0 / sqrt((double)D));
  p.debug_flags = a.debug_flags;
  p.item_counter = a.item_counter;
  p.bh_count = l.B * l.H;
  const int grid = a.n_items < num_sms ? a.n_items : num_sms;
  if (grid > 0) {
    wa_dq_kernel<D><<<grid, kBwdThreads, DqCfg<D>::kSmemBytes, s>>>(mq, mk, mv, mdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
  }
  if ((e = rec(2)) != cudaSuccess) return (int)e;
  if (grid > 0) {
    wa_dkdv_kernel<D><<<grid, kBwdThreads, DkvCfg<D>::kSmemBytes, s>>>(mq, mk, mv, mdo, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
  }
  if ((e = rec(3)) != cudaSuccess) return (int)e;
  if (g.G > 0) {
    const int grows = l.B * l.H * g.G;
    bwd_sum_kernel<D><<<dim3((grows + 7) / 8, 3), 256, 0, s>>>(a.ws, a.part_elems, p.dq, p.dk, p.dv, grows, g.G, l.H,
                                                                (int)g.g0, a.n_splits, l.stride_b, l.stride_l,
                                                                l.stride_h);
    if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
  }
  return (int)rec(4);
}

}  // namespace

int launch_backward(const BackwardArgs& a, void* stream, int num_sms, void* const* events) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return a.geo->layout.D == 128 ? launch_backward_d<128>(a, s, num_sms, events)
                                : launch_backward_d<64>(a, s, num_sms, events);
}

}  // namespace wa
