// Attention kernels for chunk-aligned window softmax attention on sm_103a.
//
// One persistent launch runs every work item of the plan: window items (a pair of 128-row query tiles of one
// window group against the group's key segments: its frame window, then the globals) and global-leg items (a
// pair of global query tiles against one key split of the whole sequence). This is the decomposition of the
// VDN-Minimax-H3 window-attention article, section 三: every kept (query, key) pair lies in a dense rectangle,
// and each rectangle is computed as plain dense attention with no mask except at segment tails.
//
// CTA roles (384 threads = 3 warpgroups, one CTA per SM):
//   warps 0-3   softmax warpgroup of query tile 0: one thread per query row / TMEM lane
//   warps 4-7   softmax warpgroup of query tile 1
//   warp 8      MMA issuer: S_t = Q_t K^T and O_t += P_t V with tcgen05.mma, accumulators in TMEM; the whole warp
//               runs the loop and one elect.sync-chosen lane issues (the issue model in wa_ptx.cuh)
//   warp 9      TMA producer (the whole warp runs the loop, lane 0 issues): Q tiles and rings of K / V tiles,
//               128-byte swizzled; each step's K_j and V_{j-1} complete on one bundle barrier. It also claims the
//               CTA's next work item from a global counter when it is ready for one, and passes the index to the
//               other roles through a shared ring. A segment's last V tile lands on a barrier of its own first:
//               the 32 lanes zero its rows past the segment's end (tokens outside the rows' kept sets, where P is 0
//               but 0 x Inf would be NaN) and only then release the bundle, so the MMA and softmax roles never
//               see a ragged tail
//   warps 10-11 idle
// Full window tiles (D = 128) leave through a shared-memory stage and TMA stores; the rest is stored directly.
// The launch gives every thread 168 registers (384 x 168 = 64512); setmaxnreg then moves them to where the work
// is: the softmax warpgroups rise to 192 (a full 128-column score row stays in registers), the third warpgroup
// drops to 120. 2 x 128 x 192 + 128 x 120 = 64512, the launch's total. Each role branch ends with its own copy of
// the teardown, so that no code is shared by regions with different register counts.
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256, 256+D), O_1 [384, 384+D). P_t (bf16) overwrites the
// first 64 columns of S_t and is the A operand of the P.V MMA, read straight from TMEM.
// The two query tiles ping-pong: while one warpgroup runs the softmax of its tile, the tensor core works on the
// other tile's products. An item with a single query tile (the rows of a group past its last full pair of tiles)
// alternates its key tiles between the two slots instead and merges the two halves at the end, so that it keeps
// the ping-pong too.
//
// Softmax state is fp32 in registers: a reference max m (in log2 units of the scaled score) and row sum l. Each
// step exponentiates against m and checks only the step's row sum: the exact row max is taken (and m raised, O
// and l rescaled) when that sum exceeds 2^16 or is not finite, i.e. at an item's first step (m starts at -inf) and
// when the scores jump. This is exact because the final normalisation uses the same m. Every wait is bounded; on expiry the kernel latches an error in the plan's
// error word and unwinds.
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

constexpr int kThreads = 384;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr uint32_t kSoftmaxRegs = 192;
constexpr uint32_t kControlRegs = 120;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168, "register split exceeds the launch");
constexpr float kLazyLimit = 65536.0f;  // a step's row sum above this (relative to the reference m) raises m
constexpr int kItemConsumers = 9;  // warps that take every work item from the producer: the MMA warp, 8 softmax

// kF8: q and k are e4m3 (one byte per element) and the scores use kind::f8f6f4 MMAs; v, P and O stay bf16 / fp32.
template <int D, bool kF8>
struct Cfg {
  static constexpr int kQKRowBytes = D * (kF8 ? 1 : 2);
  static constexpr int kQKBoxes = kQKRowBytes / 128;           // 128-byte swizzle boxes per q / k row
  static constexpr int kQKBoxElems = kF8 ? 128 : 64;           // elements in one 128-byte box row
  static constexpr int kQTileBytes = kTileRows * kQKRowBytes;  // one query tile (also one key tile)
  static constexpr int kVBoxes = D / 64;                       // v is bf16: 64 elements per 128-byte box row
  static constexpr int kVTileBytes = kTileRows * D * 2;
  static constexpr int kBoxBytes = kTileRows * 128;            // one box: 128 rows x 128 bytes
  static constexpr int kSKSteps = kF8 ? D / 32 : D / 16;       // score MMAs per tile (32 bytes of K each)
  static_assert(kQKBoxes >= 1 && kQKRowBytes % 128 == 0, "q / k rows must be whole 128-byte boxes");
  // Separate K and V rings; the producer runs K one tile ahead of V (K is needed a step earlier than V).
  static constexpr int kKSlots = kF8 ? 3 : (D == 128 ? 2 : 4);
  static constexpr int kVSlots = kF8 ? 3 : (D == 128 ? 2 : 4);
  // Step bundles: the copies of step j (K_j and V_{j-1}) complete on one barrier and are released by one commit.
  // Bundle b reuses a K slot last read in bundle <= b - kKSlots and a V slot last read in bundle <= b - kVSlots,
  // so the producer waits for bundle b - kLag's release, kLag = min(kKSlots, kVSlots) (also the barrier count).
  static constexpr int kLag = kKSlots < kVSlots ? kKSlots : kVSlots;
  // D = 128: full window tiles leave through shared memory and one TMA store per 64 columns (16 KB per query tile:
  // each store instruction of the softmax warps then fills whole 128-byte rows of shared memory, instead of
  // touching 32 rows of out). A bundle's K slot is never reused sooner than kLag bundles later, so K slots beyond
  // kLag would sit idle: their space holds the two tiles' staging.
  static constexpr bool kStage = D == 128;
  static constexpr int kStageTileBytes = kTileRows * 128;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kQTileBytes;
  static constexpr int kVOff = kKOff + kKSlots * kQTileBytes;
  static constexpr int kStageOff = kVOff + kVSlots * kVTileBytes;
  static constexpr int kBarOff = kStageOff + (kStage ? 2 * kStageTileBytes : 0);
  // barriers: q_full[2] q_empty[2] s_full[2] p_full[2] o_full[2] drain b_full[kLag] b_empty[kLag]
  //           item ring full[kItemRingSlots] empty[kItemRingSlots]  stage_full[2] stage_free[2] v_land
  //           xchg_full o1_free
  static constexpr int kNumBars = 11 + 2 * kLag + 2 * kItemRingSlots + 7;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM address, abort flag, 2 spare words, item ring
  // (m, l) of the 128 rows of an alternating-key item's second half, handed to the first warpgroup (8 bytes a row)
  static constexpr int kXchgOff = kMiscOff + 16 + 4 * kItemRingSlots;
  static constexpr int kSmemBytes = kXchgOff + kTileRows * 8 + 1024;  // + slack for 1024-byte alignment
  static constexpr uint32_t kTmemO = 256;
  static constexpr uint32_t kIdescS = kF8 ? idesc_e4m3_f32(128, 128)
                                         : idesc_bf16_f32(128, 128, 0, 0);  // Q K-major, K K-major
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);   // P from TMEM, V MN-major (D contiguous)
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Params {
  const Item* items;
  int n_items;
  __nv_bfloat16* out;
  float* ws_o;
  float* ws_lse;
  int* err;
  int64_t sb, sl, sh;  // element strides of out
  int H, G, g0, n_splits;
  float c_scale;  // log2(e) / sqrt(D)
  int debug_flags;
  float* lse;     // optional [B][H][L] row log-sum-exp output (natural log); nullptr when not wanted
  int L;
  int* item_counter;  // ItemFeed counter (two ints, zero at launch); nullptr: static striding
  int bh_count;       // B * H (index checks of a debug build)
};

// Shared-memory barrier layout, relative to the barrier block: q_full[2] q_empty[2] s_full[2] p_full[2]
// o_full[2] drain, then the step-bundle barriers, then the item ring's. Addresses are computed, never indexed from
// a local array.
template <int NB>
struct BarAddr {
  uint32_t base;
  __device__ __forceinline__ uint32_t q_full(int t) const { return base + 8 * (0 + t); }
  __device__ __forceinline__ uint32_t q_empty(int t) const { return base + 8 * (2 + t); }
  __device__ __forceinline__ uint32_t s_full(int t) const { return base + 8 * (4 + t); }
  __device__ __forceinline__ uint32_t p_full(int t) const { return base + 8 * (6 + t); }
  __device__ __forceinline__ uint32_t o_full(int t) const { return base + 8 * (8 + t); }
  __device__ __forceinline__ uint32_t drain() const { return base + 8 * 10; }
  // bundle b: full (copies landed) and empty (the MMAs reading it completed)
  __device__ __forceinline__ uint32_t b_full(uint32_t b) const { return base + 8 * (11 + b % NB); }
  __device__ __forceinline__ uint32_t b_empty(uint32_t b) const { return base + 8 * (11 + NB + b % NB); }
  // the work-item ring's barriers (ItemFeed)
  __device__ __forceinline__ uint32_t item_ring() const { return base + 8 * (11 + 2 * NB); }
  // query tile t's epilogue staging: written by its 4 warps (full), read out by the store (free)
  __device__ __forceinline__ uint32_t stage_full(int t) const { return base + 8 * (11 + 2 * NB + 2 * kItemRingSlots + t); }
  __device__ __forceinline__ uint32_t stage_free(int t) const {
    return base + 8 * (13 + 2 * NB + 2 * kItemRingSlots + t);
  }
  // a segment's last V tile lands here (not on its bundle's barrier) so the producer can clean it first
  __device__ __forceinline__ uint32_t v_land() const { return base + 8 * (15 + 2 * NB + 2 * kItemRingSlots); }
  // alternating-key items: the second warpgroup's (m, l) are in shared memory (xchg_full); the first warpgroup has
  // read them and the second half's O out of TMEM (o1_free)
  __device__ __forceinline__ uint32_t xchg_full() const { return base + 8 * (16 + 2 * NB + 2 * kItemRingSlots); }
  __device__ __forceinline__ uint32_t o1_free() const { return base + 8 * (17 + 2 * NB + 2 * kItemRingSlots); }
};

// An item with a single query tile and at least two key tiles runs with alternating keys: key tile j goes to tile
// slot j % 2, so the two slots (their S/P and O regions in TMEM and their softmax warpgroups) ping-pong on the same
// query rows exactly as two query tiles would, and the tile costs half the time it would alone. Each slot keeps its
// own (O, m, l) over its keys; the first warpgroup merges the two by log-sum-exp in the epilogue.
__device__ __forceinline__ bool alternating_keys(int ntq, int nt) { return ntq == 1 && nt >= 2; }

// Exponentiate one 128-column score row into bf16 P (written to TMEM over the row's S columns, 16 columns per
// store) and return the fp32 row sum.
__device__ __forceinline__ float exp_store_row(const float (&s)[128], float c_scale, float neg_m, uint32_t tS) {
  float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // 4 independent pairs: short add chains
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float x0, x1;
      fma2(x0, x1, s[32 * q4 + 2 * c], s[32 * q4 + 2 * c + 1], c_scale, c_scale, neg_m, neg_m);
      const float p0 = ex2(x0);
      const float p1 = ex2(x1);
      add2(sum[2 * (c & 3)], sum[2 * (c & 3) + 1], sum[2 * (c & 3)], sum[2 * (c & 3) + 1], p0, p1);
      pk[c] = pack_bf16(p0, p1);
    }
    tmem_st_x16(tS + 16 * q4, pk);
  }
  return ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
}

template <int D, bool kF8>
__global__ void __launch_bounds__(kThreads, 1)
    window_attention_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_o,
                            const Params prm) {
  using C = Cfg<D, kF8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + C::kQOff;
  const uint32_t sK = s_base + C::kKOff;
  const uint32_t sV = s_base + C::kVOff;
  const uint32_t bar0 = s_base + C::kBarOff;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const BarAddr<C::kLag> bars{bar0};
  const ItemFeed feed{prm.item_counter, prm.n_items, reinterpret_cast<volatile int*>(smem + C::kMiscOff + 16),
                      bars.item_ring()};

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.q_full(t), 1);
      mbar_init(bars.q_empty(t), 1);
      mbar_init(bars.s_full(t), 1);
      mbar_init(bars.p_full(t), 4);  // one arrive per softmax warp
      mbar_init(bars.o_full(t), 1);
    }
    mbar_init(bars.drain(), 1);
    for (int s = 0; s < C::kLag; ++s) {
      mbar_init(bars.b_full(s), 1);
      mbar_init(bars.b_empty(s), 1);
    }
    feed.init(kItemConsumers);
    for (int t = 0; t < 2; ++t) {
      mbar_init(bars.stage_full(t), 4);  // one arrive per warp of the tile's warpgroup
      mbar_init(bars.stage_free(t), 1);  // the store issuer, once the copy engine has read the stage
    }
    mbar_init(bars.v_land(), 1);
    mbar_init(bars.xchg_full(), 4);  // one arrive per warp of the second warpgroup
    mbar_init(bars.o1_free(), 4);    // one arrive per warp of the first warpgroup
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  int* err = prm.err;

  auto teardown = [&]() {  // every thread: wait for all roles, then warp 0 frees the tensor memory
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) feed.finish();  // this CTA's claims are over (the last CTA out rewinds the counter)
    if (warp == 0) {
      __syncwarp();  // tcgen05.dealloc is warp-collective: reconverge after the role branches
      tmem_dealloc(tmem, 512);
    }
  };

  if (warp >= 8) {
    regs_dec<kControlRegs>();
    if (warp == kLoadWarp) {
    // ------------------------------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (waits are warp-wide); lane 0 claims the items and issues the copies.
    {
      const bool leader = lane == 0;
      uint32_t k_n = 0, v_n = 0, b_n = 0;  // K tiles, V tiles and step bundles loaded so far
      uint32_t vt_n = 0;                   // segment-final V tiles landed on v_land so far
      uint32_t q_n0 = 0, q_n1 = 0;
      bool dropped = false;
      bool ok = true;
      for (uint32_t n = 0; ok; ++n) {
        const int idx = feed.claim_warp(n, abort_flag, err, ok);
        if (idx < 0) break;
#ifdef WA_DEBUG
        Item it = load_item(prm.items, idx);
        if ((prm.debug_flags & 8) && n == 0 && blockIdx.x == 0)
          it.s0_hi = prm.L + 1000;  // test hook: a key segment past the sequence (the check must catch it)
        if (!item_in_bounds(it, ItemBounds{prm.bh_count, prm.L, prm.g0, prm.G, prm.n_splits})) {
          if (leader) {
            atomicOr(err, kErrBounds);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
#else
        const Item it = load_item(prm.items, idx);
#endif
        const int b = it.bh / prm.H, h = it.bh % prm.H;
        const int ntq = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t >= ntq || !ok) break;
          uint32_t& qn = t ? q_n1 : q_n0;
          ok = mbar_wait_warp(bars.q_empty(t), (qn & 1) ^ 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          if (!ok) break;
          if (leader) {
            mbar_arrive_expect_tx(bars.q_full(t), C::kQTileBytes);
#pragma unroll
            for (int hf = 0; hf < C::kQKBoxes; ++hf)
              tma_load_4d(sQ + t * C::kQTileBytes + hf * C::kBoxBytes, &tmap_q, bars.q_full(t), hf * C::kQKBoxElems,
                          h, it.q_lo + t * kTileRows, b);
          }
          qn++;
        }
        const int nt0 = seg_tiles(it.s0_lo, it.s0_hi);
        const int nt = nt0 + seg_tiles(it.s1_lo, it.s1_hi);
        auto row_of = [&](int j) { return j < nt0 ? it.s0_lo + j * kTileRows : it.s1_lo + (j - nt0) * kTileRows; };
        // Bundle j of the item: K_j (j < nt, for S(j)) and V_{j-1} (j >= 1, for P(j-1).V).
        for (int j = 0; j <= nt && ok; ++j) {
          if (b_n >= (uint32_t)C::kLag) {
            const uint32_t w = b_n - C::kLag;
            ok = mbar_wait_warp(bars.b_empty(w), (w / C::kLag) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
            if (!ok) break;
          }
          const uint32_t full = bars.b_full(b_n);
          const uint32_t kbytes = j < nt ? C::kQTileBytes : 0;
          // V_{j-1} ends a segment mid-tile: it lands on v_land and the bundle is released after the cleaning below
          const int vvalid = j >= 1 ? tile_valid(it, j - 1, nt0) : kTileRows;
          const bool vtail = vvalid < kTileRows;
          const uint32_t vslot = v_n % C::kVSlots;
          if (leader) {
            if (vtail) {
              mbar_expect_tx(full, kbytes);  // the pending arrival is made once the V tile is clean
              mbar_arrive_expect_tx(bars.v_land(), C::kVTileBytes);
            } else {
              mbar_arrive_expect_tx(full, kbytes + (j >= 1 ? C::kVTileBytes : 0));
            }
            if ((prm.debug_flags & 1) && !dropped && blockIdx.x == 0 && j < nt) {
              dropped = true;  // fault injection for the watchdog test: this key tile is never loaded
            } else if (j < nt) {
              const uint32_t slot = k_n % C::kKSlots;
#pragma unroll
              for (int hf = 0; hf < C::kQKBoxes; ++hf)
                tma_load_4d(sK + slot * C::kQTileBytes + hf * C::kBoxBytes, &tmap_k, full, hf * C::kQKBoxElems, h,
                            row_of(j), b);
            }
            if (j >= 1) {
              const uint32_t vbar = vtail ? bars.v_land() : full;
#pragma unroll
              for (int hf = 0; hf < C::kVBoxes; ++hf)
                tma_load_4d(sV + vslot * C::kVTileBytes + hf * C::kBoxBytes, &tmap_v, vbar, hf * 64, h,
                            row_of(j - 1), b);
            }
          }
          if (j < nt) k_n++;
          if (j >= 1) v_n++;
          b_n++;
          if (vtail) {
            ok = mbar_wait_warp(bars.v_land(), vt_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
            vt_n++;
            if (ok) zero_tile_rows(sV + vslot * C::kVTileBytes, C::kVBoxes, vvalid, lane);
            if (leader) mbar_arrive(full);  // release the bundle (also when unwinding, so that it can drain)
          }
        }
      }
      if (!ok && leader) {
        // Unwinding: wait (briefly) for the copies still in flight so that none lands after the CTA exits.
        for (uint32_t n = b_n > (uint32_t)C::kLag ? b_n - C::kLag : 0; n < b_n; ++n)
          mbar_wait_drain(bars.b_full(n), (n / C::kLag) & 1, kDrainLimitNs);
        if (vt_n) mbar_wait_drain(bars.v_land(), (vt_n - 1) & 1, kDrainLimitNs);
        if (q_n0) mbar_wait_drain(bars.q_full(0), (q_n0 - 1) & 1, kDrainLimitNs);
        if (q_n1) mbar_wait_drain(bars.q_full(1), (q_n1 - 1) & 1, kDrainLimitNs);
      }
    }
    } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------------------------- MMA issuer
    // The whole warp runs this loop (see the issue model in wa_ptx.cuh); one elected lane issues the MMAs.
    {
      uint32_t k_n = 0, v_n = 0, b_n = 0;
      uint32_t q_n0 = 0, q_n1 = 0, p_n0 = 0, p_n1 = 0;
      bool ok = true;
      // Descriptors are built once; a shared-memory offset is added to the start-address field (address >> 4,
      // 14 bits: every address of the 227 KB window fits, so the addition never carries out of the field, nor out
      // of the low word).
      const uint64_t dq = sdesc_sw128(sQ, 16, 1024);                 // Q tiles, K-major
      const uint64_t dk = sdesc_sw128(sK, 16, 1024);                 // K tiles, K-major
      const uint64_t dv = sdesc_sw128(sV, C::kBoxBytes, 1024);       // V tiles, MN-major (D contiguous)
      // O_t (+)= P_t V, P_t read from TMEM (aliasing S_t), V from ring slot `vslot`
      // All three descriptor families share one high word (stride byte offset 1024, version, 128-byte swizzle).
      const uint32_t desc_hi = (uint32_t)(dq >> 32);
      auto issue_pv = [&](int t, uint32_t vslot, bool acc_first) {
        const uint32_t d0 = (uint32_t)dv + ((vslot * C::kVTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk)
          mma_ts(tmem + C::kTmemO + t * 128, tmem + t * 128 + kk * 8, d0 + ((kk * 2048) >> 4), desc_hi,
                 C::kIdescPV, (acc_first || kk > 0) ? 1u : 0u);
      };
      // S_u = Q_qt K^T into the S region of slot u, both K-major; each MMA takes 32 bytes of K (16 bf16 or 32
      // e4m3 elements) inside a 128-byte swizzle row, then moves to the next box
      auto issue_s = [&](int qt, int u, uint32_t kslot) {
        const uint32_t q0 = (uint32_t)dq + ((qt * C::kQTileBytes) >> 4);
        const uint32_t k0 = (uint32_t)dk + ((kslot * C::kQTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::kSKSteps; ++kk) {
          const uint32_t off = ((kk / 4) * C::kBoxBytes + (kk % 4) * 32) >> 4;
          if constexpr (kF8)
            mma_ss_f8(tmem + u * 128, q0 + off, k0 + off, desc_hi, C::kIdescS, kk > 0 ? 1u : 0u);
          else
            mma_ss(tmem + u * 128, q0 + off, k0 + off, desc_hi, C::kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      for (uint32_t n = 0; ok; ++n) {
        const int idx = feed.fetch(n, abort_flag, err, ok);
        if (idx < 0) break;
        const Item it = load_item(prm.items, idx);
        const int ntq = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
        const int nt0 = seg_tiles(it.s0_lo, it.s0_hi);
        const int nt = nt0 + seg_tiles(it.s1_lo, it.s1_hi);
        ok = mbar_wait_warp(bars.q_full(0), q_n0 & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
        q_n0++;
        if (ok && ntq > 1) {
          ok = mbar_wait_warp(bars.q_full(1), q_n1 & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          q_n1++;
        }
        if (!ok) break;
        if (alternating_keys(ntq, nt)) {
          // Step j: S = Q_0 K_j^T into slot j % 2 first (that region was last read by the P.V of key tile j - 2,
          // issued one step earlier: the tensor pipe runs in issue order), then O_u += P_u(j-1) V_{j-1} for the
          // slot u of key tile j - 1 once its softmax has written P; j = nt only drains. Each slot's O is complete
          // after its last key tile (nt - 1 or nt - 2).
          for (int j = 0; j <= nt; ++j) {
            ok = mbar_wait_warp(bars.b_full(b_n), (b_n / C::kLag) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
            if (!ok) break;
            tc_fence_after();
            const uint32_t kslot = k_n % C::kKSlots, vslot = v_n % C::kVSlots;
            if (j < nt) {
              issue_s(0, j & 1, kslot);
              mma_commit(bars.s_full(j & 1));
            }
            if (j > 0) {
              const int u = (j - 1) & 1;
              uint32_t& pn = u ? p_n1 : p_n0;
              ok = mbar_wait_warp(bars.p_full(u), pn & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
              pn++;
              if (!ok) break;
              tc_fence_after();
              issue_pv(u, vslot, j - 1 >= 2);
              if (j - 1 >= nt - 2) mma_commit(bars.o_full(u));
            }
            mma_commit(bars.b_empty(b_n));
            if (j == nt - 1) mma_commit(bars.q_empty(0));
            if (j < nt) k_n++;
            if (j >= 1) v_n++;
            b_n++;
          }
          continue;
        }
        // Step j: O_t += P_t(j-1) V_{j-1} (j >= 1), then S_t = Q_t K_j^T (j < nt), per tile; j = nt only drains.
        for (int j = 0; j <= nt; ++j) {
          ok = mbar_wait_warp(bars.b_full(b_n), (b_n / C::kLag) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kslot = k_n % C::kKSlots, vslot = v_n % C::kVSlots;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= ntq) break;
            if (j > 0) {
              uint32_t& pn = t ? p_n1 : p_n0;
              ok = mbar_wait_warp(bars.p_full(t), pn & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
              pn++;
              if (!ok) break;
              tc_fence_after();
              issue_pv(t, vslot, j > 1);  // O_t += P_t(j-1) V_{j-1}
              if (j == nt) mma_commit(bars.o_full(t));
            }
            if (j < nt) {
              issue_s(t, t, kslot);  // S_t = Q_t K_j^T
              mma_commit(bars.s_full(t));
            }
          }
          if (!ok) break;
          mma_commit(bars.b_empty(b_n));  // K_j and V_{j-1} are free once these MMAs complete
          if (j == nt - 1) {
            mma_commit(bars.q_empty(0));
            if (ntq > 1) mma_commit(bars.q_empty(1));
          }
          if (j < nt) k_n++;
          if (j >= 1) v_n++;
          b_n++;
        }
      }
      // Every MMA and every completion arrive must have landed before the CTA tears down.
      mma_commit(bars.drain());
      mbar_wait_drain(bars.drain(), 0, ok ? kWaitLimitNs : kDrainLimitNs);
    }
    }
    teardown();
  } else {
    regs_inc<kSoftmaxRegs>();
    // ---------------------------------------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;            // query tile of this warpgroup
    const int row_in_tile = tid & 127;  // == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + C::kTmemO + t * 128;
    const uint32_t bar_s = bars.s_full(t), bar_p = bars.p_full(t), bar_o = bars.o_full(t);
    uint32_t s_n = 0, o_n = 0, st_n = 0;  // st_n: staged halves of this warpgroup
    // Alternating-key items (one query tile, keys alternating between the slots): xk_n counts them (the phase of
    // xchg_full and o1_free); the first warpgroup counts the completions of slot 1's o_full in o1_n (it waits on
    // that barrier only in these items); the second warpgroup must see o1_free before its next item (whose P.V
    // overwrites O_1, which the first warpgroup reads in the merge, and which may write the exchange again).
    uint32_t xk_n = 0, o1_n = 0;
    bool o1_pending = false;
    const uint32_t xchg = s_base + C::kXchgOff + row_in_tile * 8;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int idx = feed.fetch(n, abort_flag, err, ok);  // every softmax warp takes every item
      if (idx < 0) break;
      const Item it = load_item(prm.items, idx);
      const int ntq = (it.q_hi - it.q_lo > kTileRows) ? 2 : 1;
      const int nt0 = seg_tiles(it.s0_lo, it.s0_hi);
      const int nt = nt0 + seg_tiles(it.s1_lo, it.s1_hi);
      const bool alt = alternating_keys(ntq, nt);
      if (t == 0 && ntq > 1) o1_n++;  // slot 1's O completes once in every two-tile item
      if (t >= ntq && !alt) continue;
      if (o1_pending) {  // this item's first P would let a P.V overwrite O_1: wait until the merge has read it
        ok = mbar_wait(bars.o1_free(), (xk_n - 1) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        o1_pending = false;
        if (!ok) break;
      }
      float m = -INFINITY, l = 0.f;
      // One pass over this slot's key tiles j0, j0 + dj, ... (instantiated twice below with constant strides, so
      // that the two-tile path compiles exactly as a plain loop from key tile 0).
      auto slot_pass = [&](const int j0, const int dj) {
        for (int j = j0; j < nt; j += dj) {
          const bool first = j == j0;
          const int valid = tile_valid(it, j, nt0);
          ok = mbar_wait(bar_s, s_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          ok = __all_sync(0xffffffffu, ok);
          s_n++;
          if (!ok) break;
          tc_fence_after();
          uint32_t sr[128];
          tmem_ld_x128(tS, sr);
          float(&s)[128] = *reinterpret_cast<float(*)[128]>(sr);
          if (valid < kTileRows) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= valid) s[c] = -INFINITY;
          }
          // P = 2^(s*c - m) against the current reference m, and its row sum. The reference only has to keep P finite
          // and within a sane range, not equal the row max: the final normalisation divides by l built against the
          // same reference. So the exact row max is computed only when this step's sum exceeds 2^16 (or is not
          // finite): then the warp takes the max, raises m, redoes the exponentials and rescales l and, after the
          // first step, O. The first step starts from m = -inf, so it takes the exact max straight away.
          float row_sum = first ? INFINITY : exp_store_row(s, prm.c_scale, -m, tS);
          const bool need = !(row_sum <= kLazyLimit);
          if (__any_sync(0xffffffffu, need)) {  // warp-uniform: tcgen05.ld/st are warp-collective
            float alpha = 1.f;
            if (need) {
              // Row max: 8 independent chains of three-input maxima over 16 columns each.
              float mx[8];
#pragma unroll
              for (int a = 0; a < 8; ++a) {
                mx[a] = fmaxf(s[16 * a], s[16 * a + 15]);
#pragma unroll
                for (int c = 1; c < 15; c += 2) mx[a] = max3(mx[a], s[16 * a + c], s[16 * a + c + 1]);
              }
              const float m_cand =
                  fmaxf(max3(mx[0], mx[1], mx[2]), max3(mx[3], max3(mx[4], mx[5], mx[6]), mx[7])) * prm.c_scale;
              alpha = first ? 0.f : ex2(m - m_cand);
              m = m_cand;
            }
            row_sum = exp_store_row(s, prm.c_scale, -m, tS);  // the same P again for the lanes that kept m
            l = l * alpha + row_sum;
            if (!first) {  // O holds earlier steps' sums only after the first step
#pragma unroll
              for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld_x32(tO + c0, o);
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                tmem_st_x32(tO + c0, o);
              }
            }
          } else {
            l += row_sum;
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_p);
        }
      };
      if (alt)
        slot_pass(t, 2);
      else
        slot_pass(0, 1);
      if (!ok) break;
      if (alt && t == 1) {
        // Second half of an alternating-key item: hand (m, l) to the first warpgroup, which merges the halves and
        // waits for O_1 (o_full(1) completes for this item without this warpgroup waiting on it: count it).
        sts_f2(xchg, m, l);
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.xchg_full());
        xk_n++;
        o_n++;
        o1_pending = true;
        continue;
      }
      ok = mbar_wait(bar_o, o_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      o_n++;
      if (!ok) break;
      // Merge weights of the two halves of an alternating-key item: O = (a0 O_0 + a1 O_1) / (a0 l_0 + a1 l_1)
      // against the larger reference m (log-sum-exp merge); a0 = 1, a1 = 0 otherwise.
      float a0 = 1.f, a1 = 0.f;
      if (alt) {
        ok = mbar_wait(bars.o_full(1), o1_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
        o1_n++;
        if (ok) ok = mbar_wait(bars.xchg_full(), xk_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        xk_n++;
        if (!ok) break;
        const float2 ml1 = lds_f2(xchg);
        const float mm = fmaxf(m, ml1.x);
        a0 = ex2(m - mm);
        a1 = ex2(ml1.x - mm);
        l = a0 * l + a1 * ml1.y;
        m = mm;
      }
      tc_fence_after();
      // O of this row (columns [c0, c0 + 32)): this slot's, or the merge of both slots' for alternating keys
      const uint32_t tO1 = tmem + lane_base + C::kTmemO + 128;
      auto load_o = [&](int c0, uint32_t (&o)[32]) {
        tmem_ld_x32(tO + c0, o);
        if (alt) {
          uint32_t o1[32];
          tmem_ld_x32(tO1 + c0, o1);
#pragma unroll
          for (int c = 0; c < 32; ++c)
            o[c] = __float_as_uint(fmaf(a1, __uint_as_float(o1[c]), a0 * __uint_as_float(o[c])));
        }
      };
      // Epilogue: O / l, straight into this row's place (no scatter pass).
      const int row = it.q_lo + t * kTileRows + row_in_tile;
      const bool row_ok = row < it.q_hi;
      const float inv_l = 1.f / l;
      const int b = it.bh / prm.H, h = it.bh % prm.H;
      const int row0 = it.q_lo + t * kTileRows;
      if (C::kStage && it.split < 0 && row0 + kTileRows <= it.q_hi) {
        // A full tile: each 64-column half is packed in registers, written to this tile's stage in the store's
        // 128-byte swizzle, and stored with TMA by one thread of the warpgroup once all four warps have written
        // their rows. That thread waits for the copy engine to have read a half from the stage only when the stage
        // is needed again (for the next half, or in the next full-tile epilogue), so the read overlaps the TMEM
        // loads of what comes next.
        const uint32_t stage = s_base + C::kStageOff + t * C::kStageTileBytes;
        const bool issuer = (warp & 3) == 0 && lane == 0;
#pragma unroll 1
        for (int half = 0; half < 2 && ok; ++half) {
          uint32_t pk[32];  // the half's 64 columns of this row as bf16 pairs
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t o[32];
            load_o(half * 64 + c0, o);
#pragma unroll
            for (int c = 0; c < 16; ++c)
              pk[c0 / 2 + c] = pack_bf16(__uint_as_float(o[2 * c]) * inv_l, __uint_as_float(o[2 * c + 1]) * inv_l);
          }
          if (issuer && st_n > 0) {  // the previous store out of this stage (this tile's or an earlier one's)
            bulk_wait_read();
            mbar_arrive(bars.stage_free(t));
          }
          ok = mbar_wait(bars.stage_free(t), (st_n & 1) ^ 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          const uint32_t row_addr = stage + row_in_tile * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)  // 16-byte chunk c of the row sits at chunk c ^ (row % 8)
            sts_u4(row_addr + ((c ^ (row_in_tile & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.stage_full(t));
          if (issuer) {
            ok = mbar_wait(bars.stage_full(t), st_n & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
            if (ok) {
              tma_store_4d(&tmap_o, stage, half * 64, h, row0, b);
              bulk_commit();
            }
          }
          ok = __all_sync(0xffffffffu, ok);
          st_n++;
        }
        if (prm.lse != nullptr)  // m and l are in log2 units of the scaled score
          prm.lse[(int64_t)it.bh * prm.L + row] = (m + __log2f(l)) * 0.6931471805599453f;
      } else if (it.split < 0) {
        __nv_bfloat16* dst = prm.out + (int64_t)b * prm.sb + (int64_t)row * prm.sl + (int64_t)h * prm.sh;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          load_o(c0, o);
          uint32_t w[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            w[c] = pack_bf16(__uint_as_float(o[2 * c]) * inv_l, __uint_as_float(o[2 * c + 1]) * inv_l);
          if (row_ok) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
            for (int c = 0; c < 4; ++c) d4[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
          }
        }
        if (prm.lse != nullptr && row_ok)  // m and l are in log2 units of the scaled score
          prm.lse[(int64_t)it.bh * prm.L + row] = (m + __log2f(l)) * 0.6931471805599453f;
      } else {
        const int64_t grow = (int64_t)row - prm.g0;
        const int64_t slot = ((int64_t)it.bh * prm.G + grow) * prm.n_splits + it.split;
        float* dst = prm.ws_o + slot * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          load_o(c0, o);
          if (row_ok) {  // 32-byte stores: each fills a whole sector of the row
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * c + e]) * inv_l;
              asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + c0 + 8 * c),
                           "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7])
                           : "memory");
            }
          }
        }
        if (row_ok) prm.ws_lse[slot] = m + __log2f(l);
      }
      tc_fence_before();
      if (alt) {  // O_1 and the exchange have been read (tcgen05.ld waits are in the loads): slot 1 may move on
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.o1_free());
      }
    }
    // The warpgroup's last stores must have written out (and read their stage) before the CTA leaves.
    if (C::kStage && (warp & 3) == 0 && lane == 0) bulk_wait();
    teardown();
  }
}

// Merge the key splits of the global rows: out = sum_p 2^(lse_p - lse*) O_p with lse* the log2-sum-exp of the
// split values (each O_p is already normalised by its own row sum). One warp per global row.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                                                      __nv_bfloat16* __restrict__ out, int rows, int G, int H, int g0,
                                                      int P, int64_t sb, int64_t sl, int64_t sh, float* lse_out,
                                                      int L, int h0, int nh) {
  // rows = B * nh * G global rows of the heads [h0, h0 + nh)
  const int rr = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (rr >= rows) return;
  const int r = ((rr / (nh * G)) * H + h0 + (rr / G) % nh) * G + rr % G;  // index over all B * H * G rows
  constexpr int kPer = D / 32;
  const float* lse = ws_lse + (int64_t)r * P;
  const float* o = ws_o + (int64_t)r * P * D;
  float mx = -INFINITY;
  for (int p = 0; p < P; ++p) mx = fmaxf(mx, __ldg(lse + p));
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  float den = 0.f;
  for (int p = 0; p < P; ++p) {
    const float w = ex2(__ldg(lse + p) - mx);
    den += w;
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = fmaf(w, __ldg(o + (int64_t)p * D + lane + 32 * i), acc[i]);
  }
  const float inv = 1.f / den;
  const int bh = r / G, gr = r % G;
  const int b = bh / H, h = bh % H;
  __nv_bfloat16* dst = out + (int64_t)b * sb + (int64_t)(g0 + gr) * sl + (int64_t)h * sh;
#pragma unroll
  for (int i = 0; i < kPer; ++i) dst[lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
  if (lse_out != nullptr && lane == 0) lse_out[(int64_t)bh * L + g0 + gr] = (mx + __log2f(den)) * 0.6931471805599453f;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // Looked up once, by a thread-safe static initialisation (the driver entry point is the same in every context).
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// 4-D map over (D, H, L, B) with a (128 bytes) x 1 x 128 x 1 box and 128-byte swizzle; rows past L read as
// zeros. elem_bytes 2: bf16; 1: e4m3 (as 8-bit integers: the copy does not interpret them).
bool make_map(CUtensorMap* m, const void* ptr, const Geometry& g, int elem_bytes) {
  auto enc = encode_fn();
  if (!enc) return false;
  const wa_layout_t& l = g.layout;
  const cuuint64_t eb = (cuuint64_t)elem_bytes;
  cuuint64_t dims[4] = {(cuuint64_t)l.D, (cuuint64_t)l.H, (cuuint64_t)g.L, (cuuint64_t)l.B};
  cuuint64_t strides[3] = {(cuuint64_t)l.stride_h * eb, (cuuint64_t)l.stride_l * eb, (cuuint64_t)l.stride_b * eb};
  cuuint32_t box[4] = {(cuuint32_t)(128 / elem_bytes), 1, (cuuint32_t)kTileRows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
             const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool kF8>
int launch_attention_d(const LaunchArgs& a, cudaStream_t s, int num_sms) {
  using C = Cfg<D, kF8>;
  if (int e = ensure_smem_attr(reinterpret_cast<const void*>(&window_attention_kernel<D, kF8>), C::kSmemBytes))
    return e;
  CUtensorMap mq, mk, mv, mo;
  const int qk_bytes = kF8 ? 1 : 2;
  if (!make_map(&mq, a.q, *a.geo, qk_bytes) || !make_map(&mk, a.k, *a.geo, qk_bytes) ||
      !make_map(&mv, a.v, *a.geo, 2) || !make_map(&mo, a.out, *a.geo, 2))
    return (int)cudaErrorInvalidValue;
  const wa_layout_t& l = a.geo->layout;
  Params p;
  p.items = a.items;
  p.n_items = a.n_items;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.ws_o = a.ws_o;
  p.ws_lse = a.ws_lse;
  p.err = a.err;
  p.sb = l.stride_b;
  p.sl = l.stride_l;
  p.sh = l.stride_h;
  p.H = l.H;
  p.G = a.geo->G;
  p.g0 = (int)a.geo->g0;
  p.n_splits = a.n_splits;
  p.c_scale = (float)(1.4426950408889634 / sqrt((double)D) * (double)a.qk_scale);
  p.debug_flags = a.debug_flags;
  p.lse = a.lse;
  p.L = (int)a.geo->L;
  p.item_counter = a.item_counter;
  p.bh_count = l.B * l.H;
  const int grid = a.n_items < num_sms ? a.n_items : num_sms;
  window_attention_kernel<D, kF8><<<grid, kThreads, C::kSmemBytes, s>>>(mq, mk, mv, mo, p);
  return (int)cudaGetLastError();
}

}  // namespace

bool make_tile_map(void* map, const void* ptr, const Geometry& g, int elem_bytes) {
  return make_map(reinterpret_cast<CUtensorMap*>(map), ptr, g, elem_bytes);
}

int launch_attention(const LaunchArgs& a, void* stream, int num_sms) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (a.qk_fp8) return a.geo->layout.D == 128 ? launch_attention_d<128, true>(a, s, num_sms) : (int)cudaErrorInvalidValue;
  return a.geo->layout.D == 128 ? launch_attention_d<128, false>(a, s, num_sms)
                                : launch_attention_d<64, false>(a, s, num_sms);
}

int launch_combine(const LaunchArgs& a, void* stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Geometry& g = *a.geo;
  const wa_layout_t& l = g.layout;
  const int nh = a.head_count > 0 ? a.head_count : l.H;
  const int rows = l.B * nh * g.G;
  const int blocks = (rows + 7) / 8;
  if (l.D == 128)
    combine_kernel<128><<<blocks, 256, 0, s>>>(a.ws_o, a.ws_lse, reinterpret_cast<__nv_bfloat16*>(a.out), rows, g.G,
                                               l.H, (int)g.g0, a.n_splits, l.stride_b, l.stride_l, l.stride_h, a.lse,
                                               (int)g.L, a.head_first, nh);
  else
    combine_kernel<64><<<blocks, 256, 0, s>>>(a.ws_o, a.ws_lse, reinterpret_cast<__nv_bfloat16*>(a.out), rows, g.G,
                                              l.H, (int)g.g0, a.n_splits, l.stride_b, l.stride_l, l.stride_h, a.lse,
                                              (int)g.L, a.head_first, nh);
  return (int)cudaGetLastError();
}

}  // namespace wa
