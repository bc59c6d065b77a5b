// Device helpers shared by the forward and backward kernels: the work-item view and its hand-out to the CTAs of
// a persistent launch, wait limits and bf16 packing.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "wa_internal.h"
#include "wa_ptx.cuh"

namespace wa {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr uint64_t kDrainLimitNs = 20000000ull;   // 20 ms: waiting for in-flight copies while unwinding

// One work item, read as two 16-byte loads.
__device__ __forceinline__ Item load_item(const Item* items, int idx) {
  const int4* p = reinterpret_cast<const int4*>(items + idx);
  int4 a = __ldg(p), b = __ldg(p + 1);
  return Item{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
}

// Number of 128-row tiles of the half-open row range [lo, hi).
__device__ __forceinline__ int seg_tiles(int lo, int hi) { return hi > lo ? (hi - lo + kTileRows - 1) / kTileRows : 0; }

// Rows of the j-th 128-row tile of an item's key segments that lie inside the segment (128 except in a segment's
// last tile); nt0 = seg_tiles of segment 0.
__device__ __forceinline__ int tile_valid(const Item& it, int j, int nt0) {
  return j < nt0 ? min(kTileRows, it.s0_hi - (it.s0_lo + j * kTileRows))
                 : min(kTileRows, it.s1_hi - (it.s1_lo + (j - nt0) * kTileRows));
}

// Index checks of a debug build (compiled with -DWA_DEBUG; they stand in for a memory checker). An item is in
// bounds when its head index is below B*H, its query rows are a non-empty range of at most two tiles inside [0, L),
// segment 0 is a non-empty and segment 1 a possibly empty range inside [0, L), and a global split item's split index
// is below n_splits and its query rows lie inside the global rows [g0, g0 + G). Every copy coordinate and store row
// of the kernels derives from these fields. The claiming thread checks each item before any role uses it; a failed
// check latches the bounds error and unwinds the CTA without touching memory for that item.
struct ItemBounds {
  int bh_count, L, g0, G, n_splits;
};
__device__ __forceinline__ bool item_in_bounds(const Item& it, const ItemBounds& b) {
  const bool head = it.bh >= 0 && it.bh < b.bh_count;
  const bool rows = it.q_lo >= 0 && it.q_lo < it.q_hi && it.q_hi <= b.L && it.q_hi - it.q_lo <= kItemRows;
  const bool seg0 = it.s0_lo >= 0 && it.s0_lo < it.s0_hi && it.s0_hi <= b.L;
  const bool seg1 = it.s1_lo >= 0 && it.s1_lo <= it.s1_hi && it.s1_hi <= b.L;
  const bool split = it.split == -1 ||
                     (it.split >= 0 && it.split < b.n_splits && it.q_lo >= b.g0 && it.q_hi <= b.g0 + b.G);
  return head && rows && seg0 && seg1 && split;
}

// Zero rows [valid, 128) of a 128-row tile held in shared memory as `boxes` consecutive boxes of 128 rows x 128
// bytes (a row of a box is 128 contiguous bytes, so the 128-byte swizzle inside a row does not matter). A segment's
// last tile is copied whole and so holds rows past the segment's end: tokens outside the rows' kept sets, or past
// the sequence (zero-filled by the copy). Their scores or probabilities are masked to zero, but a tensor-core
// product of zero with an Inf or NaN there would still be NaN; zeroing the rows keeps every result independent of
// tokens outside its kept set. Called by all 32 lanes of a warp after the tile's copy has completed; the writes are
// fenced for the tensor core's (async-proxy) reads and the warp is reconverged before it returns.
__device__ __forceinline__ void zero_tile_rows(uint32_t tile, int boxes, int valid, int lane) {
  const uint32_t chunks = (uint32_t)(kTileRows - valid) * 8;  // 16-byte chunks per box
  for (int hf = 0; hf < boxes; ++hf) {
    const uint32_t base = tile + (uint32_t)(hf * kTileRows * 128 + valid * 128);
    for (uint32_t c = lane; c < chunks; c += 32) ptx::sts_u4(base + 16 * c, 0u, 0u, 0u, 0u);
  }
  ptx::fence_proxy_async_smem();
  __syncwarp();
}

// Hand-out of the work items of a persistent launch to its CTAs. Without a counter, CTA c runs the items c,
// c + grid, c + 2 grid, ... With a counter (two device ints, zero when the launch starts: items claimed so far and
// CTAs finished), one producer thread of each CTA claims the next unclaimed item when it is ready for one, so CTAs
// that run faster take more items and all of them finish within about one item of each other; it passes the index
// to the CTA's consuming warps through a ring of kItemRingSlots shared-memory slots, each guarded by a "full"
// mbarrier (the index is written) and an "empty" one (every consuming warp has read it). The last CTA to finish
// sets the counter back to zero for the next launch. Every wait is bounded.
constexpr int kItemRingSlots = 4;

struct ItemFeed {
  int* counter;         // nullptr: static striding
  int n_items;
  volatile int* ring;   // kItemRingSlots ints of shared memory
  uint32_t bars;        // 2 * kItemRingSlots mbarriers (8 bytes each): full[kItemRingSlots], then empty[...]

  __device__ __forceinline__ bool dynamic() const { return counter != nullptr; }
  __device__ __forceinline__ uint32_t full(uint32_t n) const { return bars + 8 * (n % kItemRingSlots); }
  __device__ __forceinline__ uint32_t empty(uint32_t n) const {
    return bars + 8 * (kItemRingSlots + n % kItemRingSlots);
  }
  __device__ __forceinline__ int static_item(uint32_t n) const {
    const int64_t i = blockIdx.x + (int64_t)n * gridDim.x;
    return i < n_items ? (int)i : -1;
  }
  // One thread, before the CTA's first barrier sync: `consumers` warps read every index.
  __device__ __forceinline__ void init(int consumers) const {
    for (int s = 0; s < kItemRingSlots; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), consumers);
    }
  }
  // The producer thread: the item of its n-th iteration, or -1 when there are no more (or on an error: ok = false).
  __device__ __forceinline__ int claim(uint32_t n, volatile int* abort_flag, int* err, bool& ok) const {
    if (!dynamic()) return static_item(n);
    if (n >= (uint32_t)kItemRingSlots) {  // the slot's previous index must have been read by every consumer
      const uint32_t w = n - kItemRingSlots;
      ok = ptx::mbar_wait(empty(w), (w / kItemRingSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
      if (!ok) return -1;
    }
    int i = atomicAdd(counter, 1);
    if (i >= n_items) i = -1;
    ring[n % kItemRingSlots] = i;
    ptx::mbar_arrive(full(n));  // release: the index is visible to whoever completes the wait
    return i;
  }
  // claim() for a producer that is a whole warp: lane 0 claims, every lane gets the index and the outcome.
  __device__ __forceinline__ int claim_warp(uint32_t n, volatile int* abort_flag, int* err, bool& ok) const {
    int i = -1;
    bool good = true;
    if ((threadIdx.x & 31) == 0) i = claim(n, abort_flag, err, good);
    i = __shfl_sync(0xffffffffu, i, 0);
    if (!__shfl_sync(0xffffffffu, (int)good, 0)) ok = false;
    return i;
  }
  // A whole consuming warp: the same item as the producer's n-th iteration, or -1 (ok = false on an error).
  __device__ __forceinline__ int fetch(uint32_t n, volatile int* abort_flag, int* err, bool& ok) const {
    if (!dynamic()) return static_item(n);
    ok = ptx::mbar_wait(full(n), (n / kItemRingSlots) & 1, abort_flag, err, kErrTimeout, kWaitLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return -1;
    const int i = ring[n % kItemRingSlots];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(empty(n));
    return i;
  }
  // One thread per CTA, once every role of the CTA is done: the last CTA out rewinds the counter.
  __device__ __forceinline__ void finish() const {
    if (!dynamic()) return;
    __threadfence();
    if (atomicAdd(counter + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(counter, 0);
      atomicExch(counter + 1, 0);
    }
  }
};

// Two fp32 values rounded to nearest-even bf16 and packed low-first into 32 bits.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v2 = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v2);
}

}  // namespace wa
