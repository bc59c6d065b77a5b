// Device helpers shared by the forward and backward kernels: the work-item view, wait limits and bf16 packing.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "wa_internal.h"

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

// Two fp32 values rounded to nearest-even bf16 and packed low-first into 32 bits.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v2 = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v2);
}

}  // namespace wa
