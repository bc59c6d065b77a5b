// Internal declarations shared by the host plan/ABI code and the CUDA launchers.
#pragma once

#include <stdint.h>

#include <new>
#include <stdexcept>
#include <utility>
#include <vector>

#include "../../include/wa.h"

namespace wa {

constexpr int kTileRows = 128;    // query rows per tile and key rows per key tile
constexpr int kItemQTiles = 2;    // query tiles per work item (they share the key tiles)
constexpr int kItemRows = kTileRows * kItemQTiles;

// One work item of the attention kernel, 8 x int32 (two 16-byte loads on the device).
//   split < 0: window item, the query rows [q_lo, q_hi) are written as bf16 rows of `out`.
//   split >= 0: global-leg item, the rows are written as fp32 partials + log2-sum-exp to the workspace at
//               split index `split`.
// Keys: segment 0 [s0_lo, s0_hi) then segment 1 [s1_lo, s1_hi) (empty when equal), processed in key tiles of
// kTileRows rows; the last tile of each segment is column-masked.
struct Item {
  int32_t bh, split, q_lo, q_hi, s0_lo, s0_hi, s1_lo, s1_hi;
};
static_assert(sizeof(Item) == 32, "work item is 32 bytes");

struct Geometry {
  int T, S, K, r, G;
  wa_layout_t layout;
  int64_t nc, F, L, f0, g0;
};

struct HostPlan {
  Geometry geo;
  wa_plan_info_t info;
  std::vector<wa_group_t> groups;
  std::vector<Item> items;
  int n_splits;
};

// The piece schedule of the host-buffer forward: blocks of sequence rows x heads (all batch entries) copied in one
// after the other; after piece p, launch p of the items whose rows have all arrived; after launch p, the blocks of
// out it completed are copied back.
struct HostBlock {
  int64_t lo, hi;  // sequence rows [lo, hi)
  int h_lo, h_hi;  // heads [h_lo, h_hi)
};
struct HostSchedule {
  bool rows = false;                         // pieces are row blocks (else one piece: the whole tensors)
  std::vector<HostBlock> pieces;             // in copy order
  std::vector<int> launch;                   // per item of HostPlan::items (same order): the launch that runs it
  std::vector<std::vector<HostBlock>> out;    // per launch: the blocks of out (frame rows) it completes
  std::vector<std::vector<HostBlock>> merge;  // per launch: global-row blocks whose heads' split items are all done
                                              // after it (merged, then copied back, right behind it)
};

// Validate arguments; on success fill `geo`.
wa_status make_geometry(int T, int S, int K, int r, int G, const wa_layout_t* layout, Geometry* geo);
// Key splits of the global leg, in multiples of the longest window item (when the global rows are plentiful): the
// device plans' work list, and the host-buffer forward's own list (which keeps the last split short).
constexpr int kDeviceSplitMult = 4;
constexpr int kHostSplitMult = 2;
// Build groups, splits and the ordered work list on the host.
void build_host_plan(const Geometry& geo, HostPlan* hp, int split_mult = kDeviceSplitMult);
// Build the host-buffer forward's piece schedule for a plan (host only).
void build_host_schedule(const HostPlan& hp, HostSchedule* hs);
// Run `build` (which fills host-side tables) so that no C++ exception leaves the C ABI: a failed host allocation
// becomes WA_ERR_OOM. Geometries that pass make_geometry have bounded tables, so this is only reached when the host
// itself is out of memory.
template <class F>
wa_status host_tables(F&& build) {
  try {
    build();
  } catch (const std::bad_alloc&) {
    return WA_ERR_OOM;
  } catch (const std::length_error&) {
    return WA_ERR_OOM;
  }
  return WA_OK;
}

// Arguments of one attention launch (device pointers; tensor maps are built by the launcher).
struct LaunchArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const Item* items;
  int n_items;
  float* ws_o;      // [B*H][G][n_splits][D] fp32 (global leg partial outputs, normalised per split)
  float* ws_lse;    // [B*H][G][n_splits] fp32 (log2-domain log-sum-exp of the scaled scores per split)
  int* err;         // device error word
  int n_splits;
  int debug_flags;  // test-only fault injection on the host-visible error path (0 in normal use)
  const Geometry* geo;
  float* lse = nullptr;    // optional [B][H][L] fp32 output: natural-log sum of exp of each row's scaled scores
  int qk_fp8 = 0;          // q and k are e4m3 (scores by kind::f8f6f4 MMAs); v and out stay bf16
  float qk_scale = 1.0f;   // dequantisation factor of the scores: q_scale * k_scale (1 for bf16 inputs)
  int head_first = 0;      // the merge covers the heads [head_first, head_first + head_count) of every batch entry
  int head_count = 0;      // (0: all heads)
  int* item_counter = nullptr;  // two device ints, zero before the launch and zero again after it: items are claimed
                                // dynamically by the CTAs (nullptr: CTA c runs items c, c + grid, ...)
};

// Encode the tensor maps and launch the attention kernel; returns a CUDA error code (0 on success).
int launch_attention(const LaunchArgs& a, void* stream, int num_sms);
// Launch the log-sum-exp merge of the global rows; returns a CUDA error code.
int launch_combine(const LaunchArgs& a, void* stream);

// Arguments of one backward pass (device pointers; every [B, L, H, D] tensor has the plan's strides).
struct BackwardArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* out;    // the forward's output
  const void* dout;   // gradient of the loss with respect to out
  const float* lse;   // [B][H][L] natural-log row log-sum-exp written by the forward
  void* dq;
  void* dk;
  void* dv;
  const Item* items;
  int n_items;
  float* dvec;        // [B*H][L] scratch: dout_i . out_i
  float* ws;          // 3 x part_elems fp32 scratch: split partials of the global rows' dq, dk, dv
  int64_t part_elems; // B*H*G*n_splits*D
  int* err;
  int n_splits;
  int debug_flags;
  const Geometry* geo;
  int* item_counter = nullptr;  // as LaunchArgs::item_counter, shared by the dq and dk/dv launches (stream-ordered)
};

// Launch the backward (row dot products, dq kernel, dk/dv kernel, split sums) on `stream`. `events`, when not null,
// holds five CUDA events recorded before, between and after the four launches. Returns a CUDA error code.
int launch_backward(const BackwardArgs& a, void* stream, int num_sms, void* const* events);

// Identity of the CUDA context current on the calling thread (the driver's context id: unique for the life of the
// process, so a context created after cudaDeviceReset gets a new one). Makes the device's primary context current
// first when the runtime has not yet done so. Returns 0 when it cannot be read.
unsigned long long current_context_id();
// Opt `func` into `bytes` of dynamic shared memory in the current context, once per (kernel, context): the
// attribute belongs to the context, so a second device (or a context rebuilt after a reset) needs its own call.
// Thread-safe. Returns a CUDA error code (0 on success).
int ensure_smem_attr(const void* func, int bytes);
// Capture state of a stream: 0 = not capturing, 1 = being captured into a CUDA graph, -1 = the query failed or the
// capture was invalidated. A captured call runs whenever the graph is launched, on the stream it is launched on, so
// it takes no part in a plan's cross-stream ordering: the caller orders graph launches against other uses of the
// plan (or of the allocation-free entry point's shared array).
int capture_state(void* stream);

// Encode the 4-D TMA map of a [B, L, H, D] tensor (box 128 bytes x 1 x 128 rows x 1, 128-byte swizzle) into
// `map` (a 64-byte aligned CUtensorMap). elem_bytes 2: bf16, 1: 8-bit. Returns false if encoding fails.
bool make_tile_map(void* map, const void* ptr, const Geometry& g, int elem_bytes);

// Device error word bits.
constexpr int kErrTimeout = 1;
constexpr int kErrBounds = 2;

}  // namespace wa
