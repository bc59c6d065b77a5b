// Host side of the library: argument checks, the window-group plan, the work list, the plan cache and the C ABI.
//
// The plan follows the VDN-Minimax-H3 window-attention article, section 三 ("the mask is a union of a few dense
// rectangles"): query rows whose kept key sets are identical form a group, and each group is one plain dense
// attention. A chunk's kept set is its clamped frame window plus the globals (section 一), so groups are runs of
// consecutive chunks whose clamped windows coincide. The article caches one plan per geometry, at most four
// (section 三, _Plan); this cache does the same and evicts the least recently used unreferenced plan.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <new>
#include <stdexcept>
#include <list>
#include <mutex>
#include <utility>

#include "wa_internal.h"

struct wa_plan {
  wa::HostPlan hp;
  std::mutex mu;  // guards the per-call host state below (last stream, profiling records, debug flags)
  int device = -1;
  int num_sms = 0;
  int refcount = 0;
  bool cached = false;
  uint64_t lru = 0;
  wa::Item* d_items = nullptr;
  float* d_ws = nullptr;  // partial outputs followed by the log-sum-exp values
  int* d_err = nullptr;       // the device error word, then two item counters of the attention kernel
  int* d_counters = nullptr;  // = d_err + 1: two ints per counter; counter 0 for wa_forward, counters 0 and 1 for the
                              // host path's two compute streams (launches on one stream are ordered)
  int64_t ws_o_elems = 0;
  cudaStream_t last_stream = nullptr;
  bool have_last = false;
  cudaEvent_t done = nullptr;
  int debug_flags = 0;
  // Launch timing (wa_plan_profile): three events per forward, recorded on the forward's stream before the
  // attention kernel, between the two kernels and after the merge kernel.
  bool profiling = false;
  int prof_n = 0;
  std::vector<cudaEvent_t> prof_ev;
  // Backward workspace (allocated by the first wa_backward): row dot products, then the split partials of the
  // global rows' dq, dk and dv. Five profiling events per recorded backward.
  float* d_bws = nullptr;
  int bprof_n = 0;
  std::vector<cudaEvent_t> bprof_ev;
  // Host-buffer forward (allocated by the first wa_forward_host): device copies of q, k, v and out with the plan's
  // layout, and the sequence cut into row pieces that are copied in one after the other. After piece p has arrived,
  // launch p runs the work items whose rows have all arrived (their list regrouped by launch), and the frame rows of
  // out that launch p completes are copied back while later pieces are still on their way.
  uint8_t* d_stage = nullptr;
  wa::Item* d_items_pc = nullptr;
  wa::HostSchedule hs;
  std::vector<int> pc_item_off;                  // launch p: items [pc_item_off[p], pc_item_off[p + 1])
  cudaStream_t s_in = nullptr, s_out = nullptr, s_c2 = nullptr;
  std::vector<cudaEvent_t> pc_ev;                // per piece: copies in, launch done; then four for the whole call
  wa::HostPlan hp_host;                          // the work list of the host path (its own global key splits)
  float* d_ws_host = nullptr;                    // its global-leg workspace: partial outputs, then log-sum-exp
  int64_t ws_o_elems_host = 0;
  bool host_ready = false;                       // all of the above set up (a failed set-up leaves none of it)
};

namespace wa {

static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

unsigned long long current_context_id() {
  // Driver entry points, looked up once (a thread-safe static initialisation).
  struct Fns {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
  };
  static const Fns fns = [] {
    Fns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
    return f;
  }();
  if (!fns.get_current || !fns.get_id) return 0;
  CUcontext ctx = nullptr;
  if (fns.get_current(&ctx) != CUDA_SUCCESS) return 0;
  if (!ctx) {  // the runtime has not made its primary context current on this thread yet: let it
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (fns.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  }
  unsigned long long id = 0;
  if (fns.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id + 1;  // never 0 for a valid context
}

int capture_state(void* stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing((cudaStream_t)stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (cs == cudaStreamCaptureStatusNone) return 0;
  return cs == cudaStreamCaptureStatusActive ? 1 : -1;
}

int ensure_smem_attr(const void* func, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, unsigned long long>> done;  // (kernel, context) pairs already set
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(mu);
  if (ctx != 0)
    for (auto& d : done)
      if (d.first == func && d.second == ctx) return 0;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return (int)e;
  if (ctx != 0) done.emplace_back(func, ctx);  // context unknown: set it again on every launch
  return 0;
}

wa_status make_geometry(int T, int S, int K, int r, int G, const wa_layout_t* layout, Geometry* geo) {
  if (!layout || !geo) return WA_ERR_INVALID;
  if (T < 1 || S < 1 || K < 1 || r < 0 || G < 0) return WA_ERR_INVALID;
  const wa_layout_t& l = *layout;
  if (l.global_pos != 0 && l.global_pos != 1) return WA_ERR_INVALID;
  if (l.B < 1 || l.H < 1 || l.D < 1) return WA_ERR_INVALID;
  if (l.D != 64 && l.D != 128) return WA_ERR_UNSUPPORTED;
  int64_t L = (int64_t)T * S + G;
  if (L >= ((int64_t)1 << 31) - kTileRows) return WA_ERR_UNSUPPORTED;
  if (l.stride_b < 1 || l.stride_l < 1 || l.stride_h < 1) return WA_ERR_INVALID;
  if (l.stride_b % 8 || l.stride_l % 8 || l.stride_h % 8) return WA_ERR_INVALID;
  // The strides must map distinct (b, l, h, d) to distinct elements: sort the outer axes by stride and check
  // that each axis starts past the end of the previous ones (d is contiguous, extent D).
  struct Ax { int64_t stride, extent; } ax[3] = {{l.stride_b, l.B}, {l.stride_l, L}, {l.stride_h, l.H}};
  std::sort(ax, ax + 3, [](const Ax& a, const Ax& b) { return a.stride < b.stride; });
  int64_t span = l.D;
  for (auto& a : ax) {
    if (a.extent == 1) continue;
    if (a.stride < span) return WA_ERR_INVALID;
    // Element offsets stay far inside int64 (and byte offsets too): 2^60 elements is past any device's memory.
    if (a.stride > (((int64_t)1 << 60) / a.extent)) return WA_ERR_UNSUPPORTED;
    span = a.stride * a.extent;
  }
  // Work items carry 32-bit (b, h) indices and are counted in 32 bits: bound the count over all B*H slices. Per
  // slice at most ceil(F / item rows) + nc window items (one partial item per group, at most nc groups) and, with
  // globals, ceil(G / item rows) items for each of at most 64 key splits. Any geometry whose four tensors fit in
  // device memory stays far below the bound (B*H*L < 2^30 elements of D >= 64 at 288 GB).
  const int64_t BH = (int64_t)l.B * l.H;
  const int64_t nc = cdiv(T, K);
  const int64_t per_slice = cdiv((int64_t)T * S, kItemRows) + nc + (G > 0 ? 64 * cdiv(G, kItemRows) : 0);
  if (per_slice > (int64_t)INT32_MAX / BH) return WA_ERR_UNSUPPORTED;
  geo->T = T; geo->S = S; geo->K = K; geo->r = r; geo->G = G;
  geo->layout = l;
  geo->nc = cdiv(T, K);
  geo->F = (int64_t)T * S;
  geo->L = L;
  geo->f0 = l.global_pos ? G : 0;
  geo->g0 = l.global_pos ? 0 : geo->F;
  return WA_OK;
}

static int64_t seg_tiles(int64_t lo, int64_t hi) { return hi > lo ? cdiv(hi - lo, kTileRows) : 0; }

void build_host_plan(const Geometry& g, HostPlan* hp, int split_mult) {
  const int64_t KS = (int64_t)g.K * g.S;
  hp->geo = g;
  hp->groups.clear();
  hp->items.clear();
  // Window groups: runs of chunks with the same clamped window [max(0, c-r), min(nc-1, c+r)].
  int64_t prev_lo = -1, prev_hi = -1;
  for (int64_t c = 0; c < g.nc; ++c) {
    int64_t lo = std::max<int64_t>(0, c - g.r), hi = std::min<int64_t>(g.nc - 1, c + g.r);
    int64_t q_lo = g.f0 + c * KS, q_hi = g.f0 + std::min<int64_t>(g.T, (c + 1) * (int64_t)g.K) * g.S;
    if (lo == prev_lo && hi == prev_hi) {
      hp->groups.back().q_hi = q_hi;
      continue;
    }
    prev_lo = lo; prev_hi = hi;
    wa_group_t gr;
    gr.q_lo = q_lo; gr.q_hi = q_hi;
    gr.kv0_lo = g.f0 + lo * KS;
    gr.kv0_hi = g.f0 + std::min<int64_t>(g.T, (hi + 1) * (int64_t)g.K) * g.S;
    gr.kv1_lo = gr.kv1_hi = 0;
    if (g.G > 0) {
      if (gr.kv0_hi == g.g0) {              // globals right after the window: one contiguous segment
        gr.kv0_hi = g.g0 + g.G;
      } else if (g.g0 + g.G == gr.kv0_lo) {  // globals right before the window
        gr.kv0_lo = g.g0;
      } else {
        gr.kv1_lo = g.g0; gr.kv1_hi = g.g0 + g.G;
      }
    }
    hp->groups.push_back(gr);
  }
  // Split count of the global leg: splits about as long as the longest window item, so that every item of the
  // persistent kernel costs about the same; split_mult times that when the global rows fill at least four items'
  // query tile pairs per head, since their split items are then plentiful, are claimed first (longest first) and
  // leave the window items to even out the finish, and longer splits mean fewer item switches (a split item's
  // switch is about four times a window item's: it writes fp32 partial rows) and a smaller merge. Measured at 56
  // heads x 99,968 rows, 2,048 global rows: twice the window item against once, forward -0.8 %, backward -1.0 %;
  // four times against twice (the device plan's kDeviceSplitMult), forward -0.3 %, the backward unchanged, and
  // -2.1 to -2.4 % on the same shape with one-frame chunks and r = 0. The host-buffer forward keeps twice
  // (kHostSplitMult): it can run a split only once every row of its key range has arrived, so a longer last split
  // leaves more work after the last copy (four times: 1.6-1.9 % slower there). With 77 global rows, one partly
  // filled query tile per head, longer splits made the forward 1.6 % slower.
  int64_t wmax = 1;
  for (auto& gr : hp->groups) wmax = std::max(wmax, seg_tiles(gr.kv0_lo, gr.kv0_hi) + seg_tiles(gr.kv1_lo, gr.kv1_hi));
  int64_t Lt = cdiv(g.L, kTileRows);
  int n_splits = 1;
  int64_t tps = Lt;
  if (g.G > 0) {
    const int64_t split_tiles = g.G >= 4 * kItemRows ? split_mult * wmax : wmax;
    int64_t p = std::min<int64_t>(64, std::max<int64_t>(1, cdiv(Lt, split_tiles)));
    tps = cdiv(Lt, p);
    n_splits = (int)cdiv(Lt, tps);
  }
  hp->n_splits = n_splits;

  const int BH = (int)((int64_t)g.layout.B * g.layout.H);  // below 2^31: bounded by make_geometry
  std::vector<Item> items;
  for (int bh = 0; bh < BH; ++bh) {
    for (auto& gr : hp->groups) {
      for (int64_t q = gr.q_lo; q < gr.q_hi; q += kItemRows) {
        Item it{bh, -1, (int32_t)q, (int32_t)std::min<int64_t>(gr.q_hi, q + kItemRows), (int32_t)gr.kv0_lo,
                (int32_t)gr.kv0_hi, (int32_t)gr.kv1_lo, (int32_t)gr.kv1_hi};
        items.push_back(it);
      }
    }
    if (g.G > 0) {
      for (int64_t q = g.g0; q < g.g0 + g.G; q += kItemRows) {
        for (int p = 0; p < n_splits; ++p) {
          int64_t lo = (int64_t)p * tps * kTileRows, hi = std::min<int64_t>(g.L, (int64_t)(p + 1) * tps * kTileRows);
          Item it{bh, p, (int32_t)q, (int32_t)std::min<int64_t>(g.g0 + g.G, q + kItemRows), (int32_t)lo,
                  (int32_t)hi, 0, 0};
          items.push_back(it);
        }
      }
    }
  }
  // Longest first (stable, so the items of one group and head stay adjacent and share keys in L2).
  auto tiles = [](const Item& it) { return seg_tiles(it.s0_lo, it.s0_hi) + seg_tiles(it.s1_lo, it.s1_hi); };
  std::stable_sort(items.begin(), items.end(), [&](const Item& a, const Item& b) { return tiles(a) > tiles(b); });
  hp->items = std::move(items);

  wa_plan_info_t& in = hp->info;
  memset(&in, 0, sizeof(in));
  in.n_chunks = (int32_t)g.nc;
  in.n_groups = (int32_t)hp->groups.size();
  in.n_splits = n_splits;
  in.n_items = (int32_t)hp->items.size();
  in.L = g.L;
  int64_t wp = 0;
  for (auto& gr : hp->groups) wp += (gr.q_hi - gr.q_lo) * ((gr.kv0_hi - gr.kv0_lo) + (gr.kv1_hi - gr.kv1_lo));
  in.window_pairs = wp;
  in.global_pairs = (int64_t)g.G * g.L;
  in.kept_pairs = wp + in.global_pairs;
  in.workspace_bytes = g.G > 0 ? (int64_t)BH * g.G * n_splits * (g.layout.D + 1) * 4 : 0;
  int64_t kt = 0;
  for (auto& it : hp->items) kt += tiles(it);
  in.kv_tiles = kt;
}


// At most this many pieces (and launches) per host-buffer forward; geometries with more window groups merge
// neighbouring pieces.
constexpr int kMaxPieces = 64;
// Head ranges of the first pieces (the globals and the first window group's rows) and of the last frame piece.
constexpr int kStartHeadSplits = 2;
constexpr int kEndHeadSplits = 4;

// One past the last sequence row that the attention kernel reads for the row range [lo, hi): it reads whole 128-row
// tiles from the start of the range, so the last tile also reads rows past its end (rows past L read as zeros).
// Those scores are masked, but 0 times a row that has not arrived yet could be NaN, so those rows must have arrived.
static int64_t read_end(const Geometry& g, int64_t lo, int64_t hi) {
  return hi > lo ? std::min<int64_t>(g.L, lo + cdiv(hi - lo, kTileRows) * kTileRows) : lo;
}

void build_host_schedule(const HostPlan& hp, HostSchedule* hs) {
  const Geometry& g = hp.geo;
  const wa_layout_t& l = g.layout;
  const int H = l.H;
  // With the heads of a row adjacent (stride_h == D), a block of sequence rows x consecutive heads of one batch
  // entry is one strided 2-D copy at full speed. Otherwise the tensors are copied whole as one piece.
  hs->rows = H == 1 || l.stride_h == l.D;
  hs->pieces.clear();
  if (!hs->rows) {
    hs->pieces.push_back({0, g.L, 0, H});
  } else {
    // The globals first (every window item reads them), then the frames in order, cut where a window group's reads
    // end: each group can start as soon as the piece holding its last row has arrived. Measured at 56 heads x
    // 99,968 rows (34 groups of one chunk; a row block copies at the full 211 GB/s host-to-device rate): 24.2 ms
    // with one chunk per piece, 24.5 with two, 25.4 with four; head groups copied as strided blocks took 27.4 ms.
    // The first launch waits for the globals and the first group's rows; to start it sooner, those two pieces
    // are split into kStartHeadSplits head ranges, so that the first group's first heads start after a fraction
    // of that copy. The copies set the pace (4.3 GB in at 211 GB/s, slowed by the copies out), so what matters
    // most is the work left after the last byte arrives: the last frame piece is split into kEndHeadSplits head
    // ranges, and each range's global rows are merged and copied back as soon as its last launch is done.
    const int64_t f_lo = g.f0, f_hi = g.f0 + g.F;
    // The last frame row read for [lo, hi), plus one (f_lo when the reads hold no frame row, e.g. the globals).
    auto frame_end = [&](int64_t lo, int64_t hi) {
      const int64_t e = std::min(read_end(g, lo, hi), f_hi);
      return hi > lo && std::max(lo, f_lo) < e ? e : f_lo;
    };
    std::vector<int64_t> cuts;  // increasing frame rows where pieces end
    for (const wa_group_t& gr : hp.groups) {
      const int64_t q_last = gr.q_lo + (gr.q_hi - gr.q_lo - 1) / kItemRows * kItemRows;  // the last item's rows
      const int64_t end = std::max({frame_end(gr.kv0_lo, gr.kv0_hi), frame_end(gr.kv1_lo, gr.kv1_hi),
                                    frame_end(q_last, gr.q_hi), f_lo + 1});
      if (cuts.empty() || end > cuts.back()) cuts.push_back(end);
    }
    if (cuts.empty() || cuts.back() != f_hi) cuts.push_back(f_hi);
    const int splits = std::min(H, kStartHeadSplits), end_splits = std::min(H, kEndHeadSplits);
    const int start_pieces = splits * (g.G > 0 ? 2 : 1);
    const int max_frame_pieces = kMaxPieces - start_pieces - end_splits + 2;
    const int n_cuts = (int)cuts.size();
    std::vector<std::pair<int64_t, int64_t>> frames;
    int64_t lo = f_lo;
    for (int i = 0; i < std::min(n_cuts, max_frame_pieces); ++i) {
      // every cut when they fit, else evenly spaced ones (always including the last)
      const int64_t hi =
          n_cuts <= max_frame_pieces ? cuts[i] : cuts[(int64_t)(i + 1) * n_cuts / max_frame_pieces - 1];
      frames.emplace_back(lo, hi);
      lo = hi;
    }
    for (int s = 0; s < splits; ++s) {
      const int h_lo = (int)((int64_t)H * s / splits), h_hi = (int)((int64_t)H * (s + 1) / splits);
      if (g.G > 0) hs->pieces.push_back({g.g0, g.g0 + g.G, h_lo, h_hi});
      hs->pieces.push_back({frames[0].first, frames[0].second, h_lo, h_hi});
    }
    for (size_t i = 1; i < frames.size(); ++i) {
      if (i + 1 < frames.size()) {
        hs->pieces.push_back({frames[i].first, frames[i].second, 0, H});
        continue;
      }
      for (int s = 0; s < end_splits; ++s)
        hs->pieces.push_back({frames[i].first, frames[i].second, (int)((int64_t)H * s / end_splits),
                              (int)((int64_t)H * (s + 1) / end_splits)});
    }
  }
  const int n_pieces = (int)hs->pieces.size();
  // The launch of an item: the latest piece among those holding a row it reads, for the item's head.
  auto last_piece = [&](int h, int64_t lo, int64_t hi) {
    int last = 0;
    if (hi <= lo) return last;
    hi = read_end(g, lo, hi);
    for (int p = 0; p < n_pieces; ++p) {
      const HostBlock& pc = hs->pieces[p];
      if (pc.h_lo <= h && h < pc.h_hi && pc.lo < hi && lo < pc.hi) last = p;
    }
    return last;
  };
  auto launch_of = [&](const Item& it) {
    const int h = it.bh % H;
    return std::max({last_piece(h, it.q_lo, it.q_hi), last_piece(h, it.s0_lo, it.s0_hi),
                     last_piece(h, it.s1_lo, it.s1_hi)});
  };
  hs->launch.resize(hp.items.size());
  for (size_t i = 0; i < hp.items.size(); ++i) hs->launch[i] = launch_of(hp.items[i]);
  // A window group's rows of out, for one head, are complete after the launch of the group's items of that head
  // (the same launch for all of them: they read the same rows). Runs of heads finished by the same launch form one
  // block; blocks of adjacent groups with the same heads and launch are merged. Without row pieces the whole of out
  // is copied back at the end instead.
  hs->out.assign(n_pieces, {});
  if (hs->rows) {
    std::vector<int> head_launch(H);
    for (const wa_group_t& gr : hp.groups) {
      for (int h = 0; h < H; ++h) {
        int launch = 0;
        for (int64_t q = gr.q_lo; q < gr.q_hi; q += kItemRows) {
          const Item it{h, -1, (int32_t)q, (int32_t)std::min<int64_t>(gr.q_hi, q + kItemRows), (int32_t)gr.kv0_lo,
                        (int32_t)gr.kv0_hi, (int32_t)gr.kv1_lo, (int32_t)gr.kv1_hi};
          launch = std::max(launch, launch_of(it));
        }
        head_launch[h] = launch;
      }
      for (int h0 = 0; h0 < H;) {
        int h1 = h0 + 1;
        while (h1 < H && head_launch[h1] == head_launch[h0]) ++h1;
        auto& blocks = hs->out[head_launch[h0]];
        if (!blocks.empty() && blocks.back().hi == gr.q_lo && blocks.back().h_lo == h0 && blocks.back().h_hi == h1)
          blocks.back().hi = gr.q_hi;
        else
          blocks.push_back({gr.q_lo, gr.q_hi, h0, h1});
        h0 = h1;
      }
    }
  }
  // The global rows of a head can be merged once its last split item has run: runs of heads whose last split item
  // is in the same launch form one merge block of that launch. Without row pieces everything is merged at the end.
  hs->merge.assign(n_pieces, {});
  if (hs->rows && g.G > 0) {
    std::vector<int> head_last(H, 0);
    for (size_t i = 0; i < hp.items.size(); ++i)
      if (hp.items[i].split >= 0) {
        const int h = hp.items[i].bh % H;
        head_last[h] = std::max(head_last[h], hs->launch[i]);
      }
    for (int h0 = 0; h0 < H;) {
      int h1 = h0 + 1;
      while (h1 < H && head_last[h1] == head_last[h0]) ++h1;
      hs->merge[head_last[h0]].push_back({g.g0, g.g0 + g.G, h0, h1});
      h0 = h1;
    }
  }
}

}  // namespace wa

// ------------------------------------------------------------------------------------------- plan cache
namespace {

std::mutex g_mu;
std::list<wa_plan*> g_cache;  // cached plans (referenced or not)
uint64_t g_tick = 0;
constexpr size_t kMaxCached = 4;

bool same_key(const wa_plan* p, int dev, const wa::Geometry& g) {
  const wa::Geometry& a = p->hp.geo;
  return p->device == dev && a.T == g.T && a.S == g.S && a.K == g.K && a.r == g.r && a.G == g.G &&
         memcmp(&a.layout, &g.layout, sizeof(wa_layout_t)) == 0;
}

void free_plan(wa_plan* p) {
  if (!p) return;
  int cur = -1;
  cudaGetDevice(&cur);
  if (p->device >= 0 && cur != p->device) cudaSetDevice(p->device);
  if (p->d_items) cudaFree(p->d_items);
  if (p->d_ws) cudaFree(p->d_ws);
  if (p->d_bws) cudaFree(p->d_bws);
  if (p->d_stage) cudaFree(p->d_stage);
  if (p->d_items_pc) cudaFree(p->d_items_pc);
  if (p->d_ws_host) cudaFree(p->d_ws_host);
  for (cudaEvent_t e : p->pc_ev)
    if (e) cudaEventDestroy(e);
  if (p->s_in) cudaStreamDestroy(p->s_in);
  if (p->s_out) cudaStreamDestroy(p->s_out);
  if (p->s_c2) cudaStreamDestroy(p->s_c2);
  if (p->d_err) cudaFree(p->d_err);
  if (p->done) cudaEventDestroy(p->done);
  for (cudaEvent_t e : p->prof_ev) cudaEventDestroy(e);
  for (cudaEvent_t e : p->bprof_ev) cudaEventDestroy(e);
  if (p->device >= 0 && cur >= 0 && cur != p->device) cudaSetDevice(cur);
  delete p;
}

bool env_flag(const char* name) {
  const char* s = getenv(name);
  return s && s[0] && strcmp(s, "0") != 0;
}

template <class T>
cudaError_t dev_alloc(T** ptr, size_t bytes) {
  if (env_flag("WA_TEST_FAIL_ALLOC")) {
    *ptr = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc((void**)ptr, bytes);
}

wa_status create_uncached(const wa::Geometry& g, int dev, wa_plan** out) {
  wa_plan* p = new (std::nothrow) wa_plan();
  if (!p) return WA_ERR_OOM;
  p->device = dev;
  if (wa::host_tables([&] { wa::build_host_plan(g, &p->hp, wa::kDeviceSplitMult); }) != WA_OK) {
    delete p;
    return WA_ERR_OOM;
  }
  if (cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete p;
    return WA_ERR_CUDA;
  }
  const size_t items_bytes = std::max<size_t>(1, p->hp.items.size()) * sizeof(wa::Item);
  const wa_plan_info_t& in = p->hp.info;
  p->ws_o_elems = (int64_t)g.layout.B * g.layout.H * g.G * p->hp.n_splits * g.layout.D;
  cudaError_t e = dev_alloc(&p->d_items, items_bytes);
  if (e == cudaSuccess && in.workspace_bytes > 0) e = dev_alloc(&p->d_ws, (size_t)in.workspace_bytes);
  if (e == cudaSuccess) e = dev_alloc(&p->d_err, 5 * sizeof(int));
  if (e == cudaSuccess) p->d_counters = p->d_err + 1;
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free allocation error
    free_plan(p);
    return e == cudaErrorMemoryAllocation ? WA_ERR_OOM : WA_ERR_CUDA;
  }
  if (cudaMemcpy(p->d_items, p->hp.items.data(), p->hp.items.size() * sizeof(wa::Item), cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      cudaMemset(p->d_err, 0, 5 * sizeof(int)) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming) != cudaSuccess) {
    free_plan(p);
    return WA_ERR_CUDA;
  }
  if (env_flag("WA_LOG")) {
    fprintf(stderr,
            "[wa] plan T=%d S=%d K=%d r=%d G=%d B=%d H=%d D=%d: %d groups, %d splits, %d items, %lld kept pairs/head, "
            "workspace %lld B\n",
            g.T, g.S, g.K, g.r, g.G, g.layout.B, g.layout.H, g.layout.D, in.n_groups, in.n_splits, in.n_items,
            (long long)in.kept_pairs, (long long)in.workspace_bytes);
  }
  *out = p;
  return WA_OK;
}

constexpr int kMaxProfiled = 4096;

bool ranges_overlap(uintptr_t a, size_t na, uintptr_t b, size_t nb) { return a < b + nb && b < a + na; }


}  // namespace

extern "C" {

const char* wa_status_string(wa_status s) {
  switch (s) {
    case WA_OK: return "WA_OK";
    case WA_ERR_INVALID: return "WA_ERR_INVALID";
    case WA_ERR_UNSUPPORTED: return "WA_ERR_UNSUPPORTED";
    case WA_ERR_OOM: return "WA_ERR_OOM";
    case WA_ERR_CUDA: return "WA_ERR_CUDA";
    case WA_ERR_DEVICE_TIMEOUT: return "WA_ERR_DEVICE_TIMEOUT";
    case WA_ERR_DEVICE_BOUNDS: return "WA_ERR_DEVICE_BOUNDS";
  }
  return "WA_UNKNOWN";
}

wa_status wa_geometry_describe(int T, int S, int K, int r, int G, const wa_layout_t* layout, wa_plan_info_t* info,
                               wa_group_t* groups, int64_t groups_cap, int64_t* items, int64_t items_cap) {
  if (!info) return WA_ERR_INVALID;
  wa::Geometry g;
  wa_status st = wa::make_geometry(T, S, K, r, G, layout, &g);
  if (st != WA_OK) return st;
  wa::HostPlan hp;
  st = wa::host_tables([&] { wa::build_host_plan(g, &hp, wa::kDeviceSplitMult); });
  if (st != WA_OK) return st;
  *info = hp.info;
  if (groups)
    for (int64_t i = 0; i < std::min<int64_t>(groups_cap, (int64_t)hp.groups.size()); ++i) groups[i] = hp.groups[i];
  if (items)
    for (int64_t i = 0; i < std::min<int64_t>(items_cap, (int64_t)hp.items.size()); ++i) {
      const wa::Item& it = hp.items[i];
      int64_t* o = items + 8 * i;
      o[0] = it.bh; o[1] = it.split < 0 ? 0 : 1; o[2] = it.q_lo; o[3] = it.q_hi;
      o[4] = it.s0_lo; o[5] = it.s0_hi; o[6] = it.s1_lo; o[7] = it.s1_hi;
    }
  return WA_OK;
}

wa_status wa_host_schedule_describe(int T, int S, int K, int r, int G, const wa_layout_t* layout, int64_t* pieces,
                                    int64_t pieces_cap, int64_t* items, int32_t* item_launch, int64_t items_cap,
                                    int64_t* out_ranges, int64_t out_cap, int64_t* n_pieces, int64_t* n_items,
                                    int64_t* n_out, int32_t* row_pieces) {
  if (!n_pieces || !n_items || !n_out || !row_pieces) return WA_ERR_INVALID;
  wa::Geometry g;
  wa_status st = wa::make_geometry(T, S, K, r, G, layout, &g);
  if (st != WA_OK) return st;
  wa::HostPlan hp;
  wa::HostSchedule hs;
  st = wa::host_tables([&] {
    wa::build_host_plan(g, &hp, wa::kHostSplitMult);
    wa::build_host_schedule(hp, &hs);
  });
  if (st != WA_OK) return st;
  *n_pieces = (int64_t)hs.pieces.size();
  *n_items = (int64_t)hp.items.size();
  *row_pieces = hs.rows ? 1 : 0;
  if (pieces)
    for (int64_t i = 0; i < std::min<int64_t>(pieces_cap, *n_pieces); ++i) {
      const wa::HostBlock& pc = hs.pieces[i];
      int64_t* o = pieces + 4 * i;
      o[0] = pc.lo; o[1] = pc.hi; o[2] = pc.h_lo; o[3] = pc.h_hi;
    }
  for (int64_t i = 0; i < std::min<int64_t>(items_cap, *n_items); ++i) {
    const wa::Item& it = hp.items[i];
    if (items) {
      int64_t* o = items + 8 * i;
      o[0] = it.bh; o[1] = it.split < 0 ? 0 : 1; o[2] = it.q_lo; o[3] = it.q_hi;
      o[4] = it.s0_lo; o[5] = it.s0_hi; o[6] = it.s1_lo; o[7] = it.s1_hi;
    }
    if (item_launch) item_launch[i] = hs.launch[i];
  }
  int64_t n = 0;
  for (size_t p = 0; p < hs.out.size(); ++p)
    for (const auto* list : {&hs.out[p], &hs.merge[p]})
      for (const wa::HostBlock& blk : *list) {
        if (out_ranges && n < out_cap) {
          int64_t* o = out_ranges + 5 * n;
          o[0] = (int64_t)p; o[1] = blk.lo; o[2] = blk.hi; o[3] = blk.h_lo; o[4] = blk.h_hi;
        }
        ++n;
      }
  *n_out = n;
  return WA_OK;
}

wa_status wa_plan_create(int T, int S, int K, int r, int G, const wa_layout_t* layout, wa_plan_t** out) {
  if (!out) return WA_ERR_INVALID;
  *out = nullptr;
  wa::Geometry g;
  wa_status st = wa::make_geometry(T, S, K, r, G, layout, &g);
  if (st != WA_OK) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return WA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  for (wa_plan* p : g_cache) {
    if (same_key(p, dev, g)) {
      p->refcount++;
      p->lru = ++g_tick;
      *out = p;
      return WA_OK;
    }
  }
  wa_plan* p = nullptr;
  st = create_uncached(g, dev, &p);
  if (st != WA_OK) return st;
  p->refcount = 1;
  p->lru = ++g_tick;
  // Make room: evict least recently used unreferenced plans; if every cached plan is in use, this one stays
  // uncached and is freed on its last release.
  while (g_cache.size() >= kMaxCached) {
    wa_plan* victim = nullptr;
    for (wa_plan* c : g_cache)
      if (c->refcount == 0 && (!victim || c->lru < victim->lru)) victim = c;
    if (!victim) break;
    g_cache.remove(victim);
    free_plan(victim);
  }
  if (g_cache.size() < kMaxCached &&
      wa::host_tables([&] { g_cache.push_back(p); }) == WA_OK)  // else the plan stays uncached
    p->cached = true;
  *out = p;
  return WA_OK;
}

void wa_plan_release(wa_plan_t* plan) {
  if (!plan) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (plan->refcount > 0) plan->refcount--;
  if (plan->refcount == 0 && !plan->cached) free_plan(plan);
}

wa_status wa_plan_info(const wa_plan_t* plan, wa_plan_info_t* info) {
  if (!plan || !info) return WA_ERR_INVALID;
  *info = plan->hp.info;
  return WA_OK;
}

// Test hook (not in the public header): set fault-injection flags of a plan.
int wa_plan_set_debug_flags(wa_plan_t* plan, int flags) {
  if (!plan) return WA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(plan->mu);
  plan->debug_flags = flags;
  return WA_OK;
}

// Test hook: number of cached plans and the reference count of a plan.
int wa_cache_size(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return (int)g_cache.size();
}
int wa_plan_refcount(const wa_plan_t* plan) { return plan ? plan->refcount : -1; }

}  // extern "C"

namespace {

// Shared body of the forward entry points. qk_bytes: element size of q and k (2 bf16, 1 e4m3); qk_scale multiplies
// the scores (the product of the e4m3 tensors' dequantisation factors; 1 for bf16).
wa_status forward_impl(wa_plan_t* plan, const void* q, const void* k, const void* v, void* out, wa_stream_t stream,
                       int qk_bytes, float qk_scale, float* lse = nullptr) {
  if (!plan || !q || !k || !v || !out) return WA_ERR_INVALID;
  if (lse && ((uintptr_t)lse & 3)) return WA_ERR_INVALID;
  auto al = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  if (!al(q) || !al(k) || !al(v) || !al(out)) return WA_ERR_INVALID;
  const wa::Geometry& g = plan->hp.geo;
  const wa_layout_t& l = g.layout;
  const size_t elems = (size_t)((l.B - 1) * l.stride_b + (g.L - 1) * l.stride_l + (l.H - 1) * l.stride_h + l.D);
  const size_t span = 2 * elems, qk_span = (size_t)qk_bytes * elems;
  uintptr_t o = (uintptr_t)out;
  if (ranges_overlap(o, span, (uintptr_t)q, qk_span) || ranges_overlap(o, span, (uintptr_t)k, qk_span) ||
      ranges_overlap(o, span, (uintptr_t)v, span))
    return WA_ERR_INVALID;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) {
    cudaGetLastError();
    return WA_ERR_INVALID;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int cap = wa::capture_state(s);
  if (cap < 0) return WA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(plan->mu);  // forwards on one plan share its workspace: serialise the host side
  if (!cap && plan->have_last && plan->last_stream != s) {
    if (cudaStreamWaitEvent(s, plan->done, 0) != cudaSuccess) return WA_ERR_CUDA;
  }
  wa::LaunchArgs a;
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.items = plan->d_items;
  a.n_items = (int)plan->hp.items.size();
  a.ws_o = plan->d_ws;
  a.ws_lse = plan->d_ws ? plan->d_ws + plan->ws_o_elems : nullptr;
  a.err = plan->d_err;
  a.n_splits = plan->hp.n_splits;
  a.debug_flags = plan->debug_flags;
  a.geo = &g;
  a.qk_fp8 = qk_bytes == 1;
  a.qk_scale = qk_scale;
  a.lse = lse;
  a.item_counter = plan->d_counters;
  cudaEvent_t* ev = nullptr;
  if (!cap && plan->profiling && plan->prof_n < kMaxProfiled) {
    while ((int)plan->prof_ev.size() < 3 * (plan->prof_n + 1)) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return WA_ERR_CUDA;
      if (wa::host_tables([&] { plan->prof_ev.push_back(e); }) != WA_OK) {
        cudaEventDestroy(e);
        return WA_ERR_OOM;
      }
    }
    ev = &plan->prof_ev[3 * plan->prof_n++];
  }
  if (ev && cudaEventRecord(ev[0], s) != cudaSuccess) return WA_ERR_CUDA;
  if (a.n_items > 0 && wa::launch_attention(a, (void*)s, plan->num_sms) != 0) return WA_ERR_CUDA;
  if (ev && cudaEventRecord(ev[1], s) != cudaSuccess) return WA_ERR_CUDA;
  if (g.G > 0 && wa::launch_combine(a, (void*)s) != 0) return WA_ERR_CUDA;
  if (ev && cudaEventRecord(ev[2], s) != cudaSuccess) return WA_ERR_CUDA;
  if (cap) return WA_OK;  // captured: the graph's launches are ordered by the stream the graph is launched on
  if (cudaEventRecord(plan->done, s) != cudaSuccess) return WA_ERR_CUDA;
  plan->last_stream = s;
  plan->have_last = true;
  return WA_OK;
}

}  // namespace

extern "C" {

wa_status wa_forward(wa_plan_t* plan, const void* q, const void* k, const void* v, void* out, wa_stream_t stream) {
  return forward_impl(plan, q, k, v, out, stream, 2, 1.0f);
}

wa_status wa_forward_lse(wa_plan_t* plan, const void* q, const void* k, const void* v, void* out, float* lse,
                         wa_stream_t stream) {
  if (!lse) return WA_ERR_INVALID;
  return forward_impl(plan, q, k, v, out, stream, 2, 1.0f, lse);
}

wa_status wa_forward_fp8(wa_plan_t* plan, const void* q8, const void* k8, const void* v, void* out, float q_scale,
                         float k_scale, wa_stream_t stream) {
  if (!plan) return WA_ERR_INVALID;
  if (!(q_scale > 0.f) || !(k_scale > 0.f) || !std::isfinite(q_scale) || !std::isfinite(k_scale) ||
      !std::isfinite(q_scale * k_scale))
    return WA_ERR_INVALID;
  if (plan->hp.geo.layout.D != 128) return WA_ERR_UNSUPPORTED;
  return forward_impl(plan, q8, k8, v, out, stream, 1, q_scale * k_scale);
}

wa_status wa_backward(wa_plan_t* plan, const void* q, const void* k, const void* v, const void* out, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, wa_stream_t stream) {
  if (!plan || !q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return WA_ERR_INVALID;
  auto al = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  if (!al(q) || !al(k) || !al(v) || !al(out) || !al(dout) || !al(dq) || !al(dk) || !al(dv) || ((uintptr_t)lse & 3))
    return WA_ERR_INVALID;
  const wa::Geometry& g = plan->hp.geo;
  const wa_layout_t& l = g.layout;
  const size_t span = 2 * (size_t)((l.B - 1) * l.stride_b + (g.L - 1) * l.stride_l + (l.H - 1) * l.stride_h + l.D);
  const size_t lse_span = (size_t)4 * l.B * l.H * g.L;
  const void* outs[3] = {dq, dk, dv};
  const void* ins[6] = {q, k, v, out, dout, lse};
  for (int i = 0; i < 3; ++i) {
    for (int j = i + 1; j < 3; ++j)
      if (ranges_overlap((uintptr_t)outs[i], span, (uintptr_t)outs[j], span)) return WA_ERR_INVALID;
    for (int j = 0; j < 6; ++j)
      if (ranges_overlap((uintptr_t)outs[i], span, (uintptr_t)ins[j], j == 5 ? lse_span : span))
        return WA_ERR_INVALID;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) {
    cudaGetLastError();
    return WA_ERR_INVALID;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int cap = wa::capture_state(s);
  if (cap < 0) return WA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(plan->mu);
  const int64_t BH = (int64_t)l.B * l.H;
  const int64_t part = BH * g.G * plan->hp.n_splits * l.D;
  // The partials are written with 16-byte vector stores: start them on a 256-byte boundary after the row dots.
  const int64_t dvec_elems = (BH * g.L + 63) / 64 * 64;
  if (!plan->d_bws) {
    if (cap) return WA_ERR_UNSUPPORTED;  // the workspace is allocated by a first call outside a capture
    const size_t bytes = (size_t)(dvec_elems + 3 * part) * sizeof(float);
    if (dev_alloc(&plan->d_bws, bytes) != cudaSuccess) {
      cudaGetLastError();
      plan->d_bws = nullptr;
      return WA_ERR_OOM;
    }
  }
  if (!cap && plan->have_last && plan->last_stream != s) {
    if (cudaStreamWaitEvent(s, plan->done, 0) != cudaSuccess) return WA_ERR_CUDA;
  }
  wa::BackwardArgs a;
  a.q = q; a.k = k; a.v = v; a.out = out; a.dout = dout; a.lse = lse;
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.items = plan->d_items;
  a.n_items = (int)plan->hp.items.size();
  a.dvec = plan->d_bws;
  a.ws = plan->d_bws + dvec_elems;
  a.part_elems = part;
  a.err = plan->d_err;
  a.n_splits = plan->hp.n_splits;
  a.debug_flags = plan->debug_flags;
  a.geo = &g;
  a.item_counter = plan->d_counters;
  void* const* ev = nullptr;
  if (!cap && plan->profiling && plan->bprof_n < kMaxProfiled) {
    while ((int)plan->bprof_ev.size() < 5 * (plan->bprof_n + 1)) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return WA_ERR_CUDA;
      if (wa::host_tables([&] { plan->bprof_ev.push_back(e); }) != WA_OK) {
        cudaEventDestroy(e);
        return WA_ERR_OOM;
      }
    }
    ev = reinterpret_cast<void* const*>(&plan->bprof_ev[5 * plan->bprof_n++]);
  }
  if (wa::launch_backward(a, (void*)s, plan->num_sms, ev) != 0) return WA_ERR_CUDA;
  if (cap) return WA_OK;  // captured: as in the forward, no cross-stream bookkeeping
  if (cudaEventRecord(plan->done, s) != cudaSuccess) return WA_ERR_CUDA;
  plan->last_stream = s;
  plan->have_last = true;
  return WA_OK;
}

namespace {

// Undo a partial set-up of the host path: the next wa_forward_host starts it again from nothing.
void release_host_path(wa_plan_t* plan) {
  for (cudaEvent_t& ev : plan->pc_ev)
    if (ev) cudaEventDestroy(ev);
  plan->pc_ev.clear();
  for (cudaStream_t* st : {&plan->s_in, &plan->s_out, &plan->s_c2}) {
    if (*st) cudaStreamDestroy(*st);
    *st = nullptr;
  }
  if (plan->d_items_pc) cudaFree(plan->d_items_pc);
  plan->d_items_pc = nullptr;
  if (plan->d_stage) cudaFree(plan->d_stage);
  plan->d_stage = nullptr;
  if (plan->d_ws_host) cudaFree(plan->d_ws_host);
  plan->d_ws_host = nullptr;
  cudaGetLastError();  // clear a non-sticky error of the failed step
}

// Lazily set up what wa_forward_host needs; called with plan->mu held. All or nothing: the host tables are built
// first (a failed host allocation throws before anything exists on the device), then every device resource; if one
// of those fails, everything set up so far is released.
wa_status prepare_host_path(wa_plan_t* plan, size_t span_bytes) {
  if (plan->host_ready) return WA_OK;
  wa::build_host_plan(plan->hp.geo, &plan->hp_host, wa::kHostSplitMult);
  const wa::HostPlan& hh = plan->hp_host;
  wa::build_host_schedule(hh, &plan->hs);
  const int n_pieces = (int)plan->hs.pieces.size();
  std::vector<std::vector<wa::Item>> by_launch(n_pieces);
  for (size_t i = 0; i < hh.items.size(); ++i)  // keeps the longest-first order inside each launch
    by_launch[plan->hs.launch[i]].push_back(hh.items[i]);
  std::vector<wa::Item> regrouped;
  regrouped.reserve(hh.items.size());
  plan->pc_item_off.assign(n_pieces + 1, 0);
  for (int p = 0; p < n_pieces; ++p) {
    regrouped.insert(regrouped.end(), by_launch[p].begin(), by_launch[p].end());
    plan->pc_item_off[p + 1] = (int)regrouped.size();
  }
  plan->pc_ev.assign(3 * n_pieces + 4, nullptr);
  const wa::Geometry& g = hh.geo;
  plan->ws_o_elems_host = (int64_t)g.layout.B * g.layout.H * g.G * hh.n_splits * g.layout.D;
  cudaError_t e = dev_alloc(&plan->d_stage, 4 * span_bytes);
  if (e == cudaSuccess) e = dev_alloc(&plan->d_items_pc, std::max<size_t>(1, regrouped.size()) * sizeof(wa::Item));
  if (e == cudaSuccess && hh.info.workspace_bytes > 0)
    e = dev_alloc(&plan->d_ws_host, (size_t)hh.info.workspace_bytes);
  if (e != cudaSuccess) {
    release_host_path(plan);
    return e == cudaErrorMemoryAllocation ? WA_ERR_OOM : WA_ERR_CUDA;
  }
  bool ok = cudaMemcpy(plan->d_items_pc, regrouped.data(), regrouped.size() * sizeof(wa::Item),
                       cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaStreamCreateWithFlags(&plan->s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&plan->s_out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&plan->s_c2, cudaStreamNonBlocking) == cudaSuccess;
  for (cudaEvent_t& ev : plan->pc_ev)
    ok = ok && cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    release_host_path(plan);
    return WA_ERR_CUDA;
  }
  plan->host_ready = true;
  return WA_OK;
}

// Copy one block (sequence rows [lo, hi) x heads [h_lo, h_hi) of every batch entry) between two buffers of the
// plan's layout: one strided 2-D copy per batch entry.
cudaError_t copy_block(const wa::Geometry& g, void* dst, const void* src, const wa::HostBlock& blk,
                       cudaMemcpyKind kind, cudaStream_t st) {
  const wa_layout_t& l = g.layout;
  const size_t width = (size_t)((blk.h_hi - blk.h_lo - 1) * l.stride_h + l.D) * 2;
  const size_t pitch = std::max<size_t>((size_t)l.stride_l * 2, width);
  for (int b = 0; b < l.B; ++b) {
    const size_t off = (size_t)(b * l.stride_b + blk.lo * l.stride_l + (int64_t)blk.h_lo * l.stride_h) * 2;
    cudaError_t e = cudaMemcpy2DAsync((uint8_t*)dst + off, pitch, (const uint8_t*)src + off, pitch, width,
                                      (size_t)(blk.hi - blk.lo), kind, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

wa_status wa_forward_host(wa_plan_t* plan, const void* q, const void* k, const void* v, void* out,
                          wa_stream_t stream) {
  if (!plan || !q || !k || !v || !out) return WA_ERR_INVALID;
  const wa::Geometry& g = plan->hp.geo;
  const wa_layout_t& l = g.layout;
  const size_t elems = (size_t)((l.B - 1) * l.stride_b + (g.L - 1) * l.stride_l + (l.H - 1) * l.stride_h + l.D);
  const size_t span = 2 * elems;
  uintptr_t o = (uintptr_t)out;
  if (ranges_overlap(o, span, (uintptr_t)q, span) || ranges_overlap(o, span, (uintptr_t)k, span) ||
      ranges_overlap(o, span, (uintptr_t)v, span))
    return WA_ERR_INVALID;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) {
    cudaGetLastError();
    return WA_ERR_INVALID;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int cap = wa::capture_state(s);
  if (cap) return cap > 0 ? WA_ERR_UNSUPPORTED : WA_ERR_CUDA;  // host copies are not captured into graphs
  std::lock_guard<std::mutex> lk(plan->mu);
  const size_t stage_span = (span + 255) / 256 * 256;
  wa_status st = WA_OK;
  if (wa::host_tables([&] { st = prepare_host_path(plan, stage_span); }) != WA_OK) return WA_ERR_OOM;
  if (st != WA_OK) return st;
  if (plan->have_last && plan->last_stream != s) {
    if (cudaStreamWaitEvent(s, plan->done, 0) != cudaSuccess) return WA_ERR_CUDA;
  }
  uint8_t* dq = plan->d_stage;
  uint8_t* dk = dq + stage_span;
  uint8_t* dv = dk + stage_span;
  uint8_t* dout = dv + stage_span;
  const int n_pieces = (int)plan->hs.pieces.size();
  cudaEvent_t* ev_in = &plan->pc_ev[0];                // piece p copied in
  cudaEvent_t* ev_comp = &plan->pc_ev[n_pieces];       // launch p done
  cudaEvent_t* ev_post = &plan->pc_ev[2 * n_pieces];   // launch p and its merges done
  cudaEvent_t ev_start = plan->pc_ev[3 * n_pieces], ev_c2 = plan->pc_ev[3 * n_pieces + 1];
  cudaEvent_t ev_merged = plan->pc_ev[3 * n_pieces + 2], ev_outdone = plan->pc_ev[3 * n_pieces + 3];
  // The helper streams start behind everything already queued on the caller's stream (earlier users of the staging).
  if (cudaEventRecord(ev_start, s) != cudaSuccess || cudaStreamWaitEvent(plan->s_in, ev_start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(plan->s_out, ev_start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(plan->s_c2, ev_start, 0) != cudaSuccess)
    return WA_ERR_CUDA;
  const void* src[3] = {q, k, v};
  uint8_t* dst[3] = {dq, dk, dv};
  wa::LaunchArgs a;
  a.q = dq; a.k = dk; a.v = dv; a.out = dout;
  a.ws_o = plan->d_ws_host;
  a.ws_lse = plan->d_ws_host ? plan->d_ws_host + plan->ws_o_elems_host : nullptr;
  a.err = plan->d_err;
  a.n_splits = plan->hp_host.n_splits;
  a.debug_flags = 0;
  a.geo = &g;
  for (int p = 0; p < n_pieces; ++p) {
    for (int x = 0; x < 3; ++x) {
      cudaError_t e = plan->hs.rows
                          ? copy_block(g, dst[x], src[x], plan->hs.pieces[p], cudaMemcpyHostToDevice, plan->s_in)
                          : cudaMemcpyAsync(dst[x], src[x], span, cudaMemcpyHostToDevice, plan->s_in);
      if (e != cudaSuccess) return WA_ERR_CUDA;
    }
    // Launches alternate between two streams, so that one launch's last items overlap the next launch's first.
    cudaStream_t cs = (p & 1) ? plan->s_c2 : s;
    if (cudaEventRecord(ev_in[p], plan->s_in) != cudaSuccess || cudaStreamWaitEvent(cs, ev_in[p], 0) != cudaSuccess)
      return WA_ERR_CUDA;
    a.items = plan->d_items_pc + plan->pc_item_off[p];
    a.n_items = plan->pc_item_off[p + 1] - plan->pc_item_off[p];
    a.item_counter = plan->d_counters + 2 * (p & 1);  // one per compute stream
    if (a.n_items > 0 && wa::launch_attention(a, (void*)cs, plan->num_sms) != 0) return WA_ERR_CUDA;
    if (cudaEventRecord(ev_comp[p], cs) != cudaSuccess) return WA_ERR_CUDA;
    const auto& merges = plan->hs.merge[p];
    if (!merges.empty()) {
      // The heads' earlier split items may have run in the other stream's launches: wait for its latest one.
      if (p >= 1 && cudaStreamWaitEvent(cs, ev_comp[p - 1], 0) != cudaSuccess) return WA_ERR_CUDA;
      for (const wa::HostBlock& blk : merges) {
        a.head_first = blk.h_lo;
        a.head_count = blk.h_hi - blk.h_lo;
        if (wa::launch_combine(a, (void*)cs) != 0) return WA_ERR_CUDA;
      }
    }
    if (plan->hs.out[p].empty() && merges.empty()) continue;
    if (cudaEventRecord(ev_post[p], cs) != cudaSuccess || cudaStreamWaitEvent(plan->s_out, ev_post[p], 0) != cudaSuccess)
      return WA_ERR_CUDA;
    for (const wa::HostBlock& blk : plan->hs.out[p])
      if (copy_block(g, out, dout, blk, cudaMemcpyDeviceToHost, plan->s_out) != cudaSuccess) return WA_ERR_CUDA;
    for (const wa::HostBlock& blk : merges)
      if (copy_block(g, out, dout, blk, cudaMemcpyDeviceToHost, plan->s_out) != cudaSuccess) return WA_ERR_CUDA;
  }
  if (cudaEventRecord(ev_c2, plan->s_c2) != cudaSuccess || cudaStreamWaitEvent(s, ev_c2, 0) != cudaSuccess)
    return WA_ERR_CUDA;
  if (!plan->hs.rows) {
    // One piece: merge every global row after the launch, then copy the whole of out back.
    a.head_first = 0;
    a.head_count = 0;
    if (g.G > 0 && wa::launch_combine(a, (void*)s) != 0) return WA_ERR_CUDA;
    if (cudaEventRecord(ev_merged, s) != cudaSuccess || cudaStreamWaitEvent(plan->s_out, ev_merged, 0) != cudaSuccess ||
        cudaMemcpyAsync(out, dout, span, cudaMemcpyDeviceToHost, plan->s_out) != cudaSuccess)
      return WA_ERR_CUDA;
  }
  if (cudaEventRecord(ev_outdone, plan->s_out) != cudaSuccess || cudaStreamWaitEvent(s, ev_outdone, 0) != cudaSuccess ||
      cudaEventRecord(plan->done, s) != cudaSuccess)
    return WA_ERR_CUDA;
  plan->last_stream = s;
  plan->have_last = true;
  return WA_OK;
}

int wa_plan_profile(wa_plan_t* plan, int enable) {
  if (!plan) return WA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(plan->mu);
  plan->profiling = enable != 0;
  plan->prof_n = 0;
  plan->bprof_n = 0;
  return WA_OK;
}

int wa_plan_profile_read_backward(wa_plan_t* plan, double* ms, int* n_backwards) {
  if (!plan || !ms || !n_backwards) return WA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(plan->mu);
  for (int k = 0; k < 4; ++k) ms[k] = 0.0;
  *n_backwards = plan->bprof_n;
  for (int i = 0; i < plan->bprof_n; ++i) {
    cudaEvent_t* ev = &plan->bprof_ev[5 * i];
    if (cudaEventSynchronize(ev[4]) != cudaSuccess) return WA_ERR_CUDA;
    for (int k = 0; k < 4; ++k) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, ev[k], ev[k + 1]) != cudaSuccess) return WA_ERR_CUDA;
      ms[k] += t;
    }
  }
  return WA_OK;
}

int wa_plan_profile_read(wa_plan_t* plan, double* attention_ms, double* combine_ms, int* n_forwards) {
  if (!plan || !attention_ms || !combine_ms || !n_forwards) return WA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(plan->mu);
  *attention_ms = *combine_ms = 0.0;
  *n_forwards = plan->prof_n;
  for (int i = 0; i < plan->prof_n; ++i) {
    cudaEvent_t* ev = &plan->prof_ev[3 * i];
    float a = 0.f, c = 0.f;
    if (cudaEventSynchronize(ev[2]) != cudaSuccess || cudaEventElapsedTime(&a, ev[0], ev[1]) != cudaSuccess ||
        cudaEventElapsedTime(&c, ev[1], ev[2]) != cudaSuccess)
      return WA_ERR_CUDA;
    *attention_ms += a;
    *combine_ms += c;
  }
  return WA_OK;
}

wa_status wa_plan_check_error(wa_plan_t* plan, wa_stream_t stream) {
  if (!plan) return WA_ERR_INVALID;
  const int cap = wa::capture_state(stream);
  if (cap) return cap > 0 ? WA_ERR_UNSUPPORTED : WA_ERR_CUDA;  // it synchronises: never inside a capture
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return WA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, plan->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return WA_ERR_CUDA;
  if (h && cudaMemset(plan->d_err, 0, sizeof(int)) != cudaSuccess) return WA_ERR_CUDA;
  if (h & wa::kErrTimeout) return WA_ERR_DEVICE_TIMEOUT;
  if (h & wa::kErrBounds) return WA_ERR_DEVICE_BOUNDS;
  return WA_OK;
}

}  // extern "C"
