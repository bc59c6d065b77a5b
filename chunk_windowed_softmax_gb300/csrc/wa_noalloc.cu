// wa_forward_static: the forward pass for callers that may not allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention: a framework that hands out device
// memory only from its own pool and counts every byte, a process that runs under a fixed device-memory budget,
// or code that must not trigger the device-wide synchronisation that cudaMalloc / cudaFree can cause. wa_forward
// needs a plan, and a plan allocates its work-list table, its global-leg workspace and its error word. This entry
// point runs the same two kernels with all of that scratch placed in one file-scope __device__ array instead,
// so it allocates no device memory at all: the caller passes only the inputs and the output.
//
// The array is kScratchBytes (32 MiB) and exists on every GPU where this library's device code is loaded, until
// the process exits. Geometries whose scratch does not fit are rejected with WA_ERR_UNSUPPORTED before anything
// is launched. All calls share the one array, so calls that overlap on the GPU (two streams, two threads) race
// on it; calls on one stream are ordered and safe.
#include <cuda_runtime.h>

#include <mutex>
#include <utility>
#include <vector>

#include "wa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

// [0, 256): device error word; then the work list; then the fp32 partial outputs; then the log2-sum-exp values.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// The work list is written on the device by expand_items_kernel, from per-head item templates passed by value as
// kernel parameters: nothing is copied from host memory. The plan's list is the per-head list (one template per
// window query-tile pair and per global query-tile pair and split) repeated for every (b, h) and sorted stably,
// longest first; so the templates are the per-head list sorted the same way, and a template t in the run [a, b)
// of templates with equal key-tile counts lands at a * BH + bh * (b - a) + (t - a) for head index bh.
struct ItemTemplate {
  int32_t split, q_lo, q_hi, s0_lo, s0_hi, s1_lo, s1_hi;
  int32_t base;    // a * BH + (t - a)
  int32_t stride;  // b - a
};
constexpr int kTemplatesPerLaunch = 800;  // 28.8 KB of parameters, under the 32,764-byte kernel-parameter limit
struct ExpandParams {
  int n_tpl;  // templates in this launch
  int BH;
  int* err;   // non-null in the first launch: the error word is cleared
  ItemTemplate tpl[kTemplatesPerLaunch];
};
static_assert(sizeof(ExpandParams) <= 32764, "kernel parameter limit");

__global__ void expand_items_kernel(const __grid_constant__ ExpandParams p, wa::Item* items) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0 && p.err != nullptr) *p.err = 0;
  if (i >= p.n_tpl * p.BH) return;
  const int bh = i / p.n_tpl;
  const ItemTemplate& t = p.tpl[i % p.n_tpl];
  items[t.base + bh * t.stride] = wa::Item{bh, t.split, t.q_lo, t.q_hi, t.s0_lo, t.s0_hi, t.s1_lo, t.s1_hi};
}

std::mutex g_mu;
// Device address of g_scratch per CUDA context (context id, address), looked up once per context with that
// context current. A context created after cudaDeviceReset has a new id, so its address is looked up again.
std::vector<std::pair<unsigned long long, void*>> g_scratch_addr;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool overlap(uintptr_t a, size_t na, uintptr_t b, size_t nb) { return a < b + nb && b < a + na; }

}  // namespace

extern "C" wa_status wa_forward_static(int T, int S, int K, int r, int G, const wa_layout_t* layout, const void* q,
                                       const void* k, const void* v, void* out, wa_stream_t stream) {
  if (!q || !k || !v || !out) return WA_ERR_INVALID;
  wa::Geometry g;
  wa_status st = wa::make_geometry(T, S, K, r, G, layout, &g);
  if (st != WA_OK) return st;
  auto aligned = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
  if (!aligned(q) || !aligned(k) || !aligned(v) || !aligned(out)) return WA_ERR_INVALID;
  const wa_layout_t& l = g.layout;
  const size_t span = 2 * (size_t)((l.B - 1) * l.stride_b + (g.L - 1) * l.stride_l + (l.H - 1) * l.stride_h + l.D);
  const uintptr_t o = (uintptr_t)out;
  if (overlap(o, span, (uintptr_t)q, span) || overlap(o, span, (uintptr_t)k, span) ||
      overlap(o, span, (uintptr_t)v, span))
    return WA_ERR_INVALID;

  // The per-head work list, built on the host exactly as for a plan (a geometry with one (b, h) slice: groups and
  // splits do not depend on B or H), already sorted longest first.
  wa::Geometry g1 = g;
  g1.layout.B = 1;
  g1.layout.H = 1;
  wa::HostPlan hp;
  if (wa::host_tables([&] { wa::build_host_plan(g1, &hp); }) != WA_OK) return WA_ERR_OOM;
  const int BH = l.B * l.H;
  const size_t n_tpl = hp.items.size();
  const size_t n_items = n_tpl * (size_t)BH;
  const size_t items_bytes = align256(n_items * sizeof(wa::Item));
  const size_t ws_rows = (size_t)BH * g.G * hp.n_splits;
  const size_t ws_o_bytes = align256(ws_rows * l.D * sizeof(float));
  const size_t need = 256 + items_bytes + ws_o_bytes + ws_rows * sizeof(float);
  if (need > kScratchBytes) return WA_ERR_UNSUPPORTED;

  int dev = -1, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return WA_ERR_CUDA;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int cap = wa::capture_state(s);
  if (cap < 0) return WA_ERR_CUDA;
  void* base = nullptr;
  {
    // First call in a context: look up the array's device address with that context current. In host code the
    // name g_scratch is only a host-side stand-in and must never be handed to a kernel.
    const unsigned long long ctx = wa::current_context_id();
    std::lock_guard<std::mutex> lk(g_mu);
    if (ctx != 0)
      for (auto& e : g_scratch_addr)
        if (e.first == ctx) base = e.second;
    if (!base) {
      if (cap) return WA_ERR_UNSUPPORTED;  // the address is looked up by a first call outside a capture
      if (cudaGetSymbolAddress(&base, g_scratch) != cudaSuccess || !base) {
        cudaGetLastError();
        return WA_ERR_CUDA;
      }
      if (ctx != 0)  // context unknown (or no room to remember it): look it up on every call
        wa::host_tables([&] { g_scratch_addr.emplace_back(ctx, base); });
    }
  }
  unsigned char* b = static_cast<unsigned char*>(base);
  int* err = reinterpret_cast<int*>(b);
  wa::Item* items = reinterpret_cast<wa::Item*>(b + 256);
  float* ws_o = reinterpret_cast<float*>(b + 256 + items_bytes);
  float* ws_lse = reinterpret_cast<float*>(b + 256 + items_bytes + ws_o_bytes);

  // The array keeps the previous call's contents: the first expansion launch clears the error word; the work list
  // is rewritten in full; every workspace entry the merge reads is written by the attention kernel first.
  {
    std::vector<int> run_lo, run_hi;  // the run of equal key-tile counts each template belongs to
    if (wa::host_tables([&] {
          run_lo.resize(n_tpl);
          run_hi.resize(n_tpl);
        }) != WA_OK)
      return WA_ERR_OOM;
    auto tiles = [](const wa::Item& it) {
      auto seg = [](int lo, int hi) { return hi > lo ? (hi - lo + wa::kTileRows - 1) / wa::kTileRows : 0; };
      return seg(it.s0_lo, it.s0_hi) + seg(it.s1_lo, it.s1_hi);
    };
    for (size_t a = 0; a < n_tpl;) {
      size_t e = a + 1;
      while (e < n_tpl && tiles(hp.items[e]) == tiles(hp.items[a])) ++e;
      for (size_t t = a; t < e; ++t) {
        run_lo[t] = (int)a;
        run_hi[t] = (int)e;
      }
      a = e;
    }
    static ExpandParams prm;  // 29 KB: kept off the stack; guarded by the lock below
    static std::mutex prm_mu;
    std::lock_guard<std::mutex> lk(prm_mu);
    for (size_t t0 = 0; t0 < n_tpl; t0 += kTemplatesPerLaunch) {
      const int n = (int)std::min<size_t>(kTemplatesPerLaunch, n_tpl - t0);
      prm.n_tpl = n;
      prm.BH = BH;
      prm.err = t0 == 0 ? err : nullptr;
      for (int i = 0; i < n; ++i) {
        const size_t t = t0 + i;
        const wa::Item& it = hp.items[t];
        prm.tpl[i] = ItemTemplate{it.split, it.q_lo, it.q_hi, it.s0_lo, it.s0_hi, it.s1_lo, it.s1_hi,
                                  (int32_t)((size_t)run_lo[t] * BH + (t - run_lo[t])), run_hi[t] - run_lo[t]};
      }
      const int threads = 256, total = n * BH;
      expand_items_kernel<<<(total + threads - 1) / threads, threads, 0, s>>>(prm, items);
      if (cudaGetLastError() != cudaSuccess) return WA_ERR_CUDA;
    }
  }

  wa::LaunchArgs a;
  a.q = q; a.k = k; a.v = v; a.out = out;
  a.items = items;
  a.n_items = (int)n_items;
  a.ws_o = g.G > 0 ? ws_o : nullptr;
  a.ws_lse = g.G > 0 ? ws_lse : nullptr;
  a.err = err;
  a.n_splits = hp.n_splits;
  a.debug_flags = 0;
  a.geo = &g;
  if (wa::launch_attention(a, (void*)s, num_sms) != 0) return WA_ERR_CUDA;
  if (g.G > 0 && wa::launch_combine(a, (void*)s) != 0) return WA_ERR_CUDA;
  return WA_OK;
}
