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

#include "wa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

// [0, 256): device error word; then the work list; then the fp32 partial outputs; then the log2-sum-exp values.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_scratch per device, looked up once

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

  // The work list is built on the host exactly as for a plan; it is copied into the scratch on every call.
  wa::HostPlan hp;
  wa::build_host_plan(g, &hp);
  const size_t n_items = hp.items.size();
  const size_t items_bytes = align256(n_items * sizeof(wa::Item));
  const size_t ws_rows = (size_t)l.B * l.H * g.G * hp.n_splits;
  const size_t ws_o_bytes = align256(ws_rows * l.D * sizeof(float));
  const size_t need = 256 + items_bytes + ws_o_bytes + ws_rows * sizeof(float);
  if (need > kScratchBytes) return WA_ERR_UNSUPPORTED;

  int dev = -1, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return WA_ERR_CUDA;
  }
  void* base = nullptr;
  {
    // First call on a device: look up the array's device address with that device current. In host code the
    // name g_scratch is only a host-side stand-in and must never be handed to a kernel.
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return WA_ERR_CUDA;
      }
      g_scratch_addr[dev] = p;
    }
    base = g_scratch_addr[dev];
  }
  unsigned char* b = static_cast<unsigned char*>(base);
  int* err = reinterpret_cast<int*>(b);
  wa::Item* items = reinterpret_cast<wa::Item*>(b + 256);
  float* ws_o = reinterpret_cast<float*>(b + 256 + items_bytes);
  float* ws_lse = reinterpret_cast<float*>(b + 256 + items_bytes + ws_o_bytes);

  cudaStream_t s = (cudaStream_t)stream;
  // The array keeps the previous call's contents: the error word must start at zero; the work list is rewritten;
  // every workspace entry the merge reads is written by the attention kernel first.
  if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess ||
      cudaMemcpyAsync(items, hp.items.data(), n_items * sizeof(wa::Item), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return WA_ERR_CUDA;

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
