/*
 * wa.h -- chunk-aligned window softmax attention for GB300 (sm_103a): the C ABI.
 *
 * The operation (VDN-Minimax-H3 window-attention article, lqnn.cn, sections 一 and 三):
 *   The packed sequence holds T latent frames of S spatial tokens each plus G global (text/audio) tokens,
 *   L = T*S + G rows. Frames are grouped into chunks of K consecutive frames (chunk c = floor(t / K); the
 *   last chunk may be partial). A query token of a frame in chunk c attends to every token of the chunks in
 *   [c - r, c + r] that exist, plus all G global tokens; a global query attends to all L tokens. Each query's
 *   softmax is normalised over exactly that kept set; scores are scaled by 1/sqrt(D); non-causal.
 *   The library computes it the article's "decomposed" way (section 三): query rows with identical kept sets
 *   form a group and each group is one dense attention over its frame window plus the globals (the window
 *   leg); the G global rows run one dense attention over the whole sequence (the global leg, split along the
 *   keys and merged by log-sum-exp). The legs write disjoint row sets straight into the output.
 *
 * Layout: q, k, v and out are bf16 device tensors of logical shape [B, L, H, D] with the element strides given
 * in wa_layout_t (the D axis contiguous). Frame token (t, s) is row f0 + t*S + s, global token g is row g0 + g,
 * where (f0, g0) = (0, T*S) when global_pos == 0 (globals after the frames) and (G, 0) when global_pos == 1.
 *
 * Threading: every function may be called from any host thread; the plan cache is mutex-guarded.
 * Errors: argument errors are returned synchronously and launch nothing. Device-side watchdog and bounds
 * failures are latched in the plan and reported by wa_plan_check_error().
 */
#ifndef WA_H_
#define WA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (a CUDA runtime/driver stream handle). NULL is the legacy default stream. */
typedef struct CUstream_st* wa_stream_t;

typedef enum {
  WA_OK = 0,
  WA_ERR_INVALID = 1,         /* bad argument: geometry, pointer, alignment, stride, aliasing */
  WA_ERR_UNSUPPORTED = 2,     /* valid but not built: head dim other than 64/128, sizes past int32 rows or items */
  WA_ERR_OOM = 3,             /* device (or host) allocation of the plan's tables or workspace failed */
  WA_ERR_CUDA = 4,            /* a CUDA call failed (launch error, no device, wrong architecture) */
  WA_ERR_DEVICE_TIMEOUT = 5,  /* a device-side wait ran past its limit; the kernel gave up and returned */
  WA_ERR_DEVICE_BOUNDS = 6    /* a device-side index check failed; the access was skipped */
} wa_status;

/* How the four tensors are laid out. All four (q, k, v, out) share it.
 * A range of heads [h0, h0 + nh) of larger tensors is itself such a layout: H = nh with the larger tensors' strides,
 * and every pointer advanced by h0 * stride_h elements. A head-sharded (Ulysses-style) run uses this, or the
 * contiguous [B, L, H/N, D] head shard it receives from its all-to-all (MiniMax-H3 Ulysses pull request, sglang
 * #43164, Motivation): (b, h) slices are independent, so a head range needs nothing from the other heads. */
typedef struct {
  int32_t global_pos; /* 0 = globals after the frame tokens, 1 = before them */
  int32_t B;          /* batch */
  int32_t H;          /* heads */
  int32_t D;          /* head dim: 64 or 128 */
  int64_t stride_b;   /* element stride between batch entries; multiple of 8 */
  int64_t stride_l;   /* element stride between sequence rows; multiple of 8 */
  int64_t stride_h;   /* element stride between heads; multiple of 8 (contiguous: D) */
} wa_layout_t;

/* Counts describing a plan (host-side facts; filled by wa_plan_info and wa_geometry_describe). */
typedef struct {
  int32_t n_chunks;        /* ceil(T / K) */
  int32_t n_groups;        /* window groups: chunks with identical clamped windows are merged */
  int32_t n_splits;        /* key splits of the global leg (1 when G == 0) */
  int32_t n_items;         /* work items of the attention kernel (window tiles + global split tiles) */
  int64_t L;               /* T*S + G */
  int64_t kept_pairs;      /* kept (query, key) pairs per (b, h) slice */
  int64_t window_pairs;    /* of which: frame-query pairs */
  int64_t global_pairs;    /* of which: global-query pairs (G * L) */
  int64_t workspace_bytes; /* device workspace of the global leg: B*H*G*n_splits*(D+1)*4 */
  int64_t kv_tiles;        /* sum over items of the key tiles each processes */
} wa_plan_info_t;

/* Per-group row of the window plan (wa_geometry_describe): all indices are sequence rows, half-open. */
typedef struct {
  int64_t q_lo, q_hi;   /* query rows of the group */
  int64_t kv0_lo, kv0_hi; /* key segment 0: the window's frame tokens (merged with the globals when adjacent) */
  int64_t kv1_lo, kv1_hi; /* key segment 1: the global tokens, or empty (lo == hi) */
} wa_group_t;

typedef struct wa_plan wa_plan_t;

/*
 * Build (or fetch from the cache) the plan for one geometry on the current CUDA device.
 *   T, S, K >= 1; r >= 0 (r >= number of chunks is valid: dense attention); G >= 0 (0 runs no global leg).
 *   layout: see wa_layout_t; B, H >= 1; D in {64, 128}; T*S + G < 2^31. Work items carry 32-bit indices, so
 *   B*H * (ceil(T*S / 256) + ceil(T / K) + 64 * ceil(G / 256)) must stay below 2^31, and no stride times its
 *   extent may reach 2^60 elements; any geometry whose tensors fit in device memory is far inside both bounds.
 * The plan holds the window groups, the work list of the attention kernel (uploaded to the device once) and
 * the global leg's workspace. The article builds its plan once per geometry and caches it (section 三, the _Plan
 * object with its window groups and gather indices, kept per geometry); here plans live in a process-wide cache
 * of up to 4 geometries keyed on (device, geometry, layout); the least recently used unreferenced entry is
 * evicted. Each successful call returns a
 * reference that the caller must drop with wa_plan_release().
 * Errors: WA_ERR_INVALID (null pointers, bad geometry), WA_ERR_UNSUPPORTED (D, the bounds above), WA_ERR_OOM (a
 * device or host allocation failed; no C++ exception leaves the library), WA_ERR_CUDA.
 */
wa_status wa_plan_create(int T, int S, int K, int r, int G, const wa_layout_t* layout, wa_plan_t** out);

/*
 * out <- window attention of (q, k, v), asynchronously on `stream`.
 *   q, k, v: device pointers to bf16 [B, L, H, D] (layout of the plan); read only.
 *   out: device pointer to bf16 [B, L, H, D]; every element is overwritten; must not overlap q, k or v.
 * Pointers must be 16-byte aligned. Host work is argument checks and building three TMA descriptors; the
 * device work is two launches (the attention kernel over the plan's work list, then the log-sum-exp merge of
 * the global rows). Forwards on one plan are serialised: a call on a different stream than the previous call
 * first waits for that call to finish on the device, since both use the plan's workspace.
 * CUDA graphs: a call on a stream that is being captured records the two launches into the graph (their arguments,
 * including q, k, v and out, are fixed at capture; the plan must outlive the graph). Each launch leaves the plan's
 * work counter as it found it, so the graph can be replayed any number of times. A captured call takes no part in
 * the cross-stream ordering above (it runs whenever the graph is launched): the caller must not let a replay run
 * at the same time as another call on the same plan, captured or not. Make the first call of a process outside a
 * capture (it sets the kernels' shared-memory attribute).
 * Errors (synchronous, nothing launched): WA_ERR_INVALID for null/misaligned/overlapping pointers;
 * WA_ERR_CUDA when a launch fails, or when `stream`'s capture state cannot be read or its capture was invalidated.
 * Device-side failures: see wa_plan_check_error().
 */
wa_status wa_forward(wa_plan_t* plan, const void* q, const void* k, const void* v, void* out, wa_stream_t stream);

/*
 * wa_forward, and also the log-sum-exp of every row's scaled scores over its kept set, as the backward pass needs:
 *   lse[(b*H + h)*L + i] = ln sum_{j kept by i} exp(q_i.k_j / sqrt(D))   (fp32, device, [B][H][L] contiguous,
 *   4-byte aligned; every element is written).
 * Errors: as wa_forward; WA_ERR_INVALID for a NULL or misaligned lse.
 */
wa_status wa_forward_lse(wa_plan_t* plan, const void* q, const void* k, const void* v, void* out, float* lse,
                         wa_stream_t stream);

/*
 * out <- window attention with 8-bit queries and keys (the article's deployment runs the model in FP8,
 * section 四: 6.41 s/NFE FP8 on one GPU; this is the attention-side counterpart).
 *   q8, k8: device pointers to e4m3 (float8 e4m3fn, 1 byte) [B, L, H, D] with the plan's element strides; the
 *           represented values are q = q_scale * q8 and k = k_scale * k8 (per-tensor dequantisation factors).
 *   v, out: bf16 as in wa_forward.
 * Scores are q8.k8 (exact products, fp32 accumulation by kind::f8f6f4 MMAs) times q_scale * k_scale / sqrt(D);
 * the softmax, P (bf16) and O (fp32 accumulation) are as in wa_forward. Uses the same plan as wa_forward.
 * Errors: as wa_forward; WA_ERR_INVALID for scales that are not finite and positive; WA_ERR_UNSUPPORTED unless
 * D == 128 (one e4m3 row is then exactly one 128-byte swizzle row).
 */
wa_status wa_forward_fp8(wa_plan_t* plan, const void* q8, const void* k8, const void* v, void* out, float q_scale,
                         float k_scale, wa_stream_t stream);

/*
 * wa_forward on HOST buffers: q, k, v are read from host memory and out is written to host memory (all bf16 with
 * the plan's layout; page-locked memory lets the copies run asynchronously and overlap the computation). The
 * library keeps device copies of the four tensors in the plan (allocated by the first call: 4 x the layout's span,
 * kept until the plan is freed). When the heads of a sequence row are adjacent in memory (stride_h == D, or H == 1),
 * the sequence is copied in as row pieces, the global rows first and then the frames one window group at a time
 * (the first frame piece holds the rows the first window group reads; it and the globals are split into two head
 * ranges, so that the first launch can start after half of that copy, and the last frame piece into four). After
 * each piece arrives, one launch computes the work items whose rows have all arrived, and the blocks of out that
 * launch completes are copied back while later pieces are still arriving; the global rows of a head range are
 * merged and copied back right after the launch that ran the range's last split items. Launches alternate between `stream` and a library-owned compute stream; copies run on two
 * library-owned copy streams; events chain all of them to `stream`. Other layouts are copied whole and computed in
 * one launch, merged, and copied back whole. The work list is the plan's, except that when the global rows fill at
 * least four query-tile pairs per head the global leg uses key splits half as long (its own workspace, allocated
 * with the device copies; see wa_host_schedule_describe). Frame rows are identical to wa_forward's bit for bit, and
 * so are global rows when the two lists split alike; otherwise global rows differ from wa_forward's only in the
 * order of the split merge (within rounding). The call is asynchronous: out is complete when `stream` reaches this point (e.g. after
 * cudaStreamSynchronize); q, k, v and out must stay valid until then.
 * Errors: WA_ERR_INVALID for null pointers or out overlapping an input; WA_ERR_OOM when the device copies cannot
 * be allocated; WA_ERR_UNSUPPORTED, nothing queued, while `stream` is being captured into a CUDA graph; WA_ERR_CUDA
 * when a copy or launch fails. Device-side failures: see wa_plan_check_error().
 */
wa_status wa_forward_host(wa_plan_t* plan, const void* q, const void* k, const void* v, void* out,
                          wa_stream_t stream);

/*
 * Gradients of a scalar loss through the forward: given dout = d(loss)/d(out), writes
 *   dq = d(loss)/dq, dk = d(loss)/dk, dv = d(loss)/dv
 * for the same kept sets as wa_forward (VDN-Minimax-H3 window-attention article, section 一 for the kept sets and
 * section 三 for the softmax restricted to them; the chain rule through that softmax, per row i with kept set J:
 * dv_j += P_ij dout_i, dS_ij = P_ij (dout_i.v_j - dout_i.out_i), dq_i = sum_j dS_ij k_j / sqrt(D),
 * dk_j += dS_ij q_i / sqrt(D)).
 *   q, k, v, out, dout, dq, dk, dv: device pointers to bf16 [B, L, H, D] with the plan's element strides,
 *     16-byte aligned. out and lse must be what wa_forward_lse wrote for these q, k, v (the probabilities are
 *     recomputed from lse, not stored). Every element of dq, dk, dv is written.
 *   lse: device fp32 [B][H][L] contiguous, 4-byte aligned.
 * Ordering: as wa_forward (calls on one plan are ordered across streams by the library). The first call on a plan
 * allocates its backward workspace: B*H*L*4 (rounded up to 256) + 3*B*H*G*n_splits*D*4 bytes, kept until the plan is freed.
 * CUDA graphs: as wa_forward; a call inside a capture needs the workspace of an earlier call outside one.
 * Errors (synchronous, nothing launched): WA_ERR_INVALID for null or misaligned pointers, or when dq, dk or dv
 * overlaps each other or any input; WA_ERR_OOM when the workspace cannot be allocated; WA_ERR_UNSUPPORTED for a
 * first call made inside a capture; WA_ERR_CUDA when a launch fails. Device-side failures: see wa_plan_check_error(); besides the wait watchdog, the dk/dv kernel at D = 128
 * reports WA_ERR_DEVICE_BOUNDS (and computes nothing) if the device gives it a dynamic shared-memory window more
 * than 768 bytes short of a 1024-byte boundary, since its buffers leave only that much room to realign it (any
 * window on a 256-byte boundary is fine).
 */
wa_status wa_backward(wa_plan_t* plan, const void* q, const void* k, const void* v, const void* out, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, wa_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the plan's device error word.
 * Returns WA_OK, WA_ERR_DEVICE_TIMEOUT, WA_ERR_DEVICE_BOUNDS, or WA_ERR_CUDA if the synchronisation failed;
 * WA_ERR_UNSUPPORTED, touching nothing, while `stream` is being captured into a CUDA graph (call it after the
 * graph's launch instead).
 */
wa_status wa_plan_check_error(wa_plan_t* plan, wa_stream_t stream);

/* Counts of a plan. Errors: WA_ERR_INVALID for null pointers. */
wa_status wa_plan_info(const wa_plan_t* plan, wa_plan_info_t* info);

/* Drop one reference. The plan is freed when unreferenced and evicted (or never cached). NULL is a no-op. */
void wa_plan_release(wa_plan_t* plan);

/*
 * Host-only: the plan a geometry would get, without touching any device. Fills `info`; when `groups` is not
 * NULL writes min(n_groups, groups_cap) group rows; when `items` is not NULL writes min(n_items, items_cap)
 * work items, 8 int64 each: {b*H + h, kind (0 window, 1 global split), q_lo, q_hi, kv0_lo, kv0_hi, kv1_lo,
 * kv1_hi}. Errors: as wa_plan_create for the arguments; WA_ERR_OOM if host memory runs out; never WA_ERR_CUDA.
 */
wa_status wa_geometry_describe(int T, int S, int K, int r, int G, const wa_layout_t* layout, wa_plan_info_t* info,
                               wa_group_t* groups, int64_t groups_cap, int64_t* items, int64_t items_cap);

/*
 * Host-only: the piece schedule wa_forward_host uses for this geometry and layout, without touching any device.
 * The host-buffer forward runs its own work list: wa_geometry_describe's, except that the key splits of the global
 * leg are half as long when the global rows fill at least four query-tile pairs per head (a split runs only once
 * every row of its key range has arrived, so a short last split leaves less work after the last copy); with fewer
 * global rows the two lists are the same. Pieces are blocks of sequence rows x heads (all batch entries) in the
 * order they are copied in; after piece p has arrived, launch p runs the work items whose rows have all arrived;
 * after launch p the blocks of out that it completed are copied back: frame rows, and the global rows of the heads
 * whose last split item it ran (merged right behind it). When the pieces are not row blocks, the whole of out is
 * merged and copied back at the end. Writes min(n_pieces, pieces_cap) blocks {lo, hi, h_lo, h_hi} (rows [lo, hi),
 * heads [h_lo, h_hi)) to `pieces`; for the first min(n_items, items_cap) work items of the host path's list, the
 * item (8 int64 each, as wa_geometry_describe writes them) to `items` and its launch index to `item_launch`; and
 * min(n_out, out_cap) blocks {launch, lo, hi, h_lo, h_hi} to `out_ranges`. Any of the four arrays may be NULL.
 * *n_pieces, *n_items and *n_out receive the full counts; *row_pieces is 1 when pieces are row blocks
 * (stride_h == D or H == 1), else 0 (one piece: the whole tensors).
 * Errors: as wa_plan_create for the arguments, WA_ERR_INVALID for a null count pointer.
 */
wa_status wa_host_schedule_describe(int T, int S, int K, int r, int G, const wa_layout_t* layout, int64_t* pieces,
                                    int64_t pieces_cap, int64_t* items, int32_t* item_launch, int64_t items_cap,
                                    int64_t* out_ranges, int64_t out_cap, int64_t* n_pieces, int64_t* n_items,
                                    int64_t* n_out, int32_t* row_pieces);

/* Static string for a status code ("WA_OK", ...); "WA_UNKNOWN" for other values. */
const char* wa_status_string(wa_status s);

/*
 * The same forward pass as wa_forward, for callers that may not allocate device memory (the article has no
 * counterpart to this entry point). Such callers include frameworks that hand out device memory only from their
 * own accounted pool, processes under a fixed device-memory budget, and code that must avoid the device-wide
 * synchronisation cudaMalloc / cudaFree can cause. It needs no plan: the work list, the global-leg workspace and
 * the device error word live in one library-owned 32 MiB __device__ array that exists on every GPU where the
 * library's device code is loaded, until the process exits. It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *   Arguments: as wa_plan_create (geometry, layout) plus q, k, v, out and stream as wa_forward. The work list is
 *   built on the host per (b, h) slice and passed by value, as kernel parameters, to a small kernel that writes the
 *   whole list into the array on every call (one launch per 800 entries of the per-slice list); no host memory is
 *   read by the device after the call returns.
 *   The first call in a CUDA context (the device's primary context, or a new one after cudaDeviceReset) looks up
 *   the array's device address (cudaGetSymbolAddress) with that context current; make that first call before any
 *   stream capture (inside a capture it returns WA_ERR_UNSUPPORTED). Later calls can be captured into a CUDA graph:
 *   the work list travels in the launches' parameters, so a replay reads nothing from the host.
 *   Every call shares the one array: calls that overlap on the GPU (different streams or threads) race on it;
 *   calls on one stream are ordered. The array keeps the previous call's contents; the call clears what must
 *   start at zero.
 * Errors: as wa_forward; WA_ERR_UNSUPPORTED, before anything is launched, when the geometry's scratch (work list
 * + B*H*G*n_splits*(D+1)*4 bytes of workspace) exceeds the 32 MiB array; WA_ERR_OOM if the host-side work list
 * cannot be built (host memory). Device-side watchdog failures are latched
 * in the array's error word and cleared by the next call; this entry point does not report them.
 */
wa_status wa_forward_static(int T, int S, int K, int r, int G, const wa_layout_t* layout, const void* q,
                            const void* k, const void* v, void* out, wa_stream_t stream);

/* ---- test hooks: not needed in normal use ---------------------------------------------------------------- */

/*
 * Fault injection for the watchdog test. flags & 1: the next forward's producer skips one key-tile copy, so the
 * consumer's bounded wait runs out (about 2 s), the kernel unwinds and latches WA_ERR_DEVICE_TIMEOUT, which
 * wa_plan_check_error() then reports. flags & 2 and flags & 4 do the same to the backward's dq kernel and dk/dv
 * kernel (one query-tile copy is never issued). The device stays usable; later calls with flags == 0 are
 * correct. flags & 8 (only in the index-checking debug build, libwa_debug.so, compiled with -DWA_DEBUG): the first
 * work item of the forward's first CTA is given a key segment past the end of the sequence; the device-side check
 * rejects it before any copy, the CTA unwinds and WA_ERR_DEVICE_BOUNDS is latched. Returns WA_ERR_INVALID for a
 * NULL plan.
 */
int wa_plan_set_debug_flags(wa_plan_t* plan, int flags);

/*
 * Launch timing. enable != 0 starts recording (and clears earlier records): each later wa_forward on the plan
 * records CUDA events on its stream before the attention kernel, between the two kernels and after the merge
 * kernel (up to 4096 forwards). wa_plan_profile_read() waits for the recorded events and returns the summed
 * device time of each kernel in milliseconds and the number of forwards recorded. Returns WA_ERR_INVALID for
 * NULL arguments, WA_ERR_CUDA if an event call fails.
 */
int wa_plan_profile(wa_plan_t* plan, int enable);
int wa_plan_profile_read(wa_plan_t* plan, double* attention_ms, double* combine_ms, int* n_forwards);
/*
 * The same for the backward passes recorded while profiling is enabled (up to 4096): ms[0..3] receive the summed
 * device time of the row dot products, the dq kernel, the dk/dv kernel and the split sums; *n_backwards the count.
 */
int wa_plan_profile_read_backward(wa_plan_t* plan, double* ms, int* n_backwards);

/* Number of plans currently held by the cache (referenced or not). */
int wa_cache_size(void);

/* Reference count of a plan; -1 for NULL. */
int wa_plan_refcount(const wa_plan_t* plan);

#ifdef __cplusplus
}
#endif

#endif /* WA_H_ */
