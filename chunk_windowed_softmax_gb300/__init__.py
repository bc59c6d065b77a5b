"""chunk_windowed_softmax_gb300: chunk-aligned window softmax attention on GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/wa.h`` (``libwa.so``, built in-tree by ``_build.build()``).
Functions keep the C names; this module only marshals arguments: every step of the computation runs in the
library's CUDA kernels. PyTorch supplies device memory and streams. There is no CPU fallback: if the library
is missing or a call fails, an exception is raised.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libwa.so")

WA_OK = 0
STATUS = {0: "WA_OK", 1: "WA_ERR_INVALID", 2: "WA_ERR_UNSUPPORTED", 3: "WA_ERR_OOM", 4: "WA_ERR_CUDA",
          5: "WA_ERR_DEVICE_TIMEOUT", 6: "WA_ERR_DEVICE_BOUNDS"}

# Symbols declared in include/wa.h (the tests check that the library exports each of them).
EXPORTS = ("wa_plan_create", "wa_forward", "wa_plan_check_error", "wa_plan_info", "wa_plan_release",
           "wa_geometry_describe", "wa_status_string", "wa_plan_set_debug_flags", "wa_cache_size", "wa_plan_refcount",
           "wa_plan_profile", "wa_plan_profile_read", "wa_forward_static", "wa_forward_fp8", "wa_forward_lse",
           "wa_backward", "wa_plan_profile_read_backward", "wa_forward_host",
           "wa_host_schedule_describe")


class WAError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


class wa_layout_t(ctypes.Structure):
    _fields_ = [("global_pos", ctypes.c_int32), ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
                ("stride_b", ctypes.c_int64), ("stride_l", ctypes.c_int64), ("stride_h", ctypes.c_int64)]


class wa_plan_info_t(ctypes.Structure):
    _fields_ = [("n_chunks", ctypes.c_int32), ("n_groups", ctypes.c_int32), ("n_splits", ctypes.c_int32),
                ("n_items", ctypes.c_int32), ("L", ctypes.c_int64), ("kept_pairs", ctypes.c_int64),
                ("window_pairs", ctypes.c_int64), ("global_pairs", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("kv_tiles", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class wa_group_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("q_lo", "q_hi", "kv0_lo", "kv0_hi", "kv1_lo", "kv1_hi")]


_lib_handle = None


def lib():
    """Load libwa.so (once). Raises if it has not been built: there is no fallback."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                               f"g.build()'` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        L.wa_plan_create.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(wa_layout_t), ctypes.POINTER(P)]
        L.wa_plan_create.restype = ctypes.c_int
        L.wa_forward.argtypes = [P, P, P, P, P, P]
        L.wa_forward.restype = ctypes.c_int
        L.wa_forward_lse.argtypes = [P, P, P, P, P, P, P]
        L.wa_forward_lse.restype = ctypes.c_int
        L.wa_forward_host.argtypes = [P] * 6
        L.wa_forward_host.restype = ctypes.c_int
        L.wa_backward.argtypes = [P] * 11
        L.wa_backward.restype = ctypes.c_int
        L.wa_plan_profile_read_backward.argtypes = [P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]
        L.wa_plan_profile_read_backward.restype = ctypes.c_int
        L.wa_forward_fp8.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float, P]
        L.wa_forward_fp8.restype = ctypes.c_int
        L.wa_plan_check_error.argtypes = [P, P]
        L.wa_plan_check_error.restype = ctypes.c_int
        L.wa_plan_info.argtypes = [P, ctypes.POINTER(wa_plan_info_t)]
        L.wa_plan_info.restype = ctypes.c_int
        L.wa_plan_release.argtypes = [P]
        L.wa_plan_release.restype = None
        L.wa_geometry_describe.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(wa_layout_t),
                                                                 ctypes.POINTER(wa_plan_info_t),
                                                                 ctypes.POINTER(wa_group_t), ctypes.c_int64,
                                                                 ctypes.POINTER(ctypes.c_int64), ctypes.c_int64]
        L.wa_geometry_describe.restype = ctypes.c_int
        i64p, i32p = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
        L.wa_host_schedule_describe.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(wa_layout_t), i64p,
                                                                      ctypes.c_int64, i64p, i32p, ctypes.c_int64,
                                                                      i64p, ctypes.c_int64, i64p, i64p, i64p, i32p]
        L.wa_host_schedule_describe.restype = ctypes.c_int
        L.wa_status_string.argtypes = [ctypes.c_int]
        L.wa_status_string.restype = ctypes.c_char_p
        L.wa_plan_set_debug_flags.argtypes = [P, ctypes.c_int]
        L.wa_plan_set_debug_flags.restype = ctypes.c_int
        L.wa_plan_profile.argtypes = [P, ctypes.c_int]
        L.wa_plan_profile.restype = ctypes.c_int
        L.wa_plan_profile_read.argtypes = [P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_int)]
        L.wa_plan_profile_read.restype = ctypes.c_int
        L.wa_forward_static.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(wa_layout_t), P, P, P, P, P]
        L.wa_forward_static.restype = ctypes.c_int
        L.wa_cache_size.argtypes = []
        L.wa_cache_size.restype = ctypes.c_int
        L.wa_plan_refcount.argtypes = [P]
        L.wa_plan_refcount.restype = ctypes.c_int
        _lib_handle = L
    return _lib_handle


def _check(st, what):
    if st != WA_OK:
        raise WAError(st, what)


def make_layout(B, L, H, D, global_pos, strides=None):
    """Layout of a [B, L, H, D] tensor; `strides` are element strides (b, l, h), contiguous by default."""
    if strides is None:
        strides = (L * H * D, H * D, D)
    return wa_layout_t(global_pos, B, H, D, *strides)


# ------------------------------------------------------------------------------------- C-named wrappers
def wa_status_string(status):
    return lib().wa_status_string(status).decode()


def wa_plan_create(T, S, K, r, G, layout):
    """Returns a plan handle (ctypes.c_void_p); raises WAError on failure."""
    h = ctypes.c_void_p()
    _check(lib().wa_plan_create(T, S, K, r, G, ctypes.byref(layout), ctypes.byref(h)), "wa_plan_create")
    return h


def wa_forward(plan, q_ptr, k_ptr, v_ptr, out_ptr, stream_ptr):
    _check(lib().wa_forward(plan, ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                            ctypes.c_void_p(out_ptr), ctypes.c_void_p(stream_ptr)), "wa_forward")


def wa_backward(plan, q_ptr, k_ptr, v_ptr, out_ptr, dout_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr, stream_ptr):
    _check(lib().wa_backward(plan, *(ctypes.c_void_p(p) for p in (q_ptr, k_ptr, v_ptr, out_ptr, dout_ptr, lse_ptr,
                                                                  dq_ptr, dk_ptr, dv_ptr, stream_ptr))),
           "wa_backward")


def wa_forward_fp8(plan, q8_ptr, k8_ptr, v_ptr, out_ptr, q_scale, k_scale, stream_ptr):
    _check(lib().wa_forward_fp8(plan, ctypes.c_void_p(q8_ptr), ctypes.c_void_p(k8_ptr), ctypes.c_void_p(v_ptr),
                                ctypes.c_void_p(out_ptr), q_scale, k_scale, ctypes.c_void_p(stream_ptr)),
           "wa_forward_fp8")


def wa_forward_static(T, S, K, r, G, layout, q_ptr, k_ptr, v_ptr, out_ptr, stream_ptr):
    """Forward pass with no device allocation (library-owned static scratch); raises WAError on failure."""
    _check(lib().wa_forward_static(T, S, K, r, G, ctypes.byref(layout), ctypes.c_void_p(q_ptr),
                                   ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr), ctypes.c_void_p(out_ptr),
                                   ctypes.c_void_p(stream_ptr)), "wa_forward_static")


def wa_plan_check_error(plan, stream_ptr):
    return lib().wa_plan_check_error(plan, ctypes.c_void_p(stream_ptr))


def wa_plan_info(plan):
    info = wa_plan_info_t()
    _check(lib().wa_plan_info(plan, ctypes.byref(info)), "wa_plan_info")
    return info.as_dict()


def wa_plan_release(plan):
    lib().wa_plan_release(plan)


def wa_geometry_describe(T, S, K, r, G, layout, with_groups=True, with_items=False):
    """Host-only plan description: (info dict, list of group dicts, list of item tuples)."""
    L = lib()
    info = wa_plan_info_t()
    _check(L.wa_geometry_describe(T, S, K, r, G, ctypes.byref(layout), ctypes.byref(info), None, 0, None, 0),
           "wa_geometry_describe")
    groups, items = [], []
    gbuf = (wa_group_t * max(1, info.n_groups))() if with_groups else None
    ibuf = (ctypes.c_int64 * (8 * max(1, info.n_items)))() if with_items else None
    _check(L.wa_geometry_describe(T, S, K, r, G, ctypes.byref(layout), ctypes.byref(info), gbuf, info.n_groups,
                                  ibuf, info.n_items), "wa_geometry_describe")
    if with_groups:
        groups = [{n: getattr(g, n) for n, _ in wa_group_t._fields_} for g in gbuf[:info.n_groups]]
    if with_items:
        items = [tuple(ibuf[8 * i:8 * i + 8]) for i in range(info.n_items)]
    return info.as_dict(), groups, items


def wa_host_schedule_describe(T, S, K, r, G, layout):
    """Host-only piece schedule of the host-buffer forward: {"row_pieces": bool, "pieces": [(lo, hi, h_lo, h_hi)] in
    copy order, "items": [the host path's work items, as wa_geometry_describe's], "item_launch": [launch per item],
    "out": [(launch, lo, hi, h_lo, h_hi)]}."""
    L = lib()
    n_pieces, n_items, n_out, rows = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    args = (T, S, K, r, G, ctypes.byref(layout))
    counts = (ctypes.byref(n_pieces), ctypes.byref(n_items), ctypes.byref(n_out), ctypes.byref(rows))
    _check(L.wa_host_schedule_describe(*args, None, 0, None, None, 0, None, 0, *counts), "wa_host_schedule_describe")
    pbuf = (ctypes.c_int64 * (4 * max(1, n_pieces.value)))()
    ibuf = (ctypes.c_int64 * (8 * max(1, n_items.value)))()
    lbuf = (ctypes.c_int32 * max(1, n_items.value))()
    obuf = (ctypes.c_int64 * (5 * max(1, n_out.value)))()
    _check(L.wa_host_schedule_describe(*args, pbuf, n_pieces.value, ibuf, lbuf, n_items.value, obuf, n_out.value,
                                       *counts), "wa_host_schedule_describe")
    return {"row_pieces": bool(rows.value),
            "pieces": [tuple(pbuf[4 * i:4 * i + 4]) for i in range(n_pieces.value)],
            "items": [tuple(ibuf[8 * i:8 * i + 8]) for i in range(n_items.value)],
            "item_launch": list(lbuf[:n_items.value]),
            "out": [tuple(obuf[5 * i:5 * i + 5]) for i in range(n_out.value)]}


# ----------------------------------------------------------------------------------------- torch side
class Plan:
    """A referenced plan for one geometry and layout on the current CUDA device."""

    def __init__(self, T, S, K, r, G, B, H, D, global_pos=0, strides=None):
        self.geometry = (T, S, K, r, G)
        self.L = T * S + G
        self.layout = make_layout(B, self.L, H, D, global_pos, strides)
        self.handle = wa_plan_create(T, S, K, r, G, self.layout)

    def info(self):
        return wa_plan_info(self.handle)

    def forward(self, q, k, v, out=None, stream=None):
        """out <- window attention of bf16 CUDA tensors q, k, v (shape [B, L, H, D], this plan's layout)."""
        import torch
        lay = self.layout
        shape = (lay.B, self.L, lay.H, lay.D)
        for name, t in (("q", q), ("k", k), ("v", v)):
            if t.dtype != torch.bfloat16 or not t.is_cuda or tuple(t.shape) != shape:
                raise ValueError(f"{name} must be a bf16 CUDA tensor of shape {shape}")
            if tuple(t.stride()) != (lay.stride_b, lay.stride_l, lay.stride_h, 1):
                raise ValueError(f"{name} strides {t.stride()} differ from the plan's layout")
        if out is None:
            out = torch.empty_strided(shape, (lay.stride_b, lay.stride_l, lay.stride_h, 1), dtype=torch.bfloat16,
                                      device=q.device)
        s = torch.cuda.current_stream(q.device) if stream is None else stream
        wa_forward(self.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), s.cuda_stream)
        return out

    def forward_host(self, q, k, v, out=None, stream=None):
        """out <- window attention of HOST (CPU) bf16 tensors with the plan's layout; the copies to and from the
        device are pipelined with the computation over pieces of the sequence (pinned tensors let them overlap).
        Returns the host tensor `out` once it is complete."""
        import torch
        lay = self.layout
        shape = (lay.B, self.L, lay.H, lay.D)
        strides = (lay.stride_b, lay.stride_l, lay.stride_h, 1)
        for name, t in (("q", q), ("k", k), ("v", v)):
            if t.dtype != torch.bfloat16 or t.is_cuda or tuple(t.shape) != shape or tuple(t.stride()) != strides:
                raise ValueError(f"{name} must be a bf16 CPU tensor of shape {shape} with the plan's strides")
        if out is None:
            out = torch.empty_strided(shape, strides, dtype=torch.bfloat16, pin_memory=q.is_pinned())
        s = torch.cuda.current_stream() if stream is None else stream
        _check(lib().wa_forward_host(self.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                     ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(s.cuda_stream)), "wa_forward_host")
        s.synchronize()
        return out

    def forward_lse(self, q, k, v, out=None, lse=None, stream=None):
        """(out, lse): the forward and each row's natural-log log-sum-exp (fp32 [B, H, L]) for the backward."""
        import torch
        lay = self.layout
        if lse is None:
            lse = torch.empty(lay.B, lay.H, self.L, dtype=torch.float32, device=q.device)
        shape = (lay.B, self.L, lay.H, lay.D)
        strides = (lay.stride_b, lay.stride_l, lay.stride_h, 1)
        for name, t in (("q", q), ("k", k), ("v", v)):
            if t.dtype != torch.bfloat16 or not t.is_cuda or tuple(t.shape) != shape or tuple(t.stride()) != strides:
                raise ValueError(f"{name} must be a bf16 CUDA tensor of shape {shape} with the plan's strides")
        if out is None:
            out = torch.empty_strided(shape, strides, dtype=torch.bfloat16, device=q.device)
        s = torch.cuda.current_stream(q.device) if stream is None else stream
        _check(lib().wa_forward_lse(self.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                    ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(s.cuda_stream)), "wa_forward_lse")
        return out, lse

    def backward(self, q, k, v, out, dout, lse, dq=None, dk=None, dv=None, stream=None):
        """(dq, dk, dv): gradients through the forward, given dout and the forward's out and lse (forward_lse)."""
        import torch
        lay = self.layout
        shape = (lay.B, self.L, lay.H, lay.D)
        strides = (lay.stride_b, lay.stride_l, lay.stride_h, 1)
        for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
            if t.dtype != torch.bfloat16 or not t.is_cuda or tuple(t.shape) != shape or tuple(t.stride()) != strides:
                raise ValueError(f"{name} must be a bf16 CUDA tensor of shape {shape} with the plan's strides")
        if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (lay.B, lay.H, self.L) \
                or not lse.is_contiguous():
            raise ValueError(f"lse must be a contiguous fp32 CUDA tensor of shape {(lay.B, lay.H, self.L)}")
        grads = [g if g is not None else torch.empty_strided(shape, strides, dtype=torch.bfloat16, device=q.device)
                 for g in (dq, dk, dv)]
        s = torch.cuda.current_stream(q.device) if stream is None else stream
        wa_backward(self.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(),
                    lse.data_ptr(), *(g.data_ptr() for g in grads), s.cuda_stream)
        return tuple(grads)

    def profile_read_backward(self):
        """([row dots, dq kernel, dk/dv kernel, split sums] ms, backwards) summed over the recorded backwards."""
        ms, n = (ctypes.c_double * 4)(), ctypes.c_int()
        _check(lib().wa_plan_profile_read_backward(self.handle, ms, ctypes.byref(n)), "wa_plan_profile_read_backward")
        return list(ms), n.value

    def forward_fp8(self, q8, k8, v, q_scale, k_scale, out=None, stream=None):
        """out <- window attention with e4m3 queries / keys (values q_scale * q8, k_scale * k8) and bf16 v."""
        import torch
        lay = self.layout
        shape = (lay.B, self.L, lay.H, lay.D)
        strides = (lay.stride_b, lay.stride_l, lay.stride_h, 1)
        for name, t, dt in (("q8", q8, torch.float8_e4m3fn), ("k8", k8, torch.float8_e4m3fn), ("v", v, torch.bfloat16)):
            if t.dtype != dt or not t.is_cuda or tuple(t.shape) != shape or tuple(t.stride()) != strides:
                raise ValueError(f"{name} must be a {dt} CUDA tensor of shape {shape} with the plan's strides")
        if out is None:
            out = torch.empty_strided(shape, strides, dtype=torch.bfloat16, device=v.device)
        s = torch.cuda.current_stream(v.device) if stream is None else stream
        wa_forward_fp8(self.handle, q8.data_ptr(), k8.data_ptr(), v.data_ptr(), out.data_ptr(), float(q_scale),
                       float(k_scale), s.cuda_stream)
        return out

    def check_error(self, stream=None):
        import torch
        s = torch.cuda.current_stream() if stream is None else stream
        return wa_plan_check_error(self.handle, s.cuda_stream)

    def profile(self, enable=True):
        """Start (or stop) recording per-kernel device times of this plan's forwards."""
        _check(lib().wa_plan_profile(self.handle, 1 if enable else 0), "wa_plan_profile")

    def profile_read(self):
        """(attention kernel ms, merge kernel ms, forwards) summed over the recorded forwards."""
        a, c, n = ctypes.c_double(), ctypes.c_double(), ctypes.c_int()
        _check(lib().wa_plan_profile_read(self.handle, ctypes.byref(a), ctypes.byref(c), ctypes.byref(n)),
               "wa_plan_profile_read")
        return a.value, c.value, n.value

    def set_debug_flags(self, flags):
        _check(lib().wa_plan_set_debug_flags(self.handle, flags), "wa_plan_set_debug_flags")

    def close(self):
        if getattr(self, "handle", None) is not None:
            wa_plan_release(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def forward(q, k, v, T, S, K, r, G, global_pos=0, out=None):
    """One-shot call: out = window attention of q, k, v ([B, L, H, D] bf16 on a CUDA device).

    CPU tensors are accepted too (end-to-end use): wa_forward_host copies them to the current CUDA device in pieces
    of sequence rows (the global rows first, then the frames one window group at a time), runs the work items whose
    rows have arrived while later pieces are still being copied (pinned tensors let the copies run asynchronously),
    and copies each finished block of the result back into a CPU tensor.
    """
    B, L, H, D = q.shape
    plan = Plan(T, S, K, r, G, B, H, D, global_pos, strides=tuple(q.stride()[:3]))
    try:
        if not q.is_cuda:
            return plan.forward_host(q, k, v, out=out)
        return plan.forward(q, k, v, out=out)
    finally:
        plan.close()


_autograd_fn = None


def _window_softmax_fn():
    """The torch.autograd.Function behind window_softmax_decomposed (defined on first use: torch is imported lazily
    by this module)."""
    global _autograd_fn
    if _autograd_fn is None:
        import torch

        class WindowSoftmaxDecomposed(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, plan):
                out, lse = plan.forward_lse(q, k, v)
                ctx.plan = plan
                ctx.save_for_backward(q, k, v, out, lse)
                return out

            @staticmethod
            def backward(ctx, dout):
                q, k, v, out, lse = ctx.saved_tensors
                lay = ctx.plan.layout
                strides = (lay.stride_b, lay.stride_l, lay.stride_h, 1)
                if dout.dtype != torch.bfloat16 or tuple(dout.stride()) != strides:
                    # the incoming gradient in the plan's layout (e.g. an expanded gradient of a sum has stride 0)
                    dout = torch.empty_strided(dout.shape, strides, dtype=torch.bfloat16,
                                               device=dout.device).copy_(dout)
                dq, dk, dv = ctx.plan.backward(q, k, v, out, dout, lse)
                need = ctx.needs_input_grad
                return (dq if need[0] else None, dk if need[1] else None, dv if need[2] else None, None)

        _autograd_fn = WindowSoftmaxDecomposed
    return _autograd_fn


def window_softmax_decomposed(q, k, v, T, S, K, r, G, global_pos=0):
    """Differentiable window attention of bf16 CUDA tensors q, k, v ([B, L, H, D], any stride order with D
    contiguous): the forward keeps each row's log-sum-exp, and autograd's backward runs this library's gradient
    kernels (dq, dk, dv) from it. This is the decomposed path of the VDN-Minimax-H3 window-attention article
    (section 三, window_softmax_decomposed) made usable for training, which the article otherwise leaves to its
    differentiable mask-based path (section 五). Every output row depends only on its kept set (section 一)."""
    B, L, H, D = q.shape
    if L != T * S + G:
        raise ValueError(f"q has {L} rows; the geometry needs T*S + G = {T * S + G}")
    plan = Plan(T, S, K, r, G, B, H, D, global_pos, strides=tuple(q.stride()[:3]))
    return _window_softmax_fn().apply(q, k, v, plan)
