#!/usr/bin/env python3
"""Throughput of chunk-aligned window softmax attention on GB300: kept-pair TFLOP/s and ms per layer call.

One step = one ``wa_forward`` call (the persistent attention kernel over every window and global-split tile, then
the log-sum-exp merge of the global rows) on the H3-scale layer: B=1, H=56, D=128, T=102 latent frames of S=960
tokens, chunks of K=3 frames, radius r=1, G=2048 global tokens after the frames (L=99,968), keys of the global
rows scaled x2. Useful work counts only kept (query, key) pairs: 4*D flops per pair.

  python bench.py [--gpus N --steps K --warmup W] [--workload h3|medium|ragged|tiny|sweep_T..] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica of the layer on its own GPU (no data exchange; the path is
replicated, not sharded) and rank 0 prints one JSON line with the whole-job throughput over the slowest rank.
``--shard heads`` instead shards one layer by heads across the ranks (all-to-all exchanges in and out, strong
scaling).
``--impl reference`` times the CPU oracle on the host cores instead (rank 0 only), on a bounded row sample.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "kept-pair TFLOP/s and ms/call (1×GB300), % of dense BF16 tensor peak"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "window_attention_kernel_h3.md")
BWD_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "backward_kernels_h3.md")
FP8_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "window_attention_kernel_e4m3_h3.md")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="h3")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--fp8", action="store_true",
                    help="time wa_forward_fp8 (e4m3 queries / keys, per-tensor scales; bf16 values and output)")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (dq, dk, dv through wa_backward) instead of the forward")
    ap.add_argument("--sweep", action="store_true",
                    help="auxiliary: one JSON line per sweep point (kept TFLOP/s vs window density), 1 GPU")
    ap.add_argument("--shard", default="replicas", choices=["replicas", "heads"],
                    help="under torchrun: independent replicas (default), or one layer sharded by heads across the "
                         "ranks (Ulysses-style all-to-all of q, k, v in and of out back; strong scaling)")
    return ap.parse_args()


def workload(name):
    from chunk_windowed_softmax_gb300 import configs
    if name in configs.ALL:
        return configs.ALL[name]
    for w in configs.sweep():
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}")


def workload_config(w, extra=None):
    cfg = {"workload": f"{w.name}: B={w.B} H={w.H} D={w.D} T={w.T} S={w.S} K={w.K} r={w.r} G={w.G} "
                       f"globals={'front' if w.global_pos else 'back'} L={w.L}",
           "B": w.B, "H": w.H, "D": w.D, "T": w.T, "S": w.S, "K": w.K, "r": w.r, "G": w.G, "L": w.L,
           "global_pos": "front" if w.global_pos else "back", "k_global_scale": w.k_global_scale,
           "parallelism": "replicas"}
    if extra:
        cfg.update(extra)
    return cfg


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p["bf16_tflops"], p.get("bf16_tflops_sustained"), p["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def profile_fields(path):
    """The `- key: value` lines of an ncu summary under profiles/ as a dict (values without backquotes)."""
    fields = {}
    for line in open(path):
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].rsplit(":", 1)  # the last colon: keys may contain one ("sha256[:16]")
            fields[k.strip()] = v.strip().strip("`")
    return fields


def stored_traffic(summary=None, source="wa_kernels.cu", key="dram bytes per full H3 launch"):
    """DRAM bytes per launch of a kernel from a committed ncu summary, if the kernel source it was taken on is the
    current one (else None)."""
    import hashlib
    try:
        src = open(os.path.join(ROOT, "chunk_windowed_softmax_gb300", "csrc", source), "rb").read()
        digest = hashlib.sha256(src).hexdigest()[:16]
        fields = profile_fields(summary or PROFILE_SUMMARY)
        if fields.get("kernel source sha256[:16]") != digest:
            return None
        return float(fields[key])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self, t0, t1):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = []
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:8]))
            except Exception:
                continue
        os.unlink(self.f.name)
        sel = [r for r in rows if t0 - 1 <= r[0] <= t1 + 1] or rows
        if not sel:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in sel for n, a in zip(names, r[3]) if a.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel)}


def oracle_sample(w, q, k, v, heads, chunks, global_rows):
    """Run the CPU oracle on a row sample; returns (seconds, kept-pair flops of the sample, rows)."""
    import oracle.ref as ref
    flops = 0.0
    t0 = time.perf_counter()
    nrows = 0
    for h in heads:
        frames = [t for c in chunks for t in ref.chunk_frames(c, w.T, w.K)]
        res = ref.window_attention_rows(q, k, v, w.T, w.S, w.K, w.r, w.G, w.global_pos, 0, h, frames=frames,
                                        global_rows=False)
        nrows += len(res)
        for t in frames:
            flops += 4.0 * w.D * w.S * len(ref.kept_set_of_frame(t, w.T, w.S, w.K, w.r, w.G, w.global_pos))
        if global_rows and w.G:
            sub = ref.window_attention_rows(q, k, v, w.T, w.S, w.K, w.r, w.G, w.global_pos, 0, h, frames=[],
                                            global_rows=True)
            nrows += len(sub)
            flops += 4.0 * w.D * w.G * w.L
    return time.perf_counter() - t0, flops, nrows


def host_inputs(w):
    """q, k, v on the host (drawn on the GPU when there is one: the same generator the GPU arm uses)."""
    import torch
    from chunk_windowed_softmax_gb300 import inputs
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    return tuple(t.cpu() for t in inputs.make_qkv(w, device=dev))


def cores_used():
    n = len(os.sched_getaffinity(0))
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            n = min(n, int(os.environ[var]))
    return n


def blas_threads():
    """The BLAS library numpy's matrix products run on and its live thread count (threadpoolctl when installed,
    else the getter that numpy's bundled OpenBLAS exports); None when neither can be read."""
    try:
        from threadpoolctl import threadpool_info
        for i in threadpool_info():
            if i.get("user_api") == "blas":
                return {"library": i.get("internal_api"), "threads": i.get("num_threads")}
    except Exception:
        pass
    import ctypes
    import glob
    import numpy
    d = os.path.dirname(numpy.__file__)
    for lib in sorted(glob.glob(os.path.join(d, "..", "numpy.libs", "*openblas*")) +
                      glob.glob(os.path.join(d, ".libs", "*openblas*"))):
        try:
            handle = ctypes.CDLL(lib)
        except OSError:
            continue
        for fn in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_", "openblas_get_num_threads"):
            if hasattr(handle, fn):
                return {"library": os.path.basename(lib), "threads": int(getattr(handle, fn)())}
    return None


def run_reference(args, w, rank):
    """The CPU oracle, as it stands, on the host cores: each step a bounded row sample of the workload."""
    if rank != 0:
        return
    import oracle.ref as ref
    q, k, v = host_inputs(w)
    nc = ref.num_chunks(w.T, w.K)

    def step(i):
        h = i % w.H
        c = (i * 7) % nc
        return oracle_sample(w, q, k, v, heads=[h], chunks=[c], global_rows=False)

    for i in range(args.warmup):
        step(i)
    tot_s, tot_f = 0.0, 0.0
    for i in range(args.steps):
        s, f, _ = step(args.warmup + i)
        tot_s += s
        tot_f += f
    value = tot_f / tot_s / 1e12
    sample = (f"per step: every row of one chunk ({w.K * w.S} rows) of one head, cycling heads and chunks; "
              f"{args.steps} steps")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, {"timed": "CPU oracle (numpy float64) on a row sample per step"}),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                         "sample": sample, "blas": blas_threads()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def max_over_ranks(x, device, world):
    """The slowest rank's value (the job finishes when the last replica does)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, flops_per_replica, seconds):
    """Whole-job TFLOP/s: every replica does the same kept-pair work; the job takes the slowest rank's time."""
    return world * flops_per_replica / seconds / 1e12


L2_BYTES = 129e6  # GB300 L2


def timed_steps(fn, steps, stream, device, resident_bytes):
    """Average milliseconds of `fn` over `steps` calls, timed with CUDA events on `stream`. When the tensors a step
    reads and writes are larger than four times L2 they cannot stay cached between steps and the steps are timed
    back to back; otherwise L2 is flushed before each step (a write of twice its size, outside the timed region) and
    each step is timed on its own. Returns (ms, note for the JSON line)."""
    import torch
    if resident_bytes > 4 * L2_BYTES:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / steps, (f"no flush: the tensors of a step ({resident_bytes / 1e9:.2f} GB) are "
                                             f"far larger than the 129 MB L2")
    flush = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=device)
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in events:
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize(device)
    return sum(a.elapsed_time(b) for a, b in events) / steps, (
        f"flushed: a {2 * L2_BYTES / 1e6:.0f} MB buffer is written before each step (the tensors of a step, "
        f"{resident_bytes / 1e9:.3f} GB, could stay in the 129 MB L2); each step timed on its own")


def run_sweep(args):
    """Kept-pair throughput across the H3-shaped sweep (T in {34, 102}, K in {1, 3, 6}, r in {0, 1, 2})."""
    import torch
    import chunk_windowed_softmax_gb300 as wa
    from chunk_windowed_softmax_gb300 import _build, configs, inputs
    _build.build()
    bf16_peak = peaks()[0]
    for w in configs.sweep():
        q, k, v = inputs.make_qkv(w, device="cuda")
        plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
        info = plan.info()
        out = torch.empty_like(q)
        for _ in range(max(3, args.warmup)):
            plan.forward(q, k, v, out=out)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(3, min(args.steps, 10))
        e0.record()
        for _ in range(n):
            plan.forward(q, k, v, out=out)
        e1.record()
        torch.cuda.synchronize()
        st = plan.check_error()
        plan.close()
        ms = e0.elapsed_time(e1) / n
        flops = 4.0 * w.D * info["kept_pairs"] * w.B * w.H
        print(json.dumps({"workload": w.name, "T": w.T, "K": w.K, "r": w.r, "density": info["kept_pairs"] / w.L ** 2,
                          "kept_tflop": flops / 1e12, "ms_per_call": ms, "tflops": flops / ms / 1e9,
                          "pct_of_bf16_peak": 100 * flops / ms / 1e9 / bf16_peak, "status": wa.wa_status_string(st)}),
              flush=True)
        del q, k, v, out


def run_backward(args, w):
    """Backward throughput on one GPU: each step is one wa_backward (row dots, dq kernel, dk/dv kernel, split sums)
    on device-resident q, k, v, out, dout and lse from one forward. Useful work is counted as the five products of
    the chain rule per kept pair (S, dP, dv, dk, dq: 10 D flops); the kernels recompute S and dP once more."""
    import torch
    import chunk_windowed_softmax_gb300 as wa
    from chunk_windowed_softmax_gb300 import _build, inputs
    _build.build()
    q, k, v = inputs.make_qkv(w, device="cuda")
    dout = inputs.make_dout(w, device="cuda")
    plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
    info = plan.info()
    pairs = info["kept_pairs"] * w.B * w.H
    out, lse = plan.forward_lse(q, k, v)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    for _ in range(max(3, args.warmup)):
        plan.backward(q, k, v, out, dout, lse, dq, dk, dv)
    st = plan.check_error()
    if st != 0:
        raise SystemExit(f"device error during warm-up: {wa.wa_status_string(st)}")
    sampler = ClockSampler(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0])
    time.sleep(0.3)
    plan.profile(True)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0 = time.time()
    step_bytes = 8 * q.numel() * 2 + lse.numel() * 4  # q, k, v, out, dout read; dq, dk, dv written; lse
    ms, l2_note = timed_steps(lambda: plan.backward(q, k, v, out, dout, lse, dq, dk, dv), args.steps, stream,
                              q.device, step_bytes)
    t1 = time.time()
    kms, n = plan.profile_read_backward()
    plan.profile(False)
    clocks = sampler.stop(t0, t1)
    st = plan.check_error()
    plan.close()
    if st != 0:
        raise SystemExit(f"device error during the timed steps: {wa.wa_status_string(st)}")
    kms = [x / max(1, n) for x in kms]
    bf16_peak = peaks()[0]
    useful = 10.0 * w.D * pairs
    dq_tf = 6.0 * w.D * pairs / (kms[1] * 1e-3) / 1e12    # S, dP, dq products
    dkdv_tf = 8.0 * w.D * pairs / (kms[2] * 1e-3) / 1e12  # S^T, dP^T, dv, dk products
    print(json.dumps({
        "metric": "backward kept-pair TFLOP/s (10 D flops per kept pair)", "value": useful / ms / 1e9,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, {"kept_pairs_per_head": info["kept_pairs"], "l2": l2_note}),
        "kernels_ms": {"row_dots": kms[0], "dq": kms[1], "dk_dv": kms[2], "split_sums": kms[3]},
        "kernel_tflops": {"dq": dq_tf, "dk_dv": dkdv_tf},
        "kernel_frac_of_bf16_peak": {"dq": dq_tf / bf16_peak, "dk_dv": dkdv_tf / bf16_peak},
        "roofline": {"bound": "tensor", "achieved": dkdv_tf, "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": dkdv_tf / bf16_peak, "frac_of_sustained": dkdv_tf / peaks()[1] if peaks()[1] else None,
                     "kernel": f"wa_dkdv_kernel<{w.D}>", "kernel_ms": kms[2],
                     "traffic": stored_traffic(BWD_PROFILE_SUMMARY, "wa_backward.cu", "dk/dv dram bytes per full H3 launch")
                     if w.name == "h3" else None},
        "gpu_launches": (3 + (1 if w.G > 0 else 0)) * args.steps, "clocks": clocks}), flush=True)


def secondary_paths(w, q, k, v, plan, bf16_peak, steps=10):
    """Short measurements of the e4m3 forward, of the backward and of the forward replayed from a CUDA graph, on the
    bench's workload, taken after the timed forward region (so they change neither its value nor its clock record)
    and reported beside the main line. Each is a few warm-up calls and `steps` timed calls with CUDA events on the
    current stream; a failure is reported as an error string instead of a number."""
    import torch
    out = {}
    stream = torch.cuda.current_stream()
    info = plan.info()
    pairs = info["kept_pairs"] * w.B * w.H
    flops = 4.0 * w.D * pairs
    try:
        sq = float(q.float().abs().max()) / 448.0
        sk = float(k.float().abs().max()) / 448.0
        q8 = (q.float() / sq).to(torch.float8_e4m3fn)
        k8 = (k.float() / sk).to(torch.float8_e4m3fn)
        o8 = torch.empty_like(v)
        for _ in range(3):
            plan.forward_fp8(q8, k8, v, sq, sk, out=o8)
        plan.profile(True)
        ms, _ = timed_steps(lambda: plan.forward_fp8(q8, k8, v, sq, sk, out=o8), steps, stream, q.device,
                            q8.numel() * 2 + v.numel() * 4)
        attn, _, n = plan.profile_read()
        plan.profile(False)
        st = plan.check_error()
        kms = attn / max(1, n)
        mixed = bf16_peak * 4.0 / 3.0
        out["e4m3_forward"] = {"ms_per_step": ms, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                               "kernel_ms": kms, "frac": flops / (kms * 1e-3) / 1e12 / mixed, "peak": mixed,
                               "steps": steps, "status": st}
        del q8, k8, o8
    except Exception as e:  # noqa: BLE001 -- reported in the line, never fatal for the main measurement
        out["e4m3_forward"] = {"error": str(e)[:200]}
    try:
        from chunk_windowed_softmax_gb300 import inputs
        dout = inputs.make_dout(w, device=q.device)
        o, lse = plan.forward_lse(q, k, v)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        for _ in range(2):
            plan.backward(q, k, v, o, dout, lse, dq, dk, dv)
        plan.profile(True)
        ms, _ = timed_steps(lambda: plan.backward(q, k, v, o, dout, lse, dq, dk, dv), max(3, steps // 2), stream,
                            q.device, 8 * q.numel() * 2)
        kms, n = plan.profile_read_backward()
        plan.profile(False)
        st = plan.check_error()
        kms = [x / max(1, n) for x in kms]
        dkdv = 8.0 * w.D * pairs / (kms[2] * 1e-3) / 1e12
        dqk = 6.0 * w.D * pairs / (kms[1] * 1e-3) / 1e12
        out["backward"] = {"ms_per_step": ms, "value": 10.0 * w.D * pairs / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                           "kernels_ms": {"row_dots": kms[0], "dq": kms[1], "dk_dv": kms[2], "split_sums": kms[3]},
                           "frac": {"dq": dqk / bf16_peak, "dk_dv": dkdv / bf16_peak}, "peak": bf16_peak,
                           "steps": max(3, steps // 2), "status": st}
        del dout, o, lse, dq, dk, dv
    except Exception as e:  # noqa: BLE001
        out["backward"] = {"error": str(e)[:200]}
    try:
        # The forward captured once into a CUDA graph and replayed: the same two launches without the per-call host
        # work (argument checks, three TMA descriptors, two launches through the runtime), which matters only
        # where a call is as short as that host work.
        og = torch.empty_like(q)
        plan.forward(q, k, v, out=og)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            plan.forward(q, k, v, out=og)
        for _ in range(3):
            graph.replay()
        ms, _ = timed_steps(graph.replay, steps, stream, q.device, 4 * q.numel() * 2)
        st = plan.check_error()
        eager = plan.forward(q, k, v)
        torch.cuda.synchronize()
        out["graph_forward"] = {"ms_per_step": ms, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                                "launches_per_replay": 1 + (1 if w.G > 0 else 0), "steps": steps,
                                "identical_to_eager": bool(torch.equal(og, eager)), "status": st}
        del graph, og, eager
    except Exception as e:  # noqa: BLE001
        out["graph_forward"] = {"error": str(e)[:200]}
    torch.cuda.empty_cache()
    return out


def run_head_sharded(args, w, rank, world, local):
    """One layer sharded by heads across the ranks: each rank starts from its shard of the packed sequence (all
    heads), q, k and v go to head shards by all-to-all, each rank computes its H/N heads over the whole sequence with
    the library, and the output goes back by all-to-all. Every step includes the four exchanges. Total work is the
    layer's, whatever N (strong scaling)."""
    import torch
    import torch.distributed as dist
    import chunk_windowed_softmax_gb300 as wa
    from chunk_windowed_softmax_gb300 import _build, inputs, sharded
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    if w.H % world:
        raise SystemExit(f"{w.H} heads do not split over {world} ranks")
    sizes = sharded.even_seq_sizes(w.L, world)
    off = sum(sizes[:rank])
    q, k, v = inputs.make_qkv(w, device=dev)  # the same seed on every rank: the shards of one layer
    qs, ks, vs = (t[:, off:off + sizes[rank]].contiguous() for t in (q, k, v))
    del q, k, v
    hn = w.H // world
    plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, hn, w.D, w.global_pos)
    info = plan.info()
    flops = 4.0 * w.D * info["kept_pairs"] * w.B * w.H  # the whole layer
    oh = torch.empty(w.B, w.L, hn, w.D, dtype=torch.bfloat16, device=dev)

    def step():
        return sharded.sharded_forward(qs, ks, vs, w.T, w.S, w.K, w.r, w.G, w.global_pos, seq_sizes=sizes,
                                       attend=lambda qh, kh, vh: plan.forward(qh, kh, vh, out=oh))
    for _ in range(max(3, args.warmup)):
        step()
    st = plan.check_error()
    if st != 0:
        raise SystemExit(f"device error during warm-up: {wa.wa_status_string(st)}")
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev, world)
    st = plan.check_error()
    plan.close()
    if st != 0:
        raise SystemExit(f"device error during the timed steps: {wa.wa_status_string(st)}")
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, {"parallelism": f"heads/{world}: all-to-all of q, k, v to head shards "
                                                         f"and of out back, every step",
                                          "seq_shard_rows": sizes, "heads_per_rank": hn,
                                          "l2": "no flush: the tensors of a step are far larger than the 129 MB L2"
                                          if w.name == "h3" else "not flushed"}),
            "gpu_launches": (2 if w.G > 0 else 1) * args.steps}), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.sweep:
        run_sweep(args)
        return
    if args.backward:
        run_backward(args, workload(args.workload))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = workload(args.workload)
    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if args.shard == "heads":
        run_head_sharded(args, w, rank, world, local)
        return

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import chunk_windowed_softmax_gb300 as wa
    from chunk_windowed_softmax_gb300 import _build, inputs
    _build.build()
    dev = torch.device("cuda", local)

    def barrier():
        if world > 1:
            dist.barrier()

    q, k, v = inputs.make_qkv(w, device=dev)
    if args.fp8:
        sq = float(q.float().abs().max()) / 448.0
        sk = float(k.float().abs().max()) / 448.0
        q8 = (q.float() / sq).to(torch.float8_e4m3fn)
        k8 = (k.float() / sk).to(torch.float8_e4m3fn)
    plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)

    def forward(out):
        if args.fp8:
            return plan.forward_fp8(q8, k8, v, sq, sk, out=out)
        return plan.forward(q, k, v, out=out)
    info = plan.info()
    flops = 4.0 * w.D * info["kept_pairs"] * w.B * w.H
    launches_per_step = 1 + (1 if w.G > 0 else 0)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        forward(out)
    st = plan.check_error()
    if st != 0:
        raise SystemExit(f"device error during warm-up: {wa.wa_status_string(st)}")

    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        gpu_index = vis.split(",")[local]
    sampler = ClockSampler(gpu_index)
    time.sleep(0.3)
    plan.profile(True)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    step_bytes = (q.numel() * (1 if args.fp8 else 2) * 2 + v.numel() * 2 + out.numel() * 2)
    ms, l2_note = timed_steps(lambda: forward(out), args.steps, stream, dev, step_bytes)
    barrier()
    t1 = time.time()
    attn_ms, comb_ms, nrec = plan.profile_read()
    plan.profile(False)
    clocks = sampler.stop(t0, t1)
    st = plan.check_error()
    if st != 0:
        raise SystemExit(f"device error during the timed steps: {wa.wa_status_string(st)}")
    ms_max = max_over_ranks(ms, dev, world)
    value = job_throughput(world, flops, ms_max * 1e-3)
    attn_avg = attn_ms / max(1, nrec)
    bf16_peak, bf16_sus, hbm, peak_kind = peaks()
    achieved = flops / (attn_avg * 1e-3) / 1e12

    if args.fp8:  # the e4m3 path has no one-shot host-tensor call; report the device-resident line only
        # Half of the kept-pair FLOPs (the scores) run as e4m3 products at twice the bf16 rate (the nominal
        # e4m3 : bf16 ratio), the other half (P.V) as bf16 products: the bound on the whole count is 4/3 of the
        # measured bf16 peak.
        mixed_peak = bf16_peak * 4.0 / 3.0
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": job_throughput(world, flops, ms_max * 1e-3),
                              "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
                              "vs_baseline": None, "dtype": "e4m3 scores, bf16 P.V", "data": "synthetic",
                              "config": workload_config(w, {"l2": l2_note,
                                                            "kept_pairs_per_head": info["kept_pairs"],
                                                            "kept_tflop_per_step": flops / 1e12}),
                              "roofline": {"bound": "tensor", "achieved": achieved, "peak": mixed_peak,
                                           "unit": "TFLOP/s", "frac": achieved / mixed_peak,
                                           "frac_of_sustained": achieved / (bf16_sus * 4.0 / 3.0) if bf16_sus else None,
                                           "traffic": stored_traffic(FP8_PROFILE_SUMMARY) if w.name == "h3" else None,
                                           "kernel": f"window_attention_kernel<{w.D}, e4m3>", "kernel_ms": attn_avg,
                                           "merge_kernel_ms": comb_ms / max(1, nrec),
                                           "peak_kind": f"{peak_kind} bf16 burst x 4/3 (e4m3 scores at twice the "
                                                        f"bf16 rate, bf16 P.V)"},
                              "gpu_launches": launches_per_step * args.steps, "clocks": clocks}), flush=True)
        plan.close()
        if world > 1:
            dist.destroy_process_group()
        return
    # The e4m3 forward and the backward, measured briefly on the same workload after the timed region (single
    # process only: a multi-GPU run times the forward replicas alone).
    secondary = secondary_paths(w, q, k, v, plan, bf16_peak) if world == 1 else None
    # End to end through the public call with host tensors: pinned host -> device copies, the forward, and the
    # device -> host copy of the result, every step.
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    del out
    wa.forward(qh, kh, vh, w.T, w.S, w.K, w.r, w.G, w.global_pos, out=oh)
    barrier()
    torch.cuda.synchronize(dev)
    tt0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        wa.forward(qh, kh, vh, w.T, w.S, w.K, w.r, w.G, w.global_pos, out=oh)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks((time.perf_counter() - tt0) / args.e2e_steps, dev, world)
    e2e_value = job_throughput(world, flops, e2e_s)
    nbytes = q.numel() * q.element_size()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        qc, kc, vc = qh, kh, vh
        import oracle.ref as ref
        nc = ref.num_chunks(w.T, w.K)
        heads = sorted({0, w.H // 2, w.H - 1})
        chunks = sorted({0, nc // 2, nc - 1})
        s, f, nrows = oracle_sample(w, qc, kc, vc, heads, chunks, global_rows=True)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
               "blas": blas_threads(),
               "sample": f"heads {heads}: all {w.G} global rows + every row of chunks {chunks} ({nrows} rows, "
                         f"{f / 1e12:.3f} kept TFLOP, {s:.1f} s); throughput of the sample"}

    if rank == 0:
        traffic = stored_traffic() if w.name == "h3" else None
        res = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, {"l2": l2_note,
                                          "kept_pairs_per_head": info["kept_pairs"],
                                          "kept_tflop_per_step": flops / 1e12}),
            "pct_of_bf16_peak": 100.0 * value / world / bf16_peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": achieved / bf16_peak, "frac_of_sustained": achieved / bf16_sus if bf16_sus else None,
                         "traffic": traffic,
                         "kernel": f"window_attention_kernel<{w.D}>", "kernel_ms": attn_avg,
                         "merge_kernel_ms": comb_ms / max(1, nrec),
                         "peak_kind": f"{peak_kind} bf16 burst (sustained {bf16_sus})"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": 3 * nbytes,
                    "d2h_bytes_per_step": nbytes, "ms_per_step": e2e_s * 1e3},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        if secondary is not None:
            res["secondary"] = dict(secondary, note="measured after the timed region, not part of value; "
                                                    "clocks not sampled")
        print(json.dumps(res), flush=True)
    plan.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
