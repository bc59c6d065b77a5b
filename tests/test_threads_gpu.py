"""Launch state shared by host threads (the header promises that every function may be called from any thread).

The one-time work of a first call (the kernels' shared-memory opt-in, which belongs to the CUDA context, and the
driver entry-point lookups) is guarded per context. The test runs in a fresh process, so that the first calls there
really are first: two threads, started together, each make their first forward and first backward on their own
geometry; both must succeed and equal the same calls made again one after the other.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys, threading
    sys.path.insert(0, {root!r})
    import torch
    import chunk_windowed_softmax_gb300 as wa
    from chunk_windowed_softmax_gb300 import configs, inputs

    geos = [configs.Workload("t0", B=1, H=2, D=128, T=8, S=90, K=2, r=1, G=40, global_pos=0, seed=61),
            configs.Workload("t1", B=1, H=3, D=64, T=9, S=70, K=3, r=1, G=33, global_pos=1, seed=62)]
    data = []
    for w in geos:
        q, k, v = inputs.make_qkv(w, device="cuda")
        data.append((q, k, v, inputs.make_dout(w, device="cuda")))
    torch.cuda.synchronize()

    def run(i):
        w = geos[i]
        q, k, v, dout = data[i]
        plan = wa.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
        try:
            out, lse = plan.forward_lse(q, k, v)
            grads = plan.backward(q, k, v, out, dout, lse)
            st = plan.check_error()
        finally:
            plan.close()
        torch.cuda.synchronize()
        return st, out, grads

    start = threading.Barrier(2)
    results = [None, None]
    errors = []

    def worker(i):
        try:
            start.wait()
            results[i] = run(i)
        except Exception as e:
            errors.append(repr(e))

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=120)
    assert not errors, errors
    assert all(r is not None for r in results), "a thread did not finish"
    for i in range(2):
        st, out, grads = results[i]
        assert st == 0, st
        st2, out2, grads2 = run(i)
        assert st2 == 0 and torch.equal(out, out2) and all(torch.equal(a, b) for a, b in zip(grads, grads2))
    print("threads ok")
""")


def test_concurrent_first_calls_in_fresh_process(cuda):
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
