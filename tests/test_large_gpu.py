"""A long sequence: 66,560,100 rows (65,000 frames of 1,024 tokens, 100 globals at the front), one head, D = 128,
so that every tensor is 17 GB and row offsets times strides pass 2^32 elements. Frame rows of the first, a
middle and the last chunk are checked against the fp64 oracle (which gathers only their kept rows). The global
rows' queries are zeroed, so each global row attends uniformly to all 66.6 M tokens and must equal the mean of v
over the whole sequence (the oracle's pinned closed form: equal scores give the mean of v over the kept set),
summed in float64 by torch. v is shifted by +0.5 so that this mean is far from zero."""
import numpy as np
import pytest
import torch

import oracle.ref as ref
from chunk_windowed_softmax_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

W = configs.Workload("long_sequence", B=1, H=1, D=128, T=65000, S=1024, K=1, r=1, G=100, global_pos=1, seed=71)
REL, ABS = 5e-3, 3e-2


def test_long_sequence_rows_and_globals(cuda):
    w = W
    free, _ = torch.cuda.mem_get_info()
    need = 8 * w.L * w.D * 2 + (8 << 30)  # q, k, v, out, the float32 draw of one tensor, slack
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB of free device memory, {free / 2**30:.0f} GiB free")
    try:
        q, k, v = inputs.make_qkv(w, device="cuda")
        q[:, :w.G] = 0  # global rows (front placement: rows [0, G)) score every key equally
        v += 0.5
        plan = cuda.Plan(w.T, w.S, w.K, w.r, w.G, w.B, w.H, w.D, w.global_pos)
        try:
            out = plan.forward(q, k, v)
            assert plan.check_error() == 0
        finally:
            plan.close()
        torch.cuda.synchronize()

        # frame rows: three chunks (the first and last have clamped windows), each row against the oracle
        nc = w.nc
        for c in (0, nc // 2, nc - 1):
            frames = ref.chunk_frames(c, w.T, w.K)
            want = ref.window_attention_rows(q, k, v, w.T, w.S, w.K, w.r, w.G, w.global_pos, 0, 0, frames=frames)
            rows = np.array(sorted(want))
            got = out[0, torch.as_tensor(rows, device=out.device), 0].double().cpu().numpy()
            ref_rows = np.stack([want[i] for i in rows])
            rel = np.linalg.norm(got - ref_rows) / np.linalg.norm(ref_rows)
            ab = np.abs(got - ref_rows).max()
            assert rel <= REL and ab <= ABS, f"chunk {c}: rel {rel:.2e} abs {ab:.2e}"

        # global rows: the mean of v over all L tokens, summed in float64 over row blocks
        total = torch.zeros(w.D, dtype=torch.float64, device=v.device)
        for lo in range(0, w.L, 1 << 22):
            total += v[0, lo:lo + (1 << 22), 0].double().sum(dim=0)
        mean = (total / w.L).cpu().numpy()
        got = out[0, :w.G, 0].double().cpu().numpy()
        want = np.broadcast_to(mean, got.shape)
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        ab = np.abs(got - want).max()
        assert rel <= REL and ab <= ABS, f"global rows: rel {rel:.2e} abs {ab:.2e}"
    finally:
        q = k = v = out = None
        torch.cuda.empty_cache()
