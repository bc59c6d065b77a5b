"""Seeded synthetic inputs, shared by the tests, the benchmark and the CPU oracle's callers.

This module draws random numbers and nothing else: it holds none of the attention arithmetic. The recipe:
a ``torch.Generator`` on the target device, seeded with the workload's seed, draws q, then k, then v, each as
float32 N(0, 1) of shape [B, L, H, D]; when ``k_global_scale`` is not 1 the keys of the global rows are
multiplied by it (x2 is exact in bf16); every tensor is then cast to bfloat16. Draws on a CUDA device use
torch's Philox generator there (milliseconds even at H3 scale); draws on the CPU use torch's CPU generator.
The two devices give different values for the same seed, so a comparison always reads the oracle's inputs back
from the very tensors the GPU used. The backward's upstream gradient dout is drawn the same way from its own
generator, seeded with the workload's seed + 7919, as float32 N(0, 1) cast to bfloat16.
"""
import torch


def make_qkv(w, seed=None, device="cpu"):
    """Return (q, k, v) as contiguous bf16 tensors of shape [B, L, H, D] for workload ``w`` on ``device``."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    shape = (w.B, w.L, w.H, w.D)
    out = []
    for which in ("q", "k", "v"):
        x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
        if which == "k" and w.k_global_scale != 1.0 and w.G > 0:
            x[:, w.g0:w.g0 + w.G] *= w.k_global_scale
        out.append(x.to(torch.bfloat16).contiguous())
        del x
    return tuple(out)


def make_dout(w, seed=None, device="cpu"):
    """Return dout, a contiguous bf16 tensor of shape [B, L, H, D]: the upstream gradient for workload ``w``."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed((w.seed if seed is None else seed) + 7919)
    x = torch.randn((w.B, w.L, w.H, w.D), generator=g, dtype=torch.float32, device=device)
    return x.to(torch.bfloat16).contiguous()
