"""Seeded synthetic inputs shaped like the CodonFM-5B layer workloads.

This module holds none of the quantization arithmetic: it only draws bf16
tensors.  The same tensor feeds both the CUDA path and (as host bit patterns)
the CPU oracle.

Recipe: ``randn`` in fp32 from a ``torch.Generator`` seeded with ``seed`` on
the target device, times ``std``; optionally ``round(outlier_frac * numel)``
entries chosen by ``randperm`` are multiplied by ``outlier_scale``; then one
round-to-nearest-even cast to bf16.
"""
import torch


def bf16_normal(shape, std=1.0, seed=0, device="cuda", outlier_frac=0.0, outlier_scale=1.0):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    x.mul_(float(std))
    if outlier_frac > 0:
        n = x.numel()
        k = int(round(outlier_frac * n))
        if k > 0:
            idx = torch.randperm(n, generator=g, device=device)[:k]
            x.view(-1)[idx] *= float(outlier_scale)
    return x.to(torch.bfloat16)


def host_bits(x_bf16):
    """bf16 tensor -> numpy uint16 array of its bit patterns (for the oracle)."""
    return x_bf16.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


# Per-tensor distributions of the layer workloads: activations ~N(0, 1),
# weights ~N(0, 0.02^2), gradients ~N(0, (1e-3)^2).
ACT_STD, WEIGHT_STD, GRAD_STD = 1.0, 0.02, 1e-3
# Seed offsets per tensor role for the layer workloads.
SEED_X, SEED_W, SEED_DY = 0, 1, 2


def drift_std(step, steps=20, lo=1.0, hi=4.0):
    """Activation std of a drifting run: linear from lo to hi over `steps`."""
    return lo + (hi - lo) * step / max(1, steps - 1)
