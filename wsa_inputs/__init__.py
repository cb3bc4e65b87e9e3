"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA path.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and value distributions of the workloads below, so the same
bits can be handed to the GPU library and (upcast to fp64) to the oracle.

Every tensor is drawn from ``torch.randn`` in fp32 under a
``torch.Generator`` seeded with an explicit integer, scaled, then rounded once
to the storage dtype.  Seeds: q, k, v of layer L use base + 3L + {0, 1, 2}; the
outlier channel set uses base + 7919; the transition activation uses
base + 104729.  A generator on ``device='cuda'`` is deterministic but draws
different numbers from the CPU one, so a test always hands one drawn tensor to
both sides rather than drawing twice.
"""

from dataclasses import dataclass

import torch

BASE_SEED = 1234


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    W: int
    nt: int
    nh: int
    nw: int
    heads: int
    head_dim: int
    dtype: str          # "bf16" or "fp32"
    dist: str           # "normal", "normal_half_var", "outlier"
    layers: int = 2     # regular + shifted

    @property
    def num_tokens(self):
        return self.T * self.H * self.W

    @property
    def channels(self):
        return self.heads * self.head_dim

    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


# Workloads shaped like the SeedVR2 720p-reference setting of the window note.
WORKLOADS = {
    # 576 tokens, wt,wh,ww = 2,5,5, ragged edges, fp32 check.
    "tiny": Workload("tiny", 4, 9, 16, 2, 9, 16, 2, 64, "fp32", "normal"),
    # 720p-area grid, 75,600 tokens, wt,wh,ww = 6,15,27.
    "720p": Workload("720p", 21, 45, 80, 4, 3, 3, 24, 128, "bf16", "normal_half_var"),
    # 1080p-scale grid, 171,360 tokens, same window size, outlier channels in Q and K.
    "1080p": Workload("1080p", 21, 68, 120, 4, 3, 3, 24, 128, "bf16", "outlier"),
    # long clip at 720p area: temporal window capped by min(T, 30) -> wt = 8.
    "long": Workload("long", 31, 45, 80, 4, 3, 3, 24, 128, "bf16", "normal"),
    # 32 alternating layers on a 302,400-token grid.
    "32layer": Workload("32layer", 21, 90, 160, 4, 3, 3, 24, 128, "bf16", "normal", layers=32),
}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, seed, device="cpu"):
    return torch.randn(shape, generator=_gen(seed, device), dtype=torch.float32, device=device)


def outlier_channels(channels, seed=BASE_SEED + 7919, frac=0.01):
    """Seeded choice of round(frac * channels) channel indices (CPU permutation)."""
    count = max(1, int(round(frac * channels)))
    perm = torch.randperm(channels, generator=_gen(seed, "cpu"))
    return torch.sort(perm[:count]).values


def qkv(wl, layer=0, device="cpu", base_seed=BASE_SEED, tokens=None):
    """Q, K, V of one layer, shape [N, heads, head_dim], in canonical token order.

    ``tokens`` overrides N (used for packed-order inputs of the same size)."""
    n = wl.num_tokens if tokens is None else tokens
    shape = (n, wl.heads, wl.head_dim)
    out = []
    for j in range(3):
        x = randn(shape, base_seed + 3 * layer + j, device)
        if wl.dist == "normal_half_var":
            x = x * (2.0 ** -0.5)
        elif wl.dist == "outlier" and j < 2:
            idx = outlier_channels(wl.channels).to(device)
            x = x.view(n, wl.channels)
            x[:, idx] *= 8.0
            x = x.view(shape)
        out.append(x.to(wl.torch_dtype()))
    return tuple(out)


def activation(wl, device="cpu", base_seed=BASE_SEED, channels=None):
    """Hidden-state rows [N, channels] (default heads*head_dim) for a transition."""
    c = wl.channels if channels is None else channels
    x = randn((wl.num_tokens, c), base_seed + 104729, device)
    return x.to(wl.torch_dtype())


def custom(T, H, W, nt, nh, nw, heads, head_dim, dtype="bf16", dist="normal", name="custom"):
    return Workload(name, T, H, W, nt, nh, nw, heads, head_dim, dtype, dist)
