"""Seeded synthetic inputs shaped like the workloads the VC-Attention pages report.

This module holds no step of the method: it only draws random tensors.  The
CUDA path and the CPU oracle are both fed from here (the oracle receives CPU
copies of the same bf16 bits).

Shapes and distributions (the pages measure on Wan2.2 / MovieGen Bench
activations, which are not available; these stand in for them):

* ``tiny``   B=1 H=2  N=1024  d=64   Q,K ~ N(0,1); V = mixture of 8 N(0,1)
  centroids + N(0,0.1) noise, 1% of tokens scaled x20 on 4 random channels
  (per head); k=8, 5 k-means iterations.
* ``medium`` B=1 H=8  N=8192  d=128  Q,K ~ N(0,1); V = 64-centroid mixture,
  1% outlier tokens x20 on 4 channels chosen per head; k=64, 5 iterations.
* ``wan``    B=1 H=40 N=75600 d=128  Q,K ~ N(0,1) + per-(head,channel) bias
  N(0,2); V = 256-centroid mixture, 1% outlier tokens x20 on 4 channels that
  change from head to head (each head draws 4 channels, shifted by 3 h);
  k=256, warm-started.
* ``sweep``  B=1 H=24 d=128 N in {4096,...,131072}, generated like ``wan``,
  k = N/512.

Rotary tables (``rope_table``): (cos, sin) of the angle pos_a * base^(-2i/D_a)
for each channel pair, with the pairs split over the three axes of a
(frames, height, width) latent grid -- 21 x 45 x 80 = 75,600 tokens for the
``wan`` shape -- or over one token axis when no grid is given.  base = 10^4.

N(mu, v) denotes variance v.  Cluster memberships are i.i.d. uniform over
token positions (no spatial locality), so a block in sequence order holds a
mixture of clusters.  Tensors are bf16 in the layout [B, N, H, d].
"""
from dataclasses import dataclass

import torch

__all__ = ["Workload", "WORKLOADS", "make_qkv", "drift_v", "sweep_workload", "rope_table", "WAN_GRID"]

WAN_GRID = (21, 45, 80)  # latent frames x height x width of the 75,600-token shape


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    k: int
    iters: int
    centers: int
    qk_bias_var: float
    outlier_mode: str  # "random" | "per_head" | "drift"
    seed: int


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 1024, 64, 8, 5, 8, 0.0, "random", 1000),
    "medium": Workload("medium", 1, 8, 8192, 128, 64, 5, 64, 0.0, "per_head", 1001),
    "wan": Workload("wan", 1, 40, 75600, 128, 256, 3, 256, 2.0, "drift", 1002),
}


def sweep_workload(N: int) -> Workload:
    return Workload("sweep_%d" % N, 1, 24, N, 128, max(1, N // 512), 3, 256, 2.0, "drift", 1003)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _outlier_channels(w: Workload, d: int, h: int, g: torch.Generator, device) -> torch.Tensor:
    if w.outlier_mode == "drift":
        base = torch.randperm(d, generator=g, device=device)[:4]
        return (base + 3 * h) % d
    return torch.randperm(d, generator=g, device=device)[:4]


def make_qkv(w: Workload, device="cpu", B=None, H=None, N=None, d=None, seed=None):
    """Return bf16 Q, K, V of shape [B, N, H, d] on ``device``.

    Size overrides (B, H, N, d) keep the workload's distributions; they are
    used for ragged-tail and edge-case tests.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    d = w.d if d is None else d
    seed = w.seed if seed is None else seed
    dev = torch.device(device)
    g = _gen(seed, dev)
    Q = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=dev)
    K = torch.empty_like(Q)
    V = torch.empty_like(Q)
    for b in range(B):
        for h in range(H):
            q = torch.randn((N, d), generator=g, device=dev)
            k = torch.randn((N, d), generator=g, device=dev)
            if w.qk_bias_var > 0:
                sd = w.qk_bias_var ** 0.5
                q += sd * torch.randn((1, d), generator=g, device=dev)
                k += sd * torch.randn((1, d), generator=g, device=dev)
            centers = torch.randn((w.centers, d), generator=g, device=dev)
            member = torch.randint(0, w.centers, (N,), generator=g, device=dev)
            v = centers[member] + (0.1 ** 0.5) * torch.randn((N, d), generator=g, device=dev)
            rows = torch.rand((N,), generator=g, device=dev) < 0.01
            ch = _outlier_channels(w, d, h, g, dev)
            scale = torch.ones((N, d), device=dev)
            scale[rows.nonzero().flatten()[:, None], ch[None, :]] = 20.0
            v = v * scale
            Q[b, :, h] = q.to(torch.bfloat16)
            K[b, :, h] = k.to(torch.bfloat16)
            V[b, :, h] = v.to(torch.bfloat16)
    return Q, K, V


def drift_v(V: torch.Tensor, step: int, seed: int, var: float = 0.05) -> torch.Tensor:
    """V_t = V_{t-1} + N(0, var): the denoising-schedule drift."""
    g = _gen(seed * 7919 + step, V.device)
    noise = torch.randn(V.shape, generator=g, device=V.device) * (var ** 0.5)
    return (V.float() + noise).to(torch.bfloat16)


def to_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy), same shape."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")


def rope_table(N: int, d: int, grid=None, base: float = 10000.0):
    """fp32 [N, d/2, 2]: (cos, sin) of the rotary angle of each token and
    channel pair -- the memory layout of a complex64 [N, d/2] table.

    With ``grid = (F, Hh, Ww)`` (F*Hh*Ww = N, token n at frame n // (Hh*Ww),
    row (n // Ww) % Hh, column n % Ww) the d/2 pairs are split into
    d/2 - 2*(d/2 // 3) frame pairs and d/2 // 3 pairs for each spatial axis;
    otherwise all pairs follow the token index.
    """
    import numpy as np
    half = d // 2
    n = np.arange(N, dtype=np.int64)
    if grid is None:
        axes = [(n, half)]
    else:
        F, Hh, Ww = grid
        assert F * Hh * Ww == N, (grid, N)
        ps = half // 3
        axes = [(n // (Hh * Ww), half - 2 * ps), ((n // Ww) % Hh, ps), (n % Ww, ps)]
    ang = []
    for pos, pairs in axes:
        dim = 2 * pairs
        omega = base ** (-np.arange(0, dim, 2, dtype=np.float64) / dim)
        ang.append(np.outer(pos.astype(np.float64), omega))
    a = np.concatenate(ang, axis=1)
    return np.ascontiguousarray(np.stack([np.cos(a), np.sin(a)], axis=-1).astype(np.float32))
