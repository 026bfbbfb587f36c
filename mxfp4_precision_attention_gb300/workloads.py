"""Seeded synthetic attention inputs (no MXAttention arithmetic lives here).

These tensors stand in for the Wan2.2 / HunyuanVideo attention activations of
"MXAttention" section 5.1, which are not available: standard-normal Q, K, V
in bf16 with a few large "outlier" channels in Q and K, shaped like the
video-DiT and causal-LM workloads the method targets. The same generator feeds
both the CUDA path and the oracle, so both always see identical inputs.

Shapes are ``[B, H, N, 128]`` bf16, contiguous. Values depend on the device
the generator runs on (the CPU and CUDA random streams differ); a test that
compares two implementations draws once and hands the same tensor to both.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

D = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    causal: bool = False
    outlier_channels: tuple[int, ...] | None = None  # fixed channel list, or None
    n_random_outliers: int = 0                        # channels drawn from the seed
    outlier_scale: float = 20.0
    token_lognormal_sigma: float = 0.0                # per-token LogNormal(0, sigma) row scale on Q, K
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> float:
        """Algorithmic FLOP of the forward: 4*B*H*N*N*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * D
        return f / 2 if self.causal else f


WORKLOADS: dict[str, Workload] = {
    "tiny_outlier_512": Workload("tiny_outlier_512", 1, 2, 512, outlier_channels=(3, 77), seed=1,
                                 note="B1 H2 N512, channels 3 and 77 of Q and K x20"),
    "lognormal_4096": Workload("lognormal_4096", 1, 24, 4096, n_random_outliers=4, token_lognormal_sigma=0.5,
                               seed=2, note="B1 H24 N4096, 4 outlier channels x20, per-token LogNormal(0,0.5)"),
    "wan_32760": Workload("wan_32760", 1, 40, 32760, n_random_outliers=4, seed=3,
                          note="video-DiT shaped B1 H40 N32760 (21x30x52 latent tokens)"),
    "hunyuan_118800": Workload("hunyuan_118800", 1, 24, 118800, n_random_outliers=4, seed=4,
                               note="long video-DiT shaped B1 H24 N118800 (33x45x80 tokens)"),
    "causal_lm_8192": Workload("causal_lm_8192", 4, 32, 8192, causal=True, seed=5,
                               note="causal LM B4 H32 N8192, no outliers"),
}


def outlier_channels(w: Workload) -> list[int]:
    if w.outlier_channels is not None:
        return list(w.outlier_channels)
    if w.n_random_outliers == 0:
        return []
    g = torch.Generator(device="cpu")
    g.manual_seed(1_000_003 * (w.seed + 1))
    return sorted(torch.randperm(D, generator=g)[: w.n_random_outliers].tolist())


def generate(w: Workload, device: str | torch.device = "cpu", *, seed: int | None = None, N: int | None = None,
             B: int | None = None, H: int | None = None):
    """Draw (q, k, v) for workload ``w`` as bf16 ``[B, H, N, 128]`` tensors.

    ``N``, ``B`` and ``H`` override the workload's sizes (same recipe, other
    shape); ``seed`` overrides its seed."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    s = w.seed if seed is None else seed
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(s)
    shape = (B, H, N, D)
    chans = outlier_channels(w)
    out = []
    for t in range(3):
        x = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        if t < 2:
            if chans:
                x[..., chans] *= w.outlier_scale
            if w.token_lognormal_sigma > 0:
                z = torch.randn((B, H, N, 1), generator=g, device=dev, dtype=torch.float32)
                x *= torch.exp(w.token_lognormal_sigma * z)
        out.append(x.to(torch.bfloat16).contiguous())
        del x
    return tuple(out)


def as_u16(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
