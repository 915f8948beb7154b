"""Seeded synthetic workloads for the spatial self-attention block.

This module only draws random numbers: it holds none of the block's
arithmetic, and both the CUDA path (tests, bench) and the fp64 oracle are fed
from it.  Generation runs on the CPU with torch's default generator:

  torch.manual_seed(seed), then draw, in order,
  x, norm_weight, norm_bias, q_weight, q_bias, k_weight, k_bias,
  v_weight, v_bias, out_weight, out_bias;
  U(-a, a) = (rand * 2 - 1) * a;  norm_weight = 1 + 0.1 N(0,1),
  norm_bias = 0.1 N(0,1); values are drawn in fp32, then cast to the stored
  dtype.  A query sample (large problems) continues the same generator with
  randperm(H*W)[:n], sorted.

The five named shapes are the SD-VAE / U-Net attention levels (the pages name
no dataset; these are synthetic stand-ins with the same shapes and scales).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PARAM_KEYS = ("norm_weight", "norm_bias", "q_weight", "q_bias", "k_weight", "k_bias",
              "v_weight", "v_bias", "out_weight", "out_bias")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    C: int
    H: int
    W: int
    num_groups: int
    num_heads: int
    dtype: str = "f32"          # stored dtype of x, the parameters and out: 'f32' | 'bf16'
    seed: int = 0
    x_scale: float = 1.0        # x = x_scale * N(0, 1)
    w_bound: float | None = None    # U(-a, a) bound for weights and biases; None -> 1/sqrt(C)
    qk_bound: float | None = None   # U bound for q_weight/k_weight; None -> w_bound
    n_query_sample: int = 0     # >0: oracle checks this many seeded query pixels

    @property
    def N(self) -> int:
        return self.H * self.W

    @property
    def d(self) -> int:
        return self.C // self.num_heads

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs of one block forward: 8 N C^2 for the four
        projections plus 4 N^2 C for scores and P V, per sample."""
        return float(self.B) * (8.0 * self.N * self.C ** 2 + 4.0 * self.N ** 2 * self.C)

    @property
    def tokens(self) -> int:
        return self.B * self.N


WORKLOADS = {
    "tiny": Workload("tiny", 1, 64, 8, 8, 8, 2, "f32", 0, 1.0, 1.0 / 8.0),
    "vae1024": Workload("vae1024", 1, 512, 32, 32, 32, 1, "f32", 1, 1.0, 1.0 / math.sqrt(512)),
    "unet-l1": Workload("unet-l1", 2, 320, 64, 64, 32, 8, "f32", 2, 1.0, 1.0 / math.sqrt(320)),
    "unet-lowres": Workload("unet-lowres", 8, 1280, 16, 16, 32, 20, "bf16", 3, 1.0, 1.0 / math.sqrt(1280)),
    "vae16384": Workload("vae16384", 1, 512, 128, 128, 32, 1, "f32", 4, 3.0, 1.0 / math.sqrt(512),
                         4.0 / math.sqrt(512), 512),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def make_inputs(wl: Workload):
    """Return (x, params, qidx) as CPU torch tensors in the stored dtype.

    qidx is a sorted int64 tensor of wl.n_query_sample pixel indices, or None.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(wl.seed)
    C = wl.C
    a = wl.w_bound if wl.w_bound is not None else 1.0 / math.sqrt(C)
    aqk = wl.qk_bound if wl.qk_bound is not None else a

    def u(shape, bound):
        return (torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1) * bound

    x = torch.randn((wl.B, C, wl.H, wl.W), generator=g, dtype=torch.float32) * wl.x_scale
    p = {}
    p["norm_weight"] = 1 + 0.1 * torch.randn((C,), generator=g, dtype=torch.float32)
    p["norm_bias"] = 0.1 * torch.randn((C,), generator=g, dtype=torch.float32)
    p["q_weight"] = u((C, C), aqk)
    p["q_bias"] = u((C,), a)
    p["k_weight"] = u((C, C), aqk)
    p["k_bias"] = u((C,), a)
    p["v_weight"] = u((C, C), a)
    p["v_bias"] = u((C,), a)
    p["out_weight"] = u((C, C), a)
    p["out_bias"] = u((C,), a)
    qidx = None
    if wl.n_query_sample:
        qidx = torch.sort(torch.randperm(wl.N, generator=g)[: wl.n_query_sample]).values
    dt = torch_dtype(wl.dtype)
    x = x.to(dt)
    p = {k: v.to(dt).contiguous() for k, v in p.items()}
    return x.contiguous(), p, qidx


def custom(name, B, C, H, W, num_groups, num_heads, dtype="f32", seed=0, x_scale=1.0,
           w_bound=None, qk_bound=None, n_query_sample=0) -> Workload:
    """A workload of any shape, drawn with the same recipe."""
    return Workload(name, B, C, H, W, num_groups, num_heads, dtype, seed, x_scale, w_bound, qk_bound,
                    n_query_sample)
