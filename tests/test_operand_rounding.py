"""Why the tensor-core operands are fp16: an fp64 emulation of the rounding
the GPU path applies to its 16-bit operands, on the peaked statistics of the
largest workload (x = 3 N(0,1), Wq and Wk ~ U(+-4/sqrt(512)), head dim 512),
against the exact block from the oracle.

The emulation rounds, as the kernels do: Z (the GroupNorm output) and the four
weights to the operand type; Q, K and V after the fp32-accumulated projection
(bias added); P after the max-subtracted exponentials; O after the division by
the row sums; the output projection accumulates in full precision.  bf16 keeps
8 bits of mantissa against fp16's 11, and the logit error it leaves (|q||k|
grows with the peaked weights) is what pushes the branch past the 1e-2 bound
with bf16 operands while fp16 stays well inside it.  This is a CPU test of the
reasoning; the GPU comparison of the two libraries is in test_gpu_operands.py.
"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_net_spatial_gb300 import workloads as wls


def _round_f16(a):
    return a.astype(np.float16).astype(np.float64)


def _round_bf16(a):
    # to fp32 first (exact for these magnitudes up to one fp32 rounding), then
    # round-to-nearest-even on the upper 16 bits
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _emulated_branch(x, p, G, h, qi, rnd):
    """The branch y at the query pixels qi with 16-bit operands rounded by rnd."""
    x = x.double().numpy()
    B, C, H, W = x.shape
    N, d = H * W, C // h
    t = {k: v.double().numpy() for k, v in p.items()}
    z = torch.nn.functional.group_norm(torch.from_numpy(x), G, torch.from_numpy(t["norm_weight"]),
                                       torch.from_numpy(t["norm_bias"]), eps=1e-5).numpy()
    z = rnd(z.reshape(B, C, N).transpose(0, 2, 1))                       # [B, N, C]
    wq, wk, wv, wo = (rnd(t[k]) for k in ("q_weight", "k_weight", "v_weight", "out_weight"))
    q = rnd(z[:, qi] @ wq.T + t["q_bias"])
    k = rnd(z @ wk.T + t["k_bias"])
    v = rnd(z @ wv.T + t["v_bias"])
    o = np.empty((B, len(qi), C))
    for j in range(h):
        sl = slice(j * d, (j + 1) * d)
        s = q[:, :, sl] @ k[:, :, sl].transpose(0, 2, 1) / np.sqrt(d)
        e = rnd(np.exp(s - s.max(axis=-1, keepdims=True)))
        o[:, :, sl] = rnd((e @ v[:, :, sl]) / e.sum(axis=-1, keepdims=True))
    y = o @ wo.T + t["out_bias"]
    return y.transpose(0, 2, 1)                                            # [B, C, nq]


def test_bf16_operands_miss_the_bound_on_the_peaked_workload_fp16_does_not():
    base = wls.WORKLOADS["vae16384"]
    # the largest workload's statistics on a quarter of its grid (64 x 64)
    wl = wls.custom("vae-peaked-64", 1, 512, 64, 64, 32, 1, "f32", seed=base.seed, x_scale=base.x_scale,
                    w_bound=base.w_bound, qk_bound=base.qk_bound)
    x, p, _ = wls.make_inputs(wl)
    qi = np.sort(torch.randperm(wl.N, generator=torch.Generator().manual_seed(5))[:256].numpy())
    exact = oracle.forward(x, p, wl.num_groups, wl.num_heads, qidx=qi)["y"]
    err = {}
    for name, rnd in (("f16", _round_f16), ("bf16", _round_bf16)):
        y = _emulated_branch(x, p, wl.num_groups, wl.num_heads, qi, rnd)
        err[name] = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert err["f16"] < 3e-3, err
    assert err["bf16"] > 1e-2, err
    assert err["bf16"] > 4 * err["f16"], err


def test_rounding_helpers_are_round_to_nearest_even():
    v = np.array([1.0, 1.0 + 2 ** -9, 1.0 + 3 * 2 ** -9, -2.5, 3.0e-3])
    np.testing.assert_array_equal(_round_bf16(v), [1.0, 1.0, 1.0 + 2 ** -7, -2.5,
                                                   float(torch.tensor(3.0e-3).to(torch.bfloat16))])
    np.testing.assert_array_equal(_round_f16(v), v.astype(np.float16).astype(np.float64))
