"""Pins for the fp64 oracle: it is checked against things other than itself.

Each test names the passage of the tensortonic page
"diffusion-l03-spatial-self-attention" (problem statement, block equation,
hints, worked examples) or the mathematical fact it relies on.  Together they
are chosen so that a plausible slip in the oracle fails at least one: a dropped
bias, 1/d instead of 1/sqrt(d), a transposed weight, the wrong token order,
the unbiased variance, eps outside the root, cross-sample statistics, a wrong
head slice, a missing residual, a bad rounding rule.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from diffusion_net_spatial_gb300 import workloads as wls

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "worked_examples.json")))


def _params(C, seed, scale=0.5):
    g = np.random.default_rng(seed)
    p = {
        "norm_weight": 1 + 0.3 * g.standard_normal(C),
        "norm_bias": 0.3 * g.standard_normal(C),
    }
    for k in ("q", "k", "v", "out"):
        p[f"{k}_weight"] = scale * g.standard_normal((C, C))
        p[f"{k}_bias"] = scale * g.standard_normal(C)
    return p


def _x(B, C, H, W, seed, scale=1.0, shift=0.0):
    g = np.random.default_rng(seed + 1000)
    return shift + scale * g.standard_normal((B, C, H, W))


def _torch_route(x, p, G, h):
    """The block composed from torch library routines in fp64 (CPU):
    F.group_norm, flatten(2).transpose(1, 2), F.linear, the view/transpose head
    split of the hints, F.scaled_dot_product_attention (default scale
    1/sqrt(E)), F.linear, the inverse reshape, and the residual."""
    xt = torch.from_numpy(x)
    B, C, H, W = xt.shape
    t = {k: torch.from_numpy(v) for k, v in p.items()}
    gn = F.group_norm(xt, G, t["norm_weight"], t["norm_bias"], eps=1e-5)
    z = gn.flatten(2).transpose(1, 2)
    q = F.linear(z, t["q_weight"], t["q_bias"])
    k = F.linear(z, t["k_weight"], t["k_bias"])
    v = F.linear(z, t["v_weight"], t["v_bias"])
    N, d = H * W, C // h
    q, k, v = (u.view(B, N, h, d).transpose(1, 2) for u in (q, k, v))
    o = F.scaled_dot_product_attention(q, k, v)
    o = o.transpose(1, 2).reshape(B, N, C)
    y = F.linear(o, t["out_weight"], t["out_bias"])
    y = y.transpose(1, 2).reshape(B, C, H, W)
    return y.numpy()


SHAPES = [
    # B, C, H, W, G, h
    (1, 4, 2, 2, 2, 2),     # the shape of worked example 1 (d = 2)
    (1, 2, 2, 3, 1, 1),     # example 2: H != W pins the i*W + j token order
    (2, 4, 1, 1, 4, 2),     # example 3: one pixel, one channel per group
    (2, 8, 3, 5, 2, 2),
    (3, 12, 4, 3, 3, 3),
    (1, 16, 5, 7, 4, 4),
    (2, 6, 2, 7, 6, 1),
]


@pytest.mark.parametrize("B,C,H,W,G,h", SHAPES)
def test_matches_torch_library_composition(B, C, H, W, G, h):
    """Library special case: every step of the definition done by a torch
    routine instead of the oracle's loops agrees to fp64 rounding."""
    x = _x(B, C, H, W, seed=B * 100 + C, scale=1.5, shift=0.3)
    p = _params(C, seed=C + H)
    y = oracle.forward(x, p, G, h)["y"].reshape(B, C, H, W)
    ref = _torch_route(x, p, G, h)
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)


def test_scale_is_inverse_sqrt_d_not_inverse_d():
    """Worked example 1 divides the scores by sqrt(2) for d = 2.  The test is
    sensitive: the 1/d variant gives a measurably different block."""
    B, C, H, W, G, h = 1, 4, 2, 2, 2, 2
    x = _x(B, C, H, W, 7, scale=2.0)
    p = _params(C, 8, scale=1.5)
    y = oracle.forward(x, p, G, h)["y"].reshape(B, C, H, W)
    xt = torch.from_numpy(x)
    t = {k: torch.from_numpy(v) for k, v in p.items()}
    z = F.group_norm(xt, G, t["norm_weight"], t["norm_bias"], eps=1e-5).flatten(2).transpose(1, 2)
    q, k, v = (F.linear(z, t[f"{n}_weight"], t[f"{n}_bias"]).view(B, 4, h, 2).transpose(1, 2) for n in "qkv")
    for scale, expect_equal in ((1 / math.sqrt(2), True), (1 / 2, False)):
        a = torch.softmax(q @ k.transpose(-1, -2) * scale, dim=-1)
        o = (a @ v).transpose(1, 2).reshape(B, 4, C)
        yy = F.linear(o, t["out_weight"], t["out_bias"]).transpose(1, 2).reshape(B, C, H, W).numpy()
        assert np.allclose(y, yy, rtol=1e-11, atol=1e-11) == expect_equal


def test_group_norm_statistics_two_pass_library():
    """GN statistics equal numpy's mean/var (biased, ddof=0) per (sample,
    group) over contiguous channel blocks; rstd = 1/sqrt(var + 1e-5)."""
    B, C, H, W, G = 3, 12, 5, 4, 4
    x = _x(B, C, H, W, 3, scale=2.0, shift=5.0)
    mean, rstd = oracle.gn_stats(x, G)
    xg = x.reshape(B, G, -1)
    np.testing.assert_allclose(mean, xg.mean(-1), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(xg.var(-1, ddof=0) + 1e-5), rtol=1e-12)


def test_group_norm_output_has_zero_mean_unit_variance():
    """With norm_weight = 1 and norm_bias = 0, Z restricted to one (sample,
    group) has mean 0 and variance var/(var + eps) (=1 up to eps)."""
    B, C, H, W, G, h = 2, 8, 3, 4, 2, 2
    x = _x(B, C, H, W, 5, scale=3.0, shift=-2.0)
    p = _params(C, 6)
    p["norm_weight"] = np.ones(C)
    p["norm_bias"] = np.zeros(C)
    z = oracle.forward(x, p, G, h, want=("z",))["z"]          # (B, N, C)
    zg = z.reshape(B, H * W, G, C // G).transpose(0, 2, 1, 3).reshape(B, G, -1)
    var = x.reshape(B, G, -1).var(-1)
    np.testing.assert_allclose(zg.mean(-1), 0.0, atol=1e-13)
    np.testing.assert_allclose(zg.var(-1), var / (var + 1e-5), rtol=1e-12)


def test_single_pixel_closed_form():
    """H = W = 1: one token, the softmax over one key is 1, so
    out - x = Wo (Wv GN(x) + bv) + bo with GN over the C/G channels of a group."""
    B, C, G, h = 3, 8, 2, 2
    x = _x(B, C, 1, 1, 11, scale=1.3)
    p = _params(C, 12)
    y = oracle.forward(x, p, G, h)["y"][:, :, 0]               # (B, C)
    xs = x[:, :, 0, 0]
    xg = xs.reshape(B, G, -1)
    zh = (xg - xg.mean(-1, keepdims=True)) / np.sqrt(xg.var(-1, keepdims=True) + 1e-5)
    z = zh.reshape(B, C) * p["norm_weight"] + p["norm_bias"]
    v = z @ p["v_weight"].T + p["v_bias"]
    ref = v @ p["out_weight"].T + p["out_bias"]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_zero_query_key_weights_give_uniform_attention():
    """Wq = Wk = 0: every score in a row is the same constant, the softmax is
    uniform, and every pixel receives Wo mean_m(v_m) + bo."""
    B, C, H, W, G, h = 2, 8, 3, 5, 4, 2
    x = _x(B, C, H, W, 13)
    p = _params(C, 14)
    p["q_weight"][:] = 0
    p["k_weight"][:] = 0
    r = oracle.forward(x, p, G, h, want=("v",))
    vbar = r["v"].mean(axis=1)                                   # (B, C)
    ref = vbar @ p["out_weight"].T + p["out_bias"]
    np.testing.assert_allclose(r["y"], np.repeat(ref[:, :, None], H * W, axis=2), rtol=1e-12, atol=1e-12)
    # and the result cannot depend on how the channels are split into heads
    y1 = oracle.forward(x, p, G, 1)["y"]
    y4 = oracle.forward(x, p, G, 4)["y"]
    np.testing.assert_allclose(y1, y4, rtol=1e-12, atol=1e-12)


def test_softmax_rows_sum_to_one():
    """The softmax normalises over keys (hint: softmax(scores, dim=-1)); the
    example 1 explanation's weights 0.240 + 0.257 + 0.305 + 0.197 = 0.999 are
    one to their printed rounding."""
    B, C, H, W, G, h = 2, 8, 3, 3, 2, 4
    x = _x(B, C, H, W, 15, scale=2.0)
    p = _params(C, 16, scale=2.0)
    P = oracle.forward(x, p, G, h, want=("p",))["p"]
    assert (P >= 0).all()
    np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-14)
    w = GOLDEN["examples"][0]["explanation_head0_pixel0_attention"]
    assert abs(sum(w) - 1.0) <= len(w) * 0.0005


def test_pixel_permutation_equivariance_non_square():
    """Attention over pixels has no positional term: permuting the pixels of x
    permutes out - x the same way (H != W as in worked example 2)."""
    B, C, H, W, G, h = 2, 6, 2, 3, 3, 2
    x = _x(B, C, H, W, 17)
    p = _params(C, 18)
    perm = np.random.default_rng(3).permutation(H * W)
    xp = x.reshape(B, C, -1)[:, :, perm].reshape(B, C, H, W)
    y = oracle.forward(x, p, G, h)["y"]
    yp = oracle.forward(xp, p, G, h)["y"]
    np.testing.assert_allclose(yp, y[:, :, perm], rtol=1e-12, atol=1e-12)


def test_token_order_row_major():
    """tokens() puts pixel (i, j) at row i*W + j: the Z the oracle exports
    equals x.flatten(2).transpose(1, 2) of the group-normed image (the hint),
    and not the column-major order, on a non-square image."""
    B, C, H, W, G, h = 1, 4, 2, 3, 2, 2
    x = _x(B, C, H, W, 19)
    p = _params(C, 20)
    z = oracle.forward(x, p, G, h, want=("z",))["z"]
    gn = F.group_norm(torch.from_numpy(x), G, torch.from_numpy(p["norm_weight"]),
                      torch.from_numpy(p["norm_bias"]), eps=1e-5)
    np.testing.assert_allclose(z, gn.flatten(2).transpose(1, 2).numpy(), rtol=1e-12, atol=1e-12)
    zt = gn.transpose(2, 3).flatten(2).transpose(1, 2).numpy()
    assert not np.allclose(z, zt)


def test_key_bias_invariance():
    """Changing bk adds q . bk_j to every score of a row: the softmax is
    unchanged, so out is unchanged."""
    B, C, H, W, G, h = 2, 8, 3, 4, 2, 2
    x = _x(B, C, H, W, 21)
    p = _params(C, 22)
    y0 = oracle.forward(x, p, G, h)["y"]
    p["k_bias"] = p["k_bias"] + 3.0
    y1 = oracle.forward(x, p, G, h)["y"]
    np.testing.assert_allclose(y0, y1, rtol=1e-11, atol=1e-11)


def test_query_key_rescale_invariance():
    """(Wq, bq) * a together with (Wk, bk) / a leaves every score unchanged."""
    B, C, H, W, G, h = 1, 8, 4, 4, 4, 2
    x = _x(B, C, H, W, 23)
    p = _params(C, 24)
    y0 = oracle.forward(x, p, G, h)["y"]
    a = 2.5
    for k in ("q_weight", "q_bias"):
        p[k] = p[k] * a
    for k in ("k_weight", "k_bias"):
        p[k] = p[k] / a
    y1 = oracle.forward(x, p, G, h)["y"]
    np.testing.assert_allclose(y0, y1, rtol=1e-11, atol=1e-11)


def test_head_permutation_invariance():
    """Relabelling the heads (rows of Wq, Wk, Wv and entries of bq, bk, bv by
    head block, and the matching columns of Wo) leaves out unchanged; a wrong
    head slice or concat order breaks it."""
    B, C, H, W, G, h = 2, 12, 3, 3, 3, 3
    d = C // h
    x = _x(B, C, H, W, 25)
    p = _params(C, 26)
    y0 = oracle.forward(x, p, G, h)["y"]
    hp = [2, 0, 1]
    idx = np.concatenate([np.arange(j * d, (j + 1) * d) for j in hp])
    q = dict(p)
    for n in "qkv":
        q[f"{n}_weight"] = p[f"{n}_weight"][idx]
        q[f"{n}_bias"] = p[f"{n}_bias"][idx]
    q["out_weight"] = p["out_weight"][:, idx]
    y1 = oracle.forward(x, q, G, h)["y"]
    np.testing.assert_allclose(y0, y1, rtol=1e-11, atol=1e-11)


def test_value_bias_shift_closed_form():
    """Adding delta to bv adds Wo delta to every pixel, because each softmax
    row sums to one."""
    B, C, H, W, G, h = 2, 8, 3, 2, 2, 4
    x = _x(B, C, H, W, 27)
    p = _params(C, 28)
    y0 = oracle.forward(x, p, G, h)["y"]
    delta = np.linspace(-1, 1, C)
    p["v_bias"] = p["v_bias"] + delta
    y1 = oracle.forward(x, p, G, h)["y"]
    np.testing.assert_allclose(y1 - y0, np.broadcast_to((p["out_weight"] @ delta)[None, :, None], y0.shape),
                               rtol=1e-11, atol=1e-11)


def test_brute_force_python_loops_tiny():
    """Brute force: the definition evaluated with scalar Python arithmetic on
    a tiny non-square problem (d = 3, two groups of three channels)."""
    B, C, H, W, G, h = 1, 6, 2, 2, 2, 2
    x = _x(B, C, H, W, 29)
    p = _params(C, 30)
    N, d, cg = H * W, C // h, C // G
    y = oracle.forward(x, p, G, h)["y"]
    xs = x.reshape(B, C, N)
    ref = np.zeros((B, C, N))
    for b in range(B):
        z = [[0.0] * C for _ in range(N)]
        for g in range(G):
            vals = [xs[b, c, n] for c in range(g * cg, (g + 1) * cg) for n in range(N)]
            mu = sum(vals) / len(vals)
            var = sum((t - mu) ** 2 for t in vals) / len(vals)
            for c in range(g * cg, (g + 1) * cg):
                for n in range(N):
                    z[n][c] = (xs[b, c, n] - mu) / math.sqrt(var + 1e-5) * p["norm_weight"][c] + p["norm_bias"][c]

        def lin(wk, bk, row):
            return [sum(row[c] * p[wk][f][c] for c in range(C)) + p[bk][f] for f in range(C)]
        Q = [lin("q_weight", "q_bias", z[n]) for n in range(N)]
        K = [lin("k_weight", "k_bias", z[n]) for n in range(N)]
        V = [lin("v_weight", "v_bias", z[n]) for n in range(N)]
        O = [[0.0] * C for _ in range(N)]
        for j in range(h):
            for n in range(N):
                s = [sum(Q[n][j * d + e] * K[m][j * d + e] for e in range(d)) / math.sqrt(d) for m in range(N)]
                mx = max(s)
                ex = [math.exp(t - mx) for t in s]
                den = sum(ex)
                for e in range(d):
                    O[n][j * d + e] = sum(ex[m] / den * V[m][j * d + e] for m in range(N))
        for n in range(N):
            out = lin("out_weight", "out_bias", O[n])
            for c in range(C):
                ref[b, c, n] = out[c]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_example3_branch_identical_across_samples():
    """Worked example 3 (two samples, C = 4, H = W = 1, 4 groups): a group
    holds one value, so GN(x) = norm_bias for any x and the branch out - x is
    the same for both samples.  The printed outputs show this to every printed
    digit, and the oracle reproduces it for arbitrary parameters; it would give
    NaN with the unbiased variance and cross-sample statistics would break it."""
    ex = GOLDEN["examples"][2]
    x = np.array(ex["x"], dtype=np.float64)
    out = np.array(ex["out"], dtype=np.float64)
    delta = (out - x)[:, :, 0, 0]
    np.testing.assert_allclose(delta[0], delta[1], atol=2e-6)     # printed to 6 decimals
    for seed in range(3):
        p = _params(4, 40 + seed)
        y = oracle.forward(x, p, ex["num_groups"], ex["num_heads"], want=("z",))
        assert np.isfinite(y["y"]).all()
        np.testing.assert_allclose(y["y"][0], y["y"][1], rtol=0, atol=1e-15)
        np.testing.assert_allclose(y["z"][:, 0, :], np.broadcast_to(p["norm_bias"], (2, 4)), atol=1e-15)


def test_examples_shapes_and_dtype():
    """Every worked example returns (B, C, H, W) in x's dtype (return rule)."""
    for ex in GOLDEN["examples"]:
        x = torch.tensor(ex["x"], dtype=torch.float32)
        C = x.shape[1]
        p = {k: torch.from_numpy(v).float() for k, v in _params(C, 50).items()}
        out, y = oracle.block(x, p, ex["num_groups"], ex["num_heads"])
        assert out.shape == (x.shape[0], C, x.shape[2] * x.shape[3])
        # f32 rounding: the result is exactly representable in float32
        assert np.array_equal(out.astype(np.float32).astype(np.float64), out)


def test_query_sampled_mode_equals_full_mode():
    B, C, H, W, G, h = 2, 8, 4, 5, 4, 2
    x = _x(B, C, H, W, 31)
    p = _params(C, 32)
    full = oracle.forward(x, p, G, h, want=("q", "o"))
    qi = np.array([0, 3, 7, 19])
    part = oracle.forward(x, p, G, h, qidx=qi, want=("q", "o"))
    np.testing.assert_array_equal(part["y"], full["y"][:, :, qi])
    np.testing.assert_array_equal(part["o"], full["o"][:, qi])


def test_rejects_bad_shapes():
    x = _x(1, 6, 2, 2, 33)
    p = _params(6, 34)
    with pytest.raises(ValueError):
        oracle.forward(x, p, 4, 2)      # C % G != 0
    with pytest.raises(ValueError):
        oracle.forward(x, p, 2, 4)      # C % h != 0 (E_CONSTRAINT in the attention operator doc)


def test_round_to_fp32_and_bf16_nearest_even():
    """The return takes x's dtype; rounding is once, to nearest-even.
    bf16: checked against torch's fp32 -> bf16 conversion (RNE) on values that
    are exact in fp32, and on hand-made ties and the overflow edge."""
    g = np.random.default_rng(0)
    v32 = (g.standard_normal(20000) * np.exp(g.uniform(-30, 30, 20000))).astype(np.float32)
    bits = oracle.round_to(v32.astype(np.float64), "bf16")
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -130 + 2.0 ** -134,
                     3.3895313892515355e38, 3.4e38, 0.0, -0.0])
    got = oracle.bf16_bits_to_f64(oracle.round_to(ties, "bf16"))
    assert got[0] == 1.0 and got[1] == 1 + 2 * 2.0 ** -7 and got[2] == -1.0
    assert got[3] == 2.0 ** -130
    assert got[4] == 3.3895313892515355e38 and np.isinf(got[5])
    # an fp64 value a hair above a bf16 tie rounds up even though fp32 rounding
    # first would land exactly on the tie and round to even (down)
    v = 1 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.bf16_bits_to_f64(oracle.round_to(np.array([v]), "bf16"))[0] == 1 + 2.0 ** -7
    f = oracle.round_to(np.array([1 + 2.0 ** -24, 1 + 3 * 2.0 ** -24]), "f32")
    assert f[0] == np.float32(1.0) and f[1] == np.float32(1 + 2.0 ** -22)


def test_workload_generator_is_deterministic_and_shaped():
    wl = wls.WORKLOADS["tiny"]
    x1, p1, q1 = wls.make_inputs(wl)
    x2, p2, q2 = wls.make_inputs(wl)
    assert torch.equal(x1, x2) and all(torch.equal(p1[k], p2[k]) for k in p1)
    assert x1.shape == (1, 64, 8, 8) and q1 is None
    assert set(p1) == set(oracle.PARAM_KEYS)
    wl5 = wls.WORKLOADS["vae16384"]
    assert wl5.n_query_sample == 512 and wl5.d == 512
    b4 = wls.WORKLOADS["unet-lowres"]
    assert b4.dtype == "bf16" and b4.d == 64


def test_step_functions_compose_to_the_block():
    """The exported attention and output-projection steps, fed the oracle's
    own Q/K/V and O, give the same branch as the full block (they are the
    block's steps 3 and 4), and the attention step matches torch's SDPA."""
    B, C, H, W, G, h = 2, 12, 3, 5, 3, 3
    x = _x(B, C, H, W, 60)
    p = _params(C, 61)
    r = oracle.forward(x, p, G, h, want=("q", "k", "v", "o"))
    o = oracle.attention(r["q"], r["k"], r["v"], h)
    np.testing.assert_array_equal(o, r["o"])
    y = oracle.out_proj(o, p["out_weight"], p["out_bias"])
    np.testing.assert_array_equal(y, r["y"])
    qt, kt, vt = (torch.from_numpy(r[n]).view(B, H * W, h, C // h).transpose(1, 2) for n in "qkv")
    ref = F.scaled_dot_product_attention(qt, kt, vt).transpose(1, 2).reshape(B, H * W, C).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
