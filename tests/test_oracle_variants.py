"""Pins for the oracle's attention variants (HNDL "attention" operator page:
parameter table, Biases, Masking, Relative position bias and Rotary
embeddings paragraphs; vit-pytorch simple_vit_with_qk_norm.py, RMSNorm
class), applied to the block's row-major token sequence.

Each variant is checked against something other than the oracle's own loops:
a torch library composition (F.linear without bias, SDPA with is_causal or an
additive attn_mask), the complex-number form of the rotation, closed forms
(the first token under the causal mask, position 0 under the rotation) and
invariances the pages state or the mathematics fixes (a zero or constant
bias table changes nothing; rotated scores depend only on the position
difference; one token is unaffected by the rotation).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _params(C, seed, scale=0.5):
    g = np.random.default_rng(seed)
    p = {"norm_weight": 1 + 0.3 * g.standard_normal(C), "norm_bias": 0.3 * g.standard_normal(C)}
    for k in ("q", "k", "v", "out"):
        p[f"{k}_weight"] = scale * g.standard_normal((C, C))
        p[f"{k}_bias"] = scale * g.standard_normal(C)
    return p


def _x(B, C, H, W, seed):
    return np.random.default_rng(seed + 1000).standard_normal((B, C, H, W))


def _rel_table(H, W, h, seed, scale=1.0):
    return scale * np.random.default_rng(seed + 7).standard_normal(((2 * H - 1) * (2 * W - 1), h))


def _rope_complex(u, pos, h):
    """Rotary embedding through complex arithmetic: pair (a_i, b_i) of each
    head (a = first half, b = second half) is the complex number a + i b,
    multiplied by exp(i * pos * 10000**(-2i/d)).  u: (..., N, C) torch fp64."""
    *lead, N, C = u.shape
    d = C // h
    x = u.reshape(*lead, N, h, 2, d // 2)
    z = torch.complex(x[..., 0, :], x[..., 1, :])
    i = torch.arange(d // 2, dtype=torch.float64)
    theta = torch.pow(torch.tensor(10000.0, dtype=torch.float64), -2.0 * i / d)
    ang = torch.as_tensor(pos, dtype=torch.float64).reshape(N, 1, 1) * theta
    z = z * torch.polar(torch.ones_like(ang), ang)
    return torch.stack((z.real, z.imag), dim=-2).reshape(*lead, N, C)


def _rel_bias(table, H, W, h):
    """[h, T, T] bias from the table by the page's index formula, built with
    torch index tensors."""
    t = torch.arange(H * W)
    r, c = t // W, t % W
    dy = r[:, None] - r[None, :] + (H - 1)
    dx = c[:, None] - c[None, :] + (W - 1)
    idx = dy * (2 * W - 1) + dx
    tab = torch.from_numpy(table)
    return tab[idx].permute(2, 0, 1)


def _torch_route(x, p, G, h, causal=False, rope=False, rel=None):
    """The block from torch library routines in fp64 with the variants: a
    missing bias is F.linear(..., None); the causal mask is SDPA's is_causal
    (or, with a bias, the summed additive mask the page describes); the
    rotation is the complex form above."""
    xt = torch.from_numpy(x)
    B, C, H, W = xt.shape
    t = {k: (None if v is None else torch.from_numpy(v)) for k, v in p.items()}
    gn = F.group_norm(xt, G, t["norm_weight"], t["norm_bias"], eps=1e-5)
    z = gn.flatten(2).transpose(1, 2)
    q = F.linear(z, t["q_weight"], t.get("q_bias"))
    k = F.linear(z, t["k_weight"], t.get("k_bias"))
    v = F.linear(z, t["v_weight"], t.get("v_bias"))
    N, d = H * W, C // h
    if rope:
        pos = torch.arange(N)
        q, k = _rope_complex(q, pos, h), _rope_complex(k, pos, h)
    q, k, v = (u.view(B, N, h, d).transpose(1, 2) for u in (q, k, v))
    if rel is None:
        o = F.scaled_dot_product_attention(q, k, v, is_causal=causal)
    else:
        mask = _rel_bias(rel, H, W, h)
        if causal:
            mask = mask + torch.triu(torch.full((N, N), float("-inf"), dtype=torch.float64), diagonal=1)
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask)
    o = o.transpose(1, 2).reshape(B, N, C)
    y = F.linear(o, t["out_weight"], t.get("out_bias"))
    return y.transpose(1, 2).reshape(B, C, H, W).numpy()


SHAPES = [
    # B, C, H, W, G, h
    (1, 4, 2, 2, 2, 2),
    (2, 8, 3, 5, 2, 2),
    (1, 12, 4, 3, 3, 3),
    (2, 8, 2, 7, 4, 1),
]


@pytest.mark.parametrize("B,C,H,W,G,h", SHAPES)
@pytest.mark.parametrize("variant", ["no_qkv_bias", "no_out_bias", "causal", "rope", "rel", "rel_causal",
                                     "all"])
def test_variants_match_torch_composition(B, C, H, W, G, h, variant):
    x = _x(B, C, H, W, seed=C + H)
    p = _params(C, seed=W + h)
    kw = {}
    if variant == "no_qkv_bias":
        p["q_bias"] = p["k_bias"] = p["v_bias"] = None
    if variant == "no_out_bias":
        p["out_bias"] = None
    if variant in ("causal", "rel_causal", "all"):
        kw["causal"] = True
    if variant in ("rope", "all"):
        kw["rope"] = True
    if variant in ("rel", "rel_causal", "all"):
        kw["rel"] = _rel_table(H, W, h, seed=B)
    y_ref = _torch_route(x, p, G, h, **kw)
    y = oracle.forward(x, p, G, h, causal=kw.get("causal", False), rope=kw.get("rope", False),
                       rel_table=kw.get("rel"))["y"]
    np.testing.assert_allclose(y.reshape(y_ref.shape), y_ref, rtol=1e-10, atol=1e-10)


def test_missing_bias_equals_zero_bias():
    """A projection without a bias (page: 'has no bias parameter at all') is
    the projection with a zero bias."""
    x, p = _x(2, 8, 3, 4, 1), _params(8, 2)
    q = dict(p)
    for k in ("q_bias", "k_bias", "v_bias", "out_bias"):
        q[k] = np.zeros(8)
    none = dict(p)
    for k in ("q_bias", "k_bias", "v_bias", "out_bias"):
        none[k] = None
    np.testing.assert_array_equal(oracle.forward(x, q, 2, 2)["y"], oracle.forward(x, none, 2, 2)["y"])


def test_causal_first_token_attends_to_itself_only():
    """Masking paragraph: position t attends only to positions <= t, so the
    first token's head outputs are its own value row exactly."""
    x, p = _x(1, 8, 3, 3, 3), _params(8, 4)
    r = oracle.forward(x, p, 2, 2, causal=True, want=("v", "o"))
    np.testing.assert_allclose(r["o"][0, 0], r["v"][0, 0], rtol=0, atol=1e-14)
    # and the last token sees every key: its output equals the unmasked one
    r0 = oracle.forward(x, p, 2, 2, want=("o",))
    np.testing.assert_allclose(r["o"][0, -1], r0["o"][0, -1], rtol=1e-12, atol=1e-12)


def test_causal_one_pixel_is_unmasked():
    x, p = _x(2, 4, 1, 1, 5), _params(4, 6)
    np.testing.assert_array_equal(oracle.forward(x, p, 2, 2, causal=True)["y"], oracle.forward(x, p, 2, 2)["y"])


def test_rope_one_token_is_identity():
    """Rotary paragraph: at T == 1 the only angle is zero, so the layer
    matches rope=False."""
    x, p = _x(2, 8, 1, 1, 7), _params(8, 8)
    np.testing.assert_allclose(oracle.forward(x, p, 4, 2, rope=True)["y"], oracle.forward(x, p, 4, 2)["y"],
                               rtol=0, atol=1e-14)


def test_rope_matches_complex_rotation_and_keeps_norms():
    g = np.random.default_rng(11)
    m = g.standard_normal((2, 9, 12))  # (batch, tokens, C), 3 heads of 4
    r = oracle.rope(m, 3)
    ref = _rope_complex(torch.from_numpy(m), torch.arange(9), 3).numpy()
    np.testing.assert_allclose(r, ref, rtol=1e-13, atol=1e-13)
    # position 0 is untouched; each rotated pair keeps its length
    np.testing.assert_array_equal(r[:, 0], m[:, 0])
    a, b = m.reshape(2, 9, 3, 2, 2), r.reshape(2, 9, 3, 2, 2)
    np.testing.assert_allclose((b ** 2).sum(axis=3), (a ** 2).sum(axis=3), rtol=1e-12)


def test_rope_scores_depend_on_position_difference_only():
    """Rotary paragraph: rotating by absolute position makes the scores
    depend on relative distance: <R(t1) q, R(t2) k> == <R(t1+s) q, R(t2+s) k>."""
    g = np.random.default_rng(12)
    q, k = g.standard_normal((1, 16)), g.standard_normal((1, 16))
    for t1, t2, s in [(3, 7, 5), (10, 2, 100), (0, 0, 31)]:
        a = (oracle.rope(q, 2, pos=[t1]) * oracle.rope(k, 2, pos=[t2])).reshape(2, 8).sum(axis=1)
        b = (oracle.rope(q, 2, pos=[t1 + s]) * oracle.rope(k, 2, pos=[t2 + s])).reshape(2, 8).sum(axis=1)
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-11)


def test_rope_rejects_odd_head_dim():
    x, p = _x(1, 6, 2, 2, 9), _params(6, 9)
    with pytest.raises(ValueError):
        oracle.forward(x, p, 2, 2, rope=True)  # d = 3


def test_rel_bias_zero_or_constant_table_changes_nothing():
    """Relative position paragraph: the table starts at 0.0, so the layer
    starts as ordinary attention; a constant table shifts every logit of a
    row equally, which the softmax ignores."""
    x, p = _x(1, 8, 3, 4, 13), _params(8, 14)
    base = oracle.forward(x, p, 2, 2)["y"]
    zero = np.zeros((5 * 7, 2))
    np.testing.assert_array_equal(oracle.forward(x, p, 2, 2, rel_table=zero)["y"], base)
    const = np.full((5 * 7, 2), 3.25)
    np.testing.assert_allclose(oracle.forward(x, p, 2, 2, rel_table=const)["y"], base, rtol=1e-12, atol=1e-12)


def test_rel_bias_brute_force_two_tokens():
    """A 1 x 2 grid by hand: offsets dx = c(q) - c(k) + 1 in {0, 1, 2}, table
    rows (dy = 0) 0..2; single head of width 1, identity-like projections."""
    # q = k = v = z (weights identity, no biases); d = 1, scale 1
    C = 1
    p = {"norm_weight": np.ones(1), "norm_bias": np.zeros(1), "q_weight": np.eye(1), "q_bias": None,
         "k_weight": np.eye(1), "k_bias": None, "v_weight": np.eye(1), "v_bias": None,
         "out_weight": np.eye(1), "out_bias": None}
    x = np.array([[[[0.0, 2.0]]]])
    table = np.array([[0.7], [-0.2], [1.5]])  # dx = 0, 1, 2
    y = oracle.forward(x, p, 1, 1, rel_table=table, want=("z",))
    z = y["z"][0, :, 0]  # normalised tokens: (-1, 1) up to eps
    out = []
    for tq in range(2):
        s = [z[tq] * z[tk] + table[tq - tk + 1, 0] for tk in range(2)]
        w = np.exp(np.array(s) - max(s))
        out.append(float((w / w.sum()) @ z))
    np.testing.assert_allclose(y["y"][0, 0], out, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------ query-key RMS norm ---
# vit-pytorch simple_vit_with_qk_norm.py, RMSNorm class: F.normalize over the
# head dim, times sqrt(d) and a learned gamma per head and dimension.

def _gammas(h, d, seed):
    g = np.random.default_rng(seed + 31)
    return 0.5 + g.random((h, d)), 0.5 + g.random((h, d))


def _torch_qk_route(x, p, G, h, qg, kg, rope=False, causal=False):
    xt = torch.from_numpy(x)
    B, C, H, W = xt.shape
    t = {k: torch.from_numpy(v) for k, v in p.items()}
    gn = F.group_norm(xt, G, t["norm_weight"], t["norm_bias"], eps=1e-5)
    z = gn.flatten(2).transpose(1, 2)
    N, d = H * W, C // h
    q = F.linear(z, t["q_weight"], t["q_bias"]).view(B, N, h, d).transpose(1, 2)
    k = F.linear(z, t["k_weight"], t["k_bias"]).view(B, N, h, d).transpose(1, 2)
    v = F.linear(z, t["v_weight"], t["v_bias"]).view(B, N, h, d).transpose(1, 2)
    q = F.normalize(q, dim=-1) * math.sqrt(d) * torch.from_numpy(qg)[None, :, None, :]
    k = F.normalize(k, dim=-1) * math.sqrt(d) * torch.from_numpy(kg)[None, :, None, :]
    if rope:
        pos = torch.arange(N)
        q = _rope_complex(q.transpose(1, 2).reshape(B, N, C), pos, h).view(B, N, h, d).transpose(1, 2)
        k = _rope_complex(k.transpose(1, 2).reshape(B, N, C), pos, h).view(B, N, h, d).transpose(1, 2)
    o = F.scaled_dot_product_attention(q, k, v, is_causal=causal).transpose(1, 2).reshape(B, N, C)
    y = F.linear(o, t["out_weight"], t["out_bias"])
    return y.transpose(1, 2).reshape(B, C, H, W).numpy()


@pytest.mark.parametrize("B,C,H,W,G,h", SHAPES)
@pytest.mark.parametrize("rope,causal", [(False, False), (True, False), (True, True)])
def test_qk_norm_matches_torch_composition(B, C, H, W, G, h, rope, causal):
    if rope and (C // h) % 2:
        pytest.skip("odd head dim")
    x, p = _x(B, C, H, W, seed=C + W), _params(C, seed=H + h)
    qg, kg = _gammas(h, C // h, seed=B + C)
    y_ref = _torch_qk_route(x, p, G, h, qg, kg, rope=rope, causal=causal)
    y = oracle.forward(x, p, G, h, q_norm_weight=qg, k_norm_weight=kg, rope=rope, causal=causal)["y"]
    np.testing.assert_allclose(y.reshape(y_ref.shape), y_ref, rtol=1e-10, atol=1e-10)


def test_qk_norm_is_invariant_to_projection_scale():
    """Normalising Q and K per head removes any positive scale of their
    projections: scaling Wq, bq by 3 and Wk, bk by 0.25 leaves the block
    unchanged (and it does change it without the norm)."""
    x, p = _x(2, 8, 3, 4, 21), _params(8, 22)
    qg, kg = _gammas(2, 4, 23)
    s = dict(p)
    s["q_weight"], s["q_bias"] = 3 * p["q_weight"], 3 * p["q_bias"]
    s["k_weight"], s["k_bias"] = 0.25 * p["k_weight"], 0.25 * p["k_bias"]
    a = oracle.forward(x, p, 2, 2, q_norm_weight=qg, k_norm_weight=kg)["y"]
    b = oracle.forward(x, s, 2, 2, q_norm_weight=qg, k_norm_weight=kg)["y"]
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-11)
    assert np.abs(oracle.forward(x, p, 2, 2)["y"] - oracle.forward(x, s, 2, 2)["y"]).max() > 1e-3


def test_qk_norm_rows_have_rms_gamma():
    """With gamma = 1/sqrt(d) (the vit-pytorch initialisation) every head row
    of the normalised Q has unit length; with gamma = 1 its RMS is 1."""
    g = np.random.default_rng(24)
    m = g.standard_normal((5, 12))
    u = oracle.qk_norm(m, 3, np.full((3, 4), 1 / 2.0)).reshape(5, 3, 4)
    np.testing.assert_allclose(np.linalg.norm(u, axis=-1), 1.0, rtol=1e-13)
    r = oracle.qk_norm(m, 3, np.ones((3, 4))).reshape(5, 3, 4)
    np.testing.assert_allclose(np.sqrt((r ** 2).mean(axis=-1)), 1.0, rtol=1e-13)


# ------------------------------------------------ query-sampled mode + variants ---
# The largest workload is checked on sampled query pixels, so the sampled mode
# must give the same rows as the full block under every variant: the causal
# mask and the table index use the query's token position (not its row in the
# sample), and the rotation turns the sampled Q rows by their own positions.

SAMPLES = [
    np.array([0, 3, 7, 19]),        # sorted, skipping positions
    np.array([19, 7, 3, 0]),        # reversed: row t is not position t
    np.array([13, 2, 18, 6, 11]),   # scattered
]


def _sampled_kwargs(variant, H, W, h, d):
    qg, kg = _gammas(h, d, seed=H * W)
    table = _rel_table(H, W, h, seed=5)
    kw = {
        "causal": dict(causal=True),
        "rope": dict(rope=True),
        "rel": dict(rel_table=table),
        "qk_norm": dict(q_norm_weight=qg, k_norm_weight=kg),
        "all": dict(causal=True, rope=True, rel_table=table, q_norm_weight=qg, k_norm_weight=kg),
    }
    return kw[variant]


@pytest.mark.parametrize("variant", ["causal", "rope", "rel", "qk_norm", "all"])
@pytest.mark.parametrize("qi", SAMPLES, ids=["sorted", "reversed", "scattered"])
def test_query_sampled_variants_equal_full_mode(variant, qi):
    """Sampled rows equal the full block's rows bit for bit, for each variant
    and all of them together, on a non-square grid (4 x 5)."""
    B, C, H, W, G, h = 2, 8, 4, 5, 4, 2
    x, p = _x(B, C, H, W, 61), _params(C, 62)
    kw = _sampled_kwargs(variant, H, W, h, C // h)
    full = oracle.forward(x, p, G, h, want=("q", "o"), **kw)
    part = oracle.forward(x, p, G, h, qidx=qi, want=("q", "o"), **kw)
    np.testing.assert_array_equal(part["y"], full["y"][:, :, qi])
    np.testing.assert_array_equal(part["q"], full["q"][:, qi])
    np.testing.assert_array_equal(part["o"], full["o"][:, qi])


@pytest.mark.parametrize("variant", ["causal", "rope", "rel", "rel_causal_rope", "qk_norm_rope_causal"])
def test_query_sampled_variants_match_torch_composition(variant):
    """The sampled rows against the torch library routes at the same pixels
    (reversed sample, so a slip from token position to sample row shows)."""
    B, C, H, W, G, h = 2, 8, 4, 5, 4, 2
    x, p = _x(B, C, H, W, 63), _params(C, 64)
    qi = SAMPLES[1]
    if variant.startswith("qk_norm"):
        qg, kg = _gammas(h, C // h, seed=65)
        y_ref = _torch_qk_route(x, p, G, h, qg, kg, rope=True, causal=True)
        kw = dict(q_norm_weight=qg, k_norm_weight=kg, rope=True, causal=True)
    else:
        table = _rel_table(H, W, h, seed=66) if variant.startswith("rel") else None
        causal = "causal" in variant
        rope = "rope" in variant
        y_ref = _torch_route(x, p, G, h, causal=causal, rope=rope, rel=table)
        kw = dict(causal=causal, rope=rope, rel_table=table)
    y = oracle.forward(x, p, G, h, qidx=qi, **kw)["y"]
    np.testing.assert_allclose(y, y_ref.reshape(B, C, H * W)[:, :, qi], rtol=1e-10, atol=1e-10)
