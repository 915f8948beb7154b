"""GPU parity of the attention variants (HNDL "attention" operator page:
bias flags, causal mask, rotary embedding, 2-D relative position bias; the
query-key RMS normalisation of vit-pytorch simple_vit_with_qk_norm) against
the fp64 oracle, through the C ABI (ssa_forward_ex / ssa_forward_planned_ex
and the step entry points).

Tolerances as for the block (branch relative L2 <= 1e-2, max |delta| of out
<= 5e-2).  The rotation fused into the projection's epilogue takes cos/sin of
angles formed and reduced in fp64 (exact to fp32 rounding at every position);
the separate rotation pass (with the query-key norm) builds its angles in fp32
as the page prescribes, off by at most ~1e-3 rad at 16383 * theta_0, well
inside the tolerance.  The oracle rotates exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_net_spatial_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS = 5e-2


@pytest.fixture(scope="module")
def ssa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_net_spatial_gb300 as m
    m.load_library()
    return m


def _inputs(B, C, H, W, G, h, dtype, seed):
    wl = wls.custom("variant", B=B, C=C, H=H, W=W, num_groups=G, num_heads=h, dtype=dtype, seed=seed)
    x, p, qidx = wls.make_inputs(wl)
    g = torch.Generator().manual_seed(seed + 99)
    rel = ((torch.rand((2 * H - 1) * (2 * W - 1), h, generator=g) * 2 - 1) * 1.5).to(x.dtype)
    d = C // h
    qg = (0.5 + torch.rand(h, d, generator=g)).to(x.dtype)
    kg = (0.5 + torch.rand(h, d, generator=g)).to(x.dtype)
    p["_qg"], p["_kg"] = qg, kg
    return wl, x, p, rel


def _check(ssa, out, x, p, wl, qidx=None, **kw):
    B, C = x.shape[:2]
    ref, y = oracle.block(x, p, wl.num_groups, wl.num_heads, qidx=qidx, **kw)
    got = out.double().cpu().numpy().reshape(B, C, -1)
    if qidx is not None:
        got = got[:, :, qidx]
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(y), 1e-30)
    mx = np.abs(got - ref).max()
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)
    return rel, mx


SHAPES = [
    # name, B, C, H, W, G, h, dtype           attention mode
    ("d64", 1, 128, 12, 20, 8, 2, "f32"),     # single, N = 240 (ragged)
    ("d40", 1, 80, 9, 15, 8, 2, "f32"),       # single, d = 40 -> 48, N = 135
    ("d320", 1, 320, 10, 10, 16, 1, "f32"),   # double (two 160-wide O halves)
    ("d512", 1, 512, 12, 25, 32, 1, "f32"),   # pair, N = 300 (three 128-key tiles, ragged)
    ("bf16-d64", 2, 256, 8, 12, 16, 4, "bf16"),
    ("d64-w32", 1, 128, 6, 32, 8, 2, "f32"),  # quad, W % 32 == 0: the table path; N = 192 (ragged tile)
    ("d40-w64", 1, 80, 3, 64, 8, 2, "f32"),   # quad with the ones column, W = 64
    ("d64-n320", 1, 128, 16, 20, 8, 2, "f32"),  # quad, 3 query tiles: the second CTA's second tile is past N
]
VARIANTS = ["no_bias", "causal", "rope", "rel", "causal_rel", "qk_norm", "qk_norm_rope", "all"]


def _kw(variant, rel, p):
    qn = variant in ("qk_norm", "qk_norm_rope", "all")
    return {"causal": variant in ("causal", "causal_rel", "all"), "rope": variant in ("rope", "qk_norm_rope", "all"),
            "rel_table": rel if variant in ("rel", "causal_rel", "all") else None,
            "q_norm_weight": p["_qg"] if qn else None, "k_norm_weight": p["_kg"] if qn else None}


@pytest.mark.parametrize("name,B,C,H,W,G,h,dt", SHAPES, ids=[s[0] for s in SHAPES])
@pytest.mark.parametrize("variant", VARIANTS)
def test_variant_parity(ssa, name, B, C, H, W, G, h, dt, variant):
    wl, x, p, rel = _inputs(B, C, H, W, G, h, dt, seed=B * 1000 + C + H)
    if variant in ("no_bias", "all"):
        for k in ("q_bias", "k_bias", "v_bias", "out_bias"):
            p[k] = None
    kw = _kw(variant, rel, p)
    p = {k: v for k, v in p.items() if not k.startswith("_")}
    xd = x.cuda()
    pd = {k: (None if v is None else v.cuda()) for k, v in p.items()}
    dev = {k: (None if v is None or isinstance(v, bool) else v.cuda()) for k, v in kw.items()}
    out = ssa.ssa_forward(xd, pd, G, h, causal=kw["causal"], rope=kw["rope"], rel_table=dev["rel_table"],
                          q_norm_weight=dev["q_norm_weight"], k_norm_weight=dev["k_norm_weight"])
    assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
    okw = {k: (v.double().numpy() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
    _check(ssa, out, x, p, wl, **okw)


def test_rope_pass_near_2_31_pairs(ssa):
    """The separate rotary pass (it follows the query-key norm) over
    B*h*N*d/2 = 65534 * 128 * 256 = 2,147,418,112 pairs: within 2^20 of 2^31,
    where a 32-bit grid-stride index would wrap.  x is drawn on the device;
    three samples against the oracle, all of out finite."""
    B, C, H, W, G, h = 32767, 1024, 8, 16, 1, 2
    free, _ = torch.cuda.mem_get_info()
    if free < (80 << 30):
        pytest.skip("needs ~70 GB of free device memory")
    wl, _, p, _ = _inputs(1, C, H, W, G, h, "f32", seed=47)
    qg, kg = p.pop("_qg"), p.pop("_kg")
    dev = torch.device("cuda:0")
    pd = {k: v.to(dev) for k, v in p.items()}
    gen = torch.Generator(device=dev).manual_seed(53)
    xd = torch.randn((B, C, H, W), generator=gen, device=dev, dtype=torch.float32)
    try:
        out = ssa.ssa_forward(xd, pd, G, h, rope=True, q_norm_weight=qg.to(dev), k_norm_weight=kg.to(dev))
        assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
        for b in (0, 20000, B - 1):
            xb = xd[b:b + 1].cpu()
            _check(ssa, out[b:b + 1], xb, p, wl, rope=True, q_norm_weight=qg.double().numpy(),
                   k_norm_weight=kg.double().numpy())
        assert bool(torch.isfinite(out).all())
    finally:
        del xd
        torch.cuda.empty_cache()


def test_planned_variants_match_one_shot(ssa):
    wl, x, p, rel = _inputs(2, 128, 10, 14, 8, 4, "f32", seed=5)
    qg, kg = p.pop("_qg").cuda(), p.pop("_kg").cuda()
    xd = x.cuda()
    pd = {k: v.cuda() for k, v in p.items()}
    plan = ssa.SsaPlan(pd, 8, 4)
    try:
        a = plan.forward(xd, causal=True, rope=True, rel_table=rel.cuda(), q_norm_weight=qg, k_norm_weight=kg)
        b = ssa.ssa_forward(xd, pd, 8, 4, causal=True, rope=True, rel_table=rel.cuda(), q_norm_weight=qg,
                            k_norm_weight=kg)
        assert ssa.ssa_get_device_status() == 0
        assert torch.equal(a, b)
    finally:
        plan.close()


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "no-mask"])
@pytest.mark.parametrize("name", ["unet-l1", "vae16384"])
def test_named_workload_causal_rel(ssa, name, causal):
    """The two largest workloads with a relative-position table over their
    full grids (64 x 64 with 8 heads; 128 x 128 with one head of 512), with
    and without the causal mask; the oracle evaluates a seeded sample of 128
    query pixels."""
    wl = wls.WORKLOADS[name]
    x, p, _ = wls.make_inputs(wl)
    g = torch.Generator().manual_seed(17)  # (the named workloads carry no QK-norm weights)
    rel = ((torch.rand((2 * wl.H - 1) * (2 * wl.W - 1), wl.num_heads, generator=g) * 2 - 1)).to(x.dtype)
    qidx = np.sort(torch.randperm(wl.N, generator=g)[:128].numpy())
    xd = x.cuda()
    pd = {k: v.cuda() for k, v in p.items()}
    out = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads, causal=causal, rel_table=rel.cuda())
    assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
    _check(ssa, out, x, p, wl, qidx=qidx, causal=causal, rel_table=rel.double().numpy())


def test_rope_step_against_oracle(ssa):
    """ssa_rope alone on the GPU's own Q/K against the oracle's rotation."""
    B, C, H, W, h = 1, 128, 16, 16, 2
    wl, x, p, _ = _inputs(B, C, H, W, 8, h, "f32", seed=3)
    p = {k: v for k, v in p.items() if not k.startswith("_")}
    xd = x.cuda()
    pd = {k: v.cuda() for k, v in p.items()}
    _, _, a, s = ssa.ssa_gn_stats(xd, 8, pd["norm_weight"], pd["norm_bias"])
    pk = ssa.ssa_pack_weights(pd, h)
    q, k, vt = ssa.ssa_qkv_project(xd, a, s, pk["w_qkv"], pk["b_qkv"], h)
    d = C // h
    q0 = q[..., :d].double().cpu().numpy().transpose(0, 2, 1, 3).reshape(B, H * W, C)
    ssa.ssa_rope(q, k, B, C, H * W, h)
    assert ssa.ssa_get_device_status() == 0
    q1 = q[..., :d].double().cpu().numpy().transpose(0, 2, 1, 3).reshape(B, H * W, C)
    ref = oracle.rope(q0, h)
    # fp16 storage of the rotated values: relative 2^-11 per element
    np.testing.assert_allclose(q1, ref, rtol=2e-3, atol=2e-3)


def test_qk_norm_step_against_oracle(ssa):
    """ssa_qk_norm alone on the GPU's own Q/K against the oracle's norm."""
    B, C, H, W, h = 1, 128, 8, 16, 4
    wl, x, p, _ = _inputs(B, C, H, W, 8, h, "bf16", seed=6)
    qg, kg = p.pop("_qg"), p.pop("_kg")
    xd = x.cuda()
    pd = {k: v.cuda() for k, v in p.items()}
    _, _, a, s = ssa.ssa_gn_stats(xd, 8, pd["norm_weight"], pd["norm_bias"])
    pk = ssa.ssa_pack_weights(pd, h)
    q, k, vt = ssa.ssa_qkv_project(xd, a, s, pk["w_qkv"], pk["b_qkv"], h)
    d = C // h
    k0 = k[..., :d].double().cpu().numpy().transpose(0, 2, 1, 3).reshape(B, H * W, C)
    ssa.ssa_qk_norm(q, k, B, C, H * W, h, qg.cuda(), kg.cuda())
    assert ssa.ssa_get_device_status() == 0
    k1 = k[..., :d].double().cpu().numpy().transpose(0, 2, 1, 3).reshape(B, H * W, C)
    ref = oracle.qk_norm(k0, h, kg.double().numpy())
    np.testing.assert_allclose(k1, ref, rtol=3e-3, atol=3e-3)


def test_rope_rejects_odd_head_dim(ssa):
    wl, x, p, _ = _inputs(1, 48, 4, 4, 4, 16, "f32", seed=4)  # d = 3
    p = {k: v for k, v in p.items() if not k.startswith("_")}
    with pytest.raises(ssa.SsaError) as e:
        ssa.ssa_forward(x.cuda(), {k: v.cuda() for k, v in p.items()}, 4, 16, rope=True)
    assert e.value.status == 1


ROPE_STEP_SHAPES = [
    # name, B, C, H, W, G, h, dtype        epilogue path of the fused rotation
    ("d32", 1, 64, 8, 8, 8, 2, "f32"),       # the tiny shape: 16-column chunks
    ("d48", 2, 96, 9, 16, 8, 2, "f32"),      # d = dp = 48: 16-column chunks, whole pairs
    ("d64", 2, 128, 12, 20, 8, 2, "f32"),    # 32-column chunks: shuffle-transposed stores
    ("d272", 1, 272, 6, 22, 16, 1, "f32"),   # d = 272 -> 288: a chunk of pure zero padding
    ("d512", 1, 512, 12, 25, 32, 1, "f32"),  # one head of 512 across four slices
    ("c768-d64-bf16", 2, 768, 8, 16, 32, 12, "bf16"),  # C > 512: staged 8-feature halves, TMA stores
]


@pytest.mark.parametrize("case", ROPE_STEP_SHAPES, ids=[c[0] for c in ROPE_STEP_SHAPES])
def test_qkv_project_rope_step_against_oracle(ssa, case):
    """The rotation fused into the projection's epilogue: Q at sampled pixels
    and K at every pixel against the oracle's rotated projections (exact
    angles in fp64); V as without the rotation."""
    name, B, C, H, W, G, h, dt = case
    wl, x, p, _ = _inputs(B, C, H, W, G, h, dt, seed=C + H)
    p = {k: v for k, v in p.items() if not k.startswith("_")}
    xd = x.cuda()
    pd = {k: v.cuda() for k, v in p.items()}
    _, _, a, s = ssa.ssa_gn_stats(xd, G, pd["norm_weight"], pd["norm_bias"])
    pk = ssa.ssa_pack_weights(pd, h)
    q, k, vt = ssa.ssa_qkv_project_rope(xd, a, s, pk["w_qkv"], pk["b_qkv"], h)
    assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
    N, d = H * W, C // h
    qi = np.arange(0, N, 7)
    r = oracle.forward(x, p, G, h, qidx=qi, want=("q", "k", "v"), rope=True)
    qg = q[..., :d].double().cpu().numpy().transpose(0, 2, 1, 3).reshape(B, N, C)[:, qi]
    kg = k[..., :d].double().cpu().numpy().transpose(0, 2, 1, 3).reshape(B, N, C)
    vg = vt[:, :, :d, :N].double().cpu().numpy().transpose(0, 3, 1, 2).reshape(B, N, C)
    for got, ref in ((qg, r["q"]), (kg, r["k"]), (vg, r["v"])):
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 3e-3
        np.testing.assert_allclose(got, ref, rtol=4e-3, atol=4e-3)
    dp = ssa.layout(B, C, H, W, h)["dp"]
    if d < dp:
        assert torch.count_nonzero(q[..., d:dp]) == 0 and torch.count_nonzero(k[..., d:dp]) == 0


def test_qkv_project_rope_rejects_plain_order_shapes(ssa):
    """Head dims that are not a multiple of 16 keep Q/K rows in plain order
    (the rotation then runs as its own pass): the fused entry point says so."""
    wl, x, p, _ = _inputs(1, 80, 8, 8, 8, 2, "f32", seed=9)   # d = 40
    p = {k: v for k, v in p.items() if not k.startswith("_")}
    xd = x.cuda()
    pd = {k: v.cuda() for k, v in p.items()}
    _, _, a, s = ssa.ssa_gn_stats(xd, 8, pd["norm_weight"], pd["norm_bias"])
    pk = ssa.ssa_pack_weights(pd, 2)
    with pytest.raises(ssa.SsaError) as e:
        ssa.ssa_qkv_project_rope(xd, a, s, pk["w_qkv"], pk["b_qkv"], 2)
    assert e.value.status == 4


@pytest.mark.parametrize("name", ["unet-lowres", "vae16384"])
def test_named_workload_rope_positions(ssa, name):
    """Fused rotation at every token position of the named grids whose head
    dims take it (the largest angle is 16383 rad at theta_0 = 1 on
    128 x 128): K against the oracle."""
    wl = wls.WORKLOADS[name]
    x, p, _ = wls.make_inputs(wl)
    xd = x.cuda()
    pd = {k: v.cuda() for k, v in p.items()}
    _, _, a, s = ssa.ssa_gn_stats(xd, wl.num_groups, pd["norm_weight"], pd["norm_bias"])
    pk = ssa.ssa_pack_weights(pd, wl.num_heads)
    q, k, vt = ssa.ssa_qkv_project_rope(xd, a, s, pk["w_qkv"], pk["b_qkv"], wl.num_heads)
    assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
    B, C, N, h = wl.B, wl.C, wl.N, wl.num_heads
    d = C // h
    r = oracle.forward(x, p, wl.num_groups, h, qidx=np.array([N - 1]), want=("k",), rope=True)
    kg = k[..., :d].double().cpu().numpy().transpose(0, 2, 1, 3).reshape(B, N, C)
    assert np.linalg.norm(kg - r["k"]) / np.linalg.norm(r["k"]) < 3e-3
    np.testing.assert_allclose(kg, r["k"], rtol=4e-3, atol=8e-3)
