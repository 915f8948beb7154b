"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (block definition on the tensortonic page
"diffusion-l03-spatial-self-attention"; the target accuracy of fp16 tensor-core
operands with fp32 accumulation and fp32 softmax statistics):
  * branch out - x:  relative L2 error <= 1e-2
  * out:             max |delta| <= 5e-2
Per-step checks use the oracle's steps on the GPU's own inputs to that step.
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


def _to_dev(x, p):
    dev = torch.device("cuda:0")
    return x.to(dev), {k: v.to(dev) for k, v in p.items()}


def _compare(out_gpu, x, p, wl, qidx=None):
    """Returns (rel_l2_branch, max_abs_out) against the oracle.

    Both sides return the block in x's dtype (the return rule), so the branch
    is compared as out - x of the two returned tensors: the GPU's out against
    the oracle's exact result rounded once to x's dtype, normalised by the
    exact branch."""
    ref, y = oracle.block(x, p, wl.num_groups, wl.num_heads, qidx=None if qidx is None else qidx.numpy())
    B, C = x.shape[:2]
    got = out_gpu.double().cpu().numpy().reshape(B, C, -1)
    if qidx is not None:
        got = got[:, :, qidx.numpy()]
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(y), 1e-30)
    mx = np.abs(got - ref).max()
    return rel, mx


def _run(ssa, wl, inplace=False):
    x, p, qidx = wls.make_inputs(wl)
    xd, pd = _to_dev(x, p)
    if inplace:
        out = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads, out=xd)
    else:
        out = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads)
    st = ssa.ssa_get_device_status()
    assert st == 0, ssa.ssa_last_error_string()
    assert out.dtype == x.dtype and out.shape == x.shape
    return _compare(out, x, p, wl, qidx)


SMALL = [
    # name, B, C, H, W, G, h, dtype
    ("ragged-d64", 2, 128, 12, 20, 8, 2, "f32"),       # N = 240: one full 128 tile + ragged tail
    ("ragged-d40", 1, 80, 9, 15, 8, 2, "f32"),         # d = 40 -> padded to 48; N = 135
    ("ragged-d512", 1, 512, 10, 13, 32, 1, "f32"),     # d = 512 (score + output CTA pairs); N = 130
    ("d512-split3", 2, 512, 16, 24, 32, 1, "f32"),     # N = 384: every query tile shared by three SM pairs
    ("d496", 1, 496, 10, 13, 16, 1, "f32"),            # d = 496 padded to 512: the last 16 columns unwritten
    ("d500-b2", 2, 500, 9, 14, 20, 1, "f32"),          # d = 500 (not a multiple of 8): element stores
    ("d16-multihead", 2, 64, 5, 7, 4, 4, "f32"),       # N = 35 (not a multiple of 4: padded-x path)
    ("bf16-d64", 2, 256, 8, 12, 16, 4, "bf16"),
    ("bf16-n35", 2, 128, 5, 7, 8, 2, "bf16"),         # bf16 x, N = 35: 70-byte rows, the padded-x path
    ("single-pixel", 3, 64, 1, 1, 64, 2, "f32"),       # H = W = 1, one channel per group
    ("group1-head1", 1, 96, 6, 6, 1, 1, "f32"),        # one group, one head (d = 96)
    ("d32-multitile", 1, 64, 16, 24, 8, 2, "f32"),     # N = 384: three key tiles
    ("d128", 1, 256, 16, 16, 8, 2, "f32"),
    ("d256", 1, 256, 12, 12, 8, 1, "f32"),
    ("d320", 1, 320, 9, 9, 8, 1, "f32"),               # dp = 320 -> two 160-wide halves
    ("ex1-shape", 1, 4, 2, 2, 2, 2, "f32"),            # worked example 1's shape (d = 2)
    ("ex2-shape", 1, 2, 2, 3, 1, 1, "f32"),            # worked example 2's shape (H != W)
    ("ex3-shape", 2, 4, 1, 1, 4, 2, "f32"),            # worked example 3's shape
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_block_small_shapes(ssa, case):
    name, B, C, H, W, G, h, dt = case
    wl = wls.custom(name, B, C, H, W, G, h, dt, seed=11)
    rel, mx = _run(ssa, wl)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


@pytest.mark.parametrize("name", list(wls.WORKLOADS))
def test_block_named_workloads(ssa, name):
    """The five named shapes at full size; the largest is checked on its 512
    seeded query pixels (every key), the others on every pixel."""
    rel, mx = _run(ssa, wls.WORKLOADS[name])
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


def test_block_past_2_31_elements(ssa):
    """B*C*N = 32767 * 1024 * 72 = 2.4e9 elements (> 2^31), a shape the shape
    checks admit (B*h = 65534 head tiles): every kernel's offsets past 32 bits,
    the general projection (C > 512) and the split d = 512 attention.  x is
    drawn on the device; three samples against the oracle, all of out finite."""
    B, C, H, W, G, h = 32767, 1024, 8, 9, 1, 2
    free, _ = torch.cuda.mem_get_info()
    if free < (48 << 30):
        pytest.skip("needs ~45 GB of free device memory")
    _, p, _ = wls.make_inputs(wls.custom("big", 1, C, H, W, G, h, "f32", seed=41))
    dev = torch.device("cuda:0")
    pd = {k: v.to(dev) for k, v in p.items()}
    gen = torch.Generator(device=dev).manual_seed(43)
    xd = torch.randn((B, C, H, W), generator=gen, device=dev, dtype=torch.float32)
    plan = ssa.SsaPlan(pd, G, h)
    try:
        out = plan.forward(xd)
        assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
        for b in (0, 12345, B - 1):
            xb = xd[b:b + 1].cpu()
            ref, y = oracle.block(xb, p, G, h)
            got = out[b:b + 1].double().cpu().numpy().reshape(1, C, -1)
            rel = np.linalg.norm(got - ref) / max(np.linalg.norm(y), 1e-30)
            mx = np.abs(got - ref).max()
            assert rel <= REL_L2 and mx <= MAX_ABS, (b, rel, mx)
        assert bool(torch.isfinite(out).all())
    finally:
        plan.close()
        del xd
        torch.cuda.empty_cache()


def test_empty_problems(ssa):
    """B, H or W zero: no work and no error, through the one-shot, planned and
    step entry points; the output is the empty tensor of x's shape."""
    wl = wls.WORKLOADS["tiny"]
    _, p, _ = wls.make_inputs(wl)
    pd = {k: v.cuda() for k, v in p.items()}
    plan = ssa.SsaPlan(pd, wl.num_groups, wl.num_heads)
    try:
        for shape in ((0, 64, 8, 8), (2, 64, 0, 8), (2, 64, 8, 0)):
            xd = torch.empty(shape, device="cuda")
            out = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads)
            assert out.shape == xd.shape
            out = plan.forward(xd, causal=True, rope=True)
            assert out.shape == xd.shape
            assert ssa.ssa_get_device_status() == 0
    finally:
        plan.close()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_in_place(ssa, dt):
    wl = wls.custom("inplace", 2, 128, 8, 16, 8, 2, dt, seed=5)
    rel, mx = _run(ssa, wl, inplace=True)
    assert rel <= REL_L2 and mx <= MAX_ABS


def test_planned_matches_one_shot_bitwise(ssa):
    wl = wls.custom("plan", 2, 320, 16, 16, 32, 8, "f32", seed=6)
    x, p, _ = wls.make_inputs(wl)
    xd, pd = _to_dev(x, p)
    a = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads)
    plan = ssa.SsaPlan(pd, wl.num_groups, wl.num_heads)
    b = plan.forward(xd)
    c = plan.forward(xd)
    assert ssa.ssa_get_device_status() == 0
    assert torch.equal(a, b) and torch.equal(b, c)
    plan.close()


@pytest.mark.parametrize("name", ["unet-l1", "vae1024", "unet-lowres"])
def test_planned_forward_in_a_cuda_graph(ssa, name):
    """With its output and workspace given, a planned forward issues only
    stream-ordered work (no host synchronisation, no allocation), so it can be
    captured into a CUDA graph; every replay matches a direct call bit for bit.
    unet-l1 runs the quad attention mode, vae1024 the pair mode with its work
    split (a counter memset in the graph), unet-lowres bf16 x."""
    wl = wls.WORKLOADS[name]
    x, p, _ = wls.make_inputs(wl)
    xd, pd = _to_dev(x, p)
    plan = ssa.SsaPlan(pd, wl.num_groups, wl.num_heads)
    ws = torch.empty(plan.workspace_size(wl.B, wl.H, wl.W), dtype=torch.uint8, device=xd.device)
    ref = plan.forward(xd, workspace=ws)
    assert ssa.ssa_get_device_status() == 0
    out = torch.empty_like(xd)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.forward(xd, out=out, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.forward(xd, out=out, workspace=ws, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
        assert torch.equal(out, ref)
    del g
    plan.close()


def test_two_plans_on_two_streams(ssa):
    """Plans share no device state but the status word: two shapes (quad-mode
    unet-l1, split pair-mode vae1024) run concurrently on two streams, several
    times over, give exactly their results run alone."""
    runs = []
    for name in ("unet-l1", "vae1024"):
        wl = wls.WORKLOADS[name]
        x, p, _ = wls.make_inputs(wl)
        xd, pd = _to_dev(x, p)
        plan = ssa.SsaPlan(pd, wl.num_groups, wl.num_heads)
        ws = torch.empty(plan.workspace_size(wl.B, wl.H, wl.W), dtype=torch.uint8, device=xd.device)
        ref = plan.forward(xd, workspace=ws)
        runs.append((plan, xd, ws, ref, torch.cuda.Stream()))
    torch.cuda.synchronize()
    assert ssa.ssa_get_device_status() == 0
    outs = [torch.empty_like(r[1]) for r in runs]
    for _ in range(4):
        for (plan, xd, ws, _, st), out in zip(runs, outs):
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                out.zero_()
                plan.forward(xd, out=out, workspace=ws, stream=st)
        torch.cuda.synchronize()
        assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
        for (_, _, _, ref, _), out in zip(runs, outs):
            assert torch.equal(out, ref)
    for r in runs:
        r[0].close()


def test_gn_stats_step(ssa):
    """GN statistics kernel against the oracle's two-pass fp64 statistics."""
    for (B, C, H, W, G, dt, shift) in [(2, 320, 64, 64, 32, "f32", 0.0), (1, 512, 128, 128, 32, "f32", 3.0),
                                        (8, 1280, 16, 16, 32, "bf16", 0.0), (3, 12, 5, 3, 4, "f32", -7.0)]:
        wl = wls.custom("gn", B, C, H, W, G, 1, dt, seed=B + C, x_scale=2.0)
        x, p, _ = wls.make_inputs(wl)
        x = (x.float() + shift).to(x.dtype)
        xd, pd = _to_dev(x, p)
        mean, rstd, a, s = ssa.ssa_gn_stats(xd, G, pd["norm_weight"], pd["norm_bias"])
        assert ssa.ssa_get_device_status() == 0
        m_ref, r_ref = oracle.gn_stats(x, G)
        np.testing.assert_allclose(mean.cpu().double().numpy(), m_ref, rtol=1e-5, atol=1e-5 * (1 + abs(shift)))
        np.testing.assert_allclose(rstd.cpu().double().numpy(), r_ref, rtol=2e-5)
        gw = p["norm_weight"].double().numpy()
        gb = p["norm_bias"].double().numpy()
        cg = C // G
        a_ref = np.repeat(r_ref, cg, axis=1) * gw
        s_ref = gb - np.repeat(m_ref, cg, axis=1) * a_ref
        np.testing.assert_allclose(a.cpu().double().numpy(), a_ref, rtol=2e-5)
        np.testing.assert_allclose(s.cpu().double().numpy(), s_ref, rtol=2e-5, atol=2e-5 * (1 + abs(shift)))


def _step_inputs(ssa, wl):
    x, p, _ = wls.make_inputs(wl)
    xd, pd = _to_dev(x, p)
    _, _, a, s = ssa.ssa_gn_stats(xd, wl.num_groups, pd["norm_weight"], pd["norm_bias"])
    packed = ssa.ssa_pack_weights(pd, wl.num_heads)
    return x, p, xd, pd, a, s, packed


STEP_SHAPES = [("d64", 2, 128, 12, 20, 8, 2, "f32"), ("d40", 1, 80, 16, 8, 8, 2, "f32"),
               ("d512", 1, 512, 8, 32, 32, 1, "f32"), ("bf16", 2, 256, 8, 8, 16, 4, "bf16"),
               # C > 512: the general projection (fp32 x: four 32-pixel x boxes per stage) and
               # out-projection kernels; N = 208 leaves a ragged second pixel tile
               ("c640-f32", 2, 640, 13, 16, 32, 10, "f32"),
               ("c1280-bf16", 1, 1280, 12, 12, 32, 20, "bf16"),
               # C = 544: the last 64-channel k-block is half past C (zero-filled x, zero scale)
               ("c544-f32", 1, 544, 9, 12, 32, 8, "f32")]


@pytest.mark.parametrize("case", STEP_SHAPES, ids=[c[0] for c in STEP_SHAPES])
def test_qkv_attention_outproj_steps(ssa, case):
    name, B, C, H, W, G, h, dt = case
    wl = wls.custom(name, B, C, H, W, G, h, dt, seed=21)
    x, p, xd, pd, a, s, pk = _step_inputs(ssa, wl)
    N, d = H * W, C // h
    q, k, vt = ssa.ssa_qkv_project(xd, a, s, pk["w_qkv"], pk["b_qkv"], h)
    assert ssa.ssa_get_device_status() == 0
    r = oracle.forward(x, p, G, h, want=("q", "k", "v", "o"))
    # Q/K/V against the oracle's projections
    qg = q[..., :d].double().cpu().numpy().transpose(0, 2, 1, 3).reshape(B, N, C)
    kg = k[..., :d].double().cpu().numpy().transpose(0, 2, 1, 3).reshape(B, N, C)
    vg = vt[:, :, :d, :N].double().cpu().numpy().transpose(0, 3, 1, 2).reshape(B, N, C)
    for got, ref in ((qg, r["q"]), (kg, r["k"]), (vg, r["v"])):
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 3e-3
    # padded columns of Q and K are exactly zero
    if d < q.shape[-1]:
        dp = ssa.layout(B, C, H, W, h)["dp"]
        assert torch.count_nonzero(q[..., d:dp]) == 0 and torch.count_nonzero(k[..., d:dp]) == 0
    # attention on the GPU's own Q/K/V against the oracle's attention step
    o = ssa.ssa_attention(q, k, vt, B, C, N, h)
    assert ssa.ssa_get_device_status() == 0
    o_ref = oracle.attention(qg, kg, vg, h)
    og = o[..., :C].double().cpu().numpy()
    assert np.linalg.norm(og - o_ref) / np.linalg.norm(o_ref) < 3e-3
    assert np.abs(og - o_ref).max() < 2e-2
    # out-projection on the GPU's own O against the oracle's projection step
    out = ssa.ssa_out_project(o, pk["w_o"], pk["b_o"], xd)
    assert ssa.ssa_get_device_status() == 0
    y_ref = oracle.out_proj(og, p["out_weight"], p["out_bias"])
    xs = x.double().numpy().reshape(B, C, N)
    out_ref = oracle.round_to(xs + y_ref, dt)
    out_ref = oracle.bf16_bits_to_f64(out_ref) if dt == "bf16" else out_ref.astype(np.float64)
    got = out.double().cpu().numpy().reshape(B, C, N)
    assert np.linalg.norm(got - out_ref) / np.linalg.norm(y_ref) < 2e-3


# The resident out-projection (C <= 512, at least 64 pixel tiles): one CTA per
# 128-pixel tile; once its MMAs are done it streams the residual through as many
# 128-channel buffers as the freed shared memory holds.  C = 512 fp32 takes three
# (the fourth piece reloads the first buffer), bf16 four, C = 384 fp32 three.
OUTPROJ_RESIDENT = [("c512-f32", 1, 512, 64, 128, "f32"),
                    ("c512-bf16", 1, 512, 64, 128, "bf16"),
                    ("c384-f32-b2", 2, 384, 64, 64, "f32"),
                    ("c512-f32-ragged", 1, 512, 90, 92, "f32")]   # 65 tiles, the last one 88 pixels


@pytest.mark.parametrize("case", OUTPROJ_RESIDENT, ids=[c[0] for c in OUTPROJ_RESIDENT])
def test_out_projection_resident(ssa, case):
    """The out-projection step alone, on a seeded O in [-1, 1), against the
    oracle's projection plus residual."""
    name, B, C, H, W, dt = case
    h = C // 64
    wl = wls.custom(name, B, C, H, W, 32, h, dt, seed=31)
    x, p, _ = wls.make_inputs(wl)
    xd, pd = _to_dev(x, p)
    pk = ssa.ssa_pack_weights(pd, h)
    N, ldc = H * W, ssa.layout(B, C, H, W, h)["ldc"]
    g = torch.Generator().manual_seed(37)
    o_cpu = (torch.rand(B, N, ldc, generator=g) * 2 - 1).to(torch.float16)
    out = ssa.ssa_out_project(o_cpu.to(xd.device), pk["w_o"], pk["b_o"], xd)
    assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
    og = o_cpu[..., :C].double().numpy()
    y_ref = oracle.out_proj(og, p["out_weight"], p["out_bias"])
    xs = x.double().numpy().reshape(B, C, N)
    out_ref = oracle.round_to(xs + y_ref, dt)
    out_ref = oracle.bf16_bits_to_f64(out_ref) if dt == "bf16" else out_ref.astype(np.float64)
    got = out.double().cpu().numpy().reshape(B, C, N)
    assert np.linalg.norm(got - out_ref) / np.linalg.norm(y_ref) < 2e-3
    assert np.abs(got - out_ref).max() < 5e-2


def test_timeout_path_returns_status_and_context_survives(ssa):
    """A wait that nothing ends expires after its limit, latches
    SSA_ERR_TIMEOUT, and the context stays usable."""
    ssa.ssa_debug_timeout_probe(2_000_000)   # 2 ms limit
    assert ssa.ssa_get_device_status() == 7
    assert ssa.ssa_get_device_status() == 0  # read-and-clear
    rel, mx = _run(ssa, wls.WORKLOADS["tiny"])
    assert rel <= REL_L2 and mx <= MAX_ABS


def test_argument_errors(ssa):
    wl = wls.WORKLOADS["tiny"]
    x, p, _ = wls.make_inputs(wl)
    xd, pd = _to_dev(x, p)
    with pytest.raises(ssa.SsaError) as e:
        ssa.ssa_forward(xd, pd, 7, 2)          # 7 does not divide 64
    assert e.value.status == 1
    with pytest.raises(ssa.SsaError) as e:
        ssa.ssa_forward(xd, pd, 8, 3)          # 3 does not divide 64
    assert e.value.status == 1
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(ssa.SsaError) as e:
        ssa.ssa_forward(xd, pd, 8, 2, workspace=ws)
    assert e.value.status == 5
    with pytest.raises(ssa.SsaError) as e:
        ssa.ssa_forward(xd.double(), {k: v.double() for k, v in pd.items()}, 8, 2)
    assert e.value.status == 2


# ---------------------------------------------------------------------------
# Head dim 512: query tiles split between SM pairs (ssa_set_attention_split).
# The split merges fp32 parts rescaled to a common row maximum, which equals
# the unsplit online softmax up to rounding; both schedules are checked
# against the oracle on shapes where every query tile is shared by several
# clusters (ALWAYS) and where none is (NEVER).

@pytest.fixture
def split_policy(ssa):
    yield
    ssa.set_attention_split(ssa.SPLIT_AUTO)


SPLIT_CASES = [
    # name, B, C, H, W, G, h
    ("n300", 1, 512, 12, 25, 32, 1),     # 3 query tiles x 3 key tiles, ragged last tile
    ("b2-n384", 2, 512, 16, 24, 32, 1),  # 6 query tiles over 2 samples
    ("d496", 1, 496, 10, 13, 16, 1),     # padded head dim, 2 query tiles
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
@pytest.mark.parametrize("policy", ["always", "never"])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_pair_split_policies(ssa, split_policy, case, policy, causal):
    name, B, C, H, W, G, h = case
    ssa.set_attention_split(ssa.SPLIT_ALWAYS if policy == "always" else ssa.SPLIT_NEVER)
    wl = wls.custom(name, B, C, H, W, G, h, "f32", seed=21)
    x, p, _ = wls.make_inputs(wl)
    xd, pd = _to_dev(x, p)
    out = ssa.ssa_forward(xd, pd, G, h, causal=causal)
    assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
    ref, y = oracle.block(x, p, G, h, causal=causal)
    got = out.double().cpu().numpy().reshape(B, C, -1)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(y), 1e-30)
    mx = np.abs(got - ref).max()
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)


def test_pair_split_matches_whole_tiles(ssa, split_policy):
    """The split and the whole-tile schedules agree to rounding on the same
    inputs, and the attention step with scratch equals the planned block's."""
    wl = wls.custom("split-eq", 1, 512, 16, 32, 32, 1, "f32", seed=22)  # 4 query tiles x 4 key tiles
    x, p, _ = wls.make_inputs(wl)
    xd, pd = _to_dev(x, p)
    ssa.set_attention_split(ssa.SPLIT_ALWAYS)
    a = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads)
    ssa.set_attention_split(ssa.SPLIT_NEVER)
    b = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads)
    assert ssa.ssa_get_device_status() == 0
    d = (a.double() - b.double()).abs().max().item()
    assert d <= 2e-3, d
    # step API with and without scratch
    _, _, ga, gs = ssa.ssa_gn_stats(xd, wl.num_groups, pd["norm_weight"], pd["norm_bias"])
    pk = ssa.ssa_pack_weights(pd, wl.num_heads)
    q, k, vt = ssa.ssa_qkv_project(xd, ga, gs, pk["w_qkv"], pk["b_qkv"], wl.num_heads)
    nbytes = ssa.attention_workspace_size(wl.B, wl.C, wl.H, wl.W, wl.num_heads)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ssa.set_attention_split(ssa.SPLIT_ALWAYS)
    o1 = ssa.ssa_attention_ex(q, k, vt, wl.B, wl.C, wl.H, wl.W, wl.num_heads, workspace=ws)
    o2 = ssa.ssa_attention_ex(q, k, vt, wl.B, wl.C, wl.H, wl.W, wl.num_heads)
    assert ssa.ssa_get_device_status() == 0
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-3
    with pytest.raises(ssa.SsaError) as e:
        ssa.ssa_attention_ex(q, k, vt, wl.B, wl.C, wl.H, wl.W, wl.num_heads, workspace=ws[: nbytes // 2])
    assert e.value.status == 5
    with pytest.raises(ssa.SsaError) as e:
        ssa.set_attention_split(7)
    assert e.value.status == 1


ABORT_CASES = [
    # name, B, C, H, W, G, h, dtype, kernel whose producer stalls
    ("qkv-resident", 2, 320, 32, 32, 32, 8, "f32", 1),       # resident QKV (C <= 512), both producer warps
    ("qkv-general", 2, 768, 8, 16, 32, 12, "bf16", 1),       # QKV for C > 512
    ("attention-quad", 2, 320, 32, 32, 32, 8, "f32", 2),     # quad mode (head dim <= 64), d = 40
    ("attention-single", 1, 256, 32, 32, 32, 2, "f32", 2),   # single mode (two CTAs per SM), d = 128
    ("attention-double", 1, 320, 16, 16, 16, 1, "f32", 2),   # double mode (two O halves), d = 320
    ("out-proj-resident", 5, 256, 48, 48, 32, 4, "f32", 4),  # resident out-projection (C <= 512, 90 tiles)
    ("out-proj-halves", 2, 320, 64, 64, 32, 8, "f32", 4),    # 64 tiles: two CTAs per tile, half the channels each
    ("out-proj-small", 2, 320, 32, 32, 32, 8, "f32", 4),     # out-projection, one tile per CTA (16 tiles)
    ("out-proj-general", 2, 768, 8, 16, 32, 12, "bf16", 4),  # out-projection for C > 512
]


@pytest.mark.parametrize("case", ABORT_CASES, ids=[c[0] for c in ABORT_CASES])
def test_stalled_producer_times_out_and_context_survives(ssa, case):
    """The timeout path of the block's own kernels, without a fault: the test
    hook stops one kernel's TMA producer after a few loads, so its consumers
    wait for data that never comes.  With a 1 ms wait limit each wait expires,
    the kernel latches SSA_ERR_TIMEOUT, drains its copies and MMAs, frees its
    tensor memory and returns; the next call at the default limit, hook off,
    matches the oracle."""
    name, B, C, H, W, G, h, dt, mask = case
    wl = wls.custom(name, B, C, H, W, G, h, dt, seed=13)
    x, p, _ = wls.make_inputs(wl)
    xd, pd = _to_dev(x, p)
    try:
        ssa.ssa_set_wait_timeout_ns(1_000_000)
        for after in (1, 2, 3):
            ssa.ssa_debug_set_producer_stall(mask, after)
            ssa.ssa_forward(xd, pd, G, h)
            assert ssa.ssa_get_device_status() == 7, (after, ssa.ssa_last_error_string())
    finally:
        ssa.ssa_debug_set_producer_stall(0, 0)
        ssa.ssa_set_wait_timeout_ns(2_000_000_000)
    out = ssa.ssa_forward(xd, pd, G, h)
    assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
    rel, mx = _compare(out, x, p, wl)
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)
