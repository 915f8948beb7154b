"""ssa_forward_static: the block for callers that cannot allocate device memory.

Some callers may not call cudaMalloc once they are running -- fixed-memory
real-time or embedded deployments, plugins whose host forbids allocation on its
execution path, code with no device allocator at hand.  ssa_forward_static
serves them with a library-owned, fixed-size scratch array instead of a
caller workspace.  These tests call it through the C ABI (ctypes, device
pointers of caller-owned tensors) on several problems in a row, so that every
call after the first runs over the previous call's leftovers in the shared
array, and check each result against the fp64 oracle and against ssa_forward
with the tolerances of the parity tests.  The sequence covers fp32 and bf16
inputs, projections without biases (NULL pointers), and head dim 512 with the
attention work split forced on, whose per-tile counters live in the shared
array and must be cleared by the call.  The file is named to be collected
last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from diffusion_net_spatial_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS = 5e-2
KEYS = ("norm_weight", "norm_bias", "q_weight", "q_bias", "k_weight", "k_bias",
        "v_weight", "v_bias", "out_weight", "out_bias")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_net_spatial_gb300 as ssa
    lib = ssa.load_library()
    fn = lib.ssa_forward_static
    fn.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 6 + [ctypes.c_void_p] * 10 + \
        [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return ssa, lib


def _call_static(lib, xd, pd, wl, out):
    ptr = lambda t: ctypes.c_void_p(None if t is None else t.data_ptr())
    dt = 0 if xd.dtype == torch.float32 else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ssa_forward_static(ptr(xd), wl.B, wl.C, wl.H, wl.W, wl.num_groups, wl.num_heads,
                                  *[ptr(pd.get(k)) for k in KEYS], ptr(out), dt, stream)


def _rel_max(a, b, x):
    a = a.double().cpu().numpy().reshape(x.shape[0], x.shape[1], -1)
    b = np.asarray(b).reshape(a.shape)
    xs = x.double().numpy().reshape(a.shape)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b - xs), 1e-30), np.abs(a - b).max()


# Calls in this order: each runs over the leftovers of the one before.
SEQUENCE = [
    # (workload, biases left out, attention split policy)
    ("unet-lowres", (), 0),                   # bf16 in / out
    ("vae1024", (), 1),                       # head dim 512, every query tile split (scratch + counters)
    ("tiny", ("q_bias", "out_bias"), 0),      # NULL biases: that projection has no bias
    ("vae1024", ("v_bias",), 1),              # the split again, over the previous calls' data
    ("unet-l1", (), 0),
]


def test_static_scratch_matches_oracle_and_workspace_forward(lib):
    ssa, clib = lib
    try:
        for name, dropped, policy in SEQUENCE:
            wl = wls.WORKLOADS[name]
            x, p, _ = wls.make_inputs(wl)
            for k in dropped:
                p[k] = None
            xd = x.cuda()
            pd = {k: (None if v is None else v.cuda()) for k, v in p.items()}
            out = torch.full_like(xd, float("nan"))
            ssa.set_attention_split(policy)
            st = _call_static(clib, xd, pd, wl, out)
            assert st == 0, (name, clib.ssa_last_error_string())
            ref = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads)
            assert ssa.ssa_get_device_status() == 0, ssa.ssa_last_error_string()
            exact, _ = oracle.block(x, p, wl.num_groups, wl.num_heads)
            rel, mx = _rel_max(out, exact, x)
            assert rel <= REL_L2 and mx <= MAX_ABS, (name, "oracle", rel, mx)
            rel, mx = _rel_max(out, ref.double().cpu().numpy(), x)
            assert rel <= REL_L2 and mx <= MAX_ABS, (name, "ssa_forward", rel, mx)
    finally:
        ssa.set_attention_split(0)


def test_static_scratch_rejects_problems_above_its_limit(lib):
    ssa, clib = lib
    wl = wls.WORKLOADS["vae16384"]      # needs about 105 MiB of scratch
    assert ssa.ssa_workspace_size(wl.B, wl.C, wl.H, wl.W, wl.num_groups, wl.num_heads) > (48 << 20)
    xd = torch.empty((wl.B, wl.C, wl.H, wl.W), device="cuda")
    pd = {k: torch.empty((wl.C, wl.C) if k.endswith("weight") and not k.startswith("norm") else (wl.C,),
                         device="cuda") for k in KEYS}
    out = torch.empty_like(xd)
    st = _call_static(clib, xd, pd, wl, out)
    assert st == 5                       # SSA_ERR_WORKSPACE, nothing launched
    assert b"ssa_forward_static" in clib.ssa_last_error_string()
