"""ssa_forward_static: the block for callers that cannot allocate device memory.

Some callers may not call cudaMalloc once they are running -- fixed-memory
real-time or embedded deployments, plugins whose host forbids allocation on its
execution path, code with no device allocator at hand.  ssa_forward_static
serves them with a library-owned, fixed-size scratch array instead of a
caller workspace.  This test calls it through the C ABI (ctypes, device
pointers of caller-owned tensors) twice in a row, on two different problems so
that the second call runs over the first call's leftovers, and checks each
result against ssa_forward with the tolerances of the parity tests.  The file
is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

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
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    dt = 0 if xd.dtype == torch.float32 else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ssa_forward_static(ptr(xd), wl.B, wl.C, wl.H, wl.W, wl.num_groups, wl.num_heads,
                                  *[ptr(pd[k]) for k in KEYS], ptr(out), dt, stream)


def test_static_scratch_matches_workspace_forward_twice(lib):
    ssa, clib = lib
    for name in ("unet-l1", "tiny"):
        wl = wls.WORKLOADS[name]
        x, p, _ = wls.make_inputs(wl)
        xd = x.cuda()
        pd = {k: v.cuda() for k, v in p.items()}
        out = torch.empty_like(xd)
        st = _call_static(clib, xd, pd, wl, out)
        assert st == 0, clib.ssa_last_error_string()
        ref = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads)
        assert ssa.ssa_get_device_status() == 0
        a = out.double().cpu().numpy()
        b = ref.double().cpu().numpy()
        xs = x.double().numpy()
        rel = np.linalg.norm(a - b) / np.linalg.norm(b - xs)
        assert rel <= REL_L2 and np.abs(a - b).max() <= MAX_ABS, (name, rel)


def test_static_scratch_rejects_problems_above_its_limit(lib):
    ssa, clib = lib
    wl = wls.WORKLOADS["vae16384"]      # needs about 66 MiB of scratch
    assert ssa.ssa_workspace_size(wl.B, wl.C, wl.H, wl.W, wl.num_groups, wl.num_heads) > (48 << 20)
    xd = torch.empty((wl.B, wl.C, wl.H, wl.W), device="cuda")
    pd = {k: torch.empty((wl.C, wl.C) if k.endswith("weight") and not k.startswith("norm") else (wl.C,),
                         device="cuda") for k in KEYS}
    out = torch.empty_like(xd)
    st = _call_static(clib, xd, pd, wl, out)
    assert st == 5                       # SSA_ERR_WORKSPACE, nothing launched
    assert b"ssa_forward_static" in clib.ssa_last_error_string()
