"""C-ABI checks that need no GPU: the library loads, exports every function
include/ssa.h declares, sizes its workspace, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import diffusion_net_spatial_gb300 as ssa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssa.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ssa.LIB_PATH):
        from diffusion_net_spatial_gb300 import build
        build.build()
    return ssa.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for must in ("ssa_forward", "ssa_workspace_size", "ssa_plan_create", "ssa_forward_planned",
                 "ssa_plan_destroy", "ssa_get_device_status", "ssa_last_error_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(ssa.EXPORTS) <= set(_declared())


def test_workspace_size_matches_layout(lib):
    for (B, C, H, W, G, h) in [(1, 64, 8, 8, 8, 2), (2, 320, 64, 64, 32, 8), (1, 512, 128, 128, 32, 1),
                               (8, 1280, 16, 16, 32, 20), (3, 4, 1, 1, 4, 2)]:
        lay = ssa.layout(B, C, H, W, h)
        N, dp, ldq, ldn, ldc = lay["N"], lay["dp"], lay["ldq"], lay["ldn"], lay["ldc"]
        need = (2 * B * C * 4 + 3 * h * dp * ldc * 2 + 3 * h * dp * 4 + C * ldc * 2 + C * 4
                + 2 * B * h * N * ldq * 2 + B * h * dp * ldn * 2 + B * N * ldc * 2)
        if dp == 512:
            # head dim 512: parts of query tiles split between SM pairs (at most
            # 76 pieces, two parts each of 128 x 512 fp32 + row max and sum)
            # and one counter per query tile
            nqt = (N + 127) // 128
            need += 2 * min(76, B * h * nqt * nqt) * (128 * 512 + 256) * 4 + B * h * nqt * 4
        got = ssa.ssa_workspace_size(B, C, H, W, G, h, ssa.SSA_F32)
        assert need <= got <= need + 13 * 256 + B * C * (N + 4) * 4


def test_padded_head_dims():
    assert ssa.layout(2, 320, 64, 64, 8)["dp"] == 48
    assert ssa.layout(1, 512, 32, 32, 1)["dp"] == 512
    assert ssa.layout(1, 64, 8, 8, 2)["dp"] == 32
    assert ssa.layout(1, 4, 2, 2, 2)["dp"] == 16
    assert ssa.layout(1, 320, 9, 9, 1)["dp"] == 320


def test_bad_shapes_rejected_without_device(lib):
    assert ssa.ssa_workspace_size(1, 64, 8, 8, 7, 2) == 0        # C % G
    assert ssa.ssa_workspace_size(1, 64, 8, 8, 8, 3) == 0        # C % h
    assert ssa.ssa_workspace_size(1, 1024, 8, 8, 8, 1) == 0      # head dim 1024 > 512
    assert ssa.ssa_workspace_size(0, 64, 8, 8, 8, 2) == 0
    nul = [None] * 10
    # status codes come back before any CUDA call
    st = lib.ssa_forward(None, 1, 64, 8, 8, 7, 2, *nul, None, 0, None, 0, None)
    assert st == 1 and b"num_groups" in lib.ssa_last_error_string()
    st = lib.ssa_forward(None, 1, 64, 8, 8, 8, 3, *nul, None, 0, None, 0, None)
    assert st == 1
    st = lib.ssa_forward(None, 1, 64, 8, 8, 8, 2, *nul, None, 0, None, 0, None)
    assert st == 8
    st = lib.ssa_forward(None, 1, 64, 8, 8, 8, 2, *nul, None, 5, None, 0, None)
    assert st == 2
    st = lib.ssa_forward(None, 1, 1024, 8, 8, 8, 1, *nul, None, 0, None, 0, None)
    assert st == 4
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)
    ptrs = [fake] * 10
    st = lib.ssa_forward(odd, 1, 64, 8, 8, 8, 2, *ptrs, fake, 0, fake, 1 << 30, None)
    assert st == 3
    st = lib.ssa_forward(fake, 1, 64, 8, 8, 8, 2, *ptrs, fake, 0, ctypes.c_void_p(0x1010), 1 << 30, None)
    assert st == 3          # workspace not 256-byte aligned
    st = lib.ssa_forward(fake, 1, 64, 8, 8, 8, 2, *ptrs, fake, 0, fake, 16, None)
    assert st == 5          # workspace too small
    # empty problems: no work, SSA_OK, NULL pointers not read; bad splits still fail
    assert lib.ssa_forward(None, 0, 64, 8, 8, 8, 2, *nul, None, 0, None, 0, None) == 0
    assert lib.ssa_forward(None, 2, 64, 0, 8, 8, 2, *nul, None, 0, None, 0, None) == 0
    assert lib.ssa_forward(None, 0, 64, 8, 8, 7, 2, *nul, None, 0, None, 0, None) == 1
    assert lib.ssa_forward(None, -1, 64, 8, 8, 8, 2, *nul, None, 0, None, 0, None) == 1
    assert ssa.ssa_workspace_size(0, 64, 8, 8, 8, 2) == 0
    # a relative-position table of (2H-1)(2W-1) > 2^31 - 1 entries per head
    st = lib.ssa_pack_rel_table(fake, 0, 30000, 30000, 1, fake, None)
    assert st == 4 and b"relative-position table" in lib.ssa_last_error_string()


def test_launch_count(lib):
    assert ssa.ssa_launches_per_forward(False) == 5
    assert ssa.ssa_launches_per_forward(True) == 4


def test_attention_scratch_size_and_split_policy(lib):
    # head dim 512: two parts of 128 x 512 fp32 + 256 row values per cluster
    # (at most 76 clusters) and one counter per query tile; other head dims: none
    nqt = (128 * 128 + 127) // 128
    assert ssa.attention_workspace_size(1, 512, 128, 128, 1) == 2 * 76 * (128 * 512 + 256) * 4 + nqt * 4
    assert ssa.attention_workspace_size(1, 512, 4, 4, 1) == 2 * 1 * (128 * 512 + 256) * 4 + 4  # one unit
    assert ssa.attention_workspace_size(2, 320, 64, 64, 8) == 0
    assert ssa.attention_workspace_size(1, 64, 0, 8, 2) == 0
    assert lib.ssa_set_attention_split(7) == 1
    for p in (ssa.SPLIT_ALWAYS, ssa.SPLIT_NEVER, ssa.SPLIT_AUTO):
        assert lib.ssa_set_attention_split(p) == 0


def test_bf16_operand_library_exports_the_same_boundary(lib):
    """The same sources built with bf16 tensor-core operands (for the operand
    comparison) load and export every declared function too."""
    path = ssa.LIB_PATHS["bf16"]
    if not os.path.exists(path):
        from diffusion_net_spatial_gb300 import build
        build.build()
    other = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(other, name), name
