"""fp16 against bf16 tensor-core operands on the GPU, per named workload.

The library is built twice from the same sources: libssa_gb300.so with fp16
operands (the product) and libssa_gb300_bf16.so with bf16 operands (the
instruction descriptor's A/B format, every 16-bit pack, store and the P
rounding switched to bf16).  Both run the block through the C ABI on the five
named workloads and are compared with the fp64 oracle (branch relative L2
and max |delta| of out; the largest workload on its 512 seeded query pixels).
fp16 must meet the tolerance everywhere.  bf16 meets it on tiny, vae1024 and
unet-l1 (branch ~2-2.6e-3) and misses it on two: the peaked largest workload,
where the rounding of Z, Wq and Wk before the Q/K projection leaves logit
errors that put the branch at ~1.2e-2 (the fp64 emulation in
test_operand_rounding.py predicts the same), and unet-lowres, whose bf16
output rounding already costs ~4.6e-3 of its branch with fp16 operands and
~1.3e-2 with bf16 ones (measured on a GB300).  Those two are reported and
checked only against a loose bound that catches a broken build.  Run with -s
to see the table.
"""
BF16_HOLDS = ("tiny", "vae1024", "unet-l1")
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


def test_operand_types_against_the_oracle(ssa):
    rows = []
    for name, wl in wls.WORKLOADS.items():
        x, p, qidx = wls.make_inputs(wl)
        xd = x.cuda()
        pd = {k: v.cuda() for k, v in p.items()}
        ref, y = oracle.block(x, p, wl.num_groups, wl.num_heads, qidx=None if qidx is None else qidx.numpy())
        B, C = x.shape[:2]
        for op in ("f16", "bf16"):
            ssa.set_operand_type(op)
            try:
                out = ssa.ssa_forward(xd, pd, wl.num_groups, wl.num_heads)
                st = ssa.ssa_get_device_status()
            finally:
                ssa.set_operand_type("f16")
            assert st == 0, (name, op)
            got = out.double().cpu().numpy().reshape(B, C, -1)
            if qidx is not None:
                got = got[:, :, qidx.numpy()]
            rel = np.linalg.norm(got - ref) / np.linalg.norm(y)
            mx = np.abs(got - ref).max()
            rows.append((name, op, rel, mx))
    print("\nworkload        operands  branch rel-L2   max |d out|")
    for name, op, rel, mx in rows:
        print(f"{name:15s} {op:8s}  {rel:12.3e}  {mx:12.3e}")
    for name, op, rel, mx in rows:
        if op == "f16" or name in BF16_HOLDS:
            assert rel <= REL_L2 and mx <= MAX_ABS, (name, op, rel, mx)
        else:
            assert rel < 5 * REL_L2 and mx < 4 * MAX_ABS, (name, op, rel, mx)
