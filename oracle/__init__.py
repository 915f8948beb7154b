"""fp64 CPU oracle for the spatial self-attention block (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports it, and
it imports nothing from the CUDA library: the two share no code.

The arithmetic lives in ``ssa_oracle.c`` (plain loops, fp64, OpenMP over
independent rows); this module only marshals numpy arrays through ``ctypes``.
What the block computes is stated on the tensortonic page
"diffusion-l03-spatial-self-attention" (problem statement and block equation):

    out = x + image([O_1..O_n] Wo^T + bo),  O_j = softmax(Q_j K_j^T / sqrt(d)) V_j,
    Q/K/V = tokens(GN(x)) W^T + b,  GN: G groups, eps 1e-5, affine.

Parity is pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_*.py``
(library special cases, closed forms, invariants, brute force and the pages'
worked examples).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssa_oracle.so")
_lib = None

F32, BF16 = 0, 1


def build(verbose: bool = False) -> str:
    """Compile ssa_oracle.c into oracle/libssa_oracle.so (gcc, -O2, OpenMP).

    No -ffast-math: every fp64 operation keeps IEEE semantics.  Falls back to a
    single-threaded build when the compiler has no OpenMP runtime.
    """
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", _LIB_PATH, _SRC, "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:3] + extra + base[3:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            if verbose:
                print(" ".join(cmd))
            return _LIB_PATH
    raise RuntimeError("oracle build failed:\n" + r.stderr)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.ssa_oracle_gn_stats.argtypes = [dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp]
    lib.ssa_oracle_gn_stats.restype = ctypes.c_int
    lib.ssa_oracle_forward.argtypes = (
        [dp] + [ctypes.c_int] * 6 + [dp] * 10 + [ip, ctypes.c_int] + [dp] * 9
    )
    lib.ssa_oracle_forward.restype = ctypes.c_int
    lib.ssa_oracle_forward_ex.argtypes = (
        [dp] + [ctypes.c_int] * 6 + [dp] * 10 + [ctypes.c_int, ctypes.c_int, dp, dp, dp] + [ip, ctypes.c_int] +
        [dp] * 9
    )
    lib.ssa_oracle_forward_ex.restype = ctypes.c_int
    lib.ssa_oracle_attention_ex.argtypes = [dp, dp, dp] + [ctypes.c_int] * 5 + [ip, ctypes.c_int, dp,
                                                                                ctypes.c_int, ctypes.c_int, dp, dp]
    lib.ssa_oracle_attention_ex.restype = None
    lib.ssa_oracle_rope.argtypes = [dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ip]
    lib.ssa_oracle_rope.restype = None
    lib.ssa_oracle_qk_norm.argtypes = [dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp]
    lib.ssa_oracle_qk_norm.restype = None
    lib.ssa_oracle_attention.argtypes = [dp, dp, dp] + [ctypes.c_int] * 5 + [dp, dp]
    lib.ssa_oracle_attention.restype = None
    lib.ssa_oracle_out_proj.argtypes = [dp, dp, dp] + [ctypes.c_int] * 3 + [dp]
    lib.ssa_oracle_out_proj.restype = None
    lib.ssa_oracle_round.argtypes = [dp, ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p]
    lib.ssa_oracle_round.restype = None
    lib.ssa_oracle_num_threads.argtypes = []
    lib.ssa_oracle_num_threads.restype = ctypes.c_int
    lib.ssa_oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.ssa_oracle_set_num_threads.restype = None
    lib.ssa_oracle_set_num_threads(usable_cpus())
    _lib = lib
    return lib


def usable_cpus() -> int:
    """CPUs this process may actually run on: the affinity mask, capped by a
    cgroup CPU quota when one is set (so OpenMP does not oversubscribe)."""
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    try:
        with open("/sys/fs/cgroup/cpu.max") as f:
            quota, period = f.read().split()[:2]
        if quota != "max":
            n = min(n, max(1, int(int(quota) // int(period))))
    except (OSError, ValueError):
        pass
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit() and int(env) > 0:
        n = int(env)
    return max(1, n)


def _dptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    """Exact up-conversion of stored values (numpy or torch CPU) to fp64."""
    if hasattr(a, "detach"):  # a torch tensor: fp32 and bf16 widen exactly
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


PARAM_KEYS = ("norm_weight", "norm_bias", "q_weight", "q_bias", "k_weight", "k_bias",
              "v_weight", "v_bias", "out_weight", "out_bias")


def num_threads() -> int:
    return int(_load().ssa_oracle_num_threads())


def gn_stats(x, num_groups: int):
    """Per (sample, group) mean and 1/sqrt(var + 1e-5), two-pass fp64."""
    x = _f64(x)
    B, C = x.shape[0], x.shape[1]
    N = int(np.prod(x.shape[2:]))
    mean = np.empty((B, num_groups))
    rstd = np.empty((B, num_groups))
    rc = _load().ssa_oracle_gn_stats(_dptr(x), B, C, N, num_groups, _dptr(mean), _dptr(rstd))
    if rc != 0:
        raise ValueError("bad shape for group norm")
    return mean, rstd


def forward(x, params: dict, num_groups: int, num_heads: int, qidx=None, want=(), causal=False, rope=False,
            rel_table=None, q_norm_weight=None, k_norm_weight=None):
    """Run the block in fp64.

    x: (B, C, H, W); params: the 10 tensors keyed as on the page (a bias that
    is None or absent means that projection has no bias).
    qidx: None (every pixel) or a 1-D array of pixel indices (row i*W + j)
    shared by every sample.  causal / rope / rel_table ((2H-1)(2W-1), heads)
    select the attention variants of the HNDL attention operator page;
    q_norm_weight / k_norm_weight (heads, d) the query-key RMS normalisation.
    Returns a dict with 'y' (B, C, nq) = the branch image([O] Wo^T + bo) at
    those pixels, and any of 'mean', 'rstd', 'z', 'q', 'k', 'v', 'o', 'p'
    named in ``want`` ('q', 'k' after the rotary embedding when rope).
    """
    x = _f64(x)
    B, C, H, W = x.shape
    N = H * W
    p = {k: (None if params.get(k) is None else _f64(params[k])) for k in PARAM_KEYS}
    for k in ("norm_weight", "norm_bias", "q_weight", "k_weight", "v_weight", "out_weight"):
        if p[k] is None:
            raise ValueError(f"{k} is required")
    rel = None
    if rel_table is not None:
        rel = _f64(rel_table)
        if rel.shape != ((2 * H - 1) * (2 * W - 1), num_heads):
            raise ValueError("rel_table must be ((2H-1)(2W-1), heads)")
    qg = kg = None
    if (q_norm_weight is None) != (k_norm_weight is None):
        raise ValueError("q_norm_weight and k_norm_weight go together")
    if q_norm_weight is not None:
        qg = _f64(q_norm_weight).reshape(num_heads, -1)
        kg = _f64(k_norm_weight).reshape(num_heads, -1)
    G, nh = num_groups, num_heads
    if qidx is not None:
        qi = np.ascontiguousarray(np.asarray(qidx, dtype=np.int32))
        nq = int(qi.size)
        qptr = qi.ctypes.data_as(ctypes.POINTER(ctypes.c_int))
    else:
        qi, nq, qptr = None, N, None
    out = {"y": np.empty((B, C, nq))}
    shapes = {"mean": (B, G), "rstd": (B, G), "z": (B, N, C), "q": (B, nq, C),
              "k": (B, N, C), "v": (B, N, C), "o": (B, nq, C), "p": (B, nh, nq, N)}
    for k in want:
        out[k] = np.empty(shapes[k])
    rc = _load().ssa_oracle_forward_ex(
        _dptr(x), B, C, H, W, G, nh,
        *[_dptr(p[k]) for k in PARAM_KEYS],
        int(bool(causal)), int(bool(rope)), _dptr(rel), _dptr(qg), _dptr(kg),
        qptr, nq,
        _dptr(out["y"]), *[_dptr(out.get(k)) for k in ("mean", "rstd", "z", "q", "k", "v", "o", "p")])
    if rc != 0:
        raise ValueError(f"oracle rejected the problem (rc={rc})")
    return out


def attention(q, k, v, num_heads: int):
    """The attention step alone, in fp64, from given Q (B, nq, C) and K, V
    (B, N, C): per head softmax(Q_j K_j^T / sqrt(d)) V_j, heads side by side.
    Returns O (B, nq, C)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, nq, C = q.shape
    N = k.shape[1]
    if C % num_heads:
        raise ValueError("num_heads must divide C")
    o = np.empty((B, nq, C))
    _load().ssa_oracle_attention(_dptr(q), _dptr(k), _dptr(v), B, N, nq, C, num_heads, _dptr(o), None)
    return o


def attention_ex(q, k, v, num_heads: int, qpos=None, causal=False, rel_table=None, H=None, W=None):
    """The attention step with the variants: qpos (nq,) token positions of the
    query rows (None: row t is position t), causal mask, relative-position
    table ((2H-1)(2W-1), heads) over an H x W grid (H * W == N)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, nq, C = q.shape
    N = k.shape[1]
    if C % num_heads:
        raise ValueError("num_heads must divide C")
    qp = None
    if qpos is not None:
        qp = np.ascontiguousarray(np.asarray(qpos, dtype=np.int32))
    rel = None if rel_table is None else _f64(rel_table)
    if rel is not None and (H is None or W is None or H * W != N):
        raise ValueError("rel_table needs H, W with H * W == N")
    o = np.empty((B, nq, C))
    _load().ssa_oracle_attention_ex(_dptr(q), _dptr(k), _dptr(v), B, N, nq, C, num_heads,
                                    None if qp is None else qp.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                    int(bool(causal)), _dptr(rel), int(H or 1), int(W or 1), _dptr(o), None)
    return o


def rope(m, num_heads: int, pos=None):
    """Rotary embedding (rotate-half, base 10000) of rows (..., tokens, C) by
    token position (pos, broadcast over the leading axes; by default the
    index along the token axis), in fp64; returns a new array."""
    m = _f64(m).copy()
    C = m.shape[-1]
    rows = int(np.prod(m.shape[:-1]))
    if C % num_heads or (C // num_heads) % 2:
        raise ValueError("rope needs an even head dim")
    if pos is None:
        pos = np.arange(m.shape[-2])
    pp = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.int32), m.shape[:-1]).reshape(-1))
    _load().ssa_oracle_rope(_dptr(m), rows, C, num_heads, pp.ctypes.data_as(ctypes.POINTER(ctypes.c_int)))
    return m


def qk_norm(m, num_heads: int, gamma):
    """Query-key RMS normalisation of rows (..., C) per head: x / max(||x||,
    1e-12) * sqrt(d) * gamma[head], in fp64; returns a new array."""
    m = _f64(m).copy()
    C = m.shape[-1]
    g = _f64(gamma).reshape(num_heads, C // num_heads)
    _load().ssa_oracle_qk_norm(_dptr(m), int(np.prod(m.shape[:-1])), C, num_heads, _dptr(g))
    return m


def out_proj(o, out_weight, out_bias):
    """The output projection alone, in fp64: y (B, C, nq) = image(O Wo^T + bo)."""
    o, w = _f64(o), _f64(out_weight)
    b = None if out_bias is None else _f64(out_bias)
    B, nq, C = o.shape
    y = np.empty((B, C, nq))
    _load().ssa_oracle_out_proj(_dptr(o), _dptr(w), _dptr(b), B, nq, C, _dptr(y))
    return y


def round_to(v: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values once, to nearest-even, to 'f32' (float32 array) or
    'bf16' (uint16 array of bf16 bit patterns)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    if dtype == "f32":
        out = np.empty(v.shape, dtype=np.float32)
        code = F32
    elif dtype == "bf16":
        out = np.empty(v.shape, dtype=np.uint16)
        code = BF16
    else:
        raise ValueError(dtype)
    _load().ssa_oracle_round(_dptr(v), v.size, code, out.ctypes.data_as(ctypes.c_void_p))
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp64 exactly."""
    u32 = np.asarray(bits, dtype=np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)


def block(x, params: dict, num_groups: int, num_heads: int, qidx=None, causal=False, rope=False,
          rel_table=None, q_norm_weight=None, k_norm_weight=None):
    """The full block with the page's dtype rule: returns (out_f64, y_f64)
    where out_f64 is x + y rounded once to x's dtype and widened back to fp64
    for comparison.  x's dtype is read from a torch tensor ('bf16' when
    torch.bfloat16) or taken as fp32 for anything else."""
    dt = "bf16" if (hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16") else "f32"
    xf = _f64(x)
    r = forward(xf, params, num_groups, num_heads, qidx=qidx, causal=causal, rope=rope, rel_table=rel_table,
                q_norm_weight=q_norm_weight, k_norm_weight=k_norm_weight)
    y = r["y"]
    B, C = xf.shape[:2]
    xs = xf.reshape(B, C, -1)
    if qidx is not None:
        xs = xs[:, :, np.asarray(qidx)]
    exact = xs + y
    rounded = round_to(exact, dt)
    if dt == "bf16":
        out = bf16_bits_to_f64(rounded)
    else:
        out = rounded.astype(np.float64)
    return out, y
