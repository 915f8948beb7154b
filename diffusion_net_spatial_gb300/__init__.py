"""GB300 (sm_103a) spatial self-attention block: Python binding of the C ABI.

    out = x + image([O_1..O_n] Wo^T + bo),  O_j = softmax(Q_j K_j^T / sqrt(d)) V_j,
    Q/K/V = tokens(GN(x)) W^T + b        (tensortonic "diffusion-l03-spatial-self-attention")

Every step runs in the CUDA kernels of ``libssa_gb300.so``; this module only
marshals torch tensors (device memory, the current stream) into the C calls
declared in ``include/ssa.h`` and raises on a non-OK status.  There is no CPU
fallback: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libssa_gb300.so")
# The same library built with bf16 tensor-core operands (for comparing the two
# operand types; fp16 is the default).
LIB_PATHS = {"f16": LIB_PATH, "bf16": os.path.join(PKG, "libssa_gb300_bf16.so")}

SSA_F32, SSA_BF16 = 0, 1
STATUS = {0: "SSA_OK", 1: "SSA_ERR_CONSTRAINT", 2: "SSA_ERR_DTYPE", 3: "SSA_ERR_ALIGNMENT",
          4: "SSA_ERR_UNSUPPORTED", 5: "SSA_ERR_WORKSPACE", 6: "SSA_ERR_CUDA", 7: "SSA_ERR_TIMEOUT",
          8: "SSA_ERR_NULL"}
PARAM_KEYS = ("norm_weight", "norm_bias", "q_weight", "q_bias", "k_weight", "k_bias",
              "v_weight", "v_bias", "out_weight", "out_bias")
EXPORTS = ("ssa_workspace_size", "ssa_forward", "ssa_plan_create", "ssa_plan_workspace_size",
           "ssa_forward_planned", "ssa_plan_destroy", "ssa_gn_stats", "ssa_pack_weights",
           "ssa_qkv_project", "ssa_qkv_project_rope", "ssa_attention", "ssa_out_project", "ssa_get_device_status",
           "ssa_set_wait_timeout_ns", "ssa_debug_timeout_probe", "ssa_debug_set_producer_stall", "ssa_last_error_string",
           "ssa_launches_per_forward", "ssa_workspace_size_ex", "ssa_forward_ex", "ssa_plan_workspace_size_ex",
           "ssa_forward_planned_ex", "ssa_rope", "ssa_qk_norm", "ssa_pack_rel_table", "ssa_attention_ex",
           "ssa_attention_workspace_size", "ssa_attention_ws", "ssa_set_attention_split")
SPLIT_AUTO, SPLIT_ALWAYS, SPLIT_NEVER = 0, 1, 2
BIAS_KEYS = ("q_bias", "k_bias", "v_bias", "out_bias")


class SsaOptions(ctypes.Structure):
    """struct ssa_options of include/ssa.h (attention variants)."""
    _fields_ = [("causal", ctypes.c_int), ("rope", ctypes.c_int), ("rel_pos_table", ctypes.c_void_p),
                ("q_norm_weight", ctypes.c_void_p), ("k_norm_weight", ctypes.c_void_p)]


class SsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None
_libs = {}
_operand = "f16"


def set_operand_type(operand: str):
    """Selects the library the calls below go through: 'f16' (default) or
    'bf16' tensor-core operands.  Process-wide."""
    global _operand, _lib
    if operand not in LIB_PATHS:
        raise ValueError(operand)
    _operand = operand
    _lib = _libs.get(operand)


def operand_type() -> str:
    return _operand


def load_library():
    """Load libssa_gb300.so and declare the C signatures (no compute)."""
    global _lib
    if _lib is not None:
        return _lib
    path = LIB_PATHS[_operand]
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run `python -m diffusion_net_spatial_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, sz, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
    sig = {
        "ssa_workspace_size": ([i32] * 7, sz),
        "ssa_forward": ([vp] + [i32] * 6 + [vp] * 10 + [vp, i32, vp, sz, vp], i32),
        "ssa_plan_create": ([ctypes.POINTER(vp)] + [i32] * 4 + [vp] * 10 + [vp], i32),
        "ssa_plan_workspace_size": ([vp, i32, i32, i32], sz),
        "ssa_forward_planned": ([vp, vp, i32, i32, i32, vp, vp, sz, vp], i32),
        "ssa_plan_destroy": ([vp], None),
        "ssa_gn_stats": ([vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp], i32),
        "ssa_pack_weights": ([i32, i32, i32] + [vp] * 8 + [vp] * 4 + [vp], i32),
        "ssa_qkv_project": ([vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp], i32),
        "ssa_qkv_project_rope": ([vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp], i32),
        "ssa_attention": ([vp, vp, vp, i32, i32, i32, i32, vp, vp], i32),
        "ssa_out_project": ([vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp], i32),
        "ssa_get_device_status": ([vp], i32),
        "ssa_set_wait_timeout_ns": ([u64], None),
        "ssa_debug_timeout_probe": ([u64, vp], i32),
        "ssa_debug_set_producer_stall": ([ctypes.c_uint32, ctypes.c_uint32], None),
        "ssa_last_error_string": ([], ctypes.c_char_p),
        "ssa_launches_per_forward": ([i32], i32),
        "ssa_workspace_size_ex": ([i32] * 7 + [vp], sz),
        "ssa_forward_ex": ([vp] + [i32] * 6 + [vp] * 10 + [vp, i32, vp, vp, sz, vp], i32),
        "ssa_plan_workspace_size_ex": ([vp, i32, i32, i32, vp], sz),
        "ssa_forward_planned_ex": ([vp, vp, i32, i32, i32, vp, vp, vp, sz, vp], i32),
        "ssa_rope": ([vp, vp, i32, i32, i32, i32, vp], i32),
        "ssa_qk_norm": ([vp, vp, i32, i32, i32, i32, i32, vp, vp, vp], i32),
        "ssa_pack_rel_table": ([vp, i32, i32, i32, i32, vp, vp], i32),
        "ssa_attention_ex": ([vp, vp, vp] + [i32] * 6 + [vp, vp, vp], i32),
        "ssa_attention_workspace_size": ([i32] * 5, sz),
        "ssa_attention_ws": ([vp, vp, vp] + [i32] * 6 + [vp, vp, vp, sz, vp], i32),
        "ssa_set_attention_split": ([i32], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    _libs[_operand] = lib
    return lib


def _check(status: int):
    if status != 0:
        msg = load_library().ssa_last_error_string()
        raise SsaError(status, msg.decode() if msg else "")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSA_F32
    if t.dtype == torch.bfloat16:
        return SSA_BF16
    raise SsaError(2, f"x must be float32 or bfloat16, got {t.dtype}")


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _dev_tensor(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if not t.is_cuda:
        raise SsaError(8, f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise SsaError(2, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise SsaError(3, f"{name} must be contiguous")
    return t


def layout(B: int, C: int, H: int, W: int, num_heads: int) -> dict:
    """Sizes of the internal layouts (see include/ssa.h): dp, ldq, ldn, ldc."""
    d = C // num_heads
    dp = -(-d // 32) * 32 if d > 256 else -(-d // 16) * 16
    return {"N": H * W, "d": d, "dp": dp, "ldq": -(-dp // 64) * 64, "ldn": -(-(H * W) // 8) * 8,
            "ldc": -(-C // 8) * 8}


# ------------------------------------------------------------------ block ---

def ssa_workspace_size(B, C, H, W, num_groups, num_heads, dtype=SSA_F32) -> int:
    return int(load_library().ssa_workspace_size(B, C, H, W, num_groups, num_heads, dtype))


def _params_list(params: dict, dtype):
    """The 10 parameters in ABI order; a bias that is None or absent is passed
    as NULL (that projection has no bias)."""
    out = []
    for k in PARAM_KEYS:
        t = params.get(k)
        if t is None and k in BIAS_KEYS:
            out.append(None)
        else:
            out.append(_dev_tensor(t, k, dtype))
    return out


def _options(causal=False, rope=False, rel_table=None, dtype=None, q_norm_weight=None, k_norm_weight=None):
    if not causal and not rope and rel_table is None and q_norm_weight is None and k_norm_weight is None:
        return None
    for t, n in ((rel_table, "rel_table"), (q_norm_weight, "q_norm_weight"), (k_norm_weight, "k_norm_weight")):
        if t is not None:
            _dev_tensor(t, n, dtype)
    ptr = lambda t: None if t is None else t.data_ptr()
    return SsaOptions(int(bool(causal)), int(bool(rope)), ptr(rel_table), ptr(q_norm_weight), ptr(k_norm_weight))


def ssa_forward(x: torch.Tensor, params: dict, num_groups: int, num_heads: int, out=None, workspace=None,
                stream=None, causal=False, rope=False, rel_table=None, q_norm_weight=None,
                k_norm_weight=None) -> torch.Tensor:
    """The block, one shot (weights packed into the workspace on every call).
    x: (B, C, H, W) float32 or bfloat16 CUDA tensor; params: the 10 tensors
    keyed as on the page, in x's dtype (a bias may be None: no bias).
    causal / rope / rel_table ((2H-1)(2W-1), heads) select the attention
    variants (ssa_forward_ex); q_norm_weight / k_norm_weight (heads, d) the
    query-key RMS normalisation.  Returns out (x's dtype); out may be x."""
    lib = load_library()
    _dev_tensor(x, "x")
    dt = _dtype_code(x)
    B, C, H, W = x.shape
    ps = _params_list(params, x.dtype)
    if out is None:
        out = torch.empty_like(x)
    _dev_tensor(out, "out", x.dtype)
    opt = _options(causal, rope, rel_table, x.dtype, q_norm_weight, k_norm_weight)
    if opt is None:
        need = ssa_workspace_size(B, C, H, W, num_groups, num_heads, dt)
    else:
        need = int(lib.ssa_workspace_size_ex(B, C, H, W, num_groups, num_heads, dt, ctypes.byref(opt)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    if opt is None:
        _check(lib.ssa_forward(_ptr(x), B, C, H, W, num_groups, num_heads, *[_ptr(p) for p in ps], _ptr(out), dt,
                               _ptr(workspace), workspace.numel(), _stream(stream)))
    else:
        _check(lib.ssa_forward_ex(_ptr(x), B, C, H, W, num_groups, num_heads, *[_ptr(p) for p in ps], _ptr(out),
                                  dt, ctypes.byref(opt), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


class SsaPlan:
    """Steady-state form: the parameters are packed once (ssa_plan_create);
    forward() then runs the four hot-path kernels only."""

    def __init__(self, params: dict, num_groups: int, num_heads: int, stream=None):
        lib = load_library()
        ref = params["q_weight"]
        _dev_tensor(ref, "q_weight")
        self.dtype = ref.dtype
        dt = _dtype_code(ref)
        self.C = ref.shape[0]
        self.num_groups, self.num_heads = num_groups, num_heads
        self._params = dict(zip(PARAM_KEYS, _params_list(params, ref.dtype)))  # keep GN affine alive
        h = ctypes.c_void_p()
        _check(lib.ssa_plan_create(ctypes.byref(h), self.C, num_groups, num_heads, dt,
                                   *[_ptr(self._params[k]) for k in PARAM_KEYS], _stream(stream)))
        self._h = h
        self._ws = None

    def workspace_size(self, B, H, W) -> int:
        return int(load_library().ssa_plan_workspace_size(self._h, B, H, W))

    def forward(self, x: torch.Tensor, out=None, workspace=None, stream=None, causal=False, rope=False,
                rel_table=None, q_norm_weight=None, k_norm_weight=None) -> torch.Tensor:
        lib = load_library()
        _dev_tensor(x, "x", self.dtype)
        B, C, H, W = x.shape
        if out is None:
            out = torch.empty_like(x)
        opt = _options(causal, rope, rel_table, self.dtype, q_norm_weight, k_norm_weight)
        if opt is None:
            need = self.workspace_size(B, H, W)
        else:
            need = int(lib.ssa_plan_workspace_size_ex(self._h, B, H, W, ctypes.byref(opt)))
        if workspace is None:
            if self._ws is None or self._ws.numel() < need:
                self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
            workspace = self._ws
        if opt is None:
            _check(lib.ssa_forward_planned(self._h, _ptr(x), B, H, W, _ptr(out), _ptr(workspace),
                                           workspace.numel(), _stream(stream)))
        else:
            _check(lib.ssa_forward_planned_ex(self._h, _ptr(x), B, H, W, _ptr(out), ctypes.byref(opt),
                                              _ptr(workspace), workspace.numel(), _stream(stream)))
        return out

    def close(self):
        if getattr(self, "_h", None):
            load_library().ssa_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ----------------------------------------------------- steps of the path ---

def ssa_gn_stats(x: torch.Tensor, num_groups: int, norm_weight: torch.Tensor, norm_bias: torch.Tensor,
                 stream=None):
    """Returns (mean [B,G], rstd [B,G], gn_scale [B,C], gn_shift [B,C]) fp32."""
    lib = load_library()
    _dev_tensor(x, "x")
    dt = _dtype_code(x)
    B, C = x.shape[:2]
    N = x[0, 0].numel()
    f = dict(dtype=torch.float32, device=x.device)
    mean, rstd = torch.empty(B, num_groups, **f), torch.empty(B, num_groups, **f)
    a, s = torch.empty(B, C, **f), torch.empty(B, C, **f)
    _check(lib.ssa_gn_stats(_ptr(x), B, C, N, num_groups, dt, _ptr(_dev_tensor(norm_weight, "norm_weight", x.dtype)),
                            _ptr(_dev_tensor(norm_bias, "norm_bias", x.dtype)), _ptr(mean), _ptr(rstd), _ptr(a),
                            _ptr(s), _stream(stream)))
    return mean, rstd, a, s


def ssa_pack_weights(params: dict, num_heads: int, stream=None) -> dict:
    lib = load_library()
    ref = _dev_tensor(params["q_weight"], "q_weight")
    dt = _dtype_code(ref)
    C = ref.shape[0]
    lay = layout(1, C, 1, 1, num_heads)
    dev = ref.device
    w_qkv = torch.empty(3 * num_heads * lay["dp"], lay["ldc"], dtype=torch.int16, device=dev)
    b_qkv = torch.empty(3 * num_heads * lay["dp"], dtype=torch.float32, device=dev)
    w_o = torch.empty(C, lay["ldc"], dtype=torch.int16, device=dev)
    b_o = torch.empty(C, dtype=torch.float32, device=dev)
    keys = ("q_weight", "q_bias", "k_weight", "k_bias", "v_weight", "v_bias", "out_weight", "out_bias")
    given = dict(zip(PARAM_KEYS, _params_list({**{k: None for k in BIAS_KEYS}, "norm_weight": ref, "norm_bias": ref,
                                               **params}, ref.dtype)))
    _check(lib.ssa_pack_weights(C, num_heads, dt, *[_ptr(given[k]) for k in keys],
                                _ptr(w_qkv), _ptr(b_qkv), _ptr(w_o), _ptr(b_o), _stream(stream)))
    return {"w_qkv": w_qkv.view(torch.float16), "b_qkv": b_qkv, "w_o": w_o.view(torch.float16), "b_o": b_o}


def ssa_qkv_project(x: torch.Tensor, gn_scale, gn_shift, w_qkv, b_qkv, num_heads: int, stream=None):
    """Returns fp16 (q [B,h,N,ldq], k [B,h,N,ldq], vt [B,h,dp,ldn])."""
    lib = load_library()
    _dev_tensor(x, "x")
    dt = _dtype_code(x)
    B, C, H, W = x.shape
    lay = layout(B, C, H, W, num_heads)
    dev = x.device
    q = torch.empty(B, num_heads, lay["N"], lay["ldq"], dtype=torch.float16, device=dev)
    k = torch.empty_like(q)
    vt = torch.empty(B, num_heads, lay["dp"], lay["ldn"], dtype=torch.float16, device=dev)
    _check(lib.ssa_qkv_project(_ptr(x), B, C, H, W, num_heads, dt, _ptr(gn_scale), _ptr(gn_shift), _ptr(w_qkv),
                               _ptr(b_qkv), _ptr(q), _ptr(k), _ptr(vt), _stream(stream)))
    return q, k, vt


def ssa_qkv_project_rope(x: torch.Tensor, gn_scale, gn_shift, w_qkv, b_qkv, num_heads: int, stream=None):
    """ssa_qkv_project with the rotary embedding applied in the projection's
    epilogue; returns fp16 (q, k, vt) as ssa_qkv_project."""
    lib = load_library()
    _dev_tensor(x, "x")
    dt = _dtype_code(x)
    B, C, H, W = x.shape
    lay = layout(B, C, H, W, num_heads)
    dev = x.device
    q = torch.empty(B, num_heads, lay["N"], lay["ldq"], dtype=torch.float16, device=dev)
    k = torch.empty_like(q)
    vt = torch.empty(B, num_heads, lay["dp"], lay["ldn"], dtype=torch.float16, device=dev)
    _check(lib.ssa_qkv_project_rope(_ptr(x), B, C, H, W, num_heads, dt, _ptr(gn_scale), _ptr(gn_shift), _ptr(w_qkv),
                                    _ptr(b_qkv), _ptr(q), _ptr(k), _ptr(vt), _stream(stream)))
    return q, k, vt


def ssa_attention(q, k, vt, B: int, C: int, N: int, num_heads: int, o=None, stream=None):
    """Returns o fp16 [B, N, ldc] (heads side by side along channels)."""
    lib = load_library()
    lay = layout(B, C, N, 1, num_heads)
    if o is None:
        o = torch.empty(B, N, lay["ldc"], dtype=torch.float16, device=q.device)
    _check(lib.ssa_attention(_ptr(q), _ptr(k), _ptr(vt), B, C, N, num_heads, _ptr(o), _stream(stream)))
    return o


def ssa_rope(q, k, B: int, C: int, N: int, num_heads: int, stream=None):
    """Rotary embedding of q and k (q/k layout) in place, token position = row."""
    _check(load_library().ssa_rope(_ptr(q), _ptr(k), B, C, N, num_heads, _stream(stream)))
    return q, k


def ssa_qk_norm(q, k, B: int, C: int, N: int, num_heads: int, q_norm_weight, k_norm_weight, stream=None):
    """Query-key RMS normalisation of q and k (q/k layout) in place."""
    _dev_tensor(q_norm_weight, "q_norm_weight")
    dt = _dtype_code(q_norm_weight)
    _check(load_library().ssa_qk_norm(_ptr(q), _ptr(k), B, C, N, num_heads, dt, _ptr(q_norm_weight),
                                      _ptr(_dev_tensor(k_norm_weight, "k_norm_weight", q_norm_weight.dtype)),
                                      _stream(stream)))
    return q, k


def ssa_pack_rel_table(table: torch.Tensor, H: int, W: int, num_heads: int, stream=None) -> torch.Tensor:
    """table ((2H-1)(2W-1), heads) in float32/bfloat16 -> packed fp32
    (heads, (2H-1)(2W-1)), each entry times log2(e)."""
    _dev_tensor(table, "table")
    dt = _dtype_code(table)
    packed = torch.empty(num_heads, (2 * H - 1) * (2 * W - 1), dtype=torch.float32, device=table.device)
    _check(load_library().ssa_pack_rel_table(_ptr(table), dt, H, W, num_heads, _ptr(packed), _stream(stream)))
    return packed


def ssa_attention_ex(q, k, vt, B: int, C: int, H: int, W: int, num_heads: int, causal=False, rel_packed=None,
                     o=None, stream=None, workspace=None):
    """ssa_attention over the H x W token grid with the causal mask and the
    packed relative-position table (ssa_pack_rel_table).  With `workspace`
    (a uint8 device tensor of at least attention_workspace_size bytes, 256-byte
    aligned) a head dim of 512 may split query tiles between SM pairs
    (ssa_attention_ws)."""
    lib = load_library()
    lay = layout(B, C, H, W, num_heads)
    if o is None:
        o = torch.empty(B, H * W, lay["ldc"], dtype=torch.float16, device=q.device)
    if workspace is None:
        _check(lib.ssa_attention_ex(_ptr(q), _ptr(k), _ptr(vt), B, C, H, W, num_heads, int(bool(causal)),
                                    _ptr(rel_packed), _ptr(o), _stream(stream)))
    else:
        _check(lib.ssa_attention_ws(_ptr(q), _ptr(k), _ptr(vt), B, C, H, W, num_heads, int(bool(causal)),
                                    _ptr(rel_packed), _ptr(o), _ptr(workspace), workspace.numel(), _stream(stream)))
    return o


def attention_workspace_size(B: int, C: int, H: int, W: int, num_heads: int) -> int:
    """Bytes of scratch ssa_attention_ws can use for this shape (0: none)."""
    return int(load_library().ssa_attention_workspace_size(B, C, H, W, num_heads))


def set_attention_split(policy: int):
    """SPLIT_AUTO, SPLIT_ALWAYS or SPLIT_NEVER (ssa_set_attention_split)."""
    _check(load_library().ssa_set_attention_split(int(policy)))


def ssa_out_project(o, w_o, b_o, x: torch.Tensor, out=None, stream=None):
    lib = load_library()
    _dev_tensor(x, "x")
    dt = _dtype_code(x)
    B, C, H, W = x.shape
    if out is None:
        out = torch.empty_like(x)
    _check(lib.ssa_out_project(_ptr(o), _ptr(w_o), _ptr(b_o), _ptr(x), B, C, H, W, dt, _ptr(out),
                               _stream(stream)))
    return out


# ------------------------------------------------------------ diagnostics ---

def ssa_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(load_library().ssa_get_device_status(_stream(stream)))


def ssa_set_wait_timeout_ns(ns: int):
    load_library().ssa_set_wait_timeout_ns(int(ns))


STALL_QKV, STALL_ATTENTION, STALL_OUT_PROJ = 1, 2, 4


def ssa_debug_set_producer_stall(kernel_mask: int, after_loads: int):
    """Test hook: the named kernels' TMA producers stop after `after_loads`
    loads (0 = off), so their consumers' bounded waits expire."""
    load_library().ssa_debug_set_producer_stall(int(kernel_mask), int(after_loads))


def ssa_debug_timeout_probe(timeout_ns: int, stream=None):
    _check(load_library().ssa_debug_timeout_probe(int(timeout_ns), _stream(stream)))


def ssa_launches_per_forward(planned: bool) -> int:
    return int(load_library().ssa_launches_per_forward(1 if planned else 0))


def ssa_last_error_string() -> str:
    m = load_library().ssa_last_error_string()
    return m.decode() if m else ""
