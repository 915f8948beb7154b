// ssa.cu -- the C ABI (include/ssa.h): argument checks, workspace layout,
// plans, launch order and device-side error reporting for the spatial
// self-attention block of tensortonic "diffusion-l03-spatial-self-attention"
// (block equation: out = x + image([O_1..O_n] Wo^T + bo)).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/ssa.h"
#include "internal.h"
#include "ptx.cuh"

namespace ssa {

// ------------------------------------------------------------ device state --
__device__ uint32_t g_err_word;

namespace {

constexpr int kMaxDevices = 64;
thread_local char t_err[512] = "";
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_split_policy{0};
std::atomic<uint32_t> g_stall_mask{0}, g_stall_after{0};
std::mutex g_mu;
uint32_t *g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

ssa_status fail(ssa_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
ssa_status fail(ssa_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return st;
}

ssa_status cuda_fail(cudaError_t e, const char *what) {
  return fail(SSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Per-device state: the address of the device error word and the SM count.
ssa_status device_state(uint32_t **err, int *num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SSA_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_err_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    g_err_ptr[dev] = static_cast<uint32_t *>(p);
    g_num_sms[dev] = sms;
  }
  if (err) *err = g_err_ptr[dev];
  if (num_sms) *num_sms = g_num_sms[dev];
  return SSA_OK;
}

}  // namespace

int attention_split_policy() { return g_split_policy.load(); }

namespace {

ssa_status kparams(KParams *kp, int *num_sms) {
  uint32_t *err = nullptr;
  ssa_status s = device_state(&err, num_sms);
  if (s != SSA_OK) return s;
  kp->err = err;
  kp->timeout_ns = g_timeout_ns.load();
  kp->stall_mask = g_stall_mask.load();
  kp->stall_after = g_stall_after.load();
  return SSA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

// Checks shared by every entry point that takes the problem shape; a
// num_groups or num_heads of 0 means "not used by this entry point".
// An empty problem (B, H or W zero; C and its split into groups and heads
// still valid) is no work: check_shape returns kEmpty, and every entry point
// then returns SSA_OK before touching its pointers or the device.
constexpr ssa_status kEmpty = static_cast<ssa_status>(1000);

ssa_status check_shape(int B, int C, int H, int W, int G, int h) {
  if (B < 0 || C <= 0 || H < 0 || W < 0 || G < 0 || h < 0)
    return fail(SSA_ERR_CONSTRAINT, "sizes must be non-negative, C positive (B=%d C=%d H=%d W=%d G=%d h=%d)", B, C,
                H, W, G, h);
  if (G > 0 && C % G) return fail(SSA_ERR_CONSTRAINT, "num_groups (%d) must divide C (%d)", G, C);
  if (h > 0 && C % h) return fail(SSA_ERR_CONSTRAINT, "num_heads (%d) must divide C (%d)", h, C);
  if (h > 0 && C / h > 512) return fail(SSA_ERR_UNSUPPORTED, "head dim %d > 512", C / h);
  if (B == 0 || H == 0 || W == 0) return kEmpty;
  const long long N = (long long)H * W;
  if (N > (1LL << 30) || (long long)B * (G > 0 ? G : 1) > 65535 || (long long)B * (h > 0 ? h : 1) > 65535 ||
      B > 65535 || (N + 127) / 128 > 65535 || (long long)B * C * N > (1LL << 40))
    return fail(SSA_ERR_UNSUPPORTED, "problem exceeds the launch-grid limits");
  return SSA_OK;
}

// The relative-position table of an H x W grid has (2H-1)(2W-1) entries per
// head, counted and indexed in 32 bits by the table kernels.
ssa_status check_rel_grid(int H, int W) {
  const long long entries = (2LL * H - 1) * (2LL * W - 1);
  if (entries > 2147483647LL)
    return fail(SSA_ERR_UNSUPPORTED, "a relative-position table of %lld entries per head (grid %d x %d) exceeds 2^31 - 1",
                entries, H, W);
  return SSA_OK;
}

ssa_status check_dtype(ssa_dtype dt) {
  if (dt != SSA_F32 && dt != SSA_BF16) return fail(SSA_ERR_DTYPE, "dtype %d is neither SSA_F32 nor SSA_BF16", (int)dt);
  return SSA_OK;
}

int esize(ssa_dtype dt) { return dt == SSA_F32 ? 4 : 2; }

// x needs a 16-byte row pitch for its TMA map; otherwise it is first copied
// into a padded workspace buffer.
int x_pitch(int N, ssa_dtype dt) {
  const int per16 = 16 / esize(dt);
  return (N % per16 == 0) ? N : round_up(N, per16);
}

// Workspace layout of one forward call.
struct WsLayout {
  size_t ga, gs, wqkv, bqkv, wo, bo, q, k, vt, o, xpad, rel, scratch, scratch_bytes, total;
};

WsLayout ws_layout(const Dims &dm, ssa_dtype dt, bool with_weights, bool with_rel = false) {
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = al256(off + bytes);
    return at;
  };
  w.ga = take((size_t)dm.B * dm.C * 4);
  w.gs = take((size_t)dm.B * dm.C * 4);
  if (with_weights) {
    w.wqkv = take((size_t)dm.ntot * dm.ldc * 2);
    w.bqkv = take((size_t)dm.ntot * 4);
    w.wo = take((size_t)dm.C * dm.ldc * 2);
    w.bo = take((size_t)dm.C * 4);
  }
  w.q = take((size_t)dm.B * dm.h * dm.N * dm.ldq * 2);
  w.k = take((size_t)dm.B * dm.h * dm.N * dm.ldq * 2);
  w.vt = take((size_t)dm.B * dm.h * dm.dp * dm.ldn * 2);
  w.o = take((size_t)dm.B * dm.N * dm.ldc * 2);
  const int ldx = x_pitch(dm.N, dt);
  if (ldx != dm.N) w.xpad = take((size_t)dm.B * dm.C * ldx * esize(dt));
  if (with_rel) w.rel = take((size_t)dm.h * (2 * dm.H - 1) * (2 * dm.W - 1) * 4);
  w.scratch_bytes = attention_scratch_bytes(dm);
  if (w.scratch_bytes) w.scratch = take(w.scratch_bytes);
  w.total = off;
  return w;
}

__global__ void timeout_probe_kernel(uint32_t *err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Abort ab{&flag, err, limit_ns};
    (void)mbar_wait(&bar, 0, ab);  // nothing ever arrives: expires and latches the error
  }
}

struct Ptrs {
  const void *gw, *gb, *wq, *bq, *wk, *bk, *wv, *bv, *wo, *bo;
};

// Variants of the attention step (all off for the block itself).
struct Variants {
  int causal, rope;
  const void *rel_table;  // caller's table, x's dtype; packed into the workspace per call
  const void *q_gamma, *k_gamma;  // query-key RMS-norm weights [h][d], x's dtype (both or neither)
};

// Checks the variants against the problem: rope needs an even head dim.
ssa_status check_variants(const Dims &dm, const Variants &v) {
  if (v.rope && dm.d % 2) return fail(SSA_ERR_CONSTRAINT, "rope needs an even head dim (d = %d)", dm.d);
  if (v.rel_table && !aligned16(v.rel_table)) return fail(SSA_ERR_ALIGNMENT, "rel_pos_table must be 16-byte aligned");
  if (v.rel_table) {
    const ssa_status s = check_rel_grid(dm.H, dm.W);
    if (s != SSA_OK) return s;
  }
  if ((v.q_gamma == nullptr) != (v.k_gamma == nullptr))
    return fail(SSA_ERR_NULL, "q_norm_weight and k_norm_weight must be given together");
  return SSA_OK;
}

// The four steps after packing, in stream order (plus the variants' rotary
// embedding after the projection and table packing before the attention).
ssa_status run_block(const Dims &dm, ssa_dtype dt, const void *x, void *out, const Ptrs &p,
                     const uint16_t *w_qkv, const float *b_qkv, const uint16_t *w_o, const float *b_o,
                     uint8_t *ws, const WsLayout &wl, const KParams &kp, int num_sms, cudaStream_t st,
                     const Variants &var = Variants{0, 0, nullptr, nullptr, nullptr}) {
  float *ga = reinterpret_cast<float *>(ws + wl.ga);
  float *gs = reinterpret_cast<float *>(ws + wl.gs);
  uint16_t *q = reinterpret_cast<uint16_t *>(ws + wl.q);
  uint16_t *k = reinterpret_cast<uint16_t *>(ws + wl.k);
  uint16_t *vt = reinterpret_cast<uint16_t *>(ws + wl.vt);
  uint16_t *o = reinterpret_cast<uint16_t *>(ws + wl.o);
  // The rotary embedding runs inside the projection's epilogue when Q/K rows
  // are pair-interleaved; with the query-key norm (which must come first) it
  // stays a separate pass after the norm.
  const bool fuse_rope = var.rope && !var.q_gamma && qk_pair_interleaved(dm);
  cudaError_t e = launch_gn_stats(x, dm.B, dm.C, dm.N, dm.G, (int)dt, p.gw, p.gb, nullptr, nullptr, ga, gs, num_sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "gn_stats launch");
  const void *xq = x;
  int ldx = x_pitch(dm.N, dt);
  if (ldx != dm.N) {
    e = launch_pad_x(x, dm.B, dm.C, dm.N, ldx, esize(dt), ws + wl.xpad, st);
    if (e != cudaSuccess) return cuda_fail(e, "pad_x launch");
    xq = ws + wl.xpad;
  }
  int r = launch_qkv_gemm(dm, (int)dt, xq, ldx, ga, gs, w_qkv, b_qkv, q, k, vt, kp, st, fuse_rope ? 1 : 0);
  if (r == 1) return fail(SSA_ERR_CUDA, "qkv_gemm: tensor map encoding failed");
  if (r) return cuda_fail(cudaGetLastError(), "qkv_gemm launch");
  if (var.q_gamma) {
    e = launch_qk_norm(dm, (int)dt, q, k, var.q_gamma, var.k_gamma, st);
    if (e != cudaSuccess) return cuda_fail(e, "qk norm launch");
  }
  if (var.rope && !fuse_rope) {
    e = launch_rope(dm, q, k, st);
    if (e != cudaSuccess) return cuda_fail(e, "rope launch");
  }
  float *rel = nullptr;
  if (var.rel_table) {
    rel = reinterpret_cast<float *>(ws + wl.rel);
    e = launch_rel_table_pack((int)dt, var.rel_table, dm.H, dm.W, dm.h, rel, st);
    if (e != cudaSuccess) return cuda_fail(e, "rel table pack launch");
  }
  r = launch_attention(dm, q, k, vt, o, kp, st, var.causal, rel, wl.scratch_bytes ? ws + wl.scratch : nullptr);
  if (r == 1) return fail(SSA_ERR_CUDA, "attention: tensor map encoding failed");
  if (r) return cuda_fail(cudaGetLastError(), "attention launch");
  r = launch_out_proj(dm, (int)dt, o, w_o, b_o, x, out, kp, st);
  if (r == 1) return fail(SSA_ERR_CUDA, "out_proj: tensor map encoding failed");
  if (r) return cuda_fail(cudaGetLastError(), "out_proj launch");
  return SSA_OK;
}

}  // namespace

CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                      const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                      CUtensorMapSwizzle swz) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return CUDA_ERROR_NOT_FOUND;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t gdim[5], gstr[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gstr[i] = strides_bytes[i];
  return g_encode(map, dt, (cuuint32_t)rank, const_cast<void *>(base), gdim, gstr, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

cudaError_t launch_timeout_probe(const KParams &kp, cudaStream_t st) {
  timeout_probe_kernel<<<1, 32, 0, st>>>(kp.err, kp.timeout_ns);
  return cudaGetLastError();
}

}  // namespace ssa

// ===================================================================== ABI ==
using namespace ssa;

struct ssa_plan {
  Dims dm;  // C, G, h and derived head sizes (B, H, W unused)
  ssa_dtype dtype;
  int C, G, h;
  const void *gw, *gb;  // GN affine stays in the caller's memory
  uint8_t *dev;         // packed weights (owned)
  uint16_t *w_qkv, *w_o;
  float *b_qkv, *b_o;
};

extern "C" {

const char *ssa_last_error_string(void) { return t_err; }

void ssa_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

void ssa_debug_set_producer_stall(uint32_t kernel_mask, uint32_t after_loads) {
  g_stall_mask.store(after_loads ? (kernel_mask & 7u) : 0u);
  g_stall_after.store(after_loads);
}

ssa_status ssa_set_attention_split(int policy) {
  if (policy < SSA_SPLIT_AUTO || policy > SSA_SPLIT_NEVER)
    return fail(SSA_ERR_CONSTRAINT, "split policy %d is not SSA_SPLIT_AUTO, _ALWAYS or _NEVER", policy);
  g_split_policy.store(policy);
  return SSA_OK;
}

size_t ssa_attention_workspace_size(int B, int C, int H, int W, int num_heads) {
  if (num_heads <= 0 || check_shape(B, C, H, W, 0, num_heads) != SSA_OK) return 0;
  return attention_scratch_bytes(make_dims(B, C, H, W, 1, num_heads));
}

int ssa_launches_per_forward(int planned) { return planned ? 4 : 5; }

size_t ssa_workspace_size(int B, int C, int H, int W, int num_groups, int num_heads, ssa_dtype dtype) {
  if (check_shape(B, C, H, W, num_groups, num_heads) != SSA_OK || check_dtype(dtype) != SSA_OK) return 0;
  return ws_layout(make_dims(B, C, H, W, num_groups, num_heads), dtype, true).total;
}

static Variants variants_of(const ssa_options *opt) {
  if (!opt) return Variants{0, 0, nullptr, nullptr, nullptr};
  return Variants{opt->causal ? 1 : 0, opt->rope ? 1 : 0, opt->rel_pos_table, opt->q_norm_weight,
                  opt->k_norm_weight};
}

static ssa_status forward_impl(const void *x, int B, int C, int H, int W, int num_groups, int num_heads,
                               const void *norm_weight, const void *norm_bias, const void *q_weight,
                               const void *q_bias, const void *k_weight, const void *k_bias, const void *v_weight,
                               const void *v_bias, const void *out_weight, const void *out_bias, void *out,
                               ssa_dtype dtype, const Variants &var, void *workspace, size_t workspace_bytes,
                               void *stream) {
  ssa_status s = check_shape(B, C, H, W, num_groups, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if ((s = check_dtype(dtype)) != SSA_OK) return s;
  // Biases may be NULL (that projection has no bias).
  const void *ptrs[] = {x, norm_weight, norm_bias, q_weight, k_weight, v_weight, out_weight, out, workspace};
  for (const void *p : ptrs)
    if (!p) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(x) || !aligned16(out)) return fail(SSA_ERR_ALIGNMENT, "x and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(SSA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  const Dims dm = make_dims(B, C, H, W, num_groups, num_heads);
  if ((s = check_variants(dm, var)) != SSA_OK) return s;
  const WsLayout wl = ws_layout(dm, dtype, true, var.rel_table != nullptr);
  if (workspace_bytes < wl.total)
    return fail(SSA_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes, wl.total);
  KParams kp{};
  int num_sms = 0;
  if ((s = kparams(&kp, &num_sms)) != SSA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  uint16_t *w_qkv = reinterpret_cast<uint16_t *>(ws + wl.wqkv);
  float *b_qkv = reinterpret_cast<float *>(ws + wl.bqkv);
  uint16_t *w_o = reinterpret_cast<uint16_t *>(ws + wl.wo);
  float *b_o = reinterpret_cast<float *>(ws + wl.bo);
  cudaError_t e = launch_pack_weights(dm, (int)dtype, q_weight, q_bias, k_weight, k_bias, v_weight, v_bias,
                                      out_weight, out_bias, w_qkv, b_qkv, w_o, b_o, st);
  if (e != cudaSuccess) return cuda_fail(e, "pack launch");
  const Ptrs p{norm_weight, norm_bias, q_weight, q_bias, k_weight, k_bias, v_weight, v_bias, out_weight, out_bias};
  return run_block(dm, dtype, x, out, p, w_qkv, b_qkv, w_o, b_o, ws, wl, kp, num_sms, st, var);
}

ssa_status ssa_forward(const void *x, int B, int C, int H, int W, int num_groups, int num_heads,
                       const void *norm_weight, const void *norm_bias, const void *q_weight, const void *q_bias,
                       const void *k_weight, const void *k_bias, const void *v_weight, const void *v_bias,
                       const void *out_weight, const void *out_bias, void *out, ssa_dtype dtype, void *workspace,
                       size_t workspace_bytes, void *stream) {
  return forward_impl(x, B, C, H, W, num_groups, num_heads, norm_weight, norm_bias, q_weight, q_bias, k_weight,
                      k_bias, v_weight, v_bias, out_weight, out_bias, out, dtype, Variants{0, 0, nullptr, nullptr, nullptr}, workspace,
                      workspace_bytes, stream);
}

size_t ssa_workspace_size_ex(int B, int C, int H, int W, int num_groups, int num_heads, ssa_dtype dtype,
                             const ssa_options *opt) {
  if (check_shape(B, C, H, W, num_groups, num_heads) != SSA_OK || check_dtype(dtype) != SSA_OK) return 0;
  return ws_layout(make_dims(B, C, H, W, num_groups, num_heads), dtype, true, opt && opt->rel_pos_table).total;
}

ssa_status ssa_forward_ex(const void *x, int B, int C, int H, int W, int num_groups, int num_heads,
                          const void *norm_weight, const void *norm_bias, const void *q_weight, const void *q_bias,
                          const void *k_weight, const void *k_bias, const void *v_weight, const void *v_bias,
                          const void *out_weight, const void *out_bias, void *out, ssa_dtype dtype,
                          const ssa_options *opt, void *workspace, size_t workspace_bytes, void *stream) {
  return forward_impl(x, B, C, H, W, num_groups, num_heads, norm_weight, norm_bias, q_weight, q_bias, k_weight,
                      k_bias, v_weight, v_bias, out_weight, out_bias, out, dtype, variants_of(opt), workspace,
                      workspace_bytes, stream);
}

ssa_status ssa_plan_create(ssa_plan **plan, int C, int num_groups, int num_heads, ssa_dtype dtype,
                           const void *norm_weight, const void *norm_bias, const void *q_weight, const void *q_bias,
                           const void *k_weight, const void *k_bias, const void *v_weight, const void *v_bias,
                           const void *out_weight, const void *out_bias, void *stream) {
  if (!plan) return fail(SSA_ERR_NULL, "plan out-pointer is NULL");
  *plan = nullptr;
  ssa_status s = check_shape(1, C, 1, 1, num_groups, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if ((s = check_dtype(dtype)) != SSA_OK) return s;
  const void *ptrs[] = {norm_weight, norm_bias, q_weight, k_weight, v_weight, out_weight};  // biases may be NULL
  for (const void *p : ptrs)
    if (!p) return fail(SSA_ERR_NULL, "a required parameter pointer is NULL");
  if ((s = device_state(nullptr, nullptr)) != SSA_OK) return s;
  ssa_plan *pl = new ssa_plan{};
  pl->dm = make_dims(1, C, 1, 1, num_groups, num_heads);
  pl->dtype = dtype;
  pl->C = C; pl->G = num_groups; pl->h = num_heads;
  pl->gw = norm_weight; pl->gb = norm_bias;
  const Dims &dm = pl->dm;
  size_t off = 0;
  const size_t o_wqkv = off; off = al256(off + (size_t)dm.ntot * dm.ldc * 2);
  const size_t o_bqkv = off; off = al256(off + (size_t)dm.ntot * 4);
  const size_t o_wo = off; off = al256(off + (size_t)C * dm.ldc * 2);
  const size_t o_bo = off; off = al256(off + (size_t)C * 4);
  void *mem = nullptr;
  cudaError_t e = cudaMalloc(&mem, off);
  if (e != cudaSuccess) {
    delete pl;
    return cuda_fail(e, "cudaMalloc(plan)");
  }
  pl->dev = static_cast<uint8_t *>(mem);
  pl->w_qkv = reinterpret_cast<uint16_t *>(pl->dev + o_wqkv);
  pl->b_qkv = reinterpret_cast<float *>(pl->dev + o_bqkv);
  pl->w_o = reinterpret_cast<uint16_t *>(pl->dev + o_wo);
  pl->b_o = reinterpret_cast<float *>(pl->dev + o_bo);
  e = launch_pack_weights(dm, (int)dtype, q_weight, q_bias, k_weight, k_bias, v_weight, v_bias, out_weight,
                          out_bias, pl->w_qkv, pl->b_qkv, pl->w_o, pl->b_o, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaFree(mem);
    delete pl;
    return cuda_fail(e, "pack launch");
  }
  *plan = pl;
  return SSA_OK;
}

size_t ssa_plan_workspace_size(const ssa_plan *plan, int B, int H, int W) {
  if (!plan || check_shape(B, plan->C, H, W, plan->G, plan->h) != SSA_OK) return 0;
  return ws_layout(make_dims(B, plan->C, H, W, plan->G, plan->h), plan->dtype, false).total;
}

size_t ssa_plan_workspace_size_ex(const ssa_plan *plan, int B, int H, int W, const ssa_options *opt) {
  if (!plan || check_shape(B, plan->C, H, W, plan->G, plan->h) != SSA_OK) return 0;
  return ws_layout(make_dims(B, plan->C, H, W, plan->G, plan->h), plan->dtype, false, opt && opt->rel_pos_table)
      .total;
}

static ssa_status planned_impl(const ssa_plan *plan, const void *x, int B, int H, int W, void *out,
                               const Variants &var, void *workspace, size_t workspace_bytes, void *stream) {
  if (!plan) return fail(SSA_ERR_NULL, "plan is NULL");
  ssa_status s = check_shape(B, plan->C, H, W, plan->G, plan->h);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if (!x || !out || !workspace) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(x) || !aligned16(out)) return fail(SSA_ERR_ALIGNMENT, "x and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(SSA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  const Dims dm = make_dims(B, plan->C, H, W, plan->G, plan->h);
  if ((s = check_variants(dm, var)) != SSA_OK) return s;
  const WsLayout wl = ws_layout(dm, plan->dtype, false, var.rel_table != nullptr);
  if (workspace_bytes < wl.total)
    return fail(SSA_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes, wl.total);
  KParams kp{};
  int num_sms = 0;
  if ((s = kparams(&kp, &num_sms)) != SSA_OK) return s;
  const Ptrs p{plan->gw, plan->gb, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  return run_block(dm, plan->dtype, x, out, p, plan->w_qkv, plan->b_qkv, plan->w_o, plan->b_o,
                   static_cast<uint8_t *>(workspace), wl, kp, num_sms, static_cast<cudaStream_t>(stream), var);
}

ssa_status ssa_forward_planned(const ssa_plan *plan, const void *x, int B, int H, int W, void *out, void *workspace,
                               size_t workspace_bytes, void *stream) {
  return planned_impl(plan, x, B, H, W, out, Variants{0, 0, nullptr, nullptr, nullptr}, workspace, workspace_bytes, stream);
}

ssa_status ssa_forward_planned_ex(const ssa_plan *plan, const void *x, int B, int H, int W, void *out,
                                  const ssa_options *opt, void *workspace, size_t workspace_bytes, void *stream) {
  return planned_impl(plan, x, B, H, W, out, variants_of(opt), workspace, workspace_bytes, stream);
}

void ssa_plan_destroy(ssa_plan *plan) {
  if (!plan) return;
  if (plan->dev) cudaFree(plan->dev);
  delete plan;
}

ssa_status ssa_gn_stats(const void *x, int B, int C, int N, int num_groups, ssa_dtype dtype,
                        const void *norm_weight, const void *norm_bias, float *mean, float *rstd, float *gn_scale,
                        float *gn_shift, void *stream) {
  if (num_groups <= 0) return fail(SSA_ERR_CONSTRAINT, "num_groups must be positive");
  ssa_status s = check_shape(B, C, N, 1, num_groups, 0);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if ((s = check_dtype(dtype)) != SSA_OK) return s;
  if (!x || !norm_weight || !norm_bias || !gn_scale || !gn_shift) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(x)) return fail(SSA_ERR_ALIGNMENT, "x must be 16-byte aligned");
  int num_sms = 0;
  if ((s = device_state(nullptr, &num_sms)) != SSA_OK) return s;
  cudaError_t e = launch_gn_stats(x, B, C, N, num_groups, (int)dtype, norm_weight, norm_bias, mean, rstd, gn_scale,
                                  gn_shift, num_sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSA_OK : cuda_fail(e, "gn_stats launch");
}

ssa_status ssa_pack_weights(int C, int num_heads, ssa_dtype dtype, const void *q_weight, const void *q_bias,
                            const void *k_weight, const void *k_bias, const void *v_weight, const void *v_bias,
                            const void *out_weight, const void *out_bias, uint16_t *w_qkv, float *b_qkv,
                            uint16_t *w_o, float *b_o, void *stream) {
  if (num_heads <= 0) return fail(SSA_ERR_CONSTRAINT, "num_heads must be positive");
  ssa_status s = check_shape(1, C, 1, 1, 0, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if ((s = check_dtype(dtype)) != SSA_OK) return s;
  const void *ptrs[] = {q_weight, k_weight, v_weight, out_weight, w_qkv, b_qkv, w_o, b_o};  // biases may be NULL
  for (const void *p : ptrs)
    if (!p) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  const Dims dm = make_dims(1, C, 1, 1, 1, num_heads);
  cudaError_t e = launch_pack_weights(dm, (int)dtype, q_weight, q_bias, k_weight, k_bias, v_weight, v_bias,
                                      out_weight, out_bias, w_qkv, b_qkv, w_o, b_o, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSA_OK : cuda_fail(e, "pack launch");
}

ssa_status ssa_qkv_project(const void *x, int B, int C, int H, int W, int num_heads, ssa_dtype dtype,
                           const float *gn_scale, const float *gn_shift, const uint16_t *w_qkv, const float *b_qkv,
                           uint16_t *q, uint16_t *k, uint16_t *vt, void *stream) {
  if (num_heads <= 0) return fail(SSA_ERR_CONSTRAINT, "num_heads must be positive");
  ssa_status s = check_shape(B, C, H, W, 0, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if ((s = check_dtype(dtype)) != SSA_OK) return s;
  if (!x || !gn_scale || !gn_shift || !w_qkv || !b_qkv || !q || !k || !vt)
    return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(q) || !aligned16(k) || !aligned16(vt))
    return fail(SSA_ERR_ALIGNMENT, "x, w_qkv, q, k and vt must be 16-byte aligned");
  if (x_pitch(H * W, dtype) != H * W)
    return fail(SSA_ERR_ALIGNMENT, "H*W*sizeof(x) must be a multiple of 16 bytes for this entry point");
  KParams kp{};
  int num_sms = 0;
  if ((s = kparams(&kp, &num_sms)) != SSA_OK) return s;
  const Dims dm = make_dims(B, C, H, W, 1, num_heads);
  const int r = launch_qkv_gemm(dm, (int)dtype, x, dm.N, gn_scale, gn_shift, w_qkv, b_qkv, q, k, vt, kp,
                                static_cast<cudaStream_t>(stream));
  if (r == 1) return fail(SSA_ERR_CUDA, "qkv_gemm: tensor map encoding failed");
  if (r) return cuda_fail(cudaGetLastError(), "qkv_gemm launch");
  return SSA_OK;
}

ssa_status ssa_qkv_project_rope(const void *x, int B, int C, int H, int W, int num_heads, ssa_dtype dtype,
                                const float *gn_scale, const float *gn_shift, const uint16_t *w_qkv,
                                const float *b_qkv, uint16_t *q, uint16_t *k, uint16_t *vt, void *stream) {
  if (num_heads <= 0) return fail(SSA_ERR_CONSTRAINT, "num_heads must be positive");
  ssa_status s = check_shape(B, C, H, W, 0, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if ((s = check_dtype(dtype)) != SSA_OK) return s;
  if (!x || !gn_scale || !gn_shift || !w_qkv || !b_qkv || !q || !k || !vt)
    return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(q) || !aligned16(k) || !aligned16(vt))
    return fail(SSA_ERR_ALIGNMENT, "x, w_qkv, q, k and vt must be 16-byte aligned");
  if (x_pitch(H * W, dtype) != H * W)
    return fail(SSA_ERR_ALIGNMENT, "H*W*sizeof(x) must be a multiple of 16 bytes for this entry point");
  const Dims dm = make_dims(B, C, H, W, 1, num_heads);
  if (dm.d % 2) return fail(SSA_ERR_CONSTRAINT, "rope needs an even head dim (d = %d)", dm.d);
  if (!qk_pair_interleaved(dm))
    return fail(SSA_ERR_UNSUPPORTED, "this shape packs Q/K in plain order; rotate with ssa_rope after ssa_qkv_project");
  KParams kp{};
  int num_sms = 0;
  if ((s = kparams(&kp, &num_sms)) != SSA_OK) return s;
  const int r = launch_qkv_gemm(dm, (int)dtype, x, dm.N, gn_scale, gn_shift, w_qkv, b_qkv, q, k, vt, kp,
                                static_cast<cudaStream_t>(stream), 1);
  if (r == 1) return fail(SSA_ERR_CUDA, "qkv_gemm: tensor map encoding failed");
  if (r) return cuda_fail(cudaGetLastError(), "qkv_gemm launch");
  return SSA_OK;
}

ssa_status ssa_attention(const uint16_t *q, const uint16_t *k, const uint16_t *vt, int B, int C, int N,
                         int num_heads, uint16_t *o, void *stream) {
  if (num_heads <= 0) return fail(SSA_ERR_CONSTRAINT, "num_heads must be positive");
  ssa_status s = check_shape(B, C, N, 1, 0, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if (!q || !k || !vt || !o) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o))
    return fail(SSA_ERR_ALIGNMENT, "q, k, vt and o must be 16-byte aligned");
  KParams kp{};
  int num_sms = 0;
  if ((s = kparams(&kp, &num_sms)) != SSA_OK) return s;
  const Dims dm = make_dims(B, C, N, 1, 1, num_heads);
  const int r = launch_attention(dm, q, k, vt, o, kp, static_cast<cudaStream_t>(stream));
  if (r == 1) return fail(SSA_ERR_CUDA, "attention: tensor map encoding failed");
  if (r) return cuda_fail(cudaGetLastError(), "attention launch");
  return SSA_OK;
}

ssa_status ssa_rope(uint16_t *q, uint16_t *k, int B, int C, int N, int num_heads, void *stream) {
  if (num_heads <= 0) return fail(SSA_ERR_CONSTRAINT, "num_heads must be positive");
  ssa_status s = check_shape(B, C, N, 1, 0, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if (!q || !k) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  const Dims dm = make_dims(B, C, N, 1, 1, num_heads);
  if (dm.d % 2) return fail(SSA_ERR_CONSTRAINT, "rope needs an even head dim (d = %d)", dm.d);
  if ((s = device_state(nullptr, nullptr)) != SSA_OK) return s;
  const cudaError_t e = launch_rope(dm, q, k, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSA_OK : cuda_fail(e, "rope launch");
}

ssa_status ssa_qk_norm(uint16_t *q, uint16_t *k, int B, int C, int N, int num_heads, ssa_dtype dtype,
                       const void *q_norm_weight, const void *k_norm_weight, void *stream) {
  if (num_heads <= 0) return fail(SSA_ERR_CONSTRAINT, "num_heads must be positive");
  ssa_status s = check_shape(B, C, N, 1, 0, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if ((s = check_dtype(dtype)) != SSA_OK) return s;
  if (!q || !k || !q_norm_weight || !k_norm_weight) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if ((s = device_state(nullptr, nullptr)) != SSA_OK) return s;
  const Dims dm = make_dims(B, C, N, 1, 1, num_heads);
  const cudaError_t e = launch_qk_norm(dm, (int)dtype, q, k, q_norm_weight, k_norm_weight,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSA_OK : cuda_fail(e, "qk norm launch");
}

ssa_status ssa_pack_rel_table(const void *table, ssa_dtype dtype, int H, int W, int num_heads, float *packed,
                              void *stream) {
  if (H <= 0 || W <= 0 || num_heads <= 0) return fail(SSA_ERR_CONSTRAINT, "sizes must be positive");
  ssa_status s = check_dtype(dtype);
  if (s != SSA_OK) return s;
  if ((s = check_rel_grid(H, W)) != SSA_OK) return s;
  if (!table || !packed) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if ((s = device_state(nullptr, nullptr)) != SSA_OK) return s;
  const cudaError_t e = launch_rel_table_pack((int)dtype, table, H, W, num_heads, packed,
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSA_OK : cuda_fail(e, "rel table pack launch");
}

ssa_status ssa_attention_ex(const uint16_t *q, const uint16_t *k, const uint16_t *vt, int B, int C, int H, int W,
                            int num_heads, int causal, const float *rel_packed, uint16_t *o, void *stream) {
  if (num_heads <= 0) return fail(SSA_ERR_CONSTRAINT, "num_heads must be positive");
  ssa_status s = check_shape(B, C, H, W, 0, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if (!q || !k || !vt || !o) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o))
    return fail(SSA_ERR_ALIGNMENT, "q, k, vt and o must be 16-byte aligned");
  if (rel_packed && (s = check_rel_grid(H, W)) != SSA_OK) return s;
  KParams kp{};
  int num_sms = 0;
  if ((s = kparams(&kp, &num_sms)) != SSA_OK) return s;
  const Dims dm = make_dims(B, C, H, W, 1, num_heads);
  const int r = launch_attention(dm, q, k, vt, o, kp, static_cast<cudaStream_t>(stream), causal ? 1 : 0, rel_packed);
  if (r == 1) return fail(SSA_ERR_CUDA, "attention: tensor map encoding failed");
  if (r) return cuda_fail(cudaGetLastError(), "attention launch");
  return SSA_OK;
}

ssa_status ssa_attention_ws(const uint16_t *q, const uint16_t *k, const uint16_t *vt, int B, int C, int H, int W,
                            int num_heads, int causal, const float *rel_packed, uint16_t *o, void *workspace,
                            size_t workspace_bytes, void *stream) {
  if (num_heads <= 0) return fail(SSA_ERR_CONSTRAINT, "num_heads must be positive");
  ssa_status s = check_shape(B, C, H, W, 0, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if (!q || !k || !vt || !o) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o))
    return fail(SSA_ERR_ALIGNMENT, "q, k, vt and o must be 16-byte aligned");
  if (rel_packed && (s = check_rel_grid(H, W)) != SSA_OK) return s;
  const Dims dm = make_dims(B, C, H, W, 1, num_heads);
  const size_t need = attention_scratch_bytes(dm);
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(SSA_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (workspace && workspace_bytes < need)
    return fail(SSA_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  KParams kp{};
  int num_sms = 0;
  if ((s = kparams(&kp, &num_sms)) != SSA_OK) return s;
  const int r = launch_attention(dm, q, k, vt, o, kp, static_cast<cudaStream_t>(stream), causal ? 1 : 0, rel_packed,
                                 (workspace && need) ? workspace : nullptr);
  if (r == 1) return fail(SSA_ERR_CUDA, "attention: tensor map encoding failed");
  if (r) return cuda_fail(cudaGetLastError(), "attention launch");
  return SSA_OK;
}

ssa_status ssa_out_project(const uint16_t *o, const uint16_t *w_o, const float *b_o, const void *x, int B, int C,
                           int H, int W, ssa_dtype dtype, void *out, void *stream) {
  ssa_status s = check_shape(B, C, H, W, 0, 0);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if ((s = check_dtype(dtype)) != SSA_OK) return s;
  if (!o || !w_o || !b_o || !x || !out) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(o) || !aligned16(w_o)) return fail(SSA_ERR_ALIGNMENT, "o and w_o must be 16-byte aligned");
  KParams kp{};
  int num_sms = 0;
  if ((s = kparams(&kp, &num_sms)) != SSA_OK) return s;
  const Dims dm = make_dims(B, C, H, W, 1, 1);
  const int r = launch_out_proj(dm, (int)dtype, o, w_o, b_o, x, out, kp, static_cast<cudaStream_t>(stream));
  if (r == 1) return fail(SSA_ERR_CUDA, "out_proj: tensor map encoding failed");
  if (r) return cuda_fail(cudaGetLastError(), "out_proj launch");
  return SSA_OK;
}

ssa_status ssa_get_device_status(void *stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t *err = nullptr;
  ssa_status s = device_state(&err, nullptr);
  if (s != SSA_OK) return s;
  uint32_t v = 0;
  e = cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (v) {
    const uint32_t zero = 0;
    e = cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    if (v & DEV_TIMEOUT) return fail(SSA_ERR_TIMEOUT, "a bounded device wait expired (error word 0x%x)", v);
    if (v & DEV_MISALIGNED)
      return fail(SSA_ERR_CUDA, "a kernel found its shared memory misaligned and did not run (error word 0x%x)", v);
    return fail(SSA_ERR_CUDA, "device error word 0x%x", v);
  }
  return SSA_OK;
}

ssa_status ssa_debug_timeout_probe(uint64_t timeout_ns, void *stream) {
  KParams kp{};
  ssa_status s = kparams(&kp, nullptr);
  if (s != SSA_OK) return s;
  kp.timeout_ns = timeout_ns;
  cudaError_t e = launch_timeout_probe(kp, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSA_OK : cuda_fail(e, "timeout probe launch");
}

}  // extern "C"

// ======================================================= allocation-free ==
// ssa_forward_static: the same block as ssa_forward, for callers that cannot
// allocate device memory -- code that runs where cudaMalloc is not allowed or
// not wanted once set-up is over (a fixed-memory real-time or embedded
// deployment, a plugin whose host forbids allocation on its execution path,
// a caller without access to any device allocator).  Its scratch (packed
// weights, GroupNorm scale/shift, Q, K, V^T, O) lives in one file-scope
// device array of SSA_STATIC_WORKSPACE_BYTES, which every device that loads
// this library's module keeps reserved until the process exits.
namespace ssa {
namespace {

constexpr size_t kStaticWsBytes = SSA_STATIC_WORKSPACE_BYTES;
__device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];
uint8_t *g_static_ws_ptr[kMaxDevices] = {};

// The array's name is only a host-side handle; its device address is looked
// up once per device (with that device current) and cached.
ssa_status static_workspace(uint8_t **ws) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SSA_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_static_ws_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static workspace)");
    g_static_ws_ptr[dev] = static_cast<uint8_t *>(p);
  }
  *ws = g_static_ws_ptr[dev];
  return SSA_OK;
}

}  // namespace
}  // namespace ssa

extern "C" ssa_status ssa_forward_static(const void *x, int B, int C, int H, int W, int num_groups,
                                         int num_heads, const void *norm_weight, const void *norm_bias,
                                         const void *q_weight, const void *q_bias, const void *k_weight,
                                         const void *k_bias, const void *v_weight, const void *v_bias,
                                         const void *out_weight, const void *out_bias, void *out,
                                         ssa_dtype dtype, void *stream) {
  ssa_status s = check_shape(B, C, H, W, num_groups, num_heads);
  if (s == kEmpty) return SSA_OK;
  if (s != SSA_OK) return s;
  if ((s = check_dtype(dtype)) != SSA_OK) return s;
  // Biases may be NULL (that projection has no bias), as for ssa_forward.
  const void *ptrs[] = {x, norm_weight, norm_bias, q_weight, k_weight, v_weight, out_weight, out};
  for (const void *p : ptrs)
    if (!p) return fail(SSA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(x) || !aligned16(out)) return fail(SSA_ERR_ALIGNMENT, "x and out must be 16-byte aligned");
  const Dims dm = make_dims(B, C, H, W, num_groups, num_heads);
  const WsLayout wl = ws_layout(dm, dtype, true);
  if (wl.total > kStaticWsBytes)
    return fail(SSA_ERR_WORKSPACE,
                "this problem needs %zu bytes of scratch, above the %zu-byte built-in limit of "
                "ssa_forward_static; call ssa_forward with a workspace instead",
                wl.total, kStaticWsBytes);
  KParams kp{};
  int num_sms = 0;
  if ((s = kparams(&kp, &num_sms)) != SSA_OK) return s;
  uint8_t *ws = nullptr;
  if ((s = static_workspace(&ws)) != SSA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t *w_qkv = reinterpret_cast<uint16_t *>(ws + wl.wqkv);
  float *b_qkv = reinterpret_cast<float *>(ws + wl.bqkv);
  uint16_t *w_o = reinterpret_cast<uint16_t *>(ws + wl.wo);
  float *b_o = reinterpret_cast<float *>(ws + wl.bo);
  cudaError_t e = launch_pack_weights(dm, (int)dtype, q_weight, q_bias, k_weight, k_bias, v_weight, v_bias,
                                      out_weight, out_bias, w_qkv, b_qkv, w_o, b_o, st);
  if (e != cudaSuccess) return cuda_fail(e, "pack launch");
  const Ptrs p{norm_weight, norm_bias, q_weight, q_bias, k_weight, k_bias, v_weight, v_bias, out_weight, out_bias};
  return run_block(dm, dtype, x, out, p, w_qkv, b_qkv, w_o, b_o, ws, wl, kp, num_sms, st);
}
