/*
 * ssa.h -- C ABI of the GB300 (sm_103a) spatial self-attention block.
 *
 * The block (tensortonic "diffusion-l03-spatial-self-attention", problem
 * statement and block equation):
 *
 *   Z = tokens(GN(x));  Q = Z Wq^T + bq;  K = Z Wk^T + bk;  V = Z Wv^T + bv;
 *   O_j = softmax(Q_j K_j^T / sqrt(d)) V_j;  out = x + image([O_1..O_n] Wo^T + bo)
 *
 * x is (B, C, H, W); GN has num_groups groups, eps 1e-5 and the affine
 * norm_weight / norm_bias; pixel (i, j) is token row i*W + j; d = C/num_heads
 * and head j owns channels [j*d, (j+1)*d).  The result has x's dtype.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated; the
 *    library never frees them.  Tensors are dense and contiguous.
 *  - x and out are NCHW.  Weights are (C_out, C_in) row-major, as a linear
 *    layer stores them; the ten parameters share x's dtype.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous on it: no host synchronisation, no
 *    host<->device copy and no allocation happens inside ssa_forward*,
 *    ssa_gn_stats, ssa_qkv_project, ssa_attention or ssa_out_project.
 *  - Argument errors are returned at once and nothing is launched.  Errors
 *    raised on the device (a bounded wait that expired) are latched in a
 *    device flag and returned by ssa_get_device_status().
 *  - The 16-bit tensor-core operand type is fp16 (fp32 accumulation, fp32
 *    softmax statistics).  Parameters and the projected Q, K, V must lie in
 *    fp16's range: magnitudes above 65504 become infinite and values below
 *    2^-24 become zero, without a status (GroupNorm keeps Z near unit scale,
 *    so this concerns parameters of extreme magnitude only).
 */
#ifndef SSA_H
#define SSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSA_F32 = 0,   /* IEEE binary32 */
    SSA_BF16 = 1   /* bfloat16 */
} ssa_dtype;

typedef enum {
    SSA_OK = 0,
    SSA_ERR_CONSTRAINT = 1,  /* C % num_groups, C % num_heads, C <= 0 or a size < 0
                                (E_CONSTRAINT in the HNDL attention operator doc) */
    SSA_ERR_DTYPE = 2,       /* dtype is not SSA_F32 / SSA_BF16 */
    SSA_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned */
    SSA_ERR_UNSUPPORTED = 4, /* head dim above 512, or a size beyond the grid limits */
    SSA_ERR_WORKSPACE = 5,   /* workspace missing or smaller than ssa_*workspace_size */
    SSA_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed (see ssa_last_error_string) */
    SSA_ERR_TIMEOUT = 7,     /* a bounded device-side wait expired (device flag) */
    SSA_ERR_NULL = 8         /* a required pointer is NULL */
} ssa_status;

typedef struct ssa_plan ssa_plan;

/* Empty problems: with B, H or W zero (C and its split into groups and heads
 * still valid) every entry point taking the problem shape does no work and
 * returns SSA_OK at once, without reading its pointers (which may be NULL);
 * the workspace sizes are 0. */

/* ---------------------------------------------------------------- block --- */

/* Bytes of device workspace ssa_forward needs for this problem (packed
 * weights, GN scale/shift, Q, K, V^T and O).  0 on a bad shape. */
size_t ssa_workspace_size(int B, int C, int H, int W, int num_groups, int num_heads,
                          ssa_dtype dtype);

/* One-shot forward of the whole block (the page's f(x, params, num_groups,
 * num_heads)).  q_bias, k_bias, v_bias and out_bias may be NULL: that
 * projection then has no bias (the HNDL attention operator page's qkv_bias /
 * out_bias flags; the block's own definition always has all four).  Packs the weights into `workspace` on every call, then runs
 * GN statistics -> QKV projection (GN affine + NCHW->token transpose fused in
 * its prologue) -> flash attention -> output projection (bias, residual and
 * NCHW store fused in its epilogue).  `out` may equal `x` (in place);
 * otherwise it must not overlap any input.  workspace: device memory of at
 * least ssa_workspace_size(...) bytes, 256-byte aligned, contents ignored. */
ssa_status ssa_forward(const void *x, int B, int C, int H, int W, int num_groups, int num_heads,
                       const void *norm_weight, const void *norm_bias,
                       const void *q_weight, const void *q_bias,
                       const void *k_weight, const void *k_bias,
                       const void *v_weight, const void *v_bias,
                       const void *out_weight, const void *out_bias,
                       void *out, ssa_dtype dtype,
                       void *workspace, size_t workspace_bytes, void *stream);

/* Steady state: the parameters are constants of a module.  ssa_plan_create
 * packs them once into device memory that the plan owns (cudaMalloc here and
 * only here; freed by ssa_plan_destroy) and enqueues the pack on `stream`.
 * The four biases may be NULL (no bias), as for ssa_forward. */
ssa_status ssa_plan_create(ssa_plan **plan, int C, int num_groups, int num_heads, ssa_dtype dtype,
                           const void *norm_weight, const void *norm_bias,
                           const void *q_weight, const void *q_bias,
                           const void *k_weight, const void *k_bias,
                           const void *v_weight, const void *v_bias,
                           const void *out_weight, const void *out_bias, void *stream);
size_t ssa_plan_workspace_size(const ssa_plan *plan, int B, int H, int W);
ssa_status ssa_forward_planned(const ssa_plan *plan, const void *x, int B, int H, int W, void *out,
                               void *workspace, size_t workspace_bytes, void *stream);
void ssa_plan_destroy(ssa_plan *plan);

/* Built-in scratch size of ssa_forward_static (48 MiB). */
#define SSA_STATIC_WORKSPACE_BYTES ((size_t)48 << 20)

/* Allocation-free form of ssa_forward, for callers that cannot allocate
 * device memory: code running where cudaMalloc is forbidden or unwanted after
 * set-up (fixed-memory real-time or embedded deployments, plugins whose host
 * bans allocation on the execution path, callers with no device allocator
 * at hand).  The paper has no counterpart; it is a packaging of the same
 * block.  Arguments and results are those of ssa_forward minus the
 * workspace: the scratch is one library-owned device array of
 * SSA_STATIC_WORKSPACE_BYTES, reserved on every device that loads the
 * library until the process exits.  Problems whose ssa_workspace_size()
 * exceeds it are rejected with SSA_ERR_WORKSPACE.  The first call on a
 * device looks the array's address up (cudaGetSymbolAddress); make that
 * first call before any stream capture.  Every call shares the one array and
 * it keeps the last call's contents (nothing in it needs to start at zero),
 * so calls whose work can overlap on the GPU -- on different streams, or from
 * different threads -- race on it: order them on one stream. */
ssa_status ssa_forward_static(const void *x, int B, int C, int H, int W, int num_groups, int num_heads,
                              const void *norm_weight, const void *norm_bias,
                              const void *q_weight, const void *q_bias,
                              const void *k_weight, const void *k_bias,
                              const void *v_weight, const void *v_bias,
                              const void *out_weight, const void *out_bias,
                              void *out, ssa_dtype dtype, void *stream);

/* ------------------------------------------------- steps of the hot path --- *
 * Each step of the block as its own launch, with the library's internal
 * layouts, for per-step checks and timing.  Let
 *   N = H*W,  d = C/num_heads,
 *   dp = d rounded up to 16 (to 32 when d > 256)   -- MMA-padded head dim,
 *   ldq = dp rounded up to 64,  ldn = N rounded up to 8,  ldc = C rounded up to 8.
 * Layouts (fp16 unless stated):
 *   mean, rstd   [B][G] fp32           gn_scale, gn_shift [B][C] fp32
 *   w_qkv        [3][h][dp][ldc]       rows q|k|v, head-major, zero rows past d;
 *                                      for an even d the q and k rows of a head
 *                                      may be pair-interleaved (row 2i = feature
 *                                      i, row 2i+1 = feature i + d/2) so that the
 *                                      projection can apply the rotary embedding
 *                                      in its epilogue -- produced and read only
 *                                      by the library, which decides this from
 *                                      the shape (d % 16 == 0, and C <= 512 or
 *                                      d == dp); q and k below keep the plain
 *                                      feature order either way
 *   b_qkv        [3][h][dp] fp32       zero past d, same row order as w_qkv, except
 *                                      that the v bias of padded feature d is 1
 *   w_o          [C][ldc]              b_o [C] fp32
 *   q, k         [B][h][N][ldq]        columns >= dp unspecified
 *   vt           [B][h][dp][ldn]       V transposed per head; columns >= N unspecified;
 *                                      when d < dp row d holds ones (the attention
 *                                      kernels read the softmax row sums from it;
 *                                      ssa_qkv_project writes it), rows past d+1 zero
 *   o            [B][N][ldc]           heads concatenated along channels
 */

/* GroupNorm statistics (per thread a running count, mean and M2 fed by the
 * two-pass statistics of each batch of loads; Chan merges across threads and
 * across the CTAs of a cluster): per (b, g) mean and rstd =
 * 1/sqrt(var_biased + 1e-5), then the folded per-(b, c) affine
 * gn_scale = rstd * norm_weight[c], gn_shift = norm_bias[c] - mean * gn_scale,
 * so that GN(x)[b, c, :] = gn_scale[b, c] * x[b, c, :] + gn_shift[b, c].
 * mean/rstd may be NULL. */
ssa_status ssa_gn_stats(const void *x, int B, int C, int N, int num_groups, ssa_dtype dtype,
                        const void *norm_weight, const void *norm_bias,
                        float *mean, float *rstd, float *gn_scale, float *gn_shift, void *stream);

/* Cast and pack the projection weights into the layouts above (a NULL bias
 * packs as zeros). */
ssa_status ssa_pack_weights(int C, int num_heads, ssa_dtype dtype,
                            const void *q_weight, const void *q_bias,
                            const void *k_weight, const void *k_bias,
                            const void *v_weight, const void *v_bias,
                            const void *out_weight, const void *out_bias,
                            uint16_t *w_qkv, float *b_qkv, uint16_t *w_o, float *b_o, void *stream);

/* Q, K, V^T = tokens(gn_scale * x + gn_shift) w_qkv^T + b_qkv, written in the
 * q / k / vt layouts (tcgen05 GEMM, M = pixels, N = 3*h*dp, K = C). */
ssa_status ssa_qkv_project(const void *x, int B, int C, int H, int W, int num_heads, ssa_dtype dtype,
                           const float *gn_scale, const float *gn_shift,
                           const uint16_t *w_qkv, const float *b_qkv,
                           uint16_t *q, uint16_t *k, uint16_t *vt, void *stream);

/* ssa_qkv_project with the rotary embedding of the variants (HNDL attention
 * operator page, Rotary embeddings paragraph: rotate-half over the head dim,
 * base 10000) applied to Q and K in the projection's epilogue, before their
 * single rounding to fp16.  The angle t * 10000^(-2i/d) is formed from an
 * fp64 frequency (two fp32 parts) and reduced to [-pi, pi] before cos/sin,
 * so it is exact to about 1e-6 rad at every position.  SSA_ERR_CONSTRAINT for
 * an odd head dim; SSA_ERR_UNSUPPORTED for shapes whose Q/K rows are packed in
 * plain order (head dims that are not a multiple of 16; there:
 * ssa_qkv_project, then ssa_rope). */
ssa_status ssa_qkv_project_rope(const void *x, int B, int C, int H, int W, int num_heads, ssa_dtype dtype,
                                const float *gn_scale, const float *gn_shift,
                                const uint16_t *w_qkv, const float *b_qkv,
                                uint16_t *q, uint16_t *k, uint16_t *vt, void *stream);

/* O_j = softmax(Q_j K_j^T / sqrt(d)) V_j for every (b, head), never forming
 * the N x N matrix; o receives the heads side by side (layout above). */
ssa_status ssa_attention(const uint16_t *q, const uint16_t *k, const uint16_t *vt,
                         int B, int C, int N, int num_heads, uint16_t *o, void *stream);

/* out = x + image(o w_o^T + b_o), rounded once to x's dtype (tcgen05 GEMM,
 * M = pixels, N = C, K = C; bias, residual and the NCHW store in the
 * epilogue).  out may equal x. */
ssa_status ssa_out_project(const uint16_t *o, const uint16_t *w_o, const float *b_o,
                           const void *x, int B, int C, int H, int W, ssa_dtype dtype,
                           void *out, void *stream);

/* ------------------------------------------------------------ variants --- */

/* Attention variants of the HNDL "attention" operator page (parameter table
 * and its Masking, Relative position bias and Rotary embeddings paragraphs),
 * applied to the block's token sequence: T = H*W tokens, token t = pixel
 * (t / W, t % W); and the query-key RMS normalisation of the vit-pytorch
 * "simple_vit_with_qk_norm" page.  The block's own definition has none of them; an all-zero
 * ssa_options (or NULL) is the block.  A = softmax(Q K^T / sqrt(d) + bias +
 * mask) per head, after the optional rotation of Q and K. */
typedef struct ssa_options {
    int causal;                /* 1: token t attends only to tokens <= t (the strictly
                                  upper triangle of the scores is -inf) */
    int rope;                  /* 1: rotate each Q and K head by its token position,
                                  rotate-half convention over the full head dim, base
                                  10000, angles in fp32; needs an even head dim
                                  (SSA_ERR_CONSTRAINT otherwise) */
    const void *rel_pos_table; /* NULL, or the learned 2-D relative-position bias table
                                  [(2H-1)*(2W-1)][num_heads] in x's dtype (device,
                                  16-byte aligned): entry ((rq - rk + H - 1) * (2W - 1)
                                  + (cq - ck + W - 1), j) is added to head j's scaled
                                  logit of query (rq, cq) and key (rk, ck) */
    const void *q_norm_weight; /* NULL, or (with k_norm_weight) query-key RMS normalisation
                                  (vit-pytorch simple_vit_with_qk_norm.py, RMSNorm class):
                                  each Q head row becomes x / max(||x||, 1e-12) * sqrt(d)
                                  * q_norm_weight[head][:]; [num_heads][d], x's dtype,
                                  device; applied before the rotation */
    const void *k_norm_weight; /* the same for K */
} ssa_options;

/* Workspace of ssa_forward_ex (ssa_workspace_size plus the packed table). */
size_t ssa_workspace_size_ex(int B, int C, int H, int W, int num_groups, int num_heads,
                             ssa_dtype dtype, const ssa_options *opt);

/* ssa_forward with the variants: the rotation runs in the projection's
 * epilogue (or, with the query-key norm, or for shapes whose Q/K rows are
 * packed in plain order, as a separate pass after it), the table is packed
 * into the workspace, and the
 * attention kernels add the bias and apply the mask to their logits, skipping
 * key tiles that the causal mask removes entirely. */
ssa_status ssa_forward_ex(const void *x, int B, int C, int H, int W, int num_groups, int num_heads,
                          const void *norm_weight, const void *norm_bias,
                          const void *q_weight, const void *q_bias,
                          const void *k_weight, const void *k_bias,
                          const void *v_weight, const void *v_bias,
                          const void *out_weight, const void *out_bias,
                          void *out, ssa_dtype dtype, const ssa_options *opt,
                          void *workspace, size_t workspace_bytes, void *stream);

/* Planned form of ssa_forward_ex (the table is packed into the workspace on
 * every call; it is small). */
size_t ssa_plan_workspace_size_ex(const ssa_plan *plan, int B, int H, int W, const ssa_options *opt);
ssa_status ssa_forward_planned_ex(const ssa_plan *plan, const void *x, int B, int H, int W, void *out,
                                  const ssa_options *opt, void *workspace, size_t workspace_bytes,
                                  void *stream);

/* Step entry points of the variants.
 * ssa_rope: rotates q and k (q/k layout above, N tokens) in place.
 * ssa_pack_rel_table: table [(2H-1)(2W-1)][num_heads] (x's dtype) ->
 *   packed [num_heads][(2H-1)(2W-1)] fp32, each entry times log2(e).
 * ssa_attention_ex: ssa_attention over the H x W token grid with the causal
 *   mask (0/1) and the packed table (NULL: none). */
ssa_status ssa_rope(uint16_t *q, uint16_t *k, int B, int C, int N, int num_heads, void *stream);
/* ssa_qk_norm: the query-key RMS normalisation of q and k in place. */
ssa_status ssa_qk_norm(uint16_t *q, uint16_t *k, int B, int C, int N, int num_heads, ssa_dtype dtype,
                       const void *q_norm_weight, const void *k_norm_weight, void *stream);
ssa_status ssa_pack_rel_table(const void *table, ssa_dtype dtype, int H, int W, int num_heads,
                              float *packed, void *stream);
ssa_status ssa_attention_ex(const uint16_t *q, const uint16_t *k, const uint16_t *vt,
                            int B, int C, int H, int W, int num_heads, int causal,
                            const float *rel_packed, uint16_t *o, void *stream);

/* Head dimension 512 (padded) runs as two-CTA clusters, one per resident SM
 * pair.  With scratch, the (query tile, key tile) work of a call can be cut
 * into equal pieces, one per cluster, so no SM pair idles in a partial last
 * wave; a query tile shared by several clusters is finished by its last
 * contributor, which merges the others' fp32 parts (each rescaled to the
 * common row maximum, as in the online softmax) -- the result equals the
 * unsplit one up to rounding.
 *
 * ssa_attention_workspace_size: bytes of that scratch for this shape (0 when
 *   the head dim is not padded to 512, or the shape is invalid).  The
 *   ssa_forward* workspaces already include it.
 * ssa_attention_ws: ssa_attention_ex with that scratch: `workspace` (device,
 *   256-byte aligned, >= the size above, caller-owned, contents ignored) or
 *   NULL to run whole query tiles.  SSA_ERR_WORKSPACE when too small.
 * ssa_set_attention_split: when the scratch is used -- SSA_SPLIT_AUTO (when
 *   there are more query tiles than resident clusters and no causal mask:
 *   measured to pay there), SSA_SPLIT_ALWAYS, SSA_SPLIT_NEVER.  Process-wide,
 *   for launches after the call; SSA_ERR_CONSTRAINT for another value. */
#define SSA_SPLIT_AUTO 0
#define SSA_SPLIT_ALWAYS 1
#define SSA_SPLIT_NEVER 2
size_t ssa_attention_workspace_size(int B, int C, int H, int W, int num_heads);
ssa_status ssa_attention_ws(const uint16_t *q, const uint16_t *k, const uint16_t *vt,
                            int B, int C, int H, int W, int num_heads, int causal,
                            const float *rel_packed, uint16_t *o, void *workspace,
                            size_t workspace_bytes, void *stream);
ssa_status ssa_set_attention_split(int policy);

/* --------------------------------------------------------- diagnostics --- */

/* Synchronises `stream`, then reads and clears the device error flag:
 * SSA_OK, SSA_ERR_TIMEOUT (a bounded wait expired; the kernel released its
 * tensor memory and returned) or SSA_ERR_CUDA (a launch or execution error). */
ssa_status ssa_get_device_status(void *stream);

/* Limit of every device-side spin wait, in nanoseconds (default 2e9).
 * Applies to launches made after the call. */
void ssa_set_wait_timeout_ns(uint64_t ns);

/* Launches one CTA whose mbarrier wait can never complete (nothing arrives),
 * bounded by `timeout_ns`; the wait expires, latches SSA_ERR_TIMEOUT and the
 * kernel returns.  Exercises the timeout path without faulting the GPU. */
ssa_status ssa_debug_timeout_probe(uint64_t timeout_ns, void *stream);

/* Test hook for the device-side timeout path of the block's own kernels.
 * After this call the TMA producers of the kernels named in kernel_mask
 * (SSA_STALL_QKV, SSA_STALL_ATTENTION for head dims up to 256,
 * SSA_STALL_OUT_PROJ) stop after after_loads loads of a launch, as if the
 * memory system had stalled: their consumers' bounded waits then expire, the
 * kernel latches SSA_ERR_TIMEOUT, drains its copies and MMAs, frees its tensor
 * memory and returns, and ssa_get_device_status() reports it.  No fault is
 * involved.  after_loads = 0 turns the hook off.  Process-wide; applies to
 * launches after the call.  (Head dim 512 -- the two-CTA cluster kernel -- is
 * not covered.) */
#define SSA_STALL_QKV 1u
#define SSA_STALL_ATTENTION 2u
#define SSA_STALL_OUT_PROJ 4u
void ssa_debug_set_producer_stall(uint32_t kernel_mask, uint32_t after_loads);

/* Human-readable detail of the last error returned on this thread. */
const char *ssa_last_error_string(void);

/* Number of kernel launches one ssa_forward / ssa_forward_planned call makes. */
int ssa_launches_per_forward(int planned);

#ifdef __cplusplus
}
#endif

#endif /* SSA_H */
