// internal.h -- host-side declarations shared by the launcher and the kernel
// translation units: derived sizes/layouts and the per-kernel launch wrappers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ssa {

// Sizes and internal layouts derived from one problem.
//   dp  : head dim padded to the MMA K granularity (16; 32 above 256 so that
//         the two output halves each stay a multiple of 16)
//   ldq : row pitch (elements) of Q and K, a whole number of 64-element
//         swizzle rows
//   ldn : row pitch of V^T (pixels), 16-byte aligned
//   ldc : row pitch of packed weights and O (channels), 16-byte aligned
//   n_oc, d_o : the attention output of one head is produced in n_oc slices
//         of d_o columns (one slice per CTA); n_oc = 2 when dp > 256
struct Dims {
  int B, C, H, W, N, G, h, d, dp, ldq, ldn, ldc, n_oc, d_o, ntot;
};

inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

inline Dims make_dims(int B, int C, int H, int W, int G, int h) {
  Dims s{};
  s.B = B; s.C = C; s.H = H; s.W = W; s.N = H * W; s.G = G; s.h = h;
  s.d = (h > 0) ? C / h : 0;
  s.dp = (s.d > 256) ? round_up(s.d, 32) : round_up(s.d, 16);
  s.ldq = round_up(s.dp, 64);
  s.ldn = round_up(s.N, 8);
  s.ldc = round_up(C, 8);
  s.n_oc = (s.dp > 256) ? 2 : 1;
  s.d_o = s.dp / s.n_oc;
  s.ntot = 3 * h * s.dp;
  return s;
}

// Q/K packing.  When this returns true the Q and K rows of each head in the
// packed weight (and bias) are pair-interleaved: packed row 2i holds feature i
// and row 2i+1 feature i + d/2 (i < d/2), rows >= d are zero.  The rotary
// embedding (rotate-half) pairs feature i with feature i + d/2, so every pair
// then sits in two adjacent accumulator columns and the projection's epilogue
// can rotate it in registers; the epilogue writes every feature back to its
// own place, so Q and K in memory keep the plain layout.  True for an even
// head dim that is a multiple of 16 (so both halves of every 8-pair piece
// start 16-byte aligned) when the resident projection kernel runs
// (C <= 512), or, for the other kernel, when the head has no padding.
bool qk_pair_interleaved(const Dims &dm);

// Arguments every pipelined kernel receives for its bounded waits.
struct KParams {
  uint32_t *err;        // device error word
  uint64_t timeout_ns;  // limit of one spin wait
  uint32_t stall_mask;  // test hook: kernels whose TMA producers stop early (STALL_* bits)
  uint32_t stall_after; // ... after this many loads
};
enum : uint32_t { STALL_QKV = 1, STALL_ATTENTION = 2, STALL_OUT_PROJ = 4 };
inline uint32_t stall_for(const KParams &kp, uint32_t bit) { return (kp.stall_mask & bit) ? kp.stall_after : 0u; }

// cuTensorMapEncodeTiled through the runtime's driver entry point.
// dims/strides innermost first; strides in bytes for dims 1..rank-1.
CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                      const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                      CUtensorMapSwizzle swz);

// Programmatic dependent launch.  pdl_trigger lets the next kernel of the
// stream be scheduled (its CTAs then wait in pdl_wait); pdl_wait blocks until
// the previous kernel of the stream has completed and its memory is visible
// (it returns at once when the launch had no programmatic dependency).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches `kern` with programmatic dependent launch allowed: its CTAs may be
// scheduled while the previous kernel of the stream still runs; every kernel
// of this library waits (pdl_wait) before its first global memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---- launch wrappers (each returns the launch error, if any) ----
cudaError_t launch_gn_stats(const void *x, int B, int C, int N, int G, int dtype, const void *gw,
                            const void *gb, float *mean, float *rstd, float *a, float *s, int num_sms,
                            cudaStream_t st);

cudaError_t launch_pack_weights(const Dims &dm, int dtype, const void *wq, const void *bq, const void *wk,
                                const void *bk, const void *wv, const void *bv, const void *wo,
                                const void *bo, uint16_t *w_qkv, float *b_qkv, uint16_t *w_o, float *b_o,
                                cudaStream_t st);

// Copy x [B][C][N] into [B][C][ldx] with ldx*esize a multiple of 16 bytes.
cudaError_t launch_pad_x(const void *x, int B, int C, int N, int ldx, int esize, void *dst, cudaStream_t st);

// Returns 0 on success, 1 when a tensor map could not be encoded, 2 on a launch error.
// rope: Q and K are rotated in the epilogue (requires qk_pair_interleaved(dm)).
int launch_qkv_gemm(const Dims &dm, int dtype, const void *x, int ldx, const float *ga, const float *gs,
                    const uint16_t *w_qkv, const float *b_qkv, uint16_t *q, uint16_t *k, uint16_t *vt,
                    const KParams &kp, cudaStream_t st, int rope = 0);

// causal: keys after the query token are masked; rel: NULL or the packed
// relative-position table [h][(2H-1)(2W-1)] fp32 (times log2 e) over the
// dm.H x dm.W token grid.
int launch_attention(const Dims &dm, const uint16_t *q, const uint16_t *k, const uint16_t *vt, uint16_t *o,
                     const KParams &kp, cudaStream_t st, int causal = 0, const float *rel = nullptr,
                     void *scratch = nullptr);
// Scratch the attention step can use to balance its work (head dim 512 only;
// 0 otherwise): given to launch_attention it lets a query tile be split
// between SM pairs.  Depends only on the shape.
size_t attention_scratch_bytes(const Dims &dm);
// Policy for using that scratch (ssa_set_attention_split): 0 auto, 1 always,
// 2 never.
int attention_split_policy();

// Rotary embedding of Q and K in place (q/k layout), token position = row.
cudaError_t launch_rope(const Dims &dm, uint16_t *q, uint16_t *k, cudaStream_t st);
// Query-key RMS normalisation of Q and K in place; gammas [h][d] in x's dtype.
cudaError_t launch_qk_norm(const Dims &dm, int dtype, uint16_t *q, uint16_t *k, const void *q_gamma,
                           const void *k_gamma, cudaStream_t st);
// Relative-position table [(2H-1)(2W-1)][heads] (x's dtype) -> packed.
cudaError_t launch_rel_table_pack(int dtype, const void *table, int H, int W, int heads, float *packed,
                                  cudaStream_t st);

int launch_out_proj(const Dims &dm, int dtype, const uint16_t *o, const uint16_t *w_o, const float *b_o,
                    const void *x, void *out, const KParams &kp, cudaStream_t st);

cudaError_t launch_timeout_probe(const KParams &kp, cudaStream_t st);

}  // namespace ssa
