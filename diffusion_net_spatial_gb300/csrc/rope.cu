// rope.cu -- attention variants that act outside the attention kernel
// (HNDL "attention" operator page, Rotary embeddings and Relative position
// bias paragraphs), on the block's token sequence (token t = pixel i*W + j).
//
// rope_kernel: Q and K rows rotated in place by their token position, per
// head, with the rotate-half convention over the full head dim and base
// 10000:  theta_i = 10000^(-2i/d),  angle = t * theta_i  (i < d/2),
//   x'[i]       = x[i] cos(angle) - x[i + d/2] sin(angle)
//   x'[i + d/2] = x[i + d/2] cos(angle) + x[i] sin(angle).
// As on the page the angles are built in fp32; the rotation is applied in
// fp32 to the fp16 Q/K values and rounded back to fp16 once.
//
// qk_norm_kernel: query-key RMS normalisation (vit-pytorch
// simple_vit_with_qk_norm.py, RMSNorm class): each head's Q and K rows become
// x / max(||x||_2, 1e-12) * sqrt(d) * gamma[head][:], one warp per row, fp32
// sum of squares, rounded back to fp16 once.
//
// rel_table_pack_kernel: the learned table [(2H-1)(2W-1)][heads] in x's dtype
// becomes one fp32 row per head, pre-multiplied by log2(e) so that the
// attention kernels add it directly to their base-2 logits.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace {

__global__ void rope_kernel(uint16_t *q, uint16_t *k, long long rows, int N, int ldq, int d) {
  pdl_trigger();
  pdl_wait();
  const int hd = d / 2;
  const long long total = rows * hd;
  const float l2base = -2.0f * 13.287712379549449f / (float)d;  // -2 log2(10000) / d
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long row = idx / hd;
    const int i = (int)(idx - row * hd);
    const int t = (int)(row % N);
    const float theta = exp2f(l2base * (float)i);
    float sn, cs;
    sincosf((float)t * theta, &sn, &cs);
    uint16_t *bufs[2] = {q, k};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      uint16_t *p = bufs[u] + row * ldq;
      const float a = op_to_float(p[i]);
      const float b = op_to_float(p[hd + i]);
      p[i] = op_bits(a * cs - b * sn);
      p[hd + i] = op_bits(b * cs + a * sn);
    }
  }
}

template <int DT>
__device__ __forceinline__ float ld_x(const void *p, long long i) {
  if (DT == 0) return reinterpret_cast<const float *>(p)[i];
  const unsigned short u = reinterpret_cast<const unsigned short *>(p)[i];
  return __uint_as_float(((uint32_t)u) << 16);
}

template <int DT>
__global__ void qk_norm_kernel(uint16_t *q, uint16_t *k, long long rows, int N, int h, int ldq, int d,
                               const void *qg, const void *kg) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  const float sd = sqrtf((float)d);
  for (long long wr = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5); wr < 2 * rows; wr += nwarps) {
    const int which = wr >= rows ? 1 : 0;
    const long long row = wr - which * rows;
    const int head = (int)((row / N) % h);
    uint16_t *p = (which ? k : q) + row * ldq;
    const void *g = which ? kg : qg;
    float ss = 0.f;
    for (int e = lane; e < d; e += 32) {
      const float v = op_to_float(p[e]);
      ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    const float scale = sd / fmaxf(sqrtf(ss), 1e-12f);
    for (int e = lane; e < d; e += 32)
      p[e] = op_bits(op_to_float(p[e]) * scale * ld_x<DT>(g, (long long)head * d + e));
  }
}

template <int DT>
__global__ void rel_table_pack_kernel(const void *table, int entries, int heads, float *packed) {
  pdl_trigger();
  pdl_wait();
  const long long total = (long long)entries * heads;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int hh = (int)(idx / entries);
    const long long e = idx - (long long)hh * entries;
    float v;
    if (DT == 0) {
      v = reinterpret_cast<const float *>(table)[e * heads + hh];
    } else {
      const unsigned short u = reinterpret_cast<const unsigned short *>(table)[e * heads + hh];
      v = __uint_as_float(((uint32_t)u) << 16);
    }
    packed[idx] = v * 1.4426950408889634f;
  }
}

int grid_for(long long work) {
  long long g = (work + 255) / 256;
  if (g > 4096) g = 4096;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

cudaError_t launch_rope(const Dims &dm, uint16_t *q, uint16_t *k, cudaStream_t st) {
  const long long rows = (long long)dm.B * dm.h * dm.N;
  (void)launch_k(rope_kernel, dim3(grid_for(rows * (dm.d / 2))), dim3(256), 0, st, q, k, rows, dm.N, dm.ldq, dm.d);
  return cudaGetLastError();
}

cudaError_t launch_qk_norm(const Dims &dm, int dtype, uint16_t *q, uint16_t *k, const void *q_gamma,
                           const void *k_gamma, cudaStream_t st) {
  const long long rows = (long long)dm.B * dm.h * dm.N;
  long long blocks = (2 * rows + 7) / 8;  // 8 warps (rows) per block
  if (blocks > 8192) blocks = 8192;
  if (dtype == 0)
    (void)launch_k(qk_norm_kernel<0>, dim3((int)blocks), dim3(256), 0, st, q, k, rows, dm.N, dm.h, dm.ldq, dm.d, q_gamma, k_gamma);
  else
    (void)launch_k(qk_norm_kernel<1>, dim3((int)blocks), dim3(256), 0, st, q, k, rows, dm.N, dm.h, dm.ldq, dm.d, q_gamma, k_gamma);
  return cudaGetLastError();
}

cudaError_t launch_rel_table_pack(int dtype, const void *table, int H, int W, int heads, float *packed,
                                  cudaStream_t st) {
  const int entries = (2 * H - 1) * (2 * W - 1);
  if (dtype == 0)
    (void)launch_k(rel_table_pack_kernel<0>, dim3(grid_for((long long)entries * heads)), dim3(256), 0, st, table, entries, heads, packed);
  else
    (void)launch_k(rel_table_pack_kernel<1>, dim3(grid_for((long long)entries * heads)), dim3(256), 0, st, table, entries, heads, packed);
  return cudaGetLastError();
}

}  // namespace ssa
