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
// x / max(||x||_2, 1e-12) * sqrt(d) * gamma[head][:], eight lanes per row, fp32
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

// One thread per (row, pair i), consecutive threads on consecutive pairs of a
// row; the angle bases theta_i = 10000^(-2i/d) come from a table each block
// builds once in shared memory, and the index arithmetic is 32-bit.
// t0: the token position of row 0 of this launch (launches cover chunks of
// rows, so that total < 2^31).
__global__ void rope_kernel(uint16_t *q, uint16_t *k, int total, int N, int ldq, int d, int t0) {
  __shared__ float theta[256];
  pdl_trigger();
  const int hd = d / 2;
  const float l2base = -2.0f * 13.287712379549449f / (float)d;  // -2 log2(10000) / d
  for (int i = threadIdx.x; i < hd; i += blockDim.x) theta[i] = exp2f(l2base * (float)i);
  __syncthreads();
  pdl_wait();
  // Unsigned: total < 2^31 and the stride <= 2^20, so idx + stride never wraps.
  for (unsigned idx = blockIdx.x * blockDim.x + threadIdx.x; idx < (unsigned)total; idx += gridDim.x * blockDim.x) {
    const int row = (int)(idx / (unsigned)hd);
    const int i = (int)idx - row * hd;
    const float t = (float)((row + t0) % N);
    float sn, cs;
    sincosf(t * theta[i], &sn, &cs);
    uint16_t *pq = q + (long long)row * ldq;
    uint16_t *pk = k + (long long)row * ldq;
    const float qa = op_to_float(pq[i]), qb = op_to_float(pq[hd + i]);
    const float ka = op_to_float(pk[i]), kb = op_to_float(pk[hd + i]);
    pq[i] = op_bits(qa * cs - qb * sn);
    pq[hd + i] = op_bits(qb * cs + qa * sn);
    pk[i] = op_bits(ka * cs - kb * sn);
    pk[hd + i] = op_bits(kb * cs + ka * sn);
  }
}

template <int DT>
__device__ __forceinline__ float ld_x(const void *p, long long i) {
  if (DT == 0) return reinterpret_cast<const float *>(p)[i];
  const unsigned short u = reinterpret_cast<const unsigned short *>(p)[i];
  return __uint_as_float(((uint32_t)u) << 16);
}

// Eight lanes per row (Q rows, then K rows), so a warp touches four rows'
// contiguous bytes: lane j takes the 16-byte pieces j, j + 8, ... of the row
// when the head dim is a multiple of 8 (rows start 128-byte aligned), else
// elements j, j + 8, ...; the sum of squares is combined by shuffles inside
// the group of eight and the row is scaled on a second read (from L1).
template <int DT>
// hd0: the head of row 0 of this launch (launches cover chunks of whole
// heads' rows, so that 16 * rows < 2^31).
__global__ void qk_norm_kernel(uint16_t *q, uint16_t *k, int rows, int N, int h, int ldq, int d, const void *qg,
                               const void *kg, int hd0) {
  pdl_trigger();
  pdl_wait();
  const int wr = (blockIdx.x * blockDim.x + threadIdx.x) >> 3;  // uniform within a group of eight lanes
  const int j = threadIdx.x & 7;
  if (wr >= 2 * rows) return;
  const unsigned gmask = 0xFFu << (threadIdx.x & 24);
  const int which = wr >= rows ? 1 : 0;
  const int row = wr - which * rows;
  const int head = (hd0 + row / N) % h;
  uint16_t *p = (which ? k : q) + (long long)row * ldq;
  const void *g = which ? kg : qg;
  const long long g0 = (long long)head * d;
  const bool vec = (d % 8) == 0;
  float ss = 0.f;
  if (vec) {
    for (int e = 8 * j; e < d; e += 64) {
      const uint4 u = *reinterpret_cast<const uint4 *>(p + e);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float a = op_to_float((uint16_t)(w[m] & 0xFFFFu)), b = op_to_float((uint16_t)(w[m] >> 16));
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
    }
  } else {
    for (int e = j; e < d; e += 8) {
      const float v = op_to_float(p[e]);
      ss = fmaf(v, v, ss);
    }
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) ss += __shfl_xor_sync(gmask, ss, o);
  const float scale = sqrtf((float)d) / fmaxf(sqrtf(ss), 1e-12f);
  if (vec) {
    for (int e = 8 * j; e < d; e += 64) {
      uint4 u = *reinterpret_cast<const uint4 *>(p + e);
      uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float a = op_to_float((uint16_t)(w[m] & 0xFFFFu)) * scale * ld_x<DT>(g, g0 + e + 2 * m);
        const float b = op_to_float((uint16_t)(w[m] >> 16)) * scale * ld_x<DT>(g, g0 + e + 2 * m + 1);
        w[m] = (uint32_t)op_bits(a) | ((uint32_t)op_bits(b) << 16);
      }
      u.x = w[0]; u.y = w[1]; u.z = w[2]; u.w = w[3];
      *reinterpret_cast<uint4 *>(p + e) = u;
    }
  } else {
    for (int e = j; e < d; e += 8) p[e] = op_bits(op_to_float(p[e]) * scale * ld_x<DT>(g, g0 + e));
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
  const int hd = dm.d / 2;
  if (hd <= 0 || hd > 256) return cudaErrorInvalidValue;
  // Chunks of at most 2^30 pairs (whole rows); one launch for all but the
  // largest problems.
  const long long rows = (long long)dm.B * dm.h * dm.N;
  const long long per = (1LL << 30) / hd;
  for (long long r0 = 0; r0 < rows; r0 += per) {
    const long long n = rows - r0 < per ? rows - r0 : per;
    (void)launch_k(rope_kernel, dim3(grid_for(n * hd)), dim3(256), 0, st, q + r0 * dm.ldq, k + r0 * dm.ldq,
                   (int)(n * hd), dm.N, dm.ldq, dm.d, (int)(r0 % dm.N));
  }
  return cudaGetLastError();
}

cudaError_t launch_qk_norm(const Dims &dm, int dtype, uint16_t *q, uint16_t *k, const void *q_gamma,
                           const void *k_gamma, cudaStream_t st) {
  // Chunks of whole heads' rows with 16 * rows < 2^31 (one launch for all
  // but the largest problems): eight lanes per row, Q and K.
  const long long rows = (long long)dm.B * dm.h * dm.N;
  const long long per = ((1LL << 27) - 1) / dm.N * dm.N;  // N <= 2^23 here, so per >= N
  for (long long r0 = 0; r0 < rows; r0 += per) {
    const long long n = rows - r0 < per ? rows - r0 : per;
    const dim3 grid((unsigned)((16 * n + 127) / 128));
    const int hd0 = (int)((r0 / dm.N) % dm.h);
    if (dtype == 0)
      (void)launch_k(qk_norm_kernel<0>, grid, dim3(128), 0, st, q + r0 * dm.ldq, k + r0 * dm.ldq, (int)n, dm.N, dm.h,
                     dm.ldq, dm.d, q_gamma, k_gamma, hd0);
    else
      (void)launch_k(qk_norm_kernel<1>, grid, dim3(128), 0, st, q + r0 * dm.ldq, k + r0 * dm.ldq, (int)n, dm.N, dm.h,
                     dm.ldq, dm.d, q_gamma, k_gamma, hd0);
  }
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
