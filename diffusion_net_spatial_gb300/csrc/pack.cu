// pack.cu -- weight packing and the x pitch fix-up.
//
// The Q, K and V projections are linear layers (tensortonic
// "diffusion-l03-spatial-self-attention", problem statement: "used as in a
// linear layer"), so their (C_out, C_in) weights already have the K-major
// (C_in contiguous) layout the tensor cores read.  Packing only casts them to
// fp16, stacks [Wq; Wk; Wv] into one 3*h*dp x C operand (one GEMM forms Q, K
// and V together) with each head's rows padded from d to dp by zero rows, and
// keeps the biases in fp32.  When qk_pair_interleaved() holds, the Q and K
// rows of a head are ordered feature 0, d/2, 1, d/2 + 1, ... (the rotary
// embedding's pairs side by side); V rows keep their order, and when d < dp
// V's feature d gets weight 0 and bias 1, a column of ones that lets the
// attention's P V product return the softmax row sums.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace {

template <int DT>
__device__ __forceinline__ float ld_param(const void *p, long long i) {
  if (DT == 0) return reinterpret_cast<const float *>(p)[i];
  const unsigned short u = reinterpret_cast<const unsigned short *>(p)[i];
  return __uint_as_float(((uint32_t)u) << 16);
}

__device__ __forceinline__ uint16_t to_half_bits(float v) { return op_bits(v); }

template <int DT>
__global__ void pack_kernel(int C, int h, int d, int dp, int ldc, int inter, const void *wq, const void *bq,
                            const void *wk, const void *bk, const void *wv, const void *bv, const void *wo,
                            const void *bo, uint16_t *w_qkv, float *b_qkv, uint16_t *w_o, float *b_o) {
  pdl_trigger();
  pdl_wait();
  const long long n_qkv = 3LL * h * dp * ldc;
  const long long n_o = (long long)C * ldc;
  const long long total = n_qkv + n_o;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    if (i < n_qkv) {
      const int c = (int)(i % ldc);
      const long long row = i / ldc;             // (sec * h + head) * dp + e
      const int e = (int)(row % dp);
      const int head = (int)((row / dp) % h);
      const int sec = (int)(row / ((long long)dp * h));
      // feature of packed row e: pair-interleaved for Q and K (see above)
      const int f = (inter && sec < 2 && e < d) ? ((e & 1) ? d / 2 + (e >> 1) : (e >> 1)) : e;
      float v = 0.f;
      if (e < d && c < C) {
        const void *w = sec == 0 ? wq : (sec == 1 ? wk : wv);
        v = ld_param<DT>(w, (long long)(head * d + f) * C + c);
      }
      w_qkv[i] = to_half_bits(v);
      if (c == 0) {
        float bv_ = 0.f;
        if (e < d) {
          const void *bb = sec == 0 ? bq : (sec == 1 ? bk : bv);
          bv_ = bb ? ld_param<DT>(bb, head * d + f) : 0.f;  // no bias: zero
        } else if (sec == 2 && e == d) {
          bv_ = 1.f;  // V's first padding feature is 1 for every token: P V then carries the row sums
        }
        b_qkv[row] = bv_;
      }
    } else {
      const long long j = i - n_qkv;
      const int c = (int)(j % ldc);
      const int co = (int)(j / ldc);
      w_o[j] = to_half_bits(c < C ? ld_param<DT>(wo, (long long)co * C + c) : 0.f);
      if (c == 0) b_o[co] = bo ? ld_param<DT>(bo, co) : 0.f;
    }
  }
}

__global__ void pad_x_kernel(const char *x, int rows, int n_bytes, int ld_bytes, char *dst) {
  pdl_trigger();
  pdl_wait();
  const long long total = (long long)rows * ld_bytes;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / ld_bytes;
    const int c = (int)(i % ld_bytes);
    dst[i] = c < n_bytes ? x[r * n_bytes + c] : 0;
  }
}

}  // namespace

cudaError_t launch_pack_weights(const Dims &dm, int dtype, const void *wq, const void *bq, const void *wk,
                                const void *bk, const void *wv, const void *bv, const void *wo,
                                const void *bo, uint16_t *w_qkv, float *b_qkv, uint16_t *w_o, float *b_o,
                                cudaStream_t st) {
  const long long total = 3LL * dm.h * dm.dp * dm.ldc + (long long)dm.C * dm.ldc;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  const int grid = (int)(blocks < 4096 ? blocks : 4096);
  const int inter = qk_pair_interleaved(dm) ? 1 : 0;
  if (dtype == 0)
    (void)launch_k(pack_kernel<0>, dim3(grid), dim3(threads), 0, st, dm.C, dm.h, dm.d, dm.dp, dm.ldc, inter, wq, bq,
                   wk, bk, wv, bv, wo, bo, w_qkv, b_qkv, w_o, b_o);
  else
    (void)launch_k(pack_kernel<1>, dim3(grid), dim3(threads), 0, st, dm.C, dm.h, dm.d, dm.dp, dm.ldc, inter, wq, bq,
                   wk, bk, wv, bv, wo, bo, w_qkv, b_qkv, w_o, b_o);
  return cudaGetLastError();
}

cudaError_t launch_pad_x(const void *x, int B, int C, int N, int ldx, int esize, void *dst, cudaStream_t st) {
  const long long total = (long long)B * C * ldx * esize;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  const int grid = (int)(blocks < 4096 ? blocks : 4096);
  (void)launch_k(pad_x_kernel, dim3(grid), dim3(threads), 0, st, reinterpret_cast<const char *>(x), B * C, N * esize, ldx * esize,
                                         reinterpret_cast<char *>(dst));
  return cudaGetLastError();
}

}  // namespace ssa
