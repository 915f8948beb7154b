// out_proj.cu -- out = x + image([O_1..O_n] Wo^T + bo), in x's dtype
// (tensortonic "diffusion-l03-spatial-self-attention", block equation and the
// return rule; the image step undoes the tokens step, row i*W + j -> (i, j)).
//
// One CTA computes a 128-pixel x BN-channel tile (M = pixels of one sample,
// N = output channels, K = C):
//   warp 0      TMA producer: O tile [128 pixels][64 channels] and Wo tile
//               [BN][64] (fp16, 128-byte swizzle, K-major)
//   warp 1      tcgen05 MMA issuer, fp32 accumulator in tensor memory
//   warps 2..9  epilogue: tensor-memory lane = pixel, column = channel, so for
//               each channel a warp reads 32 consecutive pixels of x and
//               writes 32 consecutive pixels of out -- the residual read, the
//               bias add, the single rounding to x's dtype and the transposed
//               NCHW store are one coalesced pass.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int ST = 4;
constexpr int NEPI = 8;
constexpr int THREADS = (2 + NEPI) * 32;

struct OutArgs {
  int C, N, BN, nk, tmem_cols;
  const float *bias;
  const void *x;
  void *out;
  uint32_t *err;
  uint64_t timeout_ns;
};

__host__ __device__ inline uint32_t bars_off(int BN) { return ST * (BM * BK * 2 + BN * BK * 2); }
constexpr int NBARS = 2 * ST + 2;
__host__ __device__ inline uint32_t smem_total(int BN) { return bars_off(BN) + NBARS * 8 + 16 + 1024; }

template <int DT>
__global__ void __launch_bounds__(THREADS, 1)
    out_proj_kernel(const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap wmap,
                    const OutArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = args.BN;
  const uint32_t a_off = 0, b_off = ST * (BM * BK * 2);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + bars_off(BN));
  uint64_t *full = bars;
  uint64_t *empty = bars + ST;
  uint64_t *acc_full = bars + 2 * ST;
  uint64_t *drain = acc_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);
  volatile uint32_t *abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int p0 = blockIdx.y * BM;
  const int b = blockIdx.z;
  const int nk = args.nk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&omap);
    tma_prefetch_desc(&wmap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, (uint32_t)args.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, args.err, args.timeout_ns};

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      const uint32_t bytes = (uint32_t)(BM * BK * 2 + BN * BK * 2);
      for (; it < nk; ++it) {
        const int s = it % ST;
        if (it >= ST && !mbar_wait(&empty[s], ((it / ST) - 1) & 1, ab)) break;
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_3d(sm + a_off + s * (BM * BK * 2), &omap, &full[s], it * BK, p0, b);
        tma_load_2d(sm + b_off + s * (BN * BK * 2), &wmap, &full[s], it * BK, n0);
      }
      for (int i = (it > ST ? it - ST : 0); i < it; ++i) mbar_wait_drain(&full[i % ST], (i / ST) & 1, ab.limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(BM, (uint32_t)BN);
      bool ok = true, issued = false;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % ST;
        if (!mbar_wait(&full[s], (kb / ST) & 1, ab)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(sm + a_off + s * (BM * BK * 2));
        const uint32_t b_addr = smem_u32(sm + b_off + s * (BN * BK * 2));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_f16_ss(tmem, sdesc_k128(a_addr + kk * 32), sdesc_k128(b_addr + kk * 32), idesc,
                     (kb | kk) != 0 ? 1u : 0u);
        mma_commit(&empty[s]);
        issued = true;
      }
      if (ok) mma_commit(acc_full);
      if (!ok && issued) {
        mma_commit(drain);
        mbar_wait_drain(drain, 0, ab.limit_ns);
      }
    }
    __syncwarp();
  } else {
    if (mbar_wait_warp(acc_full, 0, ab)) {
      __syncwarp();
      tc_fence_after();
      const int ew = warp - 2;
      const int q4 = warp & 3;
      const int half = ew >> 2;
      const int row = q4 * 32 + lane;
      const int p = p0 + row;
      const bool valid = p < args.N;
      const long long plane = (long long)args.N;
      for (int c16 = half; c16 < BN / 16; c16 += 2) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(c16 * 16), r);
        tmem_wait_ld();
        if (!valid) continue;
        // All residual reads of the chunk are issued before any store: out
        // may alias x, so interleaving them would serialise every load
        // behind the previous store.
        const int cbase = n0 + c16 * 16;
        const int nc = min(16, args.C - cbase);
        const long long idx0 = ((long long)b * args.C + cbase) * plane + p;
        float xv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i < nc) {
            if (DT == 0) {
              xv[i] = reinterpret_cast<const float *>(args.x)[idx0 + i * plane];
            } else {
              const unsigned short xb = reinterpret_cast<const unsigned short *>(args.x)[idx0 + i * plane];
              xv[i] = __uint_as_float(((uint32_t)xb) << 16);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i < nc) {
            const float v = xv[i] + (__uint_as_float(r[i]) + __ldg(args.bias + cbase + i));
            if (DT == 0) {
              reinterpret_cast<float *>(args.out)[idx0 + i * plane] = v;
            } else {
              reinterpret_cast<__nv_bfloat16 *>(args.out)[idx0 + i * plane] = __float2bfloat16_rn(v);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)args.tmem_cols);
  }
}

int pick_bn(int C) {
  const int c16 = (C + 15) / 16 * 16;
  for (int bn = 256; bn >= 16; bn -= 16)
    if (c16 % bn == 0) return bn;
  return 16;
}

}  // namespace

int launch_out_proj(const Dims &dm, int dtype, const uint16_t *o, const uint16_t *w_o, const float *b_o,
                    const void *x, void *out, const KParams &kp, cudaStream_t st) {
  CUtensorMap omap, wmap;
  const int BN = pick_bn(dm.C);
  {
    const uint64_t dims[3] = {(uint64_t)dm.C, (uint64_t)dm.N, (uint64_t)dm.B};
    const uint64_t strides[2] = {(uint64_t)dm.ldc * 2, (uint64_t)dm.N * dm.ldc * 2};
    const uint32_t box[3] = {BK, BM, 1};
    if (encode_tiled(&omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, o, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
  }
  {
    const uint64_t dims[2] = {(uint64_t)dm.C, (uint64_t)dm.C};
    const uint64_t strides[1] = {(uint64_t)dm.ldc * 2};
    const uint32_t box[2] = {BK, (uint32_t)BN};
    if (encode_tiled(&wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w_o, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
  }
  OutArgs a{};
  a.C = dm.C; a.N = dm.N; a.BN = BN; a.nk = (dm.C + BK - 1) / BK;
  a.tmem_cols = BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
  a.bias = b_o; a.x = x; a.out = out; a.err = kp.err; a.timeout_ns = kp.timeout_ns;
  const uint32_t smem = smem_total(BN);
  const dim3 grid((dm.C + BN - 1) / BN, (dm.N + BM - 1) / BM, dm.B);
  if (dtype == 0) {
    cudaFuncSetAttribute(out_proj_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    out_proj_kernel<0><<<grid, THREADS, smem, st>>>(omap, wmap, a);
  } else {
    cudaFuncSetAttribute(out_proj_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    out_proj_kernel<1><<<grid, THREADS, smem, st>>>(omap, wmap, a);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace ssa
