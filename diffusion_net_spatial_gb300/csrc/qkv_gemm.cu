// qkv_gemm.cu -- Q, K, V = tokens(GN(x)) [Wq; Wk; Wv]^T + [bq; bk; bv]
// (tensortonic "diffusion-l03-spatial-self-attention", block equation:
// Z = tokens(GN(x)), Q = Z Wq^T + bq, K = Z Wk^T + bk, V = Z Wv^T + bv; the
// tokens step puts pixel (i, j) at row i*W + j).
//
// One CTA computes a 128-pixel x BN-feature tile of the stacked projection
// (M = pixels of one sample, N = 3*h*dp packed features, K = C channels):
//   warp 0      TMA producer: the raw x tile [64 channels][128 pixels] (NCHW,
//               fp32 or bf16, no swizzle) and the packed-weight tile
//               [BN][64] (fp16, 128-byte swizzle)
//   warp 1      tcgen05 MMA issuer (fp16 x fp16 -> fp32 in tensor memory);
//               owns the tensor-memory allocation
//   warps 2..9  converters: z = gn_scale * x + gn_shift, rounded to fp16 and
//               written transposed (pixel rows, channel columns) into the
//               K-major 128B-swizzled A tile -- the GN affine and the
//               NCHW -> token transpose happen here, in shared memory; after
//               the K loop the same warps run the epilogue (bias add, fp16
//               round, scatter into Q/K [b][head][pixel][ldq] and
//               V^T [b][head][e][ldn]).
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int XST = 2;      // x staging stages
constexpr int ST = 3;       // A/B operand stages
constexpr int NCONV = 8;    // converter / epilogue warps
constexpr int THREADS = (2 + NCONV) * 32;

struct QkvArgs {
  int C, N, h, dp, ldq, ldn, BN, nk, tmem_cols, xbytes;
  const float *ga;
  const float *gs;
  const float *bias;
  uint16_t *q;
  uint16_t *k;
  uint16_t *vt;
  uint32_t *err;
  uint64_t timeout_ns;
};

struct Smem {
  // offsets from the 1024-aligned base
  uint32_t xs, as, bs, slot, bars;
};

__host__ __device__ inline Smem smem_layout(int xbytes, int BN) {
  Smem s;
  s.xs = 0;
  s.as = s.xs + XST * xbytes;
  s.bs = s.as + ST * (BM * BK * 2);
  s.slot = s.bs + ST * (BN * BK * 2);
  s.bars = s.slot + NCONV * 256;
  return s;
}
// barriers: x_full[XST], x_empty[XST], b_full[ST], a_full[ST], ab_empty[ST], acc_full, drain, epi_done
constexpr int NBARS = 2 * XST + 3 * ST + 3;
__host__ __device__ inline uint32_t smem_total(int xbytes, int BN) {
  return smem_layout(xbytes, BN).bars + NBARS * 8 + 16 + 1024;  // + tmem slot, abort flag, alignment slack
}

template <int DT>
__global__ void __launch_bounds__(THREADS, 1)
    qkv_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const QkvArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Smem L = smem_layout(args.xbytes, args.BN);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bars);
  uint64_t *x_full = bars;
  uint64_t *x_empty = bars + XST;
  uint64_t *b_full = bars + 2 * XST;
  uint64_t *a_full = b_full + ST;
  uint64_t *ab_empty = a_full + ST;
  uint64_t *acc_full = ab_empty + ST;
  uint64_t *drain = acc_full + 1;
  uint64_t *epi_done = drain + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);
  volatile uint32_t *abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * args.BN;
  const int p0 = blockIdx.y * BM;
  const int b = blockIdx.z;
  const int nk = args.nk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < XST; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], NCONV);
    }
    for (int i = 0; i < ST; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&a_full[i], NCONV);
      mbar_init(&ab_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    mbar_init(epi_done, NCONV);
    *abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
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
    // ------------------------------------------------------------ producer
    int nx = 0, nb = 0;
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int sx = kb % XST, s = kb % ST;
        if (kb >= XST && !mbar_wait(&x_empty[sx], ((kb / XST) - 1) & 1, ab)) break;
        mbar_arrive_expect_tx(&x_full[sx], (uint32_t)args.xbytes);
        tma_load_3d(sm + L.xs + sx * args.xbytes, &xmap, &x_full[sx], p0, kb * BK, b);
        ++nx;
        if (kb >= ST && !mbar_wait(&ab_empty[s], ((kb / ST) - 1) & 1, ab)) break;
        mbar_arrive_expect_tx(&b_full[s], (uint32_t)(args.BN * BK * 2));
        tma_load_2d(sm + L.bs + s * (args.BN * BK * 2), &wmap, &b_full[s], kb * BK, n0);
        ++nb;
      }
      // Never leave with a copy in flight.
      for (int kb = (nx > XST ? nx - XST : 0); kb < nx; ++kb)
        mbar_wait_drain(&x_full[kb % XST], (kb / XST) & 1, ab.limit_ns);
      for (int kb = (nb > ST ? nb - ST : 0); kb < nb; ++kb)
        mbar_wait_drain(&b_full[kb % ST], (kb / ST) & 1, ab.limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and the elected lane 0 issues.
    {
      const uint32_t idesc = idesc_f16(BM, (uint32_t)args.BN);
      bool issued = false, ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % ST;
        if (!mbar_wait_warp(&b_full[s], (kb / ST) & 1, ab) || !mbar_wait_warp(&a_full[s], (kb / ST) & 1, ab)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(sm + L.as + s * (BM * BK * 2));
        const uint32_t b_addr = smem_u32(sm + L.bs + s * (args.BN * BK * 2));
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_f16_ss(tmem, sdesc_k128(a_addr + kk * 32), sdesc_k128(b_addr + kk * 32), idesc,
                       (kb | kk) != 0 ? 1u : 0u);
          mma_commit(&ab_empty[s]);
        }
        __syncwarp();
        issued = true;
      }
      if (ok) {
        if (elect_one()) mma_commit(acc_full);
        __syncwarp();
      }
      if (!ok && issued) {
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait_drain(drain, 0, ab.limit_ns);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ converters
    const int cw = warp - 2;                 // 0..7
    const int px = (cw & 3) * 32 + lane;     // pixel row of the A tile
    const int hc = cw >> 2;                  // channel half of the k-block
    float *slot = reinterpret_cast<float *>(sm + L.slot + cw * 256);
    const float *ga = args.ga + (long long)b * args.C;
    const float *gs = args.gs + (long long)b * args.C;
    bool ok = true;
    // The GN scale/shift of the next k-block are fetched one iteration ahead,
    // so their global-memory latency overlaps the current block.
    int c = hc * 32 + lane;
    float a_cur = c < args.C ? __ldg(ga + c) : 0.f;
    float s_cur = c < args.C ? __ldg(gs + c) : 0.f;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int sx = kb % XST, s = kb % ST;
      c = (kb + 1) * BK + hc * 32 + lane;
      const float a_nxt = (kb + 1 < nk && c < args.C) ? __ldg(ga + c) : 0.f;
      const float s_nxt = (kb + 1 < nk && c < args.C) ? __ldg(gs + c) : 0.f;
      if (!mbar_wait_warp(&x_full[sx], (kb / XST) & 1, ab)) { ok = false; break; }
      if (kb >= ST && !mbar_wait_warp(&ab_empty[s], ((kb / ST) - 1) & 1, ab)) { ok = false; break; }
      __syncwarp();
      slot[lane] = a_cur;
      slot[32 + lane] = s_cur;
      a_cur = a_nxt;
      s_cur = s_nxt;
      __syncwarp();
      const uint8_t *xs = sm + L.xs + sx * args.xbytes;
      const uint32_t a_tile = smem_u32(sm + L.as + s * (BM * BK * 2));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ch0 = hc * 32 + j * 8;     // channel within the k-block
        float z[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float xv;
          if (DT == 0) {
            xv = reinterpret_cast<const float *>(xs)[(ch0 + i) * BM + px];
          } else {
            const unsigned short u = reinterpret_cast<const unsigned short *>(xs)[(ch0 + i) * BM + px];
            xv = __uint_as_float(((uint32_t)u) << 16);
          }
          z[i] = fmaf(slot[j * 8 + i], xv, slot[32 + j * 8 + i]);
        }
        st_shared_v4(a_tile + sw128_offset((uint32_t)px, (uint32_t)(ch0 >> 3)), pack_half2(z[0], z[1]),
                     pack_half2(z[2], z[3]), pack_half2(z[4], z[5]), pack_half2(z[6], z[7]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&x_empty[sx]);
        mbar_arrive(&a_full[s]);
      }
    }
    // ------------------------------------------------------------ epilogue
    // The output tile is staged in the (now idle) operand ring in global
    // order, one 4 KB chunk per 16 features: Q/K chunks as [128 pixels][16]
    // (rows of the q/k layout), V chunks as [16][128 pixels] (rows of the
    // transposed v layout).  One thread then stores each chunk with TMA,
    // which clips pixels past N.
    if (ok && mbar_wait_warp(acc_full, 0, ab)) {
      __syncwarp();
      tc_fence_after();
      const int q4 = warp & 3;                // lane quarter this warp may read
      const int half = cw >> 2;
      const int row = q4 * 32 + lane;
      const int hdp = args.h * args.dp;
      uint8_t *stage = sm + L.as;
      for (int c16 = half; c16 < args.BN / 16; c16 += 2) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(c16 * 16), r);
        tmem_wait_ld();
        const int f0 = n0 + c16 * 16;
        const int sec = f0 / hdp;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]) + __ldg(args.bias + f0 + i);
        uint8_t *chunk = stage + c16 * 4096;
        if (sec < 2) {
          uint4 w0, w1;
          w0.x = pack_half2(v[0], v[1]); w0.y = pack_half2(v[2], v[3]);
          w0.z = pack_half2(v[4], v[5]); w0.w = pack_half2(v[6], v[7]);
          w1.x = pack_half2(v[8], v[9]); w1.y = pack_half2(v[10], v[11]);
          w1.z = pack_half2(v[12], v[13]); w1.w = pack_half2(v[14], v[15]);
          reinterpret_cast<uint4 *>(chunk + row * 32)[0] = w0;
          reinterpret_cast<uint4 *>(chunk + row * 32)[1] = w1;
        } else {
          __half *vt_rows = reinterpret_cast<__half *>(chunk);
#pragma unroll
          for (int i = 0; i < 16; ++i) vt_rows[i * BM + row] = __float2half_rn(v[i]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(epi_done);
      if (cw == 0 && lane == 0 && mbar_wait(epi_done, 0, ab)) {
        for (int c16 = 0; c16 < args.BN / 16; ++c16) {
          const int f0 = n0 + c16 * 16;
          const int sec = f0 / hdp;
          const int hd = (f0 / args.dp) % args.h;
          const int e0 = f0 % args.dp;
          const int bh = b * args.h + hd;
          const uint8_t *chunk = stage + c16 * 4096;
          if (sec == 0) tma_store_3d(&qmap, chunk, e0, p0, bh);
          else if (sec == 1) tma_store_3d(&kmap, chunk, e0, p0, bh);
          else tma_store_3d(&vmap, chunk, p0, e0, bh);
        }
        tma_store_commit();
        tma_store_wait_all();
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)args.tmem_cols);
  }
}

int pick_bn(int ntot) {
  for (int bn = 256; bn >= 16; bn -= 16)
    if (ntot % bn == 0) return bn;
  return 16;
}

}  // namespace

int launch_qkv_gemm(const Dims &dm, int dtype, const void *x, int ldx, const float *ga, const float *gs,
                    const uint16_t *w_qkv, const float *b_qkv, uint16_t *q, uint16_t *k, uint16_t *vt,
                    const KParams &kp, cudaStream_t st) {
  const int es = dtype == 0 ? 4 : 2;
  CUtensorMap xmap, wmap;
  {
    const uint64_t dims[3] = {(uint64_t)dm.N, (uint64_t)dm.C, (uint64_t)dm.B};
    const uint64_t strides[2] = {(uint64_t)ldx * es, (uint64_t)dm.C * ldx * es};
    const uint32_t box[3] = {BM, BK, 1};
    if (encode_tiled(&xmap, dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return 1;
  }
  const int BN = pick_bn(dm.ntot);
  {
    const uint64_t dims[2] = {(uint64_t)dm.C, (uint64_t)dm.ntot};
    const uint64_t strides[1] = {(uint64_t)dm.ldc * 2};
    const uint32_t box[2] = {BK, (uint32_t)BN};
    if (encode_tiled(&wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w_qkv, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
  }
  CUtensorMap qmap, kmap, vmap;
  {
    const uint64_t BH = (uint64_t)dm.B * dm.h;
    const uint64_t dims[3] = {(uint64_t)dm.ldq, (uint64_t)dm.N, BH};
    const uint64_t strides[2] = {(uint64_t)dm.ldq * 2, (uint64_t)dm.N * dm.ldq * 2};
    const uint32_t box[3] = {16, BM, 1};
    if (encode_tiled(&qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, q, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return 1;
    if (encode_tiled(&kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, k, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return 1;
    const uint64_t vdims[3] = {(uint64_t)dm.N, (uint64_t)dm.dp, BH};
    const uint64_t vstrides[2] = {(uint64_t)dm.ldn * 2, (uint64_t)dm.dp * dm.ldn * 2};
    const uint32_t vbox[3] = {BM, 16, 1};
    if (encode_tiled(&vmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, vt, vdims, vstrides, vbox,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return 1;
  }
  QkvArgs a{};
  a.C = dm.C; a.N = dm.N; a.h = dm.h; a.dp = dm.dp; a.ldq = dm.ldq; a.ldn = dm.ldn; a.BN = BN;
  a.nk = (dm.C + BK - 1) / BK;
  a.tmem_cols = BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
  a.xbytes = BM * BK * es;
  a.ga = ga; a.gs = gs; a.bias = b_qkv; a.q = q; a.k = k; a.vt = vt;
  a.err = kp.err; a.timeout_ns = kp.timeout_ns;
  const uint32_t smem = smem_total(a.xbytes, BN);
  const dim3 grid(dm.ntot / BN, (dm.N + BM - 1) / BM, dm.B);
  if (dtype == 0) {
    cudaFuncSetAttribute(qkv_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    qkv_gemm_kernel<0><<<grid, THREADS, smem, st>>>(xmap, wmap, qmap, kmap, vmap, a);
  } else {
    cudaFuncSetAttribute(qkv_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    qkv_gemm_kernel<1><<<grid, THREADS, smem, st>>>(xmap, wmap, qmap, kmap, vmap, a);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace ssa
