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

// Rotary embedding of one pair (HNDL "attention" operator page, Rotary
// embeddings paragraph: rotate-half, base 10000): feature i (x) and feature
// i + d/2 (y) of the token at position t turn by angle = t * theta_i,
// theta_i = 10000^(-2i/d).  theta_i comes as two fp32 parts (hi + lo, formed
// in fp64); the product t * hi is carried with its exact rounding residual,
// the angle is reduced to [-pi, pi] by Cody and Waite's two-constant scheme
// (2 pi = 6.28125 + a small remainder, so k * 6.28125 is exact for the
// |k| < 2^12 of t < 2^16), and __sincosf, accurate on that interval, gives
// cos and sin.  The rotation acts on the fp32 accumulator values (bias added)
// before their single rounding to fp16.
constexpr float kTwoPiA = 6.28125f;
constexpr float kTwoPiB = 1.9353071795864769e-3f;  // 2 pi - 6.28125
constexpr float kInvTwoPi = 0.15915494309189535f;

__device__ __forceinline__ void rope_pair(float &x, float &y, float t, float2 th) {
  const float a_hi = t * th.x;
  const float a_lo = fmaf(t, th.y, fmaf(t, th.x, -a_hi));
  const float k = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiA, a_hi);
  r = fmaf(-k, kTwoPiB, r) + a_lo;
  float sn, c;
  __sincosf(r, &sn, &c);
  const float x2 = fmaf(x, c, -y * sn);
  y = fmaf(y, c, x * sn);
  x = x2;
}

// theta_i = 10000^(-2i/d) for i < d/2, split into fp32 hi + lo, into the
// shared-memory table th[] (one entry per thread of the caller's range).
__device__ __forceinline__ void rope_thetas(float2 *th, int d, int tid, int nthreads) {
  for (int i = tid; i < d / 2; i += nthreads) {
    const double v = exp(-2.0 * (double)i / (double)d * 9.2103403719761827361);  // ln(10000)
    const float hi = (float)v;
    th[i] = make_float2(hi, (float)(v - (double)hi));
  }
}

// Writes the first n (0..M) of M fp16 values, packed two per word in w, to
// dst: 16-byte stores for a whole aligned run, else 4-byte stores where dst is
// 4-byte aligned, else 2-byte stores.
template <int M>
__device__ __forceinline__ void store_run(uint16_t *dst, const uint32_t (&w)[M / 2], int n) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
  if (n == M && (a & 15u) == 0) {
#pragma unroll
    for (int k = 0; k < M / 8; ++k)
      reinterpret_cast<uint4 *>(dst)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
  } else if ((a & 3u) == 0) {
#pragma unroll
    for (int m = 0; m < M / 2; ++m) {
      if (2 * m + 2 <= n) reinterpret_cast<uint32_t *>(dst)[m] = w[m];
      else if (2 * m < n) dst[2 * m] = (uint16_t)(w[m] & 0xFFFFu);
    }
  } else {
#pragma unroll
    for (int m = 0; m < M / 2; ++m) {
      if (2 * m < n) dst[2 * m] = (uint16_t)(w[m] & 0xFFFFu);
      if (2 * m + 1 < n) dst[2 * m + 1] = (uint16_t)(w[m] >> 16);
    }
  }
}

constexpr int XST = 4;      // x staging stages at most (args.xst: as many as shared memory allows, >= 2)
constexpr int ST = 3;       // A/B operand stages
constexpr int NCONV = 8;    // converter / epilogue warps
constexpr int THREADS = (2 + NCONV) * 32;

struct QkvArgs {
  int C, N, h, dp, ldq, ldn, BN, nk, tmem_cols, xbytes, xst;
  int d, inter;              // head dim; Q/K rows pair-interleaved (then d == dp, d % 16 == 0)
  int rope;                  // rotate Q and K in the epilogue (needs inter)
  uint32_t stall;            // test hook: the producer stops after this many loads (0: never)
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

__host__ __device__ inline Smem smem_layout(int xbytes, int BN, int xst) {
  Smem s;
  s.xs = 0;
  s.as = s.xs + xst * xbytes;
  s.bs = s.as + ST * (BM * BK * 2);
  s.slot = s.bs + ST * (BN * BK * 2);
  s.bars = s.slot + NCONV * 256;
  return s;
}
// barriers: x_full[XST], x_empty[XST], b_full[ST], a_full[ST], ab_empty[ST], acc_full, drain, epi_done
constexpr int NBARS = 2 * XST + 3 * ST + 3;
__host__ __device__ inline uint32_t smem_total(int xbytes, int BN, int xst) {
  return smem_layout(xbytes, BN, xst).bars + NBARS * 8 + 16 + 1024;  // + tmem slot, abort flag, alignment slack
}

template <int DT>
__global__ void __launch_bounds__(THREADS, 1)
    qkv_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const QkvArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Smem L = smem_layout(args.xbytes, args.BN, args.xst);
  const int xst = args.xst;
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
    for (int i = 0; i < xst; ++i) {
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
  pdl_trigger();
  pdl_wait();  // inputs of the previous kernel visible from here on
  const Abort ab{abort_flag, args.err, args.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int nx = 0, nb = 0;
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int sx = kb % xst, s = kb % ST;
        if (args.stall && (uint32_t)(nx + nb) >= args.stall) break;  // test hook: consumers' waits expire
        if (kb >= xst && !mbar_wait(&x_empty[sx], ((kb / xst) - 1) & 1, ab)) break;
        mbar_arrive_expect_tx(&x_full[sx], (uint32_t)args.xbytes);
        // [64 channels][128 pixels] as 128-byte-wide swizzled boxes of
        // 128 / sizeof(x) pixels (8 KB each)
        for (int u = 0; u < (DT == 0 ? 4 : 2); ++u)
          tma_load_3d(sm + L.xs + sx * args.xbytes + u * 8192, &xmap, &x_full[sx], p0 + u * (DT == 0 ? 32 : 64),
                      kb * BK, b);
        ++nx;
        if (kb >= ST && !mbar_wait(&ab_empty[s], ((kb / ST) - 1) & 1, ab)) break;
        mbar_arrive_expect_tx(&b_full[s], (uint32_t)(args.BN * BK * 2));
        tma_load_2d(sm + L.bs + s * (args.BN * BK * 2), &wmap, &b_full[s], kb * BK, n0);
        ++nb;
      }
      // Never leave with a copy in flight.
      for (int kb = (nx > xst ? nx - xst : 0); kb < nx; ++kb)
        mbar_wait_drain(&x_full[kb % xst], (kb / xst) & 1, drain_limit(ab));
      for (int kb = (nb > ST ? nb - ST : 0); kb < nb; ++kb)
        mbar_wait_drain(&b_full[kb % ST], (kb / ST) & 1, drain_limit(ab));
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
      if (issued) {  // every issued MMA completes before tensor memory is freed
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait_drain(drain, 0, drain_limit(ab));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ converters
    // Warp cw converts the k-block's channels 8 cw .. 8 cw + 7 for all 128
    // pixels; thread t owns channel 8 cw + t / 4 and, in each 8-pixel group,
    // the pixel pair 2 (t % 4), +1: it reads the pair with one load from the
    // swizzled x stage (the 8 channels of a load sit in 8 different 16-byte
    // bank groups) and writes the transposed A tile with stmatrix.trans, four
    // 8 x 8 pixel-by-channel blocks per instruction.
    const int cw = warp - 2;                 // 0..7
    const int cl = cw * 8 + (lane >> 2);     // this thread's channel within the k-block
    const float *ga = args.ga + (long long)b * args.C;
    const float *gs = args.gs + (long long)b * args.C;
    bool ok = true;
    // x stage offset of this thread's pixel pair in 8-pixel group T: box
    // T / (boxes of 128 bytes), 16-byte chunk XOR the channel's row phase.
    constexpr int ES = DT == 0 ? 4 : 2;
    constexpr int PPB = 128 / ES;            // pixels per 128-byte box row
    auto x_off = [&](int T) -> uint32_t {
      const int px0 = 8 * T + 2 * (lane & 3);
      const int bx = px0 / PPB, pb = (px0 % PPB) * ES;
      return (uint32_t)(bx * 8192 + cl * 128 + ((((pb >> 4) ^ (cl & 7)) << 4) | (pb & 15)));
    };
    // stmatrix row addresses: matrix i = lane / 8 (pixel group 4 g + i), row
    // lane % 8 (its pixel), chunk cw (this warp's 8 channels).
    const int prow = 8 * (lane >> 3) + (lane & 7);  // + 32 g
    // The GN scale/shift of the next k-block are fetched one iteration ahead,
    // so their global-memory latency overlaps the current block.
    int c = cl;
    float a_cur = c < args.C ? __ldg(ga + c) : 0.f;
    float s_cur = c < args.C ? __ldg(gs + c) : 0.f;
    for (int kb = 0; kb < nk && ok; ++kb) {
      const int sx = kb % xst, s = kb % ST;
      c = (kb + 1) * BK + cl;
      const float a_nxt = (kb + 1 < nk && c < args.C) ? __ldg(ga + c) : 0.f;
      const float s_nxt = (kb + 1 < nk && c < args.C) ? __ldg(gs + c) : 0.f;
      if (!mbar_wait_warp(&x_full[sx], (kb / xst) & 1, ab)) { ok = false; break; }
      if (kb >= ST && !mbar_wait_warp(&ab_empty[s], ((kb / ST) - 1) & 1, ab)) { ok = false; break; }
      const uint32_t xs = smem_u32(sm + L.xs + sx * args.xbytes);
      const uint32_t a_tile = smem_u32(sm + L.as + s * (BM * BK * 2));
      // channels past C are zero (their scale and shift are zero)
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t off = x_off(4 * g + i);
          float x0, x1;
          if (DT == 0) {
            float2 v;
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(xs + off));
            x0 = v.x;
            x1 = v.y;
          } else {
            uint32_t v;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(xs + off));
            x0 = __uint_as_float(v << 16);
            x1 = __uint_as_float(v & 0xFFFF0000u);
          }
          w[i] = pack_op2(fmaf(a_cur, x0, s_cur), fmaf(a_cur, x1, s_cur));
        }
        stmatrix_x4_trans(a_tile + sw128_offset((uint32_t)(32 * g + prow), (uint32_t)cw), w[0], w[1], w[2], w[3]);
      }
      a_cur = a_nxt;
      s_cur = s_nxt;
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
    // which clips pixels past N.  With pair-interleaved Q/K rows a chunk holds
    // 8 pairs (features i0..i0+7 and d/2+i0..d/2+i0+7): it is staged as two
    // [128 pixels][8] halves, rotated first when the rotary embedding is on.
    float2 *th = reinterpret_cast<float2 *>(sm + L.slot);  // rotation thetas (in the otherwise unused slot area)
    if (args.rope) {
      named_bar_sync(1, NCONV * 32);  // every converter has left its k-block loop
      rope_thetas(th, args.d, threadIdx.x - 64, NCONV * 32);
      named_bar_sync(1, NCONV * 32);
    }
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
        if (sec < 2 && args.inter) {
          if (args.rope) {
            const int i0 = (f0 % args.dp) >> 1;
            const float t = (float)(p0 + row);
#pragma unroll
            for (int j = 0; j < 8; ++j) rope_pair(v[2 * j], v[2 * j + 1], t, th[i0 + j]);
          }
          uint4 wx, wy;
          wx.x = pack_op2(v[0], v[2]); wx.y = pack_op2(v[4], v[6]);
          wx.z = pack_op2(v[8], v[10]); wx.w = pack_op2(v[12], v[14]);
          wy.x = pack_op2(v[1], v[3]); wy.y = pack_op2(v[5], v[7]);
          wy.z = pack_op2(v[9], v[11]); wy.w = pack_op2(v[13], v[15]);
          reinterpret_cast<uint4 *>(chunk)[row] = wx;
          reinterpret_cast<uint4 *>(chunk + 2048)[row] = wy;
        } else if (sec < 2) {
          uint4 w0, w1;
          w0.x = pack_op2(v[0], v[1]); w0.y = pack_op2(v[2], v[3]);
          w0.z = pack_op2(v[4], v[5]); w0.w = pack_op2(v[6], v[7]);
          w1.x = pack_op2(v[8], v[9]); w1.y = pack_op2(v[10], v[11]);
          w1.z = pack_op2(v[12], v[13]); w1.w = pack_op2(v[14], v[15]);
          reinterpret_cast<uint4 *>(chunk + row * 32)[0] = w0;
          reinterpret_cast<uint4 *>(chunk + row * 32)[1] = w1;
        } else {
          uint16_t *vt_rows = reinterpret_cast<uint16_t *>(chunk);
#pragma unroll
          for (int i = 0; i < 16; ++i) vt_rows[i * BM + row] = op_bits(v[i]);
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
          if (sec < 2 && args.inter) {
            // two 8-feature halves: features i0.. and d/2 + i0..
            const CUtensorMap *m = sec == 0 ? &qmap : &kmap;
            tma_store_3d(m, chunk, e0 >> 1, p0, bh);
            tma_store_3d(m, chunk + 2048, args.d / 2 + (e0 >> 1), p0, bh);
          } else if (sec == 0) tma_store_3d(&qmap, chunk, e0, p0, bh);
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


// ---------------------------------------------------------------------------
// Resident-tile variant (C <= 512): one CTA owns a 128-pixel tile and a group
// of BN-feature slices (BN <= 128).  The tile's GN-applied, transposed fp16 A
// operand (128 pixels x C) is built once into tensor-memory columns
// 256..511 and stays there while the CTA sweeps its slices (A from tensor
// memory, N = BN MMAs into two alternating 128-column accumulators), so x is
// read and converted once per tile, slice i's epilogue overlaps slice i+1's
// MMAs, and all of shared memory is a deep ring for the weight stream (every
// CTA reads all 3C x C weights; a 3-slot ring behind a shared-memory A tile
// fed them at ~40 GB/s per SM).
//   warps 0, 10  TMA producers on alternate ring loads: first the tile's x
//                blocks [64 channels][128 pixels], then the weights, two
//                [BN][64] k-blocks per 32 KB slot
//   warp 1       MMA warp (warp-uniform loop, elected lane issues)
//   warps 2..9   converters (x block -> A columns in tensor memory), then
//                epilogues (bias, the optional rotary embedding, fp16; Q/K
//                rows and V^T rows stored directly)
constexpr int RNST = 5;                  // ring slots of 32 KB (6 or 7 measured no faster: shared memory past the 164 KB carveout costs L1)
constexpr int RSLOT = 32768;
constexpr int RTHREADS = 352;
constexpr uint32_t RA_COL = 256;         // A operand: tensor-memory columns 256 .. 256 + C/2

struct ResArgs {
  int C, N, h, dp, ldq, ldn, BN, nkb, nslices, spg, xbytes;
  int w3d;  // weights as one 3-D box of two 64-channel chunks per slot (C % 64 == 0), else two 2-D boxes
  int cw;   // epilogue chunk: 32 columns (dp % 32 == 0 and BN % 64 == 0) or 16
  int d, inter;        // head dim; Q/K rows pair-interleaved (qk_pair_interleaved)
  int rope;            // rotate Q and K in the epilogue (needs inter)
  uint32_t stall;      // test hook: each producer stops at this load index (0: never)
  const float *ga;
  const float *gs;
  const float *bias;
  uint16_t *q;
  uint16_t *k;
  uint16_t *vt;
  uint32_t *err;
  uint64_t timeout_ns;
};
// barriers: full[RNST], empty[RNST], xfree[RNST], a_ready, acc_full[2], acc_empty[2], drain
constexpr int RNBARS = 3 * RNST + 6;
constexpr uint32_t RES_SLOT_OFF = RNST * RSLOT;              // converters' GN scale/shift staging
constexpr uint32_t RES_BARS_OFF = RES_SLOT_OFF + NCONV * 256;
constexpr uint32_t RES_SMEM = RES_BARS_OFF + RNBARS * 8 + 16;

// One chunk of CW accumulator columns of a slice, for the lanes' 32 pixels:
// bias, then by section
//   Q/K, pair-interleaved: pairs (x = feature i, y = feature i + d/2),
//        rotated when the table is given, written back to their own
//        features (two pieces per row; rows >= d of the packed head are the
//        zero padding [d, dp));
//   Q/K, plain order: the chunk's features as one piece per row;
//   V:   rows of V^T (feature-major), one 64-byte warp store per feature.
// Q/K rows go straight to global memory; with CW = 32 a 4 x 4 shuffle
// transpose inside each group of 4 lanes makes lanes 4g..4g+3 write the four
// 16-byte pieces of one row per store instruction.
// `bl`: lane l holds the bias of the chunk's column l (fetched by the caller
// before its wait for the accumulator), handed to every lane by shuffles.
template <int CW>
// (sec, hd, r0): section (Q, K, V), head and packed row inside the head of the
// chunk's first column F0, kept by the caller without divisions.
__device__ __forceinline__ void res_epi_chunk(const ResArgs &args, uint32_t taddr, int F0, int sec, int hd, int r0,
                                              int b, int p0, int q4, int lane, const float2 *th, float bl) {
  uint32_t r[CW];
  if constexpr (CW == 32) tmem_ld32(taddr, r);
  else tmem_ld16(taddr, r);
  tmem_wait_ld();
  float v[CW];
#pragma unroll
  for (int k = 0; k < CW; ++k) v[k] = __uint_as_float(r[k]) + __shfl_sync(0xFFFFFFFFu, bl, k);
  (void)F0;
  const int row = q4 * 32 + lane;
  const int pix = p0 + row;
  if (sec == 2) {
    // V^T row e holds feature e for every pixel: each store instruction of the
    // warp writes 32 consecutive pixels (64 contiguous bytes) of one row.
    // (Staging the rows in shared memory for TMA stores measured 2 us slower
    // on both large workloads.)
    if (pix < args.N) {
      uint16_t *dst = args.vt + (((long long)b * args.h + hd) * args.dp + r0) * args.ldn + pix;
#pragma unroll
      for (int k = 0; k < CW; ++k) dst[(long long)k * args.ldn] = op_bits(v[k]);
    }
    return;
  }
  const long long bh = (long long)b * args.h + hd;
  uint16_t *qk = (sec == 0 ? args.q : args.k) + bh * args.N * args.ldq;
  const int j4 = lane & 3, g4 = lane & ~3;
  if (args.inter) {
    const int hd2 = args.d >> 1;
    const int i0 = r0 >> 1;
    const int npair = max(0, min(hd2 - i0, CW / 2));  // pairs of this chunk
    if (args.rope) {
      const float t = (float)pix;
#pragma unroll
      for (int j = 0; j < CW / 2; ++j)
        if (j < npair) rope_pair(v[2 * j], v[2 * j + 1], t, th[i0 + j]);
    }
    if (CW == 32 && npair == 16 && (hd2 & 7) == 0) {
      // four 16-byte pieces per row: x features i0.., i0+8..; y features d/2+i0.., d/2+i0+8..
      uint32_t a[4][4];
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int j = 8 * k + 2 * m;
          a[k][m] = pack_op2(v[2 * j], v[2 * j + 2]);
          a[2 + k][m] = pack_op2(v[2 * j + 1], v[2 * j + 3]);
        }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        // transpose the 4 x 4 matrix (lane j of the group, piece k) -> (lane k, piece j)
        const uint32_t s0 = (j4 & 1) ? a[0][m] : a[1][m];
        const uint32_t s1 = (j4 & 1) ? a[2][m] : a[3][m];
        const uint32_t t0 = __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
        const uint32_t t1 = __shfl_xor_sync(0xFFFFFFFFu, s1, 1);
        if (j4 & 1) { a[0][m] = t0; a[2][m] = t1; } else { a[1][m] = t0; a[3][m] = t1; }
        const uint32_t u0 = (j4 & 2) ? a[0][m] : a[2][m];
        const uint32_t u1 = (j4 & 2) ? a[1][m] : a[3][m];
        const uint32_t w0 = __shfl_xor_sync(0xFFFFFFFFu, u0, 2);
        const uint32_t w1 = __shfl_xor_sync(0xFFFFFFFFu, u1, 2);
        if (j4 & 2) { a[0][m] = w0; a[1][m] = w1; } else { a[2][m] = w0; a[3][m] = w1; }
      }
      const int f = (j4 < 2) ? i0 + 8 * j4 : hd2 + i0 + 8 * (j4 - 2);
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        const int rp = p0 + q4 * 32 + g4 + ii;  // row written by this group in store ii
        if (rp < args.N)
          *reinterpret_cast<uint4 *>(qk + (long long)rp * args.ldq + f) = make_uint4(a[ii][0], a[ii][1], a[ii][2], a[ii][3]);
      }
      return;
    }
    if (pix >= args.N) return;
    uint16_t *dst = qk + (long long)pix * args.ldq;
    uint32_t xw[CW / 4], yw[CW / 4];
#pragma unroll
    for (int m = 0; m < CW / 4; ++m) {
      xw[m] = pack_op2(v[4 * m], v[4 * m + 2]);
      yw[m] = pack_op2(v[4 * m + 1], v[4 * m + 3]);
    }
    store_run<CW / 2>(dst + i0, xw, npair);
    store_run<CW / 2>(dst + hd2 + i0, yw, npair);
    // packed rows [d, dp) are the head's zero padding, in place
    for (int f = max(r0, args.d); f < min(r0 + CW, args.dp); ++f) dst[f] = 0;
    return;
  }
  if constexpr (CW == 32) {
    uint32_t a[4][4];  // a[k] = this row's 16-byte piece k (features 8k .. 8k+7)
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int m = 0; m < 4; ++m) a[k][m] = pack_op2(v[8 * k + 2 * m], v[8 * k + 2 * m + 1]);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t s0 = (j4 & 1) ? a[0][m] : a[1][m];
      const uint32_t s1 = (j4 & 1) ? a[2][m] : a[3][m];
      const uint32_t t0 = __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
      const uint32_t t1 = __shfl_xor_sync(0xFFFFFFFFu, s1, 1);
      if (j4 & 1) { a[0][m] = t0; a[2][m] = t1; } else { a[1][m] = t0; a[3][m] = t1; }
      const uint32_t u0 = (j4 & 2) ? a[0][m] : a[2][m];
      const uint32_t u1 = (j4 & 2) ? a[1][m] : a[3][m];
      const uint32_t w0 = __shfl_xor_sync(0xFFFFFFFFu, u0, 2);
      const uint32_t w1 = __shfl_xor_sync(0xFFFFFFFFu, u1, 2);
      if (j4 & 2) { a[0][m] = w0; a[1][m] = w1; } else { a[2][m] = w0; a[3][m] = w1; }
    }
    uint16_t *base = qk + r0 + j4 * 8;
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int rp = p0 + q4 * 32 + g4 + ii;
      if (rp < args.N)
        *reinterpret_cast<uint4 *>(base + (long long)rp * args.ldq) = make_uint4(a[ii][0], a[ii][1], a[ii][2], a[ii][3]);
    }
  } else {
    if (pix >= args.N) return;
    uint16_t *dst = qk + (long long)pix * args.ldq + r0;
    uint4 w0, w1;
    w0.x = pack_op2(v[0], v[1]); w0.y = pack_op2(v[2], v[3]);
    w0.z = pack_op2(v[4], v[5]); w0.w = pack_op2(v[6], v[7]);
    w1.x = pack_op2(v[8], v[9]); w1.y = pack_op2(v[10], v[11]);
    w1.z = pack_op2(v[12], v[13]); w1.w = pack_op2(v[14], v[15]);
    reinterpret_cast<uint4 *>(dst)[0] = w0;
    reinterpret_cast<uint4 *>(dst)[1] = w1;
  }
}

template <int DT>
__global__ void __launch_bounds__(RTHREADS, 1)
    qkv_resident_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                        const ResArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw;
  // The layout needs a 1024-byte aligned base (128B-swizzled operands) and
  // leaves no room to realign: refuse to run otherwise.
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicOr(args.err, (uint32_t)DEV_MISALIGNED);
    return;
  }
  const int nkb = args.nkb;
  const int nwl = (nkb + 1) / 2;  // weight loads per slice (two k-blocks each)
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + RES_BARS_OFF);
  uint64_t *full = bars;
  uint64_t *empty = bars + RNST;
  uint64_t *xfree = bars + 2 * RNST;
  uint64_t *a_ready = bars + 3 * RNST;
  uint64_t *acc_full = a_ready + 1;   // [2]
  uint64_t *acc_empty = acc_full + 2; // [2]
  uint64_t *drain = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + RNBARS);
  volatile uint32_t *abort_flag = tmem_slot + 1;
  uint8_t *ring = sm;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x;
  const int p0 = blockIdx.y * BM;
  const int b = blockIdx.z;
  const int sl0 = g * args.spg;
  const int nsl = min(args.spg, args.nslices - sl0);  // slices of this CTA
  const int nloads = nkb + nsl * nwl;                  // x blocks, then weight pairs
  // Slices are swept starting at a tile-dependent one: all CTAs walking the
  // weights in the same order request the same tiles at the same time, and
  // those L2 lines then serve one request after another (measured ~48 GB/s
  // per SM of weight feed that way).
  const int rot = nsl > 0 ? (int)(blockIdx.y % (unsigned)nsl) : 0;
  const uint32_t wbytes = (uint32_t)args.BN * BK * 2;  // one [BN][64] k-block

  if (threadIdx.x == 0) {
    for (int i = 0; i < RNST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&xfree[i], NCONV);
    }
    mbar_init(a_ready, NCONV);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], NCONV);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&wmap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();
  pdl_wait();  // inputs of the previous kernel visible from here on
  const Abort ab{abort_flag, args.err, args.timeout_ns};

  if (warp == 0 || warp == 10) {
    // ------------------------------------------------------------ producers
    // Load t uses slot t mod RNST.  Before refilling a slot the producer waits
    // for the release of the slot's previous load: by the converters (xfree)
    // for an x block, by the MMA's commit (empty) for a weight pair.  Each
    // barrier completes once per load of its kind in that slot, in order.
    if (lane == 0) {
      const int me = warp == 0 ? 0 : 1;
      int last = -1;
      bool stalled = false;
      for (int t = me; t < nloads; t += 2) {
        if (args.stall && (uint32_t)t >= args.stall) { stalled = true; break; }  // test hook
        const int s = t % RNST;
        const int prev = t - RNST;
        if (prev >= 0) {
          bool okw;
          if (prev < nkb) {
            okw = mbar_wait(&xfree[s], (uint32_t)((prev / RNST) & 1), ab);
          } else {
            const int first_w = nkb + ((s - nkb % RNST) + RNST) % RNST;  // first weight load in slot s
            okw = mbar_wait(&empty[s], (uint32_t)(((prev - first_w) / RNST) & 1), ab);
          }
          if (!okw) break;
        }
        if (t < nkb) {
          mbar_arrive_expect_tx(&full[s], (uint32_t)args.xbytes);
          tma_load_3d(ring + s * RSLOT, &xmap, &full[s], p0, t * BK, b);
        } else {
          const int i = (t - nkb) / nwl, kp = (t - nkb) % nwl;
          const int kb0 = 2 * kp, nk = min(2, nkb - kb0);
          const int sl = sl0 + (i + rot) % nsl;
          if (args.w3d) {
            // One box of two 64-channel chunks x BN rows (a chunk index past
            // the last reads as zeros).
            mbar_arrive_expect_tx(&full[s], 2u * wbytes);
            tma_load_3d(ring + s * RSLOT, &wmap, &full[s], 0, sl * args.BN, kb0);
          } else {
            mbar_arrive_expect_tx(&full[s], (uint32_t)nk * wbytes);
            for (int u = 0; u < nk; ++u)
              tma_load_2d(ring + s * RSLOT + u * wbytes, &wmap, &full[s], (kb0 + u) * BK, sl * args.BN);
          }
        }
        last = t;
      }
      if (*abort_flag || stalled)
        for (int t = last; t >= 0 && t > last - 2 * RNST; t -= 2)
          mbar_wait_drain(&full[t % RNST], (uint32_t)((t / RNST) & 1), drain_limit(ab));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA warp
    const uint32_t idesc = idesc_f16(BM, (uint32_t)args.BN);
    const uint64_t rd = sdesc_k128(smem_u32(ring));
    bool ok = mbar_wait_warp(a_ready, 0, ab), issued = false;
    tc_fence_after();
    int t = nkb;
    for (int i = 0; i < nsl && ok; ++i) {
      const int buf = i & 1;
      if (i >= 2 && !mbar_wait_warp(&acc_empty[buf], (uint32_t)(((i >> 1) - 1) & 1), ab)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(buf * 128);
      for (int kp = 0; kp < nwl && ok; ++kp, ++t) {
        const int s = t % RNST;
        if (!mbar_wait_warp(&full[s], (uint32_t)((t / RNST) & 1), ab)) { ok = false; break; }
        tc_fence_after();
        const int nk = min(2, nkb - 2 * kp);
        if (elect_one()) {
          for (int u = 0; u < nk; ++u) {
            const int kb = 2 * kp + u;
            const uint64_t b0 = rd + (uint64_t)((s * RSLOT + u * (int)wbytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)  // A: 16 channels = 8 columns per step
              mma_f16_ts(d, tmem + RA_COL + (uint32_t)(kb * 32 + kk * 8), b0 + (uint64_t)(kk * 2), idesc,
                         (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        __syncwarp();
        issued = true;
      }
      if (ok) {
        if (elect_one()) mma_commit(&acc_full[buf]);
        __syncwarp();
      }
    }
    if (issued) {  // every issued MMA completes before tensor memory is freed
      if (elect_one()) mma_commit(drain);
      __syncwarp();
      mbar_wait_drain(drain, 0, drain_limit(ab));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ converters
    // Warp (q4, hc) converts pixels q4*32 + lane (its tensor-memory lanes) and
    // channels hc*32 .. +31 of each k-block into 16 A columns (fp16 pairs).
    const int cw = warp - 2;                 // 0..7
    const int q4 = warp & 3;                 // TMEM lane quarter of this warp
    const int px = q4 * 32 + lane;           // pixel row of the A tile
    const int hc = cw >> 2;                  // channel half of a k-block
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    float *slot = reinterpret_cast<float *>(sm + RES_SLOT_OFF + cw * 256);
    const float *ga = args.ga + (long long)b * args.C;
    const float *gs = args.gs + (long long)b * args.C;
    bool ok = true;
    for (int kb = 0; kb < nkb && ok; ++kb) {
      const int s = kb % RNST;
      const int c = kb * BK + hc * 32 + lane;
      const float a_c = c < args.C ? __ldg(ga + c) : 0.f;
      const float s_c = c < args.C ? __ldg(gs + c) : 0.f;
      if (!mbar_wait_warp(&full[s], (uint32_t)((kb / RNST) & 1), ab)) { ok = false; break; }
      __syncwarp();
      slot[lane] = a_c;
      slot[32 + lane] = s_c;
      __syncwarp();
      const uint8_t *xs = ring + s * RSLOT;
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int ch = hc * 32 + 2 * i;
        float x0, x1;
        if (DT == 0) {
          x0 = reinterpret_cast<const float *>(xs)[ch * BM + px];
          x1 = reinterpret_cast<const float *>(xs)[(ch + 1) * BM + px];
        } else {
          x0 = __uint_as_float(((uint32_t)reinterpret_cast<const unsigned short *>(xs)[ch * BM + px]) << 16);
          x1 = __uint_as_float(((uint32_t)reinterpret_cast<const unsigned short *>(xs)[(ch + 1) * BM + px]) << 16);
        }
        // channels past C are zero (their scale and shift are zero)
        w[i] = pack_op2(fmaf(slot[2 * i], x0, slot[32 + 2 * i]), fmaf(slot[2 * i + 1], x1, slot[32 + 2 * i + 1]));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&xfree[s]);  // the x block has been read
      tmem_st16(lane_base + RA_COL + (uint32_t)(kb * 32 + hc * 16), w);
    }
    tmem_wait_st();  // also after an abort: no store may be pending when tensor memory is freed
    if (ok) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(a_ready);
    }
    // ------------------------------------------------------------ epilogues
    // Rotation thetas in the converters' (now idle) scale/shift slots.  Every
    // epilogue warp takes both barriers, whatever its state.
    float2 *th = reinterpret_cast<float2 *>(sm + RES_SLOT_OFF);
    if (args.rope) {
      named_bar_sync(1, NCONV * 32);
      rope_thetas(th, args.d, cw * 32 + lane, NCONV * 32);
      named_bar_sync(1, NCONV * 32);
    }
    const int nch = args.BN / args.cw;
    for (int i = 0; i < nsl && ok; ++i) {
      const int buf = i & 1;
      const int fs = (sl0 + (i + rot) % nsl) * args.BN;
      // this warp's chunk biases (lane l: column l of chunk u), fetched before
      // the wait so their latency hides behind it
      float bl[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = hc + 2 * u;
        bl[u] = (c < nch && lane < args.cw) ? __ldg(args.bias + fs + c * args.cw + lane) : 0.f;
      }
      if (!mbar_wait_warp(&acc_full[buf], (uint32_t)((i >> 1) & 1), ab)) { ok = false; break; }
      tc_fence_after();
      const uint32_t acc = lane_base + (uint32_t)(buf * 128);
      // Section, head and row of this warp's first chunk, then advanced by
      // two chunks at a time (no integer division per chunk).
      int F0 = fs + hc * args.cw;
      int ec = F0 / args.dp;
      int er0 = F0 - ec * args.dp;
      int esec = ec / args.h;
      int ehd = ec - esec * args.h;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = hc + 2 * u;
        if (c >= nch) break;
        if (args.cw == 32)
          res_epi_chunk<32>(args, acc + (uint32_t)(c * 32), F0, esec, ehd, er0, b, p0, q4, lane, th, bl[u]);
        else
          res_epi_chunk<16>(args, acc + (uint32_t)(c * 16), F0, esec, ehd, er0, b, p0, q4, lane, th, bl[u]);
        F0 += 2 * args.cw;
        er0 += 2 * args.cw;
        while (er0 >= args.dp) {
          er0 -= args.dp;
          if (++ehd == args.h) {
            ehd = 0;
            ++esec;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The resident-tile kernel serves C <= 512 (the A tile fits tensor-memory
// columns 256..511) when the device grants its shared memory.
bool resident_ok(const Dims &dm) {
  int max_smem = 232448, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return (dm.C + BK - 1) / BK <= 8 && (int)RES_SMEM <= max_smem;
}

int pick_bn(int ntot) {
  for (int bn = 256; bn >= 16; bn -= 16)
    if (ntot % bn == 0) return bn;
  return 16;
}

}  // namespace

bool qk_pair_interleaved(const Dims &dm) {
  if (dm.h <= 0 || dm.d % 16) return false;
  return resident_ok(dm) || dm.dp == dm.d;
}

int launch_qkv_gemm(const Dims &dm, int dtype, const void *x, int ldx, const float *ga, const float *gs,
                    const uint16_t *w_qkv, const float *b_qkv, uint16_t *q, uint16_t *k, uint16_t *vt,
                    const KParams &kp, cudaStream_t st, int rope) {
  const int es = dtype == 0 ? 4 : 2;
  const int inter = qk_pair_interleaved(dm) ? 1 : 0;
  if (rope && !inter) return 2;  // the fused rotation needs pair-interleaved Q/K rows
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
  CUtensorMap xmap_g;  // the general kernel's x stage: 128-byte-wide swizzled boxes
  {
    const uint64_t dims[3] = {(uint64_t)dm.N, (uint64_t)dm.C, (uint64_t)dm.B};
    const uint64_t strides[2] = {(uint64_t)ldx * es, (uint64_t)dm.C * ldx * es};
    const uint32_t box[3] = {(uint32_t)(128 / es), BK, 1};
    if (encode_tiled(&xmap_g, dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
  }
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
    // pair-interleaved rows leave the general kernel as 8-feature halves
    const uint32_t box[3] = {(uint32_t)((inter && !resident_ok(dm)) ? 8 : 16), BM, 1};
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
  const int nkb = (dm.C + BK - 1) / BK;
  int dev = 0;
  (void)cudaGetDevice(&dev);
  // Resident tile: A (C/2 columns) must fit tensor-memory columns 256..511,
  // a slice (BN <= 128 features) one 128-column accumulator.
  int BNr = 0;
  for (int bn = 128; bn >= 16; bn -= 16)
    if (dm.ntot % bn == 0) {
      BNr = bn;
      break;
    }
  if (resident_ok(dm) && BNr > 0 && BM * BK * es <= RSLOT) {
    CUtensorMap wmap_r;
    const int w3d = (dm.C % BK == 0) ? 1 : 0;
    if (w3d) {
      // W viewed as [64-channel chunk][feature][64 channels]: one box = two
      // chunks x BN features (32 KB for BN = 128), one TMA per ring slot --
      // half the TMA instructions of two 2-D boxes.  Only when every chunk
      // lies inside a row (C % 64 == 0).
      const uint64_t dims[3] = {64, (uint64_t)dm.ntot, (uint64_t)(dm.C / BK)};
      const uint64_t strides[2] = {(uint64_t)dm.ldc * 2, 128};
      const uint32_t box[3] = {BK, (uint32_t)BNr, 2};
      if (encode_tiled(&wmap_r, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, w_qkv, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return 1;
    } else {
      const uint64_t dims[2] = {(uint64_t)dm.C, (uint64_t)dm.ntot};
      const uint64_t strides[1] = {(uint64_t)dm.ldc * 2};
      const uint32_t box[2] = {BK, (uint32_t)BNr};
      if (encode_tiled(&wmap_r, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w_qkv, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return 1;
    }
    int nsm = 148;
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int mtiles = dm.B * ((dm.N + BM - 1) / BM);
    const int nslices = dm.ntot / BNr;
    int ng = nsm / mtiles;
    if (ng < 1) ng = 1;
    if (ng > nslices) ng = nslices;
    const int spg = (nslices + ng - 1) / ng;
    ng = (nslices + spg - 1) / spg;
    ResArgs r{};
    r.C = dm.C; r.N = dm.N; r.h = dm.h; r.dp = dm.dp; r.ldq = dm.ldq; r.ldn = dm.ldn; r.BN = BNr;
    r.nkb = nkb; r.nslices = nslices; r.spg = spg; r.xbytes = BM * BK * es; r.w3d = w3d;
    r.cw = (dm.dp % 32 == 0 && BNr % 64 == 0) ? 32 : 16;
    r.d = dm.d; r.inter = inter; r.rope = rope ? 1 : 0; r.stall = stall_for(kp, STALL_QKV);
    r.ga = ga; r.gs = gs; r.bias = b_qkv; r.q = q; r.k = k; r.vt = vt;
    r.err = kp.err; r.timeout_ns = kp.timeout_ns;
    const uint32_t smem = RES_SMEM;
    const dim3 grid(ng, (dm.N + BM - 1) / BM, dm.B);
    if (dtype == 0) {
      cudaFuncSetAttribute(qkv_resident_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      (void)launch_k(qkv_resident_kernel<0>, dim3(grid), dim3(RTHREADS), smem, st, xmap, wmap_r, r);
    } else {
      cudaFuncSetAttribute(qkv_resident_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      (void)launch_k(qkv_resident_kernel<1>, dim3(grid), dim3(RTHREADS), smem, st, xmap, wmap_r, r);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
  }
  // Here pair-interleaved rows always mean d == dp and d % 16 == 0
  // (qk_pair_interleaved), so every 16-feature chunk holds 8 whole pairs and
  // both of its 8-feature halves start 16-byte aligned.
  if (inter && !(dm.dp == dm.d && dm.d % 16 == 0)) return 2;
  QkvArgs a{};
  a.C = dm.C; a.N = dm.N; a.h = dm.h; a.dp = dm.dp; a.ldq = dm.ldq; a.ldn = dm.ldn; a.BN = BN;
  a.d = dm.d; a.inter = inter; a.rope = rope ? 1 : 0; a.stall = stall_for(kp, STALL_QKV);
  a.nk = (dm.C + BK - 1) / BK;
  a.tmem_cols = BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
  a.xbytes = BM * BK * es;
  a.ga = ga; a.gs = gs; a.bias = b_qkv; a.q = q; a.k = k; a.vt = vt;
  a.err = kp.err; a.timeout_ns = kp.timeout_ns;
  // x stages: as many as fit (up to 4), so x loads run ahead of the
  // conversion instead of waiting for it two blocks back.
  int max_smem_q = 232448;
  cudaDeviceGetAttribute(&max_smem_q, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  a.xst = XST;
  while (a.xst > 2 && (int)smem_total(a.xbytes, BN, a.xst) > max_smem_q) --a.xst;
  const uint32_t smem = smem_total(a.xbytes, BN, a.xst);
  const dim3 grid(dm.ntot / BN, (dm.N + BM - 1) / BM, dm.B);
  if (dtype == 0) {
    cudaFuncSetAttribute(qkv_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    (void)launch_k(qkv_gemm_kernel<0>, dim3(grid), dim3(THREADS), smem, st, xmap_g, wmap, qmap, kmap, vmap, a);
  } else {
    cudaFuncSetAttribute(qkv_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    (void)launch_k(qkv_gemm_kernel<1>, dim3(grid), dim3(THREADS), smem, st, xmap_g, wmap, qmap, kmap, vmap, a);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace ssa
