// out_proj.cu -- out = x + image([O_1..O_n] Wo^T + bo), in x's dtype
// (tensortonic "diffusion-l03-spatial-self-attention", block equation and the
// return rule; the image step undoes the tokens step, row i*W + j -> (i, j)).
//
// One CTA computes a 128-pixel x BN-channel tile (M = pixels of one sample,
// N = output channels, K = C):
//   warp 0      TMA producer: the residual tile x[b, n0:n0+BN, p0:p0+128]
//               (NCHW, x's dtype) once, then the O tile [128 pixels][64
//               channels] and the Wo tile [BN][64] per K step (fp16,
//               128-byte swizzle, K-major)
//   warp 1      tcgen05 MMA issuer, fp32 accumulator in tensor memory
//   warps 2..9  epilogue: tensor-memory lane = pixel, column = channel.  Each
//               thread adds its accumulator row and the bias into the staged
//               residual tile in place (x + y, one rounding to x's dtype);
//               one thread then writes the whole tile back to out with a
//               single TMA store, which clips at the image and channel edges.
// When a channel row of x is not a whole number of 16-byte units (H*W*sizeof
// not a multiple of 16) TMA cannot address it, and the epilogue reads x and
// writes out directly instead (all reads of a chunk before its writes: out
// may alias x).
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
  int C, N, BN, nk, tmem_cols, tma_epi, es;
  uint32_t stall;  // test hook: the producer stops after this many operand loads (0: never)
  const float *bias;
  const void *x;
  void *out;
  uint32_t *err;
  uint64_t timeout_ns;
};

__host__ __device__ inline uint32_t xs_off(int BN) { return ST * (BM * BK * 2 + BN * BK * 2); }
__host__ __device__ inline uint32_t bars_off(int BN, int tma_epi, int es) {
  return xs_off(BN) + (tma_epi ? (uint32_t)(BN * BM * es) : 0u);
}
// full[ST], empty[ST], acc_full, drain, x_full, epi_done
constexpr int NBARS = 2 * ST + 4;
__host__ __device__ inline uint32_t smem_total(int BN, int tma_epi, int es) {
  return bars_off(BN, tma_epi, es) + NBARS * 8 + 16 + 1024;
}

template <int DT>
__global__ void __launch_bounds__(THREADS, 1)
    out_proj_kernel(const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap outmap,
                    const OutArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = args.BN;
  const bool tma_epi = args.tma_epi != 0;
  const uint32_t a_off = 0, b_off = ST * (BM * BK * 2);
  uint8_t *xs = sm + xs_off(BN);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + bars_off(BN, args.tma_epi, args.es));
  uint64_t *full = bars;
  uint64_t *empty = bars + ST;
  uint64_t *acc_full = bars + 2 * ST;
  uint64_t *drain = acc_full + 1;
  uint64_t *x_full = drain + 1;
  uint64_t *epi_done = x_full + 1;
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
    mbar_init(x_full, 1);
    mbar_init(epi_done, NEPI);
    *abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&omap);
    tma_prefetch_desc(&wmap);
    if (tma_epi) {
      tma_prefetch_desc(&xmap);
      tma_prefetch_desc(&outmap);
    }
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
    if (lane == 0) {
      if (tma_epi) {
        mbar_arrive_expect_tx(x_full, (uint32_t)(BN * BM * args.es));
        tma_load_3d(xs, &xmap, x_full, p0, n0, b);
      }
      int it = 0;
      const uint32_t bytes = (uint32_t)(BM * BK * 2 + BN * BK * 2);
      for (; it < nk; ++it) {
        if (args.stall && (uint32_t)it >= args.stall) break;  // test hook: consumers' waits expire
        const int s = it % ST;
        if (it >= ST && !mbar_wait(&empty[s], ((it / ST) - 1) & 1, ab)) break;
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_3d(sm + a_off + s * (BM * BK * 2), &omap, &full[s], it * BK, p0, b);
        tma_load_2d(sm + b_off + s * (BN * BK * 2), &wmap, &full[s], it * BK, n0);
      }
      for (int i = (it > ST ? it - ST : 0); i < it; ++i) mbar_wait_drain(&full[i % ST], (i / ST) & 1, drain_limit(ab));
      if (tma_epi) mbar_wait_drain(x_full, 0, drain_limit(ab));
    }
    __syncwarp();
  } else if (warp == 1) {
    // The whole warp runs the loop and the elected lane 0 issues.
    {
      const uint32_t idesc = idesc_f16(BM, (uint32_t)BN);
      const uint64_t ad = sdesc_k128(smem_u32(sm + a_off));
      const uint64_t bd = sdesc_k128(smem_u32(sm + b_off));
      bool ok = true, issued = false;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % ST;
        if (!mbar_wait_warp(&full[s], (kb / ST) & 1, ab)) { ok = false; break; }
        tc_fence_after();
        const uint64_t a0 = ad + (uint64_t)((s * (BM * BK * 2)) >> 4);
        const uint64_t b0 = bd + (uint64_t)((s * (BN * BK * 2)) >> 4);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_f16_ss(tmem, a0 + (uint64_t)(kk * 2), b0 + (uint64_t)(kk * 2), idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit(&empty[s]);
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
    const int ew = warp - 2;
    const int q4 = warp & 3;
    const int half = ew >> 2;
    const int row = q4 * 32 + lane;
    const int p = p0 + row;
    bool ok = mbar_wait_warp(acc_full, 0, ab);
    if (ok && tma_epi) ok = mbar_wait_warp(x_full, 0, ab);
    if (ok) {
      __syncwarp();
      tc_fence_after();
      if (tma_epi) {
        // In place over the staged residual tile xs[channel][pixel].
        for (int c16 = half; c16 < BN / 16; c16 += 2) {
          uint32_t r[16];
          tmem_ld16(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(c16 * 16), r);
          // the chunk's biases, loaded while the accumulator load is in flight
          float bv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = n0 + c16 * 16 + i;
            bv[i] = c < args.C ? __ldg(args.bias + c) : 0.f;
          }
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int cl = c16 * 16 + i;
            const float bias = bv[i];
            if (DT == 0) {
              float *px = reinterpret_cast<float *>(xs) + cl * BM + row;
              *px = *px + (__uint_as_float(r[i]) + bias);
            } else {
              __nv_bfloat16 *px = reinterpret_cast<__nv_bfloat16 *>(xs) + cl * BM + row;
              const float xv = __bfloat162float(*px);
              *px = __float2bfloat16_rn(xv + (__uint_as_float(r[i]) + bias));
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(epi_done);
        if (ew == 0 && lane == 0 && mbar_wait(epi_done, 0, ab)) {
          tma_store_3d(&outmap, xs, p0, n0, b);
          tma_store_commit();
          tma_store_wait_all();
        }
      } else {
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)args.tmem_cols);
  }
}


// ---------------------------------------------------------------------------
// Resident variant (C <= 512, TMA-addressable x/out): one CTA owns 128 pixels
// and ALL output channels -- the O tile (128 x C fp16) is loaded once and
// stays in shared memory, Wo streams through a ring, and the whole 128 x C
// accumulator lives in tensor memory (C <= 512 columns).  After the MMAs the
// freed shared memory holds two residual pieces [128 channels][128 pixels] at
// a time: TMA loads x, eight warps add the accumulator and bias in place, TMA
// stores out (out may alias x: each piece is read before it is written and
// no CTA touches another CTA's pixels).
//   warps 0, 10  TMA producers (O tile and Wo tiles; warp 0 also runs the
//                residual pieces' loads and stores)
//   warp 1       MMA warp (warp-uniform loop, elected lane issues)
//   warps 2..9   epilogue
constexpr int ORNST = 3;
constexpr int ORSLOT = 32768;
constexpr int ORTHREADS = 352;

struct OutResArgs {
  int C, N, nkb, nch, BNc, npieces, es;
  uint32_t stall;  // test hook: each producer stops at this weight-load index (0: never)
  const float *bias;
  uint32_t *err;
  uint64_t timeout_ns;
};
// a_full, full[ORNST], empty[ORNST], acc_full, xfull[2], piece_done[2], drain
constexpr int ORNBARS = 2 * ORNST + 7;
__host__ __device__ inline uint32_t ores_ring_off(int nkb) { return (uint32_t)nkb * 16384u; }
__host__ __device__ inline uint32_t ores_bars_off(int nkb) { return ores_ring_off(nkb) + ORNST * ORSLOT; }
__host__ __device__ inline uint32_t ores_smem(int nkb) { return ores_bars_off(nkb) + ORNBARS * 8 + 16; }

template <int DT>
__global__ void __launch_bounds__(ORTHREADS, 1)
    out_proj_resident_kernel(const __grid_constant__ CUtensorMap omap, const __grid_constant__ CUtensorMap wmap,
                             const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap outmap,
                             const OutResArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw;
  // The layout needs a 1024-byte aligned base (128B-swizzled operands) and
  // leaves no room to realign: refuse to run otherwise.
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicOr(args.err, (uint32_t)DEV_MISALIGNED);
    return;
  }
  const int nkb = args.nkb, nch = args.nch, BNc = args.BNc;
  uint8_t *ring = sm + ores_ring_off(nkb);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + ores_bars_off(nkb));
  uint64_t *a_full = bars;
  uint64_t *full = bars + 1;
  uint64_t *empty = full + ORNST;
  uint64_t *acc_full = empty + ORNST;
  uint64_t *xfull = acc_full + 1;       // [2]
  uint64_t *piece_done = xfull + 2;     // [2]
  uint64_t *drain = piece_done + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + ORNBARS);
  volatile uint32_t *abort_flag = tmem_slot + 1;
  const uint32_t piece_bytes = (uint32_t)(128 * 128 * args.es);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p0 = blockIdx.x * BM;
  const int b = blockIdx.y;
  const int nloads = nkb * nch;
  // k-blocks are taken from a tile-dependent one on: CTAs walking the weights
  // in one order request the same L2 lines at the same time.
  const int rot = (int)(blockIdx.x % (unsigned)nkb);

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    for (int i = 0; i < ORNST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(acc_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&xfull[i], 1);
      mbar_init(&piece_done[i], NEPI);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&omap);
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&outmap);
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
    if (lane == 0) {
      const int me = warp == 0 ? 0 : 1;
      bool ok = true;
      if (me == 0) {
        mbar_arrive_expect_tx(a_full, (uint32_t)(nkb * 16384));
        for (int kb = 0; kb < nkb; ++kb) tma_load_3d(sm + kb * 16384, &omap, a_full, kb * BK, p0, b);
      } else {
        // Pull this tile's residual into L2 while the MMAs run.
        for (int k = 0; k < args.npieces; ++k) tma_prefetch_3d(&xmap, p0, k * 128, b);
      }
      int last = -1;
      bool stalled = false;
      for (int t = me; t < nloads; t += 2) {
        if (args.stall && (uint32_t)t >= args.stall) { stalled = true; break; }  // test hook
        const int s = t % ORNST;
        if (t >= ORNST && !mbar_wait(&empty[s], (uint32_t)(((t / ORNST) - 1) & 1), ab)) { ok = false; break; }
        mbar_arrive_expect_tx(&full[s], (uint32_t)(BNc * BK * 2));
        tma_load_2d(ring + s * ORSLOT, &wmap, &full[s], ((t / nch + rot) % nkb) * BK, (t % nch) * BNc);
        last = t;
      }
      if (*abort_flag || stalled) {
        for (int t = last; t >= 0 && t > last - 2 * ORNST; t -= 2)
          mbar_wait_drain(&full[t % ORNST], (uint32_t)((t / ORNST) & 1), drain_limit(ab));
        if (me == 0) mbar_wait_drain(a_full, 0, drain_limit(ab));
      }
      int nxl[2] = {0, 0};  // residual pieces loaded into each buffer
      if (me == 0 && ok && !*abort_flag) {
        // Residual pieces, once every MMA (the last readers of the shared
        // memory they reuse) has completed.
        if (mbar_wait(acc_full, 0, ab)) {
          for (int k = 0; k < 2 && k < args.npieces; ++k) {
            mbar_arrive_expect_tx(&xfull[k], piece_bytes);
            tma_load_3d(sm + k * piece_bytes, &xmap, &xfull[k], p0, k * 128, b);
            ++nxl[k];
          }
          for (int k = 0; k < args.npieces; ++k) {
            const int bf = k & 1;
            if (!mbar_wait(&piece_done[bf], (uint32_t)((k >> 1) & 1), ab)) break;
            tma_store_3d(&outmap, sm + bf * piece_bytes, p0, k * 128, b);
            tma_store_commit();
            if (k + 2 < args.npieces) {
              tma_store_wait_read();  // the buffer's store has read it
              mbar_arrive_expect_tx(&xfull[bf], piece_bytes);
              tma_load_3d(sm + bf * piece_bytes, &xmap, &xfull[bf], p0, (k + 2) * 128, b);
              ++nxl[bf];
            }
          }
          tma_store_wait_all();
        }
        // Each buffer's last load (phase nxl - 1) must have landed.
        if (*abort_flag)
          for (int k = 0; k < 2; ++k)
            if (nxl[k] > 0) mbar_wait_drain(&xfull[k], (uint32_t)((nxl[k] - 1) & 1), drain_limit(ab));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    const uint32_t idesc = idesc_f16(BM, (uint32_t)BNc);
    const uint64_t ad = sdesc_k128(smem_u32(sm));
    const uint64_t rd = sdesc_k128(smem_u32(ring));
    bool ok = mbar_wait_warp(a_full, 0, ab), issued = false;
    for (int t = 0; t < nloads && ok; ++t) {
      const int s = t % ORNST, kpos = t / nch, kb = (kpos + rot) % nkb, c = t % nch;
      if (!mbar_wait_warp(&full[s], (uint32_t)((t / ORNST) & 1), ab)) { ok = false; break; }
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_f16_ss(tmem + (uint32_t)(c * BNc), ad + (uint64_t)(kb * 1024 + kk * 2),
                     rd + (uint64_t)(s * (ORSLOT >> 4) + kk * 2), idesc, (kpos | kk) != 0 ? 1u : 0u);
        mma_commit(&empty[s]);
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
    __syncwarp();
  } else {
    const int ew = warp - 2;
    const int q4 = warp & 3;
    const int half = ew >> 2;
    const int row = q4 * 32 + lane;
    // This warp's biases for every piece, fetched before any wait (lane l
    // holds channel c0 + l of each 32-channel block; C <= 512 here, so at
    // most 4 pieces x 2 blocks).
    float bias_r[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = (u >> 1) * 128 + half * 64 + (u & 1) * 32 + lane;
      bias_r[u] = c < args.C ? __ldg(args.bias + c) : 0.f;
    }
    bool ok = mbar_wait_warp(acc_full, 0, ab);
    for (int k = 0; k < args.npieces && ok; ++k) {
      const int bf = k & 1;
      if (!mbar_wait_warp(&xfull[bf], (uint32_t)((k >> 1) & 1), ab)) { ok = false; break; }
      tc_fence_after();
      uint8_t *xs = sm + bf * piece_bytes;
#pragma unroll
      for (int h32 = 0; h32 < 2; ++h32) {
        const int c32 = h32 * 32;
        const int cl0 = half * 64 + c32;   // channel within the piece
        const int c0 = k * 128 + cl0;      // output channel
        if (c0 >= args.C) break;
        float bl = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          if (kk == k) bl = bias_r[2 * kk + h32];
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float y = __uint_as_float(r[i]) + __shfl_sync(0xFFFFFFFFu, bl, i);
          if (DT == 0) {
            float *px = reinterpret_cast<float *>(xs) + (cl0 + i) * BM + row;
            *px = *px + y;
          } else {
            __nv_bfloat16 *px = reinterpret_cast<__nv_bfloat16 *>(xs) + (cl0 + i) * BM + row;
            *px = __float2bfloat16_rn(__bfloat162float(*px) + y);
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&piece_done[bf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int pick_bn(int C, int cap) {
  const int c16 = (C + 15) / 16 * 16;
  for (int bn = cap; bn >= 16; bn -= 16)
    if (c16 % bn == 0) return bn;
  return 16;
}

}  // namespace

int launch_out_proj(const Dims &dm, int dtype, const uint16_t *o, const uint16_t *w_o, const float *b_o,
                    const void *x, void *out, const KParams &kp, cudaStream_t st) {
  const int es = dtype == 0 ? 4 : 2;
  const int tma_epi = ((long long)dm.N * es) % 16 == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
                              (reinterpret_cast<uintptr_t>(out) & 15u) == 0
                          ? 1
                          : 0;
  int BN = pick_bn(dm.C, tma_epi ? 128 : 256);
  int max_smem = 232448, dev = 0, nsm = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  }
  // Few pixel tiles (at most half as many as SMs): two CTAs per pixel tile,
  // each computing half of the output channels, keep more SMs busy than one
  // CTA per tile with all channels (unet-l1: 64 tiles, block 130 -> 127 us).
  const int mtiles = dm.B * ((dm.N + BM - 1) / BM);
  const bool half_split = tma_epi && 2 * mtiles <= nsm && dm.C % 32 == 0 && dm.C / 2 <= 256 &&
                          (int)smem_total(dm.C / 2, 1, es) <= max_smem;
  if (half_split) BN = dm.C / 2;
  if (!half_split && tma_epi) {
    // Channel tile by a simple cost model: each CTA streams its O tile
    // (16 KB per 64-channel K step) and its Wo slice (BN x 128 bytes per
    // step), so a wave of CTAs costs ~(16384 + 128 BN) per step, and the
    // grid takes ceil(CTAs / (SMs x CTAs per SM)) waves.  E.g. unet-lowres
    // (16 pixel tiles, C = 1280): 160 CTAs of 128 channels ran as 1 + 8/152
    // waves; 128 CTAs of 160 channels take one.
    // Tiles narrower than 64 channels are left out: their N < 64 MMAs run
    // well below the tensor rate.
    const int c16 = (dm.C + 15) / 16 * 16;
    long long best = -1;
    for (int bn = c16 < 64 ? c16 : 64; bn <= 256; bn += 16) {
      const int sm_b = (int)smem_total(bn, 1, es);
      if (c16 % bn != 0 || sm_b > max_smem) continue;
      const long long per_sm = sm_b <= 113 * 1024 ? 2 : 1;
      const long long ctas = (long long)(c16 / bn) * mtiles;
      const long long cost = (ctas + nsm * per_sm - 1) / (nsm * per_sm) * (16384LL + 128LL * bn);
      if (best < 0 || cost < best) {
        best = cost;
        BN = bn;
      }
    }
  }
  CUtensorMap omap, wmap, xmap, outmap;
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
  if (tma_epi) {
    const uint64_t dims[3] = {(uint64_t)dm.N, (uint64_t)dm.C, (uint64_t)dm.B};
    const uint64_t strides[2] = {(uint64_t)dm.N * es, (uint64_t)dm.C * dm.N * es};
    const uint32_t box[3] = {BM, (uint32_t)BN, 1};
    const CUtensorMapDataType dt = dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (encode_tiled(&xmap, dt, 3, x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS) return 1;
    if (encode_tiled(&outmap, dt, 3, out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS) return 1;
  } else {
    xmap = omap;  // unused
    outmap = omap;
  }
  const int nkb = (dm.C + BK - 1) / BK;
  const int c16 = (dm.C + 15) / 16 * 16;
  // The resident form pays off when there are enough pixel tiles to fill the
  // GPU with one CTA each.
  if (!half_split && tma_epi && c16 <= 512 && mtiles >= 64 && (int)ores_smem(nkb) <= max_smem &&
      2u * 128u * 128u * (uint32_t)es <= ores_bars_off(nkb)) {
    const int nch = (c16 + 255) / 256;
    const int BNc = ((c16 / nch + 15) / 16) * 16;
    CUtensorMap wres, xres, outres;
    {
      const uint64_t dims[2] = {(uint64_t)dm.C, (uint64_t)dm.C};
      const uint64_t strides[1] = {(uint64_t)dm.ldc * 2};
      const uint32_t box[2] = {BK, (uint32_t)BNc};
      if (encode_tiled(&wres, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w_o, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return 1;
    }
    {
      const uint64_t dims[3] = {(uint64_t)dm.N, (uint64_t)dm.C, (uint64_t)dm.B};
      const uint64_t strides[2] = {(uint64_t)dm.N * es, (uint64_t)dm.C * dm.N * es};
      const uint32_t box[3] = {BM, 128, 1};
      const CUtensorMapDataType dt = dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      if (encode_tiled(&xres, dt, 3, x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS) return 1;
      if (encode_tiled(&outres, dt, 3, out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS) return 1;
    }
    OutResArgs r{};
    r.C = dm.C; r.N = dm.N; r.nkb = nkb; r.nch = nch; r.BNc = BNc; r.npieces = (dm.C + 127) / 128; r.es = es;
    r.bias = b_o; r.err = kp.err; r.timeout_ns = kp.timeout_ns; r.stall = stall_for(kp, STALL_OUT_PROJ);
    const uint32_t smem = ores_smem(nkb);
    const dim3 grid((dm.N + BM - 1) / BM, dm.B, 1);
    if (dtype == 0) {
      cudaFuncSetAttribute(out_proj_resident_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      (void)launch_k(out_proj_resident_kernel<0>, dim3(grid), dim3(ORTHREADS), smem, st, omap, wres, xres, outres, r);
    } else {
      cudaFuncSetAttribute(out_proj_resident_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      (void)launch_k(out_proj_resident_kernel<1>, dim3(grid), dim3(ORTHREADS), smem, st, omap, wres, xres, outres, r);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 2;
  }
  OutArgs a{};
  a.C = dm.C; a.N = dm.N; a.BN = BN; a.nk = (dm.C + BK - 1) / BK;
  a.tmem_cols = BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
  a.tma_epi = tma_epi; a.es = es;
  a.bias = b_o; a.x = x; a.out = out; a.err = kp.err; a.timeout_ns = kp.timeout_ns;
  a.stall = stall_for(kp, STALL_OUT_PROJ);
  const uint32_t smem = smem_total(BN, tma_epi, es);
  const dim3 grid((dm.C + BN - 1) / BN, (dm.N + BM - 1) / BM, dm.B);
  if (dtype == 0) {
    cudaFuncSetAttribute(out_proj_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    (void)launch_k(out_proj_kernel<0>, dim3(grid), dim3(THREADS), smem, st, omap, wmap, xmap, outmap, a);
  } else {
    cudaFuncSetAttribute(out_proj_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    (void)launch_k(out_proj_kernel<1>, dim3(grid), dim3(THREADS), smem, st, omap, wmap, xmap, outmap, a);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace ssa
