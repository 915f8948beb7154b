// attention.cu -- O_j = softmax(Q_j K_j^T / sqrt(d)) V_j per (sample, head)
// (tensortonic "diffusion-l03-spatial-self-attention", block equation; the
// softmax runs over the key axis and the head outputs are concatenated along
// channels in head order; worked example 1 divides the scores by sqrt(2) for
// d = 2).
//
// Flash-style: one CTA owns 128 queries of one (sample, head) -- and one of
// the two output halves when the padded head dim exceeds 256 -- and walks the
// keys in tiles of 128, so the N x N score matrix never exists.
//   warp 0     TMA producer: Q once, then K and V^T through a ring of slots
//              (16 KB with two CTAs per SM, 32 KB with one) of 128-byte
//              swizzled, K-major boxes: K as [128 keys x 64 dims] per 16 KB,
//              V^T as [<=256 output dims x 64 keys]
//   warp 1     tcgen05 MMA issuer: S = Q K^T into tensor memory, O += P V into
//              a tensor-memory accumulator
//   warps 2-5  softmax: one query row per thread.  Scores come from tensor
//              memory, the 1/sqrt(d) scale and log2(e) fold into one FFMA
//              ahead of ex2, P is rounded to fp16 into a swizzled shared tile
//              for the next MMA.  The running maximum is only raised (and O
//              rescaled in tensor memory) when it grows by more than 2^8,
//              which keeps every P <= 256 and is exact after the final
//              division by the row sum.
// Two score-buffer modes:
//   single  S uses 128 tensor-memory columns; the MMA writes S_{j+1} as soon
//           as the softmax warps have read S_j.  With a small head dim this
//           fits 256 columns and ~113 KB of shared memory, so two CTAs share
//           an SM and their softmax warpgroups overlap.
//   double  S alternates between two 128-column buffers (512 columns in all,
//           one CTA per SM); used when O needs more than 128 columns.
// Keys past N in the last tile are zero-filled by TMA and masked to -inf.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int BLK = 16384;  // one [128 x 64] fp16 swizzled block
constexpr int THREADS = 192;
constexpr int MAX_SMEM_FALLBACK = 232448;
constexpr int SM_SMEM_PER_TWO = 115712;  // per-CTA budget when two CTAs share an SM
constexpr float RESCALE_LOG2 = 8.0f;

struct AttnArgs {
  int N, h, d, dp, ldc, d_o, n_oc, nqb, kpb, nvr, vrows, slot, nst, ntiles, single, tmem_cols, o_col;
  int p_tmem, p_col;  // P in tensor memory (and its column in single mode) or in shared memory
  float sl2;  // log2(e) / sqrt(d)
  uint16_t *o;
  uint32_t *err;
  uint64_t timeout_ns;
};

struct Layout {
  uint32_t q, p, ring, bars;
};
__host__ __device__ inline Layout layout(int nqb, int nst, int slot, int p_tmem) {
  Layout L;
  L.q = 0;
  L.p = nqb * 16384;
  L.ring = L.p + (p_tmem ? 0 : 32768);
  L.bars = L.ring + nst * slot;
  return L;
}
// full[nst], empty[nst], q_full, s_full[2], s_free, p_full, o_done, drain
__host__ __device__ inline int nbars(int nst) { return 2 * nst + 7; }
__host__ __device__ inline uint32_t smem_bytes(int nqb, int nst, int slot, int p_tmem) {
  return layout(nqb, nst, slot, p_tmem).bars + nbars(nst) * 8 + 16 + 1024;
}

template <bool SINGLE>
__global__ void __launch_bounds__(THREADS, SINGLE ? 2 : 1)
    attention_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const AttnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nst = args.nst;
  const int slot = args.slot;
  const Layout L = layout(args.nqb, nst, slot, args.p_tmem);
  const bool p_tmem = args.p_tmem != 0;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L.bars);
  uint64_t *full = bars;
  uint64_t *empty = bars + nst;
  uint64_t *q_full = bars + 2 * nst;
  uint64_t *s_full = q_full + 1;  // [2]
  uint64_t *s_free = s_full + 2;
  uint64_t *p_full = s_free + 1;
  uint64_t *o_done = p_full + 1;
  uint64_t *drain = o_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + nbars(nst));
  volatile uint32_t *abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x / args.n_oc;
  const int oc = blockIdx.x % args.n_oc;
  const int bh = blockIdx.y;
  const int q0 = qt * BQ;
  const int n = args.ntiles;
  constexpr bool single = SINGLE;
  const int nvb = 2 * args.nvr;                         // V slots per key tile
  const int nks = (args.nqb + args.kpb - 1) / args.kpb;  // K slots per key tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(s_free, 4);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
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
  const uint32_t TM_O = (uint32_t)args.o_col;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Block order (the MMA issuer consumes in the same order):
    //   K(0), K(1), then for each tile j: V(j), K(j+2).
    if (lane == 0) {
      int it = 0, s = 0;
      uint32_t ph = 0;  // parity of the ring round of slot s
      bool ok = true;
      mbar_arrive_expect_tx(q_full, (uint32_t)(args.nqb * 16384));
      for (int qb = 0; qb < args.nqb; ++qb) tma_load_3d(sm + L.q + qb * 16384, &qmap, q_full, qb * 64, q0, bh);
      auto acquire = [&]() -> bool { return it < nst || mbar_wait(&empty[s], ph ^ 1u, ab); };
      auto advance = [&]() {
        ++it;
        if (++s == nst) { s = 0; ph ^= 1u; }
      };
      auto load_k = [&](int j) {
        for (int ks = 0; ks < nks && ok; ++ks) {
          if (!acquire()) { ok = false; break; }
          const int nblk = min(args.kpb, args.nqb - ks * args.kpb);
          mbar_arrive_expect_tx(&full[s], (uint32_t)(nblk * BLK));
          for (int bl = 0; bl < nblk; ++bl)
            tma_load_3d(sm + L.ring + s * slot + bl * BLK, &kmap, &full[s], (ks * args.kpb + bl) * 64, j * BKV, bh);
          advance();
        }
      };
      auto load_v = [&](int j) {
        for (int vb = 0; vb < nvb && ok; ++vb) {
          if (!acquire()) { ok = false; break; }
          const int vh = vb / args.nvr, vr = vb - vh * args.nvr;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(args.vrows * 128));
          tma_load_3d(sm + L.ring + s * slot, &vmap, &full[s], j * BKV + 64 * vh, oc * args.d_o + vr * args.vrows, bh);
          advance();
        }
      };
      load_k(0);
      if (n > 1) load_k(1);
      for (int j = 0; j < n && ok; ++j) {
        load_v(j);
        if (j + 2 < n) load_k(j + 2);
      }
      // Never leave with a copy in flight.
      mbar_wait_drain(q_full, 0, ab.limit_ns);
      for (int i = (it > nst ? it - nst : 0); i < it; ++i)
        mbar_wait_drain(&full[i % nst], (i / nst) & 1, ab.limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Descriptors are formed once; a K step (32 B) or a 1024-B block offset
    // inside the swizzled tiles is a small add to the start-address field.
    if (lane == 0) {
      const uint32_t idesc_s = idesc_f16(BQ, BKV);
      const uint32_t idesc_o = idesc_f16(BQ, (uint32_t)args.vrows);
      const uint64_t qd = sdesc_k128(smem_u32(sm + L.q));
      const uint64_t pd = sdesc_k128(smem_u32(sm + L.p));
      const uint64_t rd = sdesc_k128(smem_u32(sm + L.ring));
      const uint32_t slot16 = (uint32_t)slot >> 4;
      const int ksteps = args.dp / 16;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true, issued = false;
      auto advance = [&]() {
        if (++s == nst) { s = 0; ph ^= 1u; }
      };
      auto issue_s = [&](int buf) {
        const uint32_t d_s = tmem + (uint32_t)(buf * BKV);
        for (int ksl = 0; ksl < nks && ok; ++ksl) {
          if (!mbar_wait(&full[s], ph, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bd = rd + (uint64_t)(s * slot16);
          const int nblk = min(args.kpb, args.nqb - ksl * args.kpb);
          for (int bl = 0; bl < nblk; ++bl) {
            const int kb = ksl * args.kpb + bl;
            const uint64_t a0 = qd + (uint64_t)(kb * 1024);
            const uint64_t b0 = bd + (uint64_t)(bl * 1024);
            const int kmax = min(4, ksteps - kb * 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if (kk < kmax) mma_f16_ss(d_s, a0 + (uint64_t)(kk * 2), b0 + (uint64_t)(kk * 2), idesc_s, (kb | kk) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
          issued = true;
          advance();
        }
        if (ok) mma_commit(&s_full[buf]);
      };
      auto issue_pv = [&](int j) {
        const uint32_t pcol = single ? (uint32_t)args.p_col : (uint32_t)((j & 1) * BKV);
        for (int vb = 0; vb < nvb && ok; ++vb) {
          if (!mbar_wait(&full[s], ph, ab)) { ok = false; break; }
          tc_fence_after();
          const int vh = vb / args.nvr, vr = vb - vh * args.nvr;
          const uint32_t d_o = tmem + TM_O + (uint32_t)(vr * args.vrows);
          const uint64_t b0 = rd + (uint64_t)(s * slot16);
          const uint32_t first = (j > 0 || vh > 0) ? 1u : 0u;
          if (p_tmem) {
            const uint32_t a0 = tmem + pcol + (uint32_t)(vh * 32);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts(d_o, a0 + (uint32_t)(kk * 8), b0 + (uint64_t)(kk * 2), idesc_o, (first | kk) ? 1u : 0u);
          } else {
            const uint64_t a0 = pd + (uint64_t)(vh * 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ss(d_o, a0 + (uint64_t)(kk * 2), b0 + (uint64_t)(kk * 2), idesc_o, (first | kk) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
          issued = true;
          advance();
        }
        if (ok) mma_commit(o_done);
      };
      if (!mbar_wait(q_full, 0, ab)) ok = false;
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; j < n && ok; ++j) {
        if (single) {
          if (j + 1 < n) {
            if (!mbar_wait(s_free, j & 1, ab)) { ok = false; break; }
            tc_fence_after();
            issue_s(0);
          }
        } else if (j == 0 && n > 1) {
          issue_s(1);
        }
        if (!ok || !mbar_wait(p_full, j & 1, ab)) { ok = false; break; }
        tc_fence_after();
        issue_pv(j);
        if (!single && j + 2 < n) issue_s(j & 1);
      }
      if (!ok && issued) {
        mma_commit(drain);
        mbar_wait_drain(drain, 0, ab.limit_ns);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const int query = q0 + row;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t p_tile = smem_u32(sm + L.p);
    const float sl2 = args.sl2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int buf = single ? 0 : (j & 1);
      const uint32_t par = single ? (uint32_t)(j & 1) : (uint32_t)((j >> 1) & 1);
      if (!mbar_wait_warp(&s_full[buf], par, ab)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + (uint32_t)(buf * BKV + 32 * c), r[c]);
      tmem_wait_ld();
      if (single) {
        // S has been read into registers: the MMA may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
      }
      const int kvalid = min(BKV, args.N - j * BKV);
      if (kvalid < BKV) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i >= kvalid) r[c][i] = __float_as_uint(-INFINITY);
      }
      // Row maximum: eight independent 3-input max chains.
      float pm[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int c = t >> 1, o = (t & 1) * 16;
        float m = __uint_as_float(r[c][o]);
#pragma unroll
        for (int i = 1; i < 15; i += 2) m = max3f(m, __uint_as_float(r[c][o + i]), __uint_as_float(r[c][o + i + 1]));
        pm[t] = fmaxf(m, __uint_as_float(r[c][o + 15]));
      }
      const float mx = max3f(max3f(pm[0], pm[1], pm[2]), max3f(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
      const float m_new = fmaxf(m_used, mx * sl2);
      // Lazy rescale: a row raises its reference maximum only when the new
      // maximum exceeds it by more than 2^RESCALE_LOG2.  The decision is made
      // per warp (any row that needs it), because the tensor-memory accesses
      // that rescale O are warp-collective; rows that did not need it use
      // their own (possibly unit) factor.
      const bool need = (j > 0) && (m_new > m_used + RESCALE_LOG2);
      const bool rescale = __any_sync(0xFFFFFFFFu, need) != 0;
      float alpha = 1.f;
      if (j == 0) {
        m_used = m_new;
      } else if (rescale && m_new > m_used) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      // p = 2^(s * log2(e)/sqrt(d) - m): one paired FMA per two scores, the
      // row sum in four paired accumulators.
      const uint64_t c2 = f2_pack(sl2, sl2);
      const uint64_t nm2 = f2_pack(-m_used, -m_used);
      uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), c2, nm2), t0, t1);
          const float e0 = ex2_approx(t0);
          const float e1 = ex2_approx(t1);
          acc2[(i >> 3) & 3] = f2_add(acc2[(i >> 3) & 3], f2_pack(e0, e1));
          pk[c >> 1][(c & 1) * 16 + (i >> 1)] = pack_half2(e0, e1);
        }
      float s0, s1, s2, s3;
      f2_unpack(f2_add(acc2[0], acc2[1]), s0, s1);
      f2_unpack(f2_add(acc2[2], acc2[3]), s2, s3);
      const float sum = (s0 + s1) + (s2 + s3);
      l = l * alpha + sum;
      if (j > 0 && !mbar_wait_warp(o_done, (j - 1) & 1, ab)) { ok = false; break; }
      if (rescale) {
        __syncwarp();
        tc_fence_after();
        for (int cc = 0; cc < args.d_o / 16; ++cc) {
          uint32_t t[16];
          tmem_ld16(lane_base + TM_O + (uint32_t)(cc * 16), t);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
          tmem_st16(lane_base + TM_O + (uint32_t)(cc * 16), t);
        }
        tmem_wait_st();
      }
      if (p_tmem) {
        // P as fp16 pairs in tensor memory: over the S buffer just read
        // (double) or in its own 64 columns (single).
        const uint32_t pcol = single ? (uint32_t)args.p_col : (uint32_t)(buf * BKV);
        __syncwarp();
        tmem_st32(lane_base + pcol, pk[0]);
        tmem_st32(lane_base + pcol + 32, pk[1]);
        tmem_wait_st();
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_shared_v4(p_tile + (c >> 3) * 16384 + sw128_offset((uint32_t)row, (uint32_t)(c & 7)),
                       pk[c >> 3][(4 * c) & 31], pk[c >> 3][(4 * c + 1) & 31], pk[c >> 3][(4 * c + 2) & 31],
                       pk[c >> 3][(4 * c + 3) & 31]);
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && mbar_wait_warp(o_done, (n - 1) & 1, ab)) {
      __syncwarp();
      tc_fence_after();
      const float inv = 1.0f / l;
      const int b = bh / args.h, hd = bh % args.h;
      const bool vec = (args.d % 8) == 0;
      uint16_t *orow = args.o + ((long long)b * args.N + query) * args.ldc + (long long)hd * args.d;
      for (int cc = 0; cc < args.d_o / 16; ++cc) {
        uint32_t t[16];
        tmem_ld16(lane_base + TM_O + (uint32_t)(cc * 16), t);
        tmem_wait_ld();
        if (query >= args.N) continue;
        const int e0 = oc * args.d_o + cc * 16;
        if (vec && e0 + 16 <= args.d) {
          uint4 w0, w1;
          w0.x = pack_half2(__uint_as_float(t[0]) * inv, __uint_as_float(t[1]) * inv);
          w0.y = pack_half2(__uint_as_float(t[2]) * inv, __uint_as_float(t[3]) * inv);
          w0.z = pack_half2(__uint_as_float(t[4]) * inv, __uint_as_float(t[5]) * inv);
          w0.w = pack_half2(__uint_as_float(t[6]) * inv, __uint_as_float(t[7]) * inv);
          w1.x = pack_half2(__uint_as_float(t[8]) * inv, __uint_as_float(t[9]) * inv);
          w1.y = pack_half2(__uint_as_float(t[10]) * inv, __uint_as_float(t[11]) * inv);
          w1.z = pack_half2(__uint_as_float(t[12]) * inv, __uint_as_float(t[13]) * inv);
          w1.w = pack_half2(__uint_as_float(t[14]) * inv, __uint_as_float(t[15]) * inv);
          reinterpret_cast<uint4 *>(orow + e0)[0] = w0;
          reinterpret_cast<uint4 *>(orow + e0)[1] = w1;
        } else {
          for (int i = 0; i < 16; ++i) {
            if (e0 + i < args.d) {
              const __half hv = __float2half_rn(__uint_as_float(t[i]) * inv);
              orow[e0 + i] = *reinterpret_cast<const uint16_t *>(&hv);
            }
          }
        }
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
// Wide mode (padded head dim 512, O in two 256-column halves over two CTAs):
// every MMA has N = 256 -- score tiles of 256 keys and a 256-wide P V --
// because on this GPU a stream that mixes MMA widths runs every MMA at the
// N = 256 cadence (the two-buffer kernel above mixes N = 128 scores with an
// N = 256 P V and is capped near half the tensor rate).  Tensor memory holds
// one 256-column score buffer and the 256-column O half; P (fp16, 256 keys)
// overwrites the first 128 columns of the scores it came from, so the score
// MMA of the next tile is issued after P V.  Eight softmax warps: warp
// (q4, half) owns 32 query rows and 128 of the 256 keys; the two halves of a
// row exchange their maxima through shared memory and combine their sums at
// the end.
constexpr int BKW = 256;
constexpr int WSLOT = 32768;
__host__ __device__ inline uint32_t wide_ring_off() { return 8u * 16384u; }  // after Q (128 x 512 fp16)
__host__ __device__ inline uint32_t wide_xch_off(int nst) { return wide_ring_off() + nst * WSLOT; }
__host__ __device__ inline uint32_t wide_bars_off(int nst) { return wide_xch_off(nst) + 2048u; }
// full[nst], empty[nst], q_full, s_full, p_full, o_done, drain, xbar[4]
__host__ __device__ inline int wide_nbars(int nst) { return 2 * nst + 9; }
__host__ __device__ inline uint32_t wide_smem(int nst) { return wide_bars_off(nst) + wide_nbars(nst) * 8 + 16; }

__global__ void __launch_bounds__(320, 1)
    attention_wide_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const AttnArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw;
  // The layout needs a 1024-byte aligned base (128B-swizzled operands) and
  // leaves no room to realign: refuse to run otherwise.
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicOr(args.err, (uint32_t)DEV_MISALIGNED);
    return;
  }
  const int nst = args.nst;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + wide_bars_off(nst));
  uint64_t *full = bars;
  uint64_t *empty = bars + nst;
  uint64_t *q_full = bars + 2 * nst;
  uint64_t *s_full = q_full + 1;
  uint64_t *p_full = s_full + 1;
  uint64_t *o_done = p_full + 1;
  uint64_t *drain = o_done + 1;
  uint64_t *xbar = drain + 1;  // [4]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + wide_nbars(nst));
  volatile uint32_t *abort_flag = tmem_slot + 1;
  float *xch = reinterpret_cast<float *>(sm + wide_xch_off(nst));  // [2 parity][2 half][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x >> 1;
  const int oc = blockIdx.x & 1;
  const int bh = blockIdx.y;
  const int q0 = qt * BQ;
  const int n = (args.N + BKW - 1) / BKW;
  const int nqb = args.nqb;  // 64-wide blocks of the head dim (8)

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 8);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&xbar[i], 2);
    *abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, args.err, args.timeout_ns};
  const uint32_t TM_O = 256;

  if (warp == 0) {
    // Block order: K(0) [nqb slots], then per tile j: V(j) [4 slots], K(j+1).
    if (lane == 0) {
      int it = 0, s = 0;
      uint32_t ph = 0;
      bool ok = true;
      mbar_arrive_expect_tx(q_full, (uint32_t)(nqb * 16384));
      for (int qb = 0; qb < nqb; ++qb) tma_load_3d(sm + qb * 16384, &qmap, q_full, qb * 64, q0, bh);
      auto acquire = [&]() -> bool { return it < nst || mbar_wait(&empty[s], ph ^ 1u, ab); };
      auto advance = [&]() {
        ++it;
        if (++s == nst) { s = 0; ph ^= 1u; }
      };
      auto load_k = [&](int j) {
        for (int kb = 0; kb < nqb && ok; ++kb) {
          if (!acquire()) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], (uint32_t)WSLOT);
          tma_load_3d(sm + wide_ring_off() + s * WSLOT, &kmap, &full[s], kb * 64, j * BKW, bh);
          advance();
        }
      };
      auto load_v = [&](int j) {
        for (int vb = 0; vb < BKW / 64 && ok; ++vb) {
          if (!acquire()) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], (uint32_t)WSLOT);
          tma_load_3d(sm + wide_ring_off() + s * WSLOT, &vmap, &full[s], j * BKW + 64 * vb, oc * 256, bh);
          advance();
        }
      };
      load_k(0);
      for (int j = 0; j < n && ok; ++j) {
        load_v(j);
        if (j + 1 < n) load_k(j + 1);
      }
      mbar_wait_drain(q_full, 0, ab.limit_ns);
      for (int i = (it > nst ? it - nst : 0); i < it; ++i)
        mbar_wait_drain(&full[i % nst], (i / nst) & 1, ab.limit_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(BQ, 256);
      const uint64_t qd = sdesc_k128(smem_u32(sm));
      const uint64_t rd = sdesc_k128(smem_u32(sm + wide_ring_off()));
      const uint32_t slot16 = (uint32_t)WSLOT >> 4;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true, issued = false;
      auto advance = [&]() {
        if (++s == nst) { s = 0; ph ^= 1u; }
      };
      if (!mbar_wait(q_full, 0, ab)) ok = false;
      if (ok) tc_fence_after();
      for (int j = 0; j < n && ok; ++j) {
        // S_j = Q K_j^T (N = 256 keys).  Issued after P V_{j-1}, which reads
        // the P that S_j overwrites (MMAs of one thread execute in order).
        for (int kb = 0; kb < nqb && ok; ++kb) {
          if (!mbar_wait(&full[s], ph, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t a0 = qd + (uint64_t)(kb * 1024);
          const uint64_t b0 = rd + (uint64_t)(s * slot16);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16_ss(tmem, a0 + (uint64_t)(kk * 2), b0 + (uint64_t)(kk * 2), idesc, (kb | kk) ? 1u : 0u);
          mma_commit(&empty[s]);
          issued = true;
          advance();
        }
        if (!ok) break;
        mma_commit(s_full);
        if (!mbar_wait(p_full, j & 1, ab)) { ok = false; break; }
        tc_fence_after();
        // O += P_j V_j: P in tensor memory, key k in column k/2.
        for (int vb = 0; vb < BKW / 64 && ok; ++vb) {
          if (!mbar_wait(&full[s], ph, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t b0 = rd + (uint64_t)(s * slot16);
          const uint32_t first = (j > 0 || vb > 0) ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16_ts(tmem + TM_O, tmem + (uint32_t)(vb * 32 + kk * 8), b0 + (uint64_t)(kk * 2), idesc,
                       (first | kk) ? 1u : 0u);
          mma_commit(&empty[s]);
          issued = true;
          advance();
        }
        if (ok) mma_commit(o_done);
      }
      if (!ok && issued) {
        mma_commit(drain);
        mbar_wait_drain(drain, 0, ab.limit_ns);
      }
    }
    __syncwarp();
  } else {
    const int sw = warp - 2;
    const int q4 = warp & 3;
    const int half = sw >> 2;
    const int row = q4 * 32 + lane;
    const int query = q0 + row;
    const int cb = half * 128;  // this thread's 128 keys of the 256-key tile
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const float sl2 = args.sl2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait_warp(s_full, (uint32_t)(j & 1), ab)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + (uint32_t)(cb + 32 * c), r[c]);
      tmem_wait_ld();
      const int kvalid = min(BKW, args.N - j * BKW) - cb;
      if (kvalid < 128) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i >= kvalid) r[c][i] = __float_as_uint(-INFINITY);
      }
      float pm[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int c = t >> 1, o = (t & 1) * 16;
        float m = __uint_as_float(r[c][o]);
#pragma unroll
        for (int i = 1; i < 15; i += 2) m = max3f(m, __uint_as_float(r[c][o + i]), __uint_as_float(r[c][o + i + 1]));
        pm[t] = fmaxf(m, __uint_as_float(r[c][o + 15]));
      }
      float mx = max3f(max3f(pm[0], pm[1], pm[2]), max3f(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
      // The other half of this row (same lanes, other warp): exchange maxima.
      // This also orders both halves' score reads before either writes P
      // over the score columns.
      xch[((j & 1) * 2 + half) * 128 + row] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xbar[q4]);
      if (!mbar_wait_warp(&xbar[q4], (uint32_t)(j & 1), ab)) { ok = false; break; }
      mx = fmaxf(mx, xch[((j & 1) * 2 + (half ^ 1)) * 128 + row]);
      const float m_new = fmaxf(m_used, mx * sl2);
      const bool need = (j > 0) && (m_new > m_used + RESCALE_LOG2);
      const bool rescale = __any_sync(0xFFFFFFFFu, need) != 0;
      float alpha = 1.f;
      if (j == 0) {
        m_used = m_new;
      } else if (rescale && m_new > m_used) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      const uint64_t c2 = f2_pack(sl2, sl2);
      const uint64_t nm2 = f2_pack(-m_used, -m_used);
      uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), c2, nm2), t0, t1);
          const float e0 = ex2_approx(t0);
          const float e1 = ex2_approx(t1);
          acc2[(i >> 3) & 3] = f2_add(acc2[(i >> 3) & 3], f2_pack(e0, e1));
          pk[c >> 1][(c & 1) * 16 + (i >> 1)] = pack_half2(e0, e1);
        }
      float s0, s1, s2, s3;
      f2_unpack(f2_add(acc2[0], acc2[1]), s0, s1);
      f2_unpack(f2_add(acc2[2], acc2[3]), s2, s3);
      l = l * alpha + ((s0 + s1) + (s2 + s3));
      if (j > 0 && !mbar_wait_warp(o_done, (j - 1) & 1, ab)) { ok = false; break; }
      if (rescale) {
        __syncwarp();
        tc_fence_after();
        for (int cc = half; cc < 16; cc += 2) {
          uint32_t t[16];
          tmem_ld16(lane_base + TM_O + (uint32_t)(cc * 16), t);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
          tmem_st16(lane_base + TM_O + (uint32_t)(cc * 16), t);
        }
        tmem_wait_st();
      }
      __syncwarp();
      tmem_st32(lane_base + (uint32_t)(cb / 2), pk[0]);
      tmem_st32(lane_base + (uint32_t)(cb / 2 + 32), pk[1]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok) {
      // Combine the two halves' row sums (exchange slot of parity n).
      xch[((n & 1) * 2 + half) * 128 + row] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xbar[q4]);
      if (!mbar_wait_warp(&xbar[q4], (uint32_t)(n & 1), ab)) ok = false;
      else l += xch[((n & 1) * 2 + (half ^ 1)) * 128 + row];
    }
    if (ok && mbar_wait_warp(o_done, (n - 1) & 1, ab)) {
      __syncwarp();
      tc_fence_after();
      const float inv = 1.0f / l;
      const int b = bh / args.h, hd = bh % args.h;
      uint16_t *orow = args.o + ((long long)b * args.N + query) * args.ldc + (long long)hd * args.d;
      for (int cc = half; cc < 16; cc += 2) {
        uint32_t t[16];
        tmem_ld16(lane_base + TM_O + (uint32_t)(cc * 16), t);
        tmem_wait_ld();
        if (query >= args.N) continue;
        const int e0 = oc * 256 + cc * 16;
        uint4 w0, w1;
        w0.x = pack_half2(__uint_as_float(t[0]) * inv, __uint_as_float(t[1]) * inv);
        w0.y = pack_half2(__uint_as_float(t[2]) * inv, __uint_as_float(t[3]) * inv);
        w0.z = pack_half2(__uint_as_float(t[4]) * inv, __uint_as_float(t[5]) * inv);
        w0.w = pack_half2(__uint_as_float(t[6]) * inv, __uint_as_float(t[7]) * inv);
        w1.x = pack_half2(__uint_as_float(t[8]) * inv, __uint_as_float(t[9]) * inv);
        w1.y = pack_half2(__uint_as_float(t[10]) * inv, __uint_as_float(t[11]) * inv);
        w1.z = pack_half2(__uint_as_float(t[12]) * inv, __uint_as_float(t[13]) * inv);
        w1.w = pack_half2(__uint_as_float(t[14]) * inv, __uint_as_float(t[15]) * inv);
        reinterpret_cast<uint4 *>(orow + e0)[0] = w0;
        reinterpret_cast<uint4 *>(orow + e0)[1] = w1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int launch_attention_wide(const Dims &dm, AttnArgs a, const uint16_t *q, const uint16_t *k, const uint16_t *vt,
                          cudaStream_t st) {
  int max_smem = MAX_SMEM_FALLBACK, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  int nst = (int)(((long long)max_smem - (long long)wide_smem(0)) / (WSLOT + 16));
  if (nst > 4) nst = 4;
  if (nst < 2) return 2;
  a.nst = nst;
  a.nqb = 8;
  CUtensorMap qmap, kmap, vmap;
  const uint64_t BH = (uint64_t)dm.B * dm.h;
  {
    const uint64_t dims[3] = {(uint64_t)dm.ldq, (uint64_t)dm.N, BH};
    const uint64_t strides[2] = {(uint64_t)dm.ldq * 2, (uint64_t)dm.N * dm.ldq * 2};
    const uint32_t qbox[3] = {64, BQ, 1};
    const uint32_t kbox[3] = {64, BKW, 1};
    if (encode_tiled(&qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, q, dims, strides, qbox,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
    if (encode_tiled(&kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, k, dims, strides, kbox,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
  }
  {
    const uint64_t dims[3] = {(uint64_t)dm.N, (uint64_t)dm.dp, BH};
    const uint64_t strides[2] = {(uint64_t)dm.ldn * 2, (uint64_t)dm.dp * dm.ldn * 2};
    const uint32_t box[3] = {64, 256, 1};
    if (encode_tiled(&vmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, vt, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
  }
  const uint32_t smem = wide_smem(nst);
  cudaFuncSetAttribute(attention_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const dim3 grid((dm.N + BQ - 1) / BQ * 2, (unsigned)BH, 1);
  attention_wide_kernel<<<grid, 320, smem, st>>>(qmap, kmap, vmap, a);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace

int launch_attention(const Dims &dm, const uint16_t *q, const uint16_t *k, const uint16_t *vt, uint16_t *o,
                     const KParams &kp, cudaStream_t st) {
  AttnArgs a{};
  a.N = dm.N; a.h = dm.h; a.d = dm.d; a.dp = dm.dp; a.ldc = dm.ldc; a.d_o = dm.d_o; a.n_oc = dm.n_oc;
  a.nqb = (dm.dp + 63) / 64;
  a.ntiles = (dm.N + BKV - 1) / BKV;
  if (dm.dp == 512 && dm.n_oc == 2) {
    a.sl2 = 1.4426950408889634f / sqrtf((float)dm.d);
    a.o = o;
    a.err = kp.err;
    a.timeout_ns = kp.timeout_ns;
    a.N = dm.N; a.h = dm.h; a.d = dm.d; a.ldc = dm.ldc;
    return launch_attention_wide(dm, a, q, k, vt, st);
  }
  int max_smem = MAX_SMEM_FALLBACK, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  // Two CTAs per SM (16 KB slots, 256 TMEM columns) when the O slice fits 128
  // columns and the ring still has >= 2 slots; P then lives in its own 64
  // TMEM columns when the O slice fits 64 (else in shared memory).  Otherwise
  // one CTA per SM, 32 KB slots, two S buffers, P over the S buffer it
  // replaces.
  const int p_tmem_single = dm.d_o <= 64 ? 1 : 0;
  int nst = (int)(((long long)SM_SMEM_PER_TWO - (long long)smem_bytes(a.nqb, 0, BLK, p_tmem_single)) / (BLK + 16));
  if (dm.d_o <= 128 && nst >= 2) {
    a.single = 1;
    a.tmem_cols = 256;
    a.p_tmem = p_tmem_single;
    a.p_col = 128;
    a.o_col = p_tmem_single ? 192 : 128;
    a.slot = BLK;
    if (nst > 4) nst = 4;
  } else {
    a.single = 0;
    a.tmem_cols = 512;
    a.p_tmem = 1;
    a.p_col = 0;
    a.o_col = 256;
    a.slot = 2 * BLK;
    nst = (int)(((long long)max_smem - (long long)smem_bytes(a.nqb, 0, a.slot, 1)) / (a.slot + 16));
    if (nst > 6) nst = 6;
  }
  a.kpb = a.slot / BLK;
  a.vrows = dm.d_o <= a.slot / 128 ? dm.d_o : a.slot / 128;
  a.nvr = (dm.d_o + a.vrows - 1) / a.vrows;
  if (nst < 2) return 2;
  a.nst = nst;
  a.sl2 = 1.4426950408889634f / sqrtf((float)dm.d);
  a.o = o;
  a.err = kp.err;
  a.timeout_ns = kp.timeout_ns;

  CUtensorMap qmap, kmap, vmap;
  const uint64_t BH = (uint64_t)dm.B * dm.h;
  {
    const uint64_t dims[3] = {(uint64_t)dm.ldq, (uint64_t)dm.N, BH};
    const uint64_t strides[2] = {(uint64_t)dm.ldq * 2, (uint64_t)dm.N * dm.ldq * 2};
    const uint32_t box[3] = {64, BQ, 1};
    if (encode_tiled(&qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, q, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
    if (encode_tiled(&kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, k, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
  }
  {
    const uint64_t dims[3] = {(uint64_t)dm.N, (uint64_t)dm.dp, BH};
    const uint64_t strides[2] = {(uint64_t)dm.ldn * 2, (uint64_t)dm.dp * dm.ldn * 2};
    const uint32_t box[3] = {64, (uint32_t)a.vrows, 1};
    if (encode_tiled(&vmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, vt, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
  }
  const uint32_t smem = smem_bytes(a.nqb, nst, a.slot, a.p_tmem);
  const dim3 grid((dm.N + BQ - 1) / BQ * dm.n_oc, (unsigned)BH, 1);
  if (a.single) {
    cudaFuncSetAttribute(attention_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attention_kernel<true><<<grid, THREADS, smem, st>>>(qmap, kmap, vmap, a);
  } else {
    cudaFuncSetAttribute(attention_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attention_kernel<false><<<grid, THREADS, smem, st>>>(qmap, kmap, vmap, a);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace ssa
