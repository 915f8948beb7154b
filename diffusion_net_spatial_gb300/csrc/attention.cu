// attention.cu -- O_j = softmax(Q_j K_j^T / sqrt(d)) V_j per (sample, head)
// (tensortonic "diffusion-l03-spatial-self-attention", block equation; the
// softmax runs over the key axis and the head outputs are concatenated along
// channels in head order; worked example 1 divides the scores by sqrt(2) for
// d = 2).
//
// Flash-style, the N x N score matrix never exists.  In the single and
// double modes one CTA owns 128 queries of one (sample, head) -- and one of
// the two output halves when the padded head dim exceeds 256 -- and walks the
// keys in tiles of 128 (the quad and pair modes are described at their
// kernels):
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
// Four modes:
//   quad    padded head dim <= 64 without the causal mask (the table only
//           when W % 32 == 0): 64-key tiles, P written over its scores, 128
//           tensor-memory columns per query tile, four query tiles per SM
//           (described at attention_quad_kernel).
//   single  S uses 128 tensor-memory columns; the MMA writes S_{j+1} as soon
//           as the softmax warps have read S_j.  With a small head dim this
//           fits 256 columns and ~113 KB of shared memory, so two CTAs share
//           an SM and their softmax warpgroups overlap.
//   double  S alternates between two 128-column buffers (512 columns in all,
//           one CTA per SM); used when O needs more than 128 columns.
//   pair    padded head dim 512: a two-CTA cluster splits scores+softmax and
//           P V between two SMs (described at attention_pair_kernel).
// Keys past N in the last tile are zero-filled by TMA and masked to -inf.
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace ssa {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int BLK = 16384;  // one [128 x 64] fp16 swizzled block
constexpr int THREADS = 192;   // double mode: producer, MMA, four softmax warps
constexpr int STHREADS = 320;  // single mode with variants: producer, MMA, eight softmax warps
constexpr int MAX_SMEM_FALLBACK = 232448;
constexpr int SM_SMEM_PER_TWO = 115712;  // per-CTA budget when two CTAs share an SM
// Lazy-rescale bounds (log2 of the largest P before O is rescaled).  Where
// the exponents are rounded to fp16 before the exponential (the fp16-pair
// paths of the padded head dims), 2^8 keeps them within 2^-9 absolute.  Where
// the exponentials are taken in fp32 and P is rounded once to fp16, whose
// relative precision does not depend on the magnitude, P may grow to 2^15
// (< 65504): a rescale rewrites all of O's columns before the next P V (512
// of them in the pair kernel, stalling its output CTA), so the higher bound
// keeps rescales to the first few key tiles of a row (vae16384 block 519.7 ->
// 446.5 us).
constexpr float RESCALE_LOG2 = 8.0f;
constexpr float RESCALE_LOG2_F32 = 15.0f;

struct AttnArgs {
  int N, h, d, dp, ldc, d_o, n_oc, nqb, kpb, nvr, vrows, slot, nst, ntiles, single, tmem_cols, o_col;
  int p_tmem, p_col;  // P in tensor memory (and its column in single mode) or in shared memory
  int vpack;          // both 64-key halves of a tile's V^T in one ring slot (single mode, d_o <= 64)
  int ones;           // single mode, d < dp: V^T row d is all ones, so O column d accumulates the row sums
  float sl2;  // log2(e) / sqrt(d)
  int causal;          // mask keys after the query token
  const float *rel;    // NULL, or packed relative-position table [h][tabn] (log2 units)
  int gh, gw, tabn;    // token grid H x W; tabn = (2H-1)(2W-1)
  int ldq;             // pair mode: row pitch of Q, K (elements)
  const uint16_t *q;   // pair mode: Q read directly into tensor memory
  int pair_split, pair_P;  // pair mode work split (see PairSplit)
  long long pair_U;
  float *part;         // pair mode scratch: contributors' parts of cut tiles
  uint32_t *cnt;       // pair mode scratch: per-tile contributor counts
  uint16_t *o;
  uint32_t *err;
  uint64_t timeout_ns;
  uint32_t stall;      // test hook (single/double modes): the producer stops after this many ring loads
};

// full[nst], empty[nst], q_full, s_full[2], s_free, p_full, o_done, drain, xbar[4]
__host__ __device__ inline int nbars(int nst) { return 2 * nst + 11; }
struct Layout {
  uint32_t q, p, ring, bars, xch;
};
__host__ __device__ inline Layout layout(int nqb, int nst, int slot, int p_tmem) {
  Layout L;
  L.q = 0;
  L.p = nqb * 16384;
  L.ring = L.p + (p_tmem ? 0 : 32768);
  L.bars = L.ring + nst * slot;
  L.xch = L.bars + nbars(nst) * 8 + 16;  // [2][2][128] f32 (single mode)
  return L;
}
__host__ __device__ inline uint32_t smem_bytes(int nqb, int nst, int slot, int p_tmem) {
  return layout(nqb, nst, slot, p_tmem).xch + 2048 + 1024;
}

// Attention variants on one thread's scores (HNDL attention operator page,
// Masking and Relative position bias paragraphs).  r holds NC chunks of 32 raw
// scores of query token `query` (row `lane` of a warp whose 32 queries are
// consecutive tokens) against keys k0 + 32c + i.
//  * causal: keys after the query become -inf (only chunks that reach past
//    the query are touched);
//  * relative-position table (packed per head, pre-scaled by log2 e): each
//    score becomes the base-2 logit s * log2(e)/sqrt(d) + table[dy, dx].
//    When W is a multiple of 32, a warp's queries share one grid row and each
//    32-key chunk lies in one grid row, so the 32 x 32 bias block is a
//    Toeplitz slice of one table row: the entry of lane l and key i is
//    p[-i] for a per-lane pointer p, one L1-resident load at a constant
//    offset per score (the rows of the next key tile are prefetched into L1
//    a tile ahead, rel_prefetch).  Other widths read the table per score with
//    full index arithmetic.
// Returns true when the scores were turned into base-2 logits.

// Pointer p of the chunk of keys kc .. kc+31 (one grid row) for this lane's
// query of the warp whose first query is qw (W % 32 == 0).
__device__ __forceinline__ const float *rel_row_ptr(const AttnArgs &args, const float *tab, int qw, int kc,
                                                    int lane) {
  const int gw = args.gw, row_len = 2 * gw - 1;
  const int rq = qw / gw, cq0 = qw - rq * gw;
  const int rk = kc / gw, ck0 = kc - rk * gw;
  return tab + (rq - rk + args.gh - 1) * row_len + (cq0 - ck0 + gw - 1) + lane;
}

// Brings the table entries of NC chunks of keys from k0 into L1 (W % 32 == 0).
template <int NC>
__device__ __forceinline__ void rel_prefetch(const AttnArgs &args, int head, int query, int k0, int lane) {
  const int qw = query - lane;
  if (args.rel == nullptr || qw >= args.N) return;
  const float *tab = args.rel + (long long)head * args.tabn;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int kc = k0 + 32 * c;
    if (kc >= args.N) continue;
    const float *p = rel_row_ptr(args, tab, qw, kc, lane);
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p - 31));
  }
}

template <int NC, bool GENERIC>
__device__ __forceinline__ bool apply_variants(uint32_t (&r)[NC][32], const AttnArgs &args, int head, int query,
                                               int k0, float sl2, int lane) {
  if (args.causal) {
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if (k0 + 32 * c + 31 > query) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (k0 + 32 * c + i > query) r[c][i] = __float_as_uint(-INFINITY);
      }
  }
  if (args.rel == nullptr) return false;
  const float *tab = args.rel + (long long)head * args.tabn;
  const int gw = args.gw, row_len = 2 * gw - 1;
  const int qw = query - lane;  // the warp's first query
  if (!GENERIC) {  // W % 32 == 0 (checked at launch)
    if (qw < args.N) {  // warp-uniform: N is a multiple of 32 here
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const int kc = k0 + 32 * c;
        if (kc >= args.N) {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[c][i] = __float_as_uint(-INFINITY);
          continue;
        }
        const float *p = rel_row_ptr(args, tab, qw, kc, lane);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[c][i] = __float_as_uint(fmaf(__uint_as_float(r[c][i]), sl2, __ldg(p - i)));
      }
    } else {
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) r[c][i] = __float_as_uint(__uint_as_float(r[c][i]) * sl2);
    }
    return true;
  }
  const bool qin = query < args.N;
  const int rq = qin ? query / gw : 0, cq = qin ? query - rq * gw : 0;
  int rk = k0 / gw, ck = k0 - (k0 / gw) * gw;
  const int base = (rq + args.gh - 1) * row_len + (cq + gw - 1);  // entry at rk = ck = 0
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int key = k0 + 32 * c + i;
      float u = __uint_as_float(r[c][i]) * sl2;
      if (qin && key < args.N) u += __ldg(tab + base - rk * row_len - ck);
      r[c][i] = __float_as_uint(u);
      if (++ck == gw) {
        ck = 0;
        ++rk;
      }
    }
  return true;
}

// VAR: 0 plain block; 1 causal mask and/or relative-position bias with W a
// multiple of 32 (or no table); 2 a table over another width (per-score
// table reads).  Separate instantiations keep the plain block's register
// budget.
template <bool SINGLE, int VAR>
__global__ void __launch_bounds__((SINGLE && VAR != 0) ? STHREADS : THREADS, SINGLE ? 2 : 1)
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
  uint64_t *xbar = drain + 1;  // [4] HALVES: row-maximum exchange of the two halves of a row
  constexpr bool HALVES = SINGLE && VAR != 0;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + nbars(nst));
  volatile uint32_t *abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Under the causal mask a query tile's work grows with its index: the grid
  // is (B*h, query tiles x O halves) and the tiles run in reverse order, so
  // the heaviest ones start first.
  const int nqt = (args.N + BQ - 1) / BQ;
  const int qt = args.causal ? nqt - 1 - (int)(blockIdx.y / args.n_oc) : (int)(blockIdx.x / args.n_oc);
  const int oc = args.causal ? (int)(blockIdx.y % args.n_oc) : (int)(blockIdx.x % args.n_oc);
  const int bh = args.causal ? (int)blockIdx.x : (int)blockIdx.y;
  const int q0 = qt * BQ;
  // Under the causal mask, key tiles past the tile's last query are skipped.
  const int n = args.causal ? min(args.ntiles, (min(q0 + BQ, args.N) - 1) / BKV + 1) : args.ntiles;
  constexpr bool single = SINGLE;
  // V slots per key tile: one when both 64-key halves share a slot (the two
  // boxes then land vrows * 128 bytes apart), else one per half and row group.
  const int nvb = args.vpack ? 1 : 2 * args.nvr;
  const int nks = (args.nqb + args.kpb - 1) / args.kpb;  // K slots per key tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(s_free, HALVES ? 8 : 4);
    mbar_init(p_full, HALVES ? 8 : 4);
    for (int i = 0; i < 4; ++i) mbar_init(&xbar[i], 2);
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
  pdl_trigger();
  pdl_wait();  // inputs of the previous kernel visible from here on
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
      auto acquire = [&]() -> bool {
        if (args.stall && (uint32_t)it >= args.stall) return false;  // test hook: consumers' waits expire
        return it < nst || mbar_wait(&empty[s], ph ^ 1u, ab);
      };
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
          if (args.vpack) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * args.vrows * 128));
            for (int vh = 0; vh < 2; ++vh)
              tma_load_3d(sm + L.ring + s * slot + vh * args.vrows * 128, &vmap, &full[s], j * BKV + 64 * vh,
                          oc * args.d_o, bh);
          } else {
            const int vh = vb / args.nvr, vr = vb - vh * args.nvr;
            mbar_arrive_expect_tx(&full[s], (uint32_t)(args.vrows * 128));
            tma_load_3d(sm + L.ring + s * slot, &vmap, &full[s], j * BKV + 64 * vh, oc * args.d_o + vr * args.vrows,
                        bh);
          }
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
      mbar_wait_drain(q_full, 0, drain_limit(ab));
      for (int i = (it > nst ? it - nst : 0); i < it; ++i)
        mbar_wait_drain(&full[i % nst], (i / nst) & 1, drain_limit(ab));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Descriptors are formed once; a K step (32 B) or a 1024-B block offset
    // inside the swizzled tiles is a small add to the start-address field.
    // The whole warp runs the loop and the elected lane 0 issues (a loop run
    // by one divergent lane cannot issue short MMAs back to back); commits
    // then track every MMA issued before them.
    {
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
          if (!mbar_wait_warp(&full[s], ph, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bd = rd + (uint64_t)(s * slot16);
          const int nblk = min(args.kpb, args.nqb - ksl * args.kpb);
          if (elect_one()) {
            for (int bl = 0; bl < nblk; ++bl) {
              const int kb = ksl * args.kpb + bl;
              const uint64_t a0 = qd + (uint64_t)(kb * 1024);
              const uint64_t b0 = bd + (uint64_t)(bl * 1024);
              const int kmax = min(4, ksteps - kb * 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                if (kk < kmax)
                  mma_f16_ss(d_s, a0 + (uint64_t)(kk * 2), b0 + (uint64_t)(kk * 2), idesc_s, (kb | kk) ? 1u : 0u);
            }
            mma_commit(&empty[s]);
          }
          __syncwarp();
          issued = true;
          advance();
        }
        if (ok) {
          if (elect_one()) mma_commit(&s_full[buf]);
          __syncwarp();
        }
      };
      auto issue_pv = [&](int j) {
        const uint32_t pcol = single ? (uint32_t)args.p_col : (uint32_t)((j & 1) * BKV);
        for (int vb = 0; vb < nvb && ok; ++vb) {
          if (!mbar_wait_warp(&full[s], ph, ab)) { ok = false; break; }
          tc_fence_after();
          if (elect_one()) {
            for (int hh = 0; hh < (args.vpack ? 2 : 1); ++hh) {
              const int vh = args.vpack ? hh : vb / args.nvr, vr = args.vpack ? 0 : vb - vh * args.nvr;
              const uint32_t d_o = tmem + TM_O + (uint32_t)(vr * args.vrows);
              const uint64_t b0 = rd + (uint64_t)(s * slot16) + (uint64_t)((hh * args.vrows * 128) >> 4);
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
            }
            mma_commit(&empty[s]);
          }
          __syncwarp();
          issued = true;
          advance();
        }
        if (ok) {
          if (elect_one()) mma_commit(o_done);
          __syncwarp();
        }
      };
      if (!mbar_wait_warp(q_full, 0, ab)) ok = false;
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; j < n && ok; ++j) {
        if (single) {
          if (j + 1 < n) {
            if (!mbar_wait_warp(s_free, j & 1, ab)) { ok = false; break; }
            tc_fence_after();
            issue_s(0);
          }
        } else if (j == 0 && n > 1) {
          issue_s(1);
        }
        if (!ok || !mbar_wait_warp(p_full, j & 1, ab)) { ok = false; break; }
        tc_fence_after();
        issue_pv(j);
        if (!single && j + 2 < n) issue_s(j & 1);
      }
      if (issued) {  // every issued MMA completes before tensor memory is freed
        if (elect_one()) mma_commit(drain);
        __syncwarp();
        mbar_wait_drain(drain, 0, drain_limit(ab));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // HALVES (single mode with a mask or a table): eight warps, warp (q4,
    // half) takes rows q4*32 .. +31 and keys half*64 .. +63 of each tile; the
    // two halves of a row exchange their maxima through shared memory and
    // add their row sums at the end -- twice the independent softmax work per
    // SM for the heavier per-score work of the variants.  Otherwise four
    // warps with whole rows (for the plain block the per-tile exchange cost
    // more than the extra warps gave: unet-l1 119 vs 111 us).
    constexpr int NC = HALVES ? 2 : 4;  // 32-key chunks per thread per tile
    const int q4 = warp & 3;
    const int half = HALVES ? ((warp - 2) >> 2) : 0;
    const int row = q4 * 32 + lane;
    const int query = q0 + row;
    const int kofs = half * (NC * 32);  // first key of this warp within a tile
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t p_tile = smem_u32(sm + L.p);
    float *xch = reinterpret_cast<float *>(sm + L.xch);  // [2 parity][2 half][128] (HALVES)
    const float sl2 = args.sl2;
    // With a mask or a bias the scores are first turned into base-2 logits
    // (apply_variants), so the scale below becomes 1.
    constexpr bool var = VAR != 0;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    if (VAR == 1) rel_prefetch<NC>(args, bh % args.h, query, kofs, lane);
    for (int j = 0; j < n; ++j) {
      const int buf = single ? 0 : (j & 1);
      const uint32_t par = single ? (uint32_t)(j & 1) : (uint32_t)((j >> 1) & 1);
      if (!mbar_wait_warp(&s_full[buf], par, ab)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[NC][32];
#pragma unroll
      for (int c = 0; c < NC; ++c) tmem_ld32(lane_base + (uint32_t)(buf * BKV + kofs + 32 * c), r[c]);
      tmem_wait_ld();
      if (single) {
        // S has been read into registers: the MMA may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
      }
      const int kvalid = min(BKV, args.N - j * BKV) - kofs;
      if (kvalid < NC * 32) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i >= kvalid) r[c][i] = __float_as_uint(-INFINITY);
      }
      float sc = sl2;  // base-2 logits when the table was added
      if (var && apply_variants<NC, VAR == 2>(r, args, bh % args.h, query, j * BKV + kofs, sl2, lane)) sc = 1.f;
      if (VAR == 1 && j + 1 < n) rel_prefetch<NC>(args, bh % args.h, query, (j + 1) * BKV + kofs, lane);
      // Row maximum: 2*NC independent 3-input max chains.
      float pm[2 * NC];
#pragma unroll
      for (int t = 0; t < 2 * NC; ++t) {
        const int c = t >> 1, o = (t & 1) * 16;
        float m = __uint_as_float(r[c][o]);
#pragma unroll
        for (int i = 1; i < 15; i += 2) m = max3f(m, __uint_as_float(r[c][o + i]), __uint_as_float(r[c][o + i + 1]));
        pm[t] = fmaxf(m, __uint_as_float(r[c][o + 15]));
      }
      float mx = fmaxf(max3f(pm[0], pm[1], pm[2]), pm[3]);
      if (NC == 4) mx = max3f(mx, max3f(pm[NC], pm[NC + 1], pm[NC + 2]), pm[2 * NC - 1]);
      if (HALVES) {
        // The other half of this row (same lanes, other warp).
        xch[((j & 1) * 2 + half) * 128 + row] = mx;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xbar[q4]);
        if (!mbar_wait_warp(&xbar[q4], (uint32_t)(j & 1), ab)) { ok = false; break; }
        mx = fmaxf(mx, xch[((j & 1) * 2 + (half ^ 1)) * 128 + row]);
      }
      const float m_new = fmaxf(m_used, mx * sc);
      // Lazy rescale: a row raises its reference maximum only when the new
      // maximum exceeds it by more than the bound (RESCALE_LOG2 on the
      // fp16-pair exponent path, RESCALE_LOG2_F32 otherwise).  The decision is made
      // per warp (any row that needs it), because the tensor-memory accesses
      // that rescale O are warp-collective; rows that did not need it use
      // their own (possibly unit) factor.  Both halves of a row see the same
      // maxima, so they decide alike.
      const bool need = (j > 0) && (m_new > m_used + (args.ones ? RESCALE_LOG2 : RESCALE_LOG2_F32));
      const bool rescale = __any_sync(0xFFFFFFFFu, need) != 0;
      float alpha = 1.f;
      if (j == 0) {
        m_used = m_new;
      } else if (rescale && m_new > m_used) {
        alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
      }
      // p = 2^(s * log2(e)/sqrt(d) - m): one paired FMA per two scores.
      const uint64_t c2 = f2_pack(sc, sc);
      const uint64_t nm2 = f2_pack(-m_used, -m_used);
      uint32_t pk[NC / 2][32];
      if (args.ones) {
        // The row sums come from V's column of ones (the P V MMA adds up
        // exactly the fp16 P it multiplies), so here only P is formed: the
        // pair of exponents rounded to fp16 once and exponentiated together
        // (one MUFU operation for two scores, already packed for the MMA).
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), c2, nm2), t0, t1);
            pk[c >> 1][(c & 1) * 16 + (i >> 1)] = exp2_pair_op(t0, t1);
          }
      } else {
        // the row sum in four paired accumulators
        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), c2, nm2), t0, t1);
            const float e0 = ex2_approx(t0);
            const float e1 = ex2_approx(t1);
            acc2[(i >> 3) & 3] = f2_add(acc2[(i >> 3) & 3], f2_pack(e0, e1));
            pk[c >> 1][(c & 1) * 16 + (i >> 1)] = pack_op2(e0, e1);
          }
        float s0, s1, s2, s3;
        f2_unpack(f2_add(acc2[0], acc2[1]), s0, s1);
        f2_unpack(f2_add(acc2[2], acc2[3]), s2, s3);
        const float sum = (s0 + s1) + (s2 + s3);
        l = l * alpha + sum;
      }
      if (j > 0 && !mbar_wait_warp(o_done, (j - 1) & 1, ab)) { ok = false; break; }
      if (rescale) {
        __syncwarp();
        tc_fence_after();
        for (int cc = half; cc < args.d_o / 16; cc += (HALVES ? 2 : 1)) {
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
        // (double) or in its own 64 columns (single; with halves, this half's 32).
        const uint32_t pcol = single ? (uint32_t)args.p_col + (uint32_t)(half * 32) : (uint32_t)(buf * BKV);
        __syncwarp();
#pragma unroll
        for (int c2i = 0; c2i < NC / 2; ++c2i) tmem_st32(lane_base + pcol + (uint32_t)(32 * c2i), pk[c2i]);
        tmem_wait_st();
      } else {
        // P as a [128 x 128] fp16 tile of two 64-key swizzled blocks; this
        // warp's keys are block `half` (single) or both blocks (double).
#pragma unroll
        for (int c = 0; c < 4 * NC; ++c)
          st_shared_v4(p_tile + (half + (c >> 3)) * 16384 + sw128_offset((uint32_t)row, (uint32_t)(c & 7)),
                       pk[c >> 3][(4 * c) & 31], pk[c >> 3][(4 * c + 1) & 31], pk[c >> 3][(4 * c + 2) & 31],
                       pk[c >> 3][(4 * c + 3) & 31]);
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ------------------------------------------------------------ epilogue
    bool eok = ok && mbar_wait_warp(o_done, (n - 1) & 1, ab);
    if (HALVES && eok && !args.ones) {
      // Row sum of the two halves (exchange slot of parity n).
      xch[((n & 1) * 2 + half) * 128 + row] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xbar[q4]);
      eok = mbar_wait_warp(&xbar[q4], (uint32_t)(n & 1), ab);
      if (eok) l += xch[((n & 1) * 2 + (half ^ 1)) * 128 + row];
    }
    if (eok) {
      __syncwarp();
      tc_fence_after();
      if (args.ones) {
        l = __uint_as_float(tmem_ld1(lane_base + TM_O + (uint32_t)args.d));  // O column d = sum of P
        tmem_wait_ld();
      }
      const float inv = 1.0f / l;
      const int b = bh / args.h, hd = bh % args.h;
      const bool vec = (args.d % 8) == 0;
      uint16_t *orow = args.o + ((long long)b * args.N + query) * args.ldc + (long long)hd * args.d;
      for (int cc = half; cc < args.d_o / 16; cc += (HALVES ? 2 : 1)) {
        uint32_t t[16];
        tmem_ld16(lane_base + TM_O + (uint32_t)(cc * 16), t);
        tmem_wait_ld();
        if (query >= args.N) continue;
        const int e0 = oc * args.d_o + cc * 16;
        if (vec && e0 + 16 <= args.d) {
          uint4 w0, w1;
          w0.x = pack_op2(__uint_as_float(t[0]) * inv, __uint_as_float(t[1]) * inv);
          w0.y = pack_op2(__uint_as_float(t[2]) * inv, __uint_as_float(t[3]) * inv);
          w0.z = pack_op2(__uint_as_float(t[4]) * inv, __uint_as_float(t[5]) * inv);
          w0.w = pack_op2(__uint_as_float(t[6]) * inv, __uint_as_float(t[7]) * inv);
          w1.x = pack_op2(__uint_as_float(t[8]) * inv, __uint_as_float(t[9]) * inv);
          w1.y = pack_op2(__uint_as_float(t[10]) * inv, __uint_as_float(t[11]) * inv);
          w1.z = pack_op2(__uint_as_float(t[12]) * inv, __uint_as_float(t[13]) * inv);
          w1.w = pack_op2(__uint_as_float(t[14]) * inv, __uint_as_float(t[15]) * inv);
          reinterpret_cast<uint4 *>(orow + e0)[0] = w0;
          reinterpret_cast<uint4 *>(orow + e0)[1] = w1;
        } else {
          for (int i = 0; i < 16; ++i) {
            if (e0 + i < args.d) {
              orow[e0 + i] = op_bits(__uint_as_float(t[i]) * inv);
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
// Quad mode (padded head dim <= 64, the block without a mask or table): four
// query tiles in flight per SM.  The single mode's 128-key tiles need 256
// tensor-memory columns per query tile (S, P, O), so an SM holds two query
// tiles: each tile's chain of softmax steps sets the pace, and on unet-l1 the
// 512 query tiles leave a partial second wave on 304 CTA slots.  Here a key
// tile is 64 keys and P is written over the scores it came from, so a query
// tile needs 128 columns; a CTA holds QT query tiles (of the same sample and
// head) that share one K/V ring:
//   tensor memory (128 per query tile t): S_j at 128t + 0..63 (fp32), then
//                P_j at 128t + 0..31 (fp16 pairs), O at 128t + 64..64+dp
//   shared memory: QT Q tiles [128 x 64] and QNST ring slots, each the K box
//                [64 keys x 64 dims] and the V^T box [dp x 64 keys]
//   warp 0   TMA producer;  warp 1 MMA: for each query tile t in turn,
//            once its softmax has written P_tj, O_t += P_tj V_j (P from
//            tensor memory), and once that has completed (same columns)
//            S_t(j+1) = Q_t K_(j+1)^T
//   warps 2.. softmax, four per query tile, one query row per thread: the
//            tile's 64 scores in one tensor-memory round trip (the longest
//            stall of the loop), the row maximum, then P per 32 keys stored
//            over scores already read
// With QT = 2 and two CTAs per SM the 152 SMs hold 608 query tiles at once
// (one wave for unet-l1), sixteen softmax warps per SM, and each K/V tile is
// loaded once for two query tiles.
constexpr int QK = 64;                           // keys per tile
constexpr int QNST = 3;                          // ring slots
constexpr int QSLOT = 16384;                     // K (8 KB) + V^T (<= 8 KB)
constexpr uint32_t Q_TM_O = 64;                  // O inside a query tile's 128 columns
template <int QT> struct QuadCfg {
  static constexpr int THREADS = 64 + 128 * QT;
  static constexpr int NBARS = 2 * QNST + 3 * QT + 2;  // full, empty, q_full, s_full[QT], p_full[QT], o_done[QT], drain
  static constexpr uint32_t OFF_RING = 16384u * QT;
  static constexpr uint32_t OFF_BARS = OFF_RING + QNST * QSLOT;
  static constexpr uint32_t SMEM = OFF_BARS + NBARS * 8 + 16;
  static constexpr uint32_t TMEM_COLS = 128u * QT;
};

// Relative-position table of the quad mode (W a multiple of 32): a warp's 32
// queries lie in one grid row and each 32-key chunk in one grid row, so the
// chunk's 32 x 32 bias block is a Toeplitz slice of one table row, read as
// p[-i] from one per-lane pointer p (one L1 load per score, coalesced).  The
// warp's grid position is fixed and the key tile's is advanced by additions,
// so no division runs per key tile.  Scores become base-2 logits
// s * log2(e)/sqrt(d) + table, two per paired FMA.
struct QuadTable {
  const float *row0;  // this head's packed table
  int row_len, gw, gh, rq_off;  // 2W - 1, W, H, (query grid row) + H - 1
  int cq_off;               // (first query's grid column) + W - 1
  int rk, ck;               // grid row and column of the current key tile's first key
  bool valid;               // the warp's queries exist
};

__device__ __forceinline__ void quad_table_init(QuadTable &t, const AttnArgs &args, int head, int qw) {
  t.row_len = 2 * args.gw - 1;
  t.gw = args.gw;
  t.gh = args.gh;
  t.valid = qw < args.N;
  const int rq = t.valid ? qw / args.gw : 0;
  t.rq_off = rq + args.gh - 1;
  t.cq_off = (t.valid ? qw - rq * args.gw : 0) + args.gw - 1;
  t.row0 = args.rel + (long long)head * args.tabn;
  t.rk = 0;
  t.ck = 0;
}

// Pointer p of the chunk whose first key is at grid (rk, ck).
__device__ __forceinline__ const float *quad_table_ptr(const QuadTable &t, int rk, int ck, int lane) {
  return t.row0 + (t.rq_off - rk) * t.row_len + (t.cq_off - ck) + lane;
}

// Logits of the key tile at (t.rk, t.ck), 64 keys; keys past N are already
// -inf and stay so.  Then t advances to the next key tile, whose table rows
// are prefetched into L1.
__device__ __forceinline__ void quad_table_apply(QuadTable &t, uint32_t (&r)[2][32], float sl2, int kvalid,
                                                 int lane) {
  const uint64_t c2 = f2_pack(sl2, sl2);
  int rk = t.rk, ck = t.ck;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (t.valid && 32 * c < kvalid) {
      const float *p = quad_table_ptr(t, rk, ck, lane);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float a0, a1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), c2,
                         f2_pack(__ldg(p - i), __ldg(p - i - 1))),
                  a0, a1);
        r[c][i] = __float_as_uint(a0);
        r[c][i + 1] = __float_as_uint(a1);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[c][i] = __float_as_uint(__uint_as_float(r[c][i]) * sl2);
    }
    ck += 32;
    if (ck == t.gw) {
      ck = 0;
      ++rk;
    }
  }
  t.rk = rk;
  t.ck = ck;
  if (t.valid) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const bool wrap = ck + 32 * c >= t.gw;
      if (rk + (wrap ? 1 : 0) >= t.gh) continue;  // past the last key row
      const float *p = quad_table_ptr(t, rk + (wrap ? 1 : 0), wrap ? ck + 32 * c - t.gw : ck + 32 * c, lane);
      asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
      asm volatile("prefetch.global.L1 [%0];" ::"l"(p - 31));
    }
  }
}

// VAR 1: the relative-position table over a width that is a multiple of 32
// (the Toeplitz path of apply_variants); its scores become base-2 logits.
template <int QT, int VAR>
__global__ void __launch_bounds__(QuadCfg<QT>::THREADS, 2)
    attention_quad_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const AttnArgs args) {
  using Cfg = QuadCfg<QT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw;
  // 128B-swizzled operands need a 1024-byte aligned base; the layout leaves
  // no room to realign, so refuse to run otherwise.
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicOr(args.err, (uint32_t)DEV_MISALIGNED);
    return;
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Cfg::OFF_BARS);
  uint64_t *full = bars;
  uint64_t *empty = bars + QNST;
  uint64_t *q_full = bars + 2 * QNST;
  uint64_t *s_full = q_full + 1;   // [QT]
  uint64_t *p_full = s_full + QT;  // [QT]
  uint64_t *o_done = p_full + QT;  // [QT]
  uint64_t *drain = o_done + QT;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::NBARS);
  volatile uint32_t *abort_flag = tmem_slot + 1;
  uint8_t *ring = sm + Cfg::OFF_RING;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * BQ * QT;
  const int bh = blockIdx.y;
  const int n = (args.N + QK - 1) / QK;  // key tiles
  const uint32_t vbytes = (uint32_t)args.dp * 128u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < QNST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(q_full, 1);
    for (int t = 0; t < QT; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0u;
    fence_barrier_init();
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
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
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 16384u * QT);
      for (int t = 0; t < QT; ++t) tma_load_3d(sm + t * 16384, &qmap, q_full, 0, q0 + t * BQ, bh);
      int it = 0;
      for (int j = 0; j < n; ++j) {
        const int s = j % QNST;
        if (args.stall && (uint32_t)it >= args.stall) break;  // test hook: consumers' waits expire
        if (j >= QNST && !mbar_wait(&empty[s], (uint32_t)(((j / QNST) - 1) & 1), ab)) break;
        mbar_arrive_expect_tx(&full[s], 8192u + vbytes);
        tma_load_3d(ring + s * QSLOT, &kmap, &full[s], 0, j * QK, bh);
        tma_load_3d(ring + s * QSLOT + 8192, &vmap, &full[s], j * QK, 0, bh);
        ++it;
      }
      // Never leave with a copy in flight.
      mbar_wait_drain(q_full, 0, drain_limit(ab));
      for (int i = (it > QNST ? it - QNST : 0); i < it; ++i)
        mbar_wait_drain(&full[i % QNST], (uint32_t)((i / QNST) & 1), drain_limit(ab));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA warp
    const uint32_t idesc_s = idesc_f16(BQ, QK);
    const uint32_t idesc_o = idesc_f16(BQ, (uint32_t)args.dp);
    const uint64_t qd = sdesc_k128(smem_u32(sm));
    const uint64_t rd = sdesc_k128(smem_u32(ring));
    const int ksteps = args.dp / 16;
    // Each query tile runs its own chain P_tj -> O_t += P_tj V_j -> S_t(j+1);
    // the tiles are served in turn, so one tile's softmax overlaps the other's
    // MMAs.  S_t(j+1) overwrites the columns P_tj V_j reads: it is issued only
    // once that P V has completed.
    auto issue_s = [&](int t, int j) {
      const uint64_t kd = rd + (uint64_t)(((j % QNST) * QSLOT) >> 4);
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          if (kk < ksteps)
            mma_f16_ss(tmem + (uint32_t)(t * 128), qd + (uint64_t)(t * 1024 + kk * 2), kd + (uint64_t)(kk * 2),
                       idesc_s, kk ? 1u : 0u);
        mma_commit(&s_full[t]);
      }
      __syncwarp();
    };
    bool ok = mbar_wait_warp(q_full, 0, ab) && mbar_wait_warp(&full[0], 0, ab), issued = false;
    if (ok) {
      for (int t = 0; t < QT; ++t) issue_s(t, 0);
      issued = true;
    }
    for (int j = 0; j < n && ok; ++j) {
      const int s = j % QNST;
      const uint64_t vd = rd + (uint64_t)((s * QSLOT + 8192) >> 4);
      bool next_full = false;
      for (int t = 0; t < QT; ++t) {
        if (!mbar_wait_warp(&p_full[t], (uint32_t)(j & 1), ab)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 16 keys (8 columns of P) per step
            mma_f16_ts(tmem + (uint32_t)(t * 128) + Q_TM_O, tmem + (uint32_t)(t * 128 + kk * 8),
                       vd + (uint64_t)(kk * 2), idesc_o, (j | kk) ? 1u : 0u);
          mma_commit(&o_done[t]);
        }
        __syncwarp();
        if (j + 1 < n) {
          if (!next_full) {
            if (!mbar_wait_warp(&full[(j + 1) % QNST], (uint32_t)(((j + 1) / QNST) & 1), ab)) { ok = false; break; }
            next_full = true;
          }
          if (!mbar_wait_warp(&o_done[t], (uint32_t)(j & 1), ab)) { ok = false; break; }
          issue_s(t, j + 1);
        }
      }
      if (ok) {  // slot s is free once this tile's MMAs complete
        if (elect_one()) mma_commit(&empty[s]);
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
    // ------------------------------------------------------------ softmax
    const int qt = (warp - 2) >> 2;  // this warp's query tile
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const int query = q0 + qt * BQ + row;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(qt * 128);
    const float sl2 = args.sl2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    QuadTable tab;
    if constexpr (VAR != 0) quad_table_init(tab, args, bh % args.h, query - lane);
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait_warp(&s_full[qt], (uint32_t)(j & 1), ab)) { ok = false; break; }
      tc_fence_after();
      const int kvalid = min(QK, args.N - j * QK);
      // The tile's 64 scores in one round trip (both loads, one wait): the
      // wait for tensor memory is the longest stall of this loop.
      uint32_t r[2][32];
      tmem_ld32(lane_base, r[0]);
      tmem_ld32(lane_base + 32u, r[1]);
      tmem_wait_ld();
      if (kvalid < QK) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i >= kvalid) r[c][i] = __float_as_uint(-INFINITY);
      }
      if constexpr (VAR != 0) quad_table_apply(tab, r, sl2, kvalid, lane);
      float alpha = 1.f, sum = 0.f;
      bool done = false;
#ifndef SSA_OPERAND_BF16
      if (VAR == 0 && j > 0 && args.ones) {
        // The exponents with the running maximum, as the fp16 pairs that
        // ex2.approx.f16x2 takes (packed in place over consumed scores); their
        // maximum by packed fp16 maxima decides the lazy rescale, so the fp32
        // row maximum is only taken on the rare tiles that need one.
        const uint64_t c2 = f2_pack(sl2, sl2);
        const uint64_t nm2 = f2_pack(-m_used, -m_used);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), c2, nm2), t0, t1);
            r[c][i >> 1] = pack_op2(t0, t1);
          }
        uint32_t h[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) h[k] = hmax2(r[k >> 3][2 * (k & 7)], r[k >> 3][2 * (k & 7) + 1]);
#pragma unroll
        for (int w = 8; w > 0; w >>= 1)
#pragma unroll
          for (int k = 0; k < w; ++k) h[k] = hmax2(h[k], h[k + w]);
        if (!__any_sync(0xFFFFFFFFu, h2_hmax(h[0]) > RESCALE_LOG2)) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int k = 0; k < 16; ++k) r[c][k] = ex2_h2(r[c][k]);
            tmem_st16_lo(lane_base + (uint32_t)(16 * c), r[c]);
          }
          done = true;
        } else {
          // Rescale: the scores again from tensor memory (P has not been written).
          tmem_ld32(lane_base, r[0]);
          tmem_ld32(lane_base + 32u, r[1]);
          tmem_wait_ld();
          if (kvalid < QK) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (32 * c + i >= kvalid) r[c][i] = __float_as_uint(-INFINITY);
          }
        }
      }
#endif
      if (!done) {
        float pm[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int c = t >> 1, o = (t & 1) * 16;
          float m = __uint_as_float(r[c][o]);
#pragma unroll
          for (int i = 1; i < 15; i += 2) m = max3f(m, __uint_as_float(r[c][o + i]), __uint_as_float(r[c][o + i + 1]));
          pm[t] = fmaxf(m, __uint_as_float(r[c][o + 15]));
        }
        const float mx = fmaxf(max3f(pm[0], pm[1], pm[2]), pm[3]);
        const float m_new = fmaxf(m_used, VAR != 0 ? mx : mx * sl2);
        // Lazy rescale, decided per warp (as in the single mode).
        const bool need = (j > 0) && (m_new > m_used + RESCALE_LOG2);
        const bool rescale = __any_sync(0xFFFFFFFFu, need) != 0;
        if (j == 0) {
          m_used = m_new;
        } else if (rescale && m_new > m_used) {
          alpha = ex2_approx(m_used - m_new);
          m_used = m_new;
        }
        if (rescale) {
          // O is idle: the P V of the previous tile completed before S_j was issued.
          for (int cc = 0; cc < args.dp / 16; ++cc) {
            uint32_t t[16];
            tmem_ld16(lane_base + Q_TM_O + (uint32_t)(cc * 16), t);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
            tmem_st16(lane_base + Q_TM_O + (uint32_t)(cc * 16), t);
          }
        }
        // P per 32 keys into columns 16c.. (scores already in registers).
        const float cs = VAR != 0 ? 1.f : sl2;  // logits already scaled
        const uint64_t c2 = f2_pack(cs, cs);
        const uint64_t nm2 = f2_pack(-m_used, -m_used);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
          if (args.ones) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float t0, t1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), c2, nm2), t0, t1);
              pk[i >> 1] = exp2_pair_op(t0, t1);
            }
          } else {
            uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float t0, t1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), c2, nm2), t0, t1);
              const float e0 = ex2_approx(t0);
              const float e1 = ex2_approx(t1);
              acc2[(i >> 1) & 1] = f2_add(acc2[(i >> 1) & 1], f2_pack(e0, e1));
              pk[i >> 1] = pack_op2(e0, e1);
            }
            float s0, s1;
            f2_unpack(f2_add(acc2[0], acc2[1]), s0, s1);
            sum += s0 + s1;
          }
          tmem_st16(lane_base + (uint32_t)(16 * c), pk);
        }
      }
      l = l * alpha + sum;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[qt]);
    }
    // ------------------------------------------------------------ epilogue
    const bool eok = ok && mbar_wait_warp(&o_done[qt], (uint32_t)((n - 1) & 1), ab);
    if (eok) {
      __syncwarp();
      tc_fence_after();
      if (args.ones) {
        l = __uint_as_float(tmem_ld1(lane_base + Q_TM_O + (uint32_t)args.d));  // O column d = sum of P
        tmem_wait_ld();
      }
      const float inv = 1.0f / l;
      const int b = bh / args.h, hd = bh % args.h;
      const bool vec = (args.d % 8) == 0;
      uint16_t *orow = args.o + ((long long)b * args.N + query) * args.ldc + (long long)hd * args.d;
      for (int cc = 0; cc < args.dp / 16; ++cc) {
        uint32_t t[16];
        tmem_ld16(lane_base + Q_TM_O + (uint32_t)(cc * 16), t);
        tmem_wait_ld();
        if (query >= args.N) continue;
        const int e0 = cc * 16;
        if (vec && e0 + 16 <= args.d) {
          uint4 w0, w1;
          w0.x = pack_op2(__uint_as_float(t[0]) * inv, __uint_as_float(t[1]) * inv);
          w0.y = pack_op2(__uint_as_float(t[2]) * inv, __uint_as_float(t[3]) * inv);
          w0.z = pack_op2(__uint_as_float(t[4]) * inv, __uint_as_float(t[5]) * inv);
          w0.w = pack_op2(__uint_as_float(t[6]) * inv, __uint_as_float(t[7]) * inv);
          w1.x = pack_op2(__uint_as_float(t[8]) * inv, __uint_as_float(t[9]) * inv);
          w1.y = pack_op2(__uint_as_float(t[10]) * inv, __uint_as_float(t[11]) * inv);
          w1.z = pack_op2(__uint_as_float(t[12]) * inv, __uint_as_float(t[13]) * inv);
          w1.w = pack_op2(__uint_as_float(t[14]) * inv, __uint_as_float(t[15]) * inv);
          reinterpret_cast<uint4 *>(orow + e0)[0] = w0;
          reinterpret_cast<uint4 *>(orow + e0)[1] = w1;
        } else {
          for (int i = 0; i < 16; ++i)
            if (e0 + i < args.d) orow[e0 + i] = op_bits(__uint_as_float(t[i]) * inv);
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Pair mode (padded head dim 512).  O for 128 queries fills all 512 tensor-
// memory columns, so one CTA cannot hold O and the scores at once.  A cluster
// of two CTAs on two SMs shares one query tile at a time and splits the work
// by role, so the scores are computed once:
//   rank 0 (score CTA)   Q (128 x 512, fp16) in tensor-memory columns
//                        256..511; S_j = Q K_j^T for 128 keys (A operand from
//                        tensor memory, N = 128) into one of two 128-column
//                        score buffers, so S_{j+1} runs while the softmax
//                        reads S_j.  Eight softmax warps (warp (q4, half): 32
//                        rows x 64 keys) round P_j to fp16 into a local
//                        swizzled staging tile; each warp then pushes its 4 KB
//                        to the output CTA with one bulk shared-to-shared
//                        copy, and the per-row rescale factors follow by
//                        st.async -- all completing one barrier there.
//   rank 1 (output CTA)  O (128 x 512 fp32) in all 512 columns; O += P_j V_j
//                        as two groups of N = 256 MMAs (P from shared memory,
//                        three buffers; V^T through a ring); four warps apply
//                        the rare rescales to O before P_j V_j; eight warps
//                        write the tile's result.
// Two producer warps per CTA issue the TMA loads (alternate ring slots): one
// issuing thread cannot keep a ring of 32 KB boxes busy on this GPU.  The
// completion of each P_j V_j is signalled to both CTAs at once (a multicast
// commit), which hands the P buffer back to the score CTA.
//
// Work split.  The (sample x head, 128-query) tiles are laid end to end as
// runs of key tiles -- one unit per key tile -- and the whole line is cut
// into P equal pieces, one per cluster, P being the number of clusters that
// fit on the GPU at once.  Every SM pair then has the same work and no
// partial second wave leaves most of the GPU idle.  A cluster walks its
// piece as segments (a query tile and a range of its key tiles).  A query
// tile cut between clusters is finished by whichever contributor ends last:
// each writes its unnormalised O with its row maxima and row sums to scratch
// and counts itself in with an atomic; the last one rescales every part to
// the common maximum, adds them to its own and writes O / l.  Nobody waits
// for another cluster.  Without scratch (and, under the causal mask, when
// there are at least as many tiles as clusters) each cluster takes one whole
// tile, the heaviest first.
constexpr int PK = 128;          // keys per tile
constexpr int PSLOT = 32768;     // ring slot: 32 KB of swizzled K or V^T blocks
constexpr int PNPB = 3;          // P buffers in the output CTA
constexpr int PNST_S = 5;        // ring slots, score CTA (after two 32 KB staging tiles)
constexpr int PNST_O = 4;        // ring slots, output CTA (after the P buffers)
constexpr int PNST_MAX = 5;
constexpr int PTHREADS = 352;    // warps: 0, 10 producers; 1 MMA; 2-9 softmax / rescale + epilogue
constexpr uint32_t P_RING_S = 2 * 32768;
constexpr uint32_t P_RING_O = PNPB * 32768;
constexpr uint32_t P_SMALL = P_RING_S + PNST_S * PSLOT;  // xch (rank 0) | alpha, flags, l, m (rank 1)
static_assert(P_RING_O + PNST_O * PSLOT <= P_SMALL, "output CTA layout");
constexpr uint32_t P_ALPHA = P_SMALL;                // [PNPB][128] f32
constexpr uint32_t P_FLAGS = P_SMALL + PNPB * 512;   // [PNPB][4 quarters] u32
constexpr uint32_t P_LSUM = P_FLAGS + PNPB * 16;     // [128] f32 row sums of the segment
constexpr uint32_t P_MROW = P_LSUM + 512;            // [128] f32 row maxima (base-2 logits)
constexpr uint32_t P_BARS = P_SMALL + 2624;
static_assert(P_MROW + 512 <= P_BARS && 2048 <= P_BARS - P_SMALL, "small area");
enum {
  PB_FULL = 0, PB_EMPTY = PB_FULL + PNST_MAX, PB_QREADY = PB_EMPTY + PNST_MAX, PB_SFULL = PB_QREADY + 1,
  PB_SFREE = PB_SFULL + 2, PB_STGFREE = PB_SFREE + 2, PB_XBAR = PB_STGFREE + 2, PB_PFULL = PB_XBAR + 4,
  PB_OREADY = PB_PFULL + PNPB, PB_PVDONE = PB_OREADY + PNPB, PB_LFULL = PB_PVDONE + PNPB, PB_LFREE = PB_LFULL + 1,
  PB_OFINAL = PB_LFREE + 1, PB_OFREE = PB_OFINAL + 1, PB_DRAIN = PB_OFREE + 1, PB_COUNT = PB_DRAIN + 1
};
constexpr uint32_t P_SMEM = P_BARS + PB_COUNT * 8 + 16;
constexpr uint32_t PMSG_BYTES = 32768 + 512 + 16;  // P tile + alpha + flags per key tile
constexpr uint32_t PLM_BYTES = 1024;               // l and m of a segment
// Scratch part of one contributor: O as [32 chunks][128 rows][16 columns]
// fp32, then the row maxima and row sums.
constexpr int PART_O_FLOATS = 128 * 512;
constexpr int PART_FLOATS = PART_O_FLOATS + 256;
constexpr int PAIR_MAX_CLUSTERS = 76;  // one per SM pair of a 152-SM GPU

// The work line of the pair kernel (see above).  Tiles t = 0 .. T-1: sample x
// head t / nqt; under the causal mask the query tiles of a head run from the
// last (heaviest) to the first, and tile i of a head has nqt - i key tiles.
struct PairSplit {
  int nqt;     // query tiles per head (= key tiles of an unmasked query tile)
  int causal;
  int split;   // 1: P equal pieces of the line; 0: cluster c takes tile c
  int P;       // clusters
  long long U; // units (key tiles) in all
  __device__ __forceinline__ int n_of(int t) const { return causal ? nqt - t % nqt : nqt; }
  __device__ __forceinline__ long long cum_of(int t) const {
    const long long bh = t / nqt, i = t % nqt;
    return causal ? bh * ((long long)nqt * (nqt + 1) / 2) + i * nqt - i * (i - 1) / 2 : (long long)t * nqt;
  }
  __device__ __forceinline__ long long ubeg(int c) const { return split ? (long long)c * U / P : cum_of(c); }
  // The cluster whose piece holds unit u (split mode).
  __device__ __forceinline__ int owner(long long u) const { return (int)(((u + 1) * P - 1) / U); }
  __device__ int tile_of(long long u) const {
    if (!causal) return (int)(u / nqt);
    const long long ub = (long long)nqt * (nqt + 1) / 2;
    const int bh = (int)(u / ub);
    const long long r = u - bh * ub;
    // largest i with i*nqt - i(i-1)/2 <= r
    const double b = 2.0 * nqt + 1.0;
    int i = (int)((b - sqrt(fmax(b * b - 8.0 * (double)r, 0.0))) * 0.5);
    i = max(0, min(i, nqt - 1));
    while (i + 1 < nqt && (long long)(i + 1) * nqt - (long long)(i + 1) * i / 2 <= r) ++i;
    while (i > 0 && (long long)i * nqt - (long long)i * (i - 1) / 2 > r) --i;
    return bh * nqt + i;
  }
};

struct PairSeg {
  int t, bh, q0, j0, j1, n;  // tile, its head and first query; key tiles [j0, j1) of n
  int rot;                   // unit j of the tile is key tile (j + rot) mod n
  long long cum;             // first unit of the tile
};

// A cluster's segments in order; every role walks the same sequence.
struct PairWalk {
  PairSplit sp;
  long long u, uend, cum;
  int t;
  __device__ PairWalk(const PairSplit &s, int c) : sp(s) {
    u = s.ubeg(c);
    uend = s.ubeg(c + 1);
    t = u < uend ? s.tile_of(u) : 0;
    cum = s.cum_of(t);
  }
  __device__ __forceinline__ bool more() const { return u < uend; }
  __device__ __forceinline__ bool next(PairSeg &g) {
    if (u >= uend) return false;
    const int n = sp.n_of(t);
    g.t = t;
    g.n = n;
    g.cum = cum;
    g.j0 = (int)(u - cum);
    g.j1 = (int)min((long long)n, uend - cum);
    g.bh = t / sp.nqt;
    // The first contributor of a tile visits key tile (its step) mod n, so
    // clusters that started together read the same K and V tiles at the same
    // time (a measured few per cent faster than scattered reads).
    g.rot = sp.split ? (int)((cum - sp.ubeg(sp.owner(cum))) % n) : 0;
    const int i = t % sp.nqt;
    g.q0 = (sp.causal ? sp.nqt - 1 - i : i) * BQ;
    u = cum + g.j1;
    cum += n;
    ++t;
    return true;
  }
};

// 32 output columns e0 .. e0+31 of a warp's 32 query rows (row = lane), as
// fp16; o_w points at column 0 of the warp's first row, rows_valid of its
// rows exist, columns at or past d are not written.  A full block goes out
// as 64 contiguous bytes per row: a 4 x 4 transpose of 16-byte pieces inside
// each group of 4 lanes lets lanes 4g..4g+3 write one row per store.
__device__ __forceinline__ void store_o32(uint16_t *o_w, int ldc, int rows_valid, int e0, int d, const float (&v)[32],
                                          int lane) {
  if ((d & 7) == 0 && e0 + 32 <= d) {
    const int j4 = lane & 3, g4 = lane & ~3;
    uint32_t a[4][4];  // a[k] = this row's 16-byte piece k (columns 8k .. 8k+7)
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int m = 0; m < 4; ++m) a[k][m] = pack_op2(v[8 * k + 2 * m], v[8 * k + 2 * m + 1]);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      // (lane j of the group, piece k) -> (lane k, piece j)
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
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int r = g4 + ii;  // row written by this group in store ii
      if (r < rows_valid)
        *reinterpret_cast<uint4 *>(o_w + (long long)r * ldc + e0 + j4 * 8) =
            make_uint4(a[ii][0], a[ii][1], a[ii][2], a[ii][3]);
    }
  } else if (lane < rows_valid) {
    uint16_t *orow = o_w + (long long)lane * ldc;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (e0 + i < d) {
        orow[e0 + i] = op_bits(v[i]);
      }
  }
}

template <int VAR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PTHREADS, 1)
    attention_pair_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const AttnArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw;
  // The layout needs a 1024-byte aligned base (128B-swizzled operands) and
  // leaves no room to realign.  The base is the same in every CTA of the
  // launch, so both CTAs of a cluster leave here together.
  if ((smem_u32(sm) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicOr(args.err, (uint32_t)DEV_MISALIGNED);
    return;
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + P_BARS);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + P_BARS + PB_COUNT * 8);
  volatile uint32_t *abort_flag = tmem_slot + 1;
  volatile uint32_t *last_flag = tmem_slot + 2;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cid = (int)(blockIdx.x >> 1);
  const PairSplit sp{(args.N + BQ - 1) / BQ, args.causal, args.pair_split, args.pair_P, args.pair_U};
  const int G = (int)(sp.ubeg(cid + 1) - sp.ubeg(cid));  // key tiles this cluster processes

  if (threadIdx.x == 0) {
    for (int i = 0; i < PNST_MAX; ++i) {
      mbar_init(&bars[PB_FULL + i], 1);
      mbar_init(&bars[PB_EMPTY + i], 1);
    }
    mbar_init(&bars[PB_QREADY], 8);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[PB_SFULL + b], 1);
      mbar_init(&bars[PB_SFREE + b], 8);
      mbar_init(&bars[PB_STGFREE + b], 1);
    }
    for (int b = 0; b < PNPB; ++b) {
      mbar_init(&bars[PB_PFULL + b], 1);
      mbar_init(&bars[PB_OREADY + b], 4);
      mbar_init(&bars[PB_PVDONE + b], 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars[PB_XBAR + i], 2);
    mbar_init(&bars[PB_LFULL], 1);
    mbar_init(&bars[PB_LFREE], 1);
    mbar_init(&bars[PB_OFINAL], 1);
    mbar_init(&bars[PB_OFREE], 8);
    mbar_init(&bars[PB_DRAIN], 1);
    *abort_flag = 0u;
    fence_barrier_init();
    if (rank == 1) {
      // Armed for the first PNPB key tiles and for the first segment's row
      // sums and maxima; the bytes come from the score CTA.
      for (int b = 0; b < PNPB && b < G; ++b) mbar_arrive_expect_tx(&bars[PB_PFULL + b], PMSG_BYTES);
      mbar_arrive_expect_tx(&bars[PB_LFULL], PLM_BYTES);
      tma_prefetch_desc(&vmap);
    } else {
      tma_prefetch_desc(&kmap);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();
  pdl_wait();  // inputs of the previous kernel visible from here on
  const Abort ab{abort_flag, args.err, args.timeout_ns};
  const uint32_t slot16 = (uint32_t)PSLOT >> 4;
  bool ok = true;

  if (warp == 0 || warp == 10) {
    // ------------------------------------------------------ TMA producers
    // Load L goes to ring slot L mod nst; warp 0 issues the even loads, warp
    // 10 the odd ones.  Rank 0: K as [2 x 64 dims] x 128 keys per load (4 per
    // key tile); rank 1: V^T as [256 output dims x 64 keys] (output half 0,
    // then half 1, two key blocks each).
    if (lane == 0) {
      const int me = warp == 0 ? 0 : 1;
      const int nst = rank == 0 ? PNST_S : PNST_O;
      uint8_t *ring = sm + (rank == 0 ? P_RING_S : P_RING_O);
      // A strided loop over this warp's own loads: a loop that visits every
      // load and skips the other warp's measured markedly slower.
      int last = -1, lbase = 0;
      PairWalk wk(sp, cid);
      PairSeg sg;
      while (ok && wk.next(sg)) {
        const int nl = (sg.j1 - sg.j0) * 4;  // lbase is a multiple of 4: the parity split holds
        for (int t = me; t < nl; t += 2) {
          const int L = lbase + t, s = L % nst, round = L / nst;
          if (round > 0 && !mbar_wait(&bars[PB_EMPTY + s], (uint32_t)((round - 1) & 1), ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars[PB_FULL + s], (uint32_t)PSLOT);
          const int j = (sg.j0 + (t >> 2) + sg.rot) % sg.n, r = t & 3;
          if (rank == 0)
            tma_load_4d(ring + s * PSLOT, &kmap, &bars[PB_FULL + s], 0, j * PK, 2 * r, sg.bh);
          else
            tma_load_3d(ring + s * PSLOT, &vmap, &bars[PB_FULL + s], j * PK + (r & 1) * 64, (r >> 1) * 256, sg.bh);
          last = L;
        }
        lbase += nl;
      }
      // After an abort no load may still be landing when the CTA leaves.
      if (*abort_flag)
        for (int t = last; t >= 0 && t > last - 2 * nst; t -= 2)
          mbar_wait_drain(&bars[PB_FULL + t % nst], (uint32_t)((t / nst) & 1), drain_limit(ab));
    }
    __syncwarp();
  } else if (rank == 0) {
    // ===================================================== score CTA ======
    if (warp == 1) {
      // The whole warp runs the issue loop and one elected lane issues: a
      // loop run by a single divergent lane cannot keep N = 128 MMAs back to
      // back.  The elected lane is always lane 0, so every commit tracks all
      // MMAs issued before it.
      const uint64_t rd = sdesc_k128(smem_u32(sm + P_RING_S));
      const uint32_t idesc = idesc_f16(BQ, PK);
      int s = 0, g = 0, si = 0;
      uint32_t ph = 0;
      bool issued = false;
      PairWalk wk(sp, cid);
      PairSeg sg;
      while (ok && wk.next(sg)) {
        // Q of this segment's tile is in tensor memory.
        if (!mbar_wait_warp(&bars[PB_QREADY], (uint32_t)(si & 1), ab)) { ok = false; break; }
        for (int j = sg.j0; j < sg.j1 && ok; ++j, ++g) {
          const int buf = g & 1, u = g >> 1;
          if (g >= 2 && !mbar_wait_warp(&bars[PB_SFREE + buf], (uint32_t)((u - 1) & 1), ab)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_s = tmem + (uint32_t)(buf * PK);
          for (int c = 0; c < 4 && ok; ++c) {
            if (!mbar_wait_warp(&bars[PB_FULL + s], ph, ab)) { ok = false; break; }
            tc_fence_after();
            const uint64_t b0 = rd + (uint64_t)(s * slot16);
            if (elect_one()) {
#pragma unroll
              for (int ks = 0; ks < 8; ++ks)  // 16 dims per step; Q dims 2c' and 2c'+1 in column 256 + c'
                mma_f16_ts(d_s, tmem + 256u + (uint32_t)((c * 8 + ks) * 8),
                           b0 + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2), idesc, (c | ks) ? 1u : 0u);
              mma_commit(&bars[PB_EMPTY + s]);
            }
            __syncwarp();
            issued = true;
            if (++s == PNST_S) { s = 0; ph ^= 1u; }
          }
          if (ok) {
            if (elect_one()) mma_commit(&bars[PB_SFULL + buf]);
            __syncwarp();
          }
        }
        ++si;
      }
      if (issued) {  // every issued MMA completes before tensor memory is freed
        if (elect_one()) mma_commit(&bars[PB_DRAIN]);
        __syncwarp();
        mbar_wait_drain(&bars[PB_DRAIN], 0, drain_limit(ab));
      }
      __syncwarp();
    } else {
      const int q4 = warp & 3;
      const int half = (warp - 2) >> 2;
      const int row = q4 * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      const float sl2 = args.sl2;
      constexpr bool var = VAR != 0;
      float *xch = reinterpret_cast<float *>(sm + P_SMALL);  // [2 parity][2 half][128]
      const uint32_t r_base = mapa_u32(smem_u32(sm), 1u);
      const uint32_t r_alpha = mapa_u32(smem_u32(sm + P_ALPHA), 1u);
      const uint32_t r_flags = mapa_u32(smem_u32(sm + P_FLAGS), 1u);
      const uint32_t r_lsum = mapa_u32(smem_u32(sm + P_LSUM), 1u);
      const uint32_t r_mrow = mapa_u32(smem_u32(sm + P_MROW), 1u);
      const uint32_t r_pfull0 = mapa_u32(smem_u32(&bars[PB_PFULL]), 1u);
      const uint32_t r_lfull = mapa_u32(smem_u32(&bars[PB_LFULL]), 1u);
      int g = 0, xi = 0, si = 0;
      PairWalk wk(sp, cid);
      PairSeg sg;
      while (ok && wk.next(sg)) {
        const int q0 = sg.q0, bh = sg.bh;
        {
          // Q rows into tensor memory: this warp's 32 rows, dims half*256 ..
          // +255 (rows past N are zero).  The previous segment's QK^T MMAs
          // all completed before its last scores were read.
          const bool qv = q0 + row < args.N;
          const uint4 *qrow = reinterpret_cast<const uint4 *>(
              args.q + ((long long)bh * args.N + (qv ? q0 + row : 0)) * args.ldq + half * 256);
          for (int c = 0; c < 4; ++c) {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 v = qv ? __ldg(qrow + c * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
              w[4 * i] = v.x;
              w[4 * i + 1] = v.y;
              w[4 * i + 2] = v.z;
              w[4 * i + 3] = v.w;
            }
            tmem_st32(lane_base + 256u + (uint32_t)(half * 128 + c * 32), w);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[PB_QREADY]);
        }
        float m_used = -INFINITY, l = 0.f;
        if (VAR == 1) rel_prefetch<2>(args, bh % args.h, q0 + row, ((sg.j0 + sg.rot) % sg.n) * PK + half * 64, lane);
        for (int j = sg.j0; j < sg.j1; ++j, ++g, ++xi) {
          const int buf = g & 1, u = g >> 1;
          if (!mbar_wait_warp(&bars[PB_SFULL + buf], (uint32_t)(u & 1), ab)) { ok = false; break; }
          tc_fence_after();
          uint32_t r[2][32];
          tmem_ld32(lane_base + (uint32_t)(buf * PK + half * 64), r[0]);
          tmem_ld32(lane_base + (uint32_t)(buf * PK + half * 64 + 32), r[1]);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[PB_SFREE + buf]);
          const int kt = (j + sg.rot) % sg.n;  // key tile
          const int kvalid = min(PK, args.N - kt * PK) - half * 64;
          if (kvalid < 64) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (32 * c + i >= kvalid) r[c][i] = __float_as_uint(-INFINITY);
          }
          float sc = sl2;  // base-2 logits when the table was added
          if (var && apply_variants<2, VAR == 2>(r, args, bh % args.h, q0 + row, kt * PK + half * 64, sl2, lane))
            sc = 1.f;
          if (VAR == 1 && j + 1 < sg.j1)
            rel_prefetch<2>(args, bh % args.h, q0 + row, ((j + 1 + sg.rot) % sg.n) * PK + half * 64, lane);
          float pm[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int c = t >> 1, o = (t & 1) * 16;
            float m = __uint_as_float(r[c][o]);
#pragma unroll
            for (int i = 1; i < 15; i += 2)
              m = max3f(m, __uint_as_float(r[c][o + i]), __uint_as_float(r[c][o + i + 1]));
            pm[t] = fmaxf(m, __uint_as_float(r[c][o + 15]));
          }
          float mx = fmaxf(max3f(pm[0], pm[1], pm[2]), pm[3]);
          // The other half of this row (same lanes, other warp): exchange maxima.
          xch[((xi & 1) * 2 + half) * 128 + row] = mx;
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[PB_XBAR + q4]);
          if (!mbar_wait_warp(&bars[PB_XBAR + q4], (uint32_t)(xi & 1), ab)) { ok = false; break; }
          mx = fmaxf(mx, xch[((xi & 1) * 2 + (half ^ 1)) * 128 + row]);
          const float m_new = fmaxf(m_used, mx * sc);
          const bool need = (j > sg.j0) && (m_new > m_used + RESCALE_LOG2_F32);
          const bool rescale = __any_sync(0xFFFFFFFFu, need) != 0;
          float alpha = 1.f;
          if (j == sg.j0) {
            m_used = m_new;
          } else if (rescale && m_new > m_used) {
            alpha = ex2_approx(m_used - m_new);
            m_used = m_new;
          }
          const uint64_t c2 = f2_pack(sc, sc);
          const uint64_t nm2 = f2_pack(-m_used, -m_used);
          uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float t0, t1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1])), c2, nm2), t0, t1);
              const float e0 = ex2_approx(t0);
              const float e1 = ex2_approx(t1);
              acc2[(i >> 3) & 3] = f2_add(acc2[(i >> 3) & 3], f2_pack(e0, e1));
              pk[c * 16 + (i >> 1)] = pack_op2(e0, e1);
            }
          float s0, s1, s2, s3;
          f2_unpack(f2_add(acc2[0], acc2[1]), s0, s1);
          f2_unpack(f2_add(acc2[2], acc2[3]), s2, s3);
          l = l * alpha + ((s0 + s1) + (s2 + s3));
          // Staging tile `buf` is free once the copy of tile g-2 has landed;
          // the output CTA's P buffer `pb` once its P V_{g-PNPB} is done.
          const int pb = g % PNPB, up = g / PNPB;
          if (g >= 2 && !mbar_wait_cluster_warp(&bars[PB_STGFREE + buf], (uint32_t)((u - 1) & 1), ab)) {
            ok = false;
            break;
          }
          if (g >= PNPB && !mbar_wait_cluster_warp(&bars[PB_PVDONE + pb], (uint32_t)((up - 1) & 1), ab)) {
            ok = false;
            break;
          }
          uint8_t *stg = sm + buf * 32768 + half * 16384;  // this half's 64 keys
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(smem_u32(stg) + sw128_offset((uint32_t)row, (uint32_t)ch), pk[ch * 4], pk[ch * 4 + 1],
                         pk[ch * 4 + 2], pk[ch * 4 + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          const uint32_t rbar = r_pfull0 + (uint32_t)(pb * 8);
          if (lane == 0)
            bulk_copy_to_cluster(r_base + (uint32_t)(pb * 32768 + half * 16384 + q4 * 4096), stg + q4 * 4096, 4096u,
                                 rbar);
          if (half == 0) {
            st_async_b32(r_alpha + (uint32_t)((pb * 128 + row) * 4), __float_as_uint(alpha), rbar);
            if (lane == 0) st_async_b32(r_flags + (uint32_t)((pb * 4 + q4) * 4), rescale ? 1u : 0u, rbar);
          }
        }
        if (!ok) break;
        // End of the segment: combine the two halves' row sums and send the
        // sums and maxima to the output CTA once it has taken the previous
        // segment's.
        xch[((xi & 1) * 2 + half) * 128 + row] = l;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[PB_XBAR + q4]);
        if (!mbar_wait_warp(&bars[PB_XBAR + q4], (uint32_t)(xi & 1), ab)) { ok = false; break; }
        l += xch[((xi & 1) * 2 + (half ^ 1)) * 128 + row];
        ++xi;
        if (half == 0) {
          if (si > 0 && !mbar_wait_cluster_warp(&bars[PB_LFREE], (uint32_t)((si - 1) & 1), ab)) { ok = false; break; }
          st_async_b32(r_lsum + (uint32_t)(row * 4), __float_as_uint(l), r_lfull);
          st_async_b32(r_mrow + (uint32_t)(row * 4), __float_as_uint(m_used), r_lfull);
        }
        ++si;
      }
      // The completions of the last P V products also arrive here; this CTA
      // stays until they have.
      if (warp == 2 && lane == 0 && ok)
        for (int gg = max(0, G - PNPB); gg < G; ++gg)
          if (!mbar_wait_cluster(&bars[PB_PVDONE + gg % PNPB], (uint32_t)((gg / PNPB) & 1), ab)) break;
      __syncwarp();
    }
  } else {
    // ==================================================== output CTA ======
    if (warp == 1) {
      // Warp-uniform issue loop, elected lane 0 issues (as in the score CTA).
      const uint64_t pd = sdesc_k128(smem_u32(sm));
      const uint64_t rd = sdesc_k128(smem_u32(sm + P_RING_O));
      const uint32_t idesc = idesc_f16(BQ, 256);
      const uint32_t r_stgfree0 = mapa_u32(smem_u32(&bars[PB_STGFREE]), 0u);
      int s = 0, g = 0, si = 0;
      uint32_t ph = 0;
      bool issued = false;
      PairWalk wk(sp, cid);
      PairSeg sg;
      while (ok && wk.next(sg)) {
        // O is free once the previous segment's result has been read out.
        if (si > 0 && !mbar_wait_warp(&bars[PB_OFREE], (uint32_t)((si - 1) & 1), ab)) { ok = false; break; }
        tc_fence_after();
        for (int j = sg.j0; j < sg.j1 && ok; ++j, ++g) {
          const int buf = g % PNPB, u = g / PNPB;
          if (!mbar_wait_cluster_warp(&bars[PB_PFULL + buf], (uint32_t)(u & 1), ab)) { ok = false; break; }
          // P_g has landed, so the score CTA's staging tile g mod 2 is free.
          // (No ordering to publish: a relaxed arrive, which keeps this warp's
          // issue loop short.)
          if (elect_one() && g + 2 < G) mbar_arrive_remote_relaxed(r_stgfree0 + (uint32_t)((g & 1) * 8));
          __syncwarp();
          if (!mbar_wait_warp(&bars[PB_OREADY + buf], (uint32_t)(u & 1), ab)) { ok = false; break; }
          if (elect_one()) {
            if (g + PNPB < G) mbar_arrive_expect_tx(&bars[PB_PFULL + buf], PMSG_BYTES);
            fence_proxy_async_smem();  // P and the rescale factors came from the other CTA
          }
          __syncwarp();
          tc_fence_after();
          for (int r = 0; r < 4 && ok; ++r) {
            if (!mbar_wait_warp(&bars[PB_FULL + s], ph, ab)) { ok = false; break; }
            tc_fence_after();
            const uint64_t a0 = pd + (uint64_t)(buf * 2048 + (r & 1) * 1024);
            const uint64_t b0 = rd + (uint64_t)(s * slot16);
            const uint32_t d_o = tmem + (uint32_t)((r >> 1) * 256);
            const uint32_t first = (j > sg.j0 || (r & 1) > 0) ? 1u : 0u;
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16_ss(d_o, a0 + (uint64_t)(kk * 2), b0 + (uint64_t)(kk * 2), idesc, (first | kk) ? 1u : 0u);
              mma_commit(&bars[PB_EMPTY + s]);
            }
            __syncwarp();
            issued = true;
            if (++s == PNST_O) { s = 0; ph ^= 1u; }
          }
          if (ok) {
            if (elect_one()) mma_commit_mc(&bars[PB_PVDONE + buf], (uint16_t)3u);  // both CTAs
            __syncwarp();
          }
        }
        if (ok) {
          if (elect_one()) mma_commit(&bars[PB_OFINAL]);
          __syncwarp();
        }
        ++si;
      }
      if (issued) {  // every issued MMA completes before tensor memory is freed
        if (elect_one()) mma_commit(&bars[PB_DRAIN]);
        __syncwarp();
        mbar_wait_drain(&bars[PB_DRAIN], 0, drain_limit(ab));
      }
      __syncwarp();
    } else {
      const int q4 = warp & 3;
      const int half = (warp - 2) >> 2;
      const int row = q4 * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      const volatile float *alpha_s = reinterpret_cast<const volatile float *>(sm + P_ALPHA);
      const volatile uint32_t *flags = reinterpret_cast<const volatile uint32_t *>(sm + P_FLAGS);
      const uint32_t r_lfree = mapa_u32(smem_u32(&bars[PB_LFREE]), 0u);
      int g = 0, si = 0;
      PairWalk wk(sp, cid);
      PairSeg sg;
      // The eight warps meet at named barriers in every segment, so none
      // leaves the loop alone: a failed wait is carried to the first barrier
      // of the segment, which every warp then leaves with the same verdict.
      while (wk.next(sg)) {
        if (warp < 6) {
          // Rescale O rows before P_j V_j when the score CTA raised their
          // running maximum.
          for (int j = sg.j0; j < sg.j1 && ok; ++j, ++g) {
            const int buf = g % PNPB, u = g / PNPB;
            if (!mbar_wait_cluster_warp(&bars[PB_PFULL + buf], (uint32_t)(u & 1), ab)) { ok = false; break; }
            if (j > sg.j0 && flags[buf * 4 + q4] != 0u) {
              if (!mbar_wait_warp(&bars[PB_PVDONE + (g - 1) % PNPB], (uint32_t)(((g - 1) / PNPB) & 1), ab)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const float a = alpha_s[buf * 128 + row];
              for (int cc = 0; cc < 32; ++cc) {
                uint32_t t[16];
                tmem_ld16(lane_base + (uint32_t)(cc * 16), t);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * a);
                tmem_st16(lane_base + (uint32_t)(cc * 16), t);
              }
              tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[PB_OREADY + buf]);
          }
        }
        // Epilogue of the segment, warps (q4, half) each taking 16 of the 32
        // 16-column chunks of their rows.
        const bool eok = ok && mbar_wait_warp(&bars[PB_OFINAL], (uint32_t)(si & 1), ab) &&
                         mbar_wait_cluster_warp(&bars[PB_LFULL], (uint32_t)(si & 1), ab);
        float m_row = 0.f, l_row = 1.f;
        if (eok) {
          tc_fence_after();
          m_row = reinterpret_cast<const volatile float *>(sm + P_MROW)[row];
          l_row = reinterpret_cast<const volatile float *>(sm + P_LSUM)[row];
        }
        // All eight warps hold this segment's l and m (or all give up).
        if (!named_bar_and(1, 256, eok)) {
          ok = false;
          break;
        }
        if (warp == 2 && lane == 0 && wk.more()) {
          mbar_arrive_expect_tx(&bars[PB_LFULL], PLM_BYTES);
          mbar_arrive_remote(r_lfree);
        }
        // Warp (q4, half) writes columns half*256 .. +255 of its 32 rows, 32
        // columns at a time.
        const int b = sg.bh / args.h, hd = sg.bh % args.h;
        const int row0 = sg.q0 + q4 * 32;
        uint16_t *o_w = args.o + ((long long)b * args.N + row0) * args.ldc + (long long)hd * args.d;
        const int rows_valid = args.N - row0;
        if (sg.j0 == 0 && sg.j1 == sg.n) {
          const float inv = 1.0f / l_row;
          for (int blk = half * 8; blk < half * 8 + 8; ++blk) {
            uint32_t t[32];
            tmem_ld32(lane_base + (uint32_t)(blk * 32), t);
            tmem_wait_ld();
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(t[i]) * inv;
            store_o32(o_w, args.ldc, rows_valid, blk * 32, args.d, v, lane);
          }
        } else {
          // Part of a tile cut between clusters: publish this part, count in.
          // Layout of a part: [16 column blocks][8 pieces][128 rows][4 floats],
          // so each store (and each load of the merge) moves 512 contiguous
          // bytes per warp.  When every other contributor has already counted
          // in (typically: this cluster ends its range with the tile's last
          // piece, the next began its range with the first), this one merges
          // straight from tensor memory without publishing its own part.
          const int c_lo = sp.owner(sg.cum), c_hi = sp.owner(sg.cum + sg.n - 1);
          if (warp == 2 && lane == 0)
            *last_flag = *reinterpret_cast<volatile uint32_t *>(args.cnt + sg.t) == (uint32_t)(c_hi - c_lo) ? 2u : 0u;
          named_bar_sync(1, 256);
          if (*last_flag != 2u) {
            const int mine = 2 * cid + (sp.ubeg(cid) < sg.cum ? 1 : 0);
            float *part = args.part + (long long)mine * PART_FLOATS;
            for (int blk = half * 8; blk < half * 8 + 8; ++blk) {
              uint32_t t[32];
              tmem_ld32(lane_base + (uint32_t)(blk * 32), t);
              tmem_wait_ld();
#pragma unroll
              for (int pc = 0; pc < 8; ++pc)
                __stcg(reinterpret_cast<uint4 *>(part + ((blk * 8 + pc) * 128 + row) * 4),
                       make_uint4(t[4 * pc], t[4 * pc + 1], t[4 * pc + 2], t[4 * pc + 3]));
            }
            if (half == 0) {
              __stcg(part + PART_O_FLOATS + row, m_row);
              __stcg(part + PART_O_FLOATS + 128 + row, l_row);
            }
            __threadfence();
            named_bar_sync(1, 256);
            if (warp == 2 && lane == 0) {
              const uint32_t prev = atomicAdd(args.cnt + sg.t, 1u);
              *last_flag = prev == (uint32_t)(c_hi - c_lo) ? 1u : 0u;
            }
            named_bar_sync(1, 256);
          }
          if (*last_flag) {
            // Every other part is published: merge them into this one, each
            // rescaled to the common row maximum.
            __threadfence();
            float M = m_row;
            for (int c = c_lo; c <= c_hi; ++c)
              if (c != cid) {
                const int sl = 2 * c + (sp.ubeg(c) < sg.cum ? 1 : 0);
                M = fmaxf(M, __ldcg(args.part + (long long)sl * PART_FLOATS + PART_O_FLOATS + row));
              }
            const float a_self = exp2f(m_row - M);
            float L = l_row * a_self;
            for (int c = c_lo; c <= c_hi; ++c)
              if (c != cid) {
                const float *pp = args.part + (long long)(2 * c + (sp.ubeg(c) < sg.cum ? 1 : 0)) * PART_FLOATS;
                L += __ldcg(pp + PART_O_FLOATS + 128 + row) * exp2f(__ldcg(pp + PART_O_FLOATS + row) - M);
              }
            const float inv = 1.0f / L;
            // Plain instance: two 32-column blocks per pass, sixteen 16-byte
            // loads of a part in flight per thread (vae16384 block 522.2 ->
            // 520.2 us); the variant instances, short of registers, one.
            constexpr int NB = VAR == 0 ? 2 : 1;
            for (int blk = half * 8; blk < half * 8 + 8; blk += NB) {
              float v[NB][32];
#pragma unroll
              for (int h2 = 0; h2 < NB; ++h2) {
                uint32_t t[32];
                tmem_ld32(lane_base + (uint32_t)((blk + h2) * 32), t);
                tmem_wait_ld();
                const float as = a_self * inv;
#pragma unroll
                for (int i = 0; i < 32; ++i) v[h2][i] = __uint_as_float(t[i]) * as;
              }
              for (int c = c_lo; c <= c_hi; ++c)
                if (c != cid) {
                  const float *pp = args.part + (long long)(2 * c + (sp.ubeg(c) < sg.cum ? 1 : 0)) * PART_FLOATS;
                  float4 f[NB][8];
#pragma unroll
                  for (int h2 = 0; h2 < NB; ++h2)
#pragma unroll
                    for (int pc = 0; pc < 8; ++pc)
                      f[h2][pc] =
                          __ldcg(reinterpret_cast<const float4 *>(pp + (((blk + h2) * 8 + pc) * 128 + row) * 4));
                  const float a = exp2f(__ldcg(pp + PART_O_FLOATS + row) - M) * inv;
#pragma unroll
                  for (int h2 = 0; h2 < NB; ++h2)
#pragma unroll
                    for (int pc = 0; pc < 8; ++pc) {
                      v[h2][4 * pc] = fmaf(f[h2][pc].x, a, v[h2][4 * pc]);
                      v[h2][4 * pc + 1] = fmaf(f[h2][pc].y, a, v[h2][4 * pc + 1]);
                      v[h2][4 * pc + 2] = fmaf(f[h2][pc].z, a, v[h2][4 * pc + 2]);
                      v[h2][4 * pc + 3] = fmaf(f[h2][pc].w, a, v[h2][4 * pc + 3]);
                    }
                }
#pragma unroll
              for (int h2 = 0; h2 < NB; ++h2) store_o32(o_w, args.ldc, rows_valid, (blk + h2) * 32, args.d, v[h2], lane);
            }
          }
        }
        // O has been read out: the next segment's P V may overwrite it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[PB_OFREE]);
        ++si;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  // Neither CTA leaves while the other may still touch its shared memory.
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Clusters of the pair kernel that are resident at once on the current device.
int pair_active_clusters(const void *kern) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * PAIR_MAX_CLUSTERS, 1, 1);
  cfg.blockDim = dim3(PTHREADS, 1, 1);
  cfg.dynamicSmemBytes = P_SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    int nsm = 0;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    n = nsm / 2;
  }
  cached[dev] = n;
  return n;
}

int launch_attention_pair(const Dims &dm, AttnArgs a, const uint16_t *q, const uint16_t *k, const uint16_t *vt,
                          void *scratch, cudaStream_t st) {
  int max_smem = MAX_SMEM_FALLBACK, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if ((int)P_SMEM > max_smem) return 2;
  a.q = q;
  a.ldq = dm.ldq;
  CUtensorMap kmap, vmap;
  const uint64_t BH = (uint64_t)dm.B * dm.h;
  {
    // K viewed as [bh][64-dim chunk][key][64 dims]: one load = 2 chunks x 128 keys.
    const uint64_t dims[4] = {64, (uint64_t)dm.N, (uint64_t)dm.ldq / 64, BH};
    const uint64_t strides[3] = {(uint64_t)dm.ldq * 2, 128, (uint64_t)dm.N * dm.ldq * 2};
    const uint32_t box[4] = {64, PK, 2, 1};
    if (encode_tiled(&kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, k, dims, strides, box,
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
  const int var = (a.rel && (a.gw & 31) != 0) ? 2 : ((a.causal || a.rel) ? 1 : 0);
  auto kern = var == 2 ? attention_pair_kernel<2> : (var == 1 ? attention_pair_kernel<1> : attention_pair_kernel<0>);
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_SMEM);
  const long long nqt = (dm.N + BQ - 1) / BQ, T = (long long)BH * nqt;
  a.pair_U = a.causal ? (long long)BH * (nqt * (nqt + 1) / 2) : T * nqt;
  // By default tiles are split only when there are more tiles than clusters
  // (a partial last wave; every piece then spans at least one tile, so a tile
  // has at most two contributors).  With fewer tiles the pieces shrink to a
  // few key tiles and the parts and merges cost more than the idle SM pairs
  // (vae1024: 69 vs 34 us); under the causal mask heaviest-first whole tiles
  // measured faster (273-281 vs 367-378 us at 128 tiles).
  const int policy = attention_split_policy();
  const int active =
      (scratch && policy != 2) ? pair_active_clusters(reinterpret_cast<const void *>(kern)) : 0;
  if (active > 0 && (policy == 1 || (!a.causal && T > active))) {
    a.pair_split = 1;
    a.pair_P = (int)std::min<long long>(std::min(active, PAIR_MAX_CLUSTERS), a.pair_U);
    a.part = static_cast<float *>(scratch);
    a.cnt = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(scratch) +
                                         (size_t)2 * a.pair_P * PART_FLOATS * sizeof(float));
    if (cudaMemsetAsync(a.cnt, 0, (size_t)T * sizeof(uint32_t), st) != cudaSuccess) return 2;
  } else {
    a.pair_split = 0;
    a.pair_P = (int)T;
  }
  (void)launch_k(kern, dim3(2u * (unsigned)a.pair_P, 1, 1), dim3(PTHREADS), P_SMEM, st, kmap, vmap, a);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

int launch_attention_quad(const Dims &dm, AttnArgs a, const uint16_t *q, const uint16_t *k, const uint16_t *vt,
                          uint16_t *o, const KParams &kp, cudaStream_t st) {
  a.sl2 = 1.4426950408889634f / sqrtf((float)dm.d);
  a.o = o;
  a.err = kp.err;
  a.timeout_ns = kp.timeout_ns;
  a.stall = stall_for(kp, STALL_ATTENTION);
  a.ones = dm.dp > dm.d ? 1 : 0;  // V^T row d holds ones (the weight pack sets that bias)
  CUtensorMap qmap, kmap, vmap;
  const uint64_t BH = (uint64_t)dm.B * dm.h;
  {
    const uint64_t dims[3] = {(uint64_t)dm.ldq, (uint64_t)dm.N, BH};
    const uint64_t strides[2] = {(uint64_t)dm.ldq * 2, (uint64_t)dm.N * dm.ldq * 2};
    const uint32_t qbox[3] = {64, BQ, 1};
    const uint32_t kbox[3] = {64, QK, 1};
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
    const uint32_t box[3] = {QK, (uint32_t)dm.dp, 1};
    if (encode_tiled(&vmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, vt, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return 1;
  }
  // Two query tiles per CTA whenever there are two; one otherwise.  The
  // table instances read the table through L1: shared memory only as large
  // as two CTAs need (the plain ones take the whole carveout).
  const int nqt = (dm.N + BQ - 1) / BQ;
  auto run = [&](auto kern, int qt, uint32_t smem, int threads, int carveout) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (carveout >= 0) cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
    (void)launch_k(kern, dim3((unsigned)((nqt + qt - 1) / qt), (unsigned)BH, 1), dim3(threads), smem, st, qmap, kmap,
                   vmap, a);
  };
  const bool table = a.rel != nullptr;
  if (nqt >= 2) {
    if (table) run(attention_quad_kernel<2, 1>, 2, QuadCfg<2>::SMEM, QuadCfg<2>::THREADS, 72);
    else run(attention_quad_kernel<2, 0>, 2, QuadCfg<2>::SMEM, QuadCfg<2>::THREADS, 100);
  } else {
    if (table) run(attention_quad_kernel<1, 1>, 1, QuadCfg<1>::SMEM, QuadCfg<1>::THREADS, -1);
    else run(attention_quad_kernel<1, 0>, 1, QuadCfg<1>::SMEM, QuadCfg<1>::THREADS, -1);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace

size_t attention_scratch_bytes(const Dims &dm) {
  if (dm.dp != 512) return 0;
  const long long nqt = (dm.N + BQ - 1) / BQ, T = (long long)dm.B * dm.h * nqt;
  const long long P = std::min<long long>(PAIR_MAX_CLUSTERS, T * nqt);
  return (size_t)2 * P * PART_FLOATS * sizeof(float) + (size_t)T * sizeof(uint32_t);
}

int launch_attention(const Dims &dm, const uint16_t *q, const uint16_t *k, const uint16_t *vt, uint16_t *o,
                     const KParams &kp, cudaStream_t st, int causal, const float *rel, void *scratch) {
  AttnArgs a{};
  a.N = dm.N; a.h = dm.h; a.d = dm.d; a.dp = dm.dp; a.ldc = dm.ldc; a.d_o = dm.d_o; a.n_oc = dm.n_oc;
  a.causal = causal; a.rel = rel; a.gh = dm.H; a.gw = dm.W; a.tabn = (2 * dm.H - 1) * (2 * dm.W - 1);
  a.nqb = (dm.dp + 63) / 64;
  a.ntiles = (dm.N + BKV - 1) / BKV;
  if (dm.dp == 512) {
    a.sl2 = 1.4426950408889634f / sqrtf((float)dm.d);
    a.o = o;
    a.err = kp.err;
    a.timeout_ns = kp.timeout_ns;
    a.N = dm.N; a.h = dm.h; a.d = dm.d; a.ldc = dm.ldc;
    return launch_attention_pair(dm, a, q, k, vt, scratch, st);
  }
  if (dm.dp <= 64 && !causal && (rel == nullptr || dm.W % 32 == 0))
    return launch_attention_quad(dm, a, q, k, vt, o, kp, st);
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
  // Single mode with d_o <= 64: a tile's two V halves share one slot, so a key
  // tile takes two ring slots instead of three and four slots prefetch two
  // tiles (per-stage timing showed P V waiting for V with three).
  a.vpack = (a.single && a.nvr == 1 && 2 * a.vrows * 128 <= a.slot && (a.vrows % 8) == 0) ? 1 : 0;
  // V^T row d holds ones whenever d < dp (the weight pack sets that bias)
  a.ones = (a.single && dm.dp > dm.d) ? 1 : 0;
  if (nst < 2) return 2;
  a.nst = nst;
  a.sl2 = 1.4426950408889634f / sqrtf((float)dm.d);
  a.o = o;
  a.err = kp.err;
  a.timeout_ns = kp.timeout_ns;
  a.stall = stall_for(kp, STALL_ATTENTION);

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
  const dim3 grid = a.causal ? dim3((unsigned)BH, (dm.N + BQ - 1) / BQ * dm.n_oc, 1)
                             : dim3((dm.N + BQ - 1) / BQ * dm.n_oc, (unsigned)BH, 1);
  const int var = (a.rel && (a.gw & 31) != 0) ? 2 : ((a.causal || a.rel) ? 1 : 0);
  if (a.single) {
    auto kern = var == 2 ? attention_kernel<true, 2> : (var == 1 ? attention_kernel<true, 1> : attention_kernel<true, 0>);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    (void)launch_k(kern, dim3(grid), dim3(var ? STHREADS : THREADS), smem, st, qmap, kmap, vmap, a);
  } else {
    auto kern =
        var == 2 ? attention_kernel<false, 2> : (var == 1 ? attention_kernel<false, 1> : attention_kernel<false, 0>);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    (void)launch_k(kern, dim3(grid), dim3(THREADS), smem, st, qmap, kmap, vmap, a);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // namespace ssa
