// gn_stats.cu -- GroupNorm statistics (tensortonic
// "diffusion-l03-spatial-self-attention", problem statement: GN with
// num_groups groups, eps 1e-5, weight norm_weight, bias norm_bias).
//
// In NCHW the (C/G) channels x N pixels of one (sample, group) are one
// contiguous span, so each group is streamed with 16-byte vector loads.  A
// thread keeps Welford-style (count, mean, M2): each batch of loads it has in
// flight (32 values) gets its mean and M2 two-pass in registers and is merged
// once; warps, the CTA and then the CTAs of a thread-block cluster combine
// with Chan's pairwise merge, the cluster step reading the other CTAs'
// partials through distributed shared memory.  No
// global scratch and no second launch are needed.  The cluster's rank-0 CTA
// writes mean, rstd = 1/sqrt(var + 1e-5) (biased variance) and the folded
// affine a = rstd * weight, s = bias - mean * a for the group's channels.
// x is read with an L2 evict-last hint: the projection reads the same x next,
// and keeping it in L2 measured 1.8 us (unet-l1) and 3.1 us (vae16384) off
// the block.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "internal.h"

namespace cg = cooperative_groups;

namespace ssa {
namespace {

constexpr int kThreads = 512;
constexpr float kEps = 1e-5f;

struct Stat {
  float n, mu, m2;
};

__device__ __forceinline__ void chan_merge(Stat &a, const Stat &b) {
  const float nn = a.n + b.n;
  if (nn == 0.f) return;
  const float delta = b.mu - a.mu;
  const float f = __fdividef(b.n, nn);  // counts: a few ulp is plenty
  a.mu = fmaf(delta, f, a.mu);
  a.m2 = a.m2 + b.m2 + delta * delta * a.n * f;
  a.n = nn;
}

template <int DT>
__device__ __forceinline__ float load_scalar(const void *x, long long i) {
  if (DT == 0) return __ldg(reinterpret_cast<const float *>(x) + i);
  const unsigned short u = __ldg(reinterpret_cast<const unsigned short *>(x) + i);
  return __uint_as_float(((uint32_t)u) << 16);
}

// 16 bytes of x, kept in L2 (evict-last) for the projection that reads x next.
__device__ __forceinline__ uint4 ld_keep(const uint4 *p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

template <int DT>
__device__ __forceinline__ float load_param(const void *p, int i) {
  return load_scalar<DT>(p, i);
}

template <int DT>
__device__ __forceinline__ void unpack(const uint4 &r, float (&f)[DT == 0 ? 4 : 8]) {
  if (DT == 0) {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
  } else {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}

// DT 0: fp32 (4 values per 16-byte vector); DT 1: bf16 (8 values).  `per`:
// elements of the group per cluster CTA (a multiple of 8).  Two CTAs per SM.
template <int DT>
__global__ void __launch_bounds__(kThreads, 2) gn_stats_kernel(const void *__restrict__ x, int C, int N, int G,
                                                               long long per, const void *__restrict__ gw,
                                                               const void *__restrict__ gb, float *mean,
                                                               float *rstd, float *ga, float *gs) {
  constexpr int VW = DT == 0 ? 4 : 8;      // elements per 16-byte vector
  constexpr int UNROLL = DT == 0 ? 8 : 4;  // vectors in flight per thread: 32 values
  pdl_trigger();
  pdl_wait();
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int cs = (int)cl.num_blocks();
  const int grp = blockIdx.y;
  const int b = grp / G, g = grp - b * G;
  const int cgc = C / G;
  const long long L = (long long)cgc * N;
  const long long base = ((long long)b * C + (long long)g * cgc) * N;

  // This CTA's slice [s0, s1) of the group.
  const long long s0 = min(L, (long long)rank * per);
  const long long s1 = min(L, s0 + per);

  Stat st{0.f, 0.f, 0.f};
  const int tid = threadIdx.x;
  // Scalar head up to the first 16-byte aligned element.
  long long a0 = s0;
  const int mis = (int)((base + s0) & (VW - 1));
  if (mis) a0 = min(s1, s0 + (VW - mis));
  for (long long i = s0 + tid; i < a0; i += kThreads) chan_merge(st, Stat{1.f, load_scalar<DT>(x, base + i), 0.f});
  const long long nvec = (s1 - a0) / VW;
  const long long a1 = a0 + nvec * VW;
  // Vector body: batches of up to UNROLL independent 16-byte loads per
  // thread, all issued before any is consumed (one memory round trip per
  // batch; most slices need one or two batches).
  const uint4 *xv = reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(x) +
                                                    (base + a0) * (DT == 0 ? 4 : 2));
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  for (long long v = tid; v < nvec; v += (long long)UNROLL * kThreads) {
    uint4 r[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const long long idx = v + (long long)u * kThreads;
      r[u] = idx < nvec ? ld_keep(xv + idx, pol) : make_uint4(0u, 0u, 0u, 0u);
    }
    // The batch's mean and M2, two-pass over its valid vectors (the
    // missing ones read as zeros and are left out of the count and of M2).
    const int nv = (int)min((long long)UNROLL, (nvec - v + kThreads - 1) / kThreads);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float f[VW];
      unpack<DT>(r[u], f);
#pragma unroll
      for (int k = 0; k < VW; ++k) acc[k & 3] += f[k];
    }
    const float cnt = (float)(nv * VW);
    const float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    const float mu = nv == UNROLL ? sum * (1.0f / (UNROLL * VW)) : __fdividef(sum, cnt);
    float m2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      if (u < nv) {
        float f[VW];
        unpack<DT>(r[u], f);
#pragma unroll
        for (int k = 0; k < VW; ++k) {
          const float t = f[k] - mu;
          m2[k & 3] = fmaf(t, t, m2[k & 3]);
        }
      }
    }
    chan_merge(st, Stat{cnt, mu, (m2[0] + m2[1]) + (m2[2] + m2[3])});
  }
  // Scalar tail.
  for (long long i = a1 + tid; i < s1; i += kThreads) chan_merge(st, Stat{1.f, load_scalar<DT>(x, base + i), 0.f});

  // Warp, then CTA merge.
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Stat o;
    o.n = __shfl_xor_sync(0xFFFFFFFFu, st.n, off);
    o.mu = __shfl_xor_sync(0xFFFFFFFFu, st.mu, off);
    o.m2 = __shfl_xor_sync(0xFFFFFFFFu, st.m2, off);
    chan_merge(st, o);
  }
  __shared__ Stat warp_stat[kThreads / 32];
  __shared__ Stat cta_stat;
  __shared__ float fin[2];
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) warp_stat[warp] = st;
  __syncthreads();
  if (warp == 0) {
    Stat t = (lane < kThreads / 32) ? warp_stat[lane] : Stat{0.f, 0.f, 0.f};
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      Stat o;
      o.n = __shfl_xor_sync(0xFFFFFFFFu, t.n, off);
      o.mu = __shfl_xor_sync(0xFFFFFFFFu, t.mu, off);
      o.m2 = __shfl_xor_sync(0xFFFFFFFFu, t.m2, off);
      chan_merge(t, o);
    }
    if (lane == 0) cta_stat = t;
  }
  // Cluster merge through distributed shared memory.
  cl.sync();
  if (rank == 0 && warp == 0) {
    Stat t{0.f, 0.f, 0.f};
    if (lane < cs) t = *cl.map_shared_rank(&cta_stat, (unsigned)lane);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      Stat o;
      o.n = __shfl_xor_sync(0xFFFFFFFFu, t.n, off);
      o.mu = __shfl_xor_sync(0xFFFFFFFFu, t.mu, off);
      o.m2 = __shfl_xor_sync(0xFFFFFFFFu, t.m2, off);
      chan_merge(t, o);
    }
    if (lane == 0) {
      const float var = fmaxf(t.m2 / t.n, 0.f);
      const float r = 1.0f / sqrtf(var + kEps);
      fin[0] = t.mu;
      fin[1] = r;
      if (mean) mean[grp] = t.mu;
      if (rstd) rstd[grp] = r;
    }
  }
  cl.sync();  // the other CTAs' shared memory has been read
  if (rank == 0) {
    __syncthreads();
    const float mu = fin[0], r = fin[1];
    for (int c = tid; c < cgc; c += kThreads) {
      const int ch = g * cgc + c;
      const float av = r * load_param<DT>(gw, ch);
      ga[(long long)b * C + ch] = av;
      gs[(long long)b * C + ch] = fmaf(-mu, av, load_param<DT>(gb, ch));
    }
  }
}

}  // namespace

cudaError_t launch_gn_stats(const void *x, int B, int C, int N, int G, int dtype, const void *gw,
                            const void *gb, float *mean, float *rstd, float *a, float *s, int num_sms,
                            cudaStream_t st) {
  const int groups = B * G;
  const long long bytes = (long long)(C / G) * N * (dtype == 0 ? 4 : 2);
  int cs = 1;
  // Split a group over a cluster of up to 8 CTAs while the doubled grid still
  // fits one wave (clusters of 8 of these CTAs fit ~51 at a time, so a
  // larger grid leaves a partial second wave for this latency-bound pass).
  while (cs < 8 && (long long)groups * cs * 2 <= 2LL * num_sms && bytes / (2LL * cs) >= 16384) cs *= 2;
  // Elements of the group per cluster CTA, on multiples of 8.
  const long long L = (long long)(C / G) * N;
  const long long per = ((L + cs - 1) / cs + 7) / 8 * 8;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(cs, groups, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (dtype == 0)
    return cudaLaunchKernelEx(&cfg, gn_stats_kernel<0>, x, C, N, G, per, gw, gb, mean, rstd, a, s);
  return cudaLaunchKernelEx(&cfg, gn_stats_kernel<1>, x, C, N, G, per, gw, gb, mean, rstd, a, s);
}

}  // namespace ssa
