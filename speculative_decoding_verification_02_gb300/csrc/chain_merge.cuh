// Merging the streaming pass's per-(row, chunk) statistics into row
// statistics, and the one-warp inverse-CDF pick over a list of masses, for
// the accept kernels of chain.cu.
#pragma once

#include "common.cuh"

namespace sv {

__device__ __forceinline__ Partial ld_partial(const Partial *p) {
  const float4 v = __ldcg(reinterpret_cast<const float4 *>(p));
  return Partial{v.x, v.y, __float_as_int(v.z), v.w};
}

constexpr int kMergeUnroll = 4;  // partials per lane whose loads are issued together

// Merges with one warp the partials of row A and, if ppB is non-null, row B:
// max, sum 2^((x - max) c), first argmax, and the drafted token's logit
// (tokchunk = the chunk holding the token, or -1).  The loads of the first
// 32 * kMergeUnroll chunks of both rows are all issued before any is used.
struct MergedRow {
  float M, S, X;
  int A;
};

template <bool SOFTMAX>
__device__ __forceinline__ MergedRow merge_prefetched(const float4 *q, const Partial *pp, int nc, float c,
                                                     int tokchunk) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY, s = 0.0f, x = -INFINITY;
  int idx = kNoIndex;
#pragma unroll
  for (int u = 0; u < kMergeUnroll; ++u) {
    const int j = lane + 32 * u;
    if (j < nc) {
      if (SOFTMAX) merge_stats(m, s, idx, q[u].x, q[u].y, __float_as_int(q[u].z), c);
      else merge_argmax(m, idx, q[u].x, __float_as_int(q[u].z));
      if (j == tokchunk) x = q[u].w;
    }
  }
  for (int j = lane + 32 * kMergeUnroll; j < nc; j += 32) {  // very long rows only
    const Partial r = ld_partial(pp + j);
    if (SOFTMAX) merge_stats(m, s, idx, r.m, r.s, r.idx, c); else merge_argmax(m, idx, r.m, r.idx);
    if (j == tokchunk) x = r.x;
  }
  if (SOFTMAX) warp_merge_stats(m, s, idx, c); else warp_merge_argmax(m, idx);
  MergedRow out;
  out.M = m;
  out.S = s;
  out.A = idx == kNoIndex ? 0 : idx;  // an all -inf row: every index ties, take 0
  out.X = tokchunk >= 0 ? __shfl_sync(0xffffffffu, x, tokchunk & 31) : -INFINITY;
  return out;
}

template <bool SOFTMAX>
__device__ __forceinline__ void warp_merge_two_rows(const Partial *ppA, const Partial *ppB, int nc, float c,
                                                    int tokA, int tokB, MergedRow &a, MergedRow &b) {
  const int lane = threadIdx.x & 31;
  const float4 neutral = make_float4(-INFINITY, 0.0f, __int_as_float(kNoIndex), -INFINITY);
  float4 qa[kMergeUnroll], qb[kMergeUnroll];
#pragma unroll
  for (int u = 0; u < kMergeUnroll; ++u) {
    const int j = lane + 32 * u;
    qa[u] = j < nc ? __ldcg(reinterpret_cast<const float4 *>(ppA + j)) : neutral;
    qb[u] = (ppB != nullptr && j < nc) ? __ldcg(reinterpret_cast<const float4 *>(ppB + j)) : neutral;
  }
  a = merge_prefetched<SOFTMAX>(qa, ppA, nc, c, tokA);
  if (ppB != nullptr) b = merge_prefetched<SOFTMAX>(qb, ppB, nc, c, tokB);
}

// One warp: the index j* in [0, n) where u * (w_0 + ... + w_{n-1}) falls,
// i.e. the smallest j with w_0 + ... + w_j > u * total, and the threshold
// relative to the start of chunk j*.  If rounding leaves no such j, the last
// j with w_j > 0 and an infinite threshold (its last positive element).
// Lane l owns the contiguous range [l*cpl, (l+1)*cpl); each weight is read
// once (kept in `cache` when n <= cap).  All lanes return the same values;
// `total` is the sum of the weights.
template <class W>
__device__ __forceinline__ void warp_pick(W weight, int n, float u, float *cache, int cap, int &jsel,
                                          float &thr_local, float &total) {
  const int lane = threadIdx.x & 31;
  const int cpl = (n + 31) / 32;
  const int j0 = min(n, lane * cpl), j1 = min(n, j0 + cpl);
  const bool cached = n <= cap;
  float ls = 0.0f;
  int lastpos = -1;
  constexpr int kUnroll = 4;  // the first kUnroll weights' loads are issued together
  float wq[kUnroll];
#pragma unroll
  for (int q = 0; q < kUnroll; ++q) wq[q] = (j0 + q < j1) ? weight(j0 + q) : 0.0f;
#pragma unroll
  for (int q = 0; q < kUnroll; ++q) {
    const int j = j0 + q;
    if (j < j1) {
      if (cached) cache[j] = wq[q];
      ls += wq[q];
      if (wq[q] > 0.0f) lastpos = j;
    }
  }
  for (int j = j0 + kUnroll; j < j1; ++j) {
    const float w = weight(j);
    if (cached) cache[j] = w;
    ls += w;
    if (w > 0.0f) lastpos = j;
  }
  __syncwarp();
  const float incl = warp_inclusive_scan(ls, lane);
  total = __shfl_sync(0xffffffffu, incl, 31);
  const float thr = u * total;
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.0f;
  const unsigned cross = __ballot_sync(0xffffffffu, incl > thr);
  if (cross) {
    const int first = __ffs(cross) - 1;
    int pick = -1;
    float base = 0.0f;
    if (lane == first) {
      float run = excl;
      for (int j = j0; j < j1; ++j) {
        const float w = cached ? cache[j] : weight(j);
        if (run + w > thr) {
          pick = j;
          base = run;
          break;
        }
        run += w;
      }
      if (pick < 0) {  // rounding inside the lane: take its last chunk with mass
        pick = lastpos >= 0 ? lastpos : j0;
        base = thr;
      }
    }
    jsel = __shfl_sync(0xffffffffu, pick, first);
    base = __shfl_sync(0xffffffffu, base, first);
    thr_local = fmaxf(thr - base, 0.0f);
  } else {
    for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
    jsel = max(lastpos, 0);
    thr_local = INFINITY;
  }
}

}  // namespace sv
