// Pieces shared by the cluster kernels (tree walk, fused chain verify), in
// which each warp of a CTA owns one contiguous range of the CTA's
// vocabulary slice: warp reductions whose result lands in every lane,
// per-lane row statistics, and the inverse-CDF draw inside a slice from
// per-warp masses.
#pragma once

#include "common.cuh"

namespace sv {

// ------------------------------------------------ warp-wide reductions

// Order-preserving map of fp32 (NaN excluded) onto int32, so that one
// integer redux finds the largest float.
__device__ __forceinline__ int float_key(float x) {
  const int b = __float_as_int(x);
  return b >= 0 ? b : b ^ 0x7fffffff;
}
__device__ __forceinline__ float key_float(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

__device__ __forceinline__ float warp_allmax(float x) {
  return key_float(__reduce_max_sync(0xffffffffu, float_key(x)));
}

// Lowest index among the lanes whose m equals the warp's max M.
__device__ __forceinline__ int warp_first_index(float m, float M, int i) {
  return static_cast<int>(__reduce_min_sync(0xffffffffu, static_cast<unsigned>(m == M ? i : kNoIndex)));
}

// (m, s, i) of all lanes merged: the max, the sums rescaled to it and added,
// the first index of the max (IDX) -- one max, one exponential per lane.
template <bool IDX>
__device__ __forceinline__ void warp_allmerge(float &m, float &s, int &i, float c) {
  const float M = warp_allmax(m);
  const float r = M == -INFINITY ? 0.0f : s * ex2((m - M) * c);
  if (IDX) i = warp_first_index(m, M, i);
  s = warp_sum(r);
  m = M;
}

__device__ __forceinline__ void warp_allargmax(float &m, int &i) {
  const float M = warp_allmax(m);
  i = warp_first_index(m, M, i);
  m = M;
}

// Block-wide merge of every thread's (m, s, i) and of the max xt; the
// result is valid in warp 0.  SOFTMAX: (max, sum rescaled to it, first
// index of the max when IDX); otherwise (max, first index).
template <bool SOFTMAX, bool IDX, int NT>
__device__ __forceinline__ void block_allmerge(float &m, float &s, int &i, float c, float &xt) {
  constexpr int NW = NT / 32;
  __shared__ float sm[NW], ss[NW], sx[NW];
  __shared__ int si[NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (SOFTMAX) warp_allmerge<IDX>(m, s, i, c);
  else warp_allargmax(m, i);
  xt = warp_allmax(xt);
  if (lane == 0) {
    sm[warp] = m;
    ss[warp] = s;
    si[warp] = i;
    sx[warp] = xt;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < NW ? sm[lane] : -INFINITY;
    s = lane < NW ? ss[lane] : 0.0f;
    i = lane < NW ? si[lane] : kNoIndex;
    xt = lane < NW ? sx[lane] : -INFINITY;
    if (SOFTMAX) warp_allmerge<IDX>(m, s, i, c);
    else warp_allargmax(m, i);
    xt = warp_allmax(xt);
  }
}

// ------------------------------------------------------ per-lane work

// Running statistics of one row over a lane's groups.
struct RowStats {
  float m;   // max logit
  float2 s;  // sum of 2^((x - m) c), two lanes
  int i;     // first index of the max
};

__device__ __forceinline__ RowStats row_stats_empty() {
  return RowStats{-INFINITY, make_float2(0.0f, 0.0f), kNoIndex};
}

template <bool SOFTMAX>
__device__ __forceinline__ void fold_one(RowStats &R, float x, int v, float c) {
  if (x > R.m) {
    if (SOFTMAX) {
      const float f = ex2((R.m - x) * c);
      R.s.x *= f;
      R.s.y *= f;
    }
    R.m = x;
    R.i = v;
  }
  if (SOFTMAX && R.m != -INFINITY) R.s.x += ex2((x - R.m) * c);
}

// Work split of a CTA's slice [lo, hi): 16-byte groups of EPG logits, group
// g holding logits lo + g EPG ...; lane l of warp w takes the groups
//     g = (w G + j) 32 + l,   j < G,
// so that each warp load instruction reads 32 consecutive groups (512
// bytes) and each warp covers one contiguous range of 32 G groups.
__device__ __forceinline__ int lane_group(int warp, int j, int G, int lane) { return ((warp * G + j) << 5) + lane; }

// The 16-byte group of `row` starting at logit e; logits >= hi read as
// -inf.  VEC: the row is 16-byte aligned and hi a multiple of the group
// size, so a group is wholly inside [.., hi) or wholly outside, and a group
// inside is one 16-byte load.
template <int DT, bool VEC>
__device__ __forceinline__ uint4 load_group(const char *row, int e, int hi) {
  constexpr uint32_t kNegInf = DT == SPEC_DTYPE_F32 ? 0xff800000u : 0xff80ff80u;  // -inf words
  if constexpr (VEC) {
    return e < hi ? __ldg(reinterpret_cast<const uint4 *>(row + static_cast<int64_t>(e) * Elems<DT>::kSize))
                  : make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (DT == SPEC_DTYPE_F32) {
        w[q] = e + q < hi ? __float_as_uint(load_one<DT>(row, e + q)) : kNegInf;
      } else {
        const uint32_t l = e + 2 * q < hi ? __float_as_uint(load_one<DT>(row, e + 2 * q)) >> 16 : 0xff80u;
        const uint32_t h = e + 2 * q + 1 < hi ? __float_as_uint(load_one<DT>(row, e + 2 * q + 1)) >> 16 : 0xff80u;
        w[q] = l | (h << 16);
      }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Max of the logits of the first n (<= kBatch) of the groups g.
template <int DT>
__device__ __forceinline__ float groups_max(const uint4 *g, int n) {
  if (DT == SPEC_DTYPE_BF16) {
    auto h2 = [](uint32_t w) { return *reinterpret_cast<const __nv_bfloat162 *>(&w); };
    __nv_bfloat162 a = __hmax2(h2(g[0].x), h2(g[0].y)), b = __hmax2(h2(g[0].z), h2(g[0].w));
#pragma unroll
    for (int u = 1; u < kBatch; ++u) {
      if (u < n) {
        a = __hmax2(a, __hmax2(h2(g[u].x), h2(g[u].y)));
        b = __hmax2(b, __hmax2(h2(g[u].z), h2(g[u].w)));
      }
    }
    const __nv_bfloat162 mx = __hmax2(a, b);
    return fmaxf(__low2float(mx), __high2float(mx));
  }
  float a = fmaxf(__uint_as_float(g[0].x), __uint_as_float(g[0].y));
  float b = fmaxf(__uint_as_float(g[0].z), __uint_as_float(g[0].w));
#pragma unroll
  for (int u = 1; u < kBatch; ++u) {
    if (u < n) {
      a = fmaxf(a, fmaxf(__uint_as_float(g[u].x), __uint_as_float(g[u].y)));
      b = fmaxf(b, fmaxf(__uint_as_float(g[u].z), __uint_as_float(g[u].w)));
    }
  }
  return fmaxf(a, b);
}

// Adds 2^((x - m) c) over the logits of the first n groups into acc (one
// packed subtract and one packed multiply per two logits, one exponential
// per logit, one packed add per two; consecutive groups alternate between
// two accumulators).
template <int DT>
__device__ __forceinline__ void groups_sumexp(const uint4 *g, int n, float c, float m, float2 &acc) {
  const float2 cc = make_float2(c, c), nm = make_float2(-m, -m);
  float2 acc2 = make_float2(0.0f, 0.0f);
  auto fold = [&](float2 &A, float a, float b) {
    const float2 z = __fmul2_rn(__fadd2_rn(make_float2(a, b), nm), cc);
    A = __fadd2_rn(A, make_float2(ex2(z.x), ex2(z.y)));
  };
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    if (u < n) {
      float2 &A = (u & 1) ? acc2 : acc;
      if (DT == SPEC_DTYPE_BF16) {
        fold(A, bf16_lo(g[u].x), bf16_hi(g[u].x));
        fold(A, bf16_lo(g[u].y), bf16_hi(g[u].y));
        fold(A, bf16_lo(g[u].z), bf16_hi(g[u].z));
        fold(A, bf16_lo(g[u].w), bf16_hi(g[u].w));
      } else {
        fold(A, __uint_as_float(g[u].x), __uint_as_float(g[u].y));
        fold(A, __uint_as_float(g[u].z), __uint_as_float(g[u].w));
      }
    }
  }
  acc = __fadd2_rn(acc, acc2);
}

// First logit equal to bm among the first n groups, group u starting at
// logit e0 + u * span; kNoIndex if none.
template <int DT>
__device__ __forceinline__ int groups_first(const uint4 *g, int n, float bm, int e0, int span) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  int first = kNoIndex;
#pragma unroll
  for (int u = kBatch - 1; u >= 0; --u) {
    if (u < n) {
      float x[EPG];
      unpack16<DT>(g[u], x);
#pragma unroll
      for (int e = EPG - 1; e >= 0; --e)
        if (x[e] == bm) first = e0 + u * span + e;
    }
  }
  return first;
}

// Folds this lane's groups (the lane_group split, G rounds) of NR rows into
// R[r]; a null rows[r] is skipped.  kBatch rounds of every row are loaded
// before any of them is folded.  SOFTMAX: the running max and the sum of
// 2^((x - max) c), rescaled once per batch when the batch raises the max
// (R[r].i is not kept); otherwise the running max and its first index.
template <int DT, bool SOFTMAX, bool VEC, int NR>
__device__ __forceinline__ void lane_rows_stats(const char *const *rows, int lo, int hi, int G, float c,
                                                RowStats *R) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  constexpr uint32_t kNegInf = DT == SPEC_DTYPE_F32 ? 0xff800000u : 0xff80ff80u;  // -inf words
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int j0 = 0; j0 < G; j0 += kBatch) {
    const int n = min(kBatch, G - j0);                        // rounds in this batch
    const int e0 = lo + lane_group(warp, j0, G, lane) * EPG;  // round j0 + u starts at e0 + u 32 EPG
    uint4 x[NR][kBatch];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        x[r][u] = (rows[r] && u < n) ? load_group<DT, VEC>(rows[r], e0 + u * 32 * EPG, hi)
                                     : make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      if (!rows[r]) continue;
      const float bm = groups_max<DT>(x[r], n);
      if (SOFTMAX) {
        if (bm > R[r].m) {
          if (R[r].m != -INFINITY) {
            const float f = ex2((R[r].m - bm) * c);
            R[r].s.x *= f;
            R[r].s.y *= f;
          }
          R[r].m = bm;
        }
        if (R[r].m != -INFINITY) groups_sumexp<DT>(x[r], n, c, R[r].m, R[r].s);
      } else if (bm > R[r].m) {
        R[r].m = bm;
        R[r].i = groups_first<DT>(x[r], n, bm, e0, 32 * EPG);
      }
    }
  }
}

// One warp walks the range of warp `wsel` of a slice (the lane_group split,
// G rounds of 32 groups), 32 groups at a time, for the first weight whose
// running sum over the range passes thr.  Returns its offset from the
// slice start, the same in every lane; when rounding leaves no crossing,
// the range's last positive weight; -1 when the range has none.
// group_weights(g, w) writes the EPG weights of group g.
template <int EPG, class GroupWeights>
__device__ __forceinline__ int warp_walk_range(int wsel, int G, float thr, GroupWeights &&group_weights) {
  const int lane = threadIdx.x & 31;
  int pick = -1, lastp = -1;
  float run = 0.0f;
  for (int j = 0; j < G; ++j) {
    const int g = lane_group(wsel, j, G, lane);
    float w[EPG];
    group_weights(g, w);
    float lm = 0.0f;
    int le = -1;  // this lane's last positive weight
#pragma unroll
    for (int e = 0; e < EPG; ++e) {
      lm += w[e];
      if (w[e] > 0.0f) le = e;
    }
    const float incl = warp_inclusive_scan(lm, lane);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.0f;
    const unsigned hit = __ballot_sync(0xffffffffu, lm > 0.0f && run + incl > thr);
    const unsigned pos = __ballot_sync(0xffffffffu, lm > 0.0f);
    if (pos) {
      const int hl = 31 - __clz(pos);
      lastp = (g - lane + hl) * EPG + __shfl_sync(0xffffffffu, le, hl);
    }
    if (hit) {
      const int lh = __ffs(hit) - 1;
      int pe = le;  // rounding inside the lane: its last positive weight
      float r = run + excl;
#pragma unroll
      for (int e = 0; e < EPG; ++e) {
        r += w[e];
        if (w[e] > 0.0f && r > thr) {
          pe = e;
          break;
        }
      }
      pick = (g - lane + lh) * EPG + __shfl_sync(0xffffffffu, pe, lh);
      break;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  return pick >= 0 ? pick : lastp;
}

// This lane's sum of the draw weights W over its groups (lane_group split
// of [lo, hi), G rounds; logits >= hi weigh 0).  With gsum, each group's
// own sum goes to gsum[g].
template <int DT, bool VEC, bool FILT>
__device__ __forceinline__ float lane_weight_sum(const Weights &W, int lo, int hi, int G, float *gsum) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc = 0.0f;
  for (int j0 = 0; j0 < G; j0 += kBatch) {
    const int g0 = lane_group(warp, j0, G, lane);  // round j0 + u: group g0 + 32 u
    uint4 xa[kBatch], xb[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (j0 + u < G) {
        xa[u] = load_group<DT, VEC>(W.a, lo + (g0 + 32 * u) * EPG, hi);
        if (W.b) xb[u] = load_group<DT, VEC>(W.b, lo + (g0 + 32 * u) * EPG, hi);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (j0 + u < G) {
        float x[EPG], y[EPG], w[EPG];
        unpack16<DT>(xa[u], x);
        if (W.b) unpack16<DT>(xb[u], y);
        weights_group<EPG, FILT>(W, x, y, w);
        float gs = 0.0f;
#pragma unroll
        for (int e = 0; e < EPG; ++e) gs += w[e];
        if (gsum != nullptr) gsum[g0 + 32 * u] = gs;
        acc += gs;
      }
    }
  }
  return acc;
}

// Inverse-CDF draw inside one CTA's slice [lo, hi) from per-warp masses
// (the lane_group split).  `wmass` is the calling warp's sum of weights
// (the same in all its lanes); the drawn logit is the first whose running
// sum over the slice passes tl (tl = INFINITY: the last positive weight).
// A scan of the warp masses finds the warp whose range holds the crossing.
// With gsum (gsum[g] = the weight sum of group g, in the same summation
// order as group_weights), that warp finds the group by one lane scan over
// its range's group sums (lane l taking G consecutive groups of the range)
// and reads only that group; without, it walks its range 32 groups at a
// time.  group_weights(g, w) writes the EPG weights of group g (0 for
// logits >= hi).  Rounding between the scans falls back to the last
// positive weight of the last warp with mass; `fallback` is returned when
// no warp has any.  Called by all NT threads.  BCAST: returns the token in
// every thread.  Otherwise (no barrier after the warp scan) it returns the
// token in every lane of one warp -- the drawing warp, or warp 0 when no
// warp has mass -- and -1 in all other threads.  wsums (or null): the NW
// warp masses already in shared memory and visible to every thread, which
// saves publishing them again.
template <int NT, int EPG, bool BCAST = true, class GroupWeights>
__device__ int range_draw(float wmass, float tl, int lo, int G, int fallback, const float *gsum,
                          GroupWeights &&group_weights, const float *wsums = nullptr) {
  constexpr int NW = NT / 32;
  __shared__ float s_wsum[NW];
  __shared__ int s_tok;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (wsums == nullptr) {
    if (lane == 0) s_wsum[warp] = wmass;
    __syncthreads();
    wsums = s_wsum;
  }
  const float wv = lane < NW ? wsums[lane] : 0.0f;
  const float winc = warp_inclusive_scan(wv, lane);
  const unsigned hit_w = __ballot_sync(0xffffffffu, wv > 0.0f && winc > tl);
  const unsigned pos_w = __ballot_sync(0xffffffffu, wv > 0.0f);
  int wsel = -1;
  float thr_local = INFINITY;
  if (hit_w) {
    wsel = __ffs(hit_w) - 1;
    const float before = __shfl_sync(0xffffffffu, winc, max(wsel - 1, 0));
    thr_local = tl - (wsel > 0 ? before : 0.0f);
  } else if (pos_w) {  // rounding: the last warp with mass, its last positive weight
    wsel = 31 - __clz(pos_w);
  }
  if (warp == wsel) {
    int pick = -1;
    // the crossing within group g, given the running sum `run` before it
    auto scan_group = [&](int g, float run, bool cross) {
      float w[EPG];
      group_weights(g, w);
      int pe = -1, le = -1;
#pragma unroll
      for (int e = 0; e < EPG; ++e) {
        run += w[e];
        if (w[e] > 0.0f) {
          le = e;
          if (cross && pe < 0 && run > thr_local) pe = e;
        }
      }
      if (pe < 0) pe = le;  // rounding inside the group: its last positive weight
      return pe < 0 ? -1 : g * EPG + pe;
    };
    if (gsum != nullptr) {
      const int g0 = wsel * 32 * G;  // the range's first group
      float ls = 0.0f;
      for (int t = 0; t < G; ++t) ls += gsum[g0 + lane * G + t];
      const float incl = warp_inclusive_scan(ls, lane);
      float excl = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) excl = 0.0f;
      const unsigned hit = __ballot_sync(0xffffffffu, ls > 0.0f && incl > thr_local);
      const unsigned pos = __ballot_sync(0xffffffffu, ls > 0.0f);
      const int lh = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
      if (lh >= 0 && lane == lh) {  // this lane's G groups hold the crossing (or the last mass)
        float run = excl;
        int gsel = -1, glast = -1;
        float base = excl, blast = excl;
        for (int t = 0; t < G; ++t) {
          const float gs = gsum[g0 + lane * G + t];
          if (gs > 0.0f) {
            glast = g0 + lane * G + t;
            blast = run;
            if (hit && gsel < 0 && run + gs > thr_local) {
              gsel = glast;
              base = run;
            }
          }
          run += gs;
        }
        if (gsel < 0) {
          gsel = glast;
          base = blast;
        }
        pick = scan_group(gsel, base, hit != 0u);
      }
      if (lh >= 0) pick = __shfl_sync(0xffffffffu, pick, lh);
    } else {
      pick = warp_walk_range<EPG>(wsel, G, thr_local, group_weights);
    }
    if (!BCAST) return pick >= 0 ? lo + pick : fallback;  // (pick is the same in every lane)
    if (lane == 0) s_tok = pick >= 0 ? lo + pick : fallback;
  } else if (wsel < 0 && threadIdx.x == 0) {
    s_tok = fallback;  // no positive weight in the slice (underflow only)
  }
  if (!BCAST) return wsel < 0 && warp == 0 ? fallback : -1;
  __syncthreads();
  const int r = s_tok;
  __syncthreads();  // the shared words are free again
  return r;
}

}  // namespace sv
