// Device helpers shared by the verification kernels (sm_103a).
//
// Numerics: logits are widened exactly to fp32 (bf16 is the top half of an
// fp32); every exponential is 2^((x - M) * c) with c = log2(e) / T, computed
// by the hardware ex2.approx unit; sums accumulate in fp32.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "spec_verify.h"

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kNoIndex = 0x7fffffff;

// Per-(row, chunk) statistics written by the streaming pass:
// m = max logit, s = sum 2^((x - m) * c) over the chunk, idx = first argmax,
// x = the logit of the row's drafted token when it falls in this chunk.
struct __align__(16) Partial {
  float m;
  float s;
  int idx;
  float x;
};

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and (in that kernel) wait until this grid has finished and its
// writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Split cluster barrier: arrive once this CTA has finished reading other
// CTAs' shared memory, wait just before exiting, so that no CTA leaves while
// another may still read from it -- without stalling at the end.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- loads

// 16-byte asynchronous copy global -> shared (L2 only), and its group
// commit / wait (hardware waits: the thread's own copies of all but the N
// most recent groups have landed).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 16-byte streaming load that does not allocate in L1 (rows are read once).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Element v of a row, widened to fp32.
template <int DT>
__device__ __forceinline__ float load_one(const char *row, int64_t v) {
  if (DT == SPEC_DTYPE_F32) return __ldg(reinterpret_cast<const float *>(row) + v);
  const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(row) + v);
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Unpack one 16-byte group: 8 bf16 or 4 fp32 values.
template <int DT>
__device__ __forceinline__ void unpack16(const uint4 &g, float *x) {
  if (DT == SPEC_DTYPE_F32) {
    x[0] = __uint_as_float(g.x);
    x[1] = __uint_as_float(g.y);
    x[2] = __uint_as_float(g.z);
    x[3] = __uint_as_float(g.w);
  } else {
    x[0] = bf16_lo(g.x); x[1] = bf16_hi(g.x);
    x[2] = bf16_lo(g.y); x[3] = bf16_hi(g.y);
    x[4] = bf16_lo(g.z); x[5] = bf16_hi(g.z);
    x[6] = bf16_lo(g.w); x[7] = bf16_hi(g.w);
  }
}

template <int DT>
struct Elems {
  static constexpr int kSize = DT == SPEC_DTYPE_F32 ? 4 : 2;  // bytes per logit
  static constexpr int kPerGroup = 16 / kSize;                // logits per 16-byte group
};

// ------------------------------------------------------------- arithmetic

// 2^x on the special-function unit (x = -inf gives +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Merge (m2, s2, i2) into (m, s, i): the running max, the sum rescaled to the
// new max, and the first index of the max (ties keep the lower index).
__device__ __forceinline__ void merge_stats(float &m, float &s, int &i, float m2, float s2, int i2,
                                            float c) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) {
    s = 0.0f;
  } else {
    s = s * ex2((m - M) * c) + s2 * ex2((m2 - M) * c);
  }
  i = (m > m2) ? i : (m2 > m) ? i2 : min(i, i2);
  m = M;
}

__device__ __forceinline__ void merge_argmax(float &m, int &i, float m2, int i2) {
  i = (m > m2) ? i : (m2 > m) ? i2 : min(i, i2);
  m = fmaxf(m, m2);
}

__device__ __forceinline__ void warp_merge_stats(float &m, float &s, int &i, float c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    merge_stats(m, s, i, m2, s2, i2, c);
  }
}

__device__ __forceinline__ void warp_merge_argmax(float &m, int &i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    merge_argmax(m, i, m2, i2);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_inclusive_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// --------------------------------------------------- weighted row selection

// Weight of element v in an inverse-CDF draw over one row (a) or a row pair
// (a, b):  w_v = max(0, alpha * 2^((a_v - Ma) c) [a_v >= ta] - beta * 2^((b_v
// - Mb) c) [b_v >= tb]).  beta = 0 (and b = nullptr) draws from the row's own
// softmax; ta, tb are the rows' top-k / top-p thresholds (-inf: unfiltered).
struct Weights {
  const char *a;
  const char *b;
  float Ma, Mb, alpha, beta, c;
  float ta, tb;
};

// The weights of two elements (a, b: their logits in the two rows), in
// packed f32x2 arithmetic: one instruction subtracts, scales or combines
// both, so a residual weight costs about nine instructions instead of
// twelve (the scans of these weights are bound by instruction issue, not by
// the exponentials).  FILT = false compiles the thresholds out (the masks
// cost a compare and a select per logit).  Every sum and scan of the
// weights, single elements included (weight_at), goes through this
// function, so they agree bit for bit.
template <bool FILT>
__device__ __forceinline__ float2 weight_pair(const Weights &W, float2 a, float2 b) {
  const float2 cc = make_float2(W.c, W.c);
  const float2 za = __fmul2_rn(__fadd2_rn(a, make_float2(-W.Ma, -W.Ma)), cc);
  float2 w = __fmul2_rn(make_float2(ex2(za.x), ex2(za.y)), make_float2(W.alpha, W.alpha));
  if (FILT) {
    if (!(a.x >= W.ta)) w.x = 0.0f;
    if (!(a.y >= W.ta)) w.y = 0.0f;
  }
  if (W.b != nullptr) {
    const float2 zb = __fmul2_rn(__fadd2_rn(b, make_float2(-W.Mb, -W.Mb)), cc);
    float2 q = make_float2(ex2(zb.x), ex2(zb.y));
    if (FILT) {
      if (!(b.x >= W.tb)) q.x = 0.0f;
      if (!(b.y >= W.tb)) q.y = 0.0f;
    }
    w = __ffma2_rn(make_float2(-W.beta, -W.beta), q, w);
  }
  return make_float2(fmaxf(w.x, 0.0f), fmaxf(w.y, 0.0f));
}

template <int DT, bool FILT = true>
__device__ __forceinline__ float weight_at(const Weights &W, float a, float b) {
  return weight_pair<FILT>(W, make_float2(a, a), make_float2(b, b)).x;
}

// The weights of EPG consecutive elements (a, b: their logits; EPG even).
template <int EPG, bool FILT = true>
__device__ __forceinline__ void weights_group(const Weights &W, const float *a, const float *b, float *w) {
#pragma unroll
  for (int e = 0; e < EPG; e += 2) {
    const float2 r = weight_pair<FILT>(W, make_float2(a[e], a[e + 1]), make_float2(b[e], b[e + 1]));
    w[e] = r.x;
    w[e + 1] = r.y;
  }
}

// True when either row of W has a top-k / top-p threshold.
__device__ __forceinline__ bool weights_filtered(const Weights &W) { return W.ta > -INFINITY || W.tb > -INFINITY; }

// A row's filter threshold (the smallest kept logit), -inf when unfiltered.
__device__ __forceinline__ float row_theta(const float *theta, int64_t row) {
  return theta ? __ldcg(theta + row) : -INFINITY;
}

// The eight weights of elements [v0, v0 + 8) (those >= hi are 0).
template <int DT, bool VEC>
__device__ __forceinline__ void weights8(const Weights &W, int v0, int hi, float *w) {
  float a[8], b[8];
  if (VEC && v0 + 8 <= hi) {
    if (DT == SPEC_DTYPE_F32) {
      unpack16<DT>(*reinterpret_cast<const uint4 *>(W.a + static_cast<int64_t>(v0) * 4), a);
      unpack16<DT>(*reinterpret_cast<const uint4 *>(W.a + static_cast<int64_t>(v0) * 4 + 16), a + 4);
      if (W.b != nullptr) {
        unpack16<DT>(*reinterpret_cast<const uint4 *>(W.b + static_cast<int64_t>(v0) * 4), b);
        unpack16<DT>(*reinterpret_cast<const uint4 *>(W.b + static_cast<int64_t>(v0) * 4 + 16), b + 4);
      }
    } else {
      unpack16<DT>(*reinterpret_cast<const uint4 *>(W.a + static_cast<int64_t>(v0) * 2), a);
      if (W.b != nullptr)
        unpack16<DT>(*reinterpret_cast<const uint4 *>(W.b + static_cast<int64_t>(v0) * 2), b);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const bool in = v0 + e < hi;
      a[e] = in ? load_one<DT>(W.a, v0 + e) : -INFINITY;
      b[e] = (in && W.b != nullptr) ? load_one<DT>(W.b, v0 + e) : -INFINITY;
    }
  }
  weights_group<8>(W, a, b, w);
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (v0 + e >= hi) w[e] = 0.0f;
}

// Block-wide inverse-CDF selection inside [lo, hi): the smallest v with
// (sum of w over [lo, v]) > thr.  If rounding leaves no such v, the last v in
// the range with w > 0 (or -1 when every weight is 0).  lo must be a
// multiple of 8.  Each thread takes a contiguous segment of kSelPerThread
// elements (all its loads in flight at once), the block scans the segment
// sums, and every thread whose prefix passes thr walks its own segment; the
// smallest proposal wins.  Called by all NT threads; returns the same
// value in every thread.
constexpr int kSelPerThread = 32;

// fill8(v0, hi, w) writes the weights of elements [v0, v0 + 8) into w (0 for
// elements >= hi).
template <int NT = kThreads, class Fill8>
__device__ int block_select_with(Fill8 &&fill8, int lo, int hi, float thr) {
  constexpr int NW = NT / 32;
  __shared__ float s_wsum[NW];
  __shared__ int s_pick, s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    s_pick = kNoIndex;
    s_last = -1;
  }
  float carry = 0.0f;
  int last_pos = -1;
  for (int base = lo; base < hi; base += NT * kSelPerThread) {
    const int v0 = base + threadIdx.x * kSelPerThread;
    float w[kSelPerThread];
#pragma unroll
    for (int q = 0; q < kSelPerThread / 8; ++q) fill8(v0 + 8 * q, hi, w + 8 * q);
    float ls = 0.0f;
#pragma unroll
    for (int e = 0; e < kSelPerThread; ++e) {
      ls += w[e];
      if (w[e] > 0.0f) last_pos = v0 + e;
    }
    const float incl = warp_inclusive_scan(ls, lane);
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    float wbase = carry, total = carry;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      if (i < warp) wbase += s_wsum[i];
      total += s_wsum[i];
    }
    if (wbase + incl > thr) {
      float run = wbase + incl - ls;
      int pick = -1, lastp = -1;
#pragma unroll
      for (int e = 0; e < kSelPerThread; ++e) {
        run += w[e];
        if (w[e] > 0.0f) lastp = v0 + e;
        if (pick < 0 && run > thr) pick = v0 + e;
      }
      if (pick < 0) pick = lastp;
      if (pick >= 0) atomicMin(&s_pick, pick);
    }
    __syncthreads();
    const bool done = s_pick != kNoIndex;
    carry = total;
    __syncthreads();
    if (done) break;
  }
  for (int o = 16; o > 0; o >>= 1) last_pos = max(last_pos, __shfl_xor_sync(0xffffffffu, last_pos, o));
  if (lane == 0) atomicMax(&s_last, last_pos);
  __syncthreads();
  const int r = s_pick != kNoIndex ? s_pick : s_last;
  __syncthreads();
  return r;
}

template <int DT, bool VEC, int NT = kThreads>
__device__ int block_select(const Weights &W, int lo, int hi, float thr) {
  return block_select_with<NT>([&](int v0, int h, float *w) { weights8<DT, VEC>(W, v0, h, w); }, lo, hi, thr);
}

// ------------------------------------------------------------ streaming

constexpr int kBatch = 4;  // 16-byte groups each thread keeps in flight

// Load flavours: a row streamed once (no L1 allocation), a row re-read from
// L2 by another CTA, a row re-read by the same CTA (L1 allocation).
enum : int { kLoadStream = 0, kLoadL2 = 1, kLoadCached = 2 };

template <int LD>
__device__ __forceinline__ uint4 load16(const uint4 *p) {
  if (LD == kLoadStream) return ld_stream16(p);
  if (LD == kLoadL2) return __ldcg(p);
  return __ldg(p);
}

// Statistics of row[v0, v1) for the calling thread (strided over the block).
// Maximum of the logits of one batch of kBatch 16-byte groups: bf16 pairs
// are compared two at a time.
template <int DT>
__device__ __forceinline__ float batch_max(const uint4 *g) {
  if (DT == SPEC_DTYPE_BF16) {
    auto h2 = [](uint32_t w) { return *reinterpret_cast<const __nv_bfloat162 *>(&w); };
    __nv_bfloat162 mx = h2(g[0].x);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (u) mx = __hmax2(mx, h2(g[u].x));
      mx = __hmax2(mx, h2(g[u].y));
      mx = __hmax2(mx, h2(g[u].z));
      mx = __hmax2(mx, h2(g[u].w));
    }
    return fmaxf(__low2float(mx), __high2float(mx));
  }
  float bm = -INFINITY;
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    bm = fmaxf(bm, fmaxf(fmaxf(__uint_as_float(g[u].x), __uint_as_float(g[u].y)),
                         fmaxf(__uint_as_float(g[u].z), __uint_as_float(g[u].w))));
  }
  return bm;
}

// Adds 2^((x - m) c) over the batch into the two-lane accumulator: one
// packed subtract and one packed multiply per two logits (x - m first, so a
// large |m c| adds no rounding offset to every exponent), one ex2 per logit,
// one packed add per two.
template <int DT>
__device__ __forceinline__ void batch_sumexp(const uint4 *g, float c, float m, float2 &acc) {
  const float2 cc = make_float2(c, c), nm = make_float2(-m, -m);
  auto fold = [&](float a, float b) {
    const float2 z = __fmul2_rn(__fadd2_rn(make_float2(a, b), nm), cc);
    acc = __fadd2_rn(acc, make_float2(ex2(z.x), ex2(z.y)));
  };
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    if (DT == SPEC_DTYPE_BF16) {
      fold(bf16_lo(g[u].x), bf16_hi(g[u].x));
      fold(bf16_lo(g[u].y), bf16_hi(g[u].y));
      fold(bf16_lo(g[u].z), bf16_hi(g[u].z));
      fold(bf16_lo(g[u].w), bf16_hi(g[u].w));
    } else {
      fold(__uint_as_float(g[u].x), __uint_as_float(g[u].y));
      fold(__uint_as_float(g[u].z), __uint_as_float(g[u].w));
    }
  }
}

// The logit at offset `off` (< 16 bytes' worth of logits) within group g.
template <int DT>
__device__ __forceinline__ float group_logit(const uint4 &g, unsigned off) {
  const unsigned wi = DT == SPEC_DTYPE_BF16 ? off >> 1 : off;
  const uint32_t w = wi == 0 ? g.x : wi == 1 ? g.y : wi == 2 ? g.z : g.w;
  if (DT == SPEC_DTYPE_F32) return __uint_as_float(w);
  return (off & 1) ? bf16_hi(w) : bf16_lo(w);
}

// Folds one batch into the running (m, two-lane sum, idx), and picks up the
// logit at index `tok` (-1: none) into xt.  The batch's groups start at
// logits first_elem + u * NT * EPG, u < kBatch.  IDX = false leaves idx
// alone (no first-index search when the batch raises the max).
template <int DT, bool SOFTMAX, int NT = kThreads, bool IDX = true>
__device__ __forceinline__ void fold_batch(const uint4 *g, int first_elem, float c, float &m, float2 &s2,
                                           int &idx, int tok, float &xt) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  constexpr int kSpan = NT * EPG;  // logits between a thread's consecutive groups
  static_assert((kSpan & (kSpan - 1)) == 0, "group spacing must be a power of two");
  // does the drafted token fall in one of this batch's groups?  (rare)
  const unsigned d = static_cast<unsigned>(tok - first_elem);
  if (d < static_cast<unsigned>(kBatch * kSpan) && (d & (kSpan - 1)) < static_cast<unsigned>(EPG)) {
    const unsigned u = d / kSpan, off = d & (kSpan - 1);
#pragma unroll
    for (int q = 0; q < kBatch; ++q)
      if (q == static_cast<int>(u)) xt = group_logit<DT>(g[q], off);
  }
  const float bm = batch_max<DT>(g);
  if (bm > m) {  // a new running max: rescale the sum, find its first index
    if (SOFTMAX) {
      const float f = ex2((m - bm) * c);
      s2.x *= f;
      s2.y *= f;
    }
    m = bm;
    if (IDX) {
      int first = kNoIndex;
#pragma unroll
      for (int u = kBatch - 1; u >= 0; --u) {
        float x[EPG];
        unpack16<DT>(g[u], x);
#pragma unroll
        for (int e = EPG - 1; e >= 0; --e)
          if (x[e] == bm) first = first_elem + u * kSpan + e;
      }
      idx = first;
    }
  }
  if (SOFTMAX && m != -INFINITY) batch_sumexp<DT>(g, c, m, s2);
}

// Statistics of row[v0, v1) for the calling thread (strided over the block):
// running max m, sum of 2^((x - m) c), first index of the max, and the logit
// at index `tok` if this thread reads it (xt, else left as is; tok = -1 for
// none).  Full batches are loaded without predicates at fixed offsets from a
// pointer that advances by one batch stride; two batches are in flight
// (ping-pong), the last, partial batch is loaded with bounds checks.
template <int DT, bool SOFTMAX, bool VEC, int LD, int NT = kThreads, bool IDX = true>
__device__ __forceinline__ void thread_chunk_stats(const char *row, int v0, int v1, float c,
                                                   float &m, float &s, int &idx, int tok, float &xt) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  constexpr int ES = Elems<DT>::kSize;
  constexpr uint32_t kNegInf = DT == SPEC_DTYPE_F32 ? 0xff800000u : 0xff80ff80u;  // -inf words
  constexpr int kStride = NT * kBatch;
  int vtail = v0;
  float2 s2 = make_float2(s, 0.0f);
  if (VEC) {
    const int ng = (v1 - v0) / EPG;
    const uint4 *p = reinterpret_cast<const uint4 *>(row + static_cast<int64_t>(v0) * ES) + threadIdx.x;
    // this thread's groups: threadIdx.x + i * NT, i < mine
    const int mine = ng > static_cast<int>(threadIdx.x) ? (ng - 1 - static_cast<int>(threadIdx.x)) / NT + 1 : 0;
    const int nfull = mine / kBatch;  // batches whose kBatch groups all exist
    int e0 = v0 + static_cast<int>(threadIdx.x) * EPG;  // first logit of the current batch
    auto load_batch = [&](uint4 *g, const uint4 *q) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u) g[u] = load16<LD>(q + u * NT);
    };
    uint4 ga[kBatch], gb[kBatch];
    int i = 0;
    if (nfull > 0) load_batch(ga, p);
    for (; i + 2 <= nfull; i += 2) {
      load_batch(gb, p + kStride);
      fold_batch<DT, SOFTMAX, NT, IDX>(ga, e0, c, m, s2, idx, tok, xt);
      e0 += kStride * EPG;
      if (i + 2 < nfull) load_batch(ga, p + 2 * kStride);
      fold_batch<DT, SOFTMAX, NT, IDX>(gb, e0, c, m, s2, idx, tok, xt);
      e0 += kStride * EPG;
      p += 2 * kStride;
    }
    if (i < nfull) {  // an odd full batch is already in ga
      fold_batch<DT, SOFTMAX, NT, IDX>(ga, e0, c, m, s2, idx, tok, xt);
      e0 += kStride * EPG;
      p += kStride;
      ++i;
    }
    const int rest = mine - nfull * kBatch;  // groups of a last, partial batch
    if (rest > 0) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        ga[u] = u < rest ? load16<LD>(p + u * NT) : make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
      fold_batch<DT, SOFTMAX, NT, IDX>(ga, e0, c, m, s2, idx, tok, xt);
    }
    vtail = v0 + ng * EPG;
  }
  s = s2.x + s2.y;
  for (int v = vtail + threadIdx.x; v < v1; v += NT) {
    const float x = load_one<DT>(row, v);
    if (v == tok) xt = x;
    if (x > m) {
      if (SOFTMAX) s *= ex2((m - x) * c);
      m = x;
      if (IDX) idx = v;
    }
    if (SOFTMAX && m != -INFINITY) s += ex2((x - m) * c);
  }
}

// Block-wide merge; the result is valid in thread 0.
template <bool SOFTMAX, int NT = kThreads>
__device__ __forceinline__ void block_merge(float &m, float &s, int &idx, float c, float &xt) {
  constexpr int NW = NT / 32;
  __shared__ float sm[NW], ss[NW], sx[NW];
  __shared__ int si[NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (SOFTMAX) warp_merge_stats(m, s, idx, c); else warp_merge_argmax(m, idx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) xt = fmaxf(xt, __shfl_xor_sync(0xffffffffu, xt, o));
  if (lane == 0) {
    sm[warp] = m;
    ss[warp] = s;
    si[warp] = idx;
    sx[warp] = xt;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < NW ? sm[lane] : -INFINITY;
    s = lane < NW ? ss[lane] : 0.0f;
    idx = lane < NW ? si[lane] : kNoIndex;
    xt = lane < NW ? sx[lane] : -INFINITY;
    if (SOFTMAX) warp_merge_stats(m, s, idx, c); else warp_merge_argmax(m, idx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) xt = fmaxf(xt, __shfl_xor_sync(0xffffffffu, xt, o));
  }
}

}  // namespace sv
