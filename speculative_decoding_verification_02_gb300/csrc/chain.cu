// Chain verification kernels: greedy prefix acceptance and lossless sampling
// acceptance with residual resampling.  Two launches per call, the second
// one a programmatic dependent launch of the first:
//
// chain_stats_kernel  one CTA per (request, row, V-chunk).  Streams the chunk
//     once with 16-byte loads, keeps a running max / sum 2^((x - max) c) /
//     first argmax per thread, reduces through warp shuffles and shared
//     memory, and writes one Partial to the workspace, together with the
//     logit of the row's drafted token when that token falls in the chunk.
//
// chain_greedy_accept_kernel  one CTA per request: merges the partials of
//     target rows 0..L into argmaxes and accepts x_i while x_i == argmax(row
//     i); at the first mismatch it emits argmax(row m)
//     ("第 13 篇：推理引擎一次猜几个字", ③ 伪代码 / 逐行要点).
//
// chain_sample_accept_kernel  one CTA per (request, V-chunk).  Every CTA of
//     a request merges the request's partials in the same order, so all of
//     them reach the same decision: p_i(x_i), q_i(x_i), accept while
//     u_i q_i(x_i) < p_i(x_i), i.e. u_i < min(1, p/q)
//     ("投机解码:为什么一个字都不改", 改进方案).  Every warp then adds up the
//     final draw's weights over its range of the chunk -- max(0, p_m - q_m)
//     after a rejection at m, p_L after a full accept -- and the CTA
//     publishes its warp masses and arrives on the request's counter (which
//     the stats kernel zeroed, so the workspace needs no initialisation).
//     The last CTA to arrive finds the chunk and the warp range where
//     u * total falls and walks that range: a draw from norm(max(0, p - q))
//     or from p_L.  When every request's thread-block cluster fits on the GPU
//     at once, the cluster accept kernel (chain_fused.cu) replaces it.
// The accept kernels read their inputs before waiting on the stats grid.
// No kernel waits on another CTA.
#include <cooperative_groups.h>

#include "chain_common.cuh"
#include "chain_merge.cuh"
#include "common.cuh"
#include "launch.h"
#include "segments.cuh"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kMaxRows = 2 * SPEC_MAX_K + 1;
constexpr int kPickCache = 512;  // chunk weights kept in shared memory by warp_pick

// Arrival counter with release (this thread's earlier writes become visible
// first) and acquire (the caller sees what earlier arrivals published).
__device__ __forceinline__ int atomic_add_acq_rel(int *p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ------------------------------------------------------------ streaming pass

template <int DT, bool SOFTMAX, bool VEC>
__global__ void __launch_bounds__(kThreads) chain_stats_kernel(const ChainParams P) {
  // Launched early behind the previous kernel in the stream: wait for it
  // before reading, and only then let the accept kernel start (it reads the
  // request's inputs, which that previous kernel may have written, before
  // its own wait).
  pdl_wait();
  pdl_launch_dependents();
  const int rows = SOFTMAX ? 2 * P.k + 1 : P.k + 1;
  const int per_req = rows * P.nc;
  const int b = blockIdx.x / per_req;
  const int rem = blockIdx.x - b * per_req;
  const int r = rem / P.nc, j = rem - r * P.nc;
  if (SOFTMAX && rem == 0 && threadIdx.x == 0) P.counter2[b] = 0;  // for the accept kernel
  const int L = P.draft_len ? P.draft_len[b] : P.k;
  if (L < 0 || L > P.k) return;  // reported by the accept kernel
  const char *row;
  int pos;
  if (r <= P.k) {
    if (r > L) return;
    pos = r;
    row = row_ptr<DT>(P.target, P.t_req, P.row, b, r);
  } else {
    pos = r - P.k - 1;
    if (pos >= L) return;
    row = row_ptr<DT>(P.draftl, P.d_req, P.row, b, pos);
  }
  const int v0 = j * P.chunk, v1 = min(P.V, v0 + P.chunk);
  // the row's drafted token: its logit is picked up while streaming
  const int tok = (SOFTMAX && pos < L) ? P.draft[static_cast<int64_t>(b) * P.k + pos] : -1;
  float m = -INFINITY, s = 0.0f, xt = -INFINITY;
  int idx = kNoIndex;
  // (the argmax is only used by greedy verification)
  thread_chunk_stats<DT, SOFTMAX, VEC, kLoadStream, kThreads, !SOFTMAX>(row, v0, v1, P.c, m, s, idx, tok, xt);
  block_allmerge<SOFTMAX, !SOFTMAX, kThreads>(m, s, idx, P.c, xt);
  if (threadIdx.x == 0)
    *reinterpret_cast<float4 *>(P.part + (static_cast<int64_t>(b) * rows + r) * P.nc + j) =
        make_float4(m, s, __int_as_float(idx), xt);
}

// --------------------------------------------------------------- accept scan

template <int DT>
__global__ void __launch_bounds__(kThreads) chain_greedy_accept_kernel(const ChainParams P) {
  __shared__ int sA[SPEC_MAX_K + 1], sTok[SPEC_MAX_K];
  __shared__ int s_m;
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Prologue pr = read_request(P, b, sTok, nullptr, false);
  pdl_wait();
  if (pr.bad) {
    write_common<false>(P, b, pr.bad, pr.L, 0, 0, sTok, nullptr, nullptr, true, -1);
    return;
  }
  const int rows = P.k + 1;
  const Partial *base = P.part + static_cast<int64_t>(b) * rows * P.nc;
  for (int r = warp; r <= pr.L; r += 2 * kWarps) {
    const int r2 = r + kWarps;
    MergedRow a, bb;
    warp_merge_two_rows<false>(base + static_cast<int64_t>(r) * P.nc,
                               r2 <= pr.L ? base + static_cast<int64_t>(r2) * P.nc : nullptr, P.nc, 1.0f, -1, -1,
                               a, bb);
    if (lane == 0) {
      sA[r] = a.A;
      if (r2 <= pr.L) sA[r2] = bb.A;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int m = 0;
    while (m < pr.L && sA[m] == sTok[m]) ++m;
    s_m = m;
  }
  __syncthreads();
  const int m = s_m;
  write_common<false>(P, b, 0, pr.L, m, max(0, min(m + 1, pr.cap)), sTok, nullptr, nullptr, true, sA[m]);
}

template <int DT, bool VEC, bool CVEC>
__global__ void __launch_bounds__(kThreads) chain_sample_accept_kernel(const ChainParams P) {
  static_assert(kWarps == 8, "a chunk's warp masses are two 16-byte words");
  __shared__ float sM[kMaxRows], sS[kMaxRows], sX[kMaxRows], sTh[kMaxRows];
  __shared__ int sTok[SPEC_MAX_K];
  __shared__ float sU[SPEC_MAX_K + 1], sP[SPEC_MAX_K], sQ[SPEC_MAX_K];
  __shared__ float s_wcache[kPickCache], s_wm[kWarps];
  __shared__ int s_last, s_j, s_jlast, s_w;
  __shared__ float s_thr;
  const int nc = P.nc, nch = P.nc2;
  const int b = blockIdx.x / nch, j = blockIdx.x - b * nch;
  const int k = P.k, rows = 2 * k + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Prologue pr = read_request(P, b, sTok, sU, true);  // (the inputs, before the wait)
  pdl_wait();
  if (pr.bad) {
    if (j == 0) write_common<true>(P, b, pr.bad, pr.L, 0, 0, sTok, sP, sQ, true, -1);
    return;
  }
  const int L = pr.L;
  // merge: target rows 0..L are rr = 0..L, draft rows 0..L-1 are rr = L+1..2L;
  // each warp takes two rows at a time with all their loads in flight
  const int nrr = 2 * L + 1;
  const Partial *base = P.part + static_cast<int64_t>(b) * rows * nc;
  auto row_of = [&](int rr) { return rr <= L ? rr : (k + 1) + (rr - L - 1); };
  auto tok_chunk = [&](int rr) {
    const int pos = rr <= L ? rr : rr - L - 1;
    return pos < L ? sTok[pos] / P.chunk : -1;
  };
  for (int rr = warp; rr < nrr; rr += 2 * kWarps) {
    const int rr2 = rr + kWarps;
    MergedRow a, bb;
    warp_merge_two_rows<true>(base + static_cast<int64_t>(row_of(rr)) * nc,
                              rr2 < nrr ? base + static_cast<int64_t>(row_of(rr2)) * nc : nullptr, nc, P.c,
                              tok_chunk(rr), rr2 < nrr ? tok_chunk(rr2) : -1, a, bb);
    if (lane == 0) {
      sM[rr] = a.M;
      sS[rr] = a.S;
      sX[rr] = a.X;
      sTh[rr] = row_theta(P.theta, static_cast<int64_t>(b) * rows + row_of(rr));
      if (rr2 < nrr) {
        sM[rr2] = bb.M;
        sS[rr2] = bb.S;
        sX[rr2] = bb.X;
        sTh[rr2] = row_theta(P.theta, static_cast<int64_t>(b) * rows + row_of(rr2));
      }
    }
  }
  __syncthreads();
  // Every warp tests the positions itself (lane i: positions i, i + 32, ...);
  // warp 0 keeps p and q for the outputs, and chunk 0's warp 0 writes them.
  int m = L;  // the first rejected position
  for (int i0 = 0; i0 < L; i0 += 32) {
    const int i = i0 + lane;
    bool ok = true;
    if (i < L) {
      // (a drafted token below its row's threshold has probability 0)
      const float p = sX[i] >= sTh[i] ? ex2((sX[i] - sM[i]) * P.c) / sS[i] : 0.0f;
      const float q = sX[L + 1 + i] >= sTh[L + 1 + i] ? ex2((sX[L + 1 + i] - sM[L + 1 + i]) * P.c) / sS[L + 1 + i]
                                                      : 0.0f;
      if (warp == 0) {
        sP[i] = p;
        sQ[i] = q;
      }
      ok = sU[i] * q < p;
    }
    const unsigned rej = __ballot_sync(0xffffffffu, !ok);
    if (rej && m == L) m = i0 + __ffs(rej) - 1;
  }
  const int ne = max(0, min(m + 1, pr.cap));
  if (j == 0 && warp == 0) {
    __syncwarp();
    write_common<true>(P, b, 0, L, m, ne, sTok, sP, sQ, false, -1, lane, 32);
  }
  const float u_final = sU[k];

  // the final draw: the residual max(0, p_m - q_m) after a rejection, p_L
  // after a full accept.  Each warp adds up the weights of its range of the
  // chunk (G rounds of 32 16-byte groups, the lane_group split); thread 0
  // publishes the chunk's warp masses and arrives; the last CTA to arrive
  // finds the chunk, then the warp range, where u * total falls, and one
  // warp walks that range.
  Weights W = m < L
                  ? Weights{row_ptr<DT>(P.target, P.t_req, P.row, b, m), row_ptr<DT>(P.draftl, P.d_req, P.row, b, m),
                            sM[m], sM[L + 1 + m], 1.0f / sS[m], 1.0f / sS[L + 1 + m], P.c, sTh[m], sTh[L + 1 + m]}
                  : Weights{row_ptr<DT>(P.target, P.t_req, P.row, b, L), nullptr, sM[L], 0.0f, 1.0f / sS[L], 0.0f,
                            P.c, sTh[L], -INFINITY};
  constexpr int EPG = Elems<DT>::kPerGroup;
  const int G = P.chunk2 / (kThreads * EPG);
  const int v0 = j * P.chunk2, v1 = min(P.V, v0 + P.chunk2);
  const bool filt = weights_filtered(W);  // (no mask in the loops without a threshold)
  const float wm = warp_sum(filt ? lane_weight_sum<DT, CVEC, true>(W, v0, v1, G, nullptr)
                                 : lane_weight_sum<DT, CVEC, false>(W, v0, v1, G, nullptr));
  if (lane == 0) s_wm[warp] = wm;
  __syncthreads();
  float *wmg = P.part2 + static_cast<int64_t>(b) * nch * kWarps;  // [chunk][warp]
  if (tid == 0) {
    // thread 0 alone publishes, then arrives (release); the last of every
    // nch arrivals draws, so a launch repeated on the same partials draws again
    float4 *dst = reinterpret_cast<float4 *>(wmg + static_cast<int64_t>(j) * kWarps);
    dst[0] = make_float4(s_wm[0], s_wm[1], s_wm[2], s_wm[3]);
    dst[1] = make_float4(s_wm[4], s_wm[5], s_wm[6], s_wm[7]);
    s_last = (atomic_add_acq_rel(P.counter2 + b, 1) + 1) % nch == 0;
    s_j = kNoIndex;
    s_jlast = -1;
  }
  __syncthreads();
  if (!s_last) return;

  // ---- the last CTA: thread t holds chunk t's warp masses (nch <= kThreads)
  float wv[kWarps];
  float cm = 0.0f;
  if (tid < nch) {
    const float4 lo4 = __ldcg(reinterpret_cast<const float4 *>(wmg + static_cast<int64_t>(tid) * kWarps));
    const float4 hi4 = __ldcg(reinterpret_cast<const float4 *>(wmg + static_cast<int64_t>(tid) * kWarps + 4));
    wv[0] = lo4.x; wv[1] = lo4.y; wv[2] = lo4.z; wv[3] = lo4.w;
    wv[4] = hi4.x; wv[5] = hi4.y; wv[6] = hi4.z; wv[7] = hi4.w;
  } else {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) wv[w] = 0.0f;
  }
#pragma unroll
  for (int w = 0; w < kWarps; ++w) cm += wv[w];
  // block-wide scan of the chunk masses in chunk order
  const float incl_w = warp_inclusive_scan(cm, lane);
  float excl_w = __shfl_up_sync(0xffffffffu, incl_w, 1);
  if (lane == 0) excl_w = 0.0f;
  if (lane == 31) s_wm[warp] = incl_w;
  __syncthreads();
  float before = 0.0f, total = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float t = s_wm[w];
    if (w < warp) before += t;
    total += t;
  }
  const bool fallback = !(total > 0.0f) && m < L;
  if (!fallback) {
    const float thr = u_final * total;
    if (cm > 0.0f) {
      if (before + incl_w > thr) atomicMin(&s_j, tid);
      atomicMax(&s_jlast, tid);
    }
    __syncthreads();
    const int jsel = s_j != kNoIndex ? s_j : max(s_jlast, 0);  // (rounding: the last chunk with mass)
    if (tid == jsel) {
      // the warp range of chunk jsel where the threshold falls
      const float thr_c = s_j != kNoIndex ? thr - (before + excl_w) : INFINITY;
      float run = 0.0f, t_w = INFINITY;
      int wsel = -1, wlast = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (wv[w] > 0.0f) {
          wlast = w;
          if (wsel < 0 && run + wv[w] > thr_c) {
            wsel = w;
            t_w = thr_c - run;
          }
        }
        run += wv[w];
      }
      s_w = wsel >= 0 ? wsel : wlast;
      s_thr = wsel >= 0 ? t_w : INFINITY;
    }
    __syncthreads();
    if (warp != 0) return;
    const int lo = jsel * P.chunk2, hi = min(P.V, lo + P.chunk2);
    auto walk = [&]<bool FILT>() {
      return warp_walk_range<EPG>(s_w, G, s_thr, [&](int g, float *w) {
        float x[EPG], y[EPG];
        unpack16<DT>(load_group<DT, CVEC>(W.a, lo + g * EPG, hi), x);
        if (W.b) unpack16<DT>(load_group<DT, CVEC>(W.b, lo + g * EPG, hi), y);
        weights_group<EPG, FILT>(W, x, y, w);
      });
    };
    const int pick = filt ? walk.template operator()<true>() : walk.template operator()<false>();
    const int tok = pick >= 0 ? lo + pick : lo;  // (a range without mass: its first logit)
    if (lane == 0) {
      if (m < ne) P.out_tokens[static_cast<int64_t>(b) * (k + 1) + m] = tok;
      if (P.resid_mass) P.resid_mass[b] = m < L ? total : 0.0f;
      if (P.final_prob)
        P.final_prob[b] = weight_at<DT>(W, load_one<DT>(W.a, tok), W.b ? load_one<DT>(W.b, tok) : 0.0f) / total;
    }
    return;
  }
  // zero residual mass (only through rounding): draw from p_m instead, its
  // chunks picked from the streaming pass's statistics
  __shared__ int s_fj;
  __shared__ float s_fthr, s_ftot;
  if (warp == 0) {
    const Partial *p1 = P.part + (static_cast<int64_t>(b) * rows + m) * nc;
    const float M = sM[m], c = P.c;
    int js;
    float th, tp;
    warp_pick([&](int jj) { const Partial q = ld_partial(p1 + jj); return q.s * ex2((q.m - M) * c); }, nc, u_final,
              s_wcache, kPickCache, js, th, tp);
    if (lane == 0) {
      s_fj = js;
      s_fthr = th;
      s_ftot = tp;
    }
  }
  __syncthreads();
  W.b = nullptr;
  W.alpha = 1.0f;
  W.beta = 0.0f;
  const int lo = s_fj * P.chunk, hi = min(P.V, lo + P.chunk);
  int tok = block_select<DT, VEC>(W, lo, hi, s_fthr);
  if (tok < 0) tok = lo;  // no positive weight in the range (a row without mass): its first logit
  if (tid == 0) {
    if (m < ne) P.out_tokens[static_cast<int64_t>(b) * (k + 1) + m] = tok;
    if (P.resid_mass) P.resid_mass[b] = 0.0f;
    if (P.final_prob)
      P.final_prob[b] = weight_at<DT>(W, load_one<DT>(W.a, tok), 0.0f) / s_ftot;
  }
}

// ------------------------------------------------------------------- host

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel in the stream is still running, and waits for it with
// griddepcontrol.wait before touching its results.
template <class K>
static cudaError_t launch_dependent(K kern, unsigned grid, cudaStream_t st, const ChainParams &P) {
  // (every kernel of the library waits with griddepcontrol.wait before it
  // reads anything the previous kernel in the stream may have written)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = trace_enabled() ? 0 : 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int DT, bool VEC, bool CVEC>
static cudaError_t launch_chain_t(const ChainParams &P, bool sample, bool stats, cudaStream_t st) {
  const int rows = sample ? 2 * P.k + 1 : P.k + 1;
  const unsigned grid1 = static_cast<unsigned>(static_cast<long long>(P.B) * rows * P.nc);
  if (sample) {
    cudaError_t e = cudaSuccess;
    if (stats)
      e = trace_launch_ex("chain_stats_sample", st, [&] {
        return launch_dependent(chain_stats_kernel<DT, true, VEC>, grid1, st, P);
      });
    if (e != cudaSuccess) return e;
    if (P.cluster > 0) return launch_chain_accept_cluster(P, CVEC, st);
    const unsigned grid2 = static_cast<unsigned>(static_cast<long long>(P.B) * P.nc2);
    return trace_launch_ex("chain_sample_accept", st, [&] {
      return launch_dependent(chain_sample_accept_kernel<DT, VEC, CVEC>, grid2, st, P);
    });
  }
  cudaError_t e = trace_launch_ex("chain_stats_greedy", st, [&] {
    return launch_dependent(chain_stats_kernel<DT, false, VEC>, grid1, st, P);
  });
  if (e != cudaSuccess) return e;
  return trace_launch_ex("chain_greedy_accept", st, [&] {
    return launch_dependent(chain_greedy_accept_kernel<DT>, static_cast<unsigned>(P.B), st, P);
  });
}

cudaError_t launch_chain(const ChainParams &P, bool sample, bool vec, bool cvec, cudaStream_t st, bool stats) {
  // (cvec implies vec: it adds V a multiple of a 16-byte group)
  if (P.dtype == SPEC_DTYPE_BF16)
    return vec ? (cvec ? launch_chain_t<SPEC_DTYPE_BF16, true, true>(P, sample, stats, st)
                       : launch_chain_t<SPEC_DTYPE_BF16, true, false>(P, sample, stats, st))
               : launch_chain_t<SPEC_DTYPE_BF16, false, false>(P, sample, stats, st);
  return vec ? (cvec ? launch_chain_t<SPEC_DTYPE_F32, true, true>(P, sample, stats, st)
                     : launch_chain_t<SPEC_DTYPE_F32, true, false>(P, sample, stats, st))
             : launch_chain_t<SPEC_DTYPE_F32, false, false>(P, sample, stats, st);
}

}  // namespace sv
