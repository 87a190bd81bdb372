// Chain verification kernels: greedy prefix acceptance and lossless sampling
// acceptance with residual resampling.  Two launches per call:
//
// chain_stats_kernel  one CTA per (request, row, V-chunk).  Streams the chunk
//     once with 16-byte loads, keeps a running max / sum 2^((x - max) c) /
//     first argmax per thread, reduces through warp shuffles and shared
//     memory, and writes one Partial to the workspace.
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
//     ("投机解码:为什么一个字都不改", 改进方案).  Then
//       all accepted  the bonus token is drawn from p_L: the chunk holding
//                     u * sum is found from the streaming pass's chunk
//                     totals and only that CTA scans its chunk;
//       rejected at m every CTA adds up max(0, p_m - q_m) over its chunk;
//                     the last to finish (an arrival counter that the
//                     stats kernel zeroed, so the workspace needs no
//                     initialisation) picks the chunk where u * R falls and
//                     scans it: a draw from norm(max(0, p - q)).
// No kernel waits on another CTA.
#include "common.cuh"
#include "launch.h"

namespace sv {

constexpr int kMaxRows = 2 * SPEC_MAX_K + 1;

__device__ __forceinline__ Partial ld_partial(const Partial *p) {
  const float4 v = __ldcg(reinterpret_cast<const float4 *>(p));
  return Partial{v.x, v.y, __float_as_int(v.z), 0};
}

template <int DT>
__device__ __forceinline__ const char *row_ptr(const char *base, int64_t req_stride,
                                               int64_t row_stride, int b, int i) {
  return base + (static_cast<int64_t>(b) * req_stride + static_cast<int64_t>(i) * row_stride) *
                    Elems<DT>::kSize;
}

// ------------------------------------------------------------ streaming pass

template <int DT, bool SOFTMAX, bool VEC>
__global__ void __launch_bounds__(kThreads) chain_stats_kernel(const ChainParams P) {
  const int rows = SOFTMAX ? 2 * P.k + 1 : P.k + 1;
  const int per_req = rows * P.nc;
  const int b = blockIdx.x / per_req;
  const int rem = blockIdx.x - b * per_req;
  const int r = rem / P.nc, j = rem - r * P.nc;
  if (SOFTMAX && rem == 0 && threadIdx.x == 0) P.counter2[b] = 0;  // for the accept kernel
  const int L = P.draft_len ? P.draft_len[b] : P.k;
  if (L < 0 || L > P.k) return;  // reported by the accept kernel
  const char *row;
  if (r <= P.k) {
    if (r > L) return;
    row = row_ptr<DT>(P.target, P.t_req, P.row, b, r);
  } else {
    if (r - P.k - 1 >= L) return;
    row = row_ptr<DT>(P.draftl, P.d_req, P.row, b, r - P.k - 1);
  }
  float m = -INFINITY, s = 0.0f;
  int idx = kNoIndex;
  const int v0 = j * P.chunk, v1 = min(P.V, v0 + P.chunk);
  thread_chunk_stats<DT, SOFTMAX, VEC, kLoadStream>(row, v0, v1, P.c, m, s, idx);
  block_merge<SOFTMAX>(m, s, idx, P.c);
  if (threadIdx.x == 0)
    *reinterpret_cast<float4 *>(P.part + (static_cast<int64_t>(b) * rows + r) * P.nc + j) =
        make_float4(m, s, __int_as_float(idx), 0.0f);
}

// --------------------------------------------------------------- accept scan

// What every CTA of a request knows after the merge.
struct Verdict {
  int bad;      // SPEC_STATUS_* (0 = fine)
  int L, m, ne;
  int final_tok;  // greedy: argmax(row m)
};

// Merges the request's partials (target rows 0..L, then for sampling draft
// rows 0..L-1) and runs the accept scan.  Called by all threads of a CTA;
// the row statistics are left in sM / sS / sA, and for sampling sXT / sXD
// hold p_i(x_i) / q_i(x_i).
template <int DT, bool SAMPLE>
__device__ Verdict accept_scan(const ChainParams &P, int b, float *sM, float *sS, int *sA,
                               float *sXT, float *sXD, int *sTok) {
  __shared__ Verdict sv;
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = P.k;
  const int rows = SAMPLE ? 2 * k + 1 : k + 1;
  const int L = P.draft_len ? P.draft_len[b] : k;
  const bool len_ok = L >= 0 && L <= k;
  if (tid == 0) s_bad = len_ok ? SPEC_STATUS_OK : SPEC_STATUS_BAD_LENGTH;
  __syncthreads();
  if (len_ok && tid < L) {
    const int t = P.draft[static_cast<int64_t>(b) * k + tid];
    sTok[tid] = t;
    if (t < 0 || t >= P.V) atomicMax(&s_bad, SPEC_STATUS_TOKEN_RANGE);
  }
  __syncthreads();
  if (s_bad != SPEC_STATUS_OK) {
    Verdict v{s_bad, L, 0, 0, -1};
    __syncthreads();
    return v;
  }
  const int nrows = SAMPLE ? 2 * L + 1 : L + 1;
  for (int rr = warp; rr < nrows; rr += kWarps) {
    const int r = rr <= L ? rr : (k + 1) + (rr - L - 1);
    const Partial *pp = P.part + (static_cast<int64_t>(b) * rows + r) * P.nc;
    float m = -INFINITY, s = 0.0f;
    int idx = kNoIndex;
    for (int j = lane; j < P.nc; j += 32) {
      const Partial q = ld_partial(pp + j);
      if (SAMPLE) merge_stats(m, s, idx, q.m, q.s, q.idx, P.c); else merge_argmax(m, idx, q.m, q.idx);
    }
    if (SAMPLE) warp_merge_stats(m, s, idx, P.c); else warp_merge_argmax(m, idx);
    if (lane == 0) {
      sM[rr] = m;
      sS[rr] = s;
      sA[rr] = idx == kNoIndex ? 0 : idx;  // an all -inf row: every index ties, take 0
    }
  }
  if (SAMPLE) {
    for (int i = tid; i < 2 * L; i += kThreads) {
      if (i < L)
        sXT[i] = load_one<DT>(row_ptr<DT>(P.target, P.t_req, P.row, b, i), sTok[i]);
      else
        sXD[i - L] = load_one<DT>(row_ptr<DT>(P.draftl, P.d_req, P.row, b, i - L), sTok[i - L]);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int m = 0;
    if (SAMPLE) {
      const float *u = P.uniforms + static_cast<int64_t>(b) * (k + 1);
      for (int i = 0; i < L; ++i) {
        const float p = ex2((sXT[i] - sM[i]) * P.c) / sS[i];
        const float q = ex2((sXD[i] - sM[L + 1 + i]) * P.c) / sS[L + 1 + i];
        sXT[i] = p;  // now p_i(x_i)
        sXD[i] = q;  // and q_i(x_i)
        if (m == i && u[i] * q < p) m = i + 1;
      }
    } else {
      while (m < L && sA[m] == sTok[m]) ++m;
    }
    const int cap = P.max_emit ? P.max_emit[b] : k + 1;
    sv = Verdict{SPEC_STATUS_OK, L, m, max(0, min(m + 1, cap)), sA[m]};
  }
  __syncthreads();
  const Verdict v = sv;
  __syncthreads();
  return v;
}

// The outputs that do not depend on the final draw (written once per request).
template <bool SAMPLE>
__device__ void write_common(const ChainParams &P, int b, const Verdict &v, const int *sTok,
                             const float *sXT, const float *sXD, bool final_known, int final_tok) {
  const int k = P.k;
  int32_t *out = P.out_tokens + static_cast<int64_t>(b) * (k + 1);
  const int tid = threadIdx.x;
  if (v.bad) {
    for (int j = tid; j <= k; j += kThreads) out[j] = -1;
  } else {
    for (int j = tid; j <= k; j += kThreads) {
      if (j == v.m && j < v.ne && !final_known) continue;  // the drawing CTA writes it
      out[j] = j < v.ne ? (j < v.m ? sTok[j] : final_tok) : -1;
    }
  }
  if (SAMPLE) {
    for (int j = tid; j < k; j += kThreads) {
      const bool ok = !v.bad && j < v.L;
      if (P.p_tok) P.p_tok[static_cast<int64_t>(b) * k + j] = ok ? sXT[j] : -1.0f;
      if (P.q_tok) P.q_tok[static_cast<int64_t>(b) * k + j] = ok ? sXD[j] : -1.0f;
    }
  }
  if (tid == 0) {
    P.accepted[b] = v.bad ? 0 : v.m;
    P.n_emit[b] = v.bad ? 0 : v.ne;
    if (P.status) P.status[b] = v.bad;
    if (SAMPLE && v.bad && P.resid_mass) P.resid_mass[b] = 0.0f;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads) chain_greedy_accept_kernel(const ChainParams P) {
  __shared__ float sM[SPEC_MAX_K + 1], sS[SPEC_MAX_K + 1];
  __shared__ int sA[SPEC_MAX_K + 1], sTok[SPEC_MAX_K];
  const int b = blockIdx.x;
  const Verdict v = accept_scan<DT, false>(P, b, sM, sS, sA, nullptr, nullptr, sTok);
  write_common<false>(P, b, v, sTok, nullptr, nullptr, true, v.final_tok);
}

// Chunk j* of a row's streaming-pass totals where u * total falls; returns
// the threshold relative to the chunk start (INFINITY when rounding left u *
// total past the end: the last chunk with mass is taken).
__device__ __forceinline__ void pick_chunk(const Partial *pp, int nc, float M, float c, float u,
                                           int &jsel_out, float &thr_out) {
  float tot = 0.0f;
  for (int j = 0; j < nc; ++j) {
    const Partial q = ld_partial(pp + j);
    tot += q.s * ex2((q.m - M) * c);
  }
  const float thr = u * tot;
  float cum = 0.0f, base = 0.0f;
  int jsel = -1, jlast = 0;
  for (int j = 0; j < nc; ++j) {
    const Partial q = ld_partial(pp + j);
    const float w = q.s * ex2((q.m - M) * c);
    if (w > 0.0f) jlast = j;
    if (jsel < 0 && cum + w > thr) {
      jsel = j;
      base = cum;
    }
    cum += w;
  }
  jsel_out = jsel >= 0 ? jsel : jlast;
  thr_out = jsel >= 0 ? thr - base : INFINITY;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) chain_sample_accept_kernel(const ChainParams P) {
  __shared__ float sM[kMaxRows], sS[kMaxRows];
  __shared__ int sA[kMaxRows], sTok[SPEC_MAX_K];
  __shared__ float sXT[SPEC_MAX_K], sXD[SPEC_MAX_K];
  __shared__ float s_red[kWarps];
  __shared__ int s_last, s_j;
  __shared__ float s_thr, s_tot;
  __shared__ bool s_fallback;
  const int nc = P.nc;
  const int b = blockIdx.x / nc, j = blockIdx.x - b * nc;
  const int k = P.k, rows = 2 * k + 1;
  const int tid = threadIdx.x;
  const Verdict v = accept_scan<DT, true>(P, b, sM, sS, sA, sXT, sXD, sTok);
  if (j == 0) write_common<true>(P, b, v, sTok, sXT, sXD, false, -1);
  if (v.bad) return;
  const int m = v.m, L = v.L;
  const float u_final = P.uniforms[static_cast<int64_t>(b) * (k + 1) + k];

  if (m == L) {
    // every draft token accepted: bonus draw from p_L
    if (tid == 0)
      pick_chunk(P.part + (static_cast<int64_t>(b) * rows + L) * nc, nc, sM[L], P.c, u_final, s_j,
                 s_thr);
    __syncthreads();
    if (j != s_j) return;
    Weights W{row_ptr<DT>(P.target, P.t_req, P.row, b, L), nullptr, sM[L], 0.0f, 1.0f, 0.0f, P.c};
    const int lo = j * P.chunk, hi = min(P.V, lo + P.chunk);
    const int tok = block_select<DT, VEC>(W, lo, hi, s_thr);
    if (tid == 0) {
      if (m < v.ne) P.out_tokens[static_cast<int64_t>(b) * (k + 1) + m] = tok;
      if (P.resid_mass) P.resid_mass[b] = 0.0f;
    }
    return;
  }

  // rejected at m: residual mass of this chunk
  Weights W{row_ptr<DT>(P.target, P.t_req, P.row, b, m), row_ptr<DT>(P.draftl, P.d_req, P.row, b, m),
            sM[m], sM[L + 1 + m], 1.0f / sS[m], 1.0f / sS[L + 1 + m], P.c};
  const int v0 = j * P.chunk, v1 = min(P.V, v0 + P.chunk);
  const float acc = warp_sum(thread_chunk_weight_sum<DT, VEC, kLoadL2>(W, v0, v1));
  if ((tid & 31) == 0) s_red[tid >> 5] = acc;
  __syncthreads();
  if (tid == 0) {
    float t = 0.0f;
    for (int w = 0; w < kWarps; ++w) t += s_red[w];
    P.part2[static_cast<int64_t>(b) * nc + j] = t;
    __threadfence();
    s_last = atomicAdd(P.counter2 + b, 1) == nc - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) {
    const float *pp = P.part2 + static_cast<int64_t>(b) * nc;
    float tot = 0.0f;
    for (int i = 0; i < nc; ++i) tot += __ldcg(pp + i);
    s_tot = tot;
    s_fallback = !(tot > 0.0f);
    if (!s_fallback) {
      const float thr = u_final * tot;
      float cum = 0.0f, base = 0.0f;
      int jsel = -1, jlast = 0;
      for (int i = 0; i < nc; ++i) {
        const float w = __ldcg(pp + i);
        if (w > 0.0f) jlast = i;
        if (jsel < 0 && cum + w > thr) {
          jsel = i;
          base = cum;
        }
        cum += w;
      }
      s_j = jsel >= 0 ? jsel : jlast;
      s_thr = jsel >= 0 ? thr - base : INFINITY;
    } else {
      // zero residual mass (only through rounding): draw from p_m instead
      pick_chunk(P.part + (static_cast<int64_t>(b) * rows + m) * nc, nc, sM[m], P.c, u_final, s_j,
                 s_thr);
    }
  }
  __syncthreads();
  if (s_fallback) {
    W.b = nullptr;
    W.alpha = 1.0f;
    W.beta = 0.0f;
  }
  const int lo = s_j * P.chunk, hi = min(P.V, lo + P.chunk);
  const int tok = block_select<DT, VEC>(W, lo, hi, s_thr);
  if (tid == 0) {
    if (m < v.ne) P.out_tokens[static_cast<int64_t>(b) * (k + 1) + m] = tok;
    if (P.resid_mass) P.resid_mass[b] = s_fallback ? 0.0f : s_tot;
  }
}

// ------------------------------------------------------------------- host

template <int DT, bool VEC>
static cudaError_t launch_chain_t(const ChainParams &P, bool sample, cudaStream_t st) {
  const int rows = sample ? 2 * P.k + 1 : P.k + 1;
  const unsigned grid1 = static_cast<unsigned>(static_cast<long long>(P.B) * rows * P.nc);
  if (sample) {
    cudaError_t e = trace_launch("chain_stats_sample", st, [&] {
      chain_stats_kernel<DT, true, VEC><<<grid1, kThreads, 0, st>>>(P);
    });
    if (e != cudaSuccess) return e;
    const unsigned grid2 = static_cast<unsigned>(static_cast<long long>(P.B) * P.nc);
    return trace_launch("chain_sample_accept", st, [&] {
      chain_sample_accept_kernel<DT, VEC><<<grid2, kThreads, 0, st>>>(P);
    });
  }
  cudaError_t e = trace_launch("chain_stats_greedy", st, [&] {
    chain_stats_kernel<DT, false, VEC><<<grid1, kThreads, 0, st>>>(P);
  });
  if (e != cudaSuccess) return e;
  return trace_launch("chain_greedy_accept", st, [&] {
    chain_greedy_accept_kernel<DT><<<P.B, kThreads, 0, st>>>(P);
  });
}

cudaError_t launch_chain(const ChainParams &P, bool sample, bool vec, cudaStream_t st) {
  if (P.dtype == SPEC_DTYPE_BF16)
    return vec ? launch_chain_t<SPEC_DTYPE_BF16, true>(P, sample, st)
               : launch_chain_t<SPEC_DTYPE_BF16, false>(P, sample, st);
  return vec ? launch_chain_t<SPEC_DTYPE_F32, true>(P, sample, st)
             : launch_chain_t<SPEC_DTYPE_F32, false>(P, sample, st);
}

}  // namespace sv
