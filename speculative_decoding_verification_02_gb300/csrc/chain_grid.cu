// Grid-resident chain verification: one cooperative launch with one CTA per
// SM (fewer for small vocabularies).  CTA j owns slice j of the vocabulary in
// every row of every request and keeps those logits in registers from the
// first load to the final draw, so each logit is read from memory once.
// Sampling follows "投机解码:为什么一个字都不改" (改进方案): accept x_i while
// u_i q_i(x_i) < p_i(x_i), then draw from norm(max(0, p_m - q_m)) after a
// rejection at m, or from p_L after a full accept; greedy accepts x_i while
// x_i == argmax(row i) and emits argmax(row m) ("第 13 篇：推理引擎一次猜几个
// 字", ③ 伪代码).
//
// Work inside a CTA: an item is (request b, position i, chunk c), a chunk
// being 32 consecutive 16-byte groups of the slice (one warp load, 512
// bytes); position i holds target row i and, when sampling and i < k, draft
// row i, side by side in the same lane.  Warp w takes items w, w + 16, ...
//   1. all loads are issued at once; each chunk is folded into (max, sum
//      2^((x - max) c)) -- greedy: (max, first argmax) -- by one warp
//      reduction, the lane holding a drafted token keeps its logit, and the
//      CTA writes one partial per (request, row) to the workspace;
//   -- grid barrier --
//   2. every CTA merges every row's partials in CTA order, so all CTAs take
//      the same decision (the accepted prefix m) from the same numbers.
//      Greedy ends here (CTA 0 writes the outputs).  Sampling: each CTA sums
//      the final draw's weights over its slice -- the residual max(0, p - q)
//      and p_m itself, for the zero-residual fallback -- per chunk, and
//      writes its slice masses;
//   -- grid barrier --
//   3. every CTA reads the slice masses and finds the slice holding
//      u_k * total; that CTA scans its chunk masses, and the warp holding
//      the chunk scans its lanes and walks one group, from its registers.
// The barrier counter lives in the first bytes of the workspace: it must be
// zero when a launch starts, and the last CTA to leave sets it back to zero.
// Every wait is bounded; a CTA whose wait runs out marks the requests
// SPEC_STATUS_SYNC_TIMEOUT and leaves.
#include <mutex>
#include <vector>

#include "chain_common.cuh"
#include "common.cuh"
#include "launch.h"
#include "segments.cuh"

namespace sv {

constexpr int kGridThreads = 512;
constexpr int kGridWarps = kGridThreads / 32;
constexpr int kGridMaxSlots = 8;                               // chunks per warp, held in registers
static_assert(kGridMaxItems == kGridWarps * kGridMaxSlots, "items per CTA");
constexpr int kGridMaxPartials = 16384;                        // partials every CTA merges after barrier 1
constexpr unsigned kGridSpinLimit = 1u << 21;                  // polls of the barrier word (about a second)

// Arrive at the grid barrier (the counter counts arrivals over the whole
// launch; this barrier is passed once it reaches `target`).  False when the
// wait ran out.  Called by all threads of the CTA.
__device__ __forceinline__ bool grid_barrier(unsigned *count, unsigned target) {
  __shared__ int s_ok;
  __syncthreads();  // the CTA's writes before the arrival
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(count) : "memory");
    unsigned v = 0, it = 0;
    do {
      asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
    } while (v < target && ++it < kGridSpinLimit);
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    s_ok = v >= target;
  }
  __syncthreads();
  return s_ok != 0;
}

// Item index -> (request, position, chunk).
struct Item {
  int b, i, c, bi;
};
__device__ __forceinline__ Item decode_item(int it, int cpr, int K1) {
  Item r;
  r.c = it % cpr;
  r.bi = it / cpr;
  r.i = r.bi % K1;
  r.b = r.bi / K1;
  return r;
}

// The EPG logits of one group, with the value at `want` (a logit index) when
// the group holds it.
template <int DT>
__device__ __forceinline__ float pick_logit(const float *x, int e, int want, float none) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  float r = none;
#pragma unroll
  for (int q = 0; q < EPG; ++q)
    if (e + q == want) r = x[q];
  return r;
}

template <int DT, bool VEC, bool SAMPLE, int NS>
__global__ void __launch_bounds__(kGridThreads, 1) chain_grid_kernel(const ChainParams P) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  constexpr uint32_t kNegInf = DT == SPEC_DTYPE_F32 ? 0xff800000u : 0xff80ff80u;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cta = blockIdx.x, ncta = gridDim.x;
  const int B = P.B, k = P.k, K1 = k + 1, V = P.V;
  const int R = SAMPLE ? 2 * k + 1 : K1;  // partial rows per request: targets 0..k, then drafts 0..k-1
  const int cpr = P.grid_cpr;
  const int W = B * K1 * cpr;
  const int lo = min(V, cta * P.grid_gps * EPG), hi = min(V, lo + P.grid_gps * EPG);
  const float c = P.c;

  // ---- 1. every lane's groups of every row it owns, all loads in flight
  uint4 xt[NS], xd[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    const int it = warp + kGridWarps * s;
    xt[s] = xd[s] = make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
    if (it < W) {
      const Item t = decode_item(it, cpr, K1);
      const int e = lo + (t.c * 32 + lane) * EPG;
      xt[s] = load_group<DT, VEC>(row_ptr<DT>(P.target, P.t_req, P.row, t.b, t.i), e, hi);
      if (SAMPLE && t.i < k) xd[s] = load_group<DT, VEC>(row_ptr<DT>(P.draftl, P.d_req, P.row, t.b, t.i), e, hi);
    }
  }
  // the requests' inputs, in flight with them
  __shared__ int s_tok[kGridMaxItems], s_L[kGridMaxItems], s_cap[kGridMaxItems], s_bad[kGridMaxItems];
  __shared__ float s_u[kGridMaxItems];
  __shared__ float s_xt[kGridMaxItems], s_xd[kGridMaxItems];  // drafted tokens' logits, per (b, i)
  for (int j = tid; j < B * k; j += kGridThreads) s_tok[j] = P.draft[j];
  if (SAMPLE)
    for (int j = tid; j < B * K1; j += kGridThreads) s_u[j] = P.uniforms[j];
  for (int j = tid; j < B * K1; j += kGridThreads) s_xt[j] = s_xd[j] = -INFINITY;
  for (int b = tid; b < B; b += kGridThreads) {
    s_L[b] = P.draft_len ? P.draft_len[b] : k;
    s_cap[b] = P.max_emit ? P.max_emit[b] : K1;
  }
  __syncthreads();
  for (int b = tid; b < B; b += kGridThreads) {
    const int L = s_L[b];
    int bad = (L >= 0 && L <= k) ? SPEC_STATUS_OK : SPEC_STATUS_BAD_LENGTH;
    for (int i = 0; bad == SPEC_STATUS_OK && i < L; ++i) {
      const int x = s_tok[b * k + i];
      if (x < 0 || x >= V) bad = SPEC_STATUS_TOKEN_RANGE;
    }
    s_bad[b] = bad;
  }

  // per-chunk statistics (one warp reduction per chunk and row)
  __shared__ float4 s_chunk[2 * kGridMaxItems];  // [side][item]: m, s, first argmax (bits), -
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    const int it = warp + kGridWarps * s;
    if (it < W) {  // the same in the whole warp
      const Item t = decode_item(it, cpr, K1);
      const int e = lo + (t.c * 32 + lane) * EPG;
      const int want = t.i < k ? s_tok[t.b * k + t.i] : -1;
#pragma unroll
      for (int side = 0; side < (SAMPLE ? 2 : 1); ++side) {
        if (side == 1 && t.i >= k) break;
        float x[EPG];
        unpack16<DT>(side ? xd[s] : xt[s], x);
        float m = -INFINITY;
        int idx = kNoIndex;
#pragma unroll
        for (int q = 0; q < EPG; ++q) {
          if (x[q] > m) {
            m = x[q];
            idx = e + q;
          }
        }
        float sum = 0.0f;
        if (SAMPLE) {
          const float M = warp_allmax(m);
          if (M != -INFINITY) {
#pragma unroll
            for (int q = 0; q < EPG; ++q) sum += ex2((x[q] - M) * c);
          }
          sum = warp_sum(sum);
          m = M;
        } else {
          warp_allargmax(m, idx);
        }
        if (lane == 0) s_chunk[side * kGridMaxItems + it] = make_float4(m, sum, __int_as_float(idx), 0.0f);
        if (SAMPLE && want >= e && want < e + EPG) {  // this lane holds the drafted token
          const float v = pick_logit<DT>(x, e, want, -INFINITY);
          if (side) s_xd[t.bi] = v;
          else s_xt[t.bi] = v;
        }
      }
    }
  }
  __syncthreads();
  // the CTA's partial of each (request, row): its chunks merged in order
  const int nrows = B * R;
  for (int j = tid; j < nrows; j += kGridThreads) {
    const int b = j / R, r = j % R;
    const int side = r < K1 ? 0 : 1, i = side ? r - K1 : r, bi = b * K1 + i;
    float m = -INFINITY, sum = 0.0f;
    int idx = kNoIndex;
    for (int q = 0; q < cpr; ++q) {
      const float4 h = s_chunk[side * kGridMaxItems + bi * cpr + q];
      if (SAMPLE) merge_stats(m, sum, idx, h.x, h.y, kNoIndex, c);
      else merge_argmax(m, idx, h.x, __float_as_int(h.z));
    }
    const float xtok = SAMPLE && i < k ? (side ? s_xd[bi] : s_xt[bi]) : -INFINITY;
    P.part[static_cast<int64_t>(j) * ncta + cta] = Partial{m, sum, idx, xtok};
  }

  auto timeout = [&]() {  // the barrier's wait ran out: no result can be trusted
    for (int b = tid; b < B; b += kGridThreads) {
      P.n_emit[b] = 0;
      P.accepted[b] = 0;
      if (P.status) P.status[b] = SPEC_STATUS_SYNC_TIMEOUT;
    }
  };
  if (!grid_barrier(P.grid_sync, ncta)) {
    timeout();
    return;
  }

  // ---- 2. every row's partials merged, in CTA order (the same in every CTA)
  __shared__ float s_M[2 * kGridMaxItems], s_S[2 * kGridMaxItems], s_X[2 * kGridMaxItems];
  __shared__ int s_A[2 * kGridMaxItems];
  for (int j = warp; j < nrows; j += kGridWarps) {
    const Partial *pp = P.part + static_cast<int64_t>(j) * ncta;
    float m = -INFINITY, sum = 0.0f, x = -INFINITY;
    int idx = kNoIndex;
    for (int q = lane; q < ncta; q += 32) {
      const float4 h = __ldcg(reinterpret_cast<const float4 *>(pp + q));
      if (SAMPLE) merge_stats(m, sum, idx, h.x, h.y, kNoIndex, c);
      else merge_argmax(m, idx, h.x, __float_as_int(h.z));
      x = fmaxf(x, h.w);
    }
    if (SAMPLE) warp_allmerge<false>(m, sum, idx, c);
    else warp_allargmax(m, idx);
    x = warp_allmax(x);
    if (lane == 0) {
      s_M[j] = m;
      s_S[j] = sum;
      s_A[j] = idx == kNoIndex ? 0 : idx;
      s_X[j] = x;
    }
  }
  __syncthreads();
  // the decision of every request
  __shared__ float s_P[kGridMaxItems], s_Q[kGridMaxItems];
  __shared__ int s_acc[kGridMaxItems], s_m[kGridMaxItems], s_ne[kGridMaxItems];
  for (int j = tid; j < B * k; j += kGridThreads) {
    const int b = j / k, i = j % k;
    int ok = 0;
    if (s_bad[b] == SPEC_STATUS_OK && i < s_L[b]) {
      if (SAMPLE) {
        const int rt = b * R + i, rd = b * R + K1 + i;
        const float p = ex2((s_X[rt] - s_M[rt]) * c) / s_S[rt];
        const float q = ex2((s_X[rd] - s_M[rd]) * c) / s_S[rd];
        s_P[j] = p;
        s_Q[j] = q;
        ok = s_u[b * K1 + i] * q < p;
      } else {
        ok = s_A[b * R + i] == s_tok[j];
      }
    }
    s_acc[j] = ok;
  }
  __syncthreads();
  for (int b = tid; b < B; b += kGridThreads) {
    const int L = s_bad[b] == SPEC_STATUS_OK ? s_L[b] : 0;
    int m = L;
    for (int i = 0; i < L; ++i) {
      if (!s_acc[b * k + i]) {
        m = i;
        break;
      }
    }
    s_m[b] = m;
    s_ne[b] = max(0, min(m + 1, s_cap[b]));
  }
  __syncthreads();
  if (cta == 0) {  // every output but a sampled final token
    for (int j = tid; j < B * K1; j += kGridThreads) {
      const int b = j / K1, i = j % K1, bad = s_bad[b], m = s_m[b], ne = s_ne[b];
      if (!bad && SAMPLE && i == m && i < ne) continue;  // the drawing CTA writes it
      P.out_tokens[j] = bad ? -1 : (i < ne ? (i < m ? s_tok[b * k + i] : s_A[b * R + m]) : -1);
    }
    if (SAMPLE) {
      for (int j = tid; j < B * k; j += kGridThreads) {
        const int b = j / k, i = j % k;
        const bool ok = s_bad[b] == SPEC_STATUS_OK && i < s_L[b];
        if (P.p_tok) P.p_tok[j] = ok ? s_P[j] : -1.0f;
        if (P.q_tok) P.q_tok[j] = ok ? s_Q[j] : -1.0f;
      }
    }
    for (int b = tid; b < B; b += kGridThreads) {
      const int bad = s_bad[b];
      P.accepted[b] = bad ? 0 : s_m[b];
      P.n_emit[b] = bad ? 0 : s_ne[b];
      if (P.status) P.status[b] = bad;
      if (SAMPLE && bad && P.resid_mass) P.resid_mass[b] = 0.0f;
    }
  }

  if (SAMPLE) {
    // the final draw's weights over this slice, per chunk: residual and p_m
    __shared__ float2 s_cw[kGridMaxItems];
    auto weights = [&](const Item &t, const uint4 &gt, const uint4 &gd, float *wr, float *wp) {
      const int b = t.b, m = s_m[b], rt = b * R + m, rd = b * R + K1 + m;
      const bool resid = m < s_L[b];
      const float Mt = s_M[rt], iSt = 1.0f / s_S[rt];
      const float Md = resid ? s_M[rd] : 0.0f, iSd = resid ? 1.0f / s_S[rd] : 0.0f;
      float x[EPG], y[EPG];
      unpack16<DT>(gt, x);
      unpack16<DT>(gd, y);
#pragma unroll
      for (int q = 0; q < EPG; ++q) {
        const float p = ex2((x[q] - Mt) * c) * iSt;
        wp[q] = p;
        wr[q] = resid ? fmaxf(0.0f, p - ex2((y[q] - Md) * c) * iSd) : p;
      }
    };
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const int it = warp + kGridWarps * s;
      if (it < W) {
        const Item t = decode_item(it, cpr, K1);
        if (s_bad[t.b] == SPEC_STATUS_OK && t.i == s_m[t.b]) {  // the same in the whole warp
          float wr[EPG], wp[EPG], ar = 0.0f, ap = 0.0f;
          weights(t, xt[s], xd[s], wr, wp);
#pragma unroll
          for (int q = 0; q < EPG; ++q) {
            ar += wr[q];
            ap += wp[q];
          }
          ar = warp_sum(ar);
          ap = warp_sum(ap);
          if (lane == 0) s_cw[it] = make_float2(ar, ap);
        }
      }
    }
    __syncthreads();
    float2 *mass = reinterpret_cast<float2 *>(P.part2);  // [b][cta]
    for (int b = tid; b < B; b += kGridThreads) {
      if (s_bad[b] != SPEC_STATUS_OK) continue;
      const int first = (b * K1 + s_m[b]) * cpr;
      float ar = 0.0f, ap = 0.0f;
      for (int q = 0; q < cpr; ++q) {
        ar += s_cw[first + q].x;
        ap += s_cw[first + q].y;
      }
      mass[static_cast<int64_t>(b) * ncta + cta] = make_float2(ar, ap);
    }
    if (!grid_barrier(P.grid_sync, 2 * ncta)) {
      timeout();
      return;
    }

    // ---- 3. the slice holding u_k * total, then the chunk, the lane, the logit
    __shared__ int s_dit[kGridMaxItems], s_duse[kGridMaxItems];
    __shared__ float s_dthr[kGridMaxItems], s_dtot[kGridMaxItems];
    const int per = (ncta + 31) / 32;  // lane l takes CTAs [l per, (l + 1) per)
    for (int b = warp; b < B; b += kGridWarps) {
      if (s_bad[b] != SPEC_STATUS_OK) continue;
      const float2 *mb = mass + static_cast<int64_t>(b) * ncta;
      const int q0 = min(ncta, lane * per), q1 = min(ncta, q0 + per);
      float lr = 0.0f, lp = 0.0f;
      for (int q = q0; q < q1; ++q) {
        const float2 v = __ldcg(mb + q);
        lr += v.x;
        lp += v.y;
      }
      const float tr = warp_sum(lr), tp = warp_sum(lp);
      const bool use_p = !(tr > 0.0f);  // zero residual mass (rounding only): draw from p_m
      const float total = use_p ? tp : tr, mine = use_p ? lp : lr;
      const float thr = s_u[b * K1 + k] * total;
      const float incl = warp_inclusive_scan(mine, lane);
      const unsigned hit = __ballot_sync(0xffffffffu, mine > 0.0f && incl > thr);
      const unsigned pos = __ballot_sync(0xffffffffu, mine > 0.0f);
      const int lh = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
      int dcta = 0;
      float before = 0.0f;
      if (lane == lh) {  // walk this lane's CTAs
        float run = incl - mine;
        int sel = -1, last = -1;
        float bsel = run, blast = run;
        for (int q = q0; q < q1; ++q) {
          const float2 v = __ldcg(mb + q);
          const float w = use_p ? v.y : v.x;
          if (w > 0.0f) {
            last = q;
            blast = run;
            if (hit && sel < 0 && run + w > thr) {
              sel = q;
              bsel = run;
            }
          }
          run += w;
        }
        dcta = sel >= 0 ? sel : last;
        before = sel >= 0 ? bsel : blast;
      }
      if (lh >= 0) {
        dcta = __shfl_sync(0xffffffffu, dcta, lh);
        before = __shfl_sync(0xffffffffu, before, lh);
      }
      if (lane == 0) {
        int dit = -2;  // -2: another CTA draws; -1: this CTA, no mass anywhere (the slice start)
        float dthr = 0.0f;
        if (dcta == cta) {
          dit = -1;
          if (lh >= 0) {
            const float tl = thr - before;
            const int first = (b * K1 + s_m[b]) * cpr;
            float run = 0.0f, blast = 0.0f;
            int sel = -1, last = -1;
            float bsel = 0.0f;
            for (int q = 0; q < cpr; ++q) {
              const float w = use_p ? s_cw[first + q].y : s_cw[first + q].x;
              if (w > 0.0f) {
                last = q;
                blast = run;
                if (hit && sel < 0 && run + w > tl) {
                  sel = q;
                  bsel = run;
                }
              }
              run += w;
            }
            const int q = sel >= 0 ? sel : last;
            if (q >= 0) {
              dit = first + q;
              dthr = sel >= 0 ? tl - bsel : INFINITY;  // rounding: the chunk's last positive weight
            }
          }
        }
        s_dit[b] = dit;
        s_dthr[b] = dthr;
        s_duse[b] = use_p;
        s_dtot[b] = total;
      }
    }
    __syncthreads();
    auto finish = [&](int b, int tok, float w) {
      const int m = s_m[b];
      const bool resid = m < s_L[b] && !s_duse[b];
      if (m < s_ne[b]) P.out_tokens[static_cast<int64_t>(b) * K1 + m] = tok;
      if (P.resid_mass) P.resid_mass[b] = resid ? s_dtot[b] : 0.0f;
      if (P.final_prob) P.final_prob[b] = s_dtot[b] > 0.0f ? w / s_dtot[b] : 0.0f;
    };
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const int it = warp + kGridWarps * s;
      if (it < W) {
        const Item t = decode_item(it, cpr, K1);
        if (s_bad[t.b] == SPEC_STATUS_OK && t.i == s_m[t.b] && s_dit[t.b] == it) {  // warp-uniform
          float wr[EPG], wp[EPG], w[EPG], lm = 0.0f;
          weights(t, xt[s], xd[s], wr, wp);
          int le = -1;
#pragma unroll
          for (int q = 0; q < EPG; ++q) {
            w[q] = s_duse[t.b] ? wp[q] : wr[q];
            lm += w[q];
            if (w[q] > 0.0f) le = q;
          }
          const float tl = s_dthr[t.b];
          const float incl = warp_inclusive_scan(lm, lane);
          const unsigned hit = __ballot_sync(0xffffffffu, lm > 0.0f && incl > tl);
          const unsigned pos = __ballot_sync(0xffffffffu, lm > 0.0f);
          const int lh = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
          if (lane == lh) {
            float r = incl - lm;
            int pe = -1;
#pragma unroll
            for (int q = 0; q < EPG; ++q) {
              r += w[q];
              if (hit && pe < 0 && w[q] > 0.0f && r > tl) pe = q;
            }
            if (pe < 0) pe = le;  // rounding inside the lane: its last positive weight
            float wsel = 0.0f;
#pragma unroll
            for (int q = 0; q < EPG; ++q)
              if (q == pe) wsel = w[q];
            finish(t.b, lo + (t.c * 32 + lane) * EPG + pe, wsel);
          }
        }
      }
    }
    for (int b = tid; b < B; b += kGridThreads)
      if (s_bad[b] == SPEC_STATUS_OK && s_dit[b] == -1) finish(b, lo, 0.0f);  // no positive weight anywhere
  }

  // the last CTA out leaves the barrier counter at zero for the next launch
  __syncthreads();
  if (tid == 0) {
    const unsigned arrivals = (SAMPLE ? 3u : 2u) * static_cast<unsigned>(ncta);
    const unsigned old = atomicAdd(P.grid_sync, 1u);
    if (old == arrivals - 1) atomicExch(P.grid_sync, 0u);
  }
}

// ------------------------------------------------------------------- host

template <int DT, bool VEC, bool SAMPLE, int NS>
static cudaError_t launch_one(const ChainParams &P, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(P.grid_ctas));
  cfg.blockDim = dim3(kGridThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return trace_launch_ex(SAMPLE ? "chain_grid_sample" : "chain_grid_greedy", st,
                         [&] { return cudaLaunchKernelEx(&cfg, chain_grid_kernel<DT, VEC, SAMPLE, NS>, P); });
}

template <int DT, bool VEC, bool SAMPLE>
static cudaError_t launch_ns(const ChainParams &P, int ns, cudaStream_t st) {
  switch (ns) {
    case 1: return launch_one<DT, VEC, SAMPLE, 1>(P, st);
    case 2: return launch_one<DT, VEC, SAMPLE, 2>(P, st);
    case 4: return launch_one<DT, VEC, SAMPLE, 4>(P, st);
    default: return launch_one<DT, VEC, SAMPLE, 8>(P, st);
  }
}

template <int DT, bool VEC, bool SAMPLE>
static int resident_per_sm(int ns) {
  int n = 0;
  cudaError_t e;
  switch (ns) {
    case 1: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_grid_kernel<DT, VEC, SAMPLE, 1>, kGridThreads, 0); break;
    case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_grid_kernel<DT, VEC, SAMPLE, 2>, kGridThreads, 0); break;
    case 4: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_grid_kernel<DT, VEC, SAMPLE, 4>, kGridThreads, 0); break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, chain_grid_kernel<DT, VEC, SAMPLE, 8>, kGridThreads, 0); break;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Device facts the plan needs (cached per device): SMs, whether cooperative
// launches are supported.
struct GridDevice {
  int dev, sms, coop;
};

static bool grid_device(GridDevice &out) {
  static std::mutex mu;
  static std::vector<GridDevice> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> g(mu);
  for (const GridDevice &d : cache)
    if (d.dev == dev) {
      out = d;
      return d.sms > 0 && d.coop;
    }
  GridDevice d{dev, 0, 0};
  if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
    cudaGetLastError();
    d.sms = 0;
  }
  cache.push_back(d);
  out = d;
  return d.sms > 0 && d.coop;
}

bool chain_grid_plan(ChainParams &P, bool sample, bool vec) {
  GridDevice d;
  if (!grid_device(d)) return false;
  const int epg = P.dtype == SPEC_DTYPE_F32 ? 4 : 8;
  const long long vg = (static_cast<long long>(P.V) + epg - 1) / epg;
  long long ncta = std::min<long long>(std::min(d.sms, kGridMaxCtas), (vg + 31) / 32);
  if (ncta < 1) ncta = 1;
  const long long gps = (vg + ncta - 1) / ncta;
  ncta = (vg + gps - 1) / gps;
  const long long cpr = (gps + 31) / 32;
  const long long items = static_cast<long long>(P.B) * (P.k + 1) * cpr;
  const long long rows = static_cast<long long>(P.B) * (sample ? 2 * P.k + 1 : P.k + 1);
  if (items > kGridMaxItems || rows * ncta > kGridMaxPartials) return false;
  const long long need = (items + kGridWarps - 1) / kGridWarps;
  const int ns = need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : 8;
  int per_sm = 0;
  if (P.dtype == SPEC_DTYPE_BF16) {
    per_sm = vec ? (sample ? resident_per_sm<SPEC_DTYPE_BF16, true, true>(ns) : resident_per_sm<SPEC_DTYPE_BF16, true, false>(ns))
                 : (sample ? resident_per_sm<SPEC_DTYPE_BF16, false, true>(ns) : resident_per_sm<SPEC_DTYPE_BF16, false, false>(ns));
  } else {
    per_sm = vec ? (sample ? resident_per_sm<SPEC_DTYPE_F32, true, true>(ns) : resident_per_sm<SPEC_DTYPE_F32, true, false>(ns))
                 : (sample ? resident_per_sm<SPEC_DTYPE_F32, false, true>(ns) : resident_per_sm<SPEC_DTYPE_F32, false, false>(ns));
  }
  if (per_sm < 1 || ncta > static_cast<long long>(per_sm) * d.sms) return false;
  P.grid_ctas = static_cast<int>(ncta);
  P.grid_gps = static_cast<int>(gps);
  P.grid_cpr = static_cast<int>(cpr);
  P.grid_slots = ns;
  return true;
}

cudaError_t launch_chain_grid(const ChainParams &P, bool sample, bool vec, cudaStream_t st) {
  if (P.dtype == SPEC_DTYPE_BF16) {
    if (vec) return sample ? launch_ns<SPEC_DTYPE_BF16, true, true>(P, P.grid_slots, st)
                           : launch_ns<SPEC_DTYPE_BF16, true, false>(P, P.grid_slots, st);
    return sample ? launch_ns<SPEC_DTYPE_BF16, false, true>(P, P.grid_slots, st)
                  : launch_ns<SPEC_DTYPE_BF16, false, false>(P, P.grid_slots, st);
  }
  if (vec) return sample ? launch_ns<SPEC_DTYPE_F32, true, true>(P, P.grid_slots, st)
                         : launch_ns<SPEC_DTYPE_F32, true, false>(P, P.grid_slots, st);
  return sample ? launch_ns<SPEC_DTYPE_F32, false, true>(P, P.grid_slots, st)
                : launch_ns<SPEC_DTYPE_F32, false, false>(P, P.grid_slots, st);
}

}  // namespace sv
