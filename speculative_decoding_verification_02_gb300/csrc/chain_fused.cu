// Fused chain verification: one thread-block cluster per request performs
// the whole call -- every row's statistics, the acceptance decision and the
// final draw -- in one launch.  Sampling mode follows the acceptance rule of
// "投机解码:为什么一个字都不改" (改进方案): accept x_i while
// u_i q_i(x_i) < p_i(x_i), then draw from norm(max(0, p_m - q_m)) after a
// rejection at m, or from p_L after a full accept; greedy mode accepts x_i
// while x_i == argmax(row i) and emits argmax(row m)
// ("第 13 篇：推理引擎一次猜几个字", ③ 伪代码).
//
// Each CTA of a request's cluster owns one slice of the vocabulary and each
// of its warps one contiguous range of that slice (lanes interleaved, so
// loads stay coalesced):
//   1. rows are streamed kRowBatch at a time with all their loads in flight;
//      each lane folds its groups of each row into (max, sum
//      2^((x - max) c)) -- greedy mode: (max, first argmax) -- and warps
//      merge those with redux and shuffle reductions;
//   2. warp w merges rows w, w + 16, ... over the CTA's warps and pushes the
//      CTA's statistics of the row into every CTA of the cluster
//      (distributed shared memory); after one cluster barrier every CTA
//      merges the slices in rank order and takes the same decision, the
//      accepted prefix m;
//   3. (sampling) each warp adds up the final draw's weights over its range;
//      the slice masses are exchanged like the statistics, the rank whose
//      slice holds u * total is found, and in that CTA a scan of the warp
//      masses and a walk of the chosen warp's range give the token.
// Used when the clusters of all requests are resident at once: one launch
// then replaces the streaming pass and the accept kernel, and the workspace
// is not touched.  The kernel waits for the previous grid in the stream
// (programmatic dependent launch) before it reads anything.
#include <cooperative_groups.h>

#include <mutex>
#include <vector>

#include "chain_common.cuh"
#include "common.cuh"
#include "launch.h"
#include "segments.cuh"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kRowBatch = 4;  // rows whose loads are in flight together
constexpr int kFusedMaxCluster = 16;
constexpr int kFusedMaxRows = 2 * SPEC_MAX_K + 1;
constexpr int kFusedMinSlice = 4096;  // fewest logits per CTA when choosing the cluster size

struct __align__(16) RowPart {
  float m, s;  // max, sum of 2^((x - m) c)
  int i;       // first argmax
  float pad;
};

// The streaming pass's statistics of one (request, row, chunk).
__device__ __forceinline__ float4 ld_part(const Partial *p) { return __ldcg(reinterpret_cast<const float4 *>(p)); }

// ACCEPT: the second launch of the two-pass path.  The row statistics are
// not streamed here but merged from the partials the streaming pass wrote
// (every CTA merges all of its request's rows, so no exchange is needed for
// them); the decision and the final draw are the same.  Its CTAs are small
// enough to share SMs with the streaming pass, so they start early and wait
// for it (programmatic dependent launch).
// FILT (accept kernel only): the rows carry top-k / top-p thresholds, which
// mask the drafted tokens' probabilities and the draw weights; without it
// the kernel reads and applies none.
template <int DT, bool VEC, bool SAMPLE, bool ACCEPT, bool FILT = false>
__global__ void __launch_bounds__(kFusedThreads, ACCEPT ? 2 : 1) chain_fused_kernel(const ChainParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int EPG = Elems<DT>::kPerGroup;
  const int CS = P.cluster;
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / CS;
  const int k = P.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows_max = SAMPLE ? 2 * k + 1 : k + 1;
  extern __shared__ RowPart dyn_parts[];
  RowPart *s_wpart = dyn_parts;                           // [warp][row] warp statistics (streamed here)
  RowPart *s_cpart = s_wpart + kFusedWarps * rows_max;    // [rank][row] slice statistics (streamed here)
  float *s_gsum = reinterpret_cast<float *>(ACCEPT ? dyn_parts : s_cpart + kFusedMaxCluster * rows_max);
  // s_gsum: [threads * groups] weight sum of each 16-byte group of the slice (sampling)
  __shared__ int sTok[SPEC_MAX_K], sA[kFusedMaxRows];
  __shared__ float sU[SPEC_MAX_K + 1], sP[SPEC_MAX_K], sQ[SPEC_MAX_K];
  __shared__ float sM[kFusedMaxRows], sS[kFusedMaxRows], sX[kFusedMaxRows], sTh[kFusedMaxRows];
  __shared__ float sIS[kFusedMaxRows];  // 1 / sS
  __shared__ float s_red[kFusedWarps], s_z[2][kFusedMaxCluster];
  const RowPart kEmpty{-INFINITY, 0.0f, kNoIndex, 0.0f};

  const float c = P.c;
  Prologue pr;
  if (ACCEPT) {
    // after the wait, warp w merges rows w, w + 16, ... of the streaming
    // pass's layout (target rows 0..k, draft rows k + 1..2k; rows the pass
    // skipped are merged too and ignored); the drafted token's logit is the
    // largest x over the chunks (the one chunk holding the token has it, the
    // others -inf)
    pdl_launch_dependents();
    // The request's own inputs do not come from the streaming pass: they are
    // read and checked while it still runs.  (This kernel starts only after
    // the streaming pass has waited for whatever kernel wrote them.)
    __shared__ int s_L, s_cap;
    if (tid == 0) s_L = P.draft_len ? P.draft_len[b] : k;
    if (tid == 32) s_cap = P.max_emit ? P.max_emit[b] : k + 1;
    if (tid < k) sTok[tid] = P.draft[static_cast<int64_t>(b) * k + tid];
    if (tid >= 64 && tid <= 64 + k) sU[tid - 64] = P.uniforms[static_cast<int64_t>(b) * (k + 1) + tid - 64];
    __syncthreads();
    pr = check_request(P, s_L, s_cap, sTok);
    pdl_wait();  // the streaming pass's partials
    const int nc = P.nc;
    const Partial *base = P.part + static_cast<int64_t>(b) * (2 * k + 1) * nc;
    for (int r = warp; r < 2 * k + 1; r += kFusedWarps) {
      const Partial *rp = base + static_cast<int64_t>(r) * nc;
      float m = -INFINITY, s = 0.0f, x = -INFINITY;
      int unused = kNoIndex;
      for (int j = lane; j < nc; j += 32) {
        const float4 q = ld_part(rp + j);
        merge_stats(m, s, unused, q.x, q.y, kNoIndex, c);
        x = fmaxf(x, q.w);
      }
      warp_allmerge<false>(m, s, unused, c);
      x = warp_allmax(x);
      if (lane == 0) {
        sM[r] = m;
        sS[r] = s;
        sIS[r] = 1.0f / s;
        sX[r] = x;
        if (FILT) sTh[r] = row_theta(P.theta, static_cast<int64_t>(b) * (2 * k + 1) + r);
      }
    }
    __syncthreads();
  } else {
    pdl_wait();  // the inputs may be the previous kernel's outputs
    pdl_launch_dependents();
    pr = read_request(P, b, sTok, sU, SAMPLE);
  }
  if (pr.bad) {  // every CTA of the cluster leaves here; no shared memory was exchanged
    if (rank == 0) write_common<SAMPLE>(P, b, pr.bad, pr.L, 0, 0, sTok, sP, sQ, true, -1);
    return;
  }
  const int L = pr.L;
  const int nrows = SAMPLE ? 2 * L + 1 : L + 1;  // target rows 0..L, then draft rows 0..L-1
  auto row_of = [&](int rr) {
    return rr <= L ? row_ptr<DT>(P.target, P.t_req, P.row, b, rr)
                   : row_ptr<DT>(P.draftl, P.d_req, P.row, b, rr - L - 1);
  };
  const int lo = min(P.V, rank * P.slice), hi = min(P.V, lo + P.slice);
  const int G = P.groups;  // rounds of 16-byte groups per lane
  if (!ACCEPT) {
    // the drafted tokens' logits (thread rr reads row rr's), in flight with the stream
    float xtok = -INFINITY;
    if (SAMPLE && tid < nrows) {
      const int pos = tid <= L ? tid : tid - L - 1;
      if (pos < L) xtok = load_one<DT>(row_of(tid), sTok[pos]);
    }

    // ---- 1. row statistics over the slice, kRowBatch rows at a time
    for (int rr0 = 0; rr0 < nrows; rr0 += kRowBatch) {
      RowStats R[kRowBatch];
      const char *rp[kRowBatch];
#pragma unroll
      for (int r = 0; r < kRowBatch; ++r) {
        R[r] = row_stats_empty();
        rp[r] = rr0 + r < nrows ? row_of(rr0 + r) : nullptr;
      }
      lane_rows_stats<DT, SAMPLE, VEC, kRowBatch>(rp, lo, hi, G, c, R);
#pragma unroll
      for (int r = 0; r < kRowBatch; ++r) {
        if (rr0 + r < nrows) {
          float m = R[r].m, s = R[r].s.x + R[r].s.y;
          int i = R[r].i;
          if (SAMPLE) warp_allmerge<false>(m, s, i, c);  // sampling needs no argmax
          else warp_allargmax(m, i);
          if (lane == 0) s_wpart[warp * rows_max + rr0 + r] = RowPart{m, s, i, 0.0f};
        }
      }
    }
    if (SAMPLE && tid < nrows) sX[tid] = xtok;
    __syncthreads();

    // ---- 2. the CTA's statistics of each row, pushed into every CTA
    for (int rr = warp; rr < nrows; rr += kFusedWarps) {
      RowPart x = lane < kFusedWarps ? s_wpart[lane * rows_max + rr] : kEmpty;
      if (SAMPLE) warp_allmerge<false>(x.m, x.s, x.i, c);
      else warp_allargmax(x.m, x.i);
      if (lane < CS) *cluster.map_shared_rank(&s_cpart[rank * rows_max + rr], lane) = x;
    }
    cluster.sync();
    // every CTA merges the slices (lane r holds rank r) and decides alike
    for (int rr = warp; rr < nrows; rr += kFusedWarps) {
      RowPart x = lane < CS ? s_cpart[lane * rows_max + rr] : kEmpty;
      if (SAMPLE) warp_allmerge<false>(x.m, x.s, x.i, c);
      else warp_allargmax(x.m, x.i);
      if (lane == 0) {
        sM[rr] = x.m;
        sS[rr] = x.s;
        sIS[rr] = 1.0f / x.s;
        sA[rr] = x.i == kNoIndex ? 0 : x.i;
      }
    }
    __syncthreads();
  }
  // the statistics of draft row i: after the target rows 0..L here, after
  // rows 0..k in the streaming pass's layout
  auto drow = [&](int i) { return (ACCEPT ? k : L) + 1 + i; };
  // Every warp tests the positions itself (lane i: positions i, i + 32),
  // so no barrier separates the test from the draw; warp 0 keeps p and q
  // for the outputs and writes the request's outputs.
  int m = L;  // the first rejected position
  for (int i0 = 0; i0 < L; i0 += 32) {
    const int i = i0 + lane;
    bool ok = true;
    if (i < L) {
      if (SAMPLE) {
        // (a drafted token below its row's threshold has probability 0)
        const float p = !FILT || sX[i] >= sTh[i] ? ex2((sX[i] - sM[i]) * c) * sIS[i] : 0.0f;
        const float q =
            !FILT || sX[drow(i)] >= sTh[drow(i)] ? ex2((sX[drow(i)] - sM[drow(i)]) * c) * sIS[drow(i)] : 0.0f;
        if (warp == 0) {
          sP[i] = p;
          sQ[i] = q;
        }
        ok = sU[i] * q < p;
      } else {
        ok = sA[i] == sTok[i];
      }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, !ok);
    if (rej && m == L) m = i0 + __ffs(rej) - 1;
  }
  const int ne = max(0, min(m + 1, pr.cap));
  if (rank == 0 && warp == 0) {
    __syncwarp();
    write_common<SAMPLE>(P, b, 0, L, m, ne, sTok, sP, sQ, !SAMPLE, sA[m], lane, 32);
  }
  if (!SAMPLE) return;

  // ---- 3. the final draw: residual after a rejection, p_L after a full accept
  Weights W = m < L ? Weights{row_of(m), row_of(L + 1 + m), sM[m], sM[drow(m)], sIS[m],
                              sIS[drow(m)], c, FILT ? sTh[m] : -INFINITY, FILT ? sTh[drow(m)] : -INFINITY}
                    : Weights{row_of(L), nullptr, sM[L], 0.0f, sIS[L], 0.0f, c, FILT ? sTh[L] : -INFINITY,
                              -INFINITY};
  float wmass = 0.0f, rmass = 0.0f, total = 0.0f;
  for (int attempt = 0; attempt < 2; ++attempt) {
    wmass = warp_sum(lane_weight_sum<DT, VEC, FILT>(W, lo, hi, G, s_gsum));  // this warp's range
    const float ws = wmass;
    if (lane == 0) s_red[warp] = ws;
    __syncthreads();
    if (warp == 0) {
      const float z = warp_sum(lane < kFusedWarps ? s_red[lane] : 0.0f);
      if (lane < CS) *cluster.map_shared_rank(&s_z[attempt][rank], lane) = z;
    }
    cluster.sync();
    rmass = lane < CS ? s_z[attempt][lane] : 0.0f;  // lane r: rank r's mass
    total = __shfl_sync(0xffffffffu, warp_inclusive_scan(rmass, lane), 31);
    if (!(total > 0.0f) && m < L && attempt == 0) {
      // zero residual mass (only through rounding): draw from p_m instead
      W.b = nullptr;
      W.beta = 0.0f;
      continue;
    }
    break;
  }
  // the rank whose slice holds u * total
  const float incl_r = warp_inclusive_scan(rmass, lane);
  const float thr = sU[k] * total;
  const unsigned hit_r = __ballot_sync(0xffffffffu, lane < CS && rmass > 0.0f && incl_r > thr);
  const unsigned pos_r = __ballot_sync(0xffffffffu, lane < CS && rmass > 0.0f);
  int draw_rank;
  float tl = INFINITY;  // threshold within the drawing rank's slice
  if (hit_r) {
    draw_rank = __ffs(hit_r) - 1;
    const float before = __shfl_sync(0xffffffffu, incl_r, max(draw_rank - 1, 0));
    tl = thr - (draw_rank > 0 ? before : 0.0f);
  } else {
    draw_rank = pos_r ? 31 - __clz(pos_r) : 0;  // rounding: the last rank with mass
  }
  if (rank != draw_rank) return;  // no CTA touches another's shared memory from here on
  // (the fallback `lo` is unreachable: the drawing rank has mass, so one of its warps has)
  // (the warp masses of the last attempt are in s_red; the drawing warp
  // writes the token)
  const int tok = range_draw<kFusedThreads, EPG, false>(wmass, tl, lo, G, lo, s_gsum, [&](int g, float *w) {
    float x[EPG], y[EPG];
    unpack16<DT>(load_group<DT, VEC>(W.a, lo + g * EPG, hi), x);
    if (W.b) unpack16<DT>(load_group<DT, VEC>(W.b, lo + g * EPG, hi), y);
    weights_group<EPG, FILT>(W, x, y, w);
  }, s_red);
  if (tok >= 0 && lane == 0) {
    if (m < ne) P.out_tokens[static_cast<int64_t>(b) * (k + 1) + m] = tok;
    if (P.resid_mass) P.resid_mass[b] = (m < L && W.b != nullptr) ? total : 0.0f;
    if (P.final_prob)
      P.final_prob[b] = weight_at<DT, FILT>(W, load_one<DT>(W.a, tok), W.b ? load_one<DT>(W.b, tok) : 0.0f) / total;
  }
}

// ------------------------------------------------------------------- host

constexpr int kAcceptMaxSlice = 32768;  // largest slice per CTA of the cluster accept kernel

// Dynamic shared memory: the warp and slice statistics of every row (only
// when streamed here), then the draw's group sums (sampling).
size_t chain_fused_smem(int k, bool sample, bool accept, int groups) {
  const int rows = sample ? 2 * k + 1 : k + 1;
  const size_t parts = accept ? 0 : sizeof(RowPart) * static_cast<size_t>(kFusedWarps + kFusedMaxCluster) * rows;
  return parts + (sample ? sizeof(float) * static_cast<size_t>(kFusedThreads) * groups : 0);
}

static int lane_groups(int V, int dtype, int cluster) {
  const int slice = ((V + cluster - 1) / cluster + 7) / 8 * 8;
  const int epg = dtype == SPEC_DTYPE_F32 ? 4 : 8;
  return ((slice + epg - 1) / epg + kFusedThreads - 1) / kFusedThreads;
}

template <int DT, bool VEC, bool SAMPLE, bool ACCEPT, bool FILT>
static cudaError_t prepare(int cluster, size_t smem) {
  auto kern = chain_fused_kernel<DT, VEC, SAMPLE, ACCEPT, FILT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess && cluster > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

static void cluster_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, int cluster, unsigned grid,
                           size_t smem, cudaStream_t st, bool pdl) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
}

// Calls f.template operator()<DT, VEC, SAMPLE, ACCEPT, FILT>() for the
// runtime choice (ACCEPT implies SAMPLE; FILT only with ACCEPT).
template <class F>
static cudaError_t dispatch(int dtype, bool vec, bool sample, bool accept, bool filt, F &&f) {
  if (dtype == SPEC_DTYPE_BF16) {
    if (vec) {
      if (accept)
        return filt ? f.template operator()<SPEC_DTYPE_BF16, true, true, true, true>()
                    : f.template operator()<SPEC_DTYPE_BF16, true, true, true, false>();
      return sample ? f.template operator()<SPEC_DTYPE_BF16, true, true, false, false>()
                    : f.template operator()<SPEC_DTYPE_BF16, true, false, false, false>();
    }
    if (accept)
      return filt ? f.template operator()<SPEC_DTYPE_BF16, false, true, true, true>()
                  : f.template operator()<SPEC_DTYPE_BF16, false, true, true, false>();
    return sample ? f.template operator()<SPEC_DTYPE_BF16, false, true, false, false>()
                  : f.template operator()<SPEC_DTYPE_BF16, false, false, false, false>();
  }
  if (vec) {
    if (accept)
      return filt ? f.template operator()<SPEC_DTYPE_F32, true, true, true, true>()
                  : f.template operator()<SPEC_DTYPE_F32, true, true, true, false>();
    return sample ? f.template operator()<SPEC_DTYPE_F32, true, true, false, false>()
                  : f.template operator()<SPEC_DTYPE_F32, true, false, false, false>();
  }
  if (accept)
    return filt ? f.template operator()<SPEC_DTYPE_F32, false, true, true, true>()
                : f.template operator()<SPEC_DTYPE_F32, false, true, true, false>();
  return sample ? f.template operator()<SPEC_DTYPE_F32, false, true, false, false>()
                : f.template operator()<SPEC_DTYPE_F32, false, false, false, false>();
}

// How many clusters of `cluster` CTAs of the kernel fit on the device at
// once (cached per device and shape).
static int resident_clusters(int dtype, bool vec, bool sample, bool accept, bool filt, int k, int V, int cluster) {
  struct Key {
    int dev, dtype, vec, sample, accept, filt, k, V, cluster, n;
  };
  static std::mutex mu;
  static std::vector<Key> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> g(mu);
    for (const Key &q : cache)
      if (q.dev == dev && q.dtype == dtype && q.vec == vec && q.sample == sample && q.accept == accept &&
          q.filt == filt && q.k == k && q.V == V && q.cluster == cluster)
        return q.n;
  }
  const size_t smem = chain_fused_smem(k, sample, accept, lane_groups(V, dtype, cluster));
  int n = 0;
  dispatch(dtype, vec, sample, accept, filt, [&]<int DT, bool VEC, bool SAMPLE, bool ACCEPT, bool FILT>() {
    cudaError_t e = prepare<DT, VEC, SAMPLE, ACCEPT, FILT>(cluster, smem);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg;
      cudaLaunchAttribute attr[2];
      cluster_config(cfg, attr, cluster, static_cast<unsigned>(cluster), smem, nullptr, false);
      e = cudaOccupancyMaxActiveClusters(&n, chain_fused_kernel<DT, VEC, SAMPLE, ACCEPT, FILT>, &cfg);
    }
    if (e != cudaSuccess) n = 0;
    return e;
  });
  cudaGetLastError();  // a refused query leaves no error behind
  std::lock_guard<std::mutex> g(mu);
  cache.push_back(Key{dev, dtype, vec, sample, accept, filt, k, V, cluster, n});
  return n;
}

// Cluster geometry: the largest cluster (at most 16 CTAs, at least
// kFusedMinSlice logits each, and for the accept kernel at most
// kAcceptMaxSlice) for which every request's cluster is resident at once.
static bool plan(ChainParams &P, bool sample, bool vec, bool accept) {
  const bool filt = accept && P.theta != nullptr;
  int cs = (P.V + kFusedMinSlice - 1) / kFusedMinSlice;
  cs = cs < 1 ? 1 : (cs > kFusedMaxCluster ? kFusedMaxCluster : cs);
  const int cs_min = accept ? (P.V + kAcceptMaxSlice - 1) / kAcceptMaxSlice : 1;
  for (; cs >= cs_min; --cs)
    if (resident_clusters(P.dtype, vec, sample, accept, filt, P.k, P.V, cs) >= P.B) break;
  if (cs < cs_min || cs < 1) return false;
  P.cluster = cs;
  P.slice = ((P.V + cs - 1) / cs + 7) / 8 * 8;
  P.groups = lane_groups(P.V, P.dtype, cs);
  return true;
}

bool chain_fused_plan(ChainParams &P, bool sample, bool vec) { return plan(P, sample, vec, false); }
bool chain_accept_plan(ChainParams &P, bool vec) { return plan(P, true, vec, true); }

static cudaError_t launch(const ChainParams &P, bool sample, bool vec, bool accept, cudaStream_t st) {
  const size_t smem = chain_fused_smem(P.k, sample, accept, P.groups);
  const bool filt = accept && P.theta != nullptr;
  return dispatch(P.dtype, vec, sample, accept, filt, [&]<int DT, bool VEC, bool SAMPLE, bool ACCEPT, bool FILT>() {
    cudaError_t e = prepare<DT, VEC, SAMPLE, ACCEPT, FILT>(P.cluster, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    cluster_config(cfg, attr, P.cluster, static_cast<unsigned>(P.B * P.cluster), smem, st, !trace_enabled());
    const char *name = ACCEPT ? "chain_sample_accept_cluster" : SAMPLE ? "chain_fused_sample" : "chain_fused_greedy";
    return trace_launch_ex(name, st, [&] {
      return cudaLaunchKernelEx(&cfg, chain_fused_kernel<DT, VEC, SAMPLE, ACCEPT, FILT>, P);
    });
  });
}

cudaError_t launch_chain_fused(const ChainParams &P, bool sample, bool vec, cudaStream_t st) {
  return launch(P, sample, vec, false, st);
}

cudaError_t launch_chain_accept_cluster(const ChainParams &P, bool vec, cudaStream_t st) {
  return launch(P, true, vec, true, st);
}

}  // namespace sv
