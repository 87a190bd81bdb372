// Tree verification: one thread-block cluster per request walks the draft
// tree from the root ("Speculative Decoding II", EAGLE section: the sampling
// rule is applied recursively at every node, as in SpecInfer).
//
// Each CTA of the cluster owns one slice of the vocabulary.  Only the rows of
// the nodes the walk visits are read.  Per visited node u:
//   1. every CTA reduces its slice of t_u (and d_u when u has children) to
//      (max, sum 2^((x - max) c), first argmax); the CTAs swap these through
//      distributed shared memory and merge them in rank order, so every CTA
//      holds the same row statistics and takes the same decisions;
//   2. children are tested in increasing id order.  The residual after j
//      rejected children is kept in closed form,
//          p^(j) = max(0, p - c_j q) / Z_j,   c_0 = 0, Z_0 = 1,
//          c_{j+1} = c_j + Z_j,  Z_{j+1} = sum_v max(0, p_v - c_{j+1} q_v),
//      which is what repeating p <- norm(max(0, p - q)) with q fixed gives
//      (induction on j; a term with p_v <= c_j q_v stays at zero).  Child x
//      is accepted iff u * q(x) * Z_j < max(0, p(x) - c_j q(x)), i.e.
//      u < min(1, p^(j)(x) / q(x)).  A rejection costs one slice pass and one
//      cluster exchange for Z_{j+1}; the first rejection at a node also
//      stores the slice's normalised p and q in shared memory, so later
//      rejections and the final draw need no more exponentials or loads;
//   3. an accepted child is descended into; otherwise the final token is
//      drawn from p^(j) with the last uniform: the rank whose slice holds the
//      crossing is found from the per-rank masses already exchanged, and that
//      CTA scans its slice.
// Greedy mode (T <= 0): per node one argmax exchange, then the first child
// whose token equals the argmax.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kMaxCluster = 16;
constexpr int kTreeThreads = 512;  // large CTAs: a slice's loads are in flight together
constexpr int kTreeWarps = kTreeThreads / 32;

struct __align__(16) Slot {
  float mt, st, md, sd;  // slice statistics of the target and draft rows
  int it;                // slice argmax of the target row
  float z;               // slice residual mass
  int pad0, pad1;
};

template <int DT>
__device__ __forceinline__ const char *node_row(const char *base, int64_t req, int64_t row, int b,
                                                int u) {
  return base + (static_cast<int64_t>(b) * req + static_cast<int64_t>(u) * row) * Elems<DT>::kSize;
}

// Asks L2 to fetch [p, p + bytes) ahead of use (no completion to wait for).
// p must be 16-byte aligned; bytes is rounded down to a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const char *p, int bytes) {
  bytes &= ~15;
  if (bytes > 0) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Writes p_v = 2^(t_v c - Mtc) iSt and q_v = 2^(d_v c - Mdc) iSd of the slice
// [lo, hi) into sp / sq (indexed from lo) and returns this thread's part of
// sum_v max(0, p_v - cres q_v).
template <int DT, bool VEC>
__device__ __forceinline__ float stage_slice(const char *trow, const char *drow, int lo, int hi, float Mtc,
                                             float Mdc, float c, float iSt, float iSd, float cres, float *sp,
                                             float *sq) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  constexpr int ES = Elems<DT>::kSize;
  float part = 0.0f;
  int vtail = lo;
  if (VEC) {
    const int ng = (hi - lo) / EPG;
    const uint4 *gt = reinterpret_cast<const uint4 *>(trow + static_cast<int64_t>(lo) * ES);
    const uint4 *gd = reinterpret_cast<const uint4 *>(drow + static_cast<int64_t>(lo) * ES);
    for (int g = threadIdx.x; g < ng; g += kTreeThreads) {
      float t[EPG], d[EPG];
      unpack16<DT>(__ldg(gt + g), t);
      unpack16<DT>(__ldg(gd + g), d);
#pragma unroll
      for (int e = 0; e < EPG; ++e) {
        const float pv = ex2(fmaf(t[e], c, -Mtc)) * iSt;
        const float qv = ex2(fmaf(d[e], c, -Mdc)) * iSd;
        sp[g * EPG + e] = pv;
        sq[g * EPG + e] = qv;
        part += fmaxf(0.0f, pv - cres * qv);
      }
    }
    vtail = lo + ng * EPG;
  }
  for (int v = vtail + threadIdx.x; v < hi; v += kTreeThreads) {
    const float pv = ex2(fmaf(load_one<DT>(trow, v), c, -Mtc)) * iSt;
    const float qv = ex2(fmaf(load_one<DT>(drow, v), c, -Mdc)) * iSd;
    sp[v - lo] = pv;
    sq[v - lo] = qv;
    part += fmaxf(0.0f, pv - cres * qv);
  }
  return part;
}

// Block sum; the result is valid in every thread.
__device__ __forceinline__ float block_sum(float v) {
  __shared__ float s[kTreeWarps];
  __shared__ float total;
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int w = 0; w < kTreeWarps; ++w) t += s[w];
    total = t;
  }
  __syncthreads();
  const float r = total;
  __syncthreads();
  return r;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kTreeThreads) tree_walk_kernel(const TreeParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  const int ncl = P.cluster;
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / ncl;
  const int N = P.N, W = P.max_depth + 1;
  const int tid = threadIdx.x;

  extern __shared__ int dyn[];
  int *s_par = dyn;          // [N]
  int *s_tok = dyn + N;      // [N]
  int *s_kids = dyn + 2 * N; // [N] children of the current node, ascending
  float *s_kt = reinterpret_cast<float *>(dyn + 3 * N);  // [N] target logit of each child's token
  float *s_kd = reinterpret_cast<float *>(dyn + 4 * N);  // [N] draft logit of each child's token
  float *s_p = reinterpret_cast<float *>(dyn + 5 * N);   // [slice] p of this CTA's slice (staged)
  float *s_q = s_p + P.slice;                            // [slice] q of this CTA's slice (staged)
  __shared__ Slot s_slot[2];
  __shared__ Slot s_all[kMaxCluster];
  __shared__ int s_path[SPEC_MAX_DEPTH + 1], s_out[SPEC_MAX_DEPTH + 1];
  __shared__ int s_bad, s_nkids, s_cnt[kTreeWarps];

  // ---- load and validate the tree (every CTA does the same)
  const int32_t *par = P.parents + static_cast<int64_t>(b) * N;
  const int32_t *tok = P.node_tok + static_cast<int64_t>(b) * N;
  if (tid == 0) s_bad = SPEC_STATUS_OK;
  __syncthreads();
  for (int i = tid; i < N; i += kTreeThreads) {
    const int p = par[i], t = tok[i];
    s_par[i] = p;
    s_tok[i] = t;
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) atomicMax(&s_bad, SPEC_STATUS_BAD_TREE);
  }
  __syncthreads();
  if (s_bad == SPEC_STATUS_OK) {
    for (int i = 1 + tid; i < N; i += kTreeThreads) {
      int d = 0, u = i;
      while (u != 0 && d <= P.max_depth) {
        u = s_par[u];
        ++d;
      }
      if (d > P.max_depth) atomicMax(&s_bad, SPEC_STATUS_BAD_TREE);
      else if (s_tok[i] < 0 || s_tok[i] >= P.V) atomicMax(&s_bad, SPEC_STATUS_TOKEN_RANGE);
    }
  }
  __syncthreads();
  int32_t *o_path = P.path_nodes + static_cast<int64_t>(b) * W;
  int32_t *o_tok = P.out_tokens + static_cast<int64_t>(b) * W;
  if (s_bad != SPEC_STATUS_OK) {
    if (rank == 0) {
      for (int j = tid; j < W; j += kTreeThreads) o_path[j] = o_tok[j] = -1;
      if (tid == 0) {
        P.accepted_len[b] = 0;
        P.n_emit[b] = 0;
        if (P.status) P.status[b] = s_bad;
      }
    }
    return;  // every CTA of the cluster leaves here; no shared memory was exchanged
  }

  const int lo = min(P.V, rank * P.slice), hi = min(P.V, lo + P.slice);
  const float c = P.c;
  const float *uni = P.uniforms + static_cast<int64_t>(b) * (N + 1);
  int phase = 0;
  // exchange: publish this CTA's slot, wait for the cluster, gather all slots
  auto exchange = [&](const Slot &mine) {
    if (tid == 0) s_slot[phase & 1] = mine;
    cluster.sync();
    if (tid < ncl) s_all[tid] = *cluster.map_shared_rank(&s_slot[phase & 1], tid);
    ++phase;
    __syncthreads();
  };

  int node = 0, nacc = 0, final_tok = -1, draw_rank = 0;
  if (tid == 0) s_path[0] = 0;
  for (;;) {
    // children of `node`, in increasing id order (block-wide ordered compaction)
    if (tid == 0) s_nkids = 0;
    __syncthreads();
    for (int base = node + 1; base < N; base += kTreeThreads) {
      const int cidx = base + tid;
      const bool is_kid = cidx < N && s_par[cidx] == node;
      const unsigned bal = __ballot_sync(0xffffffffu, is_kid);
      const int lane = tid & 31, warp = tid >> 5;
      if (lane == 0) s_cnt[warp] = __popc(bal);
      __syncthreads();
      int off = s_nkids;
      for (int w = 0; w < warp; ++w) off += s_cnt[w];
      if (is_kid) s_kids[off + __popc(bal & ((1u << lane) - 1u))] = cidx;
      __syncthreads();
      if (tid == 0) {
        int t = 0;
        for (int w = 0; w < kTreeWarps; ++w) t += s_cnt[w];
        s_nkids += t;
      }
      __syncthreads();
    }
    const int nkids = s_nkids;
    const char *trow = node_row<DT>(P.target, P.t_req, P.row, b, node);
    // the walk continues at one of these children: have L2 fetch this CTA's
    // slice of their rows while the current node is worked on
    if (VEC && tid < nkids && hi > lo) {
      const int ch = s_kids[tid];
      const int64_t off = static_cast<int64_t>(lo) * Elems<DT>::kSize;
      const int bytes = (hi - lo) * Elems<DT>::kSize;
      prefetch_l2(node_row<DT>(P.target, P.t_req, P.row, b, ch) + off, bytes);
      if (!P.greedy) prefetch_l2(node_row<DT>(P.draftl, P.d_req, P.row, b, ch) + off, bytes);
    }

    if (P.greedy) {
      float m = -INFINITY, s = 0.0f, xt = -INFINITY;
      int idx = kNoIndex;
      thread_chunk_stats<DT, false, VEC, kLoadCached, kTreeThreads>(trow, lo, hi, 1.0f, m, s, idx, -1, xt);
      block_merge<false, kTreeThreads>(m, s, idx, 1.0f, xt);
      Slot mine{m, 0.0f, 0.0f, 0.0f, idx, 0.0f, 0, 0};
      exchange(mine);
      float M = -INFINITY;
      int A = kNoIndex;
      for (int r = 0; r < ncl; ++r) merge_argmax(M, A, s_all[r].mt, s_all[r].it);
      if (A == kNoIndex) A = 0;
      int next = -1;
      for (int i = 0; i < nkids; ++i)
        if (s_tok[s_kids[i]] == A) {
          next = s_kids[i];
          break;
        }
      if (next < 0) {
        final_tok = A;
        break;
      }
      if (tid == 0) {
        s_out[nacc] = s_tok[next];
        s_path[nacc + 1] = next;
      }
      ++nacc;
      node = next;
      __syncthreads();
      continue;
    }

    // sampling: the children's token logits (their loads overlap the
    // statistics pass), then the row statistics of t_u and d_u
    const char *drow = nkids > 0 ? node_row<DT>(P.draftl, P.d_req, P.row, b, node) : nullptr;
    for (int i = tid; i < nkids; i += kTreeThreads) {
      const int x = s_tok[s_kids[i]];
      s_kt[i] = load_one<DT>(trow, x);
      s_kd[i] = load_one<DT>(drow, x);
    }
    Slot mine{-INFINITY, 0.0f, -INFINITY, 0.0f, kNoIndex, 0.0f, 0, 0};
    {
      float m = -INFINITY, s = 0.0f, xt = -INFINITY;
      int idx = kNoIndex;
      thread_chunk_stats<DT, true, VEC, kLoadCached, kTreeThreads>(trow, lo, hi, c, m, s, idx, -1, xt);
      block_merge<true, kTreeThreads>(m, s, idx, c, xt);
      if (tid == 0) {
        mine.mt = m;
        mine.st = s;
        mine.it = idx;
      }
      __syncthreads();
      if (drow) {
        m = -INFINITY;
        s = 0.0f;
        idx = kNoIndex;
        thread_chunk_stats<DT, true, VEC, kLoadCached, kTreeThreads>(drow, lo, hi, c, m, s, idx, -1, xt);
        block_merge<true, kTreeThreads>(m, s, idx, c, xt);
        if (tid == 0) {
          mine.md = m;
          mine.sd = s;
        }
      }
    }
    exchange(mine);
    float Mt = -INFINITY, St = 0.0f, Md = -INFINITY, Sd = 0.0f;
    int it = kNoIndex, id = kNoIndex;
    for (int r = 0; r < ncl; ++r) {
      merge_stats(Mt, St, it, s_all[r].mt, s_all[r].st, s_all[r].it, c);
      merge_stats(Md, Sd, id, s_all[r].md, s_all[r].sd, kNoIndex, c);
    }
    const float iSt = 1.0f / St, iSd = 1.0f / Sd;
    // per-rank mass of p (for a draw with no rejection at this node)
    float rank_mass[kMaxCluster];
    for (int r = 0; r < ncl; ++r) rank_mass[r] = s_all[r].st * ex2((s_all[r].mt - Mt) * c) * iSt;

    float cres = 0.0f, Z = 1.0f;
    bool staged = false;  // s_p / s_q hold this node's slice
    int next = -1;
    for (int ki = 0; ki < nkids; ++ki) {
      const int ch = s_kids[ki];
      const float pt = ex2((s_kt[ki] - Mt) * c) * iSt;
      const float qt = ex2((s_kd[ki] - Md) * c) * iSd;
      if (uni[ch] * qt * Z < fmaxf(0.0f, pt - cres * qt)) {
        next = ch;
        break;
      }
      // rejected: next residual  max(0, p - (cres + Z) q), its mass over the cluster
      const float cnew = cres + Z;
      float part = 0.0f;
      if (P.stage && staged) {
        for (int i = tid; i < hi - lo; i += kTreeThreads) part += fmaxf(0.0f, s_p[i] - cnew * s_q[i]);
      } else if (P.stage) {
        // first rejection here: normalise the slice into shared memory,
        // 16-byte groups of both rows at a time
        part = stage_slice<DT, VEC>(trow, drow, lo, hi, Mt * c, Md * c, c, iSt, iSd, cnew, s_p, s_q);
        staged = true;
      } else {
        Weights Wr{trow, drow, Mt, Md, iSt, cnew * iSd, c};
        part = thread_chunk_weight_sum<DT, VEC, kLoadCached, kTreeThreads>(Wr, lo, hi);
      }
      const float zs = block_sum(part);
      Slot z{0.0f, 0.0f, 0.0f, 0.0f, 0, zs, 0, 0};
      exchange(z);
      float Znew = 0.0f;
      for (int r = 0; r < ncl; ++r) Znew += s_all[r].z;
      if (Znew > 0.0f) {  // a zero-mass residual (rounding only) keeps the previous p
        cres = cnew;
        Z = Znew;
        for (int r = 0; r < ncl; ++r) rank_mass[r] = s_all[r].z;
      }
    }
    if (next >= 0) {
      if (tid == 0) {
        s_out[nacc] = s_tok[next];
        s_path[nacc + 1] = next;
      }
      ++nacc;
      node = next;
      __syncthreads();
      continue;
    }
    // final draw from p^(j): find the rank whose slice holds u * total
    float total = 0.0f;
    for (int r = 0; r < ncl; ++r) total += rank_mass[r];
    const float thr = uni[N] * total;
    float cum = 0.0f, base = 0.0f;
    int rsel = -1, rlast = 0;
    for (int r = 0; r < ncl; ++r) {
      if (rank_mass[r] > 0.0f) rlast = r;
      if (rsel < 0 && cum + rank_mass[r] > thr) {
        rsel = r;
        base = cum;
      }
      cum += rank_mass[r];
    }
    draw_rank = rsel >= 0 ? rsel : rlast;
    if (rank == draw_rank) {
      const float tl = rsel >= 0 ? thr - base : INFINITY;
      if (staged && cres > 0.0f) {
        const float cr = cres;
        final_tok = lo + block_select_with<kTreeThreads>(
                             [&](int v0, int h, float *w) {
#pragma unroll
                               for (int e = 0; e < 8; ++e)
                                 w[e] = v0 + e < h ? fmaxf(0.0f, s_p[v0 + e] - cr * s_q[v0 + e]) : 0.0f;
                             },
                             0, hi - lo, tl);
      } else {
        Weights Wf{trow, cres > 0.0f ? drow : nullptr, Mt, Md, iSt, cres > 0.0f ? cres * iSd : 0.0f, c};
        final_tok = block_select<DT, VEC, kTreeThreads>(Wf, lo, hi, tl);
      }
    }
    break;
  }

  // the CTA that found the final token writes the request's outputs
  if (rank == draw_rank) {
    for (int j = tid; j < W; j += kTreeThreads) {
      o_path[j] = j <= nacc ? s_path[j] : -1;
      o_tok[j] = j < nacc ? s_out[j] : (j == nacc ? final_tok : -1);
    }
    if (tid == 0) {
      P.accepted_len[b] = nacc;
      P.n_emit[b] = nacc + 1;
      if (P.status) P.status[b] = SPEC_STATUS_OK;
    }
  }
  cluster.sync();  // no CTA leaves while another may still read its slots
}

// Dynamic shared memory of the walk: parents, tokens, children and the
// children's two token logits (5 words per node), plus the staged p and q of
// the CTA's slice when staging is on.
size_t tree_dynamic_smem(const TreeParams &P) {
  return sizeof(int) * 5 * static_cast<size_t>(P.N) +
         (P.stage ? 2 * sizeof(float) * static_cast<size_t>(P.slice) : 0);
}

template <int DT, bool VEC>
static cudaError_t launch_tree_t(const TreeParams &P, cudaStream_t st) {
  const size_t dyn = tree_dynamic_smem(P);
  auto kern = tree_walk_kernel<DT, VEC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(dyn));
  if (e != cudaSuccess) return e;
  if (P.cluster > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(P.B * P.cluster));
  cfg.blockDim = dim3(kTreeThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return trace_launch_ex(P.greedy ? "tree_walk_greedy" : "tree_walk_sample", st,
                         [&] { return cudaLaunchKernelEx(&cfg, kern, P); });
}

cudaError_t launch_tree(const TreeParams &P, bool vec, cudaStream_t st) {
  if (P.dtype == SPEC_DTYPE_BF16)
    return vec ? launch_tree_t<SPEC_DTYPE_BF16, true>(P, st) : launch_tree_t<SPEC_DTYPE_BF16, false>(P, st);
  return vec ? launch_tree_t<SPEC_DTYPE_F32, true>(P, st) : launch_tree_t<SPEC_DTYPE_F32, false>(P, st);
}

}  // namespace sv
