// Tree verification: one thread-block cluster per request walks the draft
// tree from the root ("Speculative Decoding II", EAGLE section: the sampling
// rule is applied recursively at every node, as in SpecInfer).
//
// Each CTA of the cluster owns one slice of the vocabulary and each of its
// threads one contiguous segment of that slice.  Only the rows of the nodes
// the walk visits are read.  Per visited node u:
//   1. one pass over the segment reduces t_u, and d_u when u has children,
//      to (max, sum 2^((x - max) c), first argmax), both rows' loads in
//      flight together; warps merge with redux and shuffle reductions, warp
//      0 merges the warps and pushes the CTA's statistics into every CTA of
//      the cluster (distributed shared memory), and after one cluster
//      barrier every CTA holds all slices' statistics and takes the same
//      decisions;
//   2. children are tested in increasing id order.  The residual after j
//      rejected children is kept in closed form,
//          p^(j) = max(0, p - c_j q) / Z_j,   c_0 = 0, Z_0 = 1,
//          c_{j+1} = c_j + Z_j,  Z_{j+1} = sum_v max(0, p_v - c_{j+1} q_v),
//      which is what repeating p <- norm(max(0, p - q)) with q fixed gives
//      (induction on j; a term with p_v <= c_j q_v stays at zero).  Child x
//      is accepted iff u * q(x) * Z_j < max(0, p(x) - c_j q(x)), i.e.
//      u < min(1, p^(j)(x) / q(x)).  A rejection costs one segment pass and
//      one cluster exchange for Z_{j+1}; the first rejection at a node also
//      stores the normalised p and q of the slice in shared memory, so later
//      rejections and the final draw need no more exponentials or loads;
//   3. an accepted child is descended into; otherwise the final token is
//      drawn from p^(j) with the last uniform: the rank whose slice holds the
//      crossing is found from the per-rank masses already exchanged; in that
//      CTA a block scan of the per-thread segment masses finds the thread
//      whose segment holds it, and one warp scans that segment.
// Greedy mode (T <= 0): per node one argmax exchange, then the first child
// whose token equals the argmax.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kMaxCluster = 16;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kPrefetchKids = 2;  // children whose slices are fetched into L2 while the node is decided

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

// ------------------------------------------------ warp-wide reductions
// The results land in every lane.

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

// ------------------------------------------------- per-thread segments

// Running statistics of one row over a thread's segment.
struct RowStats {
  float m;   // max logit
  float2 s;  // sum of 2^((x - m) c), two lanes
  int i;     // first index of the max
};

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

// Folds logits [a, b) of trow into T and, unless drow is null, of drow into
// D.  a is a multiple of 8; a batch of both rows is loaded before either is
// folded.
template <int DT, bool SOFTMAX, bool VEC>
__device__ __forceinline__ void segment_stats(const char *trow, const char *drow, int a, int b, float c,
                                              RowStats &T, RowStats &D) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  constexpr int ES = Elems<DT>::kSize;
  constexpr uint32_t kNegInf = DT == SPEC_DTYPE_F32 ? 0xff800000u : 0xff80ff80u;  // -inf words
  const uint4 neg = make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
  float unused = 0.0f;
  int vt = a;
  if (VEC) {
    const int ng = b > a ? (b - a) / EPG : 0;
    const uint4 *gt = reinterpret_cast<const uint4 *>(trow + static_cast<int64_t>(a) * ES);
    const uint4 *gd = drow ? reinterpret_cast<const uint4 *>(drow + static_cast<int64_t>(a) * ES) : nullptr;
    for (int g0 = 0; g0 < ng; g0 += kBatch) {
      uint4 xt[kBatch], xd[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) xt[u] = g0 + u < ng ? __ldg(gt + g0 + u) : neg;
      if (gd) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) xd[u] = g0 + u < ng ? __ldg(gd + g0 + u) : neg;
      }
      fold_batch<DT, SOFTMAX, 1>(xt, a + g0 * EPG, c, T.m, T.s, T.i, -1, unused);
      if (gd) fold_batch<DT, SOFTMAX, 1>(xd, a + g0 * EPG, c, D.m, D.s, D.i, -1, unused);
    }
    vt = a + ng * EPG;
  }
  for (int v = vt; v < b; ++v) {
    fold_one<SOFTMAX>(T, load_one<DT>(trow, v), v, c);
    if (drow) fold_one<SOFTMAX>(D, load_one<DT>(drow, v), v, c);
  }
}

// p_v = 2^(t_v c - Mtc) iSt and q_v = 2^(d_v c - Mdc) iSd over logits
// [a, b); returns this thread's sum of max(0, p_v - cres q_v).  STORE also
// writes p_v, q_v to sp, sq at (v - a) * kTreeThreads + threadIdx.x
// (consecutive threads, consecutive words).
template <int DT, bool VEC, bool STORE>
__device__ __forceinline__ float segment_residual(const char *trow, const char *drow, int a, int b, float Mtc,
                                                  float Mdc, float c, float iSt, float iSd, float cres,
                                                  float *sp, float *sq) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  constexpr int ES = Elems<DT>::kSize;
  float part = 0.0f;
  auto one = [&](float t, float d, int o) {
    const float pv = ex2(fmaf(t, c, -Mtc)) * iSt;
    const float qv = ex2(fmaf(d, c, -Mdc)) * iSd;
    if (STORE) {
      sp[o * kTreeThreads + threadIdx.x] = pv;
      sq[o * kTreeThreads + threadIdx.x] = qv;
    }
    part += fmaxf(0.0f, pv - cres * qv);
  };
  int vt = a;
  if (VEC) {
    const int ng = b > a ? (b - a) / EPG : 0;
    const uint4 *gt = reinterpret_cast<const uint4 *>(trow + static_cast<int64_t>(a) * ES);
    const uint4 *gd = reinterpret_cast<const uint4 *>(drow + static_cast<int64_t>(a) * ES);
    for (int g0 = 0; g0 < ng; g0 += kBatch) {
      uint4 xt[kBatch], xd[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        xt[u] = g0 + u < ng ? __ldg(gt + g0 + u) : make_uint4(0u, 0u, 0u, 0u);
        xd[u] = g0 + u < ng ? __ldg(gd + g0 + u) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (g0 + u < ng) {
          float t[EPG], d[EPG];
          unpack16<DT>(xt[u], t);
          unpack16<DT>(xd[u], d);
#pragma unroll
          for (int e = 0; e < EPG; ++e) one(t[e], d[e], (g0 + u) * EPG + e);
        }
      }
    }
    vt = a + ng * EPG;
  }
  for (int v = vt; v < b; ++v) one(load_one<DT>(trow, v), load_one<DT>(drow, v), v - a);
  return part;
}

template <int DT, bool VEC, bool GREEDY>
__global__ void __launch_bounds__(kTreeThreads) tree_walk_kernel(const TreeParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  const int ncl = P.cluster;
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.x / ncl;
  const int N = P.N, W = P.max_depth + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ int dyn[];
  int *s_par = dyn;                                       // [N]
  int *s_tok = dyn + N;                                   // [N]
  int *s_kids = dyn + 2 * N;                              // [N] children of the current node, ascending
  float *s_kt = reinterpret_cast<float *>(dyn + 3 * N);   // [N] target logit of each child's token
  float *s_kd = reinterpret_cast<float *>(dyn + 4 * N);   // [N] draft logit of each child's token
  float *s_uni = reinterpret_cast<float *>(dyn + 5 * N);  // [N + 1] the request's uniforms
  float *s_p = s_uni + N + 1;                             // [seg][threads] staged p of the segments
  float *s_q = s_p + static_cast<size_t>(P.seg) * kTreeThreads;  // [seg][threads] staged q
  __shared__ Slot s_all[2][kMaxCluster];  // [exchange parity][source rank]
  __shared__ Slot s_part[kTreeWarps];
  __shared__ float s_red[kTreeWarps];
  __shared__ unsigned s_pos[kTreeWarps];
  __shared__ int s_path[SPEC_MAX_DEPTH + 1], s_out[SPEC_MAX_DEPTH + 1];
  __shared__ int s_bad, s_cnt[kTreeWarps], s_final;
  const Slot kEmpty{-INFINITY, 0.0f, -INFINITY, 0.0f, kNoIndex, 0.0f, 0, 0};

  // ---- load and validate the tree (every CTA does the same)
  const int32_t *par = P.parents + static_cast<int64_t>(b) * N;
  const int32_t *tok = P.node_tok + static_cast<int64_t>(b) * N;
  const float *uni = P.uniforms + static_cast<int64_t>(b) * (N + 1);
  if (tid == 0) s_bad = SPEC_STATUS_OK;
  __syncthreads();
  for (int i = tid; i < N; i += kTreeThreads) {
    const int p = par[i], t = tok[i];
    s_par[i] = p;
    s_tok[i] = t;
    if (i == 0 ? p != -1 : (p < 0 || p >= i)) atomicMax(&s_bad, SPEC_STATUS_BAD_TREE);
  }
  if (!GREEDY)
    for (int i = tid; i <= N; i += kTreeThreads) s_uni[i] = uni[i];
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
  const int sa = min(hi, lo + tid * P.seg), sb = min(hi, sa + P.seg);  // this thread's segment
  const float c = P.c;
  int phase = 0;

  // Warp 0's lanes < ncl push v into slot `rank` of every CTA's s_all, then
  // one cluster barrier; returns the parity written.  A slot parity is
  // rewritten two exchanges later, after a barrier that every reader of it
  // has passed.
  auto push_and_sync = [&](const Slot &v) {
    const int ph = phase & 1;
    if (warp == 0 && lane < ncl) *cluster.map_shared_rank(&s_all[ph][rank], lane) = v;
    cluster.sync();
    ++phase;
    return ph;
  };
  // Sum of x over the cluster, in every thread; lane r of every warp also
  // gets rank r's part.
  auto cluster_sum = [&](float x, float &part_of_lane) {
    const float ws = warp_sum(x);
    if (lane == 0) s_red[warp] = ws;
    __syncthreads();
    Slot z = kEmpty;
    if (warp == 0) z.z = warp_sum(lane < kTreeWarps ? s_red[lane] : 0.0f);
    const int ph = push_and_sync(z);
    part_of_lane = lane < ncl ? s_all[ph][lane].z : 0.0f;
    return warp_sum(part_of_lane);
  };
  // Children of `node` in increasing id order into s_kids; their number.
  auto children = [&](int node) {
    int nk = 0;
    for (int base = node + 1; base < N; base += kTreeThreads) {
      const int cidx = base + tid;
      const bool is_kid = cidx < N && s_par[cidx] == node;
      const unsigned bal = __ballot_sync(0xffffffffu, is_kid);
      if (lane == 0) s_cnt[warp] = __popc(bal);
      __syncthreads();
      const int cw = lane < kTreeWarps ? s_cnt[lane] : 0;
      const int before = __reduce_add_sync(0xffffffffu, lane < warp ? cw : 0);
      const int total = __reduce_add_sync(0xffffffffu, cw);
      if (is_kid) s_kids[nk + before + __popc(bal & ((1u << lane) - 1u))] = cidx;
      nk += total;
      __syncthreads();
    }
    return nk;
  };

  int node = 0, nacc = 0, final_tok = -1, draw_rank = 0;
  if (tid == 0) s_path[0] = 0;
  for (;;) {
    const int nkids = children(node);
    const char *trow = node_row<DT>(P.target, P.t_req, P.row, b, node);
    const char *drow = (!GREEDY && nkids > 0) ? node_row<DT>(P.draftl, P.d_req, P.row, b, node) : nullptr;
    // the walk is likely to continue at the first children: have L2 fetch
    // this CTA's slice of their rows while the current node is worked on
    if (VEC && tid < min(nkids, kPrefetchKids) && hi > lo) {
      const int ch = s_kids[tid];
      const int64_t off = static_cast<int64_t>(lo) * Elems<DT>::kSize;
      const int bytes = (hi - lo) * Elems<DT>::kSize;
      prefetch_l2(node_row<DT>(P.target, P.t_req, P.row, b, ch) + off, bytes);
      if (!GREEDY) prefetch_l2(node_row<DT>(P.draftl, P.d_req, P.row, b, ch) + off, bytes);
    }
    // the children's token logits: loaded now, stored after the segment pass
    float kt0 = 0.0f, kd0 = 0.0f;
    if (drow) {
      if (tid < nkids) {
        const int x = s_tok[s_kids[tid]];
        kt0 = load_one<DT>(trow, x);
        kd0 = load_one<DT>(drow, x);
      }
      for (int i = tid + kTreeThreads; i < nkids; i += kTreeThreads) {
        const int x = s_tok[s_kids[i]];
        s_kt[i] = load_one<DT>(trow, x);
        s_kd[i] = load_one<DT>(drow, x);
      }
    }

    // ---- row statistics: segment pass, warp merge, block merge, exchange
    RowStats T{-INFINITY, make_float2(0.0f, 0.0f), kNoIndex}, D = T;
    segment_stats<DT, !GREEDY, VEC>(trow, drow, sa, sb, c, T, D);
    if (drow && tid < nkids) {
      s_kt[tid] = kt0;
      s_kd[tid] = kd0;
    }
    const float th_m = T.m, th_s = T.s.x + T.s.y;  // this thread's own statistics of t
    {
      float m = T.m, s = th_s, dm = D.m, ds = D.s.x + D.s.y;
      int i = T.i, di = kNoIndex;
      if (GREEDY) warp_allargmax(m, i);
      else warp_allmerge<true>(m, s, i, c);
      if (drow) warp_allmerge<false>(dm, ds, di, c);
      if (lane == 0) s_part[warp] = Slot{m, s, dm, ds, i, 0.0f, 0, 0};
    }
    __syncthreads();
    Slot mine = kEmpty;
    if (warp == 0) {
      mine = lane < kTreeWarps ? s_part[lane] : kEmpty;
      int di = kNoIndex;
      if (GREEDY) warp_allargmax(mine.mt, mine.it);
      else warp_allmerge<true>(mine.mt, mine.st, mine.it, c);
      if (drow) warp_allmerge<false>(mine.md, mine.sd, di, c);
    }
    const int ph = push_and_sync(mine);
    const Slot r = lane < ncl ? s_all[ph][lane] : kEmpty;  // lane r: rank r's statistics

    if (GREEDY) {
      float M = r.mt;
      int A = r.it;
      warp_allargmax(M, A);
      if (A == kNoIndex) A = 0;
      int next = -1;
      for (int i0 = 0; i0 < nkids; i0 += 32) {
        const int i = i0 + lane;
        const unsigned hit = __ballot_sync(0xffffffffu, i < nkids && s_tok[s_kids[i]] == A);
        if (hit) {
          next = s_kids[i0 + __ffs(hit) - 1];
          break;
        }
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
      continue;
    }

    // ---- sampling: the node's p and q statistics over the whole row
    float Mt = r.mt, St = r.st, Md = r.md, Sd = r.sd;
    int it = r.it, id = kNoIndex;
    warp_allmerge<true>(Mt, St, it, c);
    if (drow) warp_allmerge<false>(Md, Sd, id, c);
    const float iSt = 1.0f / St, iSd = drow ? 1.0f / Sd : 0.0f;
    const int cta_it = __shfl_sync(0xffffffffu, r.it, rank);  // this slice's argmax
    // lane r: rank r's share of the current draw distribution (p so far)
    float rmass = lane < ncl ? r.st * ex2((r.mt - Mt) * c) * iSt : 0.0f;
    float my_mass = -1.0f;  // this thread's share of it; < 0: p, from the segment statistics

    float cres = 0.0f, Z = 1.0f;
    bool staged = false;  // s_p / s_q hold this node's segments
    int next = -1;
    for (int ki = 0; ki < nkids; ++ki) {
      const int ch = s_kids[ki];
      const float pt = ex2((s_kt[ki] - Mt) * c) * iSt;
      const float qt = ex2((s_kd[ki] - Md) * c) * iSd;
      if (s_uni[ch] * qt * Z < fmaxf(0.0f, pt - cres * qt)) {
        next = ch;
        break;
      }
      // rejected: next residual  max(0, p - (cres + Z) q), its mass over the cluster
      const float cnew = cres + Z;
      float part = 0.0f;
      if (staged) {
        for (int o = 0; o < sb - sa; ++o)
          part += fmaxf(0.0f, s_p[o * kTreeThreads + tid] - cnew * s_q[o * kTreeThreads + tid]);
      } else if (P.stage) {
        part = segment_residual<DT, VEC, true>(trow, drow, sa, sb, Mt * c, Md * c, c, iSt, iSd, cnew, s_p, s_q);
        staged = true;
      } else {
        part = segment_residual<DT, VEC, false>(trow, drow, sa, sb, Mt * c, Md * c, c, iSt, iSd, cnew, s_p, s_q);
      }
      float zr;
      const float Znew = cluster_sum(part, zr);
      if (Znew > 0.0f) {  // a zero-mass residual (rounding only) keeps the previous p
        cres = cnew;
        Z = Znew;
        rmass = zr;
        my_mass = part;
      }
    }
    if (next >= 0) {
      if (tid == 0) {
        s_out[nacc] = s_tok[next];
        s_path[nacc + 1] = next;
      }
      ++nacc;
      node = next;
      continue;
    }

    // ---- final draw from p^(j): the rank whose slice holds u * total
    const float incl_r = warp_inclusive_scan(rmass, lane);
    const float thr = s_uni[N] * __shfl_sync(0xffffffffu, incl_r, 31);
    const unsigned hit_r = __ballot_sync(0xffffffffu, lane < ncl && rmass > 0.0f && incl_r > thr);
    const unsigned pos_r = __ballot_sync(0xffffffffu, lane < ncl && rmass > 0.0f);
    float tl = INFINITY;  // threshold within the drawing rank's slice
    if (hit_r) {
      draw_rank = __ffs(hit_r) - 1;
      const float before = __shfl_sync(0xffffffffu, incl_r, max(draw_rank - 1, 0));
      tl = thr - (draw_rank > 0 ? before : 0.0f);
    } else {
      draw_rank = pos_r ? 31 - __clz(pos_r) : 0;  // rounding: the last rank with mass
    }
    if (rank == draw_rank) {
      // the thread whose segment holds the crossing: block scan of the masses
      const float mass =
          my_mass >= 0.0f ? my_mass : (th_m == -INFINITY ? 0.0f : th_s * ex2((th_m - Mt) * c) * iSt);
      const float incl = warp_inclusive_scan(mass, lane);
      const unsigned posw = __ballot_sync(0xffffffffu, mass > 0.0f);
      if (lane == 31) s_red[warp] = incl;
      if (lane == 0) s_pos[warp] = posw;
      __syncthreads();
      const float winc = warp_inclusive_scan(lane < kTreeWarps ? s_red[lane] : 0.0f, lane);
      const unsigned hit_w = __ballot_sync(0xffffffffu, lane < kTreeWarps && winc > tl);
      const unsigned nz_w = __ballot_sync(0xffffffffu, lane < kTreeWarps && s_pos[lane] != 0u);
      int wsel = -1, lsel = 0;
      float thr_local = INFINITY;
      if (hit_w) {
        wsel = __ffs(hit_w) - 1;
        if (warp == wsel) {
          const float wb = __shfl_sync(0xffffffffu, winc, max(wsel - 1, 0));
          const float base = wsel > 0 ? wb : 0.0f;
          const float G = base + incl;
          const unsigned hit = __ballot_sync(0xffffffffu, mass > 0.0f && G > tl);
          // (no hit: rounding between the two scans; the warp's last thread with mass)
          lsel = hit ? __ffs(hit) - 1 : (posw ? 31 - __clz(posw) : 31);
          const float gprev = __shfl_sync(0xffffffffu, G, max(lsel - 1, 0));
          thr_local = hit ? tl - (lsel > 0 ? gprev : base) : INFINITY;
        }
      } else if (nz_w) {  // rounding: the last thread with mass, its last positive weight
        wsel = 31 - __clz(nz_w);
        lsel = 31 - __clz(s_pos[wsel]);
      }
      if (warp == wsel) {
        const int tsel = wsel * 32 + lsel;
        const int a = min(hi, lo + tsel * P.seg), len = min(hi, a + P.seg) - a;
        const float Mtc = Mt * c, Mdc = Md * c;
        float run = 0.0f;
        int pick = -1, lastp = -1;
        for (int o0 = 0; o0 < len; o0 += 32) {
          const int o = o0 + lane;
          float w = 0.0f;
          if (o < len) {
            if (staged) {
              w = fmaxf(0.0f, s_p[o * kTreeThreads + tsel] - cres * s_q[o * kTreeThreads + tsel]);
            } else {
              w = ex2(fmaf(load_one<DT>(trow, a + o), c, -Mtc)) * iSt;
              if (cres > 0.0f)
                w = fmaxf(0.0f, w - cres * (ex2(fmaf(load_one<DT>(drow, a + o), c, -Mdc)) * iSd));
            }
          }
          const float inc = warp_inclusive_scan(w, lane);
          const unsigned hit = __ballot_sync(0xffffffffu, w > 0.0f && run + inc > thr_local);
          const unsigned pos = __ballot_sync(0xffffffffu, w > 0.0f);
          if (pos) lastp = o0 + 31 - __clz(pos);
          if (hit) {
            pick = o0 + __ffs(hit) - 1;
            break;
          }
          run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (pick < 0) pick = lastp;
        if (lane == 0) s_final = pick >= 0 ? a + pick : cta_it;
      } else if (wsel < 0 && tid == 0) {
        s_final = cta_it;  // no positive weight left in the slice (underflow only)
      }
      __syncthreads();
      final_tok = s_final;
    }
    break;
  }

  // The CTA that found the final token writes the request's outputs.  Every
  // exchange is a push followed by a cluster barrier, so no CTA touches
  // another's shared memory from here on and CTAs may leave independently.
  if (rank == draw_rank) {
    __syncthreads();  // s_path / s_out were written by thread 0
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
}

// Dynamic shared memory of the walk: parents, tokens, children and the
// children's two token logits (5 words per node), the uniforms (N + 1), plus
// the staged p and q of the CTA's segments when staging is on.
size_t tree_dynamic_smem(const TreeParams &P) {
  return sizeof(int) * (6 * static_cast<size_t>(P.N) + 1) +
         (P.stage ? 2 * sizeof(float) * static_cast<size_t>(P.seg) * kTreeThreads : 0);
}

template <int DT, bool VEC, bool GREEDY>
static cudaError_t launch_tree_t(const TreeParams &P, cudaStream_t st) {
  const size_t dyn = tree_dynamic_smem(P);
  auto kern = tree_walk_kernel<DT, VEC, GREEDY>;
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
  return trace_launch_ex(GREEDY ? "tree_walk_greedy" : "tree_walk_sample", st,
                         [&] { return cudaLaunchKernelEx(&cfg, kern, P); });
}

template <int DT, bool VEC>
static cudaError_t launch_tree_mode(const TreeParams &P, cudaStream_t st) {
  return P.greedy ? launch_tree_t<DT, VEC, true>(P, st) : launch_tree_t<DT, VEC, false>(P, st);
}

cudaError_t launch_tree(const TreeParams &P, bool vec, cudaStream_t st) {
  if (P.dtype == SPEC_DTYPE_BF16)
    return vec ? launch_tree_mode<SPEC_DTYPE_BF16, true>(P, st) : launch_tree_mode<SPEC_DTYPE_BF16, false>(P, st);
  return vec ? launch_tree_mode<SPEC_DTYPE_F32, true>(P, st) : launch_tree_mode<SPEC_DTYPE_F32, false>(P, st);
}

}  // namespace sv
