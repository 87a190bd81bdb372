// Tree verification: one thread-block cluster per request walks the draft
// tree from the root ("Speculative Decoding II", EAGLE section: the sampling
// rule is applied recursively at every node, as in SpecInfer).
//
// Each CTA of the cluster owns one slice of the vocabulary and each of its
// warps one contiguous range of that slice (lanes interleaved, so loads stay
// coalesced).  Only the rows of the nodes the walk visits are read.  Per
// visited node u:
//   1. one pass reduces t_u, and d_u when u has children, to (max, sum
//      2^((x - max) c)) -- greedy mode: (max, first argmax) of t_u -- both
//      rows' loads in flight together;
//      warps merge with redux and shuffle reductions, warp 0 merges the
//      warps and pushes the CTA's statistics into every CTA of the cluster
//      (distributed shared memory), and after one cluster barrier every CTA
//      holds all slices' statistics and takes the same decisions;
//   2. children are tested in increasing id order.  The residual after j
//      rejected children is kept in closed form,
//          p^(j) = max(0, p - c_j q) / Z_j,   c_0 = 0, Z_0 = 1,
//          c_{j+1} = c_j + Z_j,  Z_{j+1} = sum_v max(0, p_v - c_{j+1} q_v),
//      which is what repeating p <- norm(max(0, p - q)) with q fixed gives
//      (induction on j; a term with p_v <= c_j q_v stays at zero).  Child x
//      is accepted iff u * q(x) * Z_j < max(0, p(x) - c_j q(x)), i.e.
//      u < min(1, p^(j)(x) / q(x)).  A rejection costs one pass over the
//      slice and one cluster exchange for Z_{j+1}; the first rejection at a
//      node also stores the normalised p and q of the slice in shared
//      memory, so later rejections and the final draw need no more
//      exponentials or loads;
//   3. an accepted child is descended into; otherwise the final token is
//      drawn from p^(j) with the last uniform: the rank whose slice holds the
//      crossing is found from the per-rank masses already exchanged; in that
//      CTA a scan of the per-warp masses finds the warp whose range holds
//      it, and that warp walks its range.
// Siblings drawn without replacement (P.wor): a rejected sibling's token is
// also removed from q (q renormalised), since the next sibling was drawn from
// that distribution; then c_{j+1} = c_j + Z_j / Q_j with Q_j the q mass not
// yet removed, the acceptance test is u q(x) Z_j < max(0, p(x) - c_j q(x)) Q_j,
// and a removed token's residual keeps the coefficient of its removal (a
// correction per removed token, in the lane owning it).
// Greedy mode (T <= 0): per node one argmax exchange, then the first child
// whose token equals the argmax.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "segments.cuh"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kMaxCluster = 16;
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

// Where p_v, q_v of element e of group g are staged: the slice's groups in
// lane_group order, element-major within each warp round, so that
// consecutive lanes touch consecutive words.
__device__ __forceinline__ int stage_index(int g, int e, int epg) { return (((g >> 5) * epg + e) << 5) + (g & 31); }

// p_v = 2^((t_v - Mt) c) iSt and q_v = 2^((d_v - Md) c) iSd over this lane's
// groups (logits >= hi read as -inf, so give 0); returns the lane's sum of
// max(0, p_v - cres q_v).  STORE also writes p_v, q_v to sp, sq.
template <int DT, bool VEC, bool STORE>
__device__ __forceinline__ float lane_residual(const char *trow, const char *drow, int lo, int hi, int G,
                                               float Mt, float Md, float c, float iSt, float iSd, float cres,
                                               float *sp, float *sq) {
  constexpr int EPG = Elems<DT>::kPerGroup;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float part = 0.0f;
  for (int j0 = 0; j0 < G; j0 += kBatch) {
    const int g0 = lane_group(warp, j0, G, lane);  // round j0 + u: group g0 + 32 u
    uint4 xt[kBatch], xd[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (j0 + u < G) {
        xt[u] = load_group<DT, VEC>(trow, lo + (g0 + 32 * u) * EPG, hi);
        xd[u] = load_group<DT, VEC>(drow, lo + (g0 + 32 * u) * EPG, hi);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (j0 + u < G) {
        float t[EPG], d[EPG];
        unpack16<DT>(xt[u], t);
        unpack16<DT>(xd[u], d);
#pragma unroll
        for (int e = 0; e < EPG; ++e) {
          const float pv = ex2((t[e] - Mt) * c) * iSt;
          const float qv = ex2((d[e] - Md) * c) * iSd;
          if (STORE) {
            sp[stage_index(g0 + 32 * u, e, EPG)] = pv;
            sq[stage_index(g0 + 32 * u, e, EPG)] = qv;
          }
          part += fmaxf(0.0f, pv - cres * qv);
        }
      }
    }
  }
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
  constexpr int EPG = Elems<DT>::kPerGroup;
  const int G = P.groups;                                 // rounds of 16-byte groups per lane
  float *s_kc = s_uni + N + 1;                            // [N] removed children's coefficients (P.wor)
  float *s_p = s_kc + N;                                  // [G * EPG * threads] staged p (stage_index)
  float *s_q = s_p + static_cast<size_t>(G) * EPG * kTreeThreads;  // staged q
  __shared__ Slot s_all[2][kMaxCluster];  // [exchange parity][source rank]
  __shared__ Slot s_part[kTreeWarps];
  __shared__ float s_wz[2][kMaxCluster][kTreeWarps];  // [exchange parity][source rank][warp]
  __shared__ int s_path[SPEC_MAX_DEPTH + 1], s_out[SPEC_MAX_DEPTH + 1];
  __shared__ int s_bad, s_cnt[kTreeWarps];
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
  // gets rank r's part, and ws the calling warp's.  Every warp pushes its
  // sum into every rank (no block barrier, no second reduction in the CTA);
  // lane r adds up rank r's warp sums in warp order.
  auto cluster_sum = [&](float x, float &part_of_lane, float &ws) {
    ws = warp_sum(x);
    const int ph = phase & 1;
    if (lane < ncl) *cluster.map_shared_rank(&s_wz[ph][rank][warp], lane) = ws;
    cluster.sync();
    ++phase;
    float part = 0.0f;
    if (lane < ncl)
#pragma unroll
      for (int w = 0; w < kTreeWarps; ++w) part += s_wz[ph][lane][w];
    part_of_lane = part;
    return warp_sum(part_of_lane);
  };
  // Children of `node` in increasing id order into s_kids; their number.
  // (The walk uses this only when node's candidates need more than one
  // sweep of the block; see the loop below.)
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
    // children of `node`, in increasing id order
    int nkids, my_pos = -1, my_kid = -1;
    const bool one_sweep = N - node - 1 <= kTreeThreads;
    if (one_sweep) {
      // thread t looks at node + 1 + t; a thread that finds a child keeps its
      // slot and loads its token logits itself, and fills s_kids, s_kt, s_kd
      // after the statistics pass (one barrier fewer than the general sweep)
      const int cidx = node + 1 + tid;
      const bool is_kid = cidx < N && s_par[cidx] == node;
      const unsigned bal = __ballot_sync(0xffffffffu, is_kid);
      if (lane == 0) s_cnt[warp] = __popc(bal);
      __syncthreads();
      const int cw = lane < kTreeWarps ? s_cnt[lane] : 0;
      const int before = __reduce_add_sync(0xffffffffu, lane < warp ? cw : 0);
      nkids = __reduce_add_sync(0xffffffffu, cw);
      if (is_kid) {
        my_pos = before + __popc(bal & ((1u << lane) - 1u));
        my_kid = cidx;
      }
    } else {
      nkids = children(node);
    }
    const char *trow = node_row<DT>(P.target, P.t_req, P.row, b, node);
    const char *drow = (!GREEDY && nkids > 0) ? node_row<DT>(P.draftl, P.d_req, P.row, b, node) : nullptr;
    // the children's token logits: loaded now, stored after the statistics pass
    float kt0 = 0.0f, kd0 = 0.0f;
    if (drow) {
      if (one_sweep) {
        if (my_pos >= 0) {
          const int x = s_tok[my_kid];
          kt0 = load_one<DT>(trow, x);
          kd0 = load_one<DT>(drow, x);
        }
      } else {
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
    }
    asm volatile("" ::: "memory");  // the logit loads go out before the pass's loads

    // ---- row statistics: lane pass, warp merge, block merge, exchange
    RowStats R[2] = {row_stats_empty(), row_stats_empty()};
    const char *rows[2] = {trow, drow};
    lane_rows_stats<DT, !GREEDY, VEC, 2>(rows, lo, hi, G, c, R);
    asm volatile("" ::: "memory");  // and are stored only after it
    if (one_sweep) {
      if (my_pos >= 0) {
        s_kids[my_pos] = my_kid;
        s_kt[my_pos] = kt0;
        s_kd[my_pos] = kd0;
      }
    } else if (drow && tid < nkids) {
      s_kt[tid] = kt0;
      s_kd[tid] = kd0;
    }
    float w_m = R[0].m, w_s = R[0].s.x + R[0].s.y;  // this warp's statistics of t (after the merge)
    {
      float dm = R[1].m, ds = R[1].s.x + R[1].s.y;
      int i = R[0].i, di = kNoIndex;
      if (GREEDY) warp_allargmax(w_m, i);
      else warp_allmerge<false>(w_m, w_s, i, c);  // sampling needs no argmax
      if (drow) warp_allmerge<false>(dm, ds, di, c);
      if (lane == 0) s_part[warp] = Slot{w_m, w_s, dm, ds, i, 0.0f, 0, 0};
    }
    __syncthreads();
    Slot mine = kEmpty;
    if (warp == 0) {
      mine = lane < kTreeWarps ? s_part[lane] : kEmpty;
      int di = kNoIndex;
      if (GREEDY) warp_allargmax(mine.mt, mine.it);
      else warp_allmerge<false>(mine.mt, mine.st, mine.it, c);
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
    int unused = kNoIndex;
    warp_allmerge<false>(Mt, St, unused, c);
    if (drow) warp_allmerge<false>(Md, Sd, unused, c);
    const float iSt = 1.0f / St, iSd = drow ? 1.0f / Sd : 0.0f;
    // lane r: rank r's share of the current draw distribution (p so far)
    float rmass = lane < ncl ? r.st * ex2((r.mt - Mt) * c) * iSt : 0.0f;
    float w_mass = -1.0f;  // this warp's share of it; < 0: p, from the warp's statistics

    // the p and q of child i's token (from the children's token logits), rounded
    // as the sweeps over the slice round them
    auto pq_of = [&](int i, float &pv, float &qv) {
      pv = ex2((s_kt[i] - Mt) * c) * iSt;
      qv = ex2((s_kd[i] - Md) * c) * iSd;
    };
    // Siblings drawn without replacement (P.wor): each rejected sibling's
    // token is removed from q.  A removed token's residual keeps the
    // coefficient it had at its removal, s_kc[i] for child i (-1: child i
    // removed nothing); Qrem is the q mass not removed.  Every token never
    // removed shares the coefficient cres.
    auto removed_coef = [&](int x, int upto) {
      float a = -1.0f;
      for (int i = 0; i < upto; ++i)
        if (s_kc[i] >= 0.0f && s_tok[s_kids[i]] == x) a = s_kc[i];
      return a;
    };
    float cres = 0.0f, Z = 1.0f, Qrem = 1.0f;
    bool staged = false;  // s_p / s_q hold this node's slice
    int next = -1;
    for (int ki = 0; ki < nkids; ++ki) {
      const int ch = s_kids[ki], x = s_tok[ch];
      float pt, qt;
      pq_of(ki, pt, qt);
      const float ax = P.wor ? removed_coef(x, ki) : -1.0f;
      // a removed token, or every q mass removed: q_j(x) = 0, accepted iff p_j(x) > 0
      const bool accept = ax >= 0.0f            ? pt - ax * qt > 0.0f
                          : P.wor && !(Qrem > 0.0f) ? pt - cres * qt > 0.0f
                                                    : s_uni[ch] * qt * Z < fmaxf(0.0f, pt - cres * qt) * Qrem;
      if (accept) {
        next = ch;
        break;
      }
      if (P.wor && !(Qrem > 0.0f)) {  // q_j has no mass left: the residual is p_j itself
        s_kc[ki] = -1.0f;
        continue;
      }
      // rejected: the next residual max(0, p - cnew q), its mass over the cluster
      const float cnew = cres + (P.wor ? Z / Qrem : Z);
      float part = 0.0f;
      if (staged) {
        for (int j = 0; j < G; ++j) {
          const int g = lane_group(warp, j, G, lane);
#pragma unroll
          for (int e = 0; e < EPG; ++e)
            part += fmaxf(0.0f, s_p[stage_index(g, e, EPG)] - cnew * s_q[stage_index(g, e, EPG)]);
        }
      } else if (P.stage) {
        part = lane_residual<DT, VEC, true>(trow, drow, lo, hi, G, Mt, Md, c, iSt, iSd, cnew, s_p, s_q);
        staged = true;
      } else {
        part = lane_residual<DT, VEC, false>(trow, drow, lo, hi, G, Mt, Md, c, iSt, iSd, cnew, s_p, s_q);
      }
      if (P.wor) {
        // tokens removed earlier keep their own coefficient: the lane owning
        // such a token's group corrects its part
        for (int i = 0; i < ki; ++i) {
          const int y = s_tok[s_kids[i]];
          if (s_kc[i] < 0.0f || y < lo || y >= hi) continue;
          const int gy = (y - lo) / EPG;
          if (lane != (gy & 31) || warp != (gy >> 5) / G) continue;
          float py, qy;
          pq_of(i, py, qy);
          part += fmaxf(0.0f, py - s_kc[i] * qy) - fmaxf(0.0f, py - cnew * qy);
        }
      }
      float zr, wz;
      const float Znew = cluster_sum(part, zr, wz);
      const bool moved = Znew > 0.0f;  // a zero-mass residual (rounding only) keeps the previous p and q
      if (P.wor) s_kc[ki] = moved && ax < 0.0f ? cnew : -1.0f;  // (every thread writes the same value)
      if (moved) {
        if (P.wor && ax < 0.0f) Qrem = fmaxf(0.0f, Qrem - qt);
        cres = cnew;
        Z = Znew;
        rmass = zr;
        w_mass = wz;
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
      // the warp whose range holds the crossing, then that range
      const float mass = w_mass >= 0.0f ? w_mass : (w_m == -INFINITY ? 0.0f : w_s * ex2((w_m - Mt) * c) * iSt);
      // (the fallback `lo` is unreachable: the drawing rank has mass, so one of its warps has)
      final_tok = range_draw<kTreeThreads, EPG>(mass, tl, lo, G, lo, nullptr, [&](int g, float *w) {
        if (staged) {
#pragma unroll
          for (int e = 0; e < EPG; ++e)
            w[e] = fmaxf(0.0f, s_p[stage_index(g, e, EPG)] - cres * s_q[stage_index(g, e, EPG)]);
        } else {
          float t[EPG];
          unpack16<DT>(load_group<DT, VEC>(trow, lo + g * EPG, hi), t);
#pragma unroll
          for (int e = 0; e < EPG; ++e) w[e] = ex2((t[e] - Mt) * c) * iSt;
          if (cres > 0.0f) {
            float d[EPG];
            unpack16<DT>(load_group<DT, VEC>(drow, lo + g * EPG, hi), d);
#pragma unroll
            for (int e = 0; e < EPG; ++e) w[e] = fmaxf(0.0f, w[e] - cres * (ex2((d[e] - Md) * c) * iSd));
          }
        }
        if (P.wor) {  // removed tokens keep the coefficient of their removal
          for (int i = 0; i < nkids; ++i) {
            const int y = s_tok[s_kids[i]] - lo - g * EPG;
            if (s_kc[i] < 0.0f || y < 0 || y >= EPG) continue;
            float py, qy;
            pq_of(i, py, qy);
            const float wy = fmaxf(0.0f, py - s_kc[i] * qy);
#pragma unroll
            for (int e = 0; e < EPG; ++e)  // (no dynamic index into the register array)
              if (e == y) w[e] = wy;
          }
        }
      });
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

// Dynamic shared memory of the walk: parents, tokens, children, the
// children's two token logits and their coefficients (6 words per node), the
// uniforms (N + 1), plus the staged p and q of the CTA's slice (every lane's
// groups) when staging is on.
size_t tree_dynamic_smem(const TreeParams &P) {
  const size_t epg = P.dtype == SPEC_DTYPE_F32 ? 4 : 8;
  return sizeof(int) * (7 * static_cast<size_t>(P.N) + 1) +
         (P.stage ? 2 * sizeof(float) * static_cast<size_t>(P.groups) * epg * kTreeThreads : 0);
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
