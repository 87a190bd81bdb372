// Top-k / top-p filtering of logit rows before verification.  The pages set
// temperature, top-k and top-p aside ("投机解码:为什么一个字都不改", the
// section that leaves them to another lesson); verification stays lossless
// against the filtered target when p and q are filtered alike and the
// drafter drew from the filtered q.  The filter, applied in this order:
//   top-k (0 < top_k < V): keep every logit >= the top_k-th largest;
//   top-p (top_p < 1): over the kept logits in descending order, with p
//   renormalised to them, keep the smallest prefix whose mass reaches top_p
//   and every logit equal to its last one.
// A row is then described by its threshold: kept = {v : x_v >= theta}.
//
// One thread-block cluster per row; CTA r of the cluster holds slice r of
// the row in shared memory (staged through registers, several 16-byte loads
// in flight per thread).  Both thresholds are found by radix selection on
// an order-preserving 32-bit key of each logit (bf16 logits differ only in
// the top 16 bits: two 8-bit levels; fp32: four):
//   - each level builds a 256-bin histogram of the next digit over the
//     logits whose key matches the digits chosen so far: counts for top-k;
//     counts and masses 2^((x - M) c) for top-p, the masses in 2^-44 fixed
//     point so that the sums do not depend on the order of the atomic adds;
//   - the CTAs' histograms are added over the cluster (every CTA reads every
//     CTA's histogram through distributed shared memory, in rank order), so
//     every CTA picks the same digit: the bin holding the top_k-th largest
//     count, or the bin where the mass from the top reaches top_p times the
//     kept mass.
// Most rows never need the full radix walk.  When top-k is on, one pass
// counts the logits in the top-byte bin of the row's max and in the bin
// below it (packed bf16x2 compares), and copies the first bin's logits into
// a short list in shared memory; when that window already holds top_k
// logits (and each CTA's share fits the list), the radix walk and the top-p
// walk run over the list alone, and the kept mass is added in 2^-44 fixed
// point (so the list's order, which the appends leave unspecified, does not
// matter).  With several CTAs, each pushes its list into rank 0's shared
// memory and leaves; rank 0 finishes the row alone.  Otherwise the walk runs
// over the whole slice as above.
// Row mode, for calls with at least two rows per SM and top-k on: one CTA
// per row, no cluster and no staging; the passes read the row from global
// memory (the same steps with a cluster of one).
// The outputs are the chain verification's per-row statistics, as one
// partial per row -- (max M, sum over kept logits of 2^((x - M) c), the
// drafted token's logit) -- and theta, which the accept kernels apply as a
// mask.  Rows verification never reads (positions past the draft length)
// are skipped.
#include <cooperative_groups.h>

#include "chain_common.cuh"
#include "common.cuh"
#include "launch.h"
#include "segments.cuh"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kFilterThreads = 512;
constexpr int kFilterWarps = kFilterThreads / 32;
constexpr int kFilterListCap = 1024;             // candidate logits per CTA on the list path
constexpr int kFilterRowListCap = 4096;          // the same in row mode (one CTA per row)
constexpr int kFilterRowMinRowsPerSm = 2;       // row mode from this many rows per SM
constexpr int kFilterLoadBatch = 4;              // 16-byte loads each thread keeps in flight

constexpr double kMassScale = 17592186044416.0;  // 2^44: fixed-point unit of the histogram masses

// Order-preserving unsigned key of an fp32 value (its bits); -0 maps to +0.
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  if (bits == 0x80000000u) bits = 0u;
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}
// The value whose key has these top 8 * levels bits (the bits below are
// the same for every logit of the dtype: zero for a positive fp32 image of
// a bf16, all ones for a negative one).
template <int DT>
__device__ __forceinline__ float prefix_value(uint32_t prefix, int levels) {
  if (levels == 4) return key_value(prefix);
  const uint32_t key = prefix << 16;
  return key_value((key & 0x80000000u) ? key : (key | 0xffffu));
}

// The smallest logit of the dtype whose key has top byte d (1 <= d <= 255):
// x >= bin_floor(d) exactly when key(x) >> 24 >= d, for every non-NaN x.
template <int DT>
__device__ __forceinline__ float bin_floor(uint32_t d) {
  if (d & 0x80u) return __uint_as_float((d & 0x7fu) << 24);
  if (DT == SPEC_DTYPE_F32) return __uint_as_float(((~d & 0xffu) << 24) | 0xffffffu);
  return __uint_as_float(((((~d & 0xffu) << 8) | 0xffu)) << 16);
}

// 0x0001 in each 16-bit half of a bf16 pair that is >= the pair t2.
__device__ __forceinline__ uint32_t ge_pair(uint32_t w, uint32_t t2) {
  return __hge2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w), *reinterpret_cast<const __nv_bfloat162 *>(&t2)) &
         0x00010001u;
}

// The fixed-point (2^-44) mass of one logit, 2^((x - M) c).
__device__ __forceinline__ unsigned long long fixed_mass(float x, float c, float M) {
  return static_cast<unsigned long long>(static_cast<double>(ex2((x - M) * c)) * kMassScale);
}

template <int DT>
__device__ __forceinline__ uint32_t elem_bits(const void *s, int e) {
  if (DT == SPEC_DTYPE_F32) return reinterpret_cast<const uint32_t *>(s)[e];
  return static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(s)[e]) << 16;
}

// The filter of partial row j by the calling CTA (and, with STAGE, the
// other CTAs of its cluster, one slice each).
// STAGE = false (row mode): the CTA reads the whole row from global memory
// instead of a staged slice -- the first pass (the max) from HBM, the later
// ones from L2 -- with a longer list.
template <int DT, bool VEC, bool STAGE>
__device__ __forceinline__ void filter_row(const ChainParams &P, const int j) {
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int EPG = Elems<DT>::kPerGroup, ES = Elems<DT>::kSize;
  constexpr int kLevels = DT == SPEC_DTYPE_F32 ? 4 : 2;
  constexpr int kMaxCS = 16;
  constexpr int kCap = STAGE ? kFilterListCap : kFilterRowListCap;
  const int CS = STAGE ? P.cluster : 1, rank = STAGE ? static_cast<int>(cluster.block_rank()) : 0;
  const int k = P.k, K1 = k + 1, R = 2 * k + 1;
  const int b = j / R, r = j - b * R;
  const int side = r < K1 ? 0 : 1, i = side ? r - K1 : r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V;
  const float c = P.c;

  const int L = P.draft_len ? P.draft_len[b] : k;
  // the rows verification reads: targets 0..L, drafts 0..L-1 (the same in the whole cluster)
  if (L < 0 || L > k || (side == 0 ? i > L : i >= L)) return;
  if (r == 0 && rank == 0 && tid == 0 && P.counter2) P.counter2[b] = 0;  // for the chunked accept kernel
  const char *row = side ? row_ptr<DT>(P.draftl, P.d_req, P.row, b, i) : row_ptr<DT>(P.target, P.t_req, P.row, b, i);
  const int lo = STAGE ? min(V, rank * P.slice) : 0, hi = STAGE ? min(V, lo + P.slice) : V, n = hi - lo;
  // the drafted token's logit (rank 0 writes the partial), loaded now so the
  // two dependent reads overlap the slice's
  float xtok = -INFINITY;
  if (rank == 0 && tid == 0 && i < L) {
    const int tok = P.draft[static_cast<int64_t>(b) * k + i];
    if (tok >= 0 && tok < V) xtok = load_one<DT>(row, tok);
  }

  extern __shared__ __align__(16) unsigned char dyn_filter[];
  unsigned char *s_row = dyn_filter;  // [slice] the slice's logits (STAGE)
  // the logits every pass after the first reads: the staged slice, or the row
  const unsigned char *src = STAGE ? s_row : reinterpret_cast<const unsigned char *>(row);
  __shared__ uint32_t s_cnt[2][256];
  __shared__ unsigned long long s_mass[2][256];
  __shared__ uint32_t t_cnt[256];
  __shared__ unsigned long long t_mass[256];
  __shared__ float s_cf[kMaxCS], s_cs[kMaxCS];
  __shared__ uint32_t s_cu[kMaxCS];
  __shared__ float s_red[kFilterWarps];
  __shared__ uint32_t s_redu[kFilterWarps];
  __shared__ uint32_t s_sel_digit;
  __shared__ unsigned long long s_sel_rest;

  // ---- the slice into shared memory, and the slice max
  float mloc = -INFINITY;
  const int ng = VEC ? n / EPG : 0;  // n is a multiple of EPG on the 16-byte path
  __shared__ uint32_t s_list[kCap];
  __shared__ int s_nlist;
  if (!STAGE) {
    // row mode: one pass over the row (batches of 16-byte loads in flight per
    // thread) for its max and, with top-k on, the candidate list: each warp
    // keeps its running max and appends every logit at or above the floor of
    // that max's top-byte bin.  The threshold only rises and the row's own
    // bin floor is at least every warp's, so the list holds every logit of
    // the window the list path needs (plus smaller ones, which change
    // neither the top_k-th largest nor the kept set); the rows whose list
    // overflows, or whose window holds fewer than top_k logits, are read
    // again below.
    if (VEC) {
      const uint4 *g16 = reinterpret_cast<const uint4 *>(row);
      const bool spec = P.top_k > 0 && P.top_k < V;
      if (tid == 0) s_nlist = 0;
      __syncthreads();
      constexpr uint32_t kNegInf = DT == SPEC_DTYPE_F32 ? 0xff800000u : 0xff80ff80u;  // -inf words
      constexpr int kLoadBatch = kFilterLoadBatch;
      for (int gw = tid - lane; gw < ng; gw += kFilterThreads * kLoadBatch) {  // (warp-uniform)
        const int g0 = gw + lane;  // the lane's groups: g0 + kFilterThreads u
        uint4 w[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u)
          w[u] = g0 + u * kFilterThreads < ng ? ld_stream16(g16 + g0 + u * kFilterThreads)
                                              : make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
        float bmax = -INFINITY;  // this thread's max over the batch
        if (DT == SPEC_DTYPE_BF16) {
          __nv_bfloat162 mx2 = *reinterpret_cast<const __nv_bfloat162 *>(&w[0].x);
#pragma unroll
          for (int u = 0; u < kLoadBatch; ++u) {
            mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162 *>(&w[u].x));
            mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162 *>(&w[u].y));
            mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162 *>(&w[u].z));
            mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162 *>(&w[u].w));
          }
          bmax = fmaxf(__low2float(mx2), __high2float(mx2));
        } else {
#pragma unroll
          for (int u = 0; u < kLoadBatch; ++u)
            bmax = fmaxf(bmax, fmaxf(fmaxf(__uint_as_float(w[u].x), __uint_as_float(w[u].y)),
                                     fmaxf(__uint_as_float(w[u].z), __uint_as_float(w[u].w))));
        }
        mloc = fmaxf(mloc, bmax);
        if (spec) {
          const uint32_t dw = order_key(__float_as_uint(warp_allmax(mloc))) >> 24;
          const float tw = (dw >= 2u && (dw | 1u) != 0x81u) ? bin_floor<DT>(dw) : -INFINITY;
          // (a thread whose batch max is below tw has nothing to append; most
          // batches of most rows have no such logit in the whole warp)
          const bool has = bmax >= tw;
          if (!__any_sync(0xffffffffu, has)) continue;
          // this lane's logits >= tw, counted; one reservation of list slots
          // per warp (a shuffle scan of the counts, one atomic); then each
          // lane writes its own -- no warp-wide step inside the divergent part
          int mine = 0;
          const uint32_t t2 = (__float_as_uint(tw) >> 16) * 0x10001u;
#pragma unroll
          for (int u = 0; u < kLoadBatch; ++u) {
            if (!has || g0 + u * kFilterThreads >= ng) continue;  // (past the row's end)
            const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              if (DT == SPEC_DTYPE_BF16) mine += __popc(ge_pair(ws[h], t2));
              else mine += __uint_as_float(ws[h]) >= tw;
            }
          }
          int incl = mine;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
          }
          const int wtot = __shfl_sync(0xffffffffu, incl, 31);
          int base = 0;
          if (lane == 31 && wtot > 0) base = atomicAdd(&s_nlist, wtot);
          base = __shfl_sync(0xffffffffu, base, 31);
          int pos = base + incl - mine;
          if (mine > 0 && pos < kCap) {
#pragma unroll
            for (int u = 0; u < kLoadBatch; ++u) {
              if (g0 + u * kFilterThreads >= ng) continue;
              const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
              for (int h = 0; h < 4 * (DT == SPEC_DTYPE_BF16 ? 2 : 1); ++h) {
                const uint32_t bits = DT == SPEC_DTYPE_F32 ? ws[h]
                                      : ((h & 1) ? (ws[h >> 1] & 0xffff0000u) : (ws[h >> 1] << 16));
                if (__uint_as_float(bits) >= tw) {
                  if (pos < kCap) s_list[pos] = bits;
                  ++pos;
                }
              }
            }
          }
          __syncwarp();
        }
      }

    } else {
      for (int e = tid; e < n; e += kFilterThreads) mloc = fmaxf(mloc, load_one<DT>(row, e));
    }
  } else if (VEC) {
    // batches of kFilterLoadBatch 16-byte loads in flight per thread (into
    // registers, then shared memory), the max folded in as they land
    const uint4 *src = reinterpret_cast<const uint4 *>(row + static_cast<int64_t>(lo) * ES);
    uint4 *dst = reinterpret_cast<uint4 *>(s_row);
    __nv_bfloat162 mx2 = __float2bfloat162_rn(-INFINITY);
    for (int g0 = tid; g0 < ng; g0 += kFilterThreads * kFilterLoadBatch) {
      uint4 w[kFilterLoadBatch];
#pragma unroll
      for (int u = 0; u < kFilterLoadBatch; ++u)
        if (g0 + u * kFilterThreads < ng) w[u] = ld_stream16(src + g0 + u * kFilterThreads);
#pragma unroll
      for (int u = 0; u < kFilterLoadBatch; ++u) {
        if (g0 + u * kFilterThreads < ng) {
          dst[g0 + u * kFilterThreads] = w[u];
          if (DT == SPEC_DTYPE_BF16) {
            mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162 *>(&w[u].x));
            mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162 *>(&w[u].y));
            mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162 *>(&w[u].z));
            mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162 *>(&w[u].w));
          } else {
            mloc = fmaxf(mloc, fmaxf(fmaxf(__uint_as_float(w[u].x), __uint_as_float(w[u].y)),
                                     fmaxf(__uint_as_float(w[u].z), __uint_as_float(w[u].w))));
          }
        }
      }
    }
    if (DT == SPEC_DTYPE_BF16) mloc = fmaxf(__low2float(mx2), __high2float(mx2));
    __syncthreads();  // the slice is in shared memory
  } else {
    for (int e = tid; e < n; e += kFilterThreads) {
      const float x = load_one<DT>(row, lo + e);
      if (DT == SPEC_DTYPE_F32) reinterpret_cast<float *>(s_row)[e] = x;
      else reinterpret_cast<uint16_t *>(s_row)[e] = static_cast<uint16_t>(__float_as_uint(x) >> 16);
      mloc = fmaxf(mloc, x);
    }
  }
  mloc = warp_allmax(mloc);
  if (lane == 0) s_red[warp] = mloc;
  __syncthreads();
  mloc = warp_allmax(lane < kFilterWarps ? s_red[lane] : -INFINITY);
  if (tid < CS) *cluster.map_shared_rank(&s_cf[rank], tid) = mloc;
  cluster.sync();
  float M = -INFINITY;
  for (int q = 0; q < CS; ++q) M = fmaxf(M, s_cf[q]);

  // ---- the list path (top-k on): the window of the max's top-byte bin, or
  // of that bin and the one below, when the window holds top_k logits and
  // each CTA's share fits the list
  __shared__ uint32_t s_xc[2][kMaxCS];  // per rank: logits >= tau0, logits >= tau1
  __shared__ uint32_t s_w0[kFilterWarps], s_w1[kFilterWarps];
  bool use_list = false;  // the walk runs over s_union[0, nlist) in rank 0 alone
  bool top_bin = false;   // and every logit the walks need shares the max's top byte
  int nlist = 0;
  uint32_t *s_union = s_list;
  const uint32_t BM = order_key(__float_as_uint(M)) >> 24;
  // (not for a max in the two bins at +0, whose floors +0 and the smallest
  // normal would let a flushed subnormal compare on the wrong side)
  const bool window_ok = P.top_k > 0 && P.top_k < V && BM >= 2u && (BM | 1u) != 0x81u;
  if (!STAGE && VEC && window_ok) {
    // row mode: the list the first pass built serves when it did not
    // overflow and holds top_k logits of the max's bin.  Thread 0 reads the
    // list's length and publishes one decision, so every thread of the CTA
    // takes the same branch (and meets the same barriers).
    __shared__ int s_listn;
    if (tid == 0) {
      const int len = *reinterpret_cast<volatile int *>(&s_nlist);
      s_listn = len <= kCap ? len : -1;
    }
    __syncthreads();
    const int nl = s_listn;
    if (nl >= 0) {
      const float tau0 = bin_floor<DT>(BM);
      uint32_t c0 = 0u;
      for (int e = tid; e < nl; e += kFilterThreads) c0 += __uint_as_float(s_list[e]) >= tau0;
      c0 = __reduce_add_sync(0xffffffffu, c0);
      if (lane == 0) s_w0[warp] = c0;
      __syncthreads();
      c0 = __reduce_add_sync(0xffffffffu, lane < kFilterWarps ? s_w0[lane] : 0u);
      if (c0 >= static_cast<uint32_t>(P.top_k)) {
        use_list = true;
        top_bin = true;
        nlist = nl;
      }
      __syncthreads();  // (s_w0 is written again below)
    }
  }
  if (!use_list && window_ok) {
    const float tau0 = bin_floor<DT>(BM), tau1 = bin_floor<DT>(BM - 1u);
    // appends every logit >= tau to the list (up to its capacity); with
    // COUNT, also counts the logits >= tau0 and >= tau1 (tau = tau0)
    auto scan = [&]<bool COUNT>(float tau, uint32_t &c0, uint32_t &c1) {
      auto append = [&](uint32_t bits) {
        const int pos = atomicAdd(&s_nlist, 1);
        if (pos < kCap) s_list[pos] = bits;
      };
      if (VEC && DT == SPEC_DTYPE_BF16) {
        const uint32_t ta = (__float_as_uint(tau) >> 16) * 0x10001u;
        const uint32_t t1 = (__float_as_uint(tau1) >> 16) * 0x10001u;
        uint32_t p0 = 0u, p1 = 0u;  // two 16-bit counters each (at most 48 per half)
        for (int g = tid; g < ng; g += kFilterThreads) {
          const uint4 w = reinterpret_cast<const uint4 *>(src)[g];
          const uint32_t a0 = ge_pair(w.x, ta), a1 = ge_pair(w.y, ta), a2 = ge_pair(w.z, ta), a3 = ge_pair(w.w, ta);
          if (COUNT) {
            p0 += a0 + a1 + a2 + a3;
            p1 += ge_pair(w.x, t1) + ge_pair(w.y, t1) + ge_pair(w.z, t1) + ge_pair(w.w, t1);
          }
          if (a0 | a1 | a2 | a3) {
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              const uint32_t bits = (h & 1) ? (ws[h >> 1] & 0xffff0000u) : (ws[h >> 1] << 16);
              if (__uint_as_float(bits) >= tau) append(bits);
            }
          }
        }
        c0 = (p0 & 0xffffu) + (p0 >> 16);
        c1 = (p1 & 0xffffu) + (p1 >> 16);
      } else {
        c0 = c1 = 0u;
        for (int e = tid; e < n; e += kFilterThreads) {
          const uint32_t bits = elem_bits<DT>(src, e);
          const float x = __uint_as_float(bits);
          if (COUNT) {
            c0 += x >= tau0;
            c1 += x >= tau1;
          }
          if (x >= tau) append(bits);
        }
      }
    };
    if (tid == 0) s_nlist = 0;
    __syncthreads();
    uint32_t c0, c1;
    scan.template operator()<true>(tau0, c0, c1);
    c0 = __reduce_add_sync(0xffffffffu, c0);
    c1 = __reduce_add_sync(0xffffffffu, c1);
    if (lane == 0) {
      s_w0[warp] = c0;
      s_w1[warp] = c1;
    }
    __syncthreads();
    if (warp == 0) {
      c0 = __reduce_add_sync(0xffffffffu, lane < kFilterWarps ? s_w0[lane] : 0u);
      c1 = __reduce_add_sync(0xffffffffu, lane < kFilterWarps ? s_w1[lane] : 0u);
      if (lane < CS) {  // this CTA's counts, into every CTA of the cluster
        *cluster.map_shared_rank(&s_xc[0][rank], lane) = c0;
        *cluster.map_shared_rank(&s_xc[1][rank], lane) = c1;
      }
    }
    cluster.sync();
    uint32_t T0 = 0u, T1 = 0u, A0 = 0u, A1 = 0u;  // cluster totals, largest per-CTA counts
    for (int q = 0; q < CS; ++q) {
      T0 += s_xc[0][q];
      T1 += s_xc[1][q];
      A0 = max(A0, s_xc[0][q]);
      A1 = max(A1, s_xc[1][q]);
    }
    const uint32_t K = static_cast<uint32_t>(P.top_k);
    int win = -1;  // the window taken: 0 (>= tau0), 1 (>= tau1), -1 none
    if (T0 >= K && A0 <= static_cast<uint32_t>(kCap)) {
      win = 0;  // the lists hold every logit >= tau0
      top_bin = true;
    } else if (T1 >= K && A1 <= static_cast<uint32_t>(kCap)) {
      if (tid == 0) s_nlist = 0;
      __syncthreads();
      scan.template operator()<false>(tau1, c0, c1);
      win = 1;  // the lists hold every logit >= tau1
      cluster.sync();  // every slice scan is over before rank 0's slice buffer is reused
    }
    if (win >= 0) {
      // the union of the lists, in rank order, into rank 0's slice buffer (no
      // slice is read again on this path; CS lists of at most kFilterListCap
      // entries fit in any slice of a row that needs CS > 1); then rank 0
      // goes on alone
      use_list = true;
      __syncthreads();
      const int mine = min(*reinterpret_cast<volatile int *>(&s_nlist), kCap);
      if (STAGE && CS > 1) {
        uint32_t off = 0u, total = 0u;
        for (int q = 0; q < CS; ++q) {
          const uint32_t cq = s_xc[win][q];
          off += q < rank ? cq : 0u;
          total += cq;
        }
        uint32_t *dst = cluster.map_shared_rank(reinterpret_cast<uint32_t *>(s_row), 0) + off;
        for (int e = tid; e < mine; e += kFilterThreads) dst[e] = s_list[e];
        cluster.sync();
        if (rank != 0) return;  // (no CTA touches another's shared memory after this barrier)
        s_union = reinterpret_cast<uint32_t *>(s_row);
        nlist = static_cast<int>(total);
      } else {
        nlist = mine;
      }
    }
  }

  // ---- radix selection: one level of the histogram walk.  Builds the
  // level's cluster-wide histogram of digit (key >> shift) & 255 over the
  // logits whose key >> (shift + 8) equals `prefix` (all logits at the first
  // level) and >= floor -- on the list path, the logits of the list (which
  // holds every logit >= the answer); then warp 0 walks the bins from the top until the
  // count (BY_MASS: the mass) reaches `need` -- or, with frac > 0, frac
  // times the level's whole mass.  Returns the digit; `rest` becomes need
  // minus what the bins above the digit hold.
  int level_no = 0;
  auto level = [&](int shift, uint32_t prefix, bool first, float floor, bool by_mass,
                   unsigned long long need, unsigned long long &rest, float frac = 0.0f) -> uint32_t {
    const int buf = level_no++ & 1;  // the other buffer may still be read by other CTAs
    for (int d = tid; d < 256; d += kFilterThreads) {
      s_cnt[buf][d] = 0u;
      s_mass[buf][d] = 0ull;
    }
    __syncthreads();
    const int ne = use_list ? nlist : n;
    for (int e = tid; e < ne; e += kFilterThreads) {
      const uint32_t bits = use_list ? s_union[e] : elem_bits<DT>(src, e);
      const uint32_t key = order_key(bits);
      if (!first && (key >> (shift + 8)) != prefix) continue;
      const float x = __uint_as_float(bits);
      if (!(x >= floor)) continue;
      const uint32_t d = (key >> shift) & 255u;
      atomicAdd(&s_cnt[buf][d], 1u);
      if (by_mass) atomicAdd(&s_mass[buf][d], fixed_mass(x, c, M));
    }
    if (use_list) __syncthreads();  // rank 0 alone: its histogram is the row's
    else cluster.sync();            // every CTA's histogram is complete
    for (int d = tid; d < 256; d += kFilterThreads) {
      uint32_t cnt = 0u;
      unsigned long long ms = 0ull;
      if (use_list) {
        cnt = s_cnt[buf][d];
        ms = s_mass[buf][d];
      } else {
        for (int q = 0; q < CS; ++q) {
          cnt += *cluster.map_shared_rank(&s_cnt[buf][d], q);
          if (by_mass) ms += *cluster.map_shared_rank(&s_mass[buf][d], q);
        }
      }
      t_cnt[d] = cnt;
      t_mass[d] = ms;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255 - 8 l ... 248 - 8 l, from the top
      unsigned long long lsum = 0ull;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int d = 255 - (lane * 8 + t);
        lsum += by_mass ? t_mass[d] : t_cnt[d];
      }
      unsigned long long incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (frac > 0.0f) {
        const unsigned long long total = __shfl_sync(0xffffffffu, incl, 31);
        need = static_cast<unsigned long long>(static_cast<double>(frac) * static_cast<double>(total));
        if (need == 0ull) need = 1ull;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, lsum > 0ull && incl >= need);
      if (hit) {
        const int lh = __ffs(hit) - 1;
        if (lane == lh) {
          unsigned long long run = incl - lsum;
          int sel = -1;
          for (int t = 0; t < 8 && sel < 0; ++t) {
            const int d = 255 - (lane * 8 + t);
            const unsigned long long v = by_mass ? t_mass[d] : t_cnt[d];
            if (v > 0ull && run + v >= need) sel = d;
            else run += v;
          }
          s_sel_digit = static_cast<uint32_t>(sel);
          s_sel_rest = need - run;
        }
      } else {
        // the count or mass never reaches `need` (mass rounding): the lowest non-empty bin
        const unsigned nz = __ballot_sync(0xffffffffu, [&] {
          bool any = false;
#pragma unroll
          for (int t = 0; t < 8; ++t) any |= t_cnt[255 - (lane * 8 + t)] > 0u;
          return any;
        }());
        if (lane == 0) {
          int sel = 0;
          unsigned long long above = 0ull;
          if (nz) {
            const int ll = 31 - __clz(nz);
            for (int t = 7; t >= 0; --t)
              if (t_cnt[255 - (ll * 8 + t)] > 0u) {
                sel = 255 - (ll * 8 + t);
                break;
              }
            for (int d = 255; d > sel; --d) above += by_mass ? t_mass[d] : t_cnt[d];
          }
          s_sel_digit = static_cast<uint32_t>(sel);
          s_sel_rest = need > above ? need - above : 1ull;
        }
      }
    }
    __syncthreads();
    rest = s_sel_rest;
    return s_sel_digit;
  };

  // ---- top-k: the top_k-th largest key.  When the list holds the max's
  // top-byte bin and that bin holds top_k logits, the answer and every kept
  // logit have the max's top byte BM: the walks start at the second byte.
  const int lv0 = top_bin ? 1 : 0;
  const uint32_t prefix0 = top_bin ? BM : 0u;
  float theta = -INFINITY;
  if (P.top_k > 0 && P.top_k < V) {
    uint32_t prefix = prefix0;
    unsigned long long need = static_cast<unsigned long long>(P.top_k), rest = 0ull;
    for (int lv = lv0; lv < kLevels; ++lv) {
      const int shift = 24 - 8 * lv;
      const uint32_t d = level(shift, prefix, lv == 0, -INFINITY, false, need, rest);
      prefix = (prefix << 8) | d;
      need = rest;
    }
    theta = prefix_value<DT>(prefix, kLevels);
  }
  // ---- top-p over the logits top-k kept
  if (P.top_p < 1.0f) {
    uint32_t prefix = prefix0;
    unsigned long long need = 0ull, rest = 0ull;
    for (int lv = lv0; lv < kLevels; ++lv) {
      // the first level's walk needs top_p of the kept mass it histograms
      const uint32_t d = level(24 - 8 * lv, prefix, lv == 0, theta, true, need, rest, lv == lv0 ? P.top_p : 0.0f);
      prefix = (prefix << 8) | d;
      need = rest;
    }
    theta = fmaxf(theta, prefix_value<DT>(prefix, kLevels));
  }

  // ---- the kept logits: their mass, count and smallest value.  On the list
  // path the mass is added in 2^-44 fixed point (the list's order is not
  // fixed); on the slice, in fp32 in thread order, then in warp, block and
  // rank order.  Either way every run gives the same bits.
  float s_loc = 0.0f, mn = INFINITY;
  unsigned long long f_loc = 0ull;
  uint32_t cnt = 0u;
  if (use_list) {
    for (int e = tid; e < nlist; e += kFilterThreads) {
      const float x = __uint_as_float(s_union[e]);
      if (x >= theta) {
        f_loc += fixed_mass(x, c, M);
        mn = fminf(mn, x);
        ++cnt;
      }
    }
  } else {
    for (int e = tid; e < n; e += kFilterThreads) {
      const float x = __uint_as_float(elem_bits<DT>(src, e));
      if (x >= theta) {
        s_loc += ex2((x - M) * c);
        mn = fminf(mn, x);
        ++cnt;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) f_loc += __shfl_xor_sync(0xffffffffu, f_loc, o);
  s_loc = warp_sum(s_loc);
  mn = -warp_allmax(-mn);
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  __shared__ float s_mn[kFilterWarps];
  __shared__ unsigned long long s_redf[kFilterWarps];
  __shared__ float s_cmn[kMaxCS];
  if (lane == 0) {
    s_red[warp] = s_loc;
    s_redf[warp] = f_loc;
    s_redu[warp] = cnt;
    s_mn[warp] = mn;
  }
  __syncthreads();
  if (warp == 0) {
    s_loc = warp_sum(lane < kFilterWarps ? s_red[lane] : 0.0f);
    f_loc = lane < kFilterWarps ? s_redf[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) f_loc += __shfl_xor_sync(0xffffffffu, f_loc, o);
    cnt = __reduce_add_sync(0xffffffffu, lane < kFilterWarps ? s_redu[lane] : 0u);
    mn = -warp_allmax(-(lane < kFilterWarps ? s_mn[lane] : INFINITY));
    if (!use_list && lane < CS) {  // this CTA's sums, into every CTA of the cluster
      *cluster.map_shared_rank(&s_cs[rank], lane) = s_loc;
      *cluster.map_shared_rank(&s_cu[rank], lane) = cnt;
      *cluster.map_shared_rank(&s_cmn[rank], lane) = mn;
    }
  }
  // (after this barrier no CTA touches another's shared memory)
  if (!use_list) cluster.sync();
  if (rank == 0 && tid == 0) {
    float S = 0.0f, smallest = INFINITY;
    uint32_t kept = 0u;
    if (use_list) {  // rank 0 alone, over the whole row's list
      S = static_cast<float>(static_cast<double>(f_loc) / kMassScale);
      kept = cnt;
      smallest = mn;
    } else {
      for (int q = 0; q < CS; ++q) {
        S += s_cs[q];
        kept += s_cu[q];
        smallest = fminf(smallest, s_cmn[q]);
      }
    }
    P.part[j] = Partial{M, S, kNoIndex, xtok};
    P.theta[j] = smallest;
    if (P.kept) P.kept[j] = static_cast<int32_t>(kept);
  }
}

// STAGE: one cluster per row.  Row mode (launched without clusters): one CTA
// per row.  (Two CTAs per SM taking rows in turn measured slower, and the
// loop alone raised the kernel to 60 registers, two CTAs per SM instead of
// three.)
template <int DT, bool VEC, bool STAGE>
__global__ void __launch_bounds__(kFilterThreads, STAGE ? 2 : 4) chain_filter_kernel(const ChainParams P) {
  pdl_wait();  // the draft lengths and tokens may come from the previous kernel
  pdl_launch_dependents();
  filter_row<DT, VEC, STAGE>(P, STAGE ? static_cast<int>(blockIdx.x) / P.cluster : static_cast<int>(blockIdx.x));
}

// Cluster geometry: at most 16 CTAs, each slice at most 96 KB of logits.
constexpr int kFilterMaxSliceBytes = 96 * 1024;

bool chain_filter_plan(ChainParams &P) {
  const int es = P.dtype == SPEC_DTYPE_F32 ? 4 : 2, epg = 16 / es;
  const long long bytes = static_cast<long long>(P.V) * es;
  long long cs = (bytes + kFilterMaxSliceBytes - 1) / kFilterMaxSliceBytes;
  if (cs < 1) cs = 1;
  if (cs > 16) return false;
  P.cluster = static_cast<int>(cs);
  P.slice = static_cast<int>(((P.V + cs - 1) / cs + epg - 1) / epg * epg);
  return true;
}

cudaError_t launch_chain_filter(const ChainParams &P, bool vec, cudaStream_t st) {
  const int es = P.dtype == SPEC_DTYPE_F32 ? 4 : 2;
  const int rows = P.B * (2 * P.k + 1);
  // row mode when top-k is on (its window needs it) and the rows alone fill
  // the GPU; otherwise a cluster per row splits each row over several SMs
  const bool row_mode = P.top_k > 0 && P.top_k < P.V && rows >= kFilterRowMinRowsPerSm * device_sm_count();
  const int cs = row_mode ? 1 : P.cluster;
  const size_t smem = row_mode ? 0 : static_cast<size_t>(P.slice) * es;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess && cs > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(rows * cs));
    cfg.blockDim = dim3(kFilterThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return trace_launch_ex(row_mode ? "chain_filter_rows" : "chain_filter", st,
                           [&] { return cudaLaunchKernelEx(&cfg, kern, P); });
  };
  if (row_mode) {
    if (P.dtype == SPEC_DTYPE_BF16)
      return vec ? go(chain_filter_kernel<SPEC_DTYPE_BF16, true, false>)
                 : go(chain_filter_kernel<SPEC_DTYPE_BF16, false, false>);
    return vec ? go(chain_filter_kernel<SPEC_DTYPE_F32, true, false>) : go(chain_filter_kernel<SPEC_DTYPE_F32, false, false>);
  }
  if (P.dtype == SPEC_DTYPE_BF16)
    return vec ? go(chain_filter_kernel<SPEC_DTYPE_BF16, true, true>) : go(chain_filter_kernel<SPEC_DTYPE_BF16, false, true>);
  return vec ? go(chain_filter_kernel<SPEC_DTYPE_F32, true, true>) : go(chain_filter_kernel<SPEC_DTYPE_F32, false, true>);
}

}  // namespace sv
