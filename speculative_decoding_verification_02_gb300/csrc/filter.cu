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
// the row in shared memory.  Both thresholds are found by radix selection on
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

template <int DT>
__device__ __forceinline__ uint32_t elem_bits(const void *s, int e) {
  if (DT == SPEC_DTYPE_F32) return reinterpret_cast<const uint32_t *>(s)[e];
  return static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(s)[e]) << 16;
}

// Cluster-wide sum of one value per CTA, added in rank order (the same
// result in every CTA).  `slot` is a [kMaxCluster] array in shared memory.
template <class T>
__device__ __forceinline__ T cluster_sum_ranked(cg::cluster_group &cluster, T *slot, T v, int CS, int rank) {
  if (threadIdx.x < CS) *cluster.map_shared_rank(&slot[rank], threadIdx.x) = v;
  cluster.sync();
  T s = T(0);
  for (int q = 0; q < CS; ++q) s += slot[q];
  return s;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kFilterThreads) chain_filter_kernel(const ChainParams P) {
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int EPG = Elems<DT>::kPerGroup, ES = Elems<DT>::kSize;
  constexpr int kLevels = DT == SPEC_DTYPE_F32 ? 4 : 2;
  constexpr int kMaxCS = 16;
  const int CS = P.cluster, rank = static_cast<int>(cluster.block_rank());
  const int j = blockIdx.x / CS;  // row of the partials layout: request b, row r
  const int k = P.k, K1 = k + 1, R = 2 * k + 1;
  const int b = j / R, r = j - b * R;
  const int side = r < K1 ? 0 : 1, i = side ? r - K1 : r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = P.V;
  const float c = P.c;

  pdl_wait();  // the draft lengths and tokens may come from the previous kernel
  pdl_launch_dependents();
  const int L = P.draft_len ? P.draft_len[b] : k;
  // the rows verification reads: targets 0..L, drafts 0..L-1 (the same in the whole cluster)
  if (L < 0 || L > k || (side == 0 ? i > L : i >= L)) return;
  if (r == 0 && rank == 0 && tid == 0 && P.counter2) P.counter2[b] = 0;  // for the chunked accept kernel
  const char *row = side ? row_ptr<DT>(P.draftl, P.d_req, P.row, b, i) : row_ptr<DT>(P.target, P.t_req, P.row, b, i);
  const int lo = min(V, rank * P.slice), hi = min(V, lo + P.slice), n = hi - lo;

  extern __shared__ __align__(16) unsigned char dyn_filter[];
  unsigned char *s_row = dyn_filter;  // [slice] the slice's logits
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
  if (VEC) {
    const int ng = n / EPG;  // n is a multiple of EPG on the 16-byte path
    for (int g = tid; g < ng; g += kFilterThreads) {
      const uint4 w = __ldg(reinterpret_cast<const uint4 *>(row + static_cast<int64_t>(lo + g * EPG) * ES));
      reinterpret_cast<uint4 *>(s_row)[g] = w;
      float x[EPG];
      unpack16<DT>(w, x);
#pragma unroll
      for (int e = 0; e < EPG; ++e) mloc = fmaxf(mloc, x[e]);
    }
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
  const float Mc = M * c;

  // ---- radix selection: one level of the histogram walk.  Builds the
  // level's cluster-wide histogram of digit (key >> shift) & 255 over the
  // logits whose key >> (shift + 8) equals `prefix` (all logits at the first
  // level) and >= floor; then warp 0 walks the bins from the top until the
  // count (BY_MASS: the mass) reaches `need`.  Returns the digit; `rest`
  // becomes need minus what the bins above the digit hold.
  int level_no = 0;
  auto level = [&](int shift, uint32_t prefix, bool first, float floor, bool by_mass,
                   unsigned long long need, unsigned long long &rest) -> uint32_t {
    const int buf = level_no++ & 1;  // the other buffer may still be read by other CTAs
    for (int d = tid; d < 256; d += kFilterThreads) {
      s_cnt[buf][d] = 0u;
      s_mass[buf][d] = 0ull;
    }
    __syncthreads();
    for (int e = tid; e < n; e += kFilterThreads) {
      const uint32_t bits = elem_bits<DT>(s_row, e);
      const uint32_t key = order_key(bits);
      if (!first && (key >> (shift + 8)) != prefix) continue;
      const float x = __uint_as_float(bits);
      if (!(x >= floor)) continue;
      const uint32_t d = (key >> shift) & 255u;
      atomicAdd(&s_cnt[buf][d], 1u);
      if (by_mass) {
        const double w = static_cast<double>(ex2(fmaf(x, c, -Mc))) * kMassScale;
        atomicAdd(&s_mass[buf][d], static_cast<unsigned long long>(w));
      }
    }
    cluster.sync();  // every CTA's histogram is complete
    for (int d = tid; d < 256; d += kFilterThreads) {
      uint32_t cnt = 0u;
      unsigned long long ms = 0ull;
      for (int q = 0; q < CS; ++q) {
        cnt += *cluster.map_shared_rank(&s_cnt[buf][d], q);
        if (by_mass) ms += *cluster.map_shared_rank(&s_mass[buf][d], q);
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

  // ---- top-k: the top_k-th largest key
  float theta = -INFINITY;
  if (P.top_k > 0 && P.top_k < V) {
    uint32_t prefix = 0u;
    unsigned long long need = static_cast<unsigned long long>(P.top_k), rest = 0ull;
    for (int lv = 0; lv < kLevels; ++lv) {
      const int shift = 24 - 8 * lv;
      const uint32_t d = level(shift, prefix, lv == 0, -INFINITY, false, need, rest);
      prefix = (prefix << 8) | d;
      need = rest;
    }
    theta = prefix_value<DT>(prefix, kLevels);
  }
  // ---- top-p over the logits top-k kept
  if (P.top_p < 1.0f) {
    uint32_t prefix = 0u;
    unsigned long long need = 0ull, rest = 0ull;
    for (int lv = 0; lv < kLevels; ++lv) {
      const int shift = 24 - 8 * lv;
      if (lv == 0) {
        // the first level's histogram also gives the kept mass: need = top_p of it
        // (a first pass with need = max makes the walk fall through; the histogram stays)
        (void)level(shift, 0u, true, theta, true, ~0ull, rest);
        unsigned long long total = 0ull;
        for (int d = 0; d < 256; ++d) total += t_mass[d];
        need = static_cast<unsigned long long>(static_cast<double>(P.top_p) * static_cast<double>(total));
        if (need == 0ull) need = 1ull;
        // pick the digit from the same histogram
        if (tid == 0) {
          unsigned long long run = 0ull;
          int sel = -1, last = -1;
          for (int d = 255; d >= 0; --d) {
            if (t_cnt[d] == 0u) continue;
            last = d;
            if (run + t_mass[d] >= need) {
              sel = d;
              break;
            }
            run += t_mass[d];
          }
          if (sel < 0) {
            sel = last < 0 ? 0 : last;
            run = 0ull;
            for (int d = 255; d > sel; --d) run += t_mass[d];
          }
          s_sel_digit = static_cast<uint32_t>(sel);
          s_sel_rest = need > run ? need - run : 1ull;
        }
        __syncthreads();
        prefix = s_sel_digit;
        need = s_sel_rest;
        __syncthreads();
      } else {
        const uint32_t d = level(shift, prefix, false, theta, true, need, rest);
        prefix = (prefix << 8) | d;
        need = rest;
      }
    }
    theta = fmaxf(theta, prefix_value<DT>(prefix, kLevels));
  }

  // ---- the kept logits: their mass, count and smallest value
  float s_loc = 0.0f, mn = INFINITY;
  uint32_t cnt = 0u;
  for (int e = tid; e < n; e += kFilterThreads) {
    const float x = __uint_as_float(elem_bits<DT>(s_row, e));
    if (x >= theta) {
      s_loc += ex2(fmaf(x, c, -Mc));
      mn = fminf(mn, x);
      ++cnt;
    }
  }
  s_loc = warp_sum(s_loc);
  mn = -warp_allmax(-mn);
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  __shared__ float s_mn[kFilterWarps];
  if (lane == 0) {
    s_red[warp] = s_loc;
    s_redu[warp] = cnt;
    s_mn[warp] = mn;
  }
  __syncthreads();
  if (warp == 0) {
    s_loc = warp_sum(lane < kFilterWarps ? s_red[lane] : 0.0f);
    cnt = __reduce_add_sync(0xffffffffu, lane < kFilterWarps ? s_redu[lane] : 0u);
    mn = -warp_allmax(-(lane < kFilterWarps ? s_mn[lane] : INFINITY));
  }
  __shared__ float s_cmn[kMaxCS];
  if (tid == 0) s_red[0] = s_loc, s_redu[0] = cnt, s_mn[0] = mn;
  __syncthreads();
  if (tid < CS) *cluster.map_shared_rank(&s_cmn[rank], tid) = s_mn[0];
  const float S = cluster_sum_ranked(cluster, s_cs, s_red[0], CS, rank);
  const uint32_t kept = cluster_sum_ranked(cluster, s_cu, s_redu[0], CS, rank);
  if (rank == 0 && tid == 0) {
    float smallest = INFINITY;
    for (int q = 0; q < CS; ++q) smallest = fminf(smallest, s_cmn[q]);
    float xtok = -INFINITY;
    if (i < L) {
      const int tok = P.draft[static_cast<int64_t>(b) * k + i];
      if (tok >= 0 && tok < V) xtok = load_one<DT>(row, tok);
    }
    P.part[j] = Partial{M, S, kNoIndex, xtok};
    P.theta[j] = smallest;
    if (P.kept) P.kept[j] = static_cast<int32_t>(kept);
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
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
  const size_t smem = static_cast<size_t>(P.slice) * es;
  const int rows = P.B * (2 * P.k + 1);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess && P.cluster > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(rows * P.cluster));
    cfg.blockDim = dim3(kFilterThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return trace_launch_ex("chain_filter", st, [&] { return cudaLaunchKernelEx(&cfg, kern, P); });
  };
  if (P.dtype == SPEC_DTYPE_BF16)
    return vec ? go(chain_filter_kernel<SPEC_DTYPE_BF16, true>) : go(chain_filter_kernel<SPEC_DTYPE_BF16, false>);
  return vec ? go(chain_filter_kernel<SPEC_DTYPE_F32, true>) : go(chain_filter_kernel<SPEC_DTYPE_F32, false>);
}

}  // namespace sv
