// EAGLE-2 post-processing of candidate draft trees ("Speculative Decoding
// II", section "Context-Aware Dynamic Draft Tree" and its worked example): a
// node's value is the product of the draft confidences along its path from
// the root; the m most valuable nodes are kept (equal values: the shallower
// node, then the lower id, so the kept nodes stay a tree rooted at the
// root); they are flattened by depth for the target's forward, and each may
// attend only to itself and its ancestors.
//
// One CTA of 512 threads per request, everything in shared memory:
//   1. parents and confidences are loaded and checked;
//   2. depths by pointer jumping over the parent array;
//   3. values level by level from the root, V(i) = V(parent(i)) * c_i in
//      fp32 (the order the page multiplies in, and the order that decides
//      the ranking);
//   4. one bitonic sort of 64-bit keys (value, then shallower, then lower
//      id) ranks every node; the first m are kept;
//   5. a second bitonic sort orders the kept nodes by (depth, id);
//   6. the outputs, and the mask: the request's m x m bytes zeroed by the
//      block, then each row's thread marks the row's ancestors.
#include "common.cuh"
#include "launch.h"

namespace sv {

constexpr int kRerankThreads = 512;

__device__ __forceinline__ int pow2_ceil(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// Block-wide bitonic sort of s[0, n) (n a power of two) into descending
// order of the unsigned keys.
template <class K>
__device__ void bitonic_desc(K *s, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kRerankThreads) {
        const int l = i ^ j;
        if (l > i) {
          const K a = s[i], b = s[l];
          // descending within blocks whose bit k is clear, ascending otherwise
          if (((i & k) == 0) ? (a < b) : (a > b)) {
            s[i] = b;
            s[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kRerankThreads) tree_rerank_kernel(const RerankParams P) {
  extern __shared__ __align__(16) unsigned char dyn_rr[];
  const int N = P.N, m = P.m, b = blockIdx.x, tid = threadIdx.x;
  const int npad = pow2_ceil(N), mpad = pow2_ceil(min(m, N));
  unsigned long long *s_key = reinterpret_cast<unsigned long long *>(dyn_rr);  // [npad]
  int *s_par = reinterpret_cast<int *>(s_key + npad);                         // [N]
  float *s_val = reinterpret_cast<float *>(s_par + N);                        // [N] confidences, then values
  int *s_dep = reinterpret_cast<int *>(s_val + N);                            // [N]
  int *s_anc = s_dep + N;                                                     // [N] pointer jumping
  int *s_anc2 = s_anc + N;                                                    // [N]
  int *s_dep2 = s_anc2 + N;                                                   // [N]; then the kept nodes' slots
  __shared__ int s_bad, s_maxd;

  const int32_t *par = P.parents + static_cast<int64_t>(b) * N;
  const float *conf = P.conf + static_cast<int64_t>(b) * N;
  if (tid == 0) {
    s_bad = par[0] != -1;
    s_maxd = 0;
  }
  __syncthreads();
  // ---- 1. load and check
  for (int i = tid; i < N; i += kRerankThreads) {
    const int p = par[i];
    const float c = i == 0 ? 1.0f : conf[i];
    s_par[i] = p;
    s_val[i] = c;
    if (i > 0 && (p < 0 || p >= i || !(c >= 0.0f && c <= 1.0f))) s_bad = 1;
    s_anc[i] = i == 0 ? -1 : p;
    s_dep[i] = i == 0 ? 0 : 1;
  }
  __syncthreads();
  // ---- 2. depths: s_dep[i] edges from i up to s_anc[i]; each round doubles
  // the reach, and a depth is below N, so ceil(log2 N) rounds reach the root
  const int rounds = s_bad ? 0 : 32 - __clz(max(N - 1, 1));
  for (int round = 0; round < rounds; ++round) {
    for (int i = tid; i < N; i += kRerankThreads) {
      const int a = s_anc[i];
      s_anc2[i] = a >= 0 ? s_anc[a] : -1;
      s_dep2[i] = s_dep[i] + (a >= 0 ? s_dep[a] : 0);
    }
    __syncthreads();
    for (int i = tid; i < N; i += kRerankThreads) {
      s_anc[i] = s_anc2[i];
      s_dep[i] = s_dep2[i];
    }
    __syncthreads();
  }
  for (int i = tid; i < N && !s_bad; i += kRerankThreads) atomicMax(&s_maxd, s_dep[i]);
  __syncthreads();
  if (tid == 0 && s_maxd > P.max_depth) s_bad = 1;
  __syncthreads();

  int32_t *o_node = P.sel_nodes + static_cast<int64_t>(b) * m;
  int32_t *o_par = P.sel_parents + static_cast<int64_t>(b) * m;
  int32_t *o_dep = P.sel_depth + static_cast<int64_t>(b) * m;
  float *o_val = P.sel_value ? P.sel_value + static_cast<int64_t>(b) * m : nullptr;
  int32_t *o_tok = P.sel_tok ? P.sel_tok + static_cast<int64_t>(b) * m : nullptr;
  uint8_t *o_mask = P.mask ? P.mask + static_cast<int64_t>(b) * m * m : nullptr;
  const int n = s_bad ? 0 : min(m, N);
  // ---- 6a. padding, and the mask's zero fill (16-byte stores where aligned)
  for (int j = n + tid; j < m; j += kRerankThreads) {
    o_node[j] = o_par[j] = o_dep[j] = -1;
    if (o_val) o_val[j] = -1.0f;
    if (o_tok) o_tok[j] = -1;
  }
  if (o_mask) {
    const int64_t bytes = static_cast<int64_t>(m) * m;
    if ((reinterpret_cast<uintptr_t>(o_mask) & 15u) == 0) {
      const int64_t nv = bytes >> 4;
      for (int64_t i = tid; i < nv; i += kRerankThreads) reinterpret_cast<uint4 *>(o_mask)[i] = make_uint4(0, 0, 0, 0);
      for (int64_t i = (nv << 4) + tid; i < bytes; i += kRerankThreads) o_mask[i] = 0;
    } else {
      for (int64_t i = tid; i < bytes; i += kRerankThreads) o_mask[i] = 0;
    }
  }
  if (s_bad) {
    if (tid == 0) {
      P.n_sel[b] = 0;
      if (P.status) P.status[b] = SPEC_STATUS_BAD_TREE;
    }
    return;
  }
  // ---- 3. values from the root down, one depth at a time
  const int maxd = s_maxd;
  for (int d = 1; d <= maxd; ++d) {
    for (int i = tid; i < N; i += kRerankThreads)
      if (s_dep[i] == d) s_val[i] = s_val[s_par[i]] * s_val[i];
    __syncthreads();
  }
  // ---- 4. rank: value (non-negative, so its bits, sign cleared for a -0,
  // order like the value), then shallower, then lower id; padding keys are 0
  // and sort last
  for (int i = tid; i < npad; i += kRerankThreads) {
    s_key[i] = i < N ? (static_cast<unsigned long long>(__float_as_uint(s_val[i]) & 0x7fffffffu) << 32) |
                           (static_cast<unsigned long long>(0xFFFFu - s_dep[i]) << 16) | (0xFFFFu - i)
                     : 0ull;
  }
  __syncthreads();
  bitonic_desc(s_key, npad);
  // ---- 5. the kept nodes in (depth, id) order: descending on the complement
  // [mpad] over s_anc2 and s_dep2 (pointer jumping is done; mpad < 2N)
  unsigned *s_flat = reinterpret_cast<unsigned *>(s_anc2);
  for (int j = tid; j < mpad; j += kRerankThreads) {
    unsigned key = 0u;  // padding sorts last
    if (j < n) {
      const unsigned id = 0xFFFFu - static_cast<unsigned>(s_key[j] & 0xFFFFu);
      const unsigned dep = 0xFFFFu - static_cast<unsigned>((s_key[j] >> 16) & 0xFFFFu);
      key = ~((dep << 16) | id);
    }
    s_flat[j] = key;
  }
  int *s_pos = s_anc;  // [N] flattened slot of each kept node, -1 otherwise
  for (int i = tid; i < N; i += kRerankThreads) s_pos[i] = -1;
  __syncthreads();
  bitonic_desc(s_flat, mpad);
  for (int j = tid; j < n; j += kRerankThreads) s_pos[(~s_flat[j]) & 0xFFFFu] = j;
  __syncthreads();
  // ---- 6b. outputs (the mask's zeros are ordered before the ones by the barrier above)
  for (int j = tid; j < n; j += kRerankThreads) {
    const int u = static_cast<int>((~s_flat[j]) & 0xFFFFu);
    o_node[j] = u;
    o_par[j] = u == 0 ? -1 : s_pos[s_par[u]];
    o_dep[j] = s_dep[u];
    if (o_val) o_val[j] = s_val[u];
    if (o_tok) o_tok[j] = P.node_tok[static_cast<int64_t>(b) * N + u];
    if (o_mask) {
      uint8_t *row = o_mask + static_cast<int64_t>(j) * m;
      for (int a = u; a >= 0; a = a == 0 ? -1 : s_par[a]) row[s_pos[a]] = 1;  // ancestors are all kept
    }
  }
  if (tid == 0) {
    P.n_sel[b] = n;
    if (P.status) P.status[b] = SPEC_STATUS_OK;
  }
}

size_t tree_rerank_smem(int N, int m) {
  (void)m;
  const size_t npad = static_cast<size_t>(1) << (N > 1 ? 32 - __builtin_clz(static_cast<unsigned>(N - 1)) : 0);
  return sizeof(unsigned long long) * npad + sizeof(int) * 6 * static_cast<size_t>(N);
}

cudaError_t launch_tree_rerank(const RerankParams &P, cudaStream_t st) {
  const size_t smem = tree_rerank_smem(P.N, P.m);
  cudaError_t e = cudaFuncSetAttribute(tree_rerank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return trace_launch("tree_rerank", st, [&] {
    tree_rerank_kernel<<<P.B, kRerankThreads, smem, st>>>(P);
  });
}

}  // namespace sv
