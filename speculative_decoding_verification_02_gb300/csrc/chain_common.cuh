// Per-request pieces of chain verification shared by the two-kernel path
// (chain.cu) and the fused cluster kernel (chain_fused.cu): row addressing,
// the request prologue (draft length, tokens, uniforms, emission cap, input
// checks) and the outputs that do not depend on the final draw.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace sv {

template <int DT>
__device__ __forceinline__ const char *row_ptr(const char *base, int64_t req_stride,
                                               int64_t row_stride, int b, int i) {
  return base + (static_cast<int64_t>(b) * req_stride + static_cast<int64_t>(i) * row_stride) *
                    Elems<DT>::kSize;
}

// Inputs of one request, read before the dependency wait.
struct Prologue {
  int L, bad, cap;
};

// Validates a request whose draft length, emission cap and tokens are
// already in shared memory (called by all threads).
__device__ __forceinline__ Prologue check_request(const ChainParams &P, int L, int cap, const int *sTok) {
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = (L >= 0 && L <= P.k) ? SPEC_STATUS_OK : SPEC_STATUS_BAD_LENGTH;
  __syncthreads();
  if (s_bad == SPEC_STATUS_OK && tid < L && (sTok[tid] < 0 || sTok[tid] >= P.V))
    atomicMax(&s_bad, SPEC_STATUS_TOKEN_RANGE);
  __syncthreads();
  Prologue pr{L, s_bad, cap};
  __syncthreads();
  return pr;
}

__device__ __forceinline__ Prologue read_request(const ChainParams &P, int b, int *sTok, float *sU, bool sample) {
  __shared__ int s_L, s_cap;
  const int tid = threadIdx.x, k = P.k;
  if (tid == 0) s_L = P.draft_len ? P.draft_len[b] : k;
  if (tid == 32) s_cap = P.max_emit ? P.max_emit[b] : k + 1;
  if (tid < k) sTok[tid] = P.draft[static_cast<int64_t>(b) * k + tid];
  if (sample && tid >= 64 && tid <= 64 + k) sU[tid - 64] = P.uniforms[static_cast<int64_t>(b) * (k + 1) + tid - 64];
  __syncthreads();
  return check_request(P, s_L, s_cap, sTok);
}

// The outputs that do not depend on the final draw (written once per
// request), by threads t = 0 .. nt - 1 (the whole block by default).
template <bool SAMPLE>
__device__ __forceinline__ void write_common(const ChainParams &P, int b, int bad, int L, int m, int ne,
                                             const int *sTok, const float *sP, const float *sQ,
                                             bool final_known, int final_tok, int t = threadIdx.x,
                                             int nt = blockDim.x) {
  const int k = P.k;
  int32_t *out = P.out_tokens + static_cast<int64_t>(b) * (k + 1);
  const int tid = t;
  for (int j = tid; j <= k; j += nt) {
    if (bad) {
      out[j] = -1;
    } else {
      if (j == m && j < ne && !final_known) continue;  // the drawing CTA writes it
      out[j] = j < ne ? (j < m ? sTok[j] : final_tok) : -1;
    }
  }
  if (SAMPLE) {
    for (int j = tid; j < k; j += nt) {
      const bool ok = !bad && j < L;
      if (P.p_tok) P.p_tok[static_cast<int64_t>(b) * k + j] = ok ? sP[j] : -1.0f;
      if (P.q_tok) P.q_tok[static_cast<int64_t>(b) * k + j] = ok ? sQ[j] : -1.0f;
    }
  }
  if (tid == 0) {
    P.accepted[b] = bad ? 0 : m;
    P.n_emit[b] = bad ? 0 : ne;
    if (P.status) P.status[b] = bad;
    if (SAMPLE && bad && P.resid_mass) P.resid_mass[b] = 0.0f;
  }
}

}  // namespace sv
