// n-gram history-lookup drafter ("第 13 篇：推理引擎一次猜几个字", 逐行要点,
// the 草稿器.猜 line): the last `window` tokens of the history are the key;
// the rightmost earlier place where they occur gives the draft, namely the
// tokens that followed it there.
//
// One CTA per request.  The history is staged through shared memory in
// tiles walked from the end of the history towards its start; every thread
// compares the key at its start positions, the block keeps the largest
// matching start (atomicMax), and the walk stops at the first tile holding a
// match, since no earlier tile can hold a later start.
#include "common.cuh"
#include "launch.h"

namespace sv {

constexpr int kTile = 8192;  // start positions per tile (32 KB of history)

__global__ void __launch_bounds__(kThreads) ngram_kernel(const NgramParams P) {
  __shared__ int s_hist[kTile + SPEC_MAX_WINDOW];
  __shared__ int s_key[SPEC_MAX_WINDOW];
  __shared__ int s_best;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int n = P.hist_len[b], w = P.window, k = P.k;
  const int32_t *h = P.history + static_cast<int64_t>(b) * P.hist_stride;
  int32_t *d = P.draft + static_cast<int64_t>(b) * k;
  if (n < 0 || n > P.hist_stride) {
    for (int j = tid; j < k; j += kThreads) d[j] = -1;
    if (tid == 0) {
      P.draft_len[b] = 0;
      if (P.status) P.status[b] = SPEC_STATUS_BAD_LENGTH;
    }
    return;
  }
  if (tid == 0) s_best = -1;
  if (tid < w && n >= w) s_key[tid] = h[n - w + tid];
  __syncthreads();
  const int nstart = n - w;  // start positions i in [0, n - w)
  for (int t1 = nstart; t1 > 0; t1 -= kTile) {
    const int t0 = max(0, t1 - kTile);
    // stage h[t0, t1 + w - 1): every start in [t0, t1) with its window
#pragma unroll 8
    for (int i = tid; i < t1 - t0 + w - 1; i += kThreads) s_hist[i] = __ldg(h + t0 + i);
    __syncthreads();
    for (int i = t1 - 1 - tid; i >= t0; i -= kThreads) {
      bool same = true;
      for (int j = 0; j < w && same; ++j) same = s_hist[i - t0 + j] == s_key[j];
      if (same) atomicMax(&s_best, i);
    }
    __syncthreads();
    if (s_best >= 0) break;
  }
  const int best = s_best;
  const int len = best >= 0 ? min(k, n - (best + w)) : 0;
  for (int j = tid; j < k; j += kThreads) d[j] = j < len ? h[best + w + j] : -1;
  if (tid == 0) {
    P.draft_len[b] = len;
    if (P.status) P.status[b] = SPEC_STATUS_OK;
  }
}

cudaError_t launch_ngram(const NgramParams &P, cudaStream_t st) {
  return trace_launch("ngram_draft", st, [&] { ngram_kernel<<<P.B, kThreads, 0, st>>>(P); });
}

}  // namespace sv
