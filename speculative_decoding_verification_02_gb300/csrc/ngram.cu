// n-gram history-lookup drafter ("第 13 篇：推理引擎一次猜几个字", 逐行要点,
// the 草稿器.猜 line): the last `window` tokens of the history are the key;
// the rightmost earlier place where they occur gives the draft, namely the
// tokens that followed it there.
//
// One CTA of 512 threads per request.  The history is staged through shared
// memory in tiles of kTile start positions walked from the end of the
// history (16-byte loads when the request's row is 16-byte aligned).  Thread
// t tests the starts t, t + 512, ... of the tile against the key, so that
// consecutive threads read consecutive shared-memory words; the block keeps
// the largest matching start (a warp max, then one shared-memory max), and
// the walk stops at the first tile holding a match, since no earlier tile
// can hold a later start.  The continuation comes from the staged tile when
// it lies there.
#include "common.cuh"
#include "launch.h"

namespace sv {

constexpr int kNgramThreads = 512;
constexpr int kNgramWarps = kNgramThreads / 32;
constexpr int kTile = 8 * kNgramThreads;  // start positions per tile (16 KB of history)

__global__ void __launch_bounds__(kNgramThreads) ngram_kernel(const NgramParams P) {
  __shared__ __align__(16) int s_hist[kTile + SPEC_MAX_WINDOW + 4];
  __shared__ int s_key[SPEC_MAX_WINDOW];
  __shared__ int s_wbest[kNgramWarps];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_launch_dependents();
  pdl_wait();  // launched early behind the previous kernel in the stream: wait before reading
  const int n = P.hist_len[b], w = P.window, k = P.k;
  const int32_t *h = P.history + static_cast<int64_t>(b) * P.hist_stride;
  int32_t *d = P.draft + static_cast<int64_t>(b) * k;
  if (n < 0 || n > P.hist_stride) {
    for (int j = tid; j < k; j += kNgramThreads) d[j] = -1;
    if (tid == 0) {
      P.draft_len[b] = 0;
      if (P.status) P.status[b] = SPEC_STATUS_BAD_LENGTH;
    }
    return;
  }
  if (tid < w && n >= w) s_key[tid] = h[n - w + tid];
  const bool vec = (reinterpret_cast<uintptr_t>(h) & 15u) == 0;
  const int nstart = n - w;  // start positions i in [0, n - w)
  int best = -1, a0 = 0, cnt = 0;
  for (int t1 = nstart; t1 > 0; t1 -= kTile) {
    const int t0 = max(0, t1 - kTile);
    // stage h[a0, t1 + w - 1): every start in [t0, t1) with its window
    a0 = vec ? (t0 & ~3) : t0;
    cnt = t1 + w - 1 - a0;
    if (vec) {
      const int4 *src = reinterpret_cast<const int4 *>(h + a0);
      const int nv = cnt >> 2;
      for (int i = tid; i < nv; i += kNgramThreads) reinterpret_cast<int4 *>(s_hist)[i] = __ldg(src + i);
      for (int i = (nv << 2) + tid; i < cnt; i += kNgramThreads) s_hist[i] = __ldg(h + a0 + i);
    } else {
      for (int i = tid; i < cnt; i += kNgramThreads) s_hist[i] = __ldg(h + a0 + i);
    }
    __syncthreads();
    int mine = -1;
    for (int i = t0 + tid; i < t1; i += kNgramThreads) {  // ascending: this thread's last match wins
      bool same = true;
      for (int j = 0; j < w && same; ++j) same = s_hist[i - a0 + j] == s_key[j];
      if (same) mine = i;
    }
    mine = __reduce_max_sync(0xffffffffu, mine);
    if (lane == 0) s_wbest[warp] = mine;
    __syncthreads();
    best = __reduce_max_sync(0xffffffffu, lane < kNgramWarps ? s_wbest[lane] : -1);
    if (best >= 0) break;  // the same in every thread
  }
  const int len = best >= 0 ? min(k, n - (best + w)) : 0;
  for (int j = tid; j < k; j += kNgramThreads) {
    const int v = best + w + j;  // in [a0, n) when j < len
    d[j] = j < len ? (v - a0 < cnt ? s_hist[v - a0] : __ldg(h + v)) : -1;
  }
  if (tid == 0) {
    P.draft_len[b] = len;
    if (P.status) P.status[b] = SPEC_STATUS_OK;
  }
}

cudaError_t launch_ngram(const NgramParams &P, cudaStream_t st) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(P.B));
  cfg.blockDim = dim3(kNgramThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = trace_enabled() ? 0 : 1;
  return trace_launch_ex("ngram_draft", st, [&] { return cudaLaunchKernelEx(&cfg, ngram_kernel, P); });
}

}  // namespace sv
