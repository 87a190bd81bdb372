// Host-side parameter blocks and launchers shared by the .cu files of the
// library.  Not part of the public ABI (that is include/spec_verify.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "spec_verify.h"

namespace sv {

struct Partial;


struct ChainParams {
  const char *target;
  const char *draftl;
  int64_t t_req, d_req, row;  // element strides
  int dtype, B, k, V;
  int nc, chunk;    // streaming pass: chunks per row, logits per chunk
  int nc2, chunk2;  // chunked accept kernel: chunks per row (<= 256), logits per chunk
  float c;          // log2(e) / T
  const int32_t *draft, *draft_len, *max_emit;
  const float *uniforms;
  int32_t *accepted, *out_tokens, *n_emit, *status;
  float *p_tok, *q_tok, *resid_mass;
  float *final_prob;  // or null: the final token's probability under the distribution it was drawn from
  Partial *part;     // [B][rows][nc] streaming-pass statistics
  float *part2;      // [B][nc2][8] chunked accept kernel: the final draw's weight mass per warp range
  int *counter2;     // [B] arrival counter of the residual pass
  int cluster;       // cluster kernels: CTAs per request (sampling accept: 0 = chunked accept kernel)
  int slice;         // logits per CTA of a cluster kernel
  int groups;        // fused kernel: rounds of 16-byte groups per lane (warp ranges of the slice)
  // top-k / top-p filtering (filter.cu): the filter, and per partial row its
  // threshold (the smallest kept logit) and kept count.  theta == nullptr:
  // unfiltered (the accept kernels keep every logit).
  int top_k;
  float top_p;
  float *theta;
  int32_t *kept;
};

constexpr int kTreeThreads = 512;   // threads per tree-walk CTA
constexpr int kFusedThreads = 512;  // threads per CTA of the fused chain kernel

struct TreeParams {
  const char *target;
  const char *draftl;
  int64_t t_req, d_req, row;
  int dtype, B, N, V, max_depth;
  int cluster;     // CTAs per request
  int slice;       // logits per CTA (multiple of 8)
  int groups;      // rounds of 16-byte groups per lane (each warp: a contiguous range of the slice)
  int stage;       // 1: the first rejection at a node stages p and q of the slice in shared memory
  float c;         // log2(e) / T; unused when greedy
  int greedy;
  int wor;         // siblings drawn without replacement: rejected tokens leave q
  const int32_t *parents, *node_tok;
  const float *uniforms;
  int32_t *accepted_len, *path_nodes, *out_tokens, *n_emit, *status;
};

struct NgramParams {
  const int32_t *history, *hist_len;
  int B, hist_stride, window, k;
  int32_t *draft, *draft_len, *status;
};

// Two-pass chain path: the streaming pass (16-byte loads when vec) and an
// accept kernel -- the cluster accept kernel when P.cluster > 0 (its
// 16-byte path when cvec), else the chunked or greedy accept kernel.
// stats = false (sampling only): the accept kernel alone, on partials the
// filter kernel wrote.
cudaError_t launch_chain(const ChainParams &P, bool sample, bool vec, bool cvec, cudaStream_t st, bool stats = true);
// Streaming multiprocessors of the current device (queried once per device).
int device_sm_count();
// Cluster kernels (chain_fused.cu).  The plans pick the cluster geometry
// (cluster, slice, groups) and return false when the requests' clusters
// cannot all be resident at once.  chain_fused_plan: the fused one-launch
// kernel; chain_accept_plan: the two-pass path's cluster accept kernel.
bool chain_fused_plan(ChainParams &P, bool sample, bool vec);
bool chain_accept_plan(ChainParams &P, bool vec);
cudaError_t launch_chain_fused(const ChainParams &P, bool sample, bool vec, cudaStream_t st);
cudaError_t launch_chain_accept_cluster(const ChainParams &P, bool vec, cudaStream_t st);
// Top-k / top-p filter of every partial row (filter.cu): writes the row's
// statistics over its kept logits as partial P.part[row] (one chunk per row)
// and its threshold P.theta[row].  The plan picks the cluster geometry
// (cluster, slice) and returns false when a row is too long (more than 16
// slices of 96 KB).
bool chain_filter_plan(ChainParams &P);
cudaError_t launch_chain_filter(const ChainParams &P, bool vec, cudaStream_t st);
cudaError_t launch_tree(const TreeParams &P, bool vec, cudaStream_t st);
size_t tree_dynamic_smem(const TreeParams &P);
cudaError_t launch_ngram(const NgramParams &P, cudaStream_t st);

struct RerankParams {
  const int32_t *parents;
  const float *conf;
  const int32_t *node_tok;
  int B, N, m, max_depth;
  int32_t *sel_nodes, *sel_parents, *sel_depth;
  float *sel_value;
  int32_t *sel_tok;
  uint8_t *mask;
  int32_t *n_sel, *status;
};
cudaError_t launch_tree_rerank(const RerankParams &P, cudaStream_t st);

// Tracing hooks (api.cu).  trace_begin returns a slot (or -1 when tracing is
// off); trace_end records the closing event of that slot.
int trace_begin(const char *name, cudaStream_t st);
void trace_end(int slot, cudaStream_t st);
void count_launch();
// Sets the message spec_last_error() returns on this thread.
void set_last_error(const char *msg);
// True while spec_trace_enable(1) is in force.  Traced calls launch their
// dependent kernels without programmatic dependent launch, so that each
// kernel's event pair brackets only its own execution.
bool trace_enabled();
// Launches of each kernel inside its event pair while tracing (1 otherwise).
int trace_repeats();

template <class F>
cudaError_t trace_launch(const char *name, cudaStream_t st, F &&launch) {
  const int slot = trace_begin(name, st);
  const int reps = slot >= 0 ? trace_repeats() : 1;
  cudaError_t e = cudaSuccess;
  for (int r = 0; r < reps && e == cudaSuccess; ++r) {
    launch();
    e = cudaGetLastError();
    count_launch();
  }
  trace_end(slot, st);
  return e;
}

template <class F>
cudaError_t trace_launch_ex(const char *name, cudaStream_t st, F &&launch) {
  const int slot = trace_begin(name, st);
  const int reps = slot >= 0 ? trace_repeats() : 1;
  cudaError_t e = cudaSuccess;
  for (int r = 0; r < reps && e == cudaSuccess; ++r) {
    e = launch();
    if (e == cudaSuccess) e = cudaGetLastError();
    count_launch();
  }
  trace_end(slot, st);
  return e;
}

}  // namespace sv
