// C ABI of libspecverify.so: argument checks, workspace layout, launch
// geometry, error mapping and tracing.  The arithmetic lives in chain.cu,
// tree.cu and ngram.cu.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "launch.h"

namespace sv {
namespace {

thread_local char g_last_error[256] = "";

int fail_cuda(cudaError_t e, const char *where) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return SPEC_ECUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int dtype) { return dtype == SPEC_DTYPE_BF16 ? 2 : 4; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------ geometry

// Logits per CTA of the streaming pass, sized from the call's total bytes so
// that the grid is about four waves of four CTAs on each SM (152 on a
// GB300), between 16 KB and 128 KB of one row: small calls spread over every
// SM, large ones keep each CTA streaming long enough to amortise its
// start-up and reduction.

// Chain path (spec_set_chain_path).  In AUTO the fused kernel takes
// vocabularies up to kFusedAutoMaxV: 0, since with the cluster accept kernel
// the two-pass path measures faster on every shape tried (B=1..64,
// V=2,048..248,320).
std::atomic<int> g_chain_path{SPEC_CHAIN_AUTO};
constexpr int kFusedAutoMaxV = 0;

int stream_chunk(int dtype, long long rows_total, int V) {
  const long long es = elem_size(dtype);
  const long long target_ctas = static_cast<long long>(device_sm_count()) * 4 * 4;
  const long long per = rows_total * V * es / target_ctas;
  long long bytes = 16384;
  while (bytes < per && bytes < 131072) bytes *= 2;
  return static_cast<int>(bytes / es);
}

// Chunks of the chunked accept kernel: about one wave of its CTAs (two per
// SM) over the whole batch, and at most kThreads chunks per request (the
// last CTA to arrive reads one chunk per thread).  A chunk is G rounds of
// one 16-byte group per thread, G >= 1.
int accept_chunk(int B, int V, int dtype) {
  const long long unit = static_cast<long long>(kThreads) * (16 / elem_size(dtype));
  const long long per_req = std::max<long long>(1, 2LL * device_sm_count() / std::max(B, 1));
  long long g = (V + per_req * unit - 1) / (per_req * unit);
  g = std::max(g, (V + kThreads * unit - 1) / (kThreads * unit));
  return static_cast<int>(std::max<long long>(g, 1) * unit);
}

// Workspace: per-(row, chunk) statistics, then for sampling the draw's
// weight mass per warp range of the chunked accept kernel, one arrival
// counter per request (zeroed by the
// streaming pass of each call, so the workspace needs no initialisation)
// and each row's top-k / top-p threshold.
struct ChainLayout {
  int nc, chunk, nc2, chunk2;
  size_t part, part2, counter2, theta, total;
};

ChainLayout chain_layout(bool sample, int B, int k, int V, int dtype) {
  ChainLayout L{};
  L.chunk = stream_chunk(dtype, static_cast<long long>(B) * (sample ? 2LL * k + 1 : k + 1LL), V);
  L.nc = (V + L.chunk - 1) / L.chunk;
  L.chunk2 = accept_chunk(B, V, dtype);
  L.nc2 = (V + L.chunk2 - 1) / L.chunk2;
  const size_t rows = sample ? 2 * static_cast<size_t>(k) + 1 : static_cast<size_t>(k) + 1;
  size_t off = 0;
  L.part = off;
  off = round_up(off + sizeof(Partial) * B * rows * L.nc, 256);
  L.part2 = off;
  off = round_up(off + sizeof(float) * (sample ? B * static_cast<size_t>(L.nc2) * kWarps : 0), 256);
  L.counter2 = off;
  off = round_up(off + (sample ? sizeof(int) * B : 0), 256);
  L.theta = off;  // top-k / top-p: each row's threshold
  off = round_up(off + (sample ? sizeof(float) * B * rows : 0), 256);
  L.total = off;
  return L;
}

// Tree walk: one thread-block cluster per request, each CTA owns a slice of
// V.  Up to sixteen CTAs (at least 2,048 logits each), but no more than keep
// every cluster resident at once (one walk CTA per SM).
void tree_geometry(int B, int V, int &cluster, int &slice) {
  cluster = V >= 16 * 2048 ? 16 : V >= 8 * 2048 ? 8 : (V >= 4 * 2048 ? 4 : (V >= 2 * 2048 ? 2 : 1));
  while (cluster > 1 && static_cast<long long>(B) * cluster > device_sm_count()) cluster /= 2;
  slice = ((V + cluster - 1) / cluster + 7) / 8 * 8;
}

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// -------------------------------------------------------------- tracing

struct TraceRec {
  const char *name;
  cudaEvent_t start, stop;
};

std::mutex g_trace_mu;
bool g_trace_on = false;
int g_trace_reps = 1;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;
long long g_launches = 0;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Records ev on st.  Under stream capture the record becomes an event-record
// node of the graph (an ordinary record there only orders the capture), so
// every replay of the graph stamps the event again.
void record_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();  // (leave no error for the launch check that follows)
    cs = cudaStreamCaptureStatusNone;
  }
  if (cs == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  else cudaEventRecord(ev, st);
}

}  // namespace

int trace_begin(const char *name, cudaStream_t st) {
  std::lock_guard<std::mutex> g(g_trace_mu);
  if (!g_trace_on) return -1;
  TraceRec r{name, take_event(), take_event()};
  if (!r.start || !r.stop) return -1;
  record_event(r.start, st);
  g_trace.push_back(r);
  return static_cast<int>(g_trace.size()) - 1;
}

void trace_end(int slot, cudaStream_t st) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> g(g_trace_mu);
  if (slot < static_cast<int>(g_trace.size())) record_event(g_trace[slot].stop, st);
}

void count_launch() {
  std::lock_guard<std::mutex> g(g_trace_mu);
  ++g_launches;
}

void set_last_error(const char *msg) { std::snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

int device_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 152;  // (a GB300's count; only reached when there is no device to ask)
  }
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool trace_enabled() {
  std::lock_guard<std::mutex> g(g_trace_mu);
  return g_trace_on;
}

int trace_repeats() {
  std::lock_guard<std::mutex> g(g_trace_mu);
  return g_trace_reps;
}

}  // namespace sv

using namespace sv;

// spec_sample runs the sampling chain with k = 0 (the draw from row 0 with
// uniform 0 is the bonus draw); the accept counts it does not return live
// after the chain's workspace.
static size_t draw_workspace(int B, int V, int dtype) {
  const size_t chain = chain_layout(true, B, 0, V, dtype).total;
  return chain + round_up(2 * sizeof(int32_t) * static_cast<size_t>(B), 256);
}

extern "C" {

size_t spec_workspace_size(int op, int B, int rows_per_req, int V, int dtype) {
  if (B < 0 || rows_per_req < 0 || V <= 0 || (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16))
    return 0;
  switch (op) {
    case SPEC_OP_GREEDY: return chain_layout(false, B, rows_per_req, V, dtype).total;
    case SPEC_OP_SAMPLE: return chain_layout(true, B, rows_per_req, V, dtype).total;
    case SPEC_OP_DRAW: return draw_workspace(B, V, dtype);
    case SPEC_OP_FILTER: return round_up(sizeof(Partial) * static_cast<size_t>(B), 256);
    default: return 0;  // n-gram and tree walks need no workspace
  }
}

const char *spec_status_string(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_EINVAL: return "invalid argument";
    case SPEC_EDTYPE: return "unsupported dtype";
    case SPEC_EWORKSPACE: return "workspace missing, misaligned or too small";
    case SPEC_ECUDA: return "CUDA error (see spec_last_error)";
    case 100 + SPEC_STATUS_OK: return "request ok";
    case 100 + SPEC_STATUS_TOKEN_RANGE: return "request has a token outside [0, V)";
    case 100 + SPEC_STATUS_BAD_TREE: return "request has a malformed or too deep tree";
    case 100 + SPEC_STATUS_BAD_LENGTH: return "request has a length outside its range";
    default: return "unknown code";
  }
}

const char *spec_last_error(void) { return g_last_error; }

int spec_trace_enable(int on) {
  std::lock_guard<std::mutex> g(g_trace_mu);
  g_trace_on = on != 0;
  return SPEC_OK;
}

int spec_trace_repeat(int reps) {
  if (reps < 1 || reps > 1024) return SPEC_EINVAL;
  std::lock_guard<std::mutex> g(g_trace_mu);
  g_trace_reps = reps;
  return SPEC_OK;
}

int spec_trace_collect(const char **names, double *total_ms, int64_t *launches, int cap) {
  std::vector<TraceRec> recs;
  {
    std::lock_guard<std::mutex> g(g_trace_mu);
    recs.swap(g_trace);
  }
  std::vector<const char *> nm;
  std::vector<double> ms;
  std::vector<int64_t> cnt;
  int rc = SPEC_OK;
  for (const TraceRec &r : recs) {
    cudaError_t e = cudaEventSynchronize(r.stop);
    float t = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.start, r.stop);
    if (e != cudaSuccess) rc = fail_cuda(e, "spec_trace_collect");
    size_t i = 0;
    while (i < nm.size() && std::strcmp(nm[i], r.name) != 0) ++i;
    if (i == nm.size()) {
      nm.push_back(r.name);
      ms.push_back(0.0);
      cnt.push_back(0);
    }
    ms[i] += t;
    cnt[i] += 1;
  }
  {
    std::lock_guard<std::mutex> g(g_trace_mu);
    for (const TraceRec &r : recs) {
      g_event_pool.push_back(r.start);
      g_event_pool.push_back(r.stop);
    }
  }
  if (rc != SPEC_OK) return rc;
  for (size_t i = 0; i < nm.size() && static_cast<int>(i) < cap; ++i) {
    if (names) names[i] = nm[i];
    if (total_ms) total_ms[i] = ms[i];
    if (launches) launches[i] = cnt[i];
  }
  return static_cast<int>(nm.size());
}

int spec_set_chain_path(int path) {
  if (path != SPEC_CHAIN_AUTO && path != SPEC_CHAIN_TWO_PASS && path != SPEC_CHAIN_FUSED &&
      path != SPEC_CHAIN_CHUNKED)
    return SPEC_EINVAL;
  g_chain_path.store(path, std::memory_order_relaxed);
  return SPEC_OK;
}

int64_t spec_launch_count(void) {
  std::lock_guard<std::mutex> g(g_trace_mu);
  return g_launches;
}

int spec_ngram_draft(const int32_t *history, const int32_t *hist_len, int B, int hist_stride,
                     int window, int k, int32_t *draft, int32_t *draft_len, int32_t *status,
                     void *stream) {
  if (B < 0 || hist_stride < 0 || window < 1 || window > SPEC_MAX_WINDOW || k < 0 ||
      k > SPEC_MAX_K)
    return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  if (!hist_len || !draft_len || (k > 0 && !draft) || (hist_stride > 0 && !history))
    return SPEC_EINVAL;
  if (static_cast<int64_t>(B) > 2147483647LL) return SPEC_EINVAL;
  NgramParams P{history, hist_len, B, hist_stride, window, k, draft, draft_len, status};
  const cudaError_t e = launch_ngram(P, as_stream(stream));
  return e == cudaSuccess ? SPEC_OK : fail_cuda(e, "spec_ngram_draft");
}

static int chain_common(bool sample, const void *target, int64_t t_req, const void *draftl,
                        int64_t d_req, int64_t row, int dtype, int B, int k, int V, float T,
                        const int32_t *draft, const int32_t *draft_len, const int32_t *max_emit,
                        const float *uniforms, int32_t *accepted, int32_t *out_tokens,
                        int32_t *n_emit, float *p_tok, float *q_tok, float *resid_mass,
                        int32_t *status, void *workspace, size_t workspace_bytes, void *stream,
                        float *final_prob = nullptr, int top_k = 0, float top_p = 1.0f) {
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_EDTYPE;
  if (B < 0 || k < 0 || k > SPEC_MAX_K || V <= 0 || t_req < 0 || d_req < 0 || row < 0)
    return SPEC_EINVAL;
  if (sample && !(T > 0.0f && std::isfinite(T))) return SPEC_EINVAL;
  if (top_k < 0 || !(top_p > 0.0f && top_p <= 1.0f)) return SPEC_EINVAL;
  const bool filtered = sample && ((top_k > 0 && top_k < V) || top_p < 1.0f);
  if (B == 0) return SPEC_OK;
  if (!target || !accepted || !out_tokens || !n_emit || (k > 0 && !draft)) return SPEC_EINVAL;
  if (sample && (!uniforms || (k > 0 && !draftl))) return SPEC_EINVAL;
  const ChainLayout L = chain_layout(sample, B, k, V, dtype);
  const long long rows = sample ? 2LL * k + 1 : k + 1LL;
  if (static_cast<long long>(B) * rows * L.nc > 2147483647LL ||
      static_cast<long long>(B) * L.nc2 > 2147483647LL)
    return SPEC_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < L.total)
    return SPEC_EWORKSPACE;
  const int es = elem_size(dtype);
  const bool vec = aligned16(target) && (!sample || k == 0 || aligned16(draftl)) &&
                   (t_req * es) % 16 == 0 && (d_req * es) % 16 == 0 && (row * es) % 16 == 0;
  char *ws = static_cast<char *>(workspace);
  ChainParams P{};
  P.target = static_cast<const char *>(target);
  P.draftl = static_cast<const char *>(draftl);
  P.t_req = t_req;
  P.d_req = d_req;
  P.row = row;
  P.dtype = dtype;
  P.B = B;
  P.k = k;
  P.V = V;
  P.nc = L.nc;
  P.chunk = L.chunk;
  P.nc2 = L.nc2;
  P.chunk2 = L.chunk2;
  P.c = sample ? static_cast<float>(1.4426950408889634 / static_cast<double>(T)) : 1.0f;
  P.draft = draft;
  P.draft_len = draft_len;
  P.max_emit = max_emit;
  P.uniforms = uniforms;
  P.accepted = accepted;
  P.out_tokens = out_tokens;
  P.n_emit = n_emit;
  P.status = status;
  P.p_tok = p_tok;
  P.q_tok = q_tok;
  P.resid_mass = resid_mass;
  P.final_prob = final_prob;
  P.counter2 = reinterpret_cast<int *>(ws + L.counter2);
  P.part = reinterpret_cast<Partial *>(ws + L.part);
  P.part2 = reinterpret_cast<float *>(ws + L.part2);
  cudaError_t e;
  const bool fvec = vec && V % (16 / es) == 0;  // the fused kernel's 16-byte path also wants V a multiple of a group
  const int path = g_chain_path.load(std::memory_order_relaxed);
  const bool want_fused = path == SPEC_CHAIN_FUSED || (path == SPEC_CHAIN_AUTO && V <= kFusedAutoMaxV);
  const bool chunked = path == SPEC_CHAIN_CHUNKED;

  if (filtered) {
    // the filter kernel replaces the streaming pass: one partial per row
    // (statistics over the kept logits) and each row's threshold, then the
    // accept kernel with the thresholds as masks
    P.top_k = top_k;
    P.top_p = top_p;
    P.theta = reinterpret_cast<float *>(ws + L.theta);
    P.nc = 1;
    P.chunk = V;
    if (!chain_filter_plan(P)) return SPEC_EINVAL;  // a row longer than 16 slices of 96 KB
    e = launch_chain_filter(P, fvec, as_stream(stream));
    if (e == cudaSuccess) {
      if (chunked || !chain_accept_plan(P, fvec)) P.cluster = 0;
      e = launch_chain(P, true, vec, fvec, as_stream(stream), false);
    }
  } else if (want_fused && chain_fused_plan(P, sample, fvec)) {
    e = launch_chain_fused(P, sample, fvec, as_stream(stream));
  } else {
    // two-pass: the cluster accept kernel when every request's cluster is resident
    if (chunked || !(sample && chain_accept_plan(P, fvec))) P.cluster = 0;
    e = launch_chain(P, sample, vec, fvec, as_stream(stream));
  }
  return e == cudaSuccess ? SPEC_OK : fail_cuda(e, sample ? "spec_verify_sample" : "spec_verify_greedy");
}

int spec_sample(const void *logits, int64_t req_stride, int dtype, int B, int V, float temperature,
                const float *uniforms, int32_t *tokens, float *probs, int32_t *status, void *workspace,
                size_t workspace_bytes, void *stream) {
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_EDTYPE;
  if (B < 0 || V <= 0 || req_stride < 0 || !(temperature > 0.0f && std::isfinite(temperature))) return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  if (!logits || !uniforms || !tokens) return SPEC_EINVAL;
  const size_t need = draw_workspace(B, V, dtype);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return SPEC_EWORKSPACE;
  const size_t chain = chain_layout(true, B, 0, V, dtype).total;
  int32_t *accepted = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + chain);
  return chain_common(true, logits, req_stride, nullptr, 0, 0, dtype, B, 0, V, temperature, nullptr, nullptr,
                      nullptr, uniforms, accepted, tokens, accepted + B, nullptr, nullptr, nullptr, status,
                      workspace, chain, stream, probs);
}

int spec_sample_topkp(const void *logits, int64_t req_stride, int dtype, int B, int V, float temperature,
                      int top_k, float top_p, const float *uniforms, int32_t *tokens, float *probs,
                      int32_t *status, void *workspace, size_t workspace_bytes, void *stream) {
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_EDTYPE;
  if (B < 0 || V <= 0 || req_stride < 0 || !(temperature > 0.0f && std::isfinite(temperature))) return SPEC_EINVAL;
  if (top_k < 0 || !(top_p > 0.0f && top_p <= 1.0f)) return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  if (!logits || !uniforms || !tokens) return SPEC_EINVAL;
  const size_t need = draw_workspace(B, V, dtype);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return SPEC_EWORKSPACE;
  const size_t chain = chain_layout(true, B, 0, V, dtype).total;
  int32_t *accepted = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + chain);
  return chain_common(true, logits, req_stride, nullptr, 0, 0, dtype, B, 0, V, temperature, nullptr, nullptr,
                      nullptr, uniforms, accepted, tokens, accepted + B, nullptr, nullptr, nullptr, status,
                      workspace, chain, stream, probs, top_k, top_p);
}

int spec_filter_rows(const void *logits, int64_t row_stride, int dtype, int R, int V, float temperature, int top_k,
                     float top_p, float *theta, int32_t *kept, void *workspace, size_t workspace_bytes,
                     void *stream) {
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_EDTYPE;
  if (R < 0 || V <= 0 || row_stride < 0 || !(temperature > 0.0f && std::isfinite(temperature))) return SPEC_EINVAL;
  if (top_k < 0 || !(top_p > 0.0f && top_p <= 1.0f)) return SPEC_EINVAL;
  if (R == 0) return SPEC_OK;
  if (!logits || !theta) return SPEC_EINVAL;
  const size_t need = round_up(sizeof(Partial) * static_cast<size_t>(R), 256);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return SPEC_EWORKSPACE;
  const int es = elem_size(dtype);
  ChainParams P{};
  P.target = static_cast<const char *>(logits);
  P.t_req = row_stride;  // each row is a request with one position
  P.dtype = dtype;
  P.B = R;
  P.k = 0;
  P.V = V;
  P.c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  P.top_k = top_k;
  P.top_p = top_p;
  P.theta = theta;
  P.kept = kept;
  P.part = static_cast<Partial *>(workspace);
  if (!chain_filter_plan(P)) return SPEC_EINVAL;
  const bool vec = aligned16(logits) && (row_stride * es) % 16 == 0 && V % (16 / es) == 0;
  const cudaError_t e = launch_chain_filter(P, vec, as_stream(stream));
  return e == cudaSuccess ? SPEC_OK : fail_cuda(e, "spec_filter_rows");
}

int spec_verify_sample_topkp(const void *target, int64_t target_req_stride, const void *draft_logits,
                             int64_t draft_req_stride, int64_t row_stride, int dtype, int B, int k, int V,
                             float temperature, int top_k, float top_p, const int32_t *draft,
                             const int32_t *draft_len, const int32_t *max_emit, const float *uniforms,
                             int32_t *accepted, int32_t *out_tokens, int32_t *n_emit, float *p_tok, float *q_tok,
                             float *resid_mass, int32_t *status, void *workspace, size_t workspace_bytes,
                             void *stream) {
  return chain_common(true, target, target_req_stride, draft_logits, draft_req_stride, row_stride, dtype, B, k, V,
                      temperature, draft, draft_len, max_emit, uniforms, accepted, out_tokens, n_emit, p_tok, q_tok,
                      resid_mass, status, workspace, workspace_bytes, stream, nullptr, top_k, top_p);
}

int spec_verify_greedy(const void *target, int64_t target_req_stride, int64_t row_stride,
                       int dtype, int B, int k, int V, const int32_t *draft,
                       const int32_t *draft_len, const int32_t *max_emit, int32_t *accepted,
                       int32_t *out_tokens, int32_t *n_emit, int32_t *status, void *workspace,
                       size_t workspace_bytes, void *stream) {
  return chain_common(false, target, target_req_stride, nullptr, 0, row_stride, dtype, B, k, V,
                      1.0f, draft, draft_len, max_emit, nullptr, accepted, out_tokens, n_emit,
                      nullptr, nullptr, nullptr, status, workspace, workspace_bytes, stream);
}

int spec_verify_sample(const void *target, int64_t target_req_stride, const void *draft_logits,
                       int64_t draft_req_stride, int64_t row_stride, int dtype, int B, int k,
                       int V, float temperature, const int32_t *draft, const int32_t *draft_len,
                       const int32_t *max_emit, const float *uniforms, int32_t *accepted,
                       int32_t *out_tokens, int32_t *n_emit, float *p_tok, float *q_tok,
                       float *resid_mass, int32_t *status, void *workspace,
                       size_t workspace_bytes, void *stream) {
  return chain_common(true, target, target_req_stride, draft_logits, draft_req_stride,
                      row_stride, dtype, B, k, V, temperature, draft, draft_len, max_emit,
                      uniforms, accepted, out_tokens, n_emit, p_tok, q_tok, resid_mass, status,
                      workspace, workspace_bytes, stream);
}

int spec_tree_rerank(const int32_t *parents, const float *conf, const int32_t *node_tok, int B, int N,
                     int m, int max_depth, int32_t *sel_nodes, int32_t *sel_parents, int32_t *sel_depth,
                     float *sel_value, int32_t *sel_tok, uint8_t *mask, int32_t *n_sel, int32_t *status,
                     void *stream) {
  if (B < 0 || N < 1 || N > SPEC_MAX_NODES || m < 1 || m > SPEC_MAX_NODES || max_depth < 0 ||
      max_depth > SPEC_MAX_DEPTH)
    return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  if (!parents || !conf || !sel_nodes || !sel_parents || !sel_depth || !n_sel || (sel_tok && !node_tok))
    return SPEC_EINVAL;
  RerankParams P{parents, conf, node_tok, B, N, m, max_depth, sel_nodes, sel_parents, sel_depth,
                 sel_value, sel_tok, mask, n_sel, status};
  const cudaError_t e = launch_tree_rerank(P, as_stream(stream));
  return e == cudaSuccess ? SPEC_OK : fail_cuda(e, "spec_tree_rerank");
}

int spec_verify_tree(const void *target, int64_t target_req_stride, const void *draft_logits,
                     int64_t draft_req_stride, int64_t row_stride, int dtype, int B, int N,
                     int V, float temperature, const int32_t *parents, const int32_t *node_tok,
                     const float *uniforms, int max_depth, int32_t *accepted_len,
                     int32_t *path_nodes, int32_t *out_tokens, int32_t *n_emit,
                     int32_t *status, void *workspace, size_t workspace_bytes, void *stream) {
  return spec_verify_tree_ex(target, target_req_stride, draft_logits, draft_req_stride, row_stride, dtype, B, N, V,
                             temperature, parents, node_tok, uniforms, max_depth, 0, accepted_len, path_nodes,
                             out_tokens, n_emit, status, workspace, workspace_bytes, stream);
}

int spec_verify_tree_ex(const void *target, int64_t target_req_stride, const void *draft_logits,
                        int64_t draft_req_stride, int64_t row_stride, int dtype, int B, int N,
                        int V, float temperature, const int32_t *parents, const int32_t *node_tok,
                        const float *uniforms, int max_depth, int flags, int32_t *accepted_len,
                        int32_t *path_nodes, int32_t *out_tokens, int32_t *n_emit,
                        int32_t *status, void *workspace, size_t workspace_bytes, void *stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (flags & ~SPEC_TREE_SIBLINGS_WITHOUT_REPLACEMENT) return SPEC_EINVAL;
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_EDTYPE;
  if (std::isnan(temperature)) return SPEC_EINVAL;
  const bool greedy = !(temperature > 0.0f);
  if (B < 0 || N < 1 || N > SPEC_MAX_NODES || V <= 0 || max_depth < 0 ||
      max_depth > SPEC_MAX_DEPTH || target_req_stride < 0 || draft_req_stride < 0 ||
      row_stride < 0 || (!greedy && !std::isfinite(temperature)))
    return SPEC_EINVAL;
  if (B == 0) return SPEC_OK;
  if (!target || !parents || !node_tok || !uniforms || !accepted_len || !path_nodes ||
      !out_tokens || !n_emit || (!greedy && !draft_logits))
    return SPEC_EINVAL;
  if (B > 2147483647 / 16) return SPEC_EINVAL;
  const int es = elem_size(dtype);
  const bool vec = aligned16(target) && (greedy || aligned16(draft_logits)) &&
                   (target_req_stride * es) % 16 == 0 && (draft_req_stride * es) % 16 == 0 &&
                   (row_stride * es) % 16 == 0;
  TreeParams P{};
  P.target = static_cast<const char *>(target);
  P.draftl = static_cast<const char *>(draft_logits);
  P.t_req = target_req_stride;
  P.d_req = draft_req_stride;
  P.row = row_stride;
  P.dtype = dtype;
  P.B = B;
  P.N = N;
  P.V = V;
  P.max_depth = max_depth;
  tree_geometry(B, V, P.cluster, P.slice);
  const int epg = 16 / elem_size(dtype);
  P.groups = ((P.slice + epg - 1) / epg + kTreeThreads - 1) / kTreeThreads;
  P.stage = 1;
  if (tree_dynamic_smem(P) > 200 * 1024) P.stage = 0;  // very large V: re-read the slice instead
  P.c = greedy ? 1.0f : static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  P.greedy = greedy ? 1 : 0;
  P.wor = !greedy && (flags & SPEC_TREE_SIBLINGS_WITHOUT_REPLACEMENT) ? 1 : 0;
  P.parents = parents;
  P.node_tok = node_tok;
  P.uniforms = uniforms;
  P.accepted_len = accepted_len;
  P.path_nodes = path_nodes;
  P.out_tokens = out_tokens;
  P.n_emit = n_emit;
  P.status = status;
  // the cluster kernels' 16-byte path also wants V a multiple of a group
  const cudaError_t e = launch_tree(P, vec && V % (16 / es) == 0, as_stream(stream));
  return e == cudaSuccess ? SPEC_OK : fail_cuda(e, "spec_verify_tree_ex");
}

}  // extern "C"
