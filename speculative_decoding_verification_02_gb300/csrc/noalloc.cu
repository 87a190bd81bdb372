// spec_verify_sample_noalloc: sampling verification for callers that cannot
// allocate device memory.
//
// Some callers cannot hand over a workspace.  A serving loop may carve its
// whole device-memory budget up at start-up and forbid allocations while it
// serves; other code runs where a cudaMalloc would stall it, because an
// allocation can synchronise the device.  For them this entry point keeps
// its scratch in a fixed array compiled into the library instead.
//
// The array lives in device memory as a file-scope __device__ variable, so
// every GPU that loads the library holds SPEC_NOALLOC_SCRATCH_BYTES of it
// until the process exits.  In host code its name only stands in for the
// symbol; the device address is looked up with cudaGetSymbolAddress, once
// per device, with that device current, on the first call made there.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace sv {
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on
// the first call per device).  Returns a CUDA error code.
cudaError_t scratch_on_current_device(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace sv

extern "C" int spec_verify_sample_noalloc(
    const void *target, int64_t target_req_stride, const void *draft_logits, int64_t draft_req_stride,
    int64_t row_stride, int dtype, int B, int k, int V, float temperature, const int32_t *draft,
    const int32_t *draft_len, const int32_t *max_emit, const float *uniforms, int32_t *accepted,
    int32_t *out_tokens, int32_t *n_emit, float *p_tok, float *q_tok, float *resid_mass,
    int32_t *status, void *stream) {
  // the scratch this call would need; anything beyond the fixed array is refused
  const size_t need = spec_workspace_size(SPEC_OP_SAMPLE, B, k, V, dtype);
  if (need > SPEC_NOALLOC_SCRATCH_BYTES) {
    char msg[200];
    std::snprintf(msg, sizeof msg,
                  "spec_verify_sample_noalloc: this call needs %zu bytes of scratch, the fixed array holds "
                  "%zu; use spec_verify_sample with a workspace",
                  need, static_cast<size_t>(SPEC_NOALLOC_SCRATCH_BYTES));
    sv::set_last_error(msg);
    return SPEC_EWORKSPACE;
  }
  void *scratch = nullptr;
  const cudaError_t e = sv::scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    char msg[200];
    std::snprintf(msg, sizeof msg, "spec_verify_sample_noalloc: scratch lookup failed: %s (%s)",
                  cudaGetErrorName(e), cudaGetErrorString(e));
    sv::set_last_error(msg);
    return SPEC_ECUDA;
  }
  return spec_verify_sample(target, target_req_stride, draft_logits, draft_req_stride, row_stride,
                            dtype, B, k, V, temperature, draft, draft_len, max_emit, uniforms, accepted,
                            out_tokens, n_emit, p_tok, q_tok, resid_mass, status, scratch,
                            SPEC_NOALLOC_SCRATCH_BYTES, stream);
}
