// tsp_attention_fwd_static: the attention half of the layer for callers that
// cannot allocate device memory.
//
// Who needs it: code that runs as a plug-in inside a host application that
// owns every device allocation (an inference server, an engine with its own
// pool), where calling cudaMalloc is not allowed or would bypass the host's
// memory accounting, and latency-critical loops that must not call cudaMalloc
// because it can synchronize the device.  Such a caller still passes its
// inputs and outputs, but cannot hand the library a workspace.
//
// This entry point takes its scratch (the projected Q, K, V and the attention
// output O) from one file-scope device array of kStaticScratchBytes bytes
// instead.  The array exists on every GPU that loads the library, for as long
// as the library stays loaded.  Every call shares it: two calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on it and corrupt each other's results.  Nothing in it needs
// to start at zero: each call writes every scratch byte it later reads.
//
// The first call on a device looks up the array's device address with
// cudaGetSymbolAddress while that device is current; make that first call
// before any stream capture begins.  No call allocates or frees memory.
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(TSP_STATIC_SCRATCH_BYTES);

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[64] = {};  // device address of g_static_scratch, per device ordinal

// Returns the device address of the scratch array on the current device
// (looked up once per device), or nullptr with *err set.
void* scratch_on_current_device(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_static_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" tsp_status tsp_attention_fwd_static(const tsp_plan* plan, int batch, const void* xz,
                                               const tsp_weights* weights, void* a_out, void* lse, void* stream) {
  if (!plan) return tsp::report_error(TSP_ERR_INVALID_ARG, "tsp_attention_fwd_static: plan is NULL");
  // an empty (or negative) batch needs no scratch: validated and answered without touching the device
  if (batch <= 0) return tsp_attention_fwd(plan, batch, xz, weights, a_out, lse, nullptr, 0, stream);
  const size_t need = tsp_workspace_bytes(plan, batch, TSP_OP_ATTENTION_FWD);
  if (need > kStaticScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "tsp_attention_fwd_static: this batch needs %zu bytes of scratch, more than the %zu-byte static "
             "array; use tsp_attention_fwd with a workspace",
             need, kStaticScratchBytes);
    return tsp::report_error(TSP_ERR_WORKSPACE, msg);
  }
  // the array's address is looked up for the current device, so the work must go to that device's stream
  const tsp_status sd = tsp::check_stream_device(stream, "tsp_attention_fwd_static");
  if (sd != TSP_OK) return sd;
  cudaError_t err = cudaSuccess;
  void* scratch = scratch_on_current_device(&err);
  if (!scratch) {
    char msg[200];
    snprintf(msg, sizeof(msg), "tsp_attention_fwd_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(err));
    return tsp::report_error(TSP_ERR_CUDA, msg);
  }
  return tsp_attention_fwd(plan, batch, xz, weights, a_out, lse, scratch, kStaticScratchBytes, stream);
}
