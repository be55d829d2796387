// Allocation-free variant of the head + unmask call.
//
// Some callers cannot allocate device memory at all: a plug-in that runs
// inside a host application which owns every byte of the GPU (a serving
// process with a fixed memory budget or its own pool), or a
// latency-critical loop that cannot afford the synchronisation an allocation
// may imply. For them this file keeps the scratch memory of
// clover_lmhead_unmask in a fixed, file-scope device array that exists for as
// long as the library is loaded, so the call needs no workspace argument and
// allocates nothing.
#include <cuda_runtime.h>
#include <stdio.h>

#include "../../include/clover.h"
#include "internal.h"

namespace {

// 1 MiB: enough for up to 102 positions at hidden 2,048 (157 at hidden 256).
constexpr size_t kStaticScratchBytes = 1u << 20;

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_head_scratch[kStaticScratchBytes];

// Device address of the array in the current context. In host code the name
// g_head_scratch is only a host-side stand-in, so the address is looked up,
// with the device current, on every call: the lookup is a host-side table
// read once the module is loaded, and a cached address would go stale when
// the caller switches to another context (its own driver-API context, or a
// new primary context after cudaDeviceReset).
int scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_head_scratch);
  if (e != cudaSuccess || p == nullptr) {
    char msg[200];
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(static head scratch): %s", cudaGetErrorString(e));
    return clover::set_last_error(CLOVER_ERR_CUDA, msg);
  }
  *out = p;
  return CLOVER_OK;
}

}  // namespace

extern "C" int clover_lmhead_unmask_static(const clover_dims* dims, const uint16_t* head_w, const float* x,
                                           const float* logit_scale, float threshold, int32_t block,
                                           int32_t* tokens, uint8_t* masked, int32_t* argmax, float* max_logit,
                                           float* lse, float* max_prob, int32_t* n_committed, int32_t M,
                                           clover_stream_t stream) {
  int rc = clover::lmhead_unmask_check(dims, head_w, x, threshold, block, tokens, masked, M);
  if (rc != CLOVER_OK) return rc;
  const size_t need = clover_head_workspace_bytes(dims, M);
  if (need > kStaticScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "static scratch holds %zu bytes but hidden=%d with %d positions needs %zu; use clover_lmhead_unmask "
             "with a workspace",
             kStaticScratchBytes, dims->hidden, M, need);
    return clover::set_last_error(CLOVER_ERR_WORKSPACE_TOO_SMALL, msg);
  }
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != CLOVER_OK) return rc;
  // The array keeps whatever the previous call left; the shared routine
  // checks every argument first and only then zeroes the control words on
  // the stream, so a rejected call enqueues nothing.
  return clover::lmhead_unmask_impl(dims, head_w, x, logit_scale, threshold, block, tokens, masked, argmax, max_logit,
                                    lse, max_prob, n_committed, M, scratch, kStaticScratchBytes, stream,
                                    /*clear_ctrl=*/true);
}

extern "C" int clover_lmhead_unmask_static_status(clover_stream_t stream) {
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != CLOVER_OK) return rc;
  return clover::workspace_status_impl(scratch, kStaticScratchBytes, stream);
}
