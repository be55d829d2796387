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

#include <mutex>

#include "../../include/clover.h"

namespace clover {
int set_last_error(int code, const char* msg);
}

namespace {

// 1 MiB: enough for up to 102 positions at hidden 2,048 (157 at hidden 256).
constexpr size_t kStaticScratchBytes = 1u << 20;
constexpr size_t kControlBytes = 256;  // control words at the start of a head workspace

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_head_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {};

// Device address of the array on the current device. In host code the name
// g_head_scratch is only a host-side stand-in, so the address has to be
// looked up once per device, with that device current.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return clover::set_last_error(CLOVER_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return clover::set_last_error(CLOVER_ERR_CUDA, "device ordinal out of range");
  std::lock_guard<std::mutex> g(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_head_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[200];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(static head scratch): %s", cudaGetErrorString(e));
      return clover::set_last_error(CLOVER_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CLOVER_OK;
}

}  // namespace

extern "C" int clover_lmhead_unmask_static(const clover_dims* dims, const uint16_t* head_w, const float* x,
                                           const float* logit_scale, float threshold, int32_t block,
                                           int32_t* tokens, uint8_t* masked, int32_t* argmax, float* max_logit,
                                           float* lse, float* max_prob, int32_t* n_committed, int32_t M,
                                           clover_stream_t stream) {
  const size_t need = clover_head_workspace_bytes(dims, M);
  if (need == 0) return dims == nullptr ? CLOVER_ERR_INVALID_ARG : CLOVER_ERR_UNSUPPORTED_SHAPE;
  if (need > kStaticScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "static scratch holds %zu bytes but hidden=%d with %d positions needs %zu; use clover_lmhead_unmask "
             "with a workspace",
             kStaticScratchBytes, dims->hidden, M, need);
    return clover::set_last_error(CLOVER_ERR_WORKSPACE_TOO_SMALL, msg);
  }
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != CLOVER_OK) return rc;
  // The array keeps whatever the previous call left; its control words must
  // start at zero.
  cudaError_t e = cudaMemsetAsync(scratch, 0, kControlBytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return clover::set_last_error(CLOVER_ERR_CUDA, cudaGetErrorString(e));
  return clover_lmhead_unmask(dims, head_w, x, logit_scale, threshold, block, tokens, masked, argmax, max_logit,
                              lse, max_prob, n_committed, M, scratch, kStaticScratchBytes, stream);
}
