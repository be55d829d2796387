// Host-side routines that one translation unit of the library offers the
// others (not part of the C ABI).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/clover.h"

namespace clover {

// Records msg as the calling thread's last error (clover_last_error) and
// returns code.
int set_last_error(int code, const char* msg);

// The host-side argument checks of clover_lmhead_unmask that do not involve
// the workspace (no CUDA call).
int lmhead_unmask_check(const clover_dims* dims, const uint16_t* head_w, const float* x, float threshold,
                        int32_t block, const int32_t* tokens, const uint8_t* masked, int32_t M);

// clover_lmhead_unmask; with clear_ctrl the workspace's control words are
// zeroed on the stream after every argument check has passed.
int lmhead_unmask_impl(const clover_dims* dims, const uint16_t* head_w, const float* x, const float* logit_scale,
                       float threshold, int32_t block, int32_t* tokens, uint8_t* masked, int32_t* argmax,
                       float* max_logit, float* lse, float* max_prob, int32_t* n_committed, int32_t M,
                       void* workspace, size_t workspace_bytes, clover_stream_t stream, bool clear_ctrl);

// clover_workspace_status on any control block (a caller workspace or the
// library's static scratch).
int workspace_status_impl(void* workspace, size_t workspace_bytes, clover_stream_t stream);

}  // namespace clover
