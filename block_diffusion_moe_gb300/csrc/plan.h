// Launch planning for the persistent MoE kernels: which kernel takes a call
// and how large its grid is. Plain C++ with no CUDA dependency, so the
// decisions can be checked on a host without a GPU for any SM count.
#pragma once

namespace clover {
namespace plan {

// Largest token count of the fused layer kernel (one 32-bit mask per
// expert) and the most router rows one of its CTAs stages.
constexpr int kFusedMaxTokens = 32;
constexpr int kFusedRouterRowsPerCta = 8;

// The fused layer kernel (routing + experts + combine in one launch) takes a
// call when the tokens fit its masks, every CTA's share of the router rows
// fits its staging slices, and there is one CTA per token for the top-k
// selection (CTA t selects token t).
inline bool moe_fused(int tokens, int experts, int grid) {
  return grid >= 1 && tokens <= kFusedMaxTokens && grid >= tokens &&
         (experts + grid - 1) / grid <= kFusedRouterRowsPerCta;
}

// Grid of a persistent kernel whose CTAs wait on one another at grid
// barriers, so all of them must be resident at once. The kernels are written
// for one CTA per SM; resident_per_sm is what the occupancy query reports for
// the kernel at its shared-memory size. Returns the grid (one CTA per SM), or
// 0 when not even one CTA fits on an SM: such a launch would leave CTAs
// waiting for SMs that a barrier holds, so it is rejected instead.
inline int persistent_grid(int sms, int resident_per_sm) {
  if (sms < 1 || resident_per_sm < 1) return 0;
  return sms;
}

}  // namespace plan
}  // namespace clover
