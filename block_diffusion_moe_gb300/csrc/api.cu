// Host side of the C ABI declared in include/clover.h: argument checks,
// workspace layout, TMA descriptors, kernel launches and the denoise loop.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/clover.h"
#include "internal.h"
#include "kernels.cuh"
#include "plan.h"
#include "sm100.cuh"

using namespace clover;

static_assert(plan::kFusedMaxTokens == kLayerMaxTokens && plan::kFusedRouterRowsPerCta == kRouteExperts,
              "the launch plan and the fused layer kernel must agree on its limits");

namespace {

thread_local char g_err[512] = {0};

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(CLOVER_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Every kernel waits for its predecessor's results with griddepcontrol.wait,
// so all launches may use programmatic dependent launch.
constexpr bool kPdl = true;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Control block at the start of every workspace (and of each sub-workspace
// of the denoise workspace). Words that must be zero when a call starts are
// either reset by the kernels that use them or kept zero between calls.
constexpr size_t kCtrlBytes = 256;
enum CtrlWord : int {
  kCtrlErr = 0,          // kernel status bits
  kCtrlUnitCtr = 1,      // expert kernel work counter (reset by the kernel before its barrier)
  kCtrlMaskedLeft = 2,   // positions still masked after the last head call
  kCtrlHeadDone = 3,     // head kernel arrival counter (reset by its last CTA)
  kCtrlCommitted = 4,    // positions committed by the last head call
  kCtrlExitCtr = 5,      // expert kernel CTAs that finished (reset by the last one)
  kCtrlBarCount = 6,     // [u64, words 6-7] fused-layer grid barrier arrivals (only grows)
  kCtrlStamps = 40,      // [8 x u64] phase timestamps of the last fused-layer launch (diagnostics)
};

struct MoeLayout {
  size_t gu_done, dn_done, n_active, act, cnt, off, tok_slot, topk_idx, topk_w, topk_p, rr_idx, rr_w, fin_w, logits,
      xg, hbuf, yslot, tg_ctr, gathered, bytes;
};

// Most units tables a call can need: the standalone expert kernel cuts each
// expert's rows (and the shared expert's) into chunks of at most
// kExpertTileTokens, so there are at most E + ceil(M K / kExpertTileTokens)
// routed chunks and ceil(M / kExpertTileTokens) shared ones.
size_t max_chunks(const clover_dims& d, int M) {
  const size_t MK = static_cast<size_t>(M) * d.top_k;
  return d.n_experts + (MK + kExpertTileTokens - 1) / kExpertTileTokens +
         (M + kExpertTileTokens - 1) / kExpertTileTokens + 1;
}

MoeLayout moe_layout(const clover_dims& d, int M) {
  MoeLayout L;
  size_t o = 0;
  auto take = [&](size_t b) {
    const size_t r = o;
    o = align_up(o + b, 256);
    return r;
  };
  const size_t H = d.hidden, F = d.d_ff, E = d.n_experts, K = d.top_k;
  const size_t R = static_cast<size_t>(M) * K + M;
  const size_t NC = max_chunks(d, M);
  L.gu_done = take(NC * 4);
  L.dn_done = take((H / 128) * 4);
  L.n_active = take(4);
  L.act = take(NC * 4);
  L.cnt = take(std::max(NC, E) * 4);
  L.off = take(std::max(NC, E) * 4);
  L.tok_slot = take(M * K * 4);
  L.topk_idx = take(M * K * 4);
  L.topk_w = take(M * K * 4);
  L.topk_p = take(M * K * 4);
  L.rr_idx = take(M * K * 4);
  L.rr_w = take(M * K * 4);
  L.fin_w = take(M * K * 4);
  L.logits = take(static_cast<size_t>(M) * E * 4);
  L.xg = take(R * H * 2);
  L.hbuf = take(R * F * 2);
  L.yslot = take(R * H * 4);
  L.tg_ctr = take(((M + kRouteTileTokens - 1) / kRouteTileTokens) * 4);  // routing arrival counters (kept zero)
  L.gathered = take(NC * 4);  // rows gathered per chunk (reset by the last CTA of each launch)
  L.bytes = o;
  return L;
}

struct HeadLayout {
  size_t xn, part_m, part_s, part_a, part_t, part_zd, dec_m, dec_s, dec_a, bytes;
};

// The accept form adds two more [G][M] partial arrays.
HeadLayout head_layout(const clover_dims& d, int M, bool accept = false) {
  HeadLayout L;
  size_t o = 0;
  auto take = [&](size_t b) {
    const size_t r = o;
    o = align_up(o + b, 256);
    return r;
  };
  const size_t ms = static_cast<size_t>(std::min(M, kTileTokens));  // positions of one head sub-call
  L.xn = take(static_cast<size_t>(M) * d.hidden * 2);
  L.part_m = take(static_cast<size_t>(kHeadMaxCtas) * ms * 4);
  L.part_s = take(static_cast<size_t>(kHeadMaxCtas) * ms * 4);
  L.part_a = take(static_cast<size_t>(kHeadMaxCtas) * ms * 4);
  L.part_t = accept ? take(static_cast<size_t>(kHeadMaxCtas) * ms * 4) : 0;
  L.part_zd = accept ? take(static_cast<size_t>(kHeadMaxCtas) * ms * 4) : 0;
  L.dec_m = take(ms * 4);
  L.dec_s = accept ? take(ms * 4) : 0;
  L.dec_a = take(ms * 4);
  L.bytes = o;
  return L;
}

// Denoise workspace: [ctrl | moe ctrl | head ctrl | x | moe data | head data]
struct DenoiseLayout {
  size_t moe_ctrl, head_ctrl, x, moe, head, bytes;
};

DenoiseLayout denoise_layout(const clover_dims& d, int M) {
  DenoiseLayout L;
  L.moe_ctrl = kCtrlBytes;
  L.head_ctrl = 2 * kCtrlBytes;
  L.x = 3 * kCtrlBytes;
  L.moe = align_up(L.x + static_cast<size_t>(M) * d.hidden * 4, 256);
  L.head = align_up(L.moe + moe_layout(d, M).bytes, 256);
  L.bytes = align_up(L.head + head_layout(d, M).bytes, 256);
  return L;
}

int check_dims(const clover_dims* d) {
  if (d == nullptr) return fail(CLOVER_ERR_INVALID_ARG, "dims is NULL");
  if (d->hidden <= 0 || d->n_experts <= 0 || d->top_k <= 0 || d->d_ff <= 0 || d->vocab <= 0)
    return fail(CLOVER_ERR_INVALID_ARG, "dims must be positive");
  if (!(d->rms_eps >= 0.f) || d->rms_eps > 1.f) return fail(CLOVER_ERR_INVALID_ARG, "rms_eps out of range");
  if (d->hidden % 128 != 0 || d->hidden > 8192)
    return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "hidden=%d: must be a multiple of 128, at most 8192", d->hidden);
  if (d->d_ff % 64 != 0 || d->d_ff > 16384)
    return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "d_ff=%d: must be a multiple of 64, at most 16384", d->d_ff);
  if (d->n_experts > kMaxExperts) return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "n_experts=%d > %d", d->n_experts, kMaxExperts);
  if (d->top_k > kMaxTopK || d->top_k > d->n_experts)
    return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "top_k=%d: must be <= 32 and <= n_experts", d->top_k);
  if (d->vocab < 2) return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "vocab=%d < 2", d->vocab);
  if (d->mask_id < 0 || d->mask_id >= d->vocab)
    return fail(CLOVER_ERR_INVALID_ARG, "mask_id=%d outside [0, vocab)", d->mask_id);
  if (!(d->coreset_top_p >= 0.f && d->coreset_top_p <= 1.f))
    return fail(CLOVER_ERR_INVALID_ARG, "coreset_top_p=%g outside [0, 1]", d->coreset_top_p);
  return CLOVER_OK;
}

int check_tokens(int M) {
  if (M < 1 || M > kMaxTokens) return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "tokens=%d outside [1, %d]", M, kMaxTokens);
  return CLOVER_OK;
}

bool layer_is_q4(const clover_moe_layer& l) { return l.gate_up_q != nullptr; }

int check_layer(const clover_moe_layer* l, int i) {
  if (l == nullptr) return fail(CLOVER_ERR_INVALID_ARG, "layer %d is NULL", i);
  const void* bf[] = {l->router_w, l->gate_up, l->down, l->sh_gate_up, l->sh_down};
  const void* q4[] = {l->router_w, l->gate_up_q, l->gate_up_s, l->down_q, l->down_s, l->sh_gate_up_q,
                      l->sh_gate_up_s, l->sh_down_q, l->sh_down_s};
  const bool low = layer_is_q4(*l);
  const int n = low ? 9 : 5;
  for (int k = 0; k < n; ++k) {
    const void* p = low ? q4[k] : bf[k];
    if (p == nullptr) return fail(CLOVER_ERR_INVALID_ARG, "layer %d: NULL weight pointer", i);
    if (!aligned16(p)) return fail(CLOVER_ERR_INVALID_ARG, "layer %d: weight pointer not 16-byte aligned", i);
  }
  return CLOVER_OK;
}

// ------------------------------------------------------------ device info

struct DevInfo {
  int sms = 0;
};

int device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(CLOVER_ERR_CUDA, "device ordinal %d unsupported", dev);
  std::lock_guard<std::mutex> g(mu);
  if (cache[dev].sms == 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    cache[dev].sms = sms;
  }
  *out = cache[dev];
  return CLOVER_OK;
}

// ------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  static cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSuccess;
  std::call_once(once, [] {
    void* fn = nullptr;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) {
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
    return fail(CLOVER_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  }
  return CLOVER_OK;
}

// bf16 matrix [rows][cols], row-major; box = 64 columns x box_rows rows with
// 128-byte swizzle (the layout the UMMA descriptors expect).
int encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, const char* what) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CLOVER_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, static_cast<int>(r));
  return CLOVER_OK;
}

// A rank-n strided view (dims[0] innermost, contiguous; strides in bytes of
// dims 1..n-1).
int encode_nd(CUtensorMap* m, CUtensorMapDataType type, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle, const char* what) {
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, type, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CLOVER_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, static_cast<int>(r));
  return CLOVER_OK;
}

// The same for bf16 with 128-byte swizzle (the layout the UMMA descriptors expect).
int encode_bf16_nd(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box, const char* what) {
  return encode_nd(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                   what);
}

// The whole-stage views of one expert stack (n experts; see ExpertArgs):
// gate/up [n][2F][H], down [n][H][F]. A view is encoded only for the shapes
// whose units use it (two-group stages need an even number of K groups).
int encode_stage_maps(CUtensorMap* gu_k2, CUtensorMap* dn_k2, const void* gate_up, const void* down, uint64_t n,
                      uint64_t H, uint64_t F) {
  int rc;
  if ((H / 64) % 2 == 0) {  // (64 c, rows, gate|up, K group): gate row r, its up row r + F
    const cuuint64_t dims[4] = {64, n * 2 * F - F, 2, H / 64};
    const cuuint64_t str[3] = {H * 2, F * H * 2, 128};
    const cuuint32_t box[4] = {64, 64, 2, 2};
    if ((rc = encode_bf16_nd(gu_k2, gate_up, 4, dims, str, box, "gate_up stage view"))) return rc;
  }
  if ((F / 64) % 2 == 0) {  // (64 c, rows, K group)
    const cuuint64_t dims[3] = {64, n * H, F / 64};
    const cuuint64_t str[2] = {F * 2, 128};
    const cuuint32_t box[3] = {64, 128, 2};
    if ((rc = encode_bf16_nd(dn_k2, down, 3, dims, str, box, "down stage view"))) return rc;
  }
  return CLOVER_OK;
}

// 4-bit codes as bytes: rows of `cols_bytes`, boxes of box_cols bytes x
// box_rows (the converter warps read them).
int encode_u8_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols_bytes, uint32_t box_cols,
                 uint32_t box_rows, const char* what) {
  cuuint64_t dims[2] = {cols_bytes, rows};
  cuuint64_t strides[1] = {cols_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  // 128-byte rows take the 128-byte swizzle (16-byte chunk c of row r at
  // chunk c ^ (r % 8)), so the converter's row reads do not share banks
  const CUtensorMapSwizzle sw = box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CLOVER_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, static_cast<int>(r));
  return CLOVER_OK;
}

// ------------------------------------------------------------- profiling

struct ProfileHook {
  cudaEvent_t* begin = nullptr;
  cudaEvent_t* end = nullptr;
  int cap = 0;
  int count = 0;
} g_prof;

// ------------------------------------------------------------- launches

struct Plan {
  int sms;
};

int record(cudaEvent_t ev, cudaStream_t s) {
  cudaError_t e = cudaEventRecord(ev, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  return CLOVER_OK;
}

// Occupancy of an expert kernel at a shared-memory size, cached per
// (device, kernel, size): the query runs once per configuration.
int resident_per_sm(bool fused, bool q4, size_t smem, int* out) {
  struct Entry {
    int dev, kind;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int n_cached = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const int kind = (fused ? 2 : 0) + (q4 ? 1 : 0);
  std::lock_guard<std::mutex> g(mu);
  for (int i = 0; i < n_cached; ++i)
    if (cache[i].dev == dev && cache[i].kind == kind && cache[i].smem == smem) {
      *out = cache[i].n;
      return CLOVER_OK;
    }
  int n = 0;
  e = expert_resident_per_sm(fused, q4, smem, &n);
  if (e != cudaSuccess) return cuda_fail(e, "occupancy of the expert kernel");
  if (n_cached < 64) cache[n_cached++] = Entry{dev, kind, smem, n};
  *out = n;
  return CLOVER_OK;
}

// Route + permutation + experts for one layer. ctrl: this call's MoE control
// block; err: status word to flag. A chain of fused layers working in place
// on one x may defer each layer's combine: `defer` leaves it to the next
// launch on the same workspace (which takes `pend`) or to enqueue_combine.
int enqueue_moe_layer(const clover_dims& d, const clover_moe_layer& layer, const float* x_in, float* x_out,
                      int32_t* out_idx, float* out_w, int M, uint8_t* data, int* ctrl, int* err, const Plan& plan,
                      cudaStream_t stream, const void* next_router = nullptr, bool defer = false, bool pend = false,
                      bool xn_ready = false, bool norm_next = false, const clover_moe_layer* next_layer = nullptr) {
  const MoeLayout L = moe_layout(d, M);
  const int H = d.hidden, F = d.d_ff, E = d.n_experts, K = d.top_k;
  const int MK = M * K;
  bf16* xg = reinterpret_cast<bf16*>(data + L.xg);
  bf16* hbuf = reinterpret_cast<bf16*>(data + L.hbuf);
  int32_t* topk_idx = reinterpret_cast<int32_t*>(data + L.topk_idx);
  float* topk_w = reinterpret_cast<float*>(data + L.topk_w);

  const bool fused = plan::moe_fused(M, E, plan.sms);
  const int n_chunks = static_cast<int>(max_chunks(d, M));
  if ((defer || pend) && (!fused || x_in != x_out))
    return fail(CLOVER_ERR_INVALID_ARG, "a deferred combine needs the fused layer kernel working in place");
  if (d.coreset_top_p > 0.f && !fused)
    return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "the block coreset needs at most %d positions", kLayerMaxTokens);
  cudaError_t e = cudaSuccess;
  if (!fused) {
    RouteArgs ra;
    ra.x = x_in;
    ra.wr = reinterpret_cast<const bf16*>(layer.router_w);
    ra.bias = layer.router_bias;
    ra.logits = reinterpret_cast<float*>(data + L.logits);
    ra.xn_rows = xg + static_cast<size_t>(MK) * H;
    ra.tg_ctr = reinterpret_cast<int*>(data + L.tg_ctr);
    ra.err = ctrl + kCtrlErr;
    ra.topk_idx = topk_idx;
    ra.topk_w = topk_w;
    ra.M = M;
    ra.H = H;
    ra.E = E;
    ra.K = K;
    ra.eps = d.rms_eps;
    ra.xn_ready = xn_ready ? 1 : 0;
    e = launch_route(ra, stream, kPdl);
    if (e != cudaSuccess) return cuda_fail(e, "launch route");

  }

  ExpertArgs xa;
  memset(&xa, 0, sizeof(xa));
  xa.acc_cols = 256;
  const int R = MK + M;
  int rc;
  const bool q4 = layer_is_q4(layer);
  if (q4) {
    // K groups per staging slot: the largest of 4, 2, 1 dividing the groups
    auto slot_groups = [](int groups) { return groups % 4 == 0 ? 4 : (groups % 2 == 0 ? 2 : 1); };
    xa.kq_gu = slot_groups(H / 64);
    xa.kq_dn = slot_groups(F / 64);
    if ((rc = encode_u8_2d(&xa.tm_gu_q, layer.gate_up_q, static_cast<uint64_t>(E) * 2 * F, H / 2, xa.kq_gu * 32, 64,
                           "gate_up codes")))
      return rc;
    if ((rc = encode_u8_2d(&xa.tm_sgu_q, layer.sh_gate_up_q, 2ull * F, H / 2, xa.kq_gu * 32, 64,
                           "shared gate_up codes")))
      return rc;
    if ((rc = encode_u8_2d(&xa.tm_dn_q, layer.down_q, static_cast<uint64_t>(E) * H, F / 2, xa.kq_dn * 32, 128,
                           "down codes")))
      return rc;
    if ((rc = encode_u8_2d(&xa.tm_sdn_q, layer.sh_down_q, H, F / 2, xa.kq_dn * 32, 128, "shared down codes")))
      return rc;
    for (int sh = 0; sh < 2; ++sh) {  // the whole-slot views, routed then shared
      const uint64_t n = sh ? 1 : E;
      {  // codes: (H/2 bytes, gate rows, gate|up)
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(H / 2), n * 2 * F - F, 2};
        const cuuint64_t str[2] = {static_cast<cuuint64_t>(H / 2), static_cast<cuuint64_t>(F) * (H / 2)};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(xa.kq_gu * 32), 64, 2};
        if ((rc = encode_nd(sh ? &xa.tm_sgu_q3 : &xa.tm_gu_q3, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                            sh ? layer.sh_gate_up_q : layer.gate_up_q, 3, dims, str, box,
                            xa.kq_gu * 32 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                            "gate_up code view")))
          return rc;
      }
      {  // gate/up scales [n][H/64][2F]: (gate scale, gate|up, K group)
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(F), 2, n * (H / 64)};
        const cuuint64_t str[2] = {static_cast<cuuint64_t>(F) * 2, static_cast<cuuint64_t>(F) * 4};
        const cuuint32_t box[3] = {64, 2, static_cast<cuuint32_t>(xa.kq_gu)};
        if ((rc = encode_nd(sh ? &xa.tm_sgu_sv : &xa.tm_gu_sv, CU_TENSOR_MAP_DATA_TYPE_UINT16,
                            sh ? layer.sh_gate_up_s : layer.gate_up_s, 3, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                            "gate_up scale view")))
          return rc;
      }
      {  // down scales [n][F/64][H]: (scale, K group)
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), n * (F / 64)};
        const cuuint64_t str[1] = {static_cast<cuuint64_t>(H) * 2};
        const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(xa.kq_dn)};
        if ((rc = encode_nd(sh ? &xa.tm_sdn_sv : &xa.tm_dn_sv, CU_TENSOR_MAP_DATA_TYPE_UINT16,
                            sh ? layer.sh_down_s : layer.down_s, 2, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                            "down scale view")))
          return rc;
      }
    }
    xa.q4_views = 1;
    xa.gu_s = layer.gate_up_s;
    xa.sgu_s = layer.sh_gate_up_s;
    xa.dn_s = layer.down_s;
    xa.sdn_s = layer.sh_down_s;
    xa.q4 = 1;
  } else {
    if ((rc = encode_bf16_2d(&xa.tm_gu, layer.gate_up, static_cast<uint64_t>(E) * 2 * F, H, 64, "gate_up"))) return rc;
    if ((rc = encode_bf16_2d(&xa.tm_sgu, layer.sh_gate_up, 2ull * F, H, 64, "shared gate_up"))) return rc;
    if ((rc = encode_bf16_2d(&xa.tm_dn, layer.down, static_cast<uint64_t>(E) * H, F, 128, "down"))) return rc;
    if ((rc = encode_bf16_2d(&xa.tm_sdn, layer.sh_down, H, F, 128, "shared down"))) return rc;
    if ((rc = encode_stage_maps(&xa.tm_gu_k2, &xa.tm_dn_k2, layer.gate_up, layer.down, E, H, F))) return rc;
    if ((rc = encode_stage_maps(&xa.tm_sgu_k2, &xa.tm_sdn_k2, layer.sh_gate_up, layer.sh_down, 1, H, F))) return rc;
    xa.stage_maps = 1;
  }
  // B tiles move in boxes of up to 64 rows (one TMA instruction each), with
  // 16-row boxes for the rest; fewer, larger copies stream faster.
  const int nb_rows = std::min((M + 15) & ~15, kExpertTileTokens);
  if (fused) {  // the gate/up B operand is the dense block of normed rows
    const bf16* xn_rows = xg + static_cast<size_t>(MK) * H;
    if ((rc = encode_bf16_2d(&xa.tm_xg, xn_rows, M, H, 16, "normed rows"))) return rc;
    if ((rc = encode_bf16_2d(&xa.tm_xg_big, xn_rows, M, H, nb_rows, "normed rows"))) return rc;
    xa.xg_box = nb_rows;
  } else {
    if ((rc = encode_bf16_2d(&xa.tm_xg, xg, R, H, 16, "gathered inputs"))) return rc;
    if ((rc = encode_bf16_2d(&xa.tm_xg_big, xg, R, H, 64, "gathered inputs"))) return rc;
    xa.xg_box = 64;
  }
  if ((rc = encode_bf16_2d(&xa.tm_h, hbuf, R, F, 16, "swiglu outputs"))) return rc;
  if ((rc = encode_bf16_2d(&xa.tm_h_big, hbuf, R, F, 64, "swiglu outputs"))) return rc;
  xa.h_box = 64;
  xa.x_in = x_in;
  xa.x_out = x_out;
  xa.hbuf = hbuf;
  xa.yslot = reinterpret_cast<float*>(data + L.yslot);
  xa.n_active = reinterpret_cast<int*>(data + L.n_active);
  xa.act = reinterpret_cast<int*>(data + L.act);
  xa.cnt = reinterpret_cast<int*>(data + L.cnt);
  xa.off = reinterpret_cast<int*>(data + L.off);
  xa.tok_slot = reinterpret_cast<int32_t*>(data + L.tok_slot);
  xa.topk_w = topk_w;
  xa.topk_idx = topk_idx;
  xa.xg = xg;
  xa.xn = xg + static_cast<size_t>(MK) * H;  // the normed rows (also the shared expert's rows)
  xa.bar_count = reinterpret_cast<unsigned long long*>(ctrl + kCtrlBarCount);
  xa.out_idx = out_idx;
  xa.out_w = out_w;
  xa.unit_ctr = ctrl + kCtrlUnitCtr;
  xa.gu_done = reinterpret_cast<int*>(data + L.gu_done);
  xa.dn_done = reinterpret_cast<int*>(data + L.dn_done);
  xa.gathered = reinterpret_cast<int*>(data + L.gathered);
  xa.exit_ctr = ctrl + kCtrlExitCtr;
  xa.max_chunks = n_chunks;
  xa.err = err;
  xa.M = M;
  xa.H = H;
  xa.F = F;
  xa.E = E;
  xa.K = K;
  const int nb = std::min((M + 15) & ~15, kExpertTileTokens);  // B-tile rows: one chunk at most
  // Two K groups per A/B stage (8 MMAs per pipeline step instead of 4) up to
  // 128 token columns: every pipeline step (waits, MMAs, commits) has a fixed
  // cost of ~0.4 µs, so fewer, larger steps stream faster. The low-bit path,
  // whose A stages are written by the converter warps rather than streamed,
  // takes four (a whole staging slot, 16 MMAs per commit).
  const bool g4 = q4 && nb <= 64 && (H / 64) % 4 == 0 && (F / 64) % 4 == 0 && xa.kq_gu == 4 && xa.kq_dn == 4;
  const int kg2_cols = q4 ? 64 : 128;  // the low-bit path also needs room for its staging ring
  const int kg_gu = g4 ? 4 : ((nb <= kg2_cols && (H / 64) % 2 == 0) ? 2 : 1);
  const int kg_dn = g4 ? 4 : ((nb <= kg2_cols && (F / 64) % 2 == 0) ? 2 : 1);
  const int kg = std::max(kg_gu, kg_dn);
  xa.kg_gu = kg_gu;
  xa.kg_dn = kg_dn;
  xa.kg_stage = kg;
  if (fused && kg_gu > 1) {
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(H / 64)};
    const cuuint64_t str[2] = {static_cast<cuuint64_t>(H) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(nb_rows), static_cast<cuuint32_t>(kg_gu)};
    if ((rc = encode_bf16_nd(&xa.tm_xg_k, xg + static_cast<size_t>(MK) * H, 3, dims, str, box,
                             "normed rows stage view")))
      return rc;
    xa.xg_k = 1;
  }
  // Every chunk of the standalone kernel runs as paired units: two weight slices
  // share each B tile (an A stage of two K groups holds one K group of two
  // slices; two 128-column accumulators), halving the token rows each SM
  // takes in per weight byte. (Pairing only experts above 16, 32 or 64
  // tokens was slower on the same box: 3.68, 3.69, 3.71 against 3.64 ms per
  // Zipf step; none: 3.79.)
  xa.pair_rows = (!fused && !q4 && kg_gu == 2 && kg_dn == 2 &&
                  (F / 64) % 2 == 0 && (H / 128) % 2 == 0)
                     ? 0
                     : -1;
  const size_t a_stage = static_cast<size_t>(kg) * kATileBytes;
  const size_t b_stage = static_cast<size_t>(kg) * nb * 128;
  const size_t tables = fused ? layer_rt_bytes(M, K, E) : expert_tables_bytes(M, K, n_chunks);
  const size_t fixed = expert_smem_bytes(0, 0, 0, nb, 0, kg) + static_cast<size_t>(4 * 16) * 8 + tables;
  const size_t budget = static_cast<size_t>(kSmemBudget) - fixed;
  int sa, sb, sq = 0;
  if (q4) {
    // The staging ring carries the HBM stream (4 KiB of codes per K group,
    // 4x the weights per byte); the bf16 stages hold two slots' worth (one
    // per converter team).
    sa = kg == 4 ? 2 : 4;
    sb = kg == 4 ? 2 : 3;
    const size_t used = static_cast<size_t>(sa) * a_stage + static_cast<size_t>(sb) * b_stage;
    sq = used < budget ? static_cast<int>(std::min<size_t>(24, (budget - used) / (kQSlotBytes + 16))) : 0;
    if (sq < 1) return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "no shared memory left for the low-bit staging ring");
    // Two converter teams take slots in turn when each can own its slots
    // (an even slot count) and its bf16 stages (a multiple of twice the
    // stages one slot fills, the same for both unit kinds).
    const int per_slot_gu = xa.kq_gu / kg_gu, per_slot_dn = xa.kq_dn / kg_dn;
    xa.q_teams = 1;
    if (fused && kg == 4) {
      // A tiles in tensor memory (two 64-column accumulators, then the two
      // 128-column A stages); the staging slots take the A ring, which the
      // routing prelude uses before any slot is loaded.
      xa.a_tmem = 1;
      xa.q_in_a = 1;
      xa.acc_cols = 64;
      sq = static_cast<int>(std::min<size_t>(24, static_cast<size_t>(sa) * a_stage / kQSlotBytes));
    }
    if (per_slot_gu == per_slot_dn && sa % (2 * per_slot_gu) == 0 && sq >= 2) {
      sq &= ~1;
      xa.q_teams = 2;
    }
  } else if (nb <= 64) {
    sa = sb = static_cast<int>(std::min<size_t>(16, budget / (a_stage + b_stage)));
  } else if (kg == 2) {
    // wide B stages (bf16, 65-128 columns): two of them; the weight ring takes the rest
    sb = 2;
    const size_t used = static_cast<size_t>(sb) * b_stage;
    sa = used < budget ? static_cast<int>(std::min<size_t>(16, (budget - used) / a_stage)) : 0;
  } else {
    sb = 3;
    const size_t used = static_cast<size_t>(sb) * b_stage;
    sa = used < budget ? static_cast<int>(std::min<size_t>(16, (budget - used) / a_stage)) : 0;
  }
  if (sa < 1 || sb < 1) return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "expert pipeline does not fit in shared memory");
  // The standalone kernel builds its permutation in the weight ring.
  if (!fused && static_cast<size_t>(sa) * a_stage < perm_smem_bytes(M, K, E))
    return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "the permutation tables do not fit in the expert kernel's weight ring");
  const int smem_a = sa;
  xa.smem_a = smem_a;
  xa.stages_a = sa;
  xa.stages_b = sb;
  xa.stages_q = sq;
  xa.nb_max = nb;
  // Up to 32 tokens the down unit that completes a hidden slice combines it
  // (a few µs); with more tokens that serial walk would dominate, so a
  // parallel kernel does it.
  xa.combine = fused ? (defer ? 2 : 1) : 0;
  // the next layer's shared expert, prefetched into L2 by CTAs that have run out of units
  xa.sgu_next = (next_layer && !q4) ? reinterpret_cast<const bf16*>(next_layer->sh_gate_up) : nullptr;
  xa.sdn_next = (next_layer && !q4) ? reinterpret_cast<const bf16*>(next_layer->sh_down) : nullptr;
  xa.pend = pend ? 1 : 0;
  xa.fin_w = reinterpret_cast<float*>(data + L.fin_w);
  // (slots inside the A ring add only their barriers)
  size_t smem = xa.q_in_a ? expert_smem_bytes(smem_a, sa, sb, nb, 0, kg) + static_cast<size_t>(2 * sq) * 8
                          : expert_smem_bytes(smem_a, sa, sb, nb, sq, kg);
  if (fused) {
    xa.wr = reinterpret_cast<const bf16*>(layer.router_w);
    xa.wr_next = reinterpret_cast<const bf16*>(next_router);
    xa.bias = layer.router_bias;
    xa.logits = reinterpret_cast<float*>(data + L.logits);

    xa.pub_idx = topk_idx;
    xa.pub_w = topk_w;
    xa.pub_p = reinterpret_cast<float*>(data + L.topk_p);
    xa.pub2_idx = reinterpret_cast<int32_t*>(data + L.rr_idx);
    xa.pub2_w = reinterpret_cast<float*>(data + L.rr_w);
    xa.coreset_top_p = d.coreset_top_p;
    xa.eps = d.rms_eps;
#if CLOVER_PHASE_STAMPS
    xa.stamps = reinterpret_cast<unsigned long long*>(ctrl + kCtrlStamps);
#else
    xa.stamps = nullptr;
#endif
  }
  smem += tables;
  // Every CTA of the persistent kernel waits on other CTAs (grid barriers,
  // the chunk and unit counters), so the whole grid must be resident at
  // once: check it before launching.
  int resident = 0;
  if ((rc = resident_per_sm(fused, q4, smem, &resident))) return rc;
  const int grid = plan::persistent_grid(plan.sms, resident);
  if (grid == 0)
    return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "the %s expert kernel cannot be resident on an SM (%zu bytes of shared "
                "memory, occupancy %d)", fused ? "fused" : "standalone", smem, resident);
  if (g_prof.begin && g_prof.cap > 0) {
    if ((rc = record(g_prof.begin[g_prof.count % g_prof.cap], stream))) return rc;
  }
  e = fused ? launch_layer(xa, grid, smem, stream, kPdl) : launch_expert(xa, grid, smem, stream, kPdl);
  if (e != cudaSuccess) return cuda_fail(e, fused ? "launch layer" : "launch expert");
  if (!xa.combine) {
    CombineArgs ca;
    memset(&ca, 0, sizeof(ca));
    ca.x_in = x_in;
    ca.x_out = x_out;
    ca.yslot = xa.yslot;
    ca.tok_slot = xa.tok_slot;
    ca.topk_w = xa.topk_w;
    ca.M = M;
    ca.H = H;
    ca.K = K;
    ca.xn_out = norm_next ? xg + static_cast<size_t>(MK) * H : nullptr;
    ca.eps = d.rms_eps;
    e = norm_next ? launch_combine_norm(ca, stream, kPdl) : launch_combine(ca, stream, kPdl);
    if (e != cudaSuccess) return cuda_fail(e, "launch combine");
  }
  if (g_prof.end && g_prof.cap > 0) {
    if ((rc = record(g_prof.end[g_prof.count % g_prof.cap], stream))) return rc;
    ++g_prof.count;
  }
  return CLOVER_OK;
}

// The combine a deferring fused layer left behind (tables in its workspace),
// in place on x.
int enqueue_combine(const clover_dims& d, float* x, int M, uint8_t* data, cudaStream_t stream) {
  const MoeLayout L = moe_layout(d, M);
  CombineArgs ca;
  memset(&ca, 0, sizeof(ca));
  ca.x_in = x;
  ca.x_out = x;
  ca.yslot = reinterpret_cast<float*>(data + L.yslot);
  ca.tok_slot = reinterpret_cast<int32_t*>(data + L.tok_slot);
  ca.topk_w = reinterpret_cast<float*>(data + L.fin_w);
  ca.M = M;
  ca.H = d.hidden;
  ca.K = d.top_k;
  const cudaError_t e = launch_combine(ca, stream, kPdl);
  if (e != cudaSuccess) return cuda_fail(e, "launch combine");
  return CLOVER_OK;
}

// The accept test's inputs and outputs (null: the unmask rule).
struct AcceptCfg {
  const int32_t* draft;
  int rule;
  float ratio, delta;
  float* entropy;
  float* p_draft;
  int32_t* accept_len;
  int32_t* out_tokens;
};

// Head statistics and the unmask rule (or the accept test) on M positions.
// The positions are normalised once; the head kernel then takes them in
// sub-calls of at most kTileTokens positions made of whole blocks (one
// accumulator's width), each streaming the head once.
int enqueue_head(const clover_dims& d, const uint16_t* head_w, const float* x, const float* alpha, float threshold,
                 int block, int32_t* tokens, uint8_t* masked, int32_t* argmax, float* max_logit, float* lse,
                 float* max_prob, int32_t* n_committed, int M, uint8_t* data, int* ctrl, int* err, const Plan& plan,
                 cudaStream_t stream, const AcceptCfg* acc = nullptr) {
  const bool accept = acc != nullptr;
  const HeadLayout L = head_layout(d, M, accept);
  const int sub = M <= kTileTokens ? M : (kTileTokens / block) * block;
  if (sub < 1)
    return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "block=%d: blocks wider than %d positions need M <= %d", block,
                kTileTokens, kTileTokens);
  bf16* xn = reinterpret_cast<bf16*>(data + L.xn);
  NormArgs na;
  na.x = x;
  na.xn = xn;
  na.M = M;
  na.H = d.hidden;
  na.eps = d.rms_eps;
  cudaError_t e = launch_rmsnorm(na, stream, kPdl);
  if (e != cudaSuccess) return cuda_fail(e, "launch rmsnorm");

  int rc;
  for (int p0 = 0; p0 < M; p0 += sub) {
    const int m = std::min(sub, M - p0);
    HeadArgs ha;
    memset(&ha, 0, sizeof(ha));
    if ((rc = encode_bf16_2d(&ha.tm_w, head_w, d.vocab, d.hidden, 128, "head"))) return rc;
    // One box carries a K group of all positions (rows past m read as zeros).
    const int nb = (m + 15) & ~15;
    if ((rc = encode_bf16_2d(&ha.tm_x, xn + static_cast<size_t>(p0) * d.hidden, m, d.hidden, static_cast<uint32_t>(nb),
                             "normed positions")))
      return rc;
    ha.x_box = nb;
    ha.alpha = alpha ? alpha + p0 : nullptr;
    ha.part_m = reinterpret_cast<float*>(data + L.part_m);
    ha.part_s = reinterpret_cast<float*>(data + L.part_s);
    ha.part_a = reinterpret_cast<int*>(data + L.part_a);
    ha.done_ctr = ctrl + kCtrlHeadDone;
    ha.tokens = tokens ? tokens + p0 : nullptr;
    ha.masked = masked ? masked + p0 : nullptr;
    ha.argmax = argmax ? argmax + p0 : nullptr;
    ha.max_logit = max_logit ? max_logit + p0 : nullptr;
    ha.lse = lse ? lse + p0 : nullptr;
    ha.max_prob = max_prob ? max_prob + p0 : nullptr;
    ha.n_committed = n_committed ? n_committed : ctrl + kCtrlCommitted;
    ha.n_masked_left = ctrl + kCtrlMaskedLeft;
    ha.accumulate = p0 > 0 ? 1 : 0;
    ha.err = err;
    ha.M = m;
    ha.H = d.hidden;
    ha.V = d.vocab;
    ha.mask_id = d.mask_id;
    ha.block = block;
    ha.n_tiles = (d.vocab + 127) / 128;
    ha.threshold = threshold;
    if (accept) {
      ha.draft = acc->draft + p0;
      ha.part_t = reinterpret_cast<float*>(data + L.part_t);
      ha.part_zd = reinterpret_cast<float*>(data + L.part_zd);
      ha.entropy = acc->entropy ? acc->entropy + p0 : nullptr;
      ha.p_draft = acc->p_draft ? acc->p_draft + p0 : nullptr;
      ha.accept_len = acc->accept_len + p0 / block;
      ha.out_tokens = acc->out_tokens + p0;
      ha.rule = acc->rule;
      ha.ratio = acc->ratio;
      ha.delta = acc->delta;
    }
    // Two K groups per stage at up to 64 positions (half the pipeline steps);
    // 8 groups of weights (128 KiB) in flight per SM streamed best on GB300.
    const int kg = (nb <= 64 && (d.hidden / 64) % 2 == 0) ? 2 : 1;
    ha.kg = kg;
    const size_t fixed = head_smem_bytes(0, nb, accept, kg) + 16 * 2 * 8;
    ha.stages = static_cast<int>(std::min<size_t>(
        8 / kg, (static_cast<size_t>(kSmemBudget) - fixed) / (kg * (kATileBytes + static_cast<size_t>(nb) * 128))));
    const int grid = std::max(1, std::min(std::min(ha.n_tiles, plan.sms), kHeadMaxCtas));
    if (ha.stages < 1) return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "head pipeline does not fit in shared memory");
    ha.n_parts = grid;
    ha.dec_m = reinterpret_cast<float*>(data + L.dec_m);
    ha.dec_s = accept ? reinterpret_cast<float*>(data + L.dec_s) : nullptr;
    ha.dec_a = reinterpret_cast<int*>(data + L.dec_a);
    e = launch_head(ha, accept, grid, head_smem_bytes(ha.stages, nb, accept, kg), stream, kPdl);
    if (e != cudaSuccess) return cuda_fail(e, "launch head");
    e = launch_head_merge(ha, accept, stream, kPdl);
    if (e != cudaSuccess) return cuda_fail(e, "launch head merge");
  }
  return CLOVER_OK;
}

int check_ws(void* ws, size_t have, size_t need) {
  if (ws == nullptr) return fail(CLOVER_ERR_INVALID_ARG, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(CLOVER_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (have < need) return fail(CLOVER_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, needs %zu", have, need);
  return CLOVER_OK;
}

int check_launch_errors(const char* where) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, where);
  return CLOVER_OK;
}

int denoise_step_impl(const clover_dims* dims, const clover_moe_layer* layers, int32_t n_layers, const uint16_t* embed,
                      const float* ctx, const uint16_t* head_w, const float* logit_scale, float threshold,
                      int32_t block, int32_t* tokens, uint8_t* masked, int32_t M, void* workspace,
                      size_t workspace_bytes, clover_stream_t stream) {
  int rc;
  if ((rc = check_dims(dims))) return rc;
  if ((rc = check_tokens(M))) return rc;
  if (n_layers < 0) return fail(CLOVER_ERR_INVALID_ARG, "n_layers < 0");
  if (n_layers > 0 && layers == nullptr) return fail(CLOVER_ERR_INVALID_ARG, "layers is NULL");
  if (!embed || !ctx || !head_w || !tokens || !masked)
    return fail(CLOVER_ERR_INVALID_ARG, "NULL embed/ctx/head_w/tokens/masked");
  if (!aligned16(embed) || !aligned16(ctx) || !aligned16(head_w))
    return fail(CLOVER_ERR_INVALID_ARG, "embed/ctx/head_w must be 16-byte aligned");
  if (block < 1 || M % block != 0) return fail(CLOVER_ERR_INVALID_ARG, "block=%d must divide M=%d", block, M);
  if (dims->coreset_top_p > 0.f && block != M)
    return fail(CLOVER_ERR_UNSUPPORTED_SHAPE, "the block coreset needs one block per call (block == M)");
  if (!(threshold == threshold)) return fail(CLOVER_ERR_INVALID_ARG, "threshold is NaN");
  for (int i = 0; i < n_layers; ++i)
    if ((rc = check_layer(&layers[i], i))) return rc;
  const DenoiseLayout L = denoise_layout(*dims, M);
  if ((rc = check_ws(workspace, workspace_bytes, L.bytes))) return rc;
  if ((rc = get_encoder())) return rc;
  DevInfo di;
  if ((rc = device_info(&di))) return rc;
  const Plan plan{di.sms};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* ctrl = reinterpret_cast<int*>(ws);
  int* err = ctrl + kCtrlErr;
  float* x = reinterpret_cast<float*>(ws + L.x);

  EmbedArgs ea;
  ea.tokens = tokens;
  ea.embed = reinterpret_cast<const bf16*>(embed);
  ea.ctx = ctx;
  ea.x = x;
  ea.err = err;
  ea.M = M;
  ea.H = dims->hidden;
  ea.V = dims->vocab;
  cudaError_t e = launch_embed(ea, s, kPdl);
  if (e != cudaSuccess) return cuda_fail(e, "launch embed");
  // With the fused layer kernel each layer's combine runs at the start of
  // the next layer's launch, spread over all CTAs (one pass over the expert
  // rows instead of a serial walk at the end of the launch); the last one is
  // a combine kernel.
  const bool defer = plan::moe_fused(M, dims->n_experts, plan.sms);
  // Above 32 positions each layer's combine also writes the next layer's
  // normed rows, which the next routing kernel copies instead of
  // normalising them again in every expert tile.
  const bool chain_norm = !defer && dims->hidden <= kRouteChunk;
  for (int l = 0; l < n_layers; ++l) {
    rc = enqueue_moe_layer(*dims, layers[l], x, x, nullptr, nullptr, M, ws + L.moe,
                           reinterpret_cast<int*>(ws + L.moe_ctrl), err, plan, s,
                           l + 1 < n_layers ? layers[l + 1].router_w : nullptr, defer, defer && l > 0,
                           chain_norm && l > 0, chain_norm && l + 1 < n_layers, l + 1 < n_layers ? &layers[l + 1] : nullptr);
    if (rc) return rc;
  }
  if (defer && n_layers > 0 && (rc = enqueue_combine(*dims, x, M, ws + L.moe, s))) return rc;
  rc = enqueue_head(*dims, head_w, x, logit_scale, threshold, block, tokens, masked, nullptr, nullptr, nullptr,
                    nullptr, ctrl + kCtrlCommitted, M, ws + L.head, reinterpret_cast<int*>(ws + L.head_ctrl), err,
                    plan, s);
  if (rc) return rc;
  // The step's masked-count lands in the head control block; mirror it into
  // the top-level control block for the loop.
  e = cudaMemcpyAsync(ctrl + kCtrlMaskedLeft, reinterpret_cast<int*>(ws + L.head_ctrl) + kCtrlMaskedLeft, sizeof(int),
                      cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(masked count)");
  return check_launch_errors("denoise step");
}

}  // namespace

namespace clover {
// Lets other translation units of the library report through
// clover_last_error().
int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

// clover_lmhead_unmask with one option: clear_ctrl zeroes the workspace's
// control words on the stream (after every argument check, so a rejected
// call enqueues nothing) for scratch memory whose previous contents are not
// known.
int lmhead_unmask_check(const clover_dims* dims, const uint16_t* head_w, const float* x, float threshold,
                        int32_t block, const int32_t* tokens, const uint8_t* masked, int32_t M) {
  int rc;
  if ((rc = check_dims(dims))) return rc;
  if ((rc = check_tokens(M))) return rc;
  if (!head_w || !x || !tokens || !masked) return fail(CLOVER_ERR_INVALID_ARG, "NULL head_w/x/tokens/masked");
  if (!aligned16(head_w) || !aligned16(x)) return fail(CLOVER_ERR_INVALID_ARG, "head_w/x not 16-byte aligned");
  if (block < 1) return fail(CLOVER_ERR_INVALID_ARG, "block=%d < 1", block);
  if (!(threshold == threshold)) return fail(CLOVER_ERR_INVALID_ARG, "threshold is NaN");
  return CLOVER_OK;
}

int lmhead_unmask_impl(const clover_dims* dims, const uint16_t* head_w, const float* x, const float* logit_scale,
                       float threshold, int32_t block, int32_t* tokens, uint8_t* masked, int32_t* argmax,
                       float* max_logit, float* lse, float* max_prob, int32_t* n_committed, int32_t M,
                       void* workspace, size_t workspace_bytes, clover_stream_t stream, bool clear_ctrl) {
  int rc;
  if ((rc = lmhead_unmask_check(dims, head_w, x, threshold, block, tokens, masked, M))) return rc;
  if ((rc = check_ws(workspace, workspace_bytes, kCtrlBytes + head_layout(*dims, M).bytes))) return rc;
  if ((rc = get_encoder())) return rc;
  DevInfo di;
  if ((rc = device_info(&di))) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* ctrl = reinterpret_cast<int*>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (clear_ctrl) {
    const cudaError_t e = cudaMemsetAsync(ws, 0, kCtrlBytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the control words");
  }
  rc = enqueue_head(*dims, head_w, x, logit_scale, threshold, block, tokens, masked, argmax, max_logit, lse, max_prob,
                    n_committed, M, ws + kCtrlBytes, ctrl, ctrl + kCtrlErr, Plan{di.sms}, s);
  if (rc) return rc;
  return check_launch_errors("lmhead unmask");
}

// Synchronises the stream, reads the status word of the control block at
// `workspace`, and if it is set clears the control block and reports it.
int workspace_status_impl(void* workspace, size_t workspace_bytes, clover_stream_t stream) {
  if (workspace == nullptr || workspace_bytes < kCtrlBytes) return fail(CLOVER_ERR_INVALID_ARG, "bad workspace");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace status");
  if (word == 0) return CLOVER_OK;
  // Clear the status word and the arrival counters a failed kernel may have
  // left behind, so the workspace is usable again.
  e = cudaMemset(workspace, 0, kCtrlBytes);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace status");
  char what[200] = {0};
  snprintf(what, sizeof(what), "%s%s%s%s%s", (word & kErrMbarTimeout) ? "pipeline wait timed out; " : "",
           (word & kErrDepTimeout) ? "cross-CTA dependency wait timed out; " : "",
           (word & kErrBadToken) ? "token id out of range; " : "",
           (word & kErrBadRoute) ? "expert id out of range; " : "",
           (word & kErrState) ? "work counters inconsistent (workspace changed between calls?); " : "");
  return fail(CLOVER_ERR_DEVICE_TIMEOUT, "device status 0x%x: %s", word, what);
}
}  // namespace clover

extern "C" {

size_t clover_moe_workspace_bytes(const clover_dims* dims, int32_t max_tokens) {
  if (check_dims(dims) || check_tokens(max_tokens)) return 0;
  return kCtrlBytes + moe_layout(*dims, max_tokens).bytes;
}

int clover_moe_block_step(const clover_dims* dims, const clover_moe_layer* layer, const float* x_in, float* x_out,
                          int32_t* topk_idx, float* topk_w, int32_t M, void* workspace, size_t workspace_bytes,
                          clover_stream_t stream) {
  int rc;
  if ((rc = check_dims(dims))) return rc;
  if ((rc = check_tokens(M))) return rc;
  if ((rc = check_layer(layer, 0))) return rc;
  if (!x_in || !x_out) return fail(CLOVER_ERR_INVALID_ARG, "x_in/x_out is NULL");
  if (!aligned16(x_in) || !aligned16(x_out)) return fail(CLOVER_ERR_INVALID_ARG, "x_in/x_out not 16-byte aligned");
  const size_t xb = static_cast<size_t>(M) * dims->hidden * 4;
  const uint8_t* a0 = reinterpret_cast<const uint8_t*>(x_in);
  const uint8_t* b0 = reinterpret_cast<const uint8_t*>(x_out);
  if (a0 != b0 && a0 < b0 + xb && b0 < a0 + xb) return fail(CLOVER_ERR_INVALID_ARG, "x_in and x_out partially overlap");
  if ((rc = check_ws(workspace, workspace_bytes, kCtrlBytes + moe_layout(*dims, M).bytes))) return rc;
  if ((rc = get_encoder())) return rc;
  DevInfo di;
  if ((rc = device_info(&di))) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* ctrl = reinterpret_cast<int*>(ws);
  rc = enqueue_moe_layer(*dims, *layer, x_in, x_out, topk_idx, topk_w, M, ws + kCtrlBytes, ctrl, ctrl + kCtrlErr,
                         Plan{di.sms}, reinterpret_cast<cudaStream_t>(stream));
  if (rc) return rc;
  return check_launch_errors("moe block step");
}

size_t clover_head_workspace_bytes(const clover_dims* dims, int32_t max_tokens) {
  if (check_dims(dims) || check_tokens(max_tokens)) return 0;
  return kCtrlBytes + head_layout(*dims, max_tokens).bytes;
}

int clover_lmhead_unmask(const clover_dims* dims, const uint16_t* head_w, const float* x, const float* logit_scale,
                         float threshold, int32_t block, int32_t* tokens, uint8_t* masked, int32_t* argmax,
                         float* max_logit, float* lse, float* max_prob, int32_t* n_committed, int32_t M,
                         void* workspace, size_t workspace_bytes, clover_stream_t stream) {
  return clover::lmhead_unmask_impl(dims, head_w, x, logit_scale, threshold, block, tokens, masked, argmax, max_logit,
                                    lse, max_prob, n_committed, M, workspace, workspace_bytes, stream, false);
}

int clover_quantize_q4(const uint16_t* w, int32_t n_mats, int32_t rows, int32_t cols, uint8_t* q, uint16_t* s,
                       clover_stream_t stream) {
  if (!w || !q || !s) return fail(CLOVER_ERR_INVALID_ARG, "NULL w/q/s");
  if (!aligned16(w) || !aligned16(q) || !aligned16(s)) return fail(CLOVER_ERR_INVALID_ARG, "w/q/s not 16-byte aligned");
  if (n_mats < 1 || rows < 1 || cols < 64 || cols % 64 != 0)
    return fail(CLOVER_ERR_INVALID_ARG, "n_mats=%d rows=%d cols=%d: need >= 1 and cols %% 64 == 0", n_mats, rows, cols);
  QuantArgs a;
  a.w = reinterpret_cast<const bf16*>(w);
  a.q = q;
  a.s = s;
  a.n_mats = n_mats;
  a.rows = rows;
  a.cols = cols;
  cudaError_t e = launch_quantize_q4(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launch quantize");
  return check_launch_errors("quantize q4");
}

size_t clover_accept_workspace_bytes(const clover_dims* dims, int32_t max_rows) {
  if (check_dims(dims) || check_tokens(max_rows)) return 0;
  return kCtrlBytes + head_layout(*dims, max_rows, true).bytes;
}

int clover_lmhead_accept(const clover_dims* dims, const uint16_t* head_w, const float* x, const float* logit_scale,
                         const int32_t* draft, int32_t rule, float ratio, float delta, int32_t block,
                         int32_t* argmax, float* max_logit, float* lse, float* max_prob, float* entropy,
                         float* p_draft, int32_t* accept_len, int32_t* out_tokens, int32_t M, void* workspace,
                         size_t workspace_bytes, clover_stream_t stream) {
  int rc;
  if ((rc = check_dims(dims))) return rc;
  if ((rc = check_tokens(M))) return rc;
  if (!head_w || !x || !draft || !accept_len || !out_tokens)
    return fail(CLOVER_ERR_INVALID_ARG, "NULL head_w/x/draft/accept_len/out_tokens");
  if (!aligned16(head_w) || !aligned16(x)) return fail(CLOVER_ERR_INVALID_ARG, "head_w/x not 16-byte aligned");
  if (block < 2 || M % block != 0)
    return fail(CLOVER_ERR_INVALID_ARG, "block=%d: need >= 2 rows per block (drafts + 1) dividing M=%d", block, M);
  if (rule != CLOVER_ACCEPT_EXACT && rule != CLOVER_ACCEPT_THRESHOLD)
    return fail(CLOVER_ERR_INVALID_ARG, "rule=%d is neither exact nor threshold", rule);
  if (rule == CLOVER_ACCEPT_THRESHOLD && !(ratio > 0.f && ratio <= 1.f && delta > 0.f && delta < 1e30f))
    return fail(CLOVER_ERR_INVALID_ARG, "threshold rule needs 0 < ratio <= 1 and a finite delta > 0");
  if ((rc = check_ws(workspace, workspace_bytes, kCtrlBytes + head_layout(*dims, M, true).bytes))) return rc;
  if ((rc = get_encoder())) return rc;
  DevInfo di;
  if ((rc = device_info(&di))) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* ctrl = reinterpret_cast<int*>(ws);
  const AcceptCfg acc{draft, rule, ratio, delta, entropy, p_draft, accept_len, out_tokens};
  rc = enqueue_head(*dims, head_w, x, logit_scale, 0.f, block, nullptr, nullptr, argmax, max_logit, lse, max_prob,
                    nullptr, M, ws + kCtrlBytes, ctrl, ctrl + kCtrlErr, Plan{di.sms},
                    reinterpret_cast<cudaStream_t>(stream), &acc);
  if (rc) return rc;
  return check_launch_errors("lmhead accept");
}

size_t clover_denoise_workspace_bytes(const clover_dims* dims, int32_t max_tokens) {
  if (check_dims(dims) || check_tokens(max_tokens)) return 0;
  return denoise_layout(*dims, max_tokens).bytes;
}

size_t clover_denoise_hidden_offset(const clover_dims* dims, int32_t max_tokens) {
  if (check_dims(dims) || check_tokens(max_tokens)) return 0;
  return denoise_layout(*dims, max_tokens).x;
}

int clover_denoise_step(const clover_dims* dims, const clover_moe_layer* layers, int32_t n_layers,
                        const uint16_t* embed, const float* ctx, const uint16_t* head_w, const float* logit_scale,
                        float threshold, int32_t block, int32_t* tokens, uint8_t* masked, int32_t M,
                        void* workspace, size_t workspace_bytes, clover_stream_t stream) {
  return denoise_step_impl(dims, layers, n_layers, embed, ctx, head_w, logit_scale, threshold, block, tokens, masked,
                           M, workspace, workspace_bytes, stream);
}

int clover_denoise_block(const clover_dims* dims, const clover_moe_layer* layers, int32_t n_layers,
                         const uint16_t* embed, const float* ctx, const uint16_t* head_w, const float* logit_scale,
                         float threshold, int32_t block, int32_t* tokens, uint8_t* masked, int32_t M,
                         int32_t max_steps, int32_t* steps_taken, void* workspace, size_t workspace_bytes,
                         clover_stream_t stream) {
  if (steps_taken == nullptr) return fail(CLOVER_ERR_INVALID_ARG, "steps_taken is NULL");
  *steps_taken = 0;
  if (max_steps < 0) return fail(CLOVER_ERR_INVALID_ARG, "max_steps < 0");
  int rc;
  if ((rc = check_tokens(M))) return rc;
  if (masked == nullptr) return fail(CLOVER_ERR_INVALID_ARG, "masked is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t host_masked[kMaxTokens];  // M <= kMaxTokens (checked above)
  cudaError_t e = cudaMemcpyAsync(host_masked, masked, M, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the mask");
  int left = 0;
  for (int i = 0; i < M; ++i) left += host_masked[i] != 0;
  int steps = 0;
  while (left > 0 && steps < max_steps) {
    rc = denoise_step_impl(dims, layers, n_layers, embed, ctx, head_w, logit_scale, threshold, block, tokens, masked,
                           M, workspace, workspace_bytes, stream);
    if (rc) return rc;
    int words[3] = {0, 0, 0};
    e = cudaMemcpyAsync(words, workspace, sizeof(words), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the step status");
    ++steps;
    *steps_taken = steps;
    if (words[kCtrlErr] != 0)
      return fail(CLOVER_ERR_DEVICE_TIMEOUT, "kernel status 0x%x after step %d", words[kCtrlErr], steps);
    left = words[kCtrlMaskedLeft];
  }
  if (left > 0) return fail(CLOVER_ERR_NOT_CONVERGED, "%d positions still masked after %d steps", left, steps);
  return CLOVER_OK;
}

int clover_workspace_status(void* workspace, size_t workspace_bytes, clover_stream_t stream) {
  return clover::workspace_status_impl(workspace, workspace_bytes, stream);
}

int32_t clover_profile_expert_events(clover_event_t* begin, clover_event_t* end, int32_t capacity) {
  const int n = g_prof.count;
  g_prof.begin = reinterpret_cast<cudaEvent_t*>(begin);
  g_prof.end = reinterpret_cast<cudaEvent_t*>(end);
  g_prof.cap = (begin && end) ? capacity : 0;
  g_prof.count = 0;
  return n;
}

int32_t clover_last_error(char* buf, size_t n) {
  const size_t len = strlen(g_err);
  if (buf && n > 0) {
    const size_t c = len < n - 1 ? len : n - 1;
    memcpy(buf, g_err, c);
    buf[c] = '\0';
  }
  return static_cast<int32_t>(len);
}

int32_t clover_version(void) { return 100; }

}  // extern "C"
