// C ABI of the fused MoE layer: argument checks, workspace layout, TMA
// descriptors and the launch sequence.  Every step of the layer runs in this
// library's kernels; the host only validates and enqueues.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "moe_gb300.h"

namespace moe {
namespace {

constexpr unsigned long long kWaitLimitNs = 5000000000ull;  // 5 s per bounded wait
constexpr int kMaxExperts = 1024;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct DeviceInfo {
  int num_sms = 0;
  int major = 0, minor = 0;
};

DeviceInfo device_info(int dev) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return DeviceInfo{};
  if (!have[dev]) {
    DeviceInfo d;
    cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    cache[dev] = d;
    have[dev] = true;
  }
  return cache[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D K-major tile map: rows of `row_bytes`, boxes of (128 bytes of K) x box_rows,
// written to shared memory with the 128-byte swizzle the UMMA descriptors expect.
bool make_tmap(CUtensorMap* m, const void* base, bool bf16, uint64_t k_elems, uint64_t rows,
               uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) {
    note_cuda_error(0, "entry point not found", "cuTensorMapEncodeTiled");
    return false;
  }
  const uint64_t esize = bf16 ? 2 : 1;
  cuuint64_t dims[2] = {k_elems, rows};
  cuuint64_t strides[1] = {k_elems * esize};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) note_cuda_error(static_cast<int>(r), "CUresult", "cuTensorMapEncodeTiled");
  return r == CUDA_SUCCESS;
}

// Row-tile width of the expert GEMMs: 128 rows, the widest tile whose gate/up
// accumulators (2 x 128 columns) are still double-buffered in the 512 TMEM
// columns.  The routing is not known when the launch is planned, and a
// narrower tile would split a busy expert's rows and read its weight blocks
// once per piece (skewed routing); the weight-in-M placement only loads the
// rows a tile has, so the width costs decode nothing but shared memory.
int choose_bn_max(long long, int) { return kTokMRows; }

// CTAs the persistent GEMMs may use on the current device (also sizes the
// split-tile partial slots); 256 when no device can be queried.
int gemm_ctas() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 256;
  const DeviceInfo d = device_info(dev);
  return d.num_sms > 0 ? std::min(d.num_sms, 256) : 256;
}

// Workspace layout of the fused forward (all regions 256-byte aligned).
struct Layout {
  long long P = 0;
  int pad_max = 0;     // upper bound of aligned rows: P + E*(16-1)
  int max_mtiles = 0;  // upper bound of GEMM row tiles
  int n_partials = 0;  // router CTAs
  int bn_max = 0;
  int ctas = 0;
  int n_tile_cnt = 0;
  // Combine of the down projection: bulk reductions into an fp32 [T, H]
  // buffer (small batches), or weighted bf16 rows at the pairs' aligned rows
  // summed by a separate kernel through inv_slot (large batches, where the
  // reductions would saturate L2).
  bool combine_rows = false;
  size_t rows = 0;
  // Large batches: two-pass alignment (per-chunk histograms); FP8: x quantised
  // once per token and scattered to its aligned rows (inv_slot: row of each
  // pair, also read by the row combine).
  bool large = false;
  size_t chunk_hist = 0, inv_slot = 0;
  size_t ctrl = 0, trace = 0, partials = 0, ids = 0, wts = 0, counts = 0, offsets = 0,
         sorted = 0, sorted_w = 0, mtiles = 0, mtiles_w = 0, tile_cnt = 0, part = 0, xs = 0, h = 0, hq = 0, acc = 0,
         total = 0;
};

Layout make_layout(int T, int H, int I, int E, int k, bool fp8) {
  Layout L;
  L.P = static_cast<long long>(T) * k;
  L.pad_max = static_cast<int>(L.P + static_cast<long long>(E) * (kAlignBlock - 1));
  L.max_mtiles = L.pad_max / kAlignBlock + 1;
  L.n_partials = route_grid(T);
  L.bn_max = choose_bn_max(L.P, E);
  L.ctas = gemm_ctas();
  L.n_tile_cnt = L.max_mtiles * (I / 128);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.ctrl = take(sizeof(Ctrl));
  L.trace = take(sizeof(unsigned long long) * 2 * MOE_TRACE_MAX_CTAS * 4);
  // router amax partials: one per router CTA, or one per CTA of the
  // single-kernel small-batch path (at most one per SM)
  L.partials = take(sizeof(float) * std::max(L.n_partials, 1024));
  L.ids = take(sizeof(int32_t) * L.P);
  L.wts = take(sizeof(float) * L.P);
  L.counts = take(sizeof(int32_t) * E);
  L.offsets = take(sizeof(int32_t) * (E + 1));
  L.sorted = take(sizeof(int32_t) * L.pad_max);
  L.sorted_w = take(sizeof(float) * L.pad_max);
  L.mtiles = take(sizeof(int4) * L.max_mtiles);
  L.mtiles_w = take(sizeof(int4) * L.max_mtiles);
  L.tile_cnt = take(sizeof(int) * static_cast<size_t>(L.n_tile_cnt));
  // sized for the widest row tile (wide gate/up tiles have 256 rows)
  L.part = take(sizeof(float) * 2 * static_cast<size_t>(L.ctas) * gemm_part_slot_floats(kWideRows));
  L.xs = take(static_cast<size_t>(L.pad_max) * H * (fp8 ? 1 : 2));
  L.h = take(static_cast<size_t>(L.pad_max) * I * (fp8 ? 4 : 2));
  L.hq = take(fp8 ? static_cast<size_t>(L.pad_max) * I : 0);
  L.large = L.P > kLargePairs;
  L.chunk_hist = take(L.large ? sizeof(int32_t) * E * ((L.P + align_chunk() - 1) / align_chunk()) : 0);
  L.combine_rows = combine_by_rows(L.P, H);
  L.inv_slot = take((L.large && fp8) || L.combine_rows ? sizeof(int32_t) * L.P : 0);
  L.acc = take(L.combine_rows ? 0 : static_cast<size_t>(T) * H * sizeof(float));
  L.rows = take(L.combine_rows ? static_cast<size_t>(L.pad_max) * H * 2 : 0);
  L.total = off;
  return L;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int next_pow2(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

moe_status_t check_device(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  DeviceInfo d = device_info(dev);
  if (d.major != 10 || d.minor != 3) return MOE_ERR_UNSUPPORTED;
  *out = d;
  return MOE_OK;
}

}  // namespace

namespace {
thread_local char g_last_error[256] = "no error";
}

void note_cuda_error(int code, const char* what, const char* where) {
  snprintf(g_last_error, sizeof g_last_error, "%s: %s (%d)", where ? where : "?",
           what ? what : "?", code);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_last_error_detail(void) { return g_last_error; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_RANGE: return "device kernel met an out-of-range expert id";
  }
  return "unknown status";
}

moe_status_t moe_route_topk(const float* logits, int T, int E, int top_k, int renormalize,
                            int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || top_k < 1 || top_k > E) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
    return MOE_ERR_INVALID_ARG;
  DeviceInfo d;
  moe_status_t s = check_device(&d);
  if (s != MOE_OK) return s;
  return launch_route_topk(logits, T, E, top_k, renormalize, topk_ids, topk_w, nullptr, 0,
                           nullptr, nullptr, nullptr, 0, stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status_t moe_align_by_expert(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                                 int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                                 int32_t* tile_expert, int32_t* num_padded, moe_stream_t stream) {
  if (T < 0 || top_k < 1 || E < 1 || E > kMaxExperts || block_m < 1 || block_m > 256)
    return MOE_ERR_INVALID_ARG;
  const long long P = static_cast<long long>(T) * top_k;
  if (P + static_cast<long long>(E) * block_m >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  if (!topk_ids && P > 0) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || !sorted_ids) return MOE_ERR_INVALID_ARG;
  DeviceInfo d;
  moe_status_t s = check_device(&d);
  if (s != MOE_OK) return s;
  AlignParams p{};
  p.ids = topk_ids;
  p.P = static_cast<int>(P);
  p.E = E;
  p.bm = block_m;
  p.chunk = align_chunk();
  p.counts = counts;
  p.offsets = offsets;
  p.sorted_ids = sorted_ids;
  p.tile_expert = tile_expert;
  p.num_padded = num_padded;
  return launch_align(p, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_quantize_scratch_size(int T, int H) {
  (void)T;
  (void)H;
  return 1024 * sizeof(float);
}

moe_status_t moe_quantize_e4m3(const void* x, int T, int H, uint8_t* x_q, float* scale,
                               void* scratch, size_t scratch_bytes, moe_stream_t stream) {
  if (T < 0 || H < 16 || H % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !x_q || !scale || !aligned(x, 16) || !aligned(x_q, 16) || !aligned(scale, 4))
    return MOE_ERR_INVALID_ARG;
  if (!scratch || !aligned(scratch, 4) || scratch_bytes < moe_quantize_scratch_size(T, H))
    return MOE_ERR_WORKSPACE;
  DeviceInfo d;
  moe_status_t s = check_device(&d);
  if (s != MOE_OK) return s;
  const long long n = static_cast<long long>(T) * H;
  int parts = std::min(1024, std::max(1, d.num_sms * 4));
  parts = static_cast<int>(std::min<long long>(parts, (n / 8 + 255) / 256));
  if (parts < 1) parts = 1;
  return launch_quantize_e4m3(static_cast<const __nv_bfloat16*>(x), n, x_q, scale,
                              static_cast<float*>(scratch), parts, stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

size_t moe_inv_rope_scratch_size(int T, int NH, int D) {
  if (T < 0 || NH < 1 || NH > 4096 || D < 8 || D > 256 || (D & (D - 1)) != 0) return 0;
  return 256 + sizeof(float) * static_cast<size_t>(kRopeMaxCtas) * (NH + 1);
}

moe_status_t moe_inv_rope_quant_per_head(const void* x, const int32_t* positions,
                                         const float* cos_tab, const float* sin_tab, int T,
                                         int NH, int D, int max_pos, uint8_t* codes,
                                         float* scales, void* scratch, size_t scratch_bytes,
                                         moe_stream_t stream) {
  const size_t need = moe_inv_rope_scratch_size(T, NH, D);
  if (need == 0 || max_pos < 1) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (static_cast<long long>(T) * NH * D >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (!x || !positions || !cos_tab || !sin_tab || !codes || !scales) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(cos_tab, 16) || !aligned(sin_tab, 16) || !aligned(codes, 8) ||
      !aligned(positions, 4) || !aligned(scales, 4))
    return MOE_ERR_INVALID_ARG;
  if (!scratch || !aligned(scratch, 256) || scratch_bytes < need) return MOE_ERR_WORKSPACE;
  DeviceInfo dev;
  moe_status_t st = check_device(&dev);
  if (st != MOE_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  return launch_inv_rope_quant(static_cast<const __nv_bfloat16*>(x), positions, cos_tab, sin_tab,
                               T, NH, D, max_pos, codes, scales, reinterpret_cast<Ctrl*>(ws),
                               reinterpret_cast<float*>(ws + 256), dev.num_sms,
                               stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

size_t moe_fused_workspace_size(int T, int H, int I, int E, int top_k, moe_dtype_t dtype) {
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || E > kMaxExperts || top_k < 1 || top_k > E) return 0;
  if (dtype != MOE_DT_BF16 && dtype != MOE_DT_FP8_E4M3) return 0;
  return make_layout(T, H, I, E, top_k, dtype == MOE_DT_FP8_E4M3).total;
}

}  // extern "C"

namespace {

// On request (MOE_FLAG_ONE_KERNEL), small batches take the single-kernel
// path: the whole layer in one cooperative persistent kernel (weights in the
// MMA M slot for both GEMMs).  The shape rule (host only):
bool fused_small_shape(int T, int H, int I, int E, int k, int flags, const Layout& L) {
  const long long P = static_cast<long long>(T) * k;
  if (P > kFusedMaxPairs || E > kFusedMaxExperts || L.combine_rows) return false;
  if (!(flags & MOE_FLAG_ONE_KERNEL) || (flags & MOE_FLAG_TOKENS_IN_M)) return false;
  return H % 128 == 0 && I % 128 == 0;
}

bool fused_small(int T, int H, int I, int E, int k, int flags, const Layout& L, int device,
                 int num_sms) {
  if (!fused_small_shape(T, H, I, E, k, flags, L)) return false;
  if (num_sms < 8 || num_sms > 256) return false;  // one partial slot pair per CTA (<= 256)
  return fused_small_supported(device);
}

// Small batches take the single-CTA router + alignment kernel (which writes
// no inverse slot map, so not where the down projection combines by rows).
bool small_front(int T, int H, int E, int k) {
  const long long P = static_cast<long long>(T) * k;
  return T <= kSmallMaxTokens && P <= kSmallMaxPairs && E <= kSmallMaxExperts &&
         static_cast<long long>(T) * H <= kSmallMaxXElems && !combine_by_rows(P, H);
}

// The launch sequence.  When `events` is non-null, events[i] is recorded on
// the stream before step i (i = 0..6) and events[7] after the last step.
// phase 0: the whole layer; 1: routing through the gate/up GEMM; 2: the
// quantisation of h (with the max |h| found in the workspace), the down GEMM
// and the output (tensor-parallel shards reduce the max between the two).
moe_status_t fused_forward_impl(const moe_fused_args* a, void* workspace, size_t workspace_bytes,
                                moe_stream_t stream, cudaEvent_t const* events, int phase = 0) {
  if (!a) return MOE_ERR_INVALID_ARG;
  const int T = a->T, H = a->H, I = a->I, E = a->E, k = a->top_k;
  if (T < 0 || H <= 0 || I <= 0 || E < 1 || E > kMaxExperts || k < 1 || k > E)
    return MOE_ERR_INVALID_ARG;
  if (a->weight_dtype != MOE_DT_BF16 && a->weight_dtype != MOE_DT_FP8_E4M3)
    return MOE_ERR_INVALID_ARG;
  if ((a->debug_flags & MOE_FLAG_TOKENS_IN_M) && (a->debug_flags & MOE_FLAG_WEIGHTS_IN_M))
    return MOE_ERR_INVALID_ARG;
  const bool fp8 = a->weight_dtype == MOE_DT_FP8_E4M3;
  if (fp8 && (!a->w13_scale || !a->w2_scale)) return MOE_ERR_INVALID_ARG;
  if (!fp8 && (a->w13_scale || a->w2_scale)) return MOE_ERR_INVALID_ARG;
  if (H % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  const long long P = static_cast<long long>(T) * k;
  if (P + static_cast<long long>(E) * kAlignBlock >= (1ll << 31) / 2) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!a->x || !a->router_logits || !a->w13 || !a->w2 || !a->out) return MOE_ERR_INVALID_ARG;
  if (!aligned(a->x, 16) || !aligned(a->w13, 16) || !aligned(a->w2, 16) || !aligned(a->out, 16) ||
      !aligned(a->router_logits, 4) || (a->w13_scale && !aligned(a->w13_scale, 4)) ||
      (a->w2_scale && !aligned(a->w2_scale, 4)) ||
      (a->topk_ids_out && !aligned(a->topk_ids_out, 4)) ||
      (a->topk_w_out && !aligned(a->topk_w_out, 4)) ||
      (a->counts_out && !aligned(a->counts_out, 4)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(T, H, I, E, k, fp8);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  DeviceInfo dev;
  moe_status_t st = check_device(&dev);
  if (st != MOE_OK) return st;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  float* partials = reinterpret_cast<float*>(ws + L.partials);
  int32_t* ids = a->topk_ids_out ? a->topk_ids_out : reinterpret_cast<int32_t*>(ws + L.ids);
  float* wts = a->topk_w_out ? a->topk_w_out : reinterpret_cast<float*>(ws + L.wts);
  int32_t* counts = a->counts_out ? a->counts_out : reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
  float* sorted_w = reinterpret_cast<float*>(ws + L.sorted_w);
  int32_t* inv_slot = reinterpret_cast<int32_t*>(ws + L.inv_slot);
  int4* mtiles = reinterpret_cast<int4*>(ws + L.mtiles);
  void* xs = ws + L.xs;
  void* h = ws + L.h;
  uint8_t* hq = ws + L.hq;
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  __nv_bfloat16* pair_rows = reinterpret_cast<__nv_bfloat16*>(ws + L.rows);
  const long long acc_elems = L.combine_rows ? 0 : static_cast<long long>(T) * H;

  const long long touched = std::min<long long>(E, P);
  // Operand placement.  Gate/up: the weight block in M (the swap).  Down:
  // the weight block in M when K = I is long; with short K (I <= 2048) the
  // MMA time per tile is small and the token-in-M epilogue, which writes 16
  // consecutive outputs of one token per thread, is the cheaper one.  The two
  // flags force one placement on both GEMMs (ablation of the swap).
  const bool force_tok = (a->debug_flags & MOE_FLAG_TOKENS_IN_M) != 0;
  const bool force_w = (a->debug_flags & MOE_FLAG_WEIGHTS_IN_M) != 0;
  const bool tok_m1 = force_tok;
  const bool tok_m2 = force_tok || (!force_w && I / 128 <= 16);
  const int bn_max = L.bn_max;
  // Gate/up with the weights in M and experts of more than 256 rows on
  // average (prefill): 256-token tiles read each weight block half as often
  // (at the cost of a single TMEM accumulator buffer), from a second tile list.
  // FP8 wide tiles run on SM pairs (cta_group::2): 256 weight rows x 256
  // tokens per tile, each SM loading half of the token rows; there they pay
  // from 128 rows per expert on average, where many experts need two 128-row
  // tiles (measured at 2048 tokens, E=128, k=8, I=768: gate/up 106.5 -> 96.3
  // us uniform, 86.0 -> 63.5 us Zipf-skewed).
  const long long touched_ub = std::min<long long>(E, P);
  const long long avg_rows = (P + touched_ub - 1) / touched_ub;
  const bool pairs_ok = fp8 && I % 256 == 0 && (a->debug_flags & MOE_FLAG_NO_SM_PAIRS) == 0;
  const bool wide1 = !tok_m1 && (avg_rows > kWideRows || (pairs_ok && avg_rows >= kWideRows / 2));
  const bool pair1 = pairs_ok && wide1;
  int4* mtiles_w = reinterpret_cast<int4*>(ws + L.mtiles_w);
  int* tile_cnt = reinterpret_cast<int*>(ws + L.tile_cnt);
  float* part = reinterpret_cast<float*>(ws + L.part);

  cudaStream_t s = stream;
  if (events && cudaEventRecord(events[0], stream) != cudaSuccess) return MOE_ERR_CUDA;
  int cur_dev = 0;
  if (cudaGetDevice(&cur_dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (phase == 0 && fused_small(T, H, I, E, k, a->debug_flags, L, cur_dev, dev.num_sms)) {
    FusedParams fp{};
    fp.logits = a->router_logits;
    fp.x = static_cast<const __nv_bfloat16*>(a->x);
    fp.T = T;
    fp.H = H;
    fp.I = I;
    fp.E = E;
    fp.k = k;
    fp.renorm = a->renormalize;
    fp.w13_scale = fp8 ? a->w13_scale : nullptr;
    fp.w2_scale = fp8 ? a->w2_scale : nullptr;
    fp.out = static_cast<__nv_bfloat16*>(a->out);
    fp.ids = ids;
    fp.wts = wts;
    fp.counts_out = a->counts_out;
    fp.ctrl = ctrl;
    fp.amax_part = partials;
    fp.sorted_ids = sorted;
    fp.sorted_w = sorted_w;
    fp.xs = xs;
    fp.h = h;
    fp.hq = hq;
    fp.acc = acc;
    fp.part = part;
    fp.tile_cnt = tile_cnt;
    fp.n_tile_cnt = L.n_tile_cnt;
    fp.timeout_ns = (a->debug_flags & MOE_DEBUG_FORCE_TIMEOUT) ? MOE_DEBUG_TIMEOUT_MS * 1000000ull
                                                               : kWaitLimitNs;
    fp.debug = a->debug_flags;
    fp.trace = (a->debug_flags & MOE_DEBUG_TRACE)
                   ? reinterpret_cast<unsigned long long*>(ws + L.trace)
                   : nullptr;
    const bool bf = !fp8;
    const void* hb = fp8 ? static_cast<const void*>(hq) : static_cast<const void*>(h);
    CUtensorMap m_w13, m_xs, m_xs64, m_w2, m_h, m_h64;
    if (!make_tmap(&m_w13, a->w13, bf, H, static_cast<uint64_t>(E) * 2 * I, 128) ||
        !make_tmap(&m_xs, xs, bf, H, L.pad_max, 16) || !make_tmap(&m_xs64, xs, bf, H, L.pad_max, 64) ||
        !make_tmap(&m_w2, a->w2, bf, I, static_cast<uint64_t>(E) * H, 128) ||
        !make_tmap(&m_h, hb, bf, I, L.pad_max, 16) || !make_tmap(&m_h64, hb, bf, I, L.pad_max, 64))
      return MOE_ERR_CUDA;
    if (launch_fused_small(fp, m_w13, m_xs, m_xs64, m_w2, m_h, m_h64, dev.num_sms, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (events)
      for (int i = 1; i < MOE_TIMED_EVENTS; ++i)
        if (cudaEventRecord(events[i], stream) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (phase == 2) {
    // (routing, alignment and the x rows were written by the first call)
  } else if (small_front(T, H, E, k)) {
    // 1-2 in one CTA: routing, amax of x, alignment, tile list, s_x
    SmallFrontParams sp{};
    sp.logits = a->router_logits;
    sp.T = T;
    sp.E = E;
    sp.k = k;
    sp.renorm = a->renormalize;
    sp.ids = ids;
    sp.wts = wts;
    sp.x = fp8 ? static_cast<const __nv_bfloat16*>(a->x) : nullptr;
    sp.H = H;
    sp.ctrl = ctrl;
    sp.zero_ints = tile_cnt;
    sp.n_zero = L.n_tile_cnt;
    sp.counts = counts;
    sp.offsets = offsets;
    sp.sorted_ids = sorted;
    sp.sorted_w = sorted_w;
    sp.mtiles = mtiles;
    sp.bn_max = bn_max;
    sp.mtiles_w = wide1 ? mtiles_w : nullptr;
    if (launch_route_align_small(sp, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (events && (cudaEventRecord(events[1], stream) != cudaSuccess ||
                   cudaEventRecord(events[2], stream) != cudaSuccess))
      return MOE_ERR_CUDA;
  } else {
  // 1. routing (+ per-CTA amax of x, + reset of the control words)
  if (launch_route_topk(a->router_logits, T, E, k, a->renormalize, ids, wts,
                        static_cast<const __nv_bfloat16*>(a->x), H, fp8 ? partials : nullptr, ctrl,
                        tile_cnt, L.n_tile_cnt, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (events && cudaEventRecord(events[1], stream) != cudaSuccess) return MOE_ERR_CUDA;
  // 2. alignment by expert, GEMM row tiles, s_x
  AlignParams ap{};
  ap.ids = ids;
  ap.P = static_cast<int>(P);
  ap.E = E;
  ap.bm = kAlignBlock;
  ap.chunk = align_chunk();
  ap.counts = counts;
  ap.offsets = offsets;
  ap.sorted_ids = sorted;
  ap.wts = wts;
  ap.sorted_w = sorted_w;
  ap.inv_slot = ((L.large && fp8) || L.combine_rows) ? inv_slot : nullptr;
  ap.tile_expert = nullptr;
  ap.num_padded = nullptr;
  ap.mtiles = mtiles;
  ap.bn_max = bn_max;
  ap.mtiles_w = wide1 ? mtiles_w : nullptr;
  ap.ctrl = ctrl;
  ap.amax_partials = fp8 ? partials : nullptr;
  ap.n_partials = fp8 ? L.n_partials : 0;
  int32_t* chunk_hist = reinterpret_cast<int32_t*>(ws + L.chunk_hist);
  if (L.large) {
    if (launch_align_hist(ids, static_cast<int>(P), E, chunk_hist, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    ap.chunk_hist = chunk_hist;
  }
  if (launch_align(ap, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (events && cudaEventRecord(events[2], stream) != cudaSuccess) return MOE_ERR_CUDA;
  }
  // 3. the routed rows of x in aligned order, E4M3 with s_x (or bf16): large
  //    FP8 batches quantise each token once and scatter it to its k rows,
  //    smaller ones gather (and quantise) per aligned row; zero the combine
  //    buffer
  if (phase == 2) {
    // (written by the first call)
  } else if (L.large && fp8) {
    if (launch_quant_scatter(static_cast<const __nv_bfloat16*>(a->x), T, H, k, inv_slot, counts,
                             offsets, E, ctrl, static_cast<uint8_t*>(xs), acc, acc_elems,
                             dev.num_sms, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else if (launch_gather_x(static_cast<const __nv_bfloat16*>(a->x), H, sorted, ctrl,
                             static_cast<int>(P), k, xs, fp8, acc, acc_elems, L.pad_max,
                             dev.num_sms, s) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }

  // TMA descriptors
  CUtensorMap tm_w13, tm_xs, tm_xs64, tm_w2, tm_h, tm_h64, tm_rows;
  const bool bf16 = !fp8;
  const void* hb = fp8 ? static_cast<const void*>(hq) : static_cast<const void*>(h);
  if (!make_tmap(&tm_w13, a->w13, bf16, H, static_cast<uint64_t>(E) * 2 * I, 128) ||
      !make_tmap(&tm_xs, xs, bf16, H, L.pad_max, 16) ||
      !make_tmap(&tm_xs64, xs, bf16, H, L.pad_max, 64) ||
      !make_tmap(&tm_w2, a->w2, bf16, I, static_cast<uint64_t>(E) * H, 128) ||
      !make_tmap(&tm_h, hb, bf16, I, L.pad_max, 16) ||
      !make_tmap(&tm_h64, hb, bf16, I, L.pad_max, 64))
    return MOE_ERR_CUDA;
  // bf16 rows per pair (the down GEMM's TMA stores); else a stand-in
  if (L.combine_rows ? !make_tmap(&tm_rows, pair_rows, true, H, L.pad_max, 16) : false)
    return MOE_ERR_CUDA;
  if (!L.combine_rows) tm_rows = tm_h;

  const int k_elems = fp8 ? 128 : 64;
  const long long max_tiles = std::min<long long>(L.max_mtiles, (L.pad_max + bn_max - 1) / bn_max + touched);
  const int ctas = std::min(L.ctas, dev.num_sms);

  // 4. gate/up GEMM + SiLU*up epilogue
  GemmParams g1{};
  const int bn1 = wide1 ? kWideRows : bn_max;
  g1.mtiles = wide1 ? mtiles_w : mtiles;
  g1.wide = wide1 ? 1 : 0;
  g1.ctrl = ctrl;
  g1.nb_count = I / 128;
  g1.k_steps = H / k_elems;
  g1.k_elems = k_elems;
  g1.bn_max = bn1;
  g1.stage_smem = static_cast<unsigned>(gemm_stage_smem(true));
  g1.acc_stride = 2 * bn1;
  g1.num_acc = (4 * bn1 <= 512) ? 2 : 1;
  g1.tmem_cols = next_pow2(g1.acc_stride * g1.num_acc);
  g1.rows_per_expert = 2 * I;
  g1.wblock_rows = 128;
  g1.up_offset = I;
  g1.sorted_ids = sorted;
  g1.P = static_cast<int>(P);
  g1.top_k = k;
  g1.w_scale = fp8 ? a->w13_scale : nullptr;
  g1.act_scale_sel = fp8 ? 1 : 0;
  g1.sorted_w = sorted_w;
  g1.h_out = h;
  g1.ldh = I;
  g1.tile_cnt = tile_cnt;
  g1.part = part;
  // A weight block serves one row tile when an expert's rows fit one tile:
  // streamed once, evict-first, the whole (tile, K step) space split evenly.
  // From half a tile per expert on average, busier experts split into two
  // tiles whose weight blocks are better read once and reused from L2 (whole
  // tiles round-robin, evict-last): measured at 128 rows per expert on
  // average, gate/up 127 -> 107 us (E=128, H=2048, I=768, 2048 tokens, k=8).
  g1.weights_evict_first = (P + touched - 1) / touched <= bn1 / 2 ? 1 : 0;
  g1.pair_out = nullptr;
  g1.timeout_ns = (a->debug_flags & MOE_DEBUG_FORCE_TIMEOUT) ? MOE_DEBUG_TIMEOUT_MS * 1000000ull
                                                             : kWaitLimitNs;
  g1.debug = a->debug_flags;
  unsigned long long* trace = reinterpret_cast<unsigned long long*>(ws + L.trace);
  g1.trace = (a->debug_flags & MOE_DEBUG_TRACE) ? trace : nullptr;
  const long long max_tiles1 =
      wide1 ? std::min<long long>(L.max_mtiles, (L.pad_max + bn1 - 1) / bn1 + touched) : max_tiles;
  const long long work1 = max_tiles1 * g1.nb_count * g1.k_steps;
  const int grid1 = static_cast<int>(std::max<long long>(1, std::min<long long>(ctas, work1)));
  if (events && cudaEventRecord(events[3], stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (phase == 2) {
    // (the gate/up GEMM ran in the first call)
  } else if (pair1) {
    GemmParams gp = g1;
    gp.nb_count = I / 256;  // units: (wide row tile, pair of weight blocks)
    const long long units = max_tiles1 * gp.nb_count;
    const int max_clusters =
        static_cast<int>(std::max<long long>(1, std::min<long long>(ctas / 2, units)));
    if (launch_gemm_pair(gp, tm_w13, tm_xs, tm_xs64, max_clusters, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else if (launch_gemm(bf16, true, tok_m1, false, g1, tm_w13, tm_xs, tm_xs64, tm_rows, grid1,
                         s) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }

  if (phase == 1) return MOE_OK;  // max |h| of this call is in the workspace

  // 5. dynamic scale of h and its E4M3 codes
  if (events && cudaEventRecord(events[4], stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (fp8 && launch_quant_h(static_cast<const float*>(h), I, ctrl, hq, L.pad_max, dev.num_sms,
                            s) != cudaSuccess)
    return MOE_ERR_CUDA;

  // 6. down GEMM + weighted scatter-combine (tiles cut across CTAs add into
  //    the combine buffer like any other partial sum)
  if (events && cudaEventRecord(events[5], stream) != cudaSuccess) return MOE_ERR_CUDA;
  GemmParams g2 = g1;
  g2.mtiles = mtiles;  // 128-row tiles
  g2.wide = 0;
  g2.bn_max = bn_max;
  // unswapped: two 128-row weight blocks per tile against one token tile
  const bool pair2 = tok_m2 && H % 256 == 0;
  g2.nb_count = H / (pair2 ? 256 : 128);
  g2.k_steps = I / k_elems;
  g2.stage_smem = static_cast<unsigned>(gemm_stage_smem(false));
  g2.acc_stride = pair2 ? 2 * bn_max : bn_max;
  g2.num_acc = 2;
  g2.tmem_cols = next_pow2(2 * g2.acc_stride);
  g2.rows_per_expert = H;
  g2.wblock_rows = pair2 ? 256 : 128;
  g2.up_offset = pair2 ? 128 : 0;
  g2.w_scale = fp8 ? a->w2_scale : nullptr;
  g2.act_scale_sel = fp8 ? 2 : 0;
  g2.h_out = nullptr;
  g2.acc_out = acc;
  g2.ldo = H;
  g2.tile_cnt = nullptr;
  g2.part = nullptr;
  g2.pair_out = L.combine_rows ? pair_rows : nullptr;
  g2.trace = (a->debug_flags & MOE_DEBUG_TRACE) ? trace + MOE_TRACE_MAX_CTAS * 4 : nullptr;
  const long long work2 = max_tiles * g2.nb_count * g2.k_steps;
  const int grid2 = static_cast<int>(std::max<long long>(1, std::min<long long>(ctas, work2)));
  if (launch_gemm(bf16, false, tok_m2, pair2, g2, tm_w2, tm_h, tm_h64, tm_rows, grid2, s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;

  // 7. fp32 combine buffer -> bf16 output, or the sum of each token's k rows
  if (events && cudaEventRecord(events[6], stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (L.combine_rows) {
    if (launch_combine_rows(pair_rows, inv_slot, T, k, H, static_cast<__nv_bfloat16*>(a->out),
                            dev.num_sms, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else if (launch_finalize(acc, static_cast<__nv_bfloat16*>(a->out),
                             static_cast<long long>(T) * H, dev.num_sms, s) != cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  if (events && cudaEventRecord(events[7], stream) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_fused_forward(const moe_fused_args* a, void* workspace, size_t workspace_bytes,
                               moe_stream_t stream) {
  return fused_forward_impl(a, workspace, workspace_bytes, stream, nullptr);
}

moe_status_t moe_fused_forward_gate_up(const moe_fused_args* a, void* workspace,
                                       size_t workspace_bytes, moe_stream_t stream) {
  return fused_forward_impl(a, workspace, workspace_bytes, stream, nullptr, 1);
}

moe_status_t moe_fused_forward_down(const moe_fused_args* a, void* workspace,
                                    size_t workspace_bytes, moe_stream_t stream) {
  return fused_forward_impl(a, workspace, workspace_bytes, stream, nullptr, 2);
}

size_t moe_fused_h_amax_offset(void) { return offsetof(Ctrl, amax_h); }

size_t moe_fused_trace_offset(int T, int H, int I, int E, int top_k, moe_dtype_t dtype) {
  if (moe_fused_workspace_size(T, H, I, E, top_k, dtype) == 0) return 0;
  return make_layout(T, H, I, E, top_k, dtype == MOE_DT_FP8_E4M3).trace;
}

int moe_fused_launch_count(int T, int H, int I, int E, int top_k, moe_dtype_t dtype) {
  if (moe_fused_workspace_size(T, H, I, E, top_k, dtype) == 0) return -1;
  if (H % 128 != 0 || I % 128 != 0) return -1;
  if (T == 0) return 0;
  const bool fp8 = dtype == MOE_DT_FP8_E4M3;
  const Layout L = make_layout(T, H, I, E, top_k, fp8);
  int n = 0;
  if (small_front(T, H, E, top_k)) {
    n += 1;                          // router + alignment
  } else {
    n += 2 + (L.large ? 1 : 0);      // router, (chunk histograms), alignment
  }
  n += 1;                            // gather of x, or per-token quantise + scatter
  n += 1;                            // gate/up GEMM
  n += fp8 ? 1 : 0;                  // quantisation of h
  n += 1;                            // down GEMM
  n += 1;                            // finalize or row combine
  return n;
}

moe_status_t moe_fused_forward_timed(const moe_fused_args* a, void* workspace,
                                     size_t workspace_bytes, moe_stream_t stream,
                                     void* const* events, int n_events) {
  if (!events || n_events < MOE_TIMED_EVENTS) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < MOE_TIMED_EVENTS; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return fused_forward_impl(a, workspace, workspace_bytes, stream,
                            reinterpret_cast<cudaEvent_t const*>(events));
}

moe_status_t moe_check_status(const void* workspace, moe_stream_t stream) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  int err = 0;
  if (cudaMemcpyAsync(&err, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (err & kDevErrTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  if (err & kDevErrRange) return MOE_ERR_DEVICE_RANGE;
  return MOE_OK;
}

}  // extern "C"
