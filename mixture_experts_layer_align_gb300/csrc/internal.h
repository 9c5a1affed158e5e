// Internal (non-exported) declarations shared by the library's translation
// units: the workspace control block, kernel parameter blocks and launchers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_gb300.h"

namespace moe {

// Status bits of Ctrl::err.
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrRange = 2;

// Rows of one alignment block inside the fused path: the tcgen05 MMA with
// M = 128 takes N in multiples of 16, so each expert's token segment is
// padded to 16 rows.
constexpr int kAlignBlock = 16;

// Remembers (per host thread) the last failing CUDA call for
// moe_last_error_detail(); returns `e` unchanged.
void note_cuda_error(int code, const char* what, const char* where);
inline cudaError_t checked(cudaError_t e, const char* where) {
  if (e != cudaSuccess) note_cuda_error(static_cast<int>(e), cudaGetErrorName(e), where);
  return e;
}

// Launch with programmatic stream serialisation: the kernel may start while
// its predecessor drains; every kernel of this library calls pdl_wait()
// before touching global memory, so stream order is kept for the data.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return checked(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...), "kernel launch");
}

// Per-call control words, at the start of the workspace.
struct Ctrl {
  int err;          // kDevErr* bits set by device code
  unsigned amax_h;  // bits of max |h| (non-negative floats order like uints)
  float s_x;        // activation scale of x
  float s_h;        // activation scale of h
  int num_padded;   // rows of the aligned (sorted, padded) pair list
  int num_mtiles;   // entries of the GEMM row-tile list
  int max_tile_rows;  // rows of the largest row tile
  int num_mtiles_w;     // the same for the list of wide (256-row) tiles, when written
  int max_tile_rows_w;
  // grid-wide arrival counters of the single-kernel small-batch path (zeroed
  // by that kernel before its first grid synchronisation)
  unsigned bar[4];
  int pad[3];
};
static_assert(sizeof(Ctrl) == 64, "Ctrl layout");

// ------------------------------------------------------------ routing / align
constexpr int kRouteWarps = 8;  // tokens per router CTA (one warp per token)

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                              float* wts, const __nv_bfloat16* x, int H, float* amax_partials,
                              Ctrl* ctrl, int* zero_ints, int n_zero, cudaStream_t st);
inline int route_grid(int T) { return (T + kRouteWarps - 1) / kRouteWarps; }

struct AlignParams {
  const int32_t* ids;
  int P, E, bm, chunk;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_ids;
  int32_t* tile_expert;  // may be null
  int32_t* num_padded;   // may be null
  // per-chunk expert histograms [gridDim][E] from align_hist (large batches);
  // null: every CTA counts all pairs itself
  const int32_t* chunk_hist;
  // fused-path extras (null when unused)
  const float* wts;      // [P] router weights (read when sorted_w is set)
  float* sorted_w;       // router weight of each aligned row, 0 for padding
  int32_t* inv_slot;     // [P] aligned row of each pair, or null
  int4* mtiles;          // GEMM row tiles {expert, first row, rows, 0}
  int bn_max;            // max rows of one row tile
  int4* mtiles_w;        // second list of tiles of up to 256 rows, or null
  Ctrl* ctrl;
  const float* amax_partials;
  int n_partials;
};
cudaError_t launch_align(const AlignParams& p, cudaStream_t st);
int align_chunk();
// Router + alignment in one CTA for small batches (decode).  Used when
// T <= kSmallMaxTokens, T*k <= kSmallMaxPairs, E <= kSmallMaxExperts and
// T*H <= kSmallMaxXElems (beyond 16 tokens the separate router and alignment
// kernels were measured faster: fine-grained T=256 175 -> 136 us per call).
constexpr int kSmallMaxTokens = 16;
constexpr int kSmallMaxPairs = 2048;
// Above this many pairs: two-pass alignment (per-chunk histograms) and x
// quantised once per token before a byte-copy gather.
constexpr long long kLargePairs = 4096;
constexpr int kSmallMaxExperts = 256;
constexpr long long kSmallMaxXElems = 1ll << 19;
struct SmallFrontParams {
  const float* logits;
  int T, E, k, renorm;
  int32_t* ids;
  float* wts;
  const __nv_bfloat16* x;  // null: no activation scale (bf16 path)
  int H;
  Ctrl* ctrl;
  int* zero_ints;
  int n_zero;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_ids;
  float* sorted_w;  // router weight of each aligned row, 0 for padding
  int4* mtiles;
  int bn_max;
  int4* mtiles_w;   // second list of tiles of up to 256 rows, or null
};
cudaError_t launch_route_align_small(const SmallFrontParams& p, cudaStream_t st);

// First pass of the two-pass alignment: expert histogram of each chunk of
// align_chunk() pairs into hist[chunk][E].
cudaError_t launch_align_hist(const int32_t* ids, int P, int E, int32_t* hist, cudaStream_t st);
// Large FP8 batches: each token row of x quantised once with ctrl->s_x and
// written to its k aligned rows of xs (inv_slot[pair] = aligned row); padding
// rows of every segment zeroed; the fp32 combine buffer zeroed (acc_elems may
// be 0).
cudaError_t launch_quant_scatter(const __nv_bfloat16* x, int T, int H, int k,
                                 const int32_t* inv_slot, const int32_t* counts,
                                 const int32_t* offsets, int E, const Ctrl* ctrl, uint8_t* xs,
                                 float* acc, long long acc_elems, int num_sms, cudaStream_t st);

// Gather the routed rows of x into aligned order (E4M3 with s_x, or bf16), zero
// the fp32 combine buffer.
cudaError_t launch_gather_x(const __nv_bfloat16* x, int H, const int32_t* sorted_ids,
                            const Ctrl* ctrl, int P, int k, void* xs, bool fp8, float* acc,
                            long long acc_elems, int max_rows, int num_sms, cudaStream_t st);
// h (fp32) -> E4M3 with s_h = amax_h / 448 (stored into ctrl->s_h).
cudaError_t launch_quant_h(const float* h, int I, Ctrl* ctrl, uint8_t* hq, int max_rows,
                           int num_sms, cudaStream_t st);
// fp32 combine buffer -> bf16 output.
cudaError_t launch_finalize(const float* acc, __nv_bfloat16* out, long long n, int num_sms,
                            cudaStream_t st);
// Standalone activation quantisation.
cudaError_t launch_quantize_e4m3(const __nv_bfloat16* x, long long n, uint8_t* xq, float* scale,
                                 float* partials, int n_partials, cudaStream_t st);

// ------------------------------------------------------------ inverse RoPE + FP8
constexpr int kRopeMaxCtas = 1024;
int rope_grid(long long T, int NH, int D, int num_sms);
// partials: (grid * (NH + 1)) floats of scratch; ctrl->err gets the status.
cudaError_t launch_inv_rope_quant(const __nv_bfloat16* x, const int32_t* pos, const float* cos_t,
                                  const float* sin_t, int T, int NH, int D, int max_pos,
                                  uint8_t* codes, float* scales, Ctrl* ctrl, float* partials,
                                  int num_sms, cudaStream_t st);

// ------------------------------------------------------------ grouped GEMM
struct GemmParams {
  // Row tiles {expert, first row, rows | (tiles of this expert << 12), index of
  // the expert's first tile}, written by the alignment kernel.
  const int4* mtiles;
  Ctrl* ctrl;
  int wide;             // 1: the wide tile list (counts num_mtiles_w / max_tile_rows_w)
  int nb_count;         // 128-row weight blocks per expert (I/128 or H/128)
  int k_steps;          // K / (128 bytes of K)
  int k_elems;          // elements of K per step: 128 (E4M3) or 64 (bf16)
  int bn_max;           // max tokens (MMA N) per row tile
  unsigned stage_smem;  // shared-memory bytes for the pipeline stages
  int acc_stride;       // TMEM columns per accumulator buffer
  int num_acc;          // accumulator buffers (1 or 2)
  int tmem_cols;        // allocated TMEM columns (power of two >= 32)
  int rows_per_expert;  // 2I (gate/up) or H (down)
  int wblock_rows;      // weight rows between consecutive tile blocks: 128, or 256 for pairs
  int up_offset;        // second weight block of a stage: I (gate/up) or 128 (pairs)
  const int32_t* sorted_ids;
  int P, top_k;
  const float* w_scale;  // [E] per-expert weight scale (FP8) or null
  int act_scale_sel;     // 1: s_x, 2: s_h (FP8); 0: none
  const float* sorted_w;  // router weight of each aligned row (0 for padding)
  void* h_out;           // gate/up: [rows, I], fp32 (FP8 path) or bf16 (bf16 path)
  int ldh;
  float* acc_out;        // down, combine by reduction: [T, H] fp32
  int ldo;
  // down, combine by rows (large batches): y * s * topk_weight as bf16 at the
  // pair's aligned row of [rows, H] (the tile's own rows; tokens in M: TMA
  // stores through the tensor map passed to the kernel); a separate kernel
  // sums each token's k rows.  Null selects the bulk reductions into acc_out.
  __nv_bfloat16* pair_out;
  // gate/up tiles split across CTAs: per-tile arrival counters (zeroed by the
  // router kernel) and two partial-accumulator slots per CTA
  int* tile_cnt;
  float* part;
  int weights_evict_first;  // 1: each weight block is used by one row tile (decode)
  unsigned long long timeout_ns;
  int debug;
  unsigned long long* trace;  // [MOE_TRACE_MAX_CTAS][4] stamps or null
};

// Sum of the k weighted expert rows of every token: out[t] = sum_j
// rows[inv_slot[t*k+j]] (aligned row of each pair; fp32 accumulation in slot
// order, bf16 result).
cudaError_t launch_combine_rows(const __nv_bfloat16* rows, const int32_t* inv_slot, int T, int k,
                                int H, __nv_bfloat16* out, int num_sms, cudaStream_t st);

// The down projection combines through bf16 rows per pair (and a separate
// sum) instead of fp32 reductions into [T, H] when P x H exceeds this.
constexpr long long kCombineRowsElems = 8ll << 20;
inline bool combine_by_rows(long long P, long long H) { return P * H > kCombineRowsElems; }

// Widest row tile of any GEMM (wide gate/up tiles).
constexpr int kWideRows = 256;

// Partial-accumulator slot (gate and up, bn_max columns x 128 rows, fp32).
__host__ __device__ inline size_t gemm_part_slot_floats(int bn_max) { return static_cast<size_t>(2) * bn_max * 128; }

// warp 0 TMA, warp 1 MMA, warps 2..9 epilogue (two warps per TMEM lane
// quarter, each taking every other 16-column chunk of a tile)
constexpr int kGemmEpiWarps = 8;
constexpr int kGemmThreads = 64 + 32 * kGemmEpiWarps;
// Shared-memory bytes left for the pipeline stages (the kernel picks its
// depth from the largest row tile of the call).
size_t gemm_stage_smem(bool swiglu);
// tmb / tmb64: the token operand with 16-row and 64-row boxes.  tok_m: tokens
// in the MMA M slot (the unswapped placement; row tiles of up to 128 rows).
// pair: the unswapped down GEMM with two weight blocks per tile (H % 256 == 0).
// tmo: bf16 rows per pair [rows, H] with 64-column x 16-row boxes (128-byte
// swizzle), the target of the down GEMM's stores with tokens in M and
// p.pair_out set; any valid map otherwise (unused).
cudaError_t launch_gemm(bool bf16, bool swiglu, bool tok_m, bool pair, const GemmParams& p,
                        const CUtensorMap& tma, const CUtensorMap& tmb, const CUtensorMap& tmb64,
                        const CUtensorMap& tmo, int grid, cudaStream_t st);
// Gate/up GEMM of wide row tiles (256 tokens) on SM pairs (cluster of two,
// tcgen05 cta_group::2): E4M3, weights in M, I % 256 == 0, whole tiles;
// p.mtiles is the wide tile list and p.nb_count = I / 256.  At most
// `max_clusters` clusters (the units of the call).
cudaError_t launch_gemm_pair(const GemmParams& p, const CUtensorMap& tma, const CUtensorMap& tmb,
                             const CUtensorMap& tmb64, int max_clusters, cudaStream_t st);
// Row-tile width of the unswapped placement (the token tile fills M = 128).
constexpr int kTokMRows = 128;

// ------------------------------------------------------------ small batches, one kernel
// The whole layer for small batches in one cooperative persistent kernel (one
// CTA per SM): routing, alignment, gather, gate/up GEMM + SiLU*up, h
// quantisation, down GEMM + combine and the bf16 output, with grid-wide
// arrival counters between the phases.  Used on request (MOE_FLAG_ONE_KERNEL)
// when T*k <= kFusedMaxPairs, E <= kFusedMaxExperts and the fp32 combine
// buffer is used.
constexpr int kFusedMaxPairs = 2048;
constexpr int kFusedMaxExperts = 256;
constexpr int kFusedThreads = kGemmThreads;
struct FusedParams {
  const float* logits;
  const __nv_bfloat16* x;
  int T, H, I, E, k, renorm;
  const float* w13_scale;  // [E] (FP8) or null (bf16)
  const float* w2_scale;
  __nv_bfloat16* out;      // [T, H]
  int32_t* ids;            // [T*k] router outputs (caller's arrays or workspace)
  float* wts;
  int32_t* counts_out;     // [E] or null
  Ctrl* ctrl;
  float* amax_part;        // [gridDim] partial max |x| per CTA
  int32_t* sorted_ids;     // aligned rows: pair id (T*k for padding)
  float* sorted_w;         // aligned rows: router weight (0 for padding)
  void* xs;                // aligned rows of x: E4M3 or bf16 [rows][H]
  void* h;                 // [rows][I]: fp32 (FP8) or bf16
  uint8_t* hq;             // [rows][I] E4M3 (FP8)
  float* acc;              // [T, H] fp32 combine
  float* part;             // split gate/up tiles: two slots per CTA
  int* tile_cnt;           // per gate/up tile arrival counters
  int n_tile_cnt;
  unsigned stage_smem;     // dynamic shared memory for the pipeline stages
  unsigned long long timeout_ns;
  int debug;
  unsigned long long* trace;  // [2][MOE_TRACE_MAX_CTAS][4] or null
};
// tm_*: w13 (128-row boxes), x rows (16/64-row boxes), w2, h codes (16/64).
cudaError_t launch_fused_small(const FusedParams& p, const CUtensorMap& tm_w13,
                               const CUtensorMap& tm_xs, const CUtensorMap& tm_xs64,
                               const CUtensorMap& tm_w2, const CUtensorMap& tm_h,
                               const CUtensorMap& tm_h64, int grid, cudaStream_t st);
// Whether the device can run it (cooperative launch, one CTA per SM fits).
bool fused_small_supported(int device);
}  // namespace moe
