/*
 * moe_gb300.h — C ABI of the GB300 (sm_103a) fused Mixture-of-Experts layer.
 *
 * Source of the operation: "Amazon SageMaker AI 上的 Mixture-of-Experts 内核工程
 * 优化" (English original page).  Its Introduction defines the fused MoE layer
 * as token routing, data shuffling and the expert network computation merged
 * into one batched GPU operation; its section "Backend routing for FP8 tensor
 * quantization" adds FP8 tensor scaling and expert aggregation to the same
 * single pass; its section "Swap-AB for WGMMA utilization" (with the digest
 * page's formula B^T[N,K] x A^T[K,M] -> C^T[N,M]) gives the operand swap that
 * puts the large expert dimension in the MMA's M slot when few tokens reach an
 * expert.  The pages leave the router, the expert MLP and the scale granularity
 * open; this library reads them as:
 *   router   softmax over E fp32 logits, top-k on the raw logits with ties to
 *            the lower expert index, optional renormalisation of the k weights;
 *   expert   SwiGLU: w13 rows [0,I) gate, [I,2I) up; h = SiLU(gate) * up;
 *            y = w2 h; no bias;
 *   FP8      E4M3 weights with one fp32 scale per expert per tensor; dynamic
 *            per-tensor E4M3 activations, s = amax / 448 (1 if amax is 0),
 *            code = E4M3_rne_satfinite(fp32(v) / s);
 *   combine  out[t] = sum_j w[t,j] * y[t,j], accumulated in fp32, stored bf16.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *     row-major, 16-byte aligned.  The library allocates nothing and keeps no
 *     state between calls other than lazily cached per-device properties.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Nothing synchronises the host.
 *   - Argument errors are detected on the host before anything is enqueued and
 *     are returned synchronously with no side effect.  CUDA launch errors
 *     return MOE_ERR_CUDA.  Device-side faults of the schedule (a bounded wait
 *     that ran out, an out-of-range expert id) are recorded in the workspace's
 *     status word; moe_check_status() reads it.
 *   - All sizes are runtime values: one binary serves every shape (no per-shape
 *     compilation).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null pointer, bad size, k > E, misalignment ... */
  MOE_ERR_UNSUPPORTED = 2,    /* shape outside what the kernels tile (H or I % 128) */
  MOE_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime/driver call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait ran out (status word) */
  MOE_ERR_DEVICE_RANGE = 6    /* a device kernel met an out-of-range expert id */
} moe_status_t;

typedef enum { MOE_DT_BF16 = 0, MOE_DT_FP8_E4M3 = 1 } moe_dtype_t;

/*
 * Router (token routing, page Introduction).
 *   logits   fp32 [T, E]
 *   topk_ids int32 [T, top_k]  out: selected experts, slot order = (logit desc, index asc)
 *   topk_w   fp32 [T, top_k]   out: softmax probability of each selected expert,
 *                              divided by the sum over the k selected when renormalize != 0
 * Requires 1 <= top_k <= E <= 1024, T >= 0 (T == 0 enqueues nothing), finite logits.
 */
moe_status_t moe_route_topk(const float* logits, int T, int E, int top_k, int renormalize,
                            int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/*
 * Alignment by expert (data shuffling, page Introduction; the "fragmented
 * token arrays" of section "Backend routing for FP8 tensor quantization").
 * Pair p = t*top_k + j goes to expert topk_ids[p].
 *   counts      int32 [E]      out: pairs per expert
 *   offsets     int32 [E+1]    out: exclusive prefix sum of counts rounded up to block_m
 *   sorted_ids  int32 [T*top_k + E*(block_m-1)]
 *                              out: per expert segment, its pair ids ascending, then the
 *                              sentinel T*top_k up to the padded size; entries past
 *                              offsets[E] are left untouched
 *   tile_expert int32 [(T*top_k + E*(block_m-1)) / block_m]
 *                              out: owning expert of each block_m-row block (may be NULL)
 *   num_padded  int32 [1]      out: offsets[E]
 * Requires 1 <= E <= 1024, 1 <= block_m <= 256, T*top_k < 2^31 - E*block_m.
 * Ids outside [0, E) are skipped (not placed, not counted).
 */
moe_status_t moe_align_by_expert(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                                 int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                                 int32_t* tile_expert, int32_t* num_padded, moe_stream_t stream);

/*
 * Dynamic per-tensor activation quantisation (FP8 tensor scaling, section
 * "Backend routing for FP8 tensor quantization").
 *   x      bf16 [T, H]
 *   x_q    uint8 [T, H]  out: E4M3 codes of fp32(x) / s
 *   scale  fp32 [1]      out: s = amax|x| / 448 (1 when x is all zero)
 * Requires H % 16 == 0.  `scratch` is a caller buffer of at least
 * moe_quantize_scratch_size(T, H) bytes.
 */
size_t moe_quantize_scratch_size(int T, int H);
moe_status_t moe_quantize_e4m3(const void* x, int T, int H, uint8_t* x_q, float* scale,
                               void* scratch, size_t scratch_bytes, moe_stream_t stream);

/*
 * Same operation and results as moe_quantize_e4m3, without the caller scratch
 * buffer: the scratch (one fp32 partial maximum per amax CTA, at most
 * MOE_NOALLOC_MAX_PARTIALS of them, 4 KB) lives in a static device array of
 * the library.  The pages have no counterpart of this entry point; it exists
 * for callers that cannot allocate device memory where they call it (another
 * component owns every allocation, or the calling thread must not take
 * cudaMalloc's implicit synchronisation).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call in a CUDA context looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it under
 *     the context's unique id (cuCtxGetId); a call in another context (after
 *     cudaDeviceReset, or with another driver context current) looks it up
 *     again.  Make the first call on a device before any stream capture.
 *   - The array is shared by every call on the device and keeps the last
 *     call's contents; calls that overlap on the GPU (other streams, or other
 *     host threads) race on it and must be serialised by the caller.
 *   - Every T*H fits (the amax kernel strides over the tensor, using at most
 *     MOE_NOALLOC_MAX_PARTIALS CTAs); T, H and pointers are checked as in
 *     moe_quantize_e4m3 (MOE_ERR_INVALID_ARG), and a partial count beyond the
 *     array would return MOE_ERR_UNSUPPORTED.
 */
#define MOE_NOALLOC_MAX_PARTIALS 1024
moe_status_t moe_quantize_e4m3_noalloc(const void* x, int T, int H, uint8_t* x_q, float* scale,
                                       moe_stream_t stream);

/*
 * Inverse rotary position embedding + per-head FP8 quantisation (the fused
 * kernel named in section "Triton JIT recompilation elimination", whose
 * arithmetic the pages leave open; read here as):
 *   y[2i]   = x[2i] c + x[2i+1] s,   y[2i+1] = x[2i+1] c - x[2i] s
 *     (RoFormer's pair rotation by the negated angle; c, s = cos_tab/sin_tab
 *     [positions[t]][i]; each product rounded to fp32, then the sum),
 *   scales[h] = amax over tokens and dims of |y[., h, .]| / 448 (1 if 0),
 *   codes = E4M3_rne_satfinite(y / scales[h]) (IEEE fp32 division).
 *   x          bf16 [T, NH, D]
 *   positions  int32 [T], each in [0, max_pos)
 *   cos_tab    fp32 [max_pos, D/2]; sin_tab fp32 [max_pos, D/2]
 *   codes      uint8 [T, NH, D]  out
 *   scales     fp32 [NH]         out
 *   scratch    moe_inv_rope_scratch_size(T, NH, D) bytes, 256-byte aligned; its
 *              first word is the status word moe_check_status() reads
 *              (MOE_ERR_DEVICE_RANGE: a position outside the tables, treated
 *              as 0)
 * Requires T >= 0 (0 enqueues nothing), 1 <= NH <= 4096, D in {8, 16, 32, 64,
 * 128, 256}, max_pos >= 1, 16-byte aligned x / cos_tab / sin_tab, 8-byte
 * aligned codes; T*NH*D >= 2^31 returns MOE_ERR_UNSUPPORTED.  Enqueues on
 * `stream` one cooperative kernel (small inputs), or a memset of NH + 1 words
 * of the scratch and two kernels (large inputs); all sizes are runtime values.
 */
size_t moe_inv_rope_scratch_size(int T, int NH, int D);
moe_status_t moe_inv_rope_quant_per_head(const void* x, const int32_t* positions,
                                         const float* cos_tab, const float* sin_tab, int T,
                                         int NH, int D, int max_pos, uint8_t* codes,
                                         float* scales, void* scratch, size_t scratch_bytes,
                                         moe_stream_t stream);

/* Arguments of the fused layer forward. */
typedef struct {
  const void* x;             /* bf16 [T, H] */
  const float* router_logits;/* fp32 [T, E] */
  const void* w13;           /* [E, 2I, H]: gate rows then up rows, H contiguous.
                                E4M3 codes (FP8) or bf16 */
  const void* w2;            /* [E, H, I], I contiguous; same element type as w13 */
  const float* w13_scale;    /* fp32 [E]; required for FP8, must be NULL for BF16 */
  const float* w2_scale;     /* fp32 [E]; required for FP8, must be NULL for BF16 */
  moe_dtype_t weight_dtype;
  int T, H, I, E, top_k, renormalize;
  void* out;                 /* bf16 [T, H] */
  int32_t* topk_ids_out;     /* optional int32 [T, top_k] (NULL: not returned) */
  float* topk_w_out;         /* optional fp32 [T, top_k] */
  int32_t* counts_out;       /* optional int32 [E]: pairs routed to each expert */
  int debug_flags;           /* 0 in normal use; see MOE_DEBUG_* */
} moe_fused_args;

/* Test hook: make the expert-GEMM kernels' MMA warp wait on a barrier that
 * nothing ever arrives on, so the bounded wait runs out (about
 * MOE_DEBUG_TIMEOUT_MS) and the call reports MOE_ERR_DEVICE_TIMEOUT through
 * moe_check_status() while the CUDA context stays usable. */
#define MOE_DEBUG_FORCE_TIMEOUT 0x1
#define MOE_DEBUG_TIMEOUT_MS 200

/* Diagnostic: the two expert-GEMM kernels record, per CTA, four %globaltimer
 * stamps (ns): kernel entry, inputs ready, first weight tile landed, exit.
 * They go to uint64 [2][MOE_TRACE_MAX_CTAS][4] at byte offset
 * moe_fused_trace_offset() of the workspace (gate/up kernel first); rows of
 * CTAs that are not launched keep their previous contents (zero the region
 * first to tell them apart).  On SM pairs (wide FP8 gate/up tiles) the third
 * stamp of the second CTA of a pair is its first accumulator ready (that
 * CTA's stages complete on the first CTA's barriers).  With
 * MOE_FLAG_ONE_KERNEL the single kernel records [0][cta] = entry, token rows
 * ready, first gate/up stage, gate/up epilogue done and [1][cta] = h written
 * everywhere, h codes ready, first down stage, exit. */
#define MOE_DEBUG_TRACE 0x2
/* Operand placement (section "Swap-AB for WGMMA utilization").  By default
 * the gate/up GEMM puts the expert's weight rows in the MMA's M slot (the
 * swap) and the down GEMM does so when I > 2048; with I <= 2048 the down GEMM
 * puts the tokens (128-row tiles) in M.  MOE_FLAG_TOKENS_IN_M forces tokens
 * in M and MOE_FLAG_WEIGHTS_IN_M forces weights in M for both GEMMs (the
 * ablation of the swap); both together are MOE_ERR_INVALID_ARG.  Results are
 * the same within fp32 summation order. */
#define MOE_FLAG_TOKENS_IN_M 0x4
#define MOE_FLAG_WEIGHTS_IN_M 0x8
/* FP8 gate/up tiles of 256 tokens (I % 256 == 0 and experts averaging at
 * least 128 routed rows: prefill) run on SM pairs by default: a cluster of two
 * CTAs issues tcgen05 MMAs with M = 256 (cta_group::2), each SM holding its 128
 * weight rows and half of the token rows.  This flag runs the gate/up GEMM on
 * one SM per tile instead (ablation): 256-token tiles when experts average more
 * than 256 rows, else 128-token tiles.  Results are the same within fp32
 * summation order. */
#define MOE_FLAG_NO_SM_PAIRS 0x10
/* Small batches (T*top_k <= 2048, E <= 256): run the whole layer as one
 * cooperative persistent kernel instead of the kernel sequence (one CTA per
 * SM; its CTAs wait on one another through grid-wide counters, so it needs
 * every SM of the device at once; not with MOE_FLAG_TOKENS_IN_M).  Results
 * are the same within fp32 summation order; the sequence is the default
 * because it was measured as fast or faster on every decode workload. */
#define MOE_FLAG_ONE_KERNEL 0x20
#define MOE_TRACE_MAX_CTAS 256
size_t moe_fused_trace_offset(int T, int H, int I, int E, int top_k, moe_dtype_t dtype);

/* Workspace bytes moe_fused_forward needs for these sizes (0 if invalid). */
size_t moe_fused_workspace_size(int T, int H, int I, int E, int top_k, moe_dtype_t dtype);

/* Number of kernels one moe_fused_forward call with these sizes and
 * debug_flags = 0 launches on its stream (0 for T = 0, -1 if the sizes are
 * invalid or unsupported); MOE_FLAG_ONE_KERNEL makes it 1 where it applies.
 * Host only: no CUDA call. */
int moe_fused_launch_count(int T, int H, int I, int E, int top_k, moe_dtype_t dtype);

/*
 * Fused MoE layer forward: routing -> alignment by expert -> grouped gate/up
 * GEMM with the SiLU*up epilogue -> grouped down GEMM with the top-k weighted
 * combine, FP8-scaled when weight_dtype is MOE_DT_FP8_E4M3 (page Introduction;
 * sections "Backend routing for FP8 tensor quantization" and "Swap-AB for
 * WGMMA utilization").
 * Requires 1 <= top_k <= E <= 1024, H % 128 == 0, I % 128 == 0, T >= 0,
 * a device of compute capability 10.3, workspace of moe_fused_workspace_size()
 * bytes (256-byte aligned) that no other in-flight call uses.
 * T == 0 returns MOE_OK and enqueues nothing.
 */
moe_status_t moe_fused_forward(const moe_fused_args* args, void* workspace, size_t workspace_bytes,
                               moe_stream_t stream);

/*
 * The same forward in two calls, for tensor-parallel shards (the pages
 * measure at 8-way tensor parallelism, section "Triton JIT recompilation
 * elimination").  A rank holds, per expert, the gate and up rows of its slice
 * of I in w13 and the same columns of w2 (args.I = the slice; per-expert
 * scales unchanged); routing is replicated.
 *   moe_fused_forward_gate_up: routing, alignment, the x rows, the gate/up
 *     GEMM + SiLU*up; leaves the max |h| of this rank's h as an fp32 word at
 *     byte offset moe_fused_h_amax_offset() of the workspace (device memory).
 *   moe_fused_forward_down: the E4M3 codes of h with the scale (that word) /
 *     448, the down GEMM and the top-k weighted combine into args.out (this
 *     rank's partial output).
 * Between the two the caller replaces the word by its maximum over the ranks
 * (e.g. an all-reduce MAX of that one float on the same stream), so every
 * rank quantises h with the scale of the whole tensor, and after the second
 * call sums the ranks' outputs (all-reduce SUM).  Both calls take the same
 * args and workspace, with no other use of the workspace in between, and
 * each moe_fused_forward_down follows its own moe_fused_forward_gate_up (the
 * first call leaves the routing, the tile lists and h in the workspace for the
 * second); the first call's status word and errors are as for
 * moe_fused_forward.  With bf16 weights h is not quantised and the word is
 * unused.
 */
moe_status_t moe_fused_forward_gate_up(const moe_fused_args* args, void* workspace,
                                       size_t workspace_bytes, moe_stream_t stream);
moe_status_t moe_fused_forward_down(const moe_fused_args* args, void* workspace,
                                    size_t workspace_bytes, moe_stream_t stream);
size_t moe_fused_h_amax_offset(void);

/*
 * Same operation as moe_fused_forward, with the duration of every step made
 * measurable: events[i] (a cudaEvent_t created by the caller) is recorded on
 * `stream` before step i and events[7] after the last step.  Steps: 0 routing,
 * 1 alignment, 2 gather/quantise x, 3 gate/up GEMM + SiLU*up, 4 quantise h
 * (empty for bf16), 5 down GEMM + combine, 6 bf16 output.  Small batches
 * route and align in one kernel: events[1] and events[2] are then both
 * recorded after it (step 1 is empty).  Requires
 * n_events >= MOE_TIMED_EVENTS and non-null events; otherwise as
 * moe_fused_forward.
 */
#define MOE_TIMED_EVENTS 8
moe_status_t moe_fused_forward_timed(const moe_fused_args* args, void* workspace,
                                     size_t workspace_bytes, moe_stream_t stream,
                                     void* const* events, int n_events);

/* Synchronises `stream`, reads the status word that the last call using
 * `workspace` left there, and returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT or
 * MOE_ERR_DEVICE_RANGE (MOE_ERR_CUDA if the synchronisation itself failed). */
moe_status_t moe_check_status(const void* workspace, moe_stream_t stream);

/* Static description of a status code. */
const char* moe_status_string(moe_status_t status);

/* Text naming the last failing CUDA runtime/driver call made by this library on
 * the calling host thread and its error code (after a MOE_ERR_CUDA status).
 * Thread-local storage owned by the library, valid until that thread's next
 * failing call. */
const char* moe_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
