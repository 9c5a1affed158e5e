// Inverse rotary position embedding + per-head dynamic FP8 quantisation.
//
// "Amazon SageMaker AI 上的 Mixture-of-Experts 内核工程优化" (section "Triton JIT
// recompilation elimination") names a kernel fusing rotary position embedding
// with FP8 quantisation per head, recompiled for every new number of tokens,
// and gives none of its arithmetic.  This library reads it as:
//   - RoFormer's rotation of the consecutive pairs (2i, 2i+1) of each head
//     vector, undone: y0 = x0 c + x1 s, y1 = x1 c - x0 s with c, s the cosine
//     and sine of the position's angle for pair i, taken from caller tables
//     [max_pos][D/2]; each product rounded to fp32, then the sum/difference
//     (no fused multiply-add, so every implementation gets the same y);
//   - one dynamic E4M3 scale per head over all tokens: s_h = amax|y| / 448
//     (1 when the head is zero), code = E4M3_rne_satfinite(y / s_h) with an
//     IEEE fp32 division.
// Shapes are runtime values: one binary for every T, head count and (power of
// two) head size.
//
// Two passes over x (bf16 [T][NH][D]), a group of D/8 lanes per head vector,
// 8 elements per lane (one 16-byte load of x, one 8-byte store of codes);
// per-head maxima reduce inside each group, then one shared-memory atomic per
// group.
// Small inputs (at most two rounds of two work items per warp on one CTA of
// 512 threads per SM), one cooperative launch, rope_coop_kernel: pass 1, one
// grid synchronisation, every CTA folds the per-CTA maxima itself, pass 2
// (the latency of separate launches is what small inputs pay for).
// Large inputs: a zeroed word per head, then two launches of rope_pass_kernel
// (a warp per token, eight warps per CTA, a grid of at most eight CTAs per
// SM): pass 1 adds each CTA's maxima with one global atomic max per head;
// pass 2 forms the scales in every CTA from those words and writes the codes.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

namespace cg = cooperative_groups;


__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 4 pairs of one head vector rotated by the negated angles (cos c, sin s).
__device__ __forceinline__ void rotate8(uint4 v, float4 c, float4 s, float (&y)[8]) {
  const float xs[8] = {lo16(v.x), hi16(v.x), lo16(v.y), hi16(v.y),
                       lo16(v.z), hi16(v.z), lo16(v.w), hi16(v.w)};
  const float cs[4] = {c.x, c.y, c.z, c.w};
  const float ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float x0 = xs[2 * i], x1 = xs[2 * i + 1];
    y[2 * i] = __fadd_rn(__fmul_rn(x0, cs[i]), __fmul_rn(x1, ss[i]));
    y[2 * i + 1] = __fsub_rn(__fmul_rn(x1, cs[i]), __fmul_rn(x0, ss[i]));
  }
}

constexpr int kRopeThreads = 256;  // 8 warps: 8 tokens at a time per CTA
constexpr int kRopeBatch = 4;      // head iterations whose x loads are in flight together

// Large inputs, a warp per token.  kQuant = false: the CTA's per-head maxima
// of |y| go to the call's global maxima `gmax` [NH] (max |y| bits, zeroed
// before the launch) with one atomic max per head, and a position outside the
// tables sets gmax[NH].  kQuant = true: every CTA forms the NH scales from
// gmax (CTA 0 also stores them and the status word), then writes the codes.
// The token's first kRopeBatch loads of x are issued before its position is
// read, so they overlap the position -> cos/sin chain.
template <bool kQuant>
__global__ void __launch_bounds__(kRopeThreads)
    rope_pass_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ pos,
                     const float* __restrict__ cos_t, const float* __restrict__ sin_t, int T,
                     int NH, int D, int max_pos, unsigned* __restrict__ gmax,
                     float* __restrict__ scales, uint8_t* __restrict__ codes, Ctrl* ctrl) {
  // [NH]: max|y| bits; or the scales, then [2][NH] their bracketing reciprocals
  extern __shared__ unsigned s_head[];
  __shared__ int s_bad;
  pdl_wait();
  pdl_trigger();
  for (int h = threadIdx.x; h < NH; h += blockDim.x) {
    if (kQuant) {
      const float a = __uint_as_float(__ldcg(gmax + h));
      const float sc = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
      s_head[h] = __float_as_uint(sc);
      const E4m3Div d = e4m3_div(sc);
      s_head[NH + h] = __float_as_uint(d.rlo);
      s_head[2 * NH + h] = __float_as_uint(d.rhi);
      if (blockIdx.x == 0) scales[h] = sc;
    } else {
      s_head[h] = 0u;
    }
  }
  if (threadIdx.x == 0) {
    s_bad = 0;
    if (kQuant && blockIdx.x == 0) ctrl->err = __ldcg(gmax + NH) != 0u ? kDevErrRange : 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int n8 = D >> 3;              // lanes per head vector (a power of two <= 32)
  const int lg8 = __ffs(n8) - 1;
  const int hp = 32 >> lg8;           // head vectors per warp iteration
  const int c8 = lane & (n8 - 1);
  const int hoff = lane >> lg8;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  int bad = 0;
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nwarps) {
    const size_t row0 = static_cast<size_t>(t) * NH;
    uint4 v[kRopeBatch];
#pragma unroll
    for (int u = 0; u < kRopeBatch; ++u) {
      const int h = u * hp + hoff;
      v[u] = h < NH ? __ldg(reinterpret_cast<const uint4*>(x + (row0 + h) * D + c8 * 8))
                    : make_uint4(0, 0, 0, 0);
    }
    int p = __ldg(pos + t);
    if (p < 0 || p >= max_pos) {
      bad = 1;
      p = 0;
    }
    const size_t tab = static_cast<size_t>(p) * (D / 2) + c8 * 4;
    const float4 c = __ldg(reinterpret_cast<const float4*>(cos_t + tab));
    const float4 s = __ldg(reinterpret_cast<const float4*>(sin_t + tab));
    for (int hb = 0; hb < NH; hb += hp * kRopeBatch) {
      if (hb > 0) {
#pragma unroll
        for (int u = 0; u < kRopeBatch; ++u) {
          const int h = hb + u * hp + hoff;
          v[u] = h < NH ? __ldg(reinterpret_cast<const uint4*>(x + (row0 + h) * D + c8 * 8))
                        : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < kRopeBatch; ++u) {
        const int h = hb + u * hp + hoff;
        float y[8];
        rotate8(v[u], c, s, y);
        if (kQuant) {
          if (h < NH) {
            const E4m3Div d{__uint_as_float(s_head[h]), __uint_as_float(s_head[NH + h]),
                            __uint_as_float(s_head[2 * NH + h])};
            uint2 q;
            q.x = static_cast<uint32_t>(quant2(y[0], y[1], d)) |
                  (static_cast<uint32_t>(quant2(y[2], y[3], d)) << 16);
            q.y = static_cast<uint32_t>(quant2(y[4], y[5], d)) |
                  (static_cast<uint32_t>(quant2(y[6], y[7], d)) << 16);
            *reinterpret_cast<uint2*>(codes + (row0 + h) * D + c8 * 8) = q;
          }
        } else {
          float m = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(y[j]));
          // maximum over the group of lanes of one head vector
          for (int o = n8 >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (c8 == 0 && h < NH && m > 0.f) atomicMax(&s_head[h], __float_as_uint(m));
        }
      }
    }
  }
  if (!kQuant) {
    if (bad) s_bad = 1;
    __syncthreads();
    for (int h = threadIdx.x; h < NH; h += blockDim.x)
      if (s_head[h] != 0u) atomicMax(gmax + h, s_head[h]);
    if (threadIdx.x == 0 && s_bad) atomicOr(gmax + NH, 1u);
  }
}

constexpr int kCoopThreads = 512;  // 16 warps per CTA, at most one CTA per SM
constexpr int kCoopBatch = 2;      // warp iterations of head vectors per item

// One pass over this CTA's share of the work.  An item is (token, group of
// hp * kB head vectors); a warp takes two items per round, so that the round
// costs two dependent memory round trips for both (x and the positions, then
// the cos/sin entries of those positions), with 2 kB 16-byte loads of x per
// lane in flight.  kQuant = false: the CTA's per-head maxima of |y| into
// s_head (max |y| bits), a position outside the tables into *bad_out.
// kQuant = true: codes with the scales in s_head (fp32 bits), followed by
// their bracketing reciprocals (two arrays of NH, see E4m3Div).
template <bool kQuant, int kB>
__device__ __forceinline__ void rope_items_pass(const __nv_bfloat16* __restrict__ x,
                                          const int32_t* __restrict__ pos,
                                          const float* __restrict__ cos_t,
                                          const float* __restrict__ sin_t, int T, int NH, int D,
                                          int max_pos, unsigned* s_head,
                                          uint8_t* __restrict__ codes, int* bad_out) {
  const int lane = threadIdx.x & 31;
  const int n8 = D >> 3;              // lanes per head vector (a power of two <= 32)
  const int lg8 = __ffs(n8) - 1;
  const int hp = 32 >> lg8;           // head vectors per warp iteration
  const int c8 = lane & (n8 - 1);
  const int hoff = lane >> lg8;
  const int gh = hp * kB;     // head vectors per item
  const int ngroups = (NH + gh - 1) / gh;
  const long long n_items = static_cast<long long>(T) * ngroups;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long w0 = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int bad = 0;
  for (long long i0 = w0; i0 < n_items; i0 += 2 * nwarps) {
    uint4 v[2][kB];
    int pp[2], tt[2], hb[2];
    bool live[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const long long i = i0 + it * nwarps;
      live[it] = i < n_items;
      tt[it] = live[it] ? static_cast<int>(i / ngroups) : 0;
      hb[it] = live[it] ? static_cast<int>(i - static_cast<long long>(tt[it]) * ngroups) * gh : 0;
      pp[it] = live[it] ? pos[tt[it]] : 0;
      const size_t row0 = static_cast<size_t>(tt[it]) * NH;
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int h = hb[it] + u * hp + hoff;
        v[it][u] = (live[it] && h < NH) ? *reinterpret_cast<const uint4*>(x + (row0 + h) * D + c8 * 8)
                                        : make_uint4(0, 0, 0, 0);
      }
    }
    float4 cs[2], sn[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      int p = pp[it];
      if (live[it] && (p < 0 || p >= max_pos)) {
        bad = 1;
        p = 0;
      }
      const size_t tab = static_cast<size_t>(live[it] ? p : 0) * (D / 2) + c8 * 4;
      cs[it] = *reinterpret_cast<const float4*>(cos_t + tab);
      sn[it] = *reinterpret_cast<const float4*>(sin_t + tab);
    }
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      if (!live[it]) continue;  // uniform over the warp
      const size_t row0 = static_cast<size_t>(tt[it]) * NH;
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int h = hb[it] + u * hp + hoff;
        float y[8];
        rotate8(v[it][u], cs[it], sn[it], y);
        if (kQuant) {
          if (h < NH) {
            const E4m3Div d{__uint_as_float(s_head[h]), __uint_as_float(s_head[NH + h]),
                            __uint_as_float(s_head[2 * NH + h])};
            uint2 q;
            q.x = static_cast<uint32_t>(quant2(y[0], y[1], d)) |
                  (static_cast<uint32_t>(quant2(y[2], y[3], d)) << 16);
            q.y = static_cast<uint32_t>(quant2(y[4], y[5], d)) |
                  (static_cast<uint32_t>(quant2(y[6], y[7], d)) << 16);
            *reinterpret_cast<uint2*>(codes + (row0 + h) * D + c8 * 8) = q;
          }
        } else {
          float m = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(y[j]));
          // maximum over the group of lanes of one head vector
          for (int o = n8 >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (c8 == 0 && h < NH && m > 0.f) atomicMax(&s_head[h], __float_as_uint(m));
        }
      }
    }
  }
  if (!kQuant && bad) *bad_out = 1;
}

// The per-CTA maxima [NH][G] (head-major) folded into the NH scales, a warp
// per head, into s_head (fp32 bits); `scales` and `ctrl` (status word from the
// G flags after the maxima) when not null.
__device__ __forceinline__ void rope_fold_heads(const float* __restrict__ partials, int G, int NH,
                                                unsigned* s_head, float* __restrict__ scales,
                                                Ctrl* ctrl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int h = warp; h < NH; h += nwarps) {
    const float* ph = partials + static_cast<size_t>(h) * G;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;  // independent chains: loads in flight
    int b = lane;
    for (; b + 96 < G; b += 128) {
      a0 = fmaxf(a0, __ldcg(ph + b));
      a1 = fmaxf(a1, __ldcg(ph + b + 32));
      a2 = fmaxf(a2, __ldcg(ph + b + 64));
      a3 = fmaxf(a3, __ldcg(ph + b + 96));
    }
    for (; b < G; b += 32) a0 = fmaxf(a0, __ldcg(ph + b));
    float a = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float sc = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
    if (lane == 0) {
      s_head[h] = __float_as_uint(sc);
      if (scales != nullptr) scales[h] = sc;
    }
  }
  if (ctrl != nullptr && warp == 0) {
    int bad = 0;
    for (int b = lane; b < G; b += 32) bad |= __ldcg(partials + static_cast<size_t>(G) * NH + b) != 0.f;
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) ctrl->err = bad ? kDevErrRange : 0;
  }
}

// The whole operation: pass 1, grid synchronisation, per-head scales, pass 2.
// partials: [NH][gridDim] per-CTA maxima (head-major: a head's maxima are
// contiguous), then [gridDim] flags.
__global__ void __launch_bounds__(kCoopThreads, 1)
    rope_coop_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ pos,
                     const float* __restrict__ cos_t, const float* __restrict__ sin_t, int T,
                     int NH, int D, int max_pos, float* __restrict__ partials,
                     float* __restrict__ scales, uint8_t* __restrict__ codes, Ctrl* ctrl) {
  // [NH]: max|y| bits, then the scales, followed by [2][NH] reciprocals
  extern __shared__ unsigned s_head[];
  __shared__ int s_bad;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int G = static_cast<int>(gridDim.x);
  for (int h = threadIdx.x; h < NH; h += blockDim.x) s_head[h] = 0u;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  rope_items_pass<false, kCoopBatch>(x, pos, cos_t, sin_t, T, NH, D, max_pos, s_head, nullptr,
                                     &s_bad);
  __syncthreads();
  for (int h = threadIdx.x; h < NH; h += blockDim.x)
    partials[static_cast<size_t>(h) * G + blockIdx.x] = __uint_as_float(s_head[h]);
  if (threadIdx.x == 0) partials[static_cast<size_t>(G) * NH + blockIdx.x] = s_bad ? 1.f : 0.f;
  // nothing above waits on another CTA, so every CTA arrives here
  cg::this_grid().sync();
  // every CTA folds the per-CTA maxima into the scales
  rope_fold_heads(partials, G, NH, s_head, blockIdx.x == 0 ? scales : nullptr,
                  blockIdx.x == 0 ? ctrl : nullptr);
  __syncthreads();
  for (int h = threadIdx.x; h < NH; h += blockDim.x) {
    const E4m3Div d = e4m3_div(__uint_as_float(s_head[h]));
    s_head[NH + h] = __float_as_uint(d.rlo);
    s_head[2 * NH + h] = __float_as_uint(d.rhi);
  }
  __syncthreads();
  rope_items_pass<true, kCoopBatch>(x, pos, cos_t, sin_t, T, NH, D, max_pos, s_head, codes,
                                    nullptr);
}

}  // namespace

int rope_grid(long long T, int NH, int D, int num_sms) {
  (void)NH;
  (void)D;
  long long g = (T + (kRopeThreads / 32) - 1) / (kRopeThreads / 32);  // a warp per token
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (g > cap) g = cap;
  if (g > kRopeMaxCtas) g = kRopeMaxCtas;
  return static_cast<int>(g < 1 ? 1 : g);
}

cudaError_t launch_inv_rope_quant(const __nv_bfloat16* x, const int32_t* pos, const float* cos_t,
                                  const float* sin_t, int T, int NH, int D, int max_pos,
                                  uint8_t* codes, float* scales, Ctrl* ctrl, float* partials,
                                  int num_sms, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(NH) * sizeof(float);
  const size_t smem_q = 3 * smem;  // scales and their two reciprocals
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    const int max_q = 3 * 4096 * static_cast<int>(sizeof(float));
    cudaError_t e = checked(cudaFuncSetAttribute(rope_pass_kernel<true>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, max_q),
                            "smem attribute");
    if (e == cudaSuccess)
      e = checked(cudaFuncSetAttribute(rope_coop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       max_q),
                  "smem attribute");
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  // small inputs: at most two rounds of two items per warp on one CTA per SM
  const int gh = (32 / (D / 8)) * kCoopBatch;
  const long long items = static_cast<long long>(T) * ((NH + gh - 1) / gh);
  const long long per_cta = 2 * (kCoopThreads / 32);
  if (items <= 2 * per_cta * num_sms && num_sms <= kRopeMaxCtas) {
    const int g = static_cast<int>(
        std::min<long long>(num_sms, std::max<long long>(1, (items + per_cta - 1) / per_cta)));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(g);
    cfg.blockDim = dim3(kCoopThreads);
    cfg.dynamicSmemBytes = smem_q;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // the CTAs synchronise once
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return checked(cudaLaunchKernelEx(&cfg, rope_coop_kernel, x, pos, cos_t, sin_t, T, NH, D,
                                      max_pos, partials, scales, codes, ctrl),
                   "cooperative kernel launch");
  }
  // the call's per-head maxima and flag word, zeroed, then the two passes
  unsigned* gmax = reinterpret_cast<unsigned*>(partials);
  cudaError_t e = checked(cudaMemsetAsync(gmax, 0, sizeof(unsigned) * (static_cast<size_t>(NH) + 1), st),
                          "memset");
  if (e != cudaSuccess) return e;
  const int grid = rope_grid(T, NH, D, num_sms);
  e = launch_pdl(rope_pass_kernel<false>, dim3(grid), dim3(kRopeThreads), smem, st, x, pos, cos_t,
                 sin_t, T, NH, D, max_pos, gmax, static_cast<float*>(nullptr),
                 static_cast<uint8_t*>(nullptr), static_cast<Ctrl*>(nullptr));
  if (e != cudaSuccess) return e;
  return launch_pdl(rope_pass_kernel<true>, dim3(grid), dim3(kRopeThreads), smem_q, st, x, pos,
                    cos_t, sin_t, T, NH, D, max_pos, gmax, scales, codes, ctrl);
}

}  // namespace moe
