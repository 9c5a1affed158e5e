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
// Two passes over x (bf16 [T][NH][D]):
//   1. rope_amax_kernel: rotate, per-head maxima of |y| per CTA -> partials;
//   2. rope_quant_kernel: every CTA folds the partials into the NH scales,
//      rotates again and writes the codes (CTA 0 also writes the scales and
//      the status word).
// A thread takes 8 elements (4 pairs) of one head vector: one 16-byte load
// of x, 16-byte loads of the 4 cosines and 4 sines, one 8-byte store of codes.
// A group of D/8 lanes covers one head vector, so a warp covers 32/(D/8)
// consecutive (token, head) rows and the per-head maxima reduce inside each
// group before one shared-memory atomic per group.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRopeThreads = 256;

__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The 8 rotated values of one thread item.  Positions outside the tables are
// clamped to 0 and reported through *bad.
__device__ __forceinline__ void rotate8(const __nv_bfloat16* __restrict__ x,
                                        const int32_t* __restrict__ pos,
                                        const float* __restrict__ cos_t,
                                        const float* __restrict__ sin_t, int NH, int D,
                                        int max_pos, long long row, int c8, float (&y)[8],
                                        int* bad) {
  const int t = static_cast<int>(row / NH);
  int p = pos[t];
  if (p < 0 || p >= max_pos) {
    *bad = 1;
    p = 0;
  }
  const uint4 v = *reinterpret_cast<const uint4*>(x + row * D + c8 * 8);
  const size_t tab = static_cast<size_t>(p) * (D / 2) + c8 * 4;
  const float4 c = *reinterpret_cast<const float4*>(cos_t + tab);
  const float4 s = *reinterpret_cast<const float4*>(sin_t + tab);
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

__global__ void __launch_bounds__(kRopeThreads)
    rope_amax_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ pos,
                     const float* __restrict__ cos_t, const float* __restrict__ sin_t, int T,
                     int NH, int D, int max_pos, float* __restrict__ partials) {
  extern __shared__ unsigned s_amax[];  // [NH] bits of max|y| (non-negative floats order like uints)
  __shared__ int s_bad;
  pdl_wait();
  pdl_trigger();
  for (int h = threadIdx.x; h < NH; h += blockDim.x) s_amax[h] = 0u;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const int n8 = D / 8;                 // lanes per head vector (a power of two <= 32)
  const long long items = static_cast<long long>(T) * NH * n8;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  int bad = 0;
  // every lane of a warp runs the same number of iterations (the warp shuffle
  // below needs all of them); out-of-range items contribute 0
  const long long base0 = static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
  for (long long b = base0; b < items; b += step) {
    const long long i = b + (threadIdx.x & 31);
    float m = 0.f;
    long long row = 0;
    if (i < items) {
      row = i / n8;
      float y[8];
      rotate8(x, pos, cos_t, sin_t, NH, D, max_pos, row, static_cast<int>(i - row * n8), y, &bad);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(y[j]));
    }
    // maximum over the n8 lanes of one head vector
    for (int o = n8 >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (i < items && ((threadIdx.x & 31) & (n8 - 1)) == 0 && m > 0.f)
      atomicMax(&s_amax[static_cast<int>(row % NH)], __float_as_uint(m));
  }
  if (bad) s_bad = 1;
  __syncthreads();
  for (int h = threadIdx.x; h < NH; h += blockDim.x)
    partials[static_cast<size_t>(blockIdx.x) * NH + h] = __uint_as_float(s_amax[h]);
  if (threadIdx.x == 0) partials[static_cast<size_t>(gridDim.x) * NH + blockIdx.x] = s_bad ? 1.f : 0.f;
}

__global__ void __launch_bounds__(kRopeThreads)
    rope_quant_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ pos,
                      const float* __restrict__ cos_t, const float* __restrict__ sin_t, int T,
                      int NH, int D, int max_pos, const float* __restrict__ partials, int n_part,
                      uint8_t* __restrict__ codes, float* __restrict__ scales, Ctrl* ctrl) {
  extern __shared__ float s_scale[];  // [NH]
  pdl_wait();
  pdl_trigger();
  for (int h = threadIdx.x; h < NH; h += blockDim.x) {
    float a = 0.f;
    for (int b = 0; b < n_part; ++b) a = fmaxf(a, partials[static_cast<size_t>(b) * NH + h]);
    const float s = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
    s_scale[h] = s;
    if (blockIdx.x == 0) scales[h] = s;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    int bad = 0;
    for (int b = 0; b < n_part; ++b) bad |= partials[static_cast<size_t>(n_part) * NH + b] != 0.f;
    ctrl->err = bad ? kDevErrRange : 0;
  }
  __syncthreads();
  const int n8 = D / 8;
  const long long items = static_cast<long long>(T) * NH * n8;
  int bad = 0;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < items;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = i / n8;
    float y[8];
    rotate8(x, pos, cos_t, sin_t, NH, D, max_pos, row, static_cast<int>(i - row * n8), y, &bad);
    const float s = s_scale[static_cast<int>(row % NH)];
    uint2 q;
    q.x = static_cast<uint32_t>(cvt_e4m3x2(__fdiv_rn(y[0], s), __fdiv_rn(y[1], s))) |
          (static_cast<uint32_t>(cvt_e4m3x2(__fdiv_rn(y[2], s), __fdiv_rn(y[3], s))) << 16);
    q.y = static_cast<uint32_t>(cvt_e4m3x2(__fdiv_rn(y[4], s), __fdiv_rn(y[5], s))) |
          (static_cast<uint32_t>(cvt_e4m3x2(__fdiv_rn(y[6], s), __fdiv_rn(y[7], s))) << 16);
    *reinterpret_cast<uint2*>(codes + i * 8) = q;
  }
}

}  // namespace

int rope_grid(long long T, int NH, int D, int num_sms) {
  const long long items = T * NH * (D / 8);
  long long g = (items + kRopeThreads - 1) / kRopeThreads;
  const long long cap = static_cast<long long>(num_sms) * 4;
  if (g > cap) g = cap;
  if (g > kRopeMaxCtas) g = kRopeMaxCtas;
  return static_cast<int>(g < 1 ? 1 : g);
}

cudaError_t launch_inv_rope_quant(const __nv_bfloat16* x, const int32_t* pos, const float* cos_t,
                                  const float* sin_t, int T, int NH, int D, int max_pos,
                                  uint8_t* codes, float* scales, Ctrl* ctrl, float* partials,
                                  int num_sms, cudaStream_t st) {
  const int grid = rope_grid(T, NH, D, num_sms);
  const size_t smem = static_cast<size_t>(NH) * sizeof(float);
  cudaError_t e = launch_pdl(rope_amax_kernel, dim3(grid), dim3(kRopeThreads), smem, st, x, pos,
                             cos_t, sin_t, T, NH, D, max_pos, partials);
  if (e != cudaSuccess) return e;
  return launch_pdl(rope_quant_kernel, dim3(grid), dim3(kRopeThreads), smem, st, x, pos, cos_t,
                    sin_t, T, NH, D, max_pos, static_cast<const float*>(partials), grid, codes,
                    scales, ctrl);
}

}  // namespace moe
