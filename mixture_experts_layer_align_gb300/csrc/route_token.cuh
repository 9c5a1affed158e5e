// Warp-level router shared by the library's kernels: softmax over the E
// fp32 logits of a token and selection of its top-k experts, ties to the
// lower expert index (token routing, "Amazon SageMaker AI 上的
// Mixture-of-Experts 内核工程优化", Introduction; the router function, the
// tie rule and the slot order are this library's reading of the pages, which
// leave them open).
#pragma once

#include <math.h>
#include <stdint.h>

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// ------------------------------------------------------------------ router
// Order-preserving map of a finite float to uint32 (larger float, larger
// key; every key is > 0); -0.0 maps like +0.0 so that the two compare equal.
__device__ __forceinline__ uint32_t float_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One token, one warp.  The row of logits is staged in shared memory (`l`, E
// floats of this warp); softmax with expf on max-subtracted logits; each of
// the k rounds takes the arg-max under (logit desc, index asc) over the
// experts not taken yet (one bit per lane per 32 experts) with two warp
// reductions: the largest key among the lanes' best remaining logits, then
// the lowest expert index holding it.  Writes the k ids and weights (divided
// by their sum when renormalising; id_row / w_row may be shared or global).
__device__ void route_token(const float* __restrict__ src, int E, int k, int renorm, float* l,
                            int32_t* id_row, float* w_row, int lane) {
  uint32_t km = 0u;
  for (int e = lane; e < E; e += 32) {
    const float v = src[e];
    l[e] = v;
    km = max(km, float_key(v));
  }
  const float m = key_float(__reduce_max_sync(kFull, km));
  float z = 0.f;
  for (int e = lane; e < E; e += 32) z += expf(l[e] - m);
  z = warp_sum(z);
  __syncwarp();

  uint32_t taken = 0u;  // bit i <=> expert lane + 32 i already selected
  float sel = 0.f;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;  // 0: no candidate left in this lane
    int bi = 0;
    for (int e = lane, i = 0; e < E; e += 32, ++i) {
      if ((taken >> i) & 1u) continue;
      const uint32_t key = float_key(l[e]);
      if (key > bk) {  // ascending scan: equal keys keep the lower index
        bk = key;
        bi = e;
      }
    }
    const uint32_t kmax = __reduce_max_sync(kFull, bk);
    const int win = static_cast<int>(
        __reduce_min_sync(kFull, bk == kmax ? static_cast<uint32_t>(bi) : 0xffffffffu));
    if ((win & 31) == lane) taken |= 1u << (win >> 5);
    const float ex = expf(key_float(kmax) - m);
    sel += ex;
    if (lane == 0) {
      id_row[j] = win;
      w_row[j] = ex;
    }
  }
  __syncwarp();
  const float denom = renorm ? sel : z;
  for (int j = lane; j < k; j += 32) w_row[j] = __fdiv_rn(w_row[j], denom);
  __syncwarp();
}

// The same selection with the row's order keys in registers (E <= 32 * R):
// each lane holds experts lane + 32 i; a taken expert's key is set to 0 (every
// real key is > 0).  The full softmax sum is only formed when the weights are
// not renormalised over the k selected.  Same results as route_token.
template <int R>
__device__ void route_token_reg(const float* __restrict__ src, int E, int k, int renorm,
                                int32_t* id_row, float* w_row, int lane) {
  uint32_t key[R];
  uint32_t km = 0u;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? float_key(src[e]) : 0u;
    km = max(km, key[i]);
  }
  const float m = key_float(__reduce_max_sync(kFull, km));
  float z = 0.f;
  if (!renorm) {
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (lane + 32 * i < E) z += expf(key_float(key[i]) - m);
    z = warp_sum(z);
  }
  float sel = 0.f;
  uint32_t my_key = 0u;  // k <= 32: lane j keeps the j-th selected key
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (key[i] > bk) {  // ascending scan: equal keys keep the lower index
        bk = key[i];
        bi = lane + 32 * i;
      }
    const uint32_t kmax = __reduce_max_sync(kFull, bk);
    const int win = static_cast<int>(
        __reduce_min_sync(kFull, bk == kmax ? static_cast<uint32_t>(bi) : 0xffffffffu));
    if ((win & 31) == lane) {
#pragma unroll
      for (int i = 0; i < R; ++i)
        if (i == (win >> 5)) key[i] = 0u;
    }
    if (lane == 0) id_row[j] = win;
    if (k <= 32) {
      if (lane == j) my_key = kmax;
    } else {
      const float ex = expf(key_float(kmax) - m);
      sel += ex;
      if (lane == 0) w_row[j] = ex;
    }
  }
  if (k <= 32) {
    // the k probabilities in parallel, one lane each
    const float ex = lane < k ? expf(key_float(my_key) - m) : 0.f;
    const float denom = renorm ? warp_sum(ex) : z;
    if (lane < k) w_row[lane] = __fdiv_rn(ex, denom);
    __syncwarp();
    return;
  }
  __syncwarp();
  const float denom = renorm ? sel : z;
  for (int j = lane; j < k; j += 32) w_row[j] = __fdiv_rn(w_row[j], denom);
  __syncwarp();
}

// Dispatch on the number of experts: registers up to 256, else the shared
// memory row `l`.
__device__ __forceinline__ void route_token_any(const float* __restrict__ src, int E, int k,
                                                int renorm, float* l, int32_t* id_row,
                                                float* w_row, int lane) {
  if (E <= 32) route_token_reg<1>(src, E, k, renorm, id_row, w_row, lane);
  else if (E <= 64) route_token_reg<2>(src, E, k, renorm, id_row, w_row, lane);
  else if (E <= 128) route_token_reg<4>(src, E, k, renorm, id_row, w_row, lane);
  else if (E <= 256) route_token_reg<8>(src, E, k, renorm, id_row, w_row, lane);
  else route_token(src, E, k, renorm, l, id_row, w_row, lane);
}

}  // namespace
}  // namespace moe
