// Grouped expert GEMMs on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Operand placement follows the Swap-AB idea of "Amazon SageMaker AI 上的
// Mixture-of-Experts 内核工程优化" (section "Swap-AB for WGMMA utilization",
// and the digest page's B^T[N,K] x A^T[K,M] -> C^T[N,M]): the expert weight
// block (128 output rows) is the MMA's A operand and fills the M = 128 slot
// (128 TMEM lanes); the tokens routed to the expert are the B operand, N =
// 16..256 columns.  When an expert sees one token (decode) the MMA still does
// useful work on all 128 lanes, and the weight stream is what the kernel
// waits on.  The same tiling serves prefill, where N grows to 256.
//
// One persistent CTA per SM walks a flat list of work units
// (row tile of an expert's tokens) x (128-row weight block) [x K slice].
// Warp roles:
//   warp 0      TMA producer: weight block(s) + token tile per K step into a
//               ring of shared-memory stages (128-byte swizzle, K-major);
//   warp 1      allocates TMEM and issues tcgen05.mma (one thread), commits
//               stage release and accumulator-ready barriers;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, then either
//               gate/up:  h = SiLU(g * s) * (u * s) -> fp32 (FP8 path, with a
//                         running amax|h|) or bf16 (bf16 path)
//               down:     y * s * topk_weight -> red.add into the fp32 combine
//                         buffer (expert aggregation fused into the GEMM).
// The accumulator is double-buffered in TMEM when it fits, so the epilogue of
// one unit overlaps the MMAs of the next.  Every wait is bounded; on timeout
// the CTA records kDevErrTimeout and leaves.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kSmemLimit = 232448;  // 227 KB opt-in per CTA
constexpr int kSmemSlack = 1024 + 256;
constexpr int kMaxStages = 8;

struct Unit {
  int e, row0, n, nb, kb, ke;
};

__device__ __forceinline__ Unit decode_unit(const GemmParams& p, int u) {
  const int per_tile = p.nb_count * p.split_k;
  const int mt = u / per_tile;
  const int r = u - mt * per_tile;
  const int nb = r / p.split_k;
  const int ks = r - nb * p.split_k;
  const int4 t = p.mtiles[mt];
  Unit un;
  un.e = t.x;
  un.row0 = t.y;
  un.n = t.z;
  un.nb = nb;
  un.kb = ks * p.k_steps / p.split_k;
  un.ke = (ks + 1) * p.k_steps / p.split_k;
  return un;
}

template <bool kBF16, bool kSwiGLU>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  constexpr uint32_t kABytes = kSwiGLU ? 32768u : 16384u;
  const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(p.bn_max) * 128u;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* never = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, 4);
    }
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int num_units = p.ctrl->num_mtiles * p.nb_count * p.split_k;
  const uint64_t limit = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const Unit un = decode_unit(p, u);
        const int wrow = un.e * p.rows_per_expert + un.nb * 128;
        for (int kk = un.kb; kk < un.ke; ++kk, ++it) {
          const uint32_t s = it % S;
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait(empty + s, ph ^ 1u, abort_flag, limit)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + static_cast<size_t>(s) * stage_bytes;
          uint8_t* sb = sa + kABytes;
          mbar_arrive_expect_tx(full + s, kABytes + static_cast<uint32_t>(un.n) * 128u);
          const int kc = kk * p.k_elems;
          tma_load_2d_hint(sa, &tm_a, full + s, kc, wrow, pol_w);
          if (kSwiGLU) tma_load_2d_hint(sa + 16384, &tm_a, full + s, kc, wrow + p.up_offset, pol_w);
          for (int j = 0; j < un.n; j += 16) tma_load_2d(sb + j * 128, &tm_b, full + s, kc, un.row0 + j);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(&p.ctrl->err, kDevErrTimeout);
        // let the copies already issued land before the CTA leaves
        const uint32_t n_back = it < static_cast<uint32_t>(S) ? it : static_cast<uint32_t>(S);
        for (uint32_t b = 1; b <= n_back; ++b) {
          const uint32_t i2 = it - b;
          volatile int no_abort = 0;
          mbar_wait(full + (i2 % S), (i2 / S) & 1u, &no_abort, 20000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, tt = 0;
      bool ok = true;
      if (p.debug & MOE_DEBUG_FORCE_TIMEOUT) ok = mbar_wait(never, 0, abort_flag, limit);
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const Unit un = decode_unit(p, u);
        const uint32_t a = tt % static_cast<uint32_t>(p.num_acc);
        const uint32_t aph = (tt / static_cast<uint32_t>(p.num_acc)) & 1u;
        if (!mbar_wait(tempty + a, aph ^ 1u, abort_flag, limit)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t idesc = umma_idesc(kBF16, 128, un.n);
        const uint32_t d0 = tmem + a * static_cast<uint32_t>(p.acc_stride);
        const uint32_t d1 = d0 + static_cast<uint32_t>(p.bn_max);
        for (int kk = un.kb; kk < un.ke; ++kk, ++it) {
          const uint32_t s = it % S;
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait(full + s, ph, abort_flag, limit)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_addr(smem + static_cast<size_t>(s) * stage_bytes);
          const uint64_t da0 = sdesc_kmajor_sw128(sa);
          const uint64_t da1 = sdesc_kmajor_sw128(sa + 16384);
          const uint64_t db = sdesc_kmajor_sw128(sa + kABytes);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint32_t acc = (kk > un.kb || k4 > 0) ? 1u : 0u;
            // +2 in the start-address field = +32 bytes of K inside the swizzle atom
            if (kBF16) {
              umma_bf16(d0, da0 + 2 * k4, db + 2 * k4, idesc, acc);
              if (kSwiGLU) umma_bf16(d1, da1 + 2 * k4, db + 2 * k4, idesc, acc);
            } else {
              umma_f8(d0, da0 + 2 * k4, db + 2 * k4, idesc, acc);
              if (kSwiGLU) umma_f8(d1, da1 + 2 * k4, db + 2 * k4, idesc, acc);
            }
          }
          umma_commit(empty + s);
        }
        if (!ok) break;
        umma_commit(tfull + a);
        ++tt;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(&p.ctrl->err, kDevErrTimeout);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (4 warps)
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int row_l = q * 32 + lane;
    float act_s = 1.f;
    if (!kBF16) act_s = p.act_scale_sel == 1 ? p.ctrl->s_x : p.ctrl->s_h;
    float amax = 0.f;
    uint32_t tt = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const Unit un = decode_unit(p, u);
      const uint32_t a = tt % static_cast<uint32_t>(p.num_acc);
      const uint32_t aph = (tt / static_cast<uint32_t>(p.num_acc)) & 1u;
      int got = 0;
      if (lane == 0) got = mbar_wait(tfull + a, aph, abort_flag, limit) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float sc = kBF16 ? 1.f : act_s * p.w_scale[un.e];
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                             a * static_cast<uint32_t>(p.acc_stride);
      const int col = un.nb * 128 + row_l;
      for (int c0 = 0; c0 < un.n; c0 += 16) {
        if (kSwiGLU) {
          float g[16], v[16];
          tmem_ld16x2(tbase + c0, tbase + p.bn_max + c0, g, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = un.row0 + c0 + j;
            const float gv = g[j] * sc;
            const float uv = v[j] * sc;
            const float hv = gv / (1.f + __expf(-gv)) * uv;
            const size_t at = static_cast<size_t>(r) * p.ldh + col;
            if (kBF16) {
              // bf16 weights: h feeds the bf16 down-projection MMA directly
              static_cast<__nv_bfloat16*>(p.h_out)[at] = __float2bfloat16_rn(hv);
            } else {
              // FP8: h stays fp32 until its per-tensor scale is known; an
              // intermediate bf16 rounding would move values across E4M3
              // rounding boundaries and cost percent-level output error
              static_cast<float*>(p.h_out)[at] = hv;
              if (p.sorted_ids[r] < p.P) amax = fmaxf(amax, fabsf(hv));
            }
          }
        } else {
          float y[16];
          tmem_ld16(tbase + c0, y);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = un.row0 + c0 + j;
            const int pid = p.sorted_ids[r];
            if (pid < p.P) {
              const int t = pid / p.top_k;
              red_add_f32(p.acc_out + static_cast<size_t>(t) * p.ldo + col,
                          y[j] * sc * p.topk_w[pid]);
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty + a);
      ++tt;
    }
    if (kSwiGLU && !kBF16) {
#pragma unroll
      for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0 && amax > 0.f) atomicMax(&p.ctrl->amax_h, __float_as_uint(amax));
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(&p.ctrl->err, kDevErrTimeout);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
  }
}

template <bool kBF16, bool kSwiGLU>
cudaError_t launch_one(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb, int grid,
                       cudaStream_t st) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<kBF16, kSwiGLU>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const size_t smem = gemm_smem_bytes(kSwiGLU, p.bn_max, p.stages);
  moe_gemm_kernel<kBF16, kSwiGLU><<<grid, kGemmThreads, smem, st>>>(p, ta, tb);
  return cudaGetLastError();
}

}  // namespace

size_t gemm_smem_bytes(bool swiglu, int bn_max, int stages) {
  const size_t stage = (swiglu ? 32768u : 16384u) + static_cast<size_t>(bn_max) * 128u;
  return stage * stages + kSmemSlack;
}

int gemm_max_stages(bool swiglu, int bn_max) {
  const size_t stage = (swiglu ? 32768u : 16384u) + static_cast<size_t>(bn_max) * 128u;
  int s = static_cast<int>((kSmemLimit - kSmemSlack) / stage);
  if (s > kMaxStages) s = kMaxStages;
  return s;
}

cudaError_t launch_gemm(bool bf16, bool swiglu, const GemmParams& p, const CUtensorMap& ta,
                        const CUtensorMap& tb, int grid, cudaStream_t st) {
  if (bf16) {
    return swiglu ? launch_one<true, true>(p, ta, tb, grid, st)
                  : launch_one<true, false>(p, ta, tb, grid, st);
  }
  return swiglu ? launch_one<false, true>(p, ta, tb, grid, st)
                : launch_one<false, false>(p, ta, tb, grid, st);
}

}  // namespace moe
