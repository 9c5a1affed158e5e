// Gate/up expert GEMM of wide row tiles on SM pairs (tcgen05 cta_group::2).
//
// Placement as in the single-SM kernel (Swap-AB of "Amazon SageMaker AI 上的
// Mixture-of-Experts 内核工程优化", section "Swap-AB for WGMMA utilization"):
// expert weight rows in the MMA's M slot, routed tokens in N.  Here a cluster
// of two CTAs on two SMs shares one tile of 256 weight rows (two consecutive
// 128-row blocks, one per CTA, for gate and for up) x N <= 256 routed tokens:
// one M = 256 MMA per K step and matrix, each CTA supplying its 128 weight rows
// and half of the token rows from its own shared memory, each CTA's TMEM
// receiving its 128 rows x N.  A K step then costs an SM 32 KB of weights +
// N/2 x 128 B of tokens instead of 32 KB + N x 128 B, so four 48 KB stages fit
// where three 64 KB stages did, for the same MMA work per SM: prefill, where
// the single-SM kernel waits on its operands, gets more of them in flight.
//
// Work: units (row tile of the wide tile list, pair of weight blocks), whole
// units round-robin over the clusters in list order (the units in flight share
// weight blocks and token rows through L2).  Per CTA: warp 0 TMA producer
// (both CTAs load their halves; the byte counts complete on the rank-0 CTA's
// `full` barriers), warp 1 TMEM allocation and, on rank 0, the MMA issue
// (commits multicast to both CTAs' barriers), warps 2..9 the epilogue of the
// CTA's own 128 weight rows (h = SiLU(g s) (u s), fp32, running amax |h|;
// `tempty` on rank 0 counts both CTAs' epilogue warps).  The accumulators of a
// 256-token tile fill the 512 TMEM columns: one buffer.  Every wait is bounded;
// on timeout the CTA records kDevErrTimeout and leaves through the cluster
// barrier like any other exit.
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kPairStages = 4;
constexpr uint32_t kPairABytes = 32768;                          // gate + up, 128 rows x 128 B each
constexpr int kPairMaxN = 256;                                   // tokens per tile
constexpr uint32_t kPairBBytes = (kPairMaxN / 2) * 128;          // this CTA's half of them
constexpr uint32_t kPairStageBytes = kPairABytes + kPairBBytes;  // 48 KB
constexpr int kPairSmem = 1024 + kPairStages * kPairStageBytes + 256;
constexpr uint32_t kPairEpiBarrier = 1;
constexpr uint32_t kPairEpiThreads = 32 * kGemmEpiWarps;
constexpr uint32_t kPairTmemCols = 512;  // gate at column 0, up at 256

struct PairTile {
  int e, row0, n, nmma, nb;
};

// Unit u -> the CTA's part: row tile u / npb of the wide list (n real rows,
// MMA N = n rounded up to 32 so that each CTA holds a multiple of 16 rows),
// weight block 2 (u % npb) + rank.
__device__ __forceinline__ PairTile pair_tile(const GemmParams& p, int u, uint32_t rank) {
  const int m = u / p.nb_count;
  const int4 t = p.mtiles[m];
  PairTile r;
  r.e = t.x;
  r.row0 = t.y;
  r.n = t.z & 0xfff;
  r.nmma = (r.n + 31) & ~31;
  r.nb = 2 * (u - m * p.nb_count) + static_cast<int>(rank);
  return r;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ GemmParams p,
                         const __grid_constant__ CUtensorMap tm_a,
                         const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_b64) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int S = kPairStages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * kPairStageBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 1;
  uint64_t* never = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  // per-CTA stamps (MOE_DEBUG_TRACE): entry, inputs ready, first stage landed
  // (the leader's MMA warp; the other CTA of the pair: its first accumulator
  // ready), exit
  unsigned long long* trace =
      (p.trace != nullptr && blockIdx.x < MOE_TRACE_MAX_CTAS) ? p.trace + blockIdx.x * 4 : nullptr;
  if (trace && threadIdx.x == 0) trace[0] = global_timer_ns();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);  // rank 0: its expect_tx arrival + both CTAs' bytes
      mbar_init(empty + s, 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * kGemmEpiWarps);  // rank 0: the epilogue warps of both CTAs
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_b);
    prefetch_tensormap(&tm_b64);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kPairTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Everything above overlaps the previous kernel.  The producer also puts the
  // first stages' weight blocks in flight before that kernel has finished: the
  // tile list it reads for that was written two or more kernels back, and every
  // kernel of the library signals its dependents only after its own wait.
  const bool early_producer = (warp == 0 && lane == 0);
  if (!early_producer) {
    pdl_wait();
    pdl_trigger();
  }
  if (trace && threadIdx.x == 64) trace[1] = global_timer_ns();

  const int K = p.k_steps;
  const int units = p.ctrl->num_mtiles_w * p.nb_count;
  const int n_cl = static_cast<int>(gridDim.x) / 2;
  const int cid = static_cast<int>(blockIdx.x) / 2;
  const uint64_t limit = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_last();  // weight blocks serve several row tiles
      // weight blocks of the first S stages (fresh stages: no wait on `empty`)
      uint32_t pre = 0;
      for (int u = cid; pre < static_cast<uint32_t>(S) && u < units; u += n_cl) {
        const PairTile t = pair_tile(p, u, rank);
        const uint32_t half = static_cast<uint32_t>(t.nmma / 2);
        const int wrow = t.e * p.rows_per_expert + t.nb * 128;
        for (int kk = 0; kk < K && pre < static_cast<uint32_t>(S); ++kk, ++pre) {
          const uint32_t fb = mapa_shared(smem_addr(full + pre), 0);
          if (leader) mbar_arrive_expect_tx(full + pre, 2u * (kPairABytes + half * 128u));
          uint8_t* sa = smem + static_cast<size_t>(pre) * kPairStageBytes;
          const int kc = kk * p.k_elems;
          tma_load_2d_pair(sa, &tm_a, fb, kc, wrow, pol_w);
          tma_load_2d_pair(sa + 16384, &tm_a, fb, kc, wrow + p.up_offset, pol_w);
        }
      }
      // token rows are the previous kernels' output
      pdl_wait();
      pdl_trigger();
      uint32_t it = 0;
      bool ok = true;
      for (int u = cid; ok && u < units; u += n_cl) {
        const PairTile t = pair_tile(p, u, rank);
        const int half = t.nmma / 2;  // token rows from this CTA
        const int brow = t.row0 + static_cast<int>(rank) * half;
        const int wrow = t.e * p.rows_per_expert + t.nb * 128;
        for (int kk = 0; kk < K; ++kk, ++it) {
          const uint32_t s = it % S;
          const uint32_t ph = (it / S) & 1u;
          const uint32_t fb = mapa_shared(smem_addr(full + s), 0);
          uint8_t* sa = smem + static_cast<size_t>(s) * kPairStageBytes;
          uint8_t* sb = sa + kPairABytes;
          const int kc = kk * p.k_elems;
          if (it >= pre) {
            if (!mbar_wait(empty + s, ph ^ 1u, abort_flag, limit)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(full + s, 2u * (kPairABytes + static_cast<uint32_t>(half) * 128u));
            tma_load_2d_pair(sa, &tm_a, fb, kc, wrow, pol_w);
            tma_load_2d_pair(sa + 16384, &tm_a, fb, kc, wrow + p.up_offset, pol_w);
          }
          int j = 0;
          for (; j + 64 <= half; j += 64) tma_load_2d_pair(sb + j * 128, &tm_b64, fb, kc, brow + j);
          for (; j < half; j += 16) tma_load_2d_pair(sb + j * 128, &tm_b, fb, kc, brow + j);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(&p.ctrl->err, kDevErrTimeout);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issue (rank 0)
    if (lane == 0 && leader) {
      uint32_t it = 0, tt = 0;
      bool ok = true;
      if (p.debug & MOE_DEBUG_FORCE_TIMEOUT) ok = mbar_wait(never, 0, abort_flag, limit);
      for (int u = cid; ok && u < units; u += n_cl) {
        const PairTile t = pair_tile(p, u, 0);
        if (!mbar_wait(tempty, (tt & 1u) ^ 1u, abort_flag, limit)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t idesc = umma_idesc(false, 256, t.nmma);
        for (int kk = 0; kk < K; ++kk, ++it) {
          const uint32_t s = it % S;
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait(full + s, ph, abort_flag, limit)) {
            ok = false;
            break;
          }
          if (trace && it == 0) trace[2] = global_timer_ns();
          tc_fence_after_sync();
          const uint32_t sa = smem_addr(smem + static_cast<size_t>(s) * kPairStageBytes);
          const uint64_t da0 = sdesc_kmajor_sw128(sa);
          const uint64_t da1 = sdesc_kmajor_sw128(sa + 16384);
          const uint64_t db = sdesc_kmajor_sw128(sa + kPairABytes);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint32_t acc = (kk > 0 || k4 > 0) ? 1u : 0u;
            // +2 in the start-address field = +32 bytes of K inside the swizzle atom
            umma_f8_pair(tmem, da0 + 2 * k4, db + 2 * k4, idesc, acc);
            umma_f8_pair(tmem + kPairMaxN, da1 + 2 * k4, db + 2 * k4, idesc, acc);
          }
          umma_commit_pair(empty + s, 0x3);
        }
        if (!ok) break;
        umma_commit_pair(tfull, 0x3);
        ++tt;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(&p.ctrl->err, kDevErrTimeout);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int c_begin = 16 * ((warp - 2) >> 2);  // the two warps of a quarter alternate chunks
    const int row_l = q * 32 + lane;
    const float s_x = p.ctrl->s_x;
    const uint32_t tempty_leader = mapa_shared(smem_addr(tempty), 0);
    float amax = 0.f;
    uint32_t tt = 0;
    for (int u = cid; u < units; u += n_cl) {
      const PairTile t = pair_tile(p, u, rank);
      int got = 0;
      if (lane == 0) got = mbar_wait(tfull, tt & 1u, abort_flag, limit) ? 1 : 0;
      if (trace && !leader && tt == 0 && threadIdx.x == 64) trace[2] = global_timer_ns();
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!named_barrier_and(kPairEpiBarrier, kPairEpiThreads, got != 0)) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicOr(&p.ctrl->err, kDevErrTimeout);
        }
        break;
      }
      tc_fence_after_sync();
      const float sc = s_x * p.w_scale[t.e];
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16);
      float* hcol = static_cast<float*>(p.h_out) + t.nb * 128 + row_l;
      // columns past t.n belong to other row tiles: not stored.  Padding rows
      // inside t.n hold zero tokens, so their h is 0 and leaves amax alone.
      for (int c0 = c_begin; c0 < t.n; c0 += 32) {
        float gg[16], v[16];
        tmem_ld16x2(tbase + c0, tbase + kPairMaxN + c0, gg, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float gv = gg[j] * sc;
          const float uv = v[j] * sc;
          const float hv = __fdividef(gv, 1.f + __expf(-gv)) * uv;  // SiLU(g) * u
          hcol[static_cast<size_t>(t.row0 + c0 + j) * p.ldh] = hv;
          amax = fmaxf(amax, fabsf(hv));
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader);
      ++tt;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0 && amax > 0.f) atomicMax(&p.ctrl->amax_h, __float_as_uint(amax));
  }

  if (*abort_flag) {
    // copies already issued by either CTA land within microseconds; give them
    // that long before the shared memory is released
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // the pair's MMAs, copies and remote arrivals are done
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, kPairTmemCols);
  }
  if (trace && threadIdx.x == 0) {
    __threadfence();
    trace[3] = global_timer_ns();
  }
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                             const CUtensorMap& tb64, int max_clusters, cudaStream_t st) {
  static thread_local int configured_device = -1;
  static thread_local int resident_clusters = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = checked(cudaFuncSetAttribute(moe_gemm_pair_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kPairSmem),
                            "smem attribute");
    if (e != cudaSuccess) return e;
    // clusters of two that fit on the device at once (persistent grid)
    cudaLaunchConfig_t qc{};
    qc.gridDim = dim3(2);
    qc.blockDim = dim3(kGemmThreads);
    qc.dynamicSmemBytes = kPairSmem;
    int n = 0;
    e = checked(cudaOccupancyMaxActiveClusters(&n, moe_gemm_pair_kernel, &qc), "cluster occupancy");
    if (e != cudaSuccess) return e;
    resident_clusters = n;
    configured_device = dev;
  }
  const int clusters = std::max(1, std::min(resident_clusters, max_clusters));
  return launch_pdl(moe_gemm_pair_kernel, dim3(2 * clusters), dim3(kGemmThreads),
                    static_cast<size_t>(kPairSmem), st, p, ta, tb, tb64);
}

}  // namespace moe
