// The fused MoE layer for small batches (decode) in ONE persistent kernel.
//
// "Amazon SageMaker AI 上的 Mixture-of-Experts 内核工程优化" (English original
// page, Introduction) defines the fused MoE layer as token routing, data
// shuffling and the expert computation merged into a single batched GPU
// operation, and its section "Backend routing for FP8 tensor quantization"
// keeps FP8 scaling, the matrix multiplications and the expert aggregation in
// the same pass.  For small batches the layer is bound by streaming the
// touched experts' weights from HBM, and a chain of separate kernels leaves
// HBM idle at every kernel boundary (each GEMM restarts its weight stream).
// Here one cooperative launch of one CTA per SM does the whole layer:
//
//   phase 0  every CTA routes its share of tokens (a warp per token), takes
//            the max |x| of its slice of x, zeroes its slice of the combine
//            buffer and of the split-tile counters; one grid synchronisation;
//   phase 1  every CTA counts all pairs per expert and builds the row-tile
//            list in its own shared memory (the routing is small), so it can
//            schedule itself and put its first gate/up weight stages in
//            flight at once; its epilogue warps place their chunk of pairs
//            in expert order and write those pairs' x rows as E4M3 codes
//            (or bf16), then count themselves done (counter 0);
//   gate/up  the grouped GEMM with the Swap-AB placement (section "Swap-AB
//            for WGMMA utilization": expert weight rows in the MMA's M slot,
//            the few routed tokens in N), stream-K over (tile, K step),
//            SiLU(g)*u epilogue, running max |h|;
//   h scale  counter 1 (all of h written): every CTA quantises a slice of h
//            with the per-tensor scale, counter 2;
//   down     the same GEMM over w2 -- its weight stages are issued as soon as
//            the ring frees up, before h is quantised, so HBM keeps streaming
//            across the phase change -- with the router-weighted combine as
//            bulk fp32 reductions into the [T, H] buffer;
//   output   counter 3 (all reductions landed): every CTA converts a slice
//            of the combine buffer to bf16.
//
// Warp roles as in the grouped GEMM kernel: warp 0 TMA producer, warp 1 TMEM
// allocation + MMA issue, warps 2..9 epilogue (and the gather / h
// quantisation / output slices).  Every wait is bounded: a counter wait
// gives up at the limit or as soon as any CTA has recorded an error, and the
// CTA then records kDevErrTimeout, lets its copies land and leaves.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "gemm_sched.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "route_token.cuh"

namespace moe {

namespace {

namespace cg = cooperative_groups;

constexpr int kSmemLimit = 232448;  // 227 KB opt-in per CTA (static + dynamic)
constexpr int kMaxTiles = 512;      // row tiles of a call: at most (P + 142 E) / 128 <= 300
constexpr int kMaxChunk = 256;      // pairs placed by one CTA (grid >= P / 256)
constexpr int kMaxS = 4;            // pipeline stages of 32 KB of weights
constexpr int kRows = 128;          // rows of a row tile (MMA N <= 128)
constexpr uint32_t kABytes = 32768;  // weights per stage: gate + up, or two K chunks of w2
constexpr uint32_t kEpiBar = 1;
constexpr uint32_t kEpiThreads = 32 * kGemmEpiWarps;
constexpr int kWarps = kFusedThreads / 32;
constexpr uint32_t kStaging = kGemmEpiWarps * 2 * 16 * 32 * sizeof(float);  // combine staging
constexpr uint32_t kTmemCols = 512;  // two accumulator buffers of 2 x 128 columns

struct SmallShared {
  int4 tiles[kMaxTiles];
  int cnt[kFusedMaxExperts];
  int off[kFusedMaxExperts];
  int before[kFusedMaxExperts];  // pairs before this CTA's chunk, then its placement cursor
  int slot[kMaxChunk];           // aligned row of each pair of this CTA's chunk (-1: none)
  float red[kWarps];
  uint64_t full[kMaxS], empty[kMaxS], tfull[2], tempty[2], never;
  uint32_t tmem_slot;
  int abort_flag;
  int s_last;
  int num_tiles, max_rows, total_rows, tiles_ok;
  float s_x;
};

// Wait until the grid-wide counter reaches `target`, for at most `limit_ns`,
// or until this CTA aborts or any CTA has recorded an error.
__device__ __noinline__ bool grid_wait(const unsigned* ctr, unsigned target, const int* err,
                                       volatile int* abort, uint64_t limit_ns) {
  if (ld_acquire(ctr) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ld_acquire(ctr) >= target) return true;
    if (*abort || *reinterpret_cast<const volatile int*>(err)) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Rows [row0, row0 + n) of a K-major token matrix (n a multiple of 16) into
// consecutive 128-byte rows at `dst`: 64-row boxes, then 16-row boxes.
__device__ __forceinline__ void load_rows(uint8_t* dst, const CUtensorMap* m64,
                                          const CUtensorMap* m16, uint64_t* bar, int kc, int row0,
                                          int n) {
  int j = 0;
  for (; j + 64 <= n; j += 64) tma_load_2d(dst + j * 128, m64, bar, kc, row0 + j);
  for (; j < n; j += 16) tma_load_2d(dst + j * 128, m16, bar, kc, row0 + j);
}

// Epilogue metadata of a tile (weights in M): lane l holds the pair ids and
// router weights of columns l + 32 i; wsc is the expert's weight scale.
struct SmallMeta {
  int pid[4];
  float w[4];
  float wsc;
};

__device__ __forceinline__ SmallMeta small_meta(const FusedParams& p, const Tile& t, int lane,
                                                const float* w_scale, bool want_w, int P) {
  SmallMeta m;
#pragma unroll
  for (int s4 = 0; s4 < 4; ++s4) {
    const int c = s4 * 32 + lane;
    const bool in = c < t.n;
    m.pid[s4] = in ? __ldcg(p.sorted_ids + t.row0 + c) : P;
    m.w[s4] = (want_w && in) ? __ldcg(p.sorted_w + t.row0 + c) : 0.f;
  }
  m.wsc = w_scale != nullptr ? w_scale[t.e] : 1.f;
  return m;
}

template <int N, typename V>
__device__ __forceinline__ V pick(const V (&v)[N], int s) {
  V r = v[0];
#pragma unroll
  for (int i = 1; i < N; ++i) r = (s == i) ? v[i] : r;
  return r;
}

struct PendingRows {
  int s, row0, n, kc, n2;
};

template <bool kBF16>
__global__ void __launch_bounds__(kFusedThreads, 1)
    moe_fused_small_kernel(const __grid_constant__ FusedParams p,
                           const __grid_constant__ CUtensorMap tm_w13,
                           const __grid_constant__ CUtensorMap tm_xs,
                           const __grid_constant__ CUtensorMap tm_xs64,
                           const __grid_constant__ CUtensorMap tm_w2,
                           const __grid_constant__ CUtensorMap tm_h,
                           const __grid_constant__ CUtensorMap tm_h64) {
  __shared__ SmallShared sh;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* staging = reinterpret_cast<float*>(smem);  // per epilogue warp 2 x 16 x 32 fp32
  uint8_t* stages = smem + kStaging;                 // 1024-byte aligned
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int T = p.T, H = p.H, I = p.I, E = p.E, k = p.k;
  const int P = T * k;
  constexpr int kElems = kBF16 ? 64 : 128;  // elements of K per 128-byte step
  Ctrl* ctrl = p.ctrl;
  const uint64_t limit = p.timeout_ns;
  unsigned long long* tr0 =
      (p.trace != nullptr && c < MOE_TRACE_MAX_CTAS) ? p.trace + static_cast<size_t>(c) * 4 : nullptr;
  unsigned long long* tr1 = tr0 ? p.trace + static_cast<size_t>(MOE_TRACE_MAX_CTAS + c) * 4 : nullptr;
  if (tr0 && tid == 0) tr0[0] = global_timer_ns();
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_w13);
    prefetch_tensormap(&tm_xs);
    prefetch_tensormap(&tm_xs64);
    prefetch_tensormap(&tm_w2);
    prefetch_tensormap(&tm_h);
    prefetch_tensormap(&tm_h64);
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait();

  // ------------------------------------------------ phase 0: routing, amax slice, zeroing
  for (int t = c * kWarps + warp; t < T; t += G * kWarps) {
    const float* src = p.logits + static_cast<size_t>(t) * E;
    int32_t* idr = p.ids + static_cast<size_t>(t) * k;
    float* wr = p.wts + static_cast<size_t>(t) * k;
    if (E <= 32) route_token_reg<1>(src, E, k, p.renorm, idr, wr, lane);
    else if (E <= 64) route_token_reg<2>(src, E, k, p.renorm, idr, wr, lane);
    else if (E <= 128) route_token_reg<4>(src, E, k, p.renorm, idr, wr, lane);
    else route_token_reg<8>(src, E, k, p.renorm, idr, wr, lane);
  }
  if (!kBF16) {
    const long long n8 = static_cast<long long>(T) * H / 8;
    const long long b0 = n8 * c / G, b1 = n8 * (c + 1) / G;
    const uint4* xv = reinterpret_cast<const uint4*>(p.x);
    float m = 0.f;
    for (long long i = b0 + tid; i < b1; i += kFusedThreads) m = absmax8(__ldg(xv + i), m);
    m = warp_max(m);
    if (lane == 0) sh.red[warp] = m;
  }
  {
    const long long gt = static_cast<long long>(c) * kFusedThreads + tid;
    const long long gs = static_cast<long long>(G) * kFusedThreads;
    float4* a4 = reinterpret_cast<float4*>(p.acc);
    const long long n4 = static_cast<long long>(T) * H / 4;
    for (long long i = gt; i < n4; i += gs) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = gt; i < p.n_tile_cnt; i += gs) p.tile_cnt[i] = 0;
    if (c == 0 && tid == 0) {
      ctrl->err = 0;
      ctrl->amax_h = 0u;
      for (int b = 0; b < 4; ++b) ctrl->bar[b] = 0u;
    }
  }
  __syncthreads();
  if (!kBF16 && tid == 0) {
    float a = 0.f;
    for (int w = 0; w < kWarps; ++w) a = fmaxf(a, sh.red[w]);
    p.amax_part[c] = a;
  }
  // nothing above waits on another CTA, so every CTA arrives here
  cg::this_grid().sync();

  // ------------------------------------------------ phase 1: counts, offsets, row tiles
  // (the ids and the amax partials are requested together: one round trip)
  float amax_x = 0.f;
  if (!kBF16 && warp == 1)
    for (int i = lane; i < G; i += 32) amax_x = fmaxf(amax_x, __ldcg(p.amax_part + i));
  for (int e = tid; e < E; e += kFusedThreads) {
    sh.cnt[e] = 0;
    sh.before[e] = 0;
  }
  __syncthreads();
  const int q0 = static_cast<int>(static_cast<long long>(P) * c / G);
  const int q1 = static_cast<int>(static_cast<long long>(P) * (c + 1) / G);
  for (int q0i = 0; q0i < P; q0i += 4 * kFusedThreads) {
    int ev[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = q0i + u * kFusedThreads + tid;
      ev[u] = q < P ? __ldcg(p.ids + q) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = q0i + u * kFusedThreads + tid;
      const int e = ev[u];
      if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
        atomicAdd(&sh.cnt[e], 1);
        if (q < q0) atomicAdd(&sh.before[e], 1);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // lane l owns experts 8l .. 8l+7; segments padded to 16 rows, each split
    // into ceil(padded / 128) equal row tiles (multiples of 16 rows)
    int pad[8], nt[8];
    int pad_sum = 0, nt_sum = 0, mx = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      const int cn = e < E ? sh.cnt[e] : 0;
      pad[i] = (cn + kAlignBlock - 1) / kAlignBlock * kAlignBlock;
      nt[i] = pad[i] > 0 ? (pad[i] + kRows - 1) / kRows : 0;
      const int per = nt[i] > 0 ? ((pad[i] + nt[i] - 1) / nt[i] + kAlignBlock - 1) / kAlignBlock * kAlignBlock : 0;
      mx = max(mx, per);
      pad_sum += pad[i];
      nt_sum += nt[i];
    }
    int pi = pad_sum, ni = nt_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(kFull, pi, o), b = __shfl_up_sync(kFull, ni, o);
      if (lane >= o) {
        pi += a;
        ni += b;
      }
    }
    int off = pi - pad_sum, first = ni - nt_sum;
    bool fits = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) {
        sh.off[e] = off;
        const int per = nt[i] > 0 ? ((pad[i] + nt[i] - 1) / nt[i] + kAlignBlock - 1) / kAlignBlock * kAlignBlock : 0;
        for (int j = 0; j < nt[i]; ++j) {
          if (first + j < kMaxTiles)
            sh.tiles[first + j] = make_int4(e, off + j * per, min(per, pad[i] - j * per) | (nt[i] << 12), first);
          else
            fits = false;
        }
      }
      off += pad[i];
      first += nt[i];
    }
    const unsigned all_fit = __ballot_sync(kFull, fits);
    const int total_rows = __shfl_sync(kFull, pi, 31);
    const int num_tiles = __shfl_sync(kFull, ni, 31);
    mx = static_cast<int>(__reduce_max_sync(kFull, static_cast<unsigned>(mx)));
    if (lane == 0) {
      sh.total_rows = total_rows;
      sh.tiles_ok = (all_fit == kFull && num_tiles <= kMaxTiles) ? 1 : 0;
      sh.num_tiles = sh.tiles_ok ? num_tiles : 0;
      sh.max_rows = mx;
    }
  } else if (warp == 1) {
    const float m = warp_max(amax_x);
    if (lane == 0) sh.s_x = kBF16 ? 1.f : scale_from_amax(m);
  }
  __syncthreads();
  if (c == 0) {
    if (p.counts_out != nullptr)
      for (int e = tid; e < E; e += kFusedThreads) p.counts_out[e] = sh.cnt[e];
    if (tid == 0) {
      ctrl->s_x = sh.s_x;
      ctrl->num_padded = sh.total_rows;
      ctrl->num_mtiles = sh.num_tiles;
      ctrl->max_tile_rows = sh.max_rows;
      if (!sh.tiles_ok) atomicOr(&ctrl->err, kDevErrRange);
    }
  }

  // pipeline: a stage holds 32 KB of weights and two 128-byte K chunks of the
  // largest row tile's token rows; as many stages as fit, at most four
  const int rows_b = min(kRows, max(16, sh.max_rows));
  const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(rows_b) * 256u;
  const int S = min(kMaxS, static_cast<int>(p.stage_smem / stage_bytes));
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.tfull[a], 1);
      mbar_init(&sh.tempty[a], kGemmEpiWarps);
    }
    mbar_init(&sh.never, 1);
    sh.abort_flag = 0;
    fence_mbarrier_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_slot;
  volatile int* abort_flag = &sh.abort_flag;

  const int ntl = sh.num_tiles;
  const int nbG = I / 128, KG = H / kElems;                 // gate/up: I/128 blocks of 2 x 128 rows
  const int nbD = H / 128, KD = (I / kElems + 1) / 2;       // down: two K chunks per stage
  const Sched sG = make_sched(ntl * nbG, KG, false, false);
  const Sched sD = make_sched(ntl * nbD, KD, false, false);
  const unsigned G_u = static_cast<unsigned>(G);
  const int hq_bar = kBF16 ? 1 : 2;  // counter after which the down GEMM's token rows are final

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();  // every weight block is read once
      uint32_t it = 0;
      bool ok = true;
      // gate/up weights of the first stages (the tile list is this CTA's own)
      uint32_t pre = 0;
      {
        SegIt sj = seg_begin(sG);
        Seg gj;
        while (pre < static_cast<uint32_t>(S) && seg_next(sG, sj, gj)) {
          const Tile t = decode_tile_of(sh.tiles, nbG, gj.tile);
          const int wrow = t.e * 2 * I + t.nb * 128;
          for (int kk = gj.k0; kk < gj.k1 && pre < static_cast<uint32_t>(S); ++kk, ++pre) {
            uint8_t* sa = stages + static_cast<size_t>(pre) * stage_bytes;
            mbar_arrive_expect_tx(&sh.full[pre], kABytes + static_cast<uint32_t>(t.n) * 128u);
            tma_load_2d_hint(sa, &tm_w13, &sh.full[pre], kk * kElems, wrow, pol);
            tma_load_2d_hint(sa + 16384, &tm_w13, &sh.full[pre], kk * kElems, wrow + I, pol);
          }
        }
      }
      // token rows: written by every CTA's epilogue warps before counter 0
      ok = grid_wait(&ctrl->bar[0], G_u, &ctrl->err, abort_flag, limit);
      if (tr0) tr0[1] = global_timer_ns();
      fence_proxy_async_global();
      {
        SegIt si = seg_begin(sG);
        Seg g;
        bool have = seg_next(sG, si, g);
        while (have) {
          const Tile t = decode_tile_of(sh.tiles, nbG, g.tile);
          const int wrow = t.e * 2 * I + t.nb * 128;
          for (int kk = g.k0; kk < g.k1; ++kk, ++it) {
            const uint32_t s = it % S;
            const uint32_t ph = (it / S) & 1u;
            uint8_t* sa = stages + static_cast<size_t>(s) * stage_bytes;
            if (it >= pre) {
              if (!ok || !mbar_wait(&sh.empty[s], ph ^ 1u, abort_flag, limit)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&sh.full[s], kABytes + static_cast<uint32_t>(t.n) * 128u);
              tma_load_2d_hint(sa, &tm_w13, &sh.full[s], kk * kElems, wrow, pol);
              tma_load_2d_hint(sa + 16384, &tm_w13, &sh.full[s], kk * kElems, wrow + I, pol);
            }
            // (stages issued before the counter wait get their rows here even
            // when it failed, so that every issued stage completes)
            load_rows(sa + kABytes, &tm_xs64, &tm_xs, &sh.full[s], kk * kElems, t.row0, t.n);
          }
          if (!ok) break;
          have = seg_next(sG, si, g);
        }
      }
      // down: weights are issued into the ring as it frees up; the token rows
      // (h codes) only once counter hq_bar says every CTA has written them
      if (ok) {
        bool rows_ready = false;
        PendingRows pend[kMaxS];
        int npend = 0;
        auto flush = [&]() {
          for (int i = 0; i < npend; ++i) {
            uint8_t* sb = stages + static_cast<size_t>(pend[i].s) * stage_bytes + kABytes;
            for (int ch = 0; ch < pend[i].n2; ++ch)
              load_rows(sb + ch * rows_b * 128, &tm_h64, &tm_h, &sh.full[pend[i].s],
                        pend[i].kc + ch * kElems, pend[i].row0, pend[i].n);
          }
          npend = 0;
        };
        SegIt si = seg_begin(sD);
        Seg g;
        bool have = seg_next(sD, si, g);
        while (have && ok) {
          const Tile t = decode_tile_of(sh.tiles, nbD, g.tile);
          const int wrow = t.e * H + t.nb * 128;
          for (int kk = g.k0; kk < g.k1; ++kk, ++it) {
            const uint32_t s = it % S;
            const uint32_t ph = (it / S) & 1u;
            uint8_t* sa = stages + static_cast<size_t>(s) * stage_bytes;
            if (!mbar_wait(&sh.empty[s], ph ^ 1u, abort_flag, limit)) {
              ok = false;
              break;
            }
            const int kc = kk * 2 * kElems;
            const int n2 = (kc + kElems < I) ? 2 : 1;
            mbar_arrive_expect_tx(&sh.full[s], static_cast<uint32_t>(n2) *
                                                   (16384u + static_cast<uint32_t>(t.n) * 128u));
            tma_load_2d_hint(sa, &tm_w2, &sh.full[s], kc, wrow, pol);
            if (n2 == 2) tma_load_2d_hint(sa + 16384, &tm_w2, &sh.full[s], kc + kElems, wrow, pol);
            pend[npend++] = PendingRows{static_cast<int>(s), t.row0, t.n, kc, n2};
            if (rows_ready) {
              flush();
            } else if (npend == S) {
              ok = grid_wait(&ctrl->bar[hq_bar], G_u, &ctrl->err, abort_flag, limit);
              if (tr1) tr1[1] = global_timer_ns();
              rows_ready = true;
              fence_proxy_async_global();
              flush();  // (also on failure: every issued stage completes)
              if (!ok) break;
            }
          }
          if (!ok) break;
          have = seg_next(sD, si, g);
        }
        if (npend > 0) {
          if (!rows_ready) {
            const bool w = grid_wait(&ctrl->bar[hq_bar], G_u, &ctrl->err, abort_flag, limit);
            if (tr1) tr1[1] = global_timer_ns();
            ok = ok && w;
            fence_proxy_async_global();
          }
          flush();
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(&ctrl->err, kDevErrTimeout);
        // let the copies already issued land before the CTA leaves
        const uint32_t n_iss = it > pre ? it : pre;
        const uint32_t n_back = n_iss < static_cast<uint32_t>(S) ? n_iss : static_cast<uint32_t>(S);
        for (uint32_t b = 1; b <= n_back; ++b) {
          const uint32_t i2 = n_iss - b;
          volatile int no_abort = 0;
          mbar_wait(&sh.full[i2 % S], (i2 / S) & 1u, &no_abort, 20000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, tt = 0;
      bool ok = true;
      if (p.debug & MOE_DEBUG_FORCE_TIMEOUT) ok = mbar_wait(&sh.never, 0, abort_flag, limit);
      for (int phase = 0; phase < 2 && ok; ++phase) {
        const Sched& sc = phase == 0 ? sG : sD;
        const int nb = phase == 0 ? nbG : nbD;
        SegIt si = seg_begin(sc);
        Seg g;
        bool have = seg_next(sc, si, g);
        bool first_stage = true;
        while (ok && have) {
          const int n = decode_tile_of(sh.tiles, nb, g.tile).n;
          const uint32_t a = tt & 1u;
          const uint32_t aph = (tt >> 1) & 1u;
          if (!mbar_wait(&sh.tempty[a], aph ^ 1u, abort_flag, limit)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t idesc = umma_idesc(kBF16, 128, n);
          const uint32_t d0 = tmem + a * 256u;
          for (int kk = g.k0; kk < g.k1; ++kk, ++it) {
            const uint32_t s = it % S;
            const uint32_t ph = (it / S) & 1u;
            if (!mbar_wait(&sh.full[s], ph, abort_flag, limit)) {
              ok = false;
              break;
            }
            if (first_stage) {
              unsigned long long* trs = phase == 0 ? tr0 : tr1;
              if (trs) trs[2] = global_timer_ns();
              first_stage = false;
            }
            tc_fence_after_sync();
            const uint32_t sa = smem_addr(stages + static_cast<size_t>(s) * stage_bytes);
            if (phase == 0) {
              // gate block and up block of the same 128 rows of I: two accumulators
              const uint64_t da0 = sdesc_kmajor_sw128(sa);
              const uint64_t da1 = sdesc_kmajor_sw128(sa + 16384);
              const uint64_t db = sdesc_kmajor_sw128(sa + kABytes);
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) {
                const uint32_t acc = (kk > g.k0 || k4 > 0) ? 1u : 0u;
                if (kBF16) {
                  umma_bf16(d0, da0 + 2 * k4, db + 2 * k4, idesc, acc);
                  umma_bf16(d0 + kRows, da1 + 2 * k4, db + 2 * k4, idesc, acc);
                } else {
                  umma_f8(d0, da0 + 2 * k4, db + 2 * k4, idesc, acc);
                  umma_f8(d0 + kRows, da1 + 2 * k4, db + 2 * k4, idesc, acc);
                }
              }
            } else {
              // two consecutive 128-byte K chunks into one accumulator
              const int n2 = (kk * 2 * kElems + kElems < I) ? 2 : 1;
              for (int ch = 0; ch < n2; ++ch) {
                const uint64_t da = sdesc_kmajor_sw128(sa + ch * 16384);
                const uint64_t db = sdesc_kmajor_sw128(sa + kABytes + ch * rows_b * 128);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                  const uint32_t acc = (kk > g.k0 || ch > 0 || k4 > 0) ? 1u : 0u;
                  if (kBF16) umma_bf16(d0, da + 2 * k4, db + 2 * k4, idesc, acc);
                  else umma_f8(d0, da + 2 * k4, db + 2 * k4, idesc, acc);
                }
              }
            }
            umma_commit(&sh.empty[s]);
          }
          if (!ok) break;
          umma_commit(&sh.tfull[a]);
          ++tt;
          have = seg_next(sc, si, g);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(&ctrl->err, kDevErrTimeout);
      }
    }
  } else {
    // ------------------------------------------------ epilogue warps (+ gather, h codes, output)
    const int etid = tid - 64;
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    const int c_begin = 16 * ((warp - 2) >> 2);  // the two warps of a quarter alternate chunks
    const int row_l = q * 32 + lane;
    bool ok = true;
    // place this CTA's chunk of pairs in expert order (ascending pair id
    // within an expert: earlier CTAs' pairs come first, see `before`)
    if (warp == 2) {
      for (int g0 = q0; g0 < q1; g0 += 32) {
        const int qq = g0 + lane;
        const bool in = qq < q1;
        const int e = in ? __ldcg(p.ids + qq) : -1;
        const bool valid = in && static_cast<unsigned>(e) < static_cast<unsigned>(E);
        const unsigned mask = __match_any_sync(kFull, valid ? e : -1);
        const int leader = __ffs(mask) - 1;
        int base = 0;
        if (valid && lane == leader) {
          base = sh.off[e] + sh.before[e];
          sh.before[e] += __popc(mask);
        }
        base = __shfl_sync(kFull, base, leader);
        const int at = base + __popc(mask & ((1u << lane) - 1u));
        if (in) sh.slot[qq - q0] = valid ? at : -1;
        if (valid) {
          p.sorted_ids[at] = qq;
          p.sorted_w[at] = __ldcg(p.wts + qq);
        }
        __syncwarp();
      }
    }
    named_barrier(kEpiBar, kEpiThreads);
    // the x rows of those pairs (E4M3 with s_x, or bf16), and the padding
    // rows of the experts this CTA owns (e = c mod G): zero rows, sentinel ids
    {
      const int nvec = kBF16 ? H / 8 : H / 16;  // 16-byte outputs per row
      uint4* xs = static_cast<uint4*>(p.xs);
      const E4m3Div dx = e4m3_div(sh.s_x);
      const int chunk = q1 - q0;
      const int n_items = chunk * nvec;
      for (int i0 = 0; i0 < n_items; i0 += 4 * static_cast<int>(kEpiThreads)) {
        uint4 v[4][2];
        int dst[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int idx = i0 + u * static_cast<int>(kEpiThreads) + etid;
          dst[u] = -1;
          if (idx < n_items) {
            const int i = idx / nvec, cv = idx - i * nvec;
            const int at = sh.slot[i];
            if (at >= 0) {
              dst[u] = at * nvec + cv;
              const uint4* src =
                  reinterpret_cast<const uint4*>(p.x + static_cast<size_t>((q0 + i) / k) * H);
              if (kBF16) {
                v[u][0] = __ldg(src + cv);
              } else {
                v[u][0] = __ldg(src + 2 * cv);
                v[u][1] = __ldg(src + 2 * cv + 1);
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (dst[u] < 0) continue;
          if (kBF16) {
            xs[dst[u]] = v[u][0];
          } else {
            const uint2 lo = quant8(v[u][0], dx);
            const uint2 hi = quant8(v[u][1], dx);
            xs[dst[u]] = make_uint4(lo.x, lo.y, hi.x, hi.y);
          }
        }
      }
      for (int e = c; e < E; e += G) {
        const int cn = sh.cnt[e];
        const int r0 = sh.off[e] + cn;
        const int r1 = sh.off[e] + (cn + kAlignBlock - 1) / kAlignBlock * kAlignBlock;
        for (int idx = etid; idx < (r1 - r0) * nvec; idx += kEpiThreads)
          xs[static_cast<size_t>(r0 + idx / nvec) * nvec + idx % nvec] = make_uint4(0, 0, 0, 0);
        for (int r = r0 + etid; r < r1; r += kEpiThreads) {
          p.sorted_ids[r] = P;
          p.sorted_w[r] = 0.f;
        }
      }
    }
    fence_proxy_async_global();  // the rows are read by other CTAs' TMA
    named_barrier(kEpiBar, kEpiThreads);
    if (etid == 0) {
      __threadfence();
      red_release_add(&ctrl->bar[0], 1u);
    }
    {
      int got = 1;
      if (etid == 0) got = grid_wait(&ctrl->bar[0], G_u, &ctrl->err, abort_flag, limit) ? 1 : 0;
      ok = named_barrier_and(kEpiBar, kEpiThreads, got != 0);
    }

    uint32_t tt = 0, n_chunks = 0;
    // ---------------- gate/up epilogue: h = SiLU(g s) (u s), running max |h|
    float amax = 0.f;
    if (ok) {
      const float act_s = sh.s_x;
      SegIt si = seg_begin(sG);
      Seg g, g1;
      bool have = seg_next(sG, si, g);
      Tile t = have ? decode_tile_of(sh.tiles, nbG, g.tile) : Tile{};
      SmallMeta mt = have ? small_meta(p, t, lane, p.w13_scale, false, P) : SmallMeta{};
      bool have1 = have && seg_next(sG, si, g1);
      Tile t1 = have1 ? decode_tile_of(sh.tiles, nbG, g1.tile) : Tile{};
      while (have) {
        const SmallMeta mt1 = have1 ? small_meta(p, t1, lane, p.w13_scale, false, P) : SmallMeta{};
        Seg g2;
        const bool have2 = have1 && seg_next(sG, si, g2);
        const Tile t2 = have2 ? decode_tile_of(sh.tiles, nbG, g2.tile) : Tile{};
        const uint32_t a = tt & 1u;
        const uint32_t aph = (tt >> 1) & 1u;
        int got = 0;
        if (lane == 0) got = mbar_wait(&sh.tfull[a], aph, abort_flag, limit) ? 1 : 0;
        got = __shfl_sync(kFull, got, 0);
        if (!named_barrier_and(kEpiBar, kEpiThreads, got != 0)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const float sc = act_s * mt.wsc;
        const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + a * 256u;
        const int col = t.nb * 128 + row_l;  // this lane's row of I
        const bool whole = (g.k0 == 0 && g.k1 == KG);
        bool finish = whole;
        int c_first = 0, c_last = 0;
        if (!whole) {
          // store this contributor's partial, then count arrivals on the tile
          c_first = owner_of(g.t0, sG.tail_total);
          c_last = owner_of(g.t0 + KG - 1, sG.tail_total);
          float* mine = part_slot_of(p.part, kRows, c, g.t0, sG.tail_total);
          for (int c0 = c_begin; c0 < t.n; c0 += 32) {
            float gg[16], v[16];
            tmem_ld16x2(tbase + c0, tbase + kRows + c0, gg, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              mine[static_cast<size_t>(c0 + j) * 128 + row_l] = gg[j];
              mine[static_cast<size_t>(kRows + c0 + j) * 128 + row_l] = v[j];
            }
          }
          __threadfence();
          named_barrier(kEpiBar, kEpiThreads);
          if (etid == 0) {
            int n_seg = 0;  // contributors: CTAs in [c_first, c_last] with a non-empty range
            for (int cc = c_first; cc <= c_last; ++cc)
              n_seg += range_begin(cc, sG.tail_total) < range_begin(cc + 1, sG.tail_total) ? 1 : 0;
            sh.s_last = (atomicAdd(p.tile_cnt + g.tile, 1) == n_seg - 1) ? 1 : 0;
          }
          named_barrier(kEpiBar, kEpiThreads);
          finish = sh.s_last != 0;
          if (finish) __threadfence();
        }
        if (finish) {
          for (int c0 = c_begin; c0 < t.n; c0 += 32) {
            const int pid_c = pick<4>(mt.pid, c0 >> 5);
            float gg[16], v[16];
            tmem_ld16x2(tbase + c0, tbase + kRows + c0, gg, v);
            if (!whole) {
              for (int cc = c_first; cc <= c_last; ++cc) {
                if (cc == c || range_begin(cc, sG.tail_total) == range_begin(cc + 1, sG.tail_total))
                  continue;
                const float* other = part_slot_of(p.part, kRows, cc, g.t0, sG.tail_total);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  gg[j] += __ldcg(other + static_cast<size_t>(c0 + j) * 128 + row_l);
                  v[j] += __ldcg(other + static_cast<size_t>(kRows + c0 + j) * 128 + row_l);
                }
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float gv = gg[j] * sc;
              const float uv = v[j] * sc;
              const float hv = __fdividef(gv, 1.f + __expf(-gv)) * uv;  // SiLU(g) * u
              const size_t at = static_cast<size_t>(t.row0 + c0 + j) * I + col;
              if (kBF16) {
                static_cast<__nv_bfloat16*>(p.h)[at] = __float2bfloat16_rn(hv);
              } else {
                // h stays fp32 until its per-tensor scale is known
                static_cast<float*>(p.h)[at] = hv;
                const int pid = __shfl_sync(kFull, pid_c, (c0 & 31) + j);
                if (pid < P) amax = fmaxf(amax, fabsf(hv));
              }
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.tempty[a]);
        ++tt;
        g = g1;
        t = t1;
        mt = mt1;
        have = have1;
        g1 = g2;
        t1 = t2;
        have1 = have2;
      }
    }
    if (tr0 && etid == 0) tr0[3] = global_timer_ns();
    // ---------------- all of h written: its scale, then its E4M3 codes
    float s_h = 1.f;
    if (ok) {
      if (!kBF16) {
        amax = warp_max(amax);
        if (lane == 0 && amax > 0.f) atomicMax(&ctrl->amax_h, __float_as_uint(amax));
      }
      fence_proxy_async_global();  // bf16: h itself is the down GEMM's TMA operand
      named_barrier(kEpiBar, kEpiThreads);
      if (etid == 0) {
        __threadfence();
        red_release_add(&ctrl->bar[1], 1u);
      }
      int got = 1;
      if (etid == 0) got = grid_wait(&ctrl->bar[1], G_u, &ctrl->err, abort_flag, limit) ? 1 : 0;
      ok = named_barrier_and(kEpiBar, kEpiThreads, got != 0);
      if (tr1 && etid == 0) tr1[0] = global_timer_ns();
    }
    if (ok && !kBF16) {
      s_h = scale_from_amax(__uint_as_float(ld_acquire(&ctrl->amax_h)));
      if (c == 0 && etid == 0) ctrl->s_h = s_h;
      const E4m3Div dh = e4m3_div(s_h);
      const long long n16 = static_cast<long long>(sh.total_rows) * I / 16;
      const float4* src = static_cast<const float4*>(p.h);
      uint4* dst = reinterpret_cast<uint4*>(p.hq);
      const long long stride = static_cast<long long>(G) * kEpiThreads;
      for (long long i0 = static_cast<long long>(c) * kEpiThreads + etid; i0 < n16; i0 += 4 * stride) {
        float4 v[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const long long i = i0 + u * stride;
          if (i < n16) {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[u][j] = __ldcg(src + 4 * i + j);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const long long i = i0 + u * stride;
          if (i < n16)
            dst[i] = make_uint4(quant4(v[u][0], dh), quant4(v[u][1], dh),
                                quant4(v[u][2], dh), quant4(v[u][3], dh));
        }
      }
      fence_proxy_async_global();  // the codes are read by other CTAs' TMA
      named_barrier(kEpiBar, kEpiThreads);
      if (etid == 0) {
        __threadfence();
        red_release_add(&ctrl->bar[2], 1u);
      }
    }
    // ---------------- down epilogue: y s topk_weight added into the fp32 rows
    if (ok) {
      float* wstage = staging + static_cast<size_t>(warp - 2) * 2 * 16 * 32;
      SegIt si = seg_begin(sD);
      Seg g, g1;
      bool have = seg_next(sD, si, g);
      Tile t = have ? decode_tile_of(sh.tiles, nbD, g.tile) : Tile{};
      SmallMeta mt = have ? small_meta(p, t, lane, p.w2_scale, true, P) : SmallMeta{};
      bool have1 = have && seg_next(sD, si, g1);
      Tile t1 = have1 ? decode_tile_of(sh.tiles, nbD, g1.tile) : Tile{};
      while (have) {
        const SmallMeta mt1 = have1 ? small_meta(p, t1, lane, p.w2_scale, true, P) : SmallMeta{};
        Seg g2;
        const bool have2 = have1 && seg_next(sD, si, g2);
        const Tile t2 = have2 ? decode_tile_of(sh.tiles, nbD, g2.tile) : Tile{};
        const uint32_t a = tt & 1u;
        const uint32_t aph = (tt >> 1) & 1u;
        int got = 0;
        if (lane == 0) got = mbar_wait(&sh.tfull[a], aph, abort_flag, limit) ? 1 : 0;
        got = __shfl_sync(kFull, got, 0);
        if (!named_barrier_and(kEpiBar, kEpiThreads, got != 0)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const float sc = s_h * mt.wsc;
        const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + a * 256u;
        for (int c0 = c_begin; c0 < t.n; c0 += 32) {
          float y[16];
          tmem_ld16(tbase + c0, y);
          float* buf = wstage + (n_chunks & 1u) * 16 * 32;
          // lane j < 16 handles token column c0 + j
          const int pid = __shfl_sync(kFull, pick<4>(mt.pid, c0 >> 5), (c0 & 31) + (lane & 15));
          const float wscale = sc * __shfl_sync(kFull, pick<4>(mt.w, c0 >> 5), (c0 & 31) + (lane & 15));
          if (lane < 16) bulk_wait_read<1>();  // this buffer's reductions of two chunks ago have read it
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 16; ++j) buf[j * 32 + lane] = y[j] * __shfl_sync(kFull, wscale, j);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane < 16) {
            if (pid < P)
              bulk_reduce_add_f32(p.acc + static_cast<size_t>(pid / k) * H + t.nb * 128 + q * 32,
                                  buf + lane * 32, 128);
            bulk_commit();
          }
          ++n_chunks;
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.tempty[a]);
        ++tt;
        g = g1;
        t = t1;
        mt = mt1;
        have = have1;
        g1 = g2;
        t1 = t2;
        have1 = have2;
      }
    }
    if (lane < 16) bulk_wait_all();  // this thread's reductions have landed
    // ---------------- every reduction landed: the bf16 output
    if (ok) {
      fence_proxy_async_global();  // the bulk reductions are async-proxy writes
      named_barrier(kEpiBar, kEpiThreads);
      if (etid == 0) {
        __threadfence();
        red_release_add(&ctrl->bar[3], 1u);
      }
      int got = 1;
      if (etid == 0) got = grid_wait(&ctrl->bar[3], G_u, &ctrl->err, abort_flag, limit) ? 1 : 0;
      ok = named_barrier_and(kEpiBar, kEpiThreads, got != 0);
    }
    if (ok) {
      const long long n8 = static_cast<long long>(T) * H / 8;
      const float4* a4 = reinterpret_cast<const float4*>(p.acc);
      uint4* o = reinterpret_cast<uint4*>(p.out);
      const long long stride = static_cast<long long>(G) * kEpiThreads;
      for (long long i0 = static_cast<long long>(c) * kEpiThreads + etid; i0 < n8; i0 += 4 * stride) {
        float4 uv[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const long long i = i0 + u * stride;
          if (i < n8) {
            uv[u][0] = __ldcg(a4 + 2 * i);
            uv[u][1] = __ldcg(a4 + 2 * i + 1);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const long long i = i0 + u * stride;
          if (i >= n8) continue;
          __nv_bfloat162 b0 = __floats2bfloat162_rn(uv[u][0].x, uv[u][0].y);
          __nv_bfloat162 b1 = __floats2bfloat162_rn(uv[u][0].z, uv[u][0].w);
          __nv_bfloat162 b2 = __floats2bfloat162_rn(uv[u][1].x, uv[u][1].y);
          __nv_bfloat162 b3 = __floats2bfloat162_rn(uv[u][1].z, uv[u][1].w);
          uint4 r;
          r.x = *reinterpret_cast<uint32_t*>(&b0);
          r.y = *reinterpret_cast<uint32_t*>(&b1);
          r.z = *reinterpret_cast<uint32_t*>(&b2);
          r.w = *reinterpret_cast<uint32_t*>(&b3);
          o[i] = r;
        }
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      atomicOr(&ctrl->err, kDevErrTimeout);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tr1 && tid == 0) {
    __threadfence();
    tr1[3] = global_timer_ns();
  }
}

template <bool kBF16>
cudaError_t launch_small_one(const FusedParams& p, const CUtensorMap& a, const CUtensorMap& b,
                             const CUtensorMap& b64, const CUtensorMap& a2, const CUtensorMap& h,
                             const CUtensorMap& h64, int grid, cudaStream_t st) {
  static thread_local int configured_device = -1;
  static thread_local size_t dyn = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaFuncAttributes fa{};
    cudaError_t e = checked(cudaFuncGetAttributes(&fa, moe_fused_small_kernel<kBF16>), "func attributes");
    if (e != cudaSuccess) return e;
    dyn = kSmemLimit - fa.sharedSizeBytes;
    e = checked(cudaFuncSetAttribute(moe_fused_small_kernel<kBF16>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn)),
                "smem attribute");
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  FusedParams q = p;
  q.stage_smem = static_cast<unsigned>(dyn - 1024 - kStaging);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  // the CTAs wait on one another: all of them must be resident at once
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return checked(cudaLaunchKernelEx(&cfg, moe_fused_small_kernel<kBF16>, q, a, b, b64, a2, h, h64),
                 "cooperative kernel launch");
}

}  // namespace

bool fused_small_supported(int device) {
  static int cached[64];
  static bool have[64] = {};
  if (device < 0 || device >= 64) return false;
  if (!have[device]) {
    int coop = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    cached[device] = (coop != 0 && optin >= kSmemLimit) ? 1 : 0;
    have[device] = true;
  }
  return cached[device] != 0;
}

cudaError_t launch_fused_small(const FusedParams& p, const CUtensorMap& tm_w13,
                               const CUtensorMap& tm_xs, const CUtensorMap& tm_xs64,
                               const CUtensorMap& tm_w2, const CUtensorMap& tm_h,
                               const CUtensorMap& tm_h64, int grid, cudaStream_t st) {
  if (p.w13_scale == nullptr)
    return launch_small_one<true>(p, tm_w13, tm_xs, tm_xs64, tm_w2, tm_h, tm_h64, grid, st);
  return launch_small_one<false>(p, tm_w13, tm_xs, tm_xs64, tm_w2, tm_h, tm_h64, grid, st);
}

}  // namespace moe
