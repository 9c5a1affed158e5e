// Grouped expert GEMMs on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Operand placement follows the Swap-AB idea of "Amazon SageMaker AI 上的
// Mixture-of-Experts 内核工程优化" (section "Swap-AB for WGMMA utilization",
// and the digest page's B^T[N,K] x A^T[K,M] -> C^T[N,M]): the expert weight
// block (128 output rows) is the MMA's A operand and fills the M = 128 slot
// (128 TMEM lanes); the tokens routed to the expert are the B operand, N =
// 16..128 columns.  When an expert sees one token (decode) the MMA still does
// useful work on all 128 lanes, and the weight stream is what the kernel
// waits on.
//
// Work split: a tile is (row tile of one expert's tokens) x (128-row weight
// block) with K/128B steps; tiles of one expert are ordered weight-block-major
// so a weight block serves all of the expert's row tiles back to back.  When
// tiles share data through L2 (prefill) full waves of whole tiles go
// round-robin and only the last partial wave is split over the CTAs
// (stream-K); with nothing to share (decode) the whole (tile, K step) space is
// split, so every SM streams the same number of weight bytes.  A tile cut by a
// CTA boundary is finished by its last contributor: in the down projection the
// partial sums simply add into the combine buffer (the combine is linear); in
// the gate/up projection every contributor stores its partial accumulators and
// the last to arrive (per-tile counter) adds them and runs SiLU*up.
//
// Warp roles (one persistent CTA per SM):
//   warp 0      TMA producer: weight block(s) + token tile per K step into a
//               ring of shared-memory stages (128-byte swizzle, K-major);
//   warp 1      allocates TMEM and issues tcgen05.mma (one thread), commits
//               stage release and accumulator-ready barriers;
//   warps 2..9  epilogue (two warps per TMEM lane quarter): tcgen05.ld of the
//               accumulator, then either
//               gate/up:  h = SiLU(g * s) * (u * s) -> fp32 (FP8 path, with a
//                         running amax|h|) or bf16 (bf16 path)
//               down:     y * s * topk_weight added into the fp32 combine
//                         buffer with bulk asynchronous reductions staged in
//                         shared memory, or written as bf16 rows at the
//                         pairs' aligned rows (tokens in M: staged in shared
//                         memory and written with TMA tensor stores).
// The accumulator is double-buffered in TMEM when it fits, so the epilogue of
// one segment overlaps the MMAs of the next.  Every wait is bounded; on
// timeout the CTA records kDevErrTimeout and leaves.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gemm_sched.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kSmemLimit = 232448;  // 227 KB opt-in per CTA
constexpr int kSmemSlack = 1024 + 256;
constexpr int kMaxStages = 12;  // 2 * 12 + 5 barriers + 3 words fit the 256-byte area
// Gate/up stages (32 KB of weights each) beyond 4 were measured to slow the
// decode weight stream: more requests in flight per SM than HBM rewards.
constexpr int kMaxStagesGateUp = 4;
constexpr int kMaxStagesDown = 12;
constexpr uint32_t kEpiBarrier = 1;  // named barrier of the 4 epilogue warps
constexpr uint32_t kEpiThreads = 32 * kGemmEpiWarps;

__device__ __forceinline__ Tile decode_tile(const GemmParams& p, int u) {
  return decode_tile_of(p.mtiles, p.nb_count, u);
}

// Epilogue metadata of a tile.  Swap: lane l holds the pair ids and router
// weights of columns l + 32 i, i < N (N = 8 covers the 256-column wide
// tiles).  Unswapped: the thread's lane is token row row_l of the tile and
// entry 0 holds it.  wsc: the expert's weight scale.
template <int N>
struct Meta {
  int pid[N];
  float w[N];
  float wsc;
};

template <bool kBF16, bool kSwiGLU, bool kTokM, int N>
__device__ __forceinline__ Meta<N> load_meta(const GemmParams& p, const Tile& t, int lane,
                                             int row_l) {
  Meta<N> m;
#pragma unroll
  for (int s4 = 0; s4 < N; ++s4) {
    const int c = kTokM ? row_l : s4 * 32 + lane;
    const bool in = (kTokM ? s4 == 0 : true) && c < t.n;
    m.pid[s4] = in ? p.sorted_ids[t.row0 + c] : p.P;
    m.w[s4] = (!kSwiGLU && in) ? p.sorted_w[t.row0 + c] : 0.f;
  }
  m.wsc = kBF16 ? 1.f : p.w_scale[t.e];
  return m;
}

__device__ __forceinline__ float* part_slot(const GemmParams& p, int c, long long t0,
                                            long long total) {
  return part_slot_of(p.part, p.bn_max, c, t0, total);
}

// kTokM selects the unswapped placement (the ablation of the operand swap):
// the 128-row token tile is the A operand in the M slot and the weight block
// is B with N = 128 weight rows; lanes then hold tokens and TMEM columns hold
// weight rows.  kPair (down projection, unswapped): a tile covers two
// consecutive 128-row weight blocks against one token tile, one N = 256 MMA
// per K slice (the two blocks are contiguous in the stage, the two
// accumulators in TMEM), so the token bytes serve twice the FLOPs and the
// token operand is read from shared memory once per 256 columns.
template <bool kBF16, bool kSwiGLU, bool kTokM, bool kPair>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_b64,
                    const __grid_constant__ CUtensorMap tm_o) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // Pipeline depth from the largest row tile of this call (written by the
  // alignment kernel two or more launches back, see below): a stage holds the
  // weight block(s) and that many token rows, and as many stages as fit are
  // used, so decode (tiles of a few rows) keeps more weight bytes in flight.
  constexpr bool kTwoB = kSwiGLU || kPair;  // two weight blocks per stage
  constexpr uint32_t kABytes = kTwoB ? 32768u : 16384u;
  const int max_rows = p.wide ? p.ctrl->max_tile_rows_w : p.ctrl->max_tile_rows;
  const int rows_b = kTokM ? 128 : min(p.bn_max, max(16, max_rows));
  const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(rows_b) * 128u;
  const int S = min(kSwiGLU ? kMaxStagesGateUp : kMaxStagesDown,
                    static_cast<int>(p.stage_smem / stage_bytes));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* never = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_last = abort_flag + 1;  // "this CTA finishes the split tile" flag
  // down projection: 4 KB of staging per epilogue warp (1024-byte aligned,
  // after the barriers): two 16-column x 32-row fp32 buffers for the bulk
  // reductions into the combine buffer, or 32 bf16 rows of 128 bytes in the
  // 128-byte swizzle for the TMA stores of rows per pair
  uint8_t* stage_epi = smem + static_cast<size_t>(S) * stage_bytes + 1024;
  float* stage_out = reinterpret_cast<float*>(stage_epi);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned long long* trace =
      (p.trace != nullptr && blockIdx.x < MOE_TRACE_MAX_CTAS) ? p.trace + blockIdx.x * 4 : nullptr;
  if (trace && threadIdx.x == 0) trace[0] = global_timer_ns();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, kGemmEpiWarps);
    }
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_b);
    prefetch_tensormap(&tm_b64);
    if (kTokM && !kSwiGLU && p.pair_out != nullptr) prefetch_tensormap(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Everything above overlaps the previous kernel.  The weights are inputs of
  // the call, so the producer also puts the first stages' weight blocks in
  // flight before that kernel has finished (below); the row-tile list it reads
  // for that was written two or more kernels back, and every kernel of the
  // library signals its dependents only after its own wait, so its writers
  // have completed.  All other threads wait here.
  const bool early_producer = (warp == 0 && lane == 0);
  if (!early_producer) {
    pdl_wait();
    pdl_trigger();
  }
  if (trace && threadIdx.x == 0) trace[1] = global_timer_ns();

  const int K = p.k_steps;
  const int tiles = (p.wide ? p.ctrl->num_mtiles_w : p.ctrl->num_mtiles) * p.nb_count;
  const Sched sch = make_sched(tiles, K, p.weights_evict_first == 0,
                               !kSwiGLU && p.pair_out != nullptr);
  const uint64_t limit = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      // decode: a weight block is read once, keep it from displacing reused
      // lines; prefill: several row tiles of an expert reuse it from L2
      const uint64_t pol_w = p.weights_evict_first ? policy_evict_first() : policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      SegIt si = seg_begin(sch);
      Seg g;
      // weight blocks of the first S stages (fresh stages: no wait on `empty`)
      uint32_t pre = 0;
      {
        SegIt sj = si;
        Seg gj;
        while (pre < static_cast<uint32_t>(S) && seg_next(sch, sj, gj)) {
          const Tile t = decode_tile(p, gj.tile);
          const int wrow = t.e * p.rows_per_expert + t.nb * p.wblock_rows;
          for (int kk = gj.k0; kk < gj.k1 && pre < static_cast<uint32_t>(S); ++kk, ++pre) {
            uint8_t* sa = smem + static_cast<size_t>(pre) * stage_bytes;
            mbar_arrive_expect_tx(full + pre, kABytes + static_cast<uint32_t>(kTokM ? 128 : t.n) * 128u);
            const int kc = kk * p.k_elems;
            tma_load_2d_hint(sa, &tm_a, full + pre, kc, wrow, pol_w);
            if (kTwoB)
              tma_load_2d_hint(sa + 16384, &tm_a, full + pre, kc, wrow + p.up_offset, pol_w);
          }
        }
      }
      // token rows are the previous kernels' output
      pdl_wait();
      pdl_trigger();
      // the next segment's tile is fetched while this one's stages are issued
      bool have = seg_next(sch, si, g);
      Tile t = have ? decode_tile(p, g.tile) : Tile{};
      bool bad_rows = false;
      while (ok && have) {
        if (!kTokM && t.n > rows_b) {
          // a tile wider than the stage (the alignment kernels write none):
          // stop and report instead of writing past the stage
          bad_rows = true;
          ok = false;
          break;
        }
        Seg gn;
        const bool have_n = seg_next(sch, si, gn);
        const Tile tn = have_n ? decode_tile(p, gn.tile) : Tile{};
        const int wrow = t.e * p.rows_per_expert + t.nb * p.wblock_rows;
        for (int kk = g.k0; kk < g.k1; ++kk, ++it) {
          const uint32_t s = it % S;
          const uint32_t ph = (it / S) & 1u;
          uint8_t* sa = smem + static_cast<size_t>(s) * stage_bytes;
          uint8_t* sb = sa + kABytes;
          const int kc = kk * p.k_elems;
          if (it >= pre) {
            if (!mbar_wait(empty + s, ph ^ 1u, abort_flag, limit)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full + s, kABytes + static_cast<uint32_t>(kTokM ? 128 : t.n) * 128u);
            tma_load_2d_hint(sa, &tm_a, full + s, kc, wrow, pol_w);
            if (kTwoB) tma_load_2d_hint(sa + 16384, &tm_a, full + s, kc, wrow + p.up_offset, pol_w);
          }
          if (kTokM) {
            // tokens fill the M = 128 slot: 128 rows from the tile's first row
            // (rows past the tile belong to other tiles and are not stored;
            // rows past the buffer read as zero)
            tma_load_2d(sb, &tm_b64, full + s, kc, t.row0);
            tma_load_2d(sb + 64 * 128, &tm_b64, full + s, kc, t.row0 + 64);
          } else {
            // token rows: 64-row boxes, then 16-row boxes for the remainder
            int j = 0;
            for (; j + 64 <= t.n; j += 64) tma_load_2d(sb + j * 128, &tm_b64, full + s, kc, t.row0 + j);
            for (; j < t.n; j += 16) tma_load_2d(sb + j * 128, &tm_b, full + s, kc, t.row0 + j);
          }
        }
        g = gn;
        t = tn;
        have = have_n;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(&p.ctrl->err, bad_rows ? kDevErrRange : kDevErrTimeout);
        // let the copies already issued land before the CTA leaves (stages
        // [0, pre) had their weights issued before the loop; a stage whose
        // token rows never went out ends its wait at the limit)
        const uint32_t n_iss = it > pre ? it : pre;
        const uint32_t n_back = n_iss < static_cast<uint32_t>(S) ? n_iss : static_cast<uint32_t>(S);
        for (uint32_t b = 1; b <= n_back; ++b) {
          const uint32_t i2 = n_iss - b;
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
      SegIt si = seg_begin(sch);
      Seg g;
      bool have = seg_next(sch, si, g);
      int n_cur = have ? (kTokM ? 128 : decode_tile(p, g.tile).n) : 0;
      while (ok && have) {
        const int k0 = g.k0, k1 = g.k1;
        Seg gn;
        const bool have_n = seg_next(sch, si, gn);
        // the next tile's width (only the swap needs it) is fetched meanwhile
        const int n_next = (have_n && !kTokM) ? decode_tile(p, gn.tile).n : 128;
        const uint32_t a = tt % static_cast<uint32_t>(p.num_acc);
        const uint32_t aph = (tt / static_cast<uint32_t>(p.num_acc)) & 1u;
        if (!mbar_wait(tempty + a, aph ^ 1u, abort_flag, limit)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        // tokens in M with two weight blocks: one N = 256 MMA over both blocks
        // (contiguous in the stage) into both accumulators (contiguous in TMEM)
        constexpr bool kWideN = kTokM && kPair;
        const uint32_t idesc = umma_idesc(kBF16, 128, kWideN ? 256 : n_cur);
        const uint32_t d0 = tmem + a * static_cast<uint32_t>(p.acc_stride);
        const uint32_t d1 = d0 + static_cast<uint32_t>(p.bn_max);
        for (int kk = k0; kk < k1; ++kk, ++it) {
          const uint32_t s = it % S;
          const uint32_t ph = (it / S) & 1u;
          if (!mbar_wait(full + s, ph, abort_flag, limit)) {
            ok = false;
            break;
          }
          if (trace && it == 0) trace[2] = global_timer_ns();
          tc_fence_after_sync();
          const uint32_t sa = smem_addr(smem + static_cast<size_t>(s) * stage_bytes);
          const uint64_t da0 = sdesc_kmajor_sw128(sa);
          const uint64_t da1 = sdesc_kmajor_sw128(sa + 16384);
          const uint64_t db = sdesc_kmajor_sw128(sa + kABytes);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint32_t acc = (kk > k0 || k4 > 0) ? 1u : 0u;
            // +2 in the start-address field = +32 bytes of K inside the swizzle atom
            // swap: A = weight block, B = tokens; unswapped: A = tokens, B = weights
            const uint64_t a0 = kTokM ? db : da0, b0 = kTokM ? da0 : db;
            const uint64_t a1 = kTokM ? db : da1, b1 = kTokM ? da1 : db;
            if (kBF16) {
              umma_bf16(d0, a0 + 2 * k4, b0 + 2 * k4, idesc, acc);
              if (kTwoB && !kWideN) umma_bf16(d1, a1 + 2 * k4, b1 + 2 * k4, idesc, acc);
            } else {
              umma_f8(d0, a0 + 2 * k4, b0 + 2 * k4, idesc, acc);
              if (kTwoB && !kWideN) umma_f8(d1, a1 + 2 * k4, b1 + 2 * k4, idesc, acc);
            }
          }
          umma_commit(empty + s);
        }
        if (!ok) break;
        umma_commit(tfull + a);
        ++tt;
        g = gn;
        have = have_n;
        n_cur = n_next;
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(&p.ctrl->err, kDevErrTimeout);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (4 warps)
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    // the two warps of a quarter split a tile's 16-column chunks: this one
    // takes chunks c0 = 16 * (2 m + half)
    const int half = (warp - 2) >> 2;
    const int c_begin = 16 * half;
    const int row_l = q * 32 + lane;
    float act_s = 1.f;
    if (!kBF16) act_s = p.act_scale_sel == 1 ? p.ctrl->s_x : p.ctrl->s_h;
    float amax = 0.f;
    uint32_t n_chunks = 0;  // combine staging chunks issued by this warp
    uint32_t tt = 0;
    bool ok = true;
    // Metadata runs ahead: the tile list entry two segments ahead and the
    // pair ids / weights one segment ahead are in flight while a tile is
    // processed, so no tile starts on a chain of dependent global loads.
    SegIt si = seg_begin(sch);
    Seg g, g1;
    bool have = seg_next(sch, si, g);
    Tile t = have ? decode_tile(p, g.tile) : Tile{};
    // swap: up to 32 x kMetaN columns per tile (wide gate/up tiles have 256)
    constexpr int kMetaN = (kSwiGLU && !kTokM) ? 8 : 4;
    Meta<kMetaN> mt = have ? load_meta<kBF16, kSwiGLU, kTokM, kMetaN>(p, t, lane, row_l)
                           : Meta<kMetaN>{};
    bool have1 = have && seg_next(sch, si, g1);
    Tile t1 = have1 ? decode_tile(p, g1.tile) : Tile{};
    while (have) {
      const int k0 = g.k0, k1 = g.k1;
      const Meta<kMetaN> mt1 =
          have1 ? load_meta<kBF16, kSwiGLU, kTokM, kMetaN>(p, t1, lane, row_l) : Meta<kMetaN>{};
      Seg g2;
      const bool have2 = have1 && seg_next(sch, si, g2);
      const Tile t2 = have2 ? decode_tile(p, g2.tile) : Tile{};
      const uint32_t a = tt % static_cast<uint32_t>(p.num_acc);
      const uint32_t aph = (tt / static_cast<uint32_t>(p.num_acc)) & 1u;
      const int(&cpid)[kMetaN] = mt.pid;
      const float(&cw)[kMetaN] = mt.w;
      const float wsc = mt.wsc;
      int got = 0;
      if (lane == 0) got = mbar_wait(tfull + a, aph, abort_flag, limit) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      // all epilogue warps take the same branch (they share named barriers below)
      if (!named_barrier_and(kEpiBarrier, kEpiThreads, got != 0)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float sc = act_s * wsc;
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                             a * static_cast<uint32_t>(p.acc_stride);
      const int col = t.nb * 128 + row_l;  // swap: this lane's output row of the block
      const int ncols = kTokM ? 128 : t.n;  // accumulator columns in use
      // unswapped: this thread's token row, if it belongs to the tile
      const bool row_ok = kTokM && row_l < t.n;
      if (kSwiGLU) {
        const bool whole = (k0 == 0 && k1 == K);
        bool finish = whole;
        const long long t0 = g.t0;  // split tiles lie in the tail
        int c_first = 0, c_last = 0;
        if (!whole) {
          // store this contributor's partial, then count arrivals on the tile
          c_first = owner_of(t0, sch.tail_total);
          c_last = owner_of(t0 + K - 1, sch.tail_total);
          float* mine = part_slot(p, blockIdx.x, t0, sch.tail_total);
          for (int c0 = c_begin; c0 < ncols; c0 += 32) {
            float gg[16], v[16];
            tmem_ld16x2(tbase + c0, tbase + p.bn_max + c0, gg, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              mine[static_cast<size_t>(c0 + j) * 128 + row_l] = gg[j];
              mine[static_cast<size_t>(p.bn_max + c0 + j) * 128 + row_l] = v[j];
            }
          }
          __threadfence();
          named_barrier(kEpiBarrier, kEpiThreads);
          if (threadIdx.x == 64) {
            // contributors: CTAs in [c_first, c_last] whose range is not empty
            int n_seg = 0;
            for (int c = c_first; c <= c_last; ++c)
              n_seg += range_begin(c, sch.tail_total) < range_begin(c + 1, sch.tail_total) ? 1 : 0;
            *s_last = (atomicAdd(p.tile_cnt + g.tile, 1) == n_seg - 1) ? 1 : 0;
          }
          named_barrier(kEpiBarrier, kEpiThreads);
          finish = *s_last != 0;
          if (finish) __threadfence();
        }
        if (finish) {
          for (int c0 = c_begin; c0 < ncols; c0 += 32) {
            const int pid_c = pickn<kMetaN>(cpid, c0 >> 5);  // swap: column (c0 & 31) + lane of this block
            float gg[16], v[16];
            tmem_ld16x2(tbase + c0, tbase + p.bn_max + c0, gg, v);
            if (!whole) {
              for (int c = c_first; c <= c_last; ++c) {
                if (c == static_cast<int>(blockIdx.x) ||
                    range_begin(c, sch.tail_total) == range_begin(c + 1, sch.tail_total))
                  continue;
                const float* other = part_slot(p, c, t0, sch.tail_total);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  gg[j] += __ldcg(other + static_cast<size_t>(c0 + j) * 128 + row_l);
                  v[j] += __ldcg(other + static_cast<size_t>(p.bn_max + c0 + j) * 128 + row_l);
                }
              }
            }
            float hv[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float gv = gg[j] * sc;
              const float uv = v[j] * sc;
              hv[j] = __fdividef(gv, 1.f + __expf(-gv)) * uv;  // SiLU(g) * u
            }
            // bf16 weights: h feeds the bf16 down-projection MMA directly.
            // FP8: h stays fp32 until its per-tensor scale is known; an
            // intermediate bf16 rounding would move values across E4M3
            // rounding boundaries and cost percent-level output error.
            if (kTokM) {
              if (row_ok) {
                // 16 consecutive h values of one token row
                const size_t at = static_cast<size_t>(t.row0 + row_l) * p.ldh + t.nb * 128 + c0;
                if (kBF16) {
                  uint4 o[2];
                  uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
                  for (int j = 0; j < 8; ++j) {
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(hv[2 * j], hv[2 * j + 1]);
                    ow[j] = *reinterpret_cast<uint32_t*>(&b2);
                  }
                  uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.h_out) + at);
                  dst[0] = o[0];
                  dst[1] = o[1];
                } else {
                  float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.h_out) + at);
#pragma unroll
                  for (int j = 0; j < 4; ++j)
                    dst[j] = make_float4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]);
                  if (cpid[0] < p.P) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(hv[j]));
                  }
                }
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const size_t at = static_cast<size_t>(t.row0 + c0 + j) * p.ldh + col;
                if (kBF16) {
                  static_cast<__nv_bfloat16*>(p.h_out)[at] = __float2bfloat16_rn(hv[j]);
                } else {
                  static_cast<float*>(p.h_out)[at] = hv[j];
                  const int pid = __shfl_sync(0xffffffffu, pid_c, (c0 & 31) + j);
                  if (pid < p.P) amax = fmaxf(amax, fabsf(hv[j]));
                }
              }
            }
          }
        }
      } else if (p.pair_out != nullptr && kTokM) {
        // large batches, tokens in M: y * s * topk_weight as bf16 at the
        // tile's aligned rows (tiles are whole here, see the range split; the
        // token sum comes after).  Per weight block this warp takes 64
        // columns of its 32 rows, stages them as 128-byte rows in the
        // 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r & 7), no
        // bank conflicts) and stores them with one TMA box per 16 rows.  Row
        // tiles are multiples of 16 rows: a box is inside the tile or not
        // stored (its rows belong to the next tile).  Padding rows carry
        // router weight 0.
        uint8_t* wst = stage_epi + static_cast<size_t>(warp - 2) * 4096;
        const float w_r = sc * cw[0];
        const int c_lo = 64 * half;
        const int r0 = q * 32;
        for (int b2i = 0; b2i < (kPair ? 2 : 1); ++b2i) {
          float y[4][16];
          const uint32_t tb = tbase + static_cast<uint32_t>(b2i * p.bn_max + c_lo);
          tmem_ld16x2(tb, tb + 16, y[0], y[1]);
          tmem_ld16x2(tb + 32, tb + 48, y[2], y[3]);
          if (lane == 0) bulk_wait_read<0>();  // the previous box has left the buffer
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float* yy = &y[c >> 1][(c & 1) * 8];
            uint4 o;
            uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int j2 = 0; j2 < 4; ++j2) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(yy[2 * j2] * w_r, yy[2 * j2 + 1] * w_r);
              ow[j2] = *reinterpret_cast<uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(wst + lane * 128 + ((c ^ (lane & 7)) << 4)) = o;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int col0 = t.nb * p.wblock_rows + b2i * 128 + c_lo;
            if (r0 < t.n) tma_store_2d(&tm_o, wst, col0, t.row0 + r0);
            if (r0 + 16 < t.n) tma_store_2d(&tm_o, wst + 2048, col0, t.row0 + r0 + 16);
            bulk_commit();
          }
        }
      } else if (p.pair_out != nullptr) {
        // large batches, weights in M: y * s * topk_weight as bf16 at the
        // pair's aligned row (the tile's column), 32 consecutive output
        // columns per store instruction
        for (int c0 = c_begin; c0 < ncols; c0 += 32) {
          float y[16];
          tmem_ld16(tbase + c0, y);
          const int pid_c = pickn<kMetaN>(cpid, c0 >> 5);
          const float w_c = sc * pickn<kMetaN>(cw, c0 >> 5);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int pj = __shfl_sync(0xffffffffu, pid_c, (c0 & 31) + j);
            const float wj = __shfl_sync(0xffffffffu, w_c, (c0 & 31) + j);
            if (pj < p.P)
              p.pair_out[static_cast<size_t>(t.row0 + c0 + j) * p.ldo + col] =
                  __float2bfloat16_rn(y[j] * wj);
          }
        }
      } else if (kTokM) {
        // combine, unswapped: 16 consecutive columns of this thread's token
        // row (of each weight block of a pair), added with 16-byte vector
        // reductions
        for (int c0 = c_begin; c0 < ncols; c0 += 32) {
          float y[16], y1[16];
          tmem_ld16(tbase + c0, y);
          if (kPair) tmem_ld16(tbase + p.bn_max + c0, y1);
          if (row_ok && cpid[0] < p.P) {
            const float w_r = sc * cw[0];
#pragma unroll
            for (int b2i = 0; b2i < (kPair ? 2 : 1); ++b2i) {
              const float* yy = b2i == 0 ? y : y1;
              float* dst = p.acc_out + static_cast<size_t>(cpid[0] / p.top_k) * p.ldo +
                           t.nb * p.wblock_rows + b2i * 128 + c0;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                red_add_v4_f32(dst + 4 * j, yy[4 * j] * w_r, yy[4 * j + 1] * w_r,
                               yy[4 * j + 2] * w_r, yy[4 * j + 3] * w_r);
            }
          }
        }
      } else {
        // combine: y * s * topk_weight for 16 token columns at a time, staged
        // in shared memory and added into the token rows of the fp32 combine
        // buffer with one bulk asynchronous reduction (128 B) per column
        float* wstage = stage_out + static_cast<size_t>(warp - 2) * 2 * 16 * 32;
        for (int c0 = c_begin; c0 < t.n; c0 += 32) {
          float y[16];
          tmem_ld16(tbase + c0, y);
          float* buf = wstage + (n_chunks & 1u) * 16 * 32;
          // lane j < 16 handles column c0 + j
          const int pid = __shfl_sync(0xffffffffu, pickn<kMetaN>(cpid, c0 >> 5), (c0 & 31) + (lane & 15));
          const float wscale =
              sc * __shfl_sync(0xffffffffu, pickn<kMetaN>(cw, c0 >> 5), (c0 & 31) + (lane & 15));
          if (lane < 16) bulk_wait_read<1>();  // this buffer's reductions from two chunks ago have read it
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 16; ++j) buf[j * 32 + lane] = y[j] * __shfl_sync(0xffffffffu, wscale, j);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane < 16) {
            if (pid < p.P)
              bulk_reduce_add_f32(p.acc_out + static_cast<size_t>(pid / p.top_k) * p.ldo +
                                      t.nb * 128 + q * 32,
                                  buf + lane * 32, 128);
            bulk_commit();
          }
          ++n_chunks;
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty + a);
      ++tt;
      g = g1;
      t = t1;
      mt = mt1;
      have = have1;
      g1 = g2;
      t1 = t2;
      have1 = have2;
    }
    if (kSwiGLU && !kBF16) {
#pragma unroll
      for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0 && amax > 0.f) atomicMax(&p.ctrl->amax_h, __float_as_uint(amax));
    }
    if (!kSwiGLU && lane < 16) bulk_wait_all();  // reductions done before the CTA leaves
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
  if (trace && threadIdx.x == 0) {
    __threadfence();
    trace[3] = global_timer_ns();
  }
}

template <bool kBF16, bool kSwiGLU, bool kTokM, bool kPair = false>
cudaError_t launch_one(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                       const CUtensorMap& tb64, const CUtensorMap& to, int grid, cudaStream_t st) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = checked(cudaFuncSetAttribute(moe_gemm_kernel<kBF16, kSwiGLU, kTokM, kPair>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit), "smem attribute");
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const size_t smem = kSmemLimit;
  return launch_pdl(moe_gemm_kernel<kBF16, kSwiGLU, kTokM, kPair>, dim3(grid), dim3(kGemmThreads), smem, st, p,
                    ta, tb, tb64, to);
}

}  // namespace

// Epilogue staging of the down projection: 4 KB per epilogue warp, 1024 bytes
// after the stages (barriers first); up to 1023 bytes go to aligning the base.
constexpr size_t kCombineStaging = kGemmEpiWarps * 4096;
static_assert(kCombineStaging == kGemmEpiWarps * 2 * 16 * 32 * sizeof(float),
              "fp32 reduction staging: two 16 x 32 buffers per warp");

size_t gemm_stage_smem(bool swiglu) {
  return swiglu ? kSmemLimit - kSmemSlack : kSmemLimit - 2048 - kCombineStaging;
}

cudaError_t launch_gemm(bool bf16, bool swiglu, bool tok_m, bool pair, const GemmParams& p,
                        const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb64,
                        const CUtensorMap& to, int grid, cudaStream_t st) {
  if (pair && tok_m && !swiglu)
    return bf16 ? launch_one<true, false, true, true>(p, ta, tb, tb64, to, grid, st)
                : launch_one<false, false, true, true>(p, ta, tb, tb64, to, grid, st);
  if (pair) return cudaErrorInvalidValue;  // pairs exist for the unswapped down GEMM only
  if (tok_m) {
    if (bf16)
      return swiglu ? launch_one<true, true, true>(p, ta, tb, tb64, to, grid, st)
                    : launch_one<true, false, true>(p, ta, tb, tb64, to, grid, st);
    return swiglu ? launch_one<false, true, true>(p, ta, tb, tb64, to, grid, st)
                  : launch_one<false, false, true>(p, ta, tb, tb64, to, grid, st);
  }
  if (bf16)
    return swiglu ? launch_one<true, true, false>(p, ta, tb, tb64, to, grid, st)
                  : launch_one<true, false, false>(p, ta, tb, tb64, to, grid, st);
  return swiglu ? launch_one<false, true, false>(p, ta, tb, tb64, to, grid, st)
                : launch_one<false, false, false>(p, ta, tb, tb64, to, grid, st);
}

}  // namespace moe
