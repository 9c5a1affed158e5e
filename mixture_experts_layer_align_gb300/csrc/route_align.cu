// Token routing, alignment by expert, activation quantisation/gather and the
// small elementwise kernels of the fused MoE layer (sm_103a).
//
// Routing and "data shuffling" are the first two stages of the fused MoE
// operation ("Amazon SageMaker AI 上的 Mixture-of-Experts 内核工程优化",
// Introduction); FP8 tensor scaling is fused with them ("Backend routing for
// FP8 tensor quantization").  These kernels are HBM/latency bound: all loads
// are 16-byte vectors where the data allows, and nothing is staged through
// global memory that a CTA can keep on chip.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"
#include "route_token.cuh"

namespace moe {

namespace {

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
// `tmp` holds 32 ints of shared memory.  Every thread of the block must call it.
__device__ int block_exclusive_scan_1024(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = tmp[lane];
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(kFull, si, o);
      if (lane >= o) si += n;
    }
    tmp[lane] = si;
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? tmp[warp - 1] : 0);
  *total = tmp[31];
  __syncthreads();
  return excl;
}

// Router kernel: one warp per token, plus the per-CTA amax of x (the first
// half of the dynamic activation scale) and the per-call resets.
__global__ void __launch_bounds__(kRouteWarps * 32)
    route_topk_kernel(const float* __restrict__ logits, int T, int E, int k, int renorm,
                      int32_t* __restrict__ ids, float* __restrict__ wts,
                      const __nv_bfloat16* __restrict__ x, int H, float* __restrict__ amax_partials,
                      Ctrl* ctrl, int* __restrict__ zero_ints, int n_zero) {
  extern __shared__ float s_logits[];
  __shared__ float s_amax[kRouteWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if (ctrl != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
    ctrl->err = 0;
    ctrl->amax_h = 0u;
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x)
    zero_ints[i] = 0;
  const int t = blockIdx.x * kRouteWarps + warp;
  float xmax = 0.f;
  if (t < T) {
    // the token's first 8 x 16 bytes per lane are requested before the
    // routing, so their latency hides behind it
    const uint4* xr = x != nullptr ? reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H)
                                   : nullptr;
    const int n8 = x != nullptr ? H / 8 : 0;
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = lane + 32 * u;
      v[u] = i < n8 ? __ldg(xr + i) : make_uint4(0, 0, 0, 0);
    }
    route_token_any(logits + static_cast<size_t>(t) * E, E, k, renorm,
                s_logits + static_cast<size_t>(warp) * E, ids + static_cast<size_t>(t) * k,
                wts + static_cast<size_t>(t) * k, lane);
    if (x != nullptr) {
#pragma unroll
      for (int u = 0; u < 8; ++u) xmax = absmax8(v[u], xmax);
      for (int i0 = 256 + lane; i0 < n8; i0 += 256) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + 32 * u;
          v[u] = i < n8 ? __ldg(xr + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) xmax = absmax8(v[u], xmax);
      }
      xmax = warp_max(xmax);
    }
  }
  if (amax_partials != nullptr) {
    if (lane == 0) s_amax[warp] = xmax;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = 0.f;
#pragma unroll
      for (int w = 0; w < kRouteWarps; ++w) m = fmaxf(m, s_amax[w]);
      amax_partials[blockIdx.x] = m;
    }
  }
}

// ------------------------------------------------------------------ align
__device__ int2 write_mtiles(int tid, int E, int padded, int seg_off, int bm, int bn_max,
                             int4* __restrict__ mtiles, int* s_tmp);

// Stable counting sort of the T*k (token, slot) pairs by expert, padded per
// expert to a multiple of bm.  Each CTA owns one chunk of pair ids; it counts
// all pairs (to get the global offsets) and the pairs before its chunk (to
// get its own base inside every expert segment), so no CTA waits on another.
// Inside the chunk each warp owns a contiguous sub-range: per-warp counts are
// scanned column-wise over the 32 warps, then every warp places its pairs in
// order with __match_any_sync ranks.  The resulting order is exactly the
// ascending pair id order within each expert.  The chunk's ids are read from
// global memory once (kept in shared memory for both passes over the chunk),
// and CTA 0 writes the tile lists from the same prefix-sum pass as the
// offsets.
constexpr int kAlignThreads = 1024;
constexpr int kAlignChunk = 1024;  // pairs per CTA (<= 65535: per-warp counts are uint16)
constexpr int kAlignUnroll = 8;    // id loads in flight per thread in the histogram pass

// Block-wide exclusive scan of three ints per thread (blockDim.x == 1024),
// one pass of synchronisations for all three.  `tmp` holds 32 int3.
__device__ int3 block_exclusive_scan3_1024(int3 v, int3* tmp, int3* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int3 incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nx = __shfl_up_sync(kFull, incl.x, o);
    const int ny = __shfl_up_sync(kFull, incl.y, o);
    const int nz = __shfl_up_sync(kFull, incl.z, o);
    if (lane >= o) {
      incl.x += nx;
      incl.y += ny;
      incl.z += nz;
    }
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int3 si = tmp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nx = __shfl_up_sync(kFull, si.x, o);
      const int ny = __shfl_up_sync(kFull, si.y, o);
      const int nz = __shfl_up_sync(kFull, si.z, o);
      if (lane >= o) {
        si.x += nx;
        si.y += ny;
        si.z += nz;
      }
    }
    tmp[lane] = si;
  }
  __syncthreads();
  const int3 before = warp > 0 ? tmp[warp - 1] : make_int3(0, 0, 0);
  *total = tmp[31];
  __syncthreads();
  return make_int3(incl.x - v.x + before.x, incl.y - v.y + before.y, incl.z - v.z + before.z);
}

__global__ void __launch_bounds__(kAlignThreads) align_kernel(AlignParams p) {
  extern __shared__ int s_align[];
  __shared__ int3 s_tmp3[32];
  __shared__ float s_red[32];
  __shared__ int s_max_rows[2];  // largest row tile of each tile list
  const int E = p.E;
  int* hist_all = s_align;
  int* hist_before = hist_all + E;
  int* base = hist_before + E;
  int* seg_off = base + E;
  uint16_t* seg = reinterpret_cast<uint16_t*>(seg_off + E);  // [32][E]
  int* s_ids = reinterpret_cast<int*>(seg + 32 * E);         // this CTA's chunk of expert ids
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = p.P;
  const int cs = blockIdx.x * p.chunk;
  const int ce = min(cs + p.chunk, P);
  const int clen = max(ce - cs, 0);
  const int seglen = (clen + 31) / 32;
  const int s0 = cs + warp * seglen;
  const int s1 = min(s0 + seglen, ce);
  const bool tiles = p.mtiles != nullptr && blockIdx.x == 0;
  pdl_wait();
  pdl_trigger();
  // the router's per-CTA maxima of |x| (read at the end) are in flight meanwhile
  const float am_first =
      (tiles && p.amax_partials != nullptr && tid < p.n_partials) ? __ldg(p.amax_partials + tid) : 0.f;

  for (int e = tid; e < E; e += kAlignThreads) {
    hist_all[e] = 0;
    hist_before[e] = 0;
  }
  for (int i = tid; i < 32 * E; i += kAlignThreads) seg[i] = 0;
  if (tid < 2) s_max_rows[tid] = 0;
  __syncthreads();

  if (p.chunk_hist != nullptr) {
    // this chunk's ids into shared memory (read by both passes below)
    for (int q = cs + tid; q < ce; q += kAlignThreads) s_ids[q - cs] = __ldg(p.ids + q);
    // totals and the pairs before this chunk from the per-chunk histograms:
    // thread (e, r) sums chunks r, r + R, ... of expert e (R = 1024 / E
    // threads per expert, so all threads have loads in flight), then shared
    // atomics fold the R partial sums
    const int R = E <= kAlignThreads ? kAlignThreads / E : 1;
    const int e = tid % E, r = tid / E;
    if (r < R) {
      int tot = 0, bef = 0;
#pragma unroll 4
      for (int b = r; b < static_cast<int>(gridDim.x); b += R) {
        const int v = p.chunk_hist[static_cast<size_t>(b) * E + e];
        tot += v;
        bef += b < static_cast<int>(blockIdx.x) ? v : 0;
      }
      if (tot) atomicAdd(&hist_all[e], tot);
      if (bef) atomicAdd(&hist_before[e], bef);
    }
  }
  // histograms of every pair, and of the pairs before this chunk (loads of
  // kAlignUnroll rounds issued together: this pass is latency bound); the
  // chunk's own ids are kept in shared memory on the way
  for (int p0 = 0; p.chunk_hist == nullptr && p0 < P; p0 += kAlignThreads * kAlignUnroll) {
    int ev[kAlignUnroll];
#pragma unroll
    for (int u = 0; u < kAlignUnroll; ++u) {
      const int q = p0 + u * kAlignThreads + tid;
      ev[u] = q < P ? __ldg(p.ids + q) : -1;
    }
#pragma unroll
    for (int u = 0; u < kAlignUnroll; ++u) {
      const int q = p0 + u * kAlignThreads + tid;
      const int e = ev[u];
      if (q >= cs && q < ce) s_ids[q - cs] = e;
      const bool valid = q < P && static_cast<unsigned>(e) < static_cast<unsigned>(E);
      const unsigned mask = __match_any_sync(kFull, valid ? e : -1);
      if (valid && lane == __ffs(mask) - 1) {
        const int n = __popc(mask);
        atomicAdd(&hist_all[e], n);
        if (q < cs) atomicAdd(&hist_before[e], n);
      }
    }
  }
  __syncthreads();
  // per-warp counts of this CTA's chunk
  for (int q0 = s0; q0 < s1; q0 += 32) {
    const int q = q0 + lane;
    const int e = q < s1 ? s_ids[q - cs] : -1;
    const bool valid = q < s1 && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    const unsigned mask = __match_any_sync(kFull, valid ? e : -1);
    if (valid && lane == __ffs(mask) - 1) seg[warp * E + e] += static_cast<uint16_t>(__popc(mask));
    __syncwarp();
  }
  __syncthreads();

  // padded offsets and the row tiles of both tile lists (one expert per
  // thread; E <= 1024), all three prefix sums in one scan
  const int c = tid < E ? hist_all[tid] : 0;
  const int padded = (c + p.bm - 1) / p.bm * p.bm;
  const int nt = (p.mtiles != nullptr && padded > 0) ? (padded + p.bn_max - 1) / p.bn_max : 0;
  const int ntw = (p.mtiles_w != nullptr && padded > 0) ? (padded + kWideRows - 1) / kWideRows : 0;
  int3 tot;
  const int3 ex = block_exclusive_scan3_1024(make_int3(padded, nt, ntw), s_tmp3, &tot);
  const int off = ex.x;
  const int total = tot.x;
  if (tid < E) {
    base[tid] = off + hist_before[tid];
    seg_off[tid] = off;
    uint16_t run = 0;
    for (int w = 0; w < 32; ++w) {
      const uint16_t n = seg[w * E + tid];
      seg[w * E + tid] = run;
      run = static_cast<uint16_t>(run + n);
    }
  }
  if (blockIdx.x == 0) {
    if (tid < E) {
      p.counts[tid] = c;
      p.offsets[tid] = off;
    }
    if (tid == 0) {
      p.offsets[E] = total;
      if (p.num_padded) *p.num_padded = total;
      if (p.ctrl) p.ctrl->num_padded = total;
    }
  }
  __syncthreads();

  // stable scatter of this CTA's chunk
  for (int q0 = s0; q0 < s1; q0 += 32) {
    const int q = q0 + lane;
    const int e = q < s1 ? s_ids[q - cs] : -1;
    const bool valid = q < s1 && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    const unsigned mask = __match_any_sync(kFull, valid ? e : -1);
    const int leader = __ffs(mask) - 1;
    int slot = 0;
    if (valid && lane == leader) {
      slot = base[e] + seg[warp * E + e];
      seg[warp * E + e] = static_cast<uint16_t>(seg[warp * E + e] + __popc(mask));
    }
    slot = __shfl_sync(kFull, slot, leader);
    if (valid) {
      const int at = slot + __popc(mask & ((1u << lane) - 1u));
      p.sorted_ids[at] = q;
      if (p.sorted_w) p.sorted_w[at] = p.wts[q];
      if (p.inv_slot) p.inv_slot[q] = at;
    }
    __syncwarp();
  }

  if (blockIdx.x != 0) return;  // uniform per block

  // padding sentinels, spread over the CTA: thread i takes row r = i % bm of
  // expert i / bm's padding (rows c .. padded - 1 of its segment)
  for (int i = tid; i < E * p.bm; i += kAlignThreads) {
    const int e = i / p.bm, r = i - e * p.bm;
    const int ce2 = hist_all[e];
    const int pe = (ce2 + p.bm - 1) / p.bm * p.bm;
    if (ce2 + r < pe) {
      p.sorted_ids[seg_off[e] + ce2 + r] = P;
      if (p.sorted_w) p.sorted_w[seg_off[e] + ce2 + r] = 0.f;
    }
  }
  if (p.tile_expert && tid < E) {
    const int o = seg_off[tid];
    for (int b = o / p.bm; b < (o + padded) / p.bm; ++b) p.tile_expert[b] = tid;
  }

  if (p.mtiles != nullptr) {
    // GEMM row tiles of this thread's expert: ceil(padded / bn) tiles of equal
    // rows rounded up to the alignment block (the largest is the first)
    if (nt > 0) {
      const int per = ((padded + nt - 1) / nt + p.bm - 1) / p.bm * p.bm;
      for (int j = 0; j < nt; ++j)
        p.mtiles[ex.y + j] = make_int4(tid, off + j * per,
                                       static_cast<int>(static_cast<unsigned>(min(per, padded - j * per)) |
                                                        (static_cast<unsigned>(nt) << 12)),
                                       ex.y);
      atomicMax(&s_max_rows[0], per);
    }
    if (ntw > 0) {
      const int per = ((padded + ntw - 1) / ntw + p.bm - 1) / p.bm * p.bm;
      for (int j = 0; j < ntw; ++j)
        p.mtiles_w[ex.z + j] = make_int4(tid, off + j * per,
                                         static_cast<int>(static_cast<unsigned>(min(per, padded - j * per)) |
                                                          (static_cast<unsigned>(ntw) << 12)),
                                         ex.z);
      atomicMax(&s_max_rows[1], per);
    }
    // activation scale of x from the router's per-CTA amax values
    float m = am_first;
    for (int i = tid + kAlignThreads; i < p.n_partials; i += kAlignThreads)
      m = fmaxf(m, p.amax_partials[i]);
    m = warp_max(m);
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    if (tid == 0) {
      float a = 0.f;
      for (int w = 0; w < 32; ++w) a = fmaxf(a, s_red[w]);
      p.ctrl->s_x = p.amax_partials ? scale_from_amax(a) : 1.f;
      p.ctrl->num_mtiles = tot.y;
      p.ctrl->max_tile_rows = s_max_rows[0];
      p.ctrl->num_mtiles_w = p.mtiles_w != nullptr ? tot.z : 0;
      p.ctrl->max_tile_rows_w = p.mtiles_w != nullptr ? s_max_rows[1] : 0;
    }
  }
}

// Writes the GEMM row-tile list from the per-expert padded segments (one
// expert per thread, tid < E; all 1024 threads of the block must call).
// Each expert's segment is split into ceil(padded / bn_max) equal tiles
// (multiples of bm); every entry also carries the expert's tile count and the
// index of its first tile.  Returns {number of tiles, rows of the largest}.
__device__ int2 write_mtiles(int tid, int E, int padded, int seg_off, int bm, int bn_max,
                             int4* __restrict__ mtiles, int* s_tmp) {
  const int nt = (tid < E && padded > 0) ? (padded + bn_max - 1) / bn_max : 0;
  const int per = nt > 0 ? ((padded + nt - 1) / nt + bm - 1) / bm * bm : 0;
  int n_tiles = 0;
  const int first = block_exclusive_scan_1024(nt, s_tmp, &n_tiles);
  for (int j = 0; j < nt; ++j) {
    const int rows = min(per, padded - j * per);
    // the tile count above bit 12 is informational (the GEMMs read the low 12
    // bits); unsigned so that experts of more than 2^19 tiles wrap, not overflow
    mtiles[first + j] = make_int4(tid, seg_off + j * per,
                                  static_cast<int>(static_cast<unsigned>(rows) | (static_cast<unsigned>(nt) << 12)),
                                  first);
  }
  // the largest tile is some expert's first one
  const int wmax = static_cast<int>(__reduce_max_sync(kFull, static_cast<unsigned>(per)));
  if ((threadIdx.x & 31) == 0) s_tmp[threadIdx.x >> 5] = wmax;
  __syncthreads();
  int mx = 0;
  for (int w = 0; w < 32; ++w) mx = max(mx, s_tmp[w]);
  __syncthreads();
  return make_int2(n_tiles, mx);
}

// Small batches (decode): one CTA routes every token, takes amax |x|, aligns
// the pairs and writes the GEMM tile list, with everything in shared memory
// between the steps: the router and alignment kernels in one launch and
// without their global-memory round trips.
__global__ void __launch_bounds__(kAlignThreads, 1) route_align_small_kernel(SmallFrontParams p) {
  extern __shared__ int s_small[];
  __shared__ int s_tmp[32];
  __shared__ float s_red[32];
  const int E = p.E, k = p.k, T = p.T;
  const int P = T * k;
  float* s_logits = reinterpret_cast<float*>(s_small);  // [32][E]
  int32_t* s_ids = s_small + 32 * E;                     // [P]
  float* s_w = reinterpret_cast<float*>(s_ids + P);      // [P]
  int* s_cnt = reinterpret_cast<int*>(s_w + P);          // [E]
  int* s_run = s_cnt + E;                                // [E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Ctrl* ctrl = p.ctrl;
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    ctrl->err = 0;
    ctrl->amax_h = 0u;
  }
  for (int i = tid; i < p.n_zero; i += kAlignThreads) p.zero_ints[i] = 0;
  for (int e = tid; e < E; e += kAlignThreads) s_cnt[e] = 0;

  // amax |x| (FP8), 8 vector loads in flight per thread; the first batch goes
  // out before the routing, so that its round trip overlaps the logits'
  const uint4* xv = reinterpret_cast<const uint4*>(p.x);
  const long long n8 = p.x != nullptr ? static_cast<long long>(T) * p.H / 8 : 0;
  uint4 v[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const long long i = u * kAlignThreads + tid;
    v[u] = i < n8 ? __ldg(xv + i) : make_uint4(0, 0, 0, 0);
  }
  // routing, one warp per token
  for (int t = warp; t < T; t += 32)
    route_token_any(p.logits + static_cast<size_t>(t) * E, E, k, p.renorm, s_logits + warp * E,
                s_ids + t * k, s_w + t * k, lane);
  float xmax = 0.f;
  for (long long i0 = 0; i0 < n8; i0 += 8 * kAlignThreads) {
    if (i0 > 0) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const long long i = i0 + u * kAlignThreads + tid;
        v[u] = i < n8 ? __ldg(xv + i) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) xmax = absmax8(v[u], xmax);
  }
  xmax = warp_max(xmax);
  if (lane == 0) s_red[warp] = xmax;
  __syncthreads();

  // counts and padded offsets
  for (int q0 = 0; q0 < P; q0 += kAlignThreads) {
    const int q = q0 + tid;
    const int e = q < P ? s_ids[q] : -1;
    const bool valid = q < P && static_cast<unsigned>(e) < static_cast<unsigned>(E);
    const unsigned mask = __match_any_sync(kFull, valid ? e : -1);
    if (valid && lane == __ffs(mask) - 1) atomicAdd(&s_cnt[e], __popc(mask));
  }
  __syncthreads();
  const int c = tid < E ? s_cnt[tid] : 0;
  const int padded = (c + kAlignBlock - 1) / kAlignBlock * kAlignBlock;
  // one scan for both prefixes: padded rows (high bits) and row tiles (low 12
  // bits; at most (P + 142 E) / 128 < 4096 tiles)
  const int nt = (tid < E && padded > 0) ? (padded + p.bn_max - 1) / p.bn_max : 0;
  int tot_packed = 0;
  const int packed = block_exclusive_scan_1024((padded << 12) | nt, s_tmp, &tot_packed);
  const int off = packed >> 12;
  const int first_tile = packed & 0xfff;
  const int total = tot_packed >> 12;
  if (tid < E) s_run[tid] = off;
  __syncthreads();
  // stable placement in pair-id order (one warp), padding sentinels
  if (warp == 0) {
    for (int q0 = 0; q0 < P; q0 += 32) {
      const int q = q0 + lane;
      const int e = q < P ? s_ids[q] : -1;
      const bool valid = q < P && static_cast<unsigned>(e) < static_cast<unsigned>(E);
      const unsigned mask = __match_any_sync(kFull, valid ? e : -1);
      const int leader = __ffs(mask) - 1;
      int slot = 0;
      if (valid && lane == leader) {
        slot = s_run[e];
        s_run[e] = slot + __popc(mask);
      }
      slot = __shfl_sync(kFull, slot, leader);
      if (valid) {
        const int at = slot + __popc(mask & ((1u << lane) - 1u));
        p.sorted_ids[at] = q;
        p.sorted_w[at] = s_w[q];
      }
      __syncwarp();
    }
  }
  if (tid < E) {
    for (int i = c; i < padded; ++i) {
      p.sorted_ids[off + i] = P;
      p.sorted_w[off + i] = 0.f;
    }
    p.counts[tid] = c;
    p.offsets[tid] = off;
  }
  for (int q = tid; q < P; q += kAlignThreads) {
    p.ids[q] = s_ids[q];
    p.wts[q] = s_w[q];
  }
  // GEMM row tiles of each expert (as write_mtiles, from the packed scan)
  const int per = nt > 0 ? ((padded + nt - 1) / nt + kAlignBlock - 1) / kAlignBlock * kAlignBlock : 0;
  for (int j = 0; j < nt; ++j)
    p.mtiles[first_tile + j] = make_int4(tid, off + j * per, min(per, padded - j * per) | (nt << 12),
                                         first_tile);
  const int wmax = static_cast<int>(__reduce_max_sync(kFull, static_cast<unsigned>(per)));
  if (lane == 0) s_tmp[warp] = wmax;  // (s_tmp is free again after the scan's last sync)
  __syncthreads();
  int2 tl = make_int2(tot_packed & 0xfff, 0);
  for (int w = 0; w < 32; ++w) tl.y = max(tl.y, s_tmp[w]);
  __syncthreads();
  const int2 tw = p.mtiles_w ? write_mtiles(tid, E, padded, off, kAlignBlock, kWideRows, p.mtiles_w,
                                            s_tmp)
                             : make_int2(0, 0);
  if (tid == 0) {
    float a = 0.f;
    for (int w = 0; w < 32; ++w) a = fmaxf(a, s_red[w]);
    p.offsets[E] = total;
    ctrl->num_padded = total;
    ctrl->num_mtiles = tl.x;
    ctrl->max_tile_rows = tl.y;
    ctrl->num_mtiles_w = tw.x;
    ctrl->max_tile_rows_w = tw.y;
    ctrl->s_x = p.x != nullptr ? scale_from_amax(a) : 1.f;
  }
}

// First pass of the two-pass alignment for large batches: each CTA counts the
// experts of its own chunk of pairs only.
__global__ void __launch_bounds__(kAlignThreads)
    align_hist_kernel(const int32_t* __restrict__ ids, int P, int E, int chunk,
                      int32_t* __restrict__ hist) {
  extern __shared__ int s_hist[];
  const int tid = threadIdx.x, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  for (int e = tid; e < E; e += kAlignThreads) s_hist[e] = 0;
  __syncthreads();
  const int cs = blockIdx.x * chunk;
  const int ce = min(cs + chunk, P);
  for (int q0 = cs; q0 < ce; q0 += kAlignThreads * kAlignUnroll) {
    int ev[kAlignUnroll];
#pragma unroll
    for (int u = 0; u < kAlignUnroll; ++u) {
      const int q = q0 + u * kAlignThreads + tid;
      ev[u] = q < ce ? __ldg(ids + q) : -1;
    }
#pragma unroll
    for (int u = 0; u < kAlignUnroll; ++u) {
      const int e = ev[u];
      const bool valid = static_cast<unsigned>(e) < static_cast<unsigned>(E);
      const unsigned mask = __match_any_sync(kFull, valid ? e : -1);
      if (valid && lane == __ffs(mask) - 1) atomicAdd(&s_hist[e], __popc(mask));
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kAlignThreads) hist[static_cast<size_t>(blockIdx.x) * E + e] = s_hist[e];
}

// Large FP8 batches: every token row of x is quantised once with s_x (a warp
// per token, 16 elements per lane item) and its 16-byte code chunks are
// written to each of the token's k aligned rows (the slots the alignment
// recorded per pair); the padding rows of every expert segment are zeroed,
// and so is the fp32 combine buffer when there is one.
__global__ void __launch_bounds__(256)
    quant_scatter_kernel(const __nv_bfloat16* __restrict__ x, int T, int H, int k,
                         const int32_t* __restrict__ inv_slot, const int32_t* __restrict__ counts,
                         const int32_t* __restrict__ offsets, int E, const Ctrl* __restrict__ ctrl,
                         uint8_t* __restrict__ xs, float* __restrict__ acc, long long acc_elems) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int w0 = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const float s = ctrl->s_x;
  const E4m3Div ds = e4m3_div(s);
  const int n16 = H / 16;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  const unsigned rows = static_cast<unsigned>(ctrl->num_padded);
  for (int t = w0; t < T; t += nwarps) {
    // lane j < k holds the aligned row of pair (t, j) (k > 32: read per use)
    const int32_t* tslots = inv_slot + static_cast<size_t>(t) * k;
    const int my_slot = lane < k ? tslots[lane] : 0;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    for (int c = lane; c < n16; c += 32) {
      const uint2 lo = quant8(__ldg(src + 2 * c), ds);
      const uint2 hi = quant8(__ldg(src + 2 * c + 1), ds);
      const uint4 v = make_uint4(lo.x, lo.y, hi.x, hi.y);
      for (int j = 0; j < k; ++j) {
        const int slot = k <= 32 ? __shfl_sync(0xffffffffu, my_slot, j) : tslots[j];
        if (static_cast<unsigned>(slot) < rows)  // every routed pair has a row below num_padded
          reinterpret_cast<uint4*>(xs + static_cast<size_t>(slot) * H)[c] = v;
      }
    }
  }
  // padding rows: a warp per expert segment
  for (int e = w0; e < E; e += nwarps) {
    const int r0 = offsets[e] + counts[e], r1 = offsets[e + 1];
    for (int r = r0; r < r1; ++r) {
      uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<size_t>(r) * H);
      for (int c = lane; c < n16; c += 32) dst[c] = zero;
    }
  }
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  float4* a4 = reinterpret_cast<float4*>(acc);
  for (long long i = tid; i < acc_elems / 4; i += stride) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ gather
// The pair's token row of x for every aligned row, quantised to E4M3 with s_x
// (FP8) or copied (bf16), zero for padding rows: one thread per 16 (8 for
// bf16) elements, so a few long rows still spread over the whole grid.  The
// same grid zeroes the fp32 combine buffer.
__global__ void __launch_bounds__(256)
    gather_x_kernel(const __nv_bfloat16* __restrict__ x, int H,
                    const int32_t* __restrict__ sorted_ids, const Ctrl* __restrict__ ctrl, int P,
                    int k, void* __restrict__ xs, int fp8, float* __restrict__ acc,
                    long long acc_elems) {
  pdl_wait();
  pdl_trigger();
  const long long rows = ctrl->num_padded;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  if (fp8) {
    const float sx = ctrl->s_x;
    const E4m3Div dx = e4m3_div(sx);
    const int per_row = H / 16;
    const long long n = rows * per_row;
    uint4* dst = static_cast<uint4*>(xs);
    for (long long i = tid; i < n; i += stride) {
      const long long r = i / per_row;
      const int c = static_cast<int>(i - r * per_row);
      const int q = sorted_ids[r];
      uint4 v = zero;
      if (q < P) {
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(q / k) * H);
        const uint2 lo = quant8(__ldg(src + 2 * c), dx);
        const uint2 hi = quant8(__ldg(src + 2 * c + 1), dx);
        v = make_uint4(lo.x, lo.y, hi.x, hi.y);
      }
      dst[i] = v;
    }
  } else {
    const int per_row = H / 8;  // 8 bf16 per uint4
    const long long n = rows * per_row;
    uint4* dst = static_cast<uint4*>(xs);
    for (long long i = tid; i < n; i += stride) {
      const long long r = i / per_row;
      const int c = static_cast<int>(i - r * per_row);
      const int q = sorted_ids[r];
      dst[i] = q < P ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(q / k) * H) + c)
                     : zero;
    }
  }
  float4* a4 = reinterpret_cast<float4*>(acc);
  const long long n4 = acc_elems / 4;
  for (long long i = tid; i < n4; i += stride) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ h quant
__global__ void __launch_bounds__(256)
    quant_h_kernel(const float* __restrict__ h, int I, Ctrl* ctrl, uint8_t* __restrict__ hq) {
  pdl_wait();
  pdl_trigger();
  const float s = scale_from_amax(__uint_as_float(ctrl->amax_h));
  const E4m3Div ds = e4m3_div(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) ctrl->s_h = s;
  const long long n16 = static_cast<long long>(ctrl->num_padded) * I / 16;
  const float4* src = reinterpret_cast<const float4*>(h);
  uint4* dst = reinterpret_cast<uint4*>(hq);
  // Last rows first: the gate/up GEMM writes h in row order (experts in
  // turn), so its last rows are the ones still in L2.  Two groups of 16
  // values per thread in flight.
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long j = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; j < n16;
       j += 2 * stride) {
    const long long i0 = n16 - 1 - j;
    const long long i1 = i0 - stride;
    float4 a[4], b[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) a[c] = src[4 * i0 + c];
    if (i1 >= 0) {
#pragma unroll
      for (int c = 0; c < 4; ++c) b[c] = src[4 * i1 + c];
    }
    uint4 r;
    r.x = quant4(a[0], ds);
    r.y = quant4(a[1], ds);
    r.z = quant4(a[2], ds);
    r.w = quant4(a[3], ds);
    dst[i0] = r;
    if (i1 >= 0) {
      r.x = quant4(b[0], ds);
      r.y = quant4(b[1], ds);
      r.z = quant4(b[2], ds);
      r.w = quant4(b[3], ds);
      dst[i1] = r;
    }
  }
}

// ------------------------------------------------------------------ finalize
__global__ void __launch_bounds__(256)
    finalize_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ out, long long n8) {
  pdl_wait();
  pdl_trigger();
  const float4* a = reinterpret_cast<const float4*>(acc);
  uint4* o = reinterpret_cast<uint4*>(out);
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 u = a[2 * i], v = a[2 * i + 1];
    __nv_bfloat162 b0 = __floats2bfloat162_rn(u.x, u.y);
    __nv_bfloat162 b1 = __floats2bfloat162_rn(u.z, u.w);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b3 = __floats2bfloat162_rn(v.z, v.w);
    uint4 r;
    r.x = *reinterpret_cast<uint32_t*>(&b0);
    r.y = *reinterpret_cast<uint32_t*>(&b1);
    r.z = *reinterpret_cast<uint32_t*>(&b2);
    r.w = *reinterpret_cast<uint32_t*>(&b3);
    o[i] = r;
  }
}

// ------------------------------------------------------------------ combine rows
// out[t] = sum over the k slots of the weighted expert rows of token t (row
// inv_slot[t*k+j] of the aligned order), fp32 accumulation in slot order, one
// bf16 rounding.  8 columns per thread.
__global__ void __launch_bounds__(256, 4)
    combine_rows_kernel(const __nv_bfloat16* __restrict__ rows,
                        const int32_t* __restrict__ inv_slot, int T, int k, int H,
                        __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int per_row = H / 8;
  const long long n8 = static_cast<long long>(T) * per_row;
  const uint4* src = reinterpret_cast<const uint4*>(rows);
  uint4* dst = reinterpret_cast<uint4*>(out);
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / per_row;
    const long long c = i - t * per_row;
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int32_t* sl = inv_slot + t * k;
    for (int j0 = 0; j0 < k; j0 += 8) {
      // up to 8 rows in flight, summed in slot order
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (j0 + u < k) v[u] = __ldg(src + static_cast<long long>(__ldg(sl + j0 + u)) * per_row + c);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u < k) {
          a[0] += bf16_lo(v[u].x);
          a[1] += bf16_hi(v[u].x);
          a[2] += bf16_lo(v[u].y);
          a[3] += bf16_hi(v[u].y);
          a[4] += bf16_lo(v[u].z);
          a[5] += bf16_hi(v[u].z);
          a[6] += bf16_lo(v[u].w);
          a[7] += bf16_hi(v[u].w);
        }
      }
    }
    __nv_bfloat162 b0 = __floats2bfloat162_rn(a[0], a[1]);
    __nv_bfloat162 b1 = __floats2bfloat162_rn(a[2], a[3]);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(a[4], a[5]);
    __nv_bfloat162 b3 = __floats2bfloat162_rn(a[6], a[7]);
    uint4 r;
    r.x = *reinterpret_cast<uint32_t*>(&b0);
    r.y = *reinterpret_cast<uint32_t*>(&b1);
    r.z = *reinterpret_cast<uint32_t*>(&b2);
    r.w = *reinterpret_cast<uint32_t*>(&b3);
    dst[i] = r;
  }
}

// ------------------------------------------------------------------ quantize (standalone)
__global__ void __launch_bounds__(256)
    amax_kernel(const __nv_bfloat16* __restrict__ x, long long n8, float* __restrict__ partials) {
  __shared__ float s_red[8];
  pdl_wait();
  pdl_trigger();
  const uint4* src = reinterpret_cast<const uint4*>(x);
  float m = 0.f;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    m = absmax8(__ldg(src + i), m);
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int w = 0; w < 8; ++w) a = fmaxf(a, s_red[w]);
    partials[blockIdx.x] = a;
  }
}

__global__ void __launch_bounds__(256)
    quant_x_kernel(const __nv_bfloat16* __restrict__ x, long long n16, const float* __restrict__ partials,
                   int n_partials, uint8_t* __restrict__ xq, float* __restrict__ scale) {
  __shared__ float s_scale;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < 32) {
    float m = 0.f;
    for (int i = threadIdx.x; i < n_partials; i += 32) m = fmaxf(m, partials[i]);
    m = warp_max(m);
    if (threadIdx.x == 0) s_scale = scale_from_amax(m);
  }
  __syncthreads();
  const float s = s_scale;
  const E4m3Div ds = e4m3_div(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale = s;
  const uint4* src = reinterpret_cast<const uint4*>(x);
  uint4* dst = reinterpret_cast<uint4*>(xq);
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint2 a = quant8(__ldg(src + 2 * i), ds);
    const uint2 b = quant8(__ldg(src + 2 * i + 1), ds);
    dst[i] = make_uint4(a.x, a.y, b.x, b.y);
  }
}

}  // namespace

// ------------------------------------------------------------------ launchers
namespace {
int capped_grid(long long work, long long per_block, int num_sms, int per_sm) {
  long long g = (work + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(num_sms) * per_sm;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}
}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                              float* wts, const __nv_bfloat16* x, int H, float* amax_partials,
                              Ctrl* ctrl, int* zero_ints, int n_zero, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(kRouteWarps) * E * sizeof(float);
  return launch_pdl(route_topk_kernel, dim3(route_grid(T)), dim3(kRouteWarps * 32), smem, st,
                    logits, T, E, k, renorm, ids, wts, x, H, amax_partials, ctrl, zero_ints,
                    n_zero);
}

int align_chunk() { return kAlignChunk; }

cudaError_t launch_align(const AlignParams& p, cudaStream_t st) {
  // 4 ints and 32 per-warp counts per expert, then the CTA's chunk of ids
  const size_t smem = static_cast<size_t>(p.E) * 4 * sizeof(int) + 32u * p.E * sizeof(uint16_t) +
                      static_cast<size_t>(p.chunk) * sizeof(int);
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = checked(cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         4 * 1024 * 4 + 32 * 1024 * 2 + kAlignChunk * 4),
                            "smem attribute");
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int grid = p.P > 0 ? (p.P + p.chunk - 1) / p.chunk : 1;
  return launch_pdl(align_kernel, dim3(grid), dim3(kAlignThreads), smem, st, p);
}

cudaError_t launch_gather_x(const __nv_bfloat16* x, int H, const int32_t* sorted_ids,
                            const Ctrl* ctrl, int P, int k, void* xs, bool fp8, float* acc,
                            long long acc_elems, int max_rows, int num_sms, cudaStream_t st) {
  const long long per_row = fp8 ? H / 16 : H / 8;
  const long long work = std::max(static_cast<long long>(max_rows) * per_row, acc_elems / 4);
  const int grid = capped_grid(work, 256, num_sms, 8);
  return launch_pdl(gather_x_kernel, dim3(grid), dim3(256), 0, st, x, H, sorted_ids, ctrl, P, k,
                    xs, fp8 ? 1 : 0, acc, acc_elems);
}

cudaError_t launch_route_align_small(const SmallFrontParams& p, cudaStream_t st) {
  const size_t smem =
      (static_cast<size_t>(32) * p.E + 2 * static_cast<size_t>(p.T) * p.k + 2 * p.E) * sizeof(int);
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    const int max_smem =
        (32 * kSmallMaxExperts + 2 * kSmallMaxPairs + 2 * kSmallMaxExperts) * sizeof(int);
    cudaError_t e = checked(cudaFuncSetAttribute(route_align_small_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 max_smem),
                            "smem attribute");
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_pdl(route_align_small_kernel, dim3(1), dim3(kAlignThreads), smem, st, p);
}

cudaError_t launch_align_hist(const int32_t* ids, int P, int E, int32_t* hist, cudaStream_t st) {
  const int grid = (P + kAlignChunk - 1) / kAlignChunk;
  return launch_pdl(align_hist_kernel, dim3(grid), dim3(kAlignThreads), E * sizeof(int), st, ids,
                    P, E, kAlignChunk, hist);
}

cudaError_t launch_quant_scatter(const __nv_bfloat16* x, int T, int H, int k,
                                 const int32_t* inv_slot, const int32_t* counts,
                                 const int32_t* offsets, int E, const Ctrl* ctrl, uint8_t* xs,
                                 float* acc, long long acc_elems, int num_sms, cudaStream_t st) {
  const long long warps = std::max<long long>(T, E);
  const int grid = capped_grid(std::max(warps * 32, acc_elems / 4), 256, num_sms, 8);
  return launch_pdl(quant_scatter_kernel, dim3(grid), dim3(256), 0, st, x, T, H, k, inv_slot,
                    counts, offsets, E, ctrl, xs, acc, acc_elems);
}

cudaError_t launch_quant_h(const float* h, int I, Ctrl* ctrl, uint8_t* hq, int max_rows,
                           int num_sms, cudaStream_t st) {
  const int grid = capped_grid(static_cast<long long>(max_rows) * I / 16, 256, num_sms, 8);
  return launch_pdl(quant_h_kernel, dim3(grid), dim3(256), 0, st, h, I, ctrl, hq);
}

cudaError_t launch_finalize(const float* acc, __nv_bfloat16* out, long long n, int num_sms,
                            cudaStream_t st) {
  const int grid = capped_grid(n / 8, 256, num_sms, 8);
  return launch_pdl(finalize_kernel, dim3(grid), dim3(256), 0, st, acc, out, n / 8);
}

cudaError_t launch_combine_rows(const __nv_bfloat16* rows, const int32_t* inv_slot, int T, int k,
                                int H, __nv_bfloat16* out, int num_sms, cudaStream_t st) {
  const int grid = capped_grid(static_cast<long long>(T) * H / 8, 256, num_sms, 4);
  return launch_pdl(combine_rows_kernel, dim3(grid), dim3(256), 0, st, rows, inv_slot, T, k, H,
                    out);
}

cudaError_t launch_quantize_e4m3(const __nv_bfloat16* x, long long n, uint8_t* xq, float* scale,
                                 float* partials, int n_partials, cudaStream_t st) {
  cudaError_t e = launch_pdl(amax_kernel, dim3(n_partials), dim3(256), 0, st, x, n / 8, partials);
  if (e != cudaSuccess) return e;
  long long grid = (n / 16 + 255) / 256;
  if (grid > 4096) grid = 4096;
  if (grid < 1) grid = 1;
  return launch_pdl(quant_x_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, x, n / 16,
                    static_cast<const float*>(partials), n_partials, xq, scale);
}

}  // namespace moe
