// Work split of the persistent grouped-GEMM kernels: row tiles x weight
// blocks x K steps, whole tiles round-robin and a stream-K tail, and the
// partial-accumulator slots of tiles cut between CTAs.
#pragma once

#include <stdint.h>

#include "internal.h"

namespace moe {
namespace {

struct Tile {
  int e, row0, n, nb;
};

// Tile u -> (expert, first row, rows, weight block): row tile u / nb_count of
// the tile list `mtiles` (one load of the list), weight block u % nb_count.
// A row tile's weight blocks are consecutive tiles, and an expert's row tiles
// follow one another, so the G tiles in flight share token rows and weight
// blocks.
__device__ __forceinline__ Tile decode_tile_of(const int4* mtiles, int nb_count, int u) {
  const int m = u / nb_count;
  const int4 t = mtiles[m];
  Tile r;
  r.e = t.x;
  r.row0 = t.y;
  r.n = t.z & 0xfff;
  r.nb = u - m * nb_count;
  return r;
}

// Order in which the flat index space visits tiles: the tiles are laid out
// row-major on a grid G wide (G = CTAs) and visited column by column, so the
// contiguous range of one CTA covers tiles c, c+G, c+2G, ... spread over the
// whole weight tensor (every CTA sees the same mix of memory), while a tile
// cut at a range boundary is still shared by neighbouring CTAs only.
__device__ __forceinline__ int tile_of_seq(int s, int tiles) {
  const int G = static_cast<int>(gridDim.x);
  const int W = (tiles + G - 1) / G;         // rows
  const int r = tiles - (W - 1) * G;         // columns that have W rows
  int row, col;
  if (s < r * W) {
    col = s / W;
    row = s - col * W;
  } else {
    const int s2 = s - r * W;
    col = r + s2 / (W - 1);
    row = s2 - (col - r) * (W - 1);
  }
  return row * G + col;
}

// Work split over the flat (tile, K step) space, in two parts.
//  - The first `rr` tiles go whole and round-robin: CTA c takes tiles c, c+G,
//    c+2G, ... in natural (expert, weight block, row tile) order, so at any
//    moment the CTAs work on G consecutive tiles and the weight blocks and
//    token rows those share are read from HBM once and then hit in L2.
//  - The remaining tiles (the tail) are cut evenly over the CTAs, one
//    contiguous range of the flat tail space each (stream-K); a tile cut
//    between CTAs is finished from partial sums.
// With no reuse to keep (decode: every weight block serves one row tile) the
// whole space is tail, visited in the column-major order of tile_of_seq.
// Rows written per pair cannot take partial sums: then every tile is whole.
struct Sched {
  int tiles, K, rr;
  bool permute;          // tail order: tile_of_seq (no reuse) or natural
  long long tail_total;  // (tiles - rr) * K
  long long beg, end;    // this CTA's range of the tail space
};

__device__ __forceinline__ Sched make_sched(int tiles, int K, bool reuse, bool whole) {
  const int G = static_cast<int>(gridDim.x);
  Sched s;
  s.tiles = tiles;
  s.K = K;
  s.rr = whole ? tiles : (reuse ? tiles / G * G : 0);
  s.permute = !reuse;
  s.tail_total = static_cast<long long>(tiles - s.rr) * K;
  s.beg = s.tail_total * blockIdx.x / G;
  s.end = s.tail_total * (blockIdx.x + 1) / G;
  return s;
}

// One segment: K steps [k0, k1) of `tile`; t0 = flat start of the tile in the
// tail space (meaningful for tail tiles only).
struct Seg {
  int tile, k0, k1;
  long long t0;
};

struct SegIt {
  int u;        // next round-robin tile
  long long i;  // next flat tail index
};

__device__ __forceinline__ SegIt seg_begin(const Sched& s) {
  SegIt it;
  it.u = static_cast<int>(blockIdx.x);
  it.i = s.beg;
  return it;
}

__device__ __forceinline__ bool seg_next(const Sched& s, SegIt& it, Seg& g) {
  if (it.u < s.rr) {
    g.tile = it.u;
    g.k0 = 0;
    g.k1 = s.K;
    g.t0 = 0;
    it.u += static_cast<int>(gridDim.x);
    return true;
  }
  if (it.i >= s.end) return false;
  const int v = static_cast<int>(it.i / s.K);
  g.k0 = static_cast<int>(it.i - static_cast<long long>(v) * s.K);
  const long long rem = s.end - it.i;
  g.k1 = (static_cast<long long>(s.K) < g.k0 + rem) ? s.K : static_cast<int>(g.k0 + rem);
  g.t0 = static_cast<long long>(v) * s.K;
  g.tile = s.rr + (s.permute ? tile_of_seq(v, s.tiles - s.rr) : v);
  it.i += g.k1 - g.k0;
  return true;
}

// CTA whose tail range holds flat index i.
__device__ __forceinline__ int owner_of(long long i, long long total) {
  return static_cast<int>(((i + 1) * gridDim.x - 1) / total);
}

__device__ __forceinline__ long long range_begin(int c, long long total) {
  return total * c / gridDim.x;
}

// Partial slot of CTA c for a tile starting at flat index t0: slot 1 if c's
// range began before the tile (the tile is c's last segment), else slot 0.
__device__ __forceinline__ float* part_slot_of(float* part, int bn_max, int c, long long t0,
                                               long long total) {
  const int s = range_begin(c, total) < t0 ? 1 : 0;
  return part + (static_cast<size_t>(c) * 2 + s) * gemm_part_slot_floats(bn_max);
}

// v[s] for a warp-uniform runtime s in [0, N) without local-memory indexing.
template <int N, typename V>
__device__ __forceinline__ V pickn(const V (&v)[N], int s) {
  V r = v[0];
#pragma unroll
  for (int i = 1; i < N; ++i) r = (s == i) ? v[i] : r;
  return r;
}

}  // namespace
}  // namespace moe
