// Tile decoding shared by the dense backward kernels: a tile is a block of
// kDenseBM key rows of one KV head (and batch row, or packed sequence).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace ab {

// len: keys of the tile's sequence; qlen: its queries; off: the key position
// of query 0 (qlen, off differ from len, 0 only in a dense row with Sk != S).
struct TileInfo {
  int b, g, seq_start, len, k0, qlo, nq, valid;
  int qlen, off;
  // query heads h0 .. h0 + hn - 1 of the group; part >= 0: a last-round unit
  // whose dK/dV partial goes to slot ``part`` of the f32 partials
  int h0, hn, part;
};

// TMEM column, relative to a step's S^T buffer, of the 16-bit pair of P^T
// that holds query q (q even; the pair is queries q, q + 1).  Each softmax
// warpgroup owns ``half`` consecutive query columns of S^T and writes its P^T
// pairs into the first half of them and its dS^T pairs (same offset plus
// half / 2) into the second half, so no warp overwrites columns that another
// warp still has to read.  A K-step of 16 queries is 8 consecutive columns.
__host__ __device__ constexpr uint32_t pair_col(int q, int half) {
  return static_cast<uint32_t>((q / half) * half + (q % half) / 2);
}

// bf16 steps whose largest P exceeds this add the 16-bit rounding residuals of
// P and dS through a second pair of dV / dK MMAs (dV += P_lo^T dO, dK +=
// dS_lo^T Q).  P is rounded to the input dtype before the dV product, as the
// TileOPs page's "Tiled" program does; with bf16's 8-bit significand the
// rounding errors of large P (short causal rows) summed over a group's heads
// exceed the bf16 tolerance, while steps whose P all stay at or below 1/8 keep
// them well inside it (a bit-exact model of the rounding over group sizes up
// to 16 puts the worst element at 0.34 of the tolerance).
constexpr float kSplitP = 0.125f;
constexpr uint32_t kSplitPBf16x2 = 0x3E003E00u;  // kSplitP as two bf16 patterns
// The residuals are compiled into the bf16 kernels that serve groups of more
// than this many query heads per KV head; up to 4 heads, the same model keeps
// the plain 16-bit rounding within 0.76 of the tolerance, and those launches
// run without the check (it costs the softmax warps a few percent).
constexpr int kSplitMinGroup = 4;

// (batch, KV head) pairs whose tiles are drawn together (dense batches): at
// most kTileGroup, and no more than the CTAs in flight can cover at once
// (about one tile of every pair of the group per CTA).
constexpr int kTileGroup = 8;
// Most last-round tiles whose dK/dV partials a workspace holds (the last round
// has fewer tiles than the launch has CTAs).
constexpr int kMaxTailTiles = 256;
__host__ __device__ inline int tile_group(int ctas, int tiles_per_pair) {
  const int g = tiles_per_pair > 0 ? ctas / tiles_per_pair : kTileGroup;
  return g < 1 ? 1 : (g > kTileGroup ? kTileGroup : g);
}

// Tile t -> (batch, KV head, key block); longest tiles first (smallest key
// block index first, which is the longest under a causal mask).  Dense
// batches go through the (batch, KV head) pairs in groups of p.tile_group,
// key block major inside a group: the CTAs in flight then share the Q/dO rows
// and dQ accumulator rows of a few heads, which stay in L2, at no cost in
// load balance (each group still ends with its shortest tiles).  Long rows
// (more key tiles per pair than CTAs) take groups of one pair: all CTAs then
// work on the same KV head, whose dQ accumulator rows fit L2, instead of
// sweeping the accumulators of several heads at once.  Packed
// sequences keep key block major order over all pairs (their tile count per
// pair is known only on the device, and the draws past it end a CTA's work).
// Host code may call it too (with cu_seqlens in host memory) to check the order.
// Draws from p.tail_start on (when p.tail_tiles > 0) are last-round units:
// unit u is tile p.tail_start + u % p.tail_tiles, heads from
// (u / p.tail_tiles) * p.tail_hpu, so the units of one head slice of every
// tail tile come before the next slice.
static __host__ __device__ __forceinline__ TileInfo decode_tile(int t, const DenseParams& p) {
  TileInfo ti{};
  ti.valid = 0;
  ti.h0 = 0;
  ti.hn = p.G;
  ti.part = -1;
  const int BH = p.B * p.HKV;
  if (t < 0) return ti;
  if (p.tail_tiles > 0 && t >= p.tail_start) {
    const int u = t - p.tail_start;
    if (u >= p.tail_tiles * (p.G / p.tail_hpu)) return ti;
    ti.part = u % p.tail_tiles;
    ti.h0 = (u / p.tail_tiles) * p.tail_hpu;
    ti.hn = p.tail_hpu;
    t = p.tail_start + ti.part;
  }
  int bh, r;
  if (p.cu_seqlens == nullptr) {
    const int nt = (p.Sk + kDenseBM - 1) / kDenseBM;  // key tiles per pair
    const int grp = imin(BH, p.tile_group > 0 ? p.tile_group : kTileGroup);
    const int gi = t / (grp * nt);
    const int g0 = gi * grp;
    if (g0 >= BH) return ti;
    const int gn = imin(grp, BH - g0);  // the last group may hold fewer pairs
    const int u = t - gi * grp * nt;
    if (u >= gn * nt) return ti;
    bh = g0 + u % gn;
    r = u / gn;
  } else {
    bh = t % BH;
    r = t / BH;
  }
  ti.b = bh / p.HKV;
  ti.g = bh % p.HKV;
  if (p.cu_seqlens != nullptr) {
    bool found = false;
    for (int n = 0; n < p.num_seqs; ++n) {
      const int a = clamp_pos(p.cu_seqlens[n], p.S), e = clamp_pos(p.cu_seqlens[n + 1], p.S);
      const int nt = e > a ? (e - a + kDenseBM - 1) / kDenseBM : 0;
      if (r < nt) {
        ti.seq_start = a;
        ti.len = ti.qlen = e - a;
        ti.off = 0;
        found = true;
        break;
      }
      r -= nt;
    }
    if (!found) return ti;
  } else {
    ti.seq_start = 0;
    ti.len = p.Sk;
    ti.qlen = p.S;
    ti.off = p.Sk - p.S;
  }
  ti.k0 = r * kDenseBM;
  int lo, hi;
  query_block_range_qk(ti.k0, kDenseBM, ti.len, ti.qlen, ti.off, p.causal, p.window, p.bn, &lo, &hi);
  ti.qlo = lo;
  ti.nq = hi - lo;
  ti.valid = 1;
  return ti;
}

}  // namespace ab
