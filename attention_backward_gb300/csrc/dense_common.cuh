// Tile decoding shared by the dense backward kernels: a tile is a block of
// kDenseBM key rows of one KV head (and batch row, or packed sequence).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace ab {

struct TileInfo {
  int b, g, seq_start, len, k0, qlo, nq, valid;
};

// Tile t -> (batch, KV head, key block); longest tiles first (smallest key
// block index first, which is the longest under a causal mask).
static __device__ __forceinline__ TileInfo decode_tile(int t, const DenseParams& p) {
  TileInfo ti{};
  ti.valid = 0;
  const int BH = p.B * p.HKV;
  if (t < 0) return ti;
  const int bh = t % BH;
  int r = t / BH;
  ti.b = bh / p.HKV;
  ti.g = bh % p.HKV;
  if (p.cu_seqlens != nullptr) {
    bool found = false;
    for (int n = 0; n < p.num_seqs; ++n) {
      const int a = clamp_pos(p.cu_seqlens[n], p.S), e = clamp_pos(p.cu_seqlens[n + 1], p.S);
      const int nt = e > a ? (e - a + kDenseBM - 1) / kDenseBM : 0;
      if (r < nt) {
        ti.seq_start = a;
        ti.len = e - a;
        found = true;
        break;
      }
      r -= nt;
    }
    if (!found) return ti;
  } else {
    if (static_cast<int64_t>(r) * kDenseBM >= p.S) return ti;
    ti.seq_start = 0;
    ti.len = p.S;
  }
  ti.k0 = r * kDenseBM;
  int lo, hi;
  query_block_range(ti.k0, kDenseBM, ti.len, p.causal, p.window, p.bn, &lo, &hi);
  ti.qlo = lo;
  ti.nq = hi - lo;
  ti.valid = 1;
  return ti;
}

}  // namespace ab
