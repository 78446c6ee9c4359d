// The forward that produces the backward's inputs: O = softmax(Q K^T * scale) V
// and the natural-log LSE of every query row, for the dense masks of the
// backward (causal, sliding window, packed sequences, unequal query and key
// lengths) and grouped-query heads.  The TileOPs MHA backward page assumes
// this forward ("Summary": the backward op takes q, k, v, o, do, lse); its
// "Reference" program's first half (scores, masked softmax, LSE) is what each
// row computes here.
//
// Structure (persistent CTAs, one per SM, each walking units of two 128-row
// query tiles of one query head):
//
//   S_w  = Q_w K_j^T         tensor core, M = 128 queries, N = 128 keys, K = D
//   m    = running row max of S_w * scale * log2(e) (lazily updated, below)
//   P_w  = exp2(S_w * scale * log2(e) - m), masked; rounded to 16 bits into TMEM
//   O_w += P_w V_j           A operand = P_w from TMEM, B = V_j (MN-major)
//   l    = running row sum of P_w (f32, before rounding)
//
// and at the end O = O_w / l, LSE = (m + log2 l) * ln 2.
//
// Two softmax warpgroups, one per query tile, each own an S buffer and an O
// accumulator in TMEM (S_0 at column 0, S_1 at 128, O_0 at 256, O_1 at 256 +
// D), with one row per thread.  The MMA warp interleaves the tiles so that the
// tensor core computes one tile's P V and the next S while the other tile's
// softmax runs: S_0(j), S_1(j), P_0 V(j), S_0(j+1), P_1 V(j), S_1(j+1), ...
// An S MMA overwrites the P columns that the same tile's previous P V read;
// MMAs issued by one thread execute in issue order, so no wait separates them.
//
// Lazy rescaling: a row keeps the max m it last used.  P = exp2(s - m) stays
// at most 2^8 unless the row max grows more than 8 past m; only then does the
// row's thread wait for its tile's previous P V, scale its O row and l by
// exp2(m_old - m_new) in TMEM and adopt the new max.  Rows of random scores
// rarely need it after their first blocks.
//
// K and V come through a ring of TMA stages (2 at head dim 128, 4 at 64), K
// and V of a stage with barriers of their own.  Packed tails (rows past the
// last sequence) are zeroed in shared memory before a V tile that reaches them
// is published: a zero P times a NaN V row would be NaN.
//
// Warp roles (12 warps): 0-3 softmax of tile 0, 4-7 softmax of tile 1 (each
// also writes its tile's O and LSE), 8 TMA producer, 9 MMA issuer, 10-11 idle
// (they complete the control warpgroup of the register split).  Every wait
// is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#define AB_INLINE_WAITS 1
#include "common.cuh"
#include "cvt.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace ab {

namespace {

constexpr int BQ = 128;  // query rows per tile
constexpr int BK = 128;  // keys per block
constexpr int THREADS = 12 * 32;
// launched at 168 registers a thread (12 warps), re-split per warpgroup: the
// two softmax warpgroups hold a row of 128 scores each; the control warpgroup
// keeps the unit walk and the barrier phases of the persistent loop
constexpr uint32_t REG_SOFT = 208, REG_CTL = 88;
static_assert(2 * REG_SOFT + REG_CTL == 3 * 168, "register split must equal the launch's registers");
constexpr float kRescaleLog2 = 8.f;  // rescale once a row max grows past 2^8

template <int D>
struct FwdCfg {
  static constexpr int NSLAB = D / 64;          // 64-column (128-byte) slabs per row
  static constexpr int SLAB = BQ * 128;         // [128 rows x 64 cols] 16-bit, 128-byte swizzled
  static constexpr int TILE = NSLAB * SLAB;     // one 128-row tile of Q, K or V
  static constexpr int ST = D == 64 ? 4 : 2;    // K/V stages
  static constexpr int OFF_Q = 0;               // two query tiles
  static constexpr int OFF_KV = OFF_Q + 2 * TILE;  // stage s: K at OFF_KV + 2s*TILE, V after it
  static constexpr int OFF_BAR = OFF_KV + 2 * ST * TILE;
  static constexpr int NBAR = 32;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t T_S0 = 0, T_S1 = 128, T_O0 = 256, T_O1 = 256 + D;
};

enum FwdBar : int {
  Q_FULL = 0,
  Q_EMPTY,            // every S MMA of the unit has completed: the Q tiles may be reloaded
  K_FULL0,            // ST stages
  V_FULL0 = K_FULL0 + 4,
  KV_EMPTY0 = V_FULL0 + 4,
  S_FULL0 = KV_EMPTY0 + 4,  // per tile
  P_READY0 = S_FULL0 + 2,   // per tile: 4 softmax warps stored P
  O_DONE0 = P_READY0 + 2,   // per tile: the tile's P V MMAs issued so far completed
  O_FREE0 = O_DONE0 + 2,    // per tile: 4 softmax warps read the unit's O rows
  UNIT_FULL0 = O_FREE0 + 2,   // 2 ring slots: the producer published a unit index
  UNIT_EMPTY0 = UNIT_FULL0 + 2,  // 2 ring slots: the MMA warp and the 8 softmax warps read it
  TAIL = UNIT_EMPTY0 + 2,
  DRAIN,
  NUM_FWD_BARS
};
static_assert(NUM_FWD_BARS <= 32, "barrier storage");

// The unit a CTA owns: two query tiles of one query head, both in one
// sequence (a dense batch row or a packed sequence), and each tile's block
// range [lo, hi) of 128-key blocks.
struct FwdUnit {
  int valid, b, h, seq_start, qlen, klen, off, q0;
  int lo[2], hi[2];  // lo == hi: the tile sees no key; q0 + 128 w >= qlen: the tile is absent
};

// Key blocks [lo, hi) that query rows [q0, q1) of a row of ``qlen`` queries and
// ``klen`` keys see (query i at key position i + off).
__device__ __forceinline__ void key_block_range(int q0, int qlen, int klen, int off, int causal, int window,
                                                int* lo, int* hi) {
  *lo = *hi = 0;
  if (q0 >= qlen || klen <= 0) return;
  const int q1 = imin(q0 + BQ, qlen);
  int64_t ks = 0, ke = klen;
  if (causal || window > 0) {
    const int64_t e = static_cast<int64_t>(q1) + off;  // last visible key + 1
    ke = e < klen ? e : klen;
  }
  if (window > 0) {
    const int64_t s = static_cast<int64_t>(q0) + off - window + 1;
    ks = s > 0 ? s : 0;
  }
  if (ke <= ks) return;
  *lo = static_cast<int>(ks / BK);
  *hi = static_cast<int>((ke + BK - 1) / BK);
}

// Unit u of the launch, longest first under a causal mask (the last query
// tiles of a row see the most keys): dense rows go through the tile pairs
// from the last, each over all (batch, head) pairs; packed sequences one after
// another, each the same way over its heads.
__device__ __forceinline__ FwdUnit decode_unit(int u, const FwdParams& p) {
  FwdUnit t{};
  t.valid = 0;
  if (u < 0) return t;  // the end-of-work marker
  int pair = 0;
  if (p.cu_seqlens == nullptr) {
    const int np = (p.S + 2 * BQ - 1) / (2 * BQ);
    const int bh = p.B * p.HQ;
    if (u < 0 || u >= np * bh) return t;
    pair = np - 1 - u / bh;
    t.b = (u % bh) / p.HQ;
    t.h = (u % bh) % p.HQ;
    t.seq_start = 0;
    t.qlen = p.S;
    t.klen = p.Sk;
    t.off = p.Sk - p.S;
  } else {
    int rem = u, found = 0;
    for (int n = 0; n < p.num_seqs; ++n) {
      const int a = clamp_pos(p.cu_seqlens[n], p.S), e = clamp_pos(p.cu_seqlens[n + 1], p.S);
      const int len = e > a ? e - a : 0;
      const int np = (len + 2 * BQ - 1) / (2 * BQ);
      if (rem < np * p.HQ) {
        pair = np - 1 - rem / p.HQ;
        t.h = rem % p.HQ;
        t.b = 0;
        t.seq_start = a;
        t.qlen = t.klen = len;
        t.off = 0;
        found = 1;
        break;
      }
      rem -= np * p.HQ;
    }
    if (!found) return t;
  }
  t.q0 = pair * 2 * BQ;
  for (int w = 0; w < 2; ++w)
    key_block_range(t.q0 + w * BQ, t.qlen, t.klen, t.off, p.causal, p.window, &t.lo[w], &t.hi[w]);
  t.valid = 1;
  return t;
}

// The blocks [J0, J1) of a unit that some tile sees (J0 == J1: none).
struct UnitSpan {
  bool has[2];
  int J0, J1;
};

__device__ __forceinline__ UnitSpan unit_span(const FwdUnit& u) {
  UnitSpan s;
  s.J0 = 0x7fffffff;
  s.J1 = 0;
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    s.has[w] = u.lo[w] < u.hi[w];
    if (s.has[w]) {
      s.J0 = imin(s.J0, u.lo[w]);
      s.J1 = imax(s.J1, u.hi[w]);
    }
  }
  if (s.J1 == 0) s.J0 = 0;
  return s;
}

// Persistent: each CTA's producer draws units, longest first, from a counter
// in the workspace header (cleared by the host before the launch) and
// publishes each draw to the other roles through a two-slot ring in shared
// memory; a draw past the last unit ends every role.  Barrier phases run on
// across units (K/V stages by a block counter, the S / P / O barriers of a
// tile by that tile's block counter), and two barriers hand the shared Q tiles
// (Q_EMPTY: every S MMA of the unit has completed) and a tile's O accumulator
// (O_FREE: its softmax warps have read O) to the next unit.
template <int D, bool BF16>
__global__ void __launch_bounds__(THREADS, 1) dense_fwd_kernel(const __grid_constant__ FwdMaps maps,
                                                               const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int ST = C::ST;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 8);
  volatile int* ring = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 16);  // 2 unit indices
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if ((smem_u32(sm) & 1023u) != 0) {  // the swizzled tiles need an aligned base
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kErrAlign);
    return;
  }

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(&bars[Q_FULL], 1);
    mbar_init(&bars[Q_EMPTY], 1);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&bars[K_FULL0 + i], 1);
      mbar_init(&bars[V_FULL0 + i], 1);
      mbar_init(&bars[KV_EMPTY0 + i], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bars[S_FULL0 + w], 1);
      mbar_init(&bars[P_READY0 + w], 4);
      mbar_init(&bars[O_DONE0 + w], 1);
      mbar_init(&bars[O_FREE0 + w], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[UNIT_FULL0 + i], 1);
      mbar_init(&bars[UNIT_EMPTY0 + i], 9);
    }
    mbar_init(&bars[TAIL], 1);
    mbar_init(&bars[DRAIN], 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  auto finish = [&]() {
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
    if (warp == 9) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
  };

  // the uc-th unit of this CTA (consumers): waits for the producer's draw,
  // hands the slot back, decodes; invalid once the draws are exhausted
  auto next_unit = [&](uint32_t uc, bool* okp) -> FwdUnit {
    const uint32_t slot = uc & 1;
    FwdUnit u{};
    u.valid = 0;
    if (!(*okp = mbar_wait_warp(&bars[UNIT_FULL0 + slot], (uc >> 1) & 1, wc, kErrWaitTile))) return u;
    const int t = ring[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[UNIT_EMPTY0 + slot]);
    return decode_unit(t, p);
  };

  if (warp >= 8) {
    setmaxnreg_dec<REG_CTL>();
    if (warp == 8) {
      // ============================================================ producer
      int q_pend = -1, tail_pend = -1;
      uint32_t qc = 0, kc = 0, tail_ph = 0;
      bool ok = true;
      // key rows from tail0 on belong to no packed sequence and may hold anything
      const int rows = p.cu_seqlens ? p.S : p.Sk;
      const int tail0 = p.cu_seqlens ? clamp_pos(p.cu_seqlens[p.num_seqs], p.S) : p.Sk;
      for (uint32_t uc = 0; ok; ++uc) {
        const uint32_t slot = uc & 1;
        if (uc >= 2 && !(ok = mbar_wait_warp(&bars[UNIT_EMPTY0 + slot], ((uc >> 1) - 1) & 1, wc, kErrWaitTile)))
          break;
        int t = 0;
        if (lane == 0) t = atomicAdd(p.unit_counter, 1);
        t = __shfl_sync(0xffffffffu, t, 0);
        const FwdUnit u = decode_unit(t, p);
        if (lane == 0) {
          ring[slot] = u.valid ? t : -1;
          mbar_arrive(&bars[UNIT_FULL0 + slot]);
        }
        if (!u.valid) break;
        const UnitSpan sp = unit_span(u);
        if (sp.J1 <= sp.J0) continue;
        // the previous unit's S MMAs have read its Q tiles
        if (qc >= 1 && !(ok = mbar_wait_warp(&bars[Q_EMPTY], (qc - 1) & 1, wc, kErrWaitStageEmpty))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[Q_FULL], (sp.has[0] + sp.has[1]) * C::TILE);
          for (int w = 0; w < 2; ++w) {
            if (!sp.has[w]) continue;
#pragma unroll
            for (int s = 0; s < C::NSLAB; ++s)
              tma_load_4d(sm + C::OFF_Q + w * C::TILE + s * C::SLAB, &maps.q, &bars[Q_FULL], s * 64, u.h,
                          u.seq_start + u.q0 + w * BQ, u.b);
          }
        }
        q_pend = qc & 1;
        ++qc;
        const int kvh = u.h / p.G;
        for (int j = sp.J0; j < sp.J1; ++j, ++kc) {
          const int st = kc % ST, n = kc / ST;
          if (n >= 1 && !(ok = mbar_wait_warp(&bars[KV_EMPTY0 + st], (n - 1) & 1, wc, kErrWaitStageEmpty))) break;
          uint8_t* dk = sm + C::OFF_KV + 2 * st * C::TILE;
          uint8_t* dv = dk + C::TILE;
          const int pos = u.seq_start + j * BK;
          int r0, r1;
          tail_rows(pos, BK, tail0, rows, &r0, &r1);
          if (r0 < r1) {
            // loaded onto the producer's own barrier, the tail rows zeroed, then published
            if (lane == 0) {
              mbar_arrive_expect_tx(&bars[TAIL], 2 * C::TILE);
#pragma unroll
              for (int s = 0; s < C::NSLAB; ++s) {
                tma_load_4d(dk + s * C::SLAB, &maps.k, &bars[TAIL], s * 64, kvh, pos, u.b);
                tma_load_4d(dv + s * C::SLAB, &maps.v, &bars[TAIL], s * 64, kvh, pos, u.b);
              }
            }
            tail_pend = tail_ph & 1;
            if (!(ok = mbar_wait_warp(&bars[TAIL], tail_ph & 1, wc, kErrWaitTail))) break;
            tail_pend = -1;
            ++tail_ph;
            zero_tile_rows(dk, C::NSLAB, C::SLAB, r0, r1, lane);
            zero_tile_rows(dv, C::NSLAB, C::SLAB, r0, r1, lane);
            if (lane == 0) {
              mbar_arrive(&bars[K_FULL0 + st]);
              mbar_arrive(&bars[V_FULL0 + st]);
            }
          } else if (lane == 0) {
            mbar_arrive_expect_tx(&bars[K_FULL0 + st], C::TILE);
#pragma unroll
            for (int s = 0; s < C::NSLAB; ++s)
              tma_load_4d(dk + s * C::SLAB, &maps.k, &bars[K_FULL0 + st], s * 64, kvh, pos, u.b);
            mbar_arrive_expect_tx(&bars[V_FULL0 + st], C::TILE);
#pragma unroll
            for (int s = 0; s < C::NSLAB; ++s)
              tma_load_4d(dv + s * C::SLAB, &maps.v, &bars[V_FULL0 + st], s * 64, kvh, pos, u.b);
          }
        }
      }
      // loads still in flight land before the CTA exits: the last Q and the last ST blocks'
      if (lane == 0) {
        if (q_pend >= 0) mbar_drain(&bars[Q_FULL], q_pend);
        if (tail_pend >= 0) mbar_drain(&bars[TAIL], tail_pend);
        for (uint32_t i = kc > static_cast<uint32_t>(ST) ? kc - ST : 0u; i < kc; ++i) {
          mbar_drain(&bars[K_FULL0 + i % ST], (i / ST) & 1);
          mbar_drain(&bars[V_FULL0 + i % ST], (i / ST) & 1);
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ============================================================ MMA issuer
      constexpr uint32_t IDESC_S = idesc_f16(BF16, 128, BK, false, false);
      constexpr uint32_t IDESC_PV = idesc_f16(BF16, 128, D, false, true);
      const uint32_t sbase = smem_u32(sm);
      const uint64_t q_kmaj = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t k_kmaj = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);
      const uint64_t v_mn = sdesc_sw128(sbase + C::OFF_KV + C::TILE, C::SLAB, 1024);
      uint32_t qc = 0, kc = 0, npv0 = 0, npv1 = 0, oc0 = 0, oc1 = 0;
      bool ok = true;
      for (uint32_t uc = 0; ok; ++uc) {
        const FwdUnit u = next_unit(uc, &ok);
        if (!ok || !u.valid) break;
        const UnitSpan sp = unit_span(u);
        if (sp.J1 <= sp.J0) continue;
        const int J0 = sp.J0, J1 = sp.J1;
        const uint32_t kc0 = kc;  // block counter at the unit's first block
        auto in = [&](int w, int j) { return sp.has[w] && u.lo[w] <= j && j < u.hi[w]; };
        auto issue_s = [&](int w, int j) {
          const uint64_t ko0 = sdesc_step(2 * ((kc0 + j - J0) % ST) * C::TILE);
          const uint64_t qo = sdesc_step(w * C::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ko = sdesc_step((kk / 4) * C::SLAB + (kk % 4) * 32);
            mma_ss_w(tmem + (w ? C::T_S1 : C::T_S0), q_kmaj + qo + ko, k_kmaj + ko0 + ko, IDESC_S, kk > 0);
          }
          mma_commit_w(&bars[S_FULL0 + w]);
        };
        auto issue_pv = [&](int w, int j) -> bool {
          uint32_t& npv = w ? npv1 : npv0;
          if (!mbar_wait_warp(&bars[P_READY0 + w], npv & 1, wc, kErrWaitP)) return false;
          if (j == u.lo[w]) {
            // the tile's O accumulator: its softmax warps have read the previous unit's O
            const uint32_t oc = w ? oc1 : oc0;
            if (oc >= 1 && !mbar_wait_warp(&bars[O_FREE0 + w], (oc - 1) & 1, wc, kErrWaitDQEmpty)) return false;
          }
          tc_fence_after();
          const uint64_t vo = sdesc_step(2 * ((kc0 + j - J0) % ST) * C::TILE);
          const uint32_t ts = tmem + (w ? C::T_S1 : C::T_S0), to = tmem + (w ? C::T_O1 : C::T_O0);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_ts_w(to, ts + kk * 8, v_mn + vo + sdesc_step(kk * 2048), IDESC_PV, j > u.lo[w] || kk > 0);
          mma_commit_w(&bars[O_DONE0 + w]);
          ++npv;
          return true;
        };
        auto wait_k = [&](int j) {
          const uint32_t i = kc0 + j - J0;
          return mbar_wait_warp(&bars[K_FULL0 + i % ST], (i / ST) & 1, wc, kErrWaitKV);
        };
        ok = mbar_wait_warp(&bars[Q_FULL], qc & 1, wc, kErrWaitStageFull) && wait_k(J0);
        ++qc;
        if (ok) {
          tc_fence_after();
          if (in(0, J0)) issue_s(0, J0);
          if (in(1, J0)) issue_s(1, J0);
        }
        for (int j = J0; j < J1 && ok; ++j) {
          const uint32_t i = kc0 + j - J0;
          const int st = i % ST;
          if (!(ok = mbar_wait_warp(&bars[V_FULL0 + st], (i / ST) & 1, wc, kErrWaitKV))) break;
          tc_fence_after();
          if (in(0, j) && !(ok = issue_pv(0, j))) break;
          const bool next = j + 1 < J1;
          if (next) {
            if (!(ok = wait_k(j + 1))) break;
            tc_fence_after();
            if (in(0, j + 1)) issue_s(0, j + 1);
          }
          if (in(1, j) && !(ok = issue_pv(1, j))) break;
          mma_commit_w(&bars[KV_EMPTY0 + st]);  // every reader of K_j and V_j issued
          if (next && in(1, j + 1)) issue_s(1, j + 1);
        }
        if (!ok) break;
        mma_commit_w(&bars[Q_EMPTY]);  // every S MMA of the unit issued
        kc += J1 - J0;
        oc0 += sp.has[0] ? 1u : 0u;
        oc1 += sp.has[1] ? 1u : 0u;
      }
      // every MMA issued by this warp completes before TMEM is released
      mma_commit_w(&bars[DRAIN]);
      if (lane == 0) mbar_drain(&bars[DRAIN], 0);
      __syncwarp();
    }
    // warps 10-11: nothing to do
    finish();
    return;
  }

  setmaxnreg_inc<REG_SOFT>();
  // ============================================================ softmax of tile w (lane = query row)
  const int w = warp >> 2, quad = warp & 3;
  const int row = quad * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tS = tmem + lane_off + (w ? C::T_S1 : C::T_S0);
  const uint32_t tO = tmem + lane_off + (w ? C::T_O1 : C::T_O0);
  const bool cm = p.causal || p.window > 0;
  const int W = p.window;
  uint32_t c = 0;  // blocks of this tile over all units so far
  bool ok = true;
  for (uint32_t uc = 0; ok; ++uc) {
    const FwdUnit u = next_unit(uc, &ok);
    if (!ok || !u.valid) break;
    const int qt0 = u.q0 + w * BQ;  // first (sequence-local) query of the tile
    if (qt0 >= u.qlen) continue;    // the tile is past the end of its sequence
    const int lo_w = w ? u.lo[1] : u.lo[0], hi_w = w ? u.hi[1] : u.hi[0];
    const int q = qt0 + row;
    const uint32_t c0 = c;
    float m_used = -INFINITY, l = 0.f;
    for (int j = lo_w; j < hi_w; ++j, ++c) {
      if (!(ok = mbar_wait_warp(&bars[S_FULL0 + w], c & 1, wc, kErrWaitS))) break;
      tc_fence_after();
      uint32_t sr[BK];
#pragma unroll
      for (int ch = 0; ch < BK / 32; ++ch) tmem_ld32(tS + ch * 32, sr + ch * 32);
      tmem_ld_wait();
      const int k0 = j * BK;
      // every key and query of the block in range and inside the mask
      const bool full_vis = k0 + BK <= u.klen && qt0 + BQ <= u.qlen && (!cm || qt0 + u.off >= k0 + BK - 1) &&
                            (W <= 0 || qt0 + BQ - 1 + u.off < k0 + W);
      // row max over four independent chains
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (full_vis) {
#pragma unroll
        for (int k = 0; k < BK; ++k) mx4[k & 3] = fmaxf(mx4[k & 3], __uint_as_float(sr[k]));
      } else {
        // keys k in [k_lo, k_hi) of the block are visible to my query (one range per row)
        const int64_t d0 = static_cast<int64_t>(q) + u.off - k0;  // my key position relative to the block
        int64_t lo = 0, hi = u.klen - k0;
        if (cm) hi = hi < d0 + 1 ? hi : d0 + 1;
        if (W > 0) lo = d0 - W + 1 > 0 ? d0 - W + 1 : 0;
        if (q >= u.qlen) hi = 0;
        const int k_lo = static_cast<int>(lo > BK ? BK : lo), k_hi = static_cast<int>(hi < 0 ? 0 : (hi > BK ? BK : hi));
#pragma unroll
        for (int k = 0; k < BK; ++k) {
          const float s = (k >= k_lo && k < k_hi) ? __uint_as_float(sr[k]) : -INFINITY;
          sr[k] = __float_as_uint(s);
          mx4[k & 3] = fmaxf(mx4[k & 3], s);
        }
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      // the row max in log2 units (scale_log2 > 0 keeps the order of the raw scores)
      const float m_new = fmaxf(m_used, mx * p.scale_log2);
      // a row whose max grew past the threshold is rescaled; a row that had no
      // visible key so far adopts the new max (its O row and l are zero)
      const bool resc = m_used != -INFINITY && m_new > m_used + kRescaleLog2;
      const float f = resc ? ex2(m_used - m_new) : 1.f;
      if (__any_sync(0xffffffffu, resc)) {
        // the tile's previous P V (of this unit: m_used is finite) has completed
        // before its O rows are scaled
        if (!(ok = mbar_wait_warp(&bars[O_DONE0 + w], (c - 1) & 1, wc, kErrWaitDQFull))) break;
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(tO + ch * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
          tmem_st16(tO + ch * 32, r);
          tmem_st16(tO + ch * 32 + 16, r + 16);
        }
      }
      l *= f;
      if (resc || m_used == -INFINITY) m_used = m_new;
      const float msub = m_used == -INFINITY ? 0.f : m_used;
      // S * scale - m two keys per instruction (f32x2 FMA), the row sum in two
      // f32x2 accumulators
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-msub, -msub);
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int ch = 0; ch < BK / 32; ++ch) {
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(sr[ch * 32 + 2 * e]), __uint_as_float(sr[ch * 32 + 2 * e + 1])), sc2, nm2);
          const float2 pp = make_float2(ex2(x.x), ex2(x.y));
          sum2[e & 1] = __fadd2_rn(sum2[e & 1], pp);
          pw[e] = pack2<BF16>(pp.x, pp.y);
        }
        // P pairs of keys 32ch .. 32ch + 31 into S columns 16ch .. 16ch + 15 (the
        // scores of this row were all loaded above)
        tmem_st16(tS + ch * 16, pw);
      }
      l += (sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[P_READY0 + w]);
    }
    if (!ok) break;
    // ---- O = O_w / l and the natural-log LSE of the row
    const bool had = c > c0;  // the tile saw a key block in this unit
    if (had) {
      if (!(ok = mbar_wait_warp(&bars[O_DONE0 + w], (c - 1) & 1, wc, kErrWaitDQFull))) break;
      tc_fence_after();
    }
    const bool live = q < u.qlen;
    const int64_t pos = u.seq_start + q;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    if (live)
      p.lse[u.b * p.sl_b + u.h * p.sl_h + pos * p.sl_s] =
          l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
    uint8_t* const out = p.o + 2 * (u.b * p.so_b + pos * p.so_s + u.h * p.so_h);
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t r[32];
      if (had) {
        tmem_ld32(tO + ch * 32, r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = 0u;
      }
      if (live) {
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint4 v;
          v.x = pack2<BF16>(__uint_as_float(r[c8 * 8 + 0]) * inv, __uint_as_float(r[c8 * 8 + 1]) * inv);
          v.y = pack2<BF16>(__uint_as_float(r[c8 * 8 + 2]) * inv, __uint_as_float(r[c8 * 8 + 3]) * inv);
          v.z = pack2<BF16>(__uint_as_float(r[c8 * 8 + 4]) * inv, __uint_as_float(r[c8 * 8 + 5]) * inv);
          v.w = pack2<BF16>(__uint_as_float(r[c8 * 8 + 6]) * inv, __uint_as_float(r[c8 * 8 + 7]) * inv);
          *reinterpret_cast<uint4*>(out + 2 * (ch * 32 + c8 * 8)) = v;
        }
      }
    }
    if (had) {
      // this unit's O rows are read: the next unit's first P V may overwrite them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[O_FREE0 + w]);
    }
  }
  finish();
}

template <int D, bool BF16>
cudaError_t launch_t(const FwdParams& p, const FwdMaps& m, int grid, cudaStream_t st) {
  auto kern = dense_fwd_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, THREADS, FwdCfg<D>::SMEM, st>>>(m, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, const FwdMaps& m, bool bf16, int grid, cudaStream_t st) {
  if (p.D == 64) return bf16 ? launch_t<64, true>(p, m, grid, st) : launch_t<64, false>(p, m, grid, st);
  return bf16 ? launch_t<128, true>(p, m, grid, st) : launch_t<128, false>(p, m, grid, st);
}

}  // namespace ab
