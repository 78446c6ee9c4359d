// Launch 2 of the top-k sparse backward over shared latent rows (the tilelang
// pull request "Adaptive threads for sparse MLA backward": H = 64 query heads
// per KV group, one latent row of DQK = 576 per key with V its first DV = 512
// columns, top-k index lists).  Smaller groups (the page's tensor-parallel
// splits, "Applicability") are padded to 64 heads: the padding heads get an
// infinite LSE, so their P and dS are exactly zero, at 64/G times the work.
//
// A unit of work is one (batch, token t, KV group g) with all 64 of its query
// heads.  Its index list is processed in blocks of BK = 128 slots; per block:
//
//   gather   the 128 latent rows idx[t, slot] (TMA tile::gather4 into nine
//            64-column, 128-byte-swizzled slabs; invalid slots read zeros)
//   S^T  = K_sel Q_t^T           M = 128 slots, N = 64 heads, K = 576
//   dP^T = V_sel dO_t^T          K = 512
//   P^T  = exp2(S^T*scale*log2e - LSE2[h])   (0 for invalid slots)
//   dS^T = P^T o (dP^T - delta[h]) * scale   (scale applied here: dKV mixes
//                                             the scaled dK with the unscaled dV)
//   dQ_t^T += K_sel^T dS^T       five M-tiles of 128 head dims, accumulated in
//                                TMEM over all blocks of the token
//   dKV_sel = dS^T Q_t + [P^T dO_t, 0]   with P and dS as 16-bit hi + lo pairs
//                                (64 heads add into every latent row, so one
//                                16-bit rounding would accumulate past the
//                                tolerance); nine 64-column chunks, each
//                                scatter-added into the f32 dKV accumulator
//                                row idx[slot] with one bulk reduce per slot
//
// The token's dQ is complete when its last block is done and is written once
// in the input dtype; only dKV needs an accumulator (and a landing pass).
// Q_t and dO_t (72 KB + 64 KB) do not fit next to the 144 KB slot block, so
// they stream through a 3-slot ring of 64 x 64 chunks, twice per block (once
// for S^T/dP^T, once for dKV).  Enough gathers are kept in flight by issuing
// all 288 gather4 of a block from the 32 lanes of the producer warp as soon
// as the previous block's last reader of the slot block (dQ^T) has been issued
// (the Little's-law argument of the tilelang page, "Mechanism").
//
// Warp roles (11 warps): 0-3 dKV epilogue (lane = slot), 4-7 softmax/dS
// (lane = slot, all 64 heads) and the token's dQ output, 8 Q/dO ring
// producer, 9 MMA issuer, 10 unit scheduling, index lists and gathers (a warp
// of its own, so that the next block's gather is issued the moment dQ^T frees
// the slot block instead of queueing behind the ring loads).  Every wait is
// bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "cvt.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace ab {

namespace {

constexpr int SH = 64;                  // query heads per KV group (one unit)
constexpr int DQK = 576, DV = 512;
constexpr int BK = 128;                 // slots per block
constexpr int NSK = DQK / 64, NSV = DV / 64;  // 64-column slabs of K and V
constexpr int SLAB = BK * 128;          // [128 slots x 64 cols] 16-bit
constexpr int CHUNK = SH * 128;         // [64 heads x 64 cols] 16-bit
constexpr int RING = 3;
constexpr int STG_STRIDE = 272;         // bytes per staging row (256 + 16 of padding)
constexpr int NCHUNK = NSK + NSV;       // ring chunks per pass: Q0 dO0 Q1 dO1 ... Q7 dO7 Q8

struct UnitInfo {
  int b, t, g, nb, valid, pad[3];
  float lse2[SH];
  float delta[SH];
};

constexpr int OFF_KV = 0;
constexpr int OFF_RING = OFF_KV + NSK * SLAB;
constexpr int OFF_DS = OFF_RING + RING * CHUNK;
constexpr int OFF_STG = OFF_DS + BK * 128;
constexpr int OFF_IDX = OFF_STG + BK * STG_STRIDE;
constexpr int OFF_UNIT = OFF_IDX + 2 * BK * 4;
constexpr int OFF_BAR = OFF_UNIT + 2 * static_cast<int>(sizeof(UnitInfo));
constexpr int NBAR = 32;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM = OFF_MISC + 64;
static_assert(SMEM <= 227 * 1024, "shared memory budget");
static_assert(OFF_RING % 1024 == 0 && OFF_DS % 1024 == 0, "swizzled tiles need 1024-byte alignment");

constexpr int T_DQ = 0;     // five dQ^T tiles [128 d x 64 heads] at 64-column steps
constexpr int T_S = 320;    // S^T [128 slots x 64 heads] f32; then P^T hi (upper 32) and lo (lower 32) pairs
constexpr int T_DP = 384;   // dP^T f32; then dS^T hi (upper 32) and lo (lower 32) pairs
constexpr int T_DKV = 448;  // one dKV chunk [128 slots x 64 cols] f32
constexpr int THREADS = 11 * 32;

enum Bar : int {
  RING_FULL0 = 0,   // 3
  RING_EMPTY0 = 3,  // 3
  KV_FULL0 = 6,     // 2 (by block parity)
  KV_FREE = 8,      // dQ^T (the last reader of the slot block) issued and done
  UNIT_FULL0,       // 2
  UNIT_EMPTY0 = 11, // 2
  S_FULL = 13,
  DP_FULL,
  DS_READY,         // 4 softmax warps wrote dS (TMEM and shared) and P
  DS_SFREE,         // dQ^T read the shared dS tile
  S_FREE,           // the dKV MMAs read P^T and dS^T: S^T / dP^T may be rewritten
  DKV_FULL,
  DKV_EMPTY,        // 4 epilogue warps loaded the dKV chunk
  DQ_DONE,          // every dQ^T MMA of the unit completed
  DQ_FREE,          // 4 softmax warps loaded dQ^T
  DRAIN,
  NUM_BARS
};
static_assert(NUM_BARS <= NBAR, "barrier storage");

// 168 registers: three warps of one SM sub-partition must fit its 16K registers.
template <bool BF16>
__global__ void __maxnreg__(168)
    sparse_bwd_kernel(const __grid_constant__ SparseMaps maps, const SparseParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  UnitInfo* units = reinterpret_cast<UnitInfo*>(sm + OFF_UNIT);
  int* idx_buf = reinterpret_cast<int*>(sm + OFF_IDX);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if ((smem_u32(sm) & 1023u) != 0) {  // the swizzled tiles need an aligned base
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kErrAlign);
    return;
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < RING; ++i) {
      mbar_init(&bars[RING_FULL0 + i], 1);
      mbar_init(&bars[RING_EMPTY0 + i], 1);
    }
    mbar_init(&bars[KV_FULL0], 1);
    mbar_init(&bars[KV_FULL0 + 1], 1);
    mbar_init(&bars[KV_FREE], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[UNIT_FULL0 + i], 1);
      mbar_init(&bars[UNIT_EMPTY0 + i], 10);  // ring producer, MMA warp, 4 softmax warps, 4 epilogue warps
    }
    mbar_init(&bars[S_FULL], 1);
    mbar_init(&bars[DP_FULL], 1);
    mbar_init(&bars[DS_READY], 4);
    mbar_init(&bars[DS_SFREE], 1);
    mbar_init(&bars[S_FREE], 1);
    mbar_init(&bars[DKV_FULL], 1);
    mbar_init(&bars[DKV_EMPTY], 4);
    mbar_init(&bars[DQ_DONE], 1);
    mbar_init(&bars[DQ_FREE], 4);
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
  // the preprocess (the previous kernel on the stream) has written LSE2, delta,
  // the cleared accumulators and tile counter; the landing may be scheduled now
  grid_dependency_wait();
  grid_dependents_launch();
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
  const int units_total = p.B * p.S * p.HKV;

  if (warp == 10) {
    // ============================================================ units, index lists, gathers
    int kv_pend[2] = {-1, -1};
    uint32_t gb = 0;
    bool ok = true;
    for (int uc = 0; ok; ++uc) {
      const int slot = uc & 1;
      if (uc >= 2 && !(ok = mbar_wait_warp(&bars[UNIT_EMPTY0 + slot], ((uc >> 1) - 1) & 1, wc, kErrSparseBase + 1)))
        break;
      int u = 0;
      if (lane == 0) u = atomicAdd(p.unit_counter, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      UnitInfo* ui = &units[slot];
      const bool valid = u < units_total;
      int b = 0, t = 0, g = 0, nb = 0;
      if (valid) {
        // longest lists first: tokens in decreasing order
        const int bg = u % (p.B * p.HKV);
        t = p.S - 1 - u / (p.B * p.HKV);
        b = bg / p.HKV;
        g = bg % p.HKV;
        const int* il = p.idx + b * p.si_b + static_cast<int64_t>(t) * p.si_s + g * p.si_h;
        int last = -1;
        for (int s = lane; s < p.topk; s += 32) {
          const int j = il[s];
          if (j >= 0 && j < p.SKV) last = s;
        }
        for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
        nb = last < 0 ? 0 : last / BK + 1;
        // a group of gh < 64 heads is padded to 64: the padding heads get an
        // infinite LSE, so their P and dS are exactly 0 and add nothing to dKV
        for (int h = lane; h < SH; h += 32) {
          if (h < p.gh) {
            const int64_t r = (static_cast<int64_t>(b) * p.H + g * p.gh + h) * p.S + t;
            ui->lse2[h] = p.lse2[r];
            ui->delta[h] = p.delta[r];
          } else {
            ui->lse2[h] = __int_as_float(0x7f800000);
            ui->delta[h] = 0.f;
          }
        }
      }
      if (lane == 0) {
        ui->b = b, ui->t = t, ui->g = g, ui->nb = nb, ui->valid = valid ? 1 : 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[UNIT_FULL0 + slot]);
      if (!valid) break;
      const int* il = p.idx + b * p.si_b + static_cast<int64_t>(t) * p.si_s + g * p.si_h;
      for (int blk = 0; blk < nb && ok; ++blk, ++gb) {
        // the block's latent rows, once the previous block's dQ^T is done with the slot block
        if (gb >= 1 && !(ok = mbar_wait_warp(&bars[KV_FREE], (gb - 1) & 1, wc, kErrSparseBase + 2))) break;
        int* ib = idx_buf + (gb & 1) * BK;
        int rows[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int s = blk * BK + lane * 4 + i;
          int j = s < p.topk ? il[s] : -1;
          if (j < 0 || j >= p.SKV) j = -1;
          ib[lane * 4 + i] = j;
          rows[i] = j < 0 ? -1 : (b * p.SKV + j) * p.HKV + g;  // row of the 2-D latent map
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&bars[KV_FULL0 + (gb & 1)], NSK * SLAB);
        __syncwarp();
#pragma unroll 1
        for (int s = 0; s < NSK; ++s)
          tma_gather4(sm + OFF_KV + s * SLAB + lane * 512, &maps.kv, &bars[KV_FULL0 + (gb & 1)], s * 64, rows[0],
                      rows[1], rows[2], rows[3]);
        if (gb & 1) kv_pend[1] = (gb >> 1) & 1; else kv_pend[0] = (gb >> 1) & 1;
      }
    }
    if (lane == 0) {  // gathers in flight land before the CTA exits
      if (kv_pend[0] >= 0) mbar_drain(&bars[KV_FULL0], kv_pend[0]);
      if (kv_pend[1] >= 0) mbar_drain(&bars[KV_FULL0 + 1], kv_pend[1]);
    }
  } else if (warp == 8) {
    // ============================================================ Q/dO ring producer
    uint32_t ring_used = 0, ring_par = 0;  // per ring slot: loaded at least once, parity of its last load
    uint32_t rc = 0;
    bool ok = true;
    for (int uc = 0; ok; ++uc) {
      const int slot = uc & 1;
      if (!(ok = mbar_wait_warp(&bars[UNIT_FULL0 + slot], (uc >> 1) & 1, wc, kErrSparseBase + 21))) break;
      const int valid = units[slot].valid, nb = units[slot].nb, b = units[slot].b, t = units[slot].t,
                g = units[slot].g;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[UNIT_EMPTY0 + slot]);
      if (!valid) break;
      for (int blk = 0; blk < nb && ok; ++blk) {
        // the block's Q/dO chunks, in the MMA's order, twice
        for (int pass = 0; pass < 2 && ok; ++pass) {
          for (int i = 0; i < NCHUNK; ++i, ++rc) {
            const int rs = rc % RING;
            if (rc >= static_cast<uint32_t>(RING) &&
                !(ok = mbar_wait_warp(&bars[RING_EMPTY0 + rs], (rc / RING - 1) & 1, wc, kErrSparseBase + 3)))
              break;
            if (lane == 0) {
              mbar_arrive_expect_tx(&bars[RING_FULL0 + rs], CHUNK);
              const bool isq = (i & 1) == 0;
              const int c = i >> 1;
              tma_load_4d(sm + OFF_RING + rs * CHUNK, isq ? &maps.q : &maps.dO, &bars[RING_FULL0 + rs], c * 64, g * p.gh,
                          t, b);
            }
            ring_used |= 1u << rs;
            ring_par = (ring_par & ~(1u << rs)) | (((rc / RING) & 1u) << rs);
          }
        }
      }
    }
    if (lane == 0) {  // ring loads in flight land before the CTA exits
      for (int i = 0; i < RING; ++i)
        if ((ring_used >> i) & 1u) mbar_drain(&bars[RING_FULL0 + i], (ring_par >> i) & 1u);
    }
  } else if (warp == 9) {
    // ============================================================ MMA issuer (whole warp, one elected lane)
    constexpr uint32_t IDESC_SP = idesc_f16(BF16, 128, 64, false, false);  // S^T, dP^T
    constexpr uint32_t IDESC_DQ = idesc_f16(BF16, 128, 64, true, true);    // dQ^T
    constexpr uint32_t IDESC_KV = idesc_f16(BF16, 128, 64, false, true);   // dKV chunk
    const uint32_t sbase = smem_u32(sm);
    const uint64_t dKV_k = sdesc_sw128(sbase + OFF_KV, 16, 1024);      // slab, K-major (rows = slots)
    const uint64_t dRing_k = sdesc_sw128(sbase + OFF_RING, 16, 1024);  // chunk, K-major (rows = heads)
    const uint64_t dRing_mn = sdesc_sw128(sbase + OFF_RING, 0, 1024);  // chunk as [d x heads], MN-major
    const uint64_t dDS_mn = sdesc_sw128(sbase + OFF_DS, 0, 1024);      // dS^T as [heads x slots], MN-major
    uint32_t gb = 0, rc = 0, cc = 0;
    bool ok = true;
    for (int uc = 0; ok; ++uc) {
      const int slot = uc & 1;
      if (!(ok = mbar_wait_warp(&bars[UNIT_FULL0 + slot], (uc >> 1) & 1, wc, kErrSparseBase + 4))) break;
      const int valid = units[slot].valid, nb = units[slot].nb;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[UNIT_EMPTY0 + slot]);
      if (!valid) break;
      for (int blk = 0; blk < nb && ok; ++blk, ++gb) {
        if (!(ok = mbar_wait_warp(&bars[KV_FULL0 + (gb & 1)], (gb >> 1) & 1, wc, kErrSparseBase + 5))) break;
        if (gb >= 1 && !(ok = mbar_wait_warp(&bars[S_FREE], (gb - 1) & 1, wc, kErrSparseBase + 6))) break;
        tc_fence_after();
        // ---- S^T and dP^T over the 64-column chunks
        for (int i = 0; i < NCHUNK && ok; ++i, ++rc) {
          const int rs = rc % RING, c = i >> 1;
          if (!(ok = mbar_wait_warp(&bars[RING_FULL0 + rs], (rc / RING) & 1, wc, kErrSparseBase + 7))) break;
          tc_fence_after();
          const uint32_t acc = (i & 1) == 0 ? tmem + T_S : tmem + T_DP;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss_w(acc, dKV_k + sdesc_step(c * SLAB + kk * 32), dRing_k + sdesc_step(rs * CHUNK + kk * 32), IDESC_SP,
                     c > 0 || kk > 0);
          mma_commit_w(&bars[RING_EMPTY0 + rs]);
        }
        if (!ok) break;
        mma_commit_w(&bars[S_FULL]);
        mma_commit_w(&bars[DP_FULL]);
        // ---- dQ^T += K_sel^T dS^T (tile m: head dims 128m .. 128m+127; the last
        // tile reads slab 8 for both halves and only its first 64 rows are used)
        if (!(ok = mbar_wait_warp(&bars[DS_READY], gb & 1, wc, kErrSparseBase + 8))) break;
        if (blk == 0 && uc >= 1 && !(ok = mbar_wait_warp(&bars[DQ_FREE], (uc - 1) & 1, wc, kErrSparseBase + 9))) break;
        tc_fence_after();
#pragma unroll 1
        for (int m = 0; m < 5; ++m) {
          const uint64_t a = sdesc_sw128(sbase + OFF_KV + (2 * m < NSK ? 2 * m : NSK - 1) * SLAB, m < 4 ? SLAB : 0, 1024);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_ss_w(tmem + T_DQ + 64 * m, a + sdesc_step(kk * 2048), dDS_mn + sdesc_step(kk * 2048), IDESC_DQ,
                     blk > 0 || kk > 0);
        }
        mma_commit_w(&bars[KV_FREE]);
        mma_commit_w(&bars[DS_SFREE]);
        // ---- dKV chunks: dS^T Q_c + P^T dO_c (A from TMEM, B = chunk as [d x heads])
        for (int i = 0; i < NCHUNK && ok; ++i, ++rc) {
          const int rs = rc % RING, c = i >> 1;
          const bool isq = (i & 1) == 0;
          if (isq && cc >= 1 && !(ok = mbar_wait_warp(&bars[DKV_EMPTY], (cc - 1) & 1, wc, kErrSparseBase + 10))) break;
          if (!(ok = mbar_wait_warp(&bars[RING_FULL0 + rs], (rc / RING) & 1, wc, kErrSparseBase + 11))) break;
          tc_fence_after();
          // hi and lo halves of dS^T (with Q) or P^T (with dO)
          const uint32_t a = isq ? tmem + T_DP : tmem + T_S;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = dRing_mn + sdesc_step(rs * CHUNK + kk * 2048);
            mma_ts_w(tmem + T_DKV, a + 32 + kk * 8, bd, IDESC_KV, !isq || kk > 0);
            mma_ts_w(tmem + T_DKV, a + kk * 8, bd, IDESC_KV, 1);
          }
          mma_commit_w(&bars[RING_EMPTY0 + rs]);
          if (!isq || c == NSK - 1) {  // chunk c complete (the last chunk has no dV part)
            mma_commit_w(&bars[DKV_FULL]);
            ++cc;
          }
        }
        if (!ok) break;
        mma_commit_w(&bars[S_FREE]);
      }
      if (!ok) break;
      mma_commit_w(&bars[DQ_DONE]);
    }
    mma_commit_w(&bars[DRAIN]);
    if (lane == 0) mbar_drain(&bars[DRAIN], 0);
    __syncwarp();
  } else if (warp >= 4) {
    // ============================================================ softmax / dS, dQ output
    const int quad = warp & 3, row = quad * 32 + lane;  // slot (TMEM lane)
    const uint32_t lo = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t gb = 0;
    bool ok = true;
    for (int uc = 0; ok; ++uc) {
      const int slot = uc & 1;
      if (!(ok = mbar_wait_warp(&bars[UNIT_FULL0 + slot], (uc >> 1) & 1, wc, kErrSparseBase + 12))) break;
      const UnitInfo* ui = &units[slot];
      const int valid = ui->valid, nb = ui->nb, b = ui->b, t = ui->t, g = ui->g;
      if (!valid) break;
      for (int blk = 0; blk < nb && ok; ++blk, ++gb) {
        if (!(ok = mbar_wait_warp(&bars[KV_FULL0 + (gb & 1)], (gb >> 1) & 1, wc, kErrSparseBase + 13))) break;
        const bool sv = idx_buf[(gb & 1) * BK + row] >= 0;
        if (!(ok = mbar_wait_warp(&bars[S_FULL], gb & 1, wc, kErrSparseBase + 14))) break;
        tc_fence_after();
        // P is kept as a bf16/fp16 pair hi + lo (lo = the rounding residual of
        // hi): with 64 query heads adding into every latent row, the rounding
        // of a single 16-bit P or dS would accumulate past the tolerance of dKV.
        uint32_t ph[32], pl[32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t r[32];
          tmem_ld32(tmem + lo + T_S + ch * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float p0 = sv ? ex2(fmaf(__uint_as_float(r[c]), p.scale_log2, -ui->lse2[ch * 32 + c])) : 0.f;
            const float p1 = sv ? ex2(fmaf(__uint_as_float(r[c + 1]), p.scale_log2, -ui->lse2[ch * 32 + c + 1])) : 0.f;
            const uint32_t h = pack2<BF16>(p0, p1);
            const float2 hf = unpack2<BF16>(h);
            ph[ch * 16 + c / 2] = h;
            pl[ch * 16 + c / 2] = pack2<BF16>(p0 - hf.x, p1 - hf.y);
          }
        }
        // P^T hi over the upper 32 columns of S^T, lo over the lower 32 (all read)
        tmem_st16(tmem + lo + T_S + 32, ph);
        tmem_st16(tmem + lo + T_S + 48, ph + 16);
        tmem_st16(tmem + lo + T_S + 0, pl);
        tmem_st16(tmem + lo + T_S + 16, pl + 16);
        if (!(ok = mbar_wait_warp(&bars[DP_FULL], gb & 1, wc, kErrSparseBase + 15))) break;
        tc_fence_after();
        uint32_t dw[32], dl[32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t r[32];
          tmem_ld32(tmem + lo + T_DP + ch * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 a = unpack2<BF16>(ph[ch * 16 + c / 2]), e = unpack2<BF16>(pl[ch * 16 + c / 2]);
            const float d0 = (a.x + e.x) * (__uint_as_float(r[c]) - ui->delta[ch * 32 + c]) * p.sm_scale;
            const float d1 = (a.y + e.y) * (__uint_as_float(r[c + 1]) - ui->delta[ch * 32 + c + 1]) * p.sm_scale;
            const uint32_t h = pack2<BF16>(d0, d1);
            const float2 hf = unpack2<BF16>(h);
            dw[ch * 16 + c / 2] = h;
            dl[ch * 16 + c / 2] = pack2<BF16>(d0 - hf.x, d1 - hf.y);
          }
        }
        // dS^T hi over the upper 32 columns of dP^T, lo over the lower 32 (all read)
        tmem_st16(tmem + lo + T_DP + 32, dw);
        tmem_st16(tmem + lo + T_DP + 48, dw + 16);
        tmem_st16(tmem + lo + T_DP + 0, dl);
        tmem_st16(tmem + lo + T_DP + 16, dl + 16);
        // dS^T row into shared memory (B operand of dQ^T) once the previous dQ^T read it
        if (gb >= 1 && !(ok = mbar_wait_warp(&bars[DS_SFREE], (gb - 1) & 1, wc, kErrSparseBase + 16))) break;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          *reinterpret_cast<uint4*>(sm + OFF_DS + sw128_offset(row, c8)) =
              make_uint4(dw[c8 * 4], dw[c8 * 4 + 1], dw[c8 * 4 + 2], dw[c8 * 4 + 3]);
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[DS_READY]);
      }
      if (!ok) break;
      // ---- dQ of the token: tile m, lane = head dim 128m + row, columns = heads
      if (!(ok = mbar_wait_warp(&bars[DQ_DONE], uc & 1, wc, kErrSparseBase + 17))) break;
      tc_fence_after();
      uint8_t* dq = p.dq + 2 * (b * p.sdq_b + static_cast<int64_t>(t) * p.sdq_s + (static_cast<int64_t>(g) * p.gh) * p.sdq_h);
#pragma unroll 1
      for (int m = 0; m < 5; ++m) {
        uint32_t r[64];
        if (nb > 0) {
          tmem_ld32(tmem + lo + T_DQ + 64 * m, r);
          tmem_ld32(tmem + lo + T_DQ + 64 * m + 32, r + 32);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) r[c] = 0u;
        }
        const int d = 128 * m + row;
        if (d < DQK) {
#pragma unroll
          for (int h = 0; h < SH; ++h) {
            if (h < p.gh) {  // the group's own heads (padding heads are not written)
              const uint32_t w = pack2<BF16>(__uint_as_float(r[h]), 0.f);
              *reinterpret_cast<uint16_t*>(dq + 2 * (h * p.sdq_h + d)) = static_cast<uint16_t>(w & 0xffffu);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[DQ_FREE]);
        mbar_arrive(&bars[UNIT_EMPTY0 + slot]);  // the unit's LSE/delta are no longer read
      }
    }
  } else {
    // ============================================================ dKV epilogue (lane = slot)
    const int row = warp * 32 + lane;
    const uint32_t lo = static_cast<uint32_t>(warp * 32) << 16;
    uint8_t* stg = sm + OFF_STG + row * STG_STRIDE;
    bool issued = false;
    uint32_t gb = 0, cc = 0;
    bool ok = true;
    for (int uc = 0; ok; ++uc) {
      const int slot = uc & 1;
      if (!(ok = mbar_wait_warp(&bars[UNIT_FULL0 + slot], (uc >> 1) & 1, wc, kErrSparseBase + 18))) break;
      const int valid = units[slot].valid, nb = units[slot].nb, b = units[slot].b, g = units[slot].g;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[UNIT_EMPTY0 + slot]);
      if (!valid) break;
      for (int blk = 0; blk < nb && ok; ++blk, ++gb) {
        if (!(ok = mbar_wait_warp(&bars[KV_FULL0 + (gb & 1)], (gb >> 1) & 1, wc, kErrSparseBase + 19))) break;
        const int j = idx_buf[(gb & 1) * BK + row];
        float* dst = j >= 0 ? p.dkv_acc + ((static_cast<int64_t>(b) * p.SKV + j) * p.HKV + g) * DQK : nullptr;
        for (int c = 0; c < NSK && ok; ++c, ++cc) {
          if (!(ok = mbar_wait_warp(&bars[DKV_FULL], cc & 1, wc, kErrSparseBase + 20))) break;
          tc_fence_after();
          uint32_t r[64];
          tmem_ld32(tmem + lo + T_DKV, r);
          tmem_ld32(tmem + lo + T_DKV + 32, r + 32);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[DKV_EMPTY]);
          if (dst != nullptr) {
            if (issued) bulk_wait_read_all();  // this thread's previous reduce has read its staging row
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4)
              *reinterpret_cast<uint4*>(stg + q4 * 16) = make_uint4(r[4 * q4], r[4 * q4 + 1], r[4 * q4 + 2], r[4 * q4 + 3]);
            fence_proxy_async_smem();
            bulk_reduce_add_f32(dst + c * 64, stg, 256);
            bulk_commit_group();
            issued = true;
          }
        }
      }
    }
    if (issued) bulk_wait_all();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool BF16>
cudaError_t launch_t(const SparseParams& p, const SparseMaps& m, int grid, cudaStream_t st) {
  auto kern = sparse_bwd_kernel<BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  e = launch_after_previous(kern, grid, THREADS, SMEM, st, m, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse(const SparseParams& p, const SparseMaps& m, bool bf16, int grid, cudaStream_t st) {
  return bf16 ? launch_t<true>(p, m, grid, st) : launch_t<false>(p, m, grid, st);
}

}  // namespace ab
