// Launch 2 of the dense backward: the persistent, key-block-owned main kernel.
//
// Structure (the "Tiled" placement of the TileOPs MHA backward page, section
// "TileFoundry Description", re-designed for the 5th-generation tensor core):
// a tile is a block of BM = 128 key rows of one KV head (and batch row or
// packed sequence).  K and V stay in shared memory, dK and dV accumulate in
// tensor memory (TMEM) over every query block of every query head of the
// group (KV-head ownership, flash-linear-attention issue "Evaluate
// KV-head-owned GQA dKV backward", "Bounded scope" items 1-2), and are written
// once, in the input dtype, when the tile ends.  Per step (one query block of
// BN rows of one query head):
//
//   S^T  = K Q^T                   tensor core, M = 128 keys, N = BN, K = D
//   P^T  = exp2(S^T*scale*log2e - LSE2)  masked, rounded to 16 bits, back into TMEM
//   dP^T = V dO^T                  tensor core
//   dV  += P^T dO                  A operand = P^T from TMEM
//   dS^T = P^T o (dP^T - delta)    unscaled (the page folds the scale into dK and dQ)
//   dK  += dS^T Q                  A operand = dS^T from TMEM
//   dQ   = dS K                    from shared memory; added into the f32 workspace
//                                  accumulator with one bulk tensor reduce-add
//
// This kernel serves head dim 64 with BN = 128 queries per step and computes
// dQ = dS K (M = 128 queries); head dim 128 runs the kernel of
// dense128_bwd.cu.
//
// Pipelining: S^T is double-buffered in TMEM and the S^T of step i+1 is
// issued before dV/dK/dQ of step i, so the softmax of one step overlaps the
// tensor work of the previous one.  P^T and dS^T of a step are written over
// that step's S^T columns, and its dQ goes there once dK has read them.
// Q/dO come through a 4-stage TMA ring; the f32 dQ partial of a step is
// staged in the step's own stage and the stage goes back to the producer once
// the dQ reduces have read it.  No stage or accumulator is reused before an
// mbarrier shows that its last reader is done (the two pipelining faults the
// TileOPs page reports fixing in its older kernel, "Summary").
//
// Persistent CTAs (one per SM) draw tiles, longest first, from a counter in
// the workspace that the preprocess zeroes; each CTA's producer publishes the
// tile to the other roles through a two-slot ring in shared memory.
//
// Warp roles (16 warps): 0-3 dQ epilogue (TMEM -> shared-memory staging),
// 4-11 two warpgroups of softmax/dS work (each owns half of the BN query
// columns of all 128 key rows) that also land dK/dV, 12 TMA producer,
// 13 MMA issuer (one elected thread), 14 dQ reduce issuer, 15 idle (it
// completes the fourth warpgroup of the register split).  Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

// the register split below needs the bounded waits' slow paths inlined
#define AB_INLINE_WAITS 1
#include "common.cuh"
#include "cvt.cuh"
#include "dense_common.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace ab {

namespace {

// Q/dO stages and dS tiles in shared memory.  The f32 dQ partial of a step is
// staged in the step's own Q/dO stage once its MMAs are done, so a stage stays
// busy until the step's reduce-adds have read it; four stages cover that
// lifetime, paid for with a single dS tile.
constexpr int kStages64 = 4;
constexpr int kDsTiles64 = 1;

template <int D>
struct Cfg {
  static_assert(D == 64, "head dim 128 runs the kernel of dense128_bwd.cu");
  static constexpr int BM = kDenseBM;
  static constexpr int BN = kDenseBN;
  static constexpr int STAGES = kStages64;
  static constexpr int PREFETCH = 8;  // L2 prefetch distance of Q/dO/LSE/delta, in steps
  static constexpr int NSLAB = D / 64;  // 64-column (128-byte) slabs per row
  static constexpr int KV_SLAB = BM * 128;
  static constexpr int KV_TILE = KV_SLAB * NSLAB;
  static constexpr int Q_SLAB = BN * 128;
  static constexpr int Q_TILE = Q_SLAB * NSLAB;
  static constexpr int DS_BYTES = BM * BN * 2;
  static constexpr int NDS = kDsTiles64;  // dS tiles in shared memory
  static_assert(BN * D * 4 == 2 * Q_TILE, "the f32 dQ staging of a step fills a Q/dO stage");
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;
  static constexpr int OFF_DO = OFF_Q + STAGES * Q_TILE;
  static constexpr int OFF_DS = OFF_DO + STAGES * Q_TILE;
  static constexpr int OFF_LSE = OFF_DS + NDS * DS_BYTES;
  static constexpr int OFF_DELTA = OFF_LSE + STAGES * BN * 4;
  static constexpr int OFF_RING = OFF_DELTA + STAGES * BN * 4;
  static constexpr int OFF_BAR = OFF_RING + 2 * static_cast<int>(sizeof(TileInfo));
  static constexpr int NBAR = 40;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(OFF_Q % 1024 == 0 && OFF_DO % 1024 == 0 && OFF_DS % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  // tensor memory columns (512 allocated)
  static constexpr int T_SB = 0;           // two S^T buffers [128 x BN] f32; P^T / dS^T (16-bit pairs) overwrite them
  static constexpr int T_DP = 2 * BN;      // dP^T f32 [128 x BN]
  static constexpr int T_DV = 3 * BN;      // dV f32 [128 x D]
  static constexpr int T_DK = 3 * BN + D;  // dK f32 [128 x D]
  // dQ [128 q x 64 d] goes into the first 64 columns of its step's S^T buffer
  // once dK has read that buffer
  static_assert(3 * BN + 2 * D <= 512, "TMEM budget");
  // 16 warps in four warpgroups, launched at 128 registers each (the whole
  // register file) and re-split at entry: the softmax warpgroups take 168 so
  // that a warp keeps both halves of its S^T / dP^T columns in flight next to
  // P, the epilogue keeps 104 and the producer/MMA warpgroup 72.  Each
  // sub-partition holds one warp of every warpgroup: 32 x (104 + 168 + 168 +
  // 72) = 16384 registers, its whole file.
  static constexpr int THREADS = 16 * 32;
  static constexpr uint32_t REG_EPI = 104, REG_SOFT = 168, REG_CTL = 72;
  static_assert(REG_EPI + 2 * REG_SOFT + REG_CTL == 4 * 128, "register split must equal the launch's registers");
};

enum Bar : int {
  FULL0 = 0,                        // kStages64 stages: Q/dO loaded (+ the producer's LSE/delta arrival)
  EMPTY0 = FULL0 + kStages64,       // ... every reader of the stage is done
  KV_FULL = EMPTY0 + kStages64,
  KV_FREE,
  TILE_FULL0,                       // 2 slots
  TILE_EMPTY0 = TILE_FULL0 + 2,     // 2 slots
  S_FULL0 = TILE_EMPTY0 + 2,        // 2 buffers
  P_READY0 = S_FULL0 + 2,           // 2 buffers
  DP_FULL = P_READY0 + 2,
  DS_READY,
  DS_SFREE0,                        // kDsTiles64 dS tiles: the dQ MMAs have read them
  DQ_FULL = DS_SFREE0 + kDsTiles64,
  DQ_EMPTY,
  STG_FULL0,                        // kStages64 stages: 4 epilogue warps wrote the step's staging rows
  DKV_FULL = STG_FULL0 + kStages64,
  DKV_FREE,
  DRAIN,
  DP_FREE,
  TAIL,             // the producer's own: loads of tiles that overhang the last packed sequence
  NUM_BARS
};
static_assert(NUM_BARS <= Cfg<64>::NBAR, "barrier storage");

template <int D, bool BF16, bool SPLIT>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1) dense_bwd_kernel(const __grid_constant__ DenseMaps maps, const DenseParams p) {
  using C = Cfg<D>;
  constexpr int BM = C::BM, BN = C::BN, ST = C::STAGES, kPrefetch = C::PREFETCH;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  TileInfo* ring = reinterpret_cast<TileInfo*>(sm + C::OFF_RING);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 8);
  // per step parity: gs + 1 when a softmax warp of step gs saw a P above kSplitP (bf16)
  volatile uint32_t* split_flag = reinterpret_cast<volatile uint32_t*>(sm + C::OFF_MISC + 16);
  float* s_lse = reinterpret_cast<float*>(sm + C::OFF_LSE);
  float* s_delta = reinterpret_cast<float*>(sm + C::OFF_DELTA);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if ((smem_u32(sm) & 1023u) != 0) {  // the swizzled tiles need an aligned base
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kErrAlign);
    return;
  }
  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    split_flag[0] = split_flag[1] = 0u;
    for (int i = 0; i < ST; ++i) {
      mbar_init(&bars[FULL0 + i], 2);  // producer: expect_tx arrival + arrival after LSE/delta stores
      mbar_init(&bars[EMPTY0 + i], 1);
    }
    mbar_init(&bars[KV_FULL], 1);
    mbar_init(&bars[KV_FREE], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[TILE_FULL0 + i], 1);
      mbar_init(&bars[TILE_EMPTY0 + i], 14);  // MMA warp, 8 softmax warps, 4 epilogue warps, the reduce warp
      mbar_init(&bars[S_FULL0 + i], 1);
    }
    mbar_init(&bars[P_READY0], 8);
    mbar_init(&bars[P_READY0 + 1], 8);
    mbar_init(&bars[DP_FULL], 1);
    mbar_init(&bars[DS_READY], 8);
    for (int i = 0; i < C::NDS; ++i) mbar_init(&bars[DS_SFREE0 + i], 1);
    mbar_init(&bars[DQ_FULL], 1);
    mbar_init(&bars[DQ_EMPTY], 4);
    for (int i = 0; i < ST; ++i) mbar_init(&bars[STG_FULL0 + i], 4);
    mbar_init(&bars[DKV_FULL], 1);
    mbar_init(&bars[DKV_FREE], 8);
    mbar_init(&bars[DRAIN], 1);
    mbar_init(&bars[DP_FREE], 8);
    mbar_init(&bars[TAIL], 1);
    fence_mbar_init();
  }
  if (warp == 13) {
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

  // Every role ends here: all warps meet, then the MMA warp releases TMEM.
  // Each role runs it at its own end (and returns), so that no code is shared
  // between roles that run under different register budgets.
  auto finish = [&]() {
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(C::THREADS) : "memory");
    if (warp == 13) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
  };
  // each role sets its register budget at its own entry
  if (warp >= 14) {
    setmaxnreg_dec<C::REG_CTL>();
    if (warp == 14) {
      // ========================================================== dQ reduce issuer
      // Adds each step's staged f32 dQ partial into the workspace accumulator
      // (two bulk tensor reduce-adds) and hands the stage back to the producer
      // as soon as they have read it.  It waits for the reduce engine in a warp
      // of its own, so the epilogue warps stage the next step meanwhile.
      uint32_t gs = 0;
      bool ok = true, issued = false;
      for (int tc = 0; ok; ++tc) {
        const int slot = tc & 1;
        if (!(ok = mbar_wait_warp(&bars[TILE_FULL0 + slot], (tc >> 1) & 1, wc, kErrWaitTile))) break;
        const TileInfo ti = ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[TILE_EMPTY0 + slot]);
        if (!ti.valid) break;
        const int n = p.G * ti.nq;
        for (int j = 0; j < n; ++j, ++gs) {
          const int st = gs % ST;
          if (!(ok = mbar_wait_warp(&bars[STG_FULL0 + st], (gs / ST) & 1, wc, kErrWaitStage))) break;
          if (lane == 0) {
            const int h = ti.g * p.G + j / ti.nq, c2 = ti.seq_start + (ti.qlo + j % ti.nq) * BN;
            tma_reduce_add_4d(&maps.dq, sm + C::OFF_Q + st * C::Q_TILE, 0, h, c2, ti.b);
            tma_reduce_add_4d(&maps.dq, sm + C::OFF_DO + st * C::Q_TILE, D / 2, h, c2, ti.b);
            bulk_commit_group();
            bulk_wait_read_all();  // the stage may be reloaded once the reduces have read it
            mbar_arrive(&bars[EMPTY0 + st]);
          }
          issued = true;
          __syncwarp();
        }
      }
      if (lane == 0 && issued) bulk_wait_all();
    }
    // warp 15: spare, completes the fourth warpgroup of the register split
    finish();
    return;
  } else if (warp == 12) {
    setmaxnreg_dec<C::REG_CTL>();
    // ============================================================ producer
    int pend_full[ST];
#pragma unroll
    for (int i = 0; i < ST; ++i) pend_full[i] = -1;
    int kv_pend = -1;
    // Rows from tail0 to S belong to no packed sequence and may hold anything:
    // a tile or query block that reaches them is loaded onto the producer's
    // own barrier, those rows are zeroed, and only then is it published, so no
    // MMA multiplies them (a zero P or dS times a NaN is NaN).
    const int tail0 = p.cu_seqlens ? clamp_pos(p.cu_seqlens[p.num_seqs], p.S) : p.S;
    uint32_t tail_ph = 0;
    int tail_pend = -1;
    // loads two one-slab tiles onto TAIL, waits, zeroes rows [r0, r1) of both
    // and publishes them with a plain arrival on ``full``
    auto load_zeroed = [&](uint8_t* dst0, const CUtensorMap* m0, uint8_t* dst1, const CUtensorMap* m1, int h_,
                           int pos, int b_, int r0, int r1, uint64_t* full) -> bool {
      static_assert(C::NSLAB == 1 && C::KV_TILE == C::Q_TILE, "one-slab tiles of one size");
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[TAIL], 2 * C::Q_TILE);
        tma_load_4d(dst0, m0, &bars[TAIL], 0, h_, pos, b_);
        tma_load_4d(dst1, m1, &bars[TAIL], 0, h_, pos, b_);
      }
      tail_pend = tail_ph & 1;
      if (!mbar_wait_warp(&bars[TAIL], tail_ph & 1, wc, kErrWaitTail)) return false;
      tail_pend = -1;
      ++tail_ph;
      zero_tile_rows(dst0, 1, C::Q_SLAB, r0, r1, lane);
      zero_tile_rows(dst1, 1, C::Q_SLAB, r0, r1, lane);
      if (lane == 0) mbar_arrive(full);
      return true;
    };
    uint32_t gs = 0;
    bool ok = true;
    for (int tc = 0; ok; ++tc) {
      const int slot = tc & 1;
      if (tc >= 2 && !(ok = mbar_wait_warp(&bars[TILE_EMPTY0 + slot], ((tc >> 1) - 1) & 1, wc, kErrWaitTile))) break;
      int t = 0;
      if (lane == 0) t = atomicAdd(p.tile_counter, 1);
      t = __shfl_sync(0xffffffffu, t, 0);
      const TileInfo ti = decode_tile(t, p);
      if (lane == 0) {
        ring[slot] = ti;
        mbar_arrive(&bars[TILE_FULL0 + slot]);
      }
      if (!ti.valid) break;
      if (tc >= 1 && !(ok = mbar_wait_warp(&bars[KV_FREE], (tc - 1) & 1, wc, kErrWaitKVFree))) break;
      int kr0, kr1;
      tail_rows(ti.seq_start + ti.k0, BM, p.cu_seqlens ? tail0 : p.Sk, p.Sk, &kr0, &kr1);
      if (kr0 < kr1) {
        if (!(ok = load_zeroed(sm + C::OFF_K, &maps.k, sm + C::OFF_V, &maps.v, ti.g, ti.seq_start + ti.k0, ti.b, kr0,
                               kr1, &bars[KV_FULL])))
          break;
      } else if (lane == 0) {
        mbar_arrive_expect_tx(&bars[KV_FULL], 2 * C::KV_TILE);
#pragma unroll
        for (int s = 0; s < C::NSLAB; ++s) {
          tma_load_4d(sm + C::OFF_K + s * C::KV_SLAB, &maps.k, &bars[KV_FULL], s * 64, ti.g, ti.seq_start + ti.k0,
                      ti.b);
          tma_load_4d(sm + C::OFF_V + s * C::KV_SLAB, &maps.v, &bars[KV_FULL], s * 64, ti.g, ti.seq_start + ti.k0,
                      ti.b);
        }
      }
      kv_pend = tc & 1;
      const int n = p.G * ti.nq;
      // LSE2 / delta of a step are loaded into registers one step ahead, so
      // their global-load latency hides behind the next stage wait.
      constexpr int PER_LANE = BN / 32;
      float nl[PER_LANE], nd[PER_LANE];
      auto load_rows = [&](int jj) {
        const int hh = ti.g * p.G + jj / ti.nq, qq = (ti.qlo + jj % ti.nq) * BN;
        const int64_t rb = (static_cast<int64_t>(ti.b) * p.HQ + hh) * p.S + ti.seq_start;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
          const int q = qq + lane + 32 * i;
          nl[i] = q < ti.qlen ? p.lse2[rb + q] : 0.f;
          nd[i] = q < ti.qlen ? p.delta[rb + q] : 0.f;
        }
      };
      if (n > 0) load_rows(0);
      for (int j = 0; j < n; ++j, ++gs) {
        const int st = gs % ST;
        const uint32_t r = gs / ST;
        if (gs >= static_cast<uint32_t>(ST) &&
            !(ok = mbar_wait_warp(&bars[EMPTY0 + st], (r - 1) & 1, wc, kErrWaitStageEmpty)))
          break;
        const int h = ti.g * p.G + j / ti.nq, q0 = (ti.qlo + j % ti.nq) * BN;
        int qr0, qr1;
        tail_rows(ti.seq_start + q0, BN, tail0, p.S, &qr0, &qr1);
        if (qr0 < qr1) {
          if (!(ok = load_zeroed(sm + C::OFF_Q + st * C::Q_TILE, &maps.q, sm + C::OFF_DO + st * C::Q_TILE, &maps.dO, h,
                                 ti.seq_start + q0, ti.b, qr0, qr1, &bars[FULL0 + st])))
            break;
        } else if (lane == 0) {
          mbar_arrive_expect_tx(&bars[FULL0 + st], 2 * C::Q_TILE);
#pragma unroll
          for (int s = 0; s < C::NSLAB; ++s) {
            tma_load_4d(sm + C::OFF_Q + st * C::Q_TILE + s * C::Q_SLAB, &maps.q, &bars[FULL0 + st], s * 64, h,
                        ti.seq_start + q0, ti.b);
            tma_load_4d(sm + C::OFF_DO + st * C::Q_TILE + s * C::Q_SLAB, &maps.dO, &bars[FULL0 + st], s * 64, h,
                        ti.seq_start + q0, ti.b);
          }
        }
        // warm L2 with the operands of a step kPrefetch steps ahead
        if (j + kPrefetch < n) {
          const int hf = ti.g * p.G + (j + kPrefetch) / ti.nq, qf = (ti.qlo + (j + kPrefetch) % ti.nq) * BN;
          if (lane == 0) {
#pragma unroll
            for (int s = 0; s < C::NSLAB; ++s) {
              tma_prefetch_l2_4d(&maps.q, s * 64, hf, ti.seq_start + qf, ti.b);
              tma_prefetch_l2_4d(&maps.dO, s * 64, hf, ti.seq_start + qf, ti.b);
            }
          }
          const int64_t rf = (static_cast<int64_t>(ti.b) * p.HQ + hf) * p.S + ti.seq_start + qf;
          if (lane < BN / 32 && qf + lane * 32 < ti.qlen) {
            prefetch_l2(p.lse2 + rf + lane * 32);
            prefetch_l2(p.delta + rf + lane * 32);
          }
        }
        // negated, so that the softmax forms S*scale - LSE2 and dP - delta
        // with paired f32 adds and fused multiply-adds
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
          s_lse[st * BN + lane + 32 * i] = -nl[i];
          s_delta[st * BN + lane + 32 * i] = -nd[i];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[FULL0 + st]);
        if (j + 1 < n) load_rows(j + 1);
        pend_full[st] = r & 1;
      }
    }
    // loads still in flight land before the CTA exits
    if (lane == 0) {
      if (tail_pend >= 0) mbar_drain(&bars[TAIL], tail_pend);
      if (kv_pend >= 0) mbar_drain(&bars[KV_FULL], kv_pend);
#pragma unroll
      for (int i = 0; i < ST; ++i)
        if (pend_full[i] >= 0) mbar_drain(&bars[FULL0 + i], pend_full[i]);
    }
    finish();
    return;
  } else if (warp == 13) {
    setmaxnreg_dec<C::REG_CTL>();
    // ============================================================ MMA issuer
    // The whole warp runs this role with warp-uniform values; one elected lane
    // issues each tcgen05 instruction.
    constexpr uint32_t IDESC_S = idesc_f16(BF16, 128, BN, false, false);
    constexpr uint32_t IDESC_KV = idesc_f16(BF16, 128, D, false, true);
    constexpr uint32_t IDESC_DQ = idesc_f16(BF16, 128, 64, true, true);
    const uint32_t sbase = smem_u32(sm);
    // descriptors at the start of each operand; K-major K-steps add 32 bytes
    // inside a 128-byte row (slab kk/4), MN-major K-steps add 16 rows = 2048 bytes
    const uint64_t dK_kmaj = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
    const uint64_t dV_kmaj = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
    const uint64_t dQ_kmaj = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
    const uint64_t dO_kmaj = sdesc_sw128(sbase + C::OFF_DO, 16, 1024);
    const uint64_t dQ_mn = sdesc_sw128(sbase + C::OFF_Q, C::Q_SLAB, 1024);
    const uint64_t dO_mn = sdesc_sw128(sbase + C::OFF_DO, C::Q_SLAB, 1024);
    const uint64_t dK_mn = sdesc_sw128(sbase + C::OFF_K, C::KV_SLAB, 1024);
    const uint64_t dDS_mn = sdesc_sw128(sbase + C::OFF_DS, BM * 128, 1024);
    int64_t last_dq = -1;  // global step of the most recently issued dQ
    uint32_t gs = 0;
    bool ok = true;
    for (int tc = 0; ok; ++tc) {
      const int slot = tc & 1;
      if (!(ok = mbar_wait_warp(&bars[TILE_FULL0 + slot], (tc >> 1) & 1, wc, kErrWaitTile))) break;
      const TileInfo ti = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[TILE_EMPTY0 + slot]);
      if (!ti.valid) break;
      const int n = p.G * ti.nq;
      if (!(ok = mbar_wait_warp(&bars[KV_FULL], tc & 1, wc, kErrWaitKV))) break;
      tc_fence_after();
      for (int j = -1; j < n; ++j) {
        // j = -1: the tile's first S^T and dP^T; then per step j: the next
        // step's S^T, this step's dV, the next step's dP^T, this step's dK, dQ.
        const uint32_t cur = gs;               // step j (when j >= 0)
        const uint32_t nxt = j < 0 ? gs : gs + 1;  // step whose S^T / dP^T is issued now
        if (j + 1 < n) {
          // ---- S^T of step nxt into buffer nxt & 1
          const int st = nxt % ST;
          if (!(ok = mbar_wait_warp(&bars[FULL0 + st], (nxt / ST) & 1, wc, kErrWaitStageFull))) break;
          // the buffer's last reader is the epilogue's readout of the dQ that
          // overwrote it (readouts are in step order, so the latest issued dQ is
          // waited for)
          if (nxt >= 2 &&
              !(ok = mbar_wait_warp(&bars[DQ_EMPTY], static_cast<uint32_t>(last_dq) & 1, wc, kErrWaitDQEmpty)))
            break;
          tc_fence_after();
          const uint32_t dS_acc = tmem + C::T_SB + (nxt & 1) * BN;
          const uint64_t qo = sdesc_step(st * C::Q_TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ko = sdesc_step((kk / 4) * C::KV_SLAB + (kk % 4) * 32);
            const uint64_t qk = sdesc_step((kk / 4) * C::Q_SLAB + (kk % 4) * 32);
            mma_ss_w(dS_acc, dK_kmaj + ko, dQ_kmaj + qo + qk, IDESC_S, kk > 0);
          }
          mma_commit_w(&bars[S_FULL0 + (nxt & 1)]);
          if (j < 0) {
            // ---- dP^T of the tile's first step
            if (nxt >= 1) {
              if (!(ok = mbar_wait_warp(&bars[DP_FREE], (nxt - 1) & 1, wc, kErrWaitDP))) break;
              tc_fence_after();
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t ko = sdesc_step((kk / 4) * C::KV_SLAB + (kk % 4) * 32);
              const uint64_t qk = sdesc_step((kk / 4) * C::Q_SLAB + (kk % 4) * 32);
              mma_ss_w(tmem + C::T_DP, dV_kmaj + ko, dO_kmaj + qo + qk, IDESC_S, kk > 0);
            }
            mma_commit_w(&bars[DP_FULL]);
          }
        }
        if (j < 0) continue;
        const int st = cur % ST;
        const uint64_t qo = sdesc_step(st * C::Q_TILE);
        const uint32_t sb = tmem + C::T_SB + (cur & 1) * BN;
        // ---- dV += P^T dO (B = dO as [N = D] x [K = queries], MN-major)
        if (!(ok = mbar_wait_warp(&bars[P_READY0 + (cur & 1)], (cur >> 1) & 1, wc, kErrWaitP))) break;
        if (j == 0 && tc >= 1 && !(ok = mbar_wait_warp(&bars[DKV_FREE], (tc - 1) & 1, wc, kErrWaitDKVFree))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts_w(tmem + C::T_DV, sb + pair_col(kk * 16, BN / 2), dO_mn + qo + sdesc_step(kk * 2048), IDESC_KV,
                   j > 0 || kk > 0);
        // ---- dP^T of the next step, as soon as this step's dP^T has been loaded
        // (bf16: after this step's residual MMAs, which read residual pairs that
        // the softmax warps wrote into the dP^T columns)
        auto issue_next_dp = [&]() -> bool {
          if (j + 1 >= n) return true;
          if (!mbar_wait_warp(&bars[DP_FREE], cur & 1, wc, kErrWaitDP)) return false;
          tc_fence_after();
          const uint64_t qn = sdesc_step(((cur + 1) % ST) * C::Q_TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ko = sdesc_step((kk / 4) * C::KV_SLAB + (kk % 4) * 32);
            const uint64_t qk = sdesc_step((kk / 4) * C::Q_SLAB + (kk % 4) * 32);
            mma_ss_w(tmem + C::T_DP, dV_kmaj + ko, dO_kmaj + qn + qk, IDESC_S, kk > 0);
          }
          mma_commit_w(&bars[DP_FULL]);
          return true;
        };
        // bf16 steps with the residuals (flagged by the softmax warps before P_READY)
        bool split = false;
        if constexpr (SPLIT) split = split_flag[cur & 1] == cur + 1;
        if (!split && !(ok = issue_next_dp())) break;
        // ---- dK += dS^T Q (B = Q as [N = D] x [K = queries], MN-major)
        if (!(ok = mbar_wait_warp(&bars[DS_READY], cur & 1, wc, kErrWaitDS))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts_w(tmem + C::T_DK, sb + pair_col(kk * 16, BN / 2) + BN / 4, dQ_mn + qo + sdesc_step(kk * 2048),
                   IDESC_KV, j > 0 || kk > 0);
        if constexpr (SPLIT) {
          // a step with a large P adds the rounding residuals of P and dS (queries
          // 16kk .. 16kk + 15: P_lo pairs at dP^T column 16kk, dS_lo at 16kk + 8)
          if (split) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts_w(tmem + C::T_DV, tmem + C::T_DP + kk * 16, dO_mn + qo + sdesc_step(kk * 2048), IDESC_KV, 1u);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts_w(tmem + C::T_DK, tmem + C::T_DP + kk * 16 + 8, dQ_mn + qo + sdesc_step(kk * 2048), IDESC_KV,
                       1u);
            if (!(ok = issue_next_dp())) break;
          }
        }
        // dQ overwrites this step's S^T buffer, which dV and dK read: MMAs issued
        // by one thread run in issue order, so no wait is needed in between
        const uint32_t dq_cols = sb;
        // one dQ in flight: the epilogue has read the previous one
        if (cur >= 1 && !(ok = mbar_wait_warp(&bars[DQ_EMPTY], (cur - 1) & 1, wc, kErrWaitDQEmpty))) break;
        tc_fence_after();
        // ---- dQ over the 128 key rows (K-step = 16 key rows = 2048 bytes)
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)  // A = dS MN-major (two 64-query blocks), B = K tile MN-major
          mma_ss_w(dq_cols, dDS_mn + sdesc_step((cur % C::NDS) * C::DS_BYTES + kk * 2048),
                   dK_mn + sdesc_step(kk * 2048), IDESC_DQ, kk > 0);
        mma_commit_w(&bars[DQ_FULL]);
        mma_commit_w(&bars[DS_SFREE0 + cur % C::NDS]);
        last_dq = cur;
        ++gs;
      }
      if (!ok) break;
      if (n == 0 && tc >= 1 && !(ok = mbar_wait_warp(&bars[DKV_FREE], (tc - 1) & 1, wc, kErrWaitDKVFree))) break;
      mma_commit_w(&bars[KV_FREE]);   // last readers of K and V issued
      mma_commit_w(&bars[DKV_FULL]);  // dK, dV final once every MMA of the tile completed
    }
    // every MMA issued by this warp completes before TMEM is released
    mma_commit_w(&bars[DRAIN]);
    if (lane == 0) mbar_drain(&bars[DRAIN], 0);
    __syncwarp();
    finish();
    return;
  } else if (warp >= 4) {
    setmaxnreg_inc<C::REG_SOFT>();
    // ============================================================ softmax / dS, dK / dV landing
    const int wg = (warp - 4) >> 2, quad = warp & 3;
    const int row = quad * 32 + lane;  // key row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    constexpr int HALF = BN / 2;  // query columns of this warpgroup
    constexpr int NCH = HALF / 32;
    const bool cm = p.causal || p.window > 0;
    const int W = p.window;
    float pv[HALF];
    uint32_t gs = 0;
    bool ok = true;
    for (int tc = 0; ok; ++tc) {
      const int slot = tc & 1;
      if (!(ok = mbar_wait_warp(&bars[TILE_FULL0 + slot], (tc >> 1) & 1, wc, kErrWaitTile))) break;
      const TileInfo ti = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[TILE_EMPTY0 + slot]);
      if (!ti.valid) break;
      const int n = p.G * ti.nq;
      const int kpos = ti.k0 + row;
      const bool kvalid = kpos < ti.len;
      for (int j = 0; j < n; ++j, ++gs) {
        const int st = gs % ST;
        const uint32_t sb = tmem + lane_off + C::T_SB + (gs & 1u) * BN;
        const int q0 = (ti.qlo + j % ti.nq) * BN;
        const int qc0 = q0 + wg * HALF;  // first (sequence-local) query of my columns
        // fully visible block: every key and query in range and inside the mask
        const bool full_vis = ti.k0 + BM <= ti.len && q0 + BN <= ti.qlen &&
                              (!cm || q0 + ti.off >= ti.k0 + BM - 1) && (W <= 0 || q0 + BN - 1 + ti.off < ti.k0 + W);
        const float4* lse4 = reinterpret_cast<const float4*>(s_lse + st * BN + wg * HALF);
        const float4* dlt4 = reinterpret_cast<const float4*>(s_delta + st * BN + wg * HALF);
        if (!(ok = mbar_wait_warp(&bars[FULL0 + st], (gs / ST) & 1, wc, kErrWaitStageFull))) break;
        if (!(ok = mbar_wait_warp(&bars[S_FULL0 + (gs & 1)], (gs >> 1) & 1, wc, kErrWaitS))) break;
        tc_fence_after();
        // both 32-column halves of this warpgroup's S^T in flight at once, then P
        uint32_t sr[HALF];
        tmem_ld32(sb + wg * HALF, sr);
        tmem_ld32(sb + wg * HALF + 32, sr + 32);
        tmem_ld_wait();
        // S^T * scale - LSE2 two columns per instruction (f32x2 FMA)
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        auto x_pair = [&](int cc, float lo, float hi) {
          return __ffma2_rn(make_float2(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])), sc2,
                            make_float2(lo, hi));
        };
        // In a block that is not fully visible, my columns cc in [c_lo, c_hi) are:
        // a real query (cc < qlen - qc0), at or after my key (kpos <= qc0 + cc +
        // off) and within the window (qc0 + cc + off < kpos + W); one range per
        // step, two compares a column.  A warp whose rows all see every one of
        // their columns takes the unmasked path, one whose rows see none of them
        // writes zeros (the diagonal and window-edge blocks hold both kinds).
        int c_lo = 0, c_hi = HALF, mode = 0;  // mode 0: all visible, 1: none, 2: per column
        if (!full_vis) {
          const int64_t d0 = static_cast<int64_t>(kpos) - qc0 - ti.off;
          const int64_t hi = W > 0 ? d0 + W : HALF;
          c_lo = cm ? static_cast<int>(d0 < 0 ? 0 : (d0 > HALF ? HALF : d0)) : 0;
          c_hi = imin(ti.qlen - qc0, static_cast<int>(hi < 0 ? 0 : (hi > HALF ? HALF : hi)));
          mode = __all_sync(0xffffffffu, kvalid && c_lo == 0 && c_hi == HALF)   ? 0
                 : __all_sync(0xffffffffu, !kvalid || c_hi <= c_lo) ? 1
                                                                    : 2;
        }
        if (mode == 0) {
#pragma unroll
          for (int c4 = 0; c4 < HALF / 4; ++c4) {
            const float4 t = lse4[c4];  // -LSE2
            const float2 x0 = x_pair(4 * c4, t.x, t.y), x1 = x_pair(4 * c4 + 2, t.z, t.w);
            pv[4 * c4] = ex2(x0.x);
            pv[4 * c4 + 1] = ex2(x0.y);
            pv[4 * c4 + 2] = ex2(x1.x);
            pv[4 * c4 + 3] = ex2(x1.y);
          }
        } else if (mode == 1) {
#pragma unroll
          for (int cc = 0; cc < HALF; ++cc) pv[cc] = 0.f;
        } else {
#pragma unroll
          for (int c4 = 0; c4 < HALF / 4; ++c4) {
            const float4 t = lse4[c4];  // -LSE2
            const float2 x0 = x_pair(4 * c4, t.x, t.y), x1 = x_pair(4 * c4 + 2, t.z, t.w);
            const float x4[4] = {x0.x, x0.y, x1.x, x1.y};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int cc = 4 * c4 + e;
              const bool vis = kvalid && cc >= c_lo && cc < c_hi;
              pv[cc] = vis ? ex2(x4[e]) : 0.f;
            }
          }
        }
        // P^T pairs go into the first half of this warpgroup's own S^T columns,
        // which only this warp's lanes read (and its loads have completed); bf16
        // keeps the largest rounded P of each half-word lane (P >= 0, so the
        // 16-bit patterns order as unsigned integers)
        uint32_t pmax2 = 0u;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          uint32_t w[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            w[c] = pack2<BF16>(pv[ch * 32 + 2 * c], pv[ch * 32 + 2 * c + 1]);
            if constexpr (SPLIT) pmax2 = __vmaxu2(pmax2, w[c]);
          }
          tmem_st16(sb + wg * HALF + ch * 16, w);
        }
        // bf16: does this warp's part of the step need the rounding residuals?
        bool big = false;
        if constexpr (SPLIT) {
          big = __any_sync(0xffffffffu, __vcmpgtu2(pmax2, kSplitPBf16x2) != 0u);
          if (big && lane == 0) split_flag[gs & 1] = gs + 1;
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[P_READY0 + (gs & 1)]);

        if (!(ok = mbar_wait_warp(&bars[DP_FULL], gs & 1, wc, kErrWaitDP))) break;
        // the dS tile this step writes was last read by the dQ of step gs - NDS
        if (gs >= static_cast<uint32_t>(C::NDS) &&
            !(ok = mbar_wait_warp(&bars[DS_SFREE0 + gs % C::NDS], ((gs - C::NDS) / C::NDS) & 1, wc, kErrWaitDSFree)))
          break;
        tc_fence_after();
        // the step takes the rounding residuals if any softmax warp saw a large P
        // (the MMA warp reads the flag after every warp has signalled); a warp
        // with a large P writes its residual pairs, the others write zeros there
        const bool split = big;
        uint8_t* const dsbase = sm + C::OFF_DS + (gs % C::NDS) * C::DS_BYTES + wg * (BM * 128);
        // dS for 16 queries at a time: dS^T pairs into the second half of this
        // warpgroup's S^T columns, dS as the MN-major A operand of dQ (64-query
        // block wg, row = key, two 16-byte chunks).  The next step's dP^T may
        // overwrite this warpgroup's dP^T columns once they are loaded (DP_FREE)
        // - except in a step with the residuals, which writes those of P^T and
        // dS^T of each 16 queries into 16 of these columns (P_lo pairs, then dS_lo
        // pairs; the next dP^T is issued after the residual MMAs) and loads the
        // second half only when it reaches it, keeping the residuals within the
        // warp's registers.
        auto ds_stage = [&](auto res_c) {
          constexpr bool RES = decltype(res_c)::value;
          uint32_t dr[HALF];
          // dS = P (dP - delta), two columns per instruction (f32x2 add and multiply)
          auto ds_pair = [&](int cc, float lo, float hi) {
            return __fmul2_rn(make_float2(pv[cc], pv[cc + 1]),
                              __fadd2_rn(make_float2(__uint_as_float(dr[cc]), __uint_as_float(dr[cc + 1])),
                                         make_float2(lo, hi)));
          };
          tmem_ld32(tmem + lane_off + C::T_DP + wg * HALF, dr);
          if constexpr (!RES) tmem_ld32(tmem + lane_off + C::T_DP + wg * HALF + 32, dr + 32);
          tmem_ld_wait();
          auto dp_loaded = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[DP_FREE]);
          };
          if constexpr (!RES) {
            if constexpr (SPLIT) {
              // a warp without large P: zero residual pairs, in case another warp
              // of the step flagged it and the residual MMAs read these columns
              // (complete before the next step's dP^T may overwrite them)
              uint32_t z[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
              for (int c16 = 0; c16 < HALF / 16; ++c16)
                tmem_st16(tmem + lane_off + C::T_DP + wg * HALF + 16 * c16, z);
              tmem_st_wait();
            }
            dp_loaded();
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              uint32_t dsw[16];
#pragma unroll
              for (int c = 0; c < 32; c += 4) {
                const int cc = ch * 32 + c;
                const float4 dl = dlt4[cc / 4];  // -delta of columns cc .. cc + 3
                const float2 a0 = ds_pair(cc, dl.x, dl.y), a1 = ds_pair(cc + 2, dl.z, dl.w);
                dsw[c / 2] = pack2<BF16>(a0.x, a0.y);
                dsw[c / 2 + 1] = pack2<BF16>(a1.x, a1.y);
              }
              tmem_st16(sb + wg * HALF + HALF / 2 + ch * 16, dsw);
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4)
                *reinterpret_cast<uint4*>(dsbase + sw128_offset(row, ch * 4 + c4)) =
                    make_uint4(dsw[c4 * 4], dsw[c4 * 4 + 1], dsw[c4 * 4 + 2], dsw[c4 * 4 + 3]);
            }
          } else {
#pragma unroll
            for (int g = 0; g < HALF / 16; ++g) {
              if (g == HALF / 32) {
                tmem_ld32(tmem + lane_off + C::T_DP + wg * HALF + 32, dr + 32);
                tmem_ld_wait();
                dp_loaded();
              }
              uint32_t dsw[8], plo[8], dsl[8];
#pragma unroll
              for (int c = 0; c < 16; c += 4) {
                const int cc = g * 16 + c;
                const float4 dl = dlt4[cc / 4];  // -delta of columns cc .. cc + 3
                const float2 a0 = ds_pair(cc, dl.x, dl.y), a1 = ds_pair(cc + 2, dl.z, dl.w);
                const float d0 = a0.x, d1 = a0.y, d2 = a1.x, d3 = a1.y;
                dsw[c / 2] = pack2<BF16>(d0, d1);
                dsw[c / 2 + 1] = pack2<BF16>(d2, d3);
                dsl[c / 2] = lo_pair<BF16>(d0, d1, dsw[c / 2]);
                dsl[c / 2 + 1] = lo_pair<BF16>(d2, d3, dsw[c / 2 + 1]);
                plo[c / 2] = lo_pair<BF16>(pv[cc], pv[cc + 1], pack2<BF16>(pv[cc], pv[cc + 1]));
                plo[c / 2 + 1] = lo_pair<BF16>(pv[cc + 2], pv[cc + 3], pack2<BF16>(pv[cc + 2], pv[cc + 3]));
              }
              tmem_st8(sb + wg * HALF + HALF / 2 + g * 8, dsw);
#pragma unroll
              for (int c4 = 0; c4 < 2; ++c4)
                *reinterpret_cast<uint4*>(dsbase + sw128_offset(row, g * 2 + c4)) =
                    make_uint4(dsw[c4 * 4], dsw[c4 * 4 + 1], dsw[c4 * 4 + 2], dsw[c4 * 4 + 3]);
              const uint32_t lo_col = tmem + lane_off + C::T_DP + wg * HALF + g * 16;
              tmem_st8(lo_col, plo);
              tmem_st8(lo_col + 8, dsl);
            }
          }
        };
        if constexpr (SPLIT) {
          if (split)
            ds_stage(std::true_type{});
          else
            ds_stage(std::false_type{});
        } else {
          ds_stage(std::false_type{});
        }
        if (!ok) break;
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[DS_READY]);
      }
      if (!ok) break;
      // ---- dK / dV of the tile: warpgroup 0 lands dV, warpgroup 1 lands dK (times sm_scale)
      if (!(ok = mbar_wait_warp(&bars[DKV_FULL], tc & 1, wc, kErrWaitDKV))) break;
      tc_fence_after();
      const bool isK = wg == 1;
      const uint32_t col0 = isK ? C::T_DK : C::T_DV;
      const float mul = isK ? p.sm_scale : 1.f;
      const int64_t pos = ti.seq_start + kpos;
      uint8_t* out = isK ? p.dk + 2 * (ti.b * p.sdk_b + pos * p.sdk_s + ti.g * p.sdk_h)
                         : p.dv + 2 * (ti.b * p.sdv_b + pos * p.sdv_s + ti.g * p.sdv_h);
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_off + col0 + ch * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = 0u;
        }
        if (ch == D / 32 - 1) {  // the accumulators may be overwritten by the next tile from here on
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[DKV_FREE]);
        }
        if (kvalid) {
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint4 v;
            v.x = pack2<BF16>(__uint_as_float(r[c8 * 8 + 0]) * mul, __uint_as_float(r[c8 * 8 + 1]) * mul);
            v.y = pack2<BF16>(__uint_as_float(r[c8 * 8 + 2]) * mul, __uint_as_float(r[c8 * 8 + 3]) * mul);
            v.z = pack2<BF16>(__uint_as_float(r[c8 * 8 + 4]) * mul, __uint_as_float(r[c8 * 8 + 5]) * mul);
            v.w = pack2<BF16>(__uint_as_float(r[c8 * 8 + 6]) * mul, __uint_as_float(r[c8 * 8 + 7]) * mul);
            *reinterpret_cast<uint4*>(out + 2 * (ch * 32 + c8 * 8)) = v;
          }
        }
      }
    }
    finish();
    return;
  } else {
    setmaxnreg_dec<C::REG_EPI>();
    // ============================================================ dQ epilogue
    // The f32 dQ partial of a step is staged in the step's own Q/dO stage (every
    // MMA reading the stage was issued before dQ, so it has completed once
    // DQ_FULL has), one 128-byte-swizzled [128 q x 32 d] slab in the Q part and
    // one in the dO part; the reduce warp adds it into the accumulator.
    const int quad = warp;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t gs = 0;
    bool ok = true;
    for (int tc = 0; ok; ++tc) {
      const int slot = tc & 1;
      if (!(ok = mbar_wait_warp(&bars[TILE_FULL0 + slot], (tc >> 1) & 1, wc, kErrWaitTile))) break;
      const TileInfo ti = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[TILE_EMPTY0 + slot]);
      if (!ti.valid) break;
      const int n = p.G * ti.nq;
      for (int j = 0; j < n; ++j, ++gs) {
        const int st = gs % ST;
        if (!(ok = mbar_wait_warp(&bars[DQ_FULL], gs & 1, wc, kErrWaitDQFull))) break;
        tc_fence_after();
        uint32_t r[64];
        const uint32_t dq_cols = tmem + lane_off + C::T_SB + (gs & 1u) * BN;
        tmem_ld32(dq_cols, r);
        tmem_ld32(dq_cols + 32, r + 32);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[DQ_EMPTY]);
        uint8_t* const half0 = sm + C::OFF_Q + st * C::Q_TILE;
        uint8_t* const half1 = sm + C::OFF_DO + st * C::Q_TILE;
        // lane = query; half c / 8 is a 128-byte-swizzled slab [128 q][32 d]
        const int q = quad * 32 + lane;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          uint8_t* slab = c < 8 ? half0 : half1;
          *reinterpret_cast<float4*>(slab + sw128_offset(q, c & 7)) =
              make_float4(__uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1]), __uint_as_float(r[4 * c + 2]),
                          __uint_as_float(r[4 * c + 3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[STG_FULL0 + st]);
      }
    }
    finish();
  }
}

template <int D, bool BF16, bool SPLIT>
cudaError_t launch_dense_t(const DenseParams& p, const DenseMaps& m, int grid, cudaStream_t st) {
  auto kern = dense_bwd_kernel<D, BF16, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  e = launch_after_previous(kern, grid, Cfg<D>::THREADS, Cfg<D>::SMEM, st, m, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// One CTA waits on a barrier that nothing signals: the bounded wait must give
// up, record kErrSelftest and let the kernel return.
__global__ void selftest_timeout_kernel(int* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{&abort_flag, err, timeout_ns};
  mbar_wait_warp(&bar, 0, wc, kErrSelftest);
}

}  // namespace

cudaError_t launch_dense(const DenseParams& p, const DenseMaps& m, bool bf16, int grid, cudaStream_t st) {
  if (p.bn != kDenseBN) return cudaErrorInvalidValue;
  if (p.D == 128) return launch_dense128(p, m, bf16, grid, st);
  if (p.D != 64) return cudaErrorInvalidValue;
  if (!bf16) return launch_dense_t<64, false, false>(p, m, grid, st);
  return p.G > kSplitMinGroup ? launch_dense_t<64, true, true>(p, m, grid, st)
                              : launch_dense_t<64, true, false>(p, m, grid, st);
}

cudaError_t launch_selftest_timeout(int* err, uint64_t timeout_ns, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace ab
