// Launch 2 of the dense backward for head dim 128: the persistent,
// key-block-owned main kernel with 128-query steps.
//
// Same placement as the head-dim-64 kernel (the "Tiled" program of the TileOPs
// MHA backward page, section "TileFoundry Description"; KV-head ownership as in
// the flash-linear-attention issue "Evaluate KV-head-owned GQA dKV backward",
// "Bounded scope" items 1-2): a tile is 128 key rows of one KV head, K and V
// stay in shared memory, dK and dV accumulate in tensor memory over every
// query block of every query head of the group and are written once.  Per
// step (BN = 128 queries of one query head):
//
//   S^T  = K Q^T        M = 128 keys, N = 128 queries, K = 128   (shared x shared)
//   dP^T = V dO^T       same shape
//   P^T  = exp2(S^T*scale*log2e - LSE2), masked; dS^T = P^T o (dP^T - delta)
//   dV  += P^T dO       A = P^T from TMEM (16-bit pairs), B = dO   N = 128
//   dK  += dS^T Q       A = dS^T from TMEM                        N = 128
//   dQ   = dS K         A = dS from shared memory, M = 128 queries, N = 128
//
// Every MMA has N = 128.  An M = 128, N = 64 MMA with both operands in shared
// memory reads 6 KB per 32 cycles of tensor work, more than the 128 bytes
// per clock shared memory delivers; at N = 128 the operand bytes per flop
// drop by a quarter and the tensor pipe can run at full rate.
//
// Tensor memory (512 columns): S^T [128 x 128] f32 at 0, overwritten by P^T
// and dS^T as 16-bit pairs, each softmax warpgroup in its own 64 columns (P^T
// in the first 32, dS^T in the last 32); dP^T at 128, which
// the f32 dQ of the step overwrites once the softmax warps have read dP; dV at
// 256, dK at 384.
//
// Shared memory: K, V (32 KB each), two Q/dO stages (64 KB each), the dS tile
// (32 KB).  The f32 dQ of a step (64 KB) is staged in that step's own Q/dO
// stage once dV and dK have read it, added into the workspace accumulator with
// four TMA bulk tensor reduce-adds.  The Q half and the dO half of the stage
// go back to the producer separately, each as soon as the reduces of its own
// two staging slabs have read it.
//
// Warp roles (16 warps): 0-3 dQ epilogue (lane = query; at the end of a tile
// they also land dK/dV, lane = key row, while the softmax warps start the next
// one), 4-11 two warpgroups of softmax/dS work (each owns 64 of the 128 query
// columns of all 128 key rows), 12 TMA producer, 13 MMA issuer, 14 dQ reduce
// issuer, 15 idle (it completes the fourth warpgroup of the register split).
// A stage, a TMEM region or the dS tile is reused only after an mbarrier shows
// that its last reader is done.  Every wait is bounded.
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

constexpr int D = 128;
constexpr int BM = kDenseBM;
constexpr int BN = 128;
constexpr int ST = 2;                 // Q/dO stages
// L2 prefetch distance of Q/dO/LSE/delta, in steps.  Long tiles (unmasked GQA)
// gain from it; the short tiles of causal launches (at most 16 steps at S =
// 2048) run faster without prefetches, which this distance leaves out.
constexpr int PREFETCH = 32;
constexpr int SLAB = 128 * 128;       // [128 rows x 64 cols] 16-bit, 128-byte swizzled
constexpr int KV_TILE = 2 * SLAB;     // 128 rows x 128 cols
constexpr int Q_TILE = 2 * SLAB;
constexpr int STAGE = 2 * Q_TILE;     // Q then dO
constexpr int DS_BLOCK = BM * 128;    // dS as [128 keys x 64 queries] 16-bit
constexpr int STG_SLAB = BN * 128;    // f32 dQ staging: [128 queries x 32 d] per slab, 4 slabs

constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + KV_TILE;
constexpr int OFF_STAGE = OFF_V + KV_TILE;
constexpr int OFF_DS = OFF_STAGE + ST * STAGE;
constexpr int OFF_LSE = OFF_DS + 2 * DS_BLOCK;
constexpr int OFF_DELTA = OFF_LSE + ST * BN * 4;
constexpr int OFF_RING = OFF_DELTA + ST * BN * 4;
constexpr int OFF_BAR = OFF_RING + 2 * static_cast<int>(sizeof(TileInfo));
constexpr int NBAR = 32;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM = OFF_MISC + 64;
static_assert(SMEM <= 227 * 1024, "shared memory budget");
static_assert(4 * STG_SLAB == STAGE, "the f32 dQ staging fills one stage");
static_assert(OFF_STAGE % 1024 == 0 && OFF_DS % 1024 == 0, "swizzled tiles need 1024-byte alignment");

constexpr int T_S = 0;     // S^T f32; P^T pairs at 0-63, dS^T pairs at 64-127
constexpr int T_DP = 128;  // dP^T f32, then the step's dQ f32 [128 queries x 128 d]
constexpr int T_DV = 256;
constexpr int T_DK = 384;
// 16 warps in four warpgroups, launched at 128 registers each (the whole
// register file: 16 warps x 32 lanes x 128 = 65536) and re-split at entry:
// the softmax warpgroups take 168 so that a warp keeps both halves of its
// S^T / dP^T columns in flight next to P, the epilogue keeps 104 and the
// producer/MMA warpgroup 72.  Each sub-partition holds one warp of every
// warpgroup: 32 x (104 + 168 + 168 + 72) = 16384 registers, its whole file.
constexpr int THREADS = 16 * 32;
constexpr uint32_t REG_EPI = 104, REG_SOFT = 168, REG_CTL = 72;
static_assert(REG_EPI + 2 * REG_SOFT + REG_CTL == 4 * 128, "register split must equal the launch's registers");

// Each stage has two halves with their own barriers: Q (with the step's LSE2
// and delta) and dO.  The f32 dQ staging of a step covers both halves, and
// each half goes back to the producer as soon as the reduces of its own
// staging slabs have read it, so the next Q (needed first, by S^T and the
// softmax) does not wait for the reduces of the dO half.
enum Bar : int {
  FULL0 = 0,         // ST stages: Q half loaded (expect_tx arrival) + the producer's LSE/delta arrival
  FULLD0 = 2,        // ST stages: dO half loaded
  EMPTY0 = 4,        // ST stages: the dQ reduces have read the staging slabs in the Q half
  EMPTYD0 = 6,       // ST stages: ... in the dO half
  KV_FULL = 8,
  KV_FREE,
  TILE_FULL0 = 10,   // 2 slots
  TILE_EMPTY0 = 12,  // 2 slots
  S_FULL = 14,
  S_FREE,           // dV and dK of the step completed: S^T columns reusable
  P_READY,          // 8 softmax warps stored P^T
  DP_FULL,
  DS_READY,         // 8 softmax warps stored dS^T (TMEM) and dS (shared)
  DS_SFREE,         // dQ MMAs read the shared dS tile
  DQ_FULL,
  DQ_EMPTY,         // 4 epilogue warps loaded dQ: the dP^T columns are free
  STG_FULL0,        // ST stages: 4 epilogue warps wrote their staging rows of the Q half
  STG_FULLB0 = STG_FULL0 + ST,  // ST stages: ... of the dO half
  DKV_FULL = STG_FULLB0 + ST,
  DKV_FREE,
  DRAIN,
  TAIL,             // the producer's own: loads of tiles that overhang the last packed sequence
  NUM_BARS
};
static_assert(NUM_BARS <= NBAR, "barrier storage");

template <bool BF16, bool SPLIT>
__global__ void __launch_bounds__(THREADS, 1) dense128_bwd_kernel(const __grid_constant__ DenseMaps maps,
                                                                  const DenseParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  TileInfo* ring = reinterpret_cast<TileInfo*>(sm + OFF_RING);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC + 8);
  // per step parity: gs + 1 when a softmax warp of step gs saw a P above kSplitP (bf16)
  volatile uint32_t* split_flag = reinterpret_cast<volatile uint32_t*>(sm + OFF_MISC + 16);
  float* s_lse = reinterpret_cast<float*>(sm + OFF_LSE);
  float* s_delta = reinterpret_cast<float*>(sm + OFF_DELTA);
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
      mbar_init(&bars[FULL0 + i], 2);
      mbar_init(&bars[FULLD0 + i], 1);
      mbar_init(&bars[EMPTY0 + i], 1);
      mbar_init(&bars[EMPTYD0 + i], 1);
      mbar_init(&bars[STG_FULL0 + i], 4);
      mbar_init(&bars[STG_FULLB0 + i], 4);
    }
    mbar_init(&bars[KV_FULL], 1);
    mbar_init(&bars[KV_FREE], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[TILE_FULL0 + i], 1);
      mbar_init(&bars[TILE_EMPTY0 + i], 14);  // MMA warp, 8 softmax warps, 4 epilogue warps, the reduce warp
    }
    mbar_init(&bars[S_FULL], 1);
    mbar_init(&bars[S_FREE], 1);
    mbar_init(&bars[P_READY], 8);
    mbar_init(&bars[DP_FULL], 1);
    mbar_init(&bars[DS_READY], 8);
    mbar_init(&bars[DS_SFREE], 1);
    mbar_init(&bars[DQ_FULL], 1);
    mbar_init(&bars[DQ_EMPTY], 4);
    mbar_init(&bars[DKV_FULL], 1);
    mbar_init(&bars[DKV_FREE], 4);  // the 4 dQ epilogue warps land dK/dV
    mbar_init(&bars[DRAIN], 1);
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
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
    if (warp == 13) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
  };
  // each role sets its register budget at its own entry, so that the
  // compiler sees one budget along every path through a role
  if (warp >= 14) {
    setmaxnreg_dec<REG_CTL>();
    if (warp == 14) {
      // ========================================================== dQ reduce issuer
      // Adds each step's staged f32 dQ partial into the workspace accumulator,
      // the Q half's two slabs as soon as they are staged, then the dO half's,
      // and hands each half of the stage back to the producer as soon as its
      // reduces have read it.  It waits for the reduce engine in a warp of its
      // own, so the epilogue warps stage the next step meanwhile.
      uint32_t gs = 0;
      bool ok = true, issued = false;
      for (int tc = 0; ok; ++tc) {
        const int slot = tc & 1;
        if (!(ok = mbar_wait_warp(&bars[TILE_FULL0 + slot], (tc >> 1) & 1, wc, kErrWaitTile))) break;
        const TileInfo ti = ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[TILE_EMPTY0 + slot]);
        if (!ti.valid) break;
        const int n = ti.hn * ti.nq;
        for (int j = 0; j < n && ok; ++j, ++gs) {
          const int st = gs % ST;
          const int h = ti.g * p.G + ti.h0 + j / ti.nq, c2 = ti.seq_start + (ti.qlo + j % ti.nq) * BN;
          uint8_t* stg = sm + OFF_STAGE + st * STAGE;
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            if (!(ok = mbar_wait_warp(&bars[(hf == 0 ? STG_FULL0 : STG_FULLB0) + st], (gs / ST) & 1, wc,
                                      kErrWaitStage)))
              break;
            if (lane == 0) {
#pragma unroll
              for (int s2 = 0; s2 < 2; ++s2) {
                const int s4 = 2 * hf + s2;
                tma_reduce_add_4d(&maps.dq, stg + s4 * STG_SLAB, 32 * s4, h, c2, ti.b);
              }
              bulk_commit_group();
            }
          }
          if (!ok) break;
          if (lane == 0) {
            bulk_wait_read_1();  // the Q half may be reloaded once its reduces have read it
            mbar_arrive(&bars[EMPTY0 + st]);
            bulk_wait_read_all();
            mbar_arrive(&bars[EMPTYD0 + st]);
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
    setmaxnreg_dec<REG_CTL>();
    // ============================================================ producer
    int pend_full[ST], pend_d[ST];
#pragma unroll
    for (int i = 0; i < ST; ++i) pend_full[i] = pend_d[i] = -1;
    int kv_pend = -1;
    // Rows from tail0 to S belong to no packed sequence and may hold anything:
    // a tile or query block that reaches them is loaded onto the producer's
    // own barrier, those rows are zeroed, and only then is it published, so no
    // MMA multiplies them (a zero P or dS times a NaN is NaN).
    const int tail0 = p.cu_seqlens ? clamp_pos(p.cu_seqlens[p.num_seqs], p.S) : p.S;
    uint32_t tail_ph = 0;
    int tail_pend = -1;
    // loads the tile onto TAIL, waits, zeroes rows [r0, r1) of its slabs and
    // publishes it with a plain arrival on ``full``
    auto load_zeroed = [&](uint8_t* dst0, const CUtensorMap* m0, uint8_t* dst1, const CUtensorMap* m1, int h_,
                           int pos, int b_, int r0, int r1, uint64_t* full) -> bool {
      const uint32_t bytes = (dst1 ? 2 : 1) * Q_TILE;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[TAIL], bytes);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          tma_load_4d(dst0 + s * SLAB, m0, &bars[TAIL], s * 64, h_, pos, b_);
          if (dst1) tma_load_4d(dst1 + s * SLAB, m1, &bars[TAIL], s * 64, h_, pos, b_);
        }
      }
      tail_pend = tail_ph & 1;
      if (!mbar_wait_warp(&bars[TAIL], tail_ph & 1, wc, kErrWaitTail)) return false;
      tail_pend = -1;
      ++tail_ph;
      zero_tile_rows(dst0, 2, SLAB, r0, r1, lane);
      if (dst1) zero_tile_rows(dst1, 2, SLAB, r0, r1, lane);
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
        static_assert(KV_TILE == Q_TILE, "one tail load size");
        if (!(ok = load_zeroed(sm + OFF_K, &maps.k, sm + OFF_V, &maps.v, ti.g, ti.seq_start + ti.k0, ti.b, kr0, kr1,
                               &bars[KV_FULL])))
          break;
      } else if (lane == 0) {
        mbar_arrive_expect_tx(&bars[KV_FULL], 2 * KV_TILE);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          tma_load_4d(sm + OFF_K + s * SLAB, &maps.k, &bars[KV_FULL], s * 64, ti.g, ti.seq_start + ti.k0, ti.b);
          tma_load_4d(sm + OFF_V + s * SLAB, &maps.v, &bars[KV_FULL], s * 64, ti.g, ti.seq_start + ti.k0, ti.b);
        }
      }
      kv_pend = tc & 1;
      const int n = ti.hn * ti.nq;
      // LSE2 / delta of a step are loaded into registers one step ahead
      constexpr int PER_LANE = BN / 32;
      float nl[PER_LANE], nd[PER_LANE];
      auto load_rows = [&](int jj) {
        const int hh = ti.g * p.G + ti.h0 + jj / ti.nq, qq = (ti.qlo + jj % ti.nq) * BN;
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
        const int h = ti.g * p.G + ti.h0 + j / ti.nq, q0 = (ti.qlo + j % ti.nq) * BN;
        uint8_t* sq = sm + OFF_STAGE + st * STAGE;
        int qr0, qr1;
        tail_rows(ti.seq_start + q0, BN, tail0, p.S, &qr0, &qr1);
        if (qr0 < qr1) {
          if (!(ok = load_zeroed(sq, &maps.q, nullptr, nullptr, h, ti.seq_start + q0, ti.b, qr0, qr1,
                                 &bars[FULL0 + st])))
            break;
        } else if (lane == 0) {
          mbar_arrive_expect_tx(&bars[FULL0 + st], Q_TILE);
#pragma unroll
          for (int s = 0; s < 2; ++s)
            tma_load_4d(sq + s * SLAB, &maps.q, &bars[FULL0 + st], s * 64, h, ti.seq_start + q0, ti.b);
        }
        pend_full[st] = r & 1;
        // warm L2 with the operands of a step PREFETCH steps ahead
        if (j + PREFETCH < n) {
          const int hf = ti.g * p.G + ti.h0 + (j + PREFETCH) / ti.nq, qf = (ti.qlo + (j + PREFETCH) % ti.nq) * BN;
          if (lane == 0) {
#pragma unroll
            for (int s = 0; s < 2; ++s) {
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
        // LSE2/delta of the stage were last read by the softmax of step gs - ST,
        // which finished before that step's dQ (and so before EMPTY0)
        // negated, so that the softmax forms S*scale - LSE2 and dP - delta
        // with paired f32 adds and fused multiply-adds
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
          s_lse[st * BN + lane + 32 * i] = -nl[i];
          s_delta[st * BN + lane + 32 * i] = -nd[i];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[FULL0 + st]);
        if (gs >= static_cast<uint32_t>(ST) &&
            !(ok = mbar_wait_warp(&bars[EMPTYD0 + st], (r - 1) & 1, wc, kErrWaitStageEmpty)))
          break;
        if (qr0 < qr1) {
          if (!(ok = load_zeroed(sq + Q_TILE, &maps.dO, nullptr, nullptr, h, ti.seq_start + q0, ti.b, qr0, qr1,
                                 &bars[FULLD0 + st])))
            break;
        } else if (lane == 0) {
          mbar_arrive_expect_tx(&bars[FULLD0 + st], Q_TILE);
#pragma unroll
          for (int s = 0; s < 2; ++s)
            tma_load_4d(sq + Q_TILE + s * SLAB, &maps.dO, &bars[FULLD0 + st], s * 64, h, ti.seq_start + q0, ti.b);
        }
        pend_d[st] = r & 1;
        if (j + 1 < n) load_rows(j + 1);
      }
    }
    // loads still in flight land before the CTA exits
    if (lane == 0) {
      if (tail_pend >= 0) mbar_drain(&bars[TAIL], tail_pend);
      if (kv_pend >= 0) mbar_drain(&bars[KV_FULL], kv_pend);
#pragma unroll
      for (int i = 0; i < ST; ++i) {
        if (pend_full[i] >= 0) mbar_drain(&bars[FULL0 + i], pend_full[i]);
        if (pend_d[i] >= 0) mbar_drain(&bars[FULLD0 + i], pend_d[i]);
      }
    }
    finish();
    return;
  } else if (warp == 13) {
    setmaxnreg_dec<REG_CTL>();
    // ============================================================ MMA issuer (whole warp, one elected lane)
    constexpr uint32_t IDESC_S = idesc_f16(BF16, 128, BN, false, false);
    constexpr uint32_t IDESC_KV = idesc_f16(BF16, 128, D, false, true);
    constexpr uint32_t IDESC_DQ = idesc_f16(BF16, 128, D, true, true);
    const uint32_t sbase = smem_u32(sm);
    // K-major K-steps add 32 bytes inside a 128-byte row (slab kk/4); MN-major
    // K-steps add 16 rows = 2048 bytes
    const uint64_t dK_kmaj = sdesc_sw128(sbase + OFF_K, 16, 1024);
    const uint64_t dV_kmaj = sdesc_sw128(sbase + OFF_V, 16, 1024);
    const uint64_t dQ_kmaj = sdesc_sw128(sbase + OFF_STAGE, 16, 1024);
    const uint64_t dO_kmaj = sdesc_sw128(sbase + OFF_STAGE + Q_TILE, 16, 1024);
    const uint64_t dQ_mn = sdesc_sw128(sbase + OFF_STAGE, SLAB, 1024);
    const uint64_t dO_mn = sdesc_sw128(sbase + OFF_STAGE + Q_TILE, SLAB, 1024);
    const uint64_t dK_mn = sdesc_sw128(sbase + OFF_K, SLAB, 1024);
    const uint64_t dDS_mn = sdesc_sw128(sbase + OFF_DS, DS_BLOCK, 1024);
    uint32_t gs = 0;
    bool ok = true;
    for (int tc = 0; ok; ++tc) {
      const int slot = tc & 1;
      if (!(ok = mbar_wait_warp(&bars[TILE_FULL0 + slot], (tc >> 1) & 1, wc, kErrWaitTile))) break;
      const TileInfo ti = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[TILE_EMPTY0 + slot]);
      if (!ti.valid) break;
      const int n = ti.hn * ti.nq;
      if (!(ok = mbar_wait_warp(&bars[KV_FULL], tc & 1, wc, kErrWaitKV))) break;
      tc_fence_after();
      for (int j = 0; j < n; ++j, ++gs) {
        const int st = gs % ST;
        const uint64_t so = sdesc_step(st * STAGE);
        // ---- S^T: the stage is loaded and dV/dK of the previous step have read P^T/dS^T
        if (!(ok = mbar_wait_warp(&bars[FULL0 + st], (gs / ST) & 1, wc, kErrWaitStageFull))) break;
        if (gs >= 1 && !(ok = mbar_wait_warp(&bars[S_FREE], (gs - 1) & 1, wc, kErrWaitSFree))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ko = sdesc_step((kk / 4) * SLAB + (kk % 4) * 32);
          mma_ss_w(tmem + T_S, dK_kmaj + ko, dQ_kmaj + so + ko, IDESC_S, kk > 0);
        }
        mma_commit_w(&bars[S_FULL]);
        // ---- dP^T: the dO half is loaded and the epilogue has loaded the previous
        // step's dQ from these columns
        if (!(ok = mbar_wait_warp(&bars[FULLD0 + st], (gs / ST) & 1, wc, kErrWaitStageFull))) break;
        if (gs >= 1 && !(ok = mbar_wait_warp(&bars[DQ_EMPTY], (gs - 1) & 1, wc, kErrWaitDQEmpty))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ko = sdesc_step((kk / 4) * SLAB + (kk % 4) * 32);
          mma_ss_w(tmem + T_DP, dV_kmaj + ko, dO_kmaj + so + ko, IDESC_S, kk > 0);
        }
        mma_commit_w(&bars[DP_FULL]);
        // ---- dV += P^T dO (A = P^T pairs, 8 columns per 16 queries; B = dO MN-major)
        if (!(ok = mbar_wait_warp(&bars[P_READY], gs & 1, wc, kErrWaitP))) break;
        if (j == 0 && tc >= 1 && !(ok = mbar_wait_warp(&bars[DKV_FREE], (tc - 1) & 1, wc, kErrWaitDKVFree))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts_w(tmem + T_DV, tmem + T_S + pair_col(kk * 16, BN / 2), dO_mn + so + sdesc_step(kk * 2048), IDESC_KV, j > 0 || kk > 0);
        // ---- dK += dS^T Q
        if (!(ok = mbar_wait_warp(&bars[DS_READY], gs & 1, wc, kErrWaitDS))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts_w(tmem + T_DK, tmem + T_S + pair_col(kk * 16, BN / 2) + BN / 4, dQ_mn + so + sdesc_step(kk * 2048), IDESC_KV,
                   j > 0 || kk > 0);
        if constexpr (SPLIT) {
          // a step with a large P adds the rounding residuals of P and dS (their
          // pairs sit in the dP^T columns, which the dQ below overwrites after)
          // (queries 16kk .. 16kk + 15: P_lo pairs at dP^T column 16kk, dS_lo at 16kk + 8)
          if (split_flag[gs & 1] == gs + 1) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts_w(tmem + T_DV, tmem + T_DP + kk * 16, dO_mn + so + sdesc_step(kk * 2048), IDESC_KV, 1u);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts_w(tmem + T_DK, tmem + T_DP + kk * 16 + 8, dQ_mn + so + sdesc_step(kk * 2048), IDESC_KV, 1u);
          }
        }
        mma_commit_w(&bars[S_FREE]);
        // ---- dQ = dS K over the 128 key rows (A = dS MN-major in two 64-query blocks, B = K MN-major),
        // into the dP^T columns (the softmax warps read dP before publishing dS)
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          mma_ss_w(tmem + T_DP, dDS_mn + sdesc_step(kk * 2048), dK_mn + sdesc_step(kk * 2048), IDESC_DQ, kk > 0);
        mma_commit_w(&bars[DQ_FULL]);
        mma_commit_w(&bars[DS_SFREE]);
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
    setmaxnreg_inc<REG_SOFT>();
    // ============================================================ softmax / dS
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
      const int n = ti.hn * ti.nq;
      const int kpos = ti.k0 + row;
      const bool kvalid = kpos < ti.len;
      for (int j = 0; j < n; ++j, ++gs) {
        const int st = gs % ST;
        const uint32_t sb = tmem + lane_off + T_S;
        const int q0 = (ti.qlo + j % ti.nq) * BN;
        const int qc0 = q0 + wg * HALF;  // first (sequence-local) query of my columns
        // fully visible block: every key and query in range and inside the mask
        const bool full_vis = ti.k0 + BM <= ti.len && q0 + BN <= ti.qlen &&
                              (!cm || q0 + ti.off >= ti.k0 + BM - 1) && (W <= 0 || q0 + BN - 1 + ti.off < ti.k0 + W);
        const float4* lse4 = reinterpret_cast<const float4*>(s_lse + st * BN + wg * HALF);
        const float4* dlt4 = reinterpret_cast<const float4*>(s_delta + st * BN + wg * HALF);
        if (!(ok = mbar_wait_warp(&bars[FULL0 + st], (gs / ST) & 1, wc, kErrWaitStageFull))) break;
        if (!(ok = mbar_wait_warp(&bars[S_FULL], gs & 1, wc, kErrWaitS))) break;
        tc_fence_after();
        // both 32-column halves of this warpgroup's S^T in flight at once, then P
        // in place (LSE2 four columns at a time, so that only the S^T/P values stay live)
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
        if (full_vis) {
#pragma unroll
          for (int c4 = 0; c4 < HALF / 4; ++c4) {
            const float4 t = lse4[c4];  // -LSE2
            const float2 x0 = x_pair(4 * c4, t.x, t.y), x1 = x_pair(4 * c4 + 2, t.z, t.w);
            pv[4 * c4] = ex2(x0.x);
            pv[4 * c4 + 1] = ex2(x0.y);
            pv[4 * c4 + 2] = ex2(x1.x);
            pv[4 * c4 + 3] = ex2(x1.y);
          }
        } else {
          // my columns cc in [c_lo, c_hi) are visible: a real query (cc < qlen -
          // qc0), at or after my key (kpos <= qc0 + cc + off) and within the window
          // (qc0 + cc + off < kpos + W); one range per step, two compares a column
          const int64_t d0 = static_cast<int64_t>(kpos) - qc0 - ti.off;
          const int64_t hi = W > 0 ? d0 + W : HALF;
          const int c_lo = cm ? static_cast<int>(d0 < 0 ? 0 : (d0 > HALF ? HALF : d0)) : 0;
          const int c_hi = imin(ti.qlen - qc0, static_cast<int>(hi < 0 ? 0 : (hi > HALF ? HALF : hi)));
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
        if (lane == 0) mbar_arrive(&bars[P_READY]);

        if (!(ok = mbar_wait_warp(&bars[DP_FULL], gs & 1, wc, kErrWaitDP))) break;
        // the dS tile this step writes was last read by the previous step's dQ
        if (gs >= 1 && !(ok = mbar_wait_warp(&bars[DS_SFREE], (gs - 1) & 1, wc, kErrWaitDSFree))) break;
        tc_fence_after();
        uint8_t* dsb = sm + OFF_DS + wg * DS_BLOCK;
        // the step takes the rounding residuals if any softmax warp saw a large P
        // (the MMA warp reads the flag after every warp has signalled); a warp
        // with a large P writes its residual pairs, the others write zeros there
        const bool split = big;
        // dS for 16 queries at a time: dS^T pairs into the second half of this
        // warpgroup's S^T columns and dS as the MN-major A operand of dQ (64-query
        // block wg, row = key, two 16-byte chunks).  A step with the residuals
        // also writes those of P^T and dS^T of each 16 queries into 16 of this
        // warpgroup's dP^T columns once they are loaded (P_lo pairs, then dS_lo
        // pairs; read by the residual MMAs, then overwritten by this step's dQ),
        // and loads the second half of its dP^T columns only when it reaches
        // them, which keeps the residuals within the warp's registers.
        auto ds_stage = [&](auto res_c) {
          constexpr bool RES = decltype(res_c)::value;
          uint32_t dr[HALF];
          tmem_ld32(tmem + lane_off + T_DP + wg * HALF, dr);
          if constexpr (!RES) tmem_ld32(tmem + lane_off + T_DP + wg * HALF + 32, dr + 32);
          tmem_ld_wait();
          if constexpr (SPLIT && !RES) {
            // a warp without large P: zero residual pairs, in case another warp of
            // the step flagged it and the residual MMAs read these columns
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
            for (int c16 = 0; c16 < HALF / 16; ++c16) tmem_st16(tmem + lane_off + T_DP + wg * HALF + 16 * c16, z);
          }
#pragma unroll
          for (int g = 0; g < HALF / 16; ++g) {
            if constexpr (RES) {
              if (g == HALF / 32) {
                tmem_ld32(tmem + lane_off + T_DP + wg * HALF + 32, dr + 32);
                tmem_ld_wait();
              }
            }
            uint32_t dsw[8], plo[8], dsl[8];
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
              const int cc = g * 16 + c;
              const float4 dl = dlt4[cc / 4];  // -delta of columns cc .. cc + 3
              // dS = P (dP - delta), two columns per instruction (f32x2 add and multiply)
              const float2 a0 = __fmul2_rn(make_float2(pv[cc], pv[cc + 1]),
                                           __fadd2_rn(make_float2(__uint_as_float(dr[cc]), __uint_as_float(dr[cc + 1])),
                                                      make_float2(dl.x, dl.y)));
              const float2 a1 = __fmul2_rn(make_float2(pv[cc + 2], pv[cc + 3]),
                                           __fadd2_rn(make_float2(__uint_as_float(dr[cc + 2]), __uint_as_float(dr[cc + 3])),
                                                      make_float2(dl.z, dl.w)));
              const float d0 = a0.x, d1 = a0.y, d2 = a1.x, d3 = a1.y;
              dsw[c / 2] = pack2<BF16>(d0, d1);
              dsw[c / 2 + 1] = pack2<BF16>(d2, d3);
              if constexpr (RES) {
                dsl[c / 2] = lo_pair<BF16>(d0, d1, dsw[c / 2]);
                dsl[c / 2 + 1] = lo_pair<BF16>(d2, d3, dsw[c / 2 + 1]);
                plo[c / 2] = lo_pair<BF16>(pv[cc], pv[cc + 1], pack2<BF16>(pv[cc], pv[cc + 1]));
                plo[c / 2 + 1] = lo_pair<BF16>(pv[cc + 2], pv[cc + 3], pack2<BF16>(pv[cc + 2], pv[cc + 3]));
              }
            }
            tmem_st8(sb + wg * HALF + HALF / 2 + g * 8, dsw);
#pragma unroll
            for (int c4 = 0; c4 < 2; ++c4)
              *reinterpret_cast<uint4*>(dsb + sw128_offset(row, g * 2 + c4)) =
                  make_uint4(dsw[c4 * 4], dsw[c4 * 4 + 1], dsw[c4 * 4 + 2], dsw[c4 * 4 + 3]);
            if constexpr (RES) {
              const uint32_t lo_col = tmem + lane_off + T_DP + wg * HALF + g * 16;
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
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[DS_READY]);
      }
      if (!ok) break;
    }
    finish();
    return;
  } else {
    setmaxnreg_dec<REG_EPI>();
    // ============================================================ dQ epilogue (lane = query)
    const int quad = warp;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int q = quad * 32 + lane;  // query of the block = TMEM lane
    uint32_t gs = 0;
    bool ok = true;
    for (int tc = 0; ok; ++tc) {
      const int slot = tc & 1;
      if (!(ok = mbar_wait_warp(&bars[TILE_FULL0 + slot], (tc >> 1) & 1, wc, kErrWaitTile))) break;
      const TileInfo ti = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[TILE_EMPTY0 + slot]);
      if (!ti.valid) break;
      const int n = ti.hn * ti.nq;
      for (int j = 0; j < n; ++j, ++gs) {
        const int st = gs % ST;
        // dQ complete (so dV and dK, issued before it, have read this step's stage)
        if (!(ok = mbar_wait_warp(&bars[DQ_FULL], gs & 1, wc, kErrWaitDQFull))) break;
        tc_fence_after();
        // f32 staging in the stage: four 128-byte-swizzled slabs [128 queries x 32 d],
        // d 0-63 (slabs 0-1) in the Q half and d 64-127 (slabs 2-3) in the dO half.
        // Each half is written and handed to the reduce warp, so the Q half's
        // reduces start before the dO half is staged.
        uint8_t* stg = sm + OFF_STAGE + st * STAGE;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t r[64];
          tmem_ld32(tmem + lane_off + T_DP + 64 * hf, r);
          tmem_ld32(tmem + lane_off + T_DP + 64 * hf + 32, r + 32);
          tmem_ld_wait();
          if (hf == 1) {  // dQ fully loaded: the dP^T columns may be overwritten
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[DQ_EMPTY]);
          }
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int slab = 2 * hf + (c >> 3), chunk = c & 7;
            *reinterpret_cast<float4*>(stg + slab * STG_SLAB + sw128_offset(q, chunk)) =
                make_float4(__uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1]), __uint_as_float(r[4 * c + 2]),
                            __uint_as_float(r[4 * c + 3]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[(hf == 0 ? STG_FULL0 : STG_FULLB0) + st]);
        }
      }
      if (!ok) break;
      // ---- dK / dV of the tile, once every MMA of the tile has completed: lane =
      // key row, dV then dK (times sm_scale) in 32-column chunks.  The softmax
      // warps meanwhile start the next tile, whose first dV MMA waits for
      // DKV_FREE (all chunks loaded from TMEM).
      if (!(ok = mbar_wait_warp(&bars[DKV_FULL], tc & 1, wc, kErrWaitDKV))) break;
      tc_fence_after();
      const int kpos = ti.k0 + q;
      const bool kvalid = kpos < ti.len;
      const int64_t pos = ti.seq_start + kpos;
      uint8_t* const out_v = p.dv + 2 * (ti.b * p.sdv_b + pos * p.sdv_s + ti.g * p.sdv_h);
      uint8_t* const out_k = p.dk + 2 * (ti.b * p.sdk_b + pos * p.sdk_s + ti.g * p.sdk_h);
      constexpr int NCK = D / 32;  // chunks per accumulator
      if (ti.part >= 0) {
        // A last-round unit: add this unit's dV / dK (times sm_scale) into the
        // tile's f32 partials, column group c4 of row q at (c4 * 128 + q) * 4, so
        // that a warp adds 512 contiguous bytes per instruction; the warp whose
        // add completes its row quarter over all units casts the quarter.
        float* const acc = p.part_acc + static_cast<int64_t>(ti.part) * (2 * D * BM);
#pragma unroll 1
        for (int cc = 0; cc < 2 * NCK; ++cc) {
          const float mul = cc >= NCK ? p.sm_scale : 1.f;
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + (cc >= NCK ? T_DK + (cc - NCK) * 32 : T_DV + cc * 32), r);
          tmem_ld_wait();
          if (cc == 2 * NCK - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[DKV_FREE]);
          }
          if (n > 0) {
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
              red_add_f32x4(acc + (static_cast<int64_t>(cc * 8 + c4) * BM + q) * 4,
                            __uint_as_float(r[4 * c4]) * mul, __uint_as_float(r[4 * c4 + 1]) * mul,
                            __uint_as_float(r[4 * c4 + 2]) * mul, __uint_as_float(r[4 * c4 + 3]) * mul);
          }
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(p.part_count + ti.part * 4 + quad, 1) == p.G / p.tail_hpu - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
#pragma unroll 1
          for (int cc = 0; cc < 2 * NCK; ++cc) {
            uint8_t* const out = cc >= NCK ? out_k : out_v;
            const int ch = cc >= NCK ? cc - NCK : cc;
            if (kvalid) {
#pragma unroll
              for (int c8 = 0; c8 < 4; ++c8) {
                const float4 a = __ldcg(reinterpret_cast<const float4*>(acc) + (cc * 8 + 2 * c8) * BM + q);
                const float4 b = __ldcg(reinterpret_cast<const float4*>(acc) + (cc * 8 + 2 * c8 + 1) * BM + q);
                uint4 v;
                v.x = pack2<BF16>(a.x, a.y);
                v.y = pack2<BF16>(a.z, a.w);
                v.z = pack2<BF16>(b.x, b.y);
                v.w = pack2<BF16>(b.z, b.w);
                *reinterpret_cast<uint4*>(out + 2 * (ch * 32 + c8 * 8)) = v;
              }
            }
          }
        }
        continue;
      }
#pragma unroll 1
      for (int cc = 0; cc < 2 * NCK; ++cc) {
        const bool isK = cc >= NCK;
        const int ch = isK ? cc - NCK : cc;
        const float mul = isK ? p.sm_scale : 1.f;
        uint8_t* const out = isK ? out_k : out_v;
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_off + (isK ? T_DK : T_DV) + ch * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = 0u;
        }
        if (cc == 2 * NCK - 1) {  // the accumulators may be overwritten by the next tile from here on
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
  }
}

template <bool BF16, bool SPLIT>
cudaError_t launch_t(const DenseParams& p, const DenseMaps& m, int grid, cudaStream_t st) {
  auto kern = dense128_bwd_kernel<BF16, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  e = launch_after_previous(kern, grid, THREADS, SMEM, st, m, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense128(const DenseParams& p, const DenseMaps& m, bool bf16, int grid, cudaStream_t st) {
  if (!bf16) return launch_t<false, false>(p, m, grid, st);
  return p.G > kSplitMinGroup ? launch_t<true, true>(p, m, grid, st) : launch_t<true, false>(p, m, grid, st);
}

}  // namespace ab
