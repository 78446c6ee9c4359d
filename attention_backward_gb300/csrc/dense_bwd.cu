// Launch 2 of the dense backward: the key-block-owned main kernel.
//
// Structure (the "Tiled" placement of the TileOPs MHA backward page, section
// "TileFoundry Description", re-designed for the 5th-generation tensor core):
// one CTA owns a key tile of BM = 128 rows of one KV head (and batch row or
// packed sequence).  K and V stay in shared memory, dK and dV accumulate in
// tensor memory (TMEM) over every query block of every query head of the
// group (KV-head ownership, flash-linear-attention issue "Evaluate
// KV-head-owned GQA dKV backward", "Bounded scope" items 1-2), and are
// written once, in the input dtype, at the end.  Per query block of BN rows:
//
//   S^T  = K Q^T                   (tcgen05, M=128 keys, N=BN, K=D)
//   P^T  = exp2(S^T*scale*log2e - LSE2)  masked; rounded to 16 bit into TMEM
//   dP^T = V dO^T                  (tcgen05)
//   dV  += P^T dO                  (A = P^T from TMEM)
//   dS^T = P^T o (dP^T - delta)    unscaled (the page folds the scale into dK and dQ)
//   dK  += dS^T Q                  (A = dS^T from TMEM)
//   dQ  partial = dS K             (A/B from shared memory), added in f32 to the
//                                   workspace accumulator by atomics
//
// D = 128 uses BN = 64 and computes dQ^T = K^T dS^T (M = 128 head dims);
// D = 64 uses BN = 128 and computes dQ = dS K (M = 128 queries).
//
// Warp roles (14 warps): 0-3 dQ epilogue (TMEM -> global f32 atomics),
// 4-11 two warpgroups of softmax/dS work (each owns half of the BN query
// columns of all 128 key rows), 12 TMA producer, 13 MMA issuer (one thread).
// A Q/dO stage is released only by a tensor-core commit issued after every
// MMA that reads it; an accumulator is read only after its commit completed
// (the two pipelining faults the TileOPs page reports fixing in its older
// kernel, "Summary").
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "cvt.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace ab {

namespace {

template <int D>
struct Cfg {
  static constexpr int BM = kDenseBM;
  static constexpr int BN = dense_bn(D);
  static constexpr int STAGES = 2;
  static constexpr int NSLAB = D / 64;  // 64-column (128-byte) slabs per row
  static constexpr int KV_SLAB = BM * 128;
  static constexpr int KV_TILE = KV_SLAB * NSLAB;
  static constexpr int Q_SLAB = BN * 128;
  static constexpr int Q_TILE = Q_SLAB * NSLAB;
  static constexpr int DS_BYTES = BM * BN * 2;
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;
  static constexpr int OFF_DO = OFF_Q + STAGES * Q_TILE;
  static constexpr int OFF_DS = OFF_DO + STAGES * Q_TILE;
  static constexpr int OFF_LSE = OFF_DS + DS_BYTES;
  static constexpr int OFF_DELTA = OFF_LSE + STAGES * BN * 4;
  static constexpr int OFF_BAR = OFF_DELTA + STAGES * BN * 4;
  static constexpr int NBAR = 2 * STAGES + 16;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  // tensor memory columns (512 allocated)
  static constexpr int T_S = 0;                // S^T f32 [128 x BN]; P^T 16-bit pairs overwrite its first BN/2 columns
  static constexpr int T_DP = BN;              // dP^T f32 [128 x BN]
  static constexpr int T_DV = 2 * BN;          // dV f32 [128 x D]
  static constexpr int T_DK = 2 * BN + D;      // dK f32 [128 x D]
  static constexpr int T_DQ = 2 * BN + 2 * D;  // dQ^T [128 d x 64 q] (D=128) or dQ [128 q x 64 d] (D=64)
  static constexpr int T_DS = T_DQ + 64;       // dS^T 16-bit pairs [128 x BN/2]
  static_assert(T_DS + BN / 2 <= 512, "TMEM budget");
  static constexpr int THREADS = 14 * 32;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

enum Bar : int {
  B_FULL = 0,  // + stage
  B_EMPTY = 2, // + stage (STAGES == 2)
  B_KV = 4,
  B_S,
  B_DP,
  B_SREAD,
  B_P,
  B_DS,
  B_PFREE,
  B_DSFREE,
  B_DQFULL,
  B_DQEMPTY,
  B_DKV,
  B_DRAIN,
};

template <int D, bool BF16>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    dense_bwd_kernel(const __grid_constant__ DenseMaps maps, const DenseParams p) {
  using C = Cfg<D>;
  constexpr int BM = C::BM, BN = C::BN, STAGES = C::STAGES;
  static_assert(STAGES == 2, "barrier enum assumes two stages");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 8);
  float* s_lse = reinterpret_cast<float*>(sm + C::OFF_LSE);
  float* s_delta = reinterpret_cast<float*>(sm + C::OFF_DELTA);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- tile
  const int BH = p.B * p.HKV;
  const int bh = blockIdx.x % BH;
  int t = blockIdx.x / BH;
  const int b = bh / p.HKV, g = bh % p.HKV;
  int seq_start = 0, len = p.S;
  if (p.cu_seqlens != nullptr) {
    bool found = false;
    for (int n = 0; n < p.num_seqs; ++n) {
      const int a = clamp_pos(p.cu_seqlens[n], p.S), e = clamp_pos(p.cu_seqlens[n + 1], p.S);
      const int nt = e > a ? (e - a + BM - 1) / BM : 0;
      if (t < nt) {
        seq_start = a;
        len = e - a;
        found = true;
        break;
      }
      t -= nt;
    }
    if (!found) return;
  } else if (t * BM >= p.S) {
    return;
  }
  const int k0 = t * BM;
  int qlo, qhi;
  query_block_range(k0, BM, len, p.causal, p.window, BN, &qlo, &qhi);
  const int nq = qhi - qlo;
  const int n_steps = p.G * nq;

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&bars[B_FULL + i], 2);
      mbar_init(&bars[B_EMPTY + i], 1);
    }
    mbar_init(&bars[B_KV], 1);
    mbar_init(&bars[B_S], 1);
    mbar_init(&bars[B_DP], 1);
    mbar_init(&bars[B_SREAD], 8);
    mbar_init(&bars[B_P], 8);
    mbar_init(&bars[B_DS], 8);
    mbar_init(&bars[B_PFREE], 1);
    mbar_init(&bars[B_DSFREE], 1);
    mbar_init(&bars[B_DQFULL], 1);
    mbar_init(&bars[B_DQEMPTY], 4);
    mbar_init(&bars[B_DKV], 1);
    mbar_init(&bars[B_DRAIN], 1);
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
  const WaitCtx wc{abort_flag, p.err, p.timeout_ns};

  if (warp == 12) {
    // ============================================================ producer
    int pending[STAGES];
#pragma unroll
    for (int i = 0; i < STAGES; ++i) pending[i] = -1;
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.dO);
      mbar_arrive_expect_tx(&bars[B_KV], 2 * C::KV_TILE);
#pragma unroll
      for (int s = 0; s < C::NSLAB; ++s) {
        tma_load_4d(sm + C::OFF_K + s * C::KV_SLAB, &maps.k, &bars[B_KV], s * 64, g, seq_start + k0, b);
        tma_load_4d(sm + C::OFF_V + s * C::KV_SLAB, &maps.v, &bars[B_KV], s * 64, g, seq_start + k0, b);
      }
    }
    for (int i = 0; i < n_steps; ++i) {
      const int st = i % STAGES, r = i / STAGES;
      if (i >= STAGES && !mbar_wait_warp(&bars[B_EMPTY + st], (r - 1) & 1, wc, kErrWaitStageEmpty)) break;
      const int h = g * p.G + i / nq, q0 = (qlo + i % nq) * BN;
      const int64_t rowbase = (static_cast<int64_t>(b) * p.HQ + h) * p.S + seq_start;
      for (int c = lane; c < BN; c += 32) {
        const int q = q0 + c;
        float l = 0.f, d = 0.f;
        if (q < len) {
          l = p.lse2[rowbase + q];
          d = p.delta[rowbase + q];
        }
        s_lse[st * BN + c] = l;
        s_delta[st * BN + c] = d;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[B_FULL + st], 2 * C::Q_TILE);
#pragma unroll
        for (int s = 0; s < C::NSLAB; ++s) {
          tma_load_4d(sm + C::OFF_Q + st * C::Q_TILE + s * C::Q_SLAB, &maps.q, &bars[B_FULL + st], s * 64, h,
                      seq_start + q0, b);
          tma_load_4d(sm + C::OFF_DO + st * C::Q_TILE + s * C::Q_SLAB, &maps.dO, &bars[B_FULL + st], s * 64, h,
                      seq_start + q0, b);
        }
        mbar_arrive(&bars[B_FULL + st]);
      }
      pending[st] = r & 1;
    }
    // loads still in flight must land before the CTA exits
    if (lane == 0) {
      mbar_drain(&bars[B_KV], 0);
#pragma unroll
      for (int i = 0; i < STAGES; ++i)
        if (pending[i] >= 0) mbar_drain(&bars[B_FULL + i], pending[i]);
    }
  } else if (warp == 13) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_f16(BF16, 128, BN, false, false);
      constexpr uint32_t IDESC_KV = idesc_f16(BF16, 128, D, false, true);
      constexpr uint32_t IDESC_DQ = idesc_f16(BF16, 128, 64, true, true);
      const uint32_t sK = smem_u32(sm + C::OFF_K), sV = smem_u32(sm + C::OFF_V), sDS = smem_u32(sm + C::OFF_DS);
      auto sQ = [&](int st) { return smem_u32(sm + C::OFF_Q + st * C::Q_TILE); };
      auto sDO = [&](int st) { return smem_u32(sm + C::OFF_DO + st * C::Q_TILE); };
      // K-major operands: K-step kk of 16 elements = slab kk/4, byte offset 32*(kk%4)
      auto issue_S = [&](int st) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk / 4) * C::KV_SLAB + (kk % 4) * 32, qo = (kk / 4) * C::Q_SLAB + (kk % 4) * 32;
          mma_ss(tmem + C::T_S, sdesc_sw128(sK + ko, 16, 1024), sdesc_sw128(sQ(st) + qo, 16, 1024), IDESC_S, kk > 0);
        }
      };
      auto issue_dP = [&](int st) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk / 4) * C::KV_SLAB + (kk % 4) * 32, qo = (kk / 4) * C::Q_SLAB + (kk % 4) * 32;
          mma_ss(tmem + C::T_DP, sdesc_sw128(sV + ko, 16, 1024), sdesc_sw128(sDO(st) + qo, 16, 1024), IDESC_S,
                 kk > 0);
        }
      };
      // MN-major B (dO or Q as [N = D] x [K = queries]): K-step = 16 rows = 2048 bytes
      auto issue_dV = [&](int st, bool acc) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem + C::T_DV, tmem + C::T_S + kk * 8, sdesc_sw128(sDO(st) + kk * 2048, C::Q_SLAB, 1024), IDESC_KV,
                 acc || kk > 0);
      };
      auto issue_dK = [&](int st, bool acc) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem + C::T_DK, tmem + C::T_DS + kk * 8, sdesc_sw128(sQ(st) + kk * 2048, C::Q_SLAB, 1024), IDESC_KV,
                 acc || kk > 0);
      };
      // dQ: contraction over the 128 key rows (K-step = 16 key rows = 2048 bytes)
      auto issue_dQ = [&]() {
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
          if constexpr (D == 128)  // dQ^T = K^T dS^T: A = K tile MN-major, B = dS^T MN-major
            mma_ss(tmem + C::T_DQ, sdesc_sw128(sK + kk * 2048, C::KV_SLAB, 1024),
                   sdesc_sw128(sDS + kk * 2048, C::KV_SLAB, 1024), IDESC_DQ, kk > 0);
          else  // dQ = dS K: A = dS MN-major (two 64-query blocks), B = K tile MN-major
            mma_ss(tmem + C::T_DQ, sdesc_sw128(sDS + kk * 2048, BM * 128, 1024),
                   sdesc_sw128(sK + kk * 2048, C::KV_SLAB, 1024), IDESC_DQ, kk > 0);
        }
      };

      bool ok = mbar_wait(&bars[B_KV], 0, wc, kErrWaitKV);
      tc_fence_after();
      if (ok && n_steps > 0) {
        ok = mbar_wait(&bars[B_FULL + 0], 0, wc, kErrWaitStageFull);
        tc_fence_after();
        if (ok) {
          issue_S(0);
          mma_commit(&bars[B_S]);
          issue_dP(0);
          mma_commit(&bars[B_DP]);
        }
      }
      for (int i = 0; ok && i < n_steps; ++i) {
        const int st = i % STAGES;
        if (!(ok = mbar_wait(&bars[B_P], i & 1, wc, kErrWaitP))) break;
        tc_fence_after();
        issue_dV(st, i > 0);
        mma_commit(&bars[B_PFREE]);
        if (!(ok = mbar_wait(&bars[B_DS], i & 1, wc, kErrWaitDS))) break;
        tc_fence_after();
        issue_dK(st, i > 0);
        if (i > 0) {
          if (!(ok = mbar_wait(&bars[B_DQEMPTY], (i - 1) & 1, wc, kErrWaitDQEmpty))) break;
          tc_fence_after();
        }
        issue_dQ();
        mma_commit(&bars[B_DQFULL]);
        mma_commit(&bars[B_DSFREE]);
        mma_commit(&bars[B_EMPTY + st]);
        if (i + 1 < n_steps) {
          const int st1 = (i + 1) % STAGES;
          if (!(ok = mbar_wait(&bars[B_FULL + st1], ((i + 1) / STAGES) & 1, wc, kErrWaitStageFull))) break;
          if (!(ok = mbar_wait(&bars[B_PFREE], i & 1, wc, kErrWaitPFree))) break;
          tc_fence_after();
          issue_S(st1);
          mma_commit(&bars[B_S]);
          issue_dP(st1);
          mma_commit(&bars[B_DP]);
        }
      }
      if (ok) mma_commit(&bars[B_DKV]);
      // every MMA issued by this thread completes before TMEM is released
      mma_commit(&bars[B_DRAIN]);
      mbar_drain(&bars[B_DRAIN], 0);
    }
  } else if (warp >= 4) {
    // ============================================================ softmax / dS
    const int wg = (warp - 4) >> 2, quad = warp & 3;
    const int row = quad * 32 + lane;  // key row of the tile = TMEM lane
    const int kpos = k0 + row;
    const bool kvalid = kpos < len;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    constexpr int HALF = BN / 2;  // query columns of this warpgroup
    constexpr int NCH = HALF / 32;
    const bool cm = p.causal || p.window > 0;
    const int W = p.window;
    float pv[HALF];
    uint32_t dsw[HALF / 2];
    bool ok = true;
    for (int i = 0; ok && i < n_steps; ++i) {
      const int st = i % STAGES;
      const int qc0 = (qlo + i % nq) * BN + wg * HALF;  // first query (sequence-local) of my columns
      const float* lse = s_lse + st * BN + wg * HALF;
      const float* dlt = s_delta + st * BN + wg * HALF;
      if (!(ok = mbar_wait_warp(&bars[B_FULL + st], (i / STAGES) & 1, wc, kErrWaitStageFull))) break;
      if (!(ok = mbar_wait_warp(&bars[B_S], i & 1, wc, kErrWaitS))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::T_S + wg * HALF + ch * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int cc = ch * 32 + c, q = qc0 + cc;
          bool vis = kvalid && q < len;
          if (cm) vis = vis && kpos <= q;
          if (W > 0) vis = vis && q < kpos + W;
          pv[cc] = vis ? ex2(fmaf(__uint_as_float(r[c]), p.scale_log2, -lse[cc])) : 0.f;
        }
      }
      // P^T overwrites S^T columns that the other warpgroup reads: all eight
      // warps finish reading S^T first.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_SREAD]);
      if (!(ok = mbar_wait_warp(&bars[B_SREAD], i & 1, wc, kErrWaitSRead))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) w[c] = pack2<BF16>(pv[ch * 32 + 2 * c], pv[ch * 32 + 2 * c + 1]);
        tmem_st16(tmem + lane_off + C::T_S + (wg * HALF + ch * 32) / 2, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_P]);

      if (!(ok = mbar_wait_warp(&bars[B_DP], i & 1, wc, kErrWaitDP))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::T_DP + wg * HALF + ch * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int cc = ch * 32 + c;
          const float d0 = pv[cc] * (__uint_as_float(r[c]) - dlt[cc]);
          const float d1 = pv[cc + 1] * (__uint_as_float(r[c + 1]) - dlt[cc + 1]);
          dsw[cc / 2] = pack2<BF16>(d0, d1);
        }
      }
      if (i > 0 && !(ok = mbar_wait_warp(&bars[B_DSFREE], (i - 1) & 1, wc, kErrWaitDSFree))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) tmem_st16(tmem + lane_off + C::T_DS + (wg * HALF + ch * 32) / 2, dsw + ch * 16);
      if constexpr (D == 128) {
        // dS^T as the MN-major B operand [128 key rows x 64 queries]: my 32
        // queries are 16-byte chunks 4*wg .. 4*wg+3 of row ``row``
        uint8_t* base = sm + C::OFF_DS;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          *reinterpret_cast<uint4*>(base + sw128_offset(row, wg * 4 + c4)) =
              make_uint4(dsw[c4 * 4], dsw[c4 * 4 + 1], dsw[c4 * 4 + 2], dsw[c4 * 4 + 3]);
      } else {
        // dS as the MN-major A operand: 64-query block wg, row = key
        uint8_t* base = sm + C::OFF_DS + wg * (BM * 128);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          *reinterpret_cast<uint4*>(base + sw128_offset(row, c8)) =
              make_uint4(dsw[c8 * 4], dsw[c8 * 4 + 1], dsw[c8 * 4 + 2], dsw[c8 * 4 + 3]);
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_DS]);
    }
    // ---- dK / dV: warpgroup 0 lands dV, warpgroup 1 lands dK (times sm_scale)
    if (ok && n_steps > 0) ok = mbar_wait_warp(&bars[B_DKV], 0, wc, kErrWaitDKV);
    if (ok) {
      tc_fence_after();
      const bool isK = wg == 1;
      const uint32_t col0 = isK ? C::T_DK : C::T_DV;
      const float mul = isK ? p.sm_scale : 1.f;
      const int64_t pos = seq_start + kpos;
      uint8_t* out = isK ? p.dk + 2 * (b * p.sdk_b + pos * p.sdk_s + g * p.sdk_h)
                         : p.dv + 2 * (b * p.sdv_b + pos * p.sdv_s + g * p.sdv_h);
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        if (n_steps > 0) {
          tmem_ld32(tmem + lane_off + col0 + ch * 32, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = 0u;
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
  } else {
    // ============================================================ dQ epilogue
    const int quad = warp;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    for (int i = 0; ok && i < n_steps; ++i) {
      const int h = g * p.G + i / nq, q0 = (qlo + i % nq) * BN;
      if (!(ok = mbar_wait_warp(&bars[B_DQFULL], i & 1, wc, kErrWaitDQFull))) break;
      tc_fence_after();
      uint32_t r[64];
      tmem_ld32(tmem + lane_off + C::T_DQ, r);
      tmem_ld32(tmem + lane_off + C::T_DQ + 32, r + 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_DQEMPTY]);
      if constexpr (D == 128) {
        // lane = head dim d, columns = the BN (= 64) queries of the block
        const int d = quad * 32 + lane;
        const int nvalid = imin(BN, len - q0);
        float* base = p.dq_acc + ((static_cast<int64_t>(b) * p.S + seq_start + q0) * p.HQ + h) * D + d;
        const int64_t qstride = static_cast<int64_t>(p.HQ) * D;
#pragma unroll 8
        for (int c = 0; c < 64; ++c)
          if (c < nvalid) atomicAdd(base + c * qstride, __uint_as_float(r[c]));
      } else {
        // lane = query, columns = the 64 head dims
        const int q = q0 + quad * 32 + lane;
        if (q < len) {
          float4* base = reinterpret_cast<float4*>(
              p.dq_acc + ((static_cast<int64_t>(b) * p.S + seq_start + q) * p.HQ + h) * D);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            atomicAdd(base + c, make_float4(__uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1]),
                                            __uint_as_float(r[4 * c + 2]), __uint_as_float(r[4 * c + 3])));
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16>
cudaError_t launch_dense_t(const DenseParams& p, const DenseMaps& m, int grid, cudaStream_t st) {
  auto kern = dense_bwd_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, Cfg<D>::THREADS, Cfg<D>::SMEM, st>>>(m, p);
  return cudaGetLastError();
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
  if (p.D == 128) return bf16 ? launch_dense_t<128, true>(p, m, grid, st) : launch_dense_t<128, false>(p, m, grid, st);
  return bf16 ? launch_dense_t<64, true>(p, m, grid, st) : launch_dense_t<64, false>(p, m, grid, st);
}

cudaError_t launch_selftest_timeout(int* err, uint64_t timeout_ns, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace ab
