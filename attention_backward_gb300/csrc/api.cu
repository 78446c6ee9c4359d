// Host entry points of the C ABI declared in include/attn_bwd.h: argument
// validation, workspace layout, TMA descriptors and launches.  Nothing here
// allocates device memory or keeps state between calls other than the
// driver entry point of cuTensorMapEncodeTiled, looked up once.
//
// Every launch is prepared by a set-up function that checks its arguments and
// encodes its tensor maps without touching the device; the one-call forms set
// up all three launches of a backward before queueing the first, so a bad
// call queues nothing.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_bwd.h"
#include "attn_bwd_sink.h"
#include "common.cuh"
#include "dense_common.cuh"
#include "kernels.h"
#include "sink.h"

namespace {

using namespace ab;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// BSHD strides (elements) of a 16-bit tensor: positive, 16-byte multiples,
// within the TMA stride limit.
bool strides_ok(const attn_strides_t& s) {
  auto one = [](int64_t x) { return x > 0 && ((x * 2) % 16) == 0 && x * 2 < (int64_t(1) << 40); };
  return one(s.b) && one(s.s) && one(s.h);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

attn_status_t launch_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH; }

// 4-D tiled map over a BSHD 16-bit tensor: dims (D, H, S, B), box (64, 1,
// rows, 1), 128-byte swizzle (the layout the tcgen05 descriptors expect).
bool make_map(CUtensorMap* m, const void* base, attn_dtype_t dt, int64_t B, int64_t S, int64_t H, int64_t D,
              const attn_strides_t& st, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.h * 2), static_cast<cuuint64_t>(st.s * 2),
                           static_cast<cuuint64_t>(st.b * 2)};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty = dt == ATTN_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, ty, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// f32 accumulator [B,S,H,D] (contiguous) as the target of bulk reduce-adds:
// box (box_d, 1, rows, 1); 128-byte swizzle when box_d * 4 == 128.
bool make_acc_map(CUtensorMap* m, void* base, int64_t B, int64_t S, int64_t H, int64_t D, int box_d, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D * 4), static_cast<cuuint64_t>(H * D * 4),
                           static_cast<cuuint64_t>(S * H * D * 4)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_d), 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = box_d * 4 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over [B,S,H,Dfull] 16-bit with a box of 64 columns x 64 heads of
// one token (the sparse path's Q and dO chunks), 128-byte swizzle.
bool make_head_map(CUtensorMap* m, const void* base, attn_dtype_t dt, int64_t B, int64_t S, int64_t H, int64_t D,
                   const attn_strides_t& st) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.h * 2), static_cast<cuuint64_t>(st.s * 2),
                           static_cast<cuuint64_t>(st.b * 2)};
  cuuint32_t box[4] = {64, 64, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty = dt == ATTN_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, ty, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over ``rows`` dense rows of D 16-bit values, box 64 x 1 (for gather4).
bool make_row_map(CUtensorMap* m, const void* base, attn_dtype_t dt, int64_t rows, int64_t D, int64_t row_stride) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride * 2)};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType ty = dt == ATTN_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(m, ty, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


uint64_t wait_limit_ns() { return ab::kWaitTimeoutNs; }

bool dtype_ok(attn_dtype_t dt) { return dt == ATTN_DT_F16 || dt == ATTN_DT_BF16; }

// ---------------------------------------------------------------- set-up of each launch

struct PreSetup {
  PreprocessParams p;
  bool bf16;
};

attn_status_t setup_preprocess(PreSetup* s, const void* o, attn_strides_t so, const void* dO, attn_strides_t sdo,
                               const float* lse, attn_strides_t slse, int64_t B, int64_t S, int64_t H, int64_t Dv,
                               int64_t Dq, int64_t dkv_elems, attn_dtype_t dtype, void* workspace,
                               size_t workspace_bytes) {
  if (!o || !dO || !lse || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || Dv < 8 || Dv % 8 || Dv > 1024 || Dq < 0 || Dq % 8 || dkv_elems < 0)
    return ATTN_ERR_INVALID_ARG;
  if (B * S * H >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  if (!dtype_ok(dtype)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(workspace) || !strides_ok(so) || !strides_ok(sdo))
    return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0 || slse.b < 0 || slse.s < 0 || slse.h < 0)
    return ATTN_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(B, S, H, Dq, dkv_elems);
  if (workspace_bytes < static_cast<size_t>(L.total)) return ATTN_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PreprocessParams& p = s->p;
  p = PreprocessParams{};
  p.o = static_cast<const uint8_t*>(o);
  p.so_b = so.b, p.so_s = so.s, p.so_h = so.h;
  p.dO = static_cast<const uint8_t*>(dO);
  p.sdo_b = sdo.b, p.sdo_s = sdo.s, p.sdo_h = sdo.h;
  p.lse = lse;
  p.sl_b = slse.b, p.sl_s = slse.s, p.sl_h = slse.h;
  p.B = static_cast<int>(B), p.S = static_cast<int>(S), p.H = static_cast<int>(H), p.Dv = static_cast<int>(Dv);
  p.lse2 = reinterpret_cast<float*>(ws + L.lse2_off);
  p.delta = reinterpret_cast<float*>(ws + L.delta_off);
  p.dq_zero = reinterpret_cast<float4*>(ws + L.dq_off);
  p.dq_row_n4 = static_cast<int>(Dq / 4);
  p.zero = reinterpret_cast<float4*>(ws + L.dkv_off);
  p.zero_n4 = (L.total - L.dkv_off) / 16;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  s->bf16 = dtype == ATTN_DT_BF16;
  return ATTN_OK;
}

attn_status_t run_preprocess(const PreSetup& s, void* stream) {
  return launch_status(launch_preprocess(s.p, s.bf16, sm_count() * 8, static_cast<cudaStream_t>(stream)));
}

// The mask of a dense call: causal, window, packed sequences and the key
// length (0 in kv_len: the query length S).
struct MaskArgs {
  int causal = 0, window = -1, num_seqs = 0;
  const int32_t* cu = nullptr;
  int64_t Sk = 0;
};

attn_status_t parse_mask(const attn_mask_t* mask, int64_t B, int64_t S, MaskArgs* m) {
  *m = MaskArgs{};
  m->Sk = S;
  if (!mask) return ATTN_OK;
  m->causal = mask->causal ? 1 : 0;
  m->window = mask->window_left;
  m->cu = mask->cu_seqlens;
  m->num_seqs = mask->num_seqs;
  if (m->window == 0 || m->window < -1) return ATTN_ERR_INVALID_ARG;
  if (m->cu && (B != 1 || m->num_seqs < 1 || m->num_seqs > (1 << 20))) return ATTN_ERR_INVALID_ARG;
  if (m->cu && (reinterpret_cast<uintptr_t>(m->cu) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  if (mask->kv_len < 0 || (m->cu && mask->kv_len != 0 && mask->kv_len != S)) return ATTN_ERR_INVALID_ARG;
  if (mask->kv_len > 0) m->Sk = mask->kv_len;
  if (!m->cu) m->num_seqs = 0;
  return ATTN_OK;
}

struct DenseSetup {
  DenseParams p;
  DenseMaps m;
  bool bf16;
  int grid;
  size_t part_bytes;  // last-round partials cleared before the launch (0: no split)
};

attn_status_t setup_dense(DenseSetup* s, const void* q, attn_strides_t sq, const void* k, attn_strides_t sk,
                          const void* v, attn_strides_t sv, const void* dO, attn_strides_t sdo, int64_t B, int64_t S,
                          int64_t HQ, int64_t HKV, int64_t D, attn_dtype_t dtype, float sm_scale,
                          const attn_mask_t* mask, void* dk, attn_strides_t sdk, void* dv, attn_strides_t sdv,
                          void* workspace, size_t workspace_bytes, bool encode = true) {
  s->part_bytes = 0;
  if (!q || !k || !v || !dO || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || HQ < 1 || HKV < 1 || HQ % HKV != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!dtype_ok(dtype)) return ATTN_ERR_UNSUPPORTED;
  if (HQ / HKV > (dtype == ATTN_DT_BF16 ? ATTN_BWD_MAX_GROUP_BF16 : ATTN_BWD_MAX_GROUP_F16))
    return ATTN_ERR_UNSUPPORTED;
  if (S >= (int64_t(1) << 31) || B * HQ * S >= (int64_t(1) << 31) || B > 65535 || HQ > 65535)
    return ATTN_ERR_UNSUPPORTED;
  for (const void* ptr : {q, k, v, dO, static_cast<const void*>(dk), static_cast<const void*>(dv),
                          static_cast<const void*>(workspace)})
    if (!aligned16(ptr)) return ATTN_ERR_INVALID_ARG;
  for (const attn_strides_t* st : {&sq, &sk, &sv, &sdo, &sdk, &sdv})
    if (!strides_ok(*st)) return ATTN_ERR_INVALID_ARG;
  MaskArgs ma;
  if (const attn_status_t mst = parse_mask(mask, B, S, &ma); mst != ATTN_OK) return mst;
  const int causal = ma.causal, window = ma.window, num_seqs = ma.num_seqs;
  const int32_t* cu = ma.cu;
  const int64_t Sk = ma.Sk;  // keys per batch row
  if (B * HKV * Sk >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(B, S, HQ, D, 0);
  if (workspace_bytes < static_cast<size_t>(L.total)) return ATTN_ERR_WORKSPACE;
  // key tiles per (batch, KV head): a packed batch may add one partial tile per
  // sequence.  Persistent CTAs, one per SM, draw tiles from the counter.
  const int64_t tiles = ((Sk + kDenseBM - 1) / kDenseBM + (cu ? num_seqs : 0)) * B * HKV;
  if (tiles >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  if (!encode) return ATTN_OK;  // argument checks only: no driver call
  const int BN = kDenseBN;
  DenseMaps& m = s->m;
  if (!make_map(&m.q, q, dtype, B, S, HQ, D, sq, BN) || !make_map(&m.dO, dO, dtype, B, S, HQ, D, sdo, BN) ||
      !make_map(&m.k, k, dtype, B, Sk, HKV, D, sk, kDenseBM) || !make_map(&m.v, v, dtype, B, Sk, HKV, D, sv, kDenseBM))
    return ATTN_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // dQ partials land as [128 queries x 32 d] boxes staged with a 128-byte swizzle
  if (!make_acc_map(&m.dq, ws + L.dq_off, B, S, HQ, D, 32, BN)) return ATTN_ERR_INVALID_ARG;
  DenseParams& p = s->p;
  p = DenseParams{};
  p.B = static_cast<int>(B), p.S = static_cast<int>(S), p.HQ = static_cast<int>(HQ), p.HKV = static_cast<int>(HKV);
  p.G = static_cast<int>(HQ / HKV), p.D = static_cast<int>(D), p.Sk = static_cast<int>(Sk);
  p.causal = causal, p.window = window, p.cu_seqlens = cu, p.num_seqs = num_seqs;
  p.sm_scale = sm_scale;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.lse2 = reinterpret_cast<const float*>(ws + L.lse2_off);
  p.delta = reinterpret_cast<const float*>(ws + L.delta_off);
  p.dq_acc = reinterpret_cast<float*>(ws + L.dq_off);
  p.err = &reinterpret_cast<WsHeader*>(ws)->err;
  p.dk = static_cast<uint8_t*>(dk), p.sdk_b = sdk.b, p.sdk_s = sdk.s, p.sdk_h = sdk.h;
  p.dv = static_cast<uint8_t*>(dv), p.sdv_b = sdv.b, p.sdv_s = sdv.s, p.sdv_h = sdv.h;
  p.timeout_ns = wait_limit_ns();
  p.tile_counter = &reinterpret_cast<WsHeader*>(ws)->tile_counter;
  p.bn = BN;
  s->bf16 = dtype == ATTN_DT_BF16;
  s->grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  p.tile_group = tile_group(s->grid, static_cast<int>((Sk + kDenseBM - 1) / kDenseBM));
  return ATTN_OK;
}

// The last-round split of a dense batch's key tiles: with T equal tiles on
// ``ctas`` persistent CTAs the last round holds T mod ctas tiles, and the
// other CTAs idle meanwhile.  Drawing those tiles as units of ``hpu`` query
// heads (dK/dV partials added in f32) spreads them over all CTAs.  The
// makespan is counted in 1/G tiles; the split is taken when it shortens the
// last round by at least a quarter of a tile (half a tile at G = 2), with the
// largest head count among equal makespans.
struct TailPlan {
  int start, tiles, hpu;  // tiles = 0: no split
};
TailPlan tail_plan(int64_t T, int64_t ctas, int G) {
  TailPlan t{0, 0, 0};
  if (G < 2 || ctas < 1 || T <= ctas) return t;
  const int64_t full = T / ctas, R = T % ctas;
  if (R == 0 || R > kMaxTailTiles) return t;
  const int64_t whole = (full + 1) * G;
  int64_t best = whole;
  int hpu_best = 0;
  for (int hpu = G - 1; hpu >= 1; --hpu) {
    if (G % hpu) continue;
    const int64_t units = R * (G / hpu);
    const int64_t ms = full * G + (units + ctas - 1) / ctas * hpu;
    if (ms < best) best = ms, hpu_best = hpu;
  }
  if (hpu_best == 0 || whole - best < (G / 4 > 1 ? G / 4 : 1)) return t;
  t.start = static_cast<int>(T - R), t.tiles = static_cast<int>(R), t.hpu = hpu_best;
  return t;
}

// f32 elements of the partials region for ``tiles`` split tiles at head dim D:
// the per-quarter unit counters (padded to 256 bytes), then the partials.
int64_t tail_region_elems(int64_t tiles, int64_t D) { return round_up(tiles * 4, 64) + tiles * 2 * D * kDenseBM; }

// Enables the last-round split of a checked dense set-up when it applies (head
// dim 128, an unmasked dense batch, more than one query head per KV head) and
// the workspace has room for the partials behind the dQ accumulator; run_dense
// then clears them before the launch.
void plan_tail_split(DenseSetup* s, void* workspace, size_t workspace_bytes) {
  DenseParams& p = s->p;
  p.tail_start = p.tail_tiles = p.tail_hpu = 0;
  s->part_bytes = 0;
  if (p.D != 128 || p.cu_seqlens != nullptr || p.causal || p.window > 0) return;
  const int64_t T = static_cast<int64_t>((p.Sk + kDenseBM - 1) / kDenseBM) * p.B * p.HKV;
  const TailPlan t = tail_plan(T, s->grid, p.G);
  if (t.tiles == 0) return;
  const int64_t elems = tail_region_elems(t.tiles, p.D);
  const WsLayout L = ws_layout(p.B, p.S, p.HQ, p.D, elems);
  if (workspace_bytes < static_cast<size_t>(L.total)) return;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.tail_start = t.start, p.tail_tiles = t.tiles, p.tail_hpu = t.hpu;
  p.part_count = reinterpret_cast<int*>(ws + L.dkv_off);
  p.part_acc = reinterpret_cast<float*>(ws + L.dkv_off + round_up(t.tiles * 4, 64) * 4);
  s->part_bytes = static_cast<size_t>(elems) * 4;
}

attn_status_t run_dense(const DenseSetup& s, void* stream) {
  if (s.part_bytes > 0 && cudaMemsetAsync(s.p.part_count, 0, s.part_bytes, static_cast<cudaStream_t>(stream)) !=
                              cudaSuccess)
    return ATTN_ERR_LAUNCH;
  return launch_status(launch_dense(s.p, s.m, s.bf16, s.grid, static_cast<cudaStream_t>(stream)));
}

struct FwdSetup {
  FwdParams p;
  FwdMaps m;
  bool bf16;
  int grid;
  void* workspace;
};

attn_status_t setup_fwd(FwdSetup* s, const void* q, attn_strides_t sq, const void* k, attn_strides_t sk,
                        const void* v, attn_strides_t sv, int64_t B, int64_t S, int64_t HQ, int64_t HKV, int64_t D,
                        attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask, void* o, attn_strides_t so,
                        float* lse, attn_strides_t slse, void* workspace, size_t workspace_bytes) {
  if (!q || !k || !v || !o || !lse || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || HQ < 1 || HKV < 1 || HQ % HKV != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!dtype_ok(dtype)) return ATTN_ERR_UNSUPPORTED;
  for (const void* ptr : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(workspace)})
    if (!aligned16(ptr)) return ATTN_ERR_INVALID_ARG;
  for (const attn_strides_t* st : {&sq, &sk, &sv, &so})
    if (!strides_ok(*st)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0 || slse.b < 0 || slse.s < 0 || slse.h < 0)
    return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < static_cast<size_t>(kHeaderBytes)) return ATTN_ERR_WORKSPACE;
  MaskArgs ma;
  if (const attn_status_t mst = parse_mask(mask, B, S, &ma); mst != ATTN_OK) return mst;
  if (S >= (int64_t(1) << 31) || B * HQ * S >= (int64_t(1) << 31) || B * HKV * ma.Sk >= (int64_t(1) << 31) ||
      B > 65535 || HQ > 65535)
    return ATTN_ERR_UNSUPPORTED;
  // units of two 128-row query tiles per (batch row or sequence, query head); a
  // packed batch may add one partial unit per sequence
  const int64_t units = ((S + 255) / 256 + (ma.cu ? ma.num_seqs : 0)) * B * HQ;
  if (units >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  FwdMaps& m = s->m;
  if (!make_map(&m.q, q, dtype, B, S, HQ, D, sq, 128) || !make_map(&m.k, k, dtype, B, ma.Sk, HKV, D, sk, 128) ||
      !make_map(&m.v, v, dtype, B, ma.Sk, HKV, D, sv, 128))
    return ATTN_ERR_INVALID_ARG;
  FwdParams& p = s->p;
  p = FwdParams{};
  p.B = static_cast<int>(B), p.S = static_cast<int>(S), p.Sk = static_cast<int>(ma.Sk);
  p.HQ = static_cast<int>(HQ), p.HKV = static_cast<int>(HKV), p.G = static_cast<int>(HQ / HKV);
  p.D = static_cast<int>(D);
  p.causal = ma.causal, p.window = ma.window, p.cu_seqlens = ma.cu, p.num_seqs = ma.num_seqs;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.o = static_cast<uint8_t*>(o), p.so_b = so.b, p.so_s = so.s, p.so_h = so.h;
  p.lse = lse, p.sl_b = slse.b, p.sl_s = slse.s, p.sl_h = slse.h;
  p.err = &static_cast<WsHeader*>(workspace)->err;
  p.unit_counter = &static_cast<WsHeader*>(workspace)->tile_counter;
  p.timeout_ns = wait_limit_ns();
  s->bf16 = dtype == ATTN_DT_BF16;
  // persistent CTAs, one per SM, draw units from the counter
  s->grid = static_cast<int>(units < sm_count() ? units : sm_count());
  s->workspace = workspace;
  return ATTN_OK;
}

attn_status_t run_fwd(const FwdSetup& s, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the error word and the unit counter start clear; the kernel records the
  // first wait that ran out
  if (cudaMemsetAsync(s.workspace, 0, kHeaderBytes, st) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return launch_status(launch_fwd(s.p, s.m, s.bf16, s.grid, st));
}

struct LandSetup {
  LandParams p;
  bool bf16;
};

attn_status_t setup_dq_land(LandSetup* s, void* dq, attn_strides_t sdq, int64_t B, int64_t S, int64_t H, int64_t D,
                            attn_dtype_t dtype, float sm_scale, const void* workspace, size_t workspace_bytes) {
  if (!dq || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || H < 1 || D < 8 || D % 8) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return ATTN_ERR_INVALID_ARG;
  if (B * S * H >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  if (!dtype_ok(dtype)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(dq) || !aligned16(workspace) || !strides_ok(sdq)) return ATTN_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(B, S, H, D, 0);
  if (workspace_bytes < static_cast<size_t>(L.dkv_off)) return ATTN_ERR_WORKSPACE;
  LandParams& p = s->p;
  p = LandParams{};
  p.acc = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + L.dq_off);
  p.rows = B * S * H;
  p.B = static_cast<int>(B), p.S = static_cast<int>(S), p.H = static_cast<int>(H), p.D = static_cast<int>(D);
  p.out = static_cast<uint8_t*>(dq);
  p.s_b = sdq.b, p.s_s = sdq.s, p.s_h = sdq.h;
  p.scale = sm_scale;
  s->bf16 = dtype == ATTN_DT_BF16;
  return ATTN_OK;
}

attn_status_t run_land(const LandSetup& s, void* stream) {
  return launch_status(launch_land(s.p, s.bf16, sm_count() * 8, static_cast<cudaStream_t>(stream)));
}

struct SparseSetup {
  SparseParams p;
  SparseMaps m;
  bool bf16;
  int grid;
};

attn_status_t setup_sparse(SparseSetup* s, const void* q, attn_strides_t sq, const void* kv, attn_strides_t skv,
                           const void* dO, attn_strides_t sdo, const int32_t* idx, attn_strides_t sidx, int64_t B,
                           int64_t S, int64_t SKV, int64_t H, int64_t HKV, int64_t DQK, int64_t DV, int64_t topk,
                           attn_dtype_t dtype, float sm_scale, void* dq, attn_strides_t sdq, void* workspace,
                           size_t workspace_bytes) {
  if (!q || !kv || !dO || !idx || !dq || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || SKV < 1 || H < 1 || HKV < 1 || H % HKV != 0 || topk < 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return ATTN_ERR_INVALID_ARG;
  if (DQK != 576 || DV != 512 || H / HKV > 64) return ATTN_ERR_UNSUPPORTED;
  if (!dtype_ok(dtype)) return ATTN_ERR_UNSUPPORTED;
  if (B * S * HKV >= (int64_t(1) << 31) || B * SKV * HKV >= (int64_t(1) << 31) || topk >= (int64_t(1) << 31))
    return ATTN_ERR_UNSUPPORTED;
  for (const void* ptr : {q, kv, dO, static_cast<const void*>(idx), static_cast<const void*>(dq),
                          static_cast<const void*>(workspace)})
    if (!aligned16(ptr)) return ATTN_ERR_INVALID_ARG;
  for (const attn_strides_t* st : {&sq, &sdo, &sdq})
    if (!strides_ok(*st)) return ATTN_ERR_INVALID_ARG;
  // the latent rows are gathered as rows of a dense [B*SKV*HKV, DQK] matrix
  if (skv.h < DQK || (skv.h * 2) % 16 || skv.s != HKV * skv.h || skv.b != SKV * skv.s) return ATTN_ERR_UNSUPPORTED;
  if (sidx.b < 0 || sidx.s < 0 || sidx.h < 0) return ATTN_ERR_INVALID_ARG;
  const int64_t dkv_elems = B * SKV * HKV * DQK;
  const WsLayout L = ws_layout(B, S, H, 0, dkv_elems);
  if (workspace_bytes < static_cast<size_t>(L.total)) return ATTN_ERR_WORKSPACE;
  SparseMaps& m = s->m;
  if (!make_head_map(&m.q, q, dtype, B, S, H, DQK, sq) || !make_head_map(&m.dO, dO, dtype, B, S, H, DV, sdo) ||
      !make_row_map(&m.kv, kv, dtype, B * SKV * HKV, DQK, skv.h))
    return ATTN_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SparseParams& p = s->p;
  p = SparseParams{};
  p.B = static_cast<int>(B), p.S = static_cast<int>(S), p.SKV = static_cast<int>(SKV);
  p.H = static_cast<int>(H), p.HKV = static_cast<int>(HKV), p.topk = static_cast<int>(topk);
  p.gh = static_cast<int>(H / HKV);
  p.sm_scale = sm_scale;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.lse2 = reinterpret_cast<const float*>(ws + L.lse2_off);
  p.delta = reinterpret_cast<const float*>(ws + L.delta_off);
  p.dkv_acc = reinterpret_cast<float*>(ws + L.dkv_off);
  p.idx = idx;
  p.si_b = sidx.b, p.si_s = sidx.s, p.si_h = sidx.h;
  p.dq = static_cast<uint8_t*>(dq);
  p.sdq_b = sdq.b, p.sdq_s = sdq.s, p.sdq_h = sdq.h;
  p.err = &reinterpret_cast<WsHeader*>(ws)->err;
  p.unit_counter = &reinterpret_cast<WsHeader*>(ws)->tile_counter;
  p.timeout_ns = wait_limit_ns();
  const int64_t units = B * S * HKV;
  s->bf16 = dtype == ATTN_DT_BF16;
  s->grid = static_cast<int>(units < sm_count() ? units : sm_count());
  return ATTN_OK;
}

attn_status_t run_sparse(const SparseSetup& s, void* stream) {
  return launch_status(launch_sparse(s.p, s.m, s.bf16, s.grid, static_cast<cudaStream_t>(stream)));
}

attn_status_t setup_sparse_land(LandSetup* s, void* dkv, attn_strides_t sdkv, int64_t B, int64_t S, int64_t SKV,
                                int64_t H, int64_t HKV, int64_t DQK, attn_dtype_t dtype, const void* workspace,
                                size_t workspace_bytes) {
  if (!dkv || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || SKV < 1 || H < 1 || HKV < 1 || DQK < 8 || DQK % 8) return ATTN_ERR_INVALID_ARG;
  if (B * SKV * HKV >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  if (!dtype_ok(dtype)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(dkv) || !aligned16(workspace) || !strides_ok(sdkv)) return ATTN_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(B, S, H, 0, B * SKV * HKV * DQK);
  if (workspace_bytes < static_cast<size_t>(L.total)) return ATTN_ERR_WORKSPACE;
  LandParams& p = s->p;
  p = LandParams{};
  p.acc = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + L.dkv_off);
  p.rows = B * SKV * HKV;
  p.B = static_cast<int>(B), p.S = static_cast<int>(SKV), p.H = static_cast<int>(HKV), p.D = static_cast<int>(DQK);
  p.out = static_cast<uint8_t*>(dkv);
  p.s_b = sdkv.b, p.s_s = sdkv.s, p.s_h = sdkv.h;
  p.scale = 1.f;
  s->bf16 = dtype == ATTN_DT_BF16;
  return ATTN_OK;
}

}  // namespace

namespace ab {

// Every argument check of attn_bwd_gqa, with no device or driver call (the
// no-allocation entry point runs it before it looks up its scratch array).
attn_status_t check_gqa_call(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk, const void* v,
                             attn_strides_t sv, const void* o, attn_strides_t so, const void* dO, attn_strides_t sdo,
                             const float* lse, attn_strides_t slse, int64_t B, int64_t S, int64_t HQ, int64_t HKV,
                             int64_t D, attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask, void* dq,
                             attn_strides_t sdq, void* dk, attn_strides_t sdk, void* dv, attn_strides_t sdv,
                             void* workspace, size_t workspace_bytes) {
  DenseSetup main;
  attn_status_t st = setup_dense(&main, q, sq, k, sk, v, sv, dO, sdo, B, S, HQ, HKV, D, dtype, sm_scale, mask, dk,
                                 sdk, dv, sdv, workspace, workspace_bytes, false);
  if (st != ATTN_OK) return st;
  PreSetup pre;
  st = setup_preprocess(&pre, o, so, dO, sdo, lse, slse, B, S, HQ, D, D, 0, dtype, workspace, workspace_bytes);
  if (st != ATTN_OK) return st;
  LandSetup land;
  return setup_dq_land(&land, dq, sdq, B, S, HQ, D, dtype, sm_scale, workspace, workspace_bytes);
}

}  // namespace ab

extern "C" {

size_t attn_bwd_workspace_size(int64_t B, int64_t S, int64_t H, int64_t Dq, int64_t dkv_elems) {
  if (B < 0 || S < 0 || H < 0 || Dq < 0 || dkv_elems < 0) return 0;
  return static_cast<size_t>(ws_layout(B, S, H, Dq, dkv_elems).total);
}

size_t attn_bwd_gqa_workspace_size(int64_t B, int64_t S, int64_t HQ, int64_t D) {
  if (B < 0 || S < 0 || HQ < 0 || D < 0) return 0;
  const int64_t tiles_bound = B * HQ * ((S + kDenseBM - 1) / kDenseBM);
  const int64_t tiles = D == 128 ? (tiles_bound < kMaxTailTiles ? tiles_bound : kMaxTailTiles) : 0;
  return static_cast<size_t>(ws_layout(B, S, HQ, D, tiles > 0 ? tail_region_elems(tiles, D) : 0).total);
}

void attn_bwd_tail_plan(int64_t tiles, int32_t ctas, int32_t G, int32_t* out) {
  if (!out) return;
  const TailPlan t = tail_plan(tiles, ctas, G);
  out[0] = t.start, out[1] = t.tiles, out[2] = t.hpu;
}

const char* attn_bwd_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_LAUNCH: return "kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    case ATTN_ERR_DEVICE: return "CUDA error";
  }
  return "unknown status";
}

void attn_bwd_query_block_range(int32_t k0, int32_t block_k, int32_t len, int32_t causal, int32_t window_left,
                                int32_t block_q, int32_t* lo, int32_t* hi) {
  int l = 0, h = 0;
  if (block_k > 0 && block_q > 0) query_block_range(k0, block_k, len, causal, window_left, block_q, &l, &h);
  if (lo) *lo = l;
  if (hi) *hi = h;
}

void attn_bwd_query_block_range_qk(int32_t k0, int32_t block_k, int32_t kv_len, int32_t q_len, int32_t causal,
                                   int32_t window_left, int32_t block_q, int32_t* lo, int32_t* hi) {
  int l = 0, h = 0;
  if (block_k > 0 && block_q > 0 && kv_len >= 0 && q_len >= 0)
    query_block_range_qk(k0, block_k, kv_len, q_len, kv_len - q_len, causal, window_left, block_q, &l, &h);
  if (lo) *lo = l;
  if (hi) *hi = h;
}

void attn_bwd_tile_schedule(int32_t t, int32_t B, int32_t S, int32_t HKV, int32_t causal, int32_t window_left,
                            const int32_t* cu_seqlens, int32_t num_seqs, int32_t* out) {
  if (!out) return;
  TileInfo ti{};
  if (B >= 1 && S >= 1 && HKV >= 1 && (!cu_seqlens || num_seqs >= 1)) {
    DenseParams p{};
    p.B = B, p.S = S, p.Sk = S, p.HKV = HKV, p.G = 1;
    p.tile_group = kTileGroup;
    p.causal = causal ? 1 : 0, p.window = window_left;
    p.cu_seqlens = cu_seqlens, p.num_seqs = cu_seqlens ? num_seqs : 0;
    p.bn = kDenseBN;
    ti = decode_tile(t, p);
  }
  const int32_t v[7] = {ti.valid, ti.b, ti.g, ti.seq_start, ti.k0, ti.qlo, ti.nq};
  for (int i = 0; i < 7; ++i) out[i] = ti.valid ? v[i] : 0;
}

void attn_bwd_tile_schedule_split(int32_t t, int32_t B, int32_t S, int32_t HKV, int32_t G, int32_t tail_start,
                                  int32_t tail_tiles, int32_t tail_hpu, int32_t* out) {
  if (!out) return;
  TileInfo ti{};
  const bool split_ok = tail_tiles == 0 || (tail_tiles > 0 && tail_hpu >= 1 && G % tail_hpu == 0 && tail_start >= 0);
  if (B >= 1 && S >= 1 && HKV >= 1 && G >= 1 && split_ok) {
    DenseParams p{};
    p.B = B, p.S = S, p.Sk = S, p.HKV = HKV, p.G = G;
    p.tile_group = kTileGroup;
    p.bn = kDenseBN;
    p.tail_start = tail_start, p.tail_tiles = tail_tiles, p.tail_hpu = tail_hpu;
    ti = decode_tile(t, p);
  }
  const int32_t v[10] = {ti.valid, ti.b, ti.g, ti.seq_start, ti.k0, ti.qlo, ti.nq, ti.h0, ti.hn, ti.part};
  for (int i = 0; i < 10; ++i) out[i] = ti.valid ? v[i] : 0;
}

attn_status_t attn_bwd_preprocess(const void* o, attn_strides_t so, const void* dO, attn_strides_t sdo,
                                  const float* lse, attn_strides_t slse, int64_t B, int64_t S, int64_t H,
                                  int64_t Dv, int64_t Dq, int64_t dkv_elems, attn_dtype_t dtype, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  PreSetup s;
  const attn_status_t st =
      setup_preprocess(&s, o, so, dO, sdo, lse, slse, B, S, H, Dv, Dq, dkv_elems, dtype, workspace, workspace_bytes);
  return st != ATTN_OK ? st : run_preprocess(s, stream);
}

attn_status_t attn_bwd_gqa_main(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk, const void* v,
                                attn_strides_t sv, const void* dO, attn_strides_t sdo, int64_t B, int64_t S,
                                int64_t HQ, int64_t HKV, int64_t D, attn_dtype_t dtype, float sm_scale,
                                const attn_mask_t* mask, void* dk, attn_strides_t sdk, void* dv, attn_strides_t sdv,
                                void* workspace, size_t workspace_bytes, void* stream) {
  DenseSetup s;
  const attn_status_t st = setup_dense(&s, q, sq, k, sk, v, sv, dO, sdo, B, S, HQ, HKV, D, dtype, sm_scale, mask, dk,
                                       sdk, dv, sdv, workspace, workspace_bytes);
  if (st != ATTN_OK) return st;
  plan_tail_split(&s, workspace, workspace_bytes);
  return run_dense(s, stream);
}

attn_status_t attn_bwd_dq_land(void* dq, attn_strides_t sdq, int64_t B, int64_t S, int64_t H, int64_t D,
                               attn_dtype_t dtype, float sm_scale, const void* workspace, size_t workspace_bytes,
                               void* stream) {
  LandSetup s;
  const attn_status_t st = setup_dq_land(&s, dq, sdq, B, S, H, D, dtype, sm_scale, workspace, workspace_bytes);
  return st != ATTN_OK ? st : run_land(s, stream);
}

attn_status_t attn_bwd_gqa(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk, const void* v,
                           attn_strides_t sv, const void* o, attn_strides_t so, const void* dO, attn_strides_t sdo,
                           const float* lse, attn_strides_t slse, int64_t B, int64_t S, int64_t HQ, int64_t HKV,
                           int64_t D, attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask, void* dq,
                           attn_strides_t sdq, void* dk, attn_strides_t sdk, void* dv, attn_strides_t sdv,
                           void* workspace, size_t workspace_bytes, void* stream) {
  // the three launches are set up (checked, tensor maps encoded) before the first is queued
  DenseSetup main;
  attn_status_t st = setup_dense(&main, q, sq, k, sk, v, sv, dO, sdo, B, S, HQ, HKV, D, dtype, sm_scale, mask, dk,
                                 sdk, dv, sdv, workspace, workspace_bytes);
  if (st != ATTN_OK) return st;
  plan_tail_split(&main, workspace, workspace_bytes);
  PreSetup pre;
  st = setup_preprocess(&pre, o, so, dO, sdo, lse, slse, B, S, HQ, D, D, 0, dtype, workspace, workspace_bytes);
  if (st != ATTN_OK) return st;
  LandSetup land;
  st = setup_dq_land(&land, dq, sdq, B, S, HQ, D, dtype, sm_scale, workspace, workspace_bytes);
  if (st != ATTN_OK) return st;
  if ((st = run_preprocess(pre, stream)) != ATTN_OK) return st;
  if ((st = run_dense(main, stream)) != ATTN_OK) return st;
  return run_land(land, stream);
}

attn_status_t attn_fwd_gqa(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk, const void* v,
                           attn_strides_t sv, int64_t B, int64_t S, int64_t HQ, int64_t HKV, int64_t D,
                           attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask, void* o, attn_strides_t so,
                           float* lse, attn_strides_t slse, void* workspace, size_t workspace_bytes, void* stream) {
  FwdSetup f;
  const attn_status_t st = setup_fwd(&f, q, sq, k, sk, v, sv, B, S, HQ, HKV, D, dtype, sm_scale, mask, o, so, lse,
                                     slse, workspace, workspace_bytes);
  return st != ATTN_OK ? st : run_fwd(f, stream);
}

attn_status_t attn_bwd(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk, const void* v,
                       attn_strides_t sv, const void* o, attn_strides_t so, const void* dO, attn_strides_t sdo,
                       const float* lse, attn_strides_t slse, int64_t B, int64_t S, int64_t H, int64_t D,
                       attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask, void* dq, attn_strides_t sdq,
                       void* dk, attn_strides_t sdk, void* dv, attn_strides_t sdv, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return attn_bwd_gqa(q, sq, k, sk, v, sv, o, so, dO, sdo, lse, slse, B, S, H, H, D, dtype, sm_scale, mask, dq, sdq,
                      dk, sdk, dv, sdv, workspace, workspace_bytes, stream);
}

attn_status_t attn_bwd_sparse_main(const void* q, attn_strides_t sq, const void* kv, attn_strides_t skv,
                                   const void* dO, attn_strides_t sdo, const int32_t* idx, attn_strides_t sidx,
                                   int64_t B, int64_t S, int64_t SKV, int64_t H, int64_t HKV, int64_t DQK, int64_t DV,
                                   int64_t topk, attn_dtype_t dtype, float sm_scale, void* dq, attn_strides_t sdq,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  SparseSetup s;
  const attn_status_t st = setup_sparse(&s, q, sq, kv, skv, dO, sdo, idx, sidx, B, S, SKV, H, HKV, DQK, DV, topk,
                                        dtype, sm_scale, dq, sdq, workspace, workspace_bytes);
  return st != ATTN_OK ? st : run_sparse(s, stream);
}

attn_status_t attn_bwd_sparse_land(void* dkv, attn_strides_t sdkv, int64_t B, int64_t S, int64_t SKV, int64_t H,
                                   int64_t HKV, int64_t DQK, attn_dtype_t dtype, const void* workspace,
                                   size_t workspace_bytes, void* stream) {
  LandSetup s;
  const attn_status_t st =
      setup_sparse_land(&s, dkv, sdkv, B, S, SKV, H, HKV, DQK, dtype, workspace, workspace_bytes);
  return st != ATTN_OK ? st : run_land(s, stream);
}

attn_status_t attn_bwd_sparse(const void* q, attn_strides_t sq, const void* kv, attn_strides_t skv, const void* o,
                              attn_strides_t so, const void* dO, attn_strides_t sdo, const float* lse,
                              attn_strides_t slse, const int32_t* idx, attn_strides_t sidx, int64_t B, int64_t S,
                              int64_t SKV, int64_t H, int64_t HKV, int64_t DQK, int64_t DV, int64_t topk,
                              attn_dtype_t dtype, float sm_scale, void* dq, attn_strides_t sdq, void* dkv,
                              attn_strides_t sdkv, void* workspace, size_t workspace_bytes, void* stream) {
  SparseSetup main;
  attn_status_t st = setup_sparse(&main, q, sq, kv, skv, dO, sdo, idx, sidx, B, S, SKV, H, HKV, DQK, DV, topk, dtype,
                                  sm_scale, dq, sdq, workspace, workspace_bytes);
  if (st != ATTN_OK) return st;
  const int64_t dkv_elems = B * SKV * HKV * DQK;
  PreSetup pre;
  st = setup_preprocess(&pre, o, so, dO, sdo, lse, slse, B, S, H, DV, 0, dkv_elems, dtype, workspace,
                        workspace_bytes);
  if (st != ATTN_OK) return st;
  LandSetup land;
  st = setup_sparse_land(&land, dkv, sdkv, B, S, SKV, H, HKV, DQK, dtype, workspace, workspace_bytes);
  if (st != ATTN_OK) return st;
  if ((st = run_preprocess(pre, stream)) != ATTN_OK) return st;
  if ((st = run_sparse(main, stream)) != ATTN_OK) return st;
  return run_land(land, stream);
}

attn_status_t attn_bwd_sink_grad(const float* sink, int64_t B, int64_t S, int64_t HQ, const attn_mask_t* mask,
                                 const void* workspace, size_t workspace_bytes, float* dsink, void* stream) {
  if (!sink || !dsink || !workspace) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || HQ < 1) return ATTN_ERR_INVALID_ARG;
  if (B * S * HQ >= (int64_t(1) << 31) || HQ > 65535) return ATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(sink) & 3u) || (reinterpret_cast<uintptr_t>(dsink) & 3u) || !aligned16(workspace))
    return ATTN_ERR_INVALID_ARG;
  MaskArgs ma;
  if (const attn_status_t mst = parse_mask(mask, B, S, &ma); mst != ATTN_OK) return mst;
  const WsLayout L = ws_layout(B, S, HQ, 0, 0);
  if (workspace_bytes < static_cast<size_t>(L.dq_off)) return ATTN_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  SinkGradParams p{};
  p.sink = sink;
  p.lse2 = reinterpret_cast<const float*>(ws + L.lse2_off);
  p.delta = reinterpret_cast<const float*>(ws + L.delta_off);
  p.B = static_cast<int>(B), p.S = static_cast<int>(S), p.H = static_cast<int>(HQ);
  p.cu_seqlens = ma.cu, p.num_seqs = ma.num_seqs;
  p.dsink = dsink;
  return launch_status(launch_sink_grad(p, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_bwd_check_error(const void* workspace, void* stream, int32_t* device_code) {
  if (device_code) *device_code = 0;
  if (!workspace) return ATTN_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_DEVICE;
  WsHeader h;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_DEVICE;
  if (device_code) *device_code = h.err;
  return h.err == 0 ? ATTN_OK : ATTN_ERR_TIMEOUT;
}

attn_status_t attn_bwd_selftest_timeout(void* workspace, size_t workspace_bytes, int32_t timeout_us, void* stream) {
  if (!workspace || workspace_bytes < static_cast<size_t>(kHeaderBytes) || timeout_us < 1 || timeout_us > 10000000)
    return ATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, kHeaderBytes, st) != cudaSuccess) return ATTN_ERR_LAUNCH;
  if (launch_selftest_timeout(&static_cast<WsHeader*>(workspace)->err, static_cast<uint64_t>(timeout_us) * 1000ull,
                              st) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  return attn_bwd_check_error(workspace, stream, nullptr);
}

}  // extern "C"
