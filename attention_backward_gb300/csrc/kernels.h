// Parameter blocks and launchers of the kernels (internal to the library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_bwd.h"
#include "common.cuh"

namespace ab {

struct PreprocessParams {
  const uint8_t* o;
  int64_t so_b, so_s, so_h;  // element strides
  const uint8_t* dO;
  int64_t sdo_b, sdo_s, sdo_h;
  const float* lse;
  int64_t sl_b, sl_s, sl_h;
  int B, S, H, Dv;
  float* lse2;   // [B,H,S]
  float* delta;  // [B,H,S]
  float4* dq_zero;     // f32 dQ accumulator [B,S,H,Dq], cleared row by row with delta
  int dq_row_n4;       // float4 per accumulator row (Dq / 4; 0 without one)
  float4* zero;        // other accumulators to clear (the sparse dKV accumulator)
  int64_t zero_n4;
  WsHeader* hdr;
};

struct LandParams {
  const float* acc;  // [rows = B*S*H][D] f32
  int64_t rows;
  int B, S, H, D;
  uint8_t* out;  // 16-bit BSHD
  int64_t s_b, s_s, s_h;
  float scale;
};

struct DenseParams {
  int B, S, HQ, HKV, G, D;
  int Sk;  // key/value rows per batch row (S unless a dense row has more or fewer keys than queries)
  int causal, window;
  const int* cu_seqlens;
  int num_seqs;
  float scale_log2;  // sm_scale * log2(e)
  float sm_scale;
  const float* lse2;   // [B,HQ,S]
  const float* delta;  // [B,HQ,S]
  float* dq_acc;       // [B,S,HQ,D]
  int* err;
  uint8_t* dk;
  int64_t sdk_b, sdk_s, sdk_h;
  uint8_t* dv;
  int64_t sdv_b, sdv_s, sdv_h;
  uint64_t timeout_ns;
  int* tile_counter;  // zeroed by the preprocess; persistent CTAs draw tiles from it
  int bn;             // query rows per step (the tile schedule's query block)
  int tile_group;     // (batch, KV head) pairs drawn together, dense batches (tile_group())
  // Last-round split (head dim 128, dense batches): the tile draws from
  // tail_start on cover the last tail_tiles key tiles, each as G / tail_hpu
  // units of tail_hpu query heads; a unit adds its dK/dV partial into
  // part_acc in f32, and the last unit of each 32-row quarter of a tile
  // casts it.  tail_tiles = 0: every tile is drawn whole.
  int tail_start, tail_tiles, tail_hpu;
  int* part_count;  // [tail_tiles][4] units done per row quarter (zeroed by the preprocess)
  float* part_acc;  // [tail_tiles][2 D / 4][128 rows][4] f32, dV columns then dK (zeroed by the preprocess)
};

struct DenseMaps {
  CUtensorMap q, k, v, dO;
  CUtensorMap dq;  // f32 dQ accumulator [B,S,HQ,D] (bulk reduce-add target)
};

// The dense forward (dense_fwd.cu): O and the natural-log LSE.
struct FwdParams {
  int B, S, Sk, HQ, HKV, G, D;
  int causal, window;
  const int* cu_seqlens;
  int num_seqs;
  float scale_log2;  // sm_scale * log2(e), > 0
  uint8_t* o;        // 16-bit [B,S,HQ,D]
  int64_t so_b, so_s, so_h;
  float* lse;  // f32, lse[b*sl_b + h*sl_h + s*sl_s]
  int64_t sl_b, sl_s, sl_h;
  int* err;
  int* unit_counter;  // cleared before the launch; persistent CTAs draw units from it
  uint64_t timeout_ns;
};

struct FwdMaps {
  CUtensorMap q, k, v;  // box 64 d x 128 rows of one head
};

cudaError_t launch_fwd(const FwdParams& p, const FwdMaps& m, bool bf16, int grid, cudaStream_t st);

struct SparseParams {
  int B, S, SKV, H, HKV, topk;
  int gh;            // query heads per KV group (at most 64; a unit pads them to 64)
  float scale_log2;  // sm_scale * log2(e)
  float sm_scale;
  const float* lse2;   // [B,H,S]
  const float* delta;  // [B,H,S]
  float* dkv_acc;      // f32 [B,SKV,HKV,576]
  const int* idx;      // [B,S,HKV,topk]
  int64_t si_b, si_s, si_h;
  uint8_t* dq;  // 16-bit [B,S,H,576]
  int64_t sdq_b, sdq_s, sdq_h;
  int* err;
  int* unit_counter;
  uint64_t timeout_ns;
};

struct SparseMaps {
  CUtensorMap q;   // [B,S,H,576], box 64 d x 64 heads
  CUtensorMap dO;  // [B,S,H,512], box 64 d x 64 heads
  CUtensorMap kv;  // 2-D rows (b*SKV + j)*HKV + g of 576, box 64 x 1 (gather4)
};

cudaError_t launch_sparse(const SparseParams& p, const SparseMaps& m, bool bf16, int grid, cudaStream_t st);

cudaError_t launch_preprocess(const PreprocessParams& p, bool bf16, int grid, cudaStream_t st);
cudaError_t launch_land(const LandParams& p, bool bf16, int grid, cudaStream_t st);
cudaError_t launch_dense(const DenseParams& p, const DenseMaps& m, bool bf16, int grid, cudaStream_t st);
// Head dim 128 (dense128_bwd.cu); launch_dense forwards launches with
// p.D == 128 here and runs head dim 64 itself (dense_bwd.cu).
cudaError_t launch_dense128(const DenseParams& p, const DenseMaps& m, bool bf16, int grid, cudaStream_t st);
cudaError_t launch_selftest_timeout(int* err, uint64_t timeout_ns, cudaStream_t st);

// Every argument check of attn_bwd_gqa (api.cu), with no device or driver call.
attn_status_t check_gqa_call(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk, const void* v,
                             attn_strides_t sv, const void* o, attn_strides_t so, const void* dO, attn_strides_t sdo,
                             const float* lse, attn_strides_t slse, int64_t B, int64_t S, int64_t HQ, int64_t HKV,
                             int64_t D, attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask, void* dq,
                             attn_strides_t sdq, void* dk, attn_strides_t sdk, void* dv, attn_strides_t sdv,
                             void* workspace, size_t workspace_bytes);

// Launches ``kern`` with programmatic stream serialization: it may be scheduled
// while the previous kernel on ``st`` finishes, and waits for it with
// grid_dependency_wait before reading its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_after_previous(void (*kern)(KArgs...), int grid, int threads, int smem, cudaStream_t st,
                                  Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Block sizes of both dense kernels: keys per tile, and queries per step
// (every MMA at N = 128; 64-query steps with a double-buffered S^T measured
// slower at head dim 128 on both the causal and the unmasked workloads).
constexpr int kDenseBM = 128;
constexpr int kDenseBN = 128;

}  // namespace ab
