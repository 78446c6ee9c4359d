// Launch 1 (preprocess) and launch 3 (landing) of the backward.
//
// Preprocess: delta_i = sum_d O_id dO_id in f32 (the delta row preprocess of
// the TileOPs MHA backward page, "delta_rows"), LSE2 = LSE * log2(e) so that
// the main kernel evaluates P with one FFMA and one exp2, zeroed f32
// accumulators (the dQ accumulator row by row next to the delta of the same
// row), cleared workspace header.  HBM-bound: 16-byte loads and stores, grid
// a multiple of the SM count.
//
// Landing: out = cast(scale * acc) from an f32 accumulator laid out
// [B,S,H,D] into a strided 16-bit BSHD tensor (the page's "dq_land").
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "cvt.cuh"
#include "kernels.h"

namespace ab {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = unpack2<BF16>(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(256) preprocess_kernel(PreprocessParams p) {
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (gtid == 0) {
    p.hdr->err = 0;
    p.hdr->tile_counter = 0;
  }
  for (int64_t i = gtid; i < p.zero_n4; i += nthr) p.zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);

  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.S;
  for (int64_t r = gtid; r < rows; r += nthr) {
    const int64_t s = r % p.S, h = (r / p.S) % p.H, b = r / (static_cast<int64_t>(p.S) * p.H);
    p.lse2[r] = p.lse[b * p.sl_b + h * p.sl_h + s * p.sl_s] * kLog2e;
  }

  // delta: a group of ``gs`` lanes per (b, s, h) row, rows ordered (b, s, h)
  // so that consecutive groups read consecutive memory.
  const int chunks = p.Dv / 8;
  int gs = 1;
  while (gs * 2 <= chunks && gs * 2 <= 32) gs *= 2;
  const int lane = threadIdx.x & 31;
  const int64_t warp = gtid >> 5, nwarps = nthr >> 5;
  const int rows_per_warp = 32 / gs;
  const int sub = lane / gs, lig = lane % gs;
  for (int64_t base = warp * rows_per_warp; base < rows; base += nwarps * rows_per_warp) {
    const int64_t r = base + sub;
    float acc = 0.f;
    int64_t b = 0, s = 0, h = 0;
    if (r < rows) {
      h = r % p.H;
      s = (r / p.H) % p.S;
      b = r / (static_cast<int64_t>(p.H) * p.S);
      // the row's dQ accumulator (same (b, s, h) order), so that its writes
      // overlap the O/dO reads
      float4* z = p.dq_zero + r * p.dq_row_n4;
      for (int k = lig; k < p.dq_row_n4; k += gs) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      const uint4* o = reinterpret_cast<const uint4*>(p.o + 2 * (b * p.so_b + s * p.so_s + h * p.so_h));
      const uint4* d = reinterpret_cast<const uint4*>(p.dO + 2 * (b * p.sdo_b + s * p.sdo_s + h * p.sdo_h));
      for (int c = lig; c < chunks; c += gs) {
        float fo[8], fd[8];
        unpack8<BF16>(__ldg(o + c), fo);
        unpack8<BF16>(__ldg(d + c), fd);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(fo[e], fd[e], acc);
      }
    }
    for (int off = gs / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (r < rows && lig == 0) p.delta[(b * p.H + h) * p.S + s] = acc;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(256) land_kernel(LandParams p) {
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int cpr = p.D / 8;  // 8-element chunks per row
  const int64_t n = p.rows * cpr;
  for (int64_t i = gtid; i < n; i += nthr) {
    const int64_t row = i / cpr;
    const int c = static_cast<int>(i % cpr);
    const int64_t h = row % p.H, s = (row / p.H) % p.S, b = row / (static_cast<int64_t>(p.H) * p.S);
    const float4* a = reinterpret_cast<const float4*>(p.acc + row * p.D + c * 8);
    const float4 x = a[0], y = a[1];
    uint4 o;
    o.x = pack2<BF16>(x.x * p.scale, x.y * p.scale);
    o.y = pack2<BF16>(x.z * p.scale, x.w * p.scale);
    o.z = pack2<BF16>(y.x * p.scale, y.y * p.scale);
    o.w = pack2<BF16>(y.z * p.scale, y.w * p.scale);
    *reinterpret_cast<uint4*>(p.out + 2 * (b * p.s_b + s * p.s_s + h * p.s_h + c * 8)) = o;
  }
}

}  // namespace

cudaError_t launch_preprocess(const PreprocessParams& p, bool bf16, int grid, cudaStream_t st) {
  if (bf16)
    preprocess_kernel<true><<<grid, 256, 0, st>>>(p);
  else
    preprocess_kernel<false><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_land(const LandParams& p, bool bf16, int grid, cudaStream_t st) {
  if (bf16)
    land_kernel<true><<<grid, 256, 0, st>>>(p);
  else
    land_kernel<false><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace ab
