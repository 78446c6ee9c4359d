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
#include "sink.h"
#include "sm103.cuh"

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

// Lanes per row (a power of two, at most 32) for rows of ``chunks`` 16-byte
// chunks; a warp covers 32 / lanes rows at a time.
__device__ __forceinline__ int lanes_per_row(int chunks) {
  int g = 1;
  while (g * 2 <= chunks && g * 2 <= 32) g *= 2;
  return g;
}

// Rows of each lane group handled per loop iteration: their loads are all
// issued before any of them is used, so that enough bytes are in flight to
// cover the memory latency.  Measured on the causal MHA 2x2048x32x128 step:
// the preprocess is fastest with 2 (26.4 us against 29.5 with 4 and 37 with
// 8: with more rows per iteration fewer warps share the work), the landing
// with 4 (19.5 us against 20.7 with 2).
constexpr int kPreRowsInFlight = 2;
constexpr int kLandRowsInFlight = 4;

template <bool BF16>
__global__ void __launch_bounds__(256) preprocess_kernel(PreprocessParams p) {
  // the main kernel may be scheduled as soon as every block of this one runs
  // (it waits for this kernel's completion before reading its results)
  grid_dependents_launch();
  // grid x block < 2^31 and B*H*S < 2^31 (checked on the host): 32-bit indices
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthr = gridDim.x * blockDim.x;
  if (gtid == 0) {
    p.hdr->err = 0;
    p.hdr->tile_counter = 0;
  }
  for (int64_t i = gtid; i < p.zero_n4; i += nthr) p.zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);

  const int rows = p.B * p.H * p.S;
  for (int r = gtid; r < rows; r += nthr) {
    const int s = r % p.S, t = r / p.S, h = t % p.H, b = t / p.H;
    p.lse2[r] = p.lse[b * p.sl_b + h * p.sl_h + s * p.sl_s] * kLog2e;
  }

  // delta: a group of ``gs`` lanes per (b, s, h) row, rows ordered (b, s, h)
  // so that consecutive groups read consecutive memory.
  constexpr int U = kPreRowsInFlight;
  const int chunks = p.Dv / 8;
  const int gs = lanes_per_row(chunks);
  const int lane = threadIdx.x & 31;
  const int warp = gtid >> 5, nwarps = nthr >> 5;
  const int rows_per_warp = 32 / gs;
  const int sub = lane / gs, lig = lane % gs;
  const int span = rows_per_warp * U;
  for (int base = warp * span; base < rows; base += nwarps * span) {
    const uint4* op[U];
    const uint4* dp[U];
    int64_t di[U];
    float acc[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int r = base + k * rows_per_warp + sub;
      acc[k] = 0.f;
      op[k] = dp[k] = nullptr;
      di[k] = -1;
      if (r < rows) {
        const int h = r % p.H, t = r / p.H, s = t % p.S, b = t / p.S;
        op[k] = reinterpret_cast<const uint4*>(p.o + 2 * (b * p.so_b + s * p.so_s + h * p.so_h));
        dp[k] = reinterpret_cast<const uint4*>(p.dO + 2 * (b * p.sdo_b + s * p.sdo_s + h * p.sdo_h));
        di[k] = (static_cast<int64_t>(b) * p.H + h) * p.S + s;
      }
    }
    for (int c = lig; c < chunks; c += gs) {
      uint4 ou[U], du[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        ou[k] = du[k] = make_uint4(0u, 0u, 0u, 0u);
        if (op[k] != nullptr) {
          ou[k] = __ldg(op[k] + c);
          du[k] = __ldg(dp[k] + c);
        }
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        float fo[8], fd[8];
        unpack8<BF16>(ou[k], fo);
        unpack8<BF16>(du[k], fd);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[k] = fmaf(fo[e], fd[e], acc[k]);
      }
    }
    // the rows' dQ accumulators (same (b, s, h) order); their writes overlap
    // the O/dO reads of the next iteration
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int r = base + k * rows_per_warp + sub;
      if (r < rows) {
        float4* z = p.dq_zero + static_cast<int64_t>(r) * p.dq_row_n4;
        for (int q = lig; q < p.dq_row_n4; q += gs) z[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      for (int off = gs / 2; off > 0; off >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
      if (di[k] >= 0 && lig == 0) p.delta[di[k]] = acc[k];
    }
  }
}

template <bool BF16>
__global__ void __launch_bounds__(256) land_kernel(LandParams p) {
  grid_dependency_wait();  // the main kernel's accumulator is complete
  // rows = B*S*H < 2^31 (checked on the host); a group of ``gs`` lanes per row
  constexpr int U = kLandRowsInFlight;
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthr = gridDim.x * blockDim.x;
  const int cpr = p.D / 8;  // 8-element chunks per row
  const int gs = lanes_per_row(cpr);
  const int lane = threadIdx.x & 31;
  const int warp = gtid >> 5, nwarps = nthr >> 5;
  const int rows_per_warp = 32 / gs;
  const int sub = lane / gs, lig = lane % gs;
  const int span = rows_per_warp * U;
  const int rows = static_cast<int>(p.rows);
  for (int base = warp * span; base < rows; base += nwarps * span) {
    for (int c = lig; c < cpr; c += gs) {
      float4 x[U], y[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int r = base + k * rows_per_warp + sub;
        if (r < rows) {
          const float4* a = reinterpret_cast<const float4*>(p.acc + static_cast<int64_t>(r) * p.D + c * 8);
          x[k] = a[0];
          y[k] = a[1];
        }
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int r = base + k * rows_per_warp + sub;
        if (r < rows) {
          const int h = r % p.H, t = r / p.H, s = t % p.S, b = t / p.S;
          uint4 o;
          o.x = pack2<BF16>(x[k].x * p.scale, x[k].y * p.scale);
          o.y = pack2<BF16>(x[k].z * p.scale, x[k].w * p.scale);
          o.z = pack2<BF16>(y[k].x * p.scale, y[k].y * p.scale);
          o.w = pack2<BF16>(y[k].z * p.scale, y[k].w * p.scale);
          *reinterpret_cast<uint4*>(p.out + 2 * (b * p.s_b + s * p.s_s + h * p.s_h + c * 8)) = o;
        }
      }
    }
  }
}

// dsink_h = -sum over the rows of every sequence of exp(sink_h - LSE_i) delta_i:
// one block per head, a fixed order of additions (no atomics), so that the
// result is the same from run to run.  The data is small (8 bytes a row), so
// the block is wide and each thread keeps kSinkRows independent row loads in
// flight.  Rows whose LSE2 is not finite (no visible key and no sink in the
// forward) add nothing.
constexpr int kSinkThreads = 1024, kSinkRows = 4;
__global__ void __launch_bounds__(kSinkThreads) sink_grad_kernel(SinkGradParams p) {
  const int h = blockIdx.x;
  int r0 = 0, r1 = p.S;
  if (p.cu_seqlens != nullptr) {
    r0 = clamp_pos(p.cu_seqlens[0], p.S);
    r1 = clamp_pos(p.cu_seqlens[p.num_seqs], p.S);
  }
  const float s2 = p.sink[h] * kLog2e;
  float acc = 0.f;
  for (int b = 0; b < p.B; ++b) {
    const int64_t base = (static_cast<int64_t>(b) * p.H + h) * p.S;
    for (int r = r0 + static_cast<int>(threadIdx.x); r < r1; r += kSinkThreads * kSinkRows) {
      float l2[kSinkRows], dl[kSinkRows];
#pragma unroll
      for (int k = 0; k < kSinkRows; ++k) {
        const int rr = r + k * kSinkThreads;
        l2[k] = rr < r1 ? p.lse2[base + rr] : -INFINITY;
        dl[k] = rr < r1 ? p.delta[base + rr] : 0.f;
      }
#pragma unroll
      for (int k = 0; k < kSinkRows; ++k)
        if (isfinite(l2[k])) acc = fmaf(exp2f(s2 - l2[k]), dl[k], acc);
    }
  }
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  __shared__ float part[kSinkThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kSinkThreads / 32; ++w) t += part[w];
    p.dsink[h] = -t;
  }
}

}  // namespace

cudaError_t launch_sink_grad(const SinkGradParams& p, cudaStream_t st) {
  sink_grad_kernel<<<p.H, kSinkThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_preprocess(const PreprocessParams& p, bool bf16, int grid, cudaStream_t st) {
  if (bf16)
    preprocess_kernel<true><<<grid, 256, 0, st>>>(p);
  else
    preprocess_kernel<false><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_land(const LandParams& p, bool bf16, int grid, cudaStream_t st) {
  const cudaError_t e = bf16 ? launch_after_previous(land_kernel<true>, grid, 256, 0, st, p)
                             : launch_after_previous(land_kernel<false>, grid, 256, 0, st, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ab
