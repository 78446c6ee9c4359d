// attn_bwd_gqa_host: the dense backward from host buffers to host buffers,
// with the host<->device copies overlapped with the kernels.
//
// The problem splits into independent chunks of batch rows and KV heads (a
// batch row's KV head and its G query heads need nothing from the other rows
// and heads: dK and dV are owned per KV head, dQ and delta per query head).
// With at least as many chunks as batch rows, a chunk is one batch row and a
// range of its KV heads; with fewer, a chunk is a range of whole batch rows.
// Chunk i goes through three streams:
//
//   copy-in   strided head slices of q, k, v, o, dO, LSE -> contiguous chunk buffers
//   compute   attn_bwd_gqa (preprocess, main kernel, dQ landing) on the chunk
//   copy-out  contiguous dQ, dK, dV of the chunk -> strided host slices
//
// with two buffer slots, so that the copy-in of chunk i+1 and the copy-out of
// chunk i-1 run while chunk i computes.  Host buffers should be page-locked;
// with pageable memory the copies are correct but do not overlap.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <vector>

#include "attn_bwd.h"

namespace {

int64_t round_up(int64_t x) { return (x + 255) / 256 * 256; }

// Device scratch: the workspace of one chunk at offset 0 (so that
// attn_bwd_check_error can read the scratch pointer), then two slots of chunk
// buffers.
struct HostLayout {
  int64_t bc, hc, nb, nh, nchunks;                        // batch rows and KV heads per chunk, their counts
  int64_t q, k, v, o, dO, lse, dq, dk, dv, slot;          // offsets inside a slot, slot bytes
  int64_t ws_bytes, slot0, total;
};

HostLayout host_layout(int64_t B, int64_t S, int64_t HQ, int64_t HKV, int64_t D, int64_t chunks) {
  HostLayout L{};
  if (chunks >= B) {  // one batch row per chunk, its KV heads in chunks / B ranges
    L.bc = 1;
    const int64_t per_row = chunks / B;
    L.hc = (HKV + per_row - 1) / per_row;
  } else {  // whole batch rows, all heads
    L.bc = (B + chunks - 1) / chunks;
    L.hc = HKV;
  }
  L.nb = (B + L.bc - 1) / L.bc;
  L.nh = (HKV + L.hc - 1) / L.hc;
  L.nchunks = L.nb * L.nh;
  const int64_t G = HQ / HKV, hq = L.hc * G, Bc = L.bc;
  const int64_t qb = round_up(Bc * S * hq * D * 2), kb = round_up(Bc * S * L.hc * D * 2), lb = round_up(Bc * hq * S * 4);
  int64_t off = 0;
  L.q = off, off += qb;
  L.k = off, off += kb;
  L.v = off, off += kb;
  L.o = off, off += qb;
  L.dO = off, off += qb;
  L.lse = off, off += lb;
  L.dq = off, off += qb;
  L.dk = off, off += kb;
  L.dv = off, off += kb;
  L.slot = off;
  L.ws_bytes = round_up(static_cast<int64_t>(attn_bwd_workspace_size(Bc, S, hq, D, 0)));
  L.slot0 = L.ws_bytes;
  L.total = L.slot0 + 2 * L.slot;
  return L;
}

bool shape_ok(int64_t B, int64_t S, int64_t HQ, int64_t HKV, int64_t D, int64_t chunks) {
  return B >= 1 && S >= 1 && HQ >= 1 && HKV >= 1 && HQ % HKV == 0 && chunks >= 1 && (D == 64 || D == 128);
}

}  // namespace

extern "C" size_t attn_bwd_host_scratch_size(int64_t B, int64_t S, int64_t HQ, int64_t HKV, int64_t D,
                                             int64_t chunks) {
  if (!shape_ok(B, S, HQ, HKV, D, chunks)) return 0;
  return static_cast<size_t>(host_layout(B, S, HQ, HKV, D, chunks).total);
}

extern "C" attn_status_t attn_bwd_gqa_host(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                           const float* lse, int64_t B, int64_t S, int64_t HQ, int64_t HKV, int64_t D,
                                           attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask, void* dq,
                                           void* dk, void* dv, void* scratch, size_t scratch_bytes, int64_t chunks,
                                           void* stream, void* copy_in_stream, void* copy_out_stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || !scratch) return ATTN_ERR_INVALID_ARG;
  if (!shape_ok(B, S, HQ, HKV, D, chunks)) return D == 64 || D == 128 ? ATTN_ERR_INVALID_ARG : ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_DT_F16 && dtype != ATTN_DT_BF16) return ATTN_ERR_UNSUPPORTED;
  if (HQ / HKV > (dtype == ATTN_DT_BF16 ? ATTN_BWD_MAX_GROUP_BF16 : ATTN_BWD_MAX_GROUP_F16)) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(sm_scale)) return ATTN_ERR_INVALID_ARG;
  // chunks copy K/V as [B,S,HKV,D]: key rows of another length are not served here
  if (mask && (mask->window_left == 0 || mask->window_left < -1 ||
               (mask->cu_seqlens && (B != 1 || mask->num_seqs < 1 || mask->num_seqs > (1 << 20))) ||
               (mask->kv_len != 0 && mask->kv_len != S)))
    return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scratch) & 255u) != 0) return ATTN_ERR_INVALID_ARG;
  const HostLayout L = host_layout(B, S, HQ, HKV, D, chunks);
  if (scratch_bytes < static_cast<size_t>(L.total)) return ATTN_ERR_WORKSPACE;
  cudaStream_t sc = static_cast<cudaStream_t>(stream), si = static_cast<cudaStream_t>(copy_in_stream),
               so = static_cast<cudaStream_t>(copy_out_stream);
  const int64_t G = HQ / HKV, n = L.nchunks;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  uint8_t* ws = base;

  // events: start (orders the copies after earlier work on ``stream``), and per chunk
  std::vector<cudaEvent_t> ev(3 * n + 1, nullptr);
  attn_status_t st = ATTN_OK;
  for (auto& e : ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) st = ATTN_ERR_DEVICE;
  cudaEvent_t start = ev[0];
  auto copied_in = [&](int64_t i) { return ev[1 + i]; };
  auto computed = [&](int64_t i) { return ev[1 + n + i]; };
  auto copied_out = [&](int64_t i) { return ev[1 + 2 * n + i]; };
  auto ok = [&](cudaError_t e) {
    if (e != cudaSuccess && st == ATTN_OK) st = ATTN_ERR_DEVICE;
    return st == ATTN_OK;
  };
  if (st == ATTN_OK) ok(cudaEventRecord(start, sc));
  if (st == ATTN_OK) ok(cudaStreamWaitEvent(si, start, 0));

  const int64_t e16 = 2;  // bytes of a 16-bit element
  for (int64_t i = 0; i < n && st == ATTN_OK; ++i) {
    uint8_t* slot = base + L.slot0 + (i % 2) * L.slot;
    // chunk i: batch rows [b0, b0 + bn), KV heads [hk0, hk0 + hkn) (heads fastest)
    const int64_t b0 = (i / L.nh) * L.bc, bn = (b0 + L.bc <= B ? L.bc : B - b0);
    const int64_t hk0 = (i % L.nh) * L.hc, hkn = (hk0 + L.hc <= HKV ? L.hc : HKV - hk0), hq0 = hk0 * G, hqn = hkn * G;
    const size_t rows = static_cast<size_t>(bn * S);  // (b, s) rows of the chunk, consecutive on the host
    // ---- copy-in: the slot is free once the copy-out of chunk i-2 is done
    if (i >= 2 && !ok(cudaStreamWaitEvent(si, copied_out(i - 2), 0))) break;
    auto in_q = [&](int64_t off, const void* src) {  // a [B,S,HQ,D] slice
      return cudaMemcpy2DAsync(slot + off, hqn * D * e16,
                               static_cast<const uint8_t*>(src) + (b0 * S * HQ + hq0) * D * e16, HQ * D * e16,
                               hqn * D * e16, rows, cudaMemcpyHostToDevice, si);
    };
    auto in_k = [&](int64_t off, const void* src) {  // a [B,S,HKV,D] slice
      return cudaMemcpy2DAsync(slot + off, hkn * D * e16,
                               static_cast<const uint8_t*>(src) + (b0 * S * HKV + hk0) * D * e16, HKV * D * e16,
                               hkn * D * e16, rows, cudaMemcpyHostToDevice, si);
    };
    if (!ok(in_q(L.q, q)) || !ok(in_k(L.k, k)) || !ok(in_k(L.v, v)) || !ok(in_q(L.o, o)) || !ok(in_q(L.dO, dO)))
      break;
    if (!ok(cudaMemcpy2DAsync(slot + L.lse, hqn * S * 4, lse + (b0 * HQ + hq0) * S, HQ * S * 4, hqn * S * 4,
                              static_cast<size_t>(bn), cudaMemcpyHostToDevice, si)))
      break;
    if (!ok(cudaEventRecord(copied_in(i), si))) break;
    // ---- compute on the contiguous chunk
    if (!ok(cudaStreamWaitEvent(sc, copied_in(i), 0))) break;
    const attn_strides_t sqo{S * hqn * D, hqn * D, D}, skv{S * hkn * D, hkn * D, D}, sl{hqn * S, 1, S};
    st = attn_bwd_gqa(slot + L.q, sqo, slot + L.k, skv, slot + L.v, skv, slot + L.o, sqo, slot + L.dO, sqo,
                      reinterpret_cast<const float*>(slot + L.lse), sl, bn, S, hqn, hkn, D, dtype, sm_scale, mask,
                      slot + L.dq, sqo, slot + L.dk, skv, slot + L.dv, skv, ws, L.ws_bytes, sc);
    if (st != ATTN_OK || !ok(cudaEventRecord(computed(i), sc))) break;
    // ---- copy-out
    if (!ok(cudaStreamWaitEvent(so, computed(i), 0))) break;
    auto out_q = [&](void* dst, int64_t off) {
      return cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + (b0 * S * HQ + hq0) * D * e16, HQ * D * e16, slot + off,
                               hqn * D * e16, hqn * D * e16, rows, cudaMemcpyDeviceToHost, so);
    };
    auto out_k = [&](void* dst, int64_t off) {
      return cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + (b0 * S * HKV + hk0) * D * e16, HKV * D * e16,
                               slot + off, hkn * D * e16, hkn * D * e16, rows, cudaMemcpyDeviceToHost, so);
    };
    if (!ok(out_q(dq, L.dq)) || !ok(out_k(dk, L.dk)) || !ok(out_k(dv, L.dv))) break;
    if (!ok(cudaEventRecord(copied_out(i), so))) break;
  }
  // ``stream`` covers the whole call: it waits for the last copy-out (the
  // copy-outs are ordered on their stream)
  if (st == ATTN_OK) ok(cudaStreamWaitEvent(sc, copied_out(n - 1), 0));
  for (auto& e : ev)
    if (e) cudaEventDestroy(e);  // released once pending work that uses it completes
  return st;
}
