// attn_bwd_gqa_noalloc: the whole dense backward (preprocess, main kernel, dQ
// landing) without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they need the
// gradients: plugins hosted by a framework that owns every byte of device
// memory through its own pool (a private cudaMalloc would bypass the pool's
// budget and synchronise the device), and latency-critical loops where the
// implicit device-wide synchronisation of cudaMalloc/cudaFree is not
// acceptable.  For them this file holds the workspace itself: one file-scope
// device array of kNoAllocScratchBytes, which every GPU that loads the library
// keeps until the process exits.  Problems whose workspace
// (attn_bwd_workspace_size(B, S, HQ, D, 0)) does not fit are rejected.
//
// The array's name in host code is only a host-side stand-in for the device
// symbol, so the device address is looked up with cudaGetSymbolAddress, once
// per device, with that device current, on the first call made on it, and
// kept for the life of the process (a device reset would make it stale).
// Errors that the kernels record (a bounded wait that ran out) land in the
// array's workspace header; attn_bwd_noalloc_check_error reads them back.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "attn_bwd.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = ATTN_BWD_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size");

// The shared workspace of every attn_bwd_gqa_noalloc call on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.
attn_status_t scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_DEVICE;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_bwd_gqa_noalloc(const void* q, attn_strides_t sq, const void* k, attn_strides_t sk,
                                              const void* v, attn_strides_t sv, const void* o, attn_strides_t so,
                                              const void* dO, attn_strides_t sdo, const float* lse,
                                              attn_strides_t slse, int64_t B, int64_t S, int64_t HQ, int64_t HKV,
                                              int64_t D, attn_dtype_t dtype, float sm_scale, const attn_mask_t* mask,
                                              void* dq, attn_strides_t sdq, void* dk, attn_strides_t sdk, void* dv,
                                              attn_strides_t sdv, void* stream) {
  // Every argument, the size limit included, is checked before the device is
  // touched; the aligned placeholder stands in for the array's address, which
  // the checks never dereference.
  if (B < 1 || S < 1 || HQ < 1 || HKV < 1 || HQ % HKV != 0) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  const size_t need = attn_bwd_workspace_size(B, S, HQ, D, 0);
  if (need == 0 || need > kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
  attn_status_t st = ab::check_gqa_call(q, sq, k, sk, v, sv, o, so, dO, sdo, lse, slse, B, S, HQ, HKV, D, dtype,
                                        sm_scale, mask, dq, sdq, dk, sdk, dv, sdv, reinterpret_cast<void*>(256),
                                        kNoAllocScratchBytes);
  if (st != ATTN_OK) return st;
  void* ws = nullptr;
  st = scratch_on_current_device(&ws);
  if (st != ATTN_OK) return st;
  // The preprocess clears the error word, the tile counter and the dQ
  // accumulator, so the contents a previous call left behind do not matter.
  return attn_bwd_gqa(q, sq, k, sk, v, sv, o, so, dO, sdo, lse, slse, B, S, HQ, HKV, D, dtype, sm_scale, mask, dq,
                      sdq, dk, sdk, dv, sdv, ws, kNoAllocScratchBytes, stream);
}

extern "C" attn_status_t attn_bwd_noalloc_check_error(void* stream, int32_t* device_code) {
  if (device_code) *device_code = 0;
  void* ws = nullptr;
  const attn_status_t st = scratch_on_current_device(&ws);
  if (st != ATTN_OK) return st;
  // the array starts with a workspace header, whose error word the kernels set
  return attn_bwd_check_error(ws, stream, device_code);
}
