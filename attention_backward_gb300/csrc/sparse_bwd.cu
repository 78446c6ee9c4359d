// Top-k sparse (shared latent K/V) backward: not yet served.
#include "attn_bwd.h"

extern "C" {

attn_status_t attn_bwd_sparse(const void*, attn_strides_t, const void*, attn_strides_t, const void*, attn_strides_t,
                              const int32_t*, attn_strides_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t,
                              int64_t, int64_t, attn_dtype_t, float, void*, size_t, void*) {
  return ATTN_ERR_UNSUPPORTED;
}

attn_status_t attn_bwd_sparse_land(void*, attn_strides_t, void*, attn_strides_t, int64_t, int64_t, int64_t, int64_t,
                                   int64_t, int64_t, attn_dtype_t, const void*, size_t, void*) {
  return ATTN_ERR_UNSUPPORTED;
}

}  // extern "C"
