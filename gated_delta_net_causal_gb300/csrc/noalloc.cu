// gdn_prefill_chunked_static: the chunk-parallel prefill over a scratch
// buffer that the library reserves statically, so that the call itself
// allocates nothing and needs no workspace from the caller. One buffer per
// CUDA context, shared by all calls (see include/gdn.h for the ordering
// rule).
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace {

__device__ __align__(256) unsigned char g_prefill_scratch[GDN_STATIC_SCRATCH_BYTES];

// Device address of the scratch in the current context. Looked up on every
// call (cheap, and it allocates nothing): the address belongs to the module
// as loaded in the current context, so a cached value would go stale after
// cudaDeviceReset or under another context on the same device.
gdn_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess) return GDN_ERR_CUDA;
  *out = p;
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_prefill_chunked_static(
    const gdn_dims* dims, int32_t num_seqs, const int32_t* cu_seqlens, int64_t total_tokens,
    const void* q, int64_t q_stride, const void* k, int64_t k_stride, const void* v,
    int64_t v_stride, const void* a, const void* b, const float* decay_param,
    const float* dt_bias, int32_t flags, float* state, float* core_out, const void* z,
    const float* norm_w, void* out, void* stream) {
  int64_t need = 0;
  gdn_status st = gdn_prefill_workspace_size(dims, num_seqs, total_tokens, flags, &need);
  if (st != GDN_OK) return st;
  if (need > (int64_t)GDN_STATIC_SCRATCH_BYTES) return GDN_ERR_EXTENT;
  void* ws = nullptr;
  if (need > 0) {
    st = scratch_address(&ws);
    if (st != GDN_OK) return st;
  }
  return gdn_prefill_chunked(dims, num_seqs, cu_seqlens, total_tokens, q, q_stride, k, k_stride,
                             v, v_stride, a, b, decay_param, dt_bias, flags, state, core_out, z,
                             norm_w, out, ws, need, stream);
}
