// Host-side interface between the C ABI (abi.cu) and the kernel translation
// units. Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

struct DecodeArgs {
  const void* mixed_qkv;
  const void* a;
  const void* b;
  const float* decay_param;
  const float* dt_bias;
  const void* conv_w;
  void* conv_state;
  float* state;
  float* core_out;
  const void* z;
  const float* norm_w;
  void* out;
  // state-slot table: batch row b reads and writes state[slots[b]] and
  // conv_state[slots[b]] (slots == nullptr: slot b); num_slots bounds it
  const int32_t* slots;
  int32_t num_slots;
  // tokens per sequence (the multi-token kernel; the one-token kernel takes 1):
  // activations [B][tokens][...], outputs [B][tokens][Hv][D]
  int32_t tokens;
  int32_t Hk, Hv, rep, map, decay, C;
  float l2_eps, rms_eps, scale;
  // launched to overlap the preceding kernel on the stream (programmatic
  // dependent launch): set only where that kernel is known not to write the
  // state, the conv state or any weight (inside gdn_decode_layer)
  int32_t overlap_prev;
};

// Linear layer y = x W^T (+ bias) (linear.cu): output column n goes to
// destination r with start[r] <= n < start[r + 1] (r < count), at
// dst[r] + m * ld[r] + (n - start[r]); columns at or past start[count] are
// not written. Starts, strides and destination addresses are multiples of 8
// elements.
constexpr int kLinearRoutes = 4;
struct LinearRoute {
  int32_t count;
  int32_t start[kLinearRoutes + 1];
  int64_t ld[kLinearRoutes];
  void* dst[kLinearRoutes];
};
struct LinearArgs {
  int32_t M, N, K, splits, stages;  // splits and stages are chosen by launch_linear
  const float* bias;        // [N] or null
  LinearRoute route;
  // launched to overlap the preceding kernel (programmatic dependent
  // launch): set only where that kernel does not write w or the bias
  int32_t overlap_prev;
};

struct ConvArgs {
  const int32_t* cu_seqlens;
  int32_t N;
  int64_t T;
  int32_t C;
  const void* x;
  const void* conv_w;
  void* conv_state;
  void* y;
};

struct RmsNormArgs {
  int64_t rows;
  const float* o;
  const void* z;
  const float* norm_w;
  void* y;
  float eps;
};

struct PrefillArgs {
  const int32_t* cu_seqlens;
  int32_t N;
  int64_t T;
  const void* q;
  int64_t q_stride;
  const void* k;
  int64_t k_stride;
  const void* v;
  int64_t v_stride;
  const void* a;
  const void* b;
  const float* decay_param;
  const float* dt_bias;
  int32_t flags;
  float* state;
  float* core_out;
  const void* z;
  const float* norm_w;
  void* out;
  int32_t Hk, Hv, rep, map, decay;
  float l2_eps, rms_eps, scale;
};

// Each launcher dispatches on (io dtype, head_dim) and returns the launch
// status (cudaSuccess when everything was enqueued).
cudaError_t launch_decode(const DecodeArgs& p, int32_t dtype, int32_t D, int32_t batch,
                          cudaStream_t stream);
cudaError_t launch_decode_multi(const DecodeArgs& p, int32_t dtype, int32_t D, int32_t batch,
                                cudaStream_t stream);
cudaError_t launch_conv(const ConvArgs& p, int32_t dtype, cudaStream_t stream);
cudaError_t launch_rmsnorm(const RmsNormArgs& p, int32_t dtype, int32_t D, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& p, int32_t dtype, int32_t D, cudaStream_t stream);
// tensor-core chunked prefill (head_dim 128, f16/bf16 activations)
bool prefill_tc_supported(const PrefillArgs& p, int32_t dtype, int32_t D);
cudaError_t launch_prefill_tc(const PrefillArgs& p, int32_t dtype, cudaStream_t stream);
// chunk-parallel tensor-core prefill (head_dim 128, bf16) over a workspace
int64_t prefill_cp_workspace_bytes(int32_t N, int64_t T, int32_t Hk, int32_t Hv);
bool prefill_cp_supported(const PrefillArgs& p, int32_t dtype, int32_t D);
// whether launch_prefill_cp carries the state with the sliced kernel
bool prefill_cp_sliced(const PrefillArgs& p);
cudaError_t launch_prefill_cp(const PrefillArgs& p, void* workspace, cudaStream_t stream);

// Device error words, one per kernel translation unit.
cudaError_t read_error_decode(int32_t* status, bool clear);
cudaError_t read_error_decode_mt(int32_t* status, bool clear);
cudaError_t read_error_conv(int32_t* status, bool clear);
cudaError_t read_error_rmsnorm(int32_t* status, bool clear);
cudaError_t read_error_prefill(int32_t* status, bool clear);
cudaError_t read_error_prefill_tc(int32_t* status, bool clear);
cudaError_t read_error_prefill_cp(int32_t* status, bool clear);
cudaError_t read_error_diag(int32_t* status, bool clear);
cudaError_t read_error_linear(int32_t* status, bool clear);
// linear.cu: M <= 128, N and K multiples of 64, bf16
int64_t linear_workspace_bytes(int32_t M, int32_t N, int32_t K);
bool linear_supported();
cudaError_t launch_linear(LinearArgs p, const void* x, int64_t x_stride, const void* w, void* workspace,
                          cudaStream_t stream);
// diag.cu: one warp's bounded wait on an mbarrier nothing arrives on
cudaError_t launch_wait_timeout(uint64_t limit_ns, int32_t* gave_up, cudaStream_t stream);

}  // namespace gdn

// Defines the per-translation-unit device error word reader.
#define GDN_DEFINE_ERROR_READER(NAME)                                                  \
  namespace gdn {                                                                      \
  cudaError_t read_error_##NAME(int32_t* status, bool clear) {                         \
    int32_t v = 0;                                                                     \
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));               \
    if (e != cudaSuccess) return e;                                                    \
    *status = v;                                                                       \
    if (clear && v != 0) {                                                             \
      const int32_t zero = 0;                                                          \
      e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));                     \
    }                                                                                  \
    return e;                                                                          \
  }                                                                                    \
  }
