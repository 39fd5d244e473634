// Gated RMSNorm: y = o (mean_j o_j^2 + eps)^(-1/2) w_j silu(z_j), computed in
// fp32 and rounded once to the io dtype (ferrum-kernels
// gated_delta_attention_tests.rs, `cpu_segment` output loop). One warp per
// row of D; each lane owns D/32 consecutive elements.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

template <typename T, int D>
__global__ void __launch_bounds__(256) gated_rmsnorm_kernel(const RmsNormArgs p) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= p.rows) return;
  const float* o = p.o + row * D + lane * PER;
  const T* z = static_cast<const T*>(p.z) + row * D + lane * PER;
  T* y = static_cast<T*>(p.y) + row * D + lane * PER;
  float ov[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) ov[e] = o[e];
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) ss += ov[e] * ov[e];
  ss = group_sum<32>(ss);
  const float inv = 1.f / sqrtf(ss / (float)D + p.eps);
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const float v = ov[e] * inv * p.norm_w[lane * PER + e] * silu_fast(to_f32(z[e]));
    y[e] = from_f32<T>(v);
  }
}

template <typename T>
static cudaError_t launch_rms_t(const RmsNormArgs& p, int32_t D, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  const int64_t grid = (p.rows + 7) / 8;
  switch (D) {
    case 32: gated_rmsnorm_kernel<T, 32><<<(unsigned)grid, 256, 0, stream>>>(p); break;
    case 64: gated_rmsnorm_kernel<T, 64><<<(unsigned)grid, 256, 0, stream>>>(p); break;
    case 96: gated_rmsnorm_kernel<T, 96><<<(unsigned)grid, 256, 0, stream>>>(p); break;
    case 128: gated_rmsnorm_kernel<T, 128><<<(unsigned)grid, 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const RmsNormArgs& p, int32_t dtype, int32_t D, cudaStream_t stream) {
  switch (dtype) {
    case GDN_F16: return launch_rms_t<__half>(p, D, stream);
    case GDN_BF16: return launch_rms_t<__nv_bfloat16>(p, D, stream);
    case GDN_F32: return launch_rms_t<float>(p, D, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(rmsnorm)
