// Causal depthwise conv1d (kernel 4) + SiLU over packed variable-length
// sequences, with a rolling 3-wide conv state per sequence
// (ferrum-kernels gated_delta_attention_tests.rs, `cpu_segment` conv loop and
// conv-state update; libmir-metal decode/mod.rs `convolve`).
//
// Two launches on the caller's stream:
//  1. conv_fwd_kernel: y for every token. A thread owns 16 bytes of channels
//     (8 for f16/bf16, 4 for f32) and 4 consecutive tokens; it loads the 7
//     input rows its window needs once (16-byte vectors), converts its
//     weights once, and when one sequence covers the whole window unpacks
//     each row once into the accumulators of every token it is a tap of. Only
//     windows that reach back past a sequence start take the per-token path
//     that reads the OLD conv state for the (at most three) taps before the
//     sequence's first token. The kernel is bound by instruction issue, not
//     by HBM, so every per-element instruction counts.
//  2. conv_state_kernel: the new conv state (last three raw inputs of each
//     sequence). Running it after (1) in stream order is what makes the in-place
//     state update race-free: (1) never sees a half-updated state.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

constexpr int kConvTPT = 4;    // tokens per thread
constexpr int kConvCV = 32;    // channel vectors per block
constexpr int kConvTG = 8;     // token groups per block

__device__ __forceinline__ int64_t clamp_cu(const int32_t* cu, int n, int64_t T) {
  int64_t v = cu[n];
  return v < 0 ? 0 : (v > T ? T : v);
}

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& raw, float (&out)[16 / sizeof(T)]) {
  const T* v = reinterpret_cast<const T*>(&raw);
#pragma unroll
  for (int e = 0; e < (int)(16 / sizeof(T)); ++e) out[e] = to_f32(v[e]);
}

template <typename T>
__global__ void __launch_bounds__(kConvCV* kConvTG) conv_fwd_kernel(const ConvArgs p) {
  constexpr int VEC = 16 / (int)sizeof(T);
  constexpr int NR = kConvTPT + 3;
  const int cv = threadIdx.x % kConvCV, tg = threadIdx.x / kConvCV;
  const int64_t c0 = ((int64_t)blockIdx.y * kConvCV + cv) * VEC;
  const int64_t t0 = ((int64_t)blockIdx.x * kConvTG + tg) * kConvTPT;
  const int64_t T_ = p.T, C = p.C;
  if (c0 >= C || t0 >= T_) return;
  const T* xp = static_cast<const T*>(p.x) + c0;
  const T* st = static_cast<const T*>(p.conv_state);
  T* y = static_cast<T*>(p.y);

  uint4 xr[NR];
#pragma unroll
  for (int u = 0; u < NR; ++u) {
    const int64_t tau = t0 - 3 + u;
    xr[u] = (tau >= 0 && tau < T_) ? *reinterpret_cast<const uint4*>(xp + tau * C)
                                    : make_uint4(0, 0, 0, 0);
  }
  float wf[VEC][4];
  {
    constexpr int WV = VEC * 4 * (int)sizeof(T) / 16;
    uint4 wr[WV];
    const uint4* wp = reinterpret_cast<const uint4*>(static_cast<const T*>(p.conv_w) + c0 * 4);
#pragma unroll
    for (int i = 0; i < WV; ++i) wr[i] = wp[i];
    const T* wv = reinterpret_cast<const T*>(wr);
#pragma unroll
    for (int e = 0; e < VEC; ++e)
#pragma unroll
      for (int j = 0; j < 4; ++j) wf[e][j] = to_f32(wv[e * 4 + j]);
  }
  int lo = 0, hi = p.N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (clamp_cu(p.cu_seqlens, mid, T_) <= t0) lo = mid;
    else hi = mid - 1;
  }
  int n = lo;
  int64_t s_n = clamp_cu(p.cu_seqlens, n, T_);
  int64_t s_next = n + 1 < p.N ? clamp_cu(p.cu_seqlens, n + 1, T_) : T_ + 1;

  float acc[kConvTPT][VEC];
#pragma unroll
  for (int jj = 0; jj < kConvTPT; ++jj)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[jj][e] = 0.f;
  if (s_n <= t0 - 3 && s_next > t0 + kConvTPT - 1) {
    // one sequence covers the whole window: each row is unpacked once and
    // feeds every output token it is a tap of
#pragma unroll
    for (int u = 0; u < NR; ++u) {
      float xv[VEC];
      unpack16<T>(xr[u], xv);
#pragma unroll
      for (int jj = 0; jj < kConvTPT; ++jj) {
        const int j = u - jj;  // tap index of row u for token jj
        if (j >= 0 && j < 4) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[jj][e] = fmaf(wf[e][j], xv[e], acc[jj][e]);
        }
      }
    }
  } else {
#pragma unroll
    for (int jj = 0; jj < kConvTPT; ++jj) {
      const int64_t t = t0 + jj;
      if (t >= T_) break;
      while (s_next <= t) {
        ++n;
        s_n = s_next;
        s_next = n + 1 < p.N ? clamp_cu(p.cu_seqlens, n + 1, T_) : T_ + 1;
      }
      const int64_t s = s_n > t ? t : s_n;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t tau = t + j - 3;
        float xv[VEC];
        if (tau >= s) {
          unpack16<T>(xr[jj + j], xv);
        } else {
          const int slot = 3 + (int)(tau - s);
          const T* sp = st + ((int64_t)n * C + c0) * 3 + slot;
#pragma unroll
          for (int e = 0; e < VEC; ++e) xv[e] = to_f32(sp[e * 3]);
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[jj][e] = fmaf(wf[e][j], xv[e], acc[jj][e]);
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < kConvTPT; ++jj) {
    const int64_t t = t0 + jj;
    if (t < T_) {
      uint4 packed;
      T* pv = reinterpret_cast<T*>(&packed);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float a = acc[jj][e];
        // silu with the fast exponential and divide (~2^-21 relative error,
        // far below one ulp of the 16-bit output)
        pv[e] = from_f32<T>(__fdividef(a, 1.f + __expf(-a)));
      }
      *reinterpret_cast<uint4*>(y + t * C + c0) = packed;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) conv_state_kernel(const ConvArgs p) {
  const int n = blockIdx.x;
  const int64_t c = (int64_t)blockIdx.y * 256 + threadIdx.x;
  if (c >= p.C) return;
  const int64_t T_ = p.T, C = p.C;
  const int64_t s = clamp_cu(p.cu_seqlens, n, T_);
  int64_t e = clamp_cu(p.cu_seqlens, n + 1, T_);
  if (e < s) e = s;
  const int64_t L = e - s;
  T* sp = static_cast<T*>(p.conv_state) + ((int64_t)n * C + c) * 3;
  const T* x = static_cast<const T*>(p.x);
  const T old[3] = {sp[0], sp[1], sp[2]};
  T nw[3];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const int64_t tau = L + q - 3;
    nw[q] = tau >= 0 ? x[(s + tau) * C + c] : old[3 + tau];
  }
#pragma unroll
  for (int q = 0; q < 3; ++q) sp[q] = nw[q];
}

template <typename T>
static cudaError_t launch_conv_t(const ConvArgs& p, cudaStream_t stream) {
  constexpr int VEC = 16 / (int)sizeof(T);
  if (p.T > 0) {
    const int64_t gx = (p.T + kConvTG * kConvTPT - 1) / (kConvTG * kConvTPT);
    const int64_t gy = (p.C / VEC + kConvCV - 1) / kConvCV;
    conv_fwd_kernel<T><<<dim3((unsigned)gx, (unsigned)gy), kConvCV * kConvTG, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.N > 0) {
    const int64_t gy = (p.C + 255) / 256;
    conv_state_kernel<T><<<dim3((unsigned)p.N, (unsigned)gy), 256, 0, stream>>>(p);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

cudaError_t launch_conv(const ConvArgs& p, int32_t dtype, cudaStream_t stream) {
  switch (dtype) {
    case GDN_F16: return launch_conv_t<__half>(p, stream);
    case GDN_BF16: return launch_conv_t<__nv_bfloat16>(p, stream);
    case GDN_F32: return launch_conv_t<float>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(conv)
