// Causal depthwise conv1d (kernel 4) + SiLU over packed variable-length
// sequences, with a rolling 3-wide conv state per sequence
// (ferrum-kernels gated_delta_attention_tests.rs, `cpu_segment` conv loop and
// conv-state update; libmir-metal decode/mod.rs `convolve`).
//
// Two launches on the caller's stream:
//  1. conv_fwd_kernel: y for every token, persistent, two CTAs per SM. The
//     work is cut into tiles of 64 tokens x 512 bytes of channels. A load
//     warp streams each tile's 67 input rows (three rows of history, then the
//     64 tokens) into a three-stage shared-memory ring with one TMA copy per
//     tile; rows before the first token or past the last read as zero. Eight
//     compute warps take eight tokens each: a thread holds 16 bytes of
//     channels, reads the 11 rows its window needs from shared memory once,
//     and accumulates each row into the (at most four) tokens it is a tap of,
//     two channels per paired fp32 FMA, taps in order 0..3 from zero; a token
//     is stored as soon as its last tap is in. Only windows that reach back
//     past a sequence start (or tiles past the end) take the per-token path
//     that reads the OLD conv state for the taps before the sequence's first
//     token.
//  2. conv_state_kernel: the new conv state (last three raw inputs of each
//     sequence). Running it after (1) in stream order is what makes the in-place
//     state update race-free: (1) never sees a half-updated state.
#include <cuda.h>

#include <type_traits>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {
namespace {

constexpr int kCvTok = 64;                               // output tokens per tile
constexpr int kCvRows = kCvTok + 3;                      // input rows per tile
constexpr int kCvRowBytes = 512;                         // channels per tile, in bytes
constexpr uint32_t kCvStageBytes = kCvRows * kCvRowBytes;  // 34,304
constexpr int kCvStages = 3;
constexpr int kCvWarps = 8;                   // compute warps
constexpr int kCvTpt = kCvTok / kCvWarps;     // tokens per thread
constexpr int kCvThreads = (kCvWarps + 1) * 32;  // + the load warp
constexpr int kCvCtasPerSm = 2;
constexpr uint32_t kCvSmem = kCvStages * kCvStageBytes + 128;

__device__ __forceinline__ int64_t clamp_cu(const int32_t* cu, int n, int64_t T) {
  int64_t v = cu[n];
  return v < 0 ? 0 : (v > T ? T : v);
}

// the last sequence n in [0, N) with start <= t
__device__ __forceinline__ int seq_of(const int32_t* cu, int N, int64_t T, int64_t t) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (clamp_cu(cu, mid, T) <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// 16 bytes of channels as fp32 pairs (channels 2p, 2p + 1 in pair p)
template <typename T>
__device__ __forceinline__ void unpack_pairs(const uint4& raw, float2 (&x)[16 / sizeof(T) / 2]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  if constexpr (sizeof(T) == 4) {
    x[0] = make_float2(__uint_as_float(w[0]), __uint_as_float(w[1]));
    x[1] = make_float2(__uint_as_float(w[2]), __uint_as_float(w[3]));
  } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
#pragma unroll
    for (int p = 0; p < 4; ++p) x[p] = make_float2(__uint_as_float(w[p] << 16), __uint_as_float(w[p] & 0xffff0000u));
  } else {
#pragma unroll
    for (int p = 0; p < 4; ++p) x[p] = __half22float2(*reinterpret_cast<const __half2*>(&w[p]));
  }
}

__device__ __forceinline__ float silu_conv(float a) {
  // silu with the fast exponential and divide (~2^-21 relative error, far
  // below one ulp of the 16-bit output)
  return __fdividef(a, 1.f + __expf(-a));
}

template <typename T>
__device__ __forceinline__ uint4 pack_pairs(const float2 (&v)[16 / sizeof(T) / 2]) {
  uint4 out;
  uint32_t* o = reinterpret_cast<uint32_t*>(&out);
  if constexpr (sizeof(T) == 4) {
    o[0] = __float_as_uint(silu_conv(v[0].x));
    o[1] = __float_as_uint(silu_conv(v[0].y));
    o[2] = __float_as_uint(silu_conv(v[1].x));
    o[3] = __float_as_uint(silu_conv(v[1].y));
  } else {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float a = silu_conv(v[p].x), b = silu_conv(v[p].y);
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        o[p] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __half2 h = __floats2half2_rn(a, b);
        o[p] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
  }
  return out;
}

template <typename T>
__global__ void __launch_bounds__(kCvThreads, kCvCtasPerSm)
    conv_fwd_kernel(const ConvArgs p, const __grid_constant__ CUtensorMap tm_x, int64_t ntt,
                    int64_t ntiles) {
  constexpr int VEC = 16 / (int)sizeof(T);  // channels per thread
  constexpr int NP = VEC / 2;               // channel pairs per thread
  constexpr int CPT = kCvRowBytes / (int)sizeof(T);  // channels per tile
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  __shared__ __align__(8) uint64_t full[kCvStages], empty[kCvStages];
  __shared__ int s_abort;
  volatile int* abort_flag = &s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kCvStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCvWarps);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCvWarps) {
    // load warp: tile i of this CTA into stage i % S once its previous
    // occupant is consumed
    if (lane != 0) return;
    int64_t issued = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++issued) {
      const int s = (int)(issued % kCvStages);
      if (issued >= kCvStages &&
          !mbar_wait_bounded(&empty[s], (uint32_t)(((issued / kCvStages) - 1) & 1), abort_flag))
        break;
      const int64_t cb = tile / ntt, tt = tile - cb * ntt;
      mbar_arrive_expect_tx(&full[s], kCvStageBytes);
      tc::tma_load_2d(sm + s * kCvStageBytes, &tm_x, (int)(cb * CPT), (int)(tt * kCvTok - 3), &full[s]);
    }
    // no copy may land in shared memory after the CTA has exited: wait for
    // the last S issued (each is the latest phase of its stage)
    for (int64_t i = issued > kCvStages ? issued - kCvStages : 0; i < issued; ++i)
      mbar_wait_bounded(&full[i % kCvStages], (uint32_t)((i / kCvStages) & 1), nullptr);
    return;
  }

  const int64_t T_ = p.T, C = p.C;
  const T* st = static_cast<const T*>(p.conv_state);
  T* y = static_cast<T*>(p.y);
  float2 w[NP][4];  // weights of this thread's channel pairs, by tap
  int64_t cur_cb = -1;
  int64_t k = 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
    const int s = (int)(k % kCvStages);
    const int64_t cb = tile / ntt, tt = tile - cb * ntt;
    const int64_t c0 = cb * CPT + (int64_t)lane * VEC;
    const int64_t ta = tt * kCvTok + (int64_t)warp * kCvTpt;  // first output token of this thread
    const bool live = c0 < C && ta < T_;
    if (cb != cur_cb) {
      cur_cb = cb;
      if (c0 < C) {
        const uint4* wp = reinterpret_cast<const uint4*>(static_cast<const T*>(p.conv_w) + c0 * 4);
        constexpr int WV = VEC * 4 * (int)sizeof(T) / 16;
        uint4 wr[WV];
#pragma unroll
        for (int i = 0; i < WV; ++i) wr[i] = wp[i];
        const T* wv = reinterpret_cast<const T*>(wr);
#pragma unroll
        for (int q = 0; q < NP; ++q)
#pragma unroll
          for (int j = 0; j < 4; ++j) w[q][j] = make_float2(to_f32(wv[(2 * q) * 4 + j]), to_f32(wv[(2 * q + 1) * 4 + j]));
      }
    }
    // fast when the window of every token of this thread lies in one sequence
    bool fast = false;
    int n = 0;
    if (live) {
      const int64_t tl = ta + kCvTpt - 1 < T_ ? ta + kCvTpt - 1 : T_ - 1;
      n = seq_of(p.cu_seqlens, p.N, T_, tl);
      fast = ta + kCvTpt <= T_ && clamp_cu(p.cu_seqlens, n, T_) <= ta - 3;
    }
    const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((k / kCvStages) & 1), abort_flag);
    if (__any_sync(0xffffffffu, !ok)) break;
    // row u of this thread's window (token ta - 3 + u), its 16 bytes
    const unsigned char* rows = sm + s * kCvStageBytes + warp * kCvTpt * kCvRowBytes + lane * 16;
    if (live && fast) {
      float2 acc[4][NP];  // the four tokens in flight, token jj in acc[jj % 4]
#pragma unroll
      for (int u = 0; u < kCvTpt + 3; ++u) {
        float2 xv[NP];
        unpack_pairs<T>(*reinterpret_cast<const uint4*>(rows + u * kCvRowBytes), xv);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int jj = u - j;  // the token this row is tap j of
          if (jj >= 0 && jj < kCvTpt) {
#pragma unroll
            for (int q = 0; q < NP; ++q)
              acc[jj & 3][q] = fma2(w[q][j], xv[q], j == 0 ? make_float2(0.f, 0.f) : acc[jj & 3][q]);
          }
        }
        if (u >= 3) {
          const int jj = u - 3;
          *reinterpret_cast<uint4*>(y + (ta + jj) * C + c0) = pack_pairs<T>(acc[jj & 3]);
        }
      }
    } else if (live) {
      // per token; taps before the sequence's first token come from the old
      // conv state
      n = seq_of(p.cu_seqlens, p.N, T_, ta);
      int64_t s_n = clamp_cu(p.cu_seqlens, n, T_);
      int64_t s_next = n + 1 < p.N ? clamp_cu(p.cu_seqlens, n + 1, T_) : T_ + 1;
      for (int jj = 0; jj < kCvTpt; ++jj) {
        const int64_t t = ta + jj;
        if (t >= T_) break;
        while (s_next <= t) {
          ++n;
          s_n = s_next;
          s_next = n + 1 < p.N ? clamp_cu(p.cu_seqlens, n + 1, T_) : T_ + 1;
        }
        const int64_t sq = s_n > t ? t : s_n;
        float2 acc[NP];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t tau = t + j - 3;
          float2 xv[NP];
          if (tau >= sq) {
            unpack_pairs<T>(*reinterpret_cast<const uint4*>(rows + (jj + j) * kCvRowBytes), xv);
          } else {
            const int slot = 3 + (int)(tau - sq);
            const T* sp = st + ((int64_t)n * C + c0) * 3 + slot;
#pragma unroll
            for (int q = 0; q < NP; ++q) xv[q] = make_float2(to_f32(sp[(2 * q) * 3]), to_f32(sp[(2 * q + 1) * 3]));
          }
#pragma unroll
          for (int q = 0; q < NP; ++q) acc[q] = fma2(w[q][j], xv[q], j == 0 ? make_float2(0.f, 0.f) : acc[q]);
        }
        *reinterpret_cast<uint4*>(y + t * C + c0) = pack_pairs<T>(acc);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
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

int conv_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

template <typename T>
cudaError_t launch_conv_t(const ConvArgs& p, CUtensorMapDataType dt, cudaStream_t stream) {
  if (p.T > 0) {
    CUtensorMap tm;
    constexpr int CPT = kCvRowBytes / (int)sizeof(T);
    if (!tc::make_map_2d(&tm, p.x, p.T, p.C, p.C, sizeof(T), dt, CPT, kCvRows,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    const int64_t ntt = (p.T + kCvTok - 1) / kCvTok;
    const int64_t ncb = ((int64_t)p.C + CPT - 1) / CPT;
    const int64_t ntiles = ntt * ncb;
    const int64_t slots = (int64_t)kCvCtasPerSm * conv_sm_count();
    const int grid = (int)(ntiles < slots ? ntiles : slots);
    cudaError_t e = cudaFuncSetAttribute(conv_fwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kCvSmem);
    if (e != cudaSuccess) return e;
    conv_fwd_kernel<T><<<grid, kCvThreads, kCvSmem, stream>>>(p, tm, ntt, ntiles);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.N > 0) {
    const int64_t gy = (p.C + 255) / 256;
    conv_state_kernel<T><<<dim3((unsigned)p.N, (unsigned)gy), 256, 0, stream>>>(p);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_conv(const ConvArgs& p, int32_t dtype, cudaStream_t stream) {
  switch (dtype) {
    case GDN_F16: return launch_conv_t<__half>(p, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, stream);
    case GDN_BF16: return launch_conv_t<__nv_bfloat16>(p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, stream);
    case GDN_F32: return launch_conv_t<float>(p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(conv)
