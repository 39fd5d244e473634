// Chunked prefill on CUDA cores (fp32 throughout): the generic path for any
// supported head_dim and dtype, and the correctness reference for the tensor
// core kernel.
//
// The recurrence of gdn.rs is summed chunk-wise (chunk 64). Within a chunk of
// L tokens starting from state S0, with c_t the chunk-local inclusive cumulative
// sum of g and G_t = e^{c_t}:
//   A[t][s] = beta_t e^{c_t - c_s} (k_t . k_s)   (s < t)
//   Tm      = (I + A)^{-1}                      (unit lower triangular)
//   U       = Tm diag(beta) V,   W = Tm diag(beta G) K
//   Dm      = U - W S0^T                        (rows: the per-token d_t)
//   O       = diag(G) Q S0^T + (Q K^T o M) Dm,  M[t][s] = e^{c_t - c_s} (s <= t)
//   S_L     = G_L S0 + Dm^T diag(e^{c_L - c}) K
// which are the six stages the Metal chunk pipeline names (K gram,
// (I+A)^-1, U/W, Q K^T, carry, output; ferrum-kernels
// gated_delta_attention_tests.rs `run_chunked_core`). Decays are only ever
// applied as e^{difference <= 0}, never divided out, so strongly decaying
// heads underflow to 0 instead of overflowing.
//
// Grid: (Dv slice, V head, sequence). A CTA owns NS value rows of one head's
// state (value rows evolve independently given k, g, beta), keeps them in
// shared memory across chunks, and recomputes the key-side quantities
// (norms, K gram, Tm, W) it needs. With a fused gated RMSNorm the slices of a
// head form a thread-block cluster and exchange per-row partial sums of squares
// through distributed shared memory.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

constexpr int kChunk = 64;
constexpr int kPfThreads = 256;
constexpr int kPfNS = 32;

template <int D, int NS>
struct PfSmem {
  static constexpr int LD = D + 1;  // padded strides keep column walks conflict-free
  static constexpr int LN = NS + 1;
  static constexpr int LC = kChunk + 1;
  float K[kChunk * LD];
  float Q[kChunk * LD];
  float W[kChunk * LD];
  float S[NS * LD];
  float V[kChunk * LN];   // value slice, later the output slice
  float U[kChunk * LN];   // U, later diag(G) Q S0^T
  float Dm[kChunk * LN];
  float A[kChunk * LC];
  float Tm[kChunk * LC];
  float P[kChunk * LC];
  float g[kChunk], beta[kChunk], c[kChunk], gam[kChunk], dl[kChunk];
  float norm[2][kChunk];
};

__device__ __forceinline__ int64_t clamp_cu_pf(const int32_t* cu, int n, int64_t T) {
  int64_t v = cu[n];
  return v < 0 ? 0 : (v > T ? T : v);
}

template <typename T, int D, int NS>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_cc_kernel(const PrefillArgs p) {
  using SM = PfSmem<D, NS>;
  constexpr int LD = SM::LD, LN = SM::LN, LC = SM::LC;
  constexpr int NSL = D / NS;
  extern __shared__ __align__(16) unsigned char smraw[];
  SM& sm = *reinterpret_cast<SM*>(smraw);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int kh = k_head_of(p.map, h, p.Hk, p.rep);
  const int j0 = slice * NS;
  const int64_t seq_s = clamp_cu_pf(p.cu_seqlens, n, p.T);
  int64_t seq_e = clamp_cu_pf(p.cu_seqlens, n + 1, p.T);
  if (seq_e < seq_s) seq_e = seq_s;
  const bool prenorm = (p.flags & GDN_QK_PRENORMALIZED) != 0;
  const bool pregate = (p.flags & GDN_GATES_PRECOMPUTED) != 0;
  const bool fused_norm = p.z != nullptr;
  const T* qg = static_cast<const T*>(p.q);
  const T* kg = static_cast<const T*>(p.k);
  const T* vg = static_cast<const T*>(p.v);

  float* gS = p.state + (((size_t)n * p.Hv + h) * D + j0) * D;
  for (int e = tid; e < NS * D; e += kPfThreads) sm.S[(e / D) * LD + (e % D)] = gS[e];

  int chunk_idx = 0;
  for (int64_t c0 = seq_s; c0 < seq_e; c0 += kChunk, ++chunk_idx) {
    const int L = (int)((seq_e - c0) < kChunk ? (seq_e - c0) : kChunk);
    __syncthreads();

    // (1) loads: keys, queries, this slice of values, gates
    for (int e = tid; e < kChunk * D; e += kPfThreads) {
      const int t = e / D, i = e - (e / D) * D;
      float kv = 0.f, qv = 0.f;
      if (t < L) {
        const int64_t tok = c0 + t;
        kv = to_f32(kg[tok * p.k_stride + (int64_t)kh * D + i]);
        qv = to_f32(qg[tok * p.q_stride + (int64_t)kh * D + i]);
      }
      sm.K[t * LD + i] = kv;
      sm.Q[t * LD + i] = qv;
    }
    for (int e = tid; e < kChunk * NS; e += kPfThreads) {
      const int t = e / NS, j = e - (e / NS) * NS;
      float vv = 0.f;
      if (t < L) vv = to_f32(vg[(c0 + t) * p.v_stride + (int64_t)h * D + j0 + j]);
      sm.V[t * LN + j] = vv;
    }
    if (tid < kChunk) {
      float g = 0.f, bt = 0.f;
      if (tid < L) {
        const int64_t gi = (c0 + tid) * p.Hv + h;
        if (pregate) {
          g = static_cast<const float*>(p.a)[gi];
          bt = static_cast<const float*>(p.b)[gi];
        } else {
          g = gate_g(p.decay, p.decay_param[h], p.dt_bias[h], to_f32(static_cast<const T*>(p.a)[gi]));
          bt = sigmoid_f(to_f32(static_cast<const T*>(p.b)[gi]));
        }
      }
      sm.g[tid] = g;
      sm.beta[tid] = bt;
    }
    __syncthreads();

    // (2) l2 norms (q also scaled by 1/sqrt(D)) and the cumulative decay
    for (int t = warp; t < kChunk; t += kPfThreads / 32) {
      float kk = 0.f, qq = 0.f;
      for (int i = lane; i < D; i += 32) {
        kk += sm.K[t * LD + i] * sm.K[t * LD + i];
        qq += sm.Q[t * LD + i] * sm.Q[t * LD + i];
      }
      kk = group_sum<32>(kk);
      qq = group_sum<32>(qq);
      const float ik = prenorm ? 1.f : 1.f / sqrtf(kk + p.l2_eps);
      const float iq = (prenorm ? 1.f : 1.f / sqrtf(qq + p.l2_eps)) * p.scale;
      for (int i = lane; i < D; i += 32) {
        sm.K[t * LD + i] *= ik;
        sm.Q[t * LD + i] *= iq;
      }
    }
    if (tid == 0) {
      float run = 0.f;
      for (int t = 0; t < kChunk; ++t) {
        run += sm.g[t];
        sm.c[t] = run;
      }
    }
    __syncthreads();
    if (tid < kChunk) {
      sm.gam[tid] = expf(sm.c[tid]);
      sm.dl[tid] = tid < L ? expf(sm.c[L - 1] - sm.c[tid]) : 0.f;
    }

    // (3) key gram -> A (strictly lower), Q K^T -> P (masked, decayed)
    for (int e = tid; e < kChunk * kChunk; e += kPfThreads) {
      const int t = e / kChunk, s = e - (e / kChunk) * kChunk;
      float a = 0.f, pv = 0.f;
      if (s <= t && t < L) {
        float gk = 0.f, pq = 0.f;
        for (int i = 0; i < D; ++i) {
          const float ks = sm.K[s * LD + i];
          gk = fmaf(sm.K[t * LD + i], ks, gk);
          pq = fmaf(sm.Q[t * LD + i], ks, pq);
        }
        const float dec = expf(sm.c[t] - sm.c[s]);
        if (s < t) a = sm.beta[t] * dec * gk;
        pv = dec * pq;
      }
      sm.A[t * LC + s] = a;
      sm.P[t * LC + s] = pv;
      sm.Tm[t * LC + s] = (t == s) ? 1.f : 0.f;
    }
    __syncthreads();

    // (4) Tm = (I + A)^{-1}, row by row:
    //     Tm[t][s] = -A[t][s] - sum_{s<r<t} A[t][r] Tm[r][s]
    for (int t = 1; t < L; ++t) {
      const int s = tid >> 2, part = tid & 3;
      float acc = 0.f;
      if (s < t) {
        for (int r = s + 1 + part; r < t; r += 4) acc = fmaf(sm.A[t * LC + r], sm.Tm[r * LC + s], acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (s < t && part == 0) sm.Tm[t * LC + s] = -sm.A[t * LC + s] - acc;
      __syncthreads();
    }

    // (5) U = Tm diag(beta) V,  W = Tm diag(beta G) K
    for (int e = tid; e < kChunk * NS; e += kPfThreads) {
      const int t = e / NS, j = e - (e / NS) * NS;
      float u = 0.f;
      for (int s = 0; s <= t; ++s) u = fmaf(sm.Tm[t * LC + s] * sm.beta[s], sm.V[s * LN + j], u);
      sm.U[t * LN + j] = u;
    }
    for (int e = tid; e < kChunk * D; e += kPfThreads) {
      const int t = e / D, i = e - (e / D) * D;
      float w = 0.f;
      for (int s = 0; s <= t; ++s)
        w = fmaf(sm.Tm[t * LC + s] * sm.beta[s] * sm.gam[s], sm.K[s * LD + i], w);
      sm.W[t * LD + i] = w;
    }
    __syncthreads();

    // (6) Dm = U - W S0^T;  U <- diag(G) Q S0^T
    for (int e = tid; e < kChunk * NS; e += kPfThreads) {
      const int t = e / NS, j = e - (e / NS) * NS;
      float ws = 0.f, qs = 0.f;
      for (int i = 0; i < D; ++i) {
        const float sv = sm.S[j * LD + i];
        ws = fmaf(sm.W[t * LD + i], sv, ws);
        qs = fmaf(sm.Q[t * LD + i], sv, qs);
      }
      sm.Dm[t * LN + j] = sm.U[t * LN + j] - ws;
      sm.U[t * LN + j] = sm.gam[t] * qs;
    }
    __syncthreads();

    // (7) O = diag(G) Q S0^T + P Dm  (into V);  S <- G_L S0 + Dm^T diag(dl) K
    for (int e = tid; e < kChunk * NS; e += kPfThreads) {
      const int t = e / NS, j = e - (e / NS) * NS;
      float o = sm.U[t * LN + j];
      for (int s = 0; s <= t; ++s) o = fmaf(sm.P[t * LC + s], sm.Dm[s * LN + j], o);
      sm.V[t * LN + j] = o;
    }
    {
      const float gL = sm.gam[L - 1];
      for (int e = tid; e < NS * D; e += kPfThreads) {
        const int j = e / D, i = e - (e / D) * D;
        float acc = gL * sm.S[j * LD + i];
        for (int s = 0; s < L; ++s) acc = fmaf(sm.dl[s] * sm.Dm[s * LN + j], sm.K[s * LD + i], acc);
        sm.S[j * LD + i] = acc;
      }
    }
    __syncthreads();

    // (8) outputs
    if (p.core_out != nullptr) {
      for (int e = tid; e < L * NS; e += kPfThreads) {
        const int t = e / NS, j = e - (e / NS) * NS;
        p.core_out[((c0 + t) * p.Hv + h) * D + j0 + j] = sm.V[t * LN + j];
      }
    }
    if (fused_norm) {
      const int buf = chunk_idx & 1;
      for (int t = warp; t < kChunk; t += kPfThreads / 32) {
        float ss = 0.f;
        for (int j = lane; j < NS; j += 32) ss += sm.V[t * LN + j] * sm.V[t * LN + j];
        ss = group_sum<32>(ss);
        if (lane == 0) sm.norm[buf][t] = ss;
      }
      if (NSL > 1) {
        cluster_arrive_release();
        cluster_wait_acquire();
      } else {
        __syncthreads();
      }
      const T* zg = static_cast<const T*>(p.z);
      T* og = static_cast<T*>(p.out);
      for (int e = tid; e < L * NS; e += kPfThreads) {
        const int t = e / NS, j = e - (e / NS) * NS;
        float tot = 0.f;
        if (NSL > 1) {
          const uint32_t addr = smem_u32(&sm.norm[buf][t]);
#pragma unroll
          for (int r = 0; r < NSL; ++r) tot += ld_shared_cluster_f32(map_shared_rank(addr, r));
        } else {
          tot = sm.norm[buf][t];
        }
        const float inv = 1.f / sqrtf(tot / (float)D + p.rms_eps);
        const int64_t oi = ((c0 + t) * p.Hv + h) * D + j0 + j;
        const float y = sm.V[t * LN + j] * inv * p.norm_w[j0 + j] * silu_f(to_f32(zg[oi]));
        og[oi] = from_f32<T>(y);
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < NS * D; e += kPfThreads) gS[e] = sm.S[(e / D) * LD + (e % D)];
  if (fused_norm && NSL > 1) {
    // no CTA leaves while a peer may still read its partial sums
    cluster_arrive_release();
    cluster_wait_acquire();
  }
}

template <typename T, int D>
static cudaError_t launch_prefill_t(const PrefillArgs& p, cudaStream_t stream) {
  constexpr int NS = D < kPfNS ? D : kPfNS;
  constexpr int NSL = D / NS;
  auto kern = prefill_cc_kernel<T, D, NS>;
  const int smem = (int)sizeof(PfSmem<D, NS>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (p.N == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)NSL, (unsigned)p.Hv, (unsigned)p.N);
  cfg.blockDim = dim3(kPfThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)NSL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename T>
static cudaError_t launch_prefill_d(const PrefillArgs& p, int32_t D, cudaStream_t stream) {
  switch (D) {
    case 32: return launch_prefill_t<T, 32>(p, stream);
    case 64: return launch_prefill_t<T, 64>(p, stream);
    case 96: return launch_prefill_t<T, 96>(p, stream);
    case 128: return launch_prefill_t<T, 128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefill(const PrefillArgs& p, int32_t dtype, int32_t D, cudaStream_t stream) {
  if ((p.flags & GDN_PREFILL_CUDA_CORES) == 0 && prefill_tc_supported(p, dtype, D))
    return launch_prefill_tc(p, dtype, stream);
  switch (dtype) {
    case GDN_F16: return launch_prefill_d<__half>(p, D, stream);
    case GDN_BF16: return launch_prefill_d<__nv_bfloat16>(p, D, stream);
    case GDN_F32: return launch_prefill_d<float>(p, D, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(prefill)
