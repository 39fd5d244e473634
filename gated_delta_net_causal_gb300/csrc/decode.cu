// Fused decode step: conv + SiLU -> split q|k|v -> l2 norm -> gates ->
// gated delta-rule update of the fp32 state in place -> (gated RMSNorm).
//
// The step per value row j of V head h (ferrox-core gdn.rs, module docs and
// `delta_step`):  S_j *= a;  p = S_j . k;  d = b (v_j - p);  S_j += d k;
// o_j = S_j . q / sqrt(D).  The row is read once and written once: both
// dot products are taken from the OLD row, using
//   (a S_j) . k = a (S_j . k)   and   S_new_j . q = a (S_j . q) + d (k . q)
// (the one-pass read-out identity gdn.rs notes as exact), so the two
// reductions run side by side instead of one after the other.
//
// One CTA per (sequence, V head): it streams that head's D x D fp32 state
// (64 KB at D=128) into shared memory with eight 1-D bulk copies issued first
// thing, so the whole head is in flight while the prologue computes the conv,
// norms and gates; every global load of the prologue is issued in one round.
// Each row group is then updated in registers and written straight back to
// global memory with coalesced 16-byte stores.
//
// Conv state ownership: the q/k channels of K head kh are read by every V
// head mapped to kh (Hv/Hk CTAs). Those CTAs form one thread-block cluster;
// each reads the old conv state, arrives on the cluster barrier, and only the
// cluster's rank-0 CTA writes the new q/k conv state after waiting on it (from
// values it kept in registers). The v channels belong to one head and are
// written by its own CTA.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

constexpr int kDecodeThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kDecodeThreads) decode_step_kernel(const DecodeArgs p) {
  constexpr int NT = kDecodeThreads;
  constexpr int NW = NT / 32;
  constexpr int LPR = D / 16;             // lanes per state row (16 floats per lane)
  constexpr int RPW = 32 / LPR;           // rows per warp pass
  constexpr int NGROUPS = D / RPW;        // row groups of RPW rows
  constexpr int NCHUNK = 8;               // bulk loads per head
  constexpr int ROWS_PER_CHUNK = D / NCHUNK;
  constexpr uint32_t CHUNK_BYTES = ROWS_PER_CHUNK * D * 4;
  constexpr int NITEM = (3 * D + NT - 1) / NT;  // conv channels per thread
  static_assert(CHUNK_BYTES % 16 == 0, "bulk copy granularity");
  static_assert(2 * D <= NT, "each thread owns at most one q/k channel");

  extern __shared__ __align__(128) float sS[];  // D x D state tile
  __shared__ float sq[D], sk[D], sv[D], so[D];
  __shared__ float sred[3][NW];
  __shared__ __align__(8) uint64_t bars[NCHUNK];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bseq = blockIdx.y;
  const int kh = blockIdx.x / p.rep;
  const int r = blockIdx.x - kh * p.rep;
  const int h = p.map == GDN_MAP_TILED ? kh + r * p.Hk : blockIdx.x;
  float* gS = p.state + ((size_t)bseq * p.Hv + h) * (size_t)(D * D);

  if (tid == 0) {
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) mbar_init(&bars[c], 1);
    fence_mbar_init();
    fence_proxy_async_smem();
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) {
      mbar_arrive_expect_tx(&bars[c], CHUNK_BYTES);
      bulk_load(sS + c * ROWS_PER_CHUNK * D, gS + c * ROWS_PER_CHUNK * D, CHUNK_BYTES, &bars[c]);
    }
  }

  // ---- prologue, one round of global loads: gate scalars and conv inputs
  const int gi = bseq * p.Hv + h;
  const float a_raw = to_f32(static_cast<const T*>(p.a)[gi]);
  const float b_raw = to_f32(static_cast<const T*>(p.b)[gi]);
  const float dparam = p.decay_param[h], dtb = p.dt_bias[h];

  const size_t C = (size_t)p.C;
  const T* xrow = static_cast<const T*>(p.mixed_qkv) + (size_t)bseq * C;
  T* cstate = static_cast<T*>(p.conv_state) + (size_t)bseq * C * 3;
  const T* w = static_cast<const T*>(p.conv_w);
  const int qk_f = p.Hk * D;
  T cs0[NITEM], cs1[NITEM], cs2[NITEM], cx[NITEM], cw[NITEM][4];
  int chan[NITEM];
#pragma unroll
  for (int it = 0; it < NITEM; ++it) {
    const int idx = tid + it * NT;
    chan[it] = -1;
    if (idx < 3 * D) {
      const int which = idx / D, i = idx - which * D;
      const int c = which == 0 ? kh * D + i : which == 1 ? qk_f + kh * D + i : 2 * qk_f + h * D + i;
      chan[it] = c;
      cs0[it] = cstate[(size_t)c * 3 + 0];
      cs1[it] = cstate[(size_t)c * 3 + 1];
      cs2[it] = cstate[(size_t)c * 3 + 2];
      cx[it] = xrow[c];
#pragma unroll
      for (int j = 0; j < 4; ++j) cw[it][j] = w[(size_t)c * 4 + j];
    }
  }
  int qk_c = -1;
  T qk_s1 = T(), qk_s2 = T(), qk_x = T();
#pragma unroll
  for (int it = 0; it < NITEM; ++it) {
    const int idx = tid + it * NT;
    if (idx < 3 * D) {
      const int which = idx / D, i = idx - which * D;
      float acc = to_f32(cw[it][0]) * to_f32(cs0[it]);
      acc += to_f32(cw[it][1]) * to_f32(cs1[it]);
      acc += to_f32(cw[it][2]) * to_f32(cs2[it]);
      acc += to_f32(cw[it][3]) * to_f32(cx[it]);
      const float y = silu_f(acc);
      if (which == 2) {
        sv[i] = y;
        T* cp = cstate + (size_t)chan[it] * 3;  // v channels: this CTA is the only reader
        cp[0] = cs1[it];
        cp[1] = cs2[it];
        cp[2] = cx[it];
      } else {
        (which == 0 ? sq : sk)[i] = y;
        qk_c = chan[it];
        qk_s1 = cs1[it];
        qk_s2 = cs2[it];
        qk_x = cx[it];
      }
    }
  }
  // every CTA of the cluster has read the old q/k conv state after this
  cluster_arrive_release();
  __syncthreads();

  // ---- l2 norms of q and k and the k.q product, block-reduced; every thread
  // then forms the same scalars itself
  {
    float qq = 0.f, kk = 0.f, qk = 0.f;
    for (int i = tid; i < D; i += NT) {
      const float qv = sq[i], kv = sk[i];
      qq += qv * qv;
      kk += kv * kv;
      qk += qv * kv;
    }
    qq = group_sum<32>(qq);
    kk = group_sum<32>(kk);
    qk = group_sum<32>(qk);
    if (lane == 0) {
      sred[0][warp] = qq;
      sred[1][warp] = kk;
      sred[2][warp] = qk;
    }
  }
  __syncthreads();
  float qq = 0.f, kk = 0.f, qkr = 0.f;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    qq += sred[0][i];
    kk += sred[1][i];
    qkr += sred[2][i];
  }
  const float inv_q = 1.f / sqrtf(qq + p.l2_eps);
  const float inv_k = 1.f / sqrtf(kk + p.l2_eps);
  const float kq = qkr * inv_q * inv_k * p.scale;
  const float alpha = expf(gate_g(p.decay, dparam, dtb, a_raw));
  const float beta = sigmoid_f(b_raw);

  // ---- the state pass
  const int sub = lane % LPR, rq = lane / LPR;
  float kr[16], qr[16];
  {
    const float sqs = inv_q * p.scale;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = 4 * sub + 4 * LPR * m + e;
        kr[4 * m + e] = sk[col] * inv_k;
        qr[4 * m + e] = sq[col] * sqs;
      }
    }
  }
  bool ok = true;
  for (int grp = warp; grp < NGROUPS; grp += NW) {
    const int row0 = grp * RPW;
    if (!mbar_wait(&bars[row0 / ROWS_PER_CHUNK], 0)) {
      ok = false;
      break;
    }
    const int row = row0 + rq;
    const float* srow = sS + row * D;
    float4 s4[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
      s4[m] = *reinterpret_cast<const float4*>(srow + 4 * sub + 4 * LPR * m);
    float pk = 0.f, pq = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      pk = fmaf(s4[m].x, kr[4 * m + 0], pk);
      pq = fmaf(s4[m].x, qr[4 * m + 0], pq);
      pk = fmaf(s4[m].y, kr[4 * m + 1], pk);
      pq = fmaf(s4[m].y, qr[4 * m + 1], pq);
      pk = fmaf(s4[m].z, kr[4 * m + 2], pk);
      pq = fmaf(s4[m].z, qr[4 * m + 2], pq);
      pk = fmaf(s4[m].w, kr[4 * m + 3], pk);
      pq = fmaf(s4[m].w, qr[4 * m + 3], pq);
    }
    pk = group_sum<LPR>(pk);
    pq = group_sum<LPR>(pq);
    const float d = beta * (sv[row] - alpha * pk);
    const float o = fmaf(alpha, pq, d * kq);
    float* grow = gS + (size_t)row * D;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float4 n4;
      n4.x = fmaf(d, kr[4 * m + 0], alpha * s4[m].x);
      n4.y = fmaf(d, kr[4 * m + 1], alpha * s4[m].y);
      n4.z = fmaf(d, kr[4 * m + 2], alpha * s4[m].z);
      n4.w = fmaf(d, kr[4 * m + 3], alpha * s4[m].w);
      __stcs(reinterpret_cast<float4*>(grow + 4 * sub + 4 * LPR * m), n4);
    }
    if (sub == 0) so[row] = o;
  }
  const bool all_ok = __syncthreads_and(ok) != 0;

  // ---- outputs
  const size_t obase = ((size_t)bseq * p.Hv + h) * D;
  if (all_ok) {
    if (p.core_out != nullptr) {
      for (int j = tid; j < D; j += NT) p.core_out[obase + j] = so[j];
    }
    if (p.z != nullptr) {
      float ss = 0.f;
      for (int j = tid; j < D; j += NT) ss += so[j] * so[j];
      ss = group_sum<32>(ss);
      if (lane == 0) sred[0][warp] = ss;
      __syncthreads();
      float tot = 0.f;
#pragma unroll
      for (int i = 0; i < NW; ++i) tot += sred[0][i];
      const float inv = 1.f / sqrtf(tot / (float)D + p.rms_eps);
      const T* zr = static_cast<const T*>(p.z) + obase;
      T* outr = static_cast<T*>(p.out) + obase;
      for (int j = tid; j < D; j += NT) {
        const float y = so[j] * inv * p.norm_w[j] * silu_f(to_f32(zr[j]));
        outr[j] = from_f32<T>(y);
      }
    }
  }

  // ---- q/k conv state: written once per (sequence, K head), after every
  // CTA of the cluster has read the old values.
  cluster_wait_acquire();
  if (r == 0 && qk_c >= 0) {
    T* cp = cstate + (size_t)qk_c * 3;
    cp[0] = qk_s1;
    cp[1] = qk_s2;
    cp[2] = qk_x;
  }
}

template <typename T, int D>
static cudaError_t launch_decode_t(const DecodeArgs& p, int32_t batch, cudaStream_t stream) {
  auto kern = decode_step_kernel<T, D>;
  const int smem = D * D * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.Hv, (unsigned)batch, 1);
  cfg.blockDim = dim3(kDecodeThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.rep;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename T>
static cudaError_t launch_decode_d(const DecodeArgs& p, int32_t D, int32_t batch,
                                   cudaStream_t stream) {
  switch (D) {
    case 32: return launch_decode_t<T, 32>(p, batch, stream);
    case 64: return launch_decode_t<T, 64>(p, batch, stream);
    case 128: return launch_decode_t<T, 128>(p, batch, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const DecodeArgs& p, int32_t dtype, int32_t D, int32_t batch,
                          cudaStream_t stream) {
  switch (dtype) {
    case GDN_F16: return launch_decode_d<__half>(p, D, batch, stream);
    case GDN_BF16: return launch_decode_d<__nv_bfloat16>(p, D, batch, stream);
    case GDN_F32: return launch_decode_d<float>(p, D, batch, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(decode)
