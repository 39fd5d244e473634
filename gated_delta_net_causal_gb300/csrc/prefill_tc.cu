// Chunked prefill on the 5th-generation tensor cores (tcgen05, TMEM, TMA):
// head_dim 128, bf16/f16 activations, chunk 64.
//
// The same chunk algebra as the CUDA-core kernel (the recurrence of ferrox-core
// gdn.rs summed chunk-wise; the six stages of the Metal pipeline in
// ferrum-kernels gated_delta_attention_tests.rs `run_chunked_core`). Within a
// chunk of L tokens from state S0, with c the chunk-local cumulative decay,
// G_t = e^{c_t}, dl_t = e^{c_{L-1} - c_t}, and raw (unnormalised) k, q whose
// l2 scales invk_t, invq_t (q's includes 1/sqrt(D)) are folded into the
// small factors:
//   Gk  = K K^T, Pq = Q K^T                       bf16/f16 MMA, M=64 N=64 K=128
//   A   = beta_t e^{c_t-c_s} invk_t invk_s Gk     (s < t), Tm = (I + A)^{-1}
//   U   = Tm (diag(beta) V)                        tf32 MMA, M=64 N=32 K=64
//   W   = (Tm diag(beta G invk)) K                 tf32 MMA, M=64 N=128 K=64
//   Dm  = U - W S0^T                               tf32 MMA, M=64 N=32 K=128
//   O   = diag(G invq) Q S0^T + PM Dm,  PM = e^{c_t-c_s} invq_t invk_s Pq (s<=t)
//   S_L = G_{L-1} S0 + Dm^T diag(dl invk) K        tf32 MMA, M=128 N=32 K=64
// Decays enter only as e^{difference <= 0}.
//
// Operands live in shared memory as K-major 128-byte-swizzled tiles; raw k, q,
// v chunks arrive by TMA (k and q directly in the MMA layout), transposed fp32
// copies are written by the CUDA cores, and every accumulator lives in TMEM.
//
// Precision: raw bf16/f16 k, q, v are exact as tf32. Every other fp32 operand
// is rounded to nearest tf32 before the tensor cores see it, and the two
// products that carry the state forward, Tm diag(beta) V and K^T (dl invk Dm),
// are split as x = hi + lo (both tf32) into two MMAs each, which keeps them at
// fp32 accuracy. Q S0^T (output only) uses a 16-bit copy of the state.
// The fp32 master state stays in registers across chunks (thread owns one key
// column i of 16 value rows); its tf32 operand copy is rewritten each chunk.
//
// Grid (4 Dv slices of 32 rows, V head, sequence); the 4 slices of a head are
// one cluster, which only matters for the fused gated RMSNorm (per-row
// partial sums of squares exchanged through distributed shared memory).
#include <cuda.h>

#include <type_traits>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {

namespace {

constexpr int kTcC = 64;        // chunk
constexpr int kTcD = 128;       // head_dim
constexpr int kTcNS = 32;       // value rows per CTA
constexpr int kTcNSL = kTcD / kTcNS;
constexpr int kTcThreads = 256;

// dynamic shared memory layout (byte offsets from a 1024-aligned base)
constexpr uint32_t OFF_KBF = 0;          // k chunk, bf16 [64][128] SW128 (2 atoms)
constexpr uint32_t OFF_QBF = 16384;      // q chunk, bf16 [64][128]
constexpr uint32_t OFF_KT = 32768;       // fp32 [128 i][64 s] (k transposed)
constexpr uint32_t OFF_SB = 65536;       // io dtype [32 j][128 i] state copy for Q S0^T
constexpr uint32_t OFF_TAL = 73728;      // fp32 [64][64] low part of Tm diag(beta); the next
                                         // chunk's v lands here (row-major, 4 KB) after (D)
constexpr uint32_t OFF_DTLL = 90112;     // fp32 [32 j][64 s] low part of (dl invk Dm)^T
constexpr uint32_t OFF_VT = 98304;       // fp32 [32 j][64 s] (v transposed); later O staging
constexpr uint32_t OFF_TA = 106496;      // fp32 [64][64] Tm, then hi part of Tm diag(beta)
constexpr uint32_t OFF_TB = 122880;      // fp32 [64][64] A, then Tm diag(beta G invk)
constexpr uint32_t OFF_PM = 139264;      // fp32 [64][64]
constexpr uint32_t OFF_W = 155648;       // fp32 [64][128]
constexpr uint32_t OFF_SOP = 188416;     // fp32 [32 j][128 i] state operand
constexpr uint32_t OFF_DT = 204800;      // fp32 [32 j][64 s] Dm^T; block-inverse scratch in (C)
constexpr uint32_t OFF_DTL = 212992;     // fp32 [32 j][64 s] hi part of (dl invk Dm)^T
constexpr uint32_t SMEM_TILES = 221184;
constexpr uint32_t SMEM_DYN = SMEM_TILES + 1024;

// TMEM columns
constexpr uint32_t TM_G = 0, TM_P = 64, TM_U = 128, TM_W = 160, TM_WS = 288, TM_QS = 320,
                   TM_O = 352, TM_DS = 384, TM_COLS = 512;

__device__ __forceinline__ float* f32at(unsigned char* base, uint32_t off, int r, int k, int rows) {
  return reinterpret_cast<float*>(base + off + tc::sw128_offset(r, k, rows, 4));
}

__device__ __forceinline__ int64_t clamp_cu_tc(const int32_t* cu, int n, int64_t T) {
  int64_t v = cu[n];
  return v < 0 ? 0 : (v > T ? T : v);
}

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait(bar, parity);
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const PrefillArgs p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ float sg[kTcC], sbeta[kTcC], sc[kTcC], sgam[kTcC], sdl[kTcC], sinvk[kTcC],
      sinvq[kTcC];
  // per-row partial sums of squares of the output, from every slice of the
  // head (indexed by cluster rank), double-buffered by chunk parity
  __shared__ float snorm[2][kTcNSL][kTcC];
  __shared__ uint32_t s_tmem;
  __shared__ float sinv[kTcC];
  __shared__ __align__(8) uint64_t bar_k, bar_q, bar_v, bar_gp, bar_uw, bar_sq, bar_od;
  __shared__ __align__(8) uint64_t bar_norm[2];

  constexpr uint32_t kFmt = std::is_same<T, __half>::value ? tc::kF16 : tc::kBF16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qd = warp & 3, hh = warp >> 2;  // TMEM lane quadrant, column half
  const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int kh = k_head_of(p.map, h, p.Hk, p.rep);
  const int j0 = slice * kTcNS;
  const int64_t seq_s = clamp_cu_tc(p.cu_seqlens, n, p.T);
  int64_t seq_e = clamp_cu_tc(p.cu_seqlens, n + 1, p.T);
  if (seq_e < seq_s) seq_e = seq_s;
  const bool prenorm = (p.flags & GDN_QK_PRENORMALIZED) != 0;
  const bool pregate = (p.flags & GDN_GATES_PRECOMPUTED) != 0;
  const bool fused_norm = p.z != nullptr;

  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, TM_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_k, 1);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_gp, 1);
    mbar_init(&bar_uw, 1);
    mbar_init(&bar_sq, 1);
    mbar_init(&bar_od, 1);
    mbar_init(&bar_norm[0], 1);
    mbar_init(&bar_norm[1], 1);
    // armed for the first two chunks; each later use is re-armed right after
    // the previous one is consumed
    mbar_arrive_expect_tx(&bar_norm[0], (kTcNSL - 1) * kTcC * 4);
    mbar_arrive_expect_tx(&bar_norm[1], (kTcNSL - 1) * kTcC * 4);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  // state slice: thread owns key column i = 32 qd + lane of value rows
  // j0 + 16 hh .. +16 (fp32 master copy in registers) and writes its tf32
  // operand copy
  const int si = 32 * qd + lane;
  float* gS = p.state + (((size_t)n * p.Hv + h) * kTcD + j0) * kTcD;
  float sreg[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int j = 16 * hh + e;
    sreg[e] = gS[(size_t)j * kTcD + si];
    *f32at(sm, OFF_SOP, j, si, kTcNS) = tc::tf32_rna(sreg[e]);
    *reinterpret_cast<T*>(sm + OFF_SB + tc::sw128_offset(j, si, kTcNS, 2)) = from_f32<T>(sreg[e]);
  }
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // every CTA of the cluster has initialised its barriers before any peer
  // stores into its shared memory
  cluster_arrive_release();
  cluster_wait_acquire();
  const uint32_t tb = s_tmem;
  const uint32_t tq = tb + ((uint32_t)(32 * qd) << 16);  // this warp's TMEM quadrant

  const uint32_t a_kbf = smem_u32(sm + OFF_KBF), a_qbf = smem_u32(sm + OFF_QBF),
                 a_kt = smem_u32(sm + OFF_KT), a_sb = smem_u32(sm + OFF_SB),
                 a_tal = smem_u32(sm + OFF_TAL), a_dtll = smem_u32(sm + OFF_DTLL),
                 a_vt = smem_u32(sm + OFF_VT), a_ta = smem_u32(sm + OFF_TA),
                 a_tbm = smem_u32(sm + OFF_TB), a_pm = smem_u32(sm + OFF_PM),
                 a_w = smem_u32(sm + OFF_W), a_sop = smem_u32(sm + OFF_SOP),
                 a_dt = smem_u32(sm + OFF_DT), a_dtl = smem_u32(sm + OFF_DTL);

  // TMA issue helpers: each of k, q, v has its own barrier, completing once
  // per chunk, so the next chunk's tile is requested as soon as the current
  // one has been consumed
  auto issue_k = [&](int64_t c) {
    mbar_arrive_expect_tx(&bar_k, 16384u);
    tc::tma_load_2d(sm + OFF_KBF, &tm_k, kh * kTcD, (int)c, &bar_k);
    tc::tma_load_2d(sm + OFF_KBF + 8192, &tm_k, kh * kTcD + 64, (int)c, &bar_k);
  };
  auto issue_q = [&](int64_t c) {
    mbar_arrive_expect_tx(&bar_q, 16384u);
    tc::tma_load_2d(sm + OFF_QBF, &tm_q, kh * kTcD, (int)c, &bar_q);
    tc::tma_load_2d(sm + OFF_QBF + 8192, &tm_q, kh * kTcD + 64, (int)c, &bar_q);
  };
  auto issue_v = [&](int64_t c) {
    mbar_arrive_expect_tx(&bar_v, 4096u);
    tc::tma_load_2d(sm + OFF_TAL, &tm_v, h * kTcD + j0, (int)c, &bar_v);
  };
  if (tid == 0 && seq_s < seq_e) {
    issue_k(seq_s);
    issue_q(seq_s);
    issue_v(seq_s);
  }
  // raw gate inputs of the next chunk, prefetched into registers (tid < 64)
  float ga_next = 0.f, gb_next = 0.f;
  auto load_gates = [&](int64_t c) {
    ga_next = 0.f;
    gb_next = 0.f;
    if (tid < kTcC && c + tid < seq_e) {
      const int64_t gi = (c + tid) * p.Hv + h;
      if (pregate) {
        ga_next = static_cast<const float*>(p.a)[gi];
        gb_next = static_cast<const float*>(p.b)[gi];
      } else {
        ga_next = to_f32(static_cast<const T*>(p.a)[gi]);
        gb_next = to_f32(static_cast<const T*>(p.b)[gi]);
      }
    }
  };
  load_gates(seq_s);
  const float nw_j = fused_norm ? p.norm_w[j0 + (tid & 31)] : 0.f;
  const float gparam = pregate ? 0.f : p.decay_param[h];
  const float gdtb = pregate ? 0.f : p.dt_bias[h];
  const uint32_t my_rank = cluster_ctarank();

  int chunk = 0;
  for (int64_t c0 = seq_s; c0 < seq_e; c0 += kTcC, ++chunk) {
    const int L = (int)((seq_e - c0) < kTcC ? (seq_e - c0) : kTcC);
    const uint32_t par = (uint32_t)(chunk & 1);
    const int64_t c1 = c0 + kTcC;  // next chunk start
    const bool has_next = c1 < seq_e;

    // ---- (A) gates of this chunk (from the prefetched raw inputs)
    if (tid < kTcC) {
      float g = 0.f, bt = 0.f;
      if (tid < L) {
        if (pregate) {
          g = ga_next;
          bt = gb_next;
        } else {
          g = gate_g(p.decay, gparam, gdtb, ga_next);
          bt = sigmoid_f(gb_next);
        }
      }
      sg[tid] = g;
      sbeta[tid] = bt;
    }
    if (has_next) load_gates(c1);
    __syncthreads();
    if (warp < 2) {
      // inclusive prefix sum of g over the 64 tokens: two warp scans, then the
      // second half adds the first half's total
      float v = sg[tid];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      sc[tid] = v;
    }
    __syncthreads();
    if (warp == 1) sc[tid] += sc[31];
    tc_wait(&bar_k, par);
    tc_wait(&bar_q, par);
    tc_wait(&bar_v, par);
    __syncthreads();

    // ---- (B) K K^T and Q K^T on the tensor cores, straight from the TMA tiles
    if (tid == 0) {
      tc::fence_after_sync();
      const uint32_t id = tc::idesc(kFmt, 64, 64);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_f16(tb + TM_G, tc::sdesc_kstep(a_kbf, 64, s), tc::sdesc_kstep(a_kbf, 64, s), id,
                    s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_f16(tb + TM_P, tc::sdesc_kstep(a_qbf, 64, s), tc::sdesc_kstep(a_kbf, 64, s), id,
                    s > 0);
      tc::mma_commit(&bar_gp);
    }
    if (tid < kTcC) {
      sgam[tid] = expf(sc[tid]);
      sdl[tid] = tid < L ? expf(sc[L - 1] - sc[tid]) : 0.f;
    }
    // row norms of k and q and the K^T copy, 16 bytes at a time: four threads
    // per token row, each taking four 8-element chunks of k and of q
    {
      const int srow = tid >> 2, part = tid & 3;
      float kk = 0.f, qq = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int c16 = part + 4 * m;  // 16-byte chunk of the 256-byte row
        const uint32_t off = (uint32_t)((c16 >> 3) * (64 * 128) + (srow >> 3) * 1024 +
                                        (srow & 7) * 128 + (((c16 & 7) ^ (srow & 7)) << 4));
        const uint4 kr = *reinterpret_cast<const uint4*>(sm + OFF_KBF + off);
        const uint4 qr = *reinterpret_cast<const uint4*>(sm + OFF_QBF + off);
        const T* kv = reinterpret_cast<const T*>(&kr);
        const T* qv = reinterpret_cast<const T*>(&qr);
        const int i0 = 8 * c16;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float kf = to_f32(kv[e]), qf = to_f32(qv[e]);
          kk = fmaf(kf, kf, kk);
          qq = fmaf(qf, qf, qq);
          *f32at(sm, OFF_KT, i0 + e, srow, kTcD) = srow < L ? kf : 0.f;
        }
      }
      kk += __shfl_xor_sync(0xffffffffu, kk, 1);
      kk += __shfl_xor_sync(0xffffffffu, kk, 2);
      qq += __shfl_xor_sync(0xffffffffu, qq, 1);
      qq += __shfl_xor_sync(0xffffffffu, qq, 2);
      if (part == 0) {
        const bool live = srow < L;
        sinvk[srow] = live ? (prenorm ? 1.f : 1.f / sqrtf(kk + p.l2_eps)) : 0.f;
        sinvq[srow] = live ? (prenorm ? 1.f : 1.f / sqrtf(qq + p.l2_eps)) * p.scale : 0.f;
      }
      // V^T from the row-major staging copy: 8 values of one token row each
      const uint4 vr = *reinterpret_cast<const uint4*>(sm + OFF_TAL + (srow * kTcNS + 8 * part) * 2);
      const T* vv = reinterpret_cast<const T*>(&vr);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *f32at(sm, OFF_VT, 8 * part + e, srow, kTcNS) = srow < L ? to_f32(vv[e]) : 0.f;
    }
    __syncthreads();
    tc_wait(&bar_gp, par);
    tc::fence_after_sync();

    // ---- (C) A and PM from the tensor-core grams; Tm = (I + A)^{-1}
    // A and Tm are kept row-major (plain fp32 [64][64]) in the W tile's space,
    // which is free until (E); block products go through the Dm tiles' space.
    float* Ap = reinterpret_cast<float*>(sm + OFF_W);
    float* Tp = reinterpret_cast<float*>(sm + OFF_W + 16384);
    float* Xp = reinterpret_cast<float*>(sm + OFF_DT);
    {
      float gv[32], pv[32];
      tc::tmem_ld16(tq + TM_G + 32 * hh, *reinterpret_cast<float(*)[16]>(gv));
      tc::tmem_ld16(tq + TM_G + 32 * hh + 16, *reinterpret_cast<float(*)[16]>(gv + 16));
      tc::tmem_ld16(tq + TM_P + 32 * hh, *reinterpret_cast<float(*)[16]>(pv));
      tc::tmem_ld16(tq + TM_P + 32 * hh + 16, *reinterpret_cast<float(*)[16]>(pv + 16));
      tc::tmem_wait_ld();
      if (lane < 16) {
        const int t = 16 * qd + lane;
        const bool live = t < L;
        constexpr float kLog2e = 1.4426950408889634f;
        const float ct = sc[t] * kLog2e, bt = sbeta[t], ikt = sinvk[t], iqt = sinvq[t];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int s = 32 * hh + e;
          const float dec = exp2f(ct - sc[s] * kLog2e);  // e^{c_t - c_s} <= 1 for s <= t
          const float ks = sinvk[s];
          Ap[t * kTcC + s] = (live && s < t) ? bt * dec * gv[e] * ikt * ks : 0.f;
          *f32at(sm, OFF_PM, t, s, kTcC) = (live && s <= t) ? tc::tf32_rna(dec * pv[e] * iqt * ks) : 0.f;
        }
      }
    }
    __syncthreads();
    if (tid == 0 && has_next) issue_k(c1);  // K K^T, Q K^T done; the K copy is made
    // diagonal 16x16 blocks: warp b inverts block b by forward substitution,
    // lane l holding column 16b + l in registers
    if (warp < 4) {
      const int b0 = 16 * warp, l = lane & 15;
      float x[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) x[m] = (m == l) ? 1.f : 0.f;
#pragma unroll
      for (int m = 1; m < 16; ++m) {
        const float* arow = Ap + (b0 + m) * kTcC + b0;
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < m; ++r) acc = fmaf(arow[r], x[r], acc);
        if (m > l) x[m] = -acc;
      }
      if (lane < 16) {
#pragma unroll
        for (int m = 0; m < 16; ++m) Tp[(b0 + m) * kTcC + b0 + l] = x[m];
      }
    }
    __syncthreads();
    // off-diagonal blocks, one block diagonal at a time:
    //   T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj
    for (int d = 1; d < 4; ++d) {
      const int nblk = 4 - d;
      for (int e = tid; e < nblk * 256; e += kTcThreads) {
        const int jb = e >> 8, rr = (e >> 4) & 15, cc = e & 15, ib = jb + d;
        float acc = 0.f;
        for (int kb = jb; kb < ib; ++kb) {
          const float* arow = Ap + (16 * ib + rr) * kTcC + 16 * kb;
          const float* tcol = Tp + (16 * kb) * kTcC + 16 * jb + cc;
#pragma unroll
          for (int m = 0; m < 16; ++m) acc = fmaf(arow[m], tcol[m * kTcC], acc);
        }
        Xp[e] = acc;
      }
      __syncthreads();
      for (int e = tid; e < nblk * 256; e += kTcThreads) {
        const int jb = e >> 8, rr = (e >> 4) & 15, cc = e & 15, ib = jb + d;
        const float* trow = Tp + (16 * ib + rr) * kTcC + 16 * ib;
        const float* xcol = Xp + (jb << 8) + cc;
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = (m <= rr) ? fmaf(trow[m], xcol[m << 4], acc) : acc;
        Tp[(16 * ib + rr) * kTcC + 16 * jb + cc] = -acc;
      }
      __syncthreads();
    }
    // TA/TAL = hi/lo of Tm diag(beta); TB = Tm diag(beta G invk); zero above
    // the diagonal
    for (int e = tid; e < kTcC * kTcC; e += kTcThreads) {
      const int t = e / kTcC, s = e - (e / kTcC) * kTcC;
      const float tv = s <= t ? Tp[e] : 0.f;
      const float ta = tv * sbeta[s];
      const float hi = tc::tf32_rna(ta);
      *f32at(sm, OFF_TA, t, s, kTcC) = hi;
      *f32at(sm, OFF_TAL, t, s, kTcC) = tc::tf32_rna(ta - hi);
      *f32at(sm, OFF_TB, t, s, kTcC) = tc::tf32_rna(tv * sbeta[s] * sgam[s] * sinvk[s]);
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // ---- (D) U = Tm (beta V), W = (Tm diag(beta G invk)) K
    if (tid == 0) {
      tc::fence_after_sync();
      const uint32_t idu = tc::idesc(tc::kTF32, 64, 32), idw = tc::idesc(tc::kTF32, 64, 128);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_tf32(tb + TM_U, tc::sdesc_kstep(a_ta, 64, s), tc::sdesc_kstep(a_vt, 32, s), idu,
                     s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_tf32(tb + TM_U, tc::sdesc_kstep(a_tal, 64, s), tc::sdesc_kstep(a_vt, 32, s), idu,
                     true);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_tf32(tb + TM_W, tc::sdesc_kstep(a_tbm, 64, s), tc::sdesc_kstep(a_kt, 128, s), idw,
                     s > 0);
      tc::mma_commit(&bar_uw);
    }
    tc_wait(&bar_uw, par);
    tc::fence_after_sync();
    if (tid == 0 && has_next) issue_v(c1);  // the low part of Tm diag(beta) has been read

    // ---- (E) W to shared memory as the A operand of W S0^T
    {
      float wv[64];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        tc::tmem_ld16(tq + TM_W + 64 * hh + 16 * q4, *reinterpret_cast<float(*)[16]>(wv + 16 * q4));
      tc::tmem_wait_ld();
      if (lane < 16) {
        const int t = 16 * qd + lane;
#pragma unroll
        for (int e = 0; e < 64; ++e) *f32at(sm, OFF_W, t, 64 * hh + e, kTcC) = tc::tf32_rna(wv[e]);
      }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // ---- (F) W S0^T and Q S0^T (the state enters here)
    if (tid == 0) {
      tc::fence_after_sync();
      const uint32_t id = tc::idesc(tc::kTF32, 64, 32);
#pragma unroll
      for (int s = 0; s < 16; ++s)
        tc::mma_tf32(tb + TM_WS, tc::sdesc_kstep(a_w, 64, s), tc::sdesc_kstep(a_sop, 32, s), id,
                     s > 0);
      const uint32_t idq = tc::idesc(kFmt, 64, 32);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_f16(tb + TM_QS, tc::sdesc_kstep(a_qbf, 64, s), tc::sdesc_kstep(a_sb, 32, s), idq,
                    s > 0);
      tc::mma_commit(&bar_sq);
    }
    tc_wait(&bar_sq, par);
    tc::fence_after_sync();
    if (tid == 0 && has_next) issue_q(c1);  // Q S0^T done

    // ---- (G) Dm = U - W S0^T (transposed, twice scaled); inter-chunk output
    float oi[16];
    {
      float uv[16], wsv[16], qsv[16];
      tc::tmem_ld16(tq + TM_U + 16 * hh, uv);
      tc::tmem_ld16(tq + TM_WS + 16 * hh, wsv);
      tc::tmem_ld16(tq + TM_QS + 16 * hh, qsv);
      tc::tmem_wait_ld();
      const int t = 16 * qd + (lane & 15);
      const float gq = sgam[t] * sinvq[t], dk = sdl[t] * sinvk[t];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float dm = uv[e] - wsv[e];
        oi[e] = gq * qsv[e];
        if (lane < 16) {
          const int j = 16 * hh + e;
          *f32at(sm, OFF_DT, j, t, kTcNS) = tc::tf32_rna(dm);
          const float dt = dk * dm, dhi = tc::tf32_rna(dt);
          *f32at(sm, OFF_DTL, j, t, kTcNS) = dhi;
          *f32at(sm, OFF_DTLL, j, t, kTcNS) = tc::tf32_rna(dt - dhi);
        }
      }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // ---- (H) O = PM Dm (intra-chunk), dS^T = K^T (dl invk Dm)
    if (tid == 0) {
      tc::fence_after_sync();
      const uint32_t ido = tc::idesc(tc::kTF32, 64, 32), ids = tc::idesc(tc::kTF32, 128, 32);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_tf32(tb + TM_O, tc::sdesc_kstep(a_pm, 64, s), tc::sdesc_kstep(a_dt, 32, s), ido,
                     s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_tf32(tb + TM_DS, tc::sdesc_kstep(a_kt, 128, s), tc::sdesc_kstep(a_dtl, 32, s),
                     ids, s > 0);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_tf32(tb + TM_DS, tc::sdesc_kstep(a_kt, 128, s), tc::sdesc_kstep(a_dtll, 32, s),
                     ids, true);
      tc::mma_commit(&bar_od);
    }
    // z for this thread's output elements (row e / 32, column tid % 32), loaded
    // while the last MMAs of the chunk run
    T zpre[kTcC * kTcNS / kTcThreads];
    if (fused_norm) {
      const T* zg = static_cast<const T*>(p.z);
#pragma unroll
      for (int m = 0; m < kTcC * kTcNS / kTcThreads; ++m) {
        const int e = tid + kTcThreads * m;
        const int t = e / kTcNS;
        zpre[m] = t < L ? zg[((c0 + t) * p.Hv + h) * kTcD + j0 + (e % kTcNS)] : T();
      }
    }
    tc_wait(&bar_od, par);
    tc::fence_after_sync();

    // ---- (I) state update (registers + operand copy) and outputs
    {
      float dsv[16], ov[16];
      tc::tmem_ld16(tq + TM_DS + 16 * hh, dsv);
      tc::tmem_ld16(tq + TM_O + 16 * hh, ov);
      tc::tmem_wait_ld();
      const float gl = sgam[L - 1];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        sreg[e] = fmaf(gl, sreg[e], dsv[e]);
        *f32at(sm, OFF_SOP, 16 * hh + e, si, kTcNS) = tc::tf32_rna(sreg[e]);
        *reinterpret_cast<T*>(sm + OFF_SB + tc::sw128_offset(16 * hh + e, si, kTcNS, 2)) =
            from_f32<T>(sreg[e]);
      }
      if (lane < 16) {
        const int t = 16 * qd + lane;
        float* ostage = reinterpret_cast<float*>(sm + OFF_VT);  // [64][32] plain
#pragma unroll
        for (int e = 0; e < 16; ++e) ostage[t * kTcNS + 16 * hh + e] = ov[e] + oi[e];
      }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    {
      const float* ostage = reinterpret_cast<const float*>(sm + OFF_VT);
      if (p.core_out != nullptr) {
        for (int e = tid; e < L * kTcNS; e += kTcThreads) {
          const int t = e / kTcNS, j = e - (e / kTcNS) * kTcNS;
          p.core_out[((c0 + t) * p.Hv + h) * kTcD + j0 + j] = ostage[e];
        }
      }
      if (fused_norm) {
        const int buf = chunk & 1;
        // partial sums of squares of this slice's 32 columns, per row, sent to
        // every CTA of the cluster (own slot written locally); each CTA waits
        // for its three peers' 64 x 4 bytes on its own mbarrier
        for (int t = warp; t < kTcC; t += kTcThreads / 32) {
          float v = ostage[t * kTcNS + lane];
          v = group_sum<32>(v * v);
          if (lane < kTcNSL) {
            const uint32_t slot = smem_u32(&snorm[buf][my_rank][t]);
            if ((uint32_t)lane == my_rank) {
              snorm[buf][my_rank][t] = v;
            } else {
              st_async_cluster_f32(map_shared_rank(slot, lane), v,
                                   map_shared_rank(smem_u32(&bar_norm[buf]), lane));
            }
          }
        }
        tc_wait(&bar_norm[buf], (uint32_t)((chunk >> 1) & 1));
        __syncthreads();
        if (tid < kTcC) {
          float tot = 0.f;
#pragma unroll
          for (int r = 0; r < kTcNSL; ++r) tot += snorm[buf][r][tid];
          sinv[tid] = 1.f / sqrtf(tot / (float)kTcD + p.rms_eps);
        }
        __syncthreads();
        if (tid == 0) mbar_arrive_expect_tx(&bar_norm[buf], (kTcNSL - 1) * kTcC * 4);
        T* og = static_cast<T*>(p.out);
#pragma unroll
        for (int m = 0; m < kTcC * kTcNS / kTcThreads; ++m) {
          const int e = tid + kTcThreads * m;
          const int t = e / kTcNS;
          if (t < L) {
            const int64_t oi2 = ((c0 + t) * p.Hv + h) * kTcD + j0 + (e % kTcNS);
            og[oi2] = from_f32<T>(ostage[e] * sinv[t] * nw_j * silu_f(to_f32(zpre[m])));
          }
        }
      }
    }
    __syncthreads();  // the staging buffer and gate arrays are rewritten next chunk
  }

  // write the state back
#pragma unroll
  for (int e = 0; e < 16; ++e) gS[(size_t)(16 * hh + e) * kTcD + si] = sreg[e];
  if (fused_norm) {
    cluster_arrive_release();
    cluster_wait_acquire();
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, TM_COLS);
}

template <typename T>
cudaError_t launch_tc_t(const PrefillArgs& p, cudaStream_t stream) {
  const CUtensorMapDataType dt =
      std::is_same<T, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap mq, mk, mv;
  const int64_t qkc = (int64_t)p.Hk * kTcD, vc = (int64_t)p.Hv * kTcD;
  if (!tc::make_map_2d(&mq, p.q, p.T, qkc, p.q_stride, 2, dt, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_map_2d(&mk, p.k, p.T, qkc, p.k_stride, 2, dt, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_map_2d(&mv, p.v, p.T, vc, p.v_stride, 2, dt, kTcNS, 64, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  auto kern = prefill_tc_kernel<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_DYN);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)kTcNSL, (unsigned)p.Hv, (unsigned)p.N);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_DYN;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)kTcNSL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, mq, mk, mv);
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs& p, int32_t dtype, int32_t D) {
  if (D != kTcD || (dtype != GDN_BF16 && dtype != GDN_F16)) return false;
  if (p.T >= ((int64_t)1 << 31)) return false;  // TMA row coordinate is int32
  return tc::encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const PrefillArgs& p, int32_t dtype, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  return dtype == GDN_F16 ? launch_tc_t<__half>(p, stream) : launch_tc_t<__nv_bfloat16>(p, stream);
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(prefill_tc)
