// Chunk-parallel prefill on the 5th-generation tensor cores: head_dim 128,
// bf16 activations, chunk 64, three launches over a caller-provided
// workspace.
//
// The chunk algebra is the one of the single-pass kernel (the recurrence of
// ferrox-core gdn.rs summed chunk-wise; the stages of ferrum-kernels
// gated_delta_attention_tests.rs `run_chunked_core`), split by what depends on
// the state. Within a chunk of L tokens from state S (rows j = value, columns
// i = key), with c the chunk-local cumulative decay, G_t = e^{c_t}, raw k, q
// and their l2 scales rk_t, rq_t (rq includes 1/sqrt(D)):
//
//   state-free, every chunk at once (cp_prep_kernel, one CTA per chunk and
//   K head, looping over the V heads that read it):
//     A   = beta_t e^{c_t-c_s} rk_t rk_s (k_t . k_s)            (s < t)
//     Tb  = (I + A)^{-1} diag(beta)                              -> hi + lo bf16
//     P   = e^{c_t-c_s} rq_t rk_s (q_t . k_s)                    (s <= t) -> bf16
//     ak_t = G_t rk_t,  dk_t = e^{c_{L-1}-c_t} rk_t,  gq_t = G_t rq_t,  G_{L-1}
//   the carry, one CTA per (V head, sequence), chunk after chunk
//   (cp_chain_kernel; the state lives in TMEM as an fp32 accumulator):
//     KS^T = S K^T                  R^T[j][s] = v_s[j] - ak_s KS^T[j][s]
//     Dm^T = R^T Tb^T               (the chunk's delta-rule corrections d_t)
//     S    = G_{L-1} S + (Dm diag(dk))^T K
//     O^T  = S Q^T diag(gq) + Dm^T P^T, then the gated RMSNorm over j.
//
// Every product that carries the state forward (S K^T, R Tb^T, Dm^T K) keeps
// fp32 accuracy on bf16 tensor cores by splitting the fp32 factor as
// x = hi + lo (two bf16 values, about 16 significant bits together): S and
// Dm' are split, raw k is exact in bf16, and R Tb^T uses hi*hi + hi*lo +
// lo*hi. The two output products (S Q^T, Dm P^T) use the hi parts only.
//
// Because the carry CTA owns all 128 value rows of its head, the gated
// RMSNorm of each output row is a reduction inside the CTA: no cluster.
#include <cuda.h>
#include <string.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {

namespace {

constexpr int kC = 64;   // chunk
constexpr int kD = 128;  // head_dim
constexpr int kPrepThreads = 256;
constexpr int kCarryThreads = 256;  // warps 0-7: the state carry (two threads per value row)
constexpr int kChainThreads = 512;  // warps 8-15: output and gated norm
constexpr int kAStride = kC + 1;    // padded row pitch of the fp32 A matrix
constexpr int kMaxRep = 8;          // V heads per K head on this path

// ---------------------------------------------------------------- workspace

struct CpWork {
  int32_t* cs;         // [N+1] first chunk slot of each sequence
  __nv_bfloat16* tw;   // [3][G*Hv*64][64]: Tb hi, Tb lo, P (row-major per slot)
  __nv_bfloat16* kt;   // [G*Hk*128][64]: raw k transposed, rows t >= L zero
  float* vec;          // [G*Hv][4][64]: ak, dk, gq, {G_{L-1}, 0...}
  int64_t G;           // chunk slots
};

struct CpLayout {
  int64_t G;
  size_t off_tm, off_kt, off_vec, total;
};

CpLayout cp_layout(int32_t N, int64_t T, int32_t Hk, int32_t Hv) {
  CpLayout l{};
  // sum over sequences of ceil(len/64) <= (T + 63 N) / 64
  l.G = T > 0 ? (T + 63 * (int64_t)N) / kC : 0;
  l.off_tm = ((size_t)4 * ((size_t)N + 1) + 1023) / 1024 * 1024;
  l.off_kt = l.off_tm + (size_t)3 * l.G * Hv * kC * kC * 2;
  l.off_vec = l.off_kt + (size_t)l.G * Hk * kD * kC * 2;
  l.total = l.off_vec + (size_t)l.G * Hv * 4 * kC * 4;
  return l;
}

__device__ __forceinline__ void seq_range(const PrefillArgs& p, int n, int64_t& s, int64_t& e) {
  int64_t a = p.cu_seqlens[n], b = p.cu_seqlens[n + 1];
  a = a < 0 ? 0 : (a > p.T ? p.T : a);
  b = b < 0 ? 0 : (b > p.T ? p.T : b);
  s = a;
  e = b < a ? a : b;
}

// named barrier with an OR-reduced predicate over `count` threads
__device__ __forceinline__ bool bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void bar_named(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Byte offset of 16-byte chunk c (along K) of row r in a K-major SW128 bf16
// tile of `rows` rows (64 elements per atom).
__device__ __forceinline__ uint32_t sw_chunk(int r, int c, int rows) {
  return (uint32_t)((c >> 3) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                    (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 8 fp32 values -> their bf16 hi parts and the bf16 rounding of the remainders
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * m], x[2 * m + 1]);
    h[m] = *reinterpret_cast<const uint32_t*>(&hv);
    l[m] = pack_bf16(x[2 * m] - __low2float(hv), x[2 * m + 1] - __high2float(hv));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// ------------------------------------------------------------ chunk index

// cs[n] = sum_{m<n} ceil(len_m / 64), cs[N] = total (clamped to G + 1 so a
// cu_seqlens that overlaps itself is caught, not overflowed). One block of
// 1024 threads.
__global__ void __launch_bounds__(1024) cp_index_kernel(const PrefillArgs p, const CpWork w) {
  __shared__ int64_t swarp[32];
  __shared__ int64_t scarry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) scarry = 0;
  __syncthreads();
  for (int base = 0; base < p.N; base += 1024) {
    const int n = base + tid;
    int64_t cnt = 0;
    if (n < p.N) {
      int64_t s, e;
      seq_range(p, n, s, e);
      cnt = (e - s + kC - 1) / kC;
    }
    int64_t v = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) swarp[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int64_t x = swarp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t u = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += u;
      }
      swarp[lane] = x;
    }
    __syncthreads();
    const int64_t excl = scarry + (warp > 0 ? swarp[warp - 1] : 0) + v - cnt;
    if (n < p.N) w.cs[n] = (int32_t)(excl < w.G + 1 ? excl : w.G + 1);
    __syncthreads();
    if (tid == 1023) scarry = excl + cnt;
    __syncthreads();
  }
  if (tid == 0) w.cs[p.N] = (int32_t)(scarry < w.G + 1 ? scarry : w.G + 1);
}

// ------------------------------------------------------------------ prep

// The k and q tile is dead once the grams have completed and K^T and the l2
// scales are taken from it; the per-V-head matrices then reuse its space.
constexpr uint32_t P_OFF_KQ = 0;       // bf16 [128][128 i] SW128 (TMA): rows 0-63 k, 64-127 q
constexpr uint32_t P_OFF_A = 0;        // fp32 [64][65]
constexpr uint32_t P_OFF_T = 16640;    // fp32 [64][64] Tm (products in its upper triangle)
constexpr uint32_t P_SMEM = 33024 + 1024;

__global__ void __launch_bounds__(kPrepThreads, 4)
    cp_prep_kernel(const PrefillArgs p, const CpWork w, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(16) float sinvk[kC], sinvq[kC];
  // raw gate inputs, then per V head: beta, the chunk-local cumulative decay
  // c and G = e^c
  __shared__ __align__(16) float sga[kMaxRep][kC], sgb[kMaxRep][kC], sbeta[kMaxRep][kC],
      sc[kMaxRep][kC], sgam[kMaxRep][kC];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t bar_ld, bar_gp;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qd = warp & 3;
  const int64_t g = blockIdx.x;
  const int kh = blockIdx.y;
  const int64_t total = w.cs[p.N] < w.G ? w.cs[p.N] : w.G;
  if (g >= total) return;
  // the sequence owning slot g: the last n with cs[n] <= g
  int lo = 0, hi = p.N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (w.cs[mid] <= g) lo = mid; else hi = mid - 1;
  }
  const int n = lo;
  int64_t seq_s, seq_e;
  seq_range(p, n, seq_s, seq_e);
  const int64_t c0 = seq_s + (int64_t)kC * (g - w.cs[n]);
  const int L = (int)((seq_e - c0) < kC ? (seq_e - c0) : kC);
  const bool prenorm = (p.flags & GDN_QK_PRENORMALIZED) != 0;
  const bool pregate = (p.flags & GDN_GATES_PRECOMPUTED) != 0;

  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, 64);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_gp, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar_ld, 32768u);
    tc::tma_load_2d(sm + P_OFF_KQ, &tm_k, kh * kD, (int)c0, &bar_ld);
    tc::tma_load_2d(sm + P_OFF_KQ + 16384, &tm_k, kh * kD + 64, (int)c0, &bar_ld);
    tc::tma_load_2d(sm + P_OFF_KQ + 8192, &tm_q, kh * kD, (int)c0, &bar_ld);
    tc::tma_load_2d(sm + P_OFF_KQ + 24576, &tm_q, kh * kD + 64, (int)c0, &bar_ld);
  }
  // raw gate inputs of every V head reading this K head, fetched while the
  // k and q tiles are in flight
  for (int e = tid; e < p.rep * kC; e += kPrepThreads) {
    const int r = e >> 6, t = e & 63;
    const int h = p.map == GDN_MAP_GROUPED ? kh * p.rep + r : kh + r * p.Hk;
    float ga = 0.f, gb = 0.f;
    if (t < L) {
      const int64_t gi = (c0 + t) * p.Hv + h;
      if (pregate) {
        ga = static_cast<const float*>(p.a)[gi];
        gb = static_cast<const float*>(p.b)[gi];
      } else {
        ga = __bfloat162float(static_cast<const __nv_bfloat16*>(p.a)[gi]);
        gb = __bfloat162float(static_cast<const __nv_bfloat16*>(p.b)[gi]);
      }
    }
    sga[r][t] = ga;
    sgb[r][t] = gb;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = s_tmem;
  const uint32_t tq = tb + ((uint32_t)(32 * qd) << 16);
  const uint64_t d_kq = tc::sdesc_sw128(smem_u32(sm + P_OFF_KQ));

  bool to = !mbar_wait(&bar_ld, 0);
  if (tid == 0 && !to) {
    tc::fence_after_sync();
    // [k; q] k^T as one M=128 accumulator: rows 0-63 K K^T, rows 64-127 Q K^T
    const uint32_t id = tc::idesc(tc::kBF16, 128, 64);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      tc::mma_f16(tb, tc::sdesc_at(d_kq, 128, s), tc::sdesc_at(d_kq, 128, s), id, s > 0);
    tc::mma_commit(&bar_gp);
  }
  // l2 scales of k and q rows, four threads per row, 16 bytes at a time
  {
    const int srow = tid >> 2, part = tid & 3;
    float kk = 0.f, qq = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int c16 = part + 4 * m;
      const uint4 kr = *reinterpret_cast<const uint4*>(sm + P_OFF_KQ + sw_chunk(srow, c16, 128));
      const uint4 qr = *reinterpret_cast<const uint4*>(sm + P_OFF_KQ + sw_chunk(64 + srow, c16, 128));
      const __nv_bfloat16* kv = reinterpret_cast<const __nv_bfloat16*>(&kr);
      const __nv_bfloat16* qv = reinterpret_cast<const __nv_bfloat16*>(&qr);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float kf = __bfloat162float(kv[e]), qf = __bfloat162float(qv[e]);
        kk = fmaf(kf, kf, kk);
        qq = fmaf(qf, qf, qq);
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
  }
  // K^T of this chunk and K head for the carry's state update: thread pair
  // (i, half) gathers 32 rows t of column i
  {
    const int i = tid >> 1, th = tid & 1;
    const uint32_t col = (uint32_t)((i >> 6) * 16384 + (i & 7) * 2);
    const int ic = (i & 63) >> 3;
    uint32_t wv[16];
#pragma unroll
    for (int t2 = 0; t2 < 16; ++t2) {
      uint32_t pr = 0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int t = 32 * th + 2 * t2 + q;
        const uint32_t off = col + (uint32_t)((t >> 3) * 1024 + (t & 7) * 128 + ((ic ^ (t & 7)) << 4));
        const uint32_t x = *reinterpret_cast<const unsigned short*>(sm + P_OFF_KQ + off);
        pr |= (t < L ? x : 0u) << (16 * q);
      }
      wv[t2] = pr;
    }
    uint4* dst = reinterpret_cast<uint4*>(w.kt + ((g * p.Hk + kh) * kD + i) * kC + 32 * th);
#pragma unroll
    for (int c = 0; c < 4; ++c) dst[c] = make_uint4(wv[4 * c], wv[4 * c + 1], wv[4 * c + 2], wv[4 * c + 3]);
  }
  if (!to) to = !mbar_wait(&bar_gp, 0);
  if (__syncthreads_or(to)) {
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, 64);
    return;
  }
  tc::fence_after_sync();

  // the gates of every V head reading this K head at once: two warps per
  // head (32 tokens each) take g and beta and scan g; then the second half
  // adds the first half's total, and G = e^c
  for (int r0 = 0; r0 < p.rep; r0 += kPrepThreads / kC) {
    const int r = r0 + (warp >> 1), t = 32 * (warp & 1) + lane;
    if (r < p.rep) {
      const int h = p.map == GDN_MAP_GROUPED ? kh * p.rep + r : kh + r * p.Hk;
      float gt = 0.f, bt = 0.f;
      if (t < L) {
        if (pregate) {
          gt = sga[r][t];
          bt = sgb[r][t];
        } else {
          gt = gate_g(p.decay, p.decay_param[h], p.dt_bias[h], sga[r][t]);
          bt = sigmoid_f(sgb[r][t]);
        }
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, gt, o);
        if (lane >= o) gt += u;
      }
      sc[r][t] = gt;
      sbeta[r][t] = bt;
    }
  }
  __syncthreads();
  for (int e = tid; e < p.rep * kC; e += kPrepThreads) {
    const int r = e >> 6, t = e & 63;
    if (t >= 32) sc[r][t] += sc[r][31];
  }
  __syncthreads();
  for (int e = tid; e < p.rep * kC; e += kPrepThreads) {
    const int r = e >> 6, t = e & 63;
    sgam[r][t] = expf(sc[r][t]);
  }
  __syncthreads();

  float* Ap = reinterpret_cast<float*>(sm + P_OFF_A);
  float* Tp = reinterpret_cast<float*>(sm + P_OFF_T);
  const size_t HvG = (size_t)w.G * p.Hv;
  for (int r = 0; r < p.rep; ++r) {
    const int h = p.map == GDN_MAP_GROUPED ? kh * p.rep + r : kh + r * p.Hk;
    const size_t slot = (size_t)g * p.Hv + h;
    // A (padded rows) and P (bf16, straight to the workspace) from the grams
    // of this K head, read again for each V head: thread (row, half) takes
    // 32 columns of row `row` of the M=128 accumulator (lane = row), A for
    // rows 0-63 and P for rows 64-127
    {
      const int row = tid & 127, hc = tid >> 7;
      float gv[32];
      tc::tmem_ld16(tq + 32 * hc, *reinterpret_cast<float(*)[16]>(gv));
      tc::tmem_ld16(tq + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(gv + 16));
      tc::tmem_wait_ld();
      const bool is_a = row < kC;  // warp-uniform
      const int t = is_a ? row : row - kC;
      const bool live = t < L;
      constexpr float kLog2e = 1.4426950408889634f;
      const float ct = sc[r][t] * kLog2e;
      // e^{c_t - c_s} (<= 1 for s <= t) times rk_s for this thread's 32
      // columns s, four at a time from 16-byte loads of the per-token vectors
      float pr[32];
#pragma unroll
      for (int m4 = 0; m4 < 8; ++m4) {
        const float4 c4 = *reinterpret_cast<const float4*>(&sc[r][32 * hc + 4 * m4]);
        const float4 k4 = *reinterpret_cast<const float4*>(&sinvk[32 * hc + 4 * m4]);
        const float cv[4] = {c4.x, c4.y, c4.z, c4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = 4 * m4 + u, s = 32 * hc + e;
          pr[e] = (live && s <= t) ? exp2f(ct - cv[u] * kLog2e) * kv[u] * gv[e] : 0.f;
        }
      }
      if (is_a) {
        const float bk = sbeta[r][t] * sinvk[t];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int s = 32 * hc + e;
          Ap[t * kAStride + s] = s < t ? bk * pr[e] : 0.f;
        }
      } else {
        const float iqt = sinvq[t];
#pragma unroll
        for (int e = 0; e < 32; ++e) pr[e] *= iqt;
        uint4* dst = reinterpret_cast<uint4*>(w.tw + ((2 * HvG + slot) * kC + t) * kC + 32 * hc);
#pragma unroll
        for (int m = 0; m < 4; ++m)
          dst[m] = make_uint4(pack_bf16(pr[8 * m], pr[8 * m + 1]), pack_bf16(pr[8 * m + 2], pr[8 * m + 3]),
                              pack_bf16(pr[8 * m + 4], pr[8 * m + 5]),
                              pack_bf16(pr[8 * m + 6], pr[8 * m + 7]));
      }
    }
    __syncthreads();
    // (I + A)^{-1}: diagonal 16x16 blocks by forward substitution (warp b,
    // lane l holds column l of block b; zeros above the diagonal written)
    if (warp < 4) {
      const int b0 = 16 * warp, l = lane & 15;
      float x[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) x[m] = (m == l) ? 1.f : 0.f;
#pragma unroll
      for (int m = 1; m < 16; ++m) {
        const float* arow = Ap + (b0 + m) * kAStride + b0;
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < m; ++q) acc = fmaf(arow[q], x[q], acc);
        if (m > l) x[m] = -acc;
      }
      if (lane < 16) {
#pragma unroll
        for (int m = 0; m < 16; ++m) Tp[(b0 + m) * kC + b0 + l] = x[m];
      }
    } else {
      // zeros above the diagonal in the two 32x32 diagonal blocks too (rows
      // 0-15 x columns 16-31 and rows 32-47 x columns 48-63), so the doubling
      // below runs fixed-length loops over whole blocks
      const int e = tid - 128, zr = e >> 3, zc = (e & 7) * 2;
      *reinterpret_cast<float2*>(Tp + zr * kC + 16 + zc) = make_float2(0.f, 0.f);
      *reinterpret_cast<float2*>(Tp + (32 + zr) * kC + 48 + zc) = make_float2(0.f, 0.f);
    }
    __syncthreads();
    // The rest by doubling, T = [[T1, 0], [-T2 A21 T1, T2]] for the lower
    // triangular blocks: first both 32x32 diagonal blocks from their 16x16
    // ones, then the whole 64x64 from the two 32x32. Each product X = A21 T1
    // is kept in the (otherwise unused) upper-right 32x32 block of Tm before
    // -T2 X is formed; the loops run over whole blocks, the zeros above the
    // diagonal of T1 and T2 masking what a triangular loop would skip.
    {
      // 16 -> 32: block B's rows 16-31 x columns 0-15, one row and two
      // columns per thread; X at Tm[r][32 + 16 B + c]
      const int B = tid >> 7, u = tid & 127, r = u >> 3, c = (u & 7) * 2, o = 32 * B;
      const float* arow = Ap + (o + 16 + r) * kAStride + o;
      float x0 = 0.f, x1 = 0.f;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float2 tv = *reinterpret_cast<const float2*>(Tp + (o + q) * kC + o + c);
        const float av = arow[q];
        x0 = fmaf(av, tv.x, x0);
        x1 = fmaf(av, tv.y, x1);
      }
      *reinterpret_cast<float2*>(Tp + r * kC + 32 + 16 * B + c) = make_float2(x0, x1);
      __syncthreads();
      const float* trow = Tp + (o + 16 + r) * kC + o + 16;
      float y0 = 0.f, y1 = 0.f;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float2 xv = *reinterpret_cast<const float2*>(Tp + q * kC + 32 + 16 * B + c);
        const float tv = trow[q];
        y0 = fmaf(tv, xv.x, y0);
        y1 = fmaf(tv, xv.y, y1);
      }
      *reinterpret_cast<float2*>(Tp + (o + 16 + r) * kC + o + c) = make_float2(-y0, -y1);
      __syncthreads();
    }
    {
      // 32 -> 64: rows 32-63 x columns 0-31, a 2 x 2 tile per thread; X at
      // Tm[r][32 + c]
      const int r0 = (tid >> 4) * 2, c0 = (tid & 15) * 2;
      const float* a0 = Ap + (32 + r0) * kAStride;
      const float* a1 = a0 + kAStride;
      float x00 = 0.f, x01 = 0.f, x10 = 0.f, x11 = 0.f;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const float2 tv = *reinterpret_cast<const float2*>(Tp + q * kC + c0);
        const float av0 = a0[q], av1 = a1[q];
        x00 = fmaf(av0, tv.x, x00);
        x01 = fmaf(av0, tv.y, x01);
        x10 = fmaf(av1, tv.x, x10);
        x11 = fmaf(av1, tv.y, x11);
      }
      *reinterpret_cast<float2*>(Tp + r0 * kC + 32 + c0) = make_float2(x00, x01);
      *reinterpret_cast<float2*>(Tp + (r0 + 1) * kC + 32 + c0) = make_float2(x10, x11);
      __syncthreads();
      const float* t0 = Tp + (32 + r0) * kC + 32;
      const float* t1 = t0 + kC;
      float y00 = 0.f, y01 = 0.f, y10 = 0.f, y11 = 0.f;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const float2 xv = *reinterpret_cast<const float2*>(Tp + q * kC + 32 + c0);
        const float tv0 = t0[q], tv1 = t1[q];
        y00 = fmaf(tv0, xv.x, y00);
        y01 = fmaf(tv0, xv.y, y01);
        y10 = fmaf(tv1, xv.x, y10);
        y11 = fmaf(tv1, xv.y, y11);
      }
      *reinterpret_cast<float2*>(Tp + (32 + r0) * kC + c0) = make_float2(-y00, -y01);
      *reinterpret_cast<float2*>(Tp + (32 + r0 + 1) * kC + c0) = make_float2(-y10, -y11);
      __syncthreads();
    }
    // Tb = Tm diag(beta) as hi + lo bf16, zero above the diagonal; 16
    // consecutive elements of one row per thread
    {
      const int e0 = 16 * tid, tr = e0 >> 6, u0 = e0 & 63;
      float x[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const int s = u0 + m;
        x[m] = s <= tr ? Tp[tr * kC + s] * sbeta[r][s] : 0.f;
      }
      uint4 h0, l0, h1, l1;
      split8(x, h0, l0);
      split8(x + 8, h1, l1);
      uint4* dh = reinterpret_cast<uint4*>(w.tw + slot * (kC * kC) + e0);
      uint4* dl = reinterpret_cast<uint4*>(w.tw + (HvG + slot) * (kC * kC) + e0);
      dh[0] = h0;
      dh[1] = h1;
      dl[0] = l0;
      dl[1] = l1;
    }
    if (tid < kC) {
      const int t = tid;
      const bool live = t < L;
      float* vv = w.vec + slot * (4 * kC);
      vv[t] = live ? sgam[r][t] * sinvk[t] : 0.f;
      vv[kC + t] = live ? expf(sc[r][L - 1] - sc[r][t]) * sinvk[t] : 0.f;
      vv[2 * kC + t] = live ? sgam[r][t] * sinvq[t] : 0.f;
      vv[3 * kC + t] = t == 0 ? sgam[r][L - 1] : 0.f;
    }
    __syncthreads();  // A and Tm are rewritten for the next V head
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, 64);
}

// ----------------------------------------------------------------- carry

// shared memory (byte offsets from a 1024-aligned base)
constexpr uint32_t C_OFF_KQ = 0;         // bf16 [128][128 i] SW128 (TMA): rows 0-63 k, 64-127 q
constexpr uint32_t C_OFF_KT = 32768;     // bf16 [2][128 i][64 t] SW128 (TMA, k transposed by prep)
constexpr uint32_t C_OFF_TB = 65536;     // bf16 [2][128][64 s] SW128 (TMA): rows 0-63 Tb hi, 64-127 lo
constexpr uint32_t C_OFF_P = 98304;      // bf16 [2][64 t][64 s] SW128 (TMA): P
constexpr uint32_t C_OFF_V = 114688;     // bf16 [64 s][128 j] row-major (TMA)
constexpr uint32_t C_OFF_VEC = 131072;   // fp32 [2][4][64] (bulk copy), by chunk parity
constexpr uint32_t C_OFF_Z = 133120;     // bf16 [2][64 t][128 j] row-major: z (TMA), then out
constexpr uint32_t C_SMEM = 165888 + 1024;
// K^T, Tb and P are double-buffered by chunk parity and loaded a chunk ahead,
// together with k and q, on one barrier per parity
constexpr uint32_t kInBytes = 32768 + 16384 + 16384 + 8192;

// TMEM columns. A operands of the MMAs live in TMEM as packed bf16 pairs
// (row j in lane j, K elements 2c, 2c+1 in column c). Each region is
// rewritten only after every reader of its previous contents is known to be
// done (an MMA commit or a wait on the reading threads' barrier).
constexpr uint32_t TM_S = 0;      // fp32 S (128): the state accumulator
constexpr uint32_t TM_X = 128;    // S hi (64) | S lo (64); fp32 [R_hi Tb^T | R_hi Tb_lo^T] after (3)
constexpr uint32_t TM_XLO = 192;
constexpr uint32_t TM_Z = 256;    // R^T hi (32) | lo (32); (dk Dm)^T hi | lo after (4)
constexpr uint32_t TM_ZLO = 288;
constexpr uint32_t TM_Y = 320;    // fp32 [KS | OQ] (128); Dm^T P^T over the KS half
constexpr uint32_t TM_W = 448;    // Dm^T hi (32), A operand of Dm^T P^T
constexpr uint32_t TM_COLS = 512;

constexpr int kIssueWarp = 16;                 // every MMA (a converged warp, one elected lane)
constexpr int kLoadWarp = 17;                  // the carry's TMA loads (lane 0)
constexpr int kOutThreads = 256;               // warps 8-15
constexpr int kChainAll = kChainThreads + 64;  // + the issue and load warps

// Bounded wait that gives up at once when another role has given up.
__device__ __forceinline__ bool chain_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait_bounded(bar, parity, abort_flag);
}

// A carry warp hands one K slice of an A operand it wrote to the issue warp.
__device__ __forceinline__ void slice_done(uint64_t* bar, int lane) {
  tc::tmem_wait_st();
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Per chunk k (the issue warp's order; the carry warps hand over each K slice
// of an operand as soon as it is in TMEM, so the MMAs on slice s run while
// slice s+1 is computed):
//   (1) [KS | OQ] = S_hi [k; q]^T + S_lo k^T, K = i in two slices (bar_sc)
//   (2) R^T = V^T - diag(ak) KS^T -> hi/lo, K = s in two slices (bar_r)
//   (3) [R_hi Tb^T | R_hi Tb_lo^T] (+ R_lo Tb^T onto the first half)
//   (4) Dm^T = sum of the halves; (dk Dm)^T hi/lo and Dm^T hi (bar_d)
//   (5) S += (dk Dm)^T K (hi, lo), on the accumulator pre-scaled by G_{L-1};
//       Dm^T P^T over the KS half, for the output only
//   (6) the new state: hi/lo copies (next chunk's (1)), accumulator rescaled
// The load warp issues a buffer's next load once its last reader is done:
//   K, Q, and Tb, P, K^T of chunk k+1 (into the buffers of chunk k-1), all on
//   bar_in[(k+1) & 1], after (1) completes (its commit covers chunk k-1's
//   (3) and (5));  V after every slice of (2);  vec two chunks ahead after
//   every slice of (4)
// The output group reads OQ after (1) and Dm^T P^T after (5), then releases
// the [KS | OQ] columns (bar_oe) for chunk k+1's (1).
__global__ void __launch_bounds__(kChainAll, 1)
    cp_chain_kernel(const PrefillArgs p, const CpWork w, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_o) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bar_in[2], bar_v, bar_m1, bar_m3, bar_m5;
  __shared__ __align__(8) uint64_t bar_vec[2], bar_of, bar_oe, bar_fin, bar_z[2];
  __shared__ __align__(8) uint64_t bar_sc[2], bar_r[2], bar_d[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float spart[4][kC];
  __shared__ float sinv[kC];
  __shared__ float sgq[2][kC];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, n = blockIdx.y;
  const int kh = k_head_of(p.map, h, p.Hk, p.rep);
  const int64_t kb = w.cs[n], ke = w.cs[n + 1];
  if (ke <= kb) return;  // empty sequence: the state is left as it is
  if (ke > w.G) {
    if (tid == 0) record_device_error(GDN_ERR_INVALID_ARG);
    return;
  }
  const int nch = (int)(ke - kb);
  int64_t seq_s, seq_e;
  seq_range(p, n, seq_s, seq_e);
  const bool fused = p.z != nullptr;
  const size_t HvG = (size_t)w.G * p.Hv;

  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, TM_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_v, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_in[b], 1);
      mbar_init(&bar_vec[b], 1);
      mbar_init(&bar_z[b], 1);
      mbar_init(&bar_sc[b], kCarryThreads / 32);
      mbar_init(&bar_r[b], kCarryThreads / 32);
      mbar_init(&bar_d[b], kCarryThreads / 32);
    }
    mbar_init(&bar_m1, 1);
    mbar_init(&bar_m3, 1);
    mbar_init(&bar_m5, 1);
    mbar_init(&bar_of, 1);
    mbar_init(&bar_oe, kOutThreads);
    mbar_init(&bar_fin, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = s_tmem;
  volatile int* abort_flag = &s_abort;
  auto chunk_c0 = [&](int k) { return seq_s + (int64_t)kC * k; };
  auto slot_of = [&](int k) { return (size_t)(kb + k) * p.Hv + h; };

  // the load warp's loads; the counts let the exit path wait for copies in
  // flight
  uint32_t n_in0 = 0, n_in1 = 0, n_v = 0, n_vec0 = 0, n_vec1 = 0;
  const bool loader = warp == kLoadWarp && lane == 0;

  if (loader) {
    // the MMA operands of chunk k on bar_in[k & 1]: the expected bytes are
    // posted once per phase, the copies may land before or after
    auto arm_in = [&](int k) {
      if (k & 1) ++n_in1; else ++n_in0;
      mbar_arrive_expect_tx(&bar_in[k & 1], kInBytes);
    };
    auto load_kq = [&](int k) {
      uint64_t* bar = &bar_in[k & 1];
      const int y = (int)chunk_c0(k);
      tc::tma_load_2d(sm + C_OFF_KQ, &tm_k, kh * kD, y, bar);
      tc::tma_load_2d(sm + C_OFF_KQ + 16384, &tm_k, kh * kD + 64, y, bar);
      tc::tma_load_2d(sm + C_OFF_KQ + 8192, &tm_q, kh * kD, y, bar);
      tc::tma_load_2d(sm + C_OFF_KQ + 24576, &tm_q, kh * kD + 64, y, bar);
    };
    auto load_tbpk = [&](int k) {
      uint64_t* bar = &bar_in[k & 1];
      const int b = k & 1;
      const size_t slot = slot_of(k);
      tc::tma_load_2d(sm + C_OFF_TB + b * 16384, &tm_w, 0, (int)(slot * kC), bar);
      tc::tma_load_2d(sm + C_OFF_TB + b * 16384 + 8192, &tm_w, 0, (int)((HvG + slot) * kC), bar);
      tc::tma_load_2d(sm + C_OFF_P + b * 8192, &tm_w, 0, (int)((2 * HvG + slot) * kC), bar);
      tc::tma_load_2d(sm + C_OFF_KT + b * 16384, &tm_kt, 0, (int)(((kb + k) * p.Hk + kh) * kD), bar);
    };
    auto load_v = [&](int k) {
      ++n_v;
      mbar_arrive_expect_tx(&bar_v, 16384u);
      tc::tma_load_2d(sm + C_OFF_V, &tm_v, h * kD, (int)chunk_c0(k), &bar_v);
    };
    auto load_vec = [&](int k) {
      uint64_t* bar = &bar_vec[k & 1];
      if (k & 1) ++n_vec1; else ++n_vec0;
      mbar_arrive_expect_tx(bar, 1024u);
      bulk_load(sm + C_OFF_VEC + (k & 1) * 1024, w.vec + slot_of(k) * (4 * kC), 1024u, bar);
    };
    arm_in(0);
    load_kq(0);
    load_tbpk(0);
    load_v(0);
    load_vec(0);
    if (nch > 1) {
      arm_in(1);
      load_tbpk(1);
      load_vec(1);
    }
    for (int k = 0; k < nch; ++k) {
      const uint32_t ph = (uint32_t)(k & 1);
      const bool more = k + 1 < nch;
      if (!chain_wait(&bar_m1, ph, abort_flag)) break;
      if (more) {
        if (k >= 1) {
          arm_in(k + 1);
          load_tbpk(k + 1);  // into chunk k-1's buffers
        }
        load_kq(k + 1);
      }
      if (!chain_wait(&bar_r[1], ph, abort_flag)) break;
      if (more) load_v(k + 1);  // every slice of (2) has read V
      if (!chain_wait(&bar_d[1], ph, abort_flag)) break;
      if (k + 2 < nch) load_vec(k + 2);  // every slice of (4) has read these vectors
    }
  } else if (warp == kIssueWarp) {
    const uint32_t id64 = tc::idesc(tc::kBF16, 128, 64), id128 = tc::idesc(tc::kBF16, 128, 128);
    const uint64_t d_kq = tc::sdesc_sw128(smem_u32(sm + C_OFF_KQ)),
                   d_kt = tc::sdesc_sw128(smem_u32(sm + C_OFF_KT)),
                   d_tb = tc::sdesc_sw128(smem_u32(sm + C_OFF_TB)),
                   d_p = tc::sdesc_sw128(smem_u32(sm + C_OFF_P));
    for (int k = 0; k < nch; ++k) {
      const uint32_t ph = (uint32_t)(k & 1);
      bool ok = chain_wait(&bar_in[k & 1], (uint32_t)((k >> 1) & 1), abort_flag);
      if (ok && k >= 1) ok = chain_wait(&bar_oe, (uint32_t)((k - 1) & 1), abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      // (1) slice s of the state copies covers k-steps 2s, 2s+1, 4+2s, 5+2s
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        ok = __all_sync(0xffffffffu, chain_wait(&bar_sc[s], ph, abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ks = 2 * s + (e & 1) + 4 * (e >> 1);
          tc::mma_f16_ts_elect(tb + TM_Y, tb + TM_X + 8 * ks, tc::sdesc_at(d_kq, 128, ks), id128, ks > 0);
          tc::mma_f16_ts_elect(tb + TM_Y, tb + TM_XLO + 8 * ks, tc::sdesc_at(d_kq, 128, ks), id64, true);
        }
      }
      if (!ok) break;
      tc::mma_commit_elect(&bar_m1);
      // (3) slice s of R covers k-steps s and 2 + s; B = [Tb hi; Tb lo]
      // (N=128) for R hi, Tb hi (N=64) for R lo
      const uint64_t dtb = d_tb + (uint64_t)((k & 1) * 16384 >> 4);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        ok = __all_sync(0xffffffffu, chain_wait(&bar_r[s], ph, abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ks = s + 2 * e;
          tc::mma_f16_ts_elect(tb + TM_X, tb + TM_Z + 8 * ks, tc::sdesc_at(dtb, 128, ks), id128, ks > 0);
          tc::mma_f16_ts_elect(tb + TM_X, tb + TM_ZLO + 8 * ks, tc::sdesc_at(dtb, 64, ks), id64, true);
        }
      }
      if (!ok) break;
      tc::mma_commit_elect(&bar_m3);
      // (5) slice s of Dm covers k-steps s and 2 + s
      const uint64_t dkt = d_kt + (uint64_t)((k & 1) * 16384 >> 4);
      const uint64_t dp = d_p + (uint64_t)((k & 1) * 8192 >> 4);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        ok = __all_sync(0xffffffffu, chain_wait(&bar_d[s], ph, abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int ks = s + 2 * e;
          tc::mma_f16_ts_elect(tb + TM_S, tb + TM_Z + 8 * ks, tc::sdesc_at(dkt, 128, ks), id128, true);
          tc::mma_f16_ts_elect(tb + TM_S, tb + TM_ZLO + 8 * ks, tc::sdesc_at(dkt, 128, ks), id128, true);
        }
        if (s == 0) {
          tc::mma_f16_ts_elect(tb + TM_Y, tb + TM_W, tc::sdesc_at(dp, 64, 0), id64, false);
          tc::mma_f16_ts_elect(tb + TM_Y, tb + TM_W + 16, tc::sdesc_at(dp, 64, 2), id64, true);
        }
      }
      if (!ok) break;
      tc::mma_commit_elect(&bar_m5);
      tc::mma_f16_ts_elect(tb + TM_Y, tb + TM_W + 8, tc::sdesc_at(dp, 64, 1), id64, true);
      tc::mma_f16_ts_elect(tb + TM_Y, tb + TM_W + 24, tc::sdesc_at(dp, 64, 3), id64, true);
      tc::mma_commit_elect(&bar_of);  // OQ and Dm^T P^T of this chunk
    }
  } else if (tid < kCarryThreads) {
    // ============================ carry group: thread (j, ch) owns value row j
    // (TMEM lane j) and half ch of the columns of each per-row phase
    const int j = tid & 127, ch = tid >> 7;
    const uint32_t tl = tb + ((uint32_t)(32 * (warp & 3)) << 16);
    float* gS = p.state + (((size_t)n * p.Hv + h) * kD + j) * kD + 64 * ch;

    // 64 fp32 state values (this thread's half row) -> hi/lo A operands in
    // TMEM, one 32-wide K slice at a time, then the accumulator rescaled by gl
    auto store_state = [&](float (&v)[kC], float gl) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const float a0 = v[32 * s + 16 * q + 2 * m], a1 = v[32 * s + 16 * q + 2 * m + 1];
            const __nv_bfloat162 hv = __floats2bfloat162_rn(a0, a1);
            hw[m] = *reinterpret_cast<const uint32_t*>(&hv);
            lw[m] = pack_bf16(a0 - __low2float(hv), a1 - __high2float(hv));
          }
          tc::tmem_st8u(tl + TM_X + 32 * ch + 16 * s + 8 * q, hw);
          tc::tmem_st8u(tl + TM_XLO + 32 * ch + 16 * s + 8 * q, lw);
        }
        slice_done(&bar_sc[s], lane);
      }
#pragma unroll
      for (int e = 0; e < kC; ++e) v[e] *= gl;
#pragma unroll
      for (int m = 0; m < 4; ++m)
        tc::tmem_st16(tl + TM_S + 64 * ch + 16 * m, *reinterpret_cast<const float(*)[16]>(v + 16 * m));
    };

    bool to = !chain_wait(&bar_vec[0], 0, abort_flag);
    to = __any_sync(0xffffffffu, to);
    if (!to) {
      float v[kC];
      const float4* src = reinterpret_cast<const float4*>(gS);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float4 f = src[m];
        v[4 * m] = f.x;
        v[4 * m + 1] = f.y;
        v[4 * m + 2] = f.z;
        v[4 * m + 3] = f.w;
      }
      store_state(v, reinterpret_cast<const float*>(sm + C_OFF_VEC)[3 * kC]);
    }

    for (int k = 0; k < nch && !to; ++k) {
      const uint32_t ph = (uint32_t)(k & 1);
      const int64_t c0 = chunk_c0(k);
      const int L = (int)((seq_e - c0) < kC ? (seq_e - c0) : kC);
      const float* vec = reinterpret_cast<const float*>(sm + C_OFF_VEC + (k & 1) * 1024);
      const bool more = k + 1 < nch;

      // (2) R^T = V^T - diag(ak) KS^T (columns s >= L zero); this thread's
      // 32 columns s = 32 ch .., two slices of 16
      // (V and the vectors landed long before (1) completes: checked first)
      to = !chain_wait(&bar_v, ph, abort_flag) ||
           !chain_wait(&bar_vec[k & 1], (uint32_t)((k >> 1) & 1), abort_flag) ||
           !chain_wait(&bar_m1, ph, abort_flag);
      if (__any_sync(0xffffffffu, to)) break;
      tc::fence_after_sync();
      {
        const __nv_bfloat16* vt = reinterpret_cast<const __nv_bfloat16*>(sm + C_OFF_V) + j;
        float ks[32];
#pragma unroll
        for (int m = 0; m < 2; ++m)
          tc::tmem_ld16(tl + TM_Y + 32 * ch + 16 * m, *reinterpret_cast<float(*)[16]>(ks + 16 * m));
        tc::tmem_wait_ld();
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 a4 = reinterpret_cast<const float4*>(vec)[8 * ch + 4 * s + e4];
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            float r[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int e = 16 * s + 4 * e4 + u, t = 32 * ch + e;
              const float x = __bfloat162float(vt[t * kD]) - av[u] * ks[e];
              r[u] = t < L ? x : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const __nv_bfloat162 hv = __floats2bfloat162_rn(r[2 * u], r[2 * u + 1]);
              hw[2 * e4 + u] = *reinterpret_cast<const uint32_t*>(&hv);
              lw[2 * e4 + u] = pack_bf16(r[2 * u] - __low2float(hv), r[2 * u + 1] - __high2float(hv));
            }
          }
          tc::tmem_st8u(tl + TM_Z + 16 * ch + 8 * s, hw);
          tc::tmem_st8u(tl + TM_ZLO + 16 * ch + 8 * s, lw);
          slice_done(&bar_r[s], lane);
        }
      }

      // (4) Dm^T = [R Tb^T halves summed]; (dk Dm)^T hi/lo into R's columns
      // and Dm^T hi for the output; this thread's 32 columns t, two slices
      to = !chain_wait(&bar_m3, ph, abort_flag);
      if (__any_sync(0xffffffffu, to)) break;
      tc::fence_after_sync();
      {
        float dm[32];
        {
          float db[32];
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            tc::tmem_ld16(tl + TM_X + 32 * ch + 16 * m, *reinterpret_cast<float(*)[16]>(dm + 16 * m));
            tc::tmem_ld16(tl + TM_XLO + 32 * ch + 16 * m, *reinterpret_cast<float(*)[16]>(db + 16 * m));
          }
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) dm[e] += db[e];
        }
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          uint32_t hw[8], lw[8], dw[8];
#pragma unroll
          for (int m = 0; m < 8; ++m) dw[m] = pack_bf16(dm[16 * s + 2 * m], dm[16 * s + 2 * m + 1]);
          tc::tmem_st8u(tl + TM_W + 16 * ch + 8 * s, dw);
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 d4 = reinterpret_cast<const float4*>(vec + kC)[8 * ch + 4 * s + e4];
            const int e = 16 * s + 4 * e4;
            const float x0 = d4.x * dm[e], x1 = d4.y * dm[e + 1];
            const float x2 = d4.z * dm[e + 2], x3 = d4.w * dm[e + 3];
            const __nv_bfloat162 h01 = __floats2bfloat162_rn(x0, x1), h23 = __floats2bfloat162_rn(x2, x3);
            hw[2 * e4] = *reinterpret_cast<const uint32_t*>(&h01);
            hw[2 * e4 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
            lw[2 * e4] = pack_bf16(x0 - __low2float(h01), x1 - __high2float(h01));
            lw[2 * e4 + 1] = pack_bf16(x2 - __low2float(h23), x3 - __high2float(h23));
          }
          tc::tmem_st8u(tl + TM_Z + 16 * ch + 8 * s, hw);
          tc::tmem_st8u(tl + TM_ZLO + 16 * ch + 8 * s, lw);
          slice_done(&bar_d[s], lane);
        }
      }

      // (6) the new state: operand copies and the next chunk's decay in TMEM;
      // after the last chunk, back to global memory
      to = more && !chain_wait(&bar_vec[(k + 1) & 1], (uint32_t)(((k + 1) >> 1) & 1), abort_flag);
      to = to || !chain_wait(&bar_m5, ph, abort_flag);
      if (__any_sync(0xffffffffu, to)) break;
      tc::fence_after_sync();
      {
        float v[kC];
#pragma unroll
        for (int m = 0; m < 4; ++m)
          tc::tmem_ld16(tl + TM_S + 64 * ch + 16 * m, *reinterpret_cast<float(*)[16]>(v + 16 * m));
        tc::tmem_wait_ld();
        if (!more) {
          float4* dst = reinterpret_cast<float4*>(gS);
#pragma unroll
          for (int m = 0; m < 16; ++m)
            dst[m] = make_float4(v[4 * m], v[4 * m + 1], v[4 * m + 2], v[4 * m + 3]);
        } else {
          store_state(v, reinterpret_cast<const float*>(sm + C_OFF_VEC + ((k + 1) & 1) * 1024)[3 * kC]);
        }
      }
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
  } else if (tid < kChainThreads) {
    // ============================ output group: 8 warps; thread (j, half)
    // owns output column j = 32 (warp % 4) + lane for the 32 rows of its half.
    // OQ is read once (1) completes and Dm^T P^T once (5) completes; then
    // TMEM is released to the next chunk. With the fused norm, the per-row
    // sums of squares are reduce-scattered across lanes, z arrives by TMA into
    // a row-major tile (two, by chunk parity) that the gated result overwrites
    // in place, and each live row leaves as one 256-byte bulk store.
    const int u = tid - kCarryThreads, q4 = warp & 3, half = (warp - 8) >> 2;
    const int j = 32 * q4 + lane, t0 = 32 * half;
    const uint32_t tl = tb + ((uint32_t)(32 * q4) << 16);
    const float nwj = fused ? p.norm_w[j] : 0.f;
    uint32_t n_z0 = 0, n_z1 = 0;
    bool stored = false;
    auto load_z = [&](int k) {
      if (k & 1) ++n_z1; else ++n_z0;
      mbar_arrive_expect_tx(&bar_z[k & 1], 16384u);
      tc::tma_load_2d(sm + C_OFF_Z + (k & 1) * 16384, &tm_z, h * kD, (int)chunk_c0(k), &bar_z[k & 1]);
    };
    if (fused && u == 0) {
      load_z(0);
      if (nch > 1) load_z(1);
    }
    bool to = false;  // a bounded wait gave up (agreed on at the next barrier)
    for (int k = 0; k < nch; ++k) {
      const int64_t c0 = chunk_c0(k);
      const int L = (int)((seq_e - c0) < kC ? (seq_e - c0) : kC);
      const float* gq = sgq[k & 1] + t0;
      __nv_bfloat16* zb = reinterpret_cast<__nv_bfloat16*>(sm + C_OFF_Z + (k & 1) * 16384);
      if (u < kC) sgq[k & 1][u] = __ldg(w.vec + slot_of(k) * (4 * kC) + 2 * kC + u);
      float a[2][16], b[2][16];
      to |= !chain_wait(&bar_m1, (uint32_t)(k & 1), abort_flag);
      if (!__any_sync(0xffffffffu, to)) {
        tc::fence_after_sync();
#pragma unroll
        for (int m = 0; m < 2; ++m) tc::tmem_ld16(tl + TM_Y + 64 + t0 + 16 * m, a[m]);
        tc::tmem_wait_ld();
      }
      to |= !chain_wait(&bar_of, (uint32_t)(k & 1), abort_flag);
      if (bar_or(2, kOutThreads, to)) break;
      tc::fence_after_sync();
#pragma unroll
      for (int m = 0; m < 2; ++m) tc::tmem_ld16(tl + TM_Y + t0 + 16 * m, b[m]);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      mbar_arrive(&bar_oe);  // this chunk's output accumulators are free
      float o[32];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int e = 0; e < 16; ++e) o[16 * m + e] = fmaf(gq[16 * m + e], a[m][e], b[m][e]);
      if (p.core_out != nullptr) {
        float* cg = p.core_out + ((c0 + t0) * p.Hv + h) * kD + j;
        const int64_t cstr = (int64_t)p.Hv * kD;
        if (L == kC) {
#pragma unroll
          for (int e = 0; e < 32; ++e) cg[e * cstr] = o[e];
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (t0 + e < L) cg[e * cstr] = o[e];
        }
      }
      if (!fused) continue;
      // five halving exchanges: lane l ends with the sum of row t0 + l (the
      // first one squares on the fly)
      float sq[16];
      {
        const bool up = (lane & 16) != 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float send = up ? o[i] * o[i] : o[i + 16] * o[i + 16];
          const float keep = up ? o[i + 16] * o[i + 16] : o[i] * o[i];
          sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
      }
#pragma unroll
      for (int st = 1; st < 5; ++st) {
        const int m = 16 >> st, hv = 16 >> st;
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < hv; ++i) {
          const float send = up ? sq[i] : sq[i + hv];
          const float keep = up ? sq[i + hv] : sq[i];
          sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      spart[q4][t0 + lane] = sq[0];
      bar_named(2, kOutThreads);
      if (u < kC)
        sinv[u] = 1.f / sqrtf((spart[0][u] + spart[1][u] + spart[2][u] + spart[3][u]) / (float)kD +
                              p.rms_eps);
      // z of chunk k+1 into the tile chunk k-1 was stored from. Only a
      // sequence's last chunk can be partial, so chunk k-1 was full and left
      // as thread 0's one tile store: its own wait covers the reload.
      if (u == 0 && k >= 1 && k + 1 < nch) {
        bulk_wait_read_all();
        load_z(k + 1);
      }
      to |= !chain_wait(&bar_z[k & 1], (uint32_t)((k >> 1) & 1), abort_flag);
      bar_named(2, kOutThreads);
      // the gated result over z, in place (rows >= L hold finite values that
      // are never stored), 16 rows at a time: all loads, then the math, then
      // all stores
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float zf[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) zf[e] = __bfloat162float(zb[(t0 + 16 * hf + e) * kD + j]);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int t = t0 + 16 * hf + e;
          const float gate = __fdividef(zf[e], 1.f + __expf(-zf[e]));
          zf[e] = o[16 * hf + e] * sinv[t] * nwj * gate;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) zb[(t0 + 16 * hf + e) * kD + j] = __float2bfloat16_rn(zf[e]);
      }
      fence_proxy_async_smem();
      bar_named(2, kOutThreads);
      if (L == kC) {
        // a full chunk leaves as one tile
        if (u == 0) {
          tc::tma_store_2d(&tm_o, h * kD, (int)c0, zb);
          bulk_commit();
          stored = true;
        }
      } else if (u < L) {
        // the sequence's last chunk: row by row, so no row of the next
        // sequence is written
        bulk_store(static_cast<__nv_bfloat16*>(p.out) + ((c0 + u) * p.Hv + h) * kD, zb + u * kD,
                   (uint32_t)(kD * 2));
        bulk_commit();
        stored = true;
      }
    }
    if (stored) bulk_wait_all();
    if (u == 0) {
      if (n_z0) mbar_wait(&bar_z[0], (n_z0 - 1) & 1);
      if (n_z1) mbar_wait(&bar_z[1], (n_z1 - 1) & 1);
    }
  }

  // drain: every copy and MMA this CTA issued has completed before it exits
  // and TMEM is released (all of these have completed already unless a
  // bounded wait gave up)
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kIssueWarp) {
    tc::fence_after_sync();
    tc::mma_commit_elect(&bar_fin);
    mbar_wait(&bar_fin, 0);
    tc::fence_before_sync();
  }
  if (loader) {
    if (n_in0) mbar_wait(&bar_in[0], (n_in0 - 1) & 1);
    if (n_in1) mbar_wait(&bar_in[1], (n_in1 - 1) & 1);
    if (n_v) mbar_wait(&bar_v, (n_v - 1) & 1);
    if (n_vec0) mbar_wait(&bar_vec[0], (n_vec0 - 1) & 1);
    if (n_vec1) mbar_wait(&bar_vec[1], (n_vec1 - 1) & 1);
  }
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tb, TM_COLS);
  }
}

}  // namespace

int64_t prefill_cp_workspace_bytes(int32_t N, int64_t T, int32_t Hk, int32_t Hv) {
  return (int64_t)cp_layout(N, T, Hk, Hv).total;
}

bool prefill_cp_supported(const PrefillArgs& p, int32_t dtype, int32_t D) {
  if (D != kD || dtype != GDN_BF16 || p.rep > kMaxRep) return false;
  if (p.T >= ((int64_t)1 << 31)) return false;  // TMA row coordinates are int32
  const CpLayout l = cp_layout(p.N, p.T, p.Hk, p.Hv);
  if ((double)l.G * p.Hv * kC * 3 >= 2147483647.0) return false;
  if ((double)l.G * p.Hk * kD >= 2147483647.0) return false;
  return tc::encode_fn() != nullptr;
}

cudaError_t launch_prefill_cp(const PrefillArgs& p, void* workspace, cudaStream_t stream) {
  if (p.N == 0 || p.T == 0) return cudaSuccess;
  const CpLayout l = cp_layout(p.N, p.T, p.Hk, p.Hv);
  CpWork w{};
  w.cs = static_cast<int32_t*>(workspace);
  w.tw = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) + l.off_tm);
  w.kt = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) + l.off_kt);
  w.vec = reinterpret_cast<float*>(static_cast<char*>(workspace) + l.off_vec);
  w.G = l.G;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap mq, mk, mv, mw, mz, mkt, mo;
  memset(&mz, 0, sizeof(mz));
  memset(&mo, 0, sizeof(mo));
  const int64_t qkc = (int64_t)p.Hk * kD, vc = (int64_t)p.Hv * kD;
  if (!tc::make_map_2d(&mq, p.q, p.T, qkc, p.q_stride, 2, bf, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_map_2d(&mk, p.k, p.T, qkc, p.k_stride, 2, bf, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_map_2d(&mv, p.v, p.T, vc, p.v_stride, 2, bf, kD, 64, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !tc::make_map_2d(&mw, w.tw, 3 * l.G * p.Hv * kC, kC, kC, 2, bf, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!tc::make_map_2d(&mkt, w.kt, l.G * p.Hk * kD, kC, kC, 2, bf, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (p.z != nullptr &&
      (!tc::make_map_2d(&mz, p.z, p.T, vc, vc, 2, bf, kD, 64, CU_TENSOR_MAP_SWIZZLE_NONE) ||
       !tc::make_map_2d(&mo, p.out, p.T, vc, vc, 2, bf, kD, 64, CU_TENSOR_MAP_SWIZZLE_NONE)))
    return cudaErrorInvalidValue;
  cp_index_kernel<<<1, 1024, 0, stream>>>(p, w);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(cp_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_SMEM);
  if (e != cudaSuccess) return e;
  cp_prep_kernel<<<dim3((unsigned)l.G, (unsigned)p.Hk), kPrepThreads, P_SMEM, stream>>>(p, w, mq, mk);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(cp_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM);
  if (e != cudaSuccess) return e;
  cp_chain_kernel<<<dim3((unsigned)p.Hv, (unsigned)p.N), kChainAll, C_SMEM, stream>>>(p, w, mq, mk,
                                                                                         mv, mw, mz, mkt, mo);
  return cudaGetLastError();
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(prefill_cp)
