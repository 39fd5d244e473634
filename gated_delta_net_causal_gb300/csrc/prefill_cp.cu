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
constexpr int kAStride = kC + 4;    // padded row pitch of the fp32 A matrix (16-byte rows)
constexpr int kMaxRep = 16;         // V heads per K head on this path
// (V head, sequence) pairs up to which the sliced carry (four CTAs each) is
// chosen, and the workspace holds an fp32 core output for its separate norm
constexpr int64_t kSlMaxChains = 64;

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
  size_t off_tm, off_kt, off_vec, off_o, total;  // off_o 0: no core-output region
};

CpLayout cp_layout(int32_t N, int64_t T, int32_t Hk, int32_t Hv) {
  CpLayout l{};
  // sum over sequences of ceil(len/64) <= (T + 63 N) / 64
  l.G = T > 0 ? (T + 63 * (int64_t)N) / kC : 0;
  l.off_tm = ((size_t)4 * ((size_t)N + 1) + 1023) / 1024 * 1024;
  l.off_kt = l.off_tm + (size_t)3 * l.G * Hv * kC * kC * 2;
  l.off_vec = l.off_kt + (size_t)l.G * Hk * kD * kC * 2;
  l.total = l.off_vec + (size_t)l.G * Hv * 4 * kC * 4;
  // few (V head, sequence) pairs: [T][Hv][128] fp32 for the sliced carry's
  // core output, normalised by a separate pass when no core_out is given
  if (l.G > 0 && (int64_t)Hv * N <= kSlMaxChains) {
    l.off_o = (l.total + 255) / 256 * 256;
    l.total = l.off_o + (size_t)T * Hv * kD * 4;
  }
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
constexpr uint32_t P_OFF_T = kC * kAStride * 4;  // fp32 [64][64] Tm (products in its upper triangle)
constexpr uint32_t P_SMEM = P_OFF_T + kC * kC * 4 + 1024;

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
  // (each thread finishes its own elements; sc[r][31] is not rewritten)
  for (int e = tid; e < p.rep * kC; e += kPrepThreads) {
    const int r = e >> 6, t = e & 63;
    float c = sc[r][t];
    if (t >= 32) {
      c += sc[r][31];
      sc[r][t] = c;
    }
    sgam[r][t] = expf(c);
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
        for (int m = 0; m < 8; ++m) {
          const int s = 32 * hc + 4 * m;
          *reinterpret_cast<float4*>(Ap + t * kAStride + s) =
              make_float4(s < t ? bk * pr[4 * m] : 0.f, s + 1 < t ? bk * pr[4 * m + 1] : 0.f,
                          s + 2 < t ? bk * pr[4 * m + 2] : 0.f, s + 3 < t ? bk * pr[4 * m + 3] : 0.f);
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
        float av[16];
#pragma unroll
        for (int q4 = 0; q4 < 16; q4 += 4) {
          if (q4 < m) {
            const float4 v = *reinterpret_cast<const float4*>(arow + q4);
            av[q4] = v.x, av[q4 + 1] = v.y, av[q4 + 2] = v.z, av[q4 + 3] = v.w;
          }
        }
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < m; ++q) acc = fmaf(av[q], x[q], acc);
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
      float2 x = make_float2(0.f, 0.f);
#pragma unroll
      for (int q4 = 0; q4 < 16; q4 += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(arow + q4);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          x = fma2(make_float2(av[u], av[u]), *reinterpret_cast<const float2*>(Tp + (o + q4 + u) * kC + o + c), x);
      }
      *reinterpret_cast<float2*>(Tp + r * kC + 32 + 16 * B + c) = x;
      __syncthreads();
      const float* trow = Tp + (o + 16 + r) * kC + o + 16;
      float2 y = make_float2(0.f, 0.f);
#pragma unroll
      for (int q4 = 0; q4 < 16; q4 += 4) {
        const float4 t4 = *reinterpret_cast<const float4*>(trow + q4);
        const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          y = fma2(make_float2(tv[u], tv[u]), *reinterpret_cast<const float2*>(Tp + (q4 + u) * kC + 32 + 16 * B + c), y);
      }
      *reinterpret_cast<float2*>(Tp + (o + 16 + r) * kC + o + c) = make_float2(-y.x, -y.y);
      __syncthreads();
    }
    {
      // 32 -> 64: rows 32-63 x columns 0-31, a 2 x 2 tile per thread; X at
      // Tm[r][32 + c]
      const int r0 = (tid >> 4) * 2, c0 = (tid & 15) * 2;
      const float* a0 = Ap + (32 + r0) * kAStride;
      const float* a1 = a0 + kAStride;
      float2 x0 = make_float2(0.f, 0.f), x1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int q4 = 0; q4 < 32; q4 += 4) {
        const float4 p0 = *reinterpret_cast<const float4*>(a0 + q4);
        const float4 p1 = *reinterpret_cast<const float4*>(a1 + q4);
        const float av0[4] = {p0.x, p0.y, p0.z, p0.w}, av1[4] = {p1.x, p1.y, p1.z, p1.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 tv = *reinterpret_cast<const float2*>(Tp + (q4 + u) * kC + c0);
          x0 = fma2(make_float2(av0[u], av0[u]), tv, x0);
          x1 = fma2(make_float2(av1[u], av1[u]), tv, x1);
        }
      }
      *reinterpret_cast<float2*>(Tp + r0 * kC + 32 + c0) = x0;
      *reinterpret_cast<float2*>(Tp + (r0 + 1) * kC + 32 + c0) = x1;
      __syncthreads();
      const float* t0 = Tp + (32 + r0) * kC + 32;
      const float* t1 = t0 + kC;
      float2 y0 = make_float2(0.f, 0.f), y1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int q4 = 0; q4 < 32; q4 += 4) {
        const float4 p0 = *reinterpret_cast<const float4*>(t0 + q4);
        const float4 p1 = *reinterpret_cast<const float4*>(t1 + q4);
        const float tv0[4] = {p0.x, p0.y, p0.z, p0.w}, tv1[4] = {p1.x, p1.y, p1.z, p1.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 xv = *reinterpret_cast<const float2*>(Tp + (q4 + u) * kC + 32 + c0);
          y0 = fma2(make_float2(tv0[u], tv0[u]), xv, y0);
          y1 = fma2(make_float2(tv1[u], tv1[u]), xv, y1);
        }
      }
      *reinterpret_cast<float2*>(Tp + (32 + r0) * kC + c0) = make_float2(-y0.x, -y0.y);
      *reinterpret_cast<float2*>(Tp + (32 + r0 + 1) * kC + c0) = make_float2(-y1.x, -y1.y);
      __syncthreads();
    }
    // Tb = Tm diag(beta) as hi + lo bf16, zero above the diagonal; 16
    // consecutive elements of one row per thread
    {
      const int e0 = 16 * tid, tr = e0 >> 6, u0 = e0 & 63;
      float x[16];
#pragma unroll
      for (int m4 = 0; m4 < 16; m4 += 4) {
        const float4 tv = *reinterpret_cast<const float4*>(Tp + tr * kC + u0 + m4);
        const float4 bv = *reinterpret_cast<const float4*>(&sbeta[r][u0 + m4]);
        const float t4[4] = {tv.x, tv.y, tv.z, tv.w}, b4[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) x[m4 + u] = u0 + m4 + u <= tr ? t4[u] * b4[u] : 0.f;
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
    // no barrier here: the next V head's A/P build writes only A (every
    // read of it ended before the doubling's last barrier) and global P;
    // Tm, which this head's Tb rows still read, is rewritten only past the
    // barrier that ends that build
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


// ---------------------------------------------------------- sliced carry
//
// The carry with the 128 value rows of each (V head, sequence) split over a
// cluster of four CTAs, 32 rows j each. Given a chunk's state-free factors,
// row j of the state evolves on its own, so the CTAs share nothing but the
// gated RMSNorm's per-token sums of squares. Against cp_chain_kernel the
// orientation is turned around: the MMA M dimension runs over tokens (or key
// columns i) and this CTA's 32 value rows are N, so the state slice S_J is a
// B operand in shared memory (bf16 hi and lo, [32 j][128 i]) and its fp32
// copy lives transposed in TMEM (lane i, column j). Per chunk:
//   (1) [KS | QS] (lane t, column j) = [k; q] (S_hi + S_lo)_J^T
//   (2) R = V_J - diag(ak) KS -> hi/lo B tiles [64 s][32 j] (rows t >= L zero)
//   (3) [X | Y] = [Tb hi; Tb lo] (R_hi + R_lo): Dm = X + Y, X in lanes 0-63,
//       Y in lanes 64-127 (no exchange between lane quadrants)
//   (4) (dk X) hi/lo, (dk Y) hi, X hi, Y hi -> B tiles
//   (5) S_J^T += K^T (dk Dm) on the accumulator pre-scaled by G_{L-1} (three
//       partial accumulators, one per B tile, summed by (6));
//       P (X_hi + Y_hi) into lanes 64-127 of its own columns (A is a
//       128-row window whose rows 64-127 are P; the first half is unused)
//   (6) the new S_J hi/lo tiles and the accumulator rescaled
// and O = gq QS + P Dm, then the gated RMSNorm with the sums of squares of
// each token's row exchanged over the cluster. Each phase is a quarter of
// the per-thread work of the unsliced carry, which is latency-bound at the
// sizes where there are few (V head, sequence) pairs to spread over the SMs.

constexpr int kSl = 32;             // value rows per CTA
constexpr int kSlCta = kD / kSl;    // CTAs per cluster
constexpr int kSlThreads = 384;     // warps 0-7 carry, 8 MMA, 9 loads, 10-11 output
constexpr int kSlIssueWarp = 8;
constexpr int kSlLoadWarp = 9;
constexpr int kSlOutThreads = 64;   // warps 10-11: one token row t each

// shared memory (byte offsets from a 1024-aligned base); the per-chunk
// inputs are double-buffered by chunk parity b
constexpr uint32_t L_KQ = 0;             // bf16 [2][128 rows: k t | q t][128 i] SW128 (TMA)
constexpr uint32_t L_TB = 65536;         // bf16 [2][128 rows: Tb hi | Tb lo][64 s] SW128 (TMA)
constexpr uint32_t L_KT = 98304;         // bf16 [2][128 i][64 t] SW128 (TMA)
constexpr uint32_t L_P = 131072;         // bf16 [2][64 t][64 s] SW128 (TMA)
constexpr uint32_t L_V = 147456;         // bf16 [2][64 t][32 j] row-major (TMA)
constexpr uint32_t L_Z = 155648;         // bf16 [2][64 t][32 j] row-major: z (TMA)
constexpr uint32_t L_VEC = 163840;       // fp32 [2][4][64]: ak, dk, gq, {G_{L-1}}
constexpr uint32_t L_SH = 165888;        // bf16 [128 i][32 j] MN-major SW64: S hi
constexpr uint32_t L_SL = L_SH + 8192;   // S lo
constexpr uint32_t L_RH = L_SL + 8192;   // bf16 [64 s][32 j] MN-major SW64: R hi
constexpr uint32_t L_RL = L_RH + 4096;   // R lo
constexpr uint32_t L_DXH = L_RL + 4096;  // (dk X) hi
constexpr uint32_t L_DXL = L_DXH + 4096; // (dk X) lo
constexpr uint32_t L_DYH = L_DXL + 4096; // (dk Y) hi
constexpr uint32_t L_XH = L_DYH + 4096;  // X hi
constexpr uint32_t L_YH = L_XH + 4096;   // Y hi
constexpr uint32_t L_O = L_YH + 4096;    // bf16 [2][64 t][32 j] row-major: the gated output (TMA store)
constexpr uint32_t L_SMEM = L_O + 8192 + 1024;
static_assert(L_SH % 1024 == 0 && L_RH % 1024 == 0 && L_YH % 1024 == 0 && L_VEC + 2048 <= L_SH,
              "tile alignment");
static_assert(L_P >= 8192 && L_SMEM <= 232448, "P window and shared memory budget");
constexpr uint32_t kSlInBytes = 32768 + 16384 + 16384 + 8192;  // KQ, Tb, K^T, P
constexpr uint32_t kSlVBytes = 4096 + 1024;                    // V_J, vectors
constexpr uint32_t kNormBytes = (kSlCta - 1) * kC * 4;          // the peers' sums of squares

// TMEM columns (lane = MMA row). Each product of a hi/lo pair of B tiles is
// one MMA over both (N = 64 or 96, the tiles adjacent in shared memory), its
// parts in adjacent 32-column groups that the reader adds.
// The two that the output warps read are double-buffered by chunk parity b,
// so that the output of chunk k may finish while chunk k + 1 runs.
constexpr uint32_t T_KQS = 0;    // fp32 [2][KS (lanes 0-63) | QS (64-127)] x {S hi, S lo} (2 x 64)
constexpr uint32_t T_XY = 128;   // fp32 [X | Y] x {R hi, R lo} (64)
constexpr uint32_t T_S = 192;    // fp32 S_J^T (lane i) as three partial accumulators (96)
constexpr uint32_t T_PD = 288;   // fp32 [2] P Dm in lanes 64-127, x {X hi, Y hi} (2 x 64)
constexpr uint32_t T_SL_COLS = 512;

// The B operands of the sliced carry are MN-major with 64-byte swizzling:
// value row j (N, 32 of them) is contiguous, K index k picks a 64-byte row,
// eight K rows form a 512-byte atom, and the 16-byte group c of value rows
// 8c..8c+7 sits at group c ^ ((k % 8) / 2) of its row. A thread that holds
// 16 value rows at one K index stores them as two 16-byte words per tile.
__device__ __forceinline__ uint32_t mn64_group(int k, int c) {
  return (uint32_t)((k >> 3) * 512 + (k & 7) * 64 + ((c ^ ((k & 7) >> 1)) << 4));
}
// Descriptor of such tiles side by side along N, `lbo` bytes apart.
__device__ __forceinline__ uint64_t sdesc_mn64(uint32_t smem_addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFF) >> 4);
  d |= (uint64_t)(lbo >> 4) << 16;   // leading byte offset: between 32-row MN atoms
  d |= (uint64_t)(512 >> 4) << 32;   // stride byte offset: between 8-row K groups
  d |= (uint64_t)1 << 46;            // descriptor version
  d |= (uint64_t)4 << 61;            // SWIZZLE_64B
  return d;
}
// k-step s (16 K rows) of such a tile
__device__ __forceinline__ uint64_t sdesc_mn64_at(uint64_t base, int s) {
  return base + (uint64_t)((s * 1024) >> 4);
}
// x (value rows jl..jl+15 at K index k) rounded to bf16 into one tile
__device__ __forceinline__ void put16(unsigned char* sm, uint32_t tile, int k, int jl, const float* x) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const float* y = x + 8 * c;
    *reinterpret_cast<uint4*>(sm + tile + mn64_group(k, (jl >> 3) + c)) =
        make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
  }
}
// x split into bf16 hi parts (tile th) and the rounded remainders (tile tl)
__device__ __forceinline__ void put16_hilo(unsigned char* sm, uint32_t th, uint32_t tl, int k, int jl,
                                           const float* x) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint4 hi, lo;
    split8(x + 8 * c, hi, lo);
    const uint32_t o = mn64_group(k, (jl >> 3) + c);
    *reinterpret_cast<uint4*>(sm + th + o) = hi;
    *reinterpret_cast<uint4*>(sm + tl + o) = lo;
  }
}
// Bounded wait for the roles off the critical path (output, loads): between
// polls the thread sleeps, so that it takes no issue slots from the carry
// warps that share its SM sub-partition. `abort_flag` may be null (the wait
// then ends only on completion or the time limit).
__device__ __noinline__ bool wait_sleepy_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  const uint64_t t0 = global_ns();
  for (;;) {
    __nanosleep(100);
    if (abort_flag != nullptr && *abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      record_device_error(GDN_ERR_TIMEOUT);
      if (abort_flag != nullptr) *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_sleepy(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_try_wait(bar, parity) || wait_sleepy_slow(bar, parity, abort_flag);
}

// A warp hands shared-memory (and TMEM) operands it wrote to the MMA warp.
__device__ __forceinline__ void operands_done(uint64_t* bar, int lane) {
  fence_proxy_async_smem();
  tc::tmem_wait_st();
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

__global__ void __cluster_dims__(kSlCta, 1, 1) __launch_bounds__(kSlThreads, 1)
    cp_slice_kernel(const PrefillArgs p, const CpWork w, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_o) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bar_in[2], bar_v[2], bar_z[2], bar_nm[2], bar_free[2], bar_q[2];
  __shared__ __align__(8) uint64_t bar_m1, bar_m3, bar_m5, bar_oe[2], bar_fin;
  __shared__ __align__(8) uint64_t bar_s[4], bar_r[2], bar_d[4];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float snorm[2][kSlCta][kC];  // per token: the four slices' sums of squares
  __shared__ float snw[kSl];              // this slice's gated-norm weights

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x / kSlCta, n = blockIdx.y;
  const uint32_t rank = cluster_ctarank();
  const int j0 = kSl * (int)rank;
  const int kh = k_head_of(p.map, h, p.Hk, p.rep);
  const int64_t kb = w.cs[n], ke = w.cs[n + 1];
  // (both exits are taken by every CTA of the cluster, before any access to
  // another CTA's shared memory)
  if (ke <= kb) return;  // empty sequence: the state is left as it is
  if (ke > w.G) {
    if (tid == 0 && rank == 0) record_device_error(GDN_ERR_INVALID_ARG);
    return;
  }
  const int nch = (int)(ke - kb);
  int64_t seq_s, seq_e;
  seq_range(p, n, seq_s, seq_e);
  const bool fused = p.z != nullptr;
  const size_t HvG = (size_t)w.G * p.Hv;

  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, T_SL_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_in[b], 1);
      mbar_init(&bar_v[b], 1);
      mbar_init(&bar_z[b], 1);
      mbar_init(&bar_nm[b], 1);
      mbar_init(&bar_q[b], 1);
      mbar_init(&bar_free[b], 1);
      mbar_init(&bar_r[b], 2);
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(&bar_s[q], 2);
      mbar_init(&bar_d[q], 2);
    }
    mbar_init(&bar_m1, 1);
    mbar_init(&bar_m3, 1);
    mbar_init(&bar_m5, 1);
    mbar_init(&bar_fin, 1);
    mbar_init(&bar_oe[0], 2);
    mbar_init(&bar_oe[1], 2);
    s_abort = 0;
    fence_mbar_init();
    if (fused) {
      for (int e = 0; e < kSl; ++e) snw[e] = p.norm_w[j0 + e];
      // the norm exchange of chunks 0 and 1 (re-armed after each use): the
      // three peers' 64 sums each
      mbar_arrive_expect_tx(&bar_nm[0], kNormBytes);
      mbar_arrive_expect_tx(&bar_nm[1], kNormBytes);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  // every CTA's barriers exist before a peer can signal them
  cluster_arrive_release();
  cluster_wait_acquire();
  tc::fence_after_sync();
  const uint32_t tb = s_tmem;
  volatile int* abort_flag = &s_abort;
  auto chunk_c0 = [&](int k) { return seq_s + (int64_t)kC * k; };
  auto slot_of = [&](int k) { return (size_t)(kb + k) * p.Hv + h; };

  uint32_t n_in0 = 0, n_in1 = 0;  // loads issued per buffer (the exit path waits for them)
  const bool loader = warp == kSlLoadWarp && lane == 0;

  if (loader) {
    // chunk k's inputs into buffer k & 1; chunk k + 2 follows once the last
    // MMA reading chunk k's buffer has completed (bar_free)
    auto load = [&](int k) {
      const int b = k & 1;
      if (b) ++n_in1; else ++n_in0;
      uint64_t* bi = &bar_in[b];
      uint64_t* bv = &bar_v[b];
      mbar_arrive_expect_tx(bi, kSlInBytes);
      mbar_arrive_expect_tx(bv, kSlVBytes);
      const int y = (int)chunk_c0(k);
      unsigned char* kq = sm + L_KQ + b * 32768;
      tc::tma_load_2d(kq, &tm_k, kh * kD, y, bi);
      tc::tma_load_2d(kq + 16384, &tm_k, kh * kD + 64, y, bi);
      tc::tma_load_2d(kq + 8192, &tm_q, kh * kD, y, bi);
      tc::tma_load_2d(kq + 24576, &tm_q, kh * kD + 64, y, bi);
      const size_t slot = slot_of(k);
      tc::tma_load_2d(sm + L_TB + b * 16384, &tm_w, 0, (int)(slot * kC), bi);
      tc::tma_load_2d(sm + L_TB + b * 16384 + 8192, &tm_w, 0, (int)((HvG + slot) * kC), bi);
      tc::tma_load_2d(sm + L_P + b * 8192, &tm_w, 0, (int)((2 * HvG + slot) * kC), bi);
      tc::tma_load_2d(sm + L_KT + b * 16384, &tm_kt, 0, (int)(((kb + k) * p.Hk + kh) * kD), bi);
      tc::tma_load_2d(sm + L_V + b * 4096, &tm_v, h * kD + j0, y, bv);
      bulk_load(sm + L_VEC + b * 1024, w.vec + slot * (4 * kC), 1024u, bv);
    };
    load(0);
    if (nch > 1) load(1);
    for (int k = 0; k + 2 < nch; ++k) {
      if (!wait_sleepy(&bar_free[k & 1], (uint32_t)((k >> 1) & 1), abort_flag)) break;
      load(k + 2);
    }
  } else if (warp == kSlIssueWarp) {
    // A K-major (TMA tiles), B MN-major (bit 16): [S hi | S lo], [R hi | R lo],
    // [X hi | Y hi] (N = 64) and [(dk X) hi | (dk X) lo | (dk Y) hi] (N = 96)
    const uint32_t id64 = tc::idesc(tc::kBF16, 128, 2 * kSl) | (1u << 16);
    const uint32_t id96 = tc::idesc(tc::kBF16, 128, 3 * kSl) | (1u << 16);
    const uint64_t d_kq = tc::sdesc_sw128(smem_u32(sm + L_KQ)), d_tb = tc::sdesc_sw128(smem_u32(sm + L_TB)),
                   d_kt = tc::sdesc_sw128(smem_u32(sm + L_KT)),
                   d_pw = tc::sdesc_sw128(smem_u32(sm + L_P - 8192)),
                   d_s = sdesc_mn64(smem_u32(sm + L_SH), L_SL - L_SH),
                   d_r = sdesc_mn64(smem_u32(sm + L_RH), L_RL - L_RH),
                   d_d = sdesc_mn64(smem_u32(sm + L_DXH), L_DXL - L_DXH),
                   d_xy = sdesc_mn64(smem_u32(sm + L_XH), L_YH - L_XH);
    for (int k = 0; k < nch; ++k) {
      const uint32_t ph = (uint32_t)(k & 1);
      const int b = k & 1;
      bool ok = chain_wait(&bar_in[b], (uint32_t)((k >> 1) & 1), abort_flag);
      // the output columns of buffer b are free once chunk k - 2's are read
      if (ok && k >= 2) ok = chain_wait(&bar_oe[b], (uint32_t)(((k - 2) >> 1) & 1), abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint32_t t_kqs = tb + T_KQS + 64 * b, t_pd = tb + T_PD + 64 * b;
      const uint64_t akq = d_kq + (uint64_t)((b * 32768) >> 4), atb = d_tb + (uint64_t)((b * 16384) >> 4),
                     akt = d_kt + (uint64_t)((b * 16384) >> 4), apw = d_pw + (uint64_t)((b * 8192) >> 4);
      // (1) quadrant q of the state copies holds K = i of k-steps 2q, 2q + 1
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ok = __all_sync(0xffffffffu, chain_wait(&bar_s[q], ph, abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
        tc::mma_f16_elect2(t_kqs, tc::sdesc_at(akq, 128, 2 * q), sdesc_mn64_at(d_s, 2 * q),
                           tc::sdesc_at(akq, 128, 2 * q + 1), sdesc_mn64_at(d_s, 2 * q + 1), id64, q > 0);
      }
      if (!ok) break;
      tc::mma_commit_elect(&bar_m1);    // the carry's (2)
      tc::mma_commit_elect(&bar_q[b]);  // the output's QS (a barrier per buffer: the output
                                        // warps may be a chunk behind)
      // (3) R rows t of quadrant q (0, 1) are K = s of k-steps 2q, 2q + 1
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        ok = __all_sync(0xffffffffu, chain_wait(&bar_r[q], ph, abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
        tc::mma_f16_elect2(tb + T_XY, tc::sdesc_at(atb, 128, 2 * q), sdesc_mn64_at(d_r, 2 * q),
                           tc::sdesc_at(atb, 128, 2 * q + 1), sdesc_mn64_at(d_r, 2 * q + 1), id64, q > 0);
      }
      if (!ok) break;
      tc::mma_commit_elect(&bar_m3);
      // (5) rows t = 32h.. of dk X come from quadrant h, of dk Y from
      // quadrant 2 + h: k-steps 2h, 2h + 1 once both are in
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        ok = __all_sync(0xffffffffu, chain_wait(&bar_d[hh], ph, abort_flag) &&
                                         chain_wait(&bar_d[2 + hh], ph, abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
        tc::mma_f16_elect2(tb + T_S, tc::sdesc_at(akt, 128, 2 * hh), sdesc_mn64_at(d_d, 2 * hh),
                           tc::sdesc_at(akt, 128, 2 * hh + 1), sdesc_mn64_at(d_d, 2 * hh + 1), id96, true);
      }
      if (!ok) break;
      tc::mma_commit_elect(&bar_m5);
#pragma unroll
      for (int ks = 0; ks < 4; ks += 2)
        tc::mma_f16_elect2(t_pd, tc::sdesc_at(apw, 128, ks), sdesc_mn64_at(d_xy, ks), tc::sdesc_at(apw, 128, ks + 1),
                           sdesc_mn64_at(d_xy, ks + 1), id64, ks > 0);
      tc::mma_commit_elect(&bar_free[b]);  // the loader's reuse of buffer b, the output's P Dm
    }
  } else if (warp < 8) {
    // ============ carry: warp (q, hf) = (warp % 4, warp / 4) reads TMEM lanes
    // 32q.. and handles this CTA's value rows jl = 16 hf .. 16 hf + 15
    const int q = warp & 3, jl = 16 * (warp >> 2);
    const uint32_t tl = tb + ((uint32_t)(32 * q) << 16);
    const int i = 32 * q + lane;  // key column (state lane)
    float* gS = p.state + (((size_t)n * p.Hv + h) * kD + j0 + jl) * kD + i;  // row e at gS[e * kD]

    // the state's 16 values -> hi/lo B tiles, handed to (1) at once, then
    // the accumulator: the first partial holds the state rescaled by gl, the
    // other two restart from zero. Only (5) reads the accumulator, after
    // every carry warp's next hand-off, each of which waits for this warp's
    // TMEM stores first.
    auto store_state = [&](float (&v)[16], float gl) {
      put16_hilo(sm, L_SH, L_SL, i, jl, v);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_s[q]);
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] *= gl;
      tc::tmem_st16(tl + T_S + jl, v);
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = 0.f;
      tc::tmem_st16(tl + T_S + kSl + jl, v);
      tc::tmem_st16(tl + T_S + 2 * kSl + jl, v);
    };

    bool to = !chain_wait(&bar_v[0], 0, abort_flag);
    to = __any_sync(0xffffffffu, to);
    if (!to) {
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = gS[(size_t)e * kD];
      store_state(v, reinterpret_cast<const float*>(sm + L_VEC)[3 * kC]);
    }
    for (int k = 0; k < nch && !to; ++k) {
      const uint32_t ph = (uint32_t)(k & 1);
      const int b = k & 1;
      const int64_t c0 = chunk_c0(k);
      const int L = (int)((seq_e - c0) < kC ? (seq_e - c0) : kC);
      const float* vec = reinterpret_cast<const float*>(sm + L_VEC + b * 1024);
      const bool more = k + 1 < nch;
      to = !chain_wait(&bar_v[b], (uint32_t)((k >> 1) & 1), abort_flag);
      if (q < 2) {
        // (2) R rows t = 32q + lane (V and the vectors landed long before
        // (1) completes: checked first)
        to = to || !chain_wait(&bar_m1, ph, abort_flag);
        if (__any_sync(0xffffffffu, to)) break;
        tc::fence_after_sync();
        const int t = i;
        float ks[16], ks2[16];
        tc::tmem_ld16(tl + T_KQS + 64 * b + jl, ks);
        tc::tmem_ld16(tl + T_KQS + 64 * b + kSl + jl, ks2);
        const uint4* vp = reinterpret_cast<const uint4*>(sm + L_V + b * 4096 + t * (kSl * 2) + jl * 2);
        const uint4 va = vp[0], vb = vp[1];
        const float ak = vec[t];
        tc::tmem_wait_ld();
        const uint32_t vw[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
        const bool live = t < L;
#pragma unroll
        for (int e = 0; e < 16; ++e) ks[e] += ks2[e];
        float r[16];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&vw[m]);
          r[2 * m] = live ? __low2float(v2) - ak * ks[2 * m] : 0.f;
          r[2 * m + 1] = live ? __high2float(v2) - ak * ks[2 * m + 1] : 0.f;
        }
        put16_hilo(sm, L_RH, L_RL, t, jl, r);
        operands_done(&bar_r[q], lane);
      }
      // (4) X (quadrants 0, 1) or Y (2, 3) of rows t = 32 (q % 2) + lane
      to = to || !chain_wait(&bar_m3, ph, abort_flag);
      if (__any_sync(0xffffffffu, to)) break;
      tc::fence_after_sync();
      {
        const int t = 32 * (q & 1) + lane;
        float x[16], x2[16];
        tc::tmem_ld16(tl + T_XY + jl, x);
        tc::tmem_ld16(tl + T_XY + kSl + jl, x2);
        const float dk = vec[kC + t];
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] += x2[e];
        put16(sm, q < 2 ? L_XH : L_YH, t, jl, x);
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] *= dk;
        if (q < 2)
          put16_hilo(sm, L_DXH, L_DXL, t, jl, x);
        else
          put16(sm, L_DYH, t, jl, x);
        operands_done(&bar_d[q], lane);
      }
      // (6) the new state: operand copies and the next chunk's decay; after
      // the last chunk, back to global memory
      to = !chain_wait(&bar_m5, ph, abort_flag);
      if (more) to = to || !chain_wait(&bar_v[(k + 1) & 1], (uint32_t)(((k + 1) >> 1) & 1), abort_flag);
      if (__any_sync(0xffffffffu, to)) break;
      tc::fence_after_sync();
      float v[16], v1[16], v2[16];
      tc::tmem_ld16(tl + T_S + jl, v);
      tc::tmem_ld16(tl + T_S + kSl + jl, v1);
      tc::tmem_ld16(tl + T_S + 2 * kSl + jl, v2);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] += v1[e] + v2[e];
      if (!more) {
#pragma unroll
        for (int e = 0; e < 16; ++e) gS[(size_t)e * kD] = v[e];
      } else {
        store_state(v, reinterpret_cast<const float*>(sm + L_VEC + ((k + 1) & 1) * 1024)[3 * kC]);
      }
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
  } else if (warp >= 10) {
    // ============ output: thread u owns token row t = u (TMEM lane 64 + t)
    // and this CTA's 32 columns j. QS is read once (1) completes and P Dm
    // once its MMAs do; then TMEM is released to the next chunk but one. With
    // the fused norm each row's sum of squares goes to all four CTAs
    // (distributed shared memory), z arrives by TMA two chunks ahead into a
    // row-major tile (two, by chunk parity), and the gated result leaves from
    // a staging tile of its own (two), a full chunk as one tile store.
    const int u = tid - 10 * 32, t = u;
    const uint32_t tl = tb + ((uint32_t)(32 * (warp & 3)) << 16);
    uint32_t n_z0 = 0, n_z1 = 0;
    bool stored = false;
    auto load_z = [&](int k) {
      if (k & 1) ++n_z1; else ++n_z0;
      mbar_arrive_expect_tx(&bar_z[k & 1], 4096u);
      tc::tma_load_2d(sm + L_Z + (k & 1) * 4096, &tm_z, h * kD + j0, (int)chunk_c0(k), &bar_z[k & 1]);
    };
    if (fused && u == 0) {
      load_z(0);
      if (nch > 1) load_z(1);
    }
    // A bounded wait that gave up stops the stores but, with the fused norm,
    // not the exchange: every CTA sends its sums for every chunk and takes
    // its peers' before it goes on, so no copy into a CTA's shared memory is
    // in flight when it exits (unless a peer stops answering altogether, when
    // the time limit ends the wait).
    bool to = false;  // a bounded wait gave up (agreed on at the chunk's barrier)
    for (int k = 0; k < nch; ++k) {
      const int b = k & 1;
      const int64_t c0 = chunk_c0(k);
      const int L = (int)((seq_e - c0) < kC ? (seq_e - c0) : kC);
      const float gq = __ldg(w.vec + slot_of(k) * (4 * kC) + 2 * kC + t);
      // QS (its S hi and S lo parts summed) once (1) completes
      float a[32], o[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0.f;
      to |= !wait_sleepy(&bar_q[b], (uint32_t)((k >> 1) & 1), abort_flag);
      if (!__any_sync(0xffffffffu, to)) {
        tc::fence_after_sync();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float x[16], y[16];
          tc::tmem_ld16(tl + T_KQS + 64 * b + 16 * hh, x);
          tc::tmem_ld16(tl + T_KQS + 64 * b + kSl + 16 * hh, y);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) a[16 * hh + e] = x[e] + y[e];
        }
      }
      // then gq QS + P (X hi + Y hi)
      to |= !wait_sleepy(&bar_free[b], (uint32_t)((k >> 1) & 1), abort_flag);
      if (!__any_sync(0xffffffffu, to)) {
        tc::fence_after_sync();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float x[16], y[16];
          tc::tmem_ld16(tl + T_PD + 64 * b + 16 * hh, x);
          tc::tmem_ld16(tl + T_PD + 64 * b + kSl + 16 * hh, y);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[16 * hh + e] = fmaf(gq, a[16 * hh + e], x[e] + y[e]);
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_oe[b]);  // this chunk's output accumulators are free
      if (fused && p.core_out != nullptr && t < L && !to) {
        float4* cg = reinterpret_cast<float4*>(p.core_out + ((c0 + t) * p.Hv + h) * kD + j0);
#pragma unroll
        for (int m = 0; m < 8; ++m) cg[m] = make_float4(o[4 * m], o[4 * m + 1], o[4 * m + 2], o[4 * m + 3]);
      }
      if (fused) {
        // this slice's sum of squares of row t to the other three CTAs (an
        // asynchronous store that completes on the receiver's mbarrier), and
        // into this CTA's own slot
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) ss = fmaf(o[e], o[e], ss);
        const uint32_t slot = smem_u32(&snorm[b][rank][t]), nb = smem_u32(&bar_nm[b]);
#pragma unroll
        for (uint32_t r = 0; r < (uint32_t)kSlCta; ++r) {
          if (r == rank)
            snorm[b][rank][t] = ss;
          else
            st_async_cluster_f32(map_shared_rank(slot, r), ss, map_shared_rank(nb, r));
        }
      }
      if (!fused) {
        // the core output: a full chunk leaves as one tile store from a
        // staging tile (two, by chunk parity, in the z and output tiles'
        // space, unused without the fused norm; 16-byte group m of row t at
        // group m ^ (t % 8), the tensor map's 128-byte swizzle); a
        // sequence's last, partial chunk by rows
        const bool full_tile = L == kC;
        if (p.core_out != nullptr && !to) {
          if (full_tile) {
            unsigned char* stg = sm + (b ? L_O : L_Z);
#pragma unroll
            for (int m = 0; m < 8; ++m)
              *reinterpret_cast<float4*>(stg + t * 128 + ((m ^ (t & 7)) << 4)) =
                  make_float4(o[4 * m], o[4 * m + 1], o[4 * m + 2], o[4 * m + 3]);
            fence_proxy_async_smem();
          } else if (t < L) {
            float4* cg = reinterpret_cast<float4*>(p.core_out + ((c0 + t) * p.Hv + h) * kD + j0);
#pragma unroll
            for (int m = 0; m < 8; ++m) cg[m] = make_float4(o[4 * m], o[4 * m + 1], o[4 * m + 2], o[4 * m + 3]);
          }
        }
        // the previous chunk's tile store has read the other staging tile
        // (written again next chunk) before the rows pass the barrier
        if (u == 0 && stored) bulk_wait_read_all();
        if (bar_or(3, kSlOutThreads, to)) break;
        if (u == 0 && full_tile && p.core_out != nullptr) {
          tc::tma_store_2d(&tm_o, h * kD + j0, (int)c0, sm + (b ? L_O : L_Z));
          bulk_commit();
          stored = true;
        }
        continue;
      }
      // the gate nw silu(z) while the peers' sums are on their way
      if (!to) to = !wait_sleepy(&bar_z[b], (uint32_t)((k >> 1) & 1), abort_flag);
      const uint4* zr = reinterpret_cast<const uint4*>(sm + L_Z + b * 4096 + t * (kSl * 2));
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint4 zw = zr[m];
        const uint32_t zz[4] = {zw.x, zw.y, zw.z, zw.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const __nv_bfloat162 z2 = *reinterpret_cast<const __nv_bfloat162*>(&zz[c]);
          const int e = 8 * m + 2 * c;
          const float z0 = __low2float(z2), z1 = __high2float(z2);
          o[e] *= snw[e] * __fdividef(z0, 1.f + __expf(-z0));
          o[e + 1] *= snw[e + 1] * __fdividef(z1, 1.f + __expf(-z1));
        }
      }
      // the peers' sums (a wait limited by time only: see above; all 64 rows
      // agree on giving up)
      const bool lost = !wait_sleepy(&bar_nm[b], (uint32_t)((k >> 1) & 1), nullptr);
      if (bar_or(4, kSlOutThreads, lost)) {
        *abort_flag = 1;
        break;
      }
      float tot = 0.f;
#pragma unroll
      for (int r = 0; r < kSlCta; ++r) tot += snorm[b][r][t];
      // (a peer writes this buffer again only after every row here has sent
      // chunk k + 1's sums, i.e. after these reads)
      if (u == 0 && k + 2 < nch) mbar_arrive_expect_tx(&bar_nm[b], kNormBytes);
      const float rs = 1.f / sqrtf(tot / (float)kD + p.rms_eps);
      // (the staging tile b was last stored from two chunks ago; thread 0
      // waited for that store's reads before the previous chunk's barrier)
      uint4* orow = reinterpret_cast<uint4*>(sm + L_O + b * 4096 + t * (kSl * 2));
#pragma unroll
      for (int m = 0; m < 4; ++m)
        orow[m] = make_uint4(pack_bf16(o[8 * m] * rs, o[8 * m + 1] * rs), pack_bf16(o[8 * m + 2] * rs, o[8 * m + 3] * rs),
                             pack_bf16(o[8 * m + 4] * rs, o[8 * m + 5] * rs),
                             pack_bf16(o[8 * m + 6] * rs, o[8 * m + 7] * rs));
      fence_proxy_async_smem();
      // the previous chunk's store has read its staging tile (rewritten next
      // chunk) before this barrier
      if (u == 0 && stored) bulk_wait_read_all();
      to = bar_or(3, kSlOutThreads, to);
      if (to) continue;  // no more stores or loads; the exchange goes on
      const __nv_bfloat16* ob = reinterpret_cast<const __nv_bfloat16*>(sm + L_O + b * 4096);
      if (L == kC) {
        // a full chunk leaves as one tile
        if (u == 0) {
          tc::tma_store_2d(&tm_o, h * kD + j0, (int)c0, ob);
          bulk_commit();
          stored = true;
        }
      } else if (t < L) {
        // the sequence's last chunk: row by row, so no row of the next
        // sequence is written
        bulk_store(static_cast<__nv_bfloat16*>(p.out) + ((c0 + t) * p.Hv + h) * kD + j0, ob + t * kSl,
                   (uint32_t)(kSl * 2));
        bulk_commit();
        stored = true;
      }
      // every row has read z of chunk k: chunk k + 2's into its tile
      if (u == 0 && k + 2 < nch) load_z(k + 2);
    }
    if (stored) bulk_wait_all();
    if (u == 0) {
      if (n_z0) mbar_wait(&bar_z[0], (n_z0 - 1) & 1);
      if (n_z1) mbar_wait(&bar_z[1], (n_z1 - 1) & 1);
    }
  }

  // drain: every copy and MMA this CTA issued has completed, and every CTA
  // of the cluster is done writing into its peers' shared memory, before
  // TMEM is released and the CTA exits
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kSlIssueWarp) {
    tc::fence_after_sync();
    tc::mma_commit_elect(&bar_fin);
    mbar_wait(&bar_fin, 0);
    tc::fence_before_sync();
  }
  if (loader) {
    if (n_in0) {
      mbar_wait(&bar_in[0], (n_in0 - 1) & 1);
      mbar_wait(&bar_v[0], (n_in0 - 1) & 1);
    }
    if (n_in1) {
      mbar_wait(&bar_in[1], (n_in1 - 1) & 1);
      mbar_wait(&bar_v[1], (n_in1 - 1) & 1);
    }
  }
  __syncthreads();
  cluster_arrive_release();
  cluster_wait_acquire();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tb, T_SL_COLS);
  }
}

// ------------------------------------------------------- separate norm

// The gated RMSNorm of the sliced carry's fp32 core output (the same formula
// as the fused epilogues): rows (t, h) of the tokens the sequences cover,
// [cu_seqlens[0], cu_seqlens[N]). A warp takes four rows, each lane the same
// four columns of each (one coalesced 512-byte row per load), all eight
// loads issued before the reductions. Runs after the carry on the same
// stream.
constexpr int kNormRowsPerWarp = 4;
constexpr int kNormRowsPerBlock = 8 * kNormRowsPerWarp;  // 256 threads
__global__ void __launch_bounds__(256) cp_norm_kernel(const PrefillArgs p, const float* __restrict__ o) {
  int64_t lo = p.cu_seqlens[0], hi = p.cu_seqlens[p.N];
  lo = lo < 0 ? 0 : (lo > p.T ? p.T : lo);
  hi = hi < lo ? lo : (hi > p.T ? p.T : hi);
  const int lane = threadIdx.x & 31, c0 = 4 * lane;
  const int64_t rows_end = hi * p.Hv;
  const int64_t stride = (int64_t)gridDim.x * kNormRowsPerBlock;
  const float4 w = *reinterpret_cast<const float4*>(p.norm_w + c0);
  for (int64_t r0 = lo * p.Hv + (int64_t)blockIdx.x * kNormRowsPerBlock + kNormRowsPerWarp * (threadIdx.x >> 5);
       r0 < rows_end; r0 += stride) {
    float4 v[kNormRowsPerWarp];
    uint2 zw[kNormRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kNormRowsPerWarp; ++r) {
      v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      zw[r] = make_uint2(0u, 0u);
      if (r0 + r < rows_end) {  // (uniform across the warp)
        v[r] = *reinterpret_cast<const float4*>(o + (r0 + r) * kD + c0);
        zw[r] = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.z) + (r0 + r) * kD + c0);
      }
    }
#pragma unroll
    for (int r = 0; r < kNormRowsPerWarp; ++r) {
      const float ss = group_sum<32>(v[r].x * v[r].x + v[r].y * v[r].y + v[r].z * v[r].z + v[r].w * v[r].w);
      const float inv = 1.f / sqrtf(ss / (float)kD + p.rms_eps);
      const __nv_bfloat162 z01 = *reinterpret_cast<const __nv_bfloat162*>(&zw[r].x);
      const __nv_bfloat162 z23 = *reinterpret_cast<const __nv_bfloat162*>(&zw[r].y);
      uint2 y;
      y.x = pack_bf16(v[r].x * inv * w.x * silu_fast(__low2float(z01)),
                      v[r].y * inv * w.y * silu_fast(__high2float(z01)));
      y.y = pack_bf16(v[r].z * inv * w.z * silu_fast(__low2float(z23)),
                      v[r].w * inv * w.w * silu_fast(__high2float(z23)));
      if (r0 + r < rows_end)
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + (r0 + r) * kD + c0) = y;
    }
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

bool prefill_cp_sliced(const PrefillArgs& p) {
  if (p.flags & GDN_PREFILL_CARRY_SLICED) return true;
  if (p.flags & GDN_PREFILL_CARRY_WHOLE) return false;
  // four CTAs per (V head, sequence) pay where the whole-row carries would
  // leave most SMs idle: at most two waves of sliced CTAs
  if ((int64_t)p.Hv * p.N > kSlMaxChains) return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  return (int64_t)kSlCta * p.Hv * p.N <= 2 * (int64_t)sms;
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
  if (prefill_cp_sliced(p)) {
    // With the gated norm, the carry writes the fp32 core output (core_out,
    // else the workspace's region for it) and a separate pass normalises it:
    // the norm's work in the carry's output warps slows the carry's own
    // phases on the SMs it shares. Without such a buffer (the sliced carry
    // forced for many pairs), the carry's output warps apply it themselves.
    PrefillArgs ps = p;
    const bool defer = p.z != nullptr && (p.core_out != nullptr || l.off_o != 0);
    if (defer) {
      ps.z = nullptr;
      if (ps.core_out == nullptr) ps.core_out = reinterpret_cast<float*>(static_cast<char*>(workspace) + l.off_o);
    }
    CUtensorMap mv32, mz32, mo32;
    memset(&mz32, 0, sizeof(mz32));
    memset(&mo32, 0, sizeof(mo32));
    if (!tc::make_map_2d(&mv32, p.v, p.T, vc, p.v_stride, 2, bf, kSl, 64, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    if (ps.z != nullptr &&
        (!tc::make_map_2d(&mz32, p.z, p.T, vc, vc, 2, bf, kSl, 64, CU_TENSOR_MAP_SWIZZLE_NONE) ||
         !tc::make_map_2d(&mo32, p.out, p.T, vc, vc, 2, bf, kSl, 64, CU_TENSOR_MAP_SWIZZLE_NONE)))
      return cudaErrorInvalidValue;
    // without the fused norm the output map is the fp32 core output's, in
    // tiles of 64 tokens x 32 columns (128 bytes, swizzled)
    if (ps.z == nullptr && ps.core_out != nullptr &&
        !tc::make_map_2d(&mo32, ps.core_out, p.T, vc, vc, 4, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kSl, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(cp_slice_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L_SMEM);
    if (e != cudaSuccess) return e;
    cp_slice_kernel<<<dim3((unsigned)(kSlCta * p.Hv), (unsigned)p.N), kSlThreads, L_SMEM, stream>>>(
        ps, w, mq, mk, mv32, mw, mz32, mkt, mo32);
    e = cudaGetLastError();
    if (e != cudaSuccess || !defer) return e;
    const int64_t rows = p.T * p.Hv;
    const int64_t need = (rows + kNormRowsPerBlock - 1) / kNormRowsPerBlock;
    const int64_t blocks = need < 65536 ? need : 65536;
    cp_norm_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, ps.core_out);
    return cudaGetLastError();
  }
  e = cudaFuncSetAttribute(cp_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM);
  if (e != cudaSuccess) return e;
  cp_chain_kernel<<<dim3((unsigned)p.Hv, (unsigned)p.N), kChainAll, C_SMEM, stream>>>(p, w, mq, mk,
                                                                                         mv, mw, mz, mkt, mo);
  return cudaGetLastError();
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(prefill_cp)
