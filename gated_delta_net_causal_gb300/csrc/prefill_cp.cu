// Chunk-parallel prefill on the 5th-generation tensor cores: head_dim 128,
// bf16 activations, chunk 64, three launches over a caller-provided
// workspace.
//
// The chunk algebra (the recurrence of ferrox-core gdn.rs summed chunk-wise;
// the stages of ferrum-kernels gated_delta_attention_tests.rs
// `run_chunked_core`) is split by what depends on the state. Within a chunk
// of L tokens from state S (rows j = value, columns i = key), with c the
// chunk-local cumulative decay, G_t = e^{c_t}, raw k, q and their l2 scales
// rk_t, rq_t (rq includes 1/sqrt(D)):
//
//   state-free, every chunk at once (cp_prep_kernel, one CTA per chunk and
//   K head, looping over the V heads that read it):
//     A   = beta_t e^{c_t-c_s} rk_t rk_s (k_t . k_s)            (s < t)
//     Tb  = (I + A)^{-1} diag(beta)                              (hi + lo bf16)
//     U   = Tb V,  W = Tb diag(G rk) K       (tensor cores)      -> fp32, hi + lo bf16
//     P   = e^{c_t-c_s} rq_t rk_s (q_t . k_s)                    (s <= t) -> bf16
//     dk_t = e^{c_{L-1}-c_t} rk_t,  gq_t = G_t rq_t,  G_{L-1}
//   the scan, one CTA per (V head, sequence), chunk after chunk
//   (cp_scan_kernel; the fp32 state lives in TMEM as an MMA accumulator):
//     Dm^T = U^T - S W^T            (the chunk's delta-rule corrections d_t)
//     S    = G_{L-1} S + (Dm diag(dk))^T K
//     O^T  = S Q^T diag(gq) + Dm^T P^T, then the gated RMSNorm over j.
// Only the two products of the middle line depend on the previous chunk, so
// each chunk costs two dependent MMA groups; S Q^T and Dm^T P^T are issued
// off that chain.
//
// Every product that carries the state forward keeps fp32 accuracy on bf16
// tensor cores by splitting each fp32 factor as x = hi + lo (two bf16 values,
// about 16 significant bits together): S W^T uses S_hi W_hi + S_hi W_lo +
// S_lo W_hi, the update Dm'_hi K + Dm'_lo K, and U and W both halves of Tb
// (raw k and v are exact in bf16). The two output products use the hi parts
// only.
//
// Because the scan CTA owns all 128 value rows of its head, the gated RMSNorm
// of each output row is a reduction inside the CTA: no cluster.
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
constexpr int kAStride = kC + 1;    // padded row pitch of the fp32 A matrix
constexpr int kMaxRep = 8;          // V heads per K head on this path

// ---------------------------------------------------------------- workspace

struct CpWork {
  int32_t* cs;         // [N+1] first chunk slot of each sequence
  __nv_bfloat16* tw;   // [G*Hv*64][64]: P (row-major per slot)
  float* u;            // [G*Hv][128 j][64 t]: U^T = (Tb V)^T per slot (columns t >= L zero)
  __nv_bfloat16* wm;   // [G*Hv][2][64 t][128 i]: W hi, W lo per slot (rows t >= L zero)
  __nv_bfloat16* kt;   // [G*Hk*128][64]: raw k transposed, rows t >= L zero
  float* vec;          // [G*Hv][4][64]: ak, dk, gq, {G_{L-1}, 0...}
  int64_t G;           // chunk slots
};

struct CpLayout {
  int64_t G;
  size_t off_tm, off_u, off_wm, off_kt, off_vec, total;
};

CpLayout cp_layout(int32_t N, int64_t T, int32_t Hk, int32_t Hv) {
  CpLayout l{};
  // sum over sequences of ceil(len/64) <= (T + 63 N) / 64
  l.G = T > 0 ? (T + 63 * (int64_t)N) / kC : 0;
  l.off_tm = ((size_t)4 * ((size_t)N + 1) + 1023) / 1024 * 1024;
  l.off_u = l.off_tm + (size_t)l.G * Hv * kC * kC * 2;
  l.off_wm = l.off_u + (size_t)l.G * Hv * kD * kC * 4;
  l.off_kt = l.off_wm + (size_t)l.G * Hv * 2 * kD * kC * 2;
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

// The k rows of the k/q tile stay until W has been formed from them; the q
// rows are dead once the grams and l2 scales are taken, and then hold the V
// tile of the V head in hand. A and Tm sit after the tile; the raw gate
// inputs overlay Tm until the gates are taken. Once the inverse is complete,
// the hi/lo tiles of Tb diag(G rk) (B of W) overlay A and those of Tb (B of
// U) overlay Tm.
constexpr uint32_t P_OFF_KQ = 0;       // bf16 [128][128 i] SW128 (TMA): rows 0-63 k, 64-127 q
constexpr uint32_t P_OFF_A = 32768;    // fp32 [64][65]; later bf16 [2][64 t][64 s] SW128
constexpr uint32_t P_OFF_T = 50176;    // fp32 [64][64] Tm (products in its upper triangle); 1024-aligned
constexpr uint32_t P_SMEM = 66560 + 1024;
constexpr uint32_t P_TMEM_COLS = 128;  // grams 0-63, U^T and W 64-127
// swizzled operand tiles start on 1024-byte boundaries
static_assert(P_OFF_KQ % 1024 == 0 && P_OFF_A % 1024 == 0 && P_OFF_T % 1024 == 0, "tile alignment");

__global__ void __launch_bounds__(kPrepThreads, 3)
    cp_prep_kernel(const PrefillArgs p, const CpWork w, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(16) float sinvk[kC], sinvq[kC];
  // per V head: beta, the chunk-local cumulative decay c and G = e^c
  __shared__ __align__(16) float sbeta[kMaxRep][kC], sc[kMaxRep][kC], sgam[kMaxRep][kC];
  // raw gate inputs (in the Tm space until the first inverse)
  float (*sga)[kC] = reinterpret_cast<float (*)[kC]>(sm + P_OFF_T);
  float (*sgb)[kC] = reinterpret_cast<float (*)[kC]>(sm + P_OFF_T + kMaxRep * kC * 4);
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t bar_ld, bar_gp, bar_w, bar_v;

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
    tc::tmem_alloc(&s_tmem, P_TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_gp, 1);
    mbar_init(&bar_w, 1);
    mbar_init(&bar_v, 1);
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
  // K^T of this chunk and K head for the scan's state update (its K-major B
  // operand): thread pair (i, half) gathers 32 rows t of column i
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
    if (warp == 0) tc::tmem_dealloc(tb, P_TMEM_COLS);
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
  // the V tile of V head r into the q rows (j halves 16 KB apart)
  auto load_v = [&](int r) {
    const int h = p.map == GDN_MAP_GROUPED ? kh * p.rep + r : kh + r * p.Hk;
    mbar_arrive_expect_tx(&bar_v, 16384u);
    tc::tma_load_2d(sm + P_OFF_KQ + 8192, &tm_v, h * kD, (int)c0, &bar_v);
    tc::tma_load_2d(sm + P_OFF_KQ + 24576, &tm_v, h * kD + 64, (int)c0, &bar_v);
  };
  if (tid == 0) load_v(0);
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
      // columns s, from 16-byte loads of the per-token vectors
      float dks[32];
#pragma unroll
      for (int m4 = 0; m4 < 8; ++m4) {
        const float4 c4 = *reinterpret_cast<const float4*>(&sc[r][32 * hc + 4 * m4]);
        const float4 k4 = *reinterpret_cast<const float4*>(&sinvk[32 * hc + 4 * m4]);
        dks[4 * m4] = exp2f(ct - c4.x * kLog2e) * k4.x;
        dks[4 * m4 + 1] = exp2f(ct - c4.y * kLog2e) * k4.y;
        dks[4 * m4 + 2] = exp2f(ct - c4.z * kLog2e) * k4.z;
        dks[4 * m4 + 3] = exp2f(ct - c4.w * kLog2e) * k4.w;
      }
      if (is_a) {
        const float bk = sbeta[r][t] * sinvk[t];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int s = 32 * hc + e;
          Ap[t * kAStride + s] = (live && s < t) ? bk * dks[e] * gv[e] : 0.f;
        }
      } else {
        const float iqt = sinvq[t];
        float pr[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int s = 32 * hc + e;
          pr[e] = (live && s <= t) ? dks[e] * gv[e] * iqt : 0.f;
        }
        uint4* dst = reinterpret_cast<uint4*>(w.tw + (slot * kC + t) * kC + 32 * hc);
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
    // Tb = Tm diag(beta) and Tb diag(ak) (ak = G rk) as hi + lo bf16 tiles
    // (K-major, zero above the diagonal): Tb over Tm once every thread has
    // read its row of Tm, Tb diag(ak) over the dead A; 16 consecutive
    // elements of one row per thread
    {
      const int e0 = 16 * tid, tr = e0 >> 6, u0 = e0 & 63;
      float x[16], xa[16];
#pragma unroll
      for (int m4 = 0; m4 < 4; ++m4) {
        const float4 t4 = *reinterpret_cast<const float4*>(Tp + tr * kC + u0 + 4 * m4);
        const float4 b4 = *reinterpret_cast<const float4*>(&sbeta[r][u0 + 4 * m4]);
        const float4 g4 = *reinterpret_cast<const float4*>(&sgam[r][u0 + 4 * m4]);
        const float4 k4 = *reinterpret_cast<const float4*>(&sinvk[u0 + 4 * m4]);
        const float tv[4] = {t4.x, t4.y, t4.z, t4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
        const float gv[4] = {g4.x, g4.y, g4.z, g4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = 4 * m4 + e;
          x[m] = u0 + m <= tr ? tv[e] * bv[e] : 0.f;
          xa[m] = x[m] * (gv[e] * kv[e]);
        }
      }
      const int c16 = u0 >> 3;
      uint4 h0, l0, h1, l1;
      split8(xa, h0, l0);
      split8(xa + 8, h1, l1);
      unsigned char* ba = sm + P_OFF_A;
      *reinterpret_cast<uint4*>(ba + sw_chunk(tr, c16, kC)) = h0;
      *reinterpret_cast<uint4*>(ba + sw_chunk(tr, c16 + 1, kC)) = h1;
      *reinterpret_cast<uint4*>(ba + 8192 + sw_chunk(tr, c16, kC)) = l0;
      *reinterpret_cast<uint4*>(ba + 8192 + sw_chunk(tr, c16 + 1, kC)) = l1;
      split8(x, h0, l0);
      split8(x + 8, h1, l1);
      __syncthreads();  // Tm has been read
      unsigned char* bu = sm + P_OFF_T;
      *reinterpret_cast<uint4*>(bu + sw_chunk(tr, c16, kC)) = h0;
      *reinterpret_cast<uint4*>(bu + sw_chunk(tr, c16 + 1, kC)) = h1;
      *reinterpret_cast<uint4*>(bu + 8192 + sw_chunk(tr, c16, kC)) = l0;
      *reinterpret_cast<uint4*>(bu + 8192 + sw_chunk(tr, c16 + 1, kC)) = l1;
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
    // U^T = (Tb V)^T on the tensor cores: A = the V tile read MN-major (j
    // along M, the two j halves 16 KB apart), B = the Tb tiles over Tm; the
    // hi and lo products accumulate into TMEM columns 64-127, and row j
    // (lane j) goes to the workspace as fp32
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    {
      bool bad = false;
      if (tid == 0) {
        bad = !mbar_wait(&bar_v, (uint32_t)(r & 1));
        if (!bad) {
          tc::fence_after_sync();
          const uint32_t id = tc::idesc(tc::kBF16, 128, 64) | tc::kAMajorMN;
          const uint32_t av = smem_u32(sm + P_OFF_KQ + 8192);
          const uint64_t dbh = tc::sdesc_sw128(smem_u32(sm + P_OFF_T));
          const uint64_t dbl = tc::sdesc_sw128(smem_u32(sm + P_OFF_T + 8192));
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint64_t da = tc::sdesc_mn(av + 2048u * s, 16384u);
            tc::mma_f16(tb + 64, da, tc::sdesc_at(dbh, kC, s), id, s > 0);
            tc::mma_f16(tb + 64, da, tc::sdesc_at(dbl, kC, s), id, true);
          }
          tc::mma_commit(&bar_w);
        }
      }
      if (__syncthreads_or(bad) || __syncthreads_or(!mbar_wait(&bar_w, (uint32_t)((3 * r) & 1)))) {
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::tmem_dealloc(tb, P_TMEM_COLS);
        return;
      }
      tc::fence_after_sync();
      const int j = tid & 127, hc = tid >> 7;
      float x[32];
      tc::tmem_ld16(tq + 64 + 32 * hc, *reinterpret_cast<float(*)[16]>(x));
      tc::tmem_ld16(tq + 64 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(x + 16));
      tc::tmem_wait_ld();
      float4* du = reinterpret_cast<float4*>(w.u + (slot * kD + j) * kC + 32 * hc);
#pragma unroll
      for (int m = 0; m < 8; ++m) du[m] = make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
      tc::fence_before_sync();
      __syncthreads();  // every thread has its U columns; the V tile is free
    }
    // W = Tb diag(G rk) K on the tensor cores, rows t contiguous in i (the
    // scan's K-major B operand): A = [hi; lo] tiles of Tb diag(ak) stacked as
    // 128 rows (over the dead A), B = the k rows of the k/q tile read
    // MN-major, one 64-wide i half at a time into TMEM columns 64-127. Row
    // t' of the result is hi_t' K (t' < 64) or lo_{t'-64} K: the lo rows go
    // through shared memory (over the dead Tb tiles, 16-byte chunks
    // XOR-swizzled by row) and are added to the hi rows, which split the sum
    // as hi + lo bf16.
    auto issue_w = [&](int half) {
      tc::fence_after_sync();
      const uint32_t id = tc::idesc(tc::kBF16, 128, 64) | tc::kBMajorMN;
      const uint64_t da = tc::sdesc_sw128(smem_u32(sm + P_OFF_A));
      const uint32_t bk = smem_u32(sm + P_OFF_KQ) + 16384u * half;
#pragma unroll
      for (int s = 0; s < 4; ++s)
        tc::mma_f16(tb + 64, tc::sdesc_at(da, 128, s), tc::sdesc_mn(bk + 2048u * s, 16384u), id, s > 0);
      tc::mma_commit(&bar_w);
    };
    if (tid == 0) {
      issue_w(0);
      if (r + 1 < p.rep) load_v(r + 1);
    }
    float* xb = Tp;  // [64][64] fp32 exchange of the lo rows
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      if (__syncthreads_or(!mbar_wait(&bar_w, (uint32_t)((3 * r + 1 + half) & 1)))) {
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::tmem_dealloc(tb, P_TMEM_COLS);
        return;
      }
      tc::fence_after_sync();
      const int row = tid & 127, hc = tid >> 7;
      float x[32];
      tc::tmem_ld16(tq + 64 + 32 * hc, *reinterpret_cast<float(*)[16]>(x));
      tc::tmem_ld16(tq + 64 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(x + 16));
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncthreads();  // every thread has its columns: the next half may overwrite them
      if (tid == 0 && half == 0) issue_w(1);
      if (row >= kC) {
        const int tr = row - kC;
#pragma unroll
        for (int m = 0; m < 8; ++m)
          *reinterpret_cast<float4*>(xb + tr * kC + 4 * ((8 * hc + m) ^ (tr & 7))) =
              make_float4(x[4 * m], x[4 * m + 1], x[4 * m + 2], x[4 * m + 3]);
      }
      __syncthreads();
      if (row < kC) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const float4 lo4 = *reinterpret_cast<const float4*>(xb + row * kC + 4 * ((8 * hc + m) ^ (row & 7)));
          x[4 * m] += lo4.x;
          x[4 * m + 1] += lo4.y;
          x[4 * m + 2] += lo4.z;
          x[4 * m + 3] += lo4.w;
        }
        uint4* dh = reinterpret_cast<uint4*>(w.wm + ((slot * 2) * kC + row) * kD + 64 * half + 32 * hc);
        uint4* dl = reinterpret_cast<uint4*>(w.wm + ((slot * 2 + 1) * kC + row) * kD + 64 * half + 32 * hc);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint4 hv, lv;
          split8(x + 8 * m, hv, lv);
          dh[m] = hv;
          dl[m] = lv;
        }
      }
      __syncthreads();  // the exchange buffer is reused by the next half
    }
    tc::fence_before_sync();
    __syncthreads();  // A, Tm and the W columns are rewritten for the next V head
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, P_TMEM_COLS);
}

// ------------------------------------------------------------------ scan

// Shared memory (byte offsets from a 1024-aligned base). The per-chunk
// workspace tiles are double-buffered by chunk parity and loaded a chunk
// ahead; V, K and Q are single tiles reloaded as soon as their MMA completes.
constexpr uint32_t ST_U = 0;           // fp32 [2][128 j][32 t] SW128 (two t halves): U^T
constexpr uint32_t ST_WHI = 32768;     // bf16 [64 t][128 i] SW128 (two i halves): W hi, K-major B
constexpr uint32_t ST_WLO = 49152;     // W lo
constexpr uint32_t ST_VEC = 65536;     // fp32 [4][64]: ak, dk, gq, {G_{L-1}}
constexpr uint32_t ST_BYTES = 66560;   // one stage
constexpr uint32_t SO_P = 2 * ST_BYTES;        // bf16 [64 t][64 s] SW128: P (K-major B of Dm^T P^T)
constexpr uint32_t SO_K = SO_P + 8192;         // bf16 [128 i][64 t] SW128: k transposed, K-major B of the update
constexpr uint32_t SO_Q = SO_K + 16384;        // bf16 [64 t][128 i] two i halves: K-major B of S Q^T
constexpr uint32_t SO_DL = SO_Q + 16384;       // bf16 [128 j][64 t] SW128: Dm' lo, K-major A
constexpr uint32_t SO_Z = SO_DL + 16384;       // bf16 [2][64 t][128 j] row-major: z (TMA), then out
constexpr uint32_t S_SMEM = SO_Z + 32768 + 1024;
static_assert(ST_U % 1024 == 0 && ST_WHI % 1024 == 0 && ST_WLO % 1024 == 0 && ST_BYTES % 1024 == 0 &&
                  SO_P % 1024 == 0 && SO_K % 1024 == 0 && SO_Q % 1024 == 0 && SO_DL % 1024 == 0 &&
                  SO_Z % 1024 == 0,
              "tile alignment");

// TMEM columns. A operands are packed bf16 pairs (row j in lane j, K
// elements 2c, 2c+1 in column c). A region is rewritten only after an MMA
// commit or a barrier of its readers covers the previous contents.
constexpr uint32_t TS_HI = 0;    // S hi (64): A of S W^T and S Q^T
constexpr uint32_t TS_LO = 64;   // S lo (64)
constexpr uint32_t TS_Y = 128;   // fp32 -S W^T (64); Dm^T = U^T + this
constexpr uint32_t TS_S = 192;   // fp32 S (128): the state accumulator, pre-scaled by G_{L-1}
constexpr uint32_t TS_DH = 320;  // (dk Dm)^T hi (32): A of the update
constexpr uint32_t TS_DM = 352;  // Dm^T hi (32): A of Dm^T P^T
constexpr uint32_t TS_OQ = 384;  // fp32 S Q^T (64)
constexpr uint32_t TS_DP = 448;  // fp32 Dm^T P^T (64)

constexpr int kScanThreads = 576;  // warp 0 loads, warp 1 MMAs, 2-9 state, 10-17 output
constexpr int kOutThreads = 256;

// Bounded wait that gives up at once when another role has given up.
__device__ __forceinline__ bool chain_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait_bounded(bar, parity, abort_flag);
}

// A warp hands TMEM (and shared-memory) operands it wrote to the MMA warp.
__device__ __forceinline__ void warp_done(uint64_t* bar, int lane) {
  tc::tmem_wait_st();
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Per chunk c, the MMA warp's order (each group waits for its operands):
//   (a) Y = -(S_hi W_hi^T + S_hi W_lo^T + S_lo W_hi^T), in two K halves as
//       the state copies arrive (conv1(c-1) has read Y by then)
//   (o) OQ = S_hi Q^T                               once the output warps read OQ(c-1)
//   (c) S += Dm'_hi K + Dm'_lo K, in two K halves   as conv1(c) writes Dm'
//   (p) DP = Dm_hi P^T                              once the output warps read DP(c-1)
// The state warps: conv1(c) after (a): Dm^T = U^T + Y, Dm' = Dm diag(dk) as
// hi (TMEM) + lo (shared memory), Dm_hi (TMEM); conv2(c) after (c): the new
// state's hi/lo copies, the accumulator rescaled by the next chunk's
// G_{L-1}. Only (a) -> conv1 -> (c) -> conv2 -> (a) is a dependent chain;
// (o), (p) and the output warps' gated norm run beside it.
__global__ void __launch_bounds__(kScanThreads, 1)
    cp_scan_kernel(const PrefillArgs p, const CpWork w, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_u,
                   const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_wm,
                   const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_z,
                   const __grid_constant__ CUtensorMap tm_o) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t bar_st[2], bar_p, bar_k, bar_q, bar_z[2];
  __shared__ __align__(8) uint64_t bar_a, bar_oq, bar_cc, bar_dp, bar_fin;
  // bar_s[q]: the state copies of column batch q (k-steps {0,1,4,5} / {2,3,6,7});
  // bar_c1[b]: the corrections of token batch b (k-steps {0,2} / {1,3})
  __shared__ __align__(8) uint64_t bar_s[2], bar_c1[2], bar_oqe, bar_dpe;
  // per stage slot (so no waiter can fall two phases behind): the stage's
  // MMAs have completed, the output warps have copied its gq
  __shared__ __align__(8) uint64_t bar_sf[2], bar_gq[2];
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

  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, 512);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_st[b], 1);
      mbar_init(&bar_z[b], 1);
      mbar_init(&bar_sf[b], 1);
      mbar_init(&bar_gq[b], 8);
    }
    mbar_init(&bar_p, 1);
    mbar_init(&bar_k, 1);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_oq, 1);
    mbar_init(&bar_cc, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_fin, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_s[b], 8);
      mbar_init(&bar_c1[b], 8);
    }
    mbar_init(&bar_oqe, 8);
    mbar_init(&bar_dpe, 8);
    s_abort = 0;
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = s_tmem;
  volatile int* abort_flag = &s_abort;
  auto chunk_c0 = [&](int c) { return seq_s + (int64_t)kC * c; };
  auto slot_of = [&](int c) { return (size_t)(kb + c) * p.Hv + h; };
  auto stage = [&](int c) { return sm + (uint32_t)(c & 1) * ST_BYTES; };

  // the loader's copies in flight, for the exit path
  uint32_t n_st0 = 0, n_st1 = 0, n_p = 0, n_k = 0, n_q = 0;
  const bool loader = warp == 0 && lane == 0;

  if (warp == 0) {
    // ================================================ loads (lane 0)
    if (loader) {
      auto load_stage = [&](int c) {
        uint64_t* bar = &bar_st[c & 1];
        if (c & 1) ++n_st1; else ++n_st0;
        mbar_arrive_expect_tx(bar, ST_BYTES);
        unsigned char* st = stage(c);
        const size_t slot = slot_of(c);
        tc::tma_load_2d(st + ST_U, &tm_u, 0, (int)(slot * kD), bar);
        tc::tma_load_2d(st + ST_U + 16384, &tm_u, 32, (int)(slot * kD), bar);
        tc::tma_load_2d(st + ST_WHI, &tm_wm, 0, (int)(slot * 2 * kC), bar);
        tc::tma_load_2d(st + ST_WHI + 8192, &tm_wm, 64, (int)(slot * 2 * kC), bar);
        tc::tma_load_2d(st + ST_WLO, &tm_wm, 0, (int)(slot * 2 * kC + kC), bar);
        tc::tma_load_2d(st + ST_WLO + 8192, &tm_wm, 64, (int)(slot * 2 * kC + kC), bar);
        bulk_load(st + ST_VEC, w.vec + slot * (4 * kC), 1024u, bar);
      };
      auto load_p = [&](int c) {
        ++n_p;
        mbar_arrive_expect_tx(&bar_p, 8192u);
        tc::tma_load_2d(sm + SO_P, &tm_w, 0, (int)(slot_of(c) * kC), &bar_p);
      };
      auto load_kt = [&](int c) {
        ++n_k;
        mbar_arrive_expect_tx(&bar_k, 16384u);
        tc::tma_load_2d(sm + SO_K, &tm_kt, 0, (int)(((kb + c) * p.Hk + kh) * kD), &bar_k);
      };
      auto load_q = [&](int c) {
        ++n_q;
        mbar_arrive_expect_tx(&bar_q, 16384u);
        const int y = (int)chunk_c0(c);
        tc::tma_load_2d(sm + SO_Q, &tm_q, kh * kD, y, &bar_q);
        tc::tma_load_2d(sm + SO_Q + 8192, &tm_q, kh * kD + 64, y, &bar_q);
      };
      load_stage(0);
      if (nch > 1) load_stage(1);
      load_kt(0);
      load_q(0);
      load_p(0);
      for (int c = 0; c < nch; ++c) {
        const uint32_t ph = (uint32_t)(c & 1);
        const bool more = c + 1 < nch;
        if (!chain_wait(&bar_oq, ph, abort_flag)) break;
        if (more) load_q(c + 1);
        if (!chain_wait(&bar_cc, ph, abort_flag)) break;
        if (more) load_kt(c + 1);
        // stage c is free once its MMAs completed and the output warps have
        // copied its gq; P once (p) completed
        const uint32_t sp = (uint32_t)((c >> 1) & 1);
        if (!chain_wait(&bar_sf[c & 1], sp, abort_flag)) break;
        if (more) load_p(c + 1);
        if (!chain_wait(&bar_gq[c & 1], sp, abort_flag)) break;
        if (c + 2 < nch) load_stage(c + 2);
      }
    }
  } else if (warp == 1) {
    // ================================================ MMA issue (one warp)
    const uint32_t id_a = tc::idesc(tc::kBF16, 128, 64) | tc::kNegB;
    const uint32_t id_o = tc::idesc(tc::kBF16, 128, 64);
    const uint32_t id_c = tc::idesc(tc::kBF16, 128, 128);
    const uint64_t d_q = tc::sdesc_sw128(smem_u32(sm + SO_Q));
    const uint64_t d_kt = tc::sdesc_sw128(smem_u32(sm + SO_K));
    const uint64_t d_dl = tc::sdesc_sw128(smem_u32(sm + SO_DL));
    const uint64_t d_p = tc::sdesc_sw128(smem_u32(sm + SO_P));
    bool ok = true;
    for (int c = 0; c < nch && ok; ++c) {
      const uint32_t ph = (uint32_t)(c & 1), pp = (uint32_t)((c + 1) & 1);
      unsigned char* st = stage(c);
      const uint64_t d_wh = tc::sdesc_sw128(smem_u32(st + ST_WHI));
      const uint64_t d_wl = tc::sdesc_sw128(smem_u32(st + ST_WLO));
      // (a), in two halves as the state copies arrive
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        ok = (q > 0 || chain_wait(&bar_st[c & 1], (uint32_t)((c >> 1) & 1), abort_flag)) &&
             chain_wait(&bar_s[q], ph, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc::fence_after_sync();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int s = 2 * q + (e & 1) + 4 * (e >> 1);
          const uint64_t bh = tc::sdesc_at(d_wh, kC, s), bl = tc::sdesc_at(d_wl, kC, s);
          tc::mma_f16_ts_elect(tb + TS_Y, tb + TS_HI + 8 * s, bh, id_a, s > 0);
          tc::mma_f16_ts_elect(tb + TS_Y, tb + TS_HI + 8 * s, bl, id_a, true);
          tc::mma_f16_ts_elect(tb + TS_Y, tb + TS_LO + 8 * s, bh, id_a, true);
        }
      }
      if (!ok) break;
      tc::mma_commit_elect(&bar_a);
      // (o)
      ok = chain_wait(&bar_q, ph, abort_flag) && (c == 0 || chain_wait(&bar_oqe, pp, abort_flag));
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after_sync();
#pragma unroll
      for (int s = 0; s < 8; ++s)
        tc::mma_f16_ts_elect(tb + TS_OQ, tb + TS_HI + 8 * s, tc::sdesc_at(d_q, kC, s), id_o, s > 0);
      tc::mma_commit_elect(&bar_oq);
      // (c), in two halves as the corrections arrive
      ok = chain_wait(&bar_k, ph, abort_flag);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        ok = ok && chain_wait(&bar_c1[b], ph, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc::fence_after_sync();
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int s = b + 2 * e;
          const uint64_t bk = tc::sdesc_at(d_kt, 128, s);
          tc::mma_f16_ts_elect(tb + TS_S, tb + TS_DH + 8 * s, bk, id_c, true);
          tc::mma_f16_elect(tb + TS_S, tc::sdesc_at(d_dl, 128, s), bk, id_c, true);
        }
      }
      if (!ok) break;
      tc::mma_commit_elect(&bar_cc);
      // (p)
      ok = chain_wait(&bar_p, ph, abort_flag) && (c == 0 || chain_wait(&bar_dpe, pp, abort_flag));
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after_sync();
#pragma unroll
      for (int s = 0; s < 4; ++s)
        tc::mma_f16_ts_elect(tb + TS_DP, tb + TS_DM + 8 * s, tc::sdesc_at(d_p, kC, s), id_o, s > 0);
      tc::mma_commit_elect(&bar_dp);
      tc::mma_commit_elect(&bar_sf[c & 1]);
    }
  } else if (warp < 10) {
    // ============================ state warps: thread (j, hf) owns value row j
    // (TMEM lane j), state columns i in [64 hf, 64 hf + 64) and tokens t in
    // [32 hf, 32 hf + 32) of the per-chunk corrections
    const int q4 = warp & 3, hf = (warp - 2) >> 2;
    const int j = 32 * q4 + lane;
    const uint32_t tl = tb + ((uint32_t)(32 * q4) << 16);
    float* gS = p.state + (((size_t)n * p.Hv + h) * kD + j) * kD + 64 * hf;

    // the state -> its hi/lo copies and the accumulator rescaled by `gl`
    // (or, after the last chunk, the state to memory); 32 columns at a time,
    // every TMEM load of a batch issued before one wait
    auto pass_state = [&](bool from_memory, bool last, float gl) {
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        float v[32];
        if (from_memory) {
          const float4* src = reinterpret_cast<const float4*>(gS + 32 * qq);
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const float4 f = src[m];
            v[4 * m] = f.x;
            v[4 * m + 1] = f.y;
            v[4 * m + 2] = f.z;
            v[4 * m + 3] = f.w;
          }
        } else {
          tc::tmem_ld16(tl + TS_S + 64 * hf + 32 * qq, *reinterpret_cast<float(*)[16]>(v));
          tc::tmem_ld16(tl + TS_S + 64 * hf + 32 * qq + 16, *reinterpret_cast<float(*)[16]>(v + 16));
          tc::tmem_wait_ld();
        }
        if (last) {
          float4* dst = reinterpret_cast<float4*>(gS + 32 * qq);
#pragma unroll
          for (int m = 0; m < 8; ++m) dst[m] = make_float4(v[4 * m], v[4 * m + 1], v[4 * m + 2], v[4 * m + 3]);
          continue;
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const float a0 = v[16 * hh + 2 * m], a1 = v[16 * hh + 2 * m + 1];
            const __nv_bfloat162 hv = __floats2bfloat162_rn(a0, a1);
            hw[m] = *reinterpret_cast<const uint32_t*>(&hv);
            lw[m] = pack_bf16(a0 - __low2float(hv), a1 - __high2float(hv));
          }
          tc::tmem_st8u(tl + TS_HI + 32 * hf + 16 * qq + 8 * hh, hw);
          tc::tmem_st8u(tl + TS_LO + 32 * hf + 16 * qq + 8 * hh, lw);
        }
#pragma unroll
        for (int m = 0; m < 32; ++m) v[m] *= gl;
        warp_done(&bar_s[qq], lane);
        tc::tmem_st16(tl + TS_S + 64 * hf + 32 * qq, *reinterpret_cast<const float(*)[16]>(v));
        tc::tmem_st16(tl + TS_S + 64 * hf + 32 * qq + 16, *reinterpret_cast<const float(*)[16]>(v + 16));
      }
    };

    bool to = !chain_wait(&bar_st[0], 0, abort_flag);
    to = __any_sync(0xffffffffu, to);
    if (!to) pass_state(true, false, reinterpret_cast<const float*>(sm + ST_VEC)[3 * kC]);

    for (int c = 0; c < nch && !to; ++c) {
      const uint32_t ph = (uint32_t)(c & 1);
      const bool more = c + 1 < nch;
      const float* vec = reinterpret_cast<const float*>(stage(c) + ST_VEC);
      // conv1: Dm^T = U^T + Y; (dk Dm)^T hi -> TMEM, lo -> shared memory;
      // Dm^T hi -> TMEM
      to = !chain_wait(&bar_st[c & 1], (uint32_t)((c >> 1) & 1), abort_flag) ||
           !chain_wait(&bar_a, ph, abort_flag);
      if (__any_sync(0xffffffffu, to)) break;
      tc::fence_after_sync();
#pragma unroll
      for (int bt = 0; bt < 2; ++bt) {
        const int t0 = 32 * hf + 16 * bt;
        float y[16], dk[16];
        tc::tmem_ld16(tl + TS_Y + t0, y);
        const unsigned char* ur = stage(c) + ST_U + hf * 16384 + (j >> 3) * 1024 + (j & 7) * 128;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 d4 = reinterpret_cast<const float4*>(vec + kC + t0)[m];
          dk[4 * m] = d4.x;
          dk[4 * m + 1] = d4.y;
          dk[4 * m + 2] = d4.z;
          dk[4 * m + 3] = d4.w;
        }
        float uv[16];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 u4 = *reinterpret_cast<const float4*>(ur + (((4 * bt + m) ^ (j & 7)) << 4));
          uv[4 * m] = u4.x;
          uv[4 * m + 1] = u4.y;
          uv[4 * m + 2] = u4.z;
          uv[4 * m + 3] = u4.w;
        }
        tc::tmem_wait_ld();
#pragma unroll
        for (int m = 0; m < 16; ++m) y[m] += uv[m];
        uint32_t dh[8], dm[8], dl[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const float x0 = y[2 * m] * dk[2 * m], x1 = y[2 * m + 1] * dk[2 * m + 1];
          const __nv_bfloat162 hv = __floats2bfloat162_rn(x0, x1);
          dh[m] = *reinterpret_cast<const uint32_t*>(&hv);
          dl[m] = pack_bf16(x0 - __low2float(hv), x1 - __high2float(hv));
          dm[m] = pack_bf16(y[2 * m], y[2 * m + 1]);
        }
        tc::tmem_st8u(tl + TS_DH + t0 / 2, dh);
        tc::tmem_st8u(tl + TS_DM + t0 / 2, dm);
        *reinterpret_cast<uint4*>(sm + SO_DL + sw_chunk(j, t0 / 8, 128)) = make_uint4(dl[0], dl[1], dl[2], dl[3]);
        *reinterpret_cast<uint4*>(sm + SO_DL + sw_chunk(j, t0 / 8 + 1, 128)) = make_uint4(dl[4], dl[5], dl[6], dl[7]);
        warp_done(&bar_c1[bt], lane);
      }
      // conv2: the new state; the next chunk's G_{L-1} from its stage
      to = (more && !chain_wait(&bar_st[(c + 1) & 1], (uint32_t)(((c + 1) >> 1) & 1), abort_flag)) ||
           !chain_wait(&bar_cc, ph, abort_flag);
      if (__any_sync(0xffffffffu, to)) break;
      tc::fence_after_sync();
      pass_state(false, !more, more ? reinterpret_cast<const float*>(stage(c + 1) + ST_VEC)[3 * kC] : 1.f);
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
  } else {
    // ============================ output warps: thread (j, hf) owns output
    // column j = 32 (warp % 4) + lane for the 32 tokens t0 = 32 hf ... With
    // the fused norm, the per-token sums of squares are reduce-scattered
    // across lanes, z arrives by TMA into a row-major tile (two, by chunk
    // parity) that the gated result overwrites in place, and a full chunk
    // leaves as one 2-D TMA store.
    const int u = tid - 320, q4 = warp & 3, hf = (warp - 10) >> 2;
    const int j = 32 * q4 + lane, t0 = 32 * hf;
    const uint32_t tl = tb + ((uint32_t)(32 * q4) << 16);
    const float nwj = fused ? p.norm_w[j] : 0.f;
    uint32_t n_z0 = 0, n_z1 = 0;
    bool stored = false;
    auto load_z = [&](int c) {
      if (c & 1) ++n_z1; else ++n_z0;
      mbar_arrive_expect_tx(&bar_z[c & 1], 16384u);
      tc::tma_load_2d(sm + SO_Z + (c & 1) * 16384, &tm_z, h * kD, (int)chunk_c0(c), &bar_z[c & 1]);
    };
    if (fused && u == 0) {
      load_z(0);
      if (nch > 1) load_z(1);
    }
    bool to = false;  // a bounded wait gave up (agreed on at the next barrier)
    for (int c = 0; c < nch; ++c) {
      const int64_t c0 = chunk_c0(c);
      const int L = (int)((seq_e - c0) < kC ? (seq_e - c0) : kC);
      const float* vec = reinterpret_cast<const float*>(stage(c) + ST_VEC);
      __nv_bfloat16* zb = reinterpret_cast<__nv_bfloat16*>(sm + SO_Z + (c & 1) * 16384);
      float a[2][16], b[2][16];
      to |= !chain_wait(&bar_st[c & 1], (uint32_t)((c >> 1) & 1), abort_flag) ||
            !chain_wait(&bar_oq, (uint32_t)(c & 1), abort_flag);
      if (bar_or(2, kOutThreads, to)) break;
      tc::fence_after_sync();
#pragma unroll
      for (int m = 0; m < 2; ++m) tc::tmem_ld16(tl + TS_OQ + t0 + 16 * m, a[m]);
      tc::tmem_wait_ld();
      if (u < kC) sgq[c & 1][u] = vec[2 * kC + u];
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_oqe);       // OQ(c) read
        mbar_arrive(&bar_gq[c & 1]);  // and gq(c) copied: stage c may be reloaded
      }
      to |= !chain_wait(&bar_dp, (uint32_t)(c & 1), abort_flag);
      if (bar_or(2, kOutThreads, to)) break;
      tc::fence_after_sync();
#pragma unroll
      for (int m = 0; m < 2; ++m) tc::tmem_ld16(tl + TS_DP + t0 + 16 * m, b[m]);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_dpe);
      const float* gq = sgq[c & 1] + t0;
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
      for (int stp = 1; stp < 5; ++stp) {
        const int m = 16 >> stp, hv = 16 >> stp;
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
      // z of chunk c+1 into the tile chunk c-1 was stored from. Only a
      // sequence's last chunk can be partial, so chunk c-1 was full and left
      // as thread 0's one tile store: its own wait covers the reload.
      if (u == 0 && c >= 1 && c + 1 < nch) {
        bulk_wait_read_all();
        load_z(c + 1);
      }
      to |= !chain_wait(&bar_z[c & 1], (uint32_t)((c >> 1) & 1), abort_flag);
      bar_named(2, kOutThreads);
      // the gated result over z, in place (rows >= L hold finite values that
      // are never stored), 16 rows at a time: all loads, then the math, then
      // all stores
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float zf[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) zf[e] = __bfloat162float(zb[(t0 + 16 * hh + e) * kD + j]);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int t = t0 + 16 * hh + e;
          const float gate = __fdividef(zf[e], 1.f + __expf(-zf[e]));
          zf[e] = o[16 * hh + e] * sinv[t] * nwj * gate;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) zb[(t0 + 16 * hh + e) * kD + j] = __float2bfloat16_rn(zf[e]);
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
  if (warp == 1) {
    tc::fence_after_sync();
    tc::mma_commit_elect(&bar_fin);
    mbar_wait(&bar_fin, 0);
    tc::fence_before_sync();
  }
  if (loader) {
    if (n_st0) mbar_wait(&bar_st[0], (n_st0 - 1) & 1);
    if (n_st1) mbar_wait(&bar_st[1], (n_st1 - 1) & 1);
    if (n_p) mbar_wait(&bar_p, (n_p - 1) & 1);
    if (n_k) mbar_wait(&bar_k, (n_k - 1) & 1);
    if (n_q) mbar_wait(&bar_q, (n_q - 1) & 1);
  }
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tb, 512);
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
  if ((double)l.G * p.Hv * kD >= 2147483647.0) return false;
  if ((double)l.G * p.Hv * 2 * kC >= 2147483647.0) return false;
  if ((double)l.G * p.Hk * kD >= 2147483647.0) return false;
  return tc::encode_fn() != nullptr;
}

cudaError_t launch_prefill_cp(const PrefillArgs& p, void* workspace, cudaStream_t stream) {
  if (p.N == 0 || p.T == 0) return cudaSuccess;
  const CpLayout l = cp_layout(p.N, p.T, p.Hk, p.Hv);
  CpWork w{};
  w.cs = static_cast<int32_t*>(workspace);
  w.tw = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) + l.off_tm);
  w.u = reinterpret_cast<float*>(static_cast<char*>(workspace) + l.off_u);
  w.wm = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) + l.off_wm);
  w.kt = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) + l.off_kt);
  w.vec = reinterpret_cast<float*>(static_cast<char*>(workspace) + l.off_vec);
  w.G = l.G;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap mq, mk, mv, mw, mu, mwm, mkt, mz, mo;
  memset(&mz, 0, sizeof(mz));
  memset(&mo, 0, sizeof(mo));
  const int64_t qkc = (int64_t)p.Hk * kD, vc = (int64_t)p.Hv * kD;
  if (!tc::make_map_2d(&mq, p.q, p.T, qkc, p.q_stride, 2, bf, 64, 64, sw) ||
      !tc::make_map_2d(&mk, p.k, p.T, qkc, p.k_stride, 2, bf, 64, 64, sw) ||
      !tc::make_map_2d(&mv, p.v, p.T, vc, p.v_stride, 2, bf, 64, 64, sw) ||
      !tc::make_map_2d(&mw, w.tw, l.G * p.Hv * kC, kC, kC, 2, bf, 64, 64, sw) ||
      !tc::make_map_2d(&mu, w.u, l.G * p.Hv * kD, kC, kC, 4, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, 128,
                       sw) ||
      !tc::make_map_2d(&mwm, w.wm, l.G * p.Hv * 2 * kC, kD, kD, 2, bf, 64, 64, sw) ||
      !tc::make_map_2d(&mkt, w.kt, l.G * p.Hk * kD, kC, kC, 2, bf, 64, 128, sw))
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
  cp_prep_kernel<<<dim3((unsigned)l.G, (unsigned)p.Hk), kPrepThreads, P_SMEM, stream>>>(p, w, mq, mk, mv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(cp_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S_SMEM);
  if (e != cudaSuccess) return e;
  cp_scan_kernel<<<dim3((unsigned)p.Hv, (unsigned)p.N), kScanThreads, S_SMEM, stream>>>(p, w, mq, mk, mu, mw,
                                                                                        mwm, mkt, mz, mo);
  return cudaGetLastError();
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(prefill_cp)
