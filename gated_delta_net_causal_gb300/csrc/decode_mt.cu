// Multi-token decode: T (1..8) consecutive tokens of every sequence in one
// launch, each state read from and written to HBM once for the T tokens
// instead of once per token (the "resident state" case of a decode step:
// speculative or multi-token-prediction decode verifies several tokens of a
// sequence at a time). Per token and value row j of V head h the step is the
// one gdn_decode_step takes (ferrox-core gdn.rs, `delta_step`):
//   S_j *= a_t;  p = S_j . k_t;  d = b_t (v_tj - p);  S_j += d k_t;
//   o_tj = S_j . q_t / sqrt(D),
// applied token after token to the row while it sits in registers. Every
// token's arithmetic is written in the same order as in the one-token kernel
// (decode.cu: the conv sum, the norms, the gates, both dot products from the
// old row, the fused update and read-out), so a T-token call gives the same
// bits as T successive gdn_decode_step calls.
//
// Structure (as in decode.cu): a persistent kernel, a work item is one
// (sequence, K head) pair with its V heads. Two CTAs share each SM where
// their shared memory fits (up to four V heads per K head), so one CTA's
// per-item prologue and outputs overlap the other's state stream. One
// producer warp streams the item's state rows through a shared-memory ring
// with 1-D bulk copies, eight consumer warps update the rows. Per item the
// consumer warps (1) run the conv over the item's q, k and v channels for
// all T tokens from the old conv state (and write the new one: this CTA
// alone owns those channels), and the gates; barrier; (2) each warp takes
// the l2 norms of every token's q and k; (3) the state pass, T tokens per
// row; barrier; (4) the outputs of every (head, token) pair, one warp per
// pair. The per-item buffers are single: barrier (1)->(2) of the next item
// orders them. With 16-bit activations, where shared memory allows, the
// item's conv inputs (old conv state, the T tokens' inputs) arrive by
// asynchronous copies into a staging area during the previous item's state
// pass, and its z rows during its own, so neither (1) nor (4) waits on
// global memory.
//
// Every wait is bounded; a wait that gives up records GDN_ERR_TIMEOUT and
// raises a CTA-wide abort flag, after which no warp waits again.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kMtCW = 8;                      // consumer warps
constexpr int kMtThreads = 32 * (kMtCW + 1);  // + one producer warp
constexpr int kMtTMax = 8;                    // tokens per sequence and call
constexpr int kMtRPL = 2;                     // rows each lane updates per pass
constexpr int kMtMaxStages = 16;

// The lane geometry of the one-token decode kernel (decode.cu): LPR lanes
// per row, NV4 groups of four columns per lane (16 columns at D = 32, 64,
// 128; eight lanes of 12 at D = 96, three rows per lane so that a chunk is a
// whole 96-row head).
template <typename T, int D, int REPMAX>
struct MtGeom {
  static constexpr int LPR = D == 96 ? 8 : D / 16;  // lanes per row
  static constexpr int NV4 = D / (4 * LPR);
  static constexpr int RPL = D == 96 ? 3 : kMtRPL;
  static constexpr int RPW = 32 / LPR;
  static constexpr int WROWS = RPW * RPL;
  static constexpr int CHUNK_ROWS = WROWS * kMtCW < D ? WROWS * kMtCW : D;
  static constexpr int CPH = D / CHUNK_ROWS;
  static constexpr uint32_t SLOT_BYTES = CHUNK_ROWS * D * 4;
  static constexpr int SLOT_FLOATS = CHUNK_ROWS * D;
  // static shared memory: q, k [T][D], v and the outputs [REPMAX][T][D], plus
  // gates, norm weight, per-warp norms and barriers (under 4 KB)
  static constexpr int STATIC_BYTES = (2 + 2 * REPMAX) * kMtTMax * D * 4 + 4096;
  // two CTAs per SM (112 KB each) while that leaves a ring of two 32 KB slots
  static constexpr int CTAS_PER_SM = REPMAX <= 4 ? 2 : 1;
  static constexpr int RING_AVAIL = (CTAS_PER_SM == 2 ? 112 : 227) * 1024 - STATIC_BYTES;
  static constexpr int stages_in(int bytes) {
    return (bytes < 192 * 1024 ? bytes : 192 * 1024) / (int)SLOT_BYTES < kMtMaxStages
               ? (bytes < 192 * 1024 ? bytes : 192 * 1024) / (int)SLOT_BYTES
               : kMtMaxStages;
  }
  // Staging area (behind the ring) for the global inputs of an item's
  // prologue and outputs: the conv state and the T tokens' inputs of its
  // NCH channels, and its z rows. Used with 16-bit activations where it
  // leaves the ring at least min(its plain depth, 4) stages.
  static constexpr int NCH = (2 + REPMAX) * D;
  static constexpr int STG_X = kMtTMax * NCH;            // elements: [T][NCH]
  static constexpr int STG_CS = 3 * NCH;                 // [NCH][3]
  static constexpr int STG_Z = REPMAX * kMtTMax * D;     // [REPMAX][T][D]
  static constexpr int STG_BYTES = (STG_X + STG_CS + STG_Z) * (int)sizeof(T);
  static constexpr int STAGES_PLAIN = stages_in(RING_AVAIL);
  static constexpr int STAGES_STG = stages_in(RING_AVAIL - STG_BYTES);
  static constexpr bool STAGED =
      sizeof(T) == 2 && STAGES_STG >= (STAGES_PLAIN < 4 ? STAGES_PLAIN : 4);
  static constexpr int STAGES = STAGED ? STAGES_STG : STAGES_PLAIN;
  static constexpr int RING_BYTES = STAGES * (int)SLOT_BYTES;
  static constexpr int DYN_BYTES = RING_BYTES + (STAGED ? STG_BYTES : 0);
  static_assert(STAGES >= 2, "ring too small");
  static_assert((D * sizeof(T)) % 16 == 0 && RING_BYTES % 16 == 0 && (STG_X * sizeof(T)) % 16 == 0 &&
                    (STG_CS * sizeof(T)) % 16 == 0,
                "16-byte copy granules");
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ bool mt_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait_bounded(bar, parity, abort_flag);
}

__device__ __forceinline__ void mt_consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kMtCW * 32) : "memory");
}

template <typename T, int D, int REPMAX>
__global__ void __launch_bounds__(kMtThreads, MtGeom<T, D, REPMAX>::CTAS_PER_SM)
    decode_multi_kernel(const DecodeArgs p, const int num_items) {
  using G = MtGeom<T, D, REPMAX>;
  constexpr int LPR = G::LPR, RPW = G::RPW, STAGES = G::STAGES, NV4 = G::NV4, RPL = G::RPL;
  constexpr int NC = kMtCW * 32;
  constexpr int PER = D / 32;  // output elements per lane
  static_assert(REPMAX * kMtTMax <= NC, "one (head, token) gate per consumer thread");

  extern __shared__ __align__(128) float ring[];
  __shared__ float sq[kMtTMax][D], sk[kMtTMax][D];
  __shared__ float sv[REPMAX][kMtTMax][D], so[REPMAX][kMtTMax][D];
  __shared__ float sgate[REPMAX][kMtTMax][2];
  __shared__ float skq[kMtTMax];  // per token: k.q of the normalised vectors, scaled
  __shared__ float snw[D];
  __shared__ __align__(8) uint64_t full_bar[kMtMaxStages], empty_bar[kMtMaxStages];
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rep = p.rep, Hk = p.Hk, Hv = p.Hv, NT = p.tokens;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kMtCW);
    }
    s_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;

  if (warp == kMtCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t k = 0;
      for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
        const int b = item / Hk, kh = item - (item / Hk) * Hk;
        for (int r = 0; r < rep; ++r) {
          const int h = p.map == GDN_MAP_TILED ? kh + r * Hk : kh * rep + r;
          const float* gS = p.state + ((size_t)b * Hv + h) * (size_t)(D * D);
          for (int c = 0; c < G::CPH; ++c, ++k) {
            const int slot = (int)(k % STAGES);
            if (k >= (uint32_t)STAGES &&
                !mt_wait(&empty_bar[slot], ((k / STAGES) - 1) & 1, abort_flag))
              return;
            mbar_arrive_expect_tx(&full_bar[slot], G::SLOT_BYTES);
            bulk_load(ring + slot * G::SLOT_FLOATS, gS + (size_t)c * G::SLOT_FLOATS,
                      G::SLOT_BYTES, &full_bar[slot]);
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const size_t C = (size_t)p.C;
  const int qk_f = Hk * D;
  const T* w = static_cast<const T*>(p.conv_w);
  const int sub = lane % LPR, rq = lane / LPR;
  if (p.z != nullptr)
    for (int j = tid; j < D; j += NC) snw[j] = p.norm_w[j];

  // first global channel of channel group g (q, k, then V head g - 2) of K head kh
  auto group_base = [&](int g, int kh) -> int {
    if (g < 2) return g * qk_f + kh * D;
    const int h = p.map == GDN_MAP_TILED ? kh + (g - 2) * Hk : kh * rep + (g - 2);
    return 2 * qk_f + h * D;
  };
  // The staging area (16-bit activations): [T][NCH] inputs and [NCH][3] conv
  // state of the item's channels, [REPMAX][T][D] z. An item's conv inputs are
  // copied in while the previous item streams its state, its z rows while
  // its own state streams: every copy is issued after an item's first
  // barrier and waited for before its third, so the barriers order them.
  T* const stg_x = reinterpret_cast<T*>(reinterpret_cast<char*>(ring) + G::RING_BYTES);
  T* const stg_cs = stg_x + G::STG_X;
  T* const stg_z = stg_cs + G::STG_CS;
  constexpr int GR = D * (int)sizeof(T) / 16;  // 16-byte granules of D elements
  auto stage_conv = [&](int it) {
    if (it >= num_items) return;
    const int b = it / Hk, kh = it - (it / Hk) * Hk;
    const char* xsrc = static_cast<const char*>(p.mixed_qkv) + (size_t)b * NT * C * sizeof(T);
    const char* csrc = static_cast<const char*>(p.conv_state) + (size_t)b * C * 3 * sizeof(T);
    const int ng = 2 + rep, n_cs = ng * 3 * GR, n_all = n_cs + NT * ng * GR;
    for (int q = tid; q < n_all; q += NC) {
      if (q < n_cs) {
        const int g = q / (3 * GR), o = q - g * (3 * GR);
        cp_async16(reinterpret_cast<char*>(stg_cs + g * 3 * D) + o * 16,
                   csrc + (size_t)group_base(g, kh) * 3 * sizeof(T) + o * 16);
      } else {
        const int j = q - n_cs, t = j / (ng * GR), rr = j - t * (ng * GR);
        const int g = rr / GR, o = rr - g * GR;
        cp_async16(reinterpret_cast<char*>(stg_x + t * G::NCH + g * D) + o * 16,
                   xsrc + ((size_t)t * C + group_base(g, kh)) * sizeof(T) + o * 16);
      }
    }
  };
  auto stage_z = [&](int it) {
    if (p.z == nullptr) return;
    const int b = it / Hk, kh = it - (it / Hk) * Hk;
    for (int q = tid; q < rep * NT * GR; q += NC) {
      const int pr = q / GR, o = q - pr * GR, r = pr / NT, t = pr - r * NT;
      const int h = p.map == GDN_MAP_TILED ? kh + r * Hk : kh * rep + r;
      cp_async16(reinterpret_cast<char*>(stg_z + (r * kMtTMax + t) * D) + o * 16,
                 static_cast<const char*>(p.z) + (((size_t)b * NT + t) * Hv + h) * D * sizeof(T) +
                     o * 16);
    }
  };
  if constexpr (G::STAGED) {
    stage_conv(blockIdx.x);
    cp_async_commit();
    cp_async_wait_all();
    mt_consumer_sync();
  }

  uint32_t k = 0;
  for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
    const int b = item / Hk, kh = item - (item / Hk) * Hk;
    const T* xb = static_cast<const T*>(p.mixed_qkv) + (size_t)b * NT * C;
    T* cst = static_cast<T*>(p.conv_state) + (size_t)b * C * 3;

    // (1) conv + SiLU of the item's channels [q of kh | k of kh | v of each
    // head] for every token, rolling the 3-wide window through the tokens,
    // then the gates (their inputs loaded first, so they arrive during the
    // conv)
    float ga = 0.f, gb = 0.f, gp = 0.f, gd = 0.f;
    const int gr = tid / NT, gt = tid - (tid / NT) * NT;  // this thread's (head, token) gate
    const bool has_gate = tid < rep * NT;
    if (has_gate) {
      const int h = p.map == GDN_MAP_TILED ? kh + gr * Hk : kh * rep + gr;
      const size_t gi = ((size_t)b * NT + gt) * Hv + h;
      ga = to_f32(static_cast<const T*>(p.a)[gi]);
      gb = to_f32(static_cast<const T*>(p.b)[gi]);
      gp = p.decay_param[h];
      gd = p.dt_bias[h];
    }
    const int nch = (2 + rep) * D;
    for (int idx = tid; idx < nch; idx += NC) {
      const int which = idx / D, i = idx - which * D;
      const int c = group_base(which, kh) + i;
      float* dst = which == 0 ? &sq[0][i] : which == 1 ? &sk[0][i] : &sv[which - 2][0][i];
      T* cp = cst + (size_t)c * 3;
      T a0, a1, a2;
      T xv[kMtTMax];
      if constexpr (G::STAGED) {
        a0 = stg_cs[idx * 3 + 0];
        a1 = stg_cs[idx * 3 + 1];
        a2 = stg_cs[idx * 3 + 2];
#pragma unroll
        for (int t = 0; t < kMtTMax; ++t) xv[t] = t < NT ? stg_x[t * G::NCH + idx] : T();
      } else {
        a0 = cp[0];
        a1 = cp[1];
        a2 = cp[2];
#pragma unroll
        for (int t = 0; t < kMtTMax; ++t) xv[t] = t < NT ? xb[(size_t)t * C + c] : T();
      }
      const float w0 = to_f32(w[(size_t)c * 4 + 0]), w1 = to_f32(w[(size_t)c * 4 + 1]);
      const float w2 = to_f32(w[(size_t)c * 4 + 2]), w3 = to_f32(w[(size_t)c * 4 + 3]);
#pragma unroll
      for (int t = 0; t < kMtTMax; ++t) {
        if (t < NT) {
          float acc = w0 * to_f32(a0);
          acc += w1 * to_f32(a1);
          acc += w2 * to_f32(a2);
          acc += w3 * to_f32(xv[t]);
          dst[t * D] = silu_f(acc);
          a0 = a1;
          a1 = a2;
          a2 = xv[t];
        }
      }
      if (!*abort_flag) {
        cp[0] = a0;
        cp[1] = a1;
        cp[2] = a2;
      }
    }
    if (has_gate) {
      sgate[gr][gt][0] = expf(gate_g(p.decay, gp, gd, ga));
      sgate[gr][gt][1] = sigmoid_f(gb);
    }
    mt_consumer_sync();
    if constexpr (G::STAGED) {
      stage_conv(item + gridDim.x);
      stage_z(item);
      cp_async_commit();
    }

    // (2) warp t: the l2 norms of token t's q and k and their product, then
    // k normalised and q normalised and scaled, in place (the one-token
    // kernel's arithmetic, token by token)
    if (warp < NT) {
      const int t = warp;
      float qq = 0.f, kk = 0.f, qkr = 0.f;
#pragma unroll
      for (int i = lane; i < D; i += 32) {
        const float qv = sq[t][i], kv = sk[t][i];
        qq = fmaf(qv, qv, qq);
        kk = fmaf(kv, kv, kk);
        qkr = fmaf(qv, kv, qkr);
      }
      qq = group_sum<32>(qq);
      kk = group_sum<32>(kk);
      qkr = group_sum<32>(qkr);
      const float inv_q = 1.f / sqrtf(qq + p.l2_eps);
      const float inv_k = 1.f / sqrtf(kk + p.l2_eps);
      const float sqs = inv_q * p.scale;
      if (lane == 0) skq[t] = qkr * inv_q * inv_k * p.scale;
#pragma unroll
      for (int i = lane; i < D; i += 32) {
        sk[t][i] *= inv_k;
        sq[t][i] *= sqs;
      }
    }
    mt_consumer_sync();

    // (3) the state pass: each row read once from the ring, T token steps in
    // registers, written back once
    for (int r = 0; r < rep; ++r) {
      const int h = p.map == GDN_MAP_TILED ? kh + r * Hk : kh * rep + r;
      float* gS = p.state + ((size_t)b * Hv + h) * (size_t)(D * D);
      for (int c = 0; c < G::CPH; ++c, ++k) {
        const int slot = (int)(k % STAGES);
        const bool ready = mt_wait(&full_bar[slot], (k / STAGES) & 1, abort_flag);
        if (ready && warp * G::WROWS < G::CHUNK_ROWS) {
          float4 s4[RPL][NV4];
          int rowv[RPL];
#pragma unroll
          for (int u = 0; u < RPL; ++u) {
            const int rl = warp * G::WROWS + u * RPW + rq;
            rowv[u] = c * G::CHUNK_ROWS + rl;
            const float* srow = ring + slot * G::SLOT_FLOATS + rl * D;
#pragma unroll
            for (int m = 0; m < NV4; ++m)
              s4[u][m] = *reinterpret_cast<const float4*>(srow + 4 * sub + 4 * LPR * m);
          }
          for (int t = 0; t < NT; ++t) {
            const float kq = skq[t];
            float4 kr[NV4], qr[NV4];
#pragma unroll
            for (int m = 0; m < NV4; ++m) {
              const int col = 4 * sub + 4 * LPR * m;
              kr[m] = *reinterpret_cast<const float4*>(&sk[t][col]);
              qr[m] = *reinterpret_cast<const float4*>(&sq[t][col]);
            }
            float pk[RPL], pq[RPL];
#pragma unroll
            for (int u = 0; u < RPL; ++u) {
              pk[u] = row_dot<NV4>(s4[u], kr);
              pq[u] = row_dot<NV4>(s4[u], qr);
            }
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) {
#pragma unroll
              for (int u = 0; u < RPL; ++u) {
                pk[u] += __shfl_xor_sync(0xffffffffu, pk[u], o);
                pq[u] += __shfl_xor_sync(0xffffffffu, pq[u], o);
              }
            }
            const float alpha = sgate[r][t][0], beta = sgate[r][t][1];
#pragma unroll
            for (int u = 0; u < RPL; ++u) {
              const int row = rowv[u];
              const float d = beta * (sv[r][t][row] - alpha * pk[u]);
              const float o = fmaf(alpha, pq[u], d * kq);
              row_update<NV4>(s4[u], kr, alpha, d);
              if (sub == 0) so[r][t][row] = o;
            }
          }
#pragma unroll
          for (int u = 0; u < RPL; ++u) {
            float* grow = gS + (size_t)rowv[u] * D;
#pragma unroll
            for (int m = 0; m < NV4; ++m)
              __stcs(reinterpret_cast<float4*>(grow + 4 * sub + 4 * LPR * m), s4[u][m]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
      }
    }
    if constexpr (G::STAGED) cp_async_wait_all();  // the next item's inputs, this item's z
    mt_consumer_sync();

    // (4) outputs: one warp per (head, token) pair
    if (!*abort_flag) {
      for (int pr = warp; pr < rep * NT; pr += kMtCW) {
        const int r = pr / NT, t = pr - (pr / NT) * NT;
        const int h = p.map == GDN_MAP_TILED ? kh + r * Hk : kh * rep + r;
        const size_t obase = (((size_t)b * NT + t) * Hv + h) * D + lane * PER;
        float ov[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) ov[e] = so[r][t][lane * PER + e];
        if (p.core_out != nullptr) {
#pragma unroll
          for (int e = 0; e < PER; ++e) p.core_out[obase + e] = ov[e];
        }
        if (p.z != nullptr) {
          float ss = 0.f;
#pragma unroll
          for (int e = 0; e < PER; ++e) ss += ov[e] * ov[e];
          ss = group_sum<32>(ss);
          const float inv = 1.f / sqrtf(ss / (float)D + p.rms_eps);
          const T* zr = G::STAGED ? stg_z + (r * kMtTMax + t) * D + lane * PER
                                  : static_cast<const T*>(p.z) + obase;
          T* outr = static_cast<T*>(p.out) + obase;
#pragma unroll
          for (int e = 0; e < PER; ++e)
            outr[e] = from_f32<T>(ov[e] * inv * snw[lane * PER + e] * silu_f(to_f32(zr[e])));
        }
      }
    }
  }
}

int mt_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

template <typename T, int D, int REPMAX>
cudaError_t launch_mt_t(const DecodeArgs& p, int32_t batch, cudaStream_t stream) {
  auto kern = decode_multi_kernel<T, D, REPMAX>;
  const int smem = MtGeom<T, D, REPMAX>::DYN_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // resident CTAs per SM as the runtime computes them, asked once per variant
  // (after the shared-memory attribute above; initialised thread-safely)
  static const int per_sm = [&] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kMtThreads, smem) != cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
    return n > 0 ? n : 1;
  }();
  const int items = batch * p.Hk;
  const int slots = mt_sm_count() * per_sm;
  const int grid = items < slots ? items : slots;
  kern<<<grid, kMtThreads, smem, stream>>>(p, items);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_mt_r(const DecodeArgs& p, int32_t batch, cudaStream_t stream) {
  if (p.rep <= 2) return launch_mt_t<T, D, 2>(p, batch, stream);
  if (p.rep <= 4) return launch_mt_t<T, D, 4>(p, batch, stream);
  return launch_mt_t<T, D, 8>(p, batch, stream);
}

template <typename T>
cudaError_t launch_mt_d(const DecodeArgs& p, int32_t D, int32_t batch, cudaStream_t stream) {
  switch (D) {
    case 32: return launch_mt_r<T, 32>(p, batch, stream);
    case 64: return launch_mt_r<T, 64>(p, batch, stream);
    case 96: return launch_mt_r<T, 96>(p, batch, stream);
    case 128: return launch_mt_r<T, 128>(p, batch, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_multi(const DecodeArgs& p, int32_t dtype, int32_t D, int32_t batch,
                                cudaStream_t stream) {
  if (p.tokens < 1 || p.tokens > kMtTMax) return cudaErrorInvalidValue;
  switch (dtype) {
    case GDN_F16: return launch_mt_d<__half>(p, D, batch, stream);
    case GDN_BF16: return launch_mt_d<__nv_bfloat16>(p, D, batch, stream);
    case GDN_F32: return launch_mt_d<float>(p, D, batch, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(decode_mt)
