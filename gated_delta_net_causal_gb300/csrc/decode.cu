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
// Structure: a persistent kernel, one CTA per SM. A work item is one
// (sequence, K head) pair with all Hv/Hk V heads that read that K head, so
// the CTA that reads a K head's old q/k conv state is also the only one that
// writes the new one (no cross-CTA ordering). Items go to CTAs round-robin.
//
// Inside a CTA, one producer warp streams the state rows of its items, in
// order, through a ring of shared-memory slots with 1-D bulk copies (each
// slot has a "full" mbarrier completed by the copy's byte count and an
// "empty" mbarrier the consumer warps arrive on). The ring spans item
// boundaries, so while the consumer warps compute the next item's conv,
// norms and gates, its state is already streaming in. The eight consumer
// warps update rows in registers (a quarter-warp per 512-byte row) and write
// them back to global memory with coalesced 16-byte stores. Per item there
// is one barrier among the consumer warps (the item's q, k, v and gates are
// in shared memory); each warp takes the l2 norms itself, and an item's
// outputs are written after the next item's barrier, by when every warp has
// finished its state pass, so they overlap the next item's stream.
//
// With a state-slot table, batch row b works on state[slots[b]] and
// conv_state[slots[b]] of a larger pool (every other tensor is still indexed
// by b). The producer and the consumers look the slot up themselves and skip
// a padded row (negative slot) or an out-of-range one alike, so their ring
// positions stay in step; such a row touches neither state and gets zero
// core outputs.
//
// Every wait is bounded; a wait that gives up records GDN_ERR_TIMEOUT and
// raises a CTA-wide abort flag, after which no warp waits again, so the
// kernel always runs to its end.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {

constexpr int kDecCW = 8;                      // consumer warps
constexpr int kDecThreads = 32 * (kDecCW + 1);  // + one producer warp
constexpr int kDecMaxStages = 16;              // ring slots (upper bound)
// shared-memory ring: 192 KB, or 160 KB where the per-item buffers for 16 V
// heads per K head (about 35 KB of static shared memory) take the rest
constexpr int dec_ring_bytes(int repmax) { return repmax > 8 ? 160 * 1024 : 192 * 1024; }
constexpr int kDecRPL = 2;                     // rows each lane updates per pass

// Each row is handled by LPR lanes, each lane taking NV4 groups of four
// columns (group m of lane sub at column 4 sub + 4 LPR m): 16 columns per
// lane at D = 32, 64, 128; at D = 96 eight lanes of 12 columns, and three
// rows per lane per pass so that one 96-row chunk is a whole head.
template <int D, int REPMAX>
struct DecGeom {
  static constexpr int LPR = D == 96 ? 8 : D / 16;         // lanes per row
  static constexpr int NV4 = D / (4 * LPR);                // float4 groups per lane
  static constexpr int RPL = D == 96 ? 3 : kDecRPL;        // rows each lane updates per pass
  static constexpr int RPW = 32 / LPR;                     // rows per warp, per row slot
  static constexpr int WROWS = RPW * RPL;                  // rows per warp pass
  static constexpr int CHUNK_ROWS = WROWS * kDecCW < D ? WROWS * kDecCW : D;
  static constexpr int CPH = D / CHUNK_ROWS;               // chunks per head
  static constexpr uint32_t SLOT_BYTES = CHUNK_ROWS * D * 4;
  static constexpr int SLOT_FLOATS = CHUNK_ROWS * D;
  static constexpr int STAGES_RAW = dec_ring_bytes(REPMAX) / (int)SLOT_BYTES;
  static constexpr int STAGES = STAGES_RAW < kDecMaxStages ? STAGES_RAW : kDecMaxStages;
  static constexpr int RING_BYTES = STAGES * (int)SLOT_BYTES;
};

// Bounded wait that also gives up as soon as another warp has aborted.
__device__ __forceinline__ bool dec_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait_bounded(bar, parity, abort_flag);
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecCW * 32) : "memory");
}

template <typename T, int D, int REPMAX, bool SLOTS>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_step_kernel(const DecodeArgs p, const int num_items) {
  using G = DecGeom<D, REPMAX>;
  constexpr int LPR = G::LPR, RPW = G::RPW;
  constexpr int kDecStages = G::STAGES;
  constexpr int kDecMaxRep = REPMAX;
  constexpr int NC = kDecCW * 32;
  static_assert(2 * D <= NC, "each consumer thread owns at most one q/k channel");

  extern __shared__ __align__(128) float ring[];
  // per-item buffers are doubled (by item parity): a fast warp may start the
  // next item while slow warps finish this one, and an item's outputs are
  // written during the next item
  __shared__ float sq[2][D], sk[2][D], sv[2][kDecMaxRep][D], so[2][kDecMaxRep][D];
  __shared__ float sgate[2][kDecMaxRep][2];
  __shared__ float snw[D];
  __shared__ __align__(8) uint64_t full_bar[kDecMaxStages], empty_bar[kDecMaxStages];
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rep = p.rep, Hk = p.Hk, Hv = p.Hv;

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kDecCW);
    }
    s_abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;
  grid_launch_dependents();

  // state slot of batch row b, or -1 for a padded or out-of-range row (the
  // plain call is compiled without the table: slot b, never -1)
  auto slot_of = [&](int b) -> int {
    if (!SLOTS) return b;
    const int s = __ldg(p.slots + b);
    return (s >= 0 && s < p.num_slots) ? s : -1;
  };

  if (warp == kDecCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t k = 0;
      for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
        const int b = item / Hk, kh = item - (item / Hk) * Hk;
        const int sb = slot_of(b);
        if (SLOTS && sb < 0) continue;
        for (int r = 0; r < rep; ++r) {
          const int h = p.map == GDN_MAP_TILED ? kh + r * Hk : kh * rep + r;
          const float* gS = p.state + ((size_t)sb * Hv + h) * (size_t)(D * D);
          for (int c = 0; c < G::CPH; ++c, ++k) {
            const int slot = (int)(k % kDecStages);
            if (k >= (uint32_t)kDecStages &&
                !dec_wait(&empty_bar[slot], ((k / kDecStages) - 1) & 1, abort_flag))
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
  // The producer streams state rows at once; the consumers read the
  // activations, which the preceding kernel may have written, only after it
  // has completed (nothing to wait for without an overlapped launch).
  grid_dependency_wait();
  const size_t C = (size_t)p.C;
  const int qk_f = Hk * D;
  const T* w = static_cast<const T*>(p.conv_w);
  const int sub = lane % LPR, rq = lane / LPR;
  // Prefetch registers: the conv inputs and gate scalars of the NEXT item
  // are loaded while the current one is processed, so an item's prologue
  // never waits on global memory.
  constexpr int NIT = ((2 + kDecMaxRep) * D + NC - 1) / NC;
  T pcs0[NIT], pcs1[NIT], pcs2[NIT], pcx[NIT], pcw[NIT][4];
  int pchan[NIT];
  float pga = 0.f, pgb = 0.f, pgp = 0.f, pgd = 0.f;
  constexpr int PER = D / 32;  // output elements per lane
  // warp w writes the outputs of heads w, w + kDecCW, ... (one head each up
  // to eight heads per K head, two for sixteen)
  constexpr int HPW = (kDecMaxRep + kDecCW - 1) / kDecCW;
  T pz[HPW][PER];
  if (p.z != nullptr)
    for (int j = tid; j < D; j += NC) snw[j] = p.norm_w[j];
  auto prefetch = [&](int item) {
    const int b = item / Hk, kh = item - (item / Hk) * Hk;
    const int sb = SLOTS ? (item < num_items ? slot_of(b) : -1) : b;
    const T* xrow = static_cast<const T*>(p.mixed_qkv) + (size_t)b * C;
    const T* cst = static_cast<const T*>(p.conv_state) + (size_t)(SLOTS && sb < 0 ? 0 : sb) * C * 3;
    const int nch = (2 + rep) * D;
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int idx = tid + it * NC;
      pchan[it] = -1;
      if (item < num_items && (!SLOTS || sb >= 0) && idx < nch) {
        const int which = idx / D, i = idx - which * D;
        int c;
        if (which < 2) {
          c = which * qk_f + kh * D + i;
        } else {
          const int r = which - 2;
          const int h = p.map == GDN_MAP_TILED ? kh + r * Hk : kh * rep + r;
          c = 2 * qk_f + h * D + i;
        }
        pchan[it] = c;
        const T* cp = cst + (size_t)c * 3;
        pcs0[it] = cp[0];
        pcs1[it] = cp[1];
        pcs2[it] = cp[2];
        pcx[it] = xrow[c];
#pragma unroll
        for (int j = 0; j < 4; ++j) pcw[it][j] = w[(size_t)c * 4 + j];
      } else {
        pcs0[it] = pcs1[it] = pcs2[it] = pcx[it] = T();
#pragma unroll
        for (int j = 0; j < 4; ++j) pcw[it][j] = T();
      }
    }
    if (item < num_items && tid < rep) {
      const int h = p.map == GDN_MAP_TILED ? kh + tid * Hk : kh * rep + tid;
      const int gi = b * Hv + h;
      pga = to_f32(static_cast<const T*>(p.a)[gi]);
      pgb = to_f32(static_cast<const T*>(p.b)[gi]);
      pgp = p.decay_param[h];
      pgd = p.dt_bias[h];
    }
#pragma unroll
    for (int hw = 0; hw < HPW; ++hw) {
      const int r = warp + hw * kDecCW;
      if (item < num_items && p.z != nullptr && r < rep) {
        const int h = p.map == GDN_MAP_TILED ? kh + r * Hk : kh * rep + r;
        const T* zr = static_cast<const T*>(p.z) + ((size_t)b * Hv + h) * D + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; ++e) pz[hw][e] = zr[e];
      }
    }
  };
  prefetch(blockIdx.x);

  // Outputs of an item (core output and/or gated norm, warp r < rep taking
  // head r) are written after every warp has finished its state pass, i.e.
  // past the next item's first barrier, so they overlap the next item's
  // stream instead of holding every warp at a barrier of their own.
  auto write_outputs = [&](int it, int pb, const T (&zz)[HPW][PER]) {
    if (*abort_flag) return;
    const int b = it / Hk, kh = it - (it / Hk) * Hk;
#pragma unroll
    for (int hw = 0; hw < HPW; ++hw) {
      const int r = warp + hw * kDecCW;
      if (r >= rep) break;
      const int h = p.map == GDN_MAP_TILED ? kh + r * Hk : kh * rep + r;
      const size_t obase = ((size_t)b * Hv + h) * D + lane * PER;
      float ov[PER];
#pragma unroll
      for (int e = 0; e < PER; ++e) ov[e] = so[pb][r][lane * PER + e];
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
        T* outr = static_cast<T*>(p.out) + obase;
#pragma unroll
        for (int e = 0; e < PER; ++e)
          outr[e] = from_f32<T>(ov[e] * inv * snw[lane * PER + e] * silu_f(to_f32(zz[hw][e])));
      }
    }
  };

  uint32_t k = 0;
  int prev_item = -1, prev_buf = 0;
  T zp[HPW][PER];  // z of the previous item, for its outputs
#pragma unroll
  for (int hw = 0; hw < HPW; ++hw)
#pragma unroll
    for (int e = 0; e < PER; ++e) zp[hw][e] = T();
  for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
    const int b = item / Hk, kh = item - (item / Hk) * Hk;
    const int sb = slot_of(b);  // the producer skipped this row's state too if < 0
    if (SLOTS && sb < 0 && tid == 0 && kh == 0 && __ldg(p.slots + b) >= p.num_slots)
      record_device_error(GDN_ERR_EXTENT);
    T* cstate = static_cast<T*>(p.conv_state) + (size_t)(SLOTS && sb < 0 ? 0 : sb) * C * 3;
    const int buf = ((item - (int)blockIdx.x) / (int)gridDim.x) & 1;
    T cs1[NIT], cs2[NIT], cx[NIT];
    int chan[NIT];
    float y[NIT];
    T zc[HPW][PER];
#pragma unroll
    for (int hw = 0; hw < HPW; ++hw)
#pragma unroll
      for (int e = 0; e < PER; ++e) zc[hw][e] = pz[hw][e];
    // conv + SiLU for this item from the prefetched registers: channels
    // [q of kh | k of kh | v of each head]
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      chan[it] = pchan[it];
      cs1[it] = pcs1[it];
      cs2[it] = pcs2[it];
      cx[it] = pcx[it];
      float acc = to_f32(pcw[it][0]) * to_f32(pcs0[it]);
      acc += to_f32(pcw[it][1]) * to_f32(pcs1[it]);
      acc += to_f32(pcw[it][2]) * to_f32(pcs2[it]);
      acc += to_f32(pcw[it][3]) * to_f32(pcx[it]);
      y[it] = silu_f(acc);
    }
    if (tid < rep) {
      sgate[buf][tid][0] = expf(gate_g(p.decay, pgp, pgd, pga));
      sgate[buf][tid][1] = sigmoid_f(pgb);
    }
    prefetch(item + gridDim.x);
    int qk_c = -1;
    T qk_s1 = T(), qk_s2 = T(), qk_x = T();
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      if (chan[it] < 0) continue;
      const int idx = tid + it * NC;
      const int which = idx / D, i = idx - which * D;
      if (which >= 2) {
        sv[buf][which - 2][i] = y[it];
        T* cp = cstate + (size_t)chan[it] * 3;  // this CTA alone reads and writes these channels
        cp[0] = cs1[it];
        cp[1] = cs2[it];
        cp[2] = cx[it];
      } else {
        (which == 0 ? sq[buf] : sk[buf])[i] = y[it];
        qk_c = chan[it];
        qk_s1 = cs1[it];
        qk_s2 = cs2[it];
        qk_x = cx[it];
      }
    }
    // this item's q, k, v and gates are in shared memory, and every warp has
    // finished the previous item's state pass
    consumer_sync();
    if (prev_item >= 0) write_outputs(prev_item, prev_buf, zp);
#pragma unroll
    for (int hw = 0; hw < HPW; ++hw)
#pragma unroll
      for (int e = 0; e < PER; ++e) zp[hw][e] = zc[hw][e];
    prev_item = item;
    prev_buf = buf;

    // l2 norms of q and k and k.q, each warp over all D (no second barrier)
    float qq = 0.f, kk = 0.f, qkr = 0.f;
#pragma unroll
    for (int i = lane; i < D; i += 32) {
      const float qv = sq[buf][i], kv = sk[buf][i];
      qq = fmaf(qv, qv, qq);
      kk = fmaf(kv, kv, kk);
      qkr = fmaf(qv, kv, qkr);
    }
    qq = group_sum<32>(qq);
    kk = group_sum<32>(kk);
    qkr = group_sum<32>(qkr);
    const float inv_q = 1.f / sqrtf(qq + p.l2_eps);
    const float inv_k = 1.f / sqrtf(kk + p.l2_eps);
    const float kq = qkr * inv_q * inv_k * p.scale;
    constexpr int NV4 = G::NV4, RPL = G::RPL;
    float4 kr[NV4], qr[NV4];  // this lane's columns of the normalised k and scaled q
    {
      const float sqs = inv_q * p.scale;
#pragma unroll
      for (int m = 0; m < NV4; ++m) {
        const int col = 4 * sub + 4 * LPR * m;
        kr[m] = make_float4(sk[buf][col] * inv_k, sk[buf][col + 1] * inv_k, sk[buf][col + 2] * inv_k,
                            sk[buf][col + 3] * inv_k);
        qr[m] = make_float4(sq[buf][col] * sqs, sq[buf][col + 1] * sqs, sq[buf][col + 2] * sqs,
                            sq[buf][col + 3] * sqs);
      }
    }

    // a row without a state slot: zero core outputs, no state pass (its
    // conv channels were never loaded, so no conv state is written either)
    if (SLOTS && sb < 0) {
      for (int j = tid; j < rep * D; j += NC) so[buf][j / D][j - (j / D) * D] = 0.f;
      continue;
    }

    // the state pass over the item's heads, chunk by chunk from the ring
    for (int r = 0; r < rep; ++r) {
      const int h = p.map == GDN_MAP_TILED ? kh + r * Hk : kh * rep + r;
      float* gS = p.state + ((size_t)sb * Hv + h) * (size_t)(D * D);
      const float alpha = sgate[buf][r][0], beta = sgate[buf][r][1];
      for (int c = 0; c < G::CPH; ++c, ++k) {
        const int slot = (int)(k % kDecStages);
        const bool ready = dec_wait(&full_bar[slot], (k / kDecStages) & 1, abort_flag);
        if (ready && warp * G::WROWS < G::CHUNK_ROWS) {
          float4 s4[RPL][NV4];
          int rowv[RPL];
#pragma unroll
          for (int u = 0; u < RPL; ++u) {
            const int rl = warp * G::WROWS + u * RPW + rq;  // row within the chunk
            rowv[u] = c * G::CHUNK_ROWS + rl;
            const float* srow = ring + slot * G::SLOT_FLOATS + rl * D;
#pragma unroll
            for (int m = 0; m < NV4; ++m)
              s4[u][m] = *reinterpret_cast<const float4*>(srow + 4 * sub + 4 * LPR * m);
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
#pragma unroll
          for (int u = 0; u < RPL; ++u) {
            const int row = rowv[u];
            const float d = beta * (sv[buf][r][row] - alpha * pk[u]);
            const float o = fmaf(alpha, pq[u], d * kq);
            float* grow = gS + (size_t)row * D;
            row_update<NV4>(s4[u], kr, alpha, d);
#pragma unroll
            for (int m = 0; m < NV4; ++m) __stcs(reinterpret_cast<float4*>(grow + 4 * sub + 4 * LPR * m), s4[u][m]);
            if (sub == 0) so[buf][r][row] = o;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
      }
    }

    // new q/k conv state: this CTA read the old values itself, in the prologue
    if (qk_c >= 0 && !*abort_flag) {
      T* cp = cstate + (size_t)qk_c * 3;
      cp[0] = qk_s1;
      cp[1] = qk_s2;
      cp[2] = qk_x;
    }
  }
  // every warp has finished the last item's state pass: its outputs
  consumer_sync();
  if (prev_item >= 0) write_outputs(prev_item, prev_buf, zp);
}

static int sm_count() {
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
static cudaError_t launch_decode_t(const DecodeArgs& p, int32_t batch, cudaStream_t stream) {
  auto kern = p.slots != nullptr ? decode_step_kernel<T, D, REPMAX, true>
                                 : decode_step_kernel<T, D, REPMAX, false>;
  const int smem = DecGeom<D, REPMAX>::RING_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int items = batch * p.Hk;
  const int grid = items < sm_count() ? items : sm_count();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.overlap_prev ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, p, items);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The per-item register and shared buffers are sized for REPMAX V heads per
// K head: 2, 4, 8 or 16.
template <typename T, int D>
static cudaError_t launch_decode_r(const DecodeArgs& p, int32_t batch, cudaStream_t stream) {
  if (p.rep <= 2) return launch_decode_t<T, D, 2>(p, batch, stream);
  if (p.rep <= 4) return launch_decode_t<T, D, 4>(p, batch, stream);
  if (p.rep <= 8) return launch_decode_t<T, D, 8>(p, batch, stream);
  return launch_decode_t<T, D, 16>(p, batch, stream);
}

template <typename T>
static cudaError_t launch_decode_d(const DecodeArgs& p, int32_t D, int32_t batch,
                                   cudaStream_t stream) {
  switch (D) {
    case 32: return launch_decode_r<T, 32>(p, batch, stream);
    case 64: return launch_decode_r<T, 64>(p, batch, stream);
    case 96: return launch_decode_r<T, 96>(p, batch, stream);
    case 128: return launch_decode_r<T, 128>(p, batch, stream);
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
