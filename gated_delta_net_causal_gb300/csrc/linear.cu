// Linear layer y = x W^T (+ bias) on the 5th-generation tensor cores: the
// projections around the core in a decode step (libmir-metal decode/mod.rs,
// `build`: the qkv, gate, beta and alpha projections of the input and the
// output projection, each a `Linear::forward`, matmul then bias).
//
// x [M][K] bf16 with M <= 128 rows (the batch), W [N][K] bf16 (one row per
// output feature), fp32 accumulation in TMEM, bf16 out. At decode batch
// sizes the work is bound by streaming W once: each CTA takes a band of 64
// output features and streams its W rows (and the M rows of x) through a TMA
// ring. The MMA always spans 128 rows; rows past M of the x tile hold
// whatever the buffer held and only reach accumulator rows that are never
// stored. The output columns may be routed to up to four destinations (the
// fused input projection writes qkv | z | b | a from one launch).
//
// Split-K for narrow outputs (few bands): grid.y splits the K steps and
// the splits of a band form one thread-block cluster (at most 8). Each CTA
// keeps its fp32 partial tile in its own shared memory; the cluster adds the
// tiles in split order over distributed shared memory (so the result does
// not depend on which CTA ran first), adds the bias, rounds and stores. No
// global scratch, fence or atomic is involved.
#include <cuda.h>
#include <string.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {
namespace {

constexpr int kLBM = 128;  // MMA rows (batch rows; the x tile holds M of them)
constexpr int kLBN = 64;   // output features per CTA
constexpr int kLBK = 64;   // K per stage (one 128-byte swizzle atom of bf16)
constexpr uint32_t kLWTile = kLBN * kLBK * 2;  // 8 KB
// A stage is the x tile (M rounded up to 8 rows of 128 bytes, so a multiple
// of 1024 bytes) then the W tile; as many stages as fit in the ring budget
// below. The MMA reads 128 rows of x from
// each stage's start, so the allocation ends 128 x 128 bytes past the last
// stage's start at least (the rows past M it reads are never used).
constexpr int kLMaxStages = 12;
// three CTAs per SM with a 64 KB ring from 32 rows of x up (more weight
// streams in flight, K split over more CTAs), two with a 96 KB ring below
// (a small x tile leaves the smaller ring too few bytes in flight)
constexpr int kLCtasPerSm = 3;
__host__ __device__ constexpr int linear_ctas_per_sm(int32_t M) { return M >= 32 ? 3 : 2; }
__host__ __device__ constexpr uint32_t linear_stage_budget(int32_t M) { return M >= 32 ? 64 * 1024 : 96 * 1024; }
constexpr int kLThreads = 128;  // warp 0 lane 0 loads, warp 1 issues MMAs, all four store
constexpr int kLMaxSplits = 8;  // the portable cluster size

__global__ void __launch_bounds__(kLThreads, kLCtasPerSm)
    linear_kernel(const LinearArgs p, const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_w) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full[kLMaxStages], empty[kLMaxStages], done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int band = blockIdx.x, n0 = band * kLBN;
  const int stages = p.stages;
  const uint32_t x_tile = (uint32_t)((p.M + 7) / 8) * 1024, stage_bytes = x_tile + kLWTile;
  const int nk = p.K / kLBK;
  const int k_begin = (int)((int64_t)blockIdx.y * nk / p.splits);
  const int k_end = (int)((int64_t)(blockIdx.y + 1) * nk / p.splits);
  const int k_len = k_end - k_begin;

  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, kLBN);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tb = s_tmem;
  volatile int* abort_flag = &s_abort;
  uint32_t n_loads = 0;
  grid_launch_dependents();

  if (warp == 0 && lane == 0) {
    // producer: stage i % S holds K step k_begin + i. The first S stages'
    // weight tiles go out before x, which the preceding kernel may have
    // written, is read (after it has completed; at once without an
    // overlapped launch)
    const int first = k_len < stages ? k_len : stages;
    for (int i = 0; i < first; ++i) {
      mbar_arrive_expect_tx(&full[i], (uint32_t)p.M * (kLBK * 2) + kLWTile);
      ++n_loads;
      tc::tma_load_2d(sm + i * stage_bytes + x_tile, &tm_w, (k_begin + i) * kLBK, n0, &full[i]);
    }
    grid_dependency_wait();
    for (int i = 0; i < first; ++i) tc::tma_load_2d(sm + i * stage_bytes, &tm_x, (k_begin + i) * kLBK, 0, &full[i]);
    for (int i = first; i < k_len; ++i) {
      const int s = i % stages;
      if (!mbar_wait_bounded(&empty[s], ((i / stages) - 1) & 1, abort_flag)) break;
      mbar_arrive_expect_tx(&full[s], (uint32_t)p.M * (kLBK * 2) + kLWTile);
      ++n_loads;
      const int kx = (k_begin + i) * kLBK;
      tc::tma_load_2d(sm + s * stage_bytes, &tm_x, kx, 0, &full[s]);
      tc::tma_load_2d(sm + s * stage_bytes + x_tile, &tm_w, kx, n0, &full[s]);
    }
  } else if (warp == 1) {
    const uint32_t id = tc::idesc(tc::kBF16, kLBM, kLBN);
    const uint64_t d0 = tc::sdesc_sw128(smem_u32(sm));
    bool ok = true;
    for (int i = 0; i < k_len; ++i) {
      const int s = i % stages;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (i / stages) & 1, abort_flag));
      if (!ok) break;
      tc::fence_after_sync();
      const uint64_t da = d0 + (uint64_t)((s * stage_bytes) >> 4);
      const uint64_t dw = d0 + (uint64_t)((s * stage_bytes + x_tile) >> 4);
#pragma unroll
      for (int ks = 0; ks < kLBK / 16; ++ks)
        tc::mma_f16_elect(tb, tc::sdesc_at(da, kLBM, ks), tc::sdesc_at(dw, kLBN, ks), id, i > 0 || ks > 0);
      tc::mma_commit_elect(&empty[s]);
    }
    tc::mma_commit_elect(&done);
  }

  // epilogue: thread (warp w, lane) holds row m = 32 w + lane of the
  // accumulator (TMEM lane m), 64 columns
  const bool ok = mbar_wait_bounded(&done, 0, abort_flag) && !*abort_flag;
  tc::fence_after_sync();
  const int m = 32 * warp + lane;
  float v[kLBN];
  if (__all_sync(0xffffffffu, ok)) {
#pragma unroll
    for (int c = 0; c < kLBN / 16; ++c)
      tc::tmem_ld16(tb + ((uint32_t)(32 * warp) << 16) + 16 * c, *reinterpret_cast<float(*)[16]>(v + 16 * c));
    tc::tmem_wait_ld();
  } else {
#pragma unroll
    for (int e = 0; e < kLBN; ++e) v[e] = 0.f;
  }
  // bias, one rounding, and the destination of an 8-column group of row m
  auto store8 = [&](int m, int g8, const float* x8) {
    const int n = n0 + 8 * g8;
    if (n >= p.route.start[p.route.count]) return;  // padding columns
    int r = 0;
#pragma unroll
    for (int q = 1; q < kLinearRoutes; ++q)
      if (q < p.route.count && n >= p.route.start[q]) r = q;
    uint32_t w4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float b0 = p.bias != nullptr ? __ldg(p.bias + n + 2 * e) : 0.f;
      const float b1 = p.bias != nullptr ? __ldg(p.bias + n + 2 * e + 1) : 0.f;
      w4[e] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x8[2 * e] + b0)) |
              ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x8[2 * e + 1] + b1)) << 16);
    }
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.route.dst[r]) + (size_t)m * p.route.ld[r] +
                         (n - p.route.start[r]);
    *reinterpret_cast<uint4*>(dst) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  };
  if (p.splits == 1) {
    if (m < p.M && !*abort_flag)
#pragma unroll
      for (int g8 = 0; g8 < kLBN / 8; ++g8) store8(m, g8, v + 8 * g8);
  } else {
    // the K splits of a band are one cluster. This split's fp32 partial tile
    // goes into its own shared memory (the ring is idle: every load it
    // issued was consumed by an MMA that has completed), 16-byte group c of
    // row m at group c ^ (m % 16); after a cluster barrier every CTA sums
    // its share of the (row, 8-column group) units over the cluster's tiles
    // in rank order, so the result does not depend on which CTA ran first;
    // a second barrier keeps each tile in place until its peers have read
    // it. Every thread reaches both barriers, whatever happened before.
    float* part = reinterpret_cast<float*>(sm);
    if (m < p.M) {
#pragma unroll
      for (int c = 0; c < kLBN / 4; ++c)
        *reinterpret_cast<float4*>(part + m * kLBN + 4 * (c ^ (m & 15))) =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    const int S = p.splits, rank = (int)cluster_ctarank();
    const uint32_t base = smem_u32(part);
    if (!*abort_flag) {
      for (int u = rank * kLThreads + tid; u < p.M * (kLBN / 8); u += S * kLThreads) {
        const int um = u >> 3, g8 = u & 7;
        const uint32_t o0 = (uint32_t)(um * kLBN + 4 * ((2 * g8) ^ (um & 15))) * 4u;
        const uint32_t o1 = (uint32_t)(um * kLBN + 4 * ((2 * g8 + 1) ^ (um & 15))) * 4u;
        float x8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x8[e] = 0.f;
        for (int sp = 0; sp < S; ++sp) {
          const float4 a0 = ld_shared_cluster_f32x4(map_shared_rank(base + o0, (uint32_t)sp));
          const float4 a1 = ld_shared_cluster_f32x4(map_shared_rank(base + o1, (uint32_t)sp));
          x8[0] += a0.x, x8[1] += a0.y, x8[2] += a0.z, x8[3] += a0.w;
          x8[4] += a1.x, x8[5] += a1.y, x8[6] += a1.z, x8[7] += a1.w;
        }
        store8(um, g8, x8);
      }
    }
    cluster_arrive_release();
    cluster_wait_acquire();
  }

  // drain: every load this CTA issued has landed (the last one into each
  // stage) and its MMAs completed, before TMEM is released
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    for (uint32_t s = 0; s < (uint32_t)stages && s < n_loads; ++s) {
      const uint32_t uses = (n_loads - s + stages - 1) / stages;  // loads into stage s
      mbar_wait(&full[s], (uses - 1) & 1);
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tb, kLBN);
  }
}

int sm_count_linear() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

}  // namespace

static int max_splits(int32_t K) {
  const int half = K / kLBK / 2;  // each split at least two K steps
  return half < 1 ? 1 : (half < kLMaxSplits ? half : kLMaxSplits);
}

int64_t linear_workspace_bytes(int32_t, int32_t, int32_t) { return 0; }

bool linear_supported() { return tc::encode_fn() != nullptr; }

cudaError_t launch_linear(LinearArgs p, const void* x, int64_t x_stride, const void* w, void*,
                          cudaStream_t stream) {
  if (p.M == 0 || p.N == 0) return cudaSuccess;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap mx, mw;
  if (!tc::make_map_2d(&mx, x, p.M, p.K, x_stride, 2, bf, kLBK, (uint32_t)p.M, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc::make_map_2d(&mw, w, p.N, p.K, p.K, 2, bf, kLBK, kLBN, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
    return cudaErrorInvalidValue;
  const int bands = p.N / kLBN;
  // as many K splits as keep every CTA slot of the SMs busy in one wave
  // (each split at least two K steps, at most one cluster of kLMaxSplits)
  int splits = (linear_ctas_per_sm(p.M) * sm_count_linear()) / bands;
  if (splits > max_splits(p.K)) splits = max_splits(p.K);
  if (splits < 1) splits = 1;
  p.splits = splits;
  const uint32_t stage_bytes = (uint32_t)((p.M + 7) / 8) * 1024 + kLWTile;
  int stages = (int)(linear_stage_budget(p.M) / stage_bytes);
  p.stages = stages < kLMaxStages ? (stages < 2 ? 2 : stages) : kLMaxStages;
  const uint32_t x_tile = stage_bytes - kLWTile;
  const uint32_t smem = (uint32_t)p.stages * stage_bytes + (kLBM * 128 - (x_tile < kLBM * 128 ? x_tile : kLBM * 128)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)bands, (unsigned)splits);
  cfg.blockDim = dim3(kLThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)splits;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchAttribute attr2[2];
  int na = 0;
  if (splits > 1) attr2[na++] = attr[0];
  if (p.overlap_prev) {
    attr2[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr2[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr2;
  cfg.numAttrs = (unsigned)na;
  e = cudaLaunchKernelEx(&cfg, linear_kernel, p, mx, mw);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gdn

GDN_DEFINE_ERROR_READER(linear)
