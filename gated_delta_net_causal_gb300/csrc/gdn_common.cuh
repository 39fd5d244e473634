// Shared device helpers for the gated delta-net kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// ------------------------------------------------------------------ dtypes

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// d = a * b + c on both lanes of a pair, one rounding each (the paired
// fp32 FMA of sm_100 and later)
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// --------------------------------------------------------------- activations
// fp32 forms of the gate nonlinearities: sigmoid in two branches so exp never
// overflows; softplus linear above 20 and exp below -20 (the cut-offs of the
// Metal test's CPU helpers).

__device__ __forceinline__ float sigmoid_f(float x) {
  if (x >= 0.f) return 1.f / (1.f + expf(-x));
  const float e = expf(x);
  return e / (1.f + e);
}
__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }
// x sigmoid(x) with the fast exponential and divide (relative error about
// 1e-6; for z -> -inf the quotient flushes to 0), for the memory-bound norm
// passes where the exact form's instruction count sets the time
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.f + __expf(-x)); }
__device__ __forceinline__ float softplus_f(float x) {
  if (x > 20.f) return x;
  if (x < -20.f) return expf(x);
  return log1pf(expf(x));
}

// gate value g for V head h from the raw input a
__device__ __forceinline__ float gate_g(int decay, float param, float dt_bias, float a) {
  const float rate = decay == GDN_DECAY_LOG_RATE ? -expf(param) : param;
  return rate * softplus_f(a + dt_bias);
}

// The per-lane partial sums of a decode row over its NV4 column groups, in
// the one fixed order both decode kernels use (so they agree bit for bit).
// Dot product of a lane's share of a state row with the matching columns of
// a vector, both as NV4 groups of four: lanes (x, y) and (z, w) of the
// groups accumulate in one paired FMA chain, group after group, and the two
// halves are added last. The one- and multi-token decode kernels both use
// it, so they round identically.
template <int NV4>
__device__ __forceinline__ float row_dot(const float4 (&s)[NV4], const float4 (&v)[NV4]) {
  float2 a = fma2(make_float2(s[0].x, s[0].y), make_float2(v[0].x, v[0].y), make_float2(0.f, 0.f));
  float2 b = fma2(make_float2(s[0].z, s[0].w), make_float2(v[0].z, v[0].w), make_float2(0.f, 0.f));
#pragma unroll
  for (int m = 1; m < NV4; ++m) {
    a = fma2(make_float2(s[m].x, s[m].y), make_float2(v[m].x, v[m].y), a);
    b = fma2(make_float2(s[m].z, s[m].w), make_float2(v[m].z, v[m].w), b);
  }
  return (a.x + b.x) + (a.y + b.y);
}
// s <- alpha s + d v on a lane's groups (one rounding of alpha s, then one
// FMA per element)
template <int NV4>
__device__ __forceinline__ void row_update(float4 (&s)[NV4], const float4 (&v)[NV4], float alpha, float d) {
  const float2 al = make_float2(alpha, alpha), dd = make_float2(d, d), nz = make_float2(-0.f, -0.f);
#pragma unroll
  for (int m = 0; m < NV4; ++m) {
    const float2 lo = fma2(dd, make_float2(v[m].x, v[m].y), fma2(al, make_float2(s[m].x, s[m].y), nz));
    const float2 hi = fma2(dd, make_float2(v[m].z, v[m].w), fma2(al, make_float2(s[m].z, s[m].w), nz));
    s[m] = make_float4(lo.x, lo.y, hi.x, hi.y);
  }
}

template <int NV4>
__device__ __forceinline__ float sum_groups(const float (&a)[NV4]) {
  static_assert(NV4 == 3 || NV4 == 4, "three or four column groups per lane");
  if constexpr (NV4 == 4) return (a[0] + a[1]) + (a[2] + a[3]);
  else return (a[0] + a[1]) + a[2];
}

__device__ __forceinline__ int k_head_of(int map, int h, int Hk, int rep) {
  return map == GDN_MAP_TILED ? (h % Hk) : (h / rep);
}

// --------------------------------------------------------------- reductions

template <int W>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- PTX: misc

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Every wait on another thread's progress is bounded in time: after
// kWaitLimitNs of the global timer it records GDN_ERR_TIMEOUT in the device
// error word and gives up, and the kernel runs to its end.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// One error word per translation unit (read back by the host through
// gdn_device_error); the first recorded status wins.
static __device__ int32_t g_device_error = 0;
__device__ __forceinline__ void record_device_error(int32_t status) {
  atomicCAS(&g_device_error, 0, status);
}

// ---------------------------------------------------------- PTX: mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on the phase with the given parity. Gives up (false) when
// *abort_flag is set by another thread, or after limit_ns, recording
// GDN_ERR_TIMEOUT and raising *abort_flag so the other waiters follow.
// (The loop lives in a function of its own so that a wait that completes
// at once costs the caller no registers.)
__device__ __forceinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                            uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (abort_flag != nullptr && *abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15) == 0 && global_ns() - t0 > limit_ns) {
      record_device_error(GDN_ERR_TIMEOUT);
      if (abort_flag != nullptr) *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, limit_ns);
}
// Bounded wait without an abort flag.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_bounded(bar, parity, nullptr);
}

// ------------------------------------------------- PTX: bulk async copies
// 1-D bulk copies (no tensor map). Addresses 16-byte aligned, size a
// multiple of 16.

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ------------------------------------------- PTX: programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while
// the preceding kernel on the stream still runs. grid_dependency_wait()
// returns once that kernel has completed and its writes are visible to the
// calling thread (at once when the launch carries no such dependency);
// grid_launch_dependents() lets the next kernel of that kind start once every
// CTA of this grid has called it or exited.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------ PTX: cluster
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr), "r"(rank));
  return out;
}
// Asynchronous 4-byte store into another CTA's shared memory that completes
// 4 transaction bytes on that CTA's mbarrier (both addresses from mapa).
__device__ __forceinline__ void st_async_cluster_f32(uint32_t remote_addr, float v,
                                                     uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr),
      "r"(__float_as_uint(v)), "r"(remote_bar)
      : "memory");
}
__device__ __forceinline__ float4 ld_shared_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

}  // namespace gdn
