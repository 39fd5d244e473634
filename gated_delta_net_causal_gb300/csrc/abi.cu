// C ABI entry points: host-side validation, then one launcher call each.
// Nothing is enqueued unless every check passes.
#include <math.h>
#include <stdint.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

using gdn::DecodeArgs;

constexpr int64_t kMaxGridY = 65535;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t dtype_size(int32_t dt) {
  switch (dt) {
    case GDN_F16:
    case GDN_BF16: return 2;
    case GDN_F32: return 4;
    default: return 0;
  }
}

// a*b with overflow detection into *out; false on overflow or negative inputs
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};
Range range_of(const void* p, int64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Range{lo, lo + (uintptr_t)(bytes > 0 ? bytes : 0)};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

gdn_status check_dims(const gdn_dims* d) {
  if (d == nullptr) return GDN_ERR_INVALID_ARG;
  if (d->n_k_heads < 1 || d->n_v_heads < 1) return GDN_ERR_INVALID_ARG;
  if (d->n_v_heads % d->n_k_heads != 0) return GDN_ERR_INVALID_ARG;
  if (d->map != GDN_MAP_GROUPED && d->map != GDN_MAP_TILED) return GDN_ERR_INVALID_ARG;
  if (d->decay != GDN_DECAY_LOG_RATE && d->decay != GDN_DECAY_NEGATIVE_RATE)
    return GDN_ERR_INVALID_ARG;
  if (dtype_size(d->io_dtype) == 0) return GDN_ERR_INVALID_ARG;
  if (!(d->l2_eps >= 0.f) || !isfinite(d->l2_eps)) return GDN_ERR_INVALID_ARG;
  if (!(d->rms_eps >= 0.f) || !isfinite(d->rms_eps)) return GDN_ERR_INVALID_ARG;
  if (d->head_dim < 1) return GDN_ERR_INVALID_ARG;
  if (d->head_dim != 32 && d->head_dim != 64 && d->head_dim != 96 && d->head_dim != 128)
    return GDN_ERR_UNSUPPORTED;
  if (d->n_v_heads > kMaxGridY) return GDN_ERR_EXTENT;
  const int64_t C = (2 * (int64_t)d->n_k_heads + d->n_v_heads) * d->head_dim;
  if (C > INT32_MAX / 4) return GDN_ERR_EXTENT;
  return GDN_OK;
}

int64_t qkv_features(const gdn_dims* d) {
  return (2 * (int64_t)d->n_k_heads + d->n_v_heads) * d->head_dim;
}

gdn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// Shared by gdn_decode_step (slots == nullptr: row b owns slot b, num_slots
// = batch) and gdn_decode_step_slots.
gdn_status decode_impl(const gdn_dims* dims, int32_t batch, int32_t tokens, const int32_t* slots,
                       int32_t num_slots, const void* mixed_qkv, const void* a, const void* b,
                       const float* decay_param, const float* dt_bias, const void* conv_w,
                       void* conv_state, float* state, float* core_out, const void* z,
                       const float* norm_w, void* out, void* stream, bool overlap_prev = false) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (batch < 0 || num_slots < 0 || tokens < 1) return GDN_ERR_INVALID_ARG;
  if (tokens > 8 || (tokens > 1 && slots != nullptr)) return GDN_ERR_UNSUPPORTED;
  if (batch > kMaxGridY) return GDN_ERR_EXTENT;
  const int rep = dims->n_v_heads / dims->n_k_heads;
  // one token: up to 16 V heads per K head; several tokens: up to 8
  if (rep > (tokens > 1 ? 8 : 16)) return GDN_ERR_UNSUPPORTED;
  if (batch == 0) return GDN_OK;
  if (!mixed_qkv || !a || !b || !decay_param || !dt_bias || !conv_w || !conv_state || !state)
    return GDN_ERR_INVALID_ARG;
  if (slots != nullptr && !aligned16(slots)) return GDN_ERR_ALIGN;
  if (core_out == nullptr && z == nullptr) return GDN_ERR_INVALID_ARG;
  if (z != nullptr && (norm_w == nullptr || out == nullptr)) return GDN_ERR_INVALID_ARG;
  const void* ptrs[] = {mixed_qkv, a, b, decay_param, dt_bias, conv_w, conv_state, state};
  for (const void* q : ptrs)
    if (!aligned16(q)) return GDN_ERR_ALIGN;
  if ((core_out && !aligned16(core_out)) || (z && (!aligned16(z) || !aligned16(norm_w) || !aligned16(out))))
    return GDN_ERR_ALIGN;
  const int64_t es = dtype_size(dims->io_dtype);
  const int64_t C = qkv_features(dims), Hv = dims->n_v_heads, D = dims->head_dim;
  int64_t state_bytes = 0, tmp = 0;
  if (!mul_ok((int64_t)num_slots * Hv, D * D * 4, &state_bytes)) return GDN_ERR_EXTENT;
  if (!mul_ok((int64_t)num_slots, C * 3 * es, &tmp)) return GDN_ERR_EXTENT;
  const int64_t conv_bytes = tmp;
  const int64_t rows = (int64_t)batch * tokens;
  const int64_t x_bytes = rows * C * es;
  const int64_t o_bytes_f32 = rows * Hv * D * 4;
  const int64_t o_bytes_io = rows * Hv * D * es;
  const int64_t gate_bytes = rows * Hv * es;
  const Range inputs[] = {range_of(mixed_qkv, x_bytes), range_of(a, gate_bytes),
                          range_of(b, gate_bytes),      range_of(decay_param, Hv * 4),
                          range_of(dt_bias, Hv * 4),    range_of(conv_w, C * 4 * es),
                          range_of(z, z ? o_bytes_io : 0), range_of(norm_w, norm_w ? D * 4 : 0),
                          range_of(slots, slots ? (int64_t)batch * 4 : 0)};
  const Range rs = range_of(state, state_bytes), rc = range_of(conv_state, conv_bytes);
  const Range ro = range_of(core_out, core_out ? o_bytes_f32 : 0);
  const Range ry = range_of(out, z ? o_bytes_io : 0);
  for (const Range& in : inputs) {
    if (overlap(rs, in) || overlap(rc, in) || overlap(ro, in) || overlap(ry, in)) return GDN_ERR_ALIAS;
  }
  if (overlap(rs, rc) || overlap(rs, ro) || overlap(rs, ry) || overlap(rc, ro) || overlap(rc, ry) ||
      overlap(ro, ry))
    return GDN_ERR_ALIAS;
  DecodeArgs p{};
  p.mixed_qkv = mixed_qkv;
  p.a = a;
  p.b = b;
  p.decay_param = decay_param;
  p.dt_bias = dt_bias;
  p.conv_w = conv_w;
  p.conv_state = conv_state;
  p.state = state;
  p.core_out = core_out;
  p.z = z;
  p.norm_w = norm_w;
  p.out = out;
  p.slots = slots;
  p.num_slots = num_slots;
  p.tokens = tokens;
  p.Hk = dims->n_k_heads;
  p.Hv = dims->n_v_heads;
  p.rep = rep;
  p.map = dims->map;
  p.decay = dims->decay;
  p.C = (int32_t)C;
  p.l2_eps = dims->l2_eps;
  p.rms_eps = dims->rms_eps;
  p.scale = 1.0f / sqrtf((float)D);
  p.overlap_prev = overlap_prev ? 1 : 0;
  if (tokens > 1)
    return cuda_status(gdn::launch_decode_multi(p, dims->io_dtype, dims->head_dim, batch,
                                                static_cast<cudaStream_t>(stream)));
  return cuda_status(gdn::launch_decode(p, dims->io_dtype, dims->head_dim, batch,
                                        static_cast<cudaStream_t>(stream)));
}

}  // namespace

// gdn_prefill_chunked flags: known bits only, and not both carry choices
static bool prefill_flags_valid(int32_t flags) {
  constexpr int32_t known = GDN_QK_PRENORMALIZED | GDN_GATES_PRECOMPUTED | GDN_PREFILL_CUDA_CORES |
                            GDN_PREFILL_CARRY_WHOLE | GDN_PREFILL_CARRY_SLICED;
  if ((flags & ~known) != 0) return false;
  return (flags & (GDN_PREFILL_CARRY_WHOLE | GDN_PREFILL_CARRY_SLICED)) !=
         (GDN_PREFILL_CARRY_WHOLE | GDN_PREFILL_CARRY_SLICED);
}

extern "C" {

const char* gdn_status_string(int32_t status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: null pointer, bad enum or bad dims";
    case GDN_ERR_EXTENT: return "GDN_ERR_EXTENT: a size product exceeds the index or launch range";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: shape not implemented";
    case GDN_ERR_ALIAS: return "GDN_ERR_ALIAS: an output overlaps an input";
    case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN: pointer or stride not 16-byte aligned";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: the CUDA runtime reported an error";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a device-side bounded wait gave up";
    default: return "GDN_ERR_UNKNOWN";
  }
}

int32_t gdn_version(void) { return 400; }

gdn_status gdn_host_pointer(const void* host, void** device) {
  if (host == nullptr || device == nullptr) return GDN_ERR_INVALID_ARG;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(host), 0) != cudaSuccess || d == nullptr) {
    cudaGetLastError();  // not mapped: the error must not surface at the caller's next call
    return GDN_ERR_INVALID_ARG;
  }
  *device = d;
  return GDN_OK;
}

int64_t gdn_qkv_features(const gdn_dims* dims) {
  if (check_dims(dims) != GDN_OK) return -1;
  return qkv_features(dims);
}

gdn_status gdn_conv_update(const gdn_dims* dims, int32_t num_seqs, const int32_t* cu_seqlens,
                           int64_t total_tokens, const void* x, const void* conv_w,
                           void* conv_state, void* y, void* stream) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0 && total_tokens > 0) return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0) return GDN_OK;
  if (cu_seqlens == nullptr || conv_w == nullptr || conv_state == nullptr) return GDN_ERR_INVALID_ARG;
  if (total_tokens > 0 && (x == nullptr || y == nullptr)) return GDN_ERR_INVALID_ARG;
  const int64_t es = dtype_size(dims->io_dtype);
  const int64_t C = qkv_features(dims);
  int64_t xel = 0, xbytes = 0, sel = 0, sbytes = 0;
  if (!mul_ok(total_tokens, C, &xel) || !mul_ok(xel, es, &xbytes)) return GDN_ERR_EXTENT;
  if (!mul_ok((int64_t)num_seqs, C * 3, &sel) || !mul_ok(sel, es, &sbytes)) return GDN_ERR_EXTENT;
  if (total_tokens > INT32_MAX - 64) return GDN_ERR_EXTENT;  // TMA row coordinates are int32
  if (!aligned16(cu_seqlens) || !aligned16(conv_w) || !aligned16(conv_state)) return GDN_ERR_ALIGN;
  if (total_tokens > 0 && (!aligned16(x) || !aligned16(y))) return GDN_ERR_ALIGN;
  if (total_tokens > 0) {
    const Range ry = range_of(y, xbytes);
    if (overlap(ry, range_of(x, xbytes)) || overlap(ry, range_of(conv_state, sbytes)) ||
        overlap(ry, range_of(conv_w, C * 4 * es)))
      return GDN_ERR_ALIAS;
  }
  if (overlap(range_of(conv_state, sbytes), range_of(x, xbytes)) ||
      overlap(range_of(conv_state, sbytes), range_of(conv_w, C * 4 * es)))
    return GDN_ERR_ALIAS;
  gdn::ConvArgs a{};
  a.cu_seqlens = cu_seqlens;
  a.N = num_seqs;
  a.T = total_tokens;
  a.C = (int32_t)C;
  a.x = x;
  a.conv_w = conv_w;
  a.conv_state = conv_state;
  a.y = y;
  return cuda_status(gdn::launch_conv(a, dims->io_dtype, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_decode_step(const gdn_dims* dims, int32_t batch, const void* mixed_qkv,
                           const void* a, const void* b, const float* decay_param,
                           const float* dt_bias, const void* conv_w, void* conv_state,
                           float* state, float* core_out, const void* z, const float* norm_w,
                           void* out, void* stream) {
  return decode_impl(dims, batch, 1, nullptr, batch, mixed_qkv, a, b, decay_param, dt_bias,
                     conv_w, conv_state, state, core_out, z, norm_w, out, stream);
}

gdn_status gdn_decode_multi(const gdn_dims* dims, int32_t batch, int32_t tokens,
                            const void* mixed_qkv, const void* a, const void* b,
                            const float* decay_param, const float* dt_bias, const void* conv_w,
                            void* conv_state, float* state, float* core_out, const void* z,
                            const float* norm_w, void* out, void* stream) {
  return decode_impl(dims, batch, tokens, nullptr, batch, mixed_qkv, a, b, decay_param, dt_bias,
                     conv_w, conv_state, state, core_out, z, norm_w, out, stream);
}

gdn_status gdn_decode_step_slots(const gdn_dims* dims, int32_t batch, const int32_t* state_slots,
                                 int32_t num_slots, const void* mixed_qkv, const void* a,
                                 const void* b, const float* decay_param, const float* dt_bias,
                                 const void* conv_w, void* conv_state, float* state,
                                 float* core_out, const void* z, const float* norm_w, void* out,
                                 void* stream) {
  if (state_slots == nullptr) return GDN_ERR_INVALID_ARG;
  return decode_impl(dims, batch, 1, state_slots, num_slots, mixed_qkv, a, b, decay_param,
                     dt_bias, conv_w, conv_state, state, core_out, z, norm_w, out, stream);
}

gdn_status gdn_prefill_chunked(const gdn_dims* dims, int32_t num_seqs, const int32_t* cu_seqlens,
                               int64_t total_tokens, const void* q, int64_t q_stride,
                               const void* k, int64_t k_stride, const void* v, int64_t v_stride,
                               const void* a, const void* b, const float* decay_param,
                               const float* dt_bias, int32_t flags, float* state,
                               float* core_out, const void* z, const float* norm_w, void* out,
                               void* workspace, int64_t workspace_bytes, void* stream) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0 && total_tokens > 0) return GDN_ERR_INVALID_ARG;
  if (num_seqs > kMaxGridY) return GDN_ERR_EXTENT;
  if (!prefill_flags_valid(flags)) return GDN_ERR_INVALID_ARG;
  if (num_seqs == 0) return GDN_OK;
  const bool pregate = (flags & GDN_GATES_PRECOMPUTED) != 0;
  if (!cu_seqlens || !state) return GDN_ERR_INVALID_ARG;
  if (total_tokens > 0) {
    if (!q || !k || !v || !a || !b) return GDN_ERR_INVALID_ARG;
    if (!pregate && (!decay_param || !dt_bias)) return GDN_ERR_INVALID_ARG;
    if (core_out == nullptr && z == nullptr) return GDN_ERR_INVALID_ARG;
    if (z != nullptr && (norm_w == nullptr || out == nullptr)) return GDN_ERR_INVALID_ARG;
  }
  const int64_t es = dtype_size(dims->io_dtype);
  const int64_t Hk = dims->n_k_heads, Hv = dims->n_v_heads, D = dims->head_dim;
  if (q_stride < Hk * D || k_stride < Hk * D || v_stride < Hv * D) return GDN_ERR_INVALID_ARG;
  if ((q_stride * es) % 16 || (k_stride * es) % 16 || (v_stride * es) % 16) return GDN_ERR_ALIGN;
  int64_t tmp = 0, state_bytes = 0;
  if (!mul_ok((int64_t)num_seqs * Hv, D * D * 4, &state_bytes)) return GDN_ERR_EXTENT;
  if (!mul_ok(total_tokens, (q_stride > v_stride ? q_stride : v_stride) + k_stride, &tmp))
    return GDN_ERR_EXTENT;
  if (!mul_ok(total_tokens, Hv * D * 4, &tmp)) return GDN_ERR_EXTENT;
  if (!aligned16(cu_seqlens) || !aligned16(state)) return GDN_ERR_ALIGN;
  if (total_tokens > 0) {
    const void* ptrs[] = {q, k, v, a, b};
    for (const void* ptr : ptrs)
      if (!aligned16(ptr)) return GDN_ERR_ALIGN;
    if ((core_out && !aligned16(core_out)) || (z && (!aligned16(z) || !aligned16(norm_w) || !aligned16(out))))
      return GDN_ERR_ALIGN;
    if (!pregate && (!aligned16(decay_param) || !aligned16(dt_bias))) return GDN_ERR_ALIGN;
  }
  const int64_t T = total_tokens;
  const int64_t gate_es = pregate ? 4 : es;
  const Range inputs[] = {
      range_of(q, T > 0 ? ((T - 1) * q_stride + Hk * D) * es : 0),
      range_of(k, T > 0 ? ((T - 1) * k_stride + Hk * D) * es : 0),
      range_of(v, T > 0 ? ((T - 1) * v_stride + Hv * D) * es : 0),
      range_of(a, T * Hv * gate_es),
      range_of(b, T * Hv * gate_es),
      range_of(z, z ? T * Hv * D * es : 0),
      range_of(cu_seqlens, ((int64_t)num_seqs + 1) * 4)};
  const Range rs = range_of(state, state_bytes);
  const Range ro = range_of(core_out, core_out ? T * Hv * D * 4 : 0);
  const Range ry = range_of(out, z ? T * Hv * D * es : 0);
  for (const Range& in : inputs) {
    if (overlap(rs, in) || overlap(ro, in) || overlap(ry, in)) return GDN_ERR_ALIAS;
  }
  if (overlap(rs, ro) || overlap(rs, ry) || overlap(ro, ry)) return GDN_ERR_ALIAS;
  int64_t ws_need = 0;
  st = gdn_prefill_workspace_size(dims, num_seqs, total_tokens, flags, &ws_need);
  if (st != GDN_OK) return st;
  const bool use_ws = workspace != nullptr && ws_need > 0 && total_tokens > 0;
  if (use_ws) {
    if (workspace_bytes < ws_need) return GDN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_ALIGN;
    const Range rw = range_of(workspace, ws_need);
    for (const Range& in : inputs)
      if (overlap(rw, in)) return GDN_ERR_ALIAS;
    if (overlap(rw, rs) || overlap(rw, ro) || overlap(rw, ry) ||
        overlap(rw, range_of(decay_param, pregate ? 0 : Hv * 4)) ||
        overlap(rw, range_of(dt_bias, pregate ? 0 : Hv * 4)) ||
        overlap(rw, range_of(norm_w, z ? D * 4 : 0)))
      return GDN_ERR_ALIAS;
  }
  gdn::PrefillArgs p{};
  p.cu_seqlens = cu_seqlens;
  p.N = num_seqs;
  p.T = total_tokens;
  p.q = q;
  p.q_stride = q_stride;
  p.k = k;
  p.k_stride = k_stride;
  p.v = v;
  p.v_stride = v_stride;
  p.a = a;
  p.b = b;
  p.decay_param = decay_param;
  p.dt_bias = dt_bias;
  p.flags = flags;
  p.state = state;
  p.core_out = core_out;
  p.z = z;
  p.norm_w = norm_w;
  p.out = out;
  p.Hk = (int32_t)Hk;
  p.Hv = (int32_t)Hv;
  p.rep = (int32_t)(Hv / Hk);
  p.map = dims->map;
  p.decay = dims->decay;
  p.l2_eps = dims->l2_eps;
  p.rms_eps = dims->rms_eps;
  p.scale = 1.0f / sqrtf((float)D);
  if (use_ws && gdn::prefill_cp_supported(p, dims->io_dtype, dims->head_dim))
    return cuda_status(gdn::launch_prefill_cp(p, workspace, static_cast<cudaStream_t>(stream)));
  return cuda_status(gdn::launch_prefill(p, dims->io_dtype, dims->head_dim,
                                         static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_prefill_workspace_size(const gdn_dims* dims, int32_t num_seqs,
                                      int64_t total_tokens, int32_t flags, int64_t* bytes) {
  if (bytes == nullptr) return GDN_ERR_INVALID_ARG;
  *bytes = 0;
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (num_seqs < 0 || total_tokens < 0) return GDN_ERR_INVALID_ARG;
  if (num_seqs > kMaxGridY) return GDN_ERR_EXTENT;
  if (!prefill_flags_valid(flags)) return GDN_ERR_INVALID_ARG;
  if (dims->head_dim != 128 || dims->io_dtype != GDN_BF16 || (flags & GDN_PREFILL_CUDA_CORES) ||
      dims->n_v_heads > 16 * dims->n_k_heads || num_seqs == 0 || total_tokens == 0)
    return GDN_OK;
  // (T + 63 N) / 64 chunk slots of 25 KB per V head and 16 KB per K head,
  // plus the chunk index, plus T Hv 512 bytes for few (V head, sequence)
  // pairs (bounded here by 512 bytes per chunk-slot token and V head)
  int64_t tmp = 0;
  if (!mul_ok(total_tokens + 63 * (int64_t)num_seqs,
              (int64_t)dims->n_v_heads * 912 + (int64_t)dims->n_k_heads * 256 + 400, &tmp))
    return GDN_ERR_EXTENT;
  *bytes = gdn::prefill_cp_workspace_bytes(num_seqs, total_tokens, dims->n_k_heads,
                                           dims->n_v_heads);
  return GDN_OK;
}

gdn_status gdn_gated_rmsnorm(const gdn_dims* dims, int64_t rows, const float* o, const void* z,
                             const float* norm_w, void* y, void* stream) {
  gdn_status st = check_dims(dims);
  if (st != GDN_OK) return st;
  if (rows < 0) return GDN_ERR_INVALID_ARG;
  if (rows == 0) return GDN_OK;
  if (!o || !z || !norm_w || !y) return GDN_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(z) || !aligned16(norm_w) || !aligned16(y)) return GDN_ERR_ALIGN;
  const int64_t es = dtype_size(dims->io_dtype), D = dims->head_dim;
  int64_t el = 0;
  if (!mul_ok(rows, D * 4, &el)) return GDN_ERR_EXTENT;
  if ((rows + 7) / 8 > INT32_MAX) return GDN_ERR_EXTENT;
  const Range ry = range_of(y, rows * D * es);
  if (overlap(ry, range_of(o, rows * D * 4)) || overlap(ry, range_of(z, rows * D * es)) ||
      overlap(ry, range_of(norm_w, D * 4)))
    return GDN_ERR_ALIAS;
  gdn::RmsNormArgs p{};
  p.rows = rows;
  p.o = o;
  p.z = z;
  p.norm_w = norm_w;
  p.y = y;
  p.eps = dims->rms_eps;
  return cuda_status(
      gdn::launch_rmsnorm(p, dims->io_dtype, dims->head_dim, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_linear_workspace_size(int32_t M, int32_t N, int32_t K, int64_t* bytes) {
  if (bytes == nullptr) return GDN_ERR_INVALID_ARG;
  *bytes = 0;
  if (M < 1 || M > 128 || N < 64 || N % 64 != 0 || K < 64 || K % 64 != 0) return GDN_ERR_INVALID_ARG;
  *bytes = gdn::linear_workspace_bytes(M, N, K);
  return GDN_OK;
}

gdn_status gdn_linear(int32_t M, int32_t N, int32_t K, const void* x, int64_t x_stride, const void* w,
                      const float* bias, void* y, int64_t y_stride, void* workspace,
                      int64_t workspace_bytes, void* stream) {
  int64_t need = 0;
  gdn_status st = gdn_linear_workspace_size(M, N, K, &need);
  if (st != GDN_OK) return st;
  if (!x || !w || !y || (need > 0 && !workspace)) return GDN_ERR_INVALID_ARG;
  if (x_stride < K || x_stride % 8 != 0 || y_stride < N || y_stride % 8 != 0) return GDN_ERR_INVALID_ARG;
  if (workspace_bytes < need) return GDN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u)) ||
      (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)))
    return GDN_ERR_ALIGN;
  const Range ry = range_of(y, ((int64_t)(M - 1) * y_stride + N) * 2), rw = range_of(workspace, need);
  const Range ins[] = {range_of(x, ((int64_t)(M - 1) * x_stride + K) * 2), range_of(w, (int64_t)N * K * 2),
                       range_of(bias, bias ? (int64_t)N * 4 : 0), rw};
  for (const Range& in : ins)
    if (overlap(ry, in)) return GDN_ERR_ALIAS;
  for (int i = 0; i < 3; ++i)
    if (overlap(rw, ins[i])) return GDN_ERR_ALIAS;
  if (!gdn::linear_supported()) return GDN_ERR_UNSUPPORTED;
  gdn::LinearArgs p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.bias = bias;
  p.route.count = 1;
  p.route.start[0] = 0;
  p.route.start[1] = N;
  p.route.ld[0] = y_stride;
  p.route.dst[0] = y;
  return cuda_status(gdn::launch_linear(p, x, x_stride, w, workspace, static_cast<cudaStream_t>(stream)));
}

namespace {

struct LayerLayout {
  int64_t C, vw, n_in;  // qkv features, value width Hv D, padded input-projection rows
  size_t off_qkv, off_z, off_b, off_a, off_y, off_lin, total;
};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

gdn_status layer_layout(const gdn_dims* d, int32_t hidden, int32_t batch, LayerLayout* l) {
  gdn_status st = check_dims(d);
  if (st != GDN_OK) return st;
  if (d->io_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (hidden < 64 || hidden % 64 != 0 || batch < 1 || batch > 128) return GDN_ERR_INVALID_ARG;
  const int64_t Hv = d->n_v_heads, D = d->head_dim;
  if ((Hv * D) % 64 != 0 || Hv % 8 != 0) return GDN_ERR_UNSUPPORTED;
  l->C = qkv_features(d);
  l->vw = Hv * D;
  l->n_in = (l->C + l->vw + 2 * Hv + 63) / 64 * 64;
  if (l->n_in > INT32_MAX / 2 || (int64_t)hidden * l->n_in > INT32_MAX) return GDN_ERR_EXTENT;
  size_t off = 0;
  l->off_qkv = off;
  off = align256(off + (size_t)batch * l->C * 2);
  l->off_z = off;
  off = align256(off + (size_t)batch * l->vw * 2);
  l->off_b = off;
  off = align256(off + (size_t)batch * Hv * 2);
  l->off_a = off;
  off = align256(off + (size_t)batch * Hv * 2);
  l->off_y = off;
  off = align256(off + (size_t)batch * l->vw * 2);
  l->off_lin = off;
  const int64_t lin_in = gdn::linear_workspace_bytes(batch, (int32_t)l->n_in, hidden);
  const int64_t lin_out = gdn::linear_workspace_bytes(batch, hidden, (int32_t)l->vw);
  l->total = off + (size_t)(lin_in > lin_out ? lin_in : lin_out);
  return GDN_OK;
}

}  // namespace

gdn_status gdn_decode_layer_workspace_size(const gdn_dims* dims, int32_t hidden, int32_t batch,
                                           int64_t* bytes) {
  if (bytes == nullptr) return GDN_ERR_INVALID_ARG;
  *bytes = 0;
  LayerLayout l{};
  gdn_status st = layer_layout(dims, hidden, batch, &l);
  if (st != GDN_OK) return st;
  *bytes = (int64_t)l.total;
  return GDN_OK;
}

gdn_status gdn_decode_layer(const gdn_dims* dims, int32_t hidden, int32_t batch, const void* x,
                            const gdn_layer_weights* w, void* conv_state, float* state, void* y,
                            void* workspace, int64_t workspace_bytes, void* stream) {
  LayerLayout l{};
  gdn_status st = layer_layout(dims, hidden, batch, &l);
  if (st != GDN_OK) return st;
  if (!x || !w || !y || !workspace || !w->w_in || !w->w_out) return GDN_ERR_INVALID_ARG;
  if (workspace_bytes < (int64_t)l.total) return GDN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(w->w_in) || !aligned16(w->w_out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      (w->b_in && (reinterpret_cast<uintptr_t>(w->b_in) & 3u)) ||
      (w->b_out && (reinterpret_cast<uintptr_t>(w->b_out) & 3u)))
    return GDN_ERR_ALIGN;
  const int64_t Hv = dims->n_v_heads, D = dims->head_dim;
  // the caller's buffers against the workspace and each other
  const Range rws = range_of(workspace, (int64_t)l.total);
  const Range ry = range_of(y, (int64_t)batch * hidden * 2);
  const Range rx = range_of(x, (int64_t)batch * hidden * 2);
  const Range rs = range_of(state, (int64_t)batch * Hv * D * D * 4);
  const Range rc = range_of(conv_state, (int64_t)batch * l.C * 3 * 2);
  const Range weights_r[] = {range_of(w->w_in, l.n_in * hidden * 2), range_of(w->b_in, w->b_in ? l.n_in * 4 : 0),
                             range_of(w->w_out, (int64_t)hidden * l.vw * 2),
                             range_of(w->b_out, w->b_out ? (int64_t)hidden * 4 : 0),
                             range_of(w->conv_w, l.C * 4 * 2), range_of(w->decay_param, Hv * 4),
                             range_of(w->dt_bias, Hv * 4), range_of(w->norm_w, D * 4)};
  for (const Range& a : {rws, ry, rs, rc}) {
    if (overlap(a, rx)) return GDN_ERR_ALIAS;
    for (const Range& b : weights_r)
      if (overlap(a, b)) return GDN_ERR_ALIAS;
  }
  if (overlap(rws, ry) || overlap(rws, rs) || overlap(rws, rc) || overlap(ry, rs) || overlap(ry, rc))
    return GDN_ERR_ALIAS;
  if (!gdn::linear_supported()) return GDN_ERR_UNSUPPORTED;
  char* ws = static_cast<char*>(workspace);
  void *qkv = ws + l.off_qkv, *z = ws + l.off_z, *bb = ws + l.off_b, *aa = ws + l.off_a, *yc = ws + l.off_y;
  void* lin = ws + l.off_lin;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // (1) the fused input projection: qkv | z | b | a
  gdn::LinearArgs pin{};
  pin.M = batch;
  pin.N = (int32_t)l.n_in;
  pin.K = hidden;
  pin.bias = w->b_in;
  pin.route.count = 4;
  pin.route.start[0] = 0;
  pin.route.start[1] = (int32_t)l.C;
  pin.route.start[2] = (int32_t)(l.C + l.vw);
  pin.route.start[3] = (int32_t)(l.C + l.vw + Hv);
  pin.route.start[4] = (int32_t)(l.C + l.vw + 2 * Hv);
  pin.route.ld[0] = l.C;
  pin.route.ld[1] = l.vw;
  pin.route.ld[2] = Hv;
  pin.route.ld[3] = Hv;
  pin.route.dst[0] = qkv;
  pin.route.dst[1] = z;
  pin.route.dst[2] = bb;
  pin.route.dst[3] = aa;
  st = cuda_status(gdn::launch_linear(pin, x, hidden, w->w_in, lin, s));
  if (st != GDN_OK) return st;
  // (2) the core with its fused gated RMSNorm, launched to overlap (1)'s
  // tail: (1) writes only the projections in the workspace, so the state
  // rows stream in while it drains and the activations are read after it
  // has completed
  st = decode_impl(dims, batch, 1, nullptr, batch, qkv, aa, bb, w->decay_param, w->dt_bias, w->conv_w,
                   conv_state, state, nullptr, z, w->norm_w, yc, stream, true);
  if (st != GDN_OK) return st;
  // (3) the output projection, overlapping (2)'s tail the same way: its
  // weight tiles load while (2) drains, its input after (2) has completed
  gdn::LinearArgs pout{};
  pout.overlap_prev = 1;
  pout.M = batch;
  pout.N = hidden;
  pout.K = (int32_t)l.vw;
  pout.bias = w->b_out;
  pout.route.count = 1;
  pout.route.start[0] = 0;
  pout.route.start[1] = hidden;
  pout.route.ld[0] = hidden;
  pout.route.dst[0] = y;
  return cuda_status(gdn::launch_linear(pout, yc, l.vw, w->w_out, lin, s));
}

gdn_status gdn_selftest_wait_timeout(int64_t limit_ns, int32_t* gave_up, void* stream) {
  if (gave_up == nullptr || limit_ns < 1000 || limit_ns > 10000000000LL) return GDN_ERR_INVALID_ARG;
  return cuda_status(gdn::launch_wait_timeout((uint64_t)limit_ns, gave_up, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_device_error(int32_t* status, int32_t clear) {
  if (status == nullptr) return GDN_ERR_INVALID_ARG;
  *status = GDN_OK;
  cudaError_t (*readers[])(int32_t*, bool) = {gdn::read_error_decode, gdn::read_error_decode_mt,
                                               gdn::read_error_conv,
                                               gdn::read_error_rmsnorm, gdn::read_error_prefill,
                                               gdn::read_error_prefill_tc,
                                               gdn::read_error_prefill_cp, gdn::read_error_diag,
                                               gdn::read_error_linear};
  for (auto rd : readers) {
    int32_t v = 0;
    if (rd(&v, clear != 0) != cudaSuccess) return GDN_ERR_CUDA;
    if (v != GDN_OK && *status == GDN_OK) *status = v;
  }
  return GDN_OK;
}

}  // extern "C"
