/*
 * gdn.h -- C ABI of the GB300 gated delta-net core library (libgdn.so).
 *
 * The library computes the gated delta-net linear-attention core (the
 * Qwen3-Next / Qwen3.5 recurrence) on one sm_103a GPU:
 *
 *   per token, per V head h reading K head kh (Grouped: kh = h / (Hv/Hk),
 *   Tiled: kh = h % Hk), with the state S[h][j][i] (value row j, key col i):
 *       S  *= exp(g_h)
 *       pred = S k            d = beta_h (v - pred)
 *       S  += d k^T           o = S q / sqrt(D)
 *   -- ferrox-core 0.24.0 src/gdn.rs, module docs (the six-line formula),
 *      `HeadMap`, `delta_step`; ferrum-kernels gated_delta_attention_tests.rs
 *      `cpu_segment`.
 *
 * Conventions shared by every call:
 *  - Every pointer is a DEVICE pointer the caller owns (allocated with
 *    cudaMalloc or by a framework allocator); the library never allocates,
 *    frees or retains one past the call. The one exception is noted at
 *    gdn_decode_step: its activations and outputs may also be mapped pinned
 *    host memory (gdn_host_pointer). All work is enqueued on `stream`
 *    (a cudaStream_t; NULL = the legacy default stream) and is asynchronous.
 *  - Arguments are validated on the host before anything is enqueued; on an
 *    error nothing is launched and the status says why. A failed launch
 *    returns GDN_ERR_CUDA.
 *  - Tensors are dense row-major with the innermost dimension last, and every
 *    pointer must be 16-byte aligned.
 *  - io dtype (gdn_dims.io_dtype) is the storage type of the activations,
 *    the conv weight and the conv state; the delta state, core outputs,
 *    decay parameters, dt_bias and the norm weight are always fp32.
 *  - Supported shapes: head_dim (Dk = Dv = D) in {32, 64, 96, 128};
 *    n_v_heads a multiple of n_k_heads; conv kernel width 4 (3-wide state).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* null pointer, bad enum, bad dims */
  GDN_ERR_EXTENT = 2,      /* a size product overflows the launch/index range */
  GDN_ERR_UNSUPPORTED = 3, /* valid but not implemented (e.g. head_dim 80) */
  GDN_ERR_ALIAS = 4,       /* an output overlaps an input it must not */
  GDN_ERR_ALIGN = 5,       /* pointer or stride not 16-byte aligned */
  GDN_ERR_CUDA = 6,        /* the CUDA runtime reported an error */
  GDN_ERR_TIMEOUT = 7      /* a device-side bounded wait gave up */
} gdn_status;

/* V head -> K head map (gdn.rs `HeadMap`; enum values as the Metal test's
 * params use them: 0 = grouped, 1 = interleaved/tiled). */
typedef enum gdn_head_map { GDN_MAP_GROUPED = 0, GDN_MAP_TILED = 1 } gdn_head_map;

/* Decay parameterisation (gated_delta_attention_tests.rs, `cpu_segment`
 * gate lines): LOG_RATE: rate_h = -exp(decay_param[h]) (decay_param = A_log);
 * NEGATIVE_RATE: rate_h = decay_param[h] (already negative).
 * Then g = rate_h * softplus(a + dt_bias[h]), beta = sigmoid(b). */
typedef enum gdn_decay { GDN_DECAY_LOG_RATE = 0, GDN_DECAY_NEGATIVE_RATE = 1 } gdn_decay;

typedef enum gdn_dtype { GDN_F16 = 0, GDN_BF16 = 1, GDN_F32 = 2 } gdn_dtype;

/* gdn_prefill_chunked flags */
enum {
  GDN_QK_PRENORMALIZED = 1,  /* q and k are already l2-normalised: skip it */
  GDN_GATES_PRECOMPUTED = 2, /* a holds g and b holds beta, both fp32 [T][Hv] */
  GDN_PREFILL_CUDA_CORES = 4, /* use the fp32 CUDA-core chunk kernel even where a
                                 tensor-core one applies (head_dim 128, f16/bf16) */
  /* On the chunk-parallel path, the carry kernel: by default the sliced one
     (four CTAs per V head and sequence) when 4 Hv N is at most two waves of
     the device's SMs, else one CTA per V head and sequence. These force
     either (not both); other paths ignore them. */
  GDN_PREFILL_CARRY_WHOLE = 8,
  GDN_PREFILL_CARRY_SLICED = 16
};

typedef struct gdn_dims {
  int32_t n_k_heads; /* Hk >= 1 */
  int32_t n_v_heads; /* Hv, a multiple of Hk */
  int32_t head_dim;  /* D = Dk = Dv in {32, 64, 96, 128} */
  int32_t map;       /* gdn_head_map */
  int32_t decay;     /* gdn_decay */
  int32_t io_dtype;  /* gdn_dtype */
  float l2_eps;      /* q/k normalisation: x * (sum x^2 + l2_eps)^(-1/2); 1e-6 */
  float rms_eps;     /* gated RMSNorm: o * (mean o^2 + rms_eps)^(-1/2); 1e-6 */
} gdn_dims;

/* Human-readable name of a status code (static storage, never NULL). */
const char* gdn_status_string(int32_t status);

/* ABI version: major * 10000 + minor * 100 + patch. 0.3.0 added
 * gdn_decode_multi and gdn_decode_step_slots; 0.4.0 gdn_linear,
 * gdn_decode_layer and gdn_host_pointer. */
int32_t gdn_version(void);

/* Channels of the packed pre-conv activation: C = 2*Hk*D + Hv*D, laid out
 * [q (Hk*D) | k (Hk*D) | v (Hv*D)] (gated_delta_attention_tests.rs
 * `cpu_segment` split; libmir-metal decode/mod.rs `split_qkv`). -1 if dims
 * is invalid. */
int64_t gdn_qkv_features(const gdn_dims* dims);

/*
 * Causal depthwise conv1d (kernel 4) + SiLU over a packed batch of
 * variable-length sequences, with a rolling 3-wide conv state per sequence.
 * -- gated_delta_attention_tests.rs `cpu_segment` conv loop and conv-state
 *    update; libmir-metal decode/mod.rs `convolve`.
 *
 *   y[t][c] = silu( sum_{j=0..3} conv_w[c][j] * xh[t+j-3][c] ),
 *   xh[tau] = x[tau] inside the sequence, conv_state[n][c][3+tau'] for the
 *   three positions before its first token (tau' = -3..-1, oldest first).
 *   Afterwards conv_state[n][c][0..2] holds the last three raw inputs of
 *   sequence n (a bit copy; older entries shift in when the sequence has
 *   fewer than three tokens).
 *
 * num_seqs    N >= 0 sequences.
 * total_tokens  0 <= T <= 2^31 - 65 (GDN_ERR_EXTENT beyond).
 * cu_seqlens  device int32 [N+1], cu[0] = 0, non-decreasing, cu[N] =
 *             total_tokens; sequence n owns tokens [cu[n], cu[n+1]). Values
 *             outside [0, total_tokens] are clamped on the device.
 * x           [total_tokens][C] io dtype (C = gdn_qkv_features).
 * conv_w      [C][4] io dtype; tap 3 multiplies the current token; no bias.
 * conv_state  [N][C][3] io dtype, updated in place.
 * y           [total_tokens][C] io dtype; must not overlap x or conv_state.
 */
gdn_status gdn_conv_update(const gdn_dims* dims, int32_t num_seqs, const int32_t* cu_seqlens,
                           int64_t total_tokens, const void* x, const void* conv_w,
                           void* conv_state, void* y, void* stream);

/*
 * One decode token for each of `batch` sequences, fully fused: conv + SiLU
 * on the packed pre-conv activation, split q|k|v, l2-normalise q and k per
 * K head (q also scaled by 1/sqrt(D)), gates, the delta-rule step on the
 * fp32 state in place, and optionally the gated RMSNorm of the output.
 * -- gdn.rs `delta_step` (the step), gated_delta_attention_tests.rs
 *    `cpu_segment` (conv, norm, gates, gated norm), libmir-metal
 *    decode/mod.rs `build` (one decode layer: convolve, split, recurrence,
 *    rms_norm, gate).
 *
 * batch        B >= 0 sequences (one token each), B <= 65535.
 * mixed_qkv    [B][C] io dtype, pre-conv.
 * a, b         [B][Hv] io dtype: raw decay input (a) and raw beta input (b).
 * decay_param  [Hv] fp32: A_log (LOG_RATE) or the negative rate.
 * dt_bias      [Hv] fp32.
 * conv_w       [C][4] io dtype.
 * conv_state   [B][C][3] io dtype, in place.
 * state        [B][Hv][D][D] fp32 S[b][h][j][i], in place.
 * core_out     [B][Hv][D] fp32 core output o, or NULL.
 * z            [B][Hv][D] io dtype output-gate input, or NULL (no norm).
 * norm_w       [D] fp32 RMSNorm weight (shared by all heads); needed with z.
 * out          [B][Hv][D] io dtype gated-RMSNorm output; needed with z.
 * At least one of core_out and (z, out) must be given. Hv/Hk <= 16.
 * mixed_qkv, a, b, z, core_out and out may be device addresses of mapped
 * pinned host memory (gdn_host_pointer): the kernel then reads the
 * activations and writes the outputs in place over the host link, with no
 * separate copy (on a coherent host link such as Grace's, the cheapest way
 * to feed one serving step from the host). Every other pointer, of this and
 * every other call, must be device memory.
 */
gdn_status gdn_decode_step(const gdn_dims* dims, int32_t batch, const void* mixed_qkv,
                           const void* a, const void* b, const float* decay_param,
                           const float* dt_bias, const void* conv_w, void* conv_state,
                           float* state, float* core_out, const void* z, const float* norm_w,
                           void* out, void* stream);

/*
 * Multi-token decode: `tokens` consecutive tokens of each of `batch`
 * sequences in one call, with the state of each (sequence, V head) read
 * from and written to memory once for all of them instead of once per
 * token (speculative or multi-token-prediction decode). The result is that
 * of `tokens` successive gdn_decode_step calls, token 0 first, each fed the
 * row of every activation that belongs to that token; the arithmetic of each
 * token is ordered as in gdn_decode_step, so the two agree bit for bit.
 * The pages' decode step is one token (gdn.rs `delta_step`); applying it to
 * a block of tokens with the state held on chip is this library's own
 * reading of a decode over several tokens.
 *
 * tokens       T in 1..8 (T = 1 is gdn_decode_step); T < 1 is
 *              GDN_ERR_INVALID_ARG, T > 8 GDN_ERR_UNSUPPORTED.
 * mixed_qkv    [B][T][C] io dtype, pre-conv (row b*T + t is token t of
 *              sequence b).
 * a, b         [B][T][Hv] io dtype.
 * core_out     [B][T][Hv][D] fp32, or NULL.
 * z, out       [B][T][Hv][D] io dtype (fused gated RMSNorm), or NULL.
 * conv_state   [B][C][3], state [B][Hv][D][D]: in place, as in
 *              gdn_decode_step; afterwards they hold the state after token
 *              T-1.
 * Every other argument, and every error, is as in gdn_decode_step, except
 * that T > 1 takes at most 8 V heads per K head (GDN_ERR_UNSUPPORTED
 * beyond).
 */
gdn_status gdn_decode_multi(const gdn_dims* dims, int32_t batch, int32_t tokens,
                            const void* mixed_qkv, const void* a, const void* b,
                            const float* decay_param, const float* dt_bias, const void* conv_w,
                            void* conv_state, float* state, float* core_out, const void* z,
                            const float* norm_w, void* out, void* stream);

/*
 * gdn_decode_step over a pool of state slots: batch row b reads and updates
 * state[state_slots[b]] and conv_state[state_slots[b]] of a pool of
 * num_slots sequences, so a serving loop can batch whichever sequences are
 * live without gathering their states. The pages declare a batch submodule
 * of the decode layer (libmir-metal decode/mod.rs, `mod batch`) without
 * showing it; this indirection is this library's own reading of it.
 *
 * state_slots  device int32 [B]. A negative entry marks a padded row: it
 *              touches no state or conv state, its core_out row is zero and
 *              its out row is the gated norm of a zero row (zero for finite
 *              z). An entry >= num_slots is treated the same and also
 *              records GDN_ERR_EXTENT in the device error word
 *              (gdn_device_error). Two rows naming the same slot is a caller
 *              error: both update that state at once and the result is
 *              unspecified (no fault).
 * num_slots    P >= 0 slots in the pool.
 * conv_state   [P][C][3] io dtype, in place.
 * state        [P][Hv][D][D] fp32, in place.
 * Every other argument is indexed by the batch row, exactly as in
 * gdn_decode_step, with the same errors; state_slots NULL is
 * GDN_ERR_INVALID_ARG.
 */
gdn_status gdn_decode_step_slots(const gdn_dims* dims, int32_t batch, const int32_t* state_slots,
                                 int32_t num_slots, const void* mixed_qkv, const void* a,
                                 const void* b, const float* decay_param, const float* dt_bias,
                                 const void* conv_w, void* conv_state, float* state,
                                 float* core_out, const void* z, const float* norm_w, void* out,
                                 void* stream);

/*
 * Chunked prefill: the same recurrence as gdn_decode_step summed chunk-wise
 * (chunk 64, UT/WY form) over a packed batch of variable-length sequences,
 * each continuing from its own fp32 state (in place). q, k, v are the
 * post-conv activations (e.g. slices of gdn_conv_update's y).
 * -- gdn.rs module docs ("the same recurrence in a different summation
 *    order"); gated_delta_attention_tests.rs `run_chunked_core` (the six
 *    chunk stages: K gram, (I+A)^-1, U/W, QK^T, carry, output) and
 *    `chunked_c64_matches_recurrent_oracle_and_non_aligned_state_continuity`.
 *
 * cu_seqlens   device int32 [N+1] as for gdn_conv_update.
 * q, k         token t, K head kh, column i at q[t*q_stride + kh*D + i]
 *              (io dtype); strides in elements, multiples of 8.
 * v            token t, V head h, column j at v[t*v_stride + h*D + j].
 * a, b         [T][Hv] io dtype raw gate inputs, or with
 *              GDN_GATES_PRECOMPUTED fp32 g and beta.
 * decay_param, dt_bias  [Hv] fp32 (ignored with GDN_GATES_PRECOMPUTED).
 * flags        GDN_QK_PRENORMALIZED | GDN_GATES_PRECOMPUTED | GDN_PREFILL_CUDA_CORES.
 * state        [N][Hv][D][D] fp32, in place (initial state = its contents).
 * core_out     [T][Hv][D] fp32 core output, or NULL.
 * z, norm_w, out  optional fused gated RMSNorm as in gdn_decode_step.
 * workspace    device scratch of at least gdn_prefill_workspace_size bytes,
 *              256-byte aligned, owned by the caller, not overlapping any
 *              other argument; its contents need no initialisation and are
 *              garbage afterwards. May be NULL (workspace_bytes ignored).
 *
 * Which kernels run (all on the given stream):
 *  - head_dim 128, bf16, Hv/Hk <= 16, a workspace: the chunk-parallel
 *    tensor-core path.
 *    Every chunk's state-free factors (the K and QK grams, (I+A)^-1 diag(beta),
 *    the masked decayed QK^T) are computed at once into the workspace, then
 *    one CTA per (V head, sequence) carries the state through its chunks with
 *    the fp32 state as a TMEM accumulator; products that carry the state use
 *    bf16 hi+lo splits of their fp32 factors.
 *  - head_dim 128, f16/bf16, no workspace (or f16): a single-pass tensor-core
 *    kernel (one cluster of four CTAs per V head and sequence, every chunk
 *    stage in sequence; tf32 hi+lo splits for the state-carrying products).
 *  - other head dims, fp32 activations, or GDN_PREFILL_CUDA_CORES: fp32 CUDA
 *    cores.
 */
gdn_status gdn_prefill_chunked(const gdn_dims* dims, int32_t num_seqs, const int32_t* cu_seqlens,
                               int64_t total_tokens, const void* q, int64_t q_stride,
                               const void* k, int64_t k_stride, const void* v, int64_t v_stride,
                               const void* a, const void* b, const float* decay_param,
                               const float* dt_bias, int32_t flags, float* state,
                               float* core_out, const void* z, const float* norm_w, void* out,
                               void* workspace, int64_t workspace_bytes, void* stream);

/*
 * Bytes of workspace gdn_prefill_chunked can use for these sizes and flags
 * (0 when no workspace path applies: head_dim != 128, io dtype not bf16,
 * more than 16 V heads per K head, or GDN_PREFILL_CUDA_CORES): per 64-token chunk slot ((T + 63 N) / 64 of
 * them) 25 KB per V head and 16 KB per K head, plus 4 (N + 1) bytes rounded
 * up to 1 KB; and where Hv N <= 64 (the sliced carry), T Hv 512 bytes more
 * at a 256-byte boundary, for the fp32 core output that its separate gated
 * norm reads when core_out is NULL. Writes the size to *bytes;
 * GDN_ERR_INVALID_ARG / GDN_ERR_EXTENT for invalid dims or sizes.
 */
gdn_status gdn_prefill_workspace_size(const gdn_dims* dims, int32_t num_seqs,
                                      int64_t total_tokens, int32_t flags, int64_t* bytes);

/* Size of the static device scratch behind gdn_prefill_chunked_static. */
#define GDN_STATIC_SCRATCH_BYTES (160u << 20)

/*
 * gdn_prefill_chunked without a workspace argument that still takes the
 * chunk-parallel path: it runs over a scratch buffer of
 * GDN_STATIC_SCRATCH_BYTES that the library reserves statically in each
 * CUDA context (when the library's kernels first load there), so the call
 * allocates nothing. Its address is looked up in the calling thread's
 * current context on every call, so it stays valid across cudaDeviceReset
 * and under several contexts on one device. The pages have no counterpart
 * to this call; it serves callers that cannot hand out device memory.
 *
 * Arguments, results and errors are those of gdn_prefill_chunked, plus:
 *  - GDN_ERR_EXTENT, checked first, when gdn_prefill_workspace_size for
 *    these sizes exceeds GDN_STATIC_SCRATCH_BYTES (e.g. more than 5,025
 *    tokens in one sequence at Hk=16, Hv=32; 2,683 at Hk=16, Hv=64);
 *  - where no workspace path applies (f16, head_dim != 128,
 *    GDN_PREFILL_CUDA_CORES) it is gdn_prefill_chunked with workspace NULL.
 *
 * Races: the scratch is one buffer per context shared by every call of this
 * function. Two calls whose executions can overlap in time (on different
 * streams without an event between them, or issued from host threads
 * without ordering) write it concurrently and corrupt each other's output
 * and state. Issue them on one stream or order them with events.
 */
gdn_status gdn_prefill_chunked_static(const gdn_dims* dims, int32_t num_seqs,
                                      const int32_t* cu_seqlens, int64_t total_tokens,
                                      const void* q, int64_t q_stride, const void* k,
                                      int64_t k_stride, const void* v, int64_t v_stride,
                                      const void* a, const void* b, const float* decay_param,
                                      const float* dt_bias, int32_t flags, float* state,
                                      float* core_out, const void* z, const float* norm_w,
                                      void* out, void* stream);

/*
 * Gated RMSNorm over rows of D: y = o * (mean_j o_j^2 + rms_eps)^(-1/2)
 * * norm_w[j] * silu(z[j]), computed in fp32 and rounded once to io dtype.
 * -- gated_delta_attention_tests.rs `cpu_segment` output loop.
 *
 * rows   >= 0 (e.g. T * Hv).
 * o      [rows][D] fp32;  z [rows][D] io dtype;  norm_w [D] fp32;
 * y      [rows][D] io dtype, must not overlap o or z.
 */
gdn_status gdn_gated_rmsnorm(const gdn_dims* dims, int64_t rows, const float* o, const void* z,
                             const float* norm_w, void* y, void* stream);

/*
 * Linear layer y = x W^T (+ bias), bf16 in and out, fp32 accumulation, on
 * the tensor cores: the projections around the core in a decode layer.
 * -- libmir-metal decode/mod.rs, `Linear::forward` (matmul, then bias) and
 *    `build` (the qkv, gate, beta, alpha and output projections).
 *
 * M            rows of x and y, 1 <= M <= 128 (the decode batch).
 * N, K         output and input features, positive multiples of 64.
 * x            [M][x_stride] bf16, row m at x + m * x_stride (x_stride >= K,
 *              a multiple of 8); 16-byte aligned.
 * w            [N][K] bf16 row-major (one row per output feature); 16-byte
 *              aligned.
 * bias         [N] fp32 added before the one rounding to bf16, or NULL.
 * y            [M][y_stride] bf16 (y_stride >= N, a multiple of 8); must not
 *              overlap x, w, bias or the workspace.
 * workspace    device scratch of gdn_linear_workspace_size bytes, 256-byte
 *              aligned; may be NULL when that size is 0 (it is 0 for every
 *              shape this version accepts: narrow outputs split K over a
 *              thread-block cluster that adds the partial sums in its own
 *              shared memory, in split order).
 *
 * Errors: GDN_ERR_INVALID_ARG (sizes, NULL pointers, strides),
 * GDN_ERR_ALIGN, GDN_ERR_ALIAS, GDN_ERR_UNSUPPORTED (no TMA encoder in the
 * driver), GDN_ERR_CUDA.
 */
gdn_status gdn_linear(int32_t M, int32_t N, int32_t K, const void* x, int64_t x_stride,
                      const void* w, const float* bias, void* y, int64_t y_stride,
                      void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes gdn_linear needs for M, N, K (0 in this version: the K
 * splits of narrow outputs, at most min(8, K / 128), are summed in shared
 * memory; the result does not depend on the order in which they finish). */
gdn_status gdn_linear_workspace_size(int32_t M, int32_t N, int32_t K, int64_t* bytes);

/*
 * Weights of one layer for gdn_decode_layer. With C = (2 Hk + Hv) D and
 * N_in = C + Hv D + 2 Hv rounded up to a multiple of 64:
 * w_in         [N_in][hidden] bf16: rows 0..C-1 the qkv projection, the next
 *              Hv D rows the gate (z) projection, then Hv rows the beta (b)
 *              and Hv rows the alpha (a) projection; padding rows unused.
 * b_in         [N_in] fp32 bias of those rows, or NULL.
 * w_out        [hidden][Hv D] bf16, the output projection; b_out [hidden]
 *              fp32 or NULL.
 * conv_w, decay_param, dt_bias, norm_w  as in gdn_decode_step.
 */
typedef struct gdn_layer_weights {
  const void* w_in;
  const float* b_in;
  const void* w_out;
  const float* b_out;
  const void* conv_w;
  const float* decay_param;
  const float* dt_bias;
  const float* norm_w;
} gdn_layer_weights;

/*
 * One decode step of a whole gated delta-net layer for a batch of
 * sequences, one token each: the fused input projection (qkv | z | b | a in
 * one gdn_linear launch), gdn_decode_step with its fused gated RMSNorm, and
 * the output projection. Three kernel launches; the second and third start
 * while their predecessor inside the call drains (programmatic dependent
 * launch), reading only what that predecessor does not write until it has
 * completed.
 * -- libmir-metal decode/mod.rs, `build`: qkv projection -> `convolve` ->
 *    `split_qkv` -> gate/beta/alpha projections -> `recurrence` ->
 *    `rms_norm` -> `precise_gate` -> output projection.
 *
 * dims         io_dtype GDN_BF16; Hv D a multiple of 64; Hv/Hk <= 16.
 * hidden       model width, a positive multiple of 64.
 * batch        1 <= batch <= 128.
 * x            [batch][hidden] bf16 layer input.
 * conv_state   [batch][C][3] bf16, state [batch][Hv][D][D] fp32, in place.
 * y            [batch][hidden] bf16 layer output.
 * workspace    gdn_decode_layer_workspace_size bytes, 256-byte aligned, not
 *              overlapping any other argument; contents irrelevant.
 * Errors as gdn_linear and gdn_decode_step.
 */
gdn_status gdn_decode_layer(const gdn_dims* dims, int32_t hidden, int32_t batch, const void* x,
                            const gdn_layer_weights* weights, void* conv_state, float* state,
                            void* y, void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes of gdn_decode_layer: the projections' bf16 outputs (qkv,
 * z, b, a and the gated core output, [batch] rows each) and gdn_linear's
 * workspace for the larger of its two calls, each rounded up to 256 bytes. */
gdn_status gdn_decode_layer_workspace_size(const gdn_dims* dims, int32_t hidden, int32_t batch,
                                           int64_t* bytes);

/*
 * The device address of pinned host memory (cudaHostAlloc, or page-locked
 * by a framework's pinned allocator), for the arguments of gdn_decode_step
 * that accept it. Writes *device and returns GDN_OK if the runtime reports
 * host as mapped into the device's address space; GDN_ERR_INVALID_ARG for a
 * NULL argument or memory that is not (pageable memory, device memory).
 * Allocates nothing; the mapping lives as long as the allocation.
 */
gdn_status gdn_host_pointer(const void* host, void** device);

/*
 * Device-side error word: kernels whose bounded waits give up record a
 * status here instead of hanging. Reads it (synchronising the device) into
 * *status and, when clear != 0, resets it to GDN_OK.
 */
gdn_status gdn_device_error(int32_t* status, int32_t clear);

/*
 * Self-test of the device-side give-up path: one warp waits on an mbarrier
 * that nothing ever arrives on, with a time limit of limit_ns (1 us .. 10 s)
 * instead of the library's usual 2 s, gives up, records GDN_ERR_TIMEOUT in
 * the device error word (gdn_device_error) and exits; nothing faults or
 * hangs and the context stays usable. gave_up is a device int32 written 1
 * by the kernel when its wait gave up (0 if the wait had completed). No
 * counterpart on the pages. GDN_ERR_INVALID_ARG for a limit out of range or
 * a NULL gave_up.
 */
gdn_status gdn_selftest_wait_timeout(int64_t limit_ns, int32_t* gave_up, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
