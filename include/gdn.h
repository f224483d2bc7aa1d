/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet (GDN) sublayer library, libgdn.so.
 *
 * The sublayer, as the pages define it (pegainfer PR #1152 "Reference golden for the GDN
 * sublayer", Summary and Code review; GLM-5.3-Flash kernel TDD ledger, slices I2-I4):
 *
 *   prefill:  x --(causal depthwise conv1d, width 4, + SiLU)--> qkv (bf16)
 *             qkv --(head expansion by repeat_interleave, L2 norm of q and k,
 *                    chunk-wise gated delta rule with an fp32 [value, key] state)--> o
 *             o, z --(gated RMSNorm with a sigmoid output gate)--> out
 *   decode:   the same for one token per sequence, fused in one launch (Qwen3.8 kernel
 *             architecture and TDD ledger, "Current dense-27B kernel map": scalar GDN
 *             recurrence and fused output gate).
 *
 * The recurrence (per sequence and V head; S is Dv x Dk, rows index the value dimension):
 *   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,    o_t = q_scale S_t q_t
 * with k_t, q_t the L2-normalised key/query of K head floor(h / (Hv/Hk)).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous, row-major, and
 *     16-byte aligned (else GDN_ERR_MISALIGNED).  The library never allocates, frees or keeps
 *     a reference to caller memory after the call returns.
 *   - bf16 tensors are passed as gdn_bf16 (raw 16-bit patterns); fp32 as float.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call is
 *     asynchronous on that stream; arguments are validated on the host before any launch, and
 *     a call that returns an error has launched nothing.
 *   - Geometry: C = 2*Hk*Dk + Hv*Dv conv channels packed [q heads | k heads | v heads].  This
 *     build supports Dk = Dv = 128, conv width 4, Hv a multiple of Hk, Hk <= 64, Hv <= 192;
 *     anything else is refused with GDN_ERR_UNSUPPORTED_GEOMETRY, never silently mis-tiled.
 *   - Device-side argument faults (for example a cu_seqlens array that is not monotonic or does
 *     not end at total_tokens) are never turned into out-of-range accesses: the kernels clamp,
 *     skip the bad sequence and raise a device error word, reported by gdn_check_device_errors.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

typedef uint16_t gdn_bf16; /* IEEE bfloat16 bit pattern */
typedef uint16_t gdn_f16;  /* IEEE binary16 (half precision) bit pattern */

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARGUMENT = 1,     /* null pointer, negative size, aliasing that is not allowed */
  GDN_ERR_UNSUPPORTED_GEOMETRY = 2, /* geometry outside what the kernels are built for         */
  GDN_ERR_MISALIGNED = 3,           /* a tensor pointer is not 16-byte aligned                  */
  GDN_ERR_CUDA = 4,                 /* a CUDA runtime call or kernel launch failed              */
  GDN_ERR_TIMEOUT = 5,              /* a bounded in-kernel wait ran out (device error word)     */
  GDN_ERR_DEVICE_ARGUMENT = 6,      /* a kernel found a bad device-side argument (cu_seqlens)   */
  GDN_ERR_WORKSPACE = 7             /* workspace missing or smaller than the queried size       */
} gdn_status;

/* Head geometry.  The pages' model: 16 K heads and 48 V heads of width 128, a four-tap conv
 * (pegainfer PR #1152, Summary). */
typedef struct {
  int32_t num_k_heads; /* Hk */
  int32_t num_v_heads; /* Hv, a multiple of Hk; V head h reads K head h / (Hv/Hk) */
  int32_t head_k_dim;  /* Dk (128) */
  int32_t head_v_dim;  /* Dv (128) */
  int32_t conv_width;  /* W  (4)   */
} gdn_geometry;

/* Tokens per chunk of the chunk-wise prefill.  A chunk never crosses a sequence boundary.
 * (pegainfer PR #1152, Validation: 16- and 64-token runs fit in one chunk, 80- and 128-token
 * runs take two.) */
#define GDN_CHUNK_SIZE 64

/* Human-readable name of a status code (static storage). */
GDN_API const char* gdn_status_string(gdn_status status);

/* Detail of the last error returned on the calling host thread ("" if none). */
GDN_API const char* gdn_last_error_message(void);

/* Library version string (static storage). */
GDN_API const char* gdn_version(void);

/*
 * Causal depthwise conv1d (width W, no bias) + SiLU over packed variable-length sequences.
 * pegainfer PR #1152, Summary (a four-tap depthwise conv; conv1d.weight is its only weight) and
 * "Commands + measured numbers" (the conv leg, compared bit-exact); GLM-5.3-Flash ledger,
 * slice I3 (a decode step equals the full width-4 causal convolution).
 *
 *   y[t, c] = bf16( silu( sum_{i<W} w[c, i] * xin(t - (W-1) + i, c) ) ),  silu(a) = a*sigmoid(a)
 *
 * where xin(p, c) is x[p, c] inside the token's own sequence, the conv state of that sequence
 * for the W-1 positions before its start, and 0 when conv_state_in is NULL.  Accumulation is
 * fp32; the result is rounded once to bf16 (round to nearest even).
 *
 *   x              [total_tokens, C] bf16
 *   conv_w         [C, W] bf16; w[c, W-1] multiplies the current token
 *   cu_seqlens     [num_seqs + 1] int32 (device): sequence n is tokens cu[n] .. cu[n+1]-1;
 *                  cu[0] = 0, non-decreasing, cu[num_seqs] = total_tokens
 *   conv_state_in  [num_seqs, C, W-1] bf16 raw inputs before each sequence (oldest first), or NULL
 *   conv_state_out [num_seqs, C, W-1] bf16 last W-1 raw inputs of each sequence, or NULL; may be
 *                  the same buffer as conv_state_in (updated in place)
 *   y              [total_tokens, C] bf16; must not overlap x
 * total_tokens == 0 or num_seqs == 0 is a no-op that returns GDN_OK.
 */
GDN_API gdn_status gdn_conv1d_prefill(const gdn_geometry* geo, const gdn_bf16* x,
                                      const gdn_bf16* conv_w, const int32_t* cu_seqlens,
                                      int32_t num_seqs, int32_t total_tokens,
                                      const gdn_bf16* conv_state_in, gdn_bf16* conv_state_out,
                                      gdn_bf16* y, void* stream);

/*
 * Bytes of device workspace for the fast path of gdn_chunk_prefill at these sizes (0 when
 * num_seqs == 0).  With at least this much, the call runs as two kernels: one that forms, for
 * every 64-token chunk at once, the quantities that do not depend on the recurrent state (the
 * intra-chunk decay factors, the solve (I + A)^-1 and the masked query-key product, about 25 KB
 * per chunk and V head), and one that carries the state through the chunks.  From 4,096 tokens
 * on it also holds 32 state slots of Hv x 128 x 128 fp32 for the parts of long sequences (see
 * gdn_chunk_prefill).  The workspace contents need no initialisation and are dead when the call's
 * kernels finish.
 */
GDN_API size_t gdn_chunk_prefill_workspace_size(const gdn_geometry* geo, int32_t num_seqs,
                                                int32_t total_tokens);

/*
 * Smallest workspace gdn_chunk_prefill accepts (the per-call sequence schedule: 256 bytes plus
 * 4 bytes per sequence, rounded up to 256).  With less than gdn_chunk_prefill_workspace_size()
 * but at least this, the call runs one fused kernel that forms the state-independent quantities
 * chunk by chunk on the state chain itself: same results within the stated tolerances, slower.
 */
GDN_API size_t gdn_chunk_prefill_min_workspace_size(const gdn_geometry* geo, int32_t num_seqs,
                                                    int32_t total_tokens);

/*
 * Chunk-wise gated delta rule over packed variable-length sequences (prefill), optionally
 * fused with the sigmoid-gated RMSNorm.  pegainfer PR #1152, Consumer (stage order
 * prepare -> cumsum -> A -> solve -> recompute -> state -> output) and Code review (f32
 * recurrent state carried across chunks); GLM-5.3-Flash ledger, slice I4 (the chunk path
 * matches the sequential state and output at 63/64/65 tokens).
 *
 *   qkv        [total_tokens, C] bf16 conv output (gdn_conv1d_prefill's y): q heads | k heads | v heads
 *   g, beta    [total_tokens, Hv] fp32 log decay (<= 0) and write strength
 *   cu_seqlens [num_seqs + 1] int32 (device), as for gdn_conv1d_prefill
 *   q_scale    output scale applied to S q (1/sqrt(Dk) for the pages' model)
 *   l2_eps     epsilon of the q/k L2 norm x / sqrt(sum x^2 + eps) (1e-6)
 *   state_in   [num_seqs, Hv, Dv, Dk] fp32 initial states ([value, key]), or NULL for zeros
 *   state_out  [num_seqs, Hv, Dv, Dk] fp32 final states; may be the same buffer as state_in
 *   z, norm_w  NULL: `out` receives o = q_scale S_t q_t (bf16).  Otherwise z [total_tokens, Hv, Dv]
 *              and norm_w [Dv] bf16, and `out` receives the gated RMSNorm of o:
 *              o * (mean_d o^2 + rms_eps)^(-1/2) * norm_w * sigmoid(z), computed from the fp32 o
 *   out        [total_tokens, Hv, Dv] bf16
 *   workspace  256-byte aligned device memory of at least gdn_chunk_prefill_min_workspace_size()
 *              bytes (NULL if 0); gdn_chunk_prefill_workspace_size() bytes select the fast path
 *
 * Streams: with the fast-path workspace, a state_out buffer, at least 4,096 tokens and no stream
 * capture in progress, the call splits each sequence's chunks into segments and runs the
 * state-independent stage of segment k + 1 on a library-owned side stream (one per device, created
 * on first use and shared by every caller on that device) beside the state stage of segment k,
 * ordered by events the library creates once per host thread and device.  Everything the call
 * writes is ordered before later work on `stream`.  Calls from different streams whose side-stream
 * work is queued together run it one after the other.  Under stream capture, everything runs on
 * `stream` as one segment.
 *
 * Long sequences: from 4,096 tokens on, a sequence whose segment holds more than twice the chunks
 * one CTA slot would get (the segment's work spread over two CTAs per SM) is cut into three or four
 * parts that run at once, decided on the device from cu_seqlens; parts after the first start
 * from a state combined from the earlier parts' transitions.  Their launch runs on a second
 * library-owned stream (per device, like the side stream) and is joined to `stream` before the
 * call's work ends; under stream capture it runs on `stream`.  A part waits (bounded) for the
 * transitions it needs; a wait that runs out sets GDN_ERR_TIMEOUT in the device error word.  With
 * one segment and state_out equal to state_in, nothing is split.
 */
GDN_API gdn_status gdn_chunk_prefill(const gdn_geometry* geo, const gdn_bf16* qkv, const float* g,
                                     const float* beta, const int32_t* cu_seqlens,
                                     int32_t num_seqs, int32_t total_tokens, float q_scale,
                                     float l2_eps, const float* state_in, float* state_out,
                                     const gdn_bf16* z, const gdn_bf16* norm_w, float rms_eps,
                                     gdn_bf16* out, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * The whole prefill sublayer in one call: gdn_conv1d_prefill (its output written to qkv), then
 * gdn_chunk_prefill on it -- the "prepare" stage of pegainfer PR #1152 Consumer, conv included,
 * followed by the chunk stages.  Same arguments, results and errors as the two calls in
 * sequence (qkv: [total_tokens, C] bf16, must not overlap x; conv_state_out may alias
 * conv_state_in; workspace as for gdn_chunk_prefill), with every argument of both stages checked
 * before either is launched: a call that returns an error has launched nothing.
 */
GDN_API gdn_status gdn_prefill(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w,
                               const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                               const gdn_bf16* conv_state_in, gdn_bf16* conv_state_out,
                               gdn_bf16* qkv, const float* g, const float* beta, float q_scale,
                               float l2_eps, const float* state_in, float* state_out,
                               const gdn_bf16* z, const gdn_bf16* norm_w, float rms_eps,
                               gdn_bf16* out, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * The gates of the recurrence from their projections, for every row (token, or sequence of a
 * decode step) and V head:
 *   g[r, h]    = -exp(A_log[h]) * softplus(a[r, h] + dt_bias[h]),   softplus(x) = log(1 + e^x)
 *   beta[r, h] = sigmoid(b[r, h])
 * The pages name these inputs (Qwen3.8 kernel architecture and TDD ledger, "GDN alpha/beta
 * transforms"; PR #1152 Summary: A_log, dt_bias, the a / b projections, and a fixture that holds
 * g / beta only after this derivation) but give no formula: this is the gate of the published
 * Gated DeltaNet / Mamba-2 layers.
 *   a, b        [rows, Hv] bf16 projection outputs
 *   A_log, dt_bias  [Hv] fp32 (4-byte aligned)
 *   g, beta     [rows, Hv] fp32 outputs, ready for gdn_chunk_prefill / gdn_decode_step
 */
GDN_API gdn_status gdn_gates(const gdn_geometry* geo, const gdn_bf16* a, const gdn_bf16* b,
                             const float* A_log, const float* dt_bias, float* g, float* beta,
                             int32_t rows, void* stream);

/*
 * gdn_chunk_prefill and gdn_decode_step with the gates derived inside the kernels that use them,
 * from the projections a, b and the per-head A_log, dt_bias (the gdn_gates formula, the same
 * arithmetic, so the results have the same bits as gdn_gates followed by the plain call): g and
 * beta are never written to memory and no gates launch precedes the call.  Qwen3.8 kernel
 * architecture and TDD ledger, kernel map (the GDN alpha / beta transforms feed the recurrence);
 * pegainfer PR #1152 Summary (A_log, dt_bias and the a / b projections are the layer's inputs).
 *   a, b            [rows, Hv] bf16 (rows = total_tokens for the prefill, batch for the decode;
 *                   2-byte aligned)
 *   A_log, dt_bias  [Hv] fp32 (4-byte aligned)
 * Every other argument, the results and the errors are those of gdn_chunk_prefill and
 * gdn_decode_step (fp32 state).
 */
GDN_API gdn_status gdn_chunk_prefill_fused_gates(const gdn_geometry* geo, const gdn_bf16* qkv,
                                                 const gdn_bf16* a, const gdn_bf16* b,
                                                 const float* A_log, const float* dt_bias,
                                                 const int32_t* cu_seqlens, int32_t num_seqs,
                                                 int32_t total_tokens, float q_scale, float l2_eps,
                                                 const float* state_in, float* state_out,
                                                 const gdn_bf16* z, const gdn_bf16* norm_w,
                                                 float rms_eps, gdn_bf16* out, void* workspace,
                                                 size_t workspace_bytes, void* stream);
GDN_API gdn_status gdn_decode_step_fused_gates(const gdn_geometry* geo, const gdn_bf16* x,
                                               const gdn_bf16* conv_w, gdn_bf16* conv_state,
                                               const gdn_bf16* a, const gdn_bf16* b,
                                               const float* A_log, const float* dt_bias,
                                               float* state, const gdn_bf16* z,
                                               const gdn_bf16* norm_w, float q_scale, float l2_eps,
                                               float rms_eps, gdn_bf16* out, int32_t batch,
                                               void* stream);

/*
 * Sigmoid-gated RMSNorm, one row per (token, V head).  pegainfer PR #1152, Summary
 * (output_gate_type "sigmoid"; the in-tree kernel that hard-codes silu is wrong) and Code
 * review (rms_norm_eps == 1e-6).
 *   out[r, d] = o[r, d] * (mean_d o[r, :]^2 + eps)^(-1/2) * norm_w[d] * sigmoid(z[r, d])
 *   o, z, out  [total_tokens, Hv, Dv] bf16 (out may alias o);  norm_w [Dv] bf16
 */
GDN_API gdn_status gdn_gated_rmsnorm(const gdn_geometry* geo, const gdn_bf16* o, const gdn_bf16* z,
                                     const gdn_bf16* norm_w, float eps, gdn_bf16* out,
                                     int32_t total_tokens, void* stream);

/*
 * One fused decode step for `batch` independent sequences (one token each): conv step on the
 * conv shift register + SiLU, L2 norm of q/k, the gated delta rule update of the fp32 state in
 * place, and the sigmoid-gated RMSNorm.  Qwen3.8 kernel architecture and TDD ledger, "Current
 * dense-27B kernel map" (scalar GDN recurrence and fused output gate); spark_model
 * layer_struct.rs, the strided decode kernel fields (one launch for all sequences, state read
 * once and written once).
 *
 *   x           [batch, C] bf16 raw conv input of this token
 *   conv_w      [C, W] bf16
 *   conv_state  [batch, C, W-1] bf16, in/out: the previous W-1 raw inputs, oldest first
 *   g, beta     [batch, Hv] fp32
 *   state       [batch, Hv, Dv, Dk] fp32, in/out
 *   z           [batch, Hv, Dv] bf16;  norm_w [Dv] bf16
 *   out         [batch, Hv, Dv] bf16 gated output
 */
GDN_API gdn_status gdn_decode_step(const gdn_geometry* geo, const gdn_bf16* x,
                                   const gdn_bf16* conv_w, gdn_bf16* conv_state, const float* g,
                                   const float* beta, float* state, const gdn_bf16* z,
                                   const gdn_bf16* norm_w, float q_scale, float l2_eps,
                                   float rms_eps, gdn_bf16* out, int32_t batch, void* stream);

/*
 * gdn_decode_step with the recurrent state stored as IEEE binary16 ("FP16 h-state"): Qwen3.8
 * kernel architecture and TDD ledger, the FP16 h-state twins of the decode kernels (the same
 * arithmetic as the fp32 kernel; the state is half precision in memory only and is rounded once
 * per token boundary).  Each state element is widened to fp32 on load, the step runs exactly as in
 * gdn_decode_step (the output comes from the new state before rounding), and the new state is
 * rounded to binary16 (to nearest, ties to even) when it is stored.  This halves the state bytes
 * the step reads and writes.
 *
 *   state       [batch, Hv, Dv, Dk] binary16, in/out (16-byte aligned)
 *   all other arguments, results and errors as gdn_decode_step.
 *
 * A state element whose magnitude rounds above 65504 becomes an infinity; nothing clamps it.
 */
GDN_API gdn_status gdn_decode_step_fp16_state(const gdn_geometry* geo, const gdn_bf16* x,
                                              const gdn_bf16* conv_w, gdn_bf16* conv_state,
                                              const float* g, const float* beta, gdn_f16* state,
                                              const gdn_bf16* z, const gdn_bf16* norm_w,
                                              float q_scale, float l2_eps, float rms_eps,
                                              gdn_bf16* out, int32_t batch, void* stream);

/*
 * Multi-token verify: `rows` (K, 1..17) consecutive tokens of each of `batch` sequences run
 * through the decode step in order -- conv step, L2 norms, gated delta rule, gated RMSNorm --
 * starting from conv_state and state, exactly as K calls of gdn_decode_step would, but WITHOUT
 * modifying either state.  Every row's gated output is written; what a later commit needs is
 * written to `stash`.  Qwen3.8 kernel architecture and TDD ledger, "Transaction and width
 * vocabulary" (verify_rows; a target transaction resolves exactly once: commit publishes only the
 * selected GDN state, abort leaves the prior state); spark_model layer_struct.rs, the WY verify
 * kernels (K = 2..17) and the write-on-accept twin with its post-verdict fold.
 *
 *   x           [batch, rows, C] bf16 raw conv inputs
 *   conv_w      [C, W] bf16;  conv_state [batch, C, W-1] bf16 (read only)
 *   g, beta     [batch, rows, Hv] fp32
 *   state       [batch, Hv, Dv, Dk] fp32 (read only)
 *   z           [batch, rows, Hv, Dv] bf16;  norm_w [Dv] bf16
 *   out         [batch, rows, Hv, Dv] bf16: row r is the output of the r+1-th token
 *   stash       gdn_verify_stash_size(geo, batch, rows) bytes, 16-byte aligned; one record per
 *               (sequence, row) at ((b * rows) + r) * (stash_size / (batch * rows)) bytes: the
 *               row's raw conv inputs (C bf16), normalised keys (Hk x Dk fp32), its delta
 *               e = beta (v - decayed state . k) for every V head and value row (Hv x Dv fp32)
 *               and g (Hv fp32).
 * GDN_ERR_UNSUPPORTED_GEOMETRY when `rows` rows of Hv/Hk V heads do not fit the kernel's shared
 * memory (never for Hv/Hk <= 3).
 */
GDN_API size_t gdn_verify_stash_size(const gdn_geometry* geo, int32_t batch, int32_t rows);
GDN_API gdn_status gdn_verify(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w,
                              const gdn_bf16* conv_state, const float* g, const float* beta,
                              const float* state, const gdn_bf16* z, const gdn_bf16* norm_w,
                              float q_scale, float l2_eps, float rms_eps, gdn_bf16* out,
                              int32_t batch, int32_t rows, void* stash, size_t stash_bytes,
                              void* stream);

/*
 * Resolves a verify: for each sequence b, committed_rows[b] = m (device int32, 0..rows) rows are
 * committed -- conv_state and state become what m decode steps of that sequence's first m rows
 * would have left (m = 0: an abort, both states untouched).  Reads only stash records of rows
 * < m.  The states must be the ones the verify read (unchanged since).  A value outside
 * [0, rows] leaves that sequence untouched and raises GDN_ERR_DEVICE_ARGUMENT in the device
 * error word.  stash_bytes is the size of the stash buffer; a stash smaller than
 * gdn_verify_stash_size(geo, batch, rows) is refused with GDN_ERR_WORKSPACE (nothing launched).
 */
GDN_API gdn_status gdn_verify_commit(const gdn_geometry* geo, const int32_t* committed_rows,
                                     const void* stash, size_t stash_bytes, gdn_bf16* conv_state,
                                     float* state, int32_t batch, int32_t rows, void* stream);

/*
 * gdn_verify and gdn_verify_commit with the recurrent state stored as IEEE binary16 (Qwen3.8
 * ledger, the FP16 h-state twins of the WY verify kernels).  The verify widens the state and
 * computes in fp32 exactly as gdn_verify; the commit widens it, applies the committed rows and
 * stores the result rounded once to binary16 (to nearest, ties to even).  No per-row state is
 * ever stored, so that is the only rounding: a commit of m rows equals m calls of
 * gdn_decode_step_fp16_state up to the roundings those calls make between the rows.  The stash
 * is the same as gdn_verify's; m = 0 leaves the state's bits untouched.
 *   state       [batch, Hv, Dv, Dk] binary16 (read only in the verify; in/out in the commit)
 */
GDN_API gdn_status gdn_verify_fp16_state(const gdn_geometry* geo, const gdn_bf16* x,
                                         const gdn_bf16* conv_w, const gdn_bf16* conv_state,
                                         const float* g, const float* beta, const gdn_f16* state,
                                         const gdn_bf16* z, const gdn_bf16* norm_w, float q_scale,
                                         float l2_eps, float rms_eps, gdn_bf16* out, int32_t batch,
                                         int32_t rows, void* stash, size_t stash_bytes,
                                         void* stream);
GDN_API gdn_status gdn_verify_commit_fp16_state(const gdn_geometry* geo,
                                                const int32_t* committed_rows, const void* stash,
                                                size_t stash_bytes, gdn_bf16* conv_state,
                                                gdn_f16* state, int32_t batch, int32_t rows,
                                                void* stream);

/*
 * One fused decode step of the KDA (Kimi delta attention) layer: as gdn_decode_step, with a decay
 * per key channel instead of per head.  GLM-5.3-Flash kernel TDD ledger, slices I2 (an fp32
 * state indexed [value, key], the decay clamped then exponentiated, its own q output scale),
 * I2a (q/k normalised x / sqrt(sum x^2 + eps)) and I3 (the width-4 conv step).  Per V head:
 *   S <- S diag(exp(max(g, g_min)));   e = beta (v - S k);   S <- S + e k^T;   o = q_scale S q
 * followed by the same sigmoid-gated RMSNorm as gdn_decode_step.
 *   g           [batch, Hv, Dk] fp32 per-channel log decay (16-byte aligned)
 *   g_min       the clamp: decays below exp(g_min) are raised to it (-INFINITY: no clamp)
 *   all other arguments, results and errors as gdn_decode_step (fp32 state).
 */
GDN_API gdn_status gdn_kda_decode_step(const gdn_geometry* geo, const gdn_bf16* x,
                                       const gdn_bf16* conv_w, gdn_bf16* conv_state,
                                       const float* g, float g_min, const float* beta, float* state,
                                       const gdn_bf16* z, const gdn_bf16* norm_w, float q_scale,
                                       float l2_eps, float rms_eps, gdn_bf16* out, int32_t batch,
                                       void* stream);

/*
 * The KDA recurrence over packed variable-length sequences (the prefill's recurrent leg),
 * optionally fused with the sigmoid-gated RMSNorm: the step of gdn_kda_decode_step applied to
 * every token in order, each (sequence, V head) state carried from token to token.
 * GLM-5.3-Flash kernel TDD ledger, slices I2 (an fp32 state indexed [value, key], a per-channel
 * decay clamped then exponentiated, its own q output scale), I2a (q/k normalised
 * x / sqrt(sum x^2 + eps)) and I4 (the prefill matches the sequential state and output at every
 * length).  This is the sequential form: one CTA per (V head, sequence) walks the tokens, so a
 * call's time grows with its longest sequence.
 *   qkv        [total_tokens, C] bf16 conv output (gdn_conv1d_prefill's y): q heads | k heads | v heads
 *   g          [total_tokens, Hv, Dk] fp32 per-channel log decay (16-byte aligned)
 *   g_min      the clamp: decays below exp(g_min) are raised to it (-INFINITY: no clamp; NaN is rejected)
 *   beta       [total_tokens, Hv] fp32 write strength (4-byte aligned)
 *   cu_seqlens [num_seqs + 1] int32 (device), as for gdn_conv1d_prefill; num_seqs <= 65535.
 *              Contents that are not nondecreasing within [0, total_tokens] set
 *              GDN_ERR_DEVICE_ARGUMENT in the device error word; those sequences are not computed.
 *   q_scale, l2_eps, state_in, state_out, z, norm_w, rms_eps, out: as gdn_chunk_prefill (fp32
 *              states [num_seqs, Hv, Dv, Dk]; state_out may be state_in; a sequence of length 0
 *              copies its state).  No workspace.
 */
GDN_API gdn_status gdn_kda_recurrence(const gdn_geometry* geo, const gdn_bf16* qkv, const float* g,
                                      float g_min, const float* beta, const int32_t* cu_seqlens,
                                      int32_t num_seqs, int32_t total_tokens, float q_scale,
                                      float l2_eps, const float* state_in, float* state_out,
                                      const gdn_bf16* z, const gdn_bf16* norm_w, float rms_eps,
                                      gdn_bf16* out, void* stream);

/*
 * Workspace bytes of gdn_kda_chunk_prefill: 256 bytes of counters, the longest-first sequence
 * order and per-sequence chunk offsets (4 bytes per sequence each, rounded up to 256), then one
 * 108,032-byte record per (64-token chunk, V head) for at most (total_tokens + 63 num_seqs) / 64
 * chunks.  0 when num_seqs <= 0.
 */
GDN_API size_t gdn_kda_chunk_prefill_workspace_size(const gdn_geometry* geo, int32_t num_seqs,
                                                    int32_t total_tokens);

/*
 * The KDA recurrence of gdn_kda_recurrence in its chunk-wise form: the same arguments, results
 * and errors, computed 64 tokens at a time on the tensor cores instead of token by token, plus a
 * workspace.  GLM-5.3-Flash kernel TDD ledger, slices I2, I2a and I4 (the chunk form matches the
 * sequential state and output at 63, 64 and 65 tokens).  Per chunk of L tokens from the state S0,
 * with gamma_t the running sum of the clamped log decays of each key channel:
 *   A_ts = beta_t sum_c k^_t k^_s e^(gamma_t - gamma_s) (s < t),  T = (I + A)^-1,
 *   E = (V - S0 (K^ o e^gamma)^T) diag(beta) T^T,
 *   O = q_scale (S0 (Q^ o e^gamma)^T + E P^T),  P_ts = sum_c q^_t k^_s e^(gamma_t - gamma_s) (s <= t),
 *   S = S0 diag(e^gamma_L) + E (K^ o e^(gamma_L - gamma))
 * A first kernel forms every (chunk, V head)'s state-independent part in parallel; a second walks
 * each (sequence, V head) through its chunks with the fp32 state in tensor memory.  Every product
 * on the state's path takes bf16 high / low pairs of both operands; o's own products plain bf16.
 * Tolerances: those of gdn_chunk_prefill.
 *   g          [total_tokens, Hv, Dk] fp32 per-channel log decay (16-byte aligned); after the clamp
 *              every value must be finite and at most 0 (a decay) -- a -INFINITY log decay (with
 *              g_min = -INFINITY) makes that chunk's results NaN: clamp it, or use
 *              gdn_kda_recurrence
 *   workspace  256-byte aligned device memory of gdn_kda_chunk_prefill_workspace_size() bytes
 *              (GDN_ERR_WORKSPACE if NULL or smaller), overwritten
 *   num_seqs   at most 2^31 / Hv; cu_seqlens outside [0, total_tokens] or decreasing set
 *              GDN_ERR_DEVICE_ARGUMENT in the device error word, those sequences are not computed
 *   everything else as gdn_kda_recurrence.  Everything runs on `stream`.
 */
GDN_API gdn_status gdn_kda_chunk_prefill(const gdn_geometry* geo, const gdn_bf16* qkv, const float* g,
                                         float g_min, const float* beta, const int32_t* cu_seqlens,
                                         int32_t num_seqs, int32_t total_tokens, float q_scale,
                                         float l2_eps, const float* state_in, float* state_out,
                                         const gdn_bf16* z, const gdn_bf16* norm_w, float rms_eps,
                                         gdn_bf16* out, void* workspace, size_t workspace_bytes,
                                         void* stream);

/*
 * The KDA prefill in one call: gdn_conv1d_prefill (its output written to qkv), then
 * gdn_kda_chunk_prefill on it.  Same arguments, results and errors as the two calls in sequence
 * (qkv: [total_tokens, C] bf16, must not overlap x; conv_state_out may alias conv_state_in;
 * workspace as for gdn_kda_chunk_prefill), with every argument of both stages checked before
 * either is launched: a call that returns an error has launched nothing.
 */
GDN_API gdn_status gdn_kda_prefill(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w,
                                   const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                   const gdn_bf16* conv_state_in, gdn_bf16* conv_state_out,
                                   gdn_bf16* qkv, const float* g, float g_min, const float* beta,
                                   float q_scale, float l2_eps, const float* state_in,
                                   float* state_out, const gdn_bf16* z, const gdn_bf16* norm_w,
                                   float rms_eps, gdn_bf16* out, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* Capacity of the fixed scratch used by gdn_chunk_prefill_noalloc. */
#define GDN_NOALLOC_MAX_SEQS 16384
#define GDN_NOALLOC_SCRATCH_BYTES (256 + 4 * GDN_NOALLOC_MAX_SEQS) /* 65,792 bytes */

/*
 * gdn_chunk_prefill for callers that cannot allocate device memory when they call it -- for
 * example a host that hands all device memory to its own pool up front, or a latency-critical
 * loop where cudaMalloc/cudaFree (which can synchronise the device) are not allowed.  Same
 * arguments, results and errors as gdn_chunk_prefill, without the workspace pair: the call
 * allocates nothing and calls no allocating routine.
 *
 * Its scratch is one fixed device array of GDN_NOALLOC_SCRATCH_BYTES inside the library, which
 * every GPU that loads the library keeps until the process exits; it holds the schedule of up to
 * GDN_NOALLOC_MAX_SEQS sequences, and a larger num_seqs is refused with GDN_ERR_INVALID_ARGUMENT
 * (nothing launched).  The first call on a device looks up that array's device address with the
 * device current (cudaGetSymbolAddress) and the kernels' launch attributes, which under lazy
 * module loading may load the library's module and reserve its static arrays on that device:
 * make this first call before any stream capture, and before a caller's pool takes the device
 * memory it will not give back.  The address is kept per device index for the life of the
 * process; after cudaDeviceReset it is stale, and the call must not be used again.  Host threads
 * making their first call at the same time store the same address (the cache is atomic).
 * All calls on a device share
 * the array and it keeps the last call's contents: each call rewrites the whole schedule and
 * zeroes its work counter before the main kernel reads them, but two calls whose kernels overlap
 * on the GPU (for example on two unordered streams) race on the array and give wrong results.
 * The scratch holds the minimum workspace only, so the call runs gdn_chunk_prefill's one-kernel
 * path.  There is no counterpart of this entry point on the pages.
 */
GDN_API gdn_status gdn_chunk_prefill_noalloc(const gdn_geometry* geo, const gdn_bf16* qkv, const float* g,
                                             const float* beta, const int32_t* cu_seqlens, int32_t num_seqs,
                                             int32_t total_tokens, float q_scale, float l2_eps,
                                             const float* state_in, float* state_out, const gdn_bf16* z,
                                             const gdn_bf16* norm_w, float rms_eps, gdn_bf16* out,
                                             void* stream);

/*
 * Waits for `stream`, then reads and clears the library's device error word.  Returns GDN_OK,
 * GDN_ERR_DEVICE_ARGUMENT (a kernel skipped a sequence with bad cu_seqlens entries),
 * GDN_ERR_TIMEOUT (a bounded in-kernel wait ran out) or GDN_ERR_CUDA.  The word is per device
 * and shared by all streams; the kernels only ever set bits in it.
 */
GDN_API gdn_status gdn_check_device_errors(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
