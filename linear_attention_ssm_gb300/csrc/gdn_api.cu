// gdn_api.cu -- the C ABI of libgdn.so: host-side validation, then one launch per call.
//
// Every entry point checks its arguments on the host before it launches anything; a call that
// returns an error has launched nothing.  Device-side faults (bad cu_seqlens contents, a bounded
// wait that ran out) set bits in a per-device error word that gdn_check_device_errors() reads.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/gdn.h"
#ifdef GDN_TEST_HOOKS
#include "../../include/gdn_debug.h"
#endif
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace {

__device__ unsigned g_gdn_error_word;

thread_local std::string g_last_error;
#ifdef GDN_TEST_HOOKS
std::atomic<int> g_chunk_mode{0};  // the test library's chunk-design selection (gdn_debug.h)
#else
constexpr int g_chunk_mode = 0;    // the product library always takes the default design
#endif

constexpr int kMaxDevices = 64;
// Device address of the error word, per device index, looked up on the first call that needs it.
// Two host threads making their first call at once both store the same address.
std::atomic<unsigned*> g_err_ptr[kMaxDevices] = {};

gdn_status fail(gdn_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
gdn_status fail(gdn_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

gdn_status ok() {
  g_last_error.clear();
  return GDN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

gdn_status check_geometry(const gdn_geometry* geo) {
  if (!geo) return fail(GDN_ERR_INVALID_ARGUMENT, "geometry is NULL");
  if (geo->num_k_heads <= 0 || geo->num_v_heads <= 0 || geo->num_v_heads % geo->num_k_heads != 0)
    return fail(GDN_ERR_UNSUPPORTED_GEOMETRY, "num_v_heads (%d) must be a positive multiple of num_k_heads (%d)",
                geo->num_v_heads, geo->num_k_heads);
  if (geo->head_k_dim != gdn::kHeadDim || geo->head_v_dim != gdn::kHeadDim)
    return fail(GDN_ERR_UNSUPPORTED_GEOMETRY, "head dims must be %d (got Dk=%d, Dv=%d)", gdn::kHeadDim,
                geo->head_k_dim, geo->head_v_dim);
  if (geo->conv_width != gdn::kConvWidth)
    return fail(GDN_ERR_UNSUPPORTED_GEOMETRY, "conv width must be %d (got %d)", gdn::kConvWidth, geo->conv_width);
  if (geo->num_k_heads > 64 || geo->num_v_heads > 192)
    return fail(GDN_ERR_UNSUPPORTED_GEOMETRY, "at most 64 K heads and 192 V heads (got %d, %d)", geo->num_k_heads,
                geo->num_v_heads);
  return GDN_OK;
}

int conv_channels(const gdn_geometry* g) {
  return 2 * g->num_k_heads * g->head_k_dim + g->num_v_heads * g->head_v_dim;
}

#define GDN_REQUIRE(ptr, name)                                                            \
  do {                                                                                    \
    if (!(ptr)) return fail(GDN_ERR_INVALID_ARGUMENT, "%s is NULL", name);                \
    if (!aligned16(ptr)) return fail(GDN_ERR_MISALIGNED, "%s is not 16-byte aligned", name); \
  } while (0)
#define GDN_OPTIONAL(ptr, name)                                                           \
  do {                                                                                    \
    if ((ptr) && !aligned16(ptr)) return fail(GDN_ERR_MISALIGNED, "%s is not 16-byte aligned", name); \
  } while (0)

gdn_status make_env(void* stream, gdn::LaunchEnv* env) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_CUDA, "device index %d out of range", dev);
  unsigned* err = g_err_ptr[dev].load(std::memory_order_acquire);
  if (!err) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_gdn_error_word);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    err = static_cast<unsigned*>(p);
    g_err_ptr[dev].store(err, std::memory_order_release);
  }
  env->err = err;
  env->num_sms = 0;
  env->stream = static_cast<cudaStream_t>(stream);
  return GDN_OK;
}

gdn_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARGUMENT: return "GDN_ERR_INVALID_ARGUMENT";
    case GDN_ERR_UNSUPPORTED_GEOMETRY: return "GDN_ERR_UNSUPPORTED_GEOMETRY";
    case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    case GDN_ERR_DEVICE_ARGUMENT: return "GDN_ERR_DEVICE_ARGUMENT";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
  }
  return "GDN_ERR_UNKNOWN";
}

const char* gdn_last_error_message(void) { return g_last_error.c_str(); }

const char* gdn_version(void) { return "gdn-gb300 0.1 (sm_103a)"; }

gdn_status gdn_conv1d_prefill(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w,
                              const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                              const gdn_bf16* conv_state_in, gdn_bf16* conv_state_out, gdn_bf16* y, void* stream) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (num_seqs < 0 || total_tokens < 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "negative size (num_seqs=%d, total_tokens=%d)", num_seqs, total_tokens);
  if (num_seqs == 0 && total_tokens > 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "total_tokens=%d with no sequence", total_tokens);
  if (num_seqs == 0) return ok();
  GDN_REQUIRE(conv_w, "conv_w");
  if (!cu_seqlens) return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens is NULL");
  if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) return fail(GDN_ERR_MISALIGNED, "cu_seqlens is not 4-byte aligned");
  GDN_OPTIONAL(conv_state_in, "conv_state_in");
  GDN_OPTIONAL(conv_state_out, "conv_state_out");
  const int C = conv_channels(geo);
  if (total_tokens > 0) {
    GDN_REQUIRE(x, "x");
    GDN_REQUIRE(y, "y");
    const size_t bytes = (size_t)total_tokens * C * 2;
    if (overlaps(x, bytes, y, bytes)) return fail(GDN_ERR_INVALID_ARGUMENT, "y overlaps x");
  } else if (!conv_state_out) {
    return ok();
  }
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  return launched(gdn::launch_conv1d_prefill(env, x, conv_w, cu_seqlens, num_seqs, total_tokens, C, conv_state_in,
                                             conv_state_out, y),
                  "conv1d launch");
}

size_t gdn_chunk_prefill_workspace_size(const gdn_geometry* geo, int32_t num_seqs, int32_t total_tokens) {
  if (!geo || num_seqs <= 0 || total_tokens < 0 || geo->num_k_heads <= 0 || geo->num_v_heads <= 0) return 0;
  return gdn::split_workspace_bytes(num_seqs, total_tokens, geo->num_k_heads, geo->num_v_heads);
}

size_t gdn_chunk_prefill_min_workspace_size(const gdn_geometry* geo, int32_t num_seqs, int32_t total_tokens) {
  (void)geo;
  (void)total_tokens;
  return num_seqs > 0 ? gdn::chunk_prefill_workspace_bytes(num_seqs) : 0;
}

}  // extern "C"

namespace {
// The gate inputs of a call: g and beta, or the projections a, b with A_log and dt_bias.
gdn_status check_gates(const gdn::GateSrc& gs) {
  if (gs.a) {
    if (!gs.b || !gs.A_log || !gs.dt_bias) return fail(GDN_ERR_INVALID_ARGUMENT, "a, b, A_log or dt_bias is NULL");
    if ((reinterpret_cast<uintptr_t>(gs.a) | reinterpret_cast<uintptr_t>(gs.b)) & 1u)
      return fail(GDN_ERR_MISALIGNED, "a or b is not 2-byte aligned");
    if ((reinterpret_cast<uintptr_t>(gs.A_log) | reinterpret_cast<uintptr_t>(gs.dt_bias)) & 3u)
      return fail(GDN_ERR_MISALIGNED, "A_log or dt_bias is not 4-byte aligned");
    return GDN_OK;
  }
  if (!gs.g || !gs.beta) return fail(GDN_ERR_INVALID_ARGUMENT, "g or beta is NULL");
  if ((reinterpret_cast<uintptr_t>(gs.g) | reinterpret_cast<uintptr_t>(gs.beta)) & 3u)
    return fail(GDN_ERR_MISALIGNED, "g or beta is not 4-byte aligned");
  return GDN_OK;
}

// The conv stage that gdn_prefill runs ahead of the chunk prefill (its output is the chunk stage's qkv).
struct ConvStage {
  const gdn_bf16* x;
  const gdn_bf16* w;
  const gdn_bf16* state_in;
  gdn_bf16* state_out;
  int C;
};

gdn_status chunk_prefill(const gdn_geometry* geo, const gdn_bf16* qkv, const gdn::GateSrc& gates,
                         const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens, float q_scale,
                         float l2_eps, const float* state_in, float* state_out, const gdn_bf16* z,
                         const gdn_bf16* norm_w, float rms_eps, gdn_bf16* out, void* workspace,
                         size_t workspace_bytes, void* stream, const ConvStage* conv = nullptr) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (num_seqs < 0 || total_tokens < 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "negative size (num_seqs=%d, total_tokens=%d)", num_seqs, total_tokens);
  if (num_seqs == 0 && total_tokens > 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "total_tokens=%d with no sequence", total_tokens);
  if ((long)num_seqs * geo->num_v_heads > 0x7FFFFFFFL)
    return fail(GDN_ERR_INVALID_ARGUMENT, "num_seqs * num_v_heads exceeds the grid limit");
  if (num_seqs == 0) return ok();
  if (!cu_seqlens) return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens is NULL");
  if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) return fail(GDN_ERR_MISALIGNED, "cu_seqlens is not 4-byte aligned");
  if (total_tokens > 0) {
    GDN_REQUIRE(qkv, "qkv");
    GDN_REQUIRE(out, "out");
    if ((s = check_gates(gates)) != GDN_OK) return s;
  }
  GDN_OPTIONAL(state_in, "state_in");
  GDN_OPTIONAL(state_out, "state_out");
  if (z) {
    GDN_REQUIRE(z, "z");
    GDN_REQUIRE(norm_w, "norm_w");
  }
  if (!(l2_eps >= 0.f) || !(rms_eps >= 0.f)) return fail(GDN_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  const size_t need = gdn_chunk_prefill_min_workspace_size(geo, num_seqs, total_tokens);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need, workspace_bytes);
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(GDN_ERR_MISALIGNED, "workspace is not 256-byte aligned");
  if (state_in && state_out && state_in != state_out) {
    const size_t sb = (size_t)num_seqs * geo->num_v_heads * gdn::kHeadDim * gdn::kHeadDim * 4;
    if (overlaps(state_in, sb, state_out, sb))
      return fail(GDN_ERR_INVALID_ARGUMENT, "state_out partially overlaps state_in");
  }
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  if (conv && (total_tokens > 0 || conv->state_out)) {  // every argument checked: the conv stage first
    s = launched(gdn::launch_conv1d_prefill(env, conv->x, conv->w, cu_seqlens, num_seqs, total_tokens, conv->C,
                                            conv->state_in, conv->state_out, const_cast<gdn_bf16*>(qkv)),
                 "conv1d launch");
    if (s != GDN_OK) return s;
  }
  return launched(gdn::launch_chunk_prefill(env, g_chunk_mode, qkv, gates, cu_seqlens, num_seqs, total_tokens,
                                            geo->num_k_heads, geo->num_v_heads, q_scale, l2_eps, state_in,
                                            state_out, z, norm_w, rms_eps, out, workspace, workspace_bytes),
                  "chunk prefill launch");
}
}  // namespace

extern "C" {

gdn_status gdn_chunk_prefill(const gdn_geometry* geo, const gdn_bf16* qkv, const float* g, const float* beta,
                             const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens, float q_scale,
                             float l2_eps, const float* state_in, float* state_out, const gdn_bf16* z,
                             const gdn_bf16* norm_w, float rms_eps, gdn_bf16* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  const gdn::GateSrc gates = {g, beta, nullptr, nullptr, nullptr, nullptr};
  return chunk_prefill(geo, qkv, gates, cu_seqlens, num_seqs, total_tokens, q_scale, l2_eps, state_in, state_out, z,
                       norm_w, rms_eps, out, workspace, workspace_bytes, stream);
}

gdn_status gdn_prefill(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w, const int32_t* cu_seqlens,
                       int32_t num_seqs, int32_t total_tokens, const gdn_bf16* conv_state_in,
                       gdn_bf16* conv_state_out, gdn_bf16* qkv, const float* g, const float* beta, float q_scale,
                       float l2_eps, const float* state_in, float* state_out, const gdn_bf16* z,
                       const gdn_bf16* norm_w, float rms_eps, gdn_bf16* out, void* workspace, size_t workspace_bytes,
                       void* stream) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (num_seqs > 0) {  // the conv stage's own arguments (the chunk stage checks the rest)
    GDN_REQUIRE(conv_w, "conv_w");
    GDN_OPTIONAL(conv_state_in, "conv_state_in");
    GDN_OPTIONAL(conv_state_out, "conv_state_out");
    if (total_tokens > 0) {
      GDN_REQUIRE(x, "x");
      GDN_REQUIRE(qkv, "qkv");
      const size_t bytes = (size_t)total_tokens * conv_channels(geo) * 2;
      if (overlaps(x, bytes, qkv, bytes)) return fail(GDN_ERR_INVALID_ARGUMENT, "qkv overlaps x");
    }
  }
  const gdn::GateSrc gates = {g, beta, nullptr, nullptr, nullptr, nullptr};
  const ConvStage conv = {x, conv_w, conv_state_in, conv_state_out, conv_channels(geo)};
  return chunk_prefill(geo, qkv, gates, cu_seqlens, num_seqs, total_tokens, q_scale, l2_eps, state_in, state_out, z,
                       norm_w, rms_eps, out, workspace, workspace_bytes, stream, &conv);
}

gdn_status gdn_chunk_prefill_fused_gates(const gdn_geometry* geo, const gdn_bf16* qkv, const gdn_bf16* a,
                                         const gdn_bf16* b, const float* A_log, const float* dt_bias,
                                         const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                         float q_scale, float l2_eps, const float* state_in, float* state_out,
                                         const gdn_bf16* z, const gdn_bf16* norm_w, float rms_eps, gdn_bf16* out,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!a) return fail(GDN_ERR_INVALID_ARGUMENT, "a is NULL");
  const gdn::GateSrc gates = {nullptr, nullptr, a, b, A_log, dt_bias};
  return chunk_prefill(geo, qkv, gates, cu_seqlens, num_seqs, total_tokens, q_scale, l2_eps, state_in, state_out, z,
                       norm_w, rms_eps, out, workspace, workspace_bytes, stream);
}

gdn_status gdn_gated_rmsnorm(const gdn_geometry* geo, const gdn_bf16* o, const gdn_bf16* z, const gdn_bf16* norm_w,
                             float eps, gdn_bf16* out, int32_t total_tokens, void* stream) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (total_tokens < 0) return fail(GDN_ERR_INVALID_ARGUMENT, "negative total_tokens");
  if (total_tokens == 0) return ok();
  GDN_REQUIRE(o, "o");
  GDN_REQUIRE(z, "z");
  GDN_REQUIRE(norm_w, "norm_w");
  GDN_REQUIRE(out, "out");
  if (!(eps >= 0.f)) return fail(GDN_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  return launched(gdn::launch_gated_rmsnorm(env, o, z, norm_w, eps, out, (long)total_tokens * geo->num_v_heads),
                  "gated rmsnorm launch");
}

}  // extern "C"

namespace {
gdn_status decode_step(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w, gdn_bf16* conv_state,
                       const gdn::GateSrc& gates, void* state, bool fp16_state, const gdn_bf16* z,
                       const gdn_bf16* norm_w, float q_scale, float l2_eps, float rms_eps, gdn_bf16* out,
                       int32_t batch, void* stream) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (geo->num_v_heads / geo->num_k_heads > gdn::decode_max_ratio())
    return fail(GDN_ERR_UNSUPPORTED_GEOMETRY, "decode supports at most %d V heads per K head",
                gdn::decode_max_ratio());
  if (batch < 0 || batch > 65535) return fail(GDN_ERR_INVALID_ARGUMENT, "batch must be in [0, 65535] (got %d)", batch);
  if (batch == 0) return ok();
  GDN_REQUIRE(x, "x");
  GDN_REQUIRE(conv_w, "conv_w");
  GDN_REQUIRE(conv_state, "conv_state");
  GDN_REQUIRE(state, "state");
  GDN_REQUIRE(z, "z");
  GDN_REQUIRE(norm_w, "norm_w");
  GDN_REQUIRE(out, "out");
  if ((s = check_gates(gates)) != GDN_OK) return s;
  if (!(l2_eps >= 0.f) || !(rms_eps >= 0.f)) return fail(GDN_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  return launched(gdn::launch_decode_step(env, x, conv_w, conv_state, gates, state, fp16_state, z, norm_w,
                                          q_scale, l2_eps, rms_eps, out, batch, geo->num_k_heads,
                                          geo->num_v_heads),
                  "decode launch");
}
}  // namespace

extern "C" {

gdn_status gdn_decode_step(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w, gdn_bf16* conv_state,
                           const float* g, const float* beta, float* state, const gdn_bf16* z,
                           const gdn_bf16* norm_w, float q_scale, float l2_eps, float rms_eps, gdn_bf16* out,
                           int32_t batch, void* stream) {
  const gdn::GateSrc gates = {g, beta, nullptr, nullptr, nullptr, nullptr};
  return decode_step(geo, x, conv_w, conv_state, gates, state, false, z, norm_w, q_scale, l2_eps, rms_eps, out,
                     batch, stream);
}

gdn_status gdn_decode_step_fused_gates(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w,
                                       gdn_bf16* conv_state, const gdn_bf16* a, const gdn_bf16* b, const float* A_log,
                                       const float* dt_bias, float* state, const gdn_bf16* z, const gdn_bf16* norm_w,
                                       float q_scale, float l2_eps, float rms_eps, gdn_bf16* out, int32_t batch,
                                       void* stream) {
  if (batch > 0 && !a) return fail(GDN_ERR_INVALID_ARGUMENT, "a is NULL");
  const gdn::GateSrc gates = {nullptr, nullptr, a, b, A_log, dt_bias};
  return decode_step(geo, x, conv_w, conv_state, gates, state, false, z, norm_w, q_scale, l2_eps, rms_eps, out,
                     batch, stream);
}

gdn_status gdn_kda_decode_step(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w,
                               gdn_bf16* conv_state, const float* g, float g_min, const float* beta, float* state,
                               const gdn_bf16* z, const gdn_bf16* norm_w, float q_scale, float l2_eps,
                               float rms_eps, gdn_bf16* out, int32_t batch, void* stream) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (geo->num_v_heads / geo->num_k_heads > gdn::decode_max_ratio())
    return fail(GDN_ERR_UNSUPPORTED_GEOMETRY, "decode supports at most %d V heads per K head",
                gdn::decode_max_ratio());
  if (batch < 0 || batch > 65535) return fail(GDN_ERR_INVALID_ARGUMENT, "batch must be in [0, 65535] (got %d)", batch);
  if (batch == 0) return ok();
  GDN_REQUIRE(x, "x");
  GDN_REQUIRE(conv_w, "conv_w");
  GDN_REQUIRE(conv_state, "conv_state");
  GDN_REQUIRE(g, "g");
  GDN_REQUIRE(state, "state");
  GDN_REQUIRE(z, "z");
  GDN_REQUIRE(norm_w, "norm_w");
  GDN_REQUIRE(out, "out");
  if (!beta) return fail(GDN_ERR_INVALID_ARGUMENT, "beta is NULL");
  if (reinterpret_cast<uintptr_t>(beta) & 3u) return fail(GDN_ERR_MISALIGNED, "beta is not 4-byte aligned");
  if (g_min != g_min) return fail(GDN_ERR_INVALID_ARGUMENT, "g_min is NaN");
  if (!(l2_eps >= 0.f) || !(rms_eps >= 0.f)) return fail(GDN_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  return launched(gdn::launch_kda_decode_step(env, x, conv_w, conv_state, g, g_min, beta, state, z, norm_w, q_scale,
                                              l2_eps, rms_eps, out, batch, geo->num_k_heads, geo->num_v_heads),
                  "KDA decode launch");
}

gdn_status gdn_kda_recurrence(const gdn_geometry* geo, const gdn_bf16* qkv, const float* g, float g_min,
                              const float* beta, const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                              float q_scale, float l2_eps, const float* state_in, float* state_out, const gdn_bf16* z,
                              const gdn_bf16* norm_w, float rms_eps, gdn_bf16* out, void* stream) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (num_seqs < 0 || total_tokens < 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "negative size (num_seqs=%d, total_tokens=%d)", num_seqs, total_tokens);
  if (num_seqs == 0 && total_tokens > 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "total_tokens=%d with no sequence", total_tokens);
  if (num_seqs > 65535) return fail(GDN_ERR_INVALID_ARGUMENT, "num_seqs must be at most 65535 (got %d)", num_seqs);
  if (num_seqs == 0) return ok();
  if (!cu_seqlens) return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens is NULL");
  if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) return fail(GDN_ERR_MISALIGNED, "cu_seqlens is not 4-byte aligned");
  if (total_tokens > 0) {
    GDN_REQUIRE(qkv, "qkv");
    GDN_REQUIRE(g, "g");
    GDN_REQUIRE(out, "out");
    if (!beta) return fail(GDN_ERR_INVALID_ARGUMENT, "beta is NULL");
    if (reinterpret_cast<uintptr_t>(beta) & 3u) return fail(GDN_ERR_MISALIGNED, "beta is not 4-byte aligned");
  }
  GDN_OPTIONAL(state_in, "state_in");
  GDN_OPTIONAL(state_out, "state_out");
  if (z) {
    GDN_REQUIRE(z, "z");
    GDN_REQUIRE(norm_w, "norm_w");
  }
  if (g_min != g_min) return fail(GDN_ERR_INVALID_ARGUMENT, "g_min is NaN");
  if (!(l2_eps >= 0.f) || !(rms_eps >= 0.f)) return fail(GDN_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  if (state_in && state_out && state_in != state_out) {
    const size_t sb = (size_t)num_seqs * geo->num_v_heads * gdn::kHeadDim * gdn::kHeadDim * 4;
    if (overlaps(state_in, sb, state_out, sb))
      return fail(GDN_ERR_INVALID_ARGUMENT, "state_out partially overlaps state_in");
  }
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  return launched(gdn::launch_kda_prefill(env, qkv, g, g_min, beta, cu_seqlens, num_seqs, total_tokens,
                                          geo->num_k_heads, geo->num_v_heads, q_scale, l2_eps, state_in, state_out,
                                          z, norm_w, rms_eps, out),
                  "KDA recurrence launch");
}

size_t gdn_kda_chunk_prefill_workspace_size(const gdn_geometry* geo, int32_t num_seqs, int32_t total_tokens) {
  if (!geo || num_seqs <= 0 || total_tokens < 0 || geo->num_v_heads <= 0) return 0;
  return gdn::kda_chunk_workspace_bytes(num_seqs, total_tokens, geo->num_v_heads);
}

static gdn_status kda_chunk_prefill(const gdn_geometry* geo, const gdn_bf16* qkv, const float* g, float g_min,
                                 const float* beta, const int32_t* cu_seqlens, int32_t num_seqs,
                                 int32_t total_tokens, float q_scale, float l2_eps, const float* state_in,
                                 float* state_out, const gdn_bf16* z, const gdn_bf16* norm_w, float rms_eps,
                                 gdn_bf16* out, void* workspace, size_t workspace_bytes, void* stream,
                                 const ConvStage* conv = nullptr) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (num_seqs < 0 || total_tokens < 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "negative size (num_seqs=%d, total_tokens=%d)", num_seqs, total_tokens);
  if (num_seqs == 0 && total_tokens > 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "total_tokens=%d with no sequence", total_tokens);
  if ((long)num_seqs * geo->num_v_heads > 0x7FFFFFFFL)
    return fail(GDN_ERR_INVALID_ARGUMENT, "num_seqs * num_v_heads exceeds the grid limit");
  if (num_seqs == 0) return ok();
  if (!cu_seqlens) return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens is NULL");
  if (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) return fail(GDN_ERR_MISALIGNED, "cu_seqlens is not 4-byte aligned");
  if (total_tokens > 0) {
    GDN_REQUIRE(qkv, "qkv");
    GDN_REQUIRE(g, "g");
    GDN_REQUIRE(out, "out");
    if (!beta) return fail(GDN_ERR_INVALID_ARGUMENT, "beta is NULL");
    if (reinterpret_cast<uintptr_t>(beta) & 3u) return fail(GDN_ERR_MISALIGNED, "beta is not 4-byte aligned");
  }
  GDN_OPTIONAL(state_in, "state_in");
  GDN_OPTIONAL(state_out, "state_out");
  if (z) {
    GDN_REQUIRE(z, "z");
    GDN_REQUIRE(norm_w, "norm_w");
  }
  if (g_min != g_min) return fail(GDN_ERR_INVALID_ARGUMENT, "g_min is NaN");
  if (!(l2_eps >= 0.f) || !(rms_eps >= 0.f)) return fail(GDN_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  const size_t need = gdn_kda_chunk_prefill_workspace_size(geo, num_seqs, total_tokens);
  if (!workspace || workspace_bytes < need)
    return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need, workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(GDN_ERR_MISALIGNED, "workspace is not 256-byte aligned");
  if (state_in && state_out && state_in != state_out) {
    const size_t sb = (size_t)num_seqs * geo->num_v_heads * gdn::kHeadDim * gdn::kHeadDim * 4;
    if (overlaps(state_in, sb, state_out, sb))
      return fail(GDN_ERR_INVALID_ARGUMENT, "state_out partially overlaps state_in");
  }
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  if (conv && (total_tokens > 0 || conv->state_out)) {  // every argument checked: the conv stage first
    s = launched(gdn::launch_conv1d_prefill(env, conv->x, conv->w, cu_seqlens, num_seqs, total_tokens, conv->C,
                                            conv->state_in, conv->state_out, const_cast<gdn_bf16*>(qkv)),
                 "conv1d launch");
    if (s != GDN_OK) return s;
  }
  return launched(gdn::launch_kda_chunk_prefill(env, qkv, g, g_min, beta, cu_seqlens, num_seqs, total_tokens,
                                                geo->num_k_heads, geo->num_v_heads, q_scale, l2_eps, state_in,
                                                state_out, z, norm_w, rms_eps, out, workspace),
                  "KDA chunk prefill launch");
}

gdn_status gdn_kda_chunk_prefill(const gdn_geometry* geo, const gdn_bf16* qkv, const float* g, float g_min,
                                 const float* beta, const int32_t* cu_seqlens, int32_t num_seqs,
                                 int32_t total_tokens, float q_scale, float l2_eps, const float* state_in,
                                 float* state_out, const gdn_bf16* z, const gdn_bf16* norm_w, float rms_eps,
                                 gdn_bf16* out, void* workspace, size_t workspace_bytes, void* stream) {
  return kda_chunk_prefill(geo, qkv, g, g_min, beta, cu_seqlens, num_seqs, total_tokens, q_scale, l2_eps, state_in,
                           state_out, z, norm_w, rms_eps, out, workspace, workspace_bytes, stream);
}

gdn_status gdn_kda_prefill(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w,
                           const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                           const gdn_bf16* conv_state_in, gdn_bf16* conv_state_out, gdn_bf16* qkv, const float* g,
                           float g_min, const float* beta, float q_scale, float l2_eps, const float* state_in,
                           float* state_out, const gdn_bf16* z, const gdn_bf16* norm_w, float rms_eps,
                           gdn_bf16* out, void* workspace, size_t workspace_bytes, void* stream) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (num_seqs > 0) {  // the conv stage's own arguments (the chunk stage checks the rest)
    GDN_REQUIRE(conv_w, "conv_w");
    GDN_OPTIONAL(conv_state_in, "conv_state_in");
    GDN_OPTIONAL(conv_state_out, "conv_state_out");
    if (total_tokens > 0) {
      GDN_REQUIRE(x, "x");
      GDN_REQUIRE(qkv, "qkv");
      const size_t bytes = (size_t)total_tokens * conv_channels(geo) * 2;
      if (overlaps(x, bytes, qkv, bytes)) return fail(GDN_ERR_INVALID_ARGUMENT, "qkv overlaps x");
    }
  }
  const ConvStage conv = {x, conv_w, conv_state_in, conv_state_out, conv_channels(geo)};
  return kda_chunk_prefill(geo, qkv, g, g_min, beta, cu_seqlens, num_seqs, total_tokens, q_scale, l2_eps, state_in,
                           state_out, z, norm_w, rms_eps, out, workspace, workspace_bytes, stream, &conv);
}

gdn_status gdn_decode_step_fp16_state(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w,
                                      gdn_bf16* conv_state, const float* g, const float* beta, gdn_f16* state,
                                      const gdn_bf16* z, const gdn_bf16* norm_w, float q_scale, float l2_eps,
                                      float rms_eps, gdn_bf16* out, int32_t batch, void* stream) {
  const gdn::GateSrc gates = {g, beta, nullptr, nullptr, nullptr, nullptr};
  return decode_step(geo, x, conv_w, conv_state, gates, state, true, z, norm_w, q_scale, l2_eps, rms_eps, out,
                     batch, stream);
}

gdn_status gdn_gates(const gdn_geometry* geo, const gdn_bf16* a, const gdn_bf16* b, const float* A_log,
                     const float* dt_bias, float* g, float* beta, int32_t rows, void* stream) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (rows < 0) return fail(GDN_ERR_INVALID_ARGUMENT, "negative rows");
  if (rows == 0) return ok();
  GDN_REQUIRE(a, "a");
  GDN_REQUIRE(b, "b");
  GDN_REQUIRE(g, "g");
  GDN_REQUIRE(beta, "beta");
  if (!A_log || !dt_bias) return fail(GDN_ERR_INVALID_ARGUMENT, "A_log or dt_bias is NULL");
  if ((reinterpret_cast<uintptr_t>(A_log) | reinterpret_cast<uintptr_t>(dt_bias)) & 3u)
    return fail(GDN_ERR_MISALIGNED, "A_log or dt_bias is not 4-byte aligned");
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  return launched(gdn::launch_gates(env, a, b, A_log, dt_bias, g, beta, rows, geo->num_v_heads), "gates launch");
}

size_t gdn_verify_stash_size(const gdn_geometry* geo, int32_t batch, int32_t rows) {
  if (check_geometry(geo) != GDN_OK || batch < 0 || rows < 1 || rows > gdn::kMaxVerifyRows) return 0;
  const int C = 2 * geo->num_k_heads * gdn::kHeadDim + geo->num_v_heads * gdn::kHeadDim;
  return (size_t)batch * rows * gdn::verify_stash_layout(C, geo->num_k_heads, geo->num_v_heads).bytes;
}

}  // extern "C"

namespace {
gdn_status check_verify_shape(const gdn_geometry* geo, int32_t batch, int32_t rows) {
  gdn_status s = check_geometry(geo);
  if (s != GDN_OK) return s;
  if (batch < 0 || batch > 65535) return fail(GDN_ERR_INVALID_ARGUMENT, "batch must be in [0, 65535] (got %d)", batch);
  if (rows < 1 || rows > gdn::kMaxVerifyRows)
    return fail(GDN_ERR_INVALID_ARGUMENT, "rows must be in [1, %d] (got %d)", gdn::kMaxVerifyRows, rows);
  if (!gdn::verify_supported(rows, geo->num_k_heads, geo->num_v_heads))
    return fail(GDN_ERR_UNSUPPORTED_GEOMETRY, "%d rows with %d V heads per K head exceed the verify kernel's shared memory",
                rows, geo->num_v_heads / geo->num_k_heads);
  return GDN_OK;
}

gdn_status verify(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w, const gdn_bf16* conv_state,
                  const float* g, const float* beta, const void* state, bool fp16_state, const gdn_bf16* z,
                  const gdn_bf16* norm_w, float q_scale, float l2_eps, float rms_eps, gdn_bf16* out, int32_t batch,
                  int32_t rows, void* stash, size_t stash_bytes, void* stream) {
  gdn_status s = check_verify_shape(geo, batch, rows);
  if (s != GDN_OK) return s;
  if (batch == 0) return ok();
  GDN_REQUIRE(x, "x");
  GDN_REQUIRE(conv_w, "conv_w");
  GDN_REQUIRE(conv_state, "conv_state");
  GDN_REQUIRE(state, "state");
  GDN_REQUIRE(z, "z");
  GDN_REQUIRE(norm_w, "norm_w");
  GDN_REQUIRE(out, "out");
  GDN_REQUIRE(stash, "stash");
  if (!g || !beta) return fail(GDN_ERR_INVALID_ARGUMENT, "g or beta is NULL");
  if ((reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(beta)) & 3u)
    return fail(GDN_ERR_MISALIGNED, "g or beta is not 4-byte aligned");
  if (!(l2_eps >= 0.f) || !(rms_eps >= 0.f)) return fail(GDN_ERR_INVALID_ARGUMENT, "eps must be >= 0");
  const size_t need = gdn_verify_stash_size(geo, batch, rows);
  if (stash_bytes < need) return fail(GDN_ERR_WORKSPACE, "stash of %zu bytes required (got %zu)", need, stash_bytes);
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  return launched(gdn::launch_verify(env, x, conv_w, conv_state, g, beta, state, fp16_state, z, norm_w, q_scale,
                                     l2_eps, rms_eps, out, stash, batch, rows, geo->num_k_heads, geo->num_v_heads),
                  "verify launch");
}

gdn_status verify_commit(const gdn_geometry* geo, const int32_t* committed_rows, const void* stash,
                         size_t stash_bytes, gdn_bf16* conv_state, void* state, bool fp16_state, int32_t batch,
                         int32_t rows, void* stream) {
  gdn_status s = check_verify_shape(geo, batch, rows);
  if (s != GDN_OK) return s;
  if (batch == 0) return ok();
  if (!committed_rows) return fail(GDN_ERR_INVALID_ARGUMENT, "committed_rows is NULL");
  if (reinterpret_cast<uintptr_t>(committed_rows) & 3u)
    return fail(GDN_ERR_MISALIGNED, "committed_rows is not 4-byte aligned");
  GDN_REQUIRE(stash, "stash");
  GDN_REQUIRE(conv_state, "conv_state");
  GDN_REQUIRE(state, "state");
  const size_t need = gdn_verify_stash_size(geo, batch, rows);
  if (stash_bytes < need)
    return fail(GDN_ERR_WORKSPACE, "stash of %zu bytes required for batch %d x rows %d (got %zu)", need, batch, rows,
                stash_bytes);
  gdn::LaunchEnv env;
  if ((s = make_env(stream, &env)) != GDN_OK) return s;
  return launched(gdn::launch_verify_commit(env, committed_rows, stash, conv_state, state, fp16_state, batch, rows,
                                            geo->num_k_heads, geo->num_v_heads),
                  "verify commit launch");
}
}  // namespace

extern "C" {

gdn_status gdn_verify(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w, const gdn_bf16* conv_state,
                      const float* g, const float* beta, const float* state, const gdn_bf16* z,
                      const gdn_bf16* norm_w, float q_scale, float l2_eps, float rms_eps, gdn_bf16* out,
                      int32_t batch, int32_t rows, void* stash, size_t stash_bytes, void* stream) {
  return verify(geo, x, conv_w, conv_state, g, beta, state, false, z, norm_w, q_scale, l2_eps, rms_eps, out, batch,
                rows, stash, stash_bytes, stream);
}

gdn_status gdn_verify_fp16_state(const gdn_geometry* geo, const gdn_bf16* x, const gdn_bf16* conv_w,
                                 const gdn_bf16* conv_state, const float* g, const float* beta, const gdn_f16* state,
                                 const gdn_bf16* z, const gdn_bf16* norm_w, float q_scale, float l2_eps,
                                 float rms_eps, gdn_bf16* out, int32_t batch, int32_t rows, void* stash,
                                 size_t stash_bytes, void* stream) {
  return verify(geo, x, conv_w, conv_state, g, beta, state, true, z, norm_w, q_scale, l2_eps, rms_eps, out, batch,
                rows, stash, stash_bytes, stream);
}

gdn_status gdn_verify_commit(const gdn_geometry* geo, const int32_t* committed_rows, const void* stash,
                             size_t stash_bytes, gdn_bf16* conv_state, float* state, int32_t batch, int32_t rows,
                             void* stream) {
  return verify_commit(geo, committed_rows, stash, stash_bytes, conv_state, state, false, batch, rows, stream);
}

gdn_status gdn_verify_commit_fp16_state(const gdn_geometry* geo, const int32_t* committed_rows, const void* stash,
                                        size_t stash_bytes, gdn_bf16* conv_state, gdn_f16* state, int32_t batch,
                                        int32_t rows, void* stream) {
  return verify_commit(geo, committed_rows, stash, stash_bytes, conv_state, state, true, batch, rows, stream);
}

// ---- allocation-free chunk prefill: the schedule lives in a fixed device array of this file
}  // extern "C"

namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];
// The array's device address per device index (the first call on a device looks it up; racing
// first calls store the same address).  It is not refreshed after cudaDeviceReset.
std::atomic<void*> g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

extern "C" {

gdn_status gdn_chunk_prefill_noalloc(const gdn_geometry* geo, const gdn_bf16* qkv, const float* g,
                                     const float* beta, const int32_t* cu_seqlens, int32_t num_seqs,
                                     int32_t total_tokens, float q_scale, float l2_eps, const float* state_in,
                                     float* state_out, const gdn_bf16* z, const gdn_bf16* norm_w, float rms_eps,
                                     gdn_bf16* out, void* stream) {
  if (num_seqs > GDN_NOALLOC_MAX_SEQS)
    return fail(GDN_ERR_INVALID_ARGUMENT, "num_seqs=%d exceeds the %d sequences of the fixed scratch", num_seqs,
                GDN_NOALLOC_MAX_SEQS);
  if (gdn_chunk_prefill_min_workspace_size(geo, num_seqs, total_tokens) > GDN_NOALLOC_SCRATCH_BYTES)
    return fail(GDN_ERR_INVALID_ARGUMENT, "the fixed scratch is too small for num_seqs=%d", num_seqs);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_CUDA, "device index %d out of range", dev);
  void* scratch = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (!scratch) {
    // host code only sees a stand-in for the array: its device address comes from the runtime
    e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess || !scratch)
      return fail(GDN_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev].store(scratch, std::memory_order_release);
  }
  return gdn_chunk_prefill(geo, qkv, g, beta, cu_seqlens, num_seqs, total_tokens, q_scale, l2_eps, state_in,
                           state_out, z, norm_w, rms_eps, out, scratch, GDN_NOALLOC_SCRATCH_BYTES, stream);
}

gdn_status gdn_check_device_errors(void* stream) {
  gdn::LaunchEnv env;
  gdn_status s = make_env(stream, &env);
  if (s != GDN_OK) return s;
  cudaError_t e = cudaStreamSynchronize(env.stream);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned word = 0;
  e = cudaMemcpy(&word, env.err, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
  if (word) {
    const unsigned zero = 0;
    e = cudaMemcpy(env.err, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "clearing the device error word: %s", cudaGetErrorString(e));
  }
  if (word & gdn::kErrTimeout) return fail(GDN_ERR_TIMEOUT, "an in-kernel wait ran out (word 0x%x)", word);
  if (word & gdn::kErrDeviceArgument)
    return fail(GDN_ERR_DEVICE_ARGUMENT, "a kernel rejected cu_seqlens contents (word 0x%x)", word);
  return ok();
}

#ifdef GDN_TEST_HOOKS
gdn_status gdn_debug_set_chunk_mode(int mode) {
  if (mode < 0 || mode > 2) return fail(GDN_ERR_INVALID_ARGUMENT, "mode must be 0, 1 or 2");
  g_chunk_mode.store(mode);
  return ok();
}

int gdn_debug_get_chunk_mode(void) { return g_chunk_mode.load(); }

gdn_status gdn_debug_set_dropped_copy(unsigned which) {
  if (which & ~3u) return fail(GDN_ERR_INVALID_ARGUMENT, "which must be a combination of bits 0 and 1");
  cudaError_t e = gdn::test_set_dropped_copy_decode(which & 1u);
  if (e == cudaSuccess) e = gdn::test_set_dropped_copy_chunk((which >> 1) & 1u);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "setting the dropped-copy hook: %s", cudaGetErrorString(e));
  return ok();
}
#endif

}  // extern "C"
