// gdn_kernels.h -- internal launch functions of the GDN kernels (host side of each .cu file).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_common.cuh"

namespace gdn {

cudaError_t launch_conv1d_prefill(const LaunchEnv& env, const uint16_t* x, const uint16_t* w, const int32_t* cu,
                                  int N, int T, int C, const uint16_t* state_in, uint16_t* state_out,
                                  uint16_t* y);

cudaError_t launch_gated_rmsnorm(const LaunchEnv& env, const uint16_t* o, const uint16_t* z, const uint16_t* w,
                                 float eps, uint16_t* out, long rows);

cudaError_t launch_gates(const LaunchEnv& env, const uint16_t* a, const uint16_t* b, const float* A_log,
                         const float* dt_bias, float* g, float* beta, long rows, int hv);

int decode_max_ratio();
// The KDA decode step: g is [B, Hv, Dk], a log decay per key channel, clamped below at g_min.
cudaError_t launch_kda_decode_step(const LaunchEnv& env, const uint16_t* x, const uint16_t* conv_w,
                                   uint16_t* conv_state, const float* g, float g_min, const float* beta,
                                   float* state, const uint16_t* z, const uint16_t* norm_w, float q_scale,
                                   float l2_eps, float rms_eps, uint16_t* out, int B, int Hk, int Hv);
cudaError_t launch_decode_step(const LaunchEnv& env, const uint16_t* x, const uint16_t* conv_w,
                               uint16_t* conv_state, const GateSrc& gates, void* state,
                               bool fp16_state, const uint16_t* z, const uint16_t* norm_w, float q_scale,
                               float l2_eps, float rms_eps, uint16_t* out, int B, int Hk, int Hv);

// The KDA recurrence over packed sequences (kda_prefill.cu): qkv is the conv output [T, C], g the
// per-channel log decay [T, Hv, Dk], clamped below at g_min; out receives the gated RMSNorm of o
// (o itself when z is NULL); state_out may be state_in.
size_t kda_prefill_smem_bytes();
cudaError_t launch_kda_prefill(const LaunchEnv& env, const uint16_t* qkv, const float* g, float g_min,
                               const float* beta, const int32_t* cu, int N, int T, int Hk, int Hv, float q_scale,
                               float l2_eps, const float* state_in, float* state_out, const uint16_t* z,
                               const uint16_t* norm_w, float rms_eps, uint16_t* out);
// The KDA recurrence in its chunk-wise form (kda_chunk.cu): same arguments and results as
// launch_kda_prefill (g finite after the clamp), plus a workspace of kda_chunk_workspace_bytes().
size_t kda_chunk_workspace_bytes(int N, int T, int Hv);
cudaError_t launch_kda_chunk_prefill(const LaunchEnv& env, const uint16_t* qkv, const float* g, float g_min,
                                     const float* beta, const int32_t* cu, int N, int T, int Hk, int Hv,
                                     float q_scale, float l2_eps, const float* state_in, float* state_out,
                                     const uint16_t* z, const uint16_t* norm_w, float rms_eps, uint16_t* out,
                                     void* workspace);

// Multi-token verify (verify.cu): K rows per sequence, the state read only; the commit folds an
// accepted prefix of rows into the recurrent and conv states.
constexpr int kMaxVerifyRows = 17;
constexpr size_t kMaxVerifySmem = 110 * 1024;  // two verify CTAs per SM
// One stash record per (sequence, row): the row's raw conv inputs (C bf16), its normalised keys
// (Hk x 128 fp32), the delta e = beta (v - decayed state . k) of every V head and value row
// (Hv x 128 fp32) and g (Hv fp32); records are 16-byte multiples, record (b, r) at
// (b * K + r) * bytes.
struct VerifyStash {
  size_t x_off, khat_off, e_off, g_off, bytes;
};
__host__ __device__ inline VerifyStash verify_stash_layout(int C, int Hk, int Hv) {
  VerifyStash L;
  L.x_off = 0;
  L.khat_off = (size_t)C * 2;
  L.e_off = L.khat_off + (size_t)Hk * kHeadDim * 4;
  L.g_off = L.e_off + (size_t)Hv * kHeadDim * 4;
  L.bytes = (L.g_off + (size_t)Hv * 4 + 15) & ~(size_t)15;
  return L;
}
int verify_max_rows();
bool verify_supported(int K, int Hk, int Hv);
cudaError_t launch_verify(const LaunchEnv& env, const uint16_t* x, const uint16_t* conv_w, const uint16_t* conv_state,
                          const float* g, const float* beta, const void* state, bool fp16_state, const uint16_t* z,
                          const uint16_t* norm_w, float q_scale, float l2_eps, float rms_eps, uint16_t* out,
                          void* stash, int B, int K, int Hk, int Hv);
cudaError_t launch_verify_commit(const LaunchEnv& env, const int32_t* committed, const void* stash,
                                 uint16_t* conv_state, void* state, bool fp16_state, int B, int K, int Hk, int Hv);

// Workspace of the fused chunk prefill: a work counter and the longest-first sequence order.
size_t chunk_prefill_workspace_bytes(int N);
// Workspace of the split chunk prefill (prep kernel + state kernel): the above, per-sequence
// chunk offsets, and per-chunk operand images (K^T per K head; T, P and per-token factors per
// V head).
size_t split_workspace_bytes(int N, int T, int Hk, int Hv);

cudaError_t device_sm_count(int* sms);
// Tiled 2D tensor map of a row-major bf16 matrix (no swizzle, zero fill out of bounds).
cudaError_t encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                          uint32_t box_inner, uint32_t box_outer);
// Tiled 2D tensor map of a row-major fp32 matrix (no swizzle, zero fill out of bounds).
cudaError_t encode_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_outer);
cudaError_t encode_chunk_tensor_maps(CUtensorMap* qkv_map, CUtensorMap* z_map, const uint16_t* qkv,
                                     const uint16_t* z, int T, int Hk, int Hv);
cudaError_t launch_chunk_schedule(cudaStream_t stream, const int32_t* cu, int N, int32_t* order, unsigned* counter,
                                  int32_t* chunk_off);

// mode 0: tensor cores, split path when the workspace holds it (else fused); mode 1: fused, MMAs
// emulated on CUDA cores; mode 2: fused, tensor cores.
cudaError_t launch_chunk_prefill(const LaunchEnv& env, int mode, const uint16_t* qkv, const GateSrc& gates,
                                 const int32_t* cu, int N, int T, int Hk, int Hv, float q_scale,
                                 float l2_eps, const float* state_in, float* state_out, const uint16_t* z,
                                 const uint16_t* norm_w, float rms_eps, uint16_t* out, void* workspace,
                                 size_t workspace_bytes);
cudaError_t launch_chunk_prefill_split(const LaunchEnv& env, const uint16_t* qkv, const GateSrc& gates,
                                       const int32_t* cu, int N, int T, int Hk, int Hv, float q_scale, float l2_eps,
                                       const float* state_in, float* state_out, const uint16_t* z,
                                       const uint16_t* norm_w, float rms_eps, uint16_t* out, void* workspace);

#ifdef GDN_TEST_HOOKS
// Test library only: while set (1), the copy named below is not issued although its barrier is
// armed for its bytes, so the bounded wait on it runs out (with a short limit) and the kernel reports
// a timeout -- nothing is in flight when the CTA leaves.  Set for the current device.
cudaError_t test_set_dropped_copy_decode(unsigned on);  // the binary16 decode step's state-slice copy
cudaError_t test_set_dropped_copy_chunk(unsigned on);   // the chunk state kernel's first vector-block copy
#endif

}  // namespace gdn
