// decode.cu -- one fused GDN decode step: conv step + SiLU, L2 norm of q/k, gated delta rule
// update of the recurrent state in place (fp32, or fp16 in memory), sigmoid-gated RMSNorm.
//
// Qwen3.8 kernel architecture and TDD ledger, "Current dense-27B kernel map" (scalar GDN
// recurrence and fused output gate); spark_model layer_struct.rs, fields of the strided decode
// kernels (one launch for all sequences; the state read once and written once, 1R+1W);
// GLM-5.3-Flash kernel TDD ledger, slice I3 (a conv step equals the full width-4 causal conv);
// Qwen3.8 ledger, the FP16 h-state twins of the decode kernels (same arithmetic as the fp32
// kernel, the state half precision in memory, rounded once per token); GLM ledger slice I2 (the
// KDA step: the same update with a decay per key channel, clamped and exponentiated).
//
// The conv outputs are rounded to the bf16 nearest the exact value (silu_bf16_rn).
//
// With a binary16 state the CTA's state slice (96 KB) is staged in shared memory by one bulk copy
// issued at the start, so it streams in while the conv step and the norms run.
//
// One CTA per (sequence, K head): it owns the q/k channels of that K head and the v channels of
// the Hv/Hk V heads that read it, so no two CTAs touch the same conv-state channel and the
// in-place conv-state update is race-free.  Each warp streams 16 rows ([value] index) of a
// head's 128 x 128 state: a row is 32 lanes x float4 over the key dimension, so both
// contractions (S k and S q) are warp-shuffle reductions (a halving butterfly: 16 shuffles for
// the 16 rows' sums) and every state byte is read once and written once.
#include <cuda_fp16.h>
#include <string.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerWarp = kHeadDim / (kThreads / 32);  // 16
constexpr int kMaxRatio = 12;                             // V heads per K head handled by one CTA
constexpr uint32_t kStateWaitLimit = 1u << 20;            // polls of the state-slice barrier
constexpr size_t kMaxStagedBytes = 96 * 1024;             // largest state slice staged in shared memory

#ifdef GDN_TEST_HOOKS
constexpr uint32_t kTestWaitLimit = 1u << 12;  // polls of a wait whose copy the hook dropped
__device__ unsigned g_test_drop_state_copy;    // 1: the staged state copy is not issued
#endif

// Four consecutive state elements of a row (index i counts groups of four), widened to fp32.  The
// fp16 storage form holds the state as IEEE binary16 in memory only: it is widened on load, the
// step runs in fp32 exactly as for the fp32 state, and the new state is rounded once (to nearest,
// ties to even) when it is stored.
__device__ __forceinline__ float4 load_state4(const float* S, int i) { return reinterpret_cast<const float4*>(S)[i]; }
__device__ __forceinline__ float4 load_state4(const __half* S, int i) {
  const uint2 u = reinterpret_cast<const uint2*>(S)[i];
  __half2 h01, h23;
  memcpy(&h01, &u.x, 4);
  memcpy(&h23, &u.y, 4);
  const float2 a = __half22float2(h01), b = __half22float2(h23);
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store_state4(float* S, int i, const float4 v) { reinterpret_cast<float4*>(S)[i] = v; }
__device__ __forceinline__ void store_state4(__half* S, int i, const float4 v) {
  const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  uint2 u;
  memcpy(&u.x, &a, 4);
  memcpy(&u.y, &b, 4);
  reinterpret_cast<uint2*>(S)[i] = u;
}

// Sums v[0..15] over the 32 lanes of a warp in 16 shuffles (a halving butterfly: at each of the
// five levels a lane keeps half of its values and adds its partner's copy of that half).  Every
// total is formed by the same pairwise additions as five xor-shuffle levels applied to each value
// on its own, so it has the same bits.  Lanes 2i and 2i + 1 return the total of v[i].
__device__ __forceinline__ float warp_sum16(const float (&v)[16], int lane) {
  float a[8], b4[4], c2[2];
  const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    a[k] = (h16 ? v[8 + k] : v[k]) + __shfl_xor_sync(0xffffffffu, h16 ? v[k] : v[8 + k], 16);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    b4[k] = (h8 ? a[4 + k] : a[k]) + __shfl_xor_sync(0xffffffffu, h8 ? a[k] : a[4 + k], 8);
#pragma unroll
  for (int k = 0; k < 2; ++k)
    c2[k] = (h4 ? b4[2 + k] : b4[k]) + __shfl_xor_sync(0xffffffffu, h4 ? b4[k] : b4[2 + k], 4);
  const float s = (h2 ? c2[1] : c2[0]) + __shfl_xor_sync(0xffffffffu, h2 ? c2[0] : c2[1], 2);
  return s + __shfl_xor_sync(0xffffffffu, s, 1);
}

// kStaged: the CTA's whole state slice (its R V heads, contiguous in [B, Hv, Dv, Dk]) is fetched
// into shared memory by one bulk copy issued before the conv step, so the state bytes are in
// flight while the conv and the norms are computed; the rows are then read from shared memory.
// Used when the slice fits (binary16 state, R <= 3: 96 KB).  Otherwise rows stream from global.
// kPerChannel: the KDA form -- gates.g is [B, Hv, Dk], a log decay per key channel, applied as
// exp(max(g, g_min)) to the state's key columns (GLM-5.3-Flash kernel TDD ledger, slice I2);
// otherwise one decay per head (the GDN step), read from gates.g [B, Hv] or derived from the
// projections a, b and A_log, dt_bias (load_gate) once per CTA, beside the conv step.
template <typename StateT, bool kStaged, bool kPerChannel = false>
__global__ void __launch_bounds__(kThreads, 2) decode_step_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ conv_w, uint16_t* conv_state,
    const GateSrc gates, StateT* state,
    const uint16_t* __restrict__ z, const uint16_t* __restrict__ norm_w, float q_scale, float l2_eps,
    float rms_eps, uint16_t* __restrict__ out, int Hk, int Hv, unsigned* err, float g_min = 0.f) {
  const int j = blockIdx.x;        // K head
  const int b = blockIdx.y;        // sequence
  const int R = Hv / Hk;
  const int C = 2 * Hk * kHeadDim + Hv * kHeadDim;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  __shared__ float s_q[kHeadDim], s_k[kHeadDim];
  __shared__ float s_v[kMaxRatio][kHeadDim];
  __shared__ float s_o[kMaxRatio][kHeadDim];
  __shared__ float s_norm[2];
  __shared__ float s_alpha[kMaxRatio], s_bt[kMaxRatio];  // the GDN step's per-head decay and beta
  __shared__ uint64_t s_bar;
  extern __shared__ __align__(128) uint8_t s_state[];  // kStaged: R x Dv x Dk StateT

  StateT* const slice = state + ((size_t)b * Hv + (size_t)j * R) * kHeadDim * kHeadDim;
  if constexpr (kStaged) {
    if (tid == 0) {
      const uint32_t bar = smem_u32(&s_bar);
      mbar_init(bar, 1);
      fence_mbar_init();
      const uint32_t bytes = (uint32_t)((size_t)R * kHeadDim * kHeadDim * sizeof(StateT));
      mbar_arrive_expect_tx(bar, bytes);
#ifdef GDN_TEST_HOOKS
      if (!g_test_drop_state_copy)
#endif
        bulk_load(smem_u32(s_state), slice, bytes, bar);
    }
  }

  if constexpr (!kPerChannel) {  // the gates of the CTA's R V heads (visible after the conv's barrier)
    if (tid < R) {
      float gg, bt;
      load_gate(gates, (size_t)b * Hv + j * R + tid, j * R + tid, gg, bt);
      s_alpha[tid] = expf(gg);
      s_bt[tid] = bt;
    }
  }

  // ---- conv step + SiLU for the CTA's 256 + 128R channels, one channel pair per thread and round
  const int n_pairs = (2 + R) * (kHeadDim / 2);
  for (int t = tid; t < n_pairs; t += kThreads) {
    int c;
    float* dst;
    if (t < 64) { c = j * kHeadDim + 2 * t; dst = s_q + 2 * t; }
    else if (t < 128) { c = Hk * kHeadDim + j * kHeadDim + 2 * (t - 64); dst = s_k + 2 * (t - 64); }
    else {
      const int hh = (t - 128) >> 6, o = (t - 128) & 63;
      c = 2 * Hk * kHeadDim + (j * R + hh) * kHeadDim + 2 * o;
      dst = s_v[hh] + 2 * o;
    }
    const uint32_t xu = __ldg(reinterpret_cast<const uint32_t*>(x + (size_t)b * C + c));
    const uint4 wu = __ldg(reinterpret_cast<const uint4*>(conv_w + (size_t)c * kConvWidth));  // [2][4] taps
    // conv state of channels c, c + 1: [2][3] bf16 in three 32-bit words, oldest slot first
    uint32_t* sp = reinterpret_cast<uint32_t*>(conv_state + ((size_t)b * C + c) * (kConvWidth - 1));
    const uint32_t s0 = sp[0], s1 = sp[1], s2 = sp[2];
    const float xa = __uint_as_float(xu << 16), xb = __uint_as_float(xu & 0xFFFF0000u);
    const float wa[4] = {__uint_as_float(wu.x << 16), __uint_as_float(wu.x & 0xFFFF0000u),
                         __uint_as_float(wu.y << 16), __uint_as_float(wu.y & 0xFFFF0000u)};
    const float wb[4] = {__uint_as_float(wu.z << 16), __uint_as_float(wu.z & 0xFFFF0000u),
                         __uint_as_float(wu.w << 16), __uint_as_float(wu.w & 0xFFFF0000u)};
    const float sa[3] = {__uint_as_float(s0 << 16), __uint_as_float(s0 & 0xFFFF0000u), __uint_as_float(s1 << 16)};
    const float sb[3] = {__uint_as_float(s1 & 0xFFFF0000u), __uint_as_float(s2 << 16), __uint_as_float(s2 & 0xFFFF0000u)};
    // the bf16 conv outputs, rounded as the exact values are
    dst[0] = bf2f(silu_bf16_rn(wa[0], sa[0], wa[1], sa[1], wa[2], sa[2], wa[3], xa));
    dst[1] = bf2f(silu_bf16_rn(wb[0], sb[0], wb[1], sb[1], wb[2], sb[2], wb[3], xb));
    // the shift register: [s1, s2, x] per channel (exact: bf16 values)
    sp[0] = pack_bf2(sa[1], sa[2]);
    sp[1] = pack_bf2(xa, sb[1]);
    sp[2] = pack_bf2(sb[2], xb);
  }
  __syncthreads();

  // ---- L2 norms of q and k: x / sqrt(sum x^2 + eps)
  if (warp < 2) {
    const float* src = warp == 0 ? s_q : s_k;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) { const float v = src[lane * 4 + i]; ss = fmaf(v, v, ss); }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if (lane == 0) s_norm[warp] = rsqrtf(ss + l2_eps);
  }
  __syncthreads();
  const float4 qn = make_float4(s_q[lane * 4] * s_norm[0], s_q[lane * 4 + 1] * s_norm[0],
                                s_q[lane * 4 + 2] * s_norm[0], s_q[lane * 4 + 3] * s_norm[0]);
  const float4 kn = make_float4(s_k[lane * 4] * s_norm[1], s_k[lane * 4 + 1] * s_norm[1],
                                s_k[lane * 4 + 2] * s_norm[1], s_k[lane * 4 + 3] * s_norm[1]);

  if constexpr (kStaged) {  // the state slice has landed in shared memory (bounded wait)
#ifdef GDN_TEST_HOOKS
    const uint32_t limit = g_test_drop_state_copy ? kTestWaitLimit : kStateWaitLimit;
#else
    const uint32_t limit = kStateWaitLimit;
#endif
    const bool got = mbar_wait(smem_u32(&s_bar), 0, limit);
    if (!got) raise_error(err, kErrTimeout);
    if (!__syncthreads_and(got ? 1 : 0)) {
      if (!got) mbar_wait(smem_u32(&s_bar), 0, limit);  // let the copy land before leaving
      return;
    }
  }

  // ---- state update, one V head at a time
  for (int hh = 0; hh < R; ++hh) {
    const int h = j * R + hh;
    float4 a4, kd;  // the decay of this lane's four key channels; the key they multiply (decayed)
    float bt;
    if constexpr (kPerChannel) {
      const float4 gv = __ldg(reinterpret_cast<const float4*>(gates.g + ((size_t)b * Hv + h) * kHeadDim) + lane);
      a4 = make_float4(expf(fmaxf(gv.x, g_min)), expf(fmaxf(gv.y, g_min)), expf(fmaxf(gv.z, g_min)),
                       expf(fmaxf(gv.w, g_min)));
      kd = make_float4(a4.x * kn.x, a4.y * kn.y, a4.z * kn.z, a4.w * kn.w);  // (S diag(a)) k = S (a * k)
      bt = __ldg(gates.beta + (size_t)b * Hv + h);
    } else {
      const float alpha = s_alpha[hh];
      a4 = make_float4(alpha, alpha, alpha, alpha);
      kd = kn;
      bt = s_bt[hh];
    }
    StateT* S = slice + ((size_t)hh * kHeadDim + warp * kRowsPerWarp) * kHeadDim;
    float4 row[kRowsPerWarp];
    if constexpr (kStaged) {
      const StateT* Ss = reinterpret_cast<const StateT*>(s_state) + (hh * kHeadDim + warp * kRowsPerWarp) * kHeadDim;
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) row[i] = load_state4(Ss, i * 32 + lane);
    } else {
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) row[i] = load_state4(S, i * 32 + lane);
    }
    float d[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
      d[i] = row[i].x * kd.x + row[i].y * kd.y + row[i].z * kd.z + row[i].w * kd.w;
    // lanes 2i and 2i + 1 hold row i's sum; its delta (against the decayed state) is formed there
    // and broadcast
    const int i_mine = (lane >> 1) & 15;
    const float dsum = warp_sum16(d, lane);
    const float e_mine = bt * (s_v[hh][warp * kRowsPerWarp + i_mine] - (kPerChannel ? dsum : a4.x * dsum));
    float o[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const float e = __shfl_sync(0xffffffffu, e_mine, 2 * i);
      // S <- alpha S + e k^T, element by element fma(alpha, s, e k) in f32x2 pairs
      const float2 e2 = make_float2(e, e);
      const float2 xy = __ffma2_rn(make_float2(a4.x, a4.y), make_float2(row[i].x, row[i].y),
                                   __fmul2_rn(e2, make_float2(kn.x, kn.y)));
      const float2 zw = __ffma2_rn(make_float2(a4.z, a4.w), make_float2(row[i].z, row[i].w),
                                   __fmul2_rn(e2, make_float2(kn.z, kn.w)));
      const float4 sn = make_float4(xy.x, xy.y, zw.x, zw.y);
      store_state4(S, i * 32 + lane, sn);
      o[i] = sn.x * qn.x + sn.y * qn.y + sn.z * qn.z + sn.w * qn.w;
    }
    const float o_mine = warp_sum16(o, lane);
    if (!(lane & 1)) s_o[hh][warp * kRowsPerWarp + i_mine] = q_scale * o_mine;
  }
  __syncthreads();

  // ---- sigmoid-gated RMSNorm of each V head's 128 outputs
  for (int hh = warp; hh < R; hh += kThreads / 32) {
    const int h = j * R + hh;
    float ov[4], ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) { ov[i] = s_o[hh][lane * 4 + i]; ss = fmaf(ov[i], ov[i], ss); }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float rstd = rsqrtf(ss * (1.0f / kHeadDim) + rms_eps);
    const size_t base = ((size_t)b * Hv + h) * kHeadDim + lane * 4;
    const uint2 zz = __ldg(reinterpret_cast<const uint2*>(z + base));
    const uint2 ww = __ldg(reinterpret_cast<const uint2*>(norm_w + lane * 4));
    const float zf[4] = {__uint_as_float(zz.x << 16), __uint_as_float(zz.x & 0xFFFF0000u),
                         __uint_as_float(zz.y << 16), __uint_as_float(zz.y & 0xFFFF0000u)};
    const float wf[4] = {__uint_as_float(ww.x << 16), __uint_as_float(ww.x & 0xFFFF0000u),
                         __uint_as_float(ww.y << 16), __uint_as_float(ww.y & 0xFFFF0000u)};
    float r4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) r4[i] = ov[i] * rstd * wf[i] * sigmoidf_(zf[i]);
    *reinterpret_cast<uint2*>(out + base) = make_uint2(pack_bf2(r4[0], r4[1]), pack_bf2(r4[2], r4[3]));
  }
}

}  // namespace

int decode_max_ratio() { return kMaxRatio; }

#ifdef GDN_TEST_HOOKS
cudaError_t test_set_dropped_copy_decode(unsigned on) {
  return cudaMemcpyToSymbol(g_test_drop_state_copy, &on, sizeof on);
}
#endif

cudaError_t launch_kda_decode_step(const LaunchEnv& env, const uint16_t* x, const uint16_t* conv_w,
                                   uint16_t* conv_state, const float* g, float g_min, const float* beta,
                                   float* state, const uint16_t* z, const uint16_t* norm_w, float q_scale,
                                   float l2_eps, float rms_eps, uint16_t* out, int B, int Hk, int Hv) {
  if (B <= 0) return cudaSuccess;
  const GateSrc gates = {g, beta, nullptr, nullptr, nullptr, nullptr};
  decode_step_kernel<float, false, true><<<dim3(Hk, B), kThreads, 0, env.stream>>>(
      x, conv_w, conv_state, gates, state, z, norm_w, q_scale, l2_eps, rms_eps, out, Hk, Hv, env.err, g_min);
  return cudaGetLastError();
}

cudaError_t launch_decode_step(const LaunchEnv& env, const uint16_t* x, const uint16_t* conv_w,
                               uint16_t* conv_state, const GateSrc& gates, void* state,
                               bool fp16_state, const uint16_t* z, const uint16_t* norm_w, float q_scale,
                               float l2_eps, float rms_eps, uint16_t* out, int B, int Hk, int Hv) {
  if (B <= 0) return cudaSuccess;
  dim3 grid(Hk, B);
  const size_t slice_bytes = (size_t)(Hv / Hk) * kHeadDim * kHeadDim * (fp16_state ? 2 : 4);
  if (fp16_state && slice_bytes <= kMaxStagedBytes) {
    static int configured[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
      cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<__half, true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxStagedBytes);
      // the largest shared-memory carveout, so that two staged CTAs share an SM
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_step_kernel<__half, true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return e;
      configured[dev] = 1;
    }
    decode_step_kernel<__half, true><<<grid, kThreads, slice_bytes, env.stream>>>(
        x, conv_w, conv_state, gates, static_cast<__half*>(state), z, norm_w, q_scale, l2_eps, rms_eps, out, Hk, Hv,
        env.err);
  } else if (fp16_state) {
    decode_step_kernel<__half, false><<<grid, kThreads, 0, env.stream>>>(
        x, conv_w, conv_state, gates, static_cast<__half*>(state), z, norm_w, q_scale, l2_eps, rms_eps, out, Hk, Hv,
        env.err);
  } else {
    decode_step_kernel<float, false><<<grid, kThreads, 0, env.stream>>>(
        x, conv_w, conv_state, gates, static_cast<float*>(state), z, norm_w, q_scale, l2_eps, rms_eps, out, Hk, Hv,
        env.err);
  }
  return cudaGetLastError();
}

}  // namespace gdn
