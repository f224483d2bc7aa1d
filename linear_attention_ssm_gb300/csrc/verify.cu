// verify.cu -- multi-token verify of the GDN sublayer and the commit of an accepted prefix.
//
// Qwen3.8 kernel architecture and TDD ledger, "Transaction and width vocabulary" (a verify of
// K rows per sequence resolves exactly once: commit publishes only the selected GDN state,
// abort leaves the prior state); spark_model layer_struct.rs, the WY verify kernel fields
// (K = 2..17 rows per sequence) and the write-on-accept twin with its post-verdict fold (the
// verify does not write the state; the accepted rows are folded in after the verdict).
//
// verify_kernel: one CTA per (sequence, K head), like the decode step: it owns the q/k channels
// of that K head and the v channels of its Hv/Hk V heads.  It runs the conv step for the K rows
// from the conv state (which it does not modify), the L2 norms of every row's q and k, then per V
// head streams the head's 128 x 128 fp32 state into registers (16 rows per warp, a row is 32
// lanes x float4 over the key dimension) and applies the K rows to it in registers -- decay,
// delta correction, output -- in the same fp32 expressions as the one-token decode step, without
// storing it.  The rows' gated outputs go to `out`; the per-row keys, values, gates and raw conv
// inputs go to the stash.
//
// commit_kernel: the same CTA grid; for committed_rows[b] = m it streams the state once more,
// applies the first m stashed rows (no output), stores it, and shifts the m rows' raw inputs into
// the conv state.  m = 0 leaves both states untouched.  Rows m.. of the stash are never read.
#include <cuda_fp16.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kHeadDim / kWarps;  // 16 state rows ([value] index) per warp

struct VerifyParams {
  const uint16_t* x;       // [B, K, C] raw conv inputs
  const uint16_t* conv_w;  // [C, 4]
  const uint16_t* conv_state;  // [B, C, 3], read only
  const float* g;          // [B, K, Hv]
  const float* beta;       // [B, K, Hv]
  const float* state;      // [B, Hv, Dv, Dk], read only
  const uint16_t* z;       // [B, K, Hv, Dv]
  const uint16_t* norm_w;  // [Dv]
  uint16_t* out;           // [B, K, Hv, Dv]
  uint8_t* stash;          // [B, K] records
  float q_scale, l2_eps, rms_eps;
  int K, Hk, Hv;
};

struct CommitParams {
  const int32_t* committed;  // [B]
  const uint8_t* stash;
  uint16_t* conv_state;      // [B, C, 3], in/out
  float* state;              // [B, Hv, Dv, Dk], in/out
  unsigned* err;
  int K, Hk, Hv;
};

__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

// Sums v[0..15] over the 32 lanes of a warp in 16 shuffles (a halving butterfly: at each of the
// five levels a lane keeps half of its values and adds its partner's copy of that half).  Every
// total is formed by the same pairwise additions as five xor-shuffle levels applied to each value
// on its own.  Lanes 2i and 2i + 1 return the total of v[i].
__device__ __forceinline__ float warp_sum16(const float (&v)[16], int lane) {
  float a[8], b4[4], c2[2];
  const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float keep = h16 ? v[8 + k] : v[k];
    const float send = h16 ? v[k] : v[8 + k];
    a[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float keep = h8 ? a[4 + k] : a[k];
    const float send = h8 ? a[k] : a[4 + k];
    b4[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float keep = h4 ? b4[2 + k] : b4[k];
    const float send = h4 ? b4[k] : b4[2 + k];
    c2[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const float keep = h2 ? c2[1] : c2[0];
  const float send = h2 ? c2[0] : c2[1];
  const float s = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  return s + __shfl_xor_sync(0xffffffffu, s, 1);
}

// The channel octet a CTA thread owns in the conv step: q channels of K head j (octets 0..15),
// k channels (16..31), then the v channels of V heads j*R .. j*R+R-1 (16 octets each).
__device__ __forceinline__ int octet_channel(int o, int j, int R, int Hk) {
  if (o < 16) return j * kHeadDim + o * 8;
  if (o < 32) return Hk * kHeadDim + j * kHeadDim + (o - 16) * 8;
  const int hh = (o - 32) >> 4;
  return 2 * Hk * kHeadDim + (j * R + hh) * kHeadDim + ((o - 32) & 15) * 8;
}

__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const __grid_constant__ VerifyParams p) {
  const int j = blockIdx.x;  // K head
  const int b = blockIdx.y;  // sequence
  const int K = p.K, Hk = p.Hk, Hv = p.Hv;
  const int R = Hv / Hk;
  const int C = 2 * Hk * kHeadDim + Hv * kHeadDim;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const VerifyStash L = verify_stash_layout(C, Hk, Hv);

  extern __shared__ float vsm[];
  float* s_q = vsm;                              // [K][128] conv outputs (bf16 values)
  float* s_k = s_q + K * kHeadDim;               // [K][128]
  float* s_v = s_k + K * kHeadDim;               // [K][R][128]
  float* s_o = s_v + K * R * kHeadDim;           // [K][R][128]
  float* s_norm = s_o + K * R * kHeadDim;        // [K][2] 1/sqrt(sum x^2 + eps) of q, k
  float* s_ab = s_norm + 2 * K;                  // [K][R][2] alpha = exp(g), beta

  // ---- conv step + SiLU for the K rows (the conv state is read, never written)
  const int n_oct = 32 + 16 * R;
  if (tid < n_oct) {
    const int c = octet_channel(tid, j, R, Hk);
    float wv[32], win[24];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float t8[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(p.conv_w + (size_t)c * kConvWidth) + i), t8);
#pragma unroll
      for (int e = 0; e < 8; ++e) wv[i * 8 + e] = t8[e];
    }
    const uint4* sp = reinterpret_cast<const uint4*>(p.conv_state + ((size_t)b * C + c) * (kConvWidth - 1));
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      float t8[8];
      unpack8(__ldg(sp + i), t8);
#pragma unroll
      for (int e = 0; e < 8; ++e) win[i * 8 + e] = t8[e];  // channel ch: win[ch*3 + 0..2], oldest first
    }
    for (int r = 0; r < K; ++r) {
      const uint4 xr = __ldg(reinterpret_cast<const uint4*>(p.x + ((size_t)b * K + r) * C + c));
      uint8_t* rec = p.stash + ((size_t)b * K + r) * L.bytes;
      *reinterpret_cast<uint4*>(rec + L.x_off + (size_t)c * 2) = xr;
      float xv[8], a[8];
      unpack8(xr, xv);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        float acc = wv[ch * 4 + 0] * win[ch * 3 + 0];
        acc = fmaf(wv[ch * 4 + 1], win[ch * 3 + 1], acc);
        acc = fmaf(wv[ch * 4 + 2], win[ch * 3 + 2], acc);
        acc = fmaf(wv[ch * 4 + 3], xv[ch], acc);
        a[ch] = bf2f(f2bf(acc / (1.0f + expf(-acc))));  // the bf16 conv output
        win[ch * 3 + 0] = win[ch * 3 + 1];
        win[ch * 3 + 1] = win[ch * 3 + 2];
        win[ch * 3 + 2] = xv[ch];
      }
      float* dst;
      if (tid < 16) dst = s_q + r * kHeadDim + tid * 8;
      else if (tid < 32) dst = s_k + r * kHeadDim + (tid - 16) * 8;
      else {
        const int hh = (tid - 32) >> 4, o = (tid - 32) & 15;
        dst = s_v + (r * R + hh) * kHeadDim + o * 8;
        uint4 vb;  // the v channels as bf16 (exact: they are bf16 values)
        vb.x = pack_bf2(a[0], a[1]); vb.y = pack_bf2(a[2], a[3]);
        vb.z = pack_bf2(a[4], a[5]); vb.w = pack_bf2(a[6], a[7]);
        *reinterpret_cast<uint4*>(rec + L.v_off + ((size_t)(j * R + hh) * kHeadDim + o * 8) * 2) = vb;
      }
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) dst[ch] = a[ch];
    }
  }
  // gates of the CTA's V heads for every row
  for (int t = tid; t < K * R; t += kThreads) {
    const int r = t / R, hh = t - r * R, h = j * R + hh;
    const size_t gi = ((size_t)b * K + r) * Hv + h;
    const float alpha = expf(__ldg(p.g + gi));
    const float bt = __ldg(p.beta + gi);
    s_ab[2 * t] = alpha;
    s_ab[2 * t + 1] = bt;
    uint8_t* rec = p.stash + ((size_t)b * K + r) * L.bytes;
    reinterpret_cast<float*>(rec + L.alpha_off)[h] = alpha;
    reinterpret_cast<float*>(rec + L.beta_off)[h] = bt;
  }
  __syncthreads();

  // ---- L2 norms of every row's q and k: x / sqrt(sum x^2 + eps)
  for (int t = warp; t < 2 * K; t += kWarps) {
    const float* src = (t & 1) ? s_k + (t >> 1) * kHeadDim : s_q + (t >> 1) * kHeadDim;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) { const float v = src[lane * 4 + i]; ss = fmaf(v, v, ss); }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if (lane == 0) s_norm[t] = rsqrtf(ss + p.l2_eps);
  }
  __syncthreads();
  // normalised keys of every row -> the stash (the commit folds with exactly these values)
  for (int t = tid; t < K * (kHeadDim / 4); t += kThreads) {
    const int r = t / (kHeadDim / 4), q4 = t - r * (kHeadDim / 4);
    const float nk = s_norm[2 * r + 1];
    const float* kk = s_k + r * kHeadDim + q4 * 4;
    uint8_t* rec = p.stash + ((size_t)b * K + r) * L.bytes;
    *reinterpret_cast<float4*>(rec + L.khat_off + ((size_t)j * kHeadDim + q4 * 4) * 4) =
        make_float4(kk[0] * nk, kk[1] * nk, kk[2] * nk, kk[3] * nk);
  }

  // ---- the K rows applied to each V head's state in registers (never stored)
  const int r_mine = (lane >> 1) & 15;  // the row whose sums this lane ends up holding
  for (int hh = 0; hh < R; ++hh) {
    const int h = j * R + hh;
    const float4* S = reinterpret_cast<const float4*>(
        p.state + (((size_t)b * Hv + h) * kHeadDim + warp * kRowsPerWarp) * kHeadDim);
    float4 row[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) row[i] = __ldg(S + i * 32 + lane);
    for (int r = 0; r < K; ++r) {
      const float nq = s_norm[2 * r], nk = s_norm[2 * r + 1];
      const float* qq = s_q + r * kHeadDim + lane * 4;
      const float* kk = s_k + r * kHeadDim + lane * 4;
      const float4 qn = make_float4(qq[0] * nq, qq[1] * nq, qq[2] * nq, qq[3] * nq);
      const float4 kn = make_float4(kk[0] * nk, kk[1] * nk, kk[2] * nk, kk[3] * nk);
      const float alpha = s_ab[2 * (r * R + hh)], bt = s_ab[2 * (r * R + hh) + 1];
      float d[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) d[i] = dot4(row[i], kn);
      const float dm = warp_sum16(d, lane);
      const float em = bt * (s_v[(r * R + hh) * kHeadDim + warp * kRowsPerWarp + r_mine] - alpha * dm);
      float o[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const float e = __shfl_sync(0xffffffffu, em, 2 * i);  // delta against the decayed state
        row[i].x = fmaf(alpha, row[i].x, e * kn.x);
        row[i].y = fmaf(alpha, row[i].y, e * kn.y);
        row[i].z = fmaf(alpha, row[i].z, e * kn.z);
        row[i].w = fmaf(alpha, row[i].w, e * kn.w);
        o[i] = dot4(row[i], qn);
      }
      const float om = warp_sum16(o, lane);
      if (!(lane & 1)) s_o[(r * R + hh) * kHeadDim + warp * kRowsPerWarp + r_mine] = p.q_scale * om;
    }
  }
  __syncthreads();

  // ---- sigmoid-gated RMSNorm of every (row, V head)
  const uint2 ww = __ldg(reinterpret_cast<const uint2*>(p.norm_w + lane * 4));
  const float wf[4] = {__uint_as_float(ww.x << 16), __uint_as_float(ww.x & 0xFFFF0000u),
                       __uint_as_float(ww.y << 16), __uint_as_float(ww.y & 0xFFFF0000u)};
  for (int t = warp; t < K * R; t += kWarps) {
    const int r = t / R, hh = t - r * R, h = j * R + hh;
    float ov[4], ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) { ov[i] = s_o[t * kHeadDim + lane * 4 + i]; ss = fmaf(ov[i], ov[i], ss); }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float rstd = rsqrtf(ss * (1.0f / kHeadDim) + p.rms_eps);
    const size_t base = (((size_t)b * K + r) * Hv + h) * kHeadDim + lane * 4;
    const uint2 zz = __ldg(reinterpret_cast<const uint2*>(p.z + base));
    const float zf[4] = {__uint_as_float(zz.x << 16), __uint_as_float(zz.x & 0xFFFF0000u),
                         __uint_as_float(zz.y << 16), __uint_as_float(zz.y & 0xFFFF0000u)};
    float r4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) r4[i] = ov[i] * rstd * wf[i] * sigmoidf_(zf[i]);
    *reinterpret_cast<uint2*>(p.out + base) = make_uint2(pack_bf2(r4[0], r4[1]), pack_bf2(r4[2], r4[3]));
  }
}

__global__ void __launch_bounds__(kThreads, 2) commit_kernel(const __grid_constant__ CommitParams p) {
  const int j = blockIdx.x;  // K head
  const int b = blockIdx.y;  // sequence
  const int K = p.K, Hk = p.Hk, Hv = p.Hv;
  const int R = Hv / Hk;
  const int C = 2 * Hk * kHeadDim + Hv * kHeadDim;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const VerifyStash L = verify_stash_layout(C, Hk, Hv);

  const int m = __ldg(p.committed + b);
  if (m < 0 || m > K) {  // a bad verdict: this sequence is left untouched and reported
    if (tid == 0 && j == 0) raise_error(p.err, kErrDeviceArgument);
    return;
  }
  if (m == 0) return;  // abort: the prior states stand
  const uint8_t* rec0 = p.stash + (size_t)b * K * L.bytes;

  // ---- conv state: the last 3 raw inputs of [prior conv state, rows 0 .. m-1], oldest first
  const int n_oct = 32 + 16 * R;
  if (tid < n_oct) {
    const int c = octet_channel(tid, j, R, Hk);
    uint4* sp = reinterpret_cast<uint4*>(p.conv_state + ((size_t)b * C + c) * (kConvWidth - 1));
    float old[24];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      float t8[8];
      unpack8(sp[i], t8);
#pragma unroll
      for (int e = 0; e < 8; ++e) old[i * 8 + e] = t8[e];
    }
    float nw[24];  // nw[ch*3 + s]
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      const int idx = m - 3 + s;  // index into the rows; negative: the prior state's slot 3 + idx
      if (idx >= 0) {
        float t8[8];
        unpack8(*reinterpret_cast<const uint4*>(rec0 + (size_t)idx * L.bytes + L.x_off + (size_t)c * 2), t8);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) nw[ch * 3 + s] = t8[ch];
      } else {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) nw[ch * 3 + s] = old[ch * 3 + 3 + idx];
      }
    }
    uint32_t pk[12];
#pragma unroll
    for (int i = 0; i < 12; ++i) pk[i] = pack_bf2(nw[2 * i], nw[2 * i + 1]);  // exact (bf16 inputs)
    sp[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    sp[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    sp[2] = make_uint4(pk[8], pk[9], pk[10], pk[11]);
  }

  // ---- the first m rows folded into each V head's state
  const int r_mine = (lane >> 1) & 15;
  for (int hh = 0; hh < R; ++hh) {
    const int h = j * R + hh;
    float4* S = reinterpret_cast<float4*>(p.state + (((size_t)b * Hv + h) * kHeadDim + warp * kRowsPerWarp) * kHeadDim);
    float4 row[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) row[i] = S[i * 32 + lane];
    for (int r = 0; r < m; ++r) {
      const uint8_t* rec = rec0 + (size_t)r * L.bytes;
      const float4 kn = *reinterpret_cast<const float4*>(rec + L.khat_off + ((size_t)j * kHeadDim + lane * 4) * 4);
      const float alpha = reinterpret_cast<const float*>(rec + L.alpha_off)[h];
      const float bt = reinterpret_cast<const float*>(rec + L.beta_off)[h];
      const float vm = bf2f(*reinterpret_cast<const uint16_t*>(
          rec + L.v_off + ((size_t)h * kHeadDim + warp * kRowsPerWarp + r_mine) * 2));
      float d[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) d[i] = dot4(row[i], kn);
      const float dm = warp_sum16(d, lane);
      const float em = bt * (vm - alpha * dm);
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const float e = __shfl_sync(0xffffffffu, em, 2 * i);
        row[i].x = fmaf(alpha, row[i].x, e * kn.x);
        row[i].y = fmaf(alpha, row[i].y, e * kn.y);
        row[i].z = fmaf(alpha, row[i].z, e * kn.z);
        row[i].w = fmaf(alpha, row[i].w, e * kn.w);
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) S[i * 32 + lane] = row[i];
  }
}

size_t verify_smem_bytes(int K, int R) {
  return sizeof(float) * ((size_t)2 * K * kHeadDim + (size_t)2 * K * R * kHeadDim + 2 * K + 2 * K * R);
}

}  // namespace

int verify_max_rows() { return kMaxVerifyRows; }

bool verify_supported(int K, int Hk, int Hv) {
  return K >= 1 && K <= kMaxVerifyRows && verify_smem_bytes(K, Hv / Hk) <= kMaxVerifySmem;
}

cudaError_t launch_verify(const LaunchEnv& env, const uint16_t* x, const uint16_t* conv_w, const uint16_t* conv_state,
                          const float* g, const float* beta, const float* state, const uint16_t* z,
                          const uint16_t* norm_w, float q_scale, float l2_eps, float rms_eps, uint16_t* out,
                          void* stash, int B, int K, int Hk, int Hv) {
  if (B <= 0) return cudaSuccess;
  static int configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxVerifySmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  VerifyParams p;
  p.x = x; p.conv_w = conv_w; p.conv_state = conv_state; p.g = g; p.beta = beta; p.state = state; p.z = z;
  p.norm_w = norm_w; p.out = out; p.stash = static_cast<uint8_t*>(stash);
  p.q_scale = q_scale; p.l2_eps = l2_eps; p.rms_eps = rms_eps;
  p.K = K; p.Hk = Hk; p.Hv = Hv;
  verify_kernel<<<dim3(Hk, B), kThreads, verify_smem_bytes(K, Hv / Hk), env.stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_verify_commit(const LaunchEnv& env, const int32_t* committed, const void* stash,
                                 uint16_t* conv_state, float* state, int B, int K, int Hk, int Hv) {
  if (B <= 0) return cudaSuccess;
  CommitParams p;
  p.committed = committed; p.stash = static_cast<const uint8_t*>(stash); p.conv_state = conv_state;
  p.state = state; p.err = env.err; p.K = K; p.Hk = Hk; p.Hv = Hv;
  commit_kernel<<<dim3(Hk, B), kThreads, 0, env.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
