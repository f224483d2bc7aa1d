// verify.cu -- multi-token verify of the GDN sublayer and the commit of an accepted prefix.
//
// Qwen3.8 kernel architecture and TDD ledger, "Transaction and width vocabulary" (a verify of
// K rows per sequence resolves exactly once: commit publishes only the selected GDN state,
// abort leaves the prior state); spark_model layer_struct.rs, the WY verify kernel fields
// (K = 2..17 rows per sequence) and the write-on-accept twin with its post-verdict fold (the
// verify does not write the state; the accepted rows are folded in after the verdict).
//
// verify_kernel: one CTA per (sequence, K head), like the decode step: it owns the q/k channels
// of that K head and the v channels of its Hv/Hk V heads.  It stages the rows' raw inputs, the
// conv state and the weights of its channels in shared memory, runs the conv step of every
// (row, channel octet) in parallel from the conv state (which it does not modify), the L2 norms
// of every row's q and k, and the rows' Gram matrices k_i . k_r and k_i . q_r.  The K rows are
// then applied in the WY form: for every value row v of a V head's initial state S0, the dot
// products S0[v] . k_r and S0[v] . q_r of all rows come first (independent of one another), and
// the deltas e_r = beta_r (v_r - decayed state . k_r) and outputs follow by forward substitution
// over the rows with decay-weighted Gram entries -- S_r = exp(G_r) S0 + sum_{i<=r} exp(G_r - G_i)
// e_i k_i^T written out, G_r the sum of g over rows 0..r.  The state is never written.  A warp
// holds 16 value rows of S0; a lane 4 rows x 16 keys, so a dot product is a 16-term f32x2 partial
// and a 3-level butterfly over the 8 lanes of its group.  The rows' gated outputs go to `out`;
// the per-row raw inputs, keys, deltas and g go to the stash.
//
// commit_kernel: the same CTA grid; for committed_rows[b] = m it streams the state once:
// S_m = exp(G_{m-1}) S0 + sum_{i<m} exp(G_{m-1} - G_i) e_i k_i^T (a rank-m update from the
// stashed deltas, the verify's own factors), and shifts the m rows' raw inputs into the conv
// state.  m = 0 leaves both states untouched.  Rows m.. of the stash are never read.
#include <cuda_fp16.h>
#include <string.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct VerifyParams {
  const uint16_t* x;       // [B, K, C] raw conv inputs
  const uint16_t* conv_w;  // [C, 4]
  const uint16_t* conv_state;  // [B, C, 3], read only
  const float* g;          // [B, K, Hv]
  const float* beta;       // [B, K, Hv]
  const void* state;       // [B, Hv, Dv, Dk] fp32 or binary16, read only
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
  void* state;               // [B, Hv, Dv, Dk] fp32 or binary16, in/out
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

// A warp owns 16 state rows of a V head; lane (rg, kg) = (lane / 8, lane % 8) holds rows
// 4 rg .. 4 rg + 3 of them over the 16 keys {32 q + 4 kg + e : q, e in 0..3} (4 float4 per row):
// every load or store instruction moves 4 rows x 128 contiguous bytes.
struct Slice {
  float4 s[4][4];  // [row][key quad]
};

__device__ __forceinline__ int slice_offset(int warp, int lane, int ri, int qi) {  // in floats, within a head
  return (warp * 16 + (lane >> 3) * 4 + ri) * kHeadDim + 32 * qi + 4 * (lane & 7);
}

// the lane's slice of a head's state, widened to fp32 (fp32 or binary16 storage)
__device__ __forceinline__ void load_slice(Slice& S, const float* Sg, int warp, int lane) {
#pragma unroll
  for (int ri = 0; ri < 4; ++ri)
#pragma unroll
    for (int qi = 0; qi < 4; ++qi) S.s[ri][qi] = *reinterpret_cast<const float4*>(Sg + slice_offset(warp, lane, ri, qi));
}
__device__ __forceinline__ void load_slice(Slice& S, const __half* Sg, int warp, int lane) {
#pragma unroll
  for (int ri = 0; ri < 4; ++ri)
#pragma unroll
    for (int qi = 0; qi < 4; ++qi) {
      const uint2 u = *reinterpret_cast<const uint2*>(Sg + slice_offset(warp, lane, ri, qi));
      __half2 h01, h23;
      memcpy(&h01, &u.x, 4);
      memcpy(&h23, &u.y, 4);
      const float2 a = __half22float2(h01), b = __half22float2(h23);
      S.s[ri][qi] = make_float4(a.x, a.y, b.x, b.y);
    }
}
// the slice stored back: fp32 as is, binary16 rounded to nearest even
__device__ __forceinline__ void store_slice(const Slice& S, float* Sg, int warp, int lane) {
#pragma unroll
  for (int ri = 0; ri < 4; ++ri)
#pragma unroll
    for (int qi = 0; qi < 4; ++qi) *reinterpret_cast<float4*>(Sg + slice_offset(warp, lane, ri, qi)) = S.s[ri][qi];
}
__device__ __forceinline__ void store_slice(const Slice& S, __half* Sg, int warp, int lane) {
#pragma unroll
  for (int ri = 0; ri < 4; ++ri)
#pragma unroll
    for (int qi = 0; qi < 4; ++qi) {
      const float4 v = S.s[ri][qi];
      const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
      uint2 u;
      memcpy(&u.x, &a, 4);
      memcpy(&u.y, &b, 4);
      *reinterpret_cast<uint2*>(Sg + slice_offset(warp, lane, ri, qi)) = u;
    }
}

// this lane's part of the dot product of row ri with a key-dimension vector (4 float4, own keys)
__device__ __forceinline__ float partial_dot(const Slice& S, int ri, const float4 (&u)[4]) {
  float2 acc = __fmul2_rn(make_float2(S.s[ri][0].x, S.s[ri][0].y), make_float2(u[0].x, u[0].y));
  acc = __ffma2_rn(make_float2(S.s[ri][0].z, S.s[ri][0].w), make_float2(u[0].z, u[0].w), acc);
#pragma unroll
  for (int qi = 1; qi < 4; ++qi) {
    acc = __ffma2_rn(make_float2(S.s[ri][qi].x, S.s[ri][qi].y), make_float2(u[qi].x, u[qi].y), acc);
    acc = __ffma2_rn(make_float2(S.s[ri][qi].z, S.s[ri][qi].w), make_float2(u[qi].z, u[qi].w), acc);
  }
  return acc.x + acc.y;
}

// Sums v[0..3] over the 8 lanes of a row group in 4 shuffles (a halving butterfly over lane bits
// 2, 1, 0).  Lanes 2i and 2i + 1 of the group return the total of v[i].
__device__ __forceinline__ float group_sum4(const float (&v)[4], int lane) {
  const bool h4 = lane & 4, h2 = lane & 2;
  const float a0 = (h4 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, h4 ? v[0] : v[2], 4);
  const float a1 = (h4 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, h4 ? v[1] : v[3], 4);
  const float b = (h2 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, h2 ? a0 : a1, 2);
  return b + __shfl_xor_sync(0xffffffffu, b, 1);
}

// this lane's 16 keys of a [128] vector in shared memory
__device__ __forceinline__ void load_keys(const float* v, int lane, float4 (&u)[4]) {
#pragma unroll
  for (int qi = 0; qi < 4; ++qi) u[qi] = *reinterpret_cast<const float4*>(v + 32 * qi + 4 * (lane & 7));
}

// The channel octet a CTA thread owns in the conv step: q channels of K head j (octets 0..15),
// k channels (16..31), then the v channels of V heads j*R .. j*R+R-1 (16 octets each).
__device__ __forceinline__ int octet_channel(int o, int j, int R, int Hk) {
  if (o < 16) return j * kHeadDim + o * 8;
  if (o < 32) return Hk * kHeadDim + j * kHeadDim + (o - 16) * 8;
  const int hh = (o - 32) >> 4;
  return 2 * Hk * kHeadDim + (j * R + hh) * kHeadDim + ((o - 32) & 15) * 8;
}

template <int KB, typename StateT>  // rows per sequence <= KB (register arrays of the per-row recurrence)
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const __grid_constant__ VerifyParams p) {
  const StateT* const state = static_cast<const StateT*>(p.state);
  const int j = blockIdx.x;  // K head
  const int b = blockIdx.y;  // sequence
  const int K = p.K, Hk = p.Hk, Hv = p.Hv;
  const int R = Hv / Hk;
  const int C = 2 * Hk * kHeadDim + Hv * kHeadDim;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const VerifyStash L = verify_stash_layout(C, Hk, Hv);

  // shared memory: the raw octets first (16-byte aligned), then the fp32 arrays
  const int n_oct = 32 + 16 * R;  // channel octets of the CTA (see octet_channel)
  extern __shared__ uint4 vsm_raw[];
  uint4* s_x = vsm_raw;                          // [K][n_oct] raw conv inputs of the rows
  uint4* s_cs = s_x + K * n_oct;                 // [n_oct][3] conv state (8 channels x 3 slots)
  uint4* s_w = s_cs + 3 * n_oct;                 // [n_oct][4] conv weights (8 channels x 4 taps)
  float* s_q = reinterpret_cast<float*>(s_w + 4 * n_oct);  // [K][128] conv outputs (bf16 values)
  float* s_k = s_q + K * kHeadDim;               // [K][128]
  float* s_v = s_k + K * kHeadDim;               // [K][R][128]
  float* s_o = s_v + K * R * kHeadDim;           // [K][R][128]
  float* s_norm = s_o + K * R * kHeadDim;        // [K][2] 1/sqrt(sum x^2 + eps) of q, k
  float* s_gb = s_norm + 2 * K;                  // [K][R][2] g, beta
  float* s_G = s_gb + 2 * K * R;                 // [K][K] G[i][r] = k_i . k_r (i < r)
  float* s_H = s_G + K * K;                      // [K][K] H[i][r] = k_i . q_r (i <= r)
  float* s_A = s_H + K * K;                      // [R][K][K] A[r][i] = exp(G_r - G_i) G[i][r] (i < r)
  float* s_B = s_A + R * K * K;                  // [R][K][K] B[r][i] = exp(G_r - G_i) H[i][r] (i <= r)
  float* s_D = s_B + R * K * K;                  // [R][K] exp(G_r), G_r = g_0 + .. + g_r

  // ---- the CTA's state slice (its R V heads are contiguous) and its z rows are fetched into L2
  // now, so that they arrive while the conv, the norms and the Gram matrices are computed
  if (tid < R) {  // one head per thread
    bulk_prefetch_l2(state + ((size_t)b * Hv + (size_t)j * R + tid) * kHeadDim * kHeadDim,
                     (uint32_t)(kHeadDim * kHeadDim * sizeof(StateT)));
  } else if (tid >= 32 && tid < 32 + K) {  // z of the CTA's V heads, one row per thread
    bulk_prefetch_l2(p.z + (((size_t)b * K + (tid - 32)) * Hv + (size_t)j * R) * kHeadDim,
                     (uint32_t)(R * kHeadDim * 2));
  }
  // gates of the CTA's V heads for every row
  for (int t = tid; t < K * R; t += kThreads) {
    const int r = t / R, hh = t - r * R, h = j * R + hh;
    const size_t gi = ((size_t)b * K + r) * Hv + h;
    const float gg = __ldg(p.g + gi);
    s_gb[2 * t] = gg;
    s_gb[2 * t + 1] = __ldg(p.beta + gi);
    reinterpret_cast<float*>(p.stash + ((size_t)b * K + r) * L.bytes + L.g_off)[h] = gg;
  }
  // ---- the rows' raw inputs, the conv state and the weights of the CTA's channels -> shared
  // memory in one round of independent loads; the raw inputs also go to the stash
  for (int t = tid; t < (K + 7) * n_oct; t += kThreads) {
    const int slot = t / n_oct, o = t - slot * n_oct;
    const int c = octet_channel(o, j, R, Hk);
    if (slot < K) {
      const uint4 xr = __ldg(reinterpret_cast<const uint4*>(p.x + ((size_t)b * K + slot) * C + c));
      s_x[slot * n_oct + o] = xr;
      *reinterpret_cast<uint4*>(p.stash + ((size_t)b * K + slot) * L.bytes + L.x_off + (size_t)c * 2) = xr;
    } else if (slot < K + 3) {
      const int i = slot - K;
      s_cs[o * 3 + i] = __ldg(reinterpret_cast<const uint4*>(p.conv_state + ((size_t)b * C + c) * (kConvWidth - 1)) + i);
    } else {
      const int i = slot - K - 3;
      s_w[o * 4 + i] = __ldg(reinterpret_cast<const uint4*>(p.conv_w + (size_t)c * kConvWidth) + i);
    }
  }
  __syncthreads();

  // ---- conv step + SiLU of every (row, octet), the rows in parallel (the conv state is read,
  // never written): y_r = w0 x_{r-3} + w1 x_{r-2} + w2 x_{r-1} + w3 x_r, x before row 0 from the
  // conv state, rounded to bf16 as the exact values are (as the decode step does)
  for (int t = tid; t < K * n_oct; t += kThreads) {
    const int r = t / n_oct, o = t - r * n_oct;
    float wv[32], cs[24], xw[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float t8[8];
      unpack8(s_w[o * 4 + i], t8);
#pragma unroll
      for (int e = 0; e < 8; ++e) wv[i * 8 + e] = t8[e];  // channel ch: wv[ch*4 + tap]
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      float t8[8];
      unpack8(s_cs[o * 3 + i], t8);
#pragma unroll
      for (int e = 0; e < 8; ++e) cs[i * 8 + e] = t8[e];  // channel ch: cs[ch*3 + slot], oldest first
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // window position i holds x_{r-3+i}
      const int rr = r - 3 + i;
      if (rr >= 0) {
        unpack8(s_x[rr * n_oct + o], xw[i]);
      } else {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) xw[i][ch] = cs[ch * 3 + 3 + rr];
      }
    }
    float a[8];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)  // the bf16 conv output, rounded as the exact value is
      a[ch] = bf2f(silu_bf16_rn(wv[ch * 4 + 0], xw[0][ch], wv[ch * 4 + 1], xw[1][ch], wv[ch * 4 + 2], xw[2][ch],
                                wv[ch * 4 + 3], xw[3][ch]));
    float* dst;
    if (o < 16) dst = s_q + r * kHeadDim + o * 8;
    else if (o < 32) dst = s_k + r * kHeadDim + (o - 16) * 8;
    else {
      const int hh = (o - 32) >> 4, oo = (o - 32) & 15;
      dst = s_v + (r * R + hh) * kHeadDim + oo * 8;
    }
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) dst[ch] = a[ch];
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
  // q and k of every row normalised in place; the normalised keys -> the stash (the commit folds
  // with exactly these values)
  for (int t = tid; t < K * (kHeadDim / 4); t += kThreads) {
    const int r = t / (kHeadDim / 4), q4 = t - r * (kHeadDim / 4);
    const float nq = s_norm[2 * r], nk = s_norm[2 * r + 1];
    float4* qq = reinterpret_cast<float4*>(s_q + r * kHeadDim + q4 * 4);
    float4* kk = reinterpret_cast<float4*>(s_k + r * kHeadDim + q4 * 4);
    const float4 q = *qq, k = *kk;
    *qq = make_float4(q.x * nq, q.y * nq, q.z * nq, q.w * nq);
    const float4 kn = make_float4(k.x * nk, k.y * nk, k.z * nk, k.w * nk);
    *kk = kn;
    uint8_t* rec = p.stash + ((size_t)b * K + r) * L.bytes;
    *reinterpret_cast<float4*>(rec + L.khat_off + ((size_t)j * kHeadDim + q4 * 4) * 4) = kn;
  }
  __syncthreads();

  // ---- the rows' Gram matrices G[i][r] = k_i . k_r and H[i][r] = k_i . q_r, one warp per (i <= r)
  for (int t = warp; t < K * K; t += kWarps) {
    const int i = t / K, r = t - i * K;
    if (i > r) continue;
    const float4 ki = *reinterpret_cast<const float4*>(s_k + i * kHeadDim + lane * 4);
    const float4 kr = *reinterpret_cast<const float4*>(s_k + r * kHeadDim + lane * 4);
    const float4 qr = *reinterpret_cast<const float4*>(s_q + r * kHeadDim + lane * 4);
    float gk = ki.x * kr.x + ki.y * kr.y + ki.z * kr.z + ki.w * kr.w;
    float hq = ki.x * qr.x + ki.y * qr.y + ki.z * qr.z + ki.w * qr.w;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      gk += __shfl_xor_sync(0xffffffffu, gk, m);
      hq += __shfl_xor_sync(0xffffffffu, hq, m);
    }
    if (lane == 0) {
      s_G[i * K + r] = gk;
      s_H[i * K + r] = hq;
    }
  }
  __syncthreads();
  // decay-weighted factors per V head: the decay from after row i through row r is
  // exp(g_{i+1} + .. + g_r) (summed directly, never as a difference of prefix sums)
  for (int t = tid; t < R * K * K; t += kThreads) {
    const int hh = t / (K * K), r = (t / K) % K, i = t % K;
    float A = 0.f, B = 0.f;
    if (i <= r) {
      float gs = 0.f;
      for (int jj = i + 1; jj <= r; ++jj) gs += s_gb[2 * (jj * R + hh)];
      const float dec = expf(gs);
      A = i < r ? dec * s_G[i * K + r] : 0.f;
      B = dec * s_H[i * K + r];
    }
    s_A[(hh * K + r) * K + i] = A;
    s_B[(hh * K + r) * K + i] = B;
    if (i == 0) {
      float gs = 0.f;
      for (int jj = 0; jj <= r; ++jj) gs += s_gb[2 * (jj * R + hh)];
      s_D[hh * K + r] = expf(gs);
    }
  }
  __syncthreads();

  // ---- per V head, per value row v of the initial state S0 (never modified):
  //   x_r = S0[v] . k_r,  y_r = S0[v] . q_r                       (all rows' dot products first)
  //   d_r = exp(G_r) x_r + sum_{i<r} A[r][i] e_i                  (= the decayed state . k_r)
  //   e_r = beta_r (v_r - d_r)
  //   o_r = q_scale (exp(G_r) y_r + sum_{i<=r} B[r][i] e_i)       (= S_r . q_r)
  // which is S_r = exp(G_r) S0 + sum_{i<=r} exp(G_r - G_i) e_i k_i^T written out.  The deltas e go
  // to the stash: the commit forms S_m from them.
  const int row_mine = warp * 16 + (lane >> 3) * 4 + ((lane & 7) >> 1);  // the row whose sums this lane holds
  for (int hh = 0; hh < R; ++hh) {
    const int h = j * R + hh;
    Slice S;
    load_slice(S, state + ((size_t)b * Hv + h) * kHeadDim * kHeadDim, warp, lane);
    float xe[KB];  // x_r, then e_r
#pragma unroll
    for (int r = 0; r < KB; ++r) {
      if (r < K) {
        float4 u[4];
        load_keys(s_k + r * kHeadDim, lane, u);
        float d4[4];
#pragma unroll
        for (int ri = 0; ri < 4; ++ri) d4[ri] = partial_dot(S, ri, u);
        xe[r] = group_sum4(d4, lane);
      }
    }
    const float* A = s_A + hh * K * K;
    const float* B = s_B + hh * K * K;
    const float* D = s_D + hh * K;
#pragma unroll
    for (int r = 0; r < KB; ++r) {
      if (r < K) {
        float d = D[r] * xe[r];
#pragma unroll
        for (int i = 0; i < r; ++i) d = fmaf(A[r * K + i], xe[i], d);
        const int t = r * R + hh;
        xe[r] = s_gb[2 * t + 1] * (s_v[t * kHeadDim + row_mine] - d);
        if (!(lane & 1))
          reinterpret_cast<float*>(p.stash + ((size_t)b * K + r) * L.bytes + L.e_off)[h * kHeadDim + row_mine] = xe[r];
      }
    }
#pragma unroll
    for (int r = 0; r < KB; ++r) {
      if (r < K) {
        float4 u[4];
        load_keys(s_q + r * kHeadDim, lane, u);
        float y4[4];
#pragma unroll
        for (int ri = 0; ri < 4; ++ri) y4[ri] = partial_dot(S, ri, u);
        float o = D[r] * group_sum4(y4, lane);
#pragma unroll
        for (int i = 0; i <= r; ++i) o = fmaf(B[r * K + i], xe[i], o);
        if (!(lane & 1)) s_o[(r * R + hh) * kHeadDim + row_mine] = p.q_scale * o;
      }
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

template <typename StateT>
__global__ void __launch_bounds__(kThreads, 2) commit_kernel(const __grid_constant__ CommitParams p) {
  StateT* const state = static_cast<StateT*>(p.state);
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
  if (tid < R)  // the CTA's state slice into L2 while the conv state is rewritten
    bulk_prefetch_l2(state + ((size_t)b * Hv + (size_t)j * R + tid) * kHeadDim * kHeadDim,
                     (uint32_t)(kHeadDim * kHeadDim * sizeof(StateT)));

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

  // ---- S_m = exp(G_{m-1}) S0 + sum_{i<m} exp(g_{i+1} + .. + g_{m-1}) e_i k_i^T for each V head
  // (the same factors as the verify's outputs; every element streams through once)
  for (int hh = 0; hh < R; ++hh) {
    const int h = j * R + hh;
    StateT* Sg = state + ((size_t)b * Hv + h) * kHeadDim * kHeadDim;
    Slice S;
    load_slice(S, Sg, warp, lane);
    // the total decay over rows 0 .. m-1 scales S0; then rows m-1 down to 0 with the decay after them
    float gsum = 0.f;
    for (int r = 0; r < m; ++r) gsum += reinterpret_cast<const float*>(rec0 + (size_t)r * L.bytes + L.g_off)[h];
    const float2 d2 = make_float2(expf(gsum), expf(gsum));
#pragma unroll
    for (int ri = 0; ri < 4; ++ri)
#pragma unroll
      for (int qi = 0; qi < 4; ++qi) {
        float4& v = S.s[ri][qi];
        const float2 xy = __fmul2_rn(d2, make_float2(v.x, v.y)), zw = __fmul2_rn(d2, make_float2(v.z, v.w));
        v = make_float4(xy.x, xy.y, zw.x, zw.y);
      }
    float after = 0.f;  // g_{i+1} + .. + g_{m-1}
    for (int i = m - 1; i >= 0; --i) {
      const uint8_t* rec = rec0 + (size_t)i * L.bytes;
      const float dec = expf(after);
      after += reinterpret_cast<const float*>(rec + L.g_off)[h];
      float4 u[4];
      load_keys(reinterpret_cast<const float*>(rec + L.khat_off) + (size_t)j * kHeadDim, lane, u);
      const float4 e4 = *reinterpret_cast<const float4*>(
          reinterpret_cast<const float*>(rec + L.e_off) + (size_t)h * kHeadDim + warp * 16 + (lane >> 3) * 4);
      const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
      for (int ri = 0; ri < 4; ++ri) {
        const float c = dec * ev[ri];
        const float2 c2 = make_float2(c, c);
#pragma unroll
        for (int qi = 0; qi < 4; ++qi) {
          float4& v = S.s[ri][qi];
          const float2 xy = __ffma2_rn(c2, make_float2(u[qi].x, u[qi].y), make_float2(v.x, v.y));
          const float2 zw = __ffma2_rn(c2, make_float2(u[qi].z, u[qi].w), make_float2(v.z, v.w));
          v = make_float4(xy.x, xy.y, zw.x, zw.y);
        }
      }
    }
    store_slice(S, Sg, warp, lane);
  }
}

size_t verify_smem_bytes(int K, int R) {
  const size_t n_oct = 32 + 16 * (size_t)R;
  return 16 * n_oct * (K + 3 + 4) +
         sizeof(float) * ((size_t)2 * K * kHeadDim + (size_t)2 * K * R * kHeadDim + 2 * K + 2 * K * R +
                          2 * (size_t)K * K + 2 * (size_t)R * K * K + (size_t)R * K);
}

}  // namespace

int verify_max_rows() { return kMaxVerifyRows; }

bool verify_supported(int K, int Hk, int Hv) {
  return K >= 1 && K <= kMaxVerifyRows && verify_smem_bytes(K, Hv / Hk) <= kMaxVerifySmem;
}

namespace {
template <typename StateT>
cudaError_t configure_verify() {
  static int configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && configured[dev]) return cudaSuccess;
  for (auto kern : {verify_kernel<8, StateT>, verify_kernel<kMaxVerifyRows, StateT>}) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxVerifySmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
  }
  if (dev < 64) configured[dev] = 1;
  return cudaSuccess;
}

template <typename StateT>
cudaError_t launch_verify_t(const LaunchEnv& env, const VerifyParams& p, int B, int K, int Hk, int Hv) {
  cudaError_t e = configure_verify<StateT>();
  if (e != cudaSuccess) return e;
  const size_t smem = verify_smem_bytes(K, Hv / Hk);
  if (K <= 8)
    verify_kernel<8, StateT><<<dim3(Hk, B), kThreads, smem, env.stream>>>(p);
  else
    verify_kernel<kMaxVerifyRows, StateT><<<dim3(Hk, B), kThreads, smem, env.stream>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_verify(const LaunchEnv& env, const uint16_t* x, const uint16_t* conv_w, const uint16_t* conv_state,
                          const float* g, const float* beta, const void* state, bool fp16_state, const uint16_t* z,
                          const uint16_t* norm_w, float q_scale, float l2_eps, float rms_eps, uint16_t* out,
                          void* stash, int B, int K, int Hk, int Hv) {
  if (B <= 0) return cudaSuccess;
  VerifyParams p;
  p.x = x; p.conv_w = conv_w; p.conv_state = conv_state; p.g = g; p.beta = beta; p.state = state; p.z = z;
  p.norm_w = norm_w; p.out = out; p.stash = static_cast<uint8_t*>(stash);
  p.q_scale = q_scale; p.l2_eps = l2_eps; p.rms_eps = rms_eps;
  p.K = K; p.Hk = Hk; p.Hv = Hv;
  return fp16_state ? launch_verify_t<__half>(env, p, B, K, Hk, Hv) : launch_verify_t<float>(env, p, B, K, Hk, Hv);
}

cudaError_t launch_verify_commit(const LaunchEnv& env, const int32_t* committed, const void* stash,
                                 uint16_t* conv_state, void* state, bool fp16_state, int B, int K, int Hk, int Hv) {
  if (B <= 0) return cudaSuccess;
  CommitParams p;
  p.committed = committed; p.stash = static_cast<const uint8_t*>(stash); p.conv_state = conv_state;
  p.state = state; p.err = env.err; p.K = K; p.Hk = Hk; p.Hv = Hv;
  if (fp16_state)
    commit_kernel<__half><<<dim3(Hk, B), kThreads, 0, env.stream>>>(p);
  else
    commit_kernel<float><<<dim3(Hk, B), kThreads, 0, env.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
