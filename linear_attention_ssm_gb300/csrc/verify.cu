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
// (row, channel octet) in parallel from the conv state (which it does not modify), the L2 norms of every row's q and k, then per V
// head streams the head's 128 x 128 fp32 state into registers (16 rows per warp; a lane holds 4
// rows x 16 keys, so a row's dot product is a 16-term partial and a 3-level butterfly over the 8
// lanes of its group) and applies the K rows to it there -- decay, delta correction against the
// decayed state, output -- without storing it.  The rows' gated outputs go to `out`; the
// per-row keys, values, gates and raw conv inputs go to the stash.  The commit applies a row with
// the same routine, so the state it stores is bit for bit the state the verify's outputs came
// from.
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

// A warp owns 16 state rows of a V head; lane (rg, kg) = (lane / 8, lane % 8) holds rows
// 4 rg .. 4 rg + 3 of them over the 16 keys {32 q + 4 kg + e : q, e in 0..3} (4 float4 per row):
// every load or store instruction moves 4 rows x 128 contiguous bytes.
struct Slice {
  float4 s[4][4];  // [row][key quad]
};

__device__ __forceinline__ int slice_offset(int warp, int lane, int ri, int qi) {  // in floats, within a head
  return (warp * 16 + (lane >> 3) * 4 + ri) * kHeadDim + 32 * qi + 4 * (lane & 7);
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

// One token applied to the slice: S <- alpha S;  e = beta (v - S k);  S <- S + e k^T, in the
// decode step's order (delta against the decayed state: e = beta (v - alpha (S_old k))).
// `v_mine` is the value of the row whose sum this lane ends up holding (row (lane % 8) / 2 of
// its group).
__device__ __forceinline__ void apply_token(Slice& S, const float4 (&kn)[4], float alpha, float bt, float v_mine,
                                            int lane) {
  float d[4];
#pragma unroll
  for (int ri = 0; ri < 4; ++ri) d[ri] = partial_dot(S, ri, kn);
  const float em = bt * (v_mine - alpha * group_sum4(d, lane));
  const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
  for (int ri = 0; ri < 4; ++ri) {
    const float e = __shfl_sync(0xffffffffu, em, (lane & ~7) | (2 * ri));
    const float2 e2 = make_float2(e, e);
#pragma unroll
    for (int qi = 0; qi < 4; ++qi) {
      float4& r = S.s[ri][qi];
      const float2 xy = __ffma2_rn(a2, make_float2(r.x, r.y), __fmul2_rn(e2, make_float2(kn[qi].x, kn[qi].y)));
      const float2 zw = __ffma2_rn(a2, make_float2(r.z, r.w), __fmul2_rn(e2, make_float2(kn[qi].z, kn[qi].w)));
      r = make_float4(xy.x, xy.y, zw.x, zw.y);
    }
  }
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

__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const __grid_constant__ VerifyParams p) {
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
  float* s_ab = s_norm + 2 * K;                  // [K][R][2] alpha = exp(g), beta

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
  // conv state, in the decode step's order of operations
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
    for (int ch = 0; ch < 8; ++ch) {
      float acc = wv[ch * 4 + 0] * xw[0][ch];
      acc = fmaf(wv[ch * 4 + 1], xw[1][ch], acc);
      acc = fmaf(wv[ch * 4 + 2], xw[2][ch], acc);
      acc = fmaf(wv[ch * 4 + 3], xw[3][ch], acc);
      a[ch] = bf2f(f2bf(acc / (1.0f + expf(-acc))));  // the bf16 conv output
    }
    float* dst;
    if (o < 16) dst = s_q + r * kHeadDim + o * 8;
    else if (o < 32) dst = s_k + r * kHeadDim + (o - 16) * 8;
    else {
      const int hh = (o - 32) >> 4, oo = (o - 32) & 15;
      dst = s_v + (r * R + hh) * kHeadDim + oo * 8;
      uint4 vb;  // the v channels as bf16 (exact: they are bf16 values)
      vb.x = pack_bf2(a[0], a[1]); vb.y = pack_bf2(a[2], a[3]);
      vb.z = pack_bf2(a[4], a[5]); vb.w = pack_bf2(a[6], a[7]);
      *reinterpret_cast<uint4*>(p.stash + ((size_t)b * K + r) * L.bytes + L.v_off +
                                ((size_t)(j * R + hh) * kHeadDim + oo * 8) * 2) = vb;
    }
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) dst[ch] = a[ch];
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

  // ---- the K rows applied to each V head's state in registers (never stored)
  const int row_mine = warp * 16 + (lane >> 3) * 4 + ((lane & 7) >> 1);  // the row whose sums this lane holds
  for (int hh = 0; hh < R; ++hh) {
    const int h = j * R + hh;
    const float* Sg = p.state + ((size_t)b * Hv + h) * kHeadDim * kHeadDim;
    Slice S;
#pragma unroll
    for (int ri = 0; ri < 4; ++ri)
#pragma unroll
      for (int qi = 0; qi < 4; ++qi)
        S.s[ri][qi] = __ldg(reinterpret_cast<const float4*>(Sg + slice_offset(warp, lane, ri, qi)));
    for (int r = 0; r < K; ++r) {
      const int t = r * R + hh;
      float4 u[4];
      load_keys(s_k + r * kHeadDim, lane, u);
      apply_token(S, u, s_ab[2 * t], s_ab[2 * t + 1], s_v[t * kHeadDim + row_mine], lane);
      load_keys(s_q + r * kHeadDim, lane, u);
      float o[4];
#pragma unroll
      for (int ri = 0; ri < 4; ++ri) o[ri] = partial_dot(S, ri, u);
      const float om = group_sum4(o, lane);
      if (!(lane & 1)) s_o[t * kHeadDim + row_mine] = p.q_scale * om;
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
  const int row_mine = warp * 16 + (lane >> 3) * 4 + ((lane & 7) >> 1);
  for (int hh = 0; hh < R; ++hh) {
    const int h = j * R + hh;
    float* Sg = p.state + ((size_t)b * Hv + h) * kHeadDim * kHeadDim;
    Slice S;
#pragma unroll
    for (int ri = 0; ri < 4; ++ri)
#pragma unroll
      for (int qi = 0; qi < 4; ++qi) S.s[ri][qi] = *reinterpret_cast<const float4*>(Sg + slice_offset(warp, lane, ri, qi));
    for (int r = 0; r < m; ++r) {
      const uint8_t* rec = rec0 + (size_t)r * L.bytes;
      float4 u[4];
      load_keys(reinterpret_cast<const float*>(rec + L.khat_off) + (size_t)j * kHeadDim, lane, u);
      const float alpha = reinterpret_cast<const float*>(rec + L.alpha_off)[h];
      const float bt = reinterpret_cast<const float*>(rec + L.beta_off)[h];
      const float vm = bf2f(*reinterpret_cast<const uint16_t*>(rec + L.v_off + ((size_t)h * kHeadDim + row_mine) * 2));
      apply_token(S, u, alpha, bt, vm, lane);
    }
#pragma unroll
    for (int ri = 0; ri < 4; ++ri)
#pragma unroll
      for (int qi = 0; qi < 4; ++qi) *reinterpret_cast<float4*>(Sg + slice_offset(warp, lane, ri, qi)) = S.s[ri][qi];
  }
}

size_t verify_smem_bytes(int K, int R) {
  const size_t n_oct = 32 + 16 * (size_t)R;
  return 16 * n_oct * (K + 3 + 4) +
         sizeof(float) * ((size_t)2 * K * kHeadDim + (size_t)2 * K * R * kHeadDim + 2 * K + 2 * K * R);
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
