// conv1d.cu -- causal depthwise conv1d (width 4) + SiLU over packed variable-length sequences.
//
// pegainfer PR #1152 "Reference golden for the GDN sublayer", Summary (depthwise conv, conv
// kernel 4, no bias) and "Commands + measured numbers" (the conv leg is a bf16 tensor compared
// bit-exact).  Memory-bound: every thread owns 8 consecutive channels (one 16-byte vector) and
// walks a run of consecutive tokens, keeping the 3 previous raw inputs in registers, so each
// input vector is read once per run (plus a 3-token halo) and each output vector written once.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kRun = 8;           // tokens per thread
constexpr int kThreadsX = 128;    // channel octets per block

struct Oct {
  float v[8];
};

__device__ __forceinline__ Oct load_oct(const uint16_t* p) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  Oct o;
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o.v[2 * i] = __uint_as_float(w[i] << 16);
    o.v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  return o;
}

__device__ __forceinline__ Oct zero_oct() {
  Oct o;
#pragma unroll
  for (int i = 0; i < 8; ++i) o.v[i] = 0.f;
  return o;
}

// the conv state of 8 channels: [8][3] bf16 = 48 contiguous bytes; slot j of channel i at i*3+j
__device__ __forceinline__ void load_state_oct(const uint16_t* p, Oct (&h)[3]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  uint4 a = q[0], b = q[1], c = q[2];
  const uint32_t w[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
  for (int e = 0; e < 24; ++e) {
    const uint32_t word = w[e >> 1];
    const float f = __uint_as_float((e & 1) ? (word & 0xFFFF0000u) : (word << 16));
    h[e % 3].v[e / 3] = f;
  }
}

// first sequence index n with cu[n+1] > t (cu is non-decreasing, cu[0] = 0, cu[N] = T)
__device__ __forceinline__ int seq_of_token(const int32_t* cu, int N, int t) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid + 1) > t) hi = mid; else lo = mid + 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreadsX, 4) conv1d_silu_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, const int32_t* __restrict__ cu,
    int N, int T, int C, const uint16_t* __restrict__ state_in, uint16_t* __restrict__ y,
    unsigned* err) {
  const int oct = blockIdx.x * kThreadsX + threadIdx.x;
  const int C8 = C >> 3;
  if (oct >= C8) return;
  const int t0 = blockIdx.y * kRun;
  if (t0 >= T) return;
  const int t1 = min(T, t0 + kRun);
  const int c = oct * 8;

  // weights of the 8 channels: [8][4] bf16 = 64 contiguous bytes
  float wt[8][4];
  {
    const uint4* q = reinterpret_cast<const uint4*>(w + (size_t)c * 4);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 u = __ldg(q + j);
      const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t word = ww[e >> 1];
        wt[2 * j + (e >> 2)][e & 3] = __uint_as_float((e & 1) ? (word & 0xFFFF0000u) : (word << 16));
      }
    }
  }

  int n = seq_of_token(cu, N, t0);
  int s = __ldg(cu + n), e = __ldg(cu + n + 1);
  if (s < 0 || e > T || s > t0 || e <= t0) { raise_error(err, kErrDeviceArgument); return; }

  // history: raw inputs at t-3, t-2, t-1 (index 0 = oldest)
  Oct h[3];
  auto history_at = [&](int t, int seq, int seq_start) {
    // fills h with the three raw inputs before token t of sequence `seq`
    Oct st[3];
    const bool need_state = (t - seq_start) < 3;
    if (need_state) {
      if (state_in) load_state_oct(state_in + ((size_t)seq * C + c) * 3, st);
      else { st[0] = zero_oct(); st[1] = zero_oct(); st[2] = zero_oct(); }
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int p = t - 3 + i;
      if (p >= seq_start) h[i] = load_oct(x + (size_t)p * C + c);
      else {  // p = seq_start - 3 + j  ->  slot j (selects keep st in registers)
        const int j = 3 - (seq_start - p);
#pragma unroll
        for (int k = 0; k < 8; ++k) h[i].v[k] = j == 0 ? st[0].v[k] : (j == 1 ? st[1].v[k] : st[2].v[k]);
      }
    }
  };
  history_at(t0, n, s);

  // all raw inputs of the run first, so that the whole run's loads are in flight together
  uint4 raw[kRun];
#pragma unroll
  for (int i = 0; i < kRun; ++i)
    if (t0 + i < t1) raw[i] = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + i) * C + c);
#pragma unroll
  for (int i = 0; i < kRun; ++i) {
    const int t = t0 + i;
    if (t >= t1) break;
    while (t >= e) {  // next sequence (skips empty ones)
      ++n;
      if (n >= N) { raise_error(err, kErrDeviceArgument); return; }
      s = e;
      e = __ldg(cu + n + 1);
      if (e < s || e > T) { raise_error(err, kErrDeviceArgument); return; }
      if (t < e) history_at(t, n, s);
    }
    Oct cur;
    {
      const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        cur.v[2 * k] = __uint_as_float(w4[k] << 16);
        cur.v[2 * k + 1] = __uint_as_float(w4[k] & 0xFFFF0000u);
      }
    }
    uint32_t packed[4];
#pragma unroll
    for (int q = 0; q < 8; q += 2) {
      float a[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int ch = q + u;
        float acc = wt[ch][0] * h[0].v[ch];
        acc = fmaf(wt[ch][1], h[1].v[ch], acc);
        acc = fmaf(wt[ch][2], h[2].v[ch], acc);
        acc = fmaf(wt[ch][3], cur.v[ch], acc);
        a[u] = acc * rcp_approx(1.0f + ex2_approx(-acc * kLog2e));  // silu(acc)
      }
      packed[q >> 1] = pack_bf2(a[0], a[1]);
    }
    *reinterpret_cast<uint4*>(y + (size_t)t * C + c) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    h[0] = h[1];
    h[1] = h[2];
    h[2] = cur;
  }
}

// conv_state_out[n] = the last 3 raw inputs of sequence n (conv state shifted); one thread per
// (sequence, channel octet) reads everything it needs before writing, so the output may alias
// the input state.
__global__ void conv1d_state_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ cu, int N,
                                    int T, int C, const uint16_t* state_in, uint16_t* state_out,
                                    unsigned* err) {
  const int C8 = C >> 3;
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)N * C8) return;
  const int n = (int)(idx / C8);
  const int c = (int)(idx % C8) * 8;
  const int s = __ldg(cu + n), e = __ldg(cu + n + 1);
  if (s < 0 || e < s || e > T) { raise_error(err, kErrDeviceArgument); return; }
  const int L = e - s;
  Oct st[3];
  if (state_in) load_state_oct(state_in + ((size_t)n * C + c) * 3, st);
  else { st[0] = zero_oct(); st[1] = zero_oct(); st[2] = zero_oct(); }
  Oct out[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int p = L - 3 + j;  // position relative to the sequence start
    out[j] = p >= 0 ? load_oct(x + (size_t)(s + p) * C + c) : st[3 + p];
  }
  uint16_t vals[24];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 3; ++j) vals[i * 3 + j] = f2bf(out[j].v[i]);  // exact: inputs are bf16
  uint4* dst = reinterpret_cast<uint4*>(state_out + ((size_t)n * C + c) * 3);
  const uint32_t* v32 = reinterpret_cast<const uint32_t*>(vals);
  dst[0] = make_uint4(v32[0], v32[1], v32[2], v32[3]);
  dst[1] = make_uint4(v32[4], v32[5], v32[6], v32[7]);
  dst[2] = make_uint4(v32[8], v32[9], v32[10], v32[11]);
}

}  // namespace

cudaError_t launch_conv1d_prefill(const LaunchEnv& env, const uint16_t* x, const uint16_t* w,
                                  const int32_t* cu, int N, int T, int C, const uint16_t* state_in,
                                  uint16_t* state_out, uint16_t* y) {
  const int C8 = C / 8;
  if (T > 0) {
    dim3 grid((C8 + kThreadsX - 1) / kThreadsX, (T + kRun - 1) / kRun);
    conv1d_silu_kernel<<<grid, kThreadsX, 0, env.stream>>>(x, w, cu, N, T, C, state_in, y, env.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (state_out) {
    const long work = (long)N * C8;
    const int threads = 256;
    conv1d_state_kernel<<<(unsigned)((work + threads - 1) / threads), threads, 0, env.stream>>>(
        x, cu, N, T, C, state_in, state_out, env.err);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace gdn
