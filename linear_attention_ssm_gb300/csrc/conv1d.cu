// conv1d.cu -- causal depthwise conv1d (width 4) + SiLU over packed variable-length sequences.
//
// pegainfer PR #1152 "Reference golden for the GDN sublayer", Summary (depthwise conv, conv
// kernel 4, no bias) and "Commands + measured numbers" (the conv leg is a bf16 tensor compared
// bit-exact).  Memory-bound: tiles of 128 channels x 64 tokens (plus the 3-token halo) are staged
// in shared memory by TMA through a 4-deep ring per CTA, each thread slides the 4-tap window over
// 16 tokens of a channel pair, and every output pair is written once as one 32-bit store.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

// Prefill kernel: persistent CTAs (three per SM) walk (channel slab, token tile) items; each item's
// raw inputs (kSlab channels x (kTile + 3) tokens, the 3-token halo included) are staged in shared
// memory by TMA through a kStages-deep ring, so every SM keeps ~200 KB of loads in flight.  Thread
// (channel pair, token quarter) slides a 4-tap window over its 16 tokens.
constexpr int kSlab = 128;                     // channels per tile: 256-byte rows
constexpr int kTile = 64;                      // tokens per tile
constexpr int kHalo = kConvWidth - 1;          // 3 earlier tokens
constexpr int kRows = kTile + kHalo;           // rows staged per tile
constexpr int kStages = 4;
constexpr uint32_t kStageBytes = kRows * kSlab * 2;  // 17,152
constexpr int kConvThreads = 256;              // 64 channel pairs x 4 token quarters
constexpr int kQuarter = kTile / 4;
constexpr uint32_t kConvSmem = kStages * kStageBytes + 64 + 128;
constexpr uint32_t kConvWait = 1u << 22;       // polls of one stage barrier before giving up

struct ConvParams {
  CUtensorMap tmap;  // x [T][C] bf16, box kSlab x kRows, no swizzle
  const uint16_t* w;
  const int32_t* cu;
  const uint16_t* state_in;
  uint16_t* y;
  unsigned* err;
  int N, T, C, nslab, ntile;
};

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

__device__ __forceinline__ float2 bf2x2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

__global__ void __launch_bounds__(kConvThreads, 3) conv1d_silu_kernel(const __grid_constant__ ConvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kStages * kStageBytes);
  const int tid = threadIdx.x, cp = tid & 63, tq = tid >> 6;
  const long items = (long)p.nslab * p.ntile;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
    prefetch_tensormap(&p.tmap);
  }
  __syncthreads();
  auto issue = [&](long item, int s) {
    const int tile = (int)(item / p.nslab), slab = (int)(item - (long)tile * p.nslab);
    mbar_arrive_expect_tx(smem_u32(&full[s]), kStageBytes);
    tma_load_2d(smem_u32(sm + s * kStageBytes), &p.tmap, slab * kSlab, tile * kTile - kHalo, smem_u32(&full[s]));
  };
  if (tid == 0) {
    for (int k = 0; k < kStages; ++k) {
      const long item = blockIdx.x + (long)k * gridDim.x;
      if (item < items) issue(item, k);
    }
  }

  int k = 0;
  long item = blockIdx.x;
  int n = -1;  // sequence of this thread's last first token
  for (; item < items; item += gridDim.x, ++k) {
    const int s = k % kStages;
    const bool got = mbar_wait(smem_u32(&full[s]), (uint32_t)((k / kStages) & 1), kConvWait);
    if (!got) raise_error(p.err, kErrTimeout);
    if (!__syncthreads_and(got ? 1 : 0)) break;
    const int tile = (int)(item / p.nslab), slab = (int)(item - (long)tile * p.nslab);
    const int c = slab * kSlab + 2 * cp;
    const int t_first = tile * kTile + tq * kQuarter;
    const uint8_t* st = sm + s * kStageBytes + cp * 4;  // row r holds token tile * kTile - kHalo + r
    auto x_at = [&](int t) { return bf2x2(*reinterpret_cast<const uint32_t*>(st + (t - tile * kTile + kHalo) * (kSlab * 2))); };
    if (t_first < p.T) {
      // weights of channels c, c + 1: [2][4] bf16
      const uint4 wu = __ldg(reinterpret_cast<const uint4*>(p.w + (size_t)c * 4));
      const float2 w01 = bf2x2(wu.x), w23 = bf2x2(wu.y), w45 = bf2x2(wu.z), w67 = bf2x2(wu.w);
      const float wa[4] = {w01.x, w01.y, w23.x, w23.y}, wb[4] = {w45.x, w45.y, w67.x, w67.y};
      // the sequence of t_first: this thread's tokens only grow from item to item, so advance the
      // sequence it looked up last (one binary search per CTA lifetime)
      if (n < 0) n = seq_of_token(p.cu, p.N, t_first);
      int ss = __ldg(p.cu + n), se = __ldg(p.cu + n + 1);
      while (se <= t_first && n + 1 < p.N) {
        ++n;
        ss = se;
        se = __ldg(p.cu + n + 1);
      }
      bool bad = ss < 0 || se > p.T || ss > t_first || se <= t_first;
      const float2 w0 = make_float2(wa[0], wb[0]), w1 = make_float2(wa[1], wb[1]), w2 = make_float2(wa[2], wb[2]),
                   w3 = make_float2(wa[3], wb[3]);
      auto emit = [&](int t, float2 x0, float2 x1, float2 x2, float2 x3) {  // x0 oldest, x3 = token t
        float2 acc = __fmul2_rn(w0, x0);
        acc = __ffma2_rn(w1, x1, acc);
        acc = __ffma2_rn(w2, x2, acc);
        acc = __ffma2_rn(w3, x3, acc);
        const float2 e = __fmul2_rn(acc, make_float2(-kLog2e, -kLog2e));
        const float2 d = __fadd2_rn(make_float2(ex2_approx(e.x), ex2_approx(e.y)), make_float2(1.f, 1.f));
        const float2 o = __fmul2_rn(acc, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
        *reinterpret_cast<uint32_t*>(p.y + (size_t)t * p.C + c) = pack_bf2(o.x, o.y);
      };
      if (!bad && ss <= t_first - kHalo && se >= t_first + kQuarter) {
        // the common case: the 16 tokens and their halo lie inside one sequence (and inside T)
        float2 xv[kQuarter + kHalo];
#pragma unroll
        for (int r = 0; r < kQuarter + kHalo; ++r) xv[r] = x_at(t_first - kHalo + r);
#pragma unroll
        for (int i = 0; i < kQuarter; ++i) emit(t_first + i, xv[i], xv[i + 1], xv[i + 2], xv[i + 3]);
      } else if (!bad) {
        float2 h[3];  // raw inputs at t - 3, t - 2, t - 1
        auto history = [&](int t) {  // the three raw inputs before token t of the sequence starting at ss
          float2 sv[3] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          if (t - ss < kHalo && p.state_in) {  // channels c, c + 1: 6 bf16 = three words, slot j of channel i at 3i + j
            const uint32_t* q = reinterpret_cast<const uint32_t*>(p.state_in + ((size_t)n * p.C + c) * 3);
            const uint32_t u0 = __ldg(q), u1 = __ldg(q + 1), u2 = __ldg(q + 2);
            const float2 a = bf2x2(u0), b = bf2x2(u1), d = bf2x2(u2);
            sv[0] = make_float2(a.x, b.y);
            sv[1] = make_float2(a.y, d.x);
            sv[2] = make_float2(b.x, d.y);
          }
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            const int pos = t - 3 + i;
            if (pos >= ss) {
              h[i] = x_at(pos);
            } else {  // pos = ss - 3 + j  ->  state slot j
              const int j = 3 - (ss - pos);
              h[i] = j == 0 ? sv[0] : (j == 1 ? sv[1] : sv[2]);
            }
          }
        };
        history(t_first);
        for (int i = 0; i < kQuarter; ++i) {
          const int t = t_first + i;
          if (t >= p.T) break;
          while (t >= se) {  // next sequence (skips empty ones)
            ++n;
            if (n >= p.N) { bad = true; break; }
            ss = se;
            se = __ldg(p.cu + n + 1);
            if (se < ss || se > p.T) { bad = true; break; }
            if (t < se) history(t);
          }
          if (bad) break;
          const float2 cur = x_at(t);
          emit(t, h[0], h[1], h[2], cur);
          h[0] = h[1];
          h[1] = h[2];
          h[2] = cur;
        }
      }
      if (bad) raise_error(p.err, kErrDeviceArgument);
    }
    fence_proxy_async_smem();  // this stage's reads precede the TMA write that refills it
    __syncthreads();
    if (tid == 0) {
      const long next = item + (long)kStages * gridDim.x;
      if (next < items) issue(next, s);
    }
  }
  // after an early exit, let the loads still in flight land before the CTA leaves (bounded)
  if (tid == 0) {
    for (int j = 0; j < kStages; ++j, item += gridDim.x, ++k) {
      if (item >= items) break;
      mbar_wait(smem_u32(&full[k % kStages]), (uint32_t)((k / kStages) & 1), kConvWait);
    }
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
  static int configured[64] = {0};
  const int C8 = C / 8;
  if (T > 0) {
    ConvParams p;
    memset(&p, 0, sizeof p);
    cudaError_t e = encode_bf16_2d(&p.tmap, x, (uint64_t)C, (uint64_t)T, (uint64_t)C * 2, kSlab, kRows);
    if (e != cudaSuccess) return e;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
      e = cudaFuncSetAttribute(conv1d_silu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kConvSmem);
      if (e != cudaSuccess) return e;
      configured[dev] = 1;
    }
    p.w = w; p.cu = cu; p.state_in = state_in; p.y = y; p.err = env.err;
    p.N = N; p.T = T; p.C = C; p.nslab = C / kSlab; p.ntile = (T + kTile - 1) / kTile;
    int sms = 0;
    if ((e = device_sm_count(&sms)) != cudaSuccess) return e;
    const long items = (long)p.nslab * p.ntile;
    const long slots = 3L * sms;  // three CTAs per SM (69 KB of shared memory, 80 registers)
    conv1d_silu_kernel<<<(unsigned)(items < slots ? items : slots), kConvThreads, kConvSmem, env.stream>>>(p);
    e = cudaGetLastError();
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
