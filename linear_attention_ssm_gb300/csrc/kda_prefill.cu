// kda_prefill.cu -- the KDA recurrence over packed variable-length sequences (the prefill's
// recurrent leg), token by token, with each head's fp32 [value, key] state held in registers for
// the whole sequence.
//
// GLM-5.3-Flash kernel TDD ledger, slices I2 (an fp32 state indexed [value, key], a per-channel
// decay clamped then exponentiated, its own q output scale), I2a (q and k normalised as
// x / sqrt(sum x^2 + eps)) and I4 (the prefill's state and outputs match the sequential recurrence
// at every length, 63, 64 and 65 tokens included).  Per token and V head:
//   S <- S diag(exp(max(g, g_min)));   e = beta (v - S k);   S <- S + e k^T;   o = q_scale S q
// then, when z is given, the sigmoid-gated RMSNorm of the GDN sublayer.
//
// One CTA per (V head, sequence).  Warp w holds value rows 16w .. 16w + 15 of the head's state and
// lane l the key columns 4l .. 4l + 3 of each row, so both contractions of a token (S k and S q)
// are warp-shuffle reductions and no step of a token waits for another warp: the arithmetic of a
// token is that of the KDA decode kernel up to the order of the four-term sums in each lane.  The
// token inputs (q and k of the K head, v, z, the per-channel decay and beta of the V head) are
// staged in shared memory 16 tokens at a time by asynchronous copies, double-buffered so that the
// next block streams in while this one is computed.  What does not depend on the state -- each
// token's normalised q and k and its per-channel decay factors -- is formed once per block by all
// eight warps together (a token per warp), so the chain from one token to the next holds only the
// state's own work; the block's fp32 outputs are likewise normalised by all warps together at the
// end of the block.
//
// This is the sequential form: per token it does O(Dv Dk) CUDA-core work on every head, so it is
// bound by instruction issue, not by memory.
#include <string.h>

#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = kHeadDim / kWarps;  // 16
constexpr int kBlockTokens = 16;                 // tokens per staged block

// One staged block of tokens; every array starts on a 16-byte boundary.
struct Stage {
  uint16_t q[kBlockTokens][kHeadDim];  // bf16, the K head's q row
  uint16_t k[kBlockTokens][kHeadDim];  // bf16, the K head's k row
  uint16_t v[kBlockTokens][kHeadDim];  // bf16, the V head's v row
  uint16_t z[kBlockTokens][kHeadDim];  // bf16, the output gate's input
  float g[kBlockTokens][kHeadDim];     // per-channel log decay
  float beta[kBlockTokens];
};

struct Smem {
  Stage st[2];
  float qn[kBlockTokens][kHeadDim];  // the block's normalised q
  float kn[kBlockTokens][kHeadDim];  // the block's normalised k
  float o[kBlockTokens][kHeadDim];   // q_scale S q of the block's tokens, before the norm
};
static_assert(sizeof(Stage) % 16 == 0, "stage buffers must stay 16-byte aligned");

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// waits until at most one committed group of this thread is still in flight
__device__ __forceinline__ void cp_async_wait_all_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Same lane layout and pairwise additions as the decode kernel's reduction: lanes 2i and 2i + 1
// return the warp-wide total of v[i].
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

// a.x b.x + a.y b.y + a.z b.z + a.w b.w as two f32x2 products summed pairwise
__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  const float2 p = __ffma2_rn(make_float2(a.z, a.w), make_float2(b.z, b.w),
                              __fmul2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y)));
  return p.x + p.y;
}

__device__ __forceinline__ float4 bf16x4(uint2 u) {
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xFFFF0000u));
}

// Issues the copies of tokens t0 .. t0 + nt - 1 (nt <= kBlockTokens) into one stage buffer.
__device__ __forceinline__ void stage_block(Stage& s, const uint16_t* qkv, const float* g, const float* beta,
                                            const uint16_t* z, int t0, int nt, int C, int Hk, int Hv, int j, int h,
                                            int tid) {
  // q, k, v and z: per token 16 pieces of 16 bytes each (256 copies per array)
  for (int w = tid; w < 4 * kBlockTokens * 16; w += kThreads) {
    const int arr = w / (kBlockTokens * 16), tt = (w >> 4) % kBlockTokens, piece = w & 15;
    if (tt >= nt) continue;
    const size_t t = (size_t)(t0 + tt);
    const uint16_t* src;
    uint16_t* dst;
    if (arr == 0) {
      src = qkv + t * C + (size_t)j * kHeadDim;
      dst = s.q[tt];
    } else if (arr == 1) {
      src = qkv + t * C + (size_t)(Hk + j) * kHeadDim;
      dst = s.k[tt];
    } else if (arr == 2) {
      src = qkv + t * C + (size_t)(2 * Hk + h) * kHeadDim;
      dst = s.v[tt];
    } else {
      if (!z) continue;
      src = z + (t * Hv + h) * kHeadDim;
      dst = s.z[tt];
    }
    cp_async16(dst + piece * 8, src + piece * 8);
  }
  // the decay: per token 32 pieces of four floats
  for (int w = tid; w < kBlockTokens * 32; w += kThreads) {
    const int tt = w >> 5, piece = w & 31;
    if (tt >= nt) continue;
    cp_async16(&s.g[tt][piece * 4], g + ((size_t)(t0 + tt) * Hv + h) * kHeadDim + piece * 4);
  }
  if (tid < nt) cp_async4(&s.beta[tid], beta + (size_t)(t0 + tid) * Hv + h);
}

__global__ void __launch_bounds__(kThreads, 2) kda_prefill_kernel(
    const uint16_t* __restrict__ qkv, const float* __restrict__ g, float g_min, const float* __restrict__ beta,
    const int32_t* __restrict__ cu, int T, int Hk, int Hv, float q_scale, float l2_eps, const float* state_in,
    float* state_out, const uint16_t* __restrict__ z, const uint16_t* __restrict__ norm_w, float rms_eps,
    uint16_t* __restrict__ out, unsigned* err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int h = blockIdx.x;  // V head
  const int n = blockIdx.y;  // sequence
  const int j = h / (Hv / Hk);
  const int C = (2 * Hk + Hv) * kHeadDim;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int start = __ldg(cu + n), end = __ldg(cu + n + 1);
  if (start < 0 || end < start || end > T) {  // uniform over the CTA: nothing is read or written
    if (tid == 0) raise_error(err, kErrDeviceArgument);
    return;
  }

  // the warp's 16 state rows: row i is value index 16 warp + i, this lane's key columns 4 lane ..
  const size_t sbase = ((size_t)n * Hv + h) * kHeadDim * kHeadDim + (size_t)warp * kRowsPerWarp * kHeadDim;
  float4 row[kRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i)
    row[i] = state_in ? reinterpret_cast<const float4*>(state_in + sbase)[i * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 wn = make_float4(0.f, 0.f, 0.f, 0.f);
  if (z) wn = bf16x4(__ldg(reinterpret_cast<const uint2*>(norm_w) + lane));

  const int L = end - start;
  const int nblk = (L + kBlockTokens - 1) / kBlockTokens;
  const int i_mine = (lane >> 1) & 15;  // the row whose sums this lane holds after a reduction
  if (nblk > 0) stage_block(sm.st[0], qkv, g, beta, z, start, min(kBlockTokens, L), C, Hk, Hv, j, h, tid);
  cp_async_commit();
  for (int bi = 0; bi < nblk; ++bi) {
    const int t0 = start + bi * kBlockTokens, nt = min(kBlockTokens, end - t0);
    const Stage& cur = sm.st[bi & 1];
    if (bi + 1 < nblk)
      stage_block(sm.st[(bi + 1) & 1], qkv, g, beta, z, t0 + kBlockTokens, min(kBlockTokens, end - t0 - kBlockTokens),
                  C, Hk, Hv, j, h, tid);
    cp_async_commit();
    cp_async_wait_all_but_one();  // this block's copies (every group but the one just issued)
    __syncthreads();

    // ---- the state-independent quantities of the block's tokens, a token per warp: q and k
    // normalised as x / sqrt(sum x^2 + eps), and the decay factors exp(max(g, g_min)) in place of g
    {
      Stage& cw = sm.st[bi & 1];
      for (int tt = warp; tt < nt; tt += kWarps) {
        const float4 q4 = bf16x4(*reinterpret_cast<const uint2*>(&cw.q[tt][lane * 4]));
        const float4 k4 = bf16x4(*reinterpret_cast<const uint2*>(&cw.k[tt][lane * 4]));
        float sq = 0.f, sk = 0.f;
        sq = fmaf(q4.x, q4.x, sq); sq = fmaf(q4.y, q4.y, sq); sq = fmaf(q4.z, q4.z, sq); sq = fmaf(q4.w, q4.w, sq);
        sk = fmaf(k4.x, k4.x, sk); sk = fmaf(k4.y, k4.y, sk); sk = fmaf(k4.z, k4.z, sk); sk = fmaf(k4.w, k4.w, sk);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
          sq += __shfl_xor_sync(0xffffffffu, sq, m);
          sk += __shfl_xor_sync(0xffffffffu, sk, m);
        }
        const float iq = rsqrtf(sq + l2_eps), ik = rsqrtf(sk + l2_eps);
        *reinterpret_cast<float4*>(&sm.qn[tt][lane * 4]) = make_float4(q4.x * iq, q4.y * iq, q4.z * iq, q4.w * iq);
        *reinterpret_cast<float4*>(&sm.kn[tt][lane * 4]) = make_float4(k4.x * ik, k4.y * ik, k4.z * ik, k4.w * ik);
        const float4 gv = *reinterpret_cast<const float4*>(&cw.g[tt][lane * 4]);
        *reinterpret_cast<float4*>(&cw.g[tt][lane * 4]) =
            make_float4(expf(fmaxf(gv.x, g_min)), expf(fmaxf(gv.y, g_min)), expf(fmaxf(gv.z, g_min)),
                        expf(fmaxf(gv.w, g_min)));
      }
    }
    __syncthreads();

    for (int tt = 0; tt < nt; ++tt) {
      const float4 qn = *reinterpret_cast<const float4*>(&sm.qn[tt][lane * 4]);
      const float4 kn = *reinterpret_cast<const float4*>(&sm.kn[tt][lane * 4]);
      // the decay of this lane's four key channels, and the key they multiply: (S diag(a)) k = S (a k)
      const float4 a4 = *reinterpret_cast<const float4*>(&cur.g[tt][lane * 4]);
      const float4 kd = make_float4(a4.x * kn.x, a4.y * kn.y, a4.z * kn.z, a4.w * kn.w);
      float d[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i)
        d[i] = dot4(row[i], kd);
      const float dsum = warp_sum16(d, lane);
      const float e_mine = cur.beta[tt] * (bf2f(cur.v[tt][warp * kRowsPerWarp + i_mine]) - dsum);
      float o[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const float e = __shfl_sync(0xffffffffu, e_mine, 2 * i);
        // S <- S diag(a) + e k^T, element by element fma(a, s, e k) in f32x2 pairs
        const float2 e2 = make_float2(e, e);
        const float2 xy = __ffma2_rn(make_float2(a4.x, a4.y), make_float2(row[i].x, row[i].y),
                                     __fmul2_rn(e2, make_float2(kn.x, kn.y)));
        const float2 zw = __ffma2_rn(make_float2(a4.z, a4.w), make_float2(row[i].z, row[i].w),
                                     __fmul2_rn(e2, make_float2(kn.z, kn.w)));
        row[i] = make_float4(xy.x, xy.y, zw.x, zw.y);
        o[i] = dot4(row[i], qn);
      }
      const float o_mine = warp_sum16(o, lane);
      if (!(lane & 1)) sm.o[tt][warp * kRowsPerWarp + i_mine] = q_scale * o_mine;
    }
    __syncthreads();

    // ---- the block's outputs: sigmoid-gated RMSNorm over each token's 128 values (o itself
    // without z), one token per warp at a time
    for (int tt = warp; tt < nt; tt += kWarps) {
      const float4 ov = *reinterpret_cast<const float4*>(&sm.o[tt][lane * 4]);
      float r[4] = {ov.x, ov.y, ov.z, ov.w};
      if (z) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) ss = fmaf(r[i], r[i], ss);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float rstd = rsqrtf(ss * (1.0f / kHeadDim) + rms_eps);
        const float4 zf = bf16x4(*reinterpret_cast<const uint2*>(&cur.z[tt][lane * 4]));
        r[0] = r[0] * rstd * wn.x * sigmoidf_(zf.x);
        r[1] = r[1] * rstd * wn.y * sigmoidf_(zf.y);
        r[2] = r[2] * rstd * wn.z * sigmoidf_(zf.z);
        r[3] = r[3] * rstd * wn.w * sigmoidf_(zf.w);
      }
      const size_t base = ((size_t)(t0 + tt) * Hv + h) * kHeadDim + lane * 4;
      *reinterpret_cast<uint2*>(out + base) = make_uint2(pack_bf2(r[0], r[1]), pack_bf2(r[2], r[3]));
    }
    __syncthreads();  // the next block restages the buffer read here and rewrites sm.o
  }

  if (state_out) {
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) reinterpret_cast<float4*>(state_out + sbase)[i * 32 + lane] = row[i];
  }
}

}  // namespace

size_t kda_prefill_smem_bytes() { return sizeof(Smem); }

cudaError_t launch_kda_prefill(const LaunchEnv& env, const uint16_t* qkv, const float* g, float g_min,
                               const float* beta, const int32_t* cu, int N, int T, int Hk, int Hv, float q_scale,
                               float l2_eps, const float* state_in, float* state_out, const uint16_t* z,
                               const uint16_t* norm_w, float rms_eps, uint16_t* out) {
  if (N <= 0) return cudaSuccess;
  static int configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(kda_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
    // the largest shared-memory carveout, so that two CTAs share an SM
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kda_prefill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  kda_prefill_kernel<<<dim3(Hv, N), kThreads, sizeof(Smem), env.stream>>>(
      qkv, g, g_min, beta, cu, T, Hk, Hv, q_scale, l2_eps, state_in, state_out, z, norm_w, rms_eps, out, env.err);
  return cudaGetLastError();
}

}  // namespace gdn
