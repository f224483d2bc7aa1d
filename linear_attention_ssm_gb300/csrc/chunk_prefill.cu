// chunk_prefill.cu -- chunk-wise (WY) gated delta rule prefill on the tcgen05 tensor cores.
//
// The method: pegainfer PR #1152 "Reference golden for the GDN sublayer", Consumer / Shipped-line
// diff (prepare: head-expand q/k, L2-norm, split v; then cumsum -> A -> solve -> recompute ->
// state -> output) and Code review (f32 recurrent state carried across chunks); GLM-5.3-Flash
// kernel TDD ledger, slice I4 (chunk path equals the sequential state/output at 63/64/65).
//
// For one chunk of L <= 64 tokens with start state S0 (Dv x Dk, [value, key]), gamma_t the
// within-chunk cumulative sum of g, Gamma_t = exp(gamma_t) and k^, q^ the L2-normalised keys and
// queries (k^_t = ik_t k_t, q^_t = iq_t q_t with k_t, q_t the raw bf16 conv outputs):
//   A[t,j] = beta_t exp(gamma_t - gamma_j) k^_t.k^_j  (j < t),   T = (I + A)^-1
//   E      = T (diag(beta) V - diag(beta Gamma) K^ S0^T)                       (the WY solve)
//   O      = q_scale [diag(Gamma) Q^ S0^T + (mask_{j<=t} exp(gamma_t-gamma_j) Q^ K^^T) E]
//   S_L    = Gamma_L S0 + E^T diag(exp(gamma_L - gamma)) K^
// This file evaluates it "value-major", i.e. every product is written with the value index of
// the state as the 128-row M dimension of a tcgen05 MMA (M = 128, N in {64, 128}, K = 16 per
// instruction, bf16 operands in 128-byte-swizzled shared memory, fp32 accumulators in tensor
// memory).  The fp32 state itself lives in tensor memory for the whole sequence.
//
// Precision: operands that are exact in bf16 (the raw conv outputs q, k, v) are fed as they are;
// the L2-norm factors, beta and the decay exponentials are applied in fp32 as diagonal scalings
// in the epilogues.  fp32 operands on the state path (S0, the right-hand side R, the solve T,
// the scaled E) are split into bf16 hi + lo pairs, giving ~16-bit operands; products that only
// feed the output (S0 q, E P^T) use the hi part alone.
//
// One CTA of 128 threads per (sequence, V head); thread r owns row r of every accumulator (TMEM
// lane r).  The phases of a chunk run back to back, separated by mbarrier waits on the MMAs.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 128;

// ---- shared memory map (byte offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_QK = 0;         // 32 KB: 2 K-blocks x 128 rows (k tokens 0..63, q tokens 64..127)
constexpr uint32_t OFF_KT = 32768;     // 16 KB: K^T, 128 key rows x 64 tokens
constexpr uint32_t OFF_SHI = 49152;    // 32 KB: S0 hi, 2 K-blocks x 128 value rows
constexpr uint32_t OFF_SLO = 81920;    // 32 KB: S0 lo
constexpr uint32_t OFF_RHI = 114688;   // 16 KB: R hi, then E~ hi (128 value rows x 64 tokens)
constexpr uint32_t OFF_RLO = 131072;   // 16 KB: R lo, then E~ lo
constexpr uint32_t OFF_T = 147456;     // 16 KB: T hi (8 KB) + T lo (8 KB); then E bf16 (16 KB)
constexpr uint32_t OFF_P = 163840;     //  8 KB: P, 64 token rows x 64
constexpr uint32_t OFF_V = 172032;     // 16 KB: V, [64 tokens][128] bf16, plain row-major
constexpr uint32_t OFF_WORK = 188416;  // fp32 work: solve (A, T, block temp) or output staging
constexpr uint32_t LDA = 65;           // row stride (floats) of the solve matrices
constexpr uint32_t LDO = 132;          // row stride (floats) of the output staging
constexpr uint32_t WORK_BYTES = (2 * 64 * LDA + 3 * 256) * 4;  // 36352 >= 64 * LDO * 4
constexpr uint32_t OFF_VEC = OFF_WORK + WORK_BYTES;            // per-token vectors, 8 x 64 floats
constexpr uint32_t OFF_BAR = OFF_VEC + 8 * 64 * 4;             // 4 mbarriers + TMEM address
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;               // + alignment slack
static_assert(64 * LDO * 4 <= WORK_BYTES, "output staging must fit the work area");
static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

// ---- tensor memory columns (fp32, lane = value row)
constexpr uint32_t COL_S = 0;     // 128: the recurrent state
constexpr uint32_t COL_X = 128;   //  64: S0 K^T
constexpr uint32_t COL_E = 192;   //  64: E^T
constexpr uint32_t COL_O1 = 256;  //  64: S0 Q^T
constexpr uint32_t COL_O2 = 320;  //  64: E^T P^T
constexpr uint32_t COL_G = 384;   //  64: [K; Q] K^T (Gram, rows 0..63, and Q K^T, rows 64..127)
constexpr uint32_t TMEM_COLS = 512;

constexpr uint32_t kWaitLimit = 1u << 20;  // polls of one mbarrier before giving up

struct ChunkParams {
  const uint16_t* qkv;
  const float* g;
  const float* beta;
  const int32_t* cu;
  const float* state_in;
  float* state_out;
  const uint16_t* z;
  const uint16_t* norm_w;
  uint16_t* out;
  unsigned* err;
  int N, T, Hk, Hv;
  float q_scale, l2_eps, rms_eps;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint16_t ld_shared_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Writes 8 consecutive fp32 values (columns k0..k0+7 of `row`, k0 % 8 == 0) of an fp32 matrix
// as a bf16 hi/lo pair into two K-major swizzled tiles.
__device__ __forceinline__ void store8_split(uint32_t hi_tile, uint32_t lo_tile, uint32_t kb_stride, int row, int k0,
                                             const float* v) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = v[2 * i], b = v[2 * i + 1];
    const uint16_t ah = f2bf(a), bh = f2bf(b);
    h[i] = (uint32_t)ah | ((uint32_t)bh << 16);
    l[i] = pack_bf2(a - bf2f(ah), b - bf2f(bh));
  }
  const uint32_t off = sw128_offset(row, k0, kb_stride);
  st_shared_v4(hi_tile + off, h[0], h[1], h[2], h[3]);
  if (lo_tile) st_shared_v4(lo_tile + off, l[0], l[1], l[2], l[3]);
}

// CUDA-core stand-in of one M=128 MMA group for verification: thread r computes row r of
// D (+)= A * B^T from the same swizzled operand tiles and writes it to tensor memory.
template <int N, int K>
__device__ void emu_mma(uint32_t t_lane_col, uint32_t a_tile, uint32_t a_kbs, uint32_t b_tile, uint32_t b_kbs,
                        bool accumulate, int r) {
  float arow[K];
#pragma unroll 8
  for (int k = 0; k < K; ++k) arow[k] = bf2f(ld_shared_u16(a_tile + sw128_offset(r, k, a_kbs)));
  for (int n0 = 0; n0 < N; n0 += 32) {
    float d[32];
    if (accumulate) tmem_ld32(t_lane_col + n0, d);
    else {
#pragma unroll
      for (int i = 0; i < 32; ++i) d[i] = 0.f;
    }
    for (int n = 0; n < 32; ++n) {
      float s = 0.f;
#pragma unroll 8
      for (int k = 0; k < K; ++k) s = fmaf(arow[k], bf2f(ld_shared_u16(b_tile + sw128_offset(n0 + n, k, b_kbs))), s);
      d[n] += s;
    }
    tmem_st32(t_lane_col + n0, d);
  }
}

// T = (I + A)^-1 for a strictly lower triangular 64 x 64 A (row stride LDA), by 16 x 16 blocks:
// the four diagonal blocks by forward substitution (one thread per column), then the
// off-diagonal blocks by block distance d: T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj.
__device__ void solve_unit_lower(const float* sA, float* sT, float* sM, int tid) {
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15, o = b * 16;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float v = (i == c) ? 1.f : 0.f;
#pragma unroll
      for (int k = 0; k < i; ++k) v -= sA[(o + i) * LDA + o + k] * x[k];
      x[i] = (i < c) ? 0.f : v;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sT[(o + i) * LDA + o + c] = x[i];
  }
  for (int idx = tid; idx < 64 * 64; idx += kThreads) {
    const int r = idx >> 6, cc = idx & 63;
    if ((cc >> 4) > (r >> 4)) sT[r * LDA + cc] = 0.f;
  }
  __syncthreads();
  for (int d = 1; d < 4; ++d) {
    const int nb = 4 - d;
    for (int idx = tid; idx < nb * 256; idx += kThreads) {
      const int bi = idx >> 8, e = idx & 255, r = e >> 4, cc = e & 15;
      const int i = d + bi, jb = i - d;
      float acc = 0.f;
      for (int kb = jb; kb < i; ++kb)
#pragma unroll
        for (int u = 0; u < 16; ++u) acc = fmaf(sA[(i * 16 + r) * LDA + kb * 16 + u], sT[(kb * 16 + u) * LDA + jb * 16 + cc], acc);
      sM[bi * 256 + e] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < nb * 256; idx += kThreads) {
      const int bi = idx >> 8, e = idx & 255, r = e >> 4, cc = e & 15;
      const int i = d + bi, jb = i - d;
      float acc = 0.f;
      for (int u = 0; u <= r; ++u) acc = fmaf(sT[(i * 16 + r) * LDA + i * 16 + u], sM[bi * 256 + u * 16 + cc], acc);
      sT[(i * 16 + r) * LDA + jb * 16 + cc] = -acc;
    }
    __syncthreads();
  }
}

template <bool kEmulate>
__global__ void __launch_bounds__(kThreads, 1) chunk_prefill_kernel(const ChunkParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int h = blockIdx.x % p.Hv;
  const int n = blockIdx.x / p.Hv;
  const int ratio = p.Hv / p.Hk;
  const int kh = h / ratio;
  const int C = 2 * p.Hk * kHeadDim + p.Hv * kHeadDim;
  const int seq_s = __ldg(p.cu + n), seq_e = __ldg(p.cu + n + 1);
  if (seq_s < 0 || seq_e < seq_s || seq_e > p.T) {
    if (tid == 0) raise_error(p.err, kErrDeviceArgument);
    return;
  }

  float* s_gam = reinterpret_cast<float*>(sm + OFF_VEC);
  float* s_beta = s_gam + 64;
  float* s_ik = s_gam + 128;
  float* s_iq = s_gam + 192;
  float* s_cx = s_gam + 256;   // beta_t Gamma_t ik_t
  float* s_co = s_gam + 320;   // Gamma_t iq_t q_scale
  float* s_cs = s_gam + 384;   // exp(gamma_L - gamma_t) ik_t
  float* s_g = s_gam + 448;
  float* s_work = reinterpret_cast<float*>(sm + OFF_WORK);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 32);
  const uint32_t bar_g = smem_u32(&bars[0]), bar_x = smem_u32(&bars[1]), bar_e = smem_u32(&bars[2]),
                 bar_s = smem_u32(&bars[3]);

  if (tid == 0) {
    mbar_init(bar_g, 1);
    mbar_init(bar_x, 1);
    mbar_init(bar_e, 1);
    mbar_init(bar_s, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's lane quarter, column 0

  // ---- initial state -> tensor memory (thread r: value row r)
  {
    const size_t row_off = (((size_t)n * p.Hv + h) * kHeadDim + tid) * kHeadDim;
    for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
      float v[32];
      if (p.state_in) {
        const float4* src = reinterpret_cast<const float4*>(p.state_in + row_off + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 f = __ldg(src + i);
          v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      tmem_st32(tl + COL_S + c0, v);
    }
  }

  constexpr uint32_t ID64 = idesc_bf16_f32(128, 64);
  constexpr uint32_t ID128 = idesc_bf16_f32(128, 128);
  bool ok = true;
  uint32_t phase = 0;

  // one MMA group: either issued on the tensor cores by thread 0 and awaited on `bar`, or emulated
  auto finish_group = [&](uint32_t bar) {
    if constexpr (!kEmulate) {
      if (tid == 0) mma_commit(bar);
      const bool got = mbar_wait(bar, phase, kWaitLimit);
      if (!got) raise_error(p.err, kErrTimeout);
      ok = __syncthreads_and(got ? 1 : 0) != 0;
      tc_fence_after();
    } else {
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  };
  auto operands_ready = [&]() {  // smem operand writes by all threads -> visible to the MMA
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };

  for (int c0 = seq_s; c0 < seq_e && ok; c0 += kChunk, phase ^= 1u) {
    const int L = min(kChunk, seq_e - c0);

    // ================= prepare: loads, norms, K^T, cumsum
    if (tid < 64) {
      float gv = 0.f, bv = 0.f;
      if (tid < L) {
        gv = __ldg(p.g + (size_t)(c0 + tid) * p.Hv + h);
        bv = __ldg(p.beta + (size_t)(c0 + tid) * p.Hv + h);
      }
      s_g[tid] = gv;
      s_beta[tid] = bv;
    }
    for (int i = tid; i < 64 * 16; i += kThreads) {
      const int t = i >> 4, kc = i & 15;
      uint4 kq = make_uint4(0, 0, 0, 0), qq = kq, vv = kq;
      if (t < L) {
        const uint16_t* row = p.qkv + (size_t)(c0 + t) * C;
        qq = __ldg(reinterpret_cast<const uint4*>(row + kh * kHeadDim + kc * 8));
        kq = __ldg(reinterpret_cast<const uint4*>(row + p.Hk * kHeadDim + kh * kHeadDim + kc * 8));
        vv = __ldg(reinterpret_cast<const uint4*>(row + 2 * p.Hk * kHeadDim + h * kHeadDim + kc * 8));
      }
      const uint32_t swz = (uint32_t)(((kc & 7) ^ (t & 7)) << 4);
      const uint32_t kb = (uint32_t)(kc >> 3) * 16384u;
      st_shared_v4(sb + OFF_QK + kb + t * 128 + swz, kq.x, kq.y, kq.z, kq.w);
      st_shared_v4(sb + OFF_QK + kb + (64 + t) * 128 + swz, qq.x, qq.y, qq.z, qq.w);
      st_shared_v4(sb + OFF_V + t * 256 + kc * 16, vv.x, vv.y, vv.z, vv.w);
    }
    __syncthreads();
    {
      // L2 norms: thread t < 64 -> key row t, thread 64 + t -> query row t
      const int row = tid;
      float ss = 0.f;
#pragma unroll
      for (int kc = 0; kc < 16; ++kc) {
        const uint4 u = ld_shared_v4(sb + OFF_QK + (kc >> 3) * 16384 + row * 128 + (((kc & 7) ^ (row & 7)) << 4));
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = __uint_as_float(w4[e] << 16), b = __uint_as_float(w4[e] & 0xFFFF0000u);
          ss = fmaf(a, a, ss);
          ss = fmaf(b, b, ss);
        }
      }
      const float inv = 1.0f / sqrtf(ss + p.l2_eps);
      if (tid < 64) s_ik[tid] = inv; else s_iq[tid - 64] = inv;
      // K^T: thread = key index, 8 chunks of 8 tokens
      const int nk = tid;
#pragma unroll
      for (int tc = 0; tc < 8; ++tc) {
        uint32_t w4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t0 = tc * 8 + 2 * u;
          const uint32_t a = ld_shared_u16(sb + OFF_QK + sw128_offset(t0, nk, 16384));
          const uint32_t b = ld_shared_u16(sb + OFF_QK + sw128_offset(t0 + 1, nk, 16384));
          w4[u] = a | (b << 16);
        }
        st_shared_v4(sb + OFF_KT + nk * 128 + (((tc ^ (nk & 7)) & 7) << 4), w4[0], w4[1], w4[2], w4[3]);
      }
    }
    if (tid == 0) {
      float acc = 0.f;
      for (int t = 0; t < 64; ++t) { acc += s_g[t]; s_gam[t] = acc; }
    }
    __syncthreads();
    if (tid < 64) {
      const int t = tid;
      const float gam = s_gam[t], gamL = s_gam[L - 1];
      const float Gam = expf(gam);
      s_cx[t] = s_beta[t] * Gam * s_ik[t];
      s_co[t] = Gam * s_iq[t] * p.q_scale;
      s_cs[t] = (t < L) ? expf(gamL - gam) * s_ik[t] : 0.f;
    }
    operands_ready();

    // ================= Gram: G = [K; Q] K^T  (M = 128, N = 64, K = 128)
    if constexpr (!kEmulate) {
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          mma_bf16(tmem + COL_G, sw128_desc(sb + OFF_QK + off), sw128_desc(sb + OFF_QK + off), ID64, ks > 0);
        }
      }
    } else {
      emu_mma<64, 128>(tl + COL_G, sb + OFF_QK, 16384, sb + OFF_QK, 16384, false, tid);
    }
    finish_group(bar_g);
    if (!ok) break;

    // ================= A (rows 0..63) and P (rows 64..127) from the Gram tile
    {
      float gr[64];
      tmem_ld32(tl + COL_G, *reinterpret_cast<float(*)[32]>(gr));
      tmem_ld32(tl + COL_G + 32, *reinterpret_cast<float(*)[32]>(gr + 32));
      float* sA = s_work;
      if (tid < 64) {
        const int t = tid;
        const float bt = s_beta[t] * s_ik[t], gt = s_gam[t];
#pragma unroll 8
        for (int j = 0; j < 64; ++j) sA[t * LDA + j] = (j < t) ? bt * expf(gt - s_gam[j]) * gr[j] * s_ik[j] : 0.f;
      } else {
        const int t = tid - 64;
        const float qt = s_iq[t] * p.q_scale, gt = s_gam[t];
#pragma unroll
        for (int j0 = 0; j0 < 64; j0 += 8) {
          float v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = j0 + u;
            v[u] = (j <= t) ? qt * expf(gt - s_gam[j]) * gr[j] * s_ik[j] : 0.f;
          }
          store8_split(sb + OFF_P, 0, 0, t, j0, v);
        }
      }
    }
    __syncthreads();

    // ================= solve: T = (I + A)^-1, then T hi/lo -> operand tiles
    {
      float* sA = s_work;
      float* sTf = s_work + 64 * LDA;
      float* sM = s_work + 2 * 64 * LDA;
      solve_unit_lower(sA, sTf, sM, tid);
      for (int i = tid; i < 64 * 8; i += kThreads) {
        const int t = i >> 3, k0 = (i & 7) * 8;
        store8_split(sb + OFF_T, sb + OFF_T + 8192, 0, t, k0, sTf + t * LDA + k0);
      }
    }
    // ================= S0 -> hi/lo operand tiles; tensor memory state <- Gamma_L S0
    {
      const float gL = expf(s_gam[L - 1]);
      for (int k0 = 0; k0 < kHeadDim; k0 += 32) {
        float v[32];
        tmem_ld32(tl + COL_S + k0, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) store8_split(sb + OFF_SHI, sb + OFF_SLO, 16384, tid, k0 + 8 * q, v + 8 * q);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= gL;
        tmem_st32(tl + COL_S + k0, v);
      }
    }
    operands_ready();

    // ================= X = S0 K^T (hi + lo), O1 = S0_hi Q^T
    if constexpr (!kEmulate) {
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          const uint64_t bk = sw128_desc(sb + OFF_QK + off), bq = sw128_desc(sb + OFF_QK + 8192 + off);
          mma_bf16(tmem + COL_X, sw128_desc(sb + OFF_SHI + off), bk, ID64, ks > 0);
          mma_bf16(tmem + COL_X, sw128_desc(sb + OFF_SLO + off), bk, ID64, 1);
          mma_bf16(tmem + COL_O1, sw128_desc(sb + OFF_SHI + off), bq, ID64, ks > 0);
        }
      }
    } else {
      emu_mma<64, 128>(tl + COL_X, sb + OFF_SHI, 16384, sb + OFF_QK, 16384, false, tid);
      emu_mma<64, 128>(tl + COL_X, sb + OFF_SLO, 16384, sb + OFF_QK, 16384, true, tid);
      emu_mma<64, 128>(tl + COL_O1, sb + OFF_SHI, 16384, sb + OFF_QK + 8192, 16384, false, tid);
    }
    finish_group(bar_x);
    if (!ok) break;

    // ================= R = diag(beta) V - diag(beta Gamma ik) (S0 K^T)^T  -> hi/lo (value-major)
    {
      const uint16_t* sV = reinterpret_cast<const uint16_t*>(sm + OFF_V);
      for (int t0 = 0; t0 < 64; t0 += 32) {
        float x[32];
        tmem_ld32(tl + COL_X + t0, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int t = t0 + i;
          x[i] = s_beta[t] * bf2f(sV[t * kHeadDim + tid]) - s_cx[t] * x[i];
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) store8_split(sb + OFF_RHI, sb + OFF_RLO, 0, tid, t0 + 8 * q, x + 8 * q);
      }
    }
    operands_ready();

    // ================= E^T = R T^T  (hi*hi + hi*lo + lo*hi)
    if constexpr (!kEmulate) {
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t off = ks * 32;
          const uint64_t rh = sw128_desc(sb + OFF_RHI + off), rl = sw128_desc(sb + OFF_RLO + off);
          mma_bf16(tmem + COL_E, rh, sw128_desc(sb + OFF_T + off), ID64, ks > 0);
          mma_bf16(tmem + COL_E, rh, sw128_desc(sb + OFF_T + 8192 + off), ID64, 1);
          mma_bf16(tmem + COL_E, rl, sw128_desc(sb + OFF_T + off), ID64, 1);
        }
      }
    } else {
      emu_mma<64, 64>(tl + COL_E, sb + OFF_RHI, 0, sb + OFF_T, 0, false, tid);
      emu_mma<64, 64>(tl + COL_E, sb + OFF_RHI, 0, sb + OFF_T + 8192, 0, true, tid);
      emu_mma<64, 64>(tl + COL_E, sb + OFF_RLO, 0, sb + OFF_T, 0, true, tid);
    }
    finish_group(bar_e);
    if (!ok) break;

    // ================= E~ = E diag(exp(gamma_L - gamma) ik) -> hi/lo;  E -> bf16 (output operand)
    for (int t0 = 0; t0 < 64; t0 += 32) {
      float ev[32], es[32];
      tmem_ld32(tl + COL_E + t0, ev);
#pragma unroll
      for (int i = 0; i < 32; ++i) es[i] = ev[i] * s_cs[t0 + i];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        store8_split(sb + OFF_RHI, sb + OFF_RLO, 0, tid, t0 + 8 * q, es + 8 * q);
        store8_split(sb + OFF_T, 0, 0, tid, t0 + 8 * q, ev + 8 * q);
      }
    }
    operands_ready();

    // ================= S += E~ K  (N = 128 keys; B = K^T rows),  O2 = E P^T
    if constexpr (!kEmulate) {
      if (tid == 0) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t off = ks * 32;
          const uint64_t bkt = sw128_desc(sb + OFF_KT + off);
          mma_bf16(tmem + COL_S, sw128_desc(sb + OFF_RHI + off), bkt, ID128, 1);
          mma_bf16(tmem + COL_S, sw128_desc(sb + OFF_RLO + off), bkt, ID128, 1);
          mma_bf16(tmem + COL_O2, sw128_desc(sb + OFF_T + off), sw128_desc(sb + OFF_P + off), ID64, ks > 0);
        }
      }
    } else {
      emu_mma<128, 64>(tl + COL_S, sb + OFF_RHI, 0, sb + OFF_KT, 0, true, tid);
      emu_mma<128, 64>(tl + COL_S, sb + OFF_RLO, 0, sb + OFF_KT, 0, true, tid);
      emu_mma<64, 64>(tl + COL_O2, sb + OFF_T, 0, sb + OFF_P, 0, false, tid);
    }
    finish_group(bar_s);
    if (!ok) break;

    // ================= output: o = O1 diag(Gamma iq q_scale) + O2, staged token-major, then
    // (optionally) the sigmoid-gated RMSNorm over the value dimension, coalesced bf16 stores
    for (int t0 = 0; t0 < 64; t0 += 32) {
      float o1[32], o2[32];
      tmem_ld32(tl + COL_O1 + t0, o1);
      tmem_ld32(tl + COL_O2 + t0, o2);
#pragma unroll
      for (int i = 0; i < 32; ++i) s_work[(t0 + i) * LDO + tid] = fmaf(o1[i], s_co[t0 + i], o2[i]);
    }
    __syncthreads();
    {
      float wf[4] = {1.f, 1.f, 1.f, 1.f};
      if (p.z) {
        const uint2 ww = __ldg(reinterpret_cast<const uint2*>(p.norm_w + lane * 4));
        wf[0] = __uint_as_float(ww.x << 16); wf[1] = __uint_as_float(ww.x & 0xFFFF0000u);
        wf[2] = __uint_as_float(ww.y << 16); wf[3] = __uint_as_float(ww.y & 0xFFFF0000u);
      }
      for (int t = warp; t < L; t += kThreads / 32) {
        const float4 v = *reinterpret_cast<const float4*>(s_work + t * LDO + lane * 4);
        float r4[4] = {v.x, v.y, v.z, v.w};
        const size_t base = ((size_t)(c0 + t) * p.Hv + h) * kHeadDim + lane * 4;
        if (p.z) {
          float ss = r4[0] * r4[0] + r4[1] * r4[1] + r4[2] * r4[2] + r4[3] * r4[3];
#pragma unroll
          for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
          const float rstd = rsqrtf(ss * (1.0f / kHeadDim) + p.rms_eps);
          const uint2 zz = __ldg(reinterpret_cast<const uint2*>(p.z + base));
          const float zf[4] = {__uint_as_float(zz.x << 16), __uint_as_float(zz.x & 0xFFFF0000u),
                               __uint_as_float(zz.y << 16), __uint_as_float(zz.y & 0xFFFF0000u)};
#pragma unroll
          for (int i = 0; i < 4; ++i) r4[i] = r4[i] * rstd * wf[i] * sigmoidf_(zf[i]);
        }
        *reinterpret_cast<uint2*>(p.out + base) = make_uint2(pack_bf2(r4[0], r4[1]), pack_bf2(r4[2], r4[3]));
      }
    }
    __syncthreads();
  }

  // ---- final state -> global (thread r: value row r)
  if (ok && p.state_out) {
    const size_t row_off = (((size_t)n * p.Hv + h) * kHeadDim + tid) * kHeadDim;
    for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
      float v[32];
      tmem_ld32(tl + COL_S + c0, v);
      float4* dst = reinterpret_cast<float4*>(p.state_out + row_off + c0);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <bool kEmulate>
cudaError_t launch_impl(const LaunchEnv& env, const ChunkParams& p) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(chunk_prefill_kernel<kEmulate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  const long blocks = (long)p.N * p.Hv;
  chunk_prefill_kernel<kEmulate><<<(unsigned)blocks, kThreads, SMEM_BYTES, env.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_prefill(const LaunchEnv& env, int mode, const uint16_t* qkv, const float* g,
                                 const float* beta, const int32_t* cu, int N, int T, int Hk, int Hv, float q_scale,
                                 float l2_eps, const float* state_in, float* state_out, const uint16_t* z,
                                 const uint16_t* norm_w, float rms_eps, uint16_t* out) {
  if (N <= 0) return cudaSuccess;
  ChunkParams p;
  p.qkv = qkv; p.g = g; p.beta = beta; p.cu = cu; p.state_in = state_in; p.state_out = state_out;
  p.z = z; p.norm_w = norm_w; p.out = out; p.err = env.err;
  p.N = N; p.T = T; p.Hk = Hk; p.Hv = Hv; p.q_scale = q_scale; p.l2_eps = l2_eps; p.rms_eps = rms_eps;
  return mode == 1 ? launch_impl<true>(env, p) : launch_impl<false>(env, p);
}

}  // namespace gdn
