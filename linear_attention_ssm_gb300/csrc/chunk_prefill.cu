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
// Every product is written "value-major": the value index of the state is the 128-row M
// dimension of a tcgen05 MMA (M = 128, N in {64, 128}, K = 16 per instruction, bf16 operands in
// 128-byte-swizzled K-major shared memory, fp32 accumulators in tensor memory).  The fp32 state
// lives in tensor memory for a whole sequence.
//
// Precision: operands that are exact in bf16 (the raw conv outputs q, k, v) are fed as they are;
// the L2-norm factors, beta and the decay exponentials are fp32 diagonal scalings applied in the
// epilogues.  fp32 operands on the state path (S0, the right-hand side R, the solve T, the scaled
// E) are split into bf16 hi + lo pairs (~16-bit operands); the output-only product E P^T uses
// the hi part alone.  S0 K^T and S0 Q^T share one N = 128 MMA chain (the q/k tile stacks the
// 64 key rows over the 64 query rows).
//
// Launch: a persistent grid (one CTA of 256 threads per SM) pulls (sequence, V head) work items
// from a counter in longest-sequence-first order (the order and the counter live in the caller's
// workspace and are written by a one-CTA schedule kernel launched first).  Within an item the
// chunks run in order; q/k and v tiles of the next chunk are fetched by TMA as soon as their
// buffers are free, so HBM latency hides behind the current chunk.  Thread (row, part) owns
// tensor-memory lane `row` and a quarter of the accumulator columns in every epilogue.
#include <cuda.h>

#include "chunk_common.cuh"
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

// ---- shared memory map (byte offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_QK = 0;         // 32 KB: 2 K-blocks x 128 rows (k tokens 0..63, q tokens 64..127)
constexpr uint32_t OFF_KT = 32768;     // 16 KB: K^T, 128 key rows x 64 tokens
constexpr uint32_t OFF_S = 49152;      // 64 KB: S0 hi (32 KB) + lo (32 KB); also the solve work area
                                       //        and the output staging (both dead while S0 is live)
constexpr uint32_t OFF_R = 114688;     // 32 KB: R hi/lo (16 KB each), then E~ hi/lo
constexpr uint32_t OFF_T = 147456;     // 16 KB: T hi (8 KB) + T lo (8 KB); then E bf16 (16 KB)
constexpr uint32_t OFF_P = 163840;     //  8 KB: P, 64 token rows x 64
constexpr uint32_t OFF_V = 172032;     // 16 KB: V, 2 K-blocks of 64 value columns x 64 token rows
constexpr uint32_t OFF_Z = 188416;     // 16 KB: z of the chunk, [64 tokens][128] bf16 (gate input)
constexpr uint32_t OFF_VEC = 204800;   // per-token vectors (8 x 64 floats) + norm partials
constexpr uint32_t OFF_M = OFF_VEC + (8 * 64 + 128 * kParts) * 4;  // 7.5 KB: the solve's six B_ik blocks
constexpr uint32_t OFF_BAR = OFF_M + 6 * 16 * 20 * 4;        // mbarriers, TMEM address, item slot
constexpr uint32_t SMEM_USED = OFF_BAR + 128;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;            // + alignment slack
constexpr uint32_t LDO = 132;  // row stride (floats) of the output staging
static_assert(64 * LDO * 4 <= 65536, "output staging must fit the S0 area");
static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

// ---- tensor memory columns (fp32, lane = value row)
constexpr uint32_t COL_S = 0;     // 128: the recurrent state
constexpr uint32_t COL_X = 128;   //  64: S0 K^T   } one N = 128 accumulator: S0 [K; Q]^T
constexpr uint32_t COL_O1 = 192;  //  64: S0 Q^T   }
constexpr uint32_t COL_E = 256;   //  64: E^T
constexpr uint32_t COL_O2 = 320;  //  64: E^T P^T
constexpr uint32_t COL_G = 384;   //  64: [K; Q] K^T (Gram rows 0..63, Q K^T rows 64..127)
constexpr uint32_t TMEM_COLS = 512;

struct ChunkParams {
  CUtensorMap tmap;    // qkv [T][C] bf16, box 64 x 64, 128-byte swizzle
  CUtensorMap tmap_z;  // z [T][Hv * 128] bf16, box 128 x 64, no swizzle (valid when z != NULL)
  GateSrc gates;
  const int32_t* cu;
  const int32_t* order;     // longest-first sequence order (workspace)
  unsigned* counter;        // work-item counter (workspace, zeroed by the schedule kernel)
  const float* state_in;
  float* state_out;
  const uint16_t* z;
  const uint16_t* norm_w;
  uint16_t* out;
  unsigned* err;
  int N, T, Hk, Hv;
  float q_scale, l2_eps, rms_eps;
};

template <bool kEmulate>
__global__ void __launch_bounds__(kThreads, 1) chunk_prefill_kernel(const __grid_constant__ ChunkParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, part = warp >> 2;
  const int row = q4 * 32 + lane;  // tensor-memory lane = accumulator row owned by this thread

  const int ratio = p.Hv / p.Hk;
  const long total_items = (long)p.N * p.Hv;

  float* s_gam = reinterpret_cast<float*>(sm + OFF_VEC);  // within-chunk cumsum of g, times log2(e)
  float* s_beta = s_gam + 64;
  float* s_ik = s_gam + 128;
  float* s_iq = s_gam + 192;
  float* s_cx = s_gam + 256;  // beta_t Gamma_t ik_t
  float* s_co = s_gam + 320;  // Gamma_t iq_t q_scale
  float* s_cs = s_gam + 384;  // exp(gamma_L - gamma_t) ik_t
  float* s_g = s_gam + 448;
  float* s_part = s_gam + 512;  // kParts x 128 partial sums of squares
  float* s_work = reinterpret_cast<float*>(sm + OFF_S);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 64);
  int* item_slot = reinterpret_cast<int*>(sm + OFF_BAR + 72);
  const uint32_t bar_g = smem_u32(&bars[0]), bar_x = smem_u32(&bars[1]), bar_e = smem_u32(&bars[2]),
                 bar_s = smem_u32(&bars[3]), bar_qk = smem_u32(&bars[4]), bar_v = smem_u32(&bars[5]),
                 bar_z = smem_u32(&bars[6]);

  if (tid == 0) {
    for (int i = 0; i < 7; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);  // this warp's lane quarter, column 0

  constexpr uint32_t ID64 = idesc_bf16_f32(128, 64);
  constexpr uint32_t ID128 = idesc_bf16_f32(128, 128);
  bool ok = true;
  uint32_t ph_mma = 0, ph_qk = 0, ph_v = 0, ph_z = 0;  // phase parities
  bool pend_qk = false, pend_v = false, pend_z = false;  // TMA loads issued, not yet awaited
  const bool gated = p.z != nullptr;
  float wf[4] = {1.f, 1.f, 1.f, 1.f};  // norm weight of this lane's 4 value columns
  if (gated) {
    const uint2 ww = __ldg(reinterpret_cast<const uint2*>(p.norm_w + lane * 4));
    wf[0] = __uint_as_float(ww.x << 16); wf[1] = __uint_as_float(ww.x & 0xFFFF0000u);
    wf[2] = __uint_as_float(ww.y << 16); wf[3] = __uint_as_float(ww.y & 0xFFFF0000u);
  }
  float g_next = 0.f, b_next = 0.f;  // g and beta of the next chunk (threads 0..63)

  auto wait_bar = [&](uint32_t bar, uint32_t& ph) {
    const bool got = mbar_wait(bar, ph, kWaitLimit);
    ph ^= 1u;
    if (!got) raise_error(p.err, kErrTimeout);
    ok = __syncthreads_and(got ? 1 : 0) != 0 && ok;
  };
  auto finish_group = [&](uint32_t bar) {  // MMAs of a group issued (or emulated): wait for them
    if constexpr (!kEmulate) {
      if (tid == 0) mma_commit(bar);
      uint32_t ph = ph_mma;
      wait_bar(bar, ph);
      tc_fence_after();
    } else {
      fence_proxy_async_smem();  // the emulated operand reads precede later TMA writes
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  };
  auto await_group = [&](uint32_t bar) {  // an MMA group committed earlier on `bar` (or emulated)
    if constexpr (!kEmulate) {
      uint32_t ph = ph_mma;
      wait_bar(bar, ph);
      tc_fence_after();
    } else {
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  };
  auto operands_ready = [&]() {  // generic-proxy smem writes by all threads -> visible to MMA / TMA
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  auto issue_qk = [&](int c0, int kh) {  // q and k tiles of the chunk starting at token c0
    mbar_arrive_expect_tx(bar_qk, kBytesQK);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      tma_load_2d(sb + OFF_QK + kb * 16384, &p.tmap, p.Hk * kHeadDim + kh * kHeadDim + kb * 64, c0, bar_qk);
      tma_load_2d(sb + OFF_QK + kb * 16384 + 8192, &p.tmap, kh * kHeadDim + kb * 64, c0, bar_qk);
    }
  };
  auto issue_v = [&](int c0, int h) {
    mbar_arrive_expect_tx(bar_v, kBytesV);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
      tma_load_2d(sb + OFF_V + kb * 8192, &p.tmap, 2 * p.Hk * kHeadDim + h * kHeadDim + kb * 64, c0, bar_v);
  };

  auto issue_z = [&](int c0, int h) {
    mbar_arrive_expect_tx(bar_z, kBytesZ);
    tma_load_2d(sb + OFF_Z, &p.tmap_z, h * kHeadDim, c0, bar_z);
  };
  auto load_gb = [&](int c0, int L, int h) {  // g, beta of a chunk -> registers of threads < 64
    g_next = 0.f;
    b_next = 0.f;
    if (tid < L) load_gate(p.gates, (size_t)(c0 + tid) * p.Hv + h, h, g_next, b_next);
  };

  for (;;) {
    if (tid == 0) *item_slot = (int)atomicAdd(p.counter, 1u);
    __syncthreads();
    const long w = *item_slot;
    __syncthreads();
    if (w >= total_items || !ok) break;
    const int h = (int)(w % p.Hv);
    const int ni = (int)(w / p.Hv);
    const int n = p.order ? __ldg(p.order + ni) : ni;
    const int kh = h / ratio;
    const int seq_s = __ldg(p.cu + n), seq_e = __ldg(p.cu + n + 1);
    if (n < 0 || n >= p.N || seq_s < 0 || seq_e < seq_s || seq_e > p.T) {
      if (tid == 0) raise_error(p.err, kErrDeviceArgument);
      continue;
    }
    if (tid == 0 && seq_e > seq_s) {
      issue_qk(seq_s, kh);
      issue_v(seq_s, h);
      if (gated) issue_z(seq_s, h);
    }
    pend_qk = pend_v = seq_e > seq_s;
    pend_z = gated && seq_e > seq_s;
    if (seq_e > seq_s) load_gb(seq_s, min(kChunk, seq_e - seq_s), h);

    // ---- initial state -> tensor memory (thread (row, part): 128 / kParts columns of row `row`)
    {
      const size_t row_off = (((size_t)n * p.Hv + h) * kHeadDim + row) * kHeadDim;
#pragma unroll
      for (int cq = 0; cq < 4 / kParts; ++cq) {
        const int c0 = part * (128 / kParts) + cq * 32;
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

    for (int c0 = seq_s; c0 < seq_e && ok; c0 += kChunk, ph_mma ^= 1u) {
      const int L = min(kChunk, seq_e - c0);
      const bool has_next = c0 + kChunk < seq_e;

      // ================= prepare: g, beta, norms, K^T, cumsum, per-token factors
      if (tid < 64) {  // fetched one chunk ahead
        s_g[tid] = g_next;
        s_beta[tid] = b_next;
      }
      wait_bar(bar_qk, ph_qk);
      pend_qk = false;
      if (!ok) break;
      {
        // partial sums of squares: rows 0..63 keys, 64..127 queries; each part sums 128 / kParts columns
        const int r = tid & 127, kq = tid >> 7;
        float ss = 0.f;
#pragma unroll
        for (int cc = 0; cc < 16 / kParts; ++cc) {
          const int chunk = kq * (16 / kParts) + cc, kb = chunk >> 3, c = chunk & 7;
          const uint4 u = *reinterpret_cast<const uint4*>(sm + OFF_QK + kb * 16384 + r * 128 + (((c ^ (r & 7)) & 7) << 4));
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = __uint_as_float(w4[e] << 16), b = __uint_as_float(w4[e] & 0xFFFF0000u);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
          }
        }
        s_part[kq * 128 + r] = ss;
        // K^T: thread (key n, token part) gathers 64 / kParts tokens into swizzled 16-byte chunks;
        // within a chunk of 8 tokens the source swizzle term depends on the token's low bits only
        const int nk = tid & 127, th = tid >> 7;
        const uint8_t* kb_base = sm + OFF_QK + (nk >> 6) * 16384 + ((nk & 7) << 1);
        const int nsw = (nk >> 3) & 7;
#pragma unroll
        for (int q = 0; q < 8 / kParts; ++q) {
          const int tc = th * (8 / kParts) + q;
          const uint8_t* src = kb_base + tc * 1024;
          uint32_t w4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t a = *reinterpret_cast<const uint16_t*>(src + (2 * u) * 128 + ((nsw ^ (2 * u)) << 4));
            const uint32_t b = *reinterpret_cast<const uint16_t*>(src + (2 * u + 1) * 128 + ((nsw ^ (2 * u + 1)) << 4));
            w4[u] = a | (b << 16);
          }
          *reinterpret_cast<uint4*>(sm + OFF_KT + nk * 128 + (((tc ^ (nk & 7)) & 7) << 4)) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      if (warp == 0) {
        // inclusive scan of g over the chunk, in log2 units (lane l holds tokens 2l and 2l+1)
        const float g0 = s_g[2 * lane] * kLog2e, g1 = s_g[2 * lane + 1] * kLog2e;
        float s = g0 + g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float v = __shfl_up_sync(0xffffffffu, s, o);
          if (lane >= o) s += v;
        }
        s_gam[2 * lane + 1] = s;
        s_gam[2 * lane] = s - g1;
      }
      __syncthreads();
      if (tid < 128) {
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < kParts; ++q) ss += s_part[q * 128 + tid];
        const float inv = 1.0f / sqrtf(ss + p.l2_eps);
        if (tid < 64) s_ik[tid] = inv; else s_iq[tid - 64] = inv;
      }
      __syncthreads();
      if (tid < 64) {
        const int t = tid;
        const float gam = s_gam[t], gamL = s_gam[L - 1];
        const float Gam = ex2_approx(gam);
        s_cx[t] = s_beta[t] * Gam * s_ik[t];
        s_co[t] = Gam * s_iq[t] * p.q_scale;
        s_cs[t] = (t < L) ? ex2_approx(gamL - gam) * s_ik[t] : 0.f;
      }
      operands_ready();

      // ================= Gram: G = [K; Q] K^T  (M = 128, N = 64, K = 128), issued asynchronously
      if constexpr (!kEmulate) {
        if (tid == 0) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            mma_bf16(tmem + COL_G, sw128_desc(sb + OFF_QK + off), sw128_desc(sb + OFF_QK + off), ID64, ks > 0);
          }
          mma_commit(bar_g);
        }
      } else {
        emu_mma<64, 128>(tl, COL_G, sm + OFF_QK, 16384, sm + OFF_QK, 16384, false, row, part);
      }

      // ================= S0 -> hi/lo operand tiles; tensor memory state <- Gamma_L S0 (under the Gram)
      {
        const float gL = ex2_approx(s_gam[L - 1]);
#pragma unroll
        for (int cq = 0; cq < 4 / kParts; ++cq) {
          const int k0 = part * (128 / kParts) + cq * 32;
          float v[32];
          tmem_ld32(tl + COL_S + k0, v);
#pragma unroll
          for (int q = 0; q < 4; ++q) store8_split(sm + OFF_S, sm + OFF_S + 32768, 16384, row, k0 + 8 * q, v + 8 * q);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= gL;
          tmem_st32(tl + COL_S + k0, v);
        }
      }
      operands_ready();

      // ================= [X | O1] = S0 [K; Q]^T (hi + lo, N = 128), issued asynchronously
      if constexpr (!kEmulate) {
        if (tid == 0) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            const uint64_t bkq = sw128_desc(sb + OFF_QK + off);
            mma_bf16(tmem + COL_X, sw128_desc(sb + OFF_S + off), bkq, ID128, ks > 0);
            mma_bf16(tmem + COL_X, sw128_desc(sb + OFF_S + 32768 + off), bkq, ID128, 1);
          }
          mma_commit(bar_x);
        }
      } else {
        emu_mma<128, 128>(tl, COL_X, sm + OFF_S, 16384, sm + OFF_QK, 16384, false, row, part);
        emu_mma<128, 128>(tl, COL_X, sm + OFF_S + 32768, 16384, sm + OFF_QK, 16384, true, row, part);
      }
      await_group(bar_g);
      if (!ok) break;

      // ================= A (rows 0..63) and P (rows 64..127) from the Gram tile (X/O1 run meanwhile)
      {
        float gr[kW];
        tmem_ld_cols<kW>(tl + COL_G + part * kW, gr);
        float* sA = reinterpret_cast<float*>(sm + OFF_R);  // tidx layout
        if (row < 64) {
          const int t = row;
          const float bt = s_beta[t] * s_ik[t], gt = s_gam[t];
#pragma unroll
          for (int i4 = 0; i4 < kW; i4 += 4) {
            const int j0 = part * kW + i4;
            const float4 gj = *reinterpret_cast<const float4*>(s_gam + j0);
            const float4 kj = *reinterpret_cast<const float4*>(s_ik + j0);
            const float gv[4] = {gj.x, gj.y, gj.z, gj.w}, kv[4] = {kj.x, kj.y, kj.z, kj.w};
            float a[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float val = bt * ex2_approx(gt - gv[u]) * gr[i4 + u] * kv[u];
              a[u] = (j0 + u < t) ? val : 0.f;
            }
            *reinterpret_cast<float4*>(sA + tidx(t, j0)) = make_float4(a[0], a[1], a[2], a[3]);
          }
        } else {
          const int t = row - 64;
          const float qt = s_iq[t] * p.q_scale, gt = s_gam[t];
#pragma unroll
          for (int i0 = 0; i0 < kW; i0 += 8) {
            float v[8];
            const int j0 = part * kW + i0;
            const float4 g0 = *reinterpret_cast<const float4*>(s_gam + j0);
            const float4 g1 = *reinterpret_cast<const float4*>(s_gam + j0 + 4);
            const float4 k0v = *reinterpret_cast<const float4*>(s_ik + j0);
            const float4 k1v = *reinterpret_cast<const float4*>(s_ik + j0 + 4);
            const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const float kv[8] = {k0v.x, k0v.y, k0v.z, k0v.w, k1v.x, k1v.y, k1v.z, k1v.w};
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float a = qt * ex2_approx(gt - gv[u]) * gr[i0 + u] * kv[u];
              v[u] = (j0 + u <= t) ? a : 0.f;
            }
            store8_split(sm + OFF_P, nullptr, 0, t, part * kW + i0, v);
          }
        }
      }
      __syncthreads();

      // ================= solve: T = (I + A)^-1, then T hi/lo -> operand tiles
      {
        const float* sA = reinterpret_cast<const float*>(sm + OFF_R);
        float* sTf = reinterpret_cast<float*>(sm + OFF_R + 16384);
        float* sB = reinterpret_cast<float*>(sm + OFF_M);
        solve_unit_lower(sA, sTf, sB, tid);
        for (int i = tid; i < 64 * 8; i += kThreads) {
          const int t = i >> 3, k0 = (i & 7) * 8;
          // the strictly upper blocks of T are zero (never written by the solve)
          const bool upper = (k0 >> 4) > (t >> 4);
          const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 v0 = upper ? z4 : *reinterpret_cast<const float4*>(sTf + tidx(t, k0));
          const float4 v1 = upper ? z4 : *reinterpret_cast<const float4*>(sTf + tidx(t, k0 + 4));
          const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          store8_split(sm + OFF_T, sm + OFF_T + 8192, 0, t, k0, v);
        }
      }
      await_group(bar_x);  // also orders the solve's reads of the R area before R is written
      if (!ok) break;
      // the q/k tile is free: fetch the next chunk's
      if (tid == 0 && has_next) issue_qk(c0 + kChunk, kh);
      pend_qk = has_next;
      if (has_next) load_gb(c0 + kChunk, min(kChunk, seq_e - c0 - kChunk), h);

      // ================= R = diag(beta) V - diag(beta Gamma ik) (S0 K^T)^T  -> hi/lo (value-major)
      wait_bar(bar_v, ph_v);
      pend_v = false;
      if (!ok) break;
      {
        float x[kW];
        tmem_ld_cols<kW>(tl + COL_X + part * kW, x);
        // V[t][row] for t = part * kW + i: the swizzle term depends on i & 7 only
        const uint8_t* vb = sm + OFF_V + (row >> 6) * 8192 + part * kW * 128 + ((row & 7) << 1);
        const int rsw = (row >> 3) & 7;
#pragma unroll
        for (int i4 = 0; i4 < kW; i4 += 4) {
          const float4 bt = *reinterpret_cast<const float4*>(s_beta + part * kW + i4);
          const float4 cx = *reinterpret_cast<const float4*>(s_cx + part * kW + i4);
          const float btv[4] = {bt.x, bt.y, bt.z, bt.w}, cxv[4] = {cx.x, cx.y, cx.z, cx.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i4 + u;
            const float v = bf2f(*reinterpret_cast<const uint16_t*>(vb + i * 128 + ((rsw ^ (i & 7)) << 4)));
            x[i] = btv[u] * v - cxv[u] * x[i];
          }
        }
#pragma unroll
        for (int q = 0; q < kW / 8; ++q) store8_split(sm + OFF_R, sm + OFF_R + 16384, 0, row, part * kW + 8 * q, x + 8 * q);
      }
      operands_ready();
      if (tid == 0 && has_next) issue_v(c0 + kChunk, h);
      pend_v = has_next;

      // ================= E^T = R T^T  (hi*hi + hi*lo + lo*hi)
      if constexpr (!kEmulate) {
        if (tid == 0) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t off = ks * 32;
            const uint64_t rh = sw128_desc(sb + OFF_R + off), rl = sw128_desc(sb + OFF_R + 16384 + off);
            mma_bf16(tmem + COL_E, rh, sw128_desc(sb + OFF_T + off), ID64, ks > 0);
            mma_bf16(tmem + COL_E, rh, sw128_desc(sb + OFF_T + 8192 + off), ID64, 1);
            mma_bf16(tmem + COL_E, rl, sw128_desc(sb + OFF_T + off), ID64, 1);
          }
        }
      } else {
        emu_mma<64, 64>(tl, COL_E, sm + OFF_R, 0, sm + OFF_T, 0, false, row, part);
        emu_mma<64, 64>(tl, COL_E, sm + OFF_R, 0, sm + OFF_T + 8192, 0, true, row, part);
        emu_mma<64, 64>(tl, COL_E, sm + OFF_R + 16384, 0, sm + OFF_T, 0, true, row, part);
      }
      finish_group(bar_e);
      if (!ok) break;

      // ================= E~ = E diag(exp(gamma_L - gamma) ik) -> hi/lo;  E -> bf16 (output operand)
      {
        float ev[kW], es[kW];
        tmem_ld_cols<kW>(tl + COL_E + part * kW, ev);
#pragma unroll
        for (int i4 = 0; i4 < kW; i4 += 4) {
          const float4 cs = *reinterpret_cast<const float4*>(s_cs + part * kW + i4);
          es[i4] = ev[i4] * cs.x;
          es[i4 + 1] = ev[i4 + 1] * cs.y;
          es[i4 + 2] = ev[i4 + 2] * cs.z;
          es[i4 + 3] = ev[i4 + 3] * cs.w;
        }
#pragma unroll
        for (int q = 0; q < kW / 8; ++q) {
          store8_split(sm + OFF_R, sm + OFF_R + 16384, 0, row, part * kW + 8 * q, es + 8 * q);
          store8_split(sm + OFF_T, nullptr, 0, row, part * kW + 8 * q, ev + 8 * q);
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
            mma_bf16(tmem + COL_S, sw128_desc(sb + OFF_R + off), bkt, ID128, 1);
            mma_bf16(tmem + COL_S, sw128_desc(sb + OFF_R + 16384 + off), bkt, ID128, 1);
            mma_bf16(tmem + COL_O2, sw128_desc(sb + OFF_T + off), sw128_desc(sb + OFF_P + off), ID64, ks > 0);
          }
        }
      } else {
        emu_mma<128, 64>(tl, COL_S, sm + OFF_R, 0, sm + OFF_KT, 0, true, row, part);
        emu_mma<128, 64>(tl, COL_S, sm + OFF_R + 16384, 0, sm + OFF_KT, 0, true, row, part);
        emu_mma<64, 64>(tl, COL_O2, sm + OFF_T, 0, sm + OFF_P, 0, false, row, part);
      }
      finish_group(bar_s);
      if (!ok) break;

      // ================= output: o = O1 diag(Gamma iq q_scale) + O2, staged token-major in the
      // (now dead) S0 area, then the sigmoid-gated RMSNorm over the value dimension
      {
        float o1[kW], o2[kW];
        tmem_ld_cols<kW>(tl + COL_O1 + part * kW, o1);
        tmem_ld_cols<kW>(tl + COL_O2 + part * kW, o2);
#pragma unroll
        for (int i4 = 0; i4 < kW; i4 += 4) {
          const int t0 = part * kW + i4;
          const float4 co = *reinterpret_cast<const float4*>(s_co + t0);
          s_work[t0 * LDO + row] = fmaf(o1[i4], co.x, o2[i4]);
          s_work[(t0 + 1) * LDO + row] = fmaf(o1[i4 + 1], co.y, o2[i4 + 1]);
          s_work[(t0 + 2) * LDO + row] = fmaf(o1[i4 + 2], co.z, o2[i4 + 2]);
          s_work[(t0 + 3) * LDO + row] = fmaf(o1[i4 + 3], co.w, o2[i4 + 3]);
        }
      }
      if (gated) {
        wait_bar(bar_z, ph_z);
        pend_z = false;
        if (!ok) break;
      } else {
        __syncthreads();
      }
      {
        // warp w: tokens w, w + kWarps, ..., all in flight together
        constexpr int kTok = kChunk / kWarps;
        float r[kTok][4], ss[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i) {
          const float4 v = *reinterpret_cast<const float4*>(s_work + (warp + kWarps * i) * LDO + lane * 4);
          r[i][0] = v.x; r[i][1] = v.y; r[i][2] = v.z; r[i][3] = v.w;
          ss[i] = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        if (gated) {
#pragma unroll
          for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
            for (int i = 0; i < kTok; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], m);
#pragma unroll
          for (int i = 0; i < kTok; ++i) {
            const float rstd = rsqrtf(ss[i] * (1.0f / kHeadDim) + p.rms_eps);
            const uint2 zz = *reinterpret_cast<const uint2*>(sm + OFF_Z + (warp + kWarps * i) * 256 + lane * 8);
            const float zf[4] = {__uint_as_float(zz.x << 16), __uint_as_float(zz.x & 0xFFFF0000u),
                                 __uint_as_float(zz.y << 16), __uint_as_float(zz.y & 0xFFFF0000u)};
#pragma unroll
            for (int e = 0; e < 4; ++e) r[i][e] = r[i][e] * rstd * wf[e] * sigmoid_fast(zf[e]);
          }
        }
#pragma unroll
        for (int i = 0; i < kTok; ++i) {
          const int t = warp + kWarps * i;
          if (t < L) {
            const size_t base = ((size_t)(c0 + t) * p.Hv + h) * kHeadDim + lane * 4;
            *reinterpret_cast<uint2*>(p.out + base) =
                make_uint2(pack_bf2(r[i][0], r[i][1]), pack_bf2(r[i][2], r[i][3]));
          }
        }
      }
      fence_proxy_async_smem();  // z reads above precede the next z tile's TMA write
      __syncthreads();
      if (gated && has_next) {
        if (tid == 0) issue_z(c0 + kChunk, h);
        pend_z = true;
      }
    }
    if (!ok) break;

    // ---- final state -> global
    if (p.state_out) {
      const size_t row_off = (((size_t)n * p.Hv + h) * kHeadDim + row) * kHeadDim;
#pragma unroll
      for (int cq = 0; cq < 4 / kParts; ++cq) {
        const int c0 = part * (128 / kParts) + cq * 32;
        float v[32];
        tmem_ld32(tl + COL_S + c0, v);
        float4* dst = reinterpret_cast<float4*>(p.state_out + row_off + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  // after an early exit, let loads still in flight land before the CTA leaves (bounded)
  if (pend_qk) mbar_wait(bar_qk, ph_qk, kWaitLimit);
  if (pend_v) mbar_wait(bar_v, ph_v, kWaitLimit);
  if (pend_z) mbar_wait(bar_z, ph_z, kWaitLimit);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// One CTA: longest-first order of the sequences (ties by index), a zeroed work counter and,
// when `chunk_off` is given, the exclusive prefix sum over sequences of their 64-token chunk
// counts (chunk_off[N] = total chunks).  Sequences with inconsistent cu_seqlens count as empty
// here; the main kernels report them.
__global__ void __launch_bounds__(1024) chunk_schedule_kernel(const int32_t* cu, int N, int32_t* order,
                                                              unsigned* counter, int32_t* chunk_off) {
  extern __shared__ int32_t s_len[];
  __shared__ int32_t s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) *counter = 0u;
  if (chunk_off) {
    // per-thread contiguous range, then a block-wide exclusive scan of the range totals
    const int per = (N + 1023) / 1024, lo = min(N, tid * per), hi = min(N, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += (max(0, __ldg(cu + i + 1) - __ldg(cu + i)) + kChunk - 1) / kChunk;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += v;
      }
      s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int run = incl - local + (warp > 0 ? s_warp[warp - 1] : 0);
    for (int i = lo; i < hi; ++i) {
      chunk_off[i] = run;
      run += (max(0, __ldg(cu + i + 1) - __ldg(cu + i)) + kChunk - 1) / kChunk;
    }
    if (tid == 1023) chunk_off[N] = s_warp[31];
  }
  const bool sorted = N <= kScheduleSortMax;
  for (int i = tid; i < N; i += blockDim.x) {
    if (sorted) s_len[i] = max(0, __ldg(cu + i + 1) - __ldg(cu + i));
    else order[i] = i;
  }
  if (!sorted) return;
  __syncthreads();
  for (int i = tid; i < N; i += blockDim.x) {
    const int li = s_len[i];
    int rank = 0;
    for (int j = 0; j < N; ++j) {
      const int lj = s_len[j];
      rank += (lj > li) || (lj == li && j < i);
    }
    order[rank] = i;
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
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
  int sms = 0;
  cudaError_t e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const long items = (long)p.N * p.Hv;
  const int grid = (int)(items < sms ? items : sms);
  chunk_prefill_kernel<kEmulate><<<grid, kThreads, SMEM_BYTES, env.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t device_sm_count(int* sms) {
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && sm_count[dev] > 0) {
    *sms = sm_count[dev];
    return cudaSuccess;
  }
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && dev < 64) sm_count[dev] = *sms;
  return e;
}

cudaError_t encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                          uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_chunk_tensor_maps(CUtensorMap* qkv_map, CUtensorMap* z_map, const uint16_t* qkv,
                                     const uint16_t* z, int T, int Hk, int Hv) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const int C = 2 * Hk * kHeadDim + Hv * kHeadDim;
  const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(qkv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(qkv), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  if (z && z_map) {
    const cuuint64_t zdims[2] = {(cuuint64_t)Hv * kHeadDim, (cuuint64_t)T};
    const cuuint64_t zstrides[1] = {(cuuint64_t)Hv * kHeadDim * 2};
    const cuuint32_t zbox[2] = {128, 64};
    const CUresult rz = enc(z_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(z), zdims, zstrides, zbox,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (rz != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t launch_chunk_schedule(cudaStream_t stream, const int32_t* cu, int N, int32_t* order, unsigned* counter,
                                  int32_t* chunk_off) {
  const size_t sched_smem = N <= kScheduleSortMax ? (size_t)N * sizeof(int32_t) : 0;
  chunk_schedule_kernel<<<1, 1024, sched_smem, stream>>>(cu, N, order, counter, chunk_off);
  return cudaGetLastError();
}

size_t chunk_prefill_workspace_bytes(int N) {
  return 256 + (((size_t)(N > 0 ? N : 0) * sizeof(int32_t) + 255) / 256) * 256;
}

cudaError_t launch_chunk_prefill(const LaunchEnv& env, int mode, const uint16_t* qkv, const GateSrc& gates,
                                 const int32_t* cu, int N, int T, int Hk, int Hv, float q_scale,
                                 float l2_eps, const float* state_in, float* state_out, const uint16_t* z,
                                 const uint16_t* norm_w, float rms_eps, uint16_t* out, void* workspace,
                                 size_t workspace_bytes) {
  if (N <= 0) return cudaSuccess;
  if (mode == 0 && workspace_bytes >= split_workspace_bytes(N, T, Hk, Hv))
    return launch_chunk_prefill_split(env, qkv, gates, cu, N, T, Hk, Hv, q_scale, l2_eps, state_in, state_out, z,
                                      norm_w, rms_eps, out, workspace);
  ChunkParams p;
  memset(&p, 0, sizeof p);
  if (T > 0) {
    cudaError_t e = encode_chunk_tensor_maps(&p.tmap, &p.tmap_z, qkv, z, T, Hk, Hv);
    if (e != cudaSuccess) return e;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counter = reinterpret_cast<unsigned*>(ws);
  p.order = reinterpret_cast<const int32_t*>(ws + 256);
  p.gates = gates; p.cu = cu; p.state_in = state_in; p.state_out = state_out;
  p.z = z; p.norm_w = norm_w; p.out = out; p.err = env.err;
  p.N = N; p.T = T; p.Hk = Hk; p.Hv = Hv; p.q_scale = q_scale; p.l2_eps = l2_eps; p.rms_eps = rms_eps;
  cudaError_t e = launch_chunk_schedule(env.stream, cu, N, reinterpret_cast<int32_t*>(ws + 256), p.counter, nullptr);
  if (e != cudaSuccess) return e;
  return mode == 1 ? launch_impl<true>(env, p) : launch_impl<false>(env, p);
}

}  // namespace gdn
