// kda_chunk.cu -- the KDA recurrence over packed sequences in its chunk-wise form (64-token chunks):
// the state-independent quantities of every (chunk, V head) first, then the chain of chunks of
// each (sequence, V head) on the tensor cores with the fp32 state in tensor memory.
//
// GLM-5.3-Flash kernel TDD ledger, slices I2 (an fp32 state indexed [value, key], a per-channel
// decay clamped then exponentiated, its own q output scale), I2a (q and k normalised as
// x / sqrt(sum x^2 + eps)) and I4 (the chunk path matches the sequential state and output at
// 63 / 64 / 65 tokens).  Per chunk (tokens t = 0 .. L - 1 from the state S0, gamma_t the running
// sum of the clamped log decays per key channel c):
//   X  = S0 (k^_t o e^gamma_t)^T                      (value x token)
//   A_ts = beta_t sum_c k^_t k^_s e^(gamma_t - gamma_s)    (s < t),  T = (I + A)^-1
//   R  = (V - X) diag(beta),  E = R T^T
//   o_t = q_scale (S0 (q^_t o e^gamma_t) + sum_(s <= t) P_ts E_s),
//         P_ts = sum_c q^_t k^_s e^(gamma_t - gamma_s)
//   S  = S0 diag(e^gamma_L) + E (k^ o e^(gamma_L - gamma))
// -- the sequential recurrence S <- S diag(a_t); e = beta (v - S k^); S <- S + e k^T; o = q_scale S q^
// written for a chunk at once.  A and P: where every |gamma_t - gamma_31| of the chunk stays within
// 60 nats, one tensor-core product around the chunk's middle token,
// (x_t e^(gamma_t - gamma_31)) (k^_s e^(gamma_31 - gamma_s)), its entries above the diagonal
// dropped by position; otherwise (any decay, g <= 0 after the clamp) the off-diagonal 16 x 16
// blocks as products around the last token r of the column block, where both factors are at most
// 1, and the diagonal blocks from running products of the per-token factors, so nothing overflows
// however strong the decay.  Precision as in the GDN chunk path: every state-path operand (K~, Kd,
// S0, T, R, E, and the A / P operands) is a bf16 hi + lo pair, the output-only products (Q~ against
// S0, P E) plain bf16.
#include <string.h>

#include <algorithm>

#include "chunk_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

// ---- one record per (chunk, V head), written by the prep kernel and read by the state kernel
constexpr uint32_t KR_KQ = 0;        // [K~ hi; Q~]: two 64-key blocks of 128 rows (tokens 0..63 of K~ hi,
                                     // then of Q~), 16 KB apart, 128-byte swizzle
constexpr uint32_t KR_KLO = 32768;   // K~ lo: two 64-key blocks of 64 rows, 8 KB apart
constexpr uint32_t KR_T = 49152;     // T hi, T lo (8 KB each)
constexpr uint32_t KR_KD = 65536;    // Kd hi, then Kd lo 16 KB later: two 64-key blocks of 64 token rows each
constexpr uint32_t KR_P = 98304;     // P (8 KB)
constexpr uint32_t KR_VEC = 106496;  // beta, -beta, c_s (1), c_o (q_scale): 64 floats each; e^gamma_L: 128
constexpr uint32_t kKRecVec = 384 * 4;
constexpr uint32_t KR_BYTES = KR_VEC + kKRecVec;  // 108,032
constexpr uint32_t kKRecKQ = KR_T - KR_KQ;        // K~ hi, Q~ and K~ lo: one bulk copy
constexpr uint32_t kKRecTKD = KR_P - KR_T;        // T and Kd: one bulk copy
constexpr uint32_t kKRecP = KR_VEC - KR_P;
constexpr int KV_BETA = 0, KV_NCX = 64, KV_CS = 128, KV_CO = 192, KV_GL = 256;
static_assert(KR_BYTES % 256 == 0, "records stay 256-byte aligned");

// ---- prep kernel shared memory (one CTA per SM).  The gamma span of a chunk decides how its A and
// P are formed (on the tensor cores around one reference token, or block by block on the CUDA
// cores); the buffers of the two ways share one region.
constexpr uint32_t KP_Q = 0;          // q^ [64][128] fp32
constexpr uint32_t KP_K = 32768;      // k^ [64][128]
constexpr uint32_t KP_G = 65536;      // gamma [64][128], in log2 units (first the clamped log decays)
constexpr uint32_t KP_U = 98304;      // the shared region (96 KB):
constexpr uint32_t KP_AH = KP_U;          //   tensor cores: [K'; Q'] hi, two 64-channel blocks of 128 rows
constexpr uint32_t KP_AL = KP_U + 32768;  //   [K'; Q'] lo
constexpr uint32_t KP_B = KP_U + 65536;   //   [K'' hi; K'' lo], two 64-channel blocks of 128 rows
constexpr uint32_t KP_A = KP_U;           //   CUDA cores: the per-token factors 2^g [64][128] (formed
                                          //   from the raw log decays the inputs left at KP_U + 32 KB)
constexpr uint32_t KP_P = KP_U + 32768;   //   P [64][64] fp32
constexpr uint32_t KP_KB = KP_U + 49152;  //   column block k^ e^(gamma_r - gamma) [16][128]
constexpr uint32_t KP_RK = KP_U + 57344;  //   row block k^ e^(gamma - gamma_r) [16][128]
constexpr uint32_t KP_RQ = KP_U + 65536;  //   row block q^ e^(gamma - gamma_r) [16][128]
constexpr uint32_t KP_TRI = KP_U + 98304;      // A, T and the solve's scratch (kHeadBuf)
constexpr uint32_t KP_BETA = KP_TRI + kHeadBuf;  // [2][64] (by unit parity)
constexpr uint32_t KP_BAR = KP_BETA + 512;       // the MMA and input barriers, the tensor-memory address, flags
constexpr uint32_t KP_BYTES = KP_BAR + 64 + 1024;
static_assert(KP_TRI % 1024 == 0 && KP_U % 1024 == 0, "swizzled tiles and the solve's buffers stay 1 KB aligned");
static_assert(KP_RQ + 8192 <= KP_TRI && KP_B + 32768 <= KP_TRI, "the shared region holds either set");
// Reference token of the tensor-core way, and the largest |gamma_t - gamma_ref| (log2 units) over
// the chunk's tokens and channels for which it is taken: factors stay within 2^(+-86) (e^(+-60)),
// far from fp32 overflow and from denormal operands.
constexpr int kRefToken = 31;
constexpr int kPrepThreads = 512;  // sixteen warps: the prep kernel's phases are latency-bound
constexpr float kRefSpan2 = 86.f;
constexpr float kLog2e = 1.4426950408889634f;

// ---- state kernel shared memory (two CTAs per SM).  The first 48 KB hold the chunk's [K~; Q~] and
// K~ lo until the X products have read them, then its T (hi / lo; E over T hi) and Kd (hi / lo).
constexpr uint32_t SK_QK = 0;         // [K~ hi; Q~] (record copy), then T hi / lo
constexpr uint32_t SK_KLO = 32768;    // K~ lo (same copy)
constexpr uint32_t SK_T = 0;          // T hi / lo (the second copy), then E bf16 over T hi
constexpr uint32_t SK_KD = 16384;     // Kd hi / lo (same copy), lo 16 KB after hi
constexpr uint32_t SK_W = 49152;      // 32 KB: S0 key-half hi/lo, then the output staging
constexpr uint32_t SK_V = 81920;      // V (TMA), then z
constexpr uint32_t SK_P = 98304;      // P (record copy)
constexpr uint32_t SK_VEC = 106496;   // 2 x vector block
constexpr uint32_t SK_BAR = SK_VEC + 2 * kKRecVec;
constexpr uint32_t SK_BYTES = SK_BAR + 128 + 1024;
constexpr uint32_t KSC_S = 0, KSC_X = 128, KSC_O1 = 192, KSC_COLS = 256;  // tensor-memory columns
static_assert(2 * (SK_BYTES + 1024) <= 233472, "two state CTAs must share an SM");
static_assert(KP_BYTES <= 232448, "one CTA's shared memory");
static_assert(SK_KLO - SK_QK == KR_KLO - KR_KQ && SK_KD - SK_T == KR_KD - KR_T, "record parts keep their offsets");

__device__ __forceinline__ uint8_t* align1024k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}

// element (t, s) of a 64 x 64 matrix in the solve's layout: its ten 16 x 16 blocks on and below the
// diagonal (block row i, column j at index i (i + 1) / 2 + j), rows of a block with their 16-byte
// groups XOR-permuted by (row & 3)
__device__ __forceinline__ int tri_index(int t, int s) {
  const int tb = t >> 4, sb = s >> 4, r = t & 15, c = s & 15;
  return ((tb * (tb + 1)) / 2 + sb) * 256 + r * 16 + ((((c >> 2) ^ (r & 3)) << 2) | (c & 3));
}

// two bf16 in one 32-bit word (the first in the low half) -> two floats
__device__ __forceinline__ float2 bf2x2_f(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

struct KPrepParams {
  CUtensorMap tmap_qkv;  // qkv [T][C] bf16, box 64 x 64, 128-byte swizzle (the q and k tiles)
  CUtensorMap tmap_g;    // g [T][Hv * 128] fp32, box 128 x 64, no swizzle
  const float* beta;
  const int32_t* cu;
  const int32_t* chunk_off;
  uint8_t* rec;
  unsigned* err;
  int N, T, Hk, Hv, nc_max;
  float g_min, q_scale, l2_eps;
};

// The chunk and V head of unit u, its sequence n, and the chunk's first token and length; false
// (uniformly) for a sequence whose cu_seqlens entries are outside [0, T] or decreasing.  The
// caller passes chunk_off and cu at a guessed sequence (the previous unit's), loaded ahead; the
// search over chunk_off runs only when the guess is wrong.
struct UnitGuess {
  int n, off0, off1, cu0, cu1;
};
__device__ __forceinline__ UnitGuess load_guess(const KPrepParams& p, int n) {
  return {n, __ldg(p.chunk_off + n), __ldg(p.chunk_off + n + 1), __ldg(p.cu + n), __ldg(p.cu + n + 1)};
}
__device__ __forceinline__ bool kda_unit(const KPrepParams& p, long u, const UnitGuess& gs, int& n, int& gc, int& h,
                                         int& c0, int& L) {
  gc = (int)(u / p.Hv);
  h = (int)(u - (long)gc * p.Hv);
  int s0, s1, off;
  if (gs.off0 <= gc && gc < gs.off1) {
    n = gs.n; s0 = gs.cu0; s1 = gs.cu1; off = gs.off0;
  } else {  // the last n with chunk_off[n] <= gc (a non-empty one)
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.chunk_off + mid) <= gc) lo = mid; else hi = mid - 1;
    }
    n = lo; s0 = __ldg(p.cu + lo); s1 = __ldg(p.cu + lo + 1); off = __ldg(p.chunk_off + lo);
  }
  c0 = s0 + (gc - off) * kChunk;
  L = min(kChunk, s1 - c0);
  return !(s0 < 0 || s1 < s0 || s1 > p.T || L <= 0);
}

// Named barrier kId over the kCount threads of one warp group (only those threads call it): a plain
// barrier, or one that returns the AND / OR of `v` over the group.
template <int kId, int kCount>
__device__ __forceinline__ void grp_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kId), "n"(kCount) : "memory");
}
template <int kId, int kCount>
__device__ __forceinline__ bool grp_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.and.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)(v ? 1 : 0)), "n"(kId), "n"(kCount)
      : "memory");
  return r != 0;
}
template <int kId, int kCount>
__device__ __forceinline__ bool grp_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.or.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)(v ? 1 : 0)), "n"(kId), "n"(kCount)
      : "memory");
  return r != 0;
}

// 4 fp32 values (columns k0..k0+3 of `row`, k0 % 4 == 0) -> bf16 hi (and lo) in K-major 128-byte
// swizzled tiles whose 64-column blocks are hi_kbs / lo_kbs bytes apart
__device__ __forceinline__ void store4_split(uint8_t* hi_tile, uint32_t hi_kbs, uint8_t* lo_tile, uint32_t lo_kbs,
                                             int row, int k0, float4 v) {
  const uint32_t h0 = pack_bf2(v.x, v.y), h1 = pack_bf2(v.z, v.w);
  *reinterpret_cast<uint2*>(hi_tile + sw128_offset(row, k0, hi_kbs)) = make_uint2(h0, h1);
  if (lo_tile) {
    const float2 a = bf2x2_f(h0), b = bf2x2_f(h1);
    *reinterpret_cast<uint2*>(lo_tile + sw128_offset(row, k0, lo_kbs)) =
        make_uint2(pack_bf2(v.x - a.x, v.y - a.y), pack_bf2(v.z - b.x, v.w - b.y));
  }
}

__device__ __forceinline__ float4 f4mul(float4 a, float4 b) { return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w); }
__device__ __forceinline__ float4 f4exp2_diff(float4 a, float4 b) {  // 2^(a - b) per element
  return make_float4(exp2f(a.x - b.x), exp2f(a.y - b.y), exp2f(a.z - b.z), exp2f(a.w - b.w));
}

// Persistent over the (chunk, V head) units of the call, sixteen warps per CTA (one CTA per SM):
// every phase is latency-bound, so the warps' number, not their registers, sets its speed.
// Channel c of a 128-wide row is read in float4 groups; where a warp's lanes split the channels,
// lane group g takes the groups g, g + G, ... so that the lanes of one load cover consecutive
// 16-byte words (no bank conflicts).
//
// Per unit: the front phase (the unit's raw q, k and g arrive by TMA in a shared region; q and k
// normalised, gamma = the running sum of the clamped log decays per channel, in log2 units, and its
// span around token 31) has run on warps 2..15 during the previous unit; then A and P (all warps);
// then warps 0 and 1 solve for T and write it to the record while warps 2..15 write the rest of the
// record and run the next unit's front phase; the two groups meet at one CTA barrier per unit.
//
// A and P: when every |gamma_t - gamma_31| of the chunk is small enough (always, for decays of a
// few nats per token), the whole 64 x 64 products at once on the tensor cores around the middle
// token 31 -- [K'; Q'] = [k^; q^] o 2^(gamma - gamma_31) against K'' = k^ o 2^(gamma_31 - gamma),
// each a bf16 hi / lo pair: hi x [K'' hi; K'' lo] (N = 128) and lo x K'' hi (N = 64), K = 128, into
// tensor memory, the two column halves summed when read; entries above the diagonal (whose
// factors may overflow) are discarded by position.  Otherwise the diagonal 16 x 16 blocks by
// running products of the per-token factors and the blocks below them around the last token of
// their column block, on the CUDA cores, where every factor is at most 1.
__global__ void __launch_bounds__(kPrepThreads, 1) kda_prep_kernel(const __grid_constant__ KPrepParams p) {
  constexpr int NT = kPrepThreads;
  constexpr int FT = NT - 64;  // the front group: warps 2..15
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024k(smem_raw);
  const uint32_t sb = smem_u32(sm);
  float* sQ = reinterpret_cast<float*>(sm + KP_Q);
  float* sK = reinterpret_cast<float*>(sm + KP_K);
  float* sG = reinterpret_cast<float*>(sm + KP_G);
  float* sAf = reinterpret_cast<float*>(sm + KP_A);
  float* sP = reinterpret_cast<float*>(sm + KP_P);
  float* sTri = reinterpret_cast<float*>(sm + KP_TRI);
  float* sKb = reinterpret_cast<float*>(sm + KP_KB);
  float* sRK = reinterpret_cast<float*>(sm + KP_RK);
  float* sRQ = reinterpret_cast<float*>(sm + KP_RQ);
  float* sBeta = reinterpret_cast<float*>(sm + KP_BETA);  // two buffers of 64 (by unit parity)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + KP_BAR + 16);
  // [0] the way the front phase chose (1: tensor cores); [1] the next unit's rows requested, [2] landed
  int* s_flags = reinterpret_cast<int*>(sm + KP_BAR + 24);
  const uint32_t bar_mma = sb + KP_BAR, bar_in = sb + KP_BAR + 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q4 = warp & 3, cpart = warp >> 2;  // tensor-memory lane quarter, 16-column part
  const int ft = tid - 64;                     // index in the front group (negative on warps 0, 1)
  const int ratio = p.Hv / p.Hk;
  // chunk_off[N] exceeds the record capacity only for cu_seqlens outside [0, T]; those sequences
  // are rejected below, and no record past the capacity is written
  const long units = (long)min(__ldg(p.chunk_off + p.N), p.nc_max) * p.Hv;
  const float g_min2 = p.g_min * kLog2e;  // -inf stays -inf

  if (tid == 0) {
    mbar_init(bar_mma, 1);
    mbar_init(bar_in, 1);
    fence_mbar_init();
    prefetch_tensormap(&p.tmap_qkv);
    prefetch_tensormap(&p.tmap_g);
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint32_t ph_mma = 0, ph_in = 0;
  bool ok = true, in_flight = false, mma_flight = false;
  float bt = 0.f;  // beta of the unit whose rows were requested last (front thread ft < 64: token ft)
  constexpr uint32_t ID64 = idesc_bf16_f32(128, 64), ID128 = idesc_bf16_f32(128, 128);

  // the raw rows of a unit -> the shared region by TMA (one thread): q as two 64 x 64 boxes
  // (128-byte swizzle, 8 KB apart) at 0, k likewise at 16 KB, g [64][128] fp32 at 32 KB (rows past
  // T zero, rows past L ignored); the region must be free and its generic accesses fenced.  The
  // front group's first 64 threads load the unit's beta.
  auto issue_unit = [&](int c0, int L, int h, int kh) {
    if (tid == 64) {
      mbar_arrive_expect_tx(bar_in, 65536u);
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_2d(sb + KP_U + kb * 8192, &p.tmap_qkv, kh * kHeadDim + kb * 64, c0, bar_in);
        tma_load_2d(sb + KP_U + 16384 + kb * 8192, &p.tmap_qkv, (p.Hk + kh) * kHeadDim + kb * 64, c0, bar_in);
      }
      tma_load_2d(sb + KP_U + 32768, &p.tmap_g, h * kHeadDim, c0, bar_in);
    }
    if (ft >= 0 && ft < 64) bt = ft < L ? __ldg(p.beta + (size_t)(c0 + ft) * p.Hv + h) : 0.f;
  };

  // The front phase of a unit on the front group (barrier 2): wait for its rows, q and k normalised
  // (16 lanes per token row, 8 channels each), the clamped log decays in log2 units, beta into
  // buffer `bb`, the running sums gamma (a half of the chunk per thread of the first 256, the second
  // half then shifted by the first half's total) and the way A and P take (s_flags[0]).  Returns
  // false, uniformly over the group, when the rows did not arrive in time.
  auto front = [&](int L, int bb) -> bool {
    bool got = mbar_wait(bar_in, ph_in, kWaitLimit);
    got = grp_and<2, FT>(got);
    if (!got) {
      if (ft == 0) raise_error(p.err, kErrTimeout);
      return false;
    }
    for (int i = ft; i < 64 * 16; i += FT) {  // warp-uniform trip count (FT and 1024 are multiples of 32)
      const int t = i >> 4, c8 = (i & 15) * 8;
      uint4 uq = make_uint4(0u, 0u, 0u, 0u), uk = uq;
      if (t < L) {  // 16-byte group c8 / 8 of row t in the swizzled boxes
        const uint32_t off = (c8 >> 6) * 8192 + t * 128 + (((((c8 & 63) >> 3) ^ (t & 7))) << 4);
        uq = *reinterpret_cast<const uint4*>(sm + KP_U + off);
        uk = *reinterpret_cast<const uint4*>(sm + KP_U + 16384 + off);
      }
      const float2 a0 = bf2x2_f(uq.x), a1 = bf2x2_f(uq.y), a2 = bf2x2_f(uq.z), a3 = bf2x2_f(uq.w);
      const float2 b0 = bf2x2_f(uk.x), b1 = bf2x2_f(uk.y), b2 = bf2x2_f(uk.z), b3 = bf2x2_f(uk.w);
      float sq = a0.x * a0.x + a0.y * a0.y + a1.x * a1.x + a1.y * a1.y + a2.x * a2.x + a2.y * a2.y + a3.x * a3.x +
                 a3.y * a3.y;
      float sk = b0.x * b0.x + b0.y * b0.y + b1.x * b1.x + b1.y * b1.y + b2.x * b2.x + b2.y * b2.y + b3.x * b3.x +
                 b3.y * b3.y;
#pragma unroll
      for (int m = 8; m >= 1; m >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, m);
        sk += __shfl_xor_sync(0xffffffffu, sk, m);
      }
      const float iq = t < L ? rsqrtf(sq + p.l2_eps) : 0.f, ik = t < L ? rsqrtf(sk + p.l2_eps) : 0.f;
      *reinterpret_cast<float4*>(sQ + t * 128 + c8) = make_float4(a0.x * iq, a0.y * iq, a1.x * iq, a1.y * iq);
      *reinterpret_cast<float4*>(sQ + t * 128 + c8 + 4) = make_float4(a2.x * iq, a2.y * iq, a3.x * iq, a3.y * iq);
      *reinterpret_cast<float4*>(sK + t * 128 + c8) = make_float4(b0.x * ik, b0.y * ik, b1.x * ik, b1.y * ik);
      *reinterpret_cast<float4*>(sK + t * 128 + c8 + 4) = make_float4(b2.x * ik, b2.y * ik, b3.x * ik, b3.y * ik);
    }
    for (int i = ft; i < 64 * 32; i += FT) {
      const int t = i >> 5, c4 = (i & 31) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < L) {
        v = *reinterpret_cast<const float4*>(sm + KP_U + 32768 + t * 512 + c4 * 4);
        v = make_float4(fmaxf(v.x * kLog2e, g_min2), fmaxf(v.y * kLog2e, g_min2), fmaxf(v.z * kLog2e, g_min2),
                        fmaxf(v.w * kLog2e, g_min2));
      }
      *reinterpret_cast<float4*>(sG + t * 128 + c4) = v;
    }
    if (ft < 64) sBeta[64 * bb + ft] = bt;
    grp_sync<2, FT>();
    bool wide = false;
    if (ft < 256) {
      const int c = ft & 127, t0 = (ft >> 7) * 32;
      float run = 0.f, mn = INFINITY, mx = -INFINITY;
#pragma unroll 8
      for (int t = t0; t < t0 + 32; ++t) {
        run += sG[t * 128 + c];
        sG[t * 128 + c] = run;
        mn = fminf(mn, run);
        mx = fmaxf(mx, run);
      }
      // first half: gamma_0..31 around gamma_31 = run; second half: its sums are gamma_t - gamma_31
      const float ref = t0 == 0 ? run : 0.f;
      wide = !(fmaxf(mx - ref, ref - mn) <= kRefSpan2);  // NaN or infinity: wide
    }
    wide = grp_or<2, FT>(wide);
    for (int i = ft; i < 32 * 32; i += FT) {  // the second half adds the first half's total
      const int t = 32 + (i >> 5), c4 = (i & 31) * 4;
      const float4 base = *reinterpret_cast<const float4*>(sG + 31 * 128 + c4);
      float4* dst = reinterpret_cast<float4*>(sG + t * 128 + c4);
      const float4 v = *dst;
      *dst = make_float4(v.x + base.x, v.y + base.y, v.z + base.z, v.w + base.w);
    }
    if (ft == 0) s_flags[0] = wide ? 0 : 1;
    return true;
  };

  long info_u = -1;  // the unit whose description is below
  int nn = 0, ngc = 0, nh = 0, nc0 = 0, nL = 0;
  bool nvalid = false;
  long front_done = -1;  // the unit whose front phase is in shared memory
  int bcur = 0;          // its beta buffer
  for (long u = blockIdx.x; u < units && ok; u += gridDim.x) {
    int n, gc, h, c0, L;
    bool valid;
    if (info_u == u) {
      n = nn; gc = ngc; h = nh; c0 = nc0; L = nL; valid = nvalid;
    } else {
      valid = kda_unit(p, u, load_guess(p, 0), n, gc, h, c0, L);
    }
    if (!valid) {  // uniform over the CTA
      if (tid == 0) raise_error(p.err, kErrDeviceArgument);
      continue;
    }
    // the next unit, guessed to lie in this unit's sequence: the guess loads while this unit computes
    const long un = u + gridDim.x;
    const UnitGuess guess = load_guess(p, n);
    if (front_done != u) {  // the first unit, or one after a rejected unit: its front phase now
      fence_proxy_async_smem();
      __syncthreads();
      issue_unit(c0, L, h, h / ratio);
      in_flight = true;
      const bool fok = ft >= 0 ? front(L, bcur) : true;
      ok = __syncthreads_and(fok ? 1 : 0) != 0;
      if (!ok) break;  // the rows did not arrive: in_flight stays set for the bounded wait below
      ph_in ^= 1u;
      in_flight = false;
      front_done = u;
    }
    const bool tc_way = s_flags[0] != 0;
    const float* sBc = sBeta + 64 * bcur;
    const int bnext = bcur ^ 1;
    info_u = un;
    nvalid = un < units && kda_unit(p, un, guess, nn, ngc, nh, nc0, nL);
    uint8_t* rec = p.rec + ((size_t)gc * p.Hv + h) * KR_BYTES;
    // the record's K~ = k^ e^gamma (hi / lo), Q~ = q^ e^gamma and vector block, then its
    // Kd = k^ e^(gamma_L - gamma) (hi / lo), by the front group (a warp per token row, a float4 of
    // channels per lane)
    auto kq_record = [&]() {
      for (int i = ft; i < 64 * 32; i += FT) {
        const int t = i >> 5, c4 = (i & 31) * 4;
        const float4 gm = *reinterpret_cast<const float4*>(sG + t * 128 + c4);
        const float4 kk = *reinterpret_cast<const float4*>(sK + t * 128 + c4);
        const float4 qq = *reinterpret_cast<const float4*>(sQ + t * 128 + c4);
        const float4 eg = make_float4(exp2f(gm.x), exp2f(gm.y), exp2f(gm.z), exp2f(gm.w));
        store4_split(rec + KR_KQ, 16384, rec + KR_KLO, 8192, t, c4, f4mul(kk, eg));
        store4_split(rec + KR_KQ, 16384, nullptr, 0, 64 + t, c4, f4mul(qq, eg));
      }
      float* vecg = reinterpret_cast<float*>(rec + KR_VEC);
      if (ft < 64) {
        const float b = sBc[ft];
        vecg[KV_BETA + ft] = b;
        vecg[KV_NCX + ft] = -b;
        vecg[KV_CS + ft] = 1.f;
        vecg[KV_CO + ft] = p.q_scale;
      } else if (ft < 192) {
        vecg[KV_GL + ft - 64] = exp2f(sG[63 * 128 + ft - 64]);
      }
    };
    auto kd_record = [&]() {
      for (int i = ft; i < 64 * 32; i += FT) {
        const int t = i >> 5, c4 = (i & 31) * 4;
        const float4 gm = *reinterpret_cast<const float4*>(sG + t * 128 + c4);
        const float4 gl = *reinterpret_cast<const float4*>(sG + 63 * 128 + c4);
        const float4 kk = *reinterpret_cast<const float4*>(sK + t * 128 + c4);
        store4_split(rec + KR_KD, 8192, rec + KR_KD + 16384, 8192, t, c4, f4mul(kk, f4exp2_diff(gl, gm)));
      }
    };
    // T (hi / lo) into the record, by warps 0 and 1 once their solve is done
    auto t_record = [&]() {
      const float* sT = sTri + kTriBytes / 4;
      for (int i = tid; i < 64 * 8; i += 64) {
        const int t = i >> 3, k0 = (i & 7) * 8;
        const int tb = t >> 4, kb = k0 >> 4;
        const bool upper = kb > tb;  // strictly upper blocks of T are zero
        const float* rowT = sT + ((tb * (tb + 1)) / 2 + (upper ? 0 : kb)) * 256 + (t & 15) * 16;
        const int q0 = (k0 & 15) >> 2, tx = t & 3;
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 v0 = upper ? z4 : *reinterpret_cast<const float4*>(rowT + ((q0 ^ tx) << 2));
        const float4 v1 = upper ? z4 : *reinterpret_cast<const float4*>(rowT + (((q0 + 1) ^ tx) << 2));
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        store8_split(rec + KR_T, rec + KR_T + 8192, 0, t, k0, v);
      }
    };

    bool my_ok = true;
    if (tc_way) {
      // ---- [K'; Q'] and K'' (hi / lo) into the shared region, then [K'; Q'] K''^T on the tensor cores:
      // columns 0..63 take hi x hi + lo x hi, columns 64..127 hi x lo (K = 128 as two 64-channel blocks)
      for (int i = tid; i < 64 * 32; i += NT) {
        const int t = i >> 5, c4 = (i & 31) * 4;
        const float4 gm = *reinterpret_cast<const float4*>(sG + t * 128 + c4);
        const float4 gr = *reinterpret_cast<const float4*>(sG + kRefToken * 128 + c4);
        const float4 kk = *reinterpret_cast<const float4*>(sK + t * 128 + c4);
        const float4 qq = *reinterpret_cast<const float4*>(sQ + t * 128 + c4);
        const float4 er = f4exp2_diff(gm, gr), ec = f4exp2_diff(gr, gm);
        store4_split(sm + KP_AH, 16384, sm + KP_AL, 16384, t, c4, f4mul(kk, er));
        store4_split(sm + KP_AH, 16384, sm + KP_AL, 16384, 64 + t, c4, f4mul(qq, er));
        store4_split(sm + KP_B, 16384, sm + KP_B + 8192, 16384, t, c4, f4mul(kk, ec));  // lo: row 64 + t
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (tid == 0) {
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          mma_bf16_k4<2, 2>(tmem, sw128_desc(sb + KP_AH + kb * 16384), sw128_desc(sb + KP_B + kb * 16384), ID128,
                            kb);
          mma_bf16_k4<2, 2>(tmem, sw128_desc(sb + KP_AL + kb * 16384), sw128_desc(sb + KP_B + kb * 16384), ID64, 1);
        }
        mma_commit(bar_mma);
      }
      mma_flight = true;
      if (warp < 2) {
        // ---- A from tensor memory (warp w: rows 32 w .. 32 w + 31, all 64 columns, times beta_t,
        // s < t) into the solve's layout, then T = (I + A)^-1 on these two warps
        bool got = __all_sync(0xffffffffu, mbar_wait(bar_mma, ph_mma, kWaitLimit));
        tc_fence_after();
        if (got) {
          const int t = tid, tb = t >> 4;
          const float b = sBc[t];
#pragma unroll
          for (int cp = 0; cp < 4; ++cp) {
            float v[16], w2[16];  // columns c: hi x hi + lo x hi; columns 64 + c: hi x lo
            tmem_ld_cols<16>(tmem + ((uint32_t)(warp * 32) << 16) + cp * 16, v);
            tmem_ld_cols<16>(tmem + ((uint32_t)(warp * 32) << 16) + 64 + cp * 16, w2);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += w2[j];
            if (cp <= tb) {  // a block on or below the diagonal: four float4 groups
              float* rowp = sTri + ((tb * (tb + 1)) / 2 + cp) * 256 + (t & 15) * 16;
#pragma unroll
              for (int g4 = 0; g4 < 4; ++g4) {
                const int s = 16 * cp + 4 * g4, j = 4 * g4;
                const float4 w = make_float4(s < t ? b * v[j] : 0.f, s + 1 < t ? b * v[j + 1] : 0.f,
                                             s + 2 < t ? b * v[j + 2] : 0.f, s + 3 < t ? b * v[j + 3] : 0.f);
                *reinterpret_cast<float4*>(rowp + ((g4 ^ (t & 3)) << 2)) = w;
              }
            }
          }
        }
        tc_fence_before();
        got = grp_and<1, 64>(got);  // A complete (both warps)
        if (got) {
          solve_tri_batched<true>(sm + KP_TRI, 1, tid);
          t_record();
        }
        my_ok = got;
      } else {
        // ---- the front group: K~ / Q~ while the products run; then the next unit's rows, P from
        // tensor memory (rows 64.. of the lanes, times q_scale, s <= t) into the record, Kd, and the
        // next unit's front phase beside the solve
        kq_record();
        bool got = __all_sync(0xffffffffu, mbar_wait(bar_mma, ph_mma, kWaitLimit));
        tc_fence_after();
        got = grp_and<2, FT>(got);
        const bool go = got && nvalid;
        if (go) issue_unit(nc0, nL, nh, nh / ratio);
        if (got && (q4 & 2)) {
          float v[16], w2[16];
          tmem_ld_cols<16>(tmem + ((uint32_t)(q4 * 32) << 16) + cpart * 16, v);
          tmem_ld_cols<16>(tmem + ((uint32_t)(q4 * 32) << 16) + 64 + cpart * 16, w2);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += w2[j];
          const int t = q4 * 32 + lane - 64, s0 = cpart * 16;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            float p8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) p8[e] = (s0 + 8 * q + e) <= t ? p.q_scale * v[8 * q + e] : 0.f;
            store8_split(rec + KR_P, nullptr, 0, t, s0 + 8 * q, p8);
          }
        }
        tc_fence_before();
        kd_record();
        bool landed = false;
        if (go) landed = front(nL, bnext);
        if (ft == 0) {
          s_flags[1] = go ? 1 : 0;
          s_flags[2] = landed ? 1 : 0;
        }
        my_ok = got && (!go || landed);
      }
      ph_mma ^= 1u;
      mma_flight = !my_ok;
      if (!my_ok) raise_error(p.err, kErrTimeout);
    } else {
      // the per-token decay factors 2^g from the raw log decays, still in the shared region (rows
      // past L: g = 0); A's blocks cleared; then P cleared over the factors' neighbours
      for (int i = tid; i < 64 * 32; i += NT) {
        const int t = i >> 5, c4 = (i & 31) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < L) {
          v = *reinterpret_cast<const float4*>(sm + KP_U + 32768 + t * 512 + c4 * 4);
          v = make_float4(fmaxf(v.x * kLog2e, g_min2), fmaxf(v.y * kLog2e, g_min2), fmaxf(v.z * kLog2e, g_min2),
                          fmaxf(v.w * kLog2e, g_min2));
        }
        *reinterpret_cast<float4*>(sAf + t * 128 + c4) = make_float4(exp2f(v.x), exp2f(v.y), exp2f(v.z), exp2f(v.w));
      }
      for (int i = tid; i < (int)(kTriBytes / 16); i += NT)
        reinterpret_cast<float4*>(sTri)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      __syncthreads();
      for (int i = tid; i < 64 * 64 / 4; i += NT) reinterpret_cast<float4*>(sP)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      // ---- A (beta-weighted, strictly lower) and P (q_scale) inside the four diagonal 16 x 16 blocks:
      // thread (block d, column s, channel eighth cc: float4 groups cc, cc + 8, cc + 16, cc + 24), the
      // decay 2^(gamma_t - gamma_s) as the running product of the per-token factors a_(s+1) .. a_t
      {
        const int cc = lane & 7, sl = ((warp & 3) << 2) | (lane >> 3), d = warp >> 2;
        const int s = 16 * d + sl;
        float2 ks[8], f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 kv = *reinterpret_cast<const float4*>(sK + s * 128 + 32 * j + 4 * cc);
          ks[2 * j] = make_float2(kv.x, kv.y);
          ks[2 * j + 1] = make_float2(kv.z, kv.w);
          f[2 * j] = f[2 * j + 1] = make_float2(1.f, 1.f);
        }
        __syncthreads();  // sP cleared
        for (int tl = 0; tl < 16; ++tl) {
          const int t = 16 * d + tl;
          const bool after = t > s;
          float2 pa = make_float2(0.f, 0.f), pq = pa;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int off = t * 128 + 32 * j + 4 * cc;
            const float4 av = *reinterpret_cast<const float4*>(sAf + off);
            const float4 kv = *reinterpret_cast<const float4*>(sK + off);
            const float4 qv = *reinterpret_cast<const float4*>(sQ + off);
            if (after) {
              f[2 * j] = __fmul2_rn(f[2 * j], make_float2(av.x, av.y));
              f[2 * j + 1] = __fmul2_rn(f[2 * j + 1], make_float2(av.z, av.w));
            }
            const float2 w0 = __fmul2_rn(ks[2 * j], f[2 * j]), w1 = __fmul2_rn(ks[2 * j + 1], f[2 * j + 1]);
            pa = __ffma2_rn(make_float2(kv.x, kv.y), w0, pa);
            pa = __ffma2_rn(make_float2(kv.z, kv.w), w1, pa);
            pq = __ffma2_rn(make_float2(qv.x, qv.y), w0, pq);
            pq = __ffma2_rn(make_float2(qv.z, qv.w), w1, pq);
          }
          float sa = pa.x + pa.y, sq = pq.x + pq.y;
#pragma unroll
          for (int m = 1; m <= 4; m <<= 1) {
            sa += __shfl_xor_sync(0xffffffffu, sa, m);
            sq += __shfl_xor_sync(0xffffffffu, sq, m);
          }
          if (cc == 0) {
            if (after) sTri[tri_index(t, s)] = sBc[t] * sa;
            if (t >= s) sP[t * 64 + s] = p.q_scale * sq;
          }
        }
      }

      // ---- the blocks below the diagonal: rows in block a, columns in block b < a, as one product
      // around r, the last token of block b: (x_t 2^(gamma_t - gamma_r)) (k^_s 2^(gamma_r - gamma_s))^T
      for (int b = 0; b < 3; ++b) {
        const int r = 16 * b + 15;
        __syncthreads();  // the column buffer's previous readers are done
        for (int i = tid; i < 16 * 32; i += NT) {
          const int jj = i >> 5, c4 = (i & 31) * 4, s = 16 * b + jj;
          const float4 e = f4exp2_diff(*reinterpret_cast<const float4*>(sG + r * 128 + c4),
                                       *reinterpret_cast<const float4*>(sG + s * 128 + c4));
          *reinterpret_cast<float4*>(sKb + jj * 128 + c4) = f4mul(*reinterpret_cast<const float4*>(sK + s * 128 + c4), e);
        }
        for (int a = b + 1; a < 4; ++a) {
          for (int i = tid; i < 16 * 32; i += NT) {
            const int ii = i >> 5, c4 = (i & 31) * 4, t = 16 * a + ii;
            const float4 e = f4exp2_diff(*reinterpret_cast<const float4*>(sG + t * 128 + c4),
                                         *reinterpret_cast<const float4*>(sG + r * 128 + c4));
            *reinterpret_cast<float4*>(sRK + ii * 128 + c4) = f4mul(*reinterpret_cast<const float4*>(sK + t * 128 + c4), e);
            *reinterpret_cast<float4*>(sRQ + ii * 128 + c4) = f4mul(*reinterpret_cast<const float4*>(sQ + t * 128 + c4), e);
          }
          __syncthreads();
          {
            // thread: matrix (A or P), a 4 x 4 tile of the 16 x 16 block, the float4 groups kq and
            // kq + 16 of the channels; the 16 lanes of a tile then reduce its 16 sums butterfly-wise,
            // each ending with one of them
            const int which = tid >> 8, tile = (tid >> 4) & 15, kq = tid & 15;
            const int i0 = (tile >> 2) * 4, j0 = (tile & 3) * 4;
            const float* R = which ? sRQ : sRK;
            float2 acc[16];
#pragma unroll
            for (int o = 0; o < 16; ++o) acc[o] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int cb = 64 * j + 4 * kq;
              float4 rv[4], kv[4];
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                rv[x] = *reinterpret_cast<const float4*>(R + (i0 + x) * 128 + cb);
                kv[x] = *reinterpret_cast<const float4*>(sKb + (j0 + x) * 128 + cb);
              }
#pragma unroll
              for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                  acc[4 * x + y] = __ffma2_rn(make_float2(rv[x].x, rv[x].y), make_float2(kv[y].x, kv[y].y), acc[4 * x + y]);
                  acc[4 * x + y] = __ffma2_rn(make_float2(rv[x].z, rv[x].w), make_float2(kv[y].z, kv[y].w), acc[4 * x + y]);
                }
            }
            float v16[16];
#pragma unroll
            for (int o = 0; o < 16; ++o) v16[o] = acc[o].x + acc[o].y;
            const bool b3 = kq & 8, b2 = kq & 4, b1 = kq & 2, b0 = kq & 1;
            float v8[8], v4[4], v2[2];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float send = b3 ? v16[i] : v16[i + 8], keep = b3 ? v16[i + 8] : v16[i];
              v8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float send = b2 ? v8[i] : v8[i + 4], keep = b2 ? v8[i + 4] : v8[i];
              v4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float send = b1 ? v4[i] : v4[i + 2], keep = b1 ? v4[i + 2] : v4[i];
              v2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
            }
            const float send = b0 ? v2[0] : v2[1], keep = b0 ? v2[1] : v2[0];
            const float v1 = keep + __shfl_xor_sync(0xffffffffu, send, 1);
            // this lane holds sum kq: tile row kq / 4, column kq % 4
            const int t = 16 * a + i0 + (kq >> 2), s = 16 * b + j0 + (kq & 3);
            if (which == 0) sTri[tri_index(t, s)] = sBc[t] * v1;
            else sP[t * 64 + s] = p.q_scale * v1;
          }
          __syncthreads();  // the row buffers are read before the next row block is formed
        }
      }
      for (int i = tid; i < 64 * 8; i += NT) {  // P (bf16) into the record
        const int t = i >> 3, k0 = (i & 7) * 8;
        const float4 p0 = *reinterpret_cast<const float4*>(sP + t * 64 + k0);
        const float4 p1 = *reinterpret_cast<const float4*>(sP + t * 64 + k0 + 4);
        const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        store8_split(rec + KR_P, nullptr, 0, t, k0, pv);
      }
      // the shared region's generic accesses, before the next unit's rows overwrite it
      fence_proxy_async_smem();
      __syncthreads();
      const bool go = nvalid;
      if (go) issue_unit(nc0, nL, nh, nh / ratio);
      if (warp < 2) {
        solve_tri_batched<true>(sm + KP_TRI, 1, tid);
        t_record();
      } else {
        kq_record();
        kd_record();
        bool landed = false;
        if (go) landed = front(nL, bnext);
        if (ft == 0) {
          s_flags[1] = go ? 1 : 0;
          s_flags[2] = landed ? 1 : 0;
        }
        my_ok = !go || landed;
      }
    }
    ok = __syncthreads_and(my_ok ? 1 : 0) != 0;
    {
      const bool issued = s_flags[1] != 0, landed = s_flags[2] != 0;
      if (issued && landed) {  // the next unit's front phase is done
        ph_in ^= 1u;
        front_done = un;
      }
      in_flight = issued && !landed;
    }
    bcur = bnext;
    if (!ok) break;
  }

  // after an early exit, let copies and products still in flight land (bounded)
  if (in_flight) mbar_wait(bar_in, ph_in, kWaitLimit);
  if (mma_flight) mbar_wait(bar_mma, ph_mma ^ 1u, kWaitLimit);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

struct KStateParams {
  CUtensorMap tmap;    // qkv [T][C] bf16, box 64 x 64, 128-byte swizzle (the v tiles)
  CUtensorMap tmap_z;  // z [T][Hv * 128] bf16, box 128 x 64, no swizzle (valid when z != NULL)
  const int32_t* cu;
  const int32_t* order;
  unsigned* counter;
  const int32_t* chunk_off;
  const uint8_t* rec;
  const float* state_in;
  float* state_out;
  const uint16_t* z;
  const uint16_t* norm_w;
  uint16_t* out;
  unsigned* err;
  int N, T, Hk, Hv, nc_max;
  float rms_eps;
};

// Persistent CTAs take (sequence, V head) items longest sequence first and carry the fp32 state
// [value row = tensor-memory lane, key = column] through the sequence's chunks.  Thread (row,
// part) owns value row `row` and kW of each 64-column accumulator.  Per chunk:
//   S0 -> bf16 hi / lo (one 64-key half at a time; the state takes its decay diag(e^gamma_L) there)
//   [X | O1] = S0 [K~; Q~]^T                 (X with the hi / lo pairs of S0 and K~)
//   R = (V - X) diag(beta) -> hi / lo        ->  E = R T^T   (R read from tensor memory)
//   S += E Kd (hi / lo pairs),  O2 = E P^T   ->  o = q_scale O1 + O2  ->  gated RMSNorm  ->  out
// Two CTAs per SM.  The record parts arrive by bulk copies as their buffers free up: [K~; Q~] (and
// K~ lo) once the previous chunk's state update has read that buffer's T, Kd and E; T and Kd (one
// copy, prefetched into L2 a chunk ahead) once the X products have read [K~; Q~]; P once the
// previous chunk's O2 product is done; the vector block a chunk ahead.
__global__ void __launch_bounds__(kThreads, 2) kda_state_kernel(const __grid_constant__ KStateParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024k(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, part = warp >> 2;
  const int row = q4 * 32 + lane;
  const int ratio = p.Hv / p.Hk;
  const long total_items = (long)p.N * p.Hv;

  float* s_work = reinterpret_cast<float*>(sm + SK_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SK_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SK_BAR + 96);
  int* item_slot = reinterpret_cast<int*>(sm + SK_BAR + 104);
  const uint32_t bar_qk = smem_u32(&bars[0]), bar_v = smem_u32(&bars[1]), bar_tp = smem_u32(&bars[2]),
                 bar_h = smem_u32(&bars[3]), bar_x = smem_u32(&bars[4]), bar_e = smem_u32(&bars[5]),
                 bar_s = smem_u32(&bars[6]), bar_z = smem_u32(&bars[7]), bar_kd = smem_u32(&bars[10]);
  const uint32_t bar_vec0 = smem_u32(&bars[8]);  // one barrier per vector buffer: bar_vec0 + 8 * buffer

  if (tid == 0) {
    for (int i = 0; i < 11; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
    prefetch_tensormap(&p.tmap);
    if (p.z) prefetch_tensormap(&p.tmap_z);
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), KSC_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);

  constexpr uint32_t ID64 = idesc_bf16_f32(128, 64);
  constexpr uint32_t ID128 = idesc_bf16_f32(128, 128);
  constexpr uint32_t ID128_BMN = idesc_bf16_f32_bmn(128, 128);
  bool ok = true;
  uint32_t ph_mma = 0, ph_qk = 0, ph_v = 0, ph_tp = 0, ph_z = 0, ph_kd = 0;
  uint32_t ph_vec = 0, pend_vec = 0;  // bit b: parity of / load in flight on vector buffer b
  bool pend_qk = false, pend_v = false, pend_tp = false, pend_z = false, pend_kd = false;
  const bool gated = p.z != nullptr;
  float wf[4] = {1.f, 1.f, 1.f, 1.f};
  if (gated) {
    const uint2 ww = __ldg(reinterpret_cast<const uint2*>(p.norm_w + lane * 4));
    wf[0] = __uint_as_float(ww.x << 16); wf[1] = __uint_as_float(ww.x & 0xFFFF0000u);
    wf[2] = __uint_as_float(ww.y << 16); wf[3] = __uint_as_float(ww.y & 0xFFFF0000u);
  }

  auto wait_bar = [&](uint32_t bar, uint32_t& ph) {
    const bool got = mbar_wait(bar, ph, kWaitLimit);
    ph ^= 1u;
    if (!got) raise_error(p.err, kErrTimeout);
    ok = __syncthreads_and(got ? 1 : 0) != 0 && ok;
  };
  auto wait_two = [&](uint32_t bar_a, uint32_t& ph_a, uint32_t bar_b, uint32_t& ph_b) {  // one barrier for both
    const bool got = mbar_wait(bar_a, ph_a, kWaitLimit) && mbar_wait(bar_b, ph_b, kWaitLimit);
    ph_a ^= 1u;
    ph_b ^= 1u;
    if (!got) raise_error(p.err, kErrTimeout);
    ok = __syncthreads_and(got ? 1 : 0) != 0 && ok;
  };
  auto await_mma = [&](uint32_t bar) {
    uint32_t ph = ph_mma;
    wait_bar(bar, ph);
    tc_fence_after();
  };
  auto operands_ready = [&]() {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  auto issue_v = [&](int c0, int h) {
    mbar_arrive_expect_tx(bar_v, kBytesV);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
      tma_load_2d(sb + SK_V + kb * 8192, &p.tmap, 2 * p.Hk * kHeadDim + h * kHeadDim + kb * 64, c0, bar_v);
  };
  auto issue_z = [&](int c0, int h) {  // into the V buffer, once R has consumed V
    mbar_arrive_expect_tx(bar_z, kBytesZ);
    tma_load_2d(sb + SK_V, &p.tmap_z, h * kHeadDim, c0, bar_z);
  };
  // a chunk's record: [K~ hi; Q~] and K~ lo (needed by the X MMAs), Kd (the state update), T and P
  // (from the E MMA on), and its vector block (at chunk start; double buffered, so it is fetched a
  // whole chunk ahead)
  auto recp = [&](int gc, int h) { return p.rec + ((size_t)gc * p.Hv + h) * KR_BYTES; };
  auto issue_kq = [&](int gc, int h) {
    mbar_arrive_expect_tx(bar_qk, kKRecKQ);
    bulk_load(sb + SK_QK, recp(gc, h) + KR_KQ, kKRecKQ, bar_qk);
  };
  auto issue_tkd = [&](int gc, int h) {  // into the [K~; Q~] buffer, once the X products have read it
    mbar_arrive_expect_tx(bar_kd, kKRecTKD);
    bulk_load(sb + SK_T, recp(gc, h) + KR_T, kKRecTKD, bar_kd);
  };
  auto issue_p = [&](int gc, int h) {
    mbar_arrive_expect_tx(bar_tp, kKRecP);
    bulk_load(sb + SK_P, recp(gc, h) + KR_P, kKRecP, bar_tp);
  };
  auto issue_vec = [&](int gc, int h, int vb) {
    mbar_arrive_expect_tx(bar_vec0 + 8 * vb, kKRecVec);
    bulk_load(sb + SK_VEC + vb * kKRecVec, recp(gc, h) + KR_VEC, kKRecVec, bar_vec0 + 8 * vb);
  };
  // 32 fp32 values of this thread's row (tokens part * kW ..) -> bf16 hi / lo pairs in tensor memory:
  // hi in 16 columns at `taddr`, lo in the next 16 (the even token in the low half of a column)
  auto store_split_tmem = [&](uint32_t taddr, const float (&v)[kW]) {
    float hw[kW / 2], lw[kW / 2];
#pragma unroll
    for (int j = 0; j < kW / 2; ++j) {
      const uint32_t hp = pack_bf2(v[2 * j], v[2 * j + 1]);
      const float2 rem = __ffma2_rn(make_float2(__uint_as_float(hp << 16), __uint_as_float(hp & 0xFFFF0000u)),
                                    make_float2(-1.f, -1.f), make_float2(v[2 * j], v[2 * j + 1]));
      hw[j] = __uint_as_float(hp);
      lw[j] = __uint_as_float(pack_bf2(rem.x, rem.y));
    }
    tmem_st16(taddr, hw);
    tmem_st16(taddr + kW / 2, lw);
  };
  // S0 columns [k0, k0 + 64) -> hi/lo operand tiles (64 keys = one K block); state <- S0 diag(e^gamma_L)
  // there (a decay per key column)
  auto convert_half = [&](int k0, const float* vec) {
    float v[kW];
    tmem_ld_cols<kW>(tl + KSC_S + k0 + part * kW, v);
#pragma unroll
    for (int q = 0; q < kW / 8; ++q) store8_split(sm + SK_W, sm + SK_W + 16384, 0, row, part * kW + 8 * q, v + 8 * q);
    const float* gl = vec + KV_GL + k0 + part * kW;
#pragma unroll
    for (int i = 0; i < kW; i += 4) {
      const float4 g4 = *reinterpret_cast<const float4*>(gl + i);
      const float2 m0 = __fmul2_rn(make_float2(v[i], v[i + 1]), make_float2(g4.x, g4.y));
      const float2 m1 = __fmul2_rn(make_float2(v[i + 2], v[i + 3]), make_float2(g4.z, g4.w));
      v[i] = m0.x; v[i + 1] = m0.y; v[i + 2] = m1.x; v[i + 3] = m1.y;
    }
    tmem_st32(tl + KSC_S + k0 + part * kW, v);
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
    const int seq_lo = __ldg(p.cu + n), seq_hi = __ldg(p.cu + n + 1);
    const int nch = (max(0, seq_hi - seq_lo) + kChunk - 1) / kChunk;
    const int jb = 0, je = nch;
    const int seq_s = seq_lo, seq_e = seq_hi;
    const int gc0 = __ldg(p.chunk_off + n) + jb;
    if (n < 0 || n >= p.N || seq_lo < 0 || seq_hi < seq_lo || seq_hi > p.T || gc0 < 0 ||
        gc0 + (je - jb) > p.nc_max) {
      if (tid == 0) raise_error(p.err, kErrDeviceArgument);
      continue;
    }
    (void)kh;
    if (tid == 0 && seq_e > seq_s) {
      issue_vec(gc0, h, 0);
      issue_kq(gc0, h);
      issue_v(seq_s, h);
      issue_p(gc0, h);
      bulk_prefetch_l2(recp(gc0, h) + KR_T, kKRecTKD);  // T and Kd: copied once X is done
    }
    pend_qk = pend_v = pend_tp = seq_e > seq_s;
    if (seq_e > seq_s) pend_vec |= 1u;

    // ---- initial state -> tensor memory
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
        tmem_st32(tl + KSC_S + c0, v);
      }
    }

    int vb = 0;
    for (int c0 = seq_s, gc = gc0; c0 < seq_e && ok; c0 += kChunk, ++gc, ph_mma ^= 1u, vb ^= 1) {
      const int L = min(kChunk, seq_e - c0);
      const bool has_next = c0 + kChunk < seq_e;
      const float* vec = reinterpret_cast<const float*>(sm + SK_VEC + vb * kKRecVec);

      {
        const uint32_t vec_limit = kWaitLimit;
        const bool got = mbar_wait(bar_vec0 + 8 * vb, (ph_vec >> vb) & 1u, vec_limit);
        ph_vec ^= 1u << vb;
        pend_vec &= ~(1u << vb);
        if (!got) raise_error(p.err, kErrTimeout);
        ok = __syncthreads_and(got ? 1 : 0) != 0 && ok;
      }
      if (!ok) break;

      // ================= [X | O1] = S0 [K~; Q~]^T one 64-key half at a time: X from S0 hi x K~ hi,
      // S0 hi x K~ lo and S0 lo x K~ hi, the output-only O1 from S0 hi x Q~
      convert_half(0, vec);
      fence_proxy_async_smem();
      tc_fence_before();
      wait_bar(bar_qk, ph_qk);  // the chunk's K~ / Q~ tiles
      pend_qk = false;
      tc_fence_after();
      if (!ok) break;
      if (tid == 0) {
        mma_bf16_k4<2, 2>(tmem + KSC_X, sw128_desc(sb + SK_W), sw128_desc(sb + SK_QK), ID128, 0);
        mma_bf16_k4<2, 2>(tmem + KSC_X, sw128_desc(sb + SK_W + 16384), sw128_desc(sb + SK_QK), ID64, 1);
        mma_bf16_k4<2, 2>(tmem + KSC_X, sw128_desc(sb + SK_W), sw128_desc(sb + SK_KLO), ID64, 1);
        mma_commit(bar_h);
      }
      await_mma(bar_h);
      if (!ok) break;
      convert_half(64, vec);
      operands_ready();
      if (tid == 0) {
        mma_bf16_k4<2, 2>(tmem + KSC_X, sw128_desc(sb + SK_W), sw128_desc(sb + SK_QK + 16384), ID128, 1);
        mma_bf16_k4<2, 2>(tmem + KSC_X, sw128_desc(sb + SK_W + 16384), sw128_desc(sb + SK_QK + 16384), ID64, 1);
        mma_bf16_k4<2, 2>(tmem + KSC_X, sw128_desc(sb + SK_W), sw128_desc(sb + SK_KLO + 8192), ID64, 1);
        mma_commit(bar_x);
      }
      {
        uint32_t ph = ph_mma;
        wait_two(bar_x, ph, bar_v, ph_v);
        tc_fence_after();
      }
      pend_v = false;
      if (!ok) break;
      if (tid == 0) issue_tkd(gc, h);  // the [K~; Q~] buffer is free once the X MMAs are done
      pend_kd = true;

      // ================= R = (V - X^T) diag(beta) -> hi/lo (value-major)
      {
        float x[kW];
        tmem_ld_cols<kW>(tl + KSC_X + part * kW, x);
        // V[t][row] for t = part * kW + i: the swizzle term depends on i & 7 only
        const uint8_t* vbase = sm + SK_V + (row >> 6) * 8192 + part * kW * 128 + ((row & 7) << 1);
        const int rsw = (row >> 3) & 7;
        auto v_at = [&](int i) {
          return bf2f(*reinterpret_cast<const uint16_t*>(vbase + i * 128 + ((rsw ^ (i & 7)) << 4)));
        };
#pragma unroll
        for (int i4 = 0; i4 < kW; i4 += 4) {
          const float4 bt = *reinterpret_cast<const float4*>(vec + KV_BETA + part * kW + i4);
          const float4 nc = *reinterpret_cast<const float4*>(vec + KV_NCX + part * kW + i4);
          const float2 r0 = __ffma2_rn(make_float2(nc.x, nc.y), make_float2(x[i4], x[i4 + 1]),
                                       __fmul2_rn(make_float2(bt.x, bt.y), make_float2(v_at(i4), v_at(i4 + 1))));
          const float2 r1 = __ffma2_rn(make_float2(nc.z, nc.w), make_float2(x[i4 + 2], x[i4 + 3]),
                                       __fmul2_rn(make_float2(bt.z, bt.w), make_float2(v_at(i4 + 2), v_at(i4 + 3))));
          x[i4] = r0.x; x[i4 + 1] = r0.y; x[i4 + 2] = r1.x; x[i4 + 3] = r1.y;
        }
        store_split_tmem(tl + KSC_X + part * kW, x);  // over this thread's own X columns
      }
      // O1 leaves its columns (they take E next): into registers now, staged while the E MMAs run
      float o1[kW];
      tmem_ld_cols<kW>(tl + KSC_O1 + part * kW, o1);
      fence_proxy_async_smem();
      tc_fence_before();
      wait_bar(bar_kd, ph_kd);  // T and Kd of this chunk
      pend_kd = false;
      tc_fence_after();
      if (!ok) break;
      if (tid == 0) {
        // E^T = R T^T  (hi*hi + hi*lo + lo*hi), R from tensor memory (hi / lo pairs of 32 tokens per
        // thread part: hi at columns 32 p, lo at 32 p + 16 of the X region)
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<2>(tmem + KSC_O1, tmem + KSC_X + 32 * pp, sw128_desc(sb + SK_T) + 4 * pp, ID64, pp);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<2>(tmem + KSC_O1, tmem + KSC_X + 32 * pp, sw128_desc(sb + SK_T + 8192) + 4 * pp, ID64, 1);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<2>(tmem + KSC_O1, tmem + KSC_X + 32 * pp + 16, sw128_desc(sb + SK_T) + 4 * pp, ID64, 1);
        mma_commit(bar_e);
      } else if (tid == 32) {
        // the V buffer is free: the gate input of this chunk (gated), else the next chunk's v; and
        // the next chunk's vector block into the other buffer (last read by chunk c - 1)
        if (gated) issue_z(c0, h);
        else if (has_next) issue_v(c0 + kChunk, h);
        if (has_next) issue_vec(gc + 1, h, vb ^ 1);
      }
      if (has_next) pend_vec |= 1u << (vb ^ 1);
      pend_z = gated;
      pend_v = !gated && has_next;
      // o1 diag(c_o) -> the staging area (token-major fp32), free since the X MMAs completed
#pragma unroll
      for (int i4 = 0; i4 < kW; i4 += 4) {
        const int t0 = part * kW + i4;
        const float4 co = *reinterpret_cast<const float4*>(vec + KV_CO + t0);
        const float2 a = __fmul2_rn(make_float2(o1[i4], o1[i4 + 1]), make_float2(co.x, co.y));
        const float2 b = __fmul2_rn(make_float2(o1[i4 + 2], o1[i4 + 3]), make_float2(co.z, co.w));
        s_work[t0 * 128 + row] = a.x;
        s_work[(t0 + 1) * 128 + row] = a.y;
        s_work[(t0 + 2) * 128 + row] = b.x;
        s_work[(t0 + 3) * 128 + row] = b.y;
      }
      await_mma(bar_e);
      if (!ok) break;

      // ================= E~ = E diag(c_s) -> hi/lo (tensor memory, over R);  E -> bf16 (output operand, over T)
      {
        float ev[kW], es[kW];
        tmem_ld_cols<kW>(tl + KSC_O1 + part * kW, ev);
#pragma unroll
        for (int q = 0; q < kW / 8; ++q) {
          const float4 c0v = *reinterpret_cast<const float4*>(vec + KV_CS + part * kW + 8 * q);
          const float4 c1v = *reinterpret_cast<const float4*>(vec + KV_CS + part * kW + 8 * q + 4);
          const float* e8 = ev + 8 * q;
          const float2 p0 = __fmul2_rn(make_float2(e8[0], e8[1]), make_float2(c0v.x, c0v.y));
          const float2 p1 = __fmul2_rn(make_float2(e8[2], e8[3]), make_float2(c0v.z, c0v.w));
          const float2 p2 = __fmul2_rn(make_float2(e8[4], e8[5]), make_float2(c1v.x, c1v.y));
          const float2 p3 = __fmul2_rn(make_float2(e8[6], e8[7]), make_float2(c1v.z, c1v.w));
          float* s8 = es + 8 * q;
          s8[0] = p0.x; s8[1] = p0.y; s8[2] = p1.x; s8[3] = p1.y; s8[4] = p2.x; s8[5] = p2.y; s8[6] = p3.x; s8[7] = p3.y;
          store8_split(sm + SK_T, nullptr, 0, row, part * kW + 8 * q, e8);
        }
        store_split_tmem(tl + KSC_X + part * kW, es);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      wait_bar(bar_tp, ph_tp);  // P of this chunk (fetched when the previous chunk's update was done)
      pend_tp = false;
      tc_fence_after();
      if (!ok) break;
      if (tid == 0) {
        // S += E~ Kd (E~ hi x Kd hi + E~ hi x Kd lo + E~ lo x Kd hi): B = the Kd rows read MN-major
        // (N = 128 keys, 16 tokens per step), E~ from tensor memory as R was; O2 = E P^T into the E columns
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<128>(tmem + KSC_S, tmem + KSC_X + 32 * pp, sw128_mn_desc(sb + SK_KD, 8192) + 256 * pp,
                              ID128_BMN, 1);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<128>(tmem + KSC_S, tmem + KSC_X + 32 * pp, sw128_mn_desc(sb + SK_KD + 16384, 8192) + 256 * pp,
                              ID128_BMN, 1);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<128>(tmem + KSC_S, tmem + KSC_X + 32 * pp + 16, sw128_mn_desc(sb + SK_KD, 8192) + 256 * pp,
                              ID128_BMN, 1);
        mma_bf16_k4<2, 2>(tmem + KSC_O1, sw128_desc(sb + SK_T), sw128_desc(sb + SK_P), ID64, 0);
        mma_commit(bar_s);
      }
      constexpr int kTok = kChunk / kWarps;
      await_mma(bar_s);
      if (!ok) break;
      if (has_next) {  // two issuing threads in different warps, so neither lags by both
        if (tid == 0) {
          issue_kq(gc + 1, h);  // the buffer's T, Kd and E have been read by the products
          bulk_prefetch_l2(recp(gc + 1, h) + KR_T, kKRecTKD);
        } else if (tid == 32) {
          issue_p(gc + 1, h);
        }
      }
      pend_qk = pend_tp = has_next;

      // ================= output: o = O1 diag(c_o) (staged) + O2, then the gated RMSNorm
      {
        float o2a[16], o2b[16];
        tmem_ld16x2(tl + KSC_O1 + part * kW, tl + KSC_O1 + part * kW + 16, o2a, o2b);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          s_work[(part * kW + i) * 128 + row] += o2a[i];
          s_work[(part * kW + 16 + i) * 128 + row] += o2b[i];
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
        float2 r[kTok][2];
        float ss[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i) {
          const float4 v = *reinterpret_cast<const float4*>(s_work + (warp + kWarps * i) * 128 + lane * 4);
          r[i][0] = make_float2(v.x, v.y);
          r[i][1] = make_float2(v.z, v.w);
          const float2 q2 = __ffma2_rn(r[i][1], r[i][1], __fmul2_rn(r[i][0], r[i][0]));
          ss[i] = q2.x + q2.y;
        }
        if (gated) {
#pragma unroll
          for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
            for (int i = 0; i < kTok; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], m);
          const float2 half2 = make_float2(0.5f, 0.5f);
          const float2 w01 = make_float2(wf[0], wf[1]), w23 = make_float2(wf[2], wf[3]);
#pragma unroll
          for (int i = 0; i < kTok; ++i) {
            const float rstd = rsqrtf(fmaf(ss[i], 1.0f / kHeadDim, p.rms_eps));
            const uint2 zz = *reinterpret_cast<const uint2*>(sm + SK_V + (warp + kWarps * i) * 256 + lane * 8);
            // sigmoid(z) = (1 + tanh(z / 2)) / 2, the tanh of a bf16 pair in one operation (z is bf16;
            // halving it is exact)
            const float2 s01 = __ffma2_rn(half2, tanh_half_bf16x2(zz.x), half2);
            const float2 s23 = __ffma2_rn(half2, tanh_half_bf16x2(zz.y), half2);
            const float2 rs = make_float2(rstd, rstd);
            r[i][0] = __fmul2_rn(__fmul2_rn(r[i][0], __fmul2_rn(w01, rs)), s01);
            r[i][1] = __fmul2_rn(__fmul2_rn(r[i][1], __fmul2_rn(w23, rs)), s23);
          }
        }
        // rows t < L go straight to global memory: a warp writes 256 contiguous bytes per token, and
        // the z buffer is free for the next v as soon as every warp has read its rows
#pragma unroll
        for (int i = 0; i < kTok; ++i) {
          const int t = warp + kWarps * i;
          const uint2 packed = make_uint2(pack_bf2(r[i][0].x, r[i][0].y), pack_bf2(r[i][1].x, r[i][1].y));
          if (t < L) *reinterpret_cast<uint2*>(p.out + ((size_t)(c0 + t) * p.Hv + h) * kHeadDim + lane * 4) = packed;
        }
      }
      fence_proxy_async_smem();  // vector-block and z reads -> the async proxy (the next loads)
      tc_fence_before();
      __syncthreads();  // staging reads and accumulator reads done before the next chunk reuses them
      tc_fence_after();
      if (tid == 64 && gated && has_next) issue_v(c0 + kChunk, h);
      if (gated && has_next) pend_v = true;
    }
    if (!ok) break;

    // ---- final state -> global
    if (p.state_out) {
      const size_t row_off = (((size_t)n * p.Hv + h) * kHeadDim + row) * kHeadDim;
#pragma unroll
      for (int cq = 0; cq < 4 / kParts; ++cq) {
        const int c0 = part * (128 / kParts) + cq * 32;
        float v[32];
        tmem_ld32(tl + KSC_S + c0, v);
        float4* dst = reinterpret_cast<float4*>(p.state_out + row_off + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  // after an early exit, let copies still in flight land before the CTA leaves (bounded)
  if (pend_qk) mbar_wait(bar_qk, ph_qk, kWaitLimit);
  if (pend_v) mbar_wait(bar_v, ph_v, kWaitLimit);
  if (pend_tp) mbar_wait(bar_tp, ph_tp, kWaitLimit);
  if (pend_vec & 1u) mbar_wait(bar_vec0, ph_vec & 1u, kWaitLimit);
  if (pend_vec & 2u) mbar_wait(bar_vec0 + 8, (ph_vec >> 1) & 1u, kWaitLimit);
  if (pend_z) mbar_wait(bar_z, ph_z, kWaitLimit);
  if (pend_kd) mbar_wait(bar_kd, ph_kd, kWaitLimit);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, KSC_COLS);
  }
}


}  // namespace

namespace {

size_t kpad256(size_t b) { return (b + 255) / 256 * 256; }
long kda_chunk_bound(int N, int T) { return ((long)T + 63L * N) / kChunk; }

template <typename K>
cudaError_t kda_set_smem_once(K kernel, uint32_t bytes, int (&done)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && dev < 64) done[dev] = 1;
  return e;
}

}  // namespace

size_t kda_chunk_workspace_bytes(int N, int T, int Hv) {
  if (N <= 0) return 0;
  return 256 + kpad256((size_t)4 * N) + kpad256((size_t)4 * (N + 1)) +
         (size_t)kda_chunk_bound(N, T) * (size_t)Hv * KR_BYTES;
}

cudaError_t launch_kda_chunk_prefill(const LaunchEnv& env, const uint16_t* qkv, const float* g, float g_min,
                                     const float* beta, const int32_t* cu, int N, int T, int Hk, int Hv,
                                     float q_scale, float l2_eps, const float* state_in, float* state_out,
                                     const uint16_t* z, const uint16_t* norm_w, float rms_eps, uint16_t* out,
                                     void* workspace) {
  static int prep_set[64] = {0}, state_set[64] = {0};
  if (N <= 0) return cudaSuccess;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  unsigned* counter = reinterpret_cast<unsigned*>(ws);
  int32_t* order = reinterpret_cast<int32_t*>(ws + 256);
  int32_t* chunk_off = reinterpret_cast<int32_t*>(ws + 256 + kpad256((size_t)4 * N));
  uint8_t* rec = ws + 256 + kpad256((size_t)4 * N) + kpad256((size_t)4 * (N + 1));
  const long nc_max = kda_chunk_bound(N, T);

  KStateParams sp;
  memset(&sp, 0, sizeof sp);
  if (T > 0) {
    cudaError_t e = encode_chunk_tensor_maps(&sp.tmap, &sp.tmap_z, qkv, z, T, Hk, Hv);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_chunk_schedule(env.stream, cu, N, order, counter, chunk_off);
  if (e != cudaSuccess) return e;
  if ((e = kda_set_smem_once(kda_prep_kernel, KP_BYTES, prep_set)) != cudaSuccess) return e;
  if ((e = kda_set_smem_once(kda_state_kernel, SK_BYTES, state_set)) != cudaSuccess) return e;
  int sms = env.num_sms;
  if (sms <= 0 && (e = device_sm_count(&sms)) != cudaSuccess) return e;

  if (T > 0 && nc_max > 0) {
    KPrepParams pp;
    memset(&pp, 0, sizeof pp);
    if ((e = encode_chunk_tensor_maps(&pp.tmap_qkv, nullptr, qkv, nullptr, T, Hk, Hv)) != cudaSuccess) return e;
    if ((e = encode_f32_2d(&pp.tmap_g, g, (uint64_t)Hv * kHeadDim, (uint64_t)T, (uint64_t)Hv * kHeadDim * 4, 128, 64)) !=
        cudaSuccess)
      return e;
    pp.beta = beta; pp.cu = cu; pp.chunk_off = chunk_off; pp.rec = rec; pp.err = env.err;
    pp.N = N; pp.T = T; pp.Hk = Hk; pp.Hv = Hv; pp.nc_max = (int)nc_max;
    pp.g_min = g_min; pp.q_scale = q_scale; pp.l2_eps = l2_eps;
    const long units = nc_max * Hv;  // an upper bound: the device walks chunk_off[N] x Hv units
    kda_prep_kernel<<<(unsigned)std::min<long>(units, sms), kPrepThreads, KP_BYTES, env.stream>>>(pp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  sp.cu = cu; sp.order = order; sp.counter = counter; sp.chunk_off = chunk_off; sp.rec = rec;
  sp.state_in = state_in; sp.state_out = state_out; sp.z = z; sp.norm_w = norm_w; sp.out = out; sp.err = env.err;
  sp.N = N; sp.T = T; sp.Hk = Hk; sp.Hv = Hv; sp.nc_max = (int)nc_max; sp.rms_eps = rms_eps;
  const long items = (long)N * Hv;
  kda_state_kernel<<<(unsigned)std::min<long>(items, 2L * sms), kThreads, SK_BYTES, env.stream>>>(sp);
  return cudaGetLastError();
}

}  // namespace gdn
