// chunk_split.cu -- chunk-wise (WY) gated delta rule prefill as two kernels: a parallel prep
// kernel for everything that does not depend on the recurrent state, and a persistent state
// kernel that carries the state through the chunks of each (sequence, V head).
//
// The method: pegainfer PR #1152 "Reference golden for the GDN sublayer", Consumer / Shipped-line
// diff (prepare, cumsum, A, solve are per chunk; recompute, state, output follow the state
// chain) and Code review (f32 recurrent state carried across chunks).  The algebra is the one of
// the fused kernel (chunk_prefill.cu): for one chunk of L <= 64 tokens with start state S0,
//   A[t,j] = beta_t exp(gamma_t - gamma_j) k^_t.k^_j (j < t),  T = (I + A)^-1,
//   P[t,j] = q_scale iq_t exp(gamma_t - gamma_j) q_t.k^_j (j <= t),
//   E      = T (diag(beta) V - diag(beta Gamma) K^ S0^T),
//   O      = diag(Gamma iq q_scale) Q S0^T + P E,     S_L = Gamma_L S0 + E^T diag(exp(gamma_L - gamma)) K^.
// A, T, P and the per-token factors depend on q, k, g and beta only, so the prep kernel forms
// them for every chunk at once (one CTA per (chunk, K head): the Gram [K; Q] K^T of the K head
// on the tensor cores, then per V head of the group the scalings, the blocked solve and the
// bf16 operand images) and writes them to a per-(chunk, V head) record in the workspace.  The
// state kernel then runs only the state-dependent chain per chunk:
//   S0 -> bf16 hi/lo (two key halves)  ->  [X | O1] = S0 [K; Q]^T
//   R = diag(beta) V - diag(c_x) X^T   ->  E^T = R T^T               (R read from tensor memory)
//   E~ = E diag(c_s)                   ->  S = Gamma_L S0 + E~^T K  (E~ from tensor memory, K read
//                                          MN-major from the q/k tile), O2 = E P^T
//   o = O1 diag(c_o) + O2  ->  sigmoid-gated RMSNorm  ->  out
// with the records fetched by 1D bulk copies and q/k, v, z by TMA.  The state kernel uses 256 of
// the 512 tensor-memory columns and ~108 KB of shared memory, so two CTAs share an SM and one
// CTA's waits hide behind the other's work.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "chunk_common.cuh"
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

// ---- per-(chunk, V head) record in the workspace (bytes)
constexpr uint32_t REC_T = 0;          // T hi (8 KB) + T lo (8 KB): 64 x 64 bf16, K-major 128-byte swizzle
constexpr uint32_t REC_P = 16384;      // P (8 KB), same layout
constexpr uint32_t REC_VEC = 24576;    // 5 x 64 fp32: beta, -c_x, c_s, c_o, misc (misc[0] = Gamma_L)
constexpr uint32_t kRecTP = 24576;     // T and P: one bulk copy
constexpr uint32_t kRecVec = 5 * 64 * 4;
constexpr uint32_t REC_BYTES = REC_VEC + kRecVec;  // 25,856
static_assert(REC_BYTES % 128 == 0, "records must stay 16-byte aligned");
constexpr int V_BETA = 0, V_NCX = 64, V_CS = 128, V_CO = 192, V_MISC = 256;  // float offsets in the vector block

// ---- prep kernel shared memory: up to kGroup V heads of one K head are solved together
constexpr int kGroup = 3;
constexpr uint32_t PR_QK = 0;                                // 32 KB [K; Q] tile (TMA); dead once the Gram and
                                                             // the norms are taken, then it receives the next
                                                             // unit's tile
constexpr uint32_t PR_HEADS = 32768;
constexpr uint32_t PR_VEC = PR_HEADS + kGroup * kHeadBuf;    // gamma, beta (kGroup x 64 each), ik, iq, partial sums,
                                                             // gamma - log2 ik (kGroup x 64)
constexpr uint32_t PR_BAR = PR_VEC + (3 * kGroup * 64 + 2 * 64 + kParts * 128) * 4;
constexpr uint32_t PR_USED = PR_BAR + 64;
constexpr uint32_t PR_BYTES = PR_USED + 1024;
static_assert(2 * (PR_BYTES + 1024) <= 233472, "two prep CTAs must share an SM");
static_assert(kHeadBuf % 1024 == 0 && PR_HEADS % 1024 == 0, "head buffers stay 1 KB aligned");

// ---- state kernel shared memory
constexpr uint32_t SS_QK = 0;         // 32 KB [K; Q] tile (TMA)
constexpr uint32_t SS_W = 32768;      // 32 KB: S0 key-half hi/lo, then the output staging (o1 c_o, then + O2)
constexpr uint32_t SS_T = 65536;      // 16 KB T hi/lo (record), then E bf16
constexpr uint32_t SS_P = 81920;      //  8 KB P (record; follows T so one bulk copy fills both)
constexpr uint32_t SS_V = 90112;      // 16 KB V (TMA), then z of the chunk (TMA; gate input of the output stage)
constexpr uint32_t SS_VEC = 106496;   // 2 x per-token vector block (double buffered)
constexpr uint32_t SS_BAR = SS_VEC + 2 * kRecVec;
constexpr uint32_t SS_USED = SS_BAR + 128;
constexpr uint32_t SS_BYTES = SS_USED + 1024;
static_assert(2 * (SS_BYTES + 1024) <= 233472, "two state CTAs must share an SM");
static_assert(SS_P == SS_T + 16384, "T and P must be contiguous");

// ---- state kernel tensor memory columns
constexpr uint32_t SC_S = 0;      // 128: the recurrent state
constexpr uint32_t SC_X = 128;    //  64: S0 K^T, then R (bf16 hi/lo pairs: MMA operand), then E~ (likewise)
constexpr uint32_t SC_O1 = 192;   //  64: S0 Q^T, then E^T, then E P^T
constexpr uint32_t SC_COLS = 256;

// The chunks of sequence n (nch of them) are split into nseg contiguous segments; segment k holds
// chunk indices [k nch / nseg, (k + 1) nch / nseg).  The prep kernel of segment k + 1 runs beside
// the state kernel of segment k, so only the first segment's prep is exposed.  (Equal segments:
// a short first segment measured slower once the conv kernel runs before the call.)
constexpr int kMaxSegments = 4;
__host__ __device__ __forceinline__ int seg_begin(int k, int nch, int nseg) { return (int)(((long)k * nch) / nseg); }

// Parts: the chunks of a long sequence's segment are cut into P parts that run at once.  Part p
// starts from S_p = S_(p-1) Phi_(p-1) + L_(p-1) (S_0 the segment's start state), where L_q is
// part q's end state from a zero start and Phi_q its transition (the end state from the identity
// with v = 0; rows of the state evolve independently, so S_end = S_start Phi + L for any start).
// Split sequences go to their own launch of the state kernel (the parts instantiation, on a stream
// of its own beside the launch of the other sequences): L and Phi of parts 0 .. P - 2 (no outputs)
// come first in its work order; a part item waits (bounded) for their completion flags and then
// applies its p combine steps to the segment's start state (tensor cores, hi/lo operands).  The
// wait cannot deadlock: the items it waits for were taken earlier by CTAs that are running and
// wait for nothing.  A split sequence hands its state to the next segment through a slot of its
// own, so no part reads a state that another part has already replaced.
constexpr int kMaxParts = 4;          // parts per sequence and segment (measured best of 3, 4, 5 and 8)
constexpr int kMinPart = 8;           // chunks per part at least
constexpr int kMaxSplitSeqs = 8;      // split sequences per call
constexpr int kSlotCap = 32;          // [Hv][128][128] fp32 state slots per call (L, Phi, hand-off)
constexpr int kSplitMinTokens = 64 * kChunk;  // calls shorter than this never split (and get no slots)
constexpr uint32_t kFlagWaitLimit = 1u << 22;  // polls (about 256 ns apart) of a part's completion flag
__host__ __device__ __forceinline__ int part_begin(int p, int m, int P) { return (int)(((long)p * m) / P); }
// slot of (segment k, kind 0 = L / 1 = Phi / 2 = hand-off, part q) of a sequence split into P parts
__host__ __device__ __forceinline__ int part_slot(int base, int k, int P, int kind, int q) {
  return base + k * (2 * P - 1) + (kind == 2 ? 2 * (P - 1) : kind * (P - 1) + q);
}

#ifdef GDN_TEST_HOOKS
constexpr uint32_t kTestWaitLimit = 1u << 12;  // polls of a wait whose copy the hook dropped
__device__ unsigned g_test_drop_vec_copy;      // 1: an item's first vector-block copy is not issued
#endif

struct PrepParams {
  CUtensorMap tmap;  // qkv [T][C] bf16, box 64 x 64, 128-byte swizzle
  GateSrc gates;
  const int32_t* cu;
  const int32_t* chunk_off;
  const int32_t* seg_pref;  // this segment's exclusive prefix over sequences of their chunk counts [N + 1]
  uint8_t* rec;
  unsigned* err;
  int N, T, Hk, Hv, seg, nseg, nc_max;
  float q_scale, l2_eps;
};

struct StateParams {
  int seg, nseg;              // chunk segment processed by this launch
  const int2* items;          // parts launch: item_count[1] items (sequence, part | kind << 16) computing L /
  const int32_t* item_count;  //   Phi, then (sequence, part) items with outputs, item_count[0] in all;
                              //   main launch: item_count[0] sequences of `order` (NULL: N)
  int* flags;                 // [kSlotCap][Hv] completion flags of the L / Phi slots
  const int32_t* part_cnt;    // parts per sequence (NULL: 1)
  const int32_t* slot_base;   // first state slot of a split sequence
  float* slots;               // [kSlotCap][Hv][128][128]
  const float* state_src;     // state at the segment start: state_in (may be NULL) for the first, else state_out
  CUtensorMap tmap;
  CUtensorMap tmap_z;    // z [T][Hv * 128] bf16, box 128 x 64, no swizzle (valid when z != NULL)
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

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}

// q and k tiles of K head kh for the chunk starting at token c0: K rows 0..63, Q rows 64..127 of
// each 64-feature block (blocks 16 KB apart)
__device__ __forceinline__ void issue_qk_tiles(uint32_t dst, const CUtensorMap* tmap, int Hk, int c0, int kh,
                                               uint32_t bar) {
  mbar_arrive_expect_tx(bar, kBytesQK);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    tma_load_2d(dst + kb * 16384, tmap, Hk * kHeadDim + kh * kHeadDim + kb * 64, c0, bar);
    tma_load_2d(dst + kb * 16384 + 8192, tmap, kh * kHeadDim + kb * 64, c0, bar);
  }
}


// Persistent CTAs walk the (chunk, K head) units of one chunk segment.  Thread (row, part) owns
// Gram row `row` (rows 0..63: key t, the A side; rows 64..127: query t, the P side) and kW of its
// columns.  The V heads of the K head are processed kGroup at a time.
__global__ void __launch_bounds__(kThreads, 2) chunk_prep_kernel(const __grid_constant__ PrepParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, part = warp >> 2;
  const int row = q4 * 32 + lane;
  const int ratio = p.Hv / p.Hk;
  const long units = (long)__ldg(p.seg_pref + p.N) * p.Hk;
  if ((long)blockIdx.x >= units) return;  // uniform over the CTA

  float* s_gam = reinterpret_cast<float*>(sm + PR_VEC);  // [kGroup][64] cumsum of g, log2 units
  float* s_beta = s_gam + kGroup * 64;                    // [kGroup][64]
  float* s_ik = s_beta + kGroup * 64;
  float* s_iq = s_ik + 64;
  float* s_part = s_iq + 64;
  float* s_gk = s_part + kParts * 128;  // [kGroup][64] gamma_j - log2 ik_j: exp2(gamma_t - s_gk[j]) = decay ik_j
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + PR_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + PR_BAR + 32);
  const uint32_t bar_qk = smem_u32(&bars[0]), bar_g = smem_u32(&bars[1]);

  if (tid == 0) {
    mbar_init(bar_qk, 1);
    mbar_init(bar_g, 1);
    fence_mbar_init();
    prefetch_tensormap(&p.tmap);
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);

  // A unit's chunk: its sequence (the last n with seg_pref[n] <= unit / Hk: never one without
  // chunks here), first token, length and record index; false when cu_seqlens is inconsistent.
  struct Unit {
    int kh, c0, L, gc;
  };
  auto unit_of = [&](long u, Unit& un) {
    const int cu_ = (int)(u / p.Hk);
    un.kh = (int)(u - (long)cu_ * p.Hk);
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.seg_pref + mid) <= cu_) lo = mid; else hi = mid - 1;
    }
    const int n = lo;
    const int seq_s = __ldg(p.cu + n), seq_e = __ldg(p.cu + n + 1);
    const int nch = (max(0, seq_e - seq_s) + kChunk - 1) / kChunk;
    const int j = seg_begin(p.seg, nch, p.nseg) + (cu_ - __ldg(p.seg_pref + n));
    un.gc = __ldg(p.chunk_off + n) + j;
    un.c0 = seq_s + j * kChunk;
    un.L = min(kChunk, seq_e - un.c0);
    return !(seq_s < 0 || seq_e < seq_s || seq_e > p.T || un.c0 >= seq_e || un.gc < 0 || un.gc >= p.nc_max);
  };
  // g, beta of a group of V heads of a unit: thread -> (token tid / G, head tid % G), zero past the
  // sequence end
  float g_next = 0.f, b_next = 0.f;
  auto load_gb = [&](const Unit& un, int h0, int G) {
    g_next = 0.f;
    b_next = 0.f;
    const int t = tid / G;
    if (tid < 64 * G && t < un.L) {
      const int hh = h0 + (tid - t * G);
      load_gate(p.gates, (size_t)(un.c0 + t) * p.Hv + hh, hh, g_next, b_next);
    }
  };

  // The [K; Q] tile of a unit is dead once its Gram and norms are taken: the next unit's tile is
  // fetched into the same buffer from there, and the next unit's first g / beta once the current
  // unit's last group has taken its own, so both arrive while the current unit is solved.
  bool ok = true, qk_pending = false, gram_pending = false, have_next = false;
  uint32_t ph_qk = 0, ph_g = 0;  // parities: bar_qk completes once per tile, bar_g once per Gram
  for (long u = blockIdx.x; u < units && ok; u += gridDim.x) {
  Unit un;
  if (!unit_of(u, un)) {  // never prefetched (the prefetch checks the same condition)
    if (tid == 0) raise_error(p.err, kErrDeviceArgument);
    have_next = false;
    continue;
  }
  const int kh = un.kh, gc = un.gc, c0 = un.c0, L = un.L;
  if (!have_next) {
    if (tid == 0) issue_qk_tiles(sb + PR_QK, &p.tmap, p.Hk, c0, kh, bar_qk);
    load_gb(un, kh * ratio, min(kGroup, ratio));
  }
  qk_pending = true;
  have_next = false;
  Unit nx;
  const long u_next = u + gridDim.x;
  const bool next_ok = u_next < units && unit_of(u_next, nx);

  {
    const bool got = mbar_wait(bar_qk, ph_qk, kWaitLimit);
    if (got) ph_qk ^= 1u;  // after a timeout ph_qk stays the parity of the copy still in flight
    if (!got) raise_error(p.err, kErrTimeout);
    ok = __syncthreads_and(got ? 1 : 0) != 0;
    qk_pending = !ok;
  }
  if (ok) {
    // Gram G = [K; Q] K^T (M = 128, N = 64, K = 128) on the raw bf16 tiles
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        mma_bf16(tmem, sw128_desc(sb + PR_QK + off), sw128_desc(sb + PR_QK + off), idesc_bf16_f32(128, 64), ks > 0);
      }
      mma_commit(bar_g);
    }
    gram_pending = true;
    // L2-norm factors: rows 0..63 keys, 64..127 queries; each part sums 64 of the 128 features
    {
      const int r = tid & 127, kq = tid >> 7;
      float ss = 0.f;
#pragma unroll
      for (int cc = 0; cc < 16 / kParts; ++cc) {
        const int chunk = kq * (16 / kParts) + cc, kb = chunk >> 3, c = chunk & 7;
        const uint4 u = *reinterpret_cast<const uint4*>(sm + PR_QK + kb * 16384 + r * 128 + (((c ^ (r & 7)) & 7) << 4));
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = __uint_as_float(w4[e] << 16), b = __uint_as_float(w4[e] & 0xFFFF0000u);
          ss = fmaf(a, a, ss);
          ss = fmaf(b, b, ss);
        }
      }
      s_part[kq * 128 + r] = ss;
    }
    __syncthreads();
    if (tid < 128) {
      float ss = 0.f;
#pragma unroll
      for (int q = 0; q < kParts; ++q) ss += s_part[q * 128 + tid];
      const float inv = 1.0f / sqrtf(ss + p.l2_eps);
      if (tid < 64) s_ik[tid] = inv; else s_iq[tid - 64] = inv;
    }
    fence_proxy_async_smem();  // this thread's generic reads of the tile (the norms) before its refill
    const bool got = mbar_wait(bar_g, ph_g, kWaitLimit);
    if (got) ph_g ^= 1u;
    if (!got) raise_error(p.err, kErrTimeout);
    ok = __syncthreads_and(got ? 1 : 0) != 0;  // also: the q/k tile is dead from here on
    gram_pending = !ok;
    tc_fence_after();
    if (ok && next_ok) {  // the next unit's tile into the freed buffer
      if (tid == 0) issue_qk_tiles(sb + PR_QK, &p.tmap, p.Hk, nx.c0, nx.kh, bar_qk);
      qk_pending = true;
      have_next = true;
    }
  }
  if (ok) {
    for (int g0 = 0; g0 < ratio; g0 += kGroup) {
      const int G = min(kGroup, ratio - g0), h0 = kh * ratio + g0;
      if (tid < 64 * G) {
        const int t = tid / G, g = tid - t * G;
        s_gam[g * 64 + t] = g_next * kLog2e;
        s_beta[g * 64 + t] = b_next;
      }
      __syncthreads();
      if (warp < G) {  // inclusive scan of g over the chunk (lane l holds tokens 2l, 2l + 1)
        float* gam = s_gam + warp * 64;
        const float g0v = gam[2 * lane], g1v = gam[2 * lane + 1];
        float sc = g0v + g1v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float v = __shfl_up_sync(0xffffffffu, sc, o);
          if (lane >= o) sc += v;
        }
        gam[2 * lane + 1] = sc;
        gam[2 * lane] = sc - g1v;
      }
      __syncthreads();
      if (g0 + kGroup < ratio) load_gb(un, h0 + kGroup, min(kGroup, ratio - g0 - kGroup));  // in flight meanwhile
      else if (have_next) load_gb(nx, nx.kh * ratio, min(kGroup, ratio));  // the next unit's first group
      if (tid < 64 * G) {  // per-token factors of the G heads
        const int g = tid >> 6, t = tid & 63;
        const float* gam = s_gam + g * 64;
        const float gt = gam[t], gL = gam[L - 1];
        const float Gam = ex2_approx(gt), bt = s_beta[g * 64 + t];
        float* vec = reinterpret_cast<float*>(p.rec + ((size_t)gc * p.Hv + h0 + g) * REC_BYTES + REC_VEC);
        vec[V_BETA + t] = bt;
        vec[V_NCX + t] = -(bt * Gam * s_ik[t]);
        vec[V_CS + t] = (t < L) ? ex2_approx(gL - gt) * s_ik[t] : 0.f;
        vec[V_CO + t] = Gam * s_iq[t] * p.q_scale;
        vec[V_MISC + t] = (t == 0) ? ex2_approx(gL) : 0.f;
        s_gk[g * 64 + t] = gt - lg2_approx(s_ik[t]);
      }
      __syncthreads();
      // A (rows 0..63, blocks on and below the diagonal) and P (rows 64..127, straight to the record);
      // the warps whose 32 rows and 32 columns all lie above the diagonal (token j > t) have no work
      float gr[kW];  // raw Gram row `row`, columns part * kW ..
      tmem_ld_cols<kW>(tl + part * kW, gr);
      const bool all_masked = part == 1 && (q4 & 1) == 0;
      if (all_masked && row >= 64) {  // P is zero there (A's blocks above the diagonal are never read)
        const float zero8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int g = 0; g < G; ++g) {
          uint8_t* rec = p.rec + ((size_t)gc * p.Hv + h0 + g) * REC_BYTES;
#pragma unroll
          for (int i0 = 0; i0 < kW; i0 += 8) store8_split(rec + REC_P, nullptr, 0, row - 64, part * kW + i0, zero8);
        }
      }
      for (int g = 0; g < G && !all_masked; ++g) {
        // a pair of columns j, j + 1: scale * gram * exp2(gamma_t - gk_j), with gk_j = gamma_j - log2 ik_j
        const float* gk = s_gk + g * 64;
        const int t = row & 63;
        const float gt = s_gam[g * 64 + t];
        const float scale = row < 64 ? s_beta[g * 64 + t] * s_ik[t] : s_iq[t] * p.q_scale;
        const float2 gt2 = make_float2(gt, gt), neg1 = make_float2(-1.f, -1.f);
        auto pair = [&](int j, int i) {  // columns j, j + 1 (this thread's gram entries i, i + 1)
          const float2 d = __ffma2_rn(*reinterpret_cast<const float2*>(gk + j), neg1, gt2);
          return __fmul2_rn(__fmul2_rn(make_float2(gr[i], gr[i + 1]), make_float2(scale, scale)),
                            make_float2(ex2_approx(d.x), ex2_approx(d.y)));
        };
        if (row < 64) {
          // row t of A, blocks (t / 16, 2 part) and (t / 16, 2 part + 1) of the tri layout
          float* sA = reinterpret_cast<float*>(sm + PR_HEADS + g * kHeadBuf);
          const int tb = t >> 4, tx = t & 3;
          float* rowA = sA + ((tb * (tb + 1)) / 2 + 2 * part) * 256 + (t & 15) * 16;
#pragma unroll
          for (int i4 = 0; i4 < kW; i4 += 4) {
            const int j0 = part * kW + i4;
            if ((j0 >> 4) > tb) continue;  // above the diagonal blocks: never read
            const float2 a01 = pair(j0, i4), a23 = pair(j0 + 2, i4 + 2);
            *reinterpret_cast<float4*>(rowA + (i4 >> 4) * 256 + ((((i4 & 15) >> 2) ^ tx) << 2)) =
                make_float4(j0 < t ? a01.x : 0.f, j0 + 1 < t ? a01.y : 0.f, j0 + 2 < t ? a23.x : 0.f,
                            j0 + 3 < t ? a23.y : 0.f);
          }
        } else {
          uint8_t* rec = p.rec + ((size_t)gc * p.Hv + h0 + g) * REC_BYTES;
#pragma unroll
          for (int i0 = 0; i0 < kW; i0 += 8) {
            const int j0 = part * kW + i0;
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; u += 2) {
              const float2 a = pair(j0 + u, i0 + u);
              v[u] = j0 + u <= t ? a.x : 0.f;
              v[u + 1] = j0 + u + 1 <= t ? a.y : 0.f;
            }
            store8_split(rec + REC_P, nullptr, 0, t, j0, v);
          }
        }
      }
      __syncthreads();
      solve_tri_batched(sm + PR_HEADS, G, tid);
      for (int i = tid; i < 64 * 8 * G; i += kThreads) {
        const int g = i >> 9, t = (i >> 3) & 63, k0 = (i & 7) * 8;
        const float* sT = reinterpret_cast<const float*>(sm + PR_HEADS + g * kHeadBuf + kTriBytes);
        uint8_t* rec = p.rec + ((size_t)gc * p.Hv + h0 + g) * REC_BYTES;
        const int tb = t >> 4, kb = k0 >> 4;
        const bool upper = kb > tb;  // strictly upper blocks of T are zero
        const float* rowT = sT + ((tb * (tb + 1)) / 2 + kb) * 256 + (t & 15) * 16;
        const int q0 = (k0 & 15) >> 2, tx = t & 3;
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 v0 = upper ? z4 : *reinterpret_cast<const float4*>(rowT + ((q0 ^ tx) << 2));
        const float4 v1 = upper ? z4 : *reinterpret_cast<const float4*>(rowT + (((q0 + 1) ^ tx) << 2));
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        store8_split(rec + REC_T, rec + REC_T + 8192, 0, t, k0, v);
      }
      __syncthreads();  // T reads done before the next group's A writes
    }
  }
  // the unit's reads of the shared buffers precede the next unit's tile load into them
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  }
  // leave only after the Gram MMA and the tile load have landed (bounded, after an early exit)
  if (qk_pending) mbar_wait(bar_qk, ph_qk, kWaitLimit);
  if (gram_pending) mbar_wait(bar_g, ph_g, kWaitLimit);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// Persistent; pulls (sequence, V head) items in longest-first order (split sequences are left to
// chunk_part_state_kernel).  Thread (row, part) owns tensor-memory lane `row` (a value row of the
// state) and kW of the 64 columns of every token-indexed accumulator.
__global__ void __launch_bounds__(kThreads, 2) chunk_state_kernel(const __grid_constant__ StateParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, part = warp >> 2;
  const int row = q4 * 32 + lane;
  const int ratio = p.Hv / p.Hk;
  const long total_items = (long)p.N * p.Hv;

  float* s_work = reinterpret_cast<float*>(sm + SS_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SS_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SS_BAR + 96);
  int* item_slot = reinterpret_cast<int*>(sm + SS_BAR + 104);
  const uint32_t bar_qk = smem_u32(&bars[0]), bar_v = smem_u32(&bars[1]), bar_tp = smem_u32(&bars[2]),
                 bar_h = smem_u32(&bars[3]), bar_x = smem_u32(&bars[4]), bar_e = smem_u32(&bars[5]),
                 bar_s = smem_u32(&bars[6]), bar_z = smem_u32(&bars[7]);
  const uint32_t bar_vec0 = smem_u32(&bars[8]);  // one barrier per vector buffer: bar_vec0 + 8 * buffer

  if (tid == 0) {
    for (int i = 0; i < 10; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
    prefetch_tensormap(&p.tmap);
    if (p.z) prefetch_tensormap(&p.tmap_z);
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), SC_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);

  constexpr uint32_t ID64 = idesc_bf16_f32(128, 64);
  constexpr uint32_t ID128 = idesc_bf16_f32(128, 128);
  constexpr uint32_t ID128_BMN = idesc_bf16_f32_bmn(128, 128);
  bool ok = true;
  uint32_t ph_mma = 0, ph_qk = 0, ph_v = 0, ph_tp = 0, ph_z = 0;
  uint32_t ph_vec = 0, pend_vec = 0;  // bit b: parity of / load in flight on vector buffer b
  bool pend_qk = false, pend_v = false, pend_tp = false, pend_z = false;
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
      tma_load_2d(sb + SS_V + kb * 8192, &p.tmap, 2 * p.Hk * kHeadDim + h * kHeadDim + kb * 64, c0, bar_v);
  };
  auto issue_z = [&](int c0, int h) {  // into the V buffer, once R has consumed V
    mbar_arrive_expect_tx(bar_z, kBytesZ);
    tma_load_2d(sb + SS_V, &p.tmap_z, h * kHeadDim, c0, bar_z);
  };
  // a chunk's record: T and P (needed from the E MMA on), and its vector block (needed at chunk
  // start; double buffered, so it is fetched a whole chunk ahead)
  auto issue_tp = [&](int gc, int h) {
    const uint8_t* rec = p.rec + ((size_t)gc * p.Hv + h) * REC_BYTES;
    mbar_arrive_expect_tx(bar_tp, kRecTP);
    bulk_load(sb + SS_T, rec + REC_T, kRecTP, bar_tp);
  };
  auto issue_vec = [&](int gc, int h, int vb, bool first = false) {
    const uint8_t* rec = p.rec + ((size_t)gc * p.Hv + h) * REC_BYTES;
    mbar_arrive_expect_tx(bar_vec0 + 8 * vb, kRecVec);
#ifdef GDN_TEST_HOOKS
    if (first && g_test_drop_vec_copy) return;
#endif
    (void)first;
    bulk_load(sb + SS_VEC + vb * kRecVec, rec + REC_VEC, kRecVec, bar_vec0 + 8 * vb);
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
  // S0 columns [k0, k0 + 64) -> hi/lo operand tiles (64 keys = one K block); state <- Gamma_L S0 there
  auto convert_half = [&](int k0, float gL) {
    float v[kW];
    tmem_ld_cols<kW>(tl + SC_S + k0 + part * kW, v);
#pragma unroll
    for (int q = 0; q < kW / 8; ++q) store8_split(sm + SS_W, sm + SS_W + 16384, 0, row, part * kW + 8 * q, v + 8 * q);
#pragma unroll
    for (int i = 0; i < kW; i += 2) {
      const float2 m = __fmul2_rn(make_float2(v[i], v[i + 1]), make_float2(gL, gL));
      v[i] = m.x;
      v[i + 1] = m.y;
    }
    tmem_st32(tl + SC_S + k0 + part * kW, v);
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
    if (p.part_cnt && p.part_cnt[n] > 1) continue;  // a split sequence: the parts launch computes it
    const int kh = h / ratio;
    const int seq_lo = __ldg(p.cu + n), seq_hi = __ldg(p.cu + n + 1);
    const int nch = (max(0, seq_hi - seq_lo) + kChunk - 1) / kChunk;
    const int jb = seg_begin(p.seg, nch, p.nseg), je = seg_begin(p.seg + 1, nch, p.nseg);
    if (p.seg > 0 && jb == je) continue;  // no chunk in this segment: the state is already in state_out
    // this launch's part of the sequence: chunks [jb, je)
    const int seq_s = seq_lo + jb * kChunk, seq_e = min(seq_hi, seq_lo + je * kChunk);
    const int gc0 = __ldg(p.chunk_off + n) + jb;
    if (n < 0 || n >= p.N || seq_lo < 0 || seq_hi < seq_lo || seq_hi > p.T || gc0 < 0 ||
        gc0 + (je - jb) > p.nc_max) {
      if (tid == 0) raise_error(p.err, kErrDeviceArgument);
      continue;
    }
    if (tid == 0 && seq_e > seq_s) {
      issue_vec(gc0, h, 0, true);
      issue_qk_tiles(sb + SS_QK, &p.tmap, p.Hk, seq_s, kh, bar_qk);
      issue_v(seq_s, h);
      issue_tp(gc0, h);
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
        if (p.state_src) {
          const float4* src = reinterpret_cast<const float4*>(p.state_src + row_off + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 f = __ldg(src + i);
            v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        tmem_st32(tl + SC_S + c0, v);
      }
    }

    int vb = 0;
    for (int c0 = seq_s, gc = gc0; c0 < seq_e && ok; c0 += kChunk, ++gc, ph_mma ^= 1u, vb ^= 1) {
      const int L = min(kChunk, seq_e - c0);
      const bool has_next = c0 + kChunk < seq_e;
      const float* vec = reinterpret_cast<const float*>(sm + SS_VEC + vb * kRecVec);

      {
#ifdef GDN_TEST_HOOKS
        const uint32_t vec_limit = g_test_drop_vec_copy ? kTestWaitLimit : kWaitLimit;
#else
        const uint32_t vec_limit = kWaitLimit;
#endif
        const bool got = mbar_wait(bar_vec0 + 8 * vb, (ph_vec >> vb) & 1u, vec_limit);
        ph_vec ^= 1u << vb;
        pend_vec &= ~(1u << vb);
        if (!got) raise_error(p.err, kErrTimeout);
        ok = __syncthreads_and(got ? 1 : 0) != 0 && ok;
      }
      if (!ok) break;
      const float gL = vec[V_MISC];


      // ================= [X | O1] = S0 [K; Q]^T one 64-key half at a time: X from the hi and lo
      // parts of S0, the output-only O1 from the hi part
      convert_half(0, gL);
      fence_proxy_async_smem();
      tc_fence_before();
      wait_bar(bar_qk, ph_qk);  // the q/k tile (its latency overlaps the conversion above)
      pend_qk = false;
      tc_fence_after();
      if (!ok) break;
      if (tid == 0) {
        mma_bf16_k4<2, 2>(tmem + SC_X, sw128_desc(sb + SS_W), sw128_desc(sb + SS_QK), ID128, 0);
        mma_bf16_k4<2, 2>(tmem + SC_X, sw128_desc(sb + SS_W + 16384), sw128_desc(sb + SS_QK), ID64, 1);
        mma_commit(bar_h);
      }
      await_mma(bar_h);
      if (!ok) break;
      convert_half(64, gL);
      operands_ready();
      if (tid == 0) {
        mma_bf16_k4<2, 2>(tmem + SC_X, sw128_desc(sb + SS_W), sw128_desc(sb + SS_QK + 16384), ID128, 1);
        mma_bf16_k4<2, 2>(tmem + SC_X, sw128_desc(sb + SS_W + 16384), sw128_desc(sb + SS_QK + 16384), ID64, 1);
        mma_commit(bar_x);
      }
      {
        uint32_t ph = ph_mma;
        wait_two(bar_x, ph, bar_v, ph_v);
        tc_fence_after();
      }
      pend_v = false;
      if (!ok) break;

      // ================= R = diag(beta) V - diag(c_x) X^T -> hi/lo (value-major)
      {
        float x[kW];
        tmem_ld_cols<kW>(tl + SC_X + part * kW, x);
        // V[t][row] for t = part * kW + i: the swizzle term depends on i & 7 only
        const uint8_t* vbase = sm + SS_V + (row >> 6) * 8192 + part * kW * 128 + ((row & 7) << 1);
        const int rsw = (row >> 3) & 7;
        auto v_at = [&](int i) {
          return bf2f(*reinterpret_cast<const uint16_t*>(vbase + i * 128 + ((rsw ^ (i & 7)) << 4)));
        };
#pragma unroll
        for (int i4 = 0; i4 < kW; i4 += 4) {
          const float4 bt = *reinterpret_cast<const float4*>(vec + V_BETA + part * kW + i4);
          const float4 nc = *reinterpret_cast<const float4*>(vec + V_NCX + part * kW + i4);
          const float2 r0 = __ffma2_rn(make_float2(nc.x, nc.y), make_float2(x[i4], x[i4 + 1]),
                                       __fmul2_rn(make_float2(bt.x, bt.y), make_float2(v_at(i4), v_at(i4 + 1))));
          const float2 r1 = __ffma2_rn(make_float2(nc.z, nc.w), make_float2(x[i4 + 2], x[i4 + 3]),
                                       __fmul2_rn(make_float2(bt.z, bt.w), make_float2(v_at(i4 + 2), v_at(i4 + 3))));
          x[i4] = r0.x; x[i4 + 1] = r0.y; x[i4 + 2] = r1.x; x[i4 + 3] = r1.y;
        }
        store_split_tmem(tl + SC_X + part * kW, x);  // over this thread's own X columns
      }
      // O1 leaves its columns (they take E next): into registers now, staged while the E MMAs run
      float o1[kW];
      tmem_ld_cols<kW>(tl + SC_O1 + part * kW, o1);
      fence_proxy_async_smem();
      tc_fence_before();
      wait_bar(bar_tp, ph_tp);  // T and P of this chunk
      pend_tp = false;
      tc_fence_after();
      if (!ok) break;
      if (tid == 0) {
        // E^T = R T^T  (hi*hi + hi*lo + lo*hi), R from tensor memory (hi / lo pairs of 32 tokens per
        // thread part: hi at columns 32 p, lo at 32 p + 16 of the X region)
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<2>(tmem + SC_O1, tmem + SC_X + 32 * pp, sw128_desc(sb + SS_T) + 4 * pp, ID64, pp);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<2>(tmem + SC_O1, tmem + SC_X + 32 * pp, sw128_desc(sb + SS_T + 8192) + 4 * pp, ID64, 1);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<2>(tmem + SC_O1, tmem + SC_X + 32 * pp + 16, sw128_desc(sb + SS_T) + 4 * pp, ID64, 1);
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
        const float4 co = *reinterpret_cast<const float4*>(vec + V_CO + t0);
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
        tmem_ld_cols<kW>(tl + SC_O1 + part * kW, ev);
#pragma unroll
        for (int q = 0; q < kW / 8; ++q) {
          const float4 c0v = *reinterpret_cast<const float4*>(vec + V_CS + part * kW + 8 * q);
          const float4 c1v = *reinterpret_cast<const float4*>(vec + V_CS + part * kW + 8 * q + 4);
          const float* e8 = ev + 8 * q;
          const float2 p0 = __fmul2_rn(make_float2(e8[0], e8[1]), make_float2(c0v.x, c0v.y));
          const float2 p1 = __fmul2_rn(make_float2(e8[2], e8[3]), make_float2(c0v.z, c0v.w));
          const float2 p2 = __fmul2_rn(make_float2(e8[4], e8[5]), make_float2(c1v.x, c1v.y));
          const float2 p3 = __fmul2_rn(make_float2(e8[6], e8[7]), make_float2(c1v.z, c1v.w));
          float* s8 = es + 8 * q;
          s8[0] = p0.x; s8[1] = p0.y; s8[2] = p1.x; s8[3] = p1.y; s8[4] = p2.x; s8[5] = p2.y; s8[6] = p3.x; s8[7] = p3.y;
          store8_split(sm + SS_T, nullptr, 0, row, part * kW + 8 * q, e8);
        }
        store_split_tmem(tl + SC_X + part * kW, es);
      }
      operands_ready();
      if (tid == 0) {
        // S += E~ K: B = the raw k rows of the q/k tile read MN-major (N = 128 keys, 16 tokens per step)
        // (E~ from tensor memory as R was), O2 = E P^T into the E columns
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<128>(tmem + SC_S, tmem + SC_X + 32 * pp, sw128_mn_desc(sb + SS_QK, 16384) + 256 * pp,
                              ID128_BMN, 1);
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
          mma_bf16_k2_ta<128>(tmem + SC_S, tmem + SC_X + 32 * pp + 16, sw128_mn_desc(sb + SS_QK, 16384) + 256 * pp,
                              ID128_BMN, 1);
        mma_bf16_k4<2, 2>(tmem + SC_O1, sw128_desc(sb + SS_T), sw128_desc(sb + SS_P), ID64, 0);
        mma_commit(bar_s);
      }
      constexpr int kTok = kChunk / kWarps;
      await_mma(bar_s);
      if (!ok) break;
      if (has_next) {  // two issuing threads in different warps, so neither lags by both
        if (tid == 0) issue_qk_tiles(sb + SS_QK, &p.tmap, p.Hk, c0 + kChunk, kh, bar_qk);
        else if (tid == 32) issue_tp(gc + 1, h);
      }
      pend_qk = pend_tp = has_next;

      // ================= output: o = O1 diag(c_o) (staged) + O2, then the gated RMSNorm
      {
        float o2a[16], o2b[16];
        tmem_ld16x2(tl + SC_O1 + part * kW, tl + SC_O1 + part * kW + 16, o2a, o2b);
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
            const uint2 zz = *reinterpret_cast<const uint2*>(sm + SS_V + (warp + kWarps * i) * 256 + lane * 8);
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
        tmem_ld32(tl + SC_S + c0, v);
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
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, SC_COLS);
  }
}

template <bool B>
struct BoolC {
  static constexpr bool value = B;
};

// The state kernel of the split sequences' parts (items from plan_parts): L and Phi items
// (no outputs), then the parts, each starting from its combined state.  The same chain as
// chunk_state_kernel, compiled once with and once without the output stage.
__global__ void __launch_bounds__(kThreads, 2) chunk_part_state_kernel(const __grid_constant__ StateParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, part = warp >> 2;
  const int row = q4 * 32 + lane;
  const int ratio = p.Hv / p.Hk;
  const long total_items = (long)p.item_count[0] * p.Hv;
  if (total_items == 0) return;  // nothing is split

  float* s_work = reinterpret_cast<float*>(sm + SS_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SS_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SS_BAR + 96);
  int* item_slot = reinterpret_cast<int*>(sm + SS_BAR + 104);
  const uint32_t bar_qk = smem_u32(&bars[0]), bar_v = smem_u32(&bars[1]), bar_tp = smem_u32(&bars[2]),
                 bar_h = smem_u32(&bars[3]), bar_x = smem_u32(&bars[4]), bar_e = smem_u32(&bars[5]),
                 bar_s = smem_u32(&bars[6]), bar_z = smem_u32(&bars[7]);
  const uint32_t bar_vec0 = smem_u32(&bars[8]);  // one barrier per vector buffer: bar_vec0 + 8 * buffer

  if (tid == 0) {
    for (int i = 0; i < 10; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
    prefetch_tensormap(&p.tmap);
    if (p.z) prefetch_tensormap(&p.tmap_z);
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), SC_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);

  constexpr uint32_t ID64 = idesc_bf16_f32(128, 64);
  constexpr uint32_t ID128 = idesc_bf16_f32(128, 128);
  constexpr uint32_t ID128_BMN = idesc_bf16_f32_bmn(128, 128);
  bool ok = true;
  uint32_t ph_mma = 0, ph_qk = 0, ph_v = 0, ph_tp = 0, ph_z = 0;
  uint32_t ph_vec = 0, pend_vec = 0;  // bit b: parity of / load in flight on vector buffer b
  bool pend_qk = false, pend_v = false, pend_tp = false, pend_z = false;
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
      tma_load_2d(sb + SS_V + kb * 8192, &p.tmap, 2 * p.Hk * kHeadDim + h * kHeadDim + kb * 64, c0, bar_v);
  };
  auto issue_z = [&](int c0, int h) {  // into the V buffer, once R has consumed V
    mbar_arrive_expect_tx(bar_z, kBytesZ);
    tma_load_2d(sb + SS_V, &p.tmap_z, h * kHeadDim, c0, bar_z);
  };
  // a chunk's record: T and P (needed from the E MMA on), and its vector block (needed at chunk
  // start; double buffered, so it is fetched a whole chunk ahead)
  auto issue_tp = [&](int gc, int h) {
    const uint8_t* rec = p.rec + ((size_t)gc * p.Hv + h) * REC_BYTES;
    mbar_arrive_expect_tx(bar_tp, kRecTP);
    bulk_load(sb + SS_T, rec + REC_T, kRecTP, bar_tp);
  };
  auto issue_vec = [&](int gc, int h, int vb, bool first = false) {
    const uint8_t* rec = p.rec + ((size_t)gc * p.Hv + h) * REC_BYTES;
    mbar_arrive_expect_tx(bar_vec0 + 8 * vb, kRecVec);
#ifdef GDN_TEST_HOOKS
    if (first && g_test_drop_vec_copy) return;
#endif
    (void)first;
    bulk_load(sb + SS_VEC + vb * kRecVec, rec + REC_VEC, kRecVec, bar_vec0 + 8 * vb);
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
  // S0 columns [k0, k0 + 64) -> hi/lo operand tiles (64 keys = one K block); state <- Gamma_L S0 there
  auto convert_half = [&](int k0, float gL) {
    float v[kW];
    tmem_ld_cols<kW>(tl + SC_S + k0 + part * kW, v);
#pragma unroll
    for (int q = 0; q < kW / 8; ++q) store8_split(sm + SS_W, sm + SS_W + 16384, 0, row, part * kW + 8 * q, v + 8 * q);
#pragma unroll
    for (int i = 0; i < kW; i += 2) {
      const float2 m = __fmul2_rn(make_float2(v[i], v[i + 1]), make_float2(gL, gL));
      v[i] = m.x;
      v[i + 1] = m.y;
    }
    tmem_st32(tl + SC_S + k0 + part * kW, v);
  };
  // One combine step of a part's start state, S <- S Phi + L (fp32 state in tensor memory; Phi, L
  // [128][128] fp32 in global memory): the sum accumulates in the X / O1 columns (set to L first),
  // 64 rows of Phi at a time with hi/lo operands -- S through the S0 buffer (as for X), Phi
  // MN-major through the q/k buffer (two 64-column blocks 8 KB apart, hi then lo) -- and then
  // replaces S.
  auto combine = [&](const float* Lb, const float* Pb) {
    const float* lrow = Lb + (size_t)row * kHeadDim + part * 64;
#pragma unroll
    for (int cq = 0; cq < 2; ++cq) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(lrow + cq * 32) + i);
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
      }
      tmem_st32(tl + SC_X + part * 64 + cq * 32, v);
    }
    uint32_t ph = ph_mma;
    for (int kh2 = 0; kh2 < 2; ++kh2) {
      convert_half(64 * kh2, 1.f);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int idx = tid + kThreads * g, r = idx >> 4, k0 = (idx & 15) * 8;
        const float4* s4 = reinterpret_cast<const float4*>(Pb + (size_t)(64 * kh2 + r) * kHeadDim + k0);
        const float4 a = __ldcg(s4), b = __ldcg(s4 + 1);
        const float v8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        store8_split(sm + SS_QK, sm + SS_QK + 16384, 8192, r, k0, v8);
      }
      operands_ready();
      if (tid == 0) {
        mma_bf16_k4<2, 128>(tmem + SC_X, sw128_desc(sb + SS_W), sw128_mn_desc(sb + SS_QK, 8192), ID128_BMN, 1);
        mma_bf16_k4<2, 128>(tmem + SC_X, sw128_desc(sb + SS_W), sw128_mn_desc(sb + SS_QK + 16384, 8192), ID128_BMN, 1);
        mma_bf16_k4<2, 128>(tmem + SC_X, sw128_desc(sb + SS_W + 16384), sw128_mn_desc(sb + SS_QK, 8192), ID128_BMN, 1);
        mma_commit(bar_h);
      }
      wait_bar(bar_h, ph);
      tc_fence_after();
      if (!ok) return;
    }
#pragma unroll
    for (int cq = 0; cq < 2; ++cq) {
      float v[32];
      tmem_ld32(tl + SC_X + part * 64 + cq * 32, v);
      tmem_st32(tl + SC_S + part * 64 + cq * 32, v);
    }
    fence_proxy_async_smem();  // the operand buffers' reads and writes precede later copies into them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };

  // work item w -> (sequence, part, kind); the V head is w % Hv
  auto decode = [&](long w, int& n, int& q, int& kind) {
    const int ii = (int)(w / p.Hv);
    const int2 it = p.items[ii];
    n = it.x;
    q = it.y & 0xFFFF;
    kind = ii < p.item_count[1] ? 1 + (it.y >> 16) : 0;
  };
  for (;;) {
    if (tid == 0) *item_slot = (int)atomicAdd(p.counter, 1u);
    __syncthreads();
    const long w = *item_slot;
    __syncthreads();
    if (w >= total_items || !ok) break;
    const int h = (int)(w % p.Hv);
    int n, q, kind;  // kind 0: an item with outputs; 1: L of part q; 2: Phi of part q (auxiliary)
    decode(w, n, q, kind);
    if (n < 0 || n >= p.N) {
      if (tid == 0) raise_error(p.err, kErrDeviceArgument);
      continue;
    }
    const int P = p.part_cnt[n];
    const int kh = h / ratio;
    const int seq_lo = __ldg(p.cu + n), seq_hi = __ldg(p.cu + n + 1);
    const int nch = (max(0, seq_hi - seq_lo) + kChunk - 1) / kChunk;
    const int sg0 = seg_begin(p.seg, nch, p.nseg), sg1 = seg_begin(p.seg + 1, nch, p.nseg);
    const int jb = sg0 + part_begin(q, sg1 - sg0, P), je = sg0 + part_begin(q + 1, sg1 - sg0, P);
    if (p.seg > 0 && jb == je && P == 1) continue;  // no chunk in this segment: the state is already in state_out
    // this item's chunks of the sequence: [jb, je)
    const int seq_s = seq_lo + jb * kChunk, seq_e = min(seq_hi, seq_lo + je * kChunk);
    const int gc0 = __ldg(p.chunk_off + n) + jb;
    if (P < 1 || P > kMaxParts || q >= P || (P > 1 && !p.slots) || seq_lo < 0 || seq_hi < seq_lo ||
        seq_hi > p.T || gc0 < 0 || gc0 + (je - jb) > p.nc_max) {
      if (tid == 0) raise_error(p.err, kErrDeviceArgument);
      continue;
    }
    // where the item's state starts and ends
    const size_t head_off = ((size_t)n * p.Hv + h) * kHeadDim * kHeadDim;
    auto slot = [&](int skind, int sq, int kseg) {
      return p.slots + ((size_t)part_slot(p.slot_base[n], kseg, P, skind, sq) * p.Hv + h) * (kHeadDim * kHeadDim);
    };
    const float* src = nullptr;  // NULL: zeros (or the identity for a transition)
    if (kind == 0) src = (P > 1 && p.seg > 0) ? slot(2, 0, p.seg - 1) : (p.state_src ? p.state_src + head_off : nullptr);
    const bool late_qk = kind == 0 && q > 0;  // the q/k buffer serves the start-state combine first
    if (tid == 0 && seq_e > seq_s) {
      issue_vec(gc0, h, 0, true);
      if (!late_qk) issue_qk_tiles(sb + SS_QK, &p.tmap, p.Hk, seq_s, kh, bar_qk);
      issue_v(seq_s, h);
      issue_tp(gc0, h);
    }
    pend_qk = !late_qk && seq_e > seq_s;
    pend_v = pend_tp = seq_e > seq_s;
    if (seq_e > seq_s) pend_vec |= 1u;

    // ---- initial state -> tensor memory
    {
#pragma unroll
      for (int cq = 0; cq < 4 / kParts; ++cq) {
        const int c0 = part * (128 / kParts) + cq * 32;
        float v[32];
        if (src) {
          const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)row * kHeadDim + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 f = __ldg(s4 + i);
            v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = (kind == 2 && c0 + i == row) ? 1.f : 0.f;
        }
        tmem_st32(tl + SC_S + c0, v);
      }
    }
    // ---- part q's start state: q combine steps from the segment's start state
    if (late_qk) {
      // L and Phi of the parts before this one: completion flags set by the items that wrote them
      bool got = true;
      if (tid == 0) {
        for (int qq = 0; qq < q && got; ++qq)
          for (int sk = 0; sk < 2 && got; ++sk) {
            const int* f = p.flags + (size_t)part_slot(p.slot_base[n], p.seg, P, sk, qq) * p.Hv + h;
            uint32_t it = 0;
            while (ld_acquire_gpu(f) == 0 && ++it < kFlagWaitLimit) __nanosleep(256);
            got = it < kFlagWaitLimit;
          }
        if (!got) raise_error(p.err, kErrTimeout);
      }
      tc_fence_before();
      ok = __syncthreads_and(got ? 1 : 0) != 0 && ok;
      tc_fence_after();
      if (!ok) break;
      for (int qq = 0; qq < q && ok; ++qq) combine(slot(0, qq, p.seg), slot(1, qq, p.seg));
      if (!ok) break;
      if (tid == 0 && seq_e > seq_s) issue_qk_tiles(sb + SS_QK, &p.tmap, p.Hk, seq_s, kh, bar_qk);
      pend_qk = seq_e > seq_s;
    }

    // the chunk chain, compiled with the output stage (parts) and without it (L and Phi items)
    auto chain = [&](auto outs_c) {
      constexpr bool outs = decltype(outs_c)::value;
      const bool zero_v = !outs && kind == 2;  // a transition: v = 0
      const bool gz = gated && outs;
      int vb = 0;
      for (int c0 = seq_s, gc = gc0; c0 < seq_e && ok; c0 += kChunk, ++gc, ph_mma ^= 1u, vb ^= 1) {
        const int L = min(kChunk, seq_e - c0);
        const bool has_next = c0 + kChunk < seq_e;
        const float* vec = reinterpret_cast<const float*>(sm + SS_VEC + vb * kRecVec);

        {
  #ifdef GDN_TEST_HOOKS
          const uint32_t vec_limit = g_test_drop_vec_copy ? kTestWaitLimit : kWaitLimit;
  #else
          const uint32_t vec_limit = kWaitLimit;
  #endif
          const bool got = mbar_wait(bar_vec0 + 8 * vb, (ph_vec >> vb) & 1u, vec_limit);
          ph_vec ^= 1u << vb;
          pend_vec &= ~(1u << vb);
          if (!got) raise_error(p.err, kErrTimeout);
          ok = __syncthreads_and(got ? 1 : 0) != 0 && ok;
        }
        if (!ok) break;
        const float gL = vec[V_MISC];


        // ================= [X | O1] = S0 [K; Q]^T one 64-key half at a time: X from the hi and lo
        // parts of S0, the output-only O1 from the hi part
        convert_half(0, gL);
        fence_proxy_async_smem();
        tc_fence_before();
        wait_bar(bar_qk, ph_qk);  // the q/k tile (its latency overlaps the conversion above)
        pend_qk = false;
        tc_fence_after();
        if (!ok) break;
        if (tid == 0) {
          mma_bf16_k4<2, 2>(tmem + SC_X, sw128_desc(sb + SS_W), sw128_desc(sb + SS_QK), ID128, 0);
          mma_bf16_k4<2, 2>(tmem + SC_X, sw128_desc(sb + SS_W + 16384), sw128_desc(sb + SS_QK), ID64, 1);
          mma_commit(bar_h);
        }
        await_mma(bar_h);
        if (!ok) break;
        convert_half(64, gL);
        operands_ready();
        if (tid == 0) {
          mma_bf16_k4<2, 2>(tmem + SC_X, sw128_desc(sb + SS_W), sw128_desc(sb + SS_QK + 16384), ID128, 1);
          mma_bf16_k4<2, 2>(tmem + SC_X, sw128_desc(sb + SS_W + 16384), sw128_desc(sb + SS_QK + 16384), ID64, 1);
          mma_commit(bar_x);
        }
        {
          uint32_t ph = ph_mma;
          wait_two(bar_x, ph, bar_v, ph_v);
          tc_fence_after();
        }
        pend_v = false;
        if (!ok) break;

        // ================= R = diag(beta) V - diag(c_x) X^T -> hi/lo (value-major)
        {
          float x[kW];
          tmem_ld_cols<kW>(tl + SC_X + part * kW, x);
          // V[t][row] for t = part * kW + i: the swizzle term depends on i & 7 only
          const uint8_t* vbase = sm + SS_V + (row >> 6) * 8192 + part * kW * 128 + ((row & 7) << 1);
          const int rsw = (row >> 3) & 7;
          auto v_at = [&](int i) {
            return bf2f(*reinterpret_cast<const uint16_t*>(vbase + i * 128 + ((rsw ^ (i & 7)) << 4)));
          };
  #pragma unroll
          for (int i4 = 0; i4 < kW; i4 += 4) {
            const float4 bt = zero_v ? make_float4(0.f, 0.f, 0.f, 0.f)
                                     : *reinterpret_cast<const float4*>(vec + V_BETA + part * kW + i4);
            const float4 nc = *reinterpret_cast<const float4*>(vec + V_NCX + part * kW + i4);
            const float2 r0 = __ffma2_rn(make_float2(nc.x, nc.y), make_float2(x[i4], x[i4 + 1]),
                                         __fmul2_rn(make_float2(bt.x, bt.y), make_float2(v_at(i4), v_at(i4 + 1))));
            const float2 r1 = __ffma2_rn(make_float2(nc.z, nc.w), make_float2(x[i4 + 2], x[i4 + 3]),
                                         __fmul2_rn(make_float2(bt.z, bt.w), make_float2(v_at(i4 + 2), v_at(i4 + 3))));
            x[i4] = r0.x; x[i4 + 1] = r0.y; x[i4 + 2] = r1.x; x[i4 + 3] = r1.y;
          }
          store_split_tmem(tl + SC_X + part * kW, x);  // over this thread's own X columns
        }
        // O1 leaves its columns (they take E next): into registers now, staged while the E MMAs run
        float o1[kW];
        if (outs) tmem_ld_cols<kW>(tl + SC_O1 + part * kW, o1);
        fence_proxy_async_smem();
        tc_fence_before();
        wait_bar(bar_tp, ph_tp);  // T and P of this chunk
        pend_tp = false;
        tc_fence_after();
        if (!ok) break;
        if (tid == 0) {
          // E^T = R T^T  (hi*hi + hi*lo + lo*hi), R from tensor memory (hi / lo pairs of 32 tokens per
          // thread part: hi at columns 32 p, lo at 32 p + 16 of the X region)
  #pragma unroll
          for (int pp = 0; pp < 2; ++pp)
            mma_bf16_k2_ta<2>(tmem + SC_O1, tmem + SC_X + 32 * pp, sw128_desc(sb + SS_T) + 4 * pp, ID64, pp);
  #pragma unroll
          for (int pp = 0; pp < 2; ++pp)
            mma_bf16_k2_ta<2>(tmem + SC_O1, tmem + SC_X + 32 * pp, sw128_desc(sb + SS_T + 8192) + 4 * pp, ID64, 1);
  #pragma unroll
          for (int pp = 0; pp < 2; ++pp)
            mma_bf16_k2_ta<2>(tmem + SC_O1, tmem + SC_X + 32 * pp + 16, sw128_desc(sb + SS_T) + 4 * pp, ID64, 1);
          mma_commit(bar_e);
        } else if (tid == 32) {
          // the V buffer is free: the gate input of this chunk (gated), else the next chunk's v; and
          // the next chunk's vector block into the other buffer (last read by chunk c - 1)
          if (gz) issue_z(c0, h);
          else if (has_next) issue_v(c0 + kChunk, h);
          if (has_next) issue_vec(gc + 1, h, vb ^ 1);
        }
        if (has_next) pend_vec |= 1u << (vb ^ 1);
        pend_z = gz;
        pend_v = !gz && has_next;
        // o1 diag(c_o) -> the staging area (token-major fp32), free since the X MMAs completed
        if (outs) {
  #pragma unroll
        for (int i4 = 0; i4 < kW; i4 += 4) {
          const int t0 = part * kW + i4;
          const float4 co = *reinterpret_cast<const float4*>(vec + V_CO + t0);
          const float2 a = __fmul2_rn(make_float2(o1[i4], o1[i4 + 1]), make_float2(co.x, co.y));
          const float2 b = __fmul2_rn(make_float2(o1[i4 + 2], o1[i4 + 3]), make_float2(co.z, co.w));
          s_work[t0 * 128 + row] = a.x;
          s_work[(t0 + 1) * 128 + row] = a.y;
          s_work[(t0 + 2) * 128 + row] = b.x;
          s_work[(t0 + 3) * 128 + row] = b.y;
        }
        }
        await_mma(bar_e);
        if (!ok) break;

        // ================= E~ = E diag(c_s) -> hi/lo (tensor memory, over R);  E -> bf16 (output operand, over T)
        {
          float ev[kW], es[kW];
          tmem_ld_cols<kW>(tl + SC_O1 + part * kW, ev);
  #pragma unroll
          for (int q = 0; q < kW / 8; ++q) {
            const float4 c0v = *reinterpret_cast<const float4*>(vec + V_CS + part * kW + 8 * q);
            const float4 c1v = *reinterpret_cast<const float4*>(vec + V_CS + part * kW + 8 * q + 4);
            const float* e8 = ev + 8 * q;
            const float2 p0 = __fmul2_rn(make_float2(e8[0], e8[1]), make_float2(c0v.x, c0v.y));
            const float2 p1 = __fmul2_rn(make_float2(e8[2], e8[3]), make_float2(c0v.z, c0v.w));
            const float2 p2 = __fmul2_rn(make_float2(e8[4], e8[5]), make_float2(c1v.x, c1v.y));
            const float2 p3 = __fmul2_rn(make_float2(e8[6], e8[7]), make_float2(c1v.z, c1v.w));
            float* s8 = es + 8 * q;
            s8[0] = p0.x; s8[1] = p0.y; s8[2] = p1.x; s8[3] = p1.y; s8[4] = p2.x; s8[5] = p2.y; s8[6] = p3.x; s8[7] = p3.y;
            if (outs) store8_split(sm + SS_T, nullptr, 0, row, part * kW + 8 * q, e8);
          }
          store_split_tmem(tl + SC_X + part * kW, es);
        }
        operands_ready();
        if (tid == 0) {
          // S += E~ K: B = the raw k rows of the q/k tile read MN-major (N = 128 keys, 16 tokens per step)
          // (E~ from tensor memory as R was), O2 = E P^T into the E columns
  #pragma unroll
          for (int pp = 0; pp < 2; ++pp)
            mma_bf16_k2_ta<128>(tmem + SC_S, tmem + SC_X + 32 * pp, sw128_mn_desc(sb + SS_QK, 16384) + 256 * pp,
                                ID128_BMN, 1);
  #pragma unroll
          for (int pp = 0; pp < 2; ++pp)
            mma_bf16_k2_ta<128>(tmem + SC_S, tmem + SC_X + 32 * pp + 16, sw128_mn_desc(sb + SS_QK, 16384) + 256 * pp,
                                ID128_BMN, 1);
          if (outs) mma_bf16_k4<2, 2>(tmem + SC_O1, sw128_desc(sb + SS_T), sw128_desc(sb + SS_P), ID64, 0);
          mma_commit(bar_s);
        }
        constexpr int kTok = kChunk / kWarps;
        await_mma(bar_s);
        if (!ok) break;
        if (has_next) {  // two issuing threads in different warps, so neither lags by both
          if (tid == 0) issue_qk_tiles(sb + SS_QK, &p.tmap, p.Hk, c0 + kChunk, kh, bar_qk);
          else if (tid == 32) issue_tp(gc + 1, h);
        }
        pend_qk = pend_tp = has_next;

        // ================= output: o = O1 diag(c_o) (staged) + O2, then the gated RMSNorm
        if (outs) {
          {
            float o2a[16], o2b[16];
            tmem_ld16x2(tl + SC_O1 + part * kW, tl + SC_O1 + part * kW + 16, o2a, o2b);
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
                const uint2 zz = *reinterpret_cast<const uint2*>(sm + SS_V + (warp + kWarps * i) * 256 + lane * 8);
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
        }
        fence_proxy_async_smem();  // vector-block and z reads -> the async proxy (the next loads)
        tc_fence_before();
        __syncthreads();  // staging reads and accumulator reads done before the next chunk reuses them
        tc_fence_after();
        if (tid == 64 && gz && has_next) issue_v(c0 + kChunk, h);
        if (gz && has_next) pend_v = true;
      }
    };
    if (kind == 0) chain(BoolC<true>{});
    else chain(BoolC<false>{});
    if (!ok) break;

    // ---- final state -> global (state_out, a part's slot, or nowhere for a part before the last);
    // the item is decoded again rather than kept in registers across the chain
    decode(*item_slot, n, q, kind);
    float* dst = nullptr;
    {
      const int Pn = p.part_cnt[n];
      const size_t hoff = ((size_t)n * p.Hv + h) * kHeadDim * kHeadDim;
      auto slot2 = [&](int skind, int sq, int kseg) {
        return p.slots + ((size_t)part_slot(p.slot_base[n], kseg, Pn, skind, sq) * p.Hv + h) * (kHeadDim * kHeadDim);
      };
      if (kind != 0) dst = slot2(kind - 1, q, p.seg);
      else if (q == Pn - 1)
        dst = (Pn > 1 && p.seg < p.nseg - 1) ? slot2(2, 0, p.seg) : (p.state_out ? p.state_out + hoff : nullptr);
    }
    if (dst) {
#pragma unroll
      for (int cq = 0; cq < 4 / kParts; ++cq) {
        const int c0 = part * (128 / kParts) + cq * 32;
        float v[32];
        tmem_ld32(tl + SC_S + c0, v);
        float4* d4 = reinterpret_cast<float4*>(dst + (size_t)row * kHeadDim + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
    if (kind != 0) {  // L or Phi of a part: complete once every row is stored
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        st_release_gpu(p.flags + (size_t)part_slot(p.slot_base[n], p.seg, p.part_cnt[n], kind - 1, q) * p.Hv + h, 1);
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
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, SC_COLS);
  }
}

// Run by the segment-table CTA after the schedule (order = longest first): which sequences are cut
// into parts, and the work items of the parts launches (the same for every segment).
// A sequence is split when its shortest segment holds more than twice the chunks one CTA slot
// would get if the segment's work were spread evenly (the share, at least kMinPart): into
// ceil(m / share) parts (3 .. kMaxParts), while state slots last.  A lower threshold split an
// evenly loaded batch (4 x 4096 tokens: 0.73 -> 1.05 ms), and two parts gain nothing, since a part
// waits for the L and Phi chains of the part before it.  `allow` is 0 where a split is not
// possible (one segment updating its state in place, or no slots in the workspace).
//   items: first (n, q) for L and (n, q | 1 << 16) for Phi, q = 0 .. P - 2 of each split sequence,
//   then the parts (n, q), q = 0 .. P - 1; counts[0]: all items, counts[1]: the L / Phi items;
//   the slots' completion flags zeroed.
__device__ __forceinline__ void plan_parts(const int32_t* cu, int N, int Hv, int nseg, int slots, int allow,
                                           const int32_t* order, int32_t* part_cnt, int32_t* slot_base, int2* items,
                                           int32_t* counts, int* flags, unsigned* counters) {
  __shared__ int s_n[kMaxSplitSeqs], s_P[kMaxSplitSeqs], s_extra[kMaxSplitSeqs + 1];
  __shared__ int s_ns;
  __shared__ long long s_total;
  const int tid = threadIdx.x;
  for (int i = tid; i < kSlotCap * Hv; i += blockDim.x) flags[i] = 0;
  if (tid < kMaxSegments) counters[4 + tid] = 0u;  // the parts launches' work counters
  if (tid == 0) s_total = 0;
  __syncthreads();
  auto nchunks = [&](int i) {
    const int a = __ldg(cu + i), b = __ldg(cu + i + 1);
    return (a < 0 || b < a) ? 0 : (b - a + kChunk - 1) / kChunk;
  };
  long long local = 0;
  for (int i = tid; i < N; i += blockDim.x) local += nchunks(i);
  atomicAdd(reinterpret_cast<unsigned long long*>(&s_total), (unsigned long long)local);
  __syncthreads();
  if (tid == 0) {
    int ns = 0, used = 0;
    if (allow && N <= kScheduleSortMax && nseg > 0 && slots > 0) {
      const long long per_slot = (s_total * Hv + (long long)nseg * slots - 1) / ((long long)nseg * slots);
      const int share = (int)max((long long)kMinPart, per_slot);
      for (int i = 0; i < N && ns < kMaxSplitSeqs; ++i) {
        const int n = __ldg(order + i);
        const int m = nchunks(n) / nseg;  // the shortest segment of this sequence
        if (m <= 2 * share) break;         // longest first: no later sequence splits either
        int P = min(kMaxParts, (m + share - 1) / share);  // at least 3 here
        while (P > 1 && used + nseg * (2 * P - 1) > kSlotCap) --P;
        if (P < 3) break;  // two parts gain nothing: a part waits for the chains of the one before
        s_n[ns] = n;
        s_P[ns] = P;
        slot_base[n] = used;
        used += nseg * (2 * P - 1);
        ++ns;
      }
    }
    s_ns = ns;
    s_extra[0] = 0;
    for (int j = 0; j < ns; ++j) s_extra[j + 1] = s_extra[j] + s_P[j] - 1;
    counts[0] = 3 * s_extra[ns] + ns;  // L / Phi items, then the parts
    counts[1] = 2 * s_extra[ns];
  }
  __syncthreads();
  const int ns = s_ns;
  const int A = 2 * s_extra[ns];
  // the split sequences are order[0 .. ns)
  for (int i = tid; i < N; i += blockDim.x) part_cnt[__ldg(order + i)] = i < ns ? s_P[i] : 1;
  if (tid < ns) {
    const int P = s_P[tid], n = s_n[tid];
    const int lp = 2 * s_extra[tid], pp = A + s_extra[tid] + tid;
    for (int q = 0; q < P - 1; ++q) {
      items[lp + 2 * q] = make_int2(n, q);
      items[lp + 2 * q + 1] = make_int2(n, q | (1 << 16));
    }
    for (int q = 0; q < P; ++q) items[pp + q] = make_int2(n, q);
  }
}

// One CTA: for every segment k < nseg, the exclusive prefix over sequences of their chunk counts in
// segment k (seg_pref[k (N + 1) + n]; the total at n = N), and the per-segment work counters zeroed.
// Sequences with inconsistent cu_seqlens count as empty here; the main kernels report them.
__global__ void __launch_bounds__(1024) chunk_segments_kernel(const int32_t* cu, int N, int nseg, int32_t* seg_pref,
                                                              unsigned* counters, int Hv, int slots, int allow,
                                                              const int32_t* order, int32_t* part_cnt,
                                                              int32_t* slot_base, int2* items, int32_t* counts,
                                                              int* flags) {
  __shared__ int32_t s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < kMaxSegments) counters[tid] = 0u;
  const int per = (N + 1023) / 1024, lo = min(N, tid * per), hi = min(N, lo + per);
  for (int k = 0; k < nseg; ++k) {
    auto len = [&](int i) {
      const int nch = (max(0, __ldg(cu + i + 1) - __ldg(cu + i)) + kChunk - 1) / kChunk;
      return seg_begin(k + 1, nch, nseg) - seg_begin(k, nch, nseg);
    };
    int local = 0;
    for (int i = lo; i < hi; ++i) local += len(i);
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
      s_warp[lane] = w;
    }
    __syncthreads();
    int32_t* pref = seg_pref + (size_t)k * (N + 1);
    int run = incl - local + (warp > 0 ? s_warp[warp - 1] : 0);
    for (int i = lo; i < hi; ++i) {
      pref[i] = run;
      run += len(i);
    }
    if (tid == 1023) pref[N] = s_warp[31];
    __syncthreads();  // s_warp is reused by the next segment
  }
  plan_parts(cu, N, Hv, nseg, slots, allow, order, part_cnt, slot_base, items, counts, flags, counters);
}


}  // namespace

namespace {

size_t pad256(size_t b) { return (b + 255) / 256 * 256; }

// upper bound of sum_n ceil(L_n / 64) for N sequences of T tokens in total
long chunk_bound(int N, int T) { return ((long)T + 63L * N) / kChunk; }

struct SplitLayout {
  unsigned* counters;  // one work counter per segment (main launches), then one per segment (aux)
  int32_t* counts;     // the numbers of main and aux items (counters + 16)
  int32_t* order;
  int32_t* part_cnt;   // [N]
  int32_t* slot_base;  // [N]
  int2* items;         // [N + 2 kSlotCap]
  int* flags;          // [kSlotCap][Hv]
  float* slots;        // [kSlotCap][Hv][128][128] when T >= kSplitMinTokens, else NULL
  int32_t* chunk_off;
  int32_t* seg_pref;   // kMaxSegments x (N + 1)
  uint8_t* rec;
};

constexpr size_t kSlotBytes = (size_t)kHeadDim * kHeadDim * 4;  // one head's state

// bytes before the records (they depend on N only)
size_t split_head_bytes(int N) {
  return 256 + pad256((size_t)N * 4) + pad256((size_t)(N + 1) * 4) + pad256((size_t)kMaxSegments * (N + 1) * 4) +
         2 * pad256((size_t)N * 4) + pad256((size_t)(N + 2 * kSlotCap) * 8) + pad256((size_t)kSlotCap * 192 * 4);
}

SplitLayout split_layout(void* workspace, int N, int T, int Hv) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SplitLayout l;
  size_t off = 256;
  l.counters = reinterpret_cast<unsigned*>(ws);
  l.counts = reinterpret_cast<int32_t*>(ws + 64);
  l.order = reinterpret_cast<int32_t*>(ws + off);
  off += pad256((size_t)N * 4);
  l.chunk_off = reinterpret_cast<int32_t*>(ws + off);
  off += pad256((size_t)(N + 1) * 4);
  l.seg_pref = reinterpret_cast<int32_t*>(ws + off);
  off += pad256((size_t)kMaxSegments * (N + 1) * 4);
  l.part_cnt = reinterpret_cast<int32_t*>(ws + off);
  off += pad256((size_t)N * 4);
  l.slot_base = reinterpret_cast<int32_t*>(ws + off);
  off += pad256((size_t)N * 4);
  l.items = reinterpret_cast<int2*>(ws + off);
  off += pad256((size_t)(N + 2 * kSlotCap) * 8);
  l.flags = reinterpret_cast<int*>(ws + off);
  off += pad256((size_t)kSlotCap * 192 * 4);  // room for the most V heads a geometry may have
  l.rec = ws + off;
  off += (size_t)chunk_bound(N, T) * (size_t)Hv * REC_BYTES;
  l.slots = T >= kSplitMinTokens ? reinterpret_cast<float*>(ws + off) : nullptr;
  return l;
}

// Per-device side stream for the prep kernels of later segments (created on first use).
cudaError_t side_stream(cudaStream_t* out, int which = 0) {
  static std::mutex mu;
  static cudaStream_t streams[2][64] = {{nullptr}};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  cudaStream_t& st = streams[which][dev];
  if (!st) {
    e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      st = nullptr;
      return e;
    }
  }
  *out = st;
  return cudaSuccess;
}

// Events ordering the segments' prep and state launches, created once per (host thread, device)
// and reused by every later call of that thread.  They are per thread because the launcher records
// an event and then makes the other stream wait on it: with events shared between threads, one
// thread's wait could pick up another thread's later record.  Within one thread each wait is
// issued right after its own record, so reuse across calls is safe.
struct SegmentEvents {
  cudaEvent_t ev[64][kMaxSegments + 1] = {};
  ~SegmentEvents() {
    for (auto& d : ev)
      for (cudaEvent_t e : d)
        if (e) cudaEventDestroy(e);  // after the context is gone this returns an error: ignored
  }
};

cudaError_t segment_events(cudaEvent_t** out) {
  thread_local SegmentEvents cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  for (int k = 0; k <= kMaxSegments; ++k) {
    if (!cache.ev[dev][k]) {
      e = cudaEventCreateWithFlags(&cache.ev[dev][k], cudaEventDisableTiming);
      if (e != cudaSuccess) {
        cache.ev[dev][k] = nullptr;
        return e;
      }
    }
  }
  *out = cache.ev[dev];
  return cudaSuccess;
}

template <typename K>
cudaError_t set_smem_once(K kernel, uint32_t bytes, int (&done)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  // the largest shared-memory carveout, so that as many CTAs as the footprint allows share an SM
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess && dev < 64) done[dev] = 1;
  return e;
}

}  // namespace

#ifdef GDN_TEST_HOOKS
cudaError_t test_set_dropped_copy_chunk(unsigned on) { return cudaMemcpyToSymbol(g_test_drop_vec_copy, &on, sizeof on); }
#endif

size_t split_workspace_bytes(int N, int T, int Hk, int Hv) {
  (void)Hk;
  if (N <= 0) return 0;
  return split_head_bytes(N) + (size_t)chunk_bound(N, T) * (size_t)Hv * REC_BYTES +
         (T >= kSplitMinTokens ? (size_t)kSlotCap * Hv * kSlotBytes : 0);
}

cudaError_t launch_chunk_prefill_split(const LaunchEnv& env, const uint16_t* qkv, const GateSrc& gates,
                                       const int32_t* cu, int N, int T, int Hk, int Hv, float q_scale, float l2_eps,
                                       const float* state_in, float* state_out, const uint16_t* z,
                                       const uint16_t* norm_w, float rms_eps, uint16_t* out, void* workspace) {
  static int prep_set[64] = {0}, state_set[64] = {0}, parts_set[64] = {0};
  if (N <= 0) return cudaSuccess;
  const SplitLayout lay = split_layout(workspace, N, T, Hv);
  const long nc_max = chunk_bound(N, T);
  CUtensorMap tmap, tmap_z;
  memset(&tmap, 0, sizeof tmap);
  memset(&tmap_z, 0, sizeof tmap_z);
  if (T > 0) {
    cudaError_t e = encode_chunk_tensor_maps(&tmap, &tmap_z, qkv, z, T, Hk, Hv);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_chunk_schedule(env.stream, cu, N, lay.order, lay.counters, lay.chunk_off);
  if (e != cudaSuccess) return e;
  if ((e = set_smem_once(chunk_prep_kernel, PR_BYTES, prep_set)) != cudaSuccess) return e;
  if ((e = set_smem_once(chunk_state_kernel, SS_BYTES, state_set)) != cudaSuccess) return e;
  if ((e = set_smem_once(chunk_part_state_kernel, SS_BYTES, parts_set)) != cudaSuccess) return e;
  int sms = 0;
  if ((e = device_sm_count(&sms)) != cudaSuccess) return e;

  // Segments: with a state_out buffer to carry the state between launches, a long enough input
  // and no stream capture in progress, the chunks of every sequence are split into three parts
  // and the prep kernel of part k + 1 (on a side stream) runs beside the state kernel of part k;
  // otherwise one part, everything on the caller's stream.
  int nseg = 1;
  cudaStream_t side = env.stream, pstream = env.stream;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (state_out && T >= 64 * kChunk && cudaStreamIsCapturing(env.stream, &cap) == cudaSuccess &&
      cap == cudaStreamCaptureStatusNone && side_stream(&side) == cudaSuccess && side_stream(&pstream, 1) == cudaSuccess)
    nseg = 3;  // measured best of 2, 3 and 4 over the batched and the varlen workloads
  if (nseg == 1) side = pstream = env.stream;
  // Two state CTAs per SM: 2 x 256 tensor-memory columns, 2 x (SS_BYTES + 1 KB reserved) of shared
  // memory and 2 x 256 threads x 128 registers all fit.  (The runtime's occupancy query reports one
  // CTA per SM for any kernel that allocates tensor memory, but the hardware co-schedules two; a
  // CTA that cannot be resident runs later, finds no work and exits.)
  constexpr int per_sm = 2;
  const long slots = (long)sms * per_sm;
  // parts of long sequences (not with one segment updating its state in place: a part would read
  // a state the last part has replaced)
  const int allow = lay.slots != nullptr && T > 0 && !(nseg == 1 && state_in && state_in == state_out);
  chunk_segments_kernel<<<1, 1024, 0, env.stream>>>(cu, N, nseg, lay.seg_pref, lay.counters, Hv, (int)slots, allow,
                                                    lay.order, lay.part_cnt, lay.slot_base, lay.items, lay.counts,
                                                    lay.flags);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  cudaEvent_t* ev = nullptr;
  if (nseg > 1) {
    e = segment_events(&ev);
    if (e == cudaSuccess) e = cudaEventRecord(ev[nseg], env.stream);  // schedule, segment and part tables written
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, ev[nseg], 0);
    if (e != cudaSuccess) return e;
  }

  PrepParams pp;
  memset(&pp, 0, sizeof pp);
  pp.tmap = tmap;
  pp.gates = gates; pp.cu = cu; pp.chunk_off = lay.chunk_off; pp.rec = lay.rec; pp.err = env.err;
  pp.N = N; pp.T = T; pp.Hk = Hk; pp.Hv = Hv; pp.nseg = nseg; pp.nc_max = (int)nc_max;
  pp.q_scale = q_scale; pp.l2_eps = l2_eps;

  StateParams sp;
  memset(&sp, 0, sizeof sp);
  sp.nseg = nseg;
  sp.tmap = tmap;
  sp.tmap_z = tmap_z;
  sp.cu = cu; sp.order = lay.order; sp.chunk_off = lay.chunk_off; sp.rec = lay.rec;
  sp.state_in = state_in; sp.state_out = state_out; sp.z = z; sp.norm_w = norm_w; sp.out = out; sp.err = env.err;
  sp.N = N; sp.T = T; sp.Hk = Hk; sp.Hv = Hv; sp.nc_max = (int)nc_max; sp.rms_eps = rms_eps;
  sp.part_cnt = lay.part_cnt;  // the main launch leaves the split sequences to the parts launch
  // the parts launch: every CTA slot (one without an item returns at once; the number of items is
  // only known on the device)
  StateParams xp = sp;
  xp.order = nullptr;
  xp.items = lay.items; xp.item_count = lay.counts; xp.part_cnt = lay.part_cnt; xp.slot_base = lay.slot_base;
  xp.slots = lay.slots; xp.flags = lay.flags;
  const long busy = std::min<long>((long)N * Hv, slots);
  const int state_grid = (int)busy;

  for (int k = 0; k < nseg && e == cudaSuccess; ++k) {
    if (T > 0 && nc_max > 0) {
      pp.seg = k;
      pp.seg_pref = lay.seg_pref + (size_t)k * (N + 1);
      // Segment 0's prep runs alone on the whole GPU.  Later ones run beside a state kernel: they
      // take only the CTA slots the state kernel leaves (a prep CTA fits beside one state CTA),
      // so the state CTAs are placed the same way whichever launch the scheduler sees first.
      const long prep_grid = k == 0 ? slots : std::max<long>(sms / 2, slots - busy);
      chunk_prep_kernel<<<(unsigned)prep_grid, kThreads, PR_BYTES, side>>>(pp);
      if ((e = cudaGetLastError()) != cudaSuccess) break;
    }
    if (nseg > 1) {
      e = cudaEventRecord(ev[k], side);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(env.stream, ev[k], 0);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(pstream, ev[k], 0);
      if (e != cudaSuccess) break;
    }
    sp.seg = k;
    sp.counter = lay.counters + k;
    sp.state_src = k == 0 ? state_in : state_out;
    chunk_state_kernel<<<state_grid, kThreads, SS_BYTES, env.stream>>>(sp);
    if ((e = cudaGetLastError()) != cudaSuccess) break;
    // the split sequences' parts, beside the other sequences; issued after them, which measured
    // faster for calls without a split (the parts launch's CTAs then find their count zero at once)
    if (lay.slots) {
      xp.seg = k;
      xp.counter = lay.counters + 4 + k;
      xp.state_src = k == 0 ? state_in : state_out;
      chunk_part_state_kernel<<<(unsigned)slots, kThreads, SS_BYTES, pstream>>>(xp);
      e = cudaGetLastError();
    }
  }
  if (e == cudaSuccess && nseg > 1 && lay.slots) {  // the caller's stream waits for the parts as well
    e = cudaEventRecord(ev[kMaxSegments], pstream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(env.stream, ev[kMaxSegments], 0);
  }
  return e;
}

}  // namespace gdn
