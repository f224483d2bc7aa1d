// gdn_common.cuh -- internal helpers shared by the GDN kernels (not part of the C ABI).
//
// Inline-PTX wrappers for the sm_100-family tensor-core path (tcgen05 MMA with accumulators in
// tensor memory, mbarriers), bf16 bit conversions, and the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kHeadDim = 128;   // Dk = Dv
constexpr int kConvWidth = 4;   // W
constexpr int kChunk = 64;      // tokens per chunk

// bits of the device error word
enum : unsigned { kErrDeviceArgument = 1u, kErrTimeout = 2u };

struct LaunchEnv {
  unsigned* err;   // device error word of the current device
  int num_sms;
  cudaStream_t stream;
};

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
// two floats -> two bf16 (round to nearest even) in one 32-bit word, `lo` in the low half
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(x) = 2^(x log2 e)


// 2^x by the hardware approximation instruction (relative error ~2^-22; results below the
// smallest normal flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// hardware base-2 logarithm approximation
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// sigmoid(x) = 1 / (1 + e^-x) from the two approximations above (output-side gate only)
__device__ __forceinline__ float sigmoid_fast(float x) { return rcp_approx(1.0f + ex2_approx(-x * kLog2e)); }

// a + b = s + e exactly (Knuth's two-sum; rounded-to-nearest operations that nothing may fuse)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// SiLU of the width-4 conv tap sum w0 x0 + w1 x1 + w2 x2 + w3 x3 (bf16 weights and inputs held as
// floats), rounded to the bf16 nearest the exact value.  Every bf16 x bf16 product is exact in
// fp32 and the sum is carried exactly as s + e1 + e2 + e3 (two-sums), so the fp32 SiLU estimate
// from it (hardware exp2 and reciprocal) errs by a few ulps (more for large negative sums, where
// exp amplifies the argument's rounding); where the estimate lies within 32 + 2 |acc| ulps of a
// bf16 rounding midpoint, the SiLU is recomputed in fp64 from the exact sum before rounding.
// the rare fp64 re-evaluation, out of line so that the fp32 path stays compact
static __device__ __noinline__ uint16_t silu_bf16_fp64(float s, float e1, float e2, float e3) {
  const double ad = (double)s + (double)e1 + (double)e2 + (double)e3;
  return __bfloat16_as_ushort(__double2bfloat16(ad / (1.0 + exp(-ad))));
}

__device__ __forceinline__ uint16_t silu_bf16_rn(float w0, float x0, float w1, float x1, float w2, float x2,
                                                 float w3, float x3) {
  float s, e1, e2, e3;
  two_sum(__fmul_rn(w0, x0), __fmul_rn(w1, x1), s, e1);
  two_sum(s, __fmul_rn(w2, x2), s, e2);
  two_sum(s, __fmul_rn(w3, x3), s, e3);
  const float acc = __fadd_rn(s, __fadd_rn(__fadd_rn(e1, e2), e3));
  // the estimate: acc / (1 + 2^(-acc log2 e)) with the hardware exp2 and reciprocal (a few ulps)
  const float y = acc * rcp_approx(1.0f + ex2_approx(-acc * kLog2e));
  const int off = (int)(__float_as_uint(y) & 0xFFFFu) - 0x8000;  // fp32 ulps from the midpoint
  const int margin = 32 + (int)fminf(2.f * fabsf(acc), 4096.f);
  if (off >= -margin && off <= margin) return silu_bf16_fp64(s, e1, e2, e3);
  return f2bf(y);
}
// hardware tanh approximation (max relative error about 2^-11)
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// tanh(z / 2) of the two bf16 values packed in `zz` (low half first), by the bf16x2 hardware tanh
// (about bf16 precision), returned as two floats
__device__ __forceinline__ float2 tanh_half_bf16x2(uint32_t zz) {
  const __nv_bfloat162 z2 = *reinterpret_cast<const __nv_bfloat162*>(&zz);
  const __nv_bfloat162 t2 = h2tanh_approx(__hmul2(z2, __floats2bfloat162_rn(0.5f, 0.5f)));
  const uint32_t t = *reinterpret_cast<const uint32_t*>(&t2);
  return make_float2(__uint_as_float(t << 16), __uint_as_float(t & 0xFFFF0000u));
}
// sigmoid(x) = (1 + tanh(x / 2)) / 2: one special-function operation
__device__ __forceinline__ float sigmoid_tanh(float x) { return fmaf(0.5f, tanh_approx(0.5f * x), 0.5f); }

// The gates of the recurrence from their projections, for one (row, V head):
//   g = -exp(A_log) softplus(a + dt_bias),  beta = sigmoid(b),  softplus(x) = log(1 + e^x)
// (the gate of the published Gated DeltaNet / Mamba-2 layers; the GDN pages name these inputs but
// give no formula).  One definition serves the standalone gates kernel and every kernel that
// derives its gates itself, so both routes compute the same bits.
__device__ __forceinline__ void gate_one(float a, float b, float A_log, float dt_bias, float& g, float& beta) {
  const float x = a + dt_bias;
  const float sp = x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));  // log(1 + e^x), no overflow
  g = -expf(A_log) * sp;
  beta = 1.0f / (1.0f + expf(-b));
}

// Where a kernel takes its gates from: g and beta given ([rows, Hv] fp32), or, when `a` is set,
// derived from the projections a, b ([rows, Hv] bf16) and the per-head A_log, dt_bias ([Hv] fp32).
struct GateSrc {
  const float* g;
  const float* beta;
  const uint16_t* a;
  const uint16_t* b;
  const float* A_log;
  const float* dt_bias;
};
// The gates of element idx = row * Hv + h.
__device__ __forceinline__ void load_gate(const GateSrc& s, size_t idx, int h, float& g, float& beta) {
  if (s.a) {
    gate_one(bf2f(__ldg(s.a + idx)), bf2f(__ldg(s.b + idx)), __ldg(s.A_log + h), __ldg(s.dt_bias + h), g, beta);
  } else {
    g = __ldg(s.g + idx);
    beta = __ldg(s.beta + idx);
  }
}

__device__ __forceinline__ void raise_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Bounded wait on the phase with the given parity.  Returns false when `limit` polls ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Arrive on the mbarrier and add `bytes` to the transaction count the phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(addr), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ TMA

// 2D tiled bulk tensor load global -> shared; completion is signalled on `bar` (complete_tx).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 1D bulk copy global -> shared of `bytes` (multiple of 16; both addresses 16-byte aligned);
// completion is signalled on `bar` (complete_tx).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// 2D tiled bulk tensor store shared -> global (bulk-group completion): x must be 16-byte aligned
// in bytes, and the box must lie where the caller may write.
__device__ __forceinline__ void tma_store_2d(const void* tmap, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap), "r"(x),
               "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the committed bulk stores of this thread have finished reading shared memory / have completed
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// L2 prefetch hints (no completion to wait for): a 2D tensor box, or `bytes` (multiple of 16,
// 16-byte aligned) of contiguous global memory.
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x), "r"(y)
               : "memory");
}
// bring a tensor map (kernel parameter) into the TMA unit's descriptor cache
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}
// acquire / release accesses of a flag shared by CTAs of one launch (GPU scope)
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ proxy / tcgen05 fences

// generic-proxy shared-memory writes -> visible to the async proxy (tensor-core operand reads)
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------ tensor memory

// Allocate `ncols` (power of two >= 32) TMEM columns; must be executed by one full warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem_addr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem_addr),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 lanes x 32 columns of 32-bit: thread i of the warp receives lane (quarter*32 + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 16 columns of 32-bit.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 16-column loads (for example of two accumulators) behind one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float (&a)[16], float (&b)[16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[16 + i]);
  }
}

// N (16 or 32) columns of this warp's 32 lanes.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32) tmem_ld32(taddr, v);
  else tmem_ld16(taddr, v);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

// ------------------------------------------------------------------ tcgen05 MMA descriptors

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte-swizzle layout:
// rows of 64 bf16 (128 bytes), groups of 8 rows 1024 bytes apart, 16-byte chunks of row r
// XOR-permuted by (r & 7).  The tile base must be 1024-byte aligned; advancing K by 16 elements
// inside the 64-element block adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)   // start address, 16-byte units
         | ((uint64_t)1 << 16)                   // leading-dimension byte offset (unused here)
         | ((uint64_t)(1024 >> 4) << 32)         // stride between 8-row groups
         | ((uint64_t)1 << 46)                   // descriptor version for tcgen05
         | ((uint64_t)2 << 61);                  // 128-byte swizzle
}

// Descriptor of an MN-major operand in the 128-byte-swizzle layout: each 128-byte row holds 64
// consecutive M/N elements of one K index, groups of 8 K rows are 1024 bytes apart and blocks
// of 64 M/N elements are `mn_block_bytes` apart.  Same physical layout as a K-major tile whose
// rows are K indices, so a TMA box of 64 tokens x 64 features serves as B with N = features.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t mn_block_bytes) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)
         | ((uint64_t)((mn_block_bytes >> 4) & 0x3FFFu) << 16)  // stride between 64-element M/N blocks
         | ((uint64_t)(1024 >> 4) << 32)                         // stride between 8-row K groups
         | ((uint64_t)1 << 46)
         | ((uint64_t)2 << 61);
}

// Instruction descriptor: D fp32, A and B bf16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// As above with B MN-major (the transpose-B bit).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_bmn(int M, int N) { return idesc_bf16_f32(M, N) | (1u << 16); }

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four consecutive K = 16 steps of one accumulation, issued back to back: the A and B descriptors
// advance by AS and BS descriptor units (16 bytes) per step.  The first step accumulates onto D
// when `acc_first` is nonzero, the other three always do.
template <uint32_t AS, uint32_t BS>
__device__ __forceinline__ void mma_bf16_k4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t acc_first) {
  asm volatile(
      "{\n.reg .pred p, q;\n.reg .b64 a1, a2, a3, b1, b2, b3;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "setp.ne.b32 q, %5, 0;\n"
      "add.s64 a1, %1, %6;\nadd.s64 a2, %1, %7;\nadd.s64 a3, %1, %8;\n"
      "add.s64 b1, %2, %9;\nadd.s64 b2, %2, %10;\nadd.s64 b3, %2, %11;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, q;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, q;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, q;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc_first), "r"(1u), "n"(AS), "n"(2 * AS), "n"(3 * AS), "n"(BS),
      "n"(2 * BS), "n"(3 * BS)
      : "memory");
}

// As mma_bf16_k4 with A in tensor memory: A (128 rows = lanes, K along columns, two bf16 per
// 32-bit column, the even K index in the low half) starts at column a_tmem and advances 8
// columns per K = 16 step.
template <uint32_t BS>
__device__ __forceinline__ void mma_bf16_k4_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t acc_first) {
  asm volatile(
      "{\n.reg .pred p, q;\n.reg .b64 b1, b2, b3;\n.reg .b32 a1, a2, a3;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "setp.ne.b32 q, %5, 0;\n"
      "add.u32 a1, %1, 8;\nadd.u32 a2, %1, 16;\nadd.u32 a3, %1, 24;\n"
      "add.s64 b1, %2, %6;\nadd.s64 b2, %2, %7;\nadd.s64 b3, %2, %8;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, q;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, q;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, q;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc_first), "r"(1u), "n"(BS), "n"(2 * BS), "n"(3 * BS)
      : "memory");
}

// Two K = 16 steps with A in tensor memory (advancing 8 columns) and B advancing BS units.
template <uint32_t BS>
__device__ __forceinline__ void mma_bf16_k2_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t acc_first) {
  asm volatile(
      "{\n.reg .pred p, q;\n.reg .b64 b1;\n.reg .b32 a1;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "setp.ne.b32 q, %5, 0;\n"
      "add.u32 a1, %1, 8;\n"
      "add.s64 b1, %2, %6;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, q;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc_first), "r"(1u), "n"(BS)
      : "memory");
}

// Arrive once on the mbarrier when every tcgen05 MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t mbar_addr) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar_addr)
               : "memory");
}

// Byte offset of bf16 element (row, k) in a K-major 128-byte-swizzle tile whose 64-column K
// blocks are `kb_stride` bytes apart.
__device__ __forceinline__ uint32_t sw128_offset(int row, int k, uint32_t kb_stride) {
  const int kb = k >> 6, kk = k & 63;
  return kb * kb_stride + row * 128 + ((((kk >> 3) ^ (row & 7)) & 7) << 4) + ((kk & 7) << 1);
}

}  // namespace gdn
