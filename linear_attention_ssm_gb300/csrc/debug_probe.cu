// debug_probe.cu -- one tcgen05 MMA tile, for verifying the descriptor and layout conventions the
// chunk-prefill kernels rely on: D[128 x N] = A[128 x 64] * B[N x 64]^T with bf16 operands and an
// fp32 accumulator in tensor memory.  A is read from 128-byte-swizzled K-major shared memory or
// from tensor memory (two bf16 per column); B from K-major or MN-major 128-byte-swizzled shared
// memory.
#include "../../include/gdn_debug.h"
#include "gdn_common.cuh"

namespace {

constexpr uint32_t kWait = 1u << 20;

template <int N>
__global__ void __launch_bounds__(128, 1) mma_probe_kernel(const uint16_t* A, const uint16_t* B, float* D,
                                                           unsigned* status, int flags) {
  __shared__ __align__(1024) uint8_t sa[128 * 128];
  __shared__ __align__(1024) uint8_t sbm[N * 128];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool a_tmem = flags & 1, b_mn = flags & 2;
  // row r of A (64 bf16 = 8 chunks of 16 B) -> swizzled row r
  for (int i = tid; i < 128 * 8; i += 128) {
    const int r = i >> 3, c = i & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(A + r * 64 + c * 8);
    *reinterpret_cast<uint4*>(sa + r * 128 + ((c ^ (r & 7)) << 4)) = v;
  }
  if (!b_mn) {
    for (int i = tid; i < N * 8; i += 128) {
      const int r = i >> 3, c = i & 7;
      const uint4 v = *reinterpret_cast<const uint4*>(B + r * 64 + c * 8);
      *reinterpret_cast<uint4*>(sbm + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
  } else {
    // MN-major: 128-byte rows hold 64 consecutive n of one k; blocks of 64 n are 64 rows (8 KB) apart
    for (int i = tid; i < N * 64; i += 128) {
      const int n = i % N, k = i / N;
      const int blk = n >> 6, nn = n & 63;
      const uint32_t off = blk * 8192 + k * 128 + ((((nn >> 3) ^ (k & 7)) & 7) << 4) + ((nn & 7) << 1);
      *reinterpret_cast<uint16_t*>(sbm + off) = B[n * 64 + k];
    }
  }
  if (tid == 0) {
    gdn::mbar_init(gdn::smem_u32(&bar), 1);
    gdn::fence_mbar_init();
  }
  if (warp == 0) gdn::tmem_alloc(gdn::smem_u32(&tslot), 256);
  gdn::fence_proxy_async_smem();
  gdn::tc_fence_before();
  __syncthreads();
  gdn::tc_fence_after();
  const uint32_t tmem = tslot;
  const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
  if (a_tmem) {  // row tid of A -> its lane, columns 128..159, two bf16 per column
    float v[32];
    for (int j = 0; j < 32; ++j)
      v[j] = __uint_as_float((uint32_t)A[tid * 64 + 2 * j] | ((uint32_t)A[tid * 64 + 2 * j + 1] << 16));
    gdn::tmem_st32(tl + 128, v);
    gdn::tc_fence_before();
    __syncthreads();
    gdn::tc_fence_after();
  }
  if (tid == 0) {
    const uint32_t b0 = gdn::smem_u32(sbm);
    const uint32_t id = b_mn ? gdn::idesc_bf16_f32_bmn(128, N) : gdn::idesc_bf16_f32(128, N);
    const uint64_t bd = b_mn ? gdn::sw128_mn_desc(b0, 8192) : gdn::sw128_desc(b0);
    if (a_tmem) {
      if (b_mn) gdn::mma_bf16_k4_ta<128>(tmem, tmem + 128, bd, id, 0);
      else gdn::mma_bf16_k4_ta<2>(tmem, tmem + 128, bd, id, 0);
    } else {
      if (b_mn) gdn::mma_bf16_k4<2, 128>(tmem, gdn::sw128_desc(gdn::smem_u32(sa)), bd, id, 0);
      else gdn::mma_bf16_k4<2, 2>(tmem, gdn::sw128_desc(gdn::smem_u32(sa)), bd, id, 0);
    }
    gdn::mma_commit(gdn::smem_u32(&bar));
  }
  const bool got = gdn::mbar_wait(gdn::smem_u32(&bar), 0, kWait);
  if (!got && tid == 0) atomicOr(status, 1u);
  const bool all = __syncthreads_and(got ? 1 : 0) != 0;
  gdn::tc_fence_after();
  if (all) {
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      gdn::tmem_ld32(tl + c0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) D[tid * N + c0 + i] = v[i];
    }
  }
  gdn::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    gdn::tc_fence_after();
    gdn::tmem_dealloc(tmem, 256);
  }
}

}  // namespace

extern "C" gdn_status gdn_debug_mma_probe_ex(const gdn_bf16* A, const gdn_bf16* B, int n_cols, int flags, float* D,
                                             unsigned* status, void* stream) {
  if (!A || !B || !D || !status || (flags & ~3)) return GDN_ERR_INVALID_ARGUMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (n_cols == 64) mma_probe_kernel<64><<<1, 128, 0, st>>>(A, B, D, status, flags);
  else if (n_cols == 128) mma_probe_kernel<128><<<1, 128, 0, st>>>(A, B, D, status, flags);
  else return GDN_ERR_INVALID_ARGUMENT;
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_debug_mma_probe(const gdn_bf16* A, const gdn_bf16* B, int n_cols, float* D,
                                          unsigned* status, void* stream) {
  return gdn_debug_mma_probe_ex(A, B, n_cols, 0, D, status, stream);
}
