// chunk_common.cuh -- device helpers shared by the chunk-wise prefill kernels (fused and split).
//
// Thread layout, operand-tile stores, the bf16 hi/lo split, the 64 x 64 fp32 solve layout and
// the blocked unit-lower-triangular inverse used for the WY form of the gated delta rule.
#pragma once

#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kParts = 2;                 // warps sharing one tensor-memory lane quarter
constexpr int kThreads = 128 * kParts;    // 8 warps
constexpr int kW = 64 / kParts;           // columns of a 64-wide accumulator per thread
constexpr int kWarps = kThreads / 32;

constexpr uint32_t kWaitLimit = 1u << 20;  // polls of one mbarrier before giving up
constexpr int kScheduleSortMax = 4096;     // longest-first ordering up to this many sequences
constexpr uint32_t kBytesQK = 4 * 64 * 128;  // four 64 x 64 bf16 boxes
constexpr uint32_t kBytesV = 2 * 64 * 128;
constexpr uint32_t kBytesZ = 64 * 256;

// Writes 8 consecutive fp32 values (columns k0..k0+7 of `row`, k0 % 8 == 0) as a bf16 hi (and
// optionally lo) pair into K-major 128-byte-swizzled tiles.
__device__ __forceinline__ void store8_split(uint8_t* hi_tile, uint8_t* lo_tile, uint32_t kb_stride, int row, int k0,
                                             const float* v) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = v[2 * i], b = v[2 * i + 1];
    h[i] = pack_bf2(a, b);
    if (lo_tile) l[i] = pack_bf2(a - __uint_as_float(h[i] << 16), b - __uint_as_float(h[i] & 0xFFFF0000u));
  }
  const uint32_t off = sw128_offset(row, k0, kb_stride);
  *reinterpret_cast<uint4*>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
  if (lo_tile) *reinterpret_cast<uint4*>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ float ld_bf(const uint8_t* base, uint32_t off) {
  return bf2f(*reinterpret_cast<const uint16_t*>(base + off));
}

// CUDA-core stand-in of one M=128 MMA group for verification: thread (row, part) computes
// columns [part*N/kParts, (part+1)*N/kParts) of row `row` of D (+)= A * B^T from the same
// swizzled tiles.
template <int N, int K>
__device__ void emu_mma(uint32_t t_lane, uint32_t col, const uint8_t* a_tile, uint32_t a_kbs, const uint8_t* b_tile,
                        uint32_t b_kbs, bool accumulate, int row, int part) {
  for (int n0 = part * (N / kParts); n0 < (part + 1) * (N / kParts); n0 += 16) {
    float d[16];
    if (accumulate) tmem_ld16(t_lane + col + n0, d);
    else {
#pragma unroll
      for (int i = 0; i < 16; ++i) d[i] = 0.f;
    }
    for (int n = 0; n < 16; ++n) {
      float s = 0.f;
      for (int k = 0; k < K; ++k)
        s = fmaf(ld_bf(a_tile, sw128_offset(row, k, a_kbs)), ld_bf(b_tile, sw128_offset(n0 + n, k, b_kbs)), s);
      d[n] += s;
    }
    tmem_st16(t_lane + col + n0, d);
  }
}

// Element (r, c) of the 64 x 64 fp32 inverse T: rows of 64 floats whose 16-byte groups are
// XOR-permuted by the row, so float4 reads of a row segment and float4 writes of a block row
// spread over the banks.
__device__ __forceinline__ int tidx(int r, int c) { return r * 64 + ((((c >> 2) ^ (r & 15)) & 15) << 2) + (c & 3); }

// Index of block pair (i, k), i > k, among the six strictly-lower 16 x 16 blocks.
__device__ __forceinline__ int pair_index(int i, int k) { return (i * (i - 1)) / 2 + k; }

// T = (I + A)^-1 for a strictly lower triangular 64 x 64 A, both in the tidx layout, by 16 x 16
// blocks (block row/column indices 0..3), in five barrier-separated steps:
//   1. T_ii = (I + A_ii)^-1 for the four diagonal blocks: right-looking forward substitution,
//      one column per thread held in registers;
//   2. B_ik = T_ii A_ik for the six blocks below the diagonal (all independent);
//   3-5. for block distance d = 1, 2, 3:  T_ij = - sum_{k=j}^{i-1} B_ik T_kj  (j = i - d),
// which is block forward substitution on (I + A) T = I with the diagonal blocks pre-inverted.
// Each 16 x 16 block product is split over two warps, a lane holding one row and four columns.
// The strictly upper blocks of T are never written; readers treat them as zero.
__device__ void solve_unit_lower(const float* sA, float* sT, float* sB, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  if (tid < 64) {
    const int b = tid >> 4, c = tid & 15, o = b * 16;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
    for (int k = 0; k < 15; ++k) {
      const float xk = x[k];
#pragma unroll
      for (int i = k + 1; i < 16; ++i) x[i] = fmaf(-sA[tidx(o + i, o + k)], xk, x[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sT[tidx(o + i, o + c)] = x[i];
  }
  __syncthreads();
  const int r = (warp & 1) * 8 + (lane >> 2);  // row inside the 16 x 16 block
  const int c0 = (lane & 3) * 4;               // first of this lane's four columns
  // step 2: twelve half-block tasks (six blocks x two row halves)
  for (int task = warp; task < 12; task += kWarps) {
    const int pidx = task >> 1;
    const int i = pidx < 1 ? 1 : (pidx < 3 ? 2 : 3), k = pidx - pair_index(i, 0);
    const int rr = (task & 1) * 8 + (lane >> 2);
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float a = sT[tidx(i * 16 + rr, i * 16 + u)];  // zero above the diagonal
      const float4 bv = *reinterpret_cast<const float4*>(sA + tidx(i * 16 + u, k * 16 + c0));
      acc0 = fmaf(a, bv.x, acc0);
      acc1 = fmaf(a, bv.y, acc1);
      acc2 = fmaf(a, bv.z, acc2);
      acc3 = fmaf(a, bv.w, acc3);
    }
    *reinterpret_cast<float4*>(sB + pidx * 320 + rr * 20 + c0) = make_float4(acc0, acc1, acc2, acc3);
  }
  __syncthreads();
  // steps 3-5
#pragma unroll
  for (int d = 1; d < 4; ++d) {
    const int nb = 4 - d;
    if (warp < 2 * nb) {
      const int i = d + (warp >> 1), jb = i - d;
      float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
      for (int kk = 0; kk < d; ++kk) {
        const int k = jb + kk;
        const float* Bik = sB + pair_index(i, k) * 320 + r * 20;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float a = Bik[u];
          const float4 bv = *reinterpret_cast<const float4*>(sT + tidx(k * 16 + u, jb * 16 + c0));
          acc0 = fmaf(a, bv.x, acc0);
          acc1 = fmaf(a, bv.y, acc1);
          acc2 = fmaf(a, bv.z, acc2);
          acc3 = fmaf(a, bv.w, acc3);
        }
      }
      *reinterpret_cast<float4*>(sT + tidx(i * 16 + r, jb * 16 + c0)) = make_float4(-acc0, -acc1, -acc2, -acc3);
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace gdn
