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

// ---- the 64 x 64 unit-lower-triangular solve of the split path's prep kernels
constexpr uint32_t kTriBytes = 10 * 16 * 16 * 4;             // the 10 lower 16 x 16 blocks of a 64 x 64 fp32 matrix
constexpr uint32_t kYBytes = 32 * 32 * 4;                    // the solve's scratch products (32 x 32 fp32)
constexpr uint32_t kHeadBuf = 2 * kTriBytes + kYBytes;       // A, T and scratch of one V head (24 KB)

// A 64 x 64 fp32 lower block-triangular matrix (A, or its inverse T) is stored as its ten 16 x 16
// blocks on and below the diagonal (block row i, column j at index i (i + 1) / 2 + j), each
// row-major with the 16-byte groups of row r XOR-permuted by r & 3: float4 accesses of one row
// segment by 32 lanes that hold 32 consecutive rows spread over all banks.

// T_g = (I + A_g)^-1 for G <= kGroup strictly lower triangular 64 x 64 matrices at once (head g's
// A, T and scratch at base + g * kHeadBuf bytes), by two levels of 2 x 2 block inversion of a lower
// block-triangular matrix, [[M11, 0], [M21, M22]]^-1 = [[T11, 0], [-T22 M21 T11, T22]]:
//   1. the four diagonal 16 x 16 blocks by forward substitution (one column per thread);
//   2. in each diagonal 32 x 32 block, the block below the diagonal: T_ba = -T_bb (A_ba T_aa);
//   3. the lower-left 32 x 32 block: T_21 = -T_22 (A_21 T_11).
// The products of steps 2 and 3 are spread over every thread (one thread: four consecutive
// columns of one row, as f32x2 pairs), each through a scratch product and a CTA barrier: five
// barriers in all, against the block-column walk by one warp per column it replaces.  With kSub,
// only threads 0..63 run it (G = 1) and its barriers are a named barrier of those two warps, so
// the other warps of the CTA can work meanwhile.
template <bool kSub = false>
__device__ __forceinline__ void solve_sync() {
  if constexpr (kSub) asm volatile("bar.sync 1, 64;" ::: "memory");
  else __syncthreads();
}
template <bool kSub = false>
__device__ void solve_tri_batched(uint8_t* base, int G, int tid) {
  // Block (bi, bj) of a tri-layout matrix; inside it, element (r, c) sits at r * 16 +
  // ((((c >> 2) ^ (r & 3)) << 2) | (c & 3)).
  auto blk = [](const float* m, int bi, int bj) { return m + ((bi * (bi + 1)) / 2 + bj) * 256; };
  auto f4 = [](const float* p) { return *reinterpret_cast<const float4*>(p); };
  if (tid < 64 * G) {  // step 1: diagonal blocks, one column per thread; A rows read as float4
    const int g = tid >> 6, b = (tid >> 4) & 3, c = tid & 15;
    const float* Ab = blk(reinterpret_cast<const float*>(base + g * kHeadBuf), b, b);
    float* Tb = const_cast<float*>(blk(reinterpret_cast<const float*>(base + g * kHeadBuf + kTriBytes), b, b));
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == c) ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) {  // x_i -= sum_{k < i} A_ik x_k (x_k final by now)
      float a[16];
#pragma unroll
      for (int q = 0; q <= (i - 1) >> 2; ++q) {
        const float4 v = f4(Ab + i * 16 + ((q ^ (i & 3)) << 2));
        a[4 * q] = v.x; a[4 * q + 1] = v.y; a[4 * q + 2] = v.z; a[4 * q + 3] = v.w;
      }
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int k = 0; k < i; ++k) {
        if (k & 1) s1 = fmaf(a[k], x[k], s1);
        else s0 = fmaf(a[k], x[k], s0);
      }
      x[i] -= s0 + s1;
    }
    const int cq = c >> 2, ce = c & 3;
#pragma unroll
    for (int i = 0; i < 16; ++i) Tb[i * 16 + (((cq ^ (i & 3)) << 2) | ce)] = x[i];  // zeros above the diagonal too
  }
  solve_sync<kSub>();
  // Register-blocked products: a thread holds a 4 x 4 output tile -- rows rb, rb + S, rb + 2S,
  // rb + 3S (so that the lanes of a warp, consecutive in rb, read rows whose 16-byte groups sit
  // in different banks) and four consecutive columns -- and takes four k at a time: four float4
  // rows of the left operand, four float4 rows of the right one, 32 f32x2 multiply-adds.
  auto fma16 = [](const float4 (&a)[4], const float4 (&b)[4], float2 (&acc)[4][2]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float av[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 aa = make_float2(av[e], av[e]);
        acc[i][0] = __ffma2_rn(aa, make_float2(b[e].x, b[e].y), acc[i][0]);
        acc[i][1] = __ffma2_rn(aa, make_float2(b[e].z, b[e].w), acc[i][1]);
      }
    }
  };
  // step 2a: Y_h = A_{b+1,b} T_{b,b} (b = 2h), rows rb + 4i of the 16-row block; item (g, h, c4, rb)
  for (int it = tid; it < G * 32; it += kThreads) {
    const int g = it >> 5, b = ((it >> 4) & 1) * 2, cq = (it >> 2) & 3, rb = it & 3;
    const float* sA = reinterpret_cast<const float*>(base + g * kHeadBuf);
    const float* L = blk(sA, b + 1, b);
    const float* R = blk(sA + kTriBytes / 4, b, b);
    float* sY = reinterpret_cast<float*>(base + g * kHeadBuf + 2 * kTriBytes) + (b >> 1) * 256;
    float2 acc[4][2] = {};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = rb + 4 * i;
        a[i] = f4(L + r * 16 + ((q ^ (r & 3)) << 2));
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) bb[e] = f4(R + (4 * q + e) * 16 + ((cq ^ e) << 2));
      fma16(a, bb, acc);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(sY + (rb + 4 * i) * 16 + cq * 4) =
          make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
  }
  solve_sync<kSub>();
  // step 2b: T_{b+1,b} = -T_{b+1,b+1} Y_h
  for (int it = tid; it < G * 32; it += kThreads) {
    const int g = it >> 5, b = ((it >> 4) & 1) * 2, cq = (it >> 2) & 3, rb = it & 3;
    float* sT = reinterpret_cast<float*>(base + g * kHeadBuf + kTriBytes);
    const float* L = blk(sT, b + 1, b + 1);
    const float* sY = reinterpret_cast<const float*>(base + g * kHeadBuf + 2 * kTriBytes) + (b >> 1) * 256;
    float2 acc[4][2] = {};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = rb + 4 * i;
        a[i] = f4(L + r * 16 + ((q ^ (r & 3)) << 2));
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) bb[e] = f4(sY + (4 * q + e) * 16 + cq * 4);
      fma16(a, bb, acc);
    }
    float* D = const_cast<float*>(blk(sT, b + 1, b));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = rb + 4 * i;
      *reinterpret_cast<float4*>(D + r * 16 + ((cq ^ (r & 3)) << 2)) =
          make_float4(-acc[i][0].x, -acc[i][0].y, -acc[i][1].x, -acc[i][1].y);
    }
  }
  solve_sync<kSub>();
  // step 3a: Y = A_21 T_11 (rows 32..63 of A, columns 0..31), rows rb + 8i; T_11 is zero above its
  // diagonal blocks, so column block cb takes key blocks cb..1.  Item (g, c4, rb).
  for (int it = tid; it < G * 64; it += kThreads) {
    const int g = it >> 6, c4 = (it >> 3) & 7, rb = it & 7, cb = c4 >> 2, cq = c4 & 3;
    const float* sA = reinterpret_cast<const float*>(base + g * kHeadBuf);
    const float* sT = sA + kTriBytes / 4;
    float* sY = reinterpret_cast<float*>(base + g * kHeadBuf + 2 * kTriBytes);
    float2 acc[4][2] = {};
    for (int kb = cb; kb < 2; ++kb) {
      const float* R = blk(sT, kb, cb);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float4 a[4], bb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = rb + 8 * i, rr = r & 15;  // row 32 + r of A: block row 2 + r / 16
          a[i] = f4(blk(sA, 2 + (r >> 4), kb) + rr * 16 + ((q ^ (rr & 3)) << 2));
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) bb[e] = f4(R + (4 * q + e) * 16 + ((cq ^ e) << 2));
        fma16(a, bb, acc);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(sY + (rb + 8 * i) * 32 + c4 * 4) =
          make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
  }
  solve_sync<kSub>();
  // step 3b: T_21 = -T_22 Y; T_22 is zero above its diagonal blocks: rows 0..15 of it take Y's
  // first 16 rows, rows 16..31 all 32
  for (int it = tid; it < G * 64; it += kThreads) {
    const int g = it >> 6, c4 = (it >> 3) & 7, rb = it & 7, cb = c4 >> 2, cq = c4 & 3;
    float* sT = reinterpret_cast<float*>(base + g * kHeadBuf + kTriBytes);
    const float* sY = reinterpret_cast<const float*>(base + g * kHeadBuf + 2 * kTriBytes);
    float2 acc[4][2] = {};
#pragma unroll
    for (int ub = 0; ub < 2; ++ub) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float4 a[4], bb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = rb + 8 * i, rr = r & 15, rblk = r >> 4;  // row 32 + r: block row 2 + rblk
          // T_22 row r, key block ub: zero when ub > rblk (above the diagonal blocks)
          a[i] = (ub <= rblk) ? f4(blk(sT, 2 + rblk, 2 + ub) + rr * 16 + ((q ^ (rr & 3)) << 2))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) bb[e] = f4(sY + (16 * ub + 4 * q + e) * 32 + c4 * 4);
        fma16(a, bb, acc);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = rb + 8 * i, rr = r & 15;
      float* D = const_cast<float*>(blk(sT, 2 + (r >> 4), cb));
      *reinterpret_cast<float4*>(D + rr * 16 + ((cq ^ (rr & 3)) << 2)) =
          make_float4(-acc[i][0].x, -acc[i][0].y, -acc[i][1].x, -acc[i][1].y);
    }
  }
  solve_sync<kSub>();
}

}  // namespace
}  // namespace gdn
