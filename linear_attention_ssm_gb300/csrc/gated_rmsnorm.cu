// gated_rmsnorm.cu -- sigmoid-gated RMSNorm, one row of Dv = 128 per (token, V head).
//
// pegainfer PR #1152 "Reference golden for the GDN sublayer", Summary (output_gate_type
// "sigmoid"; the in-tree kernel that hard-codes silu is the trap) and Code review item 6
// (rms_norm_eps == 1e-6):  out = o * (mean(o^2) + eps)^(-1/2) * w * sigmoid(z).
// Memory-bound: 16 lanes per row, one 16-byte vector of o and z per lane, shuffle reduction.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(256) gated_rmsnorm_kernel(const uint16_t* o, const uint16_t* __restrict__ z,
                                                            const uint16_t* __restrict__ w, float eps,
                                                            uint16_t* out, long rows) {
  const long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 4;
  const int sub = threadIdx.x & 15;
  const bool valid = row < rows;
  float ov[8] = {0, 0, 0, 0, 0, 0, 0, 0}, zv[8], wv[8];
  if (valid) {
    unpack8(*reinterpret_cast<const uint4*>(o + row * kHeadDim + sub * 8), ov);
    unpack8(__ldg(reinterpret_cast<const uint4*>(z + row * kHeadDim + sub * 8)), zv);
    unpack8(__ldg(reinterpret_cast<const uint4*>(w + sub * 8)), wv);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(ov[i], ov[i], ss);
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  if (!valid) return;
  const float rstd = rsqrtf(ss * (1.0f / kHeadDim) + eps);
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 8; i += 2)
    p[i >> 1] = pack_bf2(ov[i] * rstd * wv[i] * sigmoidf_(zv[i]),
                         ov[i + 1] * rstd * wv[i + 1] * sigmoidf_(zv[i + 1]));
  *reinterpret_cast<uint4*>(out + row * kHeadDim + sub * 8) = make_uint4(p[0], p[1], p[2], p[3]);
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const LaunchEnv& env, const uint16_t* o, const uint16_t* z, const uint16_t* w,
                                 float eps, uint16_t* out, long rows) {
  if (rows <= 0) return cudaSuccess;
  const int threads = 256;  // 16 rows per block
  const long blocks = (rows * 16 + threads - 1) / threads;
  gated_rmsnorm_kernel<<<(unsigned)blocks, threads, 0, env.stream>>>(o, z, w, eps, out, rows);
  return cudaGetLastError();
}

}  // namespace gdn
