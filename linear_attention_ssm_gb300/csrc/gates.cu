// gates.cu -- the gates of the gated delta rule from their projections: for every (row, V head)
//   g = -exp(A_log[h]) softplus(a + dt_bias[h]),   beta = sigmoid(b)
// The pages name the inputs (Qwen3.8 kernel architecture and TDD ledger, "GDN alpha/beta
// transforms"; pegainfer PR #1152 Summary: A_log, dt_bias, the a / b projections) but give no
// formula; this is the gate of the published Gated DeltaNet / Mamba-2 layers.  Elementwise (2 bf16
// read, 2 fp32 written per element); a grid-stride loop over octets of elements.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

// 8 consecutive elements per thread and iteration when Hv % 8 == 0 (an octet never crosses a row:
// 16-byte loads of a and b, two 16-byte stores each of g and beta); one element otherwise.
__global__ void __launch_bounds__(256) gates_kernel(const uint16_t* __restrict__ a, const uint16_t* __restrict__ b,
                                                    const float* __restrict__ A_log,
                                                    const float* __restrict__ dt_bias, float* __restrict__ g,
                                                    float* __restrict__ beta, long n, int hv) {
  const long stride = (long)gridDim.x * blockDim.x;
  if ((hv & 7) == 0) {
    for (long o = (long)blockIdx.x * blockDim.x + threadIdx.x; o < n / 8; o += stride) {
      const long i = o * 8;
      const int h0 = (int)(i % hv);
      const uint4 au = __ldg(reinterpret_cast<const uint4*>(a + i));
      const uint4 bu = __ldg(reinterpret_cast<const uint4*>(b + i));
      const uint32_t aw[4] = {au.x, au.y, au.z, au.w}, bw[4] = {bu.x, bu.y, bu.z, bu.w};
      float gv[8], bv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t wa = aw[e >> 1], wb = bw[e >> 1];
        const float av = __uint_as_float((e & 1) ? (wa & 0xFFFF0000u) : (wa << 16));
        const float bvv = __uint_as_float((e & 1) ? (wb & 0xFFFF0000u) : (wb << 16));
        gate_one(av, bvv, __ldg(A_log + h0 + e), __ldg(dt_bias + h0 + e), gv[e], bv[e]);
      }
      float4* gp = reinterpret_cast<float4*>(g + i);
      float4* bp = reinterpret_cast<float4*>(beta + i);
      gp[0] = make_float4(gv[0], gv[1], gv[2], gv[3]);
      gp[1] = make_float4(gv[4], gv[5], gv[6], gv[7]);
      bp[0] = make_float4(bv[0], bv[1], bv[2], bv[3]);
      bp[1] = make_float4(bv[4], bv[5], bv[6], bv[7]);
    }
  } else {
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
      const int h = (int)(i % hv);
      gate_one(bf2f(__ldg(a + i)), bf2f(__ldg(b + i)), __ldg(A_log + h), __ldg(dt_bias + h), g[i], beta[i]);
    }
  }
}

}  // namespace

cudaError_t launch_gates(const LaunchEnv& env, const uint16_t* a, const uint16_t* b, const float* A_log,
                         const float* dt_bias, float* g, float* beta, long rows, int hv) {
  const long n = rows * hv;
  if (n <= 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const long work = (hv & 7) == 0 ? n / 8 : n;  // threads' items
  const long blocks = (work + 255) / 256;
  const long cap = 8L * (sms > 0 ? sms : 1);  // a few waves of 256-thread blocks; the loop strides over the rest
  gates_kernel<<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, env.stream>>>(a, b, A_log, dt_bias, g, beta, n, hv);
  return cudaGetLastError();
}

}  // namespace gdn
