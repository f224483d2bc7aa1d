// gates.cu -- the gates of the gated delta rule from their projections: for every (row, V head)
//   g = -exp(A_log[h]) softplus(a + dt_bias[h]),   beta = sigmoid(b)
// The pages name the inputs (Qwen3.8 kernel architecture and TDD ledger, "GDN alpha/beta
// transforms"; pegainfer PR #1152 Summary: A_log, dt_bias, the a / b projections) but give no
// formula; this is the gate of the published Gated DeltaNet / Mamba-2 layers.  Elementwise and
// HBM-bound (2 bf16 read, 2 fp32 written per element); a grid-stride loop over the elements.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

__global__ void __launch_bounds__(256) gates_kernel(const uint16_t* __restrict__ a, const uint16_t* __restrict__ b,
                                                    const float* __restrict__ A_log,
                                                    const float* __restrict__ dt_bias, float* __restrict__ g,
                                                    float* __restrict__ beta, long n, int hv) {
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const int h = (int)(i % hv);
    const float x = bf2f(__ldg(a + i)) + __ldg(dt_bias + h);
    const float sp = x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));  // log(1 + e^x), no overflow
    g[i] = -expf(__ldg(A_log + h)) * sp;
    beta[i] = 1.0f / (1.0f + expf(-bf2f(__ldg(b + i))));
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
  const long blocks = (n + 255) / 256;
  const long cap = 8L * (sms > 0 ? sms : 1);  // a few waves of 256-thread blocks; the loop strides over the rest
  gates_kernel<<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, env.stream>>>(a, b, A_log, dt_bias, g, beta, n, hv);
  return cudaGetLastError();
}

}  // namespace gdn
