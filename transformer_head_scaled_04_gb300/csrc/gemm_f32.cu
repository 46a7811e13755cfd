// gemm_f32.cu -- Y[M,N] = act(X[M,K] W[N,K]^T + bias[N]) in fp32 FFMA (SIMT, no TF32),
// act = identity or ReLU.
// The fp32 variant of the sublayers' projections ("Attention Is All You Need", lettle.cn
// translation, 3.2.2 多头注意力; "Attention Is All You Need" on likecs.com, 1.3 按地址的前向
// 反馈网络).  64x64 output tile per 256-thread block, 4x4 per thread, K staged through
// shared memory 16 at a time.
#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kT = 64;
constexpr int kKT = 16;

__global__ void __launch_bounds__(256)
    gemm_f32_kernel(const float* __restrict__ X, int64_t ldx, const float* __restrict__ W,
                    const float* __restrict__ bias, bool relu, float* __restrict__ Y,
                    int64_t ldy, int M, int N, int K, const float* __restrict__ R) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  __shared__ float sx[kKT][kT + 4];
  __shared__ float sw[kKT][kT + 4];
  const int tx = threadIdx.x & 15;  // column group
  const int ty = threadIdx.x >> 4;  // row group
  const int m0 = blockIdx.y * kT;
  const int n0 = blockIdx.x * kT;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kKT) {
    for (int i = threadIdx.x; i < kT * kKT; i += 256) {
      const int r = i / kKT;
      const int kk = i % kKT;
      const int gm = m0 + r, gn = n0 + r, gk = k0 + kk;
      sx[kk][r] = (gm < M && gk < K) ? X[static_cast<int64_t>(gm) * ldx + gk] : 0.f;
      sw[kk][r] = (gn < N && gk < K) ? W[static_cast<int64_t>(gn) * K + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kKT; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = sx[kk][ty * 4 + i];
        w[i] = sw[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jn = 0; jn < 4; ++jn) acc[i][jn] = fmaf(a[i], w[jn], acc[i][jn]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int jn = 0; jn < 4; ++jn) {
      const int gn = n0 + tx * 4 + jn;
      if (gn >= N) continue;
      const float v = acc[i][jn] + (bias ? bias[gn] : 0.f) +
                      (R ? R[static_cast<int64_t>(gm) * ldy + gn] : 0.f);
      Y[static_cast<int64_t>(gm) * ldy + gn] = relu ? fmaxf(v, 0.f) : v;
    }
  }
}

}  // namespace

cudaError_t launch_gemm_f32(const float* X, int64_t ldx, const float* W, const float* bias,
                            bool relu, float* Y, int64_t ldy, int M, int N, int K,
                            cudaStream_t s, const float* R) {
  dim3 grid((N + kT - 1) / kT, (M + kT - 1) / kT);
  (void)launch_pdl(gemm_f32_kernel, dim3(grid), dim3(256), 0, s, X, ldx, W, bias, relu, Y, ldy, M, N, K, R);
  return cudaGetLastError();
}

}  // namespace mha
