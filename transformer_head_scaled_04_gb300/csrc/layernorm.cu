// layernorm.cu -- y = LayerNorm(x + a) * gamma + beta, the residual + post-norm step of the
// sublayer ("Attention Is All You Need", lettle.cn translation, 3.1 Encoder and Decoder
// Stacks: LayerNorm(x + Sublayer(x)); "Transformer：抛弃循环与卷积的序列建模", Residual
// Connection 与 LayerNorm).  Mean and biased variance over the row, eps inside the root.
//
// HBM-bound: one warp per row, each lane moves 16-byte vectors (8 bf16 or 2x4 fp32) so a warp
// reads 512 contiguous bytes per step; the row stays in registers between the two statistic
// passes (mean, then the sum of squared deviations) and the normalising write.
#include <cuda_bf16.h>

#include <algorithm>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kRowsPerBlock = 8;
constexpr int kSiteLnCols = 31;  // index check (MHA_DEBUG_BOUNDS builds): a row's 8-column span

template <typename T>
struct Vec8;
template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
  }
};
template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[8]) {
    float4 a = reinterpret_cast<const float4*>(p)[0];
    float4 b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};

template <typename T, int NIT>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
    residual_layernorm_kernel(const T* __restrict__ x, const T* __restrict__ a,
                              const T* __restrict__ gamma, const T* __restrict__ beta,
                              T* __restrict__ y, int M, int D, float eps, int* status) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp;
  if (row >= M) return;
  const int64_t base = static_cast<int64_t>(row) * D;
  float r[NIT][8];
  float sum = 0.f;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int col = (it * 32 + lane) * 8;
    if (col < D && span_ok(col, 8, D, status, kSiteLnCols)) {
      float xv[8], av[8];
      Vec8<T>::load(x + base + col, xv);
      Vec8<T>::load(a + base + col, av);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        r[it][e] = xv[e] + av[e];
        sum += r[it][e];
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float mean = sum / static_cast<float>(D);
  float sq = 0.f;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int col = (it * 32 + lane) * 8;
    if (col < D) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = r[it][e] - mean;
        sq = fmaf(d, d, sq);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  const float rstd = 1.0f / sqrtf(sq / static_cast<float>(D) + eps);
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int col = (it * 32 + lane) * 8;
    if (col < D && span_ok(col, 8, D, status, kSiteLnCols)) {
      float g[8], bt[8], out[8];
      if (gamma) {
        Vec8<T>::load(gamma + col, g);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = 1.f;
      }
      if (beta) {
        Vec8<T>::load(beta + col, bt);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) bt[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) out[e] = (r[it][e] - mean) * rstd * g[e] + bt[e];
      Vec8<T>::store(y + base + col, out);
    }
  }
}

// bf16 rows, persistent: warp w of the grid takes rows w, w + W, w + 2W, ... (W warps in the
// grid) and asks L2 for its next row of x and a (one bulk prefetch each) before it loads and
// normalises the current one, so the loads of the current row mostly hit L2 and DRAM keeps
// far more bytes in flight than the registers of the resident warps could hold.
template <int NIT>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
    residual_layernorm_stream_kernel(const __nv_bfloat16* __restrict__ x,
                                     const __nv_bfloat16* __restrict__ a,
                                     const __nv_bfloat16* __restrict__ gamma,
                                     const __nv_bfloat16* __restrict__ beta,
                                     __nv_bfloat16* __restrict__ y, int M, int D, float eps,
                                     int* status) {
  const int lane = threadIdx.x & 31;
  const int W = gridDim.x * kRowsPerBlock;
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output (a) is complete from here on
  int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  const uint32_t row_bytes = static_cast<uint32_t>(D) * 2;
  if (lane == 0 && row < M) {
    prefetch_l2(x + static_cast<int64_t>(row) * D, row_bytes);
    prefetch_l2(a + static_cast<int64_t>(row) * D, row_bytes);
  }
  for (; row < M; row += W) {
    const int nxt = row + W;
    if (lane == 0 && nxt < M) {
      prefetch_l2(x + static_cast<int64_t>(nxt) * D, row_bytes);
      prefetch_l2(a + static_cast<int64_t>(nxt) * D, row_bytes);
    }
    const int64_t base = static_cast<int64_t>(row) * D;
    float r[NIT][8];
    float sum = 0.f;
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int col = (it * 32 + lane) * 8;
      if (col < D && span_ok(col, 8, D, status, kSiteLnCols)) {
        float xv[8], av[8];
        Vec8<__nv_bfloat16>::load(x + base + col, xv);
        Vec8<__nv_bfloat16>::load(a + base + col, av);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          r[it][e] = xv[e] + av[e];
          sum += r[it][e];
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float mean = sum / static_cast<float>(D);
    float sq = 0.f;
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int col = (it * 32 + lane) * 8;
      if (col < D) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float d = r[it][e] - mean;
          sq = fmaf(d, d, sq);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
    const float rstd = 1.0f / sqrtf(sq / static_cast<float>(D) + eps);
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int col = (it * 32 + lane) * 8;
      if (col < D && span_ok(col, 8, D, status, kSiteLnCols)) {
        float g[8], bt[8], out[8];
        if (gamma) {
          Vec8<__nv_bfloat16>::load(gamma + col, g);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) g[e] = 1.f;
        }
        if (beta) {
          Vec8<__nv_bfloat16>::load(beta + col, bt);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) bt[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = (r[it][e] - mean) * rstd * g[e] + bt[e];
        Vec8<__nv_bfloat16>::store(y + base + col, out);
      }
    }
  }
}

cudaError_t launch_stream(int M, int D, float eps, const void* x, const void* a,
                          const void* gamma, const void* beta, void* y, const DevCtx& ctx,
                          cudaStream_t s) {
  const int blocks = (M + kRowsPerBlock - 1) / kRowsPerBlock;
  const int grid = std::min(blocks, 4 * std::max(ctx.num_sms, 1));  // 4 blocks fit an SM
  auto go = [&](auto kern) {
    return launch_pdl(kern, dim3(grid), dim3(kRowsPerBlock * 32), 0, s,
                      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(a),
                      static_cast<const __nv_bfloat16*>(gamma),
                      static_cast<const __nv_bfloat16*>(beta), static_cast<__nv_bfloat16*>(y),
                      M, D, eps, ctx.status);
  };
  switch ((D + 255) / 256) {
    case 1: return go(residual_layernorm_stream_kernel<1>);
    case 2: return go(residual_layernorm_stream_kernel<2>);
    case 3: return go(residual_layernorm_stream_kernel<3>);
    case 4: return go(residual_layernorm_stream_kernel<4>);
    case 5: return go(residual_layernorm_stream_kernel<5>);
    case 6: return go(residual_layernorm_stream_kernel<6>);
    case 7: return go(residual_layernorm_stream_kernel<7>);
    default: return go(residual_layernorm_stream_kernel<8>);
  }
}

template <typename T>
cudaError_t launch_t(int M, int D, float eps, const void* x, const void* a, const void* gamma,
                     const void* beta, void* y, int* status, cudaStream_t s) {
  const int nit = (D + 255) / 256;
  dim3 grid((M + kRowsPerBlock - 1) / kRowsPerBlock);
  dim3 block(kRowsPerBlock * 32);
  auto args = [&](auto kern) {
    (void)launch_pdl(kern, dim3(grid), dim3(block), 0, s, static_cast<const T*>(x), static_cast<const T*>(a),
                                static_cast<const T*>(gamma), static_cast<const T*>(beta),
                                static_cast<T*>(y), M, D, eps, status);
  };
  switch (nit) {
    case 1: args(residual_layernorm_kernel<T, 1>); break;
    case 2: args(residual_layernorm_kernel<T, 2>); break;
    case 3: args(residual_layernorm_kernel<T, 3>); break;
    case 4: args(residual_layernorm_kernel<T, 4>); break;
    case 5: args(residual_layernorm_kernel<T, 5>); break;
    case 6: args(residual_layernorm_kernel<T, 6>); break;
    case 7: args(residual_layernorm_kernel<T, 7>); break;
    default: args(residual_layernorm_kernel<T, 8>); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_residual_layernorm(int dtype, int M, int D, float eps, const void* x,
                                      const void* a, const void* gamma, const void* beta,
                                      void* y, const DevCtx& ctx, cudaStream_t s) {
  if (dtype == 1) return launch_stream(M, D, eps, x, a, gamma, beta, y, ctx, s);
  return launch_t<float>(M, D, eps, x, a, gamma, beta, y, ctx.status, s);
}

}  // namespace mha
