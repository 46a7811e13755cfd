// bwd_util.cu -- the memory-bound steps of the sublayer's backward pass ("Transformer：抛弃
// 循环与卷积的序列建模", Transformer 训练样例 > 反向传播: the chain rule back through the
// residual + LayerNorm step of "Attention Is All You Need", lettle.cn translation, 3.1).
//
//   layernorm_bwd: with r = x + a, rhat = (r - mean) * rstd, g = dy * gamma:
//                  dr = (g - mean(g) - rhat * mean(g * rhat)) * rstd   (one warp per row;
//                  also keeps each row's mean and rstd for the parameter gradients)
//   ln_param_partials + reduce_partials: dgamma = sum dy * rhat, dbeta = sum dy and
//                  db_o = sum dr over all rows, summed per chunk of rows and then over the
//                  chunks in a fixed order (deterministic)
//   colsum_partials + reduce_partials: a bias gradient, the column sums of a gradient matrix
//   transpose: Y = X^T with the reduced dimension padded by zero rows to a whole number of
//                  64-wide K slices, so the weight-gradient products run on the same GEMM
//                  (bf16: 64 x 64 tiles moved as 16-byte vectors)
#include <cuda_bf16.h>

#include <cstdint>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

template <typename T>
__device__ __forceinline__ float ldf(const T* p) {
  if constexpr (sizeof(T) == 2)
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
  else
    return static_cast<float>(*p);
}
template <typename T>
__device__ __forceinline__ T stf(float v) {
  if constexpr (sizeof(T) == 2)
    return __float2bfloat16_rn(v);
  else
    return v;
}

constexpr int kRows = 8;  // rows (warps) per block in the row kernels

// one warp per row, D <= 32 * NIT
template <typename T, int NIT>
__global__ void __launch_bounds__(kRows * 32)
    layernorm_bwd_kernel(const T* __restrict__ x, const T* __restrict__ a,
                         const T* __restrict__ gamma, const T* __restrict__ dy,
                         T* __restrict__ dr, float2* __restrict__ stats, int M, int D,
                         float eps) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRows + warp;
  if (row >= M) return;
  const int64_t base = static_cast<int64_t>(row) * D;
  float r[NIT], g[NIT];
  float sum = 0.f;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int col = it * 32 + lane;
    r[it] = 0.f;
    g[it] = 0.f;
    if (col < D) {
      r[it] = ldf(x + base + col) + ldf(a + base + col);
      g[it] = ldf(dy + base + col) * (gamma ? ldf(gamma + col) : 1.f);
      sum += r[it];
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float mean = sum / static_cast<float>(D);
  float sq = 0.f;
#pragma unroll
  for (int it = 0; it < NIT; ++it)
    if (it * 32 + lane < D) sq = fmaf(r[it] - mean, r[it] - mean, sq);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  const float rstd = 1.0f / sqrtf(sq / static_cast<float>(D) + eps);
  float sg = 0.f, sgr = 0.f;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    if (it * 32 + lane < D) {
      r[it] = (r[it] - mean) * rstd;  // rhat
      sg += g[it];
      sgr = fmaf(g[it], r[it], sgr);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sg += __shfl_xor_sync(0xffffffffu, sg, off);
    sgr += __shfl_xor_sync(0xffffffffu, sgr, off);
  }
  const float mg = sg / static_cast<float>(D), mgr = sgr / static_cast<float>(D);
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int col = it * 32 + lane;
    if (col < D) dr[base + col] = stf<T>((g[it] - mg - r[it] * mgr) * rstd);
  }
  if (lane == 0) stats[row] = make_float2(mean, rstd);
}

// rows [chunk * rows_per_chunk, ...) of columns [blockIdx.x * 256 + threadIdx.x]: partial
// sums of dy * rhat, dy and dr, written to part[(chunk * 3 + k) * D + col]
template <typename T>
__global__ void __launch_bounds__(256)
    ln_param_partials_kernel(const T* __restrict__ x, const T* __restrict__ a,
                             const T* __restrict__ dy, const T* __restrict__ dr,
                             const float2* __restrict__ stats, float* __restrict__ part, int M,
                             int D, int rows_per_chunk) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  const int col = blockIdx.x * 256 + threadIdx.x;
  const int chunk = blockIdx.y;
  if (col >= D) return;
  const int r0 = chunk * rows_per_chunk, r1 = min(r0 + rows_per_chunk, M);
  float sg = 0.f, sb = 0.f, sd = 0.f;
  for (int r = r0; r < r1; ++r) {
    const int64_t i = static_cast<int64_t>(r) * D + col;
    const float2 st = stats[r];
    const float rhat = (ldf(x + i) + ldf(a + i) - st.x) * st.y;
    const float d = ldf(dy + i);
    sg = fmaf(d, rhat, sg);
    sb += d;
    sd += ldf(dr + i);
  }
  float* p = part + static_cast<int64_t>(chunk) * 3 * D + col;
  p[0] = sg;
  p[D] = sb;
  p[2 * D] = sd;
}

// column sums of X [M, N] (row pitch ld) over chunks of rows: part[chunk * N + col]
template <typename T>
__global__ void __launch_bounds__(256)
    colsum_partials_kernel(const T* __restrict__ X, int64_t ld, int M, int N,
                           int rows_per_chunk, float* __restrict__ part) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  const int col = blockIdx.x * 256 + threadIdx.x;
  const int chunk = blockIdx.y;
  if (col >= N) return;
  const int r0 = chunk * rows_per_chunk, r1 = min(r0 + rows_per_chunk, M);
  float s = 0.f;
  for (int r = r0; r < r1; ++r) s += ldf(X + static_cast<int64_t>(r) * ld + col);
  part[static_cast<int64_t>(chunk) * N + col] = s;
}

// out_t[col] = sum over chunks of part[t * term_stride + chunk * chunk_stride + col] for the
// term t = blockIdx.y (up to three outputs per launch); chunk c goes to partial sum c % 4 and
// the four are added in a fixed order (deterministic)
template <typename T>
__global__ void __launch_bounds__(256)
    reduce_partials_kernel(const float* __restrict__ part, int nchunk, int64_t chunk_stride,
                           int N, int64_t term_stride, T* __restrict__ out0,
                           T* __restrict__ out1, T* __restrict__ out2) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  const int col = blockIdx.x * 256 + threadIdx.x;
  if (col >= N) return;
  const int t = blockIdx.y;
  T* out = t == 0 ? out0 : (t == 1 ? out1 : out2);
  const float* p = part + t * term_stride + col;
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
  int c = 0;
  for (; c + 4 <= nchunk; c += 4) {
#pragma unroll
    for (int q = 0; q < 4; ++q) s4[q] += p[static_cast<int64_t>(c + q) * chunk_stride];
  }
  for (int q = 0; c < nchunk; ++c, ++q) s4[q] += p[static_cast<int64_t>(c) * chunk_stride];
  out[col] = stf<T>((s4[0] + s4[1]) + (s4[2] + s4[3]));
}

// Y[c * ldy + r] = X[r * ldx + c] for r < R, c < C; rows R <= r < R_pad of Y's columns are 0
template <typename T>
__global__ void __launch_bounds__(256)
    transpose_kernel(const T* __restrict__ X, int64_t ldx, int R, int C, T* __restrict__ Y,
                     int64_t ldy, int R_pad) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  __shared__ T tile[32][33];
  const int r0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int k = ty; k < 32; k += 8) {
    const int r = r0 + k, c = c0 + tx;
    tile[k][tx] = (r < R && c < C) ? X[static_cast<int64_t>(r) * ldx + c] : stf<T>(0.f);
  }
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    const int c = c0 + k, r = r0 + tx;
    if (c < C && r < R_pad) Y[static_cast<int64_t>(c) * ldy + r] = tile[tx][k];
  }
}

// ---- bf16 with 16-byte vectors (D, N, ld multiples of 8; 16-byte aligned rows)
__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// layernorm_bwd for bf16: one warp per row, each lane 8 consecutive features per 256
template <int NIT>
__global__ void __launch_bounds__(kRows * 32)
    layernorm_bwd_v8_kernel(const __nv_bfloat16* __restrict__ x,
                            const __nv_bfloat16* __restrict__ a,
                            const __nv_bfloat16* __restrict__ gamma,
                            const __nv_bfloat16* __restrict__ dy, __nv_bfloat16* __restrict__ dr,
                            float2* __restrict__ stats, int M, int D, float eps) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRows + warp;
  if (row >= M) return;
  const int64_t base = static_cast<int64_t>(row) * D;
  float r[NIT][8], g[NIT][8];
  float sum = 0.f;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int col = (it * 32 + lane) * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) r[it][e] = g[it][e] = 0.f;
    if (col < D) {
      float xv[8], av[8], dv[8], gv[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + base + col), xv);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(a + base + col), av);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(dy + base + col), dv);
      if (gamma) {
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(gamma + col)), gv);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) gv[e] = 1.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        r[it][e] = xv[e] + av[e];
        g[it][e] = dv[e] * gv[e];
        sum += r[it][e];
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float mean = sum / static_cast<float>(D);
  float sq = 0.f;
#pragma unroll
  for (int it = 0; it < NIT; ++it)
    if ((it * 32 + lane) * 8 < D) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sq = fmaf(r[it][e] - mean, r[it][e] - mean, sq);
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  const float rstd = 1.0f / sqrtf(sq / static_cast<float>(D) + eps);
  float sg = 0.f, sgr = 0.f;
#pragma unroll
  for (int it = 0; it < NIT; ++it)
    if ((it * 32 + lane) * 8 < D) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        r[it][e] = (r[it][e] - mean) * rstd;  // rhat
        sg += g[it][e];
        sgr = fmaf(g[it][e], r[it][e], sgr);
      }
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sg += __shfl_xor_sync(0xffffffffu, sg, off);
    sgr += __shfl_xor_sync(0xffffffffu, sgr, off);
  }
  const float mg = sg / static_cast<float>(D), mgr = sgr / static_cast<float>(D);
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const int col = (it * 32 + lane) * 8;
    if (col < D) {
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = (g[it][e] - mg - r[it][e] * mgr) * rstd;
      *reinterpret_cast<uint4*>(dr + base + col) = f32_to_bf16x8(o);
    }
  }
  if (lane == 0) stats[row] = make_float2(mean, rstd);
}

// Column partial sums over a chunk of rows for bf16, 8 consecutive columns per thread:
// blockDim (kCols, kGroups); row group y takes rows r0 + y, r0 + y + kGroups, ...; the
// groups' sums are added in group order (deterministic).  kTerms = 3: dy * rhat, dy and dr
// (LayerNorm parameters and db_o); kTerms = 1: the column sums of X (a bias gradient).
template <int kTerms, int kCols, int kGroups>
__global__ void __launch_bounds__(kCols * kGroups)
    colsum_v8_kernel(const __nv_bfloat16* __restrict__ X, int64_t ld,
                     const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ a,
                     const __nv_bfloat16* __restrict__ dr, const float2* __restrict__ stats,
                     int M, int N, int rows_per_chunk, float* __restrict__ part) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  __shared__ float red[kGroups - 1][kTerms][kCols * 8];
  const int col = (blockIdx.x * kCols + threadIdx.x) * 8;
  const int chunk = blockIdx.y, grp = threadIdx.y;
  const int r0 = chunk * rows_per_chunk, r1 = min(r0 + rows_per_chunk, M);
  float acc[kTerms][8];
#pragma unroll
  for (int k = 0; k < kTerms; ++k)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[k][e] = 0.f;
  if (col < N) {
    for (int r = r0 + grp; r < r1; r += kGroups) {
      float d[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(X + static_cast<int64_t>(r) * ld + col), d);
      if (kTerms == 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[0][e] += d[e];
      } else {
        const int64_t i = static_cast<int64_t>(r) * N + col;
        const float2 st = stats[r];
        float xv[8], av[8], rv[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + i), xv);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(a + i), av);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(dr + i), rv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc[0][e] = fmaf(d[e], (xv[e] + av[e] - st.x) * st.y, acc[0][e]);
          acc[1][e] += d[e];
          acc[kTerms - 1][e] += rv[e];
        }
      }
    }
  }
  if (grp > 0) {
#pragma unroll
    for (int k = 0; k < kTerms; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) red[grp - 1][k][threadIdx.x * 8 + e] = acc[k][e];
  }
  __syncthreads();
  if (grp == 0 && col < N) {
#pragma unroll
    for (int k = 0; k < kTerms; ++k) {
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float v = acc[k][e];
#pragma unroll
        for (int q = 0; q < kGroups - 1; ++q) v += red[q][k][threadIdx.x * 8 + e];
        o[e] = v;
      }
      float4* dst = reinterpret_cast<float4*>(part + (static_cast<int64_t>(chunk) * kTerms + k) * N + col);
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
    }
  }
}

// bf16, 64 x 64 tiles moved as 16-byte vectors: each thread loads 8 consecutive elements of a
// row of X, and stores 8 consecutive elements of a row of Y gathered from 8 rows of the tile
// (row pitch 66 elements: both the 4-byte writes and the 2-byte gathers are conflict-free).
// Needs C, ldx, ldy and R_pad multiples of 8 and 16-byte aligned X and Y.
constexpr int kTp = 64;
constexpr int kTpPitch = kTp + 2;
__global__ void __launch_bounds__(256)
    transpose_v8_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx, int R, int C,
                        __nv_bfloat16* __restrict__ Y, int64_t ldy, int R_pad) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  __shared__ uint16_t tile[kTp * kTpPitch];
  const int r0 = blockIdx.x * kTp, c0 = blockIdx.y * kTp;
  const int t = threadIdx.x;
  const int sub = (t & 7) * 8;  // 8-element chunk within a 64-wide row
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int row = (t >> 3) + 32 * pass;
    const int r = r0 + row, c = c0 + sub;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);  // rows past R read as zeros (the padding)
    if (r < R && c < C) v = *reinterpret_cast<const uint4*>(X + static_cast<int64_t>(r) * ldx + c);
    uint32_t* d = reinterpret_cast<uint32_t*>(tile + row * kTpPitch + sub);
    d[0] = v.x;
    d[1] = v.y;
    d[2] = v.z;
    d[3] = v.w;
  }
  __syncthreads();
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int oc = (t >> 3) + 32 * pass;  // row of Y = column of X
    const int c = c0 + oc, r = r0 + sub;
    if (c < C && r < R_pad) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = static_cast<uint32_t>(tile[(sub + 2 * i) * kTpPitch + oc]) |
               (static_cast<uint32_t>(tile[(sub + 2 * i + 1) * kTpPitch + oc]) << 16);
      *reinterpret_cast<uint4*>(Y + static_cast<int64_t>(c) * ldy + r) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

constexpr int kChunkRows = 256;

}  // namespace

int bwd_row_chunks(int M) { return (M + kChunkRows - 1) / kChunkRows; }

cudaError_t launch_layernorm_bwd(int dtype, int M, int D, float eps, const void* x,
                                 const void* a, const void* gamma, const void* dy, void* dr,
                                 float2* stats, float* part, cudaStream_t s) {
  const dim3 grid_rows((M + kRows - 1) / kRows);
  const int nit = (D + 31) / 32;
  const dim3 grid_cols((D + 255) / 256, bwd_row_chunks(M));
  auto al16 = [](const void* q) { return q == nullptr || reinterpret_cast<uintptr_t>(q) % 16 == 0; };
  if (dtype == 1 && D % 8 == 0 && D <= 2048 && al16(x) && al16(a) && al16(gamma) && al16(dy) &&
      al16(dr)) {
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const auto* ab = static_cast<const __nv_bfloat16*>(a);
    const auto* gb = static_cast<const __nv_bfloat16*>(gamma);
    const auto* dyb = static_cast<const __nv_bfloat16*>(dy);
    auto* drb = static_cast<__nv_bfloat16*>(dr);
    switch ((D + 255) / 256) {
      case 1: (void)launch_pdl(layernorm_bwd_v8_kernel<1>, dim3(grid_rows), dim3(kRows * 32), 0, s, xb, ab, gb, dyb, drb, stats, M, D, eps); break;
      case 2: (void)launch_pdl(layernorm_bwd_v8_kernel<2>, dim3(grid_rows), dim3(kRows * 32), 0, s, xb, ab, gb, dyb, drb, stats, M, D, eps); break;
      case 3: (void)launch_pdl(layernorm_bwd_v8_kernel<3>, dim3(grid_rows), dim3(kRows * 32), 0, s, xb, ab, gb, dyb, drb, stats, M, D, eps); break;
      case 4: (void)launch_pdl(layernorm_bwd_v8_kernel<4>, dim3(grid_rows), dim3(kRows * 32), 0, s, xb, ab, gb, dyb, drb, stats, M, D, eps); break;
      case 5: case 6: (void)launch_pdl(layernorm_bwd_v8_kernel<6>, dim3(grid_rows), dim3(kRows * 32), 0, s, xb, ab, gb, dyb, drb, stats, M, D, eps); break;
      default: (void)launch_pdl(layernorm_bwd_v8_kernel<8>, dim3(grid_rows), dim3(kRows * 32), 0, s, xb, ab, gb, dyb, drb, stats, M, D, eps); break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 512 columns and eight row groups per block: a d_model of 1024 gives two blocks per
    // 256-row chunk, so every SM has work
    const dim3 g8((D + 511) / 512, bwd_row_chunks(M));
    (void)launch_pdl(colsum_v8_kernel<3, 64, 8>, dim3(g8), dim3(64, 8), 0, s, dyb,
                     static_cast<int64_t>(D), xb, ab, drb, stats, M, D, kChunkRows, part);
    return cudaGetLastError();
  }
#define MHA_LN_BWD(T, N)                                                                    \
  (void)launch_pdl(layernorm_bwd_kernel<T, N>, dim3(grid_rows), dim3(kRows * 32), 0, s, \
      static_cast<const T*>(x), static_cast<const T*>(a), static_cast<const T*>(gamma),     \
      static_cast<const T*>(dy), static_cast<T*>(dr), stats, M, D, eps)
  if (dtype == 1) {
    if (nit <= 16) MHA_LN_BWD(__nv_bfloat16, 16);
    else if (nit <= 32) MHA_LN_BWD(__nv_bfloat16, 32);
    else MHA_LN_BWD(__nv_bfloat16, 64);
  } else {
    if (nit <= 16) MHA_LN_BWD(float, 16);
    else if (nit <= 32) MHA_LN_BWD(float, 32);
    else MHA_LN_BWD(float, 64);
  }
#undef MHA_LN_BWD
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dtype == 1)
    (void)launch_pdl(ln_param_partials_kernel<__nv_bfloat16>, dim3(grid_cols), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(a),
        static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(dr), stats,
        part, M, D, kChunkRows);
  else
    (void)launch_pdl(ln_param_partials_kernel<float>, dim3(grid_cols), dim3(256), 0, s, static_cast<const float*>(x), static_cast<const float*>(a),
        static_cast<const float*>(dy), static_cast<const float*>(dr), stats, part, M, D,
        kChunkRows);
  return cudaGetLastError();
}

cudaError_t launch_colsum_partials(int dtype, const void* X, int64_t ld, int M, int N,
                                   float* part, cudaStream_t s) {
  if (dtype == 1 && N % 8 == 0 && ld % 8 == 0 && reinterpret_cast<uintptr_t>(X) % 16 == 0) {
    const dim3 g8((N + 1023) / 1024, bwd_row_chunks(M));
    (void)launch_pdl(colsum_v8_kernel<1, 128, 4>, dim3(g8), dim3(128, 4), 0, s,
                     static_cast<const __nv_bfloat16*>(X), ld, nullptr, nullptr, nullptr,
                     nullptr, M, N, kChunkRows, part);
    return cudaGetLastError();
  }
  const dim3 grid((N + 255) / 256, bwd_row_chunks(M));
  if (dtype == 1)
    (void)launch_pdl(colsum_partials_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(X), ld, M, N, kChunkRows, part);
  else
    (void)launch_pdl(colsum_partials_kernel<float>, dim3(grid), dim3(256), 0, s, static_cast<const float*>(X), ld, M, N,
                                                       kChunkRows, part);
  return cudaGetLastError();
}

cudaError_t launch_reduce_partials(int dtype, const float* part, int nchunk,
                                   int64_t chunk_stride, int N, void* out, cudaStream_t s) {
  return launch_reduce_partials3(dtype, part, nchunk, chunk_stride, N, 0, 1, out, nullptr,
                                 nullptr, s);
}

cudaError_t launch_reduce_partials3(int dtype, const float* part, int nchunk,
                                    int64_t chunk_stride, int N, int64_t term_stride,
                                    int nterm, void* out0, void* out1, void* out2,
                                    cudaStream_t s) {
  const dim3 grid((N + 255) / 256, nterm);
  if (dtype == 1)
    (void)launch_pdl(reduce_partials_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, part, nchunk,
                     chunk_stride, N, term_stride, static_cast<__nv_bfloat16*>(out0),
                     static_cast<__nv_bfloat16*>(out1), static_cast<__nv_bfloat16*>(out2));
  else
    (void)launch_pdl(reduce_partials_kernel<float>, grid, dim3(256), 0, s, part, nchunk,
                     chunk_stride, N, term_stride, static_cast<float*>(out0),
                     static_cast<float*>(out1), static_cast<float*>(out2));
  return cudaGetLastError();
}

cudaError_t launch_transpose(int dtype, const void* X, int64_t ldx, int R, int C, void* Y,
                             int64_t ldy, int R_pad, cudaStream_t s) {
  const bool v8 = dtype == 1 && C % 8 == 0 && ldx % 8 == 0 && ldy % 8 == 0 && R_pad % 8 == 0 &&
                  reinterpret_cast<uintptr_t>(X) % 16 == 0 && reinterpret_cast<uintptr_t>(Y) % 16 == 0;
  if (v8) {
    const dim3 g64((R_pad + kTp - 1) / kTp, (C + kTp - 1) / kTp);
    (void)launch_pdl(transpose_v8_kernel, dim3(g64), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(X), ldx, R, C,
                                             static_cast<__nv_bfloat16*>(Y), ldy, R_pad);
    return cudaGetLastError();
  }
  const dim3 grid((R_pad + 31) / 32, (C + 31) / 32);
  if (dtype == 1)
    (void)launch_pdl(transpose_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(X), ldx, R, C, static_cast<__nv_bfloat16*>(Y), ldy,
        R_pad);
  else
    (void)launch_pdl(transpose_kernel<float>, dim3(grid), dim3(256), 0, s, static_cast<const float*>(X), ldx, R, C,
                                                 static_cast<float*>(Y), ldy, R_pad);
  return cudaGetLastError();
}

}  // namespace mha
