// sdpa_bwd_f32.cu -- backward of scaled dot-product attention, fp32 SIMT kernels, and the
// per-row term D shared with the bf16 path.
//
// The chain rule through O = softmax(Q K^T * scale, masked) V ("Transformer：抛弃循环与卷积的
// 序列建模", Transformer 训练样例 > 反向传播; "Attention Is All You Need", lettle.cn
// translation, 3.2.1 缩放点积注意力), with the softmax weights rebuilt from the forward's
// log-sum-exp, P_ij = exp(s_ij - lse_i) (0 for excluded keys):
//   D_i  = sum_d dO_id O_id
//   dV_j = sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i . V_j - D_i)
//   dQ_i = scale * sum_j dS_ij K_j,   dK_j = scale * sum_i dS_ij Q_i
// dq: one warp per query row (lanes split the keys); dkdv: one warp per key row (lanes split
// the queries), one launch for dV and one for dK; partial sums meet in a butterfly reduction.
// expf is CUDA's accurate function.
#include <cuda_bf16.h>

#include <cmath>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kMaxD = 128;
constexpr int kWarps = 8;

// query row i may see key j (the forward's masks; key_len is read on the device)
__device__ __forceinline__ bool allowed(int mask, int i, int j, int L, int window, int Nq) {
  if (j >= L) return false;
  if (mask == 1) return j <= i;
  if (mask == kMaskWindow) return j >= i - window && j <= i + window;
  if (mask == kMaskCausalCache) return j <= L - Nq + i;
  return true;
}

__device__ __forceinline__ int keys_of(int mask, const int32_t* key_len, int b, int Nk) {
  return (mask == 2 || mask == kMaskCausalCache) ? min(max(key_len[b], 0), Nk) : Nk;
}

template <typename T>
__device__ __forceinline__ float ld(const T* p) {
  if constexpr (sizeof(T) == 2)
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
  else
    return static_cast<float>(*p);
}

// D[b,h,i] = sum_d dO[b,h,i,d] O[b,h,i,d]; one warp per row
template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
    sdpa_bwd_rowdot_kernel(const T* __restrict__ O, const T* __restrict__ dO,
                           float* __restrict__ Dv, int H, int Nq, int d_v, int64_t ob,
                           int64_t oh, int64_t on, int64_t gb, int64_t gh, int64_t gn,
                           const float* __restrict__ lse, int rows) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  // lse != null: the per-tile layout {-lse * log2 e [128], -D [128]} (negated, so the
  // tensor-core kernels add them in paired fp32 instructions) over rows up to a whole number
  // of 128-row tiles; otherwise D alone as [B, H, Nq]
  const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  if (row >= rows) return;
  float acc = 0.f;
  if (row < Nq) {
    const T* o = O + b * ob + h * oh + static_cast<int64_t>(row) * on;
    const T* g = dO + b * gb + h * gh + static_cast<int64_t>(row) * gn;
    for (int t = lane; t < d_v; t += 32) acc = fmaf(ld(o + t), ld(g + t), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  }
  if (lane != 0) return;
  const int64_t bh = static_cast<int64_t>(b) * H + h;
  if (lse == nullptr) {
    Dv[bh * Nq + row] = acc;
  } else {
    float* tile = Dv + (bh * (rows / 128) + row / 128) * 256;
    tile[row % 128] = row < Nq ? -(__ldg(lse + bh * Nq + row) * 1.4426950408889634f) : -INFINITY;
    tile[128 + row % 128] = -acc;
  }
}

// bf16 tensor-core path: per query row, D = sum_d dO_d O_d (d = 64) and the per-tile layouts
// the backward kernels read; 16-byte loads, eight lanes per row, four rows per warp.
//   stats: per (b, h, 128-row tile) -lse * log2 e [128] then -D [128] (rows past Nq: -inf, 0)
//   aug:   per tile four 128 x 8 bf16 column chunks (row r of chunk k at (k * 128 + r) * 16
//          bytes): chunk 0 = -lse / scale, chunk 2 = -D, each as three bf16 terms summing to
//          the fp32 value; chunks 1 and 3 zero.  c = scale * log2 e, so c * (-lse / scale) =
//          -lse * log2 e.  Rows past Nq get a large negative stand-in for -inf, and so does a
//          fully masked row's +inf (its keys are masked by the kernel that reads it).
//   dq_acc (may be null): the row's 64 fp32 dQ accumulators zeroed
__device__ __forceinline__ uint4 three_bf16_terms(float x) {
  if (!(fabsf(x) <= 1e30f)) x = x > 0.f ? 1e30f : -1e30f;
  const __nv_bfloat16 t0 = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(t0);
  const __nv_bfloat16 t1 = __float2bfloat16_rn(r1);
  const __nv_bfloat16 t2 = __float2bfloat16_rn(r1 - __bfloat162float(t1));
  return make_uint4(static_cast<uint32_t>(__bfloat16_as_ushort(t0)) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(t1)) << 16),
                    static_cast<uint32_t>(__bfloat16_as_ushort(t2)), 0u, 0u);
}

__global__ void __launch_bounds__(kWarps * 32)
    sdpa_bwd_rowdot_bf16_kernel(const __nv_bfloat16* __restrict__ O,
                                const __nv_bfloat16* __restrict__ dO, int H, int Nq, int64_t ob,
                                int64_t oh, int64_t on, int64_t gb, int64_t gh, int64_t gn,
                                const float* __restrict__ lse, int rows, float c,
                                float* __restrict__ stats, uint4* __restrict__ aug,
                                float* __restrict__ dq_acc) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  const int lane = threadIdx.x & 31, part = lane & 7;
  const int row = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * 4 + (lane >> 3);
  const int h = blockIdx.y, b = blockIdx.z;
  if (row >= rows) return;  // rows is a multiple of 128: whole 8-lane groups leave together
  const bool valid = row < Nq;
  float acc = 0.f;
  if (valid) {
    const uint4 o = __ldg(reinterpret_cast<const uint4*>(O + b * ob + h * oh +
                                                         static_cast<int64_t>(row) * on) + part);
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(dO + b * gb + h * gh +
                                                         static_cast<int64_t>(row) * gn) + part);
    const uint32_t ov[4] = {o.x, o.y, o.z, o.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov[i]));
      const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[i]));
      acc = fmaf(of.x, gf.x, acc);
      acc = fmaf(of.y, gf.y, acc);
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  const int64_t bh = static_cast<int64_t>(b) * H + h;
  const int64_t tile = bh * (rows / 128) + row / 128;
  const float l2 = valid ? __ldg(lse + bh * Nq + row) * 1.4426950408889634f : INFINITY;
  if (part == 0) stats[tile * 256 + row % 128] = -l2;
  if (part == 1) stats[tile * 256 + 128 + row % 128] = -acc;
  if (part < 4) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (part == 0) v = three_bf16_terms(valid ? -l2 / c : -1e30f);
    if (part == 2) v = three_bf16_terms(-acc);
    aug[tile * 512 + part * 128 + row % 128] = v;
  }
  if (dq_acc != nullptr) {
    uint4* z = reinterpret_cast<uint4*>(dq_acc + (bh * rows + row) * 64) + part * 2;
    z[0] = make_uint4(0u, 0u, 0u, 0u);
    z[1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

struct BwdF32 {
  const float *Q, *K, *V, *dO, *lse, *Dv;
  float *dQ, *dK, *dV;
  int64_t s[8][3];  // Q, K, V, O(unused), dO, dQ, dK, dV: element strides b, h, n (d = 1)
  int H, Nq, Nk, d_k, d_v, mask, window;
  const int32_t* key_len;
  float scale;
};

__global__ void __launch_bounds__(kWarps * 32) sdpa_bwd_dq_f32_kernel(const BwdF32 p) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  __shared__ float sq[kWarps][kMaxD];
  __shared__ float sg[kWarps][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kWarps + warp, h = blockIdx.y, b = blockIdx.z;
  if (i >= p.Nq) return;
  const float* q = p.Q + b * p.s[0][0] + h * p.s[0][1] + static_cast<int64_t>(i) * p.s[0][2];
  const float* g = p.dO + b * p.s[4][0] + h * p.s[4][1] + static_cast<int64_t>(i) * p.s[4][2];
  for (int t = lane; t < p.d_k; t += 32) sq[warp][t] = q[t];
  for (int t = lane; t < p.d_v; t += 32) sg[warp][t] = g[t];
  __syncwarp();
  const int64_t r = (static_cast<int64_t>(b) * p.H + h) * p.Nq + i;
  const float lse = p.lse[r], Di = p.Dv[r];
  const int L = keys_of(p.mask, p.key_len, b, p.Nk);
  const float* kb = p.K + b * p.s[1][0] + h * p.s[1][1];
  const float* vb = p.V + b * p.s[2][0] + h * p.s[2][1];
  float acc[kMaxD];
#pragma unroll
  for (int t = 0; t < kMaxD; ++t) acc[t] = 0.f;
  for (int j = lane; j < p.Nk; j += 32) {
    if (!allowed(p.mask, i, j, L, p.window, p.Nq)) continue;
    const float* kr = kb + static_cast<int64_t>(j) * p.s[1][2];
    const float* vr = vb + static_cast<int64_t>(j) * p.s[2][2];
    float s = 0.f, dp = 0.f;
    for (int t = 0; t < p.d_k; ++t) s = fmaf(sq[warp][t], kr[t], s);
    for (int t = 0; t < p.d_v; ++t) dp = fmaf(sg[warp][t], vr[t], dp);
    const float ds = expf(s * p.scale - lse) * (dp - Di);
#pragma unroll
    for (int t = 0; t < kMaxD; ++t)
      if (t < p.d_k) acc[t] = fmaf(ds, kr[t], acc[t]);
  }
  float* dq = p.dQ + b * p.s[5][0] + h * p.s[5][1] + static_cast<int64_t>(i) * p.s[5][2];
#pragma unroll
  for (int t = 0; t < kMaxD; ++t) {
    if (t < p.d_k) {
      float v = acc[t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == (t & 31)) dq[t] = v * p.scale;
    }
  }
}

// kWantK: dK (from dS and Q) or dV (from P and dO); two passes keep one accumulator row
template <bool kWantK>
__global__ void __launch_bounds__(kWarps * 32) sdpa_bwd_dkdv_f32_kernel(const BwdF32 p) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  __shared__ float sk[kWarps][kMaxD];
  __shared__ float sv[kWarps][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * kWarps + warp, h = blockIdx.y, b = blockIdx.z;
  if (j >= p.Nk) return;
  const float* k = p.K + b * p.s[1][0] + h * p.s[1][1] + static_cast<int64_t>(j) * p.s[1][2];
  const float* v = p.V + b * p.s[2][0] + h * p.s[2][1] + static_cast<int64_t>(j) * p.s[2][2];
  for (int t = lane; t < p.d_k; t += 32) sk[warp][t] = k[t];
  for (int t = lane; t < p.d_v; t += 32) sv[warp][t] = v[t];
  __syncwarp();
  const int L = keys_of(p.mask, p.key_len, b, p.Nk);
  const float* qb = p.Q + b * p.s[0][0] + h * p.s[0][1];
  const float* gb = p.dO + b * p.s[4][0] + h * p.s[4][1];
  const int64_t r0 = (static_cast<int64_t>(b) * p.H + h) * p.Nq;
  const int dout = kWantK ? p.d_k : p.d_v;
  float acc[kMaxD];
#pragma unroll
  for (int t = 0; t < kMaxD; ++t) acc[t] = 0.f;
  for (int i = lane; i < p.Nq; i += 32) {
    if (!allowed(p.mask, i, j, L, p.window, p.Nq)) continue;
    const float* qr = qb + static_cast<int64_t>(i) * p.s[0][2];
    const float* gr = gb + static_cast<int64_t>(i) * p.s[4][2];
    float s = 0.f;
    for (int t = 0; t < p.d_k; ++t) s = fmaf(qr[t], sk[warp][t], s);
    const float pij = expf(s * p.scale - p.lse[r0 + i]);
    float w = pij;
    const float* src = gr;
    if (kWantK) {
      float dp = 0.f;
      for (int t = 0; t < p.d_v; ++t) dp = fmaf(gr[t], sv[warp][t], dp);
      w = pij * (dp - p.Dv[r0 + i]);  // dS_ij
      src = qr;
    }
#pragma unroll
    for (int t = 0; t < kMaxD; ++t)
      if (t < dout) acc[t] = fmaf(w, src[t], acc[t]);
  }
  float* dst = kWantK ? p.dK + b * p.s[6][0] + h * p.s[6][1] + static_cast<int64_t>(j) * p.s[6][2]
                      : p.dV + b * p.s[7][0] + h * p.s[7][1] + static_cast<int64_t>(j) * p.s[7][2];
  const float mul = kWantK ? p.scale : 1.f;
#pragma unroll
  for (int t = 0; t < kMaxD; ++t) {
    if (t < dout) {
      float x = acc[t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      if (lane == (t & 31)) dst[t] = x * mul;
    }
  }
}

}  // namespace

cudaError_t launch_sdpa_bwd_rowdot(const SdpaBwdArgs& a, int dtype, cudaStream_t s) {
  if (dtype == 1) {
    const int rows = (a.Nq + 127) / 128 * 128;
    char* base = reinterpret_cast<char*>(a.Dv);
    (void)launch_pdl(sdpa_bwd_rowdot_bf16_kernel, dim3(rows / (4 * kWarps), a.H, a.B),
                     dim3(kWarps * 32), 0, s, static_cast<const __nv_bfloat16*>(a.O),
                     static_cast<const __nv_bfloat16*>(a.dO), a.H, a.Nq, a.st[3][0], a.st[3][1],
                     a.st[3][2], a.st[4][0], a.st[4][1], a.st[4][2], a.lse, rows,
                     a.scale * 1.4426950408889634f, a.Dv,
                     reinterpret_cast<uint4*>(base + sdpa_bwd_aug_offset(a.B, a.H, a.Nq)),
                     a.deterministic ? nullptr
                                     : reinterpret_cast<float*>(
                                           base + sdpa_bwd_dq_acc_offset(a.B, a.H, a.Nq)));
    return cudaGetLastError();
  }
  dim3 grid((a.Nq + kWarps - 1) / kWarps, a.H, a.B);
  (void)launch_pdl(sdpa_bwd_rowdot_kernel<float>, dim3(grid), dim3(kWarps * 32), 0, s,
                   static_cast<const float*>(a.O), static_cast<const float*>(a.dO), a.Dv, a.H,
                   a.Nq, a.d_v, a.st[3][0], a.st[3][1], a.st[3][2], a.st[4][0], a.st[4][1],
                   a.st[4][2], nullptr, a.Nq);
  return cudaGetLastError();
}

cudaError_t launch_sdpa_bwd_f32(const SdpaBwdArgs& a, cudaStream_t s) {
  BwdF32 p;
  p.Q = static_cast<const float*>(a.Q);
  p.K = static_cast<const float*>(a.K);
  p.V = static_cast<const float*>(a.V);
  p.dO = static_cast<const float*>(a.dO);
  p.lse = a.lse;
  p.Dv = a.Dv;
  p.dQ = static_cast<float*>(a.dQ);
  p.dK = static_cast<float*>(a.dK);
  p.dV = static_cast<float*>(a.dV);
  for (int t = 0; t < 8; ++t)
    for (int i = 0; i < 3; ++i) p.s[t][i] = a.st[t][i];
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.d_k = a.d_k;
  p.d_v = a.d_v;
  p.mask = a.mask;
  p.window = a.window;
  p.key_len = a.key_len;
  p.scale = a.scale;
  (void)launch_pdl(sdpa_bwd_dq_f32_kernel, dim3(dim3((a.Nq + kWarps - 1) / kWarps, a.H, a.B)), dim3(kWarps * 32), 0, s, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid_k((a.Nk + kWarps - 1) / kWarps, a.H, a.B);
  (void)launch_pdl(sdpa_bwd_dkdv_f32_kernel<false>, dim3(grid_k), dim3(kWarps * 32), 0, s, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  (void)launch_pdl(sdpa_bwd_dkdv_f32_kernel<true>, dim3(grid_k), dim3(kWarps * 32), 0, s, p);
  return cudaGetLastError();
}

}  // namespace mha
