// sdpa_f32.cu -- fp32 scaled dot-product attention (SIMT, no tensor cores, no TF32).
//
//   O = softmax(Q K^T * scale) V per (batch, head), optional causal / key-padding mask, the
//   neighbourhood |i - j| <= window of restricted self-attention, or a generation step's
//   bottom-right causal mask over a key/value cache
//   ("Attention Is All You Need", lettle.cn translation, 3.2.1 缩放点积注意力;
//    "Transformer：抛弃循环与卷积的序列建模", Self-Attention的优势).
//
// One warp per query row.  Lane k handles keys k, k+32, ...: pass 1 takes the row maximum
// of the allowed scores, pass 2 recomputes each score, accumulates exp(s - max) and the
// weighted value sum in fp32 registers, and a butterfly reduction across the warp joins
// the lanes' partial sums.  expf is the accurate CUDA function (no fast-math).
#include <cmath>

#include "launchers.h"

namespace mha {
namespace {

constexpr int kMaxD = 128;
constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32)
    sdpa_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                    const float* __restrict__ V, float* __restrict__ O, int Nq, int Nk, int d_k,
                    int d_v, int mask, int window, const int32_t* __restrict__ key_len,
                    float scale, float* __restrict__ lse,
                    int64_t qb, int64_t qh, int64_t qn, int64_t qd, int64_t kb, int64_t kh,
                    int64_t kn, int64_t kd, int64_t vb, int64_t vh, int64_t vn, int64_t vd,
                    int64_t ob, int64_t oh, int64_t on, int64_t od) {
  __shared__ float sq[kWarps][kMaxD];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + warp;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  if (row >= Nq) return;  // whole warp leaves together

  const float* q = Q + b * qb + h * qh + static_cast<int64_t>(row) * qn;
  for (int t = lane; t < d_k; t += 32) sq[warp][t] = q[t * qd];
  __syncwarp();

  int limit;  // allowed keys: first <= j <= limit
  int first = 0;
  if (mask == 1) {
    limit = row;
  } else if (mask == 2) {
    limit = min(max(key_len[b], 0), Nk) - 1;
  } else if (mask == kMaskWindow) {
    limit = min(row + window, Nk - 1);
    first = max(row - window, 0);
  } else if (mask == kMaskCausalCache) {
    // the Nq queries are the newest of L cached positions: row sits at L - Nq + row
    const int L = min(max(key_len[b], 0), Nk);
    limit = min(L - Nq + row, L - 1);
  } else {
    limit = Nk - 1;
  }
  const int nkeys = min(limit + 1, Nk);

  const float* kbase = K + b * kb + h * kh;
  const float* vbase = V + b * vb + h * vh;
  auto score = [&](int j) {
    const float* kr = kbase + static_cast<int64_t>(j) * kn;
    float acc = 0.f;
    for (int t = 0; t < d_k; ++t) acc = fmaf(sq[warp][t], kr[t * kd], acc);
    return acc * scale;
  };

  float m = -INFINITY;
  for (int j = first + lane; j < nkeys; j += 32) m = fmaxf(m, score(j));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));

  float l = 0.f;
  float acc[kMaxD];
#pragma unroll
  for (int t = 0; t < kMaxD; ++t) acc[t] = 0.f;
  for (int j = first + lane; j < nkeys; j += 32) {
    const float pj = expf(score(j) - m);
    l += pj;
    const float* vr = vbase + static_cast<int64_t>(j) * vn;
#pragma unroll
    for (int t = 0; t < kMaxD; ++t)
      if (t < d_v) acc[t] = fmaf(pj, vr[t * vd], acc[t]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  const float inv = (nkeys > first && l > 0.f) ? 1.f / l : 0.f;  // no allowed key: zeros
  if (lse != nullptr && lane == 0)
    lse[(static_cast<int64_t>(b) * gridDim.y + h) * Nq + row] =
        (nkeys > first && l > 0.f) ? m + logf(l) : INFINITY;
  float* o = O + b * ob + h * oh + static_cast<int64_t>(row) * on;
#pragma unroll
  for (int t = 0; t < kMaxD; ++t) {
    if (t < d_v) {  // d_v is uniform across the warp
      float v = acc[t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == (t & 31)) o[t * od] = v * inv;
    }
  }
}

}  // namespace

cudaError_t launch_sdpa_f32(const SdpaArgs& a, cudaStream_t s) {
  dim3 grid((a.Nq + kWarps - 1) / kWarps, a.H, a.B);
  sdpa_f32_kernel<<<grid, kWarps * 32, 0, s>>>(
      static_cast<const float*>(a.Q), static_cast<const float*>(a.K),
      static_cast<const float*>(a.V), static_cast<float*>(a.O), a.Nq, a.Nk, a.d_k, a.d_v,
      a.mask, a.window, a.key_len, a.scale, a.lse, a.sq[0], a.sq[1], a.sq[2], a.sq[3], a.sk[0], a.sk[1], a.sk[2],
      a.sk[3], a.sv[0], a.sv[1], a.sv[2], a.sv[3], a.so[0], a.so[1], a.so[2], a.so[3]);
  return cudaGetLastError();
}

}  // namespace mha
