// sdpa_f32.cu -- fp32 scaled dot-product attention (SIMT, no tensor cores, no TF32).
//
//   O = softmax(Q K^T * scale) V per (batch, head), optional causal / key-padding mask, the
//   neighbourhood |i - j| <= window of restricted self-attention, or a generation step's
//   bottom-right causal mask over a key/value cache
//   ("Attention Is All You Need", lettle.cn translation, 3.2.1 缩放点积注意力;
//    "Transformer：抛弃循环与卷积的序列建模", Self-Attention的优势).
//
// One warp per query row, eight rows (of one batch element and head) per block.  The block
// walks the keys its rows may see in chunks of 32: the chunk's K and V rows are staged in
// shared memory with coalesced loads (row pitch d + 1: conflict-free per-lane row reads),
// lane k scores key k of the chunk, and an online softmax (running max m, sum l, the value
// accumulator rescaled by exp(m_old - m_new) when the max grows) folds the chunk in: each
// weight is broadcast across the warp and lane k accumulates value features k, k + 32, ...
// expf is the accurate CUDA function (no fast-math).
#include <cmath>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kMaxD = 128;
constexpr int kWarps = 8;
constexpr int kChunk = 32;             // keys per shared-memory chunk
constexpr int kPitch = kMaxD + 1;      // padded row pitch of a staged K / V row
// index checks (MHA_DEBUG_BOUNDS builds)
enum : int { kSiteF32KeyLen = 51, kSiteF32KV = 52, kSiteF32Lse = 53 };

__global__ void __launch_bounds__(kWarps * 32)
    sdpa_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                    const float* __restrict__ V, float* __restrict__ O, int Nq, int Nk, int d_k,
                    int d_v, int mask, int window, const int32_t* __restrict__ key_len,
                    float scale, float* __restrict__ lse,
                    int64_t qb, int64_t qh, int64_t qn, int64_t qd, int64_t kb, int64_t kh,
                    int64_t kn, int64_t kd, int64_t vb, int64_t vh, int64_t vn, int64_t vd,
                    int64_t ob, int64_t oh, int64_t on, int64_t od, int* status) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  __shared__ float sq[kWarps][kMaxD];
  __shared__ float sk[kChunk * kPitch];
  __shared__ float sv[kChunk * kPitch];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + warp;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const bool live = row < Nq;  // warps past Nq still help stage the chunks

  if (live) {
    const float* q = Q + b * qb + h * qh + static_cast<int64_t>(row) * qn;
    for (int t = lane; t < d_k; t += 32) sq[warp][t] = q[t * qd];
  }

  // allowed keys of a row: first <= j <= limit
  auto bounds = [&](int r, int& first, int& limit) {
    first = 0;
    if (mask == 1) {
      limit = r;
    } else if (mask == 2) {
      limit = bounds_ok(b, gridDim.z, status, kSiteF32KeyLen) ? min(max(key_len[b], 0), Nk) - 1
                                                               : -1;
    } else if (mask == kMaskWindow) {
      limit = min(r + window, Nk - 1);
      first = max(r - window, 0);
    } else if (mask == kMaskCausalCache) {
      // the Nq queries are the newest of L cached positions: row r sits at L - Nq + r
      const int L = bounds_ok(b, gridDim.z, status, kSiteF32KeyLen) ? min(max(key_len[b], 0), Nk)
                                                                    : 0;
      limit = min(L - Nq + r, L - 1);
    } else {
      limit = Nk - 1;
    }
    limit = min(limit, Nk - 1);
  };
  int first, limit;
  bounds(min(row, Nq - 1), first, limit);
  // the keys any row of the block may see: rows are consecutive and both bounds grow with r
  int blk_first, blk_limit, last_first, last_limit;
  bounds(blockIdx.x * kWarps, blk_first, blk_limit);
  bounds(min(blockIdx.x * kWarps + kWarps - 1, Nq - 1), last_first, last_limit);
  blk_first = max(min(blk_first, last_first), 0);
  blk_limit = max(blk_limit, last_limit);

  const float* kbase = K + b * kb + h * kh;
  const float* vbase = V + b * vb + h * vh;
  float m = -INFINITY, l = 0.f;
  float acc[kMaxD / 32];  // value features lane, lane + 32, ...
#pragma unroll
  for (int i = 0; i < kMaxD / 32; ++i) acc[i] = 0.f;

  for (int j0 = blk_first; j0 <= blk_limit; j0 += kChunk) {
    __syncthreads();  // the previous chunk is consumed
    const int nj = min(kChunk, blk_limit + 1 - j0);
    for (int e = threadIdx.x; e < nj * d_k; e += kWarps * 32) {
      const int jj = e / d_k, t = e - jj * d_k;
      if (bounds_ok(j0 + jj, Nk, status, kSiteF32KV))
        sk[jj * kPitch + t] = kbase[static_cast<int64_t>(j0 + jj) * kn + t * kd];
    }
    for (int e = threadIdx.x; e < nj * d_v; e += kWarps * 32) {
      const int jj = e / d_v, t = e - jj * d_v;
      if (bounds_ok(j0 + jj, Nk, status, kSiteF32KV))
        sv[jj * kPitch + t] = vbase[static_cast<int64_t>(j0 + jj) * vn + t * vd];
    }
    __syncthreads();
    if (!live) continue;
    const int j = j0 + lane;
    const bool ok = lane < nj && j >= first && j <= limit;
    float sc = -INFINITY;
    if (ok) {
      float a = 0.f;
      for (int t = 0; t < d_k; ++t) a = fmaf(sq[warp][t], sk[lane * kPitch + t], a);
      sc = a * scale;
    }
    float cm = sc;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
    if (cm == -INFINITY) continue;  // no allowed key of this row in the chunk
    const float m_new = fmaxf(m, cm);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    m = m_new;
    const float pj = ok ? expf(sc - m) : 0.f;
    l = l * alpha + pj;
#pragma unroll
    for (int i = 0; i < kMaxD / 32; ++i) acc[i] *= alpha;
    for (int jj = 0; jj < nj; ++jj) {
      const float p = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
      for (int i = 0; i < kMaxD / 32; ++i)
        if (lane + 32 * i < d_v) acc[i] = fmaf(p, sv[jj * kPitch + lane + 32 * i], acc[i]);
    }
  }
  if (!live) return;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  const bool any = m != -INFINITY && l > 0.f;
  const float inv = any ? 1.f / l : 0.f;  // no allowed key: zeros
  const int64_t lse_i = (static_cast<int64_t>(b) * gridDim.y + h) * Nq + row;
  if (lse != nullptr && lane == 0 &&
      bounds_ok(lse_i, static_cast<int64_t>(gridDim.z) * gridDim.y * Nq, status, kSiteF32Lse))
    lse[lse_i] = any ? m + logf(l) : INFINITY;
  float* o = O + b * ob + h * oh + static_cast<int64_t>(row) * on;
#pragma unroll
  for (int i = 0; i < kMaxD / 32; ++i)
    if (lane + 32 * i < d_v) o[(lane + 32 * i) * od] = acc[i] * inv;
}

}  // namespace

cudaError_t launch_sdpa_f32(const SdpaArgs& a, cudaStream_t s) {
  dim3 grid((a.Nq + kWarps - 1) / kWarps, a.H, a.B);
  (void)launch_pdl(sdpa_f32_kernel, dim3(grid), dim3(kWarps * 32), 0, s, static_cast<const float*>(a.Q), static_cast<const float*>(a.K),
      static_cast<const float*>(a.V), static_cast<float*>(a.O), a.Nq, a.Nk, a.d_k, a.d_v,
      a.mask, a.window, a.key_len, a.scale, a.lse, a.sq[0], a.sq[1], a.sq[2], a.sq[3], a.sk[0], a.sk[1], a.sk[2],
      a.sk[3], a.sv[0], a.sv[1], a.sv[2], a.sv[3], a.so[0], a.so[1], a.so[2], a.so[3], a.status);
  return cudaGetLastError();
}

}  // namespace mha
