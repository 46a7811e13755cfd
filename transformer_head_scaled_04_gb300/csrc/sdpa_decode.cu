// sdpa_decode.cu -- attention for one autoregressive generation step against a key/value
// cache ("Transformer：抛弃循环与卷积的序列建模", Transformer 翻译样例 > Decoder and Transformer
// 训练样例: each step's newest target positions attend every cached position up to their own;
// "Attention Is All You Need", lettle.cn translation, 3.2.1 缩放点积注意力).
//
//   O[b,h,i] = softmax_j(Q[b,h,i] . K[b,h,j] * scale, allowed) V[b,h,j],  i < Nq (<= 16)
//   allowed: j < L_b = cache_len[b]; with the causal flag also j <= L_b - Nq + i (the Nq
//   queries are the newest of the L_b cached positions: the causal mask aligned bottom-right).
//
// A few query rows against thousands of cached keys is bound by reading the cache from HBM
// (about Nq FLOPs per byte), so the work is split along the keys (split-K):
//   decode_partial: one CTA per (256-key chunk, head, batch element).  TMA brings the chunk's
//     K and V rows into shared memory (two 128-row boxes each, 128-byte swizzle); each thread
//     scores one key against all queries, each warp takes the max and sum of a query's
//     exponentials, and for O the lanes own value columns while the warps split the keys.
//     Writes the chunk's unnormalised O, its max m (raw scores) and sum l per query.
//   decode_combine: per (batch, head, query) merges the chunks: M = max m_s,
//     O = sum_s 2^((m_s - M) c) O_s / sum_s 2^((m_s - M) c) l_s, c = scale * log2(e).
// Chunks past L_b write an empty partial (m = -inf, l = 0) without reading the cache.  Rows
// with no allowed key are written as zeros.  Every wait is bounded.
#include <cuda_bf16.h>

#include <cmath>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kChunk = 256;  // keys per CTA
constexpr int kD = 64;       // head dim (d_k = d_v)
constexpr int kThreads = 128;
static_assert(kChunk == 2 * kThreads, "each thread scores two keys of the chunk");
constexpr int kWarps = kThreads / 32;
constexpr int kBox = 128;                // rows per TMA box
constexpr int kBoxBytes = kBox * kD * 2;  // 16 KB
constexpr int kErrTimeout = -6;
constexpr int kSiteDecode = 31;

// shared memory for NQ query rows: K chunk, V chunk (1024-aligned for the swizzle), Q,
// scores, the warps' partial O, per-query max and sum, the TMA barrier
template <int NQ>
struct DecodeSmem {
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + 2 * kBoxBytes;
  static constexpr int kOffQ = kOffV + 2 * kBoxBytes;         // float [NQ][64]
  static constexpr int kOffS = kOffQ + NQ * kD * 4;           // float [NQ][256]
  static constexpr int kOffO = kOffS + NQ * kChunk * 4;       // float [warps][NQ][64]
  static constexpr int kOffStat = kOffO + kWarps * NQ * kD * 4;  // float [NQ][2]
  static constexpr int kOffBar = kOffStat + NQ * 2 * 4;
  static constexpr int kBytes = 1024 + kOffBar + 64;  // two barriers: K landed, V landed
};

struct DecodeParams {
  int H, Nq, Lmax, causal, n_split;
  const int32_t* cache_len;
  const __nv_bfloat16* Q;
  int64_t sq_b, sq_h, sq_n;
  float scale;        // multiplies q.k
  float* part;        // [B][H][n_split][Nq][kD + 2]: O, m, l
  int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// NQ: compile-time bound on the query rows (1, 2, 4, 8 or 16); p.Nq <= NQ
template <int NQ>
__global__ void __launch_bounds__(kThreads)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  using Sm = DecodeSmem<NQ>;
  constexpr int kOffK = Sm::kOffK, kOffV = Sm::kOffV, kOffQ = Sm::kOffQ, kOffS = Sm::kOffS,
                kOffO = Sm::kOffO, kOffStat = Sm::kOffStat, kOffBar = Sm::kOffBar;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* sQ = reinterpret_cast<float*>(smem + kOffQ);
  float* sS = reinterpret_cast<float*>(smem + kOffS);
  float* sO = reinterpret_cast<float*>(smem + kOffO);
  float* sStat = reinterpret_cast<float*>(smem + kOffStat);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Nq = p.Nq;
  const int L = min(max(__ldg(p.cache_len + b), 0), p.Lmax);
  const int k0 = split * kChunk;
  float* out = p.part + ((static_cast<int64_t>(b) * p.H + h) * p.n_split + split) * Nq * (kD + 2);

  if (k0 >= L) {  // nothing cached here: an empty partial
    for (int i = tid; i < Nq * (kD + 2); i += kThreads) {
      const int c = i % (kD + 2);
      out[i] = (c == kD) ? -INFINITY : 0.f;
    }
    return;
  }
  const int nk = min(kChunk, L - k0);  // cached keys in this chunk
  const int nbox = (nk + kBox - 1) / kBox;

  const uint32_t barK = smem_u32(bar), barV = smem_u32(bar + 1);
  if (tid == 0) {
    mbar_init(barK, 1);
    mbar_init(barV, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {  // K first: the scores start while V is still on its way
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    mbar_arrive_expect_tx(barK, nbox * kBoxBytes);
    for (int x = 0; x < nbox; ++x)
      tma_load_4d(smem_u32(smem + kOffK + x * kBoxBytes), &tmK, barK, 0, k0 + x * kBox, h, b);
    mbar_arrive_expect_tx(barV, nbox * kBoxBytes);
    for (int x = 0; x < nbox; ++x)
      tma_load_4d(smem_u32(smem + kOffV + x * kBoxBytes), &tmV, barV, 0, k0 + x * kBox, h, b);
  }
  // queries to shared memory as fp32 while the cache chunk is in flight
  const __nv_bfloat16* qb = p.Q + b * p.sq_b + h * p.sq_h;
  for (int i = tid; i < Nq * kD; i += kThreads)
    sQ[i] = __bfloat162float(qb[(i / kD) * p.sq_n + (i % kD)]);
  // a timed-out wait records the error, lets the copies land (bounded) and leaves
  auto give_up = [&]() {
    if (tid == 0) record_error(p.status, kErrTimeout, kSiteDecode);
    (void)mbar_wait(barK, 0, p.timeout_ns);
    (void)mbar_wait(barV, 0, p.timeout_ns);
  };
  // every thread waits (bounded); the block gives up together if any wait ran out
  if (!__syncthreads_and(mbar_wait(barK, 0, p.timeout_ns))) {
    give_up();
    return;
  }

  // ---- scores: thread t takes keys t and t + 128 of the chunk together, so each query value
  // read from shared memory serves both keys (the sum over d runs in the same order as for one)
  {
    const int kk0 = tid, kk1 = tid + kThreads;
    const bool in0 = kk0 < nk, in1 = kk1 < nk;
    float s0[NQ], s1[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) s0[q] = s1[q] = 0.f;
    const uint8_t* row0 = smem + kOffK + kk0 * 128;  // box rows are consecutive 128-byte rows
    const uint8_t* row1 = smem + kOffK + kk1 * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {  // 16-byte chunk c of row kk sits at chunk c ^ (kk & 7)
      const uint4 u0 = in0 ? *reinterpret_cast<const uint4*>(row0 + ((c ^ (kk0 & 7)) << 4))
                           : make_uint4(0, 0, 0, 0);
      const uint4 u1 = in1 ? *reinterpret_cast<const uint4*>(row1 + ((c ^ (kk1 & 7)) << 4))
                           : make_uint4(0, 0, 0, 0);
      const float k0v[8] = {bf16_lo(u0.x), bf16_hi(u0.x), bf16_lo(u0.y), bf16_hi(u0.y),
                            bf16_lo(u0.z), bf16_hi(u0.z), bf16_lo(u0.w), bf16_hi(u0.w)};
      const float k1v[8] = {bf16_lo(u1.x), bf16_hi(u1.x), bf16_lo(u1.y), bf16_hi(u1.y),
                            bf16_lo(u1.z), bf16_hi(u1.z), bf16_lo(u1.w), bf16_hi(u1.w)};
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q < Nq) {
          const float* qr = sQ + q * kD + c * 8;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float qe = qr[e];
            s0[q] = fmaf(qe, k0v[e], s0[q]);
            s1[q] = fmaf(qe, k1v[e], s1[q]);
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (q < Nq) {
        const bool ok0 = in0 && (!p.causal || k0 + kk0 <= L - Nq + q);
        const bool ok1 = in1 && (!p.causal || k0 + kk1 <= L - Nq + q);
        sS[q * kChunk + kk0] = ok0 ? s0[q] : -INFINITY;
        sS[q * kChunk + kk1] = ok1 ? s1[q] : -INFINITY;
      }
    }
  }
  __syncthreads();

  // ---- per query: max and exponentials (warp w takes queries w, w + 4, ...)
  const float c = p.scale * 1.4426950408889634f;  // scale * log2(e)
  for (int q = warp; q < Nq; q += kWarps) {
    float* srow = sS + q * kChunk;
    float m = -INFINITY;
    for (int kk = lane; kk < kChunk; kk += 32) m = fmaxf(m, srow[kk]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
    const float mc = (m == -INFINITY) ? 0.f : m * c;
    for (int kk = lane; kk < kChunk; kk += 32) {
      const float e = ex2_approx(fmaf(srow[kk], c, -mc));  // 2^-inf = 0 for excluded keys
      srow[kk] = e;
      l += e;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) {
      sStat[2 * q] = m;
      sStat[2 * q + 1] = l;
    }
  }
  if (!__syncthreads_and(mbar_wait(barV, 0, p.timeout_ns))) {
    give_up();
    return;
  }

  // ---- unnormalised O: warp w sums keys [64 w, 64 w + 64), lane owns columns 2 lane, 2 lane + 1
  float acc[NQ][2];
#pragma unroll
  for (int q = 0; q < NQ; ++q) acc[q][0] = acc[q][1] = 0.f;
  const int kend = min(kChunk / kWarps * (warp + 1), nk);
  for (int kk = kChunk / kWarps * warp; kk < kend; ++kk) {
    const uint8_t* row = smem + kOffV + kk * 128;
    // columns 2 lane, 2 lane + 1 are bytes 4 lane .. 4 lane + 3: chunk lane / 4, swizzled
    const uint32_t u = *reinterpret_cast<const uint32_t*>(
        row + ((((lane >> 2) ^ (kk & 7)) << 4) | ((lane & 3) << 2)));
    const float v0 = bf16_lo(u), v1 = bf16_hi(u);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (q < Nq) {
        const float pq = sS[q * kChunk + kk];
        acc[q][0] = fmaf(pq, v0, acc[q][0]);
        acc[q][1] = fmaf(pq, v1, acc[q][1]);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (q < Nq) {
      sO[(warp * NQ + q) * kD + 2 * lane] = acc[q][0];
      sO[(warp * NQ + q) * kD + 2 * lane + 1] = acc[q][1];
    }
  }
  __syncthreads();
  for (int i = tid; i < Nq * kD; i += kThreads) {
    const int q = i / kD, d = i % kD;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) o += sO[(w * NQ + q) * kD + d];
    out[q * (kD + 2) + d] = o;
  }
  if (tid < Nq) {
    out[tid * (kD + 2) + kD] = sStat[2 * tid];
    out[tid * (kD + 2) + kD + 1] = sStat[2 * tid + 1];
  }
}

// one block of Nq x 64 threads per (batch, head): thread (q, d) merges column d of query q over
// the chunks
__global__ void __launch_bounds__(kDecodeMaxQ * kD)
    decode_combine_kernel(const float* __restrict__ part, int H, int Nq, int n_split,
                          float scale, __nv_bfloat16* __restrict__ O, int64_t so_b,
                          int64_t so_h, int64_t so_n) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  const int h = blockIdx.x, b = blockIdx.y;
  const int q = threadIdx.x / kD, d = threadIdx.x % kD;
  if (q >= Nq) return;
  const float c = scale * 1.4426950408889634f;
  const float* base = part + (static_cast<int64_t>(b) * H + h) * n_split * Nq * (kD + 2);
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, base[(s * Nq + q) * (kD + 2) + kD]);
  float o = 0.f, l = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n_split; ++s) {
      const float* r = base + (s * Nq + q) * (kD + 2);
      const float ms = r[kD];
      if (ms == -INFINITY) continue;  // a chunk with no allowed key for this query
      const float w = ex2_approx((ms - M) * c);
      o = fmaf(w, r[d], o);
      l = fmaf(w, r[kD + 1], l);
    }
  }
  const float y = (l > 0.f) ? o / l : 0.f;
  O[b * so_b + h * so_h + q * so_n + d] = __float2bfloat16_rn(y);
}

template <int NQ>
cudaError_t launch_partial(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeParams& p,
                           dim3 grid, cudaStream_t s) {
  static_assert(NQ <= kDecodeMaxQ, "query rows beyond the decode limit");
  auto kern = decode_partial_kernel<NQ>;
  cudaError_t e =
      prepare_kernel(reinterpret_cast<const void*>(kern), DecodeSmem<NQ>::kBytes, nullptr);
  if (e != cudaSuccess) return e;
  (void)launch_pdl(kern, dim3(grid), dim3(kThreads), DecodeSmem<NQ>::kBytes, s, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace

int decode_num_splits(int Lmax) { return (Lmax + kChunk - 1) / kChunk; }

cudaError_t launch_sdpa_decode_bf16(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                    const DecodeArgs& a, float* part, const DevCtx& ctx,
                                    cudaStream_t s) {
  DecodeParams p;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Lmax = a.Lmax;
  p.causal = a.causal;
  p.n_split = decode_num_splits(a.Lmax);
  p.cache_len = a.cache_len;
  p.Q = static_cast<const __nv_bfloat16*>(a.Q);
  p.sq_b = a.sq[0];
  p.sq_h = a.sq[1];
  p.sq_n = a.sq[2];
  p.scale = a.scale;
  p.part = part;
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  const dim3 grid(p.n_split, a.H, a.B);
  cudaError_t e;
  if (a.Nq <= 1)
    e = launch_partial<1>(tmK, tmV, p, grid, s);
  else if (a.Nq <= 2)
    e = launch_partial<2>(tmK, tmV, p, grid, s);
  else if (a.Nq <= 4)
    e = launch_partial<4>(tmK, tmV, p, grid, s);
  else if (a.Nq <= 8)
    e = launch_partial<8>(tmK, tmV, p, grid, s);
  else
    e = launch_partial<16>(tmK, tmV, p, grid, s);
  if (e != cudaSuccess) return e;
  // Nq x 64 threads per (batch, head): every thread has a column to merge, and the blocks of
  // the whole step fit on the GPU at once (1024-thread blocks took ~3.4 rounds for Nq = 1)
  const int nq = a.Nq < 1 ? 1 : a.Nq;
  (void)launch_pdl(decode_combine_kernel, dim3(a.H, a.B), dim3(nq * kD), 0, s, part, a.H, a.Nq,
                   p.n_split, a.scale, static_cast<__nv_bfloat16*>(a.O), a.so[0], a.so[1],
                   a.so[2]);
  return cudaGetLastError();
}

}  // namespace mha
