// sdpa_bf16.cu -- fused scaled dot-product attention forward on the sm_103a tensor cores.
//
//   O = softmax(Q K^T / sqrt(d_k)) V per (batch, head), optional causal or key-padding mask
//   ("Attention Is All You Need", lettle.cn translation, 3.2.1 缩放点积注意力;
//    "Transformer：抛弃循环与卷积的序列建模", Scaled Dot-Product Attention, the three uses of
//    attention, and 训练样本 for the causal mask).
//
// The n x n score matrix never leaves the SM.  One CTA owns 256 query rows (two 128-row
// tiles t = 0, 1) of one (b, h) and streams K/V in 128-row tiles:
//   warp 8     TMA producer: Q tiles once, then K_j and V_j into a 3-stage ring
//   warp 9     TMEM owner + MMA issuer (one thread):
//                S_t = Q_t K_j^T           tcgen05.mma 128x128x16 x4, fp32 in TMEM
//                O_t += P_t V_j            tcgen05.mma 128x64x16 x8, P from smem, V MN-major
//              The two tiles ping-pong so the tensor core works on one tile while the
//              softmax warps of the other run.
//   warps 0-7  softmax: warpgroup t owns tile t, one query row per thread (its TMEM lane).
//              tcgen05.ld of the S row, mask, running max m and sum l, p = 2^(s*c - m*c)
//              with c = scale*log2(e), P rounded to bf16 into a 128-byte-swizzled smem tile.
//              O is rescaled (in TMEM) only when the max grows by more than 2^8; the final
//              O / l uses the same max as every p, so the result equals the softmax exactly
//              up to rounding.  At the end: O / l -> bf16 -> global, in any strided layout
//              (the head-concat layout [B, Nq, H*64] in the sublayer).
// Whole K/V tiles past the causal diagonal or past key_len[b] are never loaded.
// Every wait is bounded (see device_common.cuh); a timeout records MHA_ERR_DEVICE_TIMEOUT.
#include <cuda_bf16.h>

#include <cmath>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kBQ = 128;       // query rows per tile
constexpr int kBKV = 128;      // keys per K/V tile
constexpr int kHD = 64;        // head dim (d_k = d_v)
constexpr int kStages = 3;     // K/V ring depth
constexpr int kThreads = 320;  // 8 softmax warps + producer + MMA
constexpr int kTileBytes = kBQ * kHD * 2;  // 16 KB: a 128 x 64 bf16 tile
constexpr int kPBytes = kBQ * kBKV * 2;    // 32 KB: a 128 x 128 bf16 P tile

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + 2 * kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffP = kOffV + kStages * kTileBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kSmemBytes = 1024 + kOffBar + 256;
constexpr uint32_t kTmemCols = 512;  // S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384)

constexpr int kErrTimeout = -6;
enum : int {
  kSiteProducer = 21,
  kSiteMma = 22,
  kSiteSoftmaxS = 23,
  kSiteSoftmaxO = 24,
  kSiteEpilogue = 25
};

// barrier indices
constexpr int kBarQ = 0;
constexpr int kBarKFull = 1;
constexpr int kBarVFull = kBarKFull + kStages;
constexpr int kBarKVEmpty = kBarVFull + kStages;
constexpr int kBarSFull = kBarKVEmpty + kStages;  // 2
constexpr int kBarPFull = kBarSFull + 2;          // 2
constexpr int kBarODone = kBarPFull + 2;          // 2
constexpr int kBarDrain = kBarODone + 2;
constexpr int kNumBars = kBarDrain + 1;

struct Params {
  int B, H, Nq, Nk, mask;
  const int32_t* key_len;
  float scale_log2;  // scale * log2(e)
  float tau;         // rescale threshold in raw score units (2^8 growth)
  __nv_bfloat16* O;
  int64_t so_b, so_h, so_n;
  int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

__global__ void __launch_bounds__(kThreads, 1)
    sdpa_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sK = smem_u32(smem + kOffK);
  const uint32_t sV = smem_u32(smem + kOffV);
  uint8_t* const sP = smem + kOffP;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int q0 = (gridDim.z - 1 - blockIdx.z) * (2 * kBQ);  // heaviest causal blocks first

  // keys a row may see: causal -> j <= row; otherwise j < L
  int L = p.Nk;
  if (p.mask == 2) L = min(max(__ldg(p.key_len + b), 0), p.Nk);
  int n_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int row0 = q0 + t * kBQ;
    if (row0 >= p.Nq)
      n_t[t] = 0;
    else if (p.mask == 1)
      n_t[t] = min(p.Nq - 1, row0 + kBQ - 1) / kBKV + 1;
    else
      n_t[t] = (L + kBKV - 1) / kBKV;
  }
  const int nmax = max(n_t[0], n_t[1]);

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPFull + t), kBQ);
      mbar_init(bar(kBarODone + t), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && nmax > 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const uint32_t qbytes = (n_t[0] > 0 ? kTileBytes : 0) + (n_t[1] > 0 ? kTileBytes : 0);
      mbar_arrive_expect_tx(bar(kBarQ), qbytes);
      for (int t = 0; t < 2; ++t)
        if (n_t[t] > 0) tma_load_4d(sQ + t * kTileBytes, &tmQ, bar(kBarQ), 0, q0 + t * kBQ, h, b);
      int issued = 0;
      for (int j = 0; j < nmax; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        if (!mbar_wait(bar(kBarKVEmpty + s), ph ^ 1, p.timeout_ns)) {
          record_error(p.status, kErrTimeout, kSiteProducer);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarKFull + s), kTileBytes);
        tma_load_4d(sK + s * kTileBytes, &tmK, bar(kBarKFull + s), 0, j * kBKV, h, b);
        mbar_arrive_expect_tx(bar(kBarVFull + s), kTileBytes);
        tma_load_4d(sV + s * kTileBytes, &tmV, bar(kBarVFull + s), 0, j * kBKV, h, b);
        issued = j + 1;
      }
      // every copy started here lands before the CTA may exit
      (void)mbar_wait(bar(kBarQ), 0, p.timeout_ns);
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i) {
        (void)mbar_wait(bar(kBarKFull + i % kStages), (i / kStages) & 1, p.timeout_ns);
        (void)mbar_wait(bar(kBarVFull + i % kStages), (i / kStages) & 1, p.timeout_ns);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && nmax > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBQ, kBKV, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(kBQ, kHD, false, true);
      auto issue_s = [&](int t, int s) {
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(sQ + t * kTileBytes + kk * 32, 1024, 1024);
          const uint64_t bd = smem_desc_sw128(sK + s * kTileBytes + kk * 32, 1024, 1024);
          mma_bf16_ss(tmem + t * kBKV, ad, bd, idS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int s, bool acc) {
        const uint32_t pbase = smem_u32(sP + t * kPBytes);
#pragma unroll
        for (int kk = 0; kk < kBKV / 16; ++kk) {
          const uint64_t ad =
              smem_desc_sw128(pbase + (kk >> 2) * (kBQ * 128) + (kk & 3) * 32, 1024, 1024);
          const uint64_t bd = smem_desc_sw128(sV + s * kTileBytes + kk * 16 * 128, 1024, 1024);
          mma_bf16_ss(tmem + 256 + t * kHD, ad, bd, idO, (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(bar(kBarQ), 0, p.timeout_ns) &&
                mbar_wait(bar(kBarKFull + 0), 0, p.timeout_ns);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (n_t[t] > 0) {
            issue_s(t, 0);
            mma_commit(bar(kBarSFull + t));
          }
      }
      for (int j = 0; ok && j < nmax; ++j) {
        const int s = j % kStages;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= n_t[t]) continue;
          if (!mbar_wait(bar(kBarPFull + t), j & 1, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (j + 1 < n_t[t]) {
            const int s1 = (j + 1) % kStages;
            if (!mbar_wait(bar(kBarKFull + s1), ((j + 1) / kStages) & 1, p.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(t, s1);
            mma_commit(bar(kBarSFull + t));
          }
          if (!mbar_wait(bar(kBarVFull + s), (j / kStages) & 1, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(t, s, j > 0);
          mma_commit(bar(kBarODone + t));
        }
        if (ok) mma_commit(bar(kBarKVEmpty + s));
      }
      if (!ok) record_error(p.status, kErrTimeout, kSiteMma);
      mma_commit(bar(kBarDrain));
      (void)mbar_wait(bar(kBarDrain), 0, p.timeout_ns);  // no MMA in flight past this point
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int t = warp >> 2;
    const int quarter = warp & 3;
    const int r_local = quarter * 32 + lane;
    const int row = q0 + t * kBQ + r_local;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + t * kBKV + lane_off;
    const uint32_t tO = tmem + 256 + t * kHD + lane_off;
    uint8_t* const sPt = sP + t * kPBytes;
    const int nt = (t == 0) ? n_t[0] : n_t[1];
    const int limit = (p.mask == 1) ? row : L - 1;  // allowed keys: j <= limit
    const float c = p.scale_log2;
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;

    for (int j = 0; j < nt; ++j) {
      if (!warp_all(mbar_wait(bar(kBarSFull + t), j & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteSoftmaxS);
        ok = false;
        break;
      }
      tc_fence_after();
      const int col0 = j * kBKV;
      const bool masked = col0 + kBKV - 1 > limit;
      // pass 1: the row maximum over the allowed keys of this tile
      float mt = -INFINITY;
      {
        uint32_t r[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, r[q]);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) reg_fence(r[q]);
        if (masked) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + q * 32 + i <= limit) mt = fmaxf(mt, __uint_as_float(r[q][i]));
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 32; i += 2)
              mt = fmax3(mt, __uint_as_float(r[q][i]), __uint_as_float(r[q][i + 1]));
        }
      }

      if (j > 0 && !warp_all(mbar_wait(bar(kBarODone + t), (j - 1) & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteSoftmaxO);
        ok = false;
        break;
      }
      const float m_new = fmaxf(m_used, mt);
      if (j == 0) {
        m_used = (m_new == -INFINITY) ? 0.f : m_new;
      } else {
        const bool grow = m_new > m_used + p.tau;
        float alpha = 1.f;
        if (grow) {
          alpha = ex2_approx((m_used - m_new) * c);
          l *= alpha;
          m_used = m_new;
        }
        if (__any_sync(0xffffffffu, grow)) {  // TMEM access is warp-collective
          tc_fence_after();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            tmem_ld32(tO + half * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + half * 32, o);
          }
          tmem_wait_st();
        }
      }
      // pass 2, 32 keys at a time: p = 2^(s*c - m*c), row sum, P (bf16) into the
      // K-major 128-byte-swizzled smem tile: two 64-key halves of [128 rows][128 B]
      const float neg = -m_used * c;
      float rs = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t r[32];
        tmem_ld32(tS + q * 32, r);
        tmem_wait_ld();
        reg_fence(r);
        float pv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float sv = (masked && col0 + q * 32 + i > limit) ? -INFINITY : __uint_as_float(r[i]);
          pv[i] = ex2_approx(fmaf(sv, c, neg));
          rs += pv[i];
        }
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int u = q * 4 + w;  // 16-byte chunk index along the row (8 keys each)
          uint4 v;
          v.x = pack_bf16x2(pv[w * 8 + 0], pv[w * 8 + 1]);
          v.y = pack_bf16x2(pv[w * 8 + 2], pv[w * 8 + 3]);
          v.z = pack_bf16x2(pv[w * 8 + 4], pv[w * 8 + 5]);
          v.w = pack_bf16x2(pv[w * 8 + 6], pv[w * 8 + 7]);
          uint8_t* dst = sPt + (u >> 3) * (kBQ * 128) + r_local * 128 +
                         (((u & 7) ^ (r_local & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = v;
        }
      }
      l += rs;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + t));
    }

    // ---------------------------------------------------------------- epilogue: O / l
    float o[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) o[i] = 0.f;
    if (ok && nt > 0) {
      if (!warp_all(mbar_wait(bar(kBarODone + t), (nt - 1) & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteEpilogue);
      } else {
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32(tO, r0);
        tmem_ld32(tO + 32, r1);
        tmem_wait_ld();
        reg_fence(r0);
        reg_fence(r1);
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          o[i] = __uint_as_float(r0[i]) * inv;
          o[32 + i] = __uint_as_float(r1[i]) * inv;
        }
      }
    }
    if (row < p.Nq) {
      __nv_bfloat16* dst = p.O + static_cast<int64_t>(b) * p.so_b +
                           static_cast<int64_t>(h) * p.so_h + static_cast<int64_t>(row) * p.so_n;
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint4 v;
        v.x = pack_bf16x2(o[u * 8 + 0], o[u * 8 + 1]);
        v.y = pack_bf16x2(o[u * 8 + 2], o[u * 8 + 3]);
        v.z = pack_bf16x2(o[u * 8 + 4], o[u * 8 + 5]);
        v.w = pack_bf16x2(o[u * 8 + 6], o[u * 8 + 7]);
        d4[u] = v;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_sdpa_bf16(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, const SdpaArgs& a, const DevCtx& ctx,
                             cudaStream_t s) {
  Params p;
  p.B = a.B;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.mask = a.mask;
  p.key_len = a.key_len;
  const double c = static_cast<double>(a.scale) * 1.4426950408889634;  // log2(e)
  p.scale_log2 = static_cast<float>(c);
  p.tau = static_cast<float>(8.0 / c);
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.so_b = a.so[0];
  p.so_h = a.so[1];
  p.so_n = a.so[2];
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  cudaError_t e = cudaFuncSetAttribute(sdpa_fwd_bf16_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(a.H, a.B, (a.Nq + 2 * kBQ - 1) / (2 * kBQ));
  sdpa_fwd_bf16_kernel<<<grid, kThreads, kSmemBytes, s>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace mha
