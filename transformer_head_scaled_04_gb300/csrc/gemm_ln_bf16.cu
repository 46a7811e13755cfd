// gemm_ln_bf16.cu -- y = LayerNorm(x + C W_o^T + b_o) * gamma + beta in one kernel: the output
// projection of the attention sublayer and its residual + post-norm step
// ("Attention Is All You Need", lettle.cn translation, 3.1 Encoder and Decoder Stacks:
// LayerNorm(x + Sublayer(x)), and 3.2.2 多头注意力: MultiHead = Concat(head_1..head_h) W^O;
// "Transformer：抛弃循环与卷积的序列建模", Residual Connection 与 LayerNorm).
//
// The projection output A = C W_o^T + b_o never reaches HBM.  A row's LayerNorm needs all
// d_model of its columns, more than one CTA's tensor memory holds next to a second
// accumulator, so a cluster of CS = d_model / 256 CTAs owns each 128-row tile: CTA rank r
// computes columns [256 r, 256 r + 256) with the same persistent TMA + tcgen05 pipeline as the
// projection GEMM (128 x 256 x 16 MMAs into one of two TMEM accumulators, so a tile's
// epilogue overlaps the next tile's MMAs).  The clusters walk the row tiles.
//   warp 0     TMA producer: C and W_o K-slices (64 wide, 128-byte swizzle) into a 4-stage ring
//   warp 1     TMEM owner + MMA issuer
//   warps 2-9  epilogue: two warps per TMEM lane quarter, one row per thread, each of the
//              two covering 128 of the CTA's 256 columns:
//              1. r = x + (acc + b_o) in fp32 (the projection output is not rounded), written
//                 back over the accumulator in TMEM; the sum of the 128 values and their
//                 squared deviations from their own mean; optionally the projection output
//                 itself, rounded to bf16, to memory (what the training forward keeps for the
//                 backward);
//              2. that (sum, squared deviations) pair goes to every CTA of the cluster by an
//                 asynchronous shared-memory store that completes the receiving CTA's
//                 statistics barrier (2 * CS pairs per row arrive in each CTA);
//              3. mean and biased variance of the whole row by the exact combination of the
//                 partial results (n = 128 values each: M2 = sum_i M2_i + n (mean_i - mean)^2),
//                 then y = (r - mean) / sqrt(var + eps) * gamma + beta from r in TMEM, rounded
//                 to bf16.  x and y move between global memory and the row-per-thread
//                 registers through a 32-row x 32-column staging tile per warp, so that the
//                 global accesses are coalesced (four lanes per 64-byte piece of a row, eight
//                 rows per instruction); with each thread reading and writing its own row
//                 directly, every 16-byte access of a warp touched 32 rows, and those accesses
//                 took ~2.6 us (x) and ~3 us (y) of a tile's epilogue.  x for the next tile is
//                 requested into L2 at the start of a tile and loaded two 32-column chunks
//                 ahead; b_o, gamma and beta sit in shared memory as bf16; the elementwise
//                 arithmetic runs on fp32 pairs.
// Every wait is bounded; on a timeout the kernel records MHA_ERR_DEVICE_TIMEOUT, lets its
// in-flight copies and MMAs land, frees TMEM and returns.  All CTAs of a cluster meet at a
// cluster barrier before they exit, so no CTA leaves while a peer may still write to it.
#include <cuda_bf16.h>

#include <mutex>
#include <vector>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;  // columns per CTA
constexpr int kBK = 64;
constexpr int kThreads = 320;  // producer, MMA issuer, 8 epilogue warps
constexpr int kEpiWarps = 8;
constexpr int kHalf = kBN / 2;  // columns per epilogue warp
constexpr int kErrTimeout = -6;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kBarBytes = 256;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr int kMaxCluster = 8;

enum : int {
  kSiteProducer = 41,
  kSiteMma = 42,
  kSiteEpilogue = 43,
  kSiteStats = 44,
  kSiteVectors = 45,  // index checks (MHA_DEBUG_BOUNDS builds): b_o / gamma / beta
  kSiteX = 46,        // x
  kSiteOut = 47       // y and the optional projection output
};

// (sum, squared deviations) per row for each of the two accumulators in flight and each of the
// 2 * CS column halves of the cluster; then b_o, gamma, beta for the CTA's columns (bf16); then
// a 32-row x 32-column bf16 staging tile per epilogue warp (x in, y out)
// (4 ring stages where they fit in the 227 KB a CTA may have, else 3)
constexpr int kStageTileBytes = 32 * 64;
template <int CS>
struct LnShape {
  static constexpr int kParts = 2 * CS;
  static constexpr int kStatBytes = 2 * kParts * kBM * 8;
  static constexpr int kVecBytes = 3 * kBN * 2;
  static constexpr int kStageBytesEpi = kEpiWarps * kStageTileBytes;
  static constexpr int kRest = 1024 + kBarBytes + kStatBytes + kVecBytes + kStageBytesEpi;
  static constexpr int kStages = (kRest + 4 * kStageBytes <= 227 * 1024) ? 4 : 3;
  static constexpr int kSmemBytes = kRest + kStages * kStageBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

struct LnParams {
  const __nv_bfloat16* bias;   // b_o [D] or null
  const __nv_bfloat16* x;      // residual [M, D]
  const __nv_bfloat16* gamma;  // [D] or null (1)
  const __nv_bfloat16* beta;   // [D] or null (0)
  __nv_bfloat16* y;            // [M, D]
  __nv_bfloat16* a_out;        // optional [M, D]: bf16(C W_o^T + b_o)
  int M, D, K;
  float eps;
  int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ void unpack8_bf16(const uint4& u, float* v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ void load8_bf16(const __nv_bfloat16* p, float* v) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}

template <int CS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_ln_bf16_kernel(const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmW, const LnParams p) {
  using S = LnShape<CS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + S::kStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kStages * kStageBytes);
  // [0,ST) full, [ST,2ST) empty, acc_full[2], acc_empty[2], stats[2], drain; tmem slot after
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S::kStages + 7);
  const uint32_t sStat = smem_u32(smem + S::kStages * kStageBytes + kBarBytes);
  __nv_bfloat16* sVec = reinterpret_cast<__nv_bfloat16*>(
      smem + S::kStages * kStageBytes + kBarBytes + S::kStatBytes);  // b_o | gamma | beta
  const uint32_t sStage =
      smem_u32(smem + S::kStages * kStageBytes + kBarBytes + S::kStatBytes + S::kVecBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const int cluster = static_cast<int>(cluster_id_x());
  const int nclusters = static_cast<int>(cluster_count_x());
  const int num_kb = p.K / kBK;
  const int tiles = (p.M + kBM - 1) / kBM;
  const int n0 = static_cast<int>(crank) * kBN;  // this CTA's columns

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + S::kStages + s); };
  auto acc_full = [&](int b) { return smem_u32(bars + 2 * S::kStages + b); };
  auto acc_empty = [&](int b) { return smem_u32(bars + 2 * S::kStages + 2 + b); };
  auto stat_bar = [&](int b) { return smem_u32(bars + 2 * S::kStages + 4 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * S::kStages + 6);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), kEpiWarps);  // one arrival per epilogue warp
      mbar_init(stat_bar(b), 1);  // this CTA's expect_tx; the pairs complete its bytes
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync_all();  // every CTA's barriers exist before any peer arrives on them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output (C, x) is complete from here on

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    int it = 0;
    bool ok = true;
    for (int t = cluster; ok && t < tiles; t += nclusters) {
      const int m0 = t * kBM;
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % S::kStages;
        if (!mbar_wait_backoff(empty_bar(s), ((it / S::kStages) & 1) ^ 1, p.timeout_ns)) {
          record_error(p.status, kErrTimeout, kSiteProducer);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(full_bar(s), kStageBytes);
        tma_load_2d(smem_u32(sA + s * kABytes), &tmX, full_bar(s), kb * kBK, m0);
        tma_load_2d(smem_u32(sB + s * kBBytes), &tmW, full_bar(s), kb * kBK, n0);
      }
    }
    // let every copy this thread started land before the CTA can exit
    for (int i = (it > S::kStages ? it - S::kStages : 0); i < it; ++i)
      (void)mbar_wait(full_bar(i % S::kStages), (i / S::kStages) & 1, p.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, false);
    int it = 0, tcount = 0;
    bool ok = true;
    for (int t = cluster; ok && t < tiles; t += nclusters, ++tcount) {
      const int buf = tcount & 1;
      const uint32_t d = tmem + buf * kBN;
      if (!mbar_wait(acc_empty(buf), ((tcount >> 1) & 1) ^ 1, p.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % S::kStages;
        if (!mbar_wait(full_bar(s), (it / S::kStages) & 1, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * kABytes);
        const uint32_t b0 = smem_u32(sB + s * kBBytes);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16_ss(d, smem_desc_sw128(a0 + k * 32, 16, 1024),
                      smem_desc_sw128(b0 + k * 32, 16, 1024), idesc,
                      (kb != 0 || k != 0) ? 1u : 0u);
        mma_commit(empty_bar(s));
      }
      if (!ok) break;
      mma_commit(acc_full(buf));
    }
    if (!ok) record_error(p.status, kErrTimeout, kSiteMma);
    mma_commit(drain_bar);
    (void)mbar_wait(drain_bar, 0, p.timeout_ns);  // no MMA in flight past this point
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;          // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;      // which 128 of the CTA's 256 columns
    const int rloc = quarter * 32 + lane;
    const int c0 = half * kHalf;           // first column of this warp inside the CTA's slab
    const int part = static_cast<int>(crank) * 2 + half;
    constexpr int kParts = S::kParts;
    constexpr uint32_t kStatTx = kParts * kBM * 8;  // bytes each CTA receives per tile
    const float inv_n = 1.f / static_cast<float>(kHalf);
    const float inv_d = 1.f / static_cast<float>(p.D);
    // b_o, gamma and beta of the CTA's 256 columns, once, as fp32
    for (int i = threadIdx.x - 64; i < kBN; i += kEpiWarps * 32) {
      const int col = n0 + i;
      const bool ok_col = bounds_ok(col, p.D, p.status, kSiteVectors);
      sVec[i] = (p.bias && ok_col) ? p.bias[col] : __float2bfloat16(0.f);
      sVec[kBN + i] = (p.gamma && ok_col) ? p.gamma[col] : __float2bfloat16(1.f);
      sVec[2 * kBN + i] = (p.beta && ok_col) ? p.beta[col] : __float2bfloat16(0.f);
    }
    named_bar_sync(1, kEpiWarps * 32);
    // ask L2 for this thread's 256 bytes of x in a tile (two 128-byte lines of its row)
    auto prefetch_x = [&](int tile) {
      const int r = tile * kBM + rloc;
      if (tile < tiles && r < p.M) {
        const char* a =
            reinterpret_cast<const char*>(p.x + static_cast<int64_t>(r) * p.D + n0 + c0);
        prefetch_global_l2(a);
        prefetch_global_l2(a + 128);
      }
    };
    prefetch_x(cluster);
    int tcount = 0;
    for (int t = cluster; t < tiles; t += nclusters, ++tcount) {
      const int buf = tcount & 1;
      const int m0 = t * kBM;
      const int row = m0 + rloc;
      const bool in = row < p.M;
      prefetch_x(t + nclusters);  // the next tile's rows reach L2 while this one runs
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(buf), (tcount >> 1) & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteEpilogue);
        break;
      }
      tc_fence_after();
      const uint32_t tb =
          tmem + buf * kBN + c0 + (static_cast<uint32_t>(quarter * 32) << 16);
      // this warp's 32 x 64-byte staging tile: 16-byte chunk j of row r sits in slot
      // j ^ ((r >> 1) & 3), so both the row-per-lane reads and the 8-rows-per-instruction
      // writes hit all 32 banks once
      const uint32_t stg = sStage + (warp - 2) * kStageTileBytes;
      const int rr = lane >> 2, jj = lane & 3;  // coalesced side: rows rr + 8k, chunk jj
      const int wrow = m0 + quarter * 32;       // the warp's first row
      const uint32_t slot_w = stg + rr * 64 + ((jj ^ ((rr >> 1) & 3)) << 4);  // + k * 512
      const uint32_t slot_r = stg + lane * 64;                                 // + (j ^ sw) * 16
      const int sw_r = (lane >> 1) & 3;
      // 1. r = x + (acc + b_o), back into TMEM; sum.  x comes in coalesced (four lanes per
      // 64-byte row piece, eight rows per instruction), two 32-column chunks ahead, and goes
      // through the staging tile to the thread that owns the row.
      uint4 xa[4], xb[4];
      auto load_x = [&](int c, uint4 (&dst)[4]) {
        const int col = n0 + c0 + c * 32 + jj * 8;
        const bool ok_x = span_ok(n0 + c0 + c * 32, 32, p.D, p.status, kSiteX);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = wrow + rr + 8 * k;
          dst[k] = (ok_x && r < p.M)
                       ? __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(r) * p.D +
                                                              col))
                       : make_uint4(0, 0, 0, 0);
        }
      };
      load_x(0, xa);
      load_x(1, xb);
      float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t a[32];
        tmem_ld32(tb + c * 32, a);
#pragma unroll
        for (int k = 0; k < 4; ++k) st_shared_v4(slot_w + k * 512, xa[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k) xa[k] = xb[k];
        if (c + 2 < kHalf / 32) load_x(c + 2, xb);
        __syncwarp();
        uint4 xc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) xc[j] = ld_shared_v4(slot_r + ((j ^ sw_r) << 4));
        __syncwarp();  // the tile is free for the next chunk
        float bvec[32];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          unpack8_bf16(ld_shared_v4(smem_u32(sVec + c0 + c * 32 + 8 * j)), bvec + 8 * j);
        tmem_wait_ld();
        reg_fence(a);
        if (p.a_out != nullptr && in && span_ok(n0 + c0 + c * 32, 32, p.D, p.status, kSiteOut)) {
          uint4* ap = reinterpret_cast<uint4*>(p.a_out + static_cast<int64_t>(row) * p.D + n0 +
                                               c0 + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = v * 8 + 2 * e;
              o[e] = pack_bf16x2(__uint_as_float(a[i]) + bvec[i],
                                 __uint_as_float(a[i + 1]) + bvec[i + 1]);
            }
            ap[v] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const __nv_bfloat162* xh = reinterpret_cast<const __nv_bfloat162*>(&xc[v]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = v * 8 + 2 * e;
            const float2 xv = __bfloat1622float2(xh[e]);
            const float2 r = fadd2(xv, fadd2(make_float2(__uint_as_float(a[i]),
                                                         __uint_as_float(a[i + 1])),
                                             make_float2(bvec[i], bvec[i + 1])));
            sum2 = fadd2(sum2, r);
            a[i] = __float_as_uint(r.x);
            a[i + 1] = __float_as_uint(r.y);
          }
        }
        tmem_st32(tb + c * 32, a);
      }
      tmem_wait_st();
      const float sum = sum2.x + sum2.y;
      const float2 nmean_l = make_float2(-sum * inv_n, -sum * inv_n);
      float2 m2v = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t a[32];
        tmem_ld32(tb + c * 32, a);
        tmem_wait_ld();
        reg_fence(a);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 dv =
              fadd2(make_float2(__uint_as_float(a[i]), __uint_as_float(a[i + 1])), nmean_l);
          m2v = ffma2(dv, dv, m2v);
        }
      }
      const float m2 = m2v.x + m2v.y;
      // 2. this row's partial statistics to slot [buf][part][rloc] of every cluster CTA; the
      // store completes that CTA's statistics barrier by its 8 bytes
      if (threadIdx.x == 64) mbar_arrive_expect_tx(stat_bar(buf), kStatTx);
      const uint32_t slot = sStat + ((buf * kParts + part) * kBM + rloc) * 8;
#pragma unroll
      for (int r = 0; r < CS; ++r)
        st_async_f32x2(mapa_shared(slot, r), sum, m2, mapa_shared(stat_bar(buf), r));
      if (!__all_sync(0xffffffffu,
                      mbar_wait_cluster(stat_bar(buf), (tcount >> 1) & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteStats);
        break;
      }
      // 3. the row's mean and biased variance from the 2 * CS partial results
      float tot = 0.f;
      float2 pr[kParts];
#pragma unroll
      for (int i = 0; i < kParts; ++i) {
        pr[i] = ld_shared_f32x2(sStat + ((buf * kParts + i) * kBM + rloc) * 8);
        tot += pr[i].x;
      }
      const float mean = tot * inv_d;
      float M2 = 0.f;
#pragma unroll
      for (int i = 0; i < kParts; ++i) {
        const float dm = pr[i].x * inv_n - mean;
        M2 += pr[i].y + static_cast<float>(kHalf) * dm * dm;
      }
      const float rstd = 1.0f / sqrtf(M2 * inv_d + p.eps);
      const float2 nmean = make_float2(-mean, -mean);
      const float2 rstd2 = make_float2(rstd, rstd);
      // y, 32 columns at a time: each thread's row into the staging tile, then out coalesced
      // (four lanes per 64-byte row piece, eight rows per instruction)
#pragma unroll 1
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t a[32];
        tmem_ld32(tb + c * 32, a);
        float g[32], bt[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          unpack8_bf16(ld_shared_v4(smem_u32(sVec + kBN + c0 + c * 32 + 8 * j)), g + 8 * j);
          unpack8_bf16(ld_shared_v4(smem_u32(sVec + 2 * kBN + c0 + c * 32 + 8 * j)), bt + 8 * j);
        }
        tmem_wait_ld();
        reg_fence(a);
        if (c == kHalf / 32 - 1) {  // accumulator read: hand it back to the MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty(buf));
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = v * 8 + 2 * e;
            float2 z = fadd2(make_float2(__uint_as_float(a[i]), __uint_as_float(a[i + 1])),
                             nmean);
            z = fmul2(z, rstd2);
            z = ffma2(z, make_float2(g[i], g[i + 1]), make_float2(bt[i], bt[i + 1]));
            o[e] = pack_bf16x2(z.x, z.y);
          }
          st_shared_v4(slot_r + ((v ^ sw_r) << 4), make_uint4(o[0], o[1], o[2], o[3]));
        }
        __syncwarp();
        const bool ok_y = span_ok(n0 + c0 + c * 32, 32, p.D, p.status, kSiteOut);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = wrow + rr + 8 * k;
          const uint4 v = ld_shared_v4(slot_w + k * 512);
          if (ok_y && r < p.M)
            *reinterpret_cast<uint4*>(p.y + static_cast<int64_t>(r) * p.D + n0 + c0 + c * 32 +
                                      jj * 8) = v;
        }
        __syncwarp();  // the tile is free for the next chunk
      }
    }
  }

  tc_fence_before();
  cluster_sync_all();  // no peer writes into this CTA's shared memory any more
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Largest number of CS-CTA clusters of this kernel that fit on the device at once (cached per
// device and cluster size); 0 when the query fails.
template <int CS>
int max_clusters(int num_sms) {
  static std::mutex mu;
  static std::vector<std::pair<int, int>> cache;  // (device, clusters)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& e : cache)
    if (e.first == dev) return e.second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS * (num_sms / CS));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = LnShape<CS>::kSmemBytes;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_ln_bf16_kernel<CS>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache.push_back({dev, n});
  return n;
}

template <int CS>
cudaError_t launch_cs(const CUtensorMap& tmX, const CUtensorMap& tmW, const LnParams& p,
                      const DevCtx& ctx, cudaStream_t s) {
  auto kern = gemm_ln_bf16_kernel<CS>;
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), LnShape<CS>::kSmemBytes,
                                 nullptr);
  if (e != cudaSuccess) return e;
  const int tiles = (p.M + kBM - 1) / kBM;
  int nc = max_clusters<CS>(ctx.num_sms);
  if (nc <= 0) nc = ctx.num_sms / CS;
  if (nc > tiles) nc = tiles;
  if (nc < 1) nc = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS * nc);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = LnShape<CS>::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, p);
}

}  // namespace

bool gemm_ln_bf16_supported(int D, int K) {
  return D % kBN == 0 && D / kBN >= 1 && D / kBN <= kMaxCluster && K % kBK == 0 && K > 0;
}

cudaError_t launch_gemm_ln_bf16(const CUtensorMap& tmX, const CUtensorMap& tmW,
                                const void* bias, const void* x, const void* gamma,
                                const void* beta, void* y, int M, int D, int K, float eps,
                                const DevCtx& ctx, cudaStream_t s, void* a_out) {
  if (!gemm_ln_bf16_supported(D, K)) return cudaErrorInvalidValue;
  LnParams p;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.gamma = static_cast<const __nv_bfloat16*>(gamma);
  p.beta = static_cast<const __nv_bfloat16*>(beta);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.a_out = static_cast<__nv_bfloat16*>(a_out);
  p.M = M;
  p.D = D;
  p.K = K;
  p.eps = eps;
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  switch (D / kBN) {
    case 1: return launch_cs<1>(tmX, tmW, p, ctx, s);
    case 2: return launch_cs<2>(tmX, tmW, p, ctx, s);
    case 3: return launch_cs<3>(tmX, tmW, p, ctx, s);
    case 4: return launch_cs<4>(tmX, tmW, p, ctx, s);
    case 5: return launch_cs<5>(tmX, tmW, p, ctx, s);
    case 6: return launch_cs<6>(tmX, tmW, p, ctx, s);
    case 7: return launch_cs<7>(tmX, tmW, p, ctx, s);
    case 8: return launch_cs<8>(tmX, tmW, p, ctx, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mha
