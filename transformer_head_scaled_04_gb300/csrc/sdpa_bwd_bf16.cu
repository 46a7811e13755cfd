// sdpa_bwd_bf16.cu -- backward of scaled dot-product attention on the sm_103a tensor cores.
//
// The chain rule through O = softmax(Q K^T * scale, masked) V ("Transformer：抛弃循环与卷积的
// 序列建模", Transformer 训练样例 > 反向传播; "Attention Is All You Need", lettle.cn
// translation, 3.2.1 缩放点积注意力).  The softmax weights are rebuilt tile by tile from the
// forward's log-sum-exp, so the n x n matrices never leave the SM:
//   P = 2^(s*c - lse2) (c = scale*log2 e, lse2 = lse*log2 e),  dP = dO V^T,
//   dS = P * (dP - D),  D_i = sum_d dO_id O_id,
//   dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO
// A small prior launch writes, per 128-row query tile, -D and -lse2 (1 KB) and an 8 KB operand
// block holding -lse / scale and -D as three bf16 terms each, and zeroes an fp32 dQ
// accumulator.  Then:
//   dkdv -- one CTA per 128-key tile; Q/dO tiles (with their operand blocks) stream through a
//           TMA ring.  S^T = K Q^T and dP^T = V dO^T (tcgen05.mma 128x128x16, fp32 in TMEM),
//           each with a fifth K step against a constant "ones" operand, so TMEM already holds
//           s - lse / scale and dP - D and the math warps (one key row per thread) read no
//           statistics: p = 2^(c s'), dS = p dP'.  They write bf16 P^T into TMEM and dS^T into
//           shared memory; dV += P^T dO (A from TMEM) and dK += dS^T Q (A from shared memory)
//           accumulate in TMEM.  By default the same issuer then computes this key tile's part
//           of dQ for the query tile, dS K (A = dS^T's bytes read MN-major, B = K), which the
//           math warps move out of TMEM and add into the accumulator with one bulk tensor
//           reduction per warp (32 x 32 fp32 box); a last launch scales it into bf16 dQ.
//   dq   -- only when deterministic results are asked for (no atomics anywhere): one CTA per
//           128-row query tile rebuilds S and dP from K/V tiles streamed through a ring, four
//           math warps per column half turn them into bf16 dS in TMEM, dQ += dS K.
// Warps: 0-7 math (two per sub-partition: warps w and w+4 share TMEM lanes 32*(w%4).. and
// take the two 64-column halves of every tile), 8 TMA producer, 9 TMEM owner and issuer of S
// and dP (S^T and dP^T), then the gradient issuers: dq kernel warp 10 (dQ, with dS double-
// buffered in TMEM so the math warps write dS_{j+1} while dQ still reads dS_j), dkdv kernel
// warps 10 (dV) and 11 (dK, and dQ when fused; its math warps run at 200 registers through
// setmaxnreg).  Every wait is bounded; a timeout records MHA_ERR_DEVICE_TIMEOUT, lets
// in-flight copies and MMAs land, frees TMEM.
// Masks: none, causal (j <= i) and key padding (j < key_len[b]); fully masked tiles are
// skipped, and the d = 64 heads of the forward kernel are assumed.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kT = 128;                    // rows per tile (queries or keys)
constexpr int kHD = 64;                    // head dim
constexpr int kTileBytes = kT * kHD * 2;   // 16 KB
constexpr int kStages = 3;
constexpr int kMathWarps = 8;               // warp w: rows 32*(w%4).. of the tile, column half w/4
constexpr int kWarpProducer = kMathWarps;   // TMA
constexpr int kWarpMma = kMathWarps + 1;    // TMEM owner; issues the S and dP products
// An issuing thread spends ~75-100 cycles per tcgen05.mma here (more when the tensor pipe's
// queue is full), so the gradient products have issuers of their own and no longer wait
// behind the next tile's S / dP issue: dq kernel warp 10 (dQ); dkdv kernel warps 10 (dV)
// and 11 (dK).
constexpr int kWarpMma2 = kMathWarps + 2;
constexpr int kWarpMma3 = kMathWarps + 3;
constexpr int kQThreads = (kMathWarps + 3) * 32;
constexpr int kKThreads = (kMathWarps + 4) * 32;
constexpr int kKMathRegs = 200;
constexpr int kKControlRegs = 72;
static_assert(kMathWarps * 32 * kKMathRegs + 4 * 32 * kKControlRegs <= kKThreads * 168,
              "dkdv register split exceeds the launch allocation");
constexpr int kErrTimeout = -6;
enum : int { kSiteBwdProducer = 41, kSiteBwdMma = 42, kSiteBwdMath = 43, kSiteBwdEpi = 44 };
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int H, Nq, Nk, mask;
  const int32_t* key_len;
  float scale;       // multiplies q.k
  const float* stats;  // per (b, h, 128-row query tile): -lse * log2 e [128], then -D [128]
  const uint8_t* aug;  // per (b, h, query tile): the dkdv kernel's 8 KB extra-K-step operand
  __nv_bfloat16* out0;  // dq: dQ; dkdv: dK
  __nv_bfloat16* out1;  // dkdv: dV
  int64_t o0_b, o0_h, o0_n, o1_b, o1_h, o1_n;
  int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// number of keys query row i may see through key tile boundaries: L (key padding) or Nk
__device__ __forceinline__ int key_limit(const BwdParams& p, int b) {
  return (p.mask == 2) ? min(max(__ldg(p.key_len + b), 0), p.Nk) : p.Nk;
}

// store 64 fp32 values (times mul) of one row as bf16
__device__ __forceinline__ void store_row(__nv_bfloat16* dst, const uint32_t* r0,
                                          const uint32_t* r1, float mul) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint32_t* r = u < 4 ? r0 + 8 * u : r1 + 8 * (u - 4);
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(r[0]) * mul, __uint_as_float(r[1]) * mul);
    v.y = pack_bf16x2(__uint_as_float(r[2]) * mul, __uint_as_float(r[3]) * mul);
    v.z = pack_bf16x2(__uint_as_float(r[4]) * mul, __uint_as_float(r[5]) * mul);
    v.w = pack_bf16x2(__uint_as_float(r[6]) * mul, __uint_as_float(r[7]) * mul);
    d4[u] = v;
  }
}

// dS of one 64-key half of a query row: p = 2^(s*c - lse2) (0 past the row's last key when
// kMask), dS = p * (dP - D), packed to bf16 pairs; nl = -lse2 and nd = -D, two keys per paired
// fp32 instruction
template <bool kMask>
__device__ __forceinline__ void dq_half(const uint32_t* s0, const uint32_t* s1,
                                        const uint32_t* g0, const uint32_t* g1, int col0,
                                        int limit, float c, float nl, float nd, uint32_t* ds) {
  const float2 c2 = make_float2(c, c), nl2 = make_float2(nl, nl), nd2 = make_float2(nd, nd);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float2 sv = make_float2(__uint_as_float(i < 16 ? s0[2 * i] : s1[2 * i - 32]),
                                  __uint_as_float(i < 16 ? s0[2 * i + 1] : s1[2 * i + 1 - 32]));
    const float2 gv = make_float2(__uint_as_float(i < 16 ? g0[2 * i] : g1[2 * i - 32]),
                                  __uint_as_float(i < 16 ? g0[2 * i + 1] : g1[2 * i + 1 - 32]));
    float2 pv = ffma2(sv, c2, nl2);
    pv.x = ex2_approx(pv.x);
    pv.y = ex2_approx(pv.y);
    if (kMask) {
      if (col0 + 2 * i > limit) pv.x = 0.f;
      if (col0 + 2 * i + 1 > limit) pv.y = 0.f;
    }
    const float2 dv = fmul2(pv, fadd2(gv, nd2));
    ds[i] = pack_bf16x2(dv.x, dv.y);
  }
}

// P^T and dS^T of one 64-query half of a key row.  The products already hold the query
// statistics (an extra K step adds -lse / scale to S^T and -D to dP^T, column by column), so
// p = 2^(c s') and dS = p dP'; ca0 is the half's first query column.  kMask: query q0 + ca
// sees this key only when ca >= first_ok (causal) and the key is below the key limit (row_ok).
template <bool kMask>
__device__ __forceinline__ void dkdv_half(const uint32_t* s0, const uint32_t* s1,
                                          const uint32_t* g0, const uint32_t* g1, int ca0,
                                          bool row_ok, int first_ok, float c, uint32_t* pp,
                                          uint32_t* ds) {
  const float2 c2 = make_float2(c, c);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int ca = ca0 + 2 * i;  // query column within the tile
    const float2 sv = make_float2(__uint_as_float(i < 16 ? s0[2 * i] : s1[2 * i - 32]),
                                  __uint_as_float(i < 16 ? s0[2 * i + 1] : s1[2 * i + 1 - 32]));
    const float2 gv = make_float2(__uint_as_float(i < 16 ? g0[2 * i] : g1[2 * i - 32]),
                                  __uint_as_float(i < 16 ? g0[2 * i + 1] : g1[2 * i + 1 - 32]));
    float2 pv = fmul2(sv, c2);
    pv.x = ex2_approx(pv.x);
    pv.y = ex2_approx(pv.y);
    if (kMask) {
      if (!row_ok || ca < first_ok) pv.x = 0.f;
      if (!row_ok || ca + 1 < first_ok) pv.y = 0.f;
    }
    pp[i] = pack_bf16x2(pv.x, pv.y);
    const float2 dv = fmul2(pv, gv);
    ds[i] = pack_bf16x2(dv.x, dv.y);
  }
}

// store 32 fp32 values (times mul) of half a row as bf16
__device__ __forceinline__ void store_half_row(__nv_bfloat16* dst, const uint32_t* r,
                                               float mul) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint32_t* q = r + 8 * u;
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(q[0]) * mul, __uint_as_float(q[1]) * mul);
    v.y = pack_bf16x2(__uint_as_float(q[2]) * mul, __uint_as_float(q[3]) * mul);
    v.z = pack_bf16x2(__uint_as_float(q[4]) * mul, __uint_as_float(q[5]) * mul);
    v.w = pack_bf16x2(__uint_as_float(q[6]) * mul, __uint_as_float(q[7]) * mul);
    d4[u] = v;
  }
}

// ============================================================================ dq kernel
// smem: Q, dO (once), K ring, V ring, barriers
constexpr int kQOffQ = 0;
constexpr int kQOffG = kQOffQ + kTileBytes;
constexpr int kQOffK = kQOffG + kTileBytes;
constexpr int kQOffV = kQOffK + kStages * kTileBytes;
constexpr int kQOffBar = kQOffV + kStages * kTileBytes;
constexpr int kQSmem = 1024 + kQOffBar + 256;
// TMEM: S [0,128) dP [128,256) dS of even tiles (bf16 pairs) [256,320) dQ [320,384) dS of
// odd tiles [384,448): the math warps write dS(j+1) while dQ += dS(j) K_j still reads dS(j)
constexpr uint32_t kQColS = 0, kQColP = 128, kQColDQ = 320;
__device__ __forceinline__ uint32_t q_col_ds(int j) { return (j & 1) ? 384u : 256u; }
// barriers
constexpr int kQBarIn = 0;                     // Q, dO landed
constexpr int kQBarKV = 1;                     // [kStages] K_j, V_j landed
constexpr int kQBarKVEmpty = kQBarKV + kStages;  // [kStages] both issuers done with K_j, V_j
constexpr int kQBarSFull = kQBarKVEmpty + kStages;
constexpr int kQBarSFree = kQBarSFull + 1;   // every math warp holds its S, dP half
constexpr int kQBarDSFull = kQBarSFree + 1;  // [2] every math warp wrote its dS half
constexpr int kQBarDQDone = kQBarDSFull + 2; // [2] dQ MMA done with that dS buffer
constexpr int kQBarDrain = kQBarDQDone + 2;
constexpr int kQNumBars = kQBarDrain + 1;

__global__ void __launch_bounds__(kQThreads, 1)
    sdpa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmG, const BwdParams p) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kQNumBars);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int q0 = qt * kT;
  const int L = key_limit(p, b);
  // key tiles this query tile needs: causal stops at the diagonal tile
  int nk = (L + kT - 1) / kT;
  if (p.mask == 1) nk = min(nk, (min(q0 + kT, p.Nq) - 1) / kT + 1);

  if (threadIdx.x == 0) {
    mbar_init(bar(kQBarIn), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kQBarKV + s), 1);
      mbar_init(bar(kQBarKVEmpty + s), 2);  // the S/dP issuer and the dQ issuer
    }
    mbar_init(bar(kQBarSFull), 1);
    mbar_init(bar(kQBarSFree), kMathWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kQBarDSFull + i), kMathWarps);
      mbar_init(bar(kQBarDQDone + i), 1);
    }
    mbar_init(bar(kQBarDrain), 2);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nk > 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmG);
      mbar_arrive_expect_tx(bar(kQBarIn), 2 * kTileBytes);
      tma_load_4d(smem_u32(smem + kQOffQ), &tmQ, bar(kQBarIn), 0, q0, h, b);
      tma_load_4d(smem_u32(smem + kQOffG), &tmG, bar(kQBarIn), 0, q0, h, b);
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < nk; ++j) {
        const int s = j % kStages;
        if (!mbar_wait_backoff(bar(kQBarKVEmpty + s), ((j / kStages) & 1) ^ 1, p.timeout_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kQBarKV + s), 2 * kTileBytes);
        tma_load_4d(smem_u32(smem + kQOffK + s * kTileBytes), &tmK, bar(kQBarKV + s), 0, j * kT,
                    h, b);
        tma_load_4d(smem_u32(smem + kQOffV + s * kTileBytes), &tmV, bar(kQBarKV + s), 0, j * kT,
                    h, b);
        issued = j + 1;
      }
      if (!ok) record_error(p.status, kErrTimeout, kSiteBwdProducer);
      (void)mbar_wait(bar(kQBarIn), 0, p.timeout_ns);
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        (void)mbar_wait(bar(kQBarKV + i % kStages), (i / kStages) & 1, p.timeout_ns);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ S and dP issuer
    if (lane == 0 && nk > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kT, kT, false, false);
      const uint64_t dQd = smem_desc_sw128(smem_u32(smem + kQOffQ), 1024, 1024);
      const uint64_t dGd = smem_desc_sw128(smem_u32(smem + kQOffG), 1024, 1024);
      // S_j = Q K_j^T and dP_j = dO V_j^T into the single S/dP buffer
      auto issue_s = [&](int j) -> bool {
        const int s = j % kStages;
        if (!mbar_wait(bar(kQBarKV + s), (j / kStages) & 1, p.timeout_ns)) return false;
        tc_fence_after();
        const uint64_t dK = smem_desc_sw128(smem_u32(smem + kQOffK + s * kTileBytes), 1024, 1024);
        const uint64_t dV = smem_desc_sw128(smem_u32(smem + kQOffV + s * kTileBytes), 1024, 1024);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {  // 16 of d per MMA = 32 B in the swizzle row
          mma_bf16_ss(tmem + kQColS, dQd + kk * 2, dK + kk * 2, idS, kk > 0 ? 1u : 0u);
          mma_bf16_ss(tmem + kQColP, dGd + kk * 2, dV + kk * 2, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(kQBarSFull));
        mma_commit(bar(kQBarKVEmpty + s));  // this issuer is done with K_j, V_j
        return true;
      };
      bool ok = mbar_wait(bar(kQBarIn), 0, p.timeout_ns) && issue_s(0);
      // once the math warps hold S_j and dP_j in registers the next tile's products run
      // while they turn them into dS_j
      for (int j = 0; ok && j + 1 < nk; ++j)
        ok = mbar_wait(bar(kQBarSFree), j & 1, p.timeout_ns) && issue_s(j + 1);
      if (!ok) record_error(p.status, kErrTimeout, kSiteBwdMma);
      mma_commit(bar(kQBarDrain));
      (void)mbar_wait(bar(kQBarDrain), 0, p.timeout_ns);  // no MMA of this CTA in flight
    }
  } else if (warp == kWarpMma2) {
    // ------------------------------------------------------------ dQ issuer
    if (lane == 0 && nk > 0) {
      constexpr uint32_t idQ = idesc_bf16_f32(kT, kHD, false, true);
      bool ok = true;
      for (int j = 0; ok && j < nk; ++j) {
        const int s = j % kStages;
        // dS_j written (and K_j landed, which the S issuer saw before S_j)
        if (!mbar_wait(bar(kQBarDSFull + (j & 1)), (j >> 1) & 1, p.timeout_ns) ||
            !mbar_wait(bar(kQBarKV + s), (j / kStages) & 1, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dK = smem_desc_sw128(smem_u32(smem + kQOffK + s * kTileBytes), 1024, 1024);
        // dQ += dS K_j: 16 keys (8 TMEM columns of dS, 16 K rows) per MMA
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_bf16_ts(tmem + kQColDQ, tmem + q_col_ds(j) + kk * 8, dK + kk * ((16 * 128) >> 4),
                      idQ, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(kQBarDQDone + (j & 1)));
        mma_commit(bar(kQBarKVEmpty + s));
      }
      if (!ok) record_error(p.status, kErrTimeout, kSiteBwdMma);
      mma_commit(bar(kQBarDrain));
      (void)mbar_wait(bar(kQBarDrain), 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ math warps
    const int quarter = warp & 3, half = warp >> 2;
    const int r_local = quarter * 32 + lane;
    const int row = q0 + r_local;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const bool live = row < p.Nq;
    const float* tile_st =
        p.stats + ((static_cast<int64_t>(b) * p.H + h) * gridDim.x + qt) * (2 * kT);
    const float nl = __ldg(tile_st + r_local);  // -lse2; -inf past Nq
    const float nd = __ldg(tile_st + kT + r_local);  // -D
    const float c = p.scale * kLog2e;
    const int limit = (p.mask == 1) ? min(row, L - 1) : L - 1;  // keys j <= limit
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
      if (!warp_all(mbar_wait(bar(kQBarSFull), j & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteBwdMath);
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s0[32], s1[32], g0[32], g1[32];
      tmem_ld32(tmem + kQColS + lane_off + half * 64, s0);
      tmem_ld32(tmem + kQColS + lane_off + half * 64 + 32, s1);
      tmem_ld32(tmem + kQColP + lane_off + half * 64, g0);
      tmem_ld32(tmem + kQColP + lane_off + half * 64 + 32, g1);
      tmem_wait_ld();
      reg_fence(s0);
      reg_fence(s1);
      reg_fence(g0);
      reg_fence(g1);
      // S and dP of this half are in registers: the next tile's products may overwrite them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kQBarSFree));
      const int col0 = j * kT + half * 64;
      uint32_t ds[32];
      if (warp_all(col0 + 63 <= limit))  // no key of this half is masked for any row here
        dq_half<false>(s0, s1, g0, g1, col0, limit, c, nl, nd, ds);
      else
        dq_half<true>(s0, s1, g0, g1, col0, limit, c, nl, nd, ds);
      // dS_j goes to buffer j % 2, which dQ += dS_{j-2} K_{j-2} must have finished reading
      if (j > 1 && !warp_all(mbar_wait(bar(kQBarDQDone + (j & 1)), ((j >> 1) - 1) & 1,
                                       p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteBwdMath);
        ok = false;
        break;
      }
      tmem_st32(tmem + q_col_ds(j) + lane_off + half * 32, ds);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kQBarDSFull + (j & 1)));
    }
    // ---- epilogue: dQ * scale -> bf16, 32 of the 64 columns per warp
    __nv_bfloat16* dst =
        p.out0 + b * p.o0_b + h * p.o0_h + static_cast<int64_t>(row) * p.o0_n + half * 32;
    uint32_t r0[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r0[i] = 0u;
    if (ok && nk > 0) {
      if (warp_all(mbar_wait(bar(kQBarDQDone + ((nk - 1) & 1)), ((nk - 1) >> 1) & 1,
                             p.timeout_ns))) {
        tc_fence_after();
        tmem_ld32(tmem + kQColDQ + lane_off + half * 32, r0);
        tmem_wait_ld();
        reg_fence(r0);
      } else {
        record_error(p.status, kErrTimeout, kSiteBwdEpi);
      }
    }
    if (live) store_half_row(dst, r0, p.scale);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ dkdv kernel
// One CTA per 128-key tile.  kFused (the default path) also produces this key tile's share of
// dQ: dQ_i += dS_i K for every query tile i it walks, added in fp32 into a workspace
// accumulator by bulk tensor reductions, so no second kernel rebuilds S and dP for dQ.
// smem: K, V (once), Q ring, dO ring, ring of the query tiles' 8 KB extra-K-step operands
// (-lse / scale and -D, no swizzle), the key side's constant extra-K-step operand, then, fused,
// dS^T (two 64-query halves, each laid out like a 128-row swizzled tile) and one 32 x 32 fp32
// staging box per math warp, then barriers
constexpr int kKOffK = 0;
constexpr int kKOffV = kKOffK + kTileBytes;
constexpr int kKOffQ = kKOffV + kTileBytes;
constexpr int kKOffG = kKOffQ + kStages * kTileBytes;
constexpr int kAugBytes = 8192;
constexpr int kKOffAug = kKOffG + kStages * kTileBytes;    // [kStages][4 chunks][128][16 B]
constexpr int kKOffKAug = kKOffAug + kStages * kAugBytes;  // [2 chunks][128][16 B]
constexpr int kKOffDS = kKOffKAug + 4096;                  // fused only
constexpr int kKOffStage = kKOffDS + 2 * kTileBytes;       // fused only: [kMathWarps][4 KB]
constexpr int kStageBytes = 32 * 32 * 4;
__host__ __device__ constexpr int k_off_bar(bool fused) {
  return fused ? kKOffStage + kMathWarps * kStageBytes : kKOffDS;
}
__host__ __device__ constexpr int k_smem(bool fused) { return 1024 + k_off_bar(fused) + 256; }
static_assert(kKOffDS % 1024 == 0 && kKOffStage % 1024 == 0, "swizzled buffers need 1 KB alignment");
static_assert(k_smem(true) <= 227 * 1024, "fused dkdv shared memory");
// TMEM: S^T [0,128) dP^T [128,256) P^T [256,320) dS^T (fused: dQ of one query tile) [320,384)
// dV [384,448) dK [448,512)
constexpr uint32_t kKColS = 0, kKColP = 128, kKColPT = 256, kKColDS = 320, kKColDQ = 320,
                   kKColDV = 384, kKColDK = 448;
constexpr int kKBarIn = 0;                        // K, V landed
constexpr int kKBarQ = 1;                         // [kStages] Q_i, dO_i, lse, D landed
constexpr int kKBarQEmpty = kKBarQ + kStages;     // [kStages] all three issuers done with Q_i, dO_i
constexpr int kKBarSFull = kKBarQEmpty + kStages;
constexpr int kKBarSFree = kKBarSFull + 1;        // every math warp holds its S^T, dP^T half
constexpr int kKBarPFull = kKBarSFree + 1;        // every math warp wrote its P^T, dS^T half
constexpr int kKBarDVDone = kKBarPFull + 1;       // dV += P^T dO done with P^T
constexpr int kKBarDKDone = kKBarDVDone + 1;      // dK += dS^T Q (fused: and dQ = dS K) done
constexpr int kKBarDrain = kKBarDKDone + 1;
constexpr int kKNumBars = kKBarDrain + 1;

// 32 consecutive 32-bit words of a thread's row into a 128-byte row of a 128-byte-swizzled
// buffer: 16-byte unit u lands at u ^ (row % 8), the layout tensor-core operands and bulk
// tensor copies use (row % 8 == lane % 8 for every caller here)
__device__ __forceinline__ void st_row_sw128(uint32_t row_addr, int lane, const uint32_t* v) {
#pragma unroll
  for (int u = 0; u < 8; ++u)
    st_shared_v4(row_addr + ((u ^ (lane & 7)) << 4),
                 make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]));
}

template <bool kFused>
__global__ void __launch_bounds__(kKThreads, 1)
    sdpa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmG,
                         const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output is complete from here on
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + k_off_bar(kFused));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kKNumBars);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int k0 = kt * kT;
  const int L = key_limit(p, b);
  const int nqt = (p.Nq + kT - 1) / kT;
  // query tiles that can see any key of this tile: causal starts at the diagonal tile; a tile
  // past key_len is seen by none
  const int i0 = (p.mask == 1) ? kt : 0;
  const int ni = (k0 < L) ? max(nqt - i0, 0) : 0;

  if (threadIdx.x == 0) {
    mbar_init(bar(kKBarIn), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kKBarQ + s), 1);
      mbar_init(bar(kKBarQEmpty + s), 3);  // the S/dP, dV and dK issuers
    }
    mbar_init(bar(kKBarSFull), 1);
    mbar_init(bar(kKBarSFree), kMathWarps);
    mbar_init(bar(kKBarPFull), kMathWarps);
    mbar_init(bar(kKBarDVDone), 1);
    mbar_init(bar(kKBarDKDone), 1);
    mbar_init(bar(kKBarDrain), 3);
    fence_mbar_init();
  }
  if (threadIdx.x < kT) {
    // the key side of the extra K step: columns 0-2 of every row are 1 (they pick up the
    // three bf16 terms of the query side), the rest 0; core matrices without swizzle
    const uint32_t row = smem_u32(smem + kKOffKAug) + threadIdx.x * 16;
    st_shared_v4(row, make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u));
    st_shared_v4(row + kT * 16, make_uint4(0u, 0u, 0u, 0u));
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // register split (setmaxnreg): 384 threads launch with 168 registers each (64512); the
  // control warpgroup (producer, three issuers) drops to 72 so the math warps can take 200:
  // 256 x 200 + 128 x 72 = 60416 <= 64512
  if (warp >= kMathWarps) regs_dec<kKControlRegs>();  // first: the math warps' increase waits on it
  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer (TMA)
    if (lane == 0 && ni > 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmG);
      mbar_arrive_expect_tx(bar(kKBarIn), 2 * kTileBytes);
      tma_load_4d(smem_u32(smem + kKOffK), &tmK, bar(kKBarIn), 0, k0, h, b);
      tma_load_4d(smem_u32(smem + kKOffV), &tmV, bar(kKBarIn), 0, k0, h, b);
      const uint8_t* aug_bh = p.aug + (static_cast<int64_t>(b) * p.H + h) * nqt * kAugBytes;
      bool ok = true;
      int issued = 0;
      for (int t = 0; t < ni; ++t) {
        const int s = t % kStages;
        const int qt = i0 + t;
        if (!mbar_wait_backoff(bar(kKBarQEmpty + s), ((t / kStages) & 1) ^ 1, p.timeout_ns)) {
          ok = false;
          break;
        }
        // Q_t, dO_t and the tile's extra-K-step operand (-lse / scale, -D: 8 KB) on one barrier
        mbar_arrive_expect_tx(bar(kKBarQ + s), 2 * kTileBytes + kAugBytes);
        tma_load_4d(smem_u32(smem + kKOffQ + s * kTileBytes), &tmQ, bar(kKBarQ + s), 0, qt * kT,
                    h, b);
        tma_load_4d(smem_u32(smem + kKOffG + s * kTileBytes), &tmG, bar(kKBarQ + s), 0, qt * kT,
                    h, b);
        bulk_load(smem_u32(smem + kKOffAug + s * kAugBytes), aug_bh + qt * kAugBytes, kAugBytes,
                  bar(kKBarQ + s));
        issued = t + 1;
      }
      if (!ok) record_error(p.status, kErrTimeout, kSiteBwdProducer);
      (void)mbar_wait(bar(kKBarIn), 0, p.timeout_ns);
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        (void)mbar_wait(bar(kKBarQ + i % kStages), (i / kStages) & 1, p.timeout_ns);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ S^T and dP^T issuer
    if (lane == 0 && ni > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kT, kT, false, false);
      const uint64_t dKd = smem_desc_sw128(smem_u32(smem + kKOffK), 1024, 1024);
      const uint64_t dVd = smem_desc_sw128(smem_u32(smem + kKOffV), 1024, 1024);
      // the extra K step (no swizzle: 16-byte core-matrix rows, K chunks 2 KB apart): key side
      // all ones in columns 0-2, query side -lse / scale (chunks 0-1) or -D (chunks 2-3)
      const uint64_t dKa = smem_desc_noswizzle(smem_u32(smem + kKOffKAug), kT * 16, 128);
      // S^T_t = K Q_t^T - lse / scale and dP^T_t = V dO_t^T - D into the single S/dP buffer
      auto issue_s = [&](int t) -> bool {
        const int s = t % kStages;
        if (!mbar_wait(bar(kKBarQ + s), (t / kStages) & 1, p.timeout_ns)) return false;
        tc_fence_after();
        const uint64_t dQ = smem_desc_sw128(smem_u32(smem + kKOffQ + s * kTileBytes), 1024, 1024);
        const uint64_t dG = smem_desc_sw128(smem_u32(smem + kKOffG + s * kTileBytes), 1024, 1024);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk) {
          mma_bf16_ss(tmem + kKColS, dKd + kk * 2, dQ + kk * 2, idS, kk > 0 ? 1u : 0u);
          mma_bf16_ss(tmem + kKColP, dVd + kk * 2, dG + kk * 2, idS, kk > 0 ? 1u : 0u);
        }
        const uint64_t dA =
            smem_desc_noswizzle(smem_u32(smem + kKOffAug + s * kAugBytes), kT * 16, 128);
        mma_bf16_ss(tmem + kKColS, dKa, dA, idS, 1u);
        mma_bf16_ss(tmem + kKColP, dKa, dA + ((2 * kT * 16) >> 4), idS, 1u);
        mma_commit(bar(kKBarSFull));
        mma_commit(bar(kKBarQEmpty + s));  // this issuer is done with Q_t, dO_t
        return true;
      };
      bool ok = mbar_wait(bar(kKBarIn), 0, p.timeout_ns) && issue_s(0);
      // once the math warps hold S^T_t and dP^T_t in registers the next tile's products run
      // while they turn them into P^T_t and dS^T_t
      for (int t = 0; ok && t + 1 < ni; ++t)
        ok = mbar_wait(bar(kKBarSFree), t & 1, p.timeout_ns) && issue_s(t + 1);
      if (!ok) record_error(p.status, kErrTimeout, kSiteBwdMma);
      mma_commit(bar(kKBarDrain));
      (void)mbar_wait(bar(kKBarDrain), 0, p.timeout_ns);  // no MMA of this CTA in flight
    }
  } else if (warp == kWarpMma2 || warp == kWarpMma3) {
    // ------------------------------------------------------------ dV issuer / dK (+dQ) issuer
    if (lane == 0 && ni > 0) {
      // B = dO_t or Q_t as an MN-major operand (head dim contiguous); 16 queries per MMA
      constexpr uint32_t idO = idesc_bf16_f32(kT, kHD, false, true);
      const bool is_dv = warp == kWarpMma2;
      const uint32_t acc = tmem + (is_dv ? kKColDV : kKColDK);
      const int b_off = is_dv ? kKOffG : kKOffQ;
      const int done_bar = is_dv ? kKBarDVDone : kKBarDKDone;
      // fused dK: A = dS^T from shared memory, K-major (queries contiguous in each 64-query
      // half); dQ_t = dS K: A = the same bytes read as dS, MN-major (the two 64-query halves
      // are the leading-dimension step), B = K, MN-major; 16 keys per MMA
      constexpr uint32_t idQ = idesc_bf16_f32(kT, kHD, true, true);
      const uint32_t sDS = smem_u32(smem + kKOffDS);
      const uint64_t dsK = smem_desc_sw128(sDS, 1024, 1024);
      const uint64_t dsM = smem_desc_sw128(sDS, kTileBytes, 1024);
      const uint64_t dKt = smem_desc_sw128(smem_u32(smem + kKOffK), 1024, 1024);
      bool ok = true;
      for (int t = 0; ok && t < ni; ++t) {
        const int s = t % kStages;
        // P^T_t, dS^T_t written (and Q_t, dO_t landed, which the S issuer saw before S^T_t)
        if (!mbar_wait(bar(kKBarPFull), t & 1, p.timeout_ns) ||
            !mbar_wait(bar(kKBarQ + s), (t / kStages) & 1, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t bd = smem_desc_sw128(smem_u32(smem + b_off + s * kTileBytes), 1024, 1024);
        if (kFused && !is_dv) {
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_bf16_ss(acc, dsK + (kk >> 2) * (kTileBytes >> 4) + (kk & 3) * 2,
                        bd + kk * ((16 * 128) >> 4), idO, (t > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_bf16_ss(tmem + kKColDQ, dsM + kk * ((16 * 128) >> 4),
                        dKt + kk * ((16 * 128) >> 4), idQ, kk > 0 ? 1u : 0u);
        } else {
          // dV += P^T dO_t, dK += dS^T Q_t with A in TMEM (8 columns of bf16 pairs per MMA)
          const uint32_t a_op = tmem + (is_dv ? kKColPT : kKColDS);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            mma_bf16_ts(acc, a_op + kk * 8, bd + kk * ((16 * 128) >> 4), idO,
                        (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(done_bar));
        mma_commit(bar(kKBarQEmpty + s));
      }
      if (!ok) record_error(p.status, kErrTimeout, kSiteBwdMma);
      mma_commit(bar(kKBarDrain));
      (void)mbar_wait(bar(kKBarDrain), 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ math warps (one key row each)
    regs_inc<kKMathRegs>();
    const int quarter = warp & 3, half = warp >> 2;
    const int r_local = quarter * 32 + lane;
    const int key = k0 + r_local;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = p.scale * kLog2e;
    // fused: this warp's dQ box (query rows 32*quarter.., columns 32*half..) of one query tile
    // goes TMEM -> registers -> its staging buffer -> one bulk reduction into the accumulator
    const uint32_t sStage = smem_u32(smem + kKOffStage + warp * kStageBytes);
    auto reduce_dq = [&](const uint32_t* v, int q0) {
      if (lane == 0) bulk_wait_group_read0();  // the previous box has left the buffer
      __syncwarp();
      st_row_sw128(sStage + lane * 128, lane, v);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_4d(&tmDQ, sStage, half * 32, q0 + quarter * 32, h, b);
        bulk_commit_group();
      }
    };
    bool ok = true;
    for (int t = 0; t < ni; ++t) {
      const int q0 = (i0 + t) * kT;
      if (!warp_all(mbar_wait(bar(kKBarSFull), t & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteBwdMath);
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s0[32], s1[32], g0[32], g1[32];
      tmem_ld32(tmem + kKColS + lane_off + half * 64, s0);
      tmem_ld32(tmem + kKColS + lane_off + half * 64 + 32, s1);
      tmem_ld32(tmem + kKColP + lane_off + half * 64, g0);
      tmem_ld32(tmem + kKColP + lane_off + half * 64 + 32, g1);
      tmem_wait_ld();
      reg_fence(s0);
      reg_fence(s1);
      reg_fence(g0);
      reg_fence(g1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kKBarSFree));
      uint32_t pp[32], ds[32];
      // key j = key is seen by query q0 + ca when j < L and, for the causal mask, j <= q
      const bool row_ok = key < L;
      const int first_ok = (p.mask == 1) ? key - q0 : -kT;
      if (warp_all(row_ok && first_ok <= half * 64))  // every pair of this half is allowed
        dkdv_half<false>(s0, s1, g0, g1, half * 64, row_ok, first_ok, c, pp, ds);
      else
        dkdv_half<true>(s0, s1, g0, g1, half * 64, row_ok, first_ok, c, pp, ds);
      // the previous dV product must have read P^T, and the previous dK (and dQ) product
      // dS^T, before they change
      if (t > 0 && !warp_all(mbar_wait(bar(kKBarDVDone), (t - 1) & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteBwdMath);
        ok = false;
        break;
      }
      tmem_st32(tmem + kKColPT + lane_off + half * 32, pp);
      if (t > 0 && !warp_all(mbar_wait(bar(kKBarDKDone), (t - 1) & 1, p.timeout_ns))) {
        tmem_wait_st();
        record_error(p.status, kErrTimeout, kSiteBwdMath);
        ok = false;
        break;
      }
      if constexpr (kFused) {
        // dQ_{t-1} leaves TMEM before dQ_t (issued after this tile's PFull) overwrites it
        uint32_t dq[32];
        tc_fence_after();
        if (t > 0) tmem_ld32(tmem + kKColDQ + lane_off + half * 32, dq);
        st_row_sw128(smem_u32(smem + kKOffDS + half * kTileBytes) + r_local * 128, lane, ds);
        tmem_wait_st();
        if (t > 0) {
          tmem_wait_ld();
          reg_fence(dq);
        }
        fence_proxy_async_smem();  // dS^T visible to the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kKBarPFull));
        if (t > 0) reduce_dq(dq, q0 - kT);
      } else {
        tmem_st32(tmem + kKColDS + lane_off + half * 32, ds);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kKBarPFull));
      }
    }
    if constexpr (kFused) {
      // the last query tile's dQ box
      if (ok && ni > 0) {
        if (warp_all(mbar_wait(bar(kKBarDKDone), (ni - 1) & 1, p.timeout_ns))) {
          uint32_t dq[32];
          tc_fence_after();
          tmem_ld32(tmem + kKColDQ + lane_off + half * 32, dq);
          tmem_wait_ld();
          reg_fence(dq);
          reduce_dq(dq, (i0 + ni - 1) * kT);
        } else {
          record_error(p.status, kErrTimeout, kSiteBwdEpi);
          ok = false;
        }
      }
    }
    // ---- epilogue: warps of half 0 write dK * scale, those of half 1 dV, as bf16 (zeros for
    // keys no query sees)
    const bool live = key < p.Nk;
    uint32_t a0[32], a1[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) a0[i] = a1[i] = 0u;
    const uint32_t col = half == 0 ? kKColDK : kKColDV;
    if (ok && ni > 0) {
      if (warp_all(mbar_wait(bar(half == 0 ? kKBarDKDone : kKBarDVDone), (ni - 1) & 1,
                             p.timeout_ns))) {
        tc_fence_after();
        tmem_ld32(tmem + col + lane_off, a0);
        tmem_ld32(tmem + col + lane_off + 32, a1);
        tmem_wait_ld();
        reg_fence(a0);
        reg_fence(a1);
      } else {
        record_error(p.status, kErrTimeout, kSiteBwdEpi);
      }
    }
    if (live) {
      if (half == 0)
        store_row(p.out0 + b * p.o0_b + h * p.o0_h + static_cast<int64_t>(key) * p.o0_n, a0,
                  a1, p.scale);
      else
        store_row(p.out1 + b * p.o1_b + h * p.o1_h + static_cast<int64_t>(key) * p.o1_n, a0,
                  a1, 1.f);
    }
    // this warp's reductions have landed in global memory before the block ends
    if (kFused && lane == 0) bulk_wait_group0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dQ = scale * accumulator, as bf16 in dQ's layout; one thread per 8 consecutive values
__global__ void __launch_bounds__(256)
    sdpa_bwd_dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                               int H, int Nq, int rows, int64_t sb, int64_t sh, int64_t sn,
                               float scale, int64_t total) {
  pdl_launch_dependents();
  pdl_wait();  // the fused kernel's reductions are complete from here on
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int part = static_cast<int>(i & 7);
    const int64_t r = i >> 3;  // (b, h, n) with n < Nq
    const int n = static_cast<int>(r % Nq);
    const int64_t bh = r / Nq;
    const int hh = static_cast<int>(bh % H);
    const int64_t bb = bh / H;
    const float4* src = reinterpret_cast<const float4*>(acc + (bh * rows + n) * 64 + part * 8);
    const float4 x = __ldcs(src), y = __ldcs(src + 1);
    uint4 v;
    v.x = pack_bf16x2(x.x * scale, x.y * scale);
    v.y = pack_bf16x2(x.z * scale, x.w * scale);
    v.z = pack_bf16x2(y.x * scale, y.y * scale);
    v.w = pack_bf16x2(y.z * scale, y.w * scale);
    *reinterpret_cast<uint4*>(dq + bb * sb + hh * sh + static_cast<int64_t>(n) * sn + part * 8) =
        v;
  }
}

}  // namespace

cudaError_t launch_sdpa_bwd_bf16(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmG,
                                 const CUtensorMap& tmDQ, const SdpaBwdArgs& a,
                                 const DevCtx& ctx, cudaStream_t s) {
  BwdParams p;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.mask = a.mask;
  p.key_len = a.key_len;
  p.scale = a.scale;
  p.stats = a.Dv;
  p.aug = reinterpret_cast<const uint8_t*>(a.Dv) + sdpa_bwd_aug_offset(a.B, a.H, a.Nq);
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  const bool fused = !a.deterministic;
  const void* kdkdv = fused ? reinterpret_cast<const void*>(sdpa_bwd_dkdv_kernel<true>)
                            : reinterpret_cast<const void*>(sdpa_bwd_dkdv_kernel<false>);
  int regs = 0;
  cudaError_t e = prepare_kernel(kdkdv, k_smem(fused), &regs);
  if (e != cudaSuccess) return e;
  // the dkdv kernel's setmaxnreg split must fit in what its blocks launch with, or the
  // increase would wait forever: refuse to launch if the compiled register count is too small
  if (regs * kKThreads < kMathWarps * 32 * kKMathRegs + 4 * 32 * kKControlRegs)
    return cudaErrorInvalidConfiguration;
  if (!fused) {
    e = prepare_kernel(reinterpret_cast<const void*>(sdpa_bwd_dq_kernel), kQSmem, nullptr);
    if (e != cudaSuccess) return e;
    p.out0 = static_cast<__nv_bfloat16*>(a.dQ);
    p.o0_b = a.st[5][0];
    p.o0_h = a.st[5][1];
    p.o0_n = a.st[5][2];
    (void)launch_pdl(sdpa_bwd_dq_kernel, dim3((a.Nq + kT - 1) / kT, a.H, a.B), dim3(kQThreads),
                     kQSmem, s, tmQ, tmK, tmV, tmG, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  p.out0 = static_cast<__nv_bfloat16*>(a.dK);
  p.o0_b = a.st[6][0];
  p.o0_h = a.st[6][1];
  p.o0_n = a.st[6][2];
  p.out1 = static_cast<__nv_bfloat16*>(a.dV);
  p.o1_b = a.st[7][0];
  p.o1_h = a.st[7][1];
  p.o1_n = a.st[7][2];
  const dim3 grid((a.Nk + kT - 1) / kT, a.H, a.B);
  if (fused)
    (void)launch_pdl(sdpa_bwd_dkdv_kernel<true>, grid, dim3(kKThreads), k_smem(true), s, tmQ, tmK,
                     tmV, tmG, tmDQ, p);
  else
    (void)launch_pdl(sdpa_bwd_dkdv_kernel<false>, grid, dim3(kKThreads), k_smem(false), s, tmQ,
                     tmK, tmV, tmG, tmDQ, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || !fused) return e;
  const int rows = (a.Nq + kT - 1) / kT * kT;
  const int64_t total = static_cast<int64_t>(a.B) * a.H * a.Nq * 8;
  const int64_t want = (total + 255) / 256;
  const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(ctx.num_sms) * 8));
  (void)launch_pdl(sdpa_bwd_dq_convert_kernel, dim3(blocks), dim3(256), 0, s,
                   reinterpret_cast<const float*>(reinterpret_cast<const char*>(a.Dv) +
                                                  sdpa_bwd_dq_acc_offset(a.B, a.H, a.Nq)),
                   static_cast<__nv_bfloat16*>(a.dQ), a.H, a.Nq, rows, a.st[5][0], a.st[5][1],
                   a.st[5][2], a.scale, total);
  return cudaGetLastError();
}

}  // namespace mha
