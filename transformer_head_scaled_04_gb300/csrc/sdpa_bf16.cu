// sdpa_bf16.cu -- fused scaled dot-product attention forward on the sm_103a tensor cores.
//
//   O = softmax(Q K^T / sqrt(d_k)) V per (batch, head), optional causal, key-padding or band
//   mask ("Attention Is All You Need", lettle.cn translation, 3.2.1 缩放点积注意力;
//    "Transformer：抛弃循环与卷积的序列建模", Scaled Dot-Product Attention, the three uses of
//    attention, 训练样本 for the causal mask, Self-Attention的优势 for the restricted form).
//
// The n x n score matrix never leaves the SM.  A CTA owns one 128-row query tile of one (b, h)
// and streams K/V in 128-row tiles; with 192 threads, ~97 KB of shared memory and 256 TMEM
// columns two CTAs share each SM, so on each SMSP two softmax warps of different tiles take
// turns with the exponentials while either CTA's tensor-core products run.  (An earlier design,
// one persistent CTA per SM owning two query tiles on 384 threads and all 512 TMEM columns,
// with its two softmax warpgroups staggered and consecutive work units overlapped through
// launch-cancel takeovers, ran the big model's heads 6% slower.)
//   warps 0-3  softmax, one query row per thread (its TMEM lane): one tcgen05.ld brings the whole
//              128-key S row into registers; the mask; p = 2^(s c - m c) with c = scale
//              log2(e) in paired fp32 FMA / add against the exact row max of the first key
//              tile (later tiles take no max pass and O no rescale: p and l share the
//              reference, so O / l is exact; a tile whose row sum passes 2^64 is redone from
//              TMEM with its true max after rescaling O and l); S released, then P as bf16 into
//              TMEM once the previous P.V has read it; at the end O / l staged in the Q buffer
//              (128-byte swizzle) and written by one bulk tensor store per warp, straight into
//              any strided layout (the head-concat layout [B, Nq, H*64] in the sublayer)
//   warp 4     TMA producer: Q, then K and V through separate rings (two and three slots); it
//              sets up the barriers and requests Q and the first K and V tiles before the block
//              synchronises (their latency overlaps the TMEM allocation; -1 to -2% in A/B)
//   warp 5     TMEM owner and MMA issuer: S = Q K_j^T (tcgen05.mma 128x128x16, fp32 in TMEM)
//              as soon as the softmax warps have read S_{j-1}, O += P_j V_j (128x64x16, P from
//              TMEM, V an MN-major shared-memory operand)
// Whole K/V tiles past the causal diagonal, past key_len[b] or outside a band are never loaded.
// The query tiles of one (b, h) are adjacent in launch order (they share K/V in L2); with a
// causal mask (tile k costs k + 1 key tiles) all heads' heaviest tiles launch first.  Every
// wait is bounded (see device_common.cuh); a timeout records MHA_ERR_DEVICE_TIMEOUT and the
// CTA winds down.
#include <cuda_bf16.h>

#include <cmath>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kBQ = 128;   // query rows per CTA
constexpr int kBKV = 128;  // keys per K/V tile
constexpr int kHD = 64;    // head dim (d_k = d_v)
constexpr int kKRing = 2;  // K ring depth
constexpr int kVRing = 3;  // V ring depth (a third slot: causal 277 -> 271 us in A/B)
// 192 threads at <= 170 registers each (two CTAs per SM); the softmax warps' S row and P fit
// without a register split (the producer and issuer warps are only half a warpgroup, so they
// could not take part in one)
constexpr int kThreads = 192;
constexpr int kTileBytes = kBQ * kHD * 2;  // 16 KB
constexpr int kOffQ = 0;                   // also stages O at the end
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kKRing * kTileBytes;
constexpr int kOffBar = kOffV + kVRing * kTileBytes;
constexpr int kSmemBytes = 1024 + kOffBar + 256;
// TMEM columns: S [0,128) O [128,192) P [192,256) (P: 128 bf16 per row, two per column)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 128;
constexpr uint32_t kColP = 192;

constexpr int kErrTimeout = -6;
enum : int {
  kSiteProducer = 71,
  kSiteMma = 72,
  kSiteSoftmaxS = 73,
  kSiteSoftmaxO = 74,
  kSiteEpilogue = 75,
  kSiteKeyLen = 76,  // index checks (MHA_DEBUG_BOUNDS builds)
  kSiteLse = 77,
  kSiteZeroRows = 78
};

constexpr int kBarQ = 0;
constexpr int kBarKFull = 1;
constexpr int kBarKEmpty = kBarKFull + kKRing;
constexpr int kBarVFull = kBarKEmpty + kKRing;
constexpr int kBarVEmpty = kBarVFull + kVRing;
constexpr int kBarSFull = kBarVEmpty + kVRing;
constexpr int kBarSFree = kBarSFull + 1;
constexpr int kBarPFull = kBarSFree + 1;
constexpr int kBarODone = kBarPFull + 1;
constexpr int kBarDrain = kBarODone + 1;
constexpr int kNumBars = kBarDrain + 1;

struct Params {
  int B, H, Nq, Nk, mask, window;
  const int32_t* key_len;
  float scale_log2;
  float* lse;
  __nv_bfloat16* O;  // direct stores for rows that see no key (zeros)
  int64_t so_b, so_h, so_n;
  int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// kHeavyFirst (causal masks): the launch order maps to query tiles heaviest first across all
// heads; the other masks keep the query tiles of a head adjacent.  Two instantiations, because
// the remapping in the same code slowed unmasked attention ~1% (461 against 457 us in A/B).
template <bool kHeavyFirst>
__global__ void __launch_bounds__(kThreads, 2)
    sdpa_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmO, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sK = smem_u32(smem + kOffK);
  const uint32_t sV = smem_u32(smem + kOffV);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // the unit: query rows q0.. of head h of batch element b, key tiles kt0 .. kt0 + nt - 1
  int qt, h, b;
  if constexpr (kHeavyFirst) {
    const int lin =
        static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    const int bh = p.B * p.H;
    qt = static_cast<int>(gridDim.x) - 1 - lin / bh;
    h = (lin % bh) % p.H;
    b = (lin % bh) / p.H;
  } else {
    qt = static_cast<int>(blockIdx.x);
    h = static_cast<int>(blockIdx.y);
    b = static_cast<int>(blockIdx.z);
  }
  const int q0 = qt * kBQ;
  int L = p.Nk;
  if (p.mask == 2 && bounds_ok(b, p.B, p.status, kSiteKeyLen))
    L = min(max(__ldg(p.key_len + b), 0), p.Nk);
  const int last = min(q0 + kBQ, p.Nq) - 1;
  int kt0 = 0, nt;
  if (p.mask == 1) {
    nt = last / kBKV + 1;
  } else if (p.mask == kMaskWindow) {
    kt0 = max(q0 - p.window, 0) / kBKV;
    nt = min(last + p.window, p.Nk - 1) / kBKV - kt0 + 1;
  } else {
    nt = (L + kBKV - 1) / kBKV;
  }

  // The producer thread sets up the barriers and, once the previous kernel's output is
  // complete, asks for Q and the first K and V tiles before the block synchronises, so their
  // latency overlaps the TMEM allocation and the barrier set-up of the other warps.
  const bool producer = warp == 4 && lane == 0;
  if (producer) {
    mbar_init(bar(kBarQ), 1);
    for (int i = 0; i < kKRing; ++i) {
      mbar_init(bar(kBarKFull + i), 1);
      mbar_init(bar(kBarKEmpty + i), 1);
    }
    for (int i = 0; i < kVRing; ++i) {
      mbar_init(bar(kBarVFull + i), 1);
      mbar_init(bar(kBarVEmpty + i), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), 4);  // one arrival per softmax warp
    mbar_init(bar(kBarPFull), kBQ);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarDrain), 1);
    fence_mbar_init();
    if (nt > 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      pdl_wait();  // the previous kernel's output (Q, K, V) is complete from here on
      mbar_arrive_expect_tx(bar(kBarQ), kTileBytes);
      tma_load_4d(sQ, &tmQ, bar(kBarQ), 0, q0, h, b);
      mbar_arrive_expect_tx(bar(kBarKFull), kTileBytes);
      tma_load_4d(sK, &tmK, bar(kBarKFull), 0, kt0 * kBKV, h, b);
      mbar_arrive_expect_tx(bar(kBarVFull), kTileBytes);
      tma_load_4d(sV, &tmV, bar(kBarVFull), 0, kt0 * kBKV, h, b);
    }
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output (Q, K, V) is complete from here on

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && nt > 0) {
      bool ok = true;
      int kn = 1, vn = 1;  // K and V tiles requested (the first of each before the sync)
      for (int j = 1; ok && j < nt; ++j) {
        const int sl = j % kKRing, vs = j % kVRing;
        const uint32_t par = ((j / kKRing) & 1) ^ 1, vpar = ((j / kVRing) & 1) ^ 1;
        if (!mbar_wait_backoff(bar(kBarKEmpty + sl), par, p.timeout_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarKFull + sl), kTileBytes);
        tma_load_4d(sK + sl * kTileBytes, &tmK, bar(kBarKFull + sl), 0, (kt0 + j) * kBKV, h, b);
        ++kn;
        if (!mbar_wait_backoff(bar(kBarVEmpty + vs), vpar, p.timeout_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarVFull + vs), kTileBytes);
        tma_load_4d(sV + vs * kTileBytes, &tmV, bar(kBarVFull + vs), 0, (kt0 + j) * kBKV, h, b);
        ++vn;
      }
      if (!ok) record_error(p.status, kErrTimeout, kSiteProducer);
      // every copy started here lands before the CTA can exit
      (void)mbar_wait(bar(kBarQ), 0, p.timeout_ns);
      for (int j = (kn > kKRing ? kn - kKRing : 0); j < kn; ++j)
        (void)mbar_wait(bar(kBarKFull + j % kKRing), (j / kKRing) & 1, p.timeout_ns);
      for (int j = (vn > kVRing ? vn - kVRing : 0); j < vn; ++j)
        (void)mbar_wait(bar(kBarVFull + j % kVRing), (j / kVRing) & 1, p.timeout_ns);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBQ, kBKV, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(kBQ, kHD, false, true);
      const uint64_t dQ = smem_desc_sw128(sQ, 1024, 1024);
      const uint64_t dK0 = smem_desc_sw128(sK, 1024, 1024);
      const uint64_t dV0 = smem_desc_sw128(sV, 1024, 1024);
      bool ok = mbar_wait(bar(kBarQ), 0, p.timeout_ns);
      // S(j) = Q K(j)^T once the softmax warps have read S(j-1) out of TMEM
      auto issue_s = [&](int j) -> bool {
        const int sl = j % kKRing;
        if (!mbar_wait(bar(kBarKFull + sl), (j / kKRing) & 1, p.timeout_ns)) return false;
        if (j > 0 && !mbar_wait(bar(kBarSFree), (j - 1) & 1, p.timeout_ns)) return false;
        tc_fence_after();
        const uint64_t bk = dK0 + static_cast<uint64_t>((sl * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk)
          mma_bf16_ss(tmem, dQ + kk * 2, bk + kk * 2, idS, kk > 0 ? 1u : 0u);
        mma_commit(bar(kBarKEmpty + sl));
        mma_commit(bar(kBarSFull));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 1; ok && j <= nt; ++j) {
        if (j < nt && !(ok = issue_s(j))) break;
        // O += P(j-1) V(j-1) once the softmax warps have written P(j-1)
        const int pj = j - 1, sl = pj % kVRing;
        if (!mbar_wait(bar(kBarPFull), pj & 1, p.timeout_ns) ||
            !mbar_wait(bar(kBarVFull + sl), (pj / kVRing) & 1, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t bv = dV0 + static_cast<uint64_t>((sl * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBKV / 16; ++kk)  // 16 keys = 8 TMEM columns of P, 16 V rows
          mma_bf16_ts(tmem + kColO, tmem + kColP + kk * 8, bv + kk * ((16 * 128) >> 4), idO,
                      (pj > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(kBarVEmpty + sl));
        mma_commit(bar(kBarODone));
      }
      if (!ok) record_error(p.status, kErrTimeout, kSiteMma);
      mma_commit(bar(kBarDrain));
      (void)mbar_wait(bar(kBarDrain), 0, p.timeout_ns);  // no MMA in flight past this point
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int quarter = warp;
    const int row = q0 + quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off;
    const uint32_t tO = tmem + kColO + lane_off;
    const uint32_t tP = tmem + kColP + lane_off;
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    // allowed keys of this row: first <= key <= limit; both grow with the row, so the warp's
    // smallest limit is its first row's and its largest first key its last row's
    const int limit = (p.mask == 1)             ? row
                      : (p.mask == kMaskWindow) ? min(row + p.window, p.Nk - 1)
                                                : L - 1;
    const int first = (p.mask == kMaskWindow) ? row - p.window : 0;
    const int wr0 = q0 + quarter * 32;
    const int lim_min = (p.mask == 1)             ? wr0
                        : (p.mask == kMaskWindow) ? min(wr0 + p.window, p.Nk - 1)
                                                  : L - 1;
    const int first_max = (p.mask == kMaskWindow) ? wr0 + 31 - p.window : 0;
    bool ok = true;
    float m_used = -INFINITY;
    float l = 0.f;
    for (int j = 0; j < nt; ++j) {
      if (!warp_all(mbar_wait(bar(kBarSFull), j & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteSoftmaxS);
        ok = false;
        break;
      }
      tc_fence_after();
      const int col0 = (kt0 + j) * kBKV;
      const int hi = limit - col0;  // keys q > hi or q < lo of the tile are excluded
      const int lo = first - col0;
      const bool mask_hi = lim_min - col0 < kBKV - 1;
      const bool mask_lo = first_max - col0 > 0;
      float sv[128];
      auto load_s = [&]() {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld32(tS + 0, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_wait_ld();
        reg_fence(r0);
        reg_fence(r1);
        reg_fence(r2);
        reg_fence(r3);
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          sv[q] = __uint_as_float(r0[q]);
          sv[32 + q] = __uint_as_float(r1[q]);
          sv[64 + q] = __uint_as_float(r2[q]);
          sv[96 + q] = __uint_as_float(r3[q]);
        }
        // excluded keys get -inf (p = 0): one compare against a per-row bound per key,
        // one-sided where no row of the warp has the other end inside the tile
        if (mask_hi || mask_lo) {
          if (!mask_lo) {
#pragma unroll
            for (int q = 0; q < 128; ++q) sv[q] = q > hi ? -INFINITY : sv[q];
          } else if (!mask_hi) {
#pragma unroll
            for (int q = 0; q < 128; ++q) sv[q] = q < lo ? -INFINITY : sv[q];
          } else {
#pragma unroll
            for (int q = 0; q < 128; ++q) sv[q] = (q > hi || q < lo) ? -INFINITY : sv[q];
          }
        }
      };
      auto row_max = [&]() {
        float m4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float* v = sv + 32 * q;
          m4[q] = fmax3(v[0], v[1], v[2]);
#pragma unroll
          for (int e = 3; e < 31; e += 2) m4[q] = fmax3(m4[q], v[e], v[e + 1]);
          m4[q] = fmaxf(m4[q], v[31]);
        }
        return fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
      };
      uint32_t pk[64];
      float tile_sum;
      auto exp_tile = [&]() {
        const float2 n2 = make_float2(-m_used * c, -m_used * c);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 64; ++q) {
          float2 x = ffma2(make_float2(sv[2 * q], sv[2 * q + 1]), c2, n2);
          x.x = ex2_approx(x.x);
          x.y = ex2_approx(x.y);
          if (q & 1)
            acc1 = fadd2(acc1, x);
          else
            acc0 = fadd2(acc0, x);
          pk[q] = pack_bf16x2(x.x, x.y);
        }
        const float2 acc = fadd2(acc0, acc1);
        tile_sum = acc.x + acc.y;
      };
      load_s();
      // m_used only guards the exponentials against overflow (p and l share it, O / l is
      // taken at the end): the exact max of the first key tile, reused by later tiles, and a
      // tile whose row sum leaves [0, 2^64] is redone with the true max
      if (j == 0) {
        const float mt = row_max();
        m_used = (mt == -INFINITY) ? 0.f : mt;
      }
      exp_tile();
      float alpha = 1.f;
      bool grow = false;
      const bool redo = j > 0 && !(tile_sum <= 1.8446744e19f);  // 2^64
      if (__any_sync(0xffffffffu, redo)) {  // rare; S(j) is still in TMEM
        load_s();
        const float m_new = fmaxf(m_used, row_max());
        if (m_new > m_used) {
          grow = true;
          alpha = ex2_approx((m_used - m_new) * c);
          l *= alpha;
          m_used = m_new;
        }
        exp_tile();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSFree));  // S may now be overwritten
      // the previous P.V product must be done before O is rescaled or P overwritten
      if (j > 0 && !warp_all(mbar_wait(bar(kBarODone), (j - 1) & 1, p.timeout_ns))) {
        record_error(p.status, kErrTimeout, kSiteSoftmaxO);
        ok = false;
        break;
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
          for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
          tmem_st32(tO + half * 32, o);
        }
        tmem_wait_st();
      }
      {
        uint32_t lo32[32], hi32[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          lo32[q] = pk[q];
          hi32[q] = pk[32 + q];
        }
        tmem_st32(tP, lo32);
        tmem_st32(tP + 32, hi32);
      }
      l += tile_sum;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull));
    }

    // -------------------------------------------------------------- epilogue: O / l
    const int64_t lse_i = (static_cast<int64_t>(b) * p.H + h) * p.Nq + row;
    if (p.lse != nullptr && row < p.Nq &&
        bounds_ok(lse_i, static_cast<int64_t>(p.B) * p.H * p.Nq, p.status, kSiteLse))
      p.lse[lse_i] = (ok && l > 0.f) ? (m_used * c + log2f(l)) * 0.6931471805599453f : INFINITY;
    if (nt > 0) {
      float o[64];
#pragma unroll
      for (int q = 0; q < 64; ++q) o[q] = 0.f;
      if (ok) {
        // the last P.V (and with it every earlier product, Q's last reader included) is done
        if (!warp_all(mbar_wait(bar(kBarODone), (nt - 1) & 1, p.timeout_ns))) {
          record_error(p.status, kErrTimeout, kSiteEpilogue);
          ok = false;
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
          for (int q = 0; q < 32; ++q) {
            o[q] = __uint_as_float(r0[q]) * inv;
            o[32 + q] = __uint_as_float(r1[q]) * inv;
          }
        }
      }
      if (ok) {
        // O / l in bf16 -> this warp's 32 rows of the Q buffer (128-byte swizzle: 16-byte chunk
        // cidx of row r at chunk cidx ^ (r % 8)) -> one bulk tensor store of the rows below Nq
        const uint32_t sOw = sQ + quarter * (32 * 128);
#pragma unroll
        for (int cidx = 0; cidx < 8; ++cidx) {
          uint4 v;
          v.x = pack_bf16x2(o[cidx * 8 + 0], o[cidx * 8 + 1]);
          v.y = pack_bf16x2(o[cidx * 8 + 2], o[cidx * 8 + 3]);
          v.z = pack_bf16x2(o[cidx * 8 + 4], o[cidx * 8 + 5]);
          v.w = pack_bf16x2(o[cidx * 8 + 6], o[cidx * 8 + 7]);
          st_shared_v4(sOw + lane * 128 + ((cidx ^ (lane & 7)) << 4), v);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && wr0 < p.Nq) {
          tma_store_4d(&tmO, sOw, 0, wr0, h, b);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
      }
    } else if (row < p.Nq && bounds_ok(b, p.B, p.status, kSiteZeroRows) &&
               bounds_ok(h, p.H, p.status, kSiteZeroRows)) {
      // no key to attend: zero rows, stored directly
      uint4* d4 = reinterpret_cast<uint4*>(p.O + static_cast<int64_t>(b) * p.so_b +
                                           static_cast<int64_t>(h) * p.so_h +
                                           static_cast<int64_t>(row) * p.so_n);
#pragma unroll
      for (int q = 0; q < 8; ++q) d4[q] = make_uint4(0u, 0u, 0u, 0u);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_sdpa_bf16(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, const CUtensorMap& tmO, const SdpaArgs& a,
                             const DevCtx& ctx, cudaStream_t s) {
  Params p;
  p.B = a.B;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.mask = a.mask;
  p.window = a.window;
  p.key_len = a.key_len;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.lse = a.lse;
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.so_b = a.so[0];
  p.so_h = a.so[1];
  p.so_n = a.so[2];
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  const bool heavy_first = a.mask == 1;
  const void* fn = heavy_first ? reinterpret_cast<const void*>(sdpa_fwd_bf16_kernel<true>)
                               : reinterpret_cast<const void*>(sdpa_fwd_bf16_kernel<false>);
  cudaError_t e = prepare_kernel(fn, kSmemBytes, nullptr);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + kBQ - 1) / kBQ, a.H, a.B);
  if (heavy_first)
    return launch_pdl(sdpa_fwd_bf16_kernel<true>, grid, dim3(kThreads), kSmemBytes, s, tmQ, tmK,
                      tmV, tmO, p);
  return launch_pdl(sdpa_fwd_bf16_kernel<false>, grid, dim3(kThreads), kSmemBytes, s, tmQ, tmK,
                    tmV, tmO, p);
}

}  // namespace mha
