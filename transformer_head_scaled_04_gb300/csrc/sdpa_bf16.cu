// sdpa_bf16.cu -- fused scaled dot-product attention forward on the sm_103a tensor cores.
//
//   O = softmax(Q K^T / sqrt(d_k)) V per (batch, head), optional causal or key-padding mask
//   ("Attention Is All You Need", lettle.cn translation, 3.2.1 缩放点积注意力;
//    "Transformer：抛弃循环与卷积的序列建模", Scaled Dot-Product Attention, the three uses of
//    attention, and 训练样本 for the causal mask).
//
// The n x n score matrix never leaves the SM.  A block owns 256 query rows (two 128-row
// tiles t = 0, 1) of one (b, h), a work unit, and streams K/V in 128-row tiles.  Blocks are
// persistent: when a block is done with its rows it takes over a block of the same grid that
// has not started yet (launch-cancel request to the hardware launch queue) and runs that
// block's rows with its barriers, rings and TMEM carrying on, so the next rows' Q and first
// K tile land and their first S = Q K^T runs while the current rows' last products and O
// epilogue finish; the launch queue still hands the remaining blocks to whichever SM frees
// first.
//   warp 8     TMA producer: a unit's two Q tiles into one of two Q buffers (units alternate),
//              its first K tile into its own buffer, then K and V through separate 4-stage
//              rings (K one tile ahead; a K slot frees as soon as Q K^T has read it); after
//              a unit's last loads, the launch-cancel request for the next unit
//   warps 9-11 MMA issuers: warp 9 (also TMEM owner) issues S for both tiles, warps 10/11 the
//              P.V of tile 0/1; warps 8-11 form the control warpgroup, which hands most of
//              its registers to the softmax warps:
//                S_t = Q_t K_j^T           tcgen05.mma 128x128x16 x4, fp32 in TMEM
//                O_t += P_t V_j            tcgen05.mma 128x64x16 x8, P from TMEM, V MN-major
//              S_t(j+1) is issued as soon as the softmax warps have read S_t(j) out of TMEM,
//              so the next product runs during this tile's exponentials; the two tiles keep
//              the tensor core busy while either tile's softmax runs.
//   warps 0-7  softmax: warpgroup t owns tile t, one query row per thread (its TMEM lane).
//              One tcgen05.ld round trip brings the whole 128-key S row into registers;
//              mask, running max m and sum l, p = 2^(s*c - m*c) with c = scale*log2(e)
//              (paired fp32 FMA / add), P rounded to bf16 and stored back into TMEM.
//              The reference max m_used is the exact max of the unit's first key tile;
//              later tiles exponentiate against it without taking their own max (any
//              reference gives the exact softmax since p and l share it), and a tile whose
//              row sum overflows 2^64 is redone from TMEM with its true max after rescaling
//              O and l.  The exponentials run before the wait for the previous P.V product,
//              and tile 1 starts its first exponentials only when tile 0 has finished its
//              own, so the two warpgroups' MUFU-heavy phases interleave instead of colliding.
//              At the end of a unit: O / l -> bf16 -> staged in the unit's Q buffer (every S
//              product has read it by then) -> one bulk tensor store per warp, into any
//              strided layout (the head-concat layout [B, Nq, H*64] in the sublayer).
// Whole K/V tiles past the causal diagonal or past key_len[b] are never loaded.  The query
// blocks of one (b, h) are adjacent in launch order, so they run together and share K/V in
// L2.  Every wait is bounded (see device_common.cuh); a timeout records
// MHA_ERR_DEVICE_TIMEOUT and the block stops taking over new units.
#include <cuda_bf16.h>

#include <cmath>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kBQ = 128;       // query rows per tile
constexpr int kBKV = 128;      // keys per K/V tile
constexpr int kHD = 64;        // head dim (d_k = d_v)
constexpr int kKStages = 4;    // K ring depth
constexpr int kVStages = 4;    // V ring depth
constexpr int kThreads = 384;  // 8 softmax warps, then producer, MMA and two idle warps
// register split (setmaxnreg): ptxas gives this 384-thread kernel 168 registers per thread,
// a launch pool of 384 x 168 = 64512; the softmax warpgroups take 216, the control
// warpgroup gives back down to 72 (its unit walk spills below that):
// 256 x 216 + 128 x 72 = 64512.
constexpr int kSoftmaxRegs = 216;
constexpr int kControlRegs = 72;
static_assert(8 * 32 * kSoftmaxRegs + 4 * 32 * kControlRegs <= kThreads * 168,
              "register split exceeds the launch allocation");
constexpr int kTileBytes = kBQ * kHD * 2;  // 16 KB: a 128 x 64 bf16 tile

// Two Q buffers (consecutive units alternate); a unit's buffer also stages its O tiles for
// the bulk stores once every S product of the unit has read it.
constexpr int kOffQ = 0;
// A unit's K(0) has its own buffer; K(i), i >= 1, uses the ring slot of step i - 1, so step
// j's K(j+1) and V(j) both land in one slot, freed together when that slot's previous step is
// done.  Ring steps are counted across units.
constexpr int kOffK0 = kOffQ + 4 * kTileBytes;
constexpr int kOffK = kOffK0 + kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffBar = kOffV + kVStages * kTileBytes;
constexpr int kOffResp = kOffBar + 256;    // two 16-byte launch-cancel responses
constexpr int kSmemBytes = 1024 + kOffResp + 32;
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384) P0 [384,448) P1 [448,512)
// (P holds 128 bf16 per row, two per 32-bit column)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;

constexpr int kErrTimeout = -6;
enum : int {
  kSiteProducer = 21,
  kSiteMma = 22,
  kSiteSoftmaxS = 23,
  kSiteSoftmaxO = 24,
  kSiteEpilogue = 25,
  kSiteKeyLen = 26,    // index checks (MHA_DEBUG_BOUNDS builds)
  kSiteLse = 27,
  kSiteZeroRows = 28
};

// barrier indices
static_assert(kKStages == kVStages, "one K/V-ready barrier per pipeline step");
constexpr int kBarQ = 0;                          // [2] a Q buffer landed
constexpr int kBarQEmpty = kBarQ + 2;             // [2] S products and O staging done with it
constexpr int kBarK0 = kBarQEmpty + 2;            // a unit's K(0) landed
constexpr int kBarK0Empty = kBarK0 + 1;           // the unit's first S products done with K(0)
constexpr int kBarResp = kBarK0Empty + 1;         // [2] a launch-cancel response landed
constexpr int kBarRespEmpty = kBarResp + 2;       // [2] every role has read that response
constexpr int kBarKV = kBarRespEmpty + 2;         // step j: K(j+1) and V(j) landed
constexpr int kBarKVEmpty = kBarKV + kKStages;    // step-j slots free (both issuers done)
constexpr int kBarSFull = kBarKVEmpty + kKStages; // 2
constexpr int kBarSFree = kBarSFull + 2;          // 2
constexpr int kBarPFull = kBarSFree + 2;          // 2
constexpr int kBarODone = kBarPFull + 2;          // 2
constexpr int kBarStagger = kBarODone + 2;
constexpr int kBarDrain = kBarStagger + 1;
constexpr int kNumBars = kBarDrain + 1;

struct Params {
  int B, H, Nq, Nk, mask;
  int nqb;  // 256-row query blocks per (b, h): gridDim.x
  int window;  // kMaskWindow: query i attends keys j with |i - j| <= window
  const int32_t* key_len;
  float scale_log2;  // scale * log2(e)
  float* lse;  // optional [B, H, Nq]: (m_used * c + log2 l) * ln 2
  __nv_bfloat16* O;  // direct stores for units that see no key (zeros)
  int64_t so_b, so_h, so_n;
  int* status;
  uint64_t timeout_ns;
};

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// One work unit, the block with linear index lin: 256 query rows q0.. of head h of batch
// element b, and the key tiles its two query tiles walk (kt0 onwards, n0 and n1 of them; 0
// when the tile has no rows or sees no key).  L: keys a row may see (key padding; else Nk).
struct Unit {
  int b, h, q0, L, kt0, n0, n1;
  __device__ __forceinline__ int nmax() const { return max(n0, n1); }
  __device__ __forceinline__ int ntiles(int t) const { return t == 0 ? n0 : n1; }
};

__device__ __forceinline__ Unit unit_of(const Params& p, int lin) {
  Unit w;
  int qblk;
  // Without a causal mask every block costs the same: the blocks of one (b, h) are adjacent in
  // launch order, so they run together and share K/V in L2.  With it, block k costs ~4k+3 key
  // tiles: all heads' heaviest blocks come first (longest-processing-time order), so no long
  // block starts last.
  if (p.mask == 1) {
    const int bh = p.B * p.H;
    qblk = (p.nqb - 1) - lin / bh;
    w.h = (lin % bh) % p.H;
    w.b = (lin % bh) / p.H;
  } else {
    qblk = p.nqb - 1 - lin % p.nqb;
    w.h = (lin / p.nqb) % p.H;
    w.b = lin / (p.nqb * p.H);
  }
  w.q0 = qblk * (2 * kBQ);
  w.L = p.Nk;
  if (p.mask == 2 && bounds_ok(w.b, p.B, p.status, kSiteKeyLen))
    w.L = min(max(__ldg(p.key_len + w.b), 0), p.Nk);
  // Restricted attention: both query tiles walk the key tiles that the block's whole band
  // [q0 - window, last row + window] touches, starting at key tile kt0; rows mask the keys
  // outside their own band, so a tile can be fully masked for one of the two query tiles.
  w.kt0 = 0;
  int n_band = 0;
  if (p.mask == kMaskWindow) {
    const int last = min(w.q0 + 2 * kBQ, p.Nq) - 1;
    w.kt0 = max(w.q0 - p.window, 0) / kBKV;
    n_band = min(last + p.window, p.Nk - 1) / kBKV - w.kt0 + 1;
  }
  int n[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int row0 = w.q0 + t * kBQ;
    if (row0 >= p.Nq)
      n[t] = 0;
    else if (p.mask == 1)
      n[t] = min(p.Nq - 1, row0 + kBQ - 1) / kBKV + 1;
    else if (p.mask == kMaskWindow)
      n[t] = n_band;
    else
      n[t] = (w.L + kBKV - 1) / kBKV;
  }
  w.n0 = n[0];
  w.n1 = n[1];
  return w;
}

// kBandMask selects how a diagonal / edge tile excludes keys (the launcher takes it for causal,
// key-padding and restricted attention): one compare and select per key against per-row
// bounds, one-sided where the warp's rows allow it.  Unmasked attention keeps a per-key
// position test: its only masked tile is a ragged last one, and any other form there changed
// how the compiler scheduled the unmasked exponential loop (3% slower in A/B).
template <bool kBandMask>
__global__ void __launch_bounds__(kThreads, 1)
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
  const uint32_t sK0 = smem_u32(smem + kOffK0);
  const uint32_t sK = smem_u32(smem + kOffK);
  const uint32_t sV = smem_u32(smem + kOffV);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sResp = smem_u32(smem + kOffResp);
  const int lin0 = static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarQ + i), 1);
      mbar_init(bar(kBarQEmpty + i), 1 + 8);  // the S issuer's commit, the 8 softmax warps
      mbar_init(bar(kBarResp + i), 1);
      mbar_init(bar(kBarRespEmpty + i), 3 + 8);  // three MMA issuers, eight softmax warps
    }
    mbar_init(bar(kBarK0), 1);
    mbar_init(bar(kBarK0Empty), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(kBarKV + s), 1);
      mbar_init(bar(kBarKVEmpty + s), 3);  // the three MMA issuers
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarSFree + t), 4);  // one arrival per softmax warp
      mbar_init(bar(kBarPFull + t), kBQ);
      mbar_init(bar(kBarODone + t), 1);
    }
    mbar_init(bar(kBarDrain), 3);
    mbar_init(bar(kBarStagger), 4);
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
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output (Q, K, V) is complete from here on
  // The i-th unit of this CTA is followed by the unit named in launch-cancel response i (slot
  // i % 2), which the producer requests once it has issued the i-th unit's loads.  Every role
  // reads every response, so all roles walk the same units; -1 ends the walk.
  auto next_unit = [&](int i, bool release, bool& ok) -> int {
    if (!mbar_wait(bar(kBarResp + (i & 1)), (i >> 1) & 1, p.timeout_ns)) {
      ok = false;
      return -1;
    }
    const int nxt = launch_cancel_result(sResp + 16 * (i & 1));
    if (release) mbar_arrive(bar(kBarRespEmpty + (i & 1)));
    return nxt;
  };

  if (warp >= 8) regs_dec<kControlRegs>();  // first thing: the softmax increase waits on it
  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      bool ok = true;
      int it = 0;         // units with work so far: Q buffer it & 1, K(0) phase it & 1
      int g = 0;          // ring steps so far
      int waiting = -1;   // a response requested and not yet awaited
      for (int i = 0, lin = lin0; ok && lin >= 0; ++i) {
        const Unit w = unit_of(p, lin);
        const int nmax = w.nmax();
        if (nmax > 0) {
          const int qb = it & 1;
          // the Q buffer of two units ago (S products and O staging) and the last K(0)
          if (!mbar_wait_backoff(bar(kBarQEmpty + qb), ((it >> 1) & 1) ^ 1, p.timeout_ns) ||
              !mbar_wait_backoff(bar(kBarK0Empty), (it & 1) ^ 1, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t qbytes = (w.n0 > 0 ? kTileBytes : 0) + (w.n1 > 0 ? kTileBytes : 0);
          mbar_arrive_expect_tx(bar(kBarQ + qb), qbytes);
          for (int t = 0; t < 2; ++t)
            if (w.ntiles(t) > 0)
              tma_load_4d(sQ + (2 * qb + t) * kTileBytes, &tmQ, bar(kBarQ + qb), 0,
                          w.q0 + t * kBQ, w.h, w.b);
          mbar_arrive_expect_tx(bar(kBarK0), kTileBytes);
          tma_load_4d(sK0, &tmK, bar(kBarK0), 0, w.kt0 * kBKV, w.h, w.b);
          ++it;
          // K runs one tile ahead of V: step j brings K(j+1) and V(j), both onto one barrier,
          // since S(j+1) = Q K(j+1)^T is issued right before O += P(j) V(j).
          for (int j = 0; j < nmax; ++j, ++g) {
            const bool next_k = j + 1 < nmax;
            const int sl = g % kKStages;
            // the slot last held step g - stages' K and V: both released together after it
            if (!mbar_wait_backoff(bar(kBarKVEmpty + sl), ((g / kKStages) & 1) ^ 1,
                                   p.timeout_ns)) {
              ok = false;
              break;
            }
            const uint32_t kv = bar(kBarKV + sl);
            mbar_arrive_expect_tx(kv, next_k ? 2 * kTileBytes : kTileBytes);
            if (next_k)
              tma_load_4d(sK + sl * kTileBytes, &tmK, kv, 0, (w.kt0 + j + 1) * kBKV, w.h, w.b);
            tma_load_4d(sV + sl * kTileBytes, &tmV, kv, 0, (w.kt0 + j) * kBKV, w.h, w.b);
          }
          if (!ok) break;
        }
        // the next unit: requested as late as the loads allow, so the blocks still waiting
        // in the launch queue go to whichever SM frees first
        if (!mbar_wait_backoff(bar(kBarRespEmpty + (i & 1)), ((i >> 1) & 1) ^ 1,
                               p.timeout_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(kBarResp + (i & 1)), 16);
        launch_cancel_request(sResp + 16 * (i & 1), bar(kBarResp + (i & 1)));
        waiting = i;
        lin = next_unit(i, false, ok);
        if (ok) waiting = -1;
      }
      if (!ok) record_error(p.status, kErrTimeout, kSiteProducer);
      // nothing this thread started may land after the CTA exits: the last response, the last
      // Q buffers and K(0), the last ring steps
      if (waiting >= 0)
        (void)mbar_wait(bar(kBarResp + (waiting & 1)), (waiting >> 1) & 1, p.timeout_ns);
      for (int q = (it > 2 ? it - 2 : 0); q < it; ++q)
        (void)mbar_wait(bar(kBarQ + (q & 1)), (q >> 1) & 1, p.timeout_ns);
      if (it > 0) (void)mbar_wait(bar(kBarK0), (it - 1) & 1, p.timeout_ns);
      for (int q = (g > kKStages ? g - kKStages : 0); q < g; ++q)
        (void)mbar_wait(bar(kBarKV + q % kKStages), (q / kKStages) & 1, p.timeout_ns);
    }
  } else if (warp >= 9) {
    // ------------------------------------------------------------------ MMA issuers
    // A thread spends tens of cycles per tcgen05.mma and per barrier test, so the work is
    // spread over three issuers: warp 9 issues both tiles' S = Q K^T products, warps 10 and
    // 11 the O += P V products of tile 0 and tile 1.  Each releases the step's K/V slots.
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kBQ, kBKV, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(kBQ, kHD, false, true);
      // Descriptor start addresses are address >> 4 in the low 14 bits and every operand
      // lies below 256 KB of shared memory, so moving an operand by `off` bytes adds off >> 4.
      const uint64_t dQ0 = smem_desc_sw128(sQ, 1024, 1024);
      const uint64_t dKfirst = smem_desc_sw128(sK0, 1024, 1024);
      const uint64_t dK0 = smem_desc_sw128(sK, 1024, 1024);
      const uint64_t dV0 = smem_desc_sw128(sV, 1024, 1024);
      bool ok = true;
      int g = 0;   // ring steps so far
      int it = 0;  // units with work so far
      int cs0 = 0, cs1 = 0;  // S products issued so far per query tile (warp 9)
      int cp = 0;            // P.V products issued so far (warps 10, 11)
      // S_t = Q_t K^T once softmax t has read the previous S_t out of TMEM
      auto issue_s = [&](int t, uint64_t aq, uint64_t bk) -> bool {
        const int cs = t == 0 ? cs0 : cs1;
        if (cs > 0 && !mbar_wait(bar(kBarSFree + t), (cs - 1) & 1, p.timeout_ns)) return false;
        tc_fence_after();
        aq += static_cast<uint64_t>((t * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk)  // K steps of 16 = 32 B inside the swizzle row
          mma_bf16_ss(tmem + t * kBKV, aq + kk * 2, bk + kk * 2, idS, kk > 0 ? 1u : 0u);
        mma_commit(bar(kBarSFull + t));
        if (t == 0)
          ++cs0;
        else
          ++cs1;
        return true;
      };
      for (int i = 0, lin = lin0; ok && lin >= 0; ++i) {
        const Unit w = unit_of(p, lin);
        const int nmax = w.nmax();
        if (nmax > 0 && warp == 9) {
          const int qb = it & 1;
          const uint64_t aq = dQ0 + static_cast<uint64_t>((2 * qb * kTileBytes) >> 4);
          if (!mbar_wait(bar(kBarQ + qb), (it >> 1) & 1, p.timeout_ns) ||
              !mbar_wait(bar(kBarK0), it & 1, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int t = 0; ok && t < 2; ++t)
            if (w.ntiles(t) > 0) ok = issue_s(t, aq, dKfirst);
          if (!ok) break;
          mma_commit(bar(kBarK0Empty));  // done with this unit's K(0)
          // Every issuer waits for step j's K/V barrier before it releases step j, even when
          // it has nothing to issue: an issuer that ran a full ring ahead would otherwise put
          // its release into an earlier phase of the same barrier.
          for (int j = 0; j < nmax; ++j, ++g) {
            const int sl = g % kKStages;
            if (!mbar_wait(bar(kBarKV + sl), (g / kKStages) & 1, p.timeout_ns)) {
              ok = false;
              break;
            }
            const uint64_t bk = dK0 + static_cast<uint64_t>((sl * kTileBytes) >> 4);
            for (int t = 0; ok && t < 2; ++t)
              if (j + 1 < w.ntiles(t)) ok = issue_s(t, aq, bk);
            if (!ok) break;
            mma_commit(bar(kBarKVEmpty + sl));  // done with K(j+1)
          }
          if (!ok) break;
          mma_commit(bar(kBarQEmpty + qb));  // every S product of this unit is issued
        } else if (nmax > 0) {
          const int t = warp - 10;
          const int nt = w.ntiles(t);
          const uint32_t dO = tmem + kColO + t * kHD;
          const uint32_t aP = tmem + kColP + t * 64;
          for (int j = 0; j < nmax; ++j, ++g) {
            const int sl = g % kKStages;
            if (!mbar_wait(bar(kBarKV + sl), (g / kKStages) & 1, p.timeout_ns)) {
              ok = false;
              break;
            }
            // O_t += P_t(j) V_j once softmax t has written P_t(j); a unit's first product
            // overwrites O_t, which softmax t has read out for the previous unit by then
            if (j < nt) {
              if (!mbar_wait(bar(kBarPFull + t), cp & 1, p.timeout_ns)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t bv = dV0 + static_cast<uint64_t>((sl * kTileBytes) >> 4);
#pragma unroll
              for (int kk = 0; kk < kBKV / 16; ++kk)  // 16 keys = 8 TMEM columns of P, 16 V rows
                mma_bf16_ts(dO, aP + kk * 8, bv + kk * ((16 * 128) >> 4), idO,
                            (j > 0 || kk > 0) ? 1u : 0u);
              mma_commit(bar(kBarODone + t));
              ++cp;
            }
            mma_commit(bar(kBarKVEmpty + sl));  // done with V(j)
          }
          if (!ok) break;
        }
        if (nmax > 0) ++it;
        lin = next_unit(i, true, ok);
      }
      if (!ok) record_error(p.status, kErrTimeout, kSiteMma);
      mma_commit(bar(kBarDrain));
      (void)mbar_wait(bar(kBarDrain), 0, p.timeout_ns);  // no MMA in flight past this point
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------------ softmax warps
    regs_inc<kSoftmaxRegs>();
    const int t = warp >> 2;
    const int quarter = warp & 3;
    const int r_local = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + t * kBKV + lane_off;
    const uint32_t tO = tmem + kColO + t * kHD + lane_off;
    const uint32_t tP = tmem + kColP + t * 64 + lane_off;
    const float c = p.scale_log2;
    const float2 c2 = make_float2(c, c);
    bool ok = true;
    int k = 0;   // S tiles of this query tile consumed so far (all units)
    int it = 0;  // units with work so far (their Q buffer: it & 1)

    for (int i = 0, lin = lin0; lin >= 0; ++i) {
      const Unit w = unit_of(p, lin);
      const int row = w.q0 + t * kBQ + r_local;
      const int nt = w.ntiles(t);
      const int kt0 = w.kt0;
      // allowed keys: first <= j <= limit
      const int limit = (p.mask == 1)             ? row
                        : (p.mask == kMaskWindow) ? min(row + p.window, p.Nk - 1)
                                                  : w.L - 1;
      const int first = (p.mask == kMaskWindow) ? row - p.window : 0;
      // Both bounds grow with the row, so the warp's smallest limit is its first row's and its
      // largest first key its last row's: whether any row of the warp masks at either end of
      // a key tile is known without a vote.
      const int wr0 = w.q0 + t * kBQ + quarter * 32;
      const int lim_min = (p.mask == 1)             ? wr0
                          : (p.mask == kMaskWindow) ? min(wr0 + p.window, p.Nk - 1)
                                                    : w.L - 1;
      const int first_max = (p.mask == kMaskWindow) ? wr0 + 31 - p.window : 0;
      float m_used = -INFINITY;
      float l = 0.f;

      for (int j = 0; j < nt; ++j) {
        const int kk = k + j;
        if (!warp_all(mbar_wait(bar(kBarSFull + t), kk & 1, p.timeout_ns))) {
          record_error(p.status, kErrTimeout, kSiteSoftmaxS);
          ok = false;
          break;
        }
        tc_fence_after();
        const int col0 = (kt0 + j) * kBKV;
        // diagonal / edge tile: keys q of the tile with q > hi or q < lo are excluded; some row
        // of the warp has keys past its limit (mask_hi) or before its band (mask_lo)
        const int hi = limit - col0;
        const int lo = first - col0;
        const bool mask_hi = lim_min - col0 < kBKV - 1;
        const bool mask_lo = first_max - col0 > 0;
        const bool masked = col0 + kBKV - 1 > limit || col0 < first;  // this row
        float sv[128];
        // the whole S row of this tile: 128 fp32 in registers, one TMEM round trip
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
          // Excluded keys get -inf (p = 0).  Band form: one compare against a per-row bound
          // and one select per key; the warp takes the one-sided form when none of its rows
          // has the other end inside the tile (causal and key-padding tiles, and the edge tiles
          // of restricted attention whose radius spans whole tiles).  The per-key position
          // test costs ~9 cycles per key there.
          if constexpr (kBandMask) {
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
          } else if (masked) {
#pragma unroll
            for (int q = 0; q < 128; ++q)
              if (col0 + q > limit || col0 + q < first) sv[q] = -INFINITY;
          }
        };
        auto row_max = [&]() {
          float m4[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // four independent chains over 32-key blocks
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
        // p = 2^(s*c - m_used*c) two at a time, the tile's row sum in two independent pairs
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
        // The running max m_used only guards the exponentials against overflow: every p and
        // l use the same m_used and O / l is taken at the end, so any m_used gives the exact
        // softmax as long as nothing overflows.  It is the exact max of the unit's first
        // tile; later tiles reuse it, and a tile whose row sum leaves [0, 2^64] (overflow,
        // inf or nan) is redone with the true max after rescaling O and l.
        if (j == 0) {
          const float mt = row_max();
          m_used = (mt == -INFINITY) ? 0.f : mt;
        }
        // the CTA's first tile: tile 1 starts its exponentials when tile 0 has done its own,
        // so the two warpgroups' MUFU-heavy phases interleave instead of colliding
        if (t == 1 && kk == 0 && !warp_all(mbar_wait(bar(kBarStagger), 0, p.timeout_ns))) {
          record_error(p.status, kErrTimeout, kSiteSoftmaxO);
          ok = false;
          break;
        }
        exp_tile();
        float alpha = 1.f;
        bool grow = false;
        const bool redo = j > 0 && !(tile_sum <= 1.8446744e19f);  // 2^64
        if (__any_sync(0xffffffffu, redo)) {  // rare; S_t(j) is still in TMEM
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
        if (lane == 0) mbar_arrive(bar(kBarSFree + t));  // S_t may now be overwritten
        if (t == 0 && kk == 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarStagger));
        }
        // the previous P.V product must be done before O is rescaled or P overwritten (a
        // unit's first tile: the previous unit's last product was awaited by its epilogue)
        if (j > 0 && !warp_all(mbar_wait(bar(kBarODone + t), (kk - 1) & 1, p.timeout_ns))) {
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
        // P row -> TMEM (bf16 pairs, keys 2i and 2i+1 in column i), the A operand of P.V
        {
          uint32_t lo[32], hi[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            lo[q] = pk[q];
            hi[q] = pk[32 + q];
          }
          tmem_st32(tP, lo);
          tmem_st32(tP + 32, hi);
        }
        l += tile_sum;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + t));
      }

      // -------------------------------------------------------------- epilogue: O / l
      float o[64];
#pragma unroll
      for (int q = 0; q < 64; ++q) o[q] = 0.f;
      if (ok && nt > 0) {
        k += nt;
        if (!warp_all(mbar_wait(bar(kBarODone + t), (k - 1) & 1, p.timeout_ns))) {
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
      const int64_t lse_i = (static_cast<int64_t>(w.b) * p.H + w.h) * p.Nq + row;
      if (p.lse != nullptr && row < p.Nq &&
          bounds_ok(lse_i, static_cast<int64_t>(p.B) * p.H * p.Nq, p.status, kSiteLse))
        p.lse[lse_i] =
            (ok && l > 0.f) ? (m_used * c + log2f(l)) * 0.6931471805599453f : INFINITY;
      const int wrow0 = w.q0 + t * kBQ + quarter * 32;
      if (w.nmax() > 0 && w.q0 + t * kBQ >= p.Nq) {
        // This query tile has no rows (a sequence of at most 128 queries, or the last block of
        // a ragged one): nothing to store.  Its warps wait on nothing else of the unit, so they
        // could run two units ahead of the other tile and release the Q buffer into its
        // previous use, which the other tile may still be staging O in.  Waiting for this
        // unit's Q to land first puts the release into this unit's use: the producer loads
        // that Q only once the buffer's previous use has been released.
        const int qb = it & 1;
        if (lane == 0) {
          if (!mbar_wait(bar(kBarQ + qb), (it >> 1) & 1, p.timeout_ns)) {
            record_error(p.status, kErrTimeout, kSiteEpilogue);
            ok = false;
          }
          mbar_arrive(bar(kBarQEmpty + qb));
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        ++it;
      } else if (w.nmax() > 0) {
        // O / l in bf16 -> this warp's 32 rows of the unit's Q buffer, which every S product
        // of the unit has read by now (128-byte swizzle: 16-byte chunk c of row r at chunk
        // c ^ (r % 8), conflict-free) -> one bulk tensor store per warp, which writes only the
        // rows below Nq; the buffer is released to the producer once the copy has read it
        const int qb = it & 1;
        const uint32_t sOw = sQ + (2 * qb + t) * kTileBytes + quarter * (32 * 128);
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
        if (lane == 0) {
          if (wrow0 < p.Nq) {
            tma_store_4d(&tmO, sOw, 0, wrow0, w.h, w.b);
            bulk_commit_group();
            bulk_wait_group_read0();
          }
          mbar_arrive(bar(kBarQEmpty + qb));
        }
        ++it;
      } else if (row < p.Nq && bounds_ok(w.b, p.B, p.status, kSiteZeroRows) &&
                 bounds_ok(w.h, p.H, p.status, kSiteZeroRows)) {
        // a unit that sees no key: zero rows, stored directly
        uint4* d4 = reinterpret_cast<uint4*>(p.O + static_cast<int64_t>(w.b) * p.so_b +
                                             static_cast<int64_t>(w.h) * p.so_h +
                                             static_cast<int64_t>(row) * p.so_n);
#pragma unroll
        for (int q = 0; q < 8; ++q) d4[q] = make_uint4(0u, 0u, 0u, 0u);
      }
      // the next unit (lane 0 waits for the response and releases it for the warp)
      if (!ok) break;
      int nxt = -1;
      bool okr = true;
      if (lane == 0) nxt = next_unit(i, true, okr);
      nxt = __shfl_sync(0xffffffffu, nxt, 0);
      if (!__shfl_sync(0xffffffffu, okr ? 1 : 0, 0)) {
        record_error(p.status, kErrTimeout, kSiteSoftmaxS);
        break;
      }
      lin = nxt;
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
  const double c = static_cast<double>(a.scale) * 1.4426950408889634;  // log2(e)
  p.scale_log2 = static_cast<float>(c);
  p.lse = a.lse;
  p.nqb = (a.Nq + 2 * kBQ - 1) / (2 * kBQ);
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.so_b = a.so[0];
  p.so_h = a.so[1];
  p.so_n = a.so[2];
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  const bool band = a.mask != 0;
  const void* fn = band ? reinterpret_cast<const void*>(sdpa_fwd_bf16_kernel<true>)
                        : reinterpret_cast<const void*>(sdpa_fwd_bf16_kernel<false>);
  int regs = 0;
  cudaError_t e = prepare_kernel(fn, kSmemBytes, &regs);
  if (e != cudaSuccess) return e;
  // The setmaxnreg split must fit in what the block is launched with, or the increase would
  // wait forever: refuse to launch if the compiled register count is too small for it.
  if (regs * kThreads < 8 * 32 * kSoftmaxRegs + 4 * 32 * kControlRegs)
    return cudaErrorInvalidConfiguration;
  dim3 grid((a.Nq + 2 * kBQ - 1) / (2 * kBQ), a.H, a.B);
  if (band)
    return launch_pdl(sdpa_fwd_bf16_kernel<true>, grid, dim3(kThreads), kSmemBytes, s, tmQ, tmK,
                      tmV, tmO, p);
  return launch_pdl(sdpa_fwd_bf16_kernel<false>, grid, dim3(kThreads), kSmemBytes, s, tmQ, tmK, tmV,
                    tmO, p);
}

}  // namespace mha
