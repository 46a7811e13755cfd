// gemm2_bf16.cu -- Y[M,N] = act(X[M,K] W[N,K]^T + bias[N]) on pairs of SMs, act = identity
// or ReLU.
//
// The same projection steps as gemm_bf16.cu: the fused Q|K|V projection of every head and the
// output projection W^O ("Attention Is All You Need", lettle.cn translation, 3.2.2 多头注意力;
// "Transformer：抛弃循环与卷积的序列建模", Multi-Head Attention) and the feed-forward network's
// first map with its ReLU ("Attention Is All You Need" on likecs.com, 1.3 按地址的前向反馈网络).
//
// A cluster of two CTAs (a pair) owns a 256 x 256 output tile.  One tcgen05.mma of pair
// granularity (cta_group::2, M = 256, N = 256, K = 16), issued by the even CTA, computes it:
// CTA r of the pair holds rows [128 r, 128 r + 128) of the tile's X slice and rows
// [128 r, 128 r + 128) of its W slice in its own shared memory, and receives output rows
// [128 r, 128 r + 128), all 256 columns, in its own TMEM.  Per 64-wide K slice a CTA stores
// 32 KB instead of the 48 KB a 128 x 256 tile on one SM needs, so a ring of 6 slices fits where
// one of 4 did, and 6 slices cover the ~1200-1700 cycles a slice takes to arrive; a single SM
// with 4 slices left its MMA issuer waiting for data ~45% of the time.
//   warp 0     TMA producer (both CTAs): its X rows and W rows of each K slice; the copies of
//              both CTAs complete the even CTA's full barrier for that ring slot
//   warp 1     TMEM owner in both CTAs (512 columns allocated as a pair: two accumulators of
//              256 columns); MMA issuer in the even CTA, which also releases ring slots and
//              hands accumulators to the epilogues of both CTAs by multicast commits
//   warps 2-5  epilogue (both CTAs, its own 128 rows): tcgen05.ld, bias, ReLU if asked,
//              bf16 round to nearest even, hand the accumulator back to the even CTA, store
//              through swizzled staging boxes with bulk tensor stores
// Every wait is bounded; on a timeout the kernel records MHA_ERR_DEVICE_TIMEOUT, lets its
// copies and MMAs land, frees TMEM and returns.  Every tcgen05 instruction of this kernel has
// pair granularity (ptxas refuses a kernel that mixes it with single-CTA tcgen05 forms).
#include <cuda_bf16.h>

#include <mutex>
#include <vector>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kRows = 128;            // output rows per CTA (the pair: 256)
constexpr int kCols = 256;            // output columns per pair tile
constexpr int kSlice = 64;            // K per ring slot: one 128-byte swizzle row of bf16
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr int kABytes = kRows * kSlice * 2;        // 16 KB: this CTA's X rows
constexpr int kBBytes = (kCols / 2) * kSlice * 2;  // 16 KB: this CTA's W rows
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kOutBoxBytes = 32 * 64 * 2;          // 32 rows x 64 bf16 columns
constexpr int kOutBytes = 4 * 2 * kOutBoxBytes;    // two boxes per epilogue warp
constexpr int kBarBytes = 256;
constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kOutBytes + kBarBytes;
constexpr uint32_t kTmemCols = 2 * kCols;  // two accumulators
constexpr int kErrTimeout = -6;
enum : int {
  kSitePairProducer = 61,
  kSitePairMma = 62,
  kSitePairEpilogue = 63,
  kSitePairBias = 64  // index checks (MHA_DEBUG_BOUNDS builds)
};

// ---- pair-granularity tcgen05 forms
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  // one warp of each CTA of the pair, collectively: both receive the same address
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// One arrival, once every MMA issued so far has completed, on the mbarrier at offset `bar` in
// both CTAs of the pair.
__device__ __forceinline__ void commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}
// 2-D tile into this CTA's shared memory; the bytes complete `bar_cluster`, an mbarrier of
// either CTA of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m,
                                                 uint32_t bar_cluster, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}

template <bool kRelu>
__global__ void __launch_bounds__(kThreads, 1)
    gemm2_bias_bf16_kernel(const __grid_constant__ CUtensorMap tmX,
                           const __grid_constant__ CUtensorMap tmW,
                           const __grid_constant__ CUtensorMap tmY,
                           const __nv_bfloat16* __restrict__ bias, int M, int N, int K,
                           int* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  const uint32_t sOut = smem_u32(smem + kStages * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kOutBytes);
  // [0,ST) full, [ST,2ST) empty, then acc_full[2], acc_empty[2], drain; tmem slot after
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the even CTA, which issues the MMAs
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int pairs = static_cast<int>(gridDim.x >> 1);
  const int num_kb = K / kSlice;
  const int tiles_n = (N + kCols - 1) / kCols;
  const int tiles = tiles_n * ((M + 2 * kRows - 1) / (2 * kRows));

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };
  auto acc_full = [&](int b) { return smem_u32(bars + 2 * kStages + b); };
  auto acc_empty = [&](int b) { return smem_u32(bars + 2 * kStages + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * kStages + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);   // the even CTA's producer arms it for both CTAs' bytes
      mbar_init(empty_bar(s), 1);  // the issuer's commit (multicast to both CTAs)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);   // the issuer's commit (multicast)
      mbar_init(acc_empty(b), 8);  // the epilogue warps of both CTAs (the even CTA's counts)
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before anything signals them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output (X, the bias) is complete from here on

  bool ok = true;
  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    const uint32_t full_even = mapa_shared(full_bar(0), 0);  // the even CTA's full barriers
    int it = 0;
    for (int t = pair; ok && t < tiles; t += pairs) {
      const int m0 = (t / tiles_n) * (2 * kRows) + static_cast<int>(rank) * kRows;
      const int n0 = (t % tiles_n) * kCols + static_cast<int>(rank) * (kCols / 2);
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % kStages;
        // the slot's previous slice has been read by the pair's MMAs
        if (!mbar_wait_backoff(empty_bar(s), ((it / kStages) & 1) ^ 1, timeout_ns)) {
          record_error(status, kErrTimeout, kSitePairProducer);
          ok = false;
          break;
        }
        if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2 * kStageBytes);
        const uint32_t fb = full_even + static_cast<uint32_t>(s) * 8u;
        tma_load_2d_pair(smem_u32(sA + s * kABytes), &tmX, fb, kb * kSlice, m0);
        tma_load_2d_pair(smem_u32(sB + s * kBBytes), &tmW, fb, kb * kSlice, n0);
      }
    }
    // every copy of both CTAs completes the even CTA's full barriers: let them land there
    if (rank == 0)
      for (int i = (it > kStages ? it - kStages : 0); i < it; ++i)
        (void)mbar_wait(full_bar(i % kStages), (i / kStages) & 1, timeout_ns);
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(2 * kRows, kCols, false, false);
    int it = 0, tcount = 0;
    for (int t = pair; ok && t < tiles; t += pairs, ++tcount) {
      const int buf = tcount & 1;
      const uint32_t d = tmem + buf * kCols;
      // both CTAs' epilogues have read this accumulator's previous tile
      if (!mbar_wait_cluster(acc_empty(buf), ((tcount >> 1) & 1) ^ 1, timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % kStages;
        if (!mbar_wait(full_bar(s), (it / kStages) & 1, timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * kABytes);
        const uint32_t b0 = smem_u32(sB + s * kBBytes);
#pragma unroll
        for (int k = 0; k < kSlice / 16; ++k)  // 16 K values: 32 bytes along the swizzled row
          mma_pair(d, smem_desc_sw128(a0 + k * 32, 16, 1024),
                   smem_desc_sw128(b0 + k * 32, 16, 1024), idesc, (kb != 0 || k != 0) ? 1u : 0u);
        commit_pair(empty_bar(s));  // the slot is free in both CTAs once these have read it
      }
      if (!ok) break;
      commit_pair(acc_full(buf));
    }
    if (!ok) record_error(status, kErrTimeout, kSitePairMma);
    commit_pair(drain_bar);
    (void)mbar_wait(drain_bar, 0, timeout_ns);  // no MMA of the pair in flight past this point
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const uint32_t acc_empty_even = mapa_shared(acc_empty(0), 0);
    int tcount = 0;
    int box = 0;  // staging boxes used so far (alternating)
    for (int t = pair; t < tiles; t += pairs, ++tcount) {
      const int buf = tcount & 1;
      const int m0 = (t / tiles_n) * (2 * kRows) + static_cast<int>(rank) * kRows;
      const int n0 = (t % tiles_n) * kCols;
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(buf), (tcount >> 1) & 1, timeout_ns))) {
        record_error(status, kErrTimeout, kSitePairEpilogue);
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + buf * kCols + (static_cast<uint32_t>(quarter * 32) << 16);
      const int wrow0 = m0 + quarter * 32;  // this warp's first output row
#pragma unroll 1
      for (int c = 0; c < kCols / 64; ++c, ++box) {
        uint32_t r[64];
        {
          uint32_t r0[32], r1[32];
          tmem_ld32(tbase + c * 64, r0);
          tmem_ld32(tbase + c * 64 + 32, r1);
          tmem_wait_ld();
          reg_fence(r0);
          reg_fence(r1);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            r[i] = r0[i];
            r[32 + i] = r1[i];
          }
        }
        if (c == kCols / 64 - 1) {  // accumulator read: hand it back to the even CTA's issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty_even + static_cast<uint32_t>(buf) * 8u);
        }
        const int col = n0 + c * 64;
        if (wrow0 >= M || col >= N) continue;  // nothing of this box is inside Y
        float bv[64];
        if (bias != nullptr && span_ok(col, 64, N, status, kSitePairBias)) {
          const uint4* bp = reinterpret_cast<const uint4*>(bias + col);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            uint4 u = __ldg(bp + v);
            const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float2 f = __bfloat1622float2(hv[e]);
              bv[v * 8 + e * 2] = f.x;
              bv[v * 8 + e * 2 + 1] = f.y;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) bv[i] = 0.f;
        }
        // the store issued from this staging box two boxes ago must have read it
        const uint32_t sb = sOut + (quarter * 2 + (box & 1)) * kOutBoxBytes;
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        // row `lane` of the box, 128-byte swizzle: 16-byte chunk q at chunk q ^ (lane % 8)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v0 = __uint_as_float(r[q * 8 + 2 * e]) + bv[q * 8 + 2 * e];
            float v1 = __uint_as_float(r[q * 8 + 2 * e + 1]) + bv[q * 8 + 2 * e + 1];
            if (kRelu) {
              v0 = fmaxf(v0, 0.f);
              v1 = fmaxf(v1, 0.f);
            }
            o[e] = pack_bf16x2(v0, v1);
          }
          st_shared_v4(sb + lane * 128 + ((q ^ (lane & 7)) << 4),
                       make_uint4(o[0], o[1], o[2], o[3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {  // rows past M are not written
          tma_store_2d(&tmY, sb, col, wrow0);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group_read<0>();  // staging stays until every store has read it
  }

  tc_fence_before();
  __syncthreads();
  // the pair's MMAs have completed (the even CTA waited for them) and every copy into either
  // CTA has landed before either CTA frees TMEM or exits
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// CTA pairs that fit on the GPU at once (cached per device)
template <bool kRelu>
int max_pairs(const DevCtx& ctx) {
  static std::mutex mu;
  static std::vector<std::pair<int, int>> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& c : cache)
    if (c.first == dev) return c.second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (ctx.num_sms / 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm2_bias_bf16_kernel<kRelu>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache.push_back({dev, n});
  return n;
}

template <bool kRelu>
cudaError_t launch_relu(const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap& tmY,
                        const void* bias, int M, int N, int K, const DevCtx& ctx,
                        cudaStream_t s) {
  auto kern = gemm2_bias_bf16_kernel<kRelu>;
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), kSmemBytes, nullptr);
  if (e != cudaSuccess) return e;
  const int np = max_pairs<kRelu>(ctx);
  if (np <= 0) return cudaErrorInvalidConfiguration;
  const int64_t tiles =
      static_cast<int64_t>((N + kCols - 1) / kCols) * ((M + 2 * kRows - 1) / (2 * kRows));
  const int pairs = static_cast<int>(tiles < np ? tiles : np);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, tmY, static_cast<const __nv_bfloat16*>(bias),
                            M, N, K, ctx.status, ctx.timeout_ns);
}

}  // namespace

bool gemm2_bf16_supported(int M, int N, int K) {
  return M > 0 && N > 0 && K > 0 && K % kSlice == 0 && N % 64 == 0;
}

cudaError_t launch_gemm2_bf16(const CUtensorMap& tmX, const CUtensorMap& tmW,
                              const CUtensorMap& tmY, bool relu, const void* bias, int M, int N,
                              int K, const DevCtx& ctx, cudaStream_t s) {
  if (relu) return launch_relu<true>(tmX, tmW, tmY, bias, M, N, K, ctx, s);
  return launch_relu<false>(tmX, tmW, tmY, bias, M, N, K, ctx, s);
}

}  // namespace mha
