// gemm_bf16.cu -- Y[M,N] = act(X[M,K] W[N,K]^T + bias[N]) on the sm_103a tensor cores,
// act = identity or ReLU.
//
// These are the projection steps of the sublayers: the fused Q|K|V projection of every head
// (N = 3*d_model) and the output projection W^O ("Attention Is All You Need", lettle.cn
// translation, 3.2.2 多头注意力; "Transformer：抛弃循环与卷积的序列建模", Multi-Head
// Attention), and the two linear maps of the position-wise feed-forward network, the first
// followed by ReLU ("Attention Is All You Need" on likecs.com, 1.3 按地址的前向反馈网络;
// "Transformer：抛弃循环与卷积的序列建模", FFN).
//
// Persistent kernel: one CTA per SM walks the 128 x BN output tiles (N fastest, so the CTAs
// running together share the same X rows in L2).
//   warp 0     TMA producer: X and W K-slices (64 wide, 128-byte swizzle) into a STAGES ring
//              that runs on across tile boundaries
//   warp 1     TMEM owner + MMA issuer: tcgen05.mma kind::f16 128xBNx16 into one of two TMEM
//              accumulators, so the epilogue of tile i overlaps the MMAs of tile i+1
//   warps 2-5  epilogue: tcgen05.ld the accumulator (one TMEM lane quarter per warp), add
//              bias, ReLU if asked, round to bf16 (nearest even), hand the accumulator back;
//              each warp writes its 32 rows 64 columns at a time into one of two swizzled
//              shared-memory staging boxes and issues one bulk tensor store per box.
// Split-K (kAcc, for the weight-gradient GEMMs whose K is the token count and whose few
// output tiles would leave SMs idle): the work units are (K slice, tile) pairs, each unit's
// fp32 partial goes through the same staging boxes as 32 x 32 fp32 boxes and is added into a
// zeroed fp32 [M, N] buffer by bulk tensor reductions; a separate launch rounds it to bf16.
// MN-major operands (kMN, the weight gradients dW = dOut^T In straight from the row-major
// activations, no transposed copies): X and W are then stored [K, M] and [K, N]; each stage
// loads 64 x 64 boxes (64 K rows of 64 M or N columns, 128-byte swizzle) side by side, and the
// MMA reads them MN-major (the 64-column chunks 8 KB apart as the leading-dimension step); K
// need not be a multiple of 64 (rows past K load as zeros).
// Every wait is bounded; on a timeout the kernel records MHA_ERR_DEVICE_TIMEOUT, lets its
// in-flight copies and MMAs land, frees TMEM and returns.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "launchers.h"

namespace mha {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;  // one 128-byte swizzle row of bf16
constexpr int kThreads = 192;
constexpr int kErrTimeout = -6;

enum : int {
  kSiteGemmProducer = 11,
  kSiteGemmMma = 12,
  kSiteGemmEpilogue = 13,
  kSiteGemmBias = 14,      // index checks (MHA_DEBUG_BOUNDS builds)
  kSiteGemmResidual = 15
};

template <int BN>
struct GemmShape {
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kOutBoxBytes = 32 * 64 * 2;        // 32 rows x 64 bf16 columns
  static constexpr int kOutBytes = 4 * 2 * kOutBoxBytes;  // two boxes per epilogue warp
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kOutBytes + kBarBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators; a power of two
};

// A second problem with the same K that the same launch works through after the first one's
// tiles (kTwo: the query and the key|value projections of cross-attention)
struct GemmSecond {
  CUtensorMap tmX, tmW, tmY;
  const __nv_bfloat16* bias;
  int M, N;
};

template <int BN, bool kRelu, bool kAcc, bool kMN, bool kTwo = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bias_bf16_kernel(const __grid_constant__ CUtensorMap tmX,
                          const __grid_constant__ CUtensorMap tmW,
                          const __grid_constant__ CUtensorMap tmY,
                          const __nv_bfloat16* __restrict__ bias, __nv_bfloat16* __restrict__ Y,
                          int M, int N, int K, int64_t ldy, int* status, uint64_t timeout_ns,
                          const __nv_bfloat16* __restrict__ R, int ksplit,
                          const __grid_constant__ GemmSecond g2) {
  using S = GemmShape<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S::kStages * S::kABytes;
  const uint32_t sOut = smem_u32(smem + S::kStages * S::kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kStages * S::kStageBytes + S::kOutBytes);
  // [0,ST) full, [ST,2ST) empty, then acc_full[2], acc_empty[2], drain; tmem slot after
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S::kStages + 5);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_kb = kMN ? (K + kBK - 1) / kBK : K / kBK;
  const int tiles_n = (N + BN - 1) / BN;
  const int tiles1 = tiles_n * ((M + kBM - 1) / kBM);
  int tiles_n2 = 0, tiles2 = 0;
  if constexpr (kTwo) {  // the second problem's tiles follow the first's (ksplit is 1)
    tiles_n2 = (g2.N + BN - 1) / BN;
    tiles2 = tiles_n2 * ((g2.M + kBM - 1) / kBM);
  }
  const int tiles = tiles1 + tiles2;
  // tile -> its problem (second), first row and column
  auto tile_pos = [&](int tile, bool& second, int& m0, int& n0) {
    second = kTwo && tile >= tiles1;
    if (second) {
      const int t2 = tile - tiles1;
      m0 = (t2 / tiles_n2) * kBM;
      n0 = (t2 % tiles_n2) * BN;
    } else {
      m0 = (tile / tiles_n) * kBM;
      n0 = (tile % tiles_n) * BN;
    }
  };
  // work unit u: tile u % tiles, K slice u / tiles (units running together share K slices)
  const int units = tiles * ksplit;
  auto kb_begin = [&](int u) { return (u / tiles) * num_kb / ksplit; };
  auto kb_end = [&](int u) { return (u / tiles + 1) * num_kb / ksplit; };

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + S::kStages + s); };
  auto acc_full = [&](int b) { return smem_u32(bars + 2 * S::kStages + b); };
  auto acc_empty = [&](int b) { return smem_u32(bars + 2 * S::kStages + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * S::kStages + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();  // the previous kernel's output (X, the bias, R) is complete from here on

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    int it = 0;
    bool ok = true;
    if constexpr (kTwo) {
      prefetch_tmap(&g2.tmX);
      prefetch_tmap(&g2.tmW);
    }
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      bool second;
      int m0, n0;
      tile_pos(u % tiles, second, m0, n0);
      const CUtensorMap* mx = second ? &g2.tmX : &tmX;
      const CUtensorMap* mw = second ? &g2.tmW : &tmW;
      for (int kb = kb_begin(u), kb1 = kb_end(u); kb < kb1; ++kb, ++it) {
        const int s = it % S::kStages;
        if (!mbar_wait_backoff(empty_bar(s), ((it / S::kStages) & 1) ^ 1, timeout_ns)) {
          record_error(status, kErrTimeout, kSiteGemmProducer);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(full_bar(s), S::kStageBytes);
        if constexpr (kMN) {
#pragma unroll
          for (int c = 0; c < kBM / 64; ++c)
            tma_load_2d(smem_u32(sA + s * S::kABytes + c * 8192), &tmX, full_bar(s), m0 + c * 64,
                        kb * kBK);
#pragma unroll
          for (int c = 0; c < BN / 64; ++c)
            tma_load_2d(smem_u32(sB + s * S::kBBytes + c * 8192), &tmW, full_bar(s), n0 + c * 64,
                        kb * kBK);
        } else {
          tma_load_2d(smem_u32(sA + s * S::kABytes), mx, full_bar(s), kb * kBK, m0);
          tma_load_2d(smem_u32(sB + s * S::kBBytes), mw, full_bar(s), kb * kBK, n0);
        }
      }
    }
    // let every copy this thread started land before the CTA can exit
    for (int i = (it > S::kStages ? it - S::kStages : 0); i < it; ++i)
      (void)mbar_wait(full_bar(i % S::kStages), (i / S::kStages) & 1, timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, kMN, kMN);
    int it = 0, tcount = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++tcount) {
      const int buf = tcount & 1;
      const uint32_t d = tmem + buf * BN;
      const int kb0 = kb_begin(u);
      if (!mbar_wait(acc_empty(buf), ((tcount >> 1) & 1) ^ 1, timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = kb0, kb1 = kb_end(u); kb < kb1; ++kb, ++it) {
        const int s = it % S::kStages;
        if (!mbar_wait(full_bar(s), (it / S::kStages) & 1, timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * S::kABytes);
        const uint32_t b0 = smem_u32(sB + s * S::kBBytes);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          // K-major: 16 K values are 32 bytes along the swizzled row; MN-major: 16 K rows
          const uint64_t ad = kMN ? smem_desc_sw128(a0 + k * 2048, 8192, 1024)
                                  : smem_desc_sw128(a0 + k * 32, 16, 1024);
          const uint64_t bd = kMN ? smem_desc_sw128(b0 + k * 2048, 8192, 1024)
                                  : smem_desc_sw128(b0 + k * 32, 16, 1024);
          mma_bf16_ss(d, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
        }
        mma_commit(empty_bar(s));
      }
      if (!ok) break;
      mma_commit(acc_full(buf));
    }
    if (!ok) record_error(status, kErrTimeout, kSiteGemmMma);
    mma_commit(drain_bar);
    (void)mbar_wait(drain_bar, 0, timeout_ns);  // no MMA in flight past this point
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    int tcount = 0;
    int box = 0;  // staging boxes used so far (alternating)
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++tcount) {
      const int buf = tcount & 1;
      bool second;
      int m0, n0;
      tile_pos(u % tiles, second, m0, n0);
      const int Mt = second ? g2.M : M;  // this tile's problem
      const int Nt = second ? g2.N : N;
      const CUtensorMap* my = second ? &g2.tmY : &tmY;
      const __nv_bfloat16* bias_t = second ? g2.bias : bias;
      const int row = m0 + quarter * 32 + lane;
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(buf), (tcount >> 1) & 1, timeout_ns))) {
        record_error(status, kErrTimeout, kSiteGemmEpilogue);
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + buf * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      const int wrow0 = m0 + quarter * 32;  // this warp's first output row
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c, ++box) {
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
        if (c == BN / 64 - 1) {  // accumulator read: hand it back to the MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty(buf));
        }
        const int col = n0 + c * 64;
        if (wrow0 >= Mt || col >= Nt) continue;  // nothing of this box is inside Y
        if constexpr (kAcc) {
          // two 32 x 32 fp32 boxes (128-byte rows, swizzled) added into the fp32 buffer
#pragma unroll
          for (int hh = 0; hh < 2; ++hh, ++box) {
            const uint32_t sb = sOut + (quarter * 2 + (box & 1)) * S::kOutBoxBytes;
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_shared_v4(sb + lane * 128 + ((q ^ (lane & 7)) << 4),
                           make_uint4(r[hh * 32 + q * 4], r[hh * 32 + q * 4 + 1],
                                      r[hh * 32 + q * 4 + 2], r[hh * 32 + q * 4 + 3]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&tmY, sb, col + hh * 32, wrow0);
              bulk_commit_group();
            }
          }
          --box;  // the loop header counts one box per chunk
          continue;
        }
        float bv[64];
        if (bias_t != nullptr && span_ok(col, 64, Nt, status, kSiteGemmBias)) {
          const uint4* bp = reinterpret_cast<const uint4*>(bias_t + col);
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
        if (R != nullptr && row < M && span_ok(col, 64, N, status, kSiteGemmResidual)) {
          // a residual matrix with Y's layout joins the bias
          const uint4* rp = reinterpret_cast<const uint4*>(R + static_cast<int64_t>(row) * ldy + col);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            uint4 u = rp[v];
            const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float2 f = __bfloat1622float2(hv[e]);
              bv[v * 8 + e * 2] += f.x;
              bv[v * 8 + e * 2 + 1] += f.y;
            }
          }
        }
        // the store issued from this staging box two boxes ago must have read it
        const uint32_t sb = sOut + (quarter * 2 + (box & 1)) * S::kOutBoxBytes;
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
          st_shared_v4(sb + lane * 128 + ((q ^ (lane & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {  // rows past M are not written
          tma_store_2d(my, sb, col, wrow0);
          bulk_commit_group();
        }
      }
    }
    // staging stays until every store has read it; reductions have also landed
    if (lane == 0) {
      if (kAcc)
        bulk_wait_group0();
      else
        bulk_wait_group_read<0>();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::kTmemCols);
  }
}

template <int BN, bool kRelu, bool kAcc, bool kMN = false, bool kTwo = false>
cudaError_t launch_bn(const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap& tmY,
                      const void* bias, void* Y,
                      int M, int N, int K, int64_t ldy, const DevCtx& ctx, cudaStream_t s,
                      const void* R, int ksplit, const GemmSecond& g2 = GemmSecond{}) {
  using S = GemmShape<BN>;
  auto kern = gemm_bias_bf16_kernel<BN, kRelu, kAcc, kMN, kTwo>;
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), S::kSmemBytes, nullptr);
  if (e != cudaSuccess) return e;
  int64_t units = static_cast<int64_t>((N + BN - 1) / BN) * ((M + kBM - 1) / kBM) * ksplit;
  if (kTwo) units += static_cast<int64_t>((g2.N + BN - 1) / BN) * ((g2.M + kBM - 1) / kBM);
  const int grid = static_cast<int>(units < ctx.num_sms ? units : ctx.num_sms);
  return launch_pdl(kern, dim3(grid), dim3(kThreads), S::kSmemBytes, s, tmX, tmW, tmY,
                    static_cast<const __nv_bfloat16*>(bias), static_cast<__nv_bfloat16*>(Y), M,
                    N, K, ldy, ctx.status, ctx.timeout_ns, static_cast<const __nv_bfloat16*>(R),
                    ksplit, g2);
}

// acc [M, N] fp32 -> Y bf16 (row pitch ldy), 8 values per thread
__global__ void __launch_bounds__(256)
    acc_to_bf16_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ Y, int M,
                       int N, int64_t ldy) {
  pdl_launch_dependents();
  pdl_wait();  // the split-K GEMM's reductions are complete from here on
  const int64_t per_row = N / 8;
  const int64_t total = static_cast<int64_t>(M) * per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / per_row;
    const int col = static_cast<int>(i % per_row) * 8;
    const float4* src = reinterpret_cast<const float4*>(acc + row * N + col);
    const float4 x = __ldcs(src), y = __ldcs(src + 1);
    uint4 v;
    v.x = pack_bf16x2(x.x, x.y);
    v.y = pack_bf16x2(x.z, x.w);
    v.z = pack_bf16x2(y.x, y.y);
    v.w = pack_bf16x2(y.z, y.w);
    *reinterpret_cast<uint4*>(Y + row * ldy + col) = v;
  }
}

}  // namespace

cudaError_t launch_gemm_bf16(const CUtensorMap& tmX, const CUtensorMap& tmW,
                             const CUtensorMap& tmY, int block_n,
                             bool relu, const void* bias, void* Y, int M, int N, int K,
                             int64_t ldy, const DevCtx& ctx, cudaStream_t s, const void* R) {
  if (relu) {
    if (block_n == 256)
      return launch_bn<256, true, false>(tmX, tmW, tmY, bias, Y, M, N, K, ldy, ctx, s, R, 1);
    return launch_bn<128, true, false>(tmX, tmW, tmY, bias, Y, M, N, K, ldy, ctx, s, R, 1);
  }
  if (block_n == 256)
    return launch_bn<256, false, false>(tmX, tmW, tmY, bias, Y, M, N, K, ldy, ctx, s, R, 1);
  return launch_bn<128, false, false>(tmX, tmW, tmY, bias, Y, M, N, K, ldy, ctx, s, R, 1);
}

cudaError_t launch_gemm_bf16_two(const CUtensorMap& tmX1, const CUtensorMap& tmW1,
                                 const CUtensorMap& tmY1, const void* bias1, int M1, int N1,
                                 const CUtensorMap& tmX2, const CUtensorMap& tmW2,
                                 const CUtensorMap& tmY2, const void* bias2, int M2, int N2,
                                 int K, int block_n, const DevCtx& ctx, cudaStream_t s) {
  GemmSecond g2;
  g2.tmX = tmX2;
  g2.tmW = tmW2;
  g2.tmY = tmY2;
  g2.bias = static_cast<const __nv_bfloat16*>(bias2);
  g2.M = M2;
  g2.N = N2;
  if (block_n == 256)
    return launch_bn<256, false, false, false, true>(tmX1, tmW1, tmY1, bias1, nullptr, M1, N1, K,
                                                     N1, ctx, s, nullptr, 1, g2);
  return launch_bn<128, false, false, false, true>(tmX1, tmW1, tmY1, bias1, nullptr, M1, N1, K,
                                                   N1, ctx, s, nullptr, 1, g2);
}

cudaError_t launch_gemm_bf16_mn(const CUtensorMap& tmX, const CUtensorMap& tmW,
                                const CUtensorMap& tmY, void* Y, int M, int N, int K,
                                int64_t ldy, const DevCtx& ctx, cudaStream_t s) {
  return launch_bn<128, false, false, true>(tmX, tmW, tmY, nullptr, Y, M, N, K, ldy, ctx, s,
                                            nullptr, 1);
}

cudaError_t launch_gemm_bf16_splitk(const CUtensorMap& tmX, const CUtensorMap& tmW,
                                    const CUtensorMap& tmAcc, float* acc, int ksplit, void* Y,
                                    int M, int N, int K, int64_t ldy, const DevCtx& ctx,
                                    cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(acc, 0, static_cast<size_t>(M) * N * 4, s);
  if (e != cudaSuccess) return e;
  e = launch_bn<128, false, true, true>(tmX, tmW, tmAcc, nullptr, nullptr, M, N, K, N, ctx, s,
                                        nullptr, ksplit);
  if (e != cudaSuccess) return e;
  const int64_t total = static_cast<int64_t>(M) * (N / 8);
  const int64_t want = (total + 255) / 256;
  const int blocks =
      static_cast<int>(want < static_cast<int64_t>(ctx.num_sms) * 8 ? want : ctx.num_sms * 8);
  return launch_pdl(acc_to_bf16_kernel, dim3(blocks), dim3(256), 0, s,
                    static_cast<const float*>(acc), static_cast<__nv_bfloat16*>(Y), M, N, ldy);
}

}  // namespace mha
