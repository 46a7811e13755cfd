// capi.cu -- the C ABI of libmha.so (declared in include/mha.h): argument validation, TMA
// descriptor encoding, workspace carving and launch sequencing.  No device memory is
// allocated here; the only device state is the 4-int error word below.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "mha.h"
#include "device_common.cuh"
#include "launchers.h"

// An NVTX range over the rest of the scope: every public entry point that launches work and
// every step inside it (projection, attention, ...) shows up by name in a profiler's timeline;
// without a profiler attached the calls return at once.
namespace {
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace
#define MHA_NVTX_CAT2(a, b) a##b
#define MHA_NVTX_CAT(a, b) MHA_NVTX_CAT2(a, b)
#define MHA_NVTX_RANGE(name) NvtxRange MHA_NVTX_CAT(nvtx_range_, __LINE__)(name)

namespace {

using mha::DevCtx;

// [0] first error code, [1] site, [2] blockIdx.x, [3] blockIdx.y (see device_common.cuh)
__device__ int g_device_status[4];

// ------------------------------------------------------------------ per-device properties
constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool init = false;
  bool supported = false;
  int num_sms = 0;
  int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

uint64_t wait_timeout_ns() {
  static uint64_t v = [] {
    const char* s = std::getenv("MHA_WAIT_TIMEOUT_NS");
    if (s != nullptr) {
      const long long x = std::atoll(s);
      if (x >= 1000 && x <= 60000000000LL) return static_cast<uint64_t>(x);
    }
    return static_cast<uint64_t>(2000000000ull);  // 2 s
  }();
  return v;
}

int device_ctx(DevCtx* ctx) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MHA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return MHA_ERR_CUDA;
    }
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    if (d.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
        cudaGetLastError();
        return MHA_ERR_CUDA;
      }
      d.status = static_cast<int*>(p);
    }
    d.init = true;
  }
  if (!d.supported) return MHA_ERR_UNSUPPORTED;
  ctx->status = d.status;
  ctx->timeout_ns = wait_timeout_ns();
  ctx->num_sms = d.num_sms;
  return MHA_OK;
}

// ------------------------------------------------------------------ kernel preparation
}  // namespace

namespace mha {
cudaError_t prepare_kernel(const void* func, int smem_bytes, int* num_regs) {
  struct Entry {
    const void* func;
    int dev, smem, regs;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (const Entry& x : done)
    if (x.func == func && x.dev == dev && x.smem == smem_bytes) {
      if (num_regs != nullptr) *num_regs = x.regs;
      return cudaSuccess;
    }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, func);
  if (e != cudaSuccess) return e;
  done.push_back({func, dev, smem_bytes, fa.numRegs});
  if (num_regs != nullptr) *num_regs = fa.numRegs;
  return cudaSuccess;
}
}  // namespace mha

namespace {
// ------------------------------------------------------------------ TMA descriptors
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols] with row pitch ld (elements); box {64 cols, box_rows}.
bool map_2d_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld,
                 uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows, cols] contiguous, box {32, 32}: the split-K GEMM's accumulator
bool map_2d_f32_acc(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B, H, N, 64] bf16 tensor with element strides st = {b, h, n, d=1}; box {64, box_rows, 1, 1}.
bool map_bhnd_bf16(CUtensorMap* m, const void* base, int B, int H, int N, const int64_t* st,
                   uint32_t box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2,
                           static_cast<cuuint64_t>(st[1]) * 2,
                           static_cast<cuuint64_t>(st[0]) * 2};
  cuuint32_t box[4] = {64, box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// the fp32 dQ accumulator of the fused bf16 attention backward, [B, H, rows, 64] contiguous:
// one 32 x 32 box (128-byte rows, 128-byte swizzle) per bulk reduction
bool map_dq_acc_f32(CUtensorMap* m, const void* base, int B, int H, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {64 * 4, static_cast<cuuint64_t>(rows) * 64 * 4,
                           static_cast<cuuint64_t>(H) * rows * 64 * 4};
  cuuint32_t box[4] = {32, 32, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The sublayer's last two steps as one kernel (W^O fused with the residual LayerNorm) pay off
// once there are enough 128-row tiles for each cluster of the fused kernel to work through
// several: same-box A/B of whole sublayers, 8192 rows (base model, causal, n = 256) 51.8 ->
// 48.8 us, the big model's 32768 rows 0.703 -> 0.689 ms, the big FFN sublayer (K = 4096)
// 375 -> 373 us; at 4096 rows (base model, n = 128) the fused launch is slower (38.6 -> 40.6
// us sublayer, 33.4 -> 36.5 us FFN sublayer), so the projection and the LayerNorm stay two
// launches there.
bool use_fused_out_ln(int dtype, int M, int D, int K) {
  return dtype == MHA_BF16 && mha::gemm_ln_bf16_supported(D, K) && M >= 8192;
}

// mha_set_deterministic: the bf16 attention backward's dQ by its own kernel (bitwise
// reproducible) instead of fp32 bulk reductions in whatever order the key tiles finish
std::atomic<int> g_deterministic{0};

// ------------------------------------------------------------------ step launchers
int run_linear(int M, int N, int K, int dtype, const void* X, int64_t ldx, const void* W,
               const void* bias, void* Y, int64_t ldy, const DevCtx& ctx, cudaStream_t s,
               bool relu = false, const void* residual = nullptr) {
  MHA_NVTX_RANGE("linear");
  cudaError_t e;
  if (dtype == MHA_BF16) {
    CUtensorMap tmX, tmW, tmY;
    // at least four rounds of 256 x 256 tiles for the pairs of SMs: the two-CTA form (half of
    // each operand per SM, a deeper ring of K slices).  Same-box A/B: 32768 x 3072 x 1024 137.9
    // -> 127.6 us, 32768 x 4096 x 1024 (ReLU) 174.7 -> 162.4 us, 16384 x 2048 x 1024 53.9 ->
    // 49.8 us; with 1-3 rounds (8192 or 4096 rows, K = 512) it was ~2 us slower, so those keep
    // the single-CTA kernel.
    const int64_t pair_tiles = ((M + 255) / 256) * static_cast<int64_t>((N + 255) / 256);
    if (mha::gemm2_bf16_supported(M, N, K) && pair_tiles >= 4 * (ctx.num_sms / 2) &&
        residual == nullptr) {
      if (!map_2d_bf16(&tmX, X, K, M, ldx, 128) || !map_2d_bf16(&tmW, W, K, N, K, 128) ||
          !map_2d_bf16(&tmY, Y, N, M, ldy, 32))
        return MHA_ERR_CUDA;
      e = mha::launch_gemm2_bf16(tmX, tmW, tmY, relu, bias, M, N, K, ctx, s);
      return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
    }
    const int64_t tiles256 = ((M + 127) / 128) * static_cast<int64_t>((N + 255) / 256);
    const int bn = (tiles256 >= ctx.num_sms) ? 256 : 128;
    if (!map_2d_bf16(&tmX, X, K, M, ldx, 128) || !map_2d_bf16(&tmW, W, K, N, K, bn) ||
        !map_2d_bf16(&tmY, Y, N, M, ldy, 32))
      return MHA_ERR_CUDA;
    e = mha::launch_gemm_bf16(tmX, tmW, tmY, bn, relu, bias, Y, M, N, K, ldy, ctx, s, residual);
  } else {
    e = mha::launch_gemm_f32(static_cast<const float*>(X), ldx, static_cast<const float*>(W),
                             static_cast<const float*>(bias), relu, static_cast<float*>(Y), ldy,
                             M, N, K, s, static_cast<const float*>(residual));
  }
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

// The two projections of cross-attention, Y1 = X1 W1^T + b1 and Y2 = X2 W2^T + b2 with the same
// K.  bf16 problems too small for the pair form alone run as one launch (the CTAs take the
// second problem's tiles after the first's), so the GPU fills once; everything else is two
// run_linear calls.
int run_linear_two(int M1, int N1, const void* X1, const void* W1, const void* b1, void* Y1,
                   int M2, int N2, const void* X2, const void* W2, const void* b2, void* Y2,
                   int K, int dtype, const DevCtx& ctx, cudaStream_t s) {
  const int64_t pair_tiles = ((M1 + 255) / 256) * static_cast<int64_t>((N1 + 255) / 256) +
                             ((M2 + 255) / 256) * static_cast<int64_t>((N2 + 255) / 256);
  if (dtype == MHA_BF16 && pair_tiles < 4 * (ctx.num_sms / 2) && K % 64 == 0 &&
      N1 % 64 == 0 && N2 % 64 == 0) {
    MHA_NVTX_RANGE("linear_two");
    const int64_t tiles256 = ((M1 + 127) / 128) * static_cast<int64_t>((N1 + 255) / 256) +
                             ((M2 + 127) / 128) * static_cast<int64_t>((N2 + 255) / 256);
    const int bn = (tiles256 >= ctx.num_sms) ? 256 : 128;
    CUtensorMap tmX1, tmW1, tmY1, tmX2, tmW2, tmY2;
    if (!map_2d_bf16(&tmX1, X1, K, M1, K, 128) || !map_2d_bf16(&tmW1, W1, K, N1, K, bn) ||
        !map_2d_bf16(&tmY1, Y1, N1, M1, N1, 32) || !map_2d_bf16(&tmX2, X2, K, M2, K, 128) ||
        !map_2d_bf16(&tmW2, W2, K, N2, K, bn) || !map_2d_bf16(&tmY2, Y2, N2, M2, N2, 32))
      return MHA_ERR_CUDA;
    const cudaError_t e = mha::launch_gemm_bf16_two(tmX1, tmW1, tmY1, b1, M1, N1, tmX2, tmW2,
                                                    tmY2, b2, M2, N2, K, bn, ctx, s);
    return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
  }
  const int st = run_linear(M1, N1, K, dtype, X1, K, W1, b1, Y1, N1, ctx, s);
  if (st != MHA_OK) return st;
  return run_linear(M2, N2, K, dtype, X2, K, W2, b2, Y2, N2, ctx, s);
}

// K slices for a weight-gradient GEMM whose 128 x 128 tiles alone would fill the SMs badly:
// the smallest split whose work units fill >= 90% of their last round (else the best of
// 1..8), with at least 8 K blocks of 64 per slice
int wgrad_ksplit(int M, int N, int K, int num_sms) {
  const int64_t tiles = static_cast<int64_t>((M + 127) / 128) * ((N + 127) / 128);
  int best = 1;
  double best_eff = 0.0;
  for (int ks = 1; ks <= 8 && (K / 64) / ks >= 8; ++ks) {
    const int64_t units = tiles * ks;
    const int64_t rounds = (units + num_sms - 1) / num_sms;
    const double eff = static_cast<double>(units) / static_cast<double>(rounds * num_sms);
    if (eff >= 0.9) return ks;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = ks;
    }
  }
  return best;
}

// dW [M, N] = A^T B for the weight gradients, from the row-major activations A_st [K, M]
// (row pitch lda) and B_st [K, N] (row pitch ldb), K = tokens.  bf16: both read MN-major by
// the tensor-core GEMM, split over K when that fills the GPU better (fp32 scratch acc of M * N
// values; not in the deterministic mode).  fp32: transposed into At [M, Kpad] and Bt [N, Kpad]
// (zero-padded to Kpad, a multiple of 64) for the SIMT GEMM.
int run_linear_wgrad(int M, int N, int K, int dtype, const void* A_st, int64_t lda,
                     const void* B_st, int64_t ldb, void* Y, int64_t ldy, float* acc, void* At,
                     void* Bt, int Kpad, const DevCtx& ctx, cudaStream_t s) {
  MHA_NVTX_RANGE("linear_weight_gradient");
  if (dtype != MHA_BF16) {
    if (mha::launch_transpose(dtype, A_st, lda, K, M, At, Kpad, Kpad, s) != cudaSuccess ||
        mha::launch_transpose(dtype, B_st, ldb, K, N, Bt, Kpad, Kpad, s) != cudaSuccess)
      return MHA_ERR_CUDA;
    return run_linear(M, N, Kpad, dtype, At, Kpad, Bt, nullptr, Y, ldy, ctx, s);
  }
  CUtensorMap tmA, tmB, tmY;
  if (!map_2d_bf16(&tmA, A_st, M, K, lda, 64) || !map_2d_bf16(&tmB, B_st, N, K, ldb, 64))
    return MHA_ERR_CUDA;
  const int ks = g_deterministic.load(std::memory_order_relaxed) != 0
                     ? 1
                     : wgrad_ksplit(M, N, (K + 63) / 64 * 64, ctx.num_sms);
  cudaError_t e;
  if (ks > 1 && N % 8 == 0) {
    if (!map_2d_f32_acc(&tmY, acc, N, M)) return MHA_ERR_CUDA;
    e = mha::launch_gemm_bf16_splitk(tmA, tmB, tmY, acc, ks, Y, M, N, K, ldy, ctx, s);
  } else {
    if (!map_2d_bf16(&tmY, Y, N, M, ldy, 32)) return MHA_ERR_CUDA;
    e = mha::launch_gemm_bf16_mn(tmA, tmB, tmY, Y, M, N, K, ldy, ctx, s);
  }
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

int run_sdpa(const mha::SdpaArgs& a, int dtype, const DevCtx& ctx, cudaStream_t s) {
  MHA_NVTX_RANGE("attention");
  cudaError_t e;
  if (dtype == MHA_BF16) {
    CUtensorMap tq, tk, tv, to;
    if (!map_bhnd_bf16(&tq, a.Q, a.B, a.H, a.Nq, a.sq) ||
        !map_bhnd_bf16(&tk, a.K, a.B, a.H, a.Nk, a.sk) ||
        !map_bhnd_bf16(&tv, a.V, a.B, a.H, a.Nk, a.sv) ||
        !map_bhnd_bf16(&to, a.O, a.B, a.H, a.Nq, a.so, 32))
      return MHA_ERR_CUDA;
    e = mha::launch_sdpa_bf16(tq, tk, tv, to, a, ctx, s);
  } else {
    mha::SdpaArgs af = a;
    af.status = ctx.status;
    e = mha::launch_sdpa_f32(af, s);
  }
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

// rowdot (D) and the gradient kernels of one attention backward; a.Dv is the caller's scratch
int run_sdpa_bwd(mha::SdpaBwdArgs a, int dtype, const DevCtx& ctx, cudaStream_t s) {
  MHA_NVTX_RANGE("attention_backward");
  a.deterministic = g_deterministic.load(std::memory_order_relaxed) != 0;
  cudaError_t e = mha::launch_sdpa_bwd_rowdot(a, dtype, s);
  if (e != cudaSuccess) return MHA_ERR_CUDA;
  if (dtype == MHA_BF16) {
    CUtensorMap tq, tk, tv, tg, tdq;
    const void* acc = reinterpret_cast<const char*>(a.Dv) +
                      mha::sdpa_bwd_dq_acc_offset(a.B, a.H, a.Nq);
    if (!map_bhnd_bf16(&tq, a.Q, a.B, a.H, a.Nq, a.st[0]) ||
        !map_bhnd_bf16(&tk, a.K, a.B, a.H, a.Nk, a.st[1]) ||
        !map_bhnd_bf16(&tv, a.V, a.B, a.H, a.Nk, a.st[2]) ||
        !map_bhnd_bf16(&tg, a.dO, a.B, a.H, a.Nq, a.st[4]) ||
        !map_dq_acc_f32(&tdq, acc, a.B, a.H, (a.Nq + 127) / 128 * 128))
      return MHA_ERR_CUDA;
    e = mha::launch_sdpa_bwd_bf16(tq, tk, tv, tg, tdq, a, ctx, s);
  } else {
    e = mha::launch_sdpa_bwd_f32(a, s);
  }
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

bool valid_dtype(int dt) { return dt == MHA_F32 || dt == MHA_BF16; }
size_t elem_size(int dt) { return dt == MHA_BF16 ? 2 : 4; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct LayerPlan {
  size_t off_q, off_kv, off_c, off_a, total;
};
LayerPlan plan_layer(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype) {
  const size_t es = elem_size(dtype);
  const size_t Mq = static_cast<size_t>(B) * Nq, Mk = static_cast<size_t>(B) * Nk;
  LayerPlan p;
  // self-attention keeps Q|K|V interleaved per token in [off_q, off_c): the same bytes as
  // Q [Mq, H*d_k] followed by K|V [Mk, H*(d_k+d_v)] when Nq == Nk.
  p.off_q = 0;
  p.off_kv = round_up(Mq * H * d_k * es, 256);
  p.off_c = p.off_kv + round_up(Mk * H * (d_k + d_v) * es, 256);
  p.off_a = p.off_c + round_up(Mq * H * d_v * es, 256);
  p.total = p.off_a + round_up(Mq * D * es, 256);
  return p;
}

int check_layer_shape(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || D < 1 || d_k < 1 || d_v < 1) return MHA_ERR_INVALID;
  if (!valid_dtype(dtype)) return MHA_ERR_INVALID;
  // launch-grid and index limits (token counts index rows with 32-bit ints)
  if (B > 65535 || H > 65535 || static_cast<int64_t>(B) * Nq > (1LL << 24) ||
      static_cast<int64_t>(B) * Nk > (1LL << 24))
    return MHA_ERR_UNSUPPORTED;
  if (dtype == MHA_BF16) {
    if (d_k != 64 || d_v != 64 || D % 64 != 0) return MHA_ERR_UNSUPPORTED;
  } else {
    if (d_k > 128 || d_v > 128) return MHA_ERR_UNSUPPORTED;
  }
  if (D % 8 != 0 || D > 2048) return MHA_ERR_UNSUPPORTED;  // residual LayerNorm kernel limits
  return MHA_OK;
}

// Feed-forward sublayer scratch: the hidden activations H [M, d_ff], then FFN(x) [M, D].
struct FfnPlan {
  size_t off_h, off_f, total;
};
FfnPlan plan_ffn(int M, int D, int d_ff, int dtype) {
  const size_t es = elem_size(dtype);
  FfnPlan p;
  p.off_h = 0;
  p.off_f = round_up(static_cast<size_t>(M) * d_ff * es, 256);
  p.total = p.off_f + round_up(static_cast<size_t>(M) * D * es, 256);
  return p;
}

int check_ffn_shape(int M, int D, int d_ff, int dtype) {
  if (M < 1 || D < 1 || d_ff < 1 || !valid_dtype(dtype)) return MHA_ERR_INVALID;
  if (M > (1 << 24)) return MHA_ERR_UNSUPPORTED;
  if (dtype == MHA_BF16 && (D % 64 != 0 || d_ff % 64 != 0)) return MHA_ERR_UNSUPPORTED;
  if (D % 8 != 0 || D > 2048) return MHA_ERR_UNSUPPORTED;  // residual LayerNorm kernel limits
  return MHA_OK;
}

// Encoder layer scratch: the attention sublayer's output h [M, D], then one region that the
// attention sublayer's workspace and, after it, the feed-forward sublayer's workspace share.
struct EncoderPlan {
  size_t off_h, off_ws, total;
};
EncoderPlan plan_encoder(int B, int N, int H, int D, int d_ff, int dtype) {
  EncoderPlan p;
  p.off_h = 0;
  p.off_ws = round_up(static_cast<size_t>(B) * N * D * elem_size(dtype), 256);
  const size_t a = plan_layer(B, H, N, N, D, D / H, D / H, dtype).total;
  const size_t f = plan_ffn(B * N, D, d_ff, dtype).total;
  p.total = p.off_ws + (a > f ? a : f);
  return p;
}

// argument checks shared by the linear-map entry points (defined with them below)
int check_linear(int M, int N, int K, int dtype, const void* X, int64_t ldx, const void* W,
                 const void* bias, const void* Y, int64_t ldy);

__global__ void wait_selftest_kernel(int* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mha::mbar_init(mha::smem_u32(&bar), 1);
    mha::fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives on this barrier: the wait must give up and report
  if (!mha::mbar_wait(mha::smem_u32(&bar), 0, timeout_ns) && threadIdx.x == 0)
    mha::record_error(status, MHA_ERR_DEVICE_TIMEOUT, 99);
  __syncthreads();
}

}  // namespace

namespace mha {
cudaError_t launch_wait_selftest(const DevCtx& ctx, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(ctx.status, ctx.timeout_ns);
  return cudaGetLastError();
}
}  // namespace mha

// ==================================================================== exported C ABI
extern "C" {

int mha_abi_version(void) { return 100; }

const char* mha_status_string(int st) {
  switch (st) {
    case MHA_OK: return "MHA_OK";
    case MHA_ERR_INVALID: return "MHA_ERR_INVALID: invalid argument";
    case MHA_ERR_UNSUPPORTED: return "MHA_ERR_UNSUPPORTED: valid request not supported by this build or device";
    case MHA_ERR_ALIGN: return "MHA_ERR_ALIGN: pointer or stride misaligned";
    case MHA_ERR_WORKSPACE: return "MHA_ERR_WORKSPACE: workspace missing or too small";
    case MHA_ERR_CUDA: return "MHA_ERR_CUDA: CUDA call or launch failed";
    case MHA_ERR_DEVICE_TIMEOUT: return "MHA_ERR_DEVICE_TIMEOUT: a device-side wait ran out";
    case MHA_ERR_DEVICE_BOUNDS:
      return "MHA_ERR_DEVICE_BOUNDS: a kernel index fell outside its buffer (debug build)";
    default: return "unknown mha status";
  }
}

}  // extern "C"

namespace {
// mask: an mha_mask value or mha::kMaskWindow (then `window` is the neighbourhood radius)
int sdpa_entry(int B, int H, int Nq, int Nk, int d_k, int d_v, int dtype, int mask,
               const int32_t* key_len, int window, float scale, const void* Q, const void* K,
               const void* V, void* O, const int64_t* strides, cudaStream_t stream,
               float* lse = nullptr) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d_k < 1 || d_v < 1) return MHA_ERR_INVALID;
  if (!valid_dtype(dtype) || mask < MHA_MASK_NONE ||
      (mask > MHA_MASK_KEY_PADDING && mask != mha::kMaskWindow))
    return MHA_ERR_INVALID;
  if (mask == mha::kMaskWindow && (Nq != Nk || window < 0)) return MHA_ERR_INVALID;
  if (mask == MHA_MASK_CAUSAL && Nq != Nk) return MHA_ERR_INVALID;
  if (mask == MHA_MASK_KEY_PADDING && key_len == nullptr) return MHA_ERR_INVALID;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return MHA_ERR_INVALID;
  if (std::isnan(scale) || std::isinf(scale)) return MHA_ERR_INVALID;
  if (key_len != nullptr && !aligned(key_len, 4)) return MHA_ERR_ALIGN;
  // launch-grid limits: (H, B, Nq/256) for bf16, (Nq/8, H, B) for fp32
  if (B > 65535 || H > 65535 || (Nq + 255) / 256 > 65535) return MHA_ERR_UNSUPPORTED;

  mha::SdpaArgs a;
  a.B = B; a.H = H; a.Nq = Nq; a.Nk = Nk; a.d_k = d_k; a.d_v = d_v;
  a.mask = mask;
  a.key_len = (mask == MHA_MASK_KEY_PADDING) ? key_len : nullptr;
  // a radius of Nk or more already reaches every key
  a.window = (mask == mha::kMaskWindow) ? (window < Nk ? window : Nk) : 0;
  a.Q = Q; a.K = K; a.V = V; a.O = O;
  a.lse = lse;
  if (lse != nullptr && !aligned(lse, 4)) return MHA_ERR_ALIGN;
  const int64_t cont[4][4] = {
      {static_cast<int64_t>(H) * Nq * d_k, static_cast<int64_t>(Nq) * d_k, d_k, 1},
      {static_cast<int64_t>(H) * Nk * d_k, static_cast<int64_t>(Nk) * d_k, d_k, 1},
      {static_cast<int64_t>(H) * Nk * d_v, static_cast<int64_t>(Nk) * d_v, d_v, 1},
      {static_cast<int64_t>(H) * Nq * d_v, static_cast<int64_t>(Nq) * d_v, d_v, 1}};
  int64_t* dst[4] = {a.sq, a.sk, a.sv, a.so};
  for (int t = 0; t < 4; ++t)
    for (int i = 0; i < 4; ++i) {
      dst[t][i] = strides ? strides[4 * t + i] : cont[t][i];
      if (dst[t][i] < 0) return MHA_ERR_INVALID;
    }
  const void* ptrs[4] = {Q, K, V, O};
  if (dtype == MHA_BF16) {
    if (d_k != 64 || d_v != 64) return MHA_ERR_UNSUPPORTED;
    for (int t = 0; t < 4; ++t) {
      if (dst[t][3] != 1) return MHA_ERR_UNSUPPORTED;
      for (int i = 0; i < 3; ++i)
        if (dst[t][i] == 0 || dst[t][i] % 8 != 0) return MHA_ERR_ALIGN;
      if (!aligned(ptrs[t], 16)) return MHA_ERR_ALIGN;
    }
  } else {
    if (d_k > 128 || d_v > 128) return MHA_ERR_UNSUPPORTED;
    for (int t = 0; t < 4; ++t)
      if (!aligned(ptrs[t], 4)) return MHA_ERR_ALIGN;
  }
  DevCtx ctx;
  int st = device_ctx(&ctx);
  if (st != MHA_OK) return st;
  a.scale = scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k)));
  return run_sdpa(a, dtype, ctx, stream);
}
}  // namespace

extern "C" {

int mha_sdpa_fwd(int B, int H, int Nq, int Nk, int d_k, int d_v, int dtype, int mask,
                 const int32_t* key_len, float scale, const void* Q, const void* K, const void* V,
                 void* O, const int64_t* strides, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_sdpa_fwd");
  if (mask < MHA_MASK_NONE || mask > MHA_MASK_KEY_PADDING) return MHA_ERR_INVALID;
  return sdpa_entry(B, H, Nq, Nk, d_k, d_v, dtype, mask, key_len, 0, scale, Q, K, V, O, strides,
                    stream);
}

int mha_decode_workspace_size(int B, int H, int Nq, int Lmax, int dtype, size_t* bytes) {
  if (bytes == nullptr || B < 1 || H < 1 || Nq < 1 || Lmax < 1 || !valid_dtype(dtype))
    return MHA_ERR_INVALID;
  if (dtype == MHA_BF16 && Nq > mha::kDecodeMaxQ) return MHA_ERR_UNSUPPORTED;
  // bf16: one fp32 partial (64 columns, max, sum) per (batch, head, 256-key chunk, query);
  // the fp32 path needs none (at least 256 bytes are asked for so a buffer always exists)
  const size_t parts = static_cast<size_t>(B) * H * mha::decode_num_splits(Lmax) * Nq;
  *bytes = dtype == MHA_BF16 ? round_up(parts * 66 * sizeof(float), 256) : 256;
  return MHA_OK;
}

int mha_sdpa_decode_fwd(int B, int H, int Nq, int Lmax, int d_k, int d_v, int dtype, int causal,
                        const int32_t* cache_len, float scale, const void* Q, const void* K,
                        const void* V, void* O, const int64_t* strides, void* workspace,
                        size_t ws_bytes, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_sdpa_decode_fwd");
  if (B < 1 || H < 1 || Nq < 1 || Lmax < 1 || d_k < 1 || d_v < 1 || !valid_dtype(dtype))
    return MHA_ERR_INVALID;
  if ((causal != 0 && causal != 1) || Nq > Lmax) return MHA_ERR_INVALID;
  if (cache_len == nullptr || Q == nullptr || K == nullptr || V == nullptr || O == nullptr)
    return MHA_ERR_INVALID;
  if (std::isnan(scale) || std::isinf(scale)) return MHA_ERR_INVALID;
  if (!aligned(cache_len, 4)) return MHA_ERR_ALIGN;
  if (B > 65535 || H > 65535) return MHA_ERR_UNSUPPORTED;
  size_t need = 0;
  int st = mha_decode_workspace_size(B, H, Nq, Lmax, dtype, &need);
  if (st != MHA_OK) return st;
  if (workspace == nullptr || ws_bytes < need) return MHA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MHA_ERR_ALIGN;
  const int64_t cont[4][4] = {
      {static_cast<int64_t>(H) * Nq * d_k, static_cast<int64_t>(Nq) * d_k, d_k, 1},
      {static_cast<int64_t>(H) * Lmax * d_k, static_cast<int64_t>(Lmax) * d_k, d_k, 1},
      {static_cast<int64_t>(H) * Lmax * d_v, static_cast<int64_t>(Lmax) * d_v, d_v, 1},
      {static_cast<int64_t>(H) * Nq * d_v, static_cast<int64_t>(Nq) * d_v, d_v, 1}};
  int64_t str[4][4];
  for (int t = 0; t < 4; ++t)
    for (int i = 0; i < 4; ++i) {
      str[t][i] = strides ? strides[4 * t + i] : cont[t][i];
      if (str[t][i] < 0) return MHA_ERR_INVALID;
    }
  const void* ptrs[4] = {Q, K, V, O};
  const float sc =
      scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k)));
  if (dtype == MHA_BF16) {
    if (d_k != 64 || d_v != 64) return MHA_ERR_UNSUPPORTED;
    for (int t = 0; t < 4; ++t) {
      if (str[t][3] != 1) return MHA_ERR_UNSUPPORTED;
      for (int i = 0; i < 3; ++i)
        if (str[t][i] == 0 || str[t][i] % 8 != 0) return MHA_ERR_ALIGN;
      if (!aligned(ptrs[t], 16)) return MHA_ERR_ALIGN;
    }
    DevCtx ctx;
    st = device_ctx(&ctx);
    if (st != MHA_OK) return st;
    CUtensorMap tk, tv;
    if (!map_bhnd_bf16(&tk, K, B, H, Lmax, str[1]) || !map_bhnd_bf16(&tv, V, B, H, Lmax, str[2]))
      return MHA_ERR_CUDA;
    mha::DecodeArgs a;
    a.B = B; a.H = H; a.Nq = Nq; a.Lmax = Lmax; a.causal = causal;
    a.cache_len = cache_len;
    a.scale = sc;
    a.Q = Q; a.O = O;
    for (int i = 0; i < 4; ++i) {
      a.sq[i] = str[0][i];
      a.so[i] = str[3][i];
    }
    cudaError_t e = mha::launch_sdpa_decode_bf16(tk, tv, a, static_cast<float*>(workspace), ctx,
                                                 stream);
    return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
  }
  // fp32: the SIMT attention kernel with the cache's masks (one warp per query row)
  if (d_k > 128 || d_v > 128) return MHA_ERR_UNSUPPORTED;
  for (int t = 0; t < 4; ++t)
    if (!aligned(ptrs[t], 4)) return MHA_ERR_ALIGN;
  DevCtx ctx;
  st = device_ctx(&ctx);
  if (st != MHA_OK) return st;
  mha::SdpaArgs a;
  a.B = B; a.H = H; a.Nq = Nq; a.Nk = Lmax; a.d_k = d_k; a.d_v = d_v;
  a.mask = causal ? mha::kMaskCausalCache : MHA_MASK_KEY_PADDING;
  a.key_len = cache_len;
  a.scale = sc;
  a.Q = Q; a.K = K; a.V = V; a.O = O;
  int64_t* dst[4] = {a.sq, a.sk, a.sv, a.so};
  for (int t = 0; t < 4; ++t)
    for (int i = 0; i < 4; ++i) dst[t][i] = str[t][i];
  return run_sdpa(a, dtype, ctx, stream);
}

int mha_sdpa_fwd_lse(int B, int H, int Nq, int Nk, int d_k, int d_v, int dtype, int mask,
                     const int32_t* key_len, float scale, const void* Q, const void* K,
                     const void* V, void* O, const int64_t* strides, float* lse,
                     cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_sdpa_fwd_lse");
  if (mask < MHA_MASK_NONE || mask > MHA_MASK_KEY_PADDING || lse == nullptr)
    return MHA_ERR_INVALID;
  return sdpa_entry(B, H, Nq, Nk, d_k, d_v, dtype, mask, key_len, 0, scale, Q, K, V, O, strides,
                    stream, lse);
}

int mha_sdpa_bwd_workspace_size(int B, int H, int Nq, int dtype, size_t* bytes) {
  if (bytes == nullptr || B < 1 || H < 1 || Nq < 1 || !valid_dtype(dtype))
    return MHA_ERR_INVALID;
  *bytes = round_up(mha::sdpa_bwd_scratch_bytes(B, H, Nq, dtype), 256);  // D (and lse) per row
  return MHA_OK;
}

int mha_sdpa_bwd(int B, int H, int Nq, int Nk, int d_k, int d_v, int dtype, int mask,
                 const int32_t* key_len, float scale, const void* Q, const void* K,
                 const void* V, const void* O, const void* dO, const float* lse, void* dQ,
                 void* dK, void* dV, const int64_t* strides, void* workspace, size_t ws_bytes,
                 cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_sdpa_bwd");
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d_k < 1 || d_v < 1 || !valid_dtype(dtype))
    return MHA_ERR_INVALID;
  if (mask < MHA_MASK_NONE || mask > MHA_MASK_KEY_PADDING) return MHA_ERR_INVALID;
  if (mask == MHA_MASK_CAUSAL && Nq != Nk) return MHA_ERR_INVALID;
  if (mask == MHA_MASK_KEY_PADDING && key_len == nullptr) return MHA_ERR_INVALID;
  const void* ptrs[8] = {Q, K, V, O, dO, dQ, dK, dV};
  for (const void* q : ptrs)
    if (q == nullptr) return MHA_ERR_INVALID;
  if (lse == nullptr || std::isnan(scale) || std::isinf(scale)) return MHA_ERR_INVALID;
  if (!aligned(lse, 4) || (key_len != nullptr && !aligned(key_len, 4))) return MHA_ERR_ALIGN;
  if (B > 65535 || H > 65535 || (Nq + 127) / 128 > 65535 || (Nk + 127) / 128 > 65535)
    return MHA_ERR_UNSUPPORTED;
  size_t need = 0;
  int st = mha_sdpa_bwd_workspace_size(B, H, Nq, dtype, &need);
  if (st != MHA_OK) return st;
  if (workspace == nullptr || ws_bytes < need) return MHA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MHA_ERR_ALIGN;
  mha::SdpaBwdArgs a;
  a.B = B; a.H = H; a.Nq = Nq; a.Nk = Nk; a.d_k = d_k; a.d_v = d_v;
  a.mask = mask;
  a.window = 0;
  a.key_len = (mask == MHA_MASK_KEY_PADDING) ? key_len : nullptr;
  a.scale = scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k)));
  a.Q = Q; a.K = K; a.V = V; a.O = O; a.dO = dO;
  a.lse = lse;
  a.Dv = static_cast<float*>(workspace);
  a.dQ = dQ; a.dK = dK; a.dV = dV;
  // contiguous [B, H, N, d] unless strides are given: Q, K, V, O, dO, dQ, dK, dV
  const int rows[8] = {Nq, Nk, Nk, Nq, Nq, Nq, Nk, Nk};
  const int dims[8] = {d_k, d_k, d_v, d_v, d_v, d_k, d_k, d_v};
  for (int t = 0; t < 8; ++t) {
    const int64_t cont[4] = {static_cast<int64_t>(H) * rows[t] * dims[t],
                             static_cast<int64_t>(rows[t]) * dims[t], dims[t], 1};
    for (int i = 0; i < 4; ++i) {
      a.st[t][i] = strides ? strides[4 * t + i] : cont[i];
      if (a.st[t][i] < 0) return MHA_ERR_INVALID;
    }
  }
  if (dtype == MHA_BF16) {
    if (d_k != 64 || d_v != 64) return MHA_ERR_UNSUPPORTED;
    for (int t = 0; t < 8; ++t) {
      if (a.st[t][3] != 1) return MHA_ERR_UNSUPPORTED;
      for (int i = 0; i < 3; ++i)
        if (a.st[t][i] == 0 || a.st[t][i] % 8 != 0) return MHA_ERR_ALIGN;
      if (!aligned(ptrs[t], 16)) return MHA_ERR_ALIGN;
    }
  } else {
    if (d_k > 128 || d_v > 128) return MHA_ERR_UNSUPPORTED;
    for (int t = 0; t < 8; ++t) {
      if (a.st[t][3] != 1) return MHA_ERR_UNSUPPORTED;
      if (!aligned(ptrs[t], 4)) return MHA_ERR_ALIGN;
    }
  }
  DevCtx ctx;
  st = device_ctx(&ctx);
  if (st != MHA_OK) return st;
  return run_sdpa_bwd(a, dtype, ctx, stream);
}

int mha_sdpa_window_fwd(int B, int H, int N, int d_k, int d_v, int dtype, int window,
                        float scale, const void* Q, const void* K, const void* V, void* O,
                        const int64_t* strides, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_sdpa_window_fwd");
  return sdpa_entry(B, H, N, N, d_k, d_v, dtype, mha::kMaskWindow, nullptr, window, scale, Q, K,
                    V, O, strides, stream);
}

int mha_layer_workspace_size(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                             size_t* bytes) {
  if (bytes == nullptr) return MHA_ERR_INVALID;
  const int st = check_layer_shape(B, H, Nq, Nk, D, d_k, d_v, dtype);
  if (st != MHA_OK) return st;
  *bytes = plan_layer(B, H, Nq, Nk, D, d_k, d_v, dtype).total;
  return MHA_OK;
}

}  // extern "C"

namespace mha {
int check_layer_call(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype, int mask,
                     const int32_t* key_len, float ln_eps, const void* x_q, const void* x_kv,
                     const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                     const void* gamma, const void* beta, const void* y, const void* workspace,
                     size_t ws_bytes, bool builtin_workspace, DevCtx* ctx) {
  int st = check_layer_shape(B, H, Nq, Nk, D, d_k, d_v, dtype);
  if (st != MHA_OK) return st;
  if (mask < MHA_MASK_NONE || mask > MHA_MASK_KEY_PADDING) return MHA_ERR_INVALID;
  const bool self = (x_kv == nullptr);
  if ((self || mask == MHA_MASK_CAUSAL) && Nq != Nk) return MHA_ERR_INVALID;
  if (mask == MHA_MASK_KEY_PADDING && key_len == nullptr) return MHA_ERR_INVALID;
  if (x_q == nullptr || W_qkv == nullptr || W_o == nullptr || y == nullptr)
    return MHA_ERR_INVALID;
  if (std::isnan(ln_eps) || ln_eps < 0.f) return MHA_ERR_INVALID;
  const LayerPlan plan = plan_layer(B, H, Nq, Nk, D, d_k, d_v, dtype);
  if ((!builtin_workspace && workspace == nullptr) || ws_bytes < plan.total)
    return MHA_ERR_WORKSPACE;
  const void* all[] = {x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, y};
  for (const void* p : all)
    if (p != nullptr && !aligned(p, 16)) return MHA_ERR_ALIGN;
  if (key_len != nullptr && !aligned(key_len, 4)) return MHA_ERR_ALIGN;
  if (!builtin_workspace && !aligned(workspace, 256)) return MHA_ERR_ALIGN;
  return device_ctx(ctx);
}
}  // namespace mha

namespace {
// ev: null, or 5 events recorded on `stream` at the step boundaries (before the projections,
// before attention, before the output projection, before the residual LayerNorm, after it).
int layer_impl(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype, int mask,
               const int32_t* key_len, float ln_eps, const void* x_q, const void* x_kv,
               const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
               const void* gamma, const void* beta, void* y, void* workspace, size_t ws_bytes,
               cudaStream_t stream, const cudaEvent_t* ev) {
  auto mark = [&](int i) {
    if (ev != nullptr) cudaEventRecord(ev[i], stream);
  };
  DevCtx ctx;
  int st = mha::check_layer_call(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q,
                                 x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, y, workspace,
                                 ws_bytes, false, &ctx);
  if (st != MHA_OK) return st;
  const bool self = (x_kv == nullptr);
  const LayerPlan plan = plan_layer(B, H, Nq, Nk, D, d_k, d_v, dtype);

  const size_t es = elem_size(dtype);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int Mq = B * Nq, Mk = B * Nk;
  const int nqk = H * d_k, nv = H * d_v;
  const uint8_t* bq = static_cast<const uint8_t*>(b_qkv);
  const uint8_t* Wb = static_cast<const uint8_t*>(W_qkv);

  mha::SdpaArgs a;
  a.B = B; a.H = H; a.Nq = Nq; a.Nk = Nk; a.d_k = d_k; a.d_v = d_v;
  a.mask = mask;
  a.key_len = (mask == MHA_MASK_KEY_PADDING) ? key_len : nullptr;
  a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k)));

  mark(0);
  if (self) {
    // one GEMM: [Mq, D] x [2*nqk + nv, D]^T -> Q|K|V interleaved per token
    const int ld = 2 * nqk + nv;
    uint8_t* qkv = ws + plan.off_q;
    st = run_linear(Mq, ld, D, dtype, x_q, D, W_qkv, b_qkv, qkv, ld, ctx, stream);
    if (st != MHA_OK) return st;
    a.Q = qkv;
    a.K = qkv + nqk * es;
    a.V = qkv + 2 * nqk * es;
    const int64_t sq[4] = {static_cast<int64_t>(Nq) * ld, d_k, ld, 1};
    for (int i = 0; i < 4; ++i) a.sq[i] = a.sk[i] = a.sv[i] = sq[i];
  } else {
    uint8_t* qb = ws + plan.off_q;
    uint8_t* kvb = ws + plan.off_kv;
    const int ldkv = nqk + nv;
    st = run_linear_two(Mq, nqk, x_q, W_qkv, b_qkv, qb, Mk, ldkv, x_kv,
                        Wb + static_cast<size_t>(nqk) * D * es, bq ? bq + nqk * es : nullptr,
                        kvb, D, dtype, ctx, stream);
    if (st != MHA_OK) return st;
    a.Q = qb;
    a.K = kvb;
    a.V = kvb + nqk * es;
    const int64_t sq[4] = {static_cast<int64_t>(Nq) * nqk, d_k, nqk, 1};
    const int64_t skv[4] = {static_cast<int64_t>(Nk) * ldkv, d_k, ldkv, 1};
    for (int i = 0; i < 4; ++i) {
      a.sq[i] = sq[i];
      a.sk[i] = skv[i];
      a.sv[i] = skv[i];
    }
    a.sv[1] = d_v;
  }
  // attention writes heads side by side: C [B, Nq, H*d_v]
  uint8_t* C = ws + plan.off_c;
  a.O = C;
  a.so[0] = static_cast<int64_t>(Nq) * nv;
  a.so[1] = d_v;
  a.so[2] = nv;
  a.so[3] = 1;
  if (self) a.sv[1] = d_v;
  mark(1);
  st = run_sdpa(a, dtype, ctx, stream);
  if (st != MHA_OK) return st;
  mark(2);
  if (use_fused_out_ln(dtype, Mq, D, nv)) {
    // y = LayerNorm(x_q + C W_o^T + b_o) in one kernel: A stays on chip
    MHA_NVTX_RANGE("out_projection_layernorm");
    CUtensorMap tmC, tmWo;
    if (!map_2d_bf16(&tmC, C, nv, Mq, nv, 128) || !map_2d_bf16(&tmWo, W_o, nv, D, nv, 256))
      return MHA_ERR_CUDA;
    const cudaError_t e = mha::launch_gemm_ln_bf16(tmC, tmWo, b_o, x_q, gamma, beta, y, Mq, D,
                                                   nv, ln_eps, ctx, stream);
    mark(3);
    mark(4);
    return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
  }
  // A = C W_o^T + b_o
  uint8_t* A = ws + plan.off_a;
  st = run_linear(Mq, D, nv, dtype, C, nv, W_o, b_o, A, D, ctx, stream);
  if (st != MHA_OK) return st;
  // y = LayerNorm(x_q + A)
  mark(3);
  MHA_NVTX_RANGE("residual_layernorm");
  cudaError_t e =
      mha::launch_residual_layernorm(dtype, Mq, D, ln_eps, x_q, A, gamma, beta, y, ctx, stream);
  mark(4);
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}
}  // namespace

namespace {
// ev: null, or 4 events recorded on `stream` at the step boundaries (before the first linear
// map, before the second, before the residual LayerNorm, after it).
int ffn_impl(int M, int D, int d_ff, int dtype, float ln_eps, const void* x, const void* W1,
             const void* b1, const void* W2, const void* b2, const void* gamma,
             const void* beta, void* y, void* workspace, size_t ws_bytes, cudaStream_t stream,
             const cudaEvent_t* ev) {
  auto mark = [&](int i) {
    if (ev != nullptr) cudaEventRecord(ev[i], stream);
  };
  int st = check_ffn_shape(M, D, d_ff, dtype);
  if (st != MHA_OK) return st;
  if (x == nullptr || W1 == nullptr || W2 == nullptr || y == nullptr) return MHA_ERR_INVALID;
  if (std::isnan(ln_eps) || ln_eps < 0.f) return MHA_ERR_INVALID;
  const FfnPlan plan = plan_ffn(M, D, d_ff, dtype);
  if (workspace == nullptr || ws_bytes < plan.total) return MHA_ERR_WORKSPACE;
  const void* all[] = {x, W1, b1, W2, b2, gamma, beta, y};
  for (const void* p : all)
    if (p != nullptr && !aligned(p, 16)) return MHA_ERR_ALIGN;
  if (!aligned(workspace, 256)) return MHA_ERR_ALIGN;
  DevCtx ctx;
  st = device_ctx(&ctx);
  if (st != MHA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* Hb = ws + plan.off_h;
  uint8_t* F = ws + plan.off_f;
  mark(0);
  // H = max(0, x W1^T + b1)
  st = run_linear(M, d_ff, D, dtype, x, D, W1, b1, Hb, d_ff, ctx, stream, /*relu=*/true);
  if (st != MHA_OK) return st;
  mark(1);
  if (use_fused_out_ln(dtype, M, D, d_ff)) {
    // y = LayerNorm(x + H W2^T + b2) in one kernel: FFN(x) stays on chip
    MHA_NVTX_RANGE("linear2_layernorm");
    CUtensorMap tmH, tmW2;
    if (!map_2d_bf16(&tmH, Hb, d_ff, M, d_ff, 128) || !map_2d_bf16(&tmW2, W2, d_ff, D, d_ff, 256))
      return MHA_ERR_CUDA;
    const cudaError_t e = mha::launch_gemm_ln_bf16(tmH, tmW2, b2, x, gamma, beta, y, M, D, d_ff,
                                                   ln_eps, ctx, stream);
    mark(2);
    mark(3);
    return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
  }
  // F = H W2^T + b2
  st = run_linear(M, D, d_ff, dtype, Hb, d_ff, W2, b2, F, D, ctx, stream);
  if (st != MHA_OK) return st;
  mark(2);
  // y = LayerNorm(x + F)
  MHA_NVTX_RANGE("residual_layernorm");
  cudaError_t e = mha::launch_residual_layernorm(dtype, M, D, ln_eps, x, F, gamma, beta, y, ctx, stream);
  mark(3);
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}
}  // namespace

extern "C" {

int mha_layer_fwd(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype, int mask,
                  const int32_t* key_len, float ln_eps, const void* x_q, const void* x_kv,
                  const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                  const void* gamma, const void* beta, void* y, void* workspace,
                  size_t ws_bytes, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_layer_fwd");
  return layer_impl(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q, x_kv, W_qkv,
                    b_qkv, W_o, b_o, gamma, beta, y, workspace, ws_bytes, stream, nullptr);
}

int mha_layer_fwd_timed(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                        int mask, const int32_t* key_len, float ln_eps, const void* x_q,
                        const void* x_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                        const void* b_o, const void* gamma, const void* beta, void* y,
                        void* workspace, size_t ws_bytes, cudaStream_t stream,
                        const cudaEvent_t* events, int n_events) {
  MHA_NVTX_RANGE("mha_layer_fwd_timed");
  if (events == nullptr || n_events < 5) return MHA_ERR_INVALID;
  for (int i = 0; i < 5; ++i)
    if (events[i] == nullptr) return MHA_ERR_INVALID;
  return layer_impl(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q, x_kv, W_qkv,
                    b_qkv, W_o, b_o, gamma, beta, y, workspace, ws_bytes, stream, events);
}

int mha_linear_fwd(int M, int N, int K, int dtype, const void* X, int64_t ldx, const void* W,
                   const void* bias, void* Y, int64_t ldy, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_linear_fwd");
  const int st = check_linear(M, N, K, dtype, X, ldx, W, bias, Y, ldy);
  if (st != MHA_OK) return st;
  DevCtx ctx;
  const int sc = device_ctx(&ctx);
  if (sc != MHA_OK) return sc;
  return run_linear(M, N, K, dtype, X, ldx, W, bias, Y, ldy, ctx, stream);
}

int mha_linear2_fwd(int M1, int N1, const void* X1, const void* W1, const void* b1, void* Y1,
                    int M2, int N2, const void* X2, const void* W2, const void* b2, void* Y2,
                    int K, int dtype, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_linear2_fwd");
  int st = check_linear(M1, N1, K, dtype, X1, K, W1, b1, Y1, N1);
  if (st != MHA_OK) return st;
  st = check_linear(M2, N2, K, dtype, X2, K, W2, b2, Y2, N2);
  if (st != MHA_OK) return st;
  DevCtx ctx;
  const int sc = device_ctx(&ctx);
  if (sc != MHA_OK) return sc;
  return run_linear_two(M1, N1, X1, W1, b1, Y1, M2, N2, X2, W2, b2, Y2, K, dtype, ctx, stream);
}

}  // extern "C"

namespace {
int check_linear(int M, int N, int K, int dtype, const void* X, int64_t ldx, const void* W,
                 const void* bias, const void* Y, int64_t ldy) {
  if (M < 1 || N < 1 || K < 1 || !valid_dtype(dtype)) return MHA_ERR_INVALID;
  if (M > (1 << 24)) return MHA_ERR_UNSUPPORTED;  // grid.y = M / 128 (or / 64) <= 65535
  if (X == nullptr || W == nullptr || Y == nullptr) return MHA_ERR_INVALID;
  if (ldx < K || ldy < N) return MHA_ERR_INVALID;
  if (dtype == MHA_BF16) {
    if (K % 64 != 0 || N % 64 != 0) return MHA_ERR_UNSUPPORTED;
    if (ldx % 8 != 0 || ldy % 8 != 0) return MHA_ERR_ALIGN;
    if (!aligned(X, 16) || !aligned(W, 16) || !aligned(Y, 16) ||
        (bias != nullptr && !aligned(bias, 16)))
      return MHA_ERR_ALIGN;
  } else {
    if (!aligned(X, 4) || !aligned(W, 4) || !aligned(Y, 4) ||
        (bias != nullptr && !aligned(bias, 4)))
      return MHA_ERR_ALIGN;
  }
  return MHA_OK;
}
}  // namespace

extern "C" {

int mha_linear_relu_fwd(int M, int N, int K, int dtype, const void* X, int64_t ldx,
                        const void* W, const void* bias, void* Y, int64_t ldy,
                        cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_linear_relu_fwd");
  const int st = check_linear(M, N, K, dtype, X, ldx, W, bias, Y, ldy);
  if (st != MHA_OK) return st;
  DevCtx ctx;
  const int sc = device_ctx(&ctx);
  if (sc != MHA_OK) return sc;
  return run_linear(M, N, K, dtype, X, ldx, W, bias, Y, ldy, ctx, stream, /*relu=*/true);
}

int mha_ffn_workspace_size(int M, int D, int d_ff, int dtype, size_t* bytes) {
  if (bytes == nullptr) return MHA_ERR_INVALID;
  const int st = check_ffn_shape(M, D, d_ff, dtype);
  if (st != MHA_OK) return st;
  *bytes = plan_ffn(M, D, d_ff, dtype).total;
  return MHA_OK;
}

int mha_ffn_fwd(int M, int D, int d_ff, int dtype, float ln_eps, const void* x, const void* W1,
                const void* b1, const void* W2, const void* b2, const void* gamma,
                const void* beta, void* y, void* workspace, size_t ws_bytes,
                cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_ffn_fwd");
  return ffn_impl(M, D, d_ff, dtype, ln_eps, x, W1, b1, W2, b2, gamma, beta, y, workspace,
                  ws_bytes, stream, nullptr);
}

int mha_ffn_fwd_timed(int M, int D, int d_ff, int dtype, float ln_eps, const void* x,
                      const void* W1, const void* b1, const void* W2, const void* b2,
                      const void* gamma, const void* beta, void* y, void* workspace,
                      size_t ws_bytes, cudaStream_t stream, const cudaEvent_t* events,
                      int n_events) {
  MHA_NVTX_RANGE("mha_ffn_fwd_timed");
  if (events == nullptr || n_events < 4) return MHA_ERR_INVALID;
  for (int i = 0; i < 4; ++i)
    if (events[i] == nullptr) return MHA_ERR_INVALID;
  return ffn_impl(M, D, d_ff, dtype, ln_eps, x, W1, b1, W2, b2, gamma, beta, y, workspace,
                  ws_bytes, stream, events);
}

int mha_encoder_layer_workspace_size(int B, int N, int H, int D, int d_ff, int dtype,
                                     size_t* bytes) {
  if (bytes == nullptr) return MHA_ERR_INVALID;
  if (H < 1 || D < 1 || D % H != 0) return MHA_ERR_INVALID;
  int st = check_layer_shape(B, H, N, N, D, D / H, D / H, dtype);
  if (st != MHA_OK) return st;
  st = check_ffn_shape(B * N, D, d_ff, dtype);
  if (st != MHA_OK) return st;
  *bytes = plan_encoder(B, N, H, D, d_ff, dtype).total;
  return MHA_OK;
}

int mha_encoder_layer_fwd(int B, int N, int H, int D, int d_ff, int dtype, int mask,
                          const int32_t* key_len, float ln_eps, const void* x,
                          const void* W_qkv, const void* b_qkv, const void* W_o,
                          const void* b_o, const void* gamma1, const void* beta1,
                          const void* W1, const void* b1, const void* W2, const void* b2,
                          const void* gamma2, const void* beta2, void* y, void* workspace,
                          size_t ws_bytes, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_encoder_layer_fwd");
  size_t need = 0;
  int st = mha_encoder_layer_workspace_size(B, N, H, D, d_ff, dtype, &need);
  if (st != MHA_OK) return st;
  if (workspace == nullptr || ws_bytes < need) return MHA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MHA_ERR_ALIGN;
  if (y == x) return MHA_ERR_INVALID;  // x is read again by the second residual
  const EncoderPlan plan = plan_encoder(B, N, H, D, d_ff, dtype);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* h = ws + plan.off_h;
  // h = LayerNorm(x + MultiHead(x, x, x))
  st = layer_impl(B, H, N, N, D, D / H, D / H, dtype, mask, key_len, ln_eps, x, nullptr, W_qkv,
                  b_qkv, W_o, b_o, gamma1, beta1, h, ws + plan.off_ws, need - plan.off_ws,
                  stream, nullptr);
  if (st != MHA_OK) return st;
  // y = LayerNorm(h + FFN(h))
  return ffn_impl(B * N, D, d_ff, dtype, ln_eps, h, W1, b1, W2, b2, gamma2, beta2, y,
                  ws + plan.off_ws, need - plan.off_ws, stream, nullptr);
}

int mha_residual_layernorm_fwd(int M, int D, int dtype, float eps, const void* x, const void* a,
                               const void* gamma, const void* beta, void* y,
                               cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_residual_layernorm_fwd");
  if (M < 1 || D < 1 || !valid_dtype(dtype)) return MHA_ERR_INVALID;
  if (x == nullptr || a == nullptr || y == nullptr) return MHA_ERR_INVALID;
  if (std::isnan(eps) || eps < 0.f) return MHA_ERR_INVALID;
  if (D % 8 != 0 || D > 2048) return MHA_ERR_UNSUPPORTED;
  const void* all[] = {x, a, gamma, beta, y};
  for (const void* p : all)
    if (p != nullptr && !aligned(p, 16)) return MHA_ERR_ALIGN;
  DevCtx ctx;
  const int st = device_ctx(&ctx);
  if (st != MHA_OK) return st;
  cudaError_t e = mha::launch_residual_layernorm(dtype, M, D, eps, x, a, gamma, beta, y, ctx, stream);
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

int mha_out_proj_layernorm_fwd(int M, int D, int K, int dtype, float eps, const void* C,
                               const void* W_o, const void* b_o, const void* x,
                               const void* gamma, const void* beta, void* y,
                               cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_out_proj_layernorm_fwd");
  if (M < 1 || D < 1 || K < 1 || !valid_dtype(dtype)) return MHA_ERR_INVALID;
  if (C == nullptr || W_o == nullptr || x == nullptr || y == nullptr) return MHA_ERR_INVALID;
  if (std::isnan(eps) || eps < 0.f) return MHA_ERR_INVALID;
  if (D % 8 != 0 || D > 2048 || M > (1 << 24)) return MHA_ERR_UNSUPPORTED;
  if (dtype == MHA_BF16 && (D % 64 != 0 || K % 64 != 0)) return MHA_ERR_UNSUPPORTED;
  const void* all[] = {C, W_o, b_o, x, gamma, beta, y};
  for (const void* p : all)
    if (p != nullptr && !aligned(p, 16)) return MHA_ERR_ALIGN;
  DevCtx ctx;
  int st = device_ctx(&ctx);
  if (st != MHA_OK) return st;
  if (dtype == MHA_BF16 && mha::gemm_ln_bf16_supported(D, K)) {
    CUtensorMap tmC, tmWo;
    if (!map_2d_bf16(&tmC, C, K, M, K, 128) || !map_2d_bf16(&tmWo, W_o, K, D, K, 256))
      return MHA_ERR_CUDA;
    const cudaError_t e = mha::launch_gemm_ln_bf16(tmC, tmWo, b_o, x, gamma, beta, y, M, D, K,
                                                   eps, ctx, stream);
    return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
  }
  // two launches: the projection into y, then the LayerNorm reads it back in place (each row
  // is read whole before it is written)
  st = run_linear(M, D, K, dtype, C, K, W_o, b_o, y, D, ctx, stream);
  if (st != MHA_OK) return st;
  const cudaError_t e =
      mha::launch_residual_layernorm(dtype, M, D, eps, x, y, gamma, beta, y, ctx, stream);
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

int mha_set_deterministic(int on) {
  if (on != 0 && on != 1) return MHA_ERR_INVALID;
  g_deterministic.store(on, std::memory_order_relaxed);
  return MHA_OK;
}

int mha_get_deterministic(void) { return g_deterministic.load(std::memory_order_relaxed); }

int mha_debug_last_device_status(cudaStream_t stream) {
  DevCtx ctx;
  const int st = device_ctx(&ctx);
  if (st != MHA_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MHA_ERR_CUDA;
  int h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, ctx.status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MHA_ERR_CUDA;
  const int zero[4] = {0, 0, 0, 0};
  if (cudaMemcpy(ctx.status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return MHA_ERR_CUDA;
  return h[0];
}

int mha_debug_wait_selftest(int64_t timeout_ns, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_debug_wait_selftest");
  DevCtx ctx;
  const int st = device_ctx(&ctx);
  if (st != MHA_OK) return st;
  if (timeout_ns < 1000) timeout_ns = 1000;
  if (timeout_ns > 1000000000) timeout_ns = 1000000000;
  ctx.timeout_ns = static_cast<uint64_t>(timeout_ns);
  return mha::launch_wait_selftest(ctx, stream) == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // extern "C"

// ==================================================================== sublayer backward
namespace {

// Scratch of one sublayer backward (offsets into the caller's workspace, 256-byte aligned).
// Forward intermediates: the projections (self: Q|K|V interleaved per token; cross: Q, then
// K|V), the head-concat C, the W^O output A, the log-sum-exp; then the gradients dr, dC and
// the projections' gradients (same layouts), the transposed weights of the data-gradient
// GEMMs, the fp32 partial column sums, and for the weight-gradient GEMMs either (bf16) the
// fp32 split-K accumulator -- their operands are read in place -- or (fp32) the transposed
// token-axis operands, padded to a multiple of 64 tokens.  mha_layer_fwd_train fills the
// forward part; mha_layer_bwd_saved reads it.
struct LayerBwdPlan {
  int Mq, Mk, Mq_pad, Mk_pad, nqk, nv, ld_q, ld_kv;  // ld_q: row pitch of the Q projection
  size_t off_q, off_kv, off_c, off_a, off_lse, off_dvec, off_stats, off_part, off_dr, off_dc,
      off_dq, off_dkv, off_wot, off_wqt, off_wkvt, off_drt, off_ct, off_dqt, off_dkvt, off_xqt,
      off_xkvt, off_wacc, total;
};

LayerBwdPlan plan_layer_bwd(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                            bool self) {
  const size_t es = elem_size(dtype);
  LayerBwdPlan p;
  p.Mq = B * Nq;
  p.Mk = B * Nk;
  p.Mq_pad = (p.Mq + 63) / 64 * 64;
  p.Mk_pad = (p.Mk + 63) / 64 * 64;
  p.nqk = H * d_k;
  p.nv = H * d_v;
  p.ld_q = self ? 2 * p.nqk + p.nv : p.nqk;
  p.ld_kv = self ? 2 * p.nqk + p.nv : p.nqk + p.nv;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += round_up(bytes, 256);
    return at;
  };
  const int nchunk = mha::bwd_row_chunks(p.Mq > p.Mk ? p.Mq : p.Mk);
  const int part_cols = (3 * D > 2 * p.nqk + p.nv) ? 3 * D : 2 * p.nqk + p.nv;
  p.off_q = take(static_cast<size_t>(p.Mq) * p.ld_q * es);
  p.off_kv = self ? p.off_q : take(static_cast<size_t>(p.Mk) * p.ld_kv * es);
  p.off_c = take(static_cast<size_t>(p.Mq) * p.nv * es);
  p.off_a = take(static_cast<size_t>(p.Mq) * D * es);
  p.off_lse = take(static_cast<size_t>(B) * H * Nq * 4);
  p.off_dvec = take(mha::sdpa_bwd_scratch_bytes(B, H, Nq, dtype));
  p.off_stats = take(static_cast<size_t>(p.Mq) * 8);
  p.off_part = take(static_cast<size_t>(nchunk) * part_cols * 4);
  p.off_dr = take(static_cast<size_t>(p.Mq) * D * es);
  p.off_dc = take(static_cast<size_t>(p.Mq) * p.nv * es);
  p.off_dq = take(static_cast<size_t>(p.Mq) * p.ld_q * es);
  p.off_dkv = self ? p.off_dq : take(static_cast<size_t>(p.Mk) * p.ld_kv * es);
  p.off_wot = take(static_cast<size_t>(p.nv) * D * es);
  p.off_wqt = take(static_cast<size_t>(D) * p.ld_q * es);
  p.off_wkvt = self ? p.off_wqt : take(static_cast<size_t>(D) * p.ld_kv * es);
  // transposed activations for the fp32 weight gradients (bf16 reads them MN-major in place)
  const size_t tes = dtype == MHA_BF16 ? 0 : es;
  p.off_drt = take(static_cast<size_t>(D) * p.Mq_pad * tes);
  p.off_ct = take(static_cast<size_t>(p.nv) * p.Mq_pad * tes);
  p.off_dqt = take(static_cast<size_t>(p.ld_q) * p.Mq_pad * tes);
  p.off_dkvt = self ? p.off_dqt : take(static_cast<size_t>(p.ld_kv) * p.Mk_pad * tes);
  p.off_xqt = take(static_cast<size_t>(D) * p.Mq_pad * tes);
  p.off_xkvt = self ? p.off_xqt : take(static_cast<size_t>(D) * p.Mk_pad * tes);
  // fp32 accumulator of the split-K weight-gradient GEMMs (the largest dW)
  const size_t wmax = static_cast<size_t>(D) *
                      std::max(std::max(p.ld_q, p.ld_kv), std::max(p.nv, p.nqk + p.nv));
  p.off_wacc = take(dtype == MHA_BF16 ? wmax * 4 : 0);
  p.total = o;
  return p;
}

// phase: kLayerBwdFull (forward recomputed, then the backward), kLayerFwdTrain (the forward
// alone, y written and the activations the backward needs left in the workspace),
// kLayerBwdSaved (the backward from those saved activations)
enum { kLayerBwdFull = 0, kLayerFwdTrain = 1, kLayerBwdSaved = 2 };

int layer_bwd_impl(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype, int mask,
                   const int32_t* key_len, float ln_eps, const void* x_q, const void* x_kv,
                   const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                   const void* gamma, const void* dy, void* dx_q, void* dx_kv, void* dW_qkv,
                   void* db_qkv, void* dW_o, void* db_o, void* dgamma, void* dbeta,
                   void* workspace, size_t ws_bytes, cudaStream_t stream,
                   int phase = kLayerBwdFull, const void* beta = nullptr, void* y = nullptr) {
  int st = check_layer_shape(B, H, Nq, Nk, D, d_k, d_v, dtype);
  if (st != MHA_OK) return st;
  if (mask < MHA_MASK_NONE || mask > MHA_MASK_KEY_PADDING) return MHA_ERR_INVALID;
  const bool self = (x_kv == nullptr);
  if ((self || mask == MHA_MASK_CAUSAL) && Nq != Nk) return MHA_ERR_INVALID;
  if (mask == MHA_MASK_KEY_PADDING && key_len == nullptr) return MHA_ERR_INVALID;
  if (phase == kLayerFwdTrain) {
    if (x_q == nullptr || W_qkv == nullptr || W_o == nullptr || y == nullptr)
      return MHA_ERR_INVALID;
  } else {
    const void* need[] = {x_q, W_qkv, W_o, dy, dx_q, dW_qkv, db_qkv, dW_o, db_o, dgamma, dbeta};
    for (const void* q : need)
      if (q == nullptr) return MHA_ERR_INVALID;
    if (!self && dx_kv == nullptr) return MHA_ERR_INVALID;
  }
  if (std::isnan(ln_eps) || ln_eps < 0.f) return MHA_ERR_INVALID;
  const LayerBwdPlan pl = plan_layer_bwd(B, H, Nq, Nk, D, d_k, d_v, dtype, self);
  if (workspace == nullptr || ws_bytes < pl.total) return MHA_ERR_WORKSPACE;
  const void* all[] = {x_q,  x_kv,  W_qkv, b_qkv, W_o,    b_o,  gamma,  dy,   dx_q, dx_kv,
                       dW_qkv, db_qkv, dW_o, db_o, dgamma, dbeta, workspace, beta, y};
  for (const void* q : all)
    if (q != nullptr && !aligned(q, 16)) return MHA_ERR_ALIGN;
  if (key_len != nullptr && !aligned(key_len, 4)) return MHA_ERR_ALIGN;
  if (!aligned(workspace, 256)) return MHA_ERR_ALIGN;
  DevCtx ctx;
  st = device_ctx(&ctx);
  if (st != MHA_OK) return st;

  const size_t es = elem_size(dtype);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto W = [&](size_t off) { return static_cast<void*>(ws + off); };
  const uint8_t* Wb = static_cast<const uint8_t*>(W_qkv);
  const uint8_t* bq = static_cast<const uint8_t*>(b_qkv);
  const int Mq = pl.Mq, Mk = pl.Mk, nqk = pl.nqk, nv = pl.nv;
  const void* src_kv = self ? x_q : x_kv;
  auto ok = [](cudaError_t e) { return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA; };
#define MHA_TRY(call)          \
  do {                         \
    const int s_ = (call);     \
    if (s_ != MHA_OK) return s_; \
  } while (0)

  // ---- forward again, keeping what the backward needs
  mha::SdpaArgs a;
  a.B = B; a.H = H; a.Nq = Nq; a.Nk = Nk; a.d_k = d_k; a.d_v = d_v;
  a.mask = mask;
  a.key_len = (mask == MHA_MASK_KEY_PADDING) ? key_len : nullptr;
  a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k)));
  uint8_t* qbuf = ws + pl.off_q;
  uint8_t* kvbuf = ws + pl.off_kv;
  const bool recompute = phase != kLayerBwdSaved;
  if (self) {
    if (recompute)
      MHA_TRY(run_linear(Mq, pl.ld_q, D, dtype, x_q, D, W_qkv, b_qkv, qbuf, pl.ld_q, ctx,
                         stream));
    a.Q = qbuf;
    a.K = qbuf + nqk * es;
    a.V = qbuf + 2 * nqk * es;
  } else {
    if (recompute) {
      MHA_TRY(run_linear_two(Mq, nqk, x_q, W_qkv, b_qkv, qbuf, Mk, pl.ld_kv, x_kv,
                             Wb + static_cast<size_t>(nqk) * D * es,
                             bq ? bq + nqk * es : nullptr, kvbuf, D, dtype, ctx, stream));
    }
    a.Q = qbuf;
    a.K = kvbuf;
    a.V = kvbuf + nqk * es;
  }
  const int64_t sq[4] = {static_cast<int64_t>(Nq) * pl.ld_q, d_k, pl.ld_q, 1};
  const int64_t sk[4] = {static_cast<int64_t>(Nk) * pl.ld_kv, d_k, pl.ld_kv, 1};
  const int64_t sv[4] = {static_cast<int64_t>(Nk) * pl.ld_kv, d_v, pl.ld_kv, 1};
  const int64_t so[4] = {static_cast<int64_t>(Nq) * nv, d_v, nv, 1};
  for (int i = 0; i < 4; ++i) {
    a.sq[i] = sq[i];
    a.sk[i] = sk[i];
    a.sv[i] = sv[i];
    a.so[i] = so[i];
  }
  a.O = W(pl.off_c);
  a.lse = static_cast<float*>(W(pl.off_lse));
  if (phase == kLayerFwdTrain && use_fused_out_ln(dtype, Mq, D, nv)) {
    // y exactly as mha_layer_fwd computes it (W^O and LayerNorm in one kernel), which also
    // keeps the projection output A in bf16 for the backward
    MHA_TRY(run_sdpa(a, dtype, ctx, stream));
    CUtensorMap tmC, tmWo;
    if (!map_2d_bf16(&tmC, W(pl.off_c), nv, Mq, nv, 128) ||
        !map_2d_bf16(&tmWo, W_o, nv, D, nv, 256))
      return MHA_ERR_CUDA;
    return ok(mha::launch_gemm_ln_bf16(tmC, tmWo, b_o, x_q, gamma, beta, y, Mq, D, nv, ln_eps,
                                       ctx, stream, W(pl.off_a)));
  }
  if (phase != kLayerBwdSaved) {
    MHA_TRY(run_sdpa(a, dtype, ctx, stream));
    MHA_TRY(run_linear(Mq, D, nv, dtype, W(pl.off_c), nv, W_o, b_o, W(pl.off_a), D, ctx,
                       stream));
  }
  if (phase == kLayerFwdTrain)
    return ok(mha::launch_residual_layernorm(dtype, Mq, D, ln_eps, x_q, W(pl.off_a), gamma, beta,
                                             y, ctx, stream));

  // ---- residual + LayerNorm backward: dr; dgamma, dbeta, db_o from per-chunk partials
  float* part = static_cast<float*>(W(pl.off_part));
  MHA_TRY(ok(mha::launch_layernorm_bwd(dtype, Mq, D, ln_eps, x_q, W(pl.off_a), gamma, dy,
                                       W(pl.off_dr), static_cast<float2*>(W(pl.off_stats)),
                                       part, stream)));
  const int nch_q = mha::bwd_row_chunks(Mq);
  MHA_TRY(ok(mha::launch_reduce_partials3(dtype, part, nch_q, 3 * D, D, D, 3, dgamma, dbeta,
                                          db_o, stream)));

  // ---- W^O: dC = dr W^O (via W^O^T), dW^O = dr^T C
  MHA_TRY(ok(mha::launch_transpose(dtype, W_o, nv, D, nv, W(pl.off_wot), D, D, stream)));
  MHA_TRY(run_linear(Mq, nv, D, dtype, W(pl.off_dr), D, W(pl.off_wot), nullptr, W(pl.off_dc),
                     nv, ctx, stream));
  float* wacc = static_cast<float*>(W(pl.off_wacc));
  MHA_TRY(run_linear_wgrad(D, nv, Mq, dtype, W(pl.off_dr), D, W(pl.off_c), nv, dW_o, nv, wacc,
                           W(pl.off_drt), W(pl.off_ct), pl.Mq_pad, ctx, stream));

  // ---- attention backward: dQ, dK, dV into buffers laid out like the projections
  mha::SdpaBwdArgs g;
  g.B = B; g.H = H; g.Nq = Nq; g.Nk = Nk; g.d_k = d_k; g.d_v = d_v;
  g.mask = mask;
  g.window = 0;
  g.key_len = a.key_len;
  g.scale = a.scale;
  g.Q = a.Q; g.K = a.K; g.V = a.V; g.O = a.O; g.dO = W(pl.off_dc);
  g.lse = a.lse;
  g.Dv = static_cast<float*>(W(pl.off_dvec));
  uint8_t* dqbuf = ws + pl.off_dq;
  uint8_t* dkvbuf = ws + pl.off_dkv;
  g.dQ = dqbuf;
  g.dK = self ? dqbuf + nqk * es : dkvbuf;
  g.dV = self ? dqbuf + 2 * nqk * es : dkvbuf + nqk * es;
  const int64_t* strs[8] = {sq, sk, sv, so, so, sq, sk, sv};
  for (int t = 0; t < 8; ++t)
    for (int i = 0; i < 4; ++i) g.st[t][i] = strs[t][i];
  MHA_TRY(run_sdpa_bwd(g, dtype, ctx, stream));

  // ---- projections: dx = dProj W (+ dr on the query side), dW = dProj^T x, db = colsum
  if (self) {
    MHA_TRY(ok(mha::launch_transpose(dtype, W_qkv, D, pl.ld_q, D, W(pl.off_wqt), pl.ld_q,
                                     pl.ld_q, stream)));
    MHA_TRY(run_linear(Mq, D, pl.ld_q, dtype, dqbuf, pl.ld_q, W(pl.off_wqt), nullptr, dx_q, D,
                       ctx, stream, false, W(pl.off_dr)));
    MHA_TRY(run_linear_wgrad(pl.ld_q, D, Mq, dtype, dqbuf, pl.ld_q, x_q, D, dW_qkv, D, wacc,
                             W(pl.off_dqt), W(pl.off_xqt), pl.Mq_pad, ctx, stream));
    MHA_TRY(ok(mha::launch_colsum_partials(dtype, dqbuf, pl.ld_q, Mq, pl.ld_q, part, stream)));
    MHA_TRY(ok(mha::launch_reduce_partials(dtype, part, nch_q, pl.ld_q, pl.ld_q, db_qkv,
                                           stream)));
  } else {
    uint8_t* dWb = static_cast<uint8_t*>(dW_qkv);
    uint8_t* dbb = static_cast<uint8_t*>(db_qkv);
    // query side
    MHA_TRY(ok(mha::launch_transpose(dtype, W_qkv, D, nqk, D, W(pl.off_wqt), nqk, nqk,
                                     stream)));
    MHA_TRY(run_linear(Mq, D, nqk, dtype, dqbuf, nqk, W(pl.off_wqt), nullptr, dx_q, D, ctx,
                       stream, false, W(pl.off_dr)));
    MHA_TRY(run_linear_wgrad(nqk, D, Mq, dtype, dqbuf, nqk, x_q, D, dWb, D, wacc,
                             W(pl.off_dqt), W(pl.off_xqt), pl.Mq_pad, ctx, stream));
    MHA_TRY(ok(mha::launch_colsum_partials(dtype, dqbuf, nqk, Mq, nqk, part, stream)));
    MHA_TRY(ok(mha::launch_reduce_partials(dtype, part, nch_q, nqk, nqk, dbb, stream)));
    // key/value side
    const int nch_k = mha::bwd_row_chunks(Mk);
    MHA_TRY(ok(mha::launch_transpose(dtype, Wb + static_cast<size_t>(nqk) * D * es, D,
                                     pl.ld_kv, D, W(pl.off_wkvt), pl.ld_kv, pl.ld_kv, stream)));
    MHA_TRY(run_linear(Mk, D, pl.ld_kv, dtype, dkvbuf, pl.ld_kv, W(pl.off_wkvt), nullptr, dx_kv,
                       D, ctx, stream));
    MHA_TRY(run_linear_wgrad(pl.ld_kv, D, Mk, dtype, dkvbuf, pl.ld_kv, src_kv, D,
                             dWb + static_cast<size_t>(nqk) * D * es, D, wacc, W(pl.off_dkvt),
                             W(pl.off_xkvt), pl.Mk_pad, ctx, stream));
    MHA_TRY(ok(mha::launch_colsum_partials(dtype, dkvbuf, pl.ld_kv, Mk, pl.ld_kv, part,
                                           stream)));
    MHA_TRY(ok(mha::launch_reduce_partials(dtype, part, nch_k, pl.ld_kv, pl.ld_kv,
                                           dbb + nqk * es, stream)));
  }
#undef MHA_TRY
  return MHA_OK;
}

}  // namespace

extern "C" {

int mha_layer_bwd_workspace_size(int B, int H, int Nq, int Nk, int D, int d_k, int d_v,
                                 int dtype, int self_attention, size_t* bytes) {
  if (bytes == nullptr) return MHA_ERR_INVALID;
  const int st = check_layer_shape(B, H, Nq, Nk, D, d_k, d_v, dtype);
  if (st != MHA_OK) return st;
  if (self_attention && Nq != Nk) return MHA_ERR_INVALID;
  *bytes = plan_layer_bwd(B, H, Nq, Nk, D, d_k, d_v, dtype, self_attention != 0).total;
  return MHA_OK;
}

int mha_layer_bwd(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype, int mask,
                  const int32_t* key_len, float ln_eps, const void* x_q, const void* x_kv,
                  const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                  const void* gamma, const void* beta, const void* dy, void* dx_q, void* dx_kv,
                  void* dW_qkv, void* db_qkv, void* dW_o, void* db_o, void* dgamma, void* dbeta,
                  void* workspace, size_t ws_bytes, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_layer_bwd");
  (void)beta;  // the output shift does not enter any gradient
  return layer_bwd_impl(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q, x_kv,
                        W_qkv, b_qkv, W_o, b_o, gamma, dy, dx_q, dx_kv, dW_qkv, db_qkv, dW_o,
                        db_o, dgamma, dbeta, workspace, ws_bytes, stream);
}

int mha_layer_fwd_train(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                        int mask, const int32_t* key_len, float ln_eps, const void* x_q,
                        const void* x_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                        const void* b_o, const void* gamma, const void* beta, void* y,
                        void* workspace, size_t ws_bytes, cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_layer_fwd_train");
  return layer_bwd_impl(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q, x_kv,
                        W_qkv, b_qkv, W_o, b_o, gamma, nullptr, nullptr, nullptr, nullptr,
                        nullptr, nullptr, nullptr, nullptr, nullptr, workspace, ws_bytes, stream,
                        kLayerFwdTrain, beta, y);
}

int mha_layer_bwd_saved(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                        int mask, const int32_t* key_len, float ln_eps, const void* x_q,
                        const void* x_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                        const void* b_o, const void* gamma, const void* beta, const void* dy,
                        void* dx_q, void* dx_kv, void* dW_qkv, void* db_qkv, void* dW_o,
                        void* db_o, void* dgamma, void* dbeta, void* workspace, size_t ws_bytes,
                        cudaStream_t stream) {
  MHA_NVTX_RANGE("mha_layer_bwd_saved");
  (void)beta;
  return layer_bwd_impl(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q, x_kv,
                        W_qkv, b_qkv, W_o, b_o, gamma, dy, dx_q, dx_kv, dW_qkv, db_qkv, dW_o,
                        db_o, dgamma, dbeta, workspace, ws_bytes, stream, kLayerBwdSaved);
}

}  // extern "C"
