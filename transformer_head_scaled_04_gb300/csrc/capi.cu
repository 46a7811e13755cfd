// capi.cu -- the C ABI of libmha.so (declared in include/mha.h): argument validation, TMA
// descriptor encoding, workspace carving and launch sequencing.  No device memory is
// allocated here; the only device state is the 4-int error word below.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "mha.h"
#include "device_common.cuh"
#include "launchers.h"

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

// [B, H, N, 64] bf16 tensor with element strides st = {b, h, n, d=1}; box {64, 128, 1, 1}.
bool map_bhnd_bf16(CUtensorMap* m, const void* base, int B, int H, int N, const int64_t* st) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2,
                           static_cast<cuuint64_t>(st[1]) * 2,
                           static_cast<cuuint64_t>(st[0]) * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------------ step launchers
int run_linear(int M, int N, int K, int dtype, const void* X, int64_t ldx, const void* W,
               const void* bias, void* Y, int64_t ldy, const DevCtx& ctx, cudaStream_t s,
               bool relu = false) {
  cudaError_t e;
  if (dtype == MHA_BF16) {
    const int64_t tiles256 = ((M + 127) / 128) * static_cast<int64_t>((N + 255) / 256);
    const int bn = (tiles256 >= ctx.num_sms) ? 256 : 128;
    CUtensorMap tmX, tmW;
    if (!map_2d_bf16(&tmX, X, K, M, ldx, 128) || !map_2d_bf16(&tmW, W, K, N, K, bn))
      return MHA_ERR_CUDA;
    e = mha::launch_gemm_bf16(tmX, tmW, bn, relu, bias, Y, M, N, K, ldy, ctx, s);
  } else {
    e = mha::launch_gemm_f32(static_cast<const float*>(X), ldx, static_cast<const float*>(W),
                             static_cast<const float*>(bias), relu, static_cast<float*>(Y), ldy,
                             M, N, K, s);
  }
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

int run_sdpa(const mha::SdpaArgs& a, int dtype, const DevCtx& ctx, cudaStream_t s) {
  cudaError_t e;
  if (dtype == MHA_BF16) {
    CUtensorMap tq, tk, tv;
    if (!map_bhnd_bf16(&tq, a.Q, a.B, a.H, a.Nq, a.sq) ||
        !map_bhnd_bf16(&tk, a.K, a.B, a.H, a.Nk, a.sk) ||
        !map_bhnd_bf16(&tv, a.V, a.B, a.H, a.Nk, a.sv))
      return MHA_ERR_CUDA;
    e = mha::launch_sdpa_bf16(tq, tk, tv, a, ctx, s);
  } else {
    e = mha::launch_sdpa_f32(a, s);
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
  if (mask < MHA_MASK_NONE || mask > MHA_MASK_KEY_PADDING || lse == nullptr)
    return MHA_ERR_INVALID;
  return sdpa_entry(B, H, Nq, Nk, d_k, d_v, dtype, mask, key_len, 0, scale, Q, K, V, O, strides,
                    stream, lse);
}

int mha_sdpa_bwd_workspace_size(int B, int H, int Nq, int dtype, size_t* bytes) {
  if (bytes == nullptr || B < 1 || H < 1 || Nq < 1 || !valid_dtype(dtype))
    return MHA_ERR_INVALID;
  *bytes = round_up(static_cast<size_t>(B) * H * Nq * sizeof(float), 256);  // D = rowsum(dO O)
  return MHA_OK;
}

int mha_sdpa_bwd(int B, int H, int Nq, int Nk, int d_k, int d_v, int dtype, int mask,
                 const int32_t* key_len, float scale, const void* Q, const void* K,
                 const void* V, const void* O, const void* dO, const float* lse, void* dQ,
                 void* dK, void* dV, const int64_t* strides, void* workspace, size_t ws_bytes,
                 cudaStream_t stream) {
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
  cudaError_t e = mha::launch_sdpa_bwd_rowdot(a, dtype, stream);
  if (e != cudaSuccess) return MHA_ERR_CUDA;
  if (dtype == MHA_BF16) {
    CUtensorMap tq, tk, tv, tg;
    if (!map_bhnd_bf16(&tq, Q, B, H, Nq, a.st[0]) || !map_bhnd_bf16(&tk, K, B, H, Nk, a.st[1]) ||
        !map_bhnd_bf16(&tv, V, B, H, Nk, a.st[2]) || !map_bhnd_bf16(&tg, dO, B, H, Nq, a.st[4]))
      return MHA_ERR_CUDA;
    e = mha::launch_sdpa_bwd_bf16(tq, tk, tv, tg, a, ctx, stream);
  } else {
    e = mha::launch_sdpa_bwd_f32(a, stream);
  }
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

int mha_sdpa_window_fwd(int B, int H, int N, int d_k, int d_v, int dtype, int window,
                        float scale, const void* Q, const void* K, const void* V, void* O,
                        const int64_t* strides, cudaStream_t stream) {
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
  if (workspace == nullptr || ws_bytes < plan.total) return MHA_ERR_WORKSPACE;
  const void* all[] = {x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, y, workspace};
  for (const void* p : all)
    if (p != nullptr && !aligned(p, 16)) return MHA_ERR_ALIGN;
  if (key_len != nullptr && !aligned(key_len, 4)) return MHA_ERR_ALIGN;
  if (!aligned(workspace, 256)) return MHA_ERR_ALIGN;

  DevCtx ctx;
  st = device_ctx(&ctx);
  if (st != MHA_OK) return st;

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
    st = run_linear(Mq, nqk, D, dtype, x_q, D, W_qkv, b_qkv, qb, nqk, ctx, stream);
    if (st != MHA_OK) return st;
    const int ldkv = nqk + nv;
    st = run_linear(Mk, ldkv, D, dtype, x_kv, D, Wb + static_cast<size_t>(nqk) * D * es,
                    bq ? bq + nqk * es : nullptr, kvb, ldkv, ctx, stream);
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
  // A = C W_o^T + b_o
  uint8_t* A = ws + plan.off_a;
  mark(2);
  st = run_linear(Mq, D, nv, dtype, C, nv, W_o, b_o, A, D, ctx, stream);
  if (st != MHA_OK) return st;
  // y = LayerNorm(x_q + A)
  mark(3);
  cudaError_t e =
      mha::launch_residual_layernorm(dtype, Mq, D, ln_eps, x_q, A, gamma, beta, y, stream);
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
  // F = H W2^T + b2
  st = run_linear(M, D, d_ff, dtype, Hb, d_ff, W2, b2, F, D, ctx, stream);
  if (st != MHA_OK) return st;
  mark(2);
  // y = LayerNorm(x + F)
  cudaError_t e = mha::launch_residual_layernorm(dtype, M, D, ln_eps, x, F, gamma, beta, y, stream);
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
  return layer_impl(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q, x_kv, W_qkv,
                    b_qkv, W_o, b_o, gamma, beta, y, workspace, ws_bytes, stream, nullptr);
}

int mha_layer_fwd_timed(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                        int mask, const int32_t* key_len, float ln_eps, const void* x_q,
                        const void* x_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                        const void* b_o, const void* gamma, const void* beta, void* y,
                        void* workspace, size_t ws_bytes, cudaStream_t stream,
                        const cudaEvent_t* events, int n_events) {
  if (events == nullptr || n_events < 5) return MHA_ERR_INVALID;
  for (int i = 0; i < 5; ++i)
    if (events[i] == nullptr) return MHA_ERR_INVALID;
  return layer_impl(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q, x_kv, W_qkv,
                    b_qkv, W_o, b_o, gamma, beta, y, workspace, ws_bytes, stream, events);
}

int mha_linear_fwd(int M, int N, int K, int dtype, const void* X, int64_t ldx, const void* W,
                   const void* bias, void* Y, int64_t ldy, cudaStream_t stream) {
  const int st = check_linear(M, N, K, dtype, X, ldx, W, bias, Y, ldy);
  if (st != MHA_OK) return st;
  DevCtx ctx;
  const int sc = device_ctx(&ctx);
  if (sc != MHA_OK) return sc;
  return run_linear(M, N, K, dtype, X, ldx, W, bias, Y, ldy, ctx, stream);
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
  return ffn_impl(M, D, d_ff, dtype, ln_eps, x, W1, b1, W2, b2, gamma, beta, y, workspace,
                  ws_bytes, stream, nullptr);
}

int mha_ffn_fwd_timed(int M, int D, int d_ff, int dtype, float ln_eps, const void* x,
                      const void* W1, const void* b1, const void* W2, const void* b2,
                      const void* gamma, const void* beta, void* y, void* workspace,
                      size_t ws_bytes, cudaStream_t stream, const cudaEvent_t* events,
                      int n_events) {
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
  cudaError_t e = mha::launch_residual_layernorm(dtype, M, D, eps, x, a, gamma, beta, y, stream);
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

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
  DevCtx ctx;
  const int st = device_ctx(&ctx);
  if (st != MHA_OK) return st;
  if (timeout_ns < 1000) timeout_ns = 1000;
  if (timeout_ns > 1000000000) timeout_ns = 1000000000;
  ctx.timeout_ns = static_cast<uint64_t>(timeout_ns);
  return mha::launch_wait_selftest(ctx, stream) == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // extern "C"
