// layer_noalloc.cu -- mha_layer_fwd_noalloc: the sublayer forward for callers that cannot
// hand the library a workspace.
//
// mha_layer_fwd needs a caller-provided device workspace for its intermediates (the
// projected Q/K/V, the head-concat buffer and the W^O output).  Some callers have no way to
// obtain one: a plugin running inside a host framework that owns every byte of device memory
// and forbids allocations from its enqueue callback, or code on a latency-critical path
// where cudaMalloc's implicit device synchronisation is not acceptable.  For them this file
// keeps a fixed scratch area in the library itself, in a file-scope __device__ array that the
// CUDA runtime places in device memory when it loads this module on a device.  It stays
// there, on every GPU that loads the library, until the process exits.
//
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.  The entry point runs
// every check mha_layer_fwd makes (the current device's included), then looks up the
// array's device address (once per device) and forwards to mha_layer_fwd.
#include <cuda_runtime.h>

#include <mutex>

#include "launchers.h"
#include "mha.h"

// Largest workspace the no-alloc entry point can serve: 48 MiB.  Self-attention at
// d_model 512 (h = 8, d_k = d_v = 64) keeps 5120 bytes per token in bf16 and 10240 in fp32,
// so one call serves up to 9830 tokens (B * n) in bf16 and 4915 in fp32; cross-attention
// keeps 3072 bytes per query token and 2048 per key token in bf16 (twice that in fp32).
static constexpr size_t kLayerScratchBytes = static_cast<size_t>(48) << 20;

// The scratch itself.  Host code must not use this name as a pointer: on the host it is only
// a stand-in for the symbol, so the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_layer_scratch[kLayerScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_layer_scratch on the current device, looked up on the first call per
// device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MHA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layer_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MHA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MHA_OK;
}

}  // namespace

extern "C" int mha_layer_fwd_noalloc(int B, int H, int Nq, int Nk, int D, int d_k, int d_v,
                                     int dtype, int mask, const int32_t* key_len, float ln_eps,
                                     const void* x_q, const void* x_kv, const void* W_qkv,
                                     const void* b_qkv, const void* W_o, const void* b_o,
                                     const void* gamma, const void* beta, void* y,
                                     cudaStream_t stream) {
  // The same checks, in the same order, as mha_layer_fwd with a 48 MiB workspace, so this
  // entry point returns the codes that one would (MHA_ERR_WORKSPACE beyond 48 MiB,
  // MHA_ERR_UNSUPPORTED on a device other than sm_103) before it touches the scratch symbol.
  mha::DevCtx ctx;
  int st = mha::check_layer_call(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q,
                                 x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, y, nullptr,
                                 kLayerScratchBytes, true, &ctx);
  if (st != MHA_OK) return st;
  void* ws = nullptr;
  st = scratch_address(&ws);
  if (st != MHA_OK) return st;
  // Every region of the workspace is fully written before it is read, so the previous
  // call's contents need no clearing.
  return mha_layer_fwd(B, H, Nq, Nk, D, d_k, d_v, dtype, mask, key_len, ln_eps, x_q, x_kv,
                       W_qkv, b_qkv, W_o, b_o, gamma, beta, y, ws, kLayerScratchBytes, stream);
}
