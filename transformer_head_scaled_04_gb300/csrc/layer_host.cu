// layer_host.cu -- mha_layer_fwd_host: the self-attention sublayer ("Attention Is All You Need",
// lettle.cn translation, 3.1 and 3.2.2) for a caller whose x and y live in host memory.
//
// The batch is cut into slices of whole sequences.  Slice i's x goes to the device on a copy
// stream while slice i-1 is computed on the caller's stream and slice i-2's y comes back on a
// second copy stream; two device buffers each for x and y (in the caller's workspace) carry
// the slices, so a copy never overtakes the computation that still reads or writes its buffer.
// The two copy streams and the events that order the three streams are created once per device
// on the first call and kept until the process exits; the device memory is the caller's.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "launchers.h"
#include "mha.h"

namespace {

constexpr int kMaxDevices = 64;

struct Pipe {
  bool init = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t entry = nullptr;
  cudaEvent_t in_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
};
Pipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu[kMaxDevices];

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct HostPlan {
  int Bc = 0, chunks = 0;
  size_t slice_bytes = 0;  // x (or y) of one slice
  size_t off_x[2] = {}, off_y[2] = {}, off_ws = 0, layer_ws = 0, total = 0;
};

int plan_host(int B, int H, int N, int D, int d_k, int d_v, int dtype, int chunks, HostPlan* hp) {
  if (B < 1 || N < 1 || D < 1 || chunks < 1) return MHA_ERR_INVALID;
  if (dtype != MHA_F32 && dtype != MHA_BF16) return MHA_ERR_INVALID;
  const int c = chunks < B ? chunks : B;
  hp->Bc = (B + c - 1) / c;
  hp->chunks = (B + hp->Bc - 1) / hp->Bc;
  size_t ws = 0;
  const int st = mha_layer_workspace_size(hp->Bc, H, N, N, D, d_k, d_v, dtype, &ws);
  if (st != MHA_OK) return st;
  const size_t es = dtype == MHA_BF16 ? 2 : 4;
  hp->slice_bytes = static_cast<size_t>(hp->Bc) * N * D * es;
  const size_t slot = round_up(hp->slice_bytes, 256);
  hp->off_x[0] = 0;
  hp->off_x[1] = slot;
  hp->off_y[0] = 2 * slot;
  hp->off_y[1] = 3 * slot;
  hp->off_ws = 4 * slot;
  hp->layer_ws = ws;
  hp->total = hp->off_ws + ws;
  return MHA_OK;
}

// The copy streams and events of the current device, created on its first call.
int pipe_of(int dev, Pipe** out) {
  Pipe& p = g_pipe[dev];
  if (!p.init) {
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    if (!ok(cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking)) ||
        !ok(cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking)) ||
        !ok(cudaEventCreateWithFlags(&p.entry, cudaEventDisableTiming))) {
      cudaGetLastError();
      return MHA_ERR_CUDA;
    }
    for (int k = 0; k < 2; ++k)
      if (!ok(cudaEventCreateWithFlags(&p.in_done[k], cudaEventDisableTiming)) ||
          !ok(cudaEventCreateWithFlags(&p.comp_done[k], cudaEventDisableTiming)) ||
          !ok(cudaEventCreateWithFlags(&p.out_done[k], cudaEventDisableTiming))) {
        cudaGetLastError();
        return MHA_ERR_CUDA;
      }
    p.init = true;
  }
  *out = &p;
  return MHA_OK;
}

}  // namespace

extern "C" {

int mha_layer_host_workspace_size(int B, int H, int N, int D, int d_k, int d_v, int dtype,
                                  int chunks, size_t* bytes) {
  if (bytes == nullptr) return MHA_ERR_INVALID;
  HostPlan hp;
  const int st = plan_host(B, H, N, D, d_k, d_v, dtype, chunks, &hp);
  if (st != MHA_OK) return st;
  *bytes = hp.total;
  return MHA_OK;
}

int mha_layer_fwd_host(int B, int H, int N, int D, int d_k, int d_v, int dtype, int mask,
                       const int32_t* key_len, float ln_eps, const void* x_host,
                       const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                       const void* gamma, const void* beta, void* y_host, int chunks,
                       void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (x_host == nullptr || y_host == nullptr) return MHA_ERR_INVALID;
  HostPlan hp;
  int st = plan_host(B, H, N, D, d_k, d_v, dtype, chunks, &hp);
  if (st != MHA_OK) return st;
  if (workspace == nullptr || ws_bytes < hp.total) return MHA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return MHA_ERR_ALIGN;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // every check mha_layer_fwd makes on one slice, the device included, before anything is
  // created or enqueued
  mha::DevCtx ctx;
  st = mha::check_layer_call(hp.Bc, H, N, N, D, d_k, d_v, dtype, mask, key_len, ln_eps,
                             ws + hp.off_x[0], nullptr, W_qkv, b_qkv, W_o, b_o, gamma, beta,
                             ws + hp.off_y[0], ws + hp.off_ws, hp.layer_ws, false, &ctx);
  if (st != MHA_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MHA_ERR_CUDA;
  }
  // one caller at a time per device: the events below are reused across slices and calls
  std::lock_guard<std::mutex> lk(g_pipe_mu[dev]);
  Pipe* pp = nullptr;
  st = pipe_of(dev, &pp);
  if (st != MHA_OK) return st;
  Pipe& p = *pp;
  auto cu = [](cudaError_t e) { return e == cudaSuccess; };
  // the copy streams start after everything the caller queued before this call
  if (!cu(cudaEventRecord(p.entry, stream)) || !cu(cudaStreamWaitEvent(p.in, p.entry, 0)) ||
      !cu(cudaStreamWaitEvent(p.out, p.entry, 0)))
    return MHA_ERR_CUDA;
  const size_t es = dtype == MHA_BF16 ? 2 : 4;
  const size_t row_bytes = static_cast<size_t>(N) * D * es;  // one sequence
  for (int i = 0; i < hp.chunks; ++i) {
    const int b0 = i * hp.Bc;
    const int nb = (B - b0) < hp.Bc ? (B - b0) : hp.Bc;
    const size_t bytes = static_cast<size_t>(nb) * row_bytes;
    const int k = i & 1;
    uint8_t* xd = ws + hp.off_x[k];
    uint8_t* yd = ws + hp.off_y[k];
    // x of slice i, once slice i-2's computation has read this buffer
    if (i >= 2 && !cu(cudaStreamWaitEvent(p.in, p.comp_done[k], 0))) return MHA_ERR_CUDA;
    if (!cu(cudaMemcpyAsync(xd, static_cast<const uint8_t*>(x_host) + b0 * row_bytes, bytes,
                            cudaMemcpyHostToDevice, p.in)) ||
        !cu(cudaEventRecord(p.in_done[k], p.in)))
      return MHA_ERR_CUDA;
    // slice i on the caller's stream, once its x has landed and slice i-2's y has left
    if (!cu(cudaStreamWaitEvent(stream, p.in_done[k], 0))) return MHA_ERR_CUDA;
    if (i >= 2 && !cu(cudaStreamWaitEvent(stream, p.out_done[k], 0))) return MHA_ERR_CUDA;
    st = mha_layer_fwd(nb, H, N, N, D, d_k, d_v, dtype, mask,
                       key_len != nullptr ? key_len + b0 : nullptr, ln_eps, xd, nullptr, W_qkv,
                       b_qkv, W_o, b_o, gamma, beta, yd, ws + hp.off_ws, hp.layer_ws, stream);
    if (st != MHA_OK) return st;
    if (!cu(cudaEventRecord(p.comp_done[k], stream))) return MHA_ERR_CUDA;
    // y of slice i back to the host
    if (!cu(cudaStreamWaitEvent(p.out, p.comp_done[k], 0)) ||
        !cu(cudaMemcpyAsync(static_cast<uint8_t*>(y_host) + b0 * row_bytes, yd, bytes,
                            cudaMemcpyDeviceToHost, p.out)) ||
        !cu(cudaEventRecord(p.out_done[k], p.out)))
      return MHA_ERR_CUDA;
  }
  // the caller's stream is done when the last copy back is (the copy stream runs in order)
  if (!cu(cudaStreamWaitEvent(stream, p.out_done[(hp.chunks - 1) & 1], 0))) return MHA_ERR_CUDA;
  return MHA_OK;
}

}  // extern "C"
