// launchers.h -- host-side entry points of the kernels, used by the C ABI layer (capi.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

namespace mha {

// Per-launch device context: where kernels record errors, and how long a bounded wait may
// spin before it gives up.
struct DevCtx {
  int* status;          // 4-int device status block (see device_common.cuh)
  uint64_t timeout_ns;  // limit of every mbarrier wait
  int num_sms;
};

// ---- every check mha_layer_fwd makes before it launches anything, in its order: shapes,
// mask, required pointers, eps, workspace size, alignment, then the current device (which
// fills ctx).  builtin_workspace: the workspace is the library's own scratch area, whose
// address is looked up only after these checks pass (workspace is then ignored).
int check_layer_call(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype, int mask,
                     const int32_t* key_len, float ln_eps, const void* x_q, const void* x_kv,
                     const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                     const void* gamma, const void* beta, const void* y, const void* workspace,
                     size_t ws_bytes, bool builtin_workspace, DevCtx* ctx);

// ---- per-kernel launch preparation: raises the kernel's dynamic shared-memory limit to
// smem_bytes and reports its register count (num_regs may be null), once per (kernel, device);
// later calls return the cached result without driver calls.
cudaError_t prepare_kernel(const void* func, int smem_bytes, int* num_regs);

// ---- launch with programmatic stream serialization: the kernel may begin (its set-up up to
// pdl_wait) while the previous kernel in the stream finishes
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- projections: Y[M,N] = act(X[M,K] W[N,K]^T + bias), act = identity or ReLU (relu)
// bf16 tensor-core path.  tmX: 2-D map over X {K, M}, box {64, 128}; tmW: 2-D map over W
// {K, N}, box {64, block_n}; tmY: 2-D map over Y {N, M}, box {64, 32}; all 128-byte swizzled.
// block_n is 128 or 256.
// residual: optional R [M, N] with Y's row pitch, added in the epilogue (Y = XW^T + b + R)
cudaError_t launch_gemm_bf16(const CUtensorMap& tmX, const CUtensorMap& tmW,
                             const CUtensorMap& tmY, int block_n,
                             bool relu, const void* bias, void* Y, int M, int N, int K,
                             int64_t ldy, const DevCtx& ctx, cudaStream_t s,
                             const void* residual = nullptr);
// Two such GEMMs with the same K (no ReLU, no residual) in one launch: the persistent CTAs
// work through the first problem's tiles and then the second's, so two small projections
// share one fill of the GPU.  Both sets of maps as for launch_gemm_bf16 with this block_n.
cudaError_t launch_gemm_bf16_two(const CUtensorMap& tmX1, const CUtensorMap& tmW1,
                                 const CUtensorMap& tmY1, const void* bias1, int M1, int N1,
                                 const CUtensorMap& tmX2, const CUtensorMap& tmW2,
                                 const CUtensorMap& tmY2, const void* bias2, int M2, int N2,
                                 int K, int block_n, const DevCtx& ctx, cudaStream_t s);
// The same GEMM on pairs of SMs (gemm2_bf16.cu): a cluster of two CTAs per 256 x 256 output
// tile, one pair-granularity MMA (M = 256) with half of each operand in each CTA.  tmX: box
// {64, 128}; tmW: box {64, 128}; tmY: box {64, 32}.  Needs K % 64 == 0 and N % 64 == 0.
bool gemm2_bf16_supported(int M, int N, int K);
cudaError_t launch_gemm2_bf16(const CUtensorMap& tmX, const CUtensorMap& tmW,
                              const CUtensorMap& tmY, bool relu, const void* bias, int M, int N,
                              int K, const DevCtx& ctx, cudaStream_t s);
// Weight-gradient forms (no bias, no activation), both operands MN-major: X stored [K, M] and
// W stored [K, N] (row-major activations, tokens = K), maps {M or N, K} with box {64, 64};
// 128 x 128 tiles.  launch_gemm_bf16_mn writes Y directly.  The split-K form zeroes acc
// [M, N] fp32 scratch, adds each of ksplit K slices of every tile into it by bulk tensor
// reductions through tmAcc (fp32 {N, M}, box {32, 32}, 128-byte swizzle), then Y = bf16(acc);
// ceil(K / 64) must be at least ksplit.
cudaError_t launch_gemm_bf16_mn(const CUtensorMap& tmX, const CUtensorMap& tmW,
                                const CUtensorMap& tmY, void* Y, int M, int N, int K,
                                int64_t ldy, const DevCtx& ctx, cudaStream_t s);
cudaError_t launch_gemm_bf16_splitk(const CUtensorMap& tmX, const CUtensorMap& tmW,
                                    const CUtensorMap& tmAcc, float* acc, int ksplit, void* Y,
                                    int M, int N, int K, int64_t ldy, const DevCtx& ctx,
                                    cudaStream_t s);
// ---- W^O projection fused with the residual + LayerNorm of the sublayer (bf16):
// y = LayerNorm(x + C W^T + bias) * gamma + beta for C [M, K], W [D, K], x and y [M, D]
// (row pitch D).  tmX: 2-D map over C {K, M}, box {64, 128}; tmW: over W {K, D}, box {64, 256};
// both 128-byte swizzled.  Needs D a multiple of 256 up to 2048 and K a multiple of 64
// (gemm_ln_bf16_supported).  a_out: optional [M, D] (row pitch D) that also receives the
// projection output bf16(C W^T + bias).
bool gemm_ln_bf16_supported(int D, int K);
cudaError_t launch_gemm_ln_bf16(const CUtensorMap& tmX, const CUtensorMap& tmW,
                                const void* bias, const void* x, const void* gamma,
                                const void* beta, void* y, int M, int D, int K, float eps,
                                const DevCtx& ctx, cudaStream_t s, void* a_out = nullptr);
cudaError_t launch_gemm_f32(const float* X, int64_t ldx, const float* W, const float* bias,
                            bool relu, float* Y, int64_t ldy, int M, int N, int K,
                            cudaStream_t s, const float* residual = nullptr);

// ---- attention
// Mask kinds beyond the public mha_mask values: restricted self-attention, where query i
// attends keys j with |i - j| <= SdpaArgs::window; decoding against a cache of
// L = key_len[b] positions, where query i (one of the Nq newest) attends j <= L - Nq + i.
constexpr int kMaskWindow = 3;
constexpr int kMaskCausalCache = 4;

struct SdpaArgs {
  int B, H, Nq, Nk, d_k, d_v;
  int mask;                  // mha_mask, or kMaskWindow
  int window = 0;            // radius of the restricted-attention neighbourhood (kMaskWindow)
  const int32_t* key_len;    // device, B entries (key padding) or null
  float scale;               // multiplies q.k
  const void* Q;             // used by the f32 path (the bf16 path reads through TMA maps)
  const void* K;
  const void* V;
  void* O;
  int64_t sq[4], sk[4], sv[4], so[4];  // element strides b, h, n, d
  // optional: natural log of each row's softmax denominator, log sum_j exp(q.k_j * scale)
  // over the allowed keys (+inf for a row with none), fp32 [B, H, Nq] contiguous
  float* lse = nullptr;
  int* status = nullptr;     // device status word (the f32 kernel's index checks)
};
// bf16: Q/K/V through 4-D TMA maps {d, n, h, b} with box {64, 128, 1, 1}, 128-byte swizzle;
// O written through the same kind of map with box {64, 32, 1, 1} (one 32-row box per warp).
cudaError_t launch_sdpa_bf16(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, const CUtensorMap& tmO, const SdpaArgs& a,
                             const DevCtx& ctx, cudaStream_t s);
cudaError_t launch_sdpa_f32(const SdpaArgs& a, cudaStream_t s);

// ---- one generation step against a key/value cache (split-K over the cached keys)
constexpr int kDecodeMaxQ = 16;  // new query rows per call on the bf16 path
struct DecodeArgs {
  int B, H, Nq, Lmax;
  int causal;                // 1: query i attends keys j <= L - Nq + i; 0: every j < L
  const int32_t* cache_len;  // device, B entries: L (clamped to [0, Lmax] on the device)
  float scale;
  const void* Q;             // [B, H, Nq, 64] with element strides sq (d stride 1)
  void* O;                   // [B, H, Nq, 64] with element strides so
  int64_t sq[4], so[4];
};
int decode_num_splits(int Lmax);  // 256-key chunks per (batch, head)
// bf16: the caches through 4-D TMA maps {64, Lmax, H, B}, box {64, 128, 1, 1}; part: fp32
// scratch of B * H * decode_num_splits(Lmax) * Nq * 66 floats.
cudaError_t launch_sdpa_decode_bf16(const CUtensorMap& tmK, const CUtensorMap& tmV,
                                    const DecodeArgs& a, float* part, const DevCtx& ctx,
                                    cudaStream_t s);

// ---- attention backward (dQ, dK, dV) from Q, K, V, O, dO and the forward's log-sum-exp
struct SdpaBwdArgs {
  int B, H, Nq, Nk, d_k, d_v;
  int mask, window;          // as in SdpaArgs
  const int32_t* key_len;
  float scale;
  const void *Q, *K, *V, *O, *dO;
  const float* lse;          // [B, H, Nq] natural-log softmax denominators
  // scratch written by launch_sdpa_bwd_rowdot from O, dO and lse: fp32 path, D_i =
  // rowsum(dO * O) as [B, H, Nq]; bf16 path, per 128-row query tile of every (b, h) the
  // tile's lse * log2(e) [128] then its D [128] (rows past Nq: +inf and 0), so one 1 KB bulk
  // copy brings a tile's statistics into shared memory
  // bf16 path, after those statistics (at sdpa_bwd_aug_offset): per query tile an 8 KB
  // operand block for the dK/dV kernel's tensor-core products, four 128 x 8 bf16 column
  // chunks (row r of chunk k at (k * 128 + r) * 16 bytes, the no-swizzle K-major layout):
  // chunk 0 = (-lse / scale) as a sum of three bf16 terms, chunk 2 = -D likewise, chunks 1
  // and 3 zero; then (at sdpa_bwd_dq_acc_offset) an fp32 dQ accumulator
  // [B, H, 128 * tiles, 64] that the rowdot launch zeroes and the fused kernel adds every key
  // tile's dS K into (unused when deterministic)
  float* Dv;
  bool deterministic;        // bf16: dQ by its own kernel instead of the fused accumulation
  void *dQ, *dK, *dV;
  int64_t st[8][4];          // element strides b, h, n, d of Q, K, V, O, dO, dQ, dK, dV
};
cudaError_t launch_sdpa_bwd_rowdot(const SdpaBwdArgs& a, int dtype, cudaStream_t s);
inline size_t sdpa_bwd_aug_offset(int B, int H, int Nq) {
  return static_cast<size_t>(B) * H * ((Nq + 127) / 128) * 1024;
}
inline size_t sdpa_bwd_dq_acc_offset(int B, int H, int Nq) {
  return static_cast<size_t>(B) * H * ((Nq + 127) / 128) * (1024 + 8192);
}
// bytes of the Dv scratch above
inline size_t sdpa_bwd_scratch_bytes(int B, int H, int Nq, int dtype) {
  return dtype == 1 ? sdpa_bwd_dq_acc_offset(B, H, Nq) +
                          static_cast<size_t>(B) * H * ((Nq + 127) / 128) * 128 * 64 * 4
                    : static_cast<size_t>(B) * H * Nq * 4;
}
cudaError_t launch_sdpa_bwd_f32(const SdpaBwdArgs& a, cudaStream_t s);
// bf16 (d = 64): Q, K, V, dO through 4-D TMA maps {64, n, h, b}, box {64, 128, 1, 1};
// tmDQ: the fp32 dQ accumulator {64, 128 * tiles, h, b}, box {32, 32, 1, 1}, 128-byte
// swizzle (read only when !a.deterministic)
cudaError_t launch_sdpa_bwd_bf16(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const CUtensorMap& tmG,
                                 const CUtensorMap& tmDQ, const SdpaBwdArgs& a,
                                 const DevCtx& ctx, cudaStream_t s);

// ---- memory-bound steps of the sublayer backward (bwd_util.cu)
int bwd_row_chunks(int M);  // chunks of rows the partial column sums use
// dr = LayerNorm backward at r = x + a (one warp per row; stats[row] = (mean, rstd)), then
// part[(chunk * 3 + k) * D + col] = per-chunk sums of dy * rhat, dy, dr
cudaError_t launch_layernorm_bwd(int dtype, int M, int D, float eps, const void* x,
                                 const void* a, const void* gamma, const void* dy, void* dr,
                                 float2* stats, float* part, cudaStream_t s);
// part[chunk * N + col] = per-chunk column sums of X [M, N] (row pitch ld)
cudaError_t launch_colsum_partials(int dtype, const void* X, int64_t ld, int M, int N,
                                   float* part, cudaStream_t s);
// out[col] = sum over chunks of part[chunk * chunk_stride + col], in chunk order
cudaError_t launch_reduce_partials(int dtype, const float* part, int nchunk,
                                   int64_t chunk_stride, int N, void* out, cudaStream_t s);
// nterm (<= 3) such sums in one launch: out_t from part + t * term_stride
cudaError_t launch_reduce_partials3(int dtype, const float* part, int nchunk,
                                    int64_t chunk_stride, int N, int64_t term_stride,
                                    int nterm, void* out0, void* out1, void* out2,
                                    cudaStream_t s);
// Y [C, R_pad] (row pitch ldy) = X [R, C]^T (row pitch ldx), zero for rows R..R_pad
cudaError_t launch_transpose(int dtype, const void* X, int64_t ldx, int R, int C, void* Y,
                             int64_t ldy, int R_pad, cudaStream_t s);

// ---- residual + LayerNorm: y = LN(x + a) * gamma + beta
// bf16: persistent warps over rows with an L2 prefetch of each warp's next row; fp32: one
// warp per row.  x, a, y contiguous [M, D], 16-byte aligned, D % 8 == 0, D <= 2048.
cudaError_t launch_residual_layernorm(int dtype, int M, int D, float eps, const void* x,
                                      const void* a, const void* gamma, const void* beta,
                                      void* y, const DevCtx& ctx, cudaStream_t s);

// ---- bounded-wait self test (waits on a barrier nothing completes)
cudaError_t launch_wait_selftest(const DevCtx& ctx, cudaStream_t s);

}  // namespace mha
