/*
 * mha.h -- C ABI of the GB300 (sm_103a) multi-head attention sublayer library (libmha.so).
 *
 * The operations are those of "Attention Is All You Need" as restated by the Chinese pages
 * this library follows:
 *   [LT] lettle.cn translation: 3.1 Encoder and Decoder Stacks (post-norm sublayer),
 *        3.2.1 缩放点积注意力 (Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V),
 *        3.2.2 多头注意力 (per-head projections, concat, output projection).
 *   [TC] "Transformer 为什么抛弃循环网络" (treecat.cn): 编码器和解码器 (the encoder layer, the
 *        feed-forward formula and its 512 -> 2048 -> 512 sizes).
 *   [LC] "Attention Is All You Need" (likecs.com): 1.3 按地址的前向反馈网络 (two linear maps
 *        with a ReLU between them, applied to every position with the same parameters).
 *   [JY] "Transformer：抛弃循环与卷积的序列建模" (jiashun-ye.github.io): Multi-Head Attention,
 *        Transformer 中的三种 Attention (self / masked self / cross attention), FFN,
 *        Self-Attention的优势 and 总结 (restricted self-attention over a neighbourhood r),
 *        Transformer 翻译样例 > Decoder (one generation step at a time),
 *        Residual Connection 与 LayerNorm, 训练样本 (the causal mask), 反向传播 (padding mask),
 *        模型变体与消融实验 (d_ff = 2048 base, 4096 big).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library allocates no
 *     device memory and keeps no state besides cached per-device properties.
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream).  Outputs are
 *     valid once the caller has synchronised that stream.
 *   - Row-major layouts; "stride" always counts ELEMENTS, not bytes.
 *   - dtype MHA_BF16: bf16 storage, fp32 accumulation, bf16 (round-to-nearest-even) outputs,
 *     tensor-core (tcgen05) kernels.  dtype MHA_F32: fp32 storage and arithmetic (SIMT
 *     kernels, no TF32).
 *   - Return value: MHA_OK or a negative mha_status.  Argument errors are found on the host
 *     before anything is launched.  MHA_ERR_CUDA means a CUDA launch or API call failed.
 *     Device-side problems (a bounded wait that ran out) are recorded in a device status
 *     word that mha_debug_last_device_status() reads; no kernel traps.
 *   - The library needs an sm_103 device (GB300); other devices get MHA_ERR_UNSUPPORTED.
 */
#ifndef MHA_GB300_H
#define MHA_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MHA_OK = 0,
  MHA_ERR_INVALID = -1,        /* bad shape, null pointer, unknown enum, causal with Nq != Nk */
  MHA_ERR_UNSUPPORTED = -2,    /* valid request this build does not implement (e.g. bf16 d_k != 64) */
  MHA_ERR_ALIGN = -3,          /* pointer or stride not aligned as the kernel requires */
  MHA_ERR_WORKSPACE = -4,      /* workspace missing or smaller than the matching *_workspace_size() */
  MHA_ERR_CUDA = -5,           /* a CUDA runtime/driver call or a launch failed */
  MHA_ERR_DEVICE_TIMEOUT = -6, /* a device-side bounded wait ran out (see mha_debug_*) */
  MHA_ERR_DEVICE_BOUNDS = -7   /* a kernel of the MHA_DEBUG_BOUNDS build (libmha_debug.so)
                                  computed an index outside a buffer; the access was skipped */
} mha_status;

typedef enum { MHA_F32 = 0, MHA_BF16 = 1 } mha_dtype;

/* Mask kinds ([JY] Transformer 中的三种 Attention; 训练样本; 反向传播):
 *   NONE        every query attends every key;
 *   CAUSAL      query i attends keys j <= i (Nq must equal Nk);
 *   KEY_PADDING query rows of batch element b attend keys j < key_len[b]; a row with
 *               key_len[b] == 0 is written as zeros. */
typedef enum { MHA_MASK_NONE = 0, MHA_MASK_CAUSAL = 1, MHA_MASK_KEY_PADDING = 2 } mha_mask;

/*
 * mha_sdpa_fwd -- scaled dot-product attention per (batch, head):
 *     O[b,h] = softmax(Q[b,h] K[b,h]^T * scale, masked) V[b,h]          ([LT] 3.2.1)
 *
 *   Q [B,H,Nq,d_k], K [B,H,Nk,d_k], V [B,H,Nk,d_v], O [B,H,Nq,d_v] (written).
 *   strides: NULL for contiguous [B,H,N,d] tensors, or 16 int64 element strides laid out as
 *            {Q: b,h,n,d,  K: b,h,n,d,  V: b,h,n,d,  O: b,h,n,d}.  This lets Q/K/V be read
 *            straight out of a packed projection buffer and O be written in the head-concat
 *            layout [B,Nq,H*d_v] (O strides {Nq*H*d_v, d_v, H*d_v, 1}).
 *   key_len: device int32[B]; required iff mask == MHA_MASK_KEY_PADDING, ignored otherwise.
 *            Values are clamped to [0, Nk] on the device.
 *   scale:  > 0 uses the given factor; <= 0 means 1/sqrt(d_k).
 *   dtype MHA_BF16: d_k == d_v == 64; d strides 1; all other strides multiples of 8 and > 0;
 *            Q/K/V/O 16-byte aligned (else MHA_ERR_ALIGN).
 *   dtype MHA_F32:  1 <= d_k, d_v <= 128; pointers 4-byte aligned.
 * The n x n score matrix is never written to memory.
 */
int mha_sdpa_fwd(int B, int H, int Nq, int Nk, int d_k, int d_v, int dtype, int mask,
                 const int32_t* key_len, float scale,
                 const void* Q, const void* K, const void* V, void* O,
                 const int64_t* strides, cudaStream_t stream);

/*
 * mha_sdpa_fwd_lse -- mha_sdpa_fwd that also writes, for every query row, the natural log of
 * its softmax denominator: lse[b,h,i] = log sum_j exp(Q[b,h,i] . K[b,h,j] * scale) over the
 * allowed keys (+inf for a row with none), fp32 [B, H, Nq] contiguous, 4-byte aligned.  The
 * backward pass (mha_sdpa_bwd) rebuilds the softmax weights as exp(s - lse) from it.
 * Same arguments, limits and errors as mha_sdpa_fwd; MHA_ERR_INVALID if lse is NULL.
 */
int mha_sdpa_fwd_lse(int B, int H, int Nq, int Nk, int d_k, int d_v, int dtype, int mask,
                     const int32_t* key_len, float scale, const void* Q, const void* K,
                     const void* V, void* O, const int64_t* strides, float* lse,
                     cudaStream_t stream);

/*
 * mha_sdpa_bwd_workspace_size -- bytes of device workspace mha_sdpa_bwd needs: with
 * D_i = sum_d dO_id O_id, MHA_BF16 keeps 1 KB per (b, h, 128-row query tile) -- the tile's
 * D and lse (lse in base-2 units), both negated, read by one bulk copy -- followed by an fp32
 * dQ accumulator of 128 x 64 values (32 KB) per tile; MHA_F32 one fp32 D per query row.
 */
int mha_sdpa_bwd_workspace_size(int B, int H, int Nq, int dtype, size_t* bytes);

/*
 * mha_sdpa_bwd -- backward of scaled dot-product attention ([JY] Transformer 训练样例 >
 * 反向传播: the chain rule through the forward's steps; [LT] 3.2.1 for the forward).  With the
 * weights rebuilt from the forward's log-sum-exp, P_ij = exp(Q_i . K_j * scale - lse_i)
 * (0 for excluded keys), and D_i = sum_d dO_id O_id:
 *     dV = P^T dO,  dS = P * (dO V^T - D),  dQ = scale * dS K,  dK = scale * dS^T Q
 *   Q, O, dO, dQ [B,H,Nq,d]; K, V, dK, dV [B,H,Nk,d]; lse [B,H,Nq] fp32 from
 *   mha_sdpa_fwd_lse (same Q, K, mask and scale); O is that call's output.  mask, key_len,
 *   scale as for mha_sdpa_fwd (none / causal / key padding).  dQ, dK, dV are written
 *   (keys no query may see get zero gradients); they may not alias the inputs.
 *   strides: NULL for contiguous, or 32 element strides {Q, K, V, O, dO, dQ, dK, dV} x
 *   {b, h, n, d} (d stride 1).  workspace: mha_sdpa_bwd_workspace_size() bytes, 256-byte
 *   aligned.  dtype MHA_BF16: d_k == d_v == 64, other strides multiples of 8, 16-byte aligned
 *   pointers; tensor-core kernels.  By default one CTA per 128 keys computes dK, dV and that
 *   key tile's part of dQ (dS K for every query tile it sees), which it adds in fp32 into the
 *   workspace's accumulator with bulk tensor reductions; a last launch scales it into dQ.
 *   The additions run in whatever order the key tiles finish, so dQ can differ between
 *   calls by fp32 rounding (then rounded to bf16).  After mha_set_deterministic(1), dQ comes
 *   from its own kernel (one CTA per 128 query rows, S and dP rebuilt, no atomics) and all
 *   three gradients are bitwise reproducible.  dtype MHA_F32: d <= 128, SIMT kernels,
 *   always reproducible.
 */
int mha_sdpa_bwd(int B, int H, int Nq, int Nk, int d_k, int d_v, int dtype, int mask,
                 const int32_t* key_len, float scale, const void* Q, const void* K,
                 const void* V, const void* O, const void* dO, const float* lse, void* dQ,
                 void* dK, void* dV, const int64_t* strides, void* workspace, size_t ws_bytes,
                 cudaStream_t stream);

/*
 * mha_sdpa_window_fwd -- restricted self-attention ([JY] Self-Attention的优势, 总结): every
 * position attends only the neighbourhood of size r = 2*window + 1 centred on it,
 *     O[b,h,i] = softmax_j(Q[b,h,i] . K[b,h,j] * scale, |i - j| <= window) V[b,h,j]
 * so the work is O(r n d) instead of O(n^2 d).  The pages give the neighbourhood's size,
 * not its placement; centred on the query is the reading taken here.
 *   Q, K, V, O [B,H,N,d] (self-attention: Nq = Nk = N); strides, scale, dtype limits and
 *   errors as for mha_sdpa_fwd.  window >= 0 (0: each position sees itself only; N - 1 or
 *   more: full attention); window < 0 is MHA_ERR_INVALID.  Only the key tiles that a query
 *   block's band touches are read.
 */
int mha_sdpa_window_fwd(int B, int H, int N, int d_k, int d_v, int dtype, int window,
                        float scale, const void* Q, const void* K, const void* V, void* O,
                        const int64_t* strides, cudaStream_t stream);

/*
 * mha_decode_workspace_size -- bytes of device workspace mha_sdpa_decode_fwd needs: for
 * MHA_BF16 one fp32 partial result (64 columns, a max and a sum) per (batch, head, 256-key
 * chunk of the cache, query); for MHA_F32 a token 256 bytes (that path keeps no partials).
 * MHA_ERR_UNSUPPORTED for bf16 with Nq > 16.
 */
int mha_decode_workspace_size(int B, int H, int Nq, int Lmax, int dtype, size_t* bytes);

/*
 * mha_sdpa_decode_fwd -- attention for one autoregressive generation step against a
 * key/value cache ([JY] Transformer 翻译样例 > Decoder: each step's newest target positions
 * attend every position generated so far, and the encoder output Z; Transformer 训练样例:
 * the causal mask during training, one position at a time during generation):
 *     O[b,h,i] = softmax_j(Q[b,h,i] . K[b,h,j] * scale, allowed) V[b,h,j]
 *   allowed: j < L_b = cache_len[b] (the cache's valid prefix; cross-attention to Z), and
 *   with causal = 1 also j <= L_b - Nq + i: the Nq queries are the newest of the L_b cached
 *   positions, i.e. the causal mask aligned bottom-right (masked self-attention).
 *   Keys and values of earlier positions never change under the causal mask, so caching
 *   them computes the same result as re-running the whole prefix.
 *
 *   Q [B,H,Nq,d_k] (the new positions' queries); K, V caches [B,H,Lmax,d] (capacity Lmax,
 *   the new positions already written at L_b - Nq .. L_b - 1); O [B,H,Nq,d_v] (written).
 *   strides: NULL for contiguous, or 16 element strides {Q, K, V, O} x {b, h, n, d} as for
 *   mha_sdpa_fwd.  cache_len: device int32[B], clamped to [0, Lmax] on the device; rows that
 *   end up with no allowed key (L_b = 0, or L_b < Nq with causal = 1) are written as zeros.
 *   scale: > 0 uses it, <= 0 means 1/sqrt(d_k).  causal must be 0 or 1; Nq <= Lmax.
 *   workspace: at least mha_decode_workspace_size() bytes, 256-byte aligned, caller-owned.
 *   dtype MHA_BF16: d_k == d_v == 64, 1 <= Nq <= 16, strides and pointers as for
 *   mha_sdpa_fwd's bf16 path; memory-bound split-K kernel (256-key chunks of the cache per
 *   CTA, then one merge launch).  dtype MHA_F32: d_k, d_v <= 128 (SIMT kernel).
 */
int mha_sdpa_decode_fwd(int B, int H, int Nq, int Lmax, int d_k, int d_v, int dtype, int causal,
                        const int32_t* cache_len, float scale, const void* Q, const void* K,
                        const void* V, void* O, const int64_t* strides, void* workspace,
                        size_t ws_bytes, cudaStream_t stream);

/*
 * mha_layer_workspace_size -- bytes of device workspace mha_layer_fwd needs for these sizes.
 * The workspace holds the projected Q/K/V, the head-concat buffer and the W^O output.
 */
int mha_layer_workspace_size(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                             size_t* bytes);

/*
 * mha_layer_fwd -- one post-norm multi-head attention sublayer ([LT] 3.1, 3.2.2; [JY]
 * Multi-Head Attention, Residual Connection 与 LayerNorm):
 *     Q_i = x_q W_i^Q + b_i^Q,  K_i = x_kv W_i^K + b_i^K,  V_i = x_kv W_i^V + b_i^V
 *     head_i = Attention(Q_i, K_i, V_i)            (mask as above)
 *     A = Concat(head_1..head_H) W^O + b_o
 *     y = LayerNorm(x_q + A) * gamma + beta        (biased variance, eps = ln_eps)
 *
 *   x_q  [B,Nq,D];  x_kv [B,Nk,D], or NULL for self-attention (then Nk must equal Nq).
 *   W_qkv [H*(2*d_k+d_v), D] in nn.Linear layout [out,in]: rows 0..H*d_k-1 are W^Q (head h
 *         owns rows h*d_k..), then W^K, then W^V.   b_qkv [H*(2*d_k+d_v)] or NULL (= 0).
 *   W_o  [D, H*d_v];  b_o [D] or NULL;  gamma, beta [D] or NULL (= 1 and 0).
 *   y    [B,Nq,D] written; may not alias any input or the workspace.
 *   All of the above share `dtype`.  key_len as for mha_sdpa_fwd.
 *   workspace: device buffer of at least mha_layer_workspace_size() bytes, 256-byte aligned,
 *         owned by the caller; its contents on entry do not matter.
 *   dtype MHA_BF16 needs d_k == d_v == 64 and D a multiple of 64; MHA_F32 needs d_k, d_v <= 128.
 * Launches: one or two projection GEMMs, the attention kernel, the W^O GEMM, the residual
 * LayerNorm -- all on `stream`.
 */
int mha_layer_fwd(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype, int mask,
                  const int32_t* key_len, float ln_eps,
                  const void* x_q, const void* x_kv, const void* W_qkv, const void* b_qkv,
                  const void* W_o, const void* b_o, const void* gamma, const void* beta,
                  void* y, void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * mha_layer_fwd_timed -- mha_layer_fwd plus profiling marks: events[0..4] (created by the
 * caller, n_events >= 5) are recorded on `stream` before the Q/K/V projection(s), before the
 * attention kernel, before the W^O projection, before the residual LayerNorm and after it, so
 * that cudaEventElapsedTime between consecutive marks is each step's device time.  Same
 * arguments, results and errors as mha_layer_fwd; MHA_ERR_INVALID if events is NULL,
 * n_events < 5 or one of the five is NULL.
 */
int mha_layer_fwd_timed(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                        int mask, const int32_t* key_len, float ln_eps,
                        const void* x_q, const void* x_kv, const void* W_qkv, const void* b_qkv,
                        const void* W_o, const void* b_o, const void* gamma, const void* beta,
                        void* y, void* workspace, size_t ws_bytes, cudaStream_t stream,
                        const cudaEvent_t* events, int n_events);

/*
 * mha_layer_bwd_workspace_size -- bytes of device workspace mha_layer_bwd needs for these
 * sizes (self_attention != 0: x_kv is NULL and Nk == Nq).  It holds the recomputed forward
 * intermediates (the activations mha_layer_fwd_train leaves), the gradients between the
 * steps, the attention backward's scratch (with its fp32 dQ accumulator), and for MHA_BF16
 * the fp32 accumulator of the split-K weight-gradient products, for MHA_F32 their transposed
 * operands.
 */
int mha_layer_bwd_workspace_size(int B, int H, int Nq, int Nk, int D, int d_k, int d_v,
                                 int dtype, int self_attention, size_t* bytes);

/*
 * mha_layer_bwd -- gradients of one post-norm multi-head attention sublayer ([JY] Transformer
 * 训练样例 > 反向传播: the chain rule back through every step of mha_layer_fwd's forward).
 * Given dy = dL/dy for y = mha_layer_fwd(...), it recomputes the forward (keeping the
 * attention's log-sum-exp) and writes, with r = x_q + A and rhat = LayerNorm(r) unscaled:
 *     dgamma = sum_rows dy * rhat,  dbeta = sum_rows dy,  dr = LayerNorm'(r)^T (dy * gamma)
 *     db_o = sum_rows dr,  dW_o = dr^T C,  dC = dr W_o          (C: head concat)
 *     dQ, dK, dV = mha_sdpa_bwd(...) per head, from dC split by heads
 *     dW_qkv = [dQ|dK|dV]^T [x_q|x_kv|x_kv],  db_qkv = column sums of [dQ|dK|dV]
 *     dx_q = dr + dQ W^Q (+ dK W^K + dV W^V for self-attention),  dx_kv = dK W^K + dV W^V
 *   Inputs as for mha_layer_fwd (same arguments, same values; beta does not enter any
 *   gradient and may be NULL); dy [B,Nq,D].  mask: none, causal or key padding.
 *   Outputs (all `dtype`, written, none may alias an input, another output or the workspace):
 *   dx_q [B,Nq,D]; dx_kv [B,Nk,D] for cross-attention (ignored, may be NULL, for self);
 *   dW_qkv like W_qkv; db_qkv [H*(2*d_k+d_v)]; dW_o like W_o; db_o, dgamma, dbeta [D]
 *   (always written, also when the forward passed NULL for the bias, gamma or beta).
 *   Sums over rows run per chunk of 256 rows and then over the chunks in a fixed order.  By
 *   default (bf16) the attention backward inside accumulates dQ in fp32 (see mha_sdpa_bwd)
 *   and the weight-gradient GEMMs, whose K is the token count, split K over several CTAs
 *   whose fp32 partials are added in no fixed order when that fills the SMs better; after
 *   mha_set_deterministic(1) neither happens and every result is bitwise reproducible.  workspace: mha_layer_bwd_workspace_size() bytes, 256-byte
 *   aligned.  Limits and errors as for mha_layer_fwd; MHA_ERR_INVALID for a NULL output.
 * Launches (all on `stream`): the forward's GEMMs, attention and W^O GEMM again, the
 * LayerNorm backward, the attention backward, the data- and weight-gradient GEMMs on the
 * same tensor-core kernel as the forward, transposes and column-sum reductions.
 */
int mha_layer_bwd(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype, int mask,
                  const int32_t* key_len, float ln_eps, const void* x_q, const void* x_kv,
                  const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                  const void* gamma, const void* beta, const void* dy, void* dx_q, void* dx_kv,
                  void* dW_qkv, void* db_qkv, void* dW_o, void* db_o, void* dgamma, void* dbeta,
                  void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * mha_layer_fwd_train / mha_layer_bwd_saved -- the same sublayer forward and backward split
 * the way a training step runs them ([JY] Transformer 训练样例: a forward pass, then the
 * backward pass), so the backward does not compute the forward a second time.
 *   mha_layer_fwd_train: arguments as for mha_layer_fwd, but `workspace` must hold
 *   mha_layer_bwd_workspace_size() bytes (256-byte aligned).  Writes y (the same values as
 *   mha_layer_fwd) and leaves in the workspace what the backward reads: the projections, the
 *   head concat C, the W^O output and the attention's log-sum-exp.
 *   mha_layer_bwd_saved: arguments as for mha_layer_bwd; the workspace must be the one a
 *   preceding mha_layer_fwd_train filled with the same inputs, parameters, mask and key_len
 *   (on the same stream, or ordered after it), untouched since.  The gradients equal those of
 *   mha_layer_bwd (bitwise in the deterministic mode).  Errors as for those two calls.
 */
int mha_layer_fwd_train(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                        int mask, const int32_t* key_len, float ln_eps, const void* x_q,
                        const void* x_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                        const void* b_o, const void* gamma, const void* beta, void* y,
                        void* workspace, size_t ws_bytes, cudaStream_t stream);
int mha_layer_bwd_saved(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                        int mask, const int32_t* key_len, float ln_eps, const void* x_q,
                        const void* x_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                        const void* b_o, const void* gamma, const void* beta, const void* dy,
                        void* dx_q, void* dx_kv, void* dW_qkv, void* db_qkv, void* dW_o,
                        void* db_o, void* dgamma, void* dbeta, void* workspace, size_t ws_bytes,
                        cudaStream_t stream);

/*
 * mha_layer_host_workspace_size -- device workspace bytes mha_layer_fwd_host needs: two
 * device buffers each for a slice's x and y, and mha_layer_fwd's workspace for one slice.
 */
int mha_layer_host_workspace_size(int B, int H, int N, int D, int d_k, int d_v, int dtype,
                                  int chunks, size_t* bytes);

/*
 * mha_layer_fwd_host -- the self-attention sublayer y = LayerNorm(x + MultiHead(x, x, x))
 * ([LT] 3.1, 3.2.2) with x and y in HOST memory (pinned memory lets the copies run
 * asynchronously; pageable memory makes them synchronous).  The weights, biases, gamma, beta and
 * key_len are device memory as for mha_layer_fwd.
 *   x_host, y_host: [B, N, D] dense, row-major.  chunks: the batch is processed in
 *   min(chunks, B) slices of ceil(B / chunks) sequences; slice i's x is copied in while slice
 *   i-1 is computed on `stream` and slice i-2's y is copied back, so the copies hide behind
 *   the computation except for the first slice's x and the last slice's y.
 *   workspace: device, at least mha_layer_host_workspace_size(...) bytes, 256-byte aligned.
 *   Each slice runs exactly as mha_layer_fwd on that slice (the results equal a per-slice
 *   mha_layer_fwd bit for bit; a whole-batch call may round differently where it fuses the
 *   W^O projection with the LayerNorm, which mha_layer_fwd does from 8192 rows on).
 *   The call is asynchronous on `stream`: y_host is complete once `stream` has finished
 *   everything queued up to this call.  The first call on a device creates two copy streams
 *   and a few events for that device, kept until the process exits; calls for one device
 *   from several host threads are serialised.  Errors: those of mha_layer_fwd for one slice
 *   (checked before anything is queued), MHA_ERR_INVALID for NULL host pointers or chunks < 1,
 *   MHA_ERR_WORKSPACE, MHA_ERR_ALIGN (workspace not 256-byte aligned), MHA_ERR_CUDA.
 */
int mha_layer_fwd_host(int B, int H, int N, int D, int d_k, int d_v, int dtype, int mask,
                       const int32_t* key_len, float ln_eps, const void* x_host,
                       const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                       const void* gamma, const void* beta, void* y_host, int chunks,
                       void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * mha_layer_fwd_noalloc -- mha_layer_fwd for callers that cannot supply a workspace.
 * The pages have no counterpart: this is a packaging variant, not part of the method.
 *
 * Who needs it: code that may not allocate device memory -- e.g. a plugin whose host
 * framework owns all GPU memory and forbids allocation inside its enqueue callback, or a
 * latency-critical path that cannot afford cudaMalloc's implicit device synchronisation.
 * Instead of a caller buffer, it uses a 48 MiB scratch area built into the library (a
 * file-scope __device__ array that stays resident on every GPU that loads the library until
 * the process exits).  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, results and errors are those of mha_layer_fwd without workspace/ws_bytes: it
 * makes the same checks in the same order (the current device's last, so a device other
 * than sm_103 gives MHA_ERR_UNSUPPORTED) before it touches the scratch area.
 * Sizes whose mha_layer_workspace_size() exceeds 48 MiB (50331648 bytes) return
 * MHA_ERR_WORKSPACE before anything is launched.  At d_model 512 (h = 8, d_k = d_v = 64)
 * that is up to 9830 self-attention tokens (B * n) per call in bf16 and 4915 in fp32.
 * The first call on each device looks up the scratch area's device address with that
 * device current (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.
 * All calls on one device share that device's scratch area, which keeps the previous
 * call's intermediates; nothing in it needs clearing (every byte a call reads, the same call
 * has written first).  Calls on the same device that can overlap on the GPU (issued to
 * streams with no ordering between them) race on the scratch and corrupt each other's
 * results: order them, e.g. issue them to one stream.  Each device has its own copy, so
 * calls on different devices do not interfere.
 */
int mha_layer_fwd_noalloc(int B, int H, int Nq, int Nk, int D, int d_k, int d_v, int dtype,
                          int mask, const int32_t* key_len, float ln_eps,
                          const void* x_q, const void* x_kv, const void* W_qkv,
                          const void* b_qkv, const void* W_o, const void* b_o,
                          const void* gamma, const void* beta, void* y, cudaStream_t stream);

/*
 * mha_linear_fwd -- Y[M,N] = X[M,K] W[N,K]^T + bias[N], the projection step of the sublayer
 * ([JY] Multi-Head Attention: Q_i = X W_i^Q; the W^O projection of [LT] 3.2.2).
 *   ldx, ldy: row pitch of X and Y in elements; W is dense [N,K].  bias may be NULL.
 *   dtype MHA_BF16: K and N multiples of 64, ldx/ldy multiples of 8, 16-byte aligned pointers.
 */
int mha_linear_fwd(int M, int N, int K, int dtype, const void* X, int64_t ldx, const void* W,
                   const void* bias, void* Y, int64_t ldy, cudaStream_t stream);

/*
 * mha_linear_relu_fwd -- Y[M,N] = max(0, X[M,K] W[N,K]^T + bias[N]): the first linear map of
 * the position-wise feed-forward network with its ReLU ([LC] 1.3; [JY] FFN).  Arguments,
 * layouts, limits and errors exactly as mha_linear_fwd.
 */
int mha_linear_relu_fwd(int M, int N, int K, int dtype, const void* X, int64_t ldx,
                        const void* W, const void* bias, void* Y, int64_t ldy,
                        cudaStream_t stream);

/*
 * mha_linear2_fwd -- two projections with the same K in one launch:
 *     Y1[M1,N1] = X1[M1,K] W1[N1,K]^T + b1[N1],   Y2[M2,N2] = X2[M2,K] W2[N2,K]^T + b2[N2]
 * the query projection of the decoder states and the key|value projection of the encoder
 * output in encoder-decoder attention ([LT] 3.2.3: queries from the previous decoder layer,
 * keys and values from the encoder output).  All matrices dense (row pitch K for X1, X2, W1,
 * W2; N1 and N2 for Y1 and Y2); b1, b2 may be NULL.  Y1 and Y2 equal what two mha_linear_fwd
 * calls write, bit for bit.  Limits and errors as mha_linear_fwd for each problem.
 */
int mha_linear2_fwd(int M1, int N1, const void* X1, const void* W1, const void* b1, void* Y1,
                    int M2, int N2, const void* X2, const void* W2, const void* b2, void* Y2,
                    int K, int dtype, cudaStream_t stream);

/*
 * mha_ffn_workspace_size -- bytes of device workspace mha_ffn_fwd needs: the hidden
 * activations [M, d_ff] and the second linear map's output [M, D].
 */
int mha_ffn_workspace_size(int M, int D, int d_ff, int dtype, size_t* bytes);

/*
 * mha_ffn_fwd -- one post-norm position-wise feed-forward sublayer ([LT] 3.1; [TC]
 * 编码器和解码器; [LC] 1.3; [JY] FFN, Residual Connection 与 LayerNorm):
 *     FFN(x) = max(0, x W1 + b1) W2 + b2       (applied to every row with the same weights)
 *     y = LayerNorm(x + FFN(x)) * gamma + beta  (biased variance, eps = ln_eps)
 *
 *   x, y [M, D] dense row-major (M = tokens); y may not alias x or the workspace.
 *   W1 [d_ff, D] and W2 [D, d_ff] in nn.Linear layout [out,in]; b1 [d_ff], b2 [D], gamma and
 *   beta [D], each nullable (= 0, 0, 1, 0).  All share `dtype`; 16-byte aligned pointers.
 *   workspace: at least mha_ffn_workspace_size() bytes, 256-byte aligned, caller-owned; its
 *   contents on entry do not matter.
 *   dtype MHA_BF16: D and d_ff multiples of 64.  Both dtypes: D a multiple of 8, <= 2048.
 * Launches: the ReLU GEMM, the second GEMM and the residual LayerNorm, all on `stream`.
 */
int mha_ffn_fwd(int M, int D, int d_ff, int dtype, float ln_eps, const void* x, const void* W1,
                const void* b1, const void* W2, const void* b2, const void* gamma,
                const void* beta, void* y, void* workspace, size_t ws_bytes,
                cudaStream_t stream);

/*
 * mha_ffn_fwd_timed -- mha_ffn_fwd plus profiling marks: events[0..3] (caller-created,
 * n_events >= 4) are recorded on `stream` before the first linear map, before the second,
 * before the residual LayerNorm and after it.  Same arguments, results and errors as
 * mha_ffn_fwd; MHA_ERR_INVALID if events is NULL, n_events < 4 or one of the four is NULL.
 */
int mha_ffn_fwd_timed(int M, int D, int d_ff, int dtype, float ln_eps, const void* x,
                      const void* W1, const void* b1, const void* W2, const void* b2,
                      const void* gamma, const void* beta, void* y, void* workspace,
                      size_t ws_bytes, cudaStream_t stream, const cudaEvent_t* events,
                      int n_events);

/*
 * mha_encoder_layer_workspace_size -- bytes of device workspace mha_encoder_layer_fwd needs
 * (the attention sublayer's output plus the larger of the two sublayers' workspaces).
 */
int mha_encoder_layer_workspace_size(int B, int N, int H, int D, int d_ff, int dtype,
                                     size_t* bytes);

/*
 * mha_encoder_layer_fwd -- one encoder layer: the self-attention sublayer, then the
 * feed-forward sublayer, each with its residual and LayerNorm ([LT] 3.1; [TC] 编码器和解码器;
 * [JY] Encoder-Decoder):
 *     h = LayerNorm(x + MultiHead(x, x, x)) * gamma1 + beta1
 *     y = LayerNorm(h + FFN(h)) * gamma2 + beta2
 *   x, y [B, N, D]; y may not alias x or the workspace.  H heads of d_k = d_v = D / H.
 *   W_qkv, b_qkv, W_o, b_o, mask and key_len as for mha_layer_fwd (self-attention; a causal
 *   mask gives the masked self-attention layer); W1, b1, W2, b2 as for mha_ffn_fwd; gamma1,
 *   beta1, gamma2, beta2 [D] or NULL.  One ln_eps for both LayerNorms.
 *   workspace: at least mha_encoder_layer_workspace_size() bytes, 256-byte aligned.
 *   Limits: those of mha_layer_fwd and mha_ffn_fwd (bf16: D / H == 64).
 */
int mha_encoder_layer_fwd(int B, int N, int H, int D, int d_ff, int dtype, int mask,
                          const int32_t* key_len, float ln_eps, const void* x,
                          const void* W_qkv, const void* b_qkv, const void* W_o,
                          const void* b_o, const void* gamma1, const void* beta1,
                          const void* W1, const void* b1, const void* W2, const void* b2,
                          const void* gamma2, const void* beta2, void* y, void* workspace,
                          size_t ws_bytes, cudaStream_t stream);

/*
 * mha_residual_layernorm_fwd -- y = LayerNorm(x + a) * gamma + beta over rows of D features
 * ([LT] 3.1: LayerNorm(x + Sublayer(x))).  x, a, y [M,D] dense; gamma/beta [D] or NULL.
 *   D a multiple of 8 and at most 2048; 16-byte aligned pointers.
 */
int mha_residual_layernorm_fwd(int M, int D, int dtype, float eps, const void* x, const void* a,
                               const void* gamma, const void* beta, void* y, cudaStream_t stream);

/*
 * mha_out_proj_layernorm_fwd -- y = LayerNorm(x + C W_o^T + b_o) * gamma + beta: the W^O
 * projection of the sublayer and its residual + post-norm step in one call ([LT] 3.2.2:
 * MultiHead = Concat(head_1..head_h) W^O; [LT] 3.1: LayerNorm(x + Sublayer(x))).  This is what
 * mha_layer_fwd runs after the attention step.
 *   C [M,K] (the head concat), W_o [D,K] ([out,in]), b_o [D] or NULL, x and y [M,D], gamma /
 *   beta [D] or NULL; all dense row-major, 16-byte aligned.
 *   bf16 with D a multiple of 256 (at most 2048) and K a multiple of 64: one kernel, the
 *   projection output never written to memory and never rounded (the residual sum is formed
 *   in fp32; the two-step path rounds the projection to bf16 when it stores it).  Otherwise (fp32, or other widths with D a multiple of 8 up to 2048 and,
 *   for bf16, D and K multiples of 64): the projection into y, then the LayerNorm in place.
 *   Errors: MHA_ERR_INVALID (sizes < 1, NULL C / W_o / x / y, eps < 0 or NaN),
 *   MHA_ERR_UNSUPPORTED (limits above, or not sm_103), MHA_ERR_ALIGN, MHA_ERR_CUDA.
 */
int mha_out_proj_layernorm_fwd(int M, int D, int K, int dtype, float eps, const void* C,
                               const void* W_o, const void* b_o, const void* x,
                               const void* gamma, const void* beta, void* y,
                               cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* mha_status_string(int status);

/*
 * mha_set_deterministic -- process-wide switch (0 by default) for the bf16 backward: 1
 * computes the attention's dQ by a separate kernel that rebuilds S and dP per query tile and
 * runs mha_layer_bwd's weight-gradient GEMMs without splitting K, all bitwise reproducible;
 * 0 adds every key tile's dQ part into an fp32 accumulator by bulk reductions and lets the
 * weight-gradient GEMMs add fp32 partials of K slices the same way: faster, reproducible up
 * to the order of fp32 additions.
 * Returns MHA_ERR_INVALID unless `on` is 0 or 1.  Takes effect for calls issued after it.
 * mha_get_deterministic -- the current setting.
 */
int mha_set_deterministic(int on);
int mha_get_deterministic(void);

/*
 * mha_debug_last_device_status -- synchronises `stream`, returns the first device-side error
 * recorded on the current device since the previous call (MHA_OK if none) and clears it.
 * Meant for tests and debugging; it blocks the host.
 */
int mha_debug_last_device_status(cudaStream_t stream);

/*
 * mha_debug_wait_selftest -- launches one block whose threads wait on a shared-memory
 * barrier that nothing will complete, with a limit of `timeout_ns` nanoseconds (clamped to
 * [1e3, 1e9]).  The wait gives up, records MHA_ERR_DEVICE_TIMEOUT in the device status word
 * and the kernel returns normally.  Exercises the bounded-wait path every kernel uses,
 * without hanging or faulting the GPU.  Returns the launch status; read the outcome with
 * mha_debug_last_device_status().
 */
int mha_debug_wait_selftest(int64_t timeout_ns, cudaStream_t stream);

/* Library ABI version (major*100 + minor). */
int mha_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MHA_GB300_H */
