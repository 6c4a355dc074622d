/*
 * gpt2_ops.h -- the individual kernels of the GPT-2 training step, callable on
 * caller-owned device buffers.  gpt2.h chains exactly these operations; they
 * are exported so each one can be checked and timed on its own.
 *
 * Common rules
 *   - Every pointer is a device pointer unless marked otherwise; the caller
 *     owns all buffers.  Float buffers used with 128-bit accesses (noted
 *     "16B") must be 16-byte aligned with row strides that are multiples of 4.
 *   - `stream` is a cudaStream_t (NULL: the default stream).  Every call is
 *     asynchronous on it.  Return value: GPT2_OK or a negative GPT2_E* code for
 *     argument errors or a failed launch.  Device-side data errors (ids
 *     outside [0, V)) OR a GPT2_STATUS_* bit into *status when status != NULL.
 *   - `mode` selects the contraction arithmetic: GPT2_MODE_FP32 (CUDA cores),
 *     GPT2_MODE_TF32 or GPT2_MODE_BF16 (tensor cores, fp32 accumulation).  The
 *     linear ops below take fp32 operands (FP32 and TF32 modes); bf16 products
 *     go through gpt2_op_gemm.  In TF32
 *     mode a product whose operands the tensor-memory-access unit cannot read
 *     (a base address not 16-byte aligned, a row stride not a multiple of 4)
 *     runs on the CUDA cores instead; the model's own buffers never do.
 *   - A tensor-core kernel whose pipeline wait exceeds one second gives up,
 *     sets GPT2_STATUS_TIMEOUT in *status and returns without faulting.
 */
#ifndef GPT2_B300_OPS_H
#define GPT2_B300_OPS_H

#include <stddef.h>
#include <stdint.h>
#include "gpt2.h"

#ifdef __cplusplus
extern "C" {
#endif

/* device status bits */
#define GPT2_STATUS_BAD_TOKEN   1
#define GPT2_STATUS_BAD_TARGET  2
#define GPT2_STATUS_TIMEOUT     4

/* Encoder: x[b,t,:] = wte[tok[b,t],:] + wpe[t,:]  ("GPT-2 from scratch with
 * torch", section 从词到编码).  tok [B*T] int32; wte [V,C], wpe [>=T,C],
 * x [B*T,C] (16B).  An id outside [0,V) writes zeros and sets BAD_TOKEN. */
int gpt2_op_encoder_forward(float* x, const int* tok, const float* wte, const float* wpe,
                            int B, int T, int C, int V, int* status, void* stream);

/* Encoder backward, deterministic.  dwte[v,:] += sum over positions with
 * tok == v of dx[pos,:], summed in a fixed order (ascending positions within
 * segments of 64 sorted entries, then segment order); dwpe[t,:] =
 * sum_b dx[b,t,:] for t < T (rows t >= T of dwpe are set to 0; dwpe has maxT
 * rows).  scratch: gpt2_op_encoder_backward_scratch_bytes(B*T, V, C) bytes. */
size_t gpt2_op_encoder_backward_scratch_bytes(int BT, int V, int C);
int gpt2_op_encoder_backward(float* dwte, float* dwpe, const float* dx, const int* tok,
                             int B, int T, int maxT, int C, int V, void* scratch,
                             size_t scratch_bytes, void* stream);

/* LayerNorm over rows of x [N,C] (16B): mean, rstd = 1/sqrt(var + 1e-5)
 * (biased variance), y = (x-mean)*rstd*w + b.  mean, rstd [N] are saved for
 * the backward.  ("GPT-2 from scratch with torch", Transformer block, eps 1e-5.)
 * The _bf16 form writes y as bf16 (round to nearest even). */
int gpt2_op_layernorm_forward(float* y, float* mean, float* rstd, const float* x,
                              const float* w, const float* b, int N, int C, void* stream);
int gpt2_op_layernorm_forward_bf16(void* y, float* mean, float* rstd, const float* x,
                                   const float* w, const float* b, int N, int C, void* stream);

/* LayerNorm backward.  With g = dy*w and xhat = (x-mean)*rstd, the row
 * gradient rstd*(g - mean(g) - xhat*mean(g*xhat)) is ADDED to dx when
 * accumulate != 0 (dx is the residual stream's gradient) or written over it
 * when accumulate == 0 (dx is then not read).  dw = sum_rows dy*xhat,
 * db = sum_rows dy (OVERWRITTEN); dx_colsum [C] or NULL: sum_rows of the
 * resulting dx (the bias gradient of the projection whose output fed this
 * residual).  All column sums run in a fixed order (rows within a block, then
 * blocks).  dx_bf16 [N,C] (8-byte aligned) or NULL: also receives the new dx in
 * bf16.  C % 4 == 0, C <= 2048; x, dy, dx, w 16-byte aligned.  Rows stream
 * through shared memory by bulk copy; a copy that does not arrive within a
 * second sets GPT2_STATUS_TIMEOUT in *status (which may be NULL).
 * scratch: gpt2_op_layernorm_backward_scratch_bytes. */
size_t gpt2_op_layernorm_backward_scratch_bytes(int N, int C);
int gpt2_op_layernorm_backward(float* dx, void* dx_bf16, float* dw, float* db, float* dx_colsum,
                               const float* dy, const float* x, const float* w, const float* mean,
                               const float* rstd, int N, int C, int accumulate, void* scratch,
                               size_t scratch_bytes, int* status, void* stream);

/* Linear forward: out[n,o] = sum_i inp[n,i]*w[o,i] + bias[o] (w is [OC,IC]).
 *   bias: [OC] or NULL.  residual: [N,ld_out] or NULL -> out = residual + ...
 *   (residual may alias out).  flags & GPT2_LINEAR_GELU: the sum (+bias) goes
 *   to out_pre [N,ld_out] and out = gelu_tanh(out_pre).
 *   inp [N,IC] row stride IC; out row stride ld_out >= OC.  Columns o >= OC of
 *   out (up to ld_out) are written with 0 when flags & GPT2_LINEAR_ZERO_PAD. */
#define GPT2_LINEAR_GELU      1
#define GPT2_LINEAR_ZERO_PAD  2
int gpt2_op_linear_forward(float* out, float* out_pre, const float* inp, const float* w,
                           const float* bias, const float* residual, int N, int IC, int OC,
                           int ld_out, int flags, int mode, int* status, void* stream);

/* Linear backward, input side: dinp[n,i] = sum_o dout[n,o]*w[o,i]  (OVERWRITES
 * dinp [N,IC]).  dout row stride ld_dout >= OC (columns >= OC are ignored).
 * gelu_x [N,IC] or NULL: dinp is multiplied by gelu_tanh'(gelu_x) (the GELU that
 * produced this layer's input). */
int gpt2_op_linear_backward_input(float* dinp, const float* dout, const float* w,
                                  const float* gelu_x, int N, int IC, int OC, int ld_dout,
                                  int mode, int* status, void* stream);

/* Linear backward, weight side: dw[o,i] = sum_n dout[n,o]*inp[n,i] and, when
 * dbias != NULL, dbias[o] = sum_n dout[n,o]; both OVERWRITTEN and reduced in a
 * fixed order.  scratch: gpt2_op_linear_backward_weight_scratch_bytes. */
size_t gpt2_op_linear_backward_weight_scratch_bytes(int N, int IC, int OC, int mode);
int gpt2_op_linear_backward_weight(float* dw, float* dbias, const float* dout,
                                   const float* inp, int N, int IC, int OC, int ld_dout,
                                   void* scratch, size_t scratch_bytes, int mode, int* status,
                                   void* stream);

/* Bias gradient alone: db[o] = sum_n dout[n*ld_dout + o] for o < OC,
 * OVERWRITTEN, summed in fp32 in a fixed order (row chunks, then chunk order).
 * dout is fp32, or bf16 when dout_bf16 != 0, with any element alignment (a
 * column slice of a wider matrix is fine: unaligned rows are read one element
 * at a time, which gives the same sums).  Any N >= 1.
 * scratch: gpt2_op_bias_grad_scratch_bytes(N, OC) bytes. */
size_t gpt2_op_bias_grad_scratch_bytes(int N, int OC);
int gpt2_op_bias_grad(float* db, const void* dout, int dout_bf16, int N, int OC, int ld_dout,
                      void* scratch, size_t scratch_bytes, void* stream);

/* General GEMM on one product: D[m,n] = sum_k A(m,k) B(n,k), fp32 accumulation,
 * then the linear-layer epilogue.  A(m,k) = A[m*lda + k] when a_kmajor, else
 * A[k*lda + m]; B(n,k) = B[n*ldb + k] when b_kmajor, else B[k*ldb + n].  A and B
 * are fp32 (mode FP32 or TF32) or bf16 (bf16 != 0, mode BF16; tensor cores
 * only).  Epilogue per element, in this order: + bias[n]; GELU (out_pre = value,
 * value = gelu(value)); + residual[m*ldo+n]; * gelu'(gelu_x[m*ldg+n]); stored to
 * out[m*ldo+n] as fp32, or bf16 when out_bf16.  out_pre is bf16 when pre_bf16,
 * gelu_x bf16 when gelu_x_bf16 (else fp32).  Pointers may be NULL to skip.
 * colsum [ceil(M/32), N] fp32 (tensor-core paths only; ENOTSUP on the CUDA
 * cores): row g receives the column sums of the final values (before bf16
 * rounding) of rows 32g .. 32g+31, summed in a fixed order -- a bias gradient
 * of the product's output is the sum of these rows. */
typedef struct {
    int M, N, K;
    const void* A; int lda; int a_kmajor;
    const void* B; int ldb; int b_kmajor;
    int bf16;
    void* out; int ldo; int out_bf16;
    void* out_pre;
    const float* bias;
    const float* residual;
    const void* gelu_x; int ldg;
    int gelu;
    int pre_bf16;
    int gelu_x_bf16;
    float* colsum;
} gpt2_gemm_args;
int gpt2_op_gemm(const gpt2_gemm_args* args, int mode, int* status, void* stream);

/* fp32 -> bf16, round to nearest even, n values. */
int gpt2_op_to_bf16(void* dst, const float* src, size_t n, void* stream);

/* Allocation-free bias gradient.  Same result as gpt2_op_bias_grad, but the
 * caller passes no scratch and the library allocates nothing: the partial sums
 * live in a fixed device array inside the library (4 MiB, every GPU that loads
 * the library holds it until the process exits).  It is for callers that
 * cannot call cudaMalloc: a host application that owns the whole device memory
 * budget through its own pool and gives a plugin only input and output
 * buffers, or a loop that plans all memory at start-up and may not allocate
 * (or synchronise the device, as cudaMalloc can) once it runs.  There is no
 * counterpart on the pages; it exists for this calling convention only.
 *   Limit: ceil(N / 256) * OC <= GPT2_BIAS_GRAD_NOALLOC_MAX_PARTIALS, otherwise
 *   GPT2_ENOMEM is returned and nothing is launched.
 *   The first call on a device looks up the array's device address (with that
 *   device current); make that first call before any stream capture.
 *   All calls share the one array: calls that overlap on the GPU (other
 *   streams, other threads) race and must be serialised by the caller.  Every
 *   partial read is written earlier in the same call, so no clearing is needed
 *   between calls. */
#define GPT2_BIAS_GRAD_NOALLOC_MAX_PARTIALS (1u << 20)
int gpt2_op_bias_grad_noalloc(float* db, const float* dout, int N, int OC, int ld_dout,
                              void* stream);

/* Causal self-attention forward over qkv [B,T,3C] (queries, keys, values at
 * column offsets 0, C, 2C; head h owns columns h*hs..h*hs+hs-1 of each):
 * per (b,h), O = softmax(mask(Q K^T / sqrt(hs))) V, heads side by side in
 * y [B,T,C]; lse [B,H,T] (fp32) receives the row log-sum-exp of the scaled
 * scores.  ("GPT-2 from scratch with torch", section 自注意力.)  hs <= 64,
 * hs % 4 == 0.  qkv and y are fp32, or bf16 in GPT2_MODE_BF16 (there hs % 8 == 0,
 * else ENOTSUP). */
int gpt2_op_attention_forward(void* y, float* lse, const void* qkv, int B, int T, int C,
                              int H, int mode, int* status, void* stream);

/* Causal self-attention backward: dqkv [B,T,3C] (OVERWRITTEN) from dy [B,T,C],
 * the forward's qkv, y and lse; dqkv, dy, qkv, y are bf16 in GPT2_MODE_BF16.
 * scratch: gpt2_op_attention_backward_scratch_bytes. */
size_t gpt2_op_attention_backward_scratch_bytes(int B, int T, int H);
int gpt2_op_attention_backward(void* dqkv, const void* dy, const void* qkv, const void* y,
                               const float* lse, int B, int T, int C, int H, void* scratch,
                               size_t scratch_bytes, int mode, int* status, void* stream);

/* ---- dropout ---------------------------------------------------------------
 * Inverted dropout ("GPT-2 from scratch with torch", sections 总体架构,
 * 近看 Transformer block：自注意力, 近看 Transformer block：前馈网络（MLP）;
 * "从头搭建GPT(Andrej Karpathy) 笔记", section 继续增加改进的点): an element
 * is kept with probability 1 - p (0 <= p < 1) and scaled by 1/(1 - p).
 * Keep masks are bit-packed by rows: a row of `cols` elements takes
 * ceil(cols/32) uint32 words, bit b of word k is column 32k + b, bits past the
 * row's end are 0.  Element e = row * cols + col is kept when word e mod 4 of
 * Philox4x32-10(counter (lo32(e/4), hi32(e/4), site, step),
 * key (lo32(seed), hi32(seed))) is at least floor(p * 2^32) (Philox4x32-10:
 * Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC 2011).  gpt2_set_dropout in gpt2.h gives the sites and steps the
 * training step uses. */

/* Words of a mask of `rows` rows of `cols` elements (0 for invalid sizes). */
size_t gpt2_op_dropout_mask_words(long long rows, int cols);

/* Draw the keep bits of rows x cols elements into bits (device, that many
 * words).  causal_T > 0 marks the attention weights: cols == causal_T, rows =
 * B*H*T are (b, h, i) with i = row % T, and words whose first column is past
 * the diagonal (32k > i) are written as 0 without drawing.  Asynchronous.
 * Errors: EINVAL (bad sizes, p outside [0, 1)). */
int gpt2_op_dropout_mask(uint32_t* bits, long long rows, int cols, int causal_T, unsigned long long seed,
                         unsigned int site, unsigned int step, float p, void* stream);

/* out[N, C] = res + keep o out / (1 - p)  (res NULL: out = keep o out / (1 - p)),
 * in place; fp32, 16-byte aligned, C % 4 == 0; bits from gpt2_op_dropout_mask
 * with rows N, cols C.  The forward of a dropped c_proj output added to the
 * residual stream, and of the dropped embedding output.  Errors: EINVAL. */
int gpt2_op_dropout_residual(float* out, const float* res, const uint32_t* bits, int N, int C, float p,
                             void* stream);

/* dst[N, C] = keep o src / (1 - p): the backward of the dropout above.  src
 * fp32 (16-byte aligned); dst fp32 (may be src) or, with dst_bf16 != 0, bf16
 * (8-byte aligned); C % 4 == 0.  Errors: EINVAL. */
int gpt2_op_dropout_backward(void* dst, int dst_bf16, const float* src, const uint32_t* bits, int N, int C,
                             float p, void* stream);

/* LayerNorm backward whose residual gradient also feeds a dropped branch (a
 * c_proj output that went through dropout before the residual addition): as
 * gpt2_op_layernorm_backward, and dx_drop [N,C] receives keep o dx / (1 - p)
 * (bf16 with dx_drop_bf16 != 0, 8-byte aligned; else fp32, 16-byte aligned),
 * drop_colsum [C] (or NULL) the column sums of dx_drop in fixed order: that
 * branch's bias gradient.  bits: keep bits with rows N, cols C.  C <= 768.
 * Errors: EINVAL, ENOMEM, ENOTSUP (C > 768). */
int gpt2_op_layernorm_backward_dropout(float* dx, void* dx_drop, int dx_drop_bf16, float* dw, float* db,
                                       float* drop_colsum, const float* dy, const float* x, const float* w,
                                       const float* mean, const float* rstd, int N, int C, int accumulate,
                                       const uint32_t* bits, float p, void* scratch, size_t scratch_bytes,
                                       int* status, void* stream);

/* Attention forward and backward with dropout on the attention weights: as
 * gpt2_op_attention_forward / _backward, with A = P o K / (1 - p) in place of
 * the softmax weights P (K the keep bits of gpt2_op_dropout_mask with rows
 * B*H*T, cols = causal_T = T):  O = A V;  the backward gives dV = A^T dO,
 * dP = (dO V^T) o K / (1 - p), dS = P o (dP - rowsum(dO o O)).  lse stays the
 * log-sum-exp of the undropped scores.  bits must not be NULL.  Errors as the
 * calls without dropout, and EINVAL for p outside [0, 1). */
int gpt2_op_attention_forward_dropout(void* y, float* lse, const void* qkv, int B, int T, int C, int H,
                                      int mode, const uint32_t* bits, float p, int* status, void* stream);
int gpt2_op_attention_backward_dropout(void* dqkv, const void* dy, const void* qkv, const void* y,
                                       const float* lse, int B, int T, int C, int H, void* scratch,
                                       size_t scratch_bytes, int mode, const uint32_t* bits, float p,
                                       int* status, void* stream);

/* Fused softmax cross-entropy over logits z [N, ld] (16B, ld % 4 == 0, ld >= V):
 * losses[n] = logsumexp(z[n,:V]) - z[n,tgt[n]]; then the gradient
 * (softmax(z[n,:V])[v] - [v == tgt[n]]) * dscale for v < V and 0 for V <= v < ld
 * is written IN PLACE over z, or, when dz_bf16 != NULL, to dz_bf16 [N, ld]
 * (bf16, 8-byte aligned) with z left unchanged.  dscale is 1/(number of
 * positions) for the mean loss; 0 skips the gradient.  A target outside [0,V)
 * sets BAD_TARGET and that row's loss and gradient to 0.  ("从头搭建GPT 笔记",
 * section 计算loss.) */
int gpt2_op_crossentropy(float* losses, float* z, void* dz_bf16, const int* tgt, int N, int V,
                         int ld, float dscale, int* status, void* stream);

/* The same cross-entropy on bf16 logits z [N, ld] (16B, ld % 8 == 0, ld >= V,
 * ld <= GPT2_CE_BF16_MAX_LD): losses as above, computed from the stored bf16 values in
 * fp32; then the gradient, rounded to bf16, is written IN PLACE over z
 * (columns V <= v < ld set to 0).  dscale 0 skips the gradient and leaves z
 * unchanged.  A target outside [0,V) sets BAD_TARGET and that row's loss and
 * gradient to 0.  ("从头搭建GPT 笔记", section 计算loss.)  EINVAL for a row
 * longer than the limit or a misaligned z. */
#define GPT2_CE_BF16_MAX_LD 56320
int gpt2_op_crossentropy_bf16(float* losses, void* z, const int* tgt, int N, int V, int ld,
                              float dscale, int* status, void* stream);

/* Top-k sampling ("GPT-2 from scratch with torch", section 生成样本: keep the
 * k highest scores, turn them into probabilities, draw the next token):
 * out[n] = a token of row n of logits [N, ld] (ld >= V), drawn with the
 * caller's uniform number u[n] in [0, 1) (device, one per row; the library
 * draws no random numbers).  The kept set is the k largest of logits[n, 0..V)
 * (1 <= k <= 64), taken in the order value descending, index ascending (so the
 * lower index wins a tie at the cut), NaN entries skipped; with p_v =
 * exp(z_v - max) / sum over the kept set, out[n] is the smallest kept index v
 * whose cumulative p (over kept indices <= v) exceeds u[n], or the largest kept
 * index when rounding leaves u[n] at or above the total.  k = 1 is the greedy
 * choice.  A row with no candidate gives 0.  EINVAL for k outside [1, 64]. */
int gpt2_op_sample_topk(int* out, const float* logits, int N, int V, int ld, int k, const float* u,
                        void* stream);

/* Greedy token choice: out[n] = the index of the largest of logits[n, 0..V)
 * (row stride ld >= V), the lowest index on ties; NaN entries never win (a row
 * of NaN gives 0).  ("GPT-2 from scratch with torch", section 生成样本: the
 * next token is taken from the highest scores of the last position.) */
int gpt2_op_argmax(int* out, const float* logits, int N, int V, int ld, void* stream);

/* Sum of losses[N] in a fixed order, times `scale`, written to *out (device). */
int gpt2_op_sum(float* out, const float* losses, int N, float scale, void* stream);

/* AdamW over n parameters (16B; n % 4 == 0), bias corrections passed in:
 * m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
 * p -= lr * ((m/bc1) / (sqrt(v/bc2) + eps) + wd * p). */
int gpt2_op_adamw(float* p, const float* g, float* m, float* v, size_t n, float lr,
                  float b1, float b2, float eps, float wd, float bc1, float bc2,
                  void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_B300_OPS_H */
