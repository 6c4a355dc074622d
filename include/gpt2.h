/*
 * gpt2.h -- C ABI of one GPT-2 decoder training step on a B300 (sm_103a).
 *
 * The step: token + position encoder, L pre-norm blocks (LayerNorm, fused QKV
 * projection, causal multi-head self-attention, output projection, residual,
 * LayerNorm, c_fc, tanh-GELU, c_proj, residual), final LayerNorm, logits
 * through the transposed token embedding (tied lm_head, no bias), and the
 * mean softmax cross-entropy; then the backward pass of every layer and an
 * AdamW update.  Architecture: "GPT-2 from scratch with torch" (Posit blog),
 * sections 总体架构, Transformer block, 自注意力, 前馈网络（MLP）, 输出.
 * Training loop and per-layer hand-written backward: "1000 行 C 代码完成 GPT-2
 * 训练的 LLM.c" (bigegpt.com).
 *
 * Conventions
 *   - All pointers marked "device" point to CUDA device memory of the current
 *     device; "host" pointers to host memory.  Pointers marked "device or host"
 *     accept either (copied with cudaMemcpyDefault; pinned host memory keeps
 *     the copy asynchronous).
 *   - Every call is ordered on the stream given in gpt2_config.stream (NULL:
 *     the legacy default stream) and is asynchronous, except gpt2_forward,
 *     which reads back the mean loss (one 4-byte device-to-host copy).
 *   - Floating point data is IEEE fp32.  Token ids are int32.
 *   - Functions returning int return GPT2_OK (0) or a negative GPT2_E* code.
 *     No function aborts, throws, or traps on the device: device-side checks
 *     (token ids out of range, bounded waits) raise bits in a status word that
 *     the next synchronising call reports.
 */
#ifndef GPT2_B300_H
#define GPT2_B300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define GPT2_OK        0
#define GPT2_EINVAL   -1   /* bad configuration, shape or argument             */
#define GPT2_ENOMEM   -2   /* workspace too small or allocation failed         */
#define GPT2_ECUDA    -3   /* a CUDA runtime call failed                        */
#define GPT2_ETOKEN   -4   /* a token or target id outside [0, V)               */
#define GPT2_ESTATE   -5   /* calls out of order (backward before a forward
                              with targets, adamw before backward)              */
#define GPT2_ETIMEOUT -6   /* a bounded device wait gave up                     */
#define GPT2_ENOTSUP  -7   /* mode or shape not supported on this device        */

/* arithmetic modes for the contractions (GEMMs and attention) */
#define GPT2_MODE_FP32 0   /* strict fp32 on the CUDA cores                     */
#define GPT2_MODE_TF32 1   /* tensor cores: tf32 operands, fp32 accumulation    */
#define GPT2_MODE_BF16 2   /* tensor cores: bf16 operands, fp32 accumulation;
                              weights keep fp32 masters; the residual stream,
                              LayerNorm statistics, softmax, loss and every
                              gradient reduction stay fp32; GEMM and attention
                              operands (LayerNorm outputs, qkv, attention
                              output, GELU output, dlogits, residual-stream
                              gradient copy, dh, d(attention out), dqkv) are
                              stored in bf16 by the kernel that produces them */

typedef struct {
    int V;           /* vocabulary size (50257 for GPT-2)                       */
    int maxT;        /* context length, rows of the position table (1024)       */
    int L;           /* number of blocks                                        */
    int H;           /* attention heads; C % H == 0                             */
    int C;           /* channels; C % 4 == 0                                    */
    int maxB;        /* largest batch a forward may pass (activation capacity)  */
    int mode;        /* GPT2_MODE_*                                             */
    void* workspace; /* device memory of at least gpt2_workspace_bytes(cfg)
                        bytes, owned by the caller and kept alive until
                        gpt2_destroy; NULL: the library allocates its own       */
    size_t workspace_bytes;
    void* stream;    /* cudaStream_t for every launch; NULL: default stream     */
} gpt2_config;

typedef struct gpt2 gpt2;

/* Number of fp32 parameters in the flat layout below (124,439,808 for GPT-2
 * 124M, matching the llm.c run log on bigegpt.com).  0 for an invalid config.
 *
 * Flat parameter layout (sixteen tensors, contiguous, in this order; linear
 * weights are [out, in]):
 *   wte[V,C] wpe[maxT,C] ln1w[L,C] ln1b[L,C] qkvw[L,3C,C] qkvb[L,3C]
 *   attprojw[L,C,C] attprojb[L,C] ln2w[L,C] ln2b[L,C] fcw[L,4C,C] fcb[L,4C]
 *   fcprojw[L,C,4C] fcprojb[L,C] lnfw[C] lnfb[C]
 * Gradients and both AdamW moments use the same layout. */
size_t gpt2_num_params(const gpt2_config* cfg);

/* Bytes of device workspace the model needs: gradients, AdamW moments,
 * activations for maxB*maxT rows, logits, and scratch.  0 for an invalid cfg. */
size_t gpt2_workspace_bytes(const gpt2_config* cfg);

/* Create a model over caller-owned parameters.
 *   cfg:    validated (C % H == 0, C % 4 == 0, head size <= 128, V, L, maxT,
 *           maxB >= 1); copied.
 *   params: device, gpt2_num_params(cfg) floats, 16-byte aligned; owned by the
 *           caller, read by forward/backward and updated in place by adamw.
 *   out:    receives the handle; *out is NULL on error.
 * Zeroes both AdamW moments.  Errors: EINVAL, ENOMEM, ECUDA, ENOTSUP. */
int gpt2_create(const gpt2_config* cfg, float* params, gpt2** out);

/* Forward pass on tokens[B,T] (device or host int32, row-major), 1 <= B <= maxB,
 * 1 <= T <= maxT.  targets[B,T] (device or host int32, or NULL): the next-token
 * ids.  With targets, returns the mean cross-entropy over the B*T positions
 * (natural log) and leaves d(loss)/d(logits) in the workspace for the
 * backward; without targets, keeps the logits and returns NaN.  The inputs are
 * copied into the workspace, so the caller may reuse its buffers at once.
 * Returns NaN on error; gpt2_status() then gives the code (EINVAL, ETOKEN,
 * ECUDA).  Synchronises the stream once to read the loss. */
float gpt2_forward(gpt2* m, const int* tokens, const int* targets, int B, int T);

/* Forward-only evaluation: the mean cross-entropy of tokens[B,T] against
 * targets[B,T] (both required; same layout and rules as gpt2_forward), without
 * d(loss)/d(logits): the validation loss of the training loop ("1000 行 C 代码
 * 完成 GPT-2 训练的 LLM.c", section 快速开始吧: the run log reports a validation
 * loss before the first step and every few steps).  The same
 * kernels as gpt2_forward; the cross-entropy skips the gradient pass.  A
 * following gpt2_backward returns ESTATE.  Returns NaN on error (EINVAL,
 * ETOKEN, ECUDA via gpt2_status).  Synchronises the stream once. */
float gpt2_eval(gpt2* m, const int* tokens, const int* targets, int B, int T);

/* Autoregressive decoding with a key/value cache: advance B sequences
 * (1 <= B <= min(maxB, 16)) by one position.  tokens[B] (device or host int32)
 * are the tokens at position pos (0 <= pos < min(maxT, 1024)); pos 0 starts
 * new sequences, every later call must continue them (same B, pos one more than
 * the last call), else ESTATE.  The keys and values of every layer for position
 * pos are appended to the cache (library memory, allocated by the first call:
 * L * maxB * maxT * 2C floats; call it before any stream capture), and the
 * logits of position pos are copied to logits[B, V] (device or host, row
 * stride V) from the library's step buffer: exactly the last row of a full
 * forward over positions 0..pos.  Computed in fp32 from the fp32 parameters in
 * every mode.  The step's kernels read the position from device memory, so the
 * second call with a given B records them as one CUDA graph that later calls
 * with that B replay.  Generation feeds the chosen
 * token back at pos + 1 ("GPT-2 from scratch with torch", section 生成样本;
 * only the new row is computed: "GPT-2ベースの3000バイトCで実装された
 * ChatGPTクローン（2023）", section KVキャッシュ方式).  Asynchronous; an id
 * outside [0, V) shows up as ETOKEN in gpt2_status.  A pending backward is
 * dropped (the next gpt2_backward returns ESTATE).  Errors: EINVAL, ESTATE,
 * ENOMEM, ECUDA. */
int gpt2_decode(gpt2* m, const int* tokens, int B, int pos, float* logits);

/* Dropout for the following gpt2_forward calls (training), not for gpt2_eval or
 * gpt2_decode: with probability p in [0, 1) an element is zeroed and the kept
 * ones are scaled by 1/(1 - p), at the four places the pages put it: the
 * token + position embedding output, the attention weights after the softmax,
 * and each block's attention and MLP c_proj outputs before their residual
 * additions ("GPT-2 from scratch with torch", sections 总体架构,
 * 近看 Transformer block：自注意力 and 近看 Transformer block：前馈网络（MLP）;
 * "从头搭建GPT(Andrej Karpathy) 笔记", section 继续增加改进的点).
 * Draws: Philox4x32-10 under the 64-bit seed as key; the n-th gpt2_forward
 * after this call (n = 0, 1, ...) draws element e (row-major) of site s
 * (0 the embedding output [B,T,C]; for layer l: 1 + 3l the attention weights
 * [B,H,T,T], 2 + 3l the attention c_proj output, 3 + 3l the MLP c_proj output)
 * as word e mod 4 of Philox4x32-10(counter (lo32(e/4), hi32(e/4), s, n),
 * key (lo32(seed), hi32(seed))) and keeps it when that word is at least
 * floor(p * 2^32).  gpt2_backward uses the masks of the last forward.
 * p = 0 turns dropout off (the step is then exactly the one without dropout).
 * The first call with p > 0 allocates the mask memory (about
 * L * maxB * H * maxT * ceil(maxT/32) * 4 bytes); changing p makes the next
 * calls capture their graphs again (the library's own graphs read the draw
 * state from device memory, so every replay draws new masks).  With p > 0,
 * gpt2_forward first copies that state from host memory, so a stream capture
 * of the caller's own that records gpt2_forward fails (ECUDA).  A pending
 * backward is dropped.  Errors: EINVAL (p outside [0, 1)), ENOMEM. */
int gpt2_set_dropout(gpt2* m, float p, unsigned long long seed);

/* Graphs: gpt2_forward, gpt2_eval and gpt2_backward record their kernels into a
 * CUDA graph on the second call with the same kind of call and (B, T), and
 * replay it from the third on, on a library stream ordered after earlier work
 * of the caller's stream and before later work (events); nothing else changes.
 * Called while the caller's stream is being captured, or with tracing on, they
 * launch their kernels directly. */

/* Backward pass of the last forward (which must have had targets).
 * Overwrites the gradient buffer (no accumulation across calls); gradients
 * are those of the mean loss.  Errors: ESTATE, ECUDA. */
int gpt2_backward(gpt2* m);

/* AdamW update of the parameters in place from the current gradients, step
 * t >= 1 (bias correction 1-b1^t, 1-b2^t):
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   p -= lr * ( (m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps) + wd_i * p )
 * with wd_i = wd on the 2-D tensors (wte, wpe, qkvw, attprojw, fcw, fcprojw)
 * and 0 elsewhere.  Errors: EINVAL (t < 1), ESTATE (no backward yet), ECUDA. */
int gpt2_adamw(gpt2* m, float lr, float b1, float b2, float eps, float wd, int t);

/* Release the model (and its workspace if the library allocated it).
 * Synchronises the stream.  NULL is accepted. */
int gpt2_destroy(gpt2* m);

/* Synchronise the stream and return the first error seen by this model
 * (including device-side status bits), then clear it. */
int gpt2_status(gpt2* m);

/* Check of the failure path of the bounded device waits (no counterpart on the
 * pages; failure detection).  Every barrier wait of the tensor-core and
 * bulk-copy kernels gives up after a limit, raises a timeout bit in the
 * model's device status word, makes the other roles of its block leave, and the
 * kernel returns instead of hanging.  This call launches, on the model's
 * stream, one block that runs that same wait on two barriers nothing ever
 * completes: the first wait is limited to wait_us microseconds (1 .. 10^6),
 * the second to the library's one-second limit, and it leaves as soon as the
 * first has given up.  Afterwards gpt2_status(m) returns GPT2_ETIMEOUT (and
 * clears it); the device context and the model stay usable.  Returns EINVAL
 * for a wait_us outside the range, ECUDA if the launch failed, else OK. */
int gpt2_wait_probe(gpt2* m, int wait_us);

/* Static description of a status code. */
const char* gpt2_strerror(int code);

/* Accessors: device pointers into the workspace, valid until gpt2_destroy.
 * gpt2_grads / gpt2_adam_m / gpt2_adam_v: gpt2_num_params floats, flat layout.
 * gpt2_logits: [B*T, row_stride] floats of the last forward; row_stride is the
 * vocabulary padded to a multiple of 128 and written to *row_stride.  Columns
 * >= V hold 0.  After a forward WITH targets the buffer holds d(loss)/d(logits)
 * instead (padded columns 0), except in GPT2_MODE_BF16 (padded vocabulary up to
 * GPT2_CE_BF16_MAX_LD), where the training forward keeps logits and gradient
 * in an internal bf16 buffer and leaves this one as it was.  gpt2_losses: the B*T per-position losses. */
const float* gpt2_grads(gpt2* m);
float* gpt2_adam_m(gpt2* m);
float* gpt2_adam_v(gpt2* m);
const float* gpt2_logits(gpt2* m, int* row_stride);
const float* gpt2_losses(gpt2* m);

/* Activation access for checks: device pointer to activation `which` of
 * block `layer` from the last forward, rows B*T of the given width:
 *   0 encoder output [C]   1 ln_1 output [C]   2 qkv [3C]   3 attention out [C]
 *   4 residual after attention [C]   5 ln_2 output [C]   6 c_fc output [4C]
 *   7 GELU output [4C]   8 block output [C]   9 ln_f output [C]
 * fp32, except 1, 2, 3, 5, 6, 7 and 9 in GPT2_MODE_BF16, which are bf16 (the
 * pointer is then to bf16 values despite its type).  NULL for an invalid index. */
const float* gpt2_activation(gpt2* m, int which, int layer);

/* ---- tracing -------------------------------------------------------------
 * Per-kernel-class timing with CUDA events recorded on the model's stream
 * around every operation of the step (off by default; the events cost about
 * a microsecond of host time each).  Classes: */
#define GPT2_TRACE_ENCODER_FWD      0
#define GPT2_TRACE_LAYERNORM_FWD    1
#define GPT2_TRACE_MATMUL_FWD       2   /* every linear layer's forward GEMM      */
#define GPT2_TRACE_ATTENTION_FWD    3
#define GPT2_TRACE_CROSSENTROPY     4   /* fused softmax-CE and the loss sum      */
#define GPT2_TRACE_MATMUL_BWD_INPUT 5   /* dX GEMMs                               */
#define GPT2_TRACE_MATMUL_BWD_WEIGHT 6  /* dW GEMMs and their split-K sums          */
#define GPT2_TRACE_LAYERNORM_BWD    7
#define GPT2_TRACE_ATTENTION_BWD    8
#define GPT2_TRACE_ENCODER_BWD      9
#define GPT2_TRACE_ADAMW           10
#define GPT2_TRACE_OTHER           11   /* input copies and memsets               */
#define GPT2_TRACE_BIAS_GRAD       12   /* column sums for the bias gradients     */
#define GPT2_TRACE_DROPOUT         13   /* dropout masks and their application   */
#define GPT2_TRACE_CLASSES         14

/* Turn tracing on (1) or off (0); turning it on discards earlier records. */
int gpt2_trace_enable(gpt2* m, int on);

/* Synchronise the stream, then write, for each of the first n classes, the
 * summed device milliseconds (ms[c]) and the number of kernel launches
 * (launches[c]) recorded since the last read; the records are then cleared.
 * ms and launches are host arrays of at least n entries (either may be NULL). */
int gpt2_trace_read(gpt2* m, double* ms, long long* launches, int n);

/* Total number of kernels this library has launched in the process so far. */
long long gpt2_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_B300_H */
