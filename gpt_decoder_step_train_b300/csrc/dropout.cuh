// dropout.cuh -- inverted dropout (dropout.cu): bit-packed keep masks drawn
// with Philox4x32-10, and the element-wise kernels that apply them.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm.cuh"

namespace gpt2k {

// floor(p * 2^32): a draw w keeps its element when w >= this
uint32_t dropout_threshold(float p);
// 1 / (1 - p), the scale of the kept elements
float dropout_scale(float p);
// words of a mask of `rows` rows of `cols` elements
size_t dropout_words(long long rows, int cols);
// Keep bits of rows x cols elements of one site (element e = row * cols + col);
// causal_T > 0: rows are (b, h, i) with i = row % causal_T, and words past
// the diagonal are written as 0.  state: device {key0, key1, step} or null.
int dropout_mask(uint32_t* bits, long long rows, int cols, int causal_T, const uint32_t* state,
                 unsigned long long seed, uint32_t site, uint32_t step, float p, cudaStream_t st);
// out = res + keep o out / (1 - p), res may be null; C % 4 == 0
int dropout_residual(float* out, const float* res, const uint32_t* bits, int N, int C, float p, cudaStream_t st);
// dst = keep o src / (1 - p), dst fp32 or bf16
int dropout_backward(void* dst, bool bf16, const float* src, const uint32_t* bits, int N, int C, float p,
                     cudaStream_t st);
// Attention forward / backward with dropout on the attention weights: bits as
// written by dropout_mask with rows B*H*T, cols = causal_T = T; null: none.
int attention_forward(void* y, float* lse, const void* qkv, int B, int T, int C, int H, int mode, int* status,
                      cudaStream_t st, const uint32_t* bits, float p);
int attention_backward_dropout(void* dqkv, const void* dy, const void* qkv, const void* y, const float* lse, int B,
                               int T, int C, int H, void* scratch, size_t scratch_bytes, int mode, int* status,
                               cudaStream_t st, float* colsum, bool* colsum_done, const uint32_t* bits, float p);

// LayerNorm backward (layernorm.cu) with the operand copy dxo of dx in bf16 or
// fp32; with bits != null that copy is keep o dx / (1 - p) and dx_colsum its
// column sum (the bias gradient of the dropped branch it feeds).  The fused
// form needs layernorm_backward_fuses_dropout(C).
bool layernorm_backward_fuses_dropout(int C);
int layernorm_backward(float* dx, void* dxo, bool dxo_bf16, float* dw, float* db, float* dx_colsum, const float* dy,
                       const float* x, const float* w, const float* mean, const float* rstd, int N, int C,
                       int accumulate, void* scratch, size_t scratch_bytes, int* status, cudaStream_t st,
                       const uint32_t* bits, float p, ColReduce* defer = nullptr);

}  // namespace gpt2k
