// gemm.cuh -- the GEMM problem shared by the CUDA-core and tensor-core kernels.
//
// D[m,n] = sum_k A(m,k) * B(n,k), fp32 accumulation, then a fused epilogue.
// Each operand is row-major in memory with one contiguous dimension:
//   A "K-major":  A(m,k) = A[m*lda + k]      A "M-major": A(m,k) = A[k*lda + m]
//   B "K-major":  B(n,k) = B[n*ldb + k]      B "N-major": B(n,k) = B[k*ldb + n]
// The three products of a linear layer map onto it as
//   forward  out  = inp . W^T   A = inp (K-major), B = W (K-major)
//   dX       dinp = dout . W    A = dout (K-major), B = W (N-major)
//   dW       dW   = dout^T . inp  A = dout (M-major), B = inp (N-major)
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"

namespace gpt2k {

struct GemmEpilogue {
    void* out;               // [M, ldo], fp32, or bf16 when out_bf16
    int ldo;
    int out_bf16;
    void* out_pre;           // GELU: pre-activation written here (same ldo), fp32 or bf16
    int pre_bf16;
    const float* bias;       // [N] or null
    const float* residual;   // [M, ldo] or null: out = residual + (acc + bias)
    const void* gelu_x;      // [M, ldg] or null: out = acc * gelu'(gelu_x), fp32 or bf16
    int gelu_x_bf16;
    int ldg;
    int gelu;                // 1: out_pre = acc + bias, out = gelu(out_pre)
    float* colsum;           // [ceil(M/32), N] or null: per 32-row group, the column sums of the
                             // stored values (before any bf16 rounding); tensor-core kernel only
};

struct GemmProblem {
    int M, N, K;
    const void* A; int lda; bool a_kmajor;
    const void* B; int ldb; bool b_kmajor;
    int* status;             // device status word for bounded-wait timeouts, or null
    bool bf16 = false;       // A and B hold bf16 (tensor cores only); else fp32
};

// Epilogue of one output element; shared by every GEMM kernel.
__device__ __forceinline__ void epilogue_store(const GemmEpilogue& e, int m, int n, float acc) {
    size_t o = (size_t)m * e.ldo + n;
    float v = acc;
    if (e.bias) v += e.bias[n];
    if (e.gelu) {
        if (e.pre_bf16) reinterpret_cast<__nv_bfloat16*>(e.out_pre)[o] = __float2bfloat16_rn(v);
        else reinterpret_cast<float*>(e.out_pre)[o] = v;
        v = gelu_fwd(v);
    }
    if (e.residual) v += e.residual[o];
    if (e.gelu_x) {
        const size_t g = (size_t)m * e.ldg + n;
        v *= gelu_grad(e.gelu_x_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(e.gelu_x)[g])
                                     : reinterpret_cast<const float*>(e.gelu_x)[g]);
    }
    if (e.out_bf16) reinterpret_cast<__nv_bfloat16*>(e.out)[o] = __float2bfloat16_rn(v);
    else reinterpret_cast<float*>(e.out)[o] = v;
}

// Tiled TMA descriptor over a row-major tensor of `rank` dimensions (dims and
// box innermost first, strides in bytes for dimensions 1..rank-1), zero fill.
bool encode_tensor_map(CUtensorMap* map, bool bf16, int rank, const void* ptr, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz);

// CUDA-core fp32 GEMM (strict mode).
int gemm_simt(const GemmProblem& p, const GemmEpilogue& e, cudaStream_t st);

// tcgen05 tensor-core GEMM, tf32 (fp32 operands) or bf16 operands (p.bf16).  `split` > 1 splits K into
// that many contiguous ranges; each range writes its own [M, N] fp32 slice of
// `partial` (plain accumulators, no epilogue), to be summed in a fixed order.
int gemm_tc(const GemmProblem& p, const GemmEpilogue& e, cudaStream_t st);
int gemm_tc_splitk(const GemmProblem& p, float* partial, int split, cudaStream_t st);
bool gemm_tc_supported(const GemmProblem& p);
// Whether a bf16 product with epilogue `e` (null: none, as for split-K slices)
// runs on CTA pairs (cta_group::2, 256 x 256 tiles), and how many pairs the
// persistent grid holds.
bool gemm_tc_pair(const GemmProblem& p, const GemmEpilogue* e);
int gemm_tc_pair_slots();
bool gemm_tc_epilogue_supported(const GemmEpilogue& e);

// A column reduction left for later: dst[k][c] = sum over g of part[g * ld +
// k * seg + c] for c < seg, k < width / seg (groups summed in a fixed order).
// Ops that produce per-group partial sums (the LayerNorm backward, the fused
// bias gradients) can describe them with one of these instead of launching
// their own reduction, and the training step then sums all of them in one
// launch (colsum_batch).
struct ColReduce {
    const float* part;
    int groups, ld, width, seg;
    float* dst[3];
};
int colsum_batch(const ColReduce* r, int n, cudaStream_t st);

// Linear-layer products for any operand type (linear.cu); bf16 requires
// mode GPT2_MODE_BF16.
// A bf16 GELU pre-activation (out_pre, gelu_x) goes with bf16 operands (`bf16`).
int linear_forward(void* out, bool out_bf16, void* out_pre, const void* inp, const void* w,
                   bool bf16, const float* bias, const float* residual, int N, int IC, int OC,
                   int ld_out, int flags, int mode, int* status, cudaStream_t st);
// With db != null, db[i] = sum over rows of dinp[:, i] as well: from the
// epilogue's per-32-row column sums on the tensor cores, else by a pass over
// dinp; cs is scratch of linear_colsum_bytes(N, IC) bytes.
// With defer != null and the column sums fused into the tensor-core epilogue,
// their reduction is described in *defer (defer->part == null otherwise)
// instead of launched.
// ks / ks_bytes: optional scratch for K slices of a plain dX product (fp32
// output, no GELU' or bias sums); linear_backward_input_scratch_bytes sizes it
// for every row count up to N.
int linear_backward_input(void* dinp, bool dinp_bf16, const void* dout, const void* w, bool bf16,
                          const void* gelu_x, int N, int IC, int OC, int ld_dout, int mode,
                          int* status, cudaStream_t st, float* db = nullptr, void* cs = nullptr,
                          size_t cs_bytes = 0, ColReduce* defer = nullptr, void* ks = nullptr,
                          size_t ks_bytes = 0);
size_t linear_backward_input_scratch_bytes(int N, int IC, int OC, int mode);
size_t linear_colsum_bytes(int N, int IC);
// db[c] = sum over g of part[g * OC + c], in group order.
int colsum_reduce(float* db, const float* part, int groups, int OC, cudaStream_t st);
int linear_backward_weight(float* dw, const void* dout, const void* inp, bool bf16, int N, int IC,
                           int OC, int ld_dout, void* scratch, size_t scratch_bytes, int mode,
                           int* status, cudaStream_t st);
int bias_grad_any(float* db, const void* dout, bool bf16, int N, int OC, int ld, void* scratch,
                  size_t scratch_bytes, cudaStream_t st);
// Attention backward (gpt2_op_attention_backward); with colsum != null the
// tcgen05 kernels also leave per-32-row column sums of dqkv in colsum
// ([B * ceil(T/32), 3C]) and set *colsum_done; other paths leave it false.
int attention_backward(void* dqkv, const void* dy, const void* qkv, const void* y, const float* lse, int B,
                       int T, int C, int H, void* scratch, size_t scratch_bytes, int mode, int* status,
                       cudaStream_t st, float* colsum, bool* colsum_done);
// Decoding with a key/value cache (decode.cu), fp32, at most 16 rows; the
// position is read from device memory (*dpos) and advanced by decode_advance.
int decode_embed(float* x, const int* tok, const float* wte, const float* wpe, int B, int C, int V,
                 const int* dpos, int* status, cudaStream_t st);
int decode_gemv(float* out, int ld, const float* in, const float* W, const float* bias, const float* resid,
                int B, int IC, int OC, int act, float* cache, int maxT, const int* dpos, cudaStream_t st);
int decode_attention(float* y, const float* qkv, const float* cache, int B, int C, int H, int maxT,
                     const int* dpos, cudaStream_t st);
int decode_advance(int* dpos, cudaStream_t st);
int layernorm_forward(void* y, bool out_bf16, float* mean, float* rstd, const float* x,
                      const float* w, const float* b, int N, int C, cudaStream_t st);
int to_bf16(void* dst, const float* src, size_t n, cudaStream_t st);

}  // namespace gpt2k
