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
#include "common.cuh"

namespace gpt2k {

struct GemmEpilogue {
    float* out;              // [M, ldo]
    int ldo;
    float* out_pre;          // GELU: pre-activation written here (same ldo)
    const float* bias;       // [N] or null
    const float* residual;   // [M, ldo] or null: out = residual + (acc + bias)
    const float* gelu_x;     // [M, ldg] or null: out = acc * gelu'(gelu_x)
    int ldg;
    int gelu;                // 1: out_pre = acc + bias, out = gelu(out_pre)
};

struct GemmProblem {
    int M, N, K;
    const float* A; int lda; bool a_kmajor;
    const float* B; int ldb; bool b_kmajor;
    int* status;             // device status word for bounded-wait timeouts, or null
};

// Epilogue of one output element; shared by every GEMM kernel.
__device__ __forceinline__ void epilogue_store(const GemmEpilogue& e, int m, int n, float acc) {
    size_t o = (size_t)m * e.ldo + n;
    float v = acc;
    if (e.bias) v += e.bias[n];
    if (e.gelu) {
        e.out_pre[o] = v;
        v = gelu_fwd(v);
    }
    if (e.residual) v += e.residual[o];
    if (e.gelu_x) v *= gelu_grad(e.gelu_x[(size_t)m * e.ldg + n]);
    e.out[o] = v;
}

// CUDA-core fp32 GEMM (strict mode).
int gemm_simt(const GemmProblem& p, const GemmEpilogue& e, cudaStream_t st);

// tcgen05 tensor-core GEMM with tf32 operands.  `split` > 1 splits K into
// that many contiguous ranges; each range writes its own [M, N] fp32 slice of
// `partial` (plain accumulators, no epilogue), to be summed in a fixed order.
int gemm_tc(const GemmProblem& p, const GemmEpilogue& e, cudaStream_t st);
int gemm_tc_splitk(const GemmProblem& p, float* partial, int split, cudaStream_t st);
bool gemm_tc_supported(const GemmProblem& p);

}  // namespace gpt2k
