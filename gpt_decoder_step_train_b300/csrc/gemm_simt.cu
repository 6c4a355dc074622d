// gemm_simt.cu -- fp32 GEMM on the CUDA cores (the strict-fp32 mode).
//
// 128x128 output tile per 256-thread block, k-step 8, each thread an 8x8
// register tile; the next k-slab is prefetched into registers while the
// current one is consumed from shared memory (double buffer).  Loads are
// bounds-checked, so M, N, K need no alignment.
#include "gemm.cuh"

namespace gpt2k {

constexpr int SG_BM = 128, SG_BN = 128, SG_BK = 8, SG_PAD = 4;

template <bool AK, bool BK>
__global__ void __launch_bounds__(256)
sgemm_kernel(int M, int N, int K, const float* __restrict__ A, int lda,
             const float* __restrict__ B, int ldb, GemmEpilogue e) {
    __shared__ __align__(16) float As[2][SG_BK][SG_BM + SG_PAD];
    __shared__ __align__(16) float Bs[2][SG_BK][SG_BN + SG_PAD];
    const int tid = threadIdx.x;
    const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
    float ra[4], rb[4];

    // K-major operand: thread loads row tid/2, k = (tid%2)*4 + j
    // MN-major operand: thread loads k = tid/32, row = (tid%32)*4 + j
    auto load = [&](const float* __restrict__ X, int ld, bool kmaj, int r0, int R, int k0,
                    float* reg) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int r, k;
            if (kmaj) { r = tid >> 1; k = ((tid & 1) << 2) + j; }
            else { k = tid >> 5; r = ((tid & 31) << 2) + j; }
            int gr = r0 + r, gk = k0 + k;
            reg[j] = (gr < R && gk < K) ? (kmaj ? X[(size_t)gr * ld + gk] : X[(size_t)gk * ld + gr]) : 0.f;
        }
    };
    auto store = [&](float (*S)[SG_BM + SG_PAD], bool kmaj, const float* reg) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int r, k;
            if (kmaj) { r = tid >> 1; k = ((tid & 1) << 2) + j; }
            else { k = tid >> 5; r = ((tid & 31) << 2) + j; }
            S[k][r] = reg[j];
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) acc[i][j] = 0.f;

    const int ty = tid >> 4, tx = tid & 15;
    load(A, lda, AK, m0, M, 0, ra);
    load(B, ldb, BK, n0, N, 0, rb);
    store(As[0], AK, ra);
    store(Bs[0], BK, rb);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < K; k0 += SG_BK) {
        bool more = k0 + SG_BK < K;
        if (more) {
            load(A, lda, AK, m0, M, k0 + SG_BK, ra);
            load(B, ldb, BK, n0, N, k0 + SG_BK, rb);
        }
#pragma unroll
        for (int kk = 0; kk < SG_BK; kk++) {
            float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
            float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
            float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int j = 0; j < 8; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) {
            store(As[buf ^ 1], AK, ra);
            store(Bs[buf ^ 1], BK, rb);
        }
        __syncthreads();
        buf ^= 1;
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
        int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (n < N) epilogue_store(e, m, n, acc[i][j]);
        }
    }
}

int gemm_simt(const GemmProblem& gp, const GemmEpilogue& e, cudaStream_t st) {
    if (gp.M <= 0 || gp.N <= 0) return GPT2_OK;
    if (gp.bf16) return GPT2_ENOTSUP;
    struct {
        int M, N, K, lda, ldb;
        const float *A, *B;
        bool a_kmajor, b_kmajor;
    } p{gp.M, gp.N, gp.K, gp.lda, gp.ldb, static_cast<const float*>(gp.A),
        static_cast<const float*>(gp.B), gp.a_kmajor, gp.b_kmajor};
    dim3 grid(ceil_div(p.N, SG_BN), ceil_div(p.M, SG_BM));
    if (p.a_kmajor && p.b_kmajor)
        count_launch(), sgemm_kernel<true, true><<<grid, 256, 0, st>>>(p.M, p.N, p.K, p.A, p.lda, p.B, p.ldb, e);
    else if (p.a_kmajor && !p.b_kmajor)
        count_launch(), sgemm_kernel<true, false><<<grid, 256, 0, st>>>(p.M, p.N, p.K, p.A, p.lda, p.B, p.ldb, e);
    else if (!p.a_kmajor && !p.b_kmajor)
        count_launch(), sgemm_kernel<false, false><<<grid, 256, 0, st>>>(p.M, p.N, p.K, p.A, p.lda, p.B, p.ldb, e);
    else
        count_launch(), sgemm_kernel<false, true><<<grid, 256, 0, st>>>(p.M, p.N, p.K, p.A, p.lda, p.B, p.ldb, e);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k
