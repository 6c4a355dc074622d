// crossentropy.cu -- fused softmax cross-entropy over the vocabulary, the
// gradient written in place over the logits, and a fixed-order loss sum.
//
// loss_n = logsumexp(z_n) - z_n[target_n] (natural log; the mean over positions
// is the training loss, "从头搭建GPT(Andrej Karpathy) 笔记", section 计算loss);
// d(mean loss)/dz_n = (softmax(z_n) - onehot(target_n)) / (number of positions).
//
// One block per row.  Pass 1 streams the row once (128-bit loads) keeping a
// per-thread running maximum and rescaled sum, combined across the block; pass
// 2 re-reads the row (it is still in L2) and overwrites it with the gradient.
// DRAM traffic is one read and one write of the logits.
#include <cuda_bf16.h>

#include "common.cuh"

namespace gpt2k {

constexpr int CE_THREADS = 512;

__device__ __forceinline__ void lse_combine(float& m, float& s, float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; s = s2; return; }
    if (m2 > m) { s = s * expf(m - m2) + s2; m = m2; }
    else s += s2 * expf(m2 - m);
}

__global__ void __launch_bounds__(CE_THREADS)
crossentropy_kernel(float* __restrict__ losses, float* __restrict__ z, __nv_bfloat16* __restrict__ dz16,
                    const int* __restrict__ tgt, int V, int ld, float dscale, int* status) {
    __shared__ float sm[CE_THREADS / 32], ss[CE_THREADS / 32];
    __shared__ float s_lse, s_zt;
    const int row = blockIdx.x, tid = threadIdx.x;
    float* zr = z + (size_t)row * ld;
    float4* z4 = reinterpret_cast<float4*>(zr);
    const int n4 = ld >> 2;
    float m = -INFINITY, s = 0.f;
    for (int c = tid; c < n4; c += CE_THREADS) {
        float4 v = z4[c];
        float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            if (c * 4 + k < V) {
                float x = e[k];
                if (x > m) { s = s * expf(m - x) + 1.f; m = x; }
                else s += expf(x - m);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
        lse_combine(m, s, m2, s2);
    }
    if ((tid & 31) == 0) { sm[tid >> 5] = m; ss[tid >> 5] = s; }
    __syncthreads();
    if (tid == 0) {
        float M = sm[0], S = ss[0];
        for (int w = 1; w < CE_THREADS / 32; w++) lse_combine(M, S, sm[w], ss[w]);
        float lse = M + logf(S);
        int t = tgt[row];
        bool ok = t >= 0 && t < V;
        if (!ok) set_status(status, GPT2_STATUS_BAD_TARGET);
        s_lse = ok ? lse : INFINITY;   // INFINITY: gradient row becomes 0 below
        s_zt = ok ? zr[t] : 0.f;
        losses[row] = ok ? lse - s_zt : 0.f;
    }
    __syncthreads();
    if (dscale == 0.f) return;
    const float lse = s_lse;
    const int t = tgt[row];
    for (int c = tid; c < n4; c += CE_THREADS) {
        float4 v = z4[c];
        float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            int idx = c * 4 + k;
            float p = idx < V ? expf(e[k] - lse) : 0.f;
            e[k] = (p - (idx == t ? 1.f : 0.f)) * dscale;
            if (idx >= V || lse == INFINITY) e[k] = 0.f;
        }
        if (dz16) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(e[0], e[1]), hi = __floats2bfloat162_rn(e[2], e[3]);
            reinterpret_cast<uint2*>(dz16 + (size_t)row * ld)[c] =
                make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        } else {
            z4[c] = make_float4(e[0], e[1], e[2], e[3]);
        }
    }
}

// One block: thread t sums elements t, t+1024, ... in order; then a fixed tree.
__global__ void __launch_bounds__(1024) sum_kernel(float* __restrict__ out, const float* __restrict__ x,
                                                   int N, float scale) {
    __shared__ float sh[1024];
    float s = 0.f;
    for (int i = threadIdx.x; i < N; i += 1024) s += x[i];
    sh[threadIdx.x] = s;
    __syncthreads();
    for (int o = 512; o > 0; o >>= 1) {
        if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) *out = sh[0] * scale;
}

}  // namespace gpt2k

using namespace gpt2k;

GPT2_API int gpt2_op_crossentropy(float* losses, float* z, void* dz_bf16, const int* tgt, int N,
                                  int V, int ld, float dscale, int* status, void* stream) {
    if (!losses || !z || !tgt || N < 1 || V < 1 || ld < V || ld % 4 || !aligned16(z))
        return GPT2_EINVAL;
    if (dz_bf16 && (reinterpret_cast<uintptr_t>(dz_bf16) & 7)) return GPT2_EINVAL;
    count_launch(), crossentropy_kernel<<<N, CE_THREADS, 0, as_stream(stream)>>>(
        losses, z, static_cast<__nv_bfloat16*>(dz_bf16), tgt, V, ld, dscale, status);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

GPT2_API int gpt2_op_sum(float* out, const float* x, int N, float scale, void* stream) {
    if (!out || !x || N < 1) return GPT2_EINVAL;
    count_launch(), sum_kernel<<<1, 1024, 0, as_stream(stream)>>>(out, x, N, scale);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}
