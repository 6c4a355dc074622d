// crossentropy.cu -- fused softmax cross-entropy over the vocabulary, the
// gradient written in place over the logits, and a fixed-order loss sum.
//
// loss_n = logsumexp(z_n) - z_n[target_n] (natural log; the mean over positions
// is the training loss, "从头搭建GPT(Andrej Karpathy) 笔记", section 计算loss);
// d(mean loss)/dz_n = (softmax(z_n) - onehot(target_n)) / (number of positions).
//
// One block per row.  Pass 1 streams the row once (128-bit loads) keeping a
// per-thread running maximum and rescaled sum, combined across the block, and
// keeps the row's first 100 KB in shared memory; pass 2 re-reads the row (that
// part from shared memory, the rest from L2) and overwrites it with the
// gradient, or writes the gradient in bf16 to a separate buffer for the bf16
// products.
// DRAM traffic is one read of the logits and one write of the gradient.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"

namespace gpt2k {

constexpr int CE_THREADS = 512;
// Shared-memory cache of a row's first float4s: pass 2 reads that part from
// here and the rest from L2.  Its size also holds residency to two rows per SM,
// so the rows in flight (2 x 148 x 200 KB for GPT-2's vocabulary) fit in L2.
constexpr int CE_CACHE_BYTES = 100 * 1024;

constexpr float CE_LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float block_reduce(float v, float* sh, bool is_max) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, u) : v + u;
    }
    __syncthreads();                       // sh may still be read from the previous reduction
    if (lane == 0) sh[w] = v;
    __syncthreads();
    float r = sh[0];
    for (int k = 1; k < CE_THREADS / 32; k++) r = is_max ? fmaxf(r, sh[k]) : r + sh[k];
    return r;
}

// Pass 1 reads the row from DRAM (128-bit loads) keeping a per-thread running
// maximum and a sum of exponentials rescaled whenever the maximum grows; the
// block combines them into the log-sum-exp.  Pass 2 re-reads the row from L2
// and writes the gradient.  Exponentials are exp2 of log2(e)-scaled differences.
__global__ void __launch_bounds__(CE_THREADS, 2)
crossentropy_kernel(float* __restrict__ losses, float* __restrict__ z, __nv_bfloat16* __restrict__ dz16,
                    const int* __restrict__ tgt, int V, int ld, float dscale, int ncache, int* status) {
    __shared__ float sh[CE_THREADS / 32];
    extern __shared__ float4 zc[];                 // the row's float4s [0, ncache)
    const int row = blockIdx.x, tid = threadIdx.x;
    float* zr = z + (size_t)row * ld;
    float4* z4 = reinterpret_cast<float4*>(zr);
    const int nfull = V >> 2;                      // float4s entirely inside [0, V)
    const int n4 = ld >> 2;
    float mx = -INFINITY, sum = 0.f;               // sum of exp(z - mx) over this thread's elements
    auto add4 = [&](const float4* v, int n) {      // n float4s: one rescale, then 4n exponentials
        float m = mx;
        for (int k = 0; k < n; k++) m = fmaxf(m, fmaxf(fmaxf(v[k].x, v[k].y), fmaxf(v[k].z, v[k].w)));
        if (m > mx) {
            sum *= exp2f((mx - m) * CE_LOG2E);
            mx = m;
        }
        const float ml = mx * CE_LOG2E;
        for (int k = 0; k < n; k++)
            sum += (exp2f(fmaf(v[k].x, CE_LOG2E, -ml)) + exp2f(fmaf(v[k].y, CE_LOG2E, -ml))) +
                   (exp2f(fmaf(v[k].z, CE_LOG2E, -ml)) + exp2f(fmaf(v[k].w, CE_LOG2E, -ml)));
    };
    int c = tid;
    for (; c + 3 * CE_THREADS < nfull; c += 4 * CE_THREADS) {
        // four independent loads in flight before any arithmetic
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; k++) v[k] = z4[c + k * CE_THREADS];
#pragma unroll
        for (int k = 0; k < 4; k++)
            if (c + k * CE_THREADS < ncache) zc[c + k * CE_THREADS] = v[k];
        add4(v, 4);
    }
    for (; c < nfull; c += CE_THREADS) {
        float4 v[1] = {z4[c]};
        if (c < ncache) zc[c] = v[0];
        add4(v, 1);
    }
    for (int v = nfull * 4 + tid; v < V; v += CE_THREADS) {
        const float x = zr[v];
        if (x > mx) {
            sum *= exp2f((mx - x) * CE_LOG2E);
            mx = x;
        }
        sum += exp2f((x - mx) * CE_LOG2E);
    }
    const float M = block_reduce(mx, sh, true);
    const float S = block_reduce(mx == -INFINITY ? 0.f : sum * exp2f((mx - M) * CE_LOG2E), sh, false);
    const float lse = M + logf(S);
    const int t = tgt[row];
    const bool ok = t >= 0 && t < V;
    if (tid == 0) {
        if (!ok) set_status(status, GPT2_STATUS_BAD_TARGET);
        losses[row] = ok ? lse - zr[t] : 0.f;
    }
    if (dscale == 0.f) return;
    __syncthreads();                               // zr[t] is read before the row is overwritten
    const float lsel = lse * CE_LOG2E;
    for (int c = tid; c < n4; c += CE_THREADS) {
        const float4 v = c < ncache ? zc[c] : z4[c];
        float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int idx = c * 4 + k;
            const float p = exp2f(fmaf(e[k], CE_LOG2E, -lsel));
            e[k] = (idx < V && ok) ? (p - (idx == t ? 1.f : 0.f)) * dscale : 0.f;
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

// bf16 logits, gradient written in place (bf16).  One block per row: the row
// is staged once into shared memory with 16-byte asynchronous copies, so DRAM
// sees one read and one write of two bytes per logit.  Pass 1 takes the row
// maximum M; pass 2 computes e = exp(z - M) once per logit, sums it, and keeps
// it in shared memory over the logit as fp16 (e is in (0, 1]; fp16's 11-bit
// significand is finer than the bf16 gradient it feeds; e below 2^-24 becomes
// 0, a gradient term below 2^-24 / positions); pass 3 writes the gradient
// e / sum - [v == target], scaled.  One exponential per logit.  Two blocks per
// SM: one row's copy overlaps the other row's arithmetic.
constexpr int CE16_THREADS = 512;
constexpr int CE16_MAX_ROW_BYTES = GPT2_CE_BF16_MAX_LD * 2;   // 110 KB: two rows per SM

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        f[2 * k] = t.x;
        f[2 * k + 1] = t.y;
    }
}

__device__ __forceinline__ void unpack8_h(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
        f[2 * k] = t.x;
        f[2 * k + 1] = t.y;
    }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack2_h(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(CE16_THREADS, 2)
crossentropy_bf16_kernel(float* __restrict__ losses, __nv_bfloat16* __restrict__ z,
                         const int* __restrict__ tgt, int V, int ld, float dscale, int* status) {
    __shared__ float sh[CE16_THREADS / 32];
    extern __shared__ uint4 zs[];                   // the row, 8 logits per entry; later 8 fp16 e values
    const int row = blockIdx.x, tid = threadIdx.x;
    const int n8 = ld >> 3, nfull = V >> 3;         // 16-byte chunks: in the row, entirely inside [0, V)
    uint4* zr = reinterpret_cast<uint4*>(z + (size_t)row * ld);
    for (int c = tid; c < n8; c += CE16_THREADS)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(&zs[c])),
                     "l"(zr + c)
                     : "memory");
    asm volatile("cp.async.commit_group;\ncp.async.wait_all;" ::: "memory");
    __syncthreads();
    const __nv_bfloat16* zsh = reinterpret_cast<const __nv_bfloat16*>(zs);
    __half* esh = reinterpret_cast<__half*>(zs);
    const int t = tgt[row];
    const bool ok = t >= 0 && t < V;
    const float zt = ok ? __bfloat162float(zsh[t]) : 0.f;   // read before the row is overwritten
    float mx = -INFINITY;
    for (int c = tid; c < nfull; c += CE16_THREADS) {
        float f[8];
        unpack8(zs[c], f);
#pragma unroll
        for (int k = 0; k < 8; k++) mx = fmaxf(mx, f[k]);
    }
    for (int v = nfull * 8 + tid; v < V; v += CE16_THREADS) mx = fmaxf(mx, __bfloat162float(zsh[v]));
    const float M = block_reduce(mx, sh, true);     // its barriers also order the read of zsh[t]
    const float ml = M * CE_LOG2E;
    float sum = 0.f;
    for (int c = tid; c < nfull; c += CE16_THREADS) {
        float f[8];
        unpack8(zs[c], f);
        float s2[2] = {0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 8; k++) {
            f[k] = exp2f(fmaf(f[k], CE_LOG2E, -ml));
            s2[k & 1] += f[k];
        }
        sum += s2[0] + s2[1];
        zs[c] = make_uint4(pack2_h(f[0], f[1]), pack2_h(f[2], f[3]), pack2_h(f[4], f[5]), pack2_h(f[6], f[7]));
    }
    for (int v = nfull * 8 + tid; v < V; v += CE16_THREADS) {
        const float e = exp2f(fmaf(__bfloat162float(zsh[v]), CE_LOG2E, -ml));
        sum += e;
        esh[v] = __float2half_rn(e);
    }
    const float S = block_reduce(sum, sh, false);   // also: every e is in shared memory
    if (tid == 0) {
        if (!ok) set_status(status, GPT2_STATUS_BAD_TARGET);
        losses[row] = ok ? M + logf(S) - zt : 0.f;
    }
    if (dscale == 0.f) return;
    const float pscale = dscale / S;
    for (int c = tid; c < n8; c += CE16_THREADS) {
        float f[8];
        unpack8_h(zs[c], f);
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const int idx = c * 8 + k;
            f[k] = (idx < V && ok) ? f[k] * pscale - (idx == t ? dscale : 0.f) : 0.f;
        }
        zr[c] = make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
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
    if (smem_limit(reinterpret_cast<const void*>(crossentropy_kernel), CE_CACHE_BYTES)) return GPT2_ECUDA;
    const int ncache = std::min(V >> 2, CE_CACHE_BYTES / 16);
    count_launch(), crossentropy_kernel<<<N, CE_THREADS, (size_t)ncache * 16, as_stream(stream)>>>(
        losses, z, static_cast<__nv_bfloat16*>(dz_bf16), tgt, V, ld, dscale, ncache, status);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

GPT2_API int gpt2_op_crossentropy_bf16(float* losses, void* z, const int* tgt, int N, int V, int ld,
                                       float dscale, int* status, void* stream) {
    if (!losses || !z || !tgt || N < 1 || V < 1 || ld < V || ld % 8 || !aligned16(z) ||
        (size_t)ld * 2 > (size_t)CE16_MAX_ROW_BYTES)
        return GPT2_EINVAL;
    if (smem_limit(reinterpret_cast<const void*>(crossentropy_bf16_kernel), CE16_MAX_ROW_BYTES)) return GPT2_ECUDA;
    count_launch(), crossentropy_bf16_kernel<<<N, CE16_THREADS, (size_t)ld * 2, as_stream(stream)>>>(
        losses, static_cast<__nv_bfloat16*>(z), tgt, V, ld, dscale, status);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

GPT2_API int gpt2_op_sum(float* out, const float* x, int N, float scale, void* stream) {
    if (!out || !x || N < 1) return GPT2_EINVAL;
    count_launch(), sum_kernel<<<1, 1024, 0, as_stream(stream)>>>(out, x, N, scale);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}
