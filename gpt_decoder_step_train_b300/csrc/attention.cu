// attention.cu -- causal multi-head self-attention, forward and backward.
//
// Per (batch b, head h): S = Q K^T / sqrt(hs), S[i,j] = -inf for j > i,
// P = softmax_rows(S), O = P V ("GPT-2 from scratch with torch", section
// 自注意力: c_attn output split at C into q, k, v, viewed as (B,T,NH,hs), causal
// mask applied with -Inf before the softmax; 1/sqrt(d_k) scaling explained in
// "从头搭建GPT(Andrej Karpathy) 笔记", section attention中为什么要做scaling).
//
// The T x T matrix is never stored: the forward keeps a running row maximum
// and sum (online softmax) and saves the row log-sum-exp; the backward
// recomputes P from Q, K and the saved log-sum-exp.  Backward formulas:
//   D_i = dO_i . O_i,  dV_j = sum_i P_ij dO_i,  dP_ij = dO_i . V_j,
//   dS_ij = P_ij (dP_ij - D_i),  dQ_i = sum_j dS_ij K_j / sqrt(hs),
//   dK_j = sum_i dS_ij Q_i / sqrt(hs).
// Every output element is owned by exactly one thread, so there are no atomics
// and results are deterministic.
//
// This file holds the CUDA-core kernels: one thread per query row (forward,
// dQ) or per key row (dK, dV), with the row and its accumulator in registers
// and tiles of the other side staged in shared memory.  Keys past a block's
// last query are skipped (causal tile skipping).
#include <cuda_bf16.h>

#include "common.cuh"
#include "dropout.cuh"

namespace gpt2k {

constexpr int AT_ROWS = 128;   // rows (threads) per block
constexpr int AT_KT = 32;      // rows of the other side per shared-memory tile

// Four consecutive elements as floats, and back.
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}

// Load `HSP` values of one row (hs of them real) as floats times mul.
template <int HSP, typename Tv>
__device__ __forceinline__ void load_row(float* dst, const Tv* src, int hs, float mul) {
#pragma unroll
    for (int d = 0; d < HSP; d += 4) {
        float4 v = d < hs ? ld4(src + d) : make_float4(0.f, 0.f, 0.f, 0.f);
        dst[d] = v.x * mul; dst[d + 1] = v.y * mul; dst[d + 2] = v.z * mul; dst[d + 3] = v.w * mul;
    }
}

template <int HSP, typename Tv>
__device__ __forceinline__ void store_row(Tv* dst, const float* v, int hs, float mul) {
#pragma unroll
    for (int d = 0; d < HSP; d += 4)
        if (d < hs) st4(dst + d, make_float4(v[d] * mul, v[d + 1] * mul, v[d + 2] * mul, v[d + 3] * mul));
}

// Cooperative load of rows [r0, r0+AT_KT) (zeros past T) into a shared tile [AT_KT][HSP].
template <int HSP, typename Tv>
__device__ __forceinline__ void load_tile(float (*dst)[HSP], const Tv* base, size_t ld, int r0, int T, int hs) {
    for (int idx = threadIdx.x; idx < AT_KT * (HSP / 4); idx += blockDim.x) {
        int r = idx / (HSP / 4), d = (idx % (HSP / 4)) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r0 + r < T && d < hs) v = ld4(base + (size_t)(r0 + r) * ld + d);
        *reinterpret_cast<float4*>(&dst[r][d]) = v;
    }
}

template <int HSP>
__device__ __forceinline__ float dot_row(const float* a, const float* b) {
    float s = 0.f;
#pragma unroll
    for (int d = 0; d < HSP; d++) s = fmaf(a[d], b[d], s);
    return s;
}

// Dropout on the attention weights: `bits` holds one keep bit per (b, h, i, j),
// rows (b, h, i) of W = ceil(T/32) words (null: no dropout); kept weights are
// scaled by ks = 1/(1-p).  The softmax normaliser and the saved log-sum-exp
// are those of the undropped weights.
template <int HSP, typename Tv>
__global__ void __launch_bounds__(AT_ROWS)
attn_fwd_simt(Tv* __restrict__ y, float* __restrict__ lse, const Tv* __restrict__ qkv, int T,
              int C, int H, int hs, float scale, const uint32_t* __restrict__ bits, float ks) {
    __shared__ __align__(16) float Ks[AT_KT][HSP];
    __shared__ __align__(16) float Vs[AT_KT][HSP];
    const int b = blockIdx.z, h = blockIdx.y, q0 = blockIdx.x * AT_ROWS;
    const int i = q0 + threadIdx.x;
    const bool active = i < T;
    const size_t ld = 3 * (size_t)C;
    const Tv* base = qkv + (size_t)b * T * ld;
    const uint32_t* brow =
        bits && active ? bits + (((size_t)b * H + h) * T + i) * (size_t)((T + 31) >> 5) : nullptr;
    float q[HSP], o[HSP];
    if (active) load_row<HSP>(q, base + (size_t)i * ld + h * hs, hs, scale);
#pragma unroll
    for (int d = 0; d < HSP; d++) o[d] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int kend = min(T, q0 + AT_ROWS);
    for (int k0 = 0; k0 < kend; k0 += AT_KT) {
        __syncthreads();
        load_tile<HSP>(Ks, base + C + h * hs, ld, k0, T, hs);
        load_tile<HSP>(Vs, base + 2 * C + h * hs, ld, k0, T, hs);
        __syncthreads();
        if (!active) continue;
        const int jn = min(AT_KT, i - k0 + 1);
        if (jn <= 0) continue;
        const uint32_t mw = brow ? brow[k0 >> 5] : 0xffffffffu;
        float s[AT_KT];
        float tmax = m;
#pragma unroll
        for (int j = 0; j < AT_KT; j++) {
            if (j < jn) {
                s[j] = dot_row<HSP>(q, Ks[j]);
                tmax = fmaxf(tmax, s[j]);
            }
        }
        const float corr = expf(m - tmax);
        l *= corr;
#pragma unroll
        for (int d = 0; d < HSP; d++) o[d] *= corr;
#pragma unroll
        for (int j = 0; j < AT_KT; j++) {
            if (j < jn) {
                float p = expf(s[j] - tmax);
                l += p;
                if (!((mw >> j) & 1u)) p = 0.f;
#pragma unroll
                for (int d = 0; d < HSP; d++) o[d] = fmaf(p, Vs[j][d], o[d]);
            }
        }
        m = tmax;
    }
    if (!active) return;
    store_row<HSP>(y + ((size_t)b * T + i) * C + h * hs, o, hs, ks / l);
    lse[((size_t)b * H + h) * T + i] = m + logf(l);
}

// D[b,h,i] = dO_i . O_i (bf16 inputs)
// D[b,h,i] = dO_i . O_i over one head's hs elements.  LPR lanes share a
// (position, head) pair and read 16 bytes at a time; pairs are ordered head
// fastest, so a warp reads contiguous rows of dO and O.  Each lane sums its
// chunks in order, then the LPR partial sums meet in a fixed xor tree.
__device__ __forceinline__ float dot16(uint4 a, uint4 b, __nv_bfloat16) {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const float2 u = __bfloat1622float2(x[k]), v = __bfloat1622float2(y[k]);
        s += u.x * v.x + u.y * v.y;
    }
    return s;
}
__device__ __forceinline__ float dot16(uint4 a, uint4 b, float) {
    const float4 u = *reinterpret_cast<const float4*>(&a), v = *reinterpret_cast<const float4*>(&b);
    return (u.x * v.x + u.y * v.y) + (u.z * v.z + u.w * v.w);
}

template <typename Tv, int LPR>
__global__ void __launch_bounds__(256) attn_bwd_dot_kernel(float* __restrict__ D, const Tv* __restrict__ dy,
                                                           const Tv* __restrict__ y, int B, int T, int C,
                                                           int H, int hs) {
    constexpr int PER = 16 / sizeof(Tv);          // elements per 16-byte chunk
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long pair = gid / LPR;             // ((b * T) + t) * H + h
    const int sub = (int)(gid % LPR);
    const bool valid = pair < (long long)B * T * H;
    float s = 0.f;
    long long bt = 0;
    int h = 0;
    if (valid) {
        h = (int)(pair % H);
        bt = pair / H;
        const Tv* a = dy + bt * C + (size_t)h * hs;
        const Tv* o = y + bt * C + (size_t)h * hs;
        for (int d = sub * PER; d < hs; d += LPR * PER)
            s += dot16(__ldg(reinterpret_cast<const uint4*>(a + d)), __ldg(reinterpret_cast<const uint4*>(o + d)),
                       Tv{});
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (valid && sub == 0) {
        const int t = (int)(bt % T), b = (int)(bt / T);
        D[((size_t)b * H + h) * T + t] = s;
    }
}

template <typename Tv>
static void launch_dot(float* D, const void* dy, const void* y, int B, int T, int C, int H, int hs,
                       cudaStream_t st) {
    constexpr int PER = 16 / sizeof(Tv);
    const int chunks = hs / PER;
    const long long pairs = (long long)B * T * H;
    const Tv* g = static_cast<const Tv*>(dy);
    const Tv* o = static_cast<const Tv*>(y);
#define GPT2_DOT(L)                                                                                        \
    count_launch(), attn_bwd_dot_kernel<Tv, L><<<(unsigned)ceil_div(pairs * L, 256), 256, 0, st>>>(       \
        D, g, o, B, T, C, H, hs)
    if (chunks >= 8) GPT2_DOT(8);
    else if (chunks >= 4) GPT2_DOT(4);
    else if (chunks >= 2) GPT2_DOT(2);
    else GPT2_DOT(1);
#undef GPT2_DOT
}

// dQ: one thread per query row i; key/value tiles j <= i in shared memory.
// With dropout, dP_ij = keep_ij * ks * (dO_i . V_j).
template <int HSP, typename Tv>
__global__ void __launch_bounds__(AT_ROWS)
attn_bwd_dq_simt(Tv* __restrict__ dqkv, const Tv* __restrict__ dy, const Tv* __restrict__ qkv,
                 const float* __restrict__ lse, const float* __restrict__ D, int T, int C, int H, int hs,
                 float scale, const uint32_t* __restrict__ bits, float ks) {
    __shared__ __align__(16) float Ks[AT_KT][HSP];
    __shared__ __align__(16) float Vs[AT_KT][HSP];
    const int b = blockIdx.z, h = blockIdx.y, q0 = blockIdx.x * AT_ROWS;
    const int i = q0 + threadIdx.x;
    const bool active = i < T;
    const size_t ld = 3 * (size_t)C;
    const Tv* base = qkv + (size_t)b * T * ld;
    const uint32_t* brow =
        bits && active ? bits + (((size_t)b * H + h) * T + i) * (size_t)((T + 31) >> 5) : nullptr;
    float q[HSP], g[HSP], dq[HSP];
    float li = 0.f, Di = 0.f;
    if (active) {
        load_row<HSP>(q, base + (size_t)i * ld + h * hs, hs, scale);
        load_row<HSP>(g, dy + ((size_t)b * T + i) * C + h * hs, hs, 1.f);
        li = lse[((size_t)b * H + h) * T + i];
        Di = D[((size_t)b * H + h) * T + i];
    }
#pragma unroll
    for (int d = 0; d < HSP; d++) dq[d] = 0.f;
    const int kend = min(T, q0 + AT_ROWS);
    for (int k0 = 0; k0 < kend; k0 += AT_KT) {
        __syncthreads();
        load_tile<HSP>(Ks, base + C + h * hs, ld, k0, T, hs);
        load_tile<HSP>(Vs, base + 2 * C + h * hs, ld, k0, T, hs);
        __syncthreads();
        if (!active) continue;
        const int jn = min(AT_KT, i - k0 + 1);
        const uint32_t mw = brow && jn > 0 ? brow[k0 >> 5] : 0xffffffffu;
#pragma unroll 4
        for (int j = 0; j < jn; j++) {
            float p = expf(dot_row<HSP>(q, Ks[j]) - li);
            float dp = dot_row<HSP>(g, Vs[j]);
            if (brow) dp = ((mw >> j) & 1u) ? dp * ks : 0.f;
            float ds = p * (dp - Di);
#pragma unroll
            for (int d = 0; d < HSP; d++) dq[d] = fmaf(ds, Ks[j][d], dq[d]);
        }
    }
    if (!active) return;
    store_row<HSP>(dqkv + ((size_t)b * T + i) * ld + h * hs, dq, hs, scale);
}

// dK and dV: one thread per key row j; query tiles i >= j in shared memory.
// WANT_DK selects dK (needs V_j too) or dV.  With dropout the keep bits of a
// query tile's rows for this block's 128 keys are staged in shared memory.
template <int HSP, typename Tv, bool WANT_DK>
__global__ void __launch_bounds__(AT_ROWS)
attn_bwd_dkv_simt(Tv* __restrict__ dqkv, const Tv* __restrict__ dy, const Tv* __restrict__ qkv,
                  const float* __restrict__ lse, const float* __restrict__ D, int T, int C, int H, int hs,
                  float scale, const uint32_t* __restrict__ bits, float ks) {
    __shared__ __align__(16) float Qs[AT_KT][HSP];
    __shared__ __align__(16) float Gs[AT_KT][HSP];
    __shared__ float Ls[AT_KT], Ds[AT_KT];
    __shared__ uint32_t Ms[AT_KT][AT_ROWS / 32];
    const int b = blockIdx.z, h = blockIdx.y, k0b = blockIdx.x * AT_ROWS;
    const int j = k0b + threadIdx.x;
    const bool active = j < T;
    const size_t ld = 3 * (size_t)C;
    const Tv* base = qkv + (size_t)b * T * ld;
    const float* lse_bh = lse + ((size_t)b * H + h) * T;
    const float* D_bh = D + ((size_t)b * H + h) * T;
    const int W = (T + 31) >> 5;
    const uint32_t* bits_bh = bits ? bits + ((size_t)b * H + h) * T * (size_t)W : nullptr;
    float k[HSP], v[HSP], acc[HSP];
    if (active) {
        load_row<HSP>(k, base + (size_t)j * ld + C + h * hs, hs, scale);
        if (WANT_DK) load_row<HSP>(v, base + (size_t)j * ld + 2 * C + h * hs, hs, 1.f);
    }
#pragma unroll
    for (int d = 0; d < HSP; d++) acc[d] = 0.f;
    for (int i0 = k0b; i0 < T; i0 += AT_KT) {
        __syncthreads();
        load_tile<HSP>(Qs, base + h * hs, ld, i0, T, hs);
        load_tile<HSP>(Gs, dy + (size_t)b * T * C + h * hs, C, i0, T, hs);
        if (threadIdx.x < AT_KT) {
            int ii = i0 + threadIdx.x;
            Ls[threadIdx.x] = ii < T ? lse_bh[ii] : 0.f;
            Ds[threadIdx.x] = ii < T ? D_bh[ii] : 0.f;
        }
        if (bits_bh) {
            for (int idx = threadIdx.x; idx < AT_KT * (AT_ROWS / 32); idx += blockDim.x) {
                const int r = idx / (AT_ROWS / 32), kw = (k0b >> 5) + idx % (AT_ROWS / 32);
                Ms[r][idx % (AT_ROWS / 32)] = i0 + r < T && kw < W ? bits_bh[(size_t)(i0 + r) * W + kw] : 0u;
            }
        }
        __syncthreads();
        if (!active) continue;
        const int ibeg = max(0, j - i0), iend = min(AT_KT, T - i0);
#pragma unroll 4
        for (int r = ibeg; r < iend; r++) {
            float p = expf(dot_row<HSP>(k, Qs[r]) - Ls[r]);
            const bool kept = !bits_bh || ((Ms[r][threadIdx.x >> 5] >> (threadIdx.x & 31)) & 1u);
            if (WANT_DK) {
                float dp = dot_row<HSP>(v, Gs[r]);
                if (bits_bh) dp = kept ? dp * ks : 0.f;
                float ds = p * (dp - Ds[r]);
#pragma unroll
                for (int d = 0; d < HSP; d++) acc[d] = fmaf(ds, Qs[r][d], acc[d]);
            } else {
                const float a = bits_bh ? (kept ? p * ks : 0.f) : p;
#pragma unroll
                for (int d = 0; d < HSP; d++) acc[d] = fmaf(a, Gs[r][d], acc[d]);
            }
        }
    }
    if (!active) return;
    store_row<HSP>(dqkv + ((size_t)b * T + j) * ld + (WANT_DK ? C : 2 * C) + h * hs, acc, hs,
                   WANT_DK ? scale : 1.f);
}

template <int HSP, typename Tv>
static void launch_fwd(void* y, float* lse, const void* qkv, int B, int T, int C, int H, int hs,
                       const uint32_t* bits, float ks, cudaStream_t st) {
    dim3 grid(ceil_div(T, AT_ROWS), H, B);
    count_launch(), attn_fwd_simt<HSP, Tv><<<grid, AT_ROWS, 0, st>>>(
        static_cast<Tv*>(y), lse, static_cast<const Tv*>(qkv), T, C, H, hs, 1.f / sqrtf((float)hs), bits, ks);
}

template <int HSP, typename Tv>
static void launch_bwd(void* dqkv, const void* dy, const void* qkv, const float* lse, const float* D, int B,
                       int T, int C, int H, int hs, const uint32_t* bits, float ks, cudaStream_t st) {
    dim3 grid(ceil_div(T, AT_ROWS), H, B);
    float scale = 1.f / sqrtf((float)hs);
    Tv* o = static_cast<Tv*>(dqkv);
    const Tv* g = static_cast<const Tv*>(dy);
    const Tv* x = static_cast<const Tv*>(qkv);
    count_launch(), attn_bwd_dq_simt<HSP, Tv><<<grid, AT_ROWS, 0, st>>>(o, g, x, lse, D, T, C, H, hs, scale, bits, ks);
    count_launch(), attn_bwd_dkv_simt<HSP, Tv, true><<<grid, AT_ROWS, 0, st>>>(o, g, x, lse, D, T, C, H, hs, scale,
                                                                               bits, ks);
    count_launch(), attn_bwd_dkv_simt<HSP, Tv, false><<<grid, AT_ROWS, 0, st>>>(o, g, x, lse, D, T, C, H, hs, scale,
                                                                                bits, ks);
}

template <typename Tv>
static void simt_forward(void* y, float* lse, const void* qkv, int B, int T, int C, int H, int hs,
                         const uint32_t* bits, float ks, cudaStream_t st) {
    if (hs <= 16) launch_fwd<16, Tv>(y, lse, qkv, B, T, C, H, hs, bits, ks, st);
    else if (hs <= 32) launch_fwd<32, Tv>(y, lse, qkv, B, T, C, H, hs, bits, ks, st);
    else launch_fwd<64, Tv>(y, lse, qkv, B, T, C, H, hs, bits, ks, st);
}

template <typename Tv>
static void simt_backward(void* dqkv, const void* dy, const void* qkv, const float* lse, const float* D, int B,
                          int T, int C, int H, int hs, const uint32_t* bits, float ks, cudaStream_t st) {
    if (hs <= 16) launch_bwd<16, Tv>(dqkv, dy, qkv, lse, D, B, T, C, H, hs, bits, ks, st);
    else if (hs <= 32) launch_bwd<32, Tv>(dqkv, dy, qkv, lse, D, B, T, C, H, hs, bits, ks, st);
    else launch_bwd<64, Tv>(dqkv, dy, qkv, lse, D, B, T, C, H, hs, bits, ks, st);
}

int attention_tc_forward(float* y, float* lse, const float* qkv, int B, int T, int C, int H,
                         int* status, cudaStream_t st);
int attention_bf16_forward(void* y, float* lse, const void* qkv, int B, int T, int C, int H,
                           cudaStream_t st);
int attention_bf16_backward(void* dqkv, const void* dy, const void* qkv, const float* lse,
                            const float* D, int B, int T, int C, int H, cudaStream_t st);
int attention_tc_backward(float* dqkv, const float* dy, const float* qkv, const float* lse,
                          const float* D, int B, int T, int C, int H, int* status,
                          cudaStream_t st);
bool attention_tc_supported(int hs);
bool attention_tc05_supported(int hs, int C);
int attention_tc05_forward(void* y, float* lse, const void* qkv, int B, int T, int C, int H, int* status,
                           cudaStream_t st, const uint32_t* bits, float ks);
int attention_tc05_tf32_forward(float* y, float* lse, const float* qkv, int B, int T, int C, int H, int* status,
                                cudaStream_t st);
int attention_tc05_tf32_backward(float* dqkv, const float* dy, const float* qkv, const float* lse, const float* D,
                                 int B, int T, int C, int H, int* status, cudaStream_t st);
int attention_tc05_backward_nodrop(void* dqkv, const void* dy, const void* qkv, const void* y, const float* lse,
                                   float* D, int B, int T, int C, int H, int* status, cudaStream_t st,
                                   float* colsum);
int attention_tc05_backward(void* dqkv, const void* dy, const void* qkv, const float* lse, const float* D,
                            int B, int T, int C, int H, int* status, cudaStream_t st, float* colsum,
                            const uint32_t* bits, float ks);

static bool attn_args_ok(int B, int T, int C, int H) {
    if (B < 1 || T < 1 || C < 4 || H < 1 || C % H) return false;
    int hs = C / H;
    return hs % 4 == 0 && hs <= 64;
}

// Dispatch: BF16 mode takes the tcgen05 kernels for head size 64, the
// mma.sync kernels for head sizes 16 and 32 (no dropout), else the CUDA-core
// kernels on bf16 (head sizes that are multiples of 8: the backward's
// rowsum(dO o O) reads a head's slice 16 bytes at a time); TF32 mode takes the
// tcgen05 tf32 kernels for head size 64 and the mma.sync TF32 kernels for
// head sizes 16 and 32 (no dropout); otherwise (FP32 mode, dropout) the
// CUDA-core kernels on fp32.
int attention_forward(void* y, float* lse, const void* qkv, int B, int T, int C, int H, int mode, int* status,
                      cudaStream_t st, const uint32_t* bits, float p) {
    if (!y || !lse || !qkv || !attn_args_ok(B, T, C, H)) return GPT2_EINVAL;
    if (!aligned16(y) || !aligned16(qkv) || !(p >= 0.f && p < 1.f)) return GPT2_EINVAL;
    int hs = C / H;
    const float ks = bits ? dropout_scale(p) : 1.f;
    if (mode == GPT2_MODE_BF16) {
        if (attention_tc05_supported(hs, C))
            return attention_tc05_forward(y, lse, qkv, B, T, C, H, status, st, bits, ks);
        if (!bits && attention_tc_supported(hs)) return attention_bf16_forward(y, lse, qkv, B, T, C, H, st);
        if (hs % 8) return GPT2_ENOTSUP;
        simt_forward<__nv_bfloat16>(y, lse, qkv, B, T, C, H, hs, bits, ks, st);
        GPT2_LAUNCH_CHECK();
        return GPT2_OK;
    }
    if (mode == GPT2_MODE_TF32 && !bits && attention_tc05_supported(hs, C))
        return attention_tc05_tf32_forward(static_cast<float*>(y), lse, static_cast<const float*>(qkv), B, T, C,
                                           H, status, st);
    if (mode == GPT2_MODE_TF32 && !bits && attention_tc_supported(hs))
        return attention_tc_forward(static_cast<float*>(y), lse, static_cast<const float*>(qkv), B, T, C, H,
                                    status, st);
    simt_forward<float>(y, lse, qkv, B, T, C, H, hs, bits, ks, st);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int attention_backward_dropout(void* dqkv, const void* dy, const void* qkv, const void* y, const float* lse, int B,
                               int T, int C, int H, void* scratch, size_t scratch_bytes, int mode, int* status,
                               cudaStream_t st, float* colsum, bool* colsum_done, const uint32_t* bits, float p) {
    if (colsum_done) *colsum_done = false;
    if (!dqkv || !dy || !qkv || !y || !lse || !attn_args_ok(B, T, C, H)) return GPT2_EINVAL;
    if (!aligned16(dqkv) || !aligned16(dy) || !aligned16(qkv) || !aligned16(y) || !(p >= 0.f && p < 1.f))
        return GPT2_EINVAL;
    if (!scratch || scratch_bytes < round_up((size_t)B * H * T * sizeof(float), 256)) return GPT2_ENOMEM;
    int hs = C / H;
    const float ks = bits ? dropout_scale(p) : 1.f;
    // D = rowsum(dO o O) with O the output that met dO (after dropout)
    float* D = reinterpret_cast<float*>(scratch);
    if (mode == GPT2_MODE_BF16) {
        if (hs % 8) return GPT2_ENOTSUP;
        // without dropout, head size 64: the tcgen05 kernels compute D themselves
        if (!bits && attention_tc05_supported(hs, C)) {
            if (colsum_done) *colsum_done = colsum != nullptr;
            return attention_tc05_backward_nodrop(dqkv, dy, qkv, y, lse, D, B, T, C, H, status, st,
                                                  colsum_done ? colsum : nullptr);
        }
        launch_dot<__nv_bfloat16>(D, dy, y, B, T, C, H, hs, st);
        GPT2_LAUNCH_CHECK();
        if (attention_tc05_supported(hs, C)) {
            if (colsum_done) *colsum_done = colsum != nullptr;
            return attention_tc05_backward(dqkv, dy, qkv, lse, D, B, T, C, H, status, st,
                                           colsum_done ? colsum : nullptr, bits, ks);
        }
        if (!bits && attention_tc_supported(hs))
            return attention_bf16_backward(dqkv, dy, qkv, lse, D, B, T, C, H, st);
        simt_backward<__nv_bfloat16>(dqkv, dy, qkv, lse, D, B, T, C, H, hs, bits, ks, st);
        GPT2_LAUNCH_CHECK();
        return GPT2_OK;
    }
    launch_dot<float>(D, dy, y, B, T, C, H, hs, st);
    GPT2_LAUNCH_CHECK();
    if (mode == GPT2_MODE_TF32 && !bits && attention_tc05_supported(hs, C))
        return attention_tc05_tf32_backward(static_cast<float*>(dqkv), static_cast<const float*>(dy),
                                            static_cast<const float*>(qkv), lse, D, B, T, C, H, status, st);
    if (mode == GPT2_MODE_TF32 && !bits && attention_tc_supported(hs))
        return attention_tc_backward(static_cast<float*>(dqkv), static_cast<const float*>(dy),
                                     static_cast<const float*>(qkv), lse, D, B, T, C, H, status, st);
    simt_backward<float>(dqkv, dy, qkv, lse, D, B, T, C, H, hs, bits, ks, st);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int attention_backward(void* dqkv, const void* dy, const void* qkv, const void* y, const float* lse, int B,
                       int T, int C, int H, void* scratch, size_t scratch_bytes, int mode, int* status,
                       cudaStream_t st, float* colsum, bool* colsum_done) {
    return attention_backward_dropout(dqkv, dy, qkv, y, lse, B, T, C, H, scratch, scratch_bytes, mode, status, st,
                                      colsum, colsum_done, nullptr, 0.f);
}

}  // namespace gpt2k

using namespace gpt2k;

GPT2_API int gpt2_op_attention_forward(void* y, float* lse, const void* qkv, int B, int T, int C,
                                       int H, int mode, int* status, void* stream) {
    return attention_forward(y, lse, qkv, B, T, C, H, mode, status, as_stream(stream), nullptr, 0.f);
}

GPT2_API int gpt2_op_attention_forward_dropout(void* y, float* lse, const void* qkv, int B, int T, int C, int H,
                                               int mode, const uint32_t* bits, float p, int* status,
                                               void* stream) {
    if (!bits) return GPT2_EINVAL;
    return attention_forward(y, lse, qkv, B, T, C, H, mode, status, as_stream(stream), bits, p);
}

GPT2_API size_t gpt2_op_attention_backward_scratch_bytes(int B, int T, int H) {
    if (B < 1 || T < 1 || H < 1) return 0;
    return round_up((size_t)B * H * T * sizeof(float), 256);
}

GPT2_API int gpt2_op_attention_backward_dropout(void* dqkv, const void* dy, const void* qkv, const void* y,
                                                const float* lse, int B, int T, int C, int H, void* scratch,
                                                size_t scratch_bytes, int mode, const uint32_t* bits, float p,
                                                int* status, void* stream) {
    if (!bits) return GPT2_EINVAL;
    return attention_backward_dropout(dqkv, dy, qkv, y, lse, B, T, C, H, scratch, scratch_bytes, mode, status,
                                      as_stream(stream), nullptr, nullptr, bits, p);
}

GPT2_API int gpt2_op_attention_backward(void* dqkv, const void* dy, const void* qkv,
                                        const void* y, const float* lse, int B, int T, int C,
                                        int H, void* scratch, size_t scratch_bytes, int mode,
                                        int* status, void* stream) {
    return attention_backward(dqkv, dy, qkv, y, lse, B, T, C, H, scratch, scratch_bytes, mode, status,
                              as_stream(stream), nullptr, nullptr);
}
