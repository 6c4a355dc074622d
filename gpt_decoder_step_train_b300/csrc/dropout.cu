// dropout.cu -- inverted dropout masks and the element-wise dropout kernels.
//
// Where dropout sits: after the token + position embeddings, on the attention
// weights after the softmax, and on each block's two c_proj outputs before the
// residual addition ("GPT-2 from scratch with torch", sections 总体架构,
// 近看 Transformer block：自注意力 and 近看 Transformer block：前馈网络（MLP）;
// "从头搭建GPT(Andrej Karpathy) 笔记", section 继续增加改进的点).  Training keeps
// an element with probability 1 - p and scales it by 1/(1 - p); evaluation
// uses every element unscaled.
//
// Draws: the counter-based generator Philox4x32-10 (Salmon, Moraes, Dror and
// Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011): ten rounds of
// (c0,c1,c2,c3) <- (hi(M1*c2)^c1^k0, lo(M1*c2), hi(M0*c0)^c3^k1, lo(M0*c0)),
// M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key advanced by (0x9E3779B9,
// 0xBB67AE85) before every round but the first.  Element e (row-major index)
// of dropout site `site` in forward call `step` under the 64-bit seed:
//   w = Philox4x32-10(counter (lo32(e/4), hi32(e/4), site, step), key (lo32(seed), hi32(seed)))
//   keep(e) = w[e mod 4] >= floor(p * 2^32)
// Sites: 0 the embedding output [B,T,C]; for layer l, 1 + 3l the attention
// weights [B,NH,T,T], 2 + 3l the attention c_proj output and 3 + 3l the MLP
// c_proj output ([B,T,C]).
//
// Masks are stored one bit per element, row by row: a row of `cols` elements
// takes W = ceil(cols/32) 32-bit words, bit b of word k is element 32k + b of
// the row, and bits past the row's end are 0.  For the attention weights the
// rows are (b, h, i) and the columns the keys j; words wholly above the
// diagonal (32k > i) are written as 0 without drawing, since no key there is
// ever used.  The attention kernels read one word per 32 keys, the
// element-wise kernels one word per row chunk, and the backward reuses the
// forward's masks as they are.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "dropout.cuh"

namespace gpt2k {

// Philox4x32-10 of counter c under key (k0, k1).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; r++) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// One thread per mask word.  The key and the step come from `state`
// ({key0, key1, step}, device memory) when it is given, so that a captured
// graph draws new masks each call; else from the arguments.
//
// ALIGNED (cols % 4 == 0): a word's first element is a multiple of 4, so its
// 32 elements are exactly the 4 words of 8 consecutive draws (fewer at a row
// end); the 8 draws are independent and unrolled.  Otherwise a word's elements
// may start and end inside a draw, and each element finds its own word.
template <bool ALIGNED>
__global__ void __launch_bounds__(256)
dropout_mask_kernel(uint32_t* __restrict__ bits, long long rows, int cols, int W, int causal_T,
                    const uint32_t* __restrict__ state, uint32_t key0, uint32_t key1, uint32_t step,
                    uint32_t site, uint32_t thr) {
    if (state) {
        key0 = state[0];
        key1 = state[1];
        step = state[2];
    }
    const long long total = rows * W;
    for (long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x; w < total;
         w += (long long)gridDim.x * blockDim.x) {
        long long row;
        int k, i_diag = 0;
        if (total <= 0x7fffffffLL) {            // 32-bit division (the usual case)
            const uint32_t wu = (uint32_t)w, ru = wu / (uint32_t)W;
            row = ru;
            k = (int)(wu - ru * (uint32_t)W);
            if (causal_T) i_diag = (int)(ru % (uint32_t)causal_T);
        } else {
            row = w / W;
            k = (int)(w - row * W);
            if (causal_T) i_diag = (int)(row % causal_T);
        }
        const int c0 = 32 * k;
        uint32_t out = 0;
        if (causal_T == 0 || c0 <= i_diag) {
            const int nb = min(32, cols - c0);
            const unsigned long long e0 = (unsigned long long)row * (unsigned long long)cols + (unsigned long long)c0;
            if constexpr (ALIGNED) {
                const unsigned long long q0 = e0 >> 2;
                const int nq = nb >> 2;
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    if (j < nq) {
                        const unsigned long long q = q0 + (unsigned long long)j;
                        const uint4 r =
                            philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), site, step), key0, key1);
                        out |= ((uint32_t)(r.x >= thr) | ((uint32_t)(r.y >= thr) << 1) |
                                ((uint32_t)(r.z >= thr) << 2) | ((uint32_t)(r.w >= thr) << 3))
                               << (4 * j);
                    }
                }
            } else {
                const unsigned long long q1 = (e0 + (unsigned long long)nb - 1) >> 2;
                for (unsigned long long q = e0 >> 2; q <= q1; q++) {
                    const uint4 r =
                        philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), site, step), key0, key1);
                    const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const long long b = (long long)(4 * q + (unsigned long long)i) - (long long)e0;
                        if (b >= 0 && b < nb && wv[i] >= thr) out |= 1u << b;
                    }
                }
            }
        }
        bits[w] = out;
    }
}

// The attention sites (causal_T > 0, cols % 4 == 0): a block of 32 x 32
// threads covers 32 consecutive rows and 32 consecutive words; a warp takes one
// word of the 32 rows (lane = row), so the rows of one 32-row group of a
// (batch, head) share the decision "left of the diagonal or not" and the warp
// draws or writes zeros as a whole.  The words go through a shared tile and are
// written row by row (32 words, 128 bytes, per warp).  Same bits as the
// kernel above.
__global__ void __launch_bounds__(1024)
dropout_mask_causal_kernel(uint32_t* __restrict__ bits, long long rows, int cols, int W, int causal_T,
                           const uint32_t* __restrict__ state, uint32_t key0, uint32_t key1, uint32_t step,
                           uint32_t site, uint32_t thr) {
    __shared__ uint32_t tile[32][33];
    if (state) {
        key0 = state[0];
        key1 = state[1];
        step = state[2];
    }
    const int r = threadIdx.x, kk = threadIdx.y;
    const long long row0 = 32LL * blockIdx.x, row = row0 + r;
    const int k = 32 * (int)blockIdx.y + kk;
    uint32_t out = 0;
    if (row < rows && k < W) {
        const int i = (int)(row % causal_T), c0 = 32 * k;
        if (c0 <= i) {
            const int nq = min(32, cols - c0) >> 2;
            const unsigned long long q0 =
                ((unsigned long long)row * (unsigned long long)cols + (unsigned long long)c0) >> 2;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if (j < nq) {
                    const unsigned long long q = q0 + (unsigned long long)j;
                    const uint4 v = philox4x32_10(make_uint4((uint32_t)q, (uint32_t)(q >> 32), site, step), key0, key1);
                    out |= ((uint32_t)(v.x >= thr) | ((uint32_t)(v.y >= thr) << 1) | ((uint32_t)(v.z >= thr) << 2) |
                            ((uint32_t)(v.w >= thr) << 3))
                           << (4 * j);
                }
            }
        }
    }
    tile[kk][r] = out;
    __syncthreads();
    // thread (x, y) writes word 32 blockIdx.y + x of row row0 + y
    const long long wrow = row0 + threadIdx.y;
    const int wk = 32 * (int)blockIdx.y + threadIdx.x;
    if (wrow < rows && wk < W) bits[wrow * W + wk] = tile[threadIdx.x][threadIdx.y];
}

// out = res + keep o out / (1 - p)  (res may be null: out = keep o out / (1 - p));
// rows of C columns, C % 4 == 0, one float4 per thread.
__global__ void __launch_bounds__(256)
dropout_residual_kernel(float4* __restrict__ out, const float4* __restrict__ res, const uint32_t* __restrict__ bits,
                        long long n4, int C4, int W, float ks) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
        long long row;
        int c;
        if (n4 <= 0x7fffffffLL) {               // 32-bit division (the usual case)
            const uint32_t iu = (uint32_t)i, ru = iu / (uint32_t)C4;
            row = ru;
            c = 4 * (int)(iu - ru * (uint32_t)C4);
        } else {
            row = i / C4;
            c = 4 * (int)(i - row * C4);
        }
        const uint32_t m = __ldg(bits + row * W + (c >> 5)) >> (c & 31);
        float4 v = out[i];
        const float4 r = res ? res[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        v.x = r.x + ((m & 1u) ? v.x * ks : 0.f);
        v.y = r.y + ((m & 2u) ? v.y * ks : 0.f);
        v.z = r.z + ((m & 4u) ? v.z * ks : 0.f);
        v.w = r.w + ((m & 8u) ? v.w * ks : 0.f);
        out[i] = v;
    }
}

// dst = keep o src / (1 - p), dst fp32 (may be src) or bf16.
template <bool BF16>
__global__ void __launch_bounds__(256)
dropout_backward_kernel(void* dst, const float4* src, const uint32_t* __restrict__ bits,
                        long long n4, int C4, int W, float ks) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
        long long row;
        int c;
        if (n4 <= 0x7fffffffLL) {               // 32-bit division (the usual case)
            const uint32_t iu = (uint32_t)i, ru = iu / (uint32_t)C4;
            row = ru;
            c = 4 * (int)(iu - ru * (uint32_t)C4);
        } else {
            row = i / C4;
            c = 4 * (int)(i - row * C4);
        }
        const uint32_t m = __ldg(bits + row * W + (c >> 5)) >> (c & 31);
        const float4 g = src[i];
        const float4 v = make_float4((m & 1u) ? g.x * ks : 0.f, (m & 2u) ? g.y * ks : 0.f, (m & 4u) ? g.z * ks : 0.f,
                                     (m & 8u) ? g.w * ks : 0.f);
        if constexpr (BF16) {
            __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t*>(&a);
            u.y = *reinterpret_cast<uint32_t*>(&b);
            reinterpret_cast<uint2*>(dst)[i] = u;
        } else {
            reinterpret_cast<float4*>(dst)[i] = v;
        }
    }
}

static unsigned elementwise_blocks(long long n) {
    const long long want = (n + 255) / 256;
    return (unsigned)(want < 148LL * 16 ? (want > 0 ? want : 1) : 148LL * 16);
}

uint32_t dropout_threshold(float p) { return (uint32_t)floor((double)p * 4294967296.0); }

float dropout_scale(float p) { return 1.f / (1.f - p); }

size_t dropout_words(long long rows, int cols) { return (size_t)rows * (size_t)((cols + 31) / 32); }

int dropout_mask(uint32_t* bits, long long rows, int cols, int causal_T, const uint32_t* state,
                 unsigned long long seed, uint32_t site, uint32_t step, float p, cudaStream_t st) {
    if (rows == 0) return GPT2_OK;
    const int W = (cols + 31) / 32;
    const long long total = rows * W;
    const long long want = (total + 255) / 256;
    const unsigned blocks = (unsigned)(want < 148LL * 32 ? want : 148LL * 32);
    const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32), thr = dropout_threshold(p);
    if (causal_T > 0 && cols % 4 == 0 && (rows + 31) / 32 <= 0x7fffffffLL)
        count_launch(), dropout_mask_causal_kernel<<<dim3((unsigned)((rows + 31) / 32), (unsigned)((W + 31) / 32)),
                                                     dim3(32, 32), 0, st>>>(bits, rows, cols, W, causal_T, state, k0,
                                                                           k1, step, site, thr);
    else if (cols % 4 == 0)
        count_launch(), dropout_mask_kernel<true><<<blocks, 256, 0, st>>>(bits, rows, cols, W, causal_T, state, k0,
                                                                          k1, step, site, thr);
    else
        count_launch(), dropout_mask_kernel<false><<<blocks, 256, 0, st>>>(bits, rows, cols, W, causal_T, state, k0,
                                                                           k1, step, site, thr);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int dropout_residual(float* out, const float* res, const uint32_t* bits, int N, int C, float p, cudaStream_t st) {
    const long long n4 = (long long)N * C / 4;
    if (n4 == 0) return GPT2_OK;
    count_launch(), dropout_residual_kernel<<<elementwise_blocks(n4), 256, 0, st>>>(
        reinterpret_cast<float4*>(out), reinterpret_cast<const float4*>(res), bits, n4, C / 4, (C + 31) / 32,
        dropout_scale(p));
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int dropout_backward(void* dst, bool bf16, const float* src, const uint32_t* bits, int N, int C, float p,
                     cudaStream_t st) {
    const long long n4 = (long long)N * C / 4;
    if (n4 == 0) return GPT2_OK;
    const auto* s4 = reinterpret_cast<const float4*>(src);
    const int W = (C + 31) / 32;
    if (bf16)
        count_launch(), dropout_backward_kernel<true><<<elementwise_blocks(n4), 256, 0, st>>>(
            dst, s4, bits, n4, C / 4, W, dropout_scale(p));
    else
        count_launch(), dropout_backward_kernel<false><<<elementwise_blocks(n4), 256, 0, st>>>(
            dst, s4, bits, n4, C / 4, W, dropout_scale(p));
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k

using namespace gpt2k;

static bool p_ok(float p) { return p >= 0.f && p < 1.f; }

GPT2_API size_t gpt2_op_dropout_mask_words(long long rows, int cols) {
    if (rows < 0 || cols < 1) return 0;
    return dropout_words(rows, cols);
}

GPT2_API int gpt2_op_dropout_mask(uint32_t* bits, long long rows, int cols, int causal_T, unsigned long long seed,
                                  unsigned int site, unsigned int step, float p, void* stream) {
    if (!bits || rows < 0 || cols < 1 || causal_T < 0 || !p_ok(p)) return GPT2_EINVAL;
    if (causal_T > 0 && (cols != causal_T || rows % causal_T)) return GPT2_EINVAL;
    return dropout_mask(bits, rows, cols, causal_T, nullptr, seed, site, step, p, as_stream(stream));
}

GPT2_API int gpt2_op_dropout_residual(float* out, const float* res, const uint32_t* bits, int N, int C, float p,
                                      void* stream) {
    if (!out || !bits || N < 0 || C < 4 || C % 4 || !p_ok(p)) return GPT2_EINVAL;
    if (!aligned16(out) || (res && !aligned16(res))) return GPT2_EINVAL;
    return dropout_residual(out, res, bits, N, C, p, as_stream(stream));
}

GPT2_API int gpt2_op_dropout_backward(void* dst, int dst_bf16, const float* src, const uint32_t* bits, int N, int C,
                                      float p, void* stream) {
    if (!dst || !src || !bits || N < 0 || C < 4 || C % 4 || !p_ok(p)) return GPT2_EINVAL;
    if (!aligned16(src) || (reinterpret_cast<uintptr_t>(dst) & (dst_bf16 ? 7u : 15u))) return GPT2_EINVAL;
    return dropout_backward(dst, dst_bf16 != 0, src, bits, N, C, p, as_stream(stream));
}
