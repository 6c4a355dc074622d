// layernorm.cu -- LayerNorm forward and backward, one warp per row.
//
// Forward ("GPT-2 from scratch with torch", Transformer block: ln_1/ln_2/ln_f
// with eps 1e-5): mean, biased variance, rstd = 1/sqrt(var + eps),
// y = (x - mean) * rstd * w + b.  The row is held in registers (float4 loads),
// so x is read once and the variance is a second pass over registers.
//
// Backward (derived by hand, as the llm.c overview on bigegpt.com describes
// for every layer): with xhat = (x-mean)*rstd and g = dy*w,
//   dx += rstd * (g - mean(g) - xhat * mean(g * xhat)),
//   dw = sum_rows dy * xhat,  db = sum_rows dy.
// dw/db are reduced deterministically: each block sums its rows in a fixed
// order into a per-block partial, and a second kernel sums the partials in
// block order.
#include <cuda_bf16.h>

#include "common.cuh"

namespace gpt2k {

constexpr float LN_EPS = 1e-5f;
constexpr int LN_MAXV = 16;        // float4 per lane: C <= 32*4*16 = 2048
constexpr int LN_WARPS = 8;

template <int NV, bool OUT_BF16>
__global__ void __launch_bounds__(LN_WARPS * 32)
ln_fwd_kernel(void* __restrict__ yv, float* __restrict__ mean, float* __restrict__ rstd,
              const float* __restrict__ x, const float* __restrict__ w,
              const float* __restrict__ b, int N, int C) {
    int row = blockIdx.x * LN_WARPS + (threadIdx.x >> 5);
    int lane = threadIdx.x & 31;
    if (row >= N) return;
    int C4 = C >> 2;
    const float4* xr = reinterpret_cast<const float4*>(x + (size_t)row * C);
    float4 v[NV];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
        int c = lane + 32 * i;
        if (c < C4) {
            v[i] = xr[c];
            s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
        }
    }
    float mu = warp_sum(s) / (float)C;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < NV; i++) {
        int c = lane + 32 * i;
        if (c < C4) {
            float a = v[i].x - mu, bb = v[i].y - mu, cc = v[i].z - mu, d = v[i].w - mu;
            q += (a * a + bb * bb) + (cc * cc + d * d);
        }
    }
    float r = rsqrtf(warp_sum(q) / (float)C + LN_EPS);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    const float4* b4 = reinterpret_cast<const float4*>(b);
#pragma unroll
    for (int i = 0; i < NV; i++) {
        int c = lane + 32 * i;
        if (c < C4) {
            float4 ww = w4[c], bb = b4[c], o;
            o.x = (v[i].x - mu) * r * ww.x + bb.x;
            o.y = (v[i].y - mu) * r * ww.y + bb.y;
            o.z = (v[i].z - mu) * r * ww.z + bb.z;
            o.w = (v[i].w - mu) * r * ww.w + bb.w;
            if (OUT_BF16) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
                reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(yv) + (size_t)row * C)[c] =
                    make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
            } else {
                reinterpret_cast<float4*>(static_cast<float*>(yv) + (size_t)row * C)[c] = o;
            }
        }
    }
    if (lane == 0) {
        mean[row] = mu;
        rstd[row] = r;
    }
}

// Block `blk` handles rows [blk*rpb, min(N, (blk+1)*rpb)); warp w takes rows
// start+w, start+w+LN_WARPS, ...  partial[blk][0][C] = sum dy*xhat,
// partial[blk][1][C] = sum dy over the block's rows.
template <int NV>
__global__ void __launch_bounds__(LN_WARPS * 32)
ln_bwd_kernel(float* __restrict__ dx, __nv_bfloat16* __restrict__ dx16, float* __restrict__ partial,
              const float* __restrict__ dy,
              const float* __restrict__ x, const float* __restrict__ w,
              const float* __restrict__ mean, const float* __restrict__ rstd, int N, int C,
              int rpb) {
    extern __shared__ float4 sh4[];              // [2][C4]
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int C4 = C >> 2;
    int start = blockIdx.x * rpb, end = min(N, start + rpb);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    float4 adw[NV], adb[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        adw[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        adb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int row = start + warp; row < end; row += LN_WARPS) {
        const float4* xr = reinterpret_cast<const float4*>(x + (size_t)row * C);
        const float4* gr = reinterpret_cast<const float4*>(dy + (size_t)row * C);
        float mu = mean[row], r = rstd[row];
        float sg = 0.f, sgx = 0.f;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            int c = lane + 32 * i;
            if (c < C4) {
                float4 xv = xr[c], d = gr[c], ww = w4[c];
                float4 xh = make_float4((xv.x - mu) * r, (xv.y - mu) * r, (xv.z - mu) * r, (xv.w - mu) * r);
                float4 g = make_float4(d.x * ww.x, d.y * ww.y, d.z * ww.z, d.w * ww.w);
                sg += (g.x + g.y) + (g.z + g.w);
                sgx += (g.x * xh.x + g.y * xh.y) + (g.z * xh.z + g.w * xh.w);
                adw[i].x += d.x * xh.x; adw[i].y += d.y * xh.y;
                adw[i].z += d.z * xh.z; adw[i].w += d.w * xh.w;
                adb[i].x += d.x; adb[i].y += d.y; adb[i].z += d.z; adb[i].w += d.w;
            }
        }
        float mg = warp_sum(sg) / (float)C, mgx = warp_sum(sgx) / (float)C;
        float4* dxr = reinterpret_cast<float4*>(dx + (size_t)row * C);
        // second pass re-reads the row (L1-resident) instead of holding it in registers
#pragma unroll
        for (int i = 0; i < NV; i++) {
            int c = lane + 32 * i;
            if (c < C4) {
                float4 xv = xr[c], d = gr[c], ww = w4[c];
                float4 o = dxr[c];
                float xh, g;
                xh = (xv.x - mu) * r; g = d.x * ww.x; o.x += r * (g - mg - xh * mgx);
                xh = (xv.y - mu) * r; g = d.y * ww.y; o.y += r * (g - mg - xh * mgx);
                xh = (xv.z - mu) * r; g = d.z * ww.z; o.z += r * (g - mg - xh * mgx);
                xh = (xv.w - mu) * r; g = d.w * ww.w; o.w += r * (g - mg - xh * mgx);
                dxr[c] = o;
                if (dx16) {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
                    reinterpret_cast<uint2*>(dx16 + (size_t)row * C)[c] =
                        make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
                }
            }
        }
    }
    // fixed-order reduction over the block's warps: warp 0 stores, then 1..7 add
    float4* sdw = sh4;
    float4* sdb = sh4 + C4;
    for (int k = 0; k < LN_WARPS; k++) {
        if (warp == k) {
#pragma unroll
            for (int i = 0; i < NV; i++) {
                int c = lane + 32 * i;
                if (c < C4) {
                    if (k == 0) {
                        sdw[c] = adw[i];
                        sdb[c] = adb[i];
                    } else {
                        float4 a = sdw[c], bb = sdb[c];
                        a.x += adw[i].x; a.y += adw[i].y; a.z += adw[i].z; a.w += adw[i].w;
                        bb.x += adb[i].x; bb.y += adb[i].y; bb.z += adb[i].z; bb.w += adb[i].w;
                        sdw[c] = a;
                        sdb[c] = bb;
                    }
                }
            }
        }
        __syncthreads();
    }
    float4* out = reinterpret_cast<float4*>(partial) + (size_t)blockIdx.x * 2 * C4;
    for (int c = threadIdx.x; c < 2 * C4; c += blockDim.x) out[c] = sh4[c];
}

// dw[c] = sum_blk partial[blk][0][c], db[c] = sum_blk partial[blk][1][c].
// Block (32 columns x 16 lanes): lane y sums blocks y, y+16, ... in order, then
// the 16 lane sums are added in lane order.
__global__ void ln_bwd_reduce_kernel(float* __restrict__ dw, float* __restrict__ db,
                                     const float* __restrict__ partial, int nblk, int C) {
    __shared__ float sh[16][33];
    const int c = blockIdx.x * 32 + threadIdx.x;
    float s = 0.f;
    if (c < 2 * C)
        for (int k = threadIdx.y; k < nblk; k += 16) s += partial[(size_t)k * 2 * C + c];
    sh[threadIdx.y][threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.y == 0 && c < 2 * C) {
        float t = sh[0][threadIdx.x];
        for (int k = 1; k < 16; k++) t += sh[k][threadIdx.x];
        if (c < C) dw[c] = t;
        else db[c - C] = t;
    }
}

static int ln_bwd_blocks(int N) { return std::min(ceil_div(N, 32), 512); }

}  // namespace gpt2k

using namespace gpt2k;

namespace gpt2k {
int layernorm_forward(void* y, bool out_bf16, float* mean, float* rstd, const float* x,
                      const float* w, const float* b, int N, int C, cudaStream_t st) {
    if (!y || !mean || !rstd || !x || !w || !b || N < 1 || C < 4 || C % 4 || C > 32 * 4 * LN_MAXV)
        return GPT2_EINVAL;
    if (!aligned16(y) || !aligned16(x) || !aligned16(w) || !aligned16(b)) return GPT2_EINVAL;
    dim3 grid(ceil_div(N, LN_WARPS));
    int nv = ceil_div(C / 4, 32);
#define LNF(NVV)                                                                                   \
    (out_bf16 ? (count_launch(), ln_fwd_kernel<NVV, true><<<grid, LN_WARPS * 32, 0, st>>>(y, mean, rstd, x, w, b, N, C)) \
              : (count_launch(), ln_fwd_kernel<NVV, false><<<grid, LN_WARPS * 32, 0, st>>>(y, mean, rstd, x, w, b, N, C)))
    if (nv <= 2) LNF(2);
    else if (nv <= 6) LNF(6);
    else if (nv <= 8) LNF(8);
    else if (nv <= 13) LNF(13);
    else LNF(LN_MAXV);
#undef LNF
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}
}  // namespace gpt2k

GPT2_API int gpt2_op_layernorm_forward(float* y, float* mean, float* rstd, const float* x,
                                       const float* w, const float* b, int N, int C,
                                       void* stream) {
    return layernorm_forward(y, false, mean, rstd, x, w, b, N, C, as_stream(stream));
}

GPT2_API int gpt2_op_layernorm_forward_bf16(void* y, float* mean, float* rstd, const float* x,
                                            const float* w, const float* b, int N, int C,
                                            void* stream) {
    return layernorm_forward(y, true, mean, rstd, x, w, b, N, C, as_stream(stream));
}

GPT2_API size_t gpt2_op_layernorm_backward_scratch_bytes(int N, int C) {
    if (N < 1 || C < 1) return 0;
    return (size_t)ln_bwd_blocks(N) * 2 * C * sizeof(float);
}

GPT2_API int gpt2_op_layernorm_backward(float* dx, void* dx_bf16, float* dw, float* db,
                                        const float* dy, const float* x, const float* w,
                                        const float* mean, const float* rstd, int N, int C,
                                        void* scratch, size_t scratch_bytes, void* stream) {
    if (!dx || !dw || !db || !dy || !x || !w || !mean || !rstd || N < 1 || C < 4 || C % 4 ||
        C > 32 * 4 * LN_MAXV)
        return GPT2_EINVAL;
    if (!aligned16(dx) || !aligned16(dy) || !aligned16(x) || !aligned16(w) || !aligned16(scratch))
        return GPT2_EINVAL;
    if (!scratch || scratch_bytes < gpt2_op_layernorm_backward_scratch_bytes(N, C)) return GPT2_ENOMEM;
    int nblk = ln_bwd_blocks(N);
    int rpb = ceil_div(N, nblk);
    float* partial = reinterpret_cast<float*>(scratch);
    size_t smem = 2 * (size_t)C * sizeof(float);
    int nv = ceil_div(C / 4, 32);
    cudaStream_t st = as_stream(stream);
    __nv_bfloat16* dx16 = static_cast<__nv_bfloat16*>(dx_bf16);
    if (dx16 && (reinterpret_cast<uintptr_t>(dx16) & 7)) return GPT2_EINVAL;
#define LNB(NVV) count_launch(), ln_bwd_kernel<NVV><<<nblk, LN_WARPS * 32, smem, st>>>(dx, dx16, partial, dy, x, w, mean, rstd, N, C, rpb)
    if (nv <= 2) LNB(2);
    else if (nv <= 6) LNB(6);
    else if (nv <= 8) LNB(8);
    else if (nv <= 13) LNB(13);
    else LNB(LN_MAXV);
#undef LNB
    count_launch(), ln_bwd_reduce_kernel<<<ceil_div(2 * C, 32), dim3(32, 16), 0, st>>>(dw, db, partial, nblk, C);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}
