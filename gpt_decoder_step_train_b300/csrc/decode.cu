// decode.cu -- autoregressive decoding with a key/value cache, and greedy
// token selection.
//
// One call advances B sequences by one position: embed the new tokens, then
// per block ln_1, c_attn (the new key and value rows go into the cache), causal
// attention of the new query over the cached keys 0..pos, c_proj + residual,
// ln_2, c_fc + GELU, c_proj + residual; ln_f and the tied lm_head give the
// logits of the new position.  Generation takes the next token from the last
// position's logits and appends it ("GPT-2 from scratch with torch", section
// 生成样本); earlier positions' rows are kept and only the new row is computed
// ("GPT-2ベースの3000バイトCで実装されたChatGPTクローン（2023）", section
// KVキャッシュ方式).  Everything is fp32 from the fp32
// parameters, whatever the training mode: with B <= 16 rows each product is a
// pass over its weights, so the kernels are weight-streaming dot products
// (one warp per output column, every row at once), bound by HBM.
#include <math.h>

#include "gemm.cuh"

namespace gpt2k {

constexpr int DEC_MAXB = 16;

// The decoding position lives in device memory (*dpos), so that one captured
// graph serves every position: the step's kernels read it and the last one
// advances it.

// x[b, :] = wte[tok[b], :] + wpe[pos, :]; an id outside [0, V) gives zeros and BAD_TOKEN
__global__ void decode_embed_kernel(float* __restrict__ x, const int* __restrict__ tok,
                                    const float* __restrict__ wte, const float* __restrict__ wpe, int B,
                                    int C, int V, const int* __restrict__ dpos, int* status) {
    const int b = blockIdx.x;
    const int t = tok[b], pos = *dpos;
    const bool ok = t >= 0 && t < V;
    if (!ok && threadIdx.x == 0) set_status(status, GPT2_STATUS_BAD_TOKEN);
    for (int c = threadIdx.x; c < C; c += blockDim.x)
        x[(size_t)b * C + c] = ok ? wte[(size_t)t * C + c] + wpe[(size_t)pos * C + c] : 0.f;
}

// out[b, o] = act(sum_k in[b, k] W[o, k] + bias[o]) + resid[b, o] for b < B <= 16;
// the qkv product also stores its key and value columns (o >= kv_c) into the
// cache row of position *dpos.
// HBM-bound (each weight read once per step, applied to every row).  A block of
// 8 warps covers 8 / S output columns with S warps per column, each warp one
// S-th of the row: its lanes issue up to eight 16-byte weight loads at once,
// then apply them to every input row; the S partial sums of a column are added
// in warp order through shared memory.  S > 1 keeps enough loads in flight when
// there are few columns.  The row count is a template parameter NB >= B
// (the rows B .. NB-1 of the input buffer are computed and dropped), so the
// inner loops carry no per-row tests.  act: 0 none, 1 tanh-GELU.  in [NB, IC]
// (row stride IC), out / resid [B, ld].
constexpr int DEC_GEMV_WARPS = 8, DEC_GEMV_U = 8;

struct DecGemv {
    float* out;
    int ld;
    const float *in, *W, *bias, *resid;
    int B, IC, OC, act, S;
    float* cache;               // key/value cache of the layer, or null
    int kv_c, maxT;             // first cached column (C); positions per cache row
    const int* dpos;
};

template <int NB>
__global__ void __launch_bounds__(32 * DEC_GEMV_WARPS) decode_gemv_kernel(const DecGemv p) {
    __shared__ float red[DEC_GEMV_WARPS][NB];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.S, IC = p.IC;
    const int o = blockIdx.x * (DEC_GEMV_WARPS / S) + w / S, part = w % S;
    const int k4n = IC >> 2, per = k4n / S, k4a = part * per, k4b = k4a + per;
    const float4* x4 = reinterpret_cast<const float4*>(p.in);
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; b++) acc[b] = 0.f;
    if (o < p.OC) {
        const float4* w4 = reinterpret_cast<const float4*>(p.W + (size_t)o * IC);
        for (int k0 = k4a; k0 < k4b; k0 += 32 * DEC_GEMV_U) {
            float4 wv[DEC_GEMV_U];
#pragma unroll
            for (int u = 0; u < DEC_GEMV_U; u++) {
                const int k4 = k0 + 32 * u + lane;
                wv[u] = k4 < k4b ? __ldg(w4 + k4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < DEC_GEMV_U; u++) {
                const int k4 = k0 + 32 * u + lane;
                if (k4 < k4b) {
#pragma unroll
                    for (int b = 0; b < NB; b++) {
                        const float4 xv = __ldg(x4 + (size_t)b * k4n + k4);
                        acc[b] += (wv[u].x * xv.x + wv[u].y * xv.y) + (wv[u].z * xv.z + wv[u].w * xv.w);
                    }
                }
            }
        }
    }
    // lane b ends with row b's sum of this warp's part
    float mine = 0.f;
#pragma unroll
    for (int b = 0; b < NB; b++) {
        const float v = warp_sum(acc[b]);
        if (lane == b) mine = v;
    }
    if (S > 1) {
        if (lane < NB) red[w][lane] = mine;
        __syncthreads();
        if (part == 0 && lane < p.B) {
            float v = 0.f;
            for (int q = 0; q < S; q++) v += red[w + q][lane];
            mine = v;
        }
    }
    if (part == 0 && o < p.OC && lane < p.B) {
        float v = mine;
        if (p.bias) v += p.bias[o];
        if (p.act == 1) v = gelu_fwd(v);
        if (p.resid) v += p.resid[(size_t)lane * p.ld + o];
        p.out[(size_t)lane * p.ld + o] = v;
        if (p.cache && o >= p.kv_c)
            p.cache[((size_t)lane * p.maxT + *p.dpos) * 2 * p.kv_c + (o - p.kv_c)] = v;
    }
}

// One block per (row b, head h), four warps splitting the keys 0..pos (warp w
// takes keys w, w + 4, ...): the score of a key is the warp's sum of the
// lanes' products over the head's dimensions (lane d holds dimensions d and
// d + 32), softmax with the block's maximum subtracted, then each warp sums
// its keys' weighted values and the four partial rows and sums are added in
// warp order.  hs <= 64.
constexpr int DEC_ATT_WARPS = 4;
constexpr int DEC_MAXT = 1024;

__global__ void __launch_bounds__(32 * DEC_ATT_WARPS)
decode_attn_kernel(float* __restrict__ y, const float* __restrict__ qkv, const float* __restrict__ cache, int B,
                   int C, int H, int maxT, const int* __restrict__ dpos, float scale) {
    __shared__ float sp[DEC_MAXT];
    __shared__ float sred[DEC_ATT_WARPS];
    __shared__ float sacc[DEC_ATT_WARPS][64];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pos = min(*dpos, DEC_MAXT - 1);
    const int b = blockIdx.x / H, h = blockIdx.x % H, hs = C / H;
    const float* q = qkv + (size_t)b * 3 * C + h * hs;
    const float* kb = cache + (size_t)b * maxT * 2 * C + h * hs;          // key j at kb + j * 2C, value at + C
    const bool d0 = lane < hs, d1 = lane + 32 < hs;
    const float q0 = d0 ? q[lane] * scale : 0.f, q1 = d1 ? q[lane + 32] * scale : 0.f;
    float mx = -INFINITY;
#pragma unroll 4
    for (int j = w; j <= pos; j += DEC_ATT_WARPS) {
        const float* kr = kb + (size_t)j * 2 * C;
        float s = (d0 ? q0 * kr[lane] : 0.f) + (d1 ? q1 * kr[lane + 32] : 0.f);
        s = warp_sum(s);
        if (lane == 0) sp[j] = s;
        mx = fmaxf(mx, s);
    }
    if (lane == 0) sred[w] = mx;
    __syncthreads();
    mx = sred[0];
    for (int k = 1; k < DEC_ATT_WARPS; k++) mx = fmaxf(mx, sred[k]);
    __syncthreads();                                                    // sred is reused below
    float a0 = 0.f, a1 = 0.f, sum = 0.f;
#pragma unroll 4
    for (int j = w; j <= pos; j += DEC_ATT_WARPS) {
        const float e = expf(sp[j] - mx);
        const float* vr = kb + (size_t)j * 2 * C + C;
        if (d0) a0 += e * vr[lane];
        if (d1) a1 += e * vr[lane + 32];
        sum += e;
    }
    if (lane == 0) sred[w] = sum;
    if (d0) sacc[w][lane] = a0;
    if (d1) sacc[w][lane + 32] = a1;
    __syncthreads();
    if (w == 0) {
        float l = 0.f;
        for (int k = 0; k < DEC_ATT_WARPS; k++) l += sred[k];
        const float inv = 1.f / l;
        for (int d = lane; d < hs; d += 32) {
            float v = 0.f;
            for (int k = 0; k < DEC_ATT_WARPS; k++) v += sacc[k][d];
            y[(size_t)b * C + h * hs + d] = v * inv;
        }
    }
}

// out[n] = the index of the largest of logits[n, 0..V) (the lowest on ties; NaN
// never wins).  One block per row, fixed-order reduction.
__global__ void argmax_kernel(int* __restrict__ out, const float* __restrict__ z, int V, int ld) {
    __shared__ float sv[32];
    __shared__ int si[32];
    const float* zr = z + (size_t)blockIdx.x * ld;
    float best = -INFINITY;
    int bi = -1;
    for (int v = threadIdx.x; v < V; v += blockDim.x) {    // ascending: the first maximum stays
        const float x = zr[v];
        if (x == x && (bi < 0 || x > best)) { best = x; bi = v; }
    }
    // warp: larger value wins, lower index on ties
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi >= 0 && (bi < 0 || ov > best || (ov == best && oi < bi))) { best = ov; bi = oi; }
    }
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sv[w] = best; si[w] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float b2 = sv[0];
        int i2 = si[0];
        for (int k = 1; k < (int)(blockDim.x >> 5); k++)
            if (si[k] >= 0 && (i2 < 0 || sv[k] > b2 || (sv[k] == b2 && si[k] < i2))) { b2 = sv[k]; i2 = si[k]; }
        out[blockIdx.x] = i2 < 0 ? 0 : i2;
    }
}

// Top-k sampling of one row per block ("GPT-2 from scratch with torch", section
// 生成样本: keep the k highest scores, softmax, draw from the distribution).
// The k largest of logits[n, 0..V) are found one by one in the order (value
// descending, index ascending), NaN entries skipped; the kept tokens, taken in
// ascending index order, get p = exp(z - zmax) / sum; the token is the first
// whose cumulative p exceeds the caller's draw u[n] in [0, 1) (the last kept
// token when rounding leaves u at or above the total).
constexpr int TOPK_MAX = 64;

__device__ __forceinline__ bool topk_better(float v, int i, float bv, int bi) {
    return bi < 0 || v > bv || (v == bv && i < bi);
}

__global__ void sample_topk_kernel(int* __restrict__ out, const float* __restrict__ z, int V, int ld, int k,
                                   const float* __restrict__ u) {
    __shared__ float sv[TOPK_MAX], wv[32];
    __shared__ int si[TOPK_MAX], wi[32];
    const float* zr = z + (size_t)blockIdx.x * ld;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    float pv = INFINITY;                 // the last kept (value, index): later picks rank below it
    int pi = -1;
    int n = 0;
    for (int j = 0; j < k; j++) {
        float bv = -INFINITY;
        int bi = -1;
        for (int v = threadIdx.x; v < V; v += blockDim.x) {
            const float x = zr[v];
            const bool below = x < pv || (x == pv && v > pi);
            if (x == x && below && topk_better(x, v, bv, bi)) { bv = x; bi = v; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi >= 0 && topk_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { wv[w] = bv; wi[w] = bi; }
        __syncthreads();
        if (threadIdx.x == 0) {
            float b2 = wv[0];
            int i2 = wi[0];
            for (int q = 1; q < nw; q++)
                if (wi[q] >= 0 && topk_better(wv[q], wi[q], b2, i2)) { b2 = wv[q]; i2 = wi[q]; }
            sv[j] = b2;
            si[j] = i2;
        }
        __syncthreads();
        pv = sv[j];
        pi = si[j];
        __syncthreads();                 // wv, wi are rewritten by the next pick
        if (pi < 0) break;               // fewer than k candidates
        n = j + 1;
    }
    if (threadIdx.x == 0) {
        if (n == 0) { out[blockIdx.x] = 0; return; }
        const float zmax = sv[0];
        // ascending index order (insertion sort of at most 64)
        for (int a = 1; a < n; a++) {
            const float tv = sv[a];
            const int ti = si[a];
            int b = a - 1;
            while (b >= 0 && si[b] > ti) { sv[b + 1] = sv[b]; si[b + 1] = si[b]; b--; }
            sv[b + 1] = tv;
            si[b + 1] = ti;
        }
        float S = 0.f;
        for (int a = 0; a < n; a++) S += expf(sv[a] - zmax);
        const float target = u[blockIdx.x] * S;
        float c = 0.f;
        int pick = si[n - 1];
        for (int a = 0; a < n; a++) {
            c += expf(sv[a] - zmax);
            if (c > target) { pick = si[a]; break; }
        }
        out[blockIdx.x] = pick;
    }
}

// ---- launchers ----------------------------------------------------------------
// The step's last kernel: the next call decodes the following position.
__global__ void decode_advance_kernel(int* dpos) { *dpos += 1; }

int decode_embed(float* x, const int* tok, const float* wte, const float* wpe, int B, int C, int V,
                 const int* dpos, int* status, cudaStream_t st) {
    count_launch(), decode_embed_kernel<<<B, 256, 0, st>>>(x, tok, wte, wpe, B, C, V, dpos, status);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

// decode_gemv with an optional store of the key and value columns into the
// cache (the qkv product: cache != null).
int decode_gemv(float* out, int ld, const float* in, const float* W, const float* bias, const float* resid,
                int B, int IC, int OC, int act, float* cache, int maxT, const int* dpos, cudaStream_t st) {
    if (B < 1 || B > DEC_MAXB || IC % 4 || !aligned16(in) || !aligned16(W)) return GPT2_EINVAL;
    if (cache && (OC % 3 || !dpos)) return GPT2_EINVAL;
    // warps per column: enough warps for every SM (about 16 each), splitting the
    // row evenly
    int S = 1;
    while (S < DEC_GEMV_WARPS && (long long)OC * S < 16LL * num_sms() && (IC / 4) % (2 * S) == 0) S *= 2;
    const DecGemv p{out, ld, in, W, bias, resid, B, IC, OC, act, S, cache, OC / 3, maxT, dpos};
    const dim3 grid(ceil_div(OC, DEC_GEMV_WARPS / S)), block(32 * DEC_GEMV_WARPS);
    const int nb = B == 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16;
    if (nb == 1) count_launch(), decode_gemv_kernel<1><<<grid, block, 0, st>>>(p);
    else if (nb == 2) count_launch(), decode_gemv_kernel<2><<<grid, block, 0, st>>>(p);
    else if (nb == 4) count_launch(), decode_gemv_kernel<4><<<grid, block, 0, st>>>(p);
    else if (nb == 8) count_launch(), decode_gemv_kernel<8><<<grid, block, 0, st>>>(p);
    else count_launch(), decode_gemv_kernel<16><<<grid, block, 0, st>>>(p);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

// Positions are below min(maxT, DEC_MAXT): checked by the caller before the
// step (the kernel clamps as well).
int decode_attention(float* y, const float* qkv, const float* cache, int B, int C, int H, int maxT,
                     const int* dpos, cudaStream_t st) {
    if (C / H > 64) return GPT2_EINVAL;
    const float scale = 1.f / sqrtf((float)(C / H));
    count_launch(), decode_attn_kernel<<<B * H, 32 * DEC_ATT_WARPS, 0, st>>>(y, qkv, cache, B, C, H, maxT, dpos,
                                                                             scale);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int decode_advance(int* dpos, cudaStream_t st) {
    count_launch(), decode_advance_kernel<<<1, 1, 0, st>>>(dpos);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k

using namespace gpt2k;

GPT2_API int gpt2_op_sample_topk(int* out, const float* logits, int N, int V, int ld, int k, const float* u,
                                  void* stream) {
    if (!out || !logits || !u || N < 1 || V < 1 || ld < V || k < 1 || k > TOPK_MAX) return GPT2_EINVAL;
    count_launch(), sample_topk_kernel<<<N, 256, 0, as_stream(stream)>>>(out, logits, V, ld, k, u);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

GPT2_API int gpt2_op_argmax(int* out, const float* logits, int N, int V, int ld, void* stream) {
    if (!out || !logits || N < 1 || V < 1 || ld < V) return GPT2_EINVAL;
    count_launch(), argmax_kernel<<<N, 256, 0, as_stream(stream)>>>(out, logits, V, ld);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}
