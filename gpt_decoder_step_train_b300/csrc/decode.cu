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

// x[b, :] = wte[tok[b], :] + wpe[pos, :]; an id outside [0, V) gives zeros and BAD_TOKEN
__global__ void decode_embed_kernel(float* __restrict__ x, const int* __restrict__ tok,
                                    const float* __restrict__ wte, const float* __restrict__ wpe, int B,
                                    int C, int V, int pos, int* status) {
    const int b = blockIdx.x;
    const int t = tok[b];
    const bool ok = t >= 0 && t < V;
    if (!ok && threadIdx.x == 0) set_status(status, GPT2_STATUS_BAD_TOKEN);
    for (int c = threadIdx.x; c < C; c += blockDim.x)
        x[(size_t)b * C + c] = ok ? wte[(size_t)t * C + c] + wpe[(size_t)pos * C + c] : 0.f;
}

// out[b, o] = act(sum_k in[b, k] W[o, k] + bias[o]) + resid[b, o] for b < B <= 16.
// One warp per output column: the weight row is read once (16-byte loads) and
// applied to every input row; lane partial sums are combined in a fixed tree.
// act: 0 none, 1 tanh-GELU.  in [B, IC] (row stride IC), out / resid [B, ld].
__global__ void decode_gemv_kernel(float* __restrict__ out, int ld, const float* __restrict__ in,
                                   const float* __restrict__ W, const float* __restrict__ bias,
                                   const float* __restrict__ resid, int B, int IC, int OC, int act) {
    const int o = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (o >= OC) return;
    float acc[DEC_MAXB];
#pragma unroll
    for (int b = 0; b < DEC_MAXB; b++) acc[b] = 0.f;
    const float4* w4 = reinterpret_cast<const float4*>(W + (size_t)o * IC);
    const int k4n = IC >> 2;
    for (int k4 = lane; k4 < k4n; k4 += 32) {
        const float4 w = __ldg(w4 + k4);
#pragma unroll
        for (int b = 0; b < DEC_MAXB; b++) {
            if (b < B) {
                const float4 xv = __ldg(reinterpret_cast<const float4*>(in + (size_t)b * IC) + k4);
                acc[b] += (w.x * xv.x + w.y * xv.y) + (w.z * xv.z + w.w * xv.w);
            }
        }
    }
#pragma unroll
    for (int b = 0; b < DEC_MAXB; b++) {
        if (b < B) {
            float v = warp_sum(acc[b]);
            if (lane == b) {
                if (bias) v += bias[o];
                if (act == 1) v = gelu_fwd(v);
                if (resid) v += resid[(size_t)b * ld + o];
                out[(size_t)b * ld + o] = v;
            }
        }
    }
}

// The new position's key and value rows into the cache: cache[b][pos] = qkv[b, C:3C].
__global__ void decode_kv_store_kernel(float* __restrict__ cache, const float* __restrict__ qkv, int B, int C,
                                       int maxT, int pos) {
    const int b = blockIdx.x;
    float* dst = cache + ((size_t)b * maxT + pos) * 2 * C;
    for (int c = threadIdx.x; c < 2 * C; c += blockDim.x) dst[c] = qkv[(size_t)b * 3 * C + C + c];
}

// One warp per (row b, head h): scores of the new query against keys 0..pos,
// softmax (maximum subtracted), weighted sum of the values.  hs <= 64.
constexpr int DEC_ATT_WARPS = 4;
constexpr int DEC_MAXT = 1024;

__global__ void decode_attn_kernel(float* __restrict__ y, const float* __restrict__ qkv,
                                   const float* __restrict__ cache, int B, int C, int H, int maxT, int pos,
                                   float scale) {
    __shared__ float sp[DEC_ATT_WARPS][DEC_MAXT];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x * DEC_ATT_WARPS + w;
    if (bh >= B * H) return;
    const int b = bh / H, h = bh % H, hs = C / H;
    const float* q = qkv + (size_t)b * 3 * C + h * hs;
    const float* kb = cache + (size_t)b * maxT * 2 * C + h * hs;          // key j at kb + j * 2C
    float* p = sp[w];
    float mx = -INFINITY;
    for (int j = lane; j <= pos; j += 32) {
        const float* kr = kb + (size_t)j * 2 * C;
        float s = 0.f;
        for (int d = 0; d < hs; d++) s += q[d] * kr[d];
        s *= scale;
        p[j] = s;
        mx = fmaxf(mx, s);
    }
    mx = warp_max(mx);
    float sum = 0.f;
    for (int j = lane; j <= pos; j += 32) {
        const float e = expf(p[j] - mx);
        p[j] = e;
        sum += e;
    }
    sum = warp_sum(sum);
    __syncwarp();
    const float inv = 1.f / sum;
    for (int d = lane; d < hs; d += 32) {
        const float* vb = kb + C + d;                                       // value j, column d
        float acc = 0.f;
        for (int j = 0; j <= pos; j++) acc += p[j] * vb[(size_t)j * 2 * C];
        y[(size_t)b * C + h * hs + d] = acc * inv;
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
int decode_embed(float* x, const int* tok, const float* wte, const float* wpe, int B, int C, int V, int pos,
                 int* status, cudaStream_t st) {
    count_launch(), decode_embed_kernel<<<B, 256, 0, st>>>(x, tok, wte, wpe, B, C, V, pos, status);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int decode_gemv(float* out, int ld, const float* in, const float* W, const float* bias, const float* resid,
                int B, int IC, int OC, int act, cudaStream_t st) {
    if (B < 1 || B > DEC_MAXB || IC % 4 || !aligned16(in) || !aligned16(W)) return GPT2_EINVAL;
    constexpr int WARPS = 8;
    count_launch(), decode_gemv_kernel<<<ceil_div(OC, WARPS), 32 * WARPS, 0, st>>>(out, ld, in, W, bias, resid, B,
                                                                                IC, OC, act);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int decode_kv_store(float* cache, const float* qkv, int B, int C, int maxT, int pos, cudaStream_t st) {
    count_launch(), decode_kv_store_kernel<<<B, 256, 0, st>>>(cache, qkv, B, C, maxT, pos);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int decode_attention(float* y, const float* qkv, const float* cache, int B, int C, int H, int maxT, int pos,
                     cudaStream_t st) {
    if (pos >= DEC_MAXT || C / H > 64) return GPT2_EINVAL;
    const float scale = 1.f / sqrtf((float)(C / H));
    count_launch(), decode_attn_kernel<<<ceil_div(B * H, DEC_ATT_WARPS), 32 * DEC_ATT_WARPS, 0, st>>>(
        y, qkv, cache, B, C, H, maxT, pos, scale);
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
