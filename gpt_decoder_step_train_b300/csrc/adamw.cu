// adamw.cu -- fused AdamW update, 128-bit vectorised, one pass over p, g, m, v.
//
// The llm.c overview (bigegpt.com) runs its fine-tuning loop with Adam at
// lr 1e-4 after each forward/backward; the decoupled weight decay and bias
// correction follow the standard AdamW definition:
//   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
//   p -= lr * ((m/bc1) / (sqrt(v/bc2) + eps) + wd * p),  bc_k = 1 - b_k^t.
// Traffic: read p, g, m, v and write p, m, v: 28 bytes per parameter.
#include "common.cuh"

namespace gpt2k {

__device__ __forceinline__ float adam_one(float& p, float g, float& m, float& v, float lr, float b1,
                                          float b2, float eps, float wd, float bc1, float bc2) {
    m = b1 * m + (1.f - b1) * g;
    v = b2 * v + (1.f - b2) * g * g;
    float mh = m / bc1, vh = v / bc2;
    p -= lr * (mh / (sqrtf(vh) + eps) + wd * p);
    return p;
}

__global__ void adamw_kernel(float4* __restrict__ p, const float4* __restrict__ g, float4* __restrict__ m,
                             float4* __restrict__ v, size_t n4, float lr, float b1, float b2, float eps,
                             float wd, float bc1, float bc2) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        float4 pp = p[i], gg = __ldcs(&g[i]), mm = m[i], vv = v[i];
        adam_one(pp.x, gg.x, mm.x, vv.x, lr, b1, b2, eps, wd, bc1, bc2);
        adam_one(pp.y, gg.y, mm.y, vv.y, lr, b1, b2, eps, wd, bc1, bc2);
        adam_one(pp.z, gg.z, mm.z, vv.z, lr, b1, b2, eps, wd, bc1, bc2);
        adam_one(pp.w, gg.w, mm.w, vv.w, lr, b1, b2, eps, wd, bc1, bc2);
        p[i] = pp;
        __stcs(&m[i], mm);
        __stcs(&v[i], vv);
    }
}

}  // namespace gpt2k

using namespace gpt2k;

GPT2_API int gpt2_op_adamw(float* p, const float* g, float* m, float* v, size_t n, float lr,
                           float b1, float b2, float eps, float wd, float bc1, float bc2,
                           void* stream) {
    if (!p || !g || !m || !v || n % 4 || bc1 <= 0.f || bc2 <= 0.f) return GPT2_EINVAL;
    if (!aligned16(p) || !aligned16(g) || !aligned16(m) || !aligned16(v)) return GPT2_EINVAL;
    if (n == 0) return GPT2_OK;
    size_t n4 = n / 4;
    int blocks = (int)std::min<size_t>((n4 + 255) / 256, (size_t)num_sms() * 8);
    count_launch(), adamw_kernel<<<blocks, 256, 0, as_stream(stream)>>>(
        reinterpret_cast<float4*>(p), reinterpret_cast<const float4*>(g), reinterpret_cast<float4*>(m),
        reinterpret_cast<float4*>(v), n4, lr, b1, b2, eps, wd, bc1, bc2);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}
