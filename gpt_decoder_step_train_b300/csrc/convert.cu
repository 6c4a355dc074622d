// convert.cu -- fp32 -> bf16 (round to nearest even), 128-bit loads.
#include <cuda_bf16.h>

#include "common.cuh"

namespace gpt2k {

__global__ void to_bf16_kernel(uint2* __restrict__ dst, const float4* __restrict__ src, size_t n4) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        float4 v = src[i];
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        dst[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
}

__global__ void to_bf16_tail_kernel(__nv_bfloat16* __restrict__ dst, const float* __restrict__ src,
                                    size_t from, size_t n) {
    size_t i = from + blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (i < n) dst[i] = __float2bfloat16_rn(src[i]);
}

int to_bf16(void* dst, const float* src, size_t n, cudaStream_t st) {
    if (n == 0) return GPT2_OK;
    size_t n4 = (aligned16(src) && (reinterpret_cast<uintptr_t>(dst) & 7) == 0) ? n / 4 : 0;
    if (n4) {
        int blocks = (int)std::min<size_t>((n4 + 255) / 256, (size_t)num_sms() * 8);
        count_launch(), to_bf16_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<uint2*>(dst),
                                                              reinterpret_cast<const float4*>(src), n4);
    }
    size_t done = n4 * 4;
    if (done < n) {
        size_t rest = n - done;
        count_launch(), to_bf16_tail_kernel<<<(unsigned)((rest + 255) / 256), 256, 0, st>>>(
            reinterpret_cast<__nv_bfloat16*>(dst), src, done, n);
    }
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k

using namespace gpt2k;

GPT2_API int gpt2_op_to_bf16(void* dst, const float* src, size_t n, void* stream) {
    if (!dst || !src) return GPT2_EINVAL;
    return to_bf16(dst, src, n, as_stream(stream));
}
