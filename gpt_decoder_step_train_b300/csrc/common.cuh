// common.cuh -- shared helpers of the CUDA library (status codes, launch checks,
// vector types, GELU).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>
#include <algorithm>

#include "../../include/gpt2.h"
#include "../../include/gpt2_ops.h"

#define GPT2_API extern "C" __attribute__((visibility("default")))

namespace gpt2k {

static inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Return GPT2_ECUDA from the enclosing function when a launch or call failed.
#define GPT2_LAUNCH_CHECK()                                   \
    do {                                                      \
        if (cudaPeekAtLastError() != cudaSuccess) {           \
            (void)cudaGetLastError();                         \
            return GPT2_ECUDA;                                \
        }                                                     \
    } while (0)

#define GPT2_CUDA_TRY(call)                                   \
    do {                                                      \
        if ((call) != cudaSuccess) {                          \
            (void)cudaGetLastError();                         \
            return GPT2_ECUDA;                                \
        }                                                     \
    } while (0)

static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }
static inline size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

// Number of SMs of the current device (cached per process; one device).
int num_sms();

// Count one kernel launch (process-wide total, read by gpt2_kernel_launches).
void count_launch();

// Raise a kernel's dynamic shared-memory limit on the current device to at
// least `bytes` (never lowers it); thread-safe.  GPT2_OK or GPT2_ECUDA.
int smem_limit(const void* kernel, int bytes);

// tanh-form GELU and its derivative, fp32.  s = sqrt(2/pi).
#define GPT2_GELU_S 0.7978845608028654f
#define GPT2_GELU_K 0.044715f

__device__ __forceinline__ float gelu_fwd(float x) {
    float u = GPT2_GELU_S * (x + GPT2_GELU_K * x * x * x);
    return 0.5f * x * (1.0f + tanhf(u));
}

__device__ __forceinline__ float gelu_grad(float x) {
    float x2 = x * x;
    float u = GPT2_GELU_S * (x + GPT2_GELU_K * x2 * x);
    float th = tanhf(u);
    return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * GPT2_GELU_S * (1.0f + 3.0f * GPT2_GELU_K * x2);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Column sums over a warp whose lane i holds row i of a 32 x NV block (NV a
// power of two, 16 <= NV <= 64), in a fixed butterfly order (bit-reproducible).
// Each step halves the values a lane keeps: at offset o the lane keeps the upper
// half if (lane & o), the lower half otherwise, and adds its partner's copy of
// the kept half.  After the last step v[0 .. NV/32) (NV >= 32), or v[0] (NV 16,
// then duplicated in lanes 2j and 2j+1), hold whole-warp sums; the column of
// v[j] is warp_colsum_col<NV>(lane) + j.
template <int NV>
__device__ __forceinline__ void warp_colsum(float (&v)[NV], int lane) {
    static_assert(NV == 16 || NV == 32 || NV == 64, "16, 32 or 64 columns");
    int n = NV;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        if (n == 1) {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
            continue;
        }
        const int h = n >> 1;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < NV / 2; j++) {
            if (j < h) {
                const float send = upper ? v[j] : v[h + j];
                const float keep = upper ? v[h + j] : v[j];
                v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
        n = h;
    }
}

template <int NV>
__device__ __forceinline__ int warp_colsum_col(int lane) {
    // the kept half at offset 16, 8, ... supplies the column's bits from the top
    int col = 0, n = NV;
#pragma unroll
    for (int o = 16; o > 0 && n > 1; o >>= 1) {
        n >>= 1;
        if (lane & o) col += n;
    }
    return col;
}

__device__ __forceinline__ void set_status(int* status, int bit) {
    if (status) atomicOr(status, bit);
}

}  // namespace gpt2k
