// attention_tc05.cuh -- constants and device helpers shared by the tcgen05
// attention kernels (forward and backward, bf16 operands, head size 64):
// operand swizzle, exp2 on the special-function unit, bf16 packing, the qkv
// bias-gradient column sums, packed f32x2 arithmetic and wide tensor-memory
// loads.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gpt2k {
namespace at05 {

using namespace ptx;

constexpr int HS = 64;              // head size (one 128-byte swizzle row of bf16)
constexpr int BQ = 128;             // queries per tile (TMEM lanes)
// backward kernels: producer, MMA issuer and eight element-wise warps (two per
// TMEM lane quarter, one per half of the tile's 64 columns)
constexpr int BWD_EW_WARPS = 8;
constexpr int BWD_THREADS = 64 + 32 * BWD_EW_WARPS;
constexpr float RESCALE_LOG2 = 8.f;                // move the running maximum past 2^8 growth
constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;

// Forward work items (both forward kernels: 128-key tiles), heaviest first:
// item i is the query-tile pair npair - 1 - i / (B H) of (batch, head) number
// i % (B H); the CTAs of the persistent grid take items blockIdx.x,
// blockIdx.x + gridDim.x, ...
struct FwdItem {
    int b, h, qrow0, nkv0, nkv1, nkv;
};
__host__ __device__ __forceinline__ int fwd_items(int B, int T, int H) {
    return B * H * (((T + 127) / 128 + 1) / 2);
}
__device__ __forceinline__ FwdItem fwd_item(int i, int B, int T, int H) {
    const int npair = ((T + 127) / 128 + 1) / 2, nkt = (T + BQ - 1) / BQ;
    const int pi = npair - 1 - i / (B * H), bh = i % (B * H);
    FwdItem w;
    w.b = bh / H;
    w.h = bh % H;
    w.qrow0 = pi * 256;
    // key tiles each query tile needs (tile g ends at row qrow0 + 128 g + 127)
    w.nkv0 = min(2 * pi + 1, nkt);
    w.nkv1 = w.qrow0 + 128 < T ? min(2 * pi + 2, nkt) : 0;
    w.nkv = max(w.nkv0, w.nkv1);
    return w;
}

// Wait, bounded and ignoring the abort flag, for a barrier phase that copies
// this thread issued will complete (the drain before an aborting CTA leaves).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity) && globaltimer() - t0 < WAIT_NS) {
    }
}

// 128-byte swizzle of a K-major bf16 operand row: 16-byte chunk c of row r
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// 2^x on the special-function unit (inputs far below -126 flush to 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Column sums of one warp's 32 output rows (lane = row row0 + lane; rows past
// T hold 0) over 32 columns, for the bias gradient of the qkv projection:
// colsum [B * ceil(T/32), 3C], row group b * ceil(T/32) + row0/32, columns
// col0 .. col0+31.  Consumes v.
__device__ __forceinline__ void store_colsum(float* colsum, float (&v)[32], int lane, int b, int row0, int T,
                                             int C, int col0) {
    warp_colsum<32>(v, lane);
    if (row0 >= T) return;
    colsum[((size_t)b * ((T + 31) >> 5) + (row0 >> 5)) * 3 * C + col0 + warp_colsum_col<32>(lane)] = v[0];
}

__device__ __forceinline__ uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
// (a, b) * s + c on both lanes of a packed pair
__device__ __forceinline__ void fma2(float& a, float& b, uint64_t s, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2pack(a, b)), "l"(s), "l"(c));
    f2unpack(r, a, b);
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// 128 consecutive accumulator columns of this warp's 32 TMEM lanes into v
// (four loads, one wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
    float (&a)[32] = *reinterpret_cast<float(*)[32]>(&v[0]);
    float (&b)[32] = *reinterpret_cast<float(*)[32]>(&v[32]);
    float (&c)[32] = *reinterpret_cast<float(*)[32]>(&v[64]);
    float (&d)[32] = *reinterpret_cast<float(*)[32]>(&v[96]);
    tmem_ld32(taddr, a);
    tmem_ld32(taddr + 32, b);
    tmem_ld32(taddr + 64, c);
    tmem_ld32(taddr + 96, d);
    tmem_wait_ld(a);
    tmem_wait_ld(b);
    tmem_wait_ld(c);
    tmem_wait_ld(d);
}


}  // namespace at05
}  // namespace gpt2k
