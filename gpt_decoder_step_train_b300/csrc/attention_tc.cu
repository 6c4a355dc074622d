// attention_tc.cu -- causal multi-head self-attention on the tensor cores
// (warp-level mma.sync m16n8k8, tf32 operands, fp32 accumulation).
//
// Same mathematics as attention.cu (see there and "GPT-2 from scratch with
// torch", section 自注意力): per (b, h), S = Q K^T / sqrt(hs), causal -inf
// mask, row softmax, O = P V; lse saved; the backward recomputes P.
//
// Forward: one block per (64-query tile, head, batch), 4 warps x 16 query
// rows.  The warp keeps its Q rows as tf32 A-fragments and its O rows as
// accumulators; key/value tiles of 64 rows stream through shared memory with
// cp.async (double buffer); scores are kept in the log2 domain (Q pre-scaled
// by log2(e)/sqrt(hs)) for exp2; P is moved from the accumulator layout to the
// A-fragment layout with quad shuffles.  Key tiles beyond the block's last
// query are skipped; the diagonal tile is masked element by element.
//
// Backward, deterministic (every output element has one owner, no atomics):
//   dK/dV pass: block per 64-key tile, warp per 16 keys, looping over 32-query
//     tiles at or after the keys: P^T, dV += P^T dO, dP^T = V dO^T,
//     dS^T = P^T (dP^T - D), dK += dS^T Q.
//   dQ pass: block per 64-query tile, looping over key tiles at or before the
//     queries: P, dP = dO V^T, dS, dQ += dS K.
#include <cuda_bf16.h>

#include "common.cuh"

namespace gpt2k {
namespace atc {

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// D += A(16x8, row) * B(8x8, col), tf32 in, fp32 accumulate.
//   A: a0 (g, t) a1 (g+8, t) a2 (g, t+4) a3 (g+8, t+4)
//   B: b0 (k=t, n=g) b1 (k=t+4, n=g)
//   D: d0 (g, 2t) d1 (g, 2t+1) d2 (g+8, 2t) d3 (g+8, 2t+1)
// with g = lane/4, t = lane%4.
__device__ __forceinline__ void mma8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Accumulator fragment of a 16x8 block -> A fragment of the same block (tf32).
__device__ __forceinline__ void acc_to_a(const float (&c)[4], uint32_t (&a)[4], int lane) {
    const int t = lane & 3;
    const int s0 = (lane & ~3) | (t >> 1), s1 = (lane & ~3) | (2 + (t >> 1));
    const bool odd = t & 1;
    float x0 = __shfl_sync(0xffffffffu, c[0], s0), x1 = __shfl_sync(0xffffffffu, c[1], s0);
    float y0 = __shfl_sync(0xffffffffu, c[2], s0), y1 = __shfl_sync(0xffffffffu, c[3], s0);
    float z0 = __shfl_sync(0xffffffffu, c[0], s1), z1 = __shfl_sync(0xffffffffu, c[1], s1);
    float w0 = __shfl_sync(0xffffffffu, c[2], s1), w1 = __shfl_sync(0xffffffffu, c[3], s1);
    a[0] = tf32(odd ? x1 : x0);
    a[1] = tf32(odd ? y1 : y0);
    a[2] = tf32(odd ? z1 : z0);
    a[3] = tf32(odd ? w1 : w0);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Rows [r0, r0+R) of a row-major matrix (row stride ld, column offset already
// applied in g) into shared memory with row stride S floats; rows >= T zero.
template <int R, int HS, int S>
__device__ __forceinline__ void load_tile(float* sm, const float* g, size_t ld, int r0, int T) {
    constexpr int CH = HS / 4;
    for (int i = threadIdx.x; i < R * CH; i += blockDim.x) {
        const int r = i / CH, c = (i % CH) * 4;
        const int row = r0 + r;
        const bool valid = row < T;
        cp_async16(smem_u32(sm + r * S + c), g + (size_t)(valid ? row : 0) * ld + c, valid);
    }
}

// A fragments of 16 rows x HS of a row-major matrix (row stride ld), times mul.
template <int HS>
__device__ __forceinline__ void load_a_rows(uint32_t (&a)[HS / 8][4], const float* g, size_t ld,
                                            int row0, int T, float mul, int lane) {
    const int gi = lane >> 2, t = lane & 3;
    const int r0 = row0 + gi, r1 = r0 + 8;
#pragma unroll
    for (int kk = 0; kk < HS / 8; kk++) {
        const int c0 = kk * 8 + t, c1 = c0 + 4;
        a[kk][0] = tf32(r0 < T ? g[(size_t)r0 * ld + c0] * mul : 0.f);
        a[kk][1] = tf32(r1 < T ? g[(size_t)r1 * ld + c0] * mul : 0.f);
        a[kk][2] = tf32(r0 < T ? g[(size_t)r0 * ld + c1] * mul : 0.f);
        a[kk][3] = tf32(r1 < T ? g[(size_t)r1 * ld + c1] * mul : 0.f);
    }
}

// ---------------------------------------------------------------- forward
template <int HS>
__global__ void __launch_bounds__(128)
attn_fwd_tc(float* __restrict__ y, float* __restrict__ lse, const float* __restrict__ qkv, int T,
            int C, int H, float scale_log2) {
    constexpr int BQ = 64, BKV = 64, KS = HS + 4, VS = HS + 8;
    extern __shared__ __align__(16) float smem[];
    float* const Kbase = smem;                     // [2][BKV*KS]
    float* const Vbase = smem + 2 * BKV * KS;      // [2][BKV*VS]
    const int nq = (T + BQ - 1) / BQ;
    const int qt = nq - 1 - blockIdx.x;            // longest tiles first
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t4 = lane & 3;
    const int q0 = qt * BQ;
    const size_t ld = 3 * (size_t)C;
    const float* base = qkv + (size_t)b * T * ld;
    const float* Kg = base + C + h * HS;
    const float* Vg = base + 2 * C + h * HS;

    const int n_kt = min(q0 + BQ - 1, T - 1) / BKV + 1;
    load_tile<BKV, HS, KS>(Kbase, Kg, ld, 0, T);
    load_tile<BKV, HS, VS>(Vbase, Vg, ld, 0, T);
    cp_commit();

    uint32_t qa[HS / 8][4];
    const int rw = q0 + warp * 16;                 // first query row of this warp
    load_a_rows<HS>(qa, base + h * HS, ld, rw, T, scale_log2, lane);
    const int r0 = rw + gi, r1 = r0 + 8;

    float o[HS / 8][4];
#pragma unroll
    for (int n = 0; n < HS / 8; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int kt = 0; kt < n_kt; kt++) {
        const int buf = kt & 1;
        if (kt + 1 < n_kt) {
            load_tile<BKV, HS, KS>(Kbase + (buf ^ 1) * BKV * KS, Kg, ld, (kt + 1) * BKV, T);
            load_tile<BKV, HS, VS>(Vbase + (buf ^ 1) * BKV * VS, Vg, ld, (kt + 1) * BKV, T);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        const float* ks = Kbase + buf * BKV * KS;
        const float* vs = Vbase + buf * BKV * VS;
        const int j0 = kt * BKV;
        // S = Q K^T (log2 domain), 16 x 64 per warp
        float s[BKV / 8][4];
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < HS / 8; kk++) {
                const float* kr = ks + (nt * 8 + gi) * KS + kk * 8 + t4;
                mma8(s[nt], qa[kk], tf32(kr[0]), tf32(kr[4]));
            }
        }
        // causal / tail mask where the tile reaches past the first row of the warp
        if (j0 + BKV - 1 > rw || j0 + BKV > T) {
#pragma unroll
            for (int nt = 0; nt < BKV / 8; nt++) {
                const int j = j0 + nt * 8 + 2 * t4;
                if (j > r0 || j >= T) s[nt][0] = -INFINITY;
                if (j + 1 > r0 || j + 1 >= T) s[nt][1] = -INFINITY;
                if (j > r1 || j >= T) s[nt][2] = -INFINITY;
                if (j + 1 > r1 || j + 1 >= T) s[nt][3] = -INFINITY;
            }
        }
        float mx0 = m0, mx1 = m1;
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // every row sees key 0 in the first tile, so mx is finite from there on
        const float c0 = exp2f(m0 - mx0), c1 = exp2f(m1 - mx1);
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            s[nt][0] = exp2f(s[nt][0] - mx0);
            s[nt][1] = exp2f(s[nt][1] - mx0);
            s[nt][2] = exp2f(s[nt][2] - mx1);
            s[nt][3] = exp2f(s[nt][3] - mx1);
            ps0 += s[nt][0] + s[nt][1];
            ps1 += s[nt][2] + s[nt][3];
        }
        l0 = l0 * c0 + ps0;
        l1 = l1 * c1 + ps1;
        m0 = mx0;
        m1 = mx1;
#pragma unroll
        for (int n = 0; n < HS / 8; n++) {
            o[n][0] *= c0; o[n][1] *= c0;
            o[n][2] *= c1; o[n][3] *= c1;
        }
        // O += P V
#pragma unroll
        for (int kc = 0; kc < BKV / 8; kc++) {
            uint32_t pa[4];
            acc_to_a(s[kc], pa, lane);
#pragma unroll
            for (int nt = 0; nt < HS / 8; nt++) {
                const float* vr = vs + (kc * 8 + t4) * VS + nt * 8 + gi;
                mma8(o[nt], pa, tf32(vr[0]), tf32(vr[4 * VS]));
            }
        }
        __syncthreads();
    }
    // row sums are spread over the quad
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = 1.f / l0, i1 = 1.f / l1;
    float* y0 = y + ((size_t)b * T + r0) * C + h * HS;
    float* y1 = y + ((size_t)b * T + r1) * C + h * HS;
#pragma unroll
    for (int nt = 0; nt < HS / 8; nt++) {
        const int d = nt * 8 + 2 * t4;
        if (r0 < T) *reinterpret_cast<float2*>(y0 + d) = make_float2(o[nt][0] * i0, o[nt][1] * i0);
        if (r1 < T) *reinterpret_cast<float2*>(y1 + d) = make_float2(o[nt][2] * i1, o[nt][3] * i1);
    }
    if (t4 == 0) {
        float* lr = lse + ((size_t)b * H + h) * T;
        if (r0 < T) lr[r0] = (m0 + log2f(l0)) * LN2;
        if (r1 < T) lr[r1] = (m1 + log2f(l1)) * LN2;
    }
}

// ---------------------------------------------------------------- backward: dQ
template <int HS>
__global__ void __launch_bounds__(128)
attn_bwd_dq_tc(float* __restrict__ dqkv, const float* __restrict__ dy,
               const float* __restrict__ qkv, const float* __restrict__ lse,
               const float* __restrict__ Dg, int T, int C, int H, float scale) {
    constexpr int BQ = 64, BKV = 64, KS = HS + 4;
    extern __shared__ __align__(16) float smem[];
    float* const Kbase = smem;                     // [2][BKV*KS]
    float* const Vbase = smem + 2 * BKV * KS;      // [2][BKV*KS]
    const int nq = (T + BQ - 1) / BQ;
    const int qt = nq - 1 - blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t4 = lane & 3;
    const int q0 = qt * BQ;
    const size_t ld = 3 * (size_t)C;
    const float* base = qkv + (size_t)b * T * ld;
    const float* Kg = base + C + h * HS;
    const float* Vg = base + 2 * C + h * HS;
    const float scale_log2 = scale * LOG2E;

    const int n_kt = min(q0 + BQ - 1, T - 1) / BKV + 1;
    load_tile<BKV, HS, KS>(Kbase, Kg, ld, 0, T);
    load_tile<BKV, HS, KS>(Vbase, Vg, ld, 0, T);
    cp_commit();

    const int rw = q0 + warp * 16;
    const int r0 = rw + gi, r1 = r0 + 8;
    uint32_t qa[HS / 8][4], ga[HS / 8][4];
    load_a_rows<HS>(qa, base + h * HS, ld, rw, T, scale_log2, lane);
    load_a_rows<HS>(ga, dy + (size_t)b * T * C + h * HS, C, rw, T, 1.f, lane);
    const float* lbh = lse + ((size_t)b * H + h) * T;
    const float* dbh = Dg + ((size_t)b * H + h) * T;
    const float L0 = r0 < T ? lbh[r0] * LOG2E : INFINITY, L1 = r1 < T ? lbh[r1] * LOG2E : INFINITY;
    const float D0 = r0 < T ? dbh[r0] : 0.f, D1 = r1 < T ? dbh[r1] : 0.f;

    float dq[HS / 8][4];
#pragma unroll
    for (int n = 0; n < HS / 8; n++) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;

    for (int kt = 0; kt < n_kt; kt++) {
        const int buf = kt & 1;
        if (kt + 1 < n_kt) {
            load_tile<BKV, HS, KS>(Kbase + (buf ^ 1) * BKV * KS, Kg, ld, (kt + 1) * BKV, T);
            load_tile<BKV, HS, KS>(Vbase + (buf ^ 1) * BKV * KS, Vg, ld, (kt + 1) * BKV, T);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        const float* ks = Kbase + buf * BKV * KS;
        const float* vs = Vbase + buf * BKV * KS;
        const int j0 = kt * BKV;
        float s[BKV / 8][4], dp[BKV / 8][4];
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            dp[nt][0] = dp[nt][1] = dp[nt][2] = dp[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < HS / 8; kk++) {
                const float* kr = ks + (nt * 8 + gi) * KS + kk * 8 + t4;
                mma8(s[nt], qa[kk], tf32(kr[0]), tf32(kr[4]));
                const float* vr = vs + (nt * 8 + gi) * KS + kk * 8 + t4;
                mma8(dp[nt], ga[kk], tf32(vr[0]), tf32(vr[4]));
            }
        }
        const bool edge = j0 + BKV - 1 > rw || j0 + BKV > T;
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            const int j = j0 + nt * 8 + 2 * t4;
            float p0 = exp2f(s[nt][0] - L0), p1 = exp2f(s[nt][1] - L0);
            float p2 = exp2f(s[nt][2] - L1), p3 = exp2f(s[nt][3] - L1);
            if (edge) {
                if (j > r0 || j >= T) p0 = 0.f;
                if (j + 1 > r0 || j + 1 >= T) p1 = 0.f;
                if (j > r1 || j >= T) p2 = 0.f;
                if (j + 1 > r1 || j + 1 >= T) p3 = 0.f;
            }
            s[nt][0] = p0 * (dp[nt][0] - D0);
            s[nt][1] = p1 * (dp[nt][1] - D0);
            s[nt][2] = p2 * (dp[nt][2] - D1);
            s[nt][3] = p3 * (dp[nt][3] - D1);
        }
        // dQ += dS K
#pragma unroll
        for (int kc = 0; kc < BKV / 8; kc++) {
            uint32_t da[4];
            acc_to_a(s[kc], da, lane);
#pragma unroll
            for (int nt = 0; nt < HS / 8; nt++) {
                const float* kr = ks + (kc * 8 + t4) * KS + nt * 8 + gi;
                mma8(dq[nt], da, tf32(kr[0]), tf32(kr[4 * KS]));
            }
        }
        __syncthreads();
    }
    float* out0 = dqkv + ((size_t)b * T + r0) * ld + h * HS;
    float* out1 = dqkv + ((size_t)b * T + r1) * ld + h * HS;
#pragma unroll
    for (int nt = 0; nt < HS / 8; nt++) {
        const int d = nt * 8 + 2 * t4;
        if (r0 < T) *reinterpret_cast<float2*>(out0 + d) = make_float2(dq[nt][0] * scale, dq[nt][1] * scale);
        if (r1 < T) *reinterpret_cast<float2*>(out1 + d) = make_float2(dq[nt][2] * scale, dq[nt][3] * scale);
    }
}

// ---------------------------------------------------------------- backward: dK, dV
template <int HS>
__global__ void __launch_bounds__(128)
attn_bwd_dkv_tc(float* __restrict__ dqkv, const float* __restrict__ dy,
                const float* __restrict__ qkv, const float* __restrict__ lse,
                const float* __restrict__ Dg, int T, int C, int H, float scale) {
    constexpr int BKV = 64, BQ = 32, QS = HS + 4, GS = HS + 8;
    extern __shared__ __align__(16) float smem[];
    float* const Qbase = smem;                              // [2][BQ*QS]
    float* const Gbase = smem + 2 * BQ * QS;                // [2][BQ*GS]
    float* const Lbase = smem + 2 * BQ * (QS + GS);         // [2][BQ]
    float* const Dbase = Lbase + 2 * BQ;                    // [2][BQ]
    const int nk = (T + BKV - 1) / BKV;
    const int kt = blockIdx.x;                     // key tile; early key tiles see the most queries
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t4 = lane & 3;
    const int j0 = kt * BKV;
    const size_t ld = 3 * (size_t)C;
    const float* base = qkv + (size_t)b * T * ld;
    const float* Qg = base + h * HS;
    const float* Gg = dy + (size_t)b * T * C + h * HS;
    const float* lbh = lse + ((size_t)b * H + h) * T;
    const float* dbh = Dg + ((size_t)b * H + h) * T;
    const float scale_log2 = scale * LOG2E;
    (void)nk;

    const int it0 = j0 / BQ;                       // first query tile that reaches these keys
    const int n_it = (T + BQ - 1) / BQ;
    auto load_q = [&](int it, int bf) {
        load_tile<BQ, HS, QS>(Qbase + bf * BQ * QS, Qg, ld, it * BQ, T);
        load_tile<BQ, HS, GS>(Gbase + bf * BQ * GS, Gg, C, it * BQ, T);
        if (threadIdx.x < BQ) {
            const int i = it * BQ + threadIdx.x;
            Lbase[bf * BQ + threadIdx.x] = i < T ? lbh[i] * LOG2E : INFINITY;
            Dbase[bf * BQ + threadIdx.x] = i < T ? dbh[i] : 0.f;
        }
    };
    load_q(it0, 0);
    cp_commit();

    const int kw = j0 + warp * 16;                 // first key row of this warp
    const int k0r = kw + gi, k1r = k0r + 8;
    uint32_t ka[HS / 8][4], va[HS / 8][4];
    load_a_rows<HS>(ka, base + C + h * HS, ld, kw, T, scale_log2, lane);
    load_a_rows<HS>(va, base + 2 * C + h * HS, ld, kw, T, 1.f, lane);

    float dk[HS / 8][4], dv[HS / 8][4];
#pragma unroll
    for (int n = 0; n < HS / 8; n++) {
        dk[n][0] = dk[n][1] = dk[n][2] = dk[n][3] = 0.f;
        dv[n][0] = dv[n][1] = dv[n][2] = dv[n][3] = 0.f;
    }

    for (int it = it0; it < n_it; it++) {
        const int buf = (it - it0) & 1;
        if (it + 1 < n_it) load_q(it + 1, buf ^ 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        const float* qs = Qbase + buf * BQ * QS;
        const float* gs = Gbase + buf * BQ * GS;
        const float* Lt = Lbase + buf * BQ;
        const float* Dt = Dbase + buf * BQ;
        const int i0 = it * BQ;
        // S^T = K Q^T and dP^T = V dO^T: 16 keys x 32 queries per warp
        float st[BQ / 8][4], dpt[BQ / 8][4];
#pragma unroll
        for (int nt = 0; nt < BQ / 8; nt++) {
            st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.f;
            dpt[nt][0] = dpt[nt][1] = dpt[nt][2] = dpt[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < HS / 8; kk++) {
                const float* qr = qs + (nt * 8 + gi) * QS + kk * 8 + t4;
                mma8(st[nt], ka[kk], tf32(qr[0]), tf32(qr[4]));
                const float* gr = gs + (nt * 8 + gi) * GS + kk * 8 + t4;
                mma8(dpt[nt], va[kk], tf32(gr[0]), tf32(gr[4]));
            }
        }
        // P^T (masked where query < key or query >= T via L = +inf), dS^T
        const bool edge = i0 < kw + 16;
#pragma unroll
        for (int nt = 0; nt < BQ / 8; nt++) {
            const int ic = nt * 8 + 2 * t4;        // query column within the tile
            const int i = i0 + ic;
            float p0 = exp2f(st[nt][0] - Lt[ic]), p1 = exp2f(st[nt][1] - Lt[ic + 1]);
            float p2 = exp2f(st[nt][2] - Lt[ic]), p3 = exp2f(st[nt][3] - Lt[ic + 1]);
            if (edge) {
                if (i < k0r) p0 = 0.f;
                if (i + 1 < k0r) p1 = 0.f;
                if (i < k1r) p2 = 0.f;
                if (i + 1 < k1r) p3 = 0.f;
            }
            st[nt][0] = p0; st[nt][1] = p1; st[nt][2] = p2; st[nt][3] = p3;
            dpt[nt][0] = p0 * (dpt[nt][0] - Dt[ic]);
            dpt[nt][1] = p1 * (dpt[nt][1] - Dt[ic + 1]);
            dpt[nt][2] = p2 * (dpt[nt][2] - Dt[ic]);
            dpt[nt][3] = p3 * (dpt[nt][3] - Dt[ic + 1]);
        }
        // dV += P^T dO ; dK += dS^T Q
#pragma unroll
        for (int kc = 0; kc < BQ / 8; kc++) {
            uint32_t pa[4], sa[4];
            acc_to_a(st[kc], pa, lane);
            acc_to_a(dpt[kc], sa, lane);
#pragma unroll
            for (int nt = 0; nt < HS / 8; nt++) {
                const float* gr = gs + (kc * 8 + t4) * GS + nt * 8 + gi;
                mma8(dv[nt], pa, tf32(gr[0]), tf32(gr[4 * GS]));
                const float* qr = qs + (kc * 8 + t4) * QS + nt * 8 + gi;
                mma8(dk[nt], sa, tf32(qr[0]), tf32(qr[4 * QS]));
            }
        }
        __syncthreads();
    }
    float* dk0 = dqkv + ((size_t)b * T + k0r) * ld + C + h * HS;
    float* dk1 = dqkv + ((size_t)b * T + k1r) * ld + C + h * HS;
    float* dv0 = dk0 + C;
    float* dv1 = dk1 + C;
#pragma unroll
    for (int nt = 0; nt < HS / 8; nt++) {
        const int d = nt * 8 + 2 * t4;
        if (k0r < T) {
            *reinterpret_cast<float2*>(dk0 + d) = make_float2(dk[nt][0] * scale, dk[nt][1] * scale);
            *reinterpret_cast<float2*>(dv0 + d) = make_float2(dv[nt][0], dv[nt][1]);
        }
        if (k1r < T) {
            *reinterpret_cast<float2*>(dk1 + d) = make_float2(dk[nt][2] * scale, dk[nt][3] * scale);
            *reinterpret_cast<float2*>(dv1 + d) = make_float2(dv[nt][2], dv[nt][3]);
        }
    }
}

// ================================================================ bf16 operands
// Same three kernels with bf16 Q, K, V, dO (and bf16 O, dQ, dK, dV out) on
// mma.sync m16n8k16.  With 16-bit operands the accumulator fragment of two
// adjacent 8-column blocks is exactly the A fragment of one k16 step, so P and
// dS feed the next product without shuffles; operands needed transposed (V,
// dO, Q, K as the k-by-n side) come from ldmatrix.trans.  Tiles are rows of
// HS+8 bf16 (16-byte aligned, conflict-free for both access patterns).

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
//   A: a0 (g, 2t..2t+1) a1 (g+8, 2t..) a2 (g, 2t+8..) a3 (g+8, 2t+8..)
//   B: b0 (k = 2t..2t+1, n = g) b1 (k = 2t+8.., n = g)
__device__ __forceinline__ void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 bf16 matrices, transposed: lane L gives the row address of matrix
// L/8; r[i] is this thread's fragment of matrix i.
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// B fragments (b0, b1) for two adjacent 8-wide n-tiles (n0, n0+8) of a k16 step
// (rows k0..k0+15) of a row-major [k][n] bf16 tile with row stride S elements.
__device__ __forceinline__ void b_frags_t(uint32_t (&b)[4], const __nv_bfloat16* tile, int S, int k0,
                                          int n0, int lane) {
    const int mat = lane >> 3, rin = lane & 7;
    const int row = k0 + (mat & 1) * 8 + rin;
    const int col = n0 + (mat >> 1) * 8;
    ldsm_x4_t(b, smem_u32(tile + row * S + col));
}

// A fragments of 16 rows x HS of a bf16 row-major matrix (row stride ld).
template <int HS>
__device__ __forceinline__ void load_a_bf16(uint32_t (&a)[HS / 16][4], const __nv_bfloat16* g,
                                            size_t ld, int row0, int T, int lane) {
    const int gi = lane >> 2, t = lane & 3;
    const int r0 = row0 + gi, r1 = r0 + 8;
#pragma unroll
    for (int kk = 0; kk < HS / 16; kk++) {
        const int c0 = kk * 16 + 2 * t, c1 = c0 + 8;
        a[kk][0] = r0 < T ? *reinterpret_cast<const uint32_t*>(g + (size_t)r0 * ld + c0) : 0u;
        a[kk][1] = r1 < T ? *reinterpret_cast<const uint32_t*>(g + (size_t)r1 * ld + c0) : 0u;
        a[kk][2] = r0 < T ? *reinterpret_cast<const uint32_t*>(g + (size_t)r0 * ld + c1) : 0u;
        a[kk][3] = r1 < T ? *reinterpret_cast<const uint32_t*>(g + (size_t)r1 * ld + c1) : 0u;
    }
}

// Rows [r0, r0+R) of a bf16 row-major matrix into shared memory (row stride S
// elements); rows >= T zero.
template <int R, int HS, int S>
__device__ __forceinline__ void load_tile_bf16(__nv_bfloat16* sm, const __nv_bfloat16* g, size_t ld,
                                               int r0, int T) {
    constexpr int CH = HS / 8;                     // 16-byte chunks per row
    for (int i = threadIdx.x; i < R * CH; i += blockDim.x) {
        const int r = i / CH, c = (i % CH) * 8;
        const int row = r0 + r;
        const bool valid = row < T;
        cp_async16(smem_u32(sm + r * S + c), g + (size_t)(valid ? row : 0) * ld + c, valid);
    }
}

template <int HS>
__global__ void __launch_bounds__(128)
attn_fwd_bf16(__nv_bfloat16* __restrict__ y, float* __restrict__ lse,
              const __nv_bfloat16* __restrict__ qkv, int T, int C, int H, float scale_log2) {
    constexpr int BQ = 64, BKV = 64, S = HS + 8;
    extern __shared__ __align__(16) __nv_bfloat16 smb[];
    __nv_bfloat16* const Kbase = smb;                 // [2][BKV*S]
    __nv_bfloat16* const Vbase = smb + 2 * BKV * S;   // [2][BKV*S]
    const int nq = (T + BQ - 1) / BQ;
    const int qt = nq - 1 - blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t4 = lane & 3;
    const int q0 = qt * BQ;
    const size_t ld = 3 * (size_t)C;
    const __nv_bfloat16* base = qkv + (size_t)b * T * ld;
    const __nv_bfloat16* Kg = base + C + h * HS;
    const __nv_bfloat16* Vg = base + 2 * C + h * HS;

    const int n_kt = min(q0 + BQ - 1, T - 1) / BKV + 1;
    load_tile_bf16<BKV, HS, S>(Kbase, Kg, ld, 0, T);
    load_tile_bf16<BKV, HS, S>(Vbase, Vg, ld, 0, T);
    cp_commit();

    uint32_t qa[HS / 16][4];
    const int rw = q0 + warp * 16;
    load_a_bf16<HS>(qa, base + h * HS, ld, rw, T, lane);
    const int r0 = rw + gi, r1 = r0 + 8;

    float o[HS / 8][4];
#pragma unroll
    for (int n = 0; n < HS / 8; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int kt = 0; kt < n_kt; kt++) {
        const int buf = kt & 1;
        if (kt + 1 < n_kt) {
            load_tile_bf16<BKV, HS, S>(Kbase + (buf ^ 1) * BKV * S, Kg, ld, (kt + 1) * BKV, T);
            load_tile_bf16<BKV, HS, S>(Vbase + (buf ^ 1) * BKV * S, Vg, ld, (kt + 1) * BKV, T);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        const __nv_bfloat16* ks = Kbase + buf * BKV * S;
        const __nv_bfloat16* vs = Vbase + buf * BKV * S;
        const int j0 = kt * BKV;
        float s[BKV / 8][4];
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < HS / 16; kk++) {
                const __nv_bfloat16* kr = ks + (nt * 8 + gi) * S + kk * 16 + 2 * t4;
                mma16(s[nt], qa[kk], *reinterpret_cast<const uint32_t*>(kr),
                      *reinterpret_cast<const uint32_t*>(kr + 8));
            }
#pragma unroll
            for (int e = 0; e < 4; e++) s[nt][e] *= scale_log2;
        }
        if (j0 + BKV - 1 > rw || j0 + BKV > T) {
#pragma unroll
            for (int nt = 0; nt < BKV / 8; nt++) {
                const int j = j0 + nt * 8 + 2 * t4;
                if (j > r0 || j >= T) s[nt][0] = -INFINITY;
                if (j + 1 > r0 || j + 1 >= T) s[nt][1] = -INFINITY;
                if (j > r1 || j >= T) s[nt][2] = -INFINITY;
                if (j + 1 > r1 || j + 1 >= T) s[nt][3] = -INFINITY;
            }
        }
        float mx0 = m0, mx1 = m1;
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float c0 = exp2f(m0 - mx0), c1 = exp2f(m1 - mx1);
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            s[nt][0] = exp2f(s[nt][0] - mx0);
            s[nt][1] = exp2f(s[nt][1] - mx0);
            s[nt][2] = exp2f(s[nt][2] - mx1);
            s[nt][3] = exp2f(s[nt][3] - mx1);
            ps0 += s[nt][0] + s[nt][1];
            ps1 += s[nt][2] + s[nt][3];
        }
        l0 = l0 * c0 + ps0;
        l1 = l1 * c1 + ps1;
        m0 = mx0;
        m1 = mx1;
#pragma unroll
        for (int n = 0; n < HS / 8; n++) {
            o[n][0] *= c0; o[n][1] *= c0;
            o[n][2] *= c1; o[n][3] *= c1;
        }
        // O += P V, k16 steps over the 64 keys
#pragma unroll
        for (int j = 0; j < BKV / 16; j++) {
            uint32_t pa[4] = {pack_bf16(s[2 * j][0], s[2 * j][1]), pack_bf16(s[2 * j][2], s[2 * j][3]),
                              pack_bf16(s[2 * j + 1][0], s[2 * j + 1][1]),
                              pack_bf16(s[2 * j + 1][2], s[2 * j + 1][3])};
#pragma unroll
            for (int nt = 0; nt < HS / 8; nt += 2) {
                uint32_t bv[4];
                b_frags_t(bv, vs, S, j * 16, nt * 8, lane);
                mma16(o[nt], pa, bv[0], bv[1]);
                mma16(o[nt + 1], pa, bv[2], bv[3]);
            }
        }
        __syncthreads();
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = 1.f / l0, i1 = 1.f / l1;
    __nv_bfloat16* y0 = y + ((size_t)b * T + r0) * C + h * HS;
    __nv_bfloat16* y1 = y + ((size_t)b * T + r1) * C + h * HS;
#pragma unroll
    for (int nt = 0; nt < HS / 8; nt++) {
        const int d = nt * 8 + 2 * t4;
        if (r0 < T) *reinterpret_cast<uint32_t*>(y0 + d) = pack_bf16(o[nt][0] * i0, o[nt][1] * i0);
        if (r1 < T) *reinterpret_cast<uint32_t*>(y1 + d) = pack_bf16(o[nt][2] * i1, o[nt][3] * i1);
    }
    if (t4 == 0) {
        float* lr = lse + ((size_t)b * H + h) * T;
        if (r0 < T) lr[r0] = (m0 + log2f(l0)) * LN2;
        if (r1 < T) lr[r1] = (m1 + log2f(l1)) * LN2;
    }
}

template <int HS>
__global__ void __launch_bounds__(128)
attn_bwd_dq_bf16(__nv_bfloat16* __restrict__ dqkv, const __nv_bfloat16* __restrict__ dy,
                 const __nv_bfloat16* __restrict__ qkv, const float* __restrict__ lse,
                 const float* __restrict__ Dg, int T, int C, int H, float scale) {
    constexpr int BQ = 64, BKV = 64, S = HS + 8;
    extern __shared__ __align__(16) __nv_bfloat16 smb[];
    __nv_bfloat16* const Kbase = smb;
    __nv_bfloat16* const Vbase = smb + 2 * BKV * S;
    const int nq = (T + BQ - 1) / BQ;
    const int qt = nq - 1 - blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t4 = lane & 3;
    const int q0 = qt * BQ;
    const size_t ld = 3 * (size_t)C;
    const __nv_bfloat16* base = qkv + (size_t)b * T * ld;
    const __nv_bfloat16* Kg = base + C + h * HS;
    const __nv_bfloat16* Vg = base + 2 * C + h * HS;
    const float scale_log2 = scale * LOG2E;

    const int n_kt = min(q0 + BQ - 1, T - 1) / BKV + 1;
    load_tile_bf16<BKV, HS, S>(Kbase, Kg, ld, 0, T);
    load_tile_bf16<BKV, HS, S>(Vbase, Vg, ld, 0, T);
    cp_commit();

    const int rw = q0 + warp * 16;
    const int r0 = rw + gi, r1 = r0 + 8;
    uint32_t qa[HS / 16][4], ga[HS / 16][4];
    load_a_bf16<HS>(qa, base + h * HS, ld, rw, T, lane);
    load_a_bf16<HS>(ga, dy + (size_t)b * T * C + h * HS, C, rw, T, lane);
    const float* lbh = lse + ((size_t)b * H + h) * T;
    const float* dbh = Dg + ((size_t)b * H + h) * T;
    const float L0 = r0 < T ? lbh[r0] * LOG2E : INFINITY, L1 = r1 < T ? lbh[r1] * LOG2E : INFINITY;
    const float D0 = r0 < T ? dbh[r0] : 0.f, D1 = r1 < T ? dbh[r1] : 0.f;

    float dq[HS / 8][4];
#pragma unroll
    for (int n = 0; n < HS / 8; n++) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;

    for (int kt = 0; kt < n_kt; kt++) {
        const int buf = kt & 1;
        if (kt + 1 < n_kt) {
            load_tile_bf16<BKV, HS, S>(Kbase + (buf ^ 1) * BKV * S, Kg, ld, (kt + 1) * BKV, T);
            load_tile_bf16<BKV, HS, S>(Vbase + (buf ^ 1) * BKV * S, Vg, ld, (kt + 1) * BKV, T);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        const __nv_bfloat16* ks = Kbase + buf * BKV * S;
        const __nv_bfloat16* vs = Vbase + buf * BKV * S;
        const int j0 = kt * BKV;
        float s[BKV / 8][4], dp[BKV / 8][4];
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            dp[nt][0] = dp[nt][1] = dp[nt][2] = dp[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < HS / 16; kk++) {
                const __nv_bfloat16* kr = ks + (nt * 8 + gi) * S + kk * 16 + 2 * t4;
                mma16(s[nt], qa[kk], *reinterpret_cast<const uint32_t*>(kr),
                      *reinterpret_cast<const uint32_t*>(kr + 8));
                const __nv_bfloat16* vr = vs + (nt * 8 + gi) * S + kk * 16 + 2 * t4;
                mma16(dp[nt], ga[kk], *reinterpret_cast<const uint32_t*>(vr),
                      *reinterpret_cast<const uint32_t*>(vr + 8));
            }
        }
        const bool edge = j0 + BKV - 1 > rw || j0 + BKV > T;
#pragma unroll
        for (int nt = 0; nt < BKV / 8; nt++) {
            const int j = j0 + nt * 8 + 2 * t4;
            float p0 = exp2f(s[nt][0] * scale_log2 - L0), p1 = exp2f(s[nt][1] * scale_log2 - L0);
            float p2 = exp2f(s[nt][2] * scale_log2 - L1), p3 = exp2f(s[nt][3] * scale_log2 - L1);
            if (edge) {
                if (j > r0 || j >= T) p0 = 0.f;
                if (j + 1 > r0 || j + 1 >= T) p1 = 0.f;
                if (j > r1 || j >= T) p2 = 0.f;
                if (j + 1 > r1 || j + 1 >= T) p3 = 0.f;
            }
            s[nt][0] = p0 * (dp[nt][0] - D0);
            s[nt][1] = p1 * (dp[nt][1] - D0);
            s[nt][2] = p2 * (dp[nt][2] - D1);
            s[nt][3] = p3 * (dp[nt][3] - D1);
        }
        // dQ += dS K
#pragma unroll
        for (int j = 0; j < BKV / 16; j++) {
            uint32_t da[4] = {pack_bf16(s[2 * j][0], s[2 * j][1]), pack_bf16(s[2 * j][2], s[2 * j][3]),
                              pack_bf16(s[2 * j + 1][0], s[2 * j + 1][1]),
                              pack_bf16(s[2 * j + 1][2], s[2 * j + 1][3])};
#pragma unroll
            for (int nt = 0; nt < HS / 8; nt += 2) {
                uint32_t bk[4];
                b_frags_t(bk, ks, S, j * 16, nt * 8, lane);
                mma16(dq[nt], da, bk[0], bk[1]);
                mma16(dq[nt + 1], da, bk[2], bk[3]);
            }
        }
        __syncthreads();
    }
    __nv_bfloat16* out0 = dqkv + ((size_t)b * T + r0) * ld + h * HS;
    __nv_bfloat16* out1 = dqkv + ((size_t)b * T + r1) * ld + h * HS;
#pragma unroll
    for (int nt = 0; nt < HS / 8; nt++) {
        const int d = nt * 8 + 2 * t4;
        if (r0 < T) *reinterpret_cast<uint32_t*>(out0 + d) = pack_bf16(dq[nt][0] * scale, dq[nt][1] * scale);
        if (r1 < T) *reinterpret_cast<uint32_t*>(out1 + d) = pack_bf16(dq[nt][2] * scale, dq[nt][3] * scale);
    }
}

template <int HS>
__global__ void __launch_bounds__(128)
attn_bwd_dkv_bf16(__nv_bfloat16* __restrict__ dqkv, const __nv_bfloat16* __restrict__ dy,
                  const __nv_bfloat16* __restrict__ qkv, const float* __restrict__ lse,
                  const float* __restrict__ Dg, int T, int C, int H, float scale) {
    constexpr int BKV = 64, BQ = 32, S = HS + 8;
    extern __shared__ __align__(16) __nv_bfloat16 smb[];
    __nv_bfloat16* const Qbase = smb;                          // [2][BQ*S]
    __nv_bfloat16* const Gbase = smb + 2 * BQ * S;             // [2][BQ*S]
    float* const Lbase = reinterpret_cast<float*>(smb + 4 * BQ * S);   // [2][BQ]
    float* const Dbase = Lbase + 2 * BQ;                                // [2][BQ]
    const int kt = blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gi = lane >> 2, t4 = lane & 3;
    const int j0 = kt * BKV;
    const size_t ld = 3 * (size_t)C;
    const __nv_bfloat16* base = qkv + (size_t)b * T * ld;
    const __nv_bfloat16* Qg = base + h * HS;
    const __nv_bfloat16* Gg = dy + (size_t)b * T * C + h * HS;
    const float* lbh = lse + ((size_t)b * H + h) * T;
    const float* dbh = Dg + ((size_t)b * H + h) * T;
    const float scale_log2 = scale * LOG2E;

    const int it0 = j0 / BQ;
    const int n_it = (T + BQ - 1) / BQ;
    auto load_q = [&](int it, int bf) {
        load_tile_bf16<BQ, HS, S>(Qbase + bf * BQ * S, Qg, ld, it * BQ, T);
        load_tile_bf16<BQ, HS, S>(Gbase + bf * BQ * S, Gg, C, it * BQ, T);
        if (threadIdx.x < BQ) {
            const int i = it * BQ + threadIdx.x;
            Lbase[bf * BQ + threadIdx.x] = i < T ? lbh[i] * LOG2E : INFINITY;
            Dbase[bf * BQ + threadIdx.x] = i < T ? dbh[i] : 0.f;
        }
    };
    load_q(it0, 0);
    cp_commit();

    const int kw = j0 + warp * 16;
    const int k0r = kw + gi, k1r = k0r + 8;
    uint32_t ka[HS / 16][4], va[HS / 16][4];
    load_a_bf16<HS>(ka, base + C + h * HS, ld, kw, T, lane);
    load_a_bf16<HS>(va, base + 2 * C + h * HS, ld, kw, T, lane);

    float dk[HS / 8][4], dv[HS / 8][4];
#pragma unroll
    for (int n = 0; n < HS / 8; n++) {
        dk[n][0] = dk[n][1] = dk[n][2] = dk[n][3] = 0.f;
        dv[n][0] = dv[n][1] = dv[n][2] = dv[n][3] = 0.f;
    }

    for (int it = it0; it < n_it; it++) {
        const int buf = (it - it0) & 1;
        if (it + 1 < n_it) load_q(it + 1, buf ^ 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        const __nv_bfloat16* qs = Qbase + buf * BQ * S;
        const __nv_bfloat16* gs = Gbase + buf * BQ * S;
        const float* Lt = Lbase + buf * BQ;
        const float* Dt = Dbase + buf * BQ;
        const int i0 = it * BQ;
        float st[BQ / 8][4], dpt[BQ / 8][4];
#pragma unroll
        for (int nt = 0; nt < BQ / 8; nt++) {
            st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.f;
            dpt[nt][0] = dpt[nt][1] = dpt[nt][2] = dpt[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < HS / 16; kk++) {
                const __nv_bfloat16* qr = qs + (nt * 8 + gi) * S + kk * 16 + 2 * t4;
                mma16(st[nt], ka[kk], *reinterpret_cast<const uint32_t*>(qr),
                      *reinterpret_cast<const uint32_t*>(qr + 8));
                const __nv_bfloat16* gr = gs + (nt * 8 + gi) * S + kk * 16 + 2 * t4;
                mma16(dpt[nt], va[kk], *reinterpret_cast<const uint32_t*>(gr),
                      *reinterpret_cast<const uint32_t*>(gr + 8));
            }
        }
        const bool edge = i0 < kw + 16;
#pragma unroll
        for (int nt = 0; nt < BQ / 8; nt++) {
            const int ic = nt * 8 + 2 * t4;
            const int i = i0 + ic;
            float p0 = exp2f(st[nt][0] * scale_log2 - Lt[ic]), p1 = exp2f(st[nt][1] * scale_log2 - Lt[ic + 1]);
            float p2 = exp2f(st[nt][2] * scale_log2 - Lt[ic]), p3 = exp2f(st[nt][3] * scale_log2 - Lt[ic + 1]);
            if (edge) {
                if (i < k0r) p0 = 0.f;
                if (i + 1 < k0r) p1 = 0.f;
                if (i < k1r) p2 = 0.f;
                if (i + 1 < k1r) p3 = 0.f;
            }
            st[nt][0] = p0; st[nt][1] = p1; st[nt][2] = p2; st[nt][3] = p3;
            dpt[nt][0] = p0 * (dpt[nt][0] - Dt[ic]);
            dpt[nt][1] = p1 * (dpt[nt][1] - Dt[ic + 1]);
            dpt[nt][2] = p2 * (dpt[nt][2] - Dt[ic]);
            dpt[nt][3] = p3 * (dpt[nt][3] - Dt[ic + 1]);
        }
        // dV += P^T dO ; dK += dS^T Q   (k16 steps over the 32 queries)
#pragma unroll
        for (int j = 0; j < BQ / 16; j++) {
            uint32_t pa[4] = {pack_bf16(st[2 * j][0], st[2 * j][1]), pack_bf16(st[2 * j][2], st[2 * j][3]),
                              pack_bf16(st[2 * j + 1][0], st[2 * j + 1][1]),
                              pack_bf16(st[2 * j + 1][2], st[2 * j + 1][3])};
            uint32_t sa[4] = {pack_bf16(dpt[2 * j][0], dpt[2 * j][1]),
                              pack_bf16(dpt[2 * j][2], dpt[2 * j][3]),
                              pack_bf16(dpt[2 * j + 1][0], dpt[2 * j + 1][1]),
                              pack_bf16(dpt[2 * j + 1][2], dpt[2 * j + 1][3])};
#pragma unroll
            for (int nt = 0; nt < HS / 8; nt += 2) {
                uint32_t bg[4], bq[4];
                b_frags_t(bg, gs, S, j * 16, nt * 8, lane);
                mma16(dv[nt], pa, bg[0], bg[1]);
                mma16(dv[nt + 1], pa, bg[2], bg[3]);
                b_frags_t(bq, qs, S, j * 16, nt * 8, lane);
                mma16(dk[nt], sa, bq[0], bq[1]);
                mma16(dk[nt + 1], sa, bq[2], bq[3]);
            }
        }
        __syncthreads();
    }
    __nv_bfloat16* dk0 = dqkv + ((size_t)b * T + k0r) * ld + C + h * HS;
    __nv_bfloat16* dk1 = dqkv + ((size_t)b * T + k1r) * ld + C + h * HS;
    __nv_bfloat16* dv0 = dk0 + C;
    __nv_bfloat16* dv1 = dk1 + C;
#pragma unroll
    for (int nt = 0; nt < HS / 8; nt++) {
        const int d = nt * 8 + 2 * t4;
        if (k0r < T) {
            *reinterpret_cast<uint32_t*>(dk0 + d) = pack_bf16(dk[nt][0] * scale, dk[nt][1] * scale);
            *reinterpret_cast<uint32_t*>(dv0 + d) = pack_bf16(dv[nt][0], dv[nt][1]);
        }
        if (k1r < T) {
            *reinterpret_cast<uint32_t*>(dk1 + d) = pack_bf16(dk[nt][2] * scale, dk[nt][3] * scale);
            *reinterpret_cast<uint32_t*>(dv1 + d) = pack_bf16(dv[nt][2], dv[nt][3]);
        }
    }
}

template <int HS>
constexpr size_t fwd_smem_bf16() { return 2 * sizeof(__nv_bfloat16) * 2 * 64 * (HS + 8); }
template <int HS>
constexpr size_t dq_smem_bf16() { return 2 * sizeof(__nv_bfloat16) * 2 * 64 * (HS + 8); }
template <int HS>
constexpr size_t dkv_smem_bf16() { return sizeof(__nv_bfloat16) * 4 * 32 * (HS + 8) + sizeof(float) * 4 * 32; }

template <int HS>
static int set_smem_attrs_bf16() {
    if (smem_limit(reinterpret_cast<const void*>(attn_fwd_bf16<HS>), (int)fwd_smem_bf16<HS>()) ||
        smem_limit(reinterpret_cast<const void*>(attn_bwd_dq_bf16<HS>), (int)dq_smem_bf16<HS>()) ||
        smem_limit(reinterpret_cast<const void*>(attn_bwd_dkv_bf16<HS>), (int)dkv_smem_bf16<HS>()))
        return GPT2_ECUDA;
    return GPT2_OK;
}

template <int HS>
static int launch_fwd_bf16(void* y, float* lse, const void* qkv, int B, int T, int C, int H,
                           cudaStream_t st) {
    int rc = set_smem_attrs_bf16<HS>();
    if (rc) return rc;
    const float scale_log2 = LOG2E / sqrtf((float)HS);
    count_launch(), attn_fwd_bf16<HS><<<dim3((T + 63) / 64, H, B), 128, fwd_smem_bf16<HS>(), st>>>(
        static_cast<__nv_bfloat16*>(y), lse, static_cast<const __nv_bfloat16*>(qkv), T, C, H, scale_log2);
    return GPT2_OK;
}

template <int HS>
static int launch_bwd_bf16(void* dqkv, const void* dy, const void* qkv, const float* lse,
                           const float* D, int B, int T, int C, int H, cudaStream_t st) {
    int rc = set_smem_attrs_bf16<HS>();
    if (rc) return rc;
    const float scale = 1.f / sqrtf((float)HS);
    auto* dq = static_cast<__nv_bfloat16*>(dqkv);
    auto* g = static_cast<const __nv_bfloat16*>(dy);
    auto* x = static_cast<const __nv_bfloat16*>(qkv);
    count_launch(), attn_bwd_dkv_bf16<HS><<<dim3((T + 63) / 64, H, B), 128, dkv_smem_bf16<HS>(), st>>>(dq, g, x, lse, D, T, C, H, scale);
    count_launch(), attn_bwd_dq_bf16<HS><<<dim3((T + 63) / 64, H, B), 128, dq_smem_bf16<HS>(), st>>>(dq, g, x, lse, D, T, C, H, scale);
    return GPT2_OK;
}

template <int HS>
constexpr size_t fwd_smem() { return sizeof(float) * 2 * 64 * ((HS + 4) + (HS + 8)); }
template <int HS>
constexpr size_t dq_smem() { return sizeof(float) * 4 * 64 * (HS + 4); }
template <int HS>
constexpr size_t dkv_smem() { return sizeof(float) * (2 * 32 * ((HS + 4) + (HS + 8)) + 4 * 32); }

template <int HS>
static int set_smem_attrs() {
    if (smem_limit(reinterpret_cast<const void*>(attn_fwd_tc<HS>), (int)fwd_smem<HS>()) ||
        smem_limit(reinterpret_cast<const void*>(attn_bwd_dq_tc<HS>), (int)dq_smem<HS>()) ||
        smem_limit(reinterpret_cast<const void*>(attn_bwd_dkv_tc<HS>), (int)dkv_smem<HS>()))
        return GPT2_ECUDA;
    return GPT2_OK;
}

template <int HS>
static int launch_fwd(float* y, float* lse, const float* qkv, int B, int T, int C, int H,
                      cudaStream_t st) {
    int rc = set_smem_attrs<HS>();
    if (rc) return rc;
    dim3 grid((T + 63) / 64, H, B);
    const float scale_log2 = LOG2E / sqrtf((float)HS);
    count_launch(), attn_fwd_tc<HS><<<grid, 128, fwd_smem<HS>(), st>>>(y, lse, qkv, T, C, H, scale_log2);
    return GPT2_OK;
}

template <int HS>
static int launch_bwd(float* dqkv, const float* dy, const float* qkv, const float* lse,
                      const float* D, int B, int T, int C, int H, cudaStream_t st) {
    int rc = set_smem_attrs<HS>();
    if (rc) return rc;
    const float scale = 1.f / sqrtf((float)HS);
    count_launch(), attn_bwd_dkv_tc<HS><<<dim3((T + 63) / 64, H, B), 128, dkv_smem<HS>(), st>>>(dqkv, dy, qkv, lse, D, T, C, H, scale);
    count_launch(), attn_bwd_dq_tc<HS><<<dim3((T + 63) / 64, H, B), 128, dq_smem<HS>(), st>>>(dqkv, dy, qkv, lse, D, T, C, H, scale);
    return GPT2_OK;
}

}  // namespace atc

bool attention_tc_supported(int hs) { return hs == 16 || hs == 32 || hs == 64; }

int attention_bf16_forward(void* y, float* lse, const void* qkv, int B, int T, int C, int H,
                           cudaStream_t st) {
    const int hs = C / H;
    int rc;
    if (hs == 64) rc = atc::launch_fwd_bf16<64>(y, lse, qkv, B, T, C, H, st);
    else if (hs == 32) rc = atc::launch_fwd_bf16<32>(y, lse, qkv, B, T, C, H, st);
    else if (hs == 16) rc = atc::launch_fwd_bf16<16>(y, lse, qkv, B, T, C, H, st);
    else return GPT2_ENOTSUP;
    if (rc) return rc;
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int attention_bf16_backward(void* dqkv, const void* dy, const void* qkv, const float* lse,
                            const float* D, int B, int T, int C, int H, cudaStream_t st) {
    const int hs = C / H;
    int rc;
    if (hs == 64) rc = atc::launch_bwd_bf16<64>(dqkv, dy, qkv, lse, D, B, T, C, H, st);
    else if (hs == 32) rc = atc::launch_bwd_bf16<32>(dqkv, dy, qkv, lse, D, B, T, C, H, st);
    else if (hs == 16) rc = atc::launch_bwd_bf16<16>(dqkv, dy, qkv, lse, D, B, T, C, H, st);
    else return GPT2_ENOTSUP;
    if (rc) return rc;
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int attention_tc_forward(float* y, float* lse, const float* qkv, int B, int T, int C, int H,
                         int* status, cudaStream_t st) {
    (void)status;
    const int hs = C / H;
    int rc;
    if (hs == 64) rc = atc::launch_fwd<64>(y, lse, qkv, B, T, C, H, st);
    else if (hs == 32) rc = atc::launch_fwd<32>(y, lse, qkv, B, T, C, H, st);
    else if (hs == 16) rc = atc::launch_fwd<16>(y, lse, qkv, B, T, C, H, st);
    else return GPT2_ENOTSUP;
    if (rc) return rc;
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

int attention_tc_backward(float* dqkv, const float* dy, const float* qkv, const float* lse,
                          const float* D, int B, int T, int C, int H, int* status,
                          cudaStream_t st) {
    (void)status;
    const int hs = C / H;
    int rc;
    if (hs == 64) rc = atc::launch_bwd<64>(dqkv, dy, qkv, lse, D, B, T, C, H, st);
    else if (hs == 32) rc = atc::launch_bwd<32>(dqkv, dy, qkv, lse, D, B, T, C, H, st);
    else if (hs == 16) rc = atc::launch_bwd<16>(dqkv, dy, qkv, lse, D, B, T, C, H, st);
    else return GPT2_ENOTSUP;
    if (rc) return rc;
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k
