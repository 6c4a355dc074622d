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
// The backward also returns the column sum of the gradient it leaves in dx,
// which is the bias gradient of the projection that wrote the residual.  All
// column sums are deterministic: each block sums its rows in a fixed order
// into a per-block partial, and a second kernel sums the partials in block
// order.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "dropout.cuh"
#include "ptx.cuh"

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

// ---------------------------------------------------------------- backward
// Persistent: two blocks per SM; block blk owns the rows [blk*rpb, min(N, (blk+1)*rpb)) and
// walks them in tiles of `rb` rows.  Thread 0 streams each tile's rows of x,
// dy and (when accumulating) the incoming dx into a ring of shared-memory
// stages with bulk copies; then
//   phase 1, one warp per row: the two row means of g = dy*w and g*xhat, the
//            new dx row (fp32 and optionally bf16) written to global memory
//            and kept in the stage for phase 2;
//   phase 2, one thread per column: dw += dy*xhat, db += dy, ds += dx over the
//            tile's rows, in row order.
// Each block writes its column sums to partial[blk][3][C]; a second kernel adds
// the blocks in block order.  ds is the column sum of the gradient leaving the
// LayerNorm: the bias gradient of the projection that wrote the residual.
constexpr int LNB_THREADS = 256;
constexpr int LNB_WARPS = LNB_THREADS / 32;
constexpr int LNB_BLOCKS_PER_SM = 2;
constexpr int LNB_MAX_STAGES = 4;
constexpr int LNB_MAX_BLOCKS = 512;
constexpr size_t LNB_SMEM_BUDGET = 110 * 1024;    // per block, two blocks per SM

struct LnbPlan {
    int rb, stages, grid, rpb;
    size_t stage_bytes;
};

// The largest tile (8, 4, 2 or 1 rows) that still leaves two stages in the budget.
static LnbPlan lnb_plan(int N, int C) {
    LnbPlan p;
    p.rb = 8;
    while (p.rb > 1 && 2 * (size_t)3 * p.rb * C * sizeof(float) > LNB_SMEM_BUDGET) p.rb /= 2;
    p.stage_bytes = (size_t)3 * p.rb * C * sizeof(float);
    p.stages = (int)std::max<size_t>(1, std::min<size_t>(LNB_MAX_STAGES, LNB_SMEM_BUDGET / p.stage_bytes));
    p.grid = std::min({LNB_BLOCKS_PER_SM * num_sms(), LNB_MAX_BLOCKS, ceil_div(N, p.rb)});
    p.rpb = ceil_div(N, p.grid);
    return p;
}

template <int CPT>   // columns per thread: ceil(C / LNB_THREADS)
__global__ void __launch_bounds__(LNB_THREADS, LNB_BLOCKS_PER_SM)
ln_bwd_kernel(float* __restrict__ dx, __nv_bfloat16* __restrict__ dx16, float* __restrict__ partial,
              const float* __restrict__ dy, const float* __restrict__ x, const float* __restrict__ w,
              const float* __restrict__ mean, const float* __restrict__ rstd, int N, int C, int rpb,
              int rb, int stages, int accumulate, int* status) {
    extern __shared__ __align__(128) float lsm[];
    __shared__ __align__(8) uint64_t full[LNB_MAX_STAGES];
    __shared__ float s_mu[8], s_rs[8];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C4 = C >> 2;
    const int r0 = blockIdx.x * rpb, r1 = min(N, r0 + rpb);
    const int ntiles = r0 < r1 ? (r1 - r0 + rb - 1) / rb : 0;
    const size_t tile = (size_t)rb * C;                // floats per array per stage
    auto stage = [&](int s) { return lsm + (size_t)s * 3 * tile; };
    if (tid == 0) {
        for (int s = 0; s < stages; s++) ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    int issued = 0;                                    // thread 0: tiles requested
    auto issue = [&](int t) {
        const int tr0 = r0 + t * rb, nr = min(rb, r1 - tr0), s = t % stages;
        const uint32_t bytes = (uint32_t)nr * C * sizeof(float);
        const uint32_t bar = ptx::smem_u32(&full[s]);
        float* st = stage(s);
        ptx::mbar_expect_tx(bar, bytes * (accumulate ? 3 : 2));
        ptx::bulk_g2s(ptx::smem_u32(st), x + (size_t)tr0 * C, bytes, bar);
        ptx::bulk_g2s(ptx::smem_u32(st + tile), dy + (size_t)tr0 * C, bytes, bar);
        if (accumulate) ptx::bulk_g2s(ptx::smem_u32(st + 2 * tile), dx + (size_t)tr0 * C, bytes, bar);
        issued++;
    };
    if (tid == 0)
        for (int t = 0; t < min(stages, ntiles); t++) issue(t);
    float aw[CPT], ab[CPT], as[CPT];
#pragma unroll
    for (int j = 0; j < CPT; j++) aw[j] = ab[j] = as[j] = 0.f;
    const float4* w4 = reinterpret_cast<const float4*>(w);
    int t = 0;
    for (; t < ntiles; t++) {
        const int s = t % stages, tr0 = r0 + t * rb, nr = min(rb, r1 - tr0);
        const bool got = ptx::mbar_wait_bounded(ptx::smem_u32(&full[s]), (uint32_t)(t / stages) & 1u);
        if (!__syncthreads_and(got)) break;
        float* xs = stage(s);
        float* gs = xs + tile;
        float* os = xs + 2 * tile;                     // incoming dx, then the new dx
        // phase 1: warp per row
        for (int r = warp; r < nr; r += LNB_WARPS) {
            const int row = tr0 + r;
            const float mu = mean[row], rs = rstd[row];
            if (lane == 0) { s_mu[r] = mu; s_rs[r] = rs; }
            const float4* xr = reinterpret_cast<const float4*>(xs + (size_t)r * C);
            const float4* gr = reinterpret_cast<const float4*>(gs + (size_t)r * C);
            float4* orow = reinterpret_cast<float4*>(os + (size_t)r * C);
            float sg = 0.f, sgx = 0.f;
            for (int c = lane; c < C4; c += 32) {
                const float4 xv = xr[c], d = gr[c], ww = __ldg(w4 + c);
                const float gx = d.x * ww.x, gy = d.y * ww.y, gz = d.z * ww.z, gw = d.w * ww.w;
                sg += (gx + gy) + (gz + gw);
                sgx += (gx * (xv.x - mu) * rs + gy * (xv.y - mu) * rs) + (gz * (xv.z - mu) * rs + gw * (xv.w - mu) * rs);
            }
            const float mg = warp_sum(sg) / (float)C, mgx = warp_sum(sgx) / (float)C;
            float4* dxr = reinterpret_cast<float4*>(dx + (size_t)row * C);
            for (int c = lane; c < C4; c += 32) {
                const float4 xv = xr[c], d = gr[c], ww = __ldg(w4 + c);
                float4 o = accumulate ? orow[c] : make_float4(0.f, 0.f, 0.f, 0.f);
                o.x += rs * (d.x * ww.x - mg - (xv.x - mu) * rs * mgx);
                o.y += rs * (d.y * ww.y - mg - (xv.y - mu) * rs * mgx);
                o.z += rs * (d.z * ww.z - mg - (xv.z - mu) * rs * mgx);
                o.w += rs * (d.w * ww.w - mg - (xv.w - mu) * rs * mgx);
                orow[c] = o;
                dxr[c] = o;
                if (dx16) {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
                    reinterpret_cast<uint2*>(dx16 + (size_t)row * C)[c] =
                        make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
                }
            }
        }
        __syncthreads();
        // phase 2: thread per column, rows in order
#pragma unroll
        for (int j = 0; j < CPT; j++) {
            const int c = tid + j * LNB_THREADS;
            if (c < C) {
                for (int r = 0; r < nr; r++) {
                    const float d = gs[(size_t)r * C + c];
                    aw[j] += d * ((xs[(size_t)r * C + c] - s_mu[r]) * s_rs[r]);
                    ab[j] += d;
                    as[j] += os[(size_t)r * C + c];
                }
            }
        }
        __syncthreads();                               // the stage is free again
        if (tid == 0 && t + stages < ntiles) issue(t + stages);
    }
    if (t < ntiles) {
        // a copy never arrived: flag it, and wait (bounded) for the copies still
        // writing into this block's shared memory before leaving
        if (tid == 0) {
            set_status(status, GPT2_STATUS_TIMEOUT);
            for (int u = t; u < issued; u++)
                (void)ptx::mbar_wait_bounded(ptx::smem_u32(&full[u % stages]), (uint32_t)(u / stages) & 1u);
        }
        return;
    }
    float* out = partial + (size_t)blockIdx.x * 3 * C;
#pragma unroll
    for (int j = 0; j < CPT; j++) {
        const int c = tid + j * LNB_THREADS;
        if (c < C) {
            out[c] = aw[j];
            out[C + c] = ab[j];
            out[2 * C + c] = as[j];
        }
    }
}

// Register-streaming backward for rows of at most 32 * 4 * V4 (<= 768) columns: one block
// of LNR_WARPS warps per SM, each warp walking its own rows one at a time with
// every load of the row in flight at once (x, dy and the incoming dx as
// float4), no shared-memory staging and no block barrier until the end.  Lane
// l owns the float4 columns l, l+32, ...; its column sums of dy*xhat, dy and
// the new dx stay in registers across the warp's rows (rows in order), then
// the block adds its warps' sums in warp order through shared memory into
// partial[blk][3][C], the same partial layout the tiled kernel above writes.
constexpr int LNR_WARPS = 12;

//
// DROP: the residual-stream gradient dx also feeds a dropped branch (a c_proj
// output that went through dropout before the residual addition).  The copy
// dxo then holds keep o dx / (1 - p) (bf16 or fp32), and the third column sum
// is that of the copy: the branch's bias gradient.  bits: keep bits of the
// branch, rows of ceil(C/32) words.
template <int V4, bool DROP>
__global__ void __launch_bounds__(LNR_WARPS * 32, 1)
ln_bwd_rows_kernel(float* __restrict__ dx, void* __restrict__ dxo, int dxo_bf16, float* __restrict__ partial,
                   const float* __restrict__ dy, const float* __restrict__ x, const float* __restrict__ w,
                   const float* __restrict__ mean, const float* __restrict__ rstd, int N, int C, int rpb,
                   int accumulate, const uint32_t* __restrict__ bits, float ks) {
    extern __shared__ __align__(16) float red[];       // [LNR_WARPS][3][C]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C4 = C >> 2;
    const int r0 = blockIdx.x * rpb, r1 = min(N, r0 + rpb);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    float4 aw[V4], ab[V4], as[V4];
#pragma unroll
    for (int k = 0; k < V4; k++) aw[k] = ab[k] = as[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float inv_c = 1.f / (float)C;
    for (int row = r0 + warp; row < r1; row += LNR_WARPS) {
        const float4* xr = reinterpret_cast<const float4*>(x + (size_t)row * C);
        const float4* gr = reinterpret_cast<const float4*>(dy + (size_t)row * C);
        float4* dr = reinterpret_cast<float4*>(dx + (size_t)row * C);
        float4 xv[V4], gv[V4], ov[V4];
#pragma unroll
        for (int k = 0; k < V4; k++) {
            const int c = lane + 32 * k;
            const bool in = c < C4;
            xv[k] = in ? __ldcs(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            gv[k] = in ? __ldcs(gr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            ov[k] = in && accumulate ? __ldcs(dr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float mu = __ldg(mean + row), rs = __ldg(rstd + row);
        float sg = 0.f, sgx = 0.f;
#pragma unroll
        for (int k = 0; k < V4; k++) {
            const int c = lane + 32 * k;
            if (c < C4) {
                const float4 ww = __ldg(w4 + c);
                const float gx = gv[k].x * ww.x, gy = gv[k].y * ww.y, gz = gv[k].z * ww.z, gw = gv[k].w * ww.w;
                // xv becomes xhat from here on
                xv[k].x = (xv[k].x - mu) * rs; xv[k].y = (xv[k].y - mu) * rs;
                xv[k].z = (xv[k].z - mu) * rs; xv[k].w = (xv[k].w - mu) * rs;
                sg += (gx + gy) + (gz + gw);
                sgx += (gx * xv[k].x + gy * xv[k].y) + (gz * xv[k].z + gw * xv[k].w);
            }
        }
        const float mg = warp_sum(sg) * inv_c, mgx = warp_sum(sgx) * inv_c;
#pragma unroll
        for (int k = 0; k < V4; k++) {
            const int c = lane + 32 * k;
            if (c < C4) {
                const float4 ww = __ldg(w4 + c);
                float4 o = ov[k];
                o.x += rs * (gv[k].x * ww.x - mg - xv[k].x * mgx);
                o.y += rs * (gv[k].y * ww.y - mg - xv[k].y * mgx);
                o.z += rs * (gv[k].z * ww.z - mg - xv[k].z * mgx);
                o.w += rs * (gv[k].w * ww.w - mg - xv[k].w * mgx);
                dr[c] = o;
                float4 om = o;
                if constexpr (DROP) {
                    const uint32_t mb = __ldg(bits + (size_t)row * ((C + 31) >> 5) + ((4 * c) >> 5)) >> ((4 * c) & 31);
                    om.x = (mb & 1u) ? o.x * ks : 0.f;
                    om.y = (mb & 2u) ? o.y * ks : 0.f;
                    om.z = (mb & 4u) ? o.z * ks : 0.f;
                    om.w = (mb & 8u) ? o.w * ks : 0.f;
                }
                if (dxo) {
                    if (!DROP || dxo_bf16) {
                        __nv_bfloat162 lo = __floats2bfloat162_rn(om.x, om.y), hi = __floats2bfloat162_rn(om.z, om.w);
                        reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(dxo) + (size_t)row * C)[c] =
                            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
                    } else {
                        reinterpret_cast<float4*>(static_cast<float*>(dxo) + (size_t)row * C)[c] = om;
                    }
                }
                aw[k].x += gv[k].x * xv[k].x; aw[k].y += gv[k].y * xv[k].y;
                aw[k].z += gv[k].z * xv[k].z; aw[k].w += gv[k].w * xv[k].w;
                ab[k].x += gv[k].x; ab[k].y += gv[k].y; ab[k].z += gv[k].z; ab[k].w += gv[k].w;
                as[k].x += om.x; as[k].y += om.y; as[k].z += om.z; as[k].w += om.w;
            }
        }
    }
    // the warps' column sums, added in warp order
    float4* mine = reinterpret_cast<float4*>(red + (size_t)warp * 3 * C);
#pragma unroll
    for (int k = 0; k < V4; k++) {
        const int c = lane + 32 * k;
        if (c < C4) {
            mine[c] = aw[k];
            mine[C4 + c] = ab[k];
            mine[2 * C4 + c] = as[k];
        }
    }
    __syncthreads();
    float* out = partial + (size_t)blockIdx.x * 3 * C;
    for (int i = threadIdx.x; i < 3 * C; i += LNR_WARPS * 32) {
        float t = red[i];
        for (int k = 1; k < LNR_WARPS; k++) t += red[(size_t)k * 3 * C + i];
        out[i] = t;
    }
}

// out_k[c] = sum_blk partial[blk][k][c] for k = 0 (dw), 1 (db), 2 (ds, when
// wanted).  Block (32 columns x 16 lanes): lane y sums blocks y, y+16, ... in
// order, then the 16 lane sums are added in lane order.
__global__ void ln_bwd_reduce_kernel(float* __restrict__ dw, float* __restrict__ db, float* __restrict__ ds,
                                     const float* __restrict__ partial, int nblk, int C) {
    __shared__ float sh[16][33];
    const int c = blockIdx.x * 32 + threadIdx.x;       // over 3C
    const int width = ds ? 3 * C : 2 * C;
    float s = 0.f;
    if (c < width)
        for (int k = threadIdx.y; k < nblk; k += 16) s += partial[(size_t)k * 3 * C + c];
    sh[threadIdx.y][threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.y == 0 && c < width) {
        float t = sh[0][threadIdx.x];
        for (int k = 1; k < 16; k++) t += sh[k][threadIdx.x];
        if (c < C) dw[c] = t;
        else if (c < 2 * C) db[c - C] = t;
        else ds[c - 2 * C] = t;
    }
}

// The same register streaming for rows of up to 2048 columns (V4 float4 per
// lane, V4 > 6): the row's x, dy and incoming dx stay in registers, but the
// column sums go to the warp's own [3][C] region of shared memory after every
// row (each lane updates its own columns, so no two lanes touch one word), which
// leaves the registers to the row itself; LNR_WIDE_WARPS warps per block.  The
// block then adds its warps' regions in warp order, as above.  No dropout.
constexpr int LNR_WIDE_WARPS = 8;

template <int V4>
__global__ void __launch_bounds__(LNR_WIDE_WARPS * 32, 1)
ln_bwd_rows_wide_kernel(float* __restrict__ dx, __nv_bfloat16* __restrict__ dx16, float* __restrict__ partial,
                        const float* __restrict__ dy, const float* __restrict__ x, const float* __restrict__ w,
                        const float* __restrict__ mean, const float* __restrict__ rstd, int N, int C, int rpb,
                        int accumulate) {
    extern __shared__ __align__(16) float red[];       // [LNR_WIDE_WARPS][3][C]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C4 = C >> 2;
    const int r0 = blockIdx.x * rpb, r1 = min(N, r0 + rpb);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    float4* acc = reinterpret_cast<float4*>(red + (size_t)warp * 3 * C);   // this warp's sums
    for (int c = lane; c < 3 * C4; c += 32) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float inv_c = 1.f / (float)C;
    for (int row = r0 + warp; row < r1; row += LNR_WIDE_WARPS) {
        const float4* xr = reinterpret_cast<const float4*>(x + (size_t)row * C);
        const float4* gr = reinterpret_cast<const float4*>(dy + (size_t)row * C);
        float4* dr = reinterpret_cast<float4*>(dx + (size_t)row * C);
        float4 xv[V4], gv[V4], ov[V4];
#pragma unroll
        for (int k = 0; k < V4; k++) {
            const int c = lane + 32 * k;
            const bool in = c < C4;
            xv[k] = in ? __ldcs(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            gv[k] = in ? __ldcs(gr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            ov[k] = in && accumulate ? __ldcs(dr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float mu = __ldg(mean + row), rs = __ldg(rstd + row);
        float sg = 0.f, sgx = 0.f;
#pragma unroll
        for (int k = 0; k < V4; k++) {
            const int c = lane + 32 * k;
            if (c < C4) {
                const float4 ww = __ldg(w4 + c);
                const float gx = gv[k].x * ww.x, gy = gv[k].y * ww.y, gz = gv[k].z * ww.z, gw = gv[k].w * ww.w;
                xv[k].x = (xv[k].x - mu) * rs; xv[k].y = (xv[k].y - mu) * rs;
                xv[k].z = (xv[k].z - mu) * rs; xv[k].w = (xv[k].w - mu) * rs;
                sg += (gx + gy) + (gz + gw);
                sgx += (gx * xv[k].x + gy * xv[k].y) + (gz * xv[k].z + gw * xv[k].w);
            }
        }
        const float mg = warp_sum(sg) * inv_c, mgx = warp_sum(sgx) * inv_c;
#pragma unroll
        for (int k = 0; k < V4; k++) {
            const int c = lane + 32 * k;
            if (c < C4) {
                const float4 ww = __ldg(w4 + c);
                float4 o = ov[k];
                o.x += rs * (gv[k].x * ww.x - mg - xv[k].x * mgx);
                o.y += rs * (gv[k].y * ww.y - mg - xv[k].y * mgx);
                o.z += rs * (gv[k].z * ww.z - mg - xv[k].z * mgx);
                o.w += rs * (gv[k].w * ww.w - mg - xv[k].w * mgx);
                dr[c] = o;
                if (dx16) {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
                    reinterpret_cast<uint2*>(dx16 + (size_t)row * C)[c] =
                        make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
                }
                float4 a = acc[c], b = acc[C4 + c], d = acc[2 * C4 + c];
                a.x += gv[k].x * xv[k].x; a.y += gv[k].y * xv[k].y;
                a.z += gv[k].z * xv[k].z; a.w += gv[k].w * xv[k].w;
                b.x += gv[k].x; b.y += gv[k].y; b.z += gv[k].z; b.w += gv[k].w;
                d.x += o.x; d.y += o.y; d.z += o.z; d.w += o.w;
                acc[c] = a;
                acc[C4 + c] = b;
                acc[2 * C4 + c] = d;
            }
        }
    }
    __syncthreads();
    float* out = partial + (size_t)blockIdx.x * 3 * C;
    for (int i = threadIdx.x; i < 3 * C; i += LNR_WIDE_WARPS * 32) {
        float t = red[i];
        for (int k = 1; k < LNR_WIDE_WARPS; k++) t += red[(size_t)k * 3 * C + i];
        out[i] = t;
    }
}

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
    return (size_t)LNB_MAX_BLOCKS * 3 * C * sizeof(float);
}

namespace gpt2k {

bool layernorm_backward_fuses_dropout(int C) { return C >= 4 && C % 4 == 0 && ceil_div(C / 4, 32) <= 6; }

// gpt2_op_layernorm_backward, with the operand copy dxo of dx in bf16 or fp32
// (dxo_bf16) and, when bits != null, dropout applied to that copy and to its
// column sum (rows of up to 768 columns: layernorm_backward_fuses_dropout).
int layernorm_backward(float* dx, void* dxo, bool dxo_bf16, float* dw, float* db, float* dx_colsum, const float* dy,
                       const float* x, const float* w, const float* mean, const float* rstd, int N, int C,
                       int accumulate, void* scratch, size_t scratch_bytes, int* status, cudaStream_t st,
                       const uint32_t* bits, float p, ColReduce* defer) {
    if (!dx || !dw || !db || !dy || !x || !w || !mean || !rstd || N < 1 || C < 4 || C % 4 ||
        C > LNB_THREADS * 8)
        return GPT2_EINVAL;
    if (!aligned16(dx) || !aligned16(dy) || !aligned16(x) || !aligned16(w) || !aligned16(scratch))
        return GPT2_EINVAL;
    if (!scratch || scratch_bytes < gpt2_op_layernorm_backward_scratch_bytes(N, C)) return GPT2_ENOMEM;
    if (dxo && (reinterpret_cast<uintptr_t>(dxo) & (dxo_bf16 ? 7u : 15u))) return GPT2_EINVAL;
    if (!dxo_bf16 && !bits && dxo) return GPT2_EINVAL;     // without dropout the copy is bf16
    if (bits && (!layernorm_backward_fuses_dropout(C) || !(p >= 0.f && p < 1.f))) return GPT2_ENOTSUP;
    __nv_bfloat16* dx16 = static_cast<__nv_bfloat16*>(dxo);
    const float ks = bits ? dropout_scale(p) : 1.f;
    const LnbPlan pl = lnb_plan(N, C);
    const size_t smem = (size_t)pl.stages * pl.stage_bytes;
    float* partial = reinterpret_cast<float*>(scratch);
    const int cpt = ceil_div(C, LNB_THREADS);
#define LNB(CPT)                                                                                         \
    do {                                                                                                 \
        if (smem_limit(reinterpret_cast<const void*>(ln_bwd_kernel<CPT>), (int)(LNB_SMEM_BUDGET)))     \
            return GPT2_ECUDA;                                                                           \
        count_launch(), ln_bwd_kernel<CPT><<<pl.grid, LNB_THREADS, smem, st>>>(                          \
            dx, dx16, partial, dy, x, w, mean, rstd, N, C, pl.rpb, pl.rb, pl.stages, accumulate ? 1 : 0, status); \
    } while (0)
    int nblk = pl.grid;
    const int v4 = ceil_div(C / 4, 32);
    if (v4 <= 6) {
        // rows of up to 768 columns: the register-streaming kernel, one block per SM
        nblk = std::min({num_sms(), LNB_MAX_BLOCKS, N});
        const int rpb = ceil_div(N, nblk);
        nblk = ceil_div(N, rpb);
        const size_t rsm = (size_t)LNR_WARPS * 3 * C * sizeof(float);
#define LNR(V4, DROP)                                                                                \
    do {                                                                                             \
        if (smem_limit(reinterpret_cast<const void*>(ln_bwd_rows_kernel<V4, DROP>),                  \
                       (int)((size_t)LNR_WARPS * 3 * 768 * sizeof(float))))                          \
            return GPT2_ECUDA;                                                                       \
        count_launch(), ln_bwd_rows_kernel<V4, DROP><<<nblk, LNR_WARPS * 32, rsm, st>>>(            \
            dx, dxo, dxo_bf16 ? 1 : 0, partial, dy, x, w, mean, rstd, N, C, rpb, accumulate ? 1 : 0,  \
            bits, ks);                                                                               \
    } while (0)
        if (bits) {
            if (v4 <= 2) LNR(2, true);
            else if (v4 <= 4) LNR(4, true);
            else LNR(6, true);
        } else {
            if (v4 <= 2) LNR(2, false);
            else if (v4 <= 4) LNR(4, false);
            else LNR(6, false);
        }
#undef LNR
    } else if (!bits && v4 <= 16) {
        // rows of up to 2048 columns: register streaming with the column sums in shared memory
        nblk = std::min({num_sms(), LNB_MAX_BLOCKS, N});
        const int rpb = ceil_div(N, nblk);
        nblk = ceil_div(N, rpb);
        const size_t wsm = (size_t)LNR_WIDE_WARPS * 3 * C * sizeof(float);
#define LNW(V4)                                                                                      \
    do {                                                                                             \
        if (smem_limit(reinterpret_cast<const void*>(ln_bwd_rows_wide_kernel<V4>),                   \
                       (int)((size_t)LNR_WIDE_WARPS * 3 * 128 * V4 * sizeof(float))))                \
            return GPT2_ECUDA;                                                                       \
        count_launch(), ln_bwd_rows_wide_kernel<V4><<<nblk, LNR_WIDE_WARPS * 32, wsm, st>>>(        \
            dx, dx16, partial, dy, x, w, mean, rstd, N, C, rpb, accumulate ? 1 : 0);                 \
    } while (0)
        if (v4 <= 8) LNW(8);
        else if (v4 <= 13) LNW(13);
        else LNW(16);
#undef LNW
    } else if (cpt <= 1) LNB(1);
    else if (cpt <= 2) LNB(2);
    else if (cpt <= 3) LNB(3);
    else if (cpt <= 4) LNB(4);
    else LNB(8);
#undef LNB
    GPT2_LAUNCH_CHECK();
    if (defer) {                                   // the caller sums the partials later
        *defer = ColReduce{partial, nblk, 3 * C, dx_colsum ? 3 * C : 2 * C, C, {dw, db, dx_colsum}};
        return GPT2_OK;
    }
    count_launch(), ln_bwd_reduce_kernel<<<ceil_div(3 * C, 32), dim3(32, 16), 0, st>>>(dw, db, dx_colsum, partial,
                                                                                       nblk, C);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k

GPT2_API int gpt2_op_layernorm_backward(float* dx, void* dx_bf16, float* dw, float* db, float* dx_colsum,
                                        const float* dy, const float* x, const float* w,
                                        const float* mean, const float* rstd, int N, int C, int accumulate,
                                        void* scratch, size_t scratch_bytes, int* status, void* stream) {
    return layernorm_backward(dx, dx_bf16, true, dw, db, dx_colsum, dy, x, w, mean, rstd, N, C, accumulate, scratch,
                              scratch_bytes, status, as_stream(stream), nullptr, 0.f);
}

GPT2_API int gpt2_op_layernorm_backward_dropout(float* dx, void* dx_drop, int dx_drop_bf16, float* dw, float* db,
                                                float* drop_colsum, const float* dy, const float* x, const float* w,
                                                const float* mean, const float* rstd, int N, int C, int accumulate,
                                                const uint32_t* bits, float p, void* scratch, size_t scratch_bytes,
                                                int* status, void* stream) {
    if (!bits || !dx_drop) return GPT2_EINVAL;
    return layernorm_backward(dx, dx_drop, dx_drop_bf16 != 0, dw, db, drop_colsum, dy, x, w, mean, rstd, N, C,
                              accumulate, scratch, scratch_bytes, status, as_stream(stream), bits, p);
}
