// attention_bwd_tc05.cu -- causal self-attention backward on the tcgen05 tensor
// cores, bf16 operands, head size 64, without dropout.
//
// With c = 1/sqrt(hs), lse the forward's row log-sum-exp and D_i = dO_i . O_i
// ("GPT-2 from scratch with torch", section 自注意力, differentiated by hand):
//   P = exp(c Q K^T - lse),  dP = dO V^T,  dS = P o (dP - D),
//   dQ = c dS K,  dK = c dS^T Q,  dV = P^T dO.
// Two persistent kernels, every output row owned by one work item (no atomics,
// deterministic), 128 x 128 score tiles:
//   attn_bwd_dkv2  items are 128-key tiles (heaviest, key tile 0, first); per
//                  128-query tile S^T = K Q^T and dP^T = V dO^T (M 128, N 128,
//                  K 64), then P^T and dS^T written to tensor memory as bf16
//                  pairs, then dV += P^T dO and dK += dS^T Q (M 128, N 64,
//                  K 128, A from tensor memory, B = the query tile's dO and Q
//                  read MN-major).
//   attn_bwd_dq2   items are 128-query tiles (longest first); first D for the
//                  tile's rows from its dO and O tiles (written out for the
//                  dK/dV kernel, which runs after it); per 128-key tile
//                  S = Q K^T and dP = dO V^T, then dS to tensor memory, then
//                  dQ += dS K (K read MN-major).
// Roles, 576 threads, one CTA per SM: warp 0 loads with TMA (the item's fixed
// operands into one of two buffers, so the next item's load overlaps this one,
// and the streamed tiles into a four-stage ring); warp 1 issues the MMAs from
// one lane as their inputs become ready (polling; the score products of the
// next tile run while the element-wise warps work on this one) and holds the
// tensor memory (512 columns); warps 2-17 do the element-wise work, one score
// row per thread (its TMEM lane), four warps per row (32 columns each), so that
// every scheduler has four of them to hide each other's latencies.
// Per 32-row group the column sums of dQ, dK and dV are kept for the qkv bias
// gradient.  Every wait is bounded; a wait that gives up raises
// GPT2_STATUS_TIMEOUT, all roles leave, copies and MMAs in flight are drained
// and tensor memory is freed.
#include "attention_tc05.cuh"
#include "gemm.cuh"

namespace gpt2k {
namespace at05 {

constexpr int B2_EW = 16;                                  // element-wise warps
constexpr int B2_THREADS = 64 + 32 * B2_EW;
constexpr int B2_STAGES = 4;
constexpr uint32_t B2_TILE = 128 * HS * 2;                 // one 128-row tile of a head: 16 KB
constexpr uint32_t B2_BOX = 64 * HS * 2;                   // one 64-row TMA box: 8 KB
constexpr uint32_t B2_FIXED = 2 * B2_TILE;                  // an item's two fixed tiles: 32 KB
constexpr uint32_t B2_OFF_STAGE = 2 * B2_FIXED;             // two item buffers, then the ring
// dK/dV stage: Q tile | dO tile | lse * log2(e) [128] | D [128]
constexpr uint32_t KV2_STAGE = 2 * B2_TILE + 1024;
constexpr size_t KV2_SMEM = B2_OFF_STAGE + (size_t)B2_STAGES * KV2_STAGE + 1024;
// dQ: the item's Q, dO and O tiles (two buffers), then stages of K tile | V tile
constexpr uint32_t Q2_FIXED = 3 * B2_TILE;
constexpr uint32_t Q2_OFF_STAGE = 2 * Q2_FIXED;
constexpr uint32_t Q2_STAGE = 2 * B2_TILE;
constexpr size_t Q2_SMEM = Q2_OFF_STAGE + (size_t)B2_STAGES * Q2_STAGE + 1024;

// Work items, heaviest first: item i is tile number (dK/dV: i / (B H); dQ:
// ntiles - 1 - i / (B H)) of (batch, head) number i % (B H).
struct BwdItem {
    int b, h, tile, n;          // n: tiles of the other operand the item visits
};
__device__ __forceinline__ BwdItem dkv_item(int i, int B, int T, int H) {
    const int nt = (T + 127) / 128;
    BwdItem w;
    w.tile = i / (B * H);
    w.b = (i % (B * H)) / H;
    w.h = i % H;
    w.n = nt - w.tile;          // query tiles tile .. nt - 1 see these keys
    return w;
}
__device__ __forceinline__ BwdItem dq_item(int i, int B, int T, int H) {
    const int nt = (T + 127) / 128;
    BwdItem w;
    w.tile = nt - 1 - i / (B * H);
    w.b = (i % (B * H)) / H;
    w.h = i % H;
    w.n = w.tile + 1;           // key tiles 0 .. tile hold keys up to the tile's last query
    return w;
}

// Two 64-row TMA boxes of a head's 128-row tile: columns col .. col + 63 of rows
// row0 .. row0 + 127 of batch b.
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, int col, int row0, int b,
                                          uint32_t bar) {
    tma_load_3d(dst, map, col, row0, b, bar);
    tma_load_3d(dst + B2_BOX, map, col, row0 + 64, b, bar);
}

// 32 values as 16 bf16 pairs into 16 TMEM columns of this warp's lanes.
__device__ __forceinline__ void tmem_st_bf16x32(uint32_t taddr, const float (&v)[32]) {
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 16; c++) pk[c] = pack_bf16(v[2 * c], v[2 * c + 1]);
    tmem_st16u(taddr, pk);
}

// Final 32 columns of an accumulator row (scaled by f) to a bf16 row of dqkv,
// with the column sums of the warp's 32 rows for the qkv bias gradient.
__device__ __forceinline__ void store_out32(float (&o)[32], float f, bool valid, __nv_bfloat16* dst, float* colsum,
                                            int lane, int b, int row0, int T, int C, int col0) {
#pragma unroll
    for (int c = 0; c < 32; c++) o[c] = valid ? o[c] * f : 0.f;
    if (valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int c = 0; c < 4; c++)
            d4[c] = make_uint4(pack_bf16(o[8 * c], o[8 * c + 1]), pack_bf16(o[8 * c + 2], o[8 * c + 3]),
                               pack_bf16(o[8 * c + 4], o[8 * c + 5]), pack_bf16(o[8 * c + 6], o[8 * c + 7]));
    }
    if (colsum) store_colsum(colsum, o, lane, b, row0, T, C, col0);
}

// ---------------------------------------------------------------- dK, dV
// Shared memory: K | V of the item (two buffers) | four stages of Q, dO, lse,
// D.  Tensor memory: S^T [0, 128) | dP^T [128, 256) | dV [256, 320) |
// dK [320, 384) | P^T [384, 448) | dS^T [448, 512) (bf16 pairs).
__global__ void __launch_bounds__(B2_THREADS, 1)
attn_bwd_dkv2(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
              __nv_bfloat16* __restrict__ dqkv, const float* __restrict__ lse, const float* __restrict__ Dg, int B,
              int T, int C, int H, float scale, int* status, float* __restrict__ colsum) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t kv_full[2], kv_empty[2], st_full[B2_STAGES], st_empty[B2_STAGES], s_full, s_free,
        p_full, pv_done, drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = B * H * ((T + 127) / 128);
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int k = 0; k < 2; k++) {
            mbar_init(smem_u32(&kv_full[k]), 1);
            mbar_init(smem_u32(&kv_empty[k]), 1);
        }
        for (int s = 0; s < B2_STAGES; s++) {
            mbar_init(smem_u32(&st_full[s]), 1);
            mbar_init(smem_u32(&st_empty[s]), 1);
        }
        mbar_init(smem_u32(&s_full), 1);
        mbar_init(smem_u32(&s_free), B2_EW);
        mbar_init(smem_u32(&p_full), B2_EW);
        mbar_init(smem_u32(&pv_done), 1);
        mbar_init(smem_u32(&drain), 1);
        fence_mbar_init();
        prefetch_map(&tq);
        prefetch_map(&tdo);
    }
    if (warp == 1) tmem_alloc(&s_tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ producer (whole warp; lane 0 issues the copies)
        int last_kc[B2_STAGES], last_ic[2];
        for (int s = 0; s < B2_STAGES; s++) last_kc[s] = -1;
        last_ic[0] = last_ic[1] = -1;
        bool ok = true;
        int kc = 0, ic = 0;
        for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
            const BwdItem w = dkv_item(it, B, T, H);
            const int kb = ic & 1;
            if (lane == 0) {
                ok = mbar_wait(smem_u32(&kv_empty[kb]), ((uint32_t)(ic >> 1) & 1u) ^ 1u, &s_abort, status);
                if (ok) {
                    const uint32_t fb = smem_u32(&kv_full[kb]);
                    mbar_expect_tx(fb, B2_FIXED);
                    last_ic[kb] = ic;
                    load_tile(base + kb * B2_FIXED, &tq, C + w.h * HS, w.tile * 128, w.b, fb);
                    load_tile(base + kb * B2_FIXED + B2_TILE, &tq, 2 * C + w.h * HS, w.tile * 128, w.b, fb);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            const float* lse_bh = lse + ((size_t)w.b * H + w.h) * T;
            const float* D_bh = Dg + ((size_t)w.b * H + w.h) * T;
            for (int t = 0; t < w.n && ok; t++, kc++) {
                const int s = kc % B2_STAGES;
                if (lane == 0)
                    ok = mbar_wait(smem_u32(&st_empty[s]), ((uint32_t)(kc / B2_STAGES) & 1u) ^ 1u, &s_abort, status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const uint32_t fb = smem_u32(&st_full[s]);
                const uint32_t st = base + B2_OFF_STAGE + s * KV2_STAGE;
                const int q0 = (w.tile + t) * 128;
                if (lane == 0) {
                    // copies first; the phase cannot complete before the arrive below
                    last_kc[s] = kc;
                    load_tile(st, &tq, w.h * HS, q0, w.b, fb);
                    load_tile(st + B2_TILE, &tdo, w.h * HS, q0, w.b, fb);
                }
                // the tile's lse * log2(e) (+inf past T, which zeroes P) and D
                float* rows = reinterpret_cast<float*>(base_ptr + B2_OFF_STAGE + s * KV2_STAGE + 2 * B2_TILE);
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int q = q0 + lane + 32 * k;
                    rows[lane + 32 * k] = q < T ? __ldg(lse_bh + q) * LOG2E : INFINITY;
                    rows[128 + lane + 32 * k] = q < T ? __ldg(D_bh + q) : 0.f;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(fb, 2 * B2_TILE);   // releases the writes above
            }
        }
        if (lane == 0 && !ok) {
            for (int k = 0; k < 2; k++)
                if (last_ic[k] >= 0) drain_wait(smem_u32(&kv_full[k]), (uint32_t)(last_ic[k] >> 1) & 1u);
            for (int s = 0; s < B2_STAGES; s++)
                if (last_kc[s] >= 0) drain_wait(smem_u32(&st_full[s]), (uint32_t)(last_kc[s] / B2_STAGES) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = instr_desc(128, 128, false, false, true);   // K Q^T, V dO^T: K-major
            const uint32_t id_o = instr_desc(128, HS, false, true, true);     // P^T dO, dS^T Q: B MN-major
            const uint64_t dfix = smem_desc(base, 16, 1024, LAYOUT_SW128);
            const uint64_t dst_k = smem_desc(base + B2_OFF_STAGE, 16, 1024, LAYOUT_SW128);
            const uint64_t dst_mn = smem_desc(base + B2_OFF_STAGE, 8192, 1024, LAYOUT_SW128);
            constexpr uint32_t FIX_U = B2_FIXED >> 4, TILE_U = B2_TILE >> 4, STAGE_U = KV2_STAGE >> 4;
            bool ok = true;
            int kc = 0, ic = 0, cs = 0;
            uint64_t t_last = globaltimer();
            for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
                const BwdItem w = dkv_item(it, B, T, H);
                const int kb = ic & 1;
                if (!mbar_wait(smem_u32(&kv_full[kb]), (uint32_t)(ic >> 1) & 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                int ns = 0, no = 0;
                for (uint32_t spin = 1; ok && no < w.n; spin++) {
                    bool progress = false;
                    if (ns < w.n) {
                        const int s = (kc + ns) % B2_STAGES, g = cs + ns;
                        if (mbar_test_wait(smem_u32(&st_full[s]), (uint32_t)((kc + ns) / B2_STAGES) & 1u) &&
                            (g == 0 || mbar_test_wait(smem_u32(&s_free), (uint32_t)(g - 1) & 1u))) {
                            tc_fence_after();
                            const uint64_t q = dst_k + (uint64_t)(s * STAGE_U);
                            mma4_ss(tmem, dfix + (uint64_t)(kb * FIX_U), q, 2, 2, id_s, 0u);   // S^T = K Q^T
                            mma4_ss(tmem + 128, dfix + (uint64_t)(kb * FIX_U + TILE_U), q + TILE_U, 2, 2, id_s,
                                    0u);                                                         // dP^T = V dO^T
                            mma_commit(smem_u32(&s_full));
                            if (++ns == w.n) mma_commit(smem_u32(&kv_empty[kb]));   // K, V read for the last time
                            progress = true;
                        }
                    }
                    if (no < ns && mbar_test_wait(smem_u32(&p_full), (uint32_t)(cs + no) & 1u)) {
                        tc_fence_after();
                        const int s = (kc + no) % B2_STAGES;
                        const uint64_t qmn = dst_mn + (uint64_t)(s * STAGE_U);
                        const uint32_t acc = no > 0 ? 1u : 0u;
                        mma4_ts(tmem + 256, tmem + 384, qmn + TILE_U, 128, id_o, acc);        // dV += P^T dO
                        mma4_ts(tmem + 256, tmem + 416, qmn + TILE_U + 512, 128, id_o, 1u);
                        mma4_ts(tmem + 320, tmem + 448, qmn, 128, id_o, acc);                 // dK += dS^T Q
                        mma4_ts(tmem + 320, tmem + 480, qmn + 512, 128, id_o, 1u);
                        mma_commit(smem_u32(&pv_done));
                        mma_commit(smem_u32(&st_empty[s]));
                        no++;
                        progress = true;
                    }
                    if (progress) {
                        t_last = globaltimer();
                    } else if ((spin & 255) == 0) {
                        if (s_abort) ok = false;
                        else if (globaltimer() - t_last > WAIT_NS) {
                            s_abort = 1;
                            set_status(status, GPT2_STATUS_TIMEOUT);
                            ok = false;
                        }
                    }
                }
                kc += w.n;
                cs += w.n;
            }
            mma_commit(smem_u32(&drain));
            drain_wait(smem_u32(&drain), 0);
        }
    } else {
        // ------------------------------------------------ element-wise (warps 2-17), thread = key
        const int quarter = warp & 3, grp = (warp - 2) >> 2;     // TMEM lane quarter, 32-column group
        const int r = quarter * 32 + lane;
        const uint32_t lb = (uint32_t)(quarter * 32) << 16;
        const float c2 = scale * LOG2E;
        const uint64_t c2x2 = f2pack(c2, c2);
        bool ok = true;
        int kc = 0, cs = 0;
        for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x) {
            const BwdItem w = dkv_item(it, B, T, H);
            const int key = w.tile * 128 + r;
            for (int t = 0; t < w.n; t++) {
                const int s = (kc + t) % B2_STAGES;
                if (!mbar_wait(smem_u32(&s_full), (uint32_t)(cs + t) & 1u, &s_abort, status)) { ok = false; break; }
                tc_fence_after();
                float sv[32], dp[32];
                tmem_ld32(tmem + lb + 32 * grp, sv);
                tmem_ld32(tmem + lb + 128 + 32 * grp, dp);
                tmem_wait_ld(sv);
                tmem_wait_ld(dp);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s_free));       // the next S^T, dP^T may be computed
                // the stage's lse and D were written before its barrier completed (acquire it)
                if (!mbar_wait(smem_u32(&st_full[s]), (uint32_t)((kc + t) / B2_STAGES) & 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                const float* rows = reinterpret_cast<const float*>(base_ptr + B2_OFF_STAGE + s * KV2_STAGE +
                                                                   2 * B2_TILE) + 32 * grp;
                const int q0 = (w.tile + t) * 128 + 32 * grp;     // first query of this warp's columns
                const bool diag = q0 < key;                        // some query of these columns precedes the key
#pragma unroll
                for (int c4 = 0; c4 < 8; c4++) {
                    const float4 lv = reinterpret_cast<const float4*>(rows)[c4];
                    const float4 dv = reinterpret_cast<const float4*>(rows + 128)[c4];
                    const int c = 4 * c4;
                    float a0 = sv[c], a1 = sv[c + 1], a2 = sv[c + 2], a3 = sv[c + 3];
                    fma2(a0, a1, c2x2, f2pack(-lv.x, -lv.y));
                    fma2(a2, a3, c2x2, f2pack(-lv.z, -lv.w));
                    float p[4] = {ex2(a0), ex2(a1), ex2(a2), ex2(a3)};
                    if (diag) {
#pragma unroll
                        for (int e = 0; e < 4; e++)
                            if (q0 + c + e < key) p[e] = 0.f;
                    }
                    const float dq[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        sv[c + e] = p[e];
                        dp[c + e] = p[e] * (dp[c + e] - dq[e]);
                    }
                }
                // P^T and dS^T columns are free once the previous tile's products completed
                if (t > 0) {
                    if (!mbar_wait(smem_u32(&pv_done), (uint32_t)(cs + t - 1) & 1u, &s_abort, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                tmem_st_bf16x32(tmem + lb + 384 + 16 * grp, sv);
                tmem_st_bf16x32(tmem + lb + 448 + 16 * grp, dp);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&p_full));
            }
            if (!ok) break;
            if (!mbar_wait(smem_u32(&pv_done), (uint32_t)(cs + w.n - 1) & 1u, &s_abort, status)) break;
            tc_fence_after();
            kc += w.n;
            cs += w.n;
            {                                              // groups 0, 1: dK (times c); 2, 3: dV
                const int which = grp >> 1, half = grp & 1;
                float o[32];
                tmem_ld32(tmem + lb + (which == 0 ? 320 : 256) + 32 * half, o);
                tmem_wait_ld(o);
                const int col0 = (1 + which) * C + w.h * HS + 32 * half;
                store_out32(o, which == 0 ? scale : 1.f, key < T, dqkv + ((size_t)w.b * T + key) * 3 * C + col0,
                            colsum, lane, w.b, w.tile * 128 + quarter * 32, T, C, col0);
            }
            // the next item's first products overwrite dK and dV: every lane has read them
            tc_fence_before();
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- dQ
// Shared memory: Q | dO | O of the item (two buffers) | four stages of K, V.
// An item buffer is free again once the MMAs have read Q and dO and every
// element-wise warp has read dO and O (for D).
// Tensor memory: S [0, 128) | dP [128, 256) | dQ [256, 320) | dS [320, 384)
// (bf16 pairs).
__global__ void __launch_bounds__(B2_THREADS, 1)
attn_bwd_dq2(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
             const __grid_constant__ CUtensorMap to, __nv_bfloat16* __restrict__ dqkv, const float* __restrict__ lse,
             float* __restrict__ Dg, int B, int T, int C, int H, float scale, int* status,
             float* __restrict__ colsum) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full[2], q_empty[2], st_full[B2_STAGES], st_empty[B2_STAGES], s_full, s_free,
        p_full, pv_done, drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = B * H * ((T + 127) / 128);
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int k = 0; k < 2; k++) {
            mbar_init(smem_u32(&q_full[k]), 1);
            mbar_init(smem_u32(&q_empty[k]), 1 + B2_EW);      // the MMA thread and the element-wise warps
        }
        for (int s = 0; s < B2_STAGES; s++) {
            mbar_init(smem_u32(&st_full[s]), 1);
            mbar_init(smem_u32(&st_empty[s]), 1);
        }
        mbar_init(smem_u32(&s_full), 1);
        mbar_init(smem_u32(&s_free), B2_EW);
        mbar_init(smem_u32(&p_full), B2_EW);
        mbar_init(smem_u32(&pv_done), 1);
        mbar_init(smem_u32(&drain), 1);
        fence_mbar_init();
        prefetch_map(&tq);
        prefetch_map(&tdo);
        prefetch_map(&to);
    }
    if (warp == 1) tmem_alloc(&s_tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_kc[B2_STAGES], last_ic[2];
            for (int s = 0; s < B2_STAGES; s++) last_kc[s] = -1;
            last_ic[0] = last_ic[1] = -1;
            bool ok = true;
            int kc = 0, ic = 0;
            for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
                const BwdItem w = dq_item(it, B, T, H);
                const int qb = ic & 1;
                if (!mbar_wait(smem_u32(&q_empty[qb]), ((uint32_t)(ic >> 1) & 1u) ^ 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&q_full[qb]);
                mbar_expect_tx(fb, Q2_FIXED);
                last_ic[qb] = ic;
                load_tile(base + qb * Q2_FIXED, &tq, w.h * HS, w.tile * 128, w.b, fb);
                load_tile(base + qb * Q2_FIXED + B2_TILE, &tdo, w.h * HS, w.tile * 128, w.b, fb);
                load_tile(base + qb * Q2_FIXED + 2 * B2_TILE, &to, w.h * HS, w.tile * 128, w.b, fb);
                for (int j = 0; j < w.n; j++, kc++) {
                    const int s = kc % B2_STAGES;
                    if (!mbar_wait(smem_u32(&st_empty[s]), ((uint32_t)(kc / B2_STAGES) & 1u) ^ 1u, &s_abort,
                                   status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sb = smem_u32(&st_full[s]);
                    mbar_expect_tx(sb, 2 * B2_TILE);
                    last_kc[s] = kc;
                    const uint32_t st = base + Q2_OFF_STAGE + s * Q2_STAGE;
                    load_tile(st, &tq, C + w.h * HS, j * 128, w.b, sb);
                    load_tile(st + B2_TILE, &tq, 2 * C + w.h * HS, j * 128, w.b, sb);
                }
            }
            if (!ok) {
                for (int k = 0; k < 2; k++)
                    if (last_ic[k] >= 0) drain_wait(smem_u32(&q_full[k]), (uint32_t)(last_ic[k] >> 1) & 1u);
                for (int s = 0; s < B2_STAGES; s++)
                    if (last_kc[s] >= 0) drain_wait(smem_u32(&st_full[s]), (uint32_t)(last_kc[s] / B2_STAGES) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = instr_desc(128, 128, false, false, true);   // Q K^T, dO V^T: K-major
            const uint32_t id_o = instr_desc(128, HS, false, true, true);     // dS K: B MN-major
            const uint64_t dfix = smem_desc(base, 16, 1024, LAYOUT_SW128);
            const uint64_t dst_k = smem_desc(base + Q2_OFF_STAGE, 16, 1024, LAYOUT_SW128);
            const uint64_t dst_mn = smem_desc(base + Q2_OFF_STAGE, 8192, 1024, LAYOUT_SW128);
            constexpr uint32_t FIX_U = Q2_FIXED >> 4, TILE_U = B2_TILE >> 4, STAGE_U = Q2_STAGE >> 4;
            bool ok = true;
            int kc = 0, ic = 0, cs = 0;
            uint64_t t_last = globaltimer();
            for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
                const BwdItem w = dq_item(it, B, T, H);
                const int qb = ic & 1;
                if (!mbar_wait(smem_u32(&q_full[qb]), (uint32_t)(ic >> 1) & 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                int ns = 0, no = 0;
                for (uint32_t spin = 1; ok && no < w.n; spin++) {
                    bool progress = false;
                    if (ns < w.n) {
                        const int s = (kc + ns) % B2_STAGES, g = cs + ns;
                        if (mbar_test_wait(smem_u32(&st_full[s]), (uint32_t)((kc + ns) / B2_STAGES) & 1u) &&
                            (g == 0 || mbar_test_wait(smem_u32(&s_free), (uint32_t)(g - 1) & 1u))) {
                            tc_fence_after();
                            const uint64_t kv = dst_k + (uint64_t)(s * STAGE_U);
                            mma4_ss(tmem, dfix + (uint64_t)(qb * FIX_U), kv, 2, 2, id_s, 0u);           // S = Q K^T
                            mma4_ss(tmem + 128, dfix + (uint64_t)(qb * FIX_U + TILE_U), kv + TILE_U, 2, 2, id_s,
                                    0u);                                                                   // dP = dO V^T
                            mma_commit(smem_u32(&s_full));
                            if (++ns == w.n) mma_commit(smem_u32(&q_empty[qb]));   // Q, dO read for the last time
                            progress = true;
                        }
                    }
                    if (no < ns && mbar_test_wait(smem_u32(&p_full), (uint32_t)(cs + no) & 1u)) {
                        tc_fence_after();
                        const int s = (kc + no) % B2_STAGES;
                        const uint64_t kmn = dst_mn + (uint64_t)(s * STAGE_U);
                        const uint32_t acc = no > 0 ? 1u : 0u;
                        mma4_ts(tmem + 256, tmem + 320, kmn, 128, id_o, acc);                  // dQ += dS K
                        mma4_ts(tmem + 256, tmem + 352, kmn + 512, 128, id_o, 1u);
                        mma_commit(smem_u32(&pv_done));
                        mma_commit(smem_u32(&st_empty[s]));
                        no++;
                        progress = true;
                    }
                    if (progress) {
                        t_last = globaltimer();
                    } else if ((spin & 255) == 0) {
                        if (s_abort) ok = false;
                        else if (globaltimer() - t_last > WAIT_NS) {
                            s_abort = 1;
                            set_status(status, GPT2_STATUS_TIMEOUT);
                            ok = false;
                        }
                    }
                }
                kc += w.n;
                cs += w.n;
            }
            mma_commit(smem_u32(&drain));
            drain_wait(smem_u32(&drain), 0);
        }
    } else {
        // ------------------------------------------------ element-wise (warps 2-17), thread = query
        const int quarter = warp & 3, grp = (warp - 2) >> 2;     // TMEM lane quarter, 32-column group
        const int r = quarter * 32 + lane;
        const uint32_t lb = (uint32_t)(quarter * 32) << 16;
        const float c2 = scale * LOG2E;
        const uint64_t c2x2 = f2pack(c2, c2);
        bool ok = true;
        int cs = 0, ic = 0;
        const uint8_t* const base_ptr = smem_raw + (base - raw);
        for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
            const BwdItem w = dq_item(it, B, T, H);
            const int row = w.tile * 128 + r;
            const size_t bh = ((size_t)w.b * H + w.h) * T;
            const float lse2 = row < T ? __ldg(lse + bh + row) * LOG2E : INFINITY;   // +inf zeroes P past T
            // D = dO . O over the row's 64 head columns, from the item's tiles (every
            // warp of the row computes it; the first writes it out for dK/dV)
            const int qb = ic & 1;
            if (!mbar_wait(smem_u32(&q_full[qb]), (uint32_t)(ic >> 1) & 1u, &s_abort, status)) { ok = false; break; }
            float Drow = 0.f;
            {
                const uint8_t* tdo_s = base_ptr + qb * Q2_FIXED + B2_TILE + (r >> 6) * B2_BOX + (r & 63) * 128;
                const uint8_t* to_s = tdo_s + B2_TILE;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    const uint32_t off = (uint32_t)((c ^ (r & 7)) << 4);
                    const uint4 a = *reinterpret_cast<const uint4*>(tdo_s + off);
                    const uint4 o = *reinterpret_cast<const uint4*>(to_s + off);
                    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
                        const float2 fo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
                        Drow = fmaf(fa.x, fo.x, Drow);
                        Drow = fmaf(fa.y, fo.y, Drow);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&q_empty[qb]));     // this warp is done with dO and O
            if (row >= T) Drow = 0.f;
            else if (grp == 0) Dg[bh + row] = Drow;
            const uint64_t nl2 = f2pack(-lse2, -lse2), nd2 = f2pack(-Drow, -Drow);
            for (int j = 0; j < w.n; j++) {
                if (!mbar_wait(smem_u32(&s_full), (uint32_t)(cs + j) & 1u, &s_abort, status)) { ok = false; break; }
                tc_fence_after();
                float sv[32], dp[32];
                tmem_ld32(tmem + lb + 32 * grp, sv);
                tmem_ld32(tmem + lb + 128 + 32 * grp, dp);
                tmem_wait_ld(sv);
                tmem_wait_ld(dp);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s_free));       // the next S, dP may be computed
                const int k0 = j * 128 + 32 * grp;                    // first key of this warp's columns
                const bool edge = k0 + 31 > row || k0 + 32 > T;      // the diagonal, the sequence end
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    fma2(sv[c], sv[c + 1], c2x2, nl2);
                    float p0 = ex2(sv[c]), p1 = ex2(sv[c + 1]);
                    if (edge) {
                        if (k0 + c > row || k0 + c >= T) p0 = 0.f;
                        if (k0 + c + 1 > row || k0 + c + 1 >= T) p1 = 0.f;
                    }
                    float d0 = dp[c], d1 = dp[c + 1];
                    uint64_t t2;
                    asm("add.f32x2 %0, %1, %2;" : "=l"(t2) : "l"(f2pack(d0, d1)), "l"(nd2));
                    f2unpack(t2, d0, d1);
                    dp[c] = p0 * d0;
                    dp[c + 1] = p1 * d1;
                }
                // the dS columns are free once the previous tile's product completed
                if (j > 0) {
                    if (!mbar_wait(smem_u32(&pv_done), (uint32_t)(cs + j - 1) & 1u, &s_abort, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                tmem_st_bf16x32(tmem + lb + 320 + 16 * grp, dp);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&p_full));
            }
            if (!ok) break;
            if (!mbar_wait(smem_u32(&pv_done), (uint32_t)(cs + w.n - 1) & 1u, &s_abort, status)) break;
            tc_fence_after();
            cs += w.n;
            if (grp < 2) {                                 // dQ: 64 columns, two groups of 32
                float o[32];
                tmem_ld32(tmem + lb + 256 + 32 * grp, o);
                tmem_wait_ld(o);
                const int col0 = w.h * HS + 32 * grp;
                store_out32(o, scale, row < T, dqkv + ((size_t)w.b * T + row) * 3 * C + col0, colsum, lane, w.b,
                            w.tile * 128 + quarter * 32, T, C, col0);
            }
            // the next item's first product overwrites dQ: every lane has read it
            tc_fence_before();
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace at05

// dqkv [B,T,3C] (bf16, every element written) from dy [B,T,C], qkv, the
// forward's output y [B,T,C] and lse [B,H,T]; D [B,H,T] = rowsum(dO o O) is
// computed on the way (scratch, written by the dQ kernel, read by the dK/dV
// kernel); head size 64, no dropout.  With colsum != null also the column sums of dqkv per 32-row group
// ([B * ceil(T/32), 3C], fp32, before bf16 rounding).
int attention_tc05_backward_nodrop(void* dqkv, const void* dy, const void* qkv, const void* y, const float* lse,
                                   float* D, int B, int T, int C, int H, int* status, cudaStream_t st,
                                   float* colsum) {
    using namespace at05;
    if (C / H != HS || C % H || C % 8) return GPT2_ENOTSUP;
    if (smem_limit(reinterpret_cast<const void*>(attn_bwd_dkv2), (int)KV2_SMEM) ||
        smem_limit(reinterpret_cast<const void*>(attn_bwd_dq2), (int)Q2_SMEM))
        return GPT2_ECUDA;
    CUtensorMap tq, tdo, to;
    const cuuint64_t dq_[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t sq_[2] = {(cuuint64_t)3 * C * 2, (cuuint64_t)T * 3 * C * 2};
    const cuuint64_t dd_[3] = {(cuuint64_t)C, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t sd_[2] = {(cuuint64_t)C * 2, (cuuint64_t)T * C * 2};
    const cuuint32_t box[3] = {HS, 64, 1};
    if (!encode_tensor_map(&tq, true, 3, qkv, dq_, sq_, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&tdo, true, 3, dy, dd_, sd_, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&to, true, 3, y, dd_, sd_, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return GPT2_ENOTSUP;
    const float scale = 1.f / sqrtf((float)HS);
    auto* out = static_cast<__nv_bfloat16*>(dqkv);
    const int nitems = B * H * ((T + 127) / 128);
    const int grid = std::min(nitems, num_sms());
    count_launch(), attn_bwd_dq2<<<grid, B2_THREADS, Q2_SMEM, st>>>(tq, tdo, to, out, lse, D, B, T, C, H, scale,
                                                                    status, colsum);
    count_launch(), attn_bwd_dkv2<<<grid, B2_THREADS, KV2_SMEM, st>>>(tq, tdo, out, lse, D, B, T, C, H, scale, status,
                                                                      colsum);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k
