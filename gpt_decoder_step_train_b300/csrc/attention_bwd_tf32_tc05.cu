// attention_bwd_tf32_tc05.cu -- causal self-attention backward on the tcgen05
// tensor cores with tf32 operands (fp32 tensors read as they are stored), head
// size 64, without dropout: the backward of the tf32 tensor-core mode.
//
// With c = 1/sqrt(hs), lse the forward's row log-sum-exp and D_i = dO_i . O_i
// ("GPT-2 from scratch with torch", section 自注意力, differentiated by hand):
//   P = exp(c Q K^T - lse),  dP = dO V^T,  dS = P o (dP - D),
//   dQ = c dS K,  dK = c dS^T Q,  dV = P^T dO.
// Two persistent kernels with the roles of the bf16 ones (attention_bwd_tc05.cu),
// every output row owned by one work item (no atomics, deterministic):
//   attn_bwd_dkv_tf32  items are 128-key tiles (K, V fixed); per 64-query
//       tile S^T = K Q^T and dP^T = V dO^T (M 128, N 64), P^T and dS^T written
//       over them in tensor memory (fp32, read as tf32), then dV += P^T dO and
//       dK += dS^T Q (M 128, N 64, K 64, A from tensor memory);
//   attn_bwd_dq_tf32   items are 128-query tiles (Q, dO fixed); per 64-key
//       tile S = Q K^T and dP = dO V^T, dS written over dP, then dQ += dS K.
// What 32-bit operands change against the bf16 kernels: a tile that is read
// both K-major (a B operand of the score products) and MN-major (the B operand
// of the dV / dK / dQ products) needs two copies, since tf32 MN-major operands
// take the 128-byte swizzle of 32-byte chunks and K-major ones that of 16-byte
// chunks; the streamed tiles are therefore 64 rows (16 KB per copy), which also
// leaves tensor memory for two score buffers, so the score products of the
// next tile run while the element-wise warps work on this one.  A score buffer
// is reused once the products that read its P^T / dS^T (dS) have completed.
// D = rowsum(dO o O) comes from a separate pass before these kernels.
// Roles, 576 threads, one CTA per SM: warp 0 loads with TMA, one lane of warp 1
// issues the MMAs (polling) and warp 1 holds the tensor memory (512 columns),
// warps 2-17 do the element-wise work, one score row per thread (its TMEM
// lane), four warps per row (16 of the tile's 64 columns each).
// Every wait is bounded; a wait that gives up raises GPT2_STATUS_TIMEOUT, all
// roles leave, copies and MMAs in flight are drained and tensor memory is freed.
#include "attention_tc05.cuh"
#include "gemm.cuh"

namespace gpt2k {
namespace at05 {

constexpr int T3_EW = 16;                                  // element-wise warps
constexpr int T3_THREADS = 64 + 32 * T3_EW;
constexpr int T3_BS = 64;                                  // rows of a streamed tile
constexpr uint32_t T3_BOX = 64 * 32 * 4;                   // one TMA box: 64 rows x 32 fp32 = 8 KB
constexpr uint32_t T3_HALF = 2 * T3_BOX;                   // 32 columns of a 128-row tile: 16 KB
constexpr uint32_t T3_TILE = 2 * T3_HALF;                  // a 128-row fixed tile: 32 KB
constexpr uint32_t T3_STILE = 2 * T3_BOX;                  // a 64-row streamed tile (one copy): 16 KB
constexpr uint32_t T3_FIXED = 2 * T3_TILE;                 // an item's two fixed tiles: 64 KB
// dK/dV: the fixed K, V | three slots of Q, dO K-major | two slots of Q, dO MN-major
constexpr int KV3_KS = 3, KV3_MS = 2;
constexpr uint32_t KV3_KSLOT = 2 * T3_STILE, KV3_MSLOT = 2 * T3_STILE;
constexpr uint32_t KV3_OFF_K = T3_FIXED, KV3_OFF_M = KV3_OFF_K + KV3_KS * KV3_KSLOT;
constexpr size_t KV3_SMEM = KV3_OFF_M + (size_t)KV3_MS * KV3_MSLOT + 1024;
// dQ stage: K, V (K-major) | K (MN-major)
constexpr uint32_t Q3_STAGE = 3 * T3_STILE;
constexpr int Q3_STAGES = 3;
constexpr size_t Q3_SMEM = T3_FIXED + (size_t)Q3_STAGES * Q3_STAGE + 1024;

// Work items, heaviest first: item i is 128-row tile number (dK/dV: i / (B H);
// dQ: ntiles - 1 - i / (B H)) of (batch, head) number i % (B H); n is the
// number of 64-row tiles of the other operand that the item visits.
struct Bwd3Item {
    int b, h, tile, n;
};
__device__ __forceinline__ Bwd3Item dkv3_item(int i, int B, int T, int H) {
    const int n64 = (T + 63) / 64;
    Bwd3Item w;
    w.tile = i / (B * H);
    w.b = (i % (B * H)) / H;
    w.h = i % H;
    w.n = n64 - 2 * w.tile;     // query tiles 2 tile .. n64 - 1 see these keys
    return w;
}
__device__ __forceinline__ Bwd3Item dq3_item(int i, int B, int T, int H) {
    const int n128 = (T + 127) / 128, n64 = (T + 63) / 64;
    Bwd3Item w;
    w.tile = n128 - 1 - i / (B * H);
    w.b = (i % (B * H)) / H;
    w.h = i % H;
    w.n = min(2 * w.tile + 2, n64);   // key tiles holding keys up to the tile's last query
    return w;
}

// A 128-row fixed tile (K-major, 128-byte swizzle): columns col .. col + 63 of
// rows row0 .. row0 + 127 of batch b as four boxes (two row halves per 32
// columns).
__device__ __forceinline__ void load_fixed(uint32_t dst, const CUtensorMap* map, int col, int row0, int b,
                                           uint32_t bar) {
#pragma unroll
    for (int hf = 0; hf < 2; hf++) {
        tma_load_3d(dst + hf * T3_HALF, map, col + 32 * hf, row0, b, bar);
        tma_load_3d(dst + hf * T3_HALF + T3_BOX, map, col + 32 * hf, row0 + 64, b, bar);
    }
}
// A 64-row streamed tile: two boxes of 32 columns (K-major or MN-major by the map).
__device__ __forceinline__ void load_stile(uint32_t dst, const CUtensorMap* map, int col, int row0, int b,
                                           uint32_t bar) {
    tma_load_3d(dst, map, col, row0, b, bar);
    tma_load_3d(dst + T3_BOX, map, col + 32, row0, b, bar);
}

// Score products of one tile: two groups of 4 tf32 MMAs (K = 64), the second
// on the second 32-column half of both operands.
__device__ __forceinline__ void score8(uint32_t d, uint64_t a, uint32_t a_half_u, uint64_t b, uint32_t b_half_u,
                                       uint32_t idesc) {
    mma4_ss_tf32(d, a, b, 2, 2, idesc, 0u);
    mma4_ss_tf32(d, a + a_half_u, b + b_half_u, 2, 2, idesc, 1u);
}
// d += A (64 columns of tensor memory at a) times a 64-row MN-major tile at b:
// 8 MMAs, K = 8 rows each (1 KB of the tile).
__device__ __forceinline__ void acc8(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    mma4_ts_tf32(d, a, b, 64, idesc, accumulate);
    mma4_ts_tf32(d, a + 32, b + 4 * 64, 64, idesc, 1u);
}

// 32 columns of an accumulator row, scaled by f, to an fp32 row of dqkv.
__device__ __forceinline__ void store_row32(const float (&o)[32], float f, float* dst) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int c = 0; c < 8; c++) d4[c] = make_float4(o[4 * c] * f, o[4 * c + 1] * f, o[4 * c + 2] * f, o[4 * c + 3] * f);
}

__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float (&v)[16]) {
    uint32_t u[16];
#pragma unroll
    for (int c = 0; c < 16; c++) u[c] = __float_as_uint(v[c]);
    tmem_st16u(taddr, u);
}

// ---------------------------------------------------------------- dK, dV
// Shared memory: K | V of the item | a ring of three K-major Q, dO tile pairs
// (released once the score products have read them) | a ring of two MN-major
// Q, dO tile pairs (released once dV, dK have read them), with each MN slot a
// small static slot holding the tile's lse * log2(e) and D (the element-wise
// warps read them; the slot is reused only after the products of its tile,
// which follow the warps' P^T / dS^T).  Tensor memory: score buffer u in
// [128 u, 128 u + 128): S^T then P^T in its first 64 columns, dP^T then dS^T
// in the next 64 | dV [256, 320) | dK [320, 384).
__global__ void __launch_bounds__(T3_THREADS, 1)
attn_bwd_dkv_tf32(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tqm,
                  const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tdom,
                  float* __restrict__ dqkv, const float* __restrict__ lse, const float* __restrict__ Dg, int B, int T,
                  int C, int H, float scale, int* status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t kv_full, kv_empty, kf_full[KV3_KS], kf_empty[KV3_KS], mn_full[KV3_MS],
        mn_empty[KV3_MS], rows_full[KV3_MS], s_full[2], p_full[2], pv_done[2], drain;
    __shared__ __align__(16) float s_rows[KV3_MS][2 * T3_BS];   // per MN slot: lse * log2(e) [64], D [64]
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = B * H * ((T + 127) / 128);
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;

    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&kv_full), 1);
        mbar_init(smem_u32(&kv_empty), 1);
        for (int s = 0; s < KV3_KS; s++) {
            mbar_init(smem_u32(&kf_full[s]), 1);
            mbar_init(smem_u32(&kf_empty[s]), 1);
        }
        for (int s = 0; s < KV3_MS; s++) {
            mbar_init(smem_u32(&mn_full[s]), 1);
            mbar_init(smem_u32(&mn_empty[s]), 1);
            mbar_init(smem_u32(&rows_full[s]), 1);
        }
        for (int u = 0; u < 2; u++) {
            mbar_init(smem_u32(&s_full[u]), 1);
            mbar_init(smem_u32(&p_full[u]), T3_EW);
            mbar_init(smem_u32(&pv_done[u]), 1);
        }
        mbar_init(smem_u32(&drain), 1);
        fence_mbar_init();
        prefetch_map(&tq);
        prefetch_map(&tqm);
        prefetch_map(&tdo);
        prefetch_map(&tdom);
    }
    if (warp == 1) tmem_alloc(&s_tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ producer (whole warp; lane 0 issues the copies)
        // order per item: fixed K, V; K-major tile 0; then MN-major tile t after
        // K-major tile t + 1, so the K-major copies run a tile ahead
        int last_k[KV3_KS], last_m[KV3_MS], last_ic = -1;
        for (int s = 0; s < KV3_KS; s++) last_k[s] = -1;
        for (int s = 0; s < KV3_MS; s++) last_m[s] = -1;
        bool ok = true;
        int kc = 0, ic = 0;                            // tiles and items loaded so far
        auto k_load = [&](const Bwd3Item& w, int t, int g) -> bool {   // K-major tile t (global index g)
            const int s = g % KV3_KS;
            bool r = true;
            if (lane == 0) {
                r = mbar_wait(smem_u32(&kf_empty[s]), ((uint32_t)(g / KV3_KS) & 1u) ^ 1u, &s_abort, status);
                if (r) {
                    const uint32_t fb = smem_u32(&kf_full[s]);
                    const uint32_t dst = base + KV3_OFF_K + s * KV3_KSLOT;
                    const int q0 = (2 * w.tile + t) * T3_BS;
                    mbar_expect_tx(fb, KV3_KSLOT);
                    last_k[s] = g;
                    load_stile(dst, &tq, w.h * HS, q0, w.b, fb);
                    load_stile(dst + T3_STILE, &tdo, w.h * HS, q0, w.b, fb);
                }
            }
            return __shfl_sync(0xffffffffu, r, 0);
        };
        auto m_load = [&](const Bwd3Item& w, int t, int g) -> bool {   // MN-major tile t, with its lse and D
            const int s = g % KV3_MS;
            const int q0 = (2 * w.tile + t) * T3_BS;
            // the tile's lse * log2(e) (+inf past T, which zeroes P) and D, loaded before the wait
            const float* lse_bh = lse + ((size_t)w.b * H + w.h) * T;
            const float* D_bh = Dg + ((size_t)w.b * H + w.h) * T;
            float lv[2], dv[2];
#pragma unroll
            for (int k = 0; k < 2; k++) {
                const int q = q0 + lane + 32 * k;
                lv[k] = q < T ? __ldg(lse_bh + q) * LOG2E : INFINITY;
                dv[k] = q < T ? __ldg(D_bh + q) : 0.f;
            }
            bool r = true;
            if (lane == 0) {
                r = mbar_wait(smem_u32(&mn_empty[s]), ((uint32_t)(g / KV3_MS) & 1u) ^ 1u, &s_abort, status);
                if (r) {
                    const uint32_t fb = smem_u32(&mn_full[s]);
                    const uint32_t dst = base + KV3_OFF_M + s * KV3_MSLOT;
                    mbar_expect_tx(fb, KV3_MSLOT);
                    last_m[s] = g;
                    load_stile(dst, &tqm, w.h * HS, q0, w.b, fb);
                    load_stile(dst + T3_STILE, &tdom, w.h * HS, q0, w.b, fb);
                }
            }
            r = __shfl_sync(0xffffffffu, r, 0);
            if (!r) return false;
#pragma unroll
            for (int k = 0; k < 2; k++) {
                s_rows[s][lane + 32 * k] = lv[k];
                s_rows[s][T3_BS + lane + 32 * k] = dv[k];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&rows_full[s]));   // releases the writes above
            return true;
        };
        for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
            const Bwd3Item w = dkv3_item(it, B, T, H);
            if (lane == 0) {
                ok = mbar_wait(smem_u32(&kv_empty), ((uint32_t)ic & 1u) ^ 1u, &s_abort, status);
                if (ok) {
                    const uint32_t fb = smem_u32(&kv_full);
                    mbar_expect_tx(fb, T3_FIXED);
                    last_ic = ic;
                    load_fixed(base, &tq, C + w.h * HS, w.tile * 128, w.b, fb);
                    load_fixed(base + T3_TILE, &tq, 2 * C + w.h * HS, w.tile * 128, w.b, fb);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok) ok = k_load(w, 0, kc);
            for (int t = 0; t < w.n && ok; t++) {
                if (t + 1 < w.n) ok = k_load(w, t + 1, kc + t + 1);
                if (ok) ok = m_load(w, t, kc + t);
            }
            kc += w.n;
        }
        if (lane == 0 && !ok) {
            if (last_ic >= 0) drain_wait(smem_u32(&kv_full), (uint32_t)last_ic & 1u);
            for (int s = 0; s < KV3_KS; s++)
                if (last_k[s] >= 0) drain_wait(smem_u32(&kf_full[s]), (uint32_t)(last_k[s] / KV3_KS) & 1u);
            for (int s = 0; s < KV3_MS; s++)
                if (last_m[s] >= 0) drain_wait(smem_u32(&mn_full[s]), (uint32_t)(last_m[s] / KV3_MS) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = instr_desc(128, T3_BS, false, false, false);   // K Q^T, V dO^T: K-major
            const uint32_t id_o = instr_desc(128, HS, false, true, false);       // P^T dO, dS^T Q: B MN-major
            const uint64_t dfix = smem_desc(base, 16, 1024, LAYOUT_SW128);
            const uint64_t dk = smem_desc(base + KV3_OFF_K, 16, 1024, LAYOUT_SW128);
            const uint64_t dm = smem_desc(base + KV3_OFF_M, T3_BOX, 512, LAYOUT_SW128_32B);
            constexpr uint32_t HALF_U = T3_HALF >> 4, BOX_U = T3_BOX >> 4, TILE_U = T3_TILE >> 4,
                               STILE_U = T3_STILE >> 4, KSLOT_U = KV3_KSLOT >> 4, MSLOT_U = KV3_MSLOT >> 4;
            bool ok = true;
            int kc = 0;                                // tiles of earlier items (also the score-buffer count)
            uint64_t t_last = globaltimer();
            for (int it = blockIdx.x, ic = 0; it < nitems && ok; it += gridDim.x, ic++) {
                const Bwd3Item w = dkv3_item(it, B, T, H);
                if (!mbar_wait(smem_u32(&kv_full), (uint32_t)ic & 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                int ns = 0, no = 0;
                for (uint32_t spin = 1; ok && no < w.n; spin++) {
                    bool progress = false;
                    if (ns < w.n) {
                        // tile g goes to score buffer g & 1, free once the products of tile g - 2 completed
                        const int g = kc + ns, s = g % KV3_KS, u = g & 1;
                        if (mbar_test_wait(smem_u32(&kf_full[s]), (uint32_t)(g / KV3_KS) & 1u) &&
                            (g < 2 || mbar_test_wait(smem_u32(&pv_done[u]), (uint32_t)((g - 2) >> 1) & 1u))) {
                            tc_fence_after();
                            const uint64_t q = dk + (uint64_t)(s * KSLOT_U);
                            score8(tmem + 128 * u, dfix, HALF_U, q, BOX_U, id_s);                   // S^T = K Q^T
                            score8(tmem + 128 * u + 64, dfix + TILE_U, HALF_U, q + STILE_U, BOX_U, id_s);   // dP^T
                            mma_commit(smem_u32(&s_full[u]));
                            mma_commit(smem_u32(&kf_empty[s]));
                            if (++ns == w.n) mma_commit(smem_u32(&kv_empty));   // K, V read for the last time
                            progress = true;
                        }
                    }
                    if (no < ns) {
                        const int g = kc + no, s = g % KV3_MS, u = g & 1;
                        if (mbar_test_wait(smem_u32(&p_full[u]), (uint32_t)(g >> 1) & 1u) &&
                            mbar_test_wait(smem_u32(&mn_full[s]), (uint32_t)(g / KV3_MS) & 1u)) {
                            tc_fence_after();
                            const uint64_t qmn = dm + (uint64_t)(s * MSLOT_U);
                            const uint32_t acc = no > 0 ? 1u : 0u;
                            acc8(tmem + 256, tmem + 128 * u, qmn + STILE_U, id_o, acc);       // dV += P^T dO
                            acc8(tmem + 320, tmem + 128 * u + 64, qmn, id_o, acc);            // dK += dS^T Q
                            mma_commit(smem_u32(&pv_done[u]));
                            mma_commit(smem_u32(&mn_empty[s]));
                            no++;
                            progress = true;
                        }
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
            }
            mma_commit(smem_u32(&drain));
            drain_wait(smem_u32(&drain), 0);
        }
    } else {
        // ------------------------------------------------ element-wise (warps 2-17), thread = key
        const int quarter = warp & 3, grp = (warp - 2) >> 2;     // TMEM lane quarter, 16-column group
        const int r = quarter * 32 + lane;
        const uint32_t lb = (uint32_t)(quarter * 32) << 16;
        const float c2 = scale * LOG2E;
        const uint64_t c2x2 = f2pack(c2, c2);
        bool ok = true;
        int kc = 0;
        for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x) {
            const Bwd3Item w = dkv3_item(it, B, T, H);
            const int key = w.tile * 128 + r;
            for (int t = 0; t < w.n; t++) {
                const int g = kc + t, s = g % KV3_MS, u = g & 1;
                if (!mbar_wait(smem_u32(&s_full[u]), (uint32_t)(g >> 1) & 1u, &s_abort, status)) { ok = false; break; }
                tc_fence_after();
                uint32_t su[16], du[16];
                const uint32_t ts = tmem + lb + 128 * u + 16 * grp;
                tmem_ld16_async(ts, su);
                tmem_ld16_async(ts + 64, du);
                // the tile's lse and D (written by the producer before rows_full; acquire them)
                if (!mbar_wait(smem_u32(&rows_full[s]), (uint32_t)(g / KV3_MS) & 1u, &s_abort, status)) {
                    tmem_wait16(su);
                    tmem_wait16(du);
                    ok = false;
                    break;
                }
                tmem_wait16(su);
                tmem_wait16(du);
                const float* rows = &s_rows[s][16 * grp];
                const int q0 = (2 * w.tile + t) * T3_BS + 16 * grp;   // first query of this warp's columns
                const bool diag = q0 < key;                            // some query of these columns precedes the key
                float pv[16], dv[16];
#pragma unroll
                for (int c4 = 0; c4 < 4; c4++) {
                    const float4 lv = reinterpret_cast<const float4*>(rows)[c4];
                    const float4 dd = reinterpret_cast<const float4*>(rows + T3_BS)[c4];
                    const int c = 4 * c4;
                    float a0 = __uint_as_float(su[c]), a1 = __uint_as_float(su[c + 1]);
                    float a2 = __uint_as_float(su[c + 2]), a3 = __uint_as_float(su[c + 3]);
                    fma2(a0, a1, c2x2, f2pack(-lv.x, -lv.y));
                    fma2(a2, a3, c2x2, f2pack(-lv.z, -lv.w));
                    float p[4] = {ex2(a0), ex2(a1), ex2(a2), ex2(a3)};
                    if (diag) {
#pragma unroll
                        for (int e = 0; e < 4; e++)
                            if (q0 + c + e < key) p[e] = 0.f;
                    }
                    const float dq[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        pv[c + e] = p[e];
                        dv[c + e] = p[e] * (__uint_as_float(du[c + e]) - dq[e]);
                    }
                }
                // P^T over S^T, dS^T over dP^T (these warps own the buffer until p_full)
                tmem_st16f(ts, pv);
                tmem_st16f(ts + 64, dv);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&p_full[u]));
            }
            if (!ok) break;
            {
                const int g = kc + w.n - 1;
                if (!mbar_wait(smem_u32(&pv_done[g & 1]), (uint32_t)(g >> 1) & 1u, &s_abort, status)) break;
            }
            tc_fence_after();
            kc += w.n;
            {                                              // groups 0, 1: dK (times c); 2, 3: dV
                const int which = grp >> 1, half = grp & 1;
                float o[32];
                tmem_ld32(tmem + lb + (which == 0 ? 320 : 256) + 32 * half, o);
                tmem_wait_ld(o);
                if (key < T)
                    store_row32(o, which == 0 ? scale : 1.f,
                                dqkv + ((size_t)w.b * T + key) * 3 * C + (1 + which) * C + w.h * HS + 32 * half);
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
// Shared memory: Q | dO of the item | three stages of K, V (K-major), K
// (MN-major).  Tensor memory: score buffer u in [128 u, 128 u + 128): S in its
// first 64 columns, dP then dS in the next 64 | dQ [256, 320).
__global__ void __launch_bounds__(T3_THREADS, 1)
attn_bwd_dq_tf32(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tqm,
                 const __grid_constant__ CUtensorMap tdo, float* __restrict__ dqkv, const float* __restrict__ lse,
                 const float* __restrict__ Dg, int B, int T, int C, int H, float scale, int* status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full, q_empty, st_full[Q3_STAGES], st_empty[Q3_STAGES], s_full[2], p_full[2],
        pv_done[2], drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = B * H * ((T + 127) / 128);
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;

    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&q_full), 1);
        mbar_init(smem_u32(&q_empty), 1);
        for (int s = 0; s < Q3_STAGES; s++) {
            mbar_init(smem_u32(&st_full[s]), 1);
            mbar_init(smem_u32(&st_empty[s]), 1);
        }
        for (int u = 0; u < 2; u++) {
            mbar_init(smem_u32(&s_full[u]), 1);
            mbar_init(smem_u32(&p_full[u]), T3_EW);
            mbar_init(smem_u32(&pv_done[u]), 1);
        }
        mbar_init(smem_u32(&drain), 1);
        fence_mbar_init();
        prefetch_map(&tq);
        prefetch_map(&tqm);
        prefetch_map(&tdo);
    }
    if (warp == 1) tmem_alloc(&s_tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_kc[Q3_STAGES], last_ic = -1;
            for (int s = 0; s < Q3_STAGES; s++) last_kc[s] = -1;
            bool ok = true;
            int kc = 0, ic = 0;
            for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
                const Bwd3Item w = dq3_item(it, B, T, H);
                if (!mbar_wait(smem_u32(&q_empty), ((uint32_t)ic & 1u) ^ 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&q_full);
                mbar_expect_tx(fb, T3_FIXED);
                last_ic = ic;
                load_fixed(base, &tq, w.h * HS, w.tile * 128, w.b, fb);
                load_fixed(base + T3_TILE, &tdo, w.h * HS, w.tile * 128, w.b, fb);
                for (int j = 0; j < w.n; j++, kc++) {
                    const int s = kc % Q3_STAGES;
                    if (!mbar_wait(smem_u32(&st_empty[s]), ((uint32_t)(kc / Q3_STAGES) & 1u) ^ 1u, &s_abort,
                                   status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sb = smem_u32(&st_full[s]);
                    mbar_expect_tx(sb, Q3_STAGE);
                    last_kc[s] = kc;
                    const uint32_t st = base + T3_FIXED + s * Q3_STAGE;
                    load_stile(st, &tq, C + w.h * HS, j * T3_BS, w.b, sb);
                    load_stile(st + T3_STILE, &tq, 2 * C + w.h * HS, j * T3_BS, w.b, sb);
                    load_stile(st + 2 * T3_STILE, &tqm, C + w.h * HS, j * T3_BS, w.b, sb);
                }
            }
            if (!ok) {
                if (last_ic >= 0) drain_wait(smem_u32(&q_full), (uint32_t)last_ic & 1u);
                for (int s = 0; s < Q3_STAGES; s++)
                    if (last_kc[s] >= 0) drain_wait(smem_u32(&st_full[s]), (uint32_t)(last_kc[s] / Q3_STAGES) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = instr_desc(128, T3_BS, false, false, false);   // Q K^T, dO V^T: K-major
            const uint32_t id_o = instr_desc(128, HS, false, true, false);       // dS K: B MN-major
            const uint64_t dfix = smem_desc(base, 16, 1024, LAYOUT_SW128);
            const uint64_t dst_k = smem_desc(base + T3_FIXED, 16, 1024, LAYOUT_SW128);
            const uint64_t dst_mn = smem_desc(base + T3_FIXED + 2 * T3_STILE, T3_BOX, 512, LAYOUT_SW128_32B);
            constexpr uint32_t HALF_U = T3_HALF >> 4, BOX_U = T3_BOX >> 4, TILE_U = T3_TILE >> 4,
                               STILE_U = T3_STILE >> 4, STAGE_U = Q3_STAGE >> 4;
            bool ok = true;
            int kc = 0, cs = 0;
            uint64_t t_last = globaltimer();
            for (int it = blockIdx.x, ic = 0; it < nitems && ok; it += gridDim.x, ic++) {
                const Bwd3Item w = dq3_item(it, B, T, H);
                if (!mbar_wait(smem_u32(&q_full), (uint32_t)ic & 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                int ns = 0, no = 0;
                for (uint32_t spin = 1; ok && no < w.n; spin++) {
                    bool progress = false;
                    if (ns < w.n) {
                        const int s = (kc + ns) % Q3_STAGES, g = cs + ns, u = g & 1;
                        if (mbar_test_wait(smem_u32(&st_full[s]), (uint32_t)((kc + ns) / Q3_STAGES) & 1u) &&
                            (g < 2 || mbar_test_wait(smem_u32(&pv_done[u]), (uint32_t)((g - 2) >> 1) & 1u))) {
                            tc_fence_after();
                            const uint64_t kv = dst_k + (uint64_t)(s * STAGE_U);
                            score8(tmem + 128 * u, dfix, HALF_U, kv, BOX_U, id_s);                      // S = Q K^T
                            score8(tmem + 128 * u + 64, dfix + TILE_U, HALF_U, kv + STILE_U, BOX_U, id_s);  // dP = dO V^T
                            mma_commit(smem_u32(&s_full[u]));
                            if (++ns == w.n) mma_commit(smem_u32(&q_empty));   // Q, dO read for the last time
                            progress = true;
                        }
                    }
                    if (no < ns) {
                        const int g = cs + no, u = g & 1;
                        if (mbar_test_wait(smem_u32(&p_full[u]), (uint32_t)(g >> 1) & 1u)) {
                            tc_fence_after();
                            const int s = (kc + no) % Q3_STAGES;
                            acc8(tmem + 256, tmem + 128 * u + 64, dst_mn + (uint64_t)(s * STAGE_U), id_o,
                                 no > 0 ? 1u : 0u);                                             // dQ += dS K
                            mma_commit(smem_u32(&pv_done[u]));
                            mma_commit(smem_u32(&st_empty[s]));
                            no++;
                            progress = true;
                        }
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
        const int quarter = warp & 3, grp = (warp - 2) >> 2;     // TMEM lane quarter, 16-column group
        const int r = quarter * 32 + lane;
        const uint32_t lb = (uint32_t)(quarter * 32) << 16;
        const float c2 = scale * LOG2E;
        const uint64_t c2x2 = f2pack(c2, c2);
        bool ok = true;
        int cs = 0;
        for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x) {
            const Bwd3Item w = dq3_item(it, B, T, H);
            const int row = w.tile * 128 + r;
            const size_t bh = ((size_t)w.b * H + w.h) * T;
            const float lse2 = row < T ? __ldg(lse + bh + row) * LOG2E : INFINITY;   // +inf zeroes P past T
            const float Drow = row < T ? __ldg(Dg + bh + row) : 0.f;
            const uint64_t nl2 = f2pack(-lse2, -lse2), nd2 = f2pack(-Drow, -Drow);
            for (int j = 0; j < w.n; j++) {
                const int g = cs + j, u = g & 1;
                if (!mbar_wait(smem_u32(&s_full[u]), (uint32_t)(g >> 1) & 1u, &s_abort, status)) { ok = false; break; }
                tc_fence_after();
                uint32_t su[16], du[16];
                const uint32_t ts = tmem + lb + 128 * u + 16 * grp;
                tmem_ld16_async(ts, su);
                tmem_ld16_async(ts + 64, du);
                tmem_wait16(su);
                tmem_wait16(du);
                const int k0 = j * T3_BS + 16 * grp;                 // first key of this warp's columns
                const bool edge = k0 + 15 > row || k0 + 16 > T;      // the diagonal, the sequence end
                float dv[16];
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    float s0 = __uint_as_float(su[c]), s1 = __uint_as_float(su[c + 1]);
                    fma2(s0, s1, c2x2, nl2);
                    float p0 = ex2(s0), p1 = ex2(s1);
                    if (edge) {
                        if (k0 + c > row || k0 + c >= T) p0 = 0.f;
                        if (k0 + c + 1 > row || k0 + c + 1 >= T) p1 = 0.f;
                    }
                    float d0 = __uint_as_float(du[c]), d1 = __uint_as_float(du[c + 1]);
                    f2unpack(add2(f2pack(d0, d1), nd2), d0, d1);
                    dv[c] = p0 * d0;
                    dv[c + 1] = p1 * d1;
                }
                tmem_st16f(ts + 64, dv);                             // dS over dP
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&p_full[u]));
            }
            if (!ok) break;
            {
                const int g = cs + w.n - 1;
                if (!mbar_wait(smem_u32(&pv_done[g & 1]), (uint32_t)(g >> 1) & 1u, &s_abort, status)) break;
            }
            tc_fence_after();
            cs += w.n;
            if (grp < 2) {                                 // dQ: 64 columns, two groups of 32
                float o[32];
                tmem_ld32(tmem + lb + 256 + 32 * grp, o);
                tmem_wait_ld(o);
                if (row < T) store_row32(o, scale, dqkv + ((size_t)w.b * T + row) * 3 * C + w.h * HS + 32 * grp);
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

// dqkv [B,T,3C] (fp32, every element written) from dy [B,T,C], qkv [B,T,3C]
// (fp32), the forward's lse [B,H,T] and D [B,H,T] = rowsum(dO o O); head size
// 64, no dropout; the products on tf32 tensor cores with fp32 accumulation.
int attention_tc05_tf32_backward(float* dqkv, const float* dy, const float* qkv, const float* lse, const float* D,
                                 int B, int T, int C, int H, int* status, cudaStream_t st) {
    using namespace at05;
    if (C % H || C / H != HS || C % 8) return GPT2_ENOTSUP;
    if (smem_limit(reinterpret_cast<const void*>(attn_bwd_dkv_tf32), (int)KV3_SMEM) ||
        smem_limit(reinterpret_cast<const void*>(attn_bwd_dq_tf32), (int)Q3_SMEM))
        return GPT2_ECUDA;
    // boxes of 64 rows x 32 columns; K-major tiles with the 16-byte-chunk
    // swizzle, MN-major tiles with the 32-byte-chunk swizzle
    CUtensorMap tq, tqm, tdo, tdom;
    const cuuint64_t dq_[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t sq_[2] = {(cuuint64_t)3 * C * 4, (cuuint64_t)T * 3 * C * 4};
    const cuuint64_t dd_[3] = {(cuuint64_t)C, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t sd_[2] = {(cuuint64_t)C * 4, (cuuint64_t)T * C * 4};
    const cuuint32_t box[3] = {32, (cuuint32_t)T3_BS, 1};
    if (!encode_tensor_map(&tq, false, 3, qkv, dq_, sq_, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&tqm, false, 3, qkv, dq_, sq_, box, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B) ||
        !encode_tensor_map(&tdo, false, 3, dy, dd_, sd_, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&tdom, false, 3, dy, dd_, sd_, box, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B))
        return GPT2_ENOTSUP;
    const float scale = 1.f / sqrtf((float)HS);
    const int nitems = B * H * ((T + 127) / 128);
    const int grid = std::min(nitems, num_sms());
    count_launch(), attn_bwd_dq_tf32<<<grid, T3_THREADS, Q3_SMEM, st>>>(tq, tqm, tdo, dqkv, lse, D, B, T, C, H, scale,
                                                                        status);
    count_launch(), attn_bwd_dkv_tf32<<<grid, T3_THREADS, KV3_SMEM, st>>>(tq, tqm, tdo, tdom, dqkv, lse, D, B, T, C,
                                                                          H, scale, status);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k
