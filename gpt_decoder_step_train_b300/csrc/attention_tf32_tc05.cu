// attention_tf32_tc05.cu -- causal self-attention forward on the 5th-generation
// tensor cores with tf32 operands (the fp32 qkv read as it is stored), head
// size 64: the forward of the tf32 tensor-core mode.
//
// Per (batch b, head h): S = Q K^T / sqrt(hs), S[i,j] = -inf for j > i,
// P = softmax_rows(S), O = P V, and the row log-sum-exp of the scaled scores
// for the backward ("GPT-2 from scratch with torch", section 自注意力; the
// 1/sqrt(d_k) scaling: "从头搭建GPT(Andrej Karpathy) 笔记", section
// attention中为什么要做scaling).
//
// The roles and work items are those of the bf16 forward kernel
// (attention_tc05.cu): a persistent CTA of 384 threads per SM walks pairs of
// adjacent 128-row query tiles, heaviest first; warp 0 loads by TMA, one
// thread of warp 1 issues the MMAs of both query tiles as their inputs become
// ready, warp 2 owns the tensor memory, warps 4-7 and 8-11 run the softmax of
// query tile 0 and 1 (one row per thread).  What changes with 32-bit operands:
//   - a 128 x 64 fp32 tile is 32 KB, two 128-byte swizzle atoms along hs: Q
//     and K are K-major operands held as two 16 KB boxes of 128 rows x 32
//     columns (K steps of 32 bytes, the second box 16 KB on), V is read
//     MN-major with the 128-byte swizzle of 32-byte chunks (boxes of 128 keys
//     x 32 columns; LBO 16 KB between the two boxes, SBO 512 bytes; a K step
//     of 8 keys is 1 KB);
//   - one MMA covers K = 8: S_g(j) = Q_g K_j^T is 8 MMAs (M 128, N 128) and
//     O_g += P_g V_j 16 MMAs (M 128, N 64) with P_g read from tensor memory;
//   - P_g (fp32, 128 columns) is written over S_g in tensor memory, so
//     S_g(j + 1) is issued only once PV_g(j) has completed (the MMA thread
//     polls pv_done), and the softmax warps, handed S_g(j + 1), may rescale O_g
//     at once;
//   - shared memory: one buffer for the item's two query tiles (64 KB,
//     released when the item's last S has completed, so the next item's load
//     overlaps its last PV products), a ring of three K tiles and one of two V
//     tiles (32 KB each): 224 KB.
// Every wait is bounded (about one second); a wait that gives up raises
// GPT2_STATUS_TIMEOUT, all roles leave, in-flight copies and MMAs are drained
// and tensor memory is freed.
#include "common.cuh"
#include "gemm.cuh"
#include "ptx.cuh"
#include "attention_tc05.cuh"

namespace gpt2k {
namespace at05 {

using namespace ptx;

constexpr int G_BK = 128;                          // keys per tile
constexpr int G_KS = 3, G_VS = 2;                  // K and V ring stages
constexpr int G_THREADS = 384;
constexpr uint32_t G_TILE = 128 * HS * 4;          // one 128 x 64 fp32 tile: 32 KB
constexpr uint32_t G_BOX = G_TILE / 2;             // one box: 128 rows x 32 fp32
constexpr uint32_t G_OFF_Q = 0, G_OFF_K = 2 * G_TILE, G_OFF_V = G_OFF_K + G_KS * G_TILE,
                   G_SMEM_USED = G_OFF_V + G_VS * G_TILE;
constexpr size_t G_SMEM = G_SMEM_USED + 1024;
constexpr uint32_t G_TMEM_COLS = 512;   // S_0/P_0 [0,128) S_1/P_1 [128,256) O_0 [256,320) O_1 [320,384)

__global__ void __launch_bounds__(G_THREADS, 1)
attn_fwd_tf32_tc05(const __grid_constant__ CUtensorMap tqk, const __grid_constant__ CUtensorMap tv,
                   float* __restrict__ y, float* __restrict__ lse, int B, int T, int C, int H, float scale_log2,
                   int* status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full, q_empty, k_full[G_KS], k_empty[G_KS], v_full[G_VS], v_empty[G_VS],
        s_full[2], p_full[2], pv_done[2], drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = fwd_items(B, T, H);
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;

    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&q_full), 1);
        mbar_init(smem_u32(&q_empty), 1);
        for (int s = 0; s < G_KS; s++) {
            mbar_init(smem_u32(&k_full[s]), 1);
            mbar_init(smem_u32(&k_empty[s]), 1);
        }
        for (int s = 0; s < G_VS; s++) {
            mbar_init(smem_u32(&v_full[s]), 1);
            mbar_init(smem_u32(&v_empty[s]), 1);
        }
        for (int g = 0; g < 2; g++) {
            mbar_init(smem_u32(&s_full[g]), 1);
            mbar_init(smem_u32(&p_full[g]), 4);
            mbar_init(smem_u32(&pv_done[g]), 1);
        }
        mbar_init(smem_u32(&drain), 1);
        fence_mbar_init();
        prefetch_map(&tqk);
        prefetch_map(&tv);
    }
    if (warp == 2) tmem_alloc(&s_tmem, G_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    // registers as in the bf16 forward: 4 x 32 x 88 + 8 x 32 x 208 = 64512 = 384 x 168
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_k[G_KS], last_v[G_VS], last_q = -1;   // last fill of each buffer (abort drain)
            for (int s = 0; s < G_KS; s++) last_k[s] = -1;
            for (int s = 0; s < G_VS; s++) last_v[s] = -1;
            bool ok = true;
            int kc = 0, ic = 0;                        // key tiles and items loaded so far
            for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
                const FwdItem w = fwd_item(it, B, T, H);
                if (!mbar_wait(smem_u32(&q_empty), ((uint32_t)ic & 1u) ^ 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(smem_u32(&q_full), 2 * G_TILE);
                last_q = ic;
                for (int g = 0; g < 2; g++)
                    for (int ka = 0; ka < 2; ka++)
                        tma_load_3d(base + G_OFF_Q + g * G_TILE + ka * G_BOX, &tqk, w.h * HS + 32 * ka,
                                    w.qrow0 + 128 * g, w.b, smem_u32(&q_full));
                for (int j = 0; j < w.nkv; j++, kc++) {
                    const int sk = kc % G_KS, sv = kc % G_VS;
                    if (!mbar_wait(smem_u32(&k_empty[sk]), ((uint32_t)(kc / G_KS) & 1u) ^ 1u, &s_abort, status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(smem_u32(&k_full[sk]), G_TILE);
                    last_k[sk] = kc;
                    for (int ka = 0; ka < 2; ka++)
                        tma_load_3d(base + G_OFF_K + sk * G_TILE + ka * G_BOX, &tqk, C + w.h * HS + 32 * ka,
                                    j * G_BK, w.b, smem_u32(&k_full[sk]));
                    if (!mbar_wait(smem_u32(&v_empty[sv]), ((uint32_t)(kc / G_VS) & 1u) ^ 1u, &s_abort, status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(smem_u32(&v_full[sv]), G_TILE);
                    last_v[sv] = kc;
                    for (int nb = 0; nb < 2; nb++)
                        tma_load_3d(base + G_OFF_V + sv * G_TILE + nb * G_BOX, &tv, 2 * C + w.h * HS + 32 * nb,
                                    j * G_BK, w.b, smem_u32(&v_full[sv]));
                }
            }
            if (!ok) {
                // wait (bounded, ignoring the abort flag) for every copy this thread issued;
                // earlier fills of a buffer completed before it was refilled
                if (last_q >= 0) {
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&q_full), (uint32_t)last_q & 1u) && globaltimer() - t0 < WAIT_NS) {
                    }
                }
                for (int s = 0; s < G_KS; s++) {
                    if (last_k[s] < 0) continue;
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&k_full[s]), (uint32_t)(last_k[s] / G_KS) & 1u) &&
                           globaltimer() - t0 < WAIT_NS) {
                    }
                }
                for (int s = 0; s < G_VS; s++) {
                    if (last_v[s] < 0) continue;
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&v_full[s]), (uint32_t)(last_v[s] / G_VS) & 1u) &&
                           globaltimer() - t0 < WAIT_NS) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = instr_desc(128, G_BK, false, false, false);   // Q K^T: both K-major
            const uint32_t id_pv = instr_desc(128, HS, false, true, false);     // P V: V MN-major
            // descriptors (start addresses in 16-byte units): a K step of 8 tf32 is
            // 32 bytes along a K-major row, the second 32 columns of a tile start one
            // box (16 KB) on; a K step of 8 keys of V is 8 rows of 128 bytes
            const uint64_t dq0 = smem_desc(base + G_OFF_Q, 16, 1024, LAYOUT_SW128);
            const uint64_t dk0 = smem_desc(base + G_OFF_K, 16, 1024, LAYOUT_SW128);
            const uint64_t dv0 = smem_desc(base + G_OFF_V, G_BOX, 512, LAYOUT_SW128_32B);
            constexpr uint32_t BOX_U = G_BOX >> 4, TILE_U = G_TILE >> 4, VSTEP_U = (8 * 128) >> 4;
            bool ok = true;
            int kc = 0;                                // key tiles consumed so far
            int cs[2] = {0, 0};                        // S (and PV) groups of earlier items, per query tile
            uint64_t t_last = globaltimer();
            for (int it = blockIdx.x, ic = 0; it < nitems && ok; it += gridDim.x, ic++) {
                const FwdItem w = fwd_item(it, B, T, H);
                if (!mbar_wait(smem_u32(&q_full), (uint32_t)ic & 1u, &s_abort, status)) { ok = false; break; }
                auto issue_s = [&](int g, int j) {     // S_g = Q_g K_j^T (8 MMAs, K = 64)
                    const uint32_t d = tmem + g * G_BK;
                    const uint64_t a = dq0 + (uint64_t)(g * TILE_U);
                    const uint64_t b = dk0 + (uint64_t)(((kc + j) % G_KS) * TILE_U);
                    mma4_ss_tf32(d, a, b, 2, 2, id_s, 0u);
                    mma4_ss_tf32(d, a + BOX_U, b + BOX_U, 2, 2, id_s, 1u);
                    mma_commit(smem_u32(&s_full[g]));
                };
                auto issue_pv = [&](int g, int j) {    // O_g += P_g V_j (16 MMAs, P_g over S_g)
                    const uint64_t vb = dv0 + (uint64_t)(((kc + j) % G_VS) * TILE_U);
                    const uint32_t d = tmem + 2 * G_BK + g * HS, a = tmem + g * G_BK;
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        mma4_ts_tf32(d, a + 32 * q, vb + (uint64_t)(4 * q * VSTEP_U), VSTEP_U, id_pv,
                                     (j > 0 || q > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&pv_done[g]));
                };
                // a K (V) stage is released once every S (PV) group of this item that
                // reads it was issued: one per query tile that needs the key tile
                auto tile_uses = [&](int j) { return (j < w.nkv0 ? 1 : 0) + (j < w.nkv1 ? 1 : 0); };
                int kuse[G_KS], vuse[G_VS];
                for (int s = 0; s < G_KS; s++) kuse[s] = s < w.nkv ? tile_uses(s) : 0;
                for (int s = 0; s < G_VS; s++) vuse[s] = s < w.nkv ? tile_uses(s) : 0;
                auto k_used = [&](int j) {
                    const int s = j % G_KS;
                    if (--kuse[s] == 0) {
                        mma_commit(smem_u32(&k_empty[(kc + j) % G_KS]));
                        if (j + G_KS < w.nkv) kuse[s] = tile_uses(j + G_KS);
                    }
                };
                auto v_used = [&](int j) {
                    const int s = j % G_VS;
                    if (--vuse[s] == 0) {
                        mma_commit(smem_u32(&v_empty[(kc + j) % G_VS]));
                        if (j + G_VS < w.nkv) vuse[s] = tile_uses(j + G_VS);
                    }
                };
                const int n[2] = {w.nkv0, w.nkv1};
                int ns[2] = {0, 0}, npv[2] = {0, 0};
                bool q_released = false;
                for (uint32_t spin = 1; ok && (npv[0] < n[0] || npv[1] < n[1]); spin++) {
                    bool progress = false;
#pragma unroll
                    for (int g = 0; g < 2; g++) {
                        // S_g(j) overwrites P_g(j - 1): only after PV_g(j - 1) was issued
                        // and has completed
                        if (ns[g] < n[g] && ns[g] == npv[g]) {
                            const int j = ns[g], gs = cs[g] + j;   // this S's index over the whole run
                            if (mbar_test_wait(smem_u32(&k_full[(kc + j) % G_KS]),
                                               (uint32_t)((kc + j) / G_KS) & 1u) &&
                                (gs == 0 || mbar_test_wait(smem_u32(&pv_done[g]), (uint32_t)(gs - 1) & 1u))) {
                                tc_fence_after();
                                issue_s(g, j);
                                k_used(j);
                                ns[g]++;
                                progress = true;
                                if (!q_released && ns[0] == n[0] && ns[1] == n[1]) {
                                    mma_commit(smem_u32(&q_empty));   // lands once the item's last S has read Q
                                    q_released = true;
                                }
                            }
                        }
                        if (npv[g] < ns[g]) {
                            const int j = npv[g];
                            if (mbar_test_wait(smem_u32(&p_full[g]), (uint32_t)(cs[g] + j) & 1u) &&
                                mbar_test_wait(smem_u32(&v_full[(kc + j) % G_VS]), (uint32_t)((kc + j) / G_VS) & 1u)) {
                                tc_fence_after();
                                issue_pv(g, j);
                                v_used(j);
                                npv[g]++;
                                progress = true;
                            }
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
                if (!ok) break;
                cs[0] += n[0];
                cs[1] += n[1];
                kc += w.nkv;
            }
            // every MMA issued has completed once this commit lands
            mma_commit(smem_u32(&drain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(&drain), 0) && globaltimer() - t0 < WAIT_NS) {
            }
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 208;" ::: "memory");
        // ------------------------------------------------ softmax (warps 4-7: tile 0, 8-11: tile 1)
        const int g = (warp - 4) >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;             // row within the query tile
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_s = tmem + lane_base + g * G_BK, t_o = tmem + lane_base + 2 * G_BK + g * HS;
        const uint64_t sc2 = f2pack(scale_log2, scale_log2);
        bool ok = true;
        int cs = 0;                                    // S tiles of earlier items
        for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x) {
            const FwdItem w = fwd_item(it, B, T, H);
            const int row = w.qrow0 + 128 * g + r;
            const int n = g == 0 ? w.nkv0 : w.nkv1;
            float m_run = -INFINITY;                   // log2-domain maximum in use
            uint64_t l2 = f2pack(0.f, 0.f);            // this row's sum of P, two partial lanes
            for (int j = 0; j < n; j++) {
                // S_g(j) was issued after PV_g(j - 1) had completed: O_g and the
                // S_g / P_g columns belong to these warps until p_full
                if (!mbar_wait(smem_u32(&s_full[g]), (uint32_t)(cs + j) & 1u, &s_abort, status)) { ok = false; break; }
                tc_fence_after();
                float sv[128];
                tmem_ld128(t_s, sv);
                // mask: the diagonal tile and the sequence end
                const int k0 = j * G_BK;
                if (k0 + G_BK - 1 > row || k0 + G_BK > T) {
#pragma unroll
                    for (int c = 0; c < 128; c++)
                        if (k0 + c > row || k0 + c >= T) sv[c] = -INFINITY;
                }
                float mx;
                {
                    float m43[43];
#pragma unroll
                    for (int c = 0; c < 42; c++) m43[c] = max3(sv[3 * c], sv[3 * c + 1], sv[3 * c + 2]);
                    m43[42] = fmaxf(sv[126], sv[127]);
                    float m15[15];
#pragma unroll
                    for (int c = 0; c < 14; c++) m15[c] = max3(m43[3 * c], m43[3 * c + 1], m43[3 * c + 2]);
                    m15[14] = m43[42];
                    float m5[5];
#pragma unroll
                    for (int c = 0; c < 5; c++) m5[c] = max3(m15[3 * c], m15[3 * c + 1], m15[3 * c + 2]);
                    mx = fmaxf(max3(m5[0], m5[1], m5[2]), fmaxf(m5[3], m5[4])) * scale_log2;
                }
                float alpha = 1.f;                     // factor on O and l for this tile
                if (mx > m_run + RESCALE_LOG2 || (m_run == -INFINITY && mx > -INFINITY)) {
                    alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mx);
                    m_run = mx;
                }
                const float mref = m_run == -INFINITY ? 0.f : m_run;
                const uint64_t nm2 = f2pack(-mref, -mref);
                uint64_t acc[4] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < 128; c += 2) {
                    fma2(sv[c], sv[c + 1], sc2, nm2);
                    sv[c] = ex2(sv[c]);
                    sv[c + 1] = ex2(sv[c + 1]);
                    acc[(c >> 1) & 3] = add2(acc[(c >> 1) & 3], f2pack(sv[c], sv[c + 1]));
                }
                {
                    float a0, a1;
                    f2unpack(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])), a0, a1);
                    float l0, l1;
                    f2unpack(l2, l0, l1);
                    l2 = f2pack(l0 * alpha + a0, l1 * alpha + a1);
                }
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int hh = 0; hh < 2; hh++) {
                        float o[32];
                        tmem_ld32(t_o + 32 * hh, o);
                        tmem_wait_ld(o);
#pragma unroll
                        for (int c = 0; c < 32; c++) o[c] *= alpha;
                        tmem_st32(t_o + 32 * hh, o);
                    }
                }
                // the P row (fp32, the MMA reads it as tf32) over the S columns
#pragma unroll
                for (int q = 0; q < 4; q++) tmem_st32(t_s + 32 * q, *reinterpret_cast<const float(*)[32]>(&sv[32 * q]));
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&p_full[g]));
            }
            if (!ok || n == 0) continue;
            if (!mbar_wait(smem_u32(&pv_done[g]), (uint32_t)(cs + n - 1) & 1u, &s_abort, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            cs += n;
            float o[64];
            {
                float (&oa)[32] = *reinterpret_cast<float(*)[32]>(&o[0]);
                float (&ob)[32] = *reinterpret_cast<float(*)[32]>(&o[32]);
                tmem_ld32(t_o, oa);
                tmem_ld32(t_o + 32, ob);
                tmem_wait_ld(oa);
                tmem_wait_ld(ob);
            }
            if (row < T) {
                float l0, l1;
                f2unpack(l2, l0, l1);
                const float l = l0 + l1;
                const float inv = 1.f / l;
                float4* yr = reinterpret_cast<float4*>(y + ((size_t)w.b * T + row) * C + w.h * HS);
#pragma unroll
                for (int c = 0; c < 16; c++)
                    yr[c] = make_float4(o[4 * c] * inv, o[4 * c + 1] * inv, o[4 * c + 2] * inv, o[4 * c + 3] * inv);
                lse[((size_t)w.b * H + w.h) * T + row] = (m_run + log2f(l)) * LN2;
            }
            // the next item's PV_g(0) overwrites O_g: every lane has read it
            tc_fence_before();
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, G_TMEM_COLS);
    }
}

}  // namespace at05

bool attention_tc05_supported(int hs, int C);

// y [B,T,C] and lse [B,H,T] from qkv [B,T,3C], all fp32, head size 64; the
// products on tf32 tensor cores with fp32 accumulation.
int attention_tc05_tf32_forward(float* y, float* lse, const float* qkv, int B, int T, int C, int H, int* status,
                                cudaStream_t st) {
    using namespace at05;
    if (C % H || C / H != HS || !attention_tc05_supported(HS, C)) return GPT2_ENOTSUP;
    if (smem_limit(reinterpret_cast<const void*>(attn_fwd_tf32_tc05), (int)G_SMEM)) return GPT2_ECUDA;
    // qkv as a 3-D tensor [B][T][3C]: boxes of 128 rows x 32 columns (half a head);
    // Q and K with the 16-byte-chunk swizzle (K-major operands), V with the
    // 32-byte-chunk swizzle (MN-major operand)
    CUtensorMap tqk, tv;
    const cuuint64_t dims[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)3 * C * 4, (cuuint64_t)T * 3 * C * 4};
    const cuuint32_t box[3] = {32, 128, 1};
    if (!encode_tensor_map(&tqk, false, 3, qkv, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&tv, false, 3, qkv, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B))
        return GPT2_ENOTSUP;
    const float scale_log2 = LOG2E / sqrtf((float)HS);
    const int nitems = fwd_items(B, T, H);
    const dim3 grid(std::min(nitems, num_sms()));
    count_launch(), attn_fwd_tf32_tc05<<<grid, G_THREADS, G_SMEM, st>>>(tqk, tv, y, lse, B, T, C, H, scale_log2,
                                                                         status);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k
