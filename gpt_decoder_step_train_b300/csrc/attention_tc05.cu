// attention_tc05.cu -- causal self-attention, forward and backward, on the
// 5th-generation tensor cores (tcgen05), bf16 operands, head size 64.
//
// Per (batch b, head h): S = Q K^T / sqrt(hs), S[i,j] = -inf for j > i,
// P = softmax_rows(S), O = P V, and the row log-sum-exp of the scaled scores
// is kept for the backward ("GPT-2 from scratch with torch", section
// 自注意力; the 1/sqrt(d_k) scaling: "从头搭建GPT(Andrej Karpathy) 笔记",
// section attention中为什么要做scaling).  The kernels' layouts are described
// above each of them.
// Every wait is bounded (about one second); a wait that gives up raises
// GPT2_STATUS_TIMEOUT, all roles leave, in-flight copies and MMAs are drained
// and tensor memory is freed.
#include <cuda_bf16.h>

#include "common.cuh"
#include "gemm.cuh"
#include "ptx.cuh"
#include "attention_tc05.cuh"

namespace gpt2k {
namespace at05 {

using namespace ptx;

// Issue loop of the MMA thread.  Each tile j has two groups of MMAs:
//   A  needs the tile's operand stage (full[j % stages], phase (j / stages) & 1)
//      and its score columns, buffer j % ns of ns, released by the element-wise
//      warps after tile j - ns (s_free[j % ns], phase ((j - ns) / ns) & 1);
//   B  needs the element-wise warps' operand tile of tile j (p_full[j % np],
//      phase (j / np) & 1; np operand buffers used in turn).
// Issue order A(0), A(1), B(0), A(2), B(1), ...: the scores of tile j + 1 are
// computed while the element-wise warps work on tile j (with ns = 2 the
// element-wise warps never wait for them: the buffer of tile j + 1 was
// released two tiles earlier).  Every wait blocks
// (the thread is suspended, taking no issue slots from the element-wise warps
// on its scheduler) and is bounded.  No deadlock: A(j + 1) needs only the
// release of S_{j+1-ns}, which the warps give before they wait for B(j - 1); no phase
// can be lapped, since every barrier's next phase needs this thread to have
// consumed the current one.  Gives up (abort flag, GPT2_STATUS_TIMEOUT) when a
// wait runs out.
template <class IssueA, class IssueB>
__device__ __forceinline__ bool mma_two_group_loop(int n, uint64_t* full, int stages, uint64_t* s_free, int ns,
                                                   uint64_t* p_full, int np, volatile int* abort_flag, int* status,
                                                   IssueA&& issue_a, IssueB&& issue_b) {
    for (int j = 0; j <= n; j++) {
        if (j < n) {
            if (!mbar_wait(smem_u32(&full[j % stages]), (uint32_t)(j / stages) & 1u, abort_flag, status))
                return false;
            if (j >= ns &&
                !mbar_wait(smem_u32(&s_free[j % ns]), (uint32_t)((j - ns) / ns) & 1u, abort_flag, status))
                return false;
            tc_fence_after();
            issue_a(j);
        }
        if (j > 0) {
            const int jb = j - 1;
            if (!mbar_wait(smem_u32(&p_full[jb % np]), (uint32_t)(jb / np) & 1u, abort_flag, status)) return false;
            tc_fence_after();
            issue_b(jb);
        }
    }
    return true;
}

// ---------------------------------------------------------------- forward
// Persistent: one CTA per SM (384 threads) walks work items, each a pair of
// adjacent 128-row query tiles of one (batch, head) (rows 256 p .. 256 p + 255),
// heaviest pairs first:
//   warp 0     TMA producer: both query tiles of an item into one of two query
//              buffers (the next item's load overlaps the current item), then
//              the K and V tiles of 128 keys into a five-stage ring (128-byte
//              swizzle);
//   warp 1     from one lane issues the MMAs of both query tiles as their
//              inputs become ready (a polling loop over the barriers):
//              S_g = Q_g K_j^T (M 128, N 128, K 64) as soon as the softmax
//              warps have read S_g(j - 1) and K_j has landed, so it runs while
//              they compute; O_g += P_g V_j (M 128, N 64, K 128; P_g read
//              from tensor memory, V from shared memory read MN-major) as
//              soon as P_g(j) is written;
//   warp 2     allocates and frees the tensor memory (S_0, S_1: 128 columns
//              each; O_0, O_1: 64 columns each; P_0, P_1: 64 columns each,
//              bf16 pairs);
//   warps 4-7  softmax of query tile 0, warps 8-11 of query tile 1: one row
//              per thread (its TMEM lane) over all 128 keys of a tile, so no
//              row reduction crosses threads.  Causal mask only on the
//              diagonal tile (and past T), online maximum and sum in the log2
//              domain with the scale folded into one packed FMA before ex2,
//              the running maximum moved only when a row's maximum grows past
//              2^8 (O in tensor memory is then rescaled first), P written to
//              its tensor-memory columns as bf16 pairs (the MMA's A operand:
//              no shared-memory traffic for P).
// Per query tile the softmax warps signal s_free (S read) and p_full (P
// written); the MMA thread signals s_full (S ready) and pv_done (PV done:
// O and P may be touched again).  Key tiles past a query tile's last row are
// never visited.
constexpr int F_BK = 128;                          // keys per tile
constexpr int F_STAGES = 5;
constexpr int F_THREADS = 384;
constexpr uint32_t F_Q_BYTES = 128 * HS * 2;       // one query tile: 16 KB
constexpr uint32_t F_KV_BYTES = F_BK * HS * 2;     // one K or V tile: 16 KB
// two query buffers (the next item's pair of query tiles loads while the
// current one runs), then the K and V rings
constexpr uint32_t F_OFF_Q = 0, F_OFF_K = 4 * F_Q_BYTES, F_OFF_V = F_OFF_K + F_STAGES * F_KV_BYTES,
                   F_SMEM_USED = F_OFF_V + F_STAGES * F_KV_BYTES;
constexpr size_t F_SMEM = F_SMEM_USED + 1024;
constexpr uint32_t F_TMEM_COLS = 512;   // S_0 [0,128) S_1 [128,256) O_0 [256,320) O_1 [320,384) P_0, P_1 [384,512)

template <bool DROP>
__global__ void __launch_bounds__(F_THREADS, 1)
attn_fwd_tc05(const __grid_constant__ CUtensorMap tm, __nv_bfloat16* __restrict__ y, float* __restrict__ lse,
              int B, int T, int C, int H, float scale_log2, int* status, const uint32_t* __restrict__ bits,
              float ks) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full[2], q_empty[2], kv_full[F_STAGES], kv_empty[F_STAGES], s_full[2],
        s_free[2], p_full[2], pv_done[2], drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nitems = fwd_items(B, T, H);
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int q = 0; q < 2; q++) {
            mbar_init(smem_u32(&q_full[q]), 1);
            mbar_init(smem_u32(&q_empty[q]), 1);
        }
        for (int s = 0; s < F_STAGES; s++) {
            mbar_init(smem_u32(&kv_full[s]), 1);
            mbar_init(smem_u32(&kv_empty[s]), 1);
        }
        for (int g = 0; g < 2; g++) {
            mbar_init(smem_u32(&s_full[g]), 1);
            mbar_init(smem_u32(&s_free[g]), 4);
            mbar_init(smem_u32(&p_full[g]), 4);
            mbar_init(smem_u32(&pv_done[g]), 1);
        }
        mbar_init(smem_u32(&drain), 1);
        fence_mbar_init();
        prefetch_map(&tm);
    }
    if (warp == 2) tmem_alloc(&s_tmem, F_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    // registers: the producer / MMA warpgroup gives most of its share to the two
    // softmax warpgroups (launched with 168 per thread: 4 x 32 x 88 +
    // 8 x 32 x 208 = 64512 = 384 x 168)
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_kc[F_STAGES], last_ic[2];         // last fill of each buffer (abort drain)
            for (int s = 0; s < F_STAGES; s++) last_kc[s] = -1;
            last_ic[0] = last_ic[1] = -1;
            bool ok = true;
            int kc = 0, ic = 0;                        // K/V tiles and items loaded so far
            for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
                const FwdItem w = fwd_item(it, B, T, H);
                const int qb = ic & 1;
                if (!mbar_wait(smem_u32(&q_empty[qb]), ((uint32_t)(ic >> 1) & 1u) ^ 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(smem_u32(&q_full[qb]), 2 * F_Q_BYTES);
                last_ic[qb] = ic;
                for (int k = 0; k < 4; k++)            // four 64-row boxes: tile 0, then tile 1
                    tma_load_3d(base + F_OFF_Q + qb * 2 * F_Q_BYTES + k * (F_Q_BYTES / 2), &tm, w.h * HS,
                                w.qrow0 + 64 * k, w.b, smem_u32(&q_full[qb]));
                for (int j = 0; j < w.nkv; j++, kc++) {
                    const int s = kc % F_STAGES;
                    if (!mbar_wait(smem_u32(&kv_empty[s]), ((uint32_t)(kc / F_STAGES) & 1u) ^ 1u, &s_abort, status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&kv_full[s]);
                    mbar_expect_tx(fb, 2 * F_KV_BYTES);
                    last_kc[s] = kc;
                    for (int k = 0; k < 2; k++) {
                        tma_load_3d(base + F_OFF_K + s * F_KV_BYTES + k * (F_KV_BYTES / 2), &tm, C + w.h * HS,
                                    j * F_BK + 64 * k, w.b, fb);
                        tma_load_3d(base + F_OFF_V + s * F_KV_BYTES + k * (F_KV_BYTES / 2), &tm, 2 * C + w.h * HS,
                                    j * F_BK + 64 * k, w.b, fb);
                    }
                }
            }
            if (!ok) {
                // wait (bounded, ignoring the abort flag) for every copy this thread issued;
                // earlier fills of a buffer completed before it was refilled
                for (int q = 0; q < 2; q++) {
                    if (last_ic[q] < 0) continue;
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&q_full[q]), (uint32_t)(last_ic[q] >> 1) & 1u) &&
                           globaltimer() - t0 < WAIT_NS) {
                    }
                }
                for (int s = 0; s < F_STAGES; s++) {
                    if (last_kc[s] < 0) continue;
                    const uint32_t ph = (uint32_t)(last_kc[s] / F_STAGES) & 1u;
                    const uint64_t t1 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&kv_full[s]), ph) && globaltimer() - t1 < WAIT_NS) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = instr_desc(128, F_BK, false, false, true);   // Q K^T: both K-major
            const uint32_t id_pv = instr_desc(128, HS, false, true, true);     // P V: V MN-major
            // descriptors precomputed; a K step of 16 bf16 is 32 bytes along a
            // K-major row (2 units of 16 bytes) or 16 rows of an MN-major V tile
            // (2048 bytes, 128 units)
            const uint64_t dq0 = smem_desc(base + F_OFF_Q, 16, 1024, LAYOUT_SW128);
            const uint64_t dk0 = smem_desc(base + F_OFF_K, 16, 1024, LAYOUT_SW128);
            const uint64_t dv0 = smem_desc(base + F_OFF_V, 8192, 1024, LAYOUT_SW128);
            bool ok = true;
            int kc = 0, ic = 0;                        // K/V tiles and items consumed so far
            int cs[2] = {0, 0}, cpv[2] = {0, 0};       // S and PV groups issued so far, per query tile
            uint64_t t_last = globaltimer();
            for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x, ic++) {
                const FwdItem w = fwd_item(it, B, T, H);
                const int qb = ic & 1;
                if (!mbar_wait(smem_u32(&q_full[qb]), (uint32_t)(ic >> 1) & 1u, &s_abort, status)) { ok = false; break; }
                auto issue_s = [&](int g, int j) {     // S_g = Q_g K_j^T (4 MMAs, K = 64)
                    mma4_ss(tmem + g * F_BK, dq0 + (uint64_t)((qb * 2 + g) * (F_Q_BYTES >> 4)),
                            dk0 + (uint64_t)(((kc + j) % F_STAGES) * (F_KV_BYTES >> 4)), 2, 2, id_s, 0u);
                    mma_commit(smem_u32(&s_full[g]));
                };
                auto issue_pv = [&](int g, int j) {    // O_g += P_g V_j (8 MMAs, P_g in tensor memory)
                    const uint64_t vb = dv0 + (uint64_t)(((kc + j) % F_STAGES) * (F_KV_BYTES >> 4));
                    const uint32_t d = tmem + 2 * F_BK + g * HS, a = tmem + 2 * F_BK + 2 * HS + g * 64;
                    mma4_ts(d, a, vb, 128, id_pv, j > 0 ? 1u : 0u);
                    mma4_ts(d, a + 32, vb + 512, 128, id_pv, 1u);
                    mma_commit(smem_u32(&pv_done[g]));
                };
                // a K/V stage is released once every MMA group of this item that reads it
                // was issued (S and PV of each query tile that needs the key tile)
                auto tile_uses = [&](int j) { return (j < w.nkv0 ? 2 : 0) + (j < w.nkv1 ? 2 : 0); };
                int uses[F_STAGES];
                for (int st = 0; st < F_STAGES; st++) uses[st] = st < w.nkv ? tile_uses(st) : 0;
                auto used = [&](int j) {
                    const int st = j % F_STAGES;
                    if (--uses[st] == 0) {
                        mma_commit(smem_u32(&kv_empty[(kc + j) % F_STAGES]));
                        if (j + F_STAGES < w.nkv) uses[st] = tile_uses(j + F_STAGES);
                    }
                };
                const int n[2] = {w.nkv0, w.nkv1};
                int ns[2] = {0, 0}, npv[2] = {0, 0};
                for (uint32_t spin = 1; ok && (npv[0] < n[0] || npv[1] < n[1]); spin++) {
                    bool progress = false;
#pragma unroll
                    for (int g = 0; g < 2; g++) {
                        if (ns[g] < n[g]) {
                            const int j = ns[g], gs = cs[g] + j;   // this S's index over the whole run
                            if (mbar_test_wait(smem_u32(&kv_full[(kc + j) % F_STAGES]),
                                               (uint32_t)((kc + j) / F_STAGES) & 1u) &&
                                (gs == 0 || mbar_test_wait(smem_u32(&s_free[g]), (uint32_t)(gs - 1) & 1u))) {
                                tc_fence_after();
                                issue_s(g, j);
                                used(j);
                                ns[g]++;
                                progress = true;
                            }
                        }
                        if (npv[g] < ns[g]) {
                            const int j = npv[g];
                            if (mbar_test_wait(smem_u32(&p_full[g]), (uint32_t)(cpv[g] + j) & 1u)) {
                                tc_fence_after();
                                issue_pv(g, j);
                                used(j);
                                npv[g]++;
                                progress = true;
                            }
                        }
                    }
                    if (progress) {
                        t_last = globaltimer();
                    } else {
                        // nothing ready: poll again (non-blocking checks only; a
                        // suspended try_wait resumes too late here)
                        if ((spin & 255) == 0) {
                            if (s_abort) ok = false;
                            else if (globaltimer() - t_last > WAIT_NS) {
                                s_abort = 1;
                                set_status(status, GPT2_STATUS_TIMEOUT);
                                ok = false;
                            }
                        }
                    }
                }
                if (!ok) break;
                mma_commit(smem_u32(&q_empty[qb]));    // the item's S products have read Q
                cs[0] += n[0];
                cs[1] += n[1];
                cpv[0] += n[0];
                cpv[1] += n[1];
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
        const uint32_t t_s = tmem + lane_base + g * F_BK, t_o = tmem + lane_base + 2 * F_BK + g * HS;
        const uint32_t t_p = tmem + lane_base + 2 * F_BK + 2 * HS + g * 64;
        const uint64_t sc2 = f2pack(scale_log2, scale_log2);
        bool ok = true;
        int cs = 0, cpv = 0;                           // S tiles read and PV products waited for, so far
        for (int it = blockIdx.x; it < nitems && ok; it += gridDim.x) {
            const FwdItem w = fwd_item(it, B, T, H);
            const int row = w.qrow0 + 128 * g + r;
            const int n = g == 0 ? w.nkv0 : w.nkv1;
            float m_run = -INFINITY;                   // log2-domain maximum in use
            uint64_t l2 = f2pack(0.f, 0.f);            // this row's sum of P, two partial lanes
            const uint32_t* brow = nullptr;
            if constexpr (DROP)
                if (row < T) brow = bits + (((size_t)w.b * H + w.h) * T + row) * (size_t)((T + 31) >> 5);
            for (int j = 0; j < n; j++) {
                uint32_t keep_w[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
                if constexpr (DROP) {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const int kw = j * F_BK + 32 * q;
                        keep_w[q] = brow && kw < T ? __ldg(brow + (kw >> 5)) : 0u;
                    }
                }
                if (!mbar_wait(smem_u32(&s_full[g]), (uint32_t)(cs + j) & 1u, &s_abort, status)) { ok = false; break; }
                tc_fence_after();
                float sv[128];
                tmem_ld128(t_s, sv);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s_free[g]));   // the next S_g may be computed now
                // mask: the diagonal tile and the sequence end
                const int k0 = j * F_BK;
                if (k0 + F_BK - 1 > row || k0 + F_BK > T) {
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
                // O_g and the P_g columns are free once the previous PV_g has completed
                // (at j = 0 the previous item's epilogue waited for it)
                if (j > 0) {
                    if (!mbar_wait(smem_u32(&pv_done[g]), (uint32_t)(cpv + j - 1) & 1u, &s_abort, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
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
                    tmem_wait_st();
                }
                if constexpr (DROP) {
#pragma unroll
                    for (int c = 0; c < 128; c++)
                        if (!((keep_w[c >> 5] >> (c & 31)) & 1u)) sv[c] = 0.f;
                }
                // the P row as bf16 pairs into the P_g columns
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 32; c++) pk[c] = pack_bf16(sv[64 * hh + 2 * c], sv[64 * hh + 2 * c + 1]);
                    tmem_st32u(t_p + 32 * hh, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&p_full[g]));
            }
            if (!ok || n == 0) continue;
            if (!mbar_wait(smem_u32(&pv_done[g]), (uint32_t)(cpv + n - 1) & 1u, &s_abort, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            cs += n;
            cpv += n;
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
                const float inv = (DROP ? ks : 1.f) / l;
                uint4* yr = reinterpret_cast<uint4*>(y + ((size_t)w.b * T + row) * C + w.h * HS);
#pragma unroll
                for (int c = 0; c < 8; c++)
                    yr[c] = make_uint4(pack_bf16(o[8 * c] * inv, o[8 * c + 1] * inv),
                                       pack_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                       pack_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                       pack_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
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
        tmem_dealloc(tmem, F_TMEM_COLS);
    }
}

// ---------------------------------------------------------------- backward
// With c = 1/sqrt(hs), lse the forward's row log-sum-exp and D_i = dO_i . O_i:
//   P = exp(c Q K^T - lse),  dP = dO V^T,  dS = P o (dP - D),
//   dQ = c dS K,  dK = c dS^T Q,  dV = P^T dO.
// Two kernels, each output row owned by one CTA (no atomics, deterministic):
//   attn_bwd_dkv_tc05  one CTA per 128-key tile; TMEM lanes are keys.  Per
//       64-query tile (from the diagonal on): S^T = K Q^T and dP^T = V dO^T,
//       then P^T and dS^T as bf16 operand tiles, then dV += P^T dO and
//       dK += dS^T Q.  The Q and dO tiles serve as K-major operands of the
//       first two products and as MN-major operands of the last two.
//   attn_bwd_dq_tc05   one CTA per 128-query tile; TMEM lanes are queries.  Per
//       64-key tile: S = Q K^T and dP = dO V^T, then dS, then dQ += dS K.
// Both follow the forward's roles: a TMA warp, one MMA-issuing thread, eight
// warps on the element-wise work (one row per thread, two warps per row with
// 32 of the tile's 64 columns each; no row reduction is needed here, since lse
// and D come from the forward and the D kernel).

constexpr uint32_t BOX_BYTES = 64 * HS * 2;        // one 64-row tile of a head: 8 KB

// dK, dV for 128 keys.  Shared memory: K | V (16 KB each) | two stages of
// Q, dO (8 KB each) and the tile's lse and D | P^T, dS^T (16 KB each).  TMEM:
// S^T | dP^T | dV | dK.  The producer warp writes each query tile's lse and D
// into the stage before it arms the stage's barrier, so the element-wise
// warps need no barrier of their own.
constexpr int DKV_STAGES = 2;
// a stage: Q box | dO box | lse*log2(e) [64] | D [64], padded to 1 KB
constexpr uint32_t DKV_OFF_K = 0, DKV_OFF_V = 16384, DKV_OFF_ST = 32768, DKV_ROWS = 2 * BOX_BYTES,
                   DKV_STAGE = 2 * BOX_BYTES + 1024, DKV_OFF_P = DKV_OFF_ST + DKV_STAGES * DKV_STAGE,
                   DKV_OFF_DS = DKV_OFF_P + 16384, DKV_SMEM_USED = DKV_OFF_DS + 16384;
constexpr size_t DKV_SMEM = DKV_SMEM_USED + 1024;

template <bool DROP>
__global__ void __launch_bounds__(BWD_THREADS, 2)
attn_bwd_dkv_tc05(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                  __nv_bfloat16* __restrict__ dqkv, const float* __restrict__ lse, const float* __restrict__ Dg,
                  int T, int C, int H, float scale, int* status, float* __restrict__ colsum,
                  const uint32_t* __restrict__ bits, float ks) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t k_full, q_full[DKV_STAGES], q_empty[DKV_STAGES], s_full, s_free, p_full,
        pv_done, drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grid (H, B, key tiles): key tile 0 sees every query, so it goes first
    const int kt = blockIdx.z, h = blockIdx.x, b = blockIdx.y;
    const int k0 = kt * 128;
    const int i0 = k0 / 64, nq = (T + 63) / 64;   // query tiles i0 .. nq-1 see these keys
    const int ntile = nq - i0;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&k_full), 1);
        for (int s = 0; s < DKV_STAGES; s++) {
            mbar_init(smem_u32(&q_full[s]), 1);
            mbar_init(smem_u32(&q_empty[s]), 1);
        }
        mbar_init(smem_u32(&s_full), 1);
        mbar_init(smem_u32(&s_free), BWD_EW_WARPS);
        mbar_init(smem_u32(&p_full), BWD_EW_WARPS);
        mbar_init(smem_u32(&pv_done), 1);
        mbar_init(smem_u32(&drain), 1);
        fence_mbar_init();
        prefetch_map(&tq);
        prefetch_map(&tdo);
    }
    if (warp == 1) tmem_alloc(&s_tmem, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ producer (whole warp; lane 0 issues)
        int last_i[DKV_STAGES];
        for (int s = 0; s < DKV_STAGES; s++) last_i[s] = -1;
        bool ok = true;
        const float* lse_bh = lse + ((size_t)b * H + h) * T;
        const float* D_bh = Dg + ((size_t)b * H + h) * T;
        // each lane carries two queries' lse*log2(e) and D, loaded one tile ahead
        float nl[2], nd[2];
        auto fetch_rows = [&](int t) {
            for (int k = 0; k < 2; k++) {
                const int q = (i0 + t) * 64 + lane + 32 * k;
                nl[k] = q < T ? __ldg(lse_bh + q) * LOG2E : INFINITY;
                nd[k] = q < T ? __ldg(D_bh + q) : 0.f;
            }
        };
        fetch_rows(0);
        if (lane == 0) {
            mbar_expect_tx(smem_u32(&k_full), 4 * BOX_BYTES);
            for (int half = 0; half < 2; half++) {
                tma_load_3d(base + DKV_OFF_K + half * BOX_BYTES, &tq, C + h * HS, k0 + 64 * half, b, smem_u32(&k_full));
                tma_load_3d(base + DKV_OFF_V + half * BOX_BYTES, &tq, 2 * C + h * HS, k0 + 64 * half, b,
                            smem_u32(&k_full));
            }
        }
        for (int t = 0; t < ntile && ok; t++) {
            const int s = t % DKV_STAGES;
            if (lane == 0)
                ok = mbar_wait(smem_u32(&q_empty[s]), ((uint32_t)(t / DKV_STAGES) & 1u) ^ 1u, &s_abort, status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const uint32_t fb = smem_u32(&q_full[s]);
            if (lane == 0) {
                // copies first; the barrier's phase cannot complete before the arrive below
                last_i[s] = t;
                const uint32_t st = base + DKV_OFF_ST + s * DKV_STAGE;
                tma_load_3d(st, &tq, h * HS, (i0 + t) * 64, b, fb);
                tma_load_3d(st + BOX_BYTES, &tdo, h * HS, (i0 + t) * 64, b, fb);
                if (t + DKV_STAGES < ntile) {          // this stage's next tile, into L2
                    tma_prefetch_l2_3d(&tq, h * HS, (i0 + t + DKV_STAGES) * 64, b);
                    tma_prefetch_l2_3d(&tdo, h * HS, (i0 + t + DKV_STAGES) * 64, b);
                }
            }
            // the tile's lse (as lse*log2 e; +inf past T, which zeroes P) and D
            float* rows = reinterpret_cast<float*>(base_ptr + DKV_OFF_ST + s * DKV_STAGE + DKV_ROWS);
            for (int k = 0; k < 2; k++) {
                rows[lane + 32 * k] = nl[k];
                rows[64 + lane + 32 * k] = nd[k];
            }
            if (t + 1 < ntile) fetch_rows(t + 1);
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(fb, 2 * BOX_BYTES);   // releases the writes above
        }
        if (lane == 0) {
            if (!ok) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(smem_u32(&k_full), 0) && globaltimer() - t0 < WAIT_NS) {
                }
                for (int s = 0; s < DKV_STAGES; s++) {
                    if (last_i[s] < 0) continue;
                    const uint32_t ph = (uint32_t)(last_i[s] / DKV_STAGES) & 1u;
                    const uint64_t t1 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&q_full[s]), ph) && globaltimer() - t1 < WAIT_NS) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = instr_desc(128, 64, false, false, true);   // K Q^T, V dO^T
            const uint32_t id_o = instr_desc(128, HS, false, true, true);    // P^T dO, dS^T Q (MN-major B)
            const uint32_t t_st = tmem, t_dp = tmem + 64, t_dv = tmem + 128, t_dk = tmem + 192;
            if (mbar_wait(smem_u32(&k_full), 0, &s_abort, status)) {
                auto issue_s = [&](int t) {            // S^T = K Q_t^T, dP^T = V dO_t^T
                    const uint32_t st = base + DKV_OFF_ST + (t % DKV_STAGES) * DKV_STAGE;
#pragma unroll
                    for (int k = 0; k < HS / 16; k++) {
                        mma_issue<true>(t_st, smem_desc(base + DKV_OFF_K + k * 32, 16, 1024, LAYOUT_SW128),
                                        smem_desc(st + k * 32, 16, 1024, LAYOUT_SW128), id_s, k > 0 ? 1u : 0u);
                        mma_issue<true>(t_dp, smem_desc(base + DKV_OFF_V + k * 32, 16, 1024, LAYOUT_SW128),
                                        smem_desc(st + BOX_BYTES + k * 32, 16, 1024, LAYOUT_SW128), id_s,
                                        k > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&s_full));
                };
                auto issue_o = [&](int t) {            // dV += P^T dO_t, dK += dS^T Q_t (B read MN-major)
                    const uint32_t st = base + DKV_OFF_ST + (t % DKV_STAGES) * DKV_STAGE;
#pragma unroll
                    for (int k = 0; k < 64 / 16; k++) {
                        mma_issue<true>(t_dv, smem_desc(base + DKV_OFF_P + k * 32, 16, 1024, LAYOUT_SW128),
                                        smem_desc(st + BOX_BYTES + k * 16 * 128, 8192, 1024, LAYOUT_SW128), id_o,
                                        (t > 0 || k > 0) ? 1u : 0u);
                        mma_issue<true>(t_dk, smem_desc(base + DKV_OFF_DS + k * 32, 16, 1024, LAYOUT_SW128),
                                        smem_desc(st + k * 16 * 128, 8192, 1024, LAYOUT_SW128), id_o,
                                        (t > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&pv_done));
                    mma_commit(smem_u32(&q_empty[t % DKV_STAGES]));
                };
                mma_two_group_loop(ntile, q_full, DKV_STAGES, &s_free, 1, &p_full, 1, &s_abort, status, issue_s, issue_o);
            }
            mma_commit(smem_u32(&drain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(&drain), 0) && globaltimer() - t0 < WAIT_NS) {
            }
        }
    } else {
        // ------------------------------------------------ element-wise (warps 2..9), thread = key
        // warps w and w + 4 share a TMEM lane quarter; each takes 32 of the
        // tile's 64 query columns
        const int quarter = warp & 3, half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const int key = k0 + r;
        const uint32_t lane_base = ((uint32_t)(quarter * 32) << 16) + (uint32_t)(32 * half);
        const uint32_t t_st = tmem + lane_base, t_dp = t_st + 64, t_dv = t_st + 128, t_dk = t_st + 192;
        const float c2 = scale * LOG2E;
        uint8_t* const prow = base_ptr + DKV_OFF_P;
        uint8_t* const dsrow = base_ptr + DKV_OFF_DS;
        bool ok = true;
        // dropout: keep bits are stored by query row (one word per 32 keys); lane
        // c loads the word of query q0 + c that holds this warp's 32 keys, and a
        // ballot per key turns the 32 words around so that bit c of keep_t is
        // the flag of (query q0 + c, this thread's key)
        const int W = (T + 31) >> 5, kw = (k0 + quarter * 32) >> 5;
        const uint32_t* bits_bh = nullptr;
        if constexpr (DROP) bits_bh = bits + ((size_t)b * H + h) * T * (size_t)W;
        for (int t = 0; t < ntile; t++) {
            uint32_t keep_q = 0u;
            if constexpr (DROP) {
                const int qq = (i0 + t) * 64 + 32 * half + lane;
                keep_q = qq < T && kw < W ? __ldg(bits_bh + (size_t)qq * W + kw) : 0u;
            }
            // S^T and dP^T ready implies the stage (with lse and D) is full
            if (!mbar_wait(smem_u32(&s_full), (uint32_t)t & 1u, &s_abort, status)) { ok = false; break; }
            tc_fence_after();
            float sv[32], dp[32];
            tmem_ld32(t_st, sv);
            tmem_ld32(t_dp, dp);
            tmem_wait_ld(sv);
            tmem_wait_ld(dp);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s_free));
            const int q0 = (i0 + t) * 64 + 32 * half;  // first query of this warp's columns
            // acquire the producer's lse and D writes from the stage barrier itself
            // (its phase for this tile completed before S^T was computed)
            if (!mbar_wait(smem_u32(&q_full[t % DKV_STAGES]), (uint32_t)(t / DKV_STAGES) & 1u, &s_abort, status)) {
                ok = false;
                break;
            }
            const float* rows = reinterpret_cast<const float*>(base_ptr + DKV_OFF_ST + (t % DKV_STAGES) * DKV_STAGE +
                                                               DKV_ROWS) + 32 * half;
            const float4* l4 = reinterpret_cast<const float4*>(rows);
            const float4* d4 = reinterpret_cast<const float4*>(rows + 64);
            const bool diag = q0 < k0 + 127;           // some query of these columns precedes some key
            uint32_t keep_t = 0xffffffffu;
            if constexpr (DROP) {
#pragma unroll
                for (int kl = 0; kl < 32; kl++) {
                    const uint32_t v = __ballot_sync(0xffffffffu, (keep_q >> kl) & 1u);
                    if (lane == kl) keep_t = v;
                }
            }
#pragma unroll
            for (int c4 = 0; c4 < 8; c4++) {
                const float4 lv = l4[c4], dv = d4[c4];
                const float lq[4] = {lv.x, lv.y, lv.z, lv.w}, dq[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int c = 4 * c4 + e;
                    float pv = ex2(fmaf(sv[c], c2, -lq[e]));
                    if (diag && q0 + c < key) pv = 0.f;
                    if constexpr (DROP) {
                        // dV takes the dropped weight; dP passes the same mask
                        const bool kept = (keep_t >> c) & 1u;
                        sv[c] = kept ? pv * ks : 0.f;
                        dp[c] = pv * ((kept ? dp[c] * ks : 0.f) - dq[e]);
                    } else {
                        sv[c] = pv;
                        dp[c] = pv * (dp[c] - dq[e]);
                    }
                }
            }
            // P^T and dS^T buffers are free once the previous tile's products completed
            if (t > 0) {
                if (!mbar_wait(smem_u32(&pv_done), (uint32_t)(t - 1) & 1u, &s_abort, status)) { ok = false; break; }
                tc_fence_after();
            }
#pragma unroll
            for (int c = 0; c < 4; c++) {
                *reinterpret_cast<uint4*>(prow + sw128(r, 4 * half + c)) =
                    make_uint4(pack_bf16(sv[8 * c], sv[8 * c + 1]), pack_bf16(sv[8 * c + 2], sv[8 * c + 3]),
                               pack_bf16(sv[8 * c + 4], sv[8 * c + 5]), pack_bf16(sv[8 * c + 6], sv[8 * c + 7]));
                *reinterpret_cast<uint4*>(dsrow + sw128(r, 4 * half + c)) =
                    make_uint4(pack_bf16(dp[8 * c], dp[8 * c + 1]), pack_bf16(dp[8 * c + 2], dp[8 * c + 3]),
                               pack_bf16(dp[8 * c + 4], dp[8 * c + 5]), pack_bf16(dp[8 * c + 6], dp[8 * c + 7]));
            }
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&p_full));
        }
        if (ok && mbar_wait(smem_u32(&pv_done), (uint32_t)(ntile - 1) & 1u, &s_abort, status)) {
            tc_fence_after();
            for (int which = 0; which < 2; which++) {  // 0: dK (scaled by c), 1: dV
                float o[32];
                tmem_ld32(which == 0 ? t_dk : t_dv, o);
                tmem_wait_ld(o);
                const float f = which == 0 ? scale : 1.f;
#pragma unroll
                for (int c = 0; c < 32; c++) o[c] = key < T ? o[c] * f : 0.f;
                const int col0 = (1 + which) * C + h * HS + 32 * half;
                if (key < T) {
                    uint4* dst = reinterpret_cast<uint4*>(dqkv + ((size_t)b * T + key) * 3 * C + col0);
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        dst[c] = make_uint4(pack_bf16(o[8 * c], o[8 * c + 1]), pack_bf16(o[8 * c + 2], o[8 * c + 3]),
                                            pack_bf16(o[8 * c + 4], o[8 * c + 5]), pack_bf16(o[8 * c + 6], o[8 * c + 7]));
                }
                if (colsum) store_colsum(colsum, o, lane, b, k0 + quarter * 32, T, C, col0);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// dQ for 128 queries.  Shared memory: Q | dO (16 KB each) | three stages of
// K, V (8 KB each) | dS (16 KB).  TMEM: S | dP | dQ.
constexpr int DQ_STAGES = 3;
constexpr uint32_t DQ_OFF_Q = 0, DQ_OFF_DO = 16384, DQ_OFF_ST = 32768, DQ_STAGE = 2 * BOX_BYTES,
                   DQ_OFF_DS = DQ_OFF_ST + DQ_STAGES * DQ_STAGE, DQ_SMEM_USED = DQ_OFF_DS + 16384;
constexpr size_t DQ_SMEM = DQ_SMEM_USED + 1024;

template <bool DROP>
__global__ void __launch_bounds__(BWD_THREADS, 2)
attn_bwd_dq_tc05(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                 __nv_bfloat16* __restrict__ dqkv, const float* __restrict__ lse, const float* __restrict__ Dg,
                 int T, int C, int H, float scale, int* status, float* __restrict__ colsum,
                 const uint32_t* __restrict__ bits, float ks) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full, kv_full[DQ_STAGES], kv_empty[DQ_STAGES], s_full, s_free, p_full,
        pv_done, drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nqt = (T + BQ - 1) / BQ;
    const int qt = nqt - 1 - (int)blockIdx.z;         // grid (H, B, query tiles): longest first
    const int h = blockIdx.x, b = blockIdx.y;
    const int q0 = qt * BQ;
    const int nkv = (min(q0 + BQ, T) + 63) / 64;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&q_full), 1);
        for (int s = 0; s < DQ_STAGES; s++) {
            mbar_init(smem_u32(&kv_full[s]), 1);
            mbar_init(smem_u32(&kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&s_full), 1);
        mbar_init(smem_u32(&s_free), BWD_EW_WARPS);
        mbar_init(smem_u32(&p_full), BWD_EW_WARPS);
        mbar_init(smem_u32(&pv_done), 1);
        mbar_init(smem_u32(&drain), 1);
        fence_mbar_init();
        prefetch_map(&tq);
        prefetch_map(&tdo);
    }
    if (warp == 1) tmem_alloc(&s_tmem, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_j[DQ_STAGES];
            for (int s = 0; s < DQ_STAGES; s++) last_j[s] = -1;
            bool ok = true;
            mbar_expect_tx(smem_u32(&q_full), 4 * BOX_BYTES);
            for (int half = 0; half < 2; half++) {
                tma_load_3d(base + DQ_OFF_Q + half * BOX_BYTES, &tq, h * HS, q0 + 64 * half, b, smem_u32(&q_full));
                tma_load_3d(base + DQ_OFF_DO + half * BOX_BYTES, &tdo, h * HS, q0 + 64 * half, b, smem_u32(&q_full));
            }
            for (int j = 0; j < nkv && ok; j++) {
                const int s = j % DQ_STAGES;
                if (!mbar_wait(smem_u32(&kv_empty[s]), ((uint32_t)(j / DQ_STAGES) & 1u) ^ 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&kv_full[s]);
                mbar_expect_tx(fb, 2 * BOX_BYTES);
                last_j[s] = j;
                const uint32_t st = base + DQ_OFF_ST + s * DQ_STAGE;
                tma_load_3d(st, &tq, C + h * HS, j * 64, b, fb);
                tma_load_3d(st + BOX_BYTES, &tq, 2 * C + h * HS, j * 64, b, fb);
                if (j + DQ_STAGES < nkv) {             // this stage's next tile, into L2
                    tma_prefetch_l2_3d(&tq, C + h * HS, (j + DQ_STAGES) * 64, b);
                    tma_prefetch_l2_3d(&tq, 2 * C + h * HS, (j + DQ_STAGES) * 64, b);
                }
            }
            if (!ok) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(smem_u32(&q_full), 0) && globaltimer() - t0 < WAIT_NS) {
                }
                for (int s = 0; s < DQ_STAGES; s++) {
                    if (last_j[s] < 0) continue;
                    const uint32_t ph = (uint32_t)(last_j[s] / DQ_STAGES) & 1u;
                    const uint64_t t1 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&kv_full[s]), ph) && globaltimer() - t1 < WAIT_NS) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = instr_desc(BQ, 64, false, false, true);   // Q K^T, dO V^T
            const uint32_t id_o = instr_desc(BQ, HS, false, true, true);    // dS K (K read MN-major)
            const uint32_t t_s = tmem, t_dp = tmem + 64, t_dq = tmem + 128;
            if (mbar_wait(smem_u32(&q_full), 0, &s_abort, status)) {
                auto issue_s = [&](int j) {            // S = Q K_j^T, dP = dO V_j^T
                    const uint32_t st = base + DQ_OFF_ST + (j % DQ_STAGES) * DQ_STAGE;
#pragma unroll
                    for (int k = 0; k < HS / 16; k++) {
                        mma_issue<true>(t_s, smem_desc(base + DQ_OFF_Q + k * 32, 16, 1024, LAYOUT_SW128),
                                        smem_desc(st + k * 32, 16, 1024, LAYOUT_SW128), id_s, k > 0 ? 1u : 0u);
                        mma_issue<true>(t_dp, smem_desc(base + DQ_OFF_DO + k * 32, 16, 1024, LAYOUT_SW128),
                                        smem_desc(st + BOX_BYTES + k * 32, 16, 1024, LAYOUT_SW128), id_s,
                                        k > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&s_full));
                };
                auto issue_o = [&](int j) {            // dQ += dS K_j (K read MN-major)
                    const uint32_t st = base + DQ_OFF_ST + (j % DQ_STAGES) * DQ_STAGE;
#pragma unroll
                    for (int k = 0; k < 64 / 16; k++)
                        mma_issue<true>(t_dq, smem_desc(base + DQ_OFF_DS + k * 32, 16, 1024, LAYOUT_SW128),
                                        smem_desc(st + k * 16 * 128, 8192, 1024, LAYOUT_SW128), id_o,
                                        (j > 0 || k > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&pv_done));
                    mma_commit(smem_u32(&kv_empty[j % DQ_STAGES]));
                };
                mma_two_group_loop(nkv, kv_full, DQ_STAGES, &s_free, 1, &p_full, 1, &s_abort, status, issue_s, issue_o);
            }
            mma_commit(smem_u32(&drain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(&drain), 0) && globaltimer() - t0 < WAIT_NS) {
            }
        }
    } else {
        // ------------------------------------------------ element-wise (warps 2..9), thread = query
        // warps w and w + 4 share a TMEM lane quarter; each takes 32 of the
        // tile's 64 key columns
        const int quarter = warp & 3, half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        const int row = q0 + r;
        const uint32_t lane_base = ((uint32_t)(quarter * 32) << 16) + (uint32_t)(32 * half);
        const uint32_t t_s = tmem + lane_base, t_dp = t_s + 64, t_dq = t_s + 128;
        const float c2 = scale * LOG2E;
        const size_t bh = ((size_t)b * H + h) * T;
        const float lse2 = row < T ? lse[bh + row] * LOG2E : INFINITY;
        const float Drow = row < T ? Dg[bh + row] : 0.f;
        uint8_t* const dsrow = base_ptr + DQ_OFF_DS;
        bool ok = true;
        const uint32_t* brow = nullptr;
        if constexpr (DROP)
            if (row < T) brow = bits + (bh + row) * (size_t)((T + 31) >> 5);
        for (int j = 0; j < nkv; j++) {
            uint32_t keep_w = 0xffffffffu;
            if constexpr (DROP) {
                const int kw = j * 64 + 32 * half;
                keep_w = brow && kw < T ? __ldg(brow + (kw >> 5)) : 0u;
            }
            if (!mbar_wait(smem_u32(&s_full), (uint32_t)j & 1u, &s_abort, status)) { ok = false; break; }
            tc_fence_after();
            float sv[32], dp[32];
            tmem_ld32(t_s, sv);
            tmem_ld32(t_dp, dp);
            tmem_wait_ld(sv);
            tmem_wait_ld(dp);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s_free));
            const int k0 = j * 64 + 32 * half;        // first key of this warp's columns
            const bool diag = k0 + 31 > q0;            // some key of these columns follows some query
#pragma unroll
            for (int c = 0; c < 32; c++) {
                float pv = ex2(fmaf(sv[c], c2, -lse2));
                if (diag && (k0 + c > row || k0 + c >= T)) pv = 0.f;
                if constexpr (DROP) dp[c] = pv * ((((keep_w >> c) & 1u) ? dp[c] * ks : 0.f) - Drow);
                else dp[c] = pv * (dp[c] - Drow);
            }
            if (j > 0) {
                if (!mbar_wait(smem_u32(&pv_done), (uint32_t)(j - 1) & 1u, &s_abort, status)) { ok = false; break; }
                tc_fence_after();
            }
#pragma unroll
            for (int c = 0; c < 4; c++)
                *reinterpret_cast<uint4*>(dsrow + sw128(r, 4 * half + c)) =
                    make_uint4(pack_bf16(dp[8 * c], dp[8 * c + 1]), pack_bf16(dp[8 * c + 2], dp[8 * c + 3]),
                               pack_bf16(dp[8 * c + 4], dp[8 * c + 5]), pack_bf16(dp[8 * c + 6], dp[8 * c + 7]));
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&p_full));
        }
        if (ok && mbar_wait(smem_u32(&pv_done), (uint32_t)(nkv - 1) & 1u, &s_abort, status)) {
            tc_fence_after();
            float o[32];
            tmem_ld32(t_dq, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int c = 0; c < 32; c++) o[c] = row < T ? o[c] * scale : 0.f;
            const int col0 = h * HS + 32 * half;
            if (row < T) {
                uint4* dst = reinterpret_cast<uint4*>(dqkv + ((size_t)b * T + row) * 3 * C + col0);
#pragma unroll
                for (int c = 0; c < 4; c++)
                    dst[c] = make_uint4(pack_bf16(o[8 * c], o[8 * c + 1]), pack_bf16(o[8 * c + 2], o[8 * c + 3]),
                                        pack_bf16(o[8 * c + 4], o[8 * c + 5]), pack_bf16(o[8 * c + 6], o[8 * c + 7]));
            }
            if (colsum) store_colsum(colsum, o, lane, b, q0 + quarter * 32, T, C, col0);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace at05

bool attention_tc05_supported(int hs, int C) { return hs == at05::HS && C % 8 == 0; }

// y [B,T,C] and lse [B,H,T] from qkv [B,T,3C] (bf16), head size 64.
// With bits != null: dropout on the attention weights (keep bits by query row,
// one word per 32 keys), kept weights scaled by ks.
int attention_tc05_forward(void* y, float* lse, const void* qkv, int B, int T, int C, int H, int* status,
                           cudaStream_t st, const uint32_t* bits, float ks) {
    using namespace at05;
    if (C / H != HS || C % H || !attention_tc05_supported(HS, C)) return GPT2_ENOTSUP;
    if (smem_limit(reinterpret_cast<const void*>(attn_fwd_tc05<false>), (int)F_SMEM) ||
        smem_limit(reinterpret_cast<const void*>(attn_fwd_tc05<true>), (int)F_SMEM))
        return GPT2_ECUDA;
    // qkv as a 3-D tensor [B][T][3C]: boxes of 64 rows x 64 columns (one head)
    CUtensorMap tm;
    const cuuint64_t dims[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)3 * C * 2, (cuuint64_t)T * 3 * C * 2};
    const cuuint32_t box[3] = {HS, 64, 1};
    if (!encode_tensor_map(&tm, true, 3, qkv, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return GPT2_ENOTSUP;
    const float scale_log2 = LOG2E / sqrtf((float)HS);
    const int nitems = fwd_items(B, T, H);
    const dim3 grid(std::min(nitems, num_sms()));
    if (bits)
        count_launch(), attn_fwd_tc05<true><<<grid, F_THREADS, F_SMEM, st>>>(
            tm, static_cast<__nv_bfloat16*>(y), lse, B, T, C, H, scale_log2, status, bits, ks);
    else
        count_launch(), attn_fwd_tc05<false><<<grid, F_THREADS, F_SMEM, st>>>(
            tm, static_cast<__nv_bfloat16*>(y), lse, B, T, C, H, scale_log2, status, nullptr, 1.f);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k

namespace gpt2k {

// dqkv [B,T,3C] (bf16, every element written) from dy [B,T,C], qkv, the
// forward's lse [B,H,T] and D [B,H,T] = rowsum(dO o O); head size 64.  With
// colsum != null also the column sums of dqkv per 32-row group
// ([B * ceil(T/32), 3C], fp32, before bf16 rounding).
int attention_tc05_backward(void* dqkv, const void* dy, const void* qkv, const float* lse, const float* D,
                            int B, int T, int C, int H, int* status, cudaStream_t st, float* colsum,
                            const uint32_t* bits, float ks) {
    using namespace at05;
    if (C / H != HS || C % H || !attention_tc05_supported(HS, C)) return GPT2_ENOTSUP;
    if (smem_limit(reinterpret_cast<const void*>(attn_bwd_dkv_tc05<false>), (int)DKV_SMEM) ||
        smem_limit(reinterpret_cast<const void*>(attn_bwd_dkv_tc05<true>), (int)DKV_SMEM) ||
        smem_limit(reinterpret_cast<const void*>(attn_bwd_dq_tc05<false>), (int)DQ_SMEM) ||
        smem_limit(reinterpret_cast<const void*>(attn_bwd_dq_tc05<true>), (int)DQ_SMEM))
        return GPT2_ECUDA;
    CUtensorMap tq, tdo;
    const cuuint64_t dq_[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t sq_[2] = {(cuuint64_t)3 * C * 2, (cuuint64_t)T * 3 * C * 2};
    const cuuint64_t dd_[3] = {(cuuint64_t)C, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t sd_[2] = {(cuuint64_t)C * 2, (cuuint64_t)T * C * 2};
    const cuuint32_t box[3] = {HS, 64, 1};
    if (!encode_tensor_map(&tq, true, 3, qkv, dq_, sq_, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&tdo, true, 3, dy, dd_, sd_, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return GPT2_ENOTSUP;
    const float scale = 1.f / sqrtf((float)HS);
    auto* out = static_cast<__nv_bfloat16*>(dqkv);
    const dim3 gk(H, B, (T + 127) / 128), gq(H, B, (T + BQ - 1) / BQ);
    if (bits) {
        count_launch(), attn_bwd_dkv_tc05<true><<<gk, BWD_THREADS, DKV_SMEM, st>>>(tq, tdo, out, lse, D, T, C, H, scale,
                                                                                 status, colsum, bits, ks);
        count_launch(), attn_bwd_dq_tc05<true><<<gq, BWD_THREADS, DQ_SMEM, st>>>(tq, tdo, out, lse, D, T, C, H, scale,
                                                                               status, colsum, bits, ks);
    } else {
        count_launch(), attn_bwd_dkv_tc05<false><<<gk, BWD_THREADS, DKV_SMEM, st>>>(tq, tdo, out, lse, D, T, C, H,
                                                                                  scale, status, colsum, nullptr, 1.f);
        count_launch(), attn_bwd_dq_tc05<false><<<gq, BWD_THREADS, DQ_SMEM, st>>>(tq, tdo, out, lse, D, T, C, H,
                                                                                scale, status, colsum, nullptr, 1.f);
    }
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k
