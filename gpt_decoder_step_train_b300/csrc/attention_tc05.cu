// attention_tc05.cu -- causal self-attention forward on the 5th-generation
// tensor cores (tcgen05), bf16 operands, head size 64.
//
// Per (batch b, head h): S = Q K^T / sqrt(hs), S[i,j] = -inf for j > i,
// P = softmax_rows(S), O = P V, and the row log-sum-exp of the scaled scores
// is kept for the backward ("GPT-2 from scratch with torch", section
// 自注意力; the 1/sqrt(d_k) scaling: "从头搭建GPT(Andrej Karpathy) 笔记",
// section attention中为什么要做scaling).
//
// One CTA per (query tile of 128 rows, head, batch), 320 threads, two CTAs per SM:
//   warp 0   TMA producer: the Q tile once, then K and V tiles of 64 keys
//            into a three-stage ring (128-byte swizzle);
//   warp 1   allocates tensor memory (S: two buffers of 64 columns, O: 64
//            columns) and from one lane issues S = Q K^T (M=128, N=64, K=64) and O += P V
//            (M=128, N=64, K=64; P from shared memory, V read MN-major);
//   warps 2-9  softmax, one query row per thread (its TMEM lane), two warps
//            per row (32 key columns each, the row maximum combined through
//            shared memory): scores from tensor memory, causal mask on the
//            diagonal tiles, online maximum and sum in the log2 domain, P
//            written to shared memory as bf16 in the operand layout.  The running maximum used for P is
//            only moved when a row's true maximum exceeds it by more than
//            2^8; O in tensor memory is then rescaled before the next P V.
//            At the end O / l goes out as bf16 and the log-sum-exp as fp32.
// Key tiles past the query tile's last row are never visited (causal tile
// skipping).  While the softmax warps work on S_j, the tensor cores compute
// S_{j+1} into the other score buffer and P_{j-1} V_{j-1} (P is double-buffered
// in shared memory too), so the softmax warps wait on the tensor cores only
// when O must be rescaled.
// Every wait is bounded (about one second); a wait that gives up raises
// GPT2_STATUS_TIMEOUT, all roles leave, in-flight copies and MMAs are drained
// and tensor memory is freed.
#include <cuda_bf16.h>

#include "common.cuh"
#include "gemm.cuh"
#include "ptx.cuh"

namespace gpt2k {
namespace at05 {

using namespace ptx;

constexpr int HS = 64;              // head size (one 128-byte swizzle row of bf16)
constexpr int BQ = 128;             // queries per CTA (TMEM lanes)
constexpr int BKV = 64;             // keys per tile
constexpr int KV_STAGES = 3;
// forward: producer, MMA issuer and eight softmax warps (two per TMEM lane
// quarter, one per half of the key tile's columns)
constexpr int FWD_EW_WARPS = 8;
constexpr int FWD_THREADS = 64 + 32 * FWD_EW_WARPS;
// backward kernels: producer, MMA issuer and eight element-wise warps (two per
// TMEM lane quarter, one per half of the tile's 64 columns)
constexpr int BWD_EW_WARPS = 8;
constexpr int BWD_THREADS = 64 + 32 * BWD_EW_WARPS;
constexpr int TMEM_COLS = 256;      // S (two buffers): [0, 64), [64, 128); O: [128, 192)
constexpr uint32_t TILE_BYTES = BKV * HS * 2;     // one K or V tile: 8 KB
constexpr uint32_t Q_BYTES = BQ * HS * 2;         // 16 KB
constexpr uint32_t P_BYTES = BQ * BKV * 2;        // 16 KB
// shared memory: Q | K[2] | V[2] | P, each 1024-byte aligned
constexpr uint32_t OFF_Q = 0, OFF_K = OFF_Q + Q_BYTES, OFF_V = OFF_K + KV_STAGES * TILE_BYTES,
                   OFF_P = OFF_V + KV_STAGES * TILE_BYTES, SMEM_USED = OFF_P + 2 * P_BYTES;
constexpr size_t SMEM = SMEM_USED + 1024;          // + alignment slack
constexpr float RESCALE_LOG2 = 8.f;                // move the running maximum past 2^8 growth
constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;

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

template <bool DROP>
__global__ void __launch_bounds__(FWD_THREADS, 2)
attn_fwd_tc05(const __grid_constant__ CUtensorMap tm, __nv_bfloat16* __restrict__ y, float* __restrict__ lse,
              int T, int C, int H, float scale_log2, int* status, const uint32_t* __restrict__ bits, float ks) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full, kv_full[KV_STAGES], kv_empty[KV_STAGES], s_full[2], s_free[2], p_full[2],
        pv_done[2], drain;
    __shared__ __align__(8) uint64_t pair_bar[4][2];
    __shared__ float pair_val[2][2][BQ];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nq = (T + BQ - 1) / BQ;
    // grid (H, B, query tiles): every head's longest tile is launched first
    const int qt = nq - 1 - (int)blockIdx.z;
    const int h = blockIdx.x, b = blockIdx.y;
    const int q0 = qt * BQ;
    const int nkv = (min(q0 + BQ, T) + BKV - 1) / BKV;  // key tiles that hold keys <= the last row
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);

    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&q_full), 1);
        for (int s = 0; s < KV_STAGES; s++) {
            mbar_init(smem_u32(&kv_full[s]), 1);
            mbar_init(smem_u32(&kv_empty[s]), 1);
        }
        for (int k = 0; k < 2; k++) {
            mbar_init(smem_u32(&s_full[k]), 1);
            mbar_init(smem_u32(&s_free[k]), FWD_EW_WARPS);
        }
        for (int k = 0; k < 2; k++) {
            mbar_init(smem_u32(&p_full[k]), FWD_EW_WARPS);
            mbar_init(smem_u32(&pv_done[k]), 1);
        }
        for (int q = 0; q < 4; q++)
            for (int k = 0; k < 2; k++) mbar_init(smem_u32(&pair_bar[q][k]), 2);
        mbar_init(smem_u32(&drain), 1);
        fence_mbar_init();
        prefetch_map(&tm);
    }
    if (warp == 1) tmem_alloc(&s_tmem, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int last_j[KV_STAGES];                     // last tile issued into each stage (abort drain)
            for (int s = 0; s < KV_STAGES; s++) last_j[s] = -1;
            bool ok = true;
            mbar_expect_tx(smem_u32(&q_full), Q_BYTES);
            tma_load_3d(base + OFF_Q, &tm, h * HS, q0, b, smem_u32(&q_full));
            tma_load_3d(base + OFF_Q + Q_BYTES / 2, &tm, h * HS, q0 + 64, b, smem_u32(&q_full));
            for (int j = 0; j < nkv && ok; j++) {
                const int s = j % KV_STAGES;
                const uint32_t ph = (uint32_t)(j / KV_STAGES) & 1u;
                if (!mbar_wait(smem_u32(&kv_empty[s]), ph ^ 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(&kv_full[s]);
                mbar_expect_tx(fb, 2 * TILE_BYTES);
                last_j[s] = j;
                tma_load_3d(base + OFF_K + s * TILE_BYTES, &tm, C + h * HS, j * BKV, b, fb);
                tma_load_3d(base + OFF_V + s * TILE_BYTES, &tm, 2 * C + h * HS, j * BKV, b, fb);
                if (j + KV_STAGES < nkv) {             // this stage's next tile, into L2
                    tma_prefetch_l2_3d(&tm, C + h * HS, (j + KV_STAGES) * BKV, b);
                    tma_prefetch_l2_3d(&tm, 2 * C + h * HS, (j + KV_STAGES) * BKV, b);
                }
            }
            if (!ok) {
                // wait (bounded, ignoring the abort flag) for every copy this thread issued
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(smem_u32(&q_full), 0) && globaltimer() - t0 < WAIT_NS) {
                }
                // earlier copies into a stage completed before it was refilled, so
                // only each stage's last issue can still be in flight
                for (int s = 0; s < KV_STAGES; s++) {
                    if (last_j[s] < 0) continue;
                    const uint32_t ph = (uint32_t)(last_j[s] / KV_STAGES) & 1u;
                    const uint64_t t1 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&kv_full[s]), ph) && globaltimer() - t1 < WAIT_NS) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = instr_desc(BQ, BKV, false, false, true);   // Q K^T: both K-major
            const uint32_t id_pv = instr_desc(BQ, HS, false, true, true);    // P V: V MN-major
            const uint32_t t_s = tmem, t_o = tmem + 2 * BKV;   // S_j in columns (j & 1) * 64
            if (mbar_wait(smem_u32(&q_full), 0, &s_abort, status)) {
                auto issue_s = [&](int j) {            // S = Q K_j^T
                    const uint32_t kb = base + OFF_K + (j % KV_STAGES) * TILE_BYTES;
#pragma unroll
                    for (int k = 0; k < HS / 16; k++)
                        mma_issue<true>(t_s + (uint32_t)(j & 1) * BKV, smem_desc(base + OFF_Q + k * 32, 16, 1024, LAYOUT_SW128),
                                        smem_desc(kb + k * 32, 16, 1024, LAYOUT_SW128), id_s, k > 0 ? 1u : 0u);
                    mma_commit(smem_u32(&s_full[j & 1]));
                };
                auto issue_pv = [&](int j) {           // O += P_j V_j (P_j in buffer j & 1)
                    const uint32_t vb = base + OFF_V + (j % KV_STAGES) * TILE_BYTES;
                    const uint32_t pb = base + OFF_P + (uint32_t)(j & 1) * P_BYTES;
#pragma unroll
                    for (int k = 0; k < BKV / 16; k++)
                        mma_issue<true>(t_o, smem_desc(pb + k * 32, 16, 1024, LAYOUT_SW128),
                                        smem_desc(vb + k * 16 * 128, 8192, 1024, LAYOUT_SW128), id_pv,
                                        (j > 0 || k > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&pv_done[j & 1]));
                    mma_commit(smem_u32(&kv_empty[j % KV_STAGES]));
                };
                mma_two_group_loop(nkv, kv_full, KV_STAGES, s_free, 2, p_full, 2, &s_abort, status, issue_s, issue_pv);
            }
            // every MMA issued has completed once this commit lands
            mma_commit(smem_u32(&drain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(&drain), 0) && globaltimer() - t0 < WAIT_NS) {
            }
        }
    } else {
        // ------------------------------------------------ softmax (warps 2..9)
        // warps w and w + 4 share a TMEM lane quarter (32 rows); each takes 32 of
        // the tile's 64 key columns and 32 of O's 64 columns.  The pair combines
        // its row maxima every tile through shared memory and a two-warp
        // mbarrier (double-buffered by tile parity), so both use the same
        // running maximum; each keeps its own part of the row sum.
        const int quarter = warp & 3, half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;             // row within the tile
        const int row = q0 + r;
        const uint32_t lane_base = ((uint32_t)(quarter * 32) << 16) + (uint32_t)(32 * half);
        const uint32_t t_s = tmem + lane_base, t_o = tmem + lane_base + 2 * BKV;
        uint8_t* const pbuf = base_ptr + OFF_P;    // two P buffers, tile j in buffer j & 1
        float m_run = -INFINITY, l_run = 0.f;          // log2-domain maximum in use, this half's sum of P
        bool ok = true;
        // dropout: this row's keep bits, one word per 32 keys
        const uint32_t* brow = nullptr;
        if constexpr (DROP)
            if (row < T) brow = bits + (((size_t)b * H + h) * T + row) * (size_t)((T + 31) >> 5);
        // exchange slot of tile j: pair_val[j & 1][half][r]; barrier pair_bar[quarter][j & 1]
        auto exchange = [&](int j, float v, float* other) -> bool {
            pair_val[j & 1][half][r] = v;
            __syncwarp();
            const uint32_t bar = smem_u32(&pair_bar[quarter][j & 1]);
            if (lane == 0) mbar_arrive(bar);
            if (!mbar_wait(bar, (uint32_t)(j >> 1) & 1u, &s_abort, status)) return false;
            *other = pair_val[j & 1][half ^ 1][r];
            return true;
        };
        for (int j = 0; j < nkv; j++) {
            uint32_t keep_w = 0xffffffffu;
            if constexpr (DROP) {
                const int kw = j * BKV + 32 * half;
                keep_w = brow && kw < T ? __ldg(brow + (kw >> 5)) : 0u;
            }
            if (!mbar_wait(smem_u32(&s_full[j & 1]), (uint32_t)(j >> 1) & 1u, &s_abort, status)) { ok = false; break; }
            tc_fence_after();
            float s[32];
            tmem_ld32(t_s + (uint32_t)(j & 1) * BKV, s);
            tmem_wait_ld(s);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s_free[j & 1]));
            // mask (tiles that reach the diagonal or the sequence end), row maximum
            // of the raw scores; the scale goes into the exponent's FMA
            const int k0 = j * BKV + 32 * half;        // first key of this warp's columns
            if (k0 + 31 > q0 || k0 + 32 > T) {
#pragma unroll
                for (int c = 0; c < 32; c++)
                    if (k0 + c > row || k0 + c >= T) s[c] = -INFINITY;
            }
            float m8[8];
#pragma unroll
            for (int c = 0; c < 8; c++) m8[c] = fmaxf(fmaxf(s[c], s[c + 8]), fmaxf(s[c + 16], s[c + 24]));
            float pm = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            float om;
            if (!exchange(j, pm, &om)) { ok = false; break; }
            const float mx = fmaxf(pm, om) * scale_log2;    // log2-domain maximum of the tile's row
            float alpha = 1.f;                         // factor on O and l for this tile
            if (mx > m_run + RESCALE_LOG2 || (m_run == -INFINITY && mx > -INFINITY)) {
                alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mx);
                m_run = mx;
            }
            const float mref = m_run == -INFINITY ? 0.f : m_run;
            float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 32; c++) {
                s[c] = ex2(fmaf(s[c], scale_log2, -mref));
                ps[c & 3] += s[c];
            }
            l_run = l_run * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
            // dropped weights leave the sum (the softmax normaliser) and miss V
            if constexpr (DROP) {
#pragma unroll
                for (int c = 0; c < 32; c++)
                    if (!((keep_w >> c) & 1u)) s[c] = 0.f;
            }
            // a rescale of O needs every earlier P V complete (the last is P_{j-1} V_{j-1})
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                if (!mbar_wait(smem_u32(&pv_done[(j - 1) & 1]), (uint32_t)((j - 1) >> 1) & 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    float o[32];
                    tmem_ld32(t_o, o);
                    tmem_wait_ld(o);
#pragma unroll
                    for (int c = 0; c < 32; c++) o[c] *= alpha;
                    tmem_st32(t_o, o);
                    tmem_wait_st();
                }
            }
            // buffer j & 1 is free once P_{j-2} V_{j-2} has completed
            if (j > 1) {
                if (!mbar_wait(smem_u32(&pv_done[j & 1]), (uint32_t)((j - 2) >> 1) & 1u, &s_abort, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            uint8_t* const prow = pbuf + (size_t)(j & 1) * P_BYTES;
            // this half of the P row (bf16) into the K-major operand tile
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const uint4 v = make_uint4(pack_bf16(s[8 * c], s[8 * c + 1]), pack_bf16(s[8 * c + 2], s[8 * c + 3]),
                                           pack_bf16(s[8 * c + 4], s[8 * c + 5]),
                                           pack_bf16(s[8 * c + 6], s[8 * c + 7]));
                *reinterpret_cast<uint4*>(prow + sw128(r, 4 * half + c)) = v;
            }
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&p_full[j & 1]));
        }
        // the row sum: this half's part plus the partner's (same order in both warps)
        float l_other = 0.f;
        if (ok && !exchange(nkv, l_run, &l_other)) ok = false;
        if (ok && mbar_wait(smem_u32(&pv_done[(nkv - 1) & 1]), (uint32_t)((nkv - 1) >> 1) & 1u, &s_abort, status)) {
            tc_fence_after();
            float o[32];
            tmem_ld32(t_o, o);
            tmem_wait_ld(o);
            if (row < T) {
                const float l = half == 0 ? l_run + l_other : l_other + l_run;
                const float inv = (DROP ? ks : 1.f) / l;
                uint4* yr = reinterpret_cast<uint4*>(y + ((size_t)b * T + row) * C + h * HS + 32 * half);
#pragma unroll
                for (int c = 0; c < 4; c++)
                    yr[c] = make_uint4(pack_bf16(o[8 * c] * inv, o[8 * c + 1] * inv),
                                       pack_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                       pack_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                       pack_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
                if (half == 0) lse[((size_t)b * H + h) * T + row] = (m_run + log2f(l)) * LN2;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
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
    if (smem_limit(reinterpret_cast<const void*>(attn_fwd_tc05<false>), (int)SMEM) ||
        smem_limit(reinterpret_cast<const void*>(attn_fwd_tc05<true>), (int)SMEM))
        return GPT2_ECUDA;
    // qkv as a 3-D tensor [B][T][3C]: boxes of 64 rows x 64 columns (one head)
    CUtensorMap tm;
    const cuuint64_t dims[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)3 * C * 2, (cuuint64_t)T * 3 * C * 2};
    const cuuint32_t box[3] = {HS, 64, 1};
    if (!encode_tensor_map(&tm, true, 3, qkv, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return GPT2_ENOTSUP;
    const float scale_log2 = LOG2E / sqrtf((float)HS);
    const dim3 grid(H, B, (T + BQ - 1) / BQ);
    if (bits)
        count_launch(), attn_fwd_tc05<true><<<grid, FWD_THREADS, SMEM, st>>>(
            tm, static_cast<__nv_bfloat16*>(y), lse, T, C, H, scale_log2, status, bits, ks);
    else
        count_launch(), attn_fwd_tc05<false><<<grid, FWD_THREADS, SMEM, st>>>(
            tm, static_cast<__nv_bfloat16*>(y), lse, T, C, H, scale_log2, status, nullptr, 1.f);
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
