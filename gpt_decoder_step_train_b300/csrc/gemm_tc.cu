// gemm_tc.cu -- GEMM on the 5th-generation tensor cores (tcgen05), fed by TMA,
// fp32 accumulation in tensor memory.  Two operand types: fp32 storage read as
// tf32 (kind::tf32, K = 8 per MMA) and bf16 (kind::f16, K = 16 per MMA); a
// k-block is one 128-byte swizzle row either way (32 fp32 or 64 bf16).
//
// Persistent, warp-specialised kernel, one CTA per SM, 320 threads:
//   warp 0  TMA producer: fills a ring of shared-memory stages (A: 128 rows,
//           B: BN rows, one 128-byte swizzle row of K each) and arms each
//           stage's "full" mbarrier with the expected byte count;
//   warp 1  allocates tensor memory and, from one lane, issues tcgen05.mma
//           per K step; tcgen05.commit frees each stage and finally signals
//           the accumulator as ready;
//   warps 2-9  epilogue, two warps per TMEM lane quarter (one column half
//           each): tcgen05.ld rows of the accumulator (one TMEM lane per
//           output row), apply bias / GELU / residual / GELU' / column sums
//           and store through swizzled shared boxes with TMA stores.
// Two accumulators (2 x BN TMEM columns) let the epilogue of one tile overlap
// the main loop of the next.  Tiles are visited in groups of m-tiles so the
// B operand (the weights) is reused from L2 by concurrently running CTAs.
//
// CTA pairs (PAIR, bf16 or tf32): a cluster of two CTAs shares each 256 x 256 tile.
// Rank 0 issues tcgen05.mma.cta_group::2 (M = 256); each CTA holds 128 rows of
// A and 128 rows of B per stage and 128 rows of the accumulator; both CTAs'
// loads complete on rank 0's stage barrier, the MMA commits are multicast to
// both CTAs, and both epilogues release the accumulator on rank 0's barrier.
//
// Operand majorness follows gemm.cuh: a K-major operand is copied as one box
// {32 k, rows}; an MN-major operand as boxes {32 rows-of-MN, 32 k}, each box a
// column of 128-byte swizzle atoms.  For tf32 one MMA consumes exactly one
// 8-row swizzle atom along K, so an MN-major descriptor only needs the stride
// between MN atoms.
//
// Every mbarrier wait is bounded (about one second of device time); a wait
// that gives up raises GPT2_STATUS_TIMEOUT, makes all roles leave their loops,
// drains in-flight copies and MMAs, and frees tensor memory before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>

#include "gemm.cuh"
#include "ptx.cuh"

namespace gpt2k {
namespace tc {

constexpr int BM = 128;
// Epilogue warps: two per TMEM lane quarter on single CTAs, four on CTA pairs
// (each warp takes 32 accumulator rows and 1/2 or 1/4 of the tile's columns).
// Threads: producer, MMA issuer, epilogue.
template <bool PAIR>
struct Epi {
    static constexpr int WARPS = PAIR ? 16 : 8;
    static constexpr int PER_QUARTER = WARPS / 4;
    static constexpr int THREADS = 64 + 32 * WARPS;
};

// Per operand type: element bytes, k-block (one 128-byte row), MMA K, and the
// MN-major box (128 bytes of MN x BK k-rows).
template <bool BF16>
struct Elem {
    static constexpr int BYTES = BF16 ? 2 : 4;
    static constexpr int BK = 128 / BYTES;            // 32 fp32 or 64 bf16
    static constexpr int UMMA_K = BF16 ? 16 : 8;
    static constexpr int MN_BOX = 128 / BYTES;        // MN elements per MN-major box
    static constexpr int BOX_BYTES = 128 * BK;        // 4 KB or 8 KB
};

// Epilogue staging: each epilogue warp owns Shape::EPI_WARP bytes of shared
// memory (4 KB, or 8 KB on CTA pairs), cut into boxes of 32 rows x EC columns
// (1 KB bf16, 2 KB fp32).
constexpr int EC = 16;

// PAIR: two CTAs of a cluster share a 256-row tile through cta_group::2 MMAs;
// each holds 128 rows of A and BN/2 rows of B per stage, and 128 rows of the
// accumulator.
template <int BN, bool BF16, bool PAIR = false>
struct Shape {
    static constexpr int STAGES = PAIR ? 5 : (BN == 256 ? 4 : 6);
    static constexpr int EPI_WARP = 4096;                  // epilogue bytes per warp
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // rows of B this CTA loads
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;  // rows of A per tile
    static constexpr int A_BYTES = BM * 128;          // BM rows x 128 bytes
    static constexpr int B_BYTES = B_ROWS * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 1024 + 256 + Epi<PAIR>::WARPS * EPI_WARP;
};

struct Params {
    int M, N, K;
    int a_kmajor, b_kmajor;
    int tiles_m, tiles_n, group_m;
    int split, kb_per_split, num_kb;
    long long units;
    GemmEpilogue e;
    float* partial;         // split-K slices [split][M][N], or null
    int* status;            // device status word (timeouts), may be null
    // MN-major operand descriptor: swizzle layout type and the two byte strides
    uint32_t mn_layout, mn_lbo, mn_sbo;
    // epilogue: which tensor maps are live
    int has_aux;            // residual (aux_residual) or GELU-input tile loaded by TMA
    int aux_residual;
    int aux_bf16;           // the GELU input is bf16
    int gelu;
    int out_bf16;
    int pre_bf16;           // the GELU pre-activation is stored as bf16
    const float* bias;
    int bias_vec;           // bias is 16-byte aligned
};

// ---------------------------------------------------------------- PTX helpers
// (shared ones in ptx.cuh)
using namespace ptx;


// tanh on the special-function unit (relative error about 2^-11), for the
// tensor-core modes' GELU epilogues
__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float gelu_fwd_fast(float x) {
    return 0.5f * x * (1.0f + tanh_fast(GPT2_GELU_S * (x + GPT2_GELU_K * x * x * x)));
}
__device__ __forceinline__ float gelu_grad_fast(float x) {
    const float x2 = x * x;
    const float th = tanh_fast(GPT2_GELU_S * (x + GPT2_GELU_K * x2 * x));
    return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * GPT2_GELU_S * (1.0f + 3.0f * GPT2_GELU_K * x2);
}

// Packed pairs of fp32 (two lanes of one 64-bit register) for the CTA-pair
// epilogue: one f32x2 instruction works on two columns.
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t splat2(float a) { return f2pack(a, a); }
__device__ __forceinline__ uint32_t bf16x2(uint64_t v) {
    float a, b;
    f2unpack(v, a, b);
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
// tanh-form GELU of a pair: 0.5 x (1 + tanh(u)), u = s (x + k x^3) = x (s + s k x^2)
__device__ __forceinline__ uint64_t gelu2(uint64_t x) {
    const uint64_t x2 = mul2(x, x);
    const uint64_t u = mul2(x, fma2(x2, splat2(GPT2_GELU_S * GPT2_GELU_K), splat2(GPT2_GELU_S)));
    float u0, u1;
    f2unpack(u, u0, u1);
    const uint64_t th = f2pack(tanh_fast(u0), tanh_fast(u1));
    const uint64_t h = mul2(x, splat2(0.5f));
    return fma2(h, th, h);
}
// its derivative: 0.5 (1 + th) + 0.5 x (1 - th^2) (s + 3 s k x^2)
__device__ __forceinline__ uint64_t gelu_grad2(uint64_t x) {
    const uint64_t x2 = mul2(x, x);
    const uint64_t u = mul2(x, fma2(x2, splat2(GPT2_GELU_S * GPT2_GELU_K), splat2(GPT2_GELU_S)));
    float u0, u1;
    f2unpack(u, u0, u1);
    const float t0 = tanh_fast(u0), t1 = tanh_fast(u1);
    const uint64_t th = f2pack(t0, t1);
    const uint64_t om = fma2(f2pack(-t0, -t1), th, splat2(1.f));
    const uint64_t d1 = fma2(x2, splat2(3.f * GPT2_GELU_S * GPT2_GELU_K), splat2(GPT2_GELU_S));
    const uint64_t g = mul2(mul2(mul2(x, splat2(0.5f)), om), d1);
    return add2(fma2(th, splat2(0.5f), splat2(0.5f)), g);
}
// 128-byte swizzle: 16-byte unit `unit` of row `row` of a box with 128-byte rows
__device__ __forceinline__ uint32_t sw128(int row, int unit) {
    return (uint32_t)(row * 128 + ((unit ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------- scheduling
struct Unit {
    int split, m_tile, n_tile;
};

__device__ __forceinline__ Unit unit_coords(const Params& p, long long u) {
    long long tiles = (long long)p.tiles_m * p.tiles_n;
    Unit r;
    r.split = (int)(u / tiles);
    int t = (int)(u % tiles);
    int per_group = p.group_m * p.tiles_n;
    int g = t / per_group;
    int first_m = g * p.group_m;
    int gm = min(p.tiles_m - first_m, p.group_m);
    int in_g = t - g * per_group;
    r.m_tile = first_m + in_g % gm;
    r.n_tile = in_g / gm;
    return r;
}

// ---------------------------------------------------------------- epilogue
// Eight epilogue warps: warp w reads TMEM lane quarter w % 4 (32 accumulator
// rows, thread = row) and one half of the tile's columns, EC columns at a time.
// Per chunk it loads the accumulator from tensor memory, applies the epilogue
// in registers and writes the chunk into a swizzled shared-memory box that one
// lane stores with a TMA bulk copy (clipped at the matrix edges).  Two warps
// per scheduler hide each other's latency; each warp's 4 KB holds as many
// output boxes as fit, so stores stay in flight while later chunks are
// written.  An input tile (residual or GELU input) arrives by TMA into a ring
// of boxes filled ahead of use, and the chunk's output is written back over
// its own input box and stored from there.  fp32 boxes have 64-byte rows
// (64-byte swizzle), bf16 boxes 32-byte rows (32-byte swizzle); both keep a
// warp's 16-byte writes free of bank conflicts.
__device__ __forceinline__ uint32_t sw64(int row, int chunk) {
    return (uint32_t)(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}
__device__ __forceinline__ uint32_t sw32(int row, int chunk) {
    return (uint32_t)(row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4));
}

// 16 values of one row into a box: fp32 (64-byte rows) or bf16 (32-byte rows)
__device__ __forceinline__ void put_row16(uint8_t* box, int row, const float (&x)[16], bool bf16) {
    if (bf16) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            __nv_bfloat162 h0 = __floats2bfloat162_rn(x[8 * h], x[8 * h + 1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(x[8 * h + 2], x[8 * h + 3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(x[8 * h + 4], x[8 * h + 5]);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(x[8 * h + 6], x[8 * h + 7]);
            *reinterpret_cast<uint4*>(box + sw32(row, h)) =
                make_uint4(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1),
                           *reinterpret_cast<uint32_t*>(&h2), *reinterpret_cast<uint32_t*>(&h3));
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; j++)
            *reinterpret_cast<float4*>(box + sw64(row, j)) =
                make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    }
}

// 16 values of one row from a box
__device__ __forceinline__ void get_row16(const uint8_t* box, int row, float (&a)[16], bool bf16) {
    if (bf16) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const uint4 v = *reinterpret_cast<const uint4*>(box + sw32(row, h));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
                a[8 * h + 2 * k] = f.x;
                a[8 * h + 2 * k + 1] = f.y;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float4 v = *reinterpret_cast<const float4*>(box + sw64(row, j));
            a[4 * j] = v.x; a[4 * j + 1] = v.y; a[4 * j + 2] = v.z; a[4 * j + 3] = v.w;
        }
    }
}

// ---------------------------------------------------------------- kernel
template <int BN, bool BF16, bool PAIR>
__global__ void __launch_bounds__(Epi<PAIR>::THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmAux,
               const __grid_constant__ CUtensorMap tmPre, const Params p) {
    static_assert(!PAIR || BN == 256, "CTA pairs: 256-column tiles");
    using S = Shape<BN, BF16, PAIR>;
    using E = Elem<BF16>;
    constexpr int RING_MAX = S::EPI_WARP / 1024;      // input boxes per warp (bf16 boxes)
    constexpr int EPI_WARPS = Epi<PAIR>::WARPS;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[S::STAGES], empty_bar[S::STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], drain_bar, aux_bar[EPI_WARPS][RING_MAX];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // pair mode: rank 0 issues the MMAs; both CTAs walk the same units
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const long long u_first = PAIR ? blockIdx.x / 2 : blockIdx.x;
    const long long u_step = PAIR ? gridDim.x / 2 : gridDim.x;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const base_ptr = smem_raw + (base - raw);
    auto stage_a = [&](int s) { return base + (uint32_t)(s * S::STAGE_BYTES); };
    auto stage_b = [&](int s) { return base + (uint32_t)(s * S::STAGE_BYTES + S::A_BYTES); };

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < S::STAGES; s++) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), PAIR ? 2 * EPI_WARPS : EPI_WARPS);   // both CTAs' epilogues
        }
        mbar_init(smem_u32(&drain_bar), 1);
        for (int w = 0; w < EPI_WARPS; w++)
            for (int k = 0; k < RING_MAX; k++) mbar_init(smem_u32(&aux_bar[w][k]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_map(&tmA);
        prefetch_map(&tmB);
        prefetch_map(&tmOut);
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(&s_tmem, S::TMEM_COLS);
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(&s_tmem)),
                         "r"(S::TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();            // the peer's barriers exist before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_phase = 0;   // per-stage bits, for the abort drain
            bool ok = true;
            // a load of this CTA's shared memory counted on barrier `bar` (pair mode:
            // rank 0's barrier, which expects both CTAs' bytes)
            auto load = [&](uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
                if (PAIR) tma_load_2d_pair(dst, map, x, y, bar);
                else tma_load_2d(dst, map, x, y, bar);
            };
            for (long long u = u_first; u < p.units && ok; u += u_step) {
                Unit c = unit_coords(p, u);
                const int m0 = c.m_tile * S::TILE_M + (int)rank * BM, n0 = c.n_tile * BN + (int)rank * S::B_ROWS;
                const int kb0 = c.split * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, &s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&full_bar[stage]);
                    const uint32_t fb = PAIR ? mapa_shared(fb_local, 0) : fb_local;
                    if (rank == 0) {
                        mbar_expect_tx(fb_local, PAIR ? 2 * S::STAGE_BYTES : S::STAGE_BYTES);
                        armed |= 1u << stage;
                        armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                    }
                    const int k0 = kb * E::BK;
                    if (p.a_kmajor) {
                        load(stage_a(stage), &tmA, k0, m0, fb);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / E::MN_BOX; j++)
                            load(stage_a(stage) + j * E::BOX_BYTES, &tmA, m0 + E::MN_BOX * j, k0, fb);
                    }
                    if (p.b_kmajor) {
                        load(stage_b(stage), &tmB, k0, n0, fb);
                    } else {
#pragma unroll
                        for (int j = 0; j < S::B_ROWS / E::MN_BOX; j++)
                            load(stage_b(stage) + j * E::BOX_BYTES, &tmB, n0 + E::MN_BOX * j, k0, fb);
                    }
                    if (++stage == S::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // drain: wait (bounded, ignoring the abort flag) for copies this thread issued
                for (int s = 0; s < S::STAGES; s++) {
                    if (!(armed >> s & 1u)) continue;
                    uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&full_bar[s]), (armed_phase >> s) & 1u) &&
                           globaltimer() - t0 < WAIT_NS) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (pair mode: rank 0 only)
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = instr_desc(S::TILE_M, BN, !p.a_kmajor, !p.b_kmajor, BF16);
            // one MMA consumes UMMA_K elements: 32 bytes of a K-major row, or UMMA_K
            // 128-byte rows of an MN-major box
            constexpr uint32_t KMAJ_STEP = E::UMMA_K * E::BYTES;
            constexpr uint32_t MN_STEP = E::UMMA_K * 128;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (long long u = u_first; u < p.units && ok; u += u_step) {
                Unit c = unit_coords(p, u);
                const int kb0 = c.split * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                if (!mbar_wait(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, &s_abort, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(smem_u32(&full_bar[stage]), phase, &s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = stage_a(stage), b0 = stage_b(stage);
#pragma unroll
                    for (int k = 0; k < E::BK / E::UMMA_K; k++) {
                        uint64_t ad = p.a_kmajor
                                          ? smem_desc(a0 + k * KMAJ_STEP, 16, 1024, LAYOUT_SW128)
                                          : smem_desc(a0 + k * MN_STEP, p.mn_lbo, p.mn_sbo, p.mn_layout);
                        uint64_t bd = p.b_kmajor
                                          ? smem_desc(b0 + k * KMAJ_STEP, 16, 1024, LAYOUT_SW128)
                                          : smem_desc(b0 + k * MN_STEP, p.mn_lbo, p.mn_sbo, p.mn_layout);
                        if (PAIR) mma_issue_pair<BF16>(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        else mma_issue<BF16>(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    // the stage is free in both CTAs once these MMAs have read it
                    if (PAIR) mma_commit_pair(smem_u32(&empty_bar[stage]), 0x3);
                    else mma_commit(smem_u32(&empty_bar[stage]));
                    if (++stage == S::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (PAIR) mma_commit_pair(smem_u32(&tfull_bar[acc]), 0x3);
                else mma_commit(smem_u32(&tfull_bar[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // every MMA this thread issued has completed once drain_bar fires
            if (PAIR) mma_commit_pair(smem_u32(&drain_bar), 0x1);
            else mma_commit(smem_u32(&drain_bar));
            uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(&drain_bar), 0) && globaltimer() - t0 < WAIT_NS) {
            }
        }
    } else if (PAIR && p.out_bf16 && !p.partial && !p.aux_residual) {
        // ------------------------------------------------ epilogue, CTA pairs, bf16 output (warps 2 ..)
        // Warp ew reads TMEM lane quarter q (32 accumulator rows, thread = row) and
        // 64 of the tile's 256 columns, 16 at a time, with the next load in flight,
        // and fills one box of 32 rows x 64 columns (128-byte rows, 128-byte
        // swizzle) that one lane stores with one TMA copy: few, large stores leave
        // the copy engine to the operand loads.  The arithmetic runs on packed fp32
        // pairs.  A GELU input tile arrives by TMA into the box before the tile
        // (issued once the previous tile's store has read it) and is overwritten in
        // place.  With GELU the tile takes two passes over the accumulator: the
        // pre-activation first, then (once that store has read the box) the
        // activation.  The accumulator goes back to the MMA thread as soon as the
        // last pass has loaded its last columns.
        const int q = warp & 3;
        const int ew = warp - 2;
        const int col_lo = (ew >> 2) * 64;
        uint8_t* const box = base_ptr + S::STAGES * S::STAGE_BYTES + ew * S::EPI_WARP;
        const uint32_t box_s = smem_u32(box);
        const bool pre = p.gelu != 0;
        const bool gx = p.has_aux != 0;
        const bool use_bias = p.bias != nullptr;
        const uint32_t aux_bar_s = smem_u32(&aux_bar[ew][0]);
        uint32_t aux_issued = 0, aux_done = 0;
        // GELU input box of tile u (lane 0)
        auto aux_issue = [&](long long u) {
            Unit c = unit_coords(p, u);
            const int x0 = c.n_tile * BN + col_lo, y0 = c.m_tile * S::TILE_M + (int)rank * BM + q * 32;
            mbar_expect_tx(aux_bar_s, 4096u);
            tma_load_2d(box_s, &tmAux, x0, y0, aux_bar_s);
            aux_issued++;
        };
        if (gx && lane == 0 && u_first < p.units) aux_issue(u_first);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (long long u = u_first; u < p.units && ok; u += u_step) {
            Unit c = unit_coords(p, u);
            const int m0 = c.m_tile * S::TILE_M + (int)rank * BM, n0 = c.n_tile * BN + col_lo;
            const int row0 = m0 + q * 32;
            const int ncols = min(64, p.N - n0);
            const int nchunks = ncols > 0 ? (ncols + EC - 1) / EC : 0;
            const bool row_ok = row0 + lane < p.M;
            if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, &s_abort, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (gx) {
                if (!mbar_wait(aux_bar_s, aux_done & 1u, &s_abort, p.status)) {
                    ok = false;
                    break;
                }
                aux_done++;
            }
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + col_lo);
            const int npass = pre ? 2 : 1;
            for (int pass = 0; pass < npass; pass++) {
                // pass 0 of a GELU tile writes the pre-activation, the last pass the output
                const bool act = pre && pass == 1, pre_pass = pre && pass == 0;
                if (!gx) {
                    if (lane == 0) bulk_wait_read(0);        // the box's last store has read it
                    __syncwarp();
                }
                auto chunk = [&](int k, uint32_t (&r)[16], uint32_t (&rn)[16]) {
                    const int nc = n0 + k * EC;
                    tmem_wait16(r);
                    if (k + 1 < nchunks) {
                        tmem_ld16_async(taddr + (uint32_t)((k + 1) * EC), rn);
                    } else if (pass == npass - 1) {
                        // every column is in registers: the accumulator goes back to the MMA thread
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
                    }
                    uint64_t x[8];
#pragma unroll
                    for (int j = 0; j < 8; j++)
                        x[j] = f2pack(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                    if (use_bias) {
                        // the same 16 bias values in every lane (broadcast loads)
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            float4 v;
                            if (nc + 16 <= p.N && p.bias_vec) {
                                v = __ldg(reinterpret_cast<const float4*>(p.bias + nc) + j);
                            } else {
                                const int c0 = nc + 4 * j;
                                v.x = c0 < p.N ? __ldg(p.bias + c0) : 0.f;
                                v.y = c0 + 1 < p.N ? __ldg(p.bias + c0 + 1) : 0.f;
                                v.z = c0 + 2 < p.N ? __ldg(p.bias + c0 + 2) : 0.f;
                                v.w = c0 + 3 < p.N ? __ldg(p.bias + c0 + 3) : 0.f;
                            }
                            x[2 * j] = add2(x[2 * j], f2pack(v.x, v.y));
                            x[2 * j + 1] = add2(x[2 * j + 1], f2pack(v.z, v.w));
                        }
                    }
                    if (gx) {
                        // out = acc * gelu'(x), x read from this lane's own row of the box
#pragma unroll
                        for (int h = 0; h < 2; h++) {
                            const uint4 v = *reinterpret_cast<const uint4*>(box + sw128(lane, 2 * k + h));
                            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int i = 0; i < 4; i++) {
                                const float2 g = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
                                x[4 * h + i] = mul2(x[4 * h + i], gelu_grad2(f2pack(g.x, g.y)));
                            }
                        }
                    }
                    if (act) {
#pragma unroll
                        for (int j = 0; j < 8; j++) x[j] = gelu2(x[j]);
                    }
                    if (p.e.colsum && !pre_pass && row0 < p.M) {
                        // this chunk's column sums over the warp's 32 rows (rows past M count 0)
                        float cs[16];
#pragma unroll
                        for (int j = 0; j < 8; j++) {
                            float a0, a1;
                            f2unpack(x[j], a0, a1);
                            cs[2 * j] = row_ok ? a0 : 0.f;
                            cs[2 * j + 1] = row_ok ? a1 : 0.f;
                        }
                        warp_colsum<16>(cs, lane);
                        const int col = nc + warp_colsum_col<16>(lane);
                        if (!(lane & 1) && col < p.N) p.e.colsum[(size_t)(row0 >> 5) * p.N + col] = cs[0];
                    }
#pragma unroll
                    for (int h = 0; h < 2; h++)
                        *reinterpret_cast<uint4*>(box + sw128(lane, 2 * k + h)) =
                            make_uint4(bf16x2(x[4 * h]), bf16x2(x[4 * h + 1]), bf16x2(x[4 * h + 2]),
                                       bf16x2(x[4 * h + 3]));
                };
                uint32_t ra[16], rb[16];
                if (nchunks > 0) {
                    tmem_ld16_async(taddr, ra);
                    for (int k = 0; k < nchunks; k += 2) {
                        chunk(k, ra, rb);
                        if (k + 1 < nchunks) chunk(k + 1, rb, ra);
                    }
                } else if (pass == npass - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    if (nchunks > 0 && row0 < p.M) tma_store_2d(pre_pass ? &tmPre : &tmOut, n0, row0, box_s);
                    bulk_commit();
                }
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            // the next tile's GELU input, once this tile's store has read the box
            const long long un = u + u_step;
            if (gx && lane == 0 && un < p.units) {
                bulk_wait_read(0);
                aux_issue(un);
            }
        }
        if (gx && !ok && lane == 0) {
            // an input load still in flight lands in this CTA's shared memory: wait
            // (bounded, ignoring the abort flag) for it before leaving
            for (uint32_t g = aux_done; g != aux_issued; g++) {
                uint64_t t0 = globaltimer();
                while (!mbar_try_wait(aux_bar_s, g & 1u) && globaltimer() - t0 < WAIT_NS) {
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue, fp32 outputs on CTA pairs and
        // every single-CTA product (warps 2 ..)
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int ew = warp - 2;
        constexpr int WCOLS = BN / Epi<PAIR>::PER_QUARTER;   // this warp's share of the tile's columns
        const int col_lo = (ew >> 2) * WCOLS;
        uint8_t* const wbuf = base_ptr + S::STAGES * S::STAGE_BYTES + ew * S::EPI_WARP;
        const bool has_aux = p.has_aux != 0;
        const bool pre = p.gelu && !p.partial;
        const bool out16 = p.out_bf16 != 0, pre16 = p.pre_bf16 != 0, aux16 = p.aux_bf16 != 0;
        const int out_bytes = out16 ? 1024 : 2048;
        // output boxes (no input tile): one chunk = output box (+ pre-activation box)
        const int chunk_bytes = out_bytes + (pre ? (pre16 ? 1024 : 2048) : 0);
        const int nbuf = min(8, S::EPI_WARP / chunk_bytes);     // 1, 2, 4 or 8
        // input ring: box g of this warp's sequence uses slot g % ring, phase (g / ring) & 1
        const int aux_bytes = aux16 && !p.aux_residual ? 1024 : 2048;
        const int ring = S::EPI_WARP / aux_bytes;
        uint32_t box_seq = 0;                // output chunks stored so far
        uint32_t aux_issued = 0;             // input boxes requested (lane 0)
        uint32_t aux_seq = 0;                // input boxes consumed
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (long long u = u_first; u < p.units && ok; u += u_step) {
            Unit c = unit_coords(p, u);
            const int m0 = c.m_tile * S::TILE_M + (int)rank * BM, n0 = c.n_tile * BN + col_lo;
            const int row0 = m0 + q * 32;
            const int ncols = min(WCOLS, p.N - n0);
            const int nchunks = ncols > 0 ? (ncols + EC - 1) / EC : 0;
            auto aux_issue = [&](int k) {    // input box of chunk k of this tile (lane 0)
                const uint32_t slot = aux_issued % (uint32_t)ring;
                const uint32_t bar = smem_u32(&aux_bar[ew][slot]);
                mbar_expect_tx(bar, (uint32_t)aux_bytes);
                tma_load_2d(smem_u32(wbuf + slot * aux_bytes), &tmAux, n0 + k * EC, row0, bar);
                aux_issued++;
            };
            if (has_aux && lane == 0) {
                bulk_wait_read(0);           // earlier stores out of the ring are done reading
                for (int k = 0; k < min(ring - 1, nchunks); k++) aux_issue(k);
                // the next tile's input rows of this warp go to L2 while this tile runs
                const long long un = u + u_step;
                if (un < p.units) {
                    Unit cn = unit_coords(p, un);
                    const int nn0 = cn.n_tile * BN + col_lo, nr0 = cn.m_tile * S::TILE_M + (int)rank * BM + q * 32;
                    if (nr0 < p.M)
                        for (int k = 0; k < WCOLS && nn0 + k < p.N; k += EC) tma_prefetch_l2(&tmAux, nn0 + k, nr0);
                }
            }
            // the bias of this warp's columns: lane l holds columns n0 + 4l .. n0 + 4l + 3
            // (loaded before the accumulator is ready; shuffled out chunk by chunk)
            float4 bl = make_float4(0.f, 0.f, 0.f, 0.f);
            const bool use_bias = !p.partial && p.bias;
            if (use_bias && 4 * lane < WCOLS) {
                const int c0 = n0 + 4 * lane;
                if (c0 + 4 <= p.N) {
                    bl = __ldg(reinterpret_cast<const float4*>(p.bias + c0));
                } else {
                    if (c0 < p.N) bl.x = __ldg(p.bias + c0);
                    if (c0 + 1 < p.N) bl.y = __ldg(p.bias + c0 + 1);
                    if (c0 + 2 < p.N) bl.z = __ldg(p.bias + c0 + 2);
                }
            }
            if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, &s_abort, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + col_lo);
            // chunk k: its accumulator columns were loaded into r one chunk ahead;
            // the next chunk's load goes out before this one is processed
            auto chunk = [&](int k, uint32_t (&r)[16], uint32_t (&rn)[16]) -> bool {
                tmem_wait16(r);
                if (k + 1 < nchunks) tmem_ld16_async(taddr + (uint32_t)((k + 1) * EC), rn);
                const int nc = n0 + k * EC;
                float x[16];
#pragma unroll
                for (int j = 0; j < 16; j++) x[j] = __uint_as_float(r[j]);
                if (use_bias) {
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const int src = 4 * k + j;       // the lane holding columns nc + 4j .. nc + 4j + 3
                        x[4 * j] += __shfl_sync(0xffffffffu, bl.x, src);
                        x[4 * j + 1] += __shfl_sync(0xffffffffu, bl.y, src);
                        x[4 * j + 2] += __shfl_sync(0xffffffffu, bl.z, src);
                        x[4 * j + 3] += __shfl_sync(0xffffffffu, bl.w, src);
                    }
                }
                uint8_t* outb;
                if (has_aux) {
                    // the chunk's input box: read, then overwrite with the output
                    const uint32_t slot = aux_seq % (uint32_t)ring;
                    if (!mbar_wait(smem_u32(&aux_bar[ew][slot]), (aux_seq / (uint32_t)ring) & 1u, &s_abort,
                                   p.status)) {
                        return false;
                    }
                    aux_seq++;
                    outb = wbuf + slot * aux_bytes;
                    float a[16];
                    get_row16(outb, lane, a, aux_bytes == 1024);
                    if (p.aux_residual) {
#pragma unroll
                        for (int j = 0; j < 16; j++) x[j] += a[j];
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; j++) x[j] *= gelu_grad_fast(a[j]);
                    }
                    __syncwarp();            // every lane has read the box before it is overwritten
                } else {
                    const uint32_t b = box_seq % (uint32_t)nbuf;
                    outb = wbuf + b * chunk_bytes;
                    // the store that last read this box is done reading
                    if (lane == 0) bulk_wait_read(nbuf - 1);
                    __syncwarp();
                    if (pre) {
                        put_row16(outb + out_bytes, lane, x, pre16);
#pragma unroll
                        for (int j = 0; j < 16; j++) x[j] = gelu_fwd_fast(x[j]);
                    }
                }
                if (p.e.colsum && row0 < p.M) {
                    // this chunk's column sums over the warp's 32 rows (rows past M count 0;
                    // a group that starts past M has no slot)
                    float cs[16];
#pragma unroll
                    for (int j = 0; j < 16; j++) cs[j] = row0 + lane < p.M ? x[j] : 0.f;
                    warp_colsum<16>(cs, lane);
                    const int col = nc + warp_colsum_col<16>(lane);
                    if (!(lane & 1) && col < p.N) p.e.colsum[(size_t)(row0 >> 5) * p.N + col] = cs[0];
                }
                put_row16(outb, lane, x, out16);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    if (p.partial) tma_store_3d(&tmOut, nc, row0, c.split, smem_u32(outb));
                    else tma_store_2d(&tmOut, nc, row0, smem_u32(outb));
                    if (pre && !has_aux) tma_store_2d(&tmPre, nc, row0, smem_u32(outb + out_bytes));
                    bulk_commit();
                    // refill: the box of chunk k - 1 (stored one chunk ago) takes chunk k + ring - 1
                    if (has_aux && k + ring - 1 < nchunks) {
                        bulk_wait_read(1);
                        aux_issue(k + ring - 1);
                    }
                }
                box_seq++;
                return true;
            };
            uint32_t ra[16], rb[16];
            if (nchunks > 0) tmem_ld16_async(taddr, ra);
            for (int k = 0; k < nchunks && ok; k += 2) {
                if (!chunk(k, ra, rb) || (k + 1 < nchunks && !chunk(k + 1, rb, ra))) ok = false;
            }
            if (!ok) {
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");   // no load left in flight
                break;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // pair mode: rank 0's MMA thread waits for both CTAs' epilogues
                if (PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
                else mbar_arrive(smem_u32(&tempty_bar[acc]));
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (has_aux && !ok && lane == 0) {
            // input loads still in flight land in this CTA's shared memory: wait
            // (bounded, ignoring the abort flag) for each before leaving
            for (uint32_t g = aux_seq; g != aux_issued; g++) {
                const uint32_t bar = smem_u32(&aux_bar[ew][g % (uint32_t)ring]);
                uint64_t t0 = globaltimer();
                while (!mbar_try_wait(bar, (g / (uint32_t)ring) & 1u) && globaltimer() - t0 < WAIT_NS) {
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // pair mode: neither CTA frees its tensor memory or leaves while the peer may
    // still signal its barriers
    if (PAIR) cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR) {
            tmem_dealloc_pair(tmem_base, S::TMEM_COLS);
        } else {
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(S::TMEM_COLS)
                         : "memory");
        }
    }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            (void)cudaGetLastError();
    }
    return fn;
}

// 2-D tensor map over a row-major matrix [rows, cols] (fp32 or bf16) with row
// stride `ld` elements; box {box_cols, box_rows}, zero fill.
static bool make_map(CUtensorMap* map, const void* ptr, bool bf16, int cols, int rows, int ld,
                     int box_cols, int box_rows, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    const size_t es = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * es};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                    const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D fp32 tensor map [z][rows][cols] (plain, contiguous slices) with box
// {box_cols, box_rows, 1}: the split-K partial slices, clipped per slice.
static bool make_map_3d(CUtensorMap* map, const float* ptr, int cols, int rows, int depth, int box_cols,
                        int box_rows, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)depth};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)cols * rows * 4};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MN-major operand tiles are boxes of 128 bytes of MN x BK k-rows, side by side
// along MN.  Descriptor: LBO = stride between MN boxes, SBO = stride between the
// k-row groups of the swizzle atom.
//   tf32: 128-byte swizzle of 32-byte chunks (UMMA layout 1, TMA ATOM_32B), 4-row
//         groups: LBO 4096, SBO 512 (the layout the tensor core reads tf32
//         MN-major operands in; with the 16-byte-chunk swizzle it returns zeros).
//   bf16: 128-byte swizzle of 16-byte chunks (UMMA layout 2, TMA 128B), 8-row
//         groups: LBO 8192, SBO 1024.
struct Maps {
    CUtensorMap a, b, out, aux, pre;
};

template <int BN, bool BF16, bool PAIR>
static int prepare(const GemmProblem& g, const GemmEpilogue& e, float* partial, int split, Maps* mp,
                   Params* pp) {
    using S = Shape<BN, BF16, PAIR>;
    using E = Elem<BF16>;
    if (smem_limit(reinterpret_cast<const void*>(gemm_tc_kernel<BN, BF16, PAIR>), (int)S::SMEM)) return GPT2_ECUDA;
    const CUtensorMapSwizzle KSW = CU_TENSOR_MAP_SWIZZLE_128B;
    const CUtensorMapSwizzle MSW = BF16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
    // A: K-major [M, K] (box {BK, 128}); M-major [K, M] (box {MN_BOX, BK})
    bool ok = g.a_kmajor ? make_map(&mp->a, g.A, BF16, g.K, g.M, g.lda, E::BK, BM, KSW)
                         : make_map(&mp->a, g.A, BF16, g.M, g.K, g.lda, E::MN_BOX, E::BK, MSW);
    ok = ok && (g.b_kmajor ? make_map(&mp->b, g.B, BF16, g.K, g.N, g.ldb, E::BK, S::B_ROWS, KSW)
                           : make_map(&mp->b, g.B, BF16, g.N, g.K, g.ldb, E::MN_BOX, E::BK, MSW));
    Params p{};
    // epilogue maps.  bf16 outputs on CTA pairs: boxes of 32 rows x 64 columns
    // (128-byte rows, 128-byte swizzle); everything else: boxes of 32 rows x EC
    // columns, fp32 64-byte rows (64-byte swizzle) or bf16 32-byte rows (32-byte
    // swizzle)
    auto swz = [](bool b16) { return b16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B; };
    if (PAIR && !partial && e.out_bf16 && !e.residual) {
        const CUtensorMapSwizzle W = CU_TENSOR_MAP_SWIZZLE_128B;
        ok = ok && make_map(&mp->out, e.out, true, g.N, g.M, e.ldo, 64, 32, W);
        if (e.gelu_x) {
            ok = ok && make_map(&mp->aux, e.gelu_x, true, g.N, g.M, e.ldg, 64, 32, W);
            p.has_aux = 1;
            p.aux_bf16 = 1;
        }
        if (e.gelu) {
            ok = ok && make_map(&mp->pre, e.out_pre, true, g.N, g.M, e.ldo, 64, 32, W);
            p.pre_bf16 = 1;
        }
    } else if (partial) {
        ok = ok && make_map_3d(&mp->out, partial, g.N, g.M, split, EC, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    } else {
        ok = ok && make_map(&mp->out, e.out, e.out_bf16, g.N, g.M, e.ldo, EC, 32, swz(e.out_bf16));
        if (e.residual) {
            ok = ok && make_map(&mp->aux, e.residual, false, g.N, g.M, e.ldo, EC, 32, swz(false));
            p.has_aux = 1;
            p.aux_residual = 1;
        } else if (e.gelu_x) {
            ok = ok && make_map(&mp->aux, e.gelu_x, e.gelu_x_bf16, g.N, g.M, e.ldg, EC, 32, swz(e.gelu_x_bf16));
            p.has_aux = 1;
            p.aux_bf16 = e.gelu_x_bf16 ? 1 : 0;
        }
        if (e.gelu) {
            ok = ok && make_map(&mp->pre, e.out_pre, e.pre_bf16, g.N, g.M, e.ldo, EC, 32, swz(e.pre_bf16));
            p.pre_bf16 = e.pre_bf16 ? 1 : 0;
        }
    }
    if (!ok) return GPT2_ENOTSUP;
    if (!p.has_aux) mp->aux = mp->out;             // unused, but a valid map
    if (!e.gelu || partial) mp->pre = mp->out;
    p.M = g.M; p.N = g.N; p.K = g.K;
    p.a_kmajor = g.a_kmajor; p.b_kmajor = g.b_kmajor;
    p.tiles_m = ceil_div(g.M, S::TILE_M);
    p.tiles_n = ceil_div(g.N, BN);
    p.num_kb = ceil_div(g.K, E::BK);
    p.split = split;
    p.kb_per_split = ceil_div(p.num_kb, split);
    if (ceil_div(p.num_kb, p.kb_per_split) != split) return GPT2_EINVAL;   // an empty K slice
    p.units = (long long)p.tiles_m * p.tiles_n * split;
    // group enough m-tiles that their A rows stay in L2 while B streams past
    p.group_m = std::max(1, std::min(p.tiles_m, PAIR ? 8 : 16));
    p.e = e;
    p.partial = partial;
    p.status = g.status;
    p.mn_layout = BF16 ? LAYOUT_SW128 : LAYOUT_SW128_32B;
    p.mn_lbo = E::BOX_BYTES;
    p.mn_sbo = BF16 ? 8 * 128 : 4 * 128;
    p.gelu = partial ? 0 : e.gelu;
    p.out_bf16 = partial ? 0 : e.out_bf16;
    p.bias = partial ? nullptr : e.bias;
    p.bias_vec = p.bias && (reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0;
    *pp = p;
    return GPT2_OK;
}

// Clusters of two CTAs that can be resident at once for the pair kernel (one
// CTA per SM): the persistent grid's size.
static int pair_clusters() {
    static int n = -1;
    if (n < 0) {
        using S = Shape<256, true, true>;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2 * std::max(1, num_sms() / 2));
        cfg.blockDim = dim3(Epi<true>::THREADS);
        cfg.dynamicSmemBytes = S::SMEM;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int c = 0;
        if (cudaFuncSetAttribute(gemm_tc_kernel<256, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)S::SMEM) == cudaSuccess &&
            cudaOccupancyMaxActiveClusters(&c, gemm_tc_kernel<256, true, true>, &cfg) == cudaSuccess && c > 0)
            n = c;
        else {
            (void)cudaGetLastError();
            n = 0;
        }
    }
    return n;
}

template <int BN, bool BF16, bool PAIR>
static int run(const Maps& mp, const Params& p, cudaStream_t st) {
    if constexpr (!PAIR) {
        int grid = (int)std::min<long long>(p.units, num_sms());
        count_launch(), gemm_tc_kernel<BN, BF16, false><<<grid, Epi<false>::THREADS, Shape<BN, BF16, false>::SMEM, st>>>(
            mp.a, mp.b, mp.out, mp.aux, mp.pre, p);
        GPT2_LAUNCH_CHECK();
        return GPT2_OK;
    } else {
    const int clusters = (int)std::min<long long>(p.units, pair_clusters());
    if (clusters < 1) return GPT2_ENOTSUP;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(Epi<true>::THREADS);
    cfg.dynamicSmemBytes = Shape<BN, BF16, true>::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launch();
    GPT2_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, BF16, true>, mp.a, mp.b, mp.out, mp.aux, mp.pre, p));
    return GPT2_OK;
    }
}

template <int BN, bool BF16, bool PAIR>
static int launch(const GemmProblem& g, const GemmEpilogue& e, float* partial, int split,
                  cudaStream_t st) {
    Maps mp;
    Params p;
    int rc = prepare<BN, BF16, PAIR>(g, e, partial, split, &mp, &p);
    if (rc) return rc;
    return run<BN, BF16, PAIR>(mp, p, st);
}

template <bool BF16>
static int launch_any(const GemmProblem& g, const GemmEpilogue& e, float* partial, int split,
                      cudaStream_t st) {
    if (gemm_tc_pair(g, partial ? nullptr : &e)) return launch<256, BF16, true>(g, e, partial, split, st);
    if (g.N <= 128) return launch<128, BF16, false>(g, e, partial, split, st);
    return launch<256, BF16, false>(g, e, partial, split, st);
}

}  // namespace tc

// bf16 and tf32 products with at least 256 rows and 256 columns run on CTA
// pairs (cta_group::2, 256 x 256 tiles, sixteen epilogue warps per CTA);
// smaller ones on single CTAs (128 x 256 or 128 x 128 tiles).
// GPT2_GEMM_CTA_PAIRS=0 in the environment sends everything to single CTAs.
bool gemm_tc_pair(const GemmProblem& g, const GemmEpilogue* e) {
    static int on = -1;
    if (on < 0) {
        const char* v = getenv("GPT2_GEMM_CTA_PAIRS");
        on = (v && v[0] == '0') ? 0 : 1;
    }
    if (!on || g.M < 256 || g.N < 256 || tc::pair_clusters() <= 0) return false;
    // a bf16 output with GELU takes a bf16 pre-activation and a bf16 GELU input
    // on pairs (both go through the output's box)
    if (e && e->out_bf16 && !e->residual &&
        ((e->gelu && (!e->pre_bf16 || e->gelu_x)) || (e->gelu_x && !e->gelu_x_bf16)))
        return false;
    return true;
}

int gemm_tc_pair_slots() { return tc::pair_clusters(); }

bool encode_tensor_map(CUtensorMap* map, bool bf16, int rank, const void* ptr, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
    auto fn = tc::encode_fn();
    if (!fn) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank,
              const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gemm_tc_supported(const GemmProblem& p) {
    if (p.M < 1 || p.N < 1 || p.K < 1) return false;
    const int align = p.bf16 ? 8 : 4;             // 16-byte row strides
    if (!aligned16(p.A) || !aligned16(p.B) || (p.lda % align) || (p.ldb % align)) return false;
    return tc::encode_fn() != nullptr;
}

// The epilogue moves its tiles with TMA: 16-byte aligned bases and row strides.
bool gemm_tc_epilogue_supported(const GemmEpilogue& e) {
    const int oa = e.out_bf16 ? 8 : 4;
    if (!aligned16(e.out) || e.ldo % oa) return false;
    if (e.residual && (!aligned16(e.residual) || e.ldo % 4)) return false;
    if (e.gelu && (!aligned16(e.out_pre) || e.ldo % (e.pre_bf16 ? 8 : 4))) return false;
    if (e.gelu_x && (!aligned16(e.gelu_x) || e.ldg % (e.gelu_x_bf16 ? 8 : 4))) return false;
    if (e.bias && (reinterpret_cast<uintptr_t>(e.bias) & 15)) return false;
    return true;
}

int gemm_tc(const GemmProblem& p, const GemmEpilogue& e, cudaStream_t st) {
    return p.bf16 ? tc::launch_any<true>(p, e, nullptr, 1, st) : tc::launch_any<false>(p, e, nullptr, 1, st);
}

int gemm_tc_splitk(const GemmProblem& p, float* partial, int split, cudaStream_t st) {
    GemmEpilogue e{};
    return p.bf16 ? tc::launch_any<true>(p, e, partial, split, st)
                  : tc::launch_any<false>(p, e, partial, split, st);
}

}  // namespace gpt2k
