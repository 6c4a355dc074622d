// gemm_tc.cu -- fp32-storage GEMM on the 5th-generation tensor cores (tcgen05,
// kind::tf32, fp32 accumulation in tensor memory), fed by TMA.
//
// Persistent, warp-specialised kernel, one CTA per SM, 192 threads:
//   warp 0  TMA producer: fills a ring of shared-memory stages (A: 128 x 32,
//           B: BN x 32 fp32, 128-byte swizzle) and arms each stage's "full"
//           mbarrier with the expected byte count;
//   warp 1  allocates tensor memory and, from one lane, issues tcgen05.mma
//           (M=128, N=BN, K=8) per k-slice; tcgen05.commit frees each stage
//           and finally signals the accumulator as ready;
//   warps 2-5  epilogue: tcgen05.ld rows of the accumulator (one TMEM lane per
//           output row), apply bias / GELU / residual / GELU' and store.
// Two accumulators (2 x BN TMEM columns) let the epilogue of one tile overlap
// the main loop of the next.  Tiles are visited in groups of m-tiles so the
// B operand (the weights) is reused from L2 by concurrently running CTAs.
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

#include "gemm.cuh"

namespace gpt2k {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 32;                 // fp32 per k-block: one 128-byte swizzle row
constexpr int UMMA_K = 8;              // K of one tf32 MMA
constexpr int THREADS = 192;
constexpr int ATOM_BYTES = 32 * BK * 4;   // one MN-major box: 32 MN x 32 k = 4 KB
constexpr unsigned long long WAIT_NS = 1000000000ull;   // 1 s

template <int BN>
struct Shape {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_BYTES = BN * BK * 4;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 1024 + 256;
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
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait.  Returns false when this CTA is aborting (timeout here or elsewhere).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; i++) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > WAIT_NS) {
                *abort_flag = 1;
                set_status(status, GPT2_STATUS_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// UMMA shared-memory descriptor: start address, leading / stride byte offsets,
// version 1 (bits 46-47), swizzle layout type in bits 61-63 (2: 128-byte
// swizzle of 16-byte chunks; 1: 128-byte swizzle of 32-byte chunks).
constexpr uint32_t LAYOUT_SW128 = 2, LAYOUT_SW128_32B = 1;

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(layout & 7u) << 61;
    return d;
}

// Instruction descriptor, kind::tf32: D fp32 (bits 4-5 = 1), A and B tf32
// (bits 7-9, 10-12 = 2), majorness bits 15 (A) and 16 (B), N>>3 at bit 17,
// M>>4 at bit 24.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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
template <bool PARTIAL>
__device__ __forceinline__ void store_row(const Params& p, int row, int n, int split,
                                          const uint32_t (&r)[32]) {
    if (PARTIAL) {
        float* out = p.partial + ((size_t)split * p.M + row) * p.N + n;
        if (n + 32 <= p.N && (p.N & 3) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(out + j) =
                    make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        } else {
            for (int j = 0; j < 32 && n + j < p.N; j++) out[j] = __uint_as_float(r[j]);
        }
        return;
    }
    const GemmEpilogue& e = p.e;
    const bool vec = n + 32 <= p.N && (e.ldo & 3) == 0 && (!e.gelu_x || (e.ldg & 3) == 0);
    if (vec) {
        size_t o = (size_t)row * e.ldo + n;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float v[4] = {__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                          __uint_as_float(r[j + 3])};
            if (e.bias) {
#pragma unroll
                for (int k = 0; k < 4; k++) v[k] += __ldg(e.bias + n + j + k);
            }
            if (e.gelu) {
                *reinterpret_cast<float4*>(e.out_pre + o + j) = make_float4(v[0], v[1], v[2], v[3]);
#pragma unroll
                for (int k = 0; k < 4; k++) v[k] = gelu_fwd(v[k]);
            }
            if (e.residual) {
                float4 rr = *reinterpret_cast<const float4*>(e.residual + o + j);
                v[0] += rr.x; v[1] += rr.y; v[2] += rr.z; v[3] += rr.w;
            }
            if (e.gelu_x) {
                float4 h = *reinterpret_cast<const float4*>(e.gelu_x + (size_t)row * e.ldg + n + j);
                v[0] *= gelu_grad(h.x); v[1] *= gelu_grad(h.y);
                v[2] *= gelu_grad(h.z); v[3] *= gelu_grad(h.w);
            }
            *reinterpret_cast<float4*>(e.out + o + j) = make_float4(v[0], v[1], v[2], v[3]);
        }
    } else {
        for (int j = 0; j < 32 && n + j < p.N; j++) epilogue_store(e, row, n + j, __uint_as_float(r[j]));
    }
}

// ---------------------------------------------------------------- kernel
template <int BN>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tf32_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const Params p) {
    using S = Shape<BN>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[S::STAGES], empty_bar[S::STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
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
            mbar_init(smem_u32(&tempty_bar[a]), 4);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_map(&tmA);
        prefetch_map(&tmB);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(S::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s_tmem;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_phase = 0;   // per-stage bits, for the abort drain
            bool ok = true;
            for (long long u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                Unit c = unit_coords(p, u);
                const int m0 = c.m_tile * BM, n0 = c.n_tile * BN;
                const int kb0 = c.split * p.kb_per_split;
                const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u, &s_abort, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_expect_tx(fb, S::STAGE_BYTES);
                    armed |= 1u << stage;
                    armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                    const int k0 = kb * BK;
                    if (p.a_kmajor) {
                        tma_load_2d(stage_a(stage), &tmA, k0, m0, fb);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 32; j++)
                            tma_load_2d(stage_a(stage) + j * ATOM_BYTES, &tmA, m0 + 32 * j, k0, fb);
                    }
                    if (p.b_kmajor) {
                        tma_load_2d(stage_b(stage), &tmB, k0, n0, fb);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 32; j++)
                            tma_load_2d(stage_b(stage) + j * ATOM_BYTES, &tmB, n0 + 32 * j, k0, fb);
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
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = instr_desc(BM, BN, !p.a_kmajor, !p.b_kmajor);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (long long u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
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
                    for (int k = 0; k < BK / UMMA_K; k++) {
                        uint64_t ad = p.a_kmajor
                                          ? smem_desc(a0 + k * 32, 16, 1024, LAYOUT_SW128)
                                          : smem_desc(a0 + k * 1024, p.mn_lbo, p.mn_sbo, p.mn_layout);
                        uint64_t bd = p.b_kmajor
                                          ? smem_desc(b0 + k * 32, 16, 1024, LAYOUT_SW128)
                                          : smem_desc(b0 + k * 1024, p.mn_lbo, p.mn_sbo, p.mn_layout);
                        mma_tf32(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&empty_bar[stage]));
                    if (++stage == S::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(smem_u32(&tfull_bar[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // every MMA this thread issued has completed once drain_bar fires
            mma_commit(smem_u32(&drain_bar));
            uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(&drain_bar), 0) && globaltimer() - t0 < WAIT_NS) {
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        int acc = 0;
        uint32_t acc_phase = 0;
        for (long long u = blockIdx.x; u < p.units; u += gridDim.x) {
            Unit c = unit_coords(p, u);
            const int m0 = c.m_tile * BM, n0 = c.n_tile * BN;
            if (!mbar_wait(smem_u32(&tfull_bar[acc]), acc_phase, &s_abort, p.status)) break;
            tc_fence_after();
            const int row = m0 + q * 32 + lane;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            for (int cc = 0; cc < BN; cc += 32) {
                if (n0 + cc >= p.N) break;
                uint32_t r[32];
                tmem_ld32(taddr + (uint32_t)cc, r);
                if (row < p.M) {
                    if (p.partial) store_row<true>(p, row, n0 + cc, c.split, r);
                    else store_row<false>(p, row, n0 + cc, c.split, r);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(S::TMEM_COLS)
                     : "memory");
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

// 2-D fp32 tensor map over a row-major matrix [rows, cols] with row stride
// `ld` elements; box {box_cols, box_rows}, zero fill.  K-major operands use the
// 128-byte swizzle of 16-byte chunks; MN-major operands the 128-byte swizzle of
// 32-byte chunks, the layout the tensor core reads tf32 MN-major tiles in.
static bool make_map(CUtensorMap* map, const float* ptr, int cols, int rows, int ld, int box_cols,
                     int box_rows, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(float)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MN-major operand tiles: boxes of 32 MN x 32 k (4 KB) side by side along MN;
// within a box, k-rows of 128 bytes whose 32-byte chunks are swizzled over a
// period of 4 rows.  Descriptor: LBO = stride between MN boxes, SBO = stride
// between 4-row k groups.
constexpr uint32_t MN_LBO = ATOM_BYTES, MN_SBO = 4 * 128;

template <int BN>
static int prepare(const GemmProblem& g, const GemmEpilogue& e, float* partial, int split,
                   CUtensorMap* ma, CUtensorMap* mb, Params* pp) {
    using S = Shape<BN>;
    static bool attr_done = false;
    if (!attr_done) {
        if (cudaFuncSetAttribute(gemm_tf32_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)S::SMEM) != cudaSuccess) {
            (void)cudaGetLastError();
            return GPT2_ECUDA;
        }
        attr_done = true;
    }
    const CUtensorMapSwizzle KSW = CU_TENSOR_MAP_SWIZZLE_128B, MSW = CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
    // A: K-major [M, K] (box {32, 128}); M-major [K, M] (box {32, 32})
    bool ok = g.a_kmajor ? make_map(ma, g.A, g.K, g.M, g.lda, BK, BM, KSW)
                         : make_map(ma, g.A, g.M, g.K, g.lda, 32, BK, MSW);
    ok = ok && (g.b_kmajor ? make_map(mb, g.B, g.K, g.N, g.ldb, BK, BN, KSW)
                           : make_map(mb, g.B, g.N, g.K, g.ldb, 32, BK, MSW));
    if (!ok) return GPT2_ENOTSUP;
    Params p{};
    p.M = g.M; p.N = g.N; p.K = g.K;
    p.a_kmajor = g.a_kmajor; p.b_kmajor = g.b_kmajor;
    p.tiles_m = ceil_div(g.M, BM);
    p.tiles_n = ceil_div(g.N, BN);
    p.num_kb = ceil_div(g.K, BK);
    p.split = split;
    p.kb_per_split = ceil_div(p.num_kb, split);
    if (ceil_div(p.num_kb, p.kb_per_split) != split) return GPT2_EINVAL;   // an empty K slice
    p.units = (long long)p.tiles_m * p.tiles_n * split;
    // group enough m-tiles that their A rows stay in L2 while B streams past
    p.group_m = std::max(1, std::min(p.tiles_m, 16));
    p.e = e;
    p.partial = partial;
    p.status = g.status;
    p.mn_layout = LAYOUT_SW128_32B;
    p.mn_lbo = MN_LBO;
    p.mn_sbo = MN_SBO;
    *pp = p;
    return GPT2_OK;
}

template <int BN>
static int run(const CUtensorMap& ma, const CUtensorMap& mb, const Params& p, cudaStream_t st) {
    int grid = (int)std::min<long long>(p.units, num_sms());
    count_launch(), gemm_tf32_kernel<BN><<<grid, THREADS, Shape<BN>::SMEM, st>>>(ma, mb, p);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

template <int BN>
static int launch(const GemmProblem& g, const GemmEpilogue& e, float* partial, int split,
                  cudaStream_t st) {
    CUtensorMap ma, mb;
    Params p;
    int rc = prepare<BN>(g, e, partial, split, &ma, &mb, &p);
    if (rc) return rc;
    return run<BN>(ma, mb, p, st);
}

}  // namespace tc

bool gemm_tc_supported(const GemmProblem& p) {
    if (p.M < 1 || p.N < 1 || p.K < 1) return false;
    if (!aligned16(p.A) || !aligned16(p.B) || (p.lda & 3) || (p.ldb & 3)) return false;
    return tc::encode_fn() != nullptr;
}

int gemm_tc(const GemmProblem& p, const GemmEpilogue& e, cudaStream_t st) {
    if (p.N <= 128) return tc::launch<128>(p, e, nullptr, 1, st);
    return tc::launch<256>(p, e, nullptr, 1, st);
}

int gemm_tc_splitk(const GemmProblem& p, float* partial, int split, cudaStream_t st) {
    GemmEpilogue e{};
    if (p.N <= 128) return tc::launch<128>(p, e, partial, split, st);
    return tc::launch<256>(p, e, partial, split, st);
}

}  // namespace gpt2k
