// linear.cu -- the linear layer (nn_linear convention, W is [out, in]) and its
// two backward products, dispatched to the CUDA-core or the tcgen05 GEMM, plus
// the deterministic bias-gradient reduction.
//
// Forward out = inp . W^T + b with the epilogues the block needs fused in
// (bias, tanh-GELU keeping its input, residual add): "GPT-2 from scratch with
// torch", sections 自注意力 (c_attn, c_proj) and 前馈网络（MLP）(c_fc, GELU,
// c_proj).  Backward (hand-derived): dinp = dout . W, dW = dout^T . inp,
// db = column sums of dout.
#include <mutex>

#include <cuda_bf16.h>

#include "gemm.cuh"

namespace gpt2k {

// ---- bias gradient: db[o] = sum_n dout[n*ld + o], fixed order -------------
// Stage 1: block (32 x 8) covers 128 columns (4 per thread, one vector load per
// row) of one chunk of rows; lane y sums rows y, y+8, ... of the chunk in order;
// the 8 lanes are combined in order.  Stage 2 sums the chunks in order.
constexpr int BG_ROWS = 256;

template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
template <typename T>
__device__ __forceinline__ float to_f(T v) { return (float)v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__global__ void bias_grad_partial_kernel(float* __restrict__ partial, const T* __restrict__ dout,
                                         int N, int OC, int ld, int nchunk) {
    __shared__ float4 sh[8][33];
    const int col = (blockIdx.x * 32 + threadIdx.x) * 4;
    // vector loads need the 4 columns inside the row, an aligned row stride and
    // an aligned base (a column slice of a wider matrix may start anywhere)
    const bool vec = col + 4 <= OC && (ld & 3) == 0 &&
                     (reinterpret_cast<uintptr_t>(dout) & (4 * sizeof(T) - 1)) == 0;
    // chunks of BG_ROWS rows, grid-strided over blockIdx.y (at most 65535 blocks high)
    for (int chunk = blockIdx.y; chunk < nchunk; chunk += gridDim.y) {
        const int r0 = chunk * BG_ROWS, r1 = min(N, r0 + BG_ROWS);
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < OC) {
            if (vec) {
#pragma unroll 4
                for (int r = r0 + threadIdx.y; r < r1; r += 8) {
                    const float4 v = load4(dout + (size_t)r * ld + col);
                    s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
                }
            } else {
                for (int r = r0 + threadIdx.y; r < r1; r += 8) {
                    const T* row = dout + (size_t)r * ld + col;
                    s.x += to_f(row[0]);
                    if (col + 1 < OC) s.y += to_f(row[1]);
                    if (col + 2 < OC) s.z += to_f(row[2]);
                    if (col + 3 < OC) s.w += to_f(row[3]);
                }
            }
        }
        sh[threadIdx.y][threadIdx.x] = s;
        __syncthreads();
        if (threadIdx.y == 0 && col < OC) {
            float4 t = sh[0][threadIdx.x];
            for (int k = 1; k < 8; k++) {
                const float4 u = sh[k][threadIdx.x];
                t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
            }
            float* out = partial + (size_t)chunk * OC + col;
            out[0] = t.x;
            if (col + 1 < OC) out[1] = t.y;
            if (col + 2 < OC) out[2] = t.z;
            if (col + 3 < OC) out[3] = t.w;
        }
        __syncthreads();
    }
}

__global__ void bias_grad_reduce_kernel(float* __restrict__ db, const float* __restrict__ partial,
                                        int nchunk, int OC) {
    int col = blockIdx.x * blockDim.x + threadIdx.x;
    if (col >= OC) return;
    float s = 0.f;
    for (int k = 0; k < nchunk; k++) s += partial[(size_t)k * OC + col];
    db[col] = s;
}

static size_t bias_scratch_bytes(int N, int OC) {
    return round_up((size_t)ceil_div(N, BG_ROWS) * OC * sizeof(float), 256);
}

template <typename T>
static int bias_grad(float* db, const T* dout, int N, int OC, int ld, float* scratch,
                     cudaStream_t st) {
    const int nchunk = ceil_div(N, BG_ROWS);
    count_launch(), bias_grad_partial_kernel<T><<<dim3(ceil_div(OC, 128), std::min(nchunk, 65535)), dim3(32, 8), 0,
                                                  st>>>(scratch, dout, N, OC, ld, nchunk);
    count_launch(), bias_grad_reduce_kernel<<<ceil_div(OC, 256), 256, 0, st>>>(db, scratch, nchunk, OC);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

// ---- column sums of per-group partial sums: db[c] = sum_g part[g][c] --------
// Block (32 columns x 32 lanes): lane y sums groups y, y+32, ... in order, then
// the 32 lane sums are added in lane order; one block per 32 columns.
__global__ void __launch_bounds__(1024) colsum_reduce_kernel(float* __restrict__ db, const float* __restrict__ part,
                                                             int groups, int OC) {
    __shared__ float sh[32][33];
    const int c = blockIdx.x * 32 + threadIdx.x;
    float s = 0.f;
    if (c < OC)
        for (int g = threadIdx.y; g < groups; g += 32) s += part[(size_t)g * OC + c];
    sh[threadIdx.y][threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.y == 0 && c < OC) {
        float t = sh[0][threadIdx.x];
        for (int k = 1; k < 32; k++) t += sh[k][threadIdx.x];
        db[c] = t;
    }
}

int colsum_reduce(float* db, const float* part, int groups, int OC, cudaStream_t st) {
    if (!db || !part || groups < 1 || OC < 1) return GPT2_EINVAL;
    count_launch(), colsum_reduce_kernel<<<ceil_div(OC, 32), dim3(32, 32), 0, st>>>(db, part, groups, OC);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

// ---- many column reductions in one launch ---------------------------------
// Block (32 columns x 16 lanes) per (reduction, 32 columns): lane y sums groups
// y, y+16, ... in order, then the 16 lane sums are added in lane order.
constexpr int COLB_MAX = 400;                    // reductions per launch (kernel parameter space)
struct ColReduceBatch {
    int n;
    ColReduce r[COLB_MAX];
};

__global__ void __launch_bounds__(512) colsum_batch_kernel(const __grid_constant__ ColReduceBatch b) {
    __shared__ float sh[16][33];
    const ColReduce& r = b.r[blockIdx.y];
    const int c = blockIdx.x * 32 + threadIdx.x;
    float s = 0.f;
    if (c < r.width)
        for (int g = threadIdx.y; g < r.groups; g += 16) s += r.part[(size_t)g * r.ld + c];
    sh[threadIdx.y][threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.y == 0 && c < r.width) {
        float t = sh[0][threadIdx.x];
        for (int k = 1; k < 16; k++) t += sh[k][threadIdx.x];
        r.dst[c / r.seg][c % r.seg] = t;
    }
}

int colsum_batch(const ColReduce* r, int n, cudaStream_t st) {
    for (int i0 = 0; i0 < n; i0 += COLB_MAX) {
        ColReduceBatch b;
        b.n = std::min(COLB_MAX, n - i0);
        int wmax = 1;
        for (int i = 0; i < b.n; i++) {
            b.r[i] = r[i0 + i];
            wmax = std::max(wmax, b.r[i].width);
        }
        count_launch(), colsum_batch_kernel<<<dim3(ceil_div(wmax, 32), b.n), dim3(32, 16), 0, st>>>(b);
        GPT2_LAUNCH_CHECK();
    }
    return GPT2_OK;
}

// ---- split-K sum: out[i] = sum_s partial[s][i], in slice order -------------
__global__ void splitk_reduce_kernel(float4* __restrict__ out, const float4* __restrict__ partial,
                                     int split, size_t n4) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4 s = partial[i];
    for (int k = 1; k < split; k++) {
        float4 v = partial[(size_t)k * n4 + i];
        s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    out[i] = s;
}

// Number of K slices for the tensor-core dW product (M = OC, N = IC, K = the N
// rows), from a small cost model in microseconds: waves of units times the
// k-blocks of a unit (about 0.45 us per 128 x 256 x 128-byte k-block on one
// SM) plus about 1 us per wave of prologue and exposed epilogue, plus the fp32
// partial slices written and summed again (S + 1 tile-sized passes at about
// 5 TB/s).  More slices fill more SMs but move more partial bytes; no slice
// is left empty.
static int dw_split(int N, int IC, int OC, int mode) {
    // the product is M = OC, N = IC, K = N rows; CTA pairs take 256 x 256 tiles
    // (a pair moves through a k-block in the time one CTA takes for 128 x 256)
    GemmProblem probe{OC, IC, N, nullptr, 0, false, nullptr, 0, false, nullptr, mode == GPT2_MODE_BF16};
    const bool pair = gemm_tc_pair(probe, nullptr);
    const int bm = pair ? 256 : 128, bn = (IC <= 128 && !pair) ? 128 : 256;
    const long long tiles = (long long)ceil_div(OC, bm) * ceil_div(IC, bn);
    const int nkb = ceil_div(N, mode == GPT2_MODE_BF16 ? 64 : 32);
    const double t_kb = 0.45 * bn / 256.0, t_wave = 1.0, bytes_per_us = 5.0e6;
    const double tile_bytes = (double)bm * bn * 4.0;
    const long long sms = pair ? gemm_tc_pair_slots() : num_sms();
    int best = 1;
    double best_t = 0.0;
    for (int split = 1; split <= 16; split++) {
        const int kbps = ceil_div(nkb, split);
        if (ceil_div(nkb, kbps) != split) continue;          // a slice would be empty
        const long long waves = (tiles * split + sms - 1) / sms;
        double t = (double)waves * (kbps * t_kb + t_wave);
        if (split > 1) t += (split + 1) * (double)tiles * tile_bytes / bytes_per_us;
        if (split == 1 || t < best_t) {
            best_t = t;
            best = split;
        }
    }
    return best;
}

static int run_gemm(const GemmProblem& p, const GemmEpilogue& e, int mode, cudaStream_t st) {
    if (p.bf16) {
        if (mode != GPT2_MODE_BF16 || !gemm_tc_supported(p) || !gemm_tc_epilogue_supported(e))
            return GPT2_ENOTSUP;
        return gemm_tc(p, e, st);
    }
    if (mode == GPT2_MODE_FP32) return gemm_simt(p, e, st);
    if (mode == GPT2_MODE_TF32) {
        // operands TMA cannot address (unaligned base or row stride) take the CUDA cores
        if (!gemm_tc_supported(p) || !gemm_tc_epilogue_supported(e)) return gemm_simt(p, e, st);
        return gemm_tc(p, e, st);
    }
    return GPT2_EINVAL;
}

// ---- the three products of a linear layer, for every operand type ---------
int linear_forward(void* out, bool out_bf16, void* out_pre, const void* inp, const void* w,
                   bool bf16, const float* bias, const float* residual, int N, int IC, int OC,
                   int ld_out, int flags, int mode, int* status, cudaStream_t st) {
    if (!out || !inp || !w || N < 1 || IC < 1 || OC < 1 || ld_out < OC) return GPT2_EINVAL;
    if ((flags & GPT2_LINEAR_GELU) && (!out_pre || residual)) return GPT2_EINVAL;
    GemmProblem p{N, OC, IC, inp, IC, true, w, IC, true, status, bf16};
    GemmEpilogue e{};
    e.out = out;
    e.ldo = ld_out;
    e.out_bf16 = out_bf16;
    e.out_pre = out_pre;
    e.pre_bf16 = bf16 ? 1 : 0;
    e.bias = bias;
    e.residual = residual;
    e.gelu = (flags & GPT2_LINEAR_GELU) ? 1 : 0;
    int rc = run_gemm(p, e, mode, st);
    if (rc) return rc;
    if ((flags & GPT2_LINEAR_ZERO_PAD) && ld_out > OC) {
        const size_t es = out_bf16 ? 2 : 4;
        GPT2_CUDA_TRY(cudaMemset2DAsync(static_cast<char*>(out) + OC * es, (size_t)ld_out * es, 0,
                                        (size_t)(ld_out - OC) * es, N, st));
    }
    return GPT2_OK;
}

// Bytes of the column-sum buffer of linear_backward_input for a bias gradient.
size_t linear_colsum_bytes(int N, int IC) {
    return std::max(round_up((size_t)ceil_div(N, 32) * IC * sizeof(float), 256), bias_scratch_bytes(N, IC));
}

// K slices for a plain dX product (fp32 output, no GELU' or bias sums), by the
// dW cost model (M = N rows, N = IC, K = OC): few row tiles and a long K (the
// lm_head at small B·T) leave most SMs idle without it.  Scratch for the slices.
static int dx_split(int N, int IC, int OC, int mode) {
    return mode == GPT2_MODE_FP32 ? 1 : dw_split(OC, IC, N, mode);
}
size_t linear_backward_input_scratch_bytes(int N, int IC, int OC, int mode) {
    size_t s = 0;
    for (int n = N; n >= 1; n = n / 2) {               // every row count up to N
        const int split = dx_split(n, IC, OC, mode);
        if (split > 1) s = std::max(s, (size_t)split * n * IC * sizeof(float));
        if (n == 1) break;
    }
    return s;
}

int linear_backward_input(void* dinp, bool dinp_bf16, const void* dout, const void* w, bool bf16,
                          const void* gelu_x, int N, int IC, int OC, int ld_dout, int mode,
                          int* status, cudaStream_t st, float* db, void* cs, size_t cs_bytes, ColReduce* defer,
                          void* ks, size_t ks_bytes) {
    if (defer) defer->part = nullptr;
    if (!dinp || !dout || !w || N < 1 || IC < 1 || OC < 1 || ld_dout < OC) return GPT2_EINVAL;
    if (db && (!cs || cs_bytes < linear_colsum_bytes(N, IC))) return GPT2_ENOMEM;
    GemmProblem p{N, IC, OC, dout, ld_dout, true, w, IC, false, status, bf16};
    if (ks && !gelu_x && !db && !dinp_bf16) {
        // split K over fp32 partial slices summed in slice order
        const int split = dx_split(N, IC, OC, mode);
        if (split > 1 && (size_t)split * N * IC * sizeof(float) <= ks_bytes && gemm_tc_supported(p) &&
            (size_t)N * IC % 4 == 0 && aligned16(dinp)) {
            float* partial = reinterpret_cast<float*>(ks);
            int rc = gemm_tc_splitk(p, partial, split, st);
            if (rc) return rc;
            const size_t n4 = (size_t)N * IC / 4;
            count_launch(), splitk_reduce_kernel<<<ceil_div((long long)n4, 256), 256, 0, st>>>(
                reinterpret_cast<float4*>(dinp), reinterpret_cast<const float4*>(partial), split, n4);
            GPT2_LAUNCH_CHECK();
            return GPT2_OK;
        }
    }
    GemmEpilogue e{};
    e.out = dinp;
    e.ldo = IC;
    e.out_bf16 = dinp_bf16;
    e.gelu_x = gelu_x;
    e.gelu_x_bf16 = bf16 ? 1 : 0;
    e.ldg = IC;
    // the tensor-core epilogue leaves per-32-row column sums of dinp in cs; the
    // bias gradient is then their sum over the groups, in group order
    const bool fused = db && (bf16 || (mode == GPT2_MODE_TF32 && gemm_tc_supported(p) &&
                                       gemm_tc_epilogue_supported(e)));
    const int groups = ceil_div(N, 32);
    float* part = static_cast<float*>(cs);
    if (fused) e.colsum = part;
    int rc = run_gemm(p, e, mode, st);
    if (rc || !db) return rc;
    if (fused && defer) {
        *defer = ColReduce{part, groups, IC, IC, IC, {db, nullptr, nullptr}};
        return GPT2_OK;
    }
    if (fused) return colsum_reduce(db, part, groups, IC, st);
    if (dinp_bf16) return bias_grad(db, static_cast<const __nv_bfloat16*>(dinp), N, IC, IC, part, st);
    return bias_grad(db, static_cast<const float*>(dinp), N, IC, IC, part, st);
}

int linear_backward_weight(float* dw, const void* dout, const void* inp, bool bf16, int N, int IC,
                           int OC, int ld_dout, void* scratch, size_t scratch_bytes, int mode,
                           int* status, cudaStream_t st) {
    if (!dw || !dout || !inp || N < 1 || IC < 1 || OC < 1 || ld_dout < OC) return GPT2_EINVAL;
    if (scratch_bytes < gpt2_op_linear_backward_weight_scratch_bytes(N, IC, OC, mode) || !scratch)
        return GPT2_ENOMEM;
    GemmProblem p{OC, IC, N, dout, ld_dout, false, inp, IC, false, status, bf16};
    int split = mode != GPT2_MODE_FP32 ? dw_split(N, IC, OC, mode) : 1;
    if (split > 1 && gemm_tc_supported(p) && (size_t)OC * IC % 4 == 0 && aligned16(dw)) {
        float* partial = reinterpret_cast<float*>(scratch);
        int rc = gemm_tc_splitk(p, partial, split, st);
        if (rc) return rc;
        size_t n4 = (size_t)OC * IC / 4;
        count_launch(), splitk_reduce_kernel<<<ceil_div((long long)n4, 256), 256, 0, st>>>(
            reinterpret_cast<float4*>(dw), reinterpret_cast<const float4*>(partial), split, n4);
        GPT2_LAUNCH_CHECK();
        return GPT2_OK;
    }
    GemmEpilogue e{};
    e.out = dw;
    e.ldo = IC;
    return run_gemm(p, e, mode, st);
}

int bias_grad_any(float* db, const void* dout, bool bf16, int N, int OC, int ld, void* scratch,
                  size_t scratch_bytes, cudaStream_t st) {
    if (!db || !dout || N < 1 || OC < 1 || ld < OC) return GPT2_EINVAL;
    if (!scratch || scratch_bytes < bias_scratch_bytes(N, OC)) return GPT2_ENOMEM;
    float* sc = reinterpret_cast<float*>(scratch);
    if (bf16) return bias_grad(db, static_cast<const __nv_bfloat16*>(dout), N, OC, ld, sc, st);
    return bias_grad(db, static_cast<const float*>(dout), N, OC, ld, sc, st);
}

}  // namespace gpt2k

using namespace gpt2k;

GPT2_API int gpt2_op_linear_forward(float* out, float* out_pre, const float* inp, const float* w,
                                    const float* bias, const float* residual, int N, int IC, int OC,
                                    int ld_out, int flags, int mode, int* status, void* stream) {
    if (mode == GPT2_MODE_BF16) return GPT2_EINVAL;
    return linear_forward(out, false, out_pre, inp, w, false, bias, residual, N, IC, OC, ld_out, flags,
                          mode, status, as_stream(stream));
}

GPT2_API int gpt2_op_linear_backward_input(float* dinp, const float* dout, const float* w,
                                           const float* gelu_x, int N, int IC, int OC, int ld_dout,
                                           int mode, int* status, void* stream) {
    if (mode == GPT2_MODE_BF16) return GPT2_EINVAL;
    return linear_backward_input(dinp, false, dout, w, false, gelu_x, N, IC, OC, ld_dout, mode, status,
                                 as_stream(stream));
}

GPT2_API size_t gpt2_op_linear_backward_weight_scratch_bytes(int N, int IC, int OC, int mode) {
    if (N < 1 || IC < 1 || OC < 1) return 0;
    size_t s = bias_scratch_bytes(N, OC);
    if (mode != GPT2_MODE_FP32) {
        int split = dw_split(N, IC, OC, mode);
        if (split > 1) s = std::max(s, (size_t)split * OC * IC * sizeof(float));
    }
    return s;
}

GPT2_API int gpt2_op_linear_backward_weight(float* dw, float* dbias, const float* dout,
                                            const float* inp, int N, int IC, int OC, int ld_dout,
                                            void* scratch, size_t scratch_bytes, int mode,
                                            int* status, void* stream) {
    if (mode == GPT2_MODE_BF16) return GPT2_EINVAL;
    cudaStream_t st = as_stream(stream);
    int rc = linear_backward_weight(dw, dout, inp, false, N, IC, OC, ld_dout, scratch, scratch_bytes,
                                    mode, status, st);
    if (rc) return rc;
    if (dbias) return bias_grad(dbias, dout, N, OC, ld_dout, reinterpret_cast<float*>(scratch), st);
    return GPT2_OK;
}

GPT2_API int gpt2_op_gemm(const gpt2_gemm_args* a, int mode, int* status, void* stream) {
    if (!a || !a->A || !a->B || !a->out || a->M < 1 || a->N < 1 || a->K < 1 || a->ldo < a->N)
        return GPT2_EINVAL;
    if (a->bf16 && mode != GPT2_MODE_BF16) return GPT2_EINVAL;
    if (a->gelu && (!a->out_pre || a->residual)) return GPT2_EINVAL;
    GemmProblem p{a->M, a->N, a->K, a->A, a->lda, a->a_kmajor != 0, a->B, a->ldb, a->b_kmajor != 0,
                  status, a->bf16 != 0};
    GemmEpilogue e{};
    e.out = a->out;
    e.ldo = a->ldo;
    e.out_bf16 = a->out_bf16;
    e.out_pre = a->out_pre;
    e.pre_bf16 = a->pre_bf16;
    e.bias = a->bias;
    e.residual = a->residual;
    e.gelu_x = a->gelu_x;
    e.gelu_x_bf16 = a->gelu_x_bf16;
    e.ldg = a->ldg;
    e.gelu = a->gelu;
    e.colsum = a->colsum;
    if (e.colsum && !(p.bf16 || (mode == GPT2_MODE_TF32 && gemm_tc_supported(p) && gemm_tc_epilogue_supported(e))))
        return GPT2_ENOTSUP;
    return run_gemm(p, e, mode, as_stream(stream));
}

GPT2_API size_t gpt2_op_bias_grad_scratch_bytes(int N, int OC) {
    if (N < 1 || OC < 1) return 0;
    return bias_scratch_bytes(N, OC);
}

GPT2_API int gpt2_op_bias_grad(float* db, const void* dout, int dout_bf16, int N, int OC,
                               int ld_dout, void* scratch, size_t scratch_bytes, void* stream) {
    if (!db || !dout || N < 1 || OC < 1 || ld_dout < OC) return GPT2_EINVAL;
    if (!scratch || scratch_bytes < bias_scratch_bytes(N, OC)) return GPT2_ENOMEM;
    float* sc = reinterpret_cast<float*>(scratch);
    if (dout_bf16)
        return bias_grad(db, static_cast<const __nv_bfloat16*>(dout), N, OC, ld_dout, sc, as_stream(stream));
    return bias_grad(db, static_cast<const float*>(dout), N, OC, ld_dout, sc, as_stream(stream));
}

// ---- allocation-free bias gradient ----------------------------------------
// The partial sums live in this file-scope device array instead of caller
// scratch.  Host code must not pass the symbol itself to a kernel (on the host
// it names a stand-in, not device memory): its device address is looked up
// once per device with cudaGetSymbolAddress and cached.
static __device__ __align__(256) float g_bias_scratch[GPT2_BIAS_GRAD_NOALLOC_MAX_PARTIALS];

namespace gpt2k {
constexpr int NOALLOC_MAX_DEVICES = 64;
static std::mutex g_noalloc_mu;
static float* g_noalloc_ptr[NOALLOC_MAX_DEVICES];

static int noalloc_scratch(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { (void)cudaGetLastError(); return GPT2_ECUDA; }
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return GPT2_ENOTSUP;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bias_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return GPT2_ECUDA;
        }
        g_noalloc_ptr[dev] = reinterpret_cast<float*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return GPT2_OK;
}
}  // namespace gpt2k

GPT2_API int gpt2_op_bias_grad_noalloc(float* db, const float* dout, int N, int OC, int ld_dout,
                                       void* stream) {
    if (!db || !dout || N < 1 || OC < 1 || ld_dout < OC) return GPT2_EINVAL;
    if ((size_t)ceil_div(N, BG_ROWS) * (size_t)OC > GPT2_BIAS_GRAD_NOALLOC_MAX_PARTIALS)
        return GPT2_ENOMEM;
    float* scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    return bias_grad(db, dout, N, OC, ld_dout, scratch, as_stream(stream));
}
