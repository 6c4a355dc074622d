// encoder.cu -- token + position embedding, forward and deterministic backward.
//
// Forward: x[b,t,:] = wte[tok[b,t],:] + wpe[t,:]  ("GPT-2 from scratch with
// torch", section 从词到编码: the two embeddings are added).
//
// Backward: dwte[v,:] += sum_{pos: tok[pos]=v} dx[pos,:] and dwpe[t,:] =
// sum_b dx[b,t,:].  The token-side scatter-add is made deterministic without
// float atomics: positions are bucketed by token id with an integer counting
// sort (histogram, a two-pass scan, fill) and each bucket is put in ascending
// position order: small buckets by counting, per position, the bucket entries
// below it; buckets of more than ENC_BIG entries by a bitmap of positions in
// shared memory, one block each.  The sorted list is then cut into fixed
// segments of ENC_SEG entries, one thread block each: a bucket that lies inside
// one segment is summed and added to dwte there; a bucket that crosses segment
// boundaries leaves one partial sum per segment, and a fix-up pass adds those
// in a fixed order.  A frequent token (a Zipf stream gives the top id ~14% of
// positions) is thus spread over many blocks.
#include "common.cuh"

namespace gpt2k {

__global__ void encoder_fwd_kernel(float4* __restrict__ x, const int* __restrict__ tok,
                                   const float4* __restrict__ wte, const float4* __restrict__ wpe,
                                   int BT, int T, int C4, int V, int* status) {
    long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)BT * C4) return;
    int row = (int)(idx / C4), c = (int)(idx % C4);
    int t = row % T;
    int id = tok[row];
    if (id < 0 || id >= V) {
        if (c == 0) set_status(status, GPT2_STATUS_BAD_TOKEN);
        x[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    float4 e = wte[(size_t)id * C4 + c];
    float4 p = wpe[(size_t)t * C4 + c];
    x[idx] = make_float4(e.x + p.x, e.y + p.y, e.z + p.z, e.w + p.w);
}

// ---- counting sort of positions by token id -------------------------------

__global__ void enc_histogram_kernel(int* __restrict__ count, const int* __restrict__ tok, int BT,
                                     int V) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BT) return;
    int id = tok[i];
    if (id >= 0 && id < V) atomicAdd(&count[id], 1);
}

constexpr int ENC_BIG = 256;           // buckets above this size are ordered by a bitmap
constexpr int ENC_SCAN_BLOCK = 1024;   // ids per block of the scan
constexpr int ENC_BITMAP_MAX_BT = 1 << 20;   // positions a shared-memory bitmap covers (128 KB)

// Exclusive scan of one value per thread over the block (at most 32 warps):
// warp shuffles, then the warp totals; returns the block total in `total`.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nwarps ? s_warp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        if (lane < nwarps) s_warp[lane] = wi - w;     // exclusive prefix of the warp totals
        if (lane == 31) s_warp[32] = wi;
    }
    __syncthreads();
    const int r = s_warp[warp] + inc - v;
    total = s_warp[32];
    __syncthreads();                         // s_warp is reused by the next call
    return r;
}

// The scan of count[0..V) in two passes over blocks of ENC_SCAN_BLOCK ids.
// Pass 1: per block, the number of positions and of ids with more than
// ENC_BIG positions.
__global__ void __launch_bounds__(ENC_SCAN_BLOCK) enc_scan_sums_kernel(int* __restrict__ sums,
                                                                      const int* __restrict__ count, int V) {
    __shared__ int s_warp[33];
    const int v = blockIdx.x * ENC_SCAN_BLOCK + threadIdx.x;
    const int c = v < V ? count[v] : 0;
    int tot, totb;
    block_exclusive_scan(c, s_warp, tot);
    block_exclusive_scan(c > ENC_BIG ? 1 : 0, s_warp, totb);
    if (threadIdx.x == 0) {
        sums[2 * blockIdx.x] = tot;
        sums[2 * blockIdx.x + 1] = totb;
    }
}

// Pass 2: each block adds the sums of the blocks before it, then writes
// offset[] (exclusive scan of count; offset[V] = the total) and the ids with
// more than ENC_BIG positions, in increasing order, into big[] (*n_big).
__global__ void __launch_bounds__(ENC_SCAN_BLOCK) enc_scan_kernel(int* __restrict__ offset, int* __restrict__ big,
                                                                 int* __restrict__ n_big,
                                                                 const int* __restrict__ count,
                                                                 const int* __restrict__ sums, int V) {
    __shared__ int s_warp[33], s_pre[2];
    if (threadIdx.x < 32) {                   // warp 0: the two sums over the blocks before this one
#pragma unroll
        for (int q = 0; q < 2; q++) {
            int a = 0;
            for (int k = threadIdx.x; k < (int)blockIdx.x; k += 32) a += sums[2 * k + q];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (threadIdx.x == 0) s_pre[q] = a;
        }
    }
    const int v = blockIdx.x * ENC_SCAN_BLOCK + threadIdx.x;
    const int c = v < V ? count[v] : 0;
    int tot, totb;
    const int ex = block_exclusive_scan(c, s_warp, tot);          // its barriers also publish s_pre
    const int exb = block_exclusive_scan(c > ENC_BIG ? 1 : 0, s_warp, totb);
    const int run = s_pre[0], runb = s_pre[1];
    if (v < V) {
        offset[v] = run + ex;
        if (c > ENC_BIG) big[runb + exb] = v;
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
        offset[V] = run + tot;
        *n_big = runb + totb;
    }
}

__global__ void enc_fill_kernel(int* __restrict__ list, int* __restrict__ cursor,
                                const int* __restrict__ offset, const int* __restrict__ tok, int BT,
                                int V) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BT) return;
    int id = tok[i];
    if (id < 0 || id >= V) return;
    list[offset[id] + atomicAdd(&cursor[id], 1)] = i;
}

// Put each bucket in ascending position order: a position's rank in its bucket
// is the number of bucket entries smaller than it (positions are distinct).
__global__ void enc_rank_kernel(int* __restrict__ sorted, const int* __restrict__ list,
                                const int* __restrict__ offset, const int* __restrict__ tok, int BT,
                                int V, int skip_big) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BT) return;
    int id = tok[i];
    if (id < 0 || id >= V) return;
    int lo = offset[id], hi = offset[id + 1];
    if (skip_big && hi - lo > ENC_BIG) return;     // enc_sort_big_kernel orders this bucket
    int r = 0;
    for (int e = lo; e < hi; e++) r += list[e] < i;
    sorted[lo + r] = i;
}

// Buckets of more than ENC_BIG entries: one block per bucket (grid-strided over
// big[]) marks the bucket's positions (distinct, below BT) in a shared-memory
// bitmap of BT bits, then each thread takes a run of consecutive words, counts
// their bits, and after an exclusive scan of the counts writes its positions
// in ascending order to sorted[].
__global__ void __launch_bounds__(512) enc_sort_big_kernel(int* __restrict__ sorted, const int* __restrict__ list,
                                                          const int* __restrict__ offset,
                                                          const int* __restrict__ big,
                                                          const int* __restrict__ n_big, int BT) {
    extern __shared__ uint32_t s_bits[];
    __shared__ int s_warp[33];
    const int nw = (BT + 31) >> 5;
    const int wpt = (nw + blockDim.x - 1) / blockDim.x;      // words per thread
    const int w0 = min(nw, (int)threadIdx.x * wpt), w1 = min(nw, w0 + wpt);
    const int nb = *n_big;
    for (int k = blockIdx.x; k < nb; k += gridDim.x) {
        const int v = big[k];
        const int lo = offset[v], n = offset[v + 1] - lo;
        for (int i = threadIdx.x; i < nw; i += blockDim.x) s_bits[i] = 0u;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const int pos = list[lo + i];
            atomicOr(&s_bits[pos >> 5], 1u << (pos & 31));
        }
        __syncthreads();
        int cnt = 0;
        for (int w = w0; w < w1; w++) cnt += __popc(s_bits[w]);
        int tot;
        int at = lo + block_exclusive_scan(cnt, s_warp, tot);
        for (int w = w0; w < w1; w++) {
            uint32_t bits = s_bits[w];
            while (bits) {
                const int bpos = __ffs(bits) - 1;
                sorted[at++] = 32 * w + bpos;
                bits &= bits - 1;
            }
        }
        __syncthreads();                          // the bitmap is cleared for the next bucket
    }
}

constexpr int ENC_SEG = 16;
constexpr int ENC_FIX = 4;             // partial sums per fix-up thread loaded together ...
constexpr int ENC_FIX_Y = 4;           // ... by each of this many threads per column
constexpr int ENC_PF = 8;              // gradient rows loaded together in the segment kernel

// One block per segment of the sorted list.  All threads walk the segment's
// entries in order (same token sequence from shared memory), each thread for
// its own float4 columns, and flush the running sum at every token change.
__global__ void __launch_bounds__(256) enc_segment_kernel(float4* __restrict__ dwte, float4* __restrict__ part,
                                   const float4* __restrict__ dx, const int* __restrict__ sorted,
                                   const int* __restrict__ offset, const int* __restrict__ tok, int V,
                                   int C4) {
    __shared__ int s_pos[ENC_SEG], s_tok[ENC_SEG];
    const int seg = blockIdx.x, seg_lo = seg * ENC_SEG;
    const int total = offset[V];                   // sorted entries (positions with valid ids)
    const int cnt = min(ENC_SEG, total - seg_lo);
    if (cnt <= 0) return;
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
        const int pos = sorted[seg_lo + i];
        s_pos[i] = pos;
        s_tok[i] = tok[pos];
    }
    __syncthreads();
    for (int c = threadIdx.x; c < C4; c += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int run_start = 0;
        // the gradient rows of the segment, ENC_PF at a time: all loads of a group
        // are in flight together, then added in entry order
        float4 g[ENC_PF];
        for (int e0 = 0; e0 <= cnt; e0 += ENC_PF) {
#pragma unroll
            for (int k = 0; k < ENC_PF; k++)
                if (e0 + k < cnt) g[k] = __ldg(dx + (size_t)s_pos[e0 + k] * C4 + c);
#pragma unroll
            for (int k = 0; k < ENC_PF; k++) {
                const int e = e0 + k;
                if (e > cnt) break;
                if (e == cnt || (e > 0 && s_tok[e] != s_tok[e - 1])) {
                    const int v = s_tok[e - 1];
                    const int lo = offset[v], hi = offset[v + 1];
                    if (lo >= seg_lo && hi <= seg_lo + cnt) {        // whole bucket in this segment
                        float4 d = dwte[(size_t)v * C4 + c];
                        d.x += acc.x; d.y += acc.y; d.z += acc.z; d.w += acc.w;
                        dwte[(size_t)v * C4 + c] = d;
                    } else {                                       // slot 0: first run, 1: last run
                        part[((size_t)seg * 2 + (run_start == 0 ? 0 : 1)) * C4 + c] = acc;
                    }
                    if (e == cnt) break;
                    acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    run_start = e;
                }
                acc.x += g[k].x; acc.y += g[k].y; acc.z += g[k].z; acc.w += g[k].w;
            }
        }
    }
}

// Buckets that cross segments.  Block b looks at the boundary after segment b
// and takes the bucket that crosses it if that is the bucket's first boundary;
// it adds the bucket's per-segment partial sums into dwte.  Thread (x, y)
// takes column float4s x, x + blockDim.x, ... and segments s0 + y, s0 + y +
// ENC_FIX_Y, ..., with ENC_FIX interleaved running sums so that their loads are
// in flight together; the sums are added in a fixed order (k, then y through
// shared memory), so the result does not depend on timing.
__global__ void __launch_bounds__(1024) enc_fixup_kernel(float4* __restrict__ dwte, const float4* __restrict__ part,
                                 const int* __restrict__ sorted, const int* __restrict__ offset,
                                 const int* __restrict__ tok, int V, int C4) {
    __shared__ float4 s_acc[ENC_FIX_Y][256];
    const int bnd = blockIdx.x, e = (bnd + 1) * ENC_SEG;     // first entry after the boundary
    if (e >= offset[V]) return;
    const int v = tok[sorted[e]];
    if (tok[sorted[e - 1]] != v) return;                      // no bucket crosses here
    const int lo = offset[v], hi = offset[v + 1];
    const int s0 = lo / ENC_SEG, s1 = (hi - 1) / ENC_SEG;
    if (s0 != bnd) return;                                    // not the bucket's first boundary
    const int y = threadIdx.y;
    for (int c0 = 0; c0 < C4; c0 += blockDim.x) {
        const int c = c0 + threadIdx.x;
        float4 a[ENC_FIX];
#pragma unroll
        for (int k = 0; k < ENC_FIX; k++) a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < C4) {
            for (int sg0 = s0 + y; sg0 <= s1; sg0 += ENC_FIX * ENC_FIX_Y) {
#pragma unroll
                for (int k = 0; k < ENC_FIX; k++) {
                    const int sg = sg0 + k * ENC_FIX_Y;
                    if (sg <= s1) {
                        const int slot = (sg == s0 && lo != sg * ENC_SEG) ? 1 : 0;
                        const float4 p = part[((size_t)sg * 2 + slot) * C4 + c];
                        a[k].x += p.x; a[k].y += p.y; a[k].z += p.z; a[k].w += p.w;
                    }
                }
            }
        }
        float4 acc = a[0];
#pragma unroll
        for (int k = 1; k < ENC_FIX; k++) {
            acc.x += a[k].x; acc.y += a[k].y; acc.z += a[k].z; acc.w += a[k].w;
        }
        s_acc[y][threadIdx.x] = acc;
        __syncthreads();
        if (y == 0 && c < C4) {
#pragma unroll
            for (int j = 1; j < ENC_FIX_Y; j++) {
                const float4 t = s_acc[j][threadIdx.x];
                acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
            }
            float4 d = dwte[(size_t)v * C4 + c];
            d.x += acc.x; d.y += acc.y; d.z += acc.z; d.w += acc.w;
            dwte[(size_t)v * C4 + c] = d;
        }
        __syncthreads();
    }
}

__global__ void enc_dwpe_kernel(float4* __restrict__ dwpe, const float4* __restrict__ dx, int B,
                                int T, int maxT, int C4) {
    long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)maxT * C4) return;
    int t = (int)(idx / C4), c = (int)(idx % C4);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < T) {
        for (int b = 0; b < B; b++) {
            float4 g = dx[((size_t)b * T + t) * C4 + c];
            s.x += g.x; s.y += g.y; s.z += g.z; s.w += g.w;
        }
    }
    dwpe[idx] = s;
}

struct EncScratch {
    int *count, *cursor, *offset, *sums, *big, *n_big, *list, *sorted;
    float* part;
};

static size_t enc_layout(int BT, int V, int C, char* base, EncScratch* s) {
    size_t off = 0;
    auto take = [&](size_t n) {
        char* p = base ? base + off : nullptr;
        off += round_up(n * sizeof(int), 256);
        return reinterpret_cast<int*>(p);
    };
    EncScratch t;
    t.count = take(V);
    t.cursor = take(V);
    t.offset = take((size_t)V + 1);
    t.sums = take(2 * (size_t)ceil_div(V, ENC_SCAN_BLOCK));
    t.big = take(BT / ENC_BIG + 1);
    t.n_big = take(1);
    t.list = take(BT);
    t.sorted = take(BT);
    const size_t nseg = (size_t)ceil_div(BT, ENC_SEG);
    t.part = reinterpret_cast<float*>(take(nseg * 2 * (size_t)C));
    if (s) *s = t;
    return off;
}

}  // namespace gpt2k

using namespace gpt2k;

GPT2_API int gpt2_op_encoder_forward(float* x, const int* tok, const float* wte, const float* wpe,
                                     int B, int T, int C, int V, int* status, void* stream) {
    if (!x || !tok || !wte || !wpe || B < 1 || T < 1 || C < 4 || C % 4 || V < 1) return GPT2_EINVAL;
    if (!aligned16(x) || !aligned16(wte) || !aligned16(wpe)) return GPT2_EINVAL;
    int C4 = C / 4, BT = B * T;
    long long n = (long long)BT * C4;
    count_launch(), encoder_fwd_kernel<<<ceil_div(n, 256), 256, 0, as_stream(stream)>>>(
        reinterpret_cast<float4*>(x), tok, reinterpret_cast<const float4*>(wte),
        reinterpret_cast<const float4*>(wpe), BT, T, C4, V, status);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

GPT2_API size_t gpt2_op_encoder_backward_scratch_bytes(int BT, int V, int C) {
    if (BT < 1 || V < 1 || C < 1) return 0;
    return enc_layout(BT, V, C, nullptr, nullptr);
}

GPT2_API int gpt2_op_encoder_backward(float* dwte, float* dwpe, const float* dx, const int* tok,
                                      int B, int T, int maxT, int C, int V, void* scratch,
                                      size_t scratch_bytes, void* stream) {
    if (!dwte || !dwpe || !dx || !tok || B < 1 || T < 1 || T > maxT || C < 4 || C % 4 || V < 1)
        return GPT2_EINVAL;
    if (!aligned16(dwte) || !aligned16(dwpe) || !aligned16(dx)) return GPT2_EINVAL;
    int BT = B * T, C4 = C / 4;
    if (!scratch || scratch_bytes < gpt2_op_encoder_backward_scratch_bytes(BT, V, C)) return GPT2_ENOMEM;
    cudaStream_t st = as_stream(stream);
    EncScratch s;
    enc_layout(BT, V, C, reinterpret_cast<char*>(scratch), &s);
    GPT2_CUDA_TRY(cudaMemsetAsync(s.count, 0, sizeof(int) * V, st));
    GPT2_CUDA_TRY(cudaMemsetAsync(s.cursor, 0, sizeof(int) * V, st));
    // every launch is checked at once: a launch that fails must not leave the
    // kernels after it reading positions it did not write
    int nb = ceil_div(BT, 256);
    count_launch(), enc_histogram_kernel<<<nb, 256, 0, st>>>(s.count, tok, BT, V);
    GPT2_LAUNCH_CHECK();
    const int nsb = ceil_div(V, ENC_SCAN_BLOCK);
    count_launch(), enc_scan_sums_kernel<<<nsb, ENC_SCAN_BLOCK, 0, st>>>(s.sums, s.count, V);
    GPT2_LAUNCH_CHECK();
    count_launch(), enc_scan_kernel<<<nsb, ENC_SCAN_BLOCK, 0, st>>>(s.offset, s.big, s.n_big, s.count, s.sums, V);
    GPT2_LAUNCH_CHECK();
    count_launch(), enc_fill_kernel<<<nb, 256, 0, st>>>(s.list, s.cursor, s.offset, tok, BT, V);
    GPT2_LAUNCH_CHECK();
    const bool bitmap = BT > ENC_BIG && BT <= ENC_BITMAP_MAX_BT;
    count_launch(), enc_rank_kernel<<<nb, 256, 0, st>>>(s.sorted, s.list, s.offset, tok, BT, V, bitmap ? 1 : 0);
    GPT2_LAUNCH_CHECK();
    if (bitmap) {
        const int smem = ceil_div(BT, 32) * (int)sizeof(uint32_t);
        if (smem_limit(reinterpret_cast<const void*>(enc_sort_big_kernel), smem)) return GPT2_ECUDA;
        count_launch(), enc_sort_big_kernel<<<std::min(BT / ENC_BIG, 2 * num_sms()), 512, smem, st>>>(
            s.sorted, s.list, s.offset, s.big, s.n_big, BT);
        GPT2_LAUNCH_CHECK();
    }
    const int threads = C4 < 256 ? ((C4 + 31) / 32) * 32 : 256;
    count_launch(), enc_segment_kernel<<<ceil_div(BT, ENC_SEG), threads, 0, st>>>(
        reinterpret_cast<float4*>(dwte), reinterpret_cast<float4*>(s.part),
        reinterpret_cast<const float4*>(dx), s.sorted, s.offset, tok, V, C4);
    GPT2_LAUNCH_CHECK();
    if (BT > ENC_SEG) {
        count_launch(), enc_fixup_kernel<<<ceil_div(BT, ENC_SEG) - 1, dim3(threads, ENC_FIX_Y), 0, st>>>(
            reinterpret_cast<float4*>(dwte), reinterpret_cast<const float4*>(s.part), s.sorted, s.offset, tok, V,
            C4);
        GPT2_LAUNCH_CHECK();
    }
    long long n = (long long)maxT * C4;
    count_launch(), enc_dwpe_kernel<<<ceil_div(n, 256), 256, 0, st>>>(reinterpret_cast<float4*>(dwpe),
                                                     reinterpret_cast<const float4*>(dx), B, T,
                                                     maxT, C4);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}
