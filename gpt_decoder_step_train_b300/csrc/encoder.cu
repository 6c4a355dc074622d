// encoder.cu -- token + position embedding, forward and deterministic backward.
//
// Forward: x[b,t,:] = wte[tok[b,t],:] + wpe[t,:]  ("GPT-2 from scratch with
// torch", section 从词到编码: the two embeddings are added).
//
// Backward: dwte[v,:] += sum_{pos: tok[pos]=v} dx[pos,:] and dwpe[t,:] =
// sum_b dx[b,t,:].  The token-side scatter-add is made deterministic without
// float atomics: positions are bucketed by token id with an integer counting
// sort and each bucket is put in ascending position order.  The sorted list is
// then cut into fixed segments of 64 entries, one thread block each: a bucket
// that lies inside one segment is summed and added to dwte there; a bucket
// that crosses segment boundaries leaves one partial sum per segment, and a
// fix-up pass adds those in segment order.  A frequent token (a Zipf stream
// gives the top id ~14% of positions) is thus spread over many blocks.
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

// One block: exclusive scan of count[0..V) into offset[], and the list of
// distinct ids present (in increasing id order) into uniq[]; *n_uniq its length.
__global__ void enc_scan_kernel(int* __restrict__ offset, int* __restrict__ uniq,
                                int* __restrict__ n_uniq, const int* __restrict__ count, int V) {
    __shared__ int s_sum[1024], s_nz[1024];
    int tid = threadIdx.x, nt = blockDim.x;
    int per = (V + nt - 1) / nt;
    int lo = min(V, tid * per), hi = min(V, lo + per);
    int sum = 0, nz = 0;
    for (int v = lo; v < hi; v++) { sum += count[v]; nz += count[v] > 0; }
    s_sum[tid] = sum;
    s_nz[tid] = nz;
    __syncthreads();
    // Hillis-Steele inclusive scan over the per-thread totals
    for (int o = 1; o < nt; o <<= 1) {
        int a = tid >= o ? s_sum[tid - o] : 0;
        int b = tid >= o ? s_nz[tid - o] : 0;
        __syncthreads();
        s_sum[tid] += a;
        s_nz[tid] += b;
        __syncthreads();
    }
    int run = s_sum[tid] - sum, runu = s_nz[tid] - nz;
    for (int v = lo; v < hi; v++) {
        offset[v] = run;
        run += count[v];
        if (count[v] > 0) uniq[runu++] = v;
    }
    if (tid == nt - 1) { offset[V] = s_sum[tid]; *n_uniq = s_nz[tid]; }
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
                                int V) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BT) return;
    int id = tok[i];
    if (id < 0 || id >= V) return;
    int lo = offset[id], hi = offset[id + 1];
    int r = 0;
    for (int e = lo; e < hi; e++) r += list[e] < i;
    sorted[lo + r] = i;
}

constexpr int ENC_SEG = 64;
constexpr int ENC_PF = 8;              // gradient rows loaded together in the segment kernel

// One block per segment of the sorted list.  All threads walk the segment's
// entries in order (same token sequence from shared memory), each thread for
// its own float4 columns, and flush the running sum at every token change.
__global__ void enc_segment_kernel(float4* __restrict__ dwte, float4* __restrict__ part,
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

// Buckets that cross segments: add their per-segment partials in segment order.
__global__ void enc_fixup_kernel(float4* __restrict__ dwte, const float4* __restrict__ part,
                                 const int* __restrict__ offset, const int* __restrict__ uniq,
                                 const int* __restrict__ n_uniq, int C4) {
    const int u = blockIdx.x;
    if (u >= *n_uniq) return;
    const int v = uniq[u];
    const int lo = offset[v], hi = offset[v + 1];
    const int s0 = lo / ENC_SEG, s1 = (hi - 1) / ENC_SEG;
    if (s0 == s1) return;
    for (int c = threadIdx.x; c < C4; c += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sg = s0; sg <= s1; sg++) {
            const int slot = (sg == s0 && lo != sg * ENC_SEG) ? 1 : 0;
            const float4 p = part[((size_t)sg * 2 + slot) * C4 + c];
            acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
        }
        float4 d = dwte[(size_t)v * C4 + c];
        d.x += acc.x; d.y += acc.y; d.z += acc.z; d.w += acc.w;
        dwte[(size_t)v * C4 + c] = d;
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
    int *count, *cursor, *offset, *uniq, *n_uniq, *list, *sorted;
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
    t.uniq = take(BT);
    t.n_uniq = take(1);
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
    int nb = ceil_div(BT, 256);
    count_launch(), enc_histogram_kernel<<<nb, 256, 0, st>>>(s.count, tok, BT, V);
    count_launch(), enc_scan_kernel<<<1, 1024, 0, st>>>(s.offset, s.uniq, s.n_uniq, s.count, V);
    count_launch(), enc_fill_kernel<<<nb, 256, 0, st>>>(s.list, s.cursor, s.offset, tok, BT, V);
    count_launch(), enc_rank_kernel<<<nb, 256, 0, st>>>(s.sorted, s.list, s.offset, tok, BT, V);
    const int threads = C4 < 256 ? ((C4 + 31) / 32) * 32 : 256;
    count_launch(), enc_segment_kernel<<<ceil_div(BT, ENC_SEG), threads, 0, st>>>(
        reinterpret_cast<float4*>(dwte), reinterpret_cast<float4*>(s.part),
        reinterpret_cast<const float4*>(dx), s.sorted, s.offset, tok, V, C4);
    count_launch(), enc_fixup_kernel<<<min(BT, V), threads, 0, st>>>(
        reinterpret_cast<float4*>(dwte), reinterpret_cast<const float4*>(s.part), s.offset, s.uniq,
        s.n_uniq, C4);
    long long n = (long long)maxT * C4;
    count_launch(), enc_dwpe_kernel<<<ceil_div(n, 256), 256, 0, st>>>(reinterpret_cast<float4*>(dwpe),
                                                     reinterpret_cast<const float4*>(dx), B, T,
                                                     maxT, C4);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}
