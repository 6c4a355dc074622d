// model.cu -- the GPT-2 training step behind the C ABI of gpt2.h.
//
// One workspace block holds every buffer the step touches (gradients, AdamW
// moments, activations for maxB*maxT rows, logits, scratch), carved once at
// create time; nothing is allocated or freed while training, as the llm.c
// overview (bigegpt.com) describes for its single 1-D memory block.
//
// Forward ("GPT-2 from scratch with torch": nn_gpt2_model and the transformer
// block's forward): x = wte[tok] + wpe[t]; per block x = x + attn(ln_1(x)),
// x = x + mlp(ln_2(x)); ln_f; logits = ln_f(x) . wte^T; mean cross-entropy.
// Backward: each layer's hand-derived backward in reverse order, the residual
// stream's gradient accumulated in one buffer.  Update: AdamW.
#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <new>
#include <atomic>
#include <functional>
#include <mutex>
#include <vector>

#include "dropout.cuh"
#include "gemm.cuh"

namespace gpt2k {

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            n = v;
        else
            n = 148;
    }
    return n;
}

static std::atomic<long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int smem_limit(const void* kernel, int bytes) {
    struct Done {
        const void* k;
        int dev, bytes;
    };
    static std::mutex mu;
    static std::vector<Done> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { (void)cudaGetLastError(); return GPT2_ECUDA; }
    std::lock_guard<std::mutex> lock(mu);
    // the attribute only grows: a launch with fewer bytes than the recorded
    // limit needs no call, and lowering it would break a later larger launch
    // that an earlier call already cleared
    Done* rec = nullptr;
    for (Done& d : done)
        if (d.k == kernel && d.dev == dev) rec = &d;
    if (rec && rec->bytes >= bytes) return GPT2_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return GPT2_ECUDA;
    }
    if (rec) rec->bytes = bytes;
    else done.push_back(Done{kernel, dev, bytes});
    return GPT2_OK;
}

constexpr int NT = 16;
static const bool kDecay[NT] = {true, true, false, false, true, false, true, false,
                                false, false, true, false, true, false, false, false};
enum { WTE, WPE, LN1W, LN1B, QKVW, QKVB, ATTPROJW, ATTPROJB, LN2W, LN2B, FCW, FCB, FCPROJW,
       FCPROJB, LNFW, LNFB };

static void tensor_sizes(const gpt2_config& c, size_t* s) {
    size_t C = c.C, L = c.L;
    s[WTE] = (size_t)c.V * C;  s[WPE] = (size_t)c.maxT * C;
    s[LN1W] = L * C;           s[LN1B] = L * C;
    s[QKVW] = L * 3 * C * C;   s[QKVB] = L * 3 * C;
    s[ATTPROJW] = L * C * C;   s[ATTPROJB] = L * C;
    s[LN2W] = L * C;           s[LN2B] = L * C;
    s[FCW] = L * 4 * C * C;    s[FCB] = L * 4 * C;
    s[FCPROJW] = L * C * 4 * C; s[FCPROJB] = L * C;
    s[LNFW] = C;               s[LNFB] = C;
}

static bool config_ok(const gpt2_config* c) {
    if (!c) return false;
    if (c->V < 1 || c->maxT < 1 || c->L < 1 || c->H < 1 || c->C < 4 || c->maxB < 1) return false;
    if (c->C % 4 || c->C % c->H) return false;
    int hs = c->C / c->H;
    if (hs % 4 || hs > 64 || c->C > 2048) return false;
    if (c->mode != GPT2_MODE_FP32 && c->mode != GPT2_MODE_TF32 && c->mode != GPT2_MODE_BF16) return false;
    if (c->mode == GPT2_MODE_BF16 && hs != 16 && hs != 32 && hs != 64) return false;
    if ((long long)c->maxB * c->maxT > (1LL << 30)) return false;
    return true;
}

static int padded_vocab(int V) { return (int)round_up((size_t)V, 128); }

struct DevFlags {
    float loss;
    int status;
};

}  // namespace gpt2k

using namespace gpt2k;

struct gpt2 {
    gpt2_config cfg;
    int Vp, R;                  // padded vocabulary, activation row capacity
    size_t nparams, off[NT], sz[NT];
    float* params;
    char* ws;
    size_t ws_bytes;
    bool owns_ws;
    cudaStream_t st;
    bool bf16;                  // GPT2_MODE_BF16: operands below are bf16 (es = 2)
    size_t es;                  // bytes per element of the operand buffers
    float *grads, *m, *v;
    void* w16;                  // bf16 copy of the parameters (BF16 mode)
    int *tok, *tgt;
    DevFlags* flags;
    // fp32 activations; per-layer arrays have a fixed stride of R rows
    float *x0, *ln1_mean, *ln1_rstd, *lse, *res2, *ln2_mean, *ln2_rstd, *res3;
    float *lnf_mean, *lnf_rstd, *logits, *losses;
    // operand activations (es bytes per element): GEMM / attention inputs
    char *ln1, *qkv, *atty, *ln2, *fch, *fchg, *lnf;
    // backward: fp32 residual-stream gradient and LN-output gradient; operands
    float *dres, *dln;
    char *dres16, *dz16, *dbig, *datty, *dqkv;
    void* scratch;
    size_t scratch_bytes;
    float* colsum;              // per-layer per-32-row column sums for the fused bias gradients
    size_t colsum_fc_bytes, colsum_qkv_bytes;
    char* lnpart;               // per-call partial sums of the LayerNorm backwards
    size_t lnpart_bytes;
    // decoding: key/value cache [L][maxB][maxT][2C] and the rows of one step,
    // allocated by the first gpt2_decode
    char* dec;
    float *kv, *sx, *sx2, *sln, *sqkv, *satt, *sh, *smean, *srstd, *slog;
    int *stok, *dpos;           // the step's token ids; the position being decoded
    int dec_B, dec_next;
    // CUDA graphs of the forward, backward and decoding step, one per (kind, B,
    // T), replayed on a private stream ordered after and before the caller's
    // stream by events
    struct Graph {
        int kind, B, T, seen;
        cudaGraphExec_t exec;
        long long launches;
    };
    std::vector<Graph> graphs;
    cudaStream_t gst;
    cudaEvent_t g_in, g_out;
    bool graphs_off;
    int B, T;
    bool fwd_targets, have_grads;
    int err;
    // dropout (gpt2_set_dropout): probability, seed, training forwards drawn
    // under this seed so far, whether the last forward used it, and the device
    // buffer {key0, key1, step, 0} followed by the keep bits of every site
    float pdrop;
    unsigned long long dseed;
    uint32_t dstep;
    bool drop_fwd;
    uint32_t* dbuf;
    size_t dbuf_words;
    // tracing: event pairs recorded around each operation, with its class and launches
    bool trace_on;
    std::vector<cudaEvent_t> trace_events;
    size_t trace_used;
    std::vector<int> trace_cls;
    std::vector<long long> trace_launches;
};

namespace gpt2k {

// Lay out the workspace; with base == nullptr only computes the size.
static size_t plan(gpt2* m, char* base) {
    const gpt2_config& c = m->cfg;
    size_t off = 0;
    auto take = [&](size_t bytes) -> char* {
        char* p = base ? base + off : nullptr;
        off += round_up(bytes, 256);
        return p;
    };
    auto F = [&](size_t n) { return reinterpret_cast<float*>(take(n * sizeof(float))); };
    auto O = [&](size_t n) { return take(n * m->es); };
    const size_t R = m->R, C = c.C, L = c.L, H = c.H, N = m->nparams;
    m->grads = F(N);
    m->m = F(N);
    m->v = F(N);
    m->w16 = m->bf16 ? take(N * 2) : nullptr;
    m->tok = reinterpret_cast<int*>(take(R * sizeof(int)));
    m->tgt = reinterpret_cast<int*>(take(R * sizeof(int)));
    m->flags = reinterpret_cast<DevFlags*>(take(sizeof(DevFlags)));
    m->x0 = F(R * C);
    m->ln1 = O(L * R * C);
    m->ln1_mean = F(L * R);
    m->ln1_rstd = F(L * R);
    m->qkv = O(L * R * 3 * C);
    m->atty = O(L * R * C);
    m->lse = F(L * R * H);
    m->res2 = F(L * R * C);
    m->ln2 = O(L * R * C);
    m->ln2_mean = F(L * R);
    m->ln2_rstd = F(L * R);
    m->fch = O(L * R * 4 * C);
    m->fchg = O(L * R * 4 * C);
    m->res3 = F(L * R * C);
    m->lnf = O(R * C);
    m->lnf_mean = F(R);
    m->lnf_rstd = F(R);
    m->logits = F(R * (size_t)m->Vp);
    m->losses = F(R);
    m->dres = F(R * C);
    m->dln = F(R * C);
    m->dres16 = m->bf16 ? O(R * C) : nullptr;
    m->dz16 = m->bf16 ? O(R * (size_t)m->Vp) : nullptr;
    m->dbig = O(R * 4 * C);
    m->datty = O(R * C);
    m->dqkv = O(R * 3 * C);
    // scratch: the largest need of any backward op at full capacity
    const int Ri = (int)R, Ci = (int)C, mode = c.mode;
    size_t s = 0;
    s = std::max(s, gpt2_op_layernorm_backward_scratch_bytes(Ri, Ci));
    s = std::max(s, gpt2_op_linear_backward_weight_scratch_bytes(Ri, Ci, 3 * Ci, mode));
    s = std::max(s, gpt2_op_linear_backward_weight_scratch_bytes(Ri, Ci, Ci, mode));
    s = std::max(s, gpt2_op_linear_backward_weight_scratch_bytes(Ri, Ci, 4 * Ci, mode));
    s = std::max(s, gpt2_op_linear_backward_weight_scratch_bytes(Ri, 4 * Ci, Ci, mode));
    s = std::max(s, gpt2_op_linear_backward_weight_scratch_bytes(Ri, Ci, c.V, mode));
    s = std::max(s, linear_backward_input_scratch_bytes(Ri, Ci, c.V, mode));
    s = std::max(s, linear_backward_input_scratch_bytes(Ri, Ci, 3 * Ci, mode));
    s = std::max(s, linear_backward_input_scratch_bytes(Ri, Ci, 4 * Ci, mode));
    s = std::max(s, gpt2_op_attention_backward_scratch_bytes(c.maxB, c.maxT, c.H));
    s = std::max(s, gpt2_op_encoder_backward_scratch_bytes(Ri, c.V, Ci));
    s = std::max(s, gpt2_op_bias_grad_scratch_bytes(Ri, 4 * Ci));
    m->scratch_bytes = s;
    m->scratch = take(s);
    // per-group partial sums, kept until one reduction at the end of the
    // backward: the MLP c_fc bias (c_proj dX epilogue) and the qkv bias
    // (attention backward) of every layer, and every LayerNorm backward's
    // gamma / beta / residual-gradient column sums
    const int att_groups = c.maxB * ceil_div(c.maxT, 32);
    m->colsum_fc_bytes = round_up(linear_colsum_bytes(Ri, 4 * Ci), 256);
    m->colsum_qkv_bytes = round_up((size_t)att_groups * 3 * C * sizeof(float), 256);
    m->colsum = reinterpret_cast<float*>(take(L * (m->colsum_fc_bytes + m->colsum_qkv_bytes)));
    m->lnpart_bytes = round_up(gpt2_op_layernorm_backward_scratch_bytes(Ri, Ci), 256);
    m->lnpart = take((2 * L + 1) * m->lnpart_bytes);
    return off;
}

static float* P(gpt2* m, int t) { return m->params + m->off[t]; }
static float* G(gpt2* m, int t) { return m->grads + m->off[t]; }
// GEMM weight operand: the bf16 copy in BF16 mode, else the fp32 parameters
static const void* W(gpt2* m, int t) {
    return m->bf16 ? static_cast<const void*>(static_cast<const char*>(m->w16) + 2 * m->off[t])
                   : static_cast<const void*>(m->params + m->off[t]);
}
// operand row r (per-layer stride R rows) of an es-byte buffer
static char* Orow(gpt2* m, char* base, size_t layer, size_t width) {
    return base + layer * (size_t)m->R * width * m->es;
}

// Run one operation; when tracing, bracket it with events on the model's stream.
static int trace_op(gpt2* m, int cls, const std::function<int()>& f) {
    if (!m->trace_on) return f();
    while (m->trace_used + 2 > m->trace_events.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) { (void)cudaGetLastError(); return GPT2_ECUDA; }
        m->trace_events.push_back(e);
    }
    cudaEvent_t e0 = m->trace_events[m->trace_used], e1 = m->trace_events[m->trace_used + 1];
    long long n0 = g_launches.load(std::memory_order_relaxed);
    if (cudaEventRecord(e0, m->st) != cudaSuccess) { (void)cudaGetLastError(); return GPT2_ECUDA; }
    int rc = f();
    if (cudaEventRecord(e1, m->st) != cudaSuccess) { (void)cudaGetLastError(); return GPT2_ECUDA; }
    m->trace_used += 2;
    m->trace_cls.push_back(cls);
    m->trace_launches.push_back(g_launches.load(std::memory_order_relaxed) - n0);
    return rc;
}

#define OP(cls, call)                                                      \
    do {                                                                   \
        int rc_ = trace_op(m, GPT2_TRACE_##cls, [&]() -> int { return (call); }); \
        if (rc_) return rc_;                                               \
    } while (0)

// Keep bits of dropout site `site` for a forward of B x T: the embedding output
// (site 0), then per layer l the attention weights (1 + 3l, rows (b, h, i) of
// ceil(T/32) words), the attention c_proj output (2 + 3l) and the MLP c_proj
// output (3 + 3l), rows (b, t) of ceil(C/32) words.  The first four words of
// the buffer hold the draw state.
static size_t drop_words(const gpt2_config& c, int B, int T) {
    const size_t N = (size_t)B * T, wc = (size_t)(c.C + 31) / 32, wt = (size_t)(T + 31) / 32;
    return 4 + N * wc + (size_t)c.L * ((size_t)B * c.H * T * wt + 2 * N * wc);
}
static uint32_t* drop_bits(gpt2* m, int site) {
    const gpt2_config& c = m->cfg;
    const size_t N = (size_t)m->B * m->T, wc = (size_t)(c.C + 31) / 32, wt = (size_t)(m->T + 31) / 32;
    const size_t att = (size_t)m->B * c.H * m->T * wt, layer = att + 2 * N * wc;
    uint32_t* base = m->dbuf + 4;
    if (site == 0) return base;
    const int l = (site - 1) / 3, k = (site - 1) % 3;
    return base + N * wc + (size_t)l * layer + (k == 0 ? 0 : att + (size_t)(k - 1) * N * wc);
}

// with_targets: the cross-entropy runs; grad: it also leaves d(loss)/d(logits)
static int forward_impl(gpt2* m, int B, int T, bool with_targets, bool grad) {
    const gpt2_config& c = m->cfg;
    const int C = c.C, L = c.L, H = c.H, N = B * T, mode = c.mode;
    const bool b16 = m->bf16;
    const size_t R = m->R;
    cudaStream_t st = m->st;
    int* status = &m->flags->status;
    if (b16) OP(OTHER, to_bf16(m->w16, m->params, m->nparams, st));
    // dropout: draw every site's keep bits (key and step from the device state)
    const bool drop = m->drop_fwd;
    const float pd = m->pdrop;
    if (drop) {
        OP(DROPOUT, dropout_mask(drop_bits(m, 0), N, C, 0, m->dbuf, 0, 0, 0, pd, st));
        for (int l = 0; l < L; l++) {
            OP(DROPOUT, dropout_mask(drop_bits(m, 1 + 3 * l), (long long)B * H * T, T, T, m->dbuf, 0, 1 + 3 * l, 0,
                                     pd, st));
            OP(DROPOUT, dropout_mask(drop_bits(m, 2 + 3 * l), N, C, 0, m->dbuf, 0, 2 + 3 * l, 0, pd, st));
            OP(DROPOUT, dropout_mask(drop_bits(m, 3 + 3 * l), N, C, 0, m->dbuf, 0, 3 + 3 * l, 0, pd, st));
        }
    }
    OP(ENCODER_FWD, gpt2_op_encoder_forward(m->x0, m->tok, P(m, WTE), P(m, WPE), B, T, C, c.V, status, st));
    if (drop) OP(DROPOUT, dropout_residual(m->x0, nullptr, drop_bits(m, 0), N, C, pd, st));
    for (int l = 0; l < L; l++) {
        const float* x = l == 0 ? m->x0 : m->res3 + (size_t)(l - 1) * R * C;
        char* ln1 = Orow(m, m->ln1, l, C);
        char* qkv = Orow(m, m->qkv, l, 3 * C);
        char* atty = Orow(m, m->atty, l, C);
        float* res2 = m->res2 + l * R * C;
        char* ln2 = Orow(m, m->ln2, l, C);
        char* fch = Orow(m, m->fch, l, 4 * C);
        char* fchg = Orow(m, m->fchg, l, 4 * C);
        float* res3 = m->res3 + l * R * C;
        const size_t cc = (size_t)C * C;
        const size_t wes = b16 ? 2 : 4;
        auto Wl = [&](int t, size_t per_layer) {
            return static_cast<const void*>(static_cast<const char*>(W(m, t)) + l * per_layer * wes);
        };
        OP(LAYERNORM_FWD, layernorm_forward(ln1, b16, m->ln1_mean + l * R, m->ln1_rstd + l * R, x,
                                            P(m, LN1W) + l * C, P(m, LN1B) + l * C, N, C, st));
        OP(MATMUL_FWD, linear_forward(qkv, b16, nullptr, ln1, Wl(QKVW, 3 * cc), b16, P(m, QKVB) + l * 3 * C,
                                      nullptr, N, C, 3 * C, 3 * C, 0, mode, status, st));
        OP(ATTENTION_FWD, attention_forward(atty, m->lse + l * R * H, qkv, B, T, C, H, mode, status, st,
                                            drop ? drop_bits(m, 1 + 3 * l) : nullptr, drop ? pd : 0.f));
        // with dropout the residual is added after the c_proj output is dropped
        OP(MATMUL_FWD, linear_forward(res2, false, nullptr, atty, Wl(ATTPROJW, cc), b16, P(m, ATTPROJB) + l * C,
                                      drop ? nullptr : x, N, C, C, C, 0, mode, status, st));
        if (drop) OP(DROPOUT, dropout_residual(res2, x, drop_bits(m, 2 + 3 * l), N, C, pd, st));
        OP(LAYERNORM_FWD, layernorm_forward(ln2, b16, m->ln2_mean + l * R, m->ln2_rstd + l * R, res2,
                                            P(m, LN2W) + l * C, P(m, LN2B) + l * C, N, C, st));
        OP(MATMUL_FWD, linear_forward(fchg, b16, fch, ln2, Wl(FCW, 4 * cc), b16, P(m, FCB) + l * 4 * C, nullptr,
                                      N, C, 4 * C, 4 * C, GPT2_LINEAR_GELU, mode, status, st));
        OP(MATMUL_FWD, linear_forward(res3, false, nullptr, fchg, Wl(FCPROJW, 4 * cc), b16,
                                      P(m, FCPROJB) + l * C, drop ? nullptr : res2, N, 4 * C, C, C, 0, mode, status,
                                      st));
        if (drop) OP(DROPOUT, dropout_residual(res3, res2, drop_bits(m, 3 + 3 * l), N, C, pd, st));
    }
    const float* xL = m->res3 + (size_t)(L - 1) * R * C;
    OP(LAYERNORM_FWD, layernorm_forward(m->lnf, b16, m->lnf_mean, m->lnf_rstd, xL, P(m, LNFW), P(m, LNFB),
                                        N, C, st));
    if (b16 && with_targets && m->Vp <= GPT2_CE_BF16_MAX_LD) {
        // training forward in BF16 mode: the logits go to the bf16 buffer and
        // the cross-entropy overwrites them with their gradient (the padded
        // columns are zeroed there), the operand of the lm_head backward
        OP(MATMUL_FWD, linear_forward(m->dz16, true, nullptr, m->lnf, W(m, WTE), b16, nullptr, nullptr, N, C,
                                      c.V, m->Vp, 0, mode, status, st));
        OP(CROSSENTROPY, gpt2_op_crossentropy_bf16(m->losses, m->dz16, m->tgt, N, c.V, m->Vp,
                                                   grad ? 1.0f / (float)N : 0.f, status, st));
    } else {
        OP(MATMUL_FWD, linear_forward(m->logits, false, nullptr, m->lnf, W(m, WTE), b16, nullptr, nullptr, N,
                                      C, c.V, m->Vp, GPT2_LINEAR_ZERO_PAD, mode, status, st));
        if (with_targets)
            OP(CROSSENTROPY, gpt2_op_crossentropy(m->losses, m->logits, m->dz16, m->tgt, N, c.V, m->Vp,
                                                  grad ? 1.0f / (float)N : 0.f, status, st));
    }
    if (with_targets) OP(CROSSENTROPY, gpt2_op_sum(&m->flags->loss, m->losses, N, 1.0f / (float)N, st));
    return GPT2_OK;
}

static int backward_impl(gpt2* m) {
    const gpt2_config& c = m->cfg;
    const int B = m->B, T = m->T, C = c.C, L = c.L, H = c.H, N = B * T, mode = c.mode;
    const bool b16 = m->bf16;
    const size_t R = m->R, cc = (size_t)C * C;
    cudaStream_t st = m->st;
    void* sc = m->scratch;
    const size_t sb = m->scratch_bytes;
    int* status = &m->flags->status;
    // operand views of the residual-stream gradient and of dlogits
    const void* dres_op = b16 ? static_cast<const void*>(m->dres16) : static_cast<const void*>(m->dres);
    const void* dz_op = b16 ? static_cast<const void*>(m->dz16) : static_cast<const void*>(m->logits);
    const size_t wes = b16 ? 2 : 4;
    // dropout: the gradient of a dropped c_proj output is keep o dres / (1 - p)
    // and its bias gradient the column sum of that.  It goes over the operand
    // copy of dres (BF16 mode), else into an operand buffer that is free at that
    // point (datty before the MLP c_proj backward, dbig before the attention
    // c_proj backward).  The LayerNorm backward that produces dres writes it
    // with the column sum (rows up to 768 wide), else a separate pass does.
    const bool drop = m->drop_fwd;
    const bool fuse = drop && layernorm_backward_fuses_dropout(C);
    const float pd = m->pdrop;
    void* const dbr_mlp = b16 ? static_cast<void*>(m->dres16) : static_cast<void*>(m->datty);
    void* const dbr_att = b16 ? static_cast<void*>(m->dres16) : static_cast<void*>(m->dbig);
    const void* const op_mlp = drop ? static_cast<const void*>(dbr_mlp) : dres_op;
    const void* const op_att = drop ? static_cast<const void*>(dbr_att) : dres_op;
    // column reductions left for one launch at the end
    std::vector<ColReduce> red;
    red.reserve(4 * L + 2);
    ColReduce cr{};
    auto keep = [&]() { if (cr.part) red.push_back(cr); cr = ColReduce{}; };
    auto lnpart = [&](int k) { return static_cast<void*>(m->lnpart + (size_t)k * m->lnpart_bytes); };
    auto cs_fc = [&](int l) { return reinterpret_cast<float*>(reinterpret_cast<char*>(m->colsum) + l * m->colsum_fc_bytes); };
    auto cs_qkv = [&](int l) {
        return reinterpret_cast<float*>(reinterpret_cast<char*>(m->colsum) + L * m->colsum_fc_bytes +
                                        l * m->colsum_qkv_bytes);
    };
    // tied lm_head: d(lnf) = dz . wte ; d(wte) = dz^T . lnf (first write of dwte)
    OP(MATMUL_BWD_INPUT, linear_backward_input(m->dln, false, dz_op, W(m, WTE), b16, nullptr, N, C, c.V,
                                               m->Vp, mode, status, st, nullptr, nullptr, 0, nullptr, sc, sb));
    OP(MATMUL_BWD_WEIGHT, linear_backward_weight(G(m, WTE), dz_op, m->lnf, b16, N, C, c.V, m->Vp, sc, sb,
                                                 mode, status, st));
    // ln_f: the residual gradient starts here (written, not accumulated); its
    // column sum is the last block's MLP c_proj bias gradient
    OP(LAYERNORM_BWD, layernorm_backward(m->dres, fuse ? dbr_mlp : m->dres16, !fuse || b16, G(m, LNFW), G(m, LNFB),
                                         drop && !fuse ? nullptr : G(m, FCPROJB) + (size_t)(L - 1) * C, m->dln,
                                         m->res3 + (size_t)(L - 1) * R * C, P(m, LNFW), m->lnf_mean, m->lnf_rstd, N,
                                         C, 0, lnpart(0), m->lnpart_bytes, status, st,
                                         fuse ? drop_bits(m, 3 * L) : nullptr, pd, &cr));
    keep();
    for (int l = L - 1; l >= 0; l--) {
        const float* x = l == 0 ? m->x0 : m->res3 + (size_t)(l - 1) * R * C;
        const char* ln1 = Orow(m, m->ln1, l, C);
        const char* qkv = Orow(m, m->qkv, l, 3 * C);
        const char* atty = Orow(m, m->atty, l, C);
        const float* res2 = m->res2 + l * R * C;
        const char* ln2 = Orow(m, m->ln2, l, C);
        const char* fch = Orow(m, m->fch, l, 4 * C);
        const char* fchg = Orow(m, m->fchg, l, 4 * C);
        auto Wl = [&](int t, size_t per_layer) {
            return static_cast<const void*>(static_cast<const char*>(W(m, t)) + l * per_layer * wes);
        };
        // MLP c_proj: dh = (dres . Wfp) * gelu'(h); dWfp = dres^T . g (its bias
        // gradient came with the LayerNorm backward that produced dres)
        // (with the c_fc bias gradient: the column sums of dh)
        if (drop && !fuse) {
            OP(DROPOUT, dropout_backward(dbr_mlp, b16, m->dres, drop_bits(m, 3 + 3 * l), N, C, pd, st));
            OP(BIAS_GRAD, bias_grad_any(G(m, FCPROJB) + l * C, dbr_mlp, b16, N, C, C, sc, sb, st));
        }
        OP(MATMUL_BWD_INPUT, linear_backward_input(m->dbig, b16, op_mlp, Wl(FCPROJW, 4 * cc), b16, fch, N,
                                                   4 * C, C, C, mode, status, st, G(m, FCB) + l * 4 * C,
                                                   cs_fc(l), m->colsum_fc_bytes, &cr));
        keep();
        OP(MATMUL_BWD_WEIGHT, linear_backward_weight(G(m, FCPROJW) + l * 4 * cc, op_mlp, fchg, b16, N,
                                                     4 * C, C, C, sc, sb, mode, status, st));
        // MLP c_fc: dln2 = dh . Wfc; dWfc = dh^T . ln2; dbfc
        OP(MATMUL_BWD_INPUT, linear_backward_input(m->dln, false, m->dbig, Wl(FCW, 4 * cc), b16, nullptr, N,
                                                   C, 4 * C, 4 * C, mode, status, st, nullptr, nullptr, 0, nullptr,
                                                   sc, sb));
        OP(MATMUL_BWD_WEIGHT, linear_backward_weight(G(m, FCW) + l * 4 * cc, m->dbig, ln2, b16, N, C, 4 * C,
                                                     4 * C, sc, sb, mode, status, st));
        // ln_2: dres += LN'(dln2); the column sum of the result is the attention
        // c_proj bias gradient
        OP(LAYERNORM_BWD, layernorm_backward(m->dres, fuse ? dbr_att : m->dres16, !fuse || b16, G(m, LN2W) + l * C,
                                             G(m, LN2B) + l * C, drop && !fuse ? nullptr : G(m, ATTPROJB) + l * C,
                                             m->dln, res2, P(m, LN2W) + l * C, m->ln2_mean + l * R,
                                             m->ln2_rstd + l * R, N, C, 1, lnpart(1 + 2 * l), m->lnpart_bytes, status,
                                             st, fuse ? drop_bits(m, 2 + 3 * l) : nullptr, pd, &cr));
        keep();
        // attention c_proj (bias gradient: with ln_2's backward above)
        if (drop && !fuse) {
            OP(DROPOUT, dropout_backward(dbr_att, b16, m->dres, drop_bits(m, 2 + 3 * l), N, C, pd, st));
            OP(BIAS_GRAD, bias_grad_any(G(m, ATTPROJB) + l * C, dbr_att, b16, N, C, C, sc, sb, st));
        }
        OP(MATMUL_BWD_INPUT, linear_backward_input(m->datty, b16, op_att, Wl(ATTPROJW, cc), b16, nullptr, N,
                                                   C, C, C, mode, status, st));
        OP(MATMUL_BWD_WEIGHT, linear_backward_weight(G(m, ATTPROJW) + l * cc, op_att, atty, b16, N, C, C, C,
                                                     sc, sb, mode, status, st));
        // attention; the tcgen05 path also leaves the column sums of dqkv per
        // 32 rows, which give the qkv bias gradient at once
        bool qkv_colsum = false;
        OP(ATTENTION_BWD, attention_backward_dropout(m->dqkv, m->datty, qkv, atty, m->lse + l * R * H, B, T, C, H,
                                                     sc, sb, mode, status, st, cs_qkv(l), &qkv_colsum,
                                                     drop ? drop_bits(m, 1 + 3 * l) : nullptr, drop ? pd : 0.f));
        if (qkv_colsum)
            red.push_back(ColReduce{cs_qkv(l), B * ceil_div(T, 32), 3 * C, 3 * C, 3 * C,
                                    {G(m, QKVB) + l * 3 * C, nullptr, nullptr}});
        // c_attn
        OP(MATMUL_BWD_INPUT, linear_backward_input(m->dln, false, m->dqkv, Wl(QKVW, 3 * cc), b16, nullptr, N,
                                                   C, 3 * C, 3 * C, mode, status, st, nullptr, nullptr, 0, nullptr,
                                                   sc, sb));
        OP(MATMUL_BWD_WEIGHT, linear_backward_weight(G(m, QKVW) + l * 3 * cc, m->dqkv, ln1, b16, N, C, 3 * C,
                                                     3 * C, sc, sb, mode, status, st));
        if (!qkv_colsum)
            OP(BIAS_GRAD, bias_grad_any(G(m, QKVB) + l * 3 * C, m->dqkv, b16, N, 3 * C, 3 * C, sc, sb, st));
        // ln_1: dres += LN'(dln1); the column sum of the result is the previous
        // block's MLP c_proj bias gradient
        // (with dropout: the previous block's dropped MLP c_proj branch; the
        // first block's ln_1 feeds the dropped embedding output instead)
        const bool fuse1 = fuse && l > 0;
        OP(LAYERNORM_BWD, layernorm_backward(m->dres, fuse1 ? dbr_mlp : m->dres16, !fuse1 || b16, G(m, LN1W) + l * C,
                                             G(m, LN1B) + l * C,
                                             l > 0 && (!drop || fuse) ? G(m, FCPROJB) + (size_t)(l - 1) * C : nullptr,
                                             m->dln, x, P(m, LN1W) + l * C, m->ln1_mean + l * R, m->ln1_rstd + l * R,
                                             N, C, 1, lnpart(2 + 2 * l), m->lnpart_bytes, status, st,
                                             fuse1 ? drop_bits(m, 3 * l) : nullptr, pd, &cr));
        keep();
    }
    if (drop) OP(DROPOUT, dropout_backward(m->dres, false, m->dres, drop_bits(m, 0), N, C, pd, st));
    OP(ENCODER_BWD, gpt2_op_encoder_backward(G(m, WTE), G(m, WPE), m->dres, m->tok, B, T, c.maxT, C, c.V,
                                             sc, sb, st));
    // every deferred column sum (bias and LayerNorm gradients), in one launch
    OP(BIAS_GRAD, colsum_batch(red.data(), (int)red.size(), st));
    return GPT2_OK;
}

static void record(gpt2* m, int rc) {
    if (rc && !m->err) m->err = rc;
}

// Run fn (the operations of a forward or backward, issued on m->st) through a
// CUDA graph.  The first call of a (kind, B, T) runs fn directly (one-time
// set-up happens outside any capture); the second captures it on the private
// stream and later calls replay the graph.  Tracing, or a failed capture,
// runs fn directly from then on.
static int run_graphed(gpt2* m, int kind, int B, int T, const std::function<int()>& fn) {
    if (m->trace_on || m->graphs_off || !m->gst) return fn();
    // inside the caller's own stream capture the operations go into that graph
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(m->st, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return fn();
    }
    if (cs != cudaStreamCaptureStatusNone) return fn();
    gpt2::Graph* g = nullptr;
    for (auto& e : m->graphs)
        if (e.kind == kind && e.B == B && e.T == T) g = &e;
    if (!g) {
        m->graphs.push_back(gpt2::Graph{kind, B, T, 0, nullptr, 0});
        g = &m->graphs.back();
    }
    if (!g->exec && g->seen++ == 0) return fn();
    if (!g->exec) {
        cudaStream_t user = m->st;
        if (cudaStreamBeginCapture(m->gst, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
            (void)cudaGetLastError();
            m->graphs_off = true;
            return fn();
        }
        m->st = m->gst;
        const long long n0 = g_launches.load(std::memory_order_relaxed);
        int rc = fn();
        const long long n = g_launches.load(std::memory_order_relaxed) - n0;
        m->st = user;
        cudaGraph_t graph = nullptr;
        cudaError_t ce = cudaStreamEndCapture(m->gst, &graph);
        g_launches.fetch_sub(n, std::memory_order_relaxed);     // counted when replayed
        if (rc || ce != cudaSuccess || !graph ||
            cudaGraphInstantiate(&g->exec, graph, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            if (graph) cudaGraphDestroy(graph);
            g->exec = nullptr;
            m->graphs_off = true;
            return fn();
        }
        cudaGraphDestroy(graph);
        g->launches = n;
    }
    if (cudaEventRecord(m->g_in, m->st) != cudaSuccess || cudaStreamWaitEvent(m->gst, m->g_in, 0) != cudaSuccess ||
        cudaGraphLaunch(g->exec, m->gst) != cudaSuccess || cudaEventRecord(m->g_out, m->gst) != cudaSuccess ||
        cudaStreamWaitEvent(m->st, m->g_out, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        return GPT2_ECUDA;
    }
    g_launches.fetch_add(g->launches, std::memory_order_relaxed);
    return GPT2_OK;
}

}  // namespace gpt2k

// ============================================================================
// C ABI
// ============================================================================

GPT2_API size_t gpt2_num_params(const gpt2_config* cfg) {
    if (!config_ok(cfg)) return 0;
    size_t s[NT], n = 0;
    tensor_sizes(*cfg, s);
    for (int i = 0; i < NT; i++) n += s[i];
    return n;
}

GPT2_API size_t gpt2_workspace_bytes(const gpt2_config* cfg) {
    if (!config_ok(cfg)) return 0;
    gpt2 tmp{};
    tmp.cfg = *cfg;
    tmp.Vp = padded_vocab(cfg->V);
    tmp.R = cfg->maxB * cfg->maxT;
    tmp.nparams = gpt2_num_params(cfg);
    tmp.bf16 = cfg->mode == GPT2_MODE_BF16;
    tmp.es = tmp.bf16 ? 2 : 4;
    return plan(&tmp, nullptr);
}

GPT2_API int gpt2_create(const gpt2_config* cfg, float* params, gpt2** out) {
    if (out) *out = nullptr;
    if (!out || !config_ok(cfg) || !params || !aligned16(params)) return GPT2_EINVAL;
    gpt2* m = new (std::nothrow) gpt2{};
    if (!m) return GPT2_ENOMEM;
    m->cfg = *cfg;
    m->Vp = padded_vocab(cfg->V);
    m->R = cfg->maxB * cfg->maxT;
    m->nparams = gpt2_num_params(cfg);
    m->bf16 = cfg->mode == GPT2_MODE_BF16;
    m->es = m->bf16 ? 2 : 4;
    tensor_sizes(*cfg, m->sz);
    size_t o = 0;
    for (int i = 0; i < NT; i++) { m->off[i] = o; o += m->sz[i]; }
    m->params = params;
    m->st = as_stream(cfg->stream);
    size_t need = plan(m, nullptr);
    if (cfg->workspace) {
        if (cfg->workspace_bytes < need || !aligned16(cfg->workspace)) { delete m; return GPT2_ENOMEM; }
        m->ws = reinterpret_cast<char*>(cfg->workspace);
        m->owns_ws = false;
    } else {
        if (cudaMalloc(&m->ws, need) != cudaSuccess) { (void)cudaGetLastError(); delete m; return GPT2_ENOMEM; }
        m->owns_ws = true;
    }
    m->ws_bytes = need;
    plan(m, m->ws);
    bool ok = cudaMemsetAsync(m->m, 0, m->nparams * sizeof(float), m->st) == cudaSuccess &&
              cudaMemsetAsync(m->v, 0, m->nparams * sizeof(float), m->st) == cudaSuccess &&
              cudaMemsetAsync(m->flags, 0, sizeof(DevFlags), m->st) == cudaSuccess;
    if (!ok) {
        (void)cudaGetLastError();
        if (m->owns_ws) cudaFree(m->ws);
        delete m;
        return GPT2_ECUDA;
    }
    // the private stream that replays the step's graphs (none: no graphs)
    if (cudaStreamCreateWithFlags(&m->gst, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&m->g_in, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&m->g_out, cudaEventDisableTiming) != cudaSuccess) {
        (void)cudaGetLastError();
        m->graphs_off = true;
    }
    (void)gemm_tc_pair_slots();     // one-time occupancy query, outside any capture
    *out = m;
    return GPT2_OK;
}

namespace gpt2k {
static float forward_common(gpt2* m, const int* tokens, const int* targets, int B, int T, bool grad) {
    if (!m) return NAN;
    if (!tokens || B < 1 || T < 1 || B > m->cfg.maxB || T > m->cfg.maxT) {
        record(m, GPT2_EINVAL);
        return NAN;
    }
    size_t nb = (size_t)B * T * sizeof(int);
    m->fwd_targets = false;
    m->have_grads = false;
    int crc = trace_op(m, GPT2_TRACE_OTHER, [&]() -> int {
        bool ok = cudaMemcpyAsync(m->tok, tokens, nb, cudaMemcpyDefault, m->st) == cudaSuccess &&
                  (!targets ||
                   cudaMemcpyAsync(m->tgt, targets, nb, cudaMemcpyDefault, m->st) == cudaSuccess) &&
                  cudaMemsetAsync(m->flags, 0, sizeof(DevFlags), m->st) == cudaSuccess;
        if (!ok) (void)cudaGetLastError();
        return ok ? GPT2_OK : GPT2_ECUDA;
    });
    if (crc) {
        record(m, crc);
        return NAN;
    }
    m->B = B;
    m->T = T;
    // dropout in the training forward (not in evaluation): this call's draw
    // state goes to the device before the step, so a replayed graph draws anew
    m->drop_fwd = grad && m->pdrop > 0.f && m->dbuf;
    if (m->drop_fwd) {
        const uint32_t h[4] = {(uint32_t)m->dseed, (uint32_t)(m->dseed >> 32), m->dstep, 0u};
        if (cudaMemcpyAsync(m->dbuf, h, sizeof(h), cudaMemcpyHostToDevice, m->st) != cudaSuccess) {
            (void)cudaGetLastError();
            record(m, GPT2_ECUDA);
            return NAN;
        }
        m->dstep++;
    }
    const int kind = targets ? (grad ? 0 : 2) : 1;
    int rc = run_graphed(m, kind, B, T, [&]() -> int { return forward_impl(m, B, T, targets != nullptr, grad); });
    if (rc) { record(m, rc); return NAN; }
    DevFlags h{};
    if (cudaMemcpyAsync(&h, m->flags, sizeof(h), cudaMemcpyDeviceToHost, m->st) != cudaSuccess ||
        cudaStreamSynchronize(m->st) != cudaSuccess) {
        (void)cudaGetLastError();
        record(m, GPT2_ECUDA);
        return NAN;
    }
    if (h.status & (GPT2_STATUS_BAD_TOKEN | GPT2_STATUS_BAD_TARGET)) {
        record(m, GPT2_ETOKEN);
        return NAN;
    }
    if (h.status & GPT2_STATUS_TIMEOUT) {
        record(m, GPT2_ETIMEOUT);
        return NAN;
    }
    if (!targets) return NAN;
    m->fwd_targets = grad;
    return h.loss;
}
}  // namespace gpt2k

GPT2_API float gpt2_forward(gpt2* m, const int* tokens, const int* targets, int B, int T) {
    return forward_common(m, tokens, targets, B, T, true);
}

GPT2_API float gpt2_eval(gpt2* m, const int* tokens, const int* targets, int B, int T) {
    if (m && !targets) {
        record(m, GPT2_EINVAL);
        return NAN;
    }
    return forward_common(m, tokens, targets, B, T, false);
}

GPT2_API int gpt2_backward(gpt2* m) {
    if (!m) return GPT2_EINVAL;
    if (!m->fwd_targets) { record(m, GPT2_ESTATE); return GPT2_ESTATE; }
    int rc = run_graphed(m, 3, m->B, m->T, [&]() -> int { return backward_impl(m); });
    if (rc) { record(m, rc); return rc; }
    m->fwd_targets = false;     // dlogits were consumed; a new forward is needed
    m->have_grads = true;
    return GPT2_OK;
}

GPT2_API int gpt2_adamw(gpt2* m, float lr, float b1, float b2, float eps, float wd, int t) {
    if (!m) return GPT2_EINVAL;
    if (t < 1) { record(m, GPT2_EINVAL); return GPT2_EINVAL; }
    if (!m->have_grads) { record(m, GPT2_ESTATE); return GPT2_ESTATE; }
    float bc1 = (float)(1.0 - pow((double)b1, (double)t));
    float bc2 = (float)(1.0 - pow((double)b2, (double)t));
    // consecutive tensors with the same decay setting share one launch
    int i = 0;
    while (i < NT) {
        int j = i;
        size_t n = 0;
        while (j < NT && kDecay[j] == kDecay[i]) n += m->sz[j++];
        int rc = trace_op(m, GPT2_TRACE_ADAMW, [&]() -> int {
            return gpt2_op_adamw(m->params + m->off[i], m->grads + m->off[i], m->m + m->off[i],
                                 m->v + m->off[i], n, lr, b1, b2, eps, kDecay[i] ? wd : 0.f, bc1,
                                 bc2, m->st);
        });
        if (rc) { record(m, rc); return rc; }
        i = j;
    }
    return GPT2_OK;
}

namespace gpt2k {
constexpr int DECODE_MAXB = 16;

// Carve the decoding state (cache and step rows) from one allocation.
static int decode_alloc(gpt2* m) {
    const gpt2_config& c = m->cfg;
    const size_t C = c.C, RB = DECODE_MAXB;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += round_up(bytes, 256); return o; };
    const size_t o_kv = take((size_t)c.L * c.maxB * c.maxT * 2 * C * sizeof(float));
    const size_t o_x = take(RB * C * 4), o_x2 = take(RB * C * 4), o_ln = take(RB * C * 4);
    const size_t o_qkv = take(RB * 3 * C * 4), o_att = take(RB * C * 4), o_h = take(RB * 4 * C * 4);
    const size_t o_mu = take(RB * 4), o_rs = take(RB * 4), o_tok = take(RB * 4), o_pos = take(4);
    const size_t o_log = take(RB * c.V * 4);
    if (cudaMalloc(&m->dec, off) != cudaSuccess) { (void)cudaGetLastError(); m->dec = nullptr; return GPT2_ENOMEM; }
    auto F = [&](size_t o) { return reinterpret_cast<float*>(m->dec + o); };
    m->kv = F(o_kv); m->sx = F(o_x); m->sx2 = F(o_x2); m->sln = F(o_ln); m->sqkv = F(o_qkv);
    m->satt = F(o_att); m->sh = F(o_h); m->smean = F(o_mu); m->srstd = F(o_rs);
    m->slog = F(o_log);
    m->stok = reinterpret_cast<int*>(m->dec + o_tok);
    m->dpos = reinterpret_cast<int*>(m->dec + o_pos);
    return GPT2_OK;
}

// One decoding step of B rows at the position *dpos (the same operations for
// every position, so a captured graph replays for each): the logits go to the
// step buffer slog [B, V].
static int decode_impl(gpt2* m, int B) {
    const gpt2_config& c = m->cfg;
    const int C = c.C, L = c.L, H = c.H;
    cudaStream_t st = m->st;
    int* status = &m->flags->status;
    int rc = decode_embed(m->sx, m->stok, P(m, WTE), P(m, WPE), B, C, c.V, m->dpos, status, st);
    // per layer: LayerNorm 1, qkv (+ the key/value cache store), attention,
    // projection + residual, LayerNorm 2, c_fc + GELU, c_proj + residual
    for (int l = 0; l < L && !rc; l++) {
        const size_t cc = (size_t)C * C;
        float* kv = m->kv + (size_t)l * c.maxB * c.maxT * 2 * C;
        rc = layernorm_forward(m->sln, false, m->smean, m->srstd, m->sx, P(m, LN1W) + l * C, P(m, LN1B) + l * C,
                               B, C, st);
        if (!rc) rc = decode_gemv(m->sqkv, 3 * C, m->sln, P(m, QKVW) + l * 3 * cc, P(m, QKVB) + l * 3 * C,
                                  nullptr, B, C, 3 * C, 0, kv, c.maxT, m->dpos, st);
        if (!rc) rc = decode_attention(m->satt, m->sqkv, kv, B, C, H, c.maxT, m->dpos, st);
        if (!rc) rc = decode_gemv(m->sx2, C, m->satt, P(m, ATTPROJW) + l * cc, P(m, ATTPROJB) + l * C, m->sx, B,
                                  C, C, 0, nullptr, 0, nullptr, st);
        if (!rc) rc = layernorm_forward(m->sln, false, m->smean, m->srstd, m->sx2, P(m, LN2W) + l * C,
                                        P(m, LN2B) + l * C, B, C, st);
        if (!rc) rc = decode_gemv(m->sh, 4 * C, m->sln, P(m, FCW) + l * 4 * cc, P(m, FCB) + l * 4 * C, nullptr,
                                  B, C, 4 * C, 1, nullptr, 0, nullptr, st);
        if (!rc) rc = decode_gemv(m->sx, C, m->sh, P(m, FCPROJW) + l * 4 * cc, P(m, FCPROJB) + l * C, m->sx2,
                                  B, 4 * C, C, 0, nullptr, 0, nullptr, st);
    }
    if (!rc) rc = layernorm_forward(m->sln, false, m->smean, m->srstd, m->sx, P(m, LNFW), P(m, LNFB), B, C, st);
    if (!rc) rc = decode_gemv(m->slog, c.V, m->sln, P(m, WTE), nullptr, nullptr, B, C, c.V, 0, nullptr, 0, nullptr,
                              st);
    if (!rc) rc = decode_advance(m->dpos, st);
    return rc;
}
}  // namespace gpt2k

GPT2_API int gpt2_decode(gpt2* m, const int* tokens, int B, int pos, float* logits) {
    if (!m) return GPT2_EINVAL;
    const int maxb = std::min(m->cfg.maxB, DECODE_MAXB);
    if (!tokens || !logits || B < 1 || B > maxb || pos < 0 || pos >= std::min(m->cfg.maxT, 1024) ||
        m->cfg.C / m->cfg.H > 64) {
        record(m, GPT2_EINVAL);
        return GPT2_EINVAL;
    }
    if (pos > 0 && (B != m->dec_B || pos != m->dec_next)) {
        record(m, GPT2_ESTATE);
        return GPT2_ESTATE;
    }
    if (!m->dec) {
        int rc = decode_alloc(m);
        if (rc) { record(m, rc); return rc; }
    }
    if (cudaMemcpyAsync(m->stok, tokens, (size_t)B * sizeof(int), cudaMemcpyDefault, m->st) != cudaSuccess) {
        (void)cudaGetLastError();
        record(m, GPT2_ECUDA);
        return GPT2_ECUDA;
    }
    m->fwd_targets = false;                 // the step rows are not a training forward
    // a new sequence starts the device-side position at 0; later calls follow it
    int rc = pos == 0 && cudaMemsetAsync(m->dpos, 0, sizeof(int), m->st) != cudaSuccess ? GPT2_ECUDA : GPT2_OK;
    if (!rc) rc = run_graphed(m, 8, B, 0, [&]() -> int { return decode_impl(m, B); });
    if (!rc && cudaMemcpyAsync(logits, m->slog, (size_t)B * m->cfg.V * sizeof(float), cudaMemcpyDefault, m->st) !=
                   cudaSuccess)
        rc = GPT2_ECUDA;
    if (rc) { (void)cudaGetLastError(); record(m, rc); m->dec_next = -1; return rc; }
    m->dec_B = B;
    m->dec_next = pos + 1;
    return GPT2_OK;
}

GPT2_API int gpt2_set_dropout(gpt2* m, float p, unsigned long long seed) {
    if (!m) return GPT2_EINVAL;
    if (!(p >= 0.f && p < 1.f)) { record(m, GPT2_EINVAL); return GPT2_EINVAL; }
    if (p > 0.f && !m->dbuf) {
        const size_t words = drop_words(m->cfg, m->cfg.maxB, m->cfg.maxT);
        if (cudaStreamSynchronize(m->st) != cudaSuccess ||
            cudaMalloc(reinterpret_cast<void**>(&m->dbuf), words * sizeof(uint32_t)) != cudaSuccess) {
            (void)cudaGetLastError();
            m->dbuf = nullptr;
            record(m, GPT2_ENOMEM);
            return GPT2_ENOMEM;
        }
        m->dbuf_words = words;
    }
    if (p != m->pdrop) {
        // the captured forward and backward differ with and without dropout
        // and carry p in their launches: capture them again
        if (m->gst && cudaStreamSynchronize(m->gst) != cudaSuccess) (void)cudaGetLastError();
        for (auto& g : m->graphs)
            if (g.exec) cudaGraphExecDestroy(g.exec);
        m->graphs.clear();
    }
    m->pdrop = p;
    m->dseed = seed;
    m->dstep = 0;
    m->fwd_targets = false;     // a backward needs a forward under these settings
    return GPT2_OK;
}

GPT2_API int gpt2_destroy(gpt2* m) {
    if (!m) return GPT2_OK;
    int rc = GPT2_OK;
    if (cudaStreamSynchronize(m->st) != cudaSuccess) { (void)cudaGetLastError(); rc = GPT2_ECUDA; }
    if (m->owns_ws && cudaFree(m->ws) != cudaSuccess) { (void)cudaGetLastError(); rc = GPT2_ECUDA; }
    if (m->dec && cudaFree(m->dec) != cudaSuccess) { (void)cudaGetLastError(); rc = GPT2_ECUDA; }
    if (m->dbuf && cudaFree(m->dbuf) != cudaSuccess) { (void)cudaGetLastError(); rc = GPT2_ECUDA; }
    if (m->gst && cudaStreamSynchronize(m->gst) != cudaSuccess) { (void)cudaGetLastError(); rc = GPT2_ECUDA; }
    for (auto& g : m->graphs)
        if (g.exec) cudaGraphExecDestroy(g.exec);
    if (m->gst) cudaStreamDestroy(m->gst);
    if (m->g_in) cudaEventDestroy(m->g_in);
    if (m->g_out) cudaEventDestroy(m->g_out);
    for (cudaEvent_t e : m->trace_events) cudaEventDestroy(e);
    delete m;
    return rc;
}

namespace gpt2k {
int wait_probe(int* status, unsigned long long limit_ns, cudaStream_t st);
}

GPT2_API int gpt2_wait_probe(gpt2* m, int wait_us) {
    if (!m || wait_us < 1 || wait_us > 1000000) return GPT2_EINVAL;
    int rc = wait_probe(&m->flags->status, (unsigned long long)wait_us * 1000ull, m->st);
    if (rc) record(m, rc);
    return rc;
}

GPT2_API int gpt2_status(gpt2* m) {
    if (!m) return GPT2_EINVAL;
    DevFlags h{};
    if (cudaStreamSynchronize(m->st) != cudaSuccess ||
        cudaMemcpy(&h, m->flags, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
        (void)cudaGetLastError();
        record(m, GPT2_ECUDA);
    }
    if (h.status & (GPT2_STATUS_BAD_TOKEN | GPT2_STATUS_BAD_TARGET)) record(m, GPT2_ETOKEN);
    if (h.status & GPT2_STATUS_TIMEOUT) record(m, GPT2_ETIMEOUT);
    int rc = m->err;
    m->err = GPT2_OK;
    if (h.status) cudaMemsetAsync(&m->flags->status, 0, sizeof(int), m->st);
    return rc;
}

GPT2_API const char* gpt2_strerror(int code) {
    switch (code) {
        case GPT2_OK: return "ok";
        case GPT2_EINVAL: return "invalid argument, configuration or shape";
        case GPT2_ENOMEM: return "workspace too small or allocation failed";
        case GPT2_ECUDA: return "CUDA runtime error";
        case GPT2_ETOKEN: return "token or target id outside [0, V)";
        case GPT2_ESTATE: return "calls out of order";
        case GPT2_ETIMEOUT: return "bounded device wait timed out";
        case GPT2_ENOTSUP: return "mode or shape not supported";
        default: return "unknown status";
    }
}

GPT2_API const float* gpt2_grads(gpt2* m) { return m ? m->grads : nullptr; }
GPT2_API float* gpt2_adam_m(gpt2* m) { return m ? m->m : nullptr; }
GPT2_API float* gpt2_adam_v(gpt2* m) { return m ? m->v : nullptr; }
GPT2_API const float* gpt2_logits(gpt2* m, int* row_stride) {
    if (!m) return nullptr;
    if (row_stride) *row_stride = m->Vp;
    return m->logits;
}
GPT2_API const float* gpt2_losses(gpt2* m) { return m ? m->losses : nullptr; }

GPT2_API const float* gpt2_activation(gpt2* m, int which, int layer) {
    if (!m || layer < 0 || layer >= m->cfg.L) return nullptr;
    const size_t R = m->R, C = m->cfg.C, l = layer;
    auto op = [&](char* base, size_t width) { return reinterpret_cast<const float*>(Orow(m, base, l, width)); };
    switch (which) {
        case 0: return m->x0;
        case 1: return op(m->ln1, C);
        case 2: return op(m->qkv, 3 * C);
        case 3: return op(m->atty, C);
        case 4: return m->res2 + l * R * C;
        case 5: return op(m->ln2, C);
        case 6: return op(m->fch, 4 * C);
        case 7: return op(m->fchg, 4 * C);
        case 8: return m->res3 + l * R * C;
        case 9: return reinterpret_cast<const float*>(m->lnf);
        default: return nullptr;
    }
}

GPT2_API int gpt2_trace_enable(gpt2* m, int on) {
    if (!m) return GPT2_EINVAL;
    m->trace_on = on != 0;
    m->trace_used = 0;
    m->trace_cls.clear();
    m->trace_launches.clear();
    return GPT2_OK;
}

GPT2_API int gpt2_trace_read(gpt2* m, double* ms, long long* launches, int n) {
    if (!m || n < 0) return GPT2_EINVAL;
    if (cudaStreamSynchronize(m->st) != cudaSuccess) { (void)cudaGetLastError(); return GPT2_ECUDA; }
    for (int c = 0; c < n; c++) {
        if (ms) ms[c] = 0.0;
        if (launches) launches[c] = 0;
    }
    int rc = GPT2_OK;
    for (size_t i = 0; i < m->trace_cls.size(); i++) {
        int c = m->trace_cls[i];
        float t = 0.f;
        if (cudaEventElapsedTime(&t, m->trace_events[2 * i], m->trace_events[2 * i + 1]) != cudaSuccess) {
            (void)cudaGetLastError();
            rc = GPT2_ECUDA;
        }
        if (c < n) {
            if (ms) ms[c] += t;
            if (launches) launches[c] += m->trace_launches[i];
        }
    }
    m->trace_used = 0;
    m->trace_cls.clear();
    m->trace_launches.clear();
    return rc;
}

GPT2_API long long gpt2_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }
