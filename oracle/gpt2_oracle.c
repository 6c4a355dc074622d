/*
 * gpt2_oracle.c -- plain CPU oracle for one GPT-2 decoder training step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  The product library never
 * links, loads or calls it, and it shares no code with the CUDA path.
 *
 * What it computes, and where the pages say so:
 *   - token + position encoder, pre-norm blocks (ln_1 -> attention -> residual,
 *     ln_2 -> MLP -> residual), final LayerNorm, lm_head tied to the token
 *     embedding:  "GPT-2 from scratch with torch" (Posit blog, Chinese
 *     translation), sections "总体架构", "Transformer block", "输出".
 *   - causal self-attention with 1/sqrt(head size) scaling and -inf masking:
 *     same page, section "近看 Transformer block：自注意力"; the scaling
 *     rationale in "从头搭建GPT(Andrej Karpathy) 笔记", section
 *     "attention中为什么要做scaling".
 *   - MLP c_fc (C->4C), tanh-GELU, c_proj (4C->C): Posit page, section
 *     "近看 Transformer block：前馈网络（MLP）"; the GELU constants in the
 *     Hacker News comments on "GPT-2ベースの3000バイトCで実装された
 *     ChatGPTクローン（2023）".
 *   - softmax cross-entropy (mean over positions, natural log):
 *     "从头搭建GPT(Andrej Karpathy) 笔记", section "计算loss".
 *   - every layer's backward written out by hand and chained, then an Adam
 *     update: "1000 行 C 代码完成 GPT-2 训练的 LLM.c" (bigegpt.com), the
 *     paragraphs on the layer list and on the forward/backward/update loop.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   LayerNorm uses the biased variance with eps = 1e-5 inside the square root;
 *   GELU uses sqrt(2/pi) at full precision; positions are 0..T-1; dropout is
 *   off unless oracle_set_dropout turns it on (then inverted dropout at the
 *   four sites the pages name, with Philox4x32-10 draws: see the dropout
 *   section below); the loss is the mean over all B*T positions; the update is decoupled
 *   AdamW with bias correction, decay only on 2-D weight tensors, applied to
 *   the pre-update parameter value.
 *
 * Precision: the scalar type `real` is double unless ORACLE_FLOAT is defined;
 * the same source builds both.  All loops are plain and unblocked.  OpenMP
 * only splits independent rows/heads across threads; every sum runs in index
 * order inside one thread, so results do not depend on the thread count.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifdef ORACLE_FLOAT
typedef float real;
#define R_EXP expf
#define R_LOG logf
#define R_TANH tanhf
#define R_SQRT sqrtf
#define R_POW powf
#else
typedef double real;
#define R_EXP exp
#define R_LOG log
#define R_TANH tanh
#define R_SQRT sqrt
#define R_POW pow
#endif

#define LN_EPS ((real)1e-5)

int oracle_real_bytes(void) { return (int)sizeof(real); }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Parameter layout.  Sixteen tensors, flat and contiguous, in this order:   */
/*   wte[V,C] wpe[maxT,C] ln1w[L,C] ln1b[L,C] qkvw[L,3C,C] qkvb[L,3C]       */
/*   attprojw[L,C,C] attprojb[L,C] ln2w[L,C] ln2b[L,C] fcw[L,4C,C] fcb[L,4C] */
/*   fcprojw[L,C,4C] fcprojb[L,C] lnfw[C] lnfb[C]                             */
/* Linear weights are [out, in] (the nn_linear convention on the Posit page).*/
/* ------------------------------------------------------------------------ */
#define NTENSORS 16

void oracle_param_sizes(int V, int maxT, int L, int C, size_t* sizes) {
    size_t c = (size_t)C, l = (size_t)L;
    sizes[0] = (size_t)V * c;        /* wte */
    sizes[1] = (size_t)maxT * c;     /* wpe */
    sizes[2] = l * c;                /* ln1w */
    sizes[3] = l * c;                /* ln1b */
    sizes[4] = l * 3 * c * c;        /* qkvw */
    sizes[5] = l * 3 * c;            /* qkvb */
    sizes[6] = l * c * c;            /* attprojw */
    sizes[7] = l * c;                /* attprojb */
    sizes[8] = l * c;                /* ln2w */
    sizes[9] = l * c;                /* ln2b */
    sizes[10] = l * 4 * c * c;       /* fcw */
    sizes[11] = l * 4 * c;           /* fcb */
    sizes[12] = l * c * 4 * c;       /* fcprojw */
    sizes[13] = l * c;               /* fcprojb */
    sizes[14] = c;                   /* lnfw */
    sizes[15] = c;                   /* lnfb */
}

size_t oracle_num_params(int V, int maxT, int L, int C) {
    size_t s[NTENSORS], n = 0;
    oracle_param_sizes(V, maxT, L, C, s);
    for (int i = 0; i < NTENSORS; i++) n += s[i];
    return n;
}

typedef struct {
    real *wte, *wpe, *ln1w, *ln1b, *qkvw, *qkvb, *attprojw, *attprojb;
    real *ln2w, *ln2b, *fcw, *fcb, *fcprojw, *fcprojb, *lnfw, *lnfb;
} Tensors;

static Tensors split_params(real* base, int V, int maxT, int L, int C) {
    size_t s[NTENSORS];
    oracle_param_sizes(V, maxT, L, C, s);
    real* p[NTENSORS];
    real* cur = base;
    for (int i = 0; i < NTENSORS; i++) { p[i] = cur; cur += s[i]; }
    Tensors t = {p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7],
                 p[8], p[9], p[10], p[11], p[12], p[13], p[14], p[15]};
    return t;
}

/* ------------------------------------------------------------------------ */
/* Layers.  Each backward ADDS its contribution into the gradient buffers.   */
/* ------------------------------------------------------------------------ */

/* x[b,t,:] = wte[tok[b,t],:] + wpe[t,:] */
void oracle_encoder_forward(real* x, const int* tok, const real* wte, const real* wpe,
                            int B, int T, int C) {
    for (int b = 0; b < B; b++)
        for (int t = 0; t < T; t++) {
            const real* e = wte + (size_t)tok[b * T + t] * C;
            const real* p = wpe + (size_t)t * C;
            real* o = x + ((size_t)b * T + t) * C;
            for (int c = 0; c < C; c++) o[c] = e[c] + p[c];
        }
}

/* dwte[tok[b,t],:] += dx[b,t,:];  dwpe[t,:] += dx[b,t,:] */
void oracle_encoder_backward(real* dwte, real* dwpe, const real* dx, const int* tok,
                             int B, int T, int C) {
    for (int b = 0; b < B; b++)
        for (int t = 0; t < T; t++) {
            const real* g = dx + ((size_t)b * T + t) * C;
            real* de = dwte + (size_t)tok[b * T + t] * C;
            real* dp = dwpe + (size_t)t * C;
            for (int c = 0; c < C; c++) { de[c] += g[c]; dp[c] += g[c]; }
        }
}

/* Per row: mu = mean(x), var = mean((x-mu)^2), rstd = 1/sqrt(var+eps),
 * y = (x-mu)*rstd*w + b.  mean and rstd are kept for the backward. */
void oracle_layernorm_forward(real* y, real* mean, real* rstd, const real* x,
                              const real* w, const real* b, int N, int C) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const real* xr = x + (size_t)n * C;
        real s = 0;
        for (int c = 0; c < C; c++) s += xr[c];
        real mu = s / C;
        real v = 0;
        for (int c = 0; c < C; c++) { real d = xr[c] - mu; v += d * d; }
        v = v / C;
        real r = 1 / R_SQRT(v + LN_EPS);
        real* yr = y + (size_t)n * C;
        for (int c = 0; c < C; c++) yr[c] = (xr[c] - mu) * r * w[c] + b[c];
        mean[n] = mu;
        rstd[n] = r;
    }
}

/* With xhat = (x-mu)*rstd and g = dy*w:
 *   dx += rstd * (g - mean(g) - xhat * mean(g*xhat))
 *   dw += sum_rows dy*xhat,   db += sum_rows dy                              */
void oracle_layernorm_backward(real* dx, real* dw, real* db, const real* dy,
                               const real* x, const real* w, const real* mean,
                               const real* rstd, int N, int C) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const real* xr = x + (size_t)n * C;
        const real* dyr = dy + (size_t)n * C;
        real mu = mean[n], r = rstd[n];
        real mg = 0, mgx = 0;
        for (int c = 0; c < C; c++) {
            real xh = (xr[c] - mu) * r;
            real g = dyr[c] * w[c];
            mg += g;
            mgx += g * xh;
        }
        mg /= C;
        mgx /= C;
        real* dxr = dx + (size_t)n * C;
        for (int c = 0; c < C; c++) {
            real xh = (xr[c] - mu) * r;
            real g = dyr[c] * w[c];
            dxr[c] += r * (g - mg - xh * mgx);
        }
    }
    /* parameter grads: sum over rows, in row order, one column per thread */
    #pragma omp parallel for schedule(static)
    for (int c = 0; c < C; c++) {
        real sw = 0, sb = 0;
        for (int n = 0; n < N; n++) {
            real xh = (x[(size_t)n * C + c] - mean[n]) * rstd[n];
            real d = dy[(size_t)n * C + c];
            sw += d * xh;
            sb += d;
        }
        dw[c] += sw;
        db[c] += sb;
    }
}

/* y[n,o] = bias[o] + sum_i x[n,i] * w[o,i]   (w is [OC, IC]; bias may be NULL) */
void oracle_matmul_forward(real* y, const real* x, const real* w, const real* bias,
                           int N, int IC, int OC) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const real* xr = x + (size_t)n * IC;
        for (int o = 0; o < OC; o++) {
            const real* wr = w + (size_t)o * IC;
            real s = 0;
            for (int i = 0; i < IC; i++) s += xr[i] * wr[i];
            y[(size_t)n * OC + o] = (bias ? bias[o] : 0) + s;
        }
    }
}

/* dx[n,i] += sum_o dy[n,o] w[o,i];  dw[o,i] += sum_n dy[n,o] x[n,i];
 * dbias[o] += sum_n dy[n,o]   (dbias may be NULL) */
void oracle_matmul_backward(real* dx, real* dw, real* dbias, const real* dy,
                            const real* x, const real* w, int N, int IC, int OC) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        real* dxr = dx + (size_t)n * IC;
        for (int o = 0; o < OC; o++) {
            real d = dy[(size_t)n * OC + o];
            const real* wr = w + (size_t)o * IC;
            for (int i = 0; i < IC; i++) dxr[i] += d * wr[i];
        }
    }
    #pragma omp parallel for schedule(static)
    for (int o = 0; o < OC; o++) {
        real* dwr = dw + (size_t)o * IC;
        real sb = 0;
        for (int n = 0; n < N; n++) {
            real d = dy[(size_t)n * OC + o];
            const real* xr = x + (size_t)n * IC;
            for (int i = 0; i < IC; i++) dwr[i] += d * xr[i];
            sb += d;
        }
        if (dbias) dbias[o] += sb;
    }
}

/* ---- dropout ----------------------------------------------------------------
 * Where: after the token + position embeddings, on the attention weights after
 * the softmax, and on the output of each block's two c_proj layers before the
 * residual addition ("GPT-2 from scratch with torch", sections 总体架构,
 * 近看 Transformer block：自注意力 and 近看 Transformer block：前馈网络（MLP）;
 * "从头搭建GPT(Andrej Karpathy) 笔记", section 继续增加改进的点).  In training
 * each element is kept with probability 1 - p and the kept ones are scaled by
 * 1/(1 - p) (inverted dropout, so evaluation uses every element unscaled).
 *
 * The pages fix no random stream, so the draws come from the counter-based
 * generator Philox4x32-10 (J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC 2011), written from its definition:
 * ten rounds of
 *     (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
 * with M0 = 0xD2511F53, M1 = 0xCD9E8D57 and 32x32->64-bit products, the key
 * (k0, k1) advanced by (0x9E3779B9, 0xBB67AE85) before every round but the
 * first.  Element e (row-major index) of dropout site `site` in forward call
 * `step` under the 64-bit seed:
 *     (w0, w1, w2, w3) = Philox4x32-10(counter (lo32(e/4), hi32(e/4), site, step),
 *                                       key (lo32(seed), hi32(seed)))
 *     keep(e) = w[e mod 4] >= floor(p * 2^32)
 * Sites: 0 the embedding output [B,T,C]; for layer l, 1 + 3l the attention
 * weights [B,NH,T,T], 2 + 3l the attention c_proj output [B,T,C] and 3 + 3l
 * the MLP c_proj output [B,T,C]. */
static void philox_round(uint32_t c[4], const uint32_t k[2]) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k[0];
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = (uint32_t)p1;
    c[2] = n2;
    c[3] = (uint32_t)p0;
}

void oracle_philox4x32_10(uint32_t out[4], const uint32_t ctr[4], const uint32_t key[2]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; r++) {
        if (r > 0) {
            k[0] += 0x9E3779B9u;
            k[1] += 0xBB67AE85u;
        }
        philox_round(c, k);
    }
    for (int i = 0; i < 4; i++) out[i] = c[i];
}

/* keep[e] for elements e = 0 .. n-1 of one site (1 = kept). */
void oracle_dropout_keep(uint8_t* keep, size_t n, uint64_t seed, uint32_t site, uint32_t step,
                         double p) {
    const uint32_t thr = (uint32_t)floor(p * 4294967296.0);
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    #pragma omp parallel for schedule(static)
    for (long long g = 0; g < (long long)((n + 3) / 4); g++) {
        const uint64_t q = (uint64_t)g;
        const uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), site, step};
        uint32_t w[4];
        oracle_philox4x32_10(w, ctr, key);
        for (int i = 0; i < 4; i++) {
            const size_t e = 4 * (size_t)q + i;
            if (e < n) keep[e] = w[i] >= thr;
        }
    }
}

static real dropout_scale(double p) { return (real)1 / ((real)1 - (real)p); }

/* y = x o keep / (1 - p)  (y may be x) */
void oracle_dropout_apply(real* y, const real* x, const uint8_t* keep, size_t n, double p) {
    const real ks = dropout_scale(p);
    for (size_t i = 0; i < n; i++) y[i] = keep[i] ? x[i] * ks : 0;
}

/* Causal multi-head self-attention over qkv[B,T,3C]; columns [0,C) are the
 * queries, [C,2C) the keys, [2C,3C) the values, and head h owns columns
 * h*hs .. h*hs+hs-1 of each (split at C, then viewed as (B,T,NH,hs)).
 * For each (b,h): S = Q K^T / sqrt(hs); S[i,j] = -inf for j > i;
 * P = row softmax(S) (max-subtracted, exact in real arithmetic); O = P V.
 * O is written with the heads side by side: y[b,t,h*hs+d].
 * P is kept, [B,NH,T,T], for the backward (entries above the diagonal are 0).
 * With dropout on the attention weights (keep != NULL, flags [B,NH,T,T]):
 * O = (P o K / (1 - p)) V, K the keep flags; P itself is stored undropped. */
void oracle_attention_forward_dropout(real* y, real* P, const real* qkv, int B, int T, int C,
                                      int NH, const uint8_t* keep, double p) {
    int hs = C / NH;
    real ks = keep ? dropout_scale(p) : (real)1;
    real scale = 1 / R_SQRT((real)hs);
    size_t C3 = (size_t)3 * C;
    #pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++)
        for (int h = 0; h < NH; h++) {
            real* Pbh = P + ((size_t)b * NH + h) * T * T;
            const uint8_t* Kbh = keep ? keep + ((size_t)b * NH + h) * T * T : NULL;
            for (int i = 0; i < T; i++) {
                const real* q = qkv + ((size_t)b * T + i) * C3 + h * hs;
                real* prow = Pbh + (size_t)i * T;
                real mx = -INFINITY;
                for (int j = 0; j <= i; j++) {
                    const real* k = qkv + ((size_t)b * T + j) * C3 + C + h * hs;
                    real s = 0;
                    for (int d = 0; d < hs; d++) s += q[d] * k[d];
                    s *= scale;
                    prow[j] = s;
                    if (s > mx) mx = s;
                }
                real z = 0;
                for (int j = 0; j <= i; j++) { prow[j] = R_EXP(prow[j] - mx); z += prow[j]; }
                for (int j = 0; j <= i; j++) prow[j] /= z;
                for (int j = i + 1; j < T; j++) prow[j] = 0;   /* exp(-inf) */
                real* out = y + ((size_t)b * T + i) * C + h * hs;
                for (int d = 0; d < hs; d++) {
                    real s = 0;
                    for (int j = 0; j <= i; j++) {
                        real a = prow[j];
                        if (Kbh) a = Kbh[(size_t)i * T + j] ? a * ks : 0;
                        s += a * qkv[((size_t)b * T + j) * C3 + 2 * C + h * hs + d];
                    }
                    out[d] = s;
                }
            }
        }
}

void oracle_attention_forward(real* y, real* P, const real* qkv, int B, int T, int C, int NH) {
    oracle_attention_forward_dropout(y, P, qkv, B, T, C, NH, NULL, 0);
}

/* Backward of the attention above, from dy (heads side by side) and the saved P:
 *   dV = P^T dO;  dP = dO V^T;  dS = P o (dP - rowsum(P o dP));
 *   dQ = dS K / sqrt(hs);  dK = dS^T Q / sqrt(hs).   Added into dqkv.
 * With dropout (keep flags K, A = P o K / (1 - p) the weights that met V):
 *   dV = A^T dO;  dP = (dO V^T) o K / (1 - p);  dS as above. */
void oracle_attention_backward_dropout(real* dqkv, const real* dy, const real* qkv, const real* P,
                                       int B, int T, int C, int NH, const uint8_t* keep,
                                       double p) {
    int hs = C / NH;
    real ks = keep ? dropout_scale(p) : (real)1;
    real scale = 1 / R_SQRT((real)hs);
    size_t C3 = (size_t)3 * C;
    #pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++)
        for (int h = 0; h < NH; h++) {
            const real* Pbh = P + ((size_t)b * NH + h) * T * T;
            const uint8_t* Kbh = keep ? keep + ((size_t)b * NH + h) * T * T : NULL;
            real* dS = (real*)malloc(sizeof(real) * (size_t)T);
            real* A = (real*)malloc(sizeof(real) * (size_t)T);
            for (int i = 0; i < T; i++) {
                const real* prow = Pbh + (size_t)i * T;
                for (int j = 0; j <= i; j++)
                    A[j] = Kbh ? (Kbh[(size_t)i * T + j] ? prow[j] * ks : 0) : prow[j];
                const real* dO = dy + ((size_t)b * T + i) * C + h * hs;
                /* dP[i,j] = dO_i . v_j,   D = sum_j P[i,j] dP[i,j] */
                real D = 0;
                for (int j = 0; j <= i; j++) {
                    const real* v = qkv + ((size_t)b * T + j) * C3 + 2 * C + h * hs;
                    real dp = 0;
                    for (int d = 0; d < hs; d++) dp += dO[d] * v[d];
                    if (Kbh) dp = Kbh[(size_t)i * T + j] ? dp * ks : 0;
                    dS[j] = dp;
                    D += prow[j] * dp;
                }
                for (int j = 0; j <= i; j++) dS[j] = prow[j] * (dS[j] - D);
                const real* q = qkv + ((size_t)b * T + i) * C3 + h * hs;
                real* dq = dqkv + ((size_t)b * T + i) * C3 + h * hs;
                for (int j = 0; j <= i; j++) {
                    const real* k = qkv + ((size_t)b * T + j) * C3 + C + h * hs;
                    real* dk = dqkv + ((size_t)b * T + j) * C3 + C + h * hs;
                    real* dv = dqkv + ((size_t)b * T + j) * C3 + 2 * C + h * hs;
                    for (int d = 0; d < hs; d++) {
                        dq[d] += dS[j] * k[d] * scale;
                        dk[d] += dS[j] * q[d] * scale;
                        dv[d] += A[j] * dO[d];
                    }
                }
            }
            free(dS);
            free(A);
        }
}

void oracle_attention_backward(real* dqkv, const real* dy, const real* qkv, const real* P,
                               int B, int T, int C, int NH) {
    oracle_attention_backward_dropout(dqkv, dy, qkv, P, B, T, C, NH, NULL, 0);
}

/* GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
#define GELU_K ((real)0.044715)
static real gelu_s(void) { return R_SQRT((real)2 / (real)3.14159265358979323846); }

void oracle_gelu_forward(real* y, const real* x, size_t n) {
    real s = gelu_s();
    #pragma omp parallel for schedule(static)
    for (size_t i = 0; i < n; i++) {
        real v = x[i];
        y[i] = (real)0.5 * v * (1 + R_TANH(s * (v + GELU_K * v * v * v)));
    }
}

/* d/dx gelu = 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) s (1 + 3 k x^2),
 * u = s (x + k x^3).   dx += dy * gelu'(x). */
void oracle_gelu_backward(real* dx, const real* x, const real* dy, size_t n) {
    real s = gelu_s();
    #pragma omp parallel for schedule(static)
    for (size_t i = 0; i < n; i++) {
        real v = x[i];
        real th = R_TANH(s * (v + GELU_K * v * v * v));
        real d = (real)0.5 * (1 + th) + (real)0.5 * v * (1 - th * th) * s * (1 + 3 * GELU_K * v * v);
        dx[i] += dy[i] * d;
    }
}

/* Cross-entropy over V classes, rows of stride `ld` (>= V; columns >= V are
 * ignored).  losses[n] = logsumexp(z_n) - z_n[tgt_n]  (natural log),
 * probs[n,:] = softmax(z_n) (max-subtracted).  Returns the mean loss. */
real oracle_crossentropy_forward(real* losses, real* probs, const real* z, const int* tgt,
                                 int N, int V, int ld) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const real* zr = z + (size_t)n * ld;
        real mx = -INFINITY;
        for (int v = 0; v < V; v++) if (zr[v] > mx) mx = zr[v];
        real s = 0;
        for (int v = 0; v < V; v++) s += R_EXP(zr[v] - mx);
        real lse = mx + R_LOG(s);
        losses[n] = lse - zr[tgt[n]];
        if (probs) {
            real* pr = probs + (size_t)n * V;
            for (int v = 0; v < V; v++) pr[v] = R_EXP(zr[v] - mx) / s;
        }
    }
    real tot = 0;
    for (int n = 0; n < N; n++) tot += losses[n];
    return tot / N;
}

/* d(mean loss)/dz[n,v] = (probs[n,v] - [v == tgt_n]) / N, added into dz */
void oracle_crossentropy_backward(real* dz, const real* probs, const int* tgt, int N, int V,
                                  int ld) {
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++)
        for (int v = 0; v < V; v++)
            dz[(size_t)n * ld + v] += (probs[(size_t)n * V + v] - (v == tgt[n] ? 1 : 0)) / N;
}

/* AdamW on n values, t >= 1:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   mhat = m / (1-b1^t);  vhat = v / (1-b2^t);
 *   p -= lr * (mhat / (sqrt(vhat) + eps) + wd * p)     (p before the update) */
void oracle_adamw(real* p, const real* g, real* m, real* v, size_t n, real lr, real b1,
                  real b2, real eps, real wd, int t) {
    real c1 = 1 - R_POW(b1, (real)t), c2 = 1 - R_POW(b2, (real)t);
    #pragma omp parallel for schedule(static)
    for (size_t i = 0; i < n; i++) {
        m[i] = b1 * m[i] + (1 - b1) * g[i];
        v[i] = b2 * v[i] + (1 - b2) * g[i] * g[i];
        real mh = m[i] / c1, vh = v[i] / c2;
        p[i] -= lr * (mh / (R_SQRT(vh) + eps) + wd * p[i]);
    }
}

/* ------------------------------------------------------------------------ */
/* Whole model.                                                             */
/* ------------------------------------------------------------------------ */
typedef struct {
    int V, maxT, L, NH, C, B, T;
    int last_only;      /* lm_head and loss on the last position of each row only */
    size_t nparams;
    /* activations, per layer l (N = B*T rows) */
    real *x0;           /* [N,C] encoder output */
    real *ln1, *ln1_mean, *ln1_rstd;     /* [L,N,C], [L,N], [L,N] */
    real *qkv;          /* [L,N,3C] */
    real *atty;         /* [L,N,C] */
    real *P;            /* [L,B,NH,T,T] */
    real *res2;         /* [L,N,C] residual after attention */
    real *ln2, *ln2_mean, *ln2_rstd;
    real *h;            /* [L,N,4C] pre-activation */
    real *g;            /* [L,N,4C] GELU output */
    real *res3;         /* [L,N,C] residual after the MLP (block output) */
    real *lnf, *lnf_mean, *lnf_rstd;     /* [N,C], [N], [N] */
    real *logits;       /* [NL,V] */
    real *probs;        /* [NL,V] */
    real *losses;       /* [NL] */
    int *tok, *tgt;     /* [N] copies */
    int has_targets;
    real loss;
    /* dropout (off unless oracle_set_dropout turned it on) */
    int drop_on;
    double pdrop;
    uint64_t seed;
    uint32_t step;
    uint8_t *keep_emb;  /* [N,C]          site 0        */
    uint8_t *keep_att;  /* [L,B,NH,T,T]   sites 1 + 3l  */
    uint8_t *keep_ap;   /* [L,N,C]        sites 2 + 3l  */
    uint8_t *keep_fp;   /* [L,N,C]        sites 3 + 3l  */
} OracleModel;

static real* zalloc(size_t n) { return (real*)calloc(n ? n : 1, sizeof(real)); }

/* number of rows that reach lm_head */
static int lm_rows(const OracleModel* m) { return m->last_only ? m->B : m->B * m->T; }

OracleModel* oracle_create(int V, int maxT, int L, int NH, int C, int B, int T, int last_only) {
    if (C % NH != 0 || T > maxT || T < 1 || B < 1) return NULL;
    OracleModel* m = (OracleModel*)calloc(1, sizeof(OracleModel));
    m->V = V; m->maxT = maxT; m->L = L; m->NH = NH; m->C = C; m->B = B; m->T = T;
    m->last_only = last_only;
    m->nparams = oracle_num_params(V, maxT, L, C);
    size_t N = (size_t)B * T, c = (size_t)C, l = (size_t)L;
    m->x0 = zalloc(N * c);
    m->ln1 = zalloc(l * N * c); m->ln1_mean = zalloc(l * N); m->ln1_rstd = zalloc(l * N);
    m->qkv = zalloc(l * N * 3 * c);
    m->atty = zalloc(l * N * c);
    m->P = zalloc(l * (size_t)B * NH * T * T);
    m->res2 = zalloc(l * N * c);
    m->ln2 = zalloc(l * N * c); m->ln2_mean = zalloc(l * N); m->ln2_rstd = zalloc(l * N);
    m->h = zalloc(l * N * 4 * c);
    m->g = zalloc(l * N * 4 * c);
    m->res3 = zalloc(l * N * c);
    m->lnf = zalloc(N * c); m->lnf_mean = zalloc(N); m->lnf_rstd = zalloc(N);
    size_t NL = (size_t)lm_rows(m);
    m->logits = zalloc(NL * V);
    m->probs = zalloc(NL * V);
    m->losses = zalloc(NL);
    m->tok = (int*)calloc(N, sizeof(int));
    m->tgt = (int*)calloc(N, sizeof(int));
    return m;
}

void oracle_free(OracleModel* m) {
    if (!m) return;
    real* bufs[] = {m->x0, m->ln1, m->ln1_mean, m->ln1_rstd, m->qkv, m->atty, m->P, m->res2,
                    m->ln2, m->ln2_mean, m->ln2_rstd, m->h, m->g, m->res3, m->lnf,
                    m->lnf_mean, m->lnf_rstd, m->logits, m->probs, m->losses};
    for (size_t i = 0; i < sizeof(bufs) / sizeof(bufs[0]); i++) free(bufs[i]);
    free(m->tok); free(m->tgt);
    free(m->keep_emb); free(m->keep_att); free(m->keep_ap); free(m->keep_fp);
    free(m);
}

/* Dropout for the following forward calls: probability p in [0, 1) of zeroing
 * an element, draws from (seed, step) as the dropout section above defines.
 * p < 0 turns dropout off.  p = 0 keeps every element (scale 1).  Returns 0,
 * or -1 when p >= 1 or memory runs out. */
int oracle_set_dropout(OracleModel* m, double p, uint64_t seed, uint32_t step) {
    if (p >= 1) return -1;
    m->drop_on = p >= 0;
    m->pdrop = p;
    m->seed = seed;
    m->step = step;
    if (!m->drop_on || m->keep_emb) return 0;
    size_t N = (size_t)m->B * m->T, NC = N * m->C, l = (size_t)m->L;
    m->keep_emb = (uint8_t*)calloc(NC, 1);
    m->keep_att = (uint8_t*)calloc(l * m->B * m->NH * (size_t)m->T * m->T, 1);
    m->keep_ap = (uint8_t*)calloc(l * NC, 1);
    m->keep_fp = (uint8_t*)calloc(l * NC, 1);
    if (!m->keep_emb || !m->keep_att || !m->keep_ap || !m->keep_fp) return -1;
    return 0;
}

/* The keep flags of the last forward: which 0 embedding, 1 attention weights,
 * 2 attention c_proj, 3 MLP c_proj; layer l for 1..3. */
const uint8_t* oracle_keep(const OracleModel* m, int which, int l) {
    size_t NC = (size_t)m->B * m->T * m->C;
    if (!m->drop_on) return NULL;
    switch (which) {
        case 0: return m->keep_emb;
        case 1: return m->keep_att + (size_t)l * m->B * m->NH * m->T * m->T;
        case 2: return m->keep_ap + l * NC;
        case 3: return m->keep_fp + l * NC;
        default: return NULL;
    }
}

/* The block input of layer l: the encoder output for l = 0, else the output
 * of block l-1. */
static const real* block_input(const OracleModel* m, int l) {
    size_t NC = (size_t)m->B * m->T * m->C;
    return l == 0 ? m->x0 : m->res3 + (size_t)(l - 1) * NC;
}

/* Forward pass.  Returns the mean loss, or NAN when tgt is NULL. */
real oracle_forward(OracleModel* m, real* params, const int* tok, const int* tgt) {
    int B = m->B, T = m->T, C = m->C, L = m->L, NH = m->NH, V = m->V;
    size_t N = (size_t)B * T, NC = N * C;
    Tensors w = split_params(params, V, m->maxT, L, C);
    memcpy(m->tok, tok, N * sizeof(int));
    m->has_targets = tgt != NULL;
    if (tgt) memcpy(m->tgt, tgt, N * sizeof(int));

    oracle_encoder_forward(m->x0, tok, w.wte, w.wpe, B, T, C);
    const int drop = m->drop_on;
    const size_t att_n = (size_t)B * NH * T * T;
    if (drop) {
        oracle_dropout_keep(m->keep_emb, NC, m->seed, 0, m->step, m->pdrop);
        oracle_dropout_apply(m->x0, m->x0, m->keep_emb, NC, m->pdrop);
    }
    for (int l = 0; l < L; l++) {
        const real* x = block_input(m, l);
        real* ln1 = m->ln1 + l * NC;
        real* qkv = m->qkv + l * 3 * NC;
        real* atty = m->atty + l * NC;
        real* P = m->P + (size_t)l * B * NH * T * T;
        real* res2 = m->res2 + l * NC;
        real* ln2 = m->ln2 + l * NC;
        real* h = m->h + l * 4 * NC;
        real* g = m->g + l * 4 * NC;
        real* res3 = m->res3 + l * NC;
        size_t cc = (size_t)C * C;
        oracle_layernorm_forward(ln1, m->ln1_mean + l * N, m->ln1_rstd + l * N, x,
                                 w.ln1w + l * C, w.ln1b + l * C, (int)N, C);
        oracle_matmul_forward(qkv, ln1, w.qkvw + l * 3 * cc, w.qkvb + l * 3 * C, (int)N, C, 3 * C);
        const uint8_t* katt = NULL;
        if (drop) {
            uint8_t* ka = m->keep_att + l * att_n;
            oracle_dropout_keep(ka, att_n, m->seed, 1 + 3 * (uint32_t)l, m->step, m->pdrop);
            oracle_dropout_keep(m->keep_ap + l * NC, NC, m->seed, 2 + 3 * (uint32_t)l, m->step, m->pdrop);
            oracle_dropout_keep(m->keep_fp + l * NC, NC, m->seed, 3 + 3 * (uint32_t)l, m->step, m->pdrop);
            katt = ka;
        }
        oracle_attention_forward_dropout(atty, P, qkv, B, T, C, NH, katt, m->pdrop);
        oracle_matmul_forward(res2, atty, w.attprojw + l * cc, w.attprojb + l * C, (int)N, C, C);
        if (drop) oracle_dropout_apply(res2, res2, m->keep_ap + l * NC, NC, m->pdrop);
        for (size_t i = 0; i < NC; i++) res2[i] += x[i];            /* residual */
        oracle_layernorm_forward(ln2, m->ln2_mean + l * N, m->ln2_rstd + l * N, res2,
                                 w.ln2w + l * C, w.ln2b + l * C, (int)N, C);
        oracle_matmul_forward(h, ln2, w.fcw + l * 4 * cc, w.fcb + l * 4 * C, (int)N, C, 4 * C);
        oracle_gelu_forward(g, h, 4 * NC);
        oracle_matmul_forward(res3, g, w.fcprojw + l * 4 * cc, w.fcprojb + l * C, (int)N, 4 * C, C);
        if (drop) oracle_dropout_apply(res3, res3, m->keep_fp + l * NC, NC, m->pdrop);
        for (size_t i = 0; i < NC; i++) res3[i] += res2[i];         /* residual */
    }
    const real* xL = block_input(m, L);
    oracle_layernorm_forward(m->lnf, m->lnf_mean, m->lnf_rstd, xL, w.lnfw, w.lnfb, (int)N, C);

    /* tied lm_head: logits = lnf . wte^T (no bias) */
    int NL = lm_rows(m);
    const real* lm_in = m->lnf;
    real* tmp = NULL;
    int* tgt_rows = m->tgt;
    int* tgt_last = NULL;
    if (m->last_only) {
        tmp = zalloc((size_t)B * C);
        tgt_last = (int*)calloc(B, sizeof(int));
        for (int b = 0; b < B; b++) {
            memcpy(tmp + (size_t)b * C, m->lnf + ((size_t)b * T + T - 1) * C, C * sizeof(real));
            tgt_last[b] = m->tgt[(size_t)b * T + T - 1];
        }
        lm_in = tmp;
        tgt_rows = tgt_last;
    }
    oracle_matmul_forward(m->logits, lm_in, w.wte, NULL, NL, C, V);
    m->loss = NAN;
    if (tgt) m->loss = oracle_crossentropy_forward(m->losses, m->probs, m->logits, tgt_rows, NL, V, V);
    free(tmp);
    free(tgt_last);
    return m->loss;
}

/* Backward pass of the mean loss.  Overwrites grads (same layout as params).
 * Requires a forward with targets on the full sequence (last_only == 0). */
int oracle_backward(OracleModel* m, real* params, real* grads) {
    if (!m->has_targets || m->last_only) return -1;
    int B = m->B, T = m->T, C = m->C, L = m->L, NH = m->NH, V = m->V;
    size_t N = (size_t)B * T, NC = N * C, cc = (size_t)C * C;
    memset(grads, 0, m->nparams * sizeof(real));
    Tensors w = split_params(params, V, m->maxT, L, C);
    Tensors d = split_params(grads, V, m->maxT, L, C);

    real* dz = zalloc(N * V);
    real* dlnf = zalloc(NC);
    real* dres = zalloc(NC);     /* gradient w.r.t. the residual stream */
    real* dtmp = zalloc(NC);     /* gradient w.r.t. an LN output        */
    real* dg = zalloc(4 * NC);
    real* dh = zalloc(4 * NC);
    real* datty = zalloc(NC);
    real* dqkv = zalloc(3 * NC);
    real* dbr = zalloc(NC);      /* gradient w.r.t. a c_proj output (through dropout) */
    const int drop = m->drop_on;
    const size_t att_n = (size_t)B * NH * T * T;

    oracle_crossentropy_backward(dz, m->probs, m->tgt, (int)N, V, V);
    oracle_matmul_backward(dlnf, d.wte, NULL, dz, m->lnf, w.wte, (int)N, C, V);
    oracle_layernorm_backward(dres, d.lnfw, d.lnfb, dlnf, block_input(m, L), w.lnfw,
                              m->lnf_mean, m->lnf_rstd, (int)N, C);
    for (int l = L - 1; l >= 0; l--) {
        const real* x = block_input(m, l);
        /* MLP branch: res3 = res2 + fcproj(gelu(fc(ln2(res2)))) */
        memset(dg, 0, 4 * NC * sizeof(real));
        memset(dh, 0, 4 * NC * sizeof(real));
        memset(dtmp, 0, NC * sizeof(real));
        if (drop) oracle_dropout_apply(dbr, dres, m->keep_fp + l * NC, NC, m->pdrop);
        oracle_matmul_backward(dg, d.fcprojw + l * 4 * cc, d.fcprojb + l * C, drop ? dbr : dres,
                               m->g + l * 4 * NC, w.fcprojw + l * 4 * cc, (int)N, 4 * C, C);
        oracle_gelu_backward(dh, m->h + l * 4 * NC, dg, 4 * NC);
        oracle_matmul_backward(dtmp, d.fcw + l * 4 * cc, d.fcb + l * 4 * C, dh,
                               m->ln2 + l * NC, w.fcw + l * 4 * cc, (int)N, C, 4 * C);
        oracle_layernorm_backward(dres, d.ln2w + l * C, d.ln2b + l * C, dtmp, m->res2 + l * NC,
                                  w.ln2w + l * C, m->ln2_mean + l * N, m->ln2_rstd + l * N,
                                  (int)N, C);
        /* attention branch: res2 = x + attproj(attn(qkv(ln1(x)))) */
        memset(datty, 0, NC * sizeof(real));
        memset(dqkv, 0, 3 * NC * sizeof(real));
        memset(dtmp, 0, NC * sizeof(real));
        if (drop) oracle_dropout_apply(dbr, dres, m->keep_ap + l * NC, NC, m->pdrop);
        oracle_matmul_backward(datty, d.attprojw + l * cc, d.attprojb + l * C, drop ? dbr : dres,
                               m->atty + l * NC, w.attprojw + l * cc, (int)N, C, C);
        oracle_attention_backward_dropout(dqkv, datty, m->qkv + l * 3 * NC,
                                          m->P + (size_t)l * att_n, B, T, C, NH,
                                          drop ? m->keep_att + l * att_n : NULL, m->pdrop);
        oracle_matmul_backward(dtmp, d.qkvw + l * 3 * cc, d.qkvb + l * 3 * C, dqkv,
                               m->ln1 + l * NC, w.qkvw + l * 3 * cc, (int)N, C, 3 * C);
        oracle_layernorm_backward(dres, d.ln1w + l * C, d.ln1b + l * C, dtmp, x,
                                  w.ln1w + l * C, m->ln1_mean + l * N, m->ln1_rstd + l * N,
                                  (int)N, C);
    }
    if (drop) oracle_dropout_apply(dres, dres, m->keep_emb, NC, m->pdrop);
    oracle_encoder_backward(d.wte, d.wpe, dres, m->tok, B, T, C);
    free(dz); free(dlnf); free(dres); free(dtmp); free(dg); free(dh); free(datty); free(dqkv);
    free(dbr);
    return 0;
}

/* AdamW over the whole model: decay only on the 2-D weight tensors
 * (wte, wpe, qkvw, attprojw, fcw, fcprojw). */
void oracle_adamw_model(OracleModel* m, real* params, const real* grads, real* am, real* av,
                        real lr, real b1, real b2, real eps, real wd, int t) {
    size_t s[NTENSORS];
    oracle_param_sizes(m->V, m->maxT, m->L, m->C, s);
    static const int is2d[NTENSORS] = {1, 1, 0, 0, 1, 0, 1, 0, 0, 0, 1, 0, 1, 0, 0, 0};
    size_t off = 0;
    for (int i = 0; i < NTENSORS; i++) {
        oracle_adamw(params + off, grads + off, am + off, av + off, s[i], lr, b1, b2, eps,
                     is2d[i] ? wd : 0, t);
        off += s[i];
    }
}

/* Accessors for the tests. */
real oracle_loss(const OracleModel* m) { return m->loss; }
const real* oracle_logits(const OracleModel* m) { return m->logits; }
const real* oracle_probs(const OracleModel* m) { return m->probs; }
const real* oracle_losses(const OracleModel* m) { return m->losses; }
const real* oracle_act(const OracleModel* m, int which, int l) {
    size_t N = (size_t)m->B * m->T, NC = N * m->C;
    switch (which) {
        case 0: return m->x0;
        case 1: return m->ln1 + l * NC;
        case 2: return m->qkv + l * 3 * NC;
        case 3: return m->atty + l * NC;
        case 4: return m->res2 + l * NC;
        case 5: return m->ln2 + l * NC;
        case 6: return m->h + l * 4 * NC;
        case 7: return m->g + l * 4 * NC;
        case 8: return m->res3 + l * NC;
        case 9: return m->lnf;
        case 10: return m->P + (size_t)l * m->B * m->NH * m->T * m->T;
        case 11: return m->ln1_mean + l * N;
        case 12: return m->ln1_rstd + l * N;
        default: return NULL;
    }
}
