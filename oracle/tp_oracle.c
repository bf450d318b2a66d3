/*
 * tp_oracle.c -- plain, slow, fp64 CPU oracle of the Megatron-style
 * tensor-parallel transformer block.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the bench's
 * CPU-baseline leg load this library.  The CUDA product path never links,
 * imports or calls it, and it shares no code, header or table with that path.
 *
 * Every routine is the plain definition written out with straightforward
 * loops in double precision, with no blocking, fusion or reordering beyond
 * what the definition states.  OpenMP only splits independent output rows
 * across threads; the arithmetic of every output element is unchanged.
 *
 * Sources (web pages; cited by title and section):
 *  - "텐서 병렬화" (itwiki, Tensor parallelism): sections "행렬 곱 나누기"
 *    (splitting a matrix product: column- and row-parallel table), "MLP"
 *    (Z = GeLU(XA)B = sum_i GeLU(X A_i) B_i; SwiGLU form
 *    W2(SiLU(X W1) (.) X W3)), "셀프 어텐션" (self-attention: heads are
 *    independent, a/t heads per device, GQA KV heads replicated when fewer
 *    than t), "통신 연산 f와 g" (f = identity forward, g = all-reduce forward;
 *    norm, dropout and residual replicated).
 *  - "추론을 위한 텐서 병렬성" (transformers docs, Tensor parallelism for
 *    inference), section "설계 구현 / DTensor": a rowwise layer's bias is
 *    replicated and added once after the reduction.
 *  - "Tensor 병렬성" (diffusers docs), section "제약 조건 및 검증"
 *    (constraints and validation): tp_degree must divide the head count.
 *
 * Layouts: row-major; weights use the nn.Linear layout W[out][in]; the pages'
 * A (h x f, Y = XA) is W1 transposed.  Activations are [tokens][features],
 * tokens = batch * seq with sequence-major order (token = b * seq + p).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define TPO_OK 0
#define TPO_ERR_INVALID 1
#define TPO_ERR_NOT_DIVISIBLE 2
#define TPO_ERR_NOMEM 3

#define TPO_ACT_GELU_ERF 0
#define TPO_ACT_GELU_TANH 1
#define TPO_ACT_SWIGLU 2
#define TPO_ACT_NONE 3

int tpo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- scalars */

/* GeLU, exact form x * Phi(x) = x/2 * (1 + erf(x / sqrt 2)).  The worked MLP
 * example ("MLP" section) calls torch's F.gelu, whose default is this form. */
double tpo_gelu_erf(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }

/* GeLU, tanh approximation (an option; the pages never name it). */
double tpo_gelu_tanh(double x) {
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

/* SiLU(x) = x * sigmoid(x), the gate of the SwiGLU MLP ("MLP" section). */
double tpo_silu(double x) { return x / (1.0 + exp(-x)); }

static double act_scalar(int act, double x) {
    switch (act) {
    case TPO_ACT_GELU_ERF: return tpo_gelu_erf(x);
    case TPO_ACT_GELU_TANH: return tpo_gelu_tanh(x);
    case TPO_ACT_SWIGLU: return tpo_silu(x);
    default: return x;
    }
}

/* Round a double to the nearest bf16 (ties to even), returning its bits.
 * Used only where a test compares a value that is exactly representable in
 * fp32 (integer-valued data), so rounding straight from double is the same
 * decision the GPU takes from fp32. */
uint16_t tpo_round_bf16(double x) {
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)(u >> 16); /* inf/nan */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- linear */

/* Y[m][n] = sum_k X[m][k] * W[n][k]   (Y = X W^T, nn.Linear without bias).
 * Row strides ldx, ldw, ldy are in elements. */
void tpo_linear(const double* X, int64_t ldx, const double* W, int64_t ldw,
                int64_t M, int64_t N, int64_t K, double* Y, int64_t ldy) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const double* x = X + m * ldx;
        for (int64_t n = 0; n < N; ++n) {
            const double* w = W + n * ldw;
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += x[k] * w[k];
            Y[m * ldy + n] = s;
        }
    }
}

/* ---------------------------------------------------------------- MLP */

/* Unsharded MLP ("MLP" section):
 *   GeLU / none :  Z = act(X W1^T) W2^T            (the page's GeLU(XA)B)
 *   SwiGLU      :  Z = (SiLU(X W1^T) (.) (X W3^T)) W2^T
 * X[M][h], W1/W3[f][h], W2[h][f], Z[M][h]. */
int tpo_mlp(int act, int64_t M, int64_t h, int64_t f, const double* X,
            const double* W1, const double* W3, const double* W2, double* Z) {
    if (M < 0 || h <= 0 || f <= 0 || !X || !W1 || !W2 || !Z) return TPO_ERR_INVALID;
    if (act == TPO_ACT_SWIGLU && !W3) return TPO_ERR_INVALID;
    double* U = (double*)malloc(sizeof(double) * (size_t)(M * f + 1));
    double* G = NULL;
    if (!U) return TPO_ERR_NOMEM;
    tpo_linear(X, h, W1, h, M, f, h, U, f);
    if (act == TPO_ACT_SWIGLU) {
        G = (double*)malloc(sizeof(double) * (size_t)(M * f + 1));
        if (!G) { free(U); return TPO_ERR_NOMEM; }
        tpo_linear(X, h, W3, h, M, f, h, G, f);
        for (int64_t e = 0; e < M * f; ++e) U[e] = tpo_silu(U[e]) * G[e];
    } else {
        for (int64_t e = 0; e < M * f; ++e) U[e] = act_scalar(act, U[e]);
    }
    tpo_linear(U, f, W2, f, M, h, f, Z, h);
    free(U);
    free(G);
    return TPO_OK;
}

/* Sharded MLP, the literal t-device form ("MLP" section, and the column /
 * row-parallel table of "행렬 곱 나누기"):
 *   A_i = columns [i f/t, (i+1) f/t) of A      = rows of W1 (and W3)
 *   B_i = rows    [i f/t, (i+1) f/t) of B      = columns of W2
 *   Y_i = act(X A_i)            (no communication: X is replicated, f = id)
 *   P_i = Y_i B_i               (the partial sum device i holds)
 *   Z   = sum_{i=0}^{t-1} P_i   (g: the one all-reduce), summed i ascending
 * Chunks are contiguous and equal, so t must divide f.
 * partials (nullable) receives P_i as [t][M][h]. */
int tpo_mlp_sharded(int act, int64_t M, int64_t h, int64_t f, int64_t t,
                    const double* X, const double* W1, const double* W3,
                    const double* W2, double* partials, double* Z) {
    if (M < 0 || h <= 0 || f <= 0 || t <= 0 || !X || !W1 || !W2 || !Z) return TPO_ERR_INVALID;
    if (act == TPO_ACT_SWIGLU && !W3) return TPO_ERR_INVALID;
    if (f % t) return TPO_ERR_NOT_DIVISIBLE;
    const int64_t w = f / t;
    double* Y = (double*)malloc(sizeof(double) * (size_t)(M * w + 1));
    double* G = (double*)malloc(sizeof(double) * (size_t)(M * w + 1));
    double* P = (double*)malloc(sizeof(double) * (size_t)(t * M * h + 1));
    if (!Y || !G || !P) { free(Y); free(G); free(P); return TPO_ERR_NOMEM; }
    for (int64_t i = 0; i < t; ++i) {
        const double* W1_i = W1 + i * w * h;          /* rows of W1 */
        tpo_linear(X, h, W1_i, h, M, w, h, Y, w);
        if (act == TPO_ACT_SWIGLU) {
            const double* W3_i = W3 + i * w * h;
            tpo_linear(X, h, W3_i, h, M, w, h, G, w);
            for (int64_t e = 0; e < M * w; ++e) Y[e] = tpo_silu(Y[e]) * G[e];
        } else {
            for (int64_t e = 0; e < M * w; ++e) Y[e] = act_scalar(act, Y[e]);
        }
        const double* W2_i = W2 + i * w;               /* columns of W2, row stride f */
        tpo_linear(Y, w, W2_i, f, M, h, w, P + i * M * h, h);
    }
    for (int64_t e = 0; e < M * h; ++e) {
        double s = 0.0;
        for (int64_t i = 0; i < t; ++i) s += P[i * M * h + e];
        Z[e] = s;
    }
    if (partials) memcpy(partials, P, sizeof(double) * (size_t)(t * M * h));
    free(Y);
    free(G);
    free(P);
    return TPO_OK;
}

/* Single-precision restatement of the worked example's two forms (the page's
 * listing runs in fp32 and compares with atol 1e-4).  A is [h][f] and B is
 * [f][h] in the page's own orientation (Y = XA).  sharded != 0 selects
 * sum_i GeLU(X A_i) B_i, else GeLU(XA)B.  Accumulation is float. */
int tpo_mlp_worked_f32(int sharded, int64_t b, int64_t h, int64_t f, int64_t t,
                       const float* X, const float* A, const float* B, float* Z) {
    if (b <= 0 || h <= 0 || f <= 0 || t <= 0 || (f % t)) return TPO_ERR_INVALID;
    const int64_t nsh = sharded ? t : 1, w = f / nsh;
    for (int64_t e = 0; e < b * h; ++e) Z[e] = 0.0f;
    float* Y = (float*)malloc(sizeof(float) * (size_t)(b * w));
    float* P = (float*)malloc(sizeof(float) * (size_t)(b * h));
    if (!Y || !P) { free(Y); free(P); return TPO_ERR_NOMEM; }
    for (int64_t i = 0; i < nsh; ++i) {
        for (int64_t r = 0; r < b; ++r)
            for (int64_t c = 0; c < w; ++c) {
                float s = 0.0f;
                for (int64_t k = 0; k < h; ++k) s += X[r * h + k] * A[k * f + i * w + c];
                Y[r * w + c] = 0.5f * s * (1.0f + erff(s / sqrtf(2.0f)));
            }
        for (int64_t r = 0; r < b; ++r)
            for (int64_t c = 0; c < h; ++c) {
                float s = 0.0f;
                for (int64_t k = 0; k < w; ++k) s += Y[r * w + k] * B[(i * w + k) * h + c];
                P[r * h + c] = s;
            }
        for (int64_t e = 0; e < b * h; ++e) Z[e] += P[e];
    }
    free(Y);
    free(P);
    return TPO_OK;
}

/* ---------------------------------------------------------------- plan */

/* Validation of a t-way split ("제약 조건 및 검증" of the diffusers page:
 * tp_degree must divide the attention heads; "셀프 어텐션" of the itwiki
 * page: the head count must divide by t, KV heads are taken into account and
 * replicated when fewer than t).  Reading for GQA: a % k == 0 (each KV head
 * serves a/k consecutive query heads); if k >= t then t | k, else k | t.
 * The MLP's column chunks are equal, so t | f.  Sizes of 0 mean "absent". */
int tpo_plan_check(int64_t h, int64_t f, int64_t a, int64_t k, int64_t d, int64_t t) {
    if (h <= 0 || t <= 0 || f < 0 || a < 0 || k < 0 || d < 0) return TPO_ERR_INVALID;
    if (f > 0 && f % t) return TPO_ERR_NOT_DIVISIBLE;
    if (a > 0) {
        if (k <= 0 || d <= 0) return TPO_ERR_INVALID;
        if (a % t) return TPO_ERR_NOT_DIVISIBLE;
        if (a % k) return TPO_ERR_NOT_DIVISIBLE;
        if (k >= t) { if (k % t) return TPO_ERR_NOT_DIVISIBLE; }
        else if (t % k) return TPO_ERR_NOT_DIVISIBLE;
    }
    return TPO_OK;
}

/* Query head j lives on device floor(j / (a/t)) (a/t heads per device). */
int64_t tpo_q_head_shard(int64_t a, int64_t t, int64_t j) { return j / (a / t); }

/* Query head j reads KV head floor(j / (a/k)) (consecutive grouping). */
int64_t tpo_q_head_kv(int64_t a, int64_t k, int64_t j) { return j / (a / k); }

/* First KV head held by device i, and how many it holds: k/t own heads when
 * k >= t, else one replica of KV head floor(i k / t). */
int64_t tpo_shard_kv_first(int64_t k, int64_t t, int64_t i) {
    return (k >= t) ? i * (k / t) : (i * k) / t;
}
int64_t tpo_shard_kv_count(int64_t k, int64_t t) { return (k >= t) ? k / t : 1; }

/* ---------------------------------------------------------------- attention */

/* Causal attention of one query row against KV rows 0..p of its sequence
 * ("셀프 어텐션": per-head softmax attention; causal mask and the 1/sqrt(d)
 * scale are the standard decoder reading).  q[d]; K/V rows at stride ld;
 * o[d] receives sum_q softmax_q(q.K_q / sqrt d) V_q.  Softmax subtracts the
 * row max before exponentiating. */
static void attend_row(const double* q, const double* K, const double* V, int64_t ld,
                       int64_t p, int64_t d, double* s, double* o) {
    const double scale = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (int64_t r = 0; r <= p; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c) acc += q[c] * K[r * ld + c];
        s[r] = acc * scale;
        if (s[r] > mx) mx = s[r];
    }
    double sum = 0.0;
    for (int64_t r = 0; r <= p; ++r) { s[r] = exp(s[r] - mx); sum += s[r]; }
    for (int64_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t r = 0; r <= p; ++r) acc += s[r] * V[r * ld + c];
        o[c] = acc / sum;
    }
}

/* Attention core over all heads: Q[M][a d] (head j at columns j d),
 * K, V [M][k d]; O[M][a d].  Sequences never attend across each other.
 * Row strides ldq, ldkv, ldo in elements. */
int tpo_attention_core(int64_t batch, int64_t seq, int64_t a, int64_t k, int64_t d,
                       const double* Q, int64_t ldq, const double* K, const double* V,
                       int64_t ldkv, double* O, int64_t ldo) {
    if (batch < 0 || seq < 0 || a <= 0 || k <= 0 || d <= 0 || a % k) return TPO_ERR_INVALID;
    const int64_t M = batch * seq;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(seq + 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t m = 0; m < M; ++m) {
            const int64_t b = m / seq, p = m % seq;
            for (int64_t j = 0; j < a; ++j) {
                const int64_t g = tpo_q_head_kv(a, k, j);
                attend_row(Q + m * ldq + j * d, K + b * seq * ldkv + g * d,
                           V + b * seq * ldkv + g * d, ldkv, p, d, s, O + m * ldo + j * d);
            }
        }
        free(s);
    }
    return TPO_OK;
}

/* Unsharded attention block: Q = X Wq^T, K = X Wk^T, V = X Wv^T, causal GQA
 * attention per head, out = O Wo^T.  X[M][h], Wq[a d][h], Wk/Wv[k d][h],
 * Wo[h][a d].  O_out (nullable) receives O[M][a d]. */
int tpo_attention(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k, int64_t d,
                  const double* X, const double* Wq, const double* Wk, const double* Wv,
                  const double* Wo, double* O_out, double* out) {
    if (batch < 0 || seq < 0 || h <= 0 || a <= 0 || k <= 0 || d <= 0 || a % k) return TPO_ERR_INVALID;
    const int64_t M = batch * seq, qw = a * d, kw = k * d;
    double* Q = (double*)malloc(sizeof(double) * (size_t)(M * qw + 1));
    double* Kx = (double*)malloc(sizeof(double) * (size_t)(M * kw + 1));
    double* Vx = (double*)malloc(sizeof(double) * (size_t)(M * kw + 1));
    double* O = (double*)malloc(sizeof(double) * (size_t)(M * qw + 1));
    if (!Q || !Kx || !Vx || !O) { free(Q); free(Kx); free(Vx); free(O); return TPO_ERR_NOMEM; }
    tpo_linear(X, h, Wq, h, M, qw, h, Q, qw);
    tpo_linear(X, h, Wk, h, M, kw, h, Kx, kw);
    tpo_linear(X, h, Wv, h, M, kw, h, Vx, kw);
    tpo_attention_core(batch, seq, a, k, d, Q, qw, Kx, Vx, kw, O, qw);
    tpo_linear(O, qw, Wo, qw, M, h, qw, out, h);
    if (O_out) memcpy(O_out, O, sizeof(double) * (size_t)(M * qw));
    free(Q); free(Kx); free(Vx); free(O);
    return TPO_OK;
}

/* Head-sharded attention, the literal t-device form ("셀프 어텐션"):
 * device i takes query heads [i a/t, (i+1) a/t) -- its column block of Wq --
 * and the KV heads those read (its own k/t heads, or a replica of one KV head
 * when k < t), computes attention with no communication, multiplies by its
 * column block of Wo (row-parallel o_proj) and leaves the partial P_i;
 * out = sum_i P_i, i ascending (g).  partials (nullable): [t][M][h]. */
int tpo_attention_sharded(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k,
                          int64_t d, int64_t t, const double* X, const double* Wq,
                          const double* Wk, const double* Wv, const double* Wo,
                          double* partials, double* out) {
    int rc = tpo_plan_check(h, 0, a, k, d, t);
    if (rc) return rc;
    const int64_t M = batch * seq, ap = a / t, kvn = tpo_shard_kv_count(k, t);
    const int64_t qw = ap * d, kw = kvn * d, ad = a * d;
    double* Q = (double*)malloc(sizeof(double) * (size_t)(M * qw + 1));
    double* Kx = (double*)malloc(sizeof(double) * (size_t)(M * kw + 1));
    double* Vx = (double*)malloc(sizeof(double) * (size_t)(M * kw + 1));
    double* O = (double*)malloc(sizeof(double) * (size_t)(M * qw + 1));
    double* P = (double*)malloc(sizeof(double) * (size_t)(t * M * h + 1));
    if (!Q || !Kx || !Vx || !O || !P) {
        free(Q); free(Kx); free(Vx); free(O); free(P);
        return TPO_ERR_NOMEM;
    }
    for (int64_t i = 0; i < t; ++i) {
        const int64_t kv0 = tpo_shard_kv_first(k, t, i);
        tpo_linear(X, h, Wq + i * qw * h, h, M, qw, h, Q, qw);
        tpo_linear(X, h, Wk + kv0 * d * h, h, M, kw, h, Kx, kw);
        tpo_linear(X, h, Wv + kv0 * d * h, h, M, kw, h, Vx, kw);
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)(seq + 1));
#pragma omp for schedule(dynamic, 16)
            for (int64_t m = 0; m < M; ++m) {
                const int64_t b = m / seq, p = m % seq;
                for (int64_t jl = 0; jl < ap; ++jl) {
                    const int64_t j = i * ap + jl;
                    const int64_t gl = tpo_q_head_kv(a, k, j) - kv0; /* local KV slot */
                    attend_row(Q + m * qw + jl * d, Kx + b * seq * kw + gl * d,
                               Vx + b * seq * kw + gl * d, kw, p, d, s, O + m * qw + jl * d);
                }
            }
            free(s);
        }
        /* Row-parallel o_proj: columns [i a d / t, (i+1) a d / t) of Wo. */
        tpo_linear(O, qw, Wo + i * qw, ad, M, h, qw, P + i * M * h, h);
    }
    for (int64_t e = 0; e < M * h; ++e) {
        double s = 0.0;
        for (int64_t i = 0; i < t; ++i) s += P[i * M * h + e];
        out[e] = s;
    }
    if (partials) memcpy(partials, P, sizeof(double) * (size_t)(t * M * h));
    free(Q); free(Kx); free(Vx); free(O); free(P);
    return TPO_OK;
}

/* ---------------------------------------------------------------- g, norm */

/* The g operator's forward on one device's view ("통신 연산 f와 g"): the sum
 * of the t partials, i ascending; a rowwise bias is replicated and added once
 * after the reduction (DTensor section of the transformers page); the
 * replicated residual is added last.  partials[t][n]; bias[h] and residual[n]
 * nullable; n is a multiple of h (rows of h features). */
int tpo_reduce(int64_t t, int64_t n, int64_t h, const double* partials, const double* bias,
               const double* residual, double* out) {
    if (t <= 0 || n < 0 || h <= 0 || (n % h)) return TPO_ERR_INVALID;
    for (int64_t e = 0; e < n; ++e) {
        double s = 0.0;
        for (int64_t i = 0; i < t; ++i) s += partials[i * n + e];
        if (bias) s += bias[e % h];
        if (residual) s += residual[e];
        out[e] = s;
    }
    return TPO_OK;
}

/* RMSNorm with unit gain: y = x / sqrt(mean_j x_j^2 + eps), per row.  The
 * norm is replicated on every device ("통신 연산 f와 g"). */
int tpo_rmsnorm(int64_t M, int64_t h, double eps, const double* x, double* y) {
    if (M < 0 || h <= 0) return TPO_ERR_INVALID;
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t j = 0; j < h; ++j) ss += x[m * h + j] * x[m * h + j];
        const double r = 1.0 / sqrt(ss / (double)h + eps);
        for (int64_t j = 0; j < h; ++j) y[m * h + j] = x[m * h + j] * r;
    }
    return TPO_OK;
}

/* ---------------------------------------------------------------- layer */

/* One pre-norm transformer layer ("통신 연산 f와 g": attention then MLP, one
 * g after each; norm and residual replicated):
 *   h1 = x + Attn(RMSNorm(x)),  y = h1 + MLP_SwiGLU(RMSNorm(h1)).
 * sharded != 0 uses the literal t-device forms of both blocks. */
int tpo_layer(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k, int64_t d,
              int64_t f, int64_t t, int sharded, double eps, const double* X,
              const double* Wq, const double* Wk, const double* Wv, const double* Wo,
              const double* W1, const double* W3, const double* W2, double* Y) {
    int rc = tpo_plan_check(h, f, a, k, d, t);
    if (rc) return rc;
    const int64_t M = batch * seq;
    double* xn = (double*)malloc(sizeof(double) * (size_t)(M * h + 1));
    double* at = (double*)malloc(sizeof(double) * (size_t)(M * h + 1));
    double* h1 = (double*)malloc(sizeof(double) * (size_t)(M * h + 1));
    if (!xn || !at || !h1) { free(xn); free(at); free(h1); return TPO_ERR_NOMEM; }
    tpo_rmsnorm(M, h, eps, X, xn);
    rc = sharded ? tpo_attention_sharded(batch, seq, h, a, k, d, t, xn, Wq, Wk, Wv, Wo, NULL, at)
                 : tpo_attention(batch, seq, h, a, k, d, xn, Wq, Wk, Wv, Wo, NULL, at);
    if (!rc) {
        for (int64_t e = 0; e < M * h; ++e) h1[e] = X[e] + at[e];
        tpo_rmsnorm(M, h, eps, h1, xn);
        rc = sharded ? tpo_mlp_sharded(TPO_ACT_SWIGLU, M, h, f, t, xn, W1, W3, W2, NULL, at)
                     : tpo_mlp(TPO_ACT_SWIGLU, M, h, f, xn, W1, W3, W2, at);
        if (!rc)
            for (int64_t e = 0; e < M * h; ++e) Y[e] = h1[e] + at[e];
    }
    free(xn); free(at); free(h1);
    return rc;
}

/* The same layer evaluated only at chosen tokens.  Causal attention makes
 * token (b, p) depend on tokens (b, 0..p) alone, so this computes the
 * normalised inputs and K/V projections of those positions and then the full
 * definition for each requested token.  rows[] are token indices b*seq+p;
 * Yrows[nrows][h].  With_mlp == 0 stops after h1 (attention block only) and
 * returns h1 - x, i.e. the attention block's output, in Yrows. */
static int layer_rows_impl(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k,
                           int64_t d, int64_t f, double eps, int prenorm, int with_mlp,
                           const double* X, const double* Wq, const double* Wk,
                           const double* Wv, const double* Wo, const double* W1,
                           const double* W3, const double* W2, int64_t nrows,
                           const int64_t* rows, double* Yrows) {
    const int64_t qw = a * d, kw = k * d;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= batch * seq) return TPO_ERR_INVALID;
    double* xn = (double*)malloc(sizeof(double) * (size_t)(seq * h + 1));
    double* Kx = (double*)malloc(sizeof(double) * (size_t)(seq * kw + 1));
    double* Vx = (double*)malloc(sizeof(double) * (size_t)(seq * kw + 1));
    double* q = (double*)malloc(sizeof(double) * (size_t)(qw + 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)(qw + 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(seq + 1));
    double* v = (double*)malloc(sizeof(double) * (size_t)(h + 1));
    double* vn = (double*)malloc(sizeof(double) * (size_t)(h + 1));
    double* u = (double*)malloc(sizeof(double) * (size_t)(f + 1));
    double* gt = (double*)malloc(sizeof(double) * (size_t)(f + 1));
    int rc = TPO_OK;
    if (!xn || !Kx || !Vx || !q || !o || !s || !v || !vn || !u || !gt) { rc = TPO_ERR_NOMEM; goto done; }
    for (int64_t b = 0; b < batch; ++b) {
        int64_t maxp = -1;
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] / seq == b && rows[r] % seq > maxp) maxp = rows[r] % seq;
        if (maxp < 0) continue;
        const double* xb = X + b * seq * h;
        if (prenorm) tpo_rmsnorm(maxp + 1, h, eps, xb, xn);
        else memcpy(xn, xb, sizeof(double) * (size_t)((maxp + 1) * h));
        tpo_linear(xn, h, Wk, h, maxp + 1, kw, h, Kx, kw);
        tpo_linear(xn, h, Wv, h, maxp + 1, kw, h, Vx, kw);
        for (int64_t r = 0; r < nrows; ++r) {
            if (rows[r] / seq != b) continue;
            const int64_t p = rows[r] % seq;
            tpo_linear(xn + p * h, h, Wq, h, 1, qw, h, q, qw);
            for (int64_t j = 0; j < a; ++j) {
                const int64_t g = tpo_q_head_kv(a, k, j);
                attend_row(q + j * d, Kx + g * d, Vx + g * d, kw, p, d, s, o + j * d);
            }
            tpo_linear(o, qw, Wo, qw, 1, h, qw, v, h);      /* attention output */
            double* y = Yrows + r * h;
            if (!with_mlp) { memcpy(y, v, sizeof(double) * (size_t)h); continue; }
            for (int64_t j = 0; j < h; ++j) v[j] += xb[p * h + j];   /* h1 */
            tpo_rmsnorm(1, h, eps, v, vn);
            tpo_linear(vn, h, W1, h, 1, f, h, u, f);
            tpo_linear(vn, h, W3, h, 1, f, h, gt, f);
            for (int64_t j = 0; j < f; ++j) u[j] = tpo_silu(u[j]) * gt[j];
            tpo_linear(u, f, W2, f, 1, h, f, y, h);
            for (int64_t j = 0; j < h; ++j) y[j] += v[j];            /* y = h1 + mlp */
        }
    }
done:
    free(xn); free(Kx); free(Vx); free(q); free(o); free(s); free(v); free(vn); free(u); free(gt);
    return rc;
}

int tpo_layer_rows(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k, int64_t d,
                   int64_t f, double eps, const double* X, const double* Wq, const double* Wk,
                   const double* Wv, const double* Wo, const double* W1, const double* W3,
                   const double* W2, int64_t nrows, const int64_t* rows, double* Yrows) {
    int rc = tpo_plan_check(h, f, a, k, d, 1);
    if (rc) return rc;
    return layer_rows_impl(batch, seq, h, a, k, d, f, eps, 1, 1, X, Wq, Wk, Wv, Wo, W1, W3,
                           W2, nrows, rows, Yrows);
}

/* Attention block (no norm, no residual) at chosen tokens: out = O Wo^T. */
int tpo_attention_rows(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k, int64_t d,
                       const double* X, const double* Wq, const double* Wk, const double* Wv,
                       const double* Wo, int64_t nrows, const int64_t* rows, double* out_rows) {
    if (batch < 0 || seq < 0 || h <= 0 || a <= 0 || k <= 0 || d <= 0 || a % k) return TPO_ERR_INVALID;
    return layer_rows_impl(batch, seq, h, a, k, d, 0, 0.0, 0, 0, X, Wq, Wk, Wv, Wo, NULL, NULL,
                           NULL, nrows, rows, out_rows);
}

/* ---------------------------------------------------------------- packed */

/* Packed projections ("Tensor 병렬성", section "Fused projections"; "추론을
 * 위한 텐서 병렬성", section "패킹 전략"): one Linear whose output rows pack
 * nb logical blocks of sizes n_0..n_{nb-1} (e.g. gate and up of SwiGLU, or
 * Q, K, V, gate, up).  Each block is sharded on its own: device i holds rows
 * [off_b + i n_b / t, off_b + (i+1) n_b / t) of every block b, in block
 * order.  Every block must divide by t ("제약 조건 및 검증": each packed block
 * individually, not only their sum).  rows_out receives the packed-weight
 * row indices device i holds (sum_b n_b / t entries). */
int tpo_packed_shard_rows(const int64_t* blocks, int64_t nb, int64_t t, int64_t i,
                          int64_t* rows_out) {
    if (!blocks || nb <= 0 || t <= 0 || i < 0 || i >= t) return TPO_ERR_INVALID;
    int64_t off = 0, k = 0;
    for (int64_t b = 0; b < nb; ++b) {
        if (blocks[b] <= 0) return TPO_ERR_INVALID;
        if (blocks[b] % t) return TPO_ERR_NOT_DIVISIBLE;
        const int64_t w = blocks[b] / t;
        if (rows_out)
            for (int64_t r = 0; r < w; ++r) rows_out[k + r] = off + i * w + r;
        k += w;
        off += blocks[b];
    }
    return TPO_OK;
}

/* SwiGLU MLP from a packed gate_up weight Wgu[2f][h] (gate rows first, then
 * up rows: blocks [f, f]) and W2[h][f].  per_block != 0: the correct
 * per-block sharding (device i: gate rows [i f/t, (i+1) f/t) and the same
 * up rows, i.e. the strided interleave); per_block == 0: the naive
 * contiguous split of the packed rows ([i 2f/t, (i+1) 2f/t)) followed by
 * chunk(2) of each device's slice into gate and up -- the misplacement the
 * pages warn runs but gives a wrong result.  Z = sum_i
 * (SiLU(X G_i^T) (.) X U_i^T) W2_i^T, with W2_i the columns matching
 * device i's gate rows. */
int tpo_mlp_packed_gate_up(int per_block, int64_t M, int64_t h, int64_t f, int64_t t,
                           const double* X, const double* Wgu, const double* W2, double* Z) {
    if (M < 0 || h <= 0 || f <= 0 || t <= 0 || !X || !Wgu || !W2 || !Z) return TPO_ERR_INVALID;
    if (f % t) return TPO_ERR_NOT_DIVISIBLE;
    const int64_t w = f / t;
    double* G = (double*)malloc(sizeof(double) * (size_t)(M * w + 1));
    double* U = (double*)malloc(sizeof(double) * (size_t)(M * w + 1));
    double* P = (double*)malloc(sizeof(double) * (size_t)(M * h + 1));
    if (!G || !U || !P) { free(G); free(U); free(P); return TPO_ERR_NOMEM; }
    for (int64_t e = 0; e < M * h; ++e) Z[e] = 0.0;
    for (int64_t i = 0; i < t; ++i) {
        const int64_t g0 = per_block ? i * w : i * 2 * w;       /* first gate row */
        const int64_t u0 = per_block ? f + i * w : i * 2 * w + w; /* first up row */
        /* W2 columns matching the gate rows the device holds (for the naive
         * split this is the column block the device would be given). */
        const int64_t c0 = per_block ? i * w : (i * 2 * w) % f;
        tpo_linear(X, h, Wgu + g0 * h, h, M, w, h, G, w);
        tpo_linear(X, h, Wgu + u0 * h, h, M, w, h, U, w);
        for (int64_t e = 0; e < M * w; ++e) G[e] = tpo_silu(G[e]) * U[e];
        tpo_linear(G, w, W2 + c0, f, M, h, w, P, h);
        for (int64_t e = 0; e < M * h; ++e) Z[e] += P[e];
    }
    free(G); free(U); free(P);
    return TPO_OK;
}

/* ---------------------------------------------------------------- vocabulary */

/* Vocab-parallel embedding ("텐서 병렬화", section "임베딩과 출력층": the
 * embedding matrix is split along the vocabulary; "추론을 위한 텐서 병렬성",
 * "분할 전략": EmbeddingParallel(shard_dim=0) looks up each rank's partial
 * and all-reduces them).  E[v][h] (nn.Embedding rows); device i holds rows
 * [i v/t, (i+1) v/t); its partial for token id is E[id] if the id is in its
 * range, else zeros; out = sum of the t partials (i ascending).  An id
 * outside [0, v) is in no device's range, so its row is zero. */
int tpo_embedding_vocab_parallel(int64_t M, int64_t v, int64_t h, int64_t t, const int32_t* ids,
                                 const double* E, double* out) {
    if (M < 0 || v <= 0 || h <= 0 || t <= 0 || !ids || !E || !out) return TPO_ERR_INVALID;
    if (v % t) return TPO_ERR_NOT_DIVISIBLE;
    const int64_t w = v / t;
    for (int64_t e = 0; e < M * h; ++e) out[e] = 0.0;
    for (int64_t i = 0; i < t; ++i)
        for (int64_t m = 0; m < M; ++m) {
            const int64_t id = ids[m];
            if (id < i * w || id >= (i + 1) * w) continue; /* masked: zero partial */
            for (int64_t j = 0; j < h; ++j) out[m * h + j] += E[id * h + j];
        }
    return TPO_OK;
}

/* Cross-entropy of one row of logits, the plain definition:
 * loss = log(sum_j exp(z_j)) - z_label, computed with the max subtracted. */
int tpo_cross_entropy(int64_t M, int64_t v, const double* logits, const int32_t* labels,
                      double* loss) {
    if (M < 0 || v <= 0 || !logits || !labels || !loss) return TPO_ERR_INVALID;
    for (int64_t m = 0; m < M; ++m) {
        const double* z = logits + m * v;
        if (labels[m] == -100) { loss[m] = 0.0; continue; } /* ignored position */
        if (labels[m] < 0 || labels[m] >= v) { loss[m] = NAN; continue; }
        double mx = -INFINITY;
        for (int64_t j = 0; j < v; ++j) if (z[j] > mx) mx = z[j];
        double s = 0.0;
        for (int64_t j = 0; j < v; ++j) s += exp(z[j] - mx);
        loss[m] = log(s) + mx - z[labels[m]];
    }
    return TPO_OK;
}

/* loss_parallel ("텐서 병렬화", "임베딩과 출력층": instead of gathering the
 * b x s x v logits, each device computes the cross-entropy terms from its own
 * partial logits and only the max and the sum are exchanged, so the traffic
 * is b x s).  Device i holds logits columns [i v/t, (i+1) v/t) and computes
 *   m_i = max_j z_j,  s_i = sum_j exp(z_j - m_i),  y_i = z_label if it owns it
 * The exchange: m = max_i m_i,  s = sum_i s_i exp(m_i - m),  y = sum_i y_i,
 * and loss = log(s) + m - y.  stats (nullable) receives [3][t][M]
 * (m_i, s_i, y_i): the only values that cross devices. */
int tpo_cross_entropy_vocab_parallel(int64_t M, int64_t v, int64_t t, const double* logits,
                                     const int32_t* labels, double* stats, double* loss) {
    if (M < 0 || v <= 0 || t <= 0 || !logits || !labels || !loss) return TPO_ERR_INVALID;
    if (v % t) return TPO_ERR_NOT_DIVISIBLE;
    const int64_t w = v / t;
    double* st = (double*)malloc(sizeof(double) * (size_t)(3 * t * M + 1));
    if (!st) return TPO_ERR_NOMEM;
    for (int64_t i = 0; i < t; ++i)
        for (int64_t m = 0; m < M; ++m) {
            const double* z = logits + m * v + i * w;
            double mx = -INFINITY;
            for (int64_t j = 0; j < w; ++j) if (z[j] > mx) mx = z[j];
            double s = 0.0;
            for (int64_t j = 0; j < w; ++j) s += exp(z[j] - mx);
            const int64_t lab = labels[m];
            st[(0 * t + i) * M + m] = mx;
            st[(1 * t + i) * M + m] = s;
            st[(2 * t + i) * M + m] = (lab >= i * w && lab < (i + 1) * w) ? z[lab - i * w] : 0.0;
        }
    for (int64_t m = 0; m < M; ++m) {
        if (labels[m] == -100) { loss[m] = 0.0; continue; }
        if (labels[m] < 0 || labels[m] >= v) { loss[m] = NAN; continue; }
        double mx = -INFINITY;
        for (int64_t i = 0; i < t; ++i) if (st[(0 * t + i) * M + m] > mx) mx = st[(0 * t + i) * M + m];
        double s = 0.0, y = 0.0;
        for (int64_t i = 0; i < t; ++i) {
            s += st[(1 * t + i) * M + m] * exp(st[(0 * t + i) * M + m] - mx);
            y += st[(2 * t + i) * M + m];
        }
        loss[m] = log(s) + mx - y;
    }
    if (stats) memcpy(stats, st, sizeof(double) * (size_t)(3 * t * M));
    free(st);
    return TPO_OK;
}

/* ---------------------------------------------------------------- sequence parallel */

/* Sequence parallelism ("텐서 병렬화", section "시퀀스 병렬화"): the norm
 * and dropout regions are split along the sequence into t pieces, each
 * device keeping its own piece; entering the tensor-parallel region an
 * all-gather collects the sequence, leaving it a reduce-scatter sums the
 * partials and splits them along the sequence again (the same traffic as the
 * all-reduce).  Layout of the sequence-split tensors: [t][batch][s/t][h],
 * device i holding positions [i s/t, (i+1) s/t) of every sequence.
 * Row of token (b, pos) in that layout: */
int64_t tpo_sp_row(int64_t batch, int64_t seq, int64_t t, int64_t b, int64_t pos) {
    const int64_t w = seq / t;
    return ((pos / w) * batch + b) * w + pos % w;
}

/* All-gather: full[b s + pos] = sp[tpo_sp_row(b, pos)]. */
int tpo_sp_all_gather(int64_t batch, int64_t seq, int64_t t, int64_t h, const double* sp,
                      double* full) {
    if (batch < 0 || seq <= 0 || t <= 0 || h <= 0 || (seq % t)) return TPO_ERR_INVALID;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t pos = 0; pos < seq; ++pos)
            memcpy(full + (b * seq + pos) * h, sp + tpo_sp_row(batch, seq, t, b, pos) * h,
                   sizeof(double) * (size_t)h);
    return TPO_OK;
}

/* Reduce-scatter of t partials [t][batch seq][h] (full token order) into the
 * sequence-split layout: device i receives sum_j partials[j] at its own
 * positions (j ascending). */
int tpo_sp_reduce_scatter(int64_t batch, int64_t seq, int64_t t, int64_t h, const double* partials,
                          double* sp) {
    if (batch < 0 || seq <= 0 || t <= 0 || h <= 0 || (seq % t)) return TPO_ERR_INVALID;
    const int64_t M = batch * seq;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t pos = 0; pos < seq; ++pos) {
            double* dst = sp + tpo_sp_row(batch, seq, t, b, pos) * h;
            for (int64_t c = 0; c < h; ++c) {
                double s = 0.0;
                for (int64_t j = 0; j < t; ++j) s += partials[(j * M + b * seq + pos) * h + c];
                dst[c] = s;
            }
        }
    return TPO_OK;
}

/* One pre-norm layer in the sequence-parallel form, step by step: X_sp and
 * Y_sp in the sequence-split layout.
 *   xn_sp = RMSNorm(x_sp) on each device's piece; xn = all-gather(xn_sp)
 *   attention block (head-sharded) -> partials; a_sp = reduce-scatter
 *   h1_sp = x_sp + a_sp; hn_sp = RMSNorm(h1_sp); hn = all-gather(hn_sp)
 *   MLP (sharded SwiGLU) -> partials; m_sp = reduce-scatter; y_sp = h1_sp + m_sp */
int tpo_layer_sp(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k, int64_t d,
                 int64_t f, int64_t t, double eps, const double* X_sp, const double* Wq,
                 const double* Wk, const double* Wv, const double* Wo, const double* W1,
                 const double* W3, const double* W2, double* Y_sp) {
    int rc = tpo_plan_check(h, f, a, k, d, t);
    if (rc) return rc;
    if (seq % t) return TPO_ERR_NOT_DIVISIBLE;
    const int64_t M = batch * seq;
    double* n_sp = (double*)malloc(sizeof(double) * (size_t)(M * h + 1));
    double* full = (double*)malloc(sizeof(double) * (size_t)(M * h + 1));
    double* P = (double*)malloc(sizeof(double) * (size_t)(t * M * h + 1));
    double* h1 = (double*)malloc(sizeof(double) * (size_t)(M * h + 1));
    double* tmp = (double*)malloc(sizeof(double) * (size_t)(M * h + 1));
    if (!n_sp || !full || !P || !h1 || !tmp) { rc = TPO_ERR_NOMEM; goto done; }
    tpo_rmsnorm(M, h, eps, X_sp, n_sp);                      /* row-local: any layout */
    tpo_sp_all_gather(batch, seq, t, h, n_sp, full);
    rc = tpo_attention_sharded(batch, seq, h, a, k, d, t, full, Wq, Wk, Wv, Wo, P, tmp);
    if (rc) goto done;
    tpo_sp_reduce_scatter(batch, seq, t, h, P, tmp);
    for (int64_t e = 0; e < M * h; ++e) h1[e] = X_sp[e] + tmp[e];
    tpo_rmsnorm(M, h, eps, h1, n_sp);
    tpo_sp_all_gather(batch, seq, t, h, n_sp, full);
    rc = tpo_mlp_sharded(TPO_ACT_SWIGLU, M, h, f, t, full, W1, W3, W2, P, tmp);
    if (rc) goto done;
    tpo_sp_reduce_scatter(batch, seq, t, h, P, tmp);
    for (int64_t e = 0; e < M * h; ++e) Y_sp[e] = h1[e] + tmp[e];
done:
    free(n_sp); free(full); free(P); free(h1); free(tmp);
    return rc;
}

/* ---------------------------------------------------------------- backward */

/* d act(u) / du for the MLP activations. */
static double act_grad(int act, double u) {
    if (act == TPO_ACT_GELU_ERF)  /* Phi(u) + u phi(u) */
        return 0.5 * (1.0 + erf(u / sqrt(2.0))) + u * exp(-0.5 * u * u) / sqrt(2.0 * 3.14159265358979323846);
    if (act == TPO_ACT_GELU_TANH) {
        const double c = sqrt(2.0 / 3.14159265358979323846), a = 0.044715;
        const double th = tanh(c * (u + a * u * u * u));
        return 0.5 * (1.0 + th) + 0.5 * u * (1.0 - th * th) * c * (1.0 + 3.0 * a * u * u);
    }
    if (act == TPO_ACT_SWIGLU) {  /* d SiLU / du = s (1 + u (1 - s)), s = sigmoid(u) */
        const double s = 1.0 / (1.0 + exp(-u));
        return s * (1.0 + u * (1.0 - s));
    }
    return 1.0;
}

/* Backward of the MLP at its plain definition, given dZ = dL/dZ:
 *   U = X W1^T, G = X W3^T (SwiGLU), H = act(U) or SiLU(U) (.) G, Z = H W2^T
 *   dH = dZ W2;  dU = dH (.) act'(U)  [SwiGLU: dU = dH (.) G (.) SiLU'(U),
 *   dG = dH (.) SiLU(U)];  dX = dU W1 (+ dG W3);  dW2 = dZ^T H;
 *   dW1 = dU^T X;  dW3 = dG^T X;  and, for a bias b2 added to Z once,
 *   db2 = sum over rows of dZ.
 * dW3 may be NULL unless SwiGLU; db2 may be NULL. */
int tpo_mlp_backward(int act, int64_t M, int64_t h, int64_t f, const double* X, const double* W1,
                     const double* W3, const double* W2, const double* dZ, double* dX, double* dW1,
                     double* dW3, double* dW2, double* db2) {
    if (M <= 0 || h <= 0 || f <= 0 || !X || !W1 || !W2 || !dZ || !dX || !dW1 || !dW2)
        return TPO_ERR_INVALID;
    const int swiglu = act == TPO_ACT_SWIGLU;
    if (swiglu && (!W3 || !dW3)) return TPO_ERR_INVALID;
    double* U = (double*)malloc(sizeof(double) * (size_t)(M * f));
    double* G = (double*)malloc(sizeof(double) * (size_t)(M * f));
    double* H = (double*)malloc(sizeof(double) * (size_t)(M * f));
    double* dH = (double*)malloc(sizeof(double) * (size_t)(M * f));
    double* dU = (double*)malloc(sizeof(double) * (size_t)(M * f));
    double* dG = (double*)malloc(sizeof(double) * (size_t)(M * f));
    int rc = TPO_OK;
    if (!U || !G || !H || !dH || !dU || !dG) { rc = TPO_ERR_NOMEM; goto done; }
    tpo_linear(X, h, W1, h, M, f, h, U, f);
    if (swiglu) tpo_linear(X, h, W3, h, M, f, h, G, f);
    for (int64_t e = 0; e < M * f; ++e) H[e] = swiglu ? tpo_silu(U[e]) * G[e] : act_scalar(act, U[e]);
    if (db2)
        for (int64_t j = 0; j < h; ++j) {
            double s = 0.0;
            for (int64_t m = 0; m < M; ++m) s += dZ[m * h + j];
            db2[j] = s;
        }
    /* dH[m][n] = sum_j dZ[m][j] W2[j][n] */
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < f; ++n) {
            double s = 0.0;
            for (int64_t j = 0; j < h; ++j) s += dZ[m * h + j] * W2[j * f + n];
            dH[m * f + n] = s;
        }
    for (int64_t e = 0; e < M * f; ++e) {
        if (swiglu) {
            dU[e] = dH[e] * G[e] * act_grad(TPO_ACT_SWIGLU, U[e]);
            dG[e] = dH[e] * tpo_silu(U[e]);
        } else {
            dU[e] = dH[e] * act_grad(act, U[e]);
        }
    }
    /* dX[m][j] = sum_n dU[m][n] W1[n][j] (+ dG[m][n] W3[n][j]) */
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < h; ++j) {
            double s = 0.0;
            for (int64_t n = 0; n < f; ++n) {
                s += dU[m * f + n] * W1[n * h + j];
                if (swiglu) s += dG[m * f + n] * W3[n * h + j];
            }
            dX[m * h + j] = s;
        }
    /* dW2[j][n] = sum_m dZ[m][j] H[m][n];  dW1[n][j] = sum_m dU[m][n] X[m][j] */
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < h; ++j)
        for (int64_t n = 0; n < f; ++n) {
            double s = 0.0;
            for (int64_t m = 0; m < M; ++m) s += dZ[m * h + j] * H[m * f + n];
            dW2[j * f + n] = s;
        }
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < f; ++n)
        for (int64_t j = 0; j < h; ++j) {
            double s = 0.0, s3 = 0.0;
            for (int64_t m = 0; m < M; ++m) {
                s += dU[m * f + n] * X[m * h + j];
                if (swiglu) s3 += dG[m * f + n] * X[m * h + j];
            }
            dW1[n * h + j] = s;
            if (swiglu) dW3[n * h + j] = s3;
        }
done:
    free(U); free(G); free(H); free(dH); free(dU); free(dG);
    return rc;
}

/* The same backward in the literal t-device form ("통신 연산 f와 g"): g's
 * backward is the identity, so every device receives the same dZ; device i
 * computes its own slices dW2[:, block i], dW1[block i, :] (and dW3) and a
 * partial dX_i = dU_i W1_i (+ dG_i W3_i); f's backward is the all-reduce
 * dX = sum_i dX_i (i ascending).  dX_partials (nullable): [t][M][h]. */
int tpo_mlp_backward_sharded(int act, int64_t M, int64_t h, int64_t f, int64_t t, const double* X,
                             const double* W1, const double* W3, const double* W2, const double* dZ,
                             double* dX_partials, double* dX, double* dW1, double* dW3, double* dW2,
                             double* db2) {
    if (t <= 0 || f % t) return TPO_ERR_NOT_DIVISIBLE;
    const int64_t w = f / t;
    const int swiglu = act == TPO_ACT_SWIGLU;
    double* W1i = (double*)malloc(sizeof(double) * (size_t)(w * h));
    double* W3i = (double*)malloc(sizeof(double) * (size_t)(w * h));
    double* W2i = (double*)malloc(sizeof(double) * (size_t)(h * w));
    double* dXi = (double*)malloc(sizeof(double) * (size_t)(M * h));
    double* dW1i = (double*)malloc(sizeof(double) * (size_t)(w * h));
    double* dW3i = (double*)malloc(sizeof(double) * (size_t)(w * h));
    double* dW2i = (double*)malloc(sizeof(double) * (size_t)(h * w));
    int rc = TPO_OK;
    if (!W1i || !W3i || !W2i || !dXi || !dW1i || !dW3i || !dW2i) { rc = TPO_ERR_NOMEM; goto done; }
    for (int64_t e = 0; e < M * h; ++e) dX[e] = 0.0;
    for (int64_t i = 0; i < t; ++i) {
        memcpy(W1i, W1 + i * w * h, sizeof(double) * (size_t)(w * h));
        if (swiglu) memcpy(W3i, W3 + i * w * h, sizeof(double) * (size_t)(w * h));
        for (int64_t j = 0; j < h; ++j) memcpy(W2i + j * w, W2 + j * f + i * w, sizeof(double) * (size_t)w);
        /* the bias is added once after g's sum: its gradient is taken once */
        rc = tpo_mlp_backward(act, M, h, w, X, W1i, swiglu ? W3i : NULL, W2i, dZ, dXi, dW1i,
                              swiglu ? dW3i : NULL, dW2i, i == 0 ? db2 : NULL);
        if (rc) goto done;
        for (int64_t e = 0; e < M * h; ++e) dX[e] += dXi[e];
        if (dX_partials) memcpy(dX_partials + i * M * h, dXi, sizeof(double) * (size_t)(M * h));
        memcpy(dW1 + i * w * h, dW1i, sizeof(double) * (size_t)(w * h));
        if (swiglu) memcpy(dW3 + i * w * h, dW3i, sizeof(double) * (size_t)(w * h));
        for (int64_t j = 0; j < h; ++j) memcpy(dW2 + j * f + i * w, dW2i + j * w, sizeof(double) * (size_t)w);
    }
done:
    free(W1i); free(W3i); free(W2i); free(dXi); free(dW1i); free(dW3i); free(dW2i);
    return rc;
}

/* ---------------------------------------------------------------- attention backward */

/* C[M][N] = A[M][K] B[K][N] (plain row-major, no transposes). */
static void matmul_nn(const double* A, const double* B, int64_t M, int64_t K, int64_t N, double* C) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t q = 0; q < K; ++q) s += A[m * K + q] * B[q * N + n];
            C[m * N + n] = s;
        }
}

/* C[M][N] (+)= A[K][M]^T B[K][N]. */
static void matmul_tn(const double* A, const double* B, int64_t K, int64_t M, int64_t N, double* C,
                      int accumulate) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t q = 0; q < K; ++q) s += A[q * M + m] * B[q * N + n];
            C[m * N + n] = accumulate ? C[m * N + n] + s : s;
        }
}

/* Backward of one causal attention row (query p of its sequence), by the
 * chain rule through the row's softmax: with s_r = q.K_r / sqrt d and
 * P = softmax(s) over r <= p, o = sum_r P_r V_r, and the upstream dout:
 *   dP_r = dout . V_r,  D = sum_r P_r dP_r (= dout . o),
 *   dS_r = P_r (dP_r - D),
 *   dq   = sum_r dS_r K_r / sqrt d,   dK_r += dS_r q / sqrt d,
 *   dV_r += P_r dout.
 * dq[d] is written; dK and dV rows (stride ld) are accumulated. */
static void attend_row_backward(const double* q, const double* K, const double* V, int64_t ld,
                                int64_t p, int64_t d, const double* dout, double* P, double* dP,
                                double* dq, double* dK, double* dV) {
    const double scale = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (int64_t r = 0; r <= p; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c) acc += q[c] * K[r * ld + c];
        P[r] = acc * scale;
        if (P[r] > mx) mx = P[r];
    }
    double sum = 0.0;
    for (int64_t r = 0; r <= p; ++r) { P[r] = exp(P[r] - mx); sum += P[r]; }
    double D = 0.0;
    for (int64_t r = 0; r <= p; ++r) {
        P[r] /= sum;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c) acc += dout[c] * V[r * ld + c];
        dP[r] = acc;
        D += P[r] * acc;
    }
    for (int64_t c = 0; c < d; ++c) dq[c] = 0.0;
    for (int64_t r = 0; r <= p; ++r) {
        const double ds = P[r] * (dP[r] - D);
        for (int64_t c = 0; c < d; ++c) {
            dq[c] += ds * K[r * ld + c] * scale;
            dK[r * ld + c] += ds * q[c] * scale;
            dV[r * ld + c] += P[r] * dout[c];
        }
    }
}

/* Backward of the attention core (layout of tpo_attention_core): given
 * dO[M][a d] (stride lddo), writes dQ (stride ldq) and dK, dV (stride ldkv).
 * The gradient of a KV head sums over every query head that reads it (GQA).
 * Parallel over (sequence, KV head): each task owns its dK/dV rows. */
int tpo_attention_core_backward(int64_t batch, int64_t seq, int64_t a, int64_t k, int64_t d,
                                const double* Q, int64_t ldq, const double* K, const double* V,
                                int64_t ldkv, const double* dO, int64_t lddo, double* dQ,
                                double* dK, double* dV) {
    if (batch < 0 || seq < 0 || a <= 0 || k <= 0 || d <= 0 || a % k) return TPO_ERR_INVALID;
    for (int64_t m = 0; m < batch * seq; ++m)
        for (int64_t c = 0; c < k * d; ++c) dK[m * ldkv + c] = dV[m * ldkv + c] = 0.0;
#pragma omp parallel
    {
        double* P = (double*)malloc(sizeof(double) * (size_t)(seq + 1));
        double* dP = (double*)malloc(sizeof(double) * (size_t)(seq + 1));
#pragma omp for schedule(dynamic, 1) collapse(2)
        for (int64_t b = 0; b < batch; ++b)
            for (int64_t g = 0; g < k; ++g) {
                const int64_t r0 = b * seq;
                for (int64_t j = 0; j < a; ++j) {
                    if (tpo_q_head_kv(a, k, j) != g) continue;
                    for (int64_t p = 0; p < seq; ++p)
                        attend_row_backward(Q + (r0 + p) * ldq + j * d, K + r0 * ldkv + g * d,
                                            V + r0 * ldkv + g * d, ldkv, p, d,
                                            dO + (r0 + p) * lddo + j * d, P, dP,
                                            dQ + (r0 + p) * ldq + j * d, dK + r0 * ldkv + g * d,
                                            dV + r0 * ldkv + g * d);
                }
            }
        free(P);
        free(dP);
    }
    return TPO_OK;
}

/* Backward of the unsharded attention block of tpo_attention, given
 * dOut = dL/dout [M][h]:
 *   dO = dOut Wo,  dWo = dOut^T O,  (dQ, dK, dV) = core backward,
 *   dWq = dQ^T X,  dWk = dK^T X,  dWv = dV^T X,
 *   dX = dQ Wq + dK Wk + dV Wv. */
int tpo_attention_backward(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k, int64_t d,
                           const double* X, const double* Wq, const double* Wk, const double* Wv,
                           const double* Wo, const double* dOut, double* dX, double* dWq,
                           double* dWk, double* dWv, double* dWo) {
    if (batch < 0 || seq < 0 || h <= 0 || a <= 0 || k <= 0 || d <= 0 || a % k) return TPO_ERR_INVALID;
    const int64_t M = batch * seq, qw = a * d, kw = k * d;
    double* buf = (double*)malloc(sizeof(double) * (size_t)(4 * M * qw + 4 * M * kw + M * h + 1));
    if (!buf) return TPO_ERR_NOMEM;
    double *Q = buf, *O = Q + M * qw, *dO = O + M * qw, *dQ = dO + M * qw;
    double *Kx = dQ + M * qw, *Vx = Kx + M * kw, *dK = Vx + M * kw, *dV = dK + M * kw;
    double* t1 = dV + M * kw;
    tpo_linear(X, h, Wq, h, M, qw, h, Q, qw);
    tpo_linear(X, h, Wk, h, M, kw, h, Kx, kw);
    tpo_linear(X, h, Wv, h, M, kw, h, Vx, kw);
    tpo_attention_core(batch, seq, a, k, d, Q, qw, Kx, Vx, kw, O, qw);
    matmul_nn(dOut, Wo, M, h, qw, dO);
    matmul_tn(dOut, O, M, h, qw, dWo, 0);
    tpo_attention_core_backward(batch, seq, a, k, d, Q, qw, Kx, Vx, kw, dO, qw, dQ, dK, dV);
    matmul_tn(dQ, X, M, qw, h, dWq, 0);
    matmul_tn(dK, X, M, kw, h, dWk, 0);
    matmul_tn(dV, X, M, kw, h, dWv, 0);
    matmul_nn(dQ, Wq, M, qw, h, dX);
    matmul_nn(dK, Wk, M, kw, h, t1);
    for (int64_t e = 0; e < M * h; ++e) dX[e] += t1[e];
    matmul_nn(dV, Wv, M, kw, h, t1);
    for (int64_t e = 0; e < M * h; ++e) dX[e] += t1[e];
    free(buf);
    return TPO_OK;
}

/* The same backward in the literal t-device form ("통신 연산 f와 g" with
 * the head split of "셀프 어텐션"): device i receives the same dOut (g's
 * backward is the identity), back-propagates through its column block of Wo,
 * its query heads and the KV heads it holds (its own, or a replica), and
 * keeps the gradients of its weight slices; a replicated KV head's weight
 * gradient is the sum over the devices holding it; f's backward is
 * dX = sum_i dX_i (i ascending).  dX_partials (nullable): [t][M][h]. */
int tpo_attention_backward_sharded(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k,
                                   int64_t d, int64_t t, const double* X, const double* Wq,
                                   const double* Wk, const double* Wv, const double* Wo,
                                   const double* dOut, double* dX_partials, double* dX, double* dWq,
                                   double* dWk, double* dWv, double* dWo) {
    int rc = tpo_plan_check(h, 0, a, k, d, t);
    if (rc) return rc;
    const int64_t M = batch * seq, ap = a / t, kvn = tpo_shard_kv_count(k, t);
    const int64_t qw = ap * d, kw = kvn * d, ad = a * d;
    const size_t n = (size_t)(4 * M * qw + 4 * M * kw + 2 * M * h + qw * h + qw * h + 2 * kw * h + 1);
    double* buf = (double*)malloc(sizeof(double) * n);
    if (!buf) return TPO_ERR_NOMEM;
    double *Q = buf, *O = Q + M * qw, *dO = O + M * qw, *dQ = dO + M * qw;
    double *Kx = dQ + M * qw, *Vx = Kx + M * kw, *dK = Vx + M * kw, *dV = dK + M * kw;
    double *dXi = dV + M * kw, *t1 = dXi + M * h;
    double *Woi = t1 + M * h, *dWoi = Woi + qw * h, *dWki = dWoi + qw * h, *dWvi = dWki + kw * h;
    for (int64_t e = 0; e < M * h; ++e) dX[e] = 0.0;
    for (int64_t e = 0; e < k * d * h; ++e) dWk[e] = dWv[e] = 0.0;
    for (int64_t i = 0; i < t; ++i) {
        const int64_t kv0 = tpo_shard_kv_first(k, t, i);
        const double* Wqi = Wq + i * qw * h;
        const double* Wki = Wk + kv0 * d * h;
        const double* Wvi = Wv + kv0 * d * h;
        /* columns [i qw, (i+1) qw) of Wo, as a [h][qw] matrix */
        for (int64_t j = 0; j < h; ++j) memcpy(Woi + j * qw, Wo + j * ad + i * qw, sizeof(double) * (size_t)qw);
        tpo_linear(X, h, Wqi, h, M, qw, h, Q, qw);
        tpo_linear(X, h, Wki, h, M, kw, h, Kx, kw);
        tpo_linear(X, h, Wvi, h, M, kw, h, Vx, kw);
        /* local heads: local query head jl reads local KV slot jl / (ap / kvn) */
        tpo_attention_core(batch, seq, ap, kvn, d, Q, qw, Kx, Vx, kw, O, qw);
        matmul_nn(dOut, Woi, M, h, qw, dO);
        matmul_tn(dOut, O, M, h, qw, dWoi, 0);
        for (int64_t j = 0; j < h; ++j) memcpy(dWo + j * ad + i * qw, dWoi + j * qw, sizeof(double) * (size_t)qw);
        tpo_attention_core_backward(batch, seq, ap, kvn, d, Q, qw, Kx, Vx, kw, dO, qw, dQ, dK, dV);
        matmul_tn(dQ, X, M, qw, h, dWq + i * qw * h, 0);
        matmul_tn(dK, X, M, kw, h, dWki, 0);
        matmul_tn(dV, X, M, kw, h, dWvi, 0);
        for (int64_t e = 0; e < kw * h; ++e) {
            dWk[kv0 * d * h + e] += dWki[e];
            dWv[kv0 * d * h + e] += dWvi[e];
        }
        matmul_nn(dQ, Wqi, M, qw, h, dXi);
        matmul_nn(dK, Wki, M, kw, h, t1);
        for (int64_t e = 0; e < M * h; ++e) dXi[e] += t1[e];
        matmul_nn(dV, Wvi, M, kw, h, t1);
        for (int64_t e = 0; e < M * h; ++e) dXi[e] += t1[e];
        for (int64_t e = 0; e < M * h; ++e) dX[e] += dXi[e];
        if (dX_partials) memcpy(dX_partials + i * M * h, dXi, sizeof(double) * (size_t)(M * h));
    }
    free(buf);
    return TPO_OK;
}

/* ---------------------------------------------------------------- layer backward */

/* Backward of the unit-gain RMSNorm y = x r, r = 1 / sqrt(mean_j x_j^2 + eps),
 * per row, added to out: with g = dL/dy,
 *   dL/dx_i = r g_i - x_i r^3 (sum_j g_j x_j) / h. */
int tpo_rmsnorm_backward(int64_t M, int64_t h, double eps, const double* x, const double* g,
                         double* out) {
    if (M < 0 || h <= 0) return TPO_ERR_INVALID;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const double* xr = x + m * h;
        const double* gr = g + m * h;
        double ss = 0.0, dot = 0.0;
        for (int64_t j = 0; j < h; ++j) {
            ss += xr[j] * xr[j];
            dot += gr[j] * xr[j];
        }
        const double r = 1.0 / sqrt(ss / (double)h + eps);
        for (int64_t j = 0; j < h; ++j) out[m * h + j] += r * gr[j] - xr[j] * r * r * r * dot / (double)h;
    }
    return TPO_OK;
}

/* Backward of the layer of tpo_layer (pre-norm, SwiGLU MLP), given dY:
 *   forward: xn1 = rms(X), h1 = X + Attn(xn1), xn2 = rms(h1), Y = h1 + MLP(xn2)
 *   dh1 = dY + rms'(h1)^T (MLP backward of dY at xn2)
 *   dX  = dh1 + rms'(X)^T (attention backward of dh1 at xn1)
 * with the weight gradients of both blocks.  The blocks' own backward passes
 * are the plain (unsharded) definitions, which the t-device forms equal. */
int tpo_layer_backward(int64_t batch, int64_t seq, int64_t h, int64_t a, int64_t k, int64_t d,
                       int64_t f, double eps, const double* X, const double* Wq, const double* Wk,
                       const double* Wv, const double* Wo, const double* W1, const double* W3,
                       const double* W2, const double* dY, double* dX, double* dWq, double* dWk,
                       double* dWv, double* dWo, double* dW1, double* dW3, double* dW2) {
    if (batch < 0 || seq < 0 || h <= 0 || a <= 0 || k <= 0 || d <= 0 || f <= 0 || a % k) return TPO_ERR_INVALID;
    const int64_t M = batch * seq;
    double* buf = (double*)malloc(sizeof(double) * (size_t)(6 * M * h + 1));
    if (!buf) return TPO_ERR_NOMEM;
    double *xn1 = buf, *h1 = xn1 + M * h, *xn2 = h1 + M * h, *dxn = xn2 + M * h, *dh1 = dxn + M * h;
    double* at = dh1 + M * h;
    int rc;
    tpo_rmsnorm(M, h, eps, X, xn1);
    rc = tpo_attention(batch, seq, h, a, k, d, xn1, Wq, Wk, Wv, Wo, NULL, at);
    if (!rc) {
        for (int64_t e = 0; e < M * h; ++e) h1[e] = X[e] + at[e];
        tpo_rmsnorm(M, h, eps, h1, xn2);
        rc = tpo_mlp_backward(TPO_ACT_SWIGLU, M, h, f, xn2, W1, W3, W2, dY, dxn, dW1, dW3, dW2, NULL);
    }
    if (!rc) {
        memcpy(dh1, dY, sizeof(double) * (size_t)(M * h));
        tpo_rmsnorm_backward(M, h, eps, h1, dxn, dh1);
        rc = tpo_attention_backward(batch, seq, h, a, k, d, xn1, Wq, Wk, Wv, Wo, dh1, dxn, dWq, dWk, dWv, dWo);
    }
    if (!rc) {
        memcpy(dX, dh1, sizeof(double) * (size_t)(M * h));
        tpo_rmsnorm_backward(M, h, eps, X, dxn, dX);
    }
    free(buf);
    return rc;
}
