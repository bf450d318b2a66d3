// tp_api.cu -- the extern "C" entry points of libtp.so: plan creation and
// validation, shard tables, workspace layout, and the composition of the
// kernels into the MLP, attention and layer forwards.
//
// Sources: "Tensor 병렬성" (diffusers docs), sections "Colwise와 rowwise"
// (colwise shards weight dim 0, rowwise weight dim 1, always paired in that
// order so one all-reduce ends the block) and "제약 조건 및 검증"
// (tp_degree must divide the head count; checked before any weight is
// loaded), "한계" (unsupported combinations raise instead of silently
// falling back); "텐서 병렬화" (itwiki), sections "MLP", "셀프 어텐션",
// "통신 연산 f와 g"; "추론을 위한 텐서 병렬성" (transformers docs),
// "DTensor" (rowwise bias replicated and added once after the reduction).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <algorithm>
#include <string>

#include "tp.h"
#include "tp_internal.h"

struct tp_plan_s {
    tp_config cfg;
    int device;
    unsigned* status;  // device status word (256 bytes allocated)
    int64_t M, h, f, a, k, d, t;
    int64_t fw;     // f / t: ffn columns per shard
    int64_t ap;     // a / t: query heads per shard
    int64_t kvn;    // KV heads held per shard
    int64_t qw;     // ap * d
    int64_t kvw;    // kvn * d
    int64_t qkv_w;  // per-shard width of the QKV buffer: qw + 2 kvw
    bool has_mlp, has_attn;
    // tp_mlp_forward in FUSED mode with a GeLU (or no) activation on a
    // problem too small to fill the GPU with two GEMMs: the K pieces of the
    // one-launch MLP (tpi::mlp_fused_launch); 0 = the two-GEMM path.
    int mlp_pieces;
    uint64_t timeout_ns;
};

namespace {

thread_local std::string g_last_error = "no error";

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int fail_str(int code, const std::string& s) {
    g_last_error = s;
    return code;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int need_ptr(const void* p, const char* name) {
    if (!p) return fail(TP_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(p)) return fail(TP_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return TP_OK;
}

int opt_ptr(const void* p, const char* name) {
    if (p && !aligned16(p)) return fail(TP_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return TP_OK;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int check_device(const tp_plan_s* p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return fail(TP_ERR_CUDA, "cudaGetDevice failed");
    if (dev != p->device)
        return fail(TP_ERR_INVALID_ARG, "current device %d is not the plan's device %d", dev,
                    p->device);
    return TP_OK;
}

int64_t kv_first(int64_t k, int64_t t, int64_t i) { return (k >= t) ? i * (k / t) : (i * k) / t; }

// Workspace regions of each op, in bytes, in order.
struct Layout {
    size_t y = 0;        // MLP colwise output [M][f] bf16
    size_t mpart = 0;    // one-launch MLP: [pieces][M][h] fp32 partials (pieces > 1)
    size_t mcnt = 0;     // one-launch MLP: tile counters (zeroed by every call)
    size_t qkv = 0;      // [M][t * qkv_w] bf16
    size_t o = 0;        // [M][a d] bf16
    size_t xn = 0;       // [M][h] bf16 (normalised input of a block)
    size_t h1 = 0;       // [M][h] bf16 (residual stream after attention)
    size_t partials = 0; // [t][M][h] fp32 or bf16 (layer in PARTIALS mode)
    size_t ss = 0;       // 2 x [M] fp32 row sums of squares (layer in FUSED mode)
    size_t full = 0;     // [M][h] bf16 all-gathered block input (sequence parallel)
    size_t ug = 0;       // MLP backward: recomputed pre-activations [M][f or 2f] bf16
    size_t dug = 0;      // MLP backward: dU (| dG) [M][f or 2f] bf16
    size_t hact = 0;     // MLP backward: activations H [M][f] bf16
    size_t bdo = 0;      // attention backward: dO [M][a d] bf16
    size_t bdstat = 0;   // attention backward: D [a][batch][seq_pad] fp32
    size_t bdq = 0;      // attention backward: dQ accumulator [M][a d] fp32
    size_t bdqkv = 0;    // attention backward: dQ | dK | dV [M][(a + 2k) d] bf16
    size_t bqkv = 0;     // attention backward, recomputation: QKV [M][t qkv_w] bf16
    size_t bo = 0;       // attention backward, recomputation: O [M][a d] bf16
    size_t blse = 0;     // attention backward, recomputation: LSE [a][batch][seq_pad] fp32
    // Layer backward: the recomputed forward's saved state, the gradient
    // stream, and one region the block backward passes use in turn.
    size_t lxn1 = 0, lh1 = 0, lxn2 = 0, ldxn = 0, ldh1 = 0;  // [M][h] bf16 each
    size_t lqkv = 0, lo = 0, llse = 0;                       // attention state
    size_t lug = 0;                                          // MLP pre-activations
    size_t lshared = 0;  // max(MLP backward, attention backward workspaces, [M][f] bf16)
    size_t lspx = 0, lspdy = 0, lspdx = 0;  // sequence parallel: X, dY, dX in token order [M][h] bf16
};

int64_t seq_pad_of(const tp_plan_s* p) { return (p->cfg.seq + 63) / 64 * 64; }

size_t layout_total(const Layout& L);

size_t partial_elem_bytes(const tp_plan_s* p) { return p->cfg.partial_dtype == TP_BF16 ? 2 : 4; }

Layout layout_of(const tp_plan_s* p, int op) {
    Layout L;
    const size_t M = static_cast<size_t>(p->M);
    if (op == TP_OP_MLP || op == TP_OP_LAYER) L.y = p->has_mlp ? align_up(M * p->f * 2) : 0;
    if (op == TP_OP_MLP && p->mlp_pieces > 0) {
        if (p->mlp_pieces > 1) L.mpart = align_up(static_cast<size_t>(p->mlp_pieces) * M * p->h * 4);
        L.mcnt = align_up(static_cast<size_t>(tpi::mlp_fused_counter_words(p->M, p->h, p->f)) * 4);
    }
    if (op == TP_OP_ATTN || op == TP_OP_LAYER) {
        if (p->has_attn) {
            L.qkv = align_up(M * p->t * p->qkv_w * 2);
            L.o = align_up(M * p->a * p->d * 2);
        }
    }
    if (op == TP_OP_MLP_BACKWARD && p->has_mlp) {
        const size_t wu = (p->cfg.act == TP_ACT_SWIGLU ? 2 : 1) * static_cast<size_t>(p->f);
        L.ug = align_up(M * wu * 2);
        L.dug = align_up(M * wu * 2);
        L.hact = align_up(M * p->f * 2);
    }
    if (op == TP_OP_ATTN_BACKWARD && p->has_attn) {
        const size_t stat = static_cast<size_t>(p->a) * p->cfg.batch * seq_pad_of(p) * 4;
        L.bdo = align_up(M * p->a * p->d * 2);
        L.bdstat = align_up(stat);
        L.bdq = align_up(M * p->a * p->d * 4);
        L.bdqkv = align_up(M * (p->a + 2 * p->k) * p->d * 2);
        L.bqkv = align_up(M * p->t * p->qkv_w * 2);
        L.bo = align_up(M * p->a * p->d * 2);
        L.blse = align_up(stat);
    }
    if (op == TP_OP_LAYER_BACKWARD && p->has_attn && p->has_mlp) {
        const size_t act = align_up(M * p->h * 2);
        L.lxn1 = L.lh1 = L.lxn2 = L.ldxn = L.ldh1 = act;
        L.lqkv = align_up(M * p->t * p->qkv_w * 2);
        L.lo = align_up(M * p->a * p->d * 2);
        L.llse = align_up(static_cast<size_t>(p->a) * p->cfg.batch * seq_pad_of(p) * 4);
        L.lug = align_up(M * (p->cfg.act == TP_ACT_SWIGLU ? 2 : 1) * static_cast<size_t>(p->f) * 2);
        const size_t mb = layout_total(layout_of(p, TP_OP_MLP_BACKWARD));
        const size_t ab = layout_total(layout_of(p, TP_OP_ATTN_BACKWARD));
        L.lshared = std::max(std::max(mb, ab), align_up(M * p->f * 2));
        if (p->cfg.sequence_parallel) L.lspx = L.lspdy = L.lspdx = act;
    }
    if (op == TP_OP_LAYER) {
        L.h1 = align_up(M * p->h * 2);
        if (p->cfg.reduce_mode == TP_REDUCE_PARTIALS) {
            L.xn = align_up(M * p->h * 2);
            L.partials = align_up(static_cast<size_t>(p->t) * M * p->h * partial_elem_bytes(p));
            if (p->cfg.sequence_parallel) L.full = align_up(M * p->h * 2);
        } else {
            // Folded RMSNorm statistics: x's row sums of squares, then h1's
            // per 128-column slice of the o_proj output.
            L.ss = align_up((1 + (p->h + 127) / 128) * M * sizeof(float));
            // Sequence parallel: the gathered (token-order) copy of x or h1.
            if (p->cfg.sequence_parallel) L.full = align_up(M * p->h * 2);
        }
    }
    return L;
}

size_t layout_total(const Layout& L) {
    return L.y + L.mpart + L.mcnt + L.qkv + L.o + L.xn + L.h1 + L.partials + L.ss + L.full + L.ug + L.dug + L.hact + L.bdo +
           L.bdstat + L.bdq + L.bdqkv + L.bqkv + L.bo + L.blse + L.lxn1 + L.lh1 + L.lxn2 + L.ldxn + L.ldh1 +
           L.lqkv + L.lo + L.llse + L.lug + L.lshared + L.lspx + L.lspdy + L.lspdx;
}

int check_ws(const tp_plan_s* p, int op, void* ws, size_t bytes) {
    const size_t need = layout_total(layout_of(p, op));
    if (need == 0) return TP_OK;
    if (!ws) return fail(TP_ERR_WORKSPACE, "workspace is NULL but %zu bytes are needed", need);
    if (!aligned16(ws)) return fail(TP_ERR_WORKSPACE, "workspace is not 16-byte aligned");
    if (bytes < need)
        return fail(TP_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", bytes, need);
    return TP_OK;
}

int run(int rc, const std::string& err) {
    if (rc != TP_OK) g_last_error = err;
    return rc;
}

// ---- building blocks (arguments already validated) ----

int do_colwise(const tp_plan_s* p, const void* X, const void* W1, const void* W3, void* Y,
               cudaStream_t s, const float* row_ss = nullptr, void* UG = nullptr, int row_ss_parts = 1) {
    tpi::GemmArgs g;
    g.mode = (p->cfg.act == TP_ACT_SWIGLU) ? tpi::GEMM_COL_SWIGLU : tpi::GEMM_COL_ACT;
    g.act = p->cfg.act;
    g.M = p->M;
    g.N = p->f;
    g.A = X;
    g.K = p->h;
    g.t = static_cast<int>(p->t);
    g.B0 = W1;
    g.B0_rows = p->f;
    if (g.mode == tpi::GEMM_COL_SWIGLU) {
        g.B1 = W3;
        g.B1_rows = p->f;
    }
    g.out = Y;
    g.ldo = p->f;
    g.aux_out = UG;  // pre-activations U (| G), saved for the backward pass
    g.ldaux = (p->cfg.act == TP_ACT_SWIGLU ? 2 : 1) * p->f;
    g.n_half = p->f;
    g.row_ss = row_ss;
    g.row_ss_parts = row_ss_parts;
    g.inv_h = 1.0f / static_cast<float>(p->h);
    g.eps = p->cfg.rms_eps;
    g.status = p->status;
    g.timeout_ns = p->timeout_ns;
    std::string err;
    return run(tpi::gemm_launch(g, s, &err), err);
}

// Rowwise GEMM of A [M][t*Ks] by B [N][t*Ks]: fused (sum over shards in the
// accumulator, + bias + residual, bf16 out) or per-shard partials.
int do_rowwise(const tp_plan_s* p, const void* A, int64_t Ks, const void* B, int64_t N,
               const void* bias, const void* residual, void* partials, void* out, bool fused,
               cudaStream_t s, float* ss_out = nullptr, bool sp_rows = false) {
    tpi::GemmArgs g;
    g.mode = fused ? tpi::GEMM_ROW_FUSED : tpi::GEMM_ROW_PARTIAL;
    g.M = p->M;
    g.N = N;
    g.A = A;
    g.t = static_cast<int>(p->t);
    g.Ks = Ks;
    g.B0 = B;
    g.B0_rows = N;
    if (fused) {
        g.out = out;
        g.ldo = N;
        g.bias = bias;
        g.residual = residual;
        g.ldr = N;
        g.ss_out = ss_out;
        if (sp_rows) {  // output and residual in the sequence-split layout
            g.sp_batch = p->cfg.batch;
            g.sp_seq = p->cfg.seq;
            g.sp_t = static_cast<int>(p->t);
        }
    } else {
        g.out = partials;
        g.ldo = N;
        g.out_f32 = p->cfg.partial_dtype == TP_F32 ? 1 : 0;
    }
    g.status = p->status;
    g.timeout_ns = p->timeout_ns;
    std::string err;
    return run(tpi::gemm_launch(g, s, &err), err);
}

int do_reduce(const tp_plan_s* p, const void* partials, const void* bias, const void* residual,
              void* out, int64_t N, cudaStream_t s) {
    std::string err;
    return run(tpi::reduce_launch(partials, p->cfg.partial_dtype == TP_F32 ? 1 : 0,
                                  static_cast<int>(p->t), p->M * N, static_cast<int>(N), bias,
                                  residual, out, s, &err),
               err);
}

int do_qkv(const tp_plan_s* p, const void* X, const void* Wq, const void* Wk, const void* Wv,
           void* QKV, cudaStream_t s, const float* row_ss = nullptr) {
    tpi::GemmArgs g;
    g.mode = tpi::GEMM_COL_QKV;
    g.M = p->M;
    g.N = p->t * p->qkv_w;
    g.A = X;
    g.K = p->h;
    g.t = static_cast<int>(p->t);
    g.B0 = Wq;
    g.B0_rows = p->a * p->d;
    g.B1 = Wk;
    g.B1_rows = p->k * p->d;
    g.B2 = Wv;
    g.B2_rows = p->k * p->d;
    g.qkv_ws = p->qkv_w;
    g.qkv_qw = p->qw;
    g.qkv_kvw = p->kvw;
    g.kv_heads = static_cast<int>(p->k);
    g.head_dim = static_cast<int>(p->d);
    g.out = QKV;
    g.ldo = g.N;
    g.row_ss = row_ss;
    g.inv_h = 1.0f / static_cast<float>(p->h);
    g.eps = p->cfg.rms_eps;
    g.status = p->status;
    g.timeout_ns = p->timeout_ns;
    std::string err;
    return run(tpi::gemm_launch(g, s, &err), err);
}

int do_attn_core(const tp_plan_s* p, const void* QKV, void* O, cudaStream_t s, float* lse = nullptr) {
    tpi::AttnArgs a;
    a.lse = lse;  // base-2 log-sum-exp per (head, sequence, row), for the backward pass
    a.seq_pad = seq_pad_of(p);
    a.QKV = QKV;
    a.ld_qkv = p->t * p->qkv_w;
    a.shard_w = p->qkv_w;
    a.q_w = p->qw;
    a.kv_w = p->kvw;
    a.O = O;
    a.ld_o = p->a * p->d;
    a.batch = p->cfg.batch;
    a.seq = p->cfg.seq;
    a.heads = static_cast<int>(p->a);
    a.kv_heads = static_cast<int>(p->k);
    a.head_dim = static_cast<int>(p->d);
    a.t = static_cast<int>(p->t);
    a.status = p->status;
    a.timeout_ns = p->timeout_ns;
    std::string err;
    return run(tpi::attn_launch(a, s, &err), err);
}

uint8_t* region(void* ws, size_t off) { return static_cast<uint8_t*>(ws) + off; }

// Host-only validation of a configuration and the derived shard geometry
// ("제약 조건 및 검증": every rule is checked before any device work).
int derive_plan(const tp_config& cfg, tp_plan_s* p) {
    const tp_config* pc = &cfg;
    const tp_config c = *pc;
    if (c.tokens < 1) return fail(TP_ERR_INVALID_ARG, "tokens must be >= 1 (got %lld)", (long long)c.tokens);
    if (c.tokens > (int64_t)1 << 30) return fail(TP_ERR_UNSUPPORTED, "tokens above 2^30 are not supported");
    if (c.tp_degree < 1 || c.tp_degree > 64)
        return fail(TP_ERR_INVALID_ARG, "tp_degree must be in [1, 64] (got %d)", c.tp_degree);
    if (c.hidden < 8 || c.hidden % 8)
        return fail(TP_ERR_INVALID_ARG, "hidden must be a positive multiple of 8 (got %d)", c.hidden);
    if (c.ffn < 0 || c.n_heads < 0 || c.n_kv_heads < 0 || c.head_dim < 0)
        return fail(TP_ERR_INVALID_ARG, "sizes must be non-negative");
    if (c.act < TP_ACT_GELU_ERF || c.act > TP_ACT_NONE)
        return fail(TP_ERR_INVALID_ARG, "act %d is not one of TP_ACT_GELU_ERF(0), TP_ACT_GELU_TANH(1), "
                    "TP_ACT_SWIGLU(2), TP_ACT_NONE(3)", c.act);
    if (c.reduce_mode != TP_REDUCE_FUSED && c.reduce_mode != TP_REDUCE_PARTIALS)
        return fail(TP_ERR_INVALID_ARG, "reduce_mode %d is not one of TP_REDUCE_FUSED(0), "
                    "TP_REDUCE_PARTIALS(1)", c.reduce_mode);
    if (c.partial_dtype != TP_F32 && c.partial_dtype != TP_BF16)
        return fail(TP_ERR_INVALID_ARG, "partial_dtype %d is not one of TP_F32(0), TP_BF16(1)",
                    c.partial_dtype);
    if (c.reduce_mode == TP_REDUCE_FUSED && c.partial_dtype != TP_F32)
        return fail(TP_ERR_UNSUPPORTED, "bf16 partials only exist in TP_REDUCE_PARTIALS mode");
    const int64_t t = c.tp_degree;
    // The pages' divisibility rules first, then the kernels' alignment rules.
    if (c.ffn > 0 && c.ffn % t)
        return fail(TP_ERR_NOT_DIVISIBLE, "tp_degree %d does not divide ffn %d", c.tp_degree, c.ffn);
    if (c.n_heads > 0) {
        if (c.n_kv_heads < 1) return fail(TP_ERR_INVALID_ARG, "n_kv_heads must be >= 1 with attention");
        if (c.n_heads % t)
            return fail(TP_ERR_NOT_DIVISIBLE, "tp_degree %d does not divide n_heads %d", c.tp_degree,
                        c.n_heads);
        if (c.n_heads % c.n_kv_heads)
            return fail(TP_ERR_NOT_DIVISIBLE, "n_kv_heads %d does not divide n_heads %d", c.n_kv_heads,
                        c.n_heads);
        if (c.n_kv_heads >= t && c.n_kv_heads % t)
            return fail(TP_ERR_NOT_DIVISIBLE, "tp_degree %d does not divide n_kv_heads %d",
                        c.tp_degree, c.n_kv_heads);
        if (c.n_kv_heads < t && t % c.n_kv_heads)
            return fail(TP_ERR_NOT_DIVISIBLE,
                        "n_kv_heads %d < tp_degree %d must divide it to be replicated evenly",
                        c.n_kv_heads, c.tp_degree);
    }
    if (c.ffn > 0 && (c.ffn / t) % 8)
        return fail(TP_ERR_INVALID_ARG, "ffn / tp_degree = %lld must be a multiple of 8",
                    (long long)(c.ffn / t));
    if (c.n_heads > 0) {
        if (c.head_dim != 64 && c.head_dim != 128)
            return fail(TP_ERR_UNSUPPORTED, "head_dim %d: only 64 and 128 are built", c.head_dim);
        if (c.batch < 1 || c.seq < 1 || (int64_t)c.batch * c.seq != c.tokens)
            return fail(TP_ERR_INVALID_ARG, "tokens %lld must equal batch %d x seq %d",
                        (long long)c.tokens, c.batch, c.seq);
    }
    if (!(c.rms_eps >= 0.0f)) return fail(TP_ERR_INVALID_ARG, "rms_eps must be >= 0");
    if (c.sequence_parallel != 0 && c.sequence_parallel != 1)
        return fail(TP_ERR_INVALID_ARG, "sequence_parallel must be 0 or 1");
    if (c.sequence_parallel) {
        if (c.batch < 1 || c.seq < 1 || (int64_t)c.batch * c.seq != c.tokens)
            return fail(TP_ERR_INVALID_ARG, "sequence parallelism needs tokens == batch x seq");
        if (c.seq % t)
            return fail(TP_ERR_NOT_DIVISIBLE, "tp_degree %d does not divide seq %d (sequence split)",
                        c.tp_degree, c.seq);
    }

    *p = tp_plan_s();
    p->cfg = c;
    p->device = -1;
    p->status = nullptr;
    p->M = c.tokens;
    p->h = c.hidden;
    p->f = c.ffn;
    p->a = c.n_heads;
    p->k = c.n_kv_heads;
    p->d = c.head_dim;
    p->t = t;
    p->has_mlp = c.ffn > 0;
    p->has_attn = c.n_heads > 0;
    p->fw = p->has_mlp ? p->f / t : 0;
    if (p->has_attn) {
        p->ap = p->a / t;
        p->kvn = (p->k >= t) ? p->k / t : 1;
        p->qw = p->ap * p->d;
        p->kvw = p->kvn * p->d;
        p->qkv_w = p->qw + 2 * p->kvw;
    }
    p->timeout_ns = 2000000000ull;  // 2 s per barrier wait
    p->mlp_pieces = 0;
    return TP_OK;
}


}  // namespace

extern "C" {

const char* tp_last_error(void) { return g_last_error.c_str(); }

int tp_config_check(const tp_config* cfg) {
    if (!cfg) return fail(TP_ERR_INVALID_ARG, "cfg is NULL");
    tp_plan_s tmp;
    return derive_plan(*cfg, &tmp);
}

int tp_plan_create(const tp_config* cfg, tp_plan_t* out) {
    if (out) *out = nullptr;
    if (!cfg || !out) return fail(TP_ERR_INVALID_ARG, "cfg and out must be non-NULL");
    tp_plan_s tmp;
    int rc = derive_plan(*cfg, &tmp);
    if (rc) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(TP_ERR_CUDA, "no CUDA device");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return fail(TP_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                    dev, major, minor);
    tp_plan_s* p = new (std::nothrow) tp_plan_s(tmp);
    if (!p) return fail(TP_ERR_CUDA, "out of host memory");
    p->device = dev;
    if (p->has_mlp && p->cfg.reduce_mode == TP_REDUCE_FUSED)
        p->mlp_pieces = tpi::mlp_fused_pieces(p->M, p->h, p->f, static_cast<int>(p->t), p->cfg.act);
    cudaError_t e = cudaMalloc(&p->status, 256);
    if (e == cudaSuccess) e = cudaMemset(p->status, 0, 256);
    if (e != cudaSuccess) {
        delete p;
        return fail(TP_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
    }
    *out = p;
    return TP_OK;
}

int tp_plan_destroy(tp_plan_t plan) {
    if (!plan) return TP_OK;
    if (plan->status) cudaFree(plan->status);
    delete plan;
    return TP_OK;
}

int tp_plan_workspace_bytes(tp_plan_t plan, int op, size_t* bytes) {
    if (!plan || !bytes) return fail(TP_ERR_INVALID_ARG, "plan and bytes must be non-NULL");
    if (op < TP_OP_MLP || op > TP_OP_LAYER_BACKWARD) return fail(TP_ERR_INVALID_ARG, "unknown op %d", op);
    *bytes = layout_total(layout_of(plan, op));
    return TP_OK;
}

int tp_plan_shard_table(tp_plan_t plan, int which, int32_t* out, int64_t cap, int64_t* n) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    return tp_config_shard_table(&plan->cfg, which, out, cap, n);
}

int tp_config_shard_table(const tp_config* cfg, int which, int32_t* out, int64_t cap, int64_t* n) {
    if (!cfg || !n) return fail(TP_ERR_INVALID_ARG, "cfg and n must be non-NULL");
    tp_plan_s tmp;
    int rc = derive_plan(*cfg, &tmp);
    if (rc) return rc;
    const tp_plan_s* p = &tmp;
    int64_t cnt = 0;
    switch (which) {
        case TP_TABLE_FFN_SHARDS: cnt = 2 * p->t; break;
        case TP_TABLE_Q_HEAD_SHARD:
        case TP_TABLE_Q_HEAD_KV: cnt = p->a; break;
        case TP_TABLE_SHARD_KV: cnt = p->has_attn ? 2 * p->t : 0; break;
        case TP_TABLE_QKV_COLUMNS: cnt = p->has_attn ? 3 * p->t : 0; break;
        default: return fail(TP_ERR_INVALID_ARG, "unknown table %d", which);
    }
    *n = cnt;
    if (cnt > cap || (cnt > 0 && !out))
        return fail(TP_ERR_INVALID_ARG, "table needs %lld entries, capacity %lld", (long long)cnt,
                    (long long)cap);
    for (int64_t i = 0; i < cnt; ++i) {
        int64_t v = 0;
        switch (which) {
            case TP_TABLE_FFN_SHARDS: v = (i & 1) ? p->fw : (i >> 1) * p->fw; break;
            case TP_TABLE_Q_HEAD_SHARD: v = i / p->ap; break;
            case TP_TABLE_Q_HEAD_KV: v = i / (p->a / p->k); break;
            case TP_TABLE_SHARD_KV: v = (i & 1) ? p->kvn : kv_first(p->k, p->t, i >> 1); break;
            case TP_TABLE_QKV_COLUMNS: {
                const int64_t s = i / 3, part = i % 3;
                v = s * p->qkv_w + (part == 0 ? 0 : part == 1 ? p->qw : p->qw + p->kvw);
                break;
            }
        }
        out[i] = static_cast<int32_t>(v);
    }
    return TP_OK;
}

int tp_get_device_status(tp_plan_t plan, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    unsigned word = 0;
    cudaStream_t s = as_stream(stream);
    cudaError_t e = cudaMemcpyAsync(&word, plan->status, sizeof(word), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(TP_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (word) {
        cudaMemsetAsync(plan->status, 0, sizeof(unsigned), s);
        cudaStreamSynchronize(s);
        if (word & 1u)
            return fail(TP_ERR_DEVICE_TIMEOUT, "a device-side wait exceeded its limit (status 0x%x)", word);
        return fail(TP_ERR_CUDA, "a kernel found its shared-memory layout does not fit (status 0x%x)",
                    word);
    }
    return TP_OK;
}

int tp_reduce_partials(const void* partials, int partial_dtype, int32_t t, int64_t n, int32_t h,
                       const tp_bf16* bias, const tp_bf16* residual, tp_bf16* out, void* stream) {
    int rc;
    if ((rc = need_ptr(partials, "partials")) || (rc = need_ptr(out, "out")) ||
        (rc = opt_ptr(bias, "bias")) || (rc = opt_ptr(residual, "residual")))
        return rc;
    if (partial_dtype != TP_F32 && partial_dtype != TP_BF16)
        return fail(TP_ERR_INVALID_ARG, "partial_dtype %d is not TP_F32(0) or TP_BF16(1)", partial_dtype);
    if (t < 1 || t > 64) return fail(TP_ERR_INVALID_ARG, "t must be in [1, 64]");
    if (h < 8 || h % 8) return fail(TP_ERR_INVALID_ARG, "h must be a positive multiple of 8");
    if (n < 0 || n % h) return fail(TP_ERR_INVALID_ARG, "n must be a non-negative multiple of h");
    std::string err;
    return run(tpi::reduce_launch(partials, partial_dtype == TP_F32 ? 1 : 0, t, n, h, bias, residual,
                                  out, as_stream(stream), &err),
               err);
}

int tp_rmsnorm(const tp_bf16* x, int64_t rows, int32_t h, float eps, tp_bf16* y, void* stream) {
    int rc;
    if ((rc = need_ptr(x, "x")) || (rc = need_ptr(y, "y"))) return rc;
    if (rows < 0 || rows > (int64_t)1 << 30) return fail(TP_ERR_INVALID_ARG, "rows out of range");
    if (h < 8 || h % 8 || h > 8192) return fail(TP_ERR_INVALID_ARG, "h must be a multiple of 8 in [8, 8192]");
    if (!(eps >= 0.0f)) return fail(TP_ERR_INVALID_ARG, "eps must be >= 0");
    std::string err;
    return run(tpi::rmsnorm_launch(x, rows, h, eps, y, as_stream(stream), &err), err);
}

int tp_colwise_forward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1, const tp_bf16* W3,
                       tp_bf16* Y, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_mlp) return fail(TP_ERR_INVALID_ARG, "the plan has no MLP (ffn == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(W1, "W1")) ||
        (rc = need_ptr(Y, "Y")))
        return rc;
    if (plan->cfg.act == TP_ACT_SWIGLU) {
        if ((rc = need_ptr(W3, "W3 (SwiGLU)"))) return rc;
    } else if (W3) {
        return fail(TP_ERR_INVALID_ARG, "W3 must be NULL unless act is TP_ACT_SWIGLU");
    }
    return do_colwise(plan, X, W1, W3, Y, as_stream(stream));
}

int tp_rowwise_forward(tp_plan_t plan, const tp_bf16* Y, const tp_bf16* W2, const tp_bf16* bias,
                       const tp_bf16* residual, void* partials, tp_bf16* Z, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_mlp) return fail(TP_ERR_INVALID_ARG, "the plan has no MLP (ffn == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(Y, "Y")) || (rc = need_ptr(W2, "W2"))) return rc;
    const bool fused = plan->cfg.reduce_mode == TP_REDUCE_FUSED;
    if (fused) {
        if ((rc = need_ptr(Z, "Z")) || (rc = opt_ptr(bias, "bias")) || (rc = opt_ptr(residual, "residual")))
            return rc;
    } else if ((rc = need_ptr(partials, "partials"))) {
        return rc;
    }
    return do_rowwise(plan, Y, plan->fw, W2, plan->h, bias, residual, partials, Z, fused,
                      as_stream(stream));
}

namespace {

int mlp_forward_impl(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1, const tp_bf16* W3,
                     const tp_bf16* W2, const tp_bf16* b2, const tp_bf16* residual, void* partials,
                     tp_bf16* Z, tp_bf16* UG, void* workspace, size_t ws_bytes, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_mlp) return fail(TP_ERR_INVALID_ARG, "the plan has no MLP (ffn == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(W1, "W1")) ||
        (rc = need_ptr(W2, "W2")) || (rc = need_ptr(Z, "Z")) || (rc = opt_ptr(b2, "b2")) ||
        (rc = opt_ptr(residual, "residual")) || (rc = opt_ptr(UG, "UG")))
        return rc;
    if (plan->cfg.act == TP_ACT_SWIGLU) {
        if ((rc = need_ptr(W3, "W3 (SwiGLU)"))) return rc;
    } else if (W3) {
        return fail(TP_ERR_INVALID_ARG, "W3 must be NULL unless act is TP_ACT_SWIGLU");
    }
    const bool fused = plan->cfg.reduce_mode == TP_REDUCE_FUSED;
    if (!fused && (rc = need_ptr(partials, "partials"))) return rc;
    if ((rc = check_ws(plan, TP_OP_MLP, workspace, ws_bytes))) return rc;
    cudaStream_t s = as_stream(stream);
    void* Y = workspace;
    if (fused && !UG && plan->mlp_pieces > 0) {
        // One launch: colwise tiles, then each m-block's rowwise tiles as
        // soon as their H columns are stored ("MLP": Z = sum_i GeLU(X A_i) B_i).
        const Layout L = layout_of(plan, TP_OP_MLP);
        uint8_t* w = static_cast<uint8_t*>(workspace);
        tpi::MlpArgs m;
        m.act = plan->cfg.act;
        m.M = plan->M;
        m.h = plan->h;
        m.f = plan->f;
        m.t = static_cast<int>(plan->t);
        m.pieces = plan->mlp_pieces;
        m.X = X;
        m.W1 = W1;
        m.W2 = W2;
        m.bias = b2;
        m.residual = residual;
        m.Z = Z;
        m.H = w;
        m.partials = L.mpart ? reinterpret_cast<float*>(w + L.y) : nullptr;
        m.counters = reinterpret_cast<unsigned*>(w + L.y + L.mpart);
        m.status = plan->status;
        m.timeout_ns = plan->timeout_ns;
        cudaError_t e = cudaMemsetAsync(m.counters, 0, L.mcnt, s);
        if (e != cudaSuccess) return fail(TP_ERR_CUDA, "counter reset: %s", cudaGetErrorString(e));
        std::string err;
        return run(tpi::mlp_fused_launch(m, s, &err), err);
    }
    if ((rc = do_colwise(plan, X, W1, W3, Y, s, nullptr, UG))) return rc;
    if ((rc = do_rowwise(plan, Y, plan->fw, W2, plan->h, b2, residual, partials, Z, fused, s))) return rc;
    if (!fused) return do_reduce(plan, partials, b2, residual, Z, plan->h, s);
    return TP_OK;
}

}  // namespace

int tp_mlp_forward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1, const tp_bf16* W3,
                   const tp_bf16* W2, const tp_bf16* b2, const tp_bf16* residual, void* partials,
                   tp_bf16* Z, void* workspace, size_t ws_bytes, void* stream) {
    return mlp_forward_impl(plan, X, W1, W3, W2, b2, residual, partials, Z, nullptr, workspace,
                            ws_bytes, stream);
}

int tp_mlp_forward_train(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1, const tp_bf16* W3,
                         const tp_bf16* W2, const tp_bf16* b2, const tp_bf16* residual,
                         void* partials, tp_bf16* Z, tp_bf16* UG, void* workspace, size_t ws_bytes,
                         void* stream) {
    if (!UG) return fail(TP_ERR_INVALID_ARG, "UG is NULL");
    return mlp_forward_impl(plan, X, W1, W3, W2, b2, residual, partials, Z, UG, workspace,
                            ws_bytes, stream);
}

int tp_mlp_backward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1, const tp_bf16* W3,
                    const tp_bf16* W2, const tp_bf16* dZ, const tp_bf16* UG, tp_bf16* dX,
                    float* dW1, float* dW3, float* dW2, float* db2, int accumulate, void* workspace,
                    size_t ws_bytes, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_mlp) return fail(TP_ERR_INVALID_ARG, "the plan has no MLP (ffn == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(W1, "W1")) ||
        (rc = need_ptr(W2, "W2")) || (rc = need_ptr(dZ, "dZ")) || (rc = opt_ptr(UG, "UG")) ||
        (rc = need_ptr(dX, "dX")) || (rc = need_ptr(dW1, "dW1")) || (rc = need_ptr(dW2, "dW2")) ||
        (rc = opt_ptr(db2, "db2")))
        return rc;
    const bool glu = plan->cfg.act == TP_ACT_SWIGLU;
    if (glu) {
        if ((rc = need_ptr(W3, "W3 (SwiGLU)")) || (rc = need_ptr(dW3, "dW3 (SwiGLU)"))) return rc;
        if (plan->f % 64 != 0)
            return fail(TP_ERR_UNSUPPORTED, "the SwiGLU backward needs ffn %% 64 == 0 (ffn = %lld)",
                        static_cast<long long>(plan->f));
    } else if (W3 || dW3) {
        return fail(TP_ERR_INVALID_ARG, "W3 and dW3 must be NULL unless act is TP_ACT_SWIGLU");
    }
    if ((rc = check_ws(plan, TP_OP_MLP_BACKWARD, workspace, ws_bytes))) return rc;
    const Layout L = layout_of(plan, TP_OP_MLP_BACKWARD);
    void* ug_ws = region(workspace, 0);
    void* dug = region(workspace, L.ug);
    void* hact = region(workspace, L.ug + L.dug);
    cudaStream_t s = as_stream(stream);
    const int64_t M = plan->M, h = plan->h, f = plan->f, wu = (glu ? 2 : 1) * f;
    std::string err;
    // Pre-activations: the caller's, or recomputed together with H.
    const void* ug = UG;
    if (!UG) {
        if ((rc = do_colwise(plan, X, W1, W3, hact, s, nullptr, ug_ws))) return rc;
        ug = ug_ws;
    }
    {  // dH = dZ W2 (g backward: the same dZ for every shard), then dU (| dG), H.
        tpi::GemmArgs g;
        g.mode = tpi::GEMM_BWD_ACT;
        g.act = plan->cfg.act;
        g.M = M;
        g.N = f;
        g.K = h;
        g.A = dZ;
        g.B0 = W2;
        g.aux = ug;
        g.ldaux = wu;
        g.n_half = f;
        g.out = dug;
        g.ldo = wu;
        g.out2 = UG ? hact : nullptr;  // recomputation already wrote H
        g.ldo2 = f;
        g.status = plan->status;
        g.timeout_ns = plan->timeout_ns;
        if ((rc = run(tpi::gemm_launch(g, s, &err), err))) return rc;
    }
    {  // dX = [dU | dG] [W1 ; W3]: f's all-reduce as the K loop over all shards.
        tpi::GemmArgs g;
        g.mode = tpi::GEMM_NN;
        g.M = M;
        g.N = h;
        g.K = wu;
        g.A = dug;
        g.B0 = W1;
        g.B1 = glu ? W3 : nullptr;
        g.k_split = f;
        g.out = dX;
        g.ldo = h;
        g.status = plan->status;
        g.timeout_ns = plan->timeout_ns;
        if ((rc = run(tpi::gemm_launch(g, s, &err), err))) return rc;
    }
    {  // dW2 = dZ^T H (shard i: columns i f/t .. of dW2).
        tpi::GemmArgs g;
        g.mode = tpi::GEMM_TN;
        g.M = h;
        g.N = f;
        g.K = M;
        g.A = dZ;
        g.lda = h;
        g.B0 = hact;
        g.out = dW2;
        g.ldo = f;
        g.accumulate = accumulate ? 1 : 0;
        g.status = plan->status;
        g.timeout_ns = plan->timeout_ns;
        if ((rc = run(tpi::gemm_launch(g, s, &err), err))) return rc;
    }
    {  // [dW1 ; dW3] = [dU | dG]^T X (shard i: rows i f/t .. of each).
        tpi::GemmArgs g;
        g.mode = tpi::GEMM_TN;
        g.M = wu;
        g.N = h;
        g.K = M;
        g.A = dug;
        g.lda = wu;
        g.B0 = X;
        g.out = dW1;
        g.ldo = h;
        g.out2 = glu ? dW3 : nullptr;
        g.ldo2 = h;
        g.row_split = f;
        g.accumulate = accumulate ? 1 : 0;
        g.status = plan->status;
        g.timeout_ns = plan->timeout_ns;
        if ((rc = run(tpi::gemm_launch(g, s, &err), err))) return rc;
    }
    if (db2) return run(tpi::colsum_launch(dZ, M, static_cast<int>(h), db2, accumulate, s, &err), err);
    return TP_OK;
}

int tp_qkv_forward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* Wq, const tp_bf16* Wk,
                   const tp_bf16* Wv, tp_bf16* QKV, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_attn) return fail(TP_ERR_INVALID_ARG, "the plan has no attention (n_heads == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(Wq, "Wq")) ||
        (rc = need_ptr(Wk, "Wk")) || (rc = need_ptr(Wv, "Wv")) || (rc = need_ptr(QKV, "QKV")))
        return rc;
    return do_qkv(plan, X, Wq, Wk, Wv, QKV, as_stream(stream));
}

int tp_attn_core_forward(tp_plan_t plan, const tp_bf16* QKV, tp_bf16* O, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_attn) return fail(TP_ERR_INVALID_ARG, "the plan has no attention (n_heads == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(QKV, "QKV")) || (rc = need_ptr(O, "O"))) return rc;
    return do_attn_core(plan, QKV, O, as_stream(stream));
}

int tp_attn_forward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* Wq, const tp_bf16* Wk,
                    const tp_bf16* Wv, const tp_bf16* Wo, const tp_bf16* residual, void* partials,
                    tp_bf16* out, void* workspace, size_t ws_bytes, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_attn) return fail(TP_ERR_INVALID_ARG, "the plan has no attention (n_heads == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(Wq, "Wq")) ||
        (rc = need_ptr(Wk, "Wk")) || (rc = need_ptr(Wv, "Wv")) || (rc = need_ptr(Wo, "Wo")) ||
        (rc = need_ptr(out, "out")) || (rc = opt_ptr(residual, "residual")))
        return rc;
    const bool fused = plan->cfg.reduce_mode == TP_REDUCE_FUSED;
    if (!fused && (rc = need_ptr(partials, "partials"))) return rc;
    if ((rc = check_ws(plan, TP_OP_ATTN, workspace, ws_bytes))) return rc;
    const Layout L = layout_of(plan, TP_OP_ATTN);
    void* QKV = region(workspace, 0);
    void* O = region(workspace, L.qkv);
    cudaStream_t s = as_stream(stream);
    if ((rc = do_qkv(plan, X, Wq, Wk, Wv, QKV, s))) return rc;
    if ((rc = do_attn_core(plan, QKV, O, s))) return rc;
    if ((rc = do_rowwise(plan, O, plan->qw, Wo, plan->h, nullptr, residual, partials, out, fused, s)))
        return rc;
    if (!fused) return do_reduce(plan, partials, nullptr, residual, out, plan->h, s);
    return TP_OK;
}

int tp_plan_attn_saved_bytes(tp_plan_t plan, size_t* qkv_bytes, size_t* o_bytes, size_t* lse_bytes) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_attn) return fail(TP_ERR_INVALID_ARG, "the plan has no attention (n_heads == 0)");
    const size_t M = static_cast<size_t>(plan->M);
    if (qkv_bytes) *qkv_bytes = M * plan->t * plan->qkv_w * 2;
    if (o_bytes) *o_bytes = M * plan->a * plan->d * 2;
    if (lse_bytes) *lse_bytes = static_cast<size_t>(plan->a) * plan->cfg.batch * seq_pad_of(plan) * 4;
    return TP_OK;
}

int tp_attn_forward_train(tp_plan_t plan, const tp_bf16* X, const tp_bf16* Wq, const tp_bf16* Wk,
                          const tp_bf16* Wv, const tp_bf16* Wo, const tp_bf16* residual, void* partials,
                          tp_bf16* out, tp_bf16* QKV, tp_bf16* O, float* LSE, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_attn) return fail(TP_ERR_INVALID_ARG, "the plan has no attention (n_heads == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(Wq, "Wq")) ||
        (rc = need_ptr(Wk, "Wk")) || (rc = need_ptr(Wv, "Wv")) || (rc = need_ptr(Wo, "Wo")) ||
        (rc = need_ptr(out, "out")) || (rc = opt_ptr(residual, "residual")) || (rc = need_ptr(QKV, "QKV")) ||
        (rc = need_ptr(O, "O")) || (rc = need_ptr(LSE, "LSE")))
        return rc;
    const bool fused = plan->cfg.reduce_mode == TP_REDUCE_FUSED;
    if (!fused && (rc = need_ptr(partials, "partials"))) return rc;
    cudaStream_t s = as_stream(stream);
    if ((rc = do_qkv(plan, X, Wq, Wk, Wv, QKV, s))) return rc;
    if ((rc = do_attn_core(plan, QKV, O, s, LSE))) return rc;
    if ((rc = do_rowwise(plan, O, plan->qw, Wo, plan->h, nullptr, residual, partials, out, fused, s)))
        return rc;
    if (!fused) return do_reduce(plan, partials, nullptr, residual, out, plan->h, s);
    return TP_OK;
}

int tp_attn_backward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* Wq, const tp_bf16* Wk,
                     const tp_bf16* Wv, const tp_bf16* Wo, const tp_bf16* dOut, const tp_bf16* QKV,
                     const tp_bf16* O, const float* LSE, tp_bf16* dX, float* dWq, float* dWk, float* dWv,
                     float* dWo, int accumulate, void* workspace, size_t ws_bytes, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_attn) return fail(TP_ERR_INVALID_ARG, "the plan has no attention (n_heads == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(Wq, "Wq")) ||
        (rc = need_ptr(Wk, "Wk")) || (rc = need_ptr(Wv, "Wv")) || (rc = need_ptr(Wo, "Wo")) ||
        (rc = need_ptr(dOut, "dOut")) || (rc = opt_ptr(QKV, "QKV")) || (rc = opt_ptr(O, "O")) ||
        (rc = opt_ptr(LSE, "LSE")) || (rc = need_ptr(dX, "dX")) || (rc = need_ptr(dWq, "dWq")) ||
        (rc = need_ptr(dWk, "dWk")) || (rc = need_ptr(dWv, "dWv")) || (rc = need_ptr(dWo, "dWo")))
        return rc;
    const bool saved = QKV != nullptr;
    if (saved != (O != nullptr) || saved != (LSE != nullptr))
        return fail(TP_ERR_INVALID_ARG, "QKV, O and LSE must be all saved or all NULL");
    if ((rc = check_ws(plan, TP_OP_ATTN_BACKWARD, workspace, ws_bytes))) return rc;
    const Layout L = layout_of(plan, TP_OP_ATTN_BACKWARD);
    size_t off = 0;
    void* w_do = region(workspace, off);
    off += L.bdo;
    float* w_dstat = reinterpret_cast<float*>(region(workspace, off));
    off += L.bdstat;
    float* w_dq = reinterpret_cast<float*>(region(workspace, off));
    off += L.bdq;
    void* w_dqkv = region(workspace, off);
    off += L.bdqkv;
    void* w_qkv = region(workspace, off);
    off += L.bqkv;
    void* w_o = region(workspace, off);
    off += L.bo;
    float* w_lse = reinterpret_cast<float*>(region(workspace, off));
    cudaStream_t s = as_stream(stream);
    const int64_t M = plan->M, h = plan->h, ad = plan->a * plan->d, kd = plan->k * plan->d;
    const int64_t wd = ad + 2 * kd;  // dQ | dK | dV columns
    std::string err;
    const void* qkv = QKV;
    const void* o = O;
    const float* lse = LSE;
    if (!saved) {  // recompute what the forward would have saved
        if ((rc = do_qkv(plan, X, Wq, Wk, Wv, w_qkv, s))) return rc;
        if ((rc = do_attn_core(plan, w_qkv, w_o, s, w_lse))) return rc;
        qkv = w_qkv;
        o = w_o;
        lse = w_lse;
    }
    {  // dO = dOut Wo (g's backward: the same dOut for every shard)
        tpi::GemmArgs g;
        g.mode = tpi::GEMM_NN;
        g.M = M;
        g.N = ad;
        g.K = h;
        g.A = dOut;
        g.B0 = Wo;
        g.out = w_do;
        g.ldo = ad;
        g.status = plan->status;
        g.timeout_ns = plan->timeout_ns;
        if ((rc = run(tpi::gemm_launch(g, s, &err), err))) return rc;
    }
    {  // dWo = dOut^T O (shard i: columns of its heads)
        tpi::GemmArgs g;
        g.mode = tpi::GEMM_TN;
        g.M = h;
        g.N = ad;
        g.K = M;
        g.A = dOut;
        g.lda = h;
        g.B0 = o;
        g.out = dWo;
        g.ldo = ad;
        g.accumulate = accumulate ? 1 : 0;
        g.status = plan->status;
        g.timeout_ns = plan->timeout_ns;
        if ((rc = run(tpi::gemm_launch(g, s, &err), err))) return rc;
    }
    {  // attention core backward: dQ | dK | dV, KV gradients summed over each group
        tpi::AttnBwdArgs a;
        a.QKV = qkv;
        a.ld_qkv = plan->t * plan->qkv_w;
        a.shard_w = plan->qkv_w;
        a.q_w = plan->qw;
        a.kv_w = plan->kvw;
        a.dO = w_do;
        a.O = o;
        a.ld_do = ad;
        a.lse = lse;
        a.dstat = w_dstat;
        a.seq_pad = seq_pad_of(plan);
        a.dq = w_dq;
        a.ld_dq = ad;
        a.dqkv = w_dqkv;
        a.ld_dqkv = wd;
        a.dk_col = ad;
        a.dv_col = ad + kd;
        a.batch = plan->cfg.batch;
        a.seq = plan->cfg.seq;
        a.heads = static_cast<int>(plan->a);
        a.kv_heads = static_cast<int>(plan->k);
        a.head_dim = static_cast<int>(plan->d);
        a.t = static_cast<int>(plan->t);
        a.status = plan->status;
        a.timeout_ns = plan->timeout_ns;
        if ((rc = run(tpi::attn_bwd_launch(a, s, &err), err))) return rc;
    }
    {  // dX = [dQ | dK | dV] [Wq ; Wk ; Wv]: f's all-reduce as the K loop over all shards
        tpi::GemmArgs g;
        g.mode = tpi::GEMM_NN;
        g.M = M;
        g.N = h;
        g.K = wd;
        g.A = w_dqkv;
        g.B0 = Wq;
        g.B1 = Wk;
        g.B2 = Wv;
        g.k_split = ad;
        g.k_split2 = ad + kd;
        g.out = dX;
        g.ldo = h;
        g.status = plan->status;
        g.timeout_ns = plan->timeout_ns;
        if ((rc = run(tpi::gemm_launch(g, s, &err), err))) return rc;
    }
    {  // [dWq ; dWk ; dWv] = [dQ | dK | dV]^T X
        tpi::GemmArgs g;
        g.mode = tpi::GEMM_TN;
        g.M = wd;
        g.N = h;
        g.K = M;
        g.A = w_dqkv;
        g.lda = wd;
        g.B0 = X;
        g.out = dWq;
        g.ldo = h;
        g.out2 = dWk;
        g.ldo2 = h;
        g.row_split = ad;
        g.out3 = dWv;
        g.ldo3 = h;
        g.row_split2 = ad + kd;
        g.accumulate = accumulate ? 1 : 0;
        g.status = plan->status;
        g.timeout_ns = plan->timeout_ns;
        if ((rc = run(tpi::gemm_launch(g, s, &err), err))) return rc;
    }
    return TP_OK;
}

int tp_layer_backward(tp_plan_t plan, const tp_bf16* X, const tp_layer_weights* w, const tp_bf16* dY,
                      tp_bf16* dX, const tp_layer_grads* grads, int accumulate, void* workspace,
                      size_t ws_bytes, void* stream) {
    if (!plan || !w || !grads) return fail(TP_ERR_INVALID_ARG, "plan, weights and grads must be non-NULL");
    if (!plan->has_attn || !plan->has_mlp)
        return fail(TP_ERR_INVALID_ARG, "a layer needs both attention (n_heads > 0) and an MLP (ffn > 0)");
    if (plan->h > 8192) return fail(TP_ERR_UNSUPPORTED, "layer RMSNorm supports hidden <= 8192");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(dY, "dY")) ||
        (rc = need_ptr(dX, "dX")))
        return rc;
    if (dX == X || dX == dY) return fail(TP_ERR_INVALID_ARG, "dX may not alias X or dY");
    if ((rc = check_ws(plan, TP_OP_LAYER_BACKWARD, workspace, ws_bytes))) return rc;
    const Layout L = layout_of(plan, TP_OP_LAYER_BACKWARD);
    size_t off = 0;
    auto take = [&](size_t n) {
        void* r = region(workspace, off);
        off += n;
        return r;
    };
    void* xn1 = take(L.lxn1);
    void* h1 = take(L.lh1);
    void* xn2 = take(L.lxn2);
    void* dxn = take(L.ldxn);
    void* dh1 = take(L.ldh1);
    void* qkv = take(L.lqkv);
    void* o = take(L.lo);
    float* lse = reinterpret_cast<float*>(take(L.llse));
    void* ug = take(L.lug);
    void* shared = take(L.lshared);
    cudaStream_t s = as_stream(stream);
    const float eps = plan->cfg.rms_eps;
    const int H = static_cast<int>(plan->h);
    std::string err;
    // Sequence parallel ("시퀀스 병렬화"): X, dY and dX live in the split
    // layout [t][batch][seq/t].  The forward's all-gathers become the
    // backward's reduce-scatters and the other way round; on one GPU the
    // shards' partial input gradients are already summed inside the fused
    // backward GEMMs, so the layer runs on token-order copies: dY and X are
    // gathered, and dX is written back into the split layout.  The weight
    // gradients are the replicated layer's.
    tp_bf16* dX_sp = nullptr;
    if (plan->cfg.sequence_parallel) {
        const int64_t B = plan->cfg.batch, S = plan->cfg.seq;
        const int T = static_cast<int>(plan->t);
        void* xf = take(L.lspx);
        void* dyf = take(L.lspdy);
        void* dxf = take(L.lspdx);
        if ((rc = run(tpi::sp_all_gather_launch(X, B, S, T, H, xf, s, &err), err))) return rc;
        if ((rc = run(tpi::sp_all_gather_launch(dY, B, S, T, H, dyf, s, &err), err))) return rc;
        X = static_cast<const tp_bf16*>(xf);
        dY = static_cast<const tp_bf16*>(dyf);
        dX_sp = dX;
        dX = static_cast<tp_bf16*>(dxf);
    }
    // Forward, keeping what the backward reads.
    if ((rc = run(tpi::rmsnorm_launch(X, plan->M, H, eps, xn1, s, &err), err))) return rc;
    if ((rc = do_qkv(plan, xn1, w->Wq, w->Wk, w->Wv, qkv, s))) return rc;
    if ((rc = do_attn_core(plan, qkv, o, s, lse))) return rc;
    if ((rc = do_rowwise(plan, o, plan->qw, w->Wo, plan->h, nullptr, X, nullptr, h1, true, s))) return rc;
    if ((rc = run(tpi::rmsnorm_launch(h1, plan->M, H, eps, xn2, s, &err), err))) return rc;
    if ((rc = do_colwise(plan, xn2, w->W1, w->W3, shared, s, nullptr, ug))) return rc;
    // MLP block, then the norm and the residual: dh1 = dY + RMSNorm'(h1)^T dxn2.
    if ((rc = tp_mlp_backward(plan, static_cast<const tp_bf16*>(xn2), w->W1, w->W3, w->W2, dY,
                              static_cast<const tp_bf16*>(ug), static_cast<tp_bf16*>(dxn), grads->dW1,
                              grads->dW3, grads->dW2, nullptr, accumulate, shared, L.lshared, stream)))
        return rc;
    if ((rc = run(tpi::rmsnorm_bwd_launch(h1, dxn, dY, plan->M, H, eps, dh1, s, &err), err))) return rc;
    // Attention block, then dX = dh1 + RMSNorm'(X)^T dxn1.
    if ((rc = tp_attn_backward(plan, static_cast<const tp_bf16*>(xn1), w->Wq, w->Wk, w->Wv, w->Wo,
                               static_cast<const tp_bf16*>(dh1), static_cast<const tp_bf16*>(qkv),
                               static_cast<const tp_bf16*>(o), lse, static_cast<tp_bf16*>(dxn), grads->dWq,
                               grads->dWk, grads->dWv, grads->dWo, accumulate, shared, L.lshared, stream)))
        return rc;
    if ((rc = run(tpi::rmsnorm_bwd_launch(X, dxn, dh1, plan->M, H, eps, dX, s, &err), err))) return rc;
    if (dX_sp)
        return run(tpi::sp_split_launch(dX, plan->cfg.batch, plan->cfg.seq, static_cast<int>(plan->t), H, dX_sp, s,
                                        &err),
                   err);
    return TP_OK;
}

int tp_layer_forward(tp_plan_t plan, const tp_bf16* X, const tp_layer_weights* w, tp_bf16* Y,
                     void* workspace, size_t ws_bytes, void* stream) {
    return tp_layer_forward_traced(plan, X, w, Y, workspace, ws_bytes, stream, nullptr, 0);
}

int tp_layer_forward_traced(tp_plan_t plan, const tp_bf16* X, const tp_layer_weights* w,
                            tp_bf16* Y, void* workspace, size_t ws_bytes, void* stream,
                            void* const* events, int n_events) {
    if (!plan || !w) return fail(TP_ERR_INVALID_ARG, "plan and weights must be non-NULL");
    if (!plan->has_attn || !plan->has_mlp)
        return fail(TP_ERR_INVALID_ARG, "a layer needs both attention (n_heads > 0) and an MLP (ffn > 0)");
    if (plan->h > 8192) return fail(TP_ERR_UNSUPPORTED, "layer RMSNorm supports hidden <= 8192");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(Y, "Y")) ||
        (rc = need_ptr(w->Wq, "Wq")) || (rc = need_ptr(w->Wk, "Wk")) || (rc = need_ptr(w->Wv, "Wv")) ||
        (rc = need_ptr(w->Wo, "Wo")) || (rc = need_ptr(w->W1, "W1")) || (rc = need_ptr(w->W2, "W2")))
        return rc;
    if (plan->cfg.act == TP_ACT_SWIGLU) {
        if ((rc = need_ptr(w->W3, "W3 (SwiGLU)"))) return rc;
    } else if (w->W3) {
        return fail(TP_ERR_INVALID_ARG, "W3 must be NULL unless act is TP_ACT_SWIGLU");
    }
    if (X == Y) return fail(TP_ERR_INVALID_ARG, "X and Y must not alias");
    if ((rc = check_ws(plan, TP_OP_LAYER, workspace, ws_bytes))) return rc;
    const bool fused_mode = plan->cfg.reduce_mode == TP_REDUCE_FUSED;
    const bool sp_mode = plan->cfg.sequence_parallel != 0;
    const int need_events = fused_mode ? (sp_mode ? 9 : 7) : sp_mode ? 11 : 9;
    if (events) {
        if (n_events < need_events)
            return fail(TP_ERR_INVALID_ARG, "%d events given, %d needed", n_events, need_events);
        for (int i = 0; i < need_events; ++i)
            if (!events[i]) return fail(TP_ERR_INVALID_ARG, "event %d is NULL", i);
    }
    int ev_i = 0;
    auto mark = [&](cudaStream_t st) {
        if (events) cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[ev_i++]), st);
    };
    const Layout L = layout_of(plan, TP_OP_LAYER);
    size_t off = 0;
    void* Yb = region(workspace, off); off += L.y;
    void* QKV = region(workspace, off); off += L.qkv;
    void* O = region(workspace, off); off += L.o;
    void* xn = region(workspace, off); off += L.xn;
    void* h1 = region(workspace, off); off += L.h1;
    void* P = L.partials ? region(workspace, off) : nullptr; off += L.partials;
    float* ss1 = L.ss ? reinterpret_cast<float*>(region(workspace, off)) : nullptr;
    off += L.ss;
    void* full = L.full ? region(workspace, off) : nullptr;
    float* ss2 = ss1 ? ss1 + plan->M : nullptr;
    const float eps = plan->cfg.rms_eps;
    cudaStream_t s = as_stream(stream);
    std::string err;
    if (fused_mode && sp_mode) {
        // Sequence parallel with g in the accumulator: X, h1 and Y stay in the
        // sequence-split layout.  Each block's input is gathered into token
        // order; its norm is folded into the colwise GEMM as in the
        // replicated layer; the reduce-scatter is the rowwise GEMM's sum over
        // shards in TMEM, written (with the residual) straight into the split
        // layout, so no partials go through HBM.
        const int64_t B = plan->cfg.batch, S = plan->cfg.seq;
        const int T = (int)plan->t, Hd = (int)plan->h;
        mark(s);
        if ((rc = run(tpi::sp_all_gather_launch(X, B, S, T, Hd, full, s, &err), err))) return rc;
        mark(s);
        if ((rc = run(tpi::row_sumsq_launch(full, plan->M, Hd, ss1, nullptr, s, &err), err))) return rc;
        mark(s);
        if ((rc = do_qkv(plan, full, w->Wq, w->Wk, w->Wv, QKV, s, ss1))) return rc;
        mark(s);
        if ((rc = do_attn_core(plan, QKV, O, s))) return rc;
        mark(s);
        if ((rc = do_rowwise(plan, O, plan->qw, w->Wo, plan->h, nullptr, X, nullptr, h1, true, s, ss2, true)))
            return rc;
        mark(s);
        if ((rc = run(tpi::sp_all_gather_launch(h1, B, S, T, Hd, full, s, &err), err))) return rc;
        mark(s);
        if ((rc = do_colwise(plan, full, w->W1, w->W3, Yb, s, ss2, nullptr, static_cast<int>((plan->h + 127) / 128))))
            return rc;
        mark(s);
        if ((rc = do_rowwise(plan, Yb, plan->fw, w->W2, plan->h, nullptr, h1, nullptr, Y, true, s, nullptr, true)))
            return rc;
        mark(s);
        return TP_OK;
    }
    if (fused_mode) {
        // RMSNorm is folded into the GEMMs: a unit-gain norm is a per-row
        // scale, so RMSNorm(x) W^T = rsqrt(mean(x^2) + eps) * (x W^T).  The
        // row statistic of x comes from one read-only pass, that of h1 from
        // the o_proj epilogue as one partial per 128-column slice, summed
        // in a fixed order by the W1/W3 GEMM.
        mark(s);
        if ((rc = run(tpi::row_sumsq_launch(X, plan->M, (int)plan->h, ss1, nullptr, s, &err), err))) return rc;
        mark(s);
        if ((rc = do_qkv(plan, X, w->Wq, w->Wk, w->Wv, QKV, s, ss1))) return rc;
        mark(s);
        if ((rc = do_attn_core(plan, QKV, O, s))) return rc;
        mark(s);
        // h1 = x + sum_i O_i Wo_i^T (g in the accumulator), and sum h1^2.
        if ((rc = do_rowwise(plan, O, plan->qw, w->Wo, plan->h, nullptr, X, nullptr, h1, true, s, ss2)))
            return rc;
        mark(s);
        if ((rc = do_colwise(plan, h1, w->W1, w->W3, Yb, s, ss2, nullptr, static_cast<int>((plan->h + 127) / 128))))
            return rc;
        mark(s);
        // y = h1 + sum_i act(xn A_i) B_i.
        if ((rc = do_rowwise(plan, Yb, plan->fw, w->W2, plan->h, nullptr, h1, nullptr, Y, true, s))) return rc;
        mark(s);
        return TP_OK;
    }
    if (sp_mode) {
        // Sequence parallel: X, h1 and Y stay split along the sequence; each
        // block's input is all-gathered after its local norm, and each g is a
        // reduce-scatter (fused with the next local norm).
        const int64_t B = plan->cfg.batch, S = plan->cfg.seq;
        const int T = (int)plan->t, Hd = (int)plan->h, pf = plan->cfg.partial_dtype == TP_F32 ? 1 : 0;
        mark(s);
        if ((rc = run(tpi::rmsnorm_launch(X, plan->M, Hd, eps, xn, s, &err), err))) return rc;
        mark(s);
        if ((rc = run(tpi::sp_all_gather_launch(xn, B, S, T, Hd, full, s, &err), err))) return rc;
        mark(s);
        if ((rc = do_qkv(plan, full, w->Wq, w->Wk, w->Wv, QKV, s))) return rc;
        mark(s);
        if ((rc = do_attn_core(plan, QKV, O, s))) return rc;
        mark(s);
        if ((rc = do_rowwise(plan, O, plan->qw, w->Wo, plan->h, nullptr, nullptr, P, nullptr, false, s)))
            return rc;
        mark(s);
        if ((rc = run(tpi::reduce_norm_launch(P, pf, T, plan->M, Hd, X, h1, xn, eps, s, &err, B, S, T), err)))
            return rc;
        mark(s);
        if ((rc = run(tpi::sp_all_gather_launch(xn, B, S, T, Hd, full, s, &err), err))) return rc;
        mark(s);
        if ((rc = do_colwise(plan, full, w->W1, w->W3, Yb, s))) return rc;
        mark(s);
        if ((rc = do_rowwise(plan, Yb, plan->fw, w->W2, plan->h, nullptr, nullptr, P, nullptr, false, s)))
            return rc;
        mark(s);
        if ((rc = run(tpi::reduce_norm_launch(P, pf, T, plan->M, Hd, h1, Y, nullptr, eps, s, &err, B, S, T),
                      err)))
            return rc;
        mark(s);
        return TP_OK;
    }
    // PARTIALS: the t partials of each block go through HBM and the g reduce.
    mark(s);
    if ((rc = run(tpi::rmsnorm_launch(X, plan->M, (int)plan->h, eps, xn, s, &err), err))) return rc;
    mark(s);
    if ((rc = do_qkv(plan, xn, w->Wq, w->Wk, w->Wv, QKV, s))) return rc;
    mark(s);
    if ((rc = do_attn_core(plan, QKV, O, s))) return rc;
    mark(s);
    if ((rc = do_rowwise(plan, O, plan->qw, w->Wo, plan->h, nullptr, nullptr, P, nullptr, false, s)))
        return rc;
    mark(s);
    // g of the attention block fused with the MLP's RMSNorm.
    if ((rc = run(tpi::reduce_norm_launch(P, plan->cfg.partial_dtype == TP_F32 ? 1 : 0, (int)plan->t,
                                          plan->M, (int)plan->h, X, h1, xn, eps, s, &err),
                  err)))
        return rc;
    mark(s);
    if ((rc = do_colwise(plan, xn, w->W1, w->W3, Yb, s))) return rc;
    mark(s);
    if ((rc = do_rowwise(plan, Yb, plan->fw, w->W2, plan->h, nullptr, nullptr, P, nullptr, false, s)))
        return rc;
    mark(s);
    if ((rc = do_reduce(plan, P, nullptr, h1, Y, plan->h, s))) return rc;
    mark(s);
    return TP_OK;
}

int tp_selftest_wait_timeout(tp_plan_t plan, uint64_t timeout_ns, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (timeout_ns < 1000ull || timeout_ns > 1000000000ull)
        return fail(TP_ERR_INVALID_ARG, "timeout_ns must be in [1e3, 1e9]");
    int rc;
    if ((rc = check_device(plan))) return rc;
    std::string err;
    return run(tpi::selftest_timeout_launch(plan->status, timeout_ns, as_stream(stream), &err), err);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free MLP: scratch in a file-scope device array.
//
// For callers that cannot allocate device memory at call time.  The array
// is sized once (TP_NOALLOC_SCRATCH_BYTES) and lives for the whole process on
// every GPU that loads this library.  Host code must not pass the array's
// name to a kernel -- on the host it is only a stand-in symbol -- so its
// device address is looked up with cudaGetSymbolAddress, once per device,
// with that device current, and the looked-up pointer is what the kernels
// receive.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TP_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// Device address of the scratch array on the current device (first call on
// a device resolves and caches it).
int noalloc_scratch(int dev, void** out) {
    if (dev < 0 || dev >= 64) return fail(TP_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr)
            return fail(TP_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(e));
        g_noalloc_addr[dev] = ptr;
    }
    *out = g_noalloc_addr[dev];
    return TP_OK;
}

}  // namespace

extern "C" int tp_mlp_forward_noalloc(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1,
                                      const tp_bf16* W3, const tp_bf16* W2, const tp_bf16* b2,
                                      const tp_bf16* residual, tp_bf16* Z, void* stream) {
    if (!plan) return fail(TP_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->has_mlp) return fail(TP_ERR_INVALID_ARG, "the plan has no MLP (ffn == 0)");
    int rc;
    if ((rc = check_device(plan)) || (rc = need_ptr(X, "X")) || (rc = need_ptr(W1, "W1")) ||
        (rc = need_ptr(W2, "W2")) || (rc = need_ptr(Z, "Z")) || (rc = opt_ptr(b2, "b2")) ||
        (rc = opt_ptr(residual, "residual")))
        return rc;
    if (plan->cfg.act == TP_ACT_SWIGLU) {
        if ((rc = need_ptr(W3, "W3 (SwiGLU)"))) return rc;
    } else if (W3) {
        return fail(TP_ERR_INVALID_ARG, "W3 must be NULL unless act is TP_ACT_SWIGLU");
    }
    const bool fused = plan->cfg.reduce_mode == TP_REDUCE_FUSED;
    const size_t y_bytes = align_up(static_cast<size_t>(plan->M) * plan->f * 2);
    const size_t p_bytes =
        fused ? 0 : align_up(static_cast<size_t>(plan->t) * plan->M * plan->h * partial_elem_bytes(plan));
    if (y_bytes + p_bytes > TP_NOALLOC_SCRATCH_BYTES)
        return fail(TP_ERR_WORKSPACE,
                    "this MLP needs %zu bytes of scratch; the built-in scratch array of "
                    "tp_mlp_forward_noalloc holds %zu bytes (use tp_mlp_forward with a workspace)",
                    y_bytes + p_bytes, (size_t)TP_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(plan->device, &scratch))) return rc;
    void* Y = scratch;
    void* P = fused ? nullptr : static_cast<uint8_t*>(scratch) + y_bytes;
    cudaStream_t s = as_stream(stream);
    if ((rc = do_colwise(plan, X, W1, W3, Y, s))) return rc;
    if ((rc = do_rowwise(plan, Y, plan->fw, W2, plan->h, b2, residual, P, Z, fused, s))) return rc;
    if (!fused) return do_reduce(plan, P, b2, residual, Z, plan->h, s);
    return TP_OK;
}

// ---------------------------------------------------------------------------
// Packed projections: one Linear packing several logical blocks along its
// output rows; every block is sharded on its own ("Tensor 병렬성", "Fused
// projections"; "추론을 위한 텐서 병렬성", "패킹 전략"; each block divisible by
// t individually, "제약 조건 및 검증").
namespace {

int check_packed_blocks(const int64_t* blocks, int32_t nblocks, int32_t t) {
    if (!blocks) return fail(TP_ERR_INVALID_ARG, "blocks is NULL");
    if (nblocks < 1 || nblocks > tpi::kMaxPackedBlocks)
        return fail(TP_ERR_INVALID_ARG, "nblocks must be in [1, %d]", tpi::kMaxPackedBlocks);
    if (t < 1 || t > 64) return fail(TP_ERR_INVALID_ARG, "t must be in [1, 64]");
    int64_t total = 0;
    for (int b = 0; b < nblocks; ++b) {
        if (blocks[b] <= 0) return fail(TP_ERR_INVALID_ARG, "block %d has size %lld", b, (long long)blocks[b]);
        total += blocks[b];
    }
    for (int b = 0; b < nblocks; ++b)
        if (blocks[b] % t)
            return fail(TP_ERR_NOT_DIVISIBLE,
                        "packed block %d (size %lld) does not divide by t = %d (each block must, "
                        "not only their sum %lld)",
                        b, (long long)blocks[b], t, (long long)total);
    if (total > (int64_t)1 << 30) return fail(TP_ERR_UNSUPPORTED, "packed rows above 2^30");
    return TP_OK;
}

}  // namespace

extern "C" int tp_packed_shard_table(const int64_t* blocks, int32_t nblocks, int32_t t,
                                     int32_t* out, int64_t cap, int64_t* n) {
    if (!n) return fail(TP_ERR_INVALID_ARG, "n is NULL");
    int rc;
    if ((rc = check_packed_blocks(blocks, nblocks, t))) return rc;
    const int64_t cnt = 2LL * t * nblocks;
    *n = cnt;
    if (cnt > cap || !out)
        return fail(TP_ERR_INVALID_ARG, "table needs %lld entries, capacity %lld", (long long)cnt,
                    (long long)cap);
    for (int32_t i = 0; i < t; ++i) {
        int64_t off = 0;
        for (int32_t b = 0; b < nblocks; ++b) {
            const int64_t w = blocks[b] / t;
            out[(i * nblocks + b) * 2 + 0] = static_cast<int32_t>(off + i * w);
            out[(i * nblocks + b) * 2 + 1] = static_cast<int32_t>(w);
            off += blocks[b];
        }
    }
    return TP_OK;
}

extern "C" int tp_packed_colwise_forward(const tp_bf16* X, int64_t M, int32_t h, const tp_bf16* W,
                                         const int64_t* blocks, int32_t nblocks, int32_t t,
                                         tp_bf16* Y, void* stream) {
    int rc;
    if ((rc = need_ptr(X, "X")) || (rc = need_ptr(W, "W")) || (rc = need_ptr(Y, "Y"))) return rc;
    if (M < 1 || M > (int64_t)1 << 30) return fail(TP_ERR_INVALID_ARG, "M out of range");
    if (h < 8 || h % 8) return fail(TP_ERR_INVALID_ARG, "h must be a positive multiple of 8");
    if ((rc = check_packed_blocks(blocks, nblocks, t))) return rc;
    tpi::GemmArgs g;
    g.mode = tpi::GEMM_COL_PACKED;
    int64_t total = 0, ws = 0;
    for (int b = 0; b < nblocks; ++b) {
        const int64_t w = blocks[b] / t;
        if (w % 64)
            return fail(TP_ERR_UNSUPPORTED,
                        "packed block %d gives %lld rows per shard; the GPU path needs multiples of 64",
                        b, (long long)w);
        g.pk_w[b] = static_cast<int>(w);
        g.pk_off[b] = total;
        total += blocks[b];
        ws += w;
    }
    g.pk_nb = nblocks;
    g.pk_ws = ws;
    g.M = M;
    g.N = total;
    g.A = X;
    g.K = h;
    g.t = t;
    g.B0 = W;
    g.B0_rows = total;
    g.out = Y;
    g.ldo = total;
    std::string err;
    return run(tpi::gemm_launch(g, as_stream(stream), &err), err);
}

// ---------------------------------------------------------------------------
// Vocabulary parallelism ("텐서 병렬화", "임베딩과 출력층").
namespace {

int check_vocab(int64_t M, int64_t v, int32_t t, int64_t align) {
    if (M < 0 || M > (int64_t)1 << 31) return fail(TP_ERR_INVALID_ARG, "M out of range");
    if (t < 1 || t > 64) return fail(TP_ERR_INVALID_ARG, "t must be in [1, 64]");
    if (v < 1 || v > (int64_t)1 << 31) return fail(TP_ERR_INVALID_ARG, "v out of range");
    if (v % t) return fail(TP_ERR_NOT_DIVISIBLE, "t = %d does not divide the vocabulary v = %lld", t,
                           (long long)v);
    if ((v / t) % align)
        return fail(TP_ERR_INVALID_ARG, "v / t = %lld must be a multiple of %lld",
                    (long long)(v / t), (long long)align);
    return TP_OK;
}

}  // namespace

extern "C" int tp_vocab_embedding_forward(const int32_t* ids, int64_t M, const tp_bf16* E, int64_t v,
                                          int32_t h, int32_t t, tp_bf16* out, void* stream) {
    int rc;
    if ((rc = need_ptr(ids, "ids")) || (rc = need_ptr(E, "E")) || (rc = need_ptr(out, "out"))) return rc;
    if ((rc = check_vocab(M, v, t, 1))) return rc;
    if (h < 8 || h % 8) return fail(TP_ERR_INVALID_ARG, "h must be a positive multiple of 8");
    std::string err;
    return run(tpi::vocab_embedding_launch(ids, M, E, v, h, out, as_stream(stream), &err), err);
}

extern "C" int tp_vocab_logits_forward(const tp_bf16* H, int64_t M, int32_t h, const tp_bf16* W,
                                       int64_t v, int32_t t, tp_bf16* logits, void* stream) {
    int rc;
    if ((rc = need_ptr(H, "H")) || (rc = need_ptr(W, "W")) || (rc = need_ptr(logits, "logits"))) return rc;
    if ((rc = check_vocab(M, v, t, 8))) return rc;
    if (M < 1) return fail(TP_ERR_INVALID_ARG, "M must be >= 1");
    if (h < 8 || h % 8) return fail(TP_ERR_INVALID_ARG, "h must be a positive multiple of 8");
    // Colwise over the vocabulary: shard i's logits are columns [i v/t,
    // (i+1) v/t) of one [M][v] result (its slice of W's rows).
    tpi::GemmArgs g;
    g.mode = tpi::GEMM_COL_ACT;
    g.act = TP_ACT_NONE;
    g.M = M;
    g.N = v;
    g.A = H;
    g.K = h;
    g.t = t;
    g.B0 = W;
    g.B0_rows = v;
    g.out = logits;
    g.ldo = v;
    std::string err;
    return run(tpi::gemm_launch(g, as_stream(stream), &err), err);
}

extern "C" int tp_vocab_parallel_cross_entropy(const tp_bf16* logits, int64_t M, int64_t v,
                                               int32_t t, const int32_t* labels, float* stats,
                                               float* loss, void* stream) {
    int rc;
    if ((rc = need_ptr(logits, "logits")) || (rc = need_ptr(labels, "labels")) ||
        (rc = need_ptr(stats, "stats")) || (rc = need_ptr(loss, "loss")))
        return rc;
    if ((rc = check_vocab(M, v, t, 8))) return rc;
    std::string err;
    return run(tpi::vocab_ce_launch(logits, M, v, t, labels, stats, loss, as_stream(stream), &err), err);
}

// ---------------------------------------------------------------------------
// Sequence parallelism ("텐서 병렬화", "시퀀스 병렬화").
extern "C" int tp_sp_all_gather(const tp_bf16* sp, int32_t batch, int32_t seq, int32_t t, int32_t h,
                                tp_bf16* full, void* stream) {
    int rc;
    if ((rc = need_ptr(sp, "sp")) || (rc = need_ptr(full, "full"))) return rc;
    if (batch < 0 || seq < 1 || t < 1 || t > 64) return fail(TP_ERR_INVALID_ARG, "bad batch/seq/t");
    if (seq % t) return fail(TP_ERR_NOT_DIVISIBLE, "t = %d does not divide seq = %d", t, seq);
    if (h < 8 || h % 8) return fail(TP_ERR_INVALID_ARG, "h must be a positive multiple of 8");
    if (sp == full) return fail(TP_ERR_INVALID_ARG, "sp and full must not alias");
    std::string err;
    return run(tpi::sp_all_gather_launch(sp, batch, seq, t, h, full, as_stream(stream), &err), err);
}

extern "C" int tp_sp_reduce_scatter(const void* partials, int partial_dtype, int32_t t, int32_t batch,
                                    int32_t seq, int32_t h, const tp_bf16* residual_sp, tp_bf16* out_sp,
                                    tp_bf16* xn_sp, float eps, void* stream) {
    int rc;
    if ((rc = need_ptr(partials, "partials")) || (rc = need_ptr(out_sp, "out_sp")) ||
        (rc = opt_ptr(residual_sp, "residual_sp")) || (rc = opt_ptr(xn_sp, "xn_sp")))
        return rc;
    if (partial_dtype != TP_F32 && partial_dtype != TP_BF16)
        return fail(TP_ERR_INVALID_ARG, "partial_dtype must be TP_F32 or TP_BF16");
    if (batch < 0 || seq < 1 || t < 1 || t > 64) return fail(TP_ERR_INVALID_ARG, "bad batch/seq/t");
    if (seq % t) return fail(TP_ERR_NOT_DIVISIBLE, "t = %d does not divide seq = %d", t, seq);
    if (h < 8 || h % 8 || h > 8192) return fail(TP_ERR_INVALID_ARG, "h must be a multiple of 8 in [8, 8192]");
    if (!(eps >= 0.0f)) return fail(TP_ERR_INVALID_ARG, "eps must be >= 0");
    std::string err;
    const int64_t rows = (int64_t)batch * seq;
    return run(tpi::reduce_norm_launch(partials, partial_dtype == TP_F32 ? 1 : 0, t, rows, h, residual_sp,
                                       out_sp, xn_sp, eps, as_stream(stream), &err, batch, seq, t),
               err);
}
