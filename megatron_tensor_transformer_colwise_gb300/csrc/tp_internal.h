// tp_internal.h -- host-side interfaces shared by the translation units of
// libtp.so (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <string>

namespace tpi {

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes (its prologue overlaps that
// kernel's tail).  Every kernel launched this way calls pdl_wait() before it
// touches global memory.
inline void pdl_attribute(cudaLaunchAttribute& a) {
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    pdl_attribute(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Kinds of GEMM the tcgen05 kernel implements.  D[m][n] = sum_k A[m][k] B[n][k].
enum GemmMode {
    GEMM_COL_ACT = 0,     // colwise X W^T with a fused activation, bf16 out
    GEMM_COL_SWIGLU = 1,  // colwise SiLU(X W1^T) * (X W3^T), bf16 out
    GEMM_COL_QKV = 2,     // colwise Q|K|V per shard, bf16 out
    GEMM_ROW_FUSED = 3,   // rowwise, shards summed in the accumulator, + bias + residual
    GEMM_ROW_PARTIAL = 4, // rowwise, one [M][N] partial per shard (fp32 or bf16)
    GEMM_COL_PACKED = 5,  // colwise from a packed weight, each block sharded on its own
    // Backward GEMMs (operands read in their stored layout; "MN-major" =
    // the operand's M or N index is the contiguous one):
    GEMM_BWD_ACT = 6,     // dH = dZ W2 (B MN-major), epilogue: dU, dG, H from saved U, G
    GEMM_NN = 7,          // A K-major, B MN-major [K][N] (K rows split over B0 / B1)
    GEMM_TN = 8,          // A and B MN-major ([K][M], [K][N]), fp32 out split by rows
    GEMM_MLP = 9          // the whole sharded MLP in one persistent launch (see MlpArgs)
};

constexpr int kMaxPackedBlocks = 8;

struct GemmArgs {
    int mode = GEMM_COL_ACT;
    int act = 0;  // TP_ACT_* for GEMM_COL_ACT
    int64_t M = 0;
    int64_t N = 0;   // output columns (SwiGLU: columns of H)
    // Colwise: A is [M][K] (K = hidden).  Rowwise: A is [M][t * Ks], shard i
    // = column block i of width Ks; B is [N][t * Ks] likewise.
    const void* A = nullptr;
    int64_t K = 0;   // colwise reduction length
    int t = 1;       // shards
    int64_t Ks = 0;  // rowwise reduction length per shard
    const void* B0 = nullptr;
    const void* B1 = nullptr;
    const void* B2 = nullptr;
    int64_t B0_rows = 0, B1_rows = 0, B2_rows = 0;
    // QKV column segments of one shard: [q_w | kv_w | kv_w], shard width ws;
    // KV rows of shard i start at kv_first(i) * d.
    int64_t qkv_ws = 0, qkv_qw = 0, qkv_kvw = 0;
    int kv_heads = 0, head_dim = 0;
    // Packed blocks (GEMM_COL_PACKED): per-shard width and packed-row offset
    // of each block; a shard's output slice is the concatenation of its
    // per-block slices (pk_ws columns wide).
    int pk_nb = 0;
    int pk_w[kMaxPackedBlocks] = {0};
    int64_t pk_off[kMaxPackedBlocks] = {0};
    int64_t pk_ws = 0;
    // Output.
    void* out = nullptr;
    int64_t ldo = 0;
    int out_f32 = 0;  // GEMM_ROW_PARTIAL: 1 = fp32 partials, 0 = bf16
    const void* bias = nullptr;
    const void* residual = nullptr;
    int64_t ldr = 0;
    // RMSNorm folded into the GEMMs (unit gain): colwise modes scale each
    // accumulator row by rsqrt(sum_i row_ss[i M + row] * inv_h + eps) over
    // i < row_ss_parts when row_ss is set; GEMM_ROW_FUSED writes the sum of
    // squares of each output row's bf16 values over each 128-column slice s
    // to ss_out[s M + row] when ss_out is set (ceil(N / 128) slices, each
    // written once: the statistic is summed in a fixed order, so the layer
    // is bit-reproducible).
    const float* row_ss = nullptr;
    int row_ss_parts = 1;
    float* ss_out = nullptr;
    // GEMM_ROW_FUSED in a sequence-parallel layer: output and residual rows
    // live in the sequence-split layout [t][batch][seq/t] (token b seq + pos
    // at row ((pos / w) batch + b) w + pos % w, w = seq / t); ss_out stays in
    // token order.  sp_t == 0: token order.
    int64_t sp_batch = 0, sp_seq = 0;
    int sp_t = 0;
    float inv_h = 0.0f, eps = 0.0f;
    // Backward modes.
    //  GEMM_BWD_ACT: aux = saved pre-activations [M][ldaux] (U at column n,
    //    G at n_half + n for SwiGLU); out = dU (dG at n_half + n), ldo;
    //    out2 = H [M][ldo2] (nullable).  A = dZ [M][K], B0 = W2 [K][N].
    //  GEMM_NN: A [M][lda] K-major; B0 = [k_split][N], B1 = [k_split2 -
    //    k_split][N], B2 = [K - k_split2][N] (nullable when their K range is
    //    empty), MN-major; bf16 out.
    //  GEMM_TN: A [K][M] and B0 [K][N], both MN-major; fp32 out [M][N];
    //    rows in [row_split, row_split2) go to out2 (row - row_split), rows
    //    >= row_split2 to out3 (row - row_split2); accumulate adds.
    //  COL_ACT / COL_SWIGLU: aux_out (nullable) also receives the
    //    pre-activations (U, and G at n_half + n), ld ldaux.
    int64_t lda = 0;  // 0: K (K-major) or M (MN-major)
    const void* aux = nullptr;
    void* aux_out = nullptr;
    int64_t ldaux = 0;
    int64_t n_half = 0;
    void* out2 = nullptr;
    int64_t ldo2 = 0;
    int64_t k_split = 0, k_split2 = 0;
    void* out3 = nullptr;
    int64_t ldo3 = 0;
    int64_t row_split = 0, row_split2 = 0;
    int accumulate = 0;
    unsigned* status = nullptr;
    uint64_t timeout_ns = 2000000000ull;
};

// Encodes the tensor maps and launches the persistent tcgen05 GEMM on
// `stream`.  Returns 0 or a TP_ERR_* code with a message in *err.
int gemm_launch(const GemmArgs& a, cudaStream_t stream, std::string* err);

// Number of kernel launches gemm_launch issues (always 1).
constexpr int kGemmLaunches = 1;

// Elementwise / row kernels (tp_elementwise.cu).
int reduce_launch(const void* partials, int partial_f32, int t, int64_t n, int h,
                  const void* bias, const void* residual, void* out, cudaStream_t stream,
                  std::string* err);
// Row-wise reduce of the partials plus residual into h1 (bf16), and also
// xn = RMSNorm(h1) (unit gain) when xn != nullptr.
// sp_t > 0: residual, h1 and xn live in the sequence-split layout
// [sp_t][sp_batch][sp_seq / sp_t] (a reduce-scatter); partials in token order.
int reduce_norm_launch(const void* partials, int partial_f32, int t, int64_t rows, int h,
                       const void* residual, void* h1, void* xn, float eps, cudaStream_t stream,
                       std::string* err, int64_t sp_batch = 0, int64_t sp_seq = 0, int sp_t = 0);
// full[b * seq + pos] = sp[row of (b, pos) in [t][batch][seq / t]].
int sp_all_gather_launch(const void* sp, int64_t batch, int64_t seq, int t, int h, void* full,
                         cudaStream_t stream, std::string* err);
// sp[row of (b, pos) in [t][batch][seq / t]] = full[b * seq + pos].
int sp_split_launch(const void* full, int64_t batch, int64_t seq, int t, int h, void* sp,
                    cudaStream_t stream, std::string* err);
int rmsnorm_launch(const void* x, int64_t rows, int h, float eps, void* y, cudaStream_t stream,
                   std::string* err);
// ss[row] = sum_j x[row][j]^2 (fp32 over the bf16 values); zero[row] = 0
// when zero != nullptr (clears the next norm's accumulator).
int row_sumsq_launch(const void* x, int64_t rows, int h, float* ss, float* zero,
                     cudaStream_t stream, std::string* err);

// Attention core (tp_attn.cu).
struct AttnArgs {
    const void* QKV = nullptr;
    int64_t ld_qkv = 0;
    int64_t shard_w = 0, q_w = 0, kv_w = 0;  // column layout of one shard
    void* O = nullptr;
    int64_t ld_o = 0;
    int batch = 0, seq = 0, heads = 0, kv_heads = 0, head_dim = 0, t = 1;
    // Softmax statistics for the backward pass (nullable): lse[(j * batch +
    // b) * seq_pad + pos] = log2 of the row's sum of 2^(s / sqrt(d) * log2 e),
    // i.e. the base-2 log-sum-exp of the scaled scores, for pos < seq.
    float* lse = nullptr;
    int64_t seq_pad = 0;
    unsigned* status = nullptr;
    uint64_t timeout_ns = 2000000000ull;
};
int attn_launch(const AttnArgs& a, cudaStream_t stream, std::string* err);

// Attention core backward (tp_attn_bwd.cu), head_dim 128: three launches
// (statistics D and a zeroed dQ accumulator; the tcgen05 kernel; dQ to bf16).
struct AttnBwdArgs {
    const void* QKV = nullptr;  // the forward's shard-blocked Q | K | V buffer
    int64_t ld_qkv = 0;
    int64_t shard_w = 0, q_w = 0, kv_w = 0;
    const void* dO = nullptr;   // [tokens][a d] bf16, row stride ld_do (also O's)
    const void* O = nullptr;
    int64_t ld_do = 0;
    const float* lse = nullptr; // [a][batch][seq_pad], from the forward
    float* dstat = nullptr;     // [a][batch][seq_pad] scratch (D)
    int64_t seq_pad = 0;        // seq rounded up to a multiple of 64
    float* dq = nullptr;        // [tokens][ld_dq] fp32 scratch
    int64_t ld_dq = 0;
    void* dqkv = nullptr;       // bf16 out: dQ at columns [0, a d), dK of KV head g at
    int64_t ld_dqkv = 0;        // dk_col + g d, dV at dv_col + g d
    int64_t dk_col = 0, dv_col = 0;
    int batch = 0, seq = 0, heads = 0, kv_heads = 0, head_dim = 0, t = 1;
    unsigned* status = nullptr;
    uint64_t timeout_ns = 2000000000ull;
};
int attn_bwd_launch(const AttnBwdArgs& a, cudaStream_t stream, std::string* err);

// Vocabulary-parallel embedding and cross-entropy (tp_vocab.cu).
int vocab_embedding_launch(const int32_t* ids, int64_t M, const void* E, int64_t v, int h, void* out,
                           cudaStream_t stream, std::string* err);
int vocab_ce_launch(const void* logits, int64_t M, int64_t v, int t, const int32_t* labels,
                    float* stats, float* loss, cudaStream_t stream, std::string* err);

// out = res + RMSNorm'(x)^T g per row (unit gain; bf16 [rows][h], h % 8 == 0,
// h <= 8192); out may alias res.
int rmsnorm_bwd_launch(const void* x, const void* g, const void* res, int64_t rows, int h, float eps,
                       void* out, cudaStream_t stream, std::string* err);
// out[j] (+)= sum_r x[r][j] for a bf16 [rows][h] x (h % 8 == 0), fp32 out.
int colsum_launch(const void* x, int64_t rows, int h, float* out, int accumulate,
                  cudaStream_t stream, std::string* err);

// Self test: a kernel that waits on a barrier nobody arrives at.
int selftest_timeout_launch(unsigned* status, uint64_t timeout_ns, cudaStream_t stream,
                            std::string* err);

// The sharded MLP Z = sum_i act(X W1_i^T) W2_i^T (+ bias + residual) in one
// persistent launch, for problems too small to fill the GPU with the two
// GEMMs one after the other.  Its work units are the colwise tiles (256 x
// 256 of H = act(X W1^T), bf16) and then, per 256-row m-block, the rowwise
// tiles (256 x 256 of Z) in `pieces` K pieces of t / pieces shards each.  A
// rowwise unit starts once the colwise tiles holding its H columns are
// stored (per-tile counters); with pieces > 1 each piece writes an fp32
// partial and the last piece of a tile to arrive sums all of them in piece
// order (so the result does not depend on the arrival order) and writes Z.
struct MlpArgs {
    int act = 0;  // TP_ACT_GELU_ERF, TP_ACT_GELU_TANH or TP_ACT_NONE
    int64_t M = 0, h = 0, f = 0;
    int t = 1;
    int pieces = 1;  // divides t
    const void* X = nullptr;   // [M][h]
    const void* W1 = nullptr;  // [f][h]
    const void* W2 = nullptr;  // [h][f]
    const void* bias = nullptr;      // [h] or null
    const void* residual = nullptr;  // [M][h] or null
    void* Z = nullptr;               // [M][h] bf16
    void* H = nullptr;               // [M][f] bf16 scratch
    float* partials = nullptr;       // [pieces][M][h] fp32 scratch (pieces > 1)
    unsigned* counters = nullptr;    // mlp_fused_counter_words() words, zero at launch
    unsigned* status = nullptr;
    uint64_t timeout_ns = 0;
};
// K pieces the fused MLP launch would use for this problem on the current
// device, or 0 when the two-GEMM path suits it better (large problems,
// SwiGLU).
int mlp_fused_pieces(int64_t M, int64_t h, int64_t f, int t, int act);
int64_t mlp_fused_counter_words(int64_t M, int64_t h, int64_t f);
int mlp_fused_launch(const MlpArgs& a, cudaStream_t stream, std::string* err);

// Device properties cached per device.
int device_sm_count();

}  // namespace tpi
