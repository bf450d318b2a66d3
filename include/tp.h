/*
 * tp.h -- C ABI of the single-GPU (sm_103a) Megatron-style tensor-parallel
 * transformer block: t-way column-then-row sharded MLP (GeLU / SwiGLU),
 * head-sharded causal GQA attention, and the g-operator reduction of the t
 * shard partials.
 *
 * Sources (web pages, cited by title and section):
 *   [wiki]  "텐서 병렬화" (itwiki, Tensor parallelism): "행렬 곱 나누기"
 *           (column- and row-parallel products), "MLP", "셀프 어텐션"
 *           (self-attention), "통신 연산 f와 g" (the f and g operators).
 *   [diff]  "Tensor 병렬성" (diffusers docs, tensor parallelism): "Colwise와
 *           rowwise" (styles table), "제약 조건 및 검증" (constraints and
 *           validation), "한계" (limits: errors instead of silent fallbacks).
 *   [trf]   "추론을 위한 텐서 병렬성" (transformers docs, tensor parallelism for
 *           inference): "분할 전략" (partitioning strategies), "설계 구현 /
 *           DTensor" (Shard / Replicate / Partial placements; rowwise bias).
 *
 * One process, one GPU: the t "devices" of the pages are shard indices.  A
 * colwise output that the pages leave sharded on the last dimension is stored
 * as one row-major [M][t * w] matrix whose column block i is shard i (the
 * Shard(-1) placement, [trf] "분할 전략").  A rowwise partial awaiting the
 * all-reduce (the Partial() placement) is an HBM buffer [t][M][h]; the g
 * operator is a local reduction of it, or is folded into the rowwise GEMM's
 * accumulator so no separate pass exists.
 *
 * Conventions for every call:
 *  - All tensors are row-major.  Weights use the nn.Linear layout W[out][in]
 *    ([diff] "Colwise와 rowwise": colwise shards weight dim 0, rowwise dim 1),
 *    passed whole and unsharded; shards are views (pointer + stride), never
 *    copies.  bf16 values are passed as their 16-bit patterns (tp_bf16).
 *  - Device pointers are caller-owned (e.g. allocated by PyTorch), must be
 *    16-byte aligned and must not alias one another unless stated.  The
 *    library allocates device memory only in tp_plan_create (a 256-byte
 *    status word) and never frees caller memory.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    only enqueue work; nothing synchronises implicitly.  The library's
 *    kernels use programmatic dependent launch: a kernel may start its
 *    prologue while the previous kernel of the stream is finishing, and
 *    touches global memory only once that kernel has completed.  Stream
 *    order therefore holds as usual for the caller's work.  A caller kernel
 *    that is itself launched with programmatic stream serialization right
 *    after one of the library's must execute griddepcontrol.wait before it
 *    reads the library's outputs.
 *  - Every call returns TP_OK or a TP_ERR_* code, and on error launches
 *    nothing ([diff] "한계": an error instead of a silent fallback;
 *    "제약 조건 및 검증": checks happen before any weight is touched).
 *    tp_last_error() then returns a message naming the failed rule.
 *  - The library runs only on sm_103a; there is no CPU path.
 */
#ifndef TP_H_
#define TP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ error codes */
#define TP_OK 0
#define TP_ERR_INVALID_ARG 1    /* null / negative / misaligned / bad enum   */
#define TP_ERR_NOT_DIVISIBLE 2  /* t does not divide f or a; bad (k, t) pair */
#define TP_ERR_UNSUPPORTED 3    /* a combination the library does not provide */
#define TP_ERR_WORKSPACE 4      /* workspace missing or smaller than needed   */
#define TP_ERR_CUDA 5           /* a CUDA runtime / driver call failed        */
#define TP_ERR_DEVICE_TIMEOUT 6 /* a bounded device-side wait gave up         */

/* Exported symbols of libtp.so (everything else in the library is hidden). */
#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

typedef uint16_t tp_bf16;
typedef struct tp_plan_s* tp_plan_t;

/* Activation of the colwise MLP projection.  GELU_ERF is the exact
 * x * Phi(x) form (the default of the [wiki] "MLP" example); SWIGLU is
 * SiLU(X W1^T) * (X W3^T) with W1 and W3 both colwise ([wiki] "MLP"); NONE is
 * the identity (a linear MLP, used to check exact integer products). */
enum { TP_ACT_GELU_ERF = 0, TP_ACT_GELU_TANH = 1, TP_ACT_SWIGLU = 2, TP_ACT_NONE = 3 };

/* How the rowwise GEMM's t partials are summed (the g operator).
 * FUSED: shard loop is the outer K loop of one accumulator; no partials
 *        buffer, no separate pass.
 * PARTIALS: each shard writes its Partial() [M][h] to a [t][M][h] buffer and
 *        tp_reduce_partials sums them. */
enum { TP_REDUCE_FUSED = 0, TP_REDUCE_PARTIALS = 1 };

/* Element type of a partials buffer. */
enum { TP_F32 = 0, TP_BF16 = 1 };

/* Operations whose workspace size tp_plan_workspace_bytes reports. */
enum {
    TP_OP_MLP = 0,
    TP_OP_ATTN = 1,
    TP_OP_LAYER = 2,
    TP_OP_MLP_BACKWARD = 3,
    TP_OP_ATTN_BACKWARD = 4,
    TP_OP_LAYER_BACKWARD = 5
};

/* Index tables tp_plan_shard_table exports (int32, row-major):
 *  FFN_SHARDS  [t][2]: first column of shard i in the ffn dimension, width f/t
 *  Q_HEAD_SHARD [a]  : shard holding query head j (= j / (a/t))
 *  Q_HEAD_KV    [a]  : KV head read by query head j (= j / (a/k))
 *  SHARD_KV    [t][2]: first KV head held by shard i, number held
 *                      (k/t own heads if k >= t, else 1 replica of head i*k/t)
 *  QKV_COLUMNS [t][3]: column offsets of Q_i, K_i, V_i in the QKV buffer */
enum {
    TP_TABLE_FFN_SHARDS = 0,
    TP_TABLE_Q_HEAD_SHARD = 1,
    TP_TABLE_Q_HEAD_KV = 2,
    TP_TABLE_SHARD_KV = 3,
    TP_TABLE_QKV_COLUMNS = 4
};

/* Configuration (plain data; copied by tp_plan_create).  Names follow the
 * pages: tokens M = batch * seq, hidden h, ffn f (0 = no MLP), n_heads a,
 * n_kv_heads k, head_dim d (a = 0: no attention), tp_degree t ([diff]
 * TensorParallelConfig(tp_degree); [trf] DistributedConfig(tp_size)). */
typedef struct {
    int64_t tokens;        /* M >= 1                                          */
    int32_t batch, seq;    /* attention is causal within each sequence;
                              tokens == batch * seq when n_heads > 0           */
    int32_t hidden;        /* h, multiple of 8                                */
    int32_t ffn;           /* f, t | f, (f/t) multiple of 8; 0 = no MLP       */
    int32_t n_heads;       /* a, t | a; 0 = no attention                      */
    int32_t n_kv_heads;    /* k, k | a, and t | k (k >= t) or k | t (k < t)    */
    int32_t head_dim;      /* d in {64, 128}                                  */
    int32_t tp_degree;     /* t in [1, 64]                                    */
    int32_t act;           /* TP_ACT_* of the MLP                             */
    int32_t reduce_mode;   /* TP_REDUCE_*                                     */
    int32_t partial_dtype; /* TP_F32 or TP_BF16 (PARTIALS mode only)          */
    float rms_eps;         /* RMSNorm epsilon (layer only), > 0               */
    int32_t sequence_parallel; /* 1: layer in/out in the sequence-split layout
                                  [t][batch][seq/t][h] (needs t | seq);
                                  0: replicated [M][h]                        */
} tp_config;

/* Weights of one layer, all full nn.Linear matrices [out][in] in bf16:
 * Wq [a d][h], Wk/Wv [k d][h], Wo [h][a d], W1/W3 [f][h], W2 [h][f]. */
typedef struct {
    const tp_bf16 *Wq, *Wk, *Wv, *Wo, *W1, *W3, *W2;
} tp_layer_weights;

/* fp32 weight gradients of one layer, shaped as the weights
 * (dW3 NULL unless the MLP is SwiGLU). */
typedef struct {
    float *dWq, *dWk, *dWv, *dWo, *dW1, *dW3, *dW2;
} tp_layer_grads;

/* ------------------------------------------------------------ plan */

/* Validate a configuration and build the shard layout.  All divisibility and
 * alignment rules are checked here, before any weight is read ([diff]
 * "제약 조건 및 검증": tp_degree divides the head count, checked before
 * loading; [wiki] "셀프 어텐션": KV heads replicated when fewer than t).
 * Allocates a 256-byte device status word on the current device.
 * Returns TP_ERR_INVALID_ARG, TP_ERR_NOT_DIVISIBLE, TP_ERR_UNSUPPORTED or
 * TP_ERR_CUDA on failure, with *out set to NULL. */
TP_API int tp_plan_create(const tp_config* cfg, tp_plan_t* out);

/* Host-only validation of a configuration: the same rules as
 * tp_plan_create, with no device work (usable without a GPU). */
TP_API int tp_config_check(const tp_config* cfg);

/* Host-only form of tp_plan_shard_table for a configuration that passes
 * tp_config_check (usable without a GPU). */
TP_API int tp_config_shard_table(const tp_config* cfg, int which, int32_t* out, int64_t cap, int64_t* n);

/* Free a plan (NULL is accepted).  The caller must ensure no launched work
 * still uses it. */
TP_API int tp_plan_destroy(tp_plan_t plan);

/* Bytes of caller-provided device workspace the op needs (TP_OP_*). */
TP_API int tp_plan_workspace_bytes(tp_plan_t plan, int op, size_t* bytes);

/* Copy index table `which` (TP_TABLE_*) into host array out[cap]; *n gets
 * the number of int32 entries (also when cap is too small, which returns
 * TP_ERR_INVALID_ARG).  Host-only; no device work. */
TP_API int tp_plan_shard_table(tp_plan_t plan, int which, int32_t* out, int64_t cap, int64_t* n);

/* Read and clear the plan's device status word (synchronises `stream`).
 * TP_OK; TP_ERR_DEVICE_TIMEOUT when a kernel's bounded wait gave up;
 * TP_ERR_CUDA when a kernel found its shared-memory layout does not fit its
 * allocation and stopped without computing (its outputs are not written). */
TP_API int tp_get_device_status(tp_plan_t plan, void* stream);

/* Thread-local description of the last error (never NULL). */
TP_API const char* tp_last_error(void);

/* ------------------------------------------------------------ g operator */

/* out[e] = sum_{i<t} partials[i][e] (+ bias[e % h]) (+ residual[e]), bf16.
 * The forward of g ([wiki] "통신 연산 f와 g": all-reduce of the partial
 * sums); bias is the rowwise bias, replicated and added once after the
 * reduction ([trf] "DTensor"); residual is the replicated residual stream.
 * partials: device [t][n] of TP_F32 or TP_BF16 (partial_dtype); bias: device
 * [h] bf16 or NULL; residual, out: device [n] bf16 (residual may be NULL;
 * out may alias residual).  n % h == 0, h % 8 == 0.  Sums in fp32, shard
 * order i = 0..t-1. */
TP_API int tp_reduce_partials(const void* partials, int partial_dtype, int32_t t, int64_t n,
                       int32_t h, const tp_bf16* bias, const tp_bf16* residual, tp_bf16* out,
                       void* stream);

/* y = x / sqrt(mean_j x_j^2 + eps) per row of h (unit gain), bf16 in/out,
 * fp32 arithmetic.  The replicated norm of [wiki] "통신 연산 f와 g".
 * x, y: device [rows][h]; h % 8 == 0, h <= 8192. */
TP_API int tp_rmsnorm(const tp_bf16* x, int64_t rows, int32_t h, float eps, tp_bf16* y, void* stream);

/* ------------------------------------------------------------ MLP */

/* Colwise projection with the activation fused ([wiki] "MLP": the first
 * matrix is split by columns so the nonlinearity needs no sync):
 *   Y[:, block i] = act(X W1_i^T)              (GeLU / none)
 *   Y[:, block i] = SiLU(X W1_i^T) * (X W3_i^T) (SwiGLU)
 * X: device [M][h]; W1, W3: device [f][h] (W3 only for SwiGLU, else NULL);
 * Y: device [M][f], column block i (width f/t) is shard i.  bf16 in and out,
 * fp32 accumulation, activation applied to the fp32 accumulator. */
TP_API int tp_colwise_forward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1, const tp_bf16* W3,
                       tp_bf16* Y, void* stream);

/* Rowwise projection of the colwise output ([wiki] "행렬 곱 나누기": row
 * parallel, Y_i B_i then a sum).  Shard i multiplies column block i of Y by
 * column block i of W2 (B_i = rows of B = columns of W2).
 *   FUSED:    Z = sum_i Y_i W2_i^T (+ bias) (+ residual), bf16; partials unused.
 *   PARTIALS: partials[i] = Y_i W2_i^T as [t][M][h] (plan's partial_dtype);
 *             Z, bias, residual unused (sum with tp_reduce_partials).
 * Y: device [M][f]; W2: device [h][f]; bias: [h] or NULL; residual: [M][h]
 * or NULL (may alias Z). */
TP_API int tp_rowwise_forward(tp_plan_t plan, const tp_bf16* Y, const tp_bf16* W2, const tp_bf16* bias,
                       const tp_bf16* residual, void* partials, tp_bf16* Z, void* stream);

/* The whole sharded MLP: Z = sum_i act(X A_i) B_i (+ bias once) (+ residual)
 * ([wiki] "MLP").  In PARTIALS mode the t partials are written to `partials`
 * ([t][M][h], required) and then reduced into Z; in FUSED mode `partials`
 * may be NULL.  workspace: device, >= tp_plan_workspace_bytes(TP_OP_MLP)
 * (holds the colwise output [M][f] bf16 at offset 0). */
TP_API int tp_mlp_forward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1, const tp_bf16* W3,
                   const tp_bf16* W2, const tp_bf16* b2, const tp_bf16* residual, void* partials,
                   tp_bf16* Z, void* workspace, size_t ws_bytes, void* stream);

/* tp_mlp_forward without a workspace, for callers that cannot allocate
 * device memory when they call: e.g. a framework whose memory manager owns
 * all device memory and forbids allocations behind its back, a plugin that
 * has no allocator handle, or a latency-critical loop where cudaMalloc's
 * implicit device synchronisation would stall other streams.  The pages have
 * no counterpart of this call; it computes exactly what tp_mlp_forward does.
 *
 * Scratch (the colwise output [M][f] bf16 and, in PARTIALS mode, the
 * [t][M][h] partials) lives in one file-scope device array of
 * TP_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU loading the library
 * holds until process exit.  A plan whose scratch needs more returns
 * TP_ERR_WORKSPACE before any launch.  The call itself allocates nothing
 * (no cudaMalloc / cudaFree / allocating library routine); the plan is
 * created beforehand, at set-up time, by tp_plan_create.
 *
 * The first call on a device resolves the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array and it keeps the last call's
 * contents: calls that overlap on the GPU (different streams, or different
 * threads without ordering) race with each other.  Calls on one stream are
 * ordered and safe.  Every scratch byte read is first written by the same
 * call, so nothing needs clearing between calls.
 * Arguments as tp_mlp_forward, minus partials / workspace. */
#define TP_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
TP_API int tp_mlp_forward_noalloc(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1,
                                  const tp_bf16* W3, const tp_bf16* W2, const tp_bf16* b2,
                                  const tp_bf16* residual, tp_bf16* Z, void* stream);

/* tp_mlp_forward that also saves what its backward needs: the
 * pre-activations UG, bf16, [M][f] U = X W1^T for GeLU / none, [M][2f] for
 * SwiGLU (U at columns [0, f), G = X W3^T at [f, 2f)); shard i's slice of
 * U (and G) is its column block i of width f/t, the layout of the colwise
 * output.  Everything else as tp_mlp_forward.  UG: device, 16-byte
 * aligned, not aliasing the other buffers. */
TP_API int tp_mlp_forward_train(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1,
                                const tp_bf16* W3, const tp_bf16* W2, const tp_bf16* b2,
                                const tp_bf16* residual, void* partials, tp_bf16* Z, tp_bf16* UG,
                                void* workspace, size_t ws_bytes, void* stream);

/* Backward of the sharded MLP ([wiki] "통신 연산 f와 g": g, at the block's
 * output, is the identity in the backward pass, so every shard receives
 * the same dZ; f, at its input, becomes the all-reduce of the shards'
 * partial input gradients).  With dZ = dL/dZ [M][h]:
 *   dH_i  = dZ W2_i                                  (W2_i: columns of shard i)
 *   dU_i  = dH_i (.) act'(U_i);  SwiGLU: dU_i = dH_i (.) G_i (.) SiLU'(U_i),
 *           dG_i = dH_i (.) SiLU(U_i)
 *   dX    = sum_i dU_i W1_i (+ dG_i W3_i)           (f's all-reduce; the sum
 *           over i runs inside one accumulator, as the FUSED forward's g)
 *   dW1_i = dU_i^T X,  dW3_i = dG_i^T X,  dW2_i = dZ^T H_i,  db2 = sum_m dZ[m]
 * where H_i = act(U_i) (SwiGLU: SiLU(U_i) (.) G_i) and W1_i, W3_i are the row
 * blocks of shard i.  Any residual added in the forward passes dZ through
 * unchanged; it is the caller's.
 * X [M][h], W1, W3 [f][h], W2 [h][f], dZ [M][h]: device bf16 as in
 * tp_mlp_forward.  UG: the pre-activations tp_mlp_forward_train saved, or
 * NULL to recompute them here (one more colwise GEMM).
 * dX: device [M][h] bf16.  dW1, dW3: device [f][h] fp32 (dW3 must be NULL
 * unless act is SwiGLU), dW2: [h][f] fp32, db2: [h] fp32 or NULL.  With
 * accumulate != 0 the weight gradients are added to what the buffers hold
 * (gradient accumulation over micro-batches); else they are overwritten.
 * Workspace: tp_plan_workspace_bytes(TP_OP_MLP_BACKWARD) bytes, device.
 * SwiGLU needs f to be a multiple of 64 (TP_ERR_UNSUPPORTED otherwise);
 * the reduce mode and partial dtype of the plan do not apply. */
TP_API int tp_mlp_backward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* W1, const tp_bf16* W3,
                           const tp_bf16* W2, const tp_bf16* dZ, const tp_bf16* UG, tp_bf16* dX,
                           float* dW1, float* dW3, float* dW2, float* db2, int accumulate,
                           void* workspace, size_t ws_bytes, void* stream);

/* Sizes of what the attention backward reads from its forward: the
 * shard-blocked QKV buffer ([M][t (a/t + 2 kv_held) d] bf16, as
 * tp_qkv_forward writes it), the attention output O ([M][a d] bf16) and the
 * softmax statistics LSE ([a][batch][seq_pad] fp32, seq_pad = seq rounded up
 * to a multiple of 64; entry (j, b, pos) is the base-2 log of the row's
 * sum of 2^(s log2(e) / sqrt(d)) over its causal keys, s the raw scores).
 * Any pointer may be NULL. */
TP_API int tp_plan_attn_saved_bytes(tp_plan_t plan, size_t* qkv_bytes, size_t* o_bytes, size_t* lse_bytes);

/* tp_attn_forward that keeps what its backward reads: QKV, O and LSE (sizes
 * from tp_plan_attn_saved_bytes; device, 16-byte aligned, not aliasing).
 * These replace the forward's workspace; everything else is as in
 * tp_attn_forward. */
TP_API int tp_attn_forward_train(tp_plan_t plan, const tp_bf16* X, const tp_bf16* Wq, const tp_bf16* Wk,
                                 const tp_bf16* Wv, const tp_bf16* Wo, const tp_bf16* residual,
                                 void* partials, tp_bf16* out, tp_bf16* QKV, tp_bf16* O, float* LSE,
                                 void* stream);

/* Backward of the head-sharded attention block ([wiki] "셀프 어텐션" and
 * "통신 연산 f와 g").  g at the block's output is the identity backward:
 * every shard receives the same dOut [M][h].  Then
 *   dO_i  = dOut Wo_i,   dWo_i = dOut^T O_i         (Wo_i: columns of shard i)
 *   dQ, dK, dV per head by the chain rule through the causal softmax:
 *           dV = P^T dO, dS = P (.) (dO V^T - rowsum(dO (.) O)),
 *           dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d);
 *           a KV head's gradient sums over the query heads that read it,
 *           which also sums its replicas when k < t
 *   dX    = sum_i (dQ_i Wq_i + dK_i Wk_i + dV_i Wv_i)  (f's all-reduce; the
 *           sum over shards runs inside one accumulator)
 *   dWq = dQ^T X, dWk = dK^T X, dWv = dV^T X.
 * X, Wq, Wk, Wv, Wo as in tp_attn_forward; dOut [M][h] bf16.  QKV, O, LSE:
 * from tp_attn_forward_train, or all NULL to recompute them here (the QKV
 * GEMM and the attention forward run again).  dX: [M][h] bf16.  dWq [a d][h],
 * dWk, dWv [k d][h], dWo [h][a d]: fp32, overwritten, or added to when
 * accumulate != 0.  Workspace: tp_plan_workspace_bytes(TP_OP_ATTN_BACKWARD)
 * bytes (it covers recomputation).  Head dimensions 64 and 128 (the plan's);
 * the plan's reduce mode does not apply. */
TP_API int tp_attn_backward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* Wq, const tp_bf16* Wk,
                            const tp_bf16* Wv, const tp_bf16* Wo, const tp_bf16* dOut, const tp_bf16* QKV,
                            const tp_bf16* O, const float* LSE, tp_bf16* dX, float* dWq, float* dWk,
                            float* dWv, float* dWo, int accumulate, void* workspace, size_t ws_bytes,
                            void* stream);

/* Backward of one pre-norm layer (the layer of tp_layer_forward), a whole
 * training step but the output: the forward is recomputed with what its
 * backward reads saved in the workspace, then
 *   MLP block backward at xn2 = RMSNorm(h1) with dZ = dY  ->  dxn2
 *   dh1 = dY + RMSNorm'(h1)^T dxn2                       (residual + norm)
 *   attention block backward at xn1 = RMSNorm(X), dOut = dh1  ->  dxn1
 *   dX  = dh1 + RMSNorm'(X)^T dxn1
 * where the blocks' backward passes are those of tp_mlp_backward and
 * tp_attn_backward (g backward identity, f backward the sum of the shards'
 * partial input gradients) and RMSNorm has unit gain.  X, dY, dX: device
 * [M][h] bf16 (dX may not alias X or dY); w: the layer's weights; grads: fp32
 * weight gradients, overwritten or, with accumulate != 0, added to.
 * Workspace: tp_plan_workspace_bytes(TP_OP_LAYER_BACKWARD).  With a
 * sequence-parallel plan ([wiki] "시퀀스 병렬화") X, dY and dX are in the
 * split layout [t][batch][seq/t][h] of tp_layer_forward: the backward of the
 * forward's all-gathers is a reduce-scatter of the shards' partial input
 * gradients, whose sum the fused backward GEMMs already hold, so dX is that
 * sum written into the split layout; the weight gradients are those of the
 * replicated layer.  Needs hidden <= 8192 and for SwiGLU f % 64 == 0
 * (TP_ERR_UNSUPPORTED otherwise). */
TP_API int tp_layer_backward(tp_plan_t plan, const tp_bf16* X, const tp_layer_weights* w, const tp_bf16* dY,
                             tp_bf16* dX, const tp_layer_grads* grads, int accumulate, void* workspace,
                             size_t ws_bytes, void* stream);

/* ------------------------------------------------------------ packed projections */

/* Per-block shard layout of a packed projection: one Linear whose output
 * rows pack `nblocks` logical blocks of sizes blocks[0..nblocks) (e.g. gate
 * and up of SwiGLU as [f, f]; Q, K, V, gate, up as [h, h, h, 3h, 3h]).
 * Every block is sharded on its own ([diff] "Fused projections": plain
 * colwise slicing would cut across the concatenation; [trf] "패킹 전략":
 * each rank gets the matching slice of every block), and every block must
 * divide by t on its own, not only their sum ([diff] "제약 조건 및 검증").
 * out[(i * nblocks + b) * 2 + {0, 1}] = first packed row and row count of
 * block b held by shard i; *n = 2 t nblocks.  Host-only.
 * Errors: TP_ERR_NOT_DIVISIBLE (a block), TP_ERR_INVALID_ARG (nblocks not in
 * [1, 8], non-positive block, small capacity). */
TP_API int tp_packed_shard_table(const int64_t* blocks, int32_t nblocks, int32_t t, int32_t* out,
                                 int64_t cap, int64_t* n);

/* Colwise projection by a packed weight, all shards in one launch:
 * Y[:, shard block i] = X * (rows of W that shard i holds)^T, shard i's
 * column block being the concatenation, in block order, of its per-block
 * slices (width sum_b blocks[b] / t).  X: device [M][h]; W: device
 * [sum blocks][h]; Y: device [M][sum blocks]; bf16, fp32 accumulation.
 * Each blocks[b] / t must be a multiple of 64 (TP_ERR_UNSUPPORTED).
 * A packed SwiGLU gate_up weight W13 [2f][h] needs no copy for the MLP:
 * pass W1 = W13 and W3 = W13 + f * h to tp_colwise_forward / tp_mlp_forward
 * (their per-shard row mapping is exactly the per-block sharding); a packed
 * QKV weight [(a + 2k) d][h] likewise splits into Wq, Wk, Wv by offsets. */
TP_API int tp_packed_colwise_forward(const tp_bf16* X, int64_t M, int32_t h, const tp_bf16* W,
                                     const int64_t* blocks, int32_t nblocks, int32_t t, tp_bf16* Y,
                                     void* stream);

/* ------------------------------------------------------------ sequence parallelism */

/* Sequence-split layout ([wiki] "시퀀스 병렬화": the norm and dropout regions
 * are split along the sequence; entering the tensor-parallel region an
 * all-gather collects the sequence, leaving it a reduce-scatter sums the
 * partials and splits them along the sequence again, the same traffic as
 * the all-reduce; [wiki] "PyTorch로 쓰기": SequenceParallel on the norms,
 * Shard(1) outputs).  A sequence-split tensor is [t][batch][seq/t][h]:
 * piece i holds positions [i seq/t, (i+1) seq/t) of every sequence.
 *
 * All-gather: full[b seq + pos] = sp[piece(pos)][b][pos % (seq/t)].
 * sp, full: device bf16, [batch seq][h]; t | seq, h % 8 == 0. */
TP_API int tp_sp_all_gather(const tp_bf16* sp, int32_t batch, int32_t seq, int32_t t, int32_t h,
                            tp_bf16* full, void* stream);

/* Reduce-scatter of the t shard partials (token order, [t][batch seq][h],
 * TP_F32 or TP_BF16) into the sequence-split layout, plus the sequence-split
 * residual: out_sp = sum_i partials[i] (+ residual_sp), fp32 sums in shard
 * order, bf16 out.  xn_sp (nullable): also RMSNorm(out_sp) with unit gain
 * and `eps` (the next block's local norm, fused).  h <= 8192. */
TP_API int tp_sp_reduce_scatter(const void* partials, int partial_dtype, int32_t t, int32_t batch,
                                int32_t seq, int32_t h, const tp_bf16* residual_sp, tp_bf16* out_sp,
                                tp_bf16* xn_sp, float eps, void* stream);

/* ------------------------------------------------------------ vocabulary */

/* Vocab-parallel embedding lookup ([wiki] "임베딩과 출력층": the embedding
 * matrix is split along the vocabulary; [trf] "분할 전략":
 * EmbeddingParallel(shard_dim=0) all-reduces the partial lookups).  Shard i
 * holds rows [i v/t, (i+1) v/t) of E; its partial for an id is E[id] if it
 * owns the id, else zero, so out[m] = E[ids[m]] (a zero row when
 * ids[m] is outside [0, v): no shard owns it).  ids: device [M] int32;
 * E: device [v][h] bf16 (nn.Embedding rows); out: device [M][h] bf16.
 * Errors: TP_ERR_NOT_DIVISIBLE when t does not divide v. */
TP_API int tp_vocab_embedding_forward(const int32_t* ids, int64_t M, const tp_bf16* E, int64_t v,
                                      int32_t h, int32_t t, tp_bf16* out, void* stream);

/* Vocab-parallel output projection: logits[M][v] = H W^T with W [v][h]
 * split by rows (colwise over the vocabulary), all shards in one launch;
 * shard i's logits are columns [i v/t, (i+1) v/t).  bf16 in and out, fp32
 * accumulation.  (v / t) % 8 == 0. */
TP_API int tp_vocab_logits_forward(const tp_bf16* H, int64_t M, int32_t h, const tp_bf16* W,
                                   int64_t v, int32_t t, tp_bf16* logits, void* stream);

/* Cross-entropy from vocab-sharded logits, exchanging only per-token
 * statistics ([wiki] "임베딩과 출력층": the max and the sum, b x s values,
 * instead of the b x s x v logits).  Shard i (columns [i v/t, (i+1) v/t) of
 * logits) computes m_i = max z, s_i = sum exp(z - m_i) and y_i = z_label if
 * it owns the label (else 0) into stats[3][t][M] (fp32: the exchanged
 * values); then loss[m] = log(sum_i s_i exp(m_i - m)) + m - sum_i y_i with
 * m = max_i m_i.  labels: device [M] int32, -100 = ignored (loss 0), any
 * other value outside [0, v) gives NaN.  logits: device [M][v] bf16;
 * stats: device [3 t M] fp32 (caller-owned scratch); loss: device [M] fp32.
 * (v / t) % 8 == 0. */
TP_API int tp_vocab_parallel_cross_entropy(const tp_bf16* logits, int64_t M, int64_t v, int32_t t,
                                           const int32_t* labels, float* stats, float* loss,
                                           void* stream);

/* ------------------------------------------------------------ attention */

/* Colwise Q/K/V projection, all shards in one launch ([wiki] "셀프 어텐션":
 * Q, K, V split by columns, a/t heads per shard).  QKV: device
 * [M][t * W], W = (a/t + 2 n_kv) d with n_kv the KV heads per shard; column
 * block i holds [Q_i | K_i | V_i] (offsets from TP_TABLE_QKV_COLUMNS). */
TP_API int tp_qkv_forward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* Wq, const tp_bf16* Wk,
                   const tp_bf16* Wv, tp_bf16* QKV, void* stream);

/* Causal GQA attention of every shard's heads, no communication ([wiki]
 * "셀프 어텐션": heads are independent).  For query head j of shard i and its
 * KV head g(j) = j / (a/k):  O_j = softmax(Q_j K_g^T / sqrt d + causal) V_g,
 * fp32 softmax, within each sequence.  QKV as written by tp_qkv_forward;
 * O: device [M][a d], head j at columns j d (column block i = shard i). */
TP_API int tp_attn_core_forward(tp_plan_t plan, const tp_bf16* QKV, tp_bf16* O, void* stream);

/* The whole head-sharded attention block: QKV colwise, attention, o_proj
 * rowwise, g ([wiki] "셀프 어텐션").  out = sum_i O_i Wo_i^T (+ residual).
 * partials: [t][M][h], required in PARTIALS mode.  workspace >=
 * tp_plan_workspace_bytes(TP_OP_ATTN). */
TP_API int tp_attn_forward(tp_plan_t plan, const tp_bf16* X, const tp_bf16* Wq, const tp_bf16* Wk,
                    const tp_bf16* Wv, const tp_bf16* Wo, const tp_bf16* residual, void* partials,
                    tp_bf16* out, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------ layer */

/* One pre-norm layer with two g reductions ([wiki] "통신 연산 f와 g": one
 * all-reduce after attention and one after the MLP; norm and residual
 * replicated):  h1 = x + Attn(RMSNorm(x)),  y = h1 + MLP(RMSNorm(h1)).
 * With cfg.sequence_parallel = 1, X and Y are in the sequence-split layout,
 * every block input is an all-gather and every g a reduce-scatter ([wiki]
 * "시퀀스 병렬화").  In PARTIALS mode the reduce-scatter sums the [t][M][h]
 * partials and fuses the next local norm; in FUSED mode it is the rowwise
 * GEMM's sum over shards in the accumulator, written with the residual into
 * the split layout, and the norms are folded into the colwise GEMMs.
 * X, Y: device [M][h] bf16 (may not alias).  Requires act == TP_ACT_SWIGLU
 * or a GeLU form (W3 NULL then).  workspace >= tp_plan_workspace_bytes(
 * TP_OP_LAYER); in PARTIALS mode it also holds the [t][M][h] partials. */
TP_API int tp_layer_forward(tp_plan_t plan, const tp_bf16* X, const tp_layer_weights* w, tp_bf16* Y,
                     void* workspace, size_t ws_bytes, void* stream);

/* tp_layer_forward that also records caller-created CUDA events (cudaEvent_t
 * handles) on `stream` at the boundaries of its kernels, for per-kernel
 * timing on the launching stream: events[0] before the first kernel and
 * events[i] after kernel i.  FUSED mode launches 6 kernels (row sums of
 * squares of x, QKV with the first RMSNorm folded in, attention,
 * o_proj + g + residual + row sums of squares of h1, W1/W3 colwise with the
 * second RMSNorm folded in, W2 + g + residual) and needs n_events >= 7;
 * PARTIALS mode launches 8 (RMSNorm, QKV, attention, o_proj partials,
 * g + RMSNorm, W1/W3 colwise, W2 partials, g) and needs 9.
 * Fewer events -> TP_ERR_INVALID_ARG before any launch. */
TP_API int tp_layer_forward_traced(tp_plan_t plan, const tp_bf16* X, const tp_layer_weights* w,
                                   tp_bf16* Y, void* workspace, size_t ws_bytes, void* stream,
                                   void* const* events, int n_events);

/* ------------------------------------------------------------ self test */

/* Failure-detection check: launches one CTA that waits on a shared-memory
 * barrier nothing ever arrives at, with a wait limit of `timeout_ns`
 * nanoseconds (1e3 .. 1e9).  The kernel gives up, records
 * TP_ERR_DEVICE_TIMEOUT in the plan's status word and returns normally, so
 * the context stays usable; read it with tp_get_device_status. */
TP_API int tp_selftest_wait_timeout(tp_plan_t plan, uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TP_H_ */
