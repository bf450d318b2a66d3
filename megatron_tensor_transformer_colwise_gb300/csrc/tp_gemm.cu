// tp_gemm.cu -- the column- and row-parallel GEMMs of the tensor-parallel
// block on sm_103a tensor cores (tcgen05 / TMEM), fed by TMA.
//
// Source: "텐서 병렬화" (itwiki, Tensor parallelism), sections "행렬 곱
// 나누기" (column parallel: Y_i = X A_i with X replicated; row parallel:
// Y_i = X_i A_i, then Y = sum_i Y_i), "MLP" (A colwise with the nonlinearity
// applied per shard, B rowwise, one sum at the end; SwiGLU with W1 and W3
// colwise) and "셀프 어텐션" (Q/K/V colwise, a/t heads per shard; o_proj
// rowwise).
//
// One kernel template, one CTA per SM (persistent), CTAs in pairs
// (clusters of 2) that share a 256 x 256 output tile, 6 or 10 warps per CTA:
//   warp 0      TMA producer (one lane): this CTA's 128 rows of A and half of
//               the tile's 256 B rows into a 6-stage ring (32 KB stages);
//               completion is counted on the pair leader's barriers
//   warp 1      TMEM owner; in the leader CTA also the MMA issuer (one lane):
//               256x256x16 bf16 UMMAs (tcgen05 cta_group::2) that read both
//               CTAs' shared memory and accumulate 128 rows in each CTA's TMEM
//   warps 2..   epilogue: TMEM -> registers -> fused op -> global (4 warps,
//               one per TMEM lane quadrant; 8 for the activation-gradient
//               and GeLU epilogues, two per quadrant on halves of the tile's
//               columns)
// The accumulator is double-buffered in TMEM (2 x 256 fp32 columns) so the
// epilogue of tile n overlaps the main loop of tile n+1.  Splitting B over
// the pair halves each SM's shared-memory operand traffic per FLOP.
// Rowwise problems that fit in one wave of 256 x 128 tiles use those
// instead (UMMA N = 128, 8 stages of 24 KB, 2 x 128 TMEM columns), so that
// twice as many SMs share a short output.
//
// Shards are grid/loop indices, not devices: a colwise output tile may span
// shard boundaries (the output is the concatenation of the shards' slices);
// the rowwise GEMM addresses shard i's K block through a 3-D tensor map
// (K per shard, shard, rows), so "fused" mode runs the shard loop as the
// outer K loop of one accumulator -- the g sum happens in TMEM -- and
// "partial" mode gives every shard its own [M][N] output.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "tp_device.cuh"
#include "tp_internal.h"
#include "tp_packed.cuh"

#ifndef TP_GEMM_CTA_PAIR
#define TP_GEMM_CTA_PAIR 2
#endif

namespace {

using namespace tpk;

constexpr int BM = 128;             // rows of the tile held by one CTA (TMEM lanes)
constexpr int BN = 256;             // UMMA N (TMEM columns per accumulator)
constexpr int BK = 64;              // one 128-byte swizzle row of bf16
constexpr int UK = 16;              // K of one kind::f16 UMMA
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_CHUNK_ROWS = 64;
constexpr int B_CHUNK_BYTES = B_CHUNK_ROWS * BK * 2;  // 8 KB
// Epilogue warps per CTA: one per TMEM lane quadrant, or two, each taking
// half of the tile's columns, where the epilogue of a tile would otherwise
// outlast the next tile's main loop: the activation gradient with its loads
// and three stores, and the GeLU epilogue of short-K problems (measured on
// GB300: the 2048 x 4096 x 1024 GeLU GEMM in 22.9 us with 8 warps, 24.8 us
// with 4).  The other forward modes keep 4: with 8 the layer step took
// 2.170 ms against 2.127 ms (W1/W3 1036 against 1011 us), and 4 keeps one
// warp per 128-column slice of a narrow rowwise tile, whose sum of squares
// it writes whole.
// The fused MLP (GEMM_MLP) runs two per quadrant as well: its tiles are
// short (16 k-blocks at the GPT-sized shapes) and every one of them has a
// GeLU or a partial-sum epilogue.
template <int MODE>
__host__ __device__ constexpr int epi_warps() {
    return (MODE == tpi::GEMM_MLP || MODE == tpi::GEMM_BWD_ACT || MODE == tpi::GEMM_COL_ACT) ? 8 : 4;
}
template <int MODE>
__host__ __device__ constexpr int num_threads() {
    return 64 + 32 * epi_warps<MODE>();
}
// CTAs per cluster.  The fused MLP runs clusters of two CTA pairs that take
// adjacent n-tiles of one m-block: each A tile is read from L2 once and
// multicast to both pairs (a quarter less operand traffic per MMA); the
// other modes run one pair (or one CTA) per cluster.
// The QKV GEMM runs the same clusters on its 256-column tiles: a cluster
// unit is two adjacent n-tiles of one m-block, one per pair, and each A
// tile is read from L2 once for both pairs (multicast).  Clusters of four
// fit on 144 of GB300's 152 SMs; QKV's 768 tiles take 11 rounds either way,
// so the lighter L2 load is a net gain there (224 -> 219 us), while the
// W1/W3 and rowwise GEMMs would gain rounds (47.2 -> 49.8 and 6.7 -> 7.1)
// and ran no faster (W1/W3) or slower (W2 506 -> 560 us).
template <int MODE>
__host__ __device__ constexpr bool mc_mode() {
    return MODE == tpi::GEMM_COL_QKV;
}
template <int MODE, int CG, int BNT = BN>
__host__ __device__ constexpr int cluster_ctas() {
    return (MODE == tpi::GEMM_MLP || (mc_mode<MODE>() && CG == 2 && BNT == BN)) ? 2 * CG : CG;
}

// CG = CTAs per tile.  CG = 1: a 128 x 256 tile per CTA, 4 stages of 48 KB.
// CG = 2: a 256 x 256 tile per CTA pair (cta_group::2): each CTA loads its
// 128 rows of A and half of the 256 B rows, 6 stages of 32 KB, and the
// pair's leader issues 256 x 256 x 16 UMMAs that read both CTAs' shared
// memory and write 128 accumulator rows into each CTA's TMEM.
//
// GEMM_BWD_ACT stages its three outputs through shared memory (one 32 x 32
// bf16 box per output and epilogue warp, 64-byte swizzle) and writes them
// with TMA stores; it runs one ring stage fewer to make room.  GEMM_TN
// stages its fp32 output the same way (two 32 x 32 fp32 boxes per epilogue
// warp, alternating, 128-byte swizzle), written by TMA stores or, when
// accumulating, TMA reduce-adds.
constexpr int EPI_BOX = 32;                        // rows and columns of an output box
constexpr int EPI_BOX_BYTES = EPI_BOX * EPI_BOX * 2;  // 2 KB
template <int MODE, int CG, int BNT = BN>
struct Cfg {
    static constexpr int B_BYTES = (BNT / CG) * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr bool STAGED_OUT = MODE == tpi::GEMM_BWD_ACT || MODE == tpi::GEMM_TN;
    // GEMM_COL_ACT stages its bf16 output through two alternating 32 x 32
    // boxes per epilogue warp (64-byte swizzle) when the output allows a
    // TMA map; the six ring stages still fit beside them.
    static constexpr bool COL_STAGED = MODE == tpi::GEMM_COL_ACT && CG == 2 && BNT == BN;
    static constexpr int STAGES = CG == 1 ? 4 : (STAGED_OUT ? 5 : (BNT == BN ? 6 : 8));
    static constexpr int CHUNKS = (BNT / B_CHUNK_ROWS) / CG;  // B boxes loaded per CTA
    static constexpr int TMEM_COLS = 2 * BNT;                  // two accumulators
    static constexpr int EPI_BYTES = MODE == tpi::GEMM_MLP    ? 8 * 2 * EPI_BOX_BYTES      // 8 warps x 2 boxes
                                     : MODE == tpi::GEMM_BWD_ACT ? 8 * 3 * EPI_BOX_BYTES     // 8 warps x 3 boxes
                                     : MODE == tpi::GEMM_TN    ? 4 * 2 * 2 * EPI_BOX_BYTES  // 4 warps x 2 fp32 boxes
                                     : COL_STAGED              ? 8 * 2 * EPI_BOX_BYTES      // 8 warps x 2 boxes
                                                               : 0;
    // GEMM_MLP adds one mbarrier per output box (TMA loads into the boxes).
    static constexpr int BOX_BARS = MODE == tpi::GEMM_MLP ? 16 : 0;
    static constexpr int BAR_BYTES = 8 * (2 * STAGES + 5) + 16 + 8 * BOX_BARS;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
    static constexpr int TILE_M = BM * CG;
};

struct GemmParams {
    CUtensorMap mapA;
    CUtensorMap mapB[3];
    int M, N;
    int kb_per_shard;  // k-blocks of BK per shard (colwise: per whole K)
    int k_shards;      // shards walked inside the K loop (ROW_FUSED: t)
    int m_tiles, n_tiles, grid_shards, num_tiles;
    int n_dec;  // n-columns of the decode grid: n_tiles, or pairs of n-tiles for cluster units
    int group_m;       // m-tiles per rasterisation group (weight-tile reuse in L2)
    int act;
    int b_rows0;       // rows of B0 (out-of-range chunks read zeros)
    int qkv_ws, qkv_qw, qkv_kvw, kv_heads, head_dim, tp;
    int pk_nb, pk_ws;
    int pk_w[tpi::kMaxPackedBlocks];
    int pk_off[tpi::kMaxPackedBlocks];
    void* out;
    long long ldo;
    long long shard_stride;  // ROW_PARTIAL: elements between shard outputs
    int out_f32;
    const __nv_bfloat16* bias;
    const __nv_bfloat16* residual;
    long long ldr;
    const float* row_ss;  // colwise: scale row by rsqrt(sum of row_ss_parts partials * inv_h + eps)
    int row_ss_parts;     // partials of row_ss, M apart
    float* ss_out;        // ROW_FUSED: sum of squares of the row's bf16 outputs per 128-column slice
    long long sp_batch, sp_seq;  // ROW_FUSED: output / residual rows in the sequence-split layout
    int sp_t;                    // (0: token order)
    float inv_h, eps;
    // Backward modes (see tpi::GemmArgs).
    const __nv_bfloat16* aux;  // BWD_ACT: saved pre-activations U (| G)
    __nv_bfloat16* aux_out;    // COL_ACT / COL_SWIGLU: pre-activations out
    long long ldaux, n_half;
    void* out2;
    long long ldo2;
    int k_split, k_split2;      // GEMM_NN: first K rows read from mapB[1], mapB[2]
    int row_split, row_split2;  // GEMM_TN: first output rows written to out2, out3
    void* out3;
    long long ldo3;
    int accumulate;
    int o_staged;  // GEMM_COL_ACT: out written through mapO[0] by TMA stores
    CUtensorMap mapO[3];  // BWD_ACT: TMA-store maps of dU, dG, H (64-byte swizzle)
    // GEMM_MLP (tpi::MlpArgs): mapA / mapB[0] are X / W1 of the colwise
    // tiles, out = H (ldo = f); the rowwise tiles read H and W2 as (Ks, t,
    // rows) and write Z (+ bias + residual, ldr = h).
    CUtensorMap mapH, mapW2;
    // Output boxes (32 rows x 64 bytes, 64-byte swizzle): H and Z stores,
    // residual loads, and the fp32 partials as (h, M, pieces) in 16-column
    // boxes (stores of the lower pieces, loads by the last one).
    CUtensorMap mapHs, mapZs, mapRs, mapPs;
    int mlp_col_units;    // colwise units (m_tiles x n_tiles), first in the unit order
    int mlp_row_n_tiles;  // 256-column tiles of Z
    int mlp_pieces;       // K pieces of the rowwise sum
    int mlp_spp;          // shards per piece
    int mlp_kb_row;       // k-blocks per shard of the rowwise GEMM
    int mlp_h;            // columns of Z
    long long mlp_ks;     // columns of H per shard (f / t)
    unsigned* mlp_ready;   // [m_tiles][8]: per K piece, CTAs that stored their half of a colwise
                           // tile overlapping the piece's H columns
    unsigned* mlp_pdone;   // [m_tiles][mlp_row_n_tiles][2]: lower pieces stored, per CTA half
    float* mlp_part;       // [mlp_pieces][M][mlp_h]
    __nv_bfloat16* mlp_z;  // [M][mlp_h]
    unsigned* status;
    unsigned long long timeout_ns;
};

// Which operands a mode reads MN-major (M or N index contiguous in global
// memory, [K][M] / [K][N]); the others are K-major ([M][K] / [N][K]).
template <int MODE>
struct Major {
    static constexpr bool A_MN = MODE == tpi::GEMM_TN;
    static constexpr bool B_MN =
        MODE == tpi::GEMM_BWD_ACT || MODE == tpi::GEMM_NN || MODE == tpi::GEMM_TN;
};
// An MN-major operand tile is stored as 64-element (128-byte) MN blocks of
// BK = 64 swizzled K rows each, MN_BLOCK_BYTES apart.
constexpr int MN_BLOCK_BYTES = 64 * BK * 2;  // 8 KB

__device__ __forceinline__ void decode_tile(const GemmParams& p, int tile, int& s, int& mb,
                                            int& nb) {
    const int per_shard = p.m_tiles * p.n_dec;
    s = tile / per_shard;
    const int r = tile - s * per_shard;
    const int group_size = p.group_m * p.n_dec;
    const int g = r / group_size;
    const int first_m = g * p.group_m;
    const int gm = min(p.m_tiles - first_m, p.group_m);
    const int rr = r - g * group_size;
    mb = first_m + rr % gm;
    nb = rr / gm;
    // Odd groups sweep the n-tiles backwards: a group starts on the weight
    // tiles the previous group ended on, which are still in L2.
    if (g & 1) nb = p.n_dec - 1 - nb;
}

// GEMM_MLP unit u of a cluster: colwise units first (all m-blocks of one
// n-tile pair, then the next pair: the first H columns of every m-block
// are done first), then the rowwise units of each m-block, piece-major (the
// first piece reads the first H columns).  A unit is two adjacent n-tiles of one m-block; pair pc
// of the cluster takes n-tile 2 n + pc (past the matrix when the count is
// odd: loads read zeros, stores are skipped).
__device__ __forceinline__ void decode_mlp(const GemmParams& p, int u, int pc, bool& row, int& mb, int& nb,
                                           int& piece) {
    if (u < p.mlp_col_units) {
        row = false;
        const int nbc = u / p.m_tiles;
        mb = u - nbc * p.m_tiles;
        nb = 2 * nbc + pc;
        piece = 0;
        return;
    }
    const int nrow2 = (p.mlp_row_n_tiles + 1) >> 1;
    const int r = u - p.mlp_col_units;
    const int per_m = nrow2 * p.mlp_pieces;
    row = true;
    mb = r / per_m;
    const int rem = r - mb * per_m;
    piece = rem / nrow2;
    nb = 2 * (rem - piece * nrow2) + pc;
}

// First KV head held by shard i (k/t own heads when k >= t, else a replica
// of head i*k/t): "셀프 어텐션", GQA KV heads replicated when fewer than t.
__device__ __forceinline__ int kv_first(int k, int t, int i) {
    return (k >= t) ? i * (k / t) : (i * k) / t;
}

// 2^x and 1/x on the SFU (PTX ex2.approx.ftz / rcp.approx.ftz: relative
// error about 2^-22 and 1 ulp; 2^-inf = +0, 1/inf = +0).  The activations
// below are rounded to bf16 (8 significant bits) right after, so these are
// far below the output's resolution.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// Upper tail of the standard normal CDF: q(u) = (1 - erf(|u| / sqrt2)) / 2,
// with erf from Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26: for y >= 0, erf(y) = 1 - t (a1 + t (a2 + t (a3 + t (a4 +
// t a5)))) exp(-y^2) + e(y), t = 1 / (1 + p y), |e(y)| <= 1.5e-7.  So Phi(u)
// = 1 - q for u >= 0 and q for u < 0, and e = exp(-u^2 / 2) is returned
// for the GeLU derivative's density term.
__device__ __forceinline__ float normal_tail(float u, float& e) {
    constexpr float P = 0.3275911f * 0.70710678118654752f;  // p / sqrt2 (y = |u| / sqrt2)
    constexpr float A1 = 0.5f * 0.254829592f, A2 = 0.5f * -0.284496736f, A3 = 0.5f * 1.421413741f;
    constexpr float A4 = 0.5f * -1.453152027f, A5 = 0.5f * 1.061405429f;
    const float t = rcp_approx(fmaf(P, fabsf(u), 1.0f));
    e = ex2_approx(u * u * (-0.5f * kLog2e));
    return t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, A5, A4), A3), A2), A1) * e;
}

// GeLU, exact (erf) form: u Phi(u).
__device__ __forceinline__ float gelu_erf(float u) {
    float e;
    const float q = normal_tail(u, e);
    return u * (u >= 0.0f ? 1.0f - q : q);
}

// GeLU, tanh form: u (1 + tanh(z)) / 2 with z = sqrt(2/pi) (u + 0.044715
// u^3), through (1 + tanh(z)) / 2 = 1 / (1 + exp(-2 z)).
constexpr float kGeluC = 0.79788456080286536f, kGeluA = 0.044715f;
__device__ __forceinline__ float gelu_tanh_sigma(float u) {
    const float z = kGeluC * u * fmaf(kGeluA * u, u, 1.0f);
    return rcp_approx(1.0f + ex2_approx(-2.0f * kLog2e * z));
}

// SiLU(u) = u sigmoid(u) = u / (1 + exp(-u)).
__device__ __forceinline__ float silu(float u) { return u * rcp_approx(1.0f + ex2_approx(-kLog2e * u)); }

template <int ACT>
__device__ __forceinline__ float act_apply(float v) {
    if (ACT == TP_ACT_GELU_ERF) return gelu_erf(v);
    if (ACT == TP_ACT_GELU_TANH) return v * gelu_tanh_sigma(v);
    return v;
}

// act_apply of two values with packed FP32 arithmetic (GeLU: the same
// operations in the same order as gelu_erf and gelu_tanh_sigma, each lane
// rounded as the scalar instruction, so the results are the same bits).
template <int ACT>
__device__ __forceinline__ void act_apply2(float u0, float u1, float& h0, float& h1) {
    if (ACT == TP_ACT_GELU_ERF) {
        constexpr float P = 0.3275911f * 0.70710678118654752f;
        constexpr float A1 = 0.5f * 0.254829592f, A2 = 0.5f * -0.284496736f, A3 = 0.5f * 1.421413741f;
        constexpr float A4 = 0.5f * -1.453152027f, A5 = 0.5f * 1.061405429f;
        const uint64_t U = f2_pack(u0, u1);
        float d0, d1, s0, s1;
        f2_unpack(f2_fma(f2_pack(P, P), f2_pack(fabsf(u0), fabsf(u1)), f2_pack(1.0f, 1.0f)), d0, d1);
        f2_unpack(f2_mul(f2_mul(U, U), f2_pack(-0.5f * kLog2e, -0.5f * kLog2e)), s0, s1);
        const uint64_t T = f2_pack(rcp_approx(d0), rcp_approx(d1));
        const uint64_t E = f2_pack(ex2_approx(s0), ex2_approx(s1));
        uint64_t poly = f2_fma(T, f2_pack(A5, A5), f2_pack(A4, A4));
        poly = f2_fma(T, poly, f2_pack(A3, A3));
        poly = f2_fma(T, poly, f2_pack(A2, A2));
        poly = f2_fma(T, poly, f2_pack(A1, A1));
        float q0, q1;
        f2_unpack(f2_mul(f2_mul(T, poly), E), q0, q1);
        f2_unpack(f2_mul(U, f2_pack(u0 >= 0.0f ? 1.0f - q0 : q0, u1 >= 0.0f ? 1.0f - q1 : q1)), h0, h1);
    } else {
        h0 = act_apply<ACT>(u0);
        h1 = act_apply<ACT>(u1);
    }
}

template <int ACT>
__device__ __forceinline__ void act_backward(float u, float g, float dh, float& du, float& dg,
                                             float& hv) {
    dg = 0.0f;
    if (ACT == TP_ACT_SWIGLU) {
        const float s = rcp_approx(1.0f + ex2_approx(-kLog2e * u));  // sigmoid(u)
        const float su = u * s;
        hv = su * g;
        dg = dh * su;
        du = dh * g * (s * (1.0f + u * (1.0f - s)));
    } else if (ACT == TP_ACT_GELU_ERF) {
        float e;  // exp(-u^2 / 2)
        const float q = normal_tail(u, e);
        const float cdf = u >= 0.0f ? 1.0f - q : q;
        const float pdf = 0.39894228040143268f * e;  // 1 / sqrt(2 pi)
        hv = u * cdf;
        du = dh * (cdf + u * pdf);
    } else if (ACT == TP_ACT_GELU_TANH) {
        // sigma = (1 + tanh z) / 2; d/du [u sigma] = sigma + u 2 sigma (1 -
        // sigma) dz/du, dz/du = c (1 + 3 a u^2).
        const float sg = gelu_tanh_sigma(u);
        hv = u * sg;
        du = dh * (sg + u * 2.0f * sg * (1.0f - sg) * kGeluC * fmaf(3.0f * kGeluA * u, u, 1.0f));
    } else {
        hv = u;
        du = dh;
    }
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// U (and G) of one 32-column chunk of an epilogue row (BWD_ACT): four
// 16-byte loads each, zeros outside the matrix.
__device__ __forceinline__ void load_ug_chunk(const GemmParams& p, const __nv_bfloat16* ug, bool row_ok,
                                              bool glu, int col0, uint4 (&u)[4], uint4 (&g)[4]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int col = col0 + e * 8;
        const bool ok = row_ok && col < p.N;
        u[e] = ok ? ld_nc_v4(ug + col) : make_uint4(0, 0, 0, 0);
        g[e] = (ok && glu) ? ld_nc_v4(ug + p.n_half + col) : make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ void unpack8(uint4 w, float (&x)[8]) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(a[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}

__device__ __forceinline__ void st_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4*>(ptr) = make_uint4(a, b, c, d);
}

// Bounded wait used only while draining after an abort (ignores the flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 200000000ull) break;  // 200 ms
    }
}

// Tensor map and first row of each 64-row B box of an output tile.  Depends
// only on the tile, so the producer computes it once per tile, not per
// k-block (the QKV segment arithmetic would otherwise stall the TMA issue).
// Tensor map and first row of the 64-row B boxes [first, first + N) of an
// output tile (a CTA of a pair loads half of the tile's four boxes).
// Depends only on the tile, so the producer computes it once per tile, not
// per k-block (the QKV segment arithmetic would otherwise stall TMA issue).
template <int MODE, int N>
__device__ __forceinline__ void b_boxes(const GemmParams& p, int nb, int first,
                                        const CUtensorMap* (&map)[N], int (&row)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const int c = first + i;
        map[i] = &p.mapB[0];
        if (MODE == tpi::GEMM_COL_SWIGLU) {
            // rows [0,128) of the tile: W1; rows [128,256): W3, both for
            // output columns nb*128 .. nb*128+127.
            map[i] = (c >> 1) ? &p.mapB[1] : &p.mapB[0];
            row[i] = nb * (BN / 2) + (c & 1) * B_CHUNK_ROWS;
        } else if (MODE == tpi::GEMM_COL_QKV) {
            const int col = nb * BN + c * B_CHUNK_ROWS;
            if (col >= p.N) {
                row[i] = p.b_rows0;  // wholly out of range: zeros
            } else {
                const int sh = col / p.qkv_ws;
                const int l = col - sh * p.qkv_ws;
                if (l < p.qkv_qw) {
                    row[i] = sh * p.qkv_qw + l;
                } else {
                    const int kv0 = kv_first(p.kv_heads, p.tp, sh) * p.head_dim;
                    const int l2 = l - p.qkv_qw;
                    if (l2 < p.qkv_kvw) {
                        map[i] = &p.mapB[1];
                        row[i] = kv0 + l2;
                    } else {
                        map[i] = &p.mapB[2];
                        row[i] = kv0 + (l2 - p.qkv_kvw);
                    }
                }
            }
        } else if (MODE == tpi::GEMM_COL_PACKED) {
            // Output column -> shard, then the packed block it falls in.
            const int col = nb * BN + c * B_CHUNK_ROWS;
            if (col >= p.N) {
                row[i] = p.b_rows0;  // wholly out of range: zeros
            } else {
                const int sh = col / p.pk_ws;
                int l = col - sh * p.pk_ws, b = 0;
                while (b + 1 < p.pk_nb && l >= p.pk_w[b]) {
                    l -= p.pk_w[b];
                    ++b;
                }
                row[i] = p.pk_off[b] + sh * p.pk_w[b] + l;
            }
        } else {
            row[i] = nb * BN + c * B_CHUNK_ROWS;
        }
    }
}

template <int MODE, int CG, int BNT>
__device__ __forceinline__ void producer_loop(const GemmParams& p, uint32_t base, uint32_t bar0,
                                              uint32_t rank, volatile int* abort_flag) {
    using C = Cfg<MODE, CG, BNT>;
    constexpr bool ROW = (MODE == tpi::GEMM_ROW_FUSED || MODE == tpi::GEMM_ROW_PARTIAL);
    constexpr int CL = cluster_ctas<MODE, CG, BNT>();
    // Clusters of two pairs (MC): pair pc = rank / 2 takes n-tile 2 n + pc of
    // a unit; each CTA loads 64 of its 128 A rows (the half pc) into its own
    // stage and, by multicast, into the same-rank CTA of the other pair.
    constexpr bool MC = CL == 2 * CG;
    const int pc = MC ? static_cast<int>(rank >> 1) : 0;
    const uint32_t prank = MC ? (rank & 1u) : rank;
    const uint16_t a_mask = static_cast<uint16_t>((1u << prank) | (1u << (prank + 2)));
    constexpr uint32_t A_HALF = A_BYTES / 2;
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, last_parity = 0;
    bool ok = true;
    const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    for (int tile = cid; ok && tile < p.num_tiles; tile += ncl) {
        int s_grid, mb, nb;
        decode_tile(p, tile, s_grid, mb, nb);
        if (MC) nb = 2 * nb + pc;  // past the matrix when n_tiles is odd: B reads zeros
        const int arow = mb * C::TILE_M + static_cast<int>(prank) * BM + (MC ? pc * (BM / 2) : 0);
        const CUtensorMap* bmap[C::CHUNKS];
        int brow[C::CHUNKS];
        if (!ROW) b_boxes<MODE, C::CHUNKS>(p, nb, static_cast<int>(prank) * C::CHUNKS, bmap, brow);
        for (int ks = 0; ok && ks < p.k_shards; ++ks) {
            const int shard = (MODE == tpi::GEMM_ROW_PARTIAL) ? s_grid : ks;
            for (int kb = 0; kb < p.kb_per_shard; ++kb) {
                const uint32_t full = bar0 + 8 * stage, empty = bar0 + 8 * (C::STAGES + stage);
                // MC: both pairs have consumed this stage (each pair's MMA
                // commit arrives on every CTA's empty barrier).
                if (!mbar_wait(empty, phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                // The leader's full barrier counts the bytes of both CTAs.
                if (prank == 0) mbar_arrive_expect_tx(full, CG * C::STAGE_BYTES);
                const uint32_t full_l = (CG == 2) ? mapa_shared(full, rank & ~1u) : full;
                const uint32_t a_dst = base + stage * C::STAGE_BYTES;
                const uint32_t b_dst = a_dst + A_BYTES;
                const int kc = kb * BK;
#pragma unroll
                for (int c = -1; c < C::CHUNKS; ++c) {
                    const int cc = static_cast<int>(prank) * C::CHUNKS + c;  // B box of the tile
                    const uint32_t dst = c < 0 ? a_dst : b_dst + c * B_CHUNK_BYTES;
                    if (MC && c < 0) {
                        if (ROW) tma_load_3d_pair_mc(a_dst + pc * A_HALF, &p.mapA, full_l, kc, shard, arow, a_mask);
                        else tma_load_2d_pair_mc(a_dst + pc * A_HALF, &p.mapA, full_l, kc, arow, a_mask);
                    } else if (ROW) {
                        const CUtensorMap* map = c < 0 ? &p.mapA : &p.mapB[0];
                        const int r = c < 0 ? arow : nb * BNT + cc * B_CHUNK_ROWS;
                        if (CG == 2) tma_load_3d_pair(dst, map, full_l, kc, shard, r);
                        else tma_load_3d(dst, map, full_l, kc, shard, r);
                    } else if (c < 0 && Major<MODE>::A_MN) {
                        // [K][M] source: the CTA's 128 A rows as two 64-wide blocks.
#pragma unroll
                        for (int e = 0; e < BM / 64; ++e) {
                            if (CG == 2)
                                tma_load_2d_pair(dst + e * MN_BLOCK_BYTES, &p.mapA, full_l, arow + 64 * e, kc);
                            else tma_load_2d(dst + e * MN_BLOCK_BYTES, &p.mapA, full_l, arow + 64 * e, kc);
                        }
                    } else if (c >= 0 && Major<MODE>::B_MN) {
                        // [K][N] source; GEMM_NN takes K rows >= k_split from B1
                        // and >= k_split2 from B2.
                        const bool hi2 = MODE == tpi::GEMM_NN && kc >= p.k_split2;
                        const bool hi = MODE == tpi::GEMM_NN && kc >= p.k_split;
                        const CUtensorMap* map = hi2 ? &p.mapB[2] : (hi ? &p.mapB[1] : &p.mapB[0]);
                        const int kk = hi2 ? kc - p.k_split2 : (hi ? kc - p.k_split : kc);
                        if (CG == 2) tma_load_2d_pair(dst, map, full_l, brow[c < 0 ? 0 : c], kk);
                        else tma_load_2d(dst, map, full_l, brow[c < 0 ? 0 : c], kk);
                    } else {
                        const CUtensorMap* map = c < 0 ? &p.mapA : bmap[c < 0 ? 0 : c];
                        const int r = c < 0 ? arow : brow[c < 0 ? 0 : c];
                        if (CG == 2) tma_load_2d_pair(dst, map, full_l, kc, r);
                        else tma_load_2d(dst, map, full_l, kc, r);
                    }
                }
                issued_mask |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
    if (!ok && prank == 0) {
        // Let every copy of the pair land before the CTAs exit (the leader's
        // full barriers count both CTAs' bytes).
        for (int s = 0; s < C::STAGES; ++s)
            if (issued_mask & (1u << s)) drain_wait(bar0 + 8 * s, (last_parity >> s) & 1u);
    }
}

// Producer of the fused MLP.  A rowwise unit first waits (bounded) until
// both CTAs of every colwise tile holding its H columns have stored them;
// its loads then read H through the async proxy.
template <int CG>
__device__ __forceinline__ void mlp_producer_loop(const GemmParams& p, uint32_t base, uint32_t bar0,
                                                  uint32_t rank, volatile int* abort_flag) {
    using C = Cfg<tpi::GEMM_MLP, CG, BN>;
    constexpr int CL = cluster_ctas<tpi::GEMM_MLP, CG>();
    static_assert(CG == 2 && CL == 4, "the fused MLP runs clusters of two CTA pairs");
    // rank: 0..3 in the cluster; pair pc = rank / 2, prank = rank % 2 in it.
    const int pc = static_cast<int>(rank >> 1), prank = static_cast<int>(rank & 1u);
    // Each CTA loads 64 of its 128 A rows (the half pc) into both pairs: the
    // CTAs of the same rank in the two pairs hold the same A rows.
    const uint16_t a_mask = static_cast<uint16_t>((1u << prank) | (1u << (prank + 2)));
    constexpr uint32_t A_HALF = A_BYTES / 2;
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, last_parity = 0;
    bool ok = true;
    const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    for (int u = cid; ok && u < p.num_tiles; u += ncl) {
        bool row;
        int mb, nb, piece;
        decode_mlp(p, u, pc, row, mb, nb, piece);
        const int arow = mb * C::TILE_M + prank * BM + pc * (BM / 2);
        int s0 = 0, ns = 1, nkb = p.kb_per_shard;
        if (row) {
            s0 = piece * p.mlp_spp;
            ns = p.mlp_spp;
            nkb = p.mlp_kb_row;
            // One counter per (m-block, piece): the CTAs of every colwise tile
            // overlapping the piece's H columns count themselves in it.
            // (Polling one counter per tile in turn, each an L2 round trip,
            // saw the last store about 3 us late.)
            const long long c0 = static_cast<long long>(s0) * p.mlp_ks, c1 = c0 + ns * p.mlp_ks;
            const unsigned tiles = static_cast<unsigned>((c1 - 1) / BN - c0 / BN + 1);
            ok = flag_wait_geq(p.mlp_ready + mb * 8 + piece, CG * tiles, abort_flag, p.status, p.timeout_ns);
            if (!ok) break;
            fence_proxy_async_global();
        }
        // One k-loop per kind of unit, each issuing its loads without a
        // branch: with the colwise / rowwise choice inside the loop the
        // loads of a k-block arrived measurably later (a colwise unit's main
        // loop took 12.8 k cycles against 9.1 k).
        auto acquire = [&](uint32_t& full_l, uint32_t& a_dst) -> bool {
            const uint32_t full = bar0 + 8 * stage, empty = bar0 + 8 * (C::STAGES + stage);
            // Both pairs have consumed this stage (each pair's MMA commit
            // arrives on every CTA's empty barrier).
            if (!mbar_wait(empty, phase ^ 1u, abort_flag, p.status, p.timeout_ns)) return false;
            if (prank == 0) mbar_arrive_expect_tx(full, CG * C::STAGE_BYTES);
            full_l = mapa_shared(full, rank & ~1u);
            a_dst = base + stage * C::STAGE_BYTES;
            return true;
        };
        auto advance = [&]() {
            issued_mask |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        };
        if (!row) {
            for (int kb = 0; kb < nkb; ++kb) {
                uint32_t full_l, a_dst;
                if (!(ok = acquire(full_l, a_dst))) break;
                const int kc = kb * BK;
                tma_load_2d_pair_mc(a_dst + pc * A_HALF, &p.mapA, full_l, kc, arow, a_mask);
#pragma unroll
                for (int c = 0; c < C::CHUNKS; ++c)
                    tma_load_2d_pair(a_dst + A_BYTES + c * B_CHUNK_BYTES, &p.mapB[0], full_l, kc,
                                     nb * BN + (prank * C::CHUNKS + c) * B_CHUNK_ROWS);
                advance();
            }
        } else {
            for (int sh = s0; ok && sh < s0 + ns; ++sh) {
                for (int kb = 0; kb < nkb; ++kb) {
                    uint32_t full_l, a_dst;
                    if (!(ok = acquire(full_l, a_dst))) break;
                    const int kc = kb * BK;
                    tma_load_3d_pair_mc(a_dst + pc * A_HALF, &p.mapH, full_l, kc, sh, arow, a_mask);
#pragma unroll
                    for (int c = 0; c < C::CHUNKS; ++c)
                        tma_load_3d_pair(a_dst + A_BYTES + c * B_CHUNK_BYTES, &p.mapW2, full_l, kc, sh,
                                         nb * BN + (prank * C::CHUNKS + c) * B_CHUNK_ROWS);
                    advance();
                }
            }
        }
    }
    if (!ok && prank == 0) {
        for (int s = 0; s < C::STAGES; ++s)
            if (issued_mask & (1u << s)) drain_wait(bar0 + 8 * s, (last_parity >> s) & 1u);
    }
}

template <int MODE, int CG, int BNT>
__device__ __forceinline__ void mma_loop(const GemmParams& p, uint32_t base, uint32_t bar0,
                                         uint32_t tmem_base, volatile int* abort_flag, uint32_t rank) {
    constexpr int CL = cluster_ctas<MODE, CG, BNT>();
    // Commit masks (cluster ranks): the accumulator goes to this pair; a
    // freed stage to every CTA whose stage this pair's MMAs read (with
    // multicast A, all CTAs of the cluster); the drain to this CTA.
    const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (rank & ~1u));
    const uint16_t stage_mask = CL == 4 ? 0xF : pair_mask;
    const uint16_t self_mask = static_cast<uint16_t>(1u << rank);
    using C = Cfg<MODE, CG, BNT>;
    constexpr bool AMN = Major<MODE>::A_MN, BMN = Major<MODE>::B_MN;
    // Bits 15 / 16 of the instruction descriptor: A / B MN-major.
    constexpr uint32_t idesc =
        idesc_bf16_f32(BM * CG, BNT) | (AMN ? (1u << 15) : 0u) | (BMN ? (1u << 16) : 0u);
    // Per UMMA (K = 16): a K-major operand advances 32 bytes inside its
    // swizzle row (2 in descriptor units), an MN-major one 16 K rows of
    // 128 bytes (128 units).
    constexpr uint64_t a_step = AMN ? 128u : 2u, b_step = BMN ? 128u : 2u;
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    bool ok = true;
    const int kblocks = p.k_shards * p.kb_per_shard;
    const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    for (int tile = cid; ok && tile < p.num_tiles; tile += ncl) {
        const uint32_t tfull = bar0 + 8 * (2 * C::STAGES + acc);
        const uint32_t tempty = bar0 + 8 * (2 * C::STAGES + 2 + acc);
        if (!mbar_wait(tempty, acc_phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BNT;
        int nkb = kblocks;
        if constexpr (MODE == tpi::GEMM_MLP)
            nkb = tile < p.mlp_col_units ? p.kb_per_shard : p.mlp_spp * p.mlp_kb_row;
        for (int kb = 0; kb < nkb; ++kb) {
            const uint32_t full = bar0 + 8 * stage, empty = bar0 + 8 * (C::STAGES + stage);
            if (!mbar_wait(full, phase, abort_flag, p.status, p.timeout_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a_addr = base + stage * C::STAGE_BYTES;
            const uint64_t adesc = AMN ? sdesc_sw128_mn(a_addr, MN_BLOCK_BYTES, 1024)
                                       : sdesc_sw128(a_addr);
            const uint64_t bdesc = BMN ? sdesc_sw128_mn(a_addr + A_BYTES, MN_BLOCK_BYTES, 1024)
                                       : sdesc_sw128(a_addr + A_BYTES);
#pragma unroll
            for (int j = 0; j < BK / UK; ++j) {
                const uint32_t accum = (kb > 0 || j > 0) ? 1u : 0u;
                const uint64_t ad = adesc + a_step * j, bd = bdesc + b_step * j;
                if (CG == 2) umma_bf16_pair(d_tmem, ad, bd, idesc, accum);
                else umma_bf16(d_tmem, ad, bd, idesc, accum);
            }
            // Frees the smem stage (of both CTAs) when these UMMAs finish.
            if (CG == 2) umma_commit_pair(empty, stage_mask);
            else umma_commit(empty);
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        // Accumulator ready for the epilogue (of both CTAs).
        if (CG == 2) umma_commit_pair(tfull, pair_mask);
        else umma_commit(tfull);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
        // No UMMA may still write TMEM when it is freed.
        const uint32_t drain = bar0 + 8 * (2 * C::STAGES + 4);
        if (CG == 2) umma_commit_pair(drain, self_mask);
        else umma_commit(drain);
        drain_wait(drain, 0);
    }
}

// Epilogue of GEMM_BWD_ACT for one warp's CPW 32-column chunks of a tile:
// dH from TMEM, U (and G) from the prefetch ring (chunks c and c + 1 already
// requested; each chunk requests c + 2).  dU, dG and H of a chunk go to the
// warp's three 32 x 32 boxes in shared memory, stored in the 64-byte swizzle
// (16-byte piece j of row r at r * 64 + (j ^ ((r >> 1) & 3)) * 16, which
// also keeps the 32 rows' writes free of bank conflicts), and leave by TMA
// stores (whole rows per request; rows and columns outside the matrices are
// clipped by the tensor maps).  row0: first global row of the warp's box.
template <int ACT, int CPW>
__device__ __forceinline__ void bwd_act_tile(const GemmParams& p, const __nv_bfloat16* ug, bool row_ok,
                                             int row0, int nb, int cb, uint32_t t0, uint32_t sbuf,
                                             uint4 (&n1u)[4], uint4 (&n1g)[4], uint4 (&n2u)[4],
                                             uint4 (&n2g)[4]) {
    constexpr bool glu = ACT == TP_ACT_SWIGLU;
    const int lane = threadIdx.x & 31;
    const bool want_h = p.out2 != nullptr;
    const bool box_ok = row0 < p.M;  // warp-uniform
    const uint32_t srow = sbuf + static_cast<uint32_t>(lane) * (EPI_BOX * 2);
    const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
    uint32_t r[32];
#pragma unroll 1
    for (int cc = 0; cc < CPW; ++cc) {  // kept rolled: instruction-cache footprint
        const int c = cb + cc;
        const int col0 = nb * BN + c * 32;
        if (col0 >= p.N) break;  // warp-uniform
        uint4 cu[4], cg[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            cu[e] = n1u[e];
            cg[e] = n1g[e];
            n1u[e] = n2u[e];
            n1g[e] = n2g[e];
        }
        // The loads of chunk c + 2 are in flight during this chunk's math.
        if (cc + 2 < CPW) load_ug_chunk(p, ug, row_ok, glu, col0 + 64, n2u, n2g);
        __syncwarp();
        tmem_ld32(t0 + c * 32, r);  // dH
        tmem_ld_wait();
        // The boxes may be rewritten once the previous chunk's stores have
        // read them.
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float uu[8], gg[8];
            unpack8(cu[g], uu);
            unpack8(cg[g], gg);
            uint32_t wu[4], wg[4], wh[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float du0, dg0, h0, du1, dg1, h1;
                act_backward<ACT>(uu[2 * e], gg[2 * e], __uint_as_float(r[g * 8 + 2 * e]), du0, dg0, h0);
                act_backward<ACT>(uu[2 * e + 1], gg[2 * e + 1], __uint_as_float(r[g * 8 + 2 * e + 1]),
                                  du1, dg1, h1);
                wu[e] = pack_bf16x2(du0, du1);
                wg[e] = pack_bf16x2(dg0, dg1);
                wh[e] = pack_bf16x2(h0, h1);
            }
            const uint32_t off = (static_cast<uint32_t>(g) ^ sw) << 4;
            st_shared_v4(srow + off, wu[0], wu[1], wu[2], wu[3]);
            if (glu) st_shared_v4(srow + EPI_BOX_BYTES + off, wg[0], wg[1], wg[2], wg[3]);
            if (want_h) st_shared_v4(srow + 2 * EPI_BOX_BYTES + off, wh[0], wh[1], wh[2], wh[3]);
        }
        fence_proxy_async_smem();  // visible to the TMA engine
        __syncwarp();
        if (lane == 0 && box_ok) {
            tma_store_2d(&p.mapO[0], sbuf, col0, row0);
            if (glu) tma_store_2d(&p.mapO[1], sbuf + EPI_BOX_BYTES, col0, row0);
            if (want_h) tma_store_2d(&p.mapO[2], sbuf + 2 * EPI_BOX_BYTES, col0, row0);
            bulk_commit_group();
        }
    }
}

// GEMM_COL_ACT epilogue through shared memory: per 32-column chunk the warp
// writes its 32 rows x 32 columns as bf16 into one of its two boxes (64-byte
// swizzle: 16-byte piece g of row l at l * 64 + (g ^ ((l / 2) % 4)) * 16)
// and lane 0 issues one TMA store of the box; rows and columns past the
// output are clipped by the map.  A box is rewritten once the store two
// chunks back has read it.  row0: first global row of the warp's box.
template <int ACT, int CPW, int BNT>
__device__ __forceinline__ void col_act_tile_staged(const GemmParams& p, uint32_t t0, int cb, int nb, int row,
                                                    bool row_ok, int row0, float rs, uint32_t sbuf) {
    const int lane = threadIdx.x & 31;
    const bool box_ok = row0 < p.M;  // warp-uniform
    const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
    const uint64_t rs2 = f2_pack(rs, rs);
    uint32_t r[32];
#pragma unroll 1
    for (int c = cb; c < cb + CPW; ++c) {
        const int col0 = nb * BNT + c * 32;
        if (col0 >= p.N) break;  // warp-uniform
        __syncwarp();
        tmem_ld32(t0 + c * 32, r);
        tmem_ld_wait();
        const uint32_t box = sbuf + static_cast<uint32_t>(c & 1) * EPI_BOX_BYTES;
        const uint32_t srow = box + static_cast<uint32_t>(lane) * 64;
        if (lane == 0) bulk_wait_group_read1();  // this box's previous store has read it
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                f2_unpack(f2_mul(f2_pack(__uint_as_float(r[g * 8 + 2 * e]), __uint_as_float(r[g * 8 + 2 * e + 1])), rs2),
                          v[2 * e], v[2 * e + 1]);
            if (p.aux_out && row_ok && col0 + g * 8 < p.N)  // pre-activations for the backward pass
                st_v4(p.aux_out + static_cast<long long>(row) * p.ldaux + col0 + g * 8, pack_bf16x2(v[0], v[1]),
                      pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float h0, h1;
                act_apply2<ACT>(v[2 * e], v[2 * e + 1], h0, h1);
                w[e] = pack_bf16x2(h0, h1);
            }
            st_shared_v4(srow + ((static_cast<uint32_t>(g) ^ sw) << 4), w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();  // visible to the TMA engine
        __syncwarp();
        if (lane == 0 && box_ok) {
            tma_store_2d(&p.mapO[0], box, col0, row0);
            bulk_commit_group();
        }
    }
}

// Epilogue of the column- and row-parallel forward modes for one warp's CPW
// 32-column chunks of a tile (row: this thread's global row; rs: the folded
// RMSNorm scale of colwise rows; ssq accumulates the squares of the stored
// values when the rowwise GEMM feeds the next norm).
template <int MODE, int ACT, int CPW, int BNT>
__device__ __forceinline__ void std_tile(const GemmParams& p, uint32_t t0, int cb, int nb, int s_grid, int row,
                                         bool row_ok, float rs, float& ssq) {
    uint32_t r[32];
#pragma unroll 1
    for (int c = cb; c < cb + CPW; ++c) {
        const int col0 = nb * BNT + c * 32;
        if (col0 >= p.N) break;  // warp-uniform
        __syncwarp();
        tmem_ld32(t0 + c * 32, r);
        tmem_ld_wait();
        if (!row_ok) {
        } else if (MODE == tpi::GEMM_ROW_PARTIAL && p.out_f32) {
            float* out = reinterpret_cast<float*>(p.out) + s_grid * p.shard_stride +
                         static_cast<long long>(row) * p.ldo;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const int col = col0 + g * 4;
                if (col < p.N)
                    st_v4(out + col, r[g * 4], r[g * 4 + 1], r[g * 4 + 2], r[g * 4 + 3]);
            }
        } else {
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
            if (MODE == tpi::GEMM_ROW_PARTIAL) out += s_grid * p.shard_stride;
            // Output (and residual) row: the token's row in the sequence-split
            // layout when the layer is sequence parallel.
            long long orow = row;
            if (MODE == tpi::GEMM_ROW_FUSED && p.sp_t > 0) {
                const long long w = p.sp_seq / p.sp_t;
                const long long b = row / p.sp_seq, pos = row - b * p.sp_seq;
                orow = ((pos / w) * p.sp_batch + b) * w + pos % w;
            }
            out += orow * p.ldo;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int col = col0 + g * 8;
                if (col >= p.N) continue;
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(r[g * 8 + e]);
                if (MODE == tpi::GEMM_COL_ACT || MODE == tpi::GEMM_COL_QKV ||
                    MODE == tpi::GEMM_COL_PACKED) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] *= rs;
                }
                if (MODE == tpi::GEMM_COL_ACT) {
                    if (p.aux_out)  // pre-activations for the backward pass
                        st_v4(p.aux_out + static_cast<long long>(row) * p.ldaux + col,
                              pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                              pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = act_apply<ACT>(v[e]);
                }
                if (MODE == tpi::GEMM_ROW_FUSED) {
                    if (p.bias) {
                        const uint4 b = *reinterpret_cast<const uint4*>(p.bias + col);
                        const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_bf16x2(bw[e]);
                            v[2 * e] += f.x;
                            v[2 * e + 1] += f.y;
                        }
                    }
                    if (p.residual) {
                        const uint4 rr = *reinterpret_cast<const uint4*>(p.residual + orow * p.ldr + col);
                        const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_bf16x2(rw[e]);
                            v[2 * e] += f.x;
                            v[2 * e + 1] += f.y;
                        }
                    }
                }
                const uint32_t w0 = pack_bf16x2(v[0], v[1]), w1 = pack_bf16x2(v[2], v[3]);
                const uint32_t w2 = pack_bf16x2(v[4], v[5]), w3 = pack_bf16x2(v[6], v[7]);
                st_v4(out + col, w0, w1, w2, w3);
                if (MODE == tpi::GEMM_ROW_FUSED && p.ss_out) {
                    // The next norm reads the stored (bf16) values.
                    const uint32_t ws[4] = {w0, w1, w2, w3};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = unpack_bf16x2(ws[e]);
                        ssq = fmaf(f.x, f.x, fmaf(f.y, f.y, ssq));
                    }
                }
            }
        }
        // The row's sum of squares over each 128-column slice goes out once,
        // when the slice's last chunk is done.
        if (MODE == tpi::GEMM_ROW_FUSED && p.ss_out && ((c & 3) == 3 || col0 + 32 >= p.N || c + 1 == cb + CPW)) {
            const int slice = col0 >> 7;
            if (row_ok) p.ss_out[static_cast<long long>(slice) * p.M + row] = ssq;
            ssq = 0.0f;
        }
    }
}

// Epilogue of the fused MLP: 8 warps, two per TMEM lane quadrant, each on
// 128 of the tile's 256 columns (four 32-column chunks).  The accumulator
// arrives one row per thread (TMEM lane = row).  Global memory is reached
// only through TMA: each warp owns two 2 KB boxes in shared memory (32 rows
// x 64 bytes, 64-byte swizzle: 16-byte piece j of row r at r * 64 + (j ^
// ((r / 2) % 4)) * 16, which keeps the row-per-thread accesses free of
// bank conflicts), used in turn, each with an mbarrier for loads into it.
//  - colwise unit: act(accumulator) -> bf16 H by TMA stores; once the
//    CTA's 8 warps have seen their stores complete, one thread counts the
//    CTA's half of the tile in mlp_ready, once for each K piece whose H
//    columns the tile overlaps.
//  - rowwise unit of a lower piece (piece < pieces - 1): its fp32 partial
//    goes out by TMA stores, then the CTA counts itself in mlp_pdone.
//  - rowwise unit of the last piece: waits (bounded) until the lower
//    pieces of its tile have stored their partials, loads them by TMA and
//    sums P_0 + ... + P_(pieces-2) + its own accumulator in that order (so
//    the result does not depend on which piece finished first), adds bias
//    and residual, and stores bf16 Z.
// The 8 warps meet on hardware barrier 1 (bar.sync over 256 threads).
constexpr uint32_t kMlpEpiBar = 1;

// This thread's 64-byte row (16 words) into / out of a box.
__device__ __forceinline__ void box_put_row(uint32_t box, int lane, const uint32_t* w) {
    const uint32_t srow = box + static_cast<uint32_t>(lane) * 64, sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        st_shared_v4(srow + ((static_cast<uint32_t>(j) ^ sw) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}
__device__ __forceinline__ void box_get_row(uint32_t box, int lane, uint32_t* w) {
    const uint32_t srow = box + static_cast<uint32_t>(lane) * 64, sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 v = ld_shared_v4(srow + ((static_cast<uint32_t>(j) ^ sw) << 4));
        w[4 * j] = v.x;
        w[4 * j + 1] = v.y;
        w[4 * j + 2] = v.z;
        w[4 * j + 3] = v.w;
    }
}

template <int ACT>
__device__ __forceinline__ void mlp_act_pack(const uint32_t (&r)[32], uint32_t (&w)[16]) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        float h0, h1;
        act_apply2<ACT>(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]), h0, h1);
        w[e] = pack_bf16x2(h0, h1);
    }
}

// The warp's two boxes, used in turn.  A box is handed out once the bulk
// store that last read it has done so: when the newest store group read
// this box, all groups must have been read; otherwise the newest group read
// the other box and may still be pending.  All lanes track the same state.
struct MlpBoxes {
    uint32_t base, bars, phase, use, newest;  // newest: box of the newest store group (2: none)
    __device__ __forceinline__ uint32_t next(int lane, uint32_t& bar) {
        const uint32_t k = use & 1u;
        ++use;
        if (lane == 0) {
            if (newest == k) bulk_wait_group_read0();
            else bulk_wait_group_read1();
        }
        __syncwarp();
        bar = bars + 8 * k;
        return base + k * EPI_BOX_BYTES;
    }
    // After a bulk store (one commit group) from the box last handed out.
    __device__ __forceinline__ void stored() { newest = (use - 1) & 1u; }
    // Wait for the TMA load into the box whose barrier is `bar`.
    __device__ __forceinline__ bool wait_load(uint32_t bar, volatile int* abort_flag, const GemmParams& p) {
        const uint32_t k = (bar - bars) >> 3;
        const bool ok = mbar_wait(bar, (phase >> k) & 1u, abort_flag, p.status, p.timeout_ns);
        phase ^= 1u << k;
        return ok;
    }
};

template <int CG>
__device__ __forceinline__ void mlp_epilogue_loop(const GemmParams& p, uint32_t bar0, uint32_t epi0, uint32_t tmem_base,
                                                  uint32_t rank, volatile int* abort_flag) {
    using C = Cfg<tpi::GEMM_MLP, CG, BN>;
    constexpr int CL = cluster_ctas<tpi::GEMM_MLP, CG>();
    const int pc = static_cast<int>(rank >> 1), prank = static_cast<int>(rank & 1u);
    constexpr int EPI_WARPS = epi_warps<tpi::GEMM_MLP>();
    constexpr uint32_t EPI_THREADS = 32 * EPI_WARPS;
    constexpr int CPW = (BN / 32) / (EPI_WARPS / 4);  // 32-column chunks per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int cb = ((warp - 2) >> 2) * CPW;
    const bool leader = warp == 2 && lane == 0;
    MlpBoxes bx{epi0 + static_cast<uint32_t>(warp - 2) * 2 * EPI_BOX_BYTES,
                bar0 + 8 * (2 * C::STAGES + 5) + 16 + 16 * static_cast<uint32_t>(warp - 2), 0u, 0u, 2u};
    uint32_t acc = 0, acc_phase = 0;
    const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    for (int u = cid; u < p.num_tiles; u += ncl) {
        bool rowu;
        int mb, nb, piece;
        decode_mlp(p, u, pc, rowu, mb, nb, piece);
        const uint32_t tfull = bar0 + 8 * (2 * C::STAGES + acc);
        const uint32_t tempty = bar0 + 8 * (2 * C::STAGES + 2 + acc);
        const int row0 = mb * C::TILE_M + prank * BM + q * 32;  // the warp's first row
        const bool box_ok = row0 < p.M;  // warp-uniform
        const bool got = mbar_wait(tfull, acc_phase, abort_flag, p.status, p.timeout_ns);
        // Every epilogue warp takes the same branch, so none is left waiting
        // at a barrier below when another has given up.
        if (!named_bar_and(kMlpEpiBar, EPI_THREADS, got)) break;
        tc_fence_after();
        const uint32_t t0 = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
        const int tile_ctr = (mb * p.mlp_row_n_tiles + nb) * 2 + prank;
        const bool tile_ok = nb < (rowu ? p.mlp_row_n_tiles : p.n_tiles);  // not past the matrix
        uint32_t r[32];
        if (!rowu) {
#pragma unroll 1
            for (int c = cb; c < cb + CPW; ++c) {
                const int col0 = nb * BN + c * 32;
                if (col0 >= p.N) break;  // warp-uniform
                __syncwarp();
                tmem_ld32(t0 + c * 32, r);
                tmem_ld_wait();
                uint32_t w[16];
                switch (p.act) {
                    case TP_ACT_GELU_ERF: mlp_act_pack<TP_ACT_GELU_ERF>(r, w); break;
                    case TP_ACT_GELU_TANH: mlp_act_pack<TP_ACT_GELU_TANH>(r, w); break;
                    default: mlp_act_pack<TP_ACT_NONE>(r, w); break;
                }
                uint32_t bar;
                const uint32_t box = bx.next(lane, bar);
                box_put_row(box, lane, w);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && box_ok) {
                    tma_store_2d(&p.mapHs, box, col0, row0);
                    bulk_commit_group();
                }
                if (box_ok) bx.stored();
            }
            if (lane == 0) bulk_wait_group0();  // this warp's H stores are in global memory
            __syncwarp();
            named_bar_sync(kMlpEpiBar, EPI_THREADS);
            if (leader && tile_ok) {
                fence_proxy_async_global();
                // Every piece whose H columns this tile overlaps.
                const long long pw = static_cast<long long>(p.mlp_spp) * p.mlp_ks;
                const int q0 = static_cast<int>(static_cast<long long>(nb) * BN / pw);
                const int q1 = static_cast<int>((min(static_cast<long long>(nb + 1) * BN, static_cast<long long>(p.N)) - 1) / pw);
                for (int q = q0; q <= q1; ++q) red_release_gpu_add(p.mlp_ready + mb * 8 + q, 1u);
            }
        } else if (piece < p.mlp_pieces - 1) {
#pragma unroll 1
            for (int c = cb; c < cb + CPW; ++c) {
                const int col0 = nb * BN + c * 32;
                if (col0 >= p.mlp_h) break;  // warp-uniform
                __syncwarp();
                tmem_ld32(t0 + c * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t bar;
                    const uint32_t box = bx.next(lane, bar);
                    box_put_row(box, lane, r + 16 * hf);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && box_ok) {
                        tma_store_3d(&p.mapPs, box, col0 + 16 * hf, row0, piece);
                        bulk_commit_group();
                    }
                    if (box_ok) bx.stored();
                }
            }
            if (lane == 0) bulk_wait_group0();
            __syncwarp();
            named_bar_sync(kMlpEpiBar, EPI_THREADS);
            if (leader && tile_ok) {
                fence_proxy_async_global();
                red_release_gpu_add(p.mlp_pdone + tile_ctr, 1u);
            }
        } else {
            bool ok = true;
            if (p.mlp_pieces > 1) {
                if (leader && tile_ok)
                    ok = flag_wait_geq(p.mlp_pdone + tile_ctr, static_cast<unsigned>(p.mlp_pieces - 1), abort_flag,
                                       p.status, p.timeout_ns);
                ok = named_bar_and(kMlpEpiBar, EPI_THREADS, ok);
                if (lane == 0) fence_proxy_async_global();  // the partials are read by TMA
            }
#pragma unroll 1
            for (int c = cb; ok && c < cb + CPW; ++c) {
                const int col0 = nb * BN + c * 32;
                if (col0 >= p.mlp_h) break;  // warp-uniform
                __syncwarp();
                tmem_ld32(t0 + c * 32, r);  // this piece's sum
                tmem_ld_wait();
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
                if (p.mlp_pieces > 1) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        float sum[16];
#pragma unroll 1
                        for (int j = 0; j < p.mlp_pieces - 1; ++j) {
                            uint32_t bar;
                            const uint32_t box = bx.next(lane, bar);
                            if (lane == 0) {
                                mbar_arrive_expect_tx(bar, EPI_BOX_BYTES);
                                tma_load_3d(box, &p.mapPs, bar, col0 + 16 * hf, row0, j);
                            }
                            ok = bx.wait_load(bar, abort_flag, p) && ok;
                            uint32_t w[16];
                            box_get_row(box, lane, w);
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                sum[e] = j == 0 ? __uint_as_float(w[e]) : sum[e] + __uint_as_float(w[e]);
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[16 * hf + e] = sum[e] + v[16 * hf + e];
                    }
                }
                if (p.bias) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (col0 + 8 * g >= p.mlp_h) continue;
                        const uint4 b = *reinterpret_cast<const uint4*>(p.bias + col0 + 8 * g);
                        const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_bf16x2(bw[e]);
                            v[8 * g + 2 * e] += f.x;
                            v[8 * g + 2 * e + 1] += f.y;
                        }
                    }
                }
                if (p.residual) {
                    uint32_t bar;
                    const uint32_t box = bx.next(lane, bar);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar, EPI_BOX_BYTES);
                        tma_load_2d(box, &p.mapRs, bar, col0, row0);
                    }
                    ok = bx.wait_load(bar, abort_flag, p) && ok;
                    uint32_t w[16];
                    box_get_row(box, lane, w);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float2 f = unpack_bf16x2(w[e]);
                        v[2 * e] += f.x;
                        v[2 * e + 1] += f.y;
                    }
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
                uint32_t bar;
                const uint32_t box = bx.next(lane, bar);
                box_put_row(box, lane, w);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && box_ok) {
                    tma_store_2d(&p.mapZs, box, col0, row0);
                    bulk_commit_group();
                }
                if (box_ok) bx.stored();
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_cluster(mapa_shared(tempty, rank & ~1u));
        }
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
    }
    // Every bulk store has completed before the CTA's shared memory goes.
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
}

template <int MODE, int CG, int BNT>
__device__ __forceinline__ void epilogue_loop(const GemmParams& p, uint32_t bar0, uint32_t epi0,
                                              uint32_t tmem_base, uint32_t rank, volatile int* abort_flag) {
    using C = Cfg<MODE, CG, BNT>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    constexpr int EPI_WARPS = epi_warps<MODE>();
    const int half = (warp - 2) >> 2;  // which half of the tile's columns (8 warps)
    constexpr int CPW = (BNT / 32) / (EPI_WARPS / 4);       // 32-column chunks per warp
    constexpr int CPW_GLU = (BN / 64) / (EPI_WARPS / 4);    // SwiGLU: output chunks per warp
    const int cb = half * CPW, cb_glu = half * CPW_GLU;
    uint32_t acc = 0, acc_phase = 0;
    constexpr int CL = cluster_ctas<MODE, CG, BNT>();
    constexpr bool MC = CL == 2 * CG;  // clusters of two pairs: pair pc takes n-tile 2 n + pc
    const int pc = MC ? static_cast<int>(rank >> 1) : 0;
    const uint32_t prank = MC ? (rank & 1u) : rank;
    const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    for (int tile = cid; tile < p.num_tiles; tile += ncl) {
        int s_grid, mb, nb;
        decode_tile(p, tile, s_grid, mb, nb);
        if (MC) nb = 2 * nb + pc;  // past the matrix when n_tiles is odd: the column checks store nothing
        const uint32_t tfull = bar0 + 8 * (2 * C::STAGES + acc);
        const uint32_t tempty = bar0 + 8 * (2 * C::STAGES + 2 + acc);
        const int row = mb * C::TILE_M + static_cast<int>(prank) * BM + q * 32 + lane;
        const bool row_ok = row < p.M;
        // BWD_ACT: the saved pre-activations of the warp's first two chunks
        // are fetched while the accumulator is still being computed; each
        // chunk then prefetches the one two ahead.
        const bool glu = p.act == TP_ACT_SWIGLU;
        const __nv_bfloat16* ug =
            MODE == tpi::GEMM_BWD_ACT ? p.aux + static_cast<long long>(row_ok ? row : 0) * p.ldaux : nullptr;
        uint4 n1u[4], n1g[4], n2u[4], n2g[4];
        if (MODE == tpi::GEMM_BWD_ACT) {
            load_ug_chunk(p, ug, row_ok, glu, nb * BN + cb * 32, n1u, n1g);
            load_ug_chunk(p, ug, row_ok, glu, nb * BN + cb * 32 + 32, n2u, n2g);
        }
        const bool got = mbar_wait(tfull, acc_phase, abort_flag, p.status, p.timeout_ns);
        __syncwarp();
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after();
        // Folded RMSNorm of the A rows (colwise modes): per-row scale.
        float rs = 1.0f;
        if (MODE != tpi::GEMM_ROW_FUSED && MODE != tpi::GEMM_ROW_PARTIAL && p.row_ss && row_ok) {
            float ss = 0.0f;
            for (int i = 0; i < p.row_ss_parts; ++i) ss += p.row_ss[static_cast<long long>(i) * p.M + row];
            rs = rsqrtf(ss * p.inv_h + p.eps);
        }
        float ssq = 0.0f;
        const uint32_t t0 = tmem_base + acc * BNT + (static_cast<uint32_t>(q * 32) << 16);
        uint32_t r[32];
        if (MODE == tpi::GEMM_BWD_ACT) {
            // One branch-free chunk loop per activation, chosen once per tile.
            const int row0 = mb * C::TILE_M + static_cast<int>(prank) * BM + q * 32;
            const uint32_t sbuf = epi0 + static_cast<uint32_t>(warp - 2) * 3 * EPI_BOX_BYTES;
            switch (p.act) {
                case TP_ACT_SWIGLU:
                    bwd_act_tile<TP_ACT_SWIGLU, CPW>(p, ug, row_ok, row0, nb, cb, t0, sbuf, n1u, n1g, n2u, n2g);
                    break;
                case TP_ACT_GELU_ERF:
                    bwd_act_tile<TP_ACT_GELU_ERF, CPW>(p, ug, row_ok, row0, nb, cb, t0, sbuf, n1u, n1g, n2u, n2g);
                    break;
                case TP_ACT_GELU_TANH:
                    bwd_act_tile<TP_ACT_GELU_TANH, CPW>(p, ug, row_ok, row0, nb, cb, t0, sbuf, n1u, n1g, n2u, n2g);
                    break;
                default:
                    bwd_act_tile<TP_ACT_NONE, CPW>(p, ug, row_ok, row0, nb, cb, t0, sbuf, n1u, n1g, n2u, n2g);
                    break;
            }
        } else if (MODE == tpi::GEMM_TN) {
            // fp32 output through two alternating 32 x 32 boxes per warp
            // (128-byte swizzle: 16-byte piece j of row r at r * 128 +
            // (j ^ (r % 8)) * 16); one TMA store, or reduce-add when
            // accumulating, per 32-column chunk.  The warp's 32 rows lie in
            // one output (row splits are multiples of 32).
            const int row0 = mb * C::TILE_M + static_cast<int>(prank) * BM + q * 32;
            const bool box_ok = row0 < p.M;
            const int which = row0 >= p.row_split2 ? 2 : (row0 >= p.row_split ? 1 : 0);
            const int ybase = row0 - (which == 2 ? p.row_split2 : (which == 1 ? p.row_split : 0));
            const uint32_t sw_base = epi0 + static_cast<uint32_t>(warp - 2) * 4 * EPI_BOX_BYTES;
            const uint32_t srow = static_cast<uint32_t>(lane) * 128;
#pragma unroll 1
            for (int c = cb; c < cb + CPW; ++c) {
                const int col0 = nb * BN + c * 32;
                if (col0 >= p.N) break;  // warp-uniform
                __syncwarp();
                tmem_ld32(t0 + c * 32, r);
                tmem_ld_wait();
                const uint32_t buf = sw_base + static_cast<uint32_t>(c & 1) * 2 * EPI_BOX_BYTES;
                if (lane == 0) bulk_wait_group_read1();  // this box's previous store has read it
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(buf + srow + ((static_cast<uint32_t>(j) ^ (lane & 7)) << 4), r[4 * j],
                                 r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && box_ok) {
                    if (p.accumulate) tma_reduce_add_2d(&p.mapO[which], buf, col0, ybase);
                    else tma_store_2d(&p.mapO[which], buf, col0, ybase);
                    bulk_commit_group();
                }
            }
        } else if (MODE == tpi::GEMM_COL_SWIGLU) {
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
            for (int c = cb_glu; c < cb_glu + CPW_GLU; ++c) {
                if (nb * (BN / 2) + c * 32 >= p.N) break;  // warp-uniform
                uint32_t u[32];
                __syncwarp();
                tmem_ld32(t0 + c * 32, r);             // gate: X W1^T
                tmem_ld32(t0 + BN / 2 + c * 32, u);    // up:   X W3^T
                tmem_ld_wait();
                const int col0 = nb * (BN / 2) + c * 32;
                if (row_ok) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int col = col0 + g * 8;
                        if (col < p.N) {
                            uint32_t w[4], pg[4], pu[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float g0 = __uint_as_float(r[g * 8 + 2 * e]) * rs;
                                const float g1 = __uint_as_float(r[g * 8 + 2 * e + 1]) * rs;
                                const float u0 = __uint_as_float(u[g * 8 + 2 * e]) * rs;
                                const float u1 = __uint_as_float(u[g * 8 + 2 * e + 1]) * rs;
                                const float h0 = silu(g0) * u0;
                                const float h1 = silu(g1) * u1;
                                w[e] = pack_bf16x2(h0, h1);
                                pg[e] = pack_bf16x2(g0, g1);
                                pu[e] = pack_bf16x2(u0, u1);
                            }
                            st_v4(out + static_cast<long long>(row) * p.ldo + col, w[0], w[1],
                                  w[2], w[3]);
                            if (p.aux_out) {  // pre-activations for the backward pass
                                __nv_bfloat16* a = p.aux_out + static_cast<long long>(row) * p.ldaux;
                                st_v4(a + col, pg[0], pg[1], pg[2], pg[3]);
                                st_v4(a + p.n_half + col, pu[0], pu[1], pu[2], pu[3]);
                            }
                        }
                    }
                }
            }
        } else if (MODE == tpi::GEMM_COL_ACT && C::COL_STAGED && p.o_staged) {
            const int row0 = mb * C::TILE_M + static_cast<int>(prank) * BM + q * 32;
            const uint32_t sbuf = epi0 + static_cast<uint32_t>(warp - 2) * 2 * EPI_BOX_BYTES;
            switch (p.act) {
                case TP_ACT_GELU_ERF:
                    col_act_tile_staged<TP_ACT_GELU_ERF, CPW, BNT>(p, t0, cb, nb, row, row_ok, row0, rs, sbuf);
                    break;
                case TP_ACT_GELU_TANH:
                    col_act_tile_staged<TP_ACT_GELU_TANH, CPW, BNT>(p, t0, cb, nb, row, row_ok, row0, rs, sbuf);
                    break;
                default:
                    col_act_tile_staged<TP_ACT_NONE, CPW, BNT>(p, t0, cb, nb, row, row_ok, row0, rs, sbuf);
                    break;
            }
        } else if (MODE == tpi::GEMM_COL_ACT) {
            // One branch-free chunk loop per activation, chosen once per tile.
            switch (p.act) {
                case TP_ACT_GELU_ERF:
                    std_tile<MODE, TP_ACT_GELU_ERF, CPW, BNT>(p, t0, cb, nb, s_grid, row, row_ok, rs, ssq);
                    break;
                case TP_ACT_GELU_TANH:
                    std_tile<MODE, TP_ACT_GELU_TANH, CPW, BNT>(p, t0, cb, nb, s_grid, row, row_ok, rs, ssq);
                    break;
                default:
                    std_tile<MODE, TP_ACT_NONE, CPW, BNT>(p, t0, cb, nb, s_grid, row, row_ok, rs, ssq);
                    break;
            }
        } else {
            std_tile<MODE, TP_ACT_NONE, CPW, BNT>(p, t0, cb, nb, s_grid, row, row_ok, rs, ssq);
        }
        tc_fence_before();
        __syncwarp();
        // Release the accumulator: the leader's MMA waits for the epilogue
        // warps of both CTAs.
        if (lane == 0) {
            if (CG == 2) mbar_arrive_cluster(mapa_shared(tempty, rank & ~1u));
            else mbar_arrive(tempty);
        }
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
    }
    // Staged outputs: every TMA store has completed before the CTA moves on
    // (its shared memory stays valid until then).
    if ((C::STAGED_OUT || C::COL_STAGED) && lane == 0) bulk_wait_group0();
    __syncwarp();
}

template <int MODE, int CG, int BNT>
__global__ void __launch_bounds__(num_threads<MODE>(), 1) tp_gemm_kernel(const __grid_constant__ GemmParams p) {
    constexpr int EPI_WARPS = epi_warps<MODE>();
    using C = Cfg<MODE, CG, BNT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t epi0 = base + C::STAGES * C::STAGE_BYTES;  // staged output boxes
    const uint32_t bar0 = epi0 + C::EPI_BYTES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES +
                                                      8 * (2 * C::STAGES + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Rank in the cluster (GEMM_MLP: 0..3, pairs (0, 1) and (2, 3)).
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
    constexpr int CL = cluster_ctas<MODE, CG, BNT>();
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar0 + 8 * s, 1);                // full: leader's arrive + both CTAs' bytes
            mbar_init(bar0 + 8 * (C::STAGES + s), CL / CG);  // empty: one commit per pair reading it
        }
        mbar_init(bar0 + 8 * (2 * C::STAGES + 0), 1);       // tmem full x2: one commit
        mbar_init(bar0 + 8 * (2 * C::STAGES + 1), 1);
        mbar_init(bar0 + 8 * (2 * C::STAGES + 2), EPI_WARPS * CG);  // tmem empty x2: epilogue warps
        mbar_init(bar0 + 8 * (2 * C::STAGES + 3), EPI_WARPS * CG);
        mbar_init(bar0 + 8 * (2 * C::STAGES + 4), 1);       // drain
        for (int b = 0; b < C::BOX_BARS; ++b)                // output boxes (GEMM_MLP)
            mbar_init(bar0 + 8 * (2 * C::STAGES + 5) + 16 + 8 * b, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.mapA);
        tma_prefetch_desc(&p.mapB[0]);
        if (MODE == tpi::GEMM_MLP) {
            tma_prefetch_desc(&p.mapH);
            tma_prefetch_desc(&p.mapW2);
        }
        if (MODE == tpi::GEMM_COL_SWIGLU || MODE == tpi::GEMM_COL_QKV || MODE == tpi::GEMM_NN)
            tma_prefetch_desc(&p.mapB[1]);
        if (MODE == tpi::GEMM_COL_QKV || MODE == tpi::GEMM_NN) tma_prefetch_desc(&p.mapB[2]);
    }
    if (warp == 1) {
        if (CG == 2) {
            tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    // Both CTAs' barriers exist before either signals the other's.
    if (CG == 2) cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // The next kernel may start its prologue on SMs this grid leaves; this
    // one touches global memory only once the previous kernel is done.
    pdl_trigger();
    pdl_wait();

    if constexpr (MODE == tpi::GEMM_MLP) {
        if (warp == 0) {
            if (lane == 0) mlp_producer_loop<CG>(p, base, bar0, rank, abort_flag);
        } else if (warp == 1) {
            if (lane == 0 && (rank & 1u) == 0) mma_loop<MODE, CG, BNT>(p, base, bar0, tmem_base, abort_flag, rank);
        } else {
            mlp_epilogue_loop<CG>(p, bar0, epi0, tmem_base, rank, abort_flag);
        }
    } else {
        if (warp == 0) {
            if (lane == 0) producer_loop<MODE, CG, BNT>(p, base, bar0, rank, abort_flag);
        } else if (warp == 1) {
            if (lane == 0 && (rank & 1u) == 0) mma_loop<MODE, CG, BNT>(p, base, bar0, tmem_base, abort_flag, rank);
        } else {
            epilogue_loop<MODE, CG, BNT>(p, bar0, epi0, tmem_base, rank, abort_flag);
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    // Neither CTA leaves while the pair may still touch its shared memory.
    if (CG == 2) cluster_sync_all();
    tc_fence_after();
    if (warp == 1) {
        if (CG == 2) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(std::string* err) {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn && err) *err = "cuTensorMapEncodeTiled is not available from the driver";
    return fn;
}

// bf16 tensor map with 128-byte swizzle; dims innermost first, strides in
// bytes for dims 1.., box innermost first.
bool make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box, std::string* err,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    EncodeTiledFn fn = encode_fn(err);
    if (!fn) return false;
    cuuint64_t d[3], s[2];
    cuuint32_t b[3], e[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
    CUresult r = fn(m, dtype, rank, const_cast<void*>(ptr), d, s, b, e,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (err) *err = "cuTensorMapEncodeTiled failed with code " + std::to_string((int)r);
        return false;
    }
    return true;
}

template <int MODE, int CG, int BNT = BN>
int launch_mode(const GemmParams& p, int grid, cudaStream_t stream, std::string* err) {
    auto kern = tp_gemm_kernel<MODE, CG, BNT>;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg<MODE, CG, BNT>::SMEM);
        if (e != cudaSuccess) {
            if (err) *err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
            return TP_ERR_CUDA;
        }
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(num_threads<MODE>(), 1, 1);
    cfg.dynamicSmemBytes = Cfg<MODE, CG, BNT>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster_ctas<MODE, CG, BNT>();
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    tpi::pdl_attribute(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        if (err) *err = std::string("GEMM launch: ") + cudaGetErrorString(e);
        return TP_ERR_CUDA;
    }
    return TP_OK;
}

// Clusters of four CTAs of the wide-tile kernel of MODE that fit on the
// current device at once (0 when the query fails).
template <int MODE>
int max_clusters() {
    static int counts[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 0;
    if (!counts[dev]) {
        constexpr int CG = TP_GEMM_CTA_PAIR;
        constexpr int CL = cluster_ctas<MODE, CG, BN>();
        auto kern = tp_gemm_kernel<MODE, CG, BN>;
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<MODE, CG, BN>::SMEM) ==
            cudaSuccess) {
            cudaLaunchConfig_t cfg;
            memset(&cfg, 0, sizeof(cfg));
            cfg.gridDim = dim3(CL * 64, 1, 1);
            cfg.blockDim = dim3(num_threads<MODE>(), 1, 1);
            cfg.dynamicSmemBytes = Cfg<MODE, CG, BN>::SMEM;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = CL;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
        }
        cudaGetLastError();
        counts[dev] = n > 0 ? n : -1;
    }
    return counts[dev] > 0 ? counts[dev] : 0;
}

}  // namespace

namespace tpi {

// CTAs per output tile (1: 128 x 256 per CTA; 2: 256 x 256 per CTA pair).
constexpr int kPairTiles = TP_GEMM_CTA_PAIR;
// Output columns of the narrow rowwise tile (UMMA N = 128).
constexpr int kNarrowBN = 128;

int gemm_launch(const GemmArgs& a, cudaStream_t stream, std::string* err) {
    GemmParams p;
    memset(&p, 0, sizeof(p));
    const bool row = (a.mode == GEMM_ROW_FUSED || a.mode == GEMM_ROW_PARTIAL);
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.act = a.act;
    p.out = a.out;
    p.ldo = a.ldo;
    p.out_f32 = a.out_f32;
    p.bias = reinterpret_cast<const __nv_bfloat16*>(a.bias);
    p.residual = reinterpret_cast<const __nv_bfloat16*>(a.residual);
    p.ldr = a.ldr;
    p.row_ss = a.row_ss;
    p.row_ss_parts = a.row_ss_parts > 0 ? a.row_ss_parts : 1;
    p.sp_batch = a.sp_batch;
    p.sp_seq = a.sp_seq;
    p.sp_t = (a.mode == GEMM_ROW_FUSED && a.sp_t > 0 && a.sp_seq > 0 && a.sp_seq % a.sp_t == 0) ? a.sp_t : 0;
    p.ss_out = a.ss_out;
    p.inv_h = a.inv_h;
    p.eps = a.eps;
    p.aux = reinterpret_cast<const __nv_bfloat16*>(a.aux);
    p.aux_out = reinterpret_cast<__nv_bfloat16*>(a.aux_out);
    p.ldaux = a.ldaux;
    p.n_half = a.n_half;
    p.out2 = a.out2;
    p.ldo2 = a.ldo2;
    p.k_split = static_cast<int>(a.k_split);
    p.row_split = static_cast<int>(a.row_split);
    p.accumulate = a.accumulate;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    constexpr int CG = kPairTiles;
    constexpr int TILE_M = BM * CG;
    p.m_tiles = static_cast<int>((a.M + TILE_M - 1) / TILE_M);
    const int bn_out = (a.mode == GEMM_COL_SWIGLU) ? BN / 2 : BN;
    p.n_tiles = static_cast<int>((a.N + bn_out - 1) / bn_out);
    p.grid_shards = (a.mode == GEMM_ROW_PARTIAL) ? a.t : 1;
    // Rowwise GEMMs of small problems (few output tiles, long K) take
    // 128-column tiles when those still fit in one wave: twice the CTAs
    // busy, each tile half as long.
    bool narrow = false;
    if (row) {
        const long long units = std::max(1, device_sm_count() / CG);
        const long long n_narrow = (a.N + kNarrowBN - 1) / kNarrowBN;
        const long long thin = static_cast<long long>(p.grid_shards) * p.m_tiles * n_narrow;
        narrow = n_narrow > p.n_tiles && thin <= units;
        if (narrow) p.n_tiles = static_cast<int>(n_narrow);
    }
    p.shard_stride = a.M * a.ldo;
    // Clusters of two pairs with multicast A halves (see mc_mode).
    const bool mc = a.mode == GEMM_COL_QKV && kPairTiles == 2;
    const uint32_t a_rows = mc ? BM / 2 : BM;  // A box rows a CTA loads
    if (row) {
        p.kb_per_shard = static_cast<int>((a.Ks + BK - 1) / BK);
        p.k_shards = (a.mode == GEMM_ROW_FUSED) ? a.t : 1;
        // A: [M][t*Ks] seen as (Ks, t, M); B: [N][t*Ks] seen as (Ks, t, N).
        const uint64_t dA[3] = {(uint64_t)a.Ks, (uint64_t)a.t, (uint64_t)a.M};
        const uint64_t sA[2] = {(uint64_t)a.Ks * 2, (uint64_t)a.t * a.Ks * 2};
        const uint32_t bA[3] = {BK, 1, a_rows};
        if (!make_map(&p.mapA, a.A, 3, dA, sA, bA, err)) return TP_ERR_CUDA;
        const uint64_t dB[3] = {(uint64_t)a.Ks, (uint64_t)a.t, (uint64_t)a.N};
        const uint32_t bB[3] = {BK, 1, B_CHUNK_ROWS};
        if (!make_map(&p.mapB[0], a.B0, 3, dB, sA, bB, err)) return TP_ERR_CUDA;
    } else if (a.mode == GEMM_BWD_ACT || a.mode == GEMM_NN || a.mode == GEMM_TN) {
        p.kb_per_shard = static_cast<int>((a.K + BK - 1) / BK);
        p.k_shards = 1;
        const uint32_t box_mn[2] = {64, BK};  // 64 MN elements x 64 K rows
        if (a.mode == GEMM_TN) {
            // A stored [K][lda]: (M, K) view.
            const int64_t lda = a.lda ? a.lda : a.M;
            const uint64_t dA[2] = {(uint64_t)a.M, (uint64_t)a.K};
            const uint64_t sA[1] = {(uint64_t)lda * 2};
            if (!make_map(&p.mapA, a.A, 2, dA, sA, box_mn, err)) return TP_ERR_CUDA;
        } else {
            const int64_t lda = a.lda ? a.lda : a.K;
            const uint64_t dA[2] = {(uint64_t)a.K, (uint64_t)a.M};
            const uint64_t sA[1] = {(uint64_t)lda * 2};
            const uint32_t bA[2] = {BK, BM};
            if (!make_map(&p.mapA, a.A, 2, dA, sA, bA, err)) return TP_ERR_CUDA;
        }
        // B stored [K rows][N]: (N, K rows) views; GEMM_NN splits K rows at
        // k_split and k_split2 between B0, B1 and B2 (multiples of BK).
        const int64_t split = (a.mode == GEMM_NN && a.B1) ? a.k_split : a.K;
        const int64_t split2 = (a.mode == GEMM_NN && a.B1 && a.B2) ? a.k_split2 : a.K;
        if ((split % BK != 0 && split != a.K) || (split2 % BK != 0 && split2 != a.K) || split2 < split) {
            if (err) *err = "K splits of the NN GEMM must be ordered multiples of 64";
            return TP_ERR_INVALID_ARG;
        }
        p.k_split = static_cast<int>(split);
        p.k_split2 = static_cast<int>(split2);
        const uint64_t sB[1] = {(uint64_t)a.N * 2};
        const uint64_t dB0[2] = {(uint64_t)a.N, (uint64_t)split};
        if (!make_map(&p.mapB[0], a.B0, 2, dB0, sB, box_mn, err)) return TP_ERR_CUDA;
        p.mapB[1] = p.mapB[0];
        p.mapB[2] = p.mapB[0];
        if (split < split2) {
            const uint64_t dB1[2] = {(uint64_t)a.N, (uint64_t)(split2 - split)};
            if (!make_map(&p.mapB[1], a.B1, 2, dB1, sB, box_mn, err)) return TP_ERR_CUDA;
        }
        if (split2 < a.K) {
            const uint64_t dB2[2] = {(uint64_t)a.N, (uint64_t)(a.K - split2)};
            if (!make_map(&p.mapB[2], a.B2, 2, dB2, sB, box_mn, err)) return TP_ERR_CUDA;
        }
        p.row_split = static_cast<int>(a.mode == GEMM_TN && a.out2 ? a.row_split : a.M);
        p.row_split2 = static_cast<int>(a.mode == GEMM_TN && a.out2 && a.out3 ? a.row_split2 : a.M);
        p.out3 = a.out3;
        p.ldo3 = a.ldo3;
        if (a.mode == GEMM_TN) {
            // fp32 output boxes of 32 x 32, 128-byte swizzle: out rows [0,
            // row_split), out2 rows [row_split, row_split2), out3 the rest.
            if ((p.row_split < a.M && p.row_split % EPI_BOX) || (p.row_split2 < a.M && p.row_split2 % EPI_BOX)) {
                if (err) *err = "TN row splits must be multiples of 32";
                return TP_ERR_INVALID_ARG;
            }
            const uint32_t box_o[2] = {EPI_BOX, EPI_BOX};
            void* outs[3] = {a.out, a.out2, a.out3};
            const int64_t lds[3] = {a.ldo, a.ldo2, a.ldo3};
            const int64_t r0[3] = {0, p.row_split, p.row_split2};
            const int64_t r1[3] = {p.row_split, p.row_split2, a.M};
            for (int o = 0; o < 3; ++o) {
                p.mapO[o] = p.mapO[0];
                if (r1[o] <= r0[o] || !outs[o]) continue;
                const uint64_t dO[2] = {(uint64_t)a.N, (uint64_t)(r1[o] - r0[o])};
                const uint64_t sO[1] = {(uint64_t)lds[o] * 4};
                if (!make_map(&p.mapO[o], outs[o], 2, dO, sO, box_o, err, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
                    return TP_ERR_CUDA;
            }
        }
        if (a.mode == GEMM_BWD_ACT) {
            // Output boxes of 32 x 32 bf16, 64-byte swizzle: dU = out[:, :N],
            // dG = out[:, n_half : n_half + N] (SwiGLU), H = out2.
            const uint32_t box_o[2] = {EPI_BOX, EPI_BOX};
            const uint64_t dO[2] = {(uint64_t)a.N, (uint64_t)a.M};
            const uint64_t sO[1] = {(uint64_t)a.ldo * 2};
            const char* base = static_cast<const char*>(a.out);
            if (!make_map(&p.mapO[0], base, 2, dO, sO, box_o, err, CU_TENSOR_MAP_SWIZZLE_64B))
                return TP_ERR_CUDA;
            p.mapO[1] = p.mapO[0];
            if (a.act == TP_ACT_SWIGLU &&
                !make_map(&p.mapO[1], base + a.n_half * 2, 2, dO, sO, box_o, err, CU_TENSOR_MAP_SWIZZLE_64B))
                return TP_ERR_CUDA;
            p.mapO[2] = p.mapO[0];
            if (a.out2) {
                const uint64_t sH[1] = {(uint64_t)a.ldo2 * 2};
                if (!make_map(&p.mapO[2], a.out2, 2, dO, sH, box_o, err, CU_TENSOR_MAP_SWIZZLE_64B))
                    return TP_ERR_CUDA;
            }
        }
    } else {
        p.kb_per_shard = static_cast<int>((a.K + BK - 1) / BK);
        p.k_shards = 1;
        const uint64_t dA[2] = {(uint64_t)a.K, (uint64_t)a.M};
        const uint64_t sA[1] = {(uint64_t)a.K * 2};
        const uint32_t bA[2] = {BK, a_rows};
        if (!make_map(&p.mapA, a.A, 2, dA, sA, bA, err)) return TP_ERR_CUDA;
        const void* bs[3] = {a.B0, a.B1, a.B2};
        const int64_t rows[3] = {a.B0_rows, a.B1_rows, a.B2_rows};
        const uint32_t bB[2] = {BK, B_CHUNK_ROWS};
        for (int i = 0; i < 3; ++i) {
            if (!bs[i]) {
                p.mapB[i] = p.mapB[0];
                continue;
            }
            const uint64_t dB[2] = {(uint64_t)a.K, (uint64_t)rows[i]};
            if (!make_map(&p.mapB[i], bs[i], 2, dB, sA, bB, err)) return TP_ERR_CUDA;
        }
        p.b_rows0 = static_cast<int>(a.B0_rows);
        if (a.mode == GEMM_COL_ACT && kPairTiles == 2 && a.ldo % 8 == 0 &&
            (reinterpret_cast<uintptr_t>(a.out) & 15u) == 0) {
            // Output boxes of 32 x 32 bf16, 64-byte swizzle (rows and columns
            // past the output are clipped).
            const uint32_t box_o[2] = {EPI_BOX, EPI_BOX};
            const uint64_t dO[2] = {(uint64_t)a.N, (uint64_t)a.M};
            const uint64_t sO[1] = {(uint64_t)a.ldo * 2};
            if (!make_map(&p.mapO[0], a.out, 2, dO, sO, box_o, err, CU_TENSOR_MAP_SWIZZLE_64B))
                return TP_ERR_CUDA;
            p.o_staged = 1;
        }
        p.qkv_ws = static_cast<int>(a.qkv_ws);
        p.qkv_qw = static_cast<int>(a.qkv_qw);
        p.qkv_kvw = static_cast<int>(a.qkv_kvw);
        p.kv_heads = a.kv_heads;
        p.head_dim = a.head_dim;
        p.tp = a.t;
        p.pk_nb = a.pk_nb;
        p.pk_ws = static_cast<int>(a.pk_ws);
        for (int b = 0; b < kMaxPackedBlocks; ++b) {
            p.pk_w[b] = a.pk_w[b];
            p.pk_off[b] = static_cast<int>(a.pk_off[b]);
        }
    }
    // Tiles run in groups of group_m m-tiles sweeping all n-tiles, so a wave
    // of SM-count CTAs shares a few weight (B) tiles across many m-tiles.
    // Measured on GB300 at the layer's shapes with 256-row pair tiles: 16
    // is best for the forward colwise GEMMs (W1/W3 2005 TFLOP/s vs 1941 at
    // 32 and 1884 at 4; 930 us vs 934-947 us at 8 and 12), 8 for the
    // rowwise ones, whose A panels (all shards' K) are longer (W2 509-510 us
    // against 516-525 us at 16, and 1.06 GB of DRAM reads per launch
    // against 1.27 GB), and 8 for the backward GEMMs (MLP backward
    // 3180-3220 us against 3237-3281 us at 16).
    const bool colwise_fwd = a.mode == GEMM_COL_ACT || a.mode == GEMM_COL_SWIGLU || a.mode == GEMM_COL_QKV ||
                             a.mode == GEMM_COL_PACKED;
    p.group_m = colwise_fwd ? 16 : 8;
    p.n_dec = mc ? (p.n_tiles + 1) / 2 : p.n_tiles;
    p.num_tiles = p.grid_shards * p.m_tiles * p.n_dec;  // tiles, or cluster units of two tiles
    if (p.num_tiles == 0) return TP_OK;
    int grid = std::min(p.num_tiles, device_sm_count() / CG) * CG;
    if (mc) {
        // Every cluster resident at once: as many as fit (144 SMs on GB300).
        const int clusters = max_clusters<GEMM_COL_QKV>();
        if (clusters < 1) {
            if (err) *err = "no cluster of four CTAs fits on this device";
            return TP_ERR_CUDA;
        }
        grid = std::min(p.num_tiles, clusters) * 2 * CG;
    }
    switch (a.mode) {
        case GEMM_COL_ACT: return launch_mode<GEMM_COL_ACT, CG>(p, grid, stream, err);
        case GEMM_COL_SWIGLU: return launch_mode<GEMM_COL_SWIGLU, CG>(p, grid, stream, err);
        case GEMM_COL_QKV: return launch_mode<GEMM_COL_QKV, CG>(p, grid, stream, err);
        case GEMM_ROW_FUSED:
            return narrow ? launch_mode<GEMM_ROW_FUSED, CG, kNarrowBN>(p, grid, stream, err)
                          : launch_mode<GEMM_ROW_FUSED, CG>(p, grid, stream, err);
        case GEMM_ROW_PARTIAL:
            return narrow ? launch_mode<GEMM_ROW_PARTIAL, CG, kNarrowBN>(p, grid, stream, err)
                          : launch_mode<GEMM_ROW_PARTIAL, CG>(p, grid, stream, err);
        case GEMM_COL_PACKED: return launch_mode<GEMM_COL_PACKED, CG>(p, grid, stream, err);
        case GEMM_BWD_ACT: return launch_mode<GEMM_BWD_ACT, CG>(p, grid, stream, err);
        case GEMM_NN: return launch_mode<GEMM_NN, CG>(p, grid, stream, err);
        case GEMM_TN: return launch_mode<GEMM_TN, CG>(p, grid, stream, err);
        default:
            if (err) *err = "unknown GEMM mode";
            return TP_ERR_INVALID_ARG;
    }
}

// ---- the fused MLP (GEMM_MLP)

namespace {

// Clusters of the fused MLP kernel that fit on the current device at once
// (its persistent grid; every cluster must be resident, since units wait on
// other units' stores).  0 when the query fails.
int mlp_max_clusters() {
    static int counts[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 0;
    if (!counts[dev]) {
        constexpr int CG = kPairTiles;
        auto kern = tp_gemm_kernel<GEMM_MLP, CG, BN>;
        int n = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<GEMM_MLP, CG>::SMEM) ==
            cudaSuccess) {
            cudaLaunchConfig_t cfg;
            memset(&cfg, 0, sizeof(cfg));
            constexpr int CL = cluster_ctas<GEMM_MLP, CG>();
            cfg.gridDim = dim3(CL * 64, 1, 1);
            cfg.blockDim = dim3(num_threads<GEMM_MLP>(), 1, 1);
            cfg.dynamicSmemBytes = Cfg<GEMM_MLP, CG>::SMEM;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = CL;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
        }
        cudaGetLastError();
        counts[dev] = n > 0 ? n : -1;
    }
    return counts[dev] > 0 ? counts[dev] : 0;
}

// Makespan, in k-blocks, of `units` run round-robin over `pairs` clusters in
// the fused MLP's unit order (colwise units first), with `fix` k-blocks of
// partial-sum epilogue charged to each rowwise unit when pieces > 1.
long long mlp_makespan(long long col_units, long long kb_col, long long row_units, long long kb_row_unit,
                       long long fix, int pairs) {
    long long worst = 0;
    for (int q = 0; q < pairs; ++q) {
        long long tsum = 0;
        for (long long u = q; u < col_units + row_units; u += pairs)
            tsum += u < col_units ? kb_col : kb_row_unit + fix;
        worst = std::max(worst, tsum);
    }
    return worst;
}

}  // namespace

int64_t mlp_fused_counter_words(int64_t M, int64_t h, int64_t f) {
    (void)f;
    const int64_t mt = (M + 2 * BM - 1) / (2 * BM);
    return mt * 8 + mt * ((h + BN - 1) / BN) * 2;  // ready [mt][8 pieces] | pieces done [mt][tiles][2]
}

int mlp_fused_pieces(int64_t M, int64_t h, int64_t f, int t, int act) {
    if (kPairTiles != 2) return 0;
    if (act != TP_ACT_GELU_ERF && act != TP_ACT_GELU_TANH && act != TP_ACT_NONE) return 0;
    if (M <= 0 || t <= 0 || f % t || (f / t) % 8 || h % 8) return 0;
    const int clusters = mlp_max_clusters();
    if (clusters < 1) return 0;
    const long long mt = (M + 2 * BM - 1) / (2 * BM);
    // Units are two adjacent 256-column tiles of one m-block (one per pair
    // of a cluster).
    const long long col_units = mt * (((f + BN - 1) / BN + 1) / 2);
    // Two GEMMs of a few waves each leave SMs idle at each kernel's tail and
    // pay a launch and a pipeline fill each; beyond about three colwise waves
    // the two-GEMM path is as good and needs no scratch.
    if (col_units > 3LL * clusters) return 0;
    const long long kb_col = (h + BK - 1) / BK;
    const long long kb_shard = (f / t + BK - 1) / BK;
    const long long row_tiles = mt * (((h + BN - 1) / BN + 1) / 2);
    int best = 0;
    long long best_cost = 0;
    for (int pieces = 1; pieces <= t && pieces <= 8; pieces *= 2) {
        if (t % pieces) continue;
        // Summing a piece's partial reads one 128 KB fp32 half tile per CTA
        // per other piece: charged as two k-blocks each.
        const long long fix = pieces > 1 ? 2LL * (pieces - 1) : 0;
        const long long cost =
            mlp_makespan(col_units, kb_col, row_tiles * pieces, (t / pieces) * kb_shard, fix, clusters);
        if (best == 0 || cost < best_cost) {
            best = pieces;
            best_cost = cost;
        }
    }
    return best;
}

int mlp_fused_launch(const MlpArgs& a, cudaStream_t stream, std::string* err) {
    constexpr int CG = kPairTiles;
    static_assert(CG == 2, "the fused MLP runs on CTA pairs");
    if (a.pieces < 1 || a.pieces > 8 || a.t % a.pieces) {
        if (err) *err = "fused MLP: pieces must divide t and be at most 8";
        return TP_ERR_INVALID_ARG;
    }
    GemmParams p;
    memset(&p, 0, sizeof(p));
    const int64_t Ks = a.f / a.t;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.f);
    p.act = a.act;
    p.out = a.H;
    p.ldo = a.f;
    p.bias = reinterpret_cast<const __nv_bfloat16*>(a.bias);
    p.residual = reinterpret_cast<const __nv_bfloat16*>(a.residual);
    p.ldr = a.h;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    p.kb_per_shard = static_cast<int>((a.h + BK - 1) / BK);
    p.k_shards = 1;
    p.m_tiles = static_cast<int>((a.M + 2 * BM - 1) / (2 * BM));
    p.n_tiles = static_cast<int>((a.f + BN - 1) / BN);
    p.grid_shards = 1;
    p.group_m = 16;
    p.mlp_row_n_tiles = static_cast<int>((a.h + BN - 1) / BN);
    p.mlp_col_units = p.m_tiles * ((p.n_tiles + 1) / 2);
    p.mlp_pieces = a.pieces;
    p.mlp_spp = a.t / a.pieces;
    p.mlp_kb_row = static_cast<int>((Ks + BK - 1) / BK);
    p.mlp_h = static_cast<int>(a.h);
    p.mlp_ks = Ks;
    const int64_t ready_words = static_cast<int64_t>(p.m_tiles) * 8;
    p.mlp_ready = a.counters;
    p.mlp_pdone = a.counters + ready_words;
    p.mlp_part = a.partials;
    p.mlp_z = reinterpret_cast<__nv_bfloat16*>(a.Z);
    if (a.pieces > 1 && !a.partials) {
        if (err) *err = "fused MLP: partials buffer missing";
        return TP_ERR_INVALID_ARG;
    }
    // Colwise operands: X [M][h] (64-row boxes: each CTA loads half of its
    // 128 rows and multicasts them to both pairs), W1 [f][h].
    {
        const uint64_t dA[2] = {(uint64_t)a.h, (uint64_t)a.M};
        const uint64_t sA[1] = {(uint64_t)a.h * 2};
        const uint32_t bA[2] = {BK, BM / 2};
        if (!make_map(&p.mapA, a.X, 2, dA, sA, bA, err)) return TP_ERR_CUDA;
        const uint64_t dB[2] = {(uint64_t)a.h, (uint64_t)a.f};
        const uint32_t bB[2] = {BK, B_CHUNK_ROWS};
        if (!make_map(&p.mapB[0], a.W1, 2, dB, sA, bB, err)) return TP_ERR_CUDA;
    }
    // Rowwise operands: H [M][t Ks] and W2 [h][t Ks] seen as (Ks, t, rows).
    {
        const uint64_t sK[2] = {(uint64_t)Ks * 2, (uint64_t)a.t * Ks * 2};
        const uint64_t dH[3] = {(uint64_t)Ks, (uint64_t)a.t, (uint64_t)a.M};
        const uint32_t bH[3] = {BK, 1, BM / 2};
        if (!make_map(&p.mapH, a.H, 3, dH, sK, bH, err)) return TP_ERR_CUDA;
        const uint64_t dW[3] = {(uint64_t)Ks, (uint64_t)a.t, (uint64_t)a.h};
        const uint32_t bW[3] = {BK, 1, B_CHUNK_ROWS};
        if (!make_map(&p.mapW2, a.W2, 3, dW, sK, bW, err)) return TP_ERR_CUDA;
    }
    // Epilogue boxes: 32 x 32 bf16 (H and Z stores, residual loads) and
    // 16 x 32 fp32 (partials), 64-byte swizzle; rows and columns past the
    // matrices are clipped on stores and read as zeros.
    {
        const uint32_t box16[2] = {EPI_BOX, EPI_BOX};
        const uint64_t dHs[2] = {(uint64_t)a.f, (uint64_t)a.M};
        const uint64_t sHs[1] = {(uint64_t)a.f * 2};
        if (!make_map(&p.mapHs, a.H, 2, dHs, sHs, box16, err, CU_TENSOR_MAP_SWIZZLE_64B)) return TP_ERR_CUDA;
        const uint64_t dZ[2] = {(uint64_t)a.h, (uint64_t)a.M};
        const uint64_t sZ[1] = {(uint64_t)a.h * 2};
        if (!make_map(&p.mapZs, a.Z, 2, dZ, sZ, box16, err, CU_TENSOR_MAP_SWIZZLE_64B)) return TP_ERR_CUDA;
        p.mapRs = p.mapZs;
        if (a.residual && !make_map(&p.mapRs, a.residual, 2, dZ, sZ, box16, err, CU_TENSOR_MAP_SWIZZLE_64B))
            return TP_ERR_CUDA;
        p.mapPs = p.mapZs;
        if (a.pieces > 1) {
            const uint64_t dP[3] = {(uint64_t)a.h, (uint64_t)a.M, (uint64_t)a.pieces};
            const uint64_t sP[2] = {(uint64_t)a.h * 4, (uint64_t)a.M * a.h * 4};
            const uint32_t bP[3] = {16, EPI_BOX, 1};
            if (!make_map(&p.mapPs, a.partials, 3, dP, sP, bP, err, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
                return TP_ERR_CUDA;
        }
    }
    p.num_tiles = p.mlp_col_units + p.m_tiles * ((p.mlp_row_n_tiles + 1) / 2) * p.mlp_pieces;
    if (p.num_tiles == 0) return TP_OK;
    const int clusters = mlp_max_clusters();
    if (clusters < 1) {
        if (err) *err = "fused MLP: no cluster of its kernel fits on this device";
        return TP_ERR_UNSUPPORTED;
    }
    constexpr int CL = cluster_ctas<GEMM_MLP, CG>();
    const int grid = std::min(p.num_tiles, clusters) * CL;
    return launch_mode<GEMM_MLP, CG>(p, grid, stream, err);
}

}  // namespace tpi
