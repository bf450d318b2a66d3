// tp_attn.cu -- causal GQA attention of every shard's heads.
//
// Source: "텐서 병렬화" (itwiki, Tensor parallelism), section "셀프 어텐션"
// (self-attention): heads are independent, so with Q/K/V split by columns
// each shard computes attention for its a/t query heads with no
// communication; with grouped-query attention the KV heads are split too,
// and replicated when there are fewer KV heads than shards.
//
// Reading of what the page leaves open: scale 1/sqrt(d), causal mask
// (key position <= query position) within each sequence, fp32 softmax with
// the running row maximum subtracted, no dropout, no rotary embedding.
//
// Kernel: one CTA of 4 warps per (64 query rows, query head, sequence);
// each warp owns 16 query rows.  K/V tiles of 64 keys stream through a
// double-buffered, XOR-swizzled shared-memory ring (cp.async); S = Q K^T and
// O += P V run on bf16 mma.sync tensor-core instructions with fp32
// accumulators; the softmax is the online (running max / running sum) form,
// so the 64 x seq score matrix never exists.  Key blocks above the diagonal
// are skipped; the diagonal block is masked element-wise.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <string>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace {

using namespace tpk;

constexpr int ABM = 64;  // query rows per CTA
constexpr int ABN = 64;  // keys per tile
constexpr int ATHREADS = 128;

struct AttnParams {
    const __nv_bfloat16* qkv;
    long long ld_qkv;
    int shard_w, q_w, kv_w;
    __nv_bfloat16* o;
    long long ld_o;
    int seq, heads, kv_heads, t, heads_per_shard;
    float scale_log2;  // log2(e) / sqrt(d)
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk c of row r in a [64][D] bf16 tile whose
// chunks are XOR-swizzled by the row's low 3 bits (conflict-free ldmatrix).
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// Copy rows [row0, row0+64) x D columns of a strided bf16 matrix into a
// swizzled tile; rows at or beyond `rows_valid` are zero-filled.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t tile, const __nv_bfloat16* g, long long ld,
                                          int rows_valid) {
    constexpr int CPR = D / 8;
#pragma unroll
    for (int idx = threadIdx.x; idx < ABM * CPR; idx += ATHREADS) {
        const int r = idx / CPR, c = idx - (idx / CPR) * CPR;
        const bool ok = r < rows_valid;
        const __nv_bfloat16* src = ok ? g + static_cast<long long>(r) * ld + c * 8 : g;
        cp_async16(tile + swz<D>(r, c), src, ok ? 16 : 0);
    }
}

template <int D>
__global__ void __launch_bounds__(ATHREADS) attn_kernel(const AttnParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int TILE = ABM * D * 2;
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK = sQ + TILE;          // 2 buffers
    const uint32_t sV = sQ + 3 * TILE;      // 2 buffers

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nqb = (p.seq + ABM - 1) / ABM;
    const int qb = nqb - 1 - static_cast<int>(blockIdx.x);  // heavy blocks first
    const int j = blockIdx.y;                                // global query head
    const int b = blockIdx.z;                                // sequence
    const int shard = j / p.heads_per_shard;
    const int jl = j - shard * p.heads_per_shard;
    const int g = j / (p.heads / p.kv_heads);                // KV head read by j
    const int kv0 = (p.kv_heads >= p.t) ? shard * (p.kv_heads / p.t) : (shard * p.kv_heads) / p.t;
    const int gl = g - kv0;                                  // its slot in the shard

    const long long tok0 = static_cast<long long>(b) * p.seq;
    const __nv_bfloat16* Qg = p.qkv + (tok0 + qb * ABM) * p.ld_qkv + shard * p.shard_w + jl * D;
    const __nv_bfloat16* Kg = p.qkv + tok0 * p.ld_qkv + shard * p.shard_w + p.q_w + gl * D;
    const __nv_bfloat16* Vg = Kg + p.kv_w;

    const int q_rows = min(ABM, p.seq - qb * ABM);
    load_tile<D>(sQ, Qg, p.ld_qkv, q_rows);
    const int nkb = qb + 1;  // causal: key blocks 0..qb
    load_tile<D>(sK, Kg, p.ld_qkv, min(ABN, p.seq));
    load_tile<D>(sV, Vg, p.ld_qkv, min(ABN, p.seq));
    cp_async_commit();

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
    uint32_t qf[D / 16][4];

    const int qrow0 = qb * ABM + warp * 16 + (lane >> 2);  // rows qrow0 and qrow0 + 8

    for (int kb = 0; kb < nkb; ++kb) {
        cp_async_wait_all();
        __syncthreads();
        if (kb == 0) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = ks * 2 + (lane >> 4);
                ldsm_x4(sQ + swz<D>(r, c), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
            }
        }
        if (kb + 1 < nkb) {
            const int nb = (kb + 1) & 1;
            const int rows = min(ABN, p.seq - (kb + 1) * ABN);
            load_tile<D>(sK + nb * TILE, Kg + static_cast<long long>((kb + 1) * ABN) * p.ld_qkv,
                         p.ld_qkv, rows);
            load_tile<D>(sV + nb * TILE, Vg + static_cast<long long>((kb + 1) * ABN) * p.ld_qkv,
                         p.ld_qkv, rows);
            cp_async_commit();
        }
        const uint32_t kt = sK + (kb & 1) * TILE, vt = sV + (kb & 1) * TILE;

        // S = Q K^T for this warp's 16 rows x 64 keys.
        float s[ABN / 8][4];
#pragma unroll
        for (int i = 0; i < ABN / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int np = 0; np < ABN / 16; ++np) {
                const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = ks * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kt + swz<D>(r, c), b0, b1, b2, b3);
                mma_bf16_16816(s[2 * np], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
                mma_bf16_16816(s[2 * np + 1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
            }
        }
        // Causal / length mask (only the diagonal and the ragged last block).
        const int key0 = kb * ABN;
        if (kb == qb || key0 + ABN > p.seq) {
#pragma unroll
            for (int nt = 0; nt < ABN / 8; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = key0 + nt * 8 + (lane & 3) * 2 + (e & 1);
                    const int qpos = qrow0 + (e >> 1) * 8;
                    if (key > qpos || key >= p.seq) s[nt][e] = -INFINITY;
                }
            }
        }
        // Online softmax.
        float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
        for (int nt = 0; nt < ABN / 8; ++nt) {
            mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
            mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        }
        float alpha[2], msc[2], rs[2] = {0.0f, 0.0f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float mref = (mx[h] == -INFINITY) ? 0.0f : mx[h];
            alpha[h] = exp2f((m_run[h] - mref) * p.scale_log2);
            msc[h] = mref * p.scale_log2;
            m_run[h] = mx[h];
        }
        uint32_t pf[ABN / 16][4];
#pragma unroll
        for (int nt = 0; nt < ABN / 8; ++nt) {
            const float p0 = exp2f(fmaf(s[nt][0], p.scale_log2, -msc[0]));
            const float p1 = exp2f(fmaf(s[nt][1], p.scale_log2, -msc[0]));
            const float p2 = exp2f(fmaf(s[nt][2], p.scale_log2, -msc[1]));
            const float p3 = exp2f(fmaf(s[nt][3], p.scale_log2, -msc[1]));
            rs[0] += p0 + p1;
            rs[1] += p2 + p3;
            pf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p0, p1);
            pf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p2, p3);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * alpha[h] + rs[h];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            o[i][0] *= alpha[0];
            o[i][1] *= alpha[0];
            o[i][2] *= alpha[1];
            o[i][3] *= alpha[1];
        }
        // O += P V.  A fragment of P for keys 16ks..16ks+15 comes straight
        // from the S accumulators of n-tiles 2ks, 2ks+1.
#pragma unroll
        for (int ks = 0; ks < ABN / 16; ++ks) {
            const uint32_t a0 = pf[ks][0], a1 = pf[ks][1], a2 = pf[ks][2], a3 = pf[ks][3];
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                const int r = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = dp * 2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vt + swz<D>(r, c), b0, b1, b2, b3);
                mma_bf16_16816(o[2 * dp], a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }
    // Row sums live spread over the 4 lanes of a quad.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
        l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    const float inv0 = 1.0f / l_run[0], inv1 = 1.0f / l_run[1];
    __nv_bfloat16* Og = p.o + (tok0 + qrow0) * p.ld_o + static_cast<long long>(j) * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const int col = i * 8 + (lane & 3) * 2;
        if (qrow0 < p.seq)
            *reinterpret_cast<uint32_t*>(Og + col) = pack_bf16x2(o[i][0] * inv0, o[i][1] * inv0);
        if (qrow0 + 8 < p.seq)
            *reinterpret_cast<uint32_t*>(Og + 8 * p.ld_o + col) =
                pack_bf16x2(o[i][2] * inv1, o[i][3] * inv1);
    }
}

template <int D>
int launch_d(const tpi::AttnArgs& a, cudaStream_t stream, std::string* err) {
    AttnParams p;
    p.qkv = reinterpret_cast<const __nv_bfloat16*>(a.QKV);
    p.ld_qkv = a.ld_qkv;
    p.shard_w = static_cast<int>(a.shard_w);
    p.q_w = static_cast<int>(a.q_w);
    p.kv_w = static_cast<int>(a.kv_w);
    p.o = reinterpret_cast<__nv_bfloat16*>(a.O);
    p.ld_o = a.ld_o;
    p.seq = a.seq;
    p.heads = a.heads;
    p.kv_heads = a.kv_heads;
    p.t = a.t;
    p.heads_per_shard = a.heads / a.t;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    const int smem = 5 * ABM * D * 2;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            if (err) *err = std::string("cudaFuncSetAttribute(attn): ") + cudaGetErrorString(e);
            return TP_ERR_CUDA;
        }
        configured[dev] = true;
    }
    dim3 grid((a.seq + ABM - 1) / ABM, a.heads, a.batch);
    attn_kernel<D><<<grid, ATHREADS, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        if (err) *err = std::string("attention launch: ") + cudaGetErrorString(e);
        return TP_ERR_CUDA;
    }
    return TP_OK;
}

}  // namespace

namespace tpi {

int attn_launch(const AttnArgs& a, cudaStream_t stream, std::string* err) {
    if (a.batch == 0 || a.seq == 0) return TP_OK;
    if (a.head_dim == 128) return launch_d<128>(a, stream, err);
    if (a.head_dim == 64) return launch_d<64>(a, stream, err);
    if (err) *err = "head_dim must be 64 or 128";
    return TP_ERR_UNSUPPORTED;
}

}  // namespace tpi
