// tp_vocab.cu -- vocab-parallel embedding and the vocab-parallel ("loss
// parallel") cross-entropy.
//
// Source: "텐서 병렬화" (itwiki, Tensor parallelism), section "임베딩과
// 출력층" (embedding and output layer): the embedding matrix is split along
// the vocabulary; for the output layer, rather than gathering all logits
// (b x s x v of traffic) each device computes the cross-entropy from its
// partial logits and only the max and the sum are exchanged (b x s).
// "추론을 위한 텐서 병렬성" (transformers docs), "분할 전략":
// EmbeddingParallel(shard_dim=0) shards the vocabulary and all-reduces the
// partial lookups.
//
// On one GPU the t shards are index ranges of the vocabulary:
//  * embedding: shard i's partial for token id is E[id] when id is in its
//    rows [i v/t, (i+1) v/t), else zero, so the all-reduced sum is the row of
//    the owning shard -- one gather (ids outside [0, v) get a zero row, as in
//    the sharded sum);
//  * cross-entropy: kernel 1 computes, for every (token, shard), the shard's
//    max m_i, sum of exp(z - m_i) and the label's logit if the shard owns it:
//    [3][t][M] fp32, the values the pages exchange; kernel 2 combines them:
//    m = max m_i, s = sum s_i exp(m_i - m), loss = log s + m - z_label.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <string>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace {

using namespace tpk;

constexpr int EMB_WARPS = 8;
constexpr int CE_THREADS = 256;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// One warp per token: copy row E[id] (16-byte vectors), or zeros.
__global__ void __launch_bounds__(EMB_WARPS * 32) vocab_embedding_kernel(
    const int32_t* __restrict__ ids, long long M, const __nv_bfloat16* __restrict__ E, long long v,
    int h, __nv_bfloat16* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const long long m = static_cast<long long>(blockIdx.x) * EMB_WARPS + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (m >= M) return;
    const long long id = ids[m];
    const bool owned = id >= 0 && id < v;  // some shard owns it
    const uint4* src = reinterpret_cast<const uint4*>(E + (owned ? id : 0) * h);
    uint4* dst = reinterpret_cast<uint4*>(out + m * h);
    for (int c = lane; c < (h >> 3); c += 32) dst[c] = owned ? src[c] : make_uint4(0, 0, 0, 0);
}

// Online (max, sum of 2^(x - max)) pair in the log2 domain.
struct MS {
    float m, s;
};

__device__ __forceinline__ MS ms_merge(MS a, MS b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return {m, 0.0f};
    return {m, a.s * ex2f(a.m - m) + b.s * ex2f(b.m - m)};
}

// One CTA per (token, shard): the shard's statistics of its logits slice.
__global__ void __launch_bounds__(CE_THREADS) ce_shard_stats_kernel(
    const __nv_bfloat16* __restrict__ logits, long long M, long long v, int t,
    const int32_t* __restrict__ labels, float* __restrict__ stats) {
    pdl_trigger();
    pdl_wait();
    __shared__ MS red[CE_THREADS / 32];
    const long long m = blockIdx.x;
    const int i = blockIdx.y;
    const long long w = v / t;
    const __nv_bfloat16* z = logits + m * v + i * w;
    MS acc = {-INFINITY, 0.0f};
    for (long long c = threadIdx.x; c < (w >> 3); c += CE_THREADS) {
        const uint4 u = ld_stream(z + c * 8);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
        float x[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(wd[e]);
            x[2 * e] = f.x * LOG2E;
            x[2 * e + 1] = f.y * LOG2E;
        }
        float bm = x[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) bm = fmaxf(bm, x[e]);
        const float nm = fmaxf(acc.m, bm);
        float s = (acc.m == -INFINITY) ? 0.0f : acc.s * ex2f(acc.m - nm);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += ex2f(x[e] - nm);
        acc = {nm, s};
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MS other = {__shfl_xor_sync(0xffffffffu, acc.m, o), __shfl_xor_sync(0xffffffffu, acc.s, o)};
        acc = ms_merge(acc, other);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        MS tot = red[0];
        for (int k = 1; k < CE_THREADS / 32; ++k) tot = ms_merge(tot, red[k]);
        const long long lab = labels[m];
        const float y = (lab >= i * w && lab < (i + 1) * w) ? __bfloat162float(z[lab - i * w]) : 0.0f;
        stats[(0LL * t + i) * M + m] = tot.m * LN2;  // natural-log units
        stats[(1LL * t + i) * M + m] = tot.s;
        stats[(2LL * t + i) * M + m] = y;
    }
}

// One thread per token: combine the t shards' (max, sum, target).
__global__ void ce_combine_kernel(const float* __restrict__ stats, long long M, long long v, int t,
                                  const int32_t* __restrict__ labels, float* __restrict__ loss) {
    pdl_trigger();
    pdl_wait();
    const long long m = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (m >= M) return;
    const long long lab = labels[m];
    if (lab == -100) {
        loss[m] = 0.0f;
        return;
    }
    if (lab < 0 || lab >= v) {
        loss[m] = __int_as_float(0x7fc00000);  // NaN: label outside the vocabulary
        return;
    }
    float mx = -INFINITY;
    for (int i = 0; i < t; ++i) mx = fmaxf(mx, stats[(0LL * t + i) * M + m]);
    float s = 0.0f, y = 0.0f;
    for (int i = 0; i < t; ++i) {
        s += stats[(1LL * t + i) * M + m] * expf(stats[(0LL * t + i) * M + m] - mx);
        y += stats[(2LL * t + i) * M + m];
    }
    loss[m] = logf(s) + mx - y;
}

int check(const char* what, std::string* err) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        if (err) *err = std::string(what) + ": " + cudaGetErrorString(e);
        return TP_ERR_CUDA;
    }
    return TP_OK;
}

}  // namespace

namespace tpi {

int vocab_embedding_launch(const int32_t* ids, int64_t M, const void* E, int64_t v, int h, void* out,
                           cudaStream_t stream, std::string* err) {
    if (M == 0) return TP_OK;
    const long long blocks = (M + EMB_WARPS - 1) / EMB_WARPS;
    launch_pdl(vocab_embedding_kernel, dim3((unsigned)blocks), dim3(EMB_WARPS * 32), 0, stream, ids,
               static_cast<long long>(M), reinterpret_cast<const __nv_bfloat16*>(E), static_cast<long long>(v), h,
               reinterpret_cast<__nv_bfloat16*>(out));
    return check("embedding kernel", err);
}

int vocab_ce_launch(const void* logits, int64_t M, int64_t v, int t, const int32_t* labels,
                    float* stats, float* loss, cudaStream_t stream, std::string* err) {
    if (M == 0) return TP_OK;
    dim3 grid((unsigned)M, (unsigned)t);
    launch_pdl(ce_shard_stats_kernel, grid, dim3(CE_THREADS), 0, stream,
               reinterpret_cast<const __nv_bfloat16*>(logits), static_cast<long long>(M), static_cast<long long>(v), t,
               labels, stats);
    int rc = check("cross-entropy statistics kernel", err);
    if (rc) return rc;
    launch_pdl(ce_combine_kernel, dim3((unsigned)((M + 255) / 256)), dim3(256), 0, stream,
               static_cast<const float*>(stats), static_cast<long long>(M), static_cast<long long>(v), t, labels,
               loss);
    return check("cross-entropy combine kernel", err);
}

}  // namespace tpi
