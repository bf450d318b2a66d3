// tp_elementwise.cu -- HBM-bound kernels of the block: the g-operator
// reduction of the t shard partials, the replicated RMSNorm, and the
// reduction fused with the next RMSNorm.
//
// Source: "텐서 병렬화" (itwiki, Tensor parallelism), section "통신 연산 f와
// g": g is an all-reduce of the t partial sums in the forward pass; norm,
// dropout and residual are replicated.  "추론을 위한 텐서 병렬성"
// (transformers docs), "설계 구현 / DTensor": a rowwise bias is replicated
// and added once, after the reduction.
//
// The reduction is elementwise over t: every thread owns 8 consecutive
// outputs, loads them from each of the t partials with 128-bit streaming
// loads (all issued before the adds), sums in fp32 in shard order
// i = 0..t-1, adds bias and residual, and stores 8 bf16 with one 128-bit
// store.  No shuffles, no shared memory; a grid-stride loop over a grid of
// SM count x 8 CTAs keeps enough loads in flight to saturate HBM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "tp_device.cuh"
#include "tp_internal.h"

namespace {

using namespace tpk;

constexpr int RED_THREADS = 256;
constexpr int MAX_T = 64;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(w[e]);
        acc[2 * e] += f.x;
        acc[2 * e + 1] += f.y;
    }
}

// out[e] = sum_i P[i][e] (+ bias[e % h]) (+ residual[e]); T known at compile
// time (0 = runtime t).
template <int T, bool F32>
__global__ void __launch_bounds__(RED_THREADS) reduce_kernel(const void* __restrict__ partials, int t,
                                                             long long n, int h,
                                                             const __nv_bfloat16* __restrict__ bias,
                                                             const __nv_bfloat16* __restrict__ residual,
                                                             __nv_bfloat16* out) {
    pdl_trigger();
    pdl_wait();
    const int tt = T ? T : t;
    const long long nvec = n >> 3;
    for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < nvec;
         v += (long long)gridDim.x * blockDim.x) {
        const long long e0 = v << 3;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
        if (F32) {
            const float* P = reinterpret_cast<const float*>(partials) + e0;
            if (T) {
                uint4 lo[T ? T : 1], hi[T ? T : 1];
#pragma unroll
                for (int i = 0; i < T; ++i) {
                    lo[i] = ld_stream(P + i * n);
                    hi[i] = ld_stream(P + i * n + 4);
                }
#pragma unroll
                for (int i = 0; i < T; ++i) {
                    acc[0] += __uint_as_float(lo[i].x);
                    acc[1] += __uint_as_float(lo[i].y);
                    acc[2] += __uint_as_float(lo[i].z);
                    acc[3] += __uint_as_float(lo[i].w);
                    acc[4] += __uint_as_float(hi[i].x);
                    acc[5] += __uint_as_float(hi[i].y);
                    acc[6] += __uint_as_float(hi[i].z);
                    acc[7] += __uint_as_float(hi[i].w);
                }
            } else {
                for (int i = 0; i < tt; ++i) {
                    const uint4 lo = ld_stream(P + i * n), hi = ld_stream(P + i * n + 4);
                    acc[0] += __uint_as_float(lo.x);
                    acc[1] += __uint_as_float(lo.y);
                    acc[2] += __uint_as_float(lo.z);
                    acc[3] += __uint_as_float(lo.w);
                    acc[4] += __uint_as_float(hi.x);
                    acc[5] += __uint_as_float(hi.y);
                    acc[6] += __uint_as_float(hi.z);
                    acc[7] += __uint_as_float(hi.w);
                }
            }
        } else {
            const __nv_bfloat16* P = reinterpret_cast<const __nv_bfloat16*>(partials) + e0;
            if (T) {
                uint4 pv[T ? T : 1];
#pragma unroll
                for (int i = 0; i < T; ++i) pv[i] = ld_stream(P + i * n);
#pragma unroll
                for (int i = 0; i < T; ++i) add_bf16x8(acc, pv[i]);
            } else {
                for (int i = 0; i < tt; ++i) add_bf16x8(acc, ld_stream(P + i * n));
            }
        }
        if (bias) add_bf16x8(acc, *reinterpret_cast<const uint4*>(bias + (e0 % h)));
        if (residual) add_bf16x8(acc, *reinterpret_cast<const uint4*>(residual + e0));
        *reinterpret_cast<uint4*>(out + e0) =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                       pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
}

// Row kernel: one CTA per row of h (h/8 vectors spread over the block, at
// most 4 per thread).  h1 = sum_i P[i][row] + residual[row] (bf16-rounded),
// then optionally xn = h1 / sqrt(mean(h1^2) + eps) from the rounded h1.
constexpr int ROW_THREADS = 256;
constexpr int ROW_VEC = 4;  // vectors of 8 per thread -> h <= 8192

// Row of token `row` (= b * seq + pos) in the sequence-split layout
// [t][batch][seq/t] ("시퀀스 병렬화": device i keeps positions
// [i seq/t, (i+1) seq/t) of every sequence); identity when sp_t == 0.
__device__ __forceinline__ long long sp_out_row(long long row, long long sp_batch, long long sp_seq,
                                                int sp_t) {
    if (sp_t == 0) return row;
    const long long w = sp_seq / sp_t;
    const long long b = row / sp_seq, pos = row - b * sp_seq;
    return ((pos / w) * sp_batch + b) * w + pos % w;
}

template <bool HAS_P, bool F32>
__global__ void __launch_bounds__(ROW_THREADS) row_kernel(const void* __restrict__ partials, int t,
                                                          long long n, int h,
                                                          const __nv_bfloat16* __restrict__ src,
                                                          __nv_bfloat16* h1_out,
                                                          __nv_bfloat16* xn_out, float eps,
                                                          long long sp_batch, long long sp_seq,
                                                          int sp_t) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[ROW_THREADS / 32];
    // Partials are read at the token's row; residual and outputs live at its
    // (possibly sequence-split) output row.
    const long long prow = blockIdx.x;
    const long long row = sp_out_row(prow, sp_batch, sp_seq, sp_t);
    const int nv = h >> 3;
    float vals[ROW_VEC][8];
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < ROW_VEC; ++j) {
        const int v = threadIdx.x + j * ROW_THREADS;
#pragma unroll
        for (int e = 0; e < 8; ++e) vals[j][e] = 0.0f;
        if (v < nv) {
            const long long e0 = row * h + (long long)v * 8;
            const long long p0 = prow * h + (long long)v * 8;
            if (HAS_P) {
                for (int i = 0; i < t; ++i) {
                    if (F32) {
                        const float* P = reinterpret_cast<const float*>(partials) + i * n + p0;
                        const uint4 lo = ld_stream(P), hi = ld_stream(P + 4);
                        vals[j][0] += __uint_as_float(lo.x);
                        vals[j][1] += __uint_as_float(lo.y);
                        vals[j][2] += __uint_as_float(lo.z);
                        vals[j][3] += __uint_as_float(lo.w);
                        vals[j][4] += __uint_as_float(hi.x);
                        vals[j][5] += __uint_as_float(hi.y);
                        vals[j][6] += __uint_as_float(hi.z);
                        vals[j][7] += __uint_as_float(hi.w);
                    } else {
                        add_bf16x8(vals[j], ld_stream(reinterpret_cast<const __nv_bfloat16*>(partials) +
                                                      i * n + p0));
                    }
                }
            }
            if (src) add_bf16x8(vals[j], *reinterpret_cast<const uint4*>(src + e0));
            const uint4 packed =
                make_uint4(pack_bf16x2(vals[j][0], vals[j][1]), pack_bf16x2(vals[j][2], vals[j][3]),
                           pack_bf16x2(vals[j][4], vals[j][5]), pack_bf16x2(vals[j][6], vals[j][7]));
            if (h1_out) *reinterpret_cast<uint4*>(h1_out + e0) = packed;
            // The norm reads the residual stream as stored (bf16).
            const uint32_t w[4] = {packed.x, packed.y, packed.z, packed.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = unpack_bf16x2(w[e]);
                vals[j][2 * e] = f.x;
                vals[j][2 * e + 1] = f.y;
                ss += f.x * f.x + f.y * f.y;
            }
        }
    }
    if (!xn_out) return;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < ROW_THREADS / 32; ++w) tot += red[w];
    const float r = rsqrtf(tot / static_cast<float>(h) + eps);
#pragma unroll
    for (int j = 0; j < ROW_VEC; ++j) {
        const int v = threadIdx.x + j * ROW_THREADS;
        if (v < nv) {
            const long long e0 = row * h + (long long)v * 8;
            *reinterpret_cast<uint4*>(xn_out + e0) = make_uint4(
                pack_bf16x2(vals[j][0] * r, vals[j][1] * r), pack_bf16x2(vals[j][2] * r, vals[j][3] * r),
                pack_bf16x2(vals[j][4] * r, vals[j][5] * r), pack_bf16x2(vals[j][6] * r, vals[j][7] * r));
        }
    }
}

// Per-row sum of squares (the statistic of a unit-gain RMSNorm that the next
// colwise GEMM applies as a per-row scale).  One warp per row; 128-bit
// loads; also clears the next norm's accumulator row.
constexpr int SS_WARPS = 8;

__global__ void __launch_bounds__(SS_WARPS * 32) row_sumsq_kernel(const __nv_bfloat16* __restrict__ x,
                                                                  long long rows, int h, float* ss,
                                                                  float* zero) {
    pdl_trigger();
    pdl_wait();
    const long long row = static_cast<long long>(blockIdx.x) * SS_WARPS + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const __nv_bfloat16* xr = x + row * h;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    auto add = [&](const uint4& u) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            acc[e] = fmaf(f.x, f.x, fmaf(f.y, f.y, acc[e]));
        }
    };
    // All of a lane's 16-byte loads of the row in flight at once when the row
    // has at most 16 per lane (h <= 4096), else 8 per round: one memory
    // latency per row instead of one per four loads (the kernel streams
    // 67 MB at the layer shape; with four in flight it ran at 0.57 of HBM).
    // Plain loads: the rows stay in L2 for the GEMM that follows.
    const int nv = h >> 3;
    int v = lane;
    if (nv <= 16 * 32) {
        // Unconditional loads of a clamped (in-row) address, so that all
        // sixteen issue before the first add; out-of-range ones count zero.
        uint4 u[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) u[k] = *reinterpret_cast<const uint4*>(xr + min(v + 32 * k, nv - 1) * 8);
#pragma unroll
        for (int k = 0; k < 16; ++k) add(v + 32 * k < nv ? u[k] : make_uint4(0, 0, 0, 0));
    } else {
        for (; v + 32 * 7 < nv; v += 32 * 8) {
            uint4 u[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) u[k] = *reinterpret_cast<const uint4*>(xr + (v + 32 * k) * 8);
#pragma unroll
            for (int k = 0; k < 8; ++k) add(u[k]);
        }
        for (; v < nv; v += 32) add(*reinterpret_cast<const uint4*>(xr + v * 8));
    }
    float t = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) {
        ss[row] = t;
        if (zero) zero[row] = 0.0f;
    }
}

// Sequence-parallel all-gather ("시퀀스 병렬화": entering the tensor-parallel
// region the sequence pieces are gathered): full[row] = sp[sp_out_row(row)],
// one warp per row, 16-byte vectors.
constexpr int AG_WARPS = 8;

__global__ void __launch_bounds__(AG_WARPS * 32) sp_all_gather_kernel(
    const __nv_bfloat16* __restrict__ sp, long long rows, int h, long long batch, long long seq,
    int t, __nv_bfloat16* __restrict__ full) {
    pdl_trigger();
    pdl_wait();
    const long long row = static_cast<long long>(blockIdx.x) * AG_WARPS + (threadIdx.x >> 5);
    if (row >= rows) return;
    const uint4* src = reinterpret_cast<const uint4*>(sp + sp_out_row(row, batch, seq, t) * h);
    uint4* dst = reinterpret_cast<uint4*>(full + row * h);
    for (int c = threadIdx.x & 31; c < (h >> 3); c += 32) dst[c] = src[c];
}

// The inverse of the all-gather: a token-order tensor into the sequence-split
// layout, one warp per row, 16-byte vectors.  The sequence-parallel layer's
// backward uses it as the reduce-scatter of dX, whose sum over the shards the
// fused backward GEMMs already hold ("텐서 병렬화", "시퀀스 병렬화").
__global__ void __launch_bounds__(AG_WARPS * 32) sp_split_kernel(
    const __nv_bfloat16* __restrict__ full, long long rows, int h, long long batch, long long seq,
    int t, __nv_bfloat16* __restrict__ sp) {
    pdl_trigger();
    pdl_wait();
    const long long row = static_cast<long long>(blockIdx.x) * AG_WARPS + (threadIdx.x >> 5);
    if (row >= rows) return;
    const uint4* src = reinterpret_cast<const uint4*>(full + row * h);
    uint4* dst = reinterpret_cast<uint4*>(sp + sp_out_row(row, batch, seq, t) * h);
    for (int c = threadIdx.x & 31; c < (h >> 3); c += 32) dst[c] = src[c];
}

// Failure-detection self test: wait on a barrier that never completes.
__global__ void selftest_wait_kernel(unsigned* status, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing arrives: the bounded wait gives up and records a timeout.
        mbar_wait(smem_u32(&bar), 0, &abort_flag, status, timeout_ns);
    }
    __syncthreads();
}

std::string cuda_msg(const char* what, cudaError_t e) {
    return std::string(what) + ": " + cudaGetErrorString(e);
}

int check_launch(const char* what, std::string* err) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        if (err) *err = cuda_msg(what, e);
        return TP_ERR_CUDA;
    }
    return TP_OK;
}

// Backward of the unit-gain RMSNorm, plus a residual gradient, per row:
//   out = res + r g - x r^3 (sum_j g_j x_j) / h,  r = 1 / sqrt(mean_j x_j^2 + eps)
// (bf16 in and out, fp32 arithmetic).  One CTA of RB_THREADS per row; each
// thread keeps VPT 8-element vectors of x and g in registers.
constexpr int RB_THREADS = 128;

template <int VPT>
__global__ void __launch_bounds__(RB_THREADS) rmsnorm_bwd_kernel(const __nv_bfloat16* __restrict__ x,
                                                                const __nv_bfloat16* __restrict__ g,
                                                                const __nv_bfloat16* __restrict__ res,
                                                                int h, float eps,
                                                                __nv_bfloat16* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[2][RB_THREADS / 32];
    const long long row = blockIdx.x;
    const int nv = h / 8;
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * h);
    const uint4* gr = reinterpret_cast<const uint4*>(g + row * h);
    float xv[VPT][8], gv[VPT][8];
    float ss = 0.0f, dot = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = threadIdx.x + i * RB_THREADS;
        uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (v < nv) {
            a = xr[v];
            b = gr[v];
        }
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 fa = unpack_bf16x2(aw[e]), fb = unpack_bf16x2(bw[e]);
            xv[i][2 * e] = fa.x;
            xv[i][2 * e + 1] = fa.y;
            gv[i][2 * e] = fb.x;
            gv[i][2 * e + 1] = fb.y;
            ss = fmaf(fa.x, fa.x, fmaf(fa.y, fa.y, ss));
            dot = fmaf(fb.x, fa.x, fmaf(fb.y, fa.y, dot));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
        dot += __shfl_xor_sync(0xffffffffu, dot, o);
    }
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = ss;
        red[1][threadIdx.x >> 5] = dot;
    }
    __syncthreads();
    ss = 0.0f;
    dot = 0.0f;
#pragma unroll
    for (int w = 0; w < RB_THREADS / 32; ++w) {
        ss += red[0][w];
        dot += red[1][w];
    }
    const float inv_h = 1.0f / static_cast<float>(h);
    const float r = rsqrtf(ss * inv_h + eps);
    const float coef = r * r * r * dot * inv_h;
    const uint4* rr = reinterpret_cast<const uint4*>(res + row * h);
    uint4* orow = reinterpret_cast<uint4*>(out + row * h);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = threadIdx.x + i * RB_THREADS;
        if (v >= nv) continue;
        const uint4 c = rr[v];
        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 fc = unpack_bf16x2(cw[e]);
            w[e] = pack_bf16x2(fc.x + r * gv[i][2 * e] - xv[i][2 * e] * coef,
                               fc.y + r * gv[i][2 * e + 1] - xv[i][2 * e + 1] * coef);
        }
        orow[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Column sums of a bf16 [rows][h] matrix into fp32 (the bias gradient
// db = sum over tokens of dZ), deterministic: block (CS_X, CS_Y) owns
// CS_X * 8 columns over all rows; thread (x, y) adds rows y, y + CS_Y, ...
// in order, then a fixed-shape tree over y in shared memory.  No atomics,
// so repeated calls give identical bits.
constexpr int CS_X = 4, CS_Y = 128;

__global__ void __launch_bounds__(CS_X * CS_Y) colsum_kernel(const __nv_bfloat16* __restrict__ x,
                                                            long long rows, int h,
                                                            float* __restrict__ out, int accumulate) {
    pdl_trigger();
    pdl_wait();
    __shared__ float part[CS_Y][CS_X * 8 + 1];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int col = (blockIdx.x * CS_X + tx) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (col < h) {
        long long r = ty;
        for (; r + 3 * CS_Y < rows; r += 4 * CS_Y) {
            uint4 u[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) u[k] = *reinterpret_cast<const uint4*>(x + (r + k * CS_Y) * h + col);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = unpack_bf16x2(w[e]);
                    acc[2 * e] += f.x;
                    acc[2 * e + 1] += f.y;
                }
            }
        }
        for (; r < rows; r += CS_Y) {
            const uint4 u = *reinterpret_cast<const uint4*>(x + r * h + col);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = unpack_bf16x2(w[e]);
                acc[2 * e] += f.x;
                acc[2 * e + 1] += f.y;
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) part[ty][tx * 8 + e] = acc[e];
    __syncthreads();
    for (int sh = CS_Y / 2; sh > 0; sh >>= 1) {
        if (ty < sh) {
#pragma unroll
            for (int e = 0; e < 8; ++e) part[ty][tx * 8 + e] += part[ty + sh][tx * 8 + e];
        }
        __syncthreads();
    }
    if (ty == 0 && col < h) {
#pragma unroll
        for (int e = 0; e < 8; ++e) out[col + e] = (accumulate ? out[col + e] : 0.f) + part[0][tx * 8 + e];
    }
}

}  // namespace

namespace tpi {

int device_sm_count() {
    static int counts[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 1;
    if (!counts[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        counts[dev] = n > 0 ? n : 1;
    }
    return counts[dev];
}

int reduce_launch(const void* partials, int partial_f32, int t, int64_t n, int h, const void* bias,
                  const void* residual, void* out, cudaStream_t stream, std::string* err) {
    if (n == 0) return TP_OK;
    const long long nvec = n / 8;
    long long blocks = (nvec + RED_THREADS - 1) / RED_THREADS;
    blocks = std::min<long long>(blocks, (long long)device_sm_count() * 8);
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(bias);
    const __nv_bfloat16* r = reinterpret_cast<const __nv_bfloat16*>(residual);
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
#define TP_RED(TT, FF) \
    launch_pdl(reduce_kernel<TT, FF>, dim3((unsigned)blocks), dim3(RED_THREADS), 0, stream, partials, t, n, h, b, r, o)
    if (partial_f32) {
        switch (t) {
            case 1: TP_RED(1, true); break;
            case 2: TP_RED(2, true); break;
            case 4: TP_RED(4, true); break;
            case 8: TP_RED(8, true); break;
            default: TP_RED(0, true); break;
        }
    } else {
        switch (t) {
            case 1: TP_RED(1, false); break;
            case 2: TP_RED(2, false); break;
            case 4: TP_RED(4, false); break;
            case 8: TP_RED(8, false); break;
            default: TP_RED(0, false); break;
        }
    }
#undef TP_RED
    return check_launch("reduce kernel", err);
}

int reduce_norm_launch(const void* partials, int partial_f32, int t, int64_t rows, int h,
                       const void* residual, void* h1, void* xn, float eps, cudaStream_t stream,
                       std::string* err, int64_t sp_batch, int64_t sp_seq, int sp_t) {
    if (rows == 0) return TP_OK;
    const long long n = rows * (long long)h;
    const __nv_bfloat16* r = reinterpret_cast<const __nv_bfloat16*>(residual);
    auto* h1p = reinterpret_cast<__nv_bfloat16*>(h1);
    auto* xnp = reinterpret_cast<__nv_bfloat16*>(xn);
    if (partial_f32)
        launch_pdl(row_kernel<true, true>, dim3((unsigned)rows), dim3(ROW_THREADS), 0, stream, partials, t, n, h,
                   r, h1p, xnp, eps, sp_batch, sp_seq, sp_t);
    else
        launch_pdl(row_kernel<true, false>, dim3((unsigned)rows), dim3(ROW_THREADS), 0, stream, partials, t, n,
                   h, r, h1p, xnp, eps, sp_batch, sp_seq, sp_t);
    return check_launch("reduce+norm kernel", err);
}

int rmsnorm_launch(const void* x, int64_t rows, int h, float eps, void* y, cudaStream_t stream,
                   std::string* err) {
    if (rows == 0) return TP_OK;
    const long long n = rows * (long long)h;
    launch_pdl(row_kernel<false, true>, dim3((unsigned)rows), dim3(ROW_THREADS), 0, stream,
               static_cast<const void*>(nullptr), 0, n, h, reinterpret_cast<const __nv_bfloat16*>(x),
               static_cast<__nv_bfloat16*>(nullptr), reinterpret_cast<__nv_bfloat16*>(y), eps, 0LL, 0LL, 0);
    return check_launch("rmsnorm kernel", err);
}

int row_sumsq_launch(const void* x, int64_t rows, int h, float* ss, float* zero,
                     cudaStream_t stream, std::string* err) {
    if (rows == 0) return TP_OK;
    const long long blocks = (rows + SS_WARPS - 1) / SS_WARPS;
    launch_pdl(row_sumsq_kernel, dim3((unsigned)blocks), dim3(SS_WARPS * 32), 0, stream,
               reinterpret_cast<const __nv_bfloat16*>(x), rows, h, ss, zero);
    return check_launch("row sum-of-squares kernel", err);
}

int sp_all_gather_launch(const void* sp, int64_t batch, int64_t seq, int t, int h, void* full,
                         cudaStream_t stream, std::string* err) {
    const long long rows = batch * seq;
    if (rows == 0) return TP_OK;
    launch_pdl(sp_all_gather_kernel, dim3((unsigned)((rows + AG_WARPS - 1) / AG_WARPS)), dim3(AG_WARPS * 32), 0,
               stream, reinterpret_cast<const __nv_bfloat16*>(sp), rows, h, batch, seq, t,
               reinterpret_cast<__nv_bfloat16*>(full));
    return check_launch("all-gather kernel", err);
}

int sp_split_launch(const void* full, int64_t batch, int64_t seq, int t, int h, void* sp,
                    cudaStream_t stream, std::string* err) {
    const long long rows = batch * seq;
    if (rows == 0) return TP_OK;
    launch_pdl(sp_split_kernel, dim3((unsigned)((rows + AG_WARPS - 1) / AG_WARPS)), dim3(AG_WARPS * 32), 0,
               stream, reinterpret_cast<const __nv_bfloat16*>(full), rows, h, batch, seq, t,
               reinterpret_cast<__nv_bfloat16*>(sp));
    return check_launch("split kernel", err);
}

int rmsnorm_bwd_launch(const void* x, const void* g, const void* res, int64_t rows, int h, float eps,
                       void* out, cudaStream_t stream, std::string* err) {
    if (rows == 0) return TP_OK;
    const int nv = h / 8;
    const __nv_bfloat16* X = reinterpret_cast<const __nv_bfloat16*>(x);
    const __nv_bfloat16* G = reinterpret_cast<const __nv_bfloat16*>(g);
    const __nv_bfloat16* R = reinterpret_cast<const __nv_bfloat16*>(res);
    __nv_bfloat16* O = reinterpret_cast<__nv_bfloat16*>(out);
    const unsigned grid = static_cast<unsigned>(rows);
    if (nv <= RB_THREADS) launch_pdl(rmsnorm_bwd_kernel<1>, dim3(grid), dim3(RB_THREADS), 0, stream, X, G, R, h, eps, O);
    else if (nv <= 2 * RB_THREADS)
        launch_pdl(rmsnorm_bwd_kernel<2>, dim3(grid), dim3(RB_THREADS), 0, stream, X, G, R, h, eps, O);
    else if (nv <= 4 * RB_THREADS)
        launch_pdl(rmsnorm_bwd_kernel<4>, dim3(grid), dim3(RB_THREADS), 0, stream, X, G, R, h, eps, O);
    else if (nv <= 8 * RB_THREADS)
        launch_pdl(rmsnorm_bwd_kernel<8>, dim3(grid), dim3(RB_THREADS), 0, stream, X, G, R, h, eps, O);
    else {
        if (err) *err = "RMSNorm backward supports hidden <= 8192";
        return TP_ERR_UNSUPPORTED;
    }
    return check_launch("RMSNorm backward kernel", err);
}

int colsum_launch(const void* x, int64_t rows, int h, float* out, int accumulate,
                  cudaStream_t stream, std::string* err) {
    if (h == 0) return TP_OK;
    const unsigned gx = static_cast<unsigned>((h / 8 + CS_X - 1) / CS_X);
    launch_pdl(colsum_kernel, dim3(gx), dim3(CS_X, CS_Y), 0, stream, reinterpret_cast<const __nv_bfloat16*>(x),
               static_cast<long long>(rows), h, out, accumulate);
    return check_launch("column-sum kernel", err);
}

int selftest_timeout_launch(unsigned* status, uint64_t timeout_ns, cudaStream_t stream,
                            std::string* err) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return check_launch("self-test kernel", err);
}

}  // namespace tpi
