// tp_attn.cu -- causal GQA attention of every shard's heads on sm_103a
// tensor cores (tcgen05 / TMEM), fed by TMA.
//
// Source: "텐서 병렬화" (itwiki, Tensor parallelism), section "셀프 어텐션"
// (self-attention): heads are independent, so with Q/K/V split by columns
// each shard computes attention for its a/t query heads with no
// communication; with grouped-query attention the KV heads are split too,
// and replicated when there are fewer KV heads than shards.
//
// Reading of what the page leaves open: scale 1/sqrt(d), causal mask
// (key position <= query position) within each sequence, fp32 softmax with
// a running maximum subtracted, no dropout, no rotary embedding.
//
// Work item: 128 query rows of one query head and sequence.  A persistent
// grid of two CTAs per SM (7 warps, 256 TMEM columns and ~105 KB of shared
// memory each) walks the items longest first, in rounds of alternating
// direction (item_at), so one CTA's softmax overlaps the other's
// tensor-core work and the next item's loads overlap the current item's
// last blocks:
//   warp 0      TMA: Q once, then K and V blocks of 64 keys (2-stage rings,
//               K one block ahead) from the shard-blocked QKV buffer; an L2
//               prefetch of the next item's Q.
//   warp 1      TMEM owner and S issuer: S = Q K^T (128 x 64, fp32, two TMEM
//               buffers so S of block j+1 is computed while the softmax works
//               on block j).
//   warp 2      PV issuer: O += P V with P read from TMEM (tcgen05.mma with
//               the A operand in tensor memory) and V used as an MN-major
//               operand straight from its [key][d] layout.
//               A thread issues one tcgen05.mma about every 100 cycles
//               whatever its size (measured on GB300), while an S or PV step
//               here is 30 to 60 cycles of math, so the two products have
//               an issuing thread each.
//   warps 3..6  one query row per thread (TMEM lane = row): read the S row,
//               apply the causal mask, online softmax with exp2, write P as
//               bf16 over the first half of the same S buffer (tcgen05.st),
//               rescale the O row in TMEM when its reference maximum moves,
//               and finally write O / l as bf16 through a per-warp shared-
//               memory box and a TMA store.
// A buffer is reused for S of block j+2 once the PV of block j, which reads
// its P, has completed; the softmax warps wait for the previous PV to
// complete only when they rescale O in place.
// The reference maximum of a row only moves when the block maximum exceeds
// it by more than 2^8 (in the exp2 domain), so most blocks need no O
// rescale; P then stays below 256, well inside bf16 and fp32 range.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <string>

#include "tp_device.cuh"
#include "tp_internal.h"
#include "tp_packed.cuh"

namespace {

using namespace tpk;

constexpr int QB = 128;  // query rows per CTA (UMMA M, TMEM lanes)
constexpr int KB = 64;   // keys per block (UMMA N of S, UMMA K of PV)
constexpr int NTHREADS = 224;
constexpr int QBOX = QB * 128;  // TMA box of Q: 128 rows x 64 bf16 (16 KB)
constexpr int KBOX = KB * 128;  // TMA box of K or V: 64 rows x 64 bf16 (8 KB)
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 of the allowed growth of P

enum {
    B_Q_FULL = 0,
    B_K_FULL = 1,    // x2 (K ring)
    B_K_EMPTY = 3,   // x2
    B_V_FULL = 5,    // x2 (V ring)
    B_V_EMPTY = 7,   // x2
    B_S_FULL = 9,    // x2 (S / P buffers in TMEM)
    B_PV_DONE = 11,  // x2: the PV MMA that read P from buffer i has completed
    B_P_FULL = 13,   // x2 (per S buffer): its 4 softmax warps wrote P
    B_O_FULL = 15,
    B_DRAIN = 16,    // x2: one per issuing thread
    B_Q_EMPTY = 18,  // the item's S products are done with Q
    B_O_EMPTY = 19,  // the item's epilogue has read O (4 softmax warps)
    NUM_BARS = 20
};

// Per-CTA dynamic shared memory when two CTAs share an SM: (228 KB - 2 x
// 1 KB reserved) / 2.
constexpr int TWO_CTA_SMEM = 115712;

// Shared memory of one CTA (two CTAs share an SM):
//   Q [128][d] | K ring 2 x [64][d] | V ring 2 x [64][d] | O staging | barriers
// (P lives in TMEM, over the first half of its S buffer).  The kernel checks
// at run time that its 1024-aligned layout fits the allocation and
// otherwise stops with an error flag, touching nothing.
constexpr int STG_BOX = 32 * 64;  // 32 rows x 32 bf16 (64-byte swizzle)

template <int D>
struct Layout {
    static constexpr int QT = QB * D * 2;
    static constexpr int KT = KB * D * 2;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = QT;
    static constexpr int V_OFF = K_OFF + 2 * KT;
    static constexpr int STG_OFF = V_OFF + 2 * KT;  // O staging: one 32 x 32 bf16 box per softmax warp
    static constexpr int BAR_OFF = STG_OFF + 4 * STG_BOX;
    static constexpr int DATA = BAR_OFF + 8 * NUM_BARS + 16;
    static constexpr int SMEM = DATA + 1024 <= TWO_CTA_SMEM ? DATA + 1024 : TWO_CTA_SMEM;
    static constexpr int TMEM_COLS = 2 * KB + D <= 256 ? 256 : 512;  // S0 | S1 | O
};

struct AttnParams {
    CUtensorMap map_q;   // the QKV buffer: dims {t * W, tokens}, box {64, 128}
    CUtensorMap map_kv;  // the same buffer, box {64, 64}
    CUtensorMap map_o;   // O as {ld_o, seq, batch}, box {32, 32, 1}, 64-byte swizzle; rows
                         // past a sequence's end are outside it and not written
    int o_tma;           // 1: O leaves by TMA stores through map_o
    __nv_bfloat16* o;
    long long ld_o;
    int seq, heads, kv_heads, t, heads_per_shard, shard_w, q_w, kv_w;
    float scale_log2;  // log2(e) / sqrt(d)
    float* lse;        // nullable: base-2 log-sum-exp per (head, sequence, row)
    long long seq_pad;
    int batch;
    unsigned* status;
    unsigned long long timeout_ns;
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 200000000ull) break;  // 200 ms
    }
}

// 2^x with the SFU's approximate exp2 (PTX ex2.approx.ftz.f32: relative
// error about 2^-22, -inf -> +0); used for the softmax numerators.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


// Tiled TMA store of a 3-D box (elements outside the map are not written).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1,
                                             int32_t c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// Bring a box of a tensor map into L2 without writing shared memory.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// One work item: 128 query rows (tile qb) of query head j in sequence b.
// Items are numbered longest first: item w has tile nqb - 1 - w / (heads *
// batch), so each round of gridDim.x items has rows of one length.
struct Item {
    int q0, nkb, tok0, j, b;
    int qcol, kcol, vcol;
};

template <int D>
__device__ __forceinline__ Item item_of(const AttnParams& p, int w) {
    const int nqb = (p.seq + QB - 1) / QB;
    const int hb = p.heads * p.batch;
    const int qi = w / hb;
    const int r = w - qi * hb;
    Item x;
    x.j = r % p.heads;
    x.b = r / p.heads;
    const int qb = nqb - 1 - qi;
    const int shard = x.j / p.heads_per_shard;
    const int jl = x.j - shard * p.heads_per_shard;
    const int g = x.j / (p.heads / p.kv_heads);
    const int kv0 = (p.kv_heads >= p.t) ? shard * (p.kv_heads / p.t) : (shard * p.kv_heads) / p.t;
    x.qcol = shard * p.shard_w + jl * D;
    x.kcol = shard * p.shard_w + p.q_w + (g - kv0) * D;
    x.vcol = x.kcol + p.kv_w;
    x.tok0 = x.b * p.seq;
    x.q0 = qb * QB;
    // causal: keys 0 .. q0+127, and never past the sequence
    x.nkb = min((x.q0 + QB + KB - 1) / KB, (p.seq + KB - 1) / KB);
    return x;
}

// The k-th item of CTA c in a grid of g CTAs: rounds of g items, taken
// left to right in even rounds and right to left in odd ones, so the CTA
// that took a round's longest item takes the next round's shortest.  Item
// lengths fall with the index; a plain c, c + g, ... order gives CTA 0 the
// longest item of every round (one sequence of 2048 tokens, 512 items on
// 304 CTAs: 46 key blocks for CTA 0 against 28.6 on average).
__device__ __forceinline__ int item_at(int k, int c, int g) { return k * g + ((k & 1) ? g - 1 - c : c); }

// Persistent: CTA c takes items item_at(0, c), item_at(1, c), ...  Every
// role walks the same item list; K/V ring stages, S buffers and their barrier phases run on
// one block count across items, so the next item's Q and first K/V blocks
// load while the current item finishes.
template <int D>
__global__ void __launch_bounds__(NTHREADS, 2) attn_tc_kernel(const __grid_constant__ AttnParams p) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + L::Q_OFF, sK = base + L::K_OFF, sV = base + L::V_OFF;
    const uint32_t bar0 = base + L::BAR_OFF;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::BAR_OFF + 8 * NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    if (base - raw + static_cast<uint32_t>(L::DATA) > static_cast<uint32_t>(L::SMEM)) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, kStatusLayout);
        return;  // the aligned layout does not fit: nothing was touched
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = ((p.seq + QB - 1) / QB) * p.heads * p.batch;
    const int w0 = static_cast<int>(blockIdx.x), dw = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        mbar_init(bar(B_Q_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_K_FULL + s), 1);
            mbar_init(bar(B_K_EMPTY + s), 1);
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_PV_DONE + s), 1);
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 1);
        }
        // One P_FULL per S buffer: a warp a block ahead of the others
        // arrives on the other barrier, never on the phase they complete.
        mbar_init(bar(B_P_FULL), 4);
        mbar_init(bar(B_P_FULL + 1), 4);
        mbar_init(bar(B_O_FULL), 1);
        mbar_init(bar(B_O_EMPTY), 4);
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_DRAIN + 1), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.map_q);
        tma_prefetch_desc(&p.map_kv);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The next kernel may start its prologue on SMs this grid leaves; this
    // one touches global memory only once the previous kernel is done.
    pdl_trigger();
    pdl_wait();

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        // Per item: Q (once the previous item's S products are done with
        // it), K0, then for each block kb: K(kb+1), V(kb).  Both rings are
        // 2-stage, so a V load waits for the PV MMA two blocks back and its
        // latency stays off the PV critical path.
        if (lane == 0) {
            bool ok = true, q_issued = false;
            uint32_t kissued = 0, kpar = 0, vissued = 0, vpar = 0, qpar = 0;
            int gb = 0;  // blocks of earlier items
            auto load_kv = [&](const Item& x, int kb, bool is_v) -> bool {
                const int n = gb + kb;  // ring position
                const int st = n & 1;
                const uint32_t ph = static_cast<uint32_t>(n >> 1) & 1u;
                const int e = is_v ? B_V_EMPTY : B_K_EMPTY, f = is_v ? B_V_FULL : B_K_FULL;
                if (!mbar_wait(bar(e + st), ph ^ 1u, abort_flag, p.status, p.timeout_ns)) return false;
                mbar_arrive_expect_tx(bar(f + st), L::KT);
                const uint32_t dst = (is_v ? sV : sK) + st * L::KT;
                const int col = is_v ? x.vcol : x.kcol;
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d(dst + c * KBOX, &p.map_kv, bar(f + st), col + 64 * c, x.tok0 + kb * KB);
                if (is_v) {
                    vissued |= 1u << st;
                    vpar = (vpar & ~(1u << st)) | (ph << st);
                } else {
                    kissued |= 1u << st;
                    kpar = (kpar & ~(1u << st)) | (ph << st);
                }
                return true;
            };
            int li = 0;
            for (int w; ok && (w = item_at(li, w0, dw)) < n_items; ++li) {
                const Item x = item_of<D>(p, w);
                // The next item's Q is read from HBM for the first time: start
                // that read now, so its TMA load later hits L2.
                if (item_at(li + 1, w0, dw) < n_items) {
                    const Item y = item_of<D>(p, item_at(li + 1, w0, dw));
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) tma_prefetch_l2_2d(&p.map_q, y.qcol + 64 * c, y.tok0 + y.q0);
                }
                if (li > 0 && !mbar_wait(bar(B_Q_EMPTY), static_cast<uint32_t>(li - 1) & 1u, abort_flag, p.status,
                                         p.timeout_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(B_Q_FULL), L::QT);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d(sQ + c * QBOX, &p.map_q, bar(B_Q_FULL), x.qcol + 64 * c, x.tok0 + x.q0);
                q_issued = true;
                qpar = static_cast<uint32_t>(li) & 1u;
                ok = load_kv(x, 0, false);
                for (int kb = 0; kb < x.nkb && ok; ++kb) {
                    if (kb + 1 < x.nkb && !(ok = load_kv(x, kb + 1, false))) break;
                    ok = load_kv(x, kb, true);
                }
                gb += x.nkb;
            }
            if (!ok) {
                if (q_issued) drain_wait(bar(B_Q_FULL), qpar);
                for (int s = 0; s < 2; ++s) {
                    if (kissued & (1u << s)) drain_wait(bar(B_K_FULL + s), (kpar >> s) & 1u);
                    if (vissued & (1u << s)) drain_wait(bar(B_V_FULL + s), (vpar >> s) & 1u);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- S issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(QB, KB);
            // Descriptors built once: a step adds its constant offset (in
            // 16-byte units) to the start-address field.
            const uint64_t qdesc = sdesc_sw128(sQ);
            const uint64_t kdesc0 = sdesc_sw128(sK), kdesc1 = sdesc_sw128(sK + L::KT);
            bool ok = true;
            int gb = 0, li = 0;
            for (int w; ok && (w = item_at(li, w0, dw)) < n_items; ++li) {
                const int nkb = item_of<D>(p, w).nkb;
                if (!mbar_wait(bar(B_Q_FULL), static_cast<uint32_t>(li) & 1u, abort_flag, p.status, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                for (int kb = 0; kb < nkb && ok; ++kb, ++gb) {
                    const int st = gb & 1;
                    // Buffer st held S and then P of block gb - 2: its PV must
                    // have read that P before this S overwrites it.
                    if (gb >= 2 && !mbar_wait(bar(B_PV_DONE + st), static_cast<uint32_t>((gb - 2) >> 1) & 1u,
                                              abort_flag, p.status, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(bar(B_K_FULL + st), static_cast<uint32_t>(gb >> 1) & 1u, abort_flag, p.status,
                                   p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + st * KB;
                    const uint64_t kdesc = st ? kdesc1 : kdesc0;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        constexpr uint32_t unit = 16;
                        const uint32_t a_off = ((ks >> 2) * QBOX + (ks & 3) * 32) / unit;
                        const uint32_t b_off = ((ks >> 2) * KBOX + (ks & 3) * 32) / unit;
                        umma_bf16(d_tmem, qdesc + a_off, kdesc + b_off, idesc_s, ks > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(B_K_EMPTY + st));
                    umma_commit(bar(B_S_FULL + st));
                }
                // Q may be reloaded once this item's S products are done.
                if (ok) umma_commit(bar(B_Q_EMPTY));
            }
            if (!ok) {
                umma_commit(bar(B_DRAIN));
                drain_wait(bar(B_DRAIN), 0);
            }
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------- PV issuer
        if (lane == 0) {
            constexpr uint32_t idesc_o = idesc_bf16_f32_bmn(QB, D);
            const uint64_t vdesc0 = sdesc_sw128_mn(sV, KBOX, 1024), vdesc1 = sdesc_sw128_mn(sV + L::KT, KBOX, 1024);
            bool ok = true;
            int gb = 0, li = 0;
            for (int w; ok && (w = item_at(li, w0, dw)) < n_items; ++li) {
                const int nkb = item_of<D>(p, w).nkb;
                for (int kb = 0; kb < nkb && ok; ++kb, ++gb) {
                    const int vst = gb & 1;
                    if (!mbar_wait(bar(B_P_FULL + vst), static_cast<uint32_t>(gb >> 1) & 1u, abort_flag, p.status,
                                   p.timeout_ns) ||
                        !mbar_wait(bar(B_V_FULL + vst), static_cast<uint32_t>(gb >> 1) & 1u, abort_flag, p.status,
                                   p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    // The first PV of an item overwrites O: the previous
                    // item's epilogue must have read it.
                    if (kb == 0 && li > 0 &&
                        !mbar_wait(bar(B_O_EMPTY), static_cast<uint32_t>(li - 1) & 1u, abort_flag, p.status,
                                   p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // P of block gb: bf16 in the first KB/2 columns of S buffer
                    // gb & 1, 16 keys (8 columns) per UMMA.
                    const uint64_t vdesc = vst ? vdesc1 : vdesc0;
                    const uint32_t pcol = tmem + vst * KB;
                    const uint32_t acc0 = kb > 0 ? 1u : 0u;
#pragma unroll
                    for (int ks = 0; ks < KB / 16; ++ks)
                        umma_bf16_ts(tmem + 2 * KB, pcol + ks * 8, vdesc + (ks * 16 * 128) / 16, idesc_o,
                                     ks > 0 ? 1u : acc0);
                    umma_commit(bar(B_V_EMPTY + vst));
                    umma_commit(bar(B_PV_DONE + vst));
                }
                if (ok) umma_commit(bar(B_O_FULL));
            }
            if (!ok) {
                umma_commit(bar(B_DRAIN + 1));
                drain_wait(bar(B_DRAIN + 1), 0);
            }
        }
    } else {
        // ---------------------------------------------------------- softmax / epilogue
        const int q = warp & 3;  // TMEM lane quadrant
        const int r = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        bool ok = true;
        int gb = 0, li = 0;
        for (int w; ok && (w = item_at(li, w0, dw)) < n_items; ++li) {
            const Item x = item_of<D>(p, w);
            const int q0 = x.q0;
            const int qpos = q0 + r;
            float m_ref = -INFINITY, l_sum = 0.0f;
            for (int kb = 0; kb < x.nkb; ++kb, ++gb) {
                const int st = gb & 1;
                const bool got = mbar_wait(bar(B_S_FULL + st), static_cast<uint32_t>(gb >> 1) & 1u, abort_flag,
                                           p.status, p.timeout_ns);
                __syncwarp();
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t s[KB];
#pragma unroll
                for (int c = 0; c < KB / 32; ++c)
                    tmem_ld32(tmem + lane_off + st * KB + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
                tmem_ld_wait();

                // Keys k0 + c with c > lim are masked: later than the query
                // (causal) or past the sequence end.
                const int k0 = kb * KB;
                const int lim = min(qpos, p.seq - 1) - k0;
                if (lim < KB - 1) {
#pragma unroll
                    for (int c = 0; c < KB; ++c)
                        if (c > lim) s[c] = __float_as_uint(-INFINITY);
                }
                // Row max with 8 independent chains of three-way maxima (one
                // softmax warp per SM sub-partition and CTA leaves little to
                // hide a serial chain).
                float mx8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(__uint_as_float(s[e]), __uint_as_float(s[8 + e]));
#pragma unroll
                for (int c = 16; c < KB; c += 16)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        mx8[e] = max3(mx8[e], __uint_as_float(s[c + e]), __uint_as_float(s[c + 8 + e]));
                const float mx = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]),
                                      fmaxf(mx8[6], mx8[7]));
                const float mxs = mx * p.scale_log2;
                float alpha = 1.0f;
                bool rescale = false;
                if (mxs > m_ref + RESCALE_THRESHOLD) {
                    alpha = exp2f(m_ref - mxs);  // 0 on the first block
                    m_ref = mxs;
                    rescale = kb > 0;
                }
                const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
                const uint64_t neg2 = f2_pack(-m_ref, -m_ref);
                uint64_t acc[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] = f2_pack(0.0f, 0.0f);
                uint32_t pk[KB / 2];
#pragma unroll
                for (int c = 0; c < KB / 2; ++c) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), scale2, neg2),
                              x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    acc[c & 3] = f2_add(acc[c & 3], f2_pack(p0, p1));
                    pk[c] = pack_bf16x2(p0, p1);
                }
                float sum8[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) f2_unpack(acc[e], sum8[2 * e], sum8[2 * e + 1]);
                const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
                                  ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
                l_sum = l_sum * alpha + sum;

                if (__any_sync(0xffffffffu, rescale)) {
                    // O is rescaled in place: the PV of the previous block must be done.
                    const int pb = gb - 1;
                    const bool got2 = mbar_wait(bar(B_PV_DONE + (pb & 1)), static_cast<uint32_t>(pb >> 1) & 1u,
                                                abort_flag, p.status, p.timeout_ns);
                    __syncwarp();
                    if (!__all_sync(0xffffffffu, got2)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        const uint32_t ta = tmem + lane_off + 2 * KB + c * 32;
                        tmem_ld32(ta, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(ta, o);
                    }
                    tmem_st_wait();
                }
                // P row r over its S row in TMEM: 64 keys as 32 packed columns.
                tmem_st32(tmem + lane_off + st * KB, pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_P_FULL + st));
            }
            if (!ok) break;
            const bool got = mbar_wait(bar(B_O_FULL), static_cast<uint32_t>(li) & 1u, abort_flag, p.status,
                                       p.timeout_ns);
            __syncwarp();
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv = 1.0f / l_sum;
            if (p.lse && qpos < p.seq)
                p.lse[(static_cast<long long>(x.j) * p.batch + x.b) * p.seq_pad + qpos] = m_ref + log2f(l_sum);
            __nv_bfloat16* orow = p.o + static_cast<long long>(x.tok0 + qpos) * p.ld_o +
                                  static_cast<long long>(x.j) * D;
            // O / l as bf16, 32 columns at a time.  With a TMA map the warp
            // writes its 32 rows into its shared-memory box (16-byte piece u
            // of row l at l * 64 + (u ^ ((l / 2) % 4)) * 16) and lane 0
            // stores the box; otherwise each thread stores its row.
            const int row0 = q0 + q * 32;
            const uint32_t box = base + L::STG_OFF + static_cast<uint32_t>(q) * STG_BOX;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + 2 * KB + c * 32, o);
                tmem_ld_wait();
                if (p.o_tma) {
                    if (lane == 0) bulk_wait_group_read0();  // the box's previous store has read it
                    __syncwarp();
                    const uint32_t srow = box + static_cast<uint32_t>(lane) * 64u;
                    const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint32_t wv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            wv[e] = pack_bf16x2(__uint_as_float(o[u * 8 + 2 * e]) * inv,
                                                __uint_as_float(o[u * 8 + 2 * e + 1]) * inv);
                        st_shared_v4(srow + ((static_cast<uint32_t>(u) ^ sw) << 4), wv[0], wv[1], wv[2], wv[3]);
                    }
                    fence_proxy_async_smem();  // visible to the TMA engine
                    __syncwarp();
                    if (lane == 0 && row0 < p.seq) {
                        tma_store_3d(&p.map_o, box, x.j * D + c * 32, row0, x.b);
                        bulk_commit_group();
                    }
                } else if (qpos < p.seq) {
#pragma unroll
                    for (int g8 = 0; g8 < 4; ++g8) {
                        uint32_t wv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            wv[e] = pack_bf16x2(__uint_as_float(o[g8 * 8 + 2 * e]) * inv,
                                                __uint_as_float(o[g8 * 8 + 2 * e + 1]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + g8 * 8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                }
            }
            // O has been read from TMEM: the next item's first PV may
            // overwrite it.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_O_EMPTY));
        }
        // The O stores must have completed before the CTA exits.
        if (lane == 0) bulk_wait_group0();
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int D>
int launch_d(const tpi::AttnArgs& a, cudaStream_t stream, std::string* err) {
    AttnParams p;
    memset(&p, 0, sizeof(p));
    void* fn_ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn_ptr, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess || !fn_ptr) {
        if (err) *err = "cuTensorMapEncodeTiled is not available from the driver";
        return TP_ERR_CUDA;
    }
    EncodeTiledFn encode = reinterpret_cast<EncodeTiledFn>(fn_ptr);
    const long long tokens = static_cast<long long>(a.batch) * a.seq;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.ld_qkv), static_cast<cuuint64_t>(tokens)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.ld_qkv) * 2};
    cuuint32_t estr[2] = {1, 1};
    for (int m = 0; m < 2; ++m) {
        cuuint32_t box[2] = {64, m == 0 ? static_cast<cuuint32_t>(QB) : static_cast<cuuint32_t>(KB)};
        CUresult r = encode(m == 0 ? &p.map_q : &p.map_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                            const_cast<void*>(a.QKV), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            if (err) *err = "cuTensorMapEncodeTiled (attention QKV) failed: " + std::to_string((int)r);
            return TP_ERR_CUDA;
        }
    }
    // O as {columns, position, sequence} for the TMA stores of the epilogue
    // (16-byte aligned base and row stride); otherwise per-thread stores.
    if (a.ld_o % 8 == 0 && (reinterpret_cast<uintptr_t>(a.O) & 15u) == 0) {
        cuuint64_t odims[3] = {static_cast<cuuint64_t>(a.ld_o), static_cast<cuuint64_t>(a.seq),
                               static_cast<cuuint64_t>(a.batch)};
        cuuint64_t ostr[2] = {static_cast<cuuint64_t>(a.ld_o) * 2,
                              static_cast<cuuint64_t>(a.ld_o) * 2 * static_cast<cuuint64_t>(a.seq)};
        cuuint32_t obox[3] = {32, 32, 1};
        cuuint32_t oestr[3] = {1, 1, 1};
        CUresult r = encode(&p.map_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.O, odims, ostr, obox, oestr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            if (err) *err = "cuTensorMapEncodeTiled (attention O) failed: " + std::to_string((int)r);
            return TP_ERR_CUDA;
        }
        p.o_tma = 1;
    }
    p.o = reinterpret_cast<__nv_bfloat16*>(a.O);
    p.ld_o = a.ld_o;
    p.seq = a.seq;
    p.heads = a.heads;
    p.kv_heads = a.kv_heads;
    p.t = a.t;
    p.heads_per_shard = a.heads / a.t;
    p.shard_w = static_cast<int>(a.shard_w);
    p.q_w = static_cast<int>(a.q_w);
    p.kv_w = static_cast<int>(a.kv_w);
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    p.lse = a.lse;
    p.seq_pad = a.seq_pad;
    p.batch = a.batch;
    p.status = a.status;
    p.timeout_ns = a.timeout_ns;
    const int smem = Layout<D>::SMEM;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            if (err) *err = std::string("cudaFuncSetAttribute(attn): ") + cudaGetErrorString(e);
            return TP_ERR_CUDA;
        }
        configured[dev] = true;
    }
    // Persistent grid: two CTAs per SM, or fewer when there are fewer items.
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    const long long n_items = static_cast<long long>((a.seq + QB - 1) / QB) * a.heads * a.batch;
    dim3 grid(static_cast<unsigned>(std::min<long long>(n_items, 2LL * sms)), 1, 1);
    cudaError_t e = tpi::launch_pdl(attn_tc_kernel<D>, grid, dim3(NTHREADS), smem, stream, p);
    if (e == cudaSuccess) e = cudaGetLastError();
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
