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
// grid of one CTA per SM (11 warps, all 512 TMEM columns, ~195 KB of shared
// memory at d = 128) walks the items longest first, in rounds of
// alternating direction (item_at), and the next item's loads overlap the
// current item's last blocks:
//   warp 0      TMA: Q, then K and V blocks of 128 keys (2-stage rings, K one
//               block ahead) from the shard-blocked QKV buffer; the next
//               item's Q and first K take the place of K(nkb), and an L2
//               prefetch of the next item's Q goes out when an item starts.
//   warp 1      TMEM owner and S issuer: S = Q K^T (128 x 128, fp32) into
//               three TMEM buffers, so S of blocks j+1 and j+2 is computed
//               while the softmax works on block j.
//   warp 2      PV issuer: O += P V with P read from TMEM (tcgen05.mma with
//               the A operand in tensor memory) and V used as an MN-major
//               operand straight from its [key][d] layout.
//               One thread issues a 128 x 128 x 16 step about every 70
//               cycles, about its math time, so the two products have an
//               issuing thread each and run side by side.
//   warps 3..10 two warps per TMEM lane quadrant, one query row per thread
//               (TMEM lane = row), each warp half of a block's keys: read
//               the S half-row, apply the causal mask, agree on the row
//               maximum with the other half through shared memory, online
//               softmax with exp2, write P as bf16 over the first half of
//               the same S buffer (tcgen05.st), rescale its half of the O
//               row in TMEM when the row's reference maximum moves.  After
//               the next item's first block they write O / l as bf16
//               through per-warp shared-memory boxes and TMA stores.
// A buffer is reused for S of block j+3 once the PV of block j, which reads
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
constexpr int QBOX = QB * 128;  // TMA box of Q: 128 rows x 64 bf16 (16 KB)
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 of the allowed growth of P
constexpr int MAX_NS = 3;  // S buffers in TMEM, at most

enum {
    B_Q_FULL = 0,
    B_K_FULL = 1,    // x2 (K ring)
    B_K_EMPTY = 3,   // x2
    B_V_FULL = 5,    // x2 (V ring)
    B_V_EMPTY = 7,   // x2
    B_S_FULL = 9,    // x NS (S / P buffers in TMEM)
    B_PV_DONE = B_S_FULL + MAX_NS,   // x NS: the PV MMA that read P from buffer i has completed
    B_P_FULL = B_PV_DONE + MAX_NS,   // x NS (per S buffer): its softmax warps wrote P
    B_O_FULL = B_P_FULL + MAX_NS,
    B_DRAIN = B_O_FULL + 1,          // x2: one per issuing thread
    B_Q_EMPTY = B_DRAIN + 2,         // the item's S products are done with Q
    B_O_EMPTY = B_Q_EMPTY + 1,       // the item's epilogue has read O (all softmax warps)
    NUM_BARS = B_O_EMPTY + 1
};

// Per-CTA dynamic shared memory when two CTAs share an SM: (228 KB - 2 x
// 1 KB reserved) / 2.
constexpr int TWO_CTA_SMEM = 115712;

// Shared memory of one CTA:
//   Q [128][d] | K ring 2 x [KB][d] | V ring 2 x [KB][d] | O staging |
//   row-max / row-sum exchange | barriers
// (P lives in TMEM, over the first half of its S buffer).  The kernel checks
// at run time that its 1024-aligned layout fits the allocation and
// otherwise stops with an error flag, touching nothing.
constexpr int STG_BOX = 32 * 64;  // 32 rows x 32 bf16 (64-byte swizzle)

// The kernel's configuration: head dimension D, keys per block KB (UMMA N of
// S, UMMA K of PV), S buffers in TMEM NS (S of later blocks is computed while
// the softmax and the PV products of earlier ones run) and CTAs per SM.
template <int D_, int KB_, int NS_, int CTAS_, int SPLIT_>
struct Layout {
    static constexpr int D = D_, KB = KB_, NS = NS_, CTAS = CTAS_;
    // Softmax warps per TMEM lane quadrant (each takes KB / SPLIT keys of a block).
    static constexpr int SPLIT = SPLIT_;
    // Warp 0 TMA, warp 1 S issuer, warp 2 PV issuer, then 4 * SPLIT softmax warps.
    static constexpr int NTHREADS = 96 + 128 * SPLIT;
    static constexpr int KBOX = KB * 128;  // TMA box of K or V: KB rows x 64 bf16
    static constexpr int QT = QB * D * 2;
    static constexpr int KT = KB * D * 2;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = QT;
    static constexpr int V_OFF = K_OFF + 2 * KT;
    // O staging: one 32 x 32 bf16 box per softmax warp and 32 columns of O,
    // so an item's stores never wait for each other.
    static constexpr int STG_OFF = V_OFF + 2 * KT;
    // Row maxima of the two block parities and row sums exchanged between
    // the softmax warps of a quadrant: [3][SPLIT][128] fp32.
    static constexpr int XCH_OFF = STG_OFF + 4 * (D / 32) * STG_BOX;
    static constexpr int BAR_OFF = XCH_OFF + 3 * SPLIT * QB * 4;
    static constexpr int DATA = BAR_OFF + 8 * NUM_BARS + 16;
    static constexpr int SMEM_CAP = CTAS == 2 ? TWO_CTA_SMEM : 232448;
    static constexpr int SMEM = DATA + 1024 <= SMEM_CAP ? DATA + 1024 : SMEM_CAP;
    static constexpr int O_COL = NS * KB;  // TMEM: S_0 | ... | S_(NS-1) | O
    static constexpr int TMEM_COLS = O_COL + D <= 256 ? 256 : 512;
    static_assert(NS >= 2 && NS <= MAX_NS && O_COL + D <= 512 && KB % 32 == 0, "configuration");
    static_assert((SPLIT == 1 || SPLIT == 2) && (KB / SPLIT) % 32 == 0 && (D / SPLIT) % 32 == 0, "split");
    static_assert(CTAS == 1 || TMEM_COLS <= 256, "two CTAs per SM share its 512 TMEM columns");
};

// Division by a run-time constant d with a multiply and a shift
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, the round-up method): with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1, n / d = (umulhi(n, m) + n) >> s for
// every n < 2^31.  Item decoding runs at each item start on the softmax
// warps' critical path, where a hardware-less integer division costs tens of
// instructions.
struct FastDiv {
    uint32_t m, s;
};
FastDiv make_fastdiv(uint32_t d) {
    FastDiv f{0, 0};
    while ((1ull << f.s) < d) ++f.s;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.s) - d)) / d + 1);
    return f;
}
__device__ __forceinline__ int fdiv(int n, FastDiv f) {
    return static_cast<int>((__umulhi(static_cast<uint32_t>(n), f.m) + static_cast<uint32_t>(n)) >> f.s);
}

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
    // Item decoding: divisors heads * batch, heads, heads per shard, query
    // heads per KV head and t; query tiles per sequence, key blocks per
    // sequence and KV heads per shard (when there are at least t).
    FastDiv f_hb, f_heads, f_hps, f_grp, f_t;
    int nqb, nkb_seq, kv_per_shard;
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

template <class L>
__device__ __forceinline__ Item item_of(const AttnParams& p, int w) {
    constexpr int D = L::D, KB = L::KB;
    const int qi = fdiv(w, p.f_hb);
    const int r = w - qi * (p.heads * p.batch);
    Item x;
    x.b = fdiv(r, p.f_heads);
    x.j = r - x.b * p.heads;
    const int qb = p.nqb - 1 - qi;
    const int shard = fdiv(x.j, p.f_hps);
    const int jl = x.j - shard * p.heads_per_shard;
    const int g = fdiv(x.j, p.f_grp);
    const int kv0 = (p.kv_heads >= p.t) ? shard * p.kv_per_shard : fdiv(shard * p.kv_heads, p.f_t);
    x.qcol = shard * p.shard_w + jl * D;
    x.kcol = shard * p.shard_w + p.q_w + (g - kv0) * D;
    x.vcol = x.kcol + p.kv_w;
    x.tok0 = x.b * p.seq;
    x.q0 = qb * QB;
    // causal: keys 0 .. q0+127, and never past the sequence
    x.nkb = min((x.q0 + QB + KB - 1) / KB, p.nkb_seq);
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
template <class L>
__global__ void __launch_bounds__(L::NTHREADS, L::CTAS) attn_tc_kernel(const __grid_constant__ AttnParams p) {
    constexpr int D = L::D, KB = L::KB, NS = L::NS, KBOX = L::KBOX;
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
    const int n_items = p.nqb * p.heads * p.batch;
    const int w0 = static_cast<int>(blockIdx.x), dw = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        mbar_init(bar(B_Q_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_K_FULL + s), 1);
            mbar_init(bar(B_K_EMPTY + s), 1);
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 1);
        }
        // One P_FULL per S buffer: a warp a block ahead of the others
        // arrives on another barrier, never on the phase they complete.
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_PV_DONE + s), 1);
            mbar_init(bar(B_P_FULL + s), 4 * L::SPLIT);
        }
        mbar_init(bar(B_O_FULL), 1);
        mbar_init(bar(B_O_EMPTY), 4 * L::SPLIT);
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
            // K or V block kb of item x, whose first block has ring position g0.
            auto load_kv = [&](const Item& x, int g0, int kb, bool is_v) -> bool {
                const int n = g0 + kb;  // ring position
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
            // Q of item number li (once the previous item's S products are done with Q).
            auto load_q = [&](const Item& x, int li) -> bool {
                if (li > 0 && !mbar_wait(bar(B_Q_EMPTY), static_cast<uint32_t>(li - 1) & 1u, abort_flag, p.status,
                                         p.timeout_ns))
                    return false;
                mbar_arrive_expect_tx(bar(B_Q_FULL), L::QT);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d(sQ + c * QBOX, &p.map_q, bar(B_Q_FULL), x.qcol + 64 * c, x.tok0 + x.q0);
                q_issued = true;
                qpar = static_cast<uint32_t>(li) & 1u;
                return true;
            };
            // Per item: for each block kb, K(kb + 1) then V(kb).  In place of
            // K(nkb) come the next item's Q and K(0), so they load while
            // the item's last blocks are still in flight rather than after
            // its last V.
            int li = 0;
            bool have = item_at(0, w0, dw) < n_items;
            Item x{};
            if (have) {
                x = item_of<L>(p, item_at(0, w0, dw));
                ok = load_q(x, 0) && load_kv(x, 0, 0, false);
            }
            for (; ok && have; ++li) {
                const int wn = item_at(li + 1, w0, dw);
                const bool has_next = wn < n_items;
                Item y{};
                if (has_next) {
                    y = item_of<L>(p, wn);
                    // The next item's Q is read from HBM for the first time:
                    // start that read now, so its TMA load later hits L2.
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) tma_prefetch_l2_2d(&p.map_q, y.qcol + 64 * c, y.tok0 + y.q0);
                }
                for (int kb = 0; kb < x.nkb && ok; ++kb) {
                    if (kb + 1 < x.nkb)
                        ok = load_kv(x, gb, kb + 1, false);
                    else if (has_next)
                        ok = load_q(y, li + 1) && load_kv(y, gb + x.nkb, 0, false);
                    if (ok) ok = load_kv(x, gb, kb, true);
                }
                gb += x.nkb;
                x = y;
                have = has_next;
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
                const int nkb = item_of<L>(p, w).nkb;
                if (!mbar_wait(bar(B_Q_FULL), static_cast<uint32_t>(li) & 1u, abort_flag, p.status, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                for (int kb = 0; kb < nkb && ok; ++kb, ++gb) {
                    const int st = gb & 1;       // K ring stage
                    const int sb = gb % NS;      // S buffer
                    // Buffer sb held S and then P of block gb - NS: its PV must
                    // have read that P before this S overwrites it.
                    if (gb >= NS && !mbar_wait(bar(B_PV_DONE + sb), static_cast<uint32_t>((gb - NS) / NS) & 1u,
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
                    const uint32_t d_tmem = tmem + sb * KB;
                    const uint64_t kdesc = st ? kdesc1 : kdesc0;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        constexpr uint32_t unit = 16;
                        const uint32_t a_off = ((ks >> 2) * QBOX + (ks & 3) * 32) / unit;
                        const uint32_t b_off = ((ks >> 2) * KBOX + (ks & 3) * 32) / unit;
                        umma_bf16(d_tmem, qdesc + a_off, kdesc + b_off, idesc_s, ks > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(B_K_EMPTY + st));
                    umma_commit(bar(B_S_FULL + sb));
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
                const int nkb = item_of<L>(p, w).nkb;
                for (int kb = 0; kb < nkb && ok; ++kb, ++gb) {
                    const int vst = gb & 1;   // V ring stage
                    const int pb = gb % NS;   // P buffer (the block's S buffer)
                    if (!mbar_wait(bar(B_P_FULL + pb), static_cast<uint32_t>(gb / NS) & 1u, abort_flag, p.status,
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
                    // P of block gb: bf16 in the first KB/2 columns of its S
                    // buffer, 16 keys (8 columns) per UMMA.
                    const uint64_t vdesc = vst ? vdesc1 : vdesc0;
                    const uint32_t pcol = tmem + pb * KB;
                    const uint32_t acc0 = kb > 0 ? 1u : 0u;
#pragma unroll
                    for (int ks = 0; ks < KB / 16; ++ks)
                        umma_bf16_ts(tmem + L::O_COL, pcol + ks * 8, vdesc + (ks * 16 * 128) / 16, idesc_o,
                                     ks > 0 ? 1u : acc0);
                    umma_commit(bar(B_V_EMPTY + vst));
                    umma_commit(bar(B_PV_DONE + pb));
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
        // SPLIT warps share each TMEM lane quadrant: warp half hf takes key
        // columns [hf * KC, (hf + 1) * KC) of every block and O columns
        // [hf * D / SPLIT, (hf + 1) * D / SPLIT).  The two halves of a row
        // agree on its running maximum through one shared-memory exchange
        // per block, so both apply the same scale; each keeps its part of
        // the row sum until the epilogue adds them in a fixed order.
        constexpr int SPLIT = L::SPLIT, KC = KB / SPLIT, DC = D / SPLIT;
        const int q = warp & 3;  // TMEM lane quadrant
        const int hf = (warp - 3) >> 2;
        const int r = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        float* xch = reinterpret_cast<float*>(gbase + L::XCH_OFF);  // [2 parities][SPLIT][128]
        // Every failure passes through one of these before the warps act on
        // it, so the two halves of a quadrant always leave together and no
        // named barrier waits for a warp that has gone.
        auto pair_all = [&](bool v) -> bool {
            if constexpr (SPLIT == 1) {
                __syncwarp();
                return __all_sync(0xffffffffu, v);
            } else {
                return named_bar_and(1u + static_cast<uint32_t>(q), 64u, v);
            }
        };
        // The epilogue of an item (O / l out of TMEM, through shared memory,
        // to global memory by TMA stores) runs after the next item's first
        // block, so the wait for the item's last PV and the stores overlap
        // that block's tensor-core work.  Returns false, in both halves of
        // the quadrant, when a wait gave up.
        auto epilogue = [&](int eq0, int ej, int eb, int eli, float m_e, float l_e, bool bad_e) -> bool {
            bool got = !bad_e && mbar_wait(bar(B_O_FULL), static_cast<uint32_t>(eli) & 1u, abort_flag, p.status,
                                           p.timeout_ns);
            got = __all_sync(0xffffffffu, got);
            if constexpr (SPLIT > 1) xch[2 * SPLIT * QB + hf * QB + r] = l_e;
            if (!pair_all(got)) return false;
            tc_fence_after();
            const int qpos = eq0 + r;
            float l_tot = l_e;
            if constexpr (SPLIT > 1) {
                // Fixed order, the same in both halves.
                l_tot = 0.0f;
#pragma unroll
                for (int h2 = 0; h2 < SPLIT; ++h2) l_tot += xch[2 * SPLIT * QB + h2 * QB + r];
            }
            const float inv = 1.0f / l_tot;
            if (hf == 0 && p.lse && qpos < p.seq)
                p.lse[(static_cast<long long>(ej) * p.batch + eb) * p.seq_pad + qpos] = m_e + log2f(l_tot);
            // O / l as bf16, 32 columns at a time.  With a TMA map the warp
            // writes its 32 rows into one shared-memory box per 32 columns
            // (16-byte piece u of row l at l * 64 + (u ^ ((l / 2) % 4)) * 16)
            // and lane 0 stores the boxes; otherwise each thread stores its
            // row.
            if (p.o_tma) {
                if (lane == 0) bulk_wait_group_read0();  // the previous item's stores have read the boxes
                __syncwarp();
            }
            const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
            const uint32_t box0 = base + L::STG_OFF + static_cast<uint32_t>(q * (D / 32) + hf * (DC / 32)) * STG_BOX;
            __nv_bfloat16* orow = p.o + (static_cast<long long>(eb) * p.seq + qpos) * p.ld_o +
                                  static_cast<long long>(ej) * D + hf * DC;
            // This half's O columns, all loads in flight at once; O is
            // released to the next item's first PV as soon as they land.
            uint32_t o[DC];
#pragma unroll
            for (int c = 0; c < DC / 32; ++c)
                tmem_ld32(tmem + lane_off + L::O_COL + hf * DC + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_O_EMPTY));
#pragma unroll
            for (int c = 0; c < DC / 32; ++c) {
                if (p.o_tma) {
                    const uint32_t srow = box0 + static_cast<uint32_t>(c) * STG_BOX + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint32_t wv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            wv[e] = pack_bf16x2(__uint_as_float(o[c * 32 + u * 8 + 2 * e]) * inv,
                                                __uint_as_float(o[c * 32 + u * 8 + 2 * e + 1]) * inv);
                        st_shared_v4(srow + ((static_cast<uint32_t>(u) ^ sw) << 4), wv[0], wv[1], wv[2], wv[3]);
                    }
                } else if (qpos < p.seq) {
#pragma unroll
                    for (int g8 = 0; g8 < 4; ++g8) {
                        uint32_t wv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            wv[e] = pack_bf16x2(__uint_as_float(o[c * 32 + g8 * 8 + 2 * e]) * inv,
                                                __uint_as_float(o[c * 32 + g8 * 8 + 2 * e + 1]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + g8 * 8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                }
            }
            if (p.o_tma) {
                fence_proxy_async_smem();  // the boxes are visible to the TMA engine
                __syncwarp();
                const int row0 = eq0 + q * 32;
                if (lane == 0 && row0 < p.seq) {
#pragma unroll
                    for (int c = 0; c < DC / 32; ++c)
                        tma_store_3d(&p.map_o, box0 + static_cast<uint32_t>(c) * STG_BOX, ej * D + hf * DC + c * 32,
                                     row0, eb);
                    bulk_commit_group();
                }
            }
            return true;
        };
        bool ok = true;
        bool pending = false;  // an item whose epilogue has not run yet
        int pq0 = 0, pj = 0, pb_ = 0, pli = 0;
        float pm = 0.0f, pl = 0.0f;
        bool pbad = false;
        int gb = 0, li = 0;
        for (int w; ok && (w = item_at(li, w0, dw)) < n_items; ++li) {
            const Item x = item_of<L>(p, w);
            const int q0 = x.q0;
            const int qpos = q0 + r;
            float m_ref = -INFINITY, l_sum = 0.0f;
            bool bad = false;  // a wait after this block's exchange gave up
            for (int kb = 0; kb < x.nkb; ++kb, ++gb) {
                const int st = gb % NS;  // S buffer
                bool got = !bad && mbar_wait(bar(B_S_FULL + st), static_cast<uint32_t>(gb / NS) & 1u, abort_flag,
                                             p.status, p.timeout_ns);
                got = __all_sync(0xffffffffu, got);
                uint32_t s[KC];
                float mxp = -INFINITY;
                if (got) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < KC / 32; ++c)
                        tmem_ld32(tmem + lane_off + st * KB + hf * KC + c * 32,
                                  *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
                    tmem_ld_wait();
                    // Keys k0 + c with c > lim are masked: later than the
                    // query (causal) or past the sequence end.
                    const int k0 = kb * KB + hf * KC;
                    const int lim = min(qpos, p.seq - 1) - k0;
                    if (lim < KC - 1) {
#pragma unroll
                        for (int c = 0; c < KC; ++c)
                            if (c > lim) s[c] = __float_as_uint(-INFINITY);
                    }
                    // Row max with 8 independent chains of three-way maxima.
                    float mx8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(__uint_as_float(s[e]), __uint_as_float(s[8 + e]));
#pragma unroll
                    for (int c = 16; c < KC; c += 16)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            mx8[e] = max3(mx8[e], __uint_as_float(s[c + e]), __uint_as_float(s[c + 8 + e]));
                    mxp = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
                    if constexpr (SPLIT > 1) xch[((gb & 1) * SPLIT + hf) * QB + r] = mxp;
                    tc_fence_before();
                }
                // The other half's S columns are in its registers once this
                // returns, so P may be written over them.
                if (!pair_all(got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float mx = mxp;
                if constexpr (SPLIT > 1) mx = fmaxf(mxp, xch[((gb & 1) * SPLIT + (hf ^ 1)) * QB + r]);
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
                uint32_t pk[KC / 2];
#pragma unroll
                for (int c = 0; c < KC / 2; ++c) {
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
                    const bool got2 = mbar_wait(bar(B_PV_DONE + pb % NS), static_cast<uint32_t>(pb / NS) & 1u,
                                                abort_flag, p.status, p.timeout_ns);
                    __syncwarp();
                    if (!__all_sync(0xffffffffu, got2)) {
                        bad = true;  // acted on at the next pair_all, with the other half
                    } else {
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < DC / 32; ++c) {
                            uint32_t o[32];
                            const uint32_t ta = tmem + lane_off + L::O_COL + hf * DC + c * 32;
                            tmem_ld32(ta, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(ta, o);
                        }
                        tmem_st_wait();
                    }
                }
                // P row r over its S row in TMEM: KC keys as KC / 2 packed columns.
#pragma unroll
                for (int c = 0; c < KC / 64; ++c)
                    tmem_st32(tmem + lane_off + st * KB + hf * (KC / 2) + c * 32,
                              *reinterpret_cast<const uint32_t(*)[32]>(&pk[c * 32]));
                if constexpr (KC % 64 == 32)
                    tmem_st16(tmem + lane_off + st * KB + hf * (KC / 2) + (KC / 64) * 32,
                              *reinterpret_cast<const uint32_t(*)[16]>(&pk[(KC / 64) * 32]));
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_P_FULL + st));
                if (kb == 0 && pending) {
                    if (!epilogue(pq0, pj, pb_, pli, pm, pl, pbad)) {
                        ok = false;
                        break;
                    }
                    pending = false;
                }
            }
            if (!ok) break;
            pending = true;
            pq0 = x.q0;
            pj = x.j;
            pb_ = x.b;
            pli = li;
            pm = m_ref;
            pl = l_sum;
            pbad = bad;
        }
        if (ok && pending) epilogue(pq0, pj, pb_, pli, pm, pl, pbad);
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

template <class L>
int launch_d(const tpi::AttnArgs& a, cudaStream_t stream, std::string* err) {
    constexpr int D = L::D, KB = L::KB;
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
    p.f_hb = make_fastdiv(static_cast<uint32_t>(a.heads * a.batch));
    p.f_heads = make_fastdiv(static_cast<uint32_t>(a.heads));
    p.f_hps = make_fastdiv(static_cast<uint32_t>(p.heads_per_shard));
    p.f_grp = make_fastdiv(static_cast<uint32_t>(a.heads / a.kv_heads));
    p.f_t = make_fastdiv(static_cast<uint32_t>(a.t));
    p.nqb = (a.seq + QB - 1) / QB;
    p.nkb_seq = (a.seq + KB - 1) / KB;
    p.kv_per_shard = a.kv_heads / a.t;
    const int smem = L::SMEM;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            if (err) *err = std::string("cudaFuncSetAttribute(attn): ") + cudaGetErrorString(e);
            return TP_ERR_CUDA;
        }
        configured[dev] = true;
    }
    // Persistent grid: L::CTAS CTAs per SM, or fewer when there are fewer items.
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    const long long n_items = static_cast<long long>((a.seq + QB - 1) / QB) * a.heads * a.batch;
    dim3 grid(static_cast<unsigned>(std::min<long long>(n_items, static_cast<long long>(L::CTAS) * sms)), 1, 1);
    cudaError_t e = tpi::launch_pdl(attn_tc_kernel<L>, grid, dim3(L::NTHREADS), smem, stream, p);
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
    if (a.head_dim == 128) return launch_d<Layout<128, 128, 3, 1, 2>>(a, stream, err);
    if (a.head_dim == 64) return launch_d<Layout<64, 128, 3, 1, 2>>(a, stream, err);
    if (err) *err = "head_dim must be 64 or 128";
    return TP_ERR_UNSUPPORTED;
}

}  // namespace tpi
