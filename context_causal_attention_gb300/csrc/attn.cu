// attn.cu -- partial causal attention with explicit positions on the sm_103a
// tensor cores (tcgen05 + TMEM + TMA), returning (o, lse).
//
// What it computes ("On Context Parallelism", Peer-to-peer / Forward:
// attention(q, k, v, q_positions, kv_positions, scale) -> (tile_output,
// tile_lse); "Context parallelism: Ring Attention and Ulysses", cp_common.py):
// for every (rank, b, h, query row i) with visible keys V(i) = {j : k_pos[j] <=
// q_pos[i]}, lse_i = ln sum_{j in V(i)} e^{scale <q_i,k_j>} and
// o_i = sum_j e^{scale <q_i,k_j> - lse_i} v_j; rows with no visible key get
// o = 0, lse = -inf.
//
// How: one persistent CTA per SM walks a list of work items (rank, b, h,
// super-block: one 256-row query block, or blocks u and nqb-1-u back to back)
// ordered longest-first, head-major within equal cost, and dealt out
// boustrophedon (cp_sched.cuh).  Inside a CTA:
//   warp 0      TMA producer: Q block (two 128-row tiles) and a ring of K/V
//               128-key stages, 128-byte swizzled;
//   warp 1      TMEM allocator (512 columns: S0 | S1 | O0 | O1) and MMA
//               issuer: S_i = Q_i K^T into TMEM (bf16 in, fp32 acc), and
//               O_i += P_i V with P_i read from TMEM;
//   warps 2-3   idle;
//   warps 4-7   softmax for query tile 0, warps 8-11 for query tile 1: one
//               thread per query row, online softmax in the log2 domain
//               ("Context Parallelism & Ring Attention", "Softmax is
//               decomposable": running max, running sum, rescaled output),
//               P written back to TMEM over S columns 64..127 as packed bf16, epilogue
//               o = O / l and lse = (m + log2 l) ln 2 (O is read from TMEM and
//               handed back to the MMA before the global stores).
// Key tiles whose smallest position exceeds the block's largest query
// position are skipped; tiles whose positions are all <= the tile's
// smallest query position run unmasked; the rest are masked per element.
// The running max m is kept an INTEGER in the log2 domain: the ceiling of the
// row max of the first key tile the row can see.  Later tiles use it as is and
// only move it (to the ceiling of their own max) when their P sum would exceed
// 2^64; O and the sums stay consistent with the stale max, every rescale is an
// exact power of two, and the bf16 rounding of P = 2^(x - m) does not
// depend on how the keys are split into partials (so a ring of partials and
// one monolithic call round P identically).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "cp_internal.h"
#include "cp_ptx.cuh"
#include "cp_sched.cuh"

namespace cpattn {

// Sticky device status word of the library (CP_ERR_DEVICE_TIMEOUT when a
// kernel gave up a bounded wait).  Read by cp_device_status().
__device__ int g_cp_device_status = 0;
// A flag nothing ever sets: the self-test holds the producer on it until its
// bounded wait runs out.
__device__ int g_cp_never_set = 0;

namespace {

// 12 warps: three per SM sub-partition, so at most 168 registers per thread
// (each sub-partition holds 16K registers).
constexpr int kThreads = 384;
constexpr int kAtomBytes = 128 * 128;  // one 128-row x 128-byte swizzle atom block (64 bf16 columns)
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Cfg {
    static constexpr int kAtoms = D / 64;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kStages = (D == 128) ? 2 : 4;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffTab = kOffV + kStages * kTileBytes;
    static constexpr int kOffOrder = kOffTab + kMaxTables * 8;
    static constexpr int kOffCost = kOffOrder + kMaxPairs * 4;
    static constexpr int kOffSeg = kOffCost + kMaxPairs * 4;
    static constexpr int kOffBar = kOffSeg + (kMaxPairs + 2) * 4;
    // barriers: q_full, q_empty, drain, k_full[S], v_full[S], k_empty[S], v_empty[S],
    //           s_full[2], p_full[2], o_full[2], o_empty[2]
    static constexpr int kNumBars = 3 + 4 * kStages + 8;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kMiscBytes = 16 + kMaxC * 4 + kMaxTables / 8;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct AttnArgs {
    const int32_t *q_pos;
    const int32_t *k_pos;
    long long q_pos_stride, k_pos_stride;
    float *o, *lse;
    int C, B, N, Nkv, Sq, Sk;
    int nqt, nkt, nqb;
    int kv_shift, kpos_shift;
    int kv_shared;  // all ranks read the same K/V (rank index 0)
    int kpr;        // key-position ranks with tables: 1 if shared, else C
    int merge_into; // LSE-merge the partial into the (o, lse) accumulator
    float scale_log2;
    unsigned long long timeout_ns;
    const int *hold;  // failure injection (self-test only), else null
    int nsp;          // super-blocks per rank
    int pair_blocks;  // a super-block holds query blocks u and nqb-1-u (else u alone)
    FastDiv div_nsp, div_n;  // by nsp, N (work-item decoding)
    PlanPtrs gp;             // the launch's plan in global memory (kernels with kGlobalPlan)
};

struct Bars {
    uint64_t *q_full, *q_empty, *drain, *k_full, *v_full, *k_empty, *v_empty, *s_full, *p_full, *o_full, *o_empty;
};

template <int D>
__device__ __forceinline__ Bars bars_at(uint8_t *base) {
    using K = Cfg<D>;
    uint64_t *b = reinterpret_cast<uint64_t *>(base + K::kOffBar);
    Bars r;
    r.q_full = b + 0;
    r.q_empty = b + 1;
    r.drain = b + 2;
    r.k_full = b + 3;
    r.v_full = b + 3 + K::kStages;
    r.k_empty = b + 3 + 2 * K::kStages;
    r.v_empty = b + 3 + 3 * K::kStages;
    r.s_full = b + 3 + 4 * K::kStages;
    r.p_full = r.s_full + 2;
    r.o_full = r.s_full + 4;
    r.o_empty = r.s_full + 6;
    return r;
}

// Work item -> (rank, query block, b, h).
struct Item {
    int r, qb, b, h, owner, kvr;
    int qmax;  // largest query position of the 256-row block (over valid rows)
};

// Work item of query block qb (a part of super item x) -> Item.
__device__ __forceinline__ Item make_item(const SuperItem &x, int qb, const AttnArgs &a, const int2 *qtab) {
    Item it;
    it.r = x.r;
    it.qb = qb;
    it.b = static_cast<int>(fdiv(static_cast<uint32_t>(x.bh), a.div_n));
    it.h = x.bh - it.b * a.N;
    it.owner = it.r + a.kpos_shift;
    if (it.owner >= a.C) it.owner -= a.C;
    if (a.kpr == 1) it.owner = 0;
    it.kvr = it.r + a.kv_shift;
    if (it.kvr >= a.C) it.kvr -= a.C;
    if (a.kv_shared) it.kvr = 0;
    const int qt0 = 2 * qb, qt1 = 2 * qb + 1;
    int qmax = qtab[it.r * a.nqt + qt0].y;
    if (qt1 < a.nqt) qmax = max(qmax, qtab[it.r * a.nqt + qt1].y);
    it.qmax = qmax;
    return it;
}

// Next key tile >= kt that this block must process (nkt if none).
__device__ __forceinline__ int next_ktile(int kt, int nkt, const int2 *ktab_owner, int qmax, bool sorted) {
    for (; kt < nkt; ++kt) {
        if (ktab_owner[kt].x <= qmax) return kt;
        if (sorted) return nkt;
    }
    return nkt;
}

// This thread's 128 scores of the current key tile from TMEM, with the causal
// mask applied (scores of keys the row may not see become -inf).  `arith`:
// the tile's positions are kmin, kmin+1, ...; else positions are read from kpos.
__device__ __forceinline__ void load_scores(uint32_t tS, bool need_mask, bool arith, int qpos, int kmin, int nvalid,
                                            const int32_t *kpos, uint32_t (&sa)[64], uint32_t (&sb)[64]) {
    tmem_ld128(tS, sa, sb);
    if (!need_mask) return;
    if (arith) {
        // column c is visible iff c <= qpos - kmin
        const long long d = static_cast<long long>(qpos) - kmin;
        const int lim = d < 0 ? -1 : static_cast<int>(min(d, static_cast<long long>(nvalid - 1)));
#pragma unroll
        for (int c = 0; c < 64; ++c)
            if (c > lim) sa[c] = 0xff800000u;
#pragma unroll
        for (int c = 0; c < 64; ++c)
            if (64 + c > lim) sb[c] = 0xff800000u;
    } else {
        // arbitrary positions: compare column by column, 16 loads at a time
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
#pragma unroll
            for (int c = c0; c < c0 + 16; ++c) {
                const int kp = (c < nvalid) ? __ldg(kpos + c) : INT_MAX;
                if (kp > qpos) sa[c] = 0xff800000u;
            }
            asm volatile("" ::: "memory");
        }
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
#pragma unroll
            for (int c = c0; c < c0 + 16; ++c) {
                const int kp = (64 + c < nvalid) ? __ldg(kpos + 64 + c) : INT_MAX;
                if (kp > qpos) sb[c] = 0xff800000u;
            }
            asm volatile("" ::: "memory");
        }
    }
}

// Causal mask of one 64-column half (columns c0 .. c0+63 of the key tile).
__device__ __forceinline__ void mask_half(bool arith, int qpos, int kmin, int nvalid, const int32_t *kpos, int c0,
                                          uint32_t (&h)[64]) {
    if (arith) {
        const long long d = static_cast<long long>(qpos) - kmin;
        const int lim = d < 0 ? -1 : static_cast<int>(min(d, static_cast<long long>(nvalid - 1)));
#pragma unroll
        for (int c = 0; c < 64; ++c)
            if (c0 + c > lim) h[c] = 0xff800000u;
    } else {
#pragma unroll
        for (int cc = 0; cc < 64; cc += 16) {
#pragma unroll
            for (int c = cc; c < cc + 16; ++c) {
                const int kp = (c0 + c < nvalid) ? __ldg(kpos + c0 + c) : INT_MAX;
                if (kp > qpos) h[c] = 0xff800000u;
            }
            asm volatile("" ::: "memory");
        }
    }
}

// p = 2^(s * sl2 - m) for 64 scores, packed to 32 bf16 pairs; returns the
// fp32 sum of p.
__device__ __forceinline__ float exp_pack64(const uint32_t (&h)[64], float sl2, float neg_m, uint32_t (&pk)[32]) {
    const uint64_t sl2x2 = f2_packf(sl2, sl2), nmx2 = f2_packf(neg_m, neg_m);
    uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
        float x0, x1, x2, x3;
        f2_unpack(f2_fma(f2_pack(h[2 * c], h[2 * c + 1]), sl2x2, nmx2), x0, x1);
        f2_unpack(f2_fma(f2_pack(h[2 * c + 2], h[2 * c + 3]), sl2x2, nmx2), x2, x3);
        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
        const float p2 = fast_exp2(x2), p3 = fast_exp2(x3);
        sum2[(c >> 1) & 1] = f2_add(sum2[(c >> 1) & 1], f2_packf(p0, p1));
        sum2[2 + ((c >> 1) & 1)] = f2_add(sum2[2 + ((c >> 1) & 1)], f2_packf(p2, p3));
        pk[c] = pack_bf16x2(p0, p1);
        pk[c + 1] = pack_bf16x2(p2, p3);
    }
    const uint64_t t = f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3]));
    float lo, hi;
    f2_unpack(t, lo, hi);
    return lo + hi;
}

// Row max of the 128 scores of one thread (raw fp32 bits), 8 independent chains.
__device__ __forceinline__ float row_max128(const uint32_t (&sa)[64], const uint32_t (&sb)[64]) {
    float mx[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
#pragma unroll
    for (int c = 0; c < 64; c += 8) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            mx[u] = fmax3(mx[u], __uint_as_float(sa[c + 2 * u]), __uint_as_float(sa[c + 2 * u + 1]));
            mx[4 + u] = fmax3(mx[4 + u], __uint_as_float(sb[c + 2 * u]), __uint_as_float(sb[c + 2 * u + 1]));
        }
    }
    return fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
}

// p = 2^(s * sl2 - m) for the 128 scores of one thread, packed to bf16 pairs
// in pa/pb; returns the sum of the fp32 p in *sum.
__device__ __forceinline__ void exp_pack128(const uint32_t (&sa)[64], const uint32_t (&sb)[64], float sl2,
                                            float neg_m, uint32_t (&pa)[32], uint32_t (&pb)[32], float *sum) {
    const uint64_t sl2x2 = f2_packf(sl2, sl2), nmx2 = f2_packf(neg_m, neg_m);
    uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        float x0, x1, x2, x3;
        f2_unpack(f2_fma(f2_pack(sa[2 * c], sa[2 * c + 1]), sl2x2, nmx2), x0, x1);
        f2_unpack(f2_fma(f2_pack(sb[2 * c], sb[2 * c + 1]), sl2x2, nmx2), x2, x3);
        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
        const float p2 = fast_exp2(x2), p3 = fast_exp2(x3);
        sum2[c & 1] = f2_add(sum2[c & 1], f2_packf(p0, p1));
        sum2[2 + (c & 1)] = f2_add(sum2[2 + (c & 1)], f2_packf(p2, p3));
        pa[c] = pack_bf16x2(p0, p1);
        pb[c] = pack_bf16x2(p2, p3);
    }
    const uint64_t t = f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3]));
    float lo, hi;
    f2_unpack(t, lo, hi);
    *sum = lo + hi;
}

// kGlobalPlan: the launch's plan (position tables, bits, sorted flags, costs,
// order) was written to global memory by the pre-pass and is read from there;
// otherwise every CTA builds it in shared memory first.
template <int D, bool kGlobalPlan>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
    using K = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    int2 *tab_s = reinterpret_cast<int2 *>(smem + K::kOffTab);  // [C*nkt] K tables, then [C*nqt] Q tables
    int *order_s = reinterpret_cast<int *>(smem + K::kOffOrder);
    // per (rank, query block): number of key tiles it processes
    int *cost_s = reinterpret_cast<int *>(smem + K::kOffCost);
    int *seg_s = reinterpret_cast<int *>(smem + K::kOffSeg);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + K::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + K::kOffMisc + 4);
    int *sorted_s = reinterpret_cast<int *>(smem + K::kOffMisc + 16);
    // bit g set: K tile g holds consecutive positions kmin, kmin+1, ... (mask = column compare)
    uint32_t *bits_s = reinterpret_cast<uint32_t *>(smem + K::kOffMisc + 16 + kMaxC * 4);
    const Bars bars = bars_at<D>(smem);
    const int2 *ktab = kGlobalPlan ? a.gp.ktab : tab_s;
    const int2 *qtab = kGlobalPlan ? a.gp.qtab : tab_s + a.kpr * a.nkt;
    const int *order = kGlobalPlan ? a.gp.order : order_s;
    const int *cost = kGlobalPlan ? a.gp.cost : cost_s;
    const int *seg_first = kGlobalPlan ? a.gp.seg_first : seg_s;
    const int *sorted_flag = kGlobalPlan ? a.gp.ksorted : sorted_s;
    const uint32_t *arith_bits = kGlobalPlan ? a.gp.kbits : bits_s;

    // ------------------------------------------------------------ set-up
    if (tid == 0) {
        *abort_flag = 0;
        if (!kGlobalPlan)
            for (int w = 0; w < kMaxTables / 32; ++w) bits_s[w] = 0u;
        mbar_init(bars.q_full, 1);
        mbar_init(bars.q_empty, 1);
        mbar_init(bars.drain, 1);
        for (int s = 0; s < K::kStages; ++s) {
            mbar_init(bars.k_full + s, 1);
            mbar_init(bars.v_full + s, 1);
            mbar_init(bars.k_empty + s, 1);
            mbar_init(bars.v_empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bars.s_full + i, 1);
            mbar_init(bars.p_full + i, 4);
            mbar_init(bars.o_full + i, 1);
            mbar_init(bars.o_empty + i, 4);
        }
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }

    __syncthreads();
    // position tables: (min, max) of every 128-row tile, K tiles per owner rank
    // first, then Q tiles per rank.
    if constexpr (!kGlobalPlan) {
        const int nk = a.kpr * a.nkt, total = nk + a.C * a.nqt;
        for (int g = warp; g < total; g += kThreads / 32) {
            const int32_t *p;
            int rows0, lim;
            if (g < nk) {
                const int j = g / a.nkt, kt = g % a.nkt;
                p = a.k_pos + j * a.k_pos_stride;
                rows0 = kt * 128;
                lim = a.Sk;
            } else {
                const int r = (g - nk) / a.nqt, qt = (g - nk) % a.nqt;
                p = a.q_pos + r * a.q_pos_stride;
                rows0 = qt * 128;
                lim = a.Sq;
            }
            int mn = INT_MAX, mx = INT_MIN;
            int vals[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int row = rows0 + lane + 32 * m;
                vals[m] = (row < lim) ? __ldg(p + row) : 0;
                if (row < lim) {
                    mn = min(mn, vals[m]);
                    mx = max(mx, vals[m]);
                }
            }
            mn = __reduce_min_sync(0xffffffffu, mn);
            mx = __reduce_max_sync(0xffffffffu, mx);
            if (lane == 0) tab_s[g] = make_int2(mn, mx);
            if (g < nk) {
                const int first = __shfl_sync(0xffffffffu, vals[0], 0);
                bool ok = true;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int row = rows0 + lane + 32 * m;
                    if (row < lim) ok &= (static_cast<long long>(vals[m]) == static_cast<long long>(first) + lane + 32 * m);
                }
                ok = __all_sync(0xffffffffu, ok);
                if (lane == 0 && ok) atomicOr(bits_s + (g >> 5), 1u << (g & 31));
            }
        }
        __syncthreads();
        if (tid < a.kpr) {
            int ok = 1;
            for (int kt = 1; kt < a.nkt; ++kt) ok &= (ktab[tid * a.nkt + kt].x >= ktab[tid * a.nkt + kt - 1].x);
            sorted_s[tid] = ok;
        }
        __syncthreads();
        // key tiles of every (rank, query block) pair, then the longest-first
        // order of the super-blocks cut into segments (see decode_super)
        const int np = a.C * a.nqb;
        for (int p = tid; p < np; p += kThreads) {
            const int r = p / a.nqb, qb = p % a.nqb;
            const int owner = (a.kpr == 1) ? 0 : (r + a.kpos_shift) % a.C;
            int qmax = qtab[r * a.nqt + 2 * qb].y;
            if (2 * qb + 1 < a.nqt) qmax = max(qmax, qtab[r * a.nqt + 2 * qb + 1].y);
            const int2 *kt_o = ktab + owner * a.nkt;
            int c = 0;
            if (sorted_flag[owner]) {
                int lo = 0, hi = a.nkt;  // first tile with kmin > qmax
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (kt_o[mid].x <= qmax) lo = mid + 1; else hi = mid;
                }
                c = lo;
            } else {
                for (int kt = 0; kt < a.nkt; ++kt) c += (kt_o[kt].x <= qmax);
            }
            cost_s[p] = c;
        }
        __syncthreads();
        build_segments<kThreads>(cost_s, a.C, a.nqb, a.pair_blocks != 0, order_s, seg_s);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_items = a.C * a.nsp * a.B * a.N;
    const int n_rounds = (n_items + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    const int hq_per_kv = a.N / a.Nkv;
    uint8_t *sQ = smem + K::kOffQ;
    uint8_t *sK = smem + K::kOffK;
    uint8_t *sV = smem + K::kOffV;

    if (warp == 0) {
        // -------------------------------------------------------- TMA producer
        if (lane == 0) {
            // K runs one tile ahead of V: a K stage is freed after the second
            // tile's Q K^T, a V stage only after the second tile's P V.
            uint32_t k_it = 0, v_it = 0, it = 0;
            bool ok = true;
            uint32_t k_issued = 0, k_par = 0, v_issued = 0, v_par = 0;  // per stage: issued / phase parity
            int q_parity = -1;
            bool pend = false;  // a V tile waits to be issued
            if (a.hold) {
                // self-test: wait (bounded) for a flag nothing sets, then give up
                // like any other wait does
                const uint64_t t0 = global_timer_ns();
                while (*reinterpret_cast<const volatile int *>(a.hold) == 0) {
                    if (global_timer_ns() - t0 > a.timeout_ns) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    __nanosleep(1000);
                }
            }
            int pend_kt = 0, pend_hk = 0, pend_row = 0;
            auto issue_v = [&]() -> bool {
                const uint32_t st = v_it % K::kStages, ph = (v_it / K::kStages) & 1u;
                if (!mbar_wait(bars.v_empty + st, ph ^ 1u, abort_flag, a.timeout_ns)) return false;
                mbar_arrive_expect_tx(bars.v_full + st, K::kTileBytes);
                for (int at = 0; at < K::kAtoms; ++at)
                    tma_load_4d(sV + st * K::kTileBytes + at * kAtomBytes, &tmV, bars.v_full + st, 64 * at, pend_hk,
                                pend_kt * 128, pend_row);
                v_issued |= 1u << st;
                v_par = (v_par & ~(1u << st)) | (ph << st);
                ++v_it;
                pend = false;
                return true;
            };
            int seg = 0;  // segment cursor of decode_super
            for (int rk = 0; rk < n_rounds && ok; ++rk) {
                const int idx = item_of_round(rk, n_items);
                if (idx < 0) continue;
                const SuperItem sup = decode_super(idx, a.B * a.N, order, seg_first, a.div_nsp, seg);
                for (int part = 0; part < 2 && ok; ++part) {
                    const int qb = super_part(sup.u, part, a.nqb, a.pair_blocks != 0);
                    if (qb < 0) continue;
                    const Item itm = make_item(sup, qb, a, qtab);
                    const int2 *kt_o = ktab + itm.owner * a.nkt;
                    const bool srt = sorted_flag[itm.owner];
                    int kt = next_ktile(0, a.nkt, kt_o, itm.qmax, srt);
                    if (kt >= a.nkt) continue;
                    if (pend && !issue_v()) { ok = false; break; }  // last V of the previous item
                    if (!mbar_wait(bars.q_empty, (it & 1u) ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    mbar_arrive_expect_tx(bars.q_full, 2 * K::kTileBytes);
                    q_parity = it & 1u;
                    const int qrow = itm.r * a.B + itm.b;
                    for (int i = 0; i < 2; ++i)
                        for (int at = 0; at < K::kAtoms; ++at)
                            tma_load_4d(sQ + i * K::kTileBytes + at * kAtomBytes, &tmQ, bars.q_full, 64 * at, itm.h,
                                        (2 * itm.qb + i) * 128, qrow);
                    ++it;
                    const int hk = itm.h / hq_per_kv;
                    const int kvrow = itm.kvr * a.B + itm.b;
                    for (; kt < a.nkt; kt = next_ktile(kt + 1, a.nkt, kt_o, itm.qmax, srt)) {
                        const uint32_t st = k_it % K::kStages, ph = (k_it / K::kStages) & 1u;
                        if (!mbar_wait(bars.k_empty + st, ph ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        mbar_arrive_expect_tx(bars.k_full + st, K::kTileBytes);
                        for (int at = 0; at < K::kAtoms; ++at)
                            tma_load_4d(sK + st * K::kTileBytes + at * kAtomBytes, &tmK, bars.k_full + st, 64 * at, hk,
                                        kt * 128, kvrow);
                        k_issued |= 1u << st;
                        k_par = (k_par & ~(1u << st)) | (ph << st);
                        ++k_it;
                        if (pend && !issue_v()) { ok = false; break; }
                        pend = true;
                        pend_kt = kt;
                        pend_hk = hk;
                        pend_row = kvrow;
                    }
                }
            }
            if (ok && pend && !issue_v()) ok = false;
            if (!ok) {
                // let every copy already issued land before shared memory goes away
                volatile int no_abort = 0;
                const unsigned long long drain_ns = 100000000ull;
                if (q_parity >= 0) mbar_wait(bars.q_full, q_parity, &no_abort, drain_ns);
                for (int st = 0; st < K::kStages; ++st) {
                    if ((k_issued >> st) & 1u) mbar_wait(bars.k_full + st, (k_par >> st) & 1u, &no_abort, drain_ns);
                    if ((v_issued >> st) & 1u) mbar_wait(bars.v_full + st, (v_par >> st) & 1u, &no_abort, drain_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, 0, 1);
            const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV);
            uint32_t kv_it = 0, it = 0;
            bool ok = true;
            // descriptors of the k-step-0 / key-0 sub-tiles, built once; the MMA
            // groups add immediate offsets (the issuing warp shares its SM
            // sub-partition with two busy softmax warps, so it is kept short)
            const uint64_t dq0 = smem_desc_sw128(q_base, 16, 1024);
            const uint64_t dq1 = smem_desc_sw128(q_base + K::kTileBytes, 16, 1024);
            const uint64_t dk0 = smem_desc_sw128(k_base, 16, 1024);
            const uint64_t dv0 = smem_desc_sw128(v_base, kAtomBytes, 1024);
            constexpr uint64_t kStageDesc = K::kTileBytes >> 4;  // one stage in descriptor units
            auto issue_qk = [&](int i, uint32_t st) {
                umma_qk_group<D / 16>(tmem + i * 128, i ? dq1 : dq0, dk0 + st * kStageDesc, kIdescQK);
            };
            auto issue_pv = [&](int i, uint32_t st, bool acc) {
                umma_pv_group(tmem + 256 + i * D, tmem + i * 128 + 64, dv0 + st * kStageDesc, kIdescPV,
                              acc ? 1u : 0u);
            };
            int seg = 0;  // segment cursor of decode_super
            for (int rk = 0; rk < n_rounds && ok; ++rk) {
                const int idx = item_of_round(rk, n_items);
                if (idx < 0) continue;
                const SuperItem sup = decode_super(idx, a.B * a.N, order, seg_first, a.div_nsp, seg);
                for (int part = 0; part < 2 && ok; ++part) {
                    const int qb = super_part(sup.u, part, a.nqb, a.pair_blocks != 0);
                    if (qb < 0) continue;
                    const Item itm = make_item(sup, qb, a, qtab);
                    const int n = cost[itm.r * a.nqb + itm.qb];  // key tiles of this item
                    if (n == 0) continue;
                    if (!mbar_wait(bars.q_full, it & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    uint32_t prev_st = 0;
                    for (int j = 0; j < n && ok; ++j) {
                        const uint32_t st = kv_it % K::kStages, ph = (kv_it / K::kStages) & 1u;
                        if (!mbar_wait(bars.k_full + st, ph, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        for (int i = 0; i < 2; ++i) {
                            if (j > 0) {
                                const uint32_t pst = (kv_it - 1) % K::kStages, pph = ((kv_it - 1) / K::kStages) & 1u;
                                // the waits that do not depend on the softmax come first, so
                                // P V follows this tile's P as closely as possible; both tiles
                                // read the same V stage, so tile 1 needs no second wait
                                if (i == 0 && !mbar_wait(bars.v_full + pst, pph, abort_flag, a.timeout_ns)) { ok = false; break; }
                                if (j == 1 && !mbar_wait(bars.o_empty + i, (it & 1u) ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                                if (!mbar_wait(bars.p_full + i, (kv_it - 1) & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                                tc_fence_after();
                                issue_pv(i, prev_st, j > 1);
                                if (i == 1) umma_commit(bars.v_empty + prev_st);
                            }
                            issue_qk(i, st);
                            umma_commit(bars.s_full + i);
                        }
                        if (ok) umma_commit(bars.k_empty + st);  // both tiles' Q K^T read this K stage
                        if (!ok) break;
                        if (j == n - 1) umma_commit(bars.q_empty);
                        prev_st = st;
                        ++kv_it;
                    }
                    if (!ok) break;
                    // tail: P V of the last key tile, then hand O to the epilogue
                    for (int i = 0; i < 2; ++i) {
                        const uint32_t pst = (kv_it - 1) % K::kStages, pph = ((kv_it - 1) / K::kStages) & 1u;
                        if (i == 0 && !mbar_wait(bars.v_full + pst, pph, abort_flag, a.timeout_ns)) { ok = false; break; }
                        if (n == 1 && !mbar_wait(bars.o_empty + i, (it & 1u) ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        if (!mbar_wait(bars.p_full + i, (kv_it - 1) & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        issue_pv(i, prev_st, n > 1);
                        if (i == 1) umma_commit(bars.v_empty + prev_st);
                        umma_commit(bars.o_full + i);
                    }
                    ++it;
                }
            }
            // no MMA may still be running when TMEM is released
            umma_commit(bars.drain);
            volatile int no_abort = 0;
            mbar_wait(bars.drain, 0, &no_abort, 100000000ull);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // -------------------------------------------------------- softmax
        const int wg = (warp - 4) >> 2;           // query tile 0 or 1
        const int wq = warp & 3;                  // TMEM lane quarter (warp % 4)
        const int row_in_tile = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + wg * 128;
        const uint32_t tO = tmem + lane_off + 256 + wg * D;
        const float sl2 = a.scale_log2;
        uint32_t kv_count = 0, it = 0;
        bool ok = true;
        int seg = 0;  // segment cursor of decode_super
        for (int rk = 0; rk < n_rounds && ok; ++rk) {
            const int idx = item_of_round(rk, n_items);
            if (idx < 0) continue;
            const SuperItem sup = decode_super(idx, a.B * a.N, order, seg_first, a.div_nsp, seg);
            for (int part = 0; part < 2 && ok; ++part) {
                const int qb = super_part(sup.u, part, a.nqb, a.pair_blocks != 0);
                if (qb < 0) continue;
                const Item itm = make_item(sup, qb, a, qtab);
                const int2 *kt_o = ktab + itm.owner * a.nkt;
                const bool srt = sorted_flag[itm.owner];
                const int qt = 2 * itm.qb + wg;
                const int row = qt * 128 + row_in_tile;
                const bool row_valid = row < a.Sq;
                const int qpos = row_valid ? __ldg(a.q_pos + itm.r * a.q_pos_stride + row) : INT_MIN;
                const int qmin_t = (qt < a.nqt) ? qtab[itm.r * a.nqt + qt].x : INT_MAX;
                const int32_t *kpos_o = a.k_pos + itm.owner * a.k_pos_stride;
                const long long orow = static_cast<long long>(itm.r * a.B + itm.b) * a.Sq + row;
                float *o_row = a.o + (orow * a.N + itm.h) * D;
                float *lse_out = a.lse + (static_cast<long long>(itm.r * a.B + itm.b) * a.N + itm.h) * a.Sq + row;
                const int n_item = cost[itm.r * a.nqb + itm.qb];  // key tiles of this item
                float m_run = -INFINITY, l_run = 0.f;
                int j = 0;
                for (int kt = next_ktile(0, a.nkt, kt_o, itm.qmax, srt); kt < a.nkt;
                     kt = next_ktile(kt + 1, a.nkt, kt_o, itm.qmax, srt), ++j) {
                    if (!mbar_wait_warp(bars.s_full + wg, kv_count & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    if (a.merge_into && row_valid && j == n_item - 1) {
                        // the epilogue will read this row of the accumulator: start it towards L2
    #pragma unroll
                        for (int c = 0; c < D; c += 32) prefetch_l2(o_row + c);
                    }
                    uint32_t sa[64], sb[64];
                    const int2 kmm = kt_o[kt];
                    const bool need_mask = (kmm.y > qmin_t) || (kt * 128 + 128 > a.Sk);
                    const int kbase = kt * 128;
                    const int gk = itm.owner * a.nkt + kt;
                    const int nvalid = min(128, a.Sk - kbase);
                    const bool arith = (arith_bits[gk >> 5] >> (gk & 31)) & 1u;
                    // P (bf16 pairs) goes to columns 64..127 of the S region, so S
                    // columns 0..63 stay readable until this tile's P V is issued.
                    uint32_t pa[32], pb[32];
                    float t_sum;
                    bool stored = false;
                    if constexpr (D == 64) {
                        // TMEM loads/stores are warp-collective: every branch around them is
                        // warp-uniform.  A row's first visible tile takes the steady code too, after the
                        // tile max of both halves has set its running max: with items of a
                        // few key tiles the per-item code is a large share, and a separate
                        // first-tile copy of the exp code ran cold in the instruction cache
                        // once per item.  (At D = 128 the shared form cost the steady loop
                        // more registers than it saved.)
                        tmem_ld64_nowait(tS, sa);
                        tmem_wait_ld(sa);
                        tmem_ld64_nowait(tS + 64, sb);
                        if (need_mask) mask_half(arith, qpos, kmm.x, nvalid, kpos_o + kbase, 0, sa);
                        const bool first = !__all_sync(0xffffffffu, m_run != -INFINITY);
                        if (first) {
                            tmem_wait_ld(sb);
                            if (need_mask) mask_half(arith, qpos, kmm.x, nvalid, kpos_o + kbase, 64, sb);
                            if (m_run == -INFINITY) {
                                const float m_tile = row_max128(sa, sb) * sl2;
                                if (m_tile > -INFINITY) m_run = ceilf(m_tile);
                            }
                        }
                        const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                        const float s0 = exp_pack64(sa, sl2, neg_m, pa);
                        tmem_wait_ld(sb);  // columns 64..127 read: P may overwrite them
                        tmem_st32_nowait(tS + 64, pa);
                        if (need_mask && !first) mask_half(arith, qpos, kmm.x, nvalid, kpos_o + kbase, 64, sb);
                        const float s1 = exp_pack64(sb, sl2, neg_m, pb);
                        tmem_st32_nowait(tS + 96, pb);
                        t_sum = s0 + s1;
                        stored = true;
                    } else if (__all_sync(0xffffffffu, m_run != -INFINITY)) {
                        // (TMEM loads/stores are warp-collective: the path must be warp-uniform)
                        // Steady state (max already set): pipeline the tile in two halves --
                        // the second half's TMEM load and the first half's P store overlap
                        // exp work.
                        tmem_ld64_nowait(tS, sa);
                        tmem_wait_ld(sa);
                        tmem_ld64_nowait(tS + 64, sb);
                        if (need_mask) mask_half(arith, qpos, kmm.x, nvalid, kpos_o + kbase, 0, sa);
                        const float s0 = exp_pack64(sa, sl2, -m_run, pa);
                        tmem_wait_ld(sb);  // columns 64..127 read: P may overwrite them
                        tmem_st32_nowait(tS + 64, pa);
                        if (need_mask) mask_half(arith, qpos, kmm.x, nvalid, kpos_o + kbase, 64, sb);
                        const float s1 = exp_pack64(sb, sl2, -m_run, pb);
                        tmem_st32_nowait(tS + 96, pb);
                        t_sum = s0 + s1;
                        stored = true;
                    } else {
                        load_scores(tS, need_mask, arith, qpos, kmm.x, nvalid, kpos_o + kbase, sa, sb);
                        // rows without a running max yet (first visible tile): set it
                        if (m_run == -INFINITY) {
                            const float m_tile = row_max128(sa, sb) * sl2;
                            if (m_tile > -INFINITY) m_run = ceilf(m_tile);
                        }
                        exp_pack128(sa, sb, sl2, (m_run == -INFINITY) ? 0.f : -m_run, pa, pb, &t_sum);
                    }
                    float factor = 1.f;
                    bool rescale = false;
                    const bool big = !(t_sum <= 0x1p64f);  // also true for inf / nan
                    if (__any_sync(0xffffffffu, big)) {
                        // rare: scores grew by more than 2^64 over the running max.  Columns
                        // 0..63 of S are still in TMEM; columns 64..127 are still in sb.
                        if (stored) tmem_wait_st();
                        tmem_ld64(tS, sa);
                        if (need_mask) mask_half(arith, qpos, kmm.x, nvalid, kpos_o + kbase, 0, sa);
                        if (big) {
                            const float m_new = ceilf(row_max128(sa, sb) * sl2);
                            // exact 2^(m_run - m_new): both are integers
                            const float dk = m_run - m_new;
                            factor = (dk >= -126.f) ? __int_as_float((127 + static_cast<int>(dk)) << 23) : 0.f;
                            rescale = true;
                            l_run *= factor;
                            m_run = m_new;
                        }
                        // every lane recomputes (unchanged rows reproduce their values)
                        exp_pack128(sa, sb, sl2, (m_run == -INFINITY) ? 0.f : -m_run, pa, pb, &t_sum);
                        stored = false;
                    }
                    l_run += t_sum;
                    if (stored) {
                        tmem_wait_st();
                    } else {
                        tmem_st64(tS + 64, pa, pb);
                    }
                    // O is quiescent here (the P V of this tile waits for p_full below)
                    if (__any_sync(0xffffffffu, rescale)) {
    #pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t ov[32];
                            tmem_ld32(tO + c0, ov);
    #pragma unroll
                            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * factor);
                            tmem_st32(tO + c0, ov);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.p_full + wg);
                    ++kv_count;
                }
                if (!ok) break;
                if (j == 0) {
                    // nothing visible for this whole block: o = 0, lse = -inf (a merge
                    // leaves the accumulator as it is)
                    if (row_valid && !a.merge_into) {
    #pragma unroll
                        for (int c = 0; c < D; c += 8) st_global_v8(o_row + c, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f);
                        *lse_out = -INFINITY;
                    }
                    continue;
                }
                if (!mbar_wait_warp(bars.o_full + wg, it & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
                const float lse_t = (l_run > 0.f) ? (m_run + __log2f(l_run)) * 0.69314718055994530942f : -INFINITY;
                // o_row <- wa * o_row + wt * O (O unnormalised in TMEM); plain write: wa = 0
                bool write = row_valid;
                float wa = 0.f, wt = inv_l, lse_new = lse_t;
                if (a.merge_into && row_valid) {
                    // "On Context Parallelism", Peer-to-peer / Forward, the tile merge
                    const float la = *lse_out;
                    if (lse_t == -INFINITY) {
                        write = false;
                    } else if (la != -INFINITY) {
                        const float mx = fmaxf(la, lse_t), mn = fminf(la, lse_t);
                        lse_new = mx + log1pf(expf(mn - mx));
                        wa = expf(la - lse_new);
                        wt = expf(lse_t - lse_new) * inv_l;
                    }
                }
                bool o_released = false;
                if (!a.merge_into) {
                    // all of O from TMEM under one wait; O is handed back before the stores
                    uint32_t ov[D / 32][32];
    #pragma unroll
                    for (int q = 0; q < D / 32; ++q) tmem_ld32_nowait(tO + 32 * q, ov[q]);
    #pragma unroll
                    for (int q = 0; q < D / 32; ++q) tmem_wait_ld32(ov[q]);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.o_empty + wg);
                    o_released = true;
                    if (write) {
    #pragma unroll
                        for (int q = 0; q < D / 32; ++q)
    #pragma unroll
                            for (int c = 0; c < 32; c += 8)
                                st_global_v8(o_row + 32 * q + c, __uint_as_float(ov[q][c]) * wt,
                                             __uint_as_float(ov[q][c + 1]) * wt, __uint_as_float(ov[q][c + 2]) * wt,
                                             __uint_as_float(ov[q][c + 3]) * wt, __uint_as_float(ov[q][c + 4]) * wt,
                                             __uint_as_float(ov[q][c + 5]) * wt, __uint_as_float(ov[q][c + 6]) * wt,
                                             __uint_as_float(ov[q][c + 7]) * wt);
                    }
                } else {
                    const bool read_acc = write && wa != 0.f;
    #pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 16) {
                        float acc[16];
                        if (read_acc) {
                            // issued before the TMEM load so both latencies overlap (the row
                            // was sent towards L2 when the item's last tile started)
                            float t8[8];
                            ld_global_v8(o_row + c0, t8);
    #pragma unroll
                            for (int e = 0; e < 8; ++e) acc[e] = t8[e];
                            ld_global_v8(o_row + c0 + 8, t8);
    #pragma unroll
                            for (int e = 0; e < 8; ++e) acc[8 + e] = t8[e];
                        }
                        uint32_t ov[16];
                        tmem_ld16(tO + c0, ov);
                        if (write) {
    #pragma unroll
                            for (int c = 0; c < 16; c += 8) {
                                float r8[8];
    #pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    r8[e] = read_acc ? fmaf(wa, acc[c + e], wt * __uint_as_float(ov[c + e]))
                                                     : wt * __uint_as_float(ov[c + e]);
                                st_global_v8(o_row + c0 + c, r8[0], r8[1], r8[2], r8[3], r8[4], r8[5], r8[6], r8[7]);
                            }
                        }
                    }
                }
                if (write) *lse_out = lse_new;
                if (!o_released) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.o_empty + wg);
                }
                ++it;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && *abort_flag) atomicExch(&g_cp_device_status, static_cast<int>(CP_ERR_DEVICE_TIMEOUT));
}

}  // namespace

// ------------------------------------------------------------ host side
namespace {
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

bool make_map(CUtensorMap *map, const void *base, int64_t D, int64_t heads, int64_t rows, int64_t outer,
              int box_rows) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(D * 2), static_cast<cuuint64_t>(heads * D * 2),
                             static_cast<cuuint64_t>(rows * heads * D * 2)};
    cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map_f32_4d(CUtensorMap *map, const float *base, int64_t d0, int64_t d1, int64_t d2, int64_t d3, int b0,
                     int b1, int b2) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(d1), static_cast<cuuint64_t>(d2),
                          static_cast<cuuint64_t>(d3)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d0 * 4), static_cast<cuuint64_t>(d0 * d1 * 4),
                             static_cast<cuuint64_t>(d0 * d1 * d2 * 4)};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(b0), static_cast<cuuint32_t>(b1), static_cast<cuuint32_t>(b2), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_map_f32_rows(CUtensorMap *map, const float *base, int64_t cols, int64_t rows, int box_cols) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 4)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), 1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// The plan of a forward launch (see PlanSpec): 128-row query and key tiles,
// cost units of two query tiles (one 256-row block).
PlanSpec fwd_plan_spec(const AttnProblem &p, bool pair_blocks) {
    PlanSpec s{};
    s.q_pos = p.q_pos;
    s.k_pos = p.k_pos;
    s.q_pos_stride = p.q_pos_stride;
    s.k_pos_stride = p.k_pos_stride;
    s.C = p.C;
    s.kpr = (p.k_pos_stride == 0) ? 1 : p.C;
    s.kpos_shift = p.kpos_shift;
    s.Sq = static_cast<int>(p.Sq);
    s.Sk = static_cast<int>(p.Sk);
    s.q_tile = 128;
    s.k_tile = 128;
    s.unit_is_k = 0;
    s.q_group = 2;
    s.pair = pair_blocks ? 1 : 0;
    return s;
}

// Does the plan fit in the kernel's shared-memory tables?
bool fwd_plan_on_chip(int64_t C, int64_t kpr, int64_t Sq, int64_t Sk) {
    const int64_t nqt = (Sq + 127) / 128, nkt = (Sk + 127) / 128;
    return kpr * nkt + C * nqt <= kMaxTables && C * ((nqt + 1) / 2) <= kMaxPairs;
}

template <int D, bool kGP>
cp_status launch_typed(const AttnProblem &p, cudaStream_t stream) {
    using K = Cfg<D>;
    CUtensorMap mq, mk, mv;
    const int64_t kv_outer = p.kv_shared ? p.B : p.C * p.B;
    if (!make_map(&mq, p.q, D, p.N, p.Sq, p.C * p.B, 128) || !make_map(&mk, p.k, D, p.Nkv, p.Sk, kv_outer, 128) ||
        !make_map(&mv, p.v, D, p.Nkv, p.Sk, kv_outer, 128))
        return CP_ERR_CUDA;
    AttnArgs a;
    a.q_pos = p.q_pos;
    a.k_pos = p.k_pos;
    a.q_pos_stride = p.q_pos_stride;
    a.k_pos_stride = p.k_pos_stride;
    a.o = p.o;
    a.lse = p.lse;
    a.C = p.C;
    a.B = static_cast<int>(p.B);
    a.N = static_cast<int>(p.N);
    a.Nkv = static_cast<int>(p.Nkv);
    a.Sq = static_cast<int>(p.Sq);
    a.Sk = static_cast<int>(p.Sk);
    a.nqt = static_cast<int>((p.Sq + 127) / 128);
    a.nkt = static_cast<int>((p.Sk + 127) / 128);
    a.nqb = (a.nqt + 1) / 2;
    a.kv_shift = p.kv_shift;
    a.kv_shared = p.kv_shared ? 1 : 0;
    a.merge_into = p.merge_into ? 1 : 0;
    a.kpr = (p.k_pos_stride == 0) ? 1 : p.C;
    a.kpos_shift = p.kpos_shift;
    a.scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634074);
    a.timeout_ns = p.timeout_ns ? p.timeout_ns : 2000000000ull;
    a.hold = p.hold;
    // query blocks u and nqb-1-u in one work item when that still leaves 8 rounds
    // (then every item costs about the same and the head-major order keeps the
    // CTAs that run together on the same K/V)
    a.pair_blocks = pair_units(a.nqb, p.C, p.B * p.N, sm_count()) ? 1 : 0;
    a.nsp = super_count(a.nqb, a.pair_blocks != 0);
    a.div_nsp = make_fastdiv(static_cast<uint32_t>(a.nsp));
    a.div_n = make_fastdiv(static_cast<uint32_t>(a.N));
    const long long n_items = static_cast<long long>(p.C) * a.nsp * p.B * p.N;
    if (n_items <= 0) return CP_OK;
    a.gp = PlanPtrs{};
    if (kGP) {
        const cp_status st = launch_plan(fwd_plan_spec(p, a.pair_blocks != 0), p.plan, &a.gp, stream);
        if (st != CP_OK) return st;
    }
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(attn_fwd_kernel<D, kGP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        K::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return CP_ERR_CUDA;
    const int grid = static_cast<int>(n_items < sm_count() ? n_items : sm_count());
    attn_fwd_kernel<D, kGP><<<grid, kThreads, K::kSmemBytes, stream>>>(mq, mk, mv, a);
    return last_launch_status();
}

}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

size_t attn_plan_need(int64_t C, int64_t kpr, int64_t Sq, int64_t Sk) {
    if (fwd_plan_on_chip(C, kpr, Sq, Sk)) return 0;
    AttnProblem p{};
    p.C = static_cast<int>(C);
    p.k_pos_stride = (kpr == 1) ? 0 : 1;
    p.Sq = Sq;
    p.Sk = Sk;
    // unpaired query blocks give the longer order, so this covers both
    return plan_bytes(fwd_plan_spec(p, false));
}

cp_status validate_attn(const AttnProblem &p, bool check_plan) {
    if (!p.q || !p.k || !p.v || !p.q_pos || !p.k_pos || !p.o || !p.lse) return CP_ERR_NULL;
    if (p.C < 1 || p.C > kMaxC || p.B < 1 || p.N < 1 || p.Nkv < 1 || p.Sq < 1 || p.Sk < 1) return CP_ERR_SHAPE;
    if (p.D != 64 && p.D != 128) return CP_ERR_UNSUPPORTED;
    if (p.N % p.Nkv != 0) return CP_ERR_DIVISIBILITY;
    if (!(std::isfinite(p.scale) && p.scale > 0.f)) return CP_ERR_ARGUMENT;
    if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !aligned16(p.q_pos) || !aligned16(p.k_pos) ||
        !aligned16(p.lse))
        return CP_ERR_ALIGNMENT;
    // the epilogue writes o rows with 32-byte stores
    if (reinterpret_cast<uintptr_t>(p.o) & 31u) return CP_ERR_ALIGNMENT;
    const int64_t nqt = (p.Sq + 127) / 128, nkt = (p.Sk + 127) / 128;
    const int64_t kpr = (p.k_pos_stride == 0) ? 1 : p.C;
    if (p.Sq > INT32_MAX / 2 || p.Sk > INT32_MAX / 2 || p.B * p.N * p.C > INT32_MAX / 4 ||
        static_cast<int64_t>(p.C) * ((nqt + 1) / 2) * p.B * p.N > INT32_MAX || kpr * nkt + p.C * nqt > INT32_MAX / 8)
        return CP_ERR_SHAPE;
    if (check_plan && !fwd_plan_on_chip(p.C, kpr, p.Sq, p.Sk)) {
        if (!p.plan || p.plan_bytes < attn_plan_need(p.C, kpr, p.Sq, p.Sk)) return CP_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(p.plan) & 255u) return CP_ERR_ALIGNMENT;
    }
    if (p.kv_shift < 0 || p.kv_shift >= p.C || p.kpos_shift < 0 || p.kpos_shift >= p.C) return CP_ERR_ARGUMENT;
    return CP_OK;
}

cp_status launch_attn(const AttnProblem &p, cudaStream_t stream) {
    cp_status st = validate_attn(p);
    if (st != CP_OK) return st;
    const bool on_chip = fwd_plan_on_chip(p.C, (p.k_pos_stride == 0) ? 1 : p.C, p.Sq, p.Sk);
    if (on_chip) return p.D == 128 ? launch_typed<128, false>(p, stream) : launch_typed<64, false>(p, stream);
    return p.D == 128 ? launch_typed<128, true>(p, stream) : launch_typed<64, true>(p, stream);
}

}  // namespace cpattn

extern "C" cp_status cp_attn_workspace_size(int64_t B, int64_t Sq, int64_t Sk, int64_t N, int64_t Nkv, int64_t D,
                                            size_t *bytes) {
    if (!bytes) return CP_ERR_NULL;
    if (B < 1 || Sq < 1 || Sk < 1 || N < 1 || Nkv < 1 || D < 1) return CP_ERR_SHAPE;
    *bytes = cpattn::attn_plan_need(1, 1, Sq, Sk);
    return CP_OK;
}

extern "C" cp_status cp_attn_partial_ws(const void *q, const void *k, const void *v, const int32_t *q_pos,
                                        const int32_t *k_pos, int64_t B, int64_t Sq, int64_t Sk, int64_t N,
                                        int64_t Nkv, int64_t D, float scale, float *o, float *lse, void *workspace,
                                        size_t ws_bytes, cudaStream_t stream) {
    cpattn::AttnProblem p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.q_pos = q_pos;
    p.k_pos = k_pos;
    p.o = o;
    p.lse = lse;
    p.C = 1;
    p.B = B;
    p.N = N;
    p.Nkv = Nkv;
    p.D = D;
    p.Sq = Sq;
    p.Sk = Sk;
    p.scale = scale;
    p.plan = workspace;
    p.plan_bytes = workspace ? ws_bytes : 0;
    return cpattn::launch_attn(p, stream);
}

extern "C" cp_status cp_attn_partial(const void *q, const void *k, const void *v, const int32_t *q_pos,
                                     const int32_t *k_pos, int64_t B, int64_t Sq, int64_t Sk, int64_t N,
                                     int64_t Nkv, int64_t D, float scale, float *o, float *lse,
                                     cudaStream_t stream) {
    cpattn::AttnProblem p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.q_pos = q_pos;
    p.k_pos = k_pos;
    p.q_pos_stride = 0;
    p.k_pos_stride = 0;
    p.o = o;
    p.lse = lse;
    p.C = 1;
    p.B = B;
    p.N = N;
    p.Nkv = Nkv;
    p.D = D;
    p.Sq = Sq;
    p.Sk = Sk;
    p.kv_shift = 0;
    p.kpos_shift = 0;
    p.scale = scale;
    return cpattn::launch_attn(p, stream);
}

extern "C" cp_status cp_selftest_stalled_producer(const void *q, const void *k, const void *v, const int32_t *pos,
                                                  float *o, float *lse, uint64_t timeout_ns, cudaStream_t stream) {
    if (timeout_ns < 1000000ull || timeout_ns > 2000000000ull) return CP_ERR_ARGUMENT;
    int *flag = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&flag), cpattn::g_cp_never_set) != cudaSuccess)
        return CP_ERR_CUDA;
    cpattn::AttnProblem p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.q_pos = pos;
    p.k_pos = pos;
    p.o = o;
    p.lse = lse;
    p.C = 1;
    p.B = 1;
    p.N = 1;
    p.Nkv = 1;
    p.D = 64;
    p.Sq = 128;
    p.Sk = 128;
    p.scale = 0.125f;
    p.hold = flag;
    p.timeout_ns = timeout_ns;
    return cpattn::launch_attn(p, stream);
}

extern "C" cp_status cp_device_status(int *code, int clear, cudaStream_t stream) {
    if (!code) return CP_ERR_NULL;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return CP_ERR_CUDA;
    int v = 0, vb = 0;
    if (cudaMemcpyFromSymbol(&v, cpattn::g_cp_device_status, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(cpattn::g_cp_device_status, &zero, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
    }
    // the backward and tf32 kernels keep their own words (other translation units)
    int vt = 0;
    cp_status st = cpattn::read_bwd_device_status(&vb, clear != 0);
    if (st == CP_OK) st = cpattn::read_tf32_device_status(&vt, clear != 0);
    if (st != CP_OK) return st;
    *code = v != 0 ? v : (vb != 0 ? vb : vt);
    return CP_OK;
}
