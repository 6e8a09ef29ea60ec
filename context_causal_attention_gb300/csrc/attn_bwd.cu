// attn_bwd.cu -- backward of the partial causal attention with explicit
// positions on the sm_103a tensor cores (tcgen05 + TMEM + TMA), and the ring
// backward over C virtual ranks built from it.
//
// What it computes ("On Context Parallelism", Peer-to-peer / Backward: the
// tile backward attention_tile_backward(q, k, v, output, grad_output, lse,
// q_positions, kv_positions, scale) -> (dq, dk, dv), which receives the FINAL
// output and lse of the whole attention): over the visible pairs
// (k_pos[j] <= q_pos[i]) with p_ij = e^{scale <q_i, k_j> - lse_i},
//   dv_j = sum_i p_ij dO_i,   dp_ij = <dO_i, v_j>,
//   ds_ij = p_ij (dp_ij - delta_i),   delta_i = <dO_i, o_i>,
//   dq_i = scale sum_j ds_ij k_j,     dk_j = scale sum_i ds_ij q_i
// (the chain rule of the forward; with N > Nkv a KV head's gradients sum over
// its query heads).
//
// Three kernels:
//   bwd_stats_kernel  per query row: nl2 = -lse log2(e) (-inf for rows that see
//                     nothing and for padding) and nd = -delta; HBM-bound.
//   bwd_dkdv_kernel   K/V-stationary.  Work item = (rank, b, KV head, 128-key
//                     tile); it streams the 128-row Q / dO tiles (of every query
//                     head of the group) that can see the keys and keeps
//                     dV += P^T dO and dK += dS^T Q in TMEM.
//   bwd_dq_kernel     Q-stationary.  Work item = (rank, b, head, 128-query tile);
//                     it streams the 128-key K / V tiles the queries can see and
//                     keeps dQ += dS K in TMEM.
// S and dP are formed in both (seven 128x128xD-class products per tile pair
// instead of five), in exchange for no atomics and deterministic sums.
// Both deal their work items like the forward (cp_sched.cuh): stationary tiles
// u and nt-1-u of a rank back to back in one item when the launch is large
// enough, equal-cost items head-major, longest first, boustrophedon.
//
// Both kernels: one persistent CTA per SM, 384 threads.
//   warp 0      TMA producer (stationary tiles once per item, a 2-stage ring
//               of streamed tiles);
//   warp 1      TMEM allocator (512 columns) and the single MMA-issuing thread;
//   warps 2-3   idle;
//   warps 4-11  compute: two warps per TMEM lane quarter (quarter = warp % 4,
//               one row of the stationary tile per thread); warps 4-7 take
//               columns 0..31 of every 64-column half, warps 8-11 columns
//               32..63, so two warps per SM sub-partition hide each other's
//               shared-memory and TMEM latencies.
// TMEM: scores S (or S^T) in columns 0..127, dP in 128..255 (128 x 128 fp32
// each, all products N = 128), then the fp32 accumulators (dV | dK, or dQ).
// The compute warps work through a streamed tile in two 64-column halves and
// write P / dS back over columns they have read, as packed bf16; the
// gradient MMAs of the first half (K = 64) run while the second half is
// computed.  The next tile's S and dP are issued after both halves' gradient
// MMAs (the tensor pipe runs them in order).
// Every mbarrier wait is bounded (2 s); a CTA that times out unwinds, lets its
// copies and MMAs land, frees TMEM and records CP_ERR_DEVICE_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "cp_internal.h"
#include "cp_hold.cuh"
#include "cp_ptx.cuh"
#include "cp_sched.cuh"
#include "cp_rounds.cuh"

namespace cpattn {
namespace {

__device__ int g_cp_bwd_status = 0;

constexpr int kBThreads = 384;  // three warps per SM sub-partition: at most 168 registers
constexpr int kBStages = 2;
constexpr uint32_t kBTmemCols = 512;
constexpr uint32_t kNegInfBits = 0xff800000u;
constexpr int kComputeWarps = 8;

template <int D>
struct Tiles {
    static constexpr int kAtoms = D / 64;
    static constexpr int kTile = 128 * D * 2;   // 128-row bf16 tile
    static constexpr int kAtom = 128 * 128;     // one 64-column swizzle atom of it
};

// K/V-stationary kernel: K, V | Q, dO stages | nl2/nd strips per stage |
// tables | order | cost | segments | barriers | misc.
template <int D>
struct CfgKV : Tiles<D> {
    using T = Tiles<D>;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = T::kTile;
    static constexpr int kOffQ = 2 * T::kTile;
    static constexpr int kOffDO = kOffQ + kBStages * T::kTile;
    static constexpr int kOffStat = kOffDO + kBStages * T::kTile;  // per stage: nl2[128] | nd[128]
    static constexpr int kOffTab = kOffStat + kBStages * 1024;
    static constexpr int kOffOrder = kOffTab + kBwdMaxTables * 8;
    static constexpr int kOffCost = kOffOrder + kBwdMaxPairs * 4;
    static constexpr int kOffSeg = kOffCost + kBwdMaxPairs * 4;
    static constexpr int kOffBar = kOffSeg + (kBwdMaxPairs + 2) * 4;
    // kv_full, kv_empty, qd_full[S], qd_empty[S], s_full, p_half, p_full, o_full, o_empty, drain
    // (p_half, p_full, o_empty: one arrival per compute warp)
    static constexpr int kNumBars = 2 + 2 * kBStages + 6;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kMiscBytes = 16 + kMaxC * 4 + kBwdMaxTables / 8;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Q-stationary kernel: Q, dO | K, V stages | tables | order | cost | segments | ...
template <int D>
struct CfgQ : Tiles<D> {
    using T = Tiles<D>;
    static constexpr int kOffQ = 0;
    static constexpr int kOffDO = T::kTile;
    static constexpr int kOffK = 2 * T::kTile;
    static constexpr int kOffV = kOffK + kBStages * T::kTile;
    static constexpr int kOffTab = kOffV + kBStages * T::kTile;
    static constexpr int kOffOrder = kOffTab + kBwdMaxTables * 8;
    static constexpr int kOffCost = kOffOrder + kBwdMaxPairs * 4;
    static constexpr int kOffSeg = kOffCost + kBwdMaxPairs * 4;
    static constexpr int kOffBar = kOffSeg + (kBwdMaxPairs + 2) * 4;
    // qd_full, qd_empty, kv_full[S], kv_empty[S], s_full, p_half, p_full, o_full, o_empty, drain
    static constexpr int kNumBars = 2 + 2 * kBStages + 6;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kMiscBytes = 16 + kMaxC * 4 + kBwdMaxTables / 8;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct BwdArgs {
    const int32_t *q_pos, *k_pos;
    long long q_pos_stride, k_pos_stride;
    const float *nl2, *nd;  // [C*B*N][sq_pad]
    long long sq_pad;
    float *dq, *dk, *dv;
    int C, B, N, Nkv, Sq, Sk;
    int nq, nk;  // 128-row query / key tiles
    int kv_shift, kpos_shift, kpr;
    int accumulate;
    float scale, scale_log2;
    unsigned long long timeout_ns;
    int pair;         // a super-block holds stationary tiles u and nt-1-u (else u alone)
    FastDiv div_nsp, div_h;  // by super-blocks per rank, heads per item
    PlanPtrs gp;      // the launch's plan in global memory (kernels with kGlobalPlan)
    const int *hold;  // failure injection (self-test only), else null
};

// (min, max) of the positions of one 128-row tile (one warp per tile); when
// `arith` is given, bit g is set if the positions are p, p+1, p+2, ...
__device__ __forceinline__ void tile_table(const int32_t *p, int row0, int lim, int lane, int2 *out, uint32_t *arith,
                                           int g) {
    int mn = INT_MAX, mx = INT_MIN, vals[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int row = row0 + lane + 32 * m;
        vals[m] = (row < lim) ? __ldg(p + row) : 0;
        if (row < lim) {
            mn = min(mn, vals[m]);
            mx = max(mx, vals[m]);
        }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) *out = make_int2(mn, mx);
    if (arith) {
        const int first = __shfl_sync(0xffffffffu, vals[0], 0);
        bool ok = true;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int row = row0 + lane + 32 * m;
            if (row < lim) ok &= (static_cast<long long>(vals[m]) == static_cast<long long>(first) + lane + 32 * m);
        }
        ok = __all_sync(0xffffffffu, ok);
        if (lane == 0 && ok) atomicOr(arith + (g >> 5), 1u << (g & 31));
    }
}

// ---- visibility of streamed tiles
// K/V-stationary: query tile qt (of rank r) can see key tile (kmin = its
// smallest key position) iff its largest query position >= kmin.  With the
// tiles' largest positions non-decreasing (`sorted`) the visible tiles are a
// suffix found by bisection.
__device__ __forceinline__ int first_q(const int2 *qt_r, int nq, int kmin, bool sorted) {
    if (sorted) {
        int lo = 0, hi = nq;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (qt_r[mid].y >= kmin) hi = mid; else lo = mid + 1;
        }
        return lo;
    }
    int qt = 0;
    while (qt < nq && qt_r[qt].y < kmin) ++qt;
    return qt;
}
__device__ __forceinline__ int next_q(int qt, const int2 *qt_r, int nq, int kmin) {
    while (qt < nq && qt_r[qt].y < kmin) ++qt;
    return qt;
}
__device__ __forceinline__ int count_q(const int2 *qt_r, int nq, int kmin, bool sorted) {
    if (sorted) return nq - first_q(qt_r, nq, kmin, true);
    int c = 0;
    for (int qt = 0; qt < nq; ++qt) c += (qt_r[qt].y >= kmin);
    return c;
}
// Q-stationary: key tile kt can be seen iff its smallest position <= qmax;
// with the smallest positions non-decreasing the visible tiles are a prefix.
__device__ __forceinline__ int next_k(int kt, const int2 *kt_o, int nk, int qmax, bool sorted) {
    for (; kt < nk; ++kt) {
        if (kt_o[kt].x <= qmax) return kt;
        if (sorted) return nk;
    }
    return nk;
}
__device__ __forceinline__ int count_k(const int2 *kt_o, int nk, int qmax, bool sorted) {
    if (sorted) {
        int lo = 0, hi = nk;  // first tile with kmin > qmax
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (kt_o[mid].x <= qmax) lo = mid + 1; else hi = mid;
        }
        return lo;
    }
    int c = 0;
    for (int kt = 0; kt < nk; ++kt) c += (kt_o[kt].x <= qmax);
    return c;
}

// Row of D fp32 values from TMEM columns [col, col + D) of this thread's lane,
// times `mul`, written to (or added to) dst (32-byte aligned).  Warp-collective.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, float *dst, float mul, bool write, bool add) {
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(taddr + c0, v);
        if (write) {
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
                float r8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) r8[e] = __uint_as_float(v[c + e]) * mul;
                if (add) {
                    float o8[8];
                    ld_global_v8(dst + c0 + c, o8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) r8[e] += o8[e];
                }
                st_global_v8(dst + c0 + c, r8[0], r8[1], r8[2], r8[3], r8[4], r8[5], r8[6], r8[7]);
            }
        }
    }
}

template <int D>
__device__ __forceinline__ void zero_row(float *dst) {
#pragma unroll
    for (int c = 0; c < D; c += 8) st_global_v8(dst + c, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Releases one half of a streamed tile to the MMA issuer (warp-collective).
__device__ __forceinline__ void release_half(uint64_t *bar, int lane) {
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// ======================================================================
// dK / dV: K/V-stationary
// ======================================================================
// kGlobalPlan (both backward kernels): the plan was written to global memory
// by the pre-pass (else every CTA builds it in shared memory).
template <int D, bool kGlobalPlan>
__global__ void __launch_bounds__(kBThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmNL2, const __grid_constant__ CUtensorMap tmND,
                    const BwdArgs a) {
    using K = CfgKV<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int2 *tab_s = reinterpret_cast<int2 *>(smem + K::kOffTab);
    int *order_s = reinterpret_cast<int *>(smem + K::kOffOrder);
    int *cost_s = reinterpret_cast<int *>(smem + K::kOffCost);  // per (rank, key tile): visible query tiles
    int *seg_s = reinterpret_cast<int *>(smem + K::kOffSeg);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + K::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + K::kOffMisc + 4);
    int *sorted_s = reinterpret_cast<int *>(smem + K::kOffMisc + 16);  // per rank
    uint32_t *bits_s = reinterpret_cast<uint32_t *>(smem + K::kOffMisc + 16 + kMaxC * 4);  // per query tile
    const int *order = kGlobalPlan ? a.gp.order : order_s;
    const int *cost = kGlobalPlan ? a.gp.cost : cost_s;
    const int *seg_first = kGlobalPlan ? a.gp.seg_first : seg_s;
    const int *sorted_flag = kGlobalPlan ? a.gp.qsorted : sorted_s;
    const uint32_t *arith_bits = kGlobalPlan ? a.gp.qbits : bits_s;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + K::kOffBar);
    uint64_t *kv_full = bar, *kv_empty = bar + 1, *qd_full = bar + 2, *qd_empty = bar + 2 + kBStages;
    uint64_t *s_full = bar + 2 + 2 * kBStages, *p_half = s_full + 1, *p_full = s_full + 2, *o_full = s_full + 3,
             *o_empty = s_full + 4, *drain = s_full + 5;
    const int2 *ktab = kGlobalPlan ? a.gp.ktab : tab_s;                // [kpr][nk] key tiles
    const int2 *qtab = kGlobalPlan ? a.gp.qtab : tab_s + a.kpr * a.nk;  // [C][nq] query tiles

    if (tid == 0) {
        *abort_flag = 0;
        if (!kGlobalPlan)
            for (int w = 0; w < kBwdMaxTables / 32; ++w) bits_s[w] = 0u;
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(qd_full + s, 1);
            mbar_init(qd_empty + s, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_half, kComputeWarps);
        mbar_init(p_full, kComputeWarps);
        mbar_init(o_full, 1);
        mbar_init(o_empty, kComputeWarps);
        mbar_init(drain, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmDO);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmNL2);
        tma_prefetch_desc(&tmND);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kBTmemCols);
        tmem_relinquish();
    }
    __syncthreads();
    if constexpr (!kGlobalPlan) {
        {
            const int nkk = a.kpr * a.nk, total = nkk + a.C * a.nq;
            for (int g = warp; g < total; g += kBThreads / 32) {
                if (g < nkk) {
                    const int j = g / a.nk, kt = g - (g / a.nk) * a.nk;
                    tile_table(a.k_pos + j * a.k_pos_stride, kt * 128, a.Sk, lane, tab_s + g, nullptr, 0);
                } else {
                    const int gq = g - nkk, r = gq / a.nq, qt = gq - (gq / a.nq) * a.nq;
                    tile_table(a.q_pos + r * a.q_pos_stride, qt * 128, a.Sq, lane, tab_s + g, bits_s, gq);
                }
            }
        }
        __syncthreads();
        if (tid < a.C) {
            int ok = 1;
            for (int qt = 1; qt < a.nq; ++qt) ok &= (qtab[tid * a.nq + qt].y >= qtab[tid * a.nq + qt - 1].y);
            sorted_s[tid] = ok;
        }
        __syncthreads();
        const int np = a.C * a.nk;
        for (int p = tid; p < np; p += kBThreads) {
            const int r = p / a.nk, kt = p - (p / a.nk) * a.nk;
            const int owner = (a.kpr == 1) ? 0 : (r + a.kpos_shift) % a.C;
            cost_s[p] = count_q(qtab + r * a.nq, a.nq, ktab[owner * a.nk + kt].x, sorted_s[r] != 0);
        }
        __syncthreads();
        build_segments<kBThreads>(cost_s, a.C, a.nk, a.pair != 0, order_s, seg_s);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_items = a.C * super_count(a.nk, a.pair != 0) * a.B * a.Nkv;
    const int n_rounds = (n_items + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    const int g_heads = a.N / a.Nkv;
    uint8_t *sK = smem + K::kOffK, *sV = smem + K::kOffV, *sQ = smem + K::kOffQ, *sDO = smem + K::kOffDO;
    float *sStat = reinterpret_cast<float *>(smem + K::kOffStat);

    // key tile `unit` of super item x -> (rank, key tile, b, KV head, ...)
    auto decode = [&](const SuperItem &x, int unit, int &r, int &kt, int &b, int &hk, int &owner, int &kvr, int &pr) {
        r = x.r;
        kt = unit;
        pr = r * a.nk + kt;
        b = static_cast<int>(fdiv(static_cast<uint32_t>(x.bh), a.div_h));
        hk = x.bh - b * a.Nkv;
        owner = (a.kpr == 1) ? 0 : (r + a.kpos_shift) % a.C;
        kvr = (r + a.kv_shift) % a.C;
    };

    if (warp == 0) {
        // -------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t it = 0, t = 0;
            bool ok = true;
            if (a.hold) ok = hold_wait(a.hold, a.timeout_ns, abort_flag);
            int kv_par = -1;
            uint32_t qd_issued = 0, qd_par = 0;
            int seg = 0;  // segment cursor of decode_super
            for (int rk = 0; rk < n_rounds && ok; ++rk) {
                const RoundWork rw = work_of_round(rk, n_items, a.pair != 0);
                if (rw.idx < 0) continue;
                const SuperItem sup = decode_super(rw.idx, a.B * a.Nkv, order, seg_first, a.div_nsp, seg);
                for (int part = rw.p0; part < rw.p1 && ok; ++part) {
                    const int unit = super_part(sup.u, part, a.nk, a.pair != 0);
                    if (unit < 0) continue;
                    int r, kt, b, hk, owner, kvr, pr;
                    decode(sup, unit, r, kt, b, hk, owner, kvr, pr);
                    if (cost[pr] == 0) continue;
                    if (!mbar_wait(kv_empty, (it & 1u) ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    mbar_arrive_expect_tx(kv_full, 2 * K::kTile);
                    kv_par = static_cast<int>(it & 1u);
                    const int kvrow = kvr * a.B + b;
                    for (int at = 0; at < K::kAtoms; ++at) {
                        tma_load_4d(sK + at * K::kAtom, &tmK, kv_full, 64 * at, hk, kt * 128, kvrow);
                        tma_load_4d(sV + at * K::kAtom, &tmV, kv_full, 64 * at, hk, kt * 128, kvrow);
                    }
                    ++it;
                    const int2 *qt_r = qtab + r * a.nq;
                    const int kmin = ktab[owner * a.nk + kt].x;
                    const bool srt = sorted_flag[r] != 0;
                    const int qrow = r * a.B + b;
                    for (int hh = 0; hh < g_heads && ok; ++hh) {
                        const int h = hk * g_heads + hh;
                        const int srow = qrow * a.N + h;
                        for (int qt = first_q(qt_r, a.nq, kmin, srt); qt < a.nq; qt = next_q(qt + 1, qt_r, a.nq, kmin)) {
                            const uint32_t st = t % kBStages, ph = (t / kBStages) & 1u;
                            if (!mbar_wait(qd_empty + st, ph ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                            mbar_arrive_expect_tx(qd_full + st, 2 * K::kTile + 1024);
                            for (int at = 0; at < K::kAtoms; ++at) {
                                tma_load_4d(sQ + st * K::kTile + at * K::kAtom, &tmQ, qd_full + st, 64 * at, h, qt * 128,
                                            qrow);
                                tma_load_4d(sDO + st * K::kTile + at * K::kAtom, &tmDO, qd_full + st, 64 * at, h, qt * 128,
                                            qrow);
                            }
                            tma_load_2d(sStat + st * 256, &tmNL2, qd_full + st, qt * 128, srow);
                            tma_load_2d(sStat + st * 256 + 128, &tmND, qd_full + st, qt * 128, srow);
                            qd_issued |= 1u << st;
                            qd_par = (qd_par & ~(1u << st)) | (ph << st);
                            ++t;
                        }
                    }
                }
            }
            if (!ok) {
                // let every copy already issued land before shared memory goes away
                volatile int no_abort = 0;
                const unsigned long long drain_ns = 100000000ull;
                if (kv_par >= 0) mbar_wait(kv_full, static_cast<uint32_t>(kv_par), &no_abort, drain_ns);
                for (int st = 0; st < kBStages; ++st)
                    if ((qd_issued >> st) & 1u) mbar_wait(qd_full + st, (qd_par >> st) & 1u, &no_abort, drain_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T: 128 keys x 128 queries
            constexpr uint32_t kIdG = idesc_bf16_f32(128, D, 0, 1);    // dV, dK: B operand MN-major
            constexpr uint64_t kStU = K::kTile >> 4;                   // one stage, descriptor units
            constexpr uint64_t kHalfU = (64 * 128) >> 4;               // 64 rows of a swizzled tile
            const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024), dV = smem_desc_sw128(smem_u32(sV), 16, 1024);
            const uint64_t dQk = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dOk = smem_desc_sw128(smem_u32(sDO), 16, 1024);
            const uint64_t dQm = smem_desc_sw128(smem_u32(sQ), K::kAtom, 1024);
            const uint64_t dOm = smem_desc_sw128(smem_u32(sDO), K::kAtom, 1024);
            uint32_t it = 0, t = 0;
            bool ok = true;
            int seg = 0;  // segment cursor of decode_super
            for (int rk = 0; rk < n_rounds && ok; ++rk) {
                const RoundWork rw = work_of_round(rk, n_items, a.pair != 0);
                if (rw.idx < 0) continue;
                const SuperItem sup = decode_super(rw.idx, a.B * a.Nkv, order, seg_first, a.div_nsp, seg);
                for (int part = rw.p0; part < rw.p1 && ok; ++part) {
                    const int unit = super_part(sup.u, part, a.nk, a.pair != 0);
                    if (unit < 0) continue;
                    int r, kt, b, hk, owner, kvr, pr;
                    decode(sup, unit, r, kt, b, hk, owner, kvr, pr);
                    const int n = g_heads * cost[pr];
                    if (n == 0) continue;
                    if (!mbar_wait(kv_full, it & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    for (int i = 0; i < n; ++i, ++t) {
                        const uint32_t st = t % kBStages, ph = (t / kBStages) & 1u;
                        if (!mbar_wait(qd_full + st, ph, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        // S^T and dP^T overwrite the previous tile's P^T / dS^T: in
                        // issue order after that tile's gradient MMAs
                        umma_ss_kgroup<D / 16, 1024, 1024>(tmem, dK, dQk + st * kStU, kIdS);
                        umma_ss_kgroup<D / 16, 1024, 1024>(tmem + 128, dV, dOk + st * kStU, kIdS);
                        umma_commit(s_full);
                        if (i == n - 1) umma_commit(kv_empty);  // K and V are read by S^T / dP^T only
                        // dV += P^T dO, dK += dS^T Q over the tile's first 64 queries,
                        // then over the second 64; `first` overwrites the accumulators
                        if (!mbar_wait(p_half, t & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        if (i == 0 && !mbar_wait(o_empty, (it & 1u) ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        umma_ts_k64_split(tmem + 256, tmem, dOm + st * kStU, kIdG, i == 0 ? 0u : 1u);
                        umma_ts_k64_split(tmem + 256 + D, tmem + 128, dQm + st * kStU, kIdG, i == 0 ? 0u : 1u);
                        if (!mbar_wait(p_full, t & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        umma_ts_k64_split(tmem + 256, tmem + 64, dOm + st * kStU + kHalfU, kIdG, 1u);
                        umma_ts_k64_split(tmem + 256 + D, tmem + 192, dQm + st * kStU + kHalfU, kIdG, 1u);
                        umma_commit(qd_empty + st);
                    }
                    if (!ok) break;
                    umma_commit(o_full);
                    ++it;
                }
            }
            // no MMA may still be running when TMEM is released
            umma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait(drain, 0, &no_abort, 100000000ull);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // -------------------------------------------------------- compute (one key row per thread)
        const int quarter = warp & 3;
        const int grp = (warp - 4) >> 2;  // columns 32 grp .. 32 grp + 31 of each half
        const int row_in = quarter * 32 + lane;
        const uint32_t tA = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint64_t sl2x2 = f2_packf(a.scale_log2, a.scale_log2);
        uint32_t it = 0, t = 0;
        bool ok = true;
        int seg = 0;  // segment cursor of decode_super
        for (int rk = 0; rk < n_rounds && ok; ++rk) {
            const RoundWork rw = work_of_round(rk, n_items, a.pair != 0);
            if (rw.idx < 0) continue;
            const SuperItem sup = decode_super(rw.idx, a.B * a.Nkv, order, seg_first, a.div_nsp, seg);
            for (int part = rw.p0; part < rw.p1 && ok; ++part) {
                const int unit = super_part(sup.u, part, a.nk, a.pair != 0);
                if (unit < 0) continue;
                int r, kt, b, hk, owner, kvr, pr;
                decode(sup, unit, r, kt, b, hk, owner, kvr, pr);
                const int key = kt * 128 + row_in;
                const bool key_valid = key < a.Sk;
                const int kpos = key_valid ? __ldg(a.k_pos + owner * a.k_pos_stride + key) : INT_MAX;
                const long long krow = (static_cast<long long>(kvr * a.B + b) * a.Sk + key) * a.Nkv + hk;
                // each group writes half of the row's D columns
                float *dk_row = a.dk + krow * D + grp * (D / 2);
                float *dv_row = a.dv + krow * D + grp * (D / 2);
                if (cost[pr] == 0) {
                    // no query sees these keys: their gradients are zero
                    if (key_valid && !a.accumulate) {
                        zero_row<D / 2>(dk_row);
                        zero_row<D / 2>(dv_row);
                    }
                    continue;
                }
                const int2 kmm = ktab[owner * a.nk + kt];
                const int2 *qt_r = qtab + r * a.nq;
                const bool srt = sorted_flag[r] != 0;
                const int32_t *qpos_r = a.q_pos + r * a.q_pos_stride;
                for (int hh = 0; hh < g_heads && ok; ++hh) {
                    for (int qt = first_q(qt_r, a.nq, kmm.x, srt); qt < a.nq;
                         qt = next_q(qt + 1, qt_r, a.nq, kmm.x), ++t) {
                        const uint32_t st = t % kBStages;
                        if (!mbar_wait_warp(s_full, t & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        const int2 qmm = qt_r[qt];
                        const int q0 = qt * 128;
                        const bool need_mask = kmm.y > qmm.x || q0 + 128 > a.Sq;
                        const int gq = r * a.nq + qt;
                        const bool arith = (arith_bits[gq >> 5] >> (gq & 31)) & 1u;
    #pragma unroll 1
                        for (int h = 0; h < 2; ++h) {
                            // this warp's columns: cb .. cb+31 = queries q0 + cb ..
                            const int cb = 64 * h + 32 * grp;
                            uint32_t s[32], dp[32];
                            tmem_ld32_nowait(tA + cb, s);
                            tmem_ld32_nowait(tA + 128 + cb, dp);
                            tmem_wait_ld32(s);
                            tmem_wait_ld32(dp);
                            if (need_mask) {
                                const int qh = q0 + cb;
                                const int nvalid = min(32, a.Sq - qh);
                                if (arith) {
                                    // query positions qmin + cb + c: column c visible iff c >= kpos - qmin - cb
                                    const long long dlo = static_cast<long long>(kpos) - qmm.x - cb;
                                    const int lo = dlo <= 0 ? 0 : (dlo > 32 ? 32 : static_cast<int>(dlo));
    #pragma unroll
                                    for (int c = 0; c < 32; ++c)
                                        if (c < lo || c >= nvalid) s[c] = kNegInfBits;
                                } else {
    #pragma unroll
                                    for (int c0 = 0; c0 < 32; c0 += 16) {
    #pragma unroll
                                        for (int c = c0; c < c0 + 16; ++c) {
                                            const int qp = (c < nvalid) ? __ldg(qpos_r + qh + c) : INT_MIN;
                                            if (kpos > qp) s[c] = kNegInfBits;
                                        }
                                        asm volatile("" ::: "memory");
                                    }
                                }
                            }
                            // P^T = 2^(s sl2 + nl2_c), dS^T = P^T (dP^T + nd_c), column stats from the stage
                            const float *nl = sStat + st * 256 + cb, *nd = nl + 128;
                            uint32_t pk_p[16], pk_d[16];
    #pragma unroll
                            for (int c = 0; c < 32; c += 4) {
                                const float4 l4 = *reinterpret_cast<const float4 *>(nl + c);
                                const float4 d4 = *reinterpret_cast<const float4 *>(nd + c);
                                float x0, x1, x2, x3, g0, g1, g2, g3;
                                f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, f2_packf(l4.x, l4.y)), x0, x1);
                                f2_unpack(f2_fma(f2_pack(s[c + 2], s[c + 3]), sl2x2, f2_packf(l4.z, l4.w)), x2, x3);
                                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1), p2 = fast_exp2(x2),
                                            p3 = fast_exp2(x3);
                                f2_unpack(f2_fma(f2_packf(p0, p1),
                                                 f2_add(f2_pack(dp[c], dp[c + 1]), f2_packf(d4.x, d4.y)), 0ull),
                                          g0, g1);
                                f2_unpack(f2_fma(f2_packf(p2, p3),
                                                 f2_add(f2_pack(dp[c + 2], dp[c + 3]), f2_packf(d4.z, d4.w)), 0ull),
                                          g2, g3);
                                pk_p[c >> 1] = pack_bf16x2(p0, p1);
                                pk_p[(c >> 1) + 1] = pack_bf16x2(p2, p3);
                                pk_d[c >> 1] = pack_bf16x2(g0, g1);
                                pk_d[(c >> 1) + 1] = pack_bf16x2(g2, g3);
                            }
                            // packed over the first 16 of this warp's own 32 columns (already
                            // read; no other warp reads them): the MMA finds the half's
                            // 64 packed queries at columns 64h + {0..15, 32..47}
                            tmem_st16_nowait(tA + cb, pk_p);
                            tmem_st16_nowait(tA + 128 + cb, pk_d);
                            release_half(h == 0 ? p_half : p_full, lane);
                        }
                    }
                }
                if (!ok) break;
                if (!mbar_wait_warp(o_full, it & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                store_acc_row<D / 2>(tA + 256 + grp * (D / 2), dv_row, 1.f, key_valid, a.accumulate != 0);
                store_acc_row<D / 2>(tA + 256 + D + grp * (D / 2), dk_row, a.scale, key_valid, a.accumulate != 0);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_empty);
                ++it;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kBTmemCols);
    }
    if (tid == 0 && *abort_flag) atomicExch(&g_cp_bwd_status, static_cast<int>(CP_ERR_DEVICE_TIMEOUT));
}

// ======================================================================
// dQ: Q-stationary
// ======================================================================
template <int D, bool kGlobalPlan>
__global__ void __launch_bounds__(kBThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const BwdArgs a) {
    using K = CfgQ<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int2 *tab_s = reinterpret_cast<int2 *>(smem + K::kOffTab);
    int *order_s = reinterpret_cast<int *>(smem + K::kOffOrder);
    int *cost_s = reinterpret_cast<int *>(smem + K::kOffCost);  // per (rank, query tile): visible key tiles
    int *seg_s = reinterpret_cast<int *>(smem + K::kOffSeg);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + K::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + K::kOffMisc + 4);
    int *sorted_s = reinterpret_cast<int *>(smem + K::kOffMisc + 16);  // per key-position rank
    uint32_t *bits_s = reinterpret_cast<uint32_t *>(smem + K::kOffMisc + 16 + kMaxC * 4);  // per key tile
    const int *order = kGlobalPlan ? a.gp.order : order_s;
    const int *cost = kGlobalPlan ? a.gp.cost : cost_s;
    const int *seg_first = kGlobalPlan ? a.gp.seg_first : seg_s;
    const int *sorted_flag = kGlobalPlan ? a.gp.ksorted : sorted_s;
    const uint32_t *arith_bits = kGlobalPlan ? a.gp.kbits : bits_s;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + K::kOffBar);
    uint64_t *qd_full = bar, *qd_empty = bar + 1, *kv_full = bar + 2, *kv_empty = bar + 2 + kBStages;
    uint64_t *s_full = bar + 2 + 2 * kBStages, *p_half = s_full + 1, *p_full = s_full + 2, *o_full = s_full + 3,
             *o_empty = s_full + 4, *drain = s_full + 5;
    const int2 *qtab = kGlobalPlan ? a.gp.qtab : tab_s;               // [C][nq] query tiles
    const int2 *ktab = kGlobalPlan ? a.gp.ktab : tab_s + a.C * a.nq;  // [kpr][nk] key tiles

    if (tid == 0) {
        *abort_flag = 0;
        if (!kGlobalPlan)
            for (int w = 0; w < kBwdMaxTables / 32; ++w) bits_s[w] = 0u;
        mbar_init(qd_full, 1);
        mbar_init(qd_empty, 1);
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(kv_full + s, 1);
            mbar_init(kv_empty + s, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_half, kComputeWarps);
        mbar_init(p_full, kComputeWarps);
        mbar_init(o_full, 1);
        mbar_init(o_empty, kComputeWarps);
        mbar_init(drain, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmDO);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kBTmemCols);
        tmem_relinquish();
    }
    __syncthreads();
    if constexpr (!kGlobalPlan) {
        {
            const int nqq = a.C * a.nq, total = nqq + a.kpr * a.nk;
            for (int g = warp; g < total; g += kBThreads / 32) {
                if (g < nqq) {
                    const int r = g / a.nq, qt = g - (g / a.nq) * a.nq;
                    tile_table(a.q_pos + r * a.q_pos_stride, qt * 128, a.Sq, lane, tab_s + g, nullptr, 0);
                } else {
                    const int gk = g - nqq, j = gk / a.nk, kt = gk - (gk / a.nk) * a.nk;
                    tile_table(a.k_pos + j * a.k_pos_stride, kt * 128, a.Sk, lane, tab_s + g, bits_s, gk);
                }
            }
        }
        __syncthreads();
        if (tid < a.kpr) {
            int ok = 1;
            for (int kt = 1; kt < a.nk; ++kt) ok &= (ktab[tid * a.nk + kt].x >= ktab[tid * a.nk + kt - 1].x);
            sorted_s[tid] = ok;
        }
        __syncthreads();
        const int np = a.C * a.nq;
        for (int p = tid; p < np; p += kBThreads) {
            const int r = p / a.nq, qt = p - (p / a.nq) * a.nq;
            const int owner = (a.kpr == 1) ? 0 : (r + a.kpos_shift) % a.C;
            cost_s[p] = count_k(ktab + owner * a.nk, a.nk, qtab[r * a.nq + qt].y, sorted_s[owner] != 0);
        }
        __syncthreads();
        build_segments<kBThreads>(cost_s, a.C, a.nq, a.pair != 0, order_s, seg_s);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_items = a.C * super_count(a.nq, a.pair != 0) * a.B * a.N;
    const int n_rounds = (n_items + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    const int g_heads = a.N / a.Nkv;
    uint8_t *sQ = smem + K::kOffQ, *sDO = smem + K::kOffDO, *sK = smem + K::kOffK, *sV = smem + K::kOffV;

    // query tile `unit` of super item x -> (rank, query tile, b, head, ...)
    auto decode = [&](const SuperItem &x, int unit, int &r, int &qt, int &b, int &h, int &owner, int &kvr, int &pr) {
        r = x.r;
        qt = unit;
        pr = r * a.nq + qt;
        b = static_cast<int>(fdiv(static_cast<uint32_t>(x.bh), a.div_h));
        h = x.bh - b * a.N;
        owner = (a.kpr == 1) ? 0 : (r + a.kpos_shift) % a.C;
        kvr = (r + a.kv_shift) % a.C;
    };

    if (warp == 0) {
        // -------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t it = 0, t = 0;
            bool ok = true;
            if (a.hold) ok = hold_wait(a.hold, a.timeout_ns, abort_flag);
            int qd_par = -1;
            uint32_t kv_issued = 0, kv_par = 0;
            int seg = 0;  // segment cursor of decode_super
            for (int rk = 0; rk < n_rounds && ok; ++rk) {
                const RoundWork rw = work_of_round(rk, n_items, a.pair != 0);
                if (rw.idx < 0) continue;
                const SuperItem sup = decode_super(rw.idx, a.B * a.N, order, seg_first, a.div_nsp, seg);
                for (int part = rw.p0; part < rw.p1 && ok; ++part) {
                    const int unit = super_part(sup.u, part, a.nq, a.pair != 0);
                    if (unit < 0) continue;
                    int r, qt, b, h, owner, kvr, pr;
                    decode(sup, unit, r, qt, b, h, owner, kvr, pr);
                    if (cost[pr] == 0) continue;
                    if (!mbar_wait(qd_empty, (it & 1u) ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    mbar_arrive_expect_tx(qd_full, 2 * K::kTile);
                    qd_par = static_cast<int>(it & 1u);
                    const int qrow = r * a.B + b;
                    for (int at = 0; at < K::kAtoms; ++at) {
                        tma_load_4d(sQ + at * K::kAtom, &tmQ, qd_full, 64 * at, h, qt * 128, qrow);
                        tma_load_4d(sDO + at * K::kAtom, &tmDO, qd_full, 64 * at, h, qt * 128, qrow);
                    }
                    ++it;
                    const int2 *kt_o = ktab + owner * a.nk;
                    const int qmax = qtab[r * a.nq + qt].y;
                    const bool srt = sorted_flag[owner] != 0;
                    const int hk = h / g_heads;
                    const int kvrow = kvr * a.B + b;
                    for (int kt = next_k(0, kt_o, a.nk, qmax, srt); kt < a.nk; kt = next_k(kt + 1, kt_o, a.nk, qmax, srt)) {
                        const uint32_t st = t % kBStages, ph = (t / kBStages) & 1u;
                        if (!mbar_wait(kv_empty + st, ph ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        mbar_arrive_expect_tx(kv_full + st, 2 * K::kTile);
                        for (int at = 0; at < K::kAtoms; ++at) {
                            tma_load_4d(sK + st * K::kTile + at * K::kAtom, &tmK, kv_full + st, 64 * at, hk, kt * 128,
                                        kvrow);
                            tma_load_4d(sV + st * K::kTile + at * K::kAtom, &tmV, kv_full + st, 64 * at, hk, kt * 128,
                                        kvrow);
                        }
                        kv_issued |= 1u << st;
                        kv_par = (kv_par & ~(1u << st)) | (ph << st);
                        ++t;
                    }
                }
            }
            if (!ok) {
                volatile int no_abort = 0;
                const unsigned long long drain_ns = 100000000ull;
                if (qd_par >= 0) mbar_wait(qd_full, static_cast<uint32_t>(qd_par), &no_abort, drain_ns);
                for (int st = 0; st < kBStages; ++st)
                    if ((kv_issued >> st) & 1u) mbar_wait(kv_full + st, (kv_par >> st) & 1u, &no_abort, drain_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);  // S, dP: 128 queries x 128 keys
            constexpr uint32_t kIdG = idesc_bf16_f32(128, D, 0, 1);    // dQ: B operand MN-major
            constexpr uint64_t kStU = K::kTile >> 4;
            constexpr uint64_t kHalfU = (64 * 128) >> 4;
            const uint64_t dQa = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dOa = smem_desc_sw128(smem_u32(sDO), 16, 1024);
            const uint64_t dKb = smem_desc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t dVb = smem_desc_sw128(smem_u32(sV), 16, 1024);
            const uint64_t dKm = smem_desc_sw128(smem_u32(sK), K::kAtom, 1024);
            uint32_t it = 0, t = 0;
            bool ok = true;
            int seg = 0;  // segment cursor of decode_super
            for (int rk = 0; rk < n_rounds && ok; ++rk) {
                const RoundWork rw = work_of_round(rk, n_items, a.pair != 0);
                if (rw.idx < 0) continue;
                const SuperItem sup = decode_super(rw.idx, a.B * a.N, order, seg_first, a.div_nsp, seg);
                for (int part = rw.p0; part < rw.p1 && ok; ++part) {
                    const int unit = super_part(sup.u, part, a.nq, a.pair != 0);
                    if (unit < 0) continue;
                    int r, qt, b, h, owner, kvr, pr;
                    decode(sup, unit, r, qt, b, h, owner, kvr, pr);
                    const int n = cost[pr];
                    if (n == 0) continue;
                    if (!mbar_wait(qd_full, it & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    for (int j = 0; j < n; ++j, ++t) {
                        const uint32_t st = t % kBStages, ph = (t / kBStages) & 1u;
                        if (!mbar_wait(kv_full + st, ph, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        umma_ss_kgroup<D / 16, 1024, 1024>(tmem, dQa, dKb + st * kStU, kIdS);
                        umma_ss_kgroup<D / 16, 1024, 1024>(tmem + 128, dOa, dVb + st * kStU, kIdS);
                        umma_commit(s_full);
                        if (j == n - 1) umma_commit(qd_empty);  // Q and dO are read by S / dP only
                        // dQ += dS K over the tile's first 64 keys, then the second 64
                        if (!mbar_wait(p_half, t & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        if (j == 0 && !mbar_wait(o_empty, (it & 1u) ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        umma_ts_k64_split(tmem + 256, tmem, dKm + st * kStU, kIdG, j == 0 ? 0u : 1u);
                        if (!mbar_wait(p_full, t & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        umma_ts_k64_split(tmem + 256, tmem + 64, dKm + st * kStU + kHalfU, kIdG, 1u);
                        umma_commit(kv_empty + st);  // K (S and dQ) and V (dP) of this stage are read
                    }
                    if (!ok) break;
                    umma_commit(o_full);
                    ++it;
                }
            }
            umma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait(drain, 0, &no_abort, 100000000ull);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // -------------------------------------------------------- compute (one query row per thread)
        const int quarter = warp & 3;
        const int grp = (warp - 4) >> 2;  // columns 32 grp .. 32 grp + 31 of each half
        const int row_in = quarter * 32 + lane;
        const uint32_t tA = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint64_t sl2x2 = f2_packf(a.scale_log2, a.scale_log2);
        uint32_t it = 0, t = 0;
        bool ok = true;
        int seg = 0;  // segment cursor of decode_super
        for (int rk = 0; rk < n_rounds && ok; ++rk) {
            const RoundWork rw = work_of_round(rk, n_items, a.pair != 0);
            if (rw.idx < 0) continue;
            const SuperItem sup = decode_super(rw.idx, a.B * a.N, order, seg_first, a.div_nsp, seg);
            for (int part = rw.p0; part < rw.p1 && ok; ++part) {
                const int unit = super_part(sup.u, part, a.nq, a.pair != 0);
                if (unit < 0) continue;
                int r, qt, b, h, owner, kvr, pr;
                decode(sup, unit, r, qt, b, h, owner, kvr, pr);
                const int row = qt * 128 + row_in;
                const bool row_valid = row < a.Sq;
                const int qpos = row_valid ? __ldg(a.q_pos + r * a.q_pos_stride + row) : INT_MIN;
                const long long qrow = static_cast<long long>(r * a.B + b);
                float *dq_row = a.dq + ((qrow * a.Sq + row) * a.N + h) * D + grp * (D / 2);
                if (cost[pr] == 0) {
                    if (row_valid && !a.accumulate) zero_row<D / 2>(dq_row);
                    continue;
                }
                // rows past Sq read the padding (-inf, 0): they see nothing
                const long long srow = (qrow * a.N + h) * a.sq_pad + row;
                const float nl2 = __ldg(a.nl2 + srow), ndv = __ldg(a.nd + srow);
                const uint64_t nl2x2 = f2_packf(nl2, nl2), ndx2 = f2_packf(ndv, ndv);
                const int2 *kt_o = ktab + owner * a.nk;
                const int2 qmm = qtab[r * a.nq + qt];
                const bool srt = sorted_flag[owner] != 0;
                const int32_t *kpos_o = a.k_pos + owner * a.k_pos_stride;
                for (int kt = next_k(0, kt_o, a.nk, qmm.y, srt); kt < a.nk;
                     kt = next_k(kt + 1, kt_o, a.nk, qmm.y, srt), ++t) {
                    if (!mbar_wait_warp(s_full, t & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    const int2 kmm = kt_o[kt];
                    const int k0 = kt * 128;
                    const bool need_mask = kmm.y > qmm.x || k0 + 128 > a.Sk;
                    const int gk = owner * a.nk + kt;
                    const bool arith = (arith_bits[gk >> 5] >> (gk & 31)) & 1u;
    #pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) {
                        // this warp's columns: cb .. cb+31 = keys k0 + cb ..
                        const int cb = 64 * hf + 32 * grp;
                        uint32_t s[32], dp[32];
                        tmem_ld32_nowait(tA + cb, s);
                        tmem_ld32_nowait(tA + 128 + cb, dp);
                        tmem_wait_ld32(s);
                        tmem_wait_ld32(dp);
                        if (need_mask) {
                            const int kh = k0 + cb;
                            const int nvalid = min(32, a.Sk - kh);
                            if (arith) {
                                // key positions kmin + cb + c: column c visible iff c <= qpos - kmin - cb
                                const long long dhi = static_cast<long long>(qpos) - kmm.x - cb;
                                const int lim = dhi < 0 ? -1 : static_cast<int>(min(dhi, static_cast<long long>(nvalid - 1)));
    #pragma unroll
                                for (int c = 0; c < 32; ++c)
                                    if (c > lim) s[c] = kNegInfBits;
                            } else {
    #pragma unroll
                                for (int c0 = 0; c0 < 32; c0 += 16) {
    #pragma unroll
                                    for (int c = c0; c < c0 + 16; ++c) {
                                        const int kp = (c < nvalid) ? __ldg(kpos_o + kh + c) : INT_MAX;
                                        if (kp > qpos) s[c] = kNegInfBits;
                                    }
                                    asm volatile("" ::: "memory");
                                }
                            }
                        }
                        // dS = 2^(s sl2 + nl2) (dP + nd)
                        uint32_t pk[16];
    #pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            float x0, x1, g0, g1;
                            f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, nl2x2), x0, x1);
                            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                            f2_unpack(f2_fma(f2_packf(p0, p1), f2_add(f2_pack(dp[c], dp[c + 1]), ndx2), 0ull), g0, g1);
                            pk[c >> 1] = pack_bf16x2(g0, g1);
                        }
                        // packed over the first 16 of this warp's own 32 columns (see dK / dV)
                        tmem_st16_nowait(tA + cb, pk);
                        release_half(hf == 0 ? p_half : p_full, lane);
                    }
                }
                if (!ok) break;
                if (!mbar_wait_warp(o_full, it & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                store_acc_row<D / 2>(tA + 256 + grp * (D / 2), dq_row, a.scale, row_valid, a.accumulate != 0);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_empty);
                ++it;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kBTmemCols);
    }
    if (tid == 0 && *abort_flag) atomicExch(&g_cp_bwd_status, static_cast<int>(CP_ERR_DEVICE_TIMEOUT));
}

// ======================================================================
// per-row statistics
// ======================================================================
__global__ void __launch_bounds__(256) bwd_stats_kernel(const float *__restrict__ o,
                                                        const __nv_bfloat16 *__restrict__ dout,
                                                        const float *__restrict__ lse, long long CB, int Sq, int N,
                                                        int D, long long sq_pad, float *__restrict__ nl2,
                                                        float *__restrict__ nd) {
    const long long total = CB * N * sq_pad;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long i = idx % sq_pad, rh = idx / sq_pad;
        const long long h = rh % N, rb = rh / N;
        float v_nl2 = -INFINITY, v_nd = 0.f;
        if (i < Sq) {
            const float l = lse[(rb * N + h) * Sq + i];
            const long long row = ((rb * Sq + i) * N + h) * D;
            const float4 *o4 = reinterpret_cast<const float4 *>(o + row);
            const uint4 *d8 = reinterpret_cast<const uint4 *>(dout + row);
            float acc = 0.f;
            for (int c = 0; c < D / 8; ++c) {
                const float4 a0 = __ldg(o4 + 2 * c), a1 = __ldg(o4 + 2 * c + 1);
                const uint4 w = __ldg(d8 + c);
                const __nv_bfloat162 *hb = reinterpret_cast<const __nv_bfloat162 *>(&w);
                const float2 f0 = __bfloat1622float2(hb[0]), f1 = __bfloat1622float2(hb[1]);
                const float2 f2 = __bfloat1622float2(hb[2]), f3 = __bfloat1622float2(hb[3]);
                acc = fmaf(a0.x, f0.x, acc);
                acc = fmaf(a0.y, f0.y, acc);
                acc = fmaf(a0.z, f1.x, acc);
                acc = fmaf(a0.w, f1.y, acc);
                acc = fmaf(a1.x, f2.x, acc);
                acc = fmaf(a1.y, f2.y, acc);
                acc = fmaf(a1.z, f3.x, acc);
                acc = fmaf(a1.w, f3.y, acc);
            }
            v_nl2 = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634074f;
            v_nd = -acc;
        }
        nl2[idx] = v_nl2;
        nd[idx] = v_nd;
    }
}

template <int D>
BwdArgs make_args(const BwdProblem &p, int nq, int nk, int heads_per_item) {
    BwdArgs a;
    a.q_pos = p.q_pos;
    a.k_pos = p.k_pos;
    a.q_pos_stride = p.q_pos_stride;
    a.k_pos_stride = p.k_pos_stride;
    a.nl2 = p.nl2;
    a.nd = p.nd;
    a.sq_pad = p.sq_pad;
    a.dq = p.dq;
    a.dk = p.dk;
    a.dv = p.dv;
    a.C = p.C;
    a.B = static_cast<int>(p.B);
    a.N = static_cast<int>(p.N);
    a.Nkv = static_cast<int>(p.Nkv);
    a.Sq = static_cast<int>(p.Sq);
    a.Sk = static_cast<int>(p.Sk);
    a.nq = nq;
    a.nk = nk;
    a.kv_shift = p.kv_shift;
    a.kpos_shift = p.kpos_shift;
    a.kpr = (p.k_pos_stride == 0) ? 1 : p.C;
    a.accumulate = p.accumulate ? 1 : 0;
    a.scale = p.scale;
    a.scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634074);
    a.timeout_ns = p.timeout_ns ? p.timeout_ns : 2000000000ull;
    a.hold = p.hold;
    a.div_h = make_fastdiv(static_cast<uint32_t>(heads_per_item));
    return a;
}

// The plans of the two backward kernels (see PlanSpec): 128-row tiles; the
// dK/dV kernel's units are key tiles, the dQ kernel's single query tiles.
PlanSpec bwd_plan_spec(const BwdProblem &p, bool dkdv, bool pair) {
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
    s.unit_is_k = dkdv ? 1 : 0;
    s.q_group = 1;
    s.pair = pair ? 1 : 0;
    return s;
}

bool bwd_plan_on_chip(int64_t C, int64_t kpr, int64_t Sq, int64_t Sk) {
    const int64_t q128 = (Sq + 127) / 128, k128 = (Sk + 127) / 128;
    return kpr * k128 + C * q128 <= kBwdMaxTables && C * k128 <= kBwdMaxPairs && C * q128 <= kBwdMaxPairs;
}

template <int D, bool kGP>
cp_status launch_dkdv_typed(const BwdProblem &p, cudaStream_t stream) {
    using K = CfgKV<D>;
    CUtensorMap mq, mdo, mk, mv, mnl, mnd;
    const int64_t CB = p.C * p.B;
    if (!make_map(&mq, p.q, D, p.N, p.Sq, CB, 128) || !make_map(&mdo, p.dout, D, p.N, p.Sq, CB, 128) ||
        !make_map(&mk, p.k, D, p.Nkv, p.Sk, CB, 128) || !make_map(&mv, p.v, D, p.Nkv, p.Sk, CB, 128) ||
        !make_map_f32_rows(&mnl, p.nl2, p.sq_pad, CB * p.N, 128) ||
        !make_map_f32_rows(&mnd, p.nd, p.sq_pad, CB * p.N, 128))
        return CP_ERR_CUDA;
    const int nq = static_cast<int>((p.Sq + 127) / 128), nk = static_cast<int>((p.Sk + 127) / 128);
    BwdArgs a = make_args<D>(p, nq, nk, static_cast<int>(p.Nkv));
    // key tiles u and nk-1-u in one work item when that still leaves 8 rounds
    a.pair = pair_units(nk, p.C, p.B * p.Nkv, sm_count()) ? 1 : 0;
    a.div_nsp = make_fastdiv(static_cast<uint32_t>(super_count(nk, a.pair != 0)));
    const long long n_items = static_cast<long long>(p.C) * super_count(nk, a.pair != 0) * p.B * p.Nkv;
    a.gp = PlanPtrs{};
    if (kGP) {
        const cp_status st = launch_plan(bwd_plan_spec(p, true, a.pair != 0), p.plan, &a.gp, stream);
        if (st != CP_OK) return st;
    }
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(bwd_dkdv_kernel<D, kGP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        K::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return cuda_status(attr_err);
    const int grid = static_cast<int>(n_items < sm_count() ? n_items : sm_count());
    bwd_dkdv_kernel<D, kGP><<<grid, kBThreads, K::kSmemBytes, stream>>>(mq, mdo, mk, mv, mnl, mnd, a);
    return last_launch_status();
}

template <int D, bool kGP>
cp_status launch_dq_typed(const BwdProblem &p, cudaStream_t stream) {
    using K = CfgQ<D>;
    CUtensorMap mq, mdo, mk, mv;
    const int64_t CB = p.C * p.B;
    if (!make_map(&mq, p.q, D, p.N, p.Sq, CB, 128) || !make_map(&mdo, p.dout, D, p.N, p.Sq, CB, 128) ||
        !make_map(&mk, p.k, D, p.Nkv, p.Sk, CB, 128) || !make_map(&mv, p.v, D, p.Nkv, p.Sk, CB, 128))
        return CP_ERR_CUDA;
    const int nq = static_cast<int>((p.Sq + 127) / 128), nk = static_cast<int>((p.Sk + 127) / 128);
    BwdArgs a = make_args<D>(p, nq, nk, static_cast<int>(p.N));
    // query tiles u and nq-1-u in one work item when that still leaves 8 rounds
    a.pair = pair_units(nq, p.C, p.B * p.N, sm_count()) ? 1 : 0;
    a.div_nsp = make_fastdiv(static_cast<uint32_t>(super_count(nq, a.pair != 0)));
    const long long n_items = static_cast<long long>(p.C) * super_count(nq, a.pair != 0) * p.B * p.N;
    a.gp = PlanPtrs{};
    if (kGP) {
        const cp_status st = launch_plan(bwd_plan_spec(p, false, a.pair != 0), p.plan, &a.gp, stream);
        if (st != CP_OK) return st;
    }
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(bwd_dq_kernel<D, kGP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        K::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return cuda_status(attr_err);
    const int grid = static_cast<int>(n_items < sm_count() ? n_items : sm_count());
    bwd_dq_kernel<D, kGP><<<grid, kBThreads, K::kSmemBytes, stream>>>(mq, mdo, mk, mv, a);
    return last_launch_status();
}

}  // namespace

cp_status launch_bwd_stats(const float *o, const void *dout, const float *lse, int64_t CB, int64_t Sq, int64_t N,
                           int64_t D, int64_t sq_pad, float *nl2, float *nd, cudaStream_t stream) {
    if (!o || !dout || !lse || !nl2 || !nd) return CP_ERR_NULL;
    if (CB < 1 || Sq < 1 || N < 1 || (D != 64 && D != 128) || sq_pad < Sq) return CP_ERR_SHAPE;
    if (!aligned16(o) || !aligned16(dout)) return CP_ERR_ALIGNMENT;
    const long long total = CB * N * sq_pad;
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    bwd_stats_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        o, static_cast<const __nv_bfloat16 *>(dout), lse, CB, static_cast<int>(Sq), static_cast<int>(N),
        static_cast<int>(D), sq_pad, nl2, nd);
    return last_launch_status();
}

size_t bwd_plan_need(int64_t C, int64_t kpr, int64_t Sq, int64_t Sk) {
    if (bwd_plan_on_chip(C, kpr, Sq, Sk)) return 0;
    BwdProblem p{};
    p.C = static_cast<int>(C);
    p.k_pos_stride = (kpr == 1) ? 0 : 1;
    p.Sq = Sq;
    p.Sk = Sk;
    // one buffer serves both launches in turn; unpaired units: the longer order
    const size_t a = plan_bytes(bwd_plan_spec(p, true, false)), b = plan_bytes(bwd_plan_spec(p, false, false));
    return a > b ? a : b;
}

cp_status validate_bwd(const BwdProblem &p, bool check_plan) {
    if (!p.q || !p.k || !p.v || !p.dout || !p.q_pos || !p.k_pos || !p.nl2 || !p.nd || !p.dq || !p.dk || !p.dv)
        return CP_ERR_NULL;
    if (p.C < 1 || p.C > kMaxC || p.B < 1 || p.N < 1 || p.Nkv < 1 || p.Sq < 1 || p.Sk < 1) return CP_ERR_SHAPE;
    if (p.D != 64 && p.D != 128) return CP_ERR_UNSUPPORTED;
    if (p.N % p.Nkv != 0) return CP_ERR_DIVISIBILITY;
    if (!(std::isfinite(p.scale) && p.scale > 0.f)) return CP_ERR_ARGUMENT;
    if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !aligned16(p.dout) || !aligned16(p.q_pos) ||
        !aligned16(p.k_pos) || !aligned16(p.nl2) || !aligned16(p.nd))
        return CP_ERR_ALIGNMENT;
    // accumulator rows are written with 32-byte stores
    if ((reinterpret_cast<uintptr_t>(p.dq) | reinterpret_cast<uintptr_t>(p.dk) | reinterpret_cast<uintptr_t>(p.dv)) &
        31u)
        return CP_ERR_ALIGNMENT;
    if (p.sq_pad < bwd_sq_pad(p.Sq) || p.sq_pad % 128 != 0) return CP_ERR_SHAPE;
    const int64_t kpr = (p.k_pos_stride == 0) ? 1 : p.C;
    const int64_t q128 = (p.Sq + 127) / 128, k128 = (p.Sk + 127) / 128;
    if (p.Sq > INT32_MAX / 2 || p.Sk > INT32_MAX / 2 || p.C * k128 * p.B * p.Nkv > INT32_MAX ||
        p.C * q128 * p.B * p.N > INT32_MAX || kpr * k128 + p.C * q128 > INT32_MAX / 8)
        return CP_ERR_SHAPE;
    if (check_plan && !bwd_plan_on_chip(p.C, kpr, p.Sq, p.Sk)) {
        if (!p.plan || p.plan_bytes < bwd_plan_need(p.C, kpr, p.Sq, p.Sk)) return CP_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(p.plan) & 255u) return CP_ERR_ALIGNMENT;
    }
    if (p.kv_shift < 0 || p.kv_shift >= p.C || p.kpos_shift < 0 || p.kpos_shift >= p.C) return CP_ERR_ARGUMENT;
    return CP_OK;
}

cp_status launch_bwd(const BwdProblem &p, cudaStream_t stream) {
    cp_status st = validate_bwd(p);
    if (st != CP_OK) return st;
    if (bwd_plan_on_chip(p.C, (p.k_pos_stride == 0) ? 1 : p.C, p.Sq, p.Sk)) {
        st = (p.D == 128) ? launch_dkdv_typed<128, false>(p, stream) : launch_dkdv_typed<64, false>(p, stream);
        if (st == CP_OK)
            st = (p.D == 128) ? launch_dq_typed<128, false>(p, stream) : launch_dq_typed<64, false>(p, stream);
        return st;
    }
    st = (p.D == 128) ? launch_dkdv_typed<128, true>(p, stream) : launch_dkdv_typed<64, true>(p, stream);
    if (st == CP_OK) st = (p.D == 128) ? launch_dq_typed<128, true>(p, stream) : launch_dq_typed<64, true>(p, stream);
    return st;
}

cp_status read_bwd_device_status(int *code, bool clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_cp_bwd_status, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
    *code = v;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_cp_bwd_status, &zero, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
    }
    return CP_OK;
}

}  // namespace cpattn

using namespace cpattn;

namespace {
inline size_t round256(size_t v) { return (v + 255) / 256 * 256; }
// workspace: the per-row statistics (nl2, nd), then the work plans when they
// do not fit on chip
size_t bwd_stats_bytes(int64_t CB, int64_t N, int64_t Sq) {
    return round256(2 * static_cast<size_t>(CB) * N * bwd_sq_pad(Sq) * sizeof(float));
}
}  // namespace

extern "C" cp_status cp_attn_bwd_workspace_size(int64_t B, int64_t Sq, int64_t Sk, int64_t N, size_t *bytes) {
    if (!bytes) return CP_ERR_NULL;
    if (B < 1 || Sq < 1 || Sk < 1 || N < 1) return CP_ERR_SHAPE;
    *bytes = bwd_stats_bytes(B, N, Sq) + bwd_plan_need(1, 1, Sq, Sk);
    return CP_OK;
}

extern "C" cp_status cp_attn_bwd_partial(const void *q, const void *k, const void *v, const float *o,
                                         const void *dout, const float *lse, const int32_t *q_pos,
                                         const int32_t *k_pos, int64_t B, int64_t Sq, int64_t Sk, int64_t N,
                                         int64_t Nkv, int64_t D, float scale, float *dq, float *dk, float *dv,
                                         int accumulate, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if (!o || !lse) return CP_ERR_NULL;
    if (B < 1 || Sq < 1 || Sk < 1 || N < 1) return CP_ERR_SHAPE;
    const int64_t pad = bwd_sq_pad(Sq);
    const size_t stats = bwd_stats_bytes(B, N, Sq), plan_need = bwd_plan_need(1, 1, Sq, Sk);
    if (!workspace || ws_bytes < stats + plan_need) return CP_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return CP_ERR_ALIGNMENT;
    BwdProblem p{};
    if (plan_need) {
        p.plan = static_cast<uint8_t *>(workspace) + stats;
        p.plan_bytes = plan_need;
    }
    p.q = q;
    p.k = k;
    p.v = v;
    p.dout = dout;
    p.q_pos = q_pos;
    p.k_pos = k_pos;
    p.q_pos_stride = 0;
    p.k_pos_stride = 0;
    p.nl2 = static_cast<float *>(workspace);
    p.nd = static_cast<float *>(workspace) + B * N * pad;
    p.sq_pad = pad;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.C = 1;
    p.B = B;
    p.N = N;
    p.Nkv = Nkv;
    p.D = D;
    p.Sq = Sq;
    p.Sk = Sk;
    p.accumulate = accumulate != 0;
    p.scale = scale;
    cp_status st = validate_bwd(p);
    if (st != CP_OK) return st;
    st = launch_bwd_stats(o, dout, lse, B, Sq, N, D, pad, const_cast<float *>(p.nl2), const_cast<float *>(p.nd),
                          stream);
    if (st == CP_OK) st = launch_bwd(p, stream);
    return st;
}

extern "C" cp_status cp_ring_bwd_workspace_size(int64_t B, int64_t S, int64_t N, int C, size_t *bytes) {
    if (!bytes) return CP_ERR_NULL;
    if (C < 1 || C > kMaxC || B < 1 || S < 1 || N < 1) return CP_ERR_SHAPE;
    if (S % C != 0) return CP_ERR_DIVISIBILITY;
    *bytes = bwd_stats_bytes(static_cast<int64_t>(C) * B, N, S / C) + bwd_plan_need(C, C, S / C, S / C);
    return CP_OK;
}

extern "C" cp_status cp_ring_attention_bwd(const void *q_sh, const void *k_sh, const void *v_sh, const float *o_sh,
                                           const float *lse_sh, const void *do_sh, const int32_t *pos, int64_t B,
                                           int64_t S, int64_t N, int64_t Nkv, int64_t D, int C, float scale,
                                           cp_layout layout, float *dq_sh, float *dk_sh, float *dv_sh,
                                           void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if (!o_sh || !lse_sh) return CP_ERR_NULL;
    if (layout != CP_ZIGZAG && layout != CP_CONTIGUOUS) return CP_ERR_ARGUMENT;
    if (C < 1 || C > kMaxC || B < 1 || S < 1 || N < 1 || Nkv < 1) return CP_ERR_SHAPE;
    if (layout == CP_ZIGZAG ? (S % (2LL * C) != 0) : (S % C != 0)) return CP_ERR_DIVISIBILITY;
    const int64_t s = S / C, pad = bwd_sq_pad(s);
    const size_t stats = bwd_stats_bytes(static_cast<int64_t>(C) * B, N, s), plan_need = bwd_plan_need(C, C, s, s);
    if (!workspace || ws_bytes < stats + plan_need) return CP_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return CP_ERR_ALIGNMENT;
    BwdProblem p{};
    if (plan_need) {
        p.plan = static_cast<uint8_t *>(workspace) + stats;
        p.plan_bytes = plan_need;
    }
    p.q = q_sh;
    p.k = k_sh;
    p.v = v_sh;
    p.dout = do_sh;
    p.q_pos = pos;
    p.k_pos = pos;
    p.q_pos_stride = s;
    p.k_pos_stride = s;
    p.nl2 = static_cast<float *>(workspace);
    p.nd = static_cast<float *>(workspace) + C * B * N * pad;
    p.sq_pad = pad;
    p.dq = dq_sh;
    p.dk = dk_sh;
    p.dv = dv_sh;
    p.C = C;
    p.B = B;
    p.N = N;
    p.Nkv = Nkv;
    p.D = D;
    p.Sq = s;
    p.Sk = s;
    p.scale = scale;
    cp_status st = validate_bwd(p);  // everything checked before anything is enqueued
    if (st != CP_OK) return st;
    st = launch_bwd_stats(o_sh, do_sh, lse_sh, C * B, s, N, D, pad, const_cast<float *>(p.nl2),
                          const_cast<float *>(p.nd), stream);
    // step `step`: rank r's queries against the K/V of owner (r - step) mod C;
    // dq of rank r and dk / dv of the owner accumulate from step 1 on (the
    // travelling dK / dV of the pages' ring are the owners' own accumulators here)
    for (int step = 0; step < C && st == CP_OK; ++step) {
        const int back = (C - step) % C;
        BwdProblem ps = p;
        ps.kv_shift = back;
        ps.kpos_shift = back;
        ps.accumulate = step > 0;
        st = launch_bwd(ps, stream);
    }
    return st;
}
