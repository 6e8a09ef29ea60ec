// plan.cu -- the work plan of a persistent attention launch, written into the
// caller's workspace by a two-kernel pre-pass when it does not fit in shared
// memory (long sequences, many virtual ranks).
//
// The plan holds exactly what the kernels otherwise build in every CTA (see
// the PlanPtrs comment in cp_internal.h): position tables and consecutive-
// position bits of every query and key tile, the sorted flags, the per-unit
// costs and the longest-first order of super-blocks cut into segments.
//   plan_tables_kernel  one warp per 32 consecutive tiles (one bit word), so
//                       the bits need no atomics and no clearing;
//   plan_order_kernel   one CTA: sorted flags, costs, then build_segments.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "cp_internal.h"
#include "cp_sched.cuh"

namespace cpattn {
namespace {

constexpr size_t kAlign = 256;
inline size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

constexpr int kOrderThreads = 1024;
constexpr int kTableThreads = 256;

struct Dims {
    int nqt, nkt, nunits, nsp;
};

Dims dims_of(const PlanSpec &s) {
    Dims d;
    d.nqt = (s.Sq + s.q_tile - 1) / s.q_tile;
    d.nkt = (s.Sk + s.k_tile - 1) / s.k_tile;
    d.nunits = s.unit_is_k ? d.nkt : (d.nqt + s.q_group - 1) / s.q_group;
    d.nsp = super_count(d.nunits, s.pair != 0);
    return d;
}

struct Offsets {
    size_t ktab, qtab, kbits, qbits, ksorted, qsorted, cost, order, seg, total;
};

Offsets offsets_of(const PlanSpec &s, const Dims &d) {
    Offsets o;
    const size_t nk = static_cast<size_t>(s.kpr) * d.nkt, nq = static_cast<size_t>(s.C) * d.nqt;
    const size_t nsup = static_cast<size_t>(s.C) * d.nsp;
    size_t off = 0;
    o.ktab = off;
    off += round_up(nk * 8);
    o.qtab = off;
    off += round_up(nq * 8);
    o.kbits = off;
    off += round_up((nk + 31) / 32 * 4);
    o.qbits = off;
    off += round_up((nq + 31) / 32 * 4);
    o.ksorted = off;
    off += round_up(static_cast<size_t>(s.kpr) * 4);
    o.qsorted = off;
    off += round_up(static_cast<size_t>(s.C) * 4);
    o.cost = off;
    off += round_up(static_cast<size_t>(s.C) * d.nunits * 4);
    o.order = off;
    off += round_up(nsup * 4);
    o.seg = off;
    off += round_up((nsup + 1) * 4);
    o.total = off;
    return o;
}

struct PlanDev {
    PlanSpec s;
    int nqt, nkt, nunits;
    int2 *ktab, *qtab;
    uint32_t *kbits, *qbits;
    int *ksorted, *qsorted, *cost, *order, *seg;
};

// (min, max) of every tile's positions and the word of consecutive-position
// bits of each 32 consecutive tiles; K tiles (kpr ranks) first, then Q tiles
// (C ranks), each in its own word range.
__global__ void __launch_bounds__(kTableThreads) plan_tables_kernel(const PlanDev d) {
    const int lane = threadIdx.x & 31;
    const PlanSpec &s = d.s;
    const int nk = s.kpr * d.nkt, nq = s.C * d.nqt;
    const int nkw = (nk + 31) / 32, nqw = (nq + 31) / 32;
    const int nw = static_cast<int>((gridDim.x * blockDim.x) >> 5);
    for (int w = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5); w < nkw + nqw; w += nw) {
        const bool isk = w < nkw;
        const int ww = isk ? w : w - nkw;
        const int n = isk ? nk : nq;
        const int per = isk ? d.nkt : d.nqt;
        const int tile = isk ? s.k_tile : s.q_tile;
        const int lim = isk ? s.Sk : s.Sq;
        const int32_t *base = isk ? s.k_pos : s.q_pos;
        const long long stride = isk ? s.k_pos_stride : s.q_pos_stride;
        int2 *tab = isk ? d.ktab : d.qtab;
        uint32_t word = 0u;
        for (int i = 0; i < 32; ++i) {
            const int g = ww * 32 + i;
            if (g >= n) break;  // warp-uniform
            const int r = g / per, t = g - r * per;
            const int32_t *p = base + r * stride;
            const int row0 = t * tile;
            const long long first = __ldg(p + row0);
            int mn = INT_MAX, mx = INT_MIN;
            bool ok = true;
            for (int m = 0; m < tile; m += 32) {
                const int row = row0 + m + lane;
                if (row < lim) {
                    const int v = __ldg(p + row);
                    mn = min(mn, v);
                    mx = max(mx, v);
                    ok &= (static_cast<long long>(v) == first + m + lane);
                }
            }
            mn = __reduce_min_sync(0xffffffffu, mn);
            mx = __reduce_max_sync(0xffffffffu, mx);
            ok = __all_sync(0xffffffffu, ok);
            if (lane == 0) tab[g] = make_int2(mn, mx);
            if (ok) word |= 1u << i;
        }
        if (lane == 0) (isk ? d.kbits : d.qbits)[ww] = word;
    }
}

// Sorted flags, per-(rank, unit) costs, then the segment order (one CTA).
__global__ void __launch_bounds__(kOrderThreads, 1) plan_order_kernel(const PlanDev d) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const PlanSpec &s = d.s;
    for (int j = warp; j < s.kpr + s.C; j += kOrderThreads / 32) {
        const bool isk = j < s.kpr;
        const int r = isk ? j : j - s.kpr;
        const int n = isk ? d.nkt : d.nqt;
        const int2 *t = isk ? d.ktab + static_cast<long long>(r) * d.nkt : d.qtab + static_cast<long long>(r) * d.nqt;
        bool ok = true;
        for (int i = 1 + lane; i < n; i += 32) ok &= isk ? (t[i].x >= t[i - 1].x) : (t[i].y >= t[i - 1].y);
        ok = __all_sync(0xffffffffu, ok);
        if (lane == 0) (isk ? d.ksorted : d.qsorted)[r] = ok ? 1 : 0;
    }
    __syncthreads();
    const int np = s.C * d.nunits;
    for (int p = tid; p < np; p += kOrderThreads) {
        const int r = p / d.nunits, u = p - r * d.nunits;
        const int owner = (s.kpr == 1) ? 0 : (r + s.kpos_shift) % s.C;
        int c = 0;
        if (!s.unit_is_k) {
            // key tiles of the owner whose smallest position is <= the unit's largest query position
            int qmax = INT_MIN;
            for (int g = 0; g < s.q_group; ++g) {
                const int qt = u * s.q_group + g;
                if (qt < d.nqt) qmax = max(qmax, d.qtab[static_cast<long long>(r) * d.nqt + qt].y);
            }
            const int2 *ko = d.ktab + static_cast<long long>(owner) * d.nkt;
            if (d.ksorted[owner]) {
                int lo = 0, hi = d.nkt;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (ko[mid].x <= qmax) lo = mid + 1; else hi = mid;
                }
                c = lo;
            } else {
                for (int kt = 0; kt < d.nkt; ++kt) c += (ko[kt].x <= qmax);
            }
        } else {
            // query tiles of the rank whose largest position is >= the key tile's smallest position
            const int kmin = d.ktab[static_cast<long long>(owner) * d.nkt + u].x;
            const int2 *qr = d.qtab + static_cast<long long>(r) * d.nqt;
            if (d.qsorted[r]) {
                int lo = 0, hi = d.nqt;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (qr[mid].y >= kmin) hi = mid; else lo = mid + 1;
                }
                c = d.nqt - lo;
            } else {
                for (int qt = 0; qt < d.nqt; ++qt) c += (qr[qt].y >= kmin);
            }
        }
        d.cost[p] = c;
    }
    __syncthreads();
    build_segments<kOrderThreads>(d.cost, s.C, d.nunits, s.pair != 0, d.order, d.seg);
}

}  // namespace

size_t plan_bytes(const PlanSpec &s) { return offsets_of(s, dims_of(s)).total; }

cp_status launch_plan(const PlanSpec &s, void *buf, PlanPtrs *out, cudaStream_t stream) {
    if (!buf || !out || !s.q_pos || !s.k_pos) return CP_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(buf) & (kAlign - 1)) return CP_ERR_ALIGNMENT;
    const Dims dm = dims_of(s);
    const Offsets o = offsets_of(s, dm);
    uint8_t *b = static_cast<uint8_t *>(buf);
    PlanDev d;
    d.s = s;
    d.nqt = dm.nqt;
    d.nkt = dm.nkt;
    d.nunits = dm.nunits;
    d.ktab = reinterpret_cast<int2 *>(b + o.ktab);
    d.qtab = reinterpret_cast<int2 *>(b + o.qtab);
    d.kbits = reinterpret_cast<uint32_t *>(b + o.kbits);
    d.qbits = reinterpret_cast<uint32_t *>(b + o.qbits);
    d.ksorted = reinterpret_cast<int *>(b + o.ksorted);
    d.qsorted = reinterpret_cast<int *>(b + o.qsorted);
    d.cost = reinterpret_cast<int *>(b + o.cost);
    d.order = reinterpret_cast<int *>(b + o.order);
    d.seg = reinterpret_cast<int *>(b + o.seg);
    const long long words = (static_cast<long long>(s.kpr) * dm.nkt + 31) / 32 +
                            (static_cast<long long>(s.C) * dm.nqt + 31) / 32;
    const long long warps_per_block = kTableThreads / 32;
    long long blocks = (words + warps_per_block - 1) / warps_per_block;
    if (blocks > 4LL * sm_count()) blocks = 4LL * sm_count();
    if (blocks < 1) blocks = 1;
    plan_tables_kernel<<<static_cast<int>(blocks), kTableThreads, 0, stream>>>(d);
    cp_status st = last_launch_status();
    if (st != CP_OK) return st;
    plan_order_kernel<<<1, kOrderThreads, 0, stream>>>(d);
    st = last_launch_status();
    if (st != CP_OK) return st;
    out->ktab = d.ktab;
    out->qtab = d.qtab;
    out->kbits = d.kbits;
    out->qbits = d.qbits;
    out->ksorted = d.ksorted;
    out->qsorted = d.qsorted;
    out->cost = d.cost;
    out->order = d.order;
    out->seg_first = d.seg;
    return CP_OK;
}

}  // namespace cpattn
