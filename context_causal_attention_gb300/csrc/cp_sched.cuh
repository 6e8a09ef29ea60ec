// cp_sched.cuh -- work-item scheduling helpers shared by the persistent
// attention kernels (forward and backward): division by run-time invariant
// divisors, the longest-first order of super-blocks cut into segments, and the
// boustrophedon dealing of that item list.
#pragma once
#include <cstdint>

namespace cpattn {

// Division by a runtime-invariant divisor 1 <= d < 2^31 for numerators
// 0 <= n < 2^31 via a multiply-high: q = (n * m) >> (31 + l) with
// l = ceil(log2 d) and m = ceil(2^(31+l) / d) < 2^32 (round-up method; the
// error m*d - 2^(31+l) < d keeps the quotient exact for n < 2^31).
struct FastDiv {
    uint32_t d, m, sh;
};
inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    f.sh = 31 + l;
    f.m = static_cast<uint32_t>(((1ull << f.sh) + d - 1) / d);
    return f;
}
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return static_cast<uint32_t>((static_cast<uint64_t>(n) * f.m) >> f.sh);
}

// Work item of this CTA in round k of the persistent schedule: items are
// sorted longest first and dealt out boustrophedon (even rounds CTA 0..G-1,
// odd rounds G-1..0), so one CTA's long and short items pair up.  Returns -1
// past the end.
__device__ __forceinline__ int item_of_round(int k, int n_items) {
    const int G = gridDim.x;
    const long long idx = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - static_cast<int>(blockIdx.x))
                                                                     : static_cast<int>(blockIdx.x));
    return idx < n_items ? static_cast<int>(idx) : -1;
}

// ---------------------------------------------------------------- super-blocks
// A kernel's stationary units (query blocks, or key / query tiles) number nt
// per rank.  With pairing, super-block u of a rank holds units u and nt-1-u
// (u alone when they coincide), else unit u; nsp super-blocks per rank.  Under
// a causal mask the costs of units u and nt-1-u add up to about the same for
// every u (contiguous and zigzag layouts alike), so paired super-blocks cost
// about the same.
__host__ __device__ inline int super_count(int nt, bool pair) { return pair ? (nt + 1) / 2 : nt; }

// Host rule: pair when that still leaves at least 8 rounds of items over the
// SMs (items = C * super-blocks * per_block, per_block being the batch x head
// items of one super-block); with fewer rounds single units balance better.
inline bool pair_units(int nt, long long C, long long per_block, int sms) {
    return nt >= 2 && C * ((nt + 1) / 2) * per_block >= 8LL * sms;
}

// Unit of part k (0 or 1) of super-block u, -1 if it has no such part.
__device__ __forceinline__ int super_part(int u, int k, int nt, bool pair) {
    if (k == 0) return u;
    const int u2 = nt - 1 - u;
    return (pair && u2 != u) ? u2 : -1;
}

// Longest-first order of the C * nsp super-blocks (ties by index: rank, then
// block), cut into segments, each a run of one rank's super-blocks of equal
// cost: order[i] is the i-th super-block (rank * nsp + u); seg_first[s] is the
// position of the first super-block of segment s, seg_first[#segments] = C*nsp.
// cost[r * nt + unit] holds the units' costs.  seg_first doubles as scratch for
// the super-block costs; needs C*nsp + 1 entries.  Called by all threads of the
// block (kThreads of them); ends without a barrier (the caller syncs before
// using the result).
template <int kThreads>
__device__ __forceinline__ void build_segments(const int *cost, int C, int nt, bool pair, int *order, int *seg_first) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsp = super_count(nt, pair), nsup = C * nsp;
    int *sp_cost = seg_first;
    for (int x = tid; x < nsup; x += kThreads) {
        const int r = x / nsp, u = x - r * nsp, u2 = super_part(u, 1, nt, pair);
        sp_cost[x] = cost[r * nt + u] + (u2 >= 0 ? cost[r * nt + u2] : 0);
    }
    __syncthreads();
    // rank by cost (descending), ties by index: the super-blocks of one rank and
    // cost are then contiguous, and the first of them opens a segment
    constexpr int kHead = 1 << 30;
    for (int x = tid; x < nsup; x += kThreads) {
        const int c = sp_cost[x];
        const int r0 = (x / nsp) * nsp;
        int rank = 0;
        bool head = true;
        for (int y = 0; y < nsup; ++y) {
            const int cy = sp_cost[y];
            rank += (cy > c) || (cy == c && y < x);
            head &= !(cy == c && y >= r0 && y < x);
        }
        order[rank] = x | (head ? kHead : 0);
    }
    __syncthreads();
    if (warp == 0) {
        int nseg = 0;
        for (int c0 = 0; c0 < nsup; c0 += 32) {
            const int i = c0 + lane;
            bool head = false;
            if (i < nsup) {
                const int v = order[i];
                head = (v & kHead) != 0;
                order[i] = v & ~kHead;
            }
            const unsigned msk = __ballot_sync(0xffffffffu, head);
            if (head) seg_first[nseg + __popc(msk & ((1u << lane) - 1u))] = i;
            nseg += __popc(msk);
        }
        if (lane == 0) seg_first[nseg] = nsup;
    }
}

// A work item: super-block u of rank r, and its batch x head index bh.
struct SuperItem {
    int r, u, bh;
};

// Work-item index -> super item.  Items are laid out segment by segment;
// inside a segment they go head-major (every super-block of the segment for
// bh = 0, then bh = 1, ...), so CTAs running at the same time share heads.
// BH: batch x head items per super-block; div_nsp divides by nsp; `seg` is the
// caller's cursor (the items of one CTA come in increasing index order).
__device__ __forceinline__ SuperItem decode_super(int idx, int BH, const int *order, const int *seg_first,
                                                  const FastDiv &div_nsp, int &seg) {
    while (seg_first[seg + 1] * BH <= idx) ++seg;
    const int f = seg_first[seg];
    const int m = seg_first[seg + 1] - f;
    const int local = idx - f * BH;
    const int bh = local / m;
    const uint32_t sp = static_cast<uint32_t>(order[f + (local - bh * m)]);
    SuperItem x;
    x.r = static_cast<int>(fdiv(sp, div_nsp));
    x.u = static_cast<int>(sp - static_cast<uint32_t>(x.r) * div_nsp.d);
    x.bh = bh;
    return x;
}

}  // namespace cpattn
