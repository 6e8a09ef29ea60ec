// cp_rounds.cuh -- the last round of a persistent schedule dealt in halves.
//
// The backward and tf32 kernels deal paired super items (cp_sched.cuh:
// super-block u of a rank holds units u and nt-1-u) one per CTA and round.
// When the super items left for the last round are at most half the grid, that
// round deals their single parts instead: twice as many pieces, each about half
// as long, so fewer CTAs sit idle at the end of the launch.  (The bf16 forward
// keeps whole items: on its zigzag ring steps the two units of a pair often
// differ in cost by the whole item, and the change cost it more in code than
// the shorter round gave back.)
#pragma once

#include "cp_sched.cuh"

namespace cpattn {

// Work of this CTA in round k: super item `idx` (-1: none) and its parts
// [p0, p1).  `pair`: the items are paired super items.
struct RoundWork {
    int idx, p0, p1;
};
__device__ __forceinline__ RoundWork work_of_round(int k, int n_items, bool pair) {
    const int G = gridDim.x;
    const int full = n_items / G, rem = n_items - full * G;
    RoundWork w{-1, 0, 2};
    if (pair && rem > 0 && 2 * rem <= G && k == full) {
        // the same boustrophedon slot order as item_of_round
        const int slot = (k & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
        if (slot < 2 * rem) {
            w.idx = full * G + (slot >> 1);
            w.p0 = slot & 1;
            w.p1 = w.p0 + 1;
        }
        return w;
    }
    w.idx = item_of_round(k, n_items);
    return w;
}

}  // namespace cpattn
