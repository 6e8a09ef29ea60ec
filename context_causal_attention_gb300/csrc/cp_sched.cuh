// cp_sched.cuh -- work-item scheduling helpers shared by the persistent
// attention kernels (forward and backward): division by run-time invariant
// divisors and the boustrophedon dealing of a longest-first item list.
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

}  // namespace cpattn
