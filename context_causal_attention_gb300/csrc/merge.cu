// merge.cu -- log-sum-exp merge of a completed partial into an accumulator
// ("On Context Parallelism", Peer-to-peer / Forward, the tile merge:
// lse = logaddexp(lse_acc, lse_tile); o = e^{lse_acc - lse} o_acc +
// e^{lse_tile - lse} o_tile), plus the fp32 -> bf16 output conversion.
//
// Bandwidth kernel with 16-byte vectors.  Rows whose tile lse is -inf (a
// causal partial that saw nothing) cost one 4-byte read and are otherwise
// skipped; rows whose accumulator lse is -inf take the tile (weight 0 on the
// accumulator).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "cp_internal.h"

namespace cpattn {
namespace {

// One warp merges 32 consecutive query rows i0..i0+31 of one (b, h): the two
// lse vectors of those rows arrive in one coalesced load each, a ballot keeps
// the rows whose tile saw anything, and those rows are merged four per lane
// group at a time with all their o loads in flight before any is used.  Lane k
// computes the merged lse of row i0+k and its two weights; every lane then
// blends one or more 16-byte pieces of each row's D values.  A row of fewer
// than 32 float4 (D < 128) takes only part of the warp, so the warp is split
// into 32 / (D/4) lane groups that each take their own rows.
// kRpp: rows per slot of the warp (1 for D >= 128, 2 for D = 64; 0: 32 / (D/4),
// computed at run time, for the other widths)
template <int kRpp>
__global__ void __launch_bounds__(256, 4) lse_merge_kernel(float *__restrict__ o_acc, float *__restrict__ lse_acc,
                                                        const float *__restrict__ o_t,
                                                        const float *__restrict__ lse_t, long long B,
                                                        long long Sq, int N, int D) {
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long nib = (Sq + 31) >> 5;  // 32-row blocks per (b, h)
    const long long units = B * N * nib;
    const int nvec = D >> 2;                // float4 per row
    for (long long u = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units;
         u += warps) {
        const long long bh = u / nib;
        const long long i0 = (u - bh * nib) << 5;
        const long long b = bh / N;
        const int h = static_cast<int>(bh - b * N);
        const long long i = i0 + lane;
        const bool valid = i < Sq;
        const long long li = bh * Sq + i;  // lse index (b*N + h)*Sq + i
        const float lt = valid ? __ldg(lse_t + li) : -INFINITY;
        const float la = valid ? lse_acc[li] : -INFINITY;
        // merged lse and weights of this lane's row
        float lse = la, wa = 1.f, wt = 0.f;
        if (lt != -INFINITY) {
            if (la == -INFINITY) {
                lse = lt;
                wa = 0.f;
                wt = 1.f;
            } else {
                const float mx = fmaxf(la, lt), mn = fminf(la, lt);
                lse = mx + log1pf(expf(mn - mx));
                wa = expf(la - lse);
                wt = expf(lt - lse);
            }
        }
        unsigned todo = __ballot_sync(0xffffffffu, lt != -INFINITY);
        const long long row0 = (b * Sq + i0) * N + h;  // o row of i0; row of i0+k is row0 + k*N
        // rows narrower than a warp (D < 128) share it: rpp rows per slot, lane
        // group `sub` takes one of them, lane c0 of the group its float4 columns
        const int rpp = kRpp > 0 ? kRpp : (nvec >= 32 ? 1 : 32 / nvec);
        const int sub = rpp == 1 ? 0 : lane / nvec;
        const int c0 = rpp == 1 ? lane : lane - sub * nvec;
        while (todo) {
            // next (up to) 4 * rpp rows of this block with a non-empty tile; slot q
            // of this lane's group holds row ks[q]
            int ks[4];
            float wsa[4], wst[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                int mine = -1;
#pragma unroll
                for (int g = 0; g < (kRpp > 0 ? kRpp : 32); ++g) {
                    if (kRpp == 0 && g >= rpp) break;
                    const int kk = todo ? __ffs(todo) - 1 : -1;
                    todo &= todo - 1;  // no-op once empty
                    if (g == sub) mine = kk;
                }
                ks[q] = mine;
                // weights of that row, from its lane (all lanes take part)
                wsa[q] = __shfl_sync(0xffffffffu, wa, mine < 0 ? 0 : mine);
                wst[q] = __shfl_sync(0xffffffffu, wt, mine < 0 ? 0 : mine);
            }
            for (int c = c0; c < nvec; c += 32) {
                float4 xa[4], xt[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (ks[q] >= 0) {
                        const long long off = (row0 + static_cast<long long>(ks[q]) * N) * D;
                        xa[q] = reinterpret_cast<const float4 *>(o_acc + off)[c];
                        xt[q] = __ldg(reinterpret_cast<const float4 *>(o_t + off) + c);
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (ks[q] >= 0) {
                        const float a = wsa[q], t = wst[q];
                        const long long off = (row0 + static_cast<long long>(ks[q]) * N) * D;
                        reinterpret_cast<float4 *>(o_acc + off)[c] =
                            make_float4(a * xa[q].x + t * xt[q].x, a * xa[q].y + t * xt[q].y,
                                        a * xa[q].z + t * xt[q].z, a * xa[q].w + t * xt[q].w);
                    }
                }
            }
        }
        if (valid && lt != -INFINITY) lse_acc[li] = lse;
    }
}

__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float4 *__restrict__ in, uint4 *__restrict__ out,
                                                          long long n8) {
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 a = __ldg(in + 2 * i), b = __ldg(in + 2 * i + 1);
        __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
        uint4 r;
        r.x = *reinterpret_cast<uint32_t *>(&p0);
        r.y = *reinterpret_cast<uint32_t *>(&p1);
        r.z = *reinterpret_cast<uint32_t *>(&p2);
        r.w = *reinterpret_cast<uint32_t *>(&p3);
        out[i] = r;
    }
}


}  // namespace

cp_status launch_merge(float *o_acc, float *lse_acc, const float *o_tile, const float *lse_tile, int64_t B,
                       int64_t Sq, int64_t N, int64_t D, cudaStream_t stream) {
    if (!o_acc || !lse_acc || !o_tile || !lse_tile) return CP_ERR_NULL;
    if (B < 1 || Sq < 1 || N < 1 || D < 1 || N > INT32_MAX || D > 4096) return CP_ERR_SHAPE;
    if (D % 4 != 0 || !aligned16(o_acc) || !aligned16(o_tile)) return CP_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(lse_acc) & 3u) || (reinterpret_cast<uintptr_t>(lse_tile) & 3u))
        return CP_ERR_ALIGNMENT;
    const long long units = B * N * ((Sq + 31) / 32);
    long long blocks = (units + 7) / 8;  // 8 warps per block
    const long long cap = static_cast<long long>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (D >= 128)
        lse_merge_kernel<1><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_acc, lse_acc, o_tile, lse_tile, B,
                                                                              Sq, static_cast<int>(N),
                                                                              static_cast<int>(D));
    else if (D == 64)
        lse_merge_kernel<2><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_acc, lse_acc, o_tile, lse_tile, B,
                                                                              Sq, static_cast<int>(N),
                                                                              static_cast<int>(D));
    else
        lse_merge_kernel<0><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_acc, lse_acc, o_tile, lse_tile, B,
                                                                              Sq, static_cast<int>(N),
                                                                              static_cast<int>(D));
    return last_launch_status();
}

cp_status launch_f32_to_bf16(const float *in, void *out, int64_t n, cudaStream_t stream) {
    if (!in || !out) return CP_ERR_NULL;
    if (n % 8 != 0 || !aligned16(in) || !aligned16(out)) return CP_ERR_ALIGNMENT;
    const long long n8 = n / 8;
    if (n8 == 0) return CP_OK;
    long long blocks = (n8 + 255) / 256;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    f32_to_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(reinterpret_cast<const float4 *>(in),
                                                                         static_cast<uint4 *>(out), n8);
    return last_launch_status();
}

}  // namespace cpattn

extern "C" cp_status cp_lse_merge(float *o_acc, float *lse_acc, const float *o_tile, const float *lse_tile,
                                  int64_t B, int64_t Sq, int64_t N, int64_t D, cudaStream_t stream) {
    return cpattn::launch_merge(o_acc, lse_acc, o_tile, lse_tile, B, Sq, N, D, stream);
}
