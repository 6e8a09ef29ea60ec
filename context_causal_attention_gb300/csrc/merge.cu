// merge.cu -- log-sum-exp merge of a completed partial into an accumulator
// ("On Context Parallelism", Peer-to-peer / Forward, the tile merge:
// lse = logaddexp(lse_acc, lse_tile); o = e^{lse_acc - lse} o_acc +
// e^{lse_tile - lse} o_tile), plus the fp32 -> bf16 output conversion.
//
// Bandwidth kernel: D/4 threads own one row (b, i, h) of D fp32 values and
// move it with 16-byte vectors; both lse values of the row are read once per
// warp (broadcast).  Rows whose tile lse is -inf (a causal partial that saw
// nothing) cost one 4-byte read and are otherwise skipped; rows whose
// accumulator lse is -inf take the tile without reading the accumulator.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "cp_internal.h"

namespace cpattn {
namespace {

__global__ void __launch_bounds__(256) lse_merge_kernel(float *__restrict__ o_acc, float *__restrict__ lse_acc,
                                                        const float *__restrict__ o_t,
                                                        const float *__restrict__ lse_t, long long rows,
                                                        long long Sq, int N, int tpr_shift, int D) {
    const int tpr = 1 << tpr_shift;  // threads per row = D / 4
    const long long gthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int sub = static_cast<int>(gid & (tpr - 1));
    for (long long row = gid >> tpr_shift; row < rows; row += gthreads >> tpr_shift) {
        // row = (b * Sq + i) * N + h
        const long long bi = row / N;
        const int h = static_cast<int>(row - bi * N);
        const long long b = bi / Sq, i = bi - b * Sq;
        const long long li = (b * N + h) * Sq + i;
        const float lt = __ldg(lse_t + li);
        if (lt == -INFINITY) continue;
        const float la = lse_acc[li];
        float4 *oa = reinterpret_cast<float4 *>(o_acc + row * D);
        const float4 *ot = reinterpret_cast<const float4 *>(o_t + row * D);
        if (la == -INFINITY) {
            for (int c = sub; c < D / 4; c += tpr) oa[c] = __ldg(ot + c);
            if (sub == 0) lse_acc[li] = lt;
            continue;
        }
        const float mx = fmaxf(la, lt), mn = fminf(la, lt);
        const float lse = mx + log1pf(expf(mn - mx));
        const float wa = expf(la - lse), wt = expf(lt - lse);
        for (int c = sub; c < D / 4; c += tpr) {
            const float4 x = oa[c];
            const float4 y = __ldg(ot + c);
            oa[c] = make_float4(wa * x.x + wt * y.x, wa * x.y + wt * y.y, wa * x.z + wt * y.z, wa * x.w + wt * y.w);
        }
        if (sub == 0) lse_acc[li] = lse;
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

int ilog2_pow2(long long v) {
    if (v <= 0 || (v & (v - 1))) return -1;
    int s = 0;
    while ((1LL << s) < v) ++s;
    return s;
}

}  // namespace

cp_status launch_merge(float *o_acc, float *lse_acc, const float *o_tile, const float *lse_tile, int64_t B,
                       int64_t Sq, int64_t N, int64_t D, cudaStream_t stream) {
    if (!o_acc || !lse_acc || !o_tile || !lse_tile) return CP_ERR_NULL;
    if (B < 1 || Sq < 1 || N < 1 || D < 1 || N > INT32_MAX || D > 4096) return CP_ERR_SHAPE;
    if (D % 4 != 0 || !aligned16(o_acc) || !aligned16(o_tile)) return CP_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(lse_acc) & 3u) || (reinterpret_cast<uintptr_t>(lse_tile) & 3u))
        return CP_ERR_ALIGNMENT;
    long long tpr = D / 4;
    if (tpr > 32) tpr = 32;
    int shift = ilog2_pow2(tpr);
    while (shift < 0) {  // largest power of two <= D/4
        --tpr;
        shift = ilog2_pow2(tpr);
    }
    const long long rows = B * Sq * N;
    long long blocks = (rows * tpr + 255) / 256;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    lse_merge_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_acc, lse_acc, o_tile, lse_tile, rows, Sq,
                                                                       static_cast<int>(N), shift,
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
