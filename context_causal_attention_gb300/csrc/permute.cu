// permute.cu -- zigzag / contiguous sharding, its inverse, the position map
// and the Ulysses relayout, as bit-exact permutation kernels.
//
// Every one of these permutations moves whole contiguous runs of bytes: a
// zigzag chunk ("On Context Parallelism", All-gather: rank r owns chunks r and
// 2C-1-r) is t rows of N*D elements that stay contiguous on both sides, and a
// Ulysses head group ("Context parallelism: Ring Attention and Ulysses",
// Ulysses: seq_to_head / head_to_seq) is N/C*D contiguous elements per row.
// So each call is a batch of "segments": `rows` rows of `row_bytes` bytes with
// a source and a destination stride.  blockIdx.y picks the segment, the
// x-blocks stream it with 16-byte vector loads and stores (four in flight per
// thread), and the grid is sized to a few waves of the SM count.
#include <cuda_runtime.h>

#include <cstdint>

#include "cp_internal.h"

namespace cpattn {
namespace {

enum SegKind : int { kZigzagShard = 0, kContigShard = 1, kUlyssesS2H = 2, kUlyssesH2S = 3 };

struct SegArgs {
    const uint8_t *src;
    uint8_t *dst;
    int kind;
    int unshard;       // shard kinds: 1 = inverse direction (swap src/dst roles)
    int global_order;  // Ulysses: 1 = sequence rows in global (unzigzagged) order
    long long B, S, N, C;
    long long row_bytes;   // bytes of one row of the segment
    long long seg_rows;    // rows per segment
    long long vec_per_row; // row_bytes / 16
    int vpr_shift;         // log2(vec_per_row) or -1
    long long seg_per_group;  // Ulysses: segments of one independent group (0 = one group)
    long long group_bytes;    // Ulysses: byte distance between groups, same on both sides
};

struct Seg {
    long long src_off, dst_off, src_stride, dst_stride;
};

__device__ __forceinline__ Seg segment(const SegArgs &a, long long y) {
    Seg s;
    long long grp = 0;
    if (a.seg_per_group) {
        grp = y / a.seg_per_group;
        y -= grp * a.seg_per_group;
    }
    if (a.kind == kZigzagShard || a.kind == kContigShard) {
        // y -> (r, b, half); one segment is a contiguous run of seg_rows rows of N*D
        const long long halves = (a.kind == kZigzagShard) ? 2 : 1;
        const long long half = y % halves;
        const long long rb = y / halves;
        const long long b = rb % a.B, r = rb / a.B;
        const long long s_loc = a.S / a.C;
        long long g0;  // first global row
        if (a.kind == kZigzagShard) {
            const long long t = a.S / (2 * a.C);
            const long long chunk = half ? (2 * a.C - 1 - r) : r;
            g0 = chunk * t;
        } else {
            g0 = r * s_loc;
        }
        const long long full_off = (b * a.S + g0) * a.row_bytes;
        const long long shard_off = ((r * a.B + b) * s_loc + half * a.seg_rows) * a.row_bytes;
        s.src_off = a.unshard ? shard_off : full_off;
        s.dst_off = a.unshard ? full_off : shard_off;
        s.src_stride = s.dst_stride = a.row_bytes;
    } else {
        // y -> (r: head group, b, j: sequence shard, half)
        const long long halves = a.global_order ? 2 : 1;
        const long long half = y % halves;
        long long rest = y / halves;
        const long long j = rest % a.C;
        rest /= a.C;
        const long long b = rest % a.B, r = rest / a.B;
        const long long s_loc = a.S / a.C, nh = a.N / a.C;
        const long long u0 = half * a.seg_rows;  // first local row of shard j
        long long row0;                          // first row in the gathered sequence
        if (a.global_order) {
            const long long t = a.S / (2 * a.C);
            row0 = (half ? (2 * a.C - 1 - j) : j) * t;
        } else {
            row0 = j * s_loc;
        }
        const long long hb = a.row_bytes;  // nh * D * esize
        const long long seq_off = (((j * a.B + b) * s_loc + u0) * a.N + r * nh) * (hb / nh);
        const long long head_off = ((r * a.B + b) * a.S + row0) * hb;
        const long long seq_stride = a.N * (hb / nh), head_stride = hb;
        if (a.kind == kUlyssesS2H) {
            s.src_off = seq_off;
            s.dst_off = head_off;
            s.src_stride = seq_stride;
            s.dst_stride = head_stride;
        } else {
            s.src_off = head_off;
            s.dst_off = seq_off;
            s.src_stride = head_stride;
            s.dst_stride = seq_stride;
        }
        s.src_off += grp * a.group_bytes;
        s.dst_off += grp * a.group_bytes;
    }
    return s;
}

__global__ void __launch_bounds__(256) segment_copy_kernel(const SegArgs a) {
    const Seg sg = segment(a, blockIdx.y);
    const uint8_t *src = a.src + sg.src_off;
    uint8_t *dst = a.dst + sg.dst_off;
    const long long total = a.seg_rows * a.vec_per_row;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    long long v = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    auto addr = [&](long long vi, long long ss) -> long long {
        long long row, col;
        if (a.vpr_shift >= 0) {
            row = vi >> a.vpr_shift;
            col = vi & (a.vec_per_row - 1);
        } else {
            row = vi / a.vec_per_row;
            col = vi - row * a.vec_per_row;
        }
        return row * ss + col * 16;
    };
    for (; v + 3 * stride < total; v += 4 * stride) {
        uint4 x0 = __ldg(reinterpret_cast<const uint4 *>(src + addr(v, sg.src_stride)));
        uint4 x1 = __ldg(reinterpret_cast<const uint4 *>(src + addr(v + stride, sg.src_stride)));
        uint4 x2 = __ldg(reinterpret_cast<const uint4 *>(src + addr(v + 2 * stride, sg.src_stride)));
        uint4 x3 = __ldg(reinterpret_cast<const uint4 *>(src + addr(v + 3 * stride, sg.src_stride)));
        *reinterpret_cast<uint4 *>(dst + addr(v, sg.dst_stride)) = x0;
        *reinterpret_cast<uint4 *>(dst + addr(v + stride, sg.dst_stride)) = x1;
        *reinterpret_cast<uint4 *>(dst + addr(v + 2 * stride, sg.dst_stride)) = x2;
        *reinterpret_cast<uint4 *>(dst + addr(v + 3 * stride, sg.dst_stride)) = x3;
    }
    for (; v < total; v += stride)
        *reinterpret_cast<uint4 *>(dst + addr(v, sg.dst_stride)) =
            __ldg(reinterpret_cast<const uint4 *>(src + addr(v, sg.src_stride)));
}

__global__ void positions_kernel(int32_t *pos, long long S, int C, int layout) {
    const long long s = S / C;
    const long long n = S;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = i / s, u = i - r * s;
        long long g;
        if (layout == CP_CONTIGUOUS) {
            g = r * s + u;
        } else {
            const long long t = s / 2;
            g = (u < t) ? (r * t + u) : ((2LL * C - 1 - r) * t + (u - t));
        }
        pos[i] = static_cast<int32_t>(g);
    }
}

int log2_exact(long long v) {
    if (v <= 0 || (v & (v - 1))) return -1;
    int s = 0;
    while ((1LL << s) < v) ++s;
    return s;
}

cp_status launch_segments(SegArgs a, long long nseg, cudaStream_t stream) {
    if (nseg <= 0 || a.seg_rows <= 0) return CP_OK;
    if (nseg > 65535) return CP_ERR_SHAPE;
    a.vec_per_row = a.row_bytes / 16;
    a.vpr_shift = log2_exact(a.vec_per_row);
    const long long vecs = a.seg_rows * a.vec_per_row;
    const long long target_blocks = static_cast<long long>(sm_count()) * 8;  // 8 x 256 threads per SM
    long long bx = (vecs + 256 * 4 - 1) / (256 * 4);
    long long cap = target_blocks / nseg;
    if (cap < 1) cap = 1;
    if (bx > cap) bx = cap;
    if (bx < 1) bx = 1;
    segment_copy_kernel<<<dim3(static_cast<unsigned>(bx), static_cast<unsigned>(nseg)), 256, 0, stream>>>(a);
    return last_launch_status();
}

// The kernels may dereference [p, p + n): memory of the current device (or
// managed memory), or host memory that is pinned and mapped into the device
// address space at the same address.  Both ends of the range are checked.
bool device_reachable(const void *p, size_t n) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const char *ends[2] = {static_cast<const char *>(p), static_cast<const char *>(p) + (n ? n - 1 : 0)};
    for (const char *e : ends) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, e) != cudaSuccess) {
            cudaGetLastError();  // clear the sticky error of the query
            return false;
        }
        if (at.type == cudaMemoryTypeManaged || (at.type == cudaMemoryTypeDevice && at.device == dev)) continue;
        if (at.type == cudaMemoryTypeHost && at.devicePointer == e) continue;
        return false;
    }
    return true;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

cp_status shard_impl(const void *x, void *x_sh, int64_t B, int64_t S, int64_t N, int64_t D, int C, cp_dtype dtype,
                     cp_layout layout, int unshard, cudaStream_t stream) {
    if (!x || !x_sh) return CP_ERR_NULL;
    if (dtype != CP_BF16 && dtype != CP_F32) return CP_ERR_DTYPE;
    if (layout != CP_ZIGZAG && layout != CP_CONTIGUOUS) return CP_ERR_ARGUMENT;
    if (B < 1 || S < 1 || N < 1 || D < 1 || C < 1) return CP_ERR_SHAPE;
    if (layout == CP_ZIGZAG ? (S % (2LL * C) != 0) : (S % C != 0)) return CP_ERR_DIVISIBILITY;
    const long long row_bytes = N * D * static_cast<long long>(dtype_size(dtype));
    if (!aligned16(x) || !aligned16(x_sh) || row_bytes % 16 != 0) return CP_ERR_ALIGNMENT;
    const size_t nbytes = static_cast<size_t>(B * S) * static_cast<size_t>(row_bytes);
    if (ranges_overlap(x, nbytes, x_sh, nbytes)) return CP_ERR_ARGUMENT;
    if (!device_reachable(x, nbytes) || !device_reachable(x_sh, nbytes)) return CP_ERR_ARGUMENT;
    SegArgs a{};
    a.src = static_cast<const uint8_t *>(unshard ? x_sh : x);
    a.dst = static_cast<uint8_t *>(unshard ? const_cast<void *>(x) : x_sh);
    a.kind = layout == CP_ZIGZAG ? kZigzagShard : kContigShard;
    a.unshard = unshard;
    a.B = B;
    a.S = S;
    a.N = N;
    a.C = C;
    // a segment is one contiguous run: treat it as a single row of seg bytes
    const long long rows = layout == CP_ZIGZAG ? S / (2LL * C) : S / C;
    a.row_bytes = row_bytes;
    a.seg_rows = rows;
    const long long nseg = static_cast<long long>(C) * B * (layout == CP_ZIGZAG ? 2 : 1);
    return launch_segments(a, nseg, stream);
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" cp_status cp_zigzag_shard(const void *x, void *x_sh, int64_t B, int64_t S, int64_t N, int64_t D, int C,
                                     cp_dtype dtype, cp_layout layout, cudaStream_t stream) {
    return shard_impl(x, x_sh, B, S, N, D, C, dtype, layout, 0, stream);
}

extern "C" cp_status cp_zigzag_unshard(const void *x_sh, void *x, int64_t B, int64_t S, int64_t N, int64_t D, int C,
                                       cp_dtype dtype, cp_layout layout, cudaStream_t stream) {
    // shard_impl(full, shard, ...) with unshard=1 copies shard -> full
    return shard_impl(x, const_cast<void *>(x_sh), B, S, N, D, C, dtype, layout, 1, stream);
}

extern "C" cp_status cp_zigzag_positions(int32_t *pos, int64_t S, int C, cp_layout layout, int on_device,
                                         cudaStream_t stream) {
    if (!pos) return CP_ERR_NULL;
    if (layout != CP_ZIGZAG && layout != CP_CONTIGUOUS) return CP_ERR_ARGUMENT;
    if (S < 1 || C < 1 || S > INT32_MAX) return CP_ERR_SHAPE;
    if (layout == CP_ZIGZAG ? (S % (2LL * C) != 0) : (S % C != 0)) return CP_ERR_DIVISIBILITY;
    if (!on_device) {
        const long long s = S / C;
        for (long long i = 0; i < S; ++i) {
            const long long r = i / s, u = i - r * s;
            long long g;
            if (layout == CP_CONTIGUOUS) {
                g = r * s + u;
            } else {
                const long long t = s / 2;
                g = (u < t) ? (r * t + u) : ((2LL * C - 1 - r) * t + (u - t));
            }
            pos[i] = static_cast<int32_t>(g);
        }
        return CP_OK;
    }
    long long blocks = (S + 255) / 256;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    positions_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(pos, S, C, layout);
    return last_launch_status();
}

namespace cpattn {

cp_status ulysses_relayout_groups(const void *in, void *out, int64_t B, int64_t S, int64_t N, int64_t D, int C,
                                  int groups, cp_dtype dtype, cp_dir dir, cp_seq_order order, cudaStream_t stream) {
    if (!in || !out) return CP_ERR_NULL;
    if (dtype != CP_BF16 && dtype != CP_F32) return CP_ERR_DTYPE;
    if ((dir != CP_SEQ_TO_HEAD && dir != CP_HEAD_TO_SEQ) || (order != CP_RANK_ORDER && order != CP_GLOBAL_ORDER))
        return CP_ERR_ARGUMENT;
    if (B < 1 || S < 1 || N < 1 || D < 1 || C < 1 || groups < 1) return CP_ERR_SHAPE;
    if (S % C != 0 || N % C != 0) return CP_ERR_DIVISIBILITY;
    if (order == CP_GLOBAL_ORDER && S % (2LL * C) != 0) return CP_ERR_DIVISIBILITY;
    const long long es = static_cast<long long>(dtype_size(dtype));
    const long long hb = (N / C) * D * es;
    if (!aligned16(in) || !aligned16(out) || hb % 16 != 0) return CP_ERR_ALIGNMENT;
    const size_t gbytes = static_cast<size_t>(B * S * N * D * es);
    const size_t nbytes = gbytes * static_cast<size_t>(groups);
    if (ranges_overlap(in, nbytes, out, nbytes)) return CP_ERR_ARGUMENT;
    SegArgs a{};
    a.src = static_cast<const uint8_t *>(in);
    a.dst = static_cast<uint8_t *>(out);
    a.kind = dir == CP_SEQ_TO_HEAD ? kUlyssesS2H : kUlyssesH2S;
    a.global_order = order == CP_GLOBAL_ORDER;
    a.B = B;
    a.S = S;
    a.N = N;
    a.C = C;
    a.row_bytes = hb;
    a.seg_rows = a.global_order ? S / (2LL * C) : S / C;
    const long long per_group = static_cast<long long>(C) * B * C * (a.global_order ? 2 : 1);
    a.seg_per_group = groups > 1 ? per_group : 0;
    a.group_bytes = static_cast<long long>(gbytes);
    return launch_segments(a, per_group * groups, stream);
}

}  // namespace cpattn

extern "C" cp_status cp_ulysses_relayout(const void *in, void *out, int64_t B, int64_t S, int64_t N, int64_t D, int C,
                                         cp_dtype dtype, cp_dir dir, cp_seq_order order, cudaStream_t stream) {
    return ulysses_relayout_groups(in, out, B, S, N, D, C, 1, dtype, dir, order, stream);
}
