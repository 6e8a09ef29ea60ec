// selftest.cu -- failure-detection self-test of the bounded device-side waits
// of every attention kernel: the tf32 forward and the two backward kernels as
// well as the bf16 forward.  The kernel's TMA producer first waits for a flag
// that nothing sets (a zeroed word of the caller's scratch) with every bounded
// wait limited to timeout_ns; the wait runs out, the other roles see the abort
// and unwind, TMEM is freed and the kernel records CP_ERR_DEVICE_TIMEOUT in the
// device status word (read with cp_device_status).  No GPU fault is involved.
#include <cuda_runtime.h>

#include <cstdint>

#include "cp_internal.h"

namespace cpattn {
namespace {

constexpr size_t kAlign = 256;
inline size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// One tiny problem: B = 1, 128 query and 128 key rows, one head, D = 64.
constexpr int64_t kRows = 128, kD = 64;

struct Layout {
    size_t flag, q, k, v, dout, qf, kf, vf, vt, o, lse, pos, dq, dk, dv, nl2, nd, total;
};

Layout layout() {
    Layout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += round_up(bytes);
        return at;
    };
    const size_t bf = kRows * kD * 2, f32 = kRows * kD * 4;
    L.flag = take(4);
    L.q = take(bf);
    L.k = take(bf);
    L.v = take(bf);
    L.dout = take(bf);
    L.qf = take(f32);
    L.kf = take(f32);
    L.vf = take(f32);
    L.vt = take(tf32_vt_bytes(1, kRows, 1, kD));
    L.o = take(f32);
    L.lse = take(kRows * 4);
    L.pos = take(kRows * 4);
    L.dq = take(f32);
    L.dk = take(f32);
    L.dv = take(f32);
    L.nl2 = take(bwd_sq_pad(kRows) * 4);
    L.nd = take(bwd_sq_pad(kRows) * 4);
    L.total = off;
    return L;
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" cp_status cp_selftest_stalled_kernel(int kernel, void *scratch, size_t scratch_bytes, uint64_t timeout_ns,
                                                cudaStream_t stream) {
    if (kernel < 0 || kernel > 2) return CP_ERR_ARGUMENT;
    if (timeout_ns < 1000000ull || timeout_ns > 2000000000ull) return CP_ERR_ARGUMENT;
    if (!scratch) return CP_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(scratch) & (kAlign - 1)) return CP_ERR_ALIGNMENT;
    const Layout L = layout();
    static_assert(CP_SELFTEST_SCRATCH_BYTES >= 4096, "scratch size");
    if (L.total > CP_SELFTEST_SCRATCH_BYTES) return CP_ERR_CUDA;  // the stated size must cover the layout
    if (scratch_bytes < CP_SELFTEST_SCRATCH_BYTES) return CP_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(scratch);
    const int *flag = reinterpret_cast<const int *>(w + L.flag);
    // everything zero: the flag is never set, positions are all 0
    cp_status st = cuda_status(cudaMemsetAsync(scratch, 0, L.total, stream));
    if (st != CP_OK) return st;
    if (kernel == 0 || kernel == 1) {
        AttnProblem p{};
        p.q = w + (kernel == 0 ? L.q : L.qf);
        p.k = w + (kernel == 0 ? L.k : L.kf);
        p.v = w + (kernel == 0 ? L.v : L.vf);
        p.q_pos = reinterpret_cast<const int32_t *>(w + L.pos);
        p.k_pos = p.q_pos;
        p.o = reinterpret_cast<float *>(w + L.o);
        p.lse = reinterpret_cast<float *>(w + L.lse);
        p.C = 1;
        p.B = 1;
        p.N = 1;
        p.Nkv = 1;
        p.D = kD;
        p.Sq = kRows;
        p.Sk = kRows;
        p.scale = 0.125f;
        p.hold = flag;
        p.timeout_ns = timeout_ns;
        return kernel == 0 ? launch_attn(p, stream)
                           : launch_attn_tf32(p, reinterpret_cast<const float *>(w + L.vt), stream);
    }
    BwdProblem p{};
    p.q = w + L.q;
    p.k = w + L.k;
    p.v = w + L.v;
    p.dout = w + L.dout;
    p.q_pos = reinterpret_cast<const int32_t *>(w + L.pos);
    p.k_pos = p.q_pos;
    p.nl2 = reinterpret_cast<const float *>(w + L.nl2);
    p.nd = reinterpret_cast<const float *>(w + L.nd);
    p.sq_pad = bwd_sq_pad(kRows);
    p.dq = reinterpret_cast<float *>(w + L.dq);
    p.dk = reinterpret_cast<float *>(w + L.dk);
    p.dv = reinterpret_cast<float *>(w + L.dv);
    p.C = 1;
    p.B = 1;
    p.N = 1;
    p.Nkv = 1;
    p.D = kD;
    p.Sq = kRows;
    p.Sk = kRows;
    p.scale = 0.125f;
    p.hold = flag;
    p.timeout_ns = timeout_ns;
    return launch_bwd(p, stream);  // the dK/dV launch, then the dQ launch: both give up
}
