// ring.cu -- ring (P2P) context-parallel attention forward over C virtual
// ranks resident on one GPU ("On Context Parallelism", Peer-to-peer /
// Forward; "Context Parallelism & Ring Attention", "The ring").
//
// Step `st` of the ring gives every rank r the K/V block of owner
// (r - st) mod C.  All C ranks of a step run in ONE attention launch (their
// work is equal under zigzag sharding, "Context Parallelism & Ring
// Attention", "The zigzag fix"), then one merge launch folds the step's
// partials into the running (o, lse); step 0 writes the accumulator directly.
//
// flags (bit set): CP_RING_FUSED_MERGE folds each step's merge into the
// attention epilogue (the partial is merged straight into the accumulator);
// CP_RING_TF32 takes fp32 q, k, v and runs the tf32 kernel (attn_tf32.cu),
// zero copy only (q and k of every rank are rounded to tf32 and v transposed
// and rounded, once per call, into the workspace).
// The inter-GPU exchange of the pages has two stand-ins here:
//   no CP_RING_PREFETCH  zero copy: the kernel reads the owner's resident block;
//   CP_RING_PREFETCH     the exchange is emulated: the K/V rotation needed by step
//                 st+1 is copied device-to-device on a second stream into a
//                 double buffer while step st computes ("start the next
//                 async send/recv before computing", Peer-to-peer / Forward),
//                 ordered with events and joined back into the caller's stream.
//                 A buffer's refill waits for the step's merge as well as its
//                 attention launch (measured: ~0.6% off the S=32768 ring step
//                 against a refill issued straight after the attention launch).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "cp_internal.h"

namespace cpattn {
namespace {

constexpr size_t kAlign = 256;
inline size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
    size_t o_tile = 0, lse_tile = 0, o_acc = 0, kv = 0, vt = 0, qr = 0, kr = 0, plan = 0, total = 0;
    size_t plan_bytes = 0;  // the attention launches' work plan (0: it fits on chip)
    size_t o_tile_bytes = 0, lse_bytes = 0, o_acc_bytes = 0, kv_bytes = 0;  // kv: one K (or V) rotation
};

Layout ws_layout(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int C, int flags, cp_dtype o_dtype) {
    Layout L;
    const int64_t s = S / C;
    const bool prefetch = (flags & CP_RING_PREFETCH) != 0, fused = (flags & CP_RING_FUSED_MERGE) != 0;
    L.o_tile_bytes = static_cast<size_t>(C) * B * s * N * D * 4;
    L.lse_bytes = static_cast<size_t>(C) * B * N * s * 4;
    L.o_acc_bytes = (o_dtype == CP_BF16) ? L.o_tile_bytes : 0;
    L.kv_bytes = (prefetch && C > 1) ? static_cast<size_t>(C) * B * s * Nkv * D * 2 : 0;
    size_t off = 0;
    L.o_tile = off;
    off += round_up(C > 1 && !fused ? L.o_tile_bytes : 0);
    L.lse_tile = off;
    off += round_up(C > 1 && !fused ? L.lse_bytes : 0);
    L.o_acc = off;
    off += round_up(L.o_acc_bytes);
    L.kv = off;
    off += 4 * round_up(L.kv_bytes);  // 2 buffers x (K, V)
    L.vt = off;
    if (flags & CP_RING_TF32) off += round_up(tf32_vt_bytes(static_cast<int64_t>(C) * B, s, Nkv, D));
    // tf32: q and k rounded to tf32 for the tensor cores (v is rounded in its transpose)
    L.qr = off;
    if (flags & CP_RING_TF32) off += round_up(static_cast<size_t>(C) * B * s * N * D * 4);
    L.kr = off;
    if (flags & CP_RING_TF32) off += round_up(static_cast<size_t>(C) * B * s * Nkv * D * 4);
    // one plan buffer, rebuilt by each step's attention launch in stream order
    L.plan_bytes = (flags & CP_RING_TF32) ? tf32_plan_need(C, C, s, s) : attn_plan_need(C, C, s, s);
    L.plan = off;
    off += round_up(L.plan_bytes);
    L.total = off;
    return L;
}

// Side stream and events for the prefetch path, pooled per device so that
// concurrent host calls never share a set.
struct SideRes {
    int device = -1;
    cudaStream_t side = nullptr;
    cudaEvent_t start = nullptr, join = nullptr, copy_done[2] = {nullptr, nullptr}, attn_done[2] = {nullptr, nullptr};
};

std::mutex g_pool_mu;
std::vector<SideRes *> g_pool;

SideRes *acquire_side(int device) {
    {
        std::lock_guard<std::mutex> lk(g_pool_mu);
        for (size_t i = 0; i < g_pool.size(); ++i)
            if (g_pool[i]->device == device) {
                SideRes *r = g_pool[i];
                g_pool.erase(g_pool.begin() + static_cast<long>(i));
                return r;
            }
    }
    SideRes *r = new SideRes();
    r->device = device;
    bool ok = cudaStreamCreateWithFlags(&r->side, cudaStreamNonBlocking) == cudaSuccess;
    cudaEvent_t *evs[6] = {&r->start, &r->join, &r->copy_done[0], &r->copy_done[1], &r->attn_done[0],
                           &r->attn_done[1]};
    for (auto *e : evs) ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        for (auto *e : evs)
            if (*e) cudaEventDestroy(*e);
        if (r->side) cudaStreamDestroy(r->side);
        delete r;
        return nullptr;
    }
    return r;
}

void release_side(SideRes *r) {
    if (!r) return;
    std::lock_guard<std::mutex> lk(g_pool_mu);
    g_pool.push_back(r);
}

// dst rank r <- src rank (r - st) mod C, for one [C][B][s][Nkv][D] tensor.
cp_status rotate_copy(void *dst, const void *src, size_t rank_bytes, int C, int st, cudaStream_t stream) {
    uint8_t *d = static_cast<uint8_t *>(dst);
    const uint8_t *s = static_cast<const uint8_t *>(src);
    // ranks [st, C) <- [0, C - st);  ranks [0, st) <- [C - st, C)
    if (cudaMemcpyAsync(d + st * rank_bytes, s, (C - st) * rank_bytes, cudaMemcpyDeviceToDevice, stream) !=
        cudaSuccess)
        return CP_ERR_CUDA;
    if (st > 0 && cudaMemcpyAsync(d, s + (C - st) * rank_bytes, st * rank_bytes, cudaMemcpyDeviceToDevice,
                                  stream) != cudaSuccess)
        return CP_ERR_CUDA;
    return CP_OK;
}

}  // namespace

// The checks of a ring call that do not involve its workspace: pointers,
// enums, flags, shapes, divisibility and the attention problem itself.  The
// fp32 accumulator of a bf16 output lives in the (256-byte aligned)
// workspace, so for that case an aligned stand-in address takes its place.
cp_status ring_check_args(const void *q_sh, const void *k_sh, const void *v_sh, const int32_t *pos, int64_t B,
                          int64_t S, int64_t N, int64_t Nkv, int64_t D, int C, float scale, cp_layout layout,
                          int flags, const void *o_sh, cp_dtype o_dtype, const float *lse_sh) {
    if (!q_sh || !k_sh || !v_sh || !pos || !o_sh || !lse_sh) return CP_ERR_NULL;
    if (o_dtype != CP_F32 && o_dtype != CP_BF16) return CP_ERR_DTYPE;
    if (layout != CP_ZIGZAG && layout != CP_CONTIGUOUS) return CP_ERR_ARGUMENT;
    if (flags & ~(CP_RING_PREFETCH | CP_RING_FUSED_MERGE | CP_RING_TF32)) return CP_ERR_ARGUMENT;
    const bool tf32 = (flags & CP_RING_TF32) != 0;
    if (tf32 && (flags & (CP_RING_PREFETCH | CP_RING_FUSED_MERGE))) return CP_ERR_UNSUPPORTED;
    if (C < 1 || C > kMaxC || B < 1 || S < 1 || N < 1 || Nkv < 1) return CP_ERR_SHAPE;
    if (layout == CP_ZIGZAG ? (S % (2LL * C) != 0) : (S % C != 0)) return CP_ERR_DIVISIBILITY;
    alignas(256) static const float acc_stand_in[1] = {0.f};
    AttnProblem chk{};
    chk.q = q_sh;
    chk.k = k_sh;
    chk.v = v_sh;
    chk.q_pos = pos;
    chk.k_pos = pos;
    chk.q_pos_stride = S / C;
    chk.k_pos_stride = S / C;
    chk.o = const_cast<float *>(o_dtype == CP_F32 ? static_cast<const float *>(o_sh) : acc_stand_in);
    chk.lse = const_cast<float *>(lse_sh);
    chk.C = C;
    chk.B = B;
    chk.N = N;
    chk.Nkv = Nkv;
    chk.D = D;
    chk.Sq = S / C;
    chk.Sk = S / C;
    chk.scale = scale;
    return tf32 ? validate_attn_tf32(chk, false) : validate_attn(chk, false);
}

namespace {

cp_status ring_impl(const void *q_sh, const void *k_sh, const void *v_sh, const int32_t *pos, int64_t B, int64_t S,
                    int64_t N, int64_t Nkv, int64_t D, int C, float scale, cp_layout layout, int flags,
                    void *o_sh, cp_dtype o_dtype, float *lse_sh, void *workspace, size_t ws_bytes,
                    cudaStream_t stream, const cudaEvent_t *events, int n_events) {
    {
        const cp_status a = ring_check_args(q_sh, k_sh, v_sh, pos, B, S, N, Nkv, D, C, scale, layout, flags, o_sh,
                                            o_dtype, lse_sh);
        if (a != CP_OK) return a;
    }
    const int prefetch = (flags & CP_RING_PREFETCH) ? 1 : 0;
    const bool fused = (flags & CP_RING_FUSED_MERGE) != 0;
    const bool tf32 = (flags & CP_RING_TF32) != 0;
    if (events && n_events < 4 * C) return CP_ERR_ARGUMENT;
    const int64_t s = S / C;
    const Layout L = ws_layout(B, S, N, Nkv, D, C, flags, o_dtype);
    if (L.total > 0 && (!workspace || ws_bytes < L.total)) return CP_ERR_WORKSPACE;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))) return CP_ERR_ALIGNMENT;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *o_tile = reinterpret_cast<float *>(ws + L.o_tile);
    float *lse_tile = reinterpret_cast<float *>(ws + L.lse_tile);
    float *o_acc = (o_dtype == CP_F32) ? static_cast<float *>(o_sh) : reinterpret_cast<float *>(ws + L.o_acc);
    uint8_t *kbuf[2] = {ws + L.kv, ws + L.kv + round_up(L.kv_bytes)};
    uint8_t *vbuf[2] = {ws + L.kv + 2 * round_up(L.kv_bytes), ws + L.kv + 3 * round_up(L.kv_bytes)};

    AttnProblem p{};
    p.q = q_sh;
    p.q_pos = pos;
    p.k_pos = pos;
    p.q_pos_stride = s;
    p.k_pos_stride = s;
    p.C = C;
    p.B = B;
    p.N = N;
    p.Nkv = Nkv;
    p.D = D;
    p.Sq = s;
    p.Sk = s;
    p.scale = scale;
    if (L.plan_bytes) {
        p.plan = ws + L.plan;
        p.plan_bytes = L.plan_bytes;
    }
    // validate everything once before enqueuing any work
    {
        AttnProblem chk = p;
        chk.k = k_sh;
        chk.v = v_sh;
        chk.o = o_acc;
        chk.lse = lse_sh;
        cp_status st = tf32 ? validate_attn_tf32(chk) : validate_attn(chk);
        if (st != CP_OK) return st;
        if (C > 1 && !fused && (!aligned16(o_tile) || !aligned16(lse_tile))) return CP_ERR_ALIGNMENT;
    }
    const bool use_prefetch = prefetch && C > 1;
    SideRes *res = nullptr;
    if (use_prefetch) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return CP_ERR_CUDA;
        res = acquire_side(dev);
        if (!res) return CP_ERR_CUDA;
    }
    const size_t rank_kv_bytes = static_cast<size_t>(B) * s * Nkv * D * 2;
    cp_status st = CP_OK;
    auto rec = [&](int idx) {
        if (events && st == CP_OK && cudaEventRecord(events[idx], stream) != cudaSuccess) st = CP_ERR_CUDA;
    };
    auto issue_copy = [&](int step) {  // rotation for `step` into buffer step % 2
        if (st != CP_OK) return;
        const int b = step % 2;
        st = rotate_copy(kbuf[b], k_sh, rank_kv_bytes, C, step, res->side);
        if (st == CP_OK) st = rotate_copy(vbuf[b], v_sh, rank_kv_bytes, C, step, res->side);
        if (st == CP_OK && cudaEventRecord(res->copy_done[b], res->side) != cudaSuccess) st = CP_ERR_CUDA;
    };
    float *vt = reinterpret_cast<float *>(ws + L.vt);
    float *qr = reinterpret_cast<float *>(ws + L.qr), *kr = reinterpret_cast<float *>(ws + L.kr);
    if (tf32) {
        st = launch_tf32_round(static_cast<const float *>(q_sh), qr, static_cast<int64_t>(C) * B * s * N * D, stream);
        if (st == CP_OK)
            st = launch_tf32_round(static_cast<const float *>(k_sh), kr, static_cast<int64_t>(C) * B * s * Nkv * D,
                                   stream);
        if (st == CP_OK)
            st = launch_tf32_transpose(static_cast<const float *>(v_sh), vt, static_cast<int64_t>(C) * B, s, Nkv, D,
                                       stream);
        p.q = qr;
    }
    if (use_prefetch) {
        if (cudaEventRecord(res->start, stream) != cudaSuccess || cudaStreamWaitEvent(res->side, res->start, 0) !=
                                                                        cudaSuccess)
            st = CP_ERR_CUDA;
        issue_copy(1);
    }
    for (int step = 0; step < C && st == CP_OK; ++step) {
        const int back = (C - step) % C;  // owner = (r - step) mod C = (r + back) mod C
        AttnProblem ps = p;
        ps.kpos_shift = back;
        if (step == 0 || !use_prefetch) {
            ps.k = tf32 ? static_cast<const void *>(kr) : k_sh;
            ps.v = v_sh;
            ps.kv_shift = back;
        } else {
            if (cudaStreamWaitEvent(stream, res->copy_done[step % 2], 0) != cudaSuccess) {
                st = CP_ERR_CUDA;
                break;
            }
            ps.k = kbuf[step % 2];
            ps.v = vbuf[step % 2];
            ps.kv_shift = 0;
        }
        // fused: steps >= 1 merge their partial into the accumulator in the
        // attention epilogue; otherwise they write the partial and a merge follows
        ps.merge_into = fused && step > 0;
        ps.o = (step == 0 || fused) ? o_acc : o_tile;
        ps.lse = (step == 0 || fused) ? lse_sh : lse_tile;
        rec(4 * step + 0);
        if (st == CP_OK) st = tf32 ? launch_attn_tf32(ps, vt, stream) : launch_attn(ps, stream);
        rec(4 * step + 1);
        rec(4 * step + 2);
        if (step > 0 && !fused && st == CP_OK)
            st = launch_merge(o_acc, lse_sh, o_tile, lse_tile, C * B, s, N, D, stream);
        rec(4 * step + 3);
        if (use_prefetch && st == CP_OK && step + 2 < C) {
            // buffer (step+2)%2 was last read by this step's attention launch;
            // the refill is ordered after the merge too (see the file header)
            if (cudaEventRecord(res->attn_done[step % 2], stream) != cudaSuccess ||
                cudaStreamWaitEvent(res->side, res->attn_done[step % 2], 0) != cudaSuccess)
                st = CP_ERR_CUDA;
            issue_copy(step + 2);
        }
    }
    if (use_prefetch) {
        // join the side stream back into the caller's stream in every case
        if (cudaEventRecord(res->join, res->side) != cudaSuccess ||
            cudaStreamWaitEvent(stream, res->join, 0) != cudaSuccess)
            if (st == CP_OK) st = CP_ERR_CUDA;
        release_side(res);
    }
    if (st == CP_OK && o_dtype == CP_BF16) st = launch_f32_to_bf16(o_acc, o_sh, C * B * s * N * D, stream);
    return st;
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" cp_status cp_ring_workspace_size(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int C,
                                            int flags, cp_dtype o_dtype, size_t *bytes) {
    if (!bytes) return CP_ERR_NULL;
    if (o_dtype != CP_F32 && o_dtype != CP_BF16) return CP_ERR_DTYPE;
    if (C < 1 || C > kMaxC || B < 1 || S < 1 || N < 1 || Nkv < 1 || D < 1) return CP_ERR_SHAPE;
    if (S % C != 0) return CP_ERR_DIVISIBILITY;
    if (flags & ~(CP_RING_PREFETCH | CP_RING_FUSED_MERGE | CP_RING_TF32)) return CP_ERR_ARGUMENT;
    *bytes = ws_layout(B, S, N, Nkv, D, C, flags, o_dtype).total;
    return CP_OK;
}

extern "C" cp_status cp_ring_attention_fwd(const void *q_sh, const void *k_sh, const void *v_sh, const int32_t *pos,
                                           int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int C,
                                           float scale, cp_layout layout, int flags, void *o_sh,
                                           cp_dtype o_dtype, float *lse_sh, void *workspace, size_t ws_bytes,
                                           cudaStream_t stream) {
    return ring_impl(q_sh, k_sh, v_sh, pos, B, S, N, Nkv, D, C, scale, layout, flags, o_sh, o_dtype, lse_sh,
                     workspace, ws_bytes, stream, nullptr, 0);
}

extern "C" cp_status cp_ring_attention_fwd_traced(const void *q_sh, const void *k_sh, const void *v_sh,
                                                  const int32_t *pos, int64_t B, int64_t S, int64_t N,
                                                  int64_t Nkv, int64_t D, int C, float scale, cp_layout layout,
                                                  int flags, void *o_sh, cp_dtype o_dtype, float *lse_sh,
                                                  void *workspace, size_t ws_bytes, cudaStream_t stream,
                                                  cudaEvent_t const *events, int n_events) {
    if (!events) return CP_ERR_NULL;
    return ring_impl(q_sh, k_sh, v_sh, pos, B, S, N, Nkv, D, C, scale, layout, flags, o_sh, o_dtype, lse_sh,
                     workspace, ws_bytes, stream, events, n_events);
}
