// strategies.cu -- the all-gather and the all-to-all (Ulysses) forms of
// context-parallel causal attention, for C virtual ranks on one GPU, built
// from the library's own kernels.
//
// All-gather ("On Context Parallelism", All-gather / Forward): every rank
// keeps its local queries; K and V are gathered from all ranks and put back in
// global order (here: cp_zigzag_unshard of the resident shards), and each
// rank's queries attend to the full sequence with their own global positions
// against positions 0..S-1.  All C ranks run in one launch sharing the
// gathered K/V.
//
// All-to-all ("On Context Parallelism", All-to-all; "Context parallelism:
// Ring Attention and Ulysses", Ulysses): q, k and v are relaid from sequence
// sharding [C][B][S/C][N][D] to head sharding [C][B][S][N/C][D] (in global
// sequence order), every head-group rank computes ordinary causal attention
// over the whole sequence for its N/C heads, and the output is relaid back.
// The C head-group ranks are independent problems with the same positions,
// so they run as one launch with the rank folded into the batch.
//
// A2A x P2P mesh ("On Context Parallelism", Peer-to-peer + All-to-all): the
// C = A*R ranks form A2A groups of A consecutive ranks (g*A .. g*A+A-1) and
// P2P groups of R ranks with stride A (a, A+a, 2A+a, ...).  Inside each A2A
// group the sequence shards become head shards (rank order, N/A heads each,
// the group's A*S/C positions concatenated in rank order); each P2P group then
// runs the ring over its R ranks with those concatenated positions, and the
// output goes back through the inverse relayout.  In memory the relaid tensors
// are [R][A][B][S/R][N/A][D]: the A2A index joins the batch, so the A
// independent P2P rings are one ring of R ranks over batch A*B.
#include <cuda_runtime.h>

#include <cstdint>

#include "cp_internal.h"

namespace cpattn {
namespace {

constexpr size_t kAlign = 256;
inline size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct AgLayout {
    size_t k = 0, v = 0, pos = 0, plan = 0, plan_bytes = 0, total = 0;
};
AgLayout ag_layout(int64_t B, int64_t S, int64_t Nkv, int64_t D, int C) {
    AgLayout L;
    const size_t kv = static_cast<size_t>(B) * S * Nkv * D * 2;
    L.k = 0;
    L.v = round_up(kv);
    L.pos = 2 * round_up(kv);
    L.plan = L.pos + round_up(static_cast<size_t>(S) * 4);
    // C query ranks of S/C rows against the one shared key sequence
    L.plan_bytes = (C >= 1 && S % C == 0) ? attn_plan_need(C, 1, S / C, S) : 0;
    L.total = L.plan + round_up(L.plan_bytes);
    return L;
}

struct MeshLayout {
    size_t q = 0, k = 0, v = 0, o = 0, ring = 0, ring_bytes = 0, total = 0;
};
MeshLayout mesh_layout(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int A, int R, int flags,
                       cp_status *st) {
    MeshLayout L;
    const size_t qb = static_cast<size_t>(B) * S * N * D * 2, kvb = static_cast<size_t>(B) * S * Nkv * D * 2;
    L.q = 0;
    L.k = round_up(qb);
    L.v = L.k + round_up(kvb);
    L.o = L.v + round_up(kvb);
    L.ring = L.o + round_up(static_cast<size_t>(B) * S * N * D * 4);
    *st = cp_ring_workspace_size(static_cast<int64_t>(A) * B, S, N / A, Nkv / A, D, R, flags, CP_F32, &L.ring_bytes);
    L.total = L.ring + round_up(L.ring_bytes);
    return L;
}

struct UlLayout {
    size_t q = 0, k = 0, v = 0, o = 0, pos = 0, plan = 0, plan_bytes = 0, total = 0;
};
UlLayout ul_layout(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D) {
    UlLayout L;
    const size_t qb = static_cast<size_t>(B) * S * N * D * 2, kvb = static_cast<size_t>(B) * S * Nkv * D * 2;
    L.q = 0;
    L.k = round_up(qb);
    L.v = L.k + round_up(kvb);
    L.o = L.v + round_up(kvb);
    L.pos = L.o + round_up(static_cast<size_t>(B) * S * N * D * 4);
    L.plan = L.pos + round_up(static_cast<size_t>(S) * 4);
    L.plan_bytes = attn_plan_need(1, 1, S, S);  // head groups folded into the batch: one rank
    L.total = L.plan + round_up(L.plan_bytes);
    return L;
}

cp_status check_common(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int C, cp_layout layout) {
    if (layout != CP_ZIGZAG && layout != CP_CONTIGUOUS) return CP_ERR_ARGUMENT;
    if (C < 1 || C > kMaxC || B < 1 || S < 1 || N < 1 || Nkv < 1) return CP_ERR_SHAPE;
    if (D != 64 && D != 128) return CP_ERR_UNSUPPORTED;
    if (layout == CP_ZIGZAG ? (S % (2LL * C) != 0) : (S % C != 0)) return CP_ERR_DIVISIBILITY;
    if (S > INT32_MAX / 2) return CP_ERR_SHAPE;
    return CP_OK;
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" cp_status cp_allgather_workspace_size(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int C,
                                                 size_t *bytes) {
    if (!bytes) return CP_ERR_NULL;
    if (C < 1 || B < 1 || S < 1 || N < 1 || Nkv < 1 || D < 1) return CP_ERR_SHAPE;
    *bytes = ag_layout(B, S, Nkv, D, C).total;
    return CP_OK;
}

extern "C" cp_status cp_allgather_attention_fwd(const void *q_sh, const void *k_sh, const void *v_sh,
                                                const int32_t *pos, int64_t B, int64_t S, int64_t N, int64_t Nkv,
                                                int64_t D, int C, float scale, cp_layout layout, float *o_sh,
                                                float *lse_sh, void *workspace, size_t ws_bytes,
                                                cudaStream_t stream) {
    if (!q_sh || !k_sh || !v_sh || !pos || !o_sh || !lse_sh) return CP_ERR_NULL;
    cp_status st = check_common(B, S, N, Nkv, D, C, layout);
    if (st != CP_OK) return st;
    const AgLayout L = ag_layout(B, S, Nkv, D, C);
    if (!workspace || ws_bytes < L.total) return CP_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) return CP_ERR_ALIGNMENT;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *k_full = ws + L.k, *v_full = ws + L.v;
    int32_t *gpos = reinterpret_cast<int32_t *>(ws + L.pos);
    const int64_t s = S / C;
    AttnProblem p{};
    p.q = q_sh;
    p.k = k_full;
    p.v = v_full;
    p.kv_shared = true;
    p.q_pos = pos;
    p.q_pos_stride = s;
    p.k_pos = gpos;
    p.k_pos_stride = 0;
    p.o = o_sh;
    p.lse = lse_sh;
    p.C = C;
    p.B = B;
    p.N = N;
    p.Nkv = Nkv;
    p.D = D;
    p.Sq = s;
    p.Sk = S;
    p.scale = scale;
    if (L.plan_bytes) {
        p.plan = ws + L.plan;
        p.plan_bytes = L.plan_bytes;
    }
    st = validate_attn(p);  // everything checked before anything is enqueued
    if (st != CP_OK) return st;
    st = cp_zigzag_unshard(k_sh, k_full, B, S, Nkv, D, C, CP_BF16, layout, stream);
    if (st == CP_OK) st = cp_zigzag_unshard(v_sh, v_full, B, S, Nkv, D, C, CP_BF16, layout, stream);
    if (st == CP_OK) st = cp_zigzag_positions(gpos, S, 1, CP_CONTIGUOUS, 1, stream);  // 0 .. S-1
    if (st == CP_OK) st = launch_attn(p, stream);
    return st;
}

extern "C" cp_status cp_ulysses_workspace_size(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int C,
                                               size_t *bytes) {
    if (!bytes) return CP_ERR_NULL;
    if (C < 1 || B < 1 || S < 1 || N < 1 || Nkv < 1 || D < 1) return CP_ERR_SHAPE;
    *bytes = ul_layout(B, S, N, Nkv, D).total;
    return CP_OK;
}

extern "C" cp_status cp_ulysses_attention_fwd(const void *q_sh, const void *k_sh, const void *v_sh, int64_t B,
                                              int64_t S, int64_t N, int64_t Nkv, int64_t D, int C, float scale,
                                              cp_layout layout, float *o_sh, float *lse_h, void *workspace,
                                              size_t ws_bytes, cudaStream_t stream) {
    if (!q_sh || !k_sh || !v_sh || !o_sh || !lse_h) return CP_ERR_NULL;
    cp_status st = check_common(B, S, N, Nkv, D, C, layout);
    if (st != CP_OK) return st;
    if (N % C != 0 || Nkv % C != 0) return CP_ERR_DIVISIBILITY;
    const UlLayout L = ul_layout(B, S, N, Nkv, D);
    if (!workspace || ws_bytes < L.total) return CP_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) return CP_ERR_ALIGNMENT;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *q_h = ws + L.q, *k_h = ws + L.k, *v_h = ws + L.v;
    float *o_h = reinterpret_cast<float *>(ws + L.o);
    int32_t *gpos = reinterpret_cast<int32_t *>(ws + L.pos);
    // contiguous shards concatenated in rank order already are global order
    const cp_seq_order order = (layout == CP_ZIGZAG) ? CP_GLOBAL_ORDER : CP_RANK_ORDER;
    AttnProblem p{};
    p.q = q_h;
    p.k = k_h;
    p.v = v_h;
    p.q_pos = gpos;
    p.k_pos = gpos;
    p.q_pos_stride = 0;
    p.k_pos_stride = 0;
    p.o = o_h;
    p.lse = lse_h;
    p.C = 1;          // head-group ranks folded into the batch: [C*B][S][N/C][D]
    p.B = C * B;
    p.N = N / C;
    p.Nkv = Nkv / C;
    p.D = D;
    p.Sq = S;
    p.Sk = S;
    p.scale = scale;
    if (L.plan_bytes) {
        p.plan = ws + L.plan;
        p.plan_bytes = L.plan_bytes;
    }
    st = validate_attn(p);
    if (st != CP_OK) return st;
    st = cp_ulysses_relayout(q_sh, q_h, B, S, N, D, C, CP_BF16, CP_SEQ_TO_HEAD, order, stream);
    if (st == CP_OK) st = cp_ulysses_relayout(k_sh, k_h, B, S, Nkv, D, C, CP_BF16, CP_SEQ_TO_HEAD, order, stream);
    if (st == CP_OK) st = cp_ulysses_relayout(v_sh, v_h, B, S, Nkv, D, C, CP_BF16, CP_SEQ_TO_HEAD, order, stream);
    if (st == CP_OK) st = cp_zigzag_positions(gpos, S, 1, CP_CONTIGUOUS, 1, stream);
    if (st == CP_OK) st = launch_attn(p, stream);
    if (st == CP_OK) st = cp_ulysses_relayout(o_h, o_sh, B, S, N, D, C, CP_F32, CP_HEAD_TO_SEQ, order, stream);
    return st;
}

extern "C" cp_status cp_mesh_workspace_size(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int A, int R,
                                            int flags, size_t *bytes) {
    if (!bytes) return CP_ERR_NULL;
    if (A < 1 || R < 1 || B < 1 || S < 1 || N < 1 || Nkv < 1 || D < 1) return CP_ERR_SHAPE;
    if (N % A != 0 || Nkv % A != 0 || S % (static_cast<int64_t>(A) * R) != 0) return CP_ERR_DIVISIBILITY;
    if (flags & ~(CP_RING_PREFETCH | CP_RING_FUSED_MERGE)) return CP_ERR_ARGUMENT;  // bf16 shards only
    cp_status st = CP_OK;
    const MeshLayout L = mesh_layout(B, S, N, Nkv, D, A, R, flags, &st);
    if (st != CP_OK) return st;
    *bytes = L.total;
    return CP_OK;
}

extern "C" cp_status cp_mesh_attention_fwd(const void *q_sh, const void *k_sh, const void *v_sh, const int32_t *pos,
                                           int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int A, int R,
                                           float scale, cp_layout layout, int flags, float *o_sh, float *lse_h,
                                           void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if (!q_sh || !k_sh || !v_sh || !pos || !o_sh || !lse_h) return CP_ERR_NULL;
    if (A < 1 || R < 1 || static_cast<int64_t>(A) * R > kMaxC) return CP_ERR_SHAPE;
    const int C = A * R;
    cp_status st = check_common(B, S, N, Nkv, D, C, layout);
    if (st != CP_OK) return st;
    if (N % A != 0 || Nkv % A != 0) return CP_ERR_DIVISIBILITY;
    if (flags & ~(CP_RING_PREFETCH | CP_RING_FUSED_MERGE)) return CP_ERR_ARGUMENT;  // bf16 shards only
    const MeshLayout L = mesh_layout(B, S, N, Nkv, D, A, R, flags, &st);
    if (st != CP_OK) return st;
    if (!workspace || ws_bytes < L.total) return CP_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) return CP_ERR_ALIGNMENT;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *q_h = ws + L.q, *k_h = ws + L.k, *v_h = ws + L.v;
    float *o_h = reinterpret_cast<float *>(ws + L.o);
    const int64_t sg = S / R;  // positions of one A2A group (A shards, rank order)
    // the relayouts are enqueued before the ring validates its own launch, so
    // check here, before anything is enqueued, the problem the ring will run
    {
        AttnProblem p{};
        p.q = q_h;
        p.k = k_h;
        p.v = v_h;
        p.q_pos = pos;
        p.k_pos = pos;
        p.q_pos_stride = sg;
        p.k_pos_stride = sg;
        p.o = o_h;
        p.lse = lse_h;
        p.C = R;
        p.B = static_cast<int64_t>(A) * B;
        p.N = N / A;
        p.Nkv = Nkv / A;
        p.D = D;
        p.Sq = sg;
        p.Sk = sg;
        p.scale = scale;
        st = validate_attn(p, false);  // the ring's workspace (inside this one) holds its plan
        if (st != CP_OK) return st;
        if (flags & ~(CP_RING_PREFETCH | CP_RING_FUSED_MERGE)) return CP_ERR_ARGUMENT;
    }
    // pos [C][S/C] read as [R][S/R] is each A2A group's concatenation in rank order
    st = ulysses_relayout_groups(q_sh, q_h, B, sg, N, D, A, R, CP_BF16, CP_SEQ_TO_HEAD, CP_RANK_ORDER, stream);
    if (st == CP_OK)
        st = ulysses_relayout_groups(k_sh, k_h, B, sg, Nkv, D, A, R, CP_BF16, CP_SEQ_TO_HEAD, CP_RANK_ORDER, stream);
    if (st == CP_OK)
        st = ulysses_relayout_groups(v_sh, v_h, B, sg, Nkv, D, A, R, CP_BF16, CP_SEQ_TO_HEAD, CP_RANK_ORDER, stream);
    if (st == CP_OK)
        st = cp_ring_attention_fwd(q_h, k_h, v_h, pos, static_cast<int64_t>(A) * B, S, N / A, Nkv / A, D, R, scale,
                                   CP_CONTIGUOUS, flags, o_h, CP_F32, lse_h, ws + L.ring, L.ring_bytes, stream);
    if (st == CP_OK)
        st = ulysses_relayout_groups(o_h, o_sh, B, sg, N, D, A, R, CP_F32, CP_HEAD_TO_SEQ, CP_RANK_ORDER, stream);
    return st;
}
