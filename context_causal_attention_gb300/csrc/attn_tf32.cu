// attn_tf32.cu -- the partial causal attention of attn.cu for fp32 inputs, with
// the tensor cores in tf32 (tcgen05.mma kind::tf32: 10-bit mantissa operands,
// fp32 accumulation).  Same result definition ("On Context Parallelism",
// Peer-to-peer / Forward: (o, lse) of the queries against one K/V block with
// positions), same rank batching (AttnProblem), same causal tile skipping and
// the same lazy integer running max in the log2 domain as the bf16 kernel.
//
// Layout of the work: one persistent CTA per SM, 256 threads; work items are
// (rank, b, h, 128-row query tile, or tiles u and nqt-1-u back to back), in the
// shared order of cp_sched.cuh.
//   warp 0      TMA producer: the 128-row fp32 query tile of the item, then
//               2-stage rings of 64-key K tiles and 64-key V^T tiles (128-byte
//               swizzle, 32 fp32 columns per swizzle atom), with separate
//               barriers: a K stage is refilled as soon as its scores are
//               computed, and each V^T tile is loaded one tile after its K;
//   warp 1      TMEM allocator (256 columns: S0 | S1 | O) and MMA issuer:
//               S_b = Q K^T (M = 128, N = 64, K = 8 per instruction) into the
//               score buffer b = tile parity, O += P V with P read from TMEM;
//   warps 2-3   idle;
//   warps 4-7   softmax, one thread per query row: P = 2^(s*scale*log2 e - m)
//               written back over S as fp32 (the A operand of P V).
// S is double buffered, so the MMA of tile j+1 runs while the softmax works on
// tile j.  Every tf32 operand is K-major: P V takes V^T ([D][keys], written by
// tf32_transpose_kernel into the caller's workspace) as its B operand.  When a
// row's running max must move, O is rescaled in TMEM after the previous tile's
// P V has completed (a per-tile completion barrier).
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "cp_internal.h"
#include "cp_hold.cuh"
#include "cp_ptx.cuh"
#include "cp_sched.cuh"
#include "cp_rounds.cuh"

namespace cpattn {

// Sticky device status word of the tf32 kernel (read by cp_device_status).
__device__ int g_cp_device_status_tf32 = 0;

namespace {

constexpr int kTThreads = 256;
constexpr int kTStages = 2;
constexpr uint32_t kTTmemCols = 256;
constexpr uint32_t kTNegInf = 0xff800000u;

template <int D>
struct CfgT {
    static constexpr int kAtoms = D / 32;              // 32 fp32 columns per 128-byte swizzle atom
    static constexpr int kQBytes = 128 * D * 4;        // 128-row query tile
    static constexpr int kKBytes = 64 * D * 4;         // 64-key tile
    static constexpr int kQAtom = 128 * 128, kKAtom = 64 * 128;
    static constexpr int kVtAtom = D * 128;             // V^T tile: D rows x 32 keys per atom, 2 atoms
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kQBytes;
    static constexpr int kOffV = kOffK + kTStages * kKBytes;
    static constexpr int kOffTab = kOffV + kTStages * kKBytes;
    static constexpr int kOffOrder = kOffTab + kMaxTables * 8;
    static constexpr int kOffCost = kOffOrder + kMaxPairs * 4;
    static constexpr int kOffSeg = kOffCost + kMaxPairs * 4;
    // q_full, q_empty, k_full[S], k_empty[S], s_full[2], p_full[2], pv_done, o_full,
    // o_empty, drain, v_full[S], v_empty[S]
    static constexpr int kNumBars = 2 + 2 * kTStages + 9 + 2 * kTStages;
    static constexpr int kOffBar = kOffSeg + (kMaxPairs + 2) * 4;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kMiscBytes = 16 + kMaxC * 4 + kMaxTables / 8;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct TArgs {
    const int32_t *q_pos, *k_pos;
    long long q_pos_stride, k_pos_stride;
    float *o, *lse;
    int C, B, N, Nkv, Sq, Sk;
    int nqt, nkt;  // 128-row query tiles, 64-key tiles
    int kv_shift, kpos_shift, kv_shared, kpr;
    float scale_log2;
    unsigned long long timeout_ns;
    int pair;  // a super-block holds query tiles u and nqt-1-u (else u alone)
    FastDiv div_nsp, div_n;
    PlanPtrs gp;  // the launch's plan in global memory (kernels with kGlobalPlan)
    const int *hold;  // failure injection (self-test only), else null
};

// kind::tf32 instruction descriptor: D fp32 (bits 4-5 = 1), A and B tf32
// (bits 7-9 = 2, 10-12 = 2), A/B major in bits 15/16, N >> 3 in 17-22,
// M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(uint32_t M, uint32_t N, uint32_t a_mn_major,
                                                      uint32_t b_mn_major) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (a_mn_major << 15) | (b_mn_major << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}
__device__ __forceinline__ void umma_tf32_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void umma_tf32_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// fp32 -> tf32 (10-bit mantissa) by rounding to nearest (ties away from zero)
// in the fp32 container; the tensor core reads the top 19 bits.
__device__ __forceinline__ uint32_t round_tf32(float x) { return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u; }

__device__ __forceinline__ void tile_minmax(const int32_t *p, int row0, int rows, int lim, int lane, int2 *out,
                                            uint32_t *arith, int g) {
    int mn = INT_MAX, mx = INT_MIN, first = 0;
    bool ok = true;
    for (int m = 0; m < rows / 32; ++m) {
        const int row = row0 + lane + 32 * m;
        const int val = (row < lim) ? __ldg(p + row) : 0;
        if (m == 0) first = __shfl_sync(0xffffffffu, val, 0);
        if (row < lim) {
            mn = min(mn, val);
            mx = max(mx, val);
            ok &= (static_cast<long long>(val) == static_cast<long long>(first) + lane + 32 * m);
        }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    ok = __all_sync(0xffffffffu, ok);
    if (lane == 0) {
        *out = make_int2(mn, mx);
        if (arith && ok) atomicOr(arith + (g >> 5), 1u << (g & 31));
    }
}

// kGlobalPlan: the plan was written to global memory by the pre-pass (else
// every CTA builds it in shared memory).
template <int D, bool kGlobalPlan>
__global__ void __launch_bounds__(kTThreads, 1)
    attn_tf32_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmVt, const TArgs a) {
    using K = CfgT<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int2 *tab_s = reinterpret_cast<int2 *>(smem + K::kOffTab);
    int *order_s = reinterpret_cast<int *>(smem + K::kOffOrder);
    int *cost_s = reinterpret_cast<int *>(smem + K::kOffCost);
    int *seg_s = reinterpret_cast<int *>(smem + K::kOffSeg);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + K::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + K::kOffMisc + 4);
    int *sorted_s = reinterpret_cast<int *>(smem + K::kOffMisc + 16);
    uint32_t *bits_s = reinterpret_cast<uint32_t *>(smem + K::kOffMisc + 16 + kMaxC * 4);
    const int *order = kGlobalPlan ? a.gp.order : order_s;
    const int *cost = kGlobalPlan ? a.gp.cost : cost_s;
    const int *seg_first = kGlobalPlan ? a.gp.seg_first : seg_s;
    const int *sorted_flag = kGlobalPlan ? a.gp.ksorted : sorted_s;
    const uint32_t *arith_bits = kGlobalPlan ? a.gp.kbits : bits_s;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + K::kOffBar);
    uint64_t *q_full = bar, *q_empty = bar + 1, *k_full = bar + 2, *k_empty = bar + 2 + kTStages;
    uint64_t *s_full = bar + 2 + 2 * kTStages, *p_full = s_full + 2, *pv_done = s_full + 4, *o_full = s_full + 5,
             *o_empty = s_full + 6, *drain = s_full + 7;
    uint64_t *v_full = s_full + 8, *v_empty = v_full + kTStages;
    const int2 *ktab = kGlobalPlan ? a.gp.ktab : tab_s;                 // [kpr][nkt] 64-key tiles
    const int2 *qtab = kGlobalPlan ? a.gp.qtab : tab_s + a.kpr * a.nkt;  // [C][nqt] 128-row query tiles

    if (tid == 0) {
        *abort_flag = 0;
        if (!kGlobalPlan)
            for (int w = 0; w < kMaxTables / 32; ++w) bits_s[w] = 0u;
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < kTStages; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, 1);
            mbar_init(v_full + s, 1);
            mbar_init(v_empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full + i, 1);
            mbar_init(p_full + i, 4);
        }
        mbar_init(pv_done, 1);
        mbar_init(o_full, 1);
        mbar_init(o_empty, 4);
        mbar_init(drain, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmVt);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTTmemCols);
        tmem_relinquish();
    }
    __syncthreads();
    if constexpr (!kGlobalPlan) {
        {
            const int nk = a.kpr * a.nkt, total = nk + a.C * a.nqt;
            for (int g = warp; g < total; g += kTThreads / 32) {
                if (g < nk) {
                    const int j = g / a.nkt, kt = g - (g / a.nkt) * a.nkt;
                    tile_minmax(a.k_pos + j * a.k_pos_stride, kt * 64, 64, a.Sk, lane, tab_s + g, bits_s, g);
                } else {
                    const int gq = g - nk, r = gq / a.nqt, qt = gq - (gq / a.nqt) * a.nqt;
                    tile_minmax(a.q_pos + r * a.q_pos_stride, qt * 128, 128, a.Sq, lane, tab_s + g, nullptr, 0);
                }
            }
        }
        __syncthreads();
        if (tid < a.kpr) {
            int ok = 1;
            for (int kt = 1; kt < a.nkt; ++kt) ok &= (ktab[tid * a.nkt + kt].x >= ktab[tid * a.nkt + kt - 1].x);
            sorted_s[tid] = ok;
        }
        __syncthreads();
        const int np = a.C * a.nqt;
        for (int p = tid; p < np; p += kTThreads) {
            const int r = p / a.nqt, qt = p - (p / a.nqt) * a.nqt;
            const int owner = (a.kpr == 1) ? 0 : (r + a.kpos_shift) % a.C;
            const int qmax = qtab[r * a.nqt + qt].y;
            const int2 *kt_o = ktab + owner * a.nkt;
            int c = 0;
            for (int kt = 0; kt < a.nkt; ++kt) c += (kt_o[kt].x <= qmax);
            cost_s[p] = c;
        }
        __syncthreads();
        build_segments<kTThreads>(cost_s, a.C, a.nqt, a.pair != 0, order_s, seg_s);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_items = a.C * super_count(a.nqt, a.pair != 0) * a.B * a.N;
    const int n_rounds = (n_items + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    const int hq_per_kv = a.N / a.Nkv;
    uint8_t *sQ = smem + K::kOffQ, *sK = smem + K::kOffK, *sV = smem + K::kOffV;  // sV holds V^T tiles
    // query tile `unit` of super item x -> (rank, query tile, b, head, ...)
    auto decode = [&](const SuperItem &x, int unit, int &r, int &qt, int &b, int &h, int &owner, int &kvr, int &pr) {
        r = x.r;
        qt = unit;
        pr = r * a.nqt + qt;
        b = static_cast<int>(fdiv(static_cast<uint32_t>(x.bh), a.div_n));
        h = x.bh - b * a.N;
        owner = (a.kpr == 1) ? 0 : (r + a.kpos_shift) % a.C;
        kvr = a.kv_shared ? 0 : (r + a.kv_shift) % a.C;
    };
    // key tiles an item processes: those whose smallest position <= the tile's largest query position
    auto next_kt = [&](int kt, const int2 *kt_o, int qmax, bool srt) {
        for (; kt < a.nkt; ++kt) {
            if (kt_o[kt].x <= qmax) return kt;
            if (srt) return a.nkt;
        }
        return a.nkt;
    };

    if (warp == 0) {
        // -------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t it = 0, t = 0, k_issued = 0, k_par = 0, v_issued = 0, v_par = 0;
            int q_par = -1;
            // V^T of a tile is loaded one tile after its K: a K stage is freed as soon
            // as that tile's scores are computed, so the next K loads while the
            // softmax and P V of earlier tiles run
            auto load_v = [&](int kt, uint32_t st, uint32_t ph, int hk, int kvrow) -> bool {
                if (!mbar_wait(v_empty + st, ph ^ 1u, abort_flag, a.timeout_ns)) return false;
                mbar_arrive_expect_tx(v_full + st, K::kKBytes);
                // V^T [D rows][keys kt*64 ..]: two atoms of 32 keys
                for (int at = 0; at < 2; ++at)
                    tma_load_4d(sV + st * K::kKBytes + at * K::kVtAtom, &tmVt, v_full + st, kt * 64 + 32 * at, 0, hk,
                                kvrow);
                v_issued |= 1u << st;
                v_par = (v_par & ~(1u << st)) | (ph << st);
                return true;
            };
            bool ok = true;
            if (a.hold) ok = hold_wait(a.hold, a.timeout_ns, abort_flag);
            int seg = 0;  // segment cursor of decode_super
            for (int rk = 0; rk < n_rounds && ok; ++rk) {
                const RoundWork rw = work_of_round(rk, n_items, a.pair != 0);
                if (rw.idx < 0) continue;
                const SuperItem sup = decode_super(rw.idx, a.B * a.N, order, seg_first, a.div_nsp, seg);
                for (int part = rw.p0; part < rw.p1 && ok; ++part) {
                    const int unit = super_part(sup.u, part, a.nqt, a.pair != 0);
                    if (unit < 0) continue;
                    int r, qt, b, h, owner, kvr, pr;
                    decode(sup, unit, r, qt, b, h, owner, kvr, pr);
                    if (cost[pr] == 0) continue;
                    if (!mbar_wait(q_empty, (it & 1u) ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    mbar_arrive_expect_tx(q_full, K::kQBytes);
                    q_par = static_cast<int>(it & 1u);
                    for (int at = 0; at < K::kAtoms; ++at)
                        tma_load_4d(sQ + at * K::kQAtom, &tmQ, q_full, 32 * at, h, qt * 128, r * a.B + b);
                    ++it;
                    const int2 *kt_o = ktab + owner * a.nkt;
                    const int qmax = qtab[r * a.nqt + qt].y;
                    const bool srt = sorted_flag[owner] != 0;
                    const int hk = h / hq_per_kv, kvrow = kvr * a.B + b;
                    int pkt = -1;  // tile whose V^T is still to be loaded
                    uint32_t pst = 0, pph = 0;
                    for (int kt = next_kt(0, kt_o, qmax, srt); kt < a.nkt; kt = next_kt(kt + 1, kt_o, qmax, srt)) {
                        const uint32_t st = t % kTStages, ph = (t / kTStages) & 1u;
                        if (!mbar_wait(k_empty + st, ph ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        mbar_arrive_expect_tx(k_full + st, K::kKBytes);
                        for (int at = 0; at < K::kAtoms; ++at)
                            tma_load_4d(sK + st * K::kKBytes + at * K::kKAtom, &tmK, k_full + st, 32 * at, hk, kt * 64, kvrow);
                        k_issued |= 1u << st;
                        k_par = (k_par & ~(1u << st)) | (ph << st);
                        if (pkt >= 0 && !load_v(pkt, pst, pph, hk, kvrow)) { ok = false; break; }
                        pkt = kt;
                        pst = st;
                        pph = ph;
                        ++t;
                    }
                    if (ok && pkt >= 0 && !load_v(pkt, pst, pph, hk, kvrow)) ok = false;
                }
            }
            if (!ok) {
                volatile int no_abort = 0;
                if (q_par >= 0) mbar_wait(q_full, static_cast<uint32_t>(q_par), &no_abort, 100000000ull);
                for (int st = 0; st < kTStages; ++st) {
                    if ((k_issued >> st) & 1u) mbar_wait(k_full + st, (k_par >> st) & 1u, &no_abort, 100000000ull);
                    if ((v_issued >> st) & 1u) mbar_wait(v_full + st, (v_par >> st) & 1u, &no_abort, 100000000ull);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_tf32_f32(128, 64, 0, 0);
            constexpr uint32_t kIdO = idesc_tf32_f32(128, D, 0, 0);  // B = V^T, K-major
            constexpr uint64_t kKU = K::kKBytes >> 4;
            const uint64_t dq = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dk = smem_desc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t dv = smem_desc_sw128(smem_u32(sV), 16, 1024);
            uint32_t it = 0, t = 0;
            bool ok = true;
            // S_b = Q K^T of the tile in stage st: D/8 k-steps of 8 fp32 (32 bytes);
            // k-step kk at (kk / 4) swizzle atoms + (kk % 4) * 32 bytes
            auto issue_s = [&](uint32_t b, uint32_t st) {
                for (int kk = 0; kk < D / 8; ++kk)
                    umma_tf32_ss(tmem + 64 * b, dq + (kk >> 2) * (K::kQAtom >> 4) + (kk & 3) * 2,
                                 dk + st * kKU + (kk >> 2) * (K::kKAtom >> 4) + (kk & 3) * 2, kIdS, kk > 0 ? 1u : 0u);
                umma_commit(s_full + b);
                umma_commit(k_empty + st);  // the K stage is free once the scores are done
            };
            int seg = 0;  // segment cursor of decode_super
            for (int rk = 0; rk < n_rounds && ok; ++rk) {
                const RoundWork rw = work_of_round(rk, n_items, a.pair != 0);
                if (rw.idx < 0) continue;
                const SuperItem sup = decode_super(rw.idx, a.B * a.N, order, seg_first, a.div_nsp, seg);
                for (int part = rw.p0; part < rw.p1 && ok; ++part) {
                    const int unit = super_part(sup.u, part, a.nqt, a.pair != 0);
                    if (unit < 0) continue;
                    int r, qt, b, h, owner, kvr, pr;
                    decode(sup, unit, r, qt, b, h, owner, kvr, pr);
                    const int n = cost[pr];
                    if (n == 0) continue;
                    if (!mbar_wait(q_full, it & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    // the first two tiles' scores, then per tile: P V, and the scores
                    // of the tile after next into the buffer P V has just read
                    for (int j = 0; j < 2 && j < n; ++j) {
                        const uint32_t st = (t + j) % kTStages, ph = ((t + j) / kTStages) & 1u;
                        if (!mbar_wait(k_full + st, ph, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        issue_s((t + j) & 1u, st);
                    }
                    if (!ok) break;
                    if (n <= 2) umma_commit(q_empty);
                    for (int j = 0; j < n; ++j, ++t) {
                        const uint32_t bb = t & 1u, st = t % kTStages, ph = (t / kTStages) & 1u;
                        const uint32_t st2 = (t + 2) % kTStages, ph2 = ((t + 2) / kTStages) & 1u;
                        // the waits that do not depend on the softmax come first, so P V
                        // and the next scores follow this tile's P directly
                        if (j == 0 && !mbar_wait(o_empty, (it & 1u) ^ 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        if (!mbar_wait(v_full + st, ph, abort_flag, a.timeout_ns)) { ok = false; break; }
                        if (j + 2 < n && !mbar_wait(k_full + st2, ph2, abort_flag, a.timeout_ns)) { ok = false; break; }
                        if (!mbar_wait(p_full + bb, (t >> 1) & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
                        // O (+)= P V: 64 keys in 8 k-steps of 8 (P columns +8; V^T k-step kk
                        // at (kk / 4) atoms + (kk % 4) * 32 bytes)
                        for (int kk = 0; kk < 8; ++kk)
                            umma_tf32_ts(tmem + 128, tmem + 64 * bb + 8 * kk,
                                         dv + st * kKU + (kk >> 2) * (K::kVtAtom >> 4) + (kk & 3) * 2, kIdO,
                                         (j > 0 || kk > 0) ? 1u : 0u);
                        umma_commit(pv_done);
                        umma_commit(v_empty + st);
                        if (j + 2 < n) {
                            issue_s(bb, st2);
                            if (j + 3 == n) umma_commit(q_empty);
                        }
                    }
                    if (!ok) break;
                    umma_commit(o_full);
                    ++it;
                }
            }
            umma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait(drain, 0, &no_abort, 100000000ull);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // -------------------------------------------------------- softmax
        const int wq = warp & 3;
        const int row_in = wq * 32 + lane;
        const uint32_t tA = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const float sl2 = a.scale_log2;
        uint32_t it = 0, t = 0;
        bool ok = true;
        int seg = 0;  // segment cursor of decode_super
        for (int rk = 0; rk < n_rounds && ok; ++rk) {
            const RoundWork rw = work_of_round(rk, n_items, a.pair != 0);
            if (rw.idx < 0) continue;
            const SuperItem sup = decode_super(rw.idx, a.B * a.N, order, seg_first, a.div_nsp, seg);
            for (int part = rw.p0; part < rw.p1 && ok; ++part) {
                const int unit = super_part(sup.u, part, a.nqt, a.pair != 0);
                if (unit < 0) continue;
                int r, qt, b, h, owner, kvr, pr;
                decode(sup, unit, r, qt, b, h, owner, kvr, pr);
                const int row = qt * 128 + row_in;
                const bool row_valid = row < a.Sq;
                const int qpos = row_valid ? __ldg(a.q_pos + r * a.q_pos_stride + row) : INT_MIN;
                const long long orow = static_cast<long long>(r * a.B + b) * a.Sq + row;
                float *o_row = a.o + (orow * a.N + h) * D;
                float *lse_out = a.lse + (static_cast<long long>(r * a.B + b) * a.N + h) * a.Sq + row;
                if (cost[pr] == 0) {
                    if (row_valid) {
                        for (int c = 0; c < D; c += 8) st_global_v8(o_row + c, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f);
                        *lse_out = -INFINITY;
                    }
                    continue;
                }
                const int2 *kt_o = ktab + owner * a.nkt;
                const int2 qmm = qtab[r * a.nqt + qt];
                const bool srt = sorted_flag[owner] != 0;
                const int32_t *kpos_o = a.k_pos + owner * a.k_pos_stride;
                float m_run = -INFINITY, l_run = 0.f;
                bool first_tile = true;
                for (int kt = next_kt(0, kt_o, qmm.y, srt); kt < a.nkt; kt = next_kt(kt + 1, kt_o, qmm.y, srt), ++t) {
                    const uint32_t bb = t & 1u;
                    if (!mbar_wait_warp(s_full + bb, (t >> 1) & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    uint32_t s[64];
                    tmem_ld64(tA + 64 * bb, s);
                    const int2 kmm = kt_o[kt];
                    const int k0 = kt * 64, nvalid = min(64, a.Sk - k0);
                    if (kmm.y > qmm.x || nvalid < 64) {
                        const int gk = owner * a.nkt + kt;
                        if ((arith_bits[gk >> 5] >> (gk & 31)) & 1u) {
                            const long long dhi = static_cast<long long>(qpos) - kmm.x;
                            const int lim = dhi < 0 ? -1 : static_cast<int>(min(dhi, static_cast<long long>(nvalid - 1)));
    #pragma unroll
                            for (int c = 0; c < 64; ++c)
                                if (c > lim) s[c] = kTNegInf;
                        } else {
    #pragma unroll
                            for (int c0 = 0; c0 < 64; c0 += 16) {
    #pragma unroll
                                for (int c = c0; c < c0 + 16; ++c) {
                                    const int kp = (c < nvalid) ? __ldg(kpos_o + k0 + c) : INT_MAX;
                                    if (kp > qpos) s[c] = kTNegInf;
                                }
                                asm volatile("" ::: "memory");
                            }
                        }
                    }
                    // lazy integer max (log2 domain): set on the row's first visible tile,
                    // moved only when a score exceeds it by more than 57 (64 keys x 2^57
                    // keeps a tile's P sum below 2^64)
                    float mx = -INFINITY;
    #pragma unroll
                    for (int c = 0; c < 64; c += 2) mx = fmax3(mx, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
                    const float m_tile = mx * sl2;
                    float factor = 1.f;
                    bool rescale = false;
                    if (m_run == -INFINITY) {
                        if (m_tile > -INFINITY) m_run = ceilf(m_tile);
                    } else if (!(m_tile - m_run <= 57.f)) {
                        const float m_new = ceilf(m_tile);
                        const float dk = m_run - m_new;
                        factor = (dk >= -126.f) ? __int_as_float((127 + static_cast<int>(dk)) << 23) : 0.f;
                        rescale = true;
                        l_run *= factor;
                        m_run = m_new;
                    }
                    const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
                    float sum = 0.f;
    #pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const float p = fast_exp2(fmaf(__uint_as_float(s[c]), sl2, neg_m));
                        sum += p;
                        s[c] = round_tf32(p);
                    }
                    l_run += sum;
                    // P over S (fp32, the A operand of P V)
                    tmem_st32_nowait(tA + 64 * bb, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                    tmem_st32_nowait(tA + 64 * bb + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                    tmem_wait_st();
                    if (__any_sync(0xffffffffu, rescale)) {
                        // O must be quiescent: the previous tile's P V has completed
                        if (!first_tile && !mbar_wait_warp(pv_done, (t - 1) & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                        tc_fence_after();
    #pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t ov[32];
                            tmem_ld32(tA + 128 + c0, ov);
    #pragma unroll
                            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * factor);
                            tmem_st32(tA + 128 + c0, ov);
                        }
                    }
                    first_tile = false;
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_full + bb);
                }
                if (!ok) break;
                if (!mbar_wait_warp(o_full, it & 1u, abort_flag, a.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
    #pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t ov[32];
                    tmem_ld32(tA + 128 + c0, ov);
                    if (row_valid) {
    #pragma unroll
                        for (int c = 0; c < 32; c += 8)
                            st_global_v8(o_row + c0 + c, __uint_as_float(ov[c]) * inv_l, __uint_as_float(ov[c + 1]) * inv_l,
                                         __uint_as_float(ov[c + 2]) * inv_l, __uint_as_float(ov[c + 3]) * inv_l,
                                         __uint_as_float(ov[c + 4]) * inv_l, __uint_as_float(ov[c + 5]) * inv_l,
                                         __uint_as_float(ov[c + 6]) * inv_l, __uint_as_float(ov[c + 7]) * inv_l);
                    }
                }
                if (row_valid)
                    *lse_out = (l_run > 0.f) ? (m_run + __log2f(l_run)) * 0.69314718055994530942f : -INFINITY;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_empty);
                ++it;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTTmemCols);
    }
    if (tid == 0 && *abort_flag) atomicExch(&g_cp_device_status_tf32, static_cast<int>(CP_ERR_DEVICE_TIMEOUT));
}

// out = in rounded to the nearest tf32 value (10-bit mantissa, ties away from
// zero), n4 float4 vectors; q and k pass through it so that the tensor cores,
// which take the top 19 bits of each fp32 operand, see rounded rather than
// truncated values.
__global__ void __launch_bounds__(256) tf32_round_kernel(const float4 *__restrict__ in, float4 *__restrict__ out,
                                                         long long n4) {
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 x = __ldg(in + i);
        out[i] = make_float4(__uint_as_float(round_tf32(x.x)), __uint_as_float(round_tf32(x.y)),
                             __uint_as_float(round_tf32(x.z)), __uint_as_float(round_tf32(x.w)));
    }
}

// vt[o][h][d][j] = v[o][j][h][d] for j < Sk, rounded to tf32 (rows padded to sk_pad with zeros)
__global__ void __launch_bounds__(256) tf32_transpose_kernel(const float *__restrict__ v, float *__restrict__ vt,
                                                             long long outer, int Sk, int Nkv, int D, int sk_pad) {
    __shared__ float tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const long long oh = blockIdx.z;                           // o * Nkv + h
    const long long o = oh / Nkv, h = oh - o * Nkv;
    const int j0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
    for (int i = ty; i < 32; i += 8) {
        const int j = j0 + i;
        tile[i][tx] = (j < Sk) ? v[((o * Sk + j) * Nkv + h) * D + d0 + tx] : 0.f;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int j = j0 + tx;
        if (j < sk_pad) vt[((o * Nkv + h) * D + d0 + i) * sk_pad + j] = __uint_as_float(round_tf32(tile[tx][i]));
    }
}

// The plan of a tf32 launch (see PlanSpec): 128-row query tiles, 64-key
// tiles, one query tile per cost unit.
PlanSpec tf32_plan_spec(const AttnProblem &p, bool pair) {
    PlanSpec s{};
    s.q_pos = p.q_pos;
    s.k_pos = p.k_pos;
    s.q_pos_stride = p.q_pos_stride;
    s.k_pos_stride = p.k_pos_stride;
    s.C = p.C;
    s.kpr = (p.k_pos_stride == 0) ? 1 : p.C;
    s.kpos_shift = p.kpos_shift;
    s.Sq = static_cast<int>(p.Sq);
    s.Sk = static_cast<int>(p.Sk);
    s.q_tile = 128;
    s.k_tile = 64;
    s.unit_is_k = 0;
    s.q_group = 1;
    s.pair = pair ? 1 : 0;
    return s;
}

bool tf32_plan_on_chip(int64_t C, int64_t kpr, int64_t Sq, int64_t Sk) {
    const int64_t nqt = (Sq + 127) / 128, nkt = (Sk + 63) / 64;
    return kpr * nkt + C * nqt <= kMaxTables && C * nqt <= kMaxPairs;
}

template <int D, bool kGP>
cp_status launch_tf32_typed(const AttnProblem &p, const float *vt, int64_t sk_pad, cudaStream_t stream) {
    using K = CfgT<D>;
    CUtensorMap mq, mk, mv;
    const int64_t kv_outer = p.kv_shared ? p.B : p.C * p.B;
    // q [C*B][Sq][N][D] and k [outer][Sk][Nkv][D]: boxes of 32 columns x 128 (64) rows;
    // vt [outer][Nkv][D][sk_pad]: boxes of 32 keys x D rows
    if (!make_map_f32_4d(&mq, static_cast<const float *>(p.q), D, p.N, p.Sq, p.C * p.B, 32, 1, 128) ||
        !make_map_f32_4d(&mk, static_cast<const float *>(p.k), D, p.Nkv, p.Sk, kv_outer, 32, 1, 64) ||
        !make_map_f32_4d(&mv, vt, sk_pad, D, p.Nkv, kv_outer, 32, D, 1))
        return CP_ERR_CUDA;
    TArgs a;
    a.q_pos = p.q_pos;
    a.k_pos = p.k_pos;
    a.q_pos_stride = p.q_pos_stride;
    a.k_pos_stride = p.k_pos_stride;
    a.o = p.o;
    a.lse = p.lse;
    a.C = p.C;
    a.B = static_cast<int>(p.B);
    a.N = static_cast<int>(p.N);
    a.Nkv = static_cast<int>(p.Nkv);
    a.Sq = static_cast<int>(p.Sq);
    a.Sk = static_cast<int>(p.Sk);
    a.nqt = static_cast<int>((p.Sq + 127) / 128);
    a.nkt = static_cast<int>((p.Sk + 63) / 64);
    a.kv_shift = p.kv_shift;
    a.kpos_shift = p.kpos_shift;
    a.kv_shared = p.kv_shared ? 1 : 0;
    a.kpr = (p.k_pos_stride == 0) ? 1 : p.C;
    a.scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634074);
    a.timeout_ns = p.timeout_ns ? p.timeout_ns : 2000000000ull;
    a.hold = p.hold;
    // query tiles u and nqt-1-u in one work item when that still leaves 8 rounds
    a.pair = pair_units(a.nqt, p.C, p.B * p.N, sm_count()) ? 1 : 0;
    a.div_nsp = make_fastdiv(static_cast<uint32_t>(super_count(a.nqt, a.pair != 0)));
    a.div_n = make_fastdiv(static_cast<uint32_t>(a.N));
    const long long n_items = static_cast<long long>(p.C) * super_count(a.nqt, a.pair != 0) * p.B * p.N;
    a.gp = PlanPtrs{};
    if (kGP) {
        const cp_status st = launch_plan(tf32_plan_spec(p, a.pair != 0), p.plan, &a.gp, stream);
        if (st != CP_OK) return st;
    }
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_tf32_kernel<D, kGP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        K::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return cuda_status(attr_err);
    const int grid = static_cast<int>(n_items < sm_count() ? n_items : sm_count());
    attn_tf32_kernel<D, kGP><<<grid, kTThreads, K::kSmemBytes, stream>>>(mq, mk, mv, a);
    return last_launch_status();
}

}  // namespace

size_t tf32_plan_need(int64_t C, int64_t kpr, int64_t Sq, int64_t Sk) {
    if (tf32_plan_on_chip(C, kpr, Sq, Sk)) return 0;
    AttnProblem p{};
    p.C = static_cast<int>(C);
    p.k_pos_stride = (kpr == 1) ? 0 : 1;
    p.Sq = Sq;
    p.Sk = Sk;
    return plan_bytes(tf32_plan_spec(p, false));  // unpaired: the longer order
}

cp_status validate_attn_tf32(const AttnProblem &p, bool check_plan) {
    if (!p.q || !p.k || !p.v || !p.q_pos || !p.k_pos || !p.o || !p.lse) return CP_ERR_NULL;
    if (p.C < 1 || p.C > kMaxC || p.B < 1 || p.N < 1 || p.Nkv < 1 || p.Sq < 1 || p.Sk < 1) return CP_ERR_SHAPE;
    if (p.D != 64 && p.D != 128) return CP_ERR_UNSUPPORTED;
    if (p.N % p.Nkv != 0) return CP_ERR_DIVISIBILITY;
    if (!(std::isfinite(p.scale) && p.scale > 0.f)) return CP_ERR_ARGUMENT;
    if (p.merge_into) return CP_ERR_UNSUPPORTED;
    if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !aligned16(p.q_pos) || !aligned16(p.k_pos) ||
        !aligned16(p.lse))
        return CP_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(p.o) & 31u) return CP_ERR_ALIGNMENT;
    const int64_t nqt = (p.Sq + 127) / 128, nkt = (p.Sk + 63) / 64;
    const int64_t kpr = (p.k_pos_stride == 0) ? 1 : p.C;
    if (p.Sq > INT32_MAX / 2 || p.Sk > INT32_MAX / 2 || static_cast<int64_t>(p.C) * nqt * p.B * p.N > INT32_MAX ||
        kpr * nkt + p.C * nqt > INT32_MAX / 8)
        return CP_ERR_SHAPE;
    if (check_plan && !tf32_plan_on_chip(p.C, kpr, p.Sq, p.Sk)) {
        if (!p.plan || p.plan_bytes < tf32_plan_need(p.C, kpr, p.Sq, p.Sk)) return CP_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(p.plan) & 255u) return CP_ERR_ALIGNMENT;
    }
    if (p.kv_shift < 0 || p.kv_shift >= p.C || p.kpos_shift < 0 || p.kpos_shift >= p.C) return CP_ERR_ARGUMENT;
    return CP_OK;
}

int64_t tf32_vt_pad(int64_t Sk) { return (Sk + 63) / 64 * 64; }

size_t tf32_vt_bytes(int64_t outer, int64_t Sk, int64_t Nkv, int64_t D) {
    return static_cast<size_t>(outer) * Nkv * D * tf32_vt_pad(Sk) * sizeof(float);
}

cp_status launch_tf32_transpose(const float *v, float *vt, int64_t outer, int64_t Sk, int64_t Nkv, int64_t D,
                                cudaStream_t stream) {
    if (!v || !vt) return CP_ERR_NULL;
    const int64_t pad = tf32_vt_pad(Sk);
    if (outer * Nkv > 65535 || D % 32 != 0) return CP_ERR_SHAPE;
    const dim3 grid(static_cast<unsigned>(pad / 32), static_cast<unsigned>(D / 32), static_cast<unsigned>(outer * Nkv));
    tf32_transpose_kernel<<<grid, 256, 0, stream>>>(v, vt, outer, static_cast<int>(Sk), static_cast<int>(Nkv),
                                                    static_cast<int>(D), static_cast<int>(pad));
    return last_launch_status();
}

cp_status launch_tf32_round(const float *in, float *out, int64_t n, cudaStream_t stream) {
    if (!in || !out) return CP_ERR_NULL;
    if (n % 4 != 0 || !aligned16(in) || !aligned16(out)) return CP_ERR_ALIGNMENT;
    const long long n4 = n / 4;
    if (n4 == 0) return CP_OK;
    long long blocks = (n4 + 255) / 256;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    tf32_round_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(reinterpret_cast<const float4 *>(in),
                                                                          reinterpret_cast<float4 *>(out), n4);
    return last_launch_status();
}

cp_status launch_attn_tf32(const AttnProblem &p, const float *vt, cudaStream_t stream) {
    cp_status st = validate_attn_tf32(p);
    if (st != CP_OK) return st;
    if (!vt || !aligned16(vt)) return CP_ERR_ALIGNMENT;
    const int64_t pad = tf32_vt_pad(p.Sk);
    if (tf32_plan_on_chip(p.C, (p.k_pos_stride == 0) ? 1 : p.C, p.Sq, p.Sk))
        return p.D == 128 ? launch_tf32_typed<128, false>(p, vt, pad, stream)
                          : launch_tf32_typed<64, false>(p, vt, pad, stream);
    return p.D == 128 ? launch_tf32_typed<128, true>(p, vt, pad, stream) : launch_tf32_typed<64, true>(p, vt, pad, stream);
}

cp_status read_tf32_device_status(int *code, bool clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_cp_device_status_tf32, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
    *code = v;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_cp_device_status_tf32, &zero, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
    }
    return CP_OK;
}

}  // namespace cpattn

namespace {
inline size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace of cp_attn_partial_f32: q and k rounded to tf32, v transposed
// (and rounded), then the work plan when it does not fit on chip.
struct F32Layout {
    size_t qr, kr, vt, plan, plan_bytes, total;
};
F32Layout f32_layout(int64_t B, int64_t Sq, int64_t Sk, int64_t N, int64_t Nkv, int64_t D) {
    F32Layout L;
    L.qr = 0;
    L.kr = round256(static_cast<size_t>(B) * Sq * N * D * 4);
    L.vt = L.kr + round256(static_cast<size_t>(B) * Sk * Nkv * D * 4);
    L.plan = L.vt + round256(cpattn::tf32_vt_bytes(B, Sk, Nkv, D));
    L.plan_bytes = cpattn::tf32_plan_need(1, 1, Sq, Sk);
    L.total = L.plan + round256(L.plan_bytes);
    return L;
}
}  // namespace

extern "C" cp_status cp_attn_f32_workspace_size(int64_t B, int64_t Sq, int64_t Sk, int64_t N, int64_t Nkv,
                                                int64_t D, size_t *bytes) {
    if (!bytes) return CP_ERR_NULL;
    if (B < 1 || Sq < 1 || Sk < 1 || N < 1 || Nkv < 1 || D < 1) return CP_ERR_SHAPE;
    *bytes = f32_layout(B, Sq, Sk, N, Nkv, D).total;
    return CP_OK;
}

extern "C" cp_status cp_attn_partial_f32(const float *q, const float *k, const float *v, const int32_t *q_pos,
                                         const int32_t *k_pos, int64_t B, int64_t Sq, int64_t Sk, int64_t N,
                                         int64_t Nkv, int64_t D, float scale, float *o, float *lse,
                                         void *workspace, size_t ws_bytes, cudaStream_t stream) {
    cpattn::AttnProblem p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.q_pos = q_pos;
    p.k_pos = k_pos;
    p.o = o;
    p.lse = lse;
    p.C = 1;
    p.B = B;
    p.N = N;
    p.Nkv = Nkv;
    p.D = D;
    p.Sq = Sq;
    p.Sk = Sk;
    p.scale = scale;
    cp_status st = cpattn::validate_attn_tf32(p, false);
    if (st != CP_OK) return st;
    const F32Layout L = f32_layout(B, Sq, Sk, N, Nkv, D);
    if (!workspace || ws_bytes < L.total) return CP_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return CP_ERR_ALIGNMENT;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *qr = reinterpret_cast<float *>(ws + L.qr), *kr = reinterpret_cast<float *>(ws + L.kr);
    float *vt = reinterpret_cast<float *>(ws + L.vt);
    p.q = qr;
    p.k = kr;
    if (L.plan_bytes) {
        p.plan = ws + L.plan;
        p.plan_bytes = L.plan_bytes;
    }
    st = cpattn::launch_tf32_round(q, qr, B * Sq * N * D, stream);
    if (st == CP_OK) st = cpattn::launch_tf32_round(k, kr, B * Sk * Nkv * D, stream);
    if (st == CP_OK) st = cpattn::launch_tf32_transpose(v, vt, B, Sk, Nkv, D, stream);
    if (st == CP_OK) st = cpattn::launch_attn_tf32(p, vt, stream);
    return st;
}
