// cp_internal.h -- host-side declarations shared by the translation units of
// libcpattn (validation helpers and internal launchers).  Not installed.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

#include "../../include/cpattn.h"

namespace cpattn {

constexpr int kTileM = 128;          // query rows per tile
constexpr int kTileN = 128;          // keys per tile
constexpr int kMaxTables = 2048;     // C * (ceil(Sq/128) + ceil(Sk/128)) limit
constexpr int kMaxPairs = 1024;      // C * ceil(Sq/256) limit
constexpr int kMaxC = 64;            // virtual ranks per launch

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t dtype_size(cp_dtype d) { return d == CP_BF16 ? 2 : (d == CP_F32 ? 4 : 0); }

// Remembers the most recent CUDA error seen by this host thread (for
// cp_last_cuda_error) and maps it to a status.
void note_cuda_error(cudaError_t e);
inline cp_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return CP_OK;
    note_cuda_error(e);
    return CP_ERR_CUDA;
}

// Reads and clears the sticky launch error of this thread.
inline cp_status last_launch_status() { return cuda_status(cudaGetLastError()); }

// Number of SMs of the current device (cached per device).
int sm_count();

// One batched attention launch over C "rank" problems.  Rank r reads its
// queries from q[r] (rank stride C-major: [C][B][Sq][N][D]), its K/V from rank
// (r + kv_shift) mod C of k/v ([C][B][Sk][Nkv][D]) -- or, with kv_shared, from
// the one K/V tensor [B][Sk][Nkv][D] all ranks share -- its query positions
// from q_pos + r*q_pos_stride and its key positions from
// k_pos + ((r + kpos_shift) mod C)*k_pos_stride (k_pos_stride 0: one shared
// key-position array).
struct AttnProblem {
    const void *q, *k, *v;
    const int32_t *q_pos, *k_pos;
    int64_t q_pos_stride, k_pos_stride;
    float *o, *lse;               // o [C][B][Sq][N][D] fp32, lse [C][B][N][Sq]
    int C;
    int64_t B, N, Nkv, D, Sq, Sk;
    int kv_shift, kpos_shift;
    bool kv_shared;
    // merge_into: o/lse hold an accumulator (o [C][B][Sq][N][D], lse
    // [C][B][N][Sq]); the partial is LSE-merged into it instead of written
    // (rows the partial cannot see are left untouched)
    bool merge_into;
    float scale;
    // failure injection (self-test only): the producer first waits for *hold
    // to become non-zero; every bounded wait uses timeout_ns (0: 2 s)
    const int *hold = nullptr;
    unsigned long long timeout_ns = 0;
    // device buffer for the launch's work plan when it does not fit in shared
    // memory (attn_plan_need bytes, 256-byte aligned); unused otherwise
    void *plan = nullptr;
    size_t plan_bytes = 0;
};

// ------------------------------------------------------------ work plans
// A persistent attention kernel starts from a plan of its launch: the
// (min, max) position of every query and key tile, a bit per tile saying its
// positions are consecutive, a "sorted" flag per rank (tile minima (K) or
// maxima (Q) non-decreasing), the streamed-tile count of every (rank,
// stationary unit), and the longest-first order of super-blocks cut into
// segments (cp_sched.cuh).  When the plan fits in shared memory every CTA
// builds it there; otherwise a pre-pass (launch_plan) writes it into the
// caller's workspace and the kernel reads it from global memory.
struct PlanPtrs {
    const int2 *ktab, *qtab;         // [kpr][nkt], [C][nqt]
    const uint32_t *kbits, *qbits;   // consecutive-positions bits of K / Q tiles
    const int *ksorted, *qsorted;    // [kpr] (K minima non-decreasing), [C] (Q maxima)
    const int *cost;                 // [C][nunits]
    const int *order, *seg_first;    // [C*nsp], [C*nsp + 1]
};

// What the plan of one launch covers.  Units: groups of `q_group` query tiles
// (cost = key tiles of the owner with min position <= the group's max query
// position), or with unit_is_k the key tiles of the owner (cost = query tiles
// of the rank with max position >= the tile's min key position).
struct PlanSpec {
    const int32_t *q_pos, *k_pos;
    long long q_pos_stride, k_pos_stride;
    int C, kpr, kpos_shift;
    int Sq, Sk;
    int q_tile, k_tile;  // rows per table entry (128; key tiles 128 or 64)
    int unit_is_k, q_group, pair;
};

// Bytes of the global plan of `s` (256-byte multiple).
size_t plan_bytes(const PlanSpec &s);
// Enqueue the plan pre-pass into buf (>= plan_bytes(s), 256-byte aligned);
// *out receives the device pointers the kernel reads.
cp_status launch_plan(const PlanSpec &s, void *buf, PlanPtrs *out, cudaStream_t stream);

// Bytes of plan buffer the forward kernel needs for C query ranks of Sq rows
// against kpr key-position ranks of Sk rows (0 when the plan fits on chip).
size_t attn_plan_need(int64_t C, int64_t kpr, int64_t Sq, int64_t Sk);

// Host validation shared by cp_attn_partial and the ring.  With check_plan,
// a problem whose plan does not fit on chip must come with a plan buffer
// (else CP_ERR_WORKSPACE).
cp_status validate_attn(const AttnProblem &p, bool check_plan = true);
// Validate then enqueue the attention kernel on `stream`.
cp_status launch_attn(const AttnProblem &p, cudaStream_t stream);

// The checks of a ring forward call that do not involve its workspace
// (pointers, enums, flags, shapes, divisibility, the attention problem).
cp_status ring_check_args(const void *q_sh, const void *k_sh, const void *v_sh, const int32_t *pos, int64_t B,
                          int64_t S, int64_t N, int64_t Nkv, int64_t D, int C, float scale, cp_layout layout,
                          int flags, const void *o_sh, cp_dtype o_dtype, const float *lse_sh);

// In-place LSE merge over `rows` rows of D fp32 values laid out as
// o [B][Sq][N][D], lse [B][N][Sq] (B may fold the rank dimension).
cp_status launch_merge(float *o_acc, float *lse_acc, const float *o_tile, const float *lse_tile, int64_t B,
                       int64_t Sq, int64_t N, int64_t D, cudaStream_t stream);

// fp32 -> bf16 (round to nearest even), n elements, n % 8 == 0.
cp_status launch_f32_to_bf16(const float *in, void *out, int64_t n, cudaStream_t stream);

// cp_ulysses_relayout applied to `groups` independent blocks laid out one
// after another (same byte offset of each block on both sides); one launch.
cp_status ulysses_relayout_groups(const void *in, void *out, int64_t B, int64_t S, int64_t N, int64_t D, int C,
                                  int groups, cp_dtype dtype, cp_dir dir, cp_seq_order order, cudaStream_t stream);

// TMA descriptors.  make_map: 4-D bf16 map over [outer][rows][heads][D],
// box 64 columns x 1 head x box_rows rows x 1, 128-byte swizzle.
// make_map_f32_rows: 2-D fp32 map over [rows][cols], box box_cols x 1.
bool make_map(CUtensorMap *map, const void *base, int64_t D, int64_t heads, int64_t rows, int64_t outer,
              int box_rows);
bool make_map_f32_rows(CUtensorMap *map, const float *base, int64_t cols, int64_t rows, int box_cols);
// 4-D fp32 map over [d3][d2][d1][d0] (d0 innermost), box b0 x b1 x b2 x 1,
// 128-byte swizzle.
bool make_map_f32_4d(CUtensorMap *map, const float *base, int64_t d0, int64_t d1, int64_t d2, int64_t d3, int b0,
                     int b1, int b2);

// ------------------------------------------------------------ tf32 path
// The attention of launch_attn for fp32 q, k, v (tensor cores in tf32); vt is
// v transposed by launch_tf32_transpose ([outer][Nkv][D][tf32_vt_pad(Sk)]).
cp_status validate_attn_tf32(const AttnProblem &p, bool check_plan = true);
// Plan bytes of the tf32 kernel (as attn_plan_need; 64-key tiles).
size_t tf32_plan_need(int64_t C, int64_t kpr, int64_t Sq, int64_t Sk);
cp_status launch_attn_tf32(const AttnProblem &p, const float *vt, cudaStream_t stream);
int64_t tf32_vt_pad(int64_t Sk);
size_t tf32_vt_bytes(int64_t outer, int64_t Sk, int64_t Nkv, int64_t D);
cp_status launch_tf32_transpose(const float *v, float *vt, int64_t outer, int64_t Sk, int64_t Nkv, int64_t D,
                                cudaStream_t stream);
// out = in rounded to the nearest tf32 value, n elements (n % 4 == 0, both 16-byte aligned).
cp_status launch_tf32_round(const float *in, float *out, int64_t n, cudaStream_t stream);
cp_status read_tf32_device_status(int *code, bool clear);

// ------------------------------------------------------------ backward
constexpr int kBwdMaxTables = 2048;  // 128-row position tables of one backward launch
constexpr int kBwdMaxPairs = 1024;   // (rank, stationary tile) pairs of one backward launch

// One batched backward launch over C "rank" problems (the tile backward of
// each rank's queries against the K/V of rank (r + kv_shift) mod C), with the
// same rank conventions as AttnProblem.  dout is bf16 like q; o fp32 (the
// final output, [C][B][Sq][N][D]); lse the final log-sum-exp [C][B][N][Sq].
// nl2 / nd: per-row statistics from launch_bwd_stats ([C][B][N][sq_pad]).
// dq [C][B][Sq][N][D]; dk, dv [C][B][Sk][Nkv][D] indexed by the K/V rank;
// accumulate: add to them instead of overwriting.
struct BwdProblem {
    const void *q, *k, *v, *dout;
    const int32_t *q_pos, *k_pos;
    int64_t q_pos_stride, k_pos_stride;
    const float *nl2, *nd;
    int64_t sq_pad;
    float *dq, *dk, *dv;
    int C;
    int64_t B, N, Nkv, D, Sq, Sk;
    int kv_shift, kpos_shift;
    bool accumulate;
    float scale;
    // device buffer for the work plans when they do not fit in shared memory
    // (bwd_plan_need bytes, 256-byte aligned; the dK/dV and dQ launches use it
    // one after the other); unused otherwise
    void *plan = nullptr;
    size_t plan_bytes = 0;
    // failure injection (self-test only): both producers first wait for *hold
    // to become non-zero; every bounded wait uses timeout_ns (0: 2 s)
    const int *hold = nullptr;
    unsigned long long timeout_ns = 0;
};
// Rows of the per-row statistics (a multiple of 128 >= Sq).
inline int64_t bwd_sq_pad(int64_t Sq) { return (Sq + 127) / 128 * 128; }
// nl2[r][i] = -lse * log2(e) (-inf where lse = -inf or i >= Sq) and
// nd[r][i] = -<dO_i, o_i> (0 for i >= Sq), rows r over C*B*N.
cp_status launch_bwd_stats(const float *o, const void *dout, const float *lse, int64_t CB, int64_t Sq, int64_t N,
                           int64_t D, int64_t sq_pad, float *nl2, float *nd, cudaStream_t stream);
cp_status validate_bwd(const BwdProblem &p, bool check_plan = true);
// Plan bytes of the two backward kernels for C query ranks of Sq rows against
// kpr key-position ranks of Sk rows (0 when both plans fit on chip).
size_t bwd_plan_need(int64_t C, int64_t kpr, int64_t Sq, int64_t Sk);
// dK / dV launch then dQ launch (both validated first).
cp_status launch_bwd(const BwdProblem &p, cudaStream_t stream);
// Sticky device status word of the backward kernels (read and optionally cleared).
cp_status read_bwd_device_status(int *code, bool clear);

}  // namespace cpattn
