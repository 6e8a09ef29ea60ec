/*
 * cpattn.h -- C ABI of libcpattn: blockwise causal attention with
 * log-sum-exp merging for ring / zigzag context parallelism, for C virtual
 * ranks held as buffers on ONE GB300 GPU (sm_103a).
 *
 * Source pages (cited by title and section):
 *   [OCP]   "On Context Parallelism": All-gather, All-to-all, Peer-to-peer
 *   [DAY74] "Context parallelism -- splitting the sequence across GPUs"
 *   [RING]  "Context Parallelism & Ring Attention"
 *   [HB]    "Context parallelism: Ring Attention and Ulysses"
 *   [APPF]  "Appendix F: Context Parallelism and MoE Parallel Folding"
 *
 * General conventions (all entry points):
 *   - Device pointers are raw CUDA device addresses owned by the caller; the
 *     library never allocates device memory on these paths and never frees
 *     caller memory.  Work that needs scratch takes a caller workspace.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) unless
 *     stated otherwise; they return as soon as the work is enqueued.
 *   - Arguments are validated on the host BEFORE anything is enqueued; on a
 *     validation error nothing is launched and the call returns the status.
 *     No call aborts, throws or prints.
 *   - Tensors are dense, row-major, with the layouts given per call:
 *       sequence-sharded, rank-major: X_sh [C][B][s][N][D], s = S/C
 *       lse: [B][N][Sq] (rank-major shards: [C][B][N][s])
 *     ([OCP] Peer-to-peer / Forward: output [B,S/C,N,D], lse [B,N,S/C].)
 *   - Every device pointer must be 16-byte aligned; rows of N*D elements
 *     must be a multiple of 16 bytes.
 *   - Failures of a launch are reported as CP_ERR_CUDA (cudaGetLastError is
 *     read and cleared).  A kernel that gives up a bounded device-side wait
 *     records CP_ERR_DEVICE_TIMEOUT in a device status word, readable with
 *     cp_device_status().
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cp_status {
    CP_OK = 0,
    CP_ERR_NULL = 1,          /* a required pointer is NULL */
    CP_ERR_SHAPE = 2,         /* a size is <= 0 or out of the supported range */
    CP_ERR_DIVISIBILITY = 3,  /* S % 2C (zigzag), S % C, N % C, Nkv % C or N % Nkv */
    CP_ERR_DTYPE = 4,         /* unknown cp_dtype */
    CP_ERR_ALIGNMENT = 5,     /* pointer or row not 16-byte aligned */
    CP_ERR_WORKSPACE = 6,     /* workspace NULL or smaller than cp_ring_workspace_size */
    CP_ERR_UNSUPPORTED = 7,   /* e.g. D not in {64, 128} for attention */
    CP_ERR_CUDA = 8,          /* a CUDA runtime call or launch failed */
    CP_ERR_DEVICE_TIMEOUT = 9,/* a kernel gave up a bounded wait (see cp_device_status) */
    CP_ERR_ARGUMENT = 10      /* any other invalid argument (scale, enum, event count) */
} cp_status;

typedef enum cp_dtype { CP_BF16 = 0, CP_F32 = 1 } cp_dtype;
typedef enum cp_layout { CP_ZIGZAG = 0, CP_CONTIGUOUS = 1 } cp_layout;
typedef enum cp_dir { CP_SEQ_TO_HEAD = 0, CP_HEAD_TO_SEQ = 1 } cp_dir;
typedef enum cp_seq_order { CP_RANK_ORDER = 0, CP_GLOBAL_ORDER = 1 } cp_seq_order;

/* Human-readable name of a status code (static string, never NULL). */
const char *cp_status_string(cp_status status);

/* Library version as "major.minor.patch" (static string). */
const char *cp_version(void);

/* Text of the most recent CUDA runtime error that made a call of this host
 * thread return CP_ERR_CUDA ("no error" if none); static string. */
const char *cp_last_cuda_error(void);

/*
 * cp_zigzag_shard -- split a full sequence into C rank-major shards.
 * [OCP] All-gather: S is cut into 2C chunks of t = S/(2C) tokens and rank r
 * owns [chunk r | chunk 2C-1-r] (layout CP_ZIGZAG; TE's "DualChunkSwap").
 * [RING] "The last remaining axis": rank r owns tokens [r*s, (r+1)*s)
 * (layout CP_CONTIGUOUS).
 *   x     : [B][S][N][D] of `dtype`, read only; memory of the current device, or pinned host
 *           memory mapped at the same address (cudaHostAlloc / cudaMallocHost /
 *           cudaHostRegister under unified addressing), which the kernel then
 *           reads across the host link (the host-to-device copy and the shard
 *           in one pass)
 *   x_sh  : device, [C][B][S/C][N][D] of `dtype`, written (must not overlap x)
 * Requires S % (2C) == 0 (zigzag) or S % C == 0 (contiguous), C >= 1.
 * Any other host memory (pageable, or pinned but not mapped at its host
 * address) is refused with CP_ERR_ARGUMENT before anything is launched.
 * The result is a bit-exact permutation of x.
 */
cp_status cp_zigzag_shard(const void *x, void *x_sh, int64_t B, int64_t S, int64_t N, int64_t D,
                          int C, cp_dtype dtype, cp_layout layout, cudaStream_t stream);

/*
 * cp_zigzag_unshard -- inverse of cp_zigzag_shard: gather the C shards back
 * into global sequence order ([OCP] All-gather: the rank-order result
 * [chunk 0, chunk 7, chunk 1, chunk 6, ...] reordered to sequence order).
 *   x_sh  : device, [C][B][S/C][N][D], read only
 *   x     : [B][S][N][D], written (must not overlap x_sh); current-device memory, or
 *           pinned host memory mapped at the same address (the kernel then
 *           writes across the host link: unshard and device-to-host copy in
 *           one pass); other host memory -> CP_ERR_ARGUMENT
 */
cp_status cp_zigzag_unshard(const void *x_sh, void *x, int64_t B, int64_t S, int64_t N, int64_t D,
                            int C, cp_dtype dtype, cp_layout layout, cudaStream_t stream);

/*
 * cp_zigzag_positions -- global position of every local token, int32 [C][S/C]:
 * zigzag: pos[r] = [r*t .. r*t+t-1] ++ [(2C-1-r)*t .. (2C-1-r)*t+t-1]
 * ([OCP] All-gather ownership; the ring's per-owner positions in
 * Peer-to-peer / Forward); contiguous: pos[r] = [r*s .. r*s+s-1].
 *   pos       : device (on_device != 0, written by a kernel on `stream`) or
 *               host (on_device == 0, written synchronously; stream unused)
 * Requires S <= INT32_MAX.
 */
cp_status cp_zigzag_positions(int32_t *pos, int64_t S, int C, cp_layout layout, int on_device,
                              cudaStream_t stream);

/*
 * cp_ulysses_relayout -- the Ulysses all-to-all as a local permutation of
 * rank-major buffers ([HB] "Ulysses" seq_to_head / head_to_seq; [OCP]
 * All-to-all; [APPF] eq. (96) [B,S/C,H,d_h] -> [B,S,H/C,d_h]).
 *   CP_SEQ_TO_HEAD: in [C][B][S/C][N][D] -> out [C][B][S][N/C][D] with
 *       out[r][b][j*s+u][h'][d] = in[j][b][u][r*N/C + h'][d]
 *     (rank r receives head group r from every shard, shards in rank order).
 *   CP_HEAD_TO_SEQ: the exact inverse (out and in swap roles).
 *   CP_GLOBAL_ORDER additionally puts the gathered sequence in global order
 *     (row j*s+u -> zigzag position of row u of rank j; [OCP] All-to-all:
 *     TE reorders the chunks into global order before attention).  Requires
 *     S % (2C) == 0.  CP_RANK_ORDER is the literal all-to-all.
 * Requires S % C == 0 and N % C == 0 (head divisibility, [OCP] All-to-all;
 * [HB] "Ulysses").  in and out must not overlap.  Bit-exact permutation.
 */
cp_status cp_ulysses_relayout(const void *in, void *out, int64_t B, int64_t S, int64_t N, int64_t D,
                              int C, cp_dtype dtype, cp_dir dir, cp_seq_order order,
                              cudaStream_t stream);

/*
 * cp_attn_partial -- partial causal attention with explicit positions,
 * returning the normalised output and the per-row log-sum-exp.
 * [OCP] Peer-to-peer / Forward (attention(q, k, v, q_positions,
 * kv_positions, scale) -> tile_output, tile_lse); [HB] cp_common.py;
 * [DAY74] the causal softmax formula.  For each (b, h, i):
 *   visible keys V(i) = { j : k_pos[j] <= q_pos[i] }
 *   s_j = scale * <q_i, k_j>,  lse_i = ln sum_{j in V(i)} e^{s_j}
 *   o_i = sum_{j in V(i)} e^{s_j - lse_i} v_j
 *   a row with no visible key gets lse = -inf and o = 0.
 *   q      : device bf16 [B][Sq][N][D]
 *   k, v   : device bf16 [B][Sk][Nkv][D]; query head h reads KV head h/(N/Nkv)
 *   q_pos  : device int32 [Sq];  k_pos : device int32 [Sk] (any values)
 *   o      : device fp32 [B][Sq][N][D], written; 32-byte aligned
 *   lse    : device fp32 [B][N][Sq], written (natural log)
 * Requires D in {64, 128}, N % Nkv == 0, scale finite and > 0.  Runs on the
 * tensor cores (bf16 products, fp32 accumulation and softmax).
 * Work plan: the kernel starts from a plan of its launch (per-tile position
 * ranges, per-block tile counts, the order of work items).  It is built in
 * shared memory when ceil(Sq/128) + ceil(Sk/128) <= 2048 and
 * ceil(Sq/256) <= 1024; beyond that it is built in device memory the caller
 * provides: call cp_attn_partial_ws with a workspace of
 * cp_attn_workspace_size bytes (cp_attn_partial then returns
 * CP_ERR_WORKSPACE).
 */
cp_status cp_attn_partial(const void *q, const void *k, const void *v, const int32_t *q_pos,
                          const int32_t *k_pos, int64_t B, int64_t Sq, int64_t Sk, int64_t N,
                          int64_t Nkv, int64_t D, float scale, float *o, float *lse,
                          cudaStream_t stream);

/*
 * cp_attn_workspace_size / cp_attn_partial_ws -- cp_attn_partial with a
 * caller workspace for the work plan, for any sequence length.
 *   *bytes receives the workspace size for these sizes (0 when the plan fits
 *   in shared memory; then workspace may be NULL).  Host only.
 *   workspace : device, >= cp_attn_workspace_size bytes, 256-byte aligned;
 *               overwritten by the call (stream-ordered), not read back.
 * Everything else as cp_attn_partial.
 */
cp_status cp_attn_workspace_size(int64_t B, int64_t Sq, int64_t Sk, int64_t N, int64_t Nkv, int64_t D,
                                 size_t *bytes);
cp_status cp_attn_partial_ws(const void *q, const void *k, const void *v, const int32_t *q_pos,
                             const int32_t *k_pos, int64_t B, int64_t Sq, int64_t Sk, int64_t N,
                             int64_t Nkv, int64_t D, float scale, float *o, float *lse, void *workspace,
                             size_t ws_bytes, cudaStream_t stream);

/*
 * cp_attn_f32_workspace_size / cp_attn_partial_f32 -- cp_attn_partial for fp32
 * inputs with the tensor cores in tf32 (tcgen05.mma kind::tf32, fp32
 * accumulation).  q, k, v and P are rounded to the nearest tf32 value (10-bit
 * mantissa, ties away from zero) before they enter the tensor cores: q and k
 * by a pass into the workspace, v in its transpose, P in the softmax.
 * Same arguments, result and conventions as cp_attn_partial except:
 *   q : device fp32 [B][Sq][N][D]; k, v : device fp32 [B][Sk][Nkv][D]
 *   workspace : device, >= cp_attn_f32_workspace_size(B, Sq, Sk, N, Nkv, D)
 *               bytes, 256-byte aligned (rounded q and k, v transposed for
 *               the K-major operand and, when ceil(Sk/64) + ceil(Sq/128) >
 *               2048 or ceil(Sq/128) > 1024, the launch's work plan)
 */
cp_status cp_attn_f32_workspace_size(int64_t B, int64_t Sq, int64_t Sk, int64_t N, int64_t Nkv, int64_t D,
                                     size_t *bytes);
cp_status cp_attn_partial_f32(const float *q, const float *k, const float *v, const int32_t *q_pos,
                              const int32_t *k_pos, int64_t B, int64_t Sq, int64_t Sk, int64_t N, int64_t Nkv,
                              int64_t D, float scale, float *o, float *lse, void *workspace, size_t ws_bytes,
                              cudaStream_t stream);

/*
 * cp_lse_merge -- merge a completed partial into an accumulator, in place.
 * [OCP] Peer-to-peer / Forward, the tile merge:
 *   lse = logaddexp(lse_acc, lse_tile)
 *   o   = e^{lse_acc - lse} * o_acc + e^{lse_tile - lse} * o_tile
 * ([HB] "Ring Attention" gives the same two formulas.)  A row whose
 * lse_tile is -inf is left untouched; a row whose lse_acc is -inf takes the
 * tile's values.
 *   o_acc, lse_acc   : device fp32 [B][Sq][N][D] / [B][N][Sq], read+written
 *   o_tile, lse_tile : device fp32, same shapes, read only
 */
cp_status cp_lse_merge(float *o_acc, float *lse_acc, const float *o_tile, const float *lse_tile,
                       int64_t B, int64_t Sq, int64_t N, int64_t D, cudaStream_t stream);

/* Ring options (bit set, argument `flags` of the ring calls). */
#define CP_RING_PREFETCH 1    /* emulate the ring exchange by side-stream K/V copies */
#define CP_RING_FUSED_MERGE 2 /* merge each step's partial in the attention epilogue */
#define CP_RING_TF32 4        /* fp32 q, k, v; tensor cores in tf32 (not with the other two flags) */

/*
 * cp_ring_workspace_size -- bytes of device workspace cp_ring_attention_fwd
 * needs for these sizes and flags: the per-step partial (fp32 o and lse for
 * all C ranks; not with CP_RING_FUSED_MERGE), an fp32 accumulator when o_dtype
 * is CP_BF16, with CP_RING_PREFETCH two K/V rotation buffers, and for long
 * shards (C * (ceil((S/C)/128) * 2) > 2048 position tables, or more than
 * 1024 query blocks in a step) the attention launches' work plan.  Host
 * only; *bytes is written on success.
 */
cp_status cp_ring_workspace_size(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int C,
                                 int flags, cp_dtype o_dtype, size_t *bytes);

/*
 * cp_ring_attention_fwd -- ring (P2P) context-parallel attention forward for
 * C virtual ranks resident on this GPU.  [OCP] Peer-to-peer / Forward;
 * [RING] "The ring"; [HB] "Ring Attention".  For step = 0 .. C-1 every rank
 * r attends its queries to the K/V block of owner (r - step) mod C (with
 * both sides' positions) and merges the partial into its running (o, lse);
 * step 0 writes the accumulator directly.  All C ranks of a step run in one
 * launch (zigzag makes their work equal, [RING] "The zigzag fix").
 *   q_sh          : device bf16 [C][B][S/C][N][D]
 *   k_sh, v_sh    : device bf16 [C][B][S/C][Nkv][D]
 *   pos           : device int32 [C][S/C] global positions (cp_zigzag_positions)
 *   layout        : selects the divisibility rule only (S % 2C for zigzag,
 *                   S % C for contiguous); masks come from `pos`
 *   flags         : bit set of
 *                   CP_RING_PREFETCH -- the ring exchange is emulated by
 *                     device copies of the next step's K/V on a second
 *                     stream, overlapped with the current step and ordered
 *                     by events (without it: zero copy, each step reads the
 *                     owner's resident block);
 *                   CP_RING_FUSED_MERGE -- steps >= 1 merge their partial
 *                     into (o, lse) inside the attention epilogue instead of
 *                     writing it and launching cp_lse_merge's kernel
 *   o_sh          : device [C][B][S/C][N][D] of o_dtype (CP_F32 or CP_BF16);
 *                   32-byte aligned when o_dtype is CP_F32
 *   lse_sh        : device fp32 [C][B][N][S/C]
 *   workspace     : device, >= cp_ring_workspace_size(...) bytes, 256-byte
 *                   aligned, caller-owned, contents need not be initialised
 * Same attention restrictions as cp_attn_partial.
 */
cp_status cp_ring_attention_fwd(const void *q_sh, const void *k_sh, const void *v_sh,
                                const int32_t *pos, int64_t B, int64_t S, int64_t N, int64_t Nkv,
                                int64_t D, int C, float scale, cp_layout layout, int flags,
                                void *o_sh, cp_dtype o_dtype, float *lse_sh, void *workspace,
                                size_t ws_bytes, cudaStream_t stream);

/*
 * cp_ring_attention_fwd_traced -- cp_ring_attention_fwd that also records
 * CUDA events on `stream` around every kernel it launches, for timing:
 *   events[4*step + 0], events[4*step + 1] : before / after the attention
 *                                            launch of `step`
 *   events[4*step + 2], events[4*step + 3] : before / after the merge launch
 *                                            of `step` (recorded back to
 *                                            back for step 0 and with
 *                                            CP_RING_FUSED_MERGE)
 * n_events must be >= 4*C; events are caller-created (cudaEventCreate).
 */
cp_status cp_ring_attention_fwd_traced(const void *q_sh, const void *k_sh, const void *v_sh,
                                       const int32_t *pos, int64_t B, int64_t S, int64_t N,
                                       int64_t Nkv, int64_t D, int C, float scale,
                                       cp_layout layout, int flags, void *o_sh,
                                       cp_dtype o_dtype, float *lse_sh, void *workspace,
                                       size_t ws_bytes, cudaStream_t stream,
                                       cudaEvent_t const *events, int n_events);

/*
 * cp_allgather_workspace_size / cp_allgather_attention_fwd -- all-gather
 * context-parallel attention forward for C virtual ranks on this GPU.
 * [OCP] All-gather / Forward: each rank keeps its local queries, K and V are
 * gathered from every rank and reordered to global sequence order, and each
 * rank's queries attend to the full sequence (query positions `pos`, key
 * positions 0..S-1).  Here the gather is cp_zigzag_unshard of the resident
 * shards into the workspace, and all C ranks share one launch.
 *   q_sh, k_sh, v_sh, pos, layout : as for cp_ring_attention_fwd
 *   o_sh   : device fp32 [C][B][S/C][N][D] (32-byte aligned), written
 *   lse_sh : device fp32 [C][B][N][S/C], written
 *   workspace : device, >= cp_allgather_workspace_size bytes (the gathered
 *               K and V, bf16 [B][S][Nkv][D] each, and S int32 positions),
 *               256-byte aligned
 * The result equals cp_ring_attention_fwd's (same partial kernel, one
 * partial instead of C merged ones).
 */
cp_status cp_allgather_workspace_size(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int C,
                                      size_t *bytes);
cp_status cp_allgather_attention_fwd(const void *q_sh, const void *k_sh, const void *v_sh,
                                     const int32_t *pos, int64_t B, int64_t S, int64_t N, int64_t Nkv,
                                     int64_t D, int C, float scale, cp_layout layout, float *o_sh,
                                     float *lse_sh, void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * cp_ulysses_workspace_size / cp_ulysses_attention_fwd -- all-to-all
 * (Ulysses) context-parallel attention forward for C virtual ranks.
 * [OCP] All-to-all; [HB] "Ulysses": q, k, v are relaid from sequence
 * sharding to head sharding (cp_ulysses_relayout, global sequence order),
 * each head-group rank computes causal attention over the whole sequence for
 * its N/C heads, and the output is relaid back to sequence sharding.
 *   q_sh : device bf16 [C][B][S/C][N][D]; k_sh, v_sh : [C][B][S/C][Nkv][D]
 *          (sharded with `layout`; N % C == 0 and Nkv % C == 0)
 *   o_sh : device fp32 [C][B][S/C][N][D], written
 *   lse_h: device fp32 [C][B][N/C][S], written: the log-sum-exp of head
 *          r*N/C + h' for global query position i is lse_h[r][b][h'][i]
 *          (head-sharded layout, global order, as the attention computes it)
 *   workspace : device, >= cp_ulysses_workspace_size bytes, 256-byte aligned
 */
cp_status cp_ulysses_workspace_size(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int C,
                                    size_t *bytes);
cp_status cp_ulysses_attention_fwd(const void *q_sh, const void *k_sh, const void *v_sh, int64_t B,
                                   int64_t S, int64_t N, int64_t Nkv, int64_t D, int C, float scale,
                                   cp_layout layout, float *o_sh, float *lse_h, void *workspace,
                                   size_t ws_bytes, cudaStream_t stream);

/*
 * cp_mesh_workspace_size / cp_mesh_attention_fwd -- A2A x P2P context-parallel
 * attention forward on a two-dimensional mesh of C = A * R virtual ranks.
 * [OCP] "Peer-to-peer + All-to-all": rank c belongs to A2A group c / A (ranks
 * g*A .. g*A+A-1) and to P2P group c % A (ranks a, A+a, 2A+a, ...).  Inside
 * each A2A group q, k, v go from sequence sharding to head sharding (N/A
 * heads; the group's A shards concatenated in rank order, S/R positions), each
 * P2P group runs the ring (as cp_ring_attention_fwd) over its R ranks with
 * those concatenated positions, and the output returns to sequence sharding.
 * A = 1 is the ring; R = 1 is Ulysses in rank order.
 *   q_sh : device bf16 [C][B][S/C][N][D]; k_sh, v_sh : [C][B][S/C][Nkv][D]
 *   pos  : device int32 [C][S/C], the global positions of each shard (for
 *          example cp_zigzag_positions with C and `layout`)
 *   A, R : A2A and P2P group sizes, 1 <= A*R <= 64; N % A == 0, Nkv % A == 0;
 *          S % (2C) == 0 for CP_ZIGZAG, S % C == 0 for CP_CONTIGUOUS
 *   flags: ring options (CP_RING_PREFETCH, CP_RING_FUSED_MERGE)
 *   o_sh : device fp32 [C][B][S/C][N][D], written
 *   lse_h: device fp32 [R][A][B][N/A][S/R], written: P2P rank g, A2A index a,
 *          head a*N/A + h', row a'*S/C + u = query u of shard g*A + a'
 *   workspace : device, >= cp_mesh_workspace_size bytes, 256-byte aligned
 *          (relaid q, k, v, the fp32 head-sharded output and the ring's own
 *          workspace)
 * Everything is validated before anything is enqueued.
 */
cp_status cp_mesh_workspace_size(int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int A, int R,
                                 int flags, size_t *bytes);
cp_status cp_mesh_attention_fwd(const void *q_sh, const void *k_sh, const void *v_sh, const int32_t *pos,
                                int64_t B, int64_t S, int64_t N, int64_t Nkv, int64_t D, int A, int R,
                                float scale, cp_layout layout, int flags, float *o_sh, float *lse_h,
                                void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * cp_attn_bwd_workspace_size / cp_attn_bwd_partial -- backward of one
 * partial attention ("tile backward"): [OCP] Peer-to-peer / Backward,
 * attention_tile_backward(q, k, v, output, grad_output, lse, q_positions,
 * kv_positions, scale) -> (dq, dk, dv).  It takes the FINAL output and lse of
 * the attention the tile belongs to, so p_ij = e^{scale <q_i,k_j> - lse_i}
 * over visible pairs (k_pos[j] <= q_pos[i]), and
 *   dv_j = sum_i p_ij dO_i,  ds_ij = p_ij (<dO_i, v_j> - <dO_i, o_i>),
 *   dq_i = scale sum_j ds_ij k_j,  dk_j = scale sum_i ds_ij q_i
 * (the chain rule of the forward; a KV head's gradients sum over its query
 * heads).  P and dS enter the tensor cores as bf16; accumulation is fp32.
 *   q, dout : device bf16 [B][Sq][N][D]; k, v : device bf16 [B][Sk][Nkv][D]
 *   o       : device fp32 [B][Sq][N][D], the final output
 *   lse     : device fp32 [B][N][Sq], the final natural-log log-sum-exp
 *             (-inf: the row sees nothing and contributes nothing)
 *   q_pos, k_pos : device int32 [Sq], [Sk]
 *   D in {64, 128}; N % Nkv == 0; scale finite and > 0
 *   dq : device fp32 [B][Sq][N][D]; dk, dv : device fp32 [B][Sk][Nkv][D];
 *        32-byte aligned; written, or added to when accumulate != 0
 *   workspace : device, >= cp_attn_bwd_workspace_size(B, Sq, Sk, N) bytes,
 *        256-byte aligned (per-row statistics and, when ceil(Sk/128) +
 *        ceil(Sq/128) > 2048 or either exceeds 1024, the kernels' work plans)
 * Other pointers 16-byte aligned.
 */
cp_status cp_attn_bwd_workspace_size(int64_t B, int64_t Sq, int64_t Sk, int64_t N, size_t *bytes);
cp_status cp_attn_bwd_partial(const void *q, const void *k, const void *v, const float *o, const void *dout,
                              const float *lse, const int32_t *q_pos, const int32_t *k_pos, int64_t B,
                              int64_t Sq, int64_t Sk, int64_t N, int64_t Nkv, int64_t D, float scale, float *dq,
                              float *dk, float *dv, int accumulate, void *workspace, size_t ws_bytes,
                              cudaStream_t stream);

/*
 * cp_ring_bwd_workspace_size / cp_ring_attention_bwd -- ring (P2P)
 * context-parallel attention backward for C virtual ranks.
 * [OCP] Peer-to-peer / Backward: at step = 0 .. C-1 rank r holds the K/V
 * block of owner (r - step) mod C and its travelling dK/dV accumulators; the
 * tile backward of rank r's queries against it (with rank r's final output
 * and lse from the forward) adds to rank r's dq and to the block's dk/dv,
 * which are back on their owner after the full rotation.  On one GPU the
 * travelling accumulators are the owners' own dk_sh / dv_sh; every step is one
 * dK/dV launch and one dQ launch over all C ranks.
 *   q_sh, do_sh : device bf16 [C][B][S/C][N][D]; k_sh, v_sh : [C][B][S/C][Nkv][D]
 *   o_sh  : device fp32 [C][B][S/C][N][D], lse_sh : fp32 [C][B][N][S/C]
 *           (cp_ring_attention_fwd's outputs with o_dtype CP_F32)
 *   pos   : device int32 [C][S/C]
 *   dq_sh : device fp32 [C][B][S/C][N][D]; dk_sh, dv_sh : [C][B][S/C][Nkv][D];
 *           written (32-byte aligned)
 *   workspace : device, >= cp_ring_bwd_workspace_size bytes, 256-byte aligned
 * Everything is validated before anything is enqueued.
 */
cp_status cp_ring_bwd_workspace_size(int64_t B, int64_t S, int64_t N, int C, size_t *bytes);
cp_status cp_ring_attention_bwd(const void *q_sh, const void *k_sh, const void *v_sh, const float *o_sh,
                                const float *lse_sh, const void *do_sh, const int32_t *pos, int64_t B, int64_t S,
                                int64_t N, int64_t Nkv, int64_t D, int C, float scale, cp_layout layout,
                                float *dq_sh, float *dk_sh, float *dv_sh, void *workspace, size_t ws_bytes,
                                cudaStream_t stream);

/*
 * cp_selftest_stalled_producer -- failure-detection self-test of the bounded
 * device-side waits (no counterpart on the pages).  Launches the attention
 * kernel on a [1][128][1][64] problem (q, k, v device bf16 [128][64], pos
 * device int32 [128], o fp32 [128][64] 32-byte aligned, lse fp32 [128]) with
 * its TMA producer held on a device flag that nothing sets and every bounded
 * wait limited to timeout_ns (1 ms .. 2 s, else CP_ERR_ARGUMENT).  The producer
 * gives up after timeout_ns, the other roles see the abort and unwind, TMEM
 * is freed, and the kernel records CP_ERR_DEVICE_TIMEOUT in the device status
 * word; o and lse are left unwritten.  The call itself returns CP_OK when the
 * launch succeeded: read the outcome with cp_device_status().  The context
 * stays usable.
 */
cp_status cp_selftest_stalled_producer(const void *q, const void *k, const void *v, const int32_t *pos, float *o,
                                       float *lse, uint64_t timeout_ns, cudaStream_t stream);

/*
 * cp_selftest_stalled_kernel -- the failure-detection self-test above for any
 * of the attention kernels (no counterpart on the pages): kernel 0 = bf16
 * forward, 1 = tf32 forward, 2 = backward (its dK/dV launch, then its dQ
 * launch).  The call zeroes `scratch` (device, 256-byte aligned, at least
 * CP_SELFTEST_SCRATCH_BYTES bytes), lays a tiny problem (one head, 128 rows,
 * D = 64) and the hold flag out in it, and launches the kernel with its TMA
 * producer held on the flag, which nothing sets, and every bounded wait limited
 * to timeout_ns (1 ms .. 2 s, else CP_ERR_ARGUMENT).  Each launch gives up
 * after timeout_ns and records CP_ERR_DEVICE_TIMEOUT in the device status word
 * (cp_device_status); the call returns CP_OK when the launches succeeded.  The
 * context stays usable.
 */
#define CP_SELFTEST_SCRATCH_BYTES ((size_t)512 << 10)
cp_status cp_selftest_stalled_kernel(int kernel, void *scratch, size_t scratch_bytes, uint64_t timeout_ns,
                                     cudaStream_t stream);

/*
 * cp_ring_attention_fwd_noalloc -- cp_ring_attention_fwd for callers that
 * cannot allocate device memory.  The source pages have no counterpart: this
 * entry point exists for callers that may not call cudaMalloc or cannot hand
 * the library a workspace -- code running inside a custom allocator's
 * callbacks (a cudaMalloc there re-enters the allocator), runtimes that
 * reserve all device memory at start-up and forbid allocation afterwards,
 * processes whose device memory pool belongs to another framework (memory
 * taken outside it escapes its accounting), and code under stream capture in
 * the global mode, where cudaMalloc is refused.
 *   Same arguments and result as cp_ring_attention_fwd with prefetch = 0
 *   (zero-copy owner rotation) and no workspace argument; the caller still
 *   passes all inputs and outputs.
 *   Scratch: the call uses one file-scope device array of
 *   CP_NOALLOC_SCRATCH_BYTES bytes inside the library (every CUDA context
 *   that loads the library's module holds one copy, until that context is
 *   destroyed: at process exit, or at cudaDeviceReset).  The ring's own
 *   argument checks (pointers, enums, shapes, divisibility, alignment) run
 *   first; then sizes whose cp_ring_workspace_size(..., prefetch = 0,
 *   o_dtype, ...) exceeds CP_NOALLOC_SCRATCH_BYTES are rejected with
 *   CP_ERR_WORKSPACE.  Either way nothing is enqueued.  The call never calls
 *   cudaMalloc, cudaFree or any allocating routine.
 *   Set-up: the first call in a CUDA context looks up the array's device
 *   address in that context (cudaGetSymbolAddress, with the caller's device
 *   and context current) and caches it, keyed by the context's id; make that
 *   first call before any stream capture in that context.  A call made in a
 *   new context (after cudaDeviceReset, or under a driver context the caller
 *   made current) looks the address up again, so no stale address is used.
 *   Sharing: all calls on a device share the array, which keeps the last
 *   call's contents (nothing needs clearing: every scratch byte a call reads
 *   it has written itself).  Calls whose executions overlap on the GPU (for
 *   instance on two streams) race on the array and give wrong results:
 *   serialise them.
 */
#define CP_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
cp_status cp_ring_attention_fwd_noalloc(const void *q_sh, const void *k_sh, const void *v_sh,
                                        const int32_t *pos, int64_t B, int64_t S, int64_t N,
                                        int64_t Nkv, int64_t D, int C, float scale, cp_layout layout,
                                        void *o_sh, cp_dtype o_dtype, float *lse_sh,
                                        cudaStream_t stream);

/*
 * cp_device_status -- synchronise `stream`, then read (and, if clear != 0,
 * reset) the library's device status word on the current device.
 * *code receives CP_OK, or CP_ERR_DEVICE_TIMEOUT if a kernel of this library
 * gave up a bounded wait since the last reset.  Host-blocking.
 */
cp_status cp_device_status(int *code, int clear, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CPATTN_H */
