/*
 * cporacle.c -- plain, slow, obviously-correct CPU reference (fp64) for
 * blockwise causal attention with log-sum-exp merging under zigzag /
 * contiguous context-parallel sharding.
 *
 * THIS IS TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or constant with the CUDA library (context_causal_attention_gb300/
 * csrc); neither side includes or links the other.
 *
 * Every function below follows a passage of the source pages; the passage is
 * named in the comment above it.  Page titles used:
 *   [OCP]  "On Context Parallelism"  (sections: All-gather (Forward,
 *          Backward), All-to-all, Peer-to-peer (Forward, Backward),
 *          Results and Conclusion)
 *   [DAY74] "Context parallelism -- splitting the sequence across GPUs"
 *          (sections: Why long contexts stress training memory, What exactly
 *          gets sharded?, How do partial softmax results combine?)
 *   [RING] "Context Parallelism & Ring Attention" (sections: Softmax is
 *          decomposable, The ring, The causal load-imbalance problem,
 *          The zigzag fix)
 *   [HB]   "Context parallelism: Ring Attention and Ulysses" (sections:
 *          Which operations partition directly / cp_common.py, Ulysses,
 *          Ring Attention, The zigzag partition)
 *
 * Conventions (readings where the pages are silent are marked READING):
 *   q  [B][Sq][N][D], k,v [B][Sk][Nkv][D], o [B][Sq][N][D], lse [B][N][Sq]
 *     ([OCP] Peer-to-peer / Forward: output [B,S/C,N,D], lse [B,N,S/C]).
 *   A key j is visible to query i iff kpos[j] <= qpos[i]
 *     ([HB] cp_common.py masks ki > qi; [DAY74] sums over j <= i).
 *   lse is the natural log of the sum of exp of the scaled scores
 *     ([OCP] Peer-to-peer: tile_lse = log(sum_j e^{s_j})).
 *   READING: a query row with no visible key yields lse = -inf and o = 0.
 *   READING: query head h reads KV head h / (N / Nkv).
 *
 * Build: gcc -O2 -std=c11 -shared -fPIC -pthread cporacle.c -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_NEG_INF (-INFINITY)

/* ------------------------------------------------------------------------ */
/* small thread pool: run fn(arg, unit) for unit in [0, n_units)            */
/* ------------------------------------------------------------------------ */
typedef void (*orc_unit_fn)(void *arg, long unit);
typedef struct {
    orc_unit_fn fn;
    void *arg;
    long n_units;
    long next;
    pthread_mutex_t mu;
} orc_pool;

static void *orc_worker(void *p) {
    orc_pool *pool = (orc_pool *)p;
    for (;;) {
        pthread_mutex_lock(&pool->mu);
        long u = pool->next++;
        pthread_mutex_unlock(&pool->mu);
        if (u >= pool->n_units) break;
        pool->fn(pool->arg, u);
    }
    return NULL;
}

static void orc_parallel(orc_unit_fn fn, void *arg, long n_units, int nthreads) {
    if (nthreads <= 1 || n_units <= 1) {
        for (long u = 0; u < n_units; ++u) fn(arg, u);
        return;
    }
    if (nthreads > 256) nthreads = 256;
    orc_pool pool;
    pool.fn = fn;
    pool.arg = arg;
    pool.n_units = n_units;
    pool.next = 0;
    pthread_mutex_init(&pool.mu, NULL);
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, orc_worker, &pool) == 0) ++started;
    if (started == 0) orc_worker(&pool);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&pool.mu);
}

/* ------------------------------------------------------------------------ */
/* Direct causal attention with explicit positions.                         */
/*                                                                          */
/* [HB] cp_common.py (attention returning output and per-row log-sum-exp)   */
/* and [DAY74] "Why long contexts stress training memory" (the softmax over */
/* eligible keys j <= i with scores q_i.k_j / sqrt(d_h)).  For one query    */
/* row: s_j = scale * <q_i, k_j> over visible j, lse = log sum_j e^{s_j},   */
/* o = sum_j e^{s_j - lse} v_j.  The max is subtracted before exponentials  */
/* only for range safety; lse = m + log sum e^{s_j - m} is the same number  */
/* ([OCP] Peer-to-peer, the tile_lse derivation).                           */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v;
    const int32_t *qpos, *kpos;
    long B, Sq, Sk, N, Nkv, D;
    double scale;
    const long *rows; /* NULL: all rows; else list of query indices */
    long nrows;       /* number of output rows per (b,h) */
    long rows_per_unit;
    double *o, *lse;
} orc_attn_job;

static void orc_attn_row(const orc_attn_job *J, long b, long h, long i, long out_i,
                         double *s /* scratch [Sk] */) {
    const long D = J->D, N = J->N, Nkv = J->Nkv;
    const long hk = h / (N / Nkv);
    const double *qi = J->q + ((b * J->Sq + i) * N + h) * D;
    double *oi = J->o + ((b * J->nrows + out_i) * N + h) * D;
    double m = ORC_NEG_INF;
    int any = 0;
    for (long j = 0; j < J->Sk; ++j) {
        if (J->kpos[j] > J->qpos[i]) continue;
        const double *kj = J->k + ((b * J->Sk + j) * Nkv + hk) * D;
        double dot = 0.0;
        for (long d = 0; d < D; ++d) dot += qi[d] * kj[d];
        s[j] = J->scale * dot;
        if (!any || s[j] > m) m = s[j];
        any = 1;
    }
    for (long d = 0; d < D; ++d) oi[d] = 0.0;
    double *lse_out = J->lse + (b * N + h) * J->nrows + out_i;
    if (!any) {
        *lse_out = ORC_NEG_INF;
        return;
    }
    double l = 0.0;
    for (long j = 0; j < J->Sk; ++j) {
        if (J->kpos[j] > J->qpos[i]) continue;
        l += exp(s[j] - m);
    }
    const double lse = m + log(l);
    for (long j = 0; j < J->Sk; ++j) {
        if (J->kpos[j] > J->qpos[i]) continue;
        const double p = exp(s[j] - lse);
        const double *vj = J->v + ((b * J->Sk + j) * Nkv + hk) * D;
        for (long d = 0; d < D; ++d) oi[d] += p * vj[d];
    }
    *lse_out = lse;
}

static void orc_attn_unit(void *arg, long unit) {
    const orc_attn_job *J = (const orc_attn_job *)arg;
    const long nblk = (J->nrows + J->rows_per_unit - 1) / J->rows_per_unit;
    const long bh = unit / nblk, blk = unit % nblk;
    const long b = bh / J->N, h = bh % J->N;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->Sk > 0 ? J->Sk : 1));
    if (!s) return;
    const long r0 = blk * J->rows_per_unit;
    long r1 = r0 + J->rows_per_unit;
    if (r1 > J->nrows) r1 = J->nrows;
    for (long r = r0; r < r1; ++r) {
        const long i = J->rows ? J->rows[r] : r;
        orc_attn_row(J, b, h, i, r, s);
    }
    free(s);
}

/* All query rows.  o [B][Sq][N][D], lse [B][N][Sq]. */
int orc_attn_direct(const double *q, const double *k, const double *v, const int32_t *qpos,
                    const int32_t *kpos, long B, long Sq, long Sk, long N, long Nkv, long D,
                    double scale, double *o, double *lse, int nthreads) {
    if (N <= 0 || Nkv <= 0 || N % Nkv != 0) return 1;
    orc_attn_job J = {q, k, v, qpos, kpos, B, Sq, Sk, N, Nkv, D, scale, NULL, Sq, 16, o, lse};
    const long nblk = (Sq + J.rows_per_unit - 1) / J.rows_per_unit;
    orc_parallel(orc_attn_unit, &J, B * N * nblk, nthreads);
    return 0;
}

/* A chosen subset of query rows (used to check very long sequences).
 * o [B][nrows][N][D], lse [B][N][nrows]; row r of the output is query rows[r]. */
int orc_attn_rows(const double *q, const double *k, const double *v, const int32_t *qpos,
                  const int32_t *kpos, long B, long Sq, long Sk, long N, long Nkv, long D,
                  double scale, const long *rows, long nrows, double *o, double *lse,
                  int nthreads) {
    if (N <= 0 || Nkv <= 0 || N % Nkv != 0) return 1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= Sq) return 2;
    orc_attn_job J = {q, k, v, qpos, kpos, B, Sq, Sk, N, Nkv, D, scale, rows, nrows, 4, o, lse};
    const long nblk = (nrows + J.rows_per_unit - 1) / J.rows_per_unit;
    orc_parallel(orc_attn_unit, &J, B * N * nblk, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Blockwise attention by the online-softmax recurrence.                    */
/*                                                                          */
/* [RING] "Softmax is decomposable": keep the running max m, the running    */
/* sum of exponentials l and the normalised output O; for a block with      */
/* local max m_b, local sum l_b and unnormalised P_b V_b:                   */
/*   m' = max(m, m_b)                                                       */
/*   l' = l e^{m-m'} + l_b e^{m_b-m'}                                       */
/*   O' = (l e^{m-m'} O + e^{m_b-m'} P_b V_b) / l'                          */
/* Initial state m = -inf, l = 0, O = 0 ([RING] "The ring", step 2).        */
/* Key blocks are consecutive key indices of length `block`.  A block with  */
/* no visible key leaves the state unchanged.  lse = m + log l at the end.  */
/* Single-threaded on purpose.                                              */
/* ------------------------------------------------------------------------ */
int orc_attn_blockwise(const double *q, const double *k, const double *v, const int32_t *qpos,
                       const int32_t *kpos, long B, long Sq, long Sk, long N, long Nkv, long D,
                       double scale, long block, double *o, double *lse) {
    if (block <= 0 || N <= 0 || Nkv <= 0 || N % Nkv != 0) return 1;
    double *s = (double *)malloc(sizeof(double) * (size_t)block);
    double *pv = (double *)malloc(sizeof(double) * (size_t)D);
    if (!s || !pv) {
        free(s);
        free(pv);
        return 3;
    }
    for (long b = 0; b < B; ++b)
        for (long h = 0; h < N; ++h) {
            const long hk = h / (N / Nkv);
            for (long i = 0; i < Sq; ++i) {
                const double *qi = q + ((b * Sq + i) * N + h) * D;
                double *Oi = o + ((b * Sq + i) * N + h) * D;
                double m = ORC_NEG_INF, l = 0.0;
                for (long d = 0; d < D; ++d) Oi[d] = 0.0;
                for (long j0 = 0; j0 < Sk; j0 += block) {
                    long j1 = j0 + block;
                    if (j1 > Sk) j1 = Sk;
                    double mb = ORC_NEG_INF;
                    int any = 0;
                    for (long j = j0; j < j1; ++j) {
                        if (kpos[j] > qpos[i]) continue;
                        const double *kj = k + ((b * Sk + j) * Nkv + hk) * D;
                        double dot = 0.0;
                        for (long d = 0; d < D; ++d) dot += qi[d] * kj[d];
                        s[j - j0] = scale * dot;
                        if (!any || s[j - j0] > mb) mb = s[j - j0];
                        any = 1;
                    }
                    if (!any) continue;
                    double lb = 0.0;
                    for (long d = 0; d < D; ++d) pv[d] = 0.0;
                    for (long j = j0; j < j1; ++j) {
                        if (kpos[j] > qpos[i]) continue;
                        const double p = exp(s[j - j0] - mb);
                        lb += p;
                        const double *vj = v + ((b * Sk + j) * Nkv + hk) * D;
                        for (long d = 0; d < D; ++d) pv[d] += p * vj[d];
                    }
                    const double mn = (m > mb) ? m : mb;
                    const double a_old = (l > 0.0) ? exp(m - mn) : 0.0;
                    const double a_blk = exp(mb - mn);
                    const double ln = l * a_old + lb * a_blk;
                    for (long d = 0; d < D; ++d) Oi[d] = (l * a_old * Oi[d] + a_blk * pv[d]) / ln;
                    m = mn;
                    l = ln;
                }
                lse[(b * N + h) * Sq + i] = (l > 0.0) ? m + log(l) : ORC_NEG_INF;
            }
        }
    free(s);
    free(pv);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* LSE merge of two completed partials, in place into (o_acc, lse_acc).     */
/*                                                                          */
/* [HB] "Ring Attention: passing the KV once around a ring": two partials   */
/* (o1, lse1), (o2, lse2) of one query row combine into                     */
/*   lse = log(e^lse1 + e^lse2),  o = o1 e^(lse1 - lse) + o2 e^(lse2 - lse) */
/* ([OCP] Peer-to-peer / Forward merges the ring's tiles with the same      */
/* result).  Evaluated with the larger lse factored out: with hi, lo the    */
/* larger and smaller of the two and r = e^(lo - hi) in (0, 1],             */
/* lse = hi + log(1 + r); the weight e^(lse_i - lse) is 1 / (1 + r) for the */
/* partial with lse hi and r / (1 + r) for the one with lse lo.             */
/* READING (the pages are silent): a row whose tile lse is -inf is left     */
/* unchanged; a row whose accumulated lse is -inf takes the tile's values.  */
/* Layouts: o [B][Sq][N][D], lse [B][N][Sq].                                */
/* ------------------------------------------------------------------------ */
void orc_lse_merge(double *o_acc, double *lse_acc, const double *o_t, const double *lse_t, long B,
                   long Sq, long N, long D) {
    for (long b = 0; b < B; ++b)
        for (long h = 0; h < N; ++h)
            for (long i = 0; i < Sq; ++i) {
                double *la = lse_acc + (b * N + h) * Sq + i;
                const double lt = lse_t[(b * N + h) * Sq + i];
                double *oa = o_acc + ((b * Sq + i) * N + h) * D;
                const double *ot = o_t + ((b * Sq + i) * N + h) * D;
                if (lt == ORC_NEG_INF) continue;
                if (*la == ORC_NEG_INF) {
                    for (long d = 0; d < D; ++d) oa[d] = ot[d];
                    *la = lt;
                    continue;
                }
                const int acc_is_hi = *la >= lt;
                const double hi = acc_is_hi ? *la : lt;
                const double lo = acc_is_hi ? lt : *la;
                const double r = exp(lo - hi);
                const double w_hi = 1.0 / (1.0 + r);
                const double w_lo = r / (1.0 + r);
                const double w_acc = acc_is_hi ? w_hi : w_lo;
                const double w_tile = acc_is_hi ? w_lo : w_hi;
                for (long d = 0; d < D; ++d) oa[d] = w_acc * oa[d] + w_tile * ot[d];
                *la = hi + log1p(r);
            }
}

/* The boxed block-combine form of [DAY74] "How do partial softmax results  */
/* combine?": o = sum_r e^{m_r - m} z_r / sum_r e^{m_r - m} l_r, with        */
/* m = max_r m_r.  Given R partials of ONE row as (lse_r, o_r) (o_r already */
/* normalised, so z_r = l_r o_r and m_r + log l_r = lse_r), writes o and     */
/* returns lse.  Used to cross-check the pairwise merge: it is symmetric in  */
/* r by construction.                                                        */
double orc_combine_row(const double *lse_r, const double *o_r, long R, long D, double *o) {
    double m = ORC_NEG_INF;
    for (long r = 0; r < R; ++r)
        if (lse_r[r] > m) m = lse_r[r];
    for (long d = 0; d < D; ++d) o[d] = 0.0;
    if (m == ORC_NEG_INF) return ORC_NEG_INF;
    double den = 0.0;
    for (long r = 0; r < R; ++r) {
        if (lse_r[r] == ORC_NEG_INF) continue;
        const double w = exp(lse_r[r] - m); /* = e^{m_r - m} l_r */
        den += w;
        for (long d = 0; d < D; ++d) o[d] += w * o_r[r * D + d];
    }
    for (long d = 0; d < D; ++d) o[d] /= den;
    return m + log(den);
}

/* ------------------------------------------------------------------------ */
/* Sharding and positions.                                                  */
/*                                                                          */
/* [OCP] All-gather: S is cut into 2C chunks of t = S/(2C) tokens; rank r   */
/* owns chunk r and chunk 2C-r-1, so its local sequence is                  */
/* [chunk r | chunk 2C-1-r] of length s = 2t.  ([RING] "The zigzag fix";    */
/* [HB] "The zigzag partition".)                                            */
/* [RING] "The last remaining axis" and [DAY74] "What exactly gets          */
/* sharded?": contiguous sharding gives rank r tokens [r s, (r+1) s).       */
/* layout 0 = zigzag, 1 = contiguous.                                       */
/* Sharded buffers are rank-major: xs [C][B][s][N][D].                      */
/* ------------------------------------------------------------------------ */
static long orc_global_pos(long S, int C, int layout, int r, long u) {
    const long s = S / C;
    if (layout == 1) return (long)r * s + u;
    const long t = S / (2L * C);
    const long chunk = (u < t) ? (long)r : (2L * C - 1 - r);
    return chunk * t + (u % t);
}

int orc_positions(int32_t *pos, long S, int C, int layout) {
    if (C <= 0) return 1;
    if (layout == 0 && S % (2L * C) != 0) return 1;
    if (layout == 1 && S % C != 0) return 1;
    const long s = S / C;
    for (int r = 0; r < C; ++r)
        for (long u = 0; u < s; ++u) pos[(long)r * s + u] = (int32_t)orc_global_pos(S, C, layout, r, u);
    return 0;
}

/* x [B][S][N][D] -> xs [C][B][s][N][D], element by element (esize bytes). */
int orc_shard(const void *x, void *xs, long B, long S, long N, long D, int C, int layout,
              long esize) {
    if (C <= 0) return 1;
    if (layout == 0 && S % (2L * C) != 0) return 1;
    if (layout == 1 && S % C != 0) return 1;
    const long s = S / C, row = N * D;
    const char *src = (const char *)x;
    char *dst = (char *)xs;
    for (int r = 0; r < C; ++r)
        for (long b = 0; b < B; ++b)
            for (long u = 0; u < s; ++u) {
                const long g = orc_global_pos(S, C, layout, r, u);
                for (long e = 0; e < row; ++e) {
                    const long di = (((long)r * B + b) * s + u) * row + e;
                    const long si = (b * S + g) * row + e;
                    memcpy(dst + di * esize, src + si * esize, (size_t)esize);
                }
            }
    return 0;
}

/* Inverse of orc_shard: the all-gather followed by the reordering of       */
/* [OCP] All-gather ("[chunk 0, chunk 7, chunk 1, ...]" back to sequence     */
/* order).                                                                   */
int orc_unshard(const void *xs, void *x, long B, long S, long N, long D, int C, int layout,
                long esize) {
    if (C <= 0) return 1;
    if (layout == 0 && S % (2L * C) != 0) return 1;
    if (layout == 1 && S % C != 0) return 1;
    const long s = S / C, row = N * D;
    const char *src = (const char *)xs;
    char *dst = (char *)x;
    for (int r = 0; r < C; ++r)
        for (long b = 0; b < B; ++b)
            for (long u = 0; u < s; ++u) {
                const long g = orc_global_pos(S, C, layout, r, u);
                for (long e = 0; e < row; ++e) {
                    const long si = (((long)r * B + b) * s + u) * row + e;
                    const long di = (b * S + g) * row + e;
                    memcpy(dst + di * esize, src + si * esize, (size_t)esize);
                }
            }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Ulysses relayout as a local permutation of rank-major buffers.           */
/*                                                                          */
/* [HB] "Ulysses" (seq_to_head / head_to_seq) and [OCP] All-to-all;         */
/* Appendix F eq. (96): [B, S/C, H, d_h] -> [B, S, H/C, d_h].               */
/* Sequence-to-head: destination rank r receives head group r (heads        */
/* [r N/C, (r+1) N/C)) from every source rank j, source shards concatenated */
/* in rank order:                                                           */
/*   out[r][b][j s + u][h'][d] = in[j][b][u][r N/C + h'][d].                */
/* order 1 (READING, the TE reorder of [OCP] All-to-all): the concatenated  */
/* sequence is put in global order, row j s + u replaced by the global      */
/* position of row u of rank j under zigzag sharding.                        */
/* Head-to-sequence (dir 1) is the exact inverse.                           */
/* in/out: SEQ side [C][B][s][N][D], HEAD side [C][B][S][N/C][D].           */
/* ------------------------------------------------------------------------ */
int orc_ulysses(const void *in, void *out, long B, long S, long N, long D, int C, long esize,
                int dir, int order) {
    if (C <= 0 || S % C != 0 || N % C != 0) return 1;
    if (order == 1 && S % (2L * C) != 0) return 1;
    const long s = S / C, nh = N / C;
    const char *src = (const char *)in;
    char *dst = (char *)out;
    for (int r = 0; r < C; ++r)         /* head-group rank */
        for (long b = 0; b < B; ++b)
            for (int j = 0; j < C; ++j) /* sequence-shard rank */
                for (long u = 0; u < s; ++u) {
                    const long row = (order == 1) ? orc_global_pos(S, C, 0, j, u) : (long)j * s + u;
                    for (long hh = 0; hh < nh; ++hh)
                        for (long d = 0; d < D; ++d) {
                            const long seq_i = ((((long)j * B + b) * s + u) * N + (long)r * nh + hh) * D + d;
                            const long head_i = ((((long)r * B + b) * S + row) * nh + hh) * D + d;
                            if (dir == 0)
                                memcpy(dst + head_i * esize, src + seq_i * esize, (size_t)esize);
                            else
                                memcpy(dst + seq_i * esize, src + head_i * esize, (size_t)esize);
                        }
                }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Ring forward over C virtual ranks.                                       */
/*                                                                          */
/* [OCP] Peer-to-peer / Forward: for step in 0..C-1 the K/V block in hand   */
/* on rank r belongs to kv_owner = (r - step) mod C; the partial attention  */
/* of the local queries against it (positions of both sides) is merged into */
/* the running (o, lse); the first partial is taken as is.                  */
/* Inputs are rank-major fp64 shards q_sh [C][B][s][N][D],                  */
/* k_sh, v_sh [C][B][s][Nkv][D], positions pos [C][s].                      */
/* Outputs o_sh [C][B][s][N][D], lse_sh [C][B][N][s].                       */
/* ------------------------------------------------------------------------ */
int orc_ring_fwd(const double *q_sh, const double *k_sh, const double *v_sh, const int32_t *pos,
                 long B, long S, long N, long Nkv, long D, int C, double scale, double *o_sh,
                 double *lse_sh, int nthreads) {
    if (C <= 0 || S % C != 0) return 1;
    const long s = S / C;
    const long qn = B * s * N * D, kn = B * s * Nkv * D, ln = B * N * s;
    double *o_t = (double *)malloc(sizeof(double) * (size_t)qn);
    double *l_t = (double *)malloc(sizeof(double) * (size_t)ln);
    if (!o_t || !l_t) {
        free(o_t);
        free(l_t);
        return 3;
    }
    for (int r = 0; r < C; ++r) {
        double *o = o_sh + (long)r * qn, *lse = lse_sh + (long)r * ln;
        for (int step = 0; step < C; ++step) {
            const int owner = ((r - step) % C + C) % C;
            int rc = orc_attn_direct(q_sh + (long)r * qn, k_sh + (long)owner * kn, v_sh + (long)owner * kn,
                                     pos + (long)r * s, pos + (long)owner * s, B, s, s, N, Nkv, D, scale,
                                     step == 0 ? o : o_t, step == 0 ? lse : l_t, nthreads);
            if (rc) {
                free(o_t);
                free(l_t);
                return rc;
            }
            if (step > 0) orc_lse_merge(o, lse, o_t, l_t, B, s, N, D);
        }
    }
    free(o_t);
    free(l_t);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward of one attention tile.                                          */
/*                                                                          */
/* [OCP] Peer-to-peer / Backward: attention_tile_backward(q, k, v, output,  */
/* grad_output, lse, q_positions, kv_positions, scale) returns the tile's   */
/* (dq, dk, dv); the call receives the FINAL output and lse of the whole    */
/* attention, so within a tile the probability of a visible pair is the     */
/* global one, p_ij = e^{s_ij - lse_i}.  The pages print no formula for it; */
/* it is the derivative of o_i = sum_j p_ij v_j with s_ij = scale <q_i,k_j> */
/* written out by the chain rule (READING: the plain definition):           */
/*   dv_j += p_ij dO_i                                                      */
/*   dp_ij = <dO_i, v_j>                                                    */
/*   ds_ij = p_ij (dp_ij - delta_i),  delta_i = sum_j' p_ij' dp_ij'         */
/*                                          = <dO_i, o_i>                   */
/*   dq_i += scale ds_ij k_j,   dk_j += scale ds_ij q_i                     */
/* (delta_i is taken as <dO_i, o_i> with the given output; over the whole   */
/* key set it equals the sum over j, which a pin checks.)                   */
/* Rows with lse = -inf see no key and contribute nothing.  With            */
/* N > Nkv the gradients of a KV head sum over its query heads.             */
/* Inputs as orc_attn_direct plus o, dO [B][Sq][N][D], lse [B][N][Sq];      */
/* outputs dq [B][Sq][N][D], dk, dv [B][Sk][Nkv][D] (overwritten).          */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v, *o, *dout, *lse;
    const int32_t *qpos, *kpos;
    long B, Sq, Sk, N, Nkv, D;
    double scale;
    double *dq, *dk, *dv;
} orc_bwd_job;

static void orc_bwd_unit(void *arg, long unit) {
    /* one unit = one (b, kv head) with all its query heads: no two units
       write the same dq, dk or dv element */
    const orc_bwd_job *J = (const orc_bwd_job *)arg;
    const long D = J->D, N = J->N, Nkv = J->Nkv, g = N / Nkv;
    const long b = unit / Nkv, hk = unit % Nkv;
    for (long j = 0; j < J->Sk; ++j)
        for (long d = 0; d < D; ++d) {
            J->dk[((b * J->Sk + j) * Nkv + hk) * D + d] = 0.0;
            J->dv[((b * J->Sk + j) * Nkv + hk) * D + d] = 0.0;
        }
    for (long h = hk * g; h < (hk + 1) * g; ++h)
        for (long i = 0; i < J->Sq; ++i) {
            const double *qi = J->q + ((b * J->Sq + i) * N + h) * D;
            const double *oi = J->o + ((b * J->Sq + i) * N + h) * D;
            const double *doi = J->dout + ((b * J->Sq + i) * N + h) * D;
            double *dqi = J->dq + ((b * J->Sq + i) * N + h) * D;
            for (long d = 0; d < D; ++d) dqi[d] = 0.0;
            const double lse = J->lse[(b * N + h) * J->Sq + i];
            if (lse == ORC_NEG_INF) continue;
            double delta = 0.0;
            for (long d = 0; d < D; ++d) delta += doi[d] * oi[d];
            for (long j = 0; j < J->Sk; ++j) {
                if (J->kpos[j] > J->qpos[i]) continue;
                const double *kj = J->k + ((b * J->Sk + j) * Nkv + hk) * D;
                const double *vj = J->v + ((b * J->Sk + j) * Nkv + hk) * D;
                double *dkj = J->dk + ((b * J->Sk + j) * Nkv + hk) * D;
                double *dvj = J->dv + ((b * J->Sk + j) * Nkv + hk) * D;
                double dot = 0.0, dp = 0.0;
                for (long d = 0; d < D; ++d) {
                    dot += qi[d] * kj[d];
                    dp += doi[d] * vj[d];
                }
                const double p = exp(J->scale * dot - lse);
                const double ds = p * (dp - delta);
                for (long d = 0; d < D; ++d) {
                    dvj[d] += p * doi[d];
                    dqi[d] += J->scale * ds * kj[d];
                    dkj[d] += J->scale * ds * qi[d];
                }
            }
        }
}

int orc_attn_bwd(const double *q, const double *k, const double *v, const double *o, const double *dout,
                 const double *lse, const int32_t *qpos, const int32_t *kpos, long B, long Sq, long Sk, long N,
                 long Nkv, long D, double scale, double *dq, double *dk, double *dv, int nthreads) {
    if (N <= 0 || Nkv <= 0 || N % Nkv != 0) return 1;
    orc_bwd_job J = {q, k, v, o, dout, lse, qpos, kpos, B, Sq, Sk, N, Nkv, D, scale, dq, dk, dv};
    orc_parallel(orc_bwd_unit, &J, B * Nkv, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Sampled gradients for sequences too long for orc_attn_bwd.               */
/*                                                                          */
/* Same definitions as orc_attn_bwd ([OCP] Peer-to-peer / Backward, the     */
/* chain rule of the forward), but nothing is taken from a forward output:  */
/* every row involved gets its lse_i, o_i and delta_i = <dO_i, o_i>          */
/* recomputed here from q, k, v in fp64.                                     */
/* ------------------------------------------------------------------------ */
typedef struct {
    const double *q, *k, *v, *dout;
    const int32_t *qpos, *kpos;
    long B, Sq, Sk, N, Nkv, D;
    double scale;
    const long *sel; /* sampled query rows (dq) or keys (dk, dv) */
    long nsel;
    double *out1, *out2;
} orc_bwd_sample_job;

/* lse, o and delta of query row i of head h (o written to o_i [D]). */
static double orc_row_stats(const orc_bwd_sample_job *J, long b, long h, long i, double *o_i, double *delta) {
    const long D = J->D, N = J->N, Nkv = J->Nkv, hk = h / (N / Nkv);
    const double *qi = J->q + ((b * J->Sq + i) * N + h) * D;
    double m = ORC_NEG_INF;
    int any = 0;
    for (long j = 0; j < J->Sk; ++j) {
        if (J->kpos[j] > J->qpos[i]) continue;
        const double *kj = J->k + ((b * J->Sk + j) * Nkv + hk) * D;
        double dot = 0.0;
        for (long d = 0; d < D; ++d) dot += qi[d] * kj[d];
        const double sj = J->scale * dot;
        if (!any || sj > m) m = sj;
        any = 1;
    }
    for (long d = 0; d < D; ++d) o_i[d] = 0.0;
    *delta = 0.0;
    if (!any) return ORC_NEG_INF;
    double l = 0.0;
    for (long j = 0; j < J->Sk; ++j) {
        if (J->kpos[j] > J->qpos[i]) continue;
        const double *kj = J->k + ((b * J->Sk + j) * Nkv + hk) * D;
        double dot = 0.0;
        for (long d = 0; d < D; ++d) dot += qi[d] * kj[d];
        l += exp(J->scale * dot - m);
    }
    const double lse = m + log(l);
    for (long j = 0; j < J->Sk; ++j) {
        if (J->kpos[j] > J->qpos[i]) continue;
        const double *kj = J->k + ((b * J->Sk + j) * Nkv + hk) * D;
        const double *vj = J->v + ((b * J->Sk + j) * Nkv + hk) * D;
        double dot = 0.0;
        for (long d = 0; d < D; ++d) dot += qi[d] * kj[d];
        const double p = exp(J->scale * dot - lse);
        for (long d = 0; d < D; ++d) o_i[d] += p * vj[d];
    }
    const double *doi = J->dout + ((b * J->Sq + i) * N + h) * D;
    for (long d = 0; d < D; ++d) *delta += doi[d] * o_i[d];
    return lse;
}

static void orc_bwd_rows_unit(void *arg, long unit) {
    /* unit = (b, h, sampled row) */
    const orc_bwd_sample_job *J = (const orc_bwd_sample_job *)arg;
    const long D = J->D, N = J->N, Nkv = J->Nkv, hk_div = N / Nkv;
    const long r = unit % J->nsel, bh = unit / J->nsel, b = bh / N, h = bh % N, hk = h / hk_div;
    const long i = J->sel[r];
    double *dq = J->out1 + ((b * J->nsel + r) * N + h) * D;
    for (long d = 0; d < D; ++d) dq[d] = 0.0;
    double *o_i = (double *)malloc(sizeof(double) * (size_t)D);
    if (!o_i) return;
    double delta;
    const double lse = orc_row_stats(J, b, h, i, o_i, &delta);
    if (lse != ORC_NEG_INF) {
        const double *qi = J->q + ((b * J->Sq + i) * N + h) * D;
        const double *doi = J->dout + ((b * J->Sq + i) * N + h) * D;
        for (long j = 0; j < J->Sk; ++j) {
            if (J->kpos[j] > J->qpos[i]) continue;
            const double *kj = J->k + ((b * J->Sk + j) * Nkv + hk) * D;
            const double *vj = J->v + ((b * J->Sk + j) * Nkv + hk) * D;
            double dot = 0.0, dp = 0.0;
            for (long d = 0; d < D; ++d) {
                dot += qi[d] * kj[d];
                dp += doi[d] * vj[d];
            }
            const double ds = exp(J->scale * dot - lse) * (dp - delta);
            for (long d = 0; d < D; ++d) dq[d] += J->scale * ds * kj[d];
        }
    }
    free(o_i);
}

/* dq of the query rows rows[0..nrows): dq [B][nrows][N][D]. */
int orc_attn_bwd_rows(const double *q, const double *k, const double *v, const double *dout, const int32_t *qpos,
                      const int32_t *kpos, long B, long Sq, long Sk, long N, long Nkv, long D, double scale,
                      const long *rows, long nrows, double *dq, int nthreads) {
    if (N <= 0 || Nkv <= 0 || N % Nkv != 0) return 1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= Sq) return 2;
    orc_bwd_sample_job J = {q, k, v, dout, qpos, kpos, B, Sq, Sk, N, Nkv, D, scale, rows, nrows, dq, NULL};
    orc_parallel(orc_bwd_rows_unit, &J, B * N * nrows, nthreads);
    return 0;
}

static void orc_bwd_keys_unit(void *arg, long unit) {
    /* unit = (b, kv head, sampled key): sums over the query heads of the group
       and over every query row that sees the key */
    const orc_bwd_sample_job *J = (const orc_bwd_sample_job *)arg;
    const long D = J->D, N = J->N, Nkv = J->Nkv, g = N / Nkv;
    const long r = unit % J->nsel, bh = unit / J->nsel, b = bh / Nkv, hk = bh % Nkv;
    const long j = J->sel[r];
    double *dk = J->out1 + ((b * J->nsel + r) * Nkv + hk) * D;
    double *dv = J->out2 + ((b * J->nsel + r) * Nkv + hk) * D;
    for (long d = 0; d < D; ++d) dk[d] = dv[d] = 0.0;
    double *o_i = (double *)malloc(sizeof(double) * (size_t)D);
    if (!o_i) return;
    const double *kj = J->k + ((b * J->Sk + j) * Nkv + hk) * D;
    const double *vj = J->v + ((b * J->Sk + j) * Nkv + hk) * D;
    for (long h = hk * g; h < (hk + 1) * g; ++h)
        for (long i = 0; i < J->Sq; ++i) {
            if (J->kpos[j] > J->qpos[i]) continue;
            double delta;
            const double lse = orc_row_stats(J, b, h, i, o_i, &delta);
            const double *qi = J->q + ((b * J->Sq + i) * N + h) * D;
            const double *doi = J->dout + ((b * J->Sq + i) * N + h) * D;
            double dot = 0.0, dp = 0.0;
            for (long d = 0; d < D; ++d) {
                dot += qi[d] * kj[d];
                dp += doi[d] * vj[d];
            }
            const double p = exp(J->scale * dot - lse);
            const double ds = p * (dp - delta);
            for (long d = 0; d < D; ++d) {
                dv[d] += p * doi[d];
                dk[d] += J->scale * ds * qi[d];
            }
        }
    free(o_i);
}

/* dk, dv of the keys keys[0..nkeys): dk, dv [B][nkeys][Nkv][D].  Cost grows
 * with the number of query rows that see each key (use late keys). */
int orc_attn_bwd_keys(const double *q, const double *k, const double *v, const double *dout, const int32_t *qpos,
                      const int32_t *kpos, long B, long Sq, long Sk, long N, long Nkv, long D, double scale,
                      const long *keys, long nkeys, double *dk, double *dv, int nthreads) {
    if (N <= 0 || Nkv <= 0 || N % Nkv != 0) return 1;
    for (long r = 0; r < nkeys; ++r)
        if (keys[r] < 0 || keys[r] >= Sk) return 2;
    orc_bwd_sample_job J = {q, k, v, dout, qpos, kpos, B, Sq, Sk, N, Nkv, D, scale, keys, nkeys, dk, dv};
    orc_parallel(orc_bwd_keys_unit, &J, B * Nkv * nkeys, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Ring backward over C virtual ranks.                                      */
/*                                                                          */
/* [OCP] Peer-to-peer / Backward: rank r keeps its queries and accumulates  */
/* dq locally; at step `step` it holds the K/V block of                     */
/* kv_owner = (r - step) mod C together with that block's travelling dk/dv  */
/* accumulators, adds the tile's (dk, dv) to them, and passes all four on;  */
/* after the full rotation each block's accumulated dk/dv is back on its    */
/* owner.  Without transport the travelling accumulator of block j is the   */
/* owner's own dk_sh[j] / dv_sh[j].  The tile backward gets the final       */
/* output and lse of rank r (saved by the forward).                         */
/* Shards as orc_ring_fwd; o_sh, do_sh [C][B][s][N][D], lse_sh [C][B][N][s]; */
/* outputs dq_sh [C][B][s][N][D], dk_sh, dv_sh [C][B][s][Nkv][D].           */
/* ------------------------------------------------------------------------ */
int orc_ring_bwd(const double *q_sh, const double *k_sh, const double *v_sh, const double *o_sh,
                 const double *do_sh, const double *lse_sh, const int32_t *pos, long B, long S, long N, long Nkv,
                 long D, int C, double scale, double *dq_sh, double *dk_sh, double *dv_sh, int nthreads) {
    if (C <= 0 || S % C != 0) return 1;
    const long s = S / C;
    const long qn = B * s * N * D, kn = B * s * Nkv * D, ln = B * N * s;
    double *tq = (double *)malloc(sizeof(double) * (size_t)qn);
    double *tk = (double *)malloc(sizeof(double) * (size_t)kn);
    double *tv = (double *)malloc(sizeof(double) * (size_t)kn);
    if (!tq || !tk || !tv) {
        free(tq);
        free(tk);
        free(tv);
        return 3;
    }
    memset(dq_sh, 0, sizeof(double) * (size_t)(C * qn));
    memset(dk_sh, 0, sizeof(double) * (size_t)(C * kn));
    memset(dv_sh, 0, sizeof(double) * (size_t)(C * kn));
    int rc = 0;
    for (int r = 0; r < C && !rc; ++r)
        for (int step = 0; step < C && !rc; ++step) {
            const int owner = ((r - step) % C + C) % C;
            rc = orc_attn_bwd(q_sh + (long)r * qn, k_sh + (long)owner * kn, v_sh + (long)owner * kn,
                              o_sh + (long)r * qn, do_sh + (long)r * qn, lse_sh + (long)r * ln, pos + (long)r * s,
                              pos + (long)owner * s, B, s, s, N, Nkv, D, scale, tq, tk, tv, nthreads);
            if (rc) break;
            for (long x = 0; x < qn; ++x) dq_sh[(long)r * qn + x] += tq[x];
            for (long x = 0; x < kn; ++x) {
                dk_sh[(long)owner * kn + x] += tk[x];
                dv_sh[(long)owner * kn + x] += tv[x];
            }
        }
    free(tq);
    free(tk);
    free(tv);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Causal work per rank.                                                    */
/*                                                                          */
/* Exact count of visible (query, key) pairs: for rank r and K/V owner j,    */
/* pairs[r][j] = #{(u, w) : pos[j][w] <= pos[r][u]}.  Plain double loop     */
/* over the rank's queries with a sorted copy of the owner's positions.     */
/* [RING] "The causal load-imbalance problem" (contiguous: work grows with  */
/* the rank) and "The zigzag fix" (equal work per rank); [HB] "The zigzag   */
/* partition".                                                              */
/* ------------------------------------------------------------------------ */
static int orc_cmp_i32(const void *a, const void *b) {
    const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

int orc_pair_counts(const int32_t *pos, long S, int C, int64_t *pairs /* [C][C] */) {
    if (C <= 0 || S % C != 0) return 1;
    const long s = S / C;
    int32_t *sorted = (int32_t *)malloc(sizeof(int32_t) * (size_t)s);
    if (!sorted) return 3;
    for (int j = 0; j < C; ++j) {
        memcpy(sorted, pos + (long)j * s, sizeof(int32_t) * (size_t)s);
        qsort(sorted, (size_t)s, sizeof(int32_t), orc_cmp_i32);
        for (int r = 0; r < C; ++r) {
            int64_t total = 0;
            for (long u = 0; u < s; ++u) {
                const int32_t qp = pos[(long)r * s + u];
                long lo = 0, hi = s; /* first index with sorted[idx] > qp */
                while (lo < hi) {
                    const long mid = (lo + hi) / 2;
                    if (sorted[mid] <= qp) lo = mid + 1; else hi = mid;
                }
                total += lo;
            }
            pairs[(long)r * C + j] = total;
        }
    }
    free(sorted);
    return 0;
}
