"""fp64 CPU oracle for blockwise causal attention with LSE merging.

TEST INFRASTRUCTURE ONLY.  The test-suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package; the CUDA library and its Python binding never do, and the two share
no code.

Each wrapper names the passage of the source pages it follows (page titles as
in ``cporacle.c``).  Arrays are numpy; floating inputs are upcast to float64
(bf16 values arrive as float32 holding the exact bf16 value).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, invariants and values printed on the pages.
"""
import ctypes
import os

import numpy as np

from . import build_oracle

_lib = None
_i64p = ctypes.POINTER(ctypes.c_int64)


def _load():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        lib = ctypes.CDLL(path)
        dp, ip, vp = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        L, I, Dd = ctypes.c_long, ctypes.c_int, ctypes.c_double
        lib.orc_attn_direct.argtypes = [dp, dp, dp, ip, ip, L, L, L, L, L, L, Dd, dp, dp, I]
        lib.orc_attn_rows.argtypes = [dp, dp, dp, ip, ip, L, L, L, L, L, L, Dd, vp, L, dp, dp, I]
        lib.orc_attn_blockwise.argtypes = [dp, dp, dp, ip, ip, L, L, L, L, L, L, Dd, L, dp, dp]
        lib.orc_lse_merge.argtypes = [dp, dp, dp, dp, L, L, L, L]
        lib.orc_lse_merge.restype = None
        lib.orc_combine_row.argtypes = [dp, dp, L, L, dp]
        lib.orc_combine_row.restype = Dd
        lib.orc_positions.argtypes = [ip, L, I, I]
        lib.orc_shard.argtypes = [vp, vp, L, L, L, L, I, I, L]
        lib.orc_unshard.argtypes = [vp, vp, L, L, L, L, I, I, L]
        lib.orc_ulysses.argtypes = [vp, vp, L, L, L, L, I, L, I, I]
        lib.orc_ring_fwd.argtypes = [dp, dp, dp, ip, L, L, L, L, L, I, Dd, dp, dp, I]
        lib.orc_pair_counts.argtypes = [ip, L, I, vp]
        lib.orc_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, ip, ip, L, L, L, L, L, L, Dd, dp, dp, dp, I]
        lib.orc_attn_bwd_rows.argtypes = [dp, dp, dp, dp, ip, ip, L, L, L, L, L, L, Dd, vp, L, dp, I]
        lib.orc_attn_bwd_keys.argtypes = [dp, dp, dp, dp, ip, ip, L, L, L, L, L, L, Dd, vp, L, dp, dp, I]
        lib.orc_ring_bwd.argtypes = [dp, dp, dp, dp, dp, dp, ip, L, L, L, L, L, I, Dd, dp, dp, dp, I]
        _lib = lib
    return _lib


ZIGZAG, CONTIGUOUS = 0, 1
SEQ_TO_HEAD, HEAD_TO_SEQ = 0, 1
RANK_ORDER, GLOBAL_ORDER = 0, 1


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads():
    return len(os.sched_getaffinity(0))


def attn_direct(q, k, v, q_pos, k_pos, scale=None, nthreads=1):
    """Causal attention with explicit positions -> (o [B,Sq,N,D], lse [B,N,Sq]).

    "Context parallelism: Ring Attention and Ulysses", cp_common.py; "Context
    parallelism -- splitting the sequence across GPUs", the causal softmax
    formula.  Key j is visible to query i iff k_pos[j] <= q_pos[i].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    qp, kp = _i32(q_pos), _i32(k_pos)
    B, Sq, N, D = q.shape
    Sk, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.empty((B, Sq, N, D))
    lse = np.empty((B, N, Sq))
    rc = _load().orc_attn_direct(_p(q), _p(k), _p(v), _p(qp), _p(kp), B, Sq, Sk, N, Nkv, D,
                                 float(scale), _p(o), _p(lse), int(nthreads))
    if rc:
        raise ValueError("orc_attn_direct: bad arguments (%d)" % rc)
    return o, lse


def attn_rows(q, k, v, q_pos, k_pos, rows, scale=None, nthreads=1):
    """Same as attn_direct for the query rows listed in ``rows`` only.

    Returns (o [B,len(rows),N,D], lse [B,N,len(rows)]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    qp, kp = _i32(q_pos), _i32(k_pos)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    B, Sq, N, D = q.shape
    Sk, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    nr = rows.shape[0]
    o = np.empty((B, nr, N, D))
    lse = np.empty((B, N, nr))
    rc = _load().orc_attn_rows(_p(q), _p(k), _p(v), _p(qp), _p(kp), B, Sq, Sk, N, Nkv, D,
                               float(scale), _p(rows), nr, _p(o), _p(lse), int(nthreads))
    if rc:
        raise ValueError("orc_attn_rows: bad arguments (%d)" % rc)
    return o, lse


def attn_blockwise(q, k, v, q_pos, k_pos, block, scale=None):
    """Online-softmax recurrence over key blocks of ``block`` keys.

    "Context Parallelism & Ring Attention", section "Softmax is decomposable".
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    qp, kp = _i32(q_pos), _i32(k_pos)
    B, Sq, N, D = q.shape
    Sk, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.empty((B, Sq, N, D))
    lse = np.empty((B, N, Sq))
    rc = _load().orc_attn_blockwise(_p(q), _p(k), _p(v), _p(qp), _p(kp), B, Sq, Sk, N, Nkv, D,
                                    float(scale), int(block), _p(o), _p(lse))
    if rc:
        raise ValueError("orc_attn_blockwise: bad arguments (%d)" % rc)
    return o, lse


def lse_merge(o_acc, lse_acc, o_tile, lse_tile):
    """Merge a completed partial into an accumulator; returns new (o, lse).

    "Context parallelism: Ring Attention and Ulysses", Ring Attention: lse =
    log(e^lse1 + e^lse2), o = o1 e^(lse1 - lse) + o2 e^(lse2 - lse) (the same
    result as the tile merge of "On Context Parallelism", Peer-to-peer /
    Forward).  Inputs are not modified.  -inf tile rows leave the accumulator unchanged.
    """
    o = _f64(o_acc).copy()
    lse = _f64(lse_acc).copy()
    ot, lt = _f64(o_tile), _f64(lse_tile)
    B, Sq, N, D = o.shape
    if lse.shape != (B, N, Sq) or ot.shape != o.shape or lt.shape != lse.shape:
        raise ValueError("lse_merge: shape mismatch")
    _load().orc_lse_merge(_p(o), _p(lse), _p(ot), _p(lt), B, Sq, N, D)
    return o, lse


def combine_row(lses, outs):
    """Boxed block-combine of one row from R partials; returns (o [D], lse).

    "Context parallelism -- splitting the sequence across GPUs", section "How
    do partial softmax results combine?".
    """
    lses = _f64(lses)
    outs = _f64(outs)
    R, D = outs.shape
    o = np.empty(D)
    lse = _load().orc_combine_row(_p(lses), _p(outs), R, D, _p(o))
    return o, lse


def positions(S, C, layout=ZIGZAG):
    """Global position of every local token: int32 [C, S/C].

    "On Context Parallelism", All-gather (zigzag: rank r owns chunks r and
    2C-r-1); "Context Parallelism & Ring Attention", "The last remaining
    axis" (contiguous).
    """
    pos = np.empty((C, S // C), dtype=np.int32)
    if _load().orc_positions(_p(pos), S, C, layout):
        raise ValueError("positions: S not divisible")
    return pos


def shard(x, C, layout=ZIGZAG):
    """x [B,S,N,D] -> rank-major shards [C,B,S/C,N,D] (any dtype, bit copy)."""
    x = np.ascontiguousarray(x)
    B, S, N, D = x.shape
    out = np.empty((C, B, S // C, N, D), dtype=x.dtype)
    if _load().orc_shard(_p(x), _p(out), B, S, N, D, C, layout, x.dtype.itemsize):
        raise ValueError("shard: S not divisible")
    return out


def unshard(xs, layout=ZIGZAG):
    """Rank-major shards [C,B,s,N,D] -> x [B,C*s,N,D] in global order.

    "On Context Parallelism", All-gather: reorder rank-order chunks to
    sequence order.
    """
    xs = np.ascontiguousarray(xs)
    C, B, s, N, D = xs.shape
    S = C * s
    out = np.empty((B, S, N, D), dtype=xs.dtype)
    if _load().orc_unshard(_p(xs), _p(out), B, S, N, D, C, layout, xs.dtype.itemsize):
        raise ValueError("unshard: S not divisible")
    return out


def ulysses(x, C, direction=SEQ_TO_HEAD, order=RANK_ORDER):
    """Ulysses relayout between [C,B,S/C,N,D] and [C,B,S,N/C,D] (bit copy).

    "Context parallelism: Ring Attention and Ulysses", section "Ulysses"
    (seq_to_head / head_to_seq); Appendix F eq. (96).
    """
    x = np.ascontiguousarray(x)
    if direction == SEQ_TO_HEAD:
        Cx, B, s, N, D = x.shape
        S = C * s
        out = np.empty((C, B, S, N // C, D), dtype=x.dtype)
    else:
        Cx, B, S, nh, D = x.shape
        N = nh * C
        out = np.empty((C, B, S // C, N, D), dtype=x.dtype)
    if Cx != C:
        raise ValueError("ulysses: leading dim must be C")
    if _load().orc_ulysses(_p(x), _p(out), B, S, N, D, C, x.dtype.itemsize, direction, order):
        raise ValueError("ulysses: divisibility")
    return out


def ring_fwd(q_sh, k_sh, v_sh, pos, scale=None, nthreads=1):
    """Ring forward over C virtual ranks -> (o_sh [C,B,s,N,D], lse_sh [C,B,N,s]).

    "On Context Parallelism", Peer-to-peer / Forward.
    """
    q_sh, k_sh, v_sh = _f64(q_sh), _f64(k_sh), _f64(v_sh)
    pos = _i32(pos)
    C, B, s, N, D = q_sh.shape
    Nkv = k_sh.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.empty_like(q_sh)
    lse = np.empty((C, B, N, s))
    rc = _load().orc_ring_fwd(_p(q_sh), _p(k_sh), _p(v_sh), _p(pos), B, C * s, N, Nkv, D, C,
                              float(scale), _p(o), _p(lse), int(nthreads))
    if rc:
        raise ValueError("ring_fwd: bad arguments (%d)" % rc)
    return o, lse


def mesh_groups(C, A):
    """A2A and P2P groups of the two-dimensional mesh of C = A*R ranks.

    "On Context Parallelism", Peer-to-peer + All-to-all: A2A groups are runs of
    A consecutive ranks, P2P groups take one rank of each A2A group (stride
    A); P2P group a handles heads [a*N/A, (a+1)*N/A).
    Returns (a2a_groups, p2p_groups), lists of rank lists.
    """
    if A < 1 or C % A:
        raise ValueError("mesh_groups: A must divide C")
    R = C // A
    a2a = [[g * A + a for a in range(A)] for g in range(R)]
    p2p = [[g * A + a for g in range(R)] for a in range(A)]
    return a2a, p2p


def mesh_fwd(q_sh, k_sh, v_sh, pos, A, scale=None, nthreads=1):
    """A2A x P2P forward over C = A*R ranks -> (o_sh [C,B,s,N,D], lse_h [R,A,B,N/A,S/R]).

    "On Context Parallelism", Peer-to-peer + All-to-all, in the order the page
    composes it: (1) inside each A2A group, sequence-to-heads all-to-all of q,
    k and v (rank order, N/A heads per rank, S/R positions); (2) the positions
    of the group's shards concatenated in rank order; (3) the peer-to-peer
    ring forward of each P2P group on those tensors and positions; (4) the
    heads-to-sequence all-to-all of the output inside each A2A group.  The
    lse stays in the head-sharded layout of step (3).
    """
    q_sh, k_sh, v_sh = _f64(q_sh), _f64(k_sh), _f64(v_sh)
    pos = _i32(pos)
    C, B, s, N, D = q_sh.shape
    a2a, p2p = mesh_groups(C, A)
    R = C // A
    # (1) per A2A group g: [A][B][A*s][N/A][D]
    heads = [[ulysses(x[grp[0]:grp[-1] + 1], A, SEQ_TO_HEAD, RANK_ORDER) for grp in a2a] for x in (q_sh, k_sh, v_sh)]
    # (2) positions of each A2A group's shards, concatenated in rank order
    pos_long = np.stack([np.concatenate([pos[c] for c in grp]) for grp in a2a])
    o_h = [None] * R
    lse_h = np.empty((R, A, B, N // A, A * s))
    for a in range(A):
        # (3) ring over P2P group a: ring rank g holds A2A index a of group g
        qr, kr, vr = (np.stack([heads[t][g][a] for g in range(R)]) for t in range(3))
        o_r, l_r = ring_fwd(qr, kr, vr, pos_long, scale=scale, nthreads=nthreads)
        for g in range(R):
            if o_h[g] is None:
                o_h[g] = np.empty((A,) + o_r.shape[1:])
            o_h[g][a] = o_r[g]
            lse_h[g, a] = l_r[g]
    # (4) back to sequence sharding inside each A2A group
    o_sh = np.concatenate([ulysses(o_h[g], A, HEAD_TO_SEQ, RANK_ORDER) for g in range(R)])
    return o_sh, lse_h


def attn_bwd(q, k, v, o, dout, lse, q_pos, k_pos, scale=None, nthreads=1):
    """Backward of one attention tile -> (dq [B,Sq,N,D], dk, dv [B,Sk,Nkv,D]).

    "On Context Parallelism", Peer-to-peer / Backward (attention_tile_backward
    with the final output and lse); the chain rule of the forward definition.
    """
    q, k, v, o, dout, lse = (_f64(x) for x in (q, k, v, o, dout, lse))
    q_pos, k_pos = _i32(q_pos), _i32(k_pos)
    B, Sq, N, D = q.shape
    Sk, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    if _load().orc_attn_bwd(_p(q), _p(k), _p(v), _p(o), _p(dout), _p(lse), _p(q_pos), _p(k_pos), B, Sq, Sk, N, Nkv,
                            D, float(scale), _p(dq), _p(dk), _p(dv), int(nthreads)):
        raise ValueError("attn_bwd: N must be a multiple of Nkv")
    return dq, dk, dv


def attn_bwd_rows(q, k, v, dout, q_pos, k_pos, rows, scale=None, nthreads=1):
    """dq of the chosen query rows -> [B, len(rows), N, D], everything
    (lse, o, delta of each row) recomputed from q, k, v.

    "On Context Parallelism", Peer-to-peer / Backward (tile backward definitions).
    """
    q, k, v, dout = (_f64(x) for x in (q, k, v, dout))
    q_pos, k_pos = _i32(q_pos), _i32(k_pos)
    B, Sq, N, D = q.shape
    Sk, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((B, len(rows), N, D))
    if _load().orc_attn_bwd_rows(_p(q), _p(k), _p(v), _p(dout), _p(q_pos), _p(k_pos), B, Sq, Sk, N, Nkv, D,
                                 float(scale), _p(rows), len(rows), _p(out), int(nthreads)):
        raise ValueError("attn_bwd_rows: bad arguments")
    return out


def attn_bwd_keys(q, k, v, dout, q_pos, k_pos, keys, scale=None, nthreads=1):
    """(dk, dv) of the chosen keys -> [B, len(keys), Nkv, D] each, with every
    query row that sees a key recomputed from q, k, v (cheap for late keys)."""
    q, k, v, dout = (_f64(x) for x in (q, k, v, dout))
    q_pos, k_pos = _i32(q_pos), _i32(k_pos)
    B, Sq, N, D = q.shape
    Sk, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    keys = np.ascontiguousarray(keys, dtype=np.int64)
    dk = np.empty((B, len(keys), Nkv, D))
    dv = np.empty((B, len(keys), Nkv, D))
    if _load().orc_attn_bwd_keys(_p(q), _p(k), _p(v), _p(dout), _p(q_pos), _p(k_pos), B, Sq, Sk, N, Nkv, D,
                                 float(scale), _p(keys), len(keys), _p(dk), _p(dv), int(nthreads)):
        raise ValueError("attn_bwd_keys: bad arguments")
    return dk, dv


def ring_bwd(q_sh, k_sh, v_sh, o_sh, do_sh, lse_sh, pos, scale=None, nthreads=1):
    """Ring backward over C virtual ranks -> (dq_sh, dk_sh, dv_sh), rank-major shards.

    "On Context Parallelism", Peer-to-peer / Backward.
    """
    q_sh, k_sh, v_sh, o_sh, do_sh, lse_sh = (_f64(x) for x in (q_sh, k_sh, v_sh, o_sh, do_sh, lse_sh))
    pos = _i32(pos)
    C, B, s, N, D = q_sh.shape
    Nkv = k_sh.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.empty_like(q_sh)
    dk = np.empty_like(k_sh)
    dv = np.empty_like(v_sh)
    rc = _load().orc_ring_bwd(_p(q_sh), _p(k_sh), _p(v_sh), _p(o_sh), _p(do_sh), _p(lse_sh), _p(pos), B, C * s, N,
                              Nkv, D, C, float(scale), _p(dq), _p(dk), _p(dv), int(nthreads))
    if rc:
        raise ValueError("ring_bwd: bad arguments (%d)" % rc)
    return dq, dk, dv


def pair_counts(pos):
    """Visible (query, key) pairs per (rank, K/V owner): int64 [C, C]."""
    pos = _i32(pos)
    C, s = pos.shape
    out = np.empty((C, C), dtype=np.int64)
    if _load().orc_pair_counts(_p(pos), C * s, C, _p(out)):
        raise ValueError("pair_counts: bad arguments")
    return out
