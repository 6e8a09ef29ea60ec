"""Pins for the fp64 CPU oracle (no GPU).

Each test ties an oracle function to something other than itself: values the
pages print (fixtures under tests/golden, cited there), closed forms, exact
invariants, or brute force on tiny inputs.  A plausible slip in the oracle (a
wrong mask direction, a dropped scale, a swapped chunk, a transposed relayout,
a wrong merge weight) fails at least one of them.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle as O
from golden_io import ints, read

RNG = np.random.default_rng(1234)


def randn(*shape):
    return RNG.standard_normal(shape)


# --------------------------------------------------------------------------
# sharding and positions
# --------------------------------------------------------------------------
def test_zigzag_c4_ownership_and_gathered_order():
    g = read("zigzag_c4.txt")
    C = int(g["C"])
    t = 5
    S = 2 * C * t
    chunk_of_token = (np.arange(S) // t).astype(np.int32).reshape(1, S, 1, 1)
    xs = O.shard(chunk_of_token, C, O.ZIGZAG)  # [C,1,2t,1,1]
    for r in range(C):
        local = xs[r, 0, :, 0, 0]
        owned = [int(local[0]), int(local[t])]
        assert owned == ints(g["owner %d" % r])
        # each owned chunk is a contiguous run of t tokens
        assert (local[:t] == owned[0]).all() and (local[t:] == owned[1]).all()
    # all-gather concatenates each rank's local tensor in rank order
    gathered = xs.reshape(-1)[::t]
    assert gathered.tolist() == ints(g["gathered_order"])


@pytest.mark.parametrize("C", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("layout", [O.ZIGZAG, O.CONTIGUOUS])
def test_shard_is_a_permutation_and_unshard_inverts_it(C, layout):
    B, t, N, D = 2, 3, 2, 4
    S = 2 * C * t
    x = RNG.integers(0, 1 << 30, size=(B, S, N, D)).astype(np.int32)
    xs = O.shard(x, C, layout)
    pos = O.positions(S, C, layout)
    # positions are a permutation of the sequence
    assert sorted(pos.reshape(-1).tolist()) == list(range(S))
    # brute force: every local row is the global row its position names
    for r in range(C):
        for b in range(B):
            for u in range(S // C):
                assert np.array_equal(xs[r, b, u], x[b, pos[r, u]])
    assert np.array_equal(O.unshard(xs, layout), x)


@pytest.mark.parametrize("C", [1, 2, 4, 8])
def test_zigzag_positions_are_two_chunks_r_and_2C_minus_1_minus_r(C):
    t = 4
    S = 2 * C * t
    pos = O.positions(S, C, O.ZIGZAG)
    for r in range(C):
        chunks = (pos[r] // t).tolist()
        assert chunks == [r] * t + [2 * C - 1 - r] * t
        assert (np.diff(pos[r][:t]) == 1).all() and (np.diff(pos[r][t:]) == 1).all()


def test_contiguous_positions():
    pos = O.positions(32, 4, O.CONTIGUOUS)
    assert np.array_equal(pos.reshape(-1), np.arange(32))


def test_rank1_visible_chunks_c4():
    g = read("rank1_visibility_c4.txt")
    C, r = int(g["C"]), int(g["rank"])
    t = 4
    S = 2 * C * t
    pos = O.positions(S, C, O.ZIGZAG)
    all_keys = pos.reshape(-1)
    for qchunk in (r, 2 * C - 1 - r):
        qrows = pos[r][(pos[r] // t) == qchunk]
        # chunks holding at least one key visible to some query of this chunk
        vis = sorted({int(kp // t) for kp in all_keys if (kp <= qrows).any()})
        assert vis == ints(g["query_chunk %d" % qchunk])


def test_divisibility_is_rejected():
    with pytest.raises(ValueError):
        O.positions(30, 4, O.ZIGZAG)  # 30 % 8 != 0
    with pytest.raises(ValueError):
        O.shard(np.zeros((1, 30, 1, 1)), 4, O.ZIGZAG)


# --------------------------------------------------------------------------
# work balance
# --------------------------------------------------------------------------
def _chunk_pairs(S, C):
    """Exact visible pairs between query chunk and key chunk (2C chunks of t)."""
    chunk_pos = O.positions(S, 2 * C, O.CONTIGUOUS)  # row c = positions of chunk c
    return O.pair_counts(chunk_pos)


def test_work_vectors_p4_half_diagonal_units():
    g = read("work_vectors_p4.txt")
    P, t = 4, 64
    S = 2 * P * t
    cp = _chunk_pairs(S, P)
    # chunk-pair units: a full chunk pair is 1, a diagonal (causal) pair rounds to 1/2
    units = np.round(2.0 * cp / (t * t)) / 2.0
    per_chunk = units.sum(axis=1)
    contiguous = [per_chunk[2 * r] + per_chunk[2 * r + 1] for r in range(P)]
    zigzag = [per_chunk[r] + per_chunk[2 * P - 1 - r] for r in range(P)]
    assert contiguous == ints(g["contiguous"])
    assert zigzag == ints(g["zigzag"])


def test_zigzag_exact_pairs_equal_per_rank_and_per_step():
    for C in (2, 4, 8):
        t = 16
        S = 2 * C * t
        pos = O.positions(S, C, O.ZIGZAG)
        pairs = O.pair_counts(pos)
        per_rank = pairs.sum(axis=1)
        assert (per_rank == (2 * C - 1) * t * t + t * (t + 1)).all()
        assert per_rank.sum() == S * (S + 1) // 2
        for r in range(C):
            for j in range(C):
                if j != r:
                    assert pairs[r, j] == 2 * t * t  # every off-diagonal ring step: same work
                else:
                    assert pairs[r, j] == t * t + t * (t + 1)


def test_contiguous_imbalance_table_and_zigzag_units():
    g = read("causal_imbalance.txt")
    for P in (2, 4, 8, 16):
        s = 8
        pos = O.positions(P * s, P, O.CONTIGUOUS)
        pairs = O.pair_counts(pos)
        blocks = (pairs > 0).sum(axis=1)  # key blocks each device must process
        line = g["P %d" % P]
        want_blocks = ints(line.split(";")[0].replace("blocks", ""))
        want_ratio = float(line.split("max_over_mean")[1])
        assert blocks.tolist() == want_blocks
        assert round(blocks.max() / blocks.mean(), 2) == want_ratio
        # exact pairs: r*s^2 + s(s+1)/2
        assert pairs.sum(axis=1).tolist() == [r * s * s + s * (s + 1) // 2 for r in range(P)]
    # zigzag in chunk units with the diagonal counted as 1
    P, t = 4, 16
    cp = _chunk_pairs(2 * P * t, P)
    units = np.ceil(cp / (t * t))
    per_chunk = units.sum(axis=1)
    zz = [per_chunk[r] + per_chunk[2 * P - 1 - r] for r in range(P)]
    assert zz == [int(g["zigzag_units P 4"])] * P


def test_ring_block_counts_contiguous_p4():
    g = read("ring_block_counts_p4.txt")
    P, S = int(g["P"]), int(g["S"])
    pairs = O.pair_counts(O.positions(S, P, O.CONTIGUOUS))
    assert (pairs > 0).sum(axis=1).tolist() == ints(g["counts"])


# --------------------------------------------------------------------------
# Ulysses relayout
# --------------------------------------------------------------------------
def test_ulysses_shapes_from_the_page():
    g = read("ulysses_shapes.txt")
    P, S, H, D = (int(g[k]) for k in ("P", "S", "H", "D"))
    x = randn(P, 1, S // P, H, D)
    y = O.ulysses(x, P, O.SEQ_TO_HEAD, O.RANK_ORDER)
    assert list(x.shape[2:]) == ints(g["input_shape"])
    assert list(y.shape[2:]) == ints(g["attention_shape"])


def test_ulysses_matches_the_pages_all_to_all_semantics():
    """Emulate the page's seq_to_head per source rank (reshape/transpose, then the
    all_to_all that sends group p to rank p) with plain numpy indexing."""
    P, B, s, H, D = 4, 2, 3, 8, 2
    x = RNG.integers(0, 1 << 20, size=(P, B, s, H, D)).astype(np.int64)
    y = O.ulysses(x, P, O.SEQ_TO_HEAD, O.RANK_ORDER)
    for b in range(B):
        # on source rank j: groups[j][p] = heads of group p for j's rows
        groups = [x[j, b].reshape(s, P, H // P, D).transpose(1, 0, 2, 3) for j in range(P)]
        for r in range(P):
            received = np.concatenate([groups[j][r] for j in range(P)], axis=0)  # rank order
            assert np.array_equal(y[r, b], received)
    # head_to_seq is the inverse
    assert np.array_equal(O.ulysses(y, P, O.HEAD_TO_SEQ, O.RANK_ORDER), x)


@pytest.mark.parametrize("order", [O.RANK_ORDER, O.GLOBAL_ORDER])
def test_ulysses_then_per_head_attention_equals_monolithic(order):
    """Ulysses: shard by sequence, relayout to heads, attend the full sequence per
    head group, relayout back -> equals monolithic causal attention."""
    C, B, N, D, t = 2, 1, 4, 8, 6
    S = 2 * C * t
    q, k, v = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    gpos = np.arange(S, dtype=np.int32)
    o_ref, _ = O.attn_direct(q, k, v, gpos, gpos)
    pos = O.positions(S, C, O.ZIGZAG)
    qs, ks, vs = (O.shard(a, C, O.ZIGZAG) for a in (q, k, v))
    qh, kh, vh = (O.ulysses(a, C, O.SEQ_TO_HEAD, order) for a in (qs, ks, vs))
    # positions of the concatenated sequence on every head-group rank
    seq_pos = pos.reshape(-1) if order == O.RANK_ORDER else gpos
    oh = np.empty_like(qh)
    for r in range(C):
        oh[r], _ = O.attn_direct(qh[r], kh[r], vh[r], seq_pos, seq_pos)
    o_sh = O.ulysses(oh, C, O.HEAD_TO_SEQ, order)
    np.testing.assert_allclose(O.unshard(o_sh, O.ZIGZAG), o_ref, rtol=0, atol=1e-13)


def test_ulysses_global_order_is_rank_order_then_unzigzag():
    C, B, s, N, D = 4, 1, 4, 8, 2
    S = C * s
    x = RNG.integers(0, 1 << 20, size=(C, B, s, N, D)).astype(np.int64)
    yr = O.ulysses(x, C, O.SEQ_TO_HEAD, O.RANK_ORDER)
    yg = O.ulysses(x, C, O.SEQ_TO_HEAD, O.GLOBAL_ORDER)
    pos = O.positions(S, C, O.ZIGZAG).reshape(-1)
    for r in range(C):
        assert np.array_equal(yg[r, :, pos], yr[r, :, np.arange(S)])


# --------------------------------------------------------------------------
# attention closed forms
# --------------------------------------------------------------------------
def _arange_pos(S):
    return np.arange(S, dtype=np.int32)


def test_single_visible_key_gives_v0_and_scaled_score():
    B, S, N, D = 1, 5, 2, 8
    q, k, v = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    scale = 0.37
    o, lse = O.attn_direct(q, k, v, _arange_pos(S), _arange_pos(S), scale)
    for h in range(N):
        np.testing.assert_array_equal(o[0, 0, h], v[0, 0, h])
        assert lse[0, h, 0] == pytest.approx(scale * float(q[0, 0, h] @ k[0, 0, h]), abs=1e-14)


def test_v_all_ones_gives_ones_so_weights_sum_to_one():
    B, S, N, D = 2, 17, 3, 4
    q, k = 3 * randn(B, S, N, D), 3 * randn(B, S, N, D)
    o, _ = O.attn_direct(q, k, np.ones((B, S, N, D)), _arange_pos(S), _arange_pos(S))
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def test_zero_query_gives_mean_of_visible_values_and_log_count():
    B, S, N, D = 1, 9, 2, 3
    k, v = randn(B, S, N, D), randn(B, S, N, D)
    o, lse = O.attn_direct(np.zeros((B, S, N, D)), k, v, _arange_pos(S), _arange_pos(S))
    for i in range(S):
        np.testing.assert_allclose(o[0, i], v[0, : i + 1].mean(axis=0), atol=1e-14)
        np.testing.assert_allclose(lse[0, :, i], np.log(i + 1), atol=1e-14)


def test_two_keys_softmax_weights():
    D = 4
    q, k, v = randn(1, 2, 1, D), randn(1, 2, 1, D), np.eye(2)[None, :, None, :]
    v = np.pad(v, ((0, 0), (0, 0), (0, 0), (0, D - 2)))
    scale = 0.5
    o, lse = O.attn_direct(q, k, v, _arange_pos(2), _arange_pos(2), scale)
    s0, s1 = scale * q[0, 1, 0] @ k[0, 0, 0], scale * q[0, 1, 0] @ k[0, 1, 0]
    w1 = 1.0 / (1.0 + np.exp(s0 - s1))
    assert o[0, 1, 0, 1] == pytest.approx(w1, abs=1e-15)
    assert o[0, 1, 0, 0] == pytest.approx(1 - w1, abs=1e-15)
    assert lse[0, 0, 1] == pytest.approx(np.log(np.exp(s0) + np.exp(s1)), abs=1e-14)


def test_mask_uses_positions_equal_positions_visible_and_empty_rows():
    B, S, N, D = 1, 6, 1, 4
    q, k, v = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    # every key strictly after every query: all rows empty -> lse -inf, o = 0
    o, lse = O.attn_direct(q, k, v, np.zeros(S, np.int32), np.ones(S, np.int32))
    assert np.isneginf(lse).all() and (o == 0).all()
    # all positions equal: every key visible to every query (non-causal softmax)
    o, lse = O.attn_direct(q, k, v, np.zeros(S, np.int32), np.zeros(S, np.int32))
    s = (q[0, :, 0] @ k[0, :, 0].T) / np.sqrt(D)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(o[0, :, 0], w @ v[0, :, 0], atol=1e-14)


def test_key_permutation_with_positions_is_invariant():
    B, S, N, D = 1, 12, 2, 4
    q, k, v = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    p = _arange_pos(S)
    o1, l1 = O.attn_direct(q, k, v, p, p)
    perm = RNG.permutation(S)
    o2, l2 = O.attn_direct(q, k[:, perm], v[:, perm], p, p[perm])
    np.testing.assert_allclose(o2, o1, atol=1e-14)
    np.testing.assert_allclose(l2, l1, atol=1e-14)


def test_against_torch_fp64_of_the_pages_attention():
    """The pages' cp_common.attention semantics ([S,H,D], offsets), in torch fp64."""
    S, H, D = 32, 8, 16
    torch.manual_seed(0)
    q, k, v = (torch.randn(S, H, D, dtype=torch.float64) for _ in range(3))
    scores = torch.einsum("qhd,khd->hqk", q, k) / D ** 0.5
    qi = torch.arange(S)[:, None]
    ki = torch.arange(S)[None, :]
    scores = scores.masked_fill(ki > qi, float("-inf"))
    lse_t = torch.logsumexp(scores, dim=-1)
    out_t = torch.einsum("hqk,khd->qhd", torch.exp(scores - lse_t[..., None]), v)
    o, lse = O.attn_direct(q.numpy()[None], k.numpy()[None], v.numpy()[None],
                           _arange_pos(S), _arange_pos(S))
    np.testing.assert_allclose(o[0], out_t.numpy(), atol=1e-13)
    np.testing.assert_allclose(lse[0], lse_t.numpy(), atol=1e-13)


def test_gqa_head_map_equals_expanded_heads():
    B, S, N, Nkv, D = 1, 10, 6, 2, 4
    q, k, v = randn(B, S, N, D), randn(B, S, Nkv, D), randn(B, S, Nkv, D)
    p = _arange_pos(S)
    o1, l1 = O.attn_direct(q, k, v, p, p)
    rep = N // Nkv
    o2, l2 = O.attn_direct(q, np.repeat(k, rep, axis=2), np.repeat(v, rep, axis=2), p, p)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_rows_subset_equals_full():
    B, S, N, D = 1, 40, 2, 8
    q, k, v = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    p = _arange_pos(S)
    o, l = O.attn_direct(q, k, v, p, p, nthreads=3)
    rows = np.array([0, 5, 39, 17])
    orow, lrow = O.attn_rows(q, k, v, p, p, rows, nthreads=2)
    np.testing.assert_array_equal(orow, o[:, rows])
    np.testing.assert_array_equal(lrow, l[:, :, rows])


# --------------------------------------------------------------------------
# blockwise recurrence
# --------------------------------------------------------------------------
@pytest.mark.parametrize("block", [1, 7, 64, 96])
def test_blockwise_equals_direct(block):
    B, S, N, D = 1, 96, 2, 16
    q, k, v = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    p = _arange_pos(S)
    o1, l1 = O.attn_direct(q, k, v, p, p)
    o2, l2 = O.attn_blockwise(q, k, v, p, p, block)
    assert np.max(np.abs(o2 - o1)) <= 1e-12
    assert np.max(np.abs(l2 - l1) / np.maximum(1.0, np.abs(l1))) <= 1e-12


def test_blockwise_with_zigzag_positions_and_empty_blocks():
    C, t, N, D = 4, 8, 1, 8
    S = 2 * C * t
    q, k, v = randn(1, S // C, N, D), randn(1, S, N, D), randn(1, S, N, D)
    pos = O.positions(S, C, O.ZIGZAG)
    qp, kp = pos[2], np.arange(S, dtype=np.int32)
    o1, l1 = O.attn_direct(q, k, v, qp, kp)
    o2, l2 = O.attn_blockwise(q, k, v, qp, kp, 5)
    assert np.max(np.abs(o2 - o1)) <= 1e-12 and np.max(np.abs(l2 - l1)) <= 1e-12


# --------------------------------------------------------------------------
# LSE merge
# --------------------------------------------------------------------------
def _split_partials(q, k, v, qp, kp, parts):
    outs = []
    for idx in parts:
        outs.append(O.attn_direct(q, k[:, idx], v[:, idx], qp, kp[idx]))
    return outs


def test_merge_of_disjoint_key_partials_equals_direct():
    B, S, N, D = 1, 30, 2, 8
    q, k, v = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    p = _arange_pos(S)
    o_ref, l_ref = O.attn_direct(q, k, v, p, p)
    parts = np.array_split(RNG.permutation(S), 3)
    partials = _split_partials(q, k, v, p, p, parts)
    o, l = partials[0]
    for ot, lt in partials[1:]:
        o, l = O.lse_merge(o, l, ot, lt)
    np.testing.assert_allclose(o, o_ref, atol=1e-13)
    np.testing.assert_allclose(l, l_ref, atol=1e-13)


def test_merge_weights_sum_to_one():
    B, Sq, N, D = 1, 7, 2, 3
    la, lt = randn(B, N, Sq) * 4, randn(B, N, Sq) * 4
    o, l = O.lse_merge(np.ones((B, Sq, N, D)), la, np.ones((B, Sq, N, D)), lt)
    np.testing.assert_allclose(o, 1.0, atol=1e-15)
    np.testing.assert_allclose(l, np.logaddexp(la, lt), atol=1e-14)


def test_merge_is_order_independent():
    B, Sq, N, D, R = 1, 5, 2, 4, 4
    parts = [(randn(B, Sq, N, D), randn(B, N, Sq) * 3) for _ in range(R)]
    results = []
    for perm in itertools.permutations(range(R)):
        o, l = parts[perm[0]]
        for i in perm[1:]:
            o, l = O.lse_merge(o, l, *parts[i])
        results.append((o, l))
    # a different bracketing: (0+1) + (2+3)
    o01 = O.lse_merge(*parts[0], *parts[1])
    o23 = O.lse_merge(*parts[2], *parts[3])
    results.append(O.lse_merge(*o01, *o23))
    for o, l in results[1:]:
        np.testing.assert_allclose(o, results[0][0], atol=1e-14)
        np.testing.assert_allclose(l, results[0][1], atol=1e-14)
    # the boxed combine form, symmetric in r by construction
    for i in range(Sq):
        for h in range(N):
            lses = np.array([p[1][0, h, i] for p in parts])
            outs = np.stack([p[0][0, i, h] for p in parts])
            oc, lc = O.combine_row(lses, outs)
            np.testing.assert_allclose(oc, results[0][0][0, i, h], atol=1e-14)
            assert lc == pytest.approx(results[0][1][0, h, i], abs=1e-14)


def test_merge_neg_inf_conventions():
    B, Sq, N, D = 1, 3, 1, 2
    oa, la = randn(B, Sq, N, D), randn(B, N, Sq)
    ot, lt = randn(B, Sq, N, D), np.full((B, N, Sq), -np.inf)
    o, l = O.lse_merge(oa, la, ot, lt)
    assert np.array_equal(o, oa) and np.array_equal(l, la)  # identity
    o, l = O.lse_merge(ot * 0, lt, oa, la)  # empty accumulator takes the tile
    assert np.array_equal(o, oa) and np.array_equal(l, la)
    o, l = O.lse_merge(np.zeros_like(oa), lt, np.zeros_like(oa), lt)
    assert np.isneginf(l).all() and (o == 0).all()


# --------------------------------------------------------------------------
# ring
# --------------------------------------------------------------------------
@pytest.mark.parametrize("C", [1, 2, 4, 8])
@pytest.mark.parametrize("layout", [O.ZIGZAG, O.CONTIGUOUS])
def test_ring_equals_direct(C, layout):
    B, N, Nkv, D, t = 1, 2, 2, 8, 3
    S = 2 * C * t
    q, k, v = randn(B, S, N, D), randn(B, S, Nkv, D), randn(B, S, Nkv, D)
    gp = _arange_pos(S)
    o_ref, l_ref = O.attn_direct(q, k, v, gp, gp)
    pos = O.positions(S, C, layout)
    o_sh, l_sh = O.ring_fwd(O.shard(q, C, layout), O.shard(k, C, layout), O.shard(v, C, layout), pos)
    np.testing.assert_allclose(O.unshard(o_sh, layout), o_ref, atol=1e-13)
    # lse: rank-major [C,B,N,s] -> global [B,N,S]
    l_glob = np.empty_like(l_ref)
    for r in range(C):
        l_glob[:, :, pos[r]] = l_sh[r]
    np.testing.assert_allclose(l_glob, l_ref, atol=1e-13)


# --------------------------------------------------------------------------
# A2A x P2P mesh
# --------------------------------------------------------------------------
def test_mesh_groups_c8_a2_from_the_page():
    g = read("mesh_groups_c8.txt")
    C, A, R = int(g["C"]), int(g["A"]), int(g["R"])
    a2a, p2p = O.mesh_groups(C, A)
    assert len(a2a) == R and len(p2p) == A
    for i in range(R):
        assert a2a[i] == ints(g["a2a_group_%d" % i])
    for a in range(A):
        assert p2p[a] == ints(g["p2p_group_%d" % a])


def test_mesh_head_groups_and_shapes_from_the_page():
    """P2P group a of the C=8, A=2, R=4 example handles heads [a N/2, (a+1) N/2):
    with q carrying its head index and k = 1, every visible score of head h is
    scale*h, so lse - log(#visible) reads the head back out of lse_h."""
    g = read("mesh_groups_c8.txt")
    C, A = int(g["C"]), int(g["A"])
    R = C // A
    B, N, D, t = 1, 4, 4, 1
    S = 2 * C * t
    s = S // C
    q = np.zeros((B, S, N, D))
    q[:, :, :, 0] = np.arange(N)[None, None, :]
    k = np.zeros((B, S, N, D))
    k[..., 0] = 1.0
    v = randn(B, S, N, D)
    pos = O.positions(S, C, O.ZIGZAG)
    _, lse_h = O.mesh_fwd(O.shard(q, C), O.shard(k, C), O.shard(v, C), pos, A)
    assert lse_h.shape == (R, A, B, N // A, S // R)  # each rank: S/R positions, N/A heads, as printed
    scale = 1.0 / np.sqrt(D)
    for a in range(A):
        lo, hi = (int(x) * N // 2 for x in ints(g["p2p_group_%d_heads_halves" % a]))
        for gg in range(R):
            for ap in range(A):
                count = pos[gg * A + ap] + 1.0  # keys at positions 0..p
                got = lse_h[gg, a, 0, :, ap * s:(ap + 1) * s] - np.log(count)[None, :]
                want = scale * np.arange(lo, hi, dtype=np.float64)[:, None] * np.ones((1, s))
                np.testing.assert_allclose(got, want, atol=1e-12)


@pytest.mark.parametrize("C,A", [(4, 1), (4, 2), (4, 4), (8, 2), (8, 4)])
@pytest.mark.parametrize("layout", [O.ZIGZAG, O.CONTIGUOUS])
def test_mesh_equals_direct(C, A, layout):
    """Whatever the mesh shape, the result is causal attention over the whole
    sequence: o by global position, lse mapped from the head-sharded layout."""
    R = C // A
    B, N, D, t = 2, 8, 8, 3
    S = 2 * C * t
    s = S // C
    q, k, v = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    gp = _arange_pos(S)
    o_ref, l_ref = O.attn_direct(q, k, v, gp, gp)
    pos = O.positions(S, C, layout)
    o_sh, lse_h = O.mesh_fwd(O.shard(q, C, layout), O.shard(k, C, layout), O.shard(v, C, layout), pos, A)
    np.testing.assert_allclose(O.unshard(o_sh, layout), o_ref, atol=1e-13)
    nh = N // A
    for g in range(R):
        for a in range(A):
            for ap in range(A):
                rows = pos[g * A + ap]
                got = lse_h[g, a, :, :, ap * s:(ap + 1) * s]
                np.testing.assert_allclose(got, l_ref[:, a * nh:(a + 1) * nh, rows], atol=1e-13)


def test_mesh_with_a1_is_the_ring():
    C, B, N, D, t = 4, 1, 2, 8, 4
    S = 2 * C * t
    q, k, v = (O.shard(randn(B, S, N, D), C) for _ in range(3))
    pos = O.positions(S, C)
    o_m, l_m = O.mesh_fwd(q, k, v, pos, 1)
    o_r, l_r = O.ring_fwd(q, k, v, pos)
    np.testing.assert_array_equal(o_m, o_r)
    np.testing.assert_array_equal(l_m[:, 0], l_r)


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------
def _loss_and_grads(q, k, v, dout, qp, kp, scale):
    """sum(dO * o) and the oracle's gradients of it (o, lse from the forward)."""
    o, lse = O.attn_direct(q, k, v, qp, kp, scale=scale)
    dq, dk, dv = O.attn_bwd(q, k, v, o, dout, lse, qp, kp, scale=scale)
    return float(np.sum(dout * o)), (dq, dk, dv)


@pytest.mark.parametrize("Nkv", [2, 1])
def test_bwd_matches_central_differences_of_the_forward(Nkv):
    """Every gradient entry against a central difference of the oracle's
    FORWARD (sum(dO * o)): independent of the backward's chain rule."""
    B, Sq, Sk, N, D = 1, 5, 6, 2, 3
    q, k, v = randn(B, Sq, N, D), randn(B, Sk, Nkv, D), randn(B, Sk, Nkv, D)
    dout = randn(B, Sq, N, D)
    qp = np.array([3, 0, 5, 2, 7], dtype=np.int32)    # unsorted, one row sees every key
    kp = np.array([1, 0, 4, 2, 6, 3], dtype=np.int32)
    scale = 0.7
    _, grads = _loss_and_grads(q, k, v, dout, qp, kp, scale)
    h = 1e-5
    for x, g in zip((q, k, v), grads):
        num = np.empty_like(x)
        for idx in np.ndindex(*x.shape):
            keep = x[idx]
            x[idx] = keep + h
            lp = float(np.sum(dout * O.attn_direct(q, k, v, qp, kp, scale=scale)[0]))
            x[idx] = keep - h
            lm = float(np.sum(dout * O.attn_direct(q, k, v, qp, kp, scale=scale)[0]))
            x[idx] = keep
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(g, num, atol=1e-8, rtol=1e-7)


def test_bwd_matches_torch_autograd_fp64():
    B, S, N, D = 2, 9, 2, 4
    q, k, v, dout = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    gp = _arange_pos(S)
    o, lse = O.attn_direct(q, k, v, gp, gp)
    dq, dk, dv = O.attn_bwd(q, k, v, o, dout, lse, gp, gp)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    sc = torch.einsum("bind,bjnd->bnij", tq, tk) / np.sqrt(D)
    sc = sc.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    out = torch.einsum("bnij,bjnd->bind", torch.softmax(sc, -1), tv)
    out.backward(torch.tensor(dout))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_bwd_single_visible_key_and_empty_rows():
    """A row that sees one key has p = 1: dv of that key gets dO, dq = dk = 0
    (ds = dp - delta = 0).  A row that sees nothing contributes nothing."""
    B, N, D = 1, 1, 3
    q, k, v = randn(B, 2, N, D), randn(B, 1, N, D), randn(B, 1, N, D)
    dout = randn(B, 2, N, D)
    qp, kp = np.array([5, 1], dtype=np.int32), np.array([4], dtype=np.int32)
    o, lse = O.attn_direct(q, k, v, qp, kp)
    assert lse[0, 0, 1] == -np.inf
    dq, dk, dv = O.attn_bwd(q, k, v, o, dout, lse, qp, kp)
    np.testing.assert_allclose(dv[0, 0], dout[0, 0], atol=1e-15)
    np.testing.assert_allclose(dq, 0.0, atol=1e-15)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)


def test_bwd_delta_identity_and_split_over_key_partials():
    """Gradients split over disjoint key sets add up (the tile backward uses
    the final o and lse), which is what lets the ring sum tile gradients."""
    B, S, N, D = 1, 12, 2, 4
    q, k, v, dout = randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D), randn(B, S, N, D)
    gp = _arange_pos(S)
    o, lse = O.attn_direct(q, k, v, gp, gp)
    full = O.attn_bwd(q, k, v, o, dout, lse, gp, gp)
    idx = [np.array([0, 3, 4, 9]), np.array([1, 2, 5, 6, 7, 8, 10, 11])]
    parts = [O.attn_bwd(q, k[:, ix], v[:, ix], o, dout, lse, gp, gp[ix]) for ix in idx]
    np.testing.assert_allclose(parts[0][0] + parts[1][0], full[0], atol=1e-13)
    for p, ix in zip(parts, idx):
        np.testing.assert_allclose(p[1], full[1][:, ix], atol=1e-13)
        np.testing.assert_allclose(p[2], full[2][:, ix], atol=1e-13)


@pytest.mark.parametrize("C", [1, 2, 4])
@pytest.mark.parametrize("layout", [O.ZIGZAG, O.CONTIGUOUS])
def test_ring_bwd_equals_direct(C, layout):
    B, N, Nkv, D, t = 1, 4, 2, 4, 3
    S = 2 * C * t
    q, k, v = randn(B, S, N, D), randn(B, S, Nkv, D), randn(B, S, Nkv, D)
    dout = randn(B, S, N, D)
    gp = _arange_pos(S)
    o, lse = O.attn_direct(q, k, v, gp, gp)
    dq, dk, dv = O.attn_bwd(q, k, v, o, dout, lse, gp, gp)
    pos = O.positions(S, C, layout)
    o_sh, l_sh = O.ring_fwd(*(O.shard(x, C, layout) for x in (q, k, v)), pos)
    g = O.ring_bwd(*(O.shard(x, C, layout) for x in (q, k, v)), o_sh, O.shard(dout, C, layout), l_sh, pos)
    for got, want in zip(g, (dq, dk, dv)):
        np.testing.assert_allclose(O.unshard(got, layout), want, atol=1e-12)


def test_bwd_sampled_rows_and_keys_equal_full():
    """The sampled-gradient functions (which recompute lse, o and delta per
    row) agree with the full backward on every chosen row and key."""
    B, Sq, Sk, N, Nkv, D = 2, 23, 19, 4, 2, 5
    q, k, v, dout = randn(B, Sq, N, D), randn(B, Sk, Nkv, D), randn(B, Sk, Nkv, D), randn(B, Sq, N, D)
    qp = np.random.default_rng(3).integers(0, 25, Sq).astype(np.int32)
    kp = np.random.default_rng(4).integers(0, 25, Sk).astype(np.int32)
    o, lse = O.attn_direct(q, k, v, qp, kp)
    dq, dk, dv = O.attn_bwd(q, k, v, o, dout, lse, qp, kp)
    rows = [0, 5, 22, 7]
    keys = [18, 0, 3]
    np.testing.assert_allclose(O.attn_bwd_rows(q, k, v, dout, qp, kp, rows, nthreads=3), dq[:, rows], atol=1e-13)
    sk, sv = O.attn_bwd_keys(q, k, v, dout, qp, kp, keys, nthreads=3)
    np.testing.assert_allclose(sk, dk[:, keys], atol=1e-13)
    np.testing.assert_allclose(sv, dv[:, keys], atol=1e-13)
