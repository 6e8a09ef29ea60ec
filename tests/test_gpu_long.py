"""Long sequences: launches whose work plan (per-tile position ranges, tile
counts, work-item order) does not fit in shared memory, so a pre-pass writes it
into the caller's workspace and the kernels read it from there.

Two kinds of check:
  * bit for bit: a ring just past the on-chip limit (32 ranks of 4224 rows)
    against the same ring computed rank by rank with single-rank calls whose
    plans fit on chip (forward, tf32 forward, backward).  Every work item does
    the same arithmetic in the same order whichever plan it came from, so the
    results must be identical;
  * against the oracle: the S=262144 workloads (C=8 and C=16) on sampled rows,
    and the ring against one monolithic call over all 262144 positions
    ("On Context Parallelism", Results and Conclusion: the >= 256K regime;
    Peer-to-peer / Forward: the ring equals attention over the whole sequence).
"""
import math

import numpy as np
import pytest
import torch

import cp_synth as SY
import oracle as O
from context_causal_attention_gb300 import ops as F

pytestmark = pytest.mark.gpu

ATOL_O = 2e-2
ATOL_LSE = 1e-3
RING_VS_MONO = 1e-3
TF32_ATOL_O, TF32_ATOL_LSE = 4e-3, 2e-3  # as in the tf32 parity tests
NTH = O.default_threads()
MAX_TABLES, MAX_PAIRS = 2048, 1024  # the kernels' on-chip plan capacity


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def fwd_plan_on_chip(C, s_q, s_k):
    nqt, nkt = -(-s_q // 128), -(-s_k // 128)
    return C * (nqt + nkt) <= MAX_TABLES and C * ((nqt + 1) // 2) <= MAX_PAIRS


# 32 ranks of 4224 rows (33 tiles, the last one ragged in the query blocks):
# 32 * (33 + 33) = 2112 position tables -> the plan goes to global memory
PAST = SY.Workload("past_limit", B=1, S=32 * 4224, N=2, Nkv=1, D=64, C=32)


def _inputs(w, dev, layout, dtype=torch.bfloat16, seed=3):
    g = torch.Generator().manual_seed(seed)
    lay = F.CP_ZIGZAG if layout == "zigzag" else F.CP_CONTIGUOUS
    q = torch.randn(w.B, w.S, w.N, w.D, generator=g).to(dtype)
    k = torch.randn(w.B, w.S, w.Nkv, w.D, generator=g).to(dtype)
    v = torch.randn(w.B, w.S, w.Nkv, w.D, generator=g).to(dtype)
    qs, ks, vs = (F.cp_zigzag_shard(t.to(dev), w.C, lay) for t in (q, k, v))
    pos = F.cp_zigzag_positions(w.S, w.C, lay, device=dev)
    return (q, k, v), (qs, ks, vs), pos, lay


def _per_rank_ring(qs, ks, vs, pos, partial):
    """The ring's steps rank by rank: step st gives rank r the block of owner
    (r - st) mod C; step 0 writes the accumulator, later steps merge."""
    C = qs.shape[0]
    o = torch.empty(qs.shape, dtype=torch.float32, device=qs.device)
    lse = torch.empty((C, qs.shape[1], qs.shape[3], qs.shape[2]), dtype=torch.float32, device=qs.device)
    for st in range(C):
        for r in range(C):
            j = (r - st) % C
            o_t, l_t = partial(qs[r], ks[j], vs[j], pos[r], pos[j])
            if st == 0:
                o[r].copy_(o_t)
                lse[r].copy_(l_t)
            else:
                F.cp_lse_merge(o[r], lse[r], o_t, l_t)
    return o, lse


@pytest.mark.parametrize("layout", ["zigzag", "contiguous"])
def test_global_plan_ring_fwd_bit_exact_vs_per_rank(cuda_dev, layout):
    w = PAST
    s = w.S // w.C
    assert not fwd_plan_on_chip(w.C, s, s) and fwd_plan_on_chip(1, s, s)
    _, (qs, ks, vs), pos, lay = _inputs(w, cuda_dev, layout)
    o_ring, l_ring = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=0)
    o_ref, l_ref = _per_rank_ring(qs, ks, vs, pos, lambda q, k, v, qp, kp: F.cp_attn_partial(q, k, v, qp, kp))
    torch.cuda.synchronize()
    assert torch.equal(o_ring, o_ref)
    assert torch.equal(l_ring, l_ref)
    # and the other ring modes agree within the ring tolerance
    o_pf, l_pf = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=1, fused_merge=True)
    assert torch.max(torch.abs(o_pf - o_ring)).item() <= RING_VS_MONO
    assert torch.max(torch.abs(l_pf - l_ring)).item() <= RING_VS_MONO
    assert F.cp_device_status() == 0


def test_global_plan_tf32_ring_bit_exact_vs_per_rank(cuda_dev):
    w = PAST
    _, (qs, ks, vs), pos, lay = _inputs(w, cuda_dev, "zigzag", dtype=torch.float32)
    o_ring, l_ring = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, tf32=True)
    o_ref, l_ref = _per_rank_ring(qs, ks, vs, pos,
                                  lambda q, k, v, qp, kp: F.cp_attn_partial_f32(q, k, v, qp, kp))
    torch.cuda.synchronize()
    assert torch.equal(o_ring, o_ref)
    assert torch.equal(l_ring, l_ref)
    assert F.cp_device_status() == 0


def test_global_plan_ring_bwd_bit_exact_vs_per_rank(cuda_dev):
    w = PAST
    _, (qs, ks, vs), pos, lay = _inputs(w, cuda_dev, "zigzag")
    g = torch.Generator().manual_seed(11)
    dos = F.cp_zigzag_shard(torch.randn(w.B, w.S, w.N, w.D, generator=g).to(torch.bfloat16).to(cuda_dev), w.C)
    o_sh, l_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=0)
    dq, dk, dv = F.cp_ring_attention_bwd(qs, ks, vs, o_sh, l_sh, dos, pos, layout=lay)
    C = w.C
    dq_r, dk_r, dv_r = (torch.empty_like(t) for t in (dq, dk, dv))
    for st in range(C):
        for r in range(C):
            j = (r - st) % C
            F.cp_attn_bwd_partial(qs[r], ks[j], vs[j], o_sh[r], dos[r], l_sh[r], pos[r], pos[j],
                                  dq=dq_r[r], dk=dk_r[j], dv=dv_r[j], accumulate=st > 0)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq_r)
    assert torch.equal(dk, dk_r)
    assert torch.equal(dv, dv_r)
    assert F.cp_device_status() == 0


def _inverse_positions(pos_np):
    C, s = pos_np.shape
    inv = np.empty((C * s, 2), dtype=np.int64)
    for r in range(C):
        inv[pos_np[r], 0] = r
        inv[pos_np[r], 1] = np.arange(s)
    return inv


def _sampled_ref(w, q, k, v, heads, n_random=32):
    """Oracle (o, lse) of sampled global rows for the given heads."""
    rows = SY.sample_rows(w, n_random=n_random, edge=1)
    gp = np.arange(w.S, dtype=np.int32)
    o_ref, l_ref = O.attn_rows(f64(q[:, :, heads]), f64(k[:, :, heads]), f64(v[:, :, heads]), gp, gp, rows,
                               nthreads=NTH)
    return rows, heads, o_ref, l_ref


def _check_sampled(ref, pos, o_sh, lse_sh, atol_o, atol_lse):
    rows, heads, o_ref, l_ref = ref
    inv = _inverse_positions(pos.cpu().numpy())
    dev = o_sh.device
    r_idx = torch.as_tensor(inv[rows, 0], device=dev)
    u_idx = torch.as_tensor(inv[rows, 1], device=dev)
    h_idx = torch.as_tensor(heads, device=dev)
    o_g = f64(o_sh[r_idx, 0, u_idx][:, h_idx])
    l_g = f64(lse_sh[r_idx, 0, :, u_idx][:, h_idx])
    do = np.max(np.abs(o_g - o_ref[0]))
    dl = np.max(np.abs(l_g - l_ref[0].T))
    assert do <= atol_o, "max|do| = %g" % do
    assert dl <= atol_lse, "max|dlse| = %g" % dl


@pytest.mark.parametrize("wname", ["s256k", "s256k_c16"])
def test_ring_s256k_sampled_rows(cuda_dev, wname):
    """S=262144, N=8, D=128 with C=8 and C=16: the ring (prefetch on, separate
    and fused merge) on sampled rows of two heads against the oracle."""
    w = SY.WORKLOADS[wname]
    s = w.S // w.C
    assert not fwd_plan_on_chip(w.C, s, s)
    q, k, v, _ = SY.make_qkv(w)
    qs, ks, vs = (F.cp_zigzag_shard(t.to(cuda_dev), w.C) for t in (q, k, v))
    pos = F.cp_zigzag_positions(w.S, w.C, device=cuda_dev)
    ref = _sampled_ref(w, q, k, v, heads=[0, w.N - 1])
    for fused in (False, True):
        o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=1, fused_merge=fused)
        torch.cuda.synchronize()
        assert torch.isfinite(o_sh).all().item() and torch.isfinite(lse_sh).all().item()
        _check_sampled(ref, pos, o_sh, lse_sh, ATOL_O, ATOL_LSE)
        del o_sh, lse_sh
    assert F.cp_device_status() == 0


def test_ring_vs_monolithic_s256k_all_rows(cuda_dev):
    """The S=262144 ring (C=8) against ONE cp_attn_partial over all 262144
    positions (its plan in a caller workspace), every row and head, <= 1e-3."""
    w = SY.WORKLOADS["s256k"]
    assert F.cp_attn_workspace_size(w.B, w.S, w.S, w.N, w.Nkv, w.D) > 0
    q, k, v, _ = SY.make_qkv(w)
    qs, ks, vs = (F.cp_zigzag_shard(t.to(cuda_dev), w.C) for t in (q, k, v))
    pos = F.cp_zigzag_positions(w.S, w.C, device=cuda_dev)
    gp = torch.arange(w.S, dtype=torch.int32, device=cuda_dev)
    qd, kd, vd = (t.to(cuda_dev) for t in (q, k, v))
    o_m, l_m = F.cp_attn_partial(qd, kd, vd, gp, gp)
    del qd, kd, vd
    o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=1)
    o_ring = F.cp_zigzag_unshard(o_sh)
    del o_sh
    l_ring = torch.empty_like(l_m)
    for r in range(w.C):
        l_ring[:, :, pos[r].long()] = lse_sh[r]
    torch.cuda.synchronize()
    d_o = torch.max(torch.abs(o_ring - o_m)).item()
    d_l = torch.max(torch.abs(l_ring - l_m)).item()
    assert d_o <= RING_VS_MONO, "max|o_ring - o_mono| = %g" % d_o
    assert d_l <= RING_VS_MONO, "max|lse_ring - lse_mono| = %g" % d_l
    # the monolithic call itself on sampled rows against the oracle
    rows = SY.sample_rows(w, n_random=16, edge=1)
    heads = [3]
    gp_np = np.arange(w.S, dtype=np.int32)
    o_ref, l_ref = O.attn_rows(f64(q[:, :, heads]), f64(k[:, :, heads]), f64(v[:, :, heads]), gp_np, gp_np, rows,
                               nthreads=NTH)
    r_idx = torch.as_tensor(rows, device=cuda_dev)
    assert np.max(np.abs(f64(o_m[:, r_idx][:, :, heads]) - o_ref)) <= ATOL_O
    assert np.max(np.abs(f64(l_m[:, heads][:, :, r_idx]) - l_ref)) <= ATOL_LSE


def test_tf32_ring_s256k_sampled_rows(cuda_dev):
    """The tf32 ring over fp32 shards at S=262144, C=8, sampled rows of one head
    against the oracle on the same fp32 inputs."""
    w = SY.WORKLOADS["s256k"]
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(w.B, w.S, n, w.D, generator=g) for n in (w.N, w.Nkv, w.Nkv))
    qs, ks, vs = (F.cp_zigzag_shard(t.to(cuda_dev), w.C) for t in (q, k, v))
    pos = F.cp_zigzag_positions(w.S, w.C, device=cuda_dev)
    o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, tf32=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o_sh).all().item()
    _check_sampled(_sampled_ref(w, q, k, v, heads=[5], n_random=16), pos, o_sh, lse_sh, TF32_ATOL_O, TF32_ATOL_LSE)
    assert F.cp_device_status() == 0


def _fwd_rounding_allowance(q, k, v, do, rows, scale):
    """Bound on how far the forward's bf16 rounding of P moves dq of the given
    rows (an error bound in fp64 from the inputs, not an expected value).

    The forward normalises by the fp32 sum of the unrounded P and rounds each
    P to bf16 for P V, so o_i is off by sum_j eps_j p_ij v_j with |eps_j| <=
    2^-8; Delta_i = <dO_i, o_i> is then off by delta_i with |delta_i| <=
    2^-8 sum_j p_ij |dp_ij| (dp_ij = <dO_i, v_j>), and dq_i = scale sum_j
    p_ij (dp_ij - Delta_i) k_j by scale |delta_i| |sum_j p_ij k_j| per
    element.  q, k, v, do: fp64 [S, D] of one head; rows: global positions
    (causal, key j visible to row i iff j <= i).  Returns [rows, D]."""
    out = np.empty((len(rows), q.shape[1]))
    for n, i in enumerate(rows):
        s_ = (k[:i + 1] @ q[i]) * scale
        p = np.exp(s_ - s_.max())
        p /= p.sum()
        dp = v[:i + 1] @ do[i]
        out[n] = scale * 2.0 ** -8 * np.sum(p * np.abs(dp)) * np.abs(p @ k[:i + 1])
    return out


def test_ring_bwd_s256k_sampled(cuda_dev):
    """Ring forward then ring backward at S=262144, C=8: dq of sampled rows and
    dk / dv of late keys of one head against the oracle's exact gradients.

    End to end, the forward's own rounding reaches dq through Delta_i =
    <dO_i, o_i> (see _fwd_rounding_allowance).  It matters on rows that see few
    keys: row 0 sees one key, its exact dq is 0, and the forward's output there
    is v_0 (1 + eps).  The dq bar is the backward bar (1e-2 max|ref|) plus that
    bound; dk and dv of late keys keep the backward bars."""
    from test_gpu_backward import assert_grad_close
    w = SY.WORKLOADS["s256k"]
    q, k, v, _ = SY.make_qkv(w)
    g = torch.Generator().manual_seed(1)
    do = torch.randn(w.B, w.S, w.N, w.D, generator=g).to(torch.bfloat16)
    qs, ks, vs, dos = (F.cp_zigzag_shard(t.to(cuda_dev), w.C) for t in (q, k, v, do))
    pos = F.cp_zigzag_positions(w.S, w.C, device=cuda_dev)
    o_sh, l_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=1)
    dq, dk, dv = F.cp_ring_attention_bwd(qs, ks, vs, o_sh, l_sh, dos, pos)
    torch.cuda.synchronize()
    assert F.cp_device_status() == 0
    inv = _inverse_positions(pos.cpu().numpy())
    heads = [2]
    gp = np.arange(w.S, dtype=np.int32)
    sub = [f64(t[:, :, heads]) for t in (q, k, v, do)]
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([[0, 1, 16383, 16384, w.S - 1], rng.integers(0, w.S, 20)]))
    ref_dq = O.attn_bwd_rows(*sub, gp, gp, rows, nthreads=NTH)[0, :, 0]          # [rows, D]
    got_dq = np.stack([f64(dq[inv[i, 0], 0, inv[i, 1], heads[0]]) for i in rows])
    prop = _fwd_rounding_allowance(*(x[0, :, 0] for x in sub), rows, 1.0 / math.sqrt(w.D))
    err = np.abs(got_dq - ref_dq)
    allow = 1e-2 * np.max(np.abs(ref_dq)) + prop
    assert np.all(err <= allow), "dq rows: worst err / allowance %g" % np.max(err / allow)
    rms = lambda x: math.sqrt(float(np.mean(x * x)))  # noqa: E731
    assert rms(err) <= 5e-3 * rms(ref_dq) + rms(prop)
    keys = np.arange(w.S - 64, w.S, 4)
    ref_dk, ref_dv = O.attn_bwd_keys(*sub, gp, gp, keys, nthreads=NTH)
    got_dk = np.stack([f64(dk[inv[j, 0], :, inv[j, 1]][:, heads]) for j in keys], axis=1)
    got_dv = np.stack([f64(dv[inv[j, 0], :, inv[j, 1]][:, heads]) for j in keys], axis=1)
    assert_grad_close("dk keys", got_dk, ref_dk)
    assert_grad_close("dv keys", got_dv, ref_dv)


def test_allgather_ulysses_mesh_s256k_vs_ring(cuda_dev):
    """The other strategies at S=262144, C=8: all-gather (one launch whose C
    query ranks share one key sequence of 262144 positions: a plan in the
    workspace), Ulysses (one launch over the whole sequence per head group) and
    the 2 x 4 mesh, all against the ring's o (every row and head) <= 1e-3."""
    w = SY.WORKLOADS["s256k"]
    q, k, v, _ = SY.make_qkv(w)
    qs, ks, vs = (F.cp_zigzag_shard(t.to(cuda_dev), w.C) for t in (q, k, v))
    del q, k, v
    pos = F.cp_zigzag_positions(w.S, w.C, device=cuda_dev)
    o_ring, l_ring = F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=1)
    o_ag, l_ag = F.cp_allgather_attention_fwd(qs, ks, vs, pos)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(o_ag - o_ring)).item() <= RING_VS_MONO
    assert torch.max(torch.abs(l_ag - l_ring)).item() <= RING_VS_MONO
    del o_ag, l_ag
    o_ul, _ = F.cp_ulysses_attention_fwd(qs, ks, vs)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(o_ul - o_ring)).item() <= RING_VS_MONO
    del o_ul
    o_me, _ = F.cp_mesh_attention_fwd(qs, ks, vs, pos, 2, 4, prefetch=1)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(o_me - o_ring)).item() <= RING_VS_MONO
    assert F.cp_device_status() == 0


def test_global_plan_unsorted_positions_vs_oracle(cuda_dev):
    """A single call past the on-chip plan limit (1100 query and 1100 key tiles)
    with shuffled key positions and unsorted query positions, so the plan's
    sorted flags are off and every count is a full scan; GQA 2:1.  Sampled rows
    against the oracle, including rows that see no key (lse = -inf, o = 0)."""
    B, Sq, Sk, N, Nkv, D = 1, 1100 * 128, 1100 * 128, 2, 1, 64
    assert F.cp_attn_workspace_size(B, Sq, Sk, N, Nkv, D) > 0
    g = torch.Generator().manual_seed(21)
    q = torch.randn(B, Sq, N, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Sk, Nkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Sk, Nkv, D, generator=g).to(torch.bfloat16)
    rng = np.random.default_rng(22)
    kp = rng.permutation(Sk).astype(np.int32) + 1000   # positions 1000 .. Sk+999, shuffled
    qp = rng.integers(0, Sk + 1000, Sq).astype(np.int32)  # some below 1000: they see nothing
    o, lse = F.cp_attn_partial(q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev), torch.as_tensor(qp).to(cuda_dev),
                               torch.as_tensor(kp).to(cuda_dev))
    torch.cuda.synchronize()
    empty = np.flatnonzero(qp < 1000)[:4]
    rows = np.unique(np.concatenate([rng.integers(0, Sq, 24), empty, [0, Sq - 1]]))
    o_ref, l_ref = O.attn_rows(f64(q), f64(k), f64(v), qp, kp, rows, nthreads=NTH)
    r_idx = torch.as_tensor(rows, device=cuda_dev)
    o_g, l_g = f64(o[:, r_idx]), f64(lse[:, :, r_idx])
    neg = np.isneginf(l_ref)
    assert neg.any() and np.array_equal(np.isneginf(l_g), neg)
    assert np.all(o_g[np.broadcast_to(np.transpose(neg, (0, 2, 1))[..., None], o_g.shape)] == 0)
    assert np.max(np.abs(o_g - o_ref)) <= ATOL_O
    assert np.max(np.abs(l_g[~neg] - l_ref[~neg])) <= ATOL_LSE
    assert F.cp_device_status() == 0
