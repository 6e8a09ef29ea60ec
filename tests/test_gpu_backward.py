"""GPU parity of the attention backward -- the tile backward
(cp_attn_bwd_partial) and the ring backward (cp_ring_attention_bwd) --
against the fp64 oracle, element by element.

Bars.  The pages state no gradient tolerance, so it is derived from the
arithmetic: P and dS enter the tensor cores rounded to bf16 (relative 2^-9
each) and everything else is fp32.  A CPU emulation of exactly those two
roundings on causal S = 1024-2048 problems gives max|err| <= 2.2e-3 max|ref|
and rms(err) <= 1.9e-3 rms(ref) for dq, dk and dv.  The tests allow, per
tensor, max|err| <= 1e-2 max|ref| and rms(err) <= 5e-3 rms(ref).
"""
import math
import zlib

import numpy as np
import pytest
import torch

import cp_synth as SY
import oracle as O
from context_causal_attention_gb300 import ops as F

pytestmark = pytest.mark.gpu

MAX_REL = 1e-2
RMS_REL = 5e-3
NTH = O.default_threads()


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_grad_close(name, got, ref):
    got = f64(got) if torch.is_tensor(got) else got
    assert got.shape == ref.shape, name
    assert np.isfinite(got).all(), name
    amax = np.max(np.abs(ref)) if ref.size else 0.0
    if amax == 0.0:
        assert np.max(np.abs(got)) == 0.0, "%s: expected exact zeros" % name
        return
    err = np.abs(got - ref)
    rms_ref = math.sqrt(float(np.mean(ref * ref)))
    rms_err = math.sqrt(float(np.mean(err * err)))
    assert err.max() <= MAX_REL * amax, "%s: max|err| %g > %g" % (name, err.max(), MAX_REL * amax)
    assert rms_err <= RMS_REL * rms_ref, "%s: rms err %g > %g" % (name, rms_err, RMS_REL * rms_ref)


def rand_bf16(*shape, gen):
    return torch.randn(*shape, generator=gen).to(torch.bfloat16)


def _zz(S, C):
    return O.positions(S, C, O.ZIGZAG)


CASES = {
    "square_d64": dict(B=1, Sq=256, Sk=256, N=2, Nkv=2, D=64, qp=lambda: np.arange(256), kp=lambda: np.arange(256)),
    "causal_d128_multi_tile": dict(B=1, Sq=1024, Sk=1024, N=2, Nkv=2, D=128, qp=lambda: np.arange(1024),
                                   kp=lambda: np.arange(1024)),
    "ragged_gqa_d128": dict(B=2, Sq=200, Sk=333, N=4, Nkv=2, D=128, qp=lambda: np.arange(133, 333),
                            kp=lambda: np.arange(333)),
    "zigzag_r1_owner0": dict(B=1, Sq=256, Sk=256, N=2, Nkv=2, D=64, qp=lambda: _zz(1024, 4)[1],
                             kp=lambda: _zz(1024, 4)[0]),
    "zigzag_r1_owner3_empty_rows": dict(B=1, Sq=256, Sk=256, N=2, Nkv=2, D=128, qp=lambda: _zz(1024, 4)[1],
                                        kp=lambda: _zz(1024, 4)[3]),
    "zigzag_diag": dict(B=1, Sq=512, Sk=512, N=2, Nkv=2, D=128, qp=lambda: _zz(2048, 4)[2],
                        kp=lambda: _zz(2048, 4)[2]),
    "unsorted_positions_gqa": dict(B=1, Sq=300, Sk=500, N=2, Nkv=1, D=64,
                                   qp=lambda: np.random.default_rng(5).integers(0, 500, 300),
                                   kp=lambda: np.random.default_rng(6).permutation(500)),
    "all_masked": dict(B=1, Sq=130, Sk=70, N=1, Nkv=1, D=64, qp=lambda: np.zeros(130), kp=lambda: np.ones(70)),
    "single_row_single_key": dict(B=1, Sq=1, Sk=1, N=1, Nkv=1, D=128, qp=lambda: [5], kp=lambda: [5]),
    "q_over_k_longer": dict(B=1, Sq=640, Sk=256, N=2, Nkv=2, D=64, qp=lambda: np.arange(640),
                            kp=lambda: np.arange(256)),
    "k_over_q_longer_gqa4": dict(B=1, Sq=192, Sk=700, N=4, Nkv=1, D=128, qp=lambda: np.arange(508, 700),
                                 kp=lambda: np.arange(700)),
}


def tile_inputs(name):
    c = CASES[name]
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()) % 1000)
    q = rand_bf16(c["B"], c["Sq"], c["N"], c["D"], gen=g)
    k = rand_bf16(c["B"], c["Sk"], c["Nkv"], c["D"], gen=g)
    v = rand_bf16(c["B"], c["Sk"], c["Nkv"], c["D"], gen=g)
    do = rand_bf16(c["B"], c["Sq"], c["N"], c["D"], gen=g)
    qp = np.asarray(c["qp"](), dtype=np.int32)
    kp = np.asarray(c["kp"](), dtype=np.int32)
    # the tile's "final" output and lse: the attention of this very tile
    o, lse = O.attn_direct(f64(q), f64(k), f64(v), qp, kp, nthreads=NTH)
    return q, k, v, do, qp, kp, o, lse


@pytest.mark.parametrize("name", sorted(CASES))
def test_attn_bwd_partial_vs_oracle(cuda_dev, name):
    q, k, v, do, qp, kp, o, lse = tile_inputs(name)
    ref = O.attn_bwd(f64(q), f64(k), f64(v), o, f64(do), lse, qp, kp, nthreads=NTH)
    dev = cuda_dev
    got = F.cp_attn_bwd_partial(q.to(dev), k.to(dev), v.to(dev), torch.tensor(o, dtype=torch.float32, device=dev),
                                do.to(dev), torch.tensor(lse, dtype=torch.float32, device=dev),
                                torch.as_tensor(qp).to(dev), torch.as_tensor(kp).to(dev))
    torch.cuda.synchronize()
    for nm, g_, r_ in zip(("dq", "dk", "dv"), got, ref):
        assert_grad_close(name + ":" + nm, g_, r_)


def test_attn_bwd_partial_accumulate_and_scale(cuda_dev):
    q, k, v, do, qp, kp, o, lse = tile_inputs("ragged_gqa_d128")
    scale = 0.3
    o, lse = O.attn_direct(f64(q), f64(k), f64(v), qp, kp, scale=scale, nthreads=NTH)
    ref = O.attn_bwd(f64(q), f64(k), f64(v), o, f64(do), lse, qp, kp, scale=scale, nthreads=NTH)
    dev = cuda_dev
    args = (q.to(dev), k.to(dev), v.to(dev), torch.tensor(o, dtype=torch.float32, device=dev), do.to(dev),
            torch.tensor(lse, dtype=torch.float32, device=dev), torch.as_tensor(qp).to(dev),
            torch.as_tensor(kp).to(dev))
    dq, dk, dv = F.cp_attn_bwd_partial(*args, scale=scale)
    F.cp_attn_bwd_partial(*args, scale=scale, dq=dq, dk=dk, dv=dv, accumulate=True)
    torch.cuda.synchronize()
    for nm, g_, r_ in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_grad_close("accumulate:" + nm, g_, 2.0 * r_)


RING = {
    "tiny": (SY.WORKLOADS["tiny"], "zigzag"),
    "s4k": (SY.WORKLOADS["s4k"], "zigzag"),
    "contig_c4": (SY.Workload("rb_contig", B=1, S=1024, N=4, Nkv=4, D=64, C=4, layout="contiguous"), "contiguous"),
    "c8_d128": (SY.Workload("rb_c8", B=1, S=2048, N=2, Nkv=2, D=128, C=8), "zigzag"),
    "gqa_c2": (SY.Workload("rb_gqa", B=2, S=768, N=8, Nkv=4, D=64, C=2), "zigzag"),
    # degenerate one-rank ring, the most virtual ranks one launch takes, and ragged 450-row shards with GQA
    "c1": (SY.Workload("rb_c1", B=1, S=640, N=2, Nkv=2, D=64, C=1), "zigzag"),
    "c64_max": (SY.Workload("rb_c64", B=1, S=8192, N=2, Nkv=1, D=64, C=64), "zigzag"),
    "ragged_gqa_c4": (SY.Workload("rb_rg", B=1, S=1800, N=4, Nkv=2, D=128, C=4), "zigzag"),
    # eight query heads per K/V head: dK, dV of a K/V head sum over all eight
    "gqa8_c2": (SY.Workload("rb_g8", B=1, S=1024, N=16, Nkv=2, D=128, C=2), "zigzag"),
}


def ring_setup(w, layout, dev):
    q, k, v, _ = SY.make_qkv(w)
    g = torch.Generator().manual_seed(17)
    do = rand_bf16(w.B, w.S, w.N, w.D, gen=g)
    lay = F.CP_ZIGZAG if layout == "zigzag" else F.CP_CONTIGUOUS
    lay_o = O.ZIGZAG if layout == "zigzag" else O.CONTIGUOUS
    sh = [F.cp_zigzag_shard(t.to(dev), w.C, lay) for t in (q, k, v, do)]
    pos = F.cp_zigzag_positions(w.S, w.C, lay, device=dev)
    return (q, k, v, do), sh, pos, lay, lay_o


@pytest.mark.parametrize("name", sorted(RING))
def test_ring_bwd_vs_oracle(cuda_dev, name):
    """The ring backward against the oracle's ring backward on the same final
    output and lse (the oracle ring forward's, rounded to fp32)."""
    w, layout = RING[name]
    (q, k, v, do), (qs, ks, vs, dos), pos, lay, lay_o = ring_setup(w, layout, cuda_dev)
    pos_np = pos.cpu().numpy()
    sh64 = [O.shard(f64(t), w.C, lay_o) for t in (q, k, v, do)]
    o_sh, l_sh = O.ring_fwd(sh64[0], sh64[1], sh64[2], pos_np, nthreads=NTH)
    ref = O.ring_bwd(sh64[0], sh64[1], sh64[2], o_sh, sh64[3], l_sh, pos_np, nthreads=NTH)
    got = F.cp_ring_attention_bwd(qs, ks, vs, torch.tensor(o_sh, dtype=torch.float32, device=cuda_dev),
                                  torch.tensor(l_sh, dtype=torch.float32, device=cuda_dev), dos, pos, layout=lay)
    torch.cuda.synchronize()
    for nm, g_, r_ in zip(("dq", "dk", "dv"), got, ref):
        assert_grad_close(name + ":" + nm, g_, r_)


def test_ring_fwd_then_bwd_end_to_end_vs_direct(cuda_dev):
    """GPU ring forward then GPU ring backward, unsharded, against the oracle's
    direct backward of the whole causal attention."""
    w = SY.WORKLOADS["s4k"]
    (q, k, v, do), (qs, ks, vs, dos), pos, lay, lay_o = ring_setup(w, "zigzag", cuda_dev)
    o_sh, l_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=1)
    dq, dk, dv = F.cp_ring_attention_bwd(qs, ks, vs, o_sh, l_sh, dos, pos, layout=lay)
    torch.cuda.synchronize()
    gp = np.arange(w.S, dtype=np.int32)
    q64, k64, v64, do64 = (f64(t) for t in (q, k, v, do))
    o, lse = O.attn_direct(q64, k64, v64, gp, gp, nthreads=NTH)
    ref = O.attn_bwd(q64, k64, v64, o, do64, lse, gp, gp, nthreads=NTH)
    for nm, g_, r_ in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_grad_close("e2e:" + nm, O.unshard(f64(g_), lay_o), r_)
    assert F.cp_device_status() == 0


def test_ring_bwd_full_size_sampled(cuda_dev):
    """S=32768 workload in the benchmark's configuration (ring forward with
    prefetch, then the ring backward): dq of sampled rows and dk / dv of late
    keys against the oracle (which recomputes every row it needs from q, k, v),
    for two heads; and two identities over every key of every head:
    sum_j dv_j = sum_i dO_i (each row's p sums to 1) and sum_j dk_j = 0 (each
    row's ds sums to 0)."""
    w = SY.WORKLOADS["s32k"]
    (q, k, v, do), (qs, ks, vs, dos), pos, lay, lay_o = ring_setup(w, "zigzag", cuda_dev)
    o_sh, l_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=1)
    dq, dk, dv = F.cp_ring_attention_bwd(qs, ks, vs, o_sh, l_sh, dos, pos, layout=lay)
    torch.cuda.synchronize()
    assert F.cp_device_status() == 0
    C, s = w.C, w.S // w.C
    pos_np = pos.cpu().numpy()
    where = np.empty((w.S, 2), dtype=np.int64)  # global position -> (rank, local row)
    for r in range(C):
        where[pos_np[r], 0] = r
        where[pos_np[r], 1] = np.arange(s)
    heads = [0, 17]
    gp = np.arange(w.S, dtype=np.int32)
    sub = [f64(t[:, :, heads]) for t in (q, k, v, do)]
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, 127, 128, 4095, 4096, w.S - 1], rng.integers(0, w.S, 58)]))
    ref_dq = O.attn_bwd_rows(*sub, gp, gp, rows, nthreads=NTH)
    got_dq = np.stack([f64(dq[where[i, 0], :, where[i, 1]][:, heads]) for i in rows], axis=1)
    assert_grad_close("dq rows", got_dq, ref_dq)
    keys = np.arange(w.S - 96, w.S, 3)
    ref_dk, ref_dv = O.attn_bwd_keys(*sub, gp, gp, keys, nthreads=NTH)
    got_dk = np.stack([f64(dk[where[j, 0], :, where[j, 1]][:, heads]) for j in keys], axis=1)
    got_dv = np.stack([f64(dv[where[j, 0], :, where[j, 1]][:, heads]) for j in keys], axis=1)
    assert_grad_close("dk keys", got_dk, ref_dk)
    assert_grad_close("dv keys", got_dv, ref_dv)
    # identities over all keys (N == Nkv here): per (b, head, d)
    sum_dv = dv.double().sum(dim=(0, 2)).cpu().numpy()             # [B, Nkv, D]
    sum_do = dos.double().sum(dim=(0, 2)).cpu().numpy()
    norm_do = np.sqrt((dos.double() ** 2).sum(dim=(0, 2)).cpu().numpy())
    assert np.max(np.abs(sum_dv - sum_do) / norm_do) <= 1e-2
    sum_dk = dk.double().sum(dim=(0, 2)).cpu().numpy()
    norm_dk = np.sqrt((dk.double() ** 2).sum(dim=(0, 2)).cpu().numpy())
    assert np.max(np.abs(sum_dk) / norm_dk) <= 1e-2
