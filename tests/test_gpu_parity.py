"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Bars: bit-exact for the permutations and positions; attention max|do| <= 2e-2
and max|dlse| <= 1e-3 against fp64 of the same bf16 inputs; ring output vs
monolithic GPU attention <= 1e-3; merge (fp32 kernel vs fp64 oracle) within
1e-5 relative (a reading: the pages state no merge tolerance, 1e-5 is a few
hundred fp32 ulps of the O(1) weights and values involved).
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

ATOL_O = 2e-2
ATOL_LSE = 1e-3
RING_VS_MONO = 1e-3
MERGE_REL = 1e-5
NTH = O.default_threads()


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def bits(t):
    """Raw bit pattern of a tensor as a numpy integer array."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.numpy()


def rand_bf16(*shape, gen, scale=1.0):
    return (torch.randn(*shape, generator=gen) * scale).to(torch.bfloat16)


def assert_attn_close(o_gpu, lse_gpu, o_ref, lse_ref, atol_o=ATOL_O, atol_lse=ATOL_LSE):
    o_g, l_g = f64(o_gpu), f64(lse_gpu)
    neg = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l_g), neg), "rows with no visible key differ"
    assert (o_g[np.broadcast_to(np.transpose(neg, (0, 2, 1))[..., None], o_g.shape)] == 0).all()
    assert np.isfinite(o_g).all()
    do = np.max(np.abs(o_g - o_ref)) if o_g.size else 0.0
    dl = np.max(np.abs(l_g[~neg] - lse_ref[~neg])) if (~neg).any() else 0.0
    assert do <= atol_o, "max|do| = %g" % do
    assert dl <= atol_lse, "max|dlse| = %g" % dl
    return do, dl


# --------------------------------------------------------------------------
# permutations
# --------------------------------------------------------------------------
SHARD_CASES = [
    # B, S, N, D, C, layout, dtype
    (1, 256, 2, 64, 2, F.CP_ZIGZAG, torch.bfloat16),
    (2, 4096, 16, 64, 4, F.CP_ZIGZAG, torch.bfloat16),
    (2, 4096, 16, 64, 4, F.CP_CONTIGUOUS, torch.bfloat16),
    (3, 96, 3, 8, 3, F.CP_CONTIGUOUS, torch.bfloat16),
    (1, 1024, 5, 4, 8, F.CP_ZIGZAG, torch.float32),
    (2, 48, 1, 8, 1, F.CP_ZIGZAG, torch.bfloat16),
]


@pytest.mark.parametrize("B,S,N,D,C,layout,dtype", SHARD_CASES)
def test_shard_unshard_bit_exact(cuda_dev, B, S, N, D, C, layout, dtype):
    g = torch.Generator().manual_seed(7)
    x = torch.randn(B, S, N, D, generator=g).to(dtype)
    xs = F.cp_zigzag_shard(x.to(cuda_dev), C, layout)
    ref = O.shard(bits(x), C, layout)
    assert np.array_equal(bits(xs), ref)
    back = F.cp_zigzag_unshard(xs, layout)
    assert np.array_equal(bits(back), bits(x))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_shard_unshard_pinned_host_direct(cuda_dev, dtype):
    """Shard straight from pinned host memory and unshard straight into it
    (the kernels cross the host link themselves): bit-identical to the
    device-to-device permutations; pageable host memory is refused."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn(2, 1024, 4, 64, generator=g).to(dtype)
    for layout in (F.CP_ZIGZAG, F.CP_CONTIGUOUS):
        ref = F.cp_zigzag_shard(x.to(cuda_dev), 4, layout)
        sh = F.cp_zigzag_shard(x.pin_memory(), 4, layout, out=torch.empty_like(ref))
        back = torch.empty(x.shape, dtype=dtype).pin_memory()
        F.cp_zigzag_unshard(ref, layout, out=back)
        torch.cuda.synchronize()
        assert np.array_equal(bits(sh), bits(ref))
        assert np.array_equal(bits(back), bits(x))
    with pytest.raises(RuntimeError):
        F.cp_zigzag_shard(x, 4, out=torch.empty_like(ref))  # pageable
    assert F.cp_device_status() == 0


@pytest.mark.parametrize("S,C,layout", [(256, 2, 0), (4096, 4, 0), (131072, 8, 0), (96, 3, 1), (8192, 8, 1)])
def test_positions_device_bit_exact(cuda_dev, S, C, layout):
    pos = F.cp_zigzag_positions(S, C, layout, device=cuda_dev)
    assert np.array_equal(pos.cpu().numpy(), O.positions(S, C, layout))


@pytest.mark.parametrize("C,B,s,N,D,dtype", [
    (4, 2, 1024, 16, 64, torch.bfloat16),   # the S=4096 workload's relayout
    (4, 1, 8, 8, 16, torch.bfloat16),       # the page's Ulysses example (P=4, S=32, H=8, D=16)
    (2, 3, 6, 4, 4, torch.float32),
    (8, 1, 64, 8, 128, torch.bfloat16),
])
@pytest.mark.parametrize("order", [F.CP_RANK_ORDER, F.CP_GLOBAL_ORDER])
def test_ulysses_relayout_bit_exact(cuda_dev, C, B, s, N, D, dtype, order):
    g = torch.Generator().manual_seed(11)
    x = torch.randn(C, B, s, N, D, generator=g).to(dtype)
    y = F.cp_ulysses_relayout(x.to(cuda_dev), C, F.CP_SEQ_TO_HEAD, order)
    assert tuple(y.shape) == (C, B, C * s, N // C, D)
    assert np.array_equal(bits(y), O.ulysses(bits(x), C, O.SEQ_TO_HEAD, order))
    back = F.cp_ulysses_relayout(y, C, F.CP_HEAD_TO_SEQ, order)
    assert np.array_equal(bits(back), bits(x))
    # inverse direction on an independent input
    z = torch.randn(C, B, C * s, N // C, D, generator=g).to(dtype)
    w = F.cp_ulysses_relayout(z.to(cuda_dev), C, F.CP_HEAD_TO_SEQ, order)
    assert np.array_equal(bits(w), O.ulysses(bits(z), C, O.HEAD_TO_SEQ, order))


# --------------------------------------------------------------------------
# LSE merge
# --------------------------------------------------------------------------
# D=64 and D=4: several rows share a warp; D=48: lane groups that do not fill it;
# D=256: two 16-byte pieces per lane and row
@pytest.mark.parametrize("B,Sq,N,D", [(2, 300, 3, 64), (1, 129, 8, 128), (1, 7, 1, 4), (3, 77, 2, 48),
                                      (1, 40, 2, 256)])
def test_lse_merge_vs_oracle(cuda_dev, B, Sq, N, D):
    o_a, l_a, o_t, l_t = SY.merge_inputs(B, Sq, N, D, seed=3, neg_inf_frac=0.3)
    # some accumulator rows empty too, and one row empty on both sides
    l_a[:, :, ::5] = float("-inf")
    l_t[:, :, 0] = float("-inf")
    l_a[:, :, 0] = float("-inf")
    o_ref, l_ref = O.lse_merge(f64(o_a), f64(l_a), f64(o_t), f64(l_t))
    oa, la = o_a.to(cuda_dev), l_a.to(cuda_dev)
    F.cp_lse_merge(oa, la, o_t.to(cuda_dev), l_t.to(cuda_dev))
    og, lg = f64(oa), f64(la)
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.all(np.abs(lg[fin] - l_ref[fin]) <= MERGE_REL * np.maximum(1.0, np.abs(l_ref[fin])))
    assert np.all(np.abs(og - o_ref) <= MERGE_REL * np.maximum(1.0, np.abs(o_ref)))
    # rows with an empty tile are untouched bit for bit
    untouched = np.transpose(np.isneginf(f64(l_t)), (0, 2, 1))
    assert np.array_equal(bits(oa)[untouched], bits(o_a)[untouched])


# --------------------------------------------------------------------------
# partial attention
# --------------------------------------------------------------------------
def run_partial(cuda_dev, q, k, v, qp, kp, scale=None):
    D = q.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    o, lse = F.cp_attn_partial(q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev),
                               torch.as_tensor(qp, dtype=torch.int32).to(cuda_dev),
                               torch.as_tensor(kp, dtype=torch.int32).to(cuda_dev), scale)
    o_ref, l_ref = O.attn_direct(f64(q), f64(k), f64(v), np.asarray(qp), np.asarray(kp), scale, nthreads=NTH)
    return o, lse, o_ref, l_ref


def test_attn_partial_tiny_workload(cuda_dev):
    w = SY.WORKLOADS["tiny"]
    q, k, v, raw = SY.make_qkv(w)
    p = np.arange(w.S, dtype=np.int32)
    o, lse, o_ref, l_ref = run_partial(cuda_dev, q, k, v, p, p)
    do, dl = assert_attn_close(o, lse, o_ref, l_ref)
    # information only: distance to the unrounded fp32 draws
    o32, l32 = O.attn_direct(*(t.numpy().astype(np.float64) for t in raw), p, p)
    print("tiny: max|do|=%.3g max|dlse|=%.3g; vs unrounded fp32 inputs: %.3g %.3g"
          % (do, dl, np.max(np.abs(f64(o) - o32)), np.max(np.abs(f64(lse) - l32))))


def _zz(S, C):
    return O.positions(S, C, O.ZIGZAG)


PARTIAL_CASES = {
    "square_d64": dict(B=1, Sq=256, Sk=256, N=2, Nkv=2, D=64, qp=lambda: np.arange(256), kp=lambda: np.arange(256)),
    "ragged_gqa_d128": dict(B=2, Sq=200, Sk=333, N=4, Nkv=2, D=128, qp=lambda: np.arange(133, 333),
                            kp=lambda: np.arange(333)),
    "zigzag_r1_owner0": dict(B=1, Sq=128, Sk=128, N=2, Nkv=2, D=64, qp=lambda: _zz(512, 4)[1],
                             kp=lambda: _zz(512, 4)[0]),
    "zigzag_r1_owner3_empty_rows": dict(B=1, Sq=128, Sk=128, N=2, Nkv=2, D=128, qp=lambda: _zz(512, 4)[1],
                                        kp=lambda: _zz(512, 4)[3]),
    "zigzag_diag_t256": dict(B=1, Sq=512, Sk=512, N=2, Nkv=2, D=128, qp=lambda: _zz(2048, 4)[2],
                             kp=lambda: _zz(2048, 4)[2]),
    "unsorted_positions": dict(B=1, Sq=300, Sk=500, N=2, Nkv=1, D=64,
                               qp=lambda: np.random.default_rng(5).integers(0, 500, 300),
                               kp=lambda: np.random.default_rng(6).permutation(500)),
    "all_masked": dict(B=1, Sq=130, Sk=70, N=1, Nkv=1, D=64, qp=lambda: np.zeros(130), kp=lambda: np.ones(70)),
    "single_row_single_key": dict(B=1, Sq=1, Sk=1, N=1, Nkv=1, D=128, qp=lambda: [5], kp=lambda: [5]),
    "multi_tile_1024": dict(B=1, Sq=1024, Sk=1024, N=3, Nkv=3, D=128, qp=lambda: np.arange(1024),
                            kp=lambda: np.arange(1024)),
    "q_over_k_longer": dict(B=1, Sq=640, Sk=256, N=2, Nkv=2, D=64, qp=lambda: np.arange(640),
                            kp=lambda: np.arange(256)),
}


@pytest.mark.parametrize("name", sorted(PARTIAL_CASES))
def test_attn_partial_vs_oracle(cuda_dev, name):
    c = PARTIAL_CASES[name]
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()) % 1000)
    q = rand_bf16(c["B"], c["Sq"], c["N"], c["D"], gen=g)
    k = rand_bf16(c["B"], c["Sk"], c["Nkv"], c["D"], gen=g)
    v = rand_bf16(c["B"], c["Sk"], c["Nkv"], c["D"], gen=g)
    qp = np.asarray(c["qp"](), dtype=np.int32)
    kp = np.asarray(c["kp"](), dtype=np.int32)
    o, lse, o_ref, l_ref = run_partial(cuda_dev, q, k, v, qp, kp)
    assert_attn_close(o, lse, o_ref, l_ref)


def test_attn_partial_large_scores_rescale_path(cuda_dev):
    """Score ranges of tens of units force the running-max rescale."""
    g = torch.Generator().manual_seed(99)
    B, S, N, D = 1, 768, 2, 128
    q = rand_bf16(B, S, N, D, gen=g, scale=3.0)
    k = rand_bf16(B, S, N, D, gen=g, scale=3.0)
    # make later keys much stronger so the max grows along the key loop
    k = (k.float() * torch.linspace(0.2, 2.0, S)[None, :, None, None]).to(torch.bfloat16)
    v = rand_bf16(B, S, N, D, gen=g)
    p = np.arange(S, dtype=np.int32)
    o, lse, o_ref, l_ref = run_partial(cuda_dev, q, k, v, p, p)
    assert_attn_close(o, lse, o_ref, l_ref)


def test_attn_partial_scale_argument(cuda_dev):
    g = torch.Generator().manual_seed(4)
    q, k, v = (rand_bf16(1, 200, 2, 64, gen=g) for _ in range(3))
    p = np.arange(200, dtype=np.int32)
    o, lse, o_ref, l_ref = run_partial(cuda_dev, q, k, v, p, p, scale=0.05)
    assert_attn_close(o, lse, o_ref, l_ref)


# --------------------------------------------------------------------------
# ring
# --------------------------------------------------------------------------
def ring_inputs(w, cuda_dev, layout):
    q, k, v, _ = SY.make_qkv(w)
    lay = F.CP_ZIGZAG if layout == "zigzag" else F.CP_CONTIGUOUS
    qs, ks, vs = (F.cp_zigzag_shard(t.to(cuda_dev), w.C, lay) for t in (q, k, v))
    pos = F.cp_zigzag_positions(w.S, w.C, lay, device=cuda_dev)
    return (q, k, v), (qs, ks, vs), pos, lay


@pytest.mark.parametrize("wname,layout", [("tiny", "zigzag"), ("s4k", "zigzag"), ("s4k_contig", "contiguous"),
                                          ("c8", "zigzag"), ("c1", "zigzag"), ("c64_max", "zigzag"),
                                          ("c64_max_contig", "contiguous"), ("ragged_gqa", "zigzag"),
                                          ("gqa8", "zigzag"), ("gqa8_contig", "contiguous")])
def test_ring_vs_oracle(cuda_dev, wname, layout):
    """Every ring mode (zero copy / prefetched K/V rotation x separate / fused
    merge) against the fp64 oracle ring."""
    extra = {
        "s4k_contig": SY.Workload("s4k_contig", B=1, S=1024, N=4, Nkv=4, D=64, C=4, layout="contiguous"),
        "c8": SY.Workload("c8", B=1, S=2048, N=2, Nkv=2, D=128, C=8),
        # degenerate ring (one rank: the monolithic call) and the most virtual ranks one launch takes
        "c1": SY.Workload("c1", B=1, S=640, N=2, Nkv=2, D=64, C=1),
        "c64_max": SY.Workload("c64", B=1, S=8192, N=2, Nkv=1, D=64, C=64),
        "c64_max_contig": SY.Workload("c64c", B=1, S=8192, N=2, Nkv=2, D=128, C=64, layout="contiguous"),
        # 450 rows per rank (a ragged last tile in every shard), two query heads per K/V head
        "ragged_gqa": SY.Workload("rg", B=2, S=1800, N=4, Nkv=2, D=128, C=4),
        # eight query heads per K/V head (query head h reads K/V head h // 8)
        "gqa8": SY.Workload("g8", B=1, S=1024, N=16, Nkv=2, D=128, C=2),
        "gqa8_contig": SY.Workload("g8c", B=2, S=768, N=8, Nkv=1, D=64, C=3, layout="contiguous"),
    }
    w = extra.get(wname) or SY.WORKLOADS[wname]
    (q, k, v), (qs, ks, vs), pos, lay = ring_inputs(w, cuda_dev, layout)
    pos_np = pos.cpu().numpy()
    o_ref, l_ref = O.ring_fwd(*(O.shard(f64(t), w.C, 0 if layout == "zigzag" else 1) for t in (q, k, v)),
                              pos_np, nthreads=NTH)
    for prefetch in (0, 1):
        for fused in (False, True):
            o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=prefetch,
                                                   fused_merge=fused)
            assert np.isfinite(f64(lse_sh)).all()
            assert np.max(np.abs(f64(o_sh) - o_ref)) <= ATOL_O, (prefetch, fused)
            assert np.max(np.abs(f64(lse_sh) - l_ref)) <= ATOL_LSE, (prefetch, fused)


def test_ring_vs_monolithic_gpu_and_bf16_output(cuda_dev):
    w = SY.WORKLOADS["s4k"]
    (q, k, v), (qs, ks, vs), pos, lay = ring_inputs(w, cuda_dev, "zigzag")
    o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=1)
    gp = torch.arange(w.S, dtype=torch.int32, device=cuda_dev)
    o_m, l_m = F.cp_attn_partial(q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev), gp, gp)
    o_ring = F.cp_zigzag_unshard(o_sh, lay)
    assert torch.max(torch.abs(o_ring - o_m)).item() <= RING_VS_MONO
    o_fu, l_fu = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=1, fused_merge=True)
    assert torch.max(torch.abs(F.cp_zigzag_unshard(o_fu, lay) - o_m)).item() <= RING_VS_MONO
    assert torch.max(torch.abs(l_fu - lse_sh)).item() <= RING_VS_MONO
    # lse: rank-major [C,B,N,s] -> [B,N,S] via positions
    l_ring = torch.empty_like(l_m)
    for r in range(w.C):
        l_ring[:, :, pos[r].long()] = lse_sh[r]
    assert torch.max(torch.abs(l_ring - l_m)).item() <= RING_VS_MONO
    # bf16 output = the fp32 result rounded once
    o_bf, l_bf = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=0, o_dtype=F.CP_BF16)
    assert o_bf.dtype == torch.bfloat16
    assert torch.equal(o_bf, o_sh.to(torch.bfloat16))
    assert torch.equal(l_bf, lse_sh)


@pytest.mark.parametrize("fused", [False, True], ids=["separate_merge", "fused_merge"])
def test_ring_vs_monolithic_s32k_all_rows(cuda_dev, fused):
    """Ring output equals attention over the whole sequence ("On Context
    Parallelism", Peer-to-peer / Forward): the S=32768 workload in the
    benchmark's launch configuration (prefetch on) against ONE monolithic
    cp_attn_partial call over all 32768 positions, every row and head compared
    on the device, o and lse, within 1e-3."""
    w = SY.WORKLOADS["s32k"]
    (q, k, v), (qs, ks, vs), pos, lay = ring_inputs(w, cuda_dev, "zigzag")
    gp = torch.arange(w.S, dtype=torch.int32, device=cuda_dev)
    qd, kd, vd = (t.to(cuda_dev) for t in (q, k, v))
    o_m, l_m = F.cp_attn_partial(qd, kd, vd, gp, gp)
    del qd, kd, vd
    o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=1, fused_merge=fused)
    o_ring = F.cp_zigzag_unshard(o_sh, lay)
    del o_sh
    torch.cuda.synchronize()
    assert torch.isfinite(o_ring).all().item() and torch.isfinite(l_m).all().item()
    d_o = torch.max(torch.abs(o_ring - o_m)).item()
    l_ring = torch.empty_like(l_m)
    for r in range(w.C):
        l_ring[:, :, pos[r].long()] = lse_sh[r]
    d_l = torch.max(torch.abs(l_ring - l_m)).item()
    assert d_o <= RING_VS_MONO, "max|o_ring - o_mono| = %g" % d_o
    assert d_l <= RING_VS_MONO, "max|lse_ring - lse_mono| = %g" % d_l


def _inverse_positions(pos_np):
    C, s = pos_np.shape
    inv = np.empty((C * s, 2), dtype=np.int64)
    for r in range(C):
        inv[pos_np[r], 0] = r
        inv[pos_np[r], 1] = np.arange(s)
    return inv


@pytest.mark.parametrize("fused", [True, False], ids=["fused_merge", "separate_merge"])
@pytest.mark.parametrize("wname", ["s32k", "s128k"])
def test_ring_full_size_sampled_rows(cuda_dev, wname, fused):
    """Full-size workloads in the benchmark's launch configuration (prefetch on,
    merge fused into the attention epilogue, fp32 output) and with the separate
    merge; sampled query rows of two heads checked against the oracle."""
    w = SY.WORKLOADS[wname]
    (q, k, v), (qs, ks, vs), pos, lay = ring_inputs(w, cuda_dev, "zigzag")
    o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=1, fused_merge=fused)
    torch.cuda.synchronize()
    assert torch.isfinite(lse_sh).all().item() and torch.isfinite(o_sh).all().item()
    rows = SY.sample_rows(w, n_random=48, edge=2)
    heads = [0, w.N - 1]
    gp = np.arange(w.S, dtype=np.int32)
    o_ref, l_ref = O.attn_rows(f64(q[:, :, heads]), f64(k[:, :, heads]), f64(v[:, :, heads]), gp, gp, rows,
                               nthreads=NTH)
    inv = _inverse_positions(pos.cpu().numpy())
    r_idx = torch.as_tensor(inv[rows, 0], device=cuda_dev)
    u_idx = torch.as_tensor(inv[rows, 1], device=cuda_dev)
    h_idx = torch.as_tensor(heads, device=cuda_dev)
    o_g = f64(o_sh[r_idx, 0, u_idx][:, h_idx])        # [rows, heads, D]
    l_g = f64(lse_sh[r_idx, 0, :, u_idx][:, h_idx])    # [rows, heads]
    assert np.max(np.abs(o_g - o_ref[0])) <= ATOL_O
    assert np.max(np.abs(l_g - l_ref[0].T)) <= ATOL_LSE


def _pairs_blocks(C, Sq, B, N):
    """The kernel pairs query blocks u and nqb-1-u into one work item when that
    still leaves at least 8 rounds of items over the SMs."""
    nqb = ((Sq + 127) // 128 + 1) // 2
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return nqb >= 2 and C * ((nqb + 1) // 2) * B * N >= 8 * sms


def test_attn_partial_paired_blocks_gqa_ragged(cuda_dev):
    """A launch large enough for paired query blocks, with 13 query heads per
    K/V head, ragged Sq / Sk and an odd number of 256-row blocks (the middle
    block is unpaired); causal positions; sampled rows of every block and head
    against the oracle."""
    B, Sq, Sk, N, Nkv, D = 2, 2800, 2900, 104, 8, 128
    assert _pairs_blocks(1, Sq, B, N)
    g = torch.Generator().manual_seed(41)
    q = rand_bf16(B, Sq, N, D, gen=g)
    k = rand_bf16(B, Sk, Nkv, D, gen=g)
    v = rand_bf16(B, Sk, Nkv, D, gen=g)
    qp = np.arange(Sk - Sq, Sk, dtype=np.int32)
    kp = np.arange(Sk, dtype=np.int32)
    scale = 1.0 / math.sqrt(D)
    o, lse = F.cp_attn_partial(q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev), torch.as_tensor(qp).to(cuda_dev),
                               torch.as_tensor(kp).to(cuda_dev), scale)
    rows = np.unique(np.concatenate([np.arange(0, Sq, 23), np.arange(Sq - 3, Sq), [127, 128, 255, 256]]))
    o_ref, l_ref = O.attn_rows(f64(q), f64(k), f64(v), qp, kp, rows, scale, nthreads=NTH)
    r_idx = torch.as_tensor(rows, device=cuda_dev)
    assert np.max(np.abs(f64(o[:, r_idx]) - o_ref)) <= ATOL_O
    assert np.max(np.abs(f64(lse[:, :, r_idx]) - l_ref)) <= ATOL_LSE


def test_ring_paired_blocks_sampled_rows(cuda_dev):
    """Zigzag ring (4 ranks, S=16384, 40 heads) whose launches pair query
    blocks; sampled rows of three heads against the oracle."""
    w = SY.Workload("pairs16k", B=1, S=16384, N=40, Nkv=40, D=128, C=4)
    assert _pairs_blocks(w.C, w.S // w.C, w.B, w.N)
    (q, k, v), (qs, ks, vs), pos, lay = ring_inputs(w, cuda_dev, "zigzag")
    o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=1)
    torch.cuda.synchronize()
    rows = SY.sample_rows(w, n_random=64, edge=2)
    heads = [0, 17, w.N - 1]
    gp = np.arange(w.S, dtype=np.int32)
    o_ref, l_ref = O.attn_rows(f64(q[:, :, heads]), f64(k[:, :, heads]), f64(v[:, :, heads]), gp, gp, rows,
                               nthreads=NTH)
    inv = _inverse_positions(pos.cpu().numpy())
    r_idx = torch.as_tensor(inv[rows, 0], device=cuda_dev)
    u_idx = torch.as_tensor(inv[rows, 1], device=cuda_dev)
    h_idx = torch.as_tensor(heads, device=cuda_dev)
    o_g = f64(o_sh[r_idx, 0, u_idx][:, h_idx])
    l_g = f64(lse_sh[r_idx, 0, :, u_idx][:, h_idx])
    assert np.max(np.abs(o_g - o_ref[0])) <= ATOL_O
    assert np.max(np.abs(l_g - l_ref[0].T)) <= ATOL_LSE


def test_device_status_clean(cuda_dev):
    assert F.cp_device_status(clear=True) == 0


# --------------------------------------------------------------------------
# tf32 input path
# --------------------------------------------------------------------------
# Bars: q, k, v and P enter the tensor cores rounded to the nearest tf32 value
# (10-bit mantissa).  A CPU emulation of exactly that (q, k, v, P rounded, the
# integer running max of the first 64-key tile, the fp32 sum of the unrounded
# P), three seeds on causal S = 256-3072, N(0,1) inputs, gives max|do| <= 1.9e-3
# and max|dlse| <= 7.9e-4 against fp64 of the fp32 inputs; the bars allow about
# twice that.
TF32_ATOL_O = 4e-3
TF32_ATOL_LSE = 2e-3

TF32_CASES = {
    "tiny_fp32_causal": dict(B=1, Sq=256, Sk=256, N=2, Nkv=2, D=64, qp=lambda: np.arange(256), kp=lambda: np.arange(256)),
    "ragged_gqa_d128": dict(B=2, Sq=200, Sk=333, N=4, Nkv=2, D=128, qp=lambda: np.arange(133, 333),
                            kp=lambda: np.arange(333)),
    "zigzag_r1_owner3_empty_rows": dict(B=1, Sq=128, Sk=128, N=2, Nkv=2, D=64, qp=lambda: _zz(512, 4)[1],
                                        kp=lambda: _zz(512, 4)[3]),
    "unsorted_positions": dict(B=1, Sq=300, Sk=500, N=2, Nkv=1, D=64,
                               qp=lambda: np.random.default_rng(5).integers(0, 500, 300),
                               kp=lambda: np.random.default_rng(6).permutation(500)),
    "multi_tile_1024": dict(B=1, Sq=1024, Sk=1024, N=2, Nkv=2, D=128, qp=lambda: np.arange(1024),
                            kp=lambda: np.arange(1024)),
    # items of a single 64-key tile: the K and V^T stages of one tile, nothing streamed after it
    "single_key_tile": dict(B=2, Sq=100, Sk=64, N=3, Nkv=3, D=128, qp=lambda: np.arange(100),
                            kp=lambda: np.arange(64)),
    "single_ragged_key_tile": dict(B=1, Sq=37, Sk=23, N=2, Nkv=1, D=64, qp=lambda: np.arange(37),
                                   kp=lambda: np.arange(23)),
}


@pytest.mark.parametrize("name", sorted(TF32_CASES))
def test_attn_partial_f32_vs_oracle(cuda_dev, name):
    c = TF32_CASES[name]
    g = torch.Generator().manual_seed(zlib.crc32(name.encode()) % 1000)
    q = torch.randn(c["B"], c["Sq"], c["N"], c["D"], generator=g)
    k = torch.randn(c["B"], c["Sk"], c["Nkv"], c["D"], generator=g)
    v = torch.randn(c["B"], c["Sk"], c["Nkv"], c["D"], generator=g)
    qp = np.asarray(c["qp"](), dtype=np.int32)
    kp = np.asarray(c["kp"](), dtype=np.int32)
    o, lse = F.cp_attn_partial_f32(q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev),
                                   torch.as_tensor(qp).to(cuda_dev), torch.as_tensor(kp).to(cuda_dev))
    torch.cuda.synchronize()
    o_ref, l_ref = O.attn_direct(f64(q), f64(k), f64(v), qp, kp, nthreads=NTH)
    assert_attn_close(o, lse, o_ref, l_ref, atol_o=TF32_ATOL_O, atol_lse=TF32_ATOL_LSE)
    assert F.cp_device_status() == 0


def test_attn_partial_f32_paired_tiles_gqa_ragged(cuda_dev):
    """tf32 path on a launch large enough for paired 128-row query tiles (23
    tiles: the middle one unpaired), 13 query heads per K/V head, ragged Sq / Sk,
    causal positions; sampled rows of every tile and head against the oracle."""
    B, Sq, Sk, N, Nkv, D = 2, 2900, 3000, 104, 8, 128
    nqt = (Sq + 127) // 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert nqt % 2 == 1 and ((nqt + 1) // 2) * B * N >= 8 * sms
    g = torch.Generator().manual_seed(43)
    q = torch.randn(B, Sq, N, D, generator=g)
    k = torch.randn(B, Sk, Nkv, D, generator=g)
    v = torch.randn(B, Sk, Nkv, D, generator=g)
    qp = np.arange(Sk - Sq, Sk, dtype=np.int32)
    kp = np.arange(Sk, dtype=np.int32)
    o, lse = F.cp_attn_partial_f32(q.to(cuda_dev), k.to(cuda_dev), v.to(cuda_dev), torch.as_tensor(qp).to(cuda_dev),
                                   torch.as_tensor(kp).to(cuda_dev))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, Sq, 23), np.arange(Sq - 3, Sq), [127, 128, 1407, 1408, 1535, 1536]]))
    o_ref, l_ref = O.attn_rows(f64(q), f64(k), f64(v), qp, kp, rows, nthreads=NTH)
    r_idx = torch.as_tensor(rows, device=cuda_dev)
    assert np.max(np.abs(f64(o[:, r_idx]) - o_ref)) <= TF32_ATOL_O
    assert np.max(np.abs(f64(lse[:, :, r_idx]) - l_ref)) <= TF32_ATOL_LSE
    assert F.cp_device_status() == 0


def test_attn_partial_f32_tiny_workload(cuda_dev):
    """The tiny workload's fp32 draws (no bf16 rounding) through the tf32 path,
    against fp64 of the same fp32 values."""
    w = SY.WORKLOADS["tiny"]
    _, _, _, raw = SY.make_qkv(w)
    q, k, v = (t.to(cuda_dev) for t in raw)
    p = torch.arange(w.S, dtype=torch.int32, device=cuda_dev)
    o, lse = F.cp_attn_partial_f32(q, k, v, p, p)
    torch.cuda.synchronize()
    pn = np.arange(w.S, dtype=np.int32)
    o_ref, l_ref = O.attn_direct(*(f64(t) for t in raw), pn, pn)
    d_o, d_l = assert_attn_close(o, lse, o_ref, l_ref, atol_o=TF32_ATOL_O, atol_lse=TF32_ATOL_LSE)
    print("tiny fp32 via tf32: max|do|=%.3g max|dlse|=%.3g" % (d_o, d_l))


@pytest.mark.parametrize("wname,layout", [("tiny", "zigzag"), ("s4k_contig", "contiguous")])
def test_ring_tf32_vs_oracle(cuda_dev, wname, layout):
    """The ring over fp32 shards (CP_RING_TF32) against the oracle ring on the
    same fp32 values (no bf16 rounding anywhere)."""
    w = {"tiny": SY.WORKLOADS["tiny"],
         "s4k_contig": SY.Workload("s4k_contig_f32", B=1, S=1024, N=4, Nkv=4, D=64, C=4, layout="contiguous")}[wname]
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn(w.B, w.S, w.N, w.D, generator=g) for _ in range(3))
    lay = F.CP_ZIGZAG if layout == "zigzag" else F.CP_CONTIGUOUS
    qs, ks, vs = (F.cp_zigzag_shard(t.to(cuda_dev), w.C, lay) for t in (q, k, v))
    pos = F.cp_zigzag_positions(w.S, w.C, lay, device=cuda_dev)
    o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, tf32=True)
    torch.cuda.synchronize()
    lay_o = O.ZIGZAG if layout == "zigzag" else O.CONTIGUOUS
    o_ref, l_ref = O.ring_fwd(*(O.shard(f64(t), w.C, lay_o) for t in (q, k, v)), pos.cpu().numpy(), nthreads=NTH)
    assert np.max(np.abs(f64(o_sh) - o_ref)) <= TF32_ATOL_O
    assert np.max(np.abs(f64(lse_sh) - l_ref)) <= TF32_ATOL_LSE
    with pytest.raises(F.CpError):
        F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, tf32=True, prefetch=1)
