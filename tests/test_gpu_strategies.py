"""GPU parity of the all-gather and all-to-all (Ulysses) forward strategies:
against the fp64 oracle (max|do| <= 2e-2, max|dlse| <= 1e-3) and against the
ring forward on the same shards (<= 1e-3, the ring-vs-monolithic bound)."""
import numpy as np
import pytest
import torch

import cp_synth as SY
import oracle as O
from context_causal_attention_gb300 import ops as F

pytestmark = pytest.mark.gpu

ATOL_O, ATOL_LSE, CROSS = 2e-2, 1e-3, 1e-3
NTH = O.default_threads()


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def setup(w, dev, layout):
    q, k, v, _ = SY.make_qkv(w)
    lay = F.CP_ZIGZAG if layout == "zigzag" else F.CP_CONTIGUOUS
    qs, ks, vs = (F.cp_zigzag_shard(t.to(dev), w.C, lay) for t in (q, k, v))
    pos = F.cp_zigzag_positions(w.S, w.C, lay, device=dev)
    gp = np.arange(w.S, dtype=np.int32)
    o_ref, l_ref = O.attn_direct(f64(q), f64(k), f64(v), gp, gp, nthreads=NTH)
    return (qs, ks, vs, pos, lay), (o_ref, l_ref)


CASES = [
    ("tiny", SY.WORKLOADS["tiny"], "zigzag"),
    ("s4k", SY.WORKLOADS["s4k"], "zigzag"),
    ("contig_c4", SY.Workload("contig_c4", B=1, S=1024, N=8, Nkv=8, D=128, C=4, layout="contiguous"), "contiguous"),
    ("gqa_c2", SY.Workload("gqa_c2", B=2, S=768, N=8, Nkv=4, D=64, C=2), "zigzag"),
]


@pytest.mark.parametrize("name,w,layout", CASES, ids=[c[0] for c in CASES])
def test_allgather_vs_oracle_and_ring(cuda_dev, name, w, layout):
    (qs, ks, vs, pos, lay), (o_ref, l_ref) = setup(w, cuda_dev, layout)
    o_ag, l_ag = F.cp_allgather_attention_fwd(qs, ks, vs, pos, layout=lay)
    o_rg, l_rg = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay)
    torch.cuda.synchronize()
    lay_o = O.ZIGZAG if layout == "zigzag" else O.CONTIGUOUS
    assert np.max(np.abs(O.unshard(f64(o_ag), lay_o) - o_ref)) <= ATOL_O
    pos_np = pos.cpu().numpy()
    l_glob = np.empty_like(l_ref)
    for r in range(w.C):
        l_glob[:, :, pos_np[r]] = f64(l_ag[r])
    assert np.max(np.abs(l_glob - l_ref)) <= ATOL_LSE
    assert torch.max(torch.abs(o_ag - o_rg)).item() <= CROSS
    assert torch.max(torch.abs(l_ag - l_rg)).item() <= CROSS


@pytest.mark.parametrize("name,w,layout", CASES, ids=[c[0] for c in CASES])
def test_ulysses_vs_oracle_and_ring(cuda_dev, name, w, layout):
    if w.N % w.C or w.Nkv % w.C:
        pytest.skip("head counts not divisible by C")
    (qs, ks, vs, pos, lay), (o_ref, l_ref) = setup(w, cuda_dev, layout)
    o_ul, l_h = F.cp_ulysses_attention_fwd(qs, ks, vs, layout=lay)
    o_rg, _ = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay)
    torch.cuda.synchronize()
    lay_o = O.ZIGZAG if layout == "zigzag" else O.CONTIGUOUS
    assert np.max(np.abs(O.unshard(f64(o_ul), lay_o) - o_ref)) <= ATOL_O
    # lse_h [C][B][N/C][S]: head r*N/C + h' in global order
    C, B, nh, S = l_h.shape
    l_glob = f64(l_h).transpose(1, 0, 2, 3).reshape(B, C * nh, S)
    assert np.max(np.abs(l_glob - l_ref)) <= ATOL_LSE
    assert torch.max(torch.abs(o_ul - o_rg)).item() <= CROSS


MESH_CASES = [
    ("c4_a2r2_zigzag", SY.Workload("m1", B=2, S=1024, N=8, Nkv=8, D=64, C=4), 2, "zigzag"),
    ("c8_a2r4_zigzag", SY.Workload("m2", B=1, S=2048, N=4, Nkv=4, D=128, C=8), 2, "zigzag"),
    ("c8_a4r2_contig", SY.Workload("m3", B=1, S=2048, N=8, Nkv=8, D=64, C=8, layout="contiguous"), 4,
     "contiguous"),
    ("c4_a4r1_zigzag", SY.Workload("m4", B=1, S=1024, N=4, Nkv=4, D=64, C=4), 4, "zigzag"),
    ("c4_a1r4_gqa", SY.Workload("m5", B=1, S=1024, N=8, Nkv=4, D=64, C=4), 1, "zigzag"),
]


@pytest.mark.parametrize("name,w,A,layout", MESH_CASES, ids=[c[0] for c in MESH_CASES])
def test_mesh_vs_oracle_and_ring(cuda_dev, name, w, A, layout):
    """A2A x P2P mesh against the oracle's mesh composition (o and the
    head-sharded lse, element by element) and against the plain ring."""
    R = w.C // A
    q, k, v, _ = SY.make_qkv(w)
    lay = F.CP_ZIGZAG if layout == "zigzag" else F.CP_CONTIGUOUS
    lay_o = O.ZIGZAG if layout == "zigzag" else O.CONTIGUOUS
    qs, ks, vs = (F.cp_zigzag_shard(t.to(cuda_dev), w.C, lay) for t in (q, k, v))
    pos = F.cp_zigzag_positions(w.S, w.C, lay, device=cuda_dev)
    o_ref, l_ref = O.mesh_fwd(*(O.shard(f64(t), w.C, lay_o) for t in (q, k, v)), pos.cpu().numpy(), A,
                              nthreads=NTH)
    for prefetch in (0, 1):
        o_m, l_m = F.cp_mesh_attention_fwd(qs, ks, vs, pos, A, R, layout=lay, prefetch=prefetch)
        torch.cuda.synchronize()
        assert np.max(np.abs(f64(o_m) - o_ref)) <= ATOL_O, prefetch
        assert np.max(np.abs(f64(l_m) - l_ref)) <= ATOL_LSE, prefetch
    o_rg, _ = F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay)
    assert torch.max(torch.abs(o_m - o_rg)).item() <= CROSS
