"""Out-of-bounds writes, checked without a sanitizer: every entry point writes
its outputs and workspace into buffers sized exactly as the header states, with
poisoned guard bytes before and after each one, at ragged sizes (a zigzag chunk
shorter than a tile, chunks that are not a tile multiple, a ring whose work plan
lives in the workspace).  After the call no guard byte may have changed, and no
input may have been modified."""
import ctypes

import numpy as np
import pytest
import torch

import cp_synth as SY
from context_causal_attention_gb300 import _lib
from context_causal_attention_gb300 import ops as F

pytestmark = pytest.mark.gpu

G = 4096        # guard bytes on each side (keeps the buffer 256-byte aligned)
POISON = 0xA5


class Guarded:
    """A device tensor of `shape` and `dtype` inside a poisoned byte buffer."""

    def __init__(self, shape, dtype, dev, fill=None):
        self.n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((G + self.n + G,), POISON, dtype=torch.uint8, device=dev)
        self.t = self.raw[G:G + self.n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        return bool((self.raw[:G] == POISON).all().item()) and bool((self.raw[G + self.n:] == POISON).all().item())


def guarded_ws(nbytes, dev):
    return Guarded((max(nbytes, 256),), torch.uint8, dev)


def rand(shape, gen, dtype=torch.bfloat16):
    return torch.randn(*shape, generator=gen).to(dtype)


def check(*gs):
    for i, g in enumerate(gs):
        assert g.intact(), "guard bytes changed around buffer %d" % i


RING_CASES = {
    # t = 96 < 128: every zigzag chunk shorter than a tile
    "t96": SY.Workload("g_t96", B=1, S=2 * 2 * 96, N=2, Nkv=2, D=64, C=2),
    # t = 200: chunks that are not a tile multiple, GQA, D = 128, odd C
    "t200_gqa": SY.Workload("g_t200", B=2, S=2 * 3 * 200, N=4, Nkv=2, D=128, C=3),
    # the work plan in the workspace (32 ranks x 4224 rows: 2112 position tables)
    "global_plan": SY.Workload("g_plan", B=1, S=32 * 4224, N=2, Nkv=1, D=64, C=32),
}


@pytest.mark.parametrize("name", sorted(RING_CASES))
def test_permutations_and_ring_forward_stay_in_bounds(cuda_dev, name):
    w = RING_CASES[name]
    g = torch.Generator().manual_seed(5)
    C, B, S, N, Nkv, D = w.C, w.B, w.S, w.N, w.Nkv, w.D
    s = S // C
    q, k, v = rand((B, S, N, D), g), rand((B, S, Nkv, D), g), rand((B, S, Nkv, D), g)
    qd, kd, vd = (t.to(cuda_dev) for t in (q, k, v))
    gq, gk, gv = (Guarded((C, B, s, n, D), torch.bfloat16, cuda_dev) for n in (N, Nkv, Nkv))
    F.cp_zigzag_shard(qd, C, out=gq.t)
    F.cp_zigzag_shard(kd, C, out=gk.t)
    F.cp_zigzag_shard(vd, C, out=gv.t)
    gpos = Guarded((C, s), torch.int32, cuda_dev)
    F.cp_zigzag_positions(S, C, out=gpos.t)
    for prefetch, fused in ((0, False), (1, False), (1, True)):
        need = F.cp_ring_workspace_size(B, S, N, Nkv, D, C, prefetch, F.CP_F32, fused)
        ws = guarded_ws(need, cuda_dev)
        go = Guarded((C, B, s, N, D), torch.float32, cuda_dev)
        gl = Guarded((C, B, N, s), torch.float32, cuda_dev)
        F.cp_ring_attention_fwd(gq.t, gk.t, gv.t, gpos.t, prefetch=prefetch, fused_merge=fused,
                                workspace=ws.t[:need] if need else ws.t, o=go.t, lse=gl.t)
        torch.cuda.synchronize()
        check(ws, go, gl)
    # bf16 output (fp32 accumulator in the workspace)
    need = F.cp_ring_workspace_size(B, S, N, Nkv, D, C, 0, F.CP_BF16, False)
    ws = guarded_ws(need, cuda_dev)
    gob = Guarded((C, B, s, N, D), torch.bfloat16, cuda_dev)
    gl = Guarded((C, B, N, s), torch.float32, cuda_dev)
    F.cp_ring_attention_fwd(gq.t, gk.t, gv.t, gpos.t, o_dtype=F.CP_BF16, workspace=ws.t[:need], o=gob.t, lse=gl.t)
    # unshard and relayouts of the shards
    gfull = Guarded((B, S, N, D), torch.bfloat16, cuda_dev)
    F.cp_zigzag_unshard(gq.t, out=gfull.t)
    torch.cuda.synchronize()
    check(ws, gob, gl, gfull, gq, gk, gv, gpos)
    assert torch.equal(gfull.t, qd)
    if N % C == 0:
        gh = Guarded((C, B, S, N // C, D), torch.bfloat16, cuda_dev)
        F.cp_ulysses_relayout(gq.t, C, F.CP_SEQ_TO_HEAD, F.CP_GLOBAL_ORDER, out=gh.t)
        gback = Guarded((C, B, s, N, D), torch.bfloat16, cuda_dev)
        F.cp_ulysses_relayout(gh.t, C, F.CP_HEAD_TO_SEQ, F.CP_GLOBAL_ORDER, out=gback.t)
        torch.cuda.synchronize()
        check(gh, gback)
        assert torch.equal(gback.t, gq.t)
    # inputs untouched
    assert torch.equal(qd, q.to(cuda_dev)) and torch.equal(kd, k.to(cuda_dev))
    assert F.cp_device_status() == 0


def test_partial_merge_tf32_and_backward_stay_in_bounds(cuda_dev):
    g = torch.Generator().manual_seed(6)
    B, Sq, Sk, N, Nkv, D = 2, 200, 333, 4, 2, 128
    dev = cuda_dev
    q, k, v, do = (Guarded(sh, torch.bfloat16, dev, rand(sh, g)) for sh in
                   ((B, Sq, N, D), (B, Sk, Nkv, D), (B, Sk, Nkv, D), (B, Sq, N, D)))
    qp = Guarded((Sq,), torch.int32, dev, torch.arange(Sk - Sq, Sk, dtype=torch.int32))
    kp = Guarded((Sk,), torch.int32, dev, torch.arange(Sk, dtype=torch.int32))
    snap = [x.t.clone() for x in (q, k, v, do, qp, kp)]
    o, l = Guarded((B, Sq, N, D), torch.float32, dev), Guarded((B, N, Sq), torch.float32, dev)
    F.cp_attn_partial(q.t, k.t, v.t, qp.t, kp.t, o=o.t, lse=l.t)
    torch.cuda.synchronize()
    check(o, l)
    # merge of a second partial into the first (in place), against a copy
    o2, l2 = Guarded((B, Sq, N, D), torch.float32, dev), Guarded((B, N, Sq), torch.float32, dev)
    F.cp_attn_partial(q.t, k.t, v.t, qp.t, kp.t, o=o2.t, lse=l2.t)
    F.cp_lse_merge(o.t, l.t, o2.t, l2.t)
    torch.cuda.synchronize()
    check(o, l, o2, l2)
    # tf32 partial (fp32 inputs), workspace exactly as stated
    qf, kf, vf = (Guarded(x.t.shape, torch.float32, dev, x.t.float()) for x in (q, k, v))
    n = ctypes.c_size_t(0)
    assert _lib.lib().cp_attn_f32_workspace_size(B, Sq, Sk, N, Nkv, D, ctypes.byref(n)) == 0
    ws = guarded_ws(n.value, dev)
    of, lf = Guarded((B, Sq, N, D), torch.float32, dev), Guarded((B, N, Sq), torch.float32, dev)
    F.cp_attn_partial_f32(qf.t, kf.t, vf.t, qp.t, kp.t, o=of.t, lse=lf.t, workspace=ws.t[:n.value])
    torch.cuda.synchronize()
    check(ws, of, lf, qf, kf, vf)
    # tile backward, written then accumulated
    assert _lib.lib().cp_attn_bwd_workspace_size(B, Sq, Sk, N, ctypes.byref(n)) == 0
    ws = guarded_ws(n.value, dev)
    dq, dk, dv = (Guarded(sh, torch.float32, dev) for sh in ((B, Sq, N, D), (B, Sk, Nkv, D), (B, Sk, Nkv, D)))
    for acc in (False, True):
        F.cp_attn_bwd_partial(q.t, k.t, v.t, o.t, do.t, l.t, qp.t, kp.t, dq=dq.t, dk=dk.t, dv=dv.t, accumulate=acc,
                              workspace=ws.t[:n.value])
    torch.cuda.synchronize()
    check(ws, dq, dk, dv)
    for x, y in zip((q, k, v, do, qp, kp), snap):
        assert torch.equal(x.t, y)
        assert x.intact()
    assert F.cp_device_status() == 0


@pytest.mark.parametrize("name", ["t96", "t200_gqa", "global_plan"])
def test_ring_backward_and_strategies_stay_in_bounds(cuda_dev, name):
    w = RING_CASES[name]
    g = torch.Generator().manual_seed(7)
    C, B, S, N, Nkv, D = w.C, w.B, w.S, w.N, w.Nkv, w.D
    s = S // C
    dev = cuda_dev
    qs, ks, vs, dos = (F.cp_zigzag_shard(rand((B, S, n, D), g).to(dev), C) for n in (N, Nkv, Nkv, N))
    pos = F.cp_zigzag_positions(S, C, device=dev)
    o_sh, l_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos)
    need = F.cp_ring_bwd_workspace_size(B, S, N, C)
    ws = guarded_ws(need, dev)
    dq, dk, dv = (Guarded(sh, torch.float32, dev) for sh in ((C, B, s, N, D), (C, B, s, Nkv, D), (C, B, s, Nkv, D)))
    F.cp_ring_attention_bwd(qs, ks, vs, o_sh, l_sh, dos, pos, workspace=ws.t[:need], dq=dq.t, dk=dk.t, dv=dv.t)
    torch.cuda.synchronize()
    check(ws, dq, dk, dv)
    L = _lib.lib()
    n = ctypes.c_size_t(0)
    assert L.cp_allgather_workspace_size(B, S, N, Nkv, D, C, ctypes.byref(n)) == 0
    ws = guarded_ws(n.value, dev)
    o, l = Guarded((C, B, s, N, D), torch.float32, dev), Guarded((C, B, N, s), torch.float32, dev)
    F.cp_allgather_attention_fwd(qs, ks, vs, pos, workspace=ws.t[:n.value], o=o.t, lse=l.t)
    torch.cuda.synchronize()
    check(ws, o, l)
    if N % C == 0 and Nkv % C == 0:
        assert L.cp_ulysses_workspace_size(B, S, N, Nkv, D, C, ctypes.byref(n)) == 0
        ws = guarded_ws(n.value, dev)
        o, l = Guarded((C, B, s, N, D), torch.float32, dev), Guarded((C, B, N // C, S), torch.float32, dev)
        F.cp_ulysses_attention_fwd(qs, ks, vs, workspace=ws.t[:n.value], o=o.t, lse=l.t)
        torch.cuda.synchronize()
        check(ws, o, l)
    assert F.cp_device_status() == 0
