"""The allocation-free ring entry point, for callers that may not call cudaMalloc.

cp_ring_attention_fwd_noalloc takes its scratch from a fixed-size array inside
the library instead of a caller workspace.  This test calls it through the C
ABI twice in a row (different inputs, so the second call runs over the first
call's leftover scratch) and compares each result with cp_ring_attention_fwd
on the same inputs, within the ring tolerance the other tests use.  It also
checks that sizes needing more scratch than the array holds are refused.

Kept in a file of its own that pytest collects last.
"""
import ctypes
import math

import pytest
import torch

import cp_synth as SY
from context_causal_attention_gb300 import _lib
from context_causal_attention_gb300 import ops as F

pytestmark = pytest.mark.gpu

TOL = 1e-3  # ring tolerance used by the parity tests
SCRATCH_LIMIT = 64 << 20  # CP_NOALLOC_SCRATCH_BYTES in include/cpattn.h


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _inputs(w, dev):
    q, k, v, _ = SY.make_qkv(w)
    qs, ks, vs = (F.cp_zigzag_shard(t.to(dev), w.C) for t in (q, k, v))
    pos = F.cp_zigzag_positions(w.S, w.C, device=dev)
    return qs, ks, vs, pos


def _noalloc(cplib, w, qs, ks, vs, pos, o_dtype, stream):
    C, B, s, N, D = qs.shape
    o = torch.full((C, B, s, N, D), float("nan"), device=qs.device,
                   dtype=torch.float32 if o_dtype == _lib.CP_F32 else torch.bfloat16)
    lse = torch.full((C, B, N, s), float("nan"), device=qs.device)
    st = cplib.cp_ring_attention_fwd_noalloc(_p(qs), _p(ks), _p(vs), _p(pos), B, w.S, N, ks.shape[3], D, C,
                                             1.0 / math.sqrt(D), _lib.CP_ZIGZAG, _p(o), o_dtype, _p(lse),
                                             ctypes.c_void_p(stream))
    assert st == 0, cplib.cp_status_string(st)
    return o, lse


def _with_workspace(cplib, w, qs, ks, vs, pos, o_dtype, stream):
    C, B, s, N, D = qs.shape
    Nkv = ks.shape[3]
    need = ctypes.c_size_t(0)
    assert cplib.cp_ring_workspace_size(B, w.S, N, Nkv, D, C, 0, o_dtype, ctypes.byref(need)) == 0
    ws = torch.empty(max(256, need.value), dtype=torch.uint8, device=qs.device)
    o = torch.empty((C, B, s, N, D), device=qs.device,
                    dtype=torch.float32 if o_dtype == _lib.CP_F32 else torch.bfloat16)
    lse = torch.empty((C, B, N, s), device=qs.device)
    st = cplib.cp_ring_attention_fwd(_p(qs), _p(ks), _p(vs), _p(pos), B, w.S, N, Nkv, D, C, 1.0 / math.sqrt(D),
                                     _lib.CP_ZIGZAG, 0, _p(o), o_dtype, _p(lse), _p(ws), ws.numel(),
                                     ctypes.c_void_p(stream))
    assert st == 0, cplib.cp_status_string(st)
    return o, lse


def test_noalloc_ring_matches_workspace_ring_twice(cplib, cuda_dev):
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(SY.WORKLOADS["s4k"], _lib.CP_F32), (SY.WORKLOADS["tiny"], _lib.CP_BF16)]
    for w, o_dtype in cases:
        qs, ks, vs, pos = _inputs(w, cuda_dev)
        o_ref, l_ref = _with_workspace(cplib, w, qs, ks, vs, pos, o_dtype, stream)
        o, l = _noalloc(cplib, w, qs, ks, vs, pos, o_dtype, stream)
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(l).all()
        assert torch.max(torch.abs(o.float() - o_ref.float())).item() <= TOL
        assert torch.max(torch.abs(l - l_ref)).item() <= TOL


def test_noalloc_rejects_sizes_beyond_its_scratch(cplib, cuda_dev):
    w = SY.WORKLOADS["s32k"]
    need = ctypes.c_size_t(0)
    assert cplib.cp_ring_workspace_size(w.B, w.S, w.N, w.Nkv, w.D, w.C, 0, _lib.CP_F32, ctypes.byref(need)) == 0
    assert need.value > SCRATCH_LIMIT
    fake = ctypes.c_void_p(4096)
    st = cplib.cp_ring_attention_fwd_noalloc(fake, fake, fake, fake, w.B, w.S, w.N, w.Nkv, w.D, w.C, 0.088,
                                             _lib.CP_ZIGZAG, fake, _lib.CP_F32, fake, None)
    assert st == 6  # CP_ERR_WORKSPACE, before anything is enqueued
