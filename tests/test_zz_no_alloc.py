"""The allocation-free ring entry point, for callers that may not call cudaMalloc.

Code running inside a custom allocator's callbacks, runtimes that forbid
allocation after start-up, and processes whose device memory pool belongs to
another framework cannot allocate a workspace for the ring.
cp_ring_attention_fwd_noalloc takes its scratch from a fixed-size array inside
the library instead.  This test calls it through the C ABI twice in a row
(different inputs and sizes, so the second call runs over the first call's
leftover scratch) and checks each result two ways: bit for bit against
cp_ring_attention_fwd on the same inputs (both run the same kernels in the
same order, so any leftover-scratch error shows), and against the fp64 oracle
ring within the attention tolerance the other tests use.  It also checks that
sizes needing more scratch than the array holds are refused.

Kept in a file of its own that pytest collects last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import cp_synth as SY
import oracle as O
from context_causal_attention_gb300 import _lib
from context_causal_attention_gb300 import ops as F

pytestmark = pytest.mark.gpu

ATOL_O = 2e-2    # attention against the fp64 oracle, as in the parity tests
ATOL_LSE = 1e-3
SCRATCH_LIMIT = 64 << 20  # CP_NOALLOC_SCRATCH_BYTES in include/cpattn.h


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


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


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def test_noalloc_ring_matches_workspace_ring_and_oracle_twice(cplib, cuda_dev):
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(SY.WORKLOADS["s4k"], _lib.CP_F32), (SY.WORKLOADS["tiny"], _lib.CP_BF16)]
    for w, o_dtype in cases:
        q, k, v, _ = SY.make_qkv(w)
        qs, ks, vs = (F.cp_zigzag_shard(t.to(cuda_dev), w.C) for t in (q, k, v))
        pos = F.cp_zigzag_positions(w.S, w.C, device=cuda_dev)
        o_ref, l_ref = _with_workspace(cplib, w, qs, ks, vs, pos, o_dtype, stream)
        o, l = _noalloc(cplib, w, qs, ks, vs, pos, o_dtype, stream)
        torch.cuda.synchronize()
        # same kernels, same order, same inputs: the results are identical
        assert torch.equal(o, o_ref), w.name
        assert torch.equal(l, l_ref), w.name
        # and they are the ring attention of the fp64 oracle
        o64, l64 = O.ring_fwd(*(O.shard(_f64(t), w.C) for t in (q, k, v)), pos.cpu().numpy(),
                              nthreads=O.default_threads())
        assert np.max(np.abs(_f64(o) - o64)) <= ATOL_O, w.name
        assert np.max(np.abs(_f64(l) - l64)) <= ATOL_LSE, w.name


def test_noalloc_rejects_sizes_beyond_its_scratch(cplib, cuda_dev):
    w = SY.WORKLOADS["s32k"]
    need = ctypes.c_size_t(0)
    assert cplib.cp_ring_workspace_size(w.B, w.S, w.N, w.Nkv, w.D, w.C, 0, _lib.CP_F32, ctypes.byref(need)) == 0
    assert need.value > SCRATCH_LIMIT
    fake = ctypes.c_void_p(4096)
    st = cplib.cp_ring_attention_fwd_noalloc(fake, fake, fake, fake, w.B, w.S, w.N, w.Nkv, w.D, w.C, 0.088,
                                             _lib.CP_ZIGZAG, fake, _lib.CP_F32, fake, None)
    assert st == 6  # CP_ERR_WORKSPACE, before anything is enqueued
