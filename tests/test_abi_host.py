"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects invalid arguments on the host before launching."""
import ctypes

import pytest

from context_causal_attention_gb300 import _lib

FAKE = ctypes.c_void_p(4096)          # aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(4096 + 8)
NULL = None


def test_every_header_symbol_is_exported(cplib):
    names = _lib.header_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(cplib, n), n


def test_status_strings(cplib):
    for code, name in _lib.STATUS_NAMES.items():
        assert cplib.cp_status_string(code).decode().startswith(name)
    assert cplib.cp_version().decode().count(".") == 2


def _attn(cplib, q=FAKE, k=FAKE, v=FAKE, qp=FAKE, kp=FAKE, B=1, Sq=256, Sk=256, N=2, Nkv=2, D=64, scale=0.125,
          o=FAKE, lse=FAKE):
    return cplib.cp_attn_partial(q, k, v, qp, kp, B, Sq, Sk, N, Nkv, D, scale, o, lse, None)


def test_attn_partial_validation(cplib):
    assert _attn(cplib, q=NULL) == 1
    assert _attn(cplib, lse=NULL) == 1
    assert _attn(cplib, D=96) == 7
    assert _attn(cplib, D=256) == 7
    assert _attn(cplib, N=3, Nkv=2) == 3
    assert _attn(cplib, Sq=0) == 2
    assert _attn(cplib, scale=float("nan")) == 10
    assert _attn(cplib, scale=-1.0) == 10
    assert _attn(cplib, q=MISALIGNED) == 5
    assert _attn(cplib, o=ctypes.c_void_p(4096 + 16)) == 5  # o needs 32-byte alignment
    # past the on-chip plan limit the call needs a workspace (cp_attn_partial_ws)
    assert _attn(cplib, Sq=200000, Sk=200000) == 6
    n = ctypes.c_size_t(0)
    assert cplib.cp_attn_workspace_size(1, 256, 256, 2, 2, 64, ctypes.byref(n)) == 0 and n.value == 0
    assert cplib.cp_attn_workspace_size(1, 200000, 200000, 2, 2, 64, ctypes.byref(n)) == 0 and n.value > 0
    need = n.value
    ws = cplib.cp_attn_partial_ws
    wargs = [FAKE, FAKE, FAKE, FAKE, FAKE, 1, 200000, 200000, 2, 2, 64, 0.125, FAKE, FAKE]
    assert ws(*wargs, NULL, 0, None) == 6
    assert ws(*wargs, FAKE, need - 1, None) == 6
    assert ws(*wargs, ctypes.c_void_p(4096 + 128), need, None) == 5  # plan buffer 256-byte aligned
    bad = list(wargs)
    bad[10] = 96
    assert ws(*bad, FAKE, need, None) == 7


def test_shard_validation(cplib):
    f = cplib.cp_zigzag_shard
    assert f(NULL, FAKE, 1, 256, 2, 64, 2, 0, 0, None) == 1
    assert f(FAKE, FAKE, 1, 250, 2, 64, 2, 0, 0, None) == 3   # S % 2C
    assert f(FAKE, FAKE, 1, 251, 2, 64, 5, 0, 1, None) == 3   # S % C (contiguous)
    assert f(FAKE, ctypes.c_void_p(1 << 30), 1, 256, 2, 64, 2, 7, 0, None) == 4  # dtype
    assert f(FAKE, ctypes.c_void_p(1 << 30), 1, 256, 1, 4, 2, 0, 0, None) == 5   # row of 8 bytes
    assert f(FAKE, FAKE, 1, 256, 2, 64, 2, 0, 0, None) == 10  # in/out overlap
    assert cplib.cp_zigzag_unshard(FAKE, MISALIGNED, 1, 256, 2, 64, 2, 0, 0, None) == 5
    # well-formed, but memory the device cannot reach: refused before any launch
    assert f(FAKE, ctypes.c_void_p(1 << 30), 1, 256, 2, 64, 2, 0, 0, None) == 10
    assert cplib.cp_zigzag_unshard(FAKE, ctypes.c_void_p(1 << 30), 1, 256, 2, 64, 2, 0, 0, None) == 10


def test_positions_and_relayout_validation(cplib):
    assert cplib.cp_zigzag_positions(NULL, 256, 2, 0, 0, None) == 1
    assert cplib.cp_zigzag_positions(FAKE, 250, 2, 0, 1, None) == 3
    r = cplib.cp_ulysses_relayout
    assert r(FAKE, ctypes.c_void_p(1 << 30), 1, 4096, 15, 64, 4, 0, 0, 0, None) == 3   # N % C
    assert r(FAKE, ctypes.c_void_p(1 << 30), 1, 4098, 16, 64, 4, 0, 0, 0, None) == 3   # S % C
    assert r(FAKE, ctypes.c_void_p(1 << 30), 1, 4100, 16, 64, 4, 0, 0, 1, None) == 3   # S % 2C, global order
    assert r(FAKE, ctypes.c_void_p(1 << 30), 1, 4096, 16, 64, 4, 0, 5, 0, None) == 10  # direction


def test_positions_host_path_matches_oracle(cplib):
    import numpy as np
    import oracle as O
    for layout in (0, 1):
        for S, C in ((256, 2), (4096, 4), (96, 3) if layout == 1 else (96, 4)):
            pos = np.zeros(S, dtype=np.int32)
            st = cplib.cp_zigzag_positions(pos.ctypes.data_as(ctypes.c_void_p), S, C, layout, 0, None)
            assert st == 0
            assert np.array_equal(pos.reshape(C, S // C), O.positions(S, C, layout))


def test_merge_and_ring_validation(cplib):
    m = cplib.cp_lse_merge
    assert m(NULL, FAKE, FAKE, FAKE, 1, 16, 2, 64, None) == 1
    assert m(FAKE, FAKE, MISALIGNED, FAKE, 1, 16, 2, 64, None) == 5
    n = ctypes.c_size_t(0)
    assert cplib.cp_ring_workspace_size(1, 256, 2, 2, 64, 2, 0, 1, ctypes.byref(n)) == 0
    assert n.value > 0
    need = n.value
    ring = cplib.cp_ring_attention_fwd
    args = [FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 2, 64, 2, 0.125, 0, 0, FAKE, 1, FAKE]
    assert ring(*args, NULL, 0, None) == 6                       # workspace missing
    assert ring(*args, FAKE, need - 1, None) == 6                # workspace too small
    bad = list(args)
    bad[5] = 254                                                 # S % 2C
    assert ring(*bad, FAKE, need, None) == 3
    bad = list(args)
    bad[14] = 9                                                  # o dtype
    assert ring(*bad, FAKE, need, None) == 4
    bad = list(args)
    bad[8] = 80                                                  # D
    assert ring(*bad, FAKE, 1 << 40, None) == 7
    ev = (ctypes.c_void_p * 3)()
    assert cplib.cp_ring_attention_fwd_traced(*args, FAKE, need, None, ev, 3) == 10  # needs 4C events
    # ring flags: unknown bits are refused; the tf32 path is zero copy and merges separately
    PREFETCH, FUSED, TF32 = 1, 2, 4
    for flags, want in [(8, 10), (TF32 | PREFETCH, 7), (TF32 | FUSED, 7)]:
        bad = list(args)
        bad[12] = flags
        assert ring(*bad, FAKE, 1 << 40, None) == want, flags


def test_noalloc_ring_validation_order(cplib):
    """The allocation-free ring runs the ring's own argument checks before its
    scratch-size check, and refuses everything on the host (no CUDA call)."""
    f = cplib.cp_ring_attention_fwd_noalloc
    # q, k, v, pos, B, S, N, Nkv, D, C, scale, layout, o, o_dtype, lse, stream: the s32k workload
    big = [FAKE, FAKE, FAKE, FAKE, 1, 32768, 32, 32, 128, 4, 0.088, 0, FAKE, 1, FAKE, None]
    assert f(*big) == 6                                  # needs more scratch than the array holds
    bad = list(big)
    bad[0] = NULL
    assert f(*bad) == 1                                  # a null pointer is reported as such
    bad = list(big)
    bad[14] = NULL
    assert f(*bad) == 1
    bad = list(big)
    bad[8] = 80
    assert f(*bad) == 7                                  # D
    bad = list(big)
    bad[5] = 32764
    assert f(*bad) == 3                                  # S % 2C
    bad = list(big)
    bad[13] = 9
    assert f(*bad) == 4                                  # o dtype
    bad = list(big)
    bad[12] = MISALIGNED
    assert f(*bad) == 5                                  # fp32 o needs 32-byte alignment


def test_allgather_and_ulysses_validation(cplib):
    n = ctypes.c_size_t(0)
    assert cplib.cp_allgather_workspace_size(1, 256, 2, 2, 64, 2, ctypes.byref(n)) == 0 and n.value > 0
    need_ag = n.value
    ag = cplib.cp_allgather_attention_fwd
    args = [FAKE, FAKE, FAKE, FAKE, 1, 256, 2, 2, 64, 2, 0.125, 0, FAKE, FAKE]
    assert ag(*args, NULL, 0, None) == 6
    assert ag(*args, FAKE, need_ag - 1, None) == 6
    bad = list(args)
    bad[8] = 96
    assert ag(*bad, FAKE, 1 << 40, None) == 7          # D
    bad = list(args)
    bad[5] = 250
    assert ag(*bad, FAKE, 1 << 40, None) == 3          # S % 2C
    bad = list(args)
    bad[0] = NULL
    assert ag(*bad, FAKE, need_ag, None) == 1
    assert cplib.cp_ulysses_workspace_size(1, 256, 4, 4, 64, 2, ctypes.byref(n)) == 0 and n.value > 0
    need_ul = n.value
    ul = cplib.cp_ulysses_attention_fwd
    uargs = [FAKE, FAKE, FAKE, 1, 256, 4, 4, 64, 2, 0.125, 0, FAKE, FAKE]
    assert ul(*uargs, FAKE, need_ul - 1, None) == 6
    bad = list(uargs)
    bad[5] = 3                                          # N % C
    assert ul(*bad, FAKE, 1 << 40, None) == 3
    bad = list(uargs)
    bad[6] = 1                                          # Nkv % C
    assert ul(*bad, FAKE, 1 << 40, None) == 3


def test_mesh_validation(cplib):
    n = ctypes.c_size_t(0)
    # B, S, N, Nkv, D, A, R, flags
    assert cplib.cp_mesh_workspace_size(1, 1024, 8, 8, 64, 2, 2, 1, ctypes.byref(n)) == 0 and n.value > 0
    need = n.value
    assert cplib.cp_mesh_workspace_size(1, 1024, 7, 7, 64, 2, 2, 0, ctypes.byref(n)) == 3   # N % A
    assert cplib.cp_mesh_workspace_size(1, 1024, 8, 8, 64, 2, 2, 4, ctypes.byref(n)) == 10  # tf32: ring only
    assert cplib.cp_mesh_workspace_size(1, 1024, 8, 8, 64, 2, 2, 8, ctypes.byref(n)) == 10  # unknown flag
    mesh = cplib.cp_mesh_attention_fwd
    # q, k, v, pos, B, S, N, Nkv, D, A, R, scale, layout, flags, o, lse
    args = [FAKE, FAKE, FAKE, FAKE, 1, 1024, 8, 8, 64, 2, 2, 0.125, 0, 1, FAKE, FAKE]
    assert mesh(*args, NULL, 0, None) == 6
    assert mesh(*args, FAKE, need - 1, None) == 6
    assert mesh(*args, MISALIGNED, need, None) == 5
    bad = list(args)
    bad[6], bad[7] = 5, 5                               # N % A
    assert mesh(*bad, FAKE, 1 << 40, None) == 3
    bad = list(args)
    bad[7] = 3                                          # Nkv % A
    assert mesh(*bad, FAKE, 1 << 40, None) == 3
    bad = list(args)
    bad[5] = 1004                                       # S % 2C
    assert mesh(*bad, FAKE, 1 << 40, None) == 3
    bad = list(args)
    bad[9], bad[10] = 8, 16                             # A*R > 64
    assert mesh(*bad, FAKE, 1 << 40, None) == 2
    bad = list(args)
    bad[8] = 96                                         # D
    assert mesh(*bad, FAKE, 1 << 40, None) == 7
    bad = list(args)
    bad[13] = 8                                         # flags
    assert mesh(*bad, FAKE, 1 << 40, None) == 10
    bad = list(args)
    bad[3] = NULL
    assert mesh(*bad, FAKE, need, None) == 1


def test_selftest_timeout_range(cplib):
    # q, k, v, pos, o, lse, timeout_ns, stream: the limit is checked before any CUDA call
    assert cplib.cp_selftest_stalled_producer(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == 10
    assert cplib.cp_selftest_stalled_producer(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 999_999, None) == 10
    assert cplib.cp_selftest_stalled_producer(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 3_000_000_000, None) == 10


def test_selftest_kernel_argument_checks(cplib):
    # kernel, scratch, bytes, timeout_ns, stream: all refused before any CUDA call
    big = 512 << 10
    f = cplib.cp_selftest_stalled_kernel
    assert f(3, FAKE, big, 10_000_000, None) == 10          # no such kernel
    assert f(-1, FAKE, big, 10_000_000, None) == 10
    assert f(1, FAKE, big, 999_999, None) == 10             # timeout below 1 ms
    assert f(1, FAKE, big, 3_000_000_000, None) == 10       # above 2 s
    assert f(2, NULL, big, 10_000_000, None) == 1
    assert f(2, ctypes.c_void_p(4096 + 16), big, 10_000_000, None) == 5
    assert f(2, FAKE, big - 1, 10_000_000, None) == 6       # scratch smaller than CP_SELFTEST_SCRATCH_BYTES


def test_binding_refuses_cpu_tensors_before_any_call():
    """The Python binding raises before reaching the library when a tensor that
    must be on the GPU is a CPU tensor (host memory is accepted only where the
    library can check and use it: the shard input, the unshard output, host
    positions)."""
    import pytest
    import torch
    from context_causal_attention_gb300 import ops as F
    q = torch.zeros(1, 128, 2, 64, dtype=torch.bfloat16)
    pos = torch.arange(128, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        F.cp_attn_partial(q, q, q, pos, pos, o=torch.zeros(1, 128, 2, 64), lse=torch.zeros(1, 2, 128))
    with pytest.raises(ValueError, match="CUDA tensor"):
        F.cp_lse_merge(torch.zeros(1, 4, 2, 64), torch.zeros(1, 2, 4), torch.zeros(1, 4, 2, 64), torch.zeros(1, 2, 4))
