"""Python binding of the libcpattn C ABI (same names as include/cpattn.h).

Argument marshalling only: shapes and pointers are read from torch tensors,
outputs are allocated with torch when not given, and the call is enqueued on
the current torch CUDA stream.  All arithmetic happens in the CUDA library.
"""
import ctypes
import math

import torch

from . import _lib
from ._lib import (CP_BF16, CP_CONTIGUOUS, CP_F32, CP_GLOBAL_ORDER, CP_HEAD_TO_SEQ, CP_RANK_ORDER,
                   CP_RING_FUSED_MERGE, CP_RING_PREFETCH, CP_RING_TF32, CP_SEQ_TO_HEAD, CP_ZIGZAG, CpError)

__all__ = [
    "cp_zigzag_shard", "cp_zigzag_unshard", "cp_zigzag_positions", "cp_ulysses_relayout", "cp_attn_partial",
    "cp_attn_workspace_size",
    "cp_lse_merge", "cp_ring_workspace_size", "cp_ring_attention_fwd", "cp_ring_attention_fwd_noalloc",
    "cp_allgather_attention_fwd", "cp_ulysses_attention_fwd",
    "cp_device_status", "cp_version",
    "CP_BF16", "CP_F32", "CP_ZIGZAG", "CP_CONTIGUOUS", "CP_SEQ_TO_HEAD", "CP_HEAD_TO_SEQ", "CP_RANK_ORDER",
    "CP_GLOBAL_ORDER", "CP_RING_PREFETCH", "CP_RING_FUSED_MERGE", "CP_RING_TF32", "CpError",
]

_DT = {torch.bfloat16: CP_BF16, torch.float32: CP_F32}


def _dtype_code(t):
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError("unsupported dtype %s (bf16 or fp32)" % t.dtype)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t, host_ok=False):
    """Raw pointer of a contiguous tensor.  Device tensors only, unless host_ok
    (the library then checks that host memory is pinned and mapped), so a CPU
    tensor never reaches a kernel by mistake."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    if not (t.is_cuda or host_ok):
        raise ValueError("tensor must be a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def cp_version():
    return _lib.lib().cp_version().decode()


def cp_zigzag_shard(x, C, layout=CP_ZIGZAG, out=None, stream=None):
    """x [B,S,N,D] -> rank-major shards [C,B,S/C,N,D] (bit-exact permutation).

    x may be a pinned host tensor: the kernel then reads it across the host
    link (copy and shard in one pass) into `out` on the current CUDA device."""
    B, S, N, D = x.shape
    if out is None:
        dev = x.device if x.is_cuda else torch.device("cuda", torch.cuda.current_device())
        out = torch.empty((C, B, S // C, N, D), dtype=x.dtype, device=dev)
    st = _lib.lib().cp_zigzag_shard(_ptr(x, host_ok=True), _ptr(out), B, S, N, D, C, _dtype_code(x), layout,
                                    _stream(stream))
    _lib.check("cp_zigzag_shard", st)
    return out


def cp_zigzag_unshard(x_sh, layout=CP_ZIGZAG, out=None, stream=None):
    """Rank-major shards [C,B,s,N,D] -> x [B,C*s,N,D] in global order.

    `out` may be a pinned host tensor: the kernel then writes it across the
    host link (unshard and device-to-host copy in one pass)."""
    C, B, s, N, D = x_sh.shape
    if out is None:
        out = torch.empty((B, C * s, N, D), dtype=x_sh.dtype, device=x_sh.device)
    st = _lib.lib().cp_zigzag_unshard(_ptr(x_sh), _ptr(out, host_ok=True), B, C * s, N, D, C, _dtype_code(x_sh),
                                      layout, _stream(stream))
    _lib.check("cp_zigzag_unshard", st)
    return out


def cp_zigzag_positions(S, C, layout=CP_ZIGZAG, device="cuda", out=None, stream=None):
    """int32 [C, S/C] global positions of every local token."""
    dev = torch.device(device)
    if out is None:
        out = torch.empty((C, S // C), dtype=torch.int32, device=dev)
    on_dev = 1 if out.is_cuda else 0
    st = _lib.lib().cp_zigzag_positions(_ptr(out, host_ok=True), S, C, layout, on_dev,
                                        _stream(stream) if on_dev else None)
    _lib.check("cp_zigzag_positions", st)
    return out


def cp_ulysses_relayout(x, C, direction=CP_SEQ_TO_HEAD, order=CP_RANK_ORDER, out=None, stream=None):
    """[C,B,S/C,N,D] <-> [C,B,S,N/C,D] (Ulysses all-to-all as a local permutation)."""
    if direction == CP_SEQ_TO_HEAD:
        Cx, B, s, N, D = x.shape
        S = C * s
        shape = (C, B, S, N // C, D)
    else:
        Cx, B, S, nh, D = x.shape
        N = nh * C
        shape = (C, B, S // C, N, D)
    if Cx != C:
        raise ValueError("leading dimension must be C")
    if out is None:
        out = torch.empty(shape, dtype=x.dtype, device=x.device)
    st = _lib.lib().cp_ulysses_relayout(_ptr(x), _ptr(out), B, S, N, D, C, _dtype_code(x), direction, order,
                                        _stream(stream))
    _lib.check("cp_ulysses_relayout", st)
    return out


def cp_attn_workspace_size(B, Sq, Sk, N, Nkv, D):
    n = ctypes.c_size_t(0)
    _lib.check("cp_attn_workspace_size", _lib.lib().cp_attn_workspace_size(B, Sq, Sk, N, Nkv, D, ctypes.byref(n)))
    return n.value


def cp_attn_partial(q, k, v, q_pos, k_pos, scale=None, o=None, lse=None, workspace=None, stream=None):
    """Partial causal attention -> (o fp32 [B,Sq,N,D], lse fp32 [B,N,Sq]).  Long
    sequences whose work plan does not fit on chip go through cp_attn_partial_ws
    with a workspace (allocated here unless given)."""
    B, Sq, N, D = q.shape
    Sk, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty((B, Sq, N, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, N, Sq), dtype=torch.float32, device=q.device)
    L = _lib.lib()
    need = cp_attn_workspace_size(B, Sq, Sk, N, Nkv, D)
    if need == 0 and workspace is None:
        st = L.cp_attn_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(q_pos), _ptr(k_pos), B, Sq, Sk, N, Nkv, D, float(scale),
                               _ptr(o), _ptr(lse), _stream(stream))
        _lib.check("cp_attn_partial", st)
        return o, lse
    if workspace is None:
        workspace = torch.empty(max(256, need), dtype=torch.uint8, device=q.device)
    st = L.cp_attn_partial_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(q_pos), _ptr(k_pos), B, Sq, Sk, N, Nkv, D, float(scale),
                              _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream(stream))
    _lib.check("cp_attn_partial_ws", st)
    return o, lse


def cp_attn_partial_f32(q, k, v, q_pos, k_pos, scale=None, o=None, lse=None, workspace=None, stream=None):
    """cp_attn_partial for fp32 q, k, v with the tensor cores in tf32 -> (o fp32, lse fp32)."""
    B, Sq, N, D = q.shape
    Sk, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = q.device
    if o is None:
        o = torch.empty((B, Sq, N, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, N, Sq), dtype=torch.float32, device=dev)
    L = _lib.lib()
    n = ctypes.c_size_t(0)
    _lib.check("cp_attn_f32_workspace_size", L.cp_attn_f32_workspace_size(B, Sq, Sk, N, Nkv, D, ctypes.byref(n)))
    if workspace is None:
        workspace = torch.empty(max(256, n.value), dtype=torch.uint8, device=dev)
    st = L.cp_attn_partial_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(q_pos), _ptr(k_pos), B, Sq, Sk, N, Nkv, D, float(scale),
                               _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _lib.check("cp_attn_partial_f32", st)
    return o, lse


def cp_lse_merge(o_acc, lse_acc, o_tile, lse_tile, stream=None):
    """In-place merge of (o_tile, lse_tile) into (o_acc, lse_acc)."""
    B, Sq, N, D = o_acc.shape
    st = _lib.lib().cp_lse_merge(_ptr(o_acc), _ptr(lse_acc), _ptr(o_tile), _ptr(lse_tile), B, Sq, N, D,
                                 _stream(stream))
    _lib.check("cp_lse_merge", st)
    return o_acc, lse_acc


def _ring_flags(prefetch, fused_merge, tf32=False):
    return ((CP_RING_PREFETCH if prefetch else 0) | (CP_RING_FUSED_MERGE if fused_merge else 0) |
            (CP_RING_TF32 if tf32 else 0))


def cp_ring_workspace_size(B, S, N, Nkv, D, C, prefetch=0, o_dtype=CP_F32, fused_merge=False, tf32=False):
    n = ctypes.c_size_t(0)
    st = _lib.lib().cp_ring_workspace_size(B, S, N, Nkv, D, C, _ring_flags(prefetch, fused_merge, tf32), o_dtype,
                                           ctypes.byref(n))
    _lib.check("cp_ring_workspace_size", st)
    return n.value


def cp_ring_attention_fwd(q_sh, k_sh, v_sh, pos, scale=None, layout=CP_ZIGZAG, prefetch=0, o_dtype=CP_F32,
                          workspace=None, o=None, lse=None, events=None, stream=None, fused_merge=False, tf32=False):
    """Ring attention forward over C resident virtual ranks.

    Returns (o_sh [C,B,s,N,D] of o_dtype, lse_sh fp32 [C,B,N,s]).  `events`, if
    given, is a list of >= 4*C recorded torch.cuda.Event objects (see the C
    header for their meaning).  tf32: fp32 shards, tensor cores in tf32."""
    C, B, s, N, D = q_sh.shape
    Nkv = k_sh.shape[3]
    S = C * s
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = q_sh.device
    if o is None:
        o = torch.empty((C, B, s, N, D), dtype=torch.float32 if o_dtype == CP_F32 else torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((C, B, N, s), dtype=torch.float32, device=dev)
    need = cp_ring_workspace_size(B, S, N, Nkv, D, C, prefetch, o_dtype, fused_merge, tf32)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    L = _lib.lib()
    args = [_ptr(q_sh), _ptr(k_sh), _ptr(v_sh), _ptr(pos), B, S, N, Nkv, D, C, float(scale), layout,
            _ring_flags(prefetch, fused_merge, tf32),
            _ptr(o), o_dtype, _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream)]
    if events is None:
        st = L.cp_ring_attention_fwd(*args)
        _lib.check("cp_ring_attention_fwd", st)
    else:
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        st = L.cp_ring_attention_fwd_traced(*args, arr, len(events))
        _lib.check("cp_ring_attention_fwd_traced", st)
    return o, lse


def cp_allgather_attention_fwd(q_sh, k_sh, v_sh, pos, scale=None, layout=CP_ZIGZAG, workspace=None, o=None,
                               lse=None, stream=None):
    """All-gather CP forward over C resident virtual ranks -> (o_sh fp32, lse_sh fp32)."""
    C, B, s, N, D = q_sh.shape
    Nkv = k_sh.shape[3]
    S = C * s
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = q_sh.device
    if o is None:
        o = torch.empty((C, B, s, N, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((C, B, N, s), dtype=torch.float32, device=dev)
    L = _lib.lib()
    n = ctypes.c_size_t(0)
    _lib.check("cp_allgather_workspace_size", L.cp_allgather_workspace_size(B, S, N, Nkv, D, C, ctypes.byref(n)))
    if workspace is None:
        workspace = torch.empty(max(256, n.value), dtype=torch.uint8, device=dev)
    st = L.cp_allgather_attention_fwd(_ptr(q_sh), _ptr(k_sh), _ptr(v_sh), _ptr(pos), B, S, N, Nkv, D, C,
                                      float(scale), layout, _ptr(o), _ptr(lse), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream))
    _lib.check("cp_allgather_attention_fwd", st)
    return o, lse


def cp_ulysses_attention_fwd(q_sh, k_sh, v_sh, scale=None, layout=CP_ZIGZAG, workspace=None, o=None, lse=None,
                             stream=None):
    """Ulysses (all-to-all) CP forward -> (o_sh fp32 [C,B,s,N,D], lse_h fp32 [C,B,N/C,S])."""
    C, B, s, N, D = q_sh.shape
    Nkv = k_sh.shape[3]
    S = C * s
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = q_sh.device
    if o is None:
        o = torch.empty((C, B, s, N, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((C, B, N // C, S), dtype=torch.float32, device=dev)
    L = _lib.lib()
    n = ctypes.c_size_t(0)
    _lib.check("cp_ulysses_workspace_size", L.cp_ulysses_workspace_size(B, S, N, Nkv, D, C, ctypes.byref(n)))
    if workspace is None:
        workspace = torch.empty(max(256, n.value), dtype=torch.uint8, device=dev)
    st = L.cp_ulysses_attention_fwd(_ptr(q_sh), _ptr(k_sh), _ptr(v_sh), B, S, N, Nkv, D, C, float(scale), layout,
                                    _ptr(o), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    _lib.check("cp_ulysses_attention_fwd", st)
    return o, lse


def cp_mesh_workspace_size(B, S, N, Nkv, D, A, R, prefetch=0, fused_merge=False):
    n = ctypes.c_size_t(0)
    st = _lib.lib().cp_mesh_workspace_size(B, S, N, Nkv, D, A, R, _ring_flags(prefetch, fused_merge), ctypes.byref(n))
    _lib.check("cp_mesh_workspace_size", st)
    return n.value


def cp_mesh_attention_fwd(q_sh, k_sh, v_sh, pos, A, R, scale=None, layout=CP_ZIGZAG, prefetch=0, fused_merge=False,
                          workspace=None, o=None, lse=None, stream=None):
    """A2A x P2P mesh CP forward over C = A*R resident virtual ranks.

    Returns (o_sh fp32 [C,B,s,N,D], lse_h fp32 [R,A,B,N/A,S/R])."""
    C, B, s, N, D = q_sh.shape
    Nkv = k_sh.shape[3]
    if A * R != C:
        raise ValueError("cp_mesh_attention_fwd: A*R must equal the number of shards")
    S = C * s
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = q_sh.device
    if o is None:
        o = torch.empty((C, B, s, N, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((R, A, B, N // A, S // R), dtype=torch.float32, device=dev)
    need = cp_mesh_workspace_size(B, S, N, Nkv, D, A, R, prefetch, fused_merge)
    if workspace is None:
        workspace = torch.empty(max(256, need), dtype=torch.uint8, device=dev)
    st = _lib.lib().cp_mesh_attention_fwd(_ptr(q_sh), _ptr(k_sh), _ptr(v_sh), _ptr(pos), B, S, N, Nkv, D, A, R,
                                          float(scale), layout, _ring_flags(prefetch, fused_merge), _ptr(o),
                                          _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream))
    _lib.check("cp_mesh_attention_fwd", st)
    return o, lse


def cp_attn_bwd_partial(q, k, v, o, dout, lse, q_pos, k_pos, scale=None, dq=None, dk=None, dv=None, accumulate=False,
                        workspace=None, stream=None):
    """Tile backward -> (dq fp32 [B,Sq,N,D], dk, dv fp32 [B,Sk,Nkv,D]) from the
    final output o (fp32) and lse; q, k, v, dout bf16."""
    B, Sq, N, D = q.shape
    Sk, Nkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = q.device
    dq = torch.empty((B, Sq, N, D), dtype=torch.float32, device=dev) if dq is None else dq
    dk = torch.empty((B, Sk, Nkv, D), dtype=torch.float32, device=dev) if dk is None else dk
    dv = torch.empty((B, Sk, Nkv, D), dtype=torch.float32, device=dev) if dv is None else dv
    L = _lib.lib()
    n = ctypes.c_size_t(0)
    _lib.check("cp_attn_bwd_workspace_size", L.cp_attn_bwd_workspace_size(B, Sq, Sk, N, ctypes.byref(n)))
    if workspace is None:
        workspace = torch.empty(max(256, n.value), dtype=torch.uint8, device=dev)
    st = L.cp_attn_bwd_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(q_pos), _ptr(k_pos), B,
                               Sq, Sk, N, Nkv, D, float(scale), _ptr(dq), _ptr(dk), _ptr(dv), 1 if accumulate else 0,
                               _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _lib.check("cp_attn_bwd_partial", st)
    return dq, dk, dv


def cp_ring_bwd_workspace_size(B, S, N, C):
    n = ctypes.c_size_t(0)
    _lib.check("cp_ring_bwd_workspace_size", _lib.lib().cp_ring_bwd_workspace_size(B, S, N, C, ctypes.byref(n)))
    return n.value


def cp_ring_attention_bwd(q_sh, k_sh, v_sh, o_sh, lse_sh, do_sh, pos, scale=None, layout=CP_ZIGZAG, workspace=None,
                          dq=None, dk=None, dv=None, stream=None):
    """Ring backward over C resident virtual ranks -> (dq_sh, dk_sh, dv_sh) fp32, rank-major."""
    C, B, s, N, D = q_sh.shape
    Nkv = k_sh.shape[3]
    S = C * s
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dev = q_sh.device
    dq = torch.empty((C, B, s, N, D), dtype=torch.float32, device=dev) if dq is None else dq
    dk = torch.empty((C, B, s, Nkv, D), dtype=torch.float32, device=dev) if dk is None else dk
    dv = torch.empty((C, B, s, Nkv, D), dtype=torch.float32, device=dev) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(max(256, cp_ring_bwd_workspace_size(B, S, N, C)), dtype=torch.uint8, device=dev)
    st = _lib.lib().cp_ring_attention_bwd(_ptr(q_sh), _ptr(k_sh), _ptr(v_sh), _ptr(o_sh), _ptr(lse_sh), _ptr(do_sh),
                                          _ptr(pos), B, S, N, Nkv, D, C, float(scale), layout, _ptr(dq), _ptr(dk),
                                          _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream))
    _lib.check("cp_ring_attention_bwd", st)
    return dq, dk, dv


def cp_ring_attention_fwd_noalloc(q_sh, k_sh, v_sh, pos, o, lse, scale=None, layout=CP_ZIGZAG, o_dtype=CP_F32,
                                  stream=None):
    """Ring forward that allocates nothing: for callers that may not call
    cudaMalloc (or cannot pass a workspace).  Its scratch is a fixed-size array
    inside the library (CP_NOALLOC_SCRATCH_BYTES); outputs o and lse must be
    given.  Calls on one device share that array: do not overlap them."""
    C, B, s, N, D = q_sh.shape
    Nkv = k_sh.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = _lib.lib().cp_ring_attention_fwd_noalloc(_ptr(q_sh), _ptr(k_sh), _ptr(v_sh), _ptr(pos), B, C * s, N, Nkv,
                                                  D, C, float(scale), layout, _ptr(o), o_dtype, _ptr(lse),
                                                  _stream(stream))
    _lib.check("cp_ring_attention_fwd_noalloc", st)
    return o, lse


def cp_selftest_stalled_producer(q, k, v, pos, o, lse, timeout_ns, stream=None):
    """Failure-detection self-test: the attention kernel with its producer held
    on a flag nothing sets; its bounded waits give up after timeout_ns and the
    device status becomes CP_ERR_DEVICE_TIMEOUT (read it with cp_device_status)."""
    st = _lib.lib().cp_selftest_stalled_producer(_ptr(q), _ptr(k), _ptr(v), _ptr(pos), _ptr(o), _ptr(lse),
                                                 int(timeout_ns), _stream(stream))
    _lib.check("cp_selftest_stalled_producer", st)


CP_SELFTEST_SCRATCH_BYTES = 512 << 10


def cp_selftest_stalled_kernel(kernel, timeout_ns, scratch=None, device="cuda", stream=None):
    """The same self-test for kernel 0 (bf16 forward), 1 (tf32 forward) or 2
    (backward: its dK/dV and dQ launches), on a tiny problem laid out in
    `scratch` (allocated here unless given)."""
    if scratch is None:
        scratch = torch.empty(CP_SELFTEST_SCRATCH_BYTES, dtype=torch.uint8, device=device)
    st = _lib.lib().cp_selftest_stalled_kernel(int(kernel), _ptr(scratch), scratch.numel() * scratch.element_size(),
                                               int(timeout_ns), _stream(stream))
    _lib.check("cp_selftest_stalled_kernel", st)


def cp_device_status(clear=True, stream=None):
    """Synchronise the stream and return the library's device status code."""
    code = ctypes.c_int(0)
    st = _lib.lib().cp_device_status(ctypes.byref(code), 1 if clear else 0, _stream(stream))
    _lib.check("cp_device_status", st)
    return code.value
