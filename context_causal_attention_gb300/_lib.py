"""ctypes loader for libcpattn.so and argument marshalling for its C ABI.

Every compute step runs in the CUDA library; this module only converts torch
tensors to pointers, sizes and stream handles.  There is no fallback: if the
library is missing or fails to load, every call raises.
"""
import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libcpattn.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "cpattn.h")

CP_OK = 0
STATUS_NAMES = {
    0: "CP_OK", 1: "CP_ERR_NULL", 2: "CP_ERR_SHAPE", 3: "CP_ERR_DIVISIBILITY", 4: "CP_ERR_DTYPE",
    5: "CP_ERR_ALIGNMENT", 6: "CP_ERR_WORKSPACE", 7: "CP_ERR_UNSUPPORTED", 8: "CP_ERR_CUDA",
    9: "CP_ERR_DEVICE_TIMEOUT", 10: "CP_ERR_ARGUMENT",
}
CP_BF16, CP_F32 = 0, 1
CP_ZIGZAG, CP_CONTIGUOUS = 0, 1
CP_SEQ_TO_HEAD, CP_HEAD_TO_SEQ = 0, 1
CP_RANK_ORDER, CP_GLOBAL_ORDER = 0, 1
CP_RING_PREFETCH, CP_RING_FUSED_MERGE, CP_RING_TF32 = 1, 2, 4


class CpError(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__("%s failed: %s" % (fn, text))
        self.status = status
        self.fn = fn


_lib = None


def header_symbols():
    """Names of every function declared in include/cpattn.h."""
    with open(HEADER) as f:
        src = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|cp_status)\s*(cp_\w+)\s*\(", src, re.M)))


def lib():
    """Load libcpattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libcpattn.so not built (expected at %s); run __graft_entry__.build()" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    sz = ctypes.c_size_t
    L.cp_status_string.argtypes = [i32]
    L.cp_status_string.restype = ctypes.c_char_p
    L.cp_version.argtypes = []
    L.cp_version.restype = ctypes.c_char_p
    L.cp_last_cuda_error.argtypes = []
    L.cp_last_cuda_error.restype = ctypes.c_char_p
    L.cp_zigzag_shard.argtypes = [vp, vp, i64, i64, i64, i64, i32, i32, i32, vp]
    L.cp_zigzag_unshard.argtypes = [vp, vp, i64, i64, i64, i64, i32, i32, i32, vp]
    L.cp_zigzag_positions.argtypes = [vp, i64, i32, i32, i32, vp]
    L.cp_ulysses_relayout.argtypes = [vp, vp, i64, i64, i64, i64, i32, i32, i32, i32, vp]
    L.cp_attn_partial.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, vp, vp, vp]
    L.cp_attn_workspace_size.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.POINTER(sz)]
    L.cp_attn_partial_ws.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, vp, vp, vp, sz, vp]
    L.cp_lse_merge.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    L.cp_ring_workspace_size.argtypes = [i64, i64, i64, i64, i64, i32, i32, i32, ctypes.POINTER(sz)]
    L.cp_ring_attention_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, f32, i32, i32, vp, i32, vp,
                                        vp, sz, vp]
    L.cp_ring_attention_fwd_traced.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, f32, i32, i32, vp,
                                               i32, vp, vp, sz, vp, vp, i32]
    L.cp_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), i32, vp]
    L.cp_allgather_workspace_size.argtypes = [i64, i64, i64, i64, i64, i32, ctypes.POINTER(sz)]
    L.cp_allgather_attention_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, f32, i32, vp, vp, vp, sz,
                                             vp]
    L.cp_ulysses_workspace_size.argtypes = [i64, i64, i64, i64, i64, i32, ctypes.POINTER(sz)]
    L.cp_ulysses_attention_fwd.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i32, f32, i32, vp, vp, vp, sz, vp]
    L.cp_mesh_workspace_size.argtypes = [i64, i64, i64, i64, i64, i32, i32, i32, ctypes.POINTER(sz)]
    L.cp_mesh_attention_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, i32, f32, i32, i32, vp, vp, vp,
                                        sz, vp]
    L.cp_attn_bwd_workspace_size.argtypes = [i64, i64, i64, i64, ctypes.POINTER(sz)]
    L.cp_attn_bwd_partial.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, vp, vp, vp,
                                      i32, vp, sz, vp]
    L.cp_ring_bwd_workspace_size.argtypes = [i64, i64, i64, i32, ctypes.POINTER(sz)]
    L.cp_ring_attention_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, f32, i32, vp, vp, vp,
                                        vp, sz, vp]
    L.cp_selftest_stalled_producer.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_uint64, vp]
    L.cp_selftest_stalled_kernel.argtypes = [i32, vp, sz, ctypes.c_uint64, vp]
    L.cp_attn_f32_workspace_size.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.POINTER(sz)]
    L.cp_attn_partial_f32.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, vp, vp, vp, sz, vp]
    L.cp_ring_attention_fwd_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, f32, i32, vp, i32, vp,
                                                vp]
    for name in header_symbols():
        if name not in ("cp_status_string", "cp_version", "cp_last_cuda_error"):
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def check(fn, status):
    if status != CP_OK:
        text = lib().cp_status_string(status).decode()
        if status == 8:
            text += " (%s)" % lib().cp_last_cuda_error().decode()
        raise CpError(fn, status, text)
