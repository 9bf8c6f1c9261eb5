"""ctypes view of libmoe.so (include/moe.h).  Argument marshalling only.

The library must exist (built by quantized_moe_decode_layer_gb300.build or
__graft_entry__.build()); there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_DEBUG_BOUNDS=1 in the environment selects the bounds-checked build
# (libmoe_debug.so); it is read once, when the library is first loaded.
DEBUG_BOUNDS = os.environ.get("MOE_DEBUG_BOUNDS", "0") not in ("", "0")
LIB_PATH = os.path.join(HERE, "libmoe_debug.so" if DEBUG_BOUNDS else "libmoe.so")

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_BUFFER_TOO_SMALL",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE", 7: "MOE_ERR_NOT_RESIDENT"}
T_ROUTER, T_SGATE, T_GATE, T_UP, T_DOWN, T_SHARED_GATE, T_SHARED_UP, T_SHARED_DOWN = range(8)

# every symbol include/moe.h declares
SYMBOLS = ["moe_pack_size", "moe_pack_weights", "moe_layer_destroy", "moe_export_canonical",
           "moe_workspace_size", "moe_workspace_init", "moe_router_topk", "moe_decode_layer",
           "moe_stack_create", "moe_stack_forward", "moe_stack_forward_host", "moe_stack_destroy",
           "moe_decode_layer_noalloc", "moe_noalloc_status",
           "moe_qkv_pack_size", "moe_qkv_pack", "moe_qkv_forward", "moe_qkv_destroy",
           "moe_attn_workspace_size", "moe_attn_decode", "moe_attn_append",
           "moe_streamed_size", "moe_streamed_create", "moe_streamed_layer", "moe_streamed_prepare",
           "moe_streamed_stats", "moe_streamed_destroy", "moe_streamed_forward",
           "moe_stream_status", "moe_build_flags", "moe_debug_inject", "moe_debug_set", "moe_debug_trace", "moe_set_grouped", "moe_set_grouped_products", "moe_gate_up_tc", "moe_down_tc", "moe_status_str",
           "moe_last_cuda_error",
           "moe_selftest_host", "moe_launch_count"]


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} (cuda error {last_cuda_error()})")


class LayerDesc(C.Structure):
    _fields_ = [("H", C.c_int), ("I", C.c_int), ("E", C.c_int), ("k", C.c_int),
                ("routed_bits", C.c_int), ("shared_bits", C.c_int), ("router_bits", C.c_int),
                ("has_shared", C.c_int), ("I_shared", C.c_int), ("eps", C.c_float)]


class SrcMatrix(C.Structure):
    _fields_ = [("codes_dev", C.c_void_p), ("scales_dev", C.c_void_p), ("biases_dev", C.c_void_p),
                ("w_dev", C.c_void_p)]


class QkvDesc(C.Structure):
    _fields_ = [("H", C.c_int), ("n_q", C.c_int), ("n_k", C.c_int), ("n_v", C.c_int), ("bits", C.c_int)]


class SrcLayer(C.Structure):
    _fields_ = [("gate", SrcMatrix), ("up", SrcMatrix), ("down", SrcMatrix),
                ("shared_gate", SrcMatrix), ("shared_up", SrcMatrix), ("shared_down", SrcMatrix),
                ("router", SrcMatrix), ("sgate", SrcMatrix),
                ("gamma_dev", C.c_void_p), ("gamma_next_dev", C.c_void_p)]


_lib = None


def lib():
    """Load libmoe.so; raise if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        vp, i, sz = C.c_void_p, C.c_int, C.c_size_t
        sig = {
            "moe_pack_size": (i, [C.POINTER(LayerDesc), C.POINTER(sz)]),
            "moe_pack_weights": (i, [C.POINTER(LayerDesc), C.POINTER(SrcLayer), vp, sz, C.POINTER(vp), vp]),
            "moe_layer_destroy": (None, [vp]),
            "moe_export_canonical": (i, [vp, i, i, vp, vp, vp, vp]),
            "moe_workspace_size": (i, [C.POINTER(LayerDesc), i, C.POINTER(sz)]),
            "moe_workspace_init": (i, [vp, sz, vp]),
            "moe_router_topk": (i, [vp, vp, i, vp, vp, vp, sz, vp]),
            "moe_decode_layer": (i, [vp, vp, i, vp, vp, vp, sz, vp]),
            "moe_stack_create": (i, [C.POINTER(vp), i, C.POINTER(vp)]),
            "moe_stack_forward": (i, [vp, vp, i, vp, vp, vp, sz, vp]),
            "moe_stack_forward_host": (i, [vp, vp, i, vp, vp, sz, vp]),
            "moe_stack_destroy": (None, [vp]),
            "moe_decode_layer_noalloc": (i, [vp, vp, i, vp, vp, vp]),
            "moe_noalloc_status": (i, [vp]),
            "moe_qkv_pack_size": (i, [C.POINTER(QkvDesc), C.POINTER(sz)]),
            "moe_qkv_pack": (i, [C.POINTER(QkvDesc), C.POINTER(SrcMatrix), C.POINTER(SrcMatrix), C.POINTER(SrcMatrix),
                                 vp, sz, C.POINTER(vp), vp]),
            "moe_qkv_forward": (i, [vp, vp, i, vp, vp, vp]),
            "moe_attn_workspace_size": (i, [i, C.POINTER(sz)]),
            "moe_attn_decode": (i, [vp, vp, vp, i, i, i, vp, vp, sz, vp, vp]),
            "moe_attn_append": (i, [vp, vp, i, i, vp, vp, i, vp]),
            "moe_streamed_size": (i, [C.POINTER(LayerDesc), i, C.POINTER(sz)]),
            "moe_streamed_create": (i, [vp, vp, sz, vp, sz, i, C.POINTER(vp), vp]),
            "moe_streamed_layer": (vp, [vp]),
            "moe_streamed_prepare": (i, [vp, vp, i, vp, C.POINTER(i)]),
            "moe_streamed_stats": (i, [vp] + [C.POINTER(C.c_longlong)] * 6),
            "moe_streamed_destroy": (None, [vp]),
            "moe_streamed_forward": (i, [vp, i, vp, i, vp, vp, vp, sz, vp, sz, i, vp, vp]),
            "moe_qkv_destroy": (None, [vp]),
            "moe_stream_status": (i, [vp, sz, vp]),
            "moe_debug_set": (i, [i, C.c_longlong]),
            "moe_build_flags": (i, []),
            "moe_set_grouped_products": (i, [i]),
            "moe_debug_inject": (i, [i]),
            "moe_debug_trace": (i, [vp, sz]),
            "moe_gate_up_tc": (i, [vp, vp, i, vp, vp, i, vp, vp, vp]),
            "moe_down_tc": (i, [vp, vp, i, vp, vp, i, vp, vp, vp]),
            "moe_set_grouped": (i, [i]),
            "moe_status_str": (C.c_char_p, [i]),
            "moe_last_cuda_error": (i, []),
            "moe_selftest_host": (i, []),
            "moe_launch_count": (C.c_longlong, [i]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def check(fn: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(fn, rc)


def last_cuda_error() -> int:
    return int(lib().moe_last_cuda_error()) if _lib is not None else 0
