"""GB300 (sm_103a) quantized MoE decode layer: a C-ABI CUDA library
(libmoe.so, include/moe.h) with a thin torch/ctypes binding."""
from .api import (QKV, AttnCache, StreamedLayer, streamed_forward, Layer, Stack, Workspace, build_flags, debug_inject, debug_set, decode_layer,
                  decode_layer_noalloc, desc_from_shape, down_tc, gate_up_tc, launch_count, layer_src_from_synth,
                  make_desc, noalloc_status, pack_size, router_topk, selftest_host, set_grouped, set_grouped_products, workspace_size)
from ._lib import SYMBOLS, MoeError, lib

__all__ = ["QKV", "AttnCache", "StreamedLayer", "streamed_forward", "Layer", "Stack", "Workspace", "build_flags", "debug_inject", "debug_set", "decode_layer",
           "decode_layer_noalloc", "desc_from_shape", "down_tc", "gate_up_tc", "noalloc_status", "selftest_host",
           "launch_count", "layer_src_from_synth", "set_grouped", "set_grouped_products", "make_desc", "pack_size", "router_topk",
           "workspace_size", "SYMBOLS", "MoeError", "lib"]
