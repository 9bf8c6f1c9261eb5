"""A small stack case for profiler captures: `--layers` distinct layer sets
of the 35B-A3B shape (about 0.66 GB each) in one persistent launch at M rows,
run `--forwards` times.  Prints one JSON line with the algorithmic bytes of
one launch (from the experts the rows actually selected).  With --tc, the
tensor-core grouped gate/up then runs on each layer's routing of the rows.
With --attn T, instead: the decode attention (moe_attn_decode) over a cache
of T positions at M rows, run `--forwards` times.

    python -m quantized_moe_decode_layer_gb300.profile_case --M 1 --layers 3
    python -m quantized_moe_decode_layer_gb300.profile_case --attn 32768 --M 3
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def tc_routing(layers, x, ws):
    """Per layer along the chain of single-layer calls on x's rows: (distinct
    experts int32 [U], their row masks int32 [U], the layer's input rows as
    fp32 [M, H]).  The input rows stand in for the normalised rows of the
    tensor-core gate/up calls that are timed or profiled with them."""
    import numpy as np
    import torch
    import quantized_moe_decode_layer_gb300 as moe
    out, h = [], x
    for lyr in layers:
        idx, _ = moe.router_topk(lyr, h, ws)
        sel = idx.cpu().numpy()
        ex = np.unique(sel)
        masks = [sum(1 << m for m in range(sel.shape[0]) if e in sel[m]) for e in ex]
        masks = [m - (1 << 32) if m >= (1 << 31) else m for m in masks]
        out.append((torch.tensor(ex, dtype=torch.int32, device=x.device),
                    torch.tensor(masks, dtype=torch.int32, device=x.device), h.float()))
        h = moe.decode_layer(lyr, h, ws)
    return out


def attn_case(a) -> None:
    import torch
    import synth
    import quantized_moe_decode_layer_gb300 as moe
    T, M = a.attn, a.M
    q, k, vt = synth.make_attn(T, T, M, 5, device="cuda")
    cache = moe.AttnCache(T, device="cuda")
    cache.k.copy_(k)
    cache.vt.copy_(vt)
    del k, vt
    out = torch.empty((M, 16, 256), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(a.forwards):
        cache.attend(q, T - M, out=out, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    print(json.dumps({"case": "attn", "T": T, "M": M, "forwards": a.forwards,
                      "bytes_per_call": T * 2 * 256 * 2 * 2 + M * 16 * 256 * 6}))


def main() -> None:
    p = argparse.ArgumentParser()
    p.add_argument("--M", type=int, default=1)
    p.add_argument("--layers", type=int, default=3)
    p.add_argument("--forwards", type=int, default=4)
    p.add_argument("--shape", default="a35b")
    p.add_argument("--correlation", type=float, default=0.6)
    p.add_argument("--tc", action="store_true",
                   help="then run the tensor-core grouped gate/up (moe_gate_up_tc) on each layer's routing")
    p.add_argument("--attn", type=int, default=0, help="run the decode attention over a cache of this many positions")
    a = p.parse_args()
    if a.attn:
        attn_case(a)
        return

    import torch
    import synth
    import quantized_moe_decode_layer_gb300 as moe
    from quantized_moe_decode_layer_gb300.accounting import unique_bytes

    shape = synth.SHAPES[a.shape]
    desc = moe.desc_from_shape(shape)
    layers = []
    for l in range(a.layers):
        L = synth.make_layer(shape, 1000 + l, device="cuda")
        layers.append(moe.Layer(desc, moe.layer_src_from_synth(L)))
        del L
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    st = moe.Stack(layers)
    ws = moe.Workspace(desc, a.M)
    x = synth.make_rows(shape, 5, a.M, correlation=a.correlation if a.M > 1 else 0.0).cuda()
    Us, h = [], x
    for lyr in layers:           # distinct experts per layer along the chain (single-layer calls)
        idx, _ = moe.router_topk(lyr, h, ws)
        Us.append(int(torch.unique(idx).numel()))
        h = moe.decode_layer(lyr, h, ws)
    for _ in range(a.forwards):
        st.forward(x, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    tc_calls = 0
    if a.tc:
        cases = tc_routing(layers, x, ws)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(a.forwards):
            for (ex, mk, hn), lyr in zip(cases, layers):
                moe.gate_up_tc(lyr, hn, ex, mk, err=err)
                tc_calls += 1
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    print(json.dumps({"shape": shape.name, "M": a.M, "layers": a.layers, "U": Us,
                      "algorithmic_bytes_per_launch": sum(unique_bytes(shape, u, a.M) for u in Us),
                      "launches": {"router_topk": a.layers, "decode_layer": a.layers, "stack": a.forwards,
                                   "router_topk_tc_routing": a.layers if a.tc else 0,
                                   "decode_layer_tc_routing": a.layers if a.tc else 0, "gate_up_tc": tc_calls}}))


if __name__ == "__main__":
    main()
