"""A small stack case for profiler captures: `--layers` distinct layer sets
of the 35B-A3B shape (about 0.66 GB each) in one persistent launch at M rows,
run `--forwards` times.  Prints one JSON line with the algorithmic bytes of
one launch (from the experts the rows actually selected).

    python -m quantized_moe_decode_layer_gb300.profile_case --M 1 --layers 3
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main() -> None:
    p = argparse.ArgumentParser()
    p.add_argument("--M", type=int, default=1)
    p.add_argument("--layers", type=int, default=3)
    p.add_argument("--forwards", type=int, default=4)
    p.add_argument("--shape", default="a35b")
    p.add_argument("--correlation", type=float, default=0.6)
    a = p.parse_args()

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
    print(json.dumps({"shape": shape.name, "M": a.M, "layers": a.layers, "U": Us,
                      "algorithmic_bytes_per_launch": sum(unique_bytes(shape, u, a.M) for u in Us),
                      "launches": {"router_topk": a.layers, "decode_layer": a.layers, "stack": a.forwards}}))


if __name__ == "__main__":
    main()
