"""Child process of test_gpu_debug_bounds.py: runs with MOE_DEBUG_BOUNDS=1,
so the binding loads the bounds-checked build.  Computes the cases of
CASES into an .npz (argv[1]) and checks the injected-id path; prints "ok"."""
import sys

import numpy as np
import torch

import synth
import quantized_moe_decode_layer_gb300 as moe

DEV = "cuda"
# (name, shape, layers, first seed, rows, row seed)
CASES = [("tiny_m1", synth.TINY, 1, 1, 1, 11), ("tiny_m3", synth.TINY, 1, 1, 3, 12),
         ("a35b_m1", synth.A35B, 2, 1000, 1, 13), ("a35b_m4", synth.A35B, 2, 1000, 4, 14)]

_built = {}


def layers_of(shape, n, seed0):
    key = (shape.name, n, seed0)
    if key not in _built:
        _built[key] = [moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(synth.make_layer(shape, seed0 + i, device=DEV)))
                       for i in range(n)]
    return _built[key]


def run_case(shape, n, seed0, M, xseed):
    layers = layers_of(shape, n, seed0)
    x = synth.make_rows(shape, xseed, M).to(DEV)
    ws = moe.Workspace(layers[0].desc, M)
    if n == 1:
        out, on = moe.decode_layer(layers[0], x, ws, normed=True)
    else:
        out, on = moe.Stack(layers).forward(x, ws, normed=True)
    st = ws.status()
    return out.view(torch.int16).cpu().numpy(), on.view(torch.int16).cpu().numpy(), st


def main(path):
    assert moe.build_flags() == 1, "the checked build is not the one loaded"
    res = {}
    for name, shape, n, s0, M, xs in CASES:
        o, on, st = run_case(shape, n, s0, M, xs)
        assert st == 0, f"{name}: status {st} on valid data"
        res[name + "_out"], res[name + "_on"] = o, on
    np.savez(path, **res)
    # an expert id out of range in the first layer's routing of row 0: the
    # checks catch it (MOE_ERR_DEVICE), the launch ends normally, and the
    # next call without the hook is clean and gives the earlier result
    for name, shape, n, s0, M, xs in CASES:
        moe.debug_inject(shape.E + 3)
        try:
            st = run_case(shape, n, s0, M, xs)[2]
        finally:
            moe.debug_inject(-1)
        assert st == 6, f"{name}: expected MOE_ERR_DEVICE (6) for the injected id, got {st}"
        o, on, st = run_case(shape, n, s0, M, xs)
        assert st == 0, f"{name}: status {st} after the injected call"
        assert np.array_equal(o, res[name + "_out"]) and np.array_equal(on, res[name + "_on"]), \
            f"{name}: the call after the injected one differs"
    print("ok")


if __name__ == "__main__":
    main(sys.argv[1])
