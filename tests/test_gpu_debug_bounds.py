"""The bounds-checked build (libmoe_debug.so, MOE_DEBUG_BOUNDS) on the GPU.

A child process loads the checked build (the library is chosen once per
process) and runs a tiny layer and a two-layer 35B-A3B stack at 1 and
several rows; this process runs the same seeded cases on the normal build.
The checked build must give the same bits (no check fires on valid data),
the tiny cases must match the oracle, and an out-of-range expert id planted
in the first layer's routing must come back as MOE_ERR_DEVICE with the
launch ending normally (bounds_case.py)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_moe_decode_layer_gb300 as moe
from quantized_moe_decode_layer_gb300 import build as b

import bounds_case
from helpers import MARGIN, assert_close

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_matches_normal_build_and_reports_bad_ids(tmp_path):
    b.build(debug_bounds=True)
    path = str(tmp_path / "checked.npz")
    env = dict(os.environ, MOE_DEBUG_BOUNDS="1")
    env["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests")])
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_case.py"), path], env=env,
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
    got = np.load(path)
    assert moe.build_flags() == 0
    for name, shape, n, s0, M, xs in bounds_case.CASES:
        o, on, st = bounds_case.run_case(shape, n, s0, M, xs)
        assert st == 0
        assert np.array_equal(o, got[name + "_out"]), f"{name}: checked build differs in out"
        assert np.array_equal(on, got[name + "_on"]), f"{name}: checked build differs in out_normed"
        if shape is synth.TINY:
            lay = oracle.Layer(synth.make_layer(shape, s0, device="cuda"))
            x = synth.make_rows(shape, xs, M)
            ref = lay.forward(synth.bf16_bits(x).numpy().view(np.uint16), normed=True)
            val = torch.from_numpy(o).view(torch.bfloat16).double().numpy()
            rows = [m for m in range(M) if ref["margin"][m] >= MARGIN]
            assert rows, f"{name}: no row above the routing margin"
            assert_close(val[rows], ref["o"][rows], name)
