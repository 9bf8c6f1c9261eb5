"""GPU parity of the configurations the benchmark times, through the C ABI.

The 40-layer 35B-A3B stack (shared expert, 8-bit router, Zipf routing) runs
as one persistent launch in which the next layer's router and shared-expert
rows are fetched while the current layer still runs; these tests run that
launch on several such layers and check it against chained single-layer
calls (bitwise) and against the fp64 oracle, teacher-forced (layer l of the
oracle on the GPU's own bf16 input of layer l; rows below the routing margin
are counted, see helpers.teacher_forced).  The same for the 397B-shaped
stack and for grouped mode (16 rows on the tensor-core path).

Source of the chaining: flash-moe (ja.news.hada.io), "Deferred GPU Expert
Compute" (combine, norm and residual stay on the GPU and feed the next
layer); PureDrive-35B-A3B-MLX model card, "Summary" (40 layers, top-8 plus a
shared expert) and "How it works" (fused add + RMSNorm between layers).
"""
import pytest
import torch

import oracle
import synth
import quantized_moe_decode_layer_gb300 as moe

from helpers import rows_with_margin, teacher_forced

pytestmark = pytest.mark.gpu
DEV = "cuda"


def build_stack(shape, n, seed0):
    built = []
    for i in range(n):
        L = synth.make_layer(shape, seed0 + i, device=DEV)
        built.append((moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L)), oracle.Layer(L)))
    return [b[0] for b in built], [b[1] for b in built]


def chained(layers, x, ws):
    h = x
    for i, lyr in enumerate(layers):
        if i == len(layers) - 1:
            h, hn = moe.decode_layer(lyr, h, ws, normed=True)
        else:
            h = moe.decode_layer(lyr, h, ws)
    return h, hn


def check_stack(shape, layers, lays, x, label):
    M = x.shape[0]
    ws = moe.Workspace(layers[0].desc, M)
    st = moe.Stack(layers)
    out, on = st.forward(x.to(DEV), ws, normed=True)
    assert ws.status() == 0
    h, hn = chained(layers, x.to(DEV), ws)
    assert torch.equal(h.view(torch.int16), out.view(torch.int16)), f"{label}: stack differs from chained calls"
    assert torch.equal(hn.view(torch.int16), on.view(torch.int16)), f"{label}: out_normed differs"
    teacher_forced(moe, layers, lays, x, ws, label)
    return out


_a35b = {}


def a35b_stack():
    if not _a35b:
        _a35b["v"] = build_stack(synth.A35B, 4, 1000)
    return _a35b["v"]


@pytest.mark.parametrize("M,corr", [(1, 0.0), (4, 0.6), (8, 0.5)])
def test_a35b_stack_matches_chained_and_oracle(M, corr):
    """The benchmarked stack shape: 4 distinct 35B-A3B layers in one launch."""
    layers, lays = a35b_stack()
    x = rows_with_margin(synth.A35B, lays[0], 900 + M, M, correlation=corr, gamma=lays[0].L["gamma"])
    check_stack(synth.A35B, layers, lays, x, f"a35b stack M={M}")


def test_a35b_stack_rows_equal_one_row_stack():
    """Row-exact verify through the stack: each row of a 4-row stack forward
    is bitwise the 1-row stack forward of that row (model card, "How it
    works": every row of the verify pass equals a one-row decode)."""
    layers, lays = a35b_stack()
    x = rows_with_margin(synth.A35B, lays[0], 950, 4, correlation=0.6, gamma=lays[0].L["gamma"]).to(DEV)
    st = moe.Stack(layers)
    ws = moe.Workspace(layers[0].desc, 4)
    out4 = st.forward(x, ws)
    for m in range(4):
        o1 = st.forward(x[m:m + 1].contiguous(), ws)
        assert torch.equal(o1.view(torch.int16), out4[m:m + 1].view(torch.int16)), f"row {m}"
    assert ws.status() == 0


def test_a35b_stack_repeated_launch_new_inputs():
    """Two stack forwards with different inputs on one workspace, then the
    first input again: the exchange words the earlier launches left behind
    are never taken for the current launch's (each launch draws its tags on
    the device), so every result matches its own single-layer chain."""
    layers, lays = a35b_stack()
    ws = moe.Workspace(layers[0].desc, 1)
    st = moe.Stack(layers)
    xs = [rows_with_margin(synth.A35B, lays[0], 960 + i, 1, gamma=lays[0].L["gamma"]).to(DEV) for i in range(2)]
    refs = [chained(layers, x, ws)[0] for x in xs]
    for x, ref in zip(xs + xs[:1], refs + refs[:1]):
        out = st.forward(x, ws)
        assert ws.status() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_b397_stack_matches_chained_and_oracle():
    """The 397B-shaped stack (4-bit routed top-10 of 512, 8-bit shared
    expert with I = 1024, uniform routing): 3 layers in one launch."""
    layers, lays = build_stack(synth.B397, 3, 3000)
    x = rows_with_margin(synth.B397, lays[0], 970, 1)
    check_stack(synth.B397, layers, lays, x, "b397 stack M=1")


@pytest.fixture
def grouped_always():
    moe.set_grouped(1)
    try:
        yield
    finally:
        moe.set_grouped(1)


def test_a35b_grouped_m16_stack(grouped_always):
    """Grouped mode (tensor-core expert products) at 16 rows, as the bench's
    sweep runs it: a 3-layer 35B-A3B stack equals chained grouped calls
    bitwise and each layer is within the tolerance of the oracle."""
    layers, lays = a35b_stack()
    layers, lays = layers[:3], lays[:3]
    x = rows_with_margin(synth.A35B, lays[0], 980, 16, gamma=lays[0].L["gamma"])
    check_stack(synth.A35B, layers, lays, x, "a35b grouped stack M=16")
