"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Bit-exact: packed codes/scales/biases, quantiser decisions, expert indices.
Tolerance on the bf16 outputs: |gpu - ref| <= 2e-3 + 1e-2 |ref| against the
unrounded fp64 oracle value (ref = o for out, on for out_normed).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_moe_decode_layer_gb300 as moe
from quantized_moe_decode_layer_gb300 import _lib

from helpers import MARGIN, assert_close, bf16_tensor_to_f64, bits_np, rows_with_margin, teacher_forced, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def build(shape, seed, device=DEV):
    """(canonical dict on device, packed layer, oracle view)."""
    L = synth.make_layer(shape, seed, device=device)
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    return L, layer, oracle.Layer(L)


_cache = {}


def cached(shape, seed):
    key = (shape.name, seed)
    if key not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        _cache[key] = build(shape, seed)
    return _cache[key]


def check_layer(shape, L, layer, lay, x, normed=True):
    ws = moe.Workspace(layer.desc, x.shape[0])
    if normed:
        out, on = moe.decode_layer(layer, x.to(DEV), ws, normed=True)
    else:
        out = moe.decode_layer(layer, x.to(DEV), ws)
    assert ws.status() == 0
    ref = lay.forward(bits_np(x), normed=normed)
    assert_close(bf16_tensor_to_f64(out), ref["o"], f"{shape.name} out")
    if normed:
        assert_close(bf16_tensor_to_f64(on), ref["on"], f"{shape.name} out_normed")
    idx, w = moe.router_topk(layer, x.to(DEV), ws)
    assert ws.status() == 0
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.allclose(w.cpu().numpy(), ref["w"], rtol=1e-4, atol=1e-6)
    return out, ref


# ------------------------------------------------------------------ packing

@pytest.mark.parametrize("shape", [synth.TINY, synth.A35B])
def test_pack_export_roundtrip(shape):
    L, layer, lay = cached(shape, 101)
    for tid, name, e in [(_lib.T_GATE, "gate", 0), (_lib.T_UP, "up", shape.E - 1), (_lib.T_DOWN, "down", 3)]:
        c, s, b = layer.export(tid, e)
        src = L[name]
        assert torch.equal(c, src["codes"][e]), name
        assert torch.equal(s.view(torch.int16), src["scales"][e].view(torch.int16)), name
        assert torch.equal(b.view(torch.int16), src["biases"][e].view(torch.int16)), name
    if shape.has_shared:
        for tid, name in [(_lib.T_SHARED_GATE, "shared_gate"), (_lib.T_SHARED_UP, "shared_up"),
                          (_lib.T_SHARED_DOWN, "shared_down")]:
            c, s, b = layer.export(tid)
            assert torch.equal(c, L[name]["codes"]), name
            assert torch.equal(s.view(torch.int16), L[name]["scales"].view(torch.int16)), name


def test_quantiser_matches_oracle_bit_exact():
    """fp32 router -> 8-bit groups: the GPU packer's codes, scales and biases
    equal the oracle quantiser's (both decide in fp32)."""
    L, layer, lay = cached(synth.A35B, 101)
    c, s, b = layer.export(_lib.T_ROUTER)
    assert np.array_equal(c.cpu().numpy(), lay.router.codes)
    assert np.array_equal(s.view(torch.int16).cpu().numpy().view(np.uint16), lay.router.scales)
    assert np.array_equal(b.view(torch.int16).cpu().numpy().view(np.uint16), lay.router.biases)
    c, s, b = layer.export(_lib.T_SGATE)
    assert np.array_equal(c.cpu().numpy(), lay.sgate.codes)


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_quantiser_fp32_experts(bits):
    """Experts given as fp32 weights are quantised on the GPU exactly as the oracle does."""
    sh = synth.LayerShape("q", 256, 128, 4, 2, bits, 8, 0, False, 0, False)
    g = torch.Generator(device=DEV).manual_seed(bits)
    gate = torch.randn((4 * 128, 256), generator=g, device=DEV) * 0.05
    up = torch.randn((4 * 128, 256), generator=g, device=DEV) * 0.05
    down = torch.randn((4 * 256, 128), generator=g, device=DEV) * 0.05
    src = {"gate": {"w": gate}, "up": {"w": up}, "down": {"w": down},
           "router": {"w": torch.randn((4, 256), generator=g, device=DEV)},
           "gamma": torch.ones(256, dtype=torch.bfloat16, device=DEV)}
    layer = moe.Layer(moe.desc_from_shape(sh), src)
    for tid, w, rows in [(_lib.T_GATE, gate, 128), (_lib.T_DOWN, down, 256)]:
        for e in (0, 3):
            c, s, b = layer.export(tid, e)
            qc, qs, qb = oracle.quantize_matrix(w[e * rows:(e + 1) * rows].cpu().numpy(), bits)
            assert np.array_equal(c.cpu().numpy(), qc)
            assert np.array_equal(s.view(torch.int16).cpu().numpy().view(np.uint16), qs)
            assert np.array_equal(b.view(torch.int16).cpu().numpy().view(np.uint16), qb)


# ------------------------------------------------------------------- layers

@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
def test_tiny_layer(M):
    shape = synth.TINY
    L, layer, lay = cached(shape, 7)
    x = rows_with_margin(shape, lay, 100 + M, M)
    check_layer(shape, L, layer, lay, x)


def test_tiny_many_rows_chunked():
    """M above the rows of one launch (19 rows): grouped mode by default;
    routing bit-exact, outputs within the tolerance."""
    shape = synth.TINY
    L, layer, lay = cached(shape, 7)
    x = rows_with_margin(shape, lay, 555, 19)
    check_layer(shape, L, layer, lay, x)


def test_a35b_m1():
    shape = synth.A35B
    L, layer, lay = cached(shape, 11)
    x = rows_with_margin(shape, lay, 1, 1, gamma=L["gamma"])
    check_layer(shape, L, layer, lay, x)


def rows_equal_one_row_calls(layer, x, out):
    """Each row of an M-row call is bitwise the one-row call of that row."""
    ws = moe.Workspace(layer.desc, 1)
    for m in range(x.shape[0]):
        o1 = moe.decode_layer(layer, x[m:m + 1].to(DEV), ws)
        assert torch.equal(o1.view(torch.int16), out[m:m + 1].view(torch.int16)), f"row {m}"
    assert ws.status() == 0


def test_a35b_m4_rows_equal_m1_bitwise():
    """1 token + 3 correlated draft rows: every row equals the one-row call bit
    for bit (PureDrive model card, "How it works": row-exact verify)."""
    shape = synth.A35B
    L, layer, lay = cached(shape, 11)
    x = rows_with_margin(shape, lay, 3, 4, correlation=0.6, gamma=L["gamma"])
    out4, ref = check_layer(shape, L, layer, lay, x)
    rows_equal_one_row_calls(layer, x, out4)


def test_a35b_m4_shared_fraction():
    """The M=4 workload (1 token + 3 draft rows at correlation 0.6): over 32
    draws, the experts chosen by two or more rows make up 30-60 % of the
    distinct experts on average (the GPU's routing)."""
    shape = synth.A35B
    L, layer, lay = cached(shape, 11)
    ws = moe.Workspace(layer.desc, 4)
    fr = []
    for seed in range(32):
        x = synth.make_rows(shape, 7000 + seed, 4, correlation=0.6, gamma=L["gamma"]).to(DEV)
        idx, _ = moe.router_topk(layer, x, ws)
        idx = idx.cpu().numpy()
        union = set(idx.ravel().tolist())
        shared = sum(1 for e in union if (idx == e).any(axis=1).sum() >= 2)
        fr.append(shared / len(union))
    assert ws.status() == 0
    print(f"shared fraction at M=4: mean {np.mean(fr):.3f}, min {min(fr):.3f}, max {max(fr):.3f}")
    assert 0.3 <= float(np.mean(fr)) <= 0.6


def test_a35b_m8():
    """8 rows in one launch: parity, and every row bitwise the one-row call."""
    shape = synth.A35B
    L, layer, lay = cached(shape, 11)
    x = rows_with_margin(shape, lay, 3, 8, correlation=0.5, gamma=L["gamma"])
    out, _ = check_layer(shape, L, layer, lay, x)
    rows_equal_one_row_calls(layer, x, out)


def test_tiny_literal_grid():
    """The workload's bias distribution taken literally (b ~ N(0, 0.01), so
    every dequantised matrix has a positive mean): parity holds as well."""
    shape = synth.TINY
    L = synth.make_layer(shape, 8, device=DEV, grid="literal")
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    lay = oracle.Layer(L)
    x = rows_with_margin(shape, lay, 108, 3)
    check_layer(shape, L, layer, lay, x)


DEFAULT_GROUPED_MIN_ROWS = 1


@pytest.fixture
def fma_only():
    moe.set_grouped(0)
    try:
        yield
    finally:
        moe.set_grouped(DEFAULT_GROUPED_MIN_ROWS)


@pytest.fixture
def grouped_always():
    moe.set_grouped(1)
    try:
        yield
    finally:
        moe.set_grouped(DEFAULT_GROUPED_MIN_ROWS)


@pytest.fixture(params=["fma", "tc"])
def grouped_products(request):
    moe.set_grouped_products(request.param == "tc")
    try:
        yield request.param
    finally:
        moe.set_grouped_products(False)


def test_a35b_m32_grouped(grouped_products):
    """32 rows: grouped mode (every expert read once for the 32 rows), with
    its products on the FMA pipes (the default) and on the tensor cores:
    routing bit-exact, outputs within the tolerance."""
    shape = synth.A35B
    L, layer, lay = cached(shape, 11)
    x = rows_with_margin(shape, lay, 4, 32, gamma=L["gamma"])
    check_layer(shape, L, layer, lay, x)


def test_grouped_fma_products_match_one_row_products():
    """The grouped FMA products run the persistent kernel's one-vector row
    kernel: with grouped mode on, a 12-row tiny call's rows are within the
    tolerance and each expert's products do not depend on the other rows
    (two calls sharing row 0 give row 0 the same output bits)."""
    shape = synth.TINY
    L, layer, lay = cached(shape, 7)
    x = rows_with_margin(shape, lay, 777, 12)
    out, _ = check_layer(shape, L, layer, lay, x)
    y = rows_with_margin(shape, lay, 778, 12)
    y[0] = x[0]
    ws = moe.Workspace(layer.desc, 12)
    out2 = moe.decode_layer(layer, y.to(DEV), ws)
    assert ws.status() == 0
    assert torch.equal(out[0].view(torch.int16), out2[0].view(torch.int16))


def test_tiny_m40_two_groups():
    """40 rows: grouped mode in two groups (32 + 8 rows); routing bit-exact,
    outputs within the tolerance."""
    shape = synth.TINY
    L, layer, lay = cached(shape, 7)
    x = rows_with_margin(shape, lay, 640, 40)
    check_layer(shape, L, layer, lay, x)


def test_a35b_m32_fma_chunks(fma_only):
    """32 rows with grouped mode off: four 8-row launches of the FMA path;
    every row is bitwise the one-row call (the mode a row-exact verify with
    more than 8 rows uses)."""
    shape = synth.A35B
    L, layer, lay = cached(shape, 11)
    x = rows_with_margin(shape, lay, 5, 32, gamma=L["gamma"])
    out, _ = check_layer(shape, L, layer, lay, x)
    rows_equal_one_row_calls(layer, x, out)


def test_grouped_stack_equals_chained_layers(grouped_always):
    """Grouped mode through a 3-layer stack (M = 12, tiny shape) gives the
    bits of chained single-layer grouped calls, and each layer is within the
    tolerance of the oracle on the GPU's own input (teacher-forced)."""
    shape = synth.TINY
    built = [build(shape, 300 + i) for i in range(3)]
    layers = [b[1] for b in built]
    lays = [b[2] for b in built]
    x = rows_with_margin(shape, lays[0], 10, 12)
    ws = moe.Workspace(layers[0].desc, 12)
    st = moe.Stack(layers)
    out, on = st.forward(x.to(DEV), ws, normed=True)
    assert ws.status() == 0
    h = x.to(DEV)
    for i, lyr in enumerate(layers):
        if i == len(layers) - 1:
            h, hn = moe.decode_layer(lyr, h, ws, normed=True)
        else:
            h = moe.decode_layer(lyr, h, ws)
    assert torch.equal(h.view(torch.int16), out.view(torch.int16))
    assert torch.equal(hn.view(torch.int16), on.view(torch.int16))
    teacher_forced(moe, layers, lays, x, ws, "tiny grouped stack M=12")


def test_b397_m1():
    shape = synth.B397
    L, layer, lay = cached(shape, 13)
    x = rows_with_margin(shape, lay, 4, 1)
    check_layer(shape, L, layer, lay, x)


def test_b397_m3_rows_equal_m1_bitwise():
    """397B shape (rows of 4096 inputs: the 8-compute-warp build), 3 rows with
    the routing warps beside the RMSNorm: parity, and every row bitwise the
    one-row call."""
    shape = synth.B397
    L, layer, lay = cached(shape, 13)
    x = rows_with_margin(shape, lay, 5, 3, correlation=0.6, gamma=L["gamma"])
    out, _ = check_layer(shape, L, layer, lay, x)
    rows_equal_one_row_calls(layer, x, out)


def test_deterministic_repeat():
    shape = synth.TINY
    L, layer, lay = cached(shape, 7)
    x = rows_with_margin(shape, lay, 77, 4).to(DEV)
    ws = moe.Workspace(layer.desc, 4)
    a = moe.decode_layer(layer, x, ws)
    b = moe.decode_layer(layer, x, ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_tiny_m5_rows_equal_m1_bitwise():
    """5 rows: more routing rows than half the compute warps, so every warp
    builds hn before the first five route (the 8-warp build); each row
    bitwise the one-row call."""
    shape = synth.TINY
    L, layer, lay = cached(shape, 7)
    x = rows_with_margin(shape, lay, 78, 5)
    out, _ = check_layer(shape, L, layer, lay, x)
    rows_equal_one_row_calls(layer, x, out)


def test_a35b_m4_deterministic_repeat():
    """35B shape, 1 token + 3 correlated draft rows (shared experts, and
    shared-expert units that come through the ring): repeated calls on one
    workspace and a call on a fresh one are bitwise equal (no race between
    the warps that route and those that build hn)."""
    shape = synth.A35B
    L, layer, lay = cached(shape, 11)
    x = synth.make_rows(shape, 61, 4, correlation=0.6, gamma=L["gamma"]).to(DEV)
    ws = moe.Workspace(layer.desc, 4)
    outs = [moe.decode_layer(layer, x, ws) for _ in range(3)]
    outs.append(moe.decode_layer(layer, x, moe.Workspace(layer.desc, 4)))
    torch.cuda.synchronize()
    assert ws.status() == 0
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_out_aliases_x():
    shape = synth.TINY
    L, layer, lay = cached(shape, 7)
    x = rows_with_margin(shape, lay, 78, 2)
    ws = moe.Workspace(layer.desc, 2)
    ref = moe.decode_layer(layer, x.to(DEV), ws)
    buf = x.to(DEV).clone()
    moe.decode_layer(layer, buf, ws, out=buf)
    assert torch.equal(buf.view(torch.int16), ref.view(torch.int16))


# -------------------------------------------------------------------- stack

def test_stack_equals_chained_layers_and_oracle():
    shape = synth.TINY
    built = [build(shape, 200 + i) for i in range(3)]
    layers = [b[1] for b in built]
    lays = [b[2] for b in built]
    x = rows_with_margin(shape, lays[0], 9, 2)
    ws = moe.Workspace(layers[0].desc, 2)
    st = moe.Stack(layers)
    out, on = st.forward(x.to(DEV), ws, normed=True)
    assert ws.status() == 0
    # chained single-layer calls give the same bits
    h = x.to(DEV)
    for i, lyr in enumerate(layers):
        if i == len(layers) - 1:
            h, hn = moe.decode_layer(lyr, h, ws, normed=True)
        else:
            h = moe.decode_layer(lyr, h, ws)
    assert torch.equal(h.view(torch.int16), out.view(torch.int16))
    assert torch.equal(hn.view(torch.int16), on.view(torch.int16))
    # teacher-forced oracle: layer l on the GPU's bf16 input of layer l
    teacher_forced(moe, layers, lays, x, ws, "tiny stack M=2")


def test_stack_host_buffers():
    shape = synth.TINY
    built = [build(shape, 300 + i) for i in range(2)]
    layers = [b[1] for b in built]
    x = rows_with_margin(shape, built[0][2], 10, 3)
    ws = moe.Workspace(layers[0].desc, 3)
    st = moe.Stack(layers)
    dev_out = st.forward(x.to(DEV), ws)
    out_h = torch.empty_like(x).pin_memory()
    st.forward_host(x.pin_memory(), out_h, ws)
    assert torch.equal(out_h.view(torch.int16), dev_out.cpu().view(torch.int16))


# -------------------------------------------------------------------- waits

def test_barrier_timeout_returns_status():
    """A router logit that is never published makes every CTA's wait for it
    run out: the call returns MOE_ERR_TIMEOUT instead of hanging, and the
    workspace works again after moe_workspace_init."""
    shape = synth.TINY
    L, layer, lay = cached(shape, 7)
    x = rows_with_margin(shape, lay, 79, 1).to(DEV)
    ws = moe.Workspace(layer.desc, 1)
    good = moe.decode_layer(layer, x, ws)
    assert ws.status() == 0
    try:
        moe.debug_set(skip_row=3, timeout_ns=50_000_000)
        moe.decode_layer(layer, x, ws)
        assert ws.status() == 5
    finally:
        moe.debug_set(-1, 0)
    ws.init()
    again = moe.decode_layer(layer, x, ws)
    assert ws.status() == 0
    assert torch.equal(again.view(torch.int16), good.view(torch.int16))


def _rows_with_distinct_margin(shape, lay, seed, gamma=None, max_attempts=200):
    """One bf16 row whose oracle logits, as a set of distinct values, are at
    least MARGIN apart down to the (k+1)-th largest expert: exact ties stay
    exact in both precisions, and no two distinct values can swap."""
    for a in range(max_attempts):
        x = synth.make_rows(shape, seed, 1, gamma=gamma, attempts=[a])
        lg = lay.route(bits_np(x))["logits"][0]
        d = np.unique(np.sort(lg)[::-1][:shape.k + 2])
        if len(d) < 2 or np.min(np.diff(d)) >= MARGIN:
            return x
    raise RuntimeError("could not draw a row with distinct-value margins")


@pytest.mark.parametrize("shape,period", [(synth.TINY, 2), (synth.A35B, 2), (synth.A35B, 4)])
def test_router_topk_exact_ties(shape, period):
    """Repeated router rows make logits tie exactly; the top k must list tied
    experts by ascending id, as the oracle does.  Period 2 at a35b: experts
    2j and 2j + 1 share a row (pairs of ties).  Period 2 at tiny and 4 at
    a35b: expert e uses row e % period; at a35b every lane of the routing
    warp then holds equal keys and 64 experts tie at the top."""
    L = synth.make_layer(shape, 23, device=DEV)
    rw = L["router_w"]
    E = shape.E
    if period == 2 and shape.E > 16:
        src = torch.arange(E, device=rw.device) // 2 * 2     # pairs (2j, 2j + 1)
    else:
        src = torch.arange(E, device=rw.device) % period
    L["router_w"] = rw[src].contiguous()
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    lay = oracle.Layer(L)
    x = _rows_with_distinct_margin(shape, lay, 31, gamma=L["gamma"] if shape.zipf else None)
    ref = lay.route(bits_np(x))
    ws = moe.Workspace(layer.desc, 1)
    idx, w = moe.router_topk(layer, x.to(DEV), ws)
    assert ws.status() == 0
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert np.allclose(w.cpu().numpy(), ref["w"], rtol=1e-4, atol=1e-6)
    # the tie structure is really there: some selected experts share a logit
    lg = ref["logits"][0][ref["idx"][0]]
    assert len(np.unique(lg)) < shape.k
