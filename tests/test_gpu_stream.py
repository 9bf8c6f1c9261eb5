"""Streamed layers (moe_streamed_*): routed experts in pinned host memory,
an HBM cache of expert slots, LRU eviction and next-layer prediction, against
the resident layers they were made from, through the C ABI.

Source: flash-moe (ja.news.hada.io), "SSD Expert Streaming" and "Trust the
OS" (only the selected experts are loaded; an LRU cache keeps the popular
ones); AiiStream Q3.6 article (648news) (the next layer's experts are
predicted and loaded ahead; output identical to the in-memory runtime);
"Qwen3.5-397B on M5 Max" (openclawradar), 効果的な最適化 (temporal expert
prediction).  The decode kernel is the resident one reading the cache
through the slot map, so every result must equal the resident layer's bits.
"""
import pytest
import torch

import synth
import quantized_moe_decode_layer_gb300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda"
SH = synth.A35B

_cache = {}


def resident_layers(n):
    if n not in _cache:
        desc = moe.desc_from_shape(SH)
        _cache[n] = [moe.Layer(desc, moe.layer_src_from_synth(synth.make_layer(SH, 4000 + i, device=DEV)))
                     for i in range(n)]
    return _cache[n]


def same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M", [1, 4])
def test_streamed_layer_equals_resident(M):
    """Route, make the selected experts resident, decode: the same bits as the
    resident layer; a second prepare of the same experts copies nothing."""
    lay = resident_layers(1)[0]
    st = moe.StreamedLayer(lay, n_slots=40)
    ws = moe.Workspace(lay.desc, M)
    x = synth.make_rows(SH, 71 + M, M, correlation=0.5 if M > 1 else 0.0).to(DEV)
    idx, _ = moe.router_topk(st, x, ws)
    ids = idx.flatten().tolist()
    n = len(set(ids))
    assert st.prepare(ids) == n
    assert st.prepare(ids) == 0
    s = st.stats()
    assert s["misses"] == n and s["hits"] == n and s["fetched"] == n and s["bytes"] == n * 2_555_904
    out, on = moe.decode_layer(st, x, ws, normed=True)
    assert ws.status() == 0
    ref, ref_n = moe.decode_layer(lay, x, ws, normed=True)
    assert same(out, ref) and same(on, ref_n)


def test_missing_expert_is_reported():
    """A decode whose selected experts were never made resident reports
    MOE_ERR_NOT_RESIDENT (the kernel reads slot 0 of the cache instead, never
    past it), and a later call after prepare is clean."""
    lay = resident_layers(1)[0]
    st = moe.StreamedLayer(lay, n_slots=8)
    ws = moe.Workspace(lay.desc, 1)
    x = synth.make_rows(SH, 81, 1).to(DEV)
    moe.decode_layer(st, x, ws)
    assert ws.status() == 7
    idx, _ = moe.router_topk(st, x, ws)
    st.prepare(idx.flatten().tolist())
    ws.init()
    out = moe.decode_layer(st, x, ws)
    assert ws.status() == 0
    assert same(out, moe.decode_layer(lay, x, ws))


def test_lru_eviction():
    """With k slots, a second set of experts evicts the first, and bringing
    the first back copies all of it again; values stay the resident ones."""
    lay = resident_layers(1)[0]
    st = moe.StreamedLayer(lay, n_slots=8)
    a = list(range(0, 8))
    b = list(range(8, 16))
    assert st.prepare(a) == 8
    assert st.prepare(b) == 8
    assert st.prepare(a[:4] + b[:4]) == 4
    s = st.stats()
    assert s["fetched"] == 20
    with pytest.raises(moe.MoeError):
        st.prepare(list(range(9)))          # more distinct experts than slots


@pytest.mark.parametrize("predict", [False, True])
def test_streamed_forward_equals_resident_chain(predict):
    """Four streamed layers with 16-slot caches over three tokens (experts
    evicted between tokens) give, token by token, the resident chain's bits;
    with prediction the next layer's predicted experts are prefetched."""
    layers = resident_layers(4)
    st = [moe.StreamedLayer(l, n_slots=16) for l in layers]
    ws = moe.Workspace(layers[0].desc, 1)
    for t in range(3):
        x = synth.make_rows(SH, 90 + t, 1).to(DEV)
        out, on = moe.streamed_forward(st, x, ws, normed=True, predict=predict)
        torch.cuda.synchronize()
        assert ws.status() == 0
        h = x
        for i, l in enumerate(layers):
            if i == len(layers) - 1:
                h, hn = moe.decode_layer(l, h, ws, normed=True)
            else:
                h = moe.decode_layer(l, h, ws)
        assert same(out, h) and same(on, hn), f"token {t}"
    tot = [s.stats() for s in st]
    assert sum(s["misses"] for s in tot) > 0
    if predict:
        assert all(s["predicted"] > 0 for s in tot[1:])
        assert sum(s["predicted_used"] for s in tot) > 0


def test_streamed_layers_in_one_persistent_launch():
    """A stack of streamed layers in one persistent launch, every layer's
    selected experts made resident beforehand, equals the resident stack."""
    layers = resident_layers(4)
    st = [moe.StreamedLayer(l, n_slots=24) for l in layers]
    ws = moe.Workspace(layers[0].desc, 3)
    x = synth.make_rows(SH, 99, 3, correlation=0.5).to(DEV)
    h = x
    for l, s in zip(layers, st):
        idx, _ = moe.router_topk(l, h, ws)
        s.prepare(idx.flatten().tolist())
        h = moe.decode_layer(l, h, ws)
    out = moe.Stack(st).forward(x, ws)
    assert ws.status() == 0
    ref = moe.Stack(layers).forward(x, ws)
    assert same(out, ref)
