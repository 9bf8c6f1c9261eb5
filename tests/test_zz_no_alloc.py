"""moe_decode_layer_noalloc: the decode call for callers that cannot allocate
device memory when they call it (stream capture into a CUDA graph, plug-ins
living inside another framework's memory pool, latency-critical paths that
must not take an allocation's synchronisation).  It uses a fixed scratch
array inside the library instead of a caller workspace; its results must
match the workspace entry point's.

This file is collected last on purpose: it adds one entry point on top of
everything else, so a run that stops at the first failure has already run the
other tests."""
import numpy as np
import pytest
import torch

import synth
import quantized_moe_decode_layer_gb300 as moe
from quantized_moe_decode_layer_gb300 import _lib

from helpers import ATOL, RTOL, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    return t.view(torch.int16) if t is not None and t.dtype == torch.bfloat16 else t


def call_noalloc(layer, x, normed):
    out = torch.empty_like(x)
    on = torch.empty_like(x) if normed else None
    rc = _lib.lib().moe_decode_layer_noalloc(layer.handle, _bits(x).data_ptr(), x.shape[0], _bits(out).data_ptr(),
                                             _bits(on).data_ptr() if on is not None else None,
                                             torch.cuda.current_stream().cuda_stream)
    assert rc == 0, _lib.STATUS.get(rc, rc)
    return out, on


def close(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    bad = np.abs(g - r) > ATOL + RTOL * np.abs(r)
    assert not bad.any(), f"{what}: {bad.sum()} elements differ"


@pytest.mark.parametrize("shape,M", [(synth.TINY, 3), (synth.A35B, 1), (synth.A35B, 4)])
def test_noalloc_matches_workspace_entry_point(shape, M):
    L = synth.make_layer(shape, 61, device=DEV)
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    x = synth.make_rows(shape, 62, M, gamma=L["gamma"], correlation=0.5 if M > 1 else 0.0).to(DEV)
    ws = moe.Workspace(layer.desc, M)
    ref, ref_n = moe.decode_layer(layer, x, ws, normed=True)
    assert ws.status() == 0
    for _ in range(2):   # two calls in a row share the same scratch array
        out, on = call_noalloc(layer, x, normed=True)
        assert moe.noalloc_status() == 0
        close(out, ref, f"{shape.name} M={M} out")
        close(on, ref_n, f"{shape.name} M={M} out_normed")
        # the same kernel with the same summation order: the bits agree too
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(on.view(torch.int16), ref_n.view(torch.int16))


def test_noalloc_python_wrapper():
    """The binding's decode_layer_noalloc gives the workspace call's result."""
    shape = synth.A35B
    L = synth.make_layer(shape, 64, device=DEV)
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    x = synth.make_rows(shape, 65, 2, gamma=L["gamma"], correlation=0.5).to(DEV)
    ws = moe.Workspace(layer.desc, 2)
    ref, ref_n = moe.decode_layer(layer, x, ws, normed=True)
    out, on = moe.decode_layer_noalloc(layer, x, normed=True)
    assert moe.noalloc_status() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(on.view(torch.int16), ref_n.view(torch.int16))


def test_noalloc_reports_a_device_timeout():
    """A device wait that runs out inside the no-alloc call is reported by
    moe_noalloc_status (the router logit of one expert is left unpublished
    through the debug switch, so every CTA's wait for it gives up after 50
    ms); the next call starts clean and gives the right result again."""
    shape = synth.TINY
    L = synth.make_layer(shape, 66, device=DEV)
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    x = synth.make_rows(shape, 67, 1).to(DEV)
    good, _ = call_noalloc(layer, x, normed=False)
    assert moe.noalloc_status() == 0
    try:
        moe.debug_set(skip_row=3, timeout_ns=50_000_000)
        call_noalloc(layer, x, normed=False)
        assert moe.noalloc_status() == 5   # MOE_ERR_TIMEOUT
    finally:
        moe.debug_set(-1, 0)
    again, _ = call_noalloc(layer, x, normed=False)
    assert moe.noalloc_status() == 0
    assert torch.equal(again.view(torch.int16), good.view(torch.int16))


def test_noalloc_rejects_rows_beyond_the_scratch():
    shape = synth.TINY
    L = synth.make_layer(shape, 63, device=DEV)
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    x = torch.zeros((1, shape.H), dtype=torch.bfloat16, device=DEV)
    too_many = 1 << 16   # the host staging area alone exceeds the scratch
    rc = _lib.lib().moe_decode_layer_noalloc(layer.handle, _bits(x).data_ptr(), too_many, _bits(x).data_ptr(), None,
                                             torch.cuda.current_stream().cuda_stream)
    assert rc == 3   # MOE_ERR_BUFFER_TOO_SMALL, nothing enqueued
