"""The C-ABI library without a GPU: it loads, exports every symbol that
include/moe.h declares, checks its arguments, and sizes blobs/workspaces."""
import ctypes as C
import os
import re

import pytest

import synth
import quantized_moe_decode_layer_gb300 as moe
from quantized_moe_decode_layer_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    L = moe.lib()
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SYMBOLS)


def test_host_selftest():
    """The code-extraction tables and the launch plans of the test shapes
    (every row count, several SM counts) meet the kernel's invariants."""
    assert moe.lib().moe_selftest_host() == 0


def test_status_strings():
    L = moe.lib()
    for code, name in _lib.STATUS.items():
        assert L.moe_status_str(code).decode() == name


@pytest.mark.parametrize("shape,per_expert", [(synth.A35B, 2_555_904), (synth.B397, 7_077_888)])
def test_pack_size_counts(shape, per_expert):
    """Blob = router (row-major, and the input-major copy with its rows padded
    to 16: one code byte per weight, one scale/bias word per group) + gammas
    + experts + shared expert; no per-row padding at these widths, so the
    expert bytes are exactly the algorithmic ones."""
    d = moe.desc_from_shape(shape)
    total = moe.pack_size(d)
    H, I, E, Is = shape.H, shape.I, shape.E, shape.I_shared
    expert = 2 * I * (H * shape.routed_bits // 8 + H // 64 * 4) + H * (I * shape.routed_bits // 8 + I // 64 * 4)
    assert expert == per_expert
    shared = 2 * Is * (H + H // 64 * 4) + H * (Is + Is // 64 * 4)
    router = (E + 1) * (H + H // 64 * 4)
    erp = (E + 1 + 15) // 16 * 16
    router_t = H * erp + H // 64 * erp * 4
    known = E * expert + shared + router + router_t + 4 * H
    assert total >= known
    assert total - known < 9 * 256


def test_argument_errors():
    L = moe.lib()
    d = moe.desc_from_shape(synth.TINY)
    n = C.c_size_t()
    assert L.moe_pack_size(None, C.byref(n)) == 1
    bad = moe.make_desc(256, 128, 16, 2, 5, router_bits=0, has_shared=False)
    assert L.moe_pack_size(C.byref(bad), C.byref(n)) == 2
    bad = moe.make_desc(256, 128, 16, 17, 4, router_bits=0, has_shared=False)   # k > E
    assert L.moe_pack_size(C.byref(bad), C.byref(n)) == 2
    bad = moe.make_desc(320, 128, 16, 2, 4, router_bits=0, has_shared=False)   # H not 256/multiple of 512
    assert L.moe_pack_size(C.byref(bad), C.byref(n)) == 2
    bad = moe.make_desc(256, 512, 16, 2, 4, router_bits=0, has_shared=False)   # I > H
    assert L.moe_pack_size(C.byref(bad), C.byref(n)) == 2
    assert L.moe_workspace_size(C.byref(d), 0, C.byref(n)) == 1
    h = C.c_void_p()
    src = _lib.SrcLayer()
    assert L.moe_pack_weights(C.byref(d), C.byref(src), None, 0, C.byref(h), None) == 1
    assert L.moe_pack_weights(C.byref(d), C.byref(src), C.c_void_p(256), 16, C.byref(h), None) == 3
    assert L.moe_decode_layer(None, None, 1, None, None, None, 0, None) == 1
    assert L.moe_router_topk(None, None, 1, None, None, None, 0, None) == 1
    assert L.moe_stack_create(None, 0, C.byref(h)) == 1
    L.moe_layer_destroy(None)
    L.moe_stack_destroy(None)


def test_workspace_sizes_grow_with_rows():
    d = moe.desc_from_shape(synth.A35B)
    assert moe.workspace_size(d, 1) < moe.workspace_size(d, 8) < moe.workspace_size(d, 32)


def test_binding_rejects_host_and_strided_tensors():
    """The binding hands the library device pointers only: a host tensor, or
    a strided view whose memory is not the logical layout, is refused before
    any call."""
    import torch
    from quantized_moe_decode_layer_gb300 import api
    assert api._ptr(None) is None
    with pytest.raises(ValueError):
        api._ptr(torch.zeros(4))
    with pytest.raises(ValueError):
        api._ptr(torch.zeros(4, 4).t())
    with pytest.raises(ValueError):
        api._need(torch.zeros((2, 8), dtype=torch.bfloat16), "x", torch.bfloat16, (None, 8))
    with pytest.raises(ValueError):
        api._need([0.0] * 8, "x", torch.bfloat16, (None, 8))


def test_binding_wrappers_for_selftest_and_noalloc():
    """The binding carries the ABI's names: the host selftest through it
    finds no violation, and the no-alloc decode refuses host tensors before
    calling the library."""
    import types

    import torch
    assert moe.selftest_host() == 0
    stand_in = types.SimpleNamespace(desc=types.SimpleNamespace(H=8))
    with pytest.raises(ValueError):
        moe.decode_layer_noalloc(stand_in, torch.zeros((1, 8), dtype=torch.bfloat16))


def test_qkv_sizes_and_argument_errors():
    """The fused projection's size query counts stacked packed rows; bad
    descriptors and missing pointers are refused before any device work."""
    L = moe.lib()
    n = C.c_size_t()
    d = _lib.QkvDesc(2048, 4096, 512, 512, 8)
    assert L.moe_qkv_pack_size(C.byref(d), C.byref(n)) == 0
    assert n.value == 5120 * (2048 + 32 * 4)        # codes + one scale/bias word per 64-group
    d6 = _lib.QkvDesc(256, 64, 32, 32, 6)
    assert L.moe_qkv_pack_size(C.byref(d6), C.byref(n)) == 0 and n.value == 128 * (192 + 16)
    for bad in (_lib.QkvDesc(2048, 4096, 512, 512, 5), _lib.QkvDesc(100, 64, 0, 0, 8), _lib.QkvDesc(256, 0, 0, 0, 8)):
        assert L.moe_qkv_pack_size(C.byref(bad), C.byref(n)) == 2
    assert L.moe_qkv_pack_size(None, C.byref(n)) == 1
    h = C.c_void_p()
    m = _lib.SrcMatrix()
    assert L.moe_qkv_pack(C.byref(d), C.byref(m), C.byref(m), C.byref(m), None, 0, C.byref(h), None) == 1
    assert L.moe_qkv_pack(C.byref(d), C.byref(m), C.byref(m), C.byref(m), C.c_void_p(256), 16, C.byref(h), None) == 3
    assert L.moe_qkv_forward(None, None, 1, None, None, None) == 1
    L.moe_qkv_destroy(None)


def _run_checked(code: str) -> str:
    """Run `code` in a child interpreter that loads the bounds-checked build."""
    import subprocess
    import sys
    from quantized_moe_decode_layer_gb300 import build as b
    b.build(debug_bounds=True)
    env = dict(os.environ, MOE_DEBUG_BOUNDS="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    return r.stdout


def test_build_flags_of_both_builds():
    """The normal build reports no flags and refuses the injection hook; the
    checked build (selected by MOE_DEBUG_BOUNDS=1 at load time) reports
    MOE_BUILD_DEBUG_BOUNDS, takes the hook, and exports the same symbols."""
    assert moe.build_flags() == 0
    assert not _lib.DEBUG_BOUNDS and _lib.LIB_PATH.endswith("libmoe.so")
    with pytest.raises(moe.MoeError) as ei:
        moe.debug_inject(3)
    assert ei.value.code == 2
    out = _run_checked(
        "import quantized_moe_decode_layer_gb300 as m\n"
        "from quantized_moe_decode_layer_gb300 import _lib\n"
        "L = m.lib()\n"
        "assert _lib.LIB_PATH.endswith('libmoe_debug.so')\n"
        "missing = [n for n in _lib.SYMBOLS if not hasattr(L, n)]\n"
        "m.debug_inject(7); m.debug_inject(-1)\n"
        "print(m.build_flags(), len(missing), L.moe_selftest_host())\n")
    assert out.split() == ["1", "0", "0"]


def test_attention_sizes_and_argument_errors():
    """Workspace size of the decode attention (per 512-position chunk: 2 KV
    heads x 64 query columns x (256 + 2) floats, the maxima and sums first;
    then for the merge, per (row, query head) of 8 x 16 and segment of 16
    chunks, a sum and 256 outputs, and a counter per (row, head); each
    region 256-aligned) and its argument checks, which reject before any
    launch."""
    L = moe.lib()
    n = C.c_size_t()

    def a256(v):
        return (v + 255) // 256 * 256
    for T_cap, chunks in ((4096, 8), (40960, 80)):
        assert L.moe_attn_workspace_size(T_cap, C.byref(n)) == 0
        segs = (chunks + 15) // 16
        po = a256(chunks * 2 * 64 * 2 * 4)
        sl = a256(po + chunks * 2 * 64 * 256 * 4)
        so = a256(sl + 128 * segs * 4)
        cnt = a256(so + 128 * segs * 256 * 4)
        assert n.value == a256(cnt + 128 * 4)
    assert L.moe_attn_workspace_size(0, C.byref(n)) == 1
    fake = 1 << 20   # never dereferenced: every call below is rejected first
    err = fake
    # M out of range, T_cap not a multiple of 8, rows past the cache, null pointers
    assert L.moe_attn_decode(fake, fake, fake, 64, 0, 0, fake, fake, 1 << 30, err, None) == 1
    assert L.moe_attn_decode(fake, fake, fake, 64, 0, 9, fake, fake, 1 << 30, err, None) == 1
    assert L.moe_attn_decode(fake, fake, fake, 60, 0, 1, fake, fake, 1 << 30, err, None) == 1
    assert L.moe_attn_decode(fake, fake, fake, 64, 63, 2, fake, fake, 1 << 30, err, None) == 1
    assert L.moe_attn_decode(None, fake, fake, 64, 0, 1, fake, fake, 1 << 30, err, None) == 1
    assert L.moe_attn_decode(fake + 8, fake, fake, 64, 0, 1, fake, fake, 1 << 30, err, None) == 1
    assert L.moe_attn_decode(fake, fake, fake, 64, 0, 1, fake, fake, 16, err, None) == 3
    assert L.moe_attn_append(fake, fake, 0, 0, fake, fake, 64, None) == 1
    assert L.moe_attn_append(fake, fake, 2, 63, fake, fake, 64, None) == 1


def test_streamed_sizes_and_argument_errors():
    """A streamed layer's device bytes: the resident parts (router, gammas,
    shared expert) plus n_slots experts plus the slot map and a table of two
    fetch jobs (32 bytes each) per slot, 256-aligned; slot
    counts below k or above E and null handles are refused."""
    L = moe.lib()
    d = moe.desc_from_shape(synth.A35B)
    n16, n8 = C.c_size_t(), C.c_size_t()
    assert L.moe_streamed_size(C.byref(d), 16, C.byref(n16)) == 0
    assert L.moe_streamed_size(C.byref(d), 8, C.byref(n8)) == 0
    # eight more experts of 2,555,904 bytes, and 8 more 512-byte pairs of gather jobs
    assert n16.value - n8.value == 8 * 2_555_904 + 512
    assert n16.value < moe.pack_size(d)
    assert L.moe_streamed_size(C.byref(d), 7, C.byref(n8)) == 1      # fewer slots than k
    assert L.moe_streamed_size(C.byref(d), 257, C.byref(n8)) == 1    # more slots than experts
    h = C.c_void_p()
    assert L.moe_streamed_create(None, 1, 1, 1, 1, 16, C.byref(h), None) == 1
    assert L.moe_streamed_prepare(None, None, 0, None, None) == 1
    assert L.moe_streamed_stats(None, None, None, None, None, None, None) == 1
    assert L.moe_streamed_forward(None, 1, None, 1, None, None, None, 0, None, 0, 0, None, None) == 1
    assert L.moe_streamed_layer(None) is None
