"""GPU parity of the tensor-core grouped products (moe_gate_up_tc,
moe_down_tc) against the fp64 oracle's dequantised weights.

The kernels split each weight w = q s + b (fp32) and each input into high and
low fp16 halves (each half rounded to 11 significant bits, so a value keeps
~22: relative error at most 2^-22 each), multiply the halves exactly and
accumulate in fp32 over K terms.  So for a dot product g = sum_k w_k x_k,
with S = sum_k |w_k| |x_k|,
    |g_gpu - g| <= eps * S,   eps = 2^-21 + 2 K 2^-24
(the accumulation term doubled for the tensor cores' own adder order), and
for act = silu(g) u (|silu'| < 1.1):
    |act_gpu - act| <= 1.1 eps S_g (|u| + eps S_u) + |silu(g)| eps S_u.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_moe_decode_layer_gb300 as moe

from helpers import bits_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _silu(g):
    return g / (1.0 + np.exp(-g))


def _case(shape, seed, M, experts, masks):
    L = synth.make_layer(shape, seed, device=DEV)
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    lay = oracle.Layer(L)
    x = synth.make_rows(shape, seed + 1, M, gamma=L["gamma"] if shape.zipf else None)
    xb = bits_np(x)
    hn64 = np.stack([oracle.rmsnorm(xb[r], lay.gamma, shape.eps) for r in range(M)])
    hn32 = hn64.astype(np.float32)
    hn = torch.from_numpy(hn32).to(DEV)
    ex = torch.tensor(experts, dtype=torch.int32, device=DEV)
    mk = torch.tensor([m - (1 << 32) if m >= (1 << 31) else m for m in masks], dtype=torch.int32, device=DEV)
    act = torch.full((len(experts), M, shape.I), float("nan"), dtype=torch.float32, device=DEV)
    act, err = moe.gate_up_tc(layer, hn, ex, mk, act=act)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = act.cpu().numpy().astype(np.float64)
    x64 = hn32.astype(np.float64)
    K = shape.H
    eps = 2.0 ** -21 + 2 * K * 2.0 ** -24
    for u, (e, m) in enumerate(zip(experts, masks)):
        Wg, Wu = (mat.dense() for mat in lay.expert(e)[:2])
        for r in range(M):
            if not (m >> r) & 1:
                assert np.isnan(got[u, r]).all(), f"row {r} outside the mask of slot {u} was written"
                continue
            g = Wg @ x64[r]
            up = Wu @ x64[r]
            Sg = np.abs(Wg) @ np.abs(x64[r])
            Su = np.abs(Wu) @ np.abs(x64[r])
            ref = _silu(g) * up
            tol = 1.1 * eps * Sg * (np.abs(up) + eps * Su) + np.abs(_silu(g)) * eps * Su
            bad = np.abs(got[u, r] - ref) > tol
            assert not bad.any(), (f"expert {e} row {r}: {bad.sum()} of {shape.I} outside the bound; "
                                   f"max err {np.abs(got[u, r] - ref).max()}, bound there {tol[bad][0]}")
    return got


def test_gate_up_tc_a35b_masks():
    """6-bit 35B-A3B experts, 32 rows: full, single, alternating, sparse and empty masks."""
    sh = synth.A35B
    full = (1 << 32) - 1
    _case(sh, 71, 32, [0, 3, 17, 128, 255, 40], [full, 1 << 31, 0x55555555, 0x00010001, 0, 0x0000000F])


def test_gate_up_tc_tiny_4bit_few_rows():
    """4-bit tiny-shape experts (I = 128: one tile), M = 3 rows."""
    sh = synth.TINY
    _case(sh, 72, 3, [0, 5, 15], [0b111, 0b010, 0b101])


def _down_case(shape, seed, M, experts, masks):
    """Down projection of random activations: y = W_down,e . a for each row of each mask."""
    L = synth.make_layer(shape, seed, device=DEV)
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    lay = oracle.Layer(L)
    g = torch.Generator().manual_seed(seed)
    a32 = (torch.randn((len(experts), M, shape.I), generator=g) * 0.3).numpy().astype(np.float32)
    ex = torch.tensor(experts, dtype=torch.int32, device=DEV)
    mk = torch.tensor([m - (1 << 32) if m >= (1 << 31) else m for m in masks], dtype=torch.int32, device=DEV)
    y = torch.full((len(experts), M, shape.H), float("nan"), dtype=torch.float32, device=DEV)
    y, err = moe.down_tc(layer, torch.from_numpy(a32).to(DEV), ex, mk, y=y)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = y.cpu().numpy().astype(np.float64)
    eps = 2.0 ** -21 + 2 * shape.I * 2.0 ** -24
    for u, (e, m) in enumerate(zip(experts, masks)):
        Wd = lay.expert(e)[2].dense()
        for r in range(M):
            if not (m >> r) & 1:
                assert np.isnan(got[u, r]).all()
                continue
            a = a32[u, r].astype(np.float64)
            ref = Wd @ a
            tol = eps * (np.abs(Wd) @ np.abs(a))
            bad = np.abs(got[u, r] - ref) > tol
            assert not bad.any(), f"expert {e} row {r}: {bad.sum()} outside the bound, max err {np.abs(got[u, r] - ref).max()}"


def test_down_tc_a35b_masks():
    """6-bit 35B-A3B down rows (K = I = 512, 16 tiles of H), 32 rows."""
    _down_case(synth.A35B, 81, 32, [2, 77, 255, 130], [(1 << 32) - 1, 0x80000001, 0x0F0F0F0F, 0])


def test_down_tc_tiny_4bit():
    """4-bit tiny down rows (K = I = 128, H = 256: two tiles), M = 5."""
    _down_case(synth.TINY, 82, 5, [1, 9], [0b10110, 0b00001])


def test_gate_up_tc_rejects_bad_args():
    sh = synth.TINY
    L = synth.make_layer(sh, 73, device=DEV)
    layer = moe.Layer(moe.desc_from_shape(sh), moe.layer_src_from_synth(L))
    hn = torch.zeros((33, sh.H), dtype=torch.float32, device=DEV)
    ex = torch.zeros(1, dtype=torch.int32, device=DEV)
    mk = torch.ones(1, dtype=torch.int32, device=DEV)
    with pytest.raises(moe.MoeError):
        moe.gate_up_tc(layer, hn, ex, mk)
    # the binding refuses, before any launch, buffers the kernel would overrun
    # or misread: an output smaller than [U, M, I], masks of another dtype
    with pytest.raises(ValueError):
        moe.gate_up_tc(layer, hn[:2], ex, mk, act=torch.zeros((1, 1, sh.I), dtype=torch.float32, device=DEV))
    with pytest.raises(ValueError):
        moe.gate_up_tc(layer, hn[:2], ex, mk.long())
