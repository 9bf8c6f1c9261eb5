"""GPU parity of the fused Q/K/V projection (moe_qkv_forward) against the
fp64 oracle, through the C ABI.  "Qwen3.5-397B on M5 Max" (openclawradar),
効果的な最適化: the Q, K and V projections fused so that the input row is
read once; the input is the MoE layer's normalised output (out_normed)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_moe_decode_layer_gb300 as moe
from quantized_moe_decode_layer_gb300 import _lib

from helpers import assert_close, bf16_tensor_to_f64, bits_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make_qkv(H, rows, bits, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    mats = [synth.quant_matrix(g, (n,), H, bits, DEV) for n in rows]
    return mats, moe.QKV(H, *mats, bits=bits), [oracle.Matrix.from_canonical(m) for m in mats]


def check(H, rows, bits, M, seed):
    mats, qkv, omats = make_qkv(H, rows, bits, seed)
    x = synth.make_rows(synth.LayerShape("x", H, 64, 2, 1, bits, 8, 0, False, 0, False), seed + 1, M)
    y, err = qkv.forward(x.to(DEV))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.qkv(omats, bits_np(x))
    got = y.double().cpu().numpy()
    assert_close(got, ref, f"qkv H={H} bits={bits} M={M}")
    # fp32 accumulation over H products: far inside the output tolerance
    scale = np.abs(np.concatenate([m.dense() for m in omats])) @ np.abs(oracle.bf16_patterns_to_double(bits_np(x))).T
    assert np.max(np.abs(got - ref) / (scale.T + 1e-30)) < 1e-5
    return qkv, x, y


@pytest.mark.parametrize("H,rows,bits,M", [(2048, (4096, 512, 512), 8, 1), (2048, (4096, 512, 512), 8, 4),
                                           (256, (64, 32, 32), 4, 3), (256, (64, 32, 32), 6, 8),
                                           (4096, (1024, 256, 256), 8, 2)])
def test_qkv_matches_oracle(H, rows, bits, M):
    check(H, rows, bits, M, 500 + H + bits + M)


def test_qkv_rows_independent_of_M():
    """Each row of a 5-row projection is bitwise the 1-row projection."""
    qkv, x, y = check(2048, (4096, 512, 512), 8, 5, 900)
    for m in range(5):
        y1, _ = qkv.forward(x[m:m + 1].contiguous().to(DEV))
        assert torch.equal(y1, y[m:m + 1])


def test_qkv_on_layer_out_normed():
    """The projection fed with a decode layer's fused out_normed, as in a
    transformer block: matches the oracle applied to the same bf16 rows."""
    shape = synth.A35B
    L = synth.make_layer(shape, 77, device=DEV)
    layer = moe.Layer(moe.desc_from_shape(shape), moe.layer_src_from_synth(L))
    ws = moe.Workspace(layer.desc, 2)
    x = synth.make_rows(shape, 78, 2, gamma=L["gamma"]).to(DEV)
    _, on = moe.decode_layer(layer, x, ws, normed=True)
    assert ws.status() == 0
    mats, qkv, omats = make_qkv(shape.H, (4096, 512, 512), 8, 79)
    y, err = qkv.forward(on)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(y.double().cpu().numpy(), oracle.qkv(omats, bits_np(on)), "qkv on out_normed")


def test_qkv_argument_errors():
    mats, qkv, _ = make_qkv(256, (64, 32, 32), 8, 3)
    lib = _lib.lib()
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((1, 128), dtype=torch.float32, device=DEV)
    e = torch.zeros(1, dtype=torch.int32, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    assert lib.moe_qkv_forward(None, x.data_ptr(), 1, y.data_ptr(), e.data_ptr(), s) == 1
    assert lib.moe_qkv_forward(qkv.handle, x.data_ptr(), 0, y.data_ptr(), e.data_ptr(), s) == 1
    assert lib.moe_qkv_forward(qkv.handle, x.data_ptr(), 1 << 20, y.data_ptr(), e.data_ptr(), s) == 2
    with pytest.raises(ValueError):
        qkv.forward(x.cpu())
