"""Pins for the fp64 CPU oracle (no GPU).

Each test ties an oracle function to something other than itself: values
computed by hand, a hand-packed bit stream, closed forms, library routines
(torch / numpy in fp64) on special cases, brute force on tiny inputs, and the
expert size printed by flash-moe (hada.io topic 27758, "SSD Expert Streaming").
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(v: float) -> int:
    """bf16 pattern of a float32-representable value via torch's converter."""
    return int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF


# ----------------------------------------------------------------- bf16 / pack

def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(0)
    vals = torch.randn(4000, generator=g, dtype=torch.float32) * torch.exp(torch.randn(4000, generator=g) * 6)
    # exact halfway cases between neighbouring bf16 values (ties to even)
    base = torch.randn(1000, generator=g, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).to(torch.int32)
    ties = ((base << 16) | 0x8000).to(torch.int32).view(torch.float32)
    vals = torch.cat([vals, ties, torch.tensor([0.0, -0.0, 1e-40, -3e-39, 3.3e38, float("inf")])])
    ref = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round_array(vals.double().numpy())
    assert np.array_equal(got, ref)


def test_pack_hand_6bit():
    # codes (1, 2, 3, 4) least significant bit first: byte0 = 1 | (2 & 3) << 6,
    # byte1 = (2 >> 2) | (3 & 15) << 4, byte2 = (3 >> 4) | 4 << 2
    assert list(oracle.pack_bits(np.array([1, 2, 3, 4]), 6)) == [0x81, 0x30, 0x10]
    assert list(oracle.pack_bits(np.array([1, 2, 15, 0]), 4)) == [0x21, 0x0F]
    assert list(oracle.pack_bits(np.array([7, 200]), 8)) == [7, 200]


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_pack_roundtrip_and_size(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=64 * 5, dtype=np.uint8)
    packed = oracle.pack_bits(codes, bits)
    assert packed.size == 64 * 5 * bits // 8
    assert np.array_equal(oracle.unpack_bits(packed, codes.size, bits), codes)
    # bit i*b+t of the stream is bit t of code i
    bitstream = np.unpackbits(packed, bitorder="little")
    for i in (0, 1, 63, 64 * 5 - 1):
        v = sum(int(bitstream[i * bits + t]) << t for t in range(bits))
        assert v == codes[i]


def test_expert_size_matches_page():
    """A 4-bit expert of the 512-expert model (hidden 4096, gate/up/down, I=1024)
    stored as 64-code groups with a bf16 scale and bias is 6.75 MiB."""
    g = json.load(open(os.path.join(GOLDEN, "page_sizes.json")))
    H, I = g["hidden_397b"], 1024
    row_codes = oracle.pack_bits(np.zeros(H, np.uint8), 4).size
    per_row = row_codes + (H // 64) * 4
    per_row_down = oracle.pack_bits(np.zeros(I, np.uint8), 4).size + (I // 64) * 4
    total = 2 * I * per_row + H * per_row_down
    assert total == 7_077_888
    assert abs(total / 2 ** 20 - g["expert_4bit_bytes_approx_MB"]) < 1e-9


# ------------------------------------------------------------------- dequant

@pytest.mark.parametrize("bits", [4, 6, 8])
def test_dequant_hand(bits):
    n = 1 << bits
    cols = max(64, n)
    codes = (np.arange(cols) % n).astype(np.uint8).reshape(1, cols)
    s = np.full((1, cols // 64), bf16(0.5), np.uint16)
    b = np.full((1, cols // 64), bf16(-1.0), np.uint16)
    m = oracle.Matrix(bits, codes, s, b)
    for c in range(cols):
        assert m.weight(0, c) == codes[0, c] / 2.0 - 1.0


def test_dequant_group_index():
    # distinct scale per group: element (r, c) must use group c // 64 of row r
    codes = np.ones((2, 128), np.uint8)
    s = np.array([[bf16(1.0), bf16(2.0)], [bf16(4.0), bf16(8.0)]], np.uint16)
    b = np.array([[bf16(0.0), bf16(0.5)], [bf16(0.25), bf16(0.125)]], np.uint16)
    m = oracle.Matrix(4, codes, s, b)
    assert m.weight(0, 63) == 1.0 and m.weight(0, 64) == 2.5
    assert m.weight(1, 0) == 4.25 and m.weight(1, 127) == 8.125


# ----------------------------------------------------------------- quantiser

@pytest.mark.parametrize("bits", [4, 6, 8])
def test_quantize_roundtrip_identity(bits):
    """Groups holding both code 0 and code 2^b-1 with bf16 (s, b) come back unchanged."""
    rng = np.random.default_rng(10 + bits)
    rows = 200
    qmax = (1 << bits) - 1
    codes = rng.integers(0, qmax + 1, size=(rows, 64), dtype=np.uint8)
    codes[:, 3] = 0
    codes[:, 40] = qmax
    s = torch.tensor(np.abs(rng.normal(0, 0.02, rows)) * 15 / qmax + 1e-4, dtype=torch.float32).to(torch.bfloat16)
    b = torch.tensor(rng.normal(0, 0.01, rows), dtype=torch.float32).to(torch.bfloat16)
    w = (torch.tensor(codes, dtype=torch.float32) * s.float()[:, None] + b.float()[:, None])
    q2, s2, b2 = oracle.quantize_matrix(w.numpy(), bits)
    assert np.array_equal(q2, codes)
    assert np.array_equal(s2[:, 0], s.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(b2[:, 0], b.view(torch.int16).numpy().view(np.uint16))


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_quantize_error_bound(bits):
    rng = np.random.default_rng(20 + bits)
    w = rng.normal(0, 0.05, size=(64, 128)).astype(np.float32)
    w[0, :64] = 0.25  # constant group: s = 0, every code 0, value = bf16(min)
    q, s, b = oracle.quantize_matrix(w, bits)
    m = oracle.Matrix(bits, q, s, b)
    deq = m.dense()
    sd = np.repeat(oracle.bf16_patterns_to_double(s), 64, axis=1)
    wg = w.astype(np.float64).reshape(64, 2, 64)
    rng_ = (wg.max(axis=2) - wg.min(axis=2)).repeat(64, axis=1)
    mn = np.repeat(wg.min(axis=2), 64, axis=1)
    bound = sd / 2 + rng_ * 2.0 ** -8 + np.abs(mn) * 2.0 ** -8 + 1e-12
    assert np.all(np.abs(deq - w) <= bound)
    assert np.all(q[0, :64] == 0) and s[0, 0] == 0
    assert int(q.max()) <= (1 << bits) - 1


# ------------------------------------------------------------------- rmsnorm

def test_rmsnorm_closed_form():
    H, eps = 256, 1e-6
    c = 0.75
    x = np.full(H, bf16(c), np.uint16)
    gam = np.array([bf16(1.0 + 0.01 * (j % 7)) for j in range(H)], np.uint16)
    hn = oracle.rmsnorm(x, gam, eps)
    expect = c / math.sqrt(c * c + eps) * oracle.bf16_patterns_to_double(gam)
    assert np.allclose(hn, expect, rtol=1e-14, atol=0)


def test_rmsnorm_matches_torch():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(2048, generator=g).to(torch.bfloat16)
    gam = (1 + 0.1 * torch.randn(2048, generator=g)).to(torch.bfloat16)
    ref = F.rms_norm(x.double()[None], (2048,), weight=gam.double(), eps=1e-6)[0].numpy()
    got = oracle.rmsnorm(synth.bf16_bits(x).numpy().view(np.uint16), synth.bf16_bits(gam).numpy().view(np.uint16), 1e-6)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------- routing

def test_topk_crafted():
    idx, w, probs, margin = oracle.topk(np.array([0.0, 1.0, 2.0, 3.0]), 2)
    assert list(idx) == [3, 2]
    s1 = 1 / (1 + math.exp(-1.0))
    assert abs(w[0] - s1) < 1e-15 and abs(w[1] - (1 - s1)) < 1e-15
    assert abs(margin - 1.0) < 1e-15
    assert abs(probs.sum() - 1) < 1e-15
    # ties go to the lower expert id, and the weights of tied experts are equal
    idx, w, _, margin = oracle.topk(np.array([1.0, 5.0, 1.0, 5.0, 0.0]), 3)
    assert list(idx) == [1, 3, 0] and margin == 0.0
    assert w[0] == w[1]


def test_topk_matches_torch():
    g = torch.Generator().manual_seed(4)
    for E, k in [(16, 2), (256, 8), (512, 10)]:
        for _ in range(20):
            lg = torch.randn(E, generator=g, dtype=torch.float64) * 2
            idx, w, probs, margin = oracle.topk(lg.numpy(), k)
            p = torch.softmax(lg, 0)
            tv, ti = torch.topk(p, k)
            assert list(idx) == ti.tolist()
            assert np.allclose(w, (tv / tv.sum()).numpy(), rtol=1e-13)
            assert abs(w.sum() - 1.0) < 1e-12
            assert np.allclose(probs, p.numpy(), rtol=1e-13)
            srt = torch.sort(lg, descending=True).values
            assert abs(margin - (srt[:k] - srt[1:k + 1]).min().item()) < 1e-13


# -------------------------------------------------------------- layer vs dense

def dense_layer(layer: oracle.Layer, x_bits: np.ndarray):
    """The layer in plain torch fp64 over fully dequantised matrices, with the
    library's RMSNorm, softmax, topk, silu and sigmoid."""
    sh = layer.shape
    x = torch.tensor(oracle.bf16_patterns_to_double(x_bits))
    gam = torch.tensor(oracle.bf16_patterns_to_double(layer.gamma))
    hn = F.rms_norm(x, (sh.H,), weight=gam, eps=sh.eps)
    R = torch.tensor(layer.router.dense())
    logits = hn @ R.T
    p = torch.softmax(logits, -1)
    tv, ti = torch.topk(p, sh.k, dim=-1)
    w = tv / tv.sum(-1, keepdim=True)
    o = x.clone()
    for m in range(x.shape[0]):
        for i in range(sh.k):
            G, U, D = (torch.tensor(t.dense()) for t in layer.expert(int(ti[m, i])))
            o[m] += w[m, i] * (D @ (F.silu(G @ hn[m]) * (U @ hn[m])))
        if layer.shared:
            G, U, D = (torch.tensor(t.dense()) for t in layer.shared)
            sg = torch.sigmoid(torch.tensor(layer.sgate.dense())[0] @ hn[m])
            o[m] += sg * (D @ (F.silu(G @ hn[m]) * (U @ hn[m])))
    return o.numpy(), ti.numpy(), w.numpy()


def test_tiny_layer_matches_dense():
    L = synth.make_layer(synth.TINY, 11)
    lay = oracle.Layer(L)
    xb = synth.bf16_bits(synth.make_rows(synth.TINY, 12, 3)).numpy().view(np.uint16)
    r = lay.forward(xb)
    o, idx, w = dense_layer(lay, xb)
    assert np.array_equal(r["idx"], idx)
    assert np.allclose(r["w"], w, rtol=1e-12)
    assert np.allclose(r["o"], o, rtol=1e-12, atol=1e-12)
    # out is the bf16 rounding of o; out_n is RMSNorm(out) * gamma_next
    assert np.array_equal(r["out"], oracle.bf16_round_array(r["o"]))
    out_d = torch.tensor(oracle.bf16_patterns_to_double(r["out"]))
    gn = torch.tensor(oracle.bf16_patterns_to_double(lay.gamma_next))
    on = F.rms_norm(out_d, (lay.H,), weight=gn, eps=lay.eps).numpy()
    assert np.allclose(r["on"], on, rtol=1e-13, atol=1e-15)


def test_shared_expert_layer_matches_dense():
    """A small shape with every feature of the 35B-A3B layer: 6-bit experts,
    8-bit router, shared expert with sigmoid gate, Zipf router term."""
    sh = synth.LayerShape("mini", 128, 64, 12, 3, 6, 8, 8, True, 128, True)
    L = synth.make_layer(sh, 5)
    lay = oracle.Layer(L)
    xb = synth.bf16_bits(synth.make_rows(sh, 6, 2, gamma=L["gamma"])).numpy().view(np.uint16)
    r = lay.forward(xb)
    o, idx, w = dense_layer(lay, xb)
    assert np.array_equal(r["idx"], idx)
    assert np.allclose(r["o"], o, rtol=1e-12, atol=1e-12)
    assert np.all(r["sigma"] > 0) and np.all(r["sigma"] < 1)


def test_k1_single_expert_is_swiglu_ffn():
    """k = 1 with one expert, no shared expert: out = x + FFN(RMSNorm(x))."""
    sh = synth.LayerShape("one", 128, 64, 1, 1, 8, 8, 0, False, 0, False)
    L = synth.make_layer(sh, 9)
    lay = oracle.Layer(L)
    xb = synth.bf16_bits(synth.make_rows(sh, 1, 1)).numpy().view(np.uint16)
    r = lay.forward(xb)
    assert r["w"][0, 0] == 1.0 and r["idx"][0, 0] == 0
    x = torch.tensor(oracle.bf16_patterns_to_double(xb))
    hn = F.rms_norm(x, (128,), weight=torch.tensor(oracle.bf16_patterns_to_double(lay.gamma)), eps=1e-6)
    G, U, D = (torch.tensor(t.dense()) for t in lay.expert(0))
    ffn = F.linear(F.silu(F.linear(hn, G)) * F.linear(hn, U), D)
    assert np.allclose(r["o"], (x + ffn).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bits,K", [(6, 2048), (8, 2048), (4, 4096), (6, 512)])
def test_matvec_full_width_matches_dense(bits, K):
    """Dequantised mat-vec at the full widths (6-bit H=2048 experts, 8-bit
    shared/router, 4-bit H=4096 experts, 6-bit I=512 down rows)."""
    g = torch.Generator().manual_seed(bits * 100 + K)
    Q = synth.quant_matrix(g, (8,), K, bits, "cpu")
    m = oracle.Matrix.from_canonical(Q)
    x = np.random.default_rng(1).normal(size=K)
    ref = m.dense() @ x
    for r in range(8):
        got = sum(m.weight(r, c) * x[c] for c in range(0, K, 1))
        assert abs(got - ref[r]) <= 1e-12 * (1 + abs(ref[r]))


def test_rows_independent():
    L = synth.make_layer(synth.TINY, 21)
    lay = oracle.Layer(L)
    xb = synth.bf16_bits(synth.make_rows(synth.TINY, 22, 4)).numpy().view(np.uint16)
    r4 = lay.forward(xb)
    for m in range(4):
        r1 = lay.forward(xb[m:m + 1])
        assert np.array_equal(r1["o"][0], r4["o"][m])
        assert np.array_equal(r1["idx"][0], r4["idx"][m])


def test_stack_is_chained_layers():
    layers = [oracle.Layer(synth.make_layer(synth.TINY, 30 + i)) for i in range(3)]
    xb = synth.bf16_bits(synth.make_rows(synth.TINY, 33, 2)).numpy().view(np.uint16)
    res = oracle.stack(layers, xb)
    x = xb
    for i, lay in enumerate(layers):
        r = lay.forward(x, normed=(i == 2))
        assert np.array_equal(r["out"], res[i]["out"])
        x = r["out"]
    assert np.array_equal(res[-1]["out_n"], oracle.bf16_round_array(res[-1]["on"]))


def test_expert_relabelling_invariance():
    """Relabelling the experts (router row e and expert e's weights both moved
    to id pi(e)) moves the selected ids to pi(idx) and leaves the weights and
    the output unchanged: the router row and the weights of one expert stay
    paired, whatever the labels."""
    sh = synth.LayerShape("mini", 128, 64, 12, 3, 6, 8, 8, True, 128, True)
    L = synth.make_layer(sh, 41)
    pi = torch.randperm(sh.E, generator=torch.Generator().manual_seed(7))
    inv = torch.argsort(pi)
    P = dict(L)
    P["router_w"] = L["router_w"][inv]
    for key in ("gate", "up", "down"):
        P[key] = {f: (v[inv] if isinstance(v, torch.Tensor) else v) for f, v in L[key].items()}
    xb = synth.bf16_bits(synth.make_rows(sh, 42, 3, gamma=L["gamma"])).numpy().view(np.uint16)
    r = oracle.Layer(L).forward(xb)
    rp = oracle.Layer(P).forward(xb)
    assert np.array_equal(rp["idx"], pi.numpy()[r["idx"]])
    assert np.allclose(rp["w"], r["w"], rtol=1e-14, atol=0)
    assert np.allclose(rp["o"], r["o"], rtol=1e-12, atol=1e-14)
    # a label that is not carried over (the down weights left in place) changes the output
    Q = dict(P)
    Q["down"] = L["down"]
    rq = oracle.Layer(Q).forward(xb)
    assert not np.allclose(rq["o"], r["o"], rtol=1e-6, atol=1e-9)


def test_threads_give_the_same_bits():
    """The all-cores oracle (mat-vec output rows over threads) equals the
    single-core oracle bit for bit."""
    L = synth.make_layer(synth.TINY, 41)
    lay = oracle.Layer(L)
    xb = synth.bf16_bits(synth.make_rows(synth.TINY, 42, 3)).numpy().view(np.uint16)
    one = lay.forward(xb)
    try:
        oracle.set_threads(max(2, oracle.max_threads()))
        many = lay.forward(xb)
    finally:
        oracle.set_threads(1)
    for key in ("o", "on", "logits", "w", "sigma"):
        assert np.array_equal(one[key], many[key]), key
    for key in ("out", "out_n", "idx"):
        assert np.array_equal(one[key], many[key]), key


@pytest.mark.parametrize("bits", [8, 4])
def test_qkv_matches_dense_product(bits):
    """The fused Q/K/V projection equals a dense fp64 product of the fully
    dequantised stacked matrix (numpy, independent of the C code), and its
    row blocks equal the three separate projections."""
    g = torch.Generator().manual_seed(77 + bits)
    H = 256
    mats = [oracle.Matrix.from_canonical(synth.quant_matrix(g, (n,), H, bits, "cpu")) for n in (64, 32, 32)]
    xb = synth.bf16_bits(synth.make_rows(synth.TINY, 5, 3)).numpy().view(np.uint16)
    y = oracle.qkv(mats, xb)
    x = oracle.bf16_patterns_to_double(xb)
    dense = np.concatenate([m.dense() for m in mats])
    assert y.shape == (3, 128)
    assert np.allclose(y, x @ dense.T, rtol=1e-12, atol=1e-12)
    off = 0
    for m in mats:
        alone = oracle.qkv([m], xb)
        assert np.array_equal(alone, y[:, off:off + m.rows])
        off += m.rows
    # a transposed operand or a dropped bias would not match
    assert not np.allclose(y, x @ (dense - dense.mean()).T, rtol=1e-6, atol=1e-6)


# ------------------------------------------------------ decode attention

def _attn_bits(t):
    return synth.bf16_bits(t).numpy().view(np.uint16)


def test_gqa_single_key_returns_its_value():
    """One key (position 0, one row): its softmax weight is 1, so every
    query head of key/value head g returns v[g][:, 0]."""
    q, k, vt = synth.make_attn(8, 1, 1, 3)
    o, oabs = oracle.gqa_decode(_attn_bits(q), _attn_bits(k), _attn_bits(vt), 0)
    v0 = vt[:, :, 0].double().numpy()
    for h in range(16):
        assert np.array_equal(o[0, h], v0[h // 8])
        assert np.array_equal(oabs[0, h], np.abs(v0[h // 8]))


def test_gqa_equal_keys_give_the_mean_of_the_values():
    """All keys equal: every score of a row is the same, so the output is the
    plain mean of the values the row sees (rows at positions 5, 6, 7)."""
    T = 16
    q, k, vt = synth.make_attn(T, 8, 3, 4)
    k = k[:, :1].expand(2, T, 256).contiguous()
    o, _ = oracle.gqa_decode(_attn_bits(q), _attn_bits(k), _attn_bits(vt), 5)
    V = vt.double().numpy()
    for m in range(3):
        n = 5 + m + 1
        for h in range(16):
            np.testing.assert_allclose(o[m, h], V[h // 8, :, :n].mean(axis=1), rtol=1e-12, atol=1e-13)


def test_gqa_matches_torch_sdpa():
    """Against torch's scaled_dot_product_attention in fp64 with the key/value
    heads repeated per query group and an explicit causal mask."""
    T, n_valid, M = 96, 77, 4
    pos0 = n_valid - M
    q, k, vt = synth.make_attn(T, n_valid, M, 5)
    o, oabs = oracle.gqa_decode(_attn_bits(q), _attn_bits(k), _attn_bits(vt), pos0)
    Q = q.double().permute(1, 0, 2)                                   # [Hq, M, D]
    K = k.double()[:, :n_valid].repeat_interleave(8, dim=0)          # [Hq, n, D]
    V = vt.double()[:, :, :n_valid].transpose(1, 2).repeat_interleave(8, dim=0)
    pos = torch.arange(n_valid)[None, :]
    allowed = pos <= (pos0 + torch.arange(M))[:, None]                # [M, n]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=allowed)
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    assert np.all(oabs >= np.abs(o) - 1e-12)


def test_gqa_rows_equal_one_row_calls():
    """Row m of an M-row call is the one-row call at position pos0 + m."""
    q, k, vt = synth.make_attn(64, 50, 3, 6)
    o, _ = oracle.gqa_decode(_attn_bits(q), _attn_bits(k), _attn_bits(vt), 47)
    for m in range(3):
        o1, _ = oracle.gqa_decode(_attn_bits(q[m:m + 1]), _attn_bits(k), _attn_bits(vt), 47 + m)
        assert np.array_equal(o1[0], o[m])


def test_gqa_rejects_rows_past_the_cache():
    q, k, vt = synth.make_attn(16, 16, 2, 7)
    with pytest.raises(ValueError):
        oracle.gqa_decode(_attn_bits(q), _attn_bits(k), _attn_bits(vt), 15)
