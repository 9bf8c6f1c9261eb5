"""GPU parity of the split-K decode attention with grouped query heads
(moe_attn_decode) against the fp64 oracle, through the C ABI.

Source: PureDrive-35B-A3B-MLX model card, "How it works" (one attention
kernel for the one-row decode and the multi-row verify, K/V read once for
all query heads and rows, split points and summation order that depend only
on the row's position) and "Beyond this checkpoint" (16 query heads, 2 KV
heads, head dimension 256).

Tolerance, derived from the kernel's arithmetic: the scores are fp32 sums of
256 exact bf16 products (|error| <= 256 * 2^-24 * sum_d |q_d k_d| / 16 per
score, the tensor core's accumulation rounding); an error e in the scores
moves the softmax-weighted mean by at most 2 e * sum_t w_t |v_t| (oabs); the
weights go to the tensor core as two bf16 halves (relative 2^-16 each) and
the column sums use the same halves, which adds 2^-15 * oabs.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_moe_decode_layer_gb300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda"


def bits(t):
    return synth.bf16_bits(t.cpu()).numpy().view(np.uint16)


def make(T_cap, n_valid, M, seed):
    q, k, vt = synth.make_attn(T_cap, n_valid, M, seed)
    cache = moe.AttnCache(T_cap, device=DEV)
    cache.k.copy_(k)
    cache.vt.copy_(vt)
    return q, k, vt, cache


def bound(q, k, n_valid, oabs):
    """Per (row, head) tolerance of the module docstring."""
    qd = q.double().abs().numpy()                        # [M, 16, 256]
    kd = k.double().abs().numpy()[:, :n_valid]           # [2, n, 256]
    M = qd.shape[0]
    tol = np.zeros_like(oabs)
    for m in range(M):
        for h in range(16):
            smax = (kd[h // 8] @ qd[m, h]).max() / 16.0
            e = 256 * 2.0 ** -24 * smax
            tol[m, h] = (2 * e + 2.0 ** -15) * oabs[m, h] + 1e-6
    return tol


def check(T_cap, n_valid, M, seed):
    q, k, vt, cache = make(T_cap, n_valid, M, seed)
    pos0 = n_valid - M
    o, err = cache.attend(q.to(DEV), pos0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, oabs = oracle.gqa_decode(bits(q), bits(k), bits(vt), pos0)
    got = o.double().cpu().numpy()
    tol = bound(q, k, n_valid, oabs)
    diff = np.abs(got - ref)
    bad = diff > tol
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside; worst {diff.max():.3g} "
                           f"(tol there {tol.flat[diff.argmax()]:.3g})")
    return q, cache, o


@pytest.mark.parametrize("T_cap,n_valid,M", [(64, 1, 1), (256, 200, 1), (1024, 700, 3), (2048, 1537, 8),
                                             (4096, 4096, 4), (640, 129, 2), (40960, 40000, 1),
                                             (65536, 50001, 4)])
def test_attention_matches_oracle(T_cap, n_valid, M):
    """Single key; ragged tiles and chunks (700 = 512 + 188, 1537 = 3 * 512 + 1,
    129 = 128 + 1); the cache full to its end; 1, 2, 3, 4 and 8 rows; more
    chunk CTAs than SMs (79 and 98 chunks per KV head), where 16 and 32
    query columns run two CTAs per SM."""
    check(T_cap, n_valid, M, 11 + M)


@pytest.mark.parametrize("T_cap,n_valid", [(2048, 1800), (45056, 40000)])
def test_attention_rows_equal_one_row_calls(T_cap, n_valid):
    """Row m of an 8-row call is bitwise the one-row call at position pos0 + m
    (at 40000 positions the one-row calls run two CTAs per SM, the 8-row call
    one)."""
    M = 8
    q, cache, o = check(T_cap, n_valid, M, 21)
    pos0 = n_valid - M
    for m in range(M):
        o1, err = cache.attend(q[m:m + 1].to(DEV), pos0 + m)
        assert torch.equal(o1[0], o[m]), f"row {m} differs from its one-row call"


def test_append_then_attend():
    """Rows appended through moe_attn_append give the same result as a cache
    written directly."""
    T_cap, n_valid, M = 1024, 600, 3
    q, k, vt = synth.make_attn(T_cap, n_valid, M, 31)
    direct = moe.AttnCache(T_cap, device=DEV)
    direct.k.copy_(k)
    direct.vt.copy_(vt)
    built = moe.AttnCache(T_cap, device=DEV)
    built.k[:, :n_valid - M].copy_(k[:, :n_valid - M])
    built.vt[:, :, :n_valid - M].copy_(vt[:, :, :n_valid - M])
    k_new = k[:, n_valid - M:n_valid].permute(1, 0, 2).contiguous().to(DEV)        # [M, 2, 256]
    v_new = vt[:, :, n_valid - M:n_valid].permute(2, 0, 1).contiguous().to(DEV)    # [M, 2, 256]
    built.append(k_new, v_new, n_valid - M)
    assert torch.equal(built.k, direct.k) and torch.equal(built.vt, direct.vt)
    o1, _ = direct.attend(q.to(DEV), n_valid - M)
    o2, _ = built.attend(q.to(DEV), n_valid - M)
    assert torch.equal(o1, o2)


def test_attention_argument_errors():
    cache = moe.AttnCache(64, device=DEV)
    q = torch.zeros((1, 16, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(moe.MoeError):
        cache.attend(q, 64)                                  # row past the cache
    with pytest.raises(moe.MoeError):
        cache.attend(torch.zeros((9, 16, 256), dtype=torch.bfloat16, device=DEV), 0)   # M > 8
