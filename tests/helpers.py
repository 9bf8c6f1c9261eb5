"""Shared helpers for the tests: seeded inputs with the routing margin the
parity checks need, oracle views and the element-wise tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

MARGIN = 1e-3          # top-k logit gap every parity row must have (oracle logits)
ATOL, RTOL = 2e-3, 1e-2  # |gpu - ref| <= ATOL + RTOL * |ref| on the bf16 outputs


def to_device(L: dict, dev) -> dict:
    out = {}
    for k, v in L.items():
        if isinstance(v, dict):
            out[k] = {kk: (vv.to(dev) if isinstance(vv, torch.Tensor) else vv) for kk, vv in v.items()}
        elif isinstance(v, torch.Tensor):
            out[k] = v.to(dev)
        else:
            out[k] = v
    return out


def bits_np(x: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(x.detach().cpu()).numpy().view(np.uint16)


def rows_with_margin(shape, lay: oracle.Layer, seed: int, M: int, correlation: float = 0.0,
                     gamma=None, max_attempts: int = 200) -> torch.Tensor:
    """bf16 rows [M, H] whose oracle top-k logit gaps are all >= MARGIN.
    A row that fails is redrawn from its next attempt stream (row 0 as well,
    which changes every correlated row)."""
    attempts = [0] * M
    for _ in range(max_attempts):
        x = synth.make_rows(shape, seed, M, gamma=gamma, correlation=correlation, attempts=attempts)
        r = lay.route(bits_np(x))
        bad = [m for m in range(M) if r["margin"][m] < MARGIN]
        if not bad:
            return x
        for m in bad:
            attempts[m] += 1
    raise RuntimeError("could not draw rows with the routing margin")


def assert_close(got: np.ndarray, ref: np.ndarray, what: str):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    tol = ATOL + RTOL * np.abs(ref)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements outside tolerance; first at "
                             f"{tuple(i)}: got {got[tuple(i)]}, ref {ref[tuple(i)]}, max err {err.max()}")


def bf16_tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def teacher_forced(moe, layers, lays, x, ws, label: str, dev="cuda", min_frac: float = 0.75,
                   normed_last: bool = True):
    """Runs the layers one call at a time from x and compares every layer with
    the oracle on the GPU's own bf16 input of that layer (teacher-forced).
    Rows whose oracle top-k margin is below MARGIN are counted and not
    compared (the GPU may then pick the other expert of a near tie); every
    other row must have bit-exact expert ids and outputs within the
    tolerance.  Fails if fewer than `min_frac` of all (layer, row) pairs
    were compared.  Returns (outputs of each layer, compared, skipped)."""
    M = x.shape[0]
    h = x.to(dev)
    outs = []
    compared = skipped = 0
    for i, (lyr, lay) in enumerate(zip(layers, lays)):
        last = normed_last and i == len(layers) - 1
        ref = lay.forward(bits_np(h), normed=last)
        idx, _ = moe.router_topk(lyr, h, ws)
        if last:
            nxt, on = moe.decode_layer(lyr, h, ws, normed=True)
        else:
            nxt = moe.decode_layer(lyr, h, ws)
        assert ws.status() == 0
        idx = idx.cpu().numpy()
        got = bf16_tensor_to_f64(nxt)
        for m in range(M):
            if ref["margin"][m] < MARGIN:
                skipped += 1
                continue
            compared += 1
            assert np.array_equal(idx[m], ref["idx"][m]), f"{label} layer {i} row {m}: expert ids differ"
            assert_close(got[m], ref["o"][m], f"{label} layer {i} row {m} out")
            if last:
                assert_close(bf16_tensor_to_f64(on)[m], ref["on"][m], f"{label} layer {i} row {m} out_normed")
        outs.append(nxt)
        h = nxt
    total = compared + skipped
    print(f"{label}: {compared} of {total} (layer, row) pairs compared, {skipped} below the routing margin")
    assert compared >= min_frac * total, f"{label}: only {compared} of {total} pairs above the routing margin"
    return outs, compared, skipped
