"""Algorithmic bytes and flops of one layer call: the numerators of the
roofline figures.

Unique bytes (the quantity the decode step must move at least once): every
distinct selected expert's packed codes and per-group scale/bias words once,
the shared expert, every router row and the shared-expert gate row, the two
RMSNorm weight vectors, and the activations (x in, the residual output and
the normalised output).  A row of K inputs at b bits takes K*b/8 code bytes
plus K/64 four-byte (scale, bias) words; an fp32 row takes 4K bytes.
(flash-moe, "Expert streaming": one 4-bit expert of the 397B model is
6.75 MB, which this count reproduces.)
"""
from __future__ import annotations


def row_bytes(K: int, bits: int) -> int:
    return K * bits // 8 + K // 64 * 4 if bits else 4 * K


def expert_bytes(H: int, I: int, bits: int) -> int:
    """gate [I,H] + up [I,H] + down [H,I]."""
    return 2 * I * row_bytes(H, bits) + H * row_bytes(I, bits)


def unique_bytes(d, U: int, M: int) -> int:
    """d: an object with H, I, E, routed_bits, shared_bits, router_bits,
    has_shared, I_shared (a moe_layer_desc or a synth shape); U distinct
    routed experts over the M rows."""
    shared = expert_bytes(d.H, d.I_shared, d.shared_bits) if d.has_shared else 0
    router = (d.E + (1 if d.has_shared else 0)) * row_bytes(d.H, d.router_bits)
    gammas = 2 * 2 * d.H
    acts = 3 * M * 2 * d.H
    return U * expert_bytes(d.H, d.I, d.routed_bits) + shared + router + gammas + acts


def layer_flops(d, U_rows: int, M: int) -> int:
    """Multiply-adds x2 of one call: U_rows = sum over rows of the experts
    each row chose (M*k), plus the shared expert and the router per row."""
    per_expert_row = 2 * 3 * d.I * d.H
    shared = 2 * 3 * d.I_shared * d.H if d.has_shared else 0
    router = 2 * (d.E + (1 if d.has_shared else 0)) * d.H
    return U_rows * per_expert_row + M * (shared + router)
