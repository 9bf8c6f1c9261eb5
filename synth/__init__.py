"""Seeded synthetic inputs for the quantized MoE decode layer.

This module only draws random numbers in the shapes and distributions of the
workloads; it holds none of the layer's arithmetic (no normalisation, no
dequantisation, no routing).  Both the CUDA path (through the tests and the
benchmark) and the CPU oracle consume what it returns.

Workloads (sizes follow the PureDrive-35B-A3B-MLX model card, "Summary": 256
experts, top-8 plus a shared expert, 6-bit experts and 8-bit shared weights;
and flash-moe (hada.io topic 27758), "モデルアーキテクチャ": 512 experts,
hidden 4096, ~6.75 MB per 4-bit expert):

  tiny   H=256  I=128  E=16  k=2   no shared expert, 4-bit experts, fp32 router
  a35b   H=2048 I=512  E=256 k=8   shared expert I=512, 6-bit experts, 8-bit router/shared
  b397   H=4096 I=1024 E=512 k=10  shared expert I=1024, 4-bit experts, 8-bit router/shared

Value recipe (one reading of the workload description):
  * expert codes uniform in [0, 2^b - 1];
  * per-group scale |N(0, 0.02)| * 15 / (2^b - 1), both rounded to bf16 (the
    15/(2^b-1) factor keeps the dequantised weight distribution of the 4-bit
    case at every width);
  * per-group bias N(0, 0.01) taken relative to the centre of the code grid:
    b = N(0, 0.01) - s (2^b - 1) / 2, so that the dequantised weights q s + b
    have mean zero as in an affine-quantised checkpoint, where the bias is the
    group's minimum (grid="centred", the default).  grid="literal" draws
    b = N(0, 0.01) as written; then every matrix carries a positive mean of
    about 7.5 E[s] = 0.12, and a stack of layers amplifies that one direction
    (the residual stream grows from rms 1 to ~1e7 within four 35B-A3B layers
    and every token row routes to the same experts);
  * router and shared-gate vector fp32 N(0, 0.05) (quantised to 8 bits by the
    library's packer where the workload asks for an 8-bit router);
  * x bf16 N(0, 1); RMSNorm weights 1 + N(0, 0.1) in bf16;
  * Zipf(1.1) popularity (a35b): router row e gets c_e * u added, with u a
    fixed unit direction and c_e = tau * ln p_e, p_e proportional to
    rank(e)^-1.1 under a fixed random permutation; every x row carries a
    component of size ZIPF_ALPHA along v = u / gamma (normalised so that
    sum_j gamma_j u_j v_j = 1), which makes u . (gamma * x) close to ZIPF_ALPHA.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    H: int
    I: int
    E: int
    k: int
    routed_bits: int
    shared_bits: int
    router_bits: int      # 0 = fp32 router
    has_shared: bool
    I_shared: int
    zipf: bool
    eps: float = 1e-6


TINY = LayerShape("tiny", 256, 128, 16, 2, 4, 8, 0, False, 0, False)
A35B = LayerShape("a35b", 2048, 512, 256, 8, 6, 8, 8, True, 512, True)
B397 = LayerShape("b397", 4096, 1024, 512, 10, 4, 8, 8, True, 1024, False)
SHAPES = {s.name: s for s in (TINY, A35B, B397)}

ZIPF_EXPONENT = 1.1
ZIPF_ALPHA = 3.0
# Gumbel-equivalent scale of the router-logit noise at a35b
# (0.05 * sqrt(2048) * sqrt(6) / pi), divided by ZIPF_ALPHA.
ZIPF_TAU = 0.05 * math.sqrt(2048.0) * math.sqrt(6.0) / math.pi / ZIPF_ALPHA


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def _codes(g, shape, bits, device):
    return torch.randint(0, 1 << bits, shape, generator=g, device=device, dtype=torch.uint8)


def _scales(g, shape, bits, device):
    s = torch.randn(shape, generator=g, device=device, dtype=torch.float32).abs_()
    s.mul_(0.02 * 15.0 / float((1 << bits) - 1))
    return s.to(torch.bfloat16)


def _biases(g, shape, device, scales=None, bits=0):
    b = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 0.01
    if scales is not None:
        b -= scales.float() * (((1 << bits) - 1) / 2.0)
    return b.to(torch.bfloat16)


GRIDS = ("centred", "literal")


def quant_matrix(g, rows_shape, K, bits, device, grid="centred"):
    """Canonical quantised matrix: codes u8 [..., K], scales/biases bf16 [..., K/64]."""
    assert grid in GRIDS
    codes = _codes(g, tuple(rows_shape) + (K,), bits, device)
    scales = _scales(g, tuple(rows_shape) + (K // 64,), bits, device)
    biases = _biases(g, tuple(rows_shape) + (K // 64,), device,
                     scales if grid == "centred" else None, bits)
    return {"codes": codes, "scales": scales, "biases": biases, "bits": bits}


def zipf_direction(shape: LayerShape, seed: int):
    """Fixed unit direction u [H] and per-expert coefficients c [E] (fp64, CPU)."""
    g = _gen(seed * 7919 + 17, "cpu")
    u = torch.randn(shape.H, generator=g, dtype=torch.float64)
    u /= u.norm()
    perm = torch.randperm(shape.E, generator=g)
    rank = torch.empty(shape.E, dtype=torch.float64)
    rank[perm] = torch.arange(1, shape.E + 1, dtype=torch.float64)
    p = rank.pow(-ZIPF_EXPONENT)
    p /= p.sum()
    c = ZIPF_TAU * torch.log(p)
    c -= c.mean()
    return u, c


def make_layer(shape: LayerShape, seed: int, device="cpu", grid="centred") -> dict:
    """Canonical weights of one layer (torch tensors on `device`); `grid`
    chooses the bias distribution (see the module docstring).

    Keys: gate/up [E, I, H], down [E, H, I] (each a dict of codes/scales/biases),
    shared_gate/shared_up [I_s, H], shared_down [H, I_s] (when present),
    router_w fp32 [E, H], sgate_w fp32 [H] (when shared), gamma bf16 [H],
    gamma_next bf16 [H].
    """
    g = _gen(seed, device)
    H, I, E = shape.H, shape.I, shape.E
    L = {"shape": shape, "seed": seed, "grid": grid}
    L["gate"] = quant_matrix(g, (E, I), H, shape.routed_bits, device, grid)
    L["up"] = quant_matrix(g, (E, I), H, shape.routed_bits, device, grid)
    L["down"] = quant_matrix(g, (E, H), I, shape.routed_bits, device, grid)
    if shape.has_shared:
        Is = shape.I_shared
        L["shared_gate"] = quant_matrix(g, (Is,), H, shape.shared_bits, device, grid)
        L["shared_up"] = quant_matrix(g, (Is,), H, shape.shared_bits, device, grid)
        L["shared_down"] = quant_matrix(g, (H,), Is, shape.shared_bits, device, grid)
    router = torch.randn((E, H), generator=g, device=device, dtype=torch.float32) * 0.05
    if shape.zipf:
        u, c = zipf_direction(shape, 0)
        router += (c[:, None] * u[None, :]).to(device=device, dtype=torch.float32)
    L["router_w"] = router
    if shape.has_shared:
        L["sgate_w"] = torch.randn((H,), generator=g, device=device, dtype=torch.float32) * 0.05
    L["gamma"] = (1.0 + 0.1 * torch.randn((H,), generator=g, device=device, dtype=torch.float32)).to(torch.bfloat16)
    L["gamma_next"] = (1.0 + 0.1 * torch.randn((H,), generator=g, device=device, dtype=torch.float32)).to(torch.bfloat16)
    return L


def make_rows(shape: LayerShape, seed: int, M: int, gamma=None, device="cpu",
              correlation: float = 0.0, attempts=None) -> torch.Tensor:
    """x rows, bf16 [M, H].

    Row r draws its noise n_r from its own stream (seed, r, attempts[r]) so that
    a row can be redrawn alone.  With correlation a > 0, row r > 0 is
    a * n_0 + sqrt(1 - a^2) * n_r (a token plus correlated draft rows).  The
    Zipf component (shapes with zipf=True) is added to every row afterwards."""
    attempts = [0] * M if attempts is None else list(attempts)
    noise = [draw_noise(shape, seed, r, attempts[r], device=device) for r in range(M)]
    x = torch.stack(noise)
    if correlation > 0.0 and M > 1:
        x[1:] = correlation * x[0][None, :] + math.sqrt(1.0 - correlation ** 2) * x[1:]
    if shape.zipf:
        x += zipf_component(shape, gamma).to(device=device, dtype=torch.float32)[None, :]
    return x.to(torch.bfloat16)


def draw_noise(shape: LayerShape, seed: int, row: int, attempt: int, device="cpu") -> torch.Tensor:
    """N(0, 1) fp32 [H] for (seed, row, attempt)."""
    g = _gen((seed * 1_000_003 + row) * 131 + attempt, device)
    return torch.randn((shape.H,), generator=g, device=device, dtype=torch.float32)


def zipf_component(shape: LayerShape, gamma=None) -> torch.Tensor:
    """ZIPF_ALPHA * v with v = u / gamma scaled so that sum_j gamma_j u_j v_j = 1 (fp64, CPU)."""
    u, _ = zipf_direction(shape, 0)
    gam = torch.ones(shape.H, dtype=torch.float64) if gamma is None else gamma.detach().to("cpu", torch.float64)
    v = u / gam
    v /= (gam * u * v).sum()
    return ZIPF_ALPHA * v


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """View a bf16 tensor as its raw 16-bit patterns (int16)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16)


# ---------------------------------------------------------- decode attention
#
# The attention shape of the 35B-A3B model (16 query heads, 2 key/value
# heads, head dimension 256) and its inputs: query rows and a bf16 cache of
# keys [Hkv, T_cap, D] and values stored transposed [Hkv, D, T_cap], all
# N(0, 1) in bf16, positions at or past the last valid one zero.

ATTN_HQ, ATTN_HKV, ATTN_D = 16, 2, 256


def make_attn(T_cap: int, n_valid: int, M: int, seed: int, device="cpu"):
    """(q [M, 16, 256], k [2, T_cap, 256], vt [2, 256, T_cap]) bf16 with keys and
    values at positions 0 .. n_valid - 1 drawn and the rest zero."""
    g = _gen(seed * 7919 + 17, device)
    q = torch.randn((M, ATTN_HQ, ATTN_D), generator=g, device=device, dtype=torch.float32)
    k = torch.zeros((ATTN_HKV, T_cap, ATTN_D), device=device, dtype=torch.float32)
    vt = torch.zeros((ATTN_HKV, ATTN_D, T_cap), device=device, dtype=torch.float32)
    k[:, :n_valid] = torch.randn((ATTN_HKV, n_valid, ATTN_D), generator=g, device=device, dtype=torch.float32)
    vt[:, :, :n_valid] = torch.randn((ATTN_HKV, ATTN_D, n_valid), generator=g, device=device, dtype=torch.float32)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), vt.to(torch.bfloat16)
