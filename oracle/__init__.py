"""Python access to the fp64 CPU oracle (oracle/moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg.  The CUDA library never imports, links or calls
anything here.

The C source is compiled with gcc into oracle/liboracle.so on first use (or by
`build()`), with -ffp-contract=off so that the fp32 quantiser decisions and the
fp64 sums round the same way on every host.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (host code only; no CUDA).  With OpenMP
    when the compiler has it (the all-cores timing run); without, the oracle
    runs on one thread."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-ffp-contract=off",
                "-fno-fast-math", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        try:
            subprocess.check_call(base[:1] + ["-fopenmp"] + base[1:], stderr=subprocess.DEVNULL)
        except subprocess.CalledProcessError:
            subprocess.check_call(base)
        os.replace(tmp, _LIB)
    return _LIB


class OqMatrix(C.Structure):
    _fields_ = [("bits", C.c_int), ("rows", C.c_int), ("cols", C.c_int),
                ("codes", C.c_void_p), ("scales", C.c_void_p), ("biases", C.c_void_p),
                ("w", C.c_void_p)]


class OqLayer(C.Structure):
    _fields_ = [("H", C.c_int), ("I", C.c_int), ("E", C.c_int), ("k", C.c_int),
                ("has_shared", C.c_int), ("I_shared", C.c_int), ("eps", C.c_double),
                ("router", OqMatrix), ("sgate", OqMatrix),
                ("gate", C.POINTER(OqMatrix)), ("up", C.POINTER(OqMatrix)), ("down", C.POINTER(OqMatrix)),
                ("shared_gate", OqMatrix), ("shared_up", OqMatrix), ("shared_down", OqMatrix),
                ("gamma", C.c_void_p), ("gamma_next", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _lib.oracle_bf16_to_double.restype = C.c_double
        _lib.oracle_bf16_to_double.argtypes = [C.c_uint16]
        _lib.oracle_bf16_from_double.restype = C.c_uint16
        _lib.oracle_bf16_from_double.argtypes = [C.c_double]
        _lib.oracle_weight.restype = C.c_double
        _lib.oracle_weight.argtypes = [C.POINTER(OqMatrix), C.c_int, C.c_int]
        _lib.oracle_layer.restype = C.c_int
        _lib.oracle_set_threads.restype = None
        _lib.oracle_set_threads.argtypes = [C.c_int]
        _lib.oracle_max_threads.restype = C.c_int
        _lib.oracle_gqa_decode.restype = C.c_int
        for name in ("oracle_pack_bits", "oracle_unpack_bits", "oracle_quantize_group",
                     "oracle_quantize_matrix", "oracle_rmsnorm", "oracle_topk",
                     "oracle_expert_ffn", "oracle_route", "oracle_qkv"):
            getattr(_lib, name).restype = None
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def _np(t, dtype=None):
    """torch tensor (any device) or array -> contiguous host numpy array."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            if t.dtype == torch.bfloat16:
                t = t.contiguous().view(torch.int16)
            a = t.detach().to("cpu").contiguous().numpy()
            if a.dtype == np.int16:
                a = a.view(np.uint16)
            return np.ascontiguousarray(a if dtype is None else a.astype(dtype))
    except ImportError:
        pass
    a = np.asarray(t)
    return np.ascontiguousarray(a if dtype is None else a.astype(dtype))


def set_threads(n: int) -> None:
    """Threads of the oracle's mat-vecs (1 = the parity reference; results
    are the same bits for any count)."""
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    """Host cores the oracle can use (1 when built without OpenMP)."""
    return int(lib().oracle_max_threads())


# ------------------------------------------------------------------ scalar ops

def bf16_from_double(v: float) -> int:
    return int(lib().oracle_bf16_from_double(float(v)))


def bf16_to_double(b: int) -> float:
    return float(lib().oracle_bf16_to_double(int(b) & 0xFFFF))


def bf16_round_array(a: np.ndarray) -> np.ndarray:
    """Elementwise double -> bf16 pattern (uint16)."""
    f = lib().oracle_bf16_from_double
    flat = np.asarray(a, dtype=np.float64).ravel()
    return np.array([f(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(a))


def bf16_patterns_to_double(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pack_bits(codes: np.ndarray, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    out = np.zeros((codes.size * bits + 7) // 8, dtype=np.uint8)
    lib().oracle_pack_bits(_p(codes), C.c_int(codes.size), C.c_int(bits), _p(out))
    return out


def unpack_bits(packed: np.ndarray, n: int, bits: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros(n, dtype=np.uint8)
    lib().oracle_unpack_bits(_p(packed), C.c_int(n), C.c_int(bits), _p(out))
    return out


def quantize_matrix(w, bits: int):
    """fp32 [rows, cols] -> (codes u8, scales bf16-patterns, biases bf16-patterns)."""
    w = _np(w, np.float32)
    rows, cols = w.shape
    codes = np.zeros((rows, cols), dtype=np.uint8)
    s = np.zeros((rows, cols // 64), dtype=np.uint16)
    b = np.zeros((rows, cols // 64), dtype=np.uint16)
    lib().oracle_quantize_matrix(C.c_int(bits), _p(w), C.c_int(rows), C.c_int(cols), _p(codes), _p(s), _p(b))
    return codes, s, b


def rmsnorm(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float) -> np.ndarray:
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    gamma_bits = np.ascontiguousarray(gamma_bits, dtype=np.uint16)
    H = x_bits.size
    hn = np.zeros(H, dtype=np.float64)
    lib().oracle_rmsnorm(_p(x_bits), _p(gamma_bits), C.c_int(H), C.c_double(eps), _p(hn))
    return hn


def topk(logits: np.ndarray, k: int):
    """-> (idx int32 [k], w float64 [k], probs float64 [E], margin)."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    E = logits.size
    idx = np.zeros(k, dtype=np.int32)
    w = np.zeros(k, dtype=np.float64)
    probs = np.zeros(E, dtype=np.float64)
    margin = C.c_double(0.0)
    lib().oracle_topk(_p(logits), C.c_int(E), C.c_int(k), _p(idx), _p(w), _p(probs), C.byref(margin))
    return idx, w, probs, margin.value


# ------------------------------------------------------------------- matrices

class Matrix:
    """Host copy of one matrix in canonical form, kept alive for ctypes."""

    def __init__(self, bits: int, codes=None, scales=None, biases=None, w=None):
        self.bits = bits
        if bits == 0:
            self.w = _np(w, np.float32)
            self.rows, self.cols = self.w.shape
            self.codes = self.scales = self.biases = None
        else:
            self.codes = _np(codes, np.uint8)
            self.scales = _np(scales, np.uint16)
            self.biases = _np(biases, np.uint16)
            self.rows, self.cols = self.codes.shape
            self.w = None

    @classmethod
    def from_canonical(cls, d):
        return cls(d["bits"], d["codes"], d["scales"], d["biases"])

    def struct(self) -> OqMatrix:
        m = OqMatrix()
        m.bits, m.rows, m.cols = self.bits, self.rows, self.cols
        if self.bits == 0:
            m.w = _p(self.w).value
        else:
            m.codes, m.scales, m.biases = _p(self.codes).value, _p(self.scales).value, _p(self.biases).value
        return m

    def weight(self, r: int, c: int) -> float:
        s = self.struct()
        return float(lib().oracle_weight(C.byref(s), r, c))

    def dense(self) -> np.ndarray:
        """Fully dequantised fp64 matrix, computed here with numpy (independent of the C code)."""
        if self.bits == 0:
            return self.w.astype(np.float64)
        s = np.repeat(bf16_patterns_to_double(self.scales), 64, axis=1)
        b = np.repeat(bf16_patterns_to_double(self.biases), 64, axis=1)
        return self.codes.astype(np.float64) * s + b


def _expert_slice(d, e):
    return {"bits": d["bits"], "codes": d["codes"][e], "scales": d["scales"][e], "biases": d["biases"][e]}


class Layer:
    """Oracle view of one layer built from synth.make_layer's canonical dict.

    The router (and shared-gate vector) are quantised here by the oracle's own
    quantiser when the shape asks for an 8-bit router.  Routed experts are
    copied to the host lazily: only the experts the routing selects are
    needed, which keeps the full-size shapes cheap."""

    def __init__(self, L: dict):
        sh = L["shape"]
        self.shape = sh
        self.L = L
        self.H, self.I, self.E, self.k = sh.H, sh.I, sh.E, sh.k
        self.eps = sh.eps
        if sh.router_bits == 0:
            self.router = Matrix(0, w=L["router_w"])
        else:
            self.router = Matrix(sh.router_bits, *quantize_matrix(L["router_w"], sh.router_bits))
        if sh.has_shared:
            sg = _np(L["sgate_w"], np.float32).reshape(1, -1)
            self.sgate = Matrix(sh.router_bits, *quantize_matrix(sg, sh.router_bits)) if sh.router_bits else Matrix(0, w=sg)
            self.shared = [Matrix.from_canonical(L["shared_gate"]), Matrix.from_canonical(L["shared_up"]),
                           Matrix.from_canonical(L["shared_down"])]
        else:
            self.sgate = None
            self.shared = None
        self.gamma = _np(L["gamma"], np.uint16)
        self.gamma_next = _np(L["gamma_next"], np.uint16)
        self.experts = {}

    def expert(self, e: int):
        if e not in self.experts:
            self.experts[e] = [Matrix.from_canonical(_expert_slice(self.L[n], e)) for n in ("gate", "up", "down")]
        return self.experts[e]

    def _struct(self, need=()):
        for e in need:
            self.expert(e)
        s = OqLayer()
        s.H, s.I, s.E, s.k = self.H, self.I, self.E, self.k
        s.has_shared = 1 if self.shared else 0
        s.I_shared = self.shape.I_shared if self.shared else 0
        s.eps = self.eps
        s.router = self.router.struct()
        if self.sgate is not None:
            s.sgate = self.sgate.struct()
        arrs = []
        for t in range(3):
            arr = (OqMatrix * self.E)()
            for e, mats in self.experts.items():
                arr[e] = mats[t].struct()
            arrs.append(arr)
        self._arrs = arrs
        s.gate, s.up, s.down = (C.cast(a, C.POINTER(OqMatrix)) for a in arrs)
        if self.shared:
            s.shared_gate, s.shared_up, s.shared_down = (m.struct() for m in self.shared)
        s.gamma = _p(self.gamma).value
        s.gamma_next = _p(self.gamma_next).value
        self._s = s
        return s

    def route(self, x_bits: np.ndarray):
        """x bf16 patterns [M, H] -> dict(logits, idx, w, sigma, margin)."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1, self.H)
        M = x_bits.shape[0]
        s = self._struct()
        logits = np.zeros((M, self.E), np.float64)
        idx = np.zeros((M, self.k), np.int32)
        w = np.zeros((M, self.k), np.float64)
        sigma = np.zeros(M, np.float64)
        margin = np.zeros(M, np.float64)
        lib().oracle_route(C.byref(s), _p(x_bits), C.c_int(M), _p(logits), _p(idx), _p(w), _p(sigma), _p(margin))
        return {"logits": logits, "idx": idx, "w": w, "sigma": sigma, "margin": margin}

    def forward(self, x_bits: np.ndarray, normed: bool = True):
        """Full layer.  Returns dict(o, out, on, out_n, logits, idx, w, sigma, margin)."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1, self.H)
        M = x_bits.shape[0]
        r = self.route(x_bits)
        s = self._struct(need=sorted(set(int(e) for e in r["idx"].ravel())))
        H = self.H
        o = np.zeros((M, H), np.float64)
        out = np.zeros((M, H), np.uint16)
        on = np.zeros((M, H), np.float64) if normed else None
        out_n = np.zeros((M, H), np.uint16) if normed else None
        logits = np.zeros((M, self.E), np.float64)
        idx = np.zeros((M, self.k), np.int32)
        w = np.zeros((M, self.k), np.float64)
        sigma = np.zeros(M, np.float64)
        margin = np.zeros(M, np.float64)
        rc = lib().oracle_layer(C.byref(s), _p(x_bits), C.c_int(M), _p(o), _p(out),
                                _p(on) if normed else None, _p(out_n) if normed else None,
                                _p(logits), _p(idx), _p(w), _p(sigma), _p(margin))
        if rc != 0:
            raise RuntimeError(f"oracle_layer: expert {-rc - 1} missing")
        return {"o": o, "out": out, "on": on, "out_n": out_n, "logits": logits, "idx": idx,
                "w": w, "sigma": sigma, "margin": margin}


def qkv(mats, x_bits: np.ndarray) -> np.ndarray:
    """Fused projection of x bf16 patterns [M, H] by the matrices in `mats`
    (Matrix objects of the same width, e.g. Q, K, V) stacked row-wise:
    returns fp64 [M, sum of their rows]."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, H = x_bits.shape
    parts = []
    for m_ in mats:
        assert m_.cols == H
    if all(m_.bits == mats[0].bits for m_ in mats) and mats[0].bits != 0:
        st = Matrix(mats[0].bits, np.concatenate([m_.codes for m_ in mats]),
                    np.concatenate([m_.scales for m_ in mats]), np.concatenate([m_.biases for m_ in mats]))
    else:
        raise ValueError("qkv: the matrices must share one code width")
    y = np.zeros((M, st.rows), np.float64)
    s = st.struct()
    lib().oracle_qkv(C.byref(s), _p(x_bits), C.c_int(M), _p(y))
    return y


def gqa_decode(q_bits: np.ndarray, k_bits: np.ndarray, vt_bits: np.ndarray, pos0: int):
    """Decode attention with grouped query heads (oracle_gqa_decode).
    q_bits [M, Hq, D], k_bits [Hkv, T_cap, D], vt_bits [Hkv, D, T_cap]: bf16
    patterns (uint16).  Row m is at position pos0 + m and attends to keys
    0 .. pos0 + m.  Returns (o, oabs), fp64 [M, Hq, D]."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    vt_bits = np.ascontiguousarray(vt_bits, dtype=np.uint16)
    M, Hq, D = q_bits.shape
    Hkv, T_cap, D2 = k_bits.shape
    if D2 != D or vt_bits.shape != (Hkv, D, T_cap):
        raise ValueError("gqa_decode: inconsistent shapes")
    o = np.zeros((M, Hq, D), np.float64)
    oabs = np.zeros((M, Hq, D), np.float64)
    rc = lib().oracle_gqa_decode(_p(q_bits), _p(k_bits), _p(vt_bits), C.c_int(T_cap), C.c_int(pos0), C.c_int(M),
                                 C.c_int(Hq), C.c_int(Hkv), C.c_int(D), _p(o), _p(oabs))
    if rc != 0:
        raise ValueError("gqa_decode: rejected arguments")
    return o, oabs


def stack(layers, x_bits: np.ndarray, normed_last: bool = True):
    """L chained layers: x_{l+1} = out_l (bf16).  Returns the per-layer results."""
    res = []
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    for i, lay in enumerate(layers):
        r = lay.forward(x, normed=normed_last and i == len(layers) - 1)
        res.append(r)
        x = r["out"]
    return res
