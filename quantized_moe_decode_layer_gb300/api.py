"""Thin Python binding over the C ABI: torch provides device memory and
streams, every step of the layer runs in libmoe.so's kernels."""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib
from ._lib import LayerDesc, QkvDesc, SrcLayer, SrcMatrix, check, lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not (t.is_cuda and t.is_contiguous()):
        raise ValueError("device tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _need(t, name: str, dtype, shape) -> None:
    """Refuse, before any call, a tensor the library would read or write out
    of its bounds: it must be a contiguous CUDA tensor of `dtype` and `shape`
    (None in `shape` matches any extent)."""
    ok = (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous() and t.dtype == dtype
          and t.dim() == len(shape) and all(n is None or t.shape[i] == n for i, n in enumerate(shape)))
    if not ok:
        want = ", ".join("*" if n is None else str(n) for n in shape)
        got = (f"{tuple(t.shape)} {t.dtype} on {t.device}, contiguous={t.is_contiguous()}"
               if isinstance(t, torch.Tensor) else type(t).__name__)
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor of shape [{want}]; got {got}")


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def make_desc(H, I, E, k, routed_bits, shared_bits=8, router_bits=8, has_shared=True, I_shared=0,
              eps=1e-6) -> LayerDesc:
    return LayerDesc(H, I, E, k, routed_bits, shared_bits, router_bits, 1 if has_shared else 0,
                     I_shared if has_shared else 0, eps)


def desc_from_shape(shape) -> LayerDesc:
    """moe_layer_desc of a synth.LayerShape-like object."""
    return make_desc(shape.H, shape.I, shape.E, shape.k, shape.routed_bits, shape.shared_bits,
                     shape.router_bits, shape.has_shared, shape.I_shared, shape.eps)


def pack_size(desc: LayerDesc) -> int:
    n = C.c_size_t()
    check("moe_pack_size", lib().moe_pack_size(C.byref(desc), C.byref(n)))
    return n.value


def workspace_size(desc: LayerDesc, max_M: int) -> int:
    n = C.c_size_t()
    check("moe_workspace_size", lib().moe_workspace_size(C.byref(desc), max_M, C.byref(n)))
    return n.value


def _bits16(t):
    if t is None:
        return None
    return t.contiguous().view(torch.int16) if t.dtype == torch.bfloat16 else t.contiguous()


def _src_matrix(d) -> tuple[SrcMatrix, list]:
    """d: dict with codes/scales/biases (canonical) or 'w' (fp32), or a tensor (fp32)."""
    keep = []
    if d is None:
        return SrcMatrix(), keep
    if isinstance(d, torch.Tensor):
        d = {"w": d}
    m = SrcMatrix()
    if d.get("codes") is not None:
        c, s, b = d["codes"].contiguous(), _bits16(d["scales"]), _bits16(d["biases"])
        keep += [c, s, b]
        m.codes_dev, m.scales_dev, m.biases_dev = _ptr(c), _ptr(s), _ptr(b)
    if d.get("w") is not None:
        w = d["w"].contiguous().float()
        keep.append(w)
        m.w_dev = _ptr(w)
    return m, keep


class Layer:
    """One packed layer: owns the device blob (a torch uint8 tensor) and the
    C handle that borrows it."""

    def __init__(self, desc: LayerDesc, src: dict, device="cuda", stream=None):
        self.desc = desc
        self.nbytes = pack_size(desc)
        self.blob = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        keep = []
        sl = SrcLayer()

        def flat(d, rows):
            if d is None or isinstance(d, torch.Tensor):
                return d
            return {k: (v.reshape(rows, -1) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}

        E, I, H = desc.E, desc.I, desc.H
        for name, d in (("gate", flat(src["gate"], E * I)), ("up", flat(src["up"], E * I)),
                        ("down", flat(src["down"], E * H)), ("router", src["router"])):
            m, k = _src_matrix(d)
            keep += k
            setattr(sl, name, m)
        if desc.has_shared:
            for name in ("shared_gate", "shared_up", "shared_down", "sgate"):
                m, k = _src_matrix(src[name])
                keep += k
                setattr(sl, name, m)
        g = _bits16(src["gamma"])
        keep.append(g)
        sl.gamma_dev = _ptr(g)
        gn = _bits16(src.get("gamma_next"))
        if gn is not None:
            keep.append(gn)
            sl.gamma_next_dev = _ptr(gn)
        h = C.c_void_p()
        check("moe_pack_weights", lib().moe_pack_weights(C.byref(desc), C.byref(sl), _ptr(self.blob),
                                                         self.nbytes, C.byref(h), _stream(stream)))
        self.handle = h
        # the sources must outlive the enqueued pack kernels
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
        del keep

    def export(self, tensor_id: int, expert: int = 0, stream=None):
        """Canonical (codes, scales bf16, biases bf16) of one packed matrix."""
        d = self.desc
        rows, cols = {
            _lib.T_ROUTER: (d.E, d.H), _lib.T_SGATE: (1, d.H), _lib.T_GATE: (d.I, d.H), _lib.T_UP: (d.I, d.H),
            _lib.T_DOWN: (d.H, d.I), _lib.T_SHARED_GATE: (d.I_shared, d.H), _lib.T_SHARED_UP: (d.I_shared, d.H),
            _lib.T_SHARED_DOWN: (d.H, d.I_shared)}[tensor_id]
        dev = self.blob.device
        codes = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        s = torch.empty((rows, cols // 64), dtype=torch.int16, device=dev)
        b = torch.empty((rows, cols // 64), dtype=torch.int16, device=dev)
        check("moe_export_canonical", lib().moe_export_canonical(self.handle, tensor_id, expert, _ptr(codes),
                                                                 _ptr(s), _ptr(b), _stream(stream)))
        return codes, s.view(torch.bfloat16), b.view(torch.bfloat16)

    def __del__(self):
        try:
            if getattr(self, "handle", None):
                lib().moe_layer_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


class Workspace:
    """Scratch for the decode calls (allocated by torch, zeroed control block)."""

    def __init__(self, desc: LayerDesc, max_M: int, device="cuda", stream=None):
        self.nbytes = workspace_size(desc, max_M)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        if self.buf.data_ptr() % 256 != 0:
            raise RuntimeError("workspace allocation is not 256-byte aligned")
        self.max_M = max_M
        self.init(stream)

    def init(self, stream=None):
        check("moe_workspace_init", lib().moe_workspace_init(_ptr(self.buf), self.nbytes, _stream(stream)))

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def status(self, stream=None) -> int:
        """Synchronise and return the device status (0 = MOE_OK)."""
        return int(lib().moe_stream_status(self.ptr, self.nbytes, _stream(stream)))


def router_topk(layer: Layer, x: torch.Tensor, ws: Workspace, stream=None):
    _need(x, "x", torch.bfloat16, (None, layer.desc.H))
    M = x.shape[0]
    idx = torch.empty((M, layer.desc.k), dtype=torch.int32, device=x.device)
    w = torch.empty((M, layer.desc.k), dtype=torch.float32, device=x.device)
    check("moe_router_topk", lib().moe_router_topk(layer.handle, _ptr(_bits16(x)), M, _ptr(idx), _ptr(w),
                                                   ws.ptr, ws.nbytes, _stream(stream)))
    return idx, w


def decode_layer(layer: Layer, x: torch.Tensor, ws: Workspace, out=None, normed: bool = False, stream=None):
    """out (and out_normed when normed) bf16 [M, H]."""
    _need(x, "x", torch.bfloat16, (None, layer.desc.H))
    M = x.shape[0]
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.bfloat16, (M, layer.desc.H))
    on = torch.empty_like(x) if normed else None
    check("moe_decode_layer", lib().moe_decode_layer(layer.handle, _ptr(_bits16(x)), M, _ptr(_bits16(out)),
                                                     _ptr(_bits16(on)) if on is not None else None,
                                                     ws.ptr, ws.nbytes, _stream(stream)))
    return (out, on) if normed else out


def decode_layer_noalloc(layer: Layer, x: torch.Tensor, out=None, normed: bool = False, stream=None):
    """moe_decode_layer_noalloc: decode_layer with the library's fixed
    scratch instead of a workspace (no device allocation at the call; calls
    must not overlap on the GPU).  Rows whose workspace would exceed the
    scratch raise MoeError (MOE_ERR_BUFFER_TOO_SMALL)."""
    _need(x, "x", torch.bfloat16, (None, layer.desc.H))
    M = x.shape[0]
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.bfloat16, (M, layer.desc.H))
    on = torch.empty_like(x) if normed else None
    check("moe_decode_layer_noalloc",
          lib().moe_decode_layer_noalloc(layer.handle, _ptr(_bits16(x)), M, _ptr(_bits16(out)),
                                         _ptr(_bits16(on)) if on is not None else None, _stream(stream)))
    return (out, on) if normed else out


def noalloc_status(stream=None) -> int:
    """moe_noalloc_status: synchronise and return the device status of the
    latest decode_layer_noalloc call (0 = MOE_OK, 5 = a device wait gave up)."""
    return int(lib().moe_noalloc_status(_stream(stream)))


def selftest_host() -> int:
    """moe_selftest_host: violations found by the library's host-side checks
    (code tables, launch plans, workspace layouts); 0 when consistent."""
    return int(lib().moe_selftest_host())


def set_grouped(min_rows: int) -> None:
    """Grouped mode (tensor-core expert products) for calls of at least
    min_rows rows above one launch's rows (default 1); 0 turns it off
    (moe_set_grouped)."""
    check("moe_set_grouped", lib().moe_set_grouped(int(min_rows)))


def gate_up_tc(layer: Layer, hn: torch.Tensor, experts: torch.Tensor, masks: torch.Tensor, act=None,
               err=None, stream=None):
    """Grouped gate/up + SwiGLU on the tensor cores (moe_gate_up_tc).

    hn fp32 [M, H] (normalised rows), experts int32 [U], masks int32 [U] (bit m
    = row m) on the device.  Returns (act fp32 [U, M, I], err int32 [1]);
    entries of rows outside a mask are left as they were in `act` (zeros when
    it is allocated here)."""
    _need(hn, "hn", torch.float32, (None, layer.desc.H))
    _need(experts, "experts", torch.int32, (None,))
    M, U, I = hn.shape[0], experts.shape[0], layer.desc.I
    _need(masks, "masks", torch.int32, (U,))
    if act is None:
        act = torch.zeros((U, M, I), dtype=torch.float32, device=hn.device)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=hn.device)
    _need(act, "act", torch.float32, (U, M, I))
    _need(err, "err", torch.int32, (1,))
    check("moe_gate_up_tc", lib().moe_gate_up_tc(layer.handle, _ptr(hn), M, _ptr(experts), _ptr(masks),
                                                 U, _ptr(act), _ptr(err), _stream(stream)))
    return act, err


def down_tc(layer: Layer, act: torch.Tensor, experts: torch.Tensor, masks: torch.Tensor, y=None, err=None,
            stream=None):
    """Grouped down projection on the tensor cores (moe_down_tc).

    act fp32 [U, M, I], experts int32 [U], masks int32 [U] on the device.
    Returns (y fp32 [U, M, H], err int32 [1])."""
    _need(act, "act", torch.float32, (None, None, layer.desc.I))
    U, M = act.shape[0], act.shape[1]
    _need(experts, "experts", torch.int32, (U,))
    _need(masks, "masks", torch.int32, (U,))
    if y is None:
        y = torch.zeros((U, M, layer.desc.H), dtype=torch.float32, device=act.device)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=act.device)
    _need(y, "y", torch.float32, (U, M, layer.desc.H))
    _need(err, "err", torch.int32, (1,))
    check("moe_down_tc", lib().moe_down_tc(layer.handle, _ptr(act), M, _ptr(experts), _ptr(masks), U,
                                           _ptr(y), _ptr(err), _stream(stream)))
    return y, err


class Stack:
    def __init__(self, layers):
        self.layers = list(layers)
        arr = (C.c_void_p * len(self.layers))(*[l.handle.value for l in self.layers])
        h = C.c_void_p()
        check("moe_stack_create", lib().moe_stack_create(arr, len(self.layers), C.byref(h)))
        self.handle = h

    def forward(self, x: torch.Tensor, ws: Workspace, out=None, normed: bool = False, stream=None):
        H = self.layers[0].desc.H
        _need(x, "x", torch.bfloat16, (None, H))
        M = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        _need(out, "out", torch.bfloat16, (M, H))
        on = torch.empty_like(x) if normed else None
        check("moe_stack_forward", lib().moe_stack_forward(self.handle, _ptr(_bits16(x)), M, _ptr(_bits16(out)),
                                                           _ptr(_bits16(on)) if on is not None else None,
                                                           ws.ptr, ws.nbytes, _stream(stream)))
        return (out, on) if normed else out

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor, ws: Workspace, stream=None):
        """Host buffers in and out (copies inside the call); synchronises."""
        for name, t in (("x_host", x_host), ("out_host", out_host)):
            if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
                raise ValueError(f"{name} must be a contiguous bfloat16 host tensor")
        if x_host.dim() != 2 or x_host.shape[1] != self.layers[0].desc.H or tuple(out_host.shape) != tuple(x_host.shape):
            raise ValueError("x_host and out_host must both have shape [M, H]")
        M = x_host.shape[0]
        check("moe_stack_forward_host",
              lib().moe_stack_forward_host(self.handle, _bits16(x_host).data_ptr(), M, _bits16(out_host).data_ptr(),
                                           ws.ptr, ws.nbytes, _stream(stream)))
        return out_host

    def __del__(self):
        try:
            if getattr(self, "handle", None):
                lib().moe_stack_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


class QKV:
    """A packed fused Q/K/V projection (moe_qkv_pack): q, k, v are canonical
    dicts (codes [n, H] uint8, scales/biases bf16 [n, H/64]) or fp32 weights
    [n, H]; the device blob is a torch uint8 tensor owned here."""

    def __init__(self, H: int, q, k, v, bits: int = 8, device="cuda", stream=None):
        mats = [q, k, v]
        rows = [(m["codes"] if isinstance(m, dict) and m.get("codes") is not None else
                 (m["w"] if isinstance(m, dict) else m)).shape[0] for m in mats]
        self.desc = QkvDesc(H, rows[0], rows[1], rows[2], bits)
        self.rows = sum(rows)
        n = C.c_size_t()
        check("moe_qkv_pack_size", lib().moe_qkv_pack_size(C.byref(self.desc), C.byref(n)))
        self.nbytes = n.value
        self.blob = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        srcs, keep = [], []
        for m in mats:
            sm, kp = _src_matrix(m)
            srcs.append(sm)
            keep += kp
        h = C.c_void_p()
        check("moe_qkv_pack", lib().moe_qkv_pack(C.byref(self.desc), C.byref(srcs[0]), C.byref(srcs[1]),
                                                 C.byref(srcs[2]), _ptr(self.blob), self.nbytes, C.byref(h),
                                                 _stream(stream)))
        self.handle = h
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
        del keep

    def forward(self, x: torch.Tensor, out=None, err=None, stream=None):
        """y fp32 [M, n_q + n_k + n_v] for x bf16 [M, H] (moe_qkv_forward);
        returns (y, err) with err an int32 [1] device flag (1 = a wait ran out)."""
        _need(x, "x", torch.bfloat16, (None, self.desc.H))
        M = x.shape[0]
        if out is None:
            out = torch.empty((M, self.rows), dtype=torch.float32, device=x.device)
        _need(out, "out", torch.float32, (M, self.rows))
        if err is None:
            err = torch.zeros(1, dtype=torch.int32, device=x.device)
        _need(err, "err", torch.int32, (1,))
        check("moe_qkv_forward", lib().moe_qkv_forward(self.handle, _ptr(_bits16(x)), M, _ptr(out), _ptr(err),
                                                       _stream(stream)))
        return out, err

    def __del__(self):
        try:
            if getattr(self, "handle", None):
                lib().moe_qkv_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


class StreamedLayer:
    """A layer whose routed experts live in pinned host memory, with an HBM
    cache of n_slots experts (moe_streamed_*).  Built from a packed Layer,
    which may be dropped afterwards; usable wherever a Layer is (decode_layer,
    router_topk, Stack), and by streamed_forward."""

    def __init__(self, layer: Layer, n_slots: int, stream=None):
        self.desc = layer.desc
        n = C.c_size_t()
        check("moe_streamed_size", lib().moe_streamed_size(C.byref(self.desc), n_slots, C.byref(n)))
        self.host = torch.empty(layer.nbytes, dtype=torch.uint8, pin_memory=True)
        self.dev = torch.empty(n.value, dtype=torch.uint8, device=layer.blob.device)
        h = C.c_void_p()
        check("moe_streamed_create", lib().moe_streamed_create(layer.handle, self.host.data_ptr(), layer.nbytes,
                                                               _ptr(self.dev), n.value, n_slots, C.byref(h),
                                                               _stream(stream)))
        self.sh = h
        self.handle = C.c_void_p(lib().moe_streamed_layer(h))
        self.n_slots = n_slots
        self.nbytes = n.value

    def prepare(self, expert_ids, stream=None) -> int:
        """Make the listed experts resident; returns how many were copied."""
        ids = (C.c_int32 * len(expert_ids))(*[int(e) for e in expert_ids])
        f = C.c_int()
        check("moe_streamed_prepare", lib().moe_streamed_prepare(self.sh, ids, len(expert_ids), _stream(stream),
                                                                 C.byref(f)))
        return f.value

    def stats(self) -> dict:
        v = [C.c_longlong() for _ in range(6)]
        check("moe_streamed_stats", lib().moe_streamed_stats(self.sh, *[C.byref(x) for x in v]))
        return dict(zip(("hits", "misses", "fetched", "bytes", "predicted", "predicted_used"), (x.value for x in v)))

    def __del__(self):
        try:
            if getattr(self, "sh", None):
                lib().moe_streamed_destroy(self.sh)
                self.sh = None
        except Exception:
            pass


def streamed_forward(layers, x: torch.Tensor, ws: Workspace, out=None, normed: bool = False, predict: bool = True,
                     stream=None, copy_stream=None):
    """One forward of x bf16 [M, H] through StreamedLayers (moe_streamed_forward)."""
    H = layers[0].desc.H
    _need(x, "x", torch.bfloat16, (None, H))
    M = x.shape[0]
    k = layers[0].desc.k
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", torch.bfloat16, (M, H))
    on = torch.empty_like(x) if normed else None
    route = torch.empty(16 * M * k, dtype=torch.uint8, device=x.device)
    if predict and copy_stream is None:
        copy_stream = torch.cuda.Stream(device=x.device)
    arr = (C.c_void_p * len(layers))(*[l.sh.value for l in layers])
    check("moe_streamed_forward",
          lib().moe_streamed_forward(arr, len(layers), _ptr(_bits16(x)), M, _ptr(_bits16(out)),
                                     _ptr(_bits16(on)) if on is not None else None, ws.ptr, ws.nbytes,
                                     _ptr(route), route.numel(), 1 if predict else 0, _stream(stream),
                                     copy_stream.cuda_stream if copy_stream is not None else None))
    return (out, on) if normed else out


class AttnCache:
    """A bf16 key/value cache of the decode attention (moe_attn_*): keys
    [2, T_cap, 256] and values stored transposed [2, 256, T_cap], zeroed, with
    the scratch the attention call needs."""

    HQ, HKV, D = 16, 2, 256

    def __init__(self, T_cap: int, device="cuda"):
        if T_cap < 8 or T_cap % 8:
            raise ValueError("T_cap must be a positive multiple of 8")
        self.T_cap = T_cap
        self.k = torch.zeros((self.HKV, T_cap, self.D), dtype=torch.bfloat16, device=device)
        self.vt = torch.zeros((self.HKV, self.D, T_cap), dtype=torch.bfloat16, device=device)
        n = C.c_size_t()
        check("moe_attn_workspace_size", lib().moe_attn_workspace_size(T_cap, C.byref(n)))
        self.ws = torch.empty(n.value, dtype=torch.uint8, device=device)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, pos0: int, stream=None) -> None:
        """Keys and values of M new rows (bf16 [M, 2, 256]) at positions pos0 .. pos0 + M - 1."""
        _need(k_new, "k_new", torch.bfloat16, (None, self.HKV, self.D))
        M = k_new.shape[0]
        _need(v_new, "v_new", torch.bfloat16, (M, self.HKV, self.D))
        check("moe_attn_append", lib().moe_attn_append(_ptr(_bits16(k_new)), _ptr(_bits16(v_new)), M, pos0,
                                                       _ptr(self.k), _ptr(self.vt), self.T_cap, _stream(stream)))

    def attend(self, q: torch.Tensor, pos0: int, out=None, err=None, stream=None):
        """o fp32 [M, 16, 256] of query rows q bf16 [M, 16, 256] at positions
        pos0 .. pos0 + M - 1 (moe_attn_decode); returns (o, err)."""
        _need(q, "q", torch.bfloat16, (None, self.HQ, self.D))
        M = q.shape[0]
        if out is None:
            out = torch.empty((M, self.HQ, self.D), dtype=torch.float32, device=q.device)
        _need(out, "out", torch.float32, (M, self.HQ, self.D))
        if err is None:
            err = torch.zeros(1, dtype=torch.int32, device=q.device)
        _need(err, "err", torch.int32, (1,))
        check("moe_attn_decode", lib().moe_attn_decode(_ptr(_bits16(q)), _ptr(self.k), _ptr(self.vt), self.T_cap,
                                                       pos0, M, _ptr(out), _ptr(self.ws), self.ws.numel(),
                                                       _ptr(err), _stream(stream)))
        return out, err


def debug_set(skip_row: int = -1, timeout_ns: int = 0) -> None:
    check("moe_debug_set", lib().moe_debug_set(skip_row, timeout_ns))


def set_grouped_products(tensor_cores: bool) -> None:
    """moe_set_grouped_products: grouped mode's expert products on the tensor
    cores (True) or the FMA pipes (False, the default)."""
    check("moe_set_grouped_products", lib().moe_set_grouped_products(1 if tensor_cores else 0))


def build_flags() -> int:
    """moe_build_flags: MOE_BUILD_DEBUG_BOUNDS (1) in the bounds-checked build."""
    return int(lib().moe_build_flags())


def debug_inject(expert: int = -1) -> None:
    """moe_debug_inject (bounds-checked build only; raises MoeError otherwise)."""
    check("moe_debug_inject", lib().moe_debug_inject(expert))


def launch_count(reset: bool = False) -> int:
    return int(lib().moe_launch_count(1 if reset else 0))


def layer_src_from_synth(L: dict) -> dict:
    """Source-tensor dict for Layer() from synth.make_layer's canonical dict."""
    src = {"gate": L["gate"], "up": L["up"], "down": L["down"], "gamma": L["gamma"],
           "gamma_next": L.get("gamma_next")}
    sh = L["shape"]
    src["router"] = {"w": L["router_w"]}
    if sh.has_shared:
        src["shared_gate"] = L["shared_gate"]
        src["shared_up"] = L["shared_up"]
        src["shared_down"] = L["shared_down"]
        src["sgate"] = {"w": L["sgate_w"].reshape(1, -1)}
    return src
