"""CPU oracle for the routed mixture-of-experts FFN (test infrastructure).

This package is the reference the CUDA library is checked against.  Only the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use
it; the library never imports, links or calls it.  The arithmetic lives in
``moe_oracle.c`` (plain C, fp64, compiled with gcc and no floating-point
contraction); this module only compiles it and marshals numpy arrays.

Every function here takes canonical-layout inputs (see ``workload.gen``):
nibble-packed int4 rows, fp16 (scale, bias) pairs per group of 64 inputs,
fp16 router weights and bf16 activations passed as their uint16 bit patterns.
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fp contraction, so x86 and Arm agree)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        base = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                "-shared", _SRC, "-o", tmp, "-lm"]
        try:   # threads over matrix rows where the compiler has OpenMP, else one thread
            subprocess.check_call(base[:1] + ["-fopenmp"] + base[1:], stderr=subprocess.DEVNULL)
        except subprocess.CalledProcessError:
            subprocess.check_call(base)
        os.replace(tmp, _SO)
    return _SO


class OrLayer(C.Structure):
    _fields_ = [("d", C.c_int), ("f", C.c_int), ("f_shared", C.c_int), ("n_experts", C.c_int),
                ("top_k", C.c_int), ("group", C.c_int), ("gelu_variant", C.c_int),
                ("router_w", C.c_void_p),
                ("gate_q", C.c_void_p), ("up_q", C.c_void_p), ("down_q", C.c_void_p),
                ("gate_sb", C.c_void_p), ("up_sb", C.c_void_p), ("down_sb", C.c_void_p),
                ("s_gate_q", C.c_void_p), ("s_up_q", C.c_void_p), ("s_down_q", C.c_void_p),
                ("s_gate_sb", C.c_void_p), ("s_up_sb", C.c_void_p), ("s_down_sb", C.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            vp, i32, i64, dbl = C.c_void_p, C.c_int, C.c_int64, C.c_double
            L.or_fp16_to_double.restype = dbl
            L.or_fp16_to_double.argtypes = [C.c_uint16]
            L.or_bf16_to_double.restype = dbl
            L.or_bf16_to_double.argtypes = [C.c_uint16]
            L.or_double_to_bf16.restype = C.c_uint16
            L.or_double_to_bf16.argtypes = [dbl]
            L.or_weight.restype = dbl
            L.or_weight.argtypes = [vp, vp, i32, i32, i32, i32]
            L.or_matvec.restype = None
            L.or_matvec.argtypes = [vp, vp, i32, i32, i32, vp, vp]
            L.or_gelu.restype = dbl
            L.or_gelu.argtypes = [dbl, i32]
            L.or_expert_ffn.restype = None
            L.or_expert_ffn.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp]
            L.or_router_logits.restype = i32
            L.or_router_logits.argtypes = [vp, vp, vp, i32, i32, vp]
            L.or_topk.restype = None
            L.or_topk.argtypes = [vp, i32, i32, vp]
            L.or_gates.restype = None
            L.or_gates.argtypes = [vp, vp, i32, vp]
            L.or_moe_layer.restype = i32
            L.or_moe_layer.argtypes = [C.POINTER(OrLayer), vp, vp, vp, vp, vp, vp]
            L.or_rmsnorm_bf16.restype = None
            L.or_rmsnorm_bf16.argtypes = [vp, i32, dbl, vp]
            L.or_residual_bf16.restype = None
            L.or_residual_bf16.argtypes = [vp, vp, i32, vp]
            L.or_lru_step.restype = i32
            L.or_lru_step.argtypes = [i32, vp, vp, vp, i32, i64, vp, vp, vp]
            L.or_lfu_step.restype = i32
            L.or_lfu_step.argtypes = [i32, vp, vp, vp, vp, i32, i64, vp, vp, vp]
            L.or_set_threads.restype = i32
            L.or_set_threads.argtypes = [i32]
            _lib = L
    return _lib


def set_threads(n: int) -> int:
    """Host threads over the rows of each matrix-vector product (results do not
    depend on it); returns the count in effect."""
    return lib().or_set_threads(n)


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def as_bits(t) -> np.ndarray:
    """uint16 bit patterns of a 16-bit float torch tensor or numpy array (CPU copy)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    return a.view(np.uint16) if a.dtype.itemsize == 2 else a


def as_np(t) -> np.ndarray:
    try:
        import torch
        if isinstance(t, torch.Tensor):
            if t.dtype in (torch.float16, torch.bfloat16):
                return as_bits(t)
            return np.ascontiguousarray(t.detach().cpu().contiguous().numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(t)


# ---------------------------------------------------------------- scalars

def fp16_to_double(bits: int) -> float:
    return lib().or_fp16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return lib().or_bf16_to_double(int(bits))


def double_to_bf16(v: float) -> int:
    return int(lib().or_double_to_bf16(float(v)))


def gelu(x: float, variant: int = 0) -> float:
    return lib().or_gelu(float(x), int(variant))


# ---------------------------------------------------------------- vectors

def matvec(q, sb, x, group: int = 64) -> np.ndarray:
    q, sb = as_np(q), as_bits(sb)
    rows, half = q.shape
    cols = 2 * half
    xd = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.zeros(rows, dtype=np.float64)
    lib().or_matvec(_p(q), _p(sb), rows, cols, group, _p(xd), _p(y))
    return y


def expert_ffn(w: dict, x, group: int = 64, variant: int = 0) -> np.ndarray:
    """w: one expert's canonical tensors (gate_q [f,d/2], ..., down_sb [d,f/g,2])."""
    gq, gsb = as_np(w["gate_q"]), as_bits(w["gate_sb"])
    uq, usb = as_np(w["up_q"]), as_bits(w["up_sb"])
    dq, dsb = as_np(w["down_q"]), as_bits(w["down_sb"])
    f, half = gq.shape
    d = 2 * half
    xd = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.zeros(d, dtype=np.float64)
    lib().or_expert_ffn(_p(gq), _p(gsb), _p(uq), _p(usb), _p(dq), _p(dsb), d, f, group, variant,
                        _p(xd), _p(y))
    return y


def router_logits(router_w, x_bits, bias=None):
    w = as_bits(router_w)
    x = as_bits(x_bits)
    E, d = w.shape
    out = np.zeros(E, dtype=np.int64)
    b = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float32))
    st = lib().or_router_logits(_p(w), _p(x), None if b is None else _p(b), E, d, _p(out))
    return out, st


def topk(logits, k: int) -> np.ndarray:
    lg = np.ascontiguousarray(np.asarray(logits, dtype=np.int64))
    ids = np.zeros(k, dtype=np.int32)
    lib().or_topk(_p(lg), lg.shape[0], k, _p(ids))
    return ids


def gates(logits, ids) -> np.ndarray:
    lg = np.ascontiguousarray(np.asarray(logits, dtype=np.int64))
    ii = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    g = np.zeros(ii.shape[0], dtype=np.float64)
    lib().or_gates(_p(lg), _p(ii), ii.shape[0], _p(g))
    return g


class Layer:
    """Holds numpy views of one layer's canonical weights for repeated calls."""

    def __init__(self, weights: dict, top_k: int, group: int = 64, gelu_variant: int = 0):
        ex, sh = weights["experts"], weights["shared"]
        self.arrays = {
            "router_w": as_bits(weights["router_w"]),
            "gate_q": as_np(ex["gate_q"]), "up_q": as_np(ex["up_q"]), "down_q": as_np(ex["down_q"]),
            "gate_sb": as_bits(ex["gate_sb"]), "up_sb": as_bits(ex["up_sb"]),
            "down_sb": as_bits(ex["down_sb"]),
            "s_gate_q": as_np(sh["gate_q"]), "s_up_q": as_np(sh["up_q"]),
            "s_down_q": as_np(sh["down_q"]), "s_gate_sb": as_bits(sh["gate_sb"]),
            "s_up_sb": as_bits(sh["up_sb"]), "s_down_sb": as_bits(sh["down_sb"]),
        }
        a = self.arrays
        E, d = a["router_w"].shape
        f = a["gate_q"].shape[1]
        fs = a["s_gate_q"].shape[0]
        self.d, self.f, self.fs, self.E, self.k, self.group = d, f, fs, E, top_k, group
        self.s = OrLayer(d, f, fs, E, top_k, group, gelu_variant,
                         *[_p(a[n]) for n in ("router_w", "gate_q", "up_q", "down_q", "gate_sb",
                                              "up_sb", "down_sb", "s_gate_q", "s_up_q", "s_down_q",
                                              "s_gate_sb", "s_up_sb", "s_down_sb")])

    def forward(self, x_bits, bias=None):
        """One token: returns (ids int32[k], gates f64[k], logits int64[E], y f64[d], status)."""
        x = np.ascontiguousarray(as_bits(x_bits).reshape(-1))
        assert x.shape[0] == self.d
        b = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float32).reshape(-1))
        ids = np.zeros(self.k, dtype=np.int32)
        g = np.zeros(self.k, dtype=np.float64)
        lg = np.zeros(self.E, dtype=np.int64)
        y = np.zeros(self.d, dtype=np.float64)
        st = lib().or_moe_layer(C.byref(self.s), _p(x), None if b is None else _p(b), _p(ids), _p(g),
                                _p(lg), _p(y))
        return ids, g, lg, y, st


def rmsnorm_bf16(h_bits, eps: float = 1e-6) -> np.ndarray:
    h = np.ascontiguousarray(as_bits(h_bits).reshape(-1))
    out = np.zeros_like(h)
    lib().or_rmsnorm_bf16(_p(h), h.shape[0], float(eps), _p(out))
    return out


def residual_bf16(h_bits, y) -> np.ndarray:
    h = np.ascontiguousarray(as_bits(h_bits).reshape(-1))
    yd = np.ascontiguousarray(np.asarray(y, dtype=np.float64).reshape(-1))
    out = np.zeros_like(h)
    lib().or_residual_bf16(_p(h), _p(yd), h.shape[0], _p(out))
    return out


class LRU:
    """One layer's LRU slot table (expert_of_slot, last_use), oracle rules."""

    def __init__(self, n_slots: int):
        self.n = n_slots
        self.expert_of_slot = np.full(n_slots, -1, dtype=np.int32)
        self.last_use = np.full(n_slots, -1, dtype=np.int64)

    def step(self, ids, t: int):
        ii = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        k = ii.shape[0]
        hit = np.zeros(k, dtype=np.int32)
        slot = np.zeros(k, dtype=np.int32)
        ev = np.zeros(k, dtype=np.int32)
        m = lib().or_lru_step(self.n, _p(self.expert_of_slot), _p(self.last_use), _p(ii), k, int(t),
                              _p(hit), _p(slot), _p(ev))
        if m < 0:
            raise ValueError("n_slots < k")
        return hit, slot, ev


class LFU:
    """One layer's LFU slot table: expert_of_slot, last_use and the whole-run
    use count of every expert (or_lfu_step rules)."""

    def __init__(self, n_slots: int, n_experts: int):
        self.n = n_slots
        self.expert_of_slot = np.full(n_slots, -1, dtype=np.int32)
        self.last_use = np.full(n_slots, -1, dtype=np.int64)
        self.use_count = np.zeros(n_experts, dtype=np.int64)

    def step(self, ids, t: int):
        ii = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        k = ii.shape[0]
        hit = np.zeros(k, dtype=np.int32)
        slot = np.zeros(k, dtype=np.int32)
        ev = np.zeros(k, dtype=np.int32)
        m = lib().or_lfu_step(self.n, _p(self.expert_of_slot), _p(self.last_use), _p(self.use_count), _p(ii), k,
                              int(t), _p(hit), _p(slot), _p(ev))
        if m < 0:
            raise ValueError("n_slots < k")
        return hit, slot, ev


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact decoding of bf16 bit patterns to float64 (vectorised, for tests)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
