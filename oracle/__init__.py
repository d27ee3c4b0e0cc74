"""ctypes wrapper around the plain C oracle (ts_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and
bench.py's cpu_baseline / ``--impl reference`` legs.  The product library
(mixture_experts_routed_logits_gb300) never imports this package, and this
package never imports the product library.

Every function takes and returns numpy arrays in the canonical layouts
described in ts_oracle.h; 16-bit floats travel as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libts_oracle.so")
# tests/test_oracle_mutations.py points this at a deliberately broken copy of the oracle
_LIB_OVERRIDE = os.environ.get("TS_ORACLE_LIB_OVERRIDE")
_lib = None

FMT = {"f16": 0, "bf16": 1, "mxfp4": 2, "int4": 3}
ACT = {"silu": 0, "gelu_tanh": 1, "gptoss": 2}
MODE = {"softmax_k": 0, "sigmoid_biased": 1, "softmax_k_scaled": 2}
ADT = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile ts_oracle.c with gcc (-O2 -ffp-contract=off -fopenmp)."""
    src = os.path.join(_HERE, "ts_oracle.c")
    hdr = os.path.join(_HERE, "ts_oracle.h")
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(src), os.path.getmtime(hdr))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-Wall", "-shared",
           "-fPIC", "-o", tmp, src, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Experts(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("act", ctypes.c_int), ("E", ctypes.c_int),
                ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("gate_s", ctypes.c_void_p), ("up_s", ctypes.c_void_p), ("down_s", ctypes.c_void_p),
                ("gate_b", ctypes.c_void_p), ("up_b", ctypes.c_void_p), ("down_b", ctypes.c_void_p),
                ("limit", ctypes.c_float), ("alpha", ctypes.c_float)]


def lib():
    global _lib
    if _lib is None:
        if _LIB_OVERRIDE:
            L = ctypes.CDLL(_LIB_OVERRIDE)
        else:
            build()
            L = ctypes.CDLL(_LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.or_f16_to_double.argtypes = [ctypes.c_uint16]
        L.or_f16_to_double.restype = ctypes.c_double
        L.or_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.or_bf16_to_double.restype = ctypes.c_double
        L.or_double_to_f16.argtypes = [ctypes.c_double]
        L.or_double_to_f16.restype = ctypes.c_uint16
        L.or_double_to_bf16.argtypes = [ctypes.c_double]
        L.or_double_to_bf16.restype = ctypes.c_uint16
        L.or_e2m1_value.argtypes = [i]
        L.or_e2m1_value.restype = ctypes.c_double
        L.or_e8m0_value.argtypes = [i]
        L.or_e8m0_value.restype = ctypes.c_double
        L.or_weight.argtypes = [ctypes.POINTER(_Experts), i, i, i, i]
        L.or_weight.restype = ctypes.c_double
        L.or_dot32f.argtypes = [vp, vp, i]
        L.or_dot32f.restype = ctypes.c_float
        L.or_act.argtypes = [i, ctypes.c_double, ctypes.c_double, f, f]
        L.or_act.restype = ctypes.c_double
        L.or_rmsnorm.argtypes = [vp, i, i, i, f, vp]
        L.or_gemma_tail.argtypes = [vp, vp, vp, vp, vp, f, f, i, i, i]
        L.or_router_logits.argtypes = [vp, vp, i, i, i, i, vp]
        L.or_route.argtypes = [vp, vp, vp, i, i, i, i, vp, vp]
        L.or_build_routes.argtypes = [vp, i, i, i, vp, vp, vp]
        L.or_expert_ffn.argtypes = [ctypes.POINTER(_Experts), i, vp, i, vp, vp]
        L.or_moe_forward.argtypes = [vp, i, i, ctypes.POINTER(_Experts), vp, vp, i,
                                     ctypes.POINTER(_Experts), vp, i, vp, vp, vp, i]
        L.or_expert_pre.argtypes = [ctypes.POINTER(_Experts), i, vp, vp, vp, vp, vp]
        L.or_act_n.argtypes = [i, vp, vp, i, f, f, vp]
        L.or_act_n.restype = None
        for name in ("or_rmsnorm", "or_gemma_tail", "or_router_logits", "or_route",
                     "or_build_routes", "or_expert_ffn", "or_expert_pre", "or_moe_forward"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    """16-bit float array (numpy float16, or uint16/int16 bits) -> contiguous uint16 bits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype in (np.uint16, np.int16), a.dtype
    return a.view(np.uint16)


class Experts:
    """Holds numpy arrays (kept alive) and the C descriptor for one expert set."""

    def __init__(self, fmt, act, E, H, I, gate, up, down, gate_s=None, up_s=None, down_s=None,
                 gate_b=None, up_b=None, down_b=None, limit=7.0, alpha=1.702):
        fmt_i = FMT[fmt] if isinstance(fmt, str) else int(fmt)
        act_i = ACT[act] if isinstance(act, str) else int(act)
        conv = (lambda a: _u16(a)) if fmt_i in (0, 1) else (lambda a: np.ascontiguousarray(a, np.uint8))
        self._keep = dict(
            gate=conv(gate), up=conv(up), down=conv(down),
            gate_s=None if gate_s is None else np.ascontiguousarray(gate_s),
            up_s=None if up_s is None else np.ascontiguousarray(up_s),
            down_s=None if down_s is None else np.ascontiguousarray(down_s),
            gate_b=None if gate_b is None else _u16(gate_b),
            up_b=None if up_b is None else _u16(up_b),
            down_b=None if down_b is None else _u16(down_b))
        k = self._keep
        self.c = _Experts(fmt_i, act_i, E, H, I, _p(k["gate"]), _p(k["up"]), _p(k["down"]),
                          _p(k["gate_s"]), _p(k["up_s"]), _p(k["down_s"]),
                          _p(k["gate_b"]), _p(k["up_b"]), _p(k["down_b"]), limit, alpha)
        self.E, self.H, self.I = E, H, I


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def rmsnorm(x, adt, eps=1e-6):
    x = _u16(x)
    T, H = x.shape
    out = np.empty_like(x)
    _check(lib().or_rmsnorm(_p(x), T, H, ADT[adt], eps, _p(out)), "rmsnorm")
    return out


def gemma_tail(y, h1, x, w_post2, w_post, adt, layer_scalar, eps=1e-6):
    """The Gemma sandwich tail on copies of y, h1, x ([T][H] 16-bit bits): returns the new
    (y, h1, x)."""
    y, h1, x = _u16(y).copy(), _u16(h1).copy(), _u16(x).copy()
    w_post2, w_post = _u16(w_post2), _u16(w_post)
    T, H = y.shape
    _check(lib().or_gemma_tail(_p(y), _p(h1), _p(x), _p(w_post2), _p(w_post), layer_scalar, eps,
                               T, H, ADT[adt]), "gemma_tail")
    return y, h1, x


def router_logits(x, Wr, adt):
    x, Wr = _u16(x), _u16(Wr)
    T, H = x.shape
    E = Wr.shape[0]
    out = np.empty((T, E), np.float32)
    _check(lib().or_router_logits(_p(x), _p(Wr), T, H, E, ADT[adt], _p(out)), "router_logits")
    return out


def route(logits, k, mode="softmax_k", bias=None, scale=None):
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    bias = None if bias is None else np.ascontiguousarray(bias, np.float32)
    scale = None if scale is None else np.ascontiguousarray(scale, np.float32)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _check(lib().or_route(_p(logits), _p(bias), _p(scale), T, E, k, MODE[mode], _p(idx), _p(w)),
           "route")
    return idx, w


def build_routes(idx, E):
    idx = np.ascontiguousarray(idx, np.int32)
    T, k = idx.shape
    off = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    _check(lib().or_build_routes(_p(idx), T, E, k, _p(off), _p(perm), _p(inv)), "build_routes")
    return off, perm, inv


def expert_ffn(ex: Experts, e, xin, adt):
    xin = np.ascontiguousarray(xin, np.float64)
    h = np.empty(ex.I, np.float64)
    eo = np.empty(ex.H, np.float32)
    _check(lib().or_expert_ffn(ctypes.byref(ex.c), e, _p(xin), ADT[adt], _p(h), _p(eo)),
           "expert_ffn")
    return h, eo


def expert_pre(ex: Experts, e, xin):
    """Phase-1 pre-activation sums of expert e for one input row (float64, biases added) and
    their absolute sums: (g [I], u [I], sum |W_g x| [I], sum |W_u x| [I])."""
    xin = np.ascontiguousarray(xin, np.float64)
    g, u, sg, su = (np.empty(ex.I, np.float64) for _ in range(4))
    _check(lib().or_expert_pre(ctypes.byref(ex.c), e, _p(xin), _p(g), _p(u), _p(sg), _p(su)),
           "expert_pre")
    return g, u, sg, su


def act(ex: Experts, g, u):
    """The expert set's gated activation over arrays g, u (float64)."""
    g = np.ascontiguousarray(g, np.float64)
    u = np.ascontiguousarray(u, np.float64)
    out = np.empty_like(g)
    lib().or_act_n(ex.c.act, _p(g), _p(u), g.size, ex.c.limit, ex.c.alpha, _p(out))
    return out


def moe_forward(x, adt, ex: Experts, idx, w, shared: Experts | None = None, tokens=None,
                nthreads=1, want_routes=False):
    """Returns (y bits [n,H] uint16, y_f32 [n,H], e_routes [n,k,H] or None)."""
    x = _u16(x)
    T, H = x.shape
    idx = np.ascontiguousarray(idx, np.int32)
    w = np.ascontiguousarray(w, np.float32)
    k = idx.shape[1]
    toks = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
    n = T if toks is None else len(toks)
    y = np.empty((n, H), np.uint16)
    yf = np.empty((n, H), np.float32)
    er = np.empty((n, k, H), np.float32) if want_routes else None
    rc = lib().or_moe_forward(_p(x), ADT[adt], T, ctypes.byref(ex.c), _p(idx), _p(w), k,
                              None if shared is None else ctypes.byref(shared.c), _p(toks), n,
                              _p(y), _p(yf), _p(er), int(nthreads))
    _check(rc, "moe_forward")
    return y, yf, er


def f16_bits_to_f64(b):
    L = lib()
    return np.array([L.or_f16_to_double(int(v)) for v in np.asarray(b).ravel()]).reshape(np.shape(b))


def bf16_bits_to_f64(b):
    b = np.asarray(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def adt_bits_to_f64(b, adt):
    b = np.asarray(b, np.uint16)
    if adt == "bf16":
        return bf16_bits_to_f64(b)
    return b.view(np.float16).astype(np.float64)
