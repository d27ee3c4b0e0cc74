"""GB300 (sm_103a) routed-expert (MoE) layer: Python binding of libts_moe.so.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels
(include/ts_moe.h documents the C ABI).  PyTorch provides device memory and streams.  There
is no CPU fallback: if the library is missing or fails to load, every call raises.

Typical use::

    import mixture_experts_routed_logits_gb300 as moe
    ex = moe.Experts.from_canonical("mxfp4", "gptoss", gate, up, down, gate_s, up_s, down_s, ...)
    idx, w, xn, _ = moe.router_route(x, W_r, k=4, router_bias=b)
    y, y32 = moe.forward(x, ex, idx, w)
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libts_moe.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "ts_moe.h")

FMT = {"f16": 0, "bf16": 1, "mxfp4": 2, "int4": 3}
ACT = {"silu": 0, "gelu_tanh": 1, "gptoss": 2}
MODE = {"softmax_k": 0, "sigmoid_biased": 1, "softmax_k_scaled": 2}
ADT = {"f16": 0, "bf16": 1}
PATH = {"auto": 0, "gemv": 1, "gemm": 2, "gemm_dequant": 3}
STATUS = {0: "TS_OK", 1: "TS_ERR_INVALID_ARG", 2: "TS_ERR_UNSUPPORTED", 3: "TS_ERR_CUDA",
          4: "TS_ERR_TIMEOUT", 5: "TS_ERR_WORKSPACE"}


class TsMoeError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class CExperts(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("act", ctypes.c_int32), ("E", ctypes.c_int32),
                ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("gate_b", ctypes.c_void_p), ("up_b", ctypes.c_void_p), ("down_b", ctypes.c_void_p),
                ("swiglu_limit", ctypes.c_float), ("swiglu_alpha", ctypes.c_float),
                ("gateup_mx", ctypes.c_void_p), ("down_mx", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded libts_moe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        pe = ctypes.POINTER(CExperts)
        sig = {
            "ts_last_error": ([], ctypes.c_char_p),
            "ts_moe_version": ([], ctypes.c_char_p),
            "ts_moe_packed_bytes": ([i32, i32, i32, i32], sz),
            "ts_moe_pack": ([i32, i32, i32, i32, vp, vp, vp, sz, vp], ctypes.c_int),
            "ts_moe_packed_mx_bytes": ([i32, i32, i32, i32], sz),
            "ts_moe_pack_mx": ([i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
            "ts_moe_route": ([vp, vp, vp, i32, i32, i32, i32, vp, vp, vp], ctypes.c_int),
            "ts_moe_router_route": ([vp, i32, i32, i32, vp, i32, i32, f32, vp, vp, i32, i32, vp,
                                     vp, vp, vp, vp], ctypes.c_int),
            "ts_moe_build_routes": ([vp, i32, i32, i32, vp, vp, vp, vp], ctypes.c_int),
            "ts_moe_workspace_size": ([i32, i32, pe, pe], sz),
            "ts_moe_forward": ([vp, i32, i32, pe, vp, vp, i32, pe, vp, vp, vp, sz, vp],
                               ctypes.c_int),
            "ts_moe_forward_path": ([vp, i32, i32, pe, vp, vp, i32, pe, vp, vp, vp, sz, i32, vp],
                                    ctypes.c_int),
            "ts_moe_route_forward": ([vp, i32, i32, vp, i32, f32, vp, vp, i32, i32, pe, pe, vp, vp,
                                      vp, vp, vp, vp, sz, i32, vp], ctypes.c_int),
            "ts_moe_device_status": ([vp, ctypes.POINTER(i32), vp], ctypes.c_int),
            "ts_moe_forward_noalloc": ([vp, i32, i32, pe, vp, vp, i32, pe, vp, vp, vp],
                                       ctypes.c_int),
            "ts_moe_noalloc_device_status": ([ctypes.POINTER(i32), vp], ctypes.c_int),
            "ts_moe_set_wait_test": ([i32], ctypes.c_int),
            "ts_moe_set_phase_events": ([ctypes.POINTER(vp), i32], ctypes.c_int),
            "ts_moe_gemma_tail": ([vp, vp, vp, vp, vp, f32, f32, i32, i32, i32, vp], ctypes.c_int),
            "ts_moe_forward_tail": ([vp, i32, i32, pe, vp, vp, i32, pe, vp, vp, vp, sz, i32, vp, vp, vp,
                                     vp, f32, f32, vp], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def header_functions():
    """Names of the functions include/ts_moe.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ts_\w+)\s*\(", text)))


def check(status):
    if status != 0:
        raise TsMoeError(status, lib().ts_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# --------------------------------------------------------------------------------- weights

def packed_bytes(fmt, nmat, R, K):
    return lib().ts_moe_packed_bytes(FMT[fmt], nmat, R, K)


def pack(fmt, codes, scales, stream=None):
    """Pack canonical quantised weights ([nmat][R][K/2] codes + scales) for the kernels."""
    import torch
    nmat, R, half_k = codes.shape
    K = half_k * 2
    nb = packed_bytes(fmt, nmat, R, K)
    if nb == 0:
        raise TsMoeError(1, f"cannot pack fmt={fmt} R={R} K={K}")
    out = torch.empty(nb, dtype=torch.uint8, device=codes.device)
    check(lib().ts_moe_pack(FMT[fmt], nmat, R, K, _ptr(codes.contiguous()),
                            _ptr(scales.contiguous()), _ptr(out), nb, _stream(stream)))
    return out


def packed_mx_bytes(nmat, R, K, pair=False):
    return lib().ts_moe_packed_mx_bytes(int(pair), nmat, R, K)


def pack_mx(codes, scales, codes_up=None, scales_up=None, stream=None):
    """Tensor-core layout of canonical MXFP4 weights ([nmat][R][K/2] codes + e8m0 scales) for
    the block-scaled MMA path (ts_moe_pack_mx); with codes_up/scales_up, gate and up together."""
    import torch
    nmat, R, half_k = codes.shape
    K = half_k * 2
    pair = codes_up is not None
    nb = packed_mx_bytes(nmat, R, K, pair)
    if nb == 0:
        raise TsMoeError(1, f"cannot pack for the tensor cores: R={R} K={K}")
    out = torch.empty(nb + 256, dtype=torch.uint8, device=codes.device)
    off = (-out.data_ptr()) % 256
    out = out[off:off + nb]
    check(lib().ts_moe_pack_mx(int(pair), nmat, R, K, _ptr(codes.contiguous()), _ptr(scales.contiguous()),
                               _ptr(None if codes_up is None else codes_up.contiguous()),
                               _ptr(None if scales_up is None else scales_up.contiguous()),
                               _ptr(out), nb, _stream(stream)))
    return out


class Experts:
    """Device weights of one expert set plus its C descriptor (tensors are kept alive)."""

    def __init__(self, fmt, act, E, H, I, gate, up, down, gate_b=None, up_b=None, down_b=None,
                 swiglu_limit=7.0, swiglu_alpha=1.702, gateup_mx=None, down_mx=None):
        self.fmt, self.act, self.E, self.H, self.I = fmt, act, E, H, I
        self._keep = [gate, up, down, gate_b, up_b, down_b, gateup_mx, down_mx]
        ptr = lambda t: None if t is None else t.data_ptr()
        self.c = CExperts(FMT[fmt], ACT[act], E, H, I, gate.data_ptr(), up.data_ptr(),
                          down.data_ptr(), ptr(gate_b), ptr(up_b), ptr(down_b), swiglu_limit,
                          swiglu_alpha, ptr(gateup_mx), ptr(down_mx))

    @classmethod
    def from_canonical(cls, fmt, act, w: dict, stream=None, with_mx=True, **kw):
        """w: gate/up/down (+ _s scales, + _b biases) in the canonical layout, on the GPU.
        MXFP4 weights also get their tensor-core layout (block-scaled MMA path) unless
        with_mx is False."""
        gate, up, down = w["gate"], w["up"], w["down"]
        mx = {}
        if fmt in ("mxfp4", "int4"):
            E, I, half_h = gate.shape
            H = half_h * 2
            if fmt == "mxfp4" and with_mx:
                mx = dict(gateup_mx=pack_mx(gate, w["gate_s"], up, w["up_s"], stream=stream),
                          down_mx=pack_mx(down, w["down_s"], stream=stream))
            gate = pack(fmt, gate, w["gate_s"], stream)
            up = pack(fmt, up, w["up_s"], stream)
            down = pack(fmt, down, w["down_s"], stream)
        else:
            E, I, H = gate.shape
            gate, up, down = gate.contiguous(), up.contiguous(), down.contiguous()
        return cls(fmt, act, E, H, I, gate, up, down, w.get("gate_b"), w.get("up_b"),
                   w.get("down_b"), **mx, **kw)


# --------------------------------------------------------------------------------- routing

def route(logits, k, mode="softmax_k", router_bias=None, per_expert_scale=None, stream=None):
    import torch
    T, E = logits.shape
    idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    check(lib().ts_moe_route(_ptr(logits.contiguous()), _ptr(router_bias), _ptr(per_expert_scale),
                             T, E, k, MODE[mode], _ptr(idx), _ptr(w), _stream(stream)))
    return idx, w


def router_route(x, W_r, k, mode="softmax_k", router_bias=None, per_expert_scale=None,
                 rmsnorm=False, eps=1e-6, want_logits=False, out=None, stream=None):
    """Returns (idx [T,k] int32, w [T,k] f32, xn [T,H] or None, logits [T,E] or None)."""
    import torch
    T, H = x.shape
    E = W_r.shape[0]
    adt = {torch.float16: "f16", torch.bfloat16: "bf16"}[x.dtype]
    if out is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, k), dtype=torch.float32, device=x.device)
        xn = torch.empty_like(x) if rmsnorm else None
        logits = torch.empty((T, E), dtype=torch.float32, device=x.device) if want_logits else None
    else:
        idx, w, xn, logits = out
    check(lib().ts_moe_router_route(_ptr(x), ADT[adt], T, H, _ptr(W_r), E, int(rmsnorm), eps,
                                    _ptr(router_bias), _ptr(per_expert_scale), k, MODE[mode],
                                    _ptr(xn), _ptr(logits), _ptr(idx), _ptr(w), _stream(stream)))
    return idx, w, xn, logits


def gemma_tail(y, h1, x, w_post2, w_post, layer_scalar, eps=1e-6, stream=None):
    """The Gemma sandwich tail in place on y, h1, x ([T,H] f16/bf16): y <- rms(y) * w_post2,
    h1 <- h1 + y, x <- (x + rms(h1) * w_post) * layer_scalar (ts_moe_gemma_tail)."""
    import torch
    T, H = y.shape
    adt = {torch.float16: "f16", torch.bfloat16: "bf16"}[y.dtype]
    check(lib().ts_moe_gemma_tail(_ptr(y), _ptr(h1), _ptr(x), _ptr(w_post2), _ptr(w_post),
                                  float(layer_scalar), float(eps), ADT[adt], T, H, _stream(stream)))
    return y, h1, x


def build_routes(idx, E, stream=None):
    import torch
    T, k = idx.shape
    off = torch.empty(E + 1, dtype=torch.int32, device=idx.device)
    perm = torch.empty(T * k, dtype=torch.int32, device=idx.device)
    inv = torch.empty(T * k, dtype=torch.int32, device=idx.device)
    check(lib().ts_moe_build_routes(_ptr(idx), T, E, k, _ptr(off), _ptr(perm), _ptr(inv),
                                    _stream(stream)))
    return off, perm, inv


# --------------------------------------------------------------------------------- experts

def workspace_size(T, k, ex: Experts, shared: Experts | None = None):
    return lib().ts_moe_workspace_size(T, k, ctypes.byref(ex.c),
                                       None if shared is None else ctypes.byref(shared.c))


def alloc_workspace(T, k, ex, shared=None, device="cuda"):
    import torch
    n = workspace_size(T, k, ex, shared)
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def forward(x, ex: Experts, idx, w, shared: Experts | None = None, want_f32=False, ws=None,
            path="auto", out=None, stream=None):
    """y[t] = adt(seed[t] + sum_s w[t,s] * expert_{idx[t,s]}(x[t])); returns (y, y_f32)."""
    import torch
    T, H = x.shape
    k = idx.shape[1]
    adt = {torch.float16: "f16", torch.bfloat16: "bf16"}[x.dtype]
    if ws is None:
        ws = alloc_workspace(T, k, ex, shared, device=x.device)
    if out is None:
        y = torch.empty_like(x)
        y32 = torch.empty((T, H), dtype=torch.float32, device=x.device) if want_f32 else None
    else:
        y, y32 = out
    check(lib().ts_moe_forward_path(_ptr(x), ADT[adt], T, ctypes.byref(ex.c), _ptr(idx), _ptr(w),
                                    k, None if shared is None else ctypes.byref(shared.c),
                                    _ptr(y), _ptr(y32), _ptr(ws), ws.numel(), PATH[path],
                                    _stream(stream)))
    return y, y32


def forward_tail(x, ex: Experts, idx, w, h1, xres, w_post2, w_post, layer_scalar, eps=1e-6,
                 shared: Experts | None = None, want_f32=False, ws=None, path="auto", out=None,
                 stream=None):
    """forward() then gemma_tail(y, h1, xres, ...) in one call (ts_moe_forward_tail): y comes
    back normalised, h1 and xres are updated in place; returns (y, y_f32)."""
    import torch
    T, H = x.shape
    k = idx.shape[1]
    adt = {torch.float16: "f16", torch.bfloat16: "bf16"}[x.dtype]
    if ws is None:
        ws = alloc_workspace(T, k, ex, shared, device=x.device)
    if out is None:
        y = torch.empty_like(x)
        y32 = torch.empty((T, H), dtype=torch.float32, device=x.device) if want_f32 else None
    else:
        y, y32 = out
    check(lib().ts_moe_forward_tail(_ptr(x), ADT[adt], T, ctypes.byref(ex.c), _ptr(idx), _ptr(w),
                                    k, None if shared is None else ctypes.byref(shared.c),
                                    _ptr(y), _ptr(y32), _ptr(ws), ws.numel(), PATH[path],
                                    _ptr(h1), _ptr(xres), _ptr(w_post2), _ptr(w_post),
                                    float(layer_scalar), float(eps), _stream(stream)))
    return y, y32


def route_forward(x, W_r, k, ex: Experts, mode="softmax_k", router_bias=None, per_expert_scale=None,
                  rmsnorm=False, eps=1e-6, shared: Experts | None = None, want_f32=False, ws=None,
                  path="auto", out=None, stream=None):
    """router_route + forward in one call (ts_moe_route_forward): returns (y, y_f32, idx, w).
    For decode batches on the block-scaled kernels the router launch also does their prep."""
    import torch
    T, H = x.shape
    adt = {torch.float16: "f16", torch.bfloat16: "bf16"}[x.dtype]
    if ws is None:
        ws = alloc_workspace(T, k, ex, shared, device=x.device)
    if out is None:
        y = torch.empty_like(x)
        y32 = torch.empty((T, H), dtype=torch.float32, device=x.device) if want_f32 else None
        idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, k), dtype=torch.float32, device=x.device)
        xn = torch.empty_like(x) if rmsnorm else None
    else:
        y, y32, idx, w, xn = out
    check(lib().ts_moe_route_forward(_ptr(x), ADT[adt], T, _ptr(W_r), int(rmsnorm), eps,
                                     _ptr(router_bias), _ptr(per_expert_scale), k, MODE[mode],
                                     ctypes.byref(ex.c), None if shared is None else ctypes.byref(shared.c),
                                     _ptr(xn), _ptr(idx), _ptr(w), _ptr(y), _ptr(y32), _ptr(ws),
                                     ws.numel(), PATH[path], _stream(stream)))
    return y, y32, idx, w


def forward_noalloc(x, ex: Experts, idx, w, shared: Experts | None = None, want_f32=False,
                    out=None, stream=None):
    """forward() without a workspace: the library's static device scratch is used (see
    ts_moe_forward_noalloc in include/ts_moe.h for its size limit and sharing rules)."""
    import torch
    T, H = x.shape
    k = idx.shape[1]
    adt = {torch.float16: "f16", torch.bfloat16: "bf16"}[x.dtype]
    if out is None:
        y = torch.empty_like(x)
        y32 = torch.empty((T, H), dtype=torch.float32, device=x.device) if want_f32 else None
    else:
        y, y32 = out
    check(lib().ts_moe_forward_noalloc(_ptr(x), ADT[adt], T, ctypes.byref(ex.c), _ptr(idx),
                                       _ptr(w), k,
                                       None if shared is None else ctypes.byref(shared.c),
                                       _ptr(y), _ptr(y32), _stream(stream)))
    return y, y32


PHASES = ("route_list", "experts_phase1", "shared_phase1", "experts_phase2", "shared_phase2",
          "combine", "router", "gemma_tail")


def set_phase_events(events):
    """Register torch.cuda.Event objects (timing enabled) recorded after each forward phase
    (see PHASES); None clears."""
    if not events:
        check(lib().ts_moe_set_phase_events(None, 0))
        return
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(ev.cuda_event) for ev in events])
    check(lib().ts_moe_set_phase_events(arr, len(events)))


def set_wait_test(mode):
    """1: the next forward() on this thread withholds its GEMV phase-1 launch's first weight
    copy, so a bounded wait runs out and the device status reports TS_ERR_TIMEOUT (test use)."""
    check(lib().ts_moe_set_wait_test(int(mode)))


def device_status(ws, stream=None):
    code = ctypes.c_int32(0)
    check(lib().ts_moe_device_status(_ptr(ws), ctypes.byref(code), _stream(stream)))
    return code.value


def noalloc_device_status(stream=None):
    """Reads and clears the status word of the scratch forward_noalloc uses on this device."""
    code = ctypes.c_int32(0)
    check(lib().ts_moe_noalloc_device_status(ctypes.byref(code), _stream(stream)))
    return code.value
