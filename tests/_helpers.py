"""Test-side helpers: turn synth layers into oracle / library arguments.

Test infrastructure: may import ``oracle`` (the CPU oracle) and the product
package, never the other way round.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

# OCP Microscaling Formats (MX) v1.0, section 5.3.3, FP4 E2M1 encodings:
# magnitudes of codes 0..7; codes 8..15 are the same magnitudes with the sign bit set.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_experts(w: dict, fmt: str, act: str, E: int, H: int, I: int,
                   limit=7.0, alpha=1.702) -> oracle.Experts:
    def arr(t):
        if t is None:
            return None
        t = t.detach().contiguous().cpu()
        if t.dtype in (torch.float16, torch.bfloat16):
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return oracle.Experts(fmt, act, E, H, I, arr(w["gate"]), arr(w["up"]), arr(w["down"]),
                          arr(w.get("gate_s")), arr(w.get("up_s")), arr(w.get("down_s")),
                          arr(w.get("gate_b")), arr(w.get("up_b")), arr(w.get("down_b")),
                          limit=limit, alpha=alpha)


def np_dequant(fmt: str, codes, scales=None) -> np.ndarray:
    """Vectorised dequantisation of a canonical [E][R][K] matrix to float64.

    Written independently of the oracle's scalar ``or_weight`` so that an indexing
    or nibble-order slip in either shows up as a mismatch."""
    if fmt in ("f16", "bf16"):
        t = codes if isinstance(codes, torch.Tensor) else torch.from_numpy(codes)
        return t.detach().cpu().double().numpy()
    c = codes.detach().cpu().numpy() if isinstance(codes, torch.Tensor) else np.asarray(codes)
    lo = (c & 0x0F).astype(np.int64)
    hi = (c >> 4).astype(np.int64)
    q = np.stack([lo, hi], axis=-1).reshape(c.shape[:-1] + (c.shape[-1] * 2,))
    if fmt == "mxfp4":
        mag = np.array(E2M1_MAGNITUDES)[q & 7]
        val = np.where(q & 8, -mag, mag)
        s = scales.detach().cpu().numpy() if isinstance(scales, torch.Tensor) else scales
        sc = np.ldexp(1.0, s.astype(np.int64) - 127)
        return val * np.repeat(sc, 32, axis=-1)
    if fmt == "int4":
        sm = scales.detach().cpu().float().double().numpy()  # [E][R][K/32][2]
        s = np.repeat(sm[..., 0], 32, axis=-1)
        m = np.repeat(sm[..., 1], 32, axis=-1)
        return q.astype(np.float64) * s + m
    raise ValueError(fmt)


# ------------------------------------------------------------------ layer -> oracle + GPU
def oracle_layer(L):
    """Oracle descriptors for a synth layer (tensors may live on any device)."""
    c = L["cfg"]
    ex = oracle_experts(L["experts"], c["fmt"], c["act"], c["E"], c["H"], c["I"])
    sh = (oracle_experts(L["shared"], "f16", c["act"], 1, c["H"], c["shared_I"])
          if L.get("shared") is not None else None)
    return ex, sh


def to_device(L, device="cuda"):
    """A copy of a synth layer with every tensor moved to `device`."""
    out = {}
    for key, v in L.items():
        if isinstance(v, torch.Tensor):
            out[key] = v.to(device)
        elif isinstance(v, dict) and key in ("experts", "shared"):
            out[key] = {n: (t.to(device) if isinstance(t, torch.Tensor) else t) for n, t in v.items()}
        else:
            out[key] = v
    return out


def gpu_layer(L):
    """Library Experts (packed where needed) for a synth layer whose tensors are on the GPU."""
    import mixture_experts_routed_logits_gb300 as moe
    c = L["cfg"]
    ex = moe.Experts.from_canonical(c["fmt"], c["act"], L["experts"])
    sh = (moe.Experts.from_canonical("f16", c["act"], L["shared"])
          if L.get("shared") is not None else None)
    return ex, sh


def oracle_route(L, x_bits):
    """Oracle steps a0-a2 for a layer: (xn bits or None, logits, idx, w)."""
    c = L["cfg"]
    xn = oracle.rmsnorm(x_bits, c["adt"], 1e-6) if c["rmsnorm"] else None
    lg = oracle.router_logits(xn if xn is not None else x_bits, bits16(L["Wr"]), c["adt"])
    bias = None if L["router_bias"] is None else L["router_bias"].cpu().numpy()
    scale = None if L["scale"] is None else L["scale"].cpu().numpy()
    idx, w = oracle.route(lg, c["k"], c["mode"], bias=bias, scale=scale)
    return xn, lg, idx, w


def parity_metrics(y_gpu_f64, y_ref_f64):
    d = np.abs(y_gpu_f64 - y_ref_f64)
    rel = np.linalg.norm(y_gpu_f64 - y_ref_f64) / max(np.linalg.norm(y_ref_f64), 1e-30)
    return float(d.max()), float(rel)


def ulp16(v, adt):
    """One unit in the last place of the 16-bit activation type at |v| (numpy, float64)."""
    v = np.abs(np.asarray(v, np.float64))
    p = 8 if adt == "bf16" else 11
    emin = -126 if adt == "bf16" else -14
    e = np.floor(np.log2(np.maximum(v, 2.0 ** emin)))
    return np.ldexp(1.0, (e - (p - 1)).astype(np.int64))


def check_outputs(y_gpu_f64, y32_gpu_f64, y_ref_bits_f64, y32_ref_f64, adt, max_abs=2e-2, rel_l2=1e-3,
                  flip_bound=None):
    """The parity bar: f32 outputs within max-abs and rel-L2; 16-bit outputs within the same
    bars, except that an element may differ by one unit in the last place of the 16-bit type
    (both sides round an f32 sum; sums a hair apart can straddle a rounding boundary).

    flip_bound: both sides also round the intermediate h to 16 bits; where an h element sits
    next to a rounding boundary the two sides can round it to neighbouring values, which moves
    the outputs that depend on it by up to ulp16(h) * |W_d| -- one such flip shifts a whole
    output row of that token.  With flip_bound set, elements beyond max_abs are accepted if they
    are at most 2 % of the outputs and each stays within flip_bound; rel-L2 is never relaxed."""
    def within(a, b, extra):
        d = np.abs(a - b)
        allow = np.maximum(max_abs, extra)
        bad = d > allow
        if flip_bound is not None and bad.any():
            ok = bad.sum() <= max(1, int(0.02 * d.size)) and np.all(d[bad] <= flip_bound)
            return ok, float(d.max()), int(bad.sum())
        return not bad.any(), float(d.max()), int(bad.sum())
    ok, dmax, nbad = within(y32_gpu_f64, y32_ref_f64, 0.0)
    rel = np.linalg.norm(y32_gpu_f64 - y32_ref_f64) / max(np.linalg.norm(y32_ref_f64), 1e-30)
    assert ok and rel <= rel_l2, ("f32 outputs", dmax, nbad, rel)
    ok, dmax16, nbad16 = within(y_gpu_f64, y_ref_bits_f64, ulp16(y_ref_bits_f64, adt))
    assert ok, ("16-bit outputs", dmax16, nbad16)
    rel16 = np.linalg.norm(y_gpu_f64 - y_ref_bits_f64) / max(np.linalg.norm(y_ref_bits_f64), 1e-30)
    assert rel16 <= rel_l2, ("16-bit rel-L2", rel16)
    return dmax, rel


def h_flip_bound(oex, xin_f64_rows, idx_rows, adt, down_f64_absmax):
    """2 * ulp16(max |h|) * max |W_d|: the most two neighbouring-value roundings of h can move
    one output (routing weights are at most 1).  max |h| from the oracle's own h of the routes."""
    import oracle
    hmax = 0.0
    for xrow, sel in zip(xin_f64_rows, idx_rows):
        for e in sel:
            h, _ = oracle.expert_ffn(oex, int(e), xrow, adt)
            hmax = max(hmax, float(np.abs(h).max()))
    return 2.0 * float(ulp16(hmax, adt)) * down_f64_absmax


def weight_absmax(fmt, codes, scales=None):
    """An upper bound of |W| over a canonical weight tensor, computed without dequantising it."""
    if fmt in ("f16", "bf16"):
        return float(codes.abs().max().item())
    if fmt == "mxfp4":
        return 6.0 * 2.0 ** (int(scales.max().item()) - 127)
    sm = scales.float()
    return float(torch.maximum(sm[..., 1].abs(), (15.0 * sm[..., 0] + sm[..., 1]).abs()).max().item())
