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


def round16(v, adt):
    """Round float64 values to the nearest 16-bit value of the activation type (ties to even),
    returned as float64 (numpy; finite values within the type's range)."""
    v = np.asarray(v, np.float64)
    q = ulp16(v, adt)
    return np.round(v / q) * q


# f32 evaluation error of a phase-1 pre-activation, as a multiple kappa of 2^-24 * sum |w_c x_c|
# (the absolute sum of its products).  The products are exact on both sides (dequantised
# weights times 16-bit activations); the GPU adds them in f32 in blocked chains, so its error is
# a small multiple of the unit roundoff times the absolute sum.  Measured on GB300 over every
# sampled h element of the five configurations (the smallest kappa that names each element the
# GPU rounded differently from the oracle): at most 0.5 on the streaming GEMV path, at most 1 on
# the tensor-core path over dequantised MXFP4 weights and at most 4 on the tensor-core path with
# 16-bit weights (its K = 4096 reduction runs through 256 chained MMA steps).  kappa = 2 for the
# GEMV path and 8 for every tensor-core path keeps a margin of at least 2x.
KAPPA_GEMV = 2.0
KAPPA_TC = 8.0
KAPPA = KAPPA_GEMV


def kappa_for(cfg, T, path):
    """kappa of the expert path a call takes (the library's automatic choice for path="auto")."""
    tc_fmt = cfg["fmt"] == "mxfp4" or cfg["fmt"] == cfg["adt"]
    tc_shape = cfg["H"] % 64 == 0 and cfg["I"] % 64 == 0
    mx = cfg["fmt"] == "mxfp4" and cfg["adt"] == "bf16"
    # block-scaled decode kernels: "gemm" at T <= 8, "auto" at 3 <= T <= 8 (MXFP4 + bf16,
    # T*k <= 64, k <= 8, H <= 4096)
    mxd = (mx and T <= 8 and T * cfg["k"] <= 64 and cfg["k"] <= 8 and cfg["H"] <= 4096
           and (path == "gemm" or (path == "auto" and T >= 3)))
    tc = mxd or ((path in ("gemm", "gemm_dequant") or (path == "auto" and T > 8)) and (mx or (tc_fmt and tc_shape)))
    return KAPPA_TC if tc else KAPPA_GEMV
# f32 evaluation of the activation itself (expf / tanhf, a divide, two multiplies), relative
ACT_REL = 2.0 ** -20
# non-flip f32 error of an output beside the flips (down projection and combine in f32)
OUT_SLACK = 1e-3


def _abs_rows(fmt, codes_e, scales_e):
    """|W| of one expert matrix as float32 [R][K] (canonical layout)."""
    if fmt in ("f16", "bf16"):
        return codes_e.detach().cpu().float().abs().numpy()
    return np.abs(np_dequant(fmt, codes_e.detach().cpu(),
                             None if scales_e is None else scales_e.detach().cpu())).astype(np.float32)


def flip_allowance(L, oex, osh, xin_rows_f64, idx_rows, w_rows, adt, kappa=KAPPA, nthreads=1):
    """Per-output allowance [n, H] for the 16-bit rounding of h, from the oracle alone.

    Both sides round the phase-1 output h to the 16-bit activation type before the down
    projection.  For each h element the oracle's exact pre-activations g, u are widened by the
    f32 evaluation error (kappa * 2^-24 * sum|products|); if the activation over that box
    straddles a 16-bit rounding boundary, the element may round to either neighbour on the GPU.
    Such an element moves output j of its token by at most gap * |W_d[j, i]| * w (gap = the two
    roundings' distance); the allowance of output j is the sum over the flagged elements of
    every route of that token (and of the shared expert, weight 1).  Elements away from a
    boundary contribute nothing, so outputs of tokens without flagged elements keep the plain
    bar.  Returns (allowance, number of flagged elements)."""
    import concurrent.futures
    c = L["cfg"]
    H = c["H"]
    n = len(xin_rows_f64)
    allow = np.zeros((n, H), np.float64)
    jobs = []                                  # (expert set, expert id, row q, weight)
    for q in range(n):
        for s, e in enumerate(idx_rows[q]):
            jobs.append(("routed", int(e), q, float(w_rows[q][s])))
        if osh is not None:
            jobs.append(("shared", 0, q, 1.0))

    def gaps(job):
        which, e, q, _ = job
        ex = oex if which == "routed" else osh
        g, u, sg, su = oracle.expert_pre(ex, e, xin_rows_f64[q])
        dg, du = kappa * 2.0 ** -24 * sg, kappa * 2.0 ** -24 * su
        h0 = oracle.act(ex, g, u)
        lo, hi = h0.copy(), h0.copy()
        for a in (-1.0, 1.0):
            for b in (-1.0, 1.0):
                hc = oracle.act(ex, g + a * dg, u + b * du)
                lo, hi = np.minimum(lo, hc), np.maximum(hi, hc)
        lo -= ACT_REL * np.abs(h0)
        hi += ACT_REL * np.abs(h0)
        return np.abs(round16(hi, adt) - round16(lo, adt))

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, nthreads)) as pool:
        gap_list = list(pool.map(gaps, jobs))
    flagged = 0
    by_expert = {}
    for job, gp in zip(jobs, gap_list):
        if gp.any():
            flagged += int(np.count_nonzero(gp))
            by_expert.setdefault((job[0], job[1]), []).append((job[2], job[3], gp))
    for (which, e), items in by_expert.items():
        d = L["experts"] if which == "routed" else L["shared"]
        fmt = c["fmt"] if which == "routed" else "f16"
        wd = _abs_rows(fmt, d["down"][e], None if d.get("down_s") is None else d["down_s"][e])
        for q, wt, gp in items:
            nz = np.nonzero(gp)[0]
            allow[q] += wt * (wd[:, nz].astype(np.float64) @ gp[nz])
    return allow, flagged


def check_outputs(y_gpu_f64, y32_gpu_f64, y_ref_bits_f64, y32_ref_f64, adt, max_abs=2e-2, rel_l2=1e-3,
                  allow=None):
    """The parity bar: f32 outputs within max-abs and rel-L2; 16-bit outputs within the same
    bars, except that an element may differ by one unit in the last place of the 16-bit type
    (both sides round an f32 sum; sums a hair apart can straddle a rounding boundary).

    allow: per-output allowance from flip_allowance (the h elements next to a 16-bit rounding
    boundary, named by the oracle).  An output beyond max_abs is accepted only if its deviation
    is covered by its own allowance (plus OUT_SLACK for the f32 arithmetic beside it); rel-L2 is
    never relaxed."""
    def within(a, b, extra):
        d = np.abs(a - b)
        bar = np.maximum(max_abs, extra)
        if allow is not None:
            bar = np.maximum(bar, allow + OUT_SLACK + extra)
        bad = d > bar
        return not bad.any(), float(d.max()), int(bad.sum())
    ok, dmax, nbad = within(y32_gpu_f64, y32_ref_f64, 0.0)
    rel = np.linalg.norm(y32_gpu_f64 - y32_ref_f64) / max(np.linalg.norm(y32_ref_f64), 1e-30)
    assert ok and rel <= rel_l2, ("f32 outputs", dmax, nbad, rel)
    ok, dmax16, nbad16 = within(y_gpu_f64, y_ref_bits_f64, ulp16(y_ref_bits_f64, adt))
    assert ok, ("16-bit outputs", dmax16, nbad16)
    rel16 = np.linalg.norm(y_gpu_f64 - y_ref_bits_f64) / max(np.linalg.norm(y_ref_bits_f64), 1e-30)
    assert rel16 <= rel_l2, ("16-bit rel-L2", rel16)
    return dmax, rel
