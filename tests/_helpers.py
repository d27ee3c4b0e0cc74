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
