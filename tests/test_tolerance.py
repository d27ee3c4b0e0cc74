"""Pins of the oracle's phase-1 pre-activation sums (or_expert_pre) and of the test-side
tolerance for the 16-bit rounding of h (tests/_helpers.flip_allowance), on the CPU."""
import numpy as np
import torch

import oracle
from mixture_experts_routed_logits_gb300 import synth
from tests import _helpers as hp
from tests._helpers import bits16, np_dequant, oracle_layer, oracle_route, round16


def test_round16_is_round_to_nearest_even_of_each_type():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 4, 20000),
                        [0.0, -0.0, 1.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -8]])
    assert np.array_equal(round16(v, "f16"), v.astype(np.float16).astype(np.float64))
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    # float64 -> float32 first is exact for these values' needs except at exact bf16 midpoints
    # of the double, which the constructed values avoid
    assert np.array_equal(round16(v, "bf16"), ref)


def _layer(cfg, shapes, T=3):
    L = synth.make_layer(cfg, T=T, shapes=shapes, device="cpu")
    c = L["cfg"]
    xb = bits16(L["x"])
    oxn, _, oidx, ow = oracle_route(L, xb)
    xin = oracle.adt_bits_to_f64(oxn if oxn is not None else xb, c["adt"])
    oex, osh = oracle_layer(L)
    return L, c, xin, oidx, ow, oex, osh


def test_expert_pre_against_an_independent_matmul():
    for cfg, shapes in [(2, dict(H=256, I=96, E=4, k=2)), (4, dict(H=128, I=64, E=4, k=2, shared_I=64)),
                        (5, dict(H=128, I=64, E=4, k=2))]:
        L, c, xin, oidx, ow, oex, _ = _layer(cfg, shapes)
        d = L["experts"]
        e = int(oidx[0, 0])
        wg = np_dequant(c["fmt"], d["gate"][e], None if d.get("gate_s") is None else d["gate_s"][e])
        wu = np_dequant(c["fmt"], d["up"][e], None if d.get("up_s") is None else d["up_s"][e])
        g, u, sg, su = oracle.expert_pre(oex, e, xin[0])
        bg = 0.0 if d.get("gate_b") is None else d["gate_b"][e].double().numpy()
        bu = 0.0 if d.get("up_b") is None else d["up_b"][e].double().numpy()
        assert np.allclose(g, wg @ xin[0] + bg, rtol=1e-12, atol=1e-12)
        assert np.allclose(u, wu @ xin[0] + bu, rtol=1e-12, atol=1e-12)
        assert np.allclose(sg, np.abs(wg) @ np.abs(xin[0]), rtol=1e-12)
        assert np.allclose(su, np.abs(wu) @ np.abs(xin[0]), rtol=1e-12)
        # the activation over the arrays is the oracle's scalar one, and its h before rounding
        h, _ = oracle.expert_ffn(oex, e, xin[0], c["adt"])
        assert np.array_equal(round16(oracle.act(oex, g, u), c["adt"]), h)


def test_flip_allowance_at_the_two_extremes(monkeypatch):
    L, c, xin, oidx, ow, oex, osh = _layer(2, dict(H=256, I=96, E=4, k=2))
    # no evaluation error: nothing is flagged (no h of this seed sits exactly on a midpoint)
    monkeypatch.setattr(hp, "ACT_REL", 0.0)
    allow, n = hp.flip_allowance(L, oex, osh, xin, oidx, ow, c["adt"], kappa=0.0)
    assert n == 0 and not allow.any()
    # an error far beyond any h: every element is flagged and the allowance of output j is
    # sum over slots w_s * sum_i |W_d[j, i]| * gap_i, computed here independently
    monkeypatch.setattr(hp, "ACT_REL", 0.0)
    allow, n = hp.flip_allowance(L, oex, osh, xin, oidx, ow, c["adt"], kappa=2.0 ** 40)
    assert n == xin.shape[0] * c["k"] * c["I"]
    d = L["experts"]
    for q in range(xin.shape[0]):
        ref = np.zeros(c["H"])
        for s in range(c["k"]):
            e = int(oidx[q, s])
            g, u, sg, su = oracle.expert_pre(oex, e, xin[q])
            dg, du = 2.0 ** 40 * 2.0 ** -24 * sg, 2.0 ** 40 * 2.0 ** -24 * su
            corners = [oracle.act(oex, g + a * dg, u + b * du) for a in (-1, 1) for b in (-1, 1)]
            h0 = oracle.act(oex, g, u)
            lo = np.minimum.reduce(corners + [h0])
            hi = np.maximum.reduce(corners + [h0])
            gap = np.abs(round16(hi, c["adt"]) - round16(lo, c["adt"]))
            wd = np.abs(np_dequant("mxfp4", d["down"][e], d["down_s"][e]))
            ref += ow[q, s] * (wd @ gap)
        assert np.allclose(allow[q], ref, rtol=1e-5)
