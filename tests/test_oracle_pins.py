"""Pins for the CPU oracle: each test checks it against something other than itself --
format definitions, closed forms, textbook/library routines, brute force and invariants
the source pages state.

Source pages (docs.rs, turbospark-runtime 0.3.0):
  gpt-oss routed-expert pass (src/families/gptoss/moe.rs), module header
  Gemma-4 batched routed prefill (src/families/gemma4/moe_batch.rs), module header + body
  Llama/Mixtral decode flow (src/families/llama/mod.rs), module header "one decoder layer"
"""
import math

import mpmath
import numpy as np
import pytest
import scipy.special
import torch

import oracle
from mixture_experts_routed_logits_gb300 import synth
from tests._helpers import E2M1_MAGNITUDES, bits16, np_dequant, oracle_experts

mpmath.mp.dps = 40


# ---------------------------------------------------------------- formats

def test_f16_round_trip_matches_numpy():
    L = oracle.lib()
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 5, 3000),
                           [0.0, -0.0, 65504.0, 65519.0, 65520.0, 2.0 ** -24, 2.0 ** -25,
                            3 * 2.0 ** -26, 1e-9]])
    for v in vals:
        with np.errstate(over="ignore"):       # values past 65520 round to inf on purpose
            ref = np.array([v], np.float64).astype(np.float16).view(np.uint16)[0]
        assert L.or_double_to_f16(float(v)) == ref, v
    for b in range(0, 65536, 7):
        ref = np.array([b], np.uint16).view(np.float16).astype(np.float64)[0]
        got = L.or_f16_to_double(b)
        assert (math.isnan(ref) and math.isnan(got)) or got == ref


def test_bf16_round_trip_matches_torch():
    L = oracle.lib()
    rng = np.random.default_rng(2)
    # f32-representable inputs: torch's f32 -> bf16 conversion rounds once (RNE)
    vals = (rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000)).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for v, r in zip(vals, ref):
        assert L.or_double_to_bf16(float(v)) == r, v
    for b in range(0, 65536, 5):
        t = torch.tensor([b], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double().item()
        got = L.or_bf16_to_double(b)
        assert (math.isnan(t) and math.isnan(got)) or got == t


def test_e2m1_table_exhaustive():
    # OCP MX v1.0, 5.3.3: E2M1 codes 0..7 -> 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign
    L = oracle.lib()
    for code in range(16):
        mag = E2M1_MAGNITUDES[code & 7]
        want = -mag if code & 8 else mag
        got = L.or_e2m1_value(code)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), code


def test_e8m0_scales():
    L = oracle.lib()
    for b, want in zip(range(119, 124), [2.0 ** -8, 2.0 ** -7, 2.0 ** -6, 2.0 ** -5, 2.0 ** -4]):
        assert L.or_e8m0_value(b) == want
    assert L.or_e8m0_value(127) == 1.0
    assert math.isnan(L.or_e8m0_value(255))


@pytest.mark.parametrize("fmt", ["f16", "bf16", "mxfp4", "int4"])
def test_weight_indexing_matches_vectorised_dequant(fmt):
    g = torch.Generator().manual_seed(11)
    E, H, I = 3, 64, 96
    w = synth.make_expert_weights(fmt, E, H, I, g, "cpu", bias_std=0.02)
    X = oracle_experts(w, fmt, "silu", E, H, I)
    L = oracle.lib()
    rng = np.random.default_rng(3)
    for mat, name, (R, K) in ((0, "gate", (I, H)), (1, "up", (I, H)), (2, "down", (H, I))):
        full = np_dequant(fmt, w[name], w[name + "_s"])
        assert full.shape == (E, R, K)
        for _ in range(300):
            e, r, c = int(rng.integers(E)), int(rng.integers(R)), int(rng.integers(K))
            assert L.or_weight(X.c, mat, e, r, c) == full[e, r, c]


def test_int4_closed_form():
    # w = q * scale + min for one group, every code
    E, H, I = 1, 32, 32
    codes = np.zeros((E, I, H // 2), np.uint8)
    codes[0, 0, :8] = [(2 * j) | ((2 * j + 1) << 4) for j in range(8)]   # q = 0..15 along K
    sm = np.zeros((E, I, 1, 2), np.float16)
    sm[0, 0, 0] = [0.00390625, -0.03125]                                   # exact f16 values
    zeros16 = np.zeros((E, H, I // 2), np.uint8)
    X = oracle.Experts("int4", "silu", E, H, I, codes, codes, zeros16, sm.view(np.uint16),
                       sm.view(np.uint16), np.zeros((E, H, 1, 2), np.uint16))
    L = oracle.lib()
    for q in range(16):
        assert L.or_weight(X.c, 0, 0, 0, q) == q * 0.00390625 - 0.03125


# ---------------------------------------------------------------- fixed-order sums

def test_dot32f_within_f32_error_bound_and_exact_on_integers():
    L = oracle.lib()
    rng = np.random.default_rng(4)
    for n in (32, 128, 2880, 4096):
        a = rng.standard_normal(n).astype(np.float32)
        b = rng.standard_normal(n).astype(np.float32)
        got = float(L.or_dot32f(oracle._p(a), oracle._p(b), n))
        exact = math.fsum(float(x) * float(y) for x, y in zip(a, b))
        bound = (n / 32 + 5) * 2.0 ** -24 * math.fsum(abs(float(x) * float(y)) for x, y in zip(a, b))
        assert abs(got - exact) <= bound
        ai = rng.integers(-8, 8, n).astype(np.float32)
        bi = rng.integers(-8, 8, n).astype(np.float32)
        assert float(L.or_dot32f(oracle._p(ai), oracle._p(bi), n)) == float(np.dot(
            ai.astype(np.int64), bi.astype(np.int64)))


def test_rmsnorm_matches_float64_formula():
    lay = synth.make_layer(4, T=3, shapes=dict(H=256, I=64, E=8, k=2, shared_I=64))
    x = bits16(lay["x"])
    xn = oracle.rmsnorm(x, "bf16", 1e-6)
    xd = oracle.bf16_bits_to_f64(x)
    r = 1.0 / np.sqrt(np.mean(xd * xd, axis=1, keepdims=True) + 1e-6)
    want = xd * r
    got = oracle.bf16_bits_to_f64(xn)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-30)


def test_router_logits_match_float64_matmul():
    lay = synth.make_layer(2, T=5, shapes=dict(H=320, I=64, E=12, k=3))
    x, Wr = bits16(lay["x"]), bits16(lay["Wr"])
    lg = oracle.router_logits(x, Wr, "bf16")
    xd, wd = oracle.bf16_bits_to_f64(x), oracle.bf16_bits_to_f64(Wr)
    exact = xd @ wd.T
    bound = (320 / 32 + 5) * 2.0 ** -24 * (np.abs(xd) @ np.abs(wd).T)
    assert np.all(np.abs(lg - exact) <= bound)


# ---------------------------------------------------------------- routing (a2)

def _brute_topk(keys, k):
    order = sorted(range(len(keys)), key=lambda e: (-keys[e], e))
    return order[:k]


def test_bias_before_topk_matches_brute_force_sort():
    # gpt-oss moe.rs module header: the bias is added to the logits before top-k sees them
    lay = synth.make_layer(2, T=64, shapes=dict(H=256, I=64))
    c = lay["cfg"]
    lg = oracle.router_logits(bits16(lay["x"]), bits16(lay["Wr"]), "bf16")
    b = lay["router_bias"].numpy()
    idx, w = oracle.route(lg, c["k"], "softmax_k", bias=b)
    for t in range(lg.shape[0]):
        keys = [float(np.float32(lg[t, e]) + np.float32(b[e])) for e in range(c["E"])]
        assert list(idx[t]) == _brute_topk(keys, c["k"])


def test_bias_after_topk_selects_different_experts():
    # negative control: adding the bias after the top-k "selects the wrong experts"
    lay = synth.make_layer(2, T=64, shapes=dict(H=256, I=64))
    k = lay["cfg"]["k"]
    lg = oracle.router_logits(bits16(lay["x"]), bits16(lay["Wr"]), "bf16")
    idx_before, _ = oracle.route(lg, k, "softmax_k", bias=lay["router_bias"].numpy())
    idx_after, _ = oracle.route(lg, k, "softmax_k", bias=None)
    differs = sum(set(a) != set(b) for a, b in zip(idx_before, idx_after))
    assert differs >= 16


def test_softmax_over_k_is_renormalised_full_softmax():
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((200, 32)).astype(np.float32) * 2
    b = rng.standard_normal(32).astype(np.float32) * 0.5
    for k in (1, 2, 4, 8, 32):
        idx, w = oracle.route(lg, k, "softmax_k", bias=b)
        keys = (lg + b).astype(np.float32).astype(np.float64)
        p = scipy.special.softmax(keys, axis=1)
        for t in range(lg.shape[0]):
            sel = idx[t]
            want = p[t, sel] / p[t, sel].sum()
            assert np.allclose(w[t], want, rtol=1e-6, atol=1e-7)
            assert abs(w[t].astype(np.float64).sum() - 1.0) <= 1e-6
            assert np.all(np.diff(keys[t, sel]) <= 0)   # slot order = rank order
        if k == 1:
            assert np.all(w == 1.0)


def test_scaled_mode_multiplies_weights_not_selection():
    rng = np.random.default_rng(6)
    lg = rng.standard_normal((50, 128)).astype(np.float32)
    sc = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    i0, w0 = oracle.route(lg, 8, "softmax_k")
    i1, w1 = oracle.route(lg, 8, "softmax_k_scaled", scale=sc)
    assert np.array_equal(i0, i1)
    assert np.allclose(w1, w0.astype(np.float64) * sc[i0], rtol=1e-6)


def test_sigmoid_biased_mode_brute_force():
    # MiniMax: selection on biased sigmoid scores, weights from the unbiased scores
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((60, 64)).astype(np.float32)
    b = (rng.standard_normal(64) * 0.1).astype(np.float32)
    idx, w = oracle.route(lg, 6, "sigmoid_biased", bias=b)
    s = scipy.special.expit(lg.astype(np.float64))
    for t in range(60):
        keys = list(s[t] + b)
        bf = _brute_topk(keys, 6)
        # brute force in float64 may order two keys closer than f32 resolution differently
        gap = sorted(keys, reverse=True)
        if min(abs(gap[i] - gap[i + 1]) for i in range(6)) > 1e-6:
            assert list(idx[t]) == bf
        assert np.allclose(w[t], s[t, idx[t]] / s[t, idx[t]].sum(), rtol=1e-6)


def test_route_ties_go_to_lower_expert_id():
    lg = np.zeros((1, 8), np.float32)
    lg[0, [2, 5, 6]] = 1.0
    idx, w = oracle.route(lg, 4, "softmax_k")
    assert list(idx[0]) == [2, 5, 6, 0]


# ---------------------------------------------------------------- route list (a3)

def test_build_routes_matches_stable_argsort():
    rng = np.random.default_rng(8)
    for T, E, k in ((1, 32, 4), (8, 128, 8), (512, 32, 4), (37, 5, 2)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        off, perm, inv = oracle.build_routes(idx, E)
        flat = idx.reshape(-1)
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
        assert np.array_equal(inv[perm], np.arange(T * k))


# ---------------------------------------------------------------- activations

@pytest.mark.parametrize("g", [-6.5, -1.0, -0.25, 0.0, 0.3, 1.0, 2.5, 9.0])
def test_silu_and_gelu_against_identities(g):
    L = oracle.lib()
    u = 1.75
    gm = mpmath.mpf(g)
    # silu(g) = g/2 * (1 + tanh(g/2))
    silu = gm / 2 * (1 + mpmath.tanh(gm / 2)) * u
    assert abs(L.or_act(0, g, u, 7.0, 1.702) - float(silu)) <= 1e-14 * max(1.0, abs(float(silu)))
    # 0.5*(1+tanh(z)) = sigmoid(2z)
    z = mpmath.sqrt(2 / mpmath.pi) * (gm + mpmath.mpf("0.044715") * gm ** 3)
    gelu = gm / (1 + mpmath.exp(-2 * z)) * u
    assert abs(L.or_act(1, g, u, 7.0, 1.702) - float(gelu)) <= 1e-14 * max(1.0, abs(float(gelu)))


def test_clamped_swiglu_spot_values():
    L = oracle.lib()
    alpha = mpmath.mpf(np.float32(1.702).item())

    def want(g, u):
        g = min(g, 7.0)
        u = max(-7.0, min(u, 7.0))
        return float(g / (1 + mpmath.exp(-alpha * g)) * (u + 1))
    for g in (-10.0, 0.0, 7.0, 10.0):
        for u in (-10.0, 0.0, 10.0):
            got = L.or_act(2, g, u, 7.0, np.float32(1.702).item())
            assert abs(got - want(g, u)) <= 1e-13 * max(1.0, abs(want(g, u)))
    # the clamp boundaries are exact: g above the limit behaves as g = limit
    assert L.or_act(2, 10.0, 3.0, 7.0, 1.702) == L.or_act(2, 7.0, 3.0, 7.0, 1.702)
    assert L.or_act(2, 1.0, 10.0, 7.0, 1.702) == L.or_act(2, 1.0, 7.0, 7.0, 1.702)
    assert L.or_act(2, 1.0, -10.0, 7.0, 1.702) == L.or_act(2, 1.0, -7.0, 7.0, 1.702)
    # u = -1 zeroes h: (u + 1) factor
    assert L.or_act(2, 3.0, -1.0, 7.0, 1.702) == 0.0


# ---------------------------------------------------------------- whole layer (a4..a7)

def _textbook_ffn(Wg, Wu, Wd, bg, bu, bd, x, act, round_h):
    g = Wg @ x + (bg if bg is not None else 0.0)
    u = Wu @ x + (bu if bu is not None else 0.0)
    if act == "silu":
        h = g / 2 * (1 + np.tanh(g / 2)) * u
    elif act == "gelu_tanh":
        z = np.sqrt(2 / np.pi) * (g + 0.044715 * g ** 3)
        h = g * scipy.special.expit(2 * z) * u
    else:
        gc = np.minimum(g, 7.0)
        uc = np.clip(u, -7.0, 7.0)
        h = gc * scipy.special.expit(np.float32(1.702).item() * gc) * (uc + 1)
    h = round_h(h)
    return Wd @ h + (bd if bd is not None else 0.0)


def _f16_round(v):
    return np.asarray(v, np.float64).astype(np.float16).astype(np.float64)


@pytest.mark.parametrize("fmt,act", [("f16", "silu"), ("mxfp4", "gptoss"), ("int4", "gelu_tanh")])
def test_single_expert_equals_one_gated_ffn(fmt, act):
    # the dense half of the llama flow: one gated FFN; E = 1, k = 1 must reduce to it
    E, H, I = 1, 64, 96
    g = torch.Generator().manual_seed(21)
    bias = 0.02 if fmt == "mxfp4" else None
    w = synth.make_expert_weights(fmt, E, H, I, g, "cpu", bias_std=bias)
    X = oracle_experts(w, fmt, act, E, H, I)
    x = (torch.randn((3, H), generator=g)).to(torch.float16)
    idx = np.zeros((3, 1), np.int32)
    wt = np.ones((3, 1), np.float32)
    y, yf, _ = oracle.moe_forward(bits16(x), "f16", X, idx, wt)
    dq = {n: np_dequant(fmt, w[n], w[n + "_s"])[0] for n in ("gate", "up", "down")}
    bb = {n: (None if w[n + "_b"] is None else w[n + "_b"][0].double().numpy())
          for n in ("gate", "up", "down")}
    for t in range(3):
        xt = x[t].double().numpy()
        e = _textbook_ffn(dq["gate"], dq["up"], dq["down"], bb["gate"], bb["up"], bb["down"], xt,
                          act, _f16_round)
        assert np.allclose(yf[t], e.astype(np.float32), rtol=2e-6, atol=1e-6)
        assert np.array_equal(y[t], yf[t].astype(np.float16).view(np.uint16))


def test_k_equals_E_is_dense_weighted_sum():
    lay = synth.make_layer(1, shapes=dict(k=8))
    c = lay["cfg"]
    E, H, I = c["E"], c["H"], c["I"]
    X = oracle_experts(lay["experts"], "f16", "silu", E, H, I)
    x = bits16(lay["x"])
    lg = oracle.router_logits(x, bits16(lay["Wr"]), "f16")
    idx, w = oracle.route(lg, E, "softmax_k")
    y, yf, _ = oracle.moe_forward(x, "f16", X, idx, w)
    p = scipy.special.softmax(lg.astype(np.float64), axis=1)
    dq = {n: np_dequant("f16", lay["experts"][n]) for n in ("gate", "up", "down")}
    xd = lay["x"].double().numpy()
    for t in range(c["T"]):
        dense = sum(p[t, e] * _textbook_ffn(dq["gate"][e], dq["up"][e], dq["down"][e], None, None,
                                            None, xd[t], "silu", _f16_round) for e in range(E))
        assert np.allclose(yf[t], dense, rtol=1e-5, atol=1e-6)


def test_zero_shared_expert_leaves_routed_sum_alone():
    lay = synth.make_layer(4, T=3, shapes=dict(H=128, I=64, E=16, k=4, shared_I=96))
    c = lay["cfg"]
    X = oracle_experts(lay["experts"], "int4", "gelu_tanh", c["E"], c["H"], c["I"])
    zero = {n: torch.zeros_like(v) if v is not None else None for n, v in lay["shared"].items()}
    S0 = oracle_experts(zero, "f16", "gelu_tanh", 1, c["H"], c["shared_I"])
    xn = oracle.rmsnorm(bits16(lay["x"]), "bf16")
    lg = oracle.router_logits(xn, bits16(lay["Wr"]), "bf16")
    idx, w = oracle.route(lg, c["k"], "softmax_k_scaled", scale=lay["scale"].numpy())
    y0, yf0, _ = oracle.moe_forward(xn, "bf16", X, idx, w, shared=None)
    y1, yf1, _ = oracle.moe_forward(xn, "bf16", X, idx, w, shared=S0)
    assert np.array_equal(yf0.view(np.uint32), yf1.view(np.uint32))
    assert np.array_equal(y0, y1)
    # and a non-zero shared expert is the seed of the combine
    S = oracle_experts(lay["shared"], "f16", "gelu_tanh", 1, c["H"], c["shared_I"])
    y2, yf2, _ = oracle.moe_forward(xn, "bf16", S, np.zeros((3, 1), np.int32),
                                    np.ones((3, 1), np.float32))
    _, yf3, _ = oracle.moe_forward(xn, "bf16", X, idx, w, shared=S)
    assert np.allclose(yf3, yf0.astype(np.float64) + yf2, rtol=1e-5, atol=1e-6)


def test_whole_layer_tiny_brute_force():
    # T=1, H=32, I=32, E=4: everything in float64 without intermediate rounding
    lay = synth.make_layer(2, T=1, shapes=dict(H=32, I=32, E=4, k=2))
    c = lay["cfg"]
    X = oracle_experts(lay["experts"], "mxfp4", "gptoss", 4, 32, 32)
    x = bits16(lay["x"])
    lg = oracle.router_logits(x, bits16(lay["Wr"]), "bf16")
    b = lay["router_bias"].numpy()
    idx, w = oracle.route(lg, 2, "softmax_k", bias=b)
    y, yf, _ = oracle.moe_forward(x, "bf16", X, idx, w)
    xd = lay["x"].double().numpy()[0]
    keys = xd @ lay["Wr"].double().numpy().T + b.astype(np.float64)
    sel = np.argsort(-keys, kind="stable")[:2]
    assert list(sel) == list(idx[0])
    p = np.exp(keys[sel] - keys[sel].max())
    p /= p.sum()
    ex = lay["experts"]
    dq = {n: np_dequant("mxfp4", ex[n], ex[n + "_s"]) for n in ("gate", "up", "down")}
    bb = {n: ex[n + "_b"].double().numpy() for n in ("gate", "up", "down")}
    ref = sum(p[s] * _textbook_ffn(dq["gate"][e], dq["up"][e], dq["down"][e], bb["gate"][e],
                                   bb["up"][e], bb["down"][e], xd, "gptoss", lambda v: v)
              for s, e in enumerate(sel))
    # the oracle rounds h to bf16 (2^-9 relative) -> compare within that
    err = np.linalg.norm(yf[0] - ref) / np.linalg.norm(ref)
    assert err < 4e-3


def test_slot_order_changes_bits_only_within_rounding():
    lay = synth.make_layer(2, T=4, shapes=dict(H=64, I=64, E=8, k=4))
    X = oracle_experts(lay["experts"], "mxfp4", "gptoss", 8, 64, 64)
    x = bits16(lay["x"])
    lg = oracle.router_logits(x, bits16(lay["Wr"]), "bf16")
    idx, w = oracle.route(lg, 4, "softmax_k", bias=lay["router_bias"].numpy())
    _, yf, _ = oracle.moe_forward(x, "bf16", X, idx, w)
    rev = np.ascontiguousarray(idx[:, ::-1])
    _, yr, _ = oracle.moe_forward(x, "bf16", X, rev, np.ascontiguousarray(w[:, ::-1]))
    assert np.allclose(yf, yr, rtol=1e-5, atol=1e-6)
    assert not np.array_equal(yf.view(np.uint32), yr.view(np.uint32))


def test_hand_example_closed_form():
    # H = I = 32, one expert, f16.  x = e_0, W_g[i][0] = 1, W_u[i][0] = 2, W_d[j][i] = 1/32 for
    # i < 32: g = 1, u = 2, h = silu(1)*2 = 2/(1+e^-1) rounded to f16, e_j = sum_i h/32 = h.
    H = I = 32
    Wg = np.zeros((1, I, H), np.float16)
    Wg[0, :, 0] = 1.0
    Wu = np.zeros((1, I, H), np.float16)
    Wu[0, :, 0] = 2.0
    Wd = np.full((1, H, I), 1.0 / 32, np.float16)
    X = oracle.Experts("f16", "silu", 1, H, I, Wg, Wu, Wd)
    x = np.zeros((1, H), np.float16)
    x[0, 0] = 1.0
    y, yf, _ = oracle.moe_forward(x, "f16", X, np.zeros((1, 1), np.int32),
                                  np.ones((1, 1), np.float32))
    h = float(np.float16(float(2 / (1 + mpmath.exp(-1)))))   # 1.462117... -> f16 1.4619140625
    assert h == 1.4619140625
    assert np.all(yf[0] == np.float32(h))


# ---------------------------------------------------------------- Gemma sandwich tail
# ([gemma4/moe_batch] routed prefill: rms-norm the routed output with
# post_feedforward_layernorm_2, add it to the dense branch h1, rms-norm that with
# post_feedforward_layernorm, add it to the residual x, multiply x by the layer scalar)

def _adt_bits(a, adt):
    t = torch.from_numpy(np.asarray(a, np.float32))
    t = t.to(torch.bfloat16 if adt == "bf16" else torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _tail_inputs(adt, T=3, H=256, seed=0):
    rng = np.random.default_rng(seed)
    y = _adt_bits(rng.standard_normal((T, H)) * 3.0, adt)
    h1 = _adt_bits(rng.standard_normal((T, H)), adt)
    x = _adt_bits(rng.standard_normal((T, H)) * 2.0, adt)
    w2 = _adt_bits(1.0 + 0.1 * rng.standard_normal(H), "bf16")
    w1 = _adt_bits(1.0 + 0.1 * rng.standard_normal(H), "bf16")
    return y, h1, x, w2, w1


@pytest.mark.parametrize("adt", ["bf16", "f16"])
def test_tail_with_unit_weights_is_two_plain_rmsnorms(adt):
    # w = 1, h1 = x = 0, scalar 1: y' = h1' = rms(y) and x' = rms(rms(y)), bit for bit, against
    # the separately pinned unweighted RMSNorm
    y = _tail_inputs(adt)[0]
    zero = np.zeros_like(y)
    one = _adt_bits(np.ones(y.shape[1]), "bf16")
    yo, ho, xo = oracle.gemma_tail(y, zero, zero, one, one, adt, 1.0)
    r1 = oracle.rmsnorm(y, adt)
    assert np.array_equal(yo, r1)
    assert np.array_equal(ho, r1)
    assert np.array_equal(xo, oracle.rmsnorm(r1, adt))


@pytest.mark.parametrize("adt", ["bf16", "f16"])
def test_tail_power_of_two_weight_and_scalar_scale_exactly(adt):
    y, h1, x, w2, w1 = _tail_inputs(adt, seed=1)
    H = y.shape[1]
    one = _adt_bits(np.ones(H), "bf16")
    two = _adt_bits(np.full(H, 2.0), "bf16")
    base = oracle.gemma_tail(y, h1, x, w2, w1, adt, 1.0)
    x4 = oracle.gemma_tail(y, h1, x, w2, w1, adt, 4.0)[2]
    assert np.array_equal(oracle.adt_bits_to_f64(x4, adt), 4.0 * oracle.adt_bits_to_f64(base[2], adt))
    y_one = oracle.gemma_tail(y, h1, x, one, w1, adt, 1.0)[0]
    y_two = oracle.gemma_tail(y, h1, x, two, w1, adt, 1.0)[0]
    assert np.array_equal(oracle.adt_bits_to_f64(y_two, adt), 2.0 * oracle.adt_bits_to_f64(y_one, adt))


@pytest.mark.parametrize("adt", ["bf16", "f16"])
def test_tail_with_zero_routed_output_normalises_the_dense_branch(adt):
    _, h1, x, w2, w1 = _tail_inputs(adt, seed=2)
    zero = np.zeros_like(h1)
    s = 0.75
    yo, ho, xo = oracle.gemma_tail(zero, h1, x, w2, w1, adt, s)
    assert not np.any(oracle.adt_bits_to_f64(yo, adt))
    assert np.array_equal(ho, h1)
    hd, xd = oracle.adt_bits_to_f64(h1, adt), oracle.adt_bits_to_f64(x, adt)
    wd = oracle.bf16_bits_to_f64(w1)
    f = hd / np.sqrt(np.mean(hd * hd, axis=1, keepdims=True) + 1e-6) * wd
    want = (xd + f) * s
    u = 2.0 ** (-7 if adt == "bf16" else -10)          # one unit in the last place, relative
    bound = (s * (np.abs(f) + np.abs(xd + f)) + np.abs(want)) * u + 1e-30
    assert np.all(np.abs(oracle.adt_bits_to_f64(xo, adt) - want) <= bound)
