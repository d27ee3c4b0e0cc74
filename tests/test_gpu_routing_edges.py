"""GPU parity of the routing step on the keys where several selections look plausible: exactly
equal keys (the tie rule decides), -0.0 against +0.0, and -inf logits.

The pages fix the selection as a top-k on the raw biased logits, slot order = the router's
ranking (gpt-oss routed-expert pass, src/families/gptoss/moe.rs, module header); they leave ties
open, and both sides read them the same way: larger key first, equal keys to the lower expert
id, -0.0 equal to +0.0.  Indices are compared bit-exactly with the oracle, weights to 1e-6.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _moe():
    import mixture_experts_routed_logits_gb300 as moe
    return moe


# exactly representable values: sums with the dyadic biases below are exact, so equal
# (logit, bias) pairs and distinct pairs with equal sums both give exactly equal keys
_VALS = np.array([-3.0, -1.5, -0.5, -0.0, 0.0, 0.25, 1.0, 2.0, -np.inf], np.float32)
_BIAS = np.array([-0.5, -0.0, 0.0, 0.25, 0.5], np.float32)


def _edge_logits(T, E, rng):
    lg = rng.choice(_VALS, size=(T, E)).astype(np.float32)
    lg[:, 0] = np.where(np.isinf(lg[:, 0]), 1.0, lg[:, 0])          # a finite key in every row
    lg[1, :] = 0.5                                                  # every key equal
    lg[2, :] = -np.inf                                              # one finite key, rest -inf
    lg[2, E // 2] = 0.0
    lg[3, :] = np.where(np.arange(E) % 2 == 0, -0.0, 0.0)           # alternating signed zeros
    lg[4, :] = np.where(np.arange(E) % 3 == 0, 2.0, -np.inf)        # ties among the finite keys
    return lg


def _check(idx, w, oidx, ow):
    gi, gw = idx.cpu().numpy(), w.cpu().numpy()
    assert np.array_equal(gi, oidx), np.argwhere(gi != oidx)[:8]
    assert np.allclose(gw, ow, rtol=1e-6, atol=1e-7), float(np.abs(gw - ow).max())


@pytest.mark.parametrize("E,k", [(8, 2), (8, 8), (32, 4), (256, 8), (256, 16)])
@pytest.mark.parametrize("mode,with_bias", [("softmax_k", False), ("softmax_k", True),
                                            ("softmax_k_scaled", False), ("sigmoid_biased", False)])
def test_route_equal_keys_signed_zeros_and_minus_inf(E, k, mode, with_bias):
    moe = _moe()
    rng = np.random.default_rng(E * 131 + k * 7 + len(mode) + with_bias)
    T = 96
    lg = _edge_logits(T, E, rng)
    bias = rng.choice(_BIAS, size=E).astype(np.float32) if with_bias else None
    scale = (rng.uniform(0.5, 1.5, size=E).astype(np.float32) if mode == "softmax_k_scaled" else None)
    oidx, ow = oracle.route(lg, k, mode, bias=bias, scale=scale)
    # the constructed rows must really hold ties at the selection boundary
    keys = lg + (bias if bias is not None else 0.0)
    srt = np.sort(keys, axis=1)[:, ::-1]
    if k < E:
        assert np.sum(srt[:, k - 1] == srt[:, k]) >= 8
    dev = lambda a: None if a is None else torch.from_numpy(a).cuda()
    idx, w = moe.route(dev(lg), k, mode=mode, router_bias=dev(bias), per_expert_scale=dev(scale))
    torch.cuda.synchronize()
    _check(idx, w, oidx, ow)


@pytest.mark.parametrize("E,k,T", [(8, 2, 8), (32, 4, 8), (32, 4, 100), (256, 8, 8), (256, 16, 70)])
def test_router_route_ties_from_duplicated_router_rows(E, k, T):
    """Through the fused router kernel: duplicated rows of W_r give bit-identical logits, so
    the top-k meets exactly equal keys (with equal biases, or none); an all-zero row gives the
    logit +0.0 and, with a -0.0 bias, the key +0.0."""
    moe = _moe()
    H = 256
    rng = np.random.default_rng(E * 17 + T)
    base = rng.standard_normal((max(2, E // 4), H)).astype(np.float32) * 0.05
    rows = rng.integers(0, base.shape[0], size=E)
    Wr = torch.from_numpy(base[rows]).to(torch.bfloat16)
    Wr[E - 1] = 0.0
    ub = rng.choice(_BIAS, size=base.shape[0]).astype(np.float32)
    bias = ub[rows].copy()
    bias[E - 1] = -0.0
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    wb = Wr.view(torch.int16).numpy().view(np.uint16)
    olg = oracle.router_logits(xb, wb, "bf16")
    for b in (None, bias):
        oidx, ow = oracle.route(olg, k, "softmax_k", bias=b)
        idx, w, _, lg = moe.router_route(x.cuda(), Wr.cuda(), k,
                                         router_bias=None if b is None else torch.from_numpy(b).cuda(),
                                         want_logits=True)
        torch.cuda.synchronize()
        assert np.array_equal(lg.cpu().numpy().view(np.uint32), olg.view(np.uint32))
        # duplicated rows put exactly equal keys at the selection boundary of some tokens
        keys = olg + (0.0 if b is None else b)
        srt = np.sort(keys, axis=1)[:, ::-1]
        assert np.sum(srt[:, k - 1] == srt[:, k]) >= 1
        _check(idx, w, oidx, ow)
