"""ts_moe_route_forward: the router and the experts in one call.  Whether or not the router
launch also does the block-scaled decode kernels' prep (their x image and counters), idx and w
are the bits ts_moe_router_route writes (the router's fixed summation order), and y / y_f32 are
the bits ts_moe_forward writes for them (gpt-oss routed-expert pass: "THE BIAS, BEFORE THE
TOP-K"; slot order = router rank)."""
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routed_logits_gb300 import synth
from tests._helpers import (bits16, check_outputs, flip_allowance, gpu_layer, kappa_for, oracle_layer,
                            oracle_route, to_device)

pytestmark = pytest.mark.gpu
NTHREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _moe():
    import mixture_experts_routed_logits_gb300 as moe
    return moe


# (config, T, shapes, path, cfg override): the first six take the decode kernels, whose prep
# the router launch then does; the rest run the forward's own launches after the router
CASES = [
    (2, 8, None, "auto", None),                                      # gpt-oss decode T=8
    (2, 4, dict(H=512, I=384, E=8, k=4), "gemm", None),
    (3, 8, None, "auto", None),                                      # skewed routing
    (2, 3, dict(H=256, I=256, E=16, k=4), "gemm", dict(mode="sigmoid_biased")),
    (2, 5, dict(H=256, I=256, E=8, k=2), "gemm", dict(mode="softmax_k_scaled")),
    (2, 6, dict(H=416, I=256, E=8, k=2), "gemm", dict(rmsnorm=True)),  # RMSNorm rows, ragged K stage
    (2, 1, None, "auto", None),                                      # T=1: the GEMV path
    (4, 8, dict(H=256, I=128, E=16, k=4, shared_I=64), "auto", None),  # RMSNorm + INT4 + shared
    (2, 16, dict(H=256, I=256, E=8, k=4), "auto", None),             # T > 8: grouped GEMM
]


def _ids(case):
    cfg, T, sh, path, over = case
    return (f"cfg{cfg}-T{T}-" + ("full" if sh is None else "x".join(f"{k}{v}" for k, v in sh.items()))
            + f"-{path}" + ("".join(f"-{k}{'' if v is True else v}" for k, v in over.items()) if over else ""))


def _layer(cfg, T, shapes, over):
    dev = "cuda" if shapes is None else "cpu"
    L = synth.make_layer(cfg, T=T, shapes=shapes, device=dev)
    if over:
        L["cfg"] = dict(L["cfg"], **over)
        if over.get("mode") == "softmax_k_scaled" and L["scale"] is None:
            g = torch.Generator().manual_seed(11)
            L["scale"] = (0.5 + torch.rand(L["cfg"]["E"], generator=g)).float()
    return L, to_device(L, "cuda")


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_route_forward_equals_router_then_forward(case):
    moe = _moe()
    cfg, T, shapes, path, mode = case
    L, D = _layer(cfg, T, shapes, mode)
    c = L["cfg"]
    ex, sh = gpu_layer(D)
    kw = dict(mode=c["mode"], router_bias=D["router_bias"], per_expert_scale=D["scale"], rmsnorm=c["rmsnorm"])
    idx0, w0, xn0, _ = moe.router_route(D["x"], D["Wr"], c["k"], **kw)
    ws = moe.alloc_workspace(T, c["k"], ex, sh)
    y0, y32_0 = moe.forward(xn0 if c["rmsnorm"] else D["x"], ex, idx0, w0, shared=sh, want_f32=True,
                            ws=ws, path=path)
    y0, y32_0 = y0.clone(), y32_0.clone()
    ws2 = moe.alloc_workspace(T, c["k"], ex, sh)
    y1, y32_1, idx1, w1 = moe.route_forward(D["x"], D["Wr"], c["k"], ex, shared=sh, want_f32=True,
                                             ws=ws2, path=path, **kw)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0 and moe.device_status(ws2) == 0
    assert torch.equal(idx1, idx0)
    assert torch.equal(w1.view(torch.int32), w0.view(torch.int32))
    assert torch.equal(y1.view(torch.int16), y0.view(torch.int16))
    assert torch.equal(y32_1.view(torch.int32), y32_0.view(torch.int32))


@pytest.mark.parametrize("case", [CASES[0], CASES[2]], ids=_ids)
def test_route_forward_parity_with_the_oracle(case):
    """The folded decode call against the plain oracle: routes bit-exact, outputs within the
    stated tolerance."""
    moe = _moe()
    cfg, T, shapes, path, mode = case
    L, D = _layer(cfg, T, shapes, mode)
    c = L["cfg"]
    ex, sh = gpu_layer(D)
    y, y32, idx, w = moe.route_forward(D["x"], D["Wr"], c["k"], ex, mode=c["mode"], router_bias=D["router_bias"],
                                       per_expert_scale=D["scale"], want_f32=True, path=path)
    torch.cuda.synchronize()
    xb = bits16(L["x"])
    _, _, oidx, ow = oracle_route(L, xb)
    assert np.array_equal(idx.cpu().numpy(), oidx)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=1e-6, atol=0)
    oex, _ = oracle_layer(L)
    oy, oy32, _ = oracle.moe_forward(xb, c["adt"], oex, oidx, ow, nthreads=NTHREADS)
    allow, _ = flip_allowance(L, oex, None, oracle.adt_bits_to_f64(xb, c["adt"]), oidx, ow, c["adt"],
                              kappa=kappa_for(c, T, path), nthreads=NTHREADS)
    check_outputs(oracle.adt_bits_to_f64(bits16(y), c["adt"]), y32.double().cpu().numpy(),
                  oracle.adt_bits_to_f64(oy, c["adt"]), oy32.astype(np.float64), c["adt"], allow=allow)


def test_route_forward_validates_its_router_arguments():
    moe = _moe()
    L, D = _layer(2, 4, dict(H=256, I=256, E=8, k=4), None)
    c = L["cfg"]
    ex, _ = gpu_layer(D)
    with pytest.raises(moe.TsMoeError):
        moe.route_forward(D["x"], D["Wr"], c["k"], ex, mode="softmax_k_scaled", per_expert_scale=None)
    with pytest.raises(moe.TsMoeError):
        moe.route_forward(D["x"], D["Wr"], 9, ex)        # k > E
