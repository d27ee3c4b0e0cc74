"""GPU parity of the block-scaled decode kernels (T <= 8 tokens, MXFP4 experts with bf16
activations, path "gemm"): the route tables built inside the kernel, the stream-K split of the
(touched expert, row block, K stage) units, the per-row activation scale and the fused
slot-ordered combine, against the CPU oracle (gpt-oss routed-expert pass: the decode pair of
phases and the slot order of the reduction)."""
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routed_logits_gb300 import synth
from tests._helpers import (bits16, check_outputs, flip_allowance, gpu_layer, kappa_for, oracle_layer, oracle_route,
                            to_device)

pytestmark = pytest.mark.gpu
NTHREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _moe():
    import mixture_experts_routed_logits_gb300 as moe
    return moe


CASES = [
    (2, 1, dict(H=512, I=384, E=8, k=4)),             # fewer units than SMs: every tile split
    (2, 3, dict(H=640, I=448, E=8, k=4)),             # ragged K stage and row blocks, odd T
    (2, 8, dict(H=256, I=256, E=128, k=8)),           # 64 routes, up to 64 touched experts
    (3, 5, dict(H=1024, I=768, E=16, k=4)),           # skewed routing: experts shared by tokens
    (2, 8, dict(H=2880, I=2880, E=32, k=4)),          # full gpt-oss widths, 32 experts
    (2, 1, None),                                     # gpt-oss-120b decode T=1
    (2, 8, None),                                     # gpt-oss-120b decode T=8
    (3, 8, None),                                     # gpt-oss shapes with skewed routing
]


def _ids(case):
    cfg, T, sh = case
    return f"cfg{cfg}-T{T}-" + ("full" if sh is None else "x".join(f"{k}{v}" for k, v in sh.items()))


def _make(cfg, T, shapes):
    dev = "cuda" if shapes is None else "cpu"
    L = synth.make_layer(cfg, T=T, shapes=shapes, device=dev)
    return L, to_device(L, "cuda")


def _check(L, D, y, y32, T):
    c = L["cfg"]
    xb = bits16(L["x"])
    _, _, oidx, ow = oracle_route(L, xb)
    oex, osh = oracle_layer(L)
    oy, oy32, _ = oracle.moe_forward(xb, c["adt"], oex, oidx, ow, shared=osh, nthreads=NTHREADS)
    allow, _ = flip_allowance(L, oex, osh, oracle.adt_bits_to_f64(xb, c["adt"]), oidx, ow, c["adt"],
                              kappa=kappa_for(c, T, "gemm"), nthreads=NTHREADS)
    check_outputs(oracle.adt_bits_to_f64(bits16(y), c["adt"]), y32.double().cpu().numpy(),
                  oracle.adt_bits_to_f64(oy, c["adt"]), oy32.astype(np.float64), c["adt"], allow=allow)
    return oidx, ow


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_mx_decode_parity(case):
    moe = _moe()
    cfg, T, shapes = case
    L, D = _make(cfg, T, shapes)
    c = L["cfg"]
    _, _, oidx, ow = oracle_route(L, bits16(L["x"]))
    ex, sh = gpu_layer(D)
    ws = moe.alloc_workspace(T, c["k"], ex, sh)
    y, y32 = moe.forward(D["x"], ex, torch.from_numpy(oidx).cuda(), torch.from_numpy(ow).cuda(),
                         shared=sh, want_f32=True, ws=ws, path="gemm")
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    _check(L, D, y, y32, T)


def test_mx_decode_with_shared_expert():
    """A shared expert's output seeds the fused combine of the second decode kernel."""
    moe = _moe()
    T = 4
    L, D = _make(2, T, dict(H=256, I=256, E=8, k=4, shared_I=128))
    c = L["cfg"]
    _, _, oidx, ow = oracle_route(L, bits16(L["x"]))
    ex, sh = gpu_layer(D)
    assert sh is not None
    ws = moe.alloc_workspace(T, c["k"], ex, sh)
    y, y32 = moe.forward(D["x"], ex, torch.from_numpy(oidx).cuda(), torch.from_numpy(ow).cuda(),
                         shared=sh, want_f32=True, ws=ws, path="gemm")
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    _check(L, D, y, y32, T)


@pytest.mark.parametrize("case", [(2, 8, None), (2, 2, dict(H=512, I=384, E=8, k=4))], ids=_ids)
def test_mx_decode_deterministic_and_reusable(case):
    """Parts of split tiles are summed in K order and the combine runs in slot order, so three
    calls on one workspace give the same bits; the counters the kernels leave behind serve the
    next call."""
    moe = _moe()
    cfg, T, shapes = case
    L, D = _make(cfg, T, shapes)
    c = L["cfg"]
    ex, sh = gpu_layer(D)
    idx, w, _, _ = moe.router_route(D["x"], D["Wr"], c["k"], mode=c["mode"], router_bias=D["router_bias"])
    ws = moe.alloc_workspace(T, c["k"], ex, sh)
    outs = []
    for _ in range(3):
        y, y32 = moe.forward(D["x"], ex, idx, w, want_f32=True, ws=ws, path="gemm")
        outs.append((y.clone(), y32.clone()))
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    for y, y32 in outs[1:]:
        assert torch.equal(y.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(y32.view(torch.int32), outs[0][1].view(torch.int32))


def test_mx_decode_matches_the_gemv_path():
    """The decode kernels and the streaming GEMV kernels compute the same layer: their f32 sums
    agree to the f32 rounding of the two reduction orders."""
    moe = _moe()
    L, D = _make(2, 8, None)
    c = L["cfg"]
    ex, _ = gpu_layer(D)
    idx, w, _, _ = moe.router_route(D["x"], D["Wr"], c["k"], mode=c["mode"], router_bias=D["router_bias"])
    _, a32 = moe.forward(D["x"], ex, idx, w, want_f32=True, path="gemv")
    _, b32 = moe.forward(D["x"], ex, idx, w, want_f32=True, path="gemm")
    torch.cuda.synchronize()
    a, b = a32.double().cpu().numpy(), b32.double().cpu().numpy()
    rel = np.linalg.norm(a - b) / np.linalg.norm(a)
    assert np.abs(a - b).max() <= 2e-2 and rel <= 1e-3, rel


def test_mx_decode_reports_out_of_range_ids():
    """Expert ids outside 0..E-1 are left out of the route tables and reported through the
    device status word; the call completes and the next valid call is exact again."""
    moe = _moe()
    T = 4
    L, D = _make(2, T, dict(H=256, I=256, E=8, k=4))
    c = L["cfg"]
    _, _, oidx, ow = oracle_route(L, bits16(L["x"]))
    ex, sh = gpu_layer(D)
    ws = moe.alloc_workspace(T, c["k"], ex, sh)
    bad = oidx.copy()
    bad[1, 2] = c["E"] + 5
    bad[3, 0] = -2
    moe.forward(D["x"], ex, torch.from_numpy(bad).cuda(), torch.from_numpy(ow).cuda(), ws=ws, path="gemm")
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 1
    y, y32 = moe.forward(D["x"], ex, torch.from_numpy(oidx).cuda(), torch.from_numpy(ow).cuda(),
                         want_f32=True, ws=ws, path="gemm")
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    _check(L, D, y, y32, T)
