"""ts_moe_forward_tail: the routed layer and the Gemma sandwich tail in one call (Gemma-4 batched
routed prefill: the per-token tail encoded right after the fused phase 2).  Decode sizes run the
tail inside the streaming GEMV's phase 2 (once every row tile is combined, CTA b takes tokens b,
b + grid, ...); larger calls launch it after the forward.  Either way every output is the bits of
ts_moe_forward_path followed by ts_moe_gemma_tail, and the tail's outputs are the oracle's tail
of the GPU's own y, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_routed_logits_gb300 import synth
from tests._helpers import bits16, gpu_layer, oracle_route, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _moe():
    import mixture_experts_routed_logits_gb300 as moe
    return moe


# (config, T, shapes, path): decode sizes take the fused tail (T * k <= 512 on the GEMV path)
CASES = [
    (4, 8, None, "auto"),                                         # Gemma decode T=8 (+ shared expert)
    (4, 1, dict(H=256, I=128, E=16, k=8, shared_I=64), "auto"),   # one token
    (4, 64, dict(H=512, I=256, E=32, k=8, shared_I=128), "auto"), # 512 routes: the largest fused call
    (1, 5, None, "auto"),                                         # f16 activations, no shared expert
    (1, 256, dict(H=128, I=256, E=8, k=2), "auto"),               # more tokens than CTAs: rows b, b + grid
    (2, 3, dict(H=1024, I=512, E=8, k=4), "gemv"),                # MXFP4 + bf16 through the GEMV
    (4, 80, dict(H=256, I=128, E=16, k=8, shared_I=64), "auto"),  # 640 routes: tail launched after
    (2, 4, dict(H=512, I=384, E=8, k=4), "gemm"),                 # decode kernels, then the tail launch
]


def _ids(case):
    cfg, T, sh, path = case
    return (f"cfg{cfg}-T{T}-" + ("full" if sh is None else "x".join(f"{k}{v}" for k, v in sh.items()))
            + f"-{path}")


def _tail_inputs(T, H, adt, seed):
    rng = np.random.default_rng(seed)
    tdt = synth.ADT_TORCH[adt]
    h1 = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(tdt)
    x = torch.from_numpy((rng.standard_normal((T, H)) * 2).astype(np.float32)).to(tdt)
    w2 = torch.from_numpy((1 + 0.1 * rng.standard_normal(H)).astype(np.float32)).to(torch.bfloat16)
    w1 = torch.from_numpy((1 + 0.1 * rng.standard_normal(H)).astype(np.float32)).to(torch.bfloat16)
    return h1, x, w2, w1


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_forward_tail_bit_exact(case):
    moe = _moe()
    cfg, T, shapes, path = case
    dev = "cuda" if shapes is None else "cpu"
    L = synth.make_layer(cfg, T=T, shapes=shapes, device=dev)
    D = to_device(L, "cuda")
    c = L["cfg"]
    H = c["H"]
    _, _, oidx, ow = oracle_route(L, bits16(L["x"]))
    idx, w = torch.from_numpy(oidx).cuda(), torch.from_numpy(ow).cuda()
    ex, sh = gpu_layer(D)
    h1, xr, w2, w1 = _tail_inputs(T, H, c["adt"], 1000 + T)
    w2, w1 = w2.cuda(), w1.cuda()
    scalar, eps = 0.8, 1e-6

    # the two calls
    ws = moe.alloc_workspace(T, c["k"], ex, sh)
    y0, y32_0 = moe.forward(D["x"], ex, idx, w, shared=sh, want_f32=True, ws=ws, path=path)
    y_fwd = y0.clone()
    gh0, gx0 = h1.cuda(), xr.cuda()
    moe.gemma_tail(y0, gh0, gx0, w2, w1, scalar, eps)
    # the one call
    ws2 = moe.alloc_workspace(T, c["k"], ex, sh)
    gh1, gx1 = h1.cuda(), xr.cuda()
    y1, y32_1 = moe.forward_tail(D["x"], ex, idx, w, gh1, gx1, w2, w1, scalar, eps, shared=sh,
                                 want_f32=True, ws=ws2, path=path)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0 and moe.device_status(ws2) == 0
    assert torch.equal(y32_1.view(torch.int32), y32_0.view(torch.int32))
    assert torch.equal(y1.view(torch.int16), y0.view(torch.int16))
    assert torch.equal(gh1.view(torch.int16), gh0.view(torch.int16))
    assert torch.equal(gx1.view(torch.int16), gx0.view(torch.int16))
    # the tail against the oracle's, on the GPU's own routed output
    oy, oh, ox = oracle.gemma_tail(bits16(y_fwd), bits16(h1), bits16(xr), bits16(w2.cpu()), bits16(w1.cpu()),
                                   c["adt"], scalar, eps=eps)
    assert np.array_equal(bits16(y1), oy)
    assert np.array_equal(bits16(gh1), oh)
    assert np.array_equal(bits16(gx1), ox)


def test_forward_tail_repeats_bit_exact():
    """Calls in a row on one workspace (the tile count is cleared by each call's phase 1)."""
    moe = _moe()
    L = synth.make_layer(4, T=8, device="cuda")
    c = L["cfg"]
    _, _, oidx, ow = oracle_route(L, bits16(L["x"]))
    idx, w = torch.from_numpy(oidx).cuda(), torch.from_numpy(ow).cuda()
    ex, sh = gpu_layer(L)
    h1, xr, w2, w1 = _tail_inputs(8, c["H"], c["adt"], 7)
    w2, w1 = w2.cuda(), w1.cuda()
    ws = moe.alloc_workspace(8, c["k"], ex, sh)
    outs = []
    for _ in range(3):
        gh, gx = h1.cuda(), xr.cuda()
        y, _ = moe.forward_tail(L["x"], ex, idx, w, gh, gx, w2, w1, 0.8, shared=sh, ws=ws)
        outs.append((y.clone(), gh, gx))
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_forward_tail_validates_its_arguments():
    moe = _moe()
    L = synth.make_layer(4, T=2, shapes=dict(H=256, I=128, E=16, k=8, shared_I=64), device="cuda")
    c = L["cfg"]
    ex, sh = gpu_layer(L)
    idx = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
    idx[:] = torch.arange(8, dtype=torch.int32, device="cuda")
    w = torch.full((2, 8), 0.125, dtype=torch.float32, device="cuda")
    h1, xr, w2, w1 = (t.cuda() for t in _tail_inputs(2, 256, c["adt"], 3))
    y = torch.empty_like(L["x"])
    with pytest.raises(moe.TsMoeError):        # y aliases h1
        moe.forward_tail(L["x"], ex, idx, w, y, xr, w2, w1, 0.8, shared=sh, out=(y, None))
