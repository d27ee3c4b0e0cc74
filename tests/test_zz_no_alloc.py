"""The no-allocation entry point, ts_moe_forward_noalloc.

It serves callers that cannot allocate device memory when they run the layer (an application
that owns all device memory itself, a runtime whose allocator is out of reach of the calling
thread, a serving loop that must not allocate): instead of a caller-provided workspace it uses
a fixed scratch array in the library's own device memory.  These tests call it through the C
ABI and check it against ts_moe_forward on the same inputs, twice in a row with different
layers (the second call reuses the scratch the first one left behind).

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from mixture_experts_routed_logits_gb300 import synth
from tests._helpers import bits16, check_outputs, gpu_layer, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _layer(cfg, T, shapes):
    import mixture_experts_routed_logits_gb300 as moe
    L = to_device(synth.make_layer(cfg, T=T, shapes=shapes, device="cpu"), "cuda")
    c = L["cfg"]
    ex, sh = gpu_layer(L)
    idx, w, xn, _ = moe.router_route(L["x"], L["Wr"], c["k"], mode=c["mode"],
                                     router_bias=L["router_bias"], per_expert_scale=L["scale"],
                                     rmsnorm=c["rmsnorm"])
    x = xn if c["rmsnorm"] else L["x"]
    return c, x, ex, sh, idx, w


def _as_f64(t, adt):
    b = bits16(t)
    if adt == "bf16":
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return b.view(np.float16).astype(np.float64)


def test_noalloc_matches_forward_two_calls_in_a_row():
    import mixture_experts_routed_logits_gb300 as moe
    layers = [_layer(2, 5, dict(H=512, I=384, E=8, k=4)),                       # MXFP4, biases
              _layer(4, 8, dict(H=256, I=96, E=16, k=8, shared_I=128))]         # INT4 + shared
    refs = []
    for c, x, ex, sh, idx, w in layers:
        refs.append(moe.forward(x, ex, idx, w, shared=sh, want_f32=True))
    outs = []
    for c, x, ex, sh, idx, w in layers:          # two no-alloc calls back to back
        outs.append(moe.forward_noalloc(x, ex, idx, w, shared=sh, want_f32=True))
    torch.cuda.synchronize()
    for (c, *_), (ry, ry32), (ny, ny32) in zip(layers, refs, outs):
        check_outputs(_as_f64(ny, c["adt"]), ny32.double().cpu().numpy(), _as_f64(ry, c["adt"]),
                      ry32.double().cpu().numpy(), c["adt"])


def test_noalloc_rejects_work_beyond_its_scratch():
    import mixture_experts_routed_logits_gb300 as moe
    c, x, ex, sh, idx, w = _layer(2, 4, dict(H=512, I=384, E=8, k=4))
    big_T = 4096                                  # needs far more than the 16 MiB scratch
    xb = torch.zeros((big_T, 512), dtype=torch.bfloat16, device="cuda")
    ib = torch.zeros((big_T, 4), dtype=torch.int32, device="cuda")
    wb = torch.zeros((big_T, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.TsMoeError) as ei:
        moe.forward_noalloc(xb, ex, ib, wb)
    assert ei.value.status == 5 and "scratch" in str(ei.value)
