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
    assert moe.noalloc_device_status() == 0


def test_noalloc_scratch_reuse_across_every_expert_path():
    """Calls of different shapes and paths back to back on the one scratch: the tensor-core
    grouped GEMM (T > 8; T*k <= 64 keeps split-K partials and counters in the scratch), the
    decode GEMV with the route list and combine fused in, and the GEMV with the route-list
    kernel and a separate combine (T*k > 512).  Each result equals ts_moe_forward's bit for bit
    (same kernels, deterministic), including a repeat of the first call after the others."""
    import mixture_experts_routed_logits_gb300 as moe
    layers = [_layer(2, 16, dict(H=256, I=256, E=8, k=4)),                      # MXFP4, GEMM, split K
              _layer(2, 5, dict(H=512, I=384, E=8, k=4)),                       # MXFP4, fused GEMV
              _layer(2, 40, dict(H=256, I=256, E=8, k=4)),                      # MXFP4, GEMM
              _layer(4, 80, dict(H=256, I=96, E=16, k=8, shared_I=128)),        # INT4 GEMV, T*k > 512
              _layer(2, 16, dict(H=256, I=256, E=8, k=4))]                      # the first again
    layers[4] = layers[0]
    refs = [moe.forward(x, ex, idx, w, shared=sh, want_f32=True) for c, x, ex, sh, idx, w in layers]
    outs = []
    for c, x, ex, sh, idx, w in layers:
        outs.append(moe.forward_noalloc(x, ex, idx, w, shared=sh, want_f32=True))
    torch.cuda.synchronize()
    for (ry, ry32), (ny, ny32) in zip(refs, outs):
        assert torch.equal(ny.view(torch.int16), ry.view(torch.int16))
        assert torch.equal(ny32.view(torch.int32), ry32.view(torch.int32))
    assert moe.noalloc_device_status() == 0


def test_noalloc_reports_device_errors():
    """An expert id outside 0..E-1 is left out of the route list and reported through the
    scratch's status word, which ts_moe_noalloc_device_status reads and clears."""
    import mixture_experts_routed_logits_gb300 as moe
    c, x, ex, sh, idx, w = _layer(2, 5, dict(H=512, I=384, E=8, k=4))
    bad = idx.clone()
    bad[1, 2] = c["E"] + 3
    moe.forward_noalloc(x, ex, bad, w, shared=sh)
    torch.cuda.synchronize()
    assert moe.noalloc_device_status() == 1
    assert moe.noalloc_device_status() == 0          # read and cleared
    moe.forward_noalloc(x, ex, idx, w, shared=sh)
    torch.cuda.synchronize()
    assert moe.noalloc_device_status() == 0


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
