"""The bounded waits of the expert kernels: a wait that runs out ends in an error status the
host reads, the call returns normally and the CUDA context stays usable.

The wait is made to run out without any GPU fault: ts_moe_set_wait_test makes the next call's
phase-1 launch (the streaming GEMV, or the block-scaled decode kernel) withhold its first weight
copy (a copy nothing else will issue), so the consumer warps' bounded wait on it expires after
about a second.  The pages' convention is to
fail with a status rather than hang or quietly degrade (Gemma-4 batched routed prefill,
src/families/gemma4/moe_batch.rs, RealForwardError::Unsupported refusals)."""
import numpy as np
import pytest
import torch

from mixture_experts_routed_logits_gb300 import synth
from tests._helpers import gpu_layer, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("path", ["gemv", "auto"])
def test_a_wait_that_runs_out_reports_timeout_and_the_context_stays_usable(path):
    """path "auto" at T = 8 with MXFP4 blobs runs the block-scaled decode kernels."""
    import mixture_experts_routed_logits_gb300 as moe
    L = to_device(synth.make_layer(2, T=8, shapes=dict(H=512, I=384, E=8, k=4), device="cpu"), "cuda")
    c = L["cfg"]
    ex, _ = gpu_layer(L)
    idx, w, _, _ = moe.router_route(L["x"], L["Wr"], c["k"], router_bias=L["router_bias"])
    ws = moe.alloc_workspace(8, c["k"], ex)
    ref, ref32 = (t.clone() for t in moe.forward(L["x"], ex, idx, w, ws=ws, want_f32=True, path=path))
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    moe.set_wait_test(1)
    moe.forward(L["x"], ex, idx, w, ws=ws, path=path)   # returns TS_OK: the failure is on the device
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 4               # TS_ERR_TIMEOUT
    assert moe.device_status(ws) == 0               # read and cleared
    # the setting was consumed and the context is usable: the next call is the first one again
    y, y32 = moe.forward(L["x"], ex, idx, w, ws=ws, want_f32=True, path=path)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(y32.view(torch.int32), ref32.view(torch.int32))


def test_wait_test_setting_is_validated():
    import mixture_experts_routed_logits_gb300 as moe
    with pytest.raises(moe.TsMoeError) as ei:
        moe.set_wait_test(2)
    assert ei.value.status == 1
    moe.set_wait_test(0)
