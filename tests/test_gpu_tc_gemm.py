"""GPU parity of the tensor-core (tcgen05) grouped GEMM path against the CPU oracle, and the
cross-check of the two expert paths on the same inputs (the Gemma-4 batched prefill pages state
that the batched route-list kernels agree with sequential per-token decode calls)."""
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
    (5, 40, dict(H=256, I=512, E=8, k=2)),            # bf16, several 64-column blocks
    (5, 37, dict(H=320, I=384, E=6, k=3)),            # ragged route tiles, partial row blocks
    (5, 300, dict(H=256, I=256, E=4, k=2)),           # > 256 routes per expert: 2+ route tiles
    (1, 20, dict(H=128, I=256, E=8, k=2)),            # f16 weights + f16 activations
    (5, 2048, None),                                  # full Mixtral-8x7B prefill chunk
    (5, 512, dict(H=1024, I=2048, E=8, k=2)),         # 256-route tiles, 32 down items on 152 SMs
    (5, 600, dict(H=1024, I=2048, E=4, k=2)),         # two route tiles per expert
    (2, 40, dict(H=512, I=384, E=8, k=4)),            # MXFP4 + clamped SwiGLU + biases (one launch)
    (2, 16, dict(H=512, I=384, E=8, k=4)),            # MXFP4, 64 routes: split K, two launches
    (2, 17, dict(H=512, I=384, E=8, k=4)),            # 68 routes: both phases in one launch
    (2, 40, dict(H=256, I=256, E=128, k=8)),          # one launch, many experts with a tile or two
    (3, 96, dict(H=1024, I=640, E=16, k=4)),          # one launch, skewed, ragged row blocks
    (3, 77, dict(H=640, I=448, E=8, k=4)),            # MXFP4, skewed, partial 128-row blocks
    (3, 512, None),                                   # full gpt-oss prefill micro-batch
    (2, 1, None),                                     # gpt-oss decode T=1 (split K)
    (2, 8, None),                                     # gpt-oss decode T=8 (split K)
    (5, 8, dict(H=4096, I=14336, E=8, k=2)),          # Mixtral decode through the tensor cores
]


def _ids(case):
    cfg, T, sh = case
    return f"cfg{cfg}-T{T}-" + ("full" if sh is None else "x".join(f"{k}{v}" for k, v in sh.items()))


def _make(cfg, T, shapes):
    dev = "cuda" if shapes is None else "cpu"
    L = synth.make_layer(cfg, T=T, shapes=shapes, device=dev)
    return L, to_device(L, "cuda")


# MXFP4 cases run on both tensor-core variants: the block-scaled MMA ("gemm": e2m1 weights,
# activations split into two e4m3 terms) and the f16 MMA over weights dequantised in shared
# memory ("gemm_dequant")
PARITY = [pytest.param(c, p, id=_ids(c) + "-" + p)
          for c in CASES for p in (("gemm", "gemm_dequant") if c[0] in (2, 3) else ("gemm",))]


@pytest.mark.parametrize("case,path", PARITY)
def test_tc_gemm_parity(case, path):
    moe = _moe()
    cfg, T, shapes = case
    L, D = _make(cfg, T, shapes)
    c = L["cfg"]
    xb = bits16(L["x"])
    _, _, oidx, ow = oracle_route(L, xb)
    ex, sh = gpu_layer(D)
    ws = moe.alloc_workspace(T, c["k"], ex, sh)
    y, y32 = moe.forward(D["x"], ex, torch.from_numpy(oidx).cuda(), torch.from_numpy(ow).cuda(),
                         want_f32=True, ws=ws, path=path)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    oex, _ = oracle_layer(L)
    toks = None if (T <= 48 and shapes is not None) else np.unique(np.linspace(0, T - 1, 6).astype(np.int32))
    oy, oy32, _ = oracle.moe_forward(xb, c["adt"], oex, oidx, ow, tokens=toks, nthreads=NTHREADS)
    rows = slice(None) if toks is None else toks
    # h elements next to a 16-bit rounding boundary (named by the oracle) and what they may move
    allow, _ = flip_allowance(L, oex, None, oracle.adt_bits_to_f64(xb[rows], c["adt"]), oidx[rows],
                              ow[rows], c["adt"], kappa=kappa_for(c, T, path), nthreads=NTHREADS)
    check_outputs(oracle.adt_bits_to_f64(bits16(y)[rows], c["adt"]), y32.double().cpu().numpy()[rows],
                  oracle.adt_bits_to_f64(oy, c["adt"]), oy32.astype(np.float64), c["adt"],
                  allow=allow)


@pytest.mark.parametrize("case", [(5, 8, dict(H=512, I=1024, E=8, k=2)), (5, 64, dict(H=256, I=512, E=8, k=2)),
                                  (2, 8, dict(H=2880, I=2880, E=32, k=4)), (3, 48, dict(H=512, I=512, E=8, k=4)),
                                  (5, 300, dict(H=1024, I=1024, E=8, k=2))],   # 256-route tiles
                         ids=_ids)
def test_gemm_and_gemv_paths_agree(case):
    moe = _moe()
    cfg, T, shapes = case
    L, D = _make(cfg, T, shapes)
    c = L["cfg"]
    ex, _ = gpu_layer(D)
    idx, w, _, _ = moe.router_route(D["x"], D["Wr"], c["k"], router_bias=D["router_bias"])
    ya, ya32 = moe.forward(D["x"], ex, idx, w, want_f32=True, path="gemv")
    yb, yb32 = moe.forward(D["x"], ex, idx, w, want_f32=True, path="gemm")
    torch.cuda.synchronize()
    a32, b32 = ya32.double().cpu().numpy(), yb32.double().cpu().numpy()
    rel = np.linalg.norm(a32 - b32) / np.linalg.norm(a32)
    assert np.abs(a32 - b32).max() <= 2e-2 and rel <= 1e-3, rel


def test_mx_one_launch_deterministic():
    """Both block-scaled phases in one launch hand items out from a counter, so a run's items
    land on other CTAs than the last run's: the outputs must not change."""
    moe = _moe()
    L, D = _make(3, 160, dict(H=512, I=512, E=32, k=4))
    ex, _ = gpu_layer(D)
    idx, w, _, _ = moe.router_route(D["x"], D["Wr"], 4, router_bias=D["router_bias"])
    outs = [moe.forward(D["x"], ex, idx, w, want_f32=True, path="gemm")[1].clone() for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))


@pytest.mark.parametrize("T,shapes", [(96, dict(H=256, I=512, E=8, k=2)),
                                      (512, dict(H=1024, I=2048, E=8, k=2))])   # 256-route tiles
def test_tc_gemm_deterministic(T, shapes):
    """Repeated calls give the same bits."""
    moe = _moe()
    L, D = _make(5, T, shapes)
    ex, _ = gpu_layer(D)
    idx, w, _, _ = moe.router_route(D["x"], D["Wr"], 2)
    ws = moe.alloc_workspace(T, 2, ex, None)
    outs = [moe.forward(D["x"], ex, idx, w, want_f32=True, ws=ws, path="gemm")[1].clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))


def test_gemm_path_refuses_int4_weights():
    moe = _moe()
    L, D = _make(4, 16, dict(H=256, I=128, E=8, k=4, shared_I=64))
    ex, _ = gpu_layer(D)
    idx, w, _, _ = moe.router_route(D["x"], D["Wr"], 4, mode="softmax_k_scaled",
                                    per_expert_scale=D["scale"])
    with pytest.raises(moe.TsMoeError) as ei:
        moe.forward(D["x"], ex, idx, w, path="gemm")
    assert ei.value.status == 2


def _widen_scales(L, lo, hi, frac, seed):
    """Replace a random `frac` of the MXFP4 block exponents of every matrix by values in [lo, hi]."""
    g = torch.Generator().manual_seed(seed)
    for name in ("gate_s", "up_s", "down_s"):
        s = L["experts"][name]
        pick = torch.rand(s.shape, generator=g) < frac
        s[pick] = torch.randint(lo, hi + 1, (int(pick.sum()),), generator=g).to(torch.uint8)


@pytest.mark.parametrize("path", ["gemm", "gemm_dequant"])
def test_tc_gemm_mxfp4_scales_outside_normal_f16(path):
    # block scales 2^-23 .. 2^1: below 2^-14 the scale itself is not a normal f16 number, yet
    # every scaled e2m1 value still is an exact f16 number, so the result must match the oracle
    moe = _moe()
    L = synth.make_layer(2, T=24, shapes=dict(H=256, I=192, E=4, k=2), device="cpu")
    _widen_scales(L, 104, 128, 0.1, 11)
    D = to_device(L, "cuda")
    c = L["cfg"]
    xb = bits16(L["x"])
    _, _, oidx, ow = oracle_route(L, xb)
    ex, _ = gpu_layer(D)
    ws = moe.alloc_workspace(24, c["k"], ex)
    y, y32 = moe.forward(D["x"], ex, torch.from_numpy(oidx).cuda(), torch.from_numpy(ow).cuda(),
                         want_f32=True, ws=ws, path=path)
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    oex, _ = oracle_layer(L)
    oy, oy32, _ = oracle.moe_forward(xb, c["adt"], oex, oidx, ow, nthreads=NTHREADS)
    check_outputs(oracle.adt_bits_to_f64(bits16(y), c["adt"]), y32.double().cpu().numpy(),
                  oracle.adt_bits_to_f64(oy, c["adt"]), oy32.astype(np.float64), c["adt"])


def test_block_scaled_path_takes_any_e8m0_scale():
    # gate/up block scales 2^-27 .. 2^23 (far outside what the f16 dequantisation represents):
    # the block-scaled MMA applies e8m0 scales in hardware, so the layer matches the oracle
    moe = _moe()
    L = synth.make_layer(2, T=24, shapes=dict(H=256, I=192, E=4, k=2), device="cpu")
    g = torch.Generator().manual_seed(5)
    for name in ("gate_s", "up_s"):
        sc = L["experts"][name]
        pick = torch.rand(sc.shape, generator=g) < 0.1
        sc[pick] = torch.randint(100, 151, (int(pick.sum()),), generator=g).to(torch.uint8)
    D = to_device(L, "cuda")
    c = L["cfg"]
    xb = bits16(L["x"])
    _, _, oidx, ow = oracle_route(L, xb)
    ex, _ = gpu_layer(D)
    ws = moe.alloc_workspace(24, c["k"], ex)
    y, y32 = moe.forward(D["x"], ex, torch.from_numpy(oidx).cuda(), torch.from_numpy(ow).cuda(),
                         want_f32=True, ws=ws, path="gemm")
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 0
    oex, _ = oracle_layer(L)
    oy, oy32, _ = oracle.moe_forward(xb, c["adt"], oex, oidx, ow, nthreads=NTHREADS)
    allow, _ = flip_allowance(L, oex, None, oracle.adt_bits_to_f64(xb, c["adt"]), oidx, ow, c["adt"],
                              kappa=kappa_for(c, 24, "gemm"), nthreads=NTHREADS)
    check_outputs(oracle.adt_bits_to_f64(bits16(y), c["adt"]), y32.double().cpu().numpy(),
                  oracle.adt_bits_to_f64(oy, c["adt"]), oy32.astype(np.float64), c["adt"], allow=allow)


def test_pack_mx_layout():
    """The tensor-core MXFP4 blob, byte for byte, against the layout built here with numpy: codes
    [nmat][KG][G][R][64 B] (128 codes of a row per group of 128 columns, gate and up side by side
    for a pair, zero codes past K), then (at a 256-byte boundary) the e8m0 scales in 512-byte
    atoms [nmat][U][KG][2][512] (atom pair = gate and up of 128 rows, or the two 128-row halves
    of 256 rows), row r and block b of an atom at 16*(r%32) + 4*(r/32) + b, 1.0 (127) for rows and
    blocks past the matrix."""
    moe = _moe()
    g = torch.Generator().manual_seed(2)
    for pair in (False, True):
        for nmat, R, K in [(3, 96, 320), (2, 2880, 2880), (1, 32, 128), (2, 288, 256)]:
            G = 2 if pair else 1
            codes = [torch.randint(0, 256, (nmat, R, K // 2), generator=g, dtype=torch.uint8) for _ in range(G)]
            scales = [torch.randint(110, 140, (nmat, R, K // 32), generator=g, dtype=torch.uint8) for _ in range(G)]
            args = (codes[1].cuda(), scales[1].cuda()) if pair else (None, None)
            blob = moe.pack_mx(codes[0].cuda(), scales[0].cuda(), *args).cpu().numpy()
            KG = (K + 127) // 128
            c = np.zeros((nmat, KG, G, R, 64), np.uint8)
            for m in range(G):
                cp = np.zeros((nmat, R, KG * 64), np.uint8)
                cp[:, :, :K // 2] = codes[m].numpy()
                c[:, :, m] = cp.reshape(nmat, R, KG, 64).transpose(0, 2, 1, 3)
            assert np.array_equal(blob[:c.size], c.reshape(-1))
            off = (c.size + 255) // 256 * 256
            U = (R + 127) // 128 if pair else (R + 255) // 256
            span = 128 if pair else 256
            sp = np.full((G, nmat, U * span, KG * 4), 127, np.uint8)
            for m in range(G):
                sp[m, :, :R, :K // 32] = scales[m].numpy()
            atoms = np.empty((nmat, U, KG, 2, 512), np.uint8)
            for b in range(512):
                rr, blk = 32 * ((b % 16) // 4) + b // 16, b % 4
                for m in range(2):
                    src = sp[m] if pair else sp[0]
                    rows = np.arange(U) * span + (0 if pair else 128 * m) + rr
                    atoms[:, :, :, m, b] = src[:, rows][:, :, blk::4][:, :, :KG]
            assert blob.size == off + atoms.size
            assert np.array_equal(blob[off:], atoms.reshape(-1))


def test_tc_gemm_reports_scales_it_cannot_represent():
    # a block scale of 2^-27: its scaled e2m1 values are not all f16 numbers; the dequantising
    # tensor-core path must say so through the device status (the GEMV path and the
    # block-scaled path compute such layers exactly)
    moe = _moe()
    L = synth.make_layer(2, T=24, shapes=dict(H=256, I=192, E=4, k=2), device="cpu")
    L["experts"]["gate_s"][1, 3, 2] = 100
    D = to_device(L, "cuda")
    c = L["cfg"]
    ex, _ = gpu_layer(D)
    idx = torch.tensor([[1, 2]] * 24, dtype=torch.int32, device="cuda")
    w = torch.full((24, 2), 0.5, dtype=torch.float32, device="cuda")
    ws = moe.alloc_workspace(24, c["k"], ex)
    moe.forward(D["x"], ex, idx, w, ws=ws, path="gemm_dequant")
    torch.cuda.synchronize()
    assert moe.device_status(ws) == 2
