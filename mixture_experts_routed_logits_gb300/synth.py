"""Seeded synthetic inputs for the routed-expert layer.

This module only draws random numbers and lays them out in the canonical
formats; it holds none of the layer's arithmetic.  The CUDA path, the tests,
the bench and the CPU oracle all read the bytes it produces.

Workloads (shapes and distributions of the five layer configurations the
layer is measured on; every draw comes from a torch.Generator seeded with
``seed``):

  1 tiny Mixtral-style   T=4,    H=128,  I=256,   E=8,   k=2, f16 weights, f16 x, SiLU
  2 gpt-oss decode       T=1|8,  H=2880, I=2880,  E=32,  k=4, MXFP4 weights, bf16 x,
                         router bias N(0,0.5) f32, expert biases bf16 N(0,0.02), clamped SwiGLU
  3 gpt-oss prefill      T=512,  as 2, plus a per-expert skew N(0,1) folded into the router bias
  4 Gemma-style          T=8,    H=2048, I=704,   E=128, k=8, INT4-affine g32 weights, bf16 x,
                         per_expert_scale U(0.5,1.5), RMSNorm eps 1e-6, shared GELU FFN
                         (inter 2048, f16 N(0,0.02)), GELU-tanh routed experts
  5 Mixtral-8x7B prefill T=2048, H=4096, I=14336, E=8,   k=2, bf16 weights N(0,0.02), bf16 x, SiLU
"""
from __future__ import annotations

import torch

CONFIGS = {
    1: dict(name="tiny_mixtral_T4_H128_I256_E8_k2_f16", T=4, H=128, I=256, E=8, k=2,
            adt="f16", fmt="f16", act="silu", mode="softmax_k", router_bias_std=None,
            skew_std=None, expert_bias_std=None, rmsnorm=False, shared_I=None),
    2: dict(name="gptoss_decode_H2880_E32_k4_mxfp4", T=8, H=2880, I=2880, E=32, k=4,
            adt="bf16", fmt="mxfp4", act="gptoss", mode="softmax_k", router_bias_std=0.5,
            skew_std=None, expert_bias_std=0.02, rmsnorm=False, shared_I=None),
    3: dict(name="gptoss_prefill_T512_H2880_E32_k4_mxfp4_skew", T=512, H=2880, I=2880, E=32,
            k=4, adt="bf16", fmt="mxfp4", act="gptoss", mode="softmax_k", router_bias_std=0.5,
            skew_std=1.0, expert_bias_std=0.02, rmsnorm=False, shared_I=None),
    4: dict(name="gemma_T8_H2048_I704_E128_k8_int4_shared2048", T=8, H=2048, I=704, E=128, k=8,
            adt="bf16", fmt="int4", act="gelu_tanh", mode="softmax_k_scaled",
            router_bias_std=None, skew_std=None, expert_bias_std=None, rmsnorm=True,
            shared_I=2048),
    5: dict(name="mixtral8x7b_prefill_T2048_H4096_I14336_E8_k2_bf16", T=2048, H=4096, I=14336,
            E=8, k=2, adt="bf16", fmt="bf16", act="silu", mode="softmax_k",
            router_bias_std=None, skew_std=None, expert_bias_std=None, rmsnorm=False,
            shared_I=None),
}

ADT_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}


def default_seed(cfg_id: int) -> int:
    return 0x5EED0000 + int(cfg_id)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, dtype, g, device):
    # drawn in f32 in row chunks to bound temporary memory, then rounded to dtype
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1, shape[-1]) if len(shape) > 1 else out.view(1, -1)
    rows = flat.shape[0]
    step = max(1, (1 << 26) // max(1, flat.shape[1]))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        flat[r0:r1] = (torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                                   dtype=torch.float32) * std).to(dtype)
    return out


def _uniform(shape, lo, hi, g, device):
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def _codes(shape, g, device):
    # uniform bytes: each 4-bit code (both nibbles) uniform over its 16 values
    return torch.randint(0, 256, shape, generator=g, device=device, dtype=torch.uint8)


def make_expert_weights(fmt, E, H, I, g, device, std=0.02, scale_exp=(-8, -4), bias_std=None):
    """Canonical per-expert weights: gate/up [E][I][H], down [E][H][I] (K contiguous).

    f16/bf16: N(0, std).  MXFP4: uniform codes, e8m0 exponents uniform in scale_exp.
    INT4-affine: uniform codes, per-32 group f16 scale ~ U(0.002, 0.006) and
    f16 min = -8*scale*(1+U(-0.05,0.05)).  Biases bf16 N(0, bias_std) when bias_std is set.
    """
    out = {}
    for name, (R, K) in (("gate", (I, H)), ("up", (I, H)), ("down", (H, I))):
        if fmt in ("f16", "bf16"):
            out[name] = _normal((E, R, K), std, ADT_TORCH[fmt], g, device)
            out[name + "_s"] = None
        elif fmt == "mxfp4":
            out[name] = _codes((E, R, K // 2), g, device)
            lo, hi = scale_exp
            out[name + "_s"] = torch.randint(127 + lo, 127 + hi + 1, (E, R, K // 32), generator=g,
                                             device=device, dtype=torch.uint8)
        elif fmt == "int4":
            out[name] = _codes((E, R, K // 2), g, device)
            sc = _uniform((E, R, K // 32), 0.002, 0.006, g, device).to(torch.float16)
            mn = (-8.0 * sc.float() * (1.0 + _uniform((E, R, K // 32), -0.05, 0.05, g, device))
                  ).to(torch.float16)
            out[name + "_s"] = torch.stack([sc, mn], dim=-1).contiguous()  # [E][R][K/32][2] f16
        else:
            raise ValueError(fmt)
        out[name + "_b"] = (_normal((E, R), bias_std, torch.bfloat16, g, device)
                            if bias_std else None)
    return out


def make_layer(cfg_id: int, T: int | None = None, seed: int | None = None, device="cpu",
               shapes: dict | None = None):
    """All inputs of one layer call.  ``shapes`` overrides H/I/E/k/shared_I for small cases."""
    c = dict(CONFIGS[cfg_id])
    if shapes:
        c.update(shapes)
    if T is not None:
        c["T"] = T
    seed = default_seed(cfg_id) if seed is None else seed
    g = _gen(device, seed)
    adt = ADT_TORCH[c["adt"]]
    T, H, I, E = c["T"], c["H"], c["I"], c["E"]
    L = dict(cfg=c, seed=seed)
    L["x"] = _normal((T, H), 1.0, adt, g, device)
    L["Wr"] = _normal((E, H), 0.02, adt, g, device)
    bias = None
    if c.get("router_bias_std"):
        bias = torch.randn((E,), generator=g, device=device) * c["router_bias_std"]
    if c.get("skew_std"):
        skew = torch.randn((E,), generator=g, device=device) * c["skew_std"]
        bias = skew if bias is None else bias + skew   # folded into the per-expert additive vector
    L["router_bias"] = None if bias is None else bias.float().contiguous()
    L["scale"] = (_uniform((E,), 0.5, 1.5, g, device).contiguous()
                  if c["mode"] == "softmax_k_scaled" else None)
    L["experts"] = make_expert_weights(c["fmt"], E, H, I, g, device,
                                       bias_std=c.get("expert_bias_std"))
    if c.get("shared_I"):
        L["shared"] = make_expert_weights("f16", 1, H, c["shared_I"], g, device)
    else:
        L["shared"] = None
    return L


def make_l2_flush(device, nbytes=512 << 20):
    """A buffer larger than the 129 MB L2, written between timed steps."""
    return torch.empty(nbytes // 4, dtype=torch.float32, device=device)
