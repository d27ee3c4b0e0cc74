"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every function
include/ts_moe.h declares, and refuses invalid arguments before launching anything."""
import ctypes

import pytest

import mixture_experts_routed_logits_gb300 as moe


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return moe.lib()


def test_exports_every_declared_function(L):
    names = moe.header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_version(L):
    assert L.ts_moe_version().decode().count(".") == 2


def test_packed_bytes(L):
    # MXFP4: 16-row tiles of 32-column blocks, 256 code bytes + 16 scale bytes per block
    assert L.ts_moe_packed_bytes(2, 32, 2880, 2880) == 32 * 180 * 90 * 272
    assert L.ts_moe_packed_bytes(3, 128, 704, 2048) == 128 * 44 * 64 * 320
    assert L.ts_moe_packed_bytes(0, 1, 16, 32) == 0      # 16-bit formats are not packed
    assert L.ts_moe_packed_bytes(2, 1, 24, 32) == 0      # rows not a multiple of 16
    assert L.ts_moe_packed_bytes(2, 1, 16, 48) == 0      # K not a multiple of 32


def _experts(fmt=2, act=2, E=32, H=2880, I=2880, ptr=0x1000):
    return moe.CExperts(fmt, act, E, H, I, ptr, ptr, ptr, None, None, None, 7.0, 1.702)


def test_workspace_size_grows_with_tokens(L):
    ex = _experts()
    a = L.ts_moe_workspace_size(1, 4, ctypes.byref(ex), None)
    b = L.ts_moe_workspace_size(8, 4, ctypes.byref(ex), None)
    assert 0 < a < b
    assert L.ts_moe_workspace_size(8, 0, ctypes.byref(ex), None) == 0


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_workspace_for_T_tokens_serves_every_smaller_batch(L, k):
    # decode-sized calls (T*k <= 64) keep split-K partials, so the size must not drop past them
    ex = _experts()
    sizes = [L.ts_moe_workspace_size(T, k, ctypes.byref(ex), None) for T in range(1, 130)]
    assert all(0 < a <= b for a, b in zip(sizes, sizes[1:]))


@pytest.mark.parametrize("case,status", [
    (dict(E=300), 2), (dict(H=100), 2), (dict(fmt=7), 1), (dict(act=9), 1), (dict(ptr=0x1001), 1),
])
def test_forward_rejects_bad_descriptor(L, case, status):
    kw = dict(fmt=2, act=2, E=32, H=2880, I=2880, ptr=0x1000)
    kw.update(case)
    ex = _experts(**kw)
    st = L.ts_moe_forward(ctypes.c_void_p(0x2000), 1, 4, ctypes.byref(ex), ctypes.c_void_p(0x3000),
                          ctypes.c_void_p(0x4000), 4, None, ctypes.c_void_p(0x5000), None,
                          ctypes.c_void_p(0x6000), 16, None)   # tiny workspace: a second line of defence
    assert st == status
    assert L.ts_last_error()


def test_forward_rejects_small_workspace_and_nulls(L):
    ex = _experts()
    args = [ctypes.c_void_p(0x2000), 1, 4, ctypes.byref(ex), ctypes.c_void_p(0x3000),
            ctypes.c_void_p(0x4000), 4, None, ctypes.c_void_p(0x5000), None,
            ctypes.c_void_p(0x6000), 16, None]
    assert L.ts_moe_forward(*args) == 5
    assert b"workspace" in L.ts_last_error()
    args[0] = None
    assert L.ts_moe_forward(*args) == 1
    args[0] = ctypes.c_void_p(0x2000)
    args[6] = 33                       # k > E
    assert L.ts_moe_forward(*args) == 1
    args[6] = 4
    args[8] = ctypes.c_void_p(0x5008)  # y not 16-byte aligned
    assert L.ts_moe_forward(*args) == 1
    assert b"aligned" in L.ts_last_error()
    args[8] = ctypes.c_void_p(0x5000)
    args[9] = ctypes.c_void_p(0x7004)  # y_f32 not 16-byte aligned
    assert L.ts_moe_forward(*args) == 1
    args[9] = None
    bf = _experts(fmt=1)
    a2 = list(args)
    a2[6] = 4
    a2[1] = 0                          # f16 activations with bf16 weights
    a2[3] = ctypes.byref(bf)
    assert L.ts_moe_forward(*a2) == 2


def test_forward_T0_is_a_noop(L):
    ex = _experts()
    st = L.ts_moe_forward(None, 1, 0, ctypes.byref(ex), None, None, 4, None, None, None, None, 0,
                          None)
    assert st == 0


def test_route_rejects_bad_k_and_E(L):
    assert L.ts_moe_route(ctypes.c_void_p(0x100), None, None, 4, 8, 9, 0, ctypes.c_void_p(0x200),
                          ctypes.c_void_p(0x300), None) == 1
    assert L.ts_moe_route(ctypes.c_void_p(0x100), None, None, 4, 257, 2, 0, ctypes.c_void_p(0x200),
                          ctypes.c_void_p(0x300), None) == 2
    assert L.ts_moe_route(ctypes.c_void_p(0x100), None, None, 4, 8, 2, 2, ctypes.c_void_p(0x200),
                          ctypes.c_void_p(0x300), None) == 1   # scaled mode without scale
    assert L.ts_moe_router_route(ctypes.c_void_p(0x100), 1, 4, 100, ctypes.c_void_p(0x100), 8, 0,
                                 1e-6, None, None, 2, 0, None, None, ctypes.c_void_p(0x200),
                                 ctypes.c_void_p(0x300), None) == 2   # H % 32
    assert L.ts_moe_router_route(ctypes.c_void_p(0x100), 1, 4, 128, ctypes.c_void_p(0x100), 8, 1,
                                 1e-6, None, None, 2, 0, None, None, ctypes.c_void_p(0x200),
                                 ctypes.c_void_p(0x300), None) == 1   # rmsnorm without xn_out


def test_build_routes_and_pack_reject(L):
    assert L.ts_moe_build_routes(None, 4, 300, 2, None, None, None, None) == 2
    assert L.ts_moe_build_routes(None, 4, 8, 2, None, None, None, None) == 1
    assert L.ts_moe_pack(2, 1, 16, 32, ctypes.c_void_p(0x100), ctypes.c_void_p(0x100),
                         ctypes.c_void_p(0x101), 1 << 20, None) == 1          # misaligned
    assert L.ts_moe_pack(2, 1, 16, 32, ctypes.c_void_p(0x100), ctypes.c_void_p(0x100),
                         ctypes.c_void_p(0x100), 10, None) == 1               # too small


def test_gemma_tail_rejects_bad_arguments(L):
    p = [ctypes.c_void_p(0x1000 + 0x100 * i) for i in range(5)]
    f = ctypes.c_float
    assert L.ts_moe_gemma_tail(*p, f(1.0), f(1e-6), 0, 0, 256, None) == 0      # T == 0: nothing
    assert L.ts_moe_gemma_tail(*p, f(1.0), f(1e-6), 5, 4, 256, None) == 1      # bad adt
    assert L.ts_moe_gemma_tail(*p, f(1.0), f(1e-6), 1, 4, 100, None) == 2      # H % 32
    assert L.ts_moe_gemma_tail(*p, f(1.0), f(1e-6), 1, 4, 8224, None) == 2     # H > 8192
    assert L.ts_moe_gemma_tail(None, *p[1:], f(1.0), f(1e-6), 1, 4, 256, None) == 1
    assert L.ts_moe_gemma_tail(p[0], p[0], *p[2:], f(1.0), f(1e-6), 1, 4, 256, None) == 1   # y == h1
    assert b"distinct" in L.ts_last_error()


def test_forward_tail_rejects_bad_arguments(L):
    """Refused before any device work: no experts, and the tail's own checks (y aliasing h1)."""
    p = [ctypes.c_void_p(0x1000 + 0x100 * i) for i in range(8)]
    f = ctypes.c_float
    args = lambda y, h1: (p[0], 1, 4, None, p[1], p[2], 2, None, y, None, p[3], 1 << 20, 0,
                          h1, p[5], p[6], p[7], f(1.0), f(1e-6), None)
    assert L.ts_moe_forward_tail(*args(p[4], p[5])) == 1                        # experts NULL
    assert b"experts" in L.ts_last_error()
