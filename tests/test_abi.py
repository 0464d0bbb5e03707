"""The C-ABI library (no GPU needed): it builds for sm_103a, exports every entry
point include/moe.h declares, and its host-side checks reject bad arguments
before any launch."""
import ctypes as C
import os
import re

import pytest

import moe_expert_layer_03_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    moe.build()
    return moe.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(moe.EXPORTS)


def test_status_strings_and_slot_bytes(L):
    assert L.moe_status_str(0) == b"ok"
    assert L.moe_status_str(3) == b"workspace too small"
    # the prepacked weights (int4: 1.59375 B per weight; bf16: 2) plus a
    # 256-byte trailer of bound exponents
    assert L.moe_slot_bytes(moe.W_INT4, 4096, 14336) == 93_585_408 + 256
    assert L.moe_slot_bytes(moe.W_BF16, 4096, 6400) == 6 * 4096 * 6400 + 256
    assert L.moe_slot_bytes(moe.W_INT4, 5120, 1536) == 12_533_760 + 256
    assert L.moe_slot_bytes(moe.W_FP8, 4096, 14336) == 178_913_280 + 256   # 3.046875 B per weight
    assert L.moe_slot_bytes(moe.W_INT4, 4096, 100) == 0          # d_ff not a multiple of 128
    assert L.moe_slot_bytes(7, 4096, 4096) == 0


def _fake_pool(E=8, d=256, F=512, fmt=moe.W_BF16):
    sb = (moe.lib().moe_slot_bytes(fmt, d, F) + 255) // 256 * 256
    return moe.MoePool(E, E, d, F, fmt, 0x10000000, sb, 0x20000000)   # never dereferenced


def test_workspace_sizes(L):
    p = _fake_pool()
    a = L.moe_layer_workspace_bytes(16, 2, C.byref(p), None)
    sh = _fake_pool(E=1)
    b = L.moe_layer_workspace_bytes(16, 2, C.byref(p), C.byref(sh))
    assert a > 16 * 2 * 256 * 2 and b > a
    assert L.moe_grouped_ffn_workspace_bytes(32, C.byref(p)) > 32 * 512 * 2
    bad = _fake_pool(d=200)
    assert L.moe_layer_workspace_bytes(16, 2, C.byref(bad), None) == 0


def test_host_checks_reject_before_launch(L):
    p = _fake_pool()
    P = C.c_void_p
    x, lg, out, ws = P(0x30000000), P(0x40000000), P(0x50000000), P(0x60000000)
    need = L.moe_layer_workspace_bytes(16, 2, C.byref(p), None)
    fwd = lambda *a: L.moe_layer_forward(*a)
    assert fwd(None, lg, 16, 2, C.byref(p), None, out, ws, need, None) == 1          # null x
    assert fwd(x, lg, 0, 2, C.byref(p), None, out, ws, need, None) == 1              # T = 0
    assert fwd(x, lg, 16, 9, C.byref(p), None, out, ws, need, None) == 1             # k > E
    assert fwd(x, lg, 16, 17, C.byref(_fake_pool(E=32)), None, out, ws, need, None) == 2   # k > 16
    assert fwd(P(0x30000002), lg, 16, 2, C.byref(p), None, out, ws, need, None) == 1  # misaligned
    assert fwd(x, lg, 16, 2, C.byref(p), None, out, ws, need - 1, None) == 3         # small ws
    mism = _fake_pool(E=1, F=1024)
    assert fwd(x, lg, 16, 2, C.byref(p), C.byref(mism), out, ws, need, None) == 2    # shared d_ff
    assert L.moe_route_topk(None, 4, 8, 2, P(0x10), P(0x20), None) == 1
    assert L.moe_route_topk(lg, 4, 300, 2, P(0x10), P(0x20), None) == 2               # E > 256
    assert L.moe_combine(P(0x10), P(0x20), P(0x30), None, 4, 2, 100, P(0x40), None) == 1


def test_router_host_checks_reject_before_launch(L):
    p = _fake_pool()
    P = C.c_void_p
    x, wr, lg, out, ws = P(0x30000000), P(0x38000000), P(0x40000000), P(0x50000000), P(0x60000000)
    rl = L.moe_router_logits
    rl.argtypes = [P, P, C.c_int, C.c_int, C.c_int, P, P]
    assert rl(None, wr, 4, 256, 8, lg, None) == 1                    # null x
    assert rl(x, wr, 0, 256, 8, lg, None) == 1                       # T = 0
    assert rl(x, wr, 4, 100, 8, lg, None) == 1                       # d % 8 != 0
    assert rl(x, wr, 4, 256, 0, lg, None) == 1                       # E = 0
    assert rl(x, wr, 4, 256, 300, lg, None) == 2                     # E > 256
    assert rl(x, P(0x38000008), 4, 256, 8, lg, None) == 1            # misaligned router weight
    need = L.moe_layer_workspace_bytes(16, 2, C.byref(p), None)
    fr = L.moe_layer_forward_router
    fr.argtypes = [P, P, C.c_int, C.c_int, C.c_void_p, C.c_void_p, P, P, P, C.c_size_t, P]
    assert fr(x, None, 16, 2, C.byref(p), None, lg, out, ws, need, None) == 1        # null router
    assert fr(x, wr, 16, 9, C.byref(p), None, lg, out, ws, need, None) == 1          # k > E
    assert fr(x, wr, 16, 2, C.byref(p), None, lg, out, ws, need - 1, None) == 3      # small ws
