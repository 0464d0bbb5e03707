"""The allocation-free layer forward (moe_layer_forward_noalloc).

Some callers cannot allocate device memory when they run the layer: code inside
stream capture, hosts that own all device memory through their own pool, and
real-time loops that forbid allocation latency.  For them the library keeps a
fixed scratch array on every device and needs only the inputs and outputs.
This file checks, through the C ABI, that the variant gives the same output as
moe_layer_forward (which takes a caller-provided workspace) on two calls in a
row -- bit for bit, since both run the same kernels on the same layout -- that
its device-side error word can be read back without a workspace pointer, and
that a call too large for the fixed scratch is refused before any launch.  It is collected last on purpose and also passes alone in a fresh
process (the per-device set-up happens on the first call).
"""
import ctypes as C

import numpy as np
import pytest
import torch

import moe_expert_layer_03_gb300 as moe
import moe_synth as ms
from layer_setup import GpuLayer, assert_close_rms

pytestmark = pytest.mark.gpu

P = C.c_void_p


def _noalloc_fn():
    f = moe.lib().moe_layer_forward_noalloc
    f.argtypes = [P, P, C.c_int, C.c_int, C.POINTER(moe.MoePool), C.POINTER(moe.MoePool), P, P]
    f.restype = C.c_int
    return f


def _call(L: GpuLayer, out: torch.Tensor) -> int:
    cfg = L.cfg
    return _noalloc_fn()(P(L.x.data_ptr()), P(L.logits.data_ptr()), cfg.T, cfg.k, L.routed.ref,
                         L.shared.ref if L.shared is not None else None, P(out.data_ptr()),
                         P(torch.cuda.current_stream().cuda_stream))


CASES = {
    "tiny_bf16": ms.CONFIGS["tiny"],
    "int4_shared": ms.LayerConfig("int4_shared", T=16, d=512, F=384, E=16, k=4, fmt="int4",
                                  logits="zipf", zipf_s=1.1, shared=True, slot_perm=True),
}


def _last_error() -> tuple[int, int]:
    f = moe.lib().moe_noalloc_last_device_error
    f.argtypes = [C.POINTER(C.c_int), P]
    f.restype = C.c_int
    code = C.c_int(-1)
    st = f(C.byref(code), P(torch.cuda.current_stream().cuda_stream))
    return st, code.value


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_layer_forward_on_two_calls(name):
    L = GpuLayer(CASES[name])
    ref, ws = L.forward()
    assert moe.last_device_error(ws) == 0
    want = ref.float().cpu().numpy()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _call(L, out) == 0
        torch.cuda.synchronize()
        assert _last_error() == (0, 0)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert_close_rms(out.float().cpu().numpy(), want, what=f"{name} noalloc")


def test_noalloc_device_error_is_readable():
    """A token routed to an expert whose slot is out of range raises the
    slot-range bit (4) in the scratch's error word; the next clean call clears it."""
    L = GpuLayer(CASES["int4_shared"])
    cfg = L.cfg
    table = torch.from_numpy(L.e2s_np.astype(np.int32)).to("cuda")
    table[int(L.logits_np[0].argmax())] = 999            # token 0's first expert
    bad = L.pool.view(table)
    out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    st = _noalloc_fn()(P(L.x.data_ptr()), P(L.logits.data_ptr()), cfg.T, cfg.k, bad.ref, L.shared.ref,
                       P(out.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    st, code = _last_error()
    assert st == 5 and code & 4                          # MOE_ERR_DEVICE, slot out of range
    assert _call(L, out) == 0
    assert _last_error() == (0, 0)


def test_noalloc_rejects_a_call_beyond_its_scratch():
    cfg = ms.CONFIGS["tiny"]
    L = GpuLayer(cfg)
    big = 40000                                      # x_perm alone needs 2 * 40000 * 256 * 2 B > 16 MiB
    x = torch.zeros(big, cfg.d, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(big, cfg.E, dtype=torch.float32, device="cuda")
    out = torch.empty(big, cfg.d, dtype=torch.bfloat16, device="cuda")
    need = moe.layer_workspace_bytes(big, cfg.k, L.routed)
    assert need > (16 << 20)
    st = _noalloc_fn()(P(x.data_ptr()), P(lg.data_ptr()), big, cfg.k, L.routed.ref, None,
                       P(out.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert st == 3                                   # MOE_ERR_WORKSPACE, nothing launched
