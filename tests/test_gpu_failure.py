"""Failure paths without a GPU fault, and out-of-bounds writes without a sanitizer.

Timeouts: every wait in the grouped-GEMM kernels is bounded.  The test hook
moe_debug_gemm_fault makes the gate/up GEMM's producer stop feeding its
pipeline after a few stages and sets a 1 ms wait limit, so the consumers' waits
run out: the call must end (no hang), report MOE_DEVERR_TIMEOUT in the error
word, and leave the context usable -- the next forward is clean and matches the
oracle.  Covered on the decode kernel (int4, fp8, and the stream-K hand-off
between CTAs) and on the prefill kernel (int4, bf16).

Guard bands: the caller-owned buffers (out, the workspace, x_perm, y_perm, the
routing outputs) are placed between 4 KB sentinel regions filled with 0xA5; after
calls on ragged shapes (T and d_ff not tile multiples, the short last row chunk
of an expert, stream-K splits) every sentinel byte must be unchanged."""
import ctypes as C

import numpy as np
import pytest
import torch

import moe_expert_layer_03_gb300 as moe
import moe_synth as ms
from layer_setup import GpuLayer, assert_close_rms

pytestmark = pytest.mark.gpu

FAULT_CASES = {
    # decode kernel (row chunks of <= 32): 8 quantisation groups per item
    "int4_decode": ms.LayerConfig("int4_decode_fault", T=16, d=1024, F=512, E=8, k=2, fmt="int4", seed=81),
    "fp8_decode": ms.LayerConfig("fp8_decode_fault", T=16, d=1024, F=512, E=8, k=2, fmt="fp8", seed=82),
    # decode kernel with the stream-K split: CTAs wait for their neighbours' partial sums
    "int4_streamk": ms.LayerConfig("int4_streamk_fault", T=16, d=256, F=3200, E=8, k=2, fmt="int4", seed=17),
    # prefill kernel (wider row chunks), quantised and bf16 weights
    "int4_prefill": ms.LayerConfig("int4_prefill_fault", T=160, d=1024, F=512, E=4, k=2, fmt="int4", seed=83),
    "bf16": ms.LayerConfig("bf16_fault", T=40, d=1024, F=512, E=8, k=2, fmt="bf16", seed=84),
}


@pytest.mark.parametrize("name", list(FAULT_CASES))
def test_gemm_wait_timeout_is_reported_and_context_stays_usable(name):
    L = GpuLayer(FAULT_CASES[name])
    try:
        moe.debug_gemm_fault(stop_stage=2, wait_ns=1_000_000)
        out, ws = moe.layer_forward(L.x, L.logits, L.cfg.k, L.routed, L.shared)
        code = moe.last_device_error(ws)             # synchronises: the call has ended
    finally:
        moe.debug_gemm_fault()
    assert code & 1, f"{name}: expected the timeout bit, error word {code}"
    out, ws = L.forward()                            # same context, defaults restored
    assert moe.last_device_error(ws) == 0
    assert_close_rms(out.float().cpu().numpy(), L.oracle_forward(), what=name)


def test_debug_hook_rejects_bad_stage():
    with pytest.raises(moe.MoeError, match="invalid"):
        moe.debug_gemm_fault(stop_stage=-2)
    moe.debug_gemm_fault()


# ----------------------------------------------------------------------------- guard bands
GUARD = 4096
SENTINEL = 0xA5


class Guarded:
    """A device buffer of `nbytes` between two GUARD-byte sentinel regions."""

    def __init__(self, nbytes: int):
        self.n = nbytes
        self.buf = torch.full((nbytes + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        assert self.buf.data_ptr() % 256 == 0

    def view(self, dtype, shape) -> torch.Tensor:
        t = self.buf[GUARD:GUARD + self.n].view(dtype)
        return t.view(*shape) if shape else t

    def ptr(self):
        return C.c_void_p(self.buf.data_ptr() + GUARD)

    def check(self, what: str):
        torch.cuda.synchronize()
        b = self.buf.cpu().numpy()
        bad = np.flatnonzero(np.concatenate([b[:GUARD], b[GUARD + self.n:]]) != SENTINEL)
        assert bad.size == 0, f"{what}: {bad.size} sentinel bytes overwritten (first at {bad[0]})"


GUARD_CASES = {
    "int4_ragged": ms.LayerConfig("int4_ragged_g", T=37, d=256, F=640, E=5, k=3, fmt="int4", seed=5),
    "int4_decode_shared": ms.LayerConfig("int4_shared_g", T=24, d=384, F=256, E=16, k=4, fmt="int4",
                                         logits="zipf", zipf_s=1.1, shared=True, slot_perm=True),
    "int4_streamk_skew": ms.LayerConfig("int4_streamk_skew_g", T=32, d=256, F=2560, E=8, k=2, fmt="int4",
                                        logits="zipf", zipf_s=1.1, shared=True, slot_perm=True, seed=19),
    "fp8_chunk64": ms.LayerConfig("fp8_chunk64_g", T=96, d=256, F=384, E=8, k=2, fmt="fp8", seed=15),
    "bf16_multichunk": ms.LayerConfig("bf16_multichunk_g", T=600, d=256, F=384, E=2, k=1, fmt="bf16", seed=3),
    "int4_wide192": ms.LayerConfig("int4_wide192_g", T=200, d=256, F=384, E=2, k=1, fmt="int4", seed=8),
}


@pytest.mark.parametrize("name", list(GUARD_CASES))
def test_layer_writes_stay_inside_out_and_workspace(name):
    L = GpuLayer(GUARD_CASES[name])
    cfg = L.cfg
    need = moe.layer_workspace_bytes(cfg.T, cfg.k, L.routed, L.shared)
    g_out = Guarded(cfg.T * cfg.d * 2)
    g_ws = Guarded(need)
    out, ws = moe.layer_forward(L.x, L.logits, cfg.k, L.routed, L.shared,
                                out=g_out.view(torch.bfloat16, (cfg.T, cfg.d)), ws=g_ws.view(torch.uint8, ()))
    assert moe.last_device_error(ws) == 0
    g_out.check(f"{name} out")
    g_ws.check(f"{name} workspace")
    assert_close_rms(out.float().cpu().numpy(), L.oracle_forward(), what=name)


@pytest.mark.parametrize("name", ["int4_ragged", "fp8_chunk64", "bf16_multichunk"])
def test_separate_calls_write_inside_their_buffers(name):
    """route -> permute -> grouped_ffn -> combine with every output guarded."""
    L = GpuLayer(GUARD_CASES[name])
    cfg = L.cfg
    T, k, E, d, A = cfg.T, cfg.k, cfg.E, cfg.d, cfg.A
    lib = moe.lib()
    st = lambda: C.c_void_p(torch.cuda.current_stream().cuda_stream)
    g_idx, g_w = Guarded(A * 4), Guarded(A * 4)
    assert lib.moe_route_topk(C.c_void_p(L.logits.data_ptr()), T, E, k, g_idx.ptr(), g_w.ptr(), st()) == 0
    g_cnt, g_off, g_roa, g_tor = Guarded(E * 4), Guarded((E + 1) * 4), Guarded(A * 4), Guarded(A * 4)
    g_xp = Guarded(A * d * 2)
    g_pws = Guarded(lib.moe_permute_workspace_bytes())
    assert lib.moe_permute(g_idx.ptr(), C.c_void_p(L.x.data_ptr()), T, k, E, d, g_cnt.ptr(), g_off.ptr(),
                           g_roa.ptr(), g_tor.ptr(), g_xp.ptr(), g_pws.ptr(), g_pws.n, st()) == 0
    g_yp = Guarded(A * d * 2)
    fws = moe.grouped_ffn_workspace_bytes(A, L.routed)
    g_fws = Guarded(fws)
    assert lib.moe_grouped_ffn(g_xp.ptr(), g_off.ptr(), A, L.routed.ref, g_yp.ptr(), g_fws.ptr(), fws, st()) == 0
    g_out = Guarded(T * d * 2)
    assert lib.moe_combine(g_yp.ptr(), g_roa.ptr(), g_w.ptr(), None, T, k, d, g_out.ptr(), st()) == 0
    torch.cuda.synchronize()
    for g, what in ((g_idx, "topk_idx"), (g_w, "topk_w"), (g_cnt, "counts"), (g_off, "offsets"),
                    (g_roa, "row_of_assign"), (g_tor, "token_of_row"), (g_xp, "x_perm"),
                    (g_pws, "permute workspace"), (g_yp, "y_perm"), (g_fws, "ffn workspace"), (g_out, "out")):
        g.check(f"{name} {what}")
    assert moe.last_device_error(g_fws.view(torch.uint8, ())) == 0
    assert_close_rms(g_out.view(torch.bfloat16, (T, d)).float().cpu().numpy(), L.oracle_forward(), what=name)
