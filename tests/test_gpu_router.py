"""GPU parity of the router GEMM (logits[t][e] = x[t] . w_router[e], bf16 inputs,
fp32 sums) against the oracle's exact fp64 dot products, and of the layer
forward that starts from the token rows and the router weight.

Tolerance, from the kernels' arithmetic (the bf16 products are exact in fp32;
|got - exact| <= gamma_n * sum_i |x_i w_i| with gamma_n = n u / (1 - n u)):
  CUDA-core kernel (T <= 64, or more than 16 experts): one fixed-order fp32 sum
  whose longest chain has n = 8 * ceil(d / 2048) + 5 + 8 roundings (a thread's
  FMAs over its K vectors, the 5-step warp butterfly, the 8 warps' sums),
  u = 2^-24;
  tensor-core kernel (T * max(E, 8) >= 8192, at most 16 experts, d % 64 == 0):
  each of the 8
  K slices accumulates 4 * ceil(d / 512) MMAs of 16 products into an fp32
  accumulator, then the 8 slice sums are added in rank order.  The tensor
  pipe may truncate rather than round when it aligns and adds, so every
  addition counts with u = 2^-23, and the 16-product block sum inside one MMA
  as 16 additions: n = 4 * ceil(d / 512) + 16 + 8."""
import math

import numpy as np
import pytest
import torch

import moe_expert_layer_03_gb300 as moe
import moe_synth as ms
import oracle
from layer_setup import GpuLayer, assert_close_rms

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def _tensor_path(T: int, d: int, E: int) -> bool:
    return E <= 16 and d % 64 == 0 and T * max(E, 8) >= 8192


def _gamma(T: int, d: int, E: int) -> float:
    if _tensor_path(T, d, E):
        n, u = 4 * math.ceil(d / 512) + 16 + 8, 2.0 ** -23
    else:
        n, u = 8 * math.ceil(d / 2048) + 5 + 8, U
    return n * u / (1 - n * u)


def _abs_dot(x: torch.Tensor, w: torch.Tensor) -> np.ndarray:
    """sum_i |x[t][i] w[e][i]| (the scale of the summation error), [T, E]."""
    xa = x.cpu().double().abs().numpy()
    wa = w.cpu().double().abs().numpy()
    return xa @ wa.T


def _draw(T, d, E, seed):
    g = np.random.default_rng(seed)
    x = torch.from_numpy(g.standard_normal((T, d), dtype=np.float32)).to(torch.bfloat16)
    w = torch.from_numpy(g.standard_normal((E, d), dtype=np.float32) * np.float32(0.02)).to(torch.bfloat16)
    return x, w


def _check_logits(got: torch.Tensor, x: torch.Tensor, w: torch.Tensor, what: str):
    want = oracle.router_logits(x.cpu(), w.cpu())
    bound = _gamma(x.shape[0], x.shape[1], w.shape[0]) * _abs_dot(x, w) + 1e-30
    err = np.abs(got.double().cpu().numpy() - want)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), f"{what}: |err| {err[worst]:.3e} > bound {bound[worst]:.3e} at {worst}"
    return want, bound


@pytest.mark.parametrize("T,d,E", [
    (16, 4096, 8),      # Mixtral-shaped decode
    (16, 5120, 128),    # 125B-class decode
    (2048, 4096, 8),    # Mixtral-shaped prefill chunk (tensor cores)
    (256, 4096, 16),    # Phi-3.5-MoE-shaped prefill chunk (CUDA cores: below the crossover)
    (600, 1024, 16),    # tensor cores, N = E = 16, ragged last token tile
    (4133, 4096, 8),    # tensor cores, more clusters than SMs, ragged last token tile
    (1100, 64, 3),      # tensor cores: one K step, so seven of the eight K slices are empty
    (1030, 576, 9),     # tensor cores: 9 K steps over 8 slices, E not a multiple of 4
    (1024, 1024, 17),   # just past the tensor path (E > 16): the CUDA-core kernel
    (37, 392, 5),       # ragged: T not a tile multiple, d not a multiple of 128, E < 8
    (1, 256, 1),        # one token, one expert
    (301, 1024, 256),   # the largest E, ragged last token tile
    (9, 8, 13),         # d = one 16-byte vector
])
def test_router_logits_vs_oracle(T, d, E):
    x, w = _draw(T, d, E, seed=T * 7 + E)
    xd, wd = x.cuda(), w.cuda()
    got = moe.router_logits(xd, wd)
    torch.cuda.synchronize()
    _check_logits(got, x, w, f"T={T} d={d} E={E}")


def test_router_logits_reproducible_and_row_independent():
    """Fixed summation order: the same call twice gives the same bits, and a
    token's logits do not depend on which other tokens share its launch."""
    x, w = _draw(64, 2048, 24, seed=5)
    xd, wd = x.cuda(), w.cuda()
    a = moe.router_logits(xd, wd)
    b = moe.router_logits(xd, wd)
    one = moe.router_logits(xd[17:18].contiguous(), wd)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(a[17:18], one)


def test_tensor_core_router_reproducible_and_row_independent():
    """The tensor-core router: the same bits twice, and a token's logits do not
    depend on its row inside the 128-token tile or on the other tokens."""
    x, w = _draw(1300, 4096, 8, seed=6)
    xd, wd = x.cuda(), w.cuda()
    a = moe.router_logits(xd, wd)
    b = moe.router_logits(xd, wd)
    tail = moe.router_logits(xd[100:].contiguous(), wd)        # 1200 tokens, shifted by 100 rows
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(a[100:], tail)


def test_tensor_core_router_wait_timeout_gives_nan_and_context_stays_usable():
    """Bounded waits: with the fault hook the router's TMA producer stops after
    two K steps, the MMA warp's wait runs out after 1 ms and the tiles' logits
    come out NaN (the call ends, no hang); afterwards the same call is exact."""
    x, w = _draw(1024, 4096, 8, seed=8)
    xd, wd = x.cuda(), w.cuda()
    try:
        moe.debug_gemm_fault(stop_stage=2, wait_ns=1_000_000)
        bad = moe.router_logits(xd, wd)
        torch.cuda.synchronize()
    finally:
        moe.debug_gemm_fault()
    assert torch.isnan(bad).all()
    got = moe.router_logits(xd, wd)
    torch.cuda.synchronize()
    _check_logits(got, x, w, "after the timeout")


@pytest.mark.parametrize("name", ["tiny_int4", "int4_shared_perm", "int4_ragged", "fused_route_max",
                                  "fused_route_bf16", "large_E_decode", "prefill_chunk", "prefill_long",
                                  "prefill_long_e16"])
def test_layer_forward_router(name):
    """The layer from x and the router weight: logits within the bound above,
    then every token whose top-k choice is unambiguous under that bound routed as
    the oracle routes its own logits, and its output within 2e-2 RMS."""
    from test_gpu_layer import SMALL
    extra = {
        # E > 32 and the shared expert on the fused path
        "large_E_decode": ms.LayerConfig("large_E_decode", T=16, d=512, F=256, E=128, k=8, fmt="int4",
                                         logits="zipf", zipf_s=1.1, shared=True, slot_perm=True, seed=71),
        # more than 64 tokens: the router GEMM as its own launch (CUDA cores)
        "prefill_chunk": ms.LayerConfig("prefill_chunk", T=200, d=384, F=256, E=8, k=2, fmt="int4", seed=72),
        # a long chunk: the tensor-core router, with the top-k gating in its launch
        "prefill_long": ms.LayerConfig("prefill_long", T=1100, d=384, F=256, E=8, k=2, fmt="int4", seed=73),
        # the same at N = E = 16, top-4, with the shared expert
        "prefill_long_e16": ms.LayerConfig("prefill_long_e16", T=600, d=256, F=256, E=16, k=4, fmt="int4",
                                           shared=True, seed=74),
    }
    cfg = SMALL[name] if name in SMALL else extra[name]
    L = GpuLayer(cfg)
    wr = ms.make_router_weight(cfg)
    out, logits, ws = moe.layer_forward_router(L.x, wr.to(L.dev), cfg.k, L.routed, L.shared)
    torch.cuda.synchronize()
    assert moe.last_device_error(ws) == 0
    want_lg, bound = _check_logits(logits, L.x, wr, name)
    # the same bits as the standalone router GEMM (same tiling, same sum order)
    assert torch.equal(logits, moe.router_logits(L.x, wr.to(L.dev)))
    # and the same layer output as moe_layer_forward on those logits
    out2, _ = moe.layer_forward(L.x, logits, cfg.k, L.routed, L.shared)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))

    # tokens whose k + 1 largest exact logits are pairwise further apart than two
    # bounds (the chosen set and its order cannot depend on the rounding)
    toks = []
    for t in range(cfg.T):
        s = np.sort(want_lg[t])[::-1][: cfg.k + 1]
        if np.all(np.diff(s) < -2 * bound[t].max()):
            toks.append(t)
    assert len(toks) >= cfg.T - 1, "synthetic router logits should be unambiguous"

    lg32 = want_lg.astype(np.float32)
    idx_gpu, _ = moe.route_topk(logits, cfg.k)
    idx_ref, _ = oracle.route_topk(lg32, cfg.k)
    np.testing.assert_array_equal(idx_gpu.cpu().numpy()[toks], idx_ref[toks])

    L.logits_np = lg32
    assert_close_rms(out.float().cpu().numpy()[toks], L.oracle_forward(toks), what=name)


def test_layer_router_launch_count():
    """Launches of one layer_forward_router call: the router inside the routing
    launch for T <= 64; its own launch above; on the tensor cores that launch
    also does the top-k gating, in place of the routing launch."""
    cases = [(ms.LayerConfig("lc_decode", T=16, d=256, F=256, E=8, k=2, fmt="int4", seed=75), 0),
             (ms.LayerConfig("lc_cuda_cores", T=200, d=256, F=256, E=8, k=2, fmt="int4", seed=76), 1),
             (ms.LayerConfig("lc_tensor", T=1100, d=256, F=256, E=8, k=2, fmt="int4", seed=77), 0),
             (ms.LayerConfig("lc_wide_E", T=1100, d=256, F=256, E=32, k=2, fmt="int4", seed=78), 1)]
    for cfg, extra in cases:
        L = GpuLayer(cfg)
        n = moe.layer_launch_count(cfg.T, cfg.k, L.routed, L.shared)
        assert moe.layer_router_launch_count(cfg.T, cfg.k, L.routed, L.shared) == n + extra, cfg.name


@pytest.mark.parametrize("T", [200, 1100])   # CUDA-core router + routing kernel; tensor-core router with its top-k
def test_router_ties_and_non_finite_rows_match_the_routing_kernel(T):
    """Duplicate router rows (experts 1 and 2, 3 and 5: equal logits wherever
    the two sums round alike, and then the lower index must win) and rows whose
    logits are not finite (an inf in x) must be routed by the same rule on both
    router paths: the layer output equals moe_layer_forward on the returned
    logits bit for bit, and the routing of every finite row equals the oracle's
    on those logits."""
    cfg = ms.LayerConfig(f"ties_{T}", T=T, d=384, F=256, E=8, k=2, fmt="int4", seed=79)
    L = GpuLayer(cfg)
    wr = ms.make_router_weight(cfg)
    wr[2] = wr[1]
    wr[5] = wr[3]
    x = L.x.clone()
    x[7, 11] = float("inf")
    x[T - 3, 0] = float("-inf")
    out, logits, ws = moe.layer_forward_router(x, wr.to(L.dev), cfg.k, L.routed, L.shared)
    out2, _ = moe.layer_forward(x, logits, cfg.k, L.routed, L.shared)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    lg = logits.cpu().numpy()
    finite = np.all(np.isfinite(lg), axis=1)
    assert not finite[7] and not finite[T - 3]
    idx_gpu, w_gpu = moe.route_topk(logits, cfg.k)
    idx_ref, w_ref = oracle.route_topk(lg[finite], cfg.k)
    np.testing.assert_array_equal(idx_gpu.cpu().numpy()[finite], idx_ref)
    np.testing.assert_allclose(w_gpu.cpu().numpy()[finite], w_ref, rtol=2e-6, atol=0)
