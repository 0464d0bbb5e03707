"""GPU parity: the grouped SwiGLU FFN, the combine and the whole layer against the
oracle, within max|err| <= 2e-2 * RMS(out) (bf16 activations, fp32 accumulation).

Small cases run the oracle on every token; the workload shapes run at full size
in the bench's launch configuration: every token at decode, and at prefill the
tokens at both ends of every expert's every row chunk."""
import numpy as np
import pytest
import torch

import moe_expert_layer_03_gb300 as moe
import moe_synth as ms
import oracle
from layer_setup import HOST_THREADS, GpuLayer, assert_close_rms, bf16_ulp, chunk_edge_tokens

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": ms.CONFIGS["tiny"],
    "tiny_int4": ms.CONFIGS["tiny"].with_(name="tiny_int4", fmt="int4"),
    "int4_shared_perm": ms.LayerConfig("int4_shared_perm", T=24, d=384, F=256, E=16, k=4,
                                       fmt="int4", logits="zipf", zipf_s=1.1, shared=True,
                                       slot_perm=True),
    "bf16_multichunk": ms.LayerConfig("bf16_multichunk", T=600, d=256, F=384, E=2, k=1,
                                      fmt="bf16", seed=3),                 # >256 rows per expert
    "int4_ragged": ms.LayerConfig("int4_ragged", T=37, d=256, F=640, E=5, k=3, fmt="int4",
                                  seed=5),                                 # T, F not tile multiples
    "k_equals_E": ms.LayerConfig("k_equals_E", T=9, d=128, F=128, E=4, k=4, fmt="bf16", seed=2),
    "single_token": ms.LayerConfig("single_token", T=1, d=256, F=256, E=8, k=2, fmt="int4"),
    "dense_E1": ms.LayerConfig("dense_E1", T=20, d=256, F=512, E=1, k=1, fmt="int4"),
    # row chunks of 32 (int4 group-scaled main loop at its wider width)
    "int4_chunk32": ms.LayerConfig("int4_chunk32", T=48, d=384, F=512, E=8, k=2, fmt="int4", seed=4),
    # row chunks of 64 (int4 prefill kernel: fp16 A tiles in TMEM, paired down tiles)
    "int4_chunk64": ms.LayerConfig("int4_chunk64", T=96, d=256, F=384, E=8, k=2, fmt="int4", seed=6),
    # row chunks of 128 with an odd number of output tiles (one down tile per item)
    "int4_wide_odd": ms.LayerConfig("int4_wide_odd", T=96, d=384, F=512, E=4, k=2, fmt="int4", seed=7),
    # row chunks of 192, the widest int4 chunk
    "int4_wide192": ms.LayerConfig("int4_wide192", T=200, d=256, F=384, E=2, k=1, fmt="int4", seed=8),
    # the one-launch routing + gather at its limits: 64 tokens, k = 16, a shared
    # expert (1088 rows, more than one per CTA), fp16 rows for the int4 prefill kernel
    "fused_route_max": ms.LayerConfig("fused_route_max", T=64, d=256, F=256, E=16, k=16, fmt="int4",
                                      shared=True, seed=10),
    # the same launch writing bf16 rows, k < E
    "fused_route_bf16": ms.LayerConfig("fused_route_bf16", T=64, d=256, F=256, E=32, k=6, fmt="bf16",
                                       seed=11),
    # 8-bit experts: decode kernel (A read from shared memory) at 16- and 32-row
    # chunks, paired and single down tiles (d/128 odd: a pair block, then a
    # tile alone), the shared expert and a permuted slot table
    "fp8_tiny": ms.CONFIGS["tiny"].with_(name="fp8_tiny", fmt="fp8"),
    "fp8_shared_perm": ms.LayerConfig("fp8_shared_perm", T=24, d=384, F=256, E=16, k=4, fmt="fp8",
                                      logits="zipf", zipf_s=1.1, shared=True, slot_perm=True, seed=13),
    "fp8_chunk32": ms.LayerConfig("fp8_chunk32", T=48, d=256, F=640, E=8, k=2, fmt="fp8", seed=14),
    # ... and the prefill kernel (fp16 A dequantised into TMEM): paired and odd tile counts
    "fp8_chunk64": ms.LayerConfig("fp8_chunk64", T=96, d=256, F=384, E=8, k=2, fmt="fp8", seed=15),
    "fp8_wide_odd": ms.LayerConfig("fp8_wide_odd", T=96, d=384, F=512, E=4, k=2, fmt="fp8", seed=16),
    # decode gate/up with ~200 work items on the persistent CTAs: a short last
    # wave, so the GEMM splits the items' groups evenly (stream-K) and CTAs hand
    # partial sums of the items cut between them to their neighbours
    "int4_streamk": ms.LayerConfig("int4_streamk", T=16, d=256, F=3200, E=8, k=2, fmt="int4", seed=17),
    "fp8_streamk": ms.LayerConfig("fp8_streamk", T=16, d=384, F=3200, E=8, k=2, fmt="fp8", seed=18),
    # stream-K with skewed routing: row chunks with more than half a tile of
    # rows next to small ones, experts with two row chunks and the shared
    # expert in tile-major order; and 32-row chunks
    "int4_streamk_skew": ms.LayerConfig("int4_streamk_skew", T=32, d=256, F=2560, E=8, k=2, fmt="int4",
                                        logits="zipf", zipf_s=1.1, shared=True, slot_perm=True, seed=19),
    "int4_streamk_g32": ms.LayerConfig("int4_streamk_g32", T=24, d=256, F=11136, E=3, k=2, fmt="int4",
                                       seed=20),
    # more than 256 tokens, top-4 and the shared expert: the combine's
    # all-rows-in-flight path for one K split at prefill widths
    "int4_prefill_shared_k4": ms.LayerConfig("int4_prefill_shared_k4", T=300, d=256, F=384, E=8, k=4,
                                             fmt="int4", shared=True, seed=21),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_small_all_tokens(name):
    L = GpuLayer(SMALL[name])
    out, ws = L.forward()
    assert moe.last_device_error(ws) == 0
    assert_close_rms(out.float().cpu().numpy(), L.oracle_forward(), what=name)


# Activation stress: each weight format on each GEMM path (decode kernel: row
# chunks of <= 32; prefill kernel: wider chunks) with token rows far from N(0,1).
STRESS_PATHS = {
    "int4_decode": ms.LayerConfig("int4_decode", T=16, d=512, F=768, E=8, k=2, fmt="int4", seed=51),
    "int4_prefill": ms.LayerConfig("int4_prefill", T=163, d=512, F=768, E=8, k=2, fmt="int4", seed=52),
    "fp8_decode": ms.LayerConfig("fp8_decode", T=16, d=512, F=768, E=8, k=2, fmt="fp8", seed=53),
    "fp8_prefill": ms.LayerConfig("fp8_prefill", T=163, d=512, F=768, E=8, k=2, fmt="fp8", seed=54),
    "bf16": ms.LayerConfig("bf16", T=40, d=512, F=768, E=8, k=2, fmt="bf16", seed=55),
    "int4_decode_shared": ms.LayerConfig("int4_decode_shared", T=12, d=384, F=512, E=16, k=4, fmt="int4",
                                         logits="zipf", zipf_s=1.1, shared=True, slot_perm=True, seed=56),
}
STRESS_X = {"outlier100": dict(x_dist="outlier", x_outlier=100.0),
            "outlier1000": dict(x_dist="outlier", x_outlier=1000.0),
            "wide": dict(x_dist="wide"), "tiny": dict(x_dist="tiny"), "onehot": dict(x_dist="onehot"),
            # every element about 200: gate and up near 250, |h| above fp16's 65504
            "scaled200": dict(x_dist="scaled", x_outlier=200.0)}


@pytest.mark.parametrize("dist", list(STRESS_X))
@pytest.mark.parametrize("path", list(STRESS_PATHS))
def test_activation_stress(path, dist):
    """Rows with outlier channels (x100, x1000), rows spanning 2^-20 .. 2^10,
    all-tiny rows (1e-6), rows of large values (200 N(0,1), whose h exceeds
    fp16's range unless scaled) and rows with one nonzero element: every token
    against the oracle within the layer's bound, on every GEMM path."""
    cfg = STRESS_PATHS[path].with_(name=f"{path}_{dist}", **STRESS_X[dist])
    L = GpuLayer(cfg)
    out, ws = L.forward()
    assert moe.last_device_error(ws) == 0
    assert_close_rms(out.float().cpu().numpy(), L.oracle_forward(), what=cfg.name)


@pytest.mark.parametrize("name", ["tiny", "tiny_int4", "int4_ragged", "bf16_multichunk"])
def test_grouped_ffn_and_combine_entry_points(name):
    """route -> permute -> grouped_ffn -> combine through the separate ABI calls:
    y_perm (bf16) row by row against the oracle's expert FFN of that row's expert,
    and the combine against the oracle's combine of the same bf16 y_perm rows."""
    L = GpuLayer(SMALL[name])
    cfg = L.cfg
    idx, w = moe.route_topk(L.logits, cfg.k)
    perm = moe.permute(idx, L.x, cfg.E)
    y_perm, ws = moe.grouped_ffn(perm["x_perm"], perm["offsets"], L.routed)
    out = moe.combine(y_perm, perm["row_of_assign"], w)
    torch.cuda.synchronize()
    assert moe.last_device_error(ws) == 0
    tor = perm["token_of_row"].cpu().numpy()
    offs = perm["offsets"].cpu().numpy()
    roa = perm["row_of_assign"].cpu().numpy()
    yp = y_perm.float().cpu().numpy()
    yb = y_perm.cpu().view(torch.int16).numpy().view(np.uint16)
    rows = np.linspace(0, cfg.A - 1, min(cfg.A, 24)).astype(int)
    for r in rows:
        e = int(np.searchsorted(offs, r, side="right") - 1)
        _, y = oracle.expert_ffn(L.x[tor[r]].cpu(), L.ref(e), cfg.d, cfg.F)
        assert_close_rms(yp[r], y, what=f"{name} row {r}")
    wc = w.cpu().numpy()
    oc = out.float().cpu().numpy()
    for t in range(min(cfg.T, 16)):
        want = oracle.combine_row([yb[roa[t * cfg.k + j]] for j in range(cfg.k)], wc[t])
        assert_close_rms(oc[t], want, what=f"{name} combine token {t}")


@pytest.mark.parametrize("fmt", ["int4", "fp8", "bf16"])
def test_slot_trailer_bounds(fmt):
    """The prepack's slot trailer: the largest row L1 norm of the dequantised
    gate and up weights (numpy float64 from the canonical weights, to fp32
    rounding) and its bound exponent ceil(log2(L (1 + 2^-7))); zero for bf16."""
    cfg = ms.LayerConfig("trailer", T=1, d=384, F=640, E=1, k=1, fmt=fmt, seed=61)
    w = ms.expert_weights(cfg, 0, "cuda")
    pool = moe.ExpertPool(1, cfg.d, cfg.F, cfg.fmt)
    pool.load_expert(0, w)
    torch.cuda.synchronize()
    tr = pool.buf[pool.slot_bytes - 256:pool.slot_bytes].cpu().numpy()
    L = tr[:8].view(np.float32)
    B = tr[8:16].view(np.int32)
    if fmt == "bf16":
        assert not tr.any()
        return
    for m, name in enumerate(("gate", "up")):
        q = w[name]["q"].cpu().numpy()
        s = np.repeat(w[name]["scale"].cpu().float().numpy().astype(np.float64), 128, axis=1)
        if fmt == "int4":
            codes = np.empty((q.shape[0], q.shape[1] * 2), np.float64)
            codes[:, 0::2] = q & 15
            codes[:, 1::2] = q >> 4
            z = np.repeat(w[name]["zero"].cpu().float().numpy().astype(np.float64), 128, axis=1)
            deq = (codes - z) * s
        else:
            deq = torch.from_numpy(q).view(torch.float8_e4m3fn).float().numpy().astype(np.float64) * s
        want = np.abs(deq).sum(axis=1).max()
        assert abs(float(L[m]) - want) <= 1e-5 * want
        assert int(B[m]) == int(np.ceil(np.log2(float(L[m]) * (1 + 2.0 ** -7))))


@pytest.mark.parametrize("T,k,d", [(5, 3, 256), (16, 8, 5120), (3, 16, 384)])
def test_combine_with_shared_rows(T, k, d):
    """The combine against the oracle's exact sum of the same bf16 rows and fp32
    weights, held to its own error: half a bf16 ulp of the result (the final
    rounding) plus the fp32 evaluation of k products and k sums,
    (2k + 1) 2^-24 sum_j |w_j y_j| + |y_shared| (a weight off by 1% fails)."""
    g = torch.Generator(device="cuda").manual_seed(T * 1000 + k)
    y = torch.randn(T * k, d, device="cuda", generator=g).to(torch.bfloat16)
    sh = torch.randn(T, d, device="cuda", generator=g).to(torch.bfloat16)
    roa = torch.randperm(T * k, device="cuda", generator=g).to(torch.int32)
    w = torch.softmax(torch.randn(T, k, device="cuda", generator=g), dim=1)
    out = moe.combine(y, roa, w, sh).float().cpu().numpy().astype(np.float64)
    yc, shc, roac, wc = y.cpu(), sh.cpu(), roa.cpu().numpy(), w.cpu().numpy()
    u = 2.0 ** -24
    for t in range(T):
        bits = [yc[roac[t * k + j]].view(torch.int16).numpy().view(np.uint16) for j in range(k)]
        want = oracle.combine_row(bits, wc[t], shc[t].view(torch.int16).numpy().view(np.uint16))
        mag = sum(np.abs(wc[t][j] * yc[roac[t * k + j]].float().numpy().astype(np.float64)) for j in range(k))
        mag = mag + np.abs(shc[t].float().numpy().astype(np.float64))
        allowed = 0.5 * bf16_ulp(np.maximum(np.abs(want), np.abs(out[t]))) + (2 * k + 1) * u * mag
        err = np.abs(out[t] - want)
        i = int(np.argmax(err / allowed))
        assert np.all(err <= allowed), f"token {t}: |err| {err[i]:.3e} > {allowed[i]:.3e} at {i}"


@pytest.mark.parametrize("name", ["mixtral_decode", "fg125b_decode", "mixtral_decode_fp8"])
def test_layer_full_size_decode_every_token(name):
    """The decode workloads at full size, in the bench's launch configuration:
    every token against the oracle (run on all host cores)."""
    cfg = ms.CONFIGS[name]
    L = GpuLayer(cfg)
    out, ws = L.forward()
    assert moe.last_device_error(ws) == 0
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert_close_rms(got, L.oracle_forward(threads=HOST_THREADS), what=name)


@pytest.mark.parametrize("name", ["phi35_prefill", "mixtral_prefill", "mixtral_prefill_fp8"])
def test_layer_full_size_prefill_every_row_chunk(name):
    """The prefill workloads at full size: the tokens holding the first and the
    last row of every row chunk of every expert (so each expert's first, middle
    and short last chunk is compared), against the oracle."""
    cfg = ms.CONFIGS[name]
    L = GpuLayer(cfg)
    out, ws = L.forward()
    assert moe.last_device_error(ws) == 0
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    toks = chunk_edge_tokens(cfg, L.logits_np)
    assert len(toks) >= cfg.E
    assert_close_rms(got[toks], L.oracle_forward(toks, threads=HOST_THREADS), what=name)


@pytest.mark.parametrize("cfg", [
    # the largest supported d_model (K = 32768 for gate/up: 256 quantisation groups)
    ms.LayerConfig("max_d", T=5, d=32768, F=128, E=2, k=1, fmt="int4", seed=31),
    # the largest supported d_ff (256 output tiles for gate/up, K = 32768 for down)
    ms.LayerConfig("max_f", T=5, d=128, F=32768, E=2, k=2, fmt="fp8", seed=32),
    # many assignments: 160000 rows through the multi-tile permutation and GEMMs
    ms.LayerConfig("large_A", T=20000, d=128, F=128, E=64, k=8, fmt="bf16", seed=33),
    # prefill-size layers on the persistent full-tile kernels: about 256 down
    # work items (one whole wave and a short last one) and 128 (fewer than CTAs)
    ms.LayerConfig("int4_prefill_tail", T=1024, d=4096, F=1024, E=8, k=2, fmt="int4", seed=34),
    ms.LayerConfig("int4_prefill_allsplit", T=512, d=4096, F=1024, E=8, k=2, fmt="int4", seed=36),
    ms.LayerConfig("bf16_prefill_tail", T=512, d=4096, F=1024, E=8, k=2, fmt="bf16", seed=35),
], ids=lambda c: c.name)
def test_size_limits_sampled(cfg):
    L = GpuLayer(cfg)
    out, ws = L.forward()
    assert moe.last_device_error(ws) == 0
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    toks = sorted({0, 1, cfg.T // 2, cfg.T - 1})
    assert_close_rms(got[toks], L.oracle_forward(toks), what=cfg.name)


def test_many_items_per_cta():
    """256 experts with d_ff = 8192 give the decode gate/up GEMM about 90 work
    items per persistent CTA, more than the per-CTA item table holds, so the
    items past it are decoded on the fly; sampled tokens against the oracle."""
    cfg = ms.LayerConfig("many_items", T=64, d=256, F=8192, E=256, k=8, fmt="int4", seed=12)
    L = GpuLayer(cfg)
    out, ws = L.forward()
    assert moe.last_device_error(ws) == 0
    got = out.float().cpu().numpy()
    toks = [0, 31, 63]
    assert_close_rms(got[toks], L.oracle_forward(toks), what=cfg.name)


@pytest.mark.parametrize("fmt", ["bf16", "int4"])
def test_one_expert_takes_every_token(fmt):
    """50 tokens on expert 0 of 16 (B tile of 16 rows -> 4 row chunks), 15 experts idle."""
    cfg = ms.LayerConfig("skew", T=50, d=256, F=256, E=16, k=1, fmt=fmt, seed=9)
    lg = ms.make_logits(cfg)
    lg[:, 0] = 10.0
    L = GpuLayer(cfg, logits=lg)
    out, ws = L.forward()
    assert moe.last_device_error(ws) == 0
    assert_close_rms(out.float().cpu().numpy(), L.oracle_forward(), what="skew")


def test_slot_permutation_is_bit_identical():
    cfg = SMALL["int4_shared_perm"]
    a = GpuLayer(cfg)
    out_a, _ = a.forward()
    b = GpuLayer(cfg, e2s=np.roll(a.e2s_np, 5))
    out_b, _ = b.forward()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


def test_token_permutation_permutes_rows():
    cfg = SMALL["int4_ragged"]
    a = GpuLayer(cfg)
    out_a, _ = a.forward()
    perm = np.random.default_rng(1).permutation(cfg.T)
    b = GpuLayer(cfg, logits=a.logits_np[perm])
    b.x = a.x[torch.from_numpy(perm).to("cuda")].contiguous()
    out_b, _ = b.forward()
    assert torch.equal(out_b.view(torch.int16), out_a[torch.from_numpy(perm).to("cuda")].view(torch.int16))


def test_slot_out_of_range_sets_device_error():
    cfg = SMALL["tiny_int4"]
    L = GpuLayer(cfg)
    bad = L.pool.view(torch.tensor([0, 1, 2, 3, 4, 5, 6, 99], dtype=torch.int32, device="cuda"))
    out, ws = moe.layer_forward(L.x, L.logits, cfg.k, bad)
    assert moe.last_device_error(ws) & 4
    out, ws = L.forward()                     # the context is still usable afterwards
    assert moe.last_device_error(ws) == 0


def test_host_side_rejections():
    cfg = SMALL["tiny"]
    L = GpuLayer(cfg)
    need = moe.layer_workspace_bytes(cfg.T, cfg.k, L.routed)
    with pytest.raises(moe.MoeError, match="workspace"):
        moe.layer_forward(L.x, L.logits, cfg.k, L.routed, ws=moe.workspace(need - 1024))
    with pytest.raises(moe.MoeError, match="invalid"):
        moe.layer_forward(L.x, L.logits, cfg.E + 1, L.routed)
    xs = torch.empty(cfg.T * cfg.d + 8, dtype=torch.bfloat16, device="cuda")[1:1 + cfg.T * cfg.d]
    with pytest.raises(moe.MoeError, match="invalid"):
        moe.layer_forward(xs.view(cfg.T, cfg.d), L.logits, cfg.k, L.routed)


@pytest.mark.parametrize("name", ["tiny", "int4_shared_perm", "int4_ragged"])
def test_layer_graph_replay(name):
    """The captured layer (moe.LayerGraph) gives the eager call's output bit for
    bit, and one capture serves new inputs: replaying after new x and logits
    have been copied in re-routes on the device and matches the oracle."""
    L = GpuLayer(SMALL[name])
    cfg = L.cfg
    g = moe.LayerGraph(cfg.T, cfg.k, L.routed, L.shared)
    g.x.copy_(L.x)
    g.logits.copy_(L.logits)
    out_g = g.replay().clone()
    out_e, _ = L.forward()
    torch.cuda.synchronize()
    assert moe.last_device_error(g.ws) == 0
    assert torch.equal(out_g, out_e)

    # new inputs: another seed's tokens and logits, same experts, same graph
    cfg2 = cfg.with_(seed=cfg.seed + 101)
    L.x = ms.make_x(cfg2).to(L.dev)
    L.logits_np = ms.make_logits(cfg2)
    L.logits = torch.from_numpy(L.logits_np).to(L.dev)
    g.x.copy_(L.x)
    g.logits.copy_(L.logits)
    out2 = g.replay().clone()
    torch.cuda.synchronize()
    assert moe.last_device_error(g.ws) == 0
    assert_close_rms(out2.float().cpu().numpy(), L.oracle_forward(), what=name + " (new inputs)")


@pytest.mark.parametrize("fmt,E,k", [("int4", 64, 2), ("fp8", 32, 2), ("bf16", 32, 6), ("int4", 256, 4)])
def test_one_launch_routing_matches_separate_kernels(fmt, E, k):
    """Up to 64 tokens route, permute and gather in one launch; 65 tokens take the
    separate kernels.
    The same 64 tokens plus a copy of token 0 must give the first 64 output rows
    bit for bit (same experts and row-chunk width, so the same GEMM tiling)."""
    cfg = ms.LayerConfig("fused_vs_split", T=64, d=256, F=256, E=E, k=k, fmt=fmt, seed=41 + E)
    L = GpuLayer(cfg)
    out64, ws64 = L.forward()
    x65 = torch.cat([L.x, L.x[:1]], 0).contiguous()
    lg65 = torch.cat([L.logits, L.logits[:1]], 0).contiguous()
    out65, ws65 = moe.layer_forward(x65, lg65, cfg.k, L.routed, L.shared)
    torch.cuda.synchronize()
    assert moe.last_device_error(ws64) == 0 and moe.last_device_error(ws65) == 0
    assert torch.equal(out64.view(torch.int16), out65[:64].view(torch.int16))
    assert_close_rms(out64.float().cpu().numpy()[:8], L.oracle_forward(range(8)), what=cfg.name)


def test_layer_graph_host_io():
    """The captured step with its host copies (LayerGraph(host_io=True)): inputs
    from pinned host buffers, output back to one, bit-identical to the eager call."""
    L = GpuLayer(SMALL["int4_shared_perm"])
    cfg = L.cfg
    g = moe.LayerGraph(cfg.T, cfg.k, L.routed, L.shared, host_io=True)
    g.x_host.copy_(L.x.cpu())
    g.logits_host.copy_(L.logits.cpu())
    g.replay()
    torch.cuda.synchronize()
    out_e, _ = L.forward()
    assert moe.last_device_error(g.ws) == 0
    assert torch.equal(g.out_host.view(torch.int16), out_e.cpu().view(torch.int16))


@pytest.mark.parametrize("name", ["int4_shared_perm", "int4_streamk_skew"])
def test_layer_pipeline_steps(name):
    """LayerPipeline: five host-to-host steps with different inputs (token rows
    of x and the logits rolled by the step index), the copies of neighbouring
    steps overlapped with compute; every step's output is bit-identical to the
    eager call on that step's inputs."""
    L = GpuLayer(SMALL[name])
    cfg = L.cfg
    pipe = moe.LayerPipeline(cfg.T, cfg.k, L.routed, L.shared)
    xs = [torch.roll(L.x, i, dims=0).contiguous() for i in range(5)]
    lgs = [torch.roll(L.logits, i, dims=0).contiguous() for i in range(5)]
    want = []
    for i in range(5):
        out_e, ws = moe.layer_forward(xs[i], lgs[i], cfg.k, L.routed, L.shared)
        torch.cuda.synchronize()
        assert moe.last_device_error(ws) == 0
        want.append(out_e.cpu())
    got = [None] * 5
    stream = torch.cuda.current_stream()
    pipe.x_host[0].copy_(xs[0].cpu())
    pipe.logits_host[0].copy_(lgs[0].cpu())
    pipe.start()
    for i in range(5):
        if i + 1 < 5:   # step i + 1's inputs into the other host slot before step i runs
            stream.synchronize()   # step i - 1 (which read that slot) is done
            pipe.x_host[(i + 1) % 2].copy_(xs[i + 1].cpu())
            pipe.logits_host[(i + 1) % 2].copy_(lgs[i + 1].cpu())
        pipe.step(i)
        if i >= 1:   # step i copied step i - 1's output out
            stream.synchronize()
            got[i - 1] = pipe.out_host[(i - 1) % 2].clone()
    pipe.finish(4)
    stream.synchronize()
    got[4] = pipe.out_host[0].clone()
    assert moe.last_device_error(pipe.ws) == 0
    for i in range(5):
        assert torch.equal(got[i].view(torch.int16), want[i].view(torch.int16)), f"step {i}"
