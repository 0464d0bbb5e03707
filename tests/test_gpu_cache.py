"""Expert streaming on the GPU: an 8-expert layer served from 4-6 HBM slots, the
other experts' images in pinned host memory, slots filled on demand (LRU).  Each
batch's output must match the oracle (every token, within the layer's bound)
and be bit-identical to the same layer with all experts resident (the GEMMs
read the same prepacked bytes, only from another slot); a token routed to an
expert that was not made resident must raise the slot-range device error rather
than read another expert's weights.  The overlapped form (prefetch on a copy
stream during the current batch's forward, commit on the compute stream) is
checked the same way over a run of batches."""
import numpy as np
import pytest
import torch

import moe_expert_layer_03_gb300 as moe
import moe_synth as ms
import oracle
from layer_setup import GpuLayer, assert_close_rms

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,mode", [("int4", 0), ("fp8", 0), ("bf16", 0), ("int4", 1)])
def test_streamed_pool_matches_resident_pool(fmt, mode):
    """mode 0: copies by the SM kernel when the host images are mapped (else the
    DMA engines); mode 1: always the DMA engines."""
    cfg = ms.LayerConfig("stream", T=2, d=256, F=512, E=8, k=2, fmt=fmt, seed=21)
    full = GpuLayer(cfg)                                   # all 8 experts resident
    hot = moe.ExpertPool(4, cfg.d, cfg.F, cfg.fmt)
    cache = moe.ExpertCache(hot, cfg.E, copy_mode=mode)
    for e in range(cfg.E):
        cache.load_expert(e, full.weights[e])
    loads = 0
    for step in range(12):                                 # a different routing every batch
        c2 = cfg.with_(seed=100 + step)
        x = ms.make_x(c2).to("cuda")
        lg_np = ms.make_logits(c2)
        lg = torch.from_numpy(lg_np).to("cuda")
        idx, _ = oracle.route_topk(lg_np, cfg.k)
        active = sorted(set(int(e) for e in idx.ravel()))
        before = cache.stats()["misses"]
        cache.ensure(active)
        out, ws = moe.layer_forward(x, lg, cfg.k, cache.view)
        ref, _ = moe.layer_forward(x, lg, cfg.k, full.routed)
        torch.cuda.synchronize()
        assert moe.last_device_error(ws) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"step {step}"
        if step % 4 == 0:   # and against the oracle
            full.x, full.logits_np = x, lg_np
            assert_close_rms(out.float().cpu().numpy(), full.oracle_forward(), what=f"{fmt} step {step}")
        loads += cache.stats()["misses"] - before
        e2s = cache.e2s.cpu().numpy()
        assert all(e2s[e] >= 0 for e in active) and (e2s >= 0).sum() <= 4
    st = cache.stats()
    assert st["misses"] == loads and st["bytes_copied"] == loads * hot.slot_bytes
    assert st["hits"] + st["misses"] >= 12 and st["misses"] >= 4


def test_expert_not_made_resident_flags_slot_error():
    cfg = ms.LayerConfig("stream_err", T=1, d=256, F=256, E=8, k=1, fmt="int4", seed=22)
    full = GpuLayer(cfg)
    hot = moe.ExpertPool(2, cfg.d, cfg.F, cfg.fmt)
    cache = moe.ExpertCache(hot, cfg.E)
    for e in range(cfg.E):
        cache.load_expert(e, full.weights[e])
    lg_np = np.full((1, cfg.E), -1.0, np.float32)
    lg_np[0, 5] = 3.0                                      # routed to expert 5 ...
    cache.ensure([0, 1])                                   # ... which is not resident
    out, ws = moe.layer_forward(full.x, torch.from_numpy(lg_np).cuda(), 1, cache.view)
    assert moe.last_device_error(ws) & 4
    cache.ensure([5])
    out, ws = moe.layer_forward(full.x, torch.from_numpy(lg_np).cuda(), 1, cache.view)
    assert moe.last_device_error(ws) == 0


@pytest.mark.parametrize("fmt,T,k,slots", [("int4", 1, 2, 5), ("int4", 2, 2, 8), ("fp8", 3, 1, 6),
                                           ("bf16", 1, 2, 4)])
def test_overlapped_streaming_matches_oracle(fmt, T, k, slots):
    """Batches of a decode loop with the next batch's experts prefetched on a copy
    stream while the current batch computes, then committed on the compute
    stream: every batch's output against the oracle (all tokens) and bit for bit
    against the all-resident pool; the copies of the slots that are reused wait
    for the forwards that read them (checked by the results)."""
    cfg = ms.LayerConfig("overlap", T=T, d=256, F=384, E=8, k=k, fmt=fmt, seed=23)
    full = GpuLayer(cfg)
    hot = moe.ExpertPool(slots, cfg.d, cfg.F, cfg.fmt)
    cache = moe.ExpertCache(hot, cfg.E)
    for e in range(cfg.E):
        cache.load_expert(e, full.weights[e])
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    n = 10
    batches = []
    for i in range(n):
        c2 = cfg.with_(seed=300 + i)
        lg_np = ms.make_logits(c2)
        idx, _ = oracle.route_topk(lg_np, cfg.k)
        batches.append((ms.make_x(c2).to("cuda"), lg_np, torch.from_numpy(lg_np).to("cuda"),
                        sorted(set(int(e) for e in idx.ravel()))))
    cache.prefetch(batches[0][3], copy)
    cache.commit(batches[0][3], compute)
    outs, wss = [], []
    for i in range(n):
        if i + 1 < n:
            cache.prefetch(batches[i + 1][3], copy)      # overlaps forward i
        x, _, lg, _ = batches[i]
        out, ws = moe.layer_forward(x, lg, cfg.k, cache.view)
        outs.append(out)
        wss.append(ws)
        if i + 1 < n:
            cache.commit(batches[i + 1][3], compute)
    torch.cuda.synchronize()
    for i in range(n):
        x, lg_np, lg, _ = batches[i]
        assert moe.last_device_error(wss[i]) == 0, f"batch {i}"
        ref, _ = moe.layer_forward(x, lg, cfg.k, full.routed)
        torch.cuda.synchronize()
        assert torch.equal(outs[i].view(torch.int16), ref.view(torch.int16)), f"batch {i}"
        full.x, full.logits_np = x, lg_np
        assert_close_rms(outs[i].float().cpu().numpy(), full.oracle_forward(), what=f"batch {i}")
    st = cache.stats()
    assert st["misses"] >= 4 and st["misses"] * hot.slot_bytes == st["bytes_copied"]


def test_prefetch_refuses_when_slots_are_short():
    """Committed and listed experts together beyond the slots: refused, nothing queued."""
    cfg = ms.LayerConfig("overlap_short", T=1, d=256, F=256, E=8, k=2, fmt="int4", seed=24)
    full = GpuLayer(cfg)
    hot = moe.ExpertPool(3, cfg.d, cfg.F, cfg.fmt)
    cache = moe.ExpertCache(hot, cfg.E)
    for e in range(cfg.E):
        cache.load_expert(e, full.weights[e])
    copy = torch.cuda.Stream()
    cache.prefetch([0, 1], copy)
    cache.commit([0, 1])
    with pytest.raises(moe.MoeError, match="unsupported"):
        cache.prefetch([2, 3], copy)                        # 2 committed + 2 new > 3 slots
    with pytest.raises(moe.MoeError, match="invalid"):
        cache.commit([4])                                   # not resident
