"""Expert streaming on the GPU: an 8-expert layer served from 4 HBM slots, the
other experts' images in pinned host memory, slots filled on demand (LRU).  Each
batch's output must be bit-identical to the same layer with all experts
resident (the GEMMs read the same prepacked bytes, only from another slot), and a
token routed to an expert that was not made resident must raise the slot-range
device error rather than read another expert's weights."""
import numpy as np
import pytest
import torch

import moe_expert_layer_03_gb300 as moe
import moe_synth as ms
import oracle
from layer_setup import GpuLayer

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
