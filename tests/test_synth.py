"""The seeded input recipes hold the properties the workloads are defined by (no GPU)."""
import numpy as np
import torch

import moe_synth as ms


def test_gap_rule_every_config():
    for cfg in ms.CONFIGS.values():
        lg = ms.make_logits(cfg)
        assert lg.dtype == np.float32 and lg.shape == (cfg.T, cfg.E)
        s = -np.sort(-lg, axis=1)
        if cfg.k < cfg.E:
            assert np.all(s[:, cfg.k - 1] - s[:, cfg.k] >= np.float32(ms.MIN_GAP))


def test_seeded_and_reproducible():
    cfg = ms.CONFIGS["tiny"]
    assert np.array_equal(ms.make_logits(cfg), ms.make_logits(cfg))
    assert torch.equal(ms.make_x(cfg), ms.make_x(cfg))
    a = ms.expert_source(cfg, 3)
    b = ms.expert_source(cfg, 3)
    assert all(torch.equal(a[m], b[m]) for m in ms.MATS)
    assert not torch.equal(ms.expert_source(cfg, 2)["gate"], a["gate"])


def test_weight_and_activation_statistics():
    cfg = ms.CONFIGS["tiny"]
    w = ms.expert_source(cfg, 0)["gate"].float()
    assert abs(w.std().item() - 0.02) < 0.001 and abs(w.mean().item()) < 0.001
    x = ms.make_x(cfg).float()
    assert abs(x.std().item() - 1.0) < 0.05


def test_zipf_skew_and_slot_permutation():
    cfg = ms.CONFIGS["fg125b_decode"].with_(T=4096)
    lg = ms.make_logits(cfg)
    top = np.argsort(-lg, axis=1, kind="stable")[:, :cfg.k]
    cnt = np.sort(np.bincount(top.ravel(), minlength=cfg.E))[::-1]
    assert cnt[:30].sum() / cnt.sum() > 0.5          # a few experts take most assignments
    st = ms.make_slot_table(ms.CONFIGS["fg125b_decode"])
    assert sorted(st.tolist()) == list(range(128)) and st.tolist() != list(range(128))


def test_reuse_fraction():
    cfg = ms.CONFIGS["mixtral_prefill"]
    lg = ms.make_logits(cfg)
    top = np.argsort(-lg, axis=1, kind="stable")[:, :2]
    same = np.mean(np.all(top[1:] == top[:-1], axis=1))
    # 44% forced reuse plus chance repeats of a fresh draw (1/56 of the rest)
    assert 0.40 < same < 0.50


def test_int4_encoding_shapes_and_ranges():
    cfg = ms.CONFIGS["tiny"].with_(fmt="int4")
    w = ms.expert_weights(cfg, 1)
    assert w["gate"]["q"].shape == (cfg.F, cfg.d // 2) and w["gate"]["q"].dtype == torch.uint8
    assert w["down"]["scale"].shape == (cfg.d, cfg.F // 128)
    z = w["up"]["zero"].float()
    assert torch.all(z == z.round()) and z.min() >= 0 and z.max() <= 15
    assert ms.active_expert_bytes(ms.CONFIGS["mixtral_decode"]) == 93_585_408
