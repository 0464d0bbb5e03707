"""The reference arm's sub-token sample on CPU: when one token per step would keep
the oracle run past its time budget, a unit of work is one token's FFN over 1/S of
d_ff (`bench.slice_weights`).  The S slices of a token must add up to the token's
full oracle output -- a wrong gate/up row range, down column range or group slice
of the scales and zero points would not."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_synth as ms  # noqa: E402
import oracle  # noqa: E402


@pytest.mark.parametrize("fmt", ["bf16", "int4", "fp8"])
def test_feature_slices_add_up_to_the_token(fmt):
    oracle.build()
    cfg = ms.LayerConfig("slices", T=4, d=256, F=512, E=4, k=2, fmt=fmt, seed=3)
    x, lg = ms.make_x(cfg), ms.make_logits(cfg)
    w = {e: ms.expert_weights(cfg, e, "cpu") for e in range(cfg.E)}
    full = oracle.layer_forward(x, lg, cfg.k, [oracle.ExpertRef(w[e], fmt) for e in range(cfg.E)], None,
                                cfg.d, cfg.F, tokens=[1])[0]
    for S in (2, 4):
        Fs = cfg.F // S
        acc = np.zeros_like(full)
        for sl in range(S):
            ex = [oracle.ExpertRef(bench.slice_weights(w[e], fmt, sl * Fs, (sl + 1) * Fs), fmt)
                  for e in range(cfg.E)]
            part = oracle.layer_forward(x, lg, cfg.k, ex, None, cfg.d, Fs, tokens=[1])[0]
            assert np.abs(part).max() > 0
            acc += part
        np.testing.assert_allclose(acc, full, rtol=0, atol=1e-12 * np.abs(full).max())
