"""GPU parity: top-k gating and the regroup-by-expert permutation, bit-exact against
the oracle (routing weights within fp32 rounding)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_03_gb300 as moe
import moe_synth as ms
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route_check(lg: np.ndarray, k: int):
    idx, w = moe.route_topk(torch.from_numpy(lg).to(DEV), k)
    torch.cuda.synchronize()
    oi, ow = oracle.route_topk(lg, k)
    assert np.array_equal(idx.cpu().numpy(), oi)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=2e-6, atol=1e-7)
    return oi


@pytest.mark.parametrize("name", list(ms.CONFIGS))
def test_route_configs(name):
    cfg = ms.CONFIGS[name]
    _route_check(ms.make_logits(cfg), cfg.k)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (3, 5, 5), (1000, 256, 16), (37, 33, 3),
                                   (64, 64, 1), (5, 128, 8), (4097, 8, 2)])
def test_route_shapes(T, E, k):
    rng = np.random.default_rng(T + E + k)
    _route_check(rng.standard_normal((T, E)).astype(np.float32), k)


def test_route_exact_ties():
    rng = np.random.default_rng(11)
    lg = rng.integers(0, 3, size=(500, 16)).astype(np.float32)   # many equal logits
    for k in (1, 2, 5, 16):
        _route_check(lg, k)
    _route_check(np.zeros((9, 7), np.float32), 4)                 # all equal -> 0..k-1


def _permute_check(idx: np.ndarray, E: int, d: int = 256):
    T, k = idx.shape
    x = torch.randn(T, d, device=DEV).to(torch.bfloat16)
    res = moe.permute(torch.from_numpy(idx).to(DEV), x, E)
    torch.cuda.synchronize()
    counts, offsets, roa, tor = oracle.permute(idx, E)
    assert np.array_equal(res["counts"].cpu().numpy(), counts)
    assert np.array_equal(res["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(res["row_of_assign"].cpu().numpy(), roa)
    assert np.array_equal(res["token_of_row"].cpu().numpy(), tor)
    assert torch.equal(res["x_perm"].view(torch.int16), x[torch.from_numpy(tor).long().to(DEV)].view(torch.int16))
    assert moe.last_device_error(res["ws"]) == 0


@pytest.mark.parametrize("name", list(ms.CONFIGS))
def test_permute_configs(name):
    cfg = ms.CONFIGS[name]
    idx, _ = oracle.route_topk(ms.make_logits(cfg), cfg.k)
    _permute_check(idx, cfg.E)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (1000, 3, 3), (3000, 256, 16), (700, 8, 2),
                                   (1025, 128, 8)])
def test_permute_shapes(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    idx, _ = oracle.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
    _permute_check(idx, E)


def test_permute_one_expert_takes_all_and_empty_experts():
    idx = np.full((2500, 1), 5, np.int32)
    _permute_check(idx, 9)
    idx = np.stack([np.full(300, 2), np.full(300, 7)], axis=1).astype(np.int32)
    _permute_check(idx, 8)


def test_permute_rejects_out_of_range_index_on_device():
    idx = np.array([[0, 1], [2, 9], [1, 0]], np.int32)           # 9 >= E = 4
    x = torch.randn(3, 128, device=DEV).to(torch.bfloat16)
    res = moe.permute(torch.from_numpy(idx).to(DEV), x, 4)
    code = moe.last_device_error(res["ws"])
    assert code & 2
    assert res["row_of_assign"].cpu().numpy()[3] == -1
