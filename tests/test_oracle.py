"""Pins of the CPU oracle against what the method and mathematics fix (no GPU).

Each test checks the oracle against something other than itself: worked cases
derived by hand (tests/golden), closed forms, invariants, brute force on tiny
inputs, or a special case that reduces to a library routine (numpy matmul,
torch's bf16 conversion).
"""
import ctypes as C
import math
import os

import numpy as np
import pytest
import torch

import moe_synth as ms
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
bf = oracle.bf16_bits_to_float


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------- numbers
def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 65536, 5000).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    L = oracle.lib()
    got = np.array([L.oracle_bf16_to_double(int(b)) for b in bits])
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.array_equal(np.isnan(got), np.isnan(want))


def test_fp16_decode_all_patterns():
    L = oracle.lib()
    pats = np.arange(65536, dtype=np.uint16)
    want = pats.view(np.float16).astype(np.float64)
    got = np.array([L.oracle_fp16_to_double(int(p)) for p in pats])
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(np.isinf(got), np.isinf(want))


# ----------------------------------------------------------------------------- fp8 (E4M3)
def test_e4m3_decode_all_patterns_match_torch():
    """All 256 E4M3 codes against torch's float8_e4m3fn (an independent decoder)."""
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.lib().oracle_e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2      # S.1111.111 only
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def _fp8_matrix(q: np.ndarray, s_bits: np.ndarray):
    q = np.ascontiguousarray(q, np.uint8)
    s_bits = np.ascontiguousarray(s_bits, np.uint16)
    m = oracle.Matrix(2, q.shape[0], q.shape[1], None, q.ctypes.data, s_bits.ctypes.data, None)
    return m, (q, s_bits)


def test_fp8_dequant_golden_group():
    """A hand-derived group (tests/golden/fp8_group.txt): w = e4m3(q) * s."""
    rows = [l.split() for l in open(os.path.join(GOLD, "fp8_group.txt"))
            if l.strip() and not l.startswith("#")]
    s_bits = int(rows[0][1], 16)
    cases = [(int(c, 16), float(w)) for c, _, w in rows[1:]]
    q = np.zeros((1, 128), np.uint8)
    for i, (c, _) in enumerate(cases):
        q[0, i] = c
    m, keep = _fp8_matrix(q, np.array([[s_bits]], np.uint16))
    for i, (_, w) in enumerate(cases):
        got = oracle.lib().oracle_weight(C.byref(m), 0, i)
        assert got == w and np.signbit(got) == np.signbit(w), (i, got, w)


def test_fp8_quantizer_roundtrip_exact_on_representable_group():
    """A group whose largest magnitude is 448 * 2^-8 and whose values are E4M3
    numbers times 2^-8 gets s = 2^-8 exactly and comes back bit for bit."""
    rng = np.random.default_rng(5)
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    finite = e4[np.isfinite(e4)]
    vals = rng.choice(finite, size=(3, 256)).astype(np.float32)
    vals[:, 0] = vals[:, 128] = 448.0                # each group's largest magnitude
    vals *= 2.0 ** -8
    enc = ms.quantize_fp8_g128(torch.from_numpy(vals).to(torch.bfloat16))
    assert np.all(enc["scale"].float().numpy() == 2.0 ** -8)
    m, keep = _fp8_matrix(enc["q"].numpy(), enc["scale"].view(torch.int16).numpy().view(np.uint16))
    back = np.array([[oracle.lib().oracle_weight(C.byref(m), r, c) for c in range(256)] for r in range(3)])
    assert np.array_equal(back, vals.astype(np.float64))


def test_fp8_quantizer_error_bound_random_groups():
    """|w - v| <= half an E4M3 ulp of v/s, times s (E4M3 keeps 3 mantissa bits;
    the subnormal spacing 2^-9 below 2^-6)."""
    rng = np.random.default_rng(6)
    v = torch.from_numpy((rng.standard_normal((8, 512)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    enc = ms.quantize_fp8_g128(v)
    m, keep = _fp8_matrix(enc["q"].numpy(), enc["scale"].view(torch.int16).numpy().view(np.uint16))
    vf = v.double().numpy()
    for r in range(8):
        for c in range(0, 512, 7):
            s = float(enc["scale"][r, c // 128])
            a = abs(vf[r, c]) / s
            ulp = 2.0 ** -9 if a < 2.0 ** -6 else 2.0 ** (np.floor(np.log2(a)) - 3)
            assert abs(oracle.lib().oracle_weight(C.byref(m), r, c) - vf[r, c]) <= 0.5 * ulp * s * (1 + 1e-12)


# ----------------------------------------------------------------------------- int4
def _golden_int4():
    kv = {}
    for line in open(os.path.join(GOLD, "int4_group.txt")):
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        kv[key] = vals
    raw = bytes(int(b, 16) for b in kv["bytes"]) * int(kv["repeat"][0])
    return (np.frombuffer(raw, np.uint8).reshape(1, 64), int(kv["scale_fp16"][0], 16),
            int(kv["zero_fp16"][0], 16), [float(v) for v in kv["expect_first16"]])


def test_int4_dequant_golden_nibble_order():
    q, s, z, first16 = _golden_int4()
    sc = np.array([[s]], np.uint16)
    zr = np.array([[z]], np.uint16)
    m = oracle.Matrix(1, 1, 128, None, q.ctypes.data, sc.ctypes.data, zr.ctypes.data)
    got = [oracle.lib().oracle_weight(m, 0, c) for c in range(128)]
    assert got[:16] == first16
    assert got == [((c % 16) - 3) * 0.5 for c in range(128)]


def test_int4_roundtrip_exact_group():
    # v_i = (q_i - 3) * 0.5, q_i = i mod 16 -> s = 0.5, z = 3 exactly and the
    # encoding followed by the oracle's dequantisation returns v bit-exactly.
    v = torch.tensor([[((i % 16) - 3) * 0.5 for i in range(256)]], dtype=torch.float32)
    enc = ms.quantize_int4_g128(v.to(torch.bfloat16))
    assert enc["scale"].float().tolist() == [[0.5, 0.5]]
    assert enc["zero"].float().tolist() == [[3.0, 3.0]]
    ref = oracle.ExpertRef({"gate": enc, "up": enc, "down": enc}, "int4")
    mat = ref.struct.gate
    got = [oracle.lib().oracle_weight(mat, 0, c) for c in range(256)]
    assert got == v[0].tolist()


def test_int4_error_bound_random_groups():
    g = torch.Generator().manual_seed(1)
    w = (torch.randn(64, 512, generator=g) * 0.02).to(torch.bfloat16)
    w[3, :128] = torch.linspace(0.1, 0.3, 128).to(torch.bfloat16)   # one-signed group
    enc = ms.quantize_int4_g128(w)
    ref = oracle.ExpertRef({"gate": enc, "up": enc, "down": enc}, "int4")
    s = enc["scale"].float().numpy()
    dq = np.array([[oracle.lib().oracle_weight(ref.struct.gate, r, c) for c in range(512)]
                   for r in range(64)])
    err = np.abs(dq - w.float().numpy())
    bound = np.repeat(s, 128, axis=1) * (0.5 + 15 * 2.0 ** -11) + 1e-12
    assert np.all(err <= bound)


# ----------------------------------------------------------------------------- router logits
def _bf16_bits_of(values) -> np.ndarray:
    return _bits(torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16))


def test_router_one_hot_rows_select_router_columns():
    """x[t] = c_t * unit vector i_t selects column i_t of the router weight, scaled
    by c_t (a power of two, exact): catches a transposed operand or a wrong index."""
    rng = np.random.default_rng(11)
    T, d, E = 6, 40, 5
    w = _bits(torch.from_numpy(rng.standard_normal((E, d)).astype(np.float32) * 0.02).to(torch.bfloat16))
    cols = [0, 39, 7, 7, 21, 13]
    scale = [1.0, 2.0, -0.5, 4.0, 1.0, -1.0]
    x = np.zeros((T, d), np.float32)
    for t in range(T):
        x[t, cols[t]] = scale[t]
    lg = oracle.router_logits(_bf16_bits_of(x), w)
    for t in range(T):
        np.testing.assert_array_equal(lg[t], scale[t] * bf(w[:, cols[t]]).astype(np.float64))


def test_router_small_integers_bruteforce():
    """Integer-valued bf16 inputs: the logits are exact integers, checked against a
    pure-Python integer triple loop."""
    rng = np.random.default_rng(12)
    T, d, E = 3, 9, 4
    xi = rng.integers(-4, 5, (T, d))
    wi = rng.integers(-4, 5, (E, d))
    lg = oracle.router_logits(_bf16_bits_of(xi), _bf16_bits_of(wi))
    for t in range(T):
        for e in range(E):
            assert lg[t, e] == sum(int(xi[t, i]) * int(wi[e, i]) for i in range(d))


def test_router_random_matches_exact_rational_sum():
    """N(0,1) tokens against N(0,0.02) router rows: the fp64 logit equals the exact
    rational dot product rounded once (the partial sums here need well under 53 bits)."""
    from fractions import Fraction
    rng = np.random.default_rng(13)
    T, d, E = 2, 64, 3
    x = _bits(torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16))
    w = _bits(torch.from_numpy(rng.standard_normal((E, d)).astype(np.float32) * 0.02).to(torch.bfloat16))
    lg = oracle.router_logits(x, w)
    xf, wf = bf(x), bf(w)
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(xf[t, i])) * Fraction(float(wf[e, i])) for i in range(d))
            assert lg[t, e] == float(exact)


# ----------------------------------------------------------------------------- top-k
def _golden_topk():
    for line in open(os.path.join(GOLD, "topk_cases.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, lg, ix, w = [p.split() for p in line.split("|")]
        yield int(k[0]), np.array(lg, np.float32), [int(i) for i in ix], [float(x) for x in w]


@pytest.mark.parametrize("case", list(_golden_topk()))
def test_topk_golden(case):
    k, lg, want_idx, want_w = case
    idx, w = oracle.route_topk(lg[None, :], k)
    assert idx[0].tolist() == want_idx
    np.testing.assert_allclose(w[0], want_w, rtol=2e-7, atol=1e-8)


def test_topk_bruteforce_tiny_with_ties():
    """Dominance check on every selected/unselected pair, logits from {0,1,2} to force ties."""
    rng = np.random.default_rng(7)
    for E in range(1, 9):
        for k in range(1, E + 1):
            lg = rng.integers(0, 3, size=(40, E)).astype(np.float32)
            idx, w = oracle.route_topk(lg, k)
            for t in range(40):
                sel = list(idx[t])
                assert len(set(sel)) == k
                beats = lambda a, b: lg[t, a] > lg[t, b] or (lg[t, a] == lg[t, b] and a < b)
                for a in sel:
                    for b in range(E):
                        if b not in sel:
                            assert beats(a, b)
                for a, b in zip(sel, sel[1:]):
                    assert beats(a, b)
                assert abs(float(np.sum(w[t], dtype=np.float64)) - 1.0) < 1e-6


def test_topk_weight_closed_forms():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((200, 6)).astype(np.float32)
    idx, w = oracle.route_topk(lg, 1)
    assert np.all(w == 1.0)
    idx, w = oracle.route_topk(lg, 2)
    l0 = lg[np.arange(200), idx[:, 0]].astype(np.float64)
    l1 = lg[np.arange(200), idx[:, 1]].astype(np.float64)
    sig = 1.0 / (1.0 + np.exp(l1 - l0))            # 2-way softmax = logistic of the gap
    np.testing.assert_allclose(w[:, 0], sig, rtol=2e-7)
    np.testing.assert_allclose(w[:, 1], 1.0 - sig, rtol=2e-6)
    eq = np.zeros((5, 8), np.float32)
    idx, w = oracle.route_topk(eq, 5)
    assert idx.tolist() == [[0, 1, 2, 3, 4]] * 5
    np.testing.assert_allclose(w, 0.2, rtol=1e-7)


# ----------------------------------------------------------------------------- permute
def test_permute_golden():
    kv = {}
    for line in open(os.path.join(GOLD, "permute_case.txt")):
        if line.startswith("#") or not line.strip():
            continue
        key, *vals = line.split()
        kv[key] = [int(v) for v in vals]
    T, k, E = kv["T"][0], kv["k"][0], kv["E"][0]
    counts, offsets, roa, tor = oracle.permute(np.array(kv["idx"], np.int32).reshape(T, k), E)
    assert counts.tolist() == kv["counts"]
    assert offsets.tolist() == kv["offsets"]
    assert roa.tolist() == kv["row_of_assign"]
    assert tor.tolist() == kv["token_of_row"]


def check_permutation_invariants(idx, counts, offsets, roa, tor, E):
    T, k = idx.shape
    A = T * k
    assert counts.sum() == A and offsets[0] == 0 and offsets[E] == A
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(roa), np.arange(A))                # bijection onto [0, A)
    flat = idx.reshape(-1)
    for a in range(A):
        assert tor[roa[a]] == a // k
        assert offsets[flat[a]] <= roa[a] < offsets[flat[a] + 1]
    for e in range(E):
        toks = tor[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(toks) > 0)                               # stable: ascending tokens


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (7, 4, 4), (33, 8, 2), (64, 128, 8), (300, 16, 2)])
def test_permute_invariants(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle.route_topk(lg, k)
    check_permutation_invariants(idx, *oracle.permute(idx, E), E)


def test_permute_all_to_one_expert():
    idx = np.zeros((50, 1), np.int32) + 3
    counts, offsets, roa, tor = oracle.permute(idx, 5)
    assert counts.tolist() == [0, 0, 0, 50, 0]
    assert roa.tolist() == list(range(50)) and tor.tolist() == list(range(50))


# ----------------------------------------------------------------------------- expert FFN
def _dense_swiglu(x_bf16: torch.Tensor, Wg, Wu, Wd):
    """Independent dense SwiGLU in float64 numpy (library matmuls)."""
    x = x_bf16.double().numpy()
    g = x @ Wg.T
    u = x @ Wu.T
    h = g / (1.0 + np.exp(-g)) * u
    return h, h @ Wd.T


def _dequant_numpy(enc):
    q = enc["q"].numpy()
    lo, hi = q & 0xF, q >> 4
    codes = np.empty((q.shape[0], q.shape[1] * 2), np.float64)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    s = np.repeat(enc["scale"].double().numpy(), 128, axis=1)
    z = np.repeat(enc["zero"].double().numpy(), 128, axis=1)
    return (codes - z) * s


def _dequant_fp8_numpy(enc):
    """E4M3 codes decoded through torch's float8 type, times the group scales."""
    codes = enc["q"].view(torch.float8_e4m3fn).double().numpy()
    return codes * np.repeat(enc["scale"].double().numpy(), 128, axis=1)


@pytest.mark.parametrize("fmt", ["bf16", "int4", "fp8"])
def test_single_expert_reduces_to_dense_swiglu(fmt):
    """E=1, k=1: the layer is one dense SwiGLU FFN (weight 1.0), d != F so a transposed operand fails."""
    cfg = ms.LayerConfig("t", T=6, d=256, F=384, E=1, k=1, fmt=fmt)
    x = ms.make_x(cfg)
    lg = ms.make_logits(cfg)
    wts = ms.expert_weights(cfg, 0)
    ref = oracle.ExpertRef(wts, fmt)
    out, idx, w = oracle.layer_forward(x, lg, 1, [ref], None, cfg.d, cfg.F)
    assert np.all(idx == 0) and np.all(w == 1.0)
    if fmt == "bf16":
        Wg, Wu, Wd = (wts[m]["w"].double().numpy() for m in ("gate", "up", "down"))
    elif fmt == "fp8":
        Wg, Wu, Wd = (_dequant_fp8_numpy(wts[m]) for m in ("gate", "up", "down"))
    else:
        Wg, Wu, Wd = (_dequant_numpy(wts[m]) for m in ("gate", "up", "down"))
    h, y = _dense_swiglu(x, Wg, Wu, Wd)
    np.testing.assert_allclose(out, y, rtol=1e-9, atol=1e-12 * np.abs(y).max())
    # the single-row entry point gives the same h and y
    h1, y1 = oracle.expert_ffn(x[2], ref, cfg.d, cfg.F)
    assert np.array_equal(y1, out[2])
    np.testing.assert_allclose(h1, h[2], rtol=1e-9, atol=1e-12 * np.abs(h).max())


def test_combine_identical_experts_is_dense_ffn():
    cfg = ms.LayerConfig("t", T=8, d=128, F=256, E=4, k=2, fmt="bf16")
    x = ms.make_x(cfg)
    lg = ms.make_logits(cfg)
    wts = ms.expert_weights(cfg, 0)
    ref = oracle.ExpertRef(wts, "bf16")
    out, _, _ = oracle.layer_forward(x, lg, 2, [ref] * 4, None, cfg.d, cfg.F)
    _, y = _dense_swiglu(x, *(wts[m]["w"].double().numpy() for m in ("gate", "up", "down")))
    np.testing.assert_allclose(out, y, rtol=1e-6, atol=1e-9)      # sum of fp32 weights = 1 +- 1e-7


def test_down_projection_linearity():
    cfg = ms.LayerConfig("t", T=5, d=128, F=256, E=3, k=2, fmt="bf16")
    x = ms.make_x(cfg)
    lg = ms.make_logits(cfg)
    wts = [ms.expert_weights(cfg, e) for e in range(3)]
    out1, _, _ = oracle.layer_forward(x, lg, 2, [oracle.ExpertRef(w, "bf16") for w in wts], None,
                                      cfg.d, cfg.F)
    w2 = [{"gate": w["gate"], "up": w["up"], "down": {"w": (w["down"]["w"].float() * 2).to(torch.bfloat16)}}
          for w in wts]
    out2, _, _ = oracle.layer_forward(x, lg, 2, [oracle.ExpertRef(w, "bf16") for w in w2], None,
                                      cfg.d, cfg.F)
    assert np.array_equal(out2, 2.0 * out1)


def test_shared_expert_alone_when_routed_down_is_zero():
    cfg = ms.LayerConfig("t", T=4, d=128, F=256, E=4, k=2, fmt="int4", shared=True)
    x = ms.make_x(cfg)
    lg = ms.make_logits(cfg)
    routed = []
    for e in range(4):
        w = ms.expert_weights(cfg, e)
        w["down"] = dict(w["down"], zero=w["down"]["zero"].clone())
        w["down"]["q"] = w["down"]["zero"].to(torch.uint8).repeat_interleave(64, dim=1) * 0x11
        routed.append(oracle.ExpertRef(w, "int4"))                # q == z everywhere -> W_down = 0
    sh = ms.expert_weights(cfg, "shared")
    shref = oracle.ExpertRef(sh, "int4")
    out, _, _ = oracle.layer_forward(x, lg, 2, routed, shref, cfg.d, cfg.F)
    for t in range(cfg.T):
        _, ysh = oracle.expert_ffn(x[t], shref, cfg.d, cfg.F)
        assert np.array_equal(out[t], ysh)


def test_combine_row_hand_values():
    one = _bits(torch.tensor([1.0, -2.0, 0.5], dtype=torch.bfloat16))
    two = _bits(torch.tensor([2.0, 4.0, 0.25], dtype=torch.bfloat16))
    sh = _bits(torch.tensor([0.5, 0.5, 0.5], dtype=torch.bfloat16))
    out = oracle.combine_row([one, two], [0.25, 0.75])
    assert out.tolist() == [1.75, 2.5, 0.3125]
    out = oracle.combine_row([one, two], [0.25, 0.75], sh)
    assert out.tolist() == [2.25, 3.0, 0.8125]


def test_bf16_ulp_helper_matches_torch_spacing():
    """The parity tests' one-ulp allowance uses the spacing of bf16 numbers: check it
    against torch's bf16 rounding (the next representable value up)."""
    from layer_setup import bf16_ulp
    rng = np.random.default_rng(21)
    v = (rng.standard_normal(2000) * np.exp2(rng.integers(-20, 20, 2000))).astype(np.float32)
    b = torch.from_numpy(v).to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().view(np.uint16).astype(np.int32)
    nxt = torch.from_numpy(((bits + 1) & 0xFFFF).astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    spacing = np.abs(nxt.double().numpy() - b.double().numpy())
    np.testing.assert_array_equal(bf16_ulp(b.double().numpy()), spacing)
