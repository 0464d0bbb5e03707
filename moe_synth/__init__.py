"""Seeded synthetic inputs for the MoE FFN layer (shared by the CUDA path and the oracle).

This module only *draws* inputs: token activations, router logits, expert weights,
the expert->slot table, and the int4 group-128 encoding of the expert weights
(offline weight preparation; the layer itself only ever dequantises).  It holds
none of the layer's arithmetic (gating, permutation, expert FFN, combine).

Workload shapes follow the five configurations the layer is measured on:

  tiny            T=16,   d=256,  F=512,   E=8,   k=2, bf16 weights
  mixtral_decode  T=16,   d=4096, F=14336, E=8,   k=2, int4 g128 weights
  phi35_prefill   T=256,  d=4096, F=6400,  E=16,  k=2, bf16, Zipf(1.0) routing
  fg125b_decode   T=16,   d=5120, F=1536,  E=128, k=8, int4, Zipf(1.1) routing,
                  + 1 always-on shared expert, permuted expert->slot table
  mixtral_prefill T=2048, d=4096, F=14336, E=8,   k=2, int4, 44% of tokens
                  reuse the previous token's expert pair
  mixtral_decode_fp8, mixtral_prefill_fp8: the two Mixtral layers with 8-bit
                  experts (E4M3 codes, one fp16 scale per row and group of 128)

Recipes (the values the layer sees; all seeded):
  * x ~ N(0,1) drawn in fp32 and rounded to bf16 ("normal").  Activation
    stress variants (x_dist) for the precision tests:
      - "outlier": N(0,1) rows with 4 seeded outlier columns, the same in every
                   token, multiplied by x_outlier (100, 1000: the few very large
                   feature channels of real LLM hidden states);
      - "wide":    magnitudes 2^u, u ~ Uniform(-20, 10), random signs, so each
                   row spans 2^-20 .. 2^10;
      - "tiny":    N(0,1) * 1e-6;
      - "scaled":  N(0,1) * x_outlier (every element large);
      - "onehot":  one nonzero element per row (a seeded column, N(0,1) value
                   pushed away from 0 by 1).
  * expert weights ~ N(0, 0.02) drawn in fp32 and rounded to bf16 ("source"),
    one independent torch Generator stream per (expert, matrix) so any single
    expert can be regenerated alone on any device.
  * router weight (optional router GEMM) [E, d] ~ N(0, 0.02), rounded to bf16.
  * router logits fp32, per row resampled until the gap between the k-th and
    (k+1)-th largest value is >= 1e-3 so the top-k set is unambiguous.
      - "normal": i.i.d. N(0,1).
      - "zipf":   logit = ln p_e + Gumbel(0,1) with p_e proportional to
                  rank(e)^-s over a seeded rank permutation, which makes the top-k
                  a draw without replacement with probabilities p.
      - "reuse":  row 0 fresh N(0,1); for t>0 with probability p_reuse a fresh
                  N(0,1) row whose two largest values are swapped onto the
                  previous token's two experts (same relative order); otherwise a
                  fresh row.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

GROUP = 128          # quantisation group along K (input dim)
MIN_GAP = 1e-3       # minimum logit gap between the k-th and (k+1)-th expert


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    d: int
    F: int
    E: int
    k: int
    fmt: str                  # "bf16", "int4" or "fp8"
    logits: str = "normal"    # "normal" | "zipf" | "reuse"
    zipf_s: float = 1.0
    reuse_p: float = 0.44
    shared: bool = False      # one always-on shared expert (weight 1.0)
    slot_perm: bool = False   # expert->slot table is a seeded random permutation
    seed: int = 0
    x_dist: str = "normal"    # "normal" | "outlier" | "wide" | "tiny" | "scaled" | "onehot"
    x_outlier: float = 1000.0

    @property
    def A(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


CONFIGS = {
    "tiny": LayerConfig("tiny", T=16, d=256, F=512, E=8, k=2, fmt="bf16"),
    "mixtral_decode": LayerConfig("mixtral_decode", T=16, d=4096, F=14336, E=8, k=2, fmt="int4"),
    "phi35_prefill": LayerConfig("phi35_prefill", T=256, d=4096, F=6400, E=16, k=2, fmt="bf16",
                                 logits="zipf", zipf_s=1.0),
    "fg125b_decode": LayerConfig("fg125b_decode", T=16, d=5120, F=1536, E=128, k=8, fmt="int4",
                                 logits="zipf", zipf_s=1.1, shared=True, slot_perm=True),
    "mixtral_prefill": LayerConfig("mixtral_prefill", T=2048, d=4096, F=14336, E=8, k=2,
                                   fmt="int4", logits="reuse", reuse_p=0.44),
    # the same two Mixtral-shaped layers with 8-bit (E4M3, group-128) experts
    "mixtral_decode_fp8": LayerConfig("mixtral_decode_fp8", T=16, d=4096, F=14336, E=8, k=2,
                                      fmt="fp8"),
    "mixtral_prefill_fp8": LayerConfig("mixtral_prefill_fp8", T=2048, d=4096, F=14336, E=8, k=2,
                                       fmt="fp8", logits="reuse", reuse_p=0.44),
}


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


# ----------------------------------------------------------------------------- activations
def make_x(cfg: LayerConfig) -> torch.Tensor:
    """Token activations, bf16 [T, d] on the CPU (distribution: cfg.x_dist)."""
    rng = _rng(cfg.seed, 1)
    v = rng.standard_normal((cfg.T, cfg.d), dtype=np.float32)
    if cfg.x_dist == "outlier":
        cols = _rng(cfg.seed, 6).choice(cfg.d, size=min(4, cfg.d), replace=False)
        v[:, cols] *= np.float32(cfg.x_outlier)
    elif cfg.x_dist == "wide":
        u = rng.uniform(-20.0, 10.0, size=(cfg.T, cfg.d))
        v = (np.sign(v) * np.exp2(u)).astype(np.float32)
    elif cfg.x_dist == "tiny":
        v = v * np.float32(1e-6)
    elif cfg.x_dist == "scaled":
        v = v * np.float32(cfg.x_outlier)
    elif cfg.x_dist == "onehot":
        col = rng.integers(0, cfg.d, size=cfg.T)
        val = v[np.arange(cfg.T), col]
        v = np.zeros_like(v)
        v[np.arange(cfg.T), col] = val + np.sign(val)
    elif cfg.x_dist != "normal":
        raise ValueError(f"unknown x_dist {cfg.x_dist!r}")
    return torch.from_numpy(np.ascontiguousarray(v)).to(torch.bfloat16)


# ----------------------------------------------------------------------------- router weight
def make_router_weight(cfg: LayerConfig) -> torch.Tensor:
    """Router weight for the optional router GEMM, bf16 [E, d] on the CPU:
    N(0, 0.02) drawn in fp32 and rounded to bf16 (same recipe as the expert
    weights), its own seeded stream."""
    v = _rng(cfg.seed, 5).standard_normal((cfg.E, cfg.d), dtype=np.float32) * np.float32(0.02)
    return torch.from_numpy(v).to(torch.bfloat16)


# ----------------------------------------------------------------------------- router logits
def _gap_ok(row: np.ndarray, k: int) -> bool:
    if k >= row.shape[0]:
        return True
    s = np.sort(row)[::-1]
    return bool(np.float32(s[k - 1]) - np.float32(s[k]) >= np.float32(MIN_GAP))


def _draw_row(cfg: LayerConfig, rng: np.random.Generator, logp: np.ndarray | None) -> np.ndarray:
    if cfg.logits == "zipf":
        u = rng.random(cfg.E)
        u = np.clip(u, 1e-12, 1.0 - 1e-12)
        return (logp - np.log(-np.log(u))).astype(np.float32)
    return rng.standard_normal(cfg.E).astype(np.float32)


def make_logits(cfg: LayerConfig) -> np.ndarray:
    """Router logits, fp32 [T, E], with the top-k gap rule applied to every row."""
    rng = _rng(cfg.seed, 2)
    logp = None
    if cfg.logits == "zipf":
        rank = rng.permutation(cfg.E)
        p = (rank + 1.0) ** (-cfg.zipf_s)
        logp = np.log(p / p.sum())
    out = np.empty((cfg.T, cfg.E), dtype=np.float32)
    prev_top: tuple[int, int] | None = None
    for t in range(cfg.T):
        reuse = (cfg.logits == "reuse" and t > 0 and cfg.E >= 2 and rng.random() < cfg.reuse_p)
        while True:
            row = _draw_row(cfg, rng, logp)
            if reuse:
                # swap the largest value onto prev_top[0], then the second largest onto prev_top[1]
                order = np.argsort(-row, kind="stable")
                a, b = int(order[0]), int(order[1])
                p0, p1 = prev_top
                row[[a, p0]] = row[[p0, a]]
                if b == p0:
                    b = a
                row[[b, p1]] = row[[p1, b]]
            if _gap_ok(row, cfg.k):
                break
        out[t] = row
        o = np.argsort(-row, kind="stable")
        prev_top = (int(o[0]), int(o[1])) if cfg.E >= 2 else None
    return out


# ----------------------------------------------------------------------------- slot table
def make_slot_table(cfg: LayerConfig) -> np.ndarray:
    """expert_to_slot int32 [E]; the shared expert (if any) lives in slot E."""
    if cfg.slot_perm:
        return _rng(cfg.seed, 3).permutation(cfg.E).astype(np.int32)
    return np.arange(cfg.E, dtype=np.int32)


# ----------------------------------------------------------------------------- expert weights
MATS = ("gate", "up", "down")


def _wshape(cfg: LayerConfig, mat: str) -> tuple[int, int]:
    return (cfg.d, cfg.F) if mat == "down" else (cfg.F, cfg.d)


def expert_source(cfg: LayerConfig, e: int | str, device="cpu") -> dict[str, torch.Tensor]:
    """bf16 source weights of expert e (or "shared"): gate/up [F, d], down [d, F]."""
    eid = cfg.E if e == "shared" else int(e)
    out = {}
    for mi, mat in enumerate(MATS):
        g = torch.Generator(device=device)
        g.manual_seed((cfg.seed * 1_000_003 + eid * 16 + mi + 7) & 0x7FFF_FFFF_FFFF)
        w = torch.randn(_wshape(cfg, mat), generator=g, device=device, dtype=torch.float32)
        out[mat] = (w * 0.02).to(torch.bfloat16)
    return out


def quantize_int4_g128(w: torch.Tensor) -> dict[str, torch.Tensor]:
    """Offline int4 encoding of a bf16 weight matrix [rows, K] (K % 128 == 0).

    Asymmetric, one fp16 scale and one fp16 zero-point (an integer 0..15) per
    row and per group of 128 consecutive K elements, with the range widened to
    include 0 (min <= 0 <= max) so a one-signed group stays representable:
        s = fp16(max(max - min, 1e-8) / 15)
        z = clamp(round(-min / s), 0, 15)
        q = clamp(round(v / s) + z, 0, 15)          (round half to even, fp32)
    Packing: byte [r, j] holds element 2j in its low nibble, 2j+1 in its high.
    Returns {"q": uint8 [rows, K/2], "scale": fp16 [rows, K/128], "zero": fp16 [rows, K/128]}.
    """
    rows, K = w.shape
    assert K % GROUP == 0
    v = w.to(torch.float32).reshape(rows, K // GROUP, GROUP)
    mn = torch.clamp(v.amin(dim=2), max=0.0)
    mx = torch.clamp(v.amax(dim=2), min=0.0)
    s = (torch.clamp(mx - mn, min=1e-8) / 15.0).to(torch.float16)
    sf = s.to(torch.float32)
    z = torch.clamp(torch.round(-mn / sf), 0, 15)
    q = torch.clamp(torch.round(v / sf.unsqueeze(2)) + z.unsqueeze(2), 0, 15).to(torch.uint8)
    q = q.reshape(rows, K)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).contiguous()
    return {"q": packed, "scale": s.contiguous(), "zero": z.to(torch.float16).contiguous()}


E4M3_MAX = 448.0


def quantize_fp8_g128(w: torch.Tensor) -> dict[str, torch.Tensor]:
    """Offline 8-bit encoding of a bf16 weight matrix [rows, K] (K % 128 == 0):
    OCP fp8 E4M3 codes with one fp16 scale per row and group of 128 K elements,
    symmetric (no zero point):
        s = fp16(max(amax, 1e-8) / 448)            (amax = largest |v| of the group)
        q = e4m3(clamp(v / s, -448, 448))           (round to nearest even, fp32)
    Returns {"q": uint8 [rows, K] (the E4M3 bit patterns), "scale": fp16 [rows, K/128]}.
    """
    rows, K = w.shape
    assert K % GROUP == 0
    v = w.to(torch.float32).reshape(rows, K // GROUP, GROUP)
    amax = v.abs().amax(dim=2)
    s = (torch.clamp(amax, min=1e-8) / E4M3_MAX).to(torch.float16)
    s = torch.where(s > 0, s, torch.full_like(s, 2.0 ** -24))   # a scale that underflowed fp16
    r = torch.clamp(v / s.to(torch.float32).unsqueeze(2), -E4M3_MAX, E4M3_MAX)
    q = r.to(torch.float8_e4m3fn).view(torch.uint8).reshape(rows, K)
    return {"q": q.contiguous(), "scale": s.contiguous()}


def expert_weights(cfg: LayerConfig, e: int | str, device="cpu") -> dict[str, dict[str, torch.Tensor]]:
    """The weights the layer consumes for expert e, in the canonical formats:
    bf16: {"gate": {"w": bf16 [F,d]}, "up": ..., "down": {"w": bf16 [d,F]}}
    int4: {"gate": {"q","scale","zero"}, ...}   (see quantize_int4_g128)
    fp8:  {"gate": {"q","scale"}, ...}          (see quantize_fp8_g128)
    """
    src = expert_source(cfg, e, device)
    if cfg.fmt == "bf16":
        return {m: {"w": src[m]} for m in MATS}
    if cfg.fmt == "fp8":
        return {m: quantize_fp8_g128(src[m]) for m in MATS}
    return {m: quantize_int4_g128(src[m]) for m in MATS}


def active_expert_bytes(cfg: LayerConfig) -> int:
    """Bytes of one expert's weights in the layer's storage format (algorithmic)."""
    if cfg.fmt == "bf16":
        return 3 * cfg.d * cfg.F * 2
    if cfg.fmt == "fp8":   # one byte per weight + one fp16 scale per row and group
        return 3 * cfg.d * cfg.F + 3 * cfg.F * (cfg.d // GROUP) * 2
    return 3 * cfg.d * cfg.F // 2 + 3 * cfg.F * (cfg.d // GROUP) * 4
