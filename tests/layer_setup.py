"""Builds one synthetic MoE layer on the GPU (through the library's C ABI) and the
matching CPU-oracle description of the same seeded inputs."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import moe_expert_layer_03_gb300 as moe
import moe_synth as ms
import oracle

# max|err| <= TOL * RMS(out) for bf16 activations with fp32 accumulation; an element
# whose one bf16 ulp exceeds that (|v| above ~2.5-5 RMS) may instead differ from the
# exact value by at most one ulp: a bf16 output cannot be closer than half an ulp,
# and the fp32 sum before its rounding may fall on either side of the midpoint.
TOL = 2e-2
HOST_THREADS = max(1, os.cpu_count() or 1)


def row_chunk_width(cfg: ms.LayerConfig) -> int:
    """The GEMMs' row-chunk width for a layer (a host-side planning rule of the
    library, restated here only to choose which token rows to compare): a power
    of two of at least twice the mean rows per routed expert, 16..256, and 192
    instead of 256 for quantised weights."""
    mean = -(-cfg.A // cfg.E)
    bn = 16
    while bn < 2 * mean and bn < 256:
        bn <<= 1
    if cfg.fmt != "bf16" and bn > 128:
        bn = 192
    return bn


def chunk_edge_tokens(cfg: ms.LayerConfig, logits_np: np.ndarray) -> list[int]:
    """Tokens whose rows are the first and the last row of every row chunk of
    every expert group (and of the shared expert's group), from the oracle's own
    routing and permutation: every chunk, the short last one included, is then
    compared."""
    idx, _ = oracle.route_topk(logits_np, cfg.k)
    counts, offsets, _, tor = oracle.permute(idx, cfg.E)
    bn = row_chunk_width(cfg)
    groups = [(int(offsets[e]), int(counts[e]), tor) for e in range(cfg.E)]
    if cfg.shared:
        groups.append((0, cfg.T, np.arange(cfg.T, dtype=np.int32)))
    toks = set()
    for start, cnt, rows_to_tok in groups:
        if cnt == 0:
            continue
        nch = -(-cnt // bn)
        rpc = (-(-cnt // nch) + 15) // 16 * 16
        for c in range(nch):
            lo, hi = c * rpc, min(cnt, (c + 1) * rpc)
            if lo < hi:
                toks.add(int(rows_to_tok[start + lo]))
                toks.add(int(rows_to_tok[start + hi - 1]))
    return sorted(toks)


class GpuLayer:
    def __init__(self, cfg: ms.LayerConfig, device="cuda", logits: np.ndarray | None = None,
                 e2s: np.ndarray | None = None):
        self.cfg = cfg
        self.dev = device
        self.x = ms.make_x(cfg).to(device)
        self.logits_np = ms.make_logits(cfg) if logits is None else logits
        self.logits = torch.from_numpy(self.logits_np).to(device)
        self.e2s_np = ms.make_slot_table(cfg) if e2s is None else e2s
        n_slots = cfg.E + (1 if cfg.shared else 0)
        self.pool = moe.ExpertPool(n_slots, cfg.d, cfg.F, cfg.fmt, device=device)
        self.weights = {}
        for e in range(cfg.E):
            self.weights[e] = ms.expert_weights(cfg, e, device)
            self.pool.load_expert(int(self.e2s_np[e]), self.weights[e])
        self.routed = self.pool.view(torch.from_numpy(self.e2s_np.astype(np.int32)).to(device))
        self.shared = None
        if cfg.shared:
            self.weights["shared"] = ms.expert_weights(cfg, "shared", device)
            self.pool.load_expert(cfg.E, self.weights["shared"])
            self.shared = self.pool.view(torch.tensor([cfg.E], dtype=torch.int32, device=device))
        self._refs = {}

    def ref(self, e) -> oracle.ExpertRef:
        if e not in self._refs:
            w = self.weights[e]
            self._refs[e] = oracle.ExpertRef({m: {k: v.cpu() for k, v in w[m].items()} for m in w},
                                             self.cfg.fmt)
        return self._refs[e]

    def forward(self, **kw):
        out, ws = moe.layer_forward(self.x, self.logits, self.cfg.k, self.routed, self.shared, **kw)
        torch.cuda.synchronize()
        return out, ws

    def oracle_forward(self, tokens=None, threads: int = 1):
        """Oracle output rows (exact, float64) for the listed tokens (all if None),
        the tokens split over `threads` host threads (the C oracle releases the GIL)."""
        cfg = self.cfg
        toks = list(range(cfg.T)) if tokens is None else list(tokens)
        idx, _ = oracle.route_topk(self.logits_np[toks], cfg.k)
        used = sorted(set(int(e) for e in idx.ravel()))
        refs = [self.ref(used[0])] * cfg.E
        for e in used:
            refs[e] = self.ref(e)
        sh = self.ref("shared") if cfg.shared else None
        x = self.x.cpu()
        n = max(1, min(threads, len(toks)))
        parts = [toks[i::n] for i in range(n)]

        def run(part):
            return oracle.layer_forward(x, self.logits_np, cfg.k, refs, sh, cfg.d, cfg.F,
                                        tokens=part)[0]

        if n == 1:
            return run(toks)
        with cf.ThreadPoolExecutor(max_workers=n) as pool:
            outs = list(pool.map(run, parts))
        out = np.zeros((len(toks), cfg.d), np.float64)
        for i, o in enumerate(outs):
            out[i::n] = o
        return out


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits; normal range)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def assert_close_rms(got: np.ndarray, want: np.ndarray, tol: float = TOL, what: str = ""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    rms = float(np.sqrt(np.mean(want ** 2)))
    e = np.abs(got - want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    allowed = np.maximum(tol * rms, bf16_ulp(want))
    i = np.unravel_index(np.argmax(e / allowed), e.shape)
    assert np.all(e <= allowed), (f"{what}: |err| {e[i]:.4e} at {i} > max({tol} * RMS {rms:.4e}, "
                                  f"1 bf16 ulp {bf16_ulp(want[i]):.4e})")
    return float(e.max()), rms
