"""GB300 (sm_103a) MoE FFN layer forward: Python binding of the C ABI in include/moe.h.

This module only marshals arguments (torch tensors -> device pointers, the
current torch stream -> cudaStream_t) and calls the CUDA library
libmoe_gb300.so; every step of the layer runs in the library's kernels.  There
is no CPU path: if the library is not built, every call raises.

Typical use::

    import moe_expert_layer_03_gb300 as moe
    pool = moe.ExpertPool(n_slots=8, d_model=4096, d_ff=14336, fmt=moe.W_INT4)
    for e in range(8):
        pool.load_expert(e, canonical_weights_of_expert[e])     # device tensors
    routed = pool.view(expert_to_slot)                          # int32 [E] on the device
    out = moe.layer_forward(x, logits, k=2, routed=routed)      # bf16 [T, d]
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

from .build import LIB, build  # noqa: F401  (build() compiles the library in-tree)

W_BF16 = 0
W_INT4 = 1
W_FP8 = 2
FMT = {"bf16": W_BF16, "int4": W_INT4, "fp8": W_FP8}
N_STAGES = 6
STAGES = ("route", "permute", "gather", "gate_up", "down", "combine")
DEVERR = {1: "timeout", 2: "expert index out of range", 4: "slot out of range", 8: "bad offsets"}

EXPORTS = ("moe_status_str", "moe_slot_bytes", "moe_prepack_expert", "moe_route_topk",
           "moe_permute_workspace_bytes", "moe_permute", "moe_grouped_ffn_workspace_bytes",
           "moe_grouped_ffn", "moe_combine", "moe_layer_workspace_bytes", "moe_layer_forward",
           "moe_layer_forward_timed", "moe_layer_launch_count", "moe_layer_router_launch_count",
           "moe_last_device_error",
           "moe_layer_forward_noalloc", "moe_noalloc_last_device_error", "moe_router_logits", "moe_layer_forward_router",
           "moe_cache_create", "moe_cache_ensure", "moe_cache_plan", "moe_cache_prefetch",
           "moe_cache_commit", "moe_cache_stats", "moe_cache_destroy", "moe_debug_gemm_fault")


class MoeError(RuntimeError):
    pass


class MoePool(C.Structure):
    _fields_ = [("n_experts", C.c_int), ("n_slots", C.c_int), ("d_model", C.c_int),
                ("d_ff", C.c_int), ("fmt", C.c_int), ("pool", C.c_void_p),
                ("slot_bytes", C.c_size_t), ("expert_to_slot", C.c_void_p)]


class CacheCounters(C.Structure):
    _fields_ = [("hits", C.c_longlong), ("misses", C.c_longlong), ("bytes_copied", C.c_longlong)]


class ExpertSrc(C.Structure):
    _fields_ = [("w", C.c_void_p * 3), ("scale", C.c_void_p * 3), ("zero", C.c_void_p * 3)]


_lib = None
_lock = threading.Lock()


def lib() -> C.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise MoeError(f"CUDA library not built ({LIB}); run moe_expert_layer_03_gb300.build()")
            L = C.CDLL(LIB)
            P, I, S = C.c_void_p, C.c_int, C.c_size_t
            L.moe_status_str.restype = C.c_char_p
            L.moe_status_str.argtypes = [I]
            L.moe_slot_bytes.restype = S
            L.moe_slot_bytes.argtypes = [I, I, I]
            L.moe_prepack_expert.argtypes = [I, I, I, C.POINTER(ExpertSrc), P, P]
            L.moe_router_logits.argtypes = [P, P, I, I, I, P, P]
            L.moe_layer_forward_router.argtypes = [P, P, I, I, C.POINTER(MoePool),
                                                   C.POINTER(MoePool), P, P, P, S, P]
            L.moe_cache_create.argtypes = [C.POINTER(MoePool), P, I, C.POINTER(P)]
            L.moe_cache_ensure.argtypes = [P, P, I, P]
            L.moe_cache_prefetch.argtypes = [P, P, I, P]
            L.moe_cache_commit.argtypes = [P, P, I, P]
            L.moe_cache_plan.argtypes = [P, P, I, P, P, C.POINTER(I)]
            L.moe_cache_stats.argtypes = [P, C.POINTER(CacheCounters)]
            L.moe_cache_destroy.argtypes = [P]
            L.moe_cache_destroy.restype = None
            L.moe_route_topk.argtypes = [P, I, I, I, P, P, P]
            L.moe_permute_workspace_bytes.restype = S
            L.moe_permute_workspace_bytes.argtypes = []
            L.moe_permute.argtypes = [P, P, I, I, I, I, P, P, P, P, P, P, S, P]
            L.moe_grouped_ffn_workspace_bytes.restype = S
            L.moe_grouped_ffn_workspace_bytes.argtypes = [I, C.POINTER(MoePool)]
            L.moe_grouped_ffn.argtypes = [P, P, I, C.POINTER(MoePool), P, P, S, P]
            L.moe_combine.argtypes = [P, P, P, P, I, I, I, P, P]
            L.moe_layer_workspace_bytes.restype = S
            L.moe_layer_workspace_bytes.argtypes = [I, I, C.POINTER(MoePool), C.POINTER(MoePool)]
            L.moe_layer_forward.argtypes = [P, P, I, I, C.POINTER(MoePool), C.POINTER(MoePool), P,
                                            P, S, P]
            L.moe_layer_forward_timed.argtypes = [P, P, I, I, C.POINTER(MoePool),
                                                  C.POINTER(MoePool), P, P, S, P, P]
            L.moe_layer_launch_count.argtypes = [I, I, C.POINTER(MoePool), C.POINTER(MoePool)]
            L.moe_layer_router_launch_count.argtypes = [I, I, C.POINTER(MoePool), C.POINTER(MoePool)]
            L.moe_last_device_error.argtypes = [P, C.POINTER(C.c_int), P]
            L.moe_debug_gemm_fault.argtypes = [I, C.c_ulonglong]
            _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise MoeError(f"{what}: {lib().moe_status_str(status).decode()} (status {status})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


# ----------------------------------------------------------------------------- expert pool
class PoolView:
    """A moe_pool struct plus the tensors it points at (kept alive)."""

    def __init__(self, pool: "ExpertPool", expert_to_slot: torch.Tensor):
        assert expert_to_slot.dtype == torch.int32 and expert_to_slot.is_cuda
        self.pool = pool
        self.e2s = expert_to_slot.contiguous()
        self.struct = MoePool(self.e2s.numel(), pool.n_slots, pool.d_model, pool.d_ff, pool.fmt,
                              pool.buf.data_ptr(), pool.slot_bytes, self.e2s.data_ptr())

    @property
    def ref(self):
        return C.byref(self.struct)


class ExpertPool:
    """HBM-resident expert pool: n_slots slots of the library's prepacked layout."""

    def __init__(self, n_slots: int, d_model: int, d_ff: int, fmt: int | str, device="cuda"):
        self.fmt = FMT[fmt] if isinstance(fmt, str) else int(fmt)
        self.n_slots, self.d_model, self.d_ff = n_slots, d_model, d_ff
        raw = lib().moe_slot_bytes(self.fmt, d_model, d_ff)
        if raw == 0:
            raise MoeError(f"unsupported expert shape d_model={d_model} d_ff={d_ff}")
        self.slot_bytes = (raw + 255) // 256 * 256
        self.buf = torch.empty(n_slots * self.slot_bytes, dtype=torch.uint8, device=device)
        assert self.buf.data_ptr() % 256 == 0

    def slot_ptr(self, slot: int) -> int:
        return self.buf.data_ptr() + slot * self.slot_bytes

    def load_expert(self, slot: int, weights: dict, stream=None):
        """Prepack one expert (canonical device tensors, see moe.h) into `slot`."""
        src = ExpertSrc()
        keep = []
        for m, name in enumerate(("gate", "up", "down")):
            wm = weights[name]
            if self.fmt == W_BF16:
                w = wm["w"].contiguous()
                keep.append(w)
                src.w[m] = w.data_ptr()
            elif self.fmt == W_FP8:
                q, s = (wm[k].contiguous() for k in ("q", "scale"))
                keep += [q, s]
                src.w[m], src.scale[m] = q.data_ptr(), s.data_ptr()
            else:
                q, s, z = (wm[k].contiguous() for k in ("q", "scale", "zero"))
                keep += [q, s, z]
                src.w[m], src.scale[m], src.zero[m] = q.data_ptr(), s.data_ptr(), z.data_ptr()
        for t in keep:
            if not t.is_cuda:
                raise MoeError("expert weights must be device tensors")
        _check(lib().moe_prepack_expert(self.fmt, self.d_model, self.d_ff, C.byref(src),
                                        C.c_void_p(self.slot_ptr(slot)), _stream(stream)),
               "moe_prepack_expert")
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()

    def view(self, expert_to_slot: torch.Tensor) -> PoolView:
        return PoolView(self, expert_to_slot)


class ExpertCache:
    """A pool larger than HBM: every expert's prepacked image in pinned host
    memory (the cold tier, reached over NVLink-C2C on a Grace-Blackwell node) and
    `pool`'s slots as the hot tier, filled on demand with LRU replacement
    (moe_cache_* in moe.h).  `view` is the routed pool view the layer takes; its
    expert -> slot table is maintained by the cache."""

    COPY_AUTO, COPY_ENGINE, COPY_SM = 0, 1, 2

    def __init__(self, pool: "ExpertPool", n_experts: int, copy_mode: int = 0):
        self.pool, self.n_experts = pool, n_experts
        self.host = torch.empty(n_experts * pool.slot_bytes, dtype=torch.uint8, pin_memory=True)
        self.e2s = torch.full((n_experts,), -1, dtype=torch.int32, device=pool.buf.device)
        self.view = PoolView(pool, self.e2s)
        h = C.c_void_p()
        _check(lib().moe_cache_create(self.view.ref, C.c_void_p(self.host.data_ptr()), copy_mode,
                                      C.byref(h)), "moe_cache_create")
        self._h = h
        self._scratch = None

    def load_expert(self, e: int, weights: dict):
        """Prepack expert e (canonical device tensors) into its host image."""
        if self._scratch is None:
            p = self.pool
            self._scratch = ExpertPool(1, p.d_model, p.d_ff, p.fmt, device=p.buf.device)
        self._scratch.load_expert(0, weights)
        sb = self.pool.slot_bytes
        self.host[e * sb:(e + 1) * sb].copy_(self._scratch.buf)

    def load_image(self, e: int, image: torch.Tensor):
        """Expert e's host image from an already prepacked slot image (uint8,
        slot_bytes long, e.g. a slot of another pool of the same shape)."""
        sb = self.pool.slot_bytes
        if image.dtype != torch.uint8 or image.numel() != sb:
            raise MoeError("expert image must be slot_bytes uint8")
        self.host[e * sb:(e + 1) * sb].copy_(image)

    def ensure(self, experts, stream=None):
        ex = (C.c_int32 * len(experts))(*[int(e) for e in experts])
        _check(lib().moe_cache_ensure(self._h, C.cast(ex, C.c_void_p), len(experts), _stream(stream)),
               "moe_cache_ensure")

    def prefetch(self, experts, stream):
        """Copies the listed experts in on `stream` (a copy stream) without touching
        the table; never evicts a committed expert (moe_cache_prefetch)."""
        ex = (C.c_int32 * max(1, len(experts)))(*[int(e) for e in experts])
        _check(lib().moe_cache_prefetch(self._h, C.cast(ex, C.c_void_p), len(experts), _stream(stream)),
               "moe_cache_prefetch")

    def commit(self, experts, stream=None):
        """Makes the listed (resident) experts the ones the layer reads, on `stream`
        (the compute stream), after their copies (moe_cache_commit)."""
        ex = (C.c_int32 * max(1, len(experts)))(*[int(e) for e in experts])
        _check(lib().moe_cache_commit(self._h, C.cast(ex, C.c_void_p), len(experts), _stream(stream)),
               "moe_cache_commit")

    def plan(self, experts):
        """The loads ensure() would do (and its bookkeeping), without CUDA work."""
        n = self.pool.n_slots
        ex = (C.c_int32 * max(1, len(experts)))(*[int(e) for e in experts])
        le, ls, nl = (C.c_int32 * n)(), (C.c_int32 * n)(), C.c_int(0)
        _check(lib().moe_cache_plan(self._h, C.cast(ex, C.c_void_p), len(experts), C.cast(le, C.c_void_p),
                                    C.cast(ls, C.c_void_p), C.byref(nl)), "moe_cache_plan")
        return [(le[i], ls[i]) for i in range(nl.value)]

    def stats(self) -> dict:
        c = CacheCounters()
        _check(lib().moe_cache_stats(self._h, C.byref(c)), "moe_cache_stats")
        return {"hits": c.hits, "misses": c.misses, "bytes_copied": c.bytes_copied}

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.moe_cache_destroy(h)
            self._h = None


# ----------------------------------------------------------------------------- workspaces
def layer_workspace_bytes(T: int, k: int, routed: PoolView, shared: PoolView | None = None) -> int:
    return lib().moe_layer_workspace_bytes(T, k, routed.ref, shared.ref if shared else None)


def grouped_ffn_workspace_bytes(A: int, pool: PoolView) -> int:
    return lib().moe_grouped_ffn_workspace_bytes(A, pool.ref)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def debug_gemm_fault(stop_stage: int = -1, wait_ns: int = 0):
    """Failure-path test hook (moe_debug_gemm_fault): the gate/up GEMM's producer
    stops after `stop_stage` stages and the GEMMs' waits give up after `wait_ns`;
    debug_gemm_fault() restores the defaults."""
    _check(lib().moe_debug_gemm_fault(stop_stage, wait_ns), "moe_debug_gemm_fault")


def last_device_error(ws: torch.Tensor, stream=None) -> int:
    """The ORed device error code of the last call that used this workspace (syncs)."""
    code = C.c_int(0)
    st = lib().moe_last_device_error(_ptr(ws), C.byref(code), _stream(stream))
    if st not in (0, 5):
        _check(st, "moe_last_device_error")
    return code.value


# ----------------------------------------------------------------------------- hot path
def router_logits(x: torch.Tensor, w_router: torch.Tensor, logits=None, stream=None):
    """fp32 [T, E] logits = x (bf16 [T, d]) . w_router (bf16 [E, d]) per row."""
    T, d = x.shape
    E = w_router.shape[0]
    logits = logits if logits is not None else torch.empty(T, E, dtype=torch.float32,
                                                           device=x.device)
    _check(lib().moe_router_logits(_ptr(x), _ptr(w_router), T, d, E, _ptr(logits),
                                   _stream(stream)), "moe_router_logits")
    return logits


def route_topk(logits: torch.Tensor, k: int, idx=None, w=None, stream=None):
    T, E = logits.shape
    idx = idx if idx is not None else torch.empty(T, k, dtype=torch.int32, device=logits.device)
    w = w if w is not None else torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _check(lib().moe_route_topk(_ptr(logits), T, E, k, _ptr(idx), _ptr(w), _stream(stream)),
           "moe_route_topk")
    return idx, w


def permute(topk_idx: torch.Tensor, x: torch.Tensor, E: int, ws=None, stream=None):
    T, k = topk_idx.shape
    d = x.shape[1]
    A = T * k
    dev = x.device
    out = {
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "row_of_assign": torch.empty(A, dtype=torch.int32, device=dev),
        "token_of_row": torch.empty(A, dtype=torch.int32, device=dev),
        "x_perm": torch.empty(A, d, dtype=torch.bfloat16, device=dev),
    }
    ws = ws if ws is not None else workspace(lib().moe_permute_workspace_bytes(), dev)
    _check(lib().moe_permute(_ptr(topk_idx), _ptr(x), T, k, E, d, _ptr(out["counts"]),
                             _ptr(out["offsets"]), _ptr(out["row_of_assign"]),
                             _ptr(out["token_of_row"]), _ptr(out["x_perm"]), _ptr(ws), ws.numel(),
                             _stream(stream)), "moe_permute")
    out["ws"] = ws
    return out


def grouped_ffn(x_perm: torch.Tensor, offsets: torch.Tensor, pool: PoolView, y_perm=None, ws=None,
                stream=None):
    A, d = x_perm.shape
    y_perm = y_perm if y_perm is not None else torch.empty(A, d, dtype=torch.bfloat16,
                                                           device=x_perm.device)
    ws = ws if ws is not None else workspace(grouped_ffn_workspace_bytes(A, pool), x_perm.device)
    _check(lib().moe_grouped_ffn(_ptr(x_perm), _ptr(offsets), A, pool.ref, _ptr(y_perm), _ptr(ws),
                                 ws.numel(), _stream(stream)), "moe_grouped_ffn")
    return y_perm, ws


def combine(y_perm: torch.Tensor, row_of_assign: torch.Tensor, topk_w: torch.Tensor,
            shared_y: torch.Tensor | None = None, out=None, stream=None):
    T, k = topk_w.shape
    d = y_perm.shape[1]
    out = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=y_perm.device)
    _check(lib().moe_combine(_ptr(y_perm), _ptr(row_of_assign), _ptr(topk_w), _ptr(shared_y), T, k,
                             d, _ptr(out), _stream(stream)), "moe_combine")
    return out


def layer_forward(x: torch.Tensor, logits: torch.Tensor, k: int, routed: PoolView,
                  shared: PoolView | None = None, out=None, ws=None, events=None, stream=None):
    """out = MoE layer(x): bf16 [T, d].  `events`: optional N_STAGES+1 torch.cuda.Event."""
    T, d = x.shape
    out = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=x.device)
    need = layer_workspace_bytes(T, k, routed, shared)
    if need == 0:
        raise MoeError("moe_layer_workspace_bytes: invalid layer description")
    ws = ws if ws is not None else workspace(need, x.device)
    sh = shared.ref if shared is not None else None
    if events is None:
        st = lib().moe_layer_forward(_ptr(x), _ptr(logits), T, k, routed.ref, sh, _ptr(out),
                                     _ptr(ws), ws.numel(), _stream(stream))
    else:
        s = stream if stream is not None else torch.cuda.current_stream()
        for e in events:          # torch creates the CUDA event on its first record
            if not e.cuda_event:
                e.record(s)
        arr = (C.c_void_p * (N_STAGES + 1))(*[e.cuda_event for e in events])
        st = lib().moe_layer_forward_timed(_ptr(x), _ptr(logits), T, k, routed.ref, sh, _ptr(out),
                                           _ptr(ws), ws.numel(), _stream(stream), arr)
    _check(st, "moe_layer_forward")
    return out, ws


def layer_forward_router(x: torch.Tensor, w_router: torch.Tensor, k: int, routed: PoolView,
                         shared: PoolView | None = None, logits=None, out=None, ws=None,
                         stream=None):
    """The layer from the token rows and the router weight (bf16 [E, d]): returns
    (out bf16 [T, d], logits fp32 [T, E], ws)."""
    T, d = x.shape
    E = routed.struct.n_experts
    out = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=x.device)
    logits = logits if logits is not None else torch.empty(T, E, dtype=torch.float32,
                                                           device=x.device)
    need = layer_workspace_bytes(T, k, routed, shared)
    if need == 0:
        raise MoeError("moe_layer_workspace_bytes: invalid layer description")
    ws = ws if ws is not None else workspace(need, x.device)
    sh = shared.ref if shared is not None else None
    _check(lib().moe_layer_forward_router(_ptr(x), _ptr(w_router), T, k, routed.ref, sh,
                                          _ptr(logits), _ptr(out), _ptr(ws), ws.numel(),
                                          _stream(stream)), "moe_layer_forward_router")
    return out, logits, ws


def layer_launch_count(T: int, k: int, routed: PoolView, shared: PoolView | None = None) -> int:
    return lib().moe_layer_launch_count(T, k, routed.ref, shared.ref if shared else None)


def layer_router_launch_count(T: int, k: int, routed: PoolView, shared: PoolView | None = None) -> int:
    """Kernel launches of one layer_forward_router call."""
    return lib().moe_layer_router_launch_count(T, k, routed.ref, shared.ref if shared else None)


class LayerGraph:
    """One layer forward captured as a CUDA graph over fixed device buffers.

    The graph reads ``self.x`` (bf16 [T, d]) and ``self.logits`` (fp32 [T, E])
    and writes ``self.out`` (bf16 [T, d]); fill the inputs (copies on the
    replaying stream), then ``replay()``.  Routing, permutation and the GEMM
    work lists are built on the device from the input values, so one capture
    serves every input of the same shape.  Replaying saves the host launch
    work and shortens the gaps between the layer's kernels (decode steps are
    a few hundred microseconds).

    host_io=True also captures the copies from pinned host buffers
    ``self.x_host`` / ``self.logits_host`` into the device inputs and from
    ``self.out`` back to ``self.out_host``: one replay is then a whole step from
    host memory to host memory (read ``out_host`` after synchronising).

    router_weight (bf16 [E, d] on the device): the step starts from the token
    rows alone (moe_layer_forward_router); ``self.logits`` is then written by
    each replay instead of read.
    """

    def __init__(self, T: int, k: int, routed: PoolView, shared: PoolView | None = None,
                 device=None, host_io: bool = False, router_weight: torch.Tensor | None = None):
        dev = torch.device(device) if device is not None else routed.e2s.device
        E, d = routed.struct.n_experts, routed.struct.d_model
        self.k, self.routed, self.shared = k, routed, shared
        self.router_weight = router_weight
        self.x = torch.zeros(T, d, dtype=torch.bfloat16, device=dev)
        self.logits = torch.zeros(T, E, dtype=torch.float32, device=dev)
        self.out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
        self.ws = workspace(layer_workspace_bytes(T, k, routed, shared), dev)
        self.host_io = host_io
        if host_io:
            self.x_host = torch.zeros(T, d, dtype=torch.bfloat16).pin_memory()
            self.logits_host = torch.zeros(T, E, dtype=torch.float32).pin_memory()
            self.out_host = torch.empty(T, d, dtype=torch.bfloat16).pin_memory()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self._forward()   # first call: one-time library set-up happens outside the capture
            side.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=side):
                self._forward()
        torch.cuda.current_stream(dev).wait_stream(side)

    def _forward(self):
        if self.host_io:
            self.x.copy_(self.x_host, non_blocking=True)
            self.logits.copy_(self.logits_host, non_blocking=True)
        if self.router_weight is not None:
            layer_forward_router(self.x, self.router_weight, self.k, self.routed, self.shared,
                                 logits=self.logits, out=self.out, ws=self.ws)
        else:
            layer_forward(self.x, self.logits, self.k, self.routed, self.shared, out=self.out, ws=self.ws)
        if self.host_io:
            self.out_host.copy_(self.out, non_blocking=True)

    def replay(self) -> torch.Tensor:
        self.graph.replay()
        return self.out


class LayerPipeline:
    """Host-to-host layer steps with the copies overlapped with compute.

    Two slots of device inputs/outputs and pinned host buffers
    (``x_host[s]``, ``logits_host[s]``, ``out_host[s]``).  Step i computes
    slot i % 2 while a second stream copies step i - 1's output back to the
    host and step i + 1's inputs in (both in the other slot), so on a stream
    the copies run under the compute instead of around it.  One CUDA graph per
    slot holds both branches; replays on one stream order the steps.

        pipe.x_host[0][...] = ...; pipe.logits_host[0][...] = ...   # step 0
        pipe.start()                      # copies step 0's inputs in
        for i in range(n):
            # before step i: the inputs of step i + 1 in the host slot (i + 1) % 2
            pipe.step(i)
        pipe.finish(n - 1)                # copies the last output out
        torch.cuda.current_stream().synchronize()
        # step i's output: out_host[i % 2], valid once step i + 1 (or finish) has run

    The host slots of step i + 1's inputs must be filled before ``step(i)`` is
    called, and ``out_host[i % 2]`` read before ``step(i + 2)`` overwrites it.
    """

    def __init__(self, T: int, k: int, routed: PoolView, shared: PoolView | None = None, device=None):
        dev = torch.device(device) if device is not None else routed.e2s.device
        E, d = routed.struct.n_experts, routed.struct.d_model
        self.k, self.routed, self.shared = k, routed, shared
        self.x = [torch.zeros(T, d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.logits = [torch.zeros(T, E, dtype=torch.float32, device=dev) for _ in range(2)]
        self.out = [torch.zeros(T, d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.x_host = [torch.zeros(T, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        self.logits_host = [torch.zeros(T, E, dtype=torch.float32).pin_memory() for _ in range(2)]
        self.out_host = [torch.zeros(T, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        self.ws = workspace(layer_workspace_bytes(T, k, routed, shared), dev)
        self.copy_stream = torch.cuda.Stream(device=dev)
        main = torch.cuda.Stream(device=dev)
        main.wait_stream(torch.cuda.current_stream(dev))
        self.graphs = []
        with torch.cuda.stream(main):
            self._forward(0)   # first call: one-time library set-up happens outside the capture
            main.synchronize()
            for s in range(2):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=main):
                    self._step_body(s, main)
                self.graphs.append(g)
        torch.cuda.current_stream(dev).wait_stream(main)

    def _forward(self, s: int):
        layer_forward(self.x[s], self.logits[s], self.k, self.routed, self.shared, out=self.out[s], ws=self.ws)

    def _step_body(self, s: int, main):
        o = 1 - s
        self.copy_stream.wait_stream(main)
        with torch.cuda.stream(self.copy_stream):   # the other slot: last output out, next inputs in
            self.out_host[o].copy_(self.out[o], non_blocking=True)
            self.x[o].copy_(self.x_host[o], non_blocking=True)
            self.logits[o].copy_(self.logits_host[o], non_blocking=True)
        self._forward(s)
        main.wait_stream(self.copy_stream)

    def start(self):
        """Copies step 0's inputs (host slot 0) to the device, on the current stream."""
        self.x[0].copy_(self.x_host[0], non_blocking=True)
        self.logits[0].copy_(self.logits_host[0], non_blocking=True)

    def step(self, i: int):
        self.graphs[i % 2].replay()

    def finish(self, last: int):
        """Copies the last step's output to ``out_host[last % 2]``, on the current stream."""
        self.out_host[last % 2].copy_(self.out[last % 2], non_blocking=True)
