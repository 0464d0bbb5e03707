"""CPU oracle of the MoE FFN layer forward -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package.  It wraps the plain C reference in moe_oracle.c (built here with
gcc; no CUDA, no code shared with the library) behind numpy/torch-friendly
functions.  Every function cites its source passage in moe_oracle.c.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (plain -O2, no fast-math, no FMA contraction)."""
    src = os.path.join(_HERE, "moe_oracle.c")
    hdr = os.path.join(_HERE, "moe_oracle.h")
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_SO) or os.path.getmtime(_SO) < max(os.path.getmtime(src), os.path.getmtime(hdr)))
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-Wall", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class Matrix(C.Structure):
    _fields_ = [("fmt", C.c_int), ("rows", C.c_int), ("cols", C.c_int),
                ("w", C.c_void_p), ("q", C.c_void_p), ("scale", C.c_void_p), ("zero", C.c_void_p)]


class Expert(C.Structure):
    _fields_ = [("gate", Matrix), ("up", Matrix), ("down", Matrix)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            L.oracle_bf16_to_double.restype = C.c_double
            L.oracle_bf16_to_double.argtypes = [C.c_uint16]
            L.oracle_fp16_to_double.restype = C.c_double
            L.oracle_fp16_to_double.argtypes = [C.c_uint16]
            L.oracle_e4m3_to_double.restype = C.c_double
            L.oracle_e4m3_to_double.argtypes = [C.c_uint8]
            L.oracle_weight.restype = C.c_double
            L.oracle_weight.argtypes = [C.POINTER(Matrix), C.c_int, C.c_int]
            L.oracle_router_logits.argtypes = [P, P, C.c_int, C.c_int, C.c_int, P]
            L.oracle_route_topk.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P]
            L.oracle_permute.argtypes = [P, C.c_int, C.c_int, C.c_int, P, P, P, P]
            L.oracle_expert_ffn.argtypes = [P, C.c_int, C.c_int, C.POINTER(Expert), P, P]
            L.oracle_combine_row.argtypes = [P, P, C.c_int, C.c_int, P, P]
            L.oracle_layer_forward.argtypes = [P, P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                               C.POINTER(Expert), C.POINTER(Expert), P, C.c_int,
                                               P, P, P]
            _lib = L
    return _lib


# ----------------------------------------------------------------------------- marshalling
def _np(a, dtype) -> np.ndarray:
    """Contiguous host numpy view with the given dtype (bf16/fp16 tensors -> raw uint16)."""
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().contiguous()
        if a.dtype in (torch.bfloat16, torch.float16):
            a = a.view(torch.int16)
        a = a.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


class ExpertRef:
    """Holds host copies of one expert's weights and its ctypes description."""

    def __init__(self, weights: dict, fmt: str):
        self.keep = []
        mats = {}
        for name in ("gate", "up", "down"):
            m = weights[name]
            if fmt == "bf16":
                w = _np(m["w"], np.uint16)
                self.keep.append(w)
                mats[name] = Matrix(0, w.shape[0], w.shape[1], _ptr(w).value, None, None, None)
            elif fmt == "fp8":
                q = _np(m["q"], np.uint8)
                s = _np(m["scale"], np.uint16)
                self.keep += [q, s]
                mats[name] = Matrix(2, q.shape[0], q.shape[1], None, _ptr(q).value,
                                    _ptr(s).value, None)
            else:
                q = _np(m["q"], np.uint8)
                s = _np(m["scale"], np.uint16)
                z = _np(m["zero"], np.uint16)
                self.keep += [q, s, z]
                mats[name] = Matrix(1, q.shape[0], q.shape[1] * 2, None, _ptr(q).value,
                                    _ptr(s).value, _ptr(z).value)
        self.struct = Expert(mats["gate"], mats["up"], mats["down"])


# ----------------------------------------------------------------------------- API
def router_logits(x, w_router):
    """float64 [T, E] logits of bf16 x [T, d] against bf16 router rows [E, d]."""
    xb = _np(x, np.uint16)
    wb = _np(w_router, np.uint16)
    T, d = xb.shape
    E = wb.shape[0]
    if wb.shape[1] != d:
        raise ValueError("router_logits: x and w_router disagree on d")
    out = np.zeros((T, E), np.float64)
    rc = lib().oracle_router_logits(_ptr(xb), _ptr(wb), T, d, E, _ptr(out))
    if rc:
        raise ValueError("oracle_router_logits: bad arguments")
    return out


def route_topk(logits, k: int):
    lg = _np(logits, np.float32)
    T, E = lg.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    rc = lib().oracle_route_topk(_ptr(lg), T, E, k, _ptr(idx), _ptr(w))
    if rc:
        raise ValueError("oracle_route_topk: bad arguments")
    return idx, w


def permute(idx, E: int):
    ix = _np(idx, np.int32)
    T, k = ix.shape
    A = T * k
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    roa = np.zeros(A, np.int32)
    tor = np.zeros(A, np.int32)
    rc = lib().oracle_permute(_ptr(ix), T, k, E, _ptr(counts), _ptr(offsets), _ptr(roa), _ptr(tor))
    if rc:
        raise ValueError("oracle_permute: bad arguments")
    return counts, offsets, roa, tor


def expert_ffn(x_row, expert: ExpertRef, d: int, F: int):
    """Returns (h [F], y [d]) in float64 for one bf16 token row."""
    xr = _np(x_row, np.uint16).reshape(-1)
    h = np.zeros(F, np.float64)
    y = np.zeros(d, np.float64)
    rc = lib().oracle_expert_ffn(_ptr(xr), d, F, C.byref(expert.struct), _ptr(h), _ptr(y))
    if rc:
        raise ValueError("oracle_expert_ffn: bad arguments")
    return h, y


def combine_row(y_rows, w, y_shared=None):
    ys = [_np(y, np.uint16).reshape(-1) for y in y_rows]
    k, d = len(ys), ys[0].shape[0]
    arr = (C.c_void_p * k)(*[_ptr(y).value for y in ys])
    wf = _np(np.asarray(w, np.float32), np.float32)
    sh = _np(y_shared, np.uint16).reshape(-1) if y_shared is not None else None
    out = np.zeros(d, np.float64)
    rc = lib().oracle_combine_row(C.cast(arr, C.c_void_p), _ptr(wf), k, d,
                                  _ptr(sh) if sh is not None else None, _ptr(out))
    if rc:
        raise ValueError("oracle_combine_row: bad arguments")
    return out


def layer_forward(x, logits, k: int, experts: list, shared: ExpertRef | None, d: int, F: int,
                  tokens=None):
    """out float64 [n, d], idx [n, k], w [n, k] for the listed tokens (all if None)."""
    xb = _np(x, np.uint16)
    lg = _np(logits, np.float32)
    T, E = lg.shape
    arr = (Expert * E)(*[e.struct for e in experts])
    tl = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, np.int32))
    n = T if tl is None else tl.shape[0]
    out = np.zeros((n, d), np.float64)
    idx = np.zeros((n, k), np.int32)
    w = np.zeros((n, k), np.float32)
    rc = lib().oracle_layer_forward(_ptr(xb), _ptr(lg), T, E, k, d, F, arr,
                                    C.byref(shared.struct) if shared is not None else None,
                                    _ptr(tl) if tl is not None else None, n, _ptr(out),
                                    _ptr(idx), _ptr(w))
    if rc:
        raise ValueError("oracle_layer_forward: bad arguments")
    return out, idx, w


def bf16_bits_to_float(a) -> np.ndarray:
    a = _np(a, np.uint16).astype(np.uint32) << 16
    return a.view(np.float32)
