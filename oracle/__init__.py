"""CPU oracle for the local W4A16 MoE forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA product path never does.

The arithmetic lives in ``w4a16_oracle.cpp`` (plain C++ loops, double for the
expert MLPs, FP32 for the top-k combine).  This module only compiles it with
g++ and marshals numpy/torch arrays into it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.cpp")
_LIB = os.path.join(_HERE, "libw4a16_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle library in place (g++, OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            L.oracle_unpack_along_k.argtypes = [P, i64, i64, P]
            L.oracle_unpack_along_rows.argtypes = [P, i64, i64, P]
            L.oracle_dequant.argtypes = [P, P, i64, i64, ctypes.c_int, P]
            L.oracle_bf16_encode.argtypes = [P, i64, P]
            L.oracle_fp16_encode.argtypes = [P, i64, P]
            L.oracle_fp16_decode.argtypes = [P, i64, P]
            L.oracle_prepare_routes.argtypes = [P, i32, P, i32, P, P, P, i64, P, P, i64, P]
            L.oracle_prepare_routes.restype = ctypes.c_int
            L.oracle_moe_forward.argtypes = [P, i32, P, P, P, P, P, P, P, i32, P, i32, P, P, i32]
            L.oracle_moe_forward.restype = ctypes.c_int
            L.oracle_num_threads.restype = ctypes.c_int
            L.oracle_route_topk.argtypes = [P, i32, i32, i32, P, P]
            L.oracle_route_topk.restype = ctypes.c_int
            L.oracle_masked_routes.argtypes = [P, i32, i32, i32, P, P]
            L.oracle_masked_routes.restype = ctypes.c_int
            L.oracle_relayout_interleaved.argtypes = [P, i32, i64, i64, i64, P]
            L.oracle_relayout_interleaved.restype = ctypes.c_int
            _lib = L
    return _lib


def _np(t, dtype=None):
    """Contiguous numpy view of a CPU tensor / array (bf16/fp16 -> uint16 bits)."""
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.view(torch.int16)
        a = t.numpy()
    else:
        a = np.ascontiguousarray(t)
    if dtype is not None:
        a = np.ascontiguousarray(a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype))
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def desc_array(cfg) -> np.ndarray:
    return np.array([cfg.num_experts, cfg.expert_offset, cfg.hidden, cfg.inter, cfg.top_k,
                     cfg.act, cfg.scale_kind, cfg.act_dtype], dtype=np.int32)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def unpack_along_k(packed, rows: int, cols: int) -> np.ndarray:
    p = _np(packed, np.uint8)
    q = np.empty((rows, cols), dtype=np.int8)
    lib().oracle_unpack_along_k(_ptr(p), rows, cols, _ptr(q))
    return q


def unpack_along_rows(packed, rows: int, cols: int) -> np.ndarray:
    p = _np(packed, np.uint8)
    q = np.empty((rows, cols), dtype=np.int8)
    lib().oracle_unpack_along_rows(_ptr(p), rows, cols, _ptr(q))
    return q


def dequant(packed, scales, rows: int, cols: int, scale_kind: int) -> np.ndarray:
    p = _np(packed, np.uint8)
    s = _np(scales, np.uint16)
    out = np.empty((rows, cols), dtype=np.float64)
    lib().oracle_dequant(_ptr(p), _ptr(s), rows, cols, scale_kind, _ptr(out))
    return out


def bf16_encode(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(a.shape, dtype=np.uint16)
    lib().oracle_bf16_encode(_ptr(a), a.size, _ptr(out))
    return out


def fp16_encode(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(a.shape, dtype=np.uint16)
    lib().oracle_fp16_encode(_ptr(a), a.size, _ptr(out))
    return out


def fp16_decode(bits) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    out = np.empty(a.shape, dtype=np.float64)
    lib().oracle_fp16_decode(_ptr(a), a.size, _ptr(out))
    return out


def prepare_routes(cfg, ids, bm: int):
    """Route layout for tile height ``bm``.  Returns a dict of numpy arrays:
    counts [E], offs [E+1], perm [offs[E]], inv [T*k], tiles [n, 4]."""
    ids_np = _np(ids, np.int32)
    T = ids_np.shape[0]
    R = T * cfg.top_k
    E = cfg.num_experts
    perm_cap = R + E * (bm - 1) + 1
    tiles_cap = R + E + 1
    counts = np.zeros(E, np.int32)
    offs = np.zeros(E + 1, np.int32)
    perm = np.zeros(perm_cap, np.int32)
    inv = np.zeros(max(R, 1), np.int32)
    tiles = np.zeros((tiles_cap, 4), np.int32)
    nt = np.zeros(1, np.int32)
    d = desc_array(cfg)
    rc = lib().oracle_prepare_routes(_ptr(d), T, _ptr(ids_np), bm, _ptr(counts), _ptr(offs),
                                     _ptr(perm), perm_cap, _ptr(inv), _ptr(tiles), tiles_cap, _ptr(nt))
    if rc != 0:
        raise RuntimeError(f"oracle_prepare_routes failed: {rc}")
    return dict(counts=counts, offs=offs, perm=perm[: offs[E]].copy(), inv=inv[:R].copy(),
                tiles=tiles[: nt[0]].copy(), num_tiles=int(nt[0]))


def relayout_interleaved(packed, scale_kind: int, E: int, N: int, K: int) -> np.ndarray:
    """The interleaved packed-weight layout of ``w4a16_moe_relayout_weights``
    (see w4a16_oracle.cpp): uint8 [E, N, K/2] from the checkpoint layout."""
    p = _np(packed, np.uint8)
    out = np.empty((E, N, K // 2), np.uint8)
    rc = lib().oracle_relayout_interleaved(_ptr(p), int(scale_kind), E, N, K, _ptr(out))
    if rc != 0:
        raise RuntimeError(f"oracle_relayout_interleaved failed: {rc}")
    return out


def route_topk(logits, top_k: int):
    """Router softmax + top-k.  logits [T, G] FP32; returns (ids int32 [T, k],
    weights float64 [T, k]) (the oracle's definition, see w4a16_oracle.cpp)."""
    lg = np.ascontiguousarray(_np(logits, np.float32))
    T, G = lg.shape
    ids = np.zeros((T, top_k), np.int32)
    w = np.zeros((T, top_k), np.float64)
    rc = lib().oracle_route_topk(_ptr(lg), T, G, top_k, _ptr(ids), _ptr(w))
    if rc != 0:
        raise RuntimeError(f"oracle_route_topk failed: {rc}")
    return ids, w


def masked_routes(counts, max_rows: int, expert_offset: int = 0):
    """Routes of the masked-count layout: (ids int32 [E * max_rows, 1],
    weights float32 [E * max_rows, 1]); see w4a16_oracle.cpp."""
    c = np.ascontiguousarray(_np(counts, np.int32))
    E = c.shape[0]
    ids = np.zeros((E * max_rows, 1), np.int32)
    w = np.zeros((E * max_rows, 1), np.float32)
    rc = lib().oracle_masked_routes(_ptr(c), E, max_rows, expert_offset, _ptr(ids), _ptr(w))
    if rc != 0:
        raise RuntimeError(f"oracle_masked_routes failed: {rc}")
    return ids, w


def masked_forward(cfg, x, weights, counts, max_rows: int, nthreads: int = 0):
    """Expert MLPs on the masked-count layout.  x [E * max_rows, H] (16-bit
    bits or tensor); cfg must have top_k == 1.  Returns (acc fp32 [E*max_rows, H],
    out bits): the forward over masked_routes()."""
    if cfg.top_k != 1:
        raise ValueError("the masked-count layout routes every row once: top_k must be 1")
    ids, w = masked_routes(counts, max_rows, cfg.expert_offset)
    return moe_forward(cfg, x, weights, torch.from_numpy(w), torch.from_numpy(ids), nthreads=nthreads)


def moe_forward(cfg, x, weights, topk_weights, ids, renormalize: bool = False,
                rows=None, nthreads: int = 0):
    """Oracle forward.  Returns (acc fp32 [n, H] before the cast, out uint16
    bits [n, H]) for the tokens in ``rows`` (all tokens when None)."""
    xb = _np(x, np.uint16)
    T = xb.shape[0]
    w13 = _np(weights.w13, np.uint8)
    s13 = _np(weights.s13, np.uint16)
    w2 = _np(weights.w2, np.uint8)
    s2 = _np(weights.s2, np.uint16)
    tw = _np(topk_weights, np.float32)
    ids_np = _np(ids, np.int32)
    if rows is None:
        n = T
        rows_np = None
    else:
        rows_np = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        n = rows_np.size
    acc = np.zeros((n, cfg.hidden), np.float32)
    out = np.zeros((n, cfg.hidden), np.uint16)
    d = desc_array(cfg)
    rc = lib().oracle_moe_forward(_ptr(d), T, _ptr(xb), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2),
                                  _ptr(tw), _ptr(ids_np), int(bool(renormalize)),
                                  _ptr(rows_np) if rows_np is not None else None, n,
                                  _ptr(acc), _ptr(out), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_moe_forward failed: {rc}")
    return acc, out
