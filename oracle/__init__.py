"""Python face of the float64 CPU oracle (``mla_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()`` and by
the benchmark's CPU-baseline leg. The library under test never imports it, and it
imports nothing from the library.

``build()`` compiles ``mla_oracle.c`` with gcc (OpenMP) into ``liboracle.so`` next to
this file; the functions below marshal numpy/torch CPU arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib: Optional[ctypes.CDLL] = None

DV = 512


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, OpenMP). Returns its path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "mla_oracle.h"))):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", _LIB_PATH, _SRC,
               "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        _lib = bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def use_library(lib: Optional[ctypes.CDLL]) -> Optional[ctypes.CDLL]:
    """Swap the shared library behind the functions below (the tests use this to run
    the pins against deliberately broken builds of the oracle). Returns the old one."""
    global _lib
    old = _lib
    _lib = lib
    return old


def bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare argument and result types of an oracle shared library."""
    P = ctypes.c_void_p
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = dbl
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_value.restype = dbl
    lib.oracle_attention.argtypes = [P, i64, i32, P, i64, P, dbl, P, i32, i32, i32, dbl, P, P,
                                     i32]
    lib.oracle_attention.restype = i32
    lib.oracle_attention_rows.argtypes = [P, i64, i32, P, i64, P, dbl, P, i32, i32, i32, dbl,
                                          P, P, P, i64, P, P, i32]
    lib.oracle_attention_rows.restype = i32
    lib.oracle_attention_range.argtypes = [P, i64, i32, P, i64, i32, i64, i64, dbl, P, dbl, P,
                                           P]
    lib.oracle_attention_range.restype = i32
    lib.oracle_merge_lse.argtypes = [P, P, i32, i64, P, P]
    lib.oracle_merge_lse.restype = None
    lib.oracle_e4m3_encode.argtypes = [dbl]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_cache_append.argtypes = [P, i64, P, P, i64, ctypes.c_float]
    lib.oracle_cache_append.restype = i32
    return lib


def _np(t, dtype) -> np.ndarray:
    """Contiguous numpy array of a CPU torch tensor (or array) holding `dtype` bits.
    bfloat16 tensors are passed through as their raw uint16 bit patterns."""
    if hasattr(t, "detach"):
        t = t.detach().cpu().contiguous()
        if str(t.dtype) == "torch.bfloat16":
            import torch
            t = t.view(torch.int16)
        t = t.numpy()
    a = np.ascontiguousarray(t)
    if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu":
        return a.view(dtype)
    return np.ascontiguousarray(a.astype(dtype))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(code)


def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(bits)


def _kv_args(inp):
    pool = _np(inp.pool, np.uint8)
    pt = _np(inp.page_table, np.int32)
    sl = _np(inp.seq_lens, np.int32)
    q = _np(inp.q, np.uint16)
    return pool, pt, sl, q


def attention(inp, n_threads: int = 0):
    """Full float64 attention for every (b, j, h) of a workload.
    Returns (out [B, n_q, H, 512] float64, lse [B, n_q, H] float64)."""
    lib = _load()
    pool, pt, sl, q = _kv_args(inp)
    B, n_q, H = q.shape[0], q.shape[1], q.shape[2]
    out = np.empty((B, n_q, H, DV), dtype=np.float64)
    lse = np.empty((B, n_q, H), dtype=np.float64)
    rc = lib.oracle_attention(_ptr(pool), pool.shape[0], pool.shape[1], _ptr(pt), pt.shape[1],
                              _ptr(sl), float(inp.kv_scale), _ptr(q), B, n_q, H,
                              float(inp.sm_scale), _ptr(out), _ptr(lse), n_threads)
    if rc != 0:
        raise ValueError("oracle_attention: bad argument (page index or length)")
    return out, lse


def attention_rows(inp, rows, n_threads: int = 0):
    """Attention for the listed rows only; rows is an int array [n, 3] of (b, j, h).
    Returns (out [n, 512], lse [n])."""
    lib = _load()
    pool, pt, sl, q = _kv_args(inp)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    rb = np.ascontiguousarray(rows[:, 0])
    rj = np.ascontiguousarray(rows[:, 1])
    rh = np.ascontiguousarray(rows[:, 2])
    n = rows.shape[0]
    out = np.empty((n, DV), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = lib.oracle_attention_rows(_ptr(pool), pool.shape[0], pool.shape[1], _ptr(pt), pt.shape[1],
                                   _ptr(sl), float(inp.kv_scale), _ptr(q), q.shape[0], q.shape[1],
                                   q.shape[2], float(inp.sm_scale), _ptr(rb), _ptr(rj), _ptr(rh),
                                   n, _ptr(out), _ptr(lse), n_threads)
    if rc != 0:
        raise ValueError("oracle_attention_rows: bad argument (page index or length)")
    return out, lse


def attention_range(inp, b: int, j: int, h: int, key_lo: int, key_hi: int):
    """Partial attention of query row (b, j, h) over keys [key_lo, key_hi) only."""
    lib = _load()
    pool, pt, sl, q = _kv_args(inp)
    qrow = np.ascontiguousarray(q[b, j, h])
    out = np.empty((DV,), dtype=np.float64)
    lse = np.empty((1,), dtype=np.float64)
    rc = lib.oracle_attention_range(_ptr(pool), pool.shape[0], pool.shape[1], _ptr(pt),
                                    pt.shape[1], b, key_lo, key_hi, float(inp.kv_scale),
                                    _ptr(qrow), float(inp.sm_scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attention_range: bad page index")
    return out, float(lse[0])


def merge_lse(part_out, part_lse):
    """part_out [S, R, 512], part_lse [S, R] -> (out [R, 512], lse [R]) in float64."""
    lib = _load()
    po = np.ascontiguousarray(np.asarray(part_out, dtype=np.float64))
    pl = np.ascontiguousarray(np.asarray(part_lse, dtype=np.float64))
    S, R = pl.shape
    out = np.empty((R, DV), dtype=np.float64)
    lse = np.empty((R,), dtype=np.float64)
    lib.oracle_merge_lse(_ptr(po), _ptr(pl), S, R, _ptr(out), _ptr(lse))
    return out, lse


def e4m3_encode(v: float) -> int:
    """e4m3fn code nearest to v (ties to even, saturating at +-448)."""
    return int(_load().oracle_e4m3_encode(float(v)))


def cache_append(pool, x, slots, kv_scale: float):
    """Append bf16 rows x [n, 576] to a copy of the paged pool (uint8 [num_pages, page_size,
    576] or [rows, 576]) at flat row slots [n] (negative: skipped). Returns the new pool
    (numpy uint8, same shape); raises if a slot is past the pool."""
    lib = _load()
    pool_np = _np(pool, np.uint8).copy()
    xs = _np(x, np.uint16)
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
    rows = pool_np.size // 576
    rc = lib.oracle_cache_append(_ptr(pool_np), rows, _ptr(xs), _ptr(sl), sl.shape[0],
                                 float(kv_scale))
    if rc != 0:
        raise ValueError("oracle_cache_append: slot past the end of the pool")
    return pool_np


def top_k_renorm_prob(probs, top_k):
    """Row-wise top-k renormalisation in float64, straight from the definition: the pivot is
    the k-th largest entry (a sort), every entry >= pivot is kept, the kept entries are
    divided by their sum; k <= 0 or k >= V keeps the row. probs [B, V]; top_k int or [B]."""
    p = np.asarray(probs, dtype=np.float64)
    B, V = p.shape
    ks = np.broadcast_to(np.asarray(top_k, dtype=np.int64), (B,))
    out = np.zeros_like(p)
    for r in range(B):
        k = int(ks[r])
        if k <= 0 or k >= V:
            keep = np.ones(V, dtype=bool)
        else:
            pivot = np.sort(p[r])[V - k]
            keep = p[r] >= pivot
        out[r, keep] = p[r, keep] / p[r, keep].sum()
    return out


def _cache_rows(cache, L: int) -> np.ndarray:
    """Dequantised rows 0..L-1 of sequence 0 of an MlaInputs cache, float64 [L][576]."""
    table = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64) * float(cache.kv_scale)
    pool = _np(cache.pool, np.uint8)
    pt = _np(cache.page_table, np.int32)
    P = pool.shape[1]
    n = np.arange(L)
    pages = pt[0, n // P]
    if (pages < 0).any() or (pages >= pool.shape[0]).any():
        raise ValueError("page index outside the pool")
    return table[pool[pages, n % P]]


def _f64(t) -> np.ndarray:
    if hasattr(t, "detach"):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def mha_prefill_rows(cache, q, w_ukv, rows=None):
    """MHA-form causal prefill of one sequence in float64, from the definition: for head h
    the key of position n is [c_n W_UK_h ; r_n] (c_n the 512-wide latent, r_n the 64 RoPE
    dims, both dequantised), its value c_n W_UV_h; new position t (of T, the last T of the
    L cached) sees keys n <= L - T + t; scores are scaled by sm_scale.
    q [T][H][192], w_ukv [512][H][256] (W_UK_h = columns 0..127, W_UV_h = 128..255).
    rows: None for every (t, h), else an int array [n, 2] of (t, h).
    Returns (out [T][H][128] or [n][128], lse [T][H] or [n])."""
    qf = _f64(q)
    W = _f64(w_ukv)
    T, H = qf.shape[0], qf.shape[1]
    L = int(_np(cache.seq_lens, np.int32)[0])
    if L < T:
        raise ValueError("the sequence must hold its T new positions")
    kv = _cache_rows(cache, L)
    c, r = kv[:, :DV], kv[:, DV:]
    sel = np.array([(t, h) for t in range(T) for h in range(H)]) if rows is None else \
        np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    out = np.zeros((sel.shape[0], 128))
    lse = np.full((sel.shape[0],), -np.inf)
    for h in np.unique(sel[:, 1]):
        K = np.concatenate([c @ W[:, h, :128], r], axis=1)   # [L][192]
        V = c @ W[:, h, 128:]                                # [L][128]
        idx = np.nonzero(sel[:, 1] == h)[0]
        ts = sel[idx, 0]
        s = float(cache.sm_scale) * (qf[ts, h, :] @ K.T)     # [n][L]
        visible = np.arange(L)[None, :] <= (L - T + ts)[:, None]
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        out[idx] = (p @ V) / l
        lse[idx] = (m + np.log(l))[:, 0]
    if rows is None:
        return out.reshape(T, H, 128), lse.reshape(T, H)
    return out, lse
