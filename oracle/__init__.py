"""fp64 CPU oracle for softmax attention and paged-KV decode (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may
import this package.  The CUDA path never does, and this package never imports
the CUDA path: the two share nothing but the seeded input generators in
``synth``.

The arithmetic lives in ``oracle.c`` (plain C, OpenMP over rows); this module
only builds and loads it and marshals numpy arrays.  Inputs are bf16 bit
patterns (``uint16``), outputs are float64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (-O2, OpenMP)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; returns the ctypes handle."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    LL = ctypes.c_longlong
    Dbl = ctypes.c_double
    lib.oracle_attn_rows.argtypes = [P, P, P, I, I, I, I, I, I, I, Dbl, LL, P, P, P, P]
    lib.oracle_attn_rows.restype = I
    lib.oracle_attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, Dbl]
    lib.oracle_attn_fwd.restype = I
    lib.oracle_paged_gather.argtypes = [P, P, P, I, I, I, I, I, I, I, P]
    lib.oracle_paged_gather.restype = I
    lib.oracle_paged_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, Dbl, P, P]
    lib.oracle_paged_decode.restype = I
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = I
    return lib


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def attn_fwd(q, k, v, causal: bool, scale: float, lib=None):
    """O [B,Hq,Tq,D] float64 and LSE [B,Hq,Tq] float64 for bf16-bit inputs.

    q [B,Hq,Tq,D], k/v [B,Hkv,Tk,D].  With causal and Tq != Tk the mask is
    aligned bottom-right (query i sees keys j <= i + Tk - Tq).
    """
    lib = lib or load()
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, Tq, D = q.shape
    _, Hkv, Tk, _ = k.shape
    o = np.zeros((B, Hq, Tq, D), dtype=np.float64)
    lse = np.zeros((B, Hq, Tq), dtype=np.float64)
    st = lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Tq, Tk,
                             D, int(bool(causal)), float(scale))
    if st:
        raise OracleError(f"oracle_attn_fwd returned {st}")
    return o, lse


def attn_rows(q, k, v, causal: bool, scale: float, rows, want_probs: bool = False, lib=None):
    """Selected rows only.  ``rows`` are flat indices ((b*Hq)+h)*Tq+i.

    Returns (O [n, D], LSE [n]) or (O, LSE, P [n, Tk]) with ``want_probs``.
    """
    lib = lib or load()
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, Tq, D = q.shape
    _, Hkv, Tk, _ = k.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = len(rows)
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    p = np.zeros((n, Tk), dtype=np.float64) if want_probs else None
    st = lib.oracle_attn_rows(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Tq, Tk, D,
                              int(bool(causal)), float(scale), n, _ptr(rows), _ptr(o), _ptr(lse),
                              _ptr(p) if p is not None else None)
    if st:
        raise OracleError(f"oracle_attn_rows returned {st}")
    return (o, lse, p) if want_probs else (o, lse)


def paged_gather(pool, block_table, seq_lens, r: int, kvh: int, lib=None):
    """Contiguous [L, D] bf16 bits of request r, kv head kvh, read via the block table."""
    lib = lib or load()
    pool = _u16(pool)
    NB, Hkv, bs, D = pool.shape
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    L = int(sl[r])
    out = np.zeros((max(L, 0), D), dtype=np.uint16)
    st = lib.oracle_paged_gather(_ptr(pool), _ptr(bt), _ptr(sl), r, kvh, Hkv, bs, D, bt.shape[1],
                                 NB, _ptr(out))
    if st:
        raise OracleError(f"oracle_paged_gather returned {st}")
    return out


def paged_decode(q, k_pool, v_pool, block_table, seq_lens, scale: float, lib=None):
    """O [S,Hq,D] float64 and LSE [S,Hq] float64 of single-token paged decode."""
    lib = lib or load()
    q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape:
        raise ValueError("pool shape mismatch")
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    o = np.zeros((S, Hq, D), dtype=np.float64)
    lse = np.zeros((S, Hq), dtype=np.float64)
    st = lib.oracle_paged_decode(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(bt), _ptr(sl), S, Hq,
                                 Hkv, D, bs, bt.shape[1], NB, float(scale), _ptr(o), _ptr(lse))
    if st:
        raise OracleError(f"oracle_paged_decode returned {st}")
    return o, lse


def paged_prefill(q, k_pool, v_pool, block_table, kv_lens, causal: bool, scale: float, lib=None):
    """O [B,Hq,Tq,D] float64 and LSE [B,Hq,Tq] of a chunk of Tq queries per batch item
    against that item's paged cache of kv_lens[b] tokens (the chunk being its newest
    tokens).  Composes the oracle's block-table gather with its attention: each
    item's K/V history is gathered through the table, then attended to with
    Tq != Tk (bottom-right causal alignment)."""
    lib = lib or load()
    q = _u16(q)
    B, Hq, Tq, D = q.shape
    NB, Hkv, bs, D2 = k_pool.shape
    kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    o = np.zeros((B, Hq, Tq, D), dtype=np.float64)
    lse = np.zeros((B, Hq, Tq), dtype=np.float64)
    for b in range(B):
        kc = np.stack([paged_gather(k_pool, block_table, kl, b, h, lib=lib) for h in range(Hkv)])
        vc = np.stack([paged_gather(v_pool, block_table, kl, b, h, lib=lib) for h in range(Hkv)])
        ob, lb = attn_fwd(q[b:b + 1], kc[None], vc[None], causal, scale, lib=lib)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


def num_threads(lib=None) -> int:
    lib = lib or load()
    return int(lib.oracle_num_threads())
