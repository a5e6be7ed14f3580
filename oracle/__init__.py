"""CPU oracle for SFI decode attention (test infrastructure).

Thin numpy/ctypes wrappers over ``sfi_oracle.c``: the plain fp64, single-threaded
restatement of what the method computes. Only the tests, the smoke check and the
benchmark's CPU-baseline leg import this package. It never imports the CUDA
library's package, and the CUDA library never imports it.

Functions take one request at a time (the oracle's own loop over requests lives
in the callers) and follow the Slow-Fast Inference paper's Figure 2 and Figure 3
captions; see ``sfi_oracle.c`` for the definitions and readings.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force on tiny inputs).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sfi_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_sfi.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle into liboracle_sfi.so next to its source (gcc, portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load(path: str):
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    Dd = ctypes.c_double
    L.oracle_dense_attn.argtypes = [P, P, P, P, I, I, I, I, I, Dd, P, P]
    L.oracle_index_attn.argtypes = [P, P, P, P, P, I, I, I, I, I, Dd, P, P]
    L.oracle_group_scores.argtypes = [P, P, P, I, I, I, I, I, I, I, Dd, P, ctypes.c_long]
    L.oracle_select_topk.argtypes = [P, I, I, I, I, P]
    L.oracle_select_topk.restype = I
    L.oracle_compact.argtypes = [P, P, P, I, I, P, I, I, I, I, I, P, P, I]
    L.oracle_fast_attn.argtypes = [P, P, P, I, I, P, P, P, I, I, I, I, I, I, I, Dd, P, P]
    L.oracle_split_merge_attn.argtypes = [P, I, P, P, P, P, I, I, I, I, Dd, P, P]
    L.oracle_paged_append.argtypes = [P, P, P, I, P, P, I, I, I]
    L.oracle_schedule.argtypes = [P, I, I, I, P]
    L.oracle_verify_attn.argtypes = [P, P, P, P, I, I, I, I, I, I, Dd, P, P]
    L.oracle_fast_multi_attn.argtypes = [P, P, P, I, I, P, P, P, I, I, I, I, I, I, I, I, Dd, P, P]
    L.oracle_verify_scores.argtypes = [P, P, P, I, I, I, I, I, I, I, I, Dd, P, ctypes.c_long]
    L.oracle_paged_append_tokens.argtypes = [P, P, P, I, I, P, P, I, I, I]
    for f in (L.oracle_dense_attn, L.oracle_index_attn, L.oracle_group_scores, L.oracle_compact,
              L.oracle_fast_attn, L.oracle_split_merge_attn, L.oracle_paged_append, L.oracle_schedule,
              L.oracle_verify_attn, L.oracle_fast_multi_attn, L.oracle_verify_scores,
              L.oracle_paged_append_tokens):
        f.restype = None
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _load(_LIB)
    return _lib


def build_variant(source: str, out_dir: str, name: str = "variant") -> str:
    """Compile a modified copy of the oracle source (used by the mutation tests only)."""
    src = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(src, "w") as f:
        f.write(source)
    subprocess.check_call(["gcc", *CFLAGS, "-o", so, src, "-lm"])
    return so


def source() -> str:
    with open(_SRC) as f:
        return f.read()


@contextlib.contextmanager
def use_library(path: str):
    """Temporarily route every wrapper in this module to another build of the oracle."""
    global _lib
    lib()
    with _lock:
        saved, _lib = _lib, _load(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def dense_attn(q, k_pool, v_pool, page_row, L, Hq, Hkv, D, P, scale=0.0):
    """Dense attention of one request: q uint16 [Hq][D] -> (out f64 [Hq][D], lse f64 [Hq])."""
    q, k_pool, v_pool, page_row = _u16(q), _u16(k_pool), _u16(v_pool), _i32(page_row)
    out = np.zeros((Hq, D), np.float64)
    lse = np.zeros(Hq, np.float64)
    lib().oracle_dense_attn(_p(q), _p(k_pool), _p(v_pool), _p(page_row), int(L), Hq, Hkv, D, P, float(scale),
                            _p(out), _p(lse))
    return out, lse


def index_attn(q, k_pool, v_pool, page_row, positions, Hq, Hkv, D, P, scale=0.0):
    """Attention over explicit positions per KV head (positions int32 [Hkv][n])."""
    q, k_pool, v_pool, page_row = _u16(q), _u16(k_pool), _u16(v_pool), _i32(page_row)
    positions = _i32(positions).reshape(Hkv, -1)
    n = positions.shape[1]
    out = np.zeros((Hq, D), np.float64)
    lse = np.zeros(Hq, np.float64)
    lib().oracle_index_attn(_p(q), _p(k_pool), _p(v_pool), _p(page_row), _p(positions), n, Hq, Hkv, D, P,
                            float(scale), _p(out), _p(lse))
    return out, lse


def group_scores(q, k_pool, page_row, L, S, W, Hq, Hkv, D, P, scale=0.0, stride=None, fill=np.nan):
    """Masked GQA-group-summed logits: float32 [Hkv][stride]; entries >= L keep `fill`."""
    q, k_pool, page_row = _u16(q), _u16(k_pool), _i32(page_row)
    stride = int(L) if stride is None else int(stride)
    scores = np.full((Hkv, stride), fill, np.float32)
    lib().oracle_group_scores(_p(q), _p(k_pool), _p(page_row), int(L), int(S), int(W), Hq, Hkv, D, P, float(scale),
                              _p(scores), stride)
    return scores


def select_topk(score_row, L, S, W, k):
    """Selector for one (request, KV head): ascending int32 positions, length k_eff."""
    score_row = np.ascontiguousarray(score_row, dtype=np.float32)
    out = np.zeros(max(1, min(max(int(k), 0), int(L))), np.int32)
    keff = lib().oracle_select_topk(_p(score_row), int(L), int(S), int(W), int(k), _p(out))
    return out[:keff].copy()


def compact(k_pool, v_pool, page_row, L, S, idx, k_eff, Hkv, D, P, cap):
    """Compact K/V of one request: (ck, cv) uint16 [Hkv][cap][D]; rows not written stay 0."""
    k_pool, v_pool, page_row = _u16(k_pool), _u16(v_pool), _i32(page_row)
    idx = _i32(idx).reshape(Hkv, -1)
    ck = np.zeros((Hkv, cap, D), np.uint16)
    cv = np.zeros((Hkv, cap, D), np.uint16)
    lib().oracle_compact(_p(k_pool), _p(v_pool), _p(page_row), int(L), int(S), _p(idx), idx.shape[1], int(k_eff),
                         Hkv, D, P, _p(ck), _p(cv), int(cap))
    return ck, cv


def fast_attn(q, ck, cv, count, k_pool, v_pool, page_row, L, S, W, Hq, Hkv, D, P, scale=0.0):
    """Fast step of one request: compact rows [0, min(S,L)+count) then paged [max(S, L-W), L)."""
    q, ck, cv = _u16(q), _u16(ck), _u16(cv)
    k_pool, v_pool, page_row = _u16(k_pool), _u16(v_pool), _i32(page_row)
    cap = ck.shape[1]
    out = np.zeros((Hq, D), np.float64)
    lse = np.zeros(Hq, np.float64)
    lib().oracle_fast_attn(_p(q), _p(ck), _p(cv), cap, int(count), _p(k_pool), _p(v_pool), _p(page_row), int(L),
                           int(S), int(W), Hq, Hkv, D, P, float(scale), _p(out), _p(lse))
    return out, lse


def split_merge_attn(q_head, kv, k_pool, v_pool, page_row, bounds, Hkv, D, P, scale=0.0):
    """Split-KV dense attention of one query head with chunk bounds [0 = b0 < ... < bn = L]."""
    q_head, k_pool, v_pool, page_row = _u16(q_head), _u16(k_pool), _u16(v_pool), _i32(page_row)
    bounds = _i32(bounds)
    out = np.zeros(D, np.float64)
    lse = np.zeros(1, np.float64)
    lib().oracle_split_merge_attn(_p(q_head), int(kv), _p(k_pool), _p(v_pool), _p(page_row), _p(bounds),
                                  len(bounds) - 1, Hkv, D, P, float(scale), _p(out), _p(lse))
    return out, float(lse[0])


def paged_append(k_pool, v_pool, page_row, L, k_new, v_new, Hkv, D, P):
    """In-place append of one token (length L after the append) into uint16 pools."""
    assert k_pool.dtype == np.uint16 and k_pool.flags["C_CONTIGUOUS"]
    assert v_pool.dtype == np.uint16 and v_pool.flags["C_CONTIGUOUS"]
    page_row, k_new, v_new = _i32(page_row), _u16(k_new), _u16(v_new)
    lib().oracle_paged_append(_p(k_pool), _p(v_pool), _p(page_row), int(L), _p(k_new), _p(v_new), Hkv, D, P)


def schedule(boundary, interval):
    """Slow(1)/fast(0) modes [steps][batch] from boundary draws uint8 [steps][batch]."""
    boundary = np.ascontiguousarray(boundary, dtype=np.uint8)
    steps, batch = boundary.shape
    modes = np.zeros_like(boundary)
    lib().oracle_schedule(_p(boundary), steps, batch, int(interval), _p(modes))
    return modes


def verify_attn(q, k_pool, v_pool, page_row, L, T, Hq, Hkv, D, P, scale=0.0):
    """Causal attention of T drafted tokens: q uint16 [T][Hq][D] -> (out [T][Hq][D], lse [T][Hq])."""
    q, k_pool, v_pool, page_row = _u16(q), _u16(k_pool), _u16(v_pool), _i32(page_row)
    out = np.zeros((T, Hq, D), np.float64)
    lse = np.zeros((T, Hq), np.float64)
    lib().oracle_verify_attn(_p(q), _p(k_pool), _p(v_pool), _p(page_row), int(L), int(T), Hq, Hkv, D, P,
                             float(scale), _p(out), _p(lse))
    return out, lse


def fast_multi_attn(q, ck, cv, count, k_pool, v_pool, page_row, L, T, S, W, Hq, Hkv, D, P, scale=0.0):
    """T query tokens over the sparse state: q uint16 [T][Hq][D] -> (out [T][Hq][D], lse [T][Hq])."""
    q, ck, cv = _u16(q), _u16(ck), _u16(cv)
    k_pool, v_pool, page_row = _u16(k_pool), _u16(v_pool), _i32(page_row)
    cap = ck.shape[1]
    out = np.zeros((T, Hq, D), np.float64)
    lse = np.zeros((T, Hq), np.float64)
    lib().oracle_fast_multi_attn(_p(q), _p(ck), _p(cv), cap, int(count), _p(k_pool), _p(v_pool), _p(page_row),
                                 int(L), int(T), int(S), int(W), Hq, Hkv, D, P, float(scale), _p(out), _p(lse))
    return out, lse


def verify_scores(q, k_pool, page_row, L, T, S, W, Hq, Hkv, D, P, scale=0.0, stride=None, fill=np.nan):
    """Verification statistics: float32 [Hkv][stride] (group- and token-summed masked logits)."""
    q, k_pool, page_row = _u16(q), _u16(k_pool), _i32(page_row)
    stride = int(L) if stride is None else int(stride)
    scores = np.full((Hkv, stride), fill, np.float32)
    lib().oracle_verify_scores(_p(q), _p(k_pool), _p(page_row), int(L), int(T), int(S), int(W), Hq, Hkv, D, P,
                               float(scale), _p(scores), stride)
    return scores


def paged_append_tokens(k_pool, v_pool, page_row, L, T, k_new, v_new, Hkv, D, P):
    """In-place append of T tokens (positions L - T .. L - 1) into uint16 pools; k_new [T][Hkv][D]."""
    assert k_pool.dtype == np.uint16 and k_pool.flags["C_CONTIGUOUS"]
    assert v_pool.dtype == np.uint16 and v_pool.flags["C_CONTIGUOUS"]
    page_row, k_new, v_new = _i32(page_row), _u16(k_new), _u16(v_new)
    lib().oracle_paged_append_tokens(_p(k_pool), _p(v_pool), _p(page_row), int(L), int(T), _p(k_new), _p(v_new),
                                     Hkv, D, P)
