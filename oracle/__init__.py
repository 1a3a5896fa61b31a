"""CPU fp64 oracle for paged KV append and mixed-batch attention.

TEST INFRASTRUCTURE ONLY: imported by the test suite, by ``smoke()`` and by the
benchmark's CPU-baseline leg, never by the product package.  It shares no code
with the CUDA library.  The arithmetic lives in ``oracle.c`` (plain loops, fp64,
OpenMP over (query row, head)); ``dense.py`` is an independent NumPy brute
force used to pin it on tiny inputs.  This module only marshals arrays.

Pinned by tests/test_oracle.py (see the header of ``oracle.c`` for the page
citations).  Parity is pinned for every function here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OR_OK, OR_ERR_ARG, OR_ERR_SHAPE, OR_ERR_PAGE = 0, -1, -2, -3


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP, strict fp)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_num_threads.restype = i32
        lib.oracle_kv_append.restype = i32
        lib.oracle_kv_append.argtypes = [P, i64, P, P, P, P, P, P, i32, i32, i32, i32]
        lib.oracle_attention.restype = i32
        lib.oracle_attention.argtypes = [P, P, i64, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                         P, i32, dbl, P, i64, P, P, P]
        lib.oracle_attention_keyrange.restype = i32
        lib.oracle_attention_keyrange.argtypes = [P, P, i64, P, P, P, P, i32, i32, i32, i32, i32,
                                                  dbl, i64, i32, i64, i64, P, P, P]
        lib.oracle_softmax_merge.restype = None
        lib.oracle_softmax_merge.argtypes = [P, P, i32, i32, P, P]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _u16(a):
    """bf16 data as uint16 bit patterns (numpy uint16 or torch bfloat16)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous().view(torch.int16).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a).view(np.uint16)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


class OracleError(RuntimeError):
    pass


def _check(st):
    if st != OR_OK:
        raise OracleError(f"oracle status {st}")


def new_pool(shape, sentinel: int) -> np.ndarray:
    """A page pool [num_pages, 2, Hkv, P, d] of bf16 bit patterns, all `sentinel`."""
    return np.full(shape, sentinel, dtype=np.uint16)


def kv_append(pool: np.ndarray, k_new, v_new, append_indptr, page_indices, kv_indptr,
              last_page_len) -> None:
    """Append in place (pool: uint16 [num_pages, 2, Hkv, P, d])."""
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous and pool.ndim == 5
    num_pages, two, Hkv, P, d = pool.shape
    k, v = _u16(k_new), _u16(v_new)
    ai, pi, ki, ll = _i32(append_indptr), _i32(page_indices), _i32(kv_indptr), _i32(last_page_len)
    batch = len(ai) - 1
    assert k.shape == v.shape and (k.size == 0 or k.shape[1:] == (Hkv, d))
    assert k.shape[0] == (ai[-1] if batch > 0 else 0)
    _check(_load().oracle_kv_append(_ptr(pool), num_pages, _ptr(k), _ptr(v), _ptr(ai), _ptr(pi),
                                    _ptr(ki), _ptr(ll), batch, Hkv, d, P))


def attention(q, pool: np.ndarray, qo_indptr, kv_indptr, page_indices, last_page_len,
              causal: bool, sm_scale: float, num_qo_heads: int, sel_rows=None, tree_mask=None):
    """Returns (out fp64 [rows, Hq, d], lse fp64 [rows, Hq], attended pairs).
    tree_mask: optional uint32 [nnz_qo, words] draft-tree mask rows."""
    num_pages, _, Hkv, P, d = pool.shape
    qq = _u16(q)
    qi, ki, pi, ll = _i32(qo_indptr), _i32(kv_indptr), _i32(page_indices), _i32(last_page_len)
    batch = len(qi) - 1
    nnz = int(qi[-1]) if batch > 0 else 0
    sel = None if sel_rows is None else np.ascontiguousarray(np.asarray(sel_rows, np.int64))
    rows = nnz if sel is None else len(sel)
    out = np.zeros((rows, num_qo_heads, d), np.float64)
    lse = np.zeros((rows, num_qo_heads), np.float64)
    pairs = ctypes.c_int64(0)
    tm = None
    if tree_mask is not None:
        tm = np.ascontiguousarray(np.asarray(tree_mask, np.uint32))
        assert tm.ndim == 2 and tm.shape[0] == nnz
    _check(_load().oracle_attention(_ptr(qq), _ptr(pool), num_pages, _ptr(qi), _ptr(ki), _ptr(pi),
                                    _ptr(ll), batch, num_qo_heads, Hkv, d, P, int(bool(causal)),
                                    _ptr(tm), 0 if tm is None else tm.shape[1],
                                    float(sm_scale), _ptr(sel), 0 if sel is None else len(sel),
                                    _ptr(out), _ptr(lse), ctypes.addressof(pairs)))
    return out, lse, int(pairs.value)


def attention_keyrange(q, pool, qo_indptr, kv_indptr, page_indices, last_page_len,
                       sm_scale, num_qo_heads, row, head, lo, hi, want_weights=False):
    """One (row, head) over keys [lo, hi) of its request: (o [d], lse, w or None)."""
    num_pages, _, Hkv, P, d = pool.shape
    qq = _u16(q)
    qi, ki, pi, ll = _i32(qo_indptr), _i32(kv_indptr), _i32(page_indices), _i32(last_page_len)
    o = np.zeros(d, np.float64)
    lse = np.zeros(1, np.float64)
    w = np.zeros(max(hi - lo, 1), np.float64) if want_weights else None
    _check(_load().oracle_attention_keyrange(_ptr(qq), _ptr(pool), num_pages, _ptr(qi), _ptr(ki),
                                             _ptr(pi), _ptr(ll), len(qi) - 1, num_qo_heads, Hkv,
                                             d, P, float(sm_scale), row, head, lo, hi, _ptr(o),
                                             _ptr(lse), _ptr(w)))
    return o, float(lse[0]), (None if w is None else w[:hi - lo])


def softmax_merge(parts_o, parts_lse):
    """Merge n partial attentions: parts_o [n, d], parts_lse [n] -> (o [d], lse)."""
    po = np.ascontiguousarray(np.asarray(parts_o, np.float64))
    pl = np.ascontiguousarray(np.asarray(parts_lse, np.float64))
    n, d = po.shape
    o = np.zeros(d, np.float64)
    lse = np.zeros(1, np.float64)
    _load().oracle_softmax_merge(_ptr(po), _ptr(pl), n, d, _ptr(o), _ptr(lse))
    return o, float(lse[0])
