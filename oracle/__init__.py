"""CPU fp64 oracle for MLA attention over a paged latent KV cache.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python binding)
never imports, links or calls anything here; only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg do.  The arithmetic lives in ``mla_oracle.c``
(plain C, IEEE double, straight loops); this module only compiles it with gcc and
marshals arguments.

What the oracle computes, with the passages it follows, is stated in the header of
``mla_oracle.c``.  Every function is pinned by ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile mla_oracle.c into liboracle.so next to it (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
               "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_mla_decode.restype = ctypes.c_int
            lib.oracle_mla_decode.argtypes = [i32, i32, i32, i32, i32, i32, P, P, i32, dbl, P, i64,
                                              P, i32, P, dbl, i32, P, i64, P, P]
            lib.oracle_mla_prefill.restype = ctypes.c_int
            lib.oracle_mla_prefill.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, dbl, P, i64, P, P]
            lib.oracle_e4m3_to_double.restype = ctypes.c_double
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> contiguous uint16 array of its bit patterns (no arithmetic)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(t) -> np.ndarray:
    return np.ascontiguousarray(torch.as_tensor(t).cpu().numpy().astype(np.int32))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def e4m3_to_double(codes) -> np.ndarray:
    """Decode e4m3fn byte codes with the oracle's own table (format definition)."""
    lib = _load()
    codes = np.asarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([lib.oracle_e4m3_to_double(int(c)) for c in codes], dtype=np.float64)


def mla_decode(q: torch.Tensor, kv_pool: torch.Tensor, page_table, seq_lens, scale: float,
               kv_scale: float = 1.0, dv: int = 512, rows=None, lens_include_drafts: bool = True,
               page_scales=None):
    """Absorbed MLA decode over a paged latent cache, in fp64.

    q: [B, T, H, D] bf16.  kv_pool: [n_pages, page_size, D] bf16, uint8 e4m3 codes or
    int8 codes (then each element is decoded and multiplied by kv_scale, or, for int8 codes
    with ``page_scales`` [n_pages], by the scale of the page that holds it).  page_table:
    [B, max_pages] int32.  seq_lens: [B] (tokens cached per request, drafts included).
    Returns (out [B,T,H,dv] float64, lse [B,T,H] float64) or, with ``rows`` (flat ids
    (b*T + t)*H + h), (out [n, dv], lse [n]).
    """
    lib = _load()
    B, T, H, D = q.shape
    n_pages, page_size, D2 = kv_pool.shape
    assert D2 == D
    if kv_pool.dtype == torch.bfloat16:
        pool = _bits16(kv_pool)
        kv_dtype = 0
    elif kv_pool.dtype == torch.uint8:
        pool = np.ascontiguousarray(kv_pool.cpu().numpy())
        kv_dtype = 1
    elif kv_pool.dtype == torch.int8:
        pool = np.ascontiguousarray(kv_pool.cpu().numpy())
        kv_dtype = 2
    else:
        raise TypeError("kv_pool must be bf16, uint8 e4m3 codes or int8 codes")
    ps = None
    if page_scales is not None:
        if kv_dtype != 2:
            raise TypeError("page_scales apply to int8 pools only")
        ps = np.ascontiguousarray(torch.as_tensor(page_scales).detach().cpu().double().numpy().reshape(-1))
        if ps.size != n_pages:
            raise ValueError("page_scales must hold one scale per page")
    qb = _bits16(q)
    pt = _i32(page_table)
    sl = _i32(seq_lens)
    max_pages = pt.shape[1]
    if rows is None:
        rows_arr, n_rows = None, B * T * H
        out = np.zeros((B, T, H, dv), dtype=np.float64)
        lse = np.zeros((B, T, H), dtype=np.float64)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n_rows = rows_arr.size
        out = np.zeros((n_rows, dv), dtype=np.float64)
        lse = np.zeros((n_rows,), dtype=np.float64)
    rc = lib.oracle_mla_decode(B, T, H, D, dv, page_size, _ptr(qb), _ptr(pool), kv_dtype,
                               float(kv_scale), _ptr(ps) if ps is not None else None, n_pages, _ptr(pt),
                               max_pages, _ptr(sl), float(scale),
                               1 if lens_include_drafts else 0,
                               _ptr(rows_arr) if rows_arr is not None else None, n_rows,
                               _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_mla_decode rejected its arguments")
    return out, lse


def mla_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q, cu_seqlens_kv,
                prefix_lens, scale: float, rows=None):
    """Ragged causal prefill with a cached prefix, in fp64.

    q: [Nq, H, Dqk] bf16, k: [Nkv, H, Dqk] bf16, v: [Nkv, H, Dv] bf16,
    cu_seqlens_q / cu_seqlens_kv: [B+1] int32, prefix_lens: [B] int32.
    Returns (out [Nq, H, Dv] float64, lse [Nq, H] float64), or per-row arrays with ``rows``
    (flat ids token*H + h).
    """
    lib = _load()
    Nq, H, Dqk = q.shape
    Dv = v.shape[2]
    cq, ck, pl = _i32(cu_seqlens_q), _i32(cu_seqlens_kv), _i32(prefix_lens)
    B = pl.shape[0]
    qb, kb, vb = _bits16(q), _bits16(k), _bits16(v)
    if rows is None:
        rows_arr, n_rows = None, Nq * H
        out = np.zeros((Nq, H, Dv), dtype=np.float64)
        lse = np.zeros((Nq, H), dtype=np.float64)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n_rows = rows_arr.size
        out = np.zeros((n_rows, Dv), dtype=np.float64)
        lse = np.zeros((n_rows,), dtype=np.float64)
    rc = lib.oracle_mla_prefill(B, H, Dqk, Dv, _ptr(cq), _ptr(ck), _ptr(pl), _ptr(qb), _ptr(kb),
                                _ptr(vb), float(scale),
                                _ptr(rows_arr) if rows_arr is not None else None, n_rows,
                                _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_mla_prefill rejected its arguments")
    return out, lse
