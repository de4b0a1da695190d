"""Loader for the C fp64 oracle (``pa_oracle.c``) and its build step.

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
baseline of the benchmark.  The product path never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")

_DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available).  Returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        L.oracle_block_layout.argtypes = [i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.oracle_block_layout.restype = i32
        L.oracle_locate.argtypes = [vp, i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.oracle_locate.restype = i32
        L.oracle_slot.argtypes = [vp, i64, i64, i64, ctypes.POINTER(i64)]
        L.oracle_slot.restype = i32
        L.oracle_write_kv.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32]
        L.oracle_write_kv.restype = i32
        L.oracle_copy_blocks.argtypes = [vp, vp, vp, i64, i32, i32, i32, i64, i32]
        L.oracle_copy_blocks.restype = i32
        L.oracle_decode.argtypes = [vp, vp, vp, vp, vp, i64, vp, i32, i32, i32, i32, i32, i64,
                                    dbl, i32, i32]
        L.oracle_decode.restype = i32
        L.oracle_prefill.argtypes = [vp, vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, i32, i64,
                                     dbl, i32, i32]
        L.oracle_prefill.restype = i32
        L.oracle_max_threads.argtypes = []
        L.oracle_max_threads.restype = i32
        _lib = L
    return _lib


def _cpu(t: torch.Tensor) -> torch.Tensor:
    t = t.detach()
    if t.device.type != "cpu" or not t.is_contiguous():
        t = t.to("cpu").contiguous()
    return t


def block_layout(tokens: int, block_size: int) -> tuple[int, int]:
    b, u = ctypes.c_int64(), ctypes.c_int64()
    if lib().oracle_block_layout(tokens, block_size, ctypes.byref(b), ctypes.byref(u)):
        raise ValueError("invalid size")
    return b.value, u.value


def locate(table_row, t: int, block_size: int) -> tuple[int, int]:
    row = np.ascontiguousarray(np.asarray(table_row, dtype=np.int32))
    p, o = ctypes.c_int64(), ctypes.c_int64()
    if lib().oracle_locate(row.ctypes.data, row.size, t, block_size, ctypes.byref(p), ctypes.byref(o)):
        raise IndexError("invalid position")
    return p.value, o.value


def slot_mapping(block_tables, token_seq, token_pos, block_size: int) -> np.ndarray:
    tables = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    out = np.empty(len(token_seq), dtype=np.int64)
    s_ = ctypes.c_int64()
    for i, (s, t) in enumerate(zip(np.asarray(token_seq).tolist(), np.asarray(token_pos).tolist())):
        row = tables[s]
        if lib().oracle_slot(row.ctypes.data, row.size, t, block_size, ctypes.byref(s_)):
            raise IndexError("invalid position")
        out[i] = s_.value
    return out


def write_kv(key, value, k_cache, v_cache, slots) -> None:
    """In place on CPU contiguous pools."""
    assert k_cache.device.type == "cpu" and k_cache.is_contiguous() and v_cache.is_contiguous()
    key, value = _cpu(key), _cpu(value)
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
    NB, Hkv, B, D = k_cache.shape
    rc = lib().oracle_write_kv(key.data_ptr(), value.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                               sl.ctypes.data, sl.size, Hkv, D, B, NB, _DTYPE_CODE[k_cache.dtype])
    if rc:
        raise IndexError("slot outside the pool")


def copy_blocks(k_cache, v_cache, pairs) -> None:
    assert k_cache.device.type == "cpu" and k_cache.is_contiguous() and v_cache.is_contiguous()
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    NB, Hkv, B, D = k_cache.shape
    rc = lib().oracle_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), pr.ctypes.data, pr.shape[0],
                                  Hkv, D, B, NB, _DTYPE_CODE[k_cache.dtype])
    if rc:
        raise IndexError("block id outside the pool")


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, nthreads: int = 0) -> np.ndarray:
    """float64 [S][Hq][D] (see ``pa_oracle.c``)."""
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    S, Hq, D = q.shape
    NB, Hkv, B, _ = k_cache.shape
    tables = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = lib().oracle_decode(out.ctypes.data, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                             tables.ctypes.data, tables.shape[1] if tables.ndim == 2 else 0,
                             lens.ctypes.data, S, Hq, Hkv, D, B, NB, float(scale),
                             _DTYPE_CODE[q.dtype], int(nthreads))
    if rc:
        raise ValueError("oracle_decode: invalid argument or index")
    return out


def prefill(q, k_cache, v_cache, block_tables, context_lens, q_start, scale: float,
            nthreads: int = 0) -> np.ndarray:
    """float64 [T][Hq][D] (see ``pa_oracle.c``, oracle_prefill)."""
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    T, Hq, D = q.shape
    NB, Hkv, B, _ = k_cache.shape
    tables = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    lens = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    qs = np.ascontiguousarray(np.asarray(q_start, dtype=np.int32))
    S = lens.size
    if qs.size != S + 1 or (S and int(qs[-1]) != T):
        raise ValueError("q_start must have num_seqs + 1 entries ending at the number of query rows")
    out = np.zeros((T, Hq, D), dtype=np.float64)
    rc = lib().oracle_prefill(out.ctypes.data, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                              tables.ctypes.data, tables.shape[1] if tables.ndim == 2 else 0, lens.ctypes.data,
                              qs.ctypes.data, S, Hq, Hkv, D, B, NB, float(scale), _DTYPE_CODE[q.dtype],
                              int(nthreads))
    if rc:
        raise ValueError("oracle_prefill: invalid argument or index")
    return out


def max_threads() -> int:
    return int(lib().oracle_max_threads())
