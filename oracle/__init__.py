"""Oracle for the DLRM sparse hot path: plain fp64 CPU definitions.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
import this package.  It shares no code with the CUDA library and imports
nothing from it.

The arithmetic lives in ``dlrm_oracle.c`` (plain loops, fp64, no fused
multiply-add); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  Every float result comes with a magnitude array (the
same computation on absolute values) that bounds the rounding error of any
summation order: a value x passes when ``|x - ref| <= rel * mag``.

Parity pins: every function here is pinned by tests that do not call it
again to check it (hand-worked examples, numpy matmul, the factorization-
machine identity, finite differences, brute force); see the test module
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dlrm_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_LIB_OMP = os.path.join(_HERE, "_build", "liboracle_omp.so")

F32, F16, BF16, INT4 = 0, 1, 2, 3
_DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16, "int4": INT4}

OK, INVALID_ARG, INDEX_OOB, BAD_OFFSETS, NO_MEMORY = 0, -1, -4, -5, -8

_lock = threading.Lock()
_lib = None
_variant = _LIB


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what} returned status {status}")
        self.status = status


def _compile(target, extra):
    tmp = target + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
                    "-Wno-unknown-pragmas"] + extra + ["-shared", "-fPIC", _SRC, "-o", tmp, "-lm"],
                   check=True, capture_output=True)
    os.replace(tmp, target)


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc into ``oracle/_build/liboracle.so``, and
    (best effort) its OpenMP build ``liboracle_omp.so``, used only to time the
    oracle on all host cores."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    for target, extra, required in ((_LIB, [], True), (_LIB_OMP, ["-fopenmp"], False)):
        if not force and os.path.exists(target) and os.path.getmtime(target) >= os.path.getmtime(_SRC):
            continue
        try:
            _compile(target, extra)
        except (subprocess.CalledProcessError, OSError):
            if required:
                raise
    return _LIB


def use_openmp(flag: bool) -> bool:
    """Switches the loaded library between the serial build (the parity
    oracle) and the OpenMP build (the same loops on all host cores; identical
    results).  Returns whether the requested build is in use."""
    global _lib, _variant
    want = _LIB_OMP if flag else _LIB
    build()
    if flag and not os.path.exists(_LIB_OMP):
        return False
    with _lock:
        if _variant != want:
            _lib = None
            _variant = want
    _load()
    return True


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_variant)
            i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
            lib.oracle_decode.argtypes = [i32, vp, i64, dp]
            lib.oracle_emb_bag_fwd.argtypes = [i32, i32, i32, vp, vp, i64, vp, vp, i64, dp, dp]
            lib.oracle_num_pairs.argtypes = [i32, i32]
            lib.oracle_num_pairs.restype = i64
            lib.oracle_interact_fwd.argtypes = [i32, i32, i64, i32, dp, dp, dp, dp, dp, dp]
            lib.oracle_interact_bwd.argtypes = [i32, i32, i64, i32, dp, dp, dp, dp, dp, dp,
                                                dp, dp, dp, dp]
            lib.oracle_coalesce.argtypes = [i32, i64, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp]
            lib.oracle_sgd.argtypes = [i32, i32, i32, vp, vp, i64, vp, i64, dp, dp,
                                       ctypes.c_double, vp, vp, vp, vp, i64, dp, dp, dp, dp]
            lib.oracle_quantize_int4.argtypes = [i64, i32, i32, vp, vp]
            lib.oracle_int4_row_bytes.argtypes = [i32]
            lib.oracle_int4_row_bytes.restype = i64
            lib.oracle_adagrad.argtypes = [i32, i32, i32, vp, vp, i64, vp, i64, dp, dp, ctypes.c_double,
                                           ctypes.c_double, vp, vp, vp, vp, i64, dp, dp, dp, dp, dp, dp, dp]
            for name in ("oracle_decode", "oracle_emb_bag_fwd", "oracle_interact_fwd",
                         "oracle_interact_bwd", "oracle_coalesce", "oracle_sgd", "oracle_adagrad",
                         "oracle_quantize_int4"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _i64(a):
    return np.ascontiguousarray(a, dtype=np.int64)


def _check(status: int, what: str):
    if status != OK:
        raise OracleError(status, what)


def _table_bits(table: np.ndarray, dtype: str) -> np.ndarray:
    """Storage of one table for the C side: float32, the 16-bit patterns, or
    the bytes of an int4 table ([rows][int4_row_bytes(d)] uint8)."""
    if dtype == "f32":
        return np.ascontiguousarray(table, dtype=np.float32)
    if dtype == "int4":
        return np.ascontiguousarray(table, dtype=np.uint8)
    if table.dtype == np.float16:
        return np.ascontiguousarray(table).view(np.uint16)
    return np.ascontiguousarray(table, dtype=np.uint16)


def decode(table: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 values of a table given in its storage type (bf16 as uint16 bits)."""
    bits = _table_bits(table, dtype)
    out = np.empty(bits.shape, dtype=np.float64)
    _check(_load().oracle_decode(_DTYPE_CODES[dtype], _ptr(bits), bits.size, _ptr(out)),
           "decode")
    return out


def num_pairs(N: int, include_self: bool) -> int:
    return int(_load().oracle_num_pairs(N, int(bool(include_self))))


def _tables_arg(tables, dtype):
    held = [_table_bits(t, dtype) for t in tables]
    arr = (ctypes.c_void_p * len(held))(*[h.ctypes.data for h in held])
    rows = np.array([h.shape[0] for h in held], dtype=np.int64)
    return held, arr, rows


def int4_row_bytes(d: int) -> int:
    """Bytes of one row of an int4 table: d/2 code bytes, fp32 scale and bias, padded to 16."""
    return int(_load().oracle_int4_row_bytes(d))


def quantize_int4(table: np.ndarray, dtype: str) -> np.ndarray:
    """Row-wise int4 encoding of a [rows][d] table: returns [rows][int4_row_bytes(d)] uint8."""
    bits = _table_bits(table, dtype)
    R, d = bits.shape
    out = np.zeros((R, int4_row_bytes(d)), dtype=np.uint8)
    _check(_load().oracle_quantize_int4(R, d, _DTYPE_CODES[dtype], _ptr(bits), _ptr(out)), "quantize_int4")
    return out


def emb_bag_fwd(tables, dtype: str, offsets, indices, B: int, d: int = None):
    """Sum-pooled lookups: returns (pooled [B][T][d], magnitude) in fp64.
    int4 tables (rows of bytes) need ``d``."""
    held, arr, rows = _tables_arg(tables, dtype)
    T = len(held)
    if d is None:
        d = held[0].shape[1]
    offsets, indices = _i64(offsets), _i64(indices)
    pooled = np.empty((B, T, d), dtype=np.float64)
    mag = np.empty_like(pooled)
    _check(_load().oracle_emb_bag_fwd(T, d, _DTYPE_CODES[dtype], arr, _ptr(rows), B,
                                      _ptr(offsets), _ptr(indices), indices.size,
                                      _ptr(pooled), _ptr(mag)), "emb_bag_fwd")
    return pooled, mag


def interact_fwd(e0, emb, include_self: bool, e0_mag=None, emb_mag=None, alongside: bool = False):
    """[e0 | pairwise dots] per sample, or [e0 | e_1 .. e_N | pairwise dots]
    with ``alongside``: returns (y [B][width], magnitude)."""
    e0, emb = _f64(e0), _f64(emb)
    B, N, d = emb.shape
    width = d * (N + 1 if alongside else 1) + num_pairs(N, include_self)
    y = np.empty((B, width), dtype=np.float64)
    ym = np.empty_like(y)
    _check(_load().oracle_interact_fwd(N, d, B, _mode(include_self, alongside), _ptr(e0),
                                       _ptr(_f64(e0_mag)), _ptr(emb), _ptr(_f64(emb_mag)),
                                       _ptr(y), _ptr(ym)), "interact_fwd")
    return y, ym


def _mode(include_self, alongside):
    return (1 if include_self else 0) | (2 if alongside else 0)


def interact_bwd(e0, emb, dy, include_self: bool, e0_mag=None, emb_mag=None, dy_mag=None,
                 alongside: bool = False):
    """Gradients of the interaction: returns (de0, de0_mag, demb, demb_mag)."""
    e0, emb, dy = _f64(e0), _f64(emb), _f64(dy)
    B, N, d = emb.shape
    width = d * (N + 1 if alongside else 1) + num_pairs(N, include_self)
    if dy.shape != (B, width) or e0.shape != (B, d):
        raise ValueError(f"interact_bwd: dy must be [{B}][{width}] and e0 [{B}][{d}]")
    de0 = np.empty((B, d), dtype=np.float64)
    de0m = np.empty_like(de0)
    demb = np.empty((B, N, d), dtype=np.float64)
    dembm = np.empty_like(demb)
    e0m, embm, dym = _f64(e0_mag), _f64(emb_mag), _f64(dy_mag)
    _check(_load().oracle_interact_bwd(N, d, B, _mode(include_self, alongside), _ptr(e0), _ptr(e0m),
                                       _ptr(emb), _ptr(embm), _ptr(dy), _ptr(dym),
                                       _ptr(de0), _ptr(de0m), _ptr(demb), _ptr(dembm)),
           "interact_bwd")
    return de0, de0m, demb, dembm


def coalesce(rows, offsets, indices, B: int):
    """Stable sort of lookups by (table, row) and run-length encoding.

    Returns a dict with sorted_pos, sorted_row, uniq_table, uniq_row, seg_off
    (length U+1) and U.
    """
    rows, offsets, indices = _i64(rows), _i64(offsets), _i64(indices)
    T, nnz = rows.size, indices.size
    sorted_pos = np.empty(nnz, dtype=np.int64)
    sorted_row = np.empty(nnz, dtype=np.int64)
    uniq_table = np.empty(nnz, dtype=np.int32)
    uniq_row = np.empty(nnz, dtype=np.int64)
    seg_off = np.empty(nnz + 1, dtype=np.int64)
    U = np.zeros(1, dtype=np.int64)
    _check(_load().oracle_coalesce(T, B, _ptr(rows), _ptr(offsets), _ptr(indices), nnz,
                                   _ptr(sorted_pos), _ptr(sorted_row), _ptr(uniq_table),
                                   _ptr(uniq_row), _ptr(seg_off), _ptr(U)), "coalesce")
    u = int(U[0])
    return dict(sorted_pos=sorted_pos, sorted_row=sorted_row, uniq_table=uniq_table[:u].copy(),
                uniq_row=uniq_row[:u].copy(), seg_off=seg_off[:u + 1].copy(), U=u)


def adagrad(tables, dtype: str, offsets, B: int, nnz: int, dpooled, lr: float, eps: float, state, co: dict,
            dpooled_mag=None):
    """Row-wise AdaGrad on the coalesced gradients, one result per unique key.

    ``state`` holds the accumulator of each unique key of ``co`` (the result of
    :func:`coalesce`), in that order.  Returns (grad, grad_mag, new_state,
    new_state_mag, new_row, new_row_mag) in fp64: [U][d], [U], [U][d].
    """
    held, arr, rows = _tables_arg(tables, dtype)
    T, d = len(held), held[0].shape[1]
    offsets = _i64(offsets)
    dpooled = _f64(dpooled)
    U = co["U"]
    grad = np.empty((U, d), dtype=np.float64)
    gm = np.empty_like(grad)
    ns = np.empty(U, dtype=np.float64)
    nsm = np.empty_like(ns)
    nr = np.empty_like(grad)
    nrm = np.empty_like(grad)
    sp = _i64(co["sorted_pos"])
    ut = np.ascontiguousarray(co["uniq_table"], dtype=np.int32)
    ur = _i64(co["uniq_row"])
    so = _i64(co["seg_off"])
    st = _f64(np.asarray(state, dtype=np.float64).reshape(U))
    _check(_load().oracle_adagrad(T, d, _DTYPE_CODES[dtype], arr, _ptr(rows), B, _ptr(offsets), nnz,
                                  _ptr(dpooled), _ptr(_f64(dpooled_mag)), float(lr), float(eps), _ptr(sp),
                                  _ptr(ut), _ptr(ur), _ptr(so), U, _ptr(st), _ptr(grad), _ptr(gm), _ptr(ns),
                                  _ptr(nsm), _ptr(nr), _ptr(nrm)), "adagrad")
    return grad, gm, ns, nsm, nr, nrm


def sgd(tables, dtype: str, offsets, B: int, nnz: int, dpooled, lr: float, co: dict,
        dpooled_mag=None):
    """Coalesced row gradients and SGD-updated rows, one per unique key.

    ``co`` is the result of :func:`coalesce`.  Returns (grad, grad_mag,
    new_row, new_row_mag), each [U][d] in fp64.
    """
    held, arr, rows = _tables_arg(tables, dtype)
    T, d = len(held), held[0].shape[1]
    offsets = _i64(offsets)
    dpooled = _f64(dpooled)
    U = co["U"]
    grad = np.empty((U, d), dtype=np.float64)
    gm = np.empty_like(grad)
    nr = np.empty_like(grad)
    nrm = np.empty_like(grad)
    sp = _i64(co["sorted_pos"])
    ut = np.ascontiguousarray(co["uniq_table"], dtype=np.int32)
    ur = _i64(co["uniq_row"])
    so = _i64(co["seg_off"])
    _check(_load().oracle_sgd(T, d, _DTYPE_CODES[dtype], arr, _ptr(rows), B, _ptr(offsets), nnz,
                              _ptr(dpooled), _ptr(_f64(dpooled_mag)), float(lr), _ptr(sp),
                              _ptr(ut), _ptr(ur), _ptr(so), U, _ptr(grad), _ptr(gm), _ptr(nr),
                              _ptr(nrm)), "sgd")
    return grad, gm, nr, nrm
