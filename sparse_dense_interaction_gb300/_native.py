"""ctypes binding of ``libdlrm_sparse.so`` (C ABI: ``include/dlrm_sparse.h``).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  The functions carry the C names and take torch CUDA tensors (torch
provides device memory and streams); they raise :class:`DlrmError` on a
non-zero status.  There is no fallback: if the library is missing the first
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

F32, F16, BF16, INT4 = 0, 1, 2, 3
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL = 0, -1, -2, -3
ERR_INDEX_OOB, ERR_BAD_OFFSETS, ERR_CAPACITY, ERR_CUDA, ERR_WAIT_TIMEOUT = -4, -5, -6, -7, -8
FLAG_INDEX_OOB, FLAG_BAD_OFFSETS, FLAG_CAPACITY, FLAG_WAIT_TIMEOUT = 1, 2, 4, 8
MAX_TABLES = 256

_TORCH_DTYPES = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

# (name, restype, argtypes) of every exported entry point
_i32, _i64, _u64, _vp, _sz, _f32 = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p,
                                    ctypes.c_size_t, ctypes.c_float)


class CoalescedView(ctypes.Structure):
    _fields_ = [("sorted_pos", _vp), ("sorted_row", _vp), ("uniq_table", _vp),
                ("uniq_row", _vp), ("seg_off", _vp), ("num_unique", _vp)]


SIGNATURES = {
    "dlrm_emb_bag_fwd": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i64, _i64, _vp, _i64, _i64,
                                _vp, _vp]),
    "dlrm_num_pairs": (_i64, [_i32, _i32]),
    "dlrm_interact_width": (_i64, [_i32, _i32, _i32]),
    "dlrm_interact_fwd": (_i32, [_vp, _i64, _vp, _i64, _i32, _i32, _i64, _i32, _vp, _i64, _vp]),
    "dlrm_interact_bwd": (_i32, [_vp, _i64, _vp, _i64, _i32, _i32, _i64, _i32, _vp, _i64, _vp,
                                 _i64, _vp, _i64, _vp]),
    "dlrm_set_interact_kernel": (_i32, [_i32]),
    "dlrm_get_interact_kernel": (_i32, []),
    "dlrm_set_wait_test_hooks": (_i32, [_i64, _i32, _i64]),
    "dlrm_emb_bag_bwd_workspace_size": (_sz, [_i32, _i64, _i64, _i32]),
    "dlrm_emb_bag_sort_plan": (_i32, [_vp, _i32, _i64, _vp, _vp]),
    "dlrm_emb_bag_bwd_sgd": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i64, _i64, _vp, _i64,
                                    _i64, _f32, _vp, _i64, _vp, _sz, ctypes.POINTER(CoalescedView),
                                    _vp, _vp]),
    "dlrm_emb_bag_bwd_sgd_atomic": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i64, _i64, _vp, _i64,
                                           _i64, _f32, _vp, _vp]),
    "dlrm_emb_bag_bwd_sgd_noalloc": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i64, _i64, _vp,
                                            _i64, _i64, _f32, _vp, _i64, ctypes.POINTER(CoalescedView),
                                            _vp, _vp]),
    "dlrm_emb_bag_interact_fwd": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i64, _i64, _vp, _i64, _i32,
                                         _vp, _i64, _vp, _i64, _i64, _vp, _vp]),
    "dlrm_emb_bag_coalesce": (_i32, [_vp, _i32, _i32, _vp, _vp, _i64, _i64, _vp, _sz,
                                     ctypes.POINTER(CoalescedView), _vp, _vp]),
    "dlrm_emb_bag_reduce_sgd": (_i32, [_vp, _vp, _i32, _i32, _i32, _i64, _i64, _vp, _i64, _i64, _f32, _vp, _i64,
                                       _vp, _sz, _vp, _vp]),
    "dlrm_emb_bag_bwd_adagrad": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _i64, _i64, _vp, _i64, _i64,
                                        _f32, _f32, _vp, _i64, _vp, _sz, ctypes.POINTER(CoalescedView), _vp,
                                        _vp]),
    "dlrm_emb_bag_reduce_adagrad": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i64, _i64, _vp, _i64, _i64, _f32,
                                           _f32, _vp, _i64, _vp, _sz, _vp, _vp]),
    "dlrm_int4_row_bytes": (_i64, [_i32]),
    "dlrm_quantize_int4": (_i32, [_vp, _i32, _i64, _i32, _vp, _vp]),
    "dlrm_read_error": (_i32, [_vp, _vp]),
    "dlrm_clear_error": (_i32, [_vp, _vp]),
    "dlrm_status_string": (ctypes.c_char_p, [_i32]),
    "dlrm_kernel_launch_count": (_u64, []),
    "dlrm_profile_events": (_i32, [_vp, _i32]),
}

_lock = threading.Lock()
_lib = None


class DlrmError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.lib_path("libdlrm_sparse.so")


def load():
    """Loads the CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it first "
                                   "(python -m sparse_dense_interaction_gb300.build)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().dlrm_status_string(status).decode()


def _check(status: int, what: str):
    if status != OK:
        raise DlrmError(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _tables(tables, d=None):
    """Pointers, rows, T, d and type of a list of tables.  uint8 tables are
    row-wise int4 tables ([rows][dlrm_int4_row_bytes(d)]) and need ``d``."""
    T = len(tables)
    ptrs = (ctypes.c_void_p * max(T, 1))(*[t.data_ptr() for t in tables])
    rows = (ctypes.c_int64 * max(T, 1))(*[t.shape[0] for t in tables])
    for t in tables:
        if t.dtype != tables[0].dtype or t.dim() != 2 or t.stride(1) != 1 or t.stride(0) != t.shape[1]:
            raise ValueError("tables must share one dtype and be contiguous [rows][d]")
    if tables[0].dtype == torch.uint8:
        if d is None or tables[0].shape[1] != dlrm_int4_row_bytes(d):
            raise ValueError("int4 tables need d, with rows of dlrm_int4_row_bytes(d) bytes")
        return ptrs, rows, T, d, INT4
    return ptrs, rows, T, tables[0].shape[1], _TORCH_DTYPES[tables[0].dtype]


def dlrm_int4_row_bytes(d: int) -> int:
    return int(load().dlrm_int4_row_bytes(d))


def dlrm_quantize_int4(src, stream=None):
    """Row-wise int4 encoding of a [rows][d] fp32/fp16/bf16 CUDA table:
    returns a uint8 [rows][dlrm_int4_row_bytes(d)] tensor."""
    if src.dim() != 2 or src.stride(1) != 1 or src.stride(0) != src.shape[1]:
        raise ValueError("src must be a contiguous [rows][d] table")
    R, d = src.shape
    dst = torch.empty((R, max(dlrm_int4_row_bytes(d), 0)), dtype=torch.uint8, device=src.device)
    _check(load().dlrm_quantize_int4(src.data_ptr(), _TORCH_DTYPES[src.dtype], R, d, dst.data_ptr(),
                                     _stream(stream)), "dlrm_quantize_int4")
    return dst


def dlrm_emb_bag_fwd(tables, offsets, indices, B: int, out, err_flag=None, stream=None, d=None):
    """Sum-pooled lookups into ``out`` ([B][T][d] fp32, any strides, last dim 1).
    ``d`` is needed only for int4 (uint8) tables."""
    ptrs, rows, T, d, dtype = _tables(tables, d)
    if out.stride(2) != 1:
        raise ValueError("out must have unit stride in its last dimension")
    _check(load().dlrm_emb_bag_fwd(ptrs, rows, T, d, dtype, offsets.data_ptr(), _ptr(indices),
                                   indices.numel(), B, out.data_ptr(), out.stride(0), out.stride(1),
                                   _ptr(err_flag), _stream(stream)), "dlrm_emb_bag_fwd")


def dlrm_num_pairs(N: int, include_self: bool) -> int:
    return int(load().dlrm_num_pairs(N, int(bool(include_self))))


INTERACT_SELF, INTERACT_ALONGSIDE = 1, 2
INTERACT_KERNEL_AUTO, INTERACT_KERNEL_CUDA_CORE = 0, 1


def dlrm_set_interact_kernel(kind: int) -> None:
    """Kernel family of the interaction calls: INTERACT_KERNEL_AUTO (tensor cores
    where they apply) or INTERACT_KERNEL_CUDA_CORE (process-wide)."""
    _check(load().dlrm_set_interact_kernel(int(kind)), "dlrm_set_interact_kernel")


def dlrm_set_wait_test_hooks(sort_wait_polls: int = -1, sort_first_tile: int = 0,
                             copy_wait_polls: int = -1) -> None:
    """Testing aid: shortens the kernels' bounded waits (see the C header);
    the defaults restore normal operation."""
    _check(load().dlrm_set_wait_test_hooks(sort_wait_polls, sort_first_tile, copy_wait_polls),
           "dlrm_set_wait_test_hooks")


def dlrm_get_interact_kernel() -> int:
    return int(load().dlrm_get_interact_kernel())


def _mode(include_self, alongside):
    return (INTERACT_SELF if include_self else 0) | (INTERACT_ALONGSIDE if alongside else 0)


def dlrm_interact_width(N: int, d: int, include_self: bool, alongside: bool = False) -> int:
    """Width of an interaction output row: [e0 | pairs], or [e0 | e_1 .. e_N | pairs] alongside."""
    return int(load().dlrm_interact_width(N, d, _mode(include_self, alongside)))


def dlrm_interact_fwd(e0, emb, include_self: bool, y, stream=None, alongside: bool = False):
    """``y[b] = [e0[b] | z_i . z_j over pairs]`` for ``emb`` of shape [B][N][d]."""
    B, N, d = emb.shape
    if emb.stride(2) != 1 or emb.stride(1) != d or e0.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("rows must be contiguous and emb's tables adjacent")
    _check(load().dlrm_interact_fwd(e0.data_ptr(), e0.stride(0), emb.data_ptr(), emb.stride(0), N, d,
                                    B, _mode(include_self, alongside), y.data_ptr(), y.stride(0),
                                    _stream(stream)), "dlrm_interact_fwd")


def dlrm_interact_bwd(e0, emb, include_self: bool, dy, de0, demb, stream=None, alongside: bool = False):
    """Gradients of :func:`dlrm_interact_fwd` into ``de0`` [B][d] and ``demb`` [B][N][d]."""
    B, N, d = emb.shape
    for t in (emb, demb):
        if t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError("rows must be contiguous and tables adjacent")
    _check(load().dlrm_interact_bwd(e0.data_ptr(), e0.stride(0), emb.data_ptr(), emb.stride(0), N, d,
                                    B, _mode(include_self, alongside), dy.data_ptr(), dy.stride(0),
                                    de0.data_ptr(), de0.stride(0), demb.data_ptr(), demb.stride(0),
                                    _stream(stream)), "dlrm_interact_bwd")


def dlrm_emb_bag_bwd_workspace_size(T: int, B: int, nnz: int, d: int) -> int:
    return int(load().dlrm_emb_bag_bwd_workspace_size(T, B, nnz, d))


def dlrm_emb_bag_sort_plan(rows, nnz: int):
    """(LSD passes, MSD bucket sort used) of the coalescing for tables of
    ``rows`` rows and ``nnz`` lookups (host only)."""
    T = len(rows)
    r = (ctypes.c_int64 * max(T, 1))(*rows)
    passes, msd = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().dlrm_emb_bag_sort_plan(r, T, nnz, ctypes.byref(passes), ctypes.byref(msd)),
           "dlrm_emb_bag_sort_plan")
    return passes.value, bool(msd.value)


def dlrm_emb_bag_bwd_sgd(tables, offsets, indices, B: int, dpooled, lr: float, workspace,
                         grad_rows=None, err_flag=None, stream=None, want_view: bool = False):
    """Coalesces duplicate lookups and applies row-wise SGD to ``tables`` in place.

    ``dpooled`` is [B][T][d] fp32 (any strides, last dim 1); ``workspace`` a
    uint8 CUDA tensor of at least :func:`dlrm_emb_bag_bwd_workspace_size`
    bytes; ``grad_rows`` an optional [cap][d] fp32 tensor for the coalesced
    gradients.  With ``want_view`` returns a dict of tensor views into the
    workspace (sorted_pos, sorted_row, uniq_table, uniq_row, seg_off as
    uint32/int32 of capacity nnz or nnz + 1, and num_unique as int64[1]).
    """
    ptrs, rows, T, d, dtype = _tables(tables)
    if dpooled.stride(2) != 1:
        raise ValueError("dpooled must have unit stride in its last dimension")
    view = CoalescedView()
    nnz = indices.numel()
    cap = 0 if grad_rows is None else grad_rows.shape[0]
    _check(load().dlrm_emb_bag_bwd_sgd(ptrs, rows, T, d, dtype, offsets.data_ptr(), _ptr(indices), nnz,
                                       B, dpooled.data_ptr(), dpooled.stride(0), dpooled.stride(1),
                                       float(lr), _ptr(grad_rows), cap, workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(),
                                       ctypes.byref(view) if want_view else None, _ptr(err_flag),
                                       _stream(stream)), "dlrm_emb_bag_bwd_sgd")
    return _view_tensors(view, workspace, nnz) if want_view else None


def _view_tensors(view, workspace, nnz):
    base = workspace.data_ptr()

    def sub(ptr, n, dt):
        off = ptr - base
        return workspace[off:off + n * 4].view(dt) if dt != torch.int64 else workspace[off:off + 8].view(dt)

    return dict(sorted_pos=sub(view.sorted_pos, nnz, torch.int32),
                sorted_row=sub(view.sorted_row, nnz, torch.int32),
                uniq_table=sub(view.uniq_table, nnz, torch.int32),
                uniq_row=sub(view.uniq_row, nnz, torch.int32),
                seg_off=sub(view.seg_off, nnz + 1, torch.int32),
                num_unique=sub(view.num_unique, 1, torch.int64))


def dlrm_emb_bag_coalesce(rows, d: int, offsets, indices, B: int, workspace, err_flag=None, stream=None,
                          want_view: bool = False):
    """The coalescing half of :func:`dlrm_emb_bag_bwd_sgd` (reads only
    ``rows``, a list of T table row counts, and the lookups)."""
    T = len(rows)
    r = (ctypes.c_int64 * max(T, 1))(*rows)
    view = CoalescedView()
    nnz = indices.numel()
    _check(load().dlrm_emb_bag_coalesce(r, T, d, offsets.data_ptr(), _ptr(indices), nnz, B,
                                        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                        ctypes.byref(view) if want_view else None, _ptr(err_flag),
                                        _stream(stream)), "dlrm_emb_bag_coalesce")
    return _view_tensors(view, workspace, nnz) if want_view else None


def dlrm_emb_bag_reduce_sgd(tables, nnz: int, B: int, dpooled, lr: float, workspace, grad_rows=None,
                            err_flag=None, stream=None):
    """The reduce + update half of :func:`dlrm_emb_bag_bwd_sgd`, on a
    workspace filled by :func:`dlrm_emb_bag_coalesce`."""
    ptrs, rows, T, d, dtype = _tables(tables)
    if dpooled.stride(2) != 1:
        raise ValueError("dpooled must have unit stride in its last dimension")
    cap = 0 if grad_rows is None else grad_rows.shape[0]
    _check(load().dlrm_emb_bag_reduce_sgd(ptrs, rows, T, d, dtype, nnz, B, dpooled.data_ptr(), dpooled.stride(0),
                                          dpooled.stride(1), float(lr), _ptr(grad_rows), cap,
                                          workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                          _ptr(err_flag), _stream(stream)), "dlrm_emb_bag_reduce_sgd")


def dlrm_emb_bag_interact_fwd(tables, offsets, indices, B: int, e0, include_self: bool, y, pooled=None,
                              err_flag=None, stream=None, alongside: bool = False, d=None):
    """Lookup + interaction forward in one call: ``y`` ([B][d + P] fp32, last
    dim 1) receives what :func:`dlrm_interact_fwd` would give on the pooled
    vectors of :func:`dlrm_emb_bag_fwd`; ``pooled`` ([B][T][d] fp32, optional)
    also receives those pooled vectors."""
    ptrs, rows, T, d, dtype = _tables(tables, d)
    if e0.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("e0 and y must have unit stride in their last dimension")
    pss = pts = 0
    if pooled is not None:
        if pooled.stride(2) != 1:
            raise ValueError("pooled must have unit stride in its last dimension")
        pss, pts = pooled.stride(0), pooled.stride(1)
    _check(load().dlrm_emb_bag_interact_fwd(ptrs, rows, T, d, dtype, offsets.data_ptr(), _ptr(indices),
                                            indices.numel(), B, e0.data_ptr(), e0.stride(0),
                                            _mode(include_self, alongside), y.data_ptr(), y.stride(0), _ptr(pooled),
                                            pss, pts, _ptr(err_flag), _stream(stream)),
           "dlrm_emb_bag_interact_fwd")


def _states(state, tables):
    if len(state) != len(tables):
        raise ValueError("one accumulator array per table")
    for s, t in zip(state, tables):
        if s.dtype != torch.float32 or s.dim() != 1 or s.shape[0] != t.shape[0] or s.stride(0) != 1:
            raise ValueError("each accumulator array is a contiguous fp32 [rows] tensor")
    return (ctypes.c_void_p * max(len(state), 1))(*[s.data_ptr() for s in state])


def dlrm_emb_bag_bwd_adagrad(tables, state, offsets, indices, B: int, dpooled, lr: float, eps: float, workspace,
                             grad_rows=None, err_flag=None, stream=None, want_view: bool = False):
    """:func:`dlrm_emb_bag_bwd_sgd` with row-wise AdaGrad: ``state`` is a list
    of fp32 [rows] accumulators, one per table, updated in place."""
    ptrs, rows, T, d, dtype = _tables(tables)
    st = _states(state, tables)
    if dpooled.stride(2) != 1:
        raise ValueError("dpooled must have unit stride in its last dimension")
    view = CoalescedView()
    nnz = indices.numel()
    cap = 0 if grad_rows is None else grad_rows.shape[0]
    _check(load().dlrm_emb_bag_bwd_adagrad(ptrs, st, rows, T, d, dtype, offsets.data_ptr(), _ptr(indices), nnz, B,
                                           dpooled.data_ptr(), dpooled.stride(0), dpooled.stride(1), float(lr),
                                           float(eps), _ptr(grad_rows), cap, workspace.data_ptr(),
                                           workspace.numel() * workspace.element_size(),
                                           ctypes.byref(view) if want_view else None, _ptr(err_flag),
                                           _stream(stream)), "dlrm_emb_bag_bwd_adagrad")
    return _view_tensors(view, workspace, nnz) if want_view else None


def dlrm_emb_bag_reduce_adagrad(tables, state, nnz: int, B: int, dpooled, lr: float, eps: float, workspace,
                                grad_rows=None, err_flag=None, stream=None):
    """The reduce + AdaGrad half, on a workspace filled by :func:`dlrm_emb_bag_coalesce`."""
    ptrs, rows, T, d, dtype = _tables(tables)
    st = _states(state, tables)
    if dpooled.stride(2) != 1:
        raise ValueError("dpooled must have unit stride in its last dimension")
    cap = 0 if grad_rows is None else grad_rows.shape[0]
    _check(load().dlrm_emb_bag_reduce_adagrad(ptrs, st, rows, T, d, dtype, nnz, B, dpooled.data_ptr(),
                                              dpooled.stride(0), dpooled.stride(1), float(lr), float(eps),
                                              _ptr(grad_rows), cap, workspace.data_ptr(),
                                              workspace.numel() * workspace.element_size(), _ptr(err_flag),
                                              _stream(stream)), "dlrm_emb_bag_reduce_adagrad")


def dlrm_emb_bag_bwd_sgd_atomic(tables, offsets, indices, B: int, dpooled, lr: float, err_flag=None,
                                stream=None):
    """Row-wise SGD on fp32 ``tables`` in place by atomic reductions, without
    coalescing the duplicate lookups (no workspace, no coalesced gradient).
    The summation order of a row touched by several bags is unspecified."""
    ptrs, rows, T, d, dtype = _tables(tables)
    if dpooled.stride(2) != 1:
        raise ValueError("dpooled must have unit stride in its last dimension")
    _check(load().dlrm_emb_bag_bwd_sgd_atomic(ptrs, rows, T, d, dtype, offsets.data_ptr(), _ptr(indices),
                                              indices.numel(), B, dpooled.data_ptr(), dpooled.stride(0),
                                              dpooled.stride(1), float(lr), _ptr(err_flag), _stream(stream)),
           "dlrm_emb_bag_bwd_sgd_atomic")


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class _DeviceArray:
    """A device pointer the library owns, described for torch.as_tensor (CUDA array interface)."""

    def __init__(self, ptr, n, typestr):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def _raw_view_tensors(view, nnz):
    def sub(ptr, n, typestr):
        return torch.as_tensor(_DeviceArray(ptr, n, typestr), device="cuda")

    return dict(sorted_pos=sub(view.sorted_pos, nnz, "<i4"), sorted_row=sub(view.sorted_row, nnz, "<i4"),
                uniq_table=sub(view.uniq_table, nnz, "<i4"), uniq_row=sub(view.uniq_row, nnz, "<i4"),
                seg_off=sub(view.seg_off, nnz + 1, "<i4"), num_unique=sub(view.num_unique, 1, "<i8"))


def dlrm_emb_bag_bwd_sgd_noalloc(tables, offsets, indices, B: int, dpooled, lr: float,
                                 grad_rows=None, err_flag=None, stream=None, want_view: bool = False):
    """:func:`dlrm_emb_bag_bwd_sgd` without a workspace: the library's fixed
    scratch array is used instead, so nothing is allocated.  For callers that
    cannot allocate device memory; sizes whose scratch exceeds
    ``NOALLOC_SCRATCH_BYTES`` raise (status DLRM_ERR_WORKSPACE_TOO_SMALL).
    With ``want_view`` returns tensors aliasing the coalescing results inside
    that array (as :func:`dlrm_emb_bag_bwd_sgd`; valid until the next call)."""
    ptrs, rows, T, d, dtype = _tables(tables)
    if dpooled.stride(2) != 1:
        raise ValueError("dpooled must have unit stride in its last dimension")
    cap = 0 if grad_rows is None else grad_rows.shape[0]
    view = CoalescedView()
    nnz = indices.numel()
    _check(load().dlrm_emb_bag_bwd_sgd_noalloc(ptrs, rows, T, d, dtype, offsets.data_ptr(), _ptr(indices),
                                               nnz, B, dpooled.data_ptr(), dpooled.stride(0),
                                               dpooled.stride(1), float(lr), _ptr(grad_rows), cap,
                                               ctypes.byref(view) if want_view else None,
                                               _ptr(err_flag), _stream(stream)),
           "dlrm_emb_bag_bwd_sgd_noalloc")
    return _raw_view_tensors(view, nnz) if want_view else None


def dlrm_read_error(err_flag, stream=None) -> int:
    """Synchronizes the stream and returns the status the flag's bits map to."""
    return int(load().dlrm_read_error(err_flag.data_ptr(), _stream(stream)))


def dlrm_clear_error(err_flag, stream=None):
    _check(load().dlrm_clear_error(err_flag.data_ptr(), _stream(stream)), "dlrm_clear_error")


def dlrm_kernel_launch_count() -> int:
    return int(load().dlrm_kernel_launch_count())


def dlrm_profile_events(events):
    """Registers torch CUDA events to be recorded after each of the library's
    next kernel launches on this thread (``[]`` unregisters).  Each event must
    have been recorded once already, so that its CUDA handle exists."""
    handles = [e.cuda_event for e in events]
    if any(h == 0 for h in handles):
        raise ValueError("record each event once before registering it")
    arr = (ctypes.c_void_p * max(len(handles), 1))(*handles)
    _check(load().dlrm_profile_events(arr, len(handles)), "dlrm_profile_events")
