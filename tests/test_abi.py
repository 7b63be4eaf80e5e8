"""The C-ABI library: it loads, exports what the header declares, and rejects
bad arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.load()


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(dlrm_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_path(lib):
    names = declared_functions()
    for required in ("dlrm_emb_bag_fwd", "dlrm_interact_fwd", "dlrm_interact_bwd",
                     "dlrm_emb_bag_bwd_sgd", "dlrm_emb_bag_bwd_workspace_size"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, f"binding lacks {name}"


def test_status_strings_and_pair_counts(lib):
    assert sdi.status_string(0) == "ok"
    assert "workspace" in sdi.status_string(-3)
    assert sdi.dlrm_num_pairs(8, False) == 36
    assert sdi.dlrm_num_pairs(26, False) == 351
    assert sdi.dlrm_num_pairs(100, True) == 5151
    assert lib.dlrm_num_pairs(-1, 0) == -1


def test_workspace_size_grows_with_the_batch(lib):
    a = sdi.dlrm_emb_bag_bwd_workspace_size(26, 65536, 1_000_000, 128)
    b = sdi.dlrm_emb_bag_bwd_workspace_size(26, 65536, 2_000_000, 128)
    assert 32 * 1_000_000 <= a < b
    assert sdi.dlrm_emb_bag_bwd_workspace_size(0, 1, 1, 1) == 0
    assert sdi.dlrm_emb_bag_bwd_workspace_size(1, 1, (1 << 31) + 1, 1) == 0


FAKE = 0x10000  # never dereferenced: every call below fails its host checks first


def _tables(n, rows=100):
    ptrs = (ctypes.c_void_p * n)(*([FAKE] * n))
    r = (ctypes.c_int64 * n)(*([rows] * n))
    return ptrs, r


def test_forward_rejects_bad_arguments(lib):
    p, r = _tables(4)
    call = lambda **kw: lib.dlrm_emb_bag_fwd(
        kw.get("tables", p), kw.get("rows", r), kw.get("T", 4), kw.get("d", 16), kw.get("dtype", 0),
        kw.get("offsets", FAKE), FAKE, 10, kw.get("B", 2), kw.get("out", FAKE), 64, 16, None, None)
    assert call(T=0) == _native.ERR_INVALID_ARG
    assert call(d=0) == _native.ERR_INVALID_ARG
    assert call(dtype=4) == _native.ERR_INVALID_ARG  # no such table type
    # int4 tables: d must be even (else invalid), a multiple of 8 and at most 512
    assert call(dtype=_native.INT4, d=13) == _native.ERR_INVALID_ARG
    assert call(dtype=_native.INT4, d=12) == _native.ERR_UNSUPPORTED
    assert call(dtype=_native.INT4, d=520) == _native.ERR_UNSUPPORTED
    assert call(tables=None) == _native.ERR_INVALID_ARG
    assert call(offsets=None) == _native.ERR_INVALID_ARG
    assert call(out=None) == _native.ERR_INVALID_ARG
    assert call(B=-1) == _native.ERR_INVALID_ARG
    big_p, big_r = _tables(_native.MAX_TABLES + 1)
    assert call(tables=big_p, rows=big_r, T=_native.MAX_TABLES + 1) == _native.ERR_UNSUPPORTED
    zero_rows = (ctypes.c_int64 * 4)(100, 0, 100, 100)
    assert call(rows=zero_rows) == _native.ERR_INVALID_ARG
    huge_rows = (ctypes.c_int64 * 4)(100, 1 << 33, 100, 100)
    assert call(rows=huge_rows) == _native.ERR_UNSUPPORTED
    assert call(B=0) == _native.OK  # nothing to do, nothing launched
    assert lib.dlrm_kernel_launch_count() == 0


def test_interaction_rejects_bad_arguments(lib):
    fwd = lambda N=4, d=8, B=2, ys=100, y=FAKE: lib.dlrm_interact_fwd(
        FAKE, d, FAKE, max(N, 1) * d, N, d, B, 0, y, ys, None)
    assert fwd(N=-1) == _native.ERR_INVALID_ARG
    assert fwd(d=0) == _native.ERR_INVALID_ARG
    assert fwd(N=128, ys=10000) == _native.ERR_UNSUPPORTED
    assert fwd(ys=8 + 10 - 1) == _native.ERR_INVALID_ARG  # width d + P = 18
    assert fwd(y=None) == _native.ERR_INVALID_ARG
    assert fwd(B=0) == _native.OK
    # the mode's unknown bits, and the alongside width (d (N + 1) + P = 40 + 10)
    mfwd = lambda mode, ys: lib.dlrm_interact_fwd(FAKE, 8, FAKE, 32, 4, 8, 2, mode, FAKE, ys, None)
    assert mfwd(4, 1000) == _native.ERR_INVALID_ARG
    assert mfwd(2, 49) == _native.ERR_INVALID_ARG
    assert lib.dlrm_interact_width(4, 8, 2) == 50 and lib.dlrm_interact_width(4, 8, 3) == 55
    assert lib.dlrm_interact_width(4, 8, 8) == -1
    bwd = lambda dys=18, de0s=8: lib.dlrm_interact_bwd(FAKE, 8, FAKE, 32, 4, 8, 2, 0, FAKE, dys, FAKE,
                                                       de0s, FAKE, 32, None)
    assert bwd(dys=17) == _native.ERR_INVALID_ARG
    assert bwd(de0s=7) == _native.ERR_INVALID_ARG
    assert lib.dlrm_kernel_launch_count() == 0


def test_fused_forward_rejects_bad_arguments(lib):
    p, r = _tables(4)
    width = 16 + 10  # d + P for F = 5 strict
    call = lambda **kw: lib.dlrm_emb_bag_interact_fwd(
        kw.get("tables", p), kw.get("rows", r), kw.get("T", 4), 16, 0, FAKE, FAKE, 10, kw.get("B", 2),
        kw.get("e0", FAKE), kw.get("e0s", 16), 0, kw.get("y", FAKE), kw.get("ys", width),
        kw.get("pooled", None), kw.get("pss", 64), 16, None, None)
    assert call(ys=width - 1) == _native.ERR_INVALID_ARG
    assert call(e0s=15) == _native.ERR_INVALID_ARG
    assert call(e0=None) == _native.ERR_INVALID_ARG
    assert call(y=None) == _native.ERR_INVALID_ARG
    assert call(pooled=FAKE, pss=-1) == _native.ERR_INVALID_ARG
    big_p, big_r = _tables(128)
    assert call(tables=big_p, rows=big_r, T=128, ys=100000) == _native.ERR_UNSUPPORTED  # N <= 127
    assert call(B=0) == _native.OK
    assert lib.dlrm_kernel_launch_count() == 0


def test_int4_calls_reject_bad_arguments(lib):
    assert lib.dlrm_int4_row_bytes(128) == 80 and lib.dlrm_int4_row_bytes(40) == 32
    assert lib.dlrm_int4_row_bytes(7) == -1 and lib.dlrm_int4_row_bytes(0) == -1
    q = lambda src_dtype=0, rows=4, d=16, dst=FAKE: lib.dlrm_quantize_int4(FAKE, src_dtype, rows, d, dst, None)
    assert q(src_dtype=3) == _native.ERR_INVALID_ARG  # int4 is not a source type
    assert q(d=15) == _native.ERR_INVALID_ARG
    assert q(d=20) == _native.ERR_UNSUPPORTED  # even, not a multiple of 8
    assert q(dst=FAKE + 8) == _native.ERR_INVALID_ARG  # the encoded rows start 16-byte aligned
    assert q(rows=0) == _native.OK
    # 4-bit tables are not trained
    p, r = _tables(2)
    need = sdi.dlrm_emb_bag_bwd_workspace_size(2, 8, 100, 16)
    assert lib.dlrm_emb_bag_bwd_sgd(p, r, 2, 16, _native.INT4, FAKE, FAKE, 100, 8, FAKE, 32, 16, 0.1, None, 0,
                                    0x100000, need, None, None, None) == _native.ERR_UNSUPPORTED
    assert lib.dlrm_kernel_launch_count() == 0


def test_backward_rejects_bad_arguments(lib):
    p, r = _tables(2)
    need = sdi.dlrm_emb_bag_bwd_workspace_size(2, 8, 100, 16)
    call = lambda **kw: lib.dlrm_emb_bag_bwd_sgd(
        p, r, 2, 16, 0, FAKE, FAKE, kw.get("nnz", 100), 8, FAKE, 32, 16, kw.get("lr", 0.1), None, 0,
        kw.get("ws", 0x100000), kw.get("ws_bytes", need), None, None, None)
    assert call(ws_bytes=need - 1) == _native.ERR_WORKSPACE_TOO_SMALL
    assert call(ws=0x100010) == _native.ERR_INVALID_ARG  # workspace not 256-byte aligned
    assert call(nnz=(1 << 31) + 1) == _native.ERR_UNSUPPORTED
    assert call(nnz=-1) == _native.ERR_INVALID_ARG
    assert call(lr=float("nan")) == _native.ERR_INVALID_ARG
    assert lib.dlrm_kernel_launch_count() == 0


def test_interaction_kernel_setting(lib):
    assert lib.dlrm_get_interact_kernel() == 0  # tensor cores where they apply
    assert lib.dlrm_set_interact_kernel(1) == 0 and lib.dlrm_get_interact_kernel() == 1
    assert lib.dlrm_set_interact_kernel(7) == _native.ERR_INVALID_ARG and lib.dlrm_get_interact_kernel() == 1
    assert lib.dlrm_set_interact_kernel(-1) == _native.ERR_INVALID_ARG
    assert lib.dlrm_set_interact_kernel(0) == 0 and lib.dlrm_get_interact_kernel() == 0


def test_read_error_needs_a_flag(lib):
    assert lib.dlrm_read_error(None, None) == _native.ERR_INVALID_ARG
    assert lib.dlrm_clear_error(None, None) == _native.ERR_INVALID_ARG


def test_atomic_backward_rejects_bad_arguments(lib):
    p, r = _tables(2)
    call = lambda **kw: lib.dlrm_emb_bag_bwd_sgd_atomic(
        p, r, 2, 16, kw.get("dtype", 0), kw.get("offsets", FAKE), FAKE, kw.get("nnz", 100), kw.get("B", 8),
        kw.get("dp", FAKE), kw.get("dpss", 32), 16, kw.get("lr", 0.1), None, None)
    assert call(dtype=_native.F16) == _native.ERR_UNSUPPORTED  # fp32 tables only
    assert call(dtype=_native.BF16) == _native.ERR_UNSUPPORTED
    assert call(dtype=_native.INT4) == _native.ERR_UNSUPPORTED
    assert call(nnz=-1) == _native.ERR_INVALID_ARG
    assert call(B=0) == _native.ERR_INVALID_ARG  # no bags cannot hold lookups
    assert call(nnz=(1 << 31) + 1) == _native.ERR_UNSUPPORTED
    assert call(lr=float("nan")) == _native.ERR_INVALID_ARG
    assert call(offsets=None) == _native.ERR_INVALID_ARG
    assert call(dp=None) == _native.ERR_INVALID_ARG
    assert call(dpss=-1) == _native.ERR_INVALID_ARG
    assert call(lr=0.0) == _native.OK  # nothing to update, nothing launched
    assert call(B=0, nnz=0) == _native.OK
    assert lib.dlrm_kernel_launch_count() == 0


def test_noalloc_returns_the_workspace_calls_statuses(lib):
    # the call without a workspace runs dlrm_emb_bag_bwd_sgd's own checks, its
    # fixed array in place of the workspace: every refused call gets the same
    # status (all of these fail on the host, before any device lookup)
    p, r = _tables(2)
    scratch = _native.NOALLOC_SCRATCH_BYTES
    big = 1 << 21  # lookups whose scratch exceeds the array
    assert sdi.dlrm_emb_bag_bwd_workspace_size(2, 8, big, 16) > scratch
    cases = [dict(T=0), dict(d=0), dict(dtype=4), dict(dtype=_native.INT4), dict(dtype=_native.INT4, d=12),
             dict(nnz=-1), dict(nnz=(1 << 31) + 1), dict(B=-1), dict(B=0), dict(lr=float("nan")),
             dict(offsets=None), dict(dp=None), dict(dpss=-1), dict(dpss=(1 << 29) + 1), dict(cap=-1),
             dict(nnz=big), dict(tables=None), dict(grad=FAKE + 2)]
    for kw in cases:
        kw.setdefault("tables", p)
        args = lambda: (kw["tables"], r, kw.get("T", 2), kw.get("d", 16), kw.get("dtype", 0),
                        kw.get("offsets", FAKE), FAKE, kw.get("nnz", 100), kw.get("B", 8), kw.get("dp", FAKE),
                        kw.get("dpss", 32), 16, kw.get("lr", 0.1), kw.get("grad", None), kw.get("cap", 0))
        want = lib.dlrm_emb_bag_bwd_sgd(*args(), 0x100000, scratch, None, None, None)
        got = lib.dlrm_emb_bag_bwd_sgd_noalloc(*args(), None, None, None)
        assert want != _native.OK, kw
        assert got == want, (kw, got, want)
    assert lib.dlrm_kernel_launch_count() == 0


def test_sort_plan_follows_the_row_bits_and_the_bucket_sizes(lib):
    # LSD passes: ceil(bits / 8) over the largest table's row bits
    assert sdi.dlrm_emb_bag_sort_plan([1000], 100) == (2, False)
    assert sdi.dlrm_emb_bag_sort_plan([256], 100) == (1, False)
    assert sdi.dlrm_emb_bag_sort_plan([257], 100) == (2, False)
    assert sdi.dlrm_emb_bag_sort_plan([4_000_000] * 26, 34_077_138) == (3, False)  # 5.1k keys per bucket
    # the bucket sort: 17+ row bits, every table above half the largest power of two,
    # 256 .. 2560 keys per (table, top digit) bucket on average
    assert sdi.dlrm_emb_bag_sort_plan([32_000_000] * 8, 16384 * 32 * 8) == (4, True)
    assert sdi.dlrm_emb_bag_sort_plan([1 << 16] * 2, 2 * 256 * 1000) == (2, False)  # 16 bits
    assert sdi.dlrm_emb_bag_sort_plan([(1 << 16) + 1] * 2, 2 * 256 * 1000) == (3, True)
    assert sdi.dlrm_emb_bag_sort_plan([200000], 256 * 256) == (3, True)
    assert sdi.dlrm_emb_bag_sort_plan([200000], 256 * 256 - 1) == (3, False)
    assert sdi.dlrm_emb_bag_sort_plan([200000], 256 * 2560) == (3, True)
    assert sdi.dlrm_emb_bag_sort_plan([200000], 256 * 2560 + 1) == (3, False)
    assert sdi.dlrm_emb_bag_sort_plan([200000, 131072], 2 * 256 * 1000) == (3, False)  # a table of 2^17 rows
    assert sdi.dlrm_emb_bag_sort_plan([200000, 131073], 2 * 256 * 1000) == (3, True)
    for bad in (([], 10), ([0], 10), ([100], -1)):
        with pytest.raises(sdi.DlrmError):
            sdi.dlrm_emb_bag_sort_plan(*bad)
