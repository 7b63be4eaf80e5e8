"""The backward with SGD applied by atomic reductions (fp32 tables, no
coalescing) against the oracle.

The oracle sums each row's gradient in sorted order and applies one update;
the atomic path adds each bag's share to the row in L2, in an unspecified
order.  Both are the same update up to rounding: an element passes when it
lies within rel 1e-5 of the oracle's magnitude (|w| + lr * sum |g|), which
covers one fp32 rounding per addition for the few additions per row these
inputs make (at most about a hundred).  Rows no lookup touches must keep
their bits.  The path yields no coalescing outputs (no sorted positions,
unique keys or gradient rows), so there is nothing integer to compare.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import _native
from sparse_dense_interaction_gb300 import workloads as W
from tests._parity import REL, assert_close, device_table_bits, host_table_bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()
    oracle.build()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _check_against_oracle(cfg, host, offsets, indices, dp, lr, what, dp_dev=None):
    tables = W.tables_to_device(host, "f32")
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    sdi.dlrm_emb_bag_bwd_sgd_atomic(tables, _t(offsets), _t(indices), cfg["B"], _t(dp) if dp_dev is None else dp_dev,
                                    lr, err_flag=flag)
    assert sdi.dlrm_read_error(flag) == 0
    co = oracle.coalesce(cfg["rows"], offsets, indices, cfg["B"])
    _, _, w_ref, w_mag = oracle.sgd(host, "f32", offsets, cfg["B"], indices.size, dp, lr, co)
    for t in range(cfg["T"]):
        us = np.nonzero(co["uniq_table"] == t)[0]
        rows_t = co["uniq_row"][us]
        dev = tables[t].cpu().numpy().astype(np.float64)
        assert_close(dev[rows_t], w_ref[us], w_mag[us], REL["f32"], f"{what} t={t}")
        untouched = np.ones(cfg["rows"][t], dtype=bool)
        untouched[rows_t] = False
        np.testing.assert_array_equal(device_table_bits(tables[t])[untouched],
                                      host_table_bits(host[t], "f32")[untouched])
    return co


CASES = {
    # spread indices over tables much larger than the batch (the call's use)
    "capacity-like": dict(name="capacity", B=2000, rows=[300000, 200000, 50000]),
    "one-hot-f32": dict(name="one-hot", B=1500, rows=[20000, 5000, 100000], dtype="f32"),
    "tiny": dict(name="tiny"),
    "d16": dict(name="tiny", B=500, rows=[4000, 3000], d=16),
    "d64": dict(name="capacity", B=700, rows=[40000, 90000], d=64, bag=("poisson", 6.0, 0, 20)),
    "d256": dict(name="capacity", B=300, rows=[30000, 9000], d=256, bag=("fixed", 7)),
    "d512": dict(name="tiny", B=200, rows=[3000, 500], d=512, bag=("poisson", 4.0, 0, 9)),
    "d17-scalar": dict(name="capacity", B=300, rows=[2000, 3000], d=17, bag=("fixed", 3)),
    "d3-scalar": dict(name="tiny", B=64, rows=[40, 50, 60], d=3),
}


@pytest.mark.parametrize("case", list(CASES))
def test_atomic_backward_matches_oracle(case):
    c = dict(CASES[case])
    cfg = W.make_config(c.pop("name"), **c)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = W.make_dpooled(cfg)
    co = _check_against_oracle(cfg, host, offsets, indices, dp, 0.05, case)
    assert co["U"] > 0


def test_atomic_backward_with_duplicates_in_and_across_bags():
    # row 5 is looked up 3 times in every bag (merged within the bag) and by
    # 90 bags; the other rows are spread
    rng = np.random.default_rng(5)
    B, d = 90, 128
    bags = [[5, 5, int(rng.integers(0, 400)), 5, int(rng.integers(0, 400))] for _ in range(B)]
    offsets = np.zeros(B + 1, dtype=np.int64)
    np.cumsum([len(b) for b in bags], out=offsets[1:])
    indices = np.array([i for b in bags for i in b], dtype=np.int64)
    cfg = W.make_config("capacity", T=1, rows=[400], B=B, d=d)
    host = W.tables_host(cfg)
    dp = W.make_dpooled(cfg)
    _check_against_oracle(cfg, host, offsets, indices, dp, 0.1, "duplicates")


def test_atomic_backward_strided_pooled_gradient():
    # the pooled gradients of a wider buffer (the demb block of the interaction backward with its sample stride)
    cfg = W.make_config("capacity", B=400, rows=[50000, 70000], bag=("fixed", 4))
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    wide = np.random.default_rng(2).standard_normal((cfg["B"], cfg["T"] + 1, cfg["d"]), dtype=np.float32)
    dp = wide[:, 1:, :]
    _check_against_oracle(cfg, host, offsets, indices, dp, 0.02, "strided", dp_dev=_t(wide)[:, 1:, :])


def test_atomic_backward_flags_and_skips_bad_lookups():
    cfg = W.make_config("tiny", B=64)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    indices[17] = 1000  # out of range of its table
    tables = W.tables_to_device(host, "f32")
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    sdi.dlrm_emb_bag_bwd_sgd_atomic(tables, _t(offsets), _t(indices), cfg["B"], _t(W.make_dpooled(cfg)), 0.05,
                                    err_flag=flag)
    assert sdi.dlrm_read_error(flag) == _native.ERR_INDEX_OOB
    offsets[10] = offsets[12] + 1  # not monotone
    flag.zero_()
    sdi.dlrm_emb_bag_bwd_sgd_atomic(tables, _t(offsets), _t(indices), cfg["B"], _t(W.make_dpooled(cfg)), 0.05,
                                    err_flag=flag)
    sdi.dlrm_read_error(flag)  # synchronizes
    assert int(flag.item()) & _native.FLAG_BAD_OFFSETS


def test_atomic_backward_zero_rate_and_half_tables():
    cfg = W.make_config("tiny", B=64)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    tables = W.tables_to_device(host, "f32")
    launches = sdi.dlrm_kernel_launch_count()
    sdi.dlrm_emb_bag_bwd_sgd_atomic(tables, _t(offsets), _t(indices), cfg["B"], _t(W.make_dpooled(cfg)), 0.0)
    assert sdi.dlrm_kernel_launch_count() == launches
    for t in range(cfg["T"]):
        np.testing.assert_array_equal(device_table_bits(tables[t]), host_table_bits(host[t], "f32"))
    half = [x.half() for x in tables]
    with pytest.raises(sdi.DlrmError) as e:
        sdi.dlrm_emb_bag_bwd_sgd_atomic(half, _t(offsets), _t(indices), cfg["B"], _t(W.make_dpooled(cfg)), 0.1)
    assert e.value.status == _native.ERR_UNSUPPORTED
