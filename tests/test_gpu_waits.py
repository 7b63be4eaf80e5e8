"""Bounded waits that run out on purpose: the kernel gives up within the
limit, reports it, and writes nothing it should not (no fault, no hang).

The waits are made to run out through the library's testing hook
(dlrm_set_wait_test_hooks), never by a fault: the radix sort's tile counters
start past the first tile, so in the second pass (the first takes its offsets
from the digit scan) the next tile waits for counts that nobody publishes; the bulk-copy interaction kernel's stage-barrier waits are given
no polls at all, so each CTA gives up before its first chunk and drains its
copies before leaving.  After each case the hooks are reset and the same
call must again match the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import _native
from sparse_dense_interaction_gb300 import workloads as W
from tests._parity import REL, assert_close, device_table_bits, device_table_f64, host_table_bits

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()
    oracle.build()


@pytest.fixture(autouse=True)
def _reset_hooks():
    yield
    sdi.dlrm_set_wait_test_hooks()
    sdi.dlrm_set_interact_kernel(_native.INTERACT_KERNEL_AUTO)


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _guarded_workspace(nbytes):
    """A workspace with a guard band of a known pattern on each side."""
    buf = torch.full((nbytes + 2 * GUARD,), 0xA5, dtype=torch.uint8, device=DEV)
    return buf, buf[GUARD:GUARD + nbytes]


def _guards_intact(buf, nbytes):
    b = buf.cpu().numpy()
    return bool((b[:GUARD] == 0xA5).all() and (b[GUARD + nbytes:] == 0xA5).all())


def test_sort_lookback_wait_runs_out_and_nothing_is_updated():
    # one table with four sort tiles and two LSD passes; the passes start
    # claiming at tile 1, so in the second pass (the first reads its offsets
    # from the digit scan and never waits) tile 1 waits for tile 0's digit
    # counts, which never come
    cfg = W.make_config("capacity", T=1, rows=[50000], B=400, bag=("fixed", 32))
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    assert indices.size > 3 * 4096
    assert sdi.dlrm_emb_bag_sort_plan(cfg["rows"], indices.size) == (2, False)
    dp = W.make_dpooled(cfg)
    nbytes = sdi.dlrm_emb_bag_bwd_workspace_size(1, cfg["B"], indices.size, cfg["d"])
    buf, ws = _guarded_workspace(nbytes)
    tables = W.tables_to_device(host, "f32")
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    off_t, idx_t, dp_t = _t(offsets), _t(indices), _t(dp)
    torch.cuda.synchronize()
    sdi.dlrm_set_wait_test_hooks(sort_wait_polls=2000, sort_first_tile=1)
    t0 = time.perf_counter()
    sdi.dlrm_emb_bag_bwd_sgd(tables, off_t, idx_t, cfg["B"], dp_t, 0.05, ws, err_flag=flag)
    status = sdi.dlrm_read_error(flag)
    elapsed = time.perf_counter() - t0
    sdi.dlrm_set_wait_test_hooks()
    assert status == _native.ERR_WAIT_TIMEOUT
    assert elapsed < 1.0, f"the wait took {elapsed:.3f} s to give up"
    assert _guards_intact(buf, nbytes), "a write left the workspace"
    np.testing.assert_array_equal(device_table_bits(tables[0]), host_table_bits(host[0], "f32"))

    # the same call with the hooks reset: correct again, in the same workspace
    flag.zero_()
    view = sdi.dlrm_emb_bag_bwd_sgd(tables, off_t, idx_t, cfg["B"], dp_t, 0.05, ws, err_flag=flag, want_view=True)
    assert sdi.dlrm_read_error(flag) == 0
    assert _guards_intact(buf, nbytes)
    co = oracle.coalesce(cfg["rows"], offsets, indices, cfg["B"])
    np.testing.assert_array_equal(view["sorted_pos"].cpu().numpy().view(np.uint32)[:indices.size],
                                  co["sorted_pos"])
    _, _, w_ref, w_mag = oracle.sgd(host, "f32", offsets, cfg["B"], indices.size, dp, 0.05, co)
    assert_close(device_table_f64(tables[0], "f32")[co["uniq_row"]], w_ref, w_mag, REL["f32"], "rows after reset")


def test_split_coalescing_wait_runs_out_and_the_reduce_updates_nothing():
    # the same failure through the split calls: the coalescing alone gives up,
    # and the reduce that follows it (on the same workspace) writes no row
    cfg = W.make_config("multi-hot", T=2, rows=[40000, 9000], B=600)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = W.make_dpooled(cfg)
    nbytes = sdi.dlrm_emb_bag_bwd_workspace_size(2, cfg["B"], indices.size, cfg["d"])
    buf, ws = _guarded_workspace(nbytes)
    tables = W.tables_to_device(host, "f16")
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    sdi.dlrm_set_wait_test_hooks(sort_wait_polls=500, sort_first_tile=1)
    sdi.dlrm_emb_bag_coalesce(cfg["rows"], cfg["d"], _t(offsets), _t(indices), cfg["B"], ws, err_flag=flag)
    sdi.dlrm_set_wait_test_hooks()
    sdi.dlrm_emb_bag_reduce_sgd(tables, indices.size, cfg["B"], _t(dp), 0.1, ws, err_flag=flag)
    assert sdi.dlrm_read_error(flag) == _native.ERR_WAIT_TIMEOUT
    assert _guards_intact(buf, nbytes)
    for t in range(2):
        np.testing.assert_array_equal(device_table_bits(tables[t]), host_table_bits(host[t], "f16"))


def test_bulk_copy_interaction_wait_runs_out_and_poisons_the_pairs():
    # the CUDA-core interaction forward fed by bulk tensor copies; with no
    # polls every CTA gives up at its first stage, drains its copies and
    # writes NaN into its samples' pairs
    rng = np.random.default_rng(9)
    B, N, d = 300, 8, 64
    e0 = rng.standard_normal((B, d), dtype=np.float32)
    emb = rng.standard_normal((B, N, d), dtype=np.float32)
    P = sdi.dlrm_num_pairs(N, False)
    y = torch.zeros((B, d + P), device=DEV)
    sdi.dlrm_set_interact_kernel(_native.INTERACT_KERNEL_CUDA_CORE)
    sdi.dlrm_set_wait_test_hooks(copy_wait_polls=0)
    t0 = time.perf_counter()
    sdi.dlrm_interact_fwd(_t(e0), _t(emb), False, y)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.0
    sdi.dlrm_set_wait_test_hooks()
    got = y.cpu().numpy()
    assert np.isnan(got[:, d:]).all(), "every sample's pairs carry the failure"
    # the same call with the hooks reset matches the oracle
    sdi.dlrm_interact_fwd(_t(e0), _t(emb), False, y)
    ref, mag = oracle.interact_fwd(e0, emb, False)
    assert_close(y.cpu().numpy(), ref, mag, REL["f32"], "interaction after reset")


def test_wait_hooks_reject_a_negative_first_tile():
    with pytest.raises(sdi.DlrmError) as e:
        sdi.dlrm_set_wait_test_hooks(sort_first_tile=-1)
    assert e.value.status == _native.ERR_INVALID_ARG
