"""Fused lookup + interaction forward (dlrm_emb_bag_interact_fwd) vs the
oracle, and vs the two calls it fuses.

y must lie within rel x magnitude of the oracle's lookup followed by its
interaction, with and without the pooled output (with it, the call may run
the lookup and the tensor-core interaction instead of the single kernel); its
first d columns are e0 bit for bit; the pooled vectors it writes on request
are bit-identical to dlrm_emb_bag_fwd's (same lane layout and add order).
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import workloads as W
from tests._parity import REL, assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()
    oracle.build()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


CASES = {  # single-kernel shapes (several samples per CTA, ragged last CTA)
    "tiny": dict(name="tiny"),
    "one-hot-f32": dict(name="one-hot", B=301, rows=[10, 17, 30, 52, 91, 5000, 100000] * 3 + [7] * 5),
    "multi-hot-f16": dict(name="multi-hot", B=301, rows=[5000, 70000, 123, 9] * 6 + [40, 41]),
    "multi-hot-bf16-self": dict(name="multi-hot", B=203, rows=[4000, 321, 77, 5000, 1], dtype="bf16",
                                include_self=True),
    "d40-f16-padded": dict(name="multi-hot", B=77, rows=[300, 20, 999], d=40),
    "d256-f32": dict(name="capacity", B=65, rows=[2000] * 26, interaction=True, include_self=False),
    "T31": dict(name="multi-hot", B=45, rows=[700] * 31),
    "T40-self-d64": dict(name="one-hot", B=50, rows=[900] * 40, include_self=True),
    "T1": dict(name="multi-hot", B=99, rows=[1234]),
}


def _cfg(case):
    c = dict(CASES[case])
    return W.make_config(c.pop("name"), **c)


def _inputs(cfg):
    host = W.tables_host(cfg)
    tables = W.tables_to_device(host, cfg["dtype"])
    offsets, indices = W.make_indices(cfg)
    e0 = W.make_e0(cfg)
    return host, tables, offsets, indices, e0


def _run(cfg, tables, offsets, indices, e0, with_pooled, flag=None):
    B, T, d = cfg["B"], cfg["T"], cfg["d"]
    inc = cfg["include_self"]
    y = torch.full((B, d + sdi.dlrm_num_pairs(T, inc)), float("nan"), device=DEV)
    pooled = torch.full((B, T, d), float("nan"), device=DEV) if with_pooled else None
    sdi.dlrm_emb_bag_interact_fwd(tables, _t(offsets), _t(indices), B, _t(e0), inc, y, pooled=pooled,
                                  err_flag=flag)
    return y, pooled


@pytest.mark.parametrize("case", list(CASES))
def test_fused_forward_matches_oracle(case):
    cfg = _cfg(case)
    host, tables, offsets, indices, e0 = _inputs(cfg)
    B, T, d, inc = cfg["B"], cfg["T"], cfg["d"], cfg["include_self"]
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, pooled = _run(cfg, tables, offsets, indices, e0, True, flag)
    assert sdi.dlrm_read_error(flag) == 0
    p_ref, p_mag = oracle.emb_bag_fwd(host, cfg["dtype"], offsets, indices, B)
    y_ref, y_mag = oracle.interact_fwd(e0, p_ref, inc, emb_mag=p_mag)
    assert_close(y.cpu().numpy(), y_ref, y_mag, REL[cfg["dtype"]], f"fused y {case}")
    np.testing.assert_array_equal(y[:, :d].cpu().numpy(), e0)

    # the pooled vectors equal the standalone lookup's bit for bit
    alone = torch.full((B, T, d), float("nan"), device=DEV)
    sdi.dlrm_emb_bag_fwd(tables, _t(offsets), _t(indices), B, alone)
    np.testing.assert_array_equal(pooled.cpu().numpy().view(np.uint32), alone.cpu().numpy().view(np.uint32))

    # without the pooled output (the single kernel) y is within tolerance too
    y2, _ = _run(cfg, tables, offsets, indices, e0, False)
    assert_close(y2.cpu().numpy(), y_ref, y_mag, REL[cfg["dtype"]], f"fused y without pooled {case}")
    np.testing.assert_array_equal(y2[:, :d].cpu().numpy(), e0)

    # and within the tolerance of the unfused interaction
    y3 = torch.empty_like(y)
    sdi.dlrm_interact_fwd(_t(e0), alone, inc, y3)
    assert_close(y.cpu().numpy(), y3.cpu().numpy().astype(np.float64), y_mag, REL[cfg["dtype"]],
                 f"fused vs unfused {case}")
    assert_close(y2.cpu().numpy(), y3.cpu().numpy().astype(np.float64), y_mag, REL[cfg["dtype"]],
                 f"single kernel vs unfused {case}")


FALLBACK_CASES = {  # Z blocks too large for one CTA, or rows not of 16-byte chunks
    "heavy-bf16": dict(name="interaction-heavy", B=20, T=100, rows=[1000] * 100),
    "d17-f16": dict(name="multi-hot", B=30, rows=[100, 200, 300], d=17),
}


@pytest.mark.parametrize("case", list(FALLBACK_CASES))
def test_two_kernel_path_needs_and_fills_pooled(case):
    c = dict(FALLBACK_CASES[case])
    cfg = W.make_config(c.pop("name"), **c)
    host, tables, offsets, indices, e0 = _inputs(cfg)
    B, inc = cfg["B"], cfg["include_self"]
    with pytest.raises(sdi.DlrmError) as ei:
        _run(cfg, tables, offsets, indices, e0, False)
    assert ei.value.status == sdi._native.ERR_UNSUPPORTED
    y, pooled = _run(cfg, tables, offsets, indices, e0, True)
    p_ref, p_mag = oracle.emb_bag_fwd(host, cfg["dtype"], offsets, indices, B)
    assert_close(pooled.cpu().numpy(), p_ref, p_mag, REL[cfg["dtype"]], f"pooled {case}")
    y_ref, y_mag = oracle.interact_fwd(e0, p_ref, inc, emb_mag=p_mag)
    assert_close(y.cpu().numpy(), y_ref, y_mag, REL[cfg["dtype"]], f"y {case}")


def test_fused_empty_bags_and_out_of_range_index():
    # T = 2, B = 3: empty bags pool to zero; index 10 is out of range (skipped, flagged)
    host = [np.arange(10 * 16, dtype=np.float32).reshape(10, 16) / 64, np.ones((3, 16), np.float32)]
    offsets = np.array([0, 0, 2, 4, 4, 5, 5], dtype=np.int64)
    indices = np.array([0, 9, 10, 3, 2], dtype=np.int64)
    e0 = np.random.default_rng(5).standard_normal((3, 16)).astype(np.float32)
    tables = W.tables_to_device(host, "f32")
    y = torch.full((3, 16 + 3), float("nan"), device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    sdi.dlrm_emb_bag_interact_fwd(tables, _t(offsets), _t(indices), 3, _t(e0), False, y, err_flag=flag)
    assert sdi.dlrm_read_error(flag) == sdi._native.ERR_INDEX_OOB
    # an out-of-range lookup contributes nothing: the oracle gets the bags without it
    p_ref, p_mag = oracle.emb_bag_fwd(host, "f32", np.array([0, 0, 2, 3, 3, 4, 4]), np.array([0, 9, 3, 2]), 3)
    y_ref, y_mag = oracle.interact_fwd(e0, p_ref, False, emb_mag=p_mag)
    assert_close(y.cpu().numpy(), y_ref, y_mag, REL["f32"], "empty/oob")
    assert np.all(y.cpu().numpy()[0, 16:] == 0.0)  # sample 0: both bags empty, every product zero


@pytest.mark.parametrize("case", ["multi-hot-f16", "T40-self-d64", "tiny"])
def test_fused_alongside_matches_oracle(case):
    cfg = _cfg(case)
    host, tables, offsets, indices, e0 = _inputs(cfg)
    B, T, d, inc = cfg["B"], cfg["T"], cfg["d"], cfg["include_self"]
    width = sdi.dlrm_interact_width(T, d, inc, alongside=True)
    y = torch.full((B, width), float("nan"), device=DEV)
    sdi.dlrm_emb_bag_interact_fwd(tables, _t(offsets), _t(indices), B, _t(e0), inc, y, alongside=True)
    p_ref, p_mag = oracle.emb_bag_fwd(host, cfg["dtype"], offsets, indices, B)
    y_ref, y_mag = oracle.interact_fwd(e0, p_ref, inc, emb_mag=p_mag, alongside=True)
    assert_close(y.cpu().numpy(), y_ref, y_mag, REL[cfg["dtype"]], f"fused alongside {case}")
    # the copies are the pooled vectors of the standalone lookup, bit for bit
    alone = torch.empty((B, T, d), device=DEV)
    sdi.dlrm_emb_bag_fwd(tables, _t(offsets), _t(indices), B, alone)
    np.testing.assert_array_equal(y[:, d:d * (T + 1)].cpu().numpy().view(np.uint32),
                                  alone.reshape(B, T * d).cpu().numpy().view(np.uint32))
