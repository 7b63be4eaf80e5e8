"""Row-wise AdaGrad (dlrm_emb_bag_bwd_adagrad, dlrm_emb_bag_reduce_adagrad)
vs the oracle.

The accumulators and the updated rows must lie within rel x magnitude of the
oracle's fp64 values (the magnitudes carry the gradient's rounding bound
through the squares and the square root to first order); the coalesced
gradient as for SGD; rows and accumulators no lookup touched keep their bits.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import workloads as W
from tests._parity import REL, assert_close, device_table_bits, device_table_f64, host_table_bits

pytestmark = pytest.mark.gpu

DEV = "cuda"
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()
    oracle.build()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


CASES = {  # (config, initial accumulators)
    "tiny-zero-state": (dict(name="tiny"), "zero"),
    "multi-hot-f16": (dict(name="multi-hot", B=1000, rows=[5000, 70000, 123, 9]), "random"),
    "multi-hot-bf16": (dict(name="multi-hot", B=700, rows=[4000, 321], dtype="bf16"), "zero"),
    "capacity-f32": (dict(name="capacity", B=400, rows=[20000, 30000, 77]), "random"),
    "heavy-bf16-d256": (dict(name="interaction-heavy", B=500, T=4, rows=[1000] * 4), "random"),
    "d200-f32": (dict(name="tiny", B=300, rows=[300, 20], d=200), "zero"),
    "d17-f16-scalar": (dict(name="multi-hot", B=300, rows=[100, 200], d=17), "random"),
    "d64-f32": (dict(name="one-hot", B=1500, rows=[10, 17, 30, 52, 91, 5000, 100000]), "zero"),
}


def _state0(cfg, kind, seed=3):
    rng = np.random.default_rng([seed, cfg["id"]])
    if kind == "zero":
        return [np.zeros(r, dtype=np.float32) for r in cfg["rows"]]
    return [rng.uniform(0.01, 2.0, r).astype(np.float32) for r in cfg["rows"]]


def _check(cfg, host, s0, offsets, indices, dp, lr, tables, state, grad, view, what):
    nnz, B, T = indices.size, cfg["B"], cfg["T"]
    co = oracle.coalesce(cfg["rows"], offsets, indices, B)
    U = co["U"]
    assert int(view["num_unique"].item()) == U
    s_in = np.array([s0[int(t)][int(r)] for t, r in zip(co["uniq_table"], co["uniq_row"])], dtype=np.float64)
    g_ref, g_mag, s_ref, s_mag, w_ref, w_mag = oracle.adagrad(host, cfg["dtype"], offsets, B, nnz, dp, lr, EPS,
                                                              s_in, co)
    rel = REL[cfg["dtype"]]
    assert_close(grad.cpu().numpy()[:U], g_ref, g_mag, rel, f"gradient {what}")
    by_t = {}
    for u in range(U):
        by_t.setdefault(int(co["uniq_table"][u]), []).append(u)
    for t in range(T):
        us = by_t.get(t, [])
        rows_t = co["uniq_row"][us]
        st = state[t].cpu().numpy()
        assert_close(st[rows_t].astype(np.float64), s_ref[us], s_mag[us], REL["f32"], f"accumulators {what} t={t}")
        dev = device_table_f64(tables[t], cfg["dtype"])
        assert_close(dev[rows_t], w_ref[us], w_mag[us], rel, f"rows {what} t={t}", table_dtype=cfg["dtype"])
        untouched = np.ones(cfg["rows"][t], dtype=bool)
        untouched[rows_t] = False
        np.testing.assert_array_equal(st[untouched].view(np.uint32), s0[t][untouched].view(np.uint32))
        np.testing.assert_array_equal(device_table_bits(tables[t])[untouched],
                                      host_table_bits(host[t], cfg["dtype"])[untouched])


@pytest.mark.parametrize("case", list(CASES))
def test_adagrad_matches_oracle(case):
    c, kind = CASES[case]
    c = dict(c)
    cfg = W.make_config(c.pop("name"), **c)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = W.make_dpooled(cfg)
    s0 = _state0(cfg, kind)
    lr, nnz = 0.05, indices.size
    tables = W.tables_to_device(host, cfg["dtype"])
    state = [_t(s) for s in s0]
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(cfg["T"], cfg["B"], nnz, cfg["d"]), dtype=torch.uint8,
                     device=DEV)
    grad = torch.full((nnz, cfg["d"]), float("nan"), device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    view = sdi.dlrm_emb_bag_bwd_adagrad(tables, state, _t(offsets), _t(indices), cfg["B"], _t(dp), lr, EPS, ws,
                                        grad_rows=grad, err_flag=flag, want_view=True)
    assert sdi.dlrm_read_error(flag) == 0
    _check(cfg, host, s0, offsets, indices, dp, lr, tables, state, grad, view, case)


@pytest.mark.parametrize("case", list(CASES))
def test_adagrad_without_a_view_gives_the_same_bits(case):
    # the sort carries bags instead of positions when no view is asked for; the sums, the
    # accumulators and the rows must equal those of the view path bit for bit
    c, kind = CASES[case]
    c = dict(c)
    cfg = W.make_config(c.pop("name"), **c)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = _t(W.make_dpooled(cfg))
    s0 = _state0(cfg, kind)
    nnz = indices.size
    out = []
    for want_view in (True, False):
        tables = W.tables_to_device(host, cfg["dtype"])
        state = [_t(s) for s in s0]
        ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(cfg["T"], cfg["B"], nnz, cfg["d"]),
                         dtype=torch.uint8, device=DEV)
        grad = torch.full((nnz, cfg["d"]), float("nan"), device=DEV)
        sdi.dlrm_emb_bag_bwd_adagrad(tables, state, _t(offsets), _t(indices), cfg["B"], dp, 0.05, EPS, ws,
                                     grad_rows=grad, want_view=want_view)
        out.append((tables, state, grad))
    (t1, s1, g1), (t2, s2, g2) = out
    np.testing.assert_array_equal(g2.cpu().numpy().view(np.uint32), g1.cpu().numpy().view(np.uint32))
    for t in range(cfg["T"]):
        np.testing.assert_array_equal(device_table_bits(t2[t]), device_table_bits(t1[t]))
        np.testing.assert_array_equal(s2[t].cpu().numpy().view(np.uint32), s1[t].cpu().numpy().view(np.uint32))


def test_adagrad_long_runs_cross_chunks():
    # almost every lookup of table 0 hits row 7: one run over many reduce
    # chunks and sort tiles, combined by the finalize (which applies AdaGrad)
    B = 3000
    rng = np.random.default_rng(12)
    bags0 = [[7] * int(rng.integers(0, 9)) for _ in range(B)]
    bags0[5] = [7, 3, 7]
    bags1 = [list(rng.integers(0, 50, int(rng.integers(0, 6)))) for _ in range(B)]
    idx, offsets = [], [0]
    for bags in (bags0, bags1):
        for bag in bags:
            idx += bag
            offsets.append(len(idx))
    offsets, indices = np.array(offsets, dtype=np.int64), np.array(idx, dtype=np.int64)
    cfg = W.make_config("multi-hot", B=B, rows=[10, 50], dtype="f32")
    host = W.tables_host(cfg)
    dp = np.random.default_rng(13).standard_normal((B, 2, cfg["d"])).astype(np.float32)
    s0 = _state0(cfg, "random")
    tables = W.tables_to_device(host, "f32")
    state = [_t(s) for s in s0]
    nnz = indices.size
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(2, B, nnz, cfg["d"]), dtype=torch.uint8, device=DEV)
    grad = torch.full((nnz, cfg["d"]), float("nan"), device=DEV)
    view = sdi.dlrm_emb_bag_bwd_adagrad(tables, state, _t(offsets), _t(indices), B, _t(dp), 0.01, EPS, ws,
                                        grad_rows=grad, want_view=True)
    _check(cfg, host, s0, offsets, indices, dp, 0.01, tables, state, grad, view, "long runs")


def test_adagrad_split_halves_equal_the_single_call():
    cfg = W.make_config("multi-hot", B=900, rows=[3000, 40000, 50])
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = _t(W.make_dpooled(cfg))
    s0 = _state0(cfg, "random")
    nnz, B, T, d = indices.size, cfg["B"], cfg["T"], cfg["d"]
    off_t, idx_t = _t(offsets), _t(indices)
    ws_bytes = sdi.dlrm_emb_bag_bwd_workspace_size(T, B, nnz, d)
    outs = []
    for split in (False, True):
        tables = W.tables_to_device(host, cfg["dtype"])
        state = [_t(s) for s in s0]
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
        if split:
            sdi.dlrm_emb_bag_coalesce(cfg["rows"], d, off_t, idx_t, B, ws)
            sdi.dlrm_emb_bag_reduce_adagrad(tables, state, nnz, B, dp, 0.02, EPS, ws)
        else:
            sdi.dlrm_emb_bag_bwd_adagrad(tables, state, off_t, idx_t, B, dp, 0.02, EPS, ws)
        outs.append(([device_table_bits(t) for t in tables], [s.cpu().numpy().view(np.uint32) for s in state]))
    for a, b in zip(outs[0][0] + outs[0][1], outs[1][0] + outs[1][1]):
        np.testing.assert_array_equal(a, b)


def test_adagrad_zero_rate_changes_nothing_but_the_gradient():
    cfg = W.make_config("tiny", B=64)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    s0 = _state0(cfg, "random")
    tables = W.tables_to_device(host, "f32")
    state = [_t(s) for s in s0]
    nnz = indices.size
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(cfg["T"], 64, nnz, cfg["d"]), dtype=torch.uint8,
                     device=DEV)
    grad = torch.zeros((nnz, cfg["d"]), device=DEV)
    sdi.dlrm_emb_bag_bwd_adagrad(tables, state, _t(offsets), _t(indices), 64, _t(W.make_dpooled(cfg)), 0.0, EPS, ws,
                                 grad_rows=grad)
    for t in range(cfg["T"]):
        np.testing.assert_array_equal(state[t].cpu().numpy(), s0[t])
        np.testing.assert_array_equal(device_table_bits(tables[t]), host_table_bits(host[t], "f32"))
    assert torch.count_nonzero(grad) > 0


def test_adagrad_rejects_wide_rows_and_bad_eps():
    cfg = W.make_config("tiny", B=8, d=260)
    tables = W.tables_to_device(W.tables_host(cfg), "f32")
    state = [torch.zeros(r, device=DEV) for r in cfg["rows"]]
    offsets, indices = W.make_indices(cfg)
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(cfg["T"], 8, indices.size, 260), dtype=torch.uint8,
                     device=DEV)
    dp = torch.zeros(8, cfg["T"], 260, device=DEV)
    with pytest.raises(sdi.DlrmError) as ei:
        sdi.dlrm_emb_bag_bwd_adagrad(tables, state, _t(offsets), _t(indices), 8, dp, 0.1, EPS, ws)
    assert ei.value.status == sdi._native.ERR_UNSUPPORTED
    cfg = W.make_config("tiny", B=8)
    tables = W.tables_to_device(W.tables_host(cfg), "f32")
    dp = torch.zeros(8, cfg["T"], cfg["d"], device=DEV)
    for eps in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(sdi.DlrmError) as ei:
            sdi.dlrm_emb_bag_bwd_adagrad(tables, state, _t(offsets), _t(indices), 8, dp, 0.1, eps, ws)
        assert ei.value.status == sdi._native.ERR_INVALID_ARG
