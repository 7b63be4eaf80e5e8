"""GPU path vs the oracle at the full workload sizes (one-hot, multi-hot,
capacity, interaction-heavy), through the same calls and launch shapes that
bench.py times.

The oracle cannot recompute every output at these sizes, so it computes
sampled outputs one by one on sub-problems that restate the same arithmetic:
a bag's pooled vector needs only that bag's rows (regenerated on the host
from the counter-based table generator); a sample's interaction needs only its
own pooled vectors; a unique row's gradient needs only its own lookups.  The
integer results of the coalescing (sorted positions, unique keys, segment
offsets, count) are compared in full with the oracle's coalescing.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import workloads as W
from tests._parity import REL, assert_close, device_table_bits, device_table_f64, host_table_bits, table_f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()
    oracle.build()


@pytest.fixture(autouse=True)
def _free_device_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _sub_tables(cfg, rows_per_table):
    """Host tables restricted to the given rows of each table, renumbered in
    increasing order (the arithmetic on them is unchanged)."""
    tabs, maps = [], []
    for t, rows in enumerate(rows_per_table):
        uniq = np.unique(np.asarray(rows, dtype=np.int64))
        if uniq.size == 0:
            uniq = np.zeros(1, dtype=np.int64)
        tabs.append(W.table_rows_host(cfg, t, uniq))
        maps.append(uniq)
    return tabs, maps


def _oracle_pooled(cfg, offsets, indices, samples):
    """Oracle pooled vectors [len(samples)][T][d] of the given samples."""
    T, B = cfg["T"], cfg["B"]
    bags = [[indices[offsets[t * B + b]:offsets[t * B + b + 1]] for b in samples] for t in range(T)]
    tabs, maps = _sub_tables(cfg, [np.concatenate(bt) if bt else [] for bt in bags])
    sub_off = [0]
    sub_idx = []
    for t in range(T):
        for bag in bags[t]:
            sub_idx.append(np.searchsorted(maps[t], bag))
            sub_off.append(sub_off[-1] + bag.size)
    return oracle.emb_bag_fwd(tabs, cfg["dtype"], np.array(sub_off), np.concatenate(sub_idx), len(samples))


def _chosen_samples(cfg, offsets, n=8, seed=0):
    """First and last samples, the sample with the longest bag, and random ones."""
    B, T = cfg["B"], cfg["T"]
    lengths = np.diff(offsets).reshape(T, B).sum(axis=0)
    rng = np.random.default_rng(seed)
    pick = {0, B - 1, int(np.argmax(lengths))} | set(rng.integers(0, B, n).tolist())
    return np.array(sorted(pick), dtype=np.int64)


def _run_forward_chain(cfg, tables, offsets, indices):
    B, T, d, inc = cfg["B"], cfg["T"], cfg["d"], cfg["include_self"]
    off_t = torch.from_numpy(offsets).to(DEV)
    idx_t = torch.from_numpy(indices).to(DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    pooled = torch.empty((B, T, d), device=DEV)
    sdi.dlrm_emb_bag_fwd(tables, off_t, idx_t, B, pooled, err_flag=flag)
    out = dict(pooled=pooled, off_t=off_t, idx_t=idx_t, flag=flag)
    if cfg["interaction"]:
        e0 = torch.from_numpy(W.make_e0(cfg)).to(DEV)
        dy = torch.from_numpy(W.make_dy(cfg)).to(DEV)
        y = torch.empty((B, d + sdi.dlrm_num_pairs(T, inc)), device=DEV)
        de0 = torch.empty((B, d), device=DEV)
        dpooled = torch.empty((B, T, d), device=DEV)
        sdi.dlrm_interact_fwd(e0, pooled, inc, y)
        sdi.dlrm_interact_bwd(e0, pooled, inc, dy, de0, dpooled)
        out.update(y=y, de0=de0, dpooled=dpooled)
    assert sdi.dlrm_read_error(flag) == 0
    return out


def _check_forward_chain(cfg, offsets, indices, res):
    rel = REL[cfg["dtype"]]
    samples = _chosen_samples(cfg, offsets)
    p_ref, p_mag = _oracle_pooled(cfg, offsets, indices, samples)
    sel = torch.from_numpy(samples).to(DEV)
    assert_close(res["pooled"][sel].cpu().numpy(), p_ref, p_mag, rel, f"{cfg['name']} pooled")
    if not cfg["interaction"]:
        return
    inc = cfg["include_self"]
    e0 = W.make_e0(cfg)[samples]
    dy = W.make_dy(cfg)[samples]
    y_ref, y_mag = oracle.interact_fwd(e0, p_ref, inc, emb_mag=p_mag)
    assert_close(res["y"][sel].cpu().numpy(), y_ref, y_mag, rel, f"{cfg['name']} interaction")
    de0_ref, de0_mag, dp_ref, dp_mag = oracle.interact_bwd(e0, p_ref, dy, inc, emb_mag=p_mag)
    assert_close(res["de0"][sel].cpu().numpy(), de0_ref, de0_mag, rel, f"{cfg['name']} de0")
    assert_close(res["dpooled"][sel].cpu().numpy(), dp_ref, dp_mag, rel, f"{cfg['name']} dpooled")


def _check_backward(cfg, tables, offsets, indices, off_t, idx_t):
    """Backward + update with a generated pooled gradient (not from the
    chain, so every oracle input comes from the generator)."""
    B, T, d = cfg["B"], cfg["T"], cfg["d"]
    nnz = indices.size
    dp_host = W.make_dpooled(cfg)
    dp = torch.from_numpy(dp_host).to(DEV)
    lr = cfg["lr"]
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(T, B, nnz, d), dtype=torch.uint8, device=DEV)
    grad = torch.empty((nnz, d), device=DEV) if cfg["update"] == "grad" else None
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    view = sdi.dlrm_emb_bag_bwd_sgd(tables, off_t, idx_t, B, dp, lr, ws, grad_rows=grad, err_flag=flag,
                                    want_view=True)
    assert sdi.dlrm_read_error(flag) == 0

    # integer results, in full
    co = oracle.coalesce(cfg["rows"], offsets, indices, B)
    U = int(view["num_unique"].item())
    assert U == co["U"]
    u32 = lambda t, n: t[:n].cpu().numpy().view(np.uint32).astype(np.int64)
    np.testing.assert_array_equal(u32(view["sorted_pos"], nnz), co["sorted_pos"])
    np.testing.assert_array_equal(u32(view["uniq_row"], U), co["uniq_row"])
    np.testing.assert_array_equal(view["uniq_table"][:U].cpu().numpy(), co["uniq_table"])
    np.testing.assert_array_equal(u32(view["seg_off"], U + 1), co["seg_off"])

    # sampled unique rows: the longest runs and random ones
    lengths = np.diff(co["seg_off"])
    rng = np.random.default_rng(1)
    us = np.unique(np.concatenate([np.argsort(lengths)[-12:], rng.integers(0, U, 96)]))
    starts, ends = co["seg_off"][us], co["seg_off"][us + 1]
    sub_co = dict(U=us.size, uniq_table=co["uniq_table"][us], uniq_row=co["uniq_row"][us],
                  sorted_pos=np.concatenate([co["sorted_pos"][a:b] for a, b in zip(starts, ends)]),
                  seg_off=np.concatenate([[0], np.cumsum(ends - starts)]))
    rows_per_table = [sub_co["uniq_row"][sub_co["uniq_table"] == t] for t in range(T)]
    tabs, maps = _sub_tables(cfg, rows_per_table)
    sub_co["uniq_row"] = np.array([np.searchsorted(maps[t], r) for t, r in
                                   zip(sub_co["uniq_table"], sub_co["uniq_row"])], dtype=np.int64)
    g_ref, g_mag, w_ref, w_mag = oracle.sgd(tabs, cfg["dtype"], offsets, B, nnz, dp_host.astype(np.float64),
                                            lr, sub_co)
    rel = REL[cfg["dtype"]]
    if grad is not None:
        assert_close(grad[torch.from_numpy(us).to(DEV)].cpu().numpy(), g_ref, g_mag, rel,
                     f"{cfg['name']} row gradients")
    got_rows = np.stack([device_table_f64(tables[int(t)][int(r):int(r) + 1], cfg["dtype"])[0]
                         for t, r in zip(co["uniq_table"][us], co["uniq_row"][us])])
    assert_close(got_rows, w_ref, w_mag, rel, f"{cfg['name']} updated rows", table_dtype=cfg["dtype"])

    # rows no lookup touched keep their bits
    touched = set(zip(co["uniq_table"].tolist(), co["uniq_row"].tolist()))
    for t in rng.choice(T, size=min(T, 4), replace=False):
        cand = rng.integers(0, cfg["rows"][t], 64)
        cand = np.array([r for r in cand if (int(t), int(r)) not in touched][:16], dtype=np.int64)
        if cand.size == 0:
            continue
        got = device_table_bits(tables[t][torch.from_numpy(cand).to(DEV)])
        np.testing.assert_array_equal(got, host_table_bits(W.table_rows_host(cfg, int(t), cand), cfg["dtype"]))


@pytest.mark.parametrize("name", ["one-hot", "multi-hot", "interaction-heavy", "capacity"])
def test_full_size_step_matches_oracle(name):
    cfg = W.make_config(name)
    need = W.table_bytes(cfg) * 1.2 + 4e9
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory, {free / 1e9:.0f} GB free")
    offsets, indices = W.make_indices(cfg)
    tables = W.make_tables_device(cfg)
    res = _run_forward_chain(cfg, tables, offsets, indices)
    _check_forward_chain(cfg, offsets, indices, res)
    off_t, idx_t = res["off_t"], res["idx_t"]
    del res
    _check_backward(cfg, tables, offsets, indices, off_t, idx_t)


def _need(cfg, extra=0.0):
    need = W.table_bytes(cfg) * 1.2 + 4e9 + extra
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory, {free / 1e9:.0f} GB free")


def test_full_size_fused_forward_multi_hot():
    cfg = W.make_config("multi-hot")
    _need(cfg)
    B, T, d, inc = cfg["B"], cfg["T"], cfg["d"], cfg["include_self"]
    offsets, indices = W.make_indices(cfg)
    tables = W.make_tables_device(cfg)
    e0 = W.make_e0(cfg)
    y = torch.empty((B, sdi.dlrm_interact_width(T, d, inc)), device=DEV)
    pooled = torch.empty((B, T, d), device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    sdi.dlrm_emb_bag_interact_fwd(tables, torch.from_numpy(offsets).to(DEV), torch.from_numpy(indices).to(DEV), B,
                                  torch.from_numpy(e0).to(DEV), inc, y, pooled=pooled, err_flag=flag)
    assert sdi.dlrm_read_error(flag) == 0
    samples = _chosen_samples(cfg, offsets)
    p_ref, p_mag = _oracle_pooled(cfg, offsets, indices, samples)
    sel = torch.from_numpy(samples).to(DEV)
    rel = REL[cfg["dtype"]]
    assert_close(pooled[sel].cpu().numpy(), p_ref, p_mag, rel, "fused pooled")
    y_ref, y_mag = oracle.interact_fwd(e0[samples], p_ref, inc, emb_mag=p_mag)
    assert_close(y[sel].cpu().numpy(), y_ref, y_mag, rel, "fused y")


def test_full_size_adagrad_multi_hot():
    cfg = W.make_config("multi-hot")
    _need(cfg, extra=0.5e9)
    B, T, d = cfg["B"], cfg["T"], cfg["d"]
    offsets, indices = W.make_indices(cfg)
    tables = W.make_tables_device(cfg)
    nnz = indices.size
    dp_host = W.make_dpooled(cfg)
    rng = np.random.default_rng(5)
    state = [torch.from_numpy(rng.uniform(0.01, 2.0, r).astype(np.float32)).to(DEV) for r in cfg["rows"]]
    state0 = [s.clone() for s in state]
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(T, B, nnz, d), dtype=torch.uint8, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    lr, eps = 0.05, 1e-6
    view = sdi.dlrm_emb_bag_bwd_adagrad(tables, state, torch.from_numpy(offsets).to(DEV),
                                        torch.from_numpy(indices).to(DEV), B, torch.from_numpy(dp_host).to(DEV), lr,
                                        eps, ws, err_flag=flag, want_view=True)
    assert sdi.dlrm_read_error(flag) == 0
    co = oracle.coalesce(cfg["rows"], offsets, indices, B)
    assert int(view["num_unique"].item()) == co["U"]
    # sampled unique rows: the longest runs and random ones, as a sub-problem
    lengths = np.diff(co["seg_off"])
    us = np.unique(np.concatenate([np.argsort(lengths)[-12:], rng.integers(0, co["U"], 96)]))
    starts, ends = co["seg_off"][us], co["seg_off"][us + 1]
    sub = dict(U=us.size, uniq_table=co["uniq_table"][us], uniq_row=co["uniq_row"][us],
               sorted_pos=np.concatenate([co["sorted_pos"][a:b] for a, b in zip(starts, ends)]),
               seg_off=np.concatenate([[0], np.cumsum(ends - starts)]))
    tabs, maps = _sub_tables(cfg, [sub["uniq_row"][sub["uniq_table"] == t] for t in range(T)])
    s_in = np.array([state0[int(t)][int(r)].item() for t, r in zip(sub["uniq_table"], sub["uniq_row"])])
    sub["uniq_row"] = np.array([np.searchsorted(maps[t], r) for t, r in zip(sub["uniq_table"], sub["uniq_row"])],
                               dtype=np.int64)
    _, _, s_ref, s_mag, w_ref, w_mag = oracle.adagrad(tabs, cfg["dtype"], offsets, B, nnz, dp_host.astype(np.float64),
                                                      lr, eps, s_in, sub)
    got_s = np.array([state[int(t)][int(r)].item() for t, r in zip(co["uniq_table"][us], co["uniq_row"][us])])
    assert_close(got_s, s_ref, s_mag, REL["f32"], "accumulators")
    got_w = np.stack([device_table_f64(tables[int(t)][int(r):int(r) + 1], cfg["dtype"])[0]
                      for t, r in zip(co["uniq_table"][us], co["uniq_row"][us])])
    assert_close(got_w, w_ref, w_mag, REL[cfg["dtype"]], "updated rows", table_dtype=cfg["dtype"])


def test_full_size_int4_capacity():
    cfg = W.make_config("capacity")
    _need(cfg, extra=W.table_bytes(cfg) / 6)
    B, T, d = cfg["B"], cfg["T"], cfg["d"]
    offsets, indices = W.make_indices(cfg)
    tables = W.make_tables_device(cfg)
    q = [sdi.dlrm_quantize_int4(t) for t in tables]
    del tables
    gc.collect()
    torch.cuda.empty_cache()
    out = torch.empty((B, T, d), device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    sdi.dlrm_emb_bag_fwd(q, torch.from_numpy(offsets).to(DEV), torch.from_numpy(indices).to(DEV), B, out,
                         err_flag=flag, d=d)
    assert sdi.dlrm_read_error(flag) == 0
    samples = _chosen_samples(cfg, offsets)
    bags = [[indices[offsets[t * B + b]:offsets[t * B + b + 1]] for b in samples] for t in range(T)]
    tabs, maps = _sub_tables(cfg, [np.concatenate(bt) for bt in bags])
    # the device's codes of the touched rows are the oracle's encoding of the generated rows
    qsub = []
    for t in range(T):
        qt = oracle.quantize_int4(tabs[t], cfg["dtype"])
        got = q[t][torch.from_numpy(maps[t]).to(DEV)].cpu().numpy()
        np.testing.assert_array_equal(got, qt)
        qsub.append(qt)
    sub_off, sub_idx = [0], []
    for t in range(T):
        for bag in bags[t]:
            sub_idx.append(np.searchsorted(maps[t], bag))
            sub_off.append(sub_off[-1] + bag.size)
    ref, mag = oracle.emb_bag_fwd(qsub, "int4", np.array(sub_off), np.concatenate(sub_idx), len(samples), d=d)
    assert_close(out[torch.from_numpy(samples).to(DEV)].cpu().numpy(), ref, mag, REL["f32"], "int4 pooled")
