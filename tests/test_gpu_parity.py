"""GPU path vs the oracle, element by element, on seeded inputs.

Sizes are small enough for the oracle to finish in seconds but span several
CTAs, sort tiles (4096 lookups) and reduce chunks (512 lookups), with ragged
tails.  Integer results of the coalescing must match bit for bit; float
results must lie within rel x magnitude of the oracle (rel 1e-5 for fp32
tables, 2e-3 for fp16/bf16 tables), where the magnitude is the oracle's
bound on the rounding error of any summation order.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import workloads as W
from tests._parity import (REL, assert_close, device_table_bits, device_table_f64,
                           host_table_bits, table_f64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()
    oracle.build()


def _t(a, dtype=None):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV) if dtype is None else \
        torch.from_numpy(np.ascontiguousarray(a)).to(DEV, dtype)


def _flag():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _u32(t):
    return t.cpu().numpy().view(np.uint32).astype(np.int64)


# --------------------------------------------------------------- forward ---

FWD_CASES = {
    "tiny": dict(name="tiny"),
    "one-hot": dict(name="one-hot", B=300, rows=[10, 17, 30, 52, 91, 5000, 100000]),
    "multi-hot-f16": dict(name="multi-hot", B=300, rows=[5000, 70000, 123, 9]),
    "multi-hot-bf16": dict(name="multi-hot", B=200, rows=[4000, 321], dtype="bf16"),
    "capacity-f32": dict(name="capacity", B=100, rows=[20000, 30000, 77]),
    "heavy-bf16": dict(name="interaction-heavy", B=96, T=5, rows=[1000] * 5),
    "d17-scalar": dict(name="multi-hot", B=64, rows=[100, 200], d=17),
    "d3-f32-scalar": dict(name="tiny", B=64, rows=[40, 50, 60], d=3),
    "d512-f32": dict(name="tiny", B=40, rows=[300, 20], d=512),
    "d8-f16": dict(name="multi-hot", B=50, rows=[300, 20], d=8),
    # half rows of 12 and 10 chunks (8 lanes of two chunks, some idle) and of 9 (16 lanes)
    "d96-f16": dict(name="multi-hot", B=120, rows=[3000, 70], d=96),
    "d80-bf16": dict(name="multi-hot", B=120, rows=[3000, 70], d=80, dtype="bf16"),
    "d72-f16": dict(name="multi-hot", B=120, rows=[3000, 70], d=72),
}


def _cfg(case):
    c = dict(FWD_CASES[case])
    return W.make_config(c.pop("name"), **c)


@pytest.mark.parametrize("case", list(FWD_CASES))
def test_emb_bag_fwd_matches_oracle(case):
    cfg = _cfg(case)
    host = W.tables_host(cfg)
    tables = W.tables_to_device(host, cfg["dtype"])
    offsets, indices = W.make_indices(cfg)
    B, T, d = cfg["B"], cfg["T"], cfg["d"]
    out = torch.full((B, T, d), float("nan"), device=DEV)
    flag = _flag()
    sdi.dlrm_emb_bag_fwd(tables, _t(offsets), _t(indices), B, out, err_flag=flag)
    assert sdi.dlrm_read_error(flag) == 0
    ref, mag = oracle.emb_bag_fwd(host, cfg["dtype"], offsets, indices, B)
    assert_close(out.cpu().numpy(), ref, mag, REL[cfg["dtype"]], f"pooled {case}")
    if cfg["bag"] == ("fixed", 1):  # pooling factor one: a bit-exact row copy
        np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), ref)


def test_emb_bag_fwd_writes_into_a_strided_buffer():
    # the pooled rows land inside a wider [B][T+1][d] block (row 0 left alone)
    cfg = W.make_config("multi-hot", B=100, rows=[500, 600, 700])
    host = W.tables_host(cfg)
    tables = W.tables_to_device(host, "f16")
    offsets, indices = W.make_indices(cfg)
    Z = torch.full((100, 4, 128), -7.0, device=DEV)
    sdi.dlrm_emb_bag_fwd(tables, _t(offsets), _t(indices), 100, Z[:, 1:, :])
    ref, mag = oracle.emb_bag_fwd(host, "f16", offsets, indices, 100)
    assert_close(Z[:, 1:].cpu().numpy(), ref, mag, REL["f16"], "strided pooled")
    assert torch.all(Z[:, 0] == -7.0)


def test_emb_bag_fwd_empty_bags_and_bounds():
    # empty bags pool to zero; first and last rows are reachable
    rows = [64, 3]
    host = [np.arange(64 * 8, dtype=np.float32).reshape(64, 8), np.ones((3, 8), np.float32)]
    offsets = np.array([0, 0, 2, 2, 2, 5, 5], dtype=np.int64)  # T=2, B=3
    indices = np.array([0, 63, 2, 0, 2], dtype=np.int64)
    out = torch.full((3, 2, 8), float("nan"), device=DEV)
    sdi.dlrm_emb_bag_fwd(W.tables_to_device(host, "f32"), _t(offsets), _t(indices), 3, out)
    ref, _ = oracle.emb_bag_fwd(host, "f32", offsets, indices, 3)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)


def test_emb_bag_fwd_out_of_range_index_is_flagged_and_skipped():
    host = [np.ones((10, 8), np.float32) * 2]
    offsets = np.array([0, 3, 4], dtype=np.int64)
    indices = np.array([1, 10, 3, -1], dtype=np.int64)
    out = torch.zeros((2, 1, 8), device=DEV)
    flag = _flag()
    sdi.dlrm_emb_bag_fwd(W.tables_to_device(host, "f32"), _t(offsets), _t(indices), 2, out, err_flag=flag)
    assert sdi.dlrm_read_error(flag) == sdi._native.ERR_INDEX_OOB
    np.testing.assert_array_equal(out.cpu().numpy()[0, 0], 4.0)  # rows 1 and 3 only
    np.testing.assert_array_equal(out.cpu().numpy()[1, 0], 0.0)


def test_emb_bag_fwd_bad_offsets_are_flagged():
    host = [np.ones((10, 8), np.float32)]
    offsets = np.array([0, 3, 1, 9], dtype=np.int64)  # decreasing, and past nnz = 4
    indices = np.array([1, 2, 3, 4], dtype=np.int64)
    out = torch.zeros((3, 1, 8), device=DEV)
    flag = _flag()
    sdi.dlrm_emb_bag_fwd(W.tables_to_device(host, "f32"), _t(offsets), _t(indices), 3, out, err_flag=flag)
    assert sdi.dlrm_read_error(flag) == sdi._native.ERR_BAD_OFFSETS


# ----------------------------------------------------------- interaction ---

INTER_CASES = [  # (B, N, d, include_self)
    (300, 26, 128, False), (301, 26, 64, False), (128, 8, 16, False), (37, 100, 256, True),
    (40, 127, 32, True), (50, 0, 16, False), (50, 0, 16, True), (33, 1, 8, True),
    (65, 5, 3, False), (21, 13, 33, True), (1, 26, 128, False),
    # 64-row and 128-row sample blocks of the tensor-core kernel, a last chunk of 8 columns
    (77, 40, 64, False), (19, 63, 40, True), (23, 64, 96, False),
    # more tiles than SMs: the persistent loop wraps its staging ring and both accumulators
    (5001, 26, 128, False), (700, 100, 256, True),
    # enough units for the tensor-core backward: 16-row Gs, two d tiles, a ragged d tile, and
    # two and three chunks of 32 vectors
    (5000, 13, 64, True), (4900, 31, 256, False), (2500, 20, 200, True), (4900, 40, 64, False),
    (4900, 70, 64, True),
    # two chunks of vectors over two d tiles, the second ragged (a sample's tiles share its Gs)
    (2500, 45, 200, True),
    # a last chunk of 21 and of 20 vectors (its last 16-byte column group half padding)
    (4900, 52, 64, False), (4900, 83, 64, True),
]

KERNELS = {"auto": sdi.INTERACT_KERNEL_AUTO, "cuda-core": sdi.INTERACT_KERNEL_CUDA_CORE}


@pytest.fixture(params=list(KERNELS))
def kernel(request):
    """Runs the test with the interaction kernels of each family."""
    sdi.dlrm_set_interact_kernel(KERNELS[request.param])
    yield request.param
    sdi.dlrm_set_interact_kernel(sdi.INTERACT_KERNEL_AUTO)


def _inter_inputs(B, N, d, inc, seed=0):
    rng = np.random.default_rng([seed, B, N, d, inc])
    e0 = rng.standard_normal((B, d), dtype=np.float32)
    emb = rng.standard_normal((B, N, d), dtype=np.float32)
    dy = rng.standard_normal((B, d + oracle.num_pairs(N, inc)), dtype=np.float32)
    return e0, emb, dy


@pytest.mark.parametrize("B,N,d,inc", INTER_CASES)
def test_interact_fwd_matches_oracle(B, N, d, inc, kernel):
    e0, emb, _ = _inter_inputs(B, N, d, inc)
    width = d + sdi.dlrm_num_pairs(N, inc)
    y = torch.full((B, width), float("nan"), device=DEV)
    sdi.dlrm_interact_fwd(_t(e0), _t(emb).reshape(B, N, d) if N else torch.empty((B, 0, d), device=DEV),
                          inc, y)
    ref, mag = oracle.interact_fwd(e0, emb, inc)
    got = y.cpu().numpy()
    np.testing.assert_array_equal(got[:, :d], e0)  # the concatenated e0 is a copy
    assert_close(got, ref, mag, REL["f32"], f"interaction fwd B={B} N={N} d={d} inc={inc}")


@pytest.mark.parametrize("B,N,d,inc", INTER_CASES)
def test_interact_bwd_matches_oracle(B, N, d, inc, kernel):
    e0, emb, dy = _inter_inputs(B, N, d, inc)
    de0 = torch.full((B, d), float("nan"), device=DEV)
    demb = torch.full((B, N, d), float("nan"), device=DEV)
    emb_t = _t(emb) if N else torch.empty((B, 0, d), device=DEV)
    sdi.dlrm_interact_bwd(_t(e0), emb_t, inc, _t(dy), de0, demb)
    r_de0, m_de0, r_demb, m_demb = oracle.interact_bwd(e0, emb, dy, inc)
    assert_close(de0.cpu().numpy(), r_de0, m_de0, REL["f32"], "de0")
    assert_close(demb.cpu().numpy(), r_demb, m_demb, REL["f32"], "demb")


@pytest.mark.parametrize("B,N,d,inc", [(4870, 127, 64, True), (2440, 100, 256, True), (4870, 64, 128, False)])
def test_interact_many_vectors_sampled(B, N, d, inc, kernel):
    # 65 to 128 vectors per sample (four chunks of 32 in the tensor-core backward), against the
    # oracle on sampled samples (first, last and a stride through the middle)
    e0, emb, dy = _inter_inputs(B, N, d, inc, seed=4)
    y = torch.full((B, d + sdi.dlrm_num_pairs(N, inc)), float("nan"), device=DEV)
    sdi.dlrm_interact_fwd(_t(e0), _t(emb), inc, y)
    de0 = torch.full((B, d), float("nan"), device=DEV)
    demb = torch.full((B, N, d), float("nan"), device=DEV)
    sdi.dlrm_interact_bwd(_t(e0), _t(emb), inc, _t(dy), de0, demb)
    rows = np.unique(np.r_[0:24, B - 24:B, 0:B:97])
    ref, mag = oracle.interact_fwd(e0[rows], emb[rows], inc)
    assert_close(y.cpu().numpy()[rows], ref, mag, REL["f32"], f"fwd B={B} N={N} d={d}")
    r_de0, m_de0, r_demb, m_demb = oracle.interact_bwd(e0[rows], emb[rows], dy[rows], inc)
    assert_close(de0.cpu().numpy()[rows], r_de0, m_de0, REL["f32"], "de0")
    assert_close(demb.cpu().numpy()[rows], r_demb, m_demb, REL["f32"], "demb")


def test_interact_with_padded_rows(kernel):
    # row strides wider than the rows (e0 and y inside larger buffers)
    B, N, d = 70, 9, 24
    e0, emb, dy = _inter_inputs(B, N, d, False)
    P = sdi.dlrm_num_pairs(N, False)
    e0_big = torch.zeros((B, d + 5), device=DEV)
    e0_big[:, :d] = _t(e0)
    y_big = torch.full((B, d + P + 3), -1.0, device=DEV)
    sdi.dlrm_interact_fwd(e0_big[:, :d], _t(emb), False, y_big[:, :d + P])
    ref, mag = oracle.interact_fwd(e0, emb, False)
    assert_close(y_big[:, :d + P].cpu().numpy(), ref, mag, REL["f32"], "padded fwd")
    assert torch.all(y_big[:, d + P:] == -1.0)


@pytest.mark.parametrize("B,N,d,inc", [(5000, 26, 128, False), (40, 100, 256, True)])
def test_interact_rows_of_very_different_scales(B, N, d, inc, kernel):
    # the error bound is relative to sum |z_i||z_j|: rows scaled by 1e-3 .. 1e3,
    # elements spanning 6 decades within a row
    rng = np.random.default_rng([11, B, N, d])
    e0 = (rng.standard_normal((B, d)) * 10.0 ** rng.uniform(-3, 3, (B, d))).astype(np.float32)
    emb = (rng.standard_normal((B, N, d)) * 10.0 ** rng.uniform(-3, 3, (B, N, 1))
           * 10.0 ** rng.uniform(-3, 3, (B, N, d))).astype(np.float32)
    dy = rng.standard_normal((B, d + oracle.num_pairs(N, inc))).astype(np.float32)
    y = torch.full((B, d + sdi.dlrm_num_pairs(N, inc)), float("nan"), device=DEV)
    sdi.dlrm_interact_fwd(_t(e0), _t(emb), inc, y)
    ref, mag = oracle.interact_fwd(e0, emb, inc)
    assert_close(y.cpu().numpy(), ref, mag, REL["f32"], "fwd, wide range")
    de0 = torch.full((B, d), float("nan"), device=DEV)
    demb = torch.full((B, N, d), float("nan"), device=DEV)
    sdi.dlrm_interact_bwd(_t(e0), _t(emb), inc, _t(dy), de0, demb)
    r_de0, m_de0, r_demb, m_demb = oracle.interact_bwd(e0, emb, dy, inc)
    assert_close(de0.cpu().numpy(), r_de0, m_de0, REL["f32"], "de0, wide range")
    assert_close(demb.cpu().numpy(), r_demb, m_demb, REL["f32"], "demb, wide range")


ALONG_CASES = [(300, 26, 128, False), (37, 100, 256, True), (65, 5, 3, False), (21, 13, 33, True),
               (50, 0, 16, True), (33, 1, 8, False), (5000, 26, 128, True)]


@pytest.mark.parametrize("B,N,d,inc", ALONG_CASES)
def test_interact_alongside_matches_oracle(B, N, d, inc, kernel):
    # [e0 | e_1 .. e_N | pairs]: forward and backward
    rng = np.random.default_rng([7, B, N, d, inc])
    e0 = rng.standard_normal((B, d), dtype=np.float32)
    emb = rng.standard_normal((B, N, d), dtype=np.float32)
    width = sdi.dlrm_interact_width(N, d, inc, alongside=True)
    assert width == d * (N + 1) + oracle.num_pairs(N, inc)
    dy = rng.standard_normal((B, width), dtype=np.float32)
    emb_t = _t(emb) if N else torch.empty((B, 0, d), device=DEV)
    y = torch.full((B, width), float("nan"), device=DEV)
    sdi.dlrm_interact_fwd(_t(e0), emb_t, inc, y, alongside=True)
    ref, mag = oracle.interact_fwd(e0, emb, inc, alongside=True)
    got = y.cpu().numpy()
    np.testing.assert_array_equal(got[:, :d * (N + 1)], ref[:, :d * (N + 1)])  # the copies
    assert_close(got, ref, mag, REL["f32"], f"alongside fwd B={B} N={N} d={d}")
    de0 = torch.full((B, d), float("nan"), device=DEV)
    demb = torch.full((B, N, d), float("nan"), device=DEV)
    sdi.dlrm_interact_bwd(_t(e0), emb_t, inc, _t(dy), de0, demb, alongside=True)
    r_de0, m_de0, r_demb, m_demb = oracle.interact_bwd(e0, emb, dy, inc, alongside=True)
    assert_close(de0.cpu().numpy(), r_de0, m_de0, REL["f32"], "alongside de0")
    assert_close(demb.cpu().numpy(), r_demb, m_demb, REL["f32"], "alongside demb")


# -------------------------------------------------------- backward + SGD ---

BWD_CASES = {
    "tiny": dict(name="tiny"),
    "one-hot": dict(name="one-hot", B=1500, rows=[10, 17, 30, 52, 91, 5000, 100000]),
    "multi-hot-f16": dict(name="multi-hot", B=1000, rows=[5000, 70000, 123, 9]),
    "multi-hot-bf16": dict(name="multi-hot", B=700, rows=[4000, 321], dtype="bf16"),
    "capacity-f32": dict(name="capacity", B=400, rows=[20000, 30000, 77]),
    "heavy-grad": dict(name="interaction-heavy", B=500, T=4, rows=[1000] * 4),
    "d17-scalar": dict(name="multi-hot", B=300, rows=[100, 200], d=17),
    "d3-f32": dict(name="tiny", B=64, rows=[40, 50, 60], d=3),
    "d512-f32": dict(name="tiny", B=300, rows=[300, 20], d=512, bag=("poisson", 5.0, 0, 12)),
    # 40 tables: the sort's tiles find their table by a search, not by one warp's ballot
    "40-tables": dict(name="multi-hot", B=200, T=40, rows=[3000] * 40),
    # rows of 18-19 bits and 256-2560 keys per top-digit bucket: one pass on the top 8 bits and a
    # shared-memory sort per bucket; with Zipf indices a hot row overflows its bucket and the LSD
    # passes sort on the device instead
    "msd-f32": dict(name="capacity", B=4096, rows=[200000, 150001]),
    "msd-f16-poisson": dict(name="multi-hot", B=6000, T=3, rows=[300000, 270000, 524288], index=("uniform",)),
    "msd-overflow-zipf": dict(name="capacity", B=4096, rows=[200000, 150001], index=("zipf", 1.2)),
}
MSD_CASES = ("msd-f32", "msd-f16-poisson", "msd-overflow-zipf")


def _run_bwd(cfg, host, offsets, indices, dp, lr, grad_cap=None, want_view=True):
    tables = W.tables_to_device(host, cfg["dtype"])
    nnz = indices.size
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(cfg["T"], cfg["B"], nnz, cfg["d"]),
                     dtype=torch.uint8, device=DEV)
    grad = None if grad_cap is None else torch.full((grad_cap, cfg["d"]), float("nan"), device=DEV)
    flag = _flag()
    view = sdi.dlrm_emb_bag_bwd_sgd(tables, _t(offsets), _t(indices), cfg["B"], _t(dp), lr, ws,
                                    grad_rows=grad, err_flag=flag, want_view=want_view)
    status = sdi.dlrm_read_error(flag)
    return tables, grad, view, status


@pytest.mark.parametrize("case", list(BWD_CASES))
def test_emb_bag_bwd_sgd_without_a_view_gives_the_same_bits(case):
    # without a view the sort carries each lookup's bag instead of its position; the runs are
    # summed in the same sorted order either way, so tables and coalesced gradients must agree
    # bit for bit with the view path, which the oracle parity test checks
    c = dict(BWD_CASES[case])
    cfg = W.make_config(c.pop("name"), **c)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = W.make_dpooled(cfg)
    nnz = indices.size
    t_view, g_view, _, s_view = _run_bwd(cfg, host, offsets, indices, dp, 0.05, grad_cap=nnz)
    t_bags, g_bags, view, s_bags = _run_bwd(cfg, host, offsets, indices, dp, 0.05, grad_cap=nnz, want_view=False)
    assert view is None
    assert s_view == 0 and s_bags == 0
    np.testing.assert_array_equal(g_bags.cpu().numpy().view(np.uint32), g_view.cpu().numpy().view(np.uint32))
    for t in range(cfg["T"]):
        np.testing.assert_array_equal(device_table_bits(t_bags[t]), device_table_bits(t_view[t]))


def test_msd_cases_take_the_bucket_sort():
    for case in MSD_CASES:
        c = dict(BWD_CASES[case])
        cfg = W.make_config(c.pop("name"), **c)
        nnz = W.make_indices(cfg)[1].size
        assert sdi.dlrm_emb_bag_sort_plan(cfg["rows"], nnz)[1], case
    cfg = W.make_config("multi-hot", B=6000, T=3, rows=[300000, 1000, 524288])  # a small table: LSD
    assert not sdi.dlrm_emb_bag_sort_plan(cfg["rows"], W.make_indices(cfg)[1].size)[1]


def _check_coalesce(view, co, nnz):
    U = int(view["num_unique"].item())
    assert U == co["U"]
    np.testing.assert_array_equal(_u32(view["sorted_pos"]), co["sorted_pos"])
    np.testing.assert_array_equal(_u32(view["sorted_row"]), co["sorted_row"])
    np.testing.assert_array_equal(view["uniq_table"].cpu().numpy()[:U], co["uniq_table"])
    np.testing.assert_array_equal(_u32(view["uniq_row"])[:U], co["uniq_row"])
    np.testing.assert_array_equal(_u32(view["seg_off"])[:U + 1], co["seg_off"])


@pytest.mark.parametrize("case", list(BWD_CASES))
def test_emb_bag_bwd_sgd_matches_oracle(case):
    c = dict(BWD_CASES[case])
    cfg = W.make_config(c.pop("name"), **c)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = W.make_dpooled(cfg)
    lr = 0.05
    nnz = indices.size
    tables, grad, view, status = _run_bwd(cfg, host, offsets, indices, dp, lr, grad_cap=nnz)
    assert status == 0
    co = oracle.coalesce(cfg["rows"], offsets, indices, cfg["B"])
    _check_coalesce(view, co, nnz)
    g_ref, g_mag, w_ref, w_mag = oracle.sgd(host, cfg["dtype"], offsets, cfg["B"], nnz, dp, lr, co)
    U = co["U"]
    rel = REL[cfg["dtype"]]
    assert_close(grad.cpu().numpy()[:U], g_ref, g_mag, rel, f"coalesced gradient {case}")
    touched = {}
    for u in range(U):
        touched.setdefault(int(co["uniq_table"][u]), []).append(u)
    for t in range(cfg["T"]):
        us = touched.get(t, [])
        rows_t = co["uniq_row"][us]
        dev = device_table_f64(tables[t], cfg["dtype"])
        assert_close(dev[rows_t], w_ref[us], w_mag[us], rel, f"updated rows {case} t={t}",
                     table_dtype=cfg["dtype"])
        untouched = np.ones(cfg["rows"][t], dtype=bool)
        untouched[rows_t] = False
        np.testing.assert_array_equal(device_table_bits(tables[t])[untouched],
                                      host_table_bits(host[t], cfg["dtype"])[untouched])


def test_long_runs_cross_chunks_and_tiles():
    # one table where almost every lookup hits row 7: a run of ~12k lookups
    # spans 24 reduce chunks and 3 sort tiles; plus a second, mixed table.
    B = 3000
    rng = np.random.default_rng(11)
    bags0 = [[7] * int(rng.integers(0, 9)) for _ in range(B)]
    bags0[5] = [7, 3, 7]
    bags1 = [list(rng.integers(0, 50, int(rng.integers(0, 6)))) for _ in range(B)]
    offsets = [0]
    idx = []
    for bags in (bags0, bags1):
        for bag in bags:
            idx += bag
            offsets.append(len(idx))
    offsets = np.array(offsets, dtype=np.int64)
    indices = np.array(idx, dtype=np.int64)
    cfg = W.make_config("tiny", T=2, rows=[16, 50], B=B, d=32)
    host = [np.asarray(h) for h in W.tables_host(cfg)]
    dp = W.make_dpooled(cfg)
    tables, grad, view, status = _run_bwd(cfg, host, offsets, indices, dp, 0.01, grad_cap=indices.size)
    assert status == 0
    co = oracle.coalesce(cfg["rows"], offsets, indices, B)
    _check_coalesce(view, co, indices.size)
    g_ref, g_mag, w_ref, w_mag = oracle.sgd(host, "f32", offsets, B, indices.size, dp, 0.01, co)
    assert_close(grad.cpu().numpy()[:co["U"]], g_ref, g_mag, REL["f32"], "long-run gradient")
    t0 = [u for u in range(co["U"]) if co["uniq_table"][u] == 0]
    assert_close(device_table_f64(tables[0], "f32")[co["uniq_row"][t0]], w_ref[t0], w_mag[t0],
                 REL["f32"], "long-run rows")


def _runs_of_lengths(rng, lengths, rows):
    """Lookups of one table in which row r_i (distinct, increasing) appears
    lengths[i] times, shuffled over the positions."""
    rws = np.sort(rng.choice(rows, size=len(lengths), replace=False))
    idx = np.repeat(rws, lengths)
    rng.shuffle(idx)
    return idx


@pytest.mark.parametrize("dtype,d", [("f32", 128), ("f16", 128), ("bf16", 64), ("f32", 96), ("f16", 256),
                                     ("f32", 16)])
def test_runs_of_every_length_short_and_long(dtype, d):
    # runs of 1 .. 9 lookups (the reduce takes runs of a few lookups that end
    # inside a tile in a separate, run-parallel phase), a few hundred long
    # runs, runs that end exactly at a tile's end or continue into the next
    # tile, and a table of only length-1 runs spanning several tiles
    rng = np.random.default_rng(17)
    B = 2500
    pattern = [1, 2, 3, 4, 5, 1, 1, 4, 4, 9, 1, 2, 3, 700, 1, 4, 2, 4100, 3, 1]
    lengths0 = (pattern * 60)[:400]
    idx0 = _runs_of_lengths(rng, lengths0, 200000)
    idx1 = _runs_of_lengths(rng, [1] * 9000, 50000)
    idx2 = _runs_of_lengths(rng, [4] * 1024 + [5] * 3 + [1] * 900, 9000)
    per_table = [idx0, idx1, idx2]
    offsets, indices = [0], []
    for idx in per_table:
        cuts = np.sort(rng.integers(0, idx.size + 1, B - 1))
        bounds = np.concatenate([[0], cuts, [idx.size]])
        for b in range(B):
            indices.extend(idx[bounds[b]:bounds[b + 1]].tolist())
            offsets.append(len(indices))
    offsets = np.array(offsets, dtype=np.int64)
    indices = np.array(indices, dtype=np.int64)
    cfg = W.make_config("multi-hot", T=3, rows=[200000, 50000, 9000], B=B, d=d, dtype=dtype)
    host = W.tables_host(cfg)
    dp = W.make_dpooled(cfg)
    lr = 0.03
    tables, grad, view, status = _run_bwd(cfg, host, offsets, indices, dp, lr, grad_cap=indices.size)
    assert status == 0
    co = oracle.coalesce(cfg["rows"], offsets, indices, B)
    _check_coalesce(view, co, indices.size)
    g_ref, g_mag, w_ref, w_mag = oracle.sgd(host, dtype, offsets, B, indices.size, dp, lr, co)
    U = co["U"]
    rel = REL[dtype]
    assert_close(grad.cpu().numpy()[:U], g_ref, g_mag, rel, f"gradient {dtype} d={d}")
    for t in range(3):
        us = np.nonzero(co["uniq_table"] == t)[0]
        rows_t = co["uniq_row"][us]
        dev = device_table_f64(tables[t], dtype)
        assert_close(dev[rows_t], w_ref[us], w_mag[us], rel, f"rows {dtype} d={d} t={t}", table_dtype=dtype)
        untouched = np.ones(cfg["rows"][t], dtype=bool)
        untouched[rows_t] = False
        np.testing.assert_array_equal(device_table_bits(tables[t])[untouched],
                                      host_table_bits(host[t], dtype)[untouched])


def test_all_duplicate_bag_gives_k_times_the_gradient():
    k = 1300
    host = [np.zeros((9, 16), np.float32)]
    offsets = np.array([0, k], dtype=np.int64)
    indices = np.full(k, 4, dtype=np.int64)
    cfg = W.make_config("tiny", T=1, rows=[9], B=1, d=16)
    dp = (np.arange(16, dtype=np.float32) / 8 - 1).reshape(1, 1, 16)  # dyadic: sums are exact
    tables, grad, view, status = _run_bwd(cfg, host, offsets, indices, dp, 0.5, grad_cap=4)
    assert status == 0 and int(view["num_unique"].item()) == 1
    np.testing.assert_array_equal(grad.cpu().numpy()[0], k * dp[0, 0])
    np.testing.assert_array_equal(tables[0].cpu().numpy()[4], -0.5 * k * dp[0, 0])


def test_bwd_is_deterministic():
    cfg = W.make_config("multi-hot", B=800, rows=[3000, 40], dtype="f16")
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = W.make_dpooled(cfg)
    a, ga, _, _ = _run_bwd(cfg, host, offsets, indices, dp, 0.1, grad_cap=indices.size)
    b, gb, _, _ = _run_bwd(cfg, host, offsets, indices, dp, 0.1, grad_cap=indices.size)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert torch.equal(ga.view(torch.int32)[:1000], gb.view(torch.int32)[:1000])


def test_lr_zero_leaves_tables_untouched():
    cfg = W.make_config("interaction-heavy", B=200, T=3, rows=[500] * 3)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = W.make_dpooled(cfg)
    tables, grad, view, status = _run_bwd(cfg, host, offsets, indices, dp, 0.0, grad_cap=indices.size)
    assert status == 0
    for t in range(3):
        np.testing.assert_array_equal(device_table_bits(tables[t]), host_table_bits(host[t], "bf16"))


def test_grad_rows_capacity_is_flagged():
    cfg = W.make_config("tiny", B=64)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = W.make_dpooled(cfg)
    _, _, _, status = _run_bwd(cfg, host, offsets, indices, dp, 0.0, grad_cap=3)
    assert status == sdi._native.ERR_CAPACITY


def test_bwd_out_of_range_index_is_flagged():
    cfg = W.make_config("tiny", B=64)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    indices[17] = 1000
    dp = W.make_dpooled(cfg)
    _, _, _, status = _run_bwd(cfg, host, offsets, indices, dp, 0.01)
    assert status == sdi._native.ERR_INDEX_OOB


def test_bwd_bad_offsets_are_flagged():
    cfg = W.make_config("tiny", B=64)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    offsets[10] = offsets[12] + 1  # not monotone
    dp = W.make_dpooled(cfg)
    _, _, _, status = _run_bwd(cfg, host, offsets, indices, dp, 0.01)
    assert status == sdi._native.ERR_BAD_OFFSETS


def test_bwd_with_no_lookups():
    cfg = W.make_config("tiny", B=4, bag=("fixed", 0))
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    assert indices.size == 0
    tables = W.tables_to_device(host, "f32")
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(8, 4, 0, 16), dtype=torch.uint8, device=DEV)
    dp = _t(W.make_dpooled(cfg))
    view = sdi.dlrm_emb_bag_bwd_sgd(tables, _t(offsets), torch.empty(0, dtype=torch.int64, device=DEV), 4,
                                    dp, 0.1, ws, want_view=True)
    assert int(view["num_unique"].item()) == 0
    for t in range(8):
        np.testing.assert_array_equal(device_table_bits(tables[t]), host_table_bits(host[t], "f32"))


# ------------------------------------------------------- the whole chain ---

@pytest.mark.parametrize("name,over", [("tiny", {}),
                                       ("one-hot", dict(B=512, rows=[10, 17, 30, 52, 91, 5000])),
                                       ("multi-hot", dict(B=600, rows=[3000, 50000, 77])),
                                       ("interaction-heavy", dict(B=64, T=20, rows=[2000] * 20))])
def test_full_step_matches_oracle(name, over):
    """fwd -> interaction fwd -> interaction bwd -> bwd + SGD, each stage fed
    by the previous one on both sides; tolerances use the chained magnitudes."""
    cfg = W.make_config(name, **over)
    B, T, d, inc = cfg["B"], cfg["T"], cfg["d"], cfg["include_self"]
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    e0 = W.make_e0(cfg)
    dy = W.make_dy(cfg)
    tables = W.tables_to_device(host, cfg["dtype"])
    P = sdi.dlrm_num_pairs(T, inc)
    pooled = torch.empty((B, T, d), device=DEV)
    y = torch.empty((B, d + P), device=DEV)
    de0 = torch.empty((B, d), device=DEV)
    dpooled = torch.empty((B, T, d), device=DEV)
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(T, B, indices.size, d), dtype=torch.uint8,
                     device=DEV)
    grad = torch.empty((indices.size, d), device=DEV)
    flag = _flag()
    e0_t, dy_t, off_t, idx_t = _t(e0), _t(dy), _t(offsets), _t(indices)
    sdi.dlrm_emb_bag_fwd(tables, off_t, idx_t, B, pooled, err_flag=flag)
    sdi.dlrm_interact_fwd(e0_t, pooled, inc, y)
    sdi.dlrm_interact_bwd(e0_t, pooled, inc, dy_t, de0, dpooled)
    view = sdi.dlrm_emb_bag_bwd_sgd(tables, off_t, idx_t, B, dpooled, cfg["lr"], ws, grad_rows=grad,
                                    err_flag=flag, want_view=True)
    assert sdi.dlrm_read_error(flag) == 0

    rel = REL[cfg["dtype"]]
    p_ref, p_mag = oracle.emb_bag_fwd(host, cfg["dtype"], offsets, indices, B)
    assert_close(pooled.cpu().numpy(), p_ref, p_mag, rel, "pooled")
    y_ref, y_mag = oracle.interact_fwd(e0, p_ref, inc, emb_mag=p_mag)
    assert_close(y.cpu().numpy(), y_ref, y_mag, rel, "interaction")
    de0_ref, de0_mag, dp_ref, dp_mag = oracle.interact_bwd(e0, p_ref, dy, inc, emb_mag=p_mag)
    assert_close(de0.cpu().numpy(), de0_ref, de0_mag, rel, "de0")
    assert_close(dpooled.cpu().numpy(), dp_ref, dp_mag, rel, "dpooled")
    co = oracle.coalesce(cfg["rows"], offsets, indices, B)
    _check_coalesce(view, co, indices.size)
    g_ref, g_mag, w_ref, w_mag = oracle.sgd(host, cfg["dtype"], offsets, B, indices.size, dp_ref,
                                            cfg["lr"], co, dpooled_mag=dp_mag)
    assert_close(grad.cpu().numpy()[:co["U"]], g_ref, g_mag, rel, "row gradient")
    for t in range(T):
        us = np.nonzero(co["uniq_table"] == t)[0]
        dev = device_table_f64(tables[t], cfg["dtype"])
        assert_close(dev[co["uniq_row"][us]], w_ref[us], w_mag[us], rel, f"table {t}",
                     table_dtype=cfg["dtype"])


def test_device_table_fill_matches_the_host_generator():
    # the two copies of the input generator agree bit for bit
    for name, over in (("tiny", {}), ("multi-hot", dict(rows=[70001, 5])),
                       ("interaction-heavy", dict(T=2, rows=[3001, 7]))):
        cfg = W.make_config(name, **over)
        dev = W.make_tables_device(cfg)
        host = W.tables_host(cfg)
        for t in range(cfg["T"]):
            np.testing.assert_array_equal(device_table_bits(dev[t]), host_table_bits(host[t], cfg["dtype"]))
