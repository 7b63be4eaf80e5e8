"""The backward's two halves (dlrm_emb_bag_coalesce, then
dlrm_emb_bag_reduce_sgd) give what the single call gives, bit for bit,
including when the coalescing runs on another stream ahead of the forward.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()
    oracle.build()


CASES = {
    "multi-hot-f16": dict(name="multi-hot", B=600, rows=[5000, 70000, 123, 9]),
    "capacity-f32": dict(name="capacity", B=200, rows=[20000, 30000, 77]),
    "tiny": dict(name="tiny"),
    "heavy-bf16": dict(name="interaction-heavy", B=96, T=5, rows=[1000] * 5),
}


def _bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


@pytest.mark.parametrize("case", list(CASES))
def test_split_backward_equals_single_call(case):
    c = dict(CASES[case])
    cfg = W.make_config(c.pop("name"), **c)
    host = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    B, T, d = cfg["B"], cfg["T"], cfg["d"]
    nnz = indices.size
    off_t, idx_t = torch.from_numpy(offsets).to(DEV), torch.from_numpy(indices).to(DEV)
    dp = torch.from_numpy(W.make_dpooled(cfg)).to(DEV)
    lr = 0.05
    ws_bytes = sdi.dlrm_emb_bag_bwd_workspace_size(T, B, nnz, d)

    tab1 = W.tables_to_device(host, cfg["dtype"])
    ws1 = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    g1 = torch.zeros(nnz, d, device=DEV)
    v1 = sdi.dlrm_emb_bag_bwd_sgd(tab1, off_t, idx_t, B, dp, lr, ws1, grad_rows=g1, want_view=True)

    # coalesce on a side stream, ordered only by an event before the reduce
    tab2 = W.tables_to_device(host, cfg["dtype"])
    ws2 = torch.full((ws_bytes,), 0xA5, dtype=torch.uint8, device=DEV)
    g2 = torch.zeros(nnz, d, device=DEV)
    side, main = torch.cuda.Stream(), torch.cuda.current_stream()
    side.wait_stream(main)
    with torch.cuda.stream(side):
        v2 = sdi.dlrm_emb_bag_coalesce(cfg["rows"], d, off_t, idx_t, B, ws2, want_view=True)
        done = torch.cuda.Event()
        done.record(side)
    main.wait_event(done)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    sdi.dlrm_emb_bag_reduce_sgd(tab2, nnz, B, dp, lr, ws2, grad_rows=g2, err_flag=flag)
    assert sdi.dlrm_read_error(flag) == 0

    U = int(v1["num_unique"].item())
    assert U == int(v2["num_unique"].item())
    for k, n in (("sorted_pos", nnz), ("sorted_row", nnz), ("uniq_table", U), ("uniq_row", U), ("seg_off", U + 1)):
        np.testing.assert_array_equal(v1[k][:n].cpu().numpy(), v2[k][:n].cpu().numpy(), err_msg=k)
    np.testing.assert_array_equal(_bits(g1[:U]), _bits(g2[:U]))
    for a, b in zip(tab1, tab2):
        np.testing.assert_array_equal(_bits(a), _bits(b))


def test_split_backward_with_no_lookups():
    cfg = W.make_config("tiny", B=4)
    tables = W.tables_to_device(W.tables_host(cfg), "f32")
    before = [t.clone() for t in tables]
    offsets = torch.zeros(cfg["T"] * 4 + 1, dtype=torch.int64, device=DEV)
    indices = torch.zeros(0, dtype=torch.int64, device=DEV)
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(cfg["T"], 4, 0, cfg["d"]), dtype=torch.uint8, device=DEV)
    v = sdi.dlrm_emb_bag_coalesce(cfg["rows"], cfg["d"], offsets, indices, 4, ws, want_view=True)
    sdi.dlrm_emb_bag_reduce_sgd(tables, 0, 4, torch.zeros(4, cfg["T"], cfg["d"], device=DEV), 0.1, ws)
    assert int(v["num_unique"].item()) == 0
    assert int(v["seg_off"][0].item()) == 0
    for a, b in zip(before, tables):
        assert torch.equal(a, b)
