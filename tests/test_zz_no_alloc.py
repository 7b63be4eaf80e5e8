"""The no-allocation backward entry point, for callers that cannot allocate.

Some callers can neither call cudaMalloc nor pass the library a workspace
(for example a plugin that only receives its input and output tensors from
the framework that hosts it).  dlrm_emb_bag_bwd_sgd_noalloc serves them from
a fixed scratch array inside the library.  This test calls it through the C
ABI twice in a row, on two different batches, and checks each result against
the workspace-based dlrm_emb_bag_bwd_sgd run on identical copies of the
inputs.  The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import _native
from sparse_dense_interaction_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
REL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()


def _run(cfg, seed, noalloc):
    host = W.tables_host(cfg, seed)
    tables = W.tables_to_device(host, cfg["dtype"])
    offsets, indices = W.make_indices(cfg, seed)
    dp = torch.from_numpy(W.make_dpooled(cfg, seed)).to(DEV)
    off_t = torch.from_numpy(offsets).to(DEV)
    idx_t = torch.from_numpy(indices).to(DEV)
    grad = torch.zeros((indices.size, cfg["d"]), device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    if noalloc:
        sdi.dlrm_emb_bag_bwd_sgd_noalloc(tables, off_t, idx_t, cfg["B"], dp, 0.05, grad_rows=grad,
                                         err_flag=flag)
    else:
        ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(cfg["T"], cfg["B"], indices.size, cfg["d"]),
                         dtype=torch.uint8, device=DEV)
        sdi.dlrm_emb_bag_bwd_sgd(tables, off_t, idx_t, cfg["B"], dp, 0.05, ws, grad_rows=grad, err_flag=flag)
    assert sdi.dlrm_read_error(flag) == 0
    return [t.float().cpu().numpy() for t in tables], grad.cpu().numpy()


def _close(a, b, rel, what):
    tol = rel * np.maximum(np.abs(a), np.abs(b)) + 1e-30
    bad = np.abs(a - b) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} elements differ beyond rel {rel}"


@pytest.mark.parametrize("name,over", [("multi-hot", dict(B=1500, rows=[3000, 70000, 50])),
                                       ("tiny", dict(B=400, d=24))])
def test_noalloc_matches_the_workspace_entry_point_twice_in_a_row(name, over):
    cfg = W.make_config(name, **over)
    for seed in (1, 2):  # two calls in a row, different batches
        t_ref, g_ref = _run(cfg, seed, noalloc=False)
        t_new, g_new = _run(cfg, seed, noalloc=True)
        rel = REL[cfg["dtype"]]
        _close(g_new, g_ref, rel, f"gradient rows, call {seed}")
        for t in range(cfg["T"]):
            _close(t_new[t], t_ref[t], rel, f"table {t}, call {seed}")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    need = sdi.dlrm_emb_bag_bwd_workspace_size(1, 4, 1 << 21, 128)
    assert need > _native.NOALLOC_SCRATCH_BYTES
    tables = [torch.zeros((10, 128), device=DEV)]
    offsets = torch.tensor([0, 0, 0, 0, 1 << 21], dtype=torch.int64, device=DEV)
    indices = torch.zeros(1 << 21, dtype=torch.int64, device=DEV)
    dp = torch.zeros((4, 1, 128), device=DEV)
    with pytest.raises(sdi.DlrmError) as e:
        sdi.dlrm_emb_bag_bwd_sgd_noalloc(tables, offsets, indices, 4, dp, 0.1)
    assert e.value.status == _native.ERR_WORKSPACE_TOO_SMALL
