"""The no-allocation backward entry point, for callers that cannot allocate.

Some callers can neither call cudaMalloc nor pass the library a workspace:
a plugin that only receives its input and output tensors from the framework
that hosts it, or a service that must not claim device memory once it runs.
dlrm_emb_bag_bwd_sgd_noalloc serves them from a fixed scratch array inside
the library.  This test calls it through the C ABI twice in a row, on two
different batches, and checks each result against the workspace-based
dlrm_emb_bag_bwd_sgd run on identical copies of the inputs: both run the
same deterministic kernels, so tables, gradient rows and the coalescing
results must agree bit for bit.  It also checks that a call after the first
claims no device memory.  The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import _native
from sparse_dense_interaction_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()


def _inputs(cfg, seed):
    host = W.tables_host(cfg, seed)
    offsets, indices = W.make_indices(cfg, seed)
    return dict(tables=W.tables_to_device(host, cfg["dtype"]), offsets=torch.from_numpy(offsets).to(DEV),
                indices=torch.from_numpy(indices).to(DEV), dp=torch.from_numpy(W.make_dpooled(cfg, seed)).to(DEV),
                grad=torch.zeros((indices.size, cfg["d"]), device=DEV),
                flag=torch.zeros(1, dtype=torch.int32, device=DEV))


def _bits(t):
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16).cpu().numpy()


VIEW_KEYS = ("sorted_pos", "sorted_row", "uniq_table", "uniq_row", "seg_off")


@pytest.mark.parametrize("name,over", [("multi-hot", dict(B=1500, rows=[3000, 70000, 50])),
                                       ("tiny", dict(B=400, d=24))])
def test_noalloc_matches_the_workspace_entry_point_twice_in_a_row(name, over):
    cfg = W.make_config(name, **over)
    # a first, empty call makes the scratch array resident on this device
    # (as a service would at start-up); later calls claim no memory
    empty = W.make_config(name, **dict(over, B=2, bag=("fixed", 0)))
    x = _inputs(empty, 0)
    sdi.dlrm_emb_bag_bwd_sgd_noalloc(x["tables"], x["offsets"], x["indices"], 2, x["dp"], 0.05)
    torch.cuda.synchronize()
    for seed in (1, 2):  # two calls in a row, different batches
        ref, new = _inputs(cfg, seed), _inputs(cfg, seed)
        nnz = ref["indices"].numel()
        ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(cfg["T"], cfg["B"], nnz, cfg["d"]),
                         dtype=torch.uint8, device=DEV)
        v_ref = sdi.dlrm_emb_bag_bwd_sgd(ref["tables"], ref["offsets"], ref["indices"], cfg["B"], ref["dp"], 0.05,
                                         ws, grad_rows=ref["grad"], err_flag=ref["flag"], want_view=True)
        assert sdi.dlrm_read_error(ref["flag"]) == 0
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        v_new = sdi.dlrm_emb_bag_bwd_sgd_noalloc(new["tables"], new["offsets"], new["indices"], cfg["B"], new["dp"],
                                                 0.05, grad_rows=new["grad"], err_flag=new["flag"], want_view=True)
        assert sdi.dlrm_read_error(new["flag"]) == 0
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before, "the call claimed device memory"
        U = int(v_ref["num_unique"].item())
        assert int(v_new["num_unique"].item()) == U
        for k in VIEW_KEYS:
            n = U + 1 if k == "seg_off" else (U if k.startswith("uniq") else nnz)
            np.testing.assert_array_equal(v_new[k][:n].cpu().numpy(), v_ref[k][:n].cpu().numpy(), err_msg=k)
        np.testing.assert_array_equal(_bits(new["grad"][:U]), _bits(ref["grad"][:U]))
        for a, b in zip(new["tables"], ref["tables"]):
            np.testing.assert_array_equal(_bits(a), _bits(b))


def test_noalloc_refuses_sizes_beyond_its_scratch():
    need = sdi.dlrm_emb_bag_bwd_workspace_size(1, 4, 1 << 21, 128)
    assert need > _native.NOALLOC_SCRATCH_BYTES
    tables = [torch.zeros((10, 128), device=DEV)]
    offsets = torch.tensor([0, 0, 0, 0, 1 << 21], dtype=torch.int64, device=DEV)
    indices = torch.zeros(1 << 21, dtype=torch.int64, device=DEV)
    dp = torch.zeros((4, 1, 128), device=DEV)
    launches = sdi.dlrm_kernel_launch_count()
    with pytest.raises(sdi.DlrmError) as e:
        sdi.dlrm_emb_bag_bwd_sgd_noalloc(tables, offsets, indices, 4, dp, 0.1)
    assert e.value.status == _native.ERR_WORKSPACE_TOO_SMALL
    assert sdi.dlrm_kernel_launch_count() == launches
