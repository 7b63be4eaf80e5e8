"""The hot path captured in a CUDA graph.

Every call runs asynchronously on the caller's stream with no host
synchronisation and no allocation, so a training step (lookup, interaction
forward and backward, coalescing on a second stream, reduce + SGD) can be
captured once and replayed.  The kernels are deterministic and reset their
own device state (tile counters, look-back words, flags) at every call, so
two replays must give, bit for bit, what two steps launched one by one give.
"""
import numpy as np
import pytest
import torch

import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


class _Step:
    def __init__(self, cfg, split):
        B, T, d = cfg["B"], cfg["T"], cfg["d"]
        self.cfg, self.split = cfg, split
        self.tables = W.tables_to_device(W.tables_host(cfg), cfg["dtype"])
        offsets, indices = W.make_indices(cfg)
        self.offsets, self.indices, self.nnz = _t(offsets), _t(indices), int(indices.size)
        self.e0, self.dy = _t(W.make_e0(cfg)), _t(W.make_dy(cfg))
        self.pooled = torch.empty((B, T, d), device=DEV)
        self.dpooled = torch.empty((B, T, d), device=DEV)
        self.y = torch.empty((B, d + sdi.dlrm_num_pairs(T, cfg["include_self"])), device=DEV)
        self.de0 = torch.empty((B, d), device=DEV)
        self.ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(T, B, self.nnz, d), dtype=torch.uint8,
                              device=DEV)
        self.flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.side = torch.cuda.Stream()
        self.done = torch.cuda.Event()

    def run(self):
        c = self.cfg
        main = torch.cuda.current_stream()
        if self.split:  # the coalescing needs only the indices: a second stream, beside the forward
            self.side.wait_stream(main)
            with torch.cuda.stream(self.side):
                sdi.dlrm_emb_bag_coalesce(c["rows"], c["d"], self.offsets, self.indices, c["B"], self.ws,
                                          err_flag=self.flag, stream=self.side)
                self.done.record(self.side)
        sdi.dlrm_emb_bag_fwd(self.tables, self.offsets, self.indices, c["B"], self.pooled, err_flag=self.flag)
        sdi.dlrm_interact_fwd(self.e0, self.pooled, c["include_self"], self.y)
        sdi.dlrm_interact_bwd(self.e0, self.pooled, c["include_self"], self.dy, self.de0, self.dpooled)
        if self.split:
            main.wait_event(self.done)
            sdi.dlrm_emb_bag_reduce_sgd(self.tables, self.nnz, c["B"], self.dpooled, c["lr"], self.ws,
                                        err_flag=self.flag)
        else:
            sdi.dlrm_emb_bag_bwd_sgd(self.tables, self.offsets, self.indices, c["B"], self.dpooled, c["lr"],
                                     self.ws, err_flag=self.flag)

    def outputs(self):
        torch.cuda.synchronize()
        out = [self.pooled, self.y, self.de0, self.dpooled] + list(self.tables)
        return [x.cpu().view(torch.uint8).numpy().copy() for x in out]


CASES = {
    "multi-hot-f16": dict(name="multi-hot", B=1024, rows=[50000, 300, 7, 4000] * 6 + [900, 20000]),
    "one-hot-f32": dict(name="one-hot", B=700, rows=[10, 57, 300, 2000, 9000] * 5 + [3]),
    "bf16-self-d64": dict(name="multi-hot", B=333, rows=[2000] * 9, dtype="bf16", d=64, include_self=True),
}


@pytest.mark.parametrize("split", [False, True], ids=["one-stream", "coalesce-beside"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_graph_replays_equal_launches_bit_for_bit(case, split):
    c = dict(CASES[case])
    cfg = W.make_config(c.pop("name"), **c)
    eager, graphed = _Step(cfg, split), _Step(cfg, split)
    for _ in range(2):
        eager.run()
    ref = eager.outputs()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # a first call of each entry point outside the capture (one-time set-up)
        graphed.run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graphed = _Step(cfg, split)  # fresh tables: the warm-up call above updated them
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.run()
    for _ in range(2):
        g.replay()
    got = graphed.outputs()
    names = ["pooled", "y", "de0", "dpooled"] + [f"table {t}" for t in range(cfg["T"])]
    for n, a, b in zip(names, got, ref):
        assert np.array_equal(a, b), f"{case}: {n} differs after two replays"
    assert sdi.dlrm_read_error(graphed.flag) == 0
