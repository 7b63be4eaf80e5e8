"""Row-wise int4 tables: the GPU encoder (bit-exact against the oracle's
encoder, which decides every code in the same fp32 arithmetic) and the pooled
lookup over int4 tables (within rel 1e-5 x magnitude of the oracle's fp64
decode-and-sum: the lookup computes in fp32)."""
import numpy as np
import pytest
import torch

import oracle
import sparse_dense_interaction_gb300 as sdi
from sparse_dense_interaction_gb300 import workloads as W
from tests._parity import REL, assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_dense_interaction_gb300 import build
    build.build()
    oracle.build()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _rows(dtype, R, d, seed):
    """Host rows with edge cases: constant rows, +-0 mixes, exact ties, wide ranges."""
    rng = np.random.default_rng([seed, R, d])
    w = rng.standard_normal((R, d)).astype(np.float32) * rng.uniform(0.01, 100, (R, 1)).astype(np.float32)
    w[0] = 1.25
    w[1] = 0.0
    w[1, ::3] = -0.0
    w[2] = np.arange(d) % 16 / 4.0  # codes on the grid, with ties (x.5) nowhere
    w[3, :] = np.where(np.arange(d) % 2 == 0, 0.0, 3.0)
    w[3, 1] = 1.5  # (1.5 - 0) / 0.2 ties at 7.5
    if dtype == "f16":
        return w.astype(np.float16)
    if dtype == "bf16":
        return W.f32_to_bf16_bits(w)
    return w


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("d", [8, 16, 24, 40, 128, 256, 512])
def test_encoder_matches_oracle_bit_for_bit(dtype, d):
    host = _rows(dtype, 300, d, 1)
    src = W.tables_to_device([host], dtype)[0]
    q = sdi.dlrm_quantize_int4(src)
    assert q.shape == (300, sdi.dlrm_int4_row_bytes(d))
    np.testing.assert_array_equal(q.cpu().numpy(), oracle.quantize_int4(host, dtype))


CASES = {
    "multi-hot-d128": dict(name="multi-hot", B=300, rows=[5000, 70000, 123, 9]),
    "one-hot-d64": dict(name="one-hot", B=400, rows=[10, 17, 30, 52, 91, 5000, 100000]),
    "capacity-d128": dict(name="capacity", B=100, rows=[20000, 30000, 77]),
    "d40-half-chunk": dict(name="multi-hot", B=77, rows=[300, 20, 999], d=40),
    "d512": dict(name="tiny", B=40, rows=[300, 20], d=512),
    "d8": dict(name="multi-hot", B=50, rows=[300, 20], d=8),
}


@pytest.mark.parametrize("case", list(CASES))
def test_int4_lookup_matches_oracle(case):
    c = dict(CASES[case])
    cfg = W.make_config(c.pop("name"), **c)
    B, T, d = cfg["B"], cfg["T"], cfg["d"]
    host = W.tables_host(cfg)
    qhost = [oracle.quantize_int4(h, cfg["dtype"]) for h in host]
    offsets, indices = W.make_indices(cfg)
    # the tables encoded on the GPU are the oracle's bytes
    src = W.tables_to_device(host, cfg["dtype"])
    qdev = [sdi.dlrm_quantize_int4(s) for s in src]
    for a, b in zip(qdev, qhost):
        np.testing.assert_array_equal(a.cpu().numpy(), b)
    out = torch.full((B, T, d), float("nan"), device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    sdi.dlrm_emb_bag_fwd(qdev, _t(offsets), _t(indices), B, out, err_flag=flag, d=d)
    assert sdi.dlrm_read_error(flag) == 0
    ref, mag = oracle.emb_bag_fwd(qhost, "int4", offsets, indices, B, d=d)
    assert_close(out.cpu().numpy(), ref, mag, REL["f32"], f"int4 pooled {case}")


def test_int4_lookup_empty_bags_and_out_of_range():
    host = [np.arange(10 * 16, dtype=np.float32).reshape(10, 16) / 7, np.ones((3, 16), np.float32)]
    q = [oracle.quantize_int4(h, "f32") for h in host]
    offsets = np.array([0, 0, 2, 4, 4, 5, 5], dtype=np.int64)  # T = 2, B = 3
    indices = np.array([0, 9, 10, 3, 2], dtype=np.int64)       # 10 is out of table 0's range
    out = torch.full((3, 2, 16), float("nan"), device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    sdi.dlrm_emb_bag_fwd([_t(x) for x in q], _t(offsets), _t(indices), 3, out, err_flag=flag, d=16)
    assert sdi.dlrm_read_error(flag) == sdi._native.ERR_INDEX_OOB
    ref, mag = oracle.emb_bag_fwd(q, "int4", np.array([0, 0, 2, 3, 3, 4, 4]), np.array([0, 9, 3, 2]), 3, d=16)
    assert_close(out.cpu().numpy(), ref, mag, REL["f32"], "int4 empty/oob")
    assert torch.all(out[0] == 0)


def test_int4_with_the_interaction_and_the_backward():
    cfg = W.make_config("multi-hot", B=90, rows=[400, 500, 600])
    B, T, d, inc = cfg["B"], cfg["T"], cfg["d"], cfg["include_self"]
    host = W.tables_host(cfg)
    q = [sdi.dlrm_quantize_int4(s) for s in W.tables_to_device(host, cfg["dtype"])]
    qhost = [x.cpu().numpy() for x in q]
    offsets, indices = W.make_indices(cfg)
    e0 = W.make_e0(cfg)
    y = torch.empty((B, sdi.dlrm_interact_width(T, d, inc)), device=DEV)
    with pytest.raises(sdi.DlrmError) as ei:  # no single-kernel path: the pooled block is needed
        sdi.dlrm_emb_bag_interact_fwd(q, _t(offsets), _t(indices), B, _t(e0), inc, y, d=d)
    assert ei.value.status == sdi._native.ERR_UNSUPPORTED
    pooled = torch.empty((B, T, d), device=DEV)
    sdi.dlrm_emb_bag_interact_fwd(q, _t(offsets), _t(indices), B, _t(e0), inc, y, pooled=pooled, d=d)
    p_ref, p_mag = oracle.emb_bag_fwd(qhost, "int4", offsets, indices, B, d=d)
    y_ref, y_mag = oracle.interact_fwd(e0, p_ref, inc, emb_mag=p_mag)
    assert_close(y.cpu().numpy(), y_ref, y_mag, REL["f32"], "int4 interaction")
    # the backward refuses int4 tables on the host, before launching anything
    ptrs, rows, _, _, _ = sdi._native._tables(q, d)
    ws = torch.empty(sdi.dlrm_emb_bag_bwd_workspace_size(T, B, indices.size, d), dtype=torch.uint8, device=DEV)
    st = sdi._native.load().dlrm_emb_bag_bwd_sgd(ptrs, rows, T, d, sdi.INT4, _t(offsets).data_ptr(),
                                                 _t(indices).data_ptr(), indices.size, B, pooled.data_ptr(), T * d,
                                                 d, 0.1, None, 0, ws.data_ptr(), ws.numel(), None, None, None)
    assert st == sdi._native.ERR_UNSUPPORTED
