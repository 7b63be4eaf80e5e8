"""Pins for the oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a fact the DLRM pages or plain
mathematics fix: hand-worked examples (tests/golden/), term counts, a
textbook matrix product (numpy), the factorization-machine identity, central
finite differences, brute force over tiny inputs, and library sorts.  A
plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a missing factor of two, an unstable sort) fails at least
one of them.
"""
import collections

import numpy as np
import pytest

import oracle
from sparse_dense_interaction_gb300 import workloads as W
from tests import _golden


def _csr(bags_per_table):
    """Table-major CSR from a list (per table) of lists (per bag) of rows."""
    T = len(bags_per_table)
    B = len(bags_per_table[0])
    offsets = [0]
    indices = []
    for t in range(T):
        for b in range(B):
            indices.extend(bags_per_table[t][b])
            offsets.append(len(indices))
    return np.array(offsets, dtype=np.int64), np.array(indices, dtype=np.int64)


def _random_bags(rng, T, B, rows, max_len, dup=True):
    bags = []
    for t in range(T):
        tb = []
        for _ in range(B):
            L = int(rng.integers(0, max_len + 1))
            if dup:
                tb.append(list(rng.integers(0, rows[t], L)))
            else:
                tb.append(list(rng.choice(rows[t], size=min(L, rows[t]), replace=False)))
        bags.append(tb)
    return bags


def _bf16_bits_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- lookup ---

def test_emb_bag_worked_example():
    g = _golden.load("emb_bag_worked_example.txt")
    tables = [g["table0"].reshape(3, 2).astype(np.float32), g["table1"].reshape(2, 2).astype(np.float32)]
    pooled, mag = oracle.emb_bag_fwd(tables, "f32", g["offsets"], g["indices"], 2)
    np.testing.assert_array_equal(pooled.reshape(-1), g["pooled"])
    np.testing.assert_array_equal(mag.reshape(-1), np.abs(g["pooled"]))  # all values positive


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_pooling_factor_one_is_row_copy(dtype):
    cfg = W.make_config("tiny", dtype=dtype, rows=[50, 70, 30], B=40)
    tables = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    pooled, _ = oracle.emb_bag_fwd(tables, dtype, offsets, indices, cfg["B"])
    for t in range(cfg["T"]):
        idx = indices[offsets[t * cfg["B"]]:offsets[(t + 1) * cfg["B"]]]
        if dtype == "bf16":
            expect = _bf16_bits_to_f64(tables[t][idx])
        else:
            expect = tables[t][idx].astype(np.float64)  # numpy's own float16 decode
        np.testing.assert_array_equal(pooled[:, t, :], expect)


def test_binary16_decode_covers_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    np.testing.assert_array_equal(np.isinf(ours), np.isinf(ref))


@pytest.mark.parametrize("dup", [False, True])
def test_pooled_equals_bruteforce_sum(dup):
    rng = np.random.default_rng(1)
    rows = [40, 9, 77]
    tables = [rng.standard_normal((r, 5)).astype(np.float32) for r in rows]
    bags = _random_bags(rng, 3, 16, rows, 8, dup=dup)
    offsets, indices = _csr(bags)
    pooled, mag = oracle.emb_bag_fwd(tables, "f32", offsets, indices, 16)
    for t in range(3):
        for b in range(16):
            r = np.array(bags[t][b], dtype=np.int64)
            got = tables[t][r].astype(np.float64)
            expect = got.sum(axis=0) if r.size else np.zeros(5)
            np.testing.assert_allclose(pooled[b, t], expect, rtol=0, atol=1e-12)
            np.testing.assert_allclose(mag[b, t], np.abs(got).sum(axis=0) if r.size else 0,
                                       rtol=0, atol=1e-12)
            assert np.all(mag[b, t] >= np.abs(pooled[b, t]))


def test_pooling_is_linear_in_the_bag():
    rng = np.random.default_rng(2)
    rows = [25, 31]
    tables = [rng.standard_normal((r, 6)).astype(np.float32) for r in rows]
    bags1 = _random_bags(rng, 2, 10, rows, 6)
    bags2 = _random_bags(rng, 2, 10, rows, 6)
    union = [[bags1[t][b] + bags2[t][b] for b in range(10)] for t in range(2)]
    p1, _ = oracle.emb_bag_fwd(tables, "f32", *_csr(bags1), 10)
    p2, _ = oracle.emb_bag_fwd(tables, "f32", *_csr(bags2), 10)
    pu, _ = oracle.emb_bag_fwd(tables, "f32", *_csr(union), 10)
    np.testing.assert_allclose(pu, p1 + p2, rtol=0, atol=1e-12)


def test_empty_bags_pool_to_zero():
    tables = [np.ones((4, 3), dtype=np.float32)]
    offsets = np.array([0, 0, 0, 2], dtype=np.int64)
    pooled, _ = oracle.emb_bag_fwd(tables, "f32", offsets, np.array([1, 3]), 3)
    np.testing.assert_array_equal(pooled[0], 0)
    np.testing.assert_array_equal(pooled[1], 0)
    np.testing.assert_array_equal(pooled[2, 0], 2)


def test_lookup_errors_are_reported():
    tables = [np.ones((4, 3), dtype=np.float32)]
    with pytest.raises(oracle.OracleError) as e:
        oracle.emb_bag_fwd(tables, "f32", np.array([0, 1]), np.array([4]), 1)
    assert e.value.status == oracle.INDEX_OOB
    with pytest.raises(oracle.OracleError) as e:
        oracle.emb_bag_fwd(tables, "f32", np.array([0, 2, 1]), np.array([0, 1]), 2)
    assert e.value.status == oracle.BAD_OFFSETS


# ----------------------------------------------------------- interaction ---

def test_pair_counts_match_the_pages():
    for N, inc, d, P, width in _golden.rows("pair_counts.txt"):
        assert oracle.num_pairs(N, bool(inc)) == P
        rng = np.random.default_rng(N)
        y, _ = oracle.interact_fwd(rng.standard_normal((2, d)), rng.standard_normal((2, N, d)),
                                   bool(inc))
        assert y.shape == (2, width)


@pytest.mark.parametrize("mode", ["strict", "inclusive"])
def test_interaction_worked_example(mode):
    g = _golden.load("interaction_worked_example.txt")
    e0 = g["e0"].reshape(1, 2)
    emb = g["emb"].reshape(1, 2, 2)
    y, _ = oracle.interact_fwd(e0, emb, mode == "inclusive")
    np.testing.assert_array_equal(y[0], g[f"y_{mode}"])
    de0, _, demb, _ = oracle.interact_bwd(e0, emb, g[f"dy_{mode}"].reshape(1, -1),
                                          mode == "inclusive")
    np.testing.assert_array_equal(de0[0], g[f"de0_{mode}"])
    np.testing.assert_array_equal(demb.reshape(-1), g[f"demb_{mode}"])


def _stack(e0, emb):
    return np.concatenate([e0[:, None, :], emb], axis=1)


@pytest.mark.parametrize("inc", [False, True])
def test_interaction_is_the_triangle_of_a_symmetric_gram_matrix(inc):
    rng = np.random.default_rng(3)
    B, N, d = 5, 7, 9
    e0 = rng.standard_normal((B, d))
    emb = rng.standard_normal((B, N, d))
    y, mag = oracle.interact_fwd(e0, emb, inc)
    Z = _stack(e0, emb)
    gram = Z @ np.swapaxes(Z, 1, 2)  # textbook matrix product
    np.testing.assert_allclose(gram, np.swapaxes(gram, 1, 2), rtol=0, atol=1e-12)
    rr, cc = np.tril_indices(N + 1, k=0 if inc else -1)  # row-major lower triangle
    np.testing.assert_array_equal(y[:, :d], e0)
    np.testing.assert_allclose(y[:, d:], gram[:, rr, cc], rtol=0, atol=1e-12)
    absgram = np.abs(Z) @ np.swapaxes(np.abs(Z), 1, 2)
    np.testing.assert_allclose(mag[:, d:], absgram[:, rr, cc], rtol=1e-14, atol=0)


def test_interaction_bruteforce_dots():
    rng = np.random.default_rng(4)
    e0 = rng.standard_normal((3, 4))
    emb = rng.standard_normal((3, 3, 4))
    y, _ = oracle.interact_fwd(e0, emb, False)
    for b in range(3):
        z = [e0[b]] + [emb[b, i] for i in range(3)]
        expect = [float(np.dot(z[i], z[j])) for i in range(4) for j in range(i)]
        np.testing.assert_allclose(y[b, 4:], expect, rtol=0, atol=1e-12)


@pytest.mark.parametrize("inc", [False, True])
def test_factorization_machine_identity(inc):
    # sum_{i<j} z_i.z_j = (|sum z|^2 - sum |z_i|^2) / 2; self pairs add sum |z_i|^2
    rng = np.random.default_rng(5)
    e0 = rng.standard_normal((6, 11))
    emb = rng.standard_normal((6, 12, 11))
    y, _ = oracle.interact_fwd(e0, emb, inc)
    Z = _stack(e0, emb)
    total = (Z.sum(axis=1) ** 2).sum(axis=1)
    squares = (Z ** 2).sum(axis=(1, 2))
    expect = 0.5 * (total + squares) if inc else 0.5 * (total - squares)
    np.testing.assert_allclose(y[:, 11:].sum(axis=1), expect, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("inc", [False, True])
def test_interaction_backward_by_finite_differences(inc):
    # L = sum(w * Y) is quadratic in the inputs, so central differences are
    # exact up to rounding.
    rng = np.random.default_rng(6)
    B, N, d = 2, 4, 3
    e0 = rng.standard_normal((B, d))
    emb = rng.standard_normal((B, N, d))
    width = d + oracle.num_pairs(N, inc)
    w = rng.standard_normal((B, width))
    de0, _, demb, _ = oracle.interact_bwd(e0, emb, w, inc)

    def loss(a, b):
        y, _ = oracle.interact_fwd(a, b, inc)
        return float((w * y).sum())

    h = 1e-3
    for idx in np.ndindex(e0.shape):
        p, m = e0.copy(), e0.copy()
        p[idx] += h
        m[idx] -= h
        fd = (loss(p, emb) - loss(m, emb)) / (2 * h)
        assert abs(fd - de0[idx]) <= 1e-6 * max(1.0, abs(fd))
    for idx in np.ndindex(emb.shape):
        p, m = emb.copy(), emb.copy()
        p[idx] += h
        m[idx] -= h
        fd = (loss(e0, p) - loss(e0, m)) / (2 * h)
        assert abs(fd - demb[idx]) <= 1e-6 * max(1.0, abs(fd))


@pytest.mark.parametrize("inc", [False, True])
def test_interaction_backward_closed_form(inc):
    # dZ = (G + G^T) Z with G the lower-triangular matrix of upstream gradients
    rng = np.random.default_rng(7)
    B, N, d = 4, 6, 5
    e0 = rng.standard_normal((B, d))
    emb = rng.standard_normal((B, N, d))
    F = N + 1
    dy = rng.standard_normal((B, d + oracle.num_pairs(N, inc)))
    de0, _, demb, _ = oracle.interact_bwd(e0, emb, dy, inc)
    rr, cc = np.tril_indices(F, k=0 if inc else -1)
    G = np.zeros((B, F, F))
    G[:, rr, cc] = dy[:, d:]
    dZ = (G + np.swapaxes(G, 1, 2)) @ _stack(e0, emb)
    np.testing.assert_allclose(de0, dy[:, :d] + dZ[:, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(demb, dZ[:, 1:], rtol=0, atol=1e-12)


# ------------------------------------------------------------ coalescing ---

def test_coalesce_worked_example():
    g = _golden.load("emb_bag_worked_example.txt")
    co = oracle.coalesce([3, 2], g["offsets"], g["indices"], 2)
    for key in ("sorted_pos", "sorted_row", "uniq_table", "uniq_row", "seg_off"):
        np.testing.assert_array_equal(co[key], g[key])
    assert co["U"] == 4


@pytest.mark.parametrize("kind", ["zipf", "uniform"])
def test_coalesce_matches_a_library_stable_sort(kind):
    cfg = W.make_config("multi-hot", rows=[500, 37, 4000, 1], B=64,
                        index=("zipf", 1.2) if kind == "zipf" else ("uniform",))
    offsets, indices = W.make_indices(cfg)
    co = oracle.coalesce(cfg["rows"], offsets, indices, cfg["B"])
    B = cfg["B"]
    table_of = np.repeat(np.arange(cfg["T"]), np.diff(offsets[::B]))
    order = np.lexsort((indices, table_of))  # numpy's lexsort is stable
    np.testing.assert_array_equal(co["sorted_pos"], order)
    np.testing.assert_array_equal(co["sorted_row"], indices[order])
    pairs = sorted(set(zip(table_of.tolist(), indices.tolist())))
    assert co["U"] == len(pairs)
    np.testing.assert_array_equal(co["uniq_table"], [p[0] for p in pairs])
    np.testing.assert_array_equal(co["uniq_row"], [p[1] for p in pairs])
    counts = collections.Counter(zip(table_of.tolist(), indices.tolist()))
    np.testing.assert_array_equal(np.diff(co["seg_off"]), [counts[p] for p in pairs])
    assert co["seg_off"][-1] == indices.size


def test_coalesce_properties_with_heavy_duplicates():
    rng = np.random.default_rng(8)
    bags = [[list(rng.integers(0, 3, 9)) for _ in range(20)] for _ in range(3)]
    offsets, indices = _csr(bags)
    co = oracle.coalesce([3, 3, 3], offsets, indices, 20)
    sp = co["sorted_pos"]
    assert sorted(sp.tolist()) == list(range(indices.size))  # a permutation
    for u in range(co["U"]):
        seg = sp[co["seg_off"][u]:co["seg_off"][u + 1]]
        assert np.all(np.diff(seg) > 0)  # ties keep their original order
        assert np.all(indices[seg] == co["uniq_row"][u])


# -------------------------------------------------------- backward + SGD ---

def test_sgd_worked_example():
    g = _golden.load("emb_bag_worked_example.txt")
    tables = [g["table0"].reshape(3, 2).astype(np.float32), g["table1"].reshape(2, 2).astype(np.float32)]
    co = oracle.coalesce([3, 2], g["offsets"], g["indices"], 2)
    grad, _, new_row, _ = oracle.sgd(tables, "f32", g["offsets"], 2, 6,
                                     g["dpooled"].reshape(2, 2, 2), float(g["lr"][0]), co)
    np.testing.assert_array_equal(grad.reshape(-1), g["grad"])
    np.testing.assert_array_equal(new_row.reshape(-1), g["new_row"])


def test_all_duplicate_bag_gives_k_times_the_gradient():
    k = 13
    tables = [np.zeros((5, 4), dtype=np.float32)]
    offsets = np.array([0, k], dtype=np.int64)
    indices = np.full(k, 3, dtype=np.int64)
    dp = np.array([[[0.25, -1.5, 3.0, 0.125]]])
    co = oracle.coalesce([5], offsets, indices, 1)
    grad, _, new_row, _ = oracle.sgd(tables, "f32", offsets, 1, k, dp, 0.5, co)
    assert co["U"] == 1 and co["uniq_row"][0] == 3
    np.testing.assert_array_equal(grad[0], k * dp[0, 0])
    np.testing.assert_array_equal(new_row[0], -0.5 * k * dp[0, 0])


def test_duplicate_updates_equal_the_summed_gradient():
    rng = np.random.default_rng(9)
    rows = [6, 11, 4]
    T, B, d = 3, 12, 3
    tables = [rng.standard_normal((r, d)).astype(np.float32) for r in rows]
    bags = _random_bags(rng, T, B, rows, 7)
    offsets, indices = _csr(bags)
    dp = rng.standard_normal((B, T, d))
    co = oracle.coalesce(rows, offsets, indices, B)
    grad, _, new_row, _ = oracle.sgd(tables, "f32", offsets, B, indices.size, dp, 0.1, co)
    brute = collections.defaultdict(lambda: np.zeros(d))
    for t in range(T):
        for b in range(B):
            for r in bags[t][b]:
                brute[(t, int(r))] += dp[b, t]
    assert co["U"] == len(brute)
    for u in range(co["U"]):
        key = (int(co["uniq_table"][u]), int(co["uniq_row"][u]))
        np.testing.assert_allclose(grad[u], brute[key], rtol=0, atol=1e-12)
        w = tables[key[0]][key[1]].astype(np.float64)
        np.testing.assert_allclose(new_row[u], w - 0.1 * brute[key], rtol=0, atol=1e-12)


def test_row_gradient_by_finite_differences():
    # L(W) = sum_{b,t} w_bt . pooled_bt(W) is linear in W; with dyadic table
    # values and step, the central difference is exact.
    rng = np.random.default_rng(10)
    rows = [7, 5]
    T, B, d = 2, 6, 3
    tables = [(rng.integers(-64, 64, (r, d)) / 64).astype(np.float32) for r in rows]
    bags = _random_bags(rng, T, B, rows, 5)
    offsets, indices = _csr(bags)
    w = (rng.integers(-8, 8, (B, T, d)) / 8).astype(np.float64)
    co = oracle.coalesce(rows, offsets, indices, B)
    grad, _, _, _ = oracle.sgd(tables, "f32", offsets, B, indices.size, w, 0.0, co)

    def loss(tabs):
        pooled, _ = oracle.emb_bag_fwd(tabs, "f32", offsets, indices, B)
        return float((w * pooled).sum())

    h = np.float32(1 / 64)
    for u in range(co["U"]):
        t, r = int(co["uniq_table"][u]), int(co["uniq_row"][u])
        for e in range(d):
            p = [x.copy() for x in tables]
            m = [x.copy() for x in tables]
            p[t][r, e] += h
            m[t][r, e] -= h
            fd = (loss(p) - loss(m)) / (2 * float(h))
            assert fd == pytest.approx(grad[u, e], abs=1e-12)
    # rows that no lookup touches have zero gradient and are not reported
    touched = set(zip(co["uniq_table"].tolist(), co["uniq_row"].tolist()))
    for t in range(T):
        for r in range(rows[t]):
            if (t, r) not in touched:
                p = [x.copy() for x in tables]
                p[t][r, 0] += h
                assert loss(p) == loss(tables)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_sgd_reads_half_tables_exactly(dtype):
    cfg = W.make_config("tiny", dtype=dtype, rows=[30, 20], B=16)
    tables = W.tables_host(cfg)
    offsets, indices = W.make_indices(cfg)
    dp = W.make_dpooled(cfg).astype(np.float64)
    co = oracle.coalesce(cfg["rows"], offsets, indices, cfg["B"])
    grad, _, new_row, _ = oracle.sgd(tables, dtype, offsets, cfg["B"], indices.size, dp, 0.01, co)
    for u in range(co["U"]):
        t, r = int(co["uniq_table"][u]), int(co["uniq_row"][u])
        wrow = (_bf16_bits_to_f64(tables[t][r]) if dtype == "bf16"
                else tables[t][r].astype(np.float64))
        np.testing.assert_allclose(new_row[u], wrow - 0.01 * grad[u], rtol=0, atol=1e-15)


# ------------------------------------------------------- row-wise AdaGrad ---

def _worked_tables(g):
    return [g["table0"].reshape(3, 2).astype(np.float32), g["table1"].reshape(2, 2).astype(np.float32)]


def test_adagrad_worked_example():
    g = _golden.load("emb_bag_worked_example.txt")
    a = _golden.load("adagrad_worked_example.txt")
    co = oracle.coalesce([3, 2], g["offsets"], g["indices"], 2)
    _, _, ns, _, nr, _ = oracle.adagrad(_worked_tables(g), "f32", g["offsets"], 2, 6, g["dpooled"].reshape(2, 2, 2),
                                        float(a["lr"][0]), float(a["eps"][0]), a["state"], co)
    np.testing.assert_array_equal(ns, a["new_state"])
    np.testing.assert_allclose(nr.reshape(-1), a["new_row"], rtol=1e-15, atol=0)


def _one_lookup(c, d=8, w=None):
    """One table, one bag holding one lookup of row 2, pooled gradient c everywhere."""
    tables = [np.zeros((4, d), dtype=np.float32) if w is None else w]
    offsets, indices = np.array([0, 1]), np.array([2])
    co = oracle.coalesce([4], offsets, indices, 1)
    return tables, offsets, co, np.full((1, 1, d), c)


def test_adagrad_constant_gradient_closed_form():
    # from s = 0 with eps = 0 a constant gradient c moves every element by lr * sign(c);
    # the second step sees s = c^2 and moves it by lr * sign(c) / sqrt(2)
    lr, c = 0.25, -0.75
    tables, offsets, co, dp = _one_lookup(c)
    _, _, s1, _, w1, _ = oracle.adagrad(tables, "f32", offsets, 1, 1, dp, lr, 0.0, [0.0], co)
    assert s1[0] == c * c
    np.testing.assert_array_equal(w1[0], np.full(8, lr))
    tables[0][2] = w1[0].astype(np.float32)
    _, _, s2, _, w2, _ = oracle.adagrad(tables, "f32", offsets, 1, 1, dp, lr, 0.0, s1, co)
    assert s2[0] == 2 * c * c
    np.testing.assert_allclose(w2[0], lr + lr / np.sqrt(2.0), rtol=1e-15)


def test_adagrad_first_step_is_scale_invariant():
    # s' = mean g^2 from s = 0: scaling every gradient leaves the step unchanged
    rng = np.random.default_rng(4)
    rows, T, B, d = [9, 5], 2, 6, 4
    tables = [rng.standard_normal((r, d)).astype(np.float32) for r in rows]
    offsets, indices = _csr(_random_bags(rng, T, B, rows, 4))
    dp = rng.standard_normal((B, T, d))
    co = oracle.coalesce(rows, offsets, indices, B)
    z = np.zeros(co["U"])
    r1 = oracle.adagrad(tables, "f32", offsets, B, indices.size, dp, 0.1, 0.0, z, co)[4]
    r2 = oracle.adagrad(tables, "f32", offsets, B, indices.size, dp * 1024.0, 0.1, 0.0, z, co)[4]
    np.testing.assert_allclose(r1, r2, rtol=1e-13, atol=1e-13)


def test_adagrad_with_a_huge_accumulator_is_sgd_with_a_scaled_rate():
    # s = 1e24: sqrt(s') = 1e12 up to a relative 1e-20, so the step is SGD at lr / 1e12
    rng = np.random.default_rng(6)
    rows, T, B, d = [7, 8, 3], 3, 10, 3
    tables = [rng.standard_normal((r, d)).astype(np.float32) for r in rows]
    offsets, indices = _csr(_random_bags(rng, T, B, rows, 5))
    dp = rng.standard_normal((B, T, d))
    co = oracle.coalesce(rows, offsets, indices, B)
    lr = 3e11
    g, _, _, _, nr, _ = oracle.adagrad(tables, "f32", offsets, B, indices.size, dp, lr, 0.0, np.full(co["U"], 1e24), co)
    g2, _, sgd_row, _ = oracle.sgd(tables, "f32", offsets, B, indices.size, dp, lr / 1e12, co)
    np.testing.assert_array_equal(g, g2)
    np.testing.assert_allclose(nr, sgd_row, rtol=1e-14, atol=1e-14)


def test_adagrad_zero_rate_and_zero_gradient():
    # lr = 0 keeps the row and still grows the accumulator; a zero gradient keeps both
    w = np.arange(32, dtype=np.float32).reshape(4, 8)
    tables, offsets, co, dp = _one_lookup(0.5, w=w)
    _, _, s, _, nr, _ = oracle.adagrad(tables, "f32", offsets, 1, 1, dp, 0.0, 1e-8, [2.0], co)
    assert s[0] == 2.0 + 0.25
    np.testing.assert_array_equal(nr[0], w[2])
    tables, offsets, co, dp = _one_lookup(0.0, w=w)
    _, _, s, _, nr, _ = oracle.adagrad(tables, "f32", offsets, 1, 1, dp, 0.1, 1e-8, [2.0], co)
    assert s[0] == 2.0
    np.testing.assert_array_equal(nr[0], w[2])


# -------------------------------------- original embeddings alongside ---

@pytest.mark.parametrize("inc", [False, True])
def test_alongside_output_is_e0_the_embeddings_then_the_pairs(inc):
    # [e0 | e_1 .. e_N | pairs]: the copies are the inputs bit for bit and the
    # pairs are those of the plain layout (pinned above by brute force and
    # the factorization-machine identity)
    rng = np.random.default_rng(21)
    B, N, d = 3, 5, 4
    e0 = rng.standard_normal((B, d))
    emb = rng.standard_normal((B, N, d))
    y, _ = oracle.interact_fwd(e0, emb, inc, alongside=True)
    plain, _ = oracle.interact_fwd(e0, emb, inc)
    assert y.shape == (B, d * (N + 1) + oracle.num_pairs(N, inc))
    np.testing.assert_array_equal(y[:, :d], e0)
    np.testing.assert_array_equal(y[:, d:d * (N + 1)], emb.reshape(B, N * d))
    np.testing.assert_array_equal(y[:, d * (N + 1):], plain[:, d:])


@pytest.mark.parametrize("inc", [False, True])
def test_alongside_backward_by_finite_differences(inc):
    rng = np.random.default_rng(22)
    B, N, d = 2, 3, 3
    e0 = rng.standard_normal((B, d))
    emb = rng.standard_normal((B, N, d))
    width = d * (N + 1) + oracle.num_pairs(N, inc)
    w = rng.standard_normal((B, width))
    de0, _, demb, _ = oracle.interact_bwd(e0, emb, w, inc, alongside=True)

    def loss(a, b):
        y, _ = oracle.interact_fwd(a, b, inc, alongside=True)
        return float((w * y).sum())

    h = 1e-3
    for arr, grad, which in ((e0, de0, 0), (emb, demb, 1)):
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            fd = ((loss(p, emb) - loss(m, emb)) if which == 0 else (loss(e0, p) - loss(e0, m))) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd))


# ------------------------------------------------------ row-wise int4 codec ---

def _unpack_int4(qt, d):
    """Independent numpy decode of an int4 table: codes, scales, biases."""
    qt = np.asarray(qt, dtype=np.uint8)
    codes = np.empty((qt.shape[0], d), dtype=np.int64)
    codes[:, 0::2] = qt[:, :d // 2] & 15
    codes[:, 1::2] = qt[:, :d // 2] >> 4
    s = qt[:, d // 2:d // 2 + 4].copy().view(np.float32)[:, 0].astype(np.float64)
    b = qt[:, d // 2 + 4:d // 2 + 8].copy().view(np.float32)[:, 0].astype(np.float64)
    return codes, s, b


def test_int4_worked_example():
    g = _golden.load("int4_worked_example.txt")
    q = oracle.quantize_int4(g["row"].reshape(1, 4).astype(np.float32), "f32")
    np.testing.assert_array_equal(q[0], g["bytes"].astype(np.uint8))
    pooled, _ = oracle.emb_bag_fwd([q], "int4", np.array([0, 1]), np.array([0]), 1, d=4)
    np.testing.assert_array_equal(pooled[0, 0], g["decoded"])


def test_int4_values_on_the_grid_round_trip_exactly():
    # rows lo + k s with s a power of two and k = 0..15 (both ends present)
    rng = np.random.default_rng(31)
    d, R = 24, 40
    lo = rng.integers(-64, 64, R).astype(np.float64) / 8
    s = 2.0 ** rng.integers(-6, 2, R).astype(np.float64)
    k = rng.integers(0, 16, (R, d))
    k[:, 0], k[:, 1] = 0, 15
    w = (lo[:, None] + s[:, None] * k).astype(np.float32)
    q = oracle.quantize_int4(w, "f32")
    codes, sc, bi = _unpack_int4(q, d)
    np.testing.assert_array_equal(codes, k)
    np.testing.assert_array_equal(sc, s)
    np.testing.assert_array_equal(bi, lo)
    assert oracle.int4_row_bytes(d) == 32 and q.shape == (R, 32) and not q[:, 20:].any()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_int4_error_is_at_most_half_a_step(dtype):
    rng = np.random.default_rng(32)
    w = rng.standard_normal((50, 64)).astype(np.float32)
    if dtype == "f16":
        w = w.astype(np.float16)
    elif dtype == "bf16":
        w = W.f32_to_bf16_bits(w)
    q = oracle.quantize_int4(w, dtype)
    codes, s, b = _unpack_int4(q, 64)
    vals = oracle.decode(w, dtype)
    np.testing.assert_array_equal(b, vals.min(axis=1).astype(np.float32))
    assert np.all(codes >= 0) and np.all(codes <= 15)
    err = np.abs(b[:, None] + s[:, None] * codes - vals)
    assert np.all(err <= s[:, None] * (0.5 + 1e-5))


def test_int4_constant_row_and_signed_zero():
    w = np.zeros((3, 8), dtype=np.float32)
    w[0] = 2.5
    w[1] = -0.0
    w[2, ::2] = -0.0  # a mix of -0 and +0 is a constant row too
    q = oracle.quantize_int4(w, "f32")
    codes, s, b = _unpack_int4(q, 8)
    assert np.all(codes == 0) and np.all(s == 0)
    np.testing.assert_array_equal(b, [2.5, 0.0, 0.0])
    assert not np.signbit(q[1, 8:12].copy().view(np.float32))[0]  # the stored bias is +0


def test_int4_pooling_sums_the_decoded_rows():
    rng = np.random.default_rng(33)
    rows, T, B, d = [13, 6], 2, 9, 16
    tables = [oracle.quantize_int4(rng.standard_normal((r, d)).astype(np.float32), "f32") for r in rows]
    offsets, indices = _csr(_random_bags(rng, T, B, rows, 5))
    pooled, _ = oracle.emb_bag_fwd(tables, "int4", offsets, indices, B, d=d)
    for t in range(T):
        codes, s, b = _unpack_int4(tables[t], d)
        dec = b[:, None] + s[:, None] * codes
        for bb in range(B):
            lo, hi = offsets[t * B + bb], offsets[t * B + bb + 1]
            np.testing.assert_allclose(pooled[bb, t], dec[indices[lo:hi]].sum(axis=0), rtol=1e-14, atol=1e-14)


# ------------------------------------------------------ the parallel build ---

def test_openmp_build_gives_identical_results():
    # the OpenMP build of the oracle (used only to time it on all host cores)
    # computes every output element in the same order: identical bits
    cfg = W.make_config("multi-hot", B=200, rows=[5000, 70000, 123, 9])
    host = W.tables_host(cfg)
    off, idx = W.make_indices(cfg)
    e0, dy = W.make_e0(cfg), W.make_dy(cfg)

    def run():
        p, pm = oracle.emb_bag_fwd(host, "f16", off, idx, cfg["B"])
        y = oracle.interact_fwd(e0, p, False, emb_mag=pm)
        a = oracle.interact_bwd(e0, p, dy, False, emb_mag=pm)
        co = oracle.coalesce(cfg["rows"], off, idx, cfg["B"])
        s = oracle.sgd(host, "f16", off, cfg["B"], idx.size, a[2], 0.01, co, dpooled_mag=a[3])
        g = oracle.adagrad(host, "f16", off, cfg["B"], idx.size, a[2], 0.01, 1e-8, np.ones(co["U"]), co)
        return [p, pm, *y, *a, *s, *g]

    try:
        serial = run()
        if not oracle.use_openmp(True):
            pytest.skip("no OpenMP build of the oracle on this host")
        parallel = run()
    finally:
        oracle.use_openmp(False)
    for x, z in zip(serial, parallel):
        np.testing.assert_array_equal(x, z)
