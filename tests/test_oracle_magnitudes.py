"""Pins for the oracle's magnitudes: the bounds every float parity test
scales its tolerance by.

Next to each float result f the oracle returns a magnitude m, and a GPU value
x passes when |x - f| <= rel * m.  For a sum of products m is the same sum
over absolute values; it is then also the largest first-order change of f
when one class of inputs moves by rel times its own magnitude.  A slip in a
magnitude (a dropped factor of two on self pairs, |g| where the gradient's
magnitude belongs, a term counted twice) would loosen or tighten every parity
test that uses it without any value changing, so each magnitude is checked
here against things that do not read the oracle's formula back:

* closed forms on absolute values: numpy matrix products, dictionary sums
  over the lookups;
* the oracle's value path, pinned elsewhere (finite differences, closed
  forms, brute force), run on absolute inputs: for the linear and bilinear
  steps the magnitude is that value;
* sensitivities measured by differences: sum_x |df/dx| m_x, which the
  magnitude must equal (linear steps) or bound (row-wise AdaGrad), and
  random or worst-case input perturbations of relative size rel, whose
  effect must stay within rel * m.

Row-wise AdaGrad is not a sum of products; its magnitudes are the
first-order bounds stated in the oracle (accumulator: |s| plus the mean of
2|g| grad_mag + g^2; row: |w| + k (grad_mag + |g|) plus the effect of the
accumulator's bound on the step size k = lr / (sqrt(s') + eps)).  They are
restated here from that statement, measured against the sensitivities, and
shown to hold under perturbation.
"""
import collections

import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import _csr, _random_bags


def _stack(e0, emb):
    return np.concatenate([e0[:, None, :], emb], axis=1)


def _pair_matrix(vals, F, inc):
    """Pair values [B][P] placed at (i, j), j < i (or j <= i), in the output order."""
    B = vals.shape[0]
    rr, cc = np.tril_indices(F, k=0 if inc else -1)  # row i ascending, column j ascending
    G = np.zeros((B, F, F))
    G[:, rr, cc] = vals
    return G


def _interact_inputs(rng, B, N, d, inc, alongside, with_mags):
    e0 = rng.standard_normal((B, d))
    emb = rng.standard_normal((B, N, d))
    width = d * (N + 1 if alongside else 1) + oracle.num_pairs(N, inc)
    dy = rng.standard_normal((B, width))
    if not with_mags:
        return e0, emb, dy, None, None, None
    # magnitudes of chained inputs: at least |x|, and not proportional to it
    grow = lambda x: np.abs(x) * (1.0 + rng.random(x.shape)) + 0.25 * rng.random(x.shape)
    return e0, emb, dy, grow(e0), grow(emb), grow(dy)


def _or_abs(mag, x):
    return np.abs(x) if mag is None else mag


# ------------------------------------------------- interaction backward ---

@pytest.mark.parametrize("inc", [False, True])
@pytest.mark.parametrize("alongside", [False, True])
@pytest.mark.parametrize("with_mags", [False, True])
def test_interact_bwd_magnitude_closed_form(inc, alongside, with_mags):
    # dZ = (G + G^T) Z, so its magnitude is (|G| + |G|^T) |Z| (a self pair
    # counts 2 |g_ii| |z_i|), plus the gradient of e0's copy for e0 and, with
    # the embeddings alongside, the gradient of each embedding's copy
    rng = np.random.default_rng(21)
    B, N, d = 4, 6, 5
    F = N + 1
    e0, emb, dy, e0m, embm, dym = _interact_inputs(rng, B, N, d, inc, alongside, with_mags)
    _, de0_mag, _, demb_mag = oracle.interact_bwd(e0, emb, dy, inc, e0_mag=e0m, emb_mag=embm, dy_mag=dym,
                                                  alongside=alongside)
    gm = _or_abs(dym, dy)
    o = d * F if alongside else d
    Gm = _pair_matrix(gm[:, o:], F, inc)
    Zm = _stack(_or_abs(e0m, e0), _or_abs(embm, emb))
    dZm = (Gm + np.swapaxes(Gm, 1, 2)) @ Zm
    np.testing.assert_allclose(de0_mag, gm[:, :d] + dZm[:, 0], rtol=1e-13, atol=0)
    expect = dZm[:, 1:].copy()
    if alongside:
        expect += gm[:, d:o].reshape(B, N, d)
    np.testing.assert_allclose(demb_mag, expect, rtol=1e-13, atol=0)


@pytest.mark.parametrize("inc", [False, True])
@pytest.mark.parametrize("alongside", [False, True])
@pytest.mark.parametrize("with_mags", [False, True])
def test_interact_bwd_magnitude_is_the_value_on_absolute_inputs(inc, alongside, with_mags):
    rng = np.random.default_rng(22)
    e0, emb, dy, e0m, embm, dym = _interact_inputs(rng, 3, 5, 4, inc, alongside, with_mags)
    _, de0_mag, _, demb_mag = oracle.interact_bwd(e0, emb, dy, inc, e0_mag=e0m, emb_mag=embm, dy_mag=dym,
                                                  alongside=alongside)
    de0_abs, _, demb_abs, _ = oracle.interact_bwd(_or_abs(e0m, e0), _or_abs(embm, emb), _or_abs(dym, dy), inc,
                                                  alongside=alongside)
    np.testing.assert_allclose(de0_mag, de0_abs, rtol=1e-13, atol=0)
    np.testing.assert_allclose(demb_mag, demb_abs, rtol=1e-13, atol=0)


def _jacobian(f, x):
    """Columns f(x + e_k) - f(x) of a map that is affine in x (exact up to fp64 rounding)."""
    f0 = f(x)
    cols = []
    for k in np.ndindex(x.shape):
        xp = x.copy()
        xp[k] += 1.0
        cols.append(f(xp) - f0)
    return np.stack(cols, axis=-1)


@pytest.mark.parametrize("inc", [False, True])
@pytest.mark.parametrize("alongside", [False, True])
def test_interact_bwd_magnitude_is_the_sensitivity_to_each_input(inc, alongside):
    # the backward is linear in dy and, for fixed dy, affine in Z: the largest
    # change of an output under |d dy| <= rel |dy| is rel * sum_k |J_k| |dy_k|,
    # and that must be the magnitude; under |dZ| <= rel |Z| it is the magnitude
    # less the copies' share (|dy| of e0's copy, and of the embeddings' copies)
    rng = np.random.default_rng(23)
    B, N, d = 1, 3, 3
    e0, emb, dy, _, _, _ = _interact_inputs(rng, B, N, d, inc, alongside, False)
    F = N + 1
    _, de0_mag, _, demb_mag = oracle.interact_bwd(e0, emb, dy, inc, alongside=alongside)
    mag = np.concatenate([de0_mag.reshape(-1), demb_mag.reshape(-1)])

    def out(e0_, emb_, dy_):
        a, _, b, _ = oracle.interact_bwd(e0_, emb_, dy_, inc, alongside=alongside)
        return np.concatenate([a.reshape(-1), b.reshape(-1)])

    Jdy = _jacobian(lambda x: out(e0, emb, x), dy)
    np.testing.assert_allclose(np.abs(Jdy) @ np.abs(dy).reshape(-1), mag, rtol=1e-12, atol=0)
    z = _stack(e0, emb)
    Jz = _jacobian(lambda x: out(x[:, 0], x[:, 1:], dy), z)
    copies = np.zeros((F, d))
    copies[0] = np.abs(dy[0, :d])
    if alongside:
        copies[1:] = np.abs(dy[0, d:d * F]).reshape(N, d)
    np.testing.assert_allclose(np.abs(Jz) @ np.abs(z).reshape(-1), mag - copies.reshape(-1), rtol=1e-12,
                               atol=1e-15)


@pytest.mark.parametrize("inc", [False, True])
def test_interact_bwd_perturbed_inputs_stay_within_the_bound(inc):
    # every input moved by up to rel/2 of its magnitude (random signs, and the
    # signs that push one output up the most): each term g z moves by at most
    # rel (1 + rel/4) of its magnitude
    rng = np.random.default_rng(24)
    B, N, d = 3, 5, 4
    rel = 1e-3
    e0, emb, dy, e0m, embm, dym = _interact_inputs(rng, B, N, d, inc, False, True)
    de0, de0_mag, demb, demb_mag = oracle.interact_bwd(e0, emb, dy, inc, e0_mag=e0m, emb_mag=embm, dy_mag=dym)
    bound0, bound1 = rel * (1 + rel) * de0_mag, rel * (1 + rel) * demb_mag
    for _ in range(40):
        s = lambda x, m: x + 0.5 * rel * m * rng.uniform(-1, 1, x.shape)
        a, _, b, _ = oracle.interact_bwd(s(e0, e0m), s(emb, embm), s(dy, dym), inc)
        assert np.all(np.abs(a - de0) <= bound0) and np.all(np.abs(b - demb) <= bound1)
    # worst case for e0's element 0 of sample 0: every pair term of row 0 and e0's copy pushed up
    F = N + 1
    G = _pair_matrix(dy[:, d:], F, inc)
    Gs = G + np.swapaxes(G, 1, 2)
    z = _stack(e0, emb)
    zm = _stack(e0m, embm)
    sz = np.sign(Gs[0, 0])[:, None] * np.ones((F, d))  # z_j pushed along the sign of its coefficient
    z2 = z.copy()
    z2[0] += 0.5 * rel * zm[0] * sz
    sg = np.zeros_like(dy)
    sg[0, 0] = 1.0
    Gsign = np.sign(z[0, :, 0])  # g_0j pushed along the sign of z_j[0]
    rr, cc = np.tril_indices(F, k=0 if inc else -1)
    for p, (i, j) in enumerate(zip(rr, cc)):
        if i == 0 or j == 0:
            sg[0, d + p] = Gsign[j if i == 0 else i]
    dy2 = dy + 0.5 * rel * dym * sg
    a, _, _, _ = oracle.interact_bwd(z2[:, 0], z2[:, 1:], dy2, inc)
    assert a[0, 0] - de0[0, 0] <= bound0[0, 0]
    # the push reaches at least rel/2 of the magnitude: the bound is not loose by more than 2x
    assert a[0, 0] - de0[0, 0] >= 0.5 * rel * de0_mag[0, 0] * (1 - 1e-9) - 0.5 * rel * (dym[0, 0] - abs(dy[0, 0]))


# ----------------------------------------------------------- SGD update ---

def _sgd_case(rng, dtype, with_mag, max_len=6):
    rows = [7, 12, 5]
    T, B, d = 3, 9, 4
    vals = [rng.standard_normal((r, d)) * 0.5 for r in rows]
    if dtype == "f32":
        tables = [v.astype(np.float32) for v in vals]
        wvals = [t.astype(np.float64) for t in tables]
    elif dtype == "f16":
        tables = [v.astype(np.float16) for v in vals]
        wvals = [t.astype(np.float64) for t in tables]
    else:  # bf16 bit patterns, truncated from fp32 (any pattern is a valid table)
        tables = [(v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16) for v in vals]
        wvals = [((t.astype(np.uint32) << 16).view(np.float32)).astype(np.float64) for t in tables]
    bags = _random_bags(rng, T, B, rows, max_len)
    offsets, indices = _csr(bags)
    dp = rng.standard_normal((B, T, d))
    dpm = np.abs(dp) * (1.0 + rng.random(dp.shape)) if with_mag else None
    return rows, T, B, d, tables, wvals, bags, offsets, indices, dp, dpm


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("with_mag", [False, True])
@pytest.mark.parametrize("lr", [0.1, -0.3, 0.0])
def test_sgd_magnitudes_by_brute_force(dtype, with_mag, lr):
    rng = np.random.default_rng(31)
    rows, T, B, d, tables, wvals, bags, offsets, indices, dp, dpm = _sgd_case(rng, dtype, with_mag)
    co = oracle.coalesce(rows, offsets, indices, B)
    _, gm, _, nrm = oracle.sgd(tables, dtype, offsets, B, indices.size, dp, lr, co, dpooled_mag=dpm)
    per_term = np.abs(dp) if dpm is None else dpm
    brute = collections.defaultdict(lambda: np.zeros(d))
    for t in range(T):
        for b in range(B):
            for r in bags[t][b]:
                brute[(t, int(r))] += per_term[b, t]
    assert co["U"] == len(brute)
    for u in range(co["U"]):
        key = (int(co["uniq_table"][u]), int(co["uniq_row"][u]))
        np.testing.assert_allclose(gm[u], brute[key], rtol=1e-14, atol=0)
        np.testing.assert_allclose(nrm[u], np.abs(wvals[key[0]][key[1]]) + abs(lr) * brute[key], rtol=1e-14,
                                   atol=0)


@pytest.mark.parametrize("with_mag", [False, True])
def test_sgd_magnitude_is_the_value_on_absolute_inputs(with_mag):
    # w - lr g on |w|, the gradients' magnitudes and -|lr|
    rng = np.random.default_rng(32)
    rows, T, B, d, tables, _, _, offsets, indices, dp, dpm = _sgd_case(rng, "f32", with_mag)
    lr = 0.37
    co = oracle.coalesce(rows, offsets, indices, B)
    _, gm, _, nrm = oracle.sgd(tables, "f32", offsets, B, indices.size, dp, lr, co, dpooled_mag=dpm)
    g_abs, _, nr_abs, _ = oracle.sgd([np.abs(t) for t in tables], "f32", offsets, B, indices.size,
                                     _or_abs(dpm, dp), -lr, co)
    np.testing.assert_allclose(gm, g_abs, rtol=1e-14, atol=0)
    np.testing.assert_allclose(nrm, nr_abs, rtol=1e-14, atol=0)


def test_sgd_worst_case_perturbation_attains_the_bound():
    # the update is linear in (w, dpooled): moving every w by +rel |w| and
    # every pooled gradient by -sign(lr) rel |dp| moves every updated element
    # up by exactly rel * magnitude (dyadic values keep it exact in fp32)
    rng = np.random.default_rng(33)
    rows, T, B, d = [6, 9], 2, 8, 3
    rel = 2.0 ** -8
    tables = [(rng.integers(-256, 256, (r, d)) / 256).astype(np.float32) for r in rows]
    offsets, indices = _csr(_random_bags(rng, T, B, rows, 5))
    dp = rng.integers(-64, 64, (B, T, d)) / 64
    lr = 0.125
    co = oracle.coalesce(rows, offsets, indices, B)
    _, _, nr, nrm = oracle.sgd(tables, "f32", offsets, B, indices.size, dp, lr, co)
    up = [t + np.float32(rel) * np.abs(t) for t in tables]
    assert all(np.array_equal(u.astype(np.float64), t + rel * np.abs(t.astype(np.float64)))
               for u, t in zip(up, tables))
    _, _, nr2, _ = oracle.sgd(up, "f32", offsets, B, indices.size, dp - np.sign(lr) * rel * np.abs(dp), lr, co)
    np.testing.assert_allclose(nr2 - nr, rel * nrm, rtol=1e-12, atol=1e-15)


# ------------------------------------------------------ row-wise AdaGrad ---

def _adagrad_case(rng, d=3, max_len=5, state_scale=1.0, rows=(5, 4), B=6, w_scale=1.0):
    rows = list(rows)
    T = len(rows)
    # dyadic table values, so that a table moved by a power-of-two step stays exact in fp32
    tables = [(w_scale * rng.integers(-128, 128, (r, d)) / 128).astype(np.float32) for r in rows]
    bags = _random_bags(rng, T, B, rows, max_len)
    offsets, indices = _csr(bags)
    dp = rng.standard_normal((B, T, d))
    co = oracle.coalesce(rows, offsets, indices, B)
    state = state_scale * rng.uniform(0.0, 2.0, co["U"])
    return rows, T, B, d, tables, bags, offsets, indices, dp, co, state


def test_adagrad_magnitudes_match_their_stated_bounds():
    # gradients' magnitudes by brute force; the accumulator's and row's
    # magnitudes as the oracle states them (first-order bounds), in numpy
    rng = np.random.default_rng(41)
    rows, T, B, d, tables, bags, offsets, indices, dp, co, state = _adagrad_case(rng, d=4)
    lr, eps = 0.05, 1e-3
    g, gm, s1, s1m, nr, nrm = oracle.adagrad(tables, "f32", offsets, B, indices.size, dp, lr, eps, state, co)
    brute = collections.defaultdict(lambda: np.zeros(d))
    for t in range(T):
        for b in range(B):
            for r in bags[t][b]:
                brute[(t, int(r))] += np.abs(dp[b, t])
    for u in range(co["U"]):
        t, r = int(co["uniq_table"][u]), int(co["uniq_row"][u])
        np.testing.assert_allclose(gm[u], brute[(t, r)], rtol=1e-14, atol=0)
        sm = abs(state[u]) + np.mean(2 * np.abs(g[u]) * gm[u] + g[u] ** 2)
        np.testing.assert_allclose(s1m[u], sm, rtol=1e-14, atol=0)
        root = np.sqrt(s1[u])
        den = root + eps
        k = lr / den
        w = tables[t][r].astype(np.float64)
        rm = np.abs(w) + k * (gm[u] + np.abs(g[u])) + np.abs(g[u]) * lr * sm / (2 * root * den * den)
        np.testing.assert_allclose(nrm[u], rm, rtol=1e-13, atol=0)


def _adagrad_sensitivity(tables, offsets, B, nnz, dp, lr, eps, state, co):
    """sum_x |df/dx| |x| of the new accumulators and rows over every input x
    (pooled gradients, accumulators, table elements), by central differences."""
    def run(tabs, dp_, st_):
        _, _, s1, _, nr, _ = oracle.adagrad(tabs, "f32", offsets, B, nnz, dp_, lr, eps, st_, co)
        return s1, nr

    s0, r0 = run(tables, dp, state)
    Ss, Sr = np.zeros_like(s0), np.zeros_like(r0)
    for k in np.ndindex(dp.shape):
        h = 1e-5 * max(1.0, abs(dp[k]))
        p, m = dp.copy(), dp.copy()
        p[k] += h
        m[k] -= h
        (sp, rp), (sm, rm) = run(tables, p, state), run(tables, m, state)
        Ss += np.abs((sp - sm) / (2 * h)) * abs(dp[k])
        Sr += np.abs((rp - rm) / (2 * h)) * abs(dp[k])
    for u in range(state.size):
        h = 1e-5 * max(1.0, abs(state[u]))
        p, m = state.copy(), state.copy()
        p[u] += h
        m[u] -= h
        (sp, rp), (sm, rm) = run(tables, dp, p), run(tables, dp, m)
        Ss += np.abs((sp - sm) / (2 * h)) * abs(state[u])
        Sr += np.abs((rp - rm) / (2 * h)) * abs(state[u])
    # the new row is w - k g with k independent of w: slope 1 in its own element
    for u in range(co["U"]):
        t, r = int(co["uniq_table"][u]), int(co["uniq_row"][u])
        Sr[u] += np.abs(tables[t][r].astype(np.float64))
    return s0, r0, Ss, Sr


def test_adagrad_magnitudes_bound_the_sensitivity_to_every_input():
    rng = np.random.default_rng(42)
    rows, T, B, d, tables, bags, offsets, indices, dp, co, state = _adagrad_case(rng)
    lr, eps = 0.05, 1e-3
    _, _, _, s1m, _, nrm = oracle.adagrad(tables, "f32", offsets, B, indices.size, dp, lr, eps, state, co)
    _, _, Ss, Sr = _adagrad_sensitivity(tables, offsets, B, indices.size, dp, lr, eps, state, co)
    g = oracle.sgd(tables, "f32", offsets, B, indices.size, dp, 0.0, co)[0]
    # the accumulator's bound is its sensitivity plus the rounding of the squares, mean g^2
    np.testing.assert_allclose(s1m, Ss + np.mean(g ** 2, axis=1), rtol=1e-7, atol=0)
    # the row's bound covers its sensitivity
    assert np.all(Sr <= nrm * (1 + 1e-7))


def test_adagrad_row_magnitude_is_tight_when_the_step_is_a_long_sum():
    # zero rows, a large accumulator and long runs of lookups: the row's
    # sensitivity is about k * grad_mag and its bound adds only terms in |g|,
    # which a long sum of signed terms keeps small; a term counted twice
    # would double the bound
    rng = np.random.default_rng(43)
    rows, T, B, d = [2], 1, 100, 2
    tables = [np.zeros((2, d), dtype=np.float32)]
    bags = [[list(rng.integers(0, 2, 10)) for _ in range(B)]]
    offsets, indices = _csr(bags)
    dp = rng.standard_normal((B, T, d))
    co = oracle.coalesce(rows, offsets, indices, B)
    state = np.full(co["U"], 1e8)
    lr, eps = 0.05, 1e-3
    _, _, _, _, _, nrm = oracle.adagrad(tables, "f32", offsets, B, indices.size, dp, lr, eps, state, co)
    _, _, _, Sr = _adagrad_sensitivity(tables, offsets, B, indices.size, dp, lr, eps, state, co)
    assert np.all(Sr <= nrm * (1 + 1e-7))
    assert np.all(nrm <= 1.2 * Sr), (nrm / Sr).max()


@pytest.mark.parametrize("state_scale", [0.0, 1.0, 100.0])
def test_adagrad_perturbed_inputs_stay_within_the_bound(state_scale):
    # pooled gradients and accumulators moved by up to rel of their size
    # (random signs, many draws), table values by +-rel exactly: every new
    # accumulator and row element moves by at most rel times its magnitude
    rng = np.random.default_rng(44)
    rows, T, B, d, tables, bags, offsets, indices, dp, co, state = _adagrad_case(rng, d=4,
                                                                               state_scale=state_scale)
    lr, eps, rel = 0.05, 1e-3, 2.0 ** -12
    _, _, s1, s1m, nr, nrm = oracle.adagrad(tables, "f32", offsets, B, indices.size, dp, lr, eps, state, co)
    for _ in range(60):
        dp2 = dp * (1 + rel * rng.uniform(-1, 1, dp.shape))
        st2 = state * (1 + rel * rng.uniform(-1, 1, state.shape))
        sign = np.float32(rng.choice([-1.0, 1.0]))
        tabs2 = [t + sign * np.float32(rel) * np.abs(t) for t in tables]  # exact: dyadic values
        _, _, s2, _, r2, _ = oracle.adagrad(tabs2, "f32", offsets, B, indices.size, dp2, lr, eps, st2, co)
        assert np.all(np.abs(s2 - s1) <= rel * s1m * (1 + 1e-6))
        assert np.all(np.abs(r2 - nr) <= rel * nrm * (1 + 1e-6))
