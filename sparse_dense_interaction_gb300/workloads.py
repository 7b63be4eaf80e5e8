"""Seeded synthetic inputs for the DLRM sparse hot path.

This module only makes input data; it holds none of the path's arithmetic
(no pooling, no dot products, no sorting, no update), and it is the one
module that the CUDA path's tests and the oracle's tests share.

The workloads stand in for the click-log benchmark the DLRM notes mention
(section 6, "The MLPerf Benchmark", on the Criteo display-advertising data),
which is not available here: the shapes follow that workload (26 categorical
features, tables of up to millions of rows, one-hot or multi-hot bags) and the
index streams are Zipf-skewed or uniform.  Nothing of the dataset itself is
reproduced.

Recipe (all seeded; ``seed`` defaults to 0):

* index streams: numpy ``Generator(PCG64(SeedSequence([seed, cfg, t, s])))``
  for config id ``cfg``, table ``t`` and stream ``s`` (1 bag lengths, 2 ranks,
  3 rank-to-row scatter, 4 e0, 5 upstream gradient dY, 6 pooled gradient);
* bag lengths: fixed, or Poisson(mean) clipped to [lo, hi];
* rows: uniform over [0, R_t), or Zipf(alpha) over ranks 1..R_t by inverse
  CDF, rank k mapped to row ((k-1)*A_t + C_t) mod R_t with A_t coprime to R_t
  so that hot rows are spread over the table;
* table values: a counter-based generator, SplitMix64 (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014), keyed per
  table; element n = row*d + col of table t is mix(s_t + (n+1)*gamma), the top
  24 bits m give v = (2m - 2^24) * 2^-24 exactly in fp32, the value is
  fp32(v * fp32(1/sqrt(R_t))) rounded once more, to nearest even, into the
  table's storage type.  The same definition runs on the host here (any subset
  of rows) and on the device in ``workloads_csrc/workload_gen.cu`` (whole tables), so a
  131 GB table set never has to exist on the host;
* e0, dY and standalone pooled gradients: N(0, 1) in fp32.
"""
from __future__ import annotations

import copy
import functools
import math

import numpy as np

CONFIG_IDS = {"tiny": 0, "one-hot": 1, "multi-hot": 2, "capacity": 3,
              "interaction-heavy": 4, "multi-hot-uniform": 5}

_BASE = {
    # 8 fp32 tables x 1000 rows, d = 16, batch 128, one uniform index per bag,
    # strict pairs, forward + backward + SGD with lr 0.01.
    "tiny": dict(T=8, rows=[1000] * 8, d=16, dtype="f32", B=128,
                 bag=("fixed", 1), index=("uniform",), interaction=True,
                 include_self=False, lr=0.01, update="sgd"),
    # 26 fp32 tables, rows log-spaced 10 .. 10M, d = 64, batch 2048, one
    # Zipf(1.05) index per bag, strict pairs, forward + backward + SGD.
    "one-hot": dict(T=26, rows=[int(math.floor(10 ** (1 + 6 * t / 25) + 0.5)) for t in range(26)],
                    d=64, dtype="f32", B=2048, bag=("fixed", 1), index=("zipf", 1.05),
                    interaction=True, include_self=False, lr=0.01, update="sgd"),
    # 26 fp16 tables x 4M rows, d = 128, batch 65536, bag length Poisson(20)
    # clipped to 1..80, Zipf(1.2) indices, strict pairs, forward + backward + SGD.
    "multi-hot": dict(T=26, rows=[4_000_000] * 26, d=128, dtype="f16", B=65536,
                      bag=("poisson", 20.0, 1, 80), index=("zipf", 1.2), interaction=True,
                      include_self=False, lr=0.01, update="sgd"),
    # 8 fp32 tables x 32M rows, d = 128 (131 GB), batch 16384, 32 uniform
    # indices per bag, no interaction, forward + backward + row-wise SGD.
    "capacity": dict(T=8, rows=[32_000_000] * 8, d=128, dtype="f32", B=16384,
                     bag=("fixed", 32), index=("uniform",), interaction=False,
                     include_self=False, lr=0.01, update="sgd"),
    # 100 bf16 tables x 100k rows, d = 256, batch 8192, one uniform index per
    # bag, self-inclusive pairs, forward + backward of interaction and lookup
    # (the lookup backward yields the coalesced row gradient, no update).
    "interaction-heavy": dict(T=100, rows=[100_000] * 100, d=256, dtype="bf16", B=8192,
                              bag=("fixed", 1), index=("uniform",), interaction=True,
                              include_self=True, lr=0.0, update="grad"),
    # the multi-hot shapes with uniform indices (cache-hostile variant)
    "multi-hot-uniform": dict(T=26, rows=[4_000_000] * 26, d=128, dtype="f16", B=65536,
                              bag=("poisson", 20.0, 1, 80), index=("uniform",),
                              interaction=True, include_self=False, lr=0.01, update="sgd"),
}

ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)


def make_config(name: str, **overrides) -> dict:
    """A named configuration, optionally with fields replaced (e.g. B=256)."""
    cfg = copy.deepcopy(_BASE[name])
    cfg["name"] = name
    cfg["id"] = CONFIG_IDS[name]
    for k, v in overrides.items():
        if k == "T":
            cfg["rows"] = (list(cfg["rows"]) * ((v + len(cfg["rows"]) - 1) // len(cfg["rows"])))[:v]
        cfg[k] = v
    if "rows" in overrides and "T" not in overrides:
        cfg["T"] = len(cfg["rows"])
    assert len(cfg["rows"]) == cfg["T"]
    return cfg


def table_stream_seed(cfg: dict, t: int, seed: int = 0) -> int:
    """Key of table t's SplitMix64 stream: seed*2^32 + config id*2^16 + t."""
    return ((seed & 0xFFFFFFFF) << 32) | ((cfg["id"] & 0xFFFF) << 16) | (t & 0xFFFF)


def table_scale(rows: int) -> np.float32:
    """fp32 half-width of the uniform initial values, 1/sqrt(rows)."""
    return np.float32(1.0 / math.sqrt(rows))


def _splitmix64(state: np.ndarray) -> np.ndarray:
    z = state.copy()
    z ^= z >> np.uint64(30)
    z *= _MIX1
    z ^= z >> np.uint64(27)
    z *= _MIX2
    z ^= z >> np.uint64(31)
    return z


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))
    return ((bits + bias) >> np.uint64(16)).astype(np.uint16)


def table_rows_host(cfg: dict, t: int, row_ids, seed: int = 0) -> np.ndarray:
    """Values of the given rows of table t in storage type.

    Returns float32 or float16 arrays, or uint16 bit patterns for bf16, with
    shape [len(row_ids)][d].
    """
    d = cfg["d"]
    row_ids = np.asarray(row_ids, dtype=np.uint64).reshape(-1, 1)
    n = row_ids * np.uint64(d) + np.arange(d, dtype=np.uint64).reshape(1, -1) + np.uint64(1)
    with np.errstate(over="ignore"):
        state = np.uint64(table_stream_seed(cfg, t, seed)) + n * _GAMMA
        z = _splitmix64(state)
    m = (z >> np.uint64(40)).astype(np.int64)
    v = (2 * m - (1 << 24)).astype(np.float32) * np.float32(2.0 ** -24)
    w = (v * table_scale(cfg["rows"][t])).astype(np.float32)
    if cfg["dtype"] == "f32":
        return w
    if cfg["dtype"] == "f16":
        return w.astype(np.float16)
    return f32_to_bf16_bits(w)


def tables_host(cfg: dict, seed: int = 0) -> list:
    """All tables on the host (small configurations only)."""
    return [table_rows_host(cfg, t, np.arange(cfg["rows"][t]), seed) for t in range(cfg["T"])]


def _rng(cfg: dict, t: int, stream: int, seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, cfg["id"], t, stream])))


@functools.lru_cache(maxsize=8)
def _zipf_cdf(R: int, alpha: float) -> np.ndarray:
    w = np.arange(1, R + 1, dtype=np.float64) ** (-alpha)
    c = np.cumsum(w)
    return c / c[-1]


def _scatter_multiplier(R: int, rng: np.random.Generator) -> int:
    while True:
        a = int(rng.integers(1, max(R, 2)))
        if math.gcd(a, R) == 1:
            return a


def bag_lengths(cfg: dict, t: int, seed: int = 0) -> np.ndarray:
    kind = cfg["bag"][0]
    B = cfg["B"]
    if kind == "fixed":
        return np.full(B, cfg["bag"][1], dtype=np.int64)
    if kind == "poisson":
        _, lam, lo, hi = cfg["bag"]
        return np.clip(_rng(cfg, t, 1, seed).poisson(lam, B), lo, hi).astype(np.int64)
    if kind == "explicit":
        return np.asarray(cfg["bag"][1][t], dtype=np.int64)
    raise ValueError(kind)


def table_indices(cfg: dict, t: int, n: int, seed: int = 0) -> np.ndarray:
    R = cfg["rows"][t]
    kind = cfg["index"][0]
    if kind == "uniform":
        return _rng(cfg, t, 2, seed).integers(0, R, size=n, dtype=np.int64)
    if kind == "zipf":
        alpha = cfg["index"][1]
        u = _rng(cfg, t, 2, seed).random(n)
        rank = np.minimum(np.searchsorted(_zipf_cdf(R, alpha), u, side="right"), R - 1)
        srng = _rng(cfg, t, 3, seed)
        a = _scatter_multiplier(R, srng)
        c = int(srng.integers(0, R))
        return (rank.astype(np.int64) * a + c) % R
    raise ValueError(kind)


def make_indices(cfg: dict, seed: int = 0):
    """Table-major CSR lookups: offsets [T*B+1] and indices [nnz], int64."""
    T, B = cfg["T"], cfg["B"]
    lengths = [bag_lengths(cfg, t, seed) for t in range(T)]
    offsets = np.zeros(T * B + 1, dtype=np.int64)
    np.cumsum(np.concatenate(lengths), out=offsets[1:])
    indices = np.empty(int(offsets[-1]), dtype=np.int64)
    for t in range(T):
        lo, hi = offsets[t * B], offsets[(t + 1) * B]
        indices[lo:hi] = table_indices(cfg, t, int(hi - lo), seed)
    return offsets, indices


def num_pairs(T: int, include_self: bool) -> int:
    """Interaction width over F = T + 1 vectors (a shape, used to size buffers)."""
    F = T + 1
    return F * (F + 1) // 2 if include_self else F * (F - 1) // 2


def make_e0(cfg: dict, seed: int = 0) -> np.ndarray:
    return _rng(cfg, 0, 4, seed).standard_normal((cfg["B"], cfg["d"]), dtype=np.float32)


def make_dy(cfg: dict, seed: int = 0) -> np.ndarray:
    width = cfg["d"] + num_pairs(cfg["T"], cfg["include_self"])
    return _rng(cfg, 0, 5, seed).standard_normal((cfg["B"], width), dtype=np.float32)


def make_dpooled(cfg: dict, seed: int = 0) -> np.ndarray:
    return _rng(cfg, 0, 6, seed).standard_normal((cfg["B"], cfg["T"], cfg["d"]),
                                                 dtype=np.float32)


def table_bytes(cfg: dict) -> int:
    return sum(cfg["rows"]) * cfg["d"] * ELEM_BYTES[cfg["dtype"]]


_fill_lib = None


def _load_fill():
    global _fill_lib
    if _fill_lib is None:
        import ctypes
        import os

        from . import build as _build
        path = _build.lib_path("libdlrm_workloads.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first "
                               "(python -m sparse_dense_interaction_gb300.build)")
        lib = ctypes.CDLL(path)
        lib.dlrm_workload_fill_table.restype = ctypes.c_int
        lib.dlrm_workload_fill_table.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                                 ctypes.c_int, ctypes.c_uint64, ctypes.c_float,
                                                 ctypes.c_void_p]
        _fill_lib = lib
    return _fill_lib


_DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


def make_tables_device(cfg: dict, seed: int = 0, device="cuda"):
    """All tables of a configuration, allocated and filled on the GPU.

    Same values as :func:`table_rows_host`, generated by the device copy of
    the counter-based generator (workload input only).
    """
    import torch
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[cfg["dtype"]]
    lib = _load_fill()
    stream = torch.cuda.current_stream(device)
    tables = []
    for t in range(cfg["T"]):
        tab = torch.empty((cfg["rows"][t], cfg["d"]), dtype=tdt, device=device)
        st = lib.dlrm_workload_fill_table(tab.data_ptr(), _DTYPE_CODE[cfg["dtype"]], cfg["rows"][t],
                                          cfg["d"], table_stream_seed(cfg, t, seed),
                                          float(table_scale(cfg["rows"][t])), stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"table fill failed with status {st}")
        tables.append(tab)
    return tables


def tables_to_device(host_tables, dtype: str, device="cuda"):
    """Uploads host tables (bf16 given as uint16 bit patterns)."""
    import torch
    out = []
    for h in host_tables:
        if dtype == "bf16":
            out.append(torch.from_numpy(h.view(np.int16).copy()).to(device).view(torch.bfloat16))
        else:
            out.append(torch.from_numpy(np.ascontiguousarray(h)).to(device))
    return out
