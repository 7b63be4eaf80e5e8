"""Element-wise comparison of GPU results with the oracle.

A float element passes when |gpu - ref| <= rel * mag, where ref is the
oracle's fp64 value and mag its magnitude (the same computation on absolute
values, a bound on the rounding error of any summation order).  rel is 1e-5
for fp32 tables and 2e-3 for fp16/bf16 tables.  A value stored back into a
half-precision table may also differ by one unit in the last place of that
type (the rounding of the fp32 result to the table type).
"""
import numpy as np

REL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


def ulp(ref, dtype):
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    if dtype == "f16":
        return np.spacing(ref.astype(np.float16)).astype(np.float64)
    if dtype == "bf16":
        e = np.floor(np.log2(np.maximum(ref, 2.0 ** -126)))
        return 2.0 ** (e - 7)
    return np.spacing(ref.astype(np.float32)).astype(np.float64)


def assert_close(gpu, ref, mag, rel, what, table_dtype=None):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mag = np.asarray(mag, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    tol = rel * mag
    if table_dtype in ("f16", "bf16"):
        tol = tol + ulp(ref, table_dtype)
    err = np.abs(gpu - ref)
    bad = ~(err <= tol)  # also catches NaN
    if bad.any():
        idx = np.argwhere(bad)[:5]
        lines = [f"{tuple(i)}: gpu={gpu[tuple(i)]!r} ref={ref[tuple(i)]!r} mag={mag[tuple(i)]!r}"
                 for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside "
                             f"rel {rel} x magnitude\n" + "\n".join(lines))


def bf16_bits_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def table_f64(host_table, dtype):
    """fp64 values of a host table (bf16 as uint16 bits)."""
    if dtype == "bf16":
        return bf16_bits_to_f64(host_table)
    return np.asarray(host_table, dtype=np.float64)


def device_table_f64(dev_table, dtype):
    import torch
    if dtype == "bf16":
        return bf16_bits_to_f64(dev_table.view(torch.int16).cpu().numpy().view(np.uint16))
    return dev_table.float().cpu().numpy().astype(np.float64)


def device_table_bits(dev_table):
    """Raw storage bits of a device table, for bit-exact comparisons."""
    import torch
    if dev_table.dtype == torch.float32:
        return dev_table.view(torch.int32).cpu().numpy()
    return dev_table.view(torch.int16).cpu().numpy()


def host_table_bits(host_table, dtype):
    if dtype == "f32":
        return np.asarray(host_table, dtype=np.float32).view(np.int32)
    if dtype == "f16":
        return np.asarray(host_table, dtype=np.float16).view(np.int16)
    return np.asarray(host_table, dtype=np.uint16).view(np.int16)
