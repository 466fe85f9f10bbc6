"""Helpers shared by the GPU parity tests (no arithmetic of the method here)."""
import numpy as np
import torch


def u16(t: torch.Tensor) -> np.ndarray:
    """bfloat16 bit patterns of a tensor (any device) as numpy uint16."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_ulp(v) -> np.ndarray:
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.maximum(np.exp2(e - 7), 2.0 ** -133)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str = ""):
    got = np.asarray(got).reshape(want.shape)
    if np.array_equal(got, want):
        return
    bad = np.argwhere(got != want)
    n = len(bad)
    i = tuple(bad[0])
    raise AssertionError(f"{what}: {n} of {want.size} elements differ; first at {i}: "
                         f"got 0x{int(got[i]):04x} want 0x{int(want[i]):04x}")


def assert_high_close(got_bits: np.ndarray, exact: np.ndarray, mag: np.ndarray, ulps: float = 2.0,
                      what: str = ""):
    """The single-pass result is within `ulps` bfloat16 ulps of the largest term
    of the exact (binary64) result."""
    g = f32(np.asarray(got_bits).reshape(exact.shape)).astype(np.float64)
    err = np.abs(g - exact)
    lim = ulps * bf16_ulp(mag)
    bad = err > lim
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond {ulps} ulp; first at {i}: "
                             f"got {g[i]!r} exact {exact[i]!r} mag {mag[i]!r}")
    return float((err / bf16_ulp(mag)).max())


def guarded(shape, device, fill=0x7E7E, pad=4096):
    """An output tensor placed inside a larger buffer whose margins hold a
    sentinel pattern; returns (view, check) where check() asserts the margins
    are untouched."""
    n = int(np.prod(shape))
    buf = torch.full((pad + n + pad,), fill, dtype=torch.int16, device=device)
    view = buf[pad:pad + n].view(torch.bfloat16).view(shape)

    def check():
        b = buf.cpu().numpy().view(np.uint16)
        assert np.all(b[:pad] == fill) and np.all(b[pad + n:] == fill), "write outside the view"

    return view, check


def par_rows(fn, rows: int, seq=None, align: int = 1, parts=None) -> list:
    """Call fn(lo, hi) on disjoint row ranges that cover [0, rows), from a pool
    of host threads, and return the results in row order.

    The oracle is plain C called through ctypes, which releases the GIL for the
    call, and it keeps no state between calls, so the ranges run on every host
    core at once.  Each output row depends only on its own input rows and its
    modulation row, so splitting the rows changes no bit of the result.  Ranges
    start at multiples of `align` (128 keeps NVFP4 scale tiles whole) and never
    cross a multiple of `seq` (so a range has one per-sample modulation row)."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    n = parts or max(1, 4 * (os.cpu_count() or 1))
    length = max(align, -(-rows // n))
    length = -(-length // align) * align
    bounds = []
    for s0 in range(0, rows, seq or rows):
        s1 = min(rows, s0 + (seq or rows))
        for lo in range(s0, s1, length):
            bounds.append((lo, min(s1, lo + length)))
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        futs = [ex.submit(fn, lo, hi) for lo, hi in bounds]
        return [f.result() for f in futs]


def host_rows(t: torch.Tensor) -> np.ndarray:
    """bfloat16 bit patterns of a device tensor as a contiguous [rows, D] host array."""
    return u16(t).reshape(-1, t.shape[-1])
