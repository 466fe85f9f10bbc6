"""Parity of the FP8 producers (LN + AdaLN, and gated residual + LN + AdaLN,
each with a static-scale E4M3 copy of the bf16 output).

Lossless: the bf16 output and every E4M3 byte equal the oracle's (the
quantiser applied to the oracle's bf16 output with the correctly rounded
1/scale).  High: the bf16 output is graded as before, and the E4M3 copy must
be the quantisation of the bf16 output the kernel wrote (checked with
PyTorch's float8_e4m3fn conversion where it does not saturate).  The E4M3
conversion itself is pinned on the GPU by mbx_selftest(5) over every binary32
pattern.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_bits_equal, assert_high_close, u16

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16 = torch.bfloat16


@pytest.fixture(scope="module")
def mbx():
    import modulation_bit_exact_gb300 as m
    m.lib()
    return m


def _b8(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def _scale(v):
    return torch.tensor([v], dtype=torch.float32, device=DEV)


def test_selftest_e4m3_conversion(mbx):
    assert tuple(mbx.selftest(5)) == (0, 0)


def _self_consistent(out, q, scale):
    """q is the E4M3 copy of the bf16 `out` (property check, any variant)."""
    inv = np.float32(1.0) / np.float32(scale)
    prod = (out.float().cpu().numpy() * inv).astype(np.float32)
    got = _b8(q)
    inr = np.abs(prod) < 448
    want = torch.from_numpy(prod[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[inr], want)
    assert np.all(got[~inr & (prod > 0)] == 0x7E) and np.all(got[~inr & (prod < 0)] == 0xFE)


@pytest.mark.parametrize("scale", [1.0, 0.0173, 0.004])
def test_ln_modulate_fp8_image_dit(mbx, scale):
    d = synth.image_dit_block()
    x, sc, sh = (d[k].to(DEV) for k in ("x", "scale", "shift"))
    X, SC, SH = u16(d["x"]).reshape(-1, 3072), u16(d["scale"]), u16(d["shift"])
    out, q = mbx.ln_modulate_fp8(x, sc, sh, _scale(scale))
    want = oracle.ln_modulate(X, SC, SH, 1e-6)
    assert_bits_equal(u16(out).reshape(-1, 3072), want, "bf16")
    assert_bits_equal(_b8(q).reshape(-1, 3072), oracle.quant_e4m3(want, scale), "e4m3")
    out_h, q_h = mbx.ln_modulate_fp8(x, sc, sh, _scale(scale), variant="high")
    _self_consistent(out_h, q_h, scale)


@pytest.mark.parametrize("D,rows,mrows,shift", [(1024, 300, 3, 0), (5120, 97, 97, 0), (1000, 50, 2, 0),
                                                (2048, 64, 2, 1), (8192, 40, 40, 0)])
def test_ln_modulate_fp8_shapes(mbx, D, rows, mrows, shift):
    """Per-sample (staged), per-token (ring), ragged D and a misaligned view
    (the pipelined kernel's FP8 store and the separate quantiser)."""
    g = torch.Generator().manual_seed(D + rows)
    x = (torch.randn(rows, D, generator=g) * 2).to(BF16)
    sc = (0.1 * torch.randn(mrows, D, generator=g)).to(BF16)
    sh = (0.1 * torch.randn(mrows, D, generator=g)).to(BF16)
    xd = x.to(DEV)
    if shift:
        buf = torch.empty(rows * D + 8, dtype=BF16, device=DEV)
        xd = buf[1:1 + rows * D].view(rows, D)
        xd.copy_(x.to(DEV))
    out, q = mbx.ln_modulate_fp8(xd, sc.to(DEV), sh.to(DEV), _scale(0.011))
    want = oracle.ln_modulate(u16(x), u16(sc), u16(sh), 1e-6)
    assert_bits_equal(u16(out), want, "bf16")
    assert_bits_equal(_b8(q), oracle.quant_e4m3(want, 0.011), "e4m3")


@pytest.mark.parametrize("bias,D", [(True, 3072), (False, 3072), (True, 8192)])
def test_gated_fp8(mbx, bias, D):
    """D = 8192 takes the composed path (gated add, then LN with the FP8 store)."""
    g = torch.Generator().manual_seed(5)
    rows = 2 * 611 if D == 3072 else 2 * 97
    r = torch.randn(rows, D, generator=g).to(BF16)
    u = torch.randn(rows, D, generator=g).to(BF16)
    gt, sc, sh = ((0.1 * torch.randn(2, D, generator=g)).to(BF16) for _ in range(3))
    b = (0.5 * torch.randn(1, D, generator=g)).to(BF16) if bias else None
    res, out, q = mbx.gated_residual_ln_modulate_fp8(r.to(DEV), gt.to(DEV), u.to(DEV), sc.to(DEV), sh.to(DEV),
                                                     _scale(0.02), bias=None if b is None else b.to(DEV))
    want_r, want_o = oracle.gated_residual_ln_modulate(u16(r), u16(gt), u16(u), None if b is None else u16(b),
                                                       u16(sc), u16(sh), 1e-6)
    assert_bits_equal(u16(res), want_r, "residual")
    assert_bits_equal(u16(out), want_o, "bf16")
    assert_bits_equal(_b8(q), oracle.quant_e4m3(want_o, 0.02), "e4m3")
    res_h, out_h, q_h = mbx.gated_residual_ln_modulate_fp8(r.to(DEV), gt.to(DEV), u.to(DEV), sc.to(DEV), sh.to(DEV),
                                                           _scale(0.02), bias=None if b is None else b.to(DEV),
                                                           variant="high")
    assert_bits_equal(u16(res_h), want_r, "residual (high)")
    _self_consistent(out_h, q_h, 0.02)


@pytest.mark.parametrize("D", [1024, 3072, 5120])
def test_gated_fp8_per_token(mbx, D):
    """Per-token gate, scale and shift (the fused kernel's per-row path, whose
    threads per row differ by width and, at 5120, by variant)."""
    g = torch.Generator().manual_seed(23 + D)
    rows = 300
    r = torch.randn(rows, D, generator=g).to(BF16)
    u = torch.randn(rows, D, generator=g).to(BF16)
    gt, sc, sh = ((0.1 * torch.randn(rows, D, generator=g)).to(BF16) for _ in range(3))
    args = (r.to(DEV), gt.to(DEV), u.to(DEV), sc.to(DEV), sh.to(DEV), _scale(0.02))
    res, out, q = mbx.gated_residual_ln_modulate_fp8(*args)
    want_r, want_o = oracle.gated_residual_ln_modulate(u16(r), u16(gt), u16(u), None, u16(sc), u16(sh), 1e-6)
    assert_bits_equal(u16(res), want_r, "residual")
    assert_bits_equal(u16(out), want_o, "bf16")
    assert_bits_equal(_b8(q), oracle.quant_e4m3(want_o, 0.02), "e4m3")
    res_h, out_h, q_h = mbx.gated_residual_ln_modulate_fp8(*args, variant="high")
    assert_bits_equal(u16(res_h), want_r, "residual (high)")
    ex, mag = oracle.ln_modulate_f64(want_r, u16(sc), u16(sh), 1e-6)
    assert_high_close(u16(out_h), ex, mag, what="bf16 (high)")
    _self_consistent(out_h, q_h, 0.02)


def test_scale_is_read_on_the_stream(mbx):
    """The scale is a device value read when the kernel runs: updating it in
    place between two calls changes the second result, with no sync."""
    g = torch.Generator().manual_seed(9)
    x = torch.randn(128, 1024, generator=g).to(BF16).to(DEV)
    sc = torch.zeros(1, 1024, dtype=BF16, device=DEV)
    s = _scale(0.05)
    _, q1 = mbx.ln_modulate_fp8(x, sc, sc, s)
    s.fill_(0.1)
    _, q2 = mbx.ln_modulate_fp8(x, sc, sc, s)
    want = oracle.ln_modulate(u16(x), u16(sc), u16(sc), 1e-6)
    want1 = oracle.quant_e4m3(want, 0.05)
    want2 = oracle.quant_e4m3(want, 0.1)
    assert_bits_equal(_b8(q1), want1, "first scale")
    assert_bits_equal(_b8(q2), want2, "second scale")
