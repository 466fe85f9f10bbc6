"""Parity of the NVFP4 producers (LN + AdaLN, and gated residual + LN + AdaLN,
each with an NVFP4 copy of the bf16 output: packed E2M1 values and E4M3 block
scales in the 128x4 tile layout).

Lossless: the bf16 output, every packed byte and every block-scale byte equal
the oracle's (the NVFP4 rule applied to the oracle's bf16 output).  High: the
bf16 output is graded as before, and the NVFP4 copy must decode to within one
E2M1 half-step of the bf16 output the kernel wrote.  The E2M1 conversion is
pinned on the GPU by mbx_selftest(6) over every binary32 pattern.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_bits_equal, u16

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16 = torch.bfloat16
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@pytest.fixture(scope="module")
def mbx():
    import modulation_bit_exact_gb300 as m
    m.lib()
    return m


def _gs(v):
    return torch.tensor([v], dtype=torch.float32, device=DEV)


def _b(t):
    return t.detach().cpu().contiguous().numpy()


def test_selftest_e2m1_conversion(mbx):
    assert tuple(mbx.selftest(6)) == (0, 0)


def _check_lossless(q, sf, want_out, gs):
    wq, wsf = oracle.quant_nvfp4(want_out, gs, sf_fill=0)
    assert_bits_equal(_b(q).reshape(wq.shape), wq, "e2m1")
    assert_bits_equal(_b(sf).reshape(-1), wsf, "block scales")


def _decode_close(out, q, sf, gs):
    """The NVFP4 copy decodes to within one E2M1 half-step of `out`."""
    y = out.float().cpu().numpy().reshape(-1, out.shape[-1]).astype(np.float64)
    rows, D = y.shape
    qb = _b(q).reshape(rows, D // 2)
    codes = np.stack([qb & 0xF, qb >> 4], axis=-1).reshape(rows, D)
    mp, kp = mbx_sf_shape(rows, D)
    S = _b(sf).reshape(mp // 128, kp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(mp, kp)[:rows, :D // 16]
    sval = torch.from_numpy(S.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    unit = np.repeat(sval, 16, axis=1) / gs
    deq = E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0) * unit
    assert np.all(np.abs(deq - y) <= unit * 1.0 + 1e-30)


def mbx_sf_shape(rows, D):
    return (rows + 127) // 128 * 128, (D // 16 + 3) // 4 * 4


def test_ln_modulate_nvfp4_image_dit(mbx):
    d = synth.image_dit_block()
    x, sc, sh = (d[k].to(DEV) for k in ("x", "scale", "shift"))
    want = oracle.ln_modulate(u16(d["x"]).reshape(-1, 3072), u16(d["scale"]), u16(d["shift"]), 1e-6)
    gs = 448.0 * 6.0 / 40.0
    out, q, sf = mbx.ln_modulate_nvfp4(x, sc, sh, _gs(gs))
    assert_bits_equal(u16(out).reshape(-1, 3072), want, "bf16")
    _check_lossless(q, sf, want, gs)
    out_h, q_h, sf_h = mbx.ln_modulate_nvfp4(x, sc, sh, _gs(gs), variant="high")
    _decode_close(out_h, q_h, sf_h, gs)


@pytest.mark.parametrize("D,rows,mrows,shift", [(1024, 300, 3, 0), (5120, 97, 97, 0), (8192, 40, 40, 0),
                                                (2048, 64, 2, 1), (64, 129, 1, 0), (48, 7, 7, 0),
                                                (2048, 256, 256, 0), (3072, 300, 300, 0), (4096, 200, 200, 0),
                                                (6144, 100, 100, 0)])
def test_ln_modulate_nvfp4_shapes(mbx, D, rows, mrows, shift):
    """Staged and per-token modulation, rows that do not fill a 128-row tile,
    D = 48 (blocks padded to 4), a misaligned view (the separate quantiser)."""
    g = torch.Generator().manual_seed(D * 3 + rows)
    x = (torch.randn(rows, D, generator=g) * 2).to(BF16)
    x[0, :16] = 0  # an all-zero block
    sc = (0.1 * torch.randn(mrows, D, generator=g)).to(BF16)
    sh = (0.1 * torch.randn(mrows, D, generator=g)).to(BF16)
    xd = x.to(DEV)
    if shift:
        buf = torch.empty(rows * D + 8, dtype=BF16, device=DEV)
        xd = buf[1:1 + rows * D].view(rows, D)
        xd.copy_(x.to(DEV))
    out, q, sf = mbx.ln_modulate_nvfp4(xd, sc.to(DEV), sh.to(DEV), _gs(500.0))
    want = oracle.ln_modulate(u16(x), u16(sc), u16(sh), 1e-6)
    assert_bits_equal(u16(out), want, "bf16")
    _check_lossless(q, sf, want, 500.0)


@pytest.mark.parametrize("bias,D", [(True, 3072), (False, 3072), (True, 8192)])
def test_gated_nvfp4(mbx, bias, D):
    g = torch.Generator().manual_seed(7 + D)
    rows = 2 * 611 if D == 3072 else 2 * 97
    r = torch.randn(rows, D, generator=g).to(BF16)
    u = torch.randn(rows, D, generator=g).to(BF16)
    gt, sc, sh = ((0.1 * torch.randn(2, D, generator=g)).to(BF16) for _ in range(3))
    b = (0.5 * torch.randn(1, D, generator=g)).to(BF16) if bias else None
    gs = 300.0
    res, out, q, sf = mbx.gated_residual_ln_modulate_nvfp4(r.to(DEV), gt.to(DEV), u.to(DEV), sc.to(DEV),
                                                           sh.to(DEV), _gs(gs),
                                                           bias=None if b is None else b.to(DEV))
    want_r, want_o = oracle.gated_residual_ln_modulate(u16(r), u16(gt), u16(u), None if b is None else u16(b),
                                                       u16(sc), u16(sh), 1e-6)
    assert_bits_equal(u16(res), want_r, "residual")
    assert_bits_equal(u16(out), want_o, "bf16")
    _check_lossless(q, sf, want_o, gs)


@pytest.mark.parametrize("D", [1024, 3072, 5120])
def test_gated_nvfp4_per_token(mbx, D):
    """Per-token gate, scale and shift: the fused kernel's per-row path (its
    threads per row differ by width)."""
    g = torch.Generator().manual_seed(11 + D)
    rows = 300
    r = torch.randn(rows, D, generator=g).to(BF16)
    u = torch.randn(rows, D, generator=g).to(BF16)
    gt, sc, sh = ((0.1 * torch.randn(rows, D, generator=g)).to(BF16) for _ in range(3))
    b = (0.5 * torch.randn(1, D, generator=g)).to(BF16)
    gs = 300.0
    res, out, q, sf = mbx.gated_residual_ln_modulate_nvfp4(r.to(DEV), gt.to(DEV), u.to(DEV), sc.to(DEV),
                                                           sh.to(DEV), _gs(gs), bias=b.to(DEV))
    want_r, want_o = oracle.gated_residual_ln_modulate(u16(r), u16(gt), u16(u), u16(b), u16(sc), u16(sh), 1e-6)
    assert_bits_equal(u16(res), want_r, "residual")
    assert_bits_equal(u16(out), want_o, "bf16")
    _check_lossless(q, sf, want_o, gs)


@pytest.mark.parametrize("gs", [0.0, 1e-44, 3e38])
def test_nvfp4_extreme_global_scales(mbx, gs):
    """A zero global scale (every block scale 0), one so small that gs / value
    underflows to zero (codes of +-0 keep their sign), and one that saturates
    every block scale."""
    g = torch.Generator().manual_seed(17)
    x = (torch.randn(256, 1024, generator=g) * 2).to(BF16)
    sc = (0.1 * torch.randn(2, 1024, generator=g)).to(BF16)
    out, q, sf = mbx.ln_modulate_nvfp4(x.to(DEV), sc.to(DEV), sc.to(DEV), _gs(gs))
    want = oracle.ln_modulate(u16(x), u16(sc), u16(sc), 1e-6)
    assert_bits_equal(u16(out), want, "bf16")
    _check_lossless(q, sf, want, gs)


def test_nvfp4_and_fp8_non_finite_rows(mbx):
    """Rows holding inf or NaN make NaN outputs (0x7FFF); their NVFP4 blocks get
    the NaN scale code 0x7F and codes 0x7, their FP8 bytes 0x7F, as in the
    oracle.  Finite rows next to them are unaffected."""
    g = torch.Generator().manual_seed(23)
    rows, D = 64, 1024
    x = torch.randn(rows, D, generator=g)
    x[3, 5] = float("inf")
    x[7, 100] = float("nan")
    x[9, :] = -float("inf")
    x = x.to(BF16)
    sc = (0.1 * torch.randn(2, D, generator=g)).to(BF16)
    out, q, sf = mbx.ln_modulate_nvfp4(x.to(DEV), sc.to(DEV), sc.to(DEV), _gs(100.0))
    want = oracle.ln_modulate(u16(x), u16(sc), u16(sc), 1e-6)
    assert_bits_equal(u16(out), want, "bf16")
    _check_lossless(q, sf, want, 100.0)
    out8, q8 = mbx.ln_modulate_fp8(x.to(DEV), sc.to(DEV), sc.to(DEV), _gs(0.05))
    assert_bits_equal(u16(out8), want, "bf16 (fp8 call)")
    assert_bits_equal(_b(q8.view(torch.uint8)), oracle.quant_e4m3(want, 0.05), "e4m3")
