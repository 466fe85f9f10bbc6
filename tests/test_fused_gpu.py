"""Parity of the gated residual update fused into LN + AdaLN modulate.

The residual stream r' and the modulated norm are both compared bit for bit
with the oracle in the lossless variant; in the high variant r' is still exact
and the norm is within 2 bfloat16 ulps of the binary64 LN + modulate of the
oracle's r'.  Shapes cover per-sample modulation staged per CTA, more samples
than a CTA can stage (ring mode), per-token modulation, ragged D, misaligned
views (the composed path), padded rows and the in-place residual update.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_bits_equal, assert_high_close, guarded, u16

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16 = torch.bfloat16


@pytest.fixture(scope="module")
def mbx():
    import modulation_bit_exact_gb300 as m
    m.lib()
    return m


def _case(batch, seq, D, per_token=False, bias=True, seed=11, pad=0):
    g = torch.Generator().manual_seed(seed * 7919 + batch * 131 + seq * 17 + D)
    mrows = batch * seq if per_token else batch

    def n(shape, std=1.0, p=0):
        t = (torch.randn(shape, generator=g) * std).to(BF16)
        return synth.padded(t, p) if p else t

    return dict(residual=n((batch * seq, D), p=pad), update=n((batch * seq, D), p=pad),
                gate=n((mrows, D), 0.1, p=pad), scale=n((mrows, D), 0.1, p=pad),
                shift=n((mrows, D), 0.1, p=pad), bias=n((1, D), 0.5) if bias else None, seq=seq)


def _oracle(c, sel=None):
    B = None if c["bias"] is None else u16(c["bias"])
    R, U = u16(c["residual"]), u16(c["update"])
    G, SC, SH = u16(c["gate"]), u16(c["scale"]), u16(c["shift"])
    if sel is not None:
        R, U = R[sel], U[sel]
        if G.shape[0] == c["residual"].shape[0]:
            G, SC, SH = G[sel], SC[sel], SH[sel]
        else:
            m = sel // c["seq"]
            G, SC, SH = G[m], SC[m], SH[m]
    return oracle.gated_residual_ln_modulate(R, G, U, B, SC, SH, 1e-6), (R, G, U, B, SC, SH)


def _dev(c, shift=()):
    """Copies on the GPU; tensors named in `shift` start one element past a
    16-byte boundary."""
    d = {}
    for k, v in c.items():
        if not torch.is_tensor(v):
            d[k] = v
        elif k in shift:
            buf = torch.empty(v.numel() + 8, dtype=BF16, device=DEV)
            d[k] = buf[1:1 + v.numel()].view(v.shape)
            d[k].copy_(v)
        else:
            d[k] = v.to(DEV)
    return d


def _gpu(mbx, c, variant="lossless", in_place=False, shift=()):
    d = _dev(c, shift)
    ro = d["residual"] if in_place else None
    return mbx.gated_residual_ln_modulate(d["residual"], d["gate"], d["update"], d["scale"],
                                          d["shift"], bias=d["bias"], variant=variant,
                                          residual_out=ro)


def _check(mbx, c, what, sel=None, shift=()):
    (want_r, want_o), ins = _oracle(c, sel)
    got_r, got_o = _gpu(mbx, c, shift=shift)
    gr, go = u16(got_r), u16(got_o)
    if sel is not None:
        gr, go = gr[sel], go[sel]
    assert_bits_equal(gr, want_r, what + " residual")
    assert_bits_equal(go, want_o, what + " out")
    # high: r' unchanged, the norm within 2 ulp of the exact LN of r'
    got_r, got_o = _gpu(mbx, c, variant="high", shift=shift)
    gr, go = u16(got_r), u16(got_o)
    if sel is not None:
        gr, go = gr[sel], go[sel]
    assert_bits_equal(gr, want_r, what + " residual (high)")
    ex, mag = oracle.ln_modulate_f64(want_r, ins[4], ins[5], 1e-6)
    assert_high_close(go, ex, mag, what=what + " out (high)")


@pytest.mark.parametrize("bias", [True, False])
def test_image_dit_full_size(mbx, bias):
    """2 x 4352 tokens of hidden 3072 with per-sample gate/scale/shift."""
    c = _case(2, 4352, 3072, bias=bias)
    rows = np.unique(np.r_[0:48, 4352 - 24:4352 + 24, 8704 - 48:8704,
                           np.random.default_rng(1).integers(0, 8704, 256)])
    (want_r, want_o), _ = _oracle(c)
    got_r, got_o = _gpu(mbx, c)
    assert_bits_equal(u16(got_r), want_r, "residual")
    assert_bits_equal(u16(got_o), want_o, "out")
    _check(mbx, c, "image high rows", sel=rows)


@pytest.mark.parametrize("batch,seq,D", [(3, 77, 1024), (64, 5, 2048), (5, 33, 5120),
                                         (2, 130, 8192), (1, 1, 3072)])
def test_shapes(mbx, batch, seq, D):
    """Staged per-sample modulation, many samples per CTA (ring mode), one row."""
    _check(mbx, _case(batch, seq, D), f"B={batch} S={seq} D={D}")


@pytest.mark.parametrize("D", [1024, 2048, 3072, 4096, 5120, 6144, 8192])
def test_per_token(mbx, D):
    _check(mbx, _case(1, 300, D, per_token=True), f"per-token D={D}")


@pytest.mark.parametrize("D", [1000, 3, 4100])
def test_ragged_d(mbx, D):
    _check(mbx, _case(2, 19, D), f"ragged D={D}")


def test_padded_rows(mbx):
    _check(mbx, _case(2, 50, 2048, per_token=True, pad=64), "padded")


@pytest.mark.parametrize("shift", [("residual",), ("update",), ("gate", "bias")])
def test_misaligned_views(mbx, shift):
    """Views offset by one element take the composed path; same bits."""
    _check(mbx, _case(2, 40, 1024), f"misaligned {shift}", shift=shift)


def test_in_place_and_guard_zones(mbx):
    c = _case(3, 64, 3072)
    (want_r, want_o), _ = _oracle(c)
    d = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in c.items()}
    out, check = guarded((192, 3072), DEV)
    res = d["residual"]
    mbx.gated_residual_ln_modulate(res, d["gate"], d["update"], d["scale"], d["shift"],
                                   bias=d["bias"], out=out, residual_out=res)
    torch.cuda.synchronize()
    check()
    assert_bits_equal(u16(res), want_r, "in-place residual")
    assert_bits_equal(u16(out), want_o, "in-place out")


@pytest.mark.parametrize("D,bias", [(8192, False), (6144, True), (2048, True)])
def test_wide_rows_modes(mbx, D, bias):
    """Rows whose per-sample vectors are read through L1 instead of staged
    (8192, 6144 by the mode policy) and the update's one-stage buffer, with and
    without a bias, over more rows than row groups."""
    _check(mbx, _case(2, 300, D, bias=bias), f"D={D} bias={bias}")


def test_in_place_wide_rows(mbx):
    """In place on the residual at the widest rows (L1 mode)."""
    c = _case(2, 97, 8192)
    (want_r, want_o), _ = _oracle(c)
    d = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in c.items()}
    res = d["residual"]
    r, o = mbx.gated_residual_ln_modulate(res, d["gate"], d["update"], d["scale"], d["shift"], bias=d["bias"],
                                          residual_out=res)
    torch.cuda.synchronize()
    assert_bits_equal(u16(res), want_r, "in-place residual")
    assert_bits_equal(u16(o), want_o, "in-place out")


def test_equals_the_two_kernels(mbx):
    """Without a bias the fused call gives exactly residual_gate_add followed
    by ln_modulate of the CUDA path."""
    c = _case(4, 257, 3072, bias=False)
    d = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in c.items()}
    r1 = mbx.residual_gate_add(d["residual"].view(4, 257, 3072), d["gate"], d["update"].view(4, 257, 3072))
    o1 = mbx.ln_modulate(r1, d["scale"], d["shift"])
    r2, o2 = _gpu(mbx, c)
    assert torch.equal(u16t(r1).reshape(-1), u16t(r2).reshape(-1))
    assert torch.equal(u16t(o1).reshape(-1), u16t(o2).reshape(-1))


def u16t(t):
    return t.view(torch.int16)
