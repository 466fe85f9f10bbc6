"""The producers (gated residual + LN, and the FP8 and NVFP4 copies of LN and
of gated LN) on the widest sweep cells: T = 65536 rows of every sweep hidden
size, every element compared.

Each D takes its own instantiation of the ring kernel (chunks per lane J =
D / 1024), so these cells cover every row-block and ring-round boundary the
production sizes reach.  Lossless: every bf16, E4M3, E2M1 and block-scale byte
equals the oracle's.  High: r' is exact, every bf16 output (plain and gated,
of the FP8 and NVFP4 producers too, which may split rows otherwise than the
plain LN) is within 2 bfloat16 ulps of the binary64 LN + modulate, and the
FP8 / NVFP4 copies are the quantisation of the bf16 output the kernel wrote (PyTorch float8 witness
for E4M3, a decode within one E2M1 half-step for NVFP4).  The oracle runs on
every host core (gpu_util.par_rows).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_bits_equal, assert_high_close, host_rows, par_rows, u16

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16 = torch.bfloat16
T = 65536
FP8_SCALE = 0.02
GS = 448.0 * 6.0 / 40.0
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@pytest.fixture(scope="module")
def mbx():
    import modulation_bit_exact_gb300 as m
    m.lib()
    return m


def _b(t):
    """Bytes of a uint8 or float8 tensor as a host uint8 array."""
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def _case(D):
    """The sweep cell's inputs (padded rows) plus a bias drawn for the gated op."""
    d = synth.sweep_case(D, T, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(D * 7 + 1)
    d["bias"] = (torch.randn(1, D, generator=g, device=DEV) * 0.5).to(BF16)
    h = dict(R=host_rows(d["residual"]), U=host_rows(d["y"]), X=host_rows(d["x"]),
             G=u16(d["gate"]), SC=u16(d["scale"]), SH=u16(d["shift"]), B=u16(d["bias"]).reshape(-1))
    return d, h


def _sf_chunk(sf_flat, lo, hi, D):
    """Bytes of the 128x4-tiled scale buffer that hold rows [lo, hi), lo a
    multiple of 128: the tiles are laid out row-tile major."""
    tile_cols = (D // 16 + 3) // 4
    a = lo // 128 * tile_cols * 512
    b = -(-hi // 128) * tile_cols * 512
    return sf_flat[a:b]


def _fp8_consistent(out_rows, q_rows, scale):
    """q is the E4M3 copy of the bf16 rows `out` (PyTorch float8 witness)."""
    inv = np.float32(1.0) / np.float32(scale)
    prod = (((out_rows.astype(np.uint32) << 16).view(np.float32)) * inv).astype(np.float32)
    inr = np.abs(prod) < 448
    want = torch.from_numpy(prod[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q_rows[inr], want)
    assert np.all(q_rows[~inr & (prod > 0)] == 0x7E) and np.all(q_rows[~inr & (prod < 0)] == 0xFE)


def _nvfp4_decode_close(out_rows, q_rows, sf_bytes, gs):
    """The NVFP4 copy of rows [lo, hi) decodes to within one E2M1 half-step."""
    y = (out_rows.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rows, D = y.shape
    codes = np.stack([q_rows & 0xF, q_rows >> 4], axis=-1).reshape(rows, D)
    mp, kp = -(-rows // 128) * 128, (D // 16 + 3) // 4 * 4
    S = sf_bytes.reshape(mp // 128, kp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(mp, kp)[:rows, :D // 16]
    sval = torch.from_numpy(np.ascontiguousarray(S)).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    unit = np.repeat(sval, 16, axis=1) / gs
    deq = E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0) * unit
    assert np.all(np.abs(deq - y) <= unit + 1e-30)


@pytest.mark.parametrize("D", synth.SWEEP_D)
def test_gated_residual_ln_modulate(mbx, D):
    d, h = _case(D)
    args = (d["residual"], d["gate"], d["y"], d["scale"], d["shift"])
    got = {}
    for v in ("lossless", "high"):
        r, o = mbx.gated_residual_ln_modulate(*args, bias=d["bias"], variant=v)
        got[v] = (host_rows(r), host_rows(o))
        del r, o

    def chk(lo, hi):
        wr, wo = oracle.gated_residual_ln_modulate(h["R"][lo:hi], h["G"], h["U"][lo:hi], h["B"], h["SC"],
                                                   h["SH"], 1e-6)
        what = f"D={D} rows {lo}:{hi}"
        assert_bits_equal(got["lossless"][0][lo:hi], wr, "residual " + what)
        assert_bits_equal(got["lossless"][1][lo:hi], wo, "out " + what)
        assert_bits_equal(got["high"][0][lo:hi], wr, "residual (high) " + what)
        assert_high_close(got["high"][1][lo:hi], *oracle.ln_modulate_f64(wr, h["SC"], h["SH"], 1e-6),
                          what="out (high) " + what)

    par_rows(chk, T)


@pytest.mark.parametrize("D", synth.SWEEP_D)
def test_fp8_producers(mbx, D):
    d, h = _case(D)
    s8 = torch.tensor([FP8_SCALE], dtype=torch.float32, device=DEV)
    ln, gated = {}, {}
    for v in ("lossless", "high"):
        o, q = mbx.ln_modulate_fp8(d["x"], d["scale"], d["shift"], s8, variant=v)
        ln[v] = (host_rows(o), _b(q).reshape(T, D))
        r, o, q = mbx.gated_residual_ln_modulate_fp8(d["residual"], d["gate"], d["y"], d["scale"], d["shift"], s8,
                                                     bias=d["bias"], variant=v)
        gated[v] = (host_rows(r), host_rows(o), _b(q).reshape(T, D))
        del o, q, r

    def chk(lo, hi):
        what = f"D={D} rows {lo}:{hi}"
        want = oracle.ln_modulate(h["X"][lo:hi], h["SC"], h["SH"], 1e-6)
        assert_bits_equal(ln["lossless"][0][lo:hi], want, "ln bf16 " + what)
        assert_bits_equal(ln["lossless"][1][lo:hi], oracle.quant_e4m3(want, FP8_SCALE), "ln e4m3 " + what)
        # the FP8 producer may run another row split than the plain LN (threads
        # per row, stages): its bf16 output is held to the high bound on its own
        assert_high_close(ln["high"][0][lo:hi], *oracle.ln_modulate_f64(h["X"][lo:hi], h["SC"], h["SH"], 1e-6),
                          what="ln bf16 (high) " + what)
        _fp8_consistent(ln["high"][0][lo:hi], ln["high"][1][lo:hi], FP8_SCALE)
        wr, wo = oracle.gated_residual_ln_modulate(h["R"][lo:hi], h["G"], h["U"][lo:hi], h["B"], h["SC"],
                                                   h["SH"], 1e-6)
        assert_bits_equal(gated["lossless"][0][lo:hi], wr, "gated residual " + what)
        assert_bits_equal(gated["lossless"][1][lo:hi], wo, "gated bf16 " + what)
        assert_bits_equal(gated["lossless"][2][lo:hi], oracle.quant_e4m3(wo, FP8_SCALE), "gated e4m3 " + what)
        assert_bits_equal(gated["high"][0][lo:hi], wr, "gated residual (high) " + what)
        assert_high_close(gated["high"][1][lo:hi], *oracle.ln_modulate_f64(wr, h["SC"], h["SH"], 1e-6),
                          what="gated bf16 (high) " + what)
        _fp8_consistent(gated["high"][1][lo:hi], gated["high"][2][lo:hi], FP8_SCALE)

    par_rows(chk, T)


@pytest.mark.parametrize("D", synth.SWEEP_D)
def test_nvfp4_producers(mbx, D):
    d, h = _case(D)
    gs = torch.tensor([GS], dtype=torch.float32, device=DEV)
    ln, gated = {}, {}
    for v in ("lossless", "high"):
        o, q, sf = mbx.ln_modulate_nvfp4(d["x"], d["scale"], d["shift"], gs, variant=v)
        ln[v] = (host_rows(o), _b(q).reshape(T, D // 2), _b(sf).reshape(-1))
        r, o, q, sf = mbx.gated_residual_ln_modulate_nvfp4(d["residual"], d["gate"], d["y"], d["scale"],
                                                           d["shift"], gs, bias=d["bias"], variant=v)
        gated[v] = (host_rows(r), host_rows(o), _b(q).reshape(T, D // 2), _b(sf).reshape(-1))
        del o, q, sf, r

    def chk(lo, hi):
        what = f"D={D} rows {lo}:{hi}"
        want = oracle.ln_modulate(h["X"][lo:hi], h["SC"], h["SH"], 1e-6)
        wq, wsf = oracle.quant_nvfp4(want, GS, sf_fill=0)
        o, q, sf = ln["lossless"]
        assert_bits_equal(o[lo:hi], want, "ln bf16 " + what)
        assert_bits_equal(q[lo:hi], wq, "ln e2m1 " + what)
        assert_bits_equal(_sf_chunk(sf, lo, hi, D), wsf, "ln block scales " + what)
        o, q, sf = ln["high"]
        assert_high_close(o[lo:hi], *oracle.ln_modulate_f64(h["X"][lo:hi], h["SC"], h["SH"], 1e-6),
                          what="ln bf16 (high) " + what)
        _nvfp4_decode_close(o[lo:hi], q[lo:hi], _sf_chunk(sf, lo, hi, D), GS)
        wr, wo = oracle.gated_residual_ln_modulate(h["R"][lo:hi], h["G"], h["U"][lo:hi], h["B"], h["SC"],
                                                   h["SH"], 1e-6)
        wq, wsf = oracle.quant_nvfp4(wo, GS, sf_fill=0)
        r, o, q, sf = gated["lossless"]
        assert_bits_equal(r[lo:hi], wr, "gated residual " + what)
        assert_bits_equal(o[lo:hi], wo, "gated bf16 " + what)
        assert_bits_equal(q[lo:hi], wq, "gated e2m1 " + what)
        assert_bits_equal(_sf_chunk(sf, lo, hi, D), wsf, "gated block scales " + what)
        r, o, q, sf = gated["high"]
        assert_bits_equal(r[lo:hi], wr, "gated residual (high) " + what)
        assert_high_close(o[lo:hi], *oracle.ln_modulate_f64(wr, h["SC"], h["SH"], 1e-6),
                          what="gated bf16 (high) " + what)
        _nvfp4_decode_close(o[lo:hi], q[lo:hi], _sf_chunk(sf, lo, hi, D), GS)

    par_rows(chk, T, align=128)
