"""Edge cases of the CUDA path against the oracle, and exhaustive checks of the
arithmetic building blocks the lossless kernels rest on."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_bits_equal, assert_high_close, guarded, u16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def mbx():
    import modulation_bit_exact_gb300 as m
    m.lib()
    return m


def bf(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)


# ------------------------------------------------------------------ building blocks


@pytest.mark.parametrize("which,what", [(0, "division by counts 1..64"),
                                        (1, "bf16x2 multiply"), (2, "bf16x2 add"),
                                        (3, "unguarded division, |d| >= 2^-100"),
                                        (4, "reciprocal square root table")])
def test_exhaustive_building_blocks(mbx, which, what):
    bad, bad_nan = mbx.selftest(which)
    assert bad == 0, f"{what}: {bad} non-NaN mismatches"
    assert bad_nan == 0, f"{what}: {bad_nan} NaN-encoding mismatches"


def test_tanh_every_bf16_input_through_the_op(mbx):
    """x = 1 gives rstd = 1 and n = 1 exactly; residual = -0 leaves out = tg for
    every gate value, signed zeros included.  All 65536 gate values."""
    g = np.arange(65536, dtype=np.uint16).reshape(8, 8192)
    x = np.full((8, 8192), 0x3F80, np.uint16)
    w = np.full(8192, 0x3F80, np.uint16)
    r = np.full((8, 8192), 0x8000, np.uint16)
    got = u16(mbx.rmsnorm_tanh_residual(bf(x).to(DEV), bf(g).to(DEV), bf(r).to(DEV), bf(w).to(DEV)))
    want = oracle.rmsnorm_tanh_residual(x, g, r, w, 1e-6)
    assert_bits_equal(got, want, "tanh")
    assert_bits_equal(got.reshape(-1), oracle.tanh_table(), "tanh table")


# ------------------------------------------------------------------ shapes and layouts


def _inputs(rows, D, mrows, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(rows, D, generator=g) * scale).to(torch.bfloat16)
    y = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    r = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    gt = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    sc = (torch.randn(mrows, D, generator=g) * 0.1).to(torch.bfloat16)
    sh = (torch.randn(mrows, D, generator=g) * 0.1).to(torch.bfloat16)
    gm = (torch.randn(mrows, D, generator=g) * 0.1).to(torch.bfloat16)
    w = (1 + 0.05 * torch.randn(D, generator=g)).to(torch.bfloat16)
    return dict(x=x, y=y, r=r, gt=gt, sc=sc, sh=sh, gm=gm, w=w)


def _all_ops(mbx, t, dev_views=None):
    """Run every row op; `dev_views` maps names to the device tensors to pass
    (possibly offset or padded views of the same values)."""
    v = dev_views or {k: a.to(DEV) for k, a in t.items()}
    U = {k: u16(a) for k, a in t.items()}
    out = {
        "ln": (u16(mbx.ln_modulate(v["x"], v["sc"], v["sh"])), oracle.ln_modulate(U["x"], U["sc"], U["sh"], 1e-6)),
        "rms": (u16(mbx.rmsnorm_scale(v["x"], v["w"], v["sc"])), oracle.rmsnorm_scale(U["x"], U["w"], U["sc"], 1e-6)),
        "tanh": (u16(mbx.rmsnorm_tanh_residual(v["x"], v["gm"], v["r"], v["w"])),
                 oracle.rmsnorm_tanh_residual(U["x"], U["gm"], U["r"], U["w"], 1e-6)),
        "tanh_tok": (u16(mbx.rmsnorm_tanh_residual(v["x"], v["gt"], v["r"], v["w"])),
                     oracle.rmsnorm_tanh_residual(U["x"], U["gt"], U["r"], U["w"], 1e-6)),
        "rga": (u16(mbx.residual_gate_add(v["x"], v["gm"], v["y"])), oracle.residual_gate_add(U["x"], U["gm"], U["y"])),
    }
    for k, (got, want) in out.items():
        assert_bits_equal(got, want, k)


@pytest.mark.parametrize("D", [1, 2, 3, 7, 8, 9, 15, 100, 1000, 1001, 1024, 1032, 3000, 5000, 8191, 8192])
def test_ragged_hidden_sizes(mbx, D):
    """Hidden sizes that are not multiples of 8 (scalar path, partial last
    chunk, lanes with fewer chunks) and ones that are."""
    _all_ops(mbx, _inputs(12, D, 3, seed=D))


@pytest.mark.parametrize("D", [64, 512, 3072])
def test_misaligned_views_take_the_scalar_path(mbx, D):
    """Views starting 2 bytes past a 16-byte boundary compute the same bits."""
    t = _inputs(6, D, 2, seed=7)
    dv = {}
    for k, a in t.items():
        flat = a.reshape(-1)
        buf = torch.zeros(flat.numel() + 1, dtype=torch.bfloat16, device=DEV)
        buf[1:] = flat.to(DEV)
        dv[k] = buf[1:].view(a.shape)
    _all_ops(mbx, t, dv)


@pytest.mark.parametrize("mrows", [1, 2, 3, 6, 12, 36])
def test_modulation_row_mapping(mbx, mrows):
    _all_ops(mbx, _inputs(36, 1024, mrows, seed=mrows))


def test_single_row_max_hidden(mbx):
    _all_ops(mbx, _inputs(1, 8192, 1, seed=3))


def test_degenerate_rows(mbx):
    """Constant rows (variance exactly 0), zero rows, tiny and huge rows."""
    t = _inputs(8, 3072, 1, seed=11)
    x = t["x"].float()
    x[0] = 0.0
    x[1] = 1.0
    x[2] = -7.5
    x[3] = 1e-30
    x[4] *= 1e30
    x[5] *= 1e-35
    x[6] = torch.where(torch.arange(3072) % 2 == 0, 1e-38, -1e-38)
    t["x"] = x.to(torch.bfloat16)
    _all_ops(mbx, t)


def test_non_finite_inputs(mbx):
    """inf and NaN propagate to the canonical NaN (0x7FFF) exactly as in the oracle."""
    t = _inputs(6, 1024, 2, seed=12)
    x = t["x"].float()
    x[0, 5] = float("inf")
    x[1, 9] = float("nan")
    x[2, 100] = -float("inf")
    t["x"] = x.to(torch.bfloat16)
    y = t["y"].float()
    y[3, 3] = float("inf")
    t["y"] = y.to(torch.bfloat16)
    gm = t["gm"].float()
    gm[1, 7] = float("nan")
    t["gm"] = gm.to(torch.bfloat16)
    _all_ops(mbx, t)


def test_extreme_values_overflow(mbx):
    t = _inputs(4, 256, 1, seed=13)
    t["x"] = (t["x"].float() * 3e38).to(torch.bfloat16)
    t["gm"] = torch.full((1, 256), 3e38).to(torch.bfloat16)
    _all_ops(mbx, t)


# ------------------------------------------------------------------ in place, bounds, streams


def test_in_place_residual_updates(mbx):
    t = _inputs(16, 3072, 2, seed=21)
    U = {k: u16(a) for k, a in t.items()}
    x = t["x"].to(DEV)
    mbx.residual_gate_add(x, t["gm"].to(DEV), t["y"].to(DEV), out=x)
    assert_bits_equal(u16(x), oracle.residual_gate_add(U["x"], U["gm"], U["y"]), "rga in place")
    r = t["r"].to(DEV)
    mbx.rmsnorm_tanh_residual(t["x"].to(DEV), t["gt"].to(DEV), r, t["w"].to(DEV), out=r)
    assert_bits_equal(u16(r), oracle.rmsnorm_tanh_residual(U["x"], U["gt"], U["r"], U["w"], 1e-6),
                      "tanh residual in place")


@pytest.mark.parametrize("D", [100, 3072])
def test_outputs_stay_inside_their_views(mbx, D):
    t = _inputs(10, D, 2, seed=31)
    v = {k: a.to(DEV) for k, a in t.items()}
    for variant in ("lossless", "high"):
        for name, run in (
            ("ln", lambda o: mbx.ln_modulate(v["x"], v["sc"], v["sh"], out=o, variant=variant)),
            ("rms", lambda o: mbx.rmsnorm_scale(v["x"], v["w"], v["sc"], out=o, variant=variant)),
            ("tanh", lambda o: mbx.rmsnorm_tanh_residual(v["x"], v["gm"], v["r"], v["w"], out=o,
                                                         variant=variant)),
            ("rga", lambda o: mbx.residual_gate_add(v["x"], v["gm"], v["y"], out=o, variant=variant)),
        ):
            o, check = guarded((10, D), DEV)
            run(o)
            torch.cuda.synchronize()
            check()


def test_padded_output_rows(mbx):
    """An output with padded rows: the pad is never written."""
    t = _inputs(9, 1000, 3, seed=41)
    buf = torch.full((9, 1064), 12345.0, dtype=torch.bfloat16, device=DEV)
    out = buf[:, :1000]
    mbx.ln_modulate(t["x"].to(DEV), t["sc"].to(DEV), t["sh"].to(DEV), out=out)
    U = {k: u16(a) for k, a in t.items()}
    assert_bits_equal(u16(out), oracle.ln_modulate(U["x"], U["sc"], U["sh"], 1e-6), "padded out")
    assert torch.all(buf[:, 1000:] == 12345.0)


def test_runs_on_the_callers_stream(mbx):
    d = synth.image_dit_block(seq=1024, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = mbx.ln_modulate(d["x"], d["scale"], d["shift"])
        out2 = mbx.residual_gate_add(out, d["gate"], d["y"])
    s.synchronize()
    X = u16(d["x"]).reshape(-1, 3072)
    ln = oracle.ln_modulate(X, u16(d["scale"]), u16(d["shift"]), 1e-6)
    want = oracle.residual_gate_add(ln, u16(d["gate"]), u16(d["y"]).reshape(-1, 3072))
    assert_bits_equal(u16(out2).reshape(-1, 3072), want, "stream chain")


def test_device_rejections(mbx):
    """Host memory and views past the end of their allocation are refused
    before anything is launched."""
    import ctypes
    from modulation_bit_exact_gb300 import _View
    x = torch.randn(4, 64, device=DEV).to(torch.bfloat16)
    sc = torch.zeros(1, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(mbx.MbxError) as e:
        mbx.ln_modulate(x, sc.cpu(), sc)
    assert e.value.status == -9
    # a fresh allocation that is its own segment (a multiple of 2 MiB); a
    # 2-row view whose second row lies past its end
    torch.cuda.empty_cache()
    n = 1 << 25
    big = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    o = torch.empty(2, 64, dtype=torch.bfloat16, device=DEV)
    xv = _View(big.data_ptr() + (n - 64) * 2, 2, 64, 64, 1)
    L = mbx.lib()
    st = L.mbx_check_ln_modulate(ctypes.byref(mbx._view(o)), ctypes.byref(xv),
                                 ctypes.byref(mbx._view(sc)), ctypes.byref(mbx._view(sc)),
                                 ctypes.c_float(1e-6), 0)
    assert st == -10
    xv_ok = _View(big.data_ptr() + (n - 128) * 2, 2, 64, 64, 1)
    st = L.mbx_check_ln_modulate(ctypes.byref(mbx._view(o)), ctypes.byref(xv_ok),
                                 ctypes.byref(mbx._view(sc)), ctypes.byref(mbx._view(sc)),
                                 ctypes.c_float(1e-6), 0)
    assert st == 0


@pytest.mark.parametrize("D,rows", [(2048, 1200), (4096, 1200), (6144, 600), (8192, 600), (4096, 16384),
                                    (3072, 32768)])
def test_per_token_modulation_every_width(mbx, D, rows):
    """Per-token modulation (each row reads its own modulation row) at the
    widths and row counts where the ring kernels change threads per row or
    stages: the plain, FP8 and RMSNorm kernels on their per-row path, both
    variants."""
    t = _inputs(rows, D, rows, seed=D + rows)
    _all_ops(mbx, t)
    v = {k: a.to(DEV) for k, a in t.items()}
    U = {k: u16(a) for k, a in t.items()}
    want = oracle.ln_modulate(U["x"], U["sc"], U["sh"], 1e-6)
    s8 = torch.tensor([0.02], dtype=torch.float32, device=DEV)
    out, q = mbx.ln_modulate_fp8(v["x"], v["sc"], v["sh"], s8)
    assert_bits_equal(u16(out), want, "fp8 ln bf16")
    assert_bits_equal(q.view(torch.uint8).cpu().numpy(), oracle.quant_e4m3(want, 0.02), "fp8 ln e4m3")
    ex, mag = oracle.ln_modulate_f64(U["x"], U["sc"], U["sh"], 1e-6)
    assert_high_close(u16(mbx.ln_modulate(v["x"], v["sc"], v["sh"], variant="high")), ex, mag, what="ln high")
    out_h, _ = mbx.ln_modulate_fp8(v["x"], v["sc"], v["sh"], s8, variant="high")
    assert_high_close(u16(out_h), ex, mag, what="fp8 ln high")


@pytest.mark.parametrize("rows,mrows,D", [(4096, 512, 1024), (6000, 3000, 3072), (2048, 1024, 5120)])
def test_modulation_changing_within_a_cta(mbx, rows, mrows, D):
    """Samples change every few rows (seq = rows / mod_rows is smaller than a
    CTA's block of rows), so the modulation rows travel with x instead of being
    staged once per CTA."""
    _all_ops(mbx, _inputs(rows, D, mrows, seed=rows + D))
