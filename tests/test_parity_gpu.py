"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Lossless variants: every element equal bit for bit.  High variants: within 2
bfloat16 ulps of the largest term of the exact binary64 result (the single-pass
error budget stated for them), see gpu_util.assert_high_close.
Inputs come from the seeded generators in synth/, outputs of the oracle from
oracle/; nothing the CUDA path computes feeds the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_bits_equal, assert_high_close, guarded, host_rows, par_rows, u16

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def mbx():
    import modulation_bit_exact_gb300 as m
    m.lib()
    return m


def _rows2(t):
    return u16(t).reshape(-1, t.shape[-1])


# ------------------------------------------------------------------ configs 1, 2


def test_tiny_ln_modulate_and_rmsnorm_scale(mbx):
    d = synth.tiny_ln_modulate()
    x, sc, sh, w = (d[k].to(DEV) for k in ("x", "scale", "shift", "weight"))
    X, SC, SH, W = _rows2(d["x"]), u16(d["scale"]), u16(d["shift"]), u16(d["weight"])
    assert_bits_equal(u16(mbx.ln_modulate(x, sc, sh)), oracle.ln_modulate(X, SC, SH, 1e-6).reshape(2, 256, 512), "ln")
    assert_bits_equal(u16(mbx.rmsnorm_scale(x, w, sc)), oracle.rmsnorm_scale(X, W, SC, 1e-6).reshape(2, 256, 512), "rms")
    ex, mag = oracle.ln_modulate_f64(X, SC, SH, 1e-6)
    assert_high_close(_rows2(mbx.ln_modulate(x, sc, sh, variant="high")), ex, mag, what="ln high")
    ex, mag = oracle.rmsnorm_scale_f64(X, W, SC, 1e-6)
    assert_high_close(_rows2(mbx.rmsnorm_scale(x, w, sc, variant="high")), ex, mag, what="rms high")


def test_image_dit_block_full_size(mbx):
    """Image-DiT norm path at its full size, as the benchmark runs it."""
    d = synth.image_dit_block()
    x, sc, sh, g, y = (d[k].to(DEV) for k in ("x", "scale", "shift", "gate", "y"))
    X, SC, SH, G, Y = _rows2(d["x"]), u16(d["scale"]), u16(d["shift"]), u16(d["gate"]), _rows2(d["y"])
    assert_bits_equal(_rows2(mbx.ln_modulate(x, sc, sh)), oracle.ln_modulate(X, SC, SH, 1e-6), "ln")
    assert_bits_equal(_rows2(mbx.residual_gate_add(x, g, y)), oracle.residual_gate_add(X, G, Y), "rga")
    got = _rows2(mbx.ln_modulate(x, sc, sh, variant="high"))
    par_rows(lambda lo, hi: assert_high_close(
        got[lo:hi], *oracle.ln_modulate_f64(X[lo:hi], SC[lo // 4352:lo // 4352 + 1], SH[lo // 4352:lo // 4352 + 1],
                                            1e-6), what=f"ln high rows {lo}:{hi}"), 8704, seq=4352)
    ex, mag = oracle.residual_gate_add_f64(X, G, Y)
    assert_high_close(_rows2(mbx.residual_gate_add(x, g, y, variant="high")), ex, mag, what="rga high")


# ------------------------------------------------------------------ config 3


def _qkv_gpu(mbx, q, variant="lossless", out=None):
    qd = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in q.items()}
    return mbx.qk_norm_rope_qkv_epilogue(
        qd["txt"], qd["img"], q["batch"], q["heads"], q["head_dim"], qd["wq_txt"], qd["wk_txt"],
        qd["wq_img"], qd["wk_img"], qd["cos_txt"], qd["sin_txt"], qd["cos_img"], qd["sin_img"],
        q["eps"], variant=variant, out=out)


def _qkv_oracle(q):
    return oracle.qkv_epilogue(
        None if q["txt"] is None else u16(q["txt"]), u16(q["img"]), q["batch"], q["heads"],
        q["head_dim"], u16(q["wq_txt"]), u16(q["wk_txt"]), u16(q["wq_img"]), u16(q["wk_img"]),
        q["cos_txt"].numpy(), q["sin_txt"].numpy(), q["cos_img"].numpy(), q["sin_img"].numpy(),
        q["eps"])


def test_qkv_epilogue_full_size(mbx):
    q = synth.qkv_epilogue_case()
    assert_bits_equal(u16(_qkv_gpu(mbx, q)), _qkv_oracle(q), "joint")


def test_qkv_epilogue_offsets_past_32_bits(mbx):
    """Text rows 2^31 elements apart: the source offsets pass 2^32, so the
    call takes the 64-bit index form (8.6 GB of address space, three rows
    written); bit-exact like the 32-bit form."""
    q = synth.qkv_epilogue_case(batch=1, s_txt=3, grid_h=4, grid_w=4, heads=2, head_dim=64)
    width = q["txt"].shape[1]
    stride = 2 ** 31
    big = torch.empty(2 * stride + width, dtype=torch.bfloat16, device=DEV)
    txt = torch.as_strided(big, (3, width), (stride, 1))
    txt.copy_(q["txt"].to(DEV))
    qd = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in q.items()}
    out = mbx.qk_norm_rope_qkv_epilogue(
        txt, qd["img"], q["batch"], q["heads"], q["head_dim"], qd["wq_txt"], qd["wk_txt"], qd["wq_img"],
        qd["wk_img"], qd["cos_txt"], qd["sin_txt"], qd["cos_img"], qd["sin_img"], q["eps"])
    assert_bits_equal(u16(out), _qkv_oracle(q), "joint (64-bit offsets)")
    del big, txt, out
    torch.cuda.empty_cache()


def _qkv_high_check(mbx, q):
    got = u16(_qkv_gpu(mbx, q, variant="high"))
    want = _qkv_oracle(q)
    B, H, hd = q["batch"], q["heads"], q["head_dim"]
    assert np.array_equal(got[:, 2], want[:, 2])  # V is a copy in both variants
    s_txt = q["txt"].shape[0] // B
    for b in range(B):
        for part in (0, 1):
            for h in range(H):
                for name, S, off, w in (("txt", s_txt, 0, "wq_txt" if part == 0 else "wk_txt"),
                                        ("img", q["img"].shape[0] // B, s_txt, "wq_img" if part == 0 else "wk_img")):
                    src = u16(q[name]).reshape(B, S, 3, H, hd)
                    tab = "txt" if name == "txt" else "img"
                    for s in range(0, S, max(1, S // 7)):
                        ex, mag = oracle.qk_head_f64(src[b, s, part, h], u16(q[w]),
                                                     q["cos_" + tab][s].numpy(), q["sin_" + tab][s].numpy())
                        assert_high_close(got[b, part, h, off + s], ex, mag, what="qkv high")


def test_qkv_epilogue_high(mbx):
    _qkv_high_check(mbx, synth.qkv_epilogue_case(batch=2, s_txt=16, grid_h=8, grid_w=8, heads=6))


@pytest.mark.parametrize("hd,heads,pad", [(64, 3, 0), (64, 8, 64), (128, 5, 8), (256, 2, 0), (256, 7, 24)])
def test_qkv_epilogue_shapes(mbx, hd, heads, pad):
    q = synth.qkv_epilogue_case(batch=3, s_txt=9, grid_h=5, grid_w=7, heads=heads, head_dim=hd, row_pad=pad)
    assert_bits_equal(u16(_qkv_gpu(mbx, q)), _qkv_oracle(q), f"hd={hd} H={heads}")


def test_qkv_epilogue_image_only_and_guard_zone(mbx):
    q = synth.qkv_epilogue_case(batch=2, s_txt=3, grid_h=4, grid_w=4, heads=4)
    q["txt"] = None
    q["cos_txt"] = q["sin_txt"] = torch.zeros(0, 64)
    out, check = guarded((2, 3, 4, 16, 128), DEV)
    _qkv_gpu(mbx, q, out=out)
    torch.cuda.synchronize()
    check()
    assert_bits_equal(u16(out), _qkv_oracle(q), "image only")


# ------------------------------------------------------------------ config 4


def test_video_dit_per_token_full_size(mbx):
    """Video-DiT per-token modulation at its full size, as the benchmark runs
    it: every element of both operations, lossless bit for bit and high
    within 2 ulps of the binary64 result."""
    d = synth.video_dit_block(device=DEV)
    x, sc, sh, g, r, w = (d[k] for k in ("x", "scale", "shift", "gate", "residual", "weight"))
    X, SC, SH, G, R, W = (host_rows(t) for t in (x, sc, sh, g, r, w))
    W = W.reshape(-1)
    T = X.shape[0]

    got = host_rows(mbx.ln_modulate(x, sc, sh))
    par_rows(lambda lo, hi: assert_bits_equal(
        got[lo:hi], oracle.ln_modulate(X[lo:hi], SC[lo:hi], SH[lo:hi], 1e-6), f"ln per-token rows {lo}:{hi}"), T)
    got = host_rows(mbx.ln_modulate(x, sc, sh, variant="high"))
    par_rows(lambda lo, hi: assert_high_close(
        got[lo:hi], *oracle.ln_modulate_f64(X[lo:hi], SC[lo:hi], SH[lo:hi], 1e-6), what=f"ln high rows {lo}:{hi}"), T)
    got = host_rows(mbx.rmsnorm_tanh_residual(x, g, r, w))
    par_rows(lambda lo, hi: assert_bits_equal(
        got[lo:hi], oracle.rmsnorm_tanh_residual(X[lo:hi], G[lo:hi], R[lo:hi], W, 1e-6),
        f"tanh residual rows {lo}:{hi}"), T)
    got = host_rows(mbx.rmsnorm_tanh_residual(x, g, r, w, variant="high"))
    par_rows(lambda lo, hi: assert_high_close(
        got[lo:hi], *oracle.rmsnorm_tanh_residual_f64(X[lo:hi], G[lo:hi], R[lo:hi], W, 1e-6),
        what=f"tanh residual high rows {lo}:{hi}"), T)


# ------------------------------------------------------------------ config 5 (sweep)


def _sweep_ops(mbx, d):
    """The four row operations on a sweep cell: {op: (gpu call(variant), oracle(lo, hi), binary64(lo, hi))}
    with the oracle sides reading host copies of the inputs."""
    x, y, gt, r, sc, sh, g, w = (d[k] for k in ("x", "y", "gate_tok", "residual", "scale", "shift", "gate", "weight"))
    X, Y, GT, R = (host_rows(t) for t in (x, y, gt, r))
    SC, SH, G, W = u16(sc), u16(sh), u16(g), u16(w)
    return {
        "ln_modulate": (lambda v: mbx.ln_modulate(x, sc, sh, variant=v),
                        lambda lo, hi: oracle.ln_modulate(X[lo:hi], SC, SH, 1e-6),
                        lambda lo, hi: oracle.ln_modulate_f64(X[lo:hi], SC, SH, 1e-6)),
        "rmsnorm_scale": (lambda v: mbx.rmsnorm_scale(x, w, sc, variant=v),
                          lambda lo, hi: oracle.rmsnorm_scale(X[lo:hi], W, SC, 1e-6),
                          lambda lo, hi: oracle.rmsnorm_scale_f64(X[lo:hi], W, SC, 1e-6)),
        "rmsnorm_tanh_residual": (lambda v: mbx.rmsnorm_tanh_residual(x, gt, r, w, variant=v),
                                  lambda lo, hi: oracle.rmsnorm_tanh_residual(X[lo:hi], GT[lo:hi], R[lo:hi], W, 1e-6),
                                  lambda lo, hi: oracle.rmsnorm_tanh_residual_f64(X[lo:hi], GT[lo:hi], R[lo:hi], W,
                                                                                  1e-6)),
        "residual_gate_add": (lambda v: mbx.residual_gate_add(x, g, y, variant=v),
                              lambda lo, hi: oracle.residual_gate_add(X[lo:hi], G, Y[lo:hi]),
                              lambda lo, hi: oracle.residual_gate_add_f64(X[lo:hi], G, Y[lo:hi])),
    }


@pytest.mark.parametrize("D", synth.SWEEP_D)
@pytest.mark.parametrize("T", synth.SWEEP_T)
def test_sweep(mbx, D, T):
    """Every element of every cell (T up to 65536 rows of D up to 8192), both
    variants, padded input rows with NaN sentinels in the pad."""
    d = synth.sweep_case(D, T, device=DEV)
    for name, (gpu, want, exact) in _sweep_ops(mbx, d).items():
        got = host_rows(gpu("lossless"))
        par_rows(lambda lo, hi: assert_bits_equal(got[lo:hi], want(lo, hi), f"{name} D={D} T={T} rows {lo}:{hi}"), T)
        got = host_rows(gpu("high"))
        par_rows(lambda lo, hi: assert_high_close(got[lo:hi], *exact(lo, hi),
                                                  what=f"{name} high D={D} T={T} rows {lo}:{hi}"), T)
        del got


@pytest.mark.parametrize("D", [1024, 4096, 8192])
def test_sweep_qkv(mbx, D):
    """The epilogue on sweep hidden sizes: H = D/128 heads of 128, a square-ish
    image grid, 77 text tokens, padded rows."""
    h, w = synth.grid_for(256)
    q = synth.qkv_epilogue_case(batch=1, s_txt=77, grid_h=h, grid_w=w, heads=D // 128, row_pad=64)
    assert_bits_equal(u16(_qkv_gpu(mbx, q)), _qkv_oracle(q), f"qkv D={D}")
