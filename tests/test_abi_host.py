"""Host-side tests of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching a device.

No kernel runs here.  Pointers are fake host addresses that the library never
dereferences: every case below fails a pure host check, which runs before the
device checks.
"""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mbx.h")


@pytest.fixture(scope="module")
def mbx():
    from modulation_bit_exact_gb300 import _build
    _build.build()
    import modulation_bit_exact_gb300 as m
    m.lib()
    return m


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MBX_API\s+[\w\s\*]+?\b(mbx_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for op in ("mbx_ln_modulate", "mbx_rmsnorm_scale", "mbx_rmsnorm_tanh_residual",
               "mbx_residual_gate_add", "mbx_qk_norm_rope_qkv_epilogue",
               "mbx_gated_residual_ln_modulate", "mbx_modulation_table_add"):
        assert op in names and op.replace("mbx_", "mbx_check_") in names


def test_library_exports_every_declared_symbol(mbx):
    L = mbx.lib()
    for name in declared_symbols():
        assert hasattr(L, name), name
    assert L.mbx_abi_version() == 1


def test_library_exports_nothing_else(mbx):
    out = os.popen(f"nm -D --defined-only {mbx.library_path}").read()
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    ours = {s for s in exported if s.startswith("mbx_")}
    assert ours == set(declared_symbols())


def test_status_strings(mbx):
    for code, name in mbx.STATUS.items():
        assert mbx.status_string(code).startswith(name)
    assert mbx.status_string(-999).startswith("MBX_E_UNKNOWN")


# ---------------------------------------------------------------- fake views

BASE = 0x10000000  # never dereferenced


def V(data=BASE, rows=4, cols=64, stride=None, dtype=1, mbx=None):
    from modulation_bit_exact_gb300 import _View
    return _View(data, rows, cols, cols if stride is None else stride, dtype)


def ref(v):
    return ctypes.byref(v)


def ln_status(L, out, x, sc, sh, eps=1e-6, variant=0):
    a = L.mbx_check_ln_modulate(ref(out), ref(x), ref(sc), ref(sh), eps, variant)
    b = L.mbx_ln_modulate(ref(out), ref(x), ref(sc), ref(sh), eps, variant, None)
    assert a == b
    return a


def views(rows=4, cols=64, mrows=2):
    return (V(BASE, rows, cols), V(BASE + 0x100000, rows, cols), V(BASE + 0x200000, mrows, cols),
            V(BASE + 0x300000, mrows, cols))


def test_ln_modulate_rejections(mbx):
    L = mbx.lib()
    o, x, sc, sh = views()
    assert L.mbx_ln_modulate(None, ref(x), ref(sc), ref(sh), 1e-6, 0, None) == -1
    assert ln_status(L, o, V(0, 4, 64), sc, sh) == -1                       # NULL data
    assert ln_status(L, o, V(BASE + 0x100000, 4, 64, dtype=0), sc, sh) == -2  # mixed dtypes
    assert ln_status(L, o, x, V(BASE + 0x200000, 2, 64, dtype=7), sh) == -2
    assert ln_status(L, V(BASE, 0, 64), V(BASE + 0x100000, 0, 64), sc, sh) == -3  # empty
    assert ln_status(L, V(BASE, 4, 0), V(BASE + 0x100000, 4, 0), sc, sh) == -3
    big = 8200
    assert ln_status(L, V(BASE, 4, big), V(BASE + 0x100000, 4, big),
                     V(BASE + 0x200000, 2, big), V(BASE + 0x300000, 2, big)) == -4  # D > 8192
    assert ln_status(L, o, x, V(BASE + 0x200000, 3, 64), V(BASE + 0x300000, 3, 64)) == -5  # 4 % 3
    assert ln_status(L, o, x, V(BASE + 0x200000, 2, 32), sh) == -5           # width
    assert ln_status(L, V(BASE, 5, 64), x, sc, sh) == -5                     # out rows
    assert ln_status(L, o, V(BASE + 0x100000, 4, 64, stride=32), sc, sh) == -6  # stride < cols
    assert ln_status(L, o, V(BASE + 0x100001, 4, 64), sc, sh) == -7          # odd address
    assert ln_status(L, o, x, sc, sh, variant=2) == -11
    for eps in (float("nan"), -1e-6, float("inf")):
        assert ln_status(L, o, x, sc, sh, eps=eps) == -12
    assert ln_status(L, o, V(BASE + 64, 4, 64), sc, sh) == -8                # partial overlap
    assert ln_status(L, o, V(BASE, 4, 64), sc, sh) == -8                     # no in-place LN


def test_residual_gate_add_in_place_only_on_x(mbx):
    L = mbx.lib()
    o, x, g, y = V(BASE, 4, 64), V(BASE, 4, 64), V(BASE + 0x200000, 2, 64), V(BASE + 0x300000, 4, 64)

    def st(o, x, g, y):
        a = L.mbx_check_residual_gate_add(ref(o), ref(x), ref(g), ref(y), 0)
        assert a == L.mbx_residual_gate_add(ref(o), ref(x), ref(g), ref(y), 0, None)
        return a

    # exact in-place passes every host check and stops at the device check
    # (there is no device here, and a fake address is no device memory anyway)
    assert st(o, x, g, y) == -9
    assert st(o, V(BASE + 2, 4, 64), g, y) == -8               # shifted: partial overlap
    assert st(o, x, g, V(BASE, 4, 64)) == -8                   # out over y
    assert st(o, V(BASE, 4, 64, stride=128), g, y) == -8       # same start, other stride
    assert st(o, x, V(BASE + 0x200000, 3, 64), y) == -5
    assert st(o, x, g, V(BASE + 0x300000, 4, 32)) == -5


def test_rmsnorm_rejections(mbx):
    L = mbx.lib()
    o, x = V(BASE, 4, 64), V(BASE + 0x100000, 4, 64)
    w, sc = V(BASE + 0x200000, 1, 64), V(BASE + 0x300000, 2, 64)

    def st(o, x, w, sc, eps=1e-6, variant=0):
        a = L.mbx_check_rmsnorm_scale(ref(o), ref(x), ref(w), ref(sc), eps, variant)
        assert a == L.mbx_rmsnorm_scale(ref(o), ref(x), ref(w), ref(sc), eps, variant, None)
        return a

    assert st(o, x, V(BASE + 0x200000, 2, 64), sc) == -5       # weight must be [1, D]
    assert st(o, x, V(BASE + 0x200000, 1, 32), sc) == -5
    assert st(o, x, w, sc, variant=-1) == -11
    assert st(o, x, w, V(BASE + 0x300000, 2, 64, dtype=2)) == -2
    assert st(o, x, w, sc) == -9                                # host checks pass

    g, r = V(BASE + 0x300000, 4, 64), V(BASE + 0x400000, 4, 64)

    def st2(o, x, g, r, w):
        a = L.mbx_check_rmsnorm_tanh_residual(ref(o), ref(x), ref(g), ref(r), ref(w), 1e-6, 0)
        assert a == L.mbx_rmsnorm_tanh_residual(ref(o), ref(x), ref(g), ref(r), ref(w), 1e-6, 0, None)
        return a

    assert st2(V(BASE + 0x400000, 4, 64), x, g, r, w) == -9     # in place on the residual
    assert st2(V(BASE + 0x100000, 4, 64), x, g, r, w) == -8     # not on x
    assert st2(o, x, g, V(BASE + 0x400000, 3, 64), w) == -5
    assert st2(o, x, V(BASE + 0x300000, 3, 64), r, w) == -5


def qkv_status(L, joint, txt, img, batch=2, heads=4, hd=128, tables=True, weights=None,
               eps=1e-6, variant=0, cos_txt=None):
    ws = weights or [V(BASE + 0x800000 + i * 0x1000, 1, hd) for i in range(4)]
    t = [BASE + 0x900000 + i * 0x100000 for i in range(4)] if tables else [None] * 4
    if cos_txt is not None:
        t[0] = cos_txt
    args = [ref(joint), ref(txt), ref(img), batch, heads, *[ref(w) for w in ws], *t, eps, variant]
    a = L.mbx_check_qk_norm_rope_qkv_epilogue(*args)
    b = L.mbx_qk_norm_rope_qkv_epilogue(*args, None)
    assert a == b
    return a


def test_qkv_epilogue_rejections(mbx):
    L = mbx.lib()
    B, H, hd, st, si = 2, 4, 128, 8, 24
    width = 3 * H * hd
    joint = V(BASE, B * 3 * H * (st + si), hd)
    txt = V(BASE + 0x1000000, B * st, width)
    img = V(BASE + 0x2000000, B * si, width, stride=width + 64)
    assert qkv_status(L, joint, txt, img) == -9                      # host checks pass
    assert qkv_status(L, joint, txt, img, hd=96,
                      weights=[V(BASE + 0x800000, 1, 96)] * 4) == -5   # weights != [1, hd]
    assert qkv_status(L, V(BASE, B * 3 * H * (st + si), 96), txt, img) == -12
    assert qkv_status(L, joint, txt, img, batch=0) == -12
    assert qkv_status(L, joint, txt, img, heads=3) == -5             # width mismatch
    assert qkv_status(L, V(BASE, B * 3 * H * (st + si) + 1, hd), txt, img) == -5
    assert qkv_status(L, joint, V(BASE + 0x1000000, B * st + 1, width), img) == -5  # rows % B
    assert qkv_status(L, joint, txt, V(BASE + 0x2000008, B * si, width)) == -7       # 16 B
    assert qkv_status(L, joint, txt, img, cos_txt=BASE + 0x900004) == -7
    assert qkv_status(L, joint, txt, img, tables=False) == -1
    assert qkv_status(L, joint, V(0, 0, width), V(0, 0, width)) == -3               # both empty
    # text branch absent: allowed (then stops at the device check)
    joint_i = V(BASE, B * 3 * H * si, hd)
    assert qkv_status(L, joint_i, V(0, 0, width), img) == -9
    assert qkv_status(L, V(BASE + 0x1000000 + 256, B * 3 * H * (st + si), hd), txt, img) == -8
    assert qkv_status(L, joint, txt, img, variant=5) == -11


def test_selftest_rejections(mbx):
    L = mbx.lib()
    assert L.mbx_selftest(0, None, None) == -1
    assert L.mbx_selftest(7, BASE, None) == -12
    assert L.mbx_selftest(8, BASE, None) == -12
    assert L.mbx_selftest(6, BASE, None) == -9  # a valid mode: only the device check refuses
    assert L.mbx_selftest(-1, BASE, None) == -12
    assert L.mbx_selftest(0, BASE + 4, None) == -7


# ---------------------------------------------------------------- Python views


def test_flat_row_rule(mbx):
    rc = mbx._rows_cols
    assert rc(torch.empty(2, 3, 8)) == (6, 8, 8)
    buf = torch.empty(6, 72)
    assert rc(buf[:, :64]) == (6, 64, 72)                      # padded rows
    assert rc(torch.empty(8)) == (1, 8, 8)
    assert rc(torch.empty(2, 1, 8)) == (2, 8, 8)               # size-1 dims skipped
    assert rc(torch.empty(4, 8).t())[2] == -1                  # last dim not contiguous
    b3 = torch.empty(2, 5, 16)
    assert rc(b3[:, :4, :])[2] == -1                           # outer dim not flat over rows
    assert rc(torch.empty(3, 4, 10)[:, :, :8]) == (12, 8, 10)


def test_cpu_tensors_are_rejected_not_computed(mbx):
    """The product path has no CPU fallback: host tensors fail the device check."""
    x = torch.randn(4, 64).to(torch.bfloat16)
    sc = torch.zeros(1, 64, dtype=torch.bfloat16)
    with pytest.raises(mbx.MbxError) as e:
        mbx.ln_modulate(x, sc, sc)
    assert e.value.status == -9
    with pytest.raises(mbx.MbxError) as e:
        mbx.ln_modulate(x.float(), sc, sc)
    assert e.value.status == -2


def test_binding_names_match_the_header(mbx):
    for name in declared_symbols():
        if name in ("mbx_status_string", "mbx_abi_version"):
            continue
        py = name[len("mbx_"):]
        assert hasattr(mbx, py), py


def test_gated_residual_ln_modulate_rejections(mbx):
    L = mbx.lib()
    rows, D = 8, 64
    ro, o, r, u = (V(BASE + i * 0x100000, rows, D) for i in range(4))
    g, sc, sh = (V(BASE + (4 + i) * 0x100000, 2, D) for i in range(3))
    b = V(BASE + 0x800000, 1, D)

    def st(ro, o, r, g, u, b, sc, sh, eps=1e-6, variant=0):
        args = [ref(ro), ref(o), ref(r), ref(g), ref(u), None if b is None else ref(b), ref(sc), ref(sh),
                ctypes.c_float(eps), variant]
        a = L.mbx_check_gated_residual_ln_modulate(*args)
        assert a == L.mbx_gated_residual_ln_modulate(*args, None)
        return a

    assert st(ro, o, r, g, u, b, sc, sh) == -9                        # host checks pass
    assert st(ro, o, r, g, u, None, sc, sh) == -9                     # bias is optional
    assert st(V(BASE + 0x200000, rows, D), o, r, g, u, b, sc, sh) == -9  # in place on the residual
    assert st(V(BASE + 0x200002, rows, D), o, r, g, u, b, sc, sh) == -8  # shifted: partial overlap
    assert st(ro, V(BASE + 0x200000, rows, D), r, g, u, b, sc, sh) == -8  # out over the residual
    assert st(ro, o, r, g, V(BASE, rows, D), b, sc, sh) == -8          # residual_out over the update
    assert st(ro, o, r, V(BASE + 0x400000, 4, D), u, b, sc, sh) == -5  # gate rows differ
    assert st(ro, o, r, g, u, V(BASE + 0x800000, 2, D), sc, sh) == -5  # bias must be [1, D]
    assert st(ro, o, r, g, V(BASE + 0x300000, rows, 32), b, sc, sh) == -5
    assert st(ro, o, r, g, u, V(BASE + 0x800000, 1, D, dtype=0), sc, sh) == -2
    assert st(ro, o, r, g, u, b, sc, sh, variant=3) == -11
    assert st(ro, o, r, g, u, V(0, 1, D), sc, sh) == -1


def test_modulation_table_add_rejections(mbx):
    L = mbx.lib()
    rows, D = 10, 48

    def st(o, t, e):
        a = L.mbx_check_modulation_table_add(ref(o), ref(t), ref(e))
        assert a == L.mbx_modulation_table_add(ref(o), ref(t), ref(e), None)
        return a

    o = V(BASE, 6 * rows, D, dtype=2)
    t = V(BASE + 0x400000, 6, D, dtype=1)
    e = V(BASE + 0x800000, rows, 6 * D, dtype=1)
    assert st(o, t, e) == -9                                        # host checks pass
    assert st(o, V(BASE + 0x400000, 6, D, dtype=2), V(BASE + 0x800000, rows, 6 * D, dtype=2)) == -9
    assert st(V(BASE, 6 * rows, D, dtype=1), t, e) == -2            # out must be binary32
    assert st(o, V(BASE + 0x400000, 6, D, dtype=3), e) == -2        # unknown dtype
    assert st(o, V(BASE + 0x400000, 5, D), e) == -5                 # table has 6 rows
    assert st(o, t, V(BASE + 0x800000, rows, 6 * D + 8)) == -5      # temb rows hold 6*D
    assert st(V(BASE, 6 * rows + 6, D, dtype=2), t, e) == -5        # out holds 6*rows rows
    assert st(V(BASE + 0x800000, 6 * rows, D, dtype=2), t, e) == -8  # out over temb
    assert st(V(BASE + 2, 6 * rows, D, dtype=2), t, e) == -7         # f32 misaligned
    assert st(o, t, V(BASE + 0x800000, rows, 6 * D, 6 * D - 1)) == -6
    assert st(o, V(0, 6, D), e) == -1


def test_fp8_producer_rejections(mbx):
    L = mbx.lib()
    rows, D = 8, 64
    o, x = V(BASE, rows, D), V(BASE + 0x100000, rows, D)
    sc, sh = V(BASE + 0x200000, 2, D), V(BASE + 0x300000, 2, D)
    q = V(BASE + 0x400000, rows, D, dtype=3)
    fs = ctypes.c_void_p(BASE + 0x500000)

    def st(o, q, x, sc, sh, fs, eps=1e-6, variant=0):
        a = L.mbx_check_ln_modulate_fp8(ref(o), ref(q), ref(x), ref(sc), ref(sh), fs, ctypes.c_float(eps), variant)
        b = L.mbx_ln_modulate_fp8(ref(o), ref(q), ref(x), ref(sc), ref(sh), fs, ctypes.c_float(eps), variant, None)
        assert a == b
        return a

    assert st(o, q, x, sc, sh, fs) == -9                                   # host checks pass
    assert st(o, V(BASE + 0x400000, rows, D, dtype=1), x, sc, sh, fs) == -2  # fp8 output must be E4M3
    assert st(o, V(BASE + 0x400000, rows, D - 8, dtype=3), x, sc, sh, fs) == -5
    assert st(o, V(BASE + 0x100000 + 64, rows, D, dtype=3), x, sc, sh, fs) == -8  # over x
    assert st(o, V(BASE + 0x40, rows, D, dtype=3), x, sc, sh, fs) == -8     # over out
    assert st(o, q, x, sc, sh, None) == -1
    assert st(o, q, x, sc, sh, ctypes.c_void_p(BASE + 0x500002)) == -7      # scale misaligned
    assert st(o, q, x, sc, sh, fs, variant=5) == -11                         # the LN checks still apply
    # the gated form runs both sets of checks
    ro, u, g = V(BASE + 0x600000, rows, D), V(BASE + 0x700000, rows, D), V(BASE + 0x800000, 2, D)
    args = [ref(ro), ref(o), ref(q), ref(x), ref(g), ref(u), None, ref(sc), ref(sh), fs, ctypes.c_float(1e-6), 0]
    assert L.mbx_check_gated_residual_ln_modulate_fp8(*args) == -9
    assert L.mbx_gated_residual_ln_modulate_fp8(*args, None) == -9
    args[2] = ref(V(BASE + 0x700000, rows, D, dtype=3))                      # fp8 over the update
    assert L.mbx_check_gated_residual_ln_modulate_fp8(*args) == -8


def test_nvfp4_producer_rejections(mbx):
    L = mbx.lib()
    rows, D = 130, 64
    o, x = V(BASE, rows, D), V(BASE + 0x100000, rows, D)
    sc, sh = V(BASE + 0x200000, 2, D), V(BASE + 0x300000, 2, D)
    q = V(BASE + 0x400000, rows, D // 2, dtype=4)
    f = V(BASE + 0x500000, 256, 4, dtype=3)
    gs = ctypes.c_void_p(BASE + 0x600000)

    def st(o, q, f, x, sc, sh, gs):
        a = L.mbx_check_ln_modulate_nvfp4(ref(o), ref(q), ref(f), ref(x), ref(sc), ref(sh), gs, ctypes.c_float(1e-6), 0)
        b = L.mbx_ln_modulate_nvfp4(ref(o), ref(q), ref(f), ref(x), ref(sc), ref(sh), gs, ctypes.c_float(1e-6), 0, None)
        assert a == b
        return a

    assert st(o, q, f, x, sc, sh, gs) == -9                                     # host checks pass
    assert st(o, V(BASE + 0x400000, rows, D // 2, dtype=3), f, x, sc, sh, gs) == -2  # values must be E2M1X2
    assert st(o, q, V(BASE + 0x500000, 256, 4, dtype=4), x, sc, sh, gs) == -2      # scales must be E4M3
    assert st(o, q, V(BASE + 0x500000, 130, 4, dtype=3), x, sc, sh, gs) == -5      # rows padded to 128
    assert st(o, q, V(BASE + 0x500000, 256, 8, dtype=3), x, sc, sh, gs) == -5      # blocks padded to 4
    assert st(o, q, V(BASE + 0x500000, 256, 4, 8, dtype=3), x, sc, sh, gs) == -6   # scales contiguous
    assert st(o, V(BASE + 0x400000, rows, D, dtype=4), f, x, sc, sh, gs) == -5     # D/2 bytes a row
    assert st(o, q, V(BASE + 0x400000 + 64, 256, 4, dtype=3), x, sc, sh, gs) == -8  # scales over values
    assert st(o, q, f, x, sc, sh, None) == -1
    d2 = 72  # not a multiple of 16
    o2, x2 = V(BASE, rows, d2), V(BASE + 0x100000, rows, d2)
    sc2, sh2 = V(BASE + 0x200000, 2, d2), V(BASE + 0x300000, 2, d2)
    assert st(o2, V(BASE + 0x400000, rows, d2 // 2, dtype=4), V(BASE + 0x500000, 256, 8, dtype=3),
              x2, sc2, sh2, gs) == -5


def test_huge_extents_are_refused_not_wrapped(mbx):
    """A view whose byte extent does not fit in 63 bits, or whose end address
    would wrap, is refused as out of bounds (-10) by the host checks: the
    overlap and bounds checks never see a wrapped size.  rows = 2^61 with
    stride = cols = 8 would wrap to 0 bytes in 64-bit arithmetic."""
    L = mbx.lib()
    o, x, sc, sh = views(rows=4, cols=8)
    huge = 1 << 61
    assert ln_status(L, V(BASE, huge, 8), V(BASE + 0x100000, huge, 8), sc, sh) == -10
    assert ln_status(L, o, V(BASE + 0x100000, 4, 8, stride=1 << 62), sc, sh) == -10
    assert ln_status(L, o, V(BASE + 0x100000, 4, 8, stride=1 << 61), sc, sh) == -10  # 3*2^62 bytes
    assert ln_status(L, o, V(0xFFFFFFFFFFFFFFF0, 4, 8), sc, sh) == -10     # end address wraps
    assert ln_status(L, o, x, V(BASE + 0x200000, 2, 8, stride=1 << 62), sh) == -10
    # the largest extent that fits is not refused by this check (the device check follows)
    assert ln_status(L, o, V(BASE + 0x100000, 4, 8, stride=1 << 40), sc, sh) == -9
    # FP8 / NVFP4 extra outputs and the table op's binary32 views take the same check
    q = V(BASE + 0x400000, huge, 8, dtype=3)
    fs = ctypes.c_void_p(BASE + 0x500000)
    assert L.mbx_check_ln_modulate_fp8(ref(o), ref(q), ref(x), ref(sc), ref(sh), fs,
                                       ctypes.c_float(1e-6), 0) in (-5, -10)
    q = V(BASE + 0x400000, 4, 8, stride=1 << 62, dtype=3)
    assert L.mbx_check_ln_modulate_fp8(ref(o), ref(q), ref(x), ref(sc), ref(sh), fs,
                                       ctypes.c_float(1e-6), 0) == -10
    t = V(BASE, 6, 8, dtype=2)
    e = V(BASE + 0x100000, 4, 48, stride=1 << 61, dtype=2)
    out = V(BASE + 0x200000, 24, 8, dtype=2)
    assert L.mbx_check_modulation_table_add(ref(out), ref(t), ref(e)) == -10


def test_qkv_huge_heads_or_batch_refused(mbx):
    L = mbx.lib()
    B, H, hd, st, si = 2, 4, 128, 8, 24
    width = 3 * H * hd
    joint = V(BASE, B * 3 * H * (st + si), hd)
    txt = V(BASE + 0x1000000, B * st, width)
    img = V(BASE + 0x2000000, B * si, width)
    assert qkv_status(L, joint, txt, img, heads=1 << 61) == -12
    assert qkv_status(L, joint, txt, img, batch=1 << 40) == -12
