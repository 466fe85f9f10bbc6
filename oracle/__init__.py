"""CPU oracle for the DiT norm/modulation path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding in ``modulation_bit_exact_gb300``) never imports it, and the two
share no code: the arithmetic lives in ``mbx_oracle.c`` (plain C, compiled with
``-ffp-contract=off`` and without fast-math), this module only marshals numpy
arrays of bfloat16 bit patterns (``uint16``) into it.

Every function cites the passage it follows in its docstring; the readings the
oracle takes where the pages are silent are listed at the top of the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mbx_oracle.c")
_SO = os.path.join(_HERE, "libmbx_oracle.so")
# The flags are part of the oracle's definition: no fused multiply-add, no
# fast-math, IEEE binary32 arithmetic rounded to nearest-even everywhere.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile ``mbx_oracle.c`` into ``libmbx_oracle.so`` next to it."""
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            sig = {
                "orc_f32_to_bf16": [_p, _p, _i64],
                "orc_bf16_to_f32": [_p, _p, _i64],
                "orc_welford128": [_p, _i64, _p, _p, _p],
                "orc_sum128_sq": [_p, _i64, _p],
                "orc_tanh_bf16_table": [_p],
                "orc_ln_modulate": [_p, _i64, _p, _i64, _i64, _i64, _p, _i64, _p, _i64, _i64, _f32],
                "orc_rmsnorm_scale": [_p, _i64, _p, _i64, _i64, _i64, _p, _p, _i64, _i64, _f32],
                "orc_rmsnorm_tanh_residual": [_p, _i64, _p, _i64, _i64, _i64, _p, _i64, _i64,
                                              _p, _i64, _p, _f32],
                "orc_residual_gate_add": [_p, _i64, _p, _i64, _i64, _i64, _p, _i64, _i64, _p, _i64],
                "orc_gated_residual_ln_modulate": [_p, _p, _p, _i64, _i64, _i64, _p, _i64, _p, _p,
                                                   _i64, _p, _i64, _p, _i64, _i64, _f32],
                "orc_f32_to_e4m3": [_p, _p, _i64],
                "orc_quant_e4m3": [_p, _i64, _p, _i64, _i64, _i64, _f32],
                "orc_f32_to_e2m1": [_p, _p, _i64],
                "orc_quant_nvfp4": [_p, _i64, _p, _p, _i64, _i64, _i64, _f32],
                "orc_modulation_table_add": [_p, _i64, _p, _i64, ctypes.c_int, _p, _i64,
                                             ctypes.c_int, _i64, _i64],
                "orc_qkv_epilogue": [_p, _p, _i64, _i64, _p, _i64, _i64, _i64, _i64, _i64,
                                     _p, _p, _p, _p, _p, _p, _p, _p, _f32],
                "orc_ln_modulate_f64": [_p, _p, _p, _i64, _i64, _i64, _p, _i64, _p, _i64, _i64, _f32],
                "orc_rmsnorm_scale_f64": [_p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _i64, _f32],
                "orc_rmsnorm_tanh_residual_f64": [_p, _p, _p, _i64, _i64, _i64, _p, _i64, _i64,
                                                  _p, _i64, _p, _f32],
                "orc_residual_gate_add_f64": [_p, _p, _p, _i64, _i64, _i64, _p, _i64, _i64, _p, _i64],
                "orc_qk_head_f64": [_p, _p, _p, _i64, _p, _p, _p, _f32],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = None
            L.orc_probe_mul_add.argtypes = [_f32, _f32, _f32]
            L.orc_probe_mul_add.restype = _f32
            _lib = L
    return _lib


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _rows(a: np.ndarray) -> tuple[np.ndarray, int]:
    """A 2-D uint16 view with a contiguous last dim; returns (array, row stride)."""
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bfloat16 bit patterns (numpy uint16)")
    if a.ndim == 1:
        a = a.reshape(1, -1)
    if a.ndim != 2:
        a = a.reshape(-1, a.shape[-1])
    if a.strides[1] != 2:
        raise ValueError("last dimension must be contiguous")
    return a, a.strides[0] // 2 if a.shape[0] > 1 else a.shape[1]


def _mat(a: np.ndarray) -> tuple[np.ndarray, int, int]:
    """A 2-D bfloat16 (uint16 bits) or binary32 matrix with a contiguous last
    dim; returns (array, row stride in elements, 1 if binary32)."""
    if a.dtype not in (np.uint16, np.float32):
        raise TypeError("expected bfloat16 bit patterns (uint16) or float32")
    if a.ndim != 2:
        a = a.reshape(-1, a.shape[-1])
    if a.strides[1] != a.itemsize:
        raise ValueError("last dimension must be contiguous")
    stride = a.strides[0] // a.itemsize if a.shape[0] > 1 else a.shape[1]
    return a, stride, int(a.dtype == np.float32)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def f32_to_bf16(v: np.ndarray) -> np.ndarray:
    """Reading R1 of the oracle: binary32 -> bfloat16 nearest-even bit patterns."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16(_ptr(v), _ptr(out), v.size)
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    lib().orc_bf16_to_f32(_ptr(b), _ptr(out), b.size)
    return out


def probe_mul_add(a: float, b: float, c: float) -> float:
    return float(lib().orc_probe_mul_add(a, b, c))


def welford128(row: np.ndarray) -> tuple[float, float, float]:
    """Welford statistics of one row in the fixed 128-lane order (mean, M2, n).

    Follows the bit-exact LayerNorm description of the tahou.com SGLang
    diffusion article, section 扩散Kernel对数值精度的敏感性 (128-thread Welford,
    fixed shuffle tree, round-to-nearest division).
    """
    row = np.ascontiguousarray(row, dtype=np.uint16).reshape(-1)
    m = np.zeros(3, dtype=np.float32)
    lib().orc_welford128(_ptr(row), row.size, _ptr(m), _ptr(m[1:]), _ptr(m[2:]))
    return float(m[0]), float(m[1]), float(m[2])


def sum128_sq(row: np.ndarray) -> float:
    """binary32 sum of bf16(x*x) over the 128-lane order (BF16-native RMSNorm)."""
    row = np.ascontiguousarray(row, dtype=np.uint16).reshape(-1)
    s = np.zeros(1, dtype=np.float32)
    lib().orc_sum128_sq(_ptr(row), row.size, _ptr(s))
    return float(s[0])


def tanh_table() -> np.ndarray:
    """All 65536 values of tanh_bf16 (the bfloat16 nearest to the exact tanh)."""
    t = np.empty(65536, dtype=np.uint16)
    lib().orc_tanh_bf16_table(_ptr(t))
    return t


def _mod_rows(x2: np.ndarray, m: np.ndarray, D: int) -> tuple[np.ndarray, int, int]:
    m2, ms = _rows(m)
    if m2.shape[1] != D:
        raise ValueError("modulation width differs from x")
    if x2.shape[0] % m2.shape[0] != 0:
        raise ValueError("rows of x must be a multiple of the modulation rows")
    return m2, ms, m2.shape[0]


def ln_modulate(x: np.ndarray, scale: np.ndarray, shift: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """LayerNorm (no affine) + AdaLN modulate, bit-exact eager chain.

    tahou.com SGLang diffusion article, section 扩散Kernel对数值精度的敏感性:
    ``y = LN(x); y = y*(1+scale)+shift`` with a BF16 store after LN and after
    each step of the multiply-add.  Row r uses modulation row r // (rows //
    mod_rows) (prhub.com.cn PR #34085 digest, 关键源码片段: batch = row //
    seq_len).
    """
    x2, xs = _rows(x)
    rows, D = x2.shape
    sc, scs, mrows = _mod_rows(x2, scale, D)
    sh, shs, mrows2 = _mod_rows(x2, shift, D)
    if mrows2 != mrows:
        raise ValueError("scale and shift rows differ")
    out = np.empty((rows, D), dtype=np.uint16)
    lib().orc_ln_modulate(_ptr(out), D, _ptr(x2), xs, rows, D, _ptr(sc), scs, _ptr(sh), shs,
                          mrows, eps)
    return out


def rmsnorm_scale(x: np.ndarray, weight: np.ndarray, scale: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """BF16-native RMSNorm * weight * scale.

    prhub.com.cn digest of SGLang PR #34085, section 关键源码片段 (the
    ``_rmsnorm_scale_kernel`` excerpt): square, sum, mean, rstd and each product
    are rounded back to bfloat16 at the points that excerpt gives.
    """
    x2, xs = _rows(x)
    rows, D = x2.shape
    w = np.ascontiguousarray(weight, dtype=np.uint16).reshape(-1)
    if w.size != D:
        raise ValueError("weight must have D elements")
    sc, scs, mrows = _mod_rows(x2, scale, D)
    out = np.empty((rows, D), dtype=np.uint16)
    lib().orc_rmsnorm_scale(_ptr(out), D, _ptr(x2), xs, rows, D, _ptr(w), _ptr(sc), scs, mrows, eps)
    return out


def rmsnorm_tanh_residual(x: np.ndarray, gate: np.ndarray, residual: np.ndarray,
                          weight: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """``out = r + tanh(g) * RMSNorm(x) * w``, BF16-native.

    prhub.com.cn PR #34085 digest, 实现拆解 item 2 (rmsnorm_tanh_residual moved
    out of Z-Image); 163.com sglang.kernels article, 3.2 (rmsnorm+tanh(gate)·x
    +residual).  The norm chain is the rmsnorm_scale chain without the scale.
    """
    x2, xs = _rows(x)
    rows, D = x2.shape
    g2, gs, grows = _mod_rows(x2, gate, D)
    r2, rs = _rows(residual)
    if r2.shape != (rows, D):
        raise ValueError("residual must match x")
    w = np.ascontiguousarray(weight, dtype=np.uint16).reshape(-1)
    out = np.empty((rows, D), dtype=np.uint16)
    lib().orc_rmsnorm_tanh_residual(_ptr(out), D, _ptr(x2), xs, rows, D, _ptr(g2), gs, grows,
                                    _ptr(r2), rs, _ptr(w), eps)
    return out


def residual_gate_add(x: np.ndarray, gate: np.ndarray, y: np.ndarray) -> np.ndarray:
    """``out = bf16(x + bf16(gate * y))`` (PR #34085 digest, 实现拆解 item 3;
    163.com sglang.kernels article, 3.2: residual + gate·update)."""
    x2, xs = _rows(x)
    rows, D = x2.shape
    g2, gs, grows = _mod_rows(x2, gate, D)
    y2, ys = _rows(y)
    if y2.shape != (rows, D):
        raise ValueError("y must match x")
    out = np.empty((rows, D), dtype=np.uint16)
    lib().orc_residual_gate_add(_ptr(out), D, _ptr(x2), xs, rows, D, _ptr(g2), gs, grows, _ptr(y2), ys)
    return out


def f32_to_e4m3(v: np.ndarray) -> np.ndarray:
    """binary32 -> FP8 E4M3 bytes: nearest-even, saturating to +-448, NaN -> 0x7F."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_f32_to_e4m3(_ptr(v), _ptr(out), v.size)
    return out


def quant_e4m3(y: np.ndarray, scale: float) -> np.ndarray:
    """Static per-tensor E4M3 copy of a bfloat16 output (tahou.com article,
    section 将FP8量化融合到前序算子): e4m3(float(y) * (1/scale)), the reciprocal
    correctly rounded in binary32."""
    y2, ys = _rows(y)
    rows, D = y2.shape
    out = np.empty((rows, D), dtype=np.uint8)
    lib().orc_quant_e4m3(_ptr(out), D, _ptr(y2), ys, rows, D, float(scale))
    return out.reshape(y.shape)


def f32_to_e2m1(v: np.ndarray) -> np.ndarray:
    """binary32 -> FP4 E2M1 codes (one per byte): nearest, ties to even,
    saturating to +-6, NaN -> +6."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_f32_to_e2m1(_ptr(v), _ptr(out), v.size)
    return out


def nvfp4_sf_shape(rows: int, D: int) -> tuple[int, int]:
    """Bytes of the 128x4-swizzled scale buffer: rows padded to 128, blocks to 4."""
    return ((rows + 127) // 128) * 128, ((D // 16 + 3) // 4) * 4


def quant_nvfp4(y: np.ndarray, gs: float, sf_fill: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4 copy of a bfloat16 output (tahou.com article, section
    将FP8量化融合到前序算子, NVFP4 path; readings at orc_quant_nvfp4): returns
    (packed E2M1 [rows, D/2] uint8, swizzled E4M3 scales, flat, padding =
    sf_fill)."""
    y2, ys = _rows(y)
    rows, D = y2.shape
    if D % 16:
        raise ValueError("D must be a multiple of 16")
    out = np.empty((rows, D // 2), dtype=np.uint8)
    mp, kp = nvfp4_sf_shape(rows, D)
    sf = np.full(mp * kp, sf_fill, dtype=np.uint8)
    lib().orc_quant_nvfp4(_ptr(out), D // 2, _ptr(sf), _ptr(y2), ys, rows, D, float(gs))
    return out, sf


def modulation_table_add(table: np.ndarray, temb: np.ndarray) -> np.ndarray:
    """Per-token modulation table in the (6, rows, D) layout, binary32.

    tahou.com article, section Wan视频模型的数据搬运优化: the eager
    ``(table.unsqueeze(0) + temb.float()).chunk(6, dim=2)``, each of the six
    chunks written as a contiguous plane; one binary32 addition per element.
    table [6, D] and temb [rows, 6*D] (or [..., 6, D]) are bfloat16 bit
    patterns (uint16) or float32.
    """
    t2, ts, tf = _mat(table)
    if t2.shape[0] != 6:
        raise ValueError("table must have 6 rows")
    D = t2.shape[1]
    e = temb.reshape(-1, 6 * D) if temb.shape[-1] != 6 * D else temb
    e2, es, ef = _mat(e)
    if e2.shape[1] != 6 * D:
        raise ValueError("temb rows must hold 6*D elements")
    rows = e2.shape[0]
    out = np.empty((6, rows, D), dtype=np.float32)
    lib().orc_modulation_table_add(_ptr(out), D, _ptr(t2), ts, tf, _ptr(e2), es, ef, rows, D)
    return out


def gated_residual_ln_modulate(residual: np.ndarray, gate: np.ndarray, update: np.ndarray,
                               bias, scale: np.ndarray, shift: np.ndarray,
                               eps: float = 1e-6) -> tuple[np.ndarray, np.ndarray]:
    """Gated residual update fused into LN + AdaLN modulate; returns (r', out).

    tahou.com SGLang diffusion article, section Qwen-Image FP8和NVFP4优化 (the
    ``residual = residual + gate * (attention + bias)`` chain, then layer_norm
    and ``* (1 + scale) + shift``), each step rounded to bfloat16 as the eager
    chain rounds it; r' is the new residual stream, out the modulated norm.
    """
    r2, rs = _rows(residual)
    rows, D = r2.shape
    u2, us = _rows(update)
    if u2.shape != (rows, D):
        raise ValueError("update must match residual")
    g2, gs, mrows = _mod_rows(r2, gate, D)
    sc, scs, m2 = _mod_rows(r2, scale, D)
    sh, shs, m3 = _mod_rows(r2, shift, D)
    if not (mrows == m2 == m3):
        raise ValueError("gate, scale and shift must share their rows")
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.uint16).reshape(-1)
    if b is not None and b.size != D:
        raise ValueError("bias must have D elements")
    res_out = np.empty((rows, D), dtype=np.uint16)
    out = np.empty((rows, D), dtype=np.uint16)
    lib().orc_gated_residual_ln_modulate(_ptr(res_out), _ptr(out), _ptr(r2), rs, rows, D, _ptr(u2), us,
                                         None if b is None else _ptr(b), _ptr(g2), gs, _ptr(sc), scs,
                                         _ptr(sh), shs, mrows, eps)
    return res_out, out


def qkv_epilogue(txt: np.ndarray | None, img: np.ndarray | None, batch: int, heads: int,
                 head_dim: int, wq_txt, wk_txt, wq_img, wk_img,
                 cos_txt, sin_txt, cos_img, sin_img, eps: float = 1e-6) -> np.ndarray:
    """Fused post-GEMM QKV epilogue into the joint [B, 3, H, S_txt+S_img, hd] buffer.

    tahou.com SGLang diffusion article, section 合并QKV投影时的数值问题: Q/K
    RMSNorm, interleaved RoPE, V copy, text and image tokens written into one
    joint QKV buffer.  Tables are per token, [S, hd/2] binary32.
    """
    width = 3 * heads * head_dim

    def branch(a):
        if a is None or a.size == 0:
            return np.zeros((0, width), dtype=np.uint16), width, 0
        a2, st = _rows(a)
        if a2.shape[1] != width or a2.shape[0] % batch:
            raise ValueError("branch must be [B*S, 3*H*hd]")
        return a2, st, a2.shape[0] // batch

    t2, ts, s_txt = branch(txt)
    i2, is_, s_img = branch(img)
    joint = np.empty((batch, 3, heads, s_txt + s_img, head_dim), dtype=np.uint16)

    def w(v):
        return np.ascontiguousarray(v, dtype=np.uint16).reshape(-1)

    def tab(v, S):
        a = np.ascontiguousarray(v, dtype=np.float32).reshape(-1)
        if a.size != S * (head_dim // 2):
            raise ValueError("tables must be [S, hd/2]")
        return a

    ws = [w(wq_txt), w(wk_txt), w(wq_img), w(wk_img)]
    tabs = [tab(cos_txt, s_txt), tab(sin_txt, s_txt), tab(cos_img, s_img), tab(sin_img, s_img)]
    lib().orc_qkv_epilogue(_ptr(joint), _ptr(t2), ts, s_txt, _ptr(i2), is_, s_img, batch, heads,
                           head_dim, *[_ptr(v) for v in ws], *[_ptr(v) for v in tabs], eps)
    return joint


# --------------------------------------------------------------------------
# binary64 references (for the single-pass "high" variants)
# --------------------------------------------------------------------------

def ln_modulate_f64(x, scale, shift, eps=1e-6):
    x2, xs = _rows(x)
    rows, D = x2.shape
    sc, scs, mrows = _mod_rows(x2, scale, D)
    sh, shs, _ = _mod_rows(x2, shift, D)
    out = np.empty((rows, D)); mag = np.empty((rows, D))
    lib().orc_ln_modulate_f64(_ptr(out), _ptr(mag), _ptr(x2), xs, rows, D, _ptr(sc), scs,
                              _ptr(sh), shs, mrows, eps)
    return out, mag


def rmsnorm_scale_f64(x, weight, scale, eps=1e-6):
    x2, xs = _rows(x)
    rows, D = x2.shape
    w = np.ascontiguousarray(weight, dtype=np.uint16).reshape(-1)
    sc, scs, mrows = _mod_rows(x2, scale, D)
    out = np.empty((rows, D)); mag = np.empty((rows, D))
    lib().orc_rmsnorm_scale_f64(_ptr(out), _ptr(mag), _ptr(x2), xs, rows, D, _ptr(w), _ptr(sc),
                                scs, mrows, eps)
    return out, mag


def rmsnorm_tanh_residual_f64(x, gate, residual, weight, eps=1e-6):
    x2, xs = _rows(x)
    rows, D = x2.shape
    g2, gs, grows = _mod_rows(x2, gate, D)
    r2, rs = _rows(residual)
    w = np.ascontiguousarray(weight, dtype=np.uint16).reshape(-1)
    out = np.empty((rows, D)); mag = np.empty((rows, D))
    lib().orc_rmsnorm_tanh_residual_f64(_ptr(out), _ptr(mag), _ptr(x2), xs, rows, D, _ptr(g2), gs,
                                        grows, _ptr(r2), rs, _ptr(w), eps)
    return out, mag


def residual_gate_add_f64(x, gate, y):
    x2, xs = _rows(x)
    rows, D = x2.shape
    g2, gs, grows = _mod_rows(x2, gate, D)
    y2, ys = _rows(y)
    out = np.empty((rows, D)); mag = np.empty((rows, D))
    lib().orc_residual_gate_add_f64(_ptr(out), _ptr(mag), _ptr(x2), xs, rows, D, _ptr(g2), gs,
                                    grows, _ptr(y2), ys)
    return out, mag


def qk_head_f64(src_row, w, cosv, sinv, eps=1e-6):
    src = np.ascontiguousarray(src_row, dtype=np.uint16).reshape(-1)
    hd = src.size
    w = np.ascontiguousarray(w, dtype=np.uint16).reshape(-1)
    c = np.ascontiguousarray(cosv, dtype=np.float32).reshape(-1)
    s = np.ascontiguousarray(sinv, dtype=np.float32).reshape(-1)
    out = np.empty(hd); mag = np.empty(hd)
    lib().orc_qk_head_f64(_ptr(out), _ptr(mag), _ptr(src), hd, _ptr(w), _ptr(c), _ptr(s), eps)
    return out, mag
