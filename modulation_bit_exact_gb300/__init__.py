"""modulation_bit_exact_gb300 -- bit-exact DiT norm/modulation kernels for GB300.

A thin binding of the C ABI in ``include/mbx.h`` (``libmbx.so``, built in-tree
for sm_103a by ``modulation_bit_exact_gb300._build``).  Every function here
only turns torch tensors into views (pointer, rows, cols, row stride), picks
the caller's current CUDA stream, calls the library and raises on a negative
status; all arithmetic runs in the library's CUDA kernels.  There is no CPU
path: if the library is missing, every call raises.

Views follow the flat-row rule of the BF16-native RMSNorm wrapper in
"#34085 [diffusion] Clean up kernels and shared fast paths" (prhub.com.cn),
section 关键源码片段: the last dimension must be contiguous; rows may be
padded (any row stride), and every outer dimension must be flat over the rows.
A tensor that breaks the rule is passed with a negative row stride, which the
library rejects (MBX_E_STRIDE).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "ln_modulate", "rmsnorm_scale", "rmsnorm_tanh_residual", "residual_gate_add",
    "qk_norm_rope_qkv_epilogue", "gated_residual_ln_modulate", "check_gated_residual_ln_modulate",
    "modulation_table_add", "check_modulation_table_add", "ln_modulate_fp8", "check_ln_modulate_fp8",
    "gated_residual_ln_modulate_fp8", "check_gated_residual_ln_modulate_fp8", "ln_modulate_nvfp4",
    "check_ln_modulate_nvfp4", "gated_residual_ln_modulate_nvfp4", "check_gated_residual_ln_modulate_nvfp4",
    "nvfp4_sf_shape",
    "check_ln_modulate", "check_rmsnorm_scale",
    "check_rmsnorm_tanh_residual", "check_residual_gate_add",
    "check_qk_norm_rope_qkv_epilogue", "selftest", "status_string", "MbxError",
    "LOSSLESS", "HIGH", "library_path",
]

LOSSLESS, HIGH = 0, 1
MBX_BF16, MBX_F32, MBX_E4M3, MBX_E2M1X2 = 1, 2, 3, 4
_VARIANTS = {"lossless": LOSSLESS, "high": HIGH, LOSSLESS: LOSSLESS, HIGH: HIGH}

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmbx.so")

STATUS = {
    0: "MBX_OK", -1: "MBX_E_NULL", -2: "MBX_E_DTYPE", -3: "MBX_E_EMPTY",
    -4: "MBX_E_DIM_TOO_LARGE", -5: "MBX_E_SHAPE", -6: "MBX_E_STRIDE", -7: "MBX_E_ALIGN",
    -8: "MBX_E_ALIAS", -9: "MBX_E_DEVICE", -10: "MBX_E_BOUNDS", -11: "MBX_E_VARIANT",
    -12: "MBX_E_ARG", -13: "MBX_E_CUDA",
}


class MbxError(ValueError):
    """A negative status from libmbx; ``.status`` holds the code."""

    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class _View(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("row_stride", ctypes.c_int64), ("dtype", ctypes.c_int32)]


_P = ctypes.POINTER(_View)
_i64, _f32, _int, _vp = ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_void_p

_lock = threading.Lock()
_lib = None


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(library_path):
            raise RuntimeError(
                f"{library_path} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc); "
                "this package has no CPU fallback")
        L = ctypes.CDLL(library_path)
        sig = {
            "mbx_ln_modulate": [_P, _P, _P, _P, _f32, _int, _vp],
            "mbx_rmsnorm_scale": [_P, _P, _P, _P, _f32, _int, _vp],
            "mbx_rmsnorm_tanh_residual": [_P, _P, _P, _P, _P, _f32, _int, _vp],
            "mbx_residual_gate_add": [_P, _P, _P, _P, _int, _vp],
            "mbx_ln_modulate_fp8": [_P, _P, _P, _P, _P, _vp, _f32, _int, _vp],
            "mbx_check_ln_modulate_fp8": [_P, _P, _P, _P, _P, _vp, _f32, _int],
            "mbx_gated_residual_ln_modulate_fp8": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _vp, _f32, _int, _vp],
            "mbx_check_gated_residual_ln_modulate_fp8": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _vp, _f32, _int],
            "mbx_ln_modulate_nvfp4": [_P, _P, _P, _P, _P, _P, _vp, _f32, _int, _vp],
            "mbx_check_ln_modulate_nvfp4": [_P, _P, _P, _P, _P, _P, _vp, _f32, _int],
            "mbx_gated_residual_ln_modulate_nvfp4": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _vp, _f32, _int, _vp],
            "mbx_check_gated_residual_ln_modulate_nvfp4": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _vp, _f32, _int],
            "mbx_modulation_table_add": [_P, _P, _P, _vp],
            "mbx_check_modulation_table_add": [_P, _P, _P],
            "mbx_gated_residual_ln_modulate": [_P, _P, _P, _P, _P, _P, _P, _P, _f32, _int, _vp],
            "mbx_check_gated_residual_ln_modulate": [_P, _P, _P, _P, _P, _P, _P, _P, _f32, _int],
            "mbx_qk_norm_rope_qkv_epilogue": [_P, _P, _P, _i64, _i64, _P, _P, _P, _P,
                                              _vp, _vp, _vp, _vp, _f32, _int, _vp],
            "mbx_check_ln_modulate": [_P, _P, _P, _P, _f32, _int],
            "mbx_check_rmsnorm_scale": [_P, _P, _P, _P, _f32, _int],
            "mbx_check_rmsnorm_tanh_residual": [_P, _P, _P, _P, _P, _f32, _int],
            "mbx_check_residual_gate_add": [_P, _P, _P, _P, _int],
            "mbx_check_qk_norm_rope_qkv_epilogue": [_P, _P, _P, _i64, _i64, _P, _P, _P, _P,
                                                    _vp, _vp, _vp, _vp, _f32, _int],
            "mbx_selftest": [_int, _vp, _vp],
            "mbx_abi_version": [],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _int
        L.mbx_status_string.argtypes = [_int]
        L.mbx_status_string.restype = ctypes.c_char_p
        _lib = L
        return L


def lib() -> ctypes.CDLL:
    return _load()


def status_string(status: int) -> str:
    return _load().mbx_status_string(int(status)).decode()


def _raise(status: int):
    if status != 0:
        raise MbxError(status, status_string(status))


# ---------------------------------------------------------------- views


def _rows_cols(t: torch.Tensor) -> tuple[int, int, int]:
    """(rows, cols, row_stride) of t under the flat-row rule; row_stride = -1
    when the rule is broken (the library then answers MBX_E_STRIDE).  Size-1
    dimensions are skipped: their strides never address anything."""
    if t.dim() == 0:
        return 1, 1, 1
    cols = t.shape[-1]
    rows = t.numel() // cols if cols else 0
    if cols > 1 and t.stride(-1) != 1:
        return rows, cols, -1
    outer = [d for d in range(t.dim() - 1) if t.shape[d] != 1]
    if not outer:
        return rows, cols, cols
    stride = t.stride(outer[-1])
    expect = stride * t.shape[outer[-1]]
    for d in reversed(outer[:-1]):
        if t.stride(d) != expect:
            return rows, cols, -1
        expect *= t.shape[d]
    return rows, cols, stride


def _view(t: torch.Tensor) -> _View:
    dtype = _DTYPES.get(t.dtype, 0)
    if t.is_contiguous() and t.dim() > 0:  # the common case, without the general walk
        cols = t.shape[-1]
        n = t.numel()
        if n:
            return _View(t.data_ptr(), n // cols, cols, cols, dtype)
    rows, cols, stride = _rows_cols(t)
    return _View(t.data_ptr() if t.numel() else None, rows, cols, stride, dtype)


_DTYPES = {torch.bfloat16: MBX_BF16, torch.float32: MBX_F32, torch.uint8: MBX_E4M3}
if hasattr(torch, "float8_e4m3fn"):
    _DTYPES[torch.float8_e4m3fn] = MBX_E4M3


def _ref(v: _View):
    return ctypes.byref(v)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t: torch.Tensor) -> int:
    """The caller's current CUDA stream on t's device (0 for host tensors,
    which the library then refuses)."""
    if not t.is_cuda:
        return 0
    if _raw_stream is not None:
        return _raw_stream(t.get_device())
    return torch.cuda.current_stream(t.device).cuda_stream


def _variant(v) -> int:
    try:
        return _VARIANTS[v]
    except KeyError:
        return 99  # rejected by the library (MBX_E_VARIANT)


def _empty_like_rows(x: torch.Tensor) -> torch.Tensor:
    return torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)


# ---------------------------------------------------------------- operations


def ln_modulate(x, scale, shift, eps: float = 1e-6, variant="lossless", out=None):
    """LayerNorm (no affine) + AdaLN modulate: out = LN(x) * (1 + scale) + shift.

    x [..., D]; scale, shift [mod_rows, D] (any flat shape), with row r of x
    using modulation row r // (rows // mod_rows).  See mbx_ln_modulate.
    """
    L = _load()
    out = _empty_like_rows(x) if out is None else out
    o, xv, sc, sh = _view(out), _view(x), _view(scale), _view(shift)
    _raise(L.mbx_ln_modulate(_ref(o), _ref(xv), _ref(sc), _ref(sh), eps, _variant(variant),
                             _stream(x)))
    return out


def rmsnorm_scale(x, weight, scale, eps: float = 1e-6, variant="lossless", out=None):
    """BF16-native RMSNorm * weight * scale (see mbx_rmsnorm_scale)."""
    L = _load()
    out = _empty_like_rows(x) if out is None else out
    o, xv, w, sc = _view(out), _view(x), _view(weight), _view(scale)
    _raise(L.mbx_rmsnorm_scale(_ref(o), _ref(xv), _ref(w), _ref(sc), eps, _variant(variant),
                               _stream(x)))
    return out


def rmsnorm_tanh_residual(x, gate, residual, weight, eps: float = 1e-6, variant="lossless",
                          out=None):
    """out = residual + tanh(gate) * RMSNorm(x) * weight (see
    mbx_rmsnorm_tanh_residual); ``out=residual`` updates the residual in place."""
    L = _load()
    out = _empty_like_rows(x) if out is None else out
    o, xv, g, r, w = _view(out), _view(x), _view(gate), _view(residual), _view(weight)
    _raise(L.mbx_rmsnorm_tanh_residual(_ref(o), _ref(xv), _ref(g), _ref(r), _ref(w), eps,
                                       _variant(variant), _stream(x)))
    return out


def residual_gate_add(x, gate, y, variant="lossless", out=None):
    """out = x + gate * y (see mbx_residual_gate_add); ``out=x`` is in place."""
    L = _load()
    out = _empty_like_rows(x) if out is None else out
    o, xv, g, yv = _view(out), _view(x), _view(gate), _view(y)
    _raise(L.mbx_residual_gate_add(_ref(o), _ref(xv), _ref(g), _ref(yv), _variant(variant),
                                   _stream(x)))
    return out


def _fp8_like(x: torch.Tensor) -> torch.Tensor:
    dt = getattr(torch, "float8_e4m3fn", torch.uint8)
    return torch.empty(x.shape, dtype=dt, device=x.device)


def ln_modulate_fp8(x, scale, shift, fp8_scale, eps: float = 1e-6, variant="lossless", out=None,
                    out_fp8=None):
    """LN + AdaLN modulate writing the bf16 result and its static E4M3 copy
    e4m3(out / fp8_scale) in one pass (see mbx_ln_modulate_fp8).  fp8_scale is a
    one-element float32 CUDA tensor.  Returns (out, out_fp8)."""
    L = _load()
    out = _empty_like_rows(x) if out is None else out
    out_fp8 = _fp8_like(x) if out_fp8 is None else out_fp8
    o, q, xv, sc, sh = _view(out), _view(out_fp8), _view(x), _view(scale), _view(shift)
    _raise(L.mbx_ln_modulate_fp8(_ref(o), _ref(q), _ref(xv), _ref(sc), _ref(sh), _ptr(fp8_scale), eps,
                                 _variant(variant), _stream(x)))
    return out, out_fp8


def check_ln_modulate_fp8(out, out_fp8, x, scale, shift, fp8_scale, eps=1e-6, variant="lossless") -> int:
    return _load().mbx_check_ln_modulate_fp8(_ref(_view(out)), _ref(_view(out_fp8)), _ref(_view(x)),
                                             _ref(_view(scale)), _ref(_view(shift)), _ptr(fp8_scale), eps,
                                             _variant(variant))


def gated_residual_ln_modulate_fp8(residual, gate, update, scale, shift, fp8_scale, bias=None,
                                   eps: float = 1e-6, variant="lossless", out=None, residual_out=None,
                                   out_fp8=None):
    """Gated residual + LN + AdaLN modulate writing r', the bf16 result and its
    static E4M3 copy (see mbx_gated_residual_ln_modulate_fp8).  Returns
    (residual_out, out, out_fp8)."""
    L = _load()
    out = _empty_like_rows(residual) if out is None else out
    residual_out = _empty_like_rows(residual) if residual_out is None else residual_out
    out_fp8 = _fp8_like(residual) if out_fp8 is None else out_fp8
    ro, o, q = _view(residual_out), _view(out), _view(out_fp8)
    r, g, u, sc, sh = _view(residual), _view(gate), _view(update), _view(scale), _view(shift)
    b = None if bias is None else _view(bias)
    _raise(L.mbx_gated_residual_ln_modulate_fp8(_ref(ro), _ref(o), _ref(q), _ref(r), _ref(g), _ref(u),
                                                None if b is None else _ref(b), _ref(sc), _ref(sh),
                                                _ptr(fp8_scale), eps, _variant(variant), _stream(residual)))
    return residual_out, out, out_fp8


def check_gated_residual_ln_modulate_fp8(residual_out, out, out_fp8, residual, gate, update, scale, shift,
                                         fp8_scale, bias=None, eps=1e-6, variant="lossless") -> int:
    b = None if bias is None else _view(bias)
    return _load().mbx_check_gated_residual_ln_modulate_fp8(
        _ref(_view(residual_out)), _ref(_view(out)), _ref(_view(out_fp8)), _ref(_view(residual)),
        _ref(_view(gate)), _ref(_view(update)), None if b is None else _ref(b), _ref(_view(scale)),
        _ref(_view(shift)), _ptr(fp8_scale), eps, _variant(variant))


def nvfp4_sf_shape(rows: int, D: int) -> tuple[int, int]:
    """Shape of the NVFP4 block-scale buffer: rows padded to 128, blocks of 16
    padded to 4 (the 128x4 tile layout)."""
    return (rows + 127) // 128 * 128, (D // 16 + 3) // 4 * 4


def _fp4_views(x: torch.Tensor, out_fp4, out_sf):
    D = x.shape[-1]
    rows = x.numel() // D
    if out_fp4 is None:
        out_fp4 = torch.empty((rows, D // 2), dtype=torch.uint8, device=x.device)
    if out_sf is None:
        out_sf = torch.zeros(nvfp4_sf_shape(rows, D), dtype=torch.uint8, device=x.device)
    q, f = _view(out_fp4), _view(out_sf)
    q.dtype, f.dtype = MBX_E2M1X2, MBX_E4M3
    return out_fp4, out_sf, q, f


def ln_modulate_nvfp4(x, scale, shift, fp4_scale, eps: float = 1e-6, variant="lossless", out=None,
                      out_fp4=None, out_sf=None):
    """LN + AdaLN modulate writing the bf16 result and its NVFP4 copy (packed
    E2M1 [rows, D/2] uint8, E4M3 block scales in the 128x4 tile layout; see
    mbx_ln_modulate_nvfp4).  fp4_scale: one-element float32 CUDA tensor (the
    global scale).  Returns (out, out_fp4, out_sf)."""
    L = _load()
    out = _empty_like_rows(x) if out is None else out
    out_fp4, out_sf, q, f = _fp4_views(x, out_fp4, out_sf)
    o, xv, sc, sh = _view(out), _view(x), _view(scale), _view(shift)
    _raise(L.mbx_ln_modulate_nvfp4(_ref(o), _ref(q), _ref(f), _ref(xv), _ref(sc), _ref(sh), _ptr(fp4_scale), eps,
                                   _variant(variant), _stream(x)))
    return out, out_fp4, out_sf


def check_ln_modulate_nvfp4(out, out_fp4, out_sf, x, scale, shift, fp4_scale, eps=1e-6, variant="lossless") -> int:
    q, f = _view(out_fp4), _view(out_sf)
    q.dtype, f.dtype = MBX_E2M1X2, MBX_E4M3
    return _load().mbx_check_ln_modulate_nvfp4(_ref(_view(out)), _ref(q), _ref(f), _ref(_view(x)),
                                               _ref(_view(scale)), _ref(_view(shift)), _ptr(fp4_scale), eps,
                                               _variant(variant))


def gated_residual_ln_modulate_nvfp4(residual, gate, update, scale, shift, fp4_scale, bias=None,
                                     eps: float = 1e-6, variant="lossless", out=None, residual_out=None,
                                     out_fp4=None, out_sf=None):
    """Gated residual + LN + AdaLN modulate writing r', the bf16 result and its
    NVFP4 copy.  Returns (residual_out, out, out_fp4, out_sf)."""
    L = _load()
    out = _empty_like_rows(residual) if out is None else out
    residual_out = _empty_like_rows(residual) if residual_out is None else residual_out
    out_fp4, out_sf, q, f = _fp4_views(residual, out_fp4, out_sf)
    ro, o = _view(residual_out), _view(out)
    r, g, u, sc, sh = _view(residual), _view(gate), _view(update), _view(scale), _view(shift)
    b = None if bias is None else _view(bias)
    _raise(L.mbx_gated_residual_ln_modulate_nvfp4(_ref(ro), _ref(o), _ref(q), _ref(f), _ref(r), _ref(g), _ref(u),
                                                  None if b is None else _ref(b), _ref(sc), _ref(sh),
                                                  _ptr(fp4_scale), eps, _variant(variant), _stream(residual)))
    return residual_out, out, out_fp4, out_sf


def check_gated_residual_ln_modulate_nvfp4(residual_out, out, out_fp4, out_sf, residual, gate, update, scale,
                                           shift, fp4_scale, bias=None, eps=1e-6, variant="lossless") -> int:
    q, f = _view(out_fp4), _view(out_sf)
    q.dtype, f.dtype = MBX_E2M1X2, MBX_E4M3
    b = None if bias is None else _view(bias)
    return _load().mbx_check_gated_residual_ln_modulate_nvfp4(
        _ref(_view(residual_out)), _ref(_view(out)), _ref(q), _ref(f), _ref(_view(residual)), _ref(_view(gate)),
        _ref(_view(update)), None if b is None else _ref(b), _ref(_view(scale)), _ref(_view(shift)),
        _ptr(fp4_scale), eps, _variant(variant))


def modulation_table_add(table, temb, out=None):
    """Per-token modulation table in the (6, rows, D) layout (see
    mbx_modulation_table_add): the eager ``(table.unsqueeze(0) +
    temb.float()).chunk(6, dim=2)`` with the six chunks written as contiguous
    binary32 planes.  table [6, D] (any leading size-1 dims), temb [..., 6, D]
    or [..., 6*D]; bfloat16 or float32.  Returns out [6, *lead, D] float32
    (``out[k]`` is chunk k)."""
    L = _load()
    D = table.shape[-1]
    if temb.dim() >= 2 and temb.shape[-2] == 6 and temb.shape[-1] == D:
        lead = tuple(temb.shape[:-2])
        e = temb.reshape(*lead, 6 * D) if temb.is_contiguous() else temb.flatten(-2)
    else:
        lead = tuple(temb.shape[:-1])
        e = temb
    if out is None:
        out = torch.empty((6, *lead, D), dtype=torch.float32, device=temb.device)
    o, t, ev = _view(out), _view(table), _view(e)
    _raise(L.mbx_modulation_table_add(_ref(o), _ref(t), _ref(ev), _stream(temb)))
    return out


def check_modulation_table_add(out, table, temb) -> int:
    return _load().mbx_check_modulation_table_add(_ref(_view(out)), _ref(_view(table)), _ref(_view(temb)))


def gated_residual_ln_modulate(residual, gate, update, scale, shift, bias=None, eps: float = 1e-6,
                               variant="lossless", out=None, residual_out=None):
    """Gated residual update fused into LN + AdaLN modulate (see
    mbx_gated_residual_ln_modulate).  Returns (residual_out, out);
    ``residual_out=residual`` updates the residual stream in place."""
    L = _load()
    out = _empty_like_rows(residual) if out is None else out
    residual_out = _empty_like_rows(residual) if residual_out is None else residual_out
    ro, o, r, g, u = _view(residual_out), _view(out), _view(residual), _view(gate), _view(update)
    sc, sh = _view(scale), _view(shift)
    b = None if bias is None else _view(bias)
    _raise(L.mbx_gated_residual_ln_modulate(_ref(ro), _ref(o), _ref(r), _ref(g), _ref(u),
                                            None if b is None else _ref(b), _ref(sc), _ref(sh), eps,
                                            _variant(variant), _stream(residual)))
    return residual_out, out


def check_gated_residual_ln_modulate(residual_out, out, residual, gate, update, scale, shift,
                                     bias=None, eps=1e-6, variant="lossless") -> int:
    ro, o, r, g, u = _view(residual_out), _view(out), _view(residual), _view(gate), _view(update)
    sc, sh = _view(scale), _view(shift)
    b = None if bias is None else _view(bias)
    return _load().mbx_check_gated_residual_ln_modulate(
        _ref(ro), _ref(o), _ref(r), _ref(g), _ref(u), None if b is None else _ref(b), _ref(sc),
        _ref(sh), eps, _variant(variant))


def _ptr(t):
    return None if t is None or t.numel() == 0 else t.data_ptr()


def _branch_view(t, width):
    if t is None:
        return _View(None, 0, width, width, MBX_BF16)
    return _view(t)


def qk_norm_rope_qkv_epilogue(txt_qkv, img_qkv, batch: int, heads: int, head_dim: int,
                              wq_txt, wk_txt, wq_img, wk_img, cos_txt, sin_txt, cos_img,
                              sin_img, eps: float = 1e-6, variant="lossless", out=None):
    """Fused post-GEMM QKV epilogue (see mbx_qk_norm_rope_qkv_epilogue).

    txt_qkv [B*S_txt, 3*H*hd] and img_qkv [B*S_img, 3*H*hd] (row views, may be
    padded; either may be None); cos/sin tables binary32 [S, hd/2].  Returns
    the joint buffer [B, 3, H, S_txt + S_img, hd].
    """
    L = _load()
    width = 3 * heads * head_dim
    ref = txt_qkv if txt_qkv is not None else img_qkv
    s_txt = 0 if txt_qkv is None else _rows_cols(txt_qkv)[0] // batch
    s_img = 0 if img_qkv is None else _rows_cols(img_qkv)[0] // batch
    if out is None:
        out = torch.empty((batch, 3, heads, s_txt + s_img, head_dim), dtype=torch.bfloat16,
                          device=ref.device)
    j = _view(out.reshape(-1, head_dim) if out.is_contiguous() else out)
    t, im = _branch_view(txt_qkv, width), _branch_view(img_qkv, width)
    ws = [_view(w) for w in (wq_txt, wk_txt, wq_img, wk_img)]
    _raise(L.mbx_qk_norm_rope_qkv_epilogue(
        _ref(j), _ref(t), _ref(im), batch, heads, *[_ref(w) for w in ws],
        _ptr(cos_txt), _ptr(sin_txt), _ptr(cos_img), _ptr(sin_img), eps, _variant(variant),
        _stream(ref)))
    return out


# ---------------------------------------------------------------- validation only


def check_ln_modulate(out, x, scale, shift, eps=1e-6, variant="lossless") -> int:
    o, xv, sc, sh = _view(out), _view(x), _view(scale), _view(shift)
    return _load().mbx_check_ln_modulate(_ref(o), _ref(xv), _ref(sc), _ref(sh), eps,
                                         _variant(variant))


def check_rmsnorm_scale(out, x, weight, scale, eps=1e-6, variant="lossless") -> int:
    o, xv, w, sc = _view(out), _view(x), _view(weight), _view(scale)
    return _load().mbx_check_rmsnorm_scale(_ref(o), _ref(xv), _ref(w), _ref(sc), eps,
                                           _variant(variant))


def check_rmsnorm_tanh_residual(out, x, gate, residual, weight, eps=1e-6,
                                variant="lossless") -> int:
    o, xv, g, r, w = _view(out), _view(x), _view(gate), _view(residual), _view(weight)
    return _load().mbx_check_rmsnorm_tanh_residual(_ref(o), _ref(xv), _ref(g), _ref(r), _ref(w),
                                                   eps, _variant(variant))


def check_residual_gate_add(out, x, gate, y, variant="lossless") -> int:
    o, xv, g, yv = _view(out), _view(x), _view(gate), _view(y)
    return _load().mbx_check_residual_gate_add(_ref(o), _ref(xv), _ref(g), _ref(yv),
                                               _variant(variant))


def check_qk_norm_rope_qkv_epilogue(out, txt_qkv, img_qkv, batch, heads, head_dim, wq_txt,
                                    wk_txt, wq_img, wk_img, cos_txt, sin_txt, cos_img,
                                    sin_img, eps=1e-6, variant="lossless") -> int:
    width = 3 * heads * head_dim
    j = _view(out.reshape(-1, head_dim) if out.is_contiguous() else out)
    t, im = _branch_view(txt_qkv, width), _branch_view(img_qkv, width)
    ws = [_view(w) for w in (wq_txt, wk_txt, wq_img, wk_img)]
    return _load().mbx_check_qk_norm_rope_qkv_epilogue(
        _ref(j), _ref(t), _ref(im), batch, heads, *[_ref(w) for w in ws], _ptr(cos_txt),
        _ptr(sin_txt), _ptr(cos_img), _ptr(sin_img), eps, _variant(variant))


def selftest(which: int, device=None) -> tuple[int, int]:
    """Run exhaustive self-test `which` (see mbx_selftest) on the current CUDA
    device; returns (mismatches, NaN-only mismatches)."""
    counts = torch.zeros(2, dtype=torch.int64, device=device or "cuda")
    _raise(_load().mbx_selftest(which, counts.data_ptr(), _stream(counts)))
    torch.cuda.synchronize(counts.device)
    c = counts.cpu().tolist()
    return int(c[0]), int(c[1])
