"""Seeded synthetic inputs for the DiT norm/modulation path.

This module is shared by the tests and the benchmark and by both sides of every
parity check (the CUDA path and the CPU oracle).  It only draws random inputs
with fixed seeds and shapes; it holds none of the method's arithmetic.

The RoPE cos/sin tables are inputs of the fused QKV epilogue (a model builds
them once per resolution and passes them to the kernel); they are built here
in binary64 from the standard rotary rule, angle = p * theta^(-2i/d), and
rounded once to binary32.

Recipes (shapes are the DiT-shaped workloads the pages discuss: Qwen-Image-like
hidden 3072 = 24 heads x 128 with 4096 image + 256 text tokens, and Wan-like
hidden 5120 with 21 x 30 x 52 = 32760 video tokens):

* all tensors are drawn in binary32 from one ``torch.Generator`` seeded per
  configuration, in declaration order, then rounded to bfloat16 by torch;
* activations ~ N(0, 1); modulation (scale/shift/gate) ~ N(0, 0.1);
  norm weights = 1 + N(0, 0.05);
* the image-DiT configuration multiplies 1 % of the activations (Bernoulli
  per element) by 20 (outliers);
* the sweep pads every input row by 64 elements (row stride D + 64), fills the
  pad with NaN sentinels that must never reach an output, makes 0.1 % of the
  rows constant (Bernoulli per row, value ~ N(0, 1)) and one row all-zero.
"""
from __future__ import annotations

import math

import torch

BF16 = torch.bfloat16

SWEEP_D = (1024, 2048, 3072, 4096, 5120, 6144, 8192)
SWEEP_T = (1, 77, 4096, 65536)
PAD = 64


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(g, shape, std=1.0, mean=0.0, device="cpu"):
    t = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(BF16)


def tiny_ln_modulate(seed: int = 0, device="cpu") -> dict:
    """x [2,256,512] ~N(0,1); per-sample scale/shift [2,512] ~N(0,0.1);
    rmsnorm weight [512] = 1+N(0,0.05); the rmsnorm_scale case reuses x and scale."""
    g = _gen(seed, device)
    x = _normal(g, (2, 256, 512), device=device)
    scale = _normal(g, (2, 512), 0.1, device=device)
    shift = _normal(g, (2, 512), 0.1, device=device)
    weight = _normal(g, (512,), 0.05, 1.0, device=device)
    return dict(x=x, scale=scale, shift=shift, weight=weight, eps=1e-6)


def image_dit_block(seed: int = 2, device="cpu", batch: int = 2, seq: int = 4352,
                    hidden: int = 3072) -> dict:
    """x [2,4352,3072] ~N(0,1) with 1 % outliers x20; per-sample scale/shift/gate
    [2,3072] ~N(0,0.1); y [2,4352,3072] ~N(0,1)."""
    g = _gen(seed, device)
    x = torch.randn((batch, seq, hidden), generator=g, dtype=torch.float32, device=device)
    mask = torch.rand((batch, seq, hidden), generator=g, device=device) < 0.01
    x = torch.where(mask, x * 20.0, x).to(BF16)
    scale = _normal(g, (batch, hidden), 0.1, device=device)
    shift = _normal(g, (batch, hidden), 0.1, device=device)
    gate = _normal(g, (batch, hidden), 0.1, device=device)
    y = _normal(g, (batch, seq, hidden), device=device)
    return dict(x=x, scale=scale, shift=shift, gate=gate, y=y, eps=1e-6)


def rope_1d(positions: torch.Tensor, dim: int, theta: float = 10000.0):
    """cos/sin [len(positions), dim/2] (binary32) for pairs i = 0..dim/2-1."""
    i = torch.arange(dim // 2, dtype=torch.float64)
    inv = torch.pow(torch.tensor(theta, dtype=torch.float64), -2.0 * i / dim)
    ang = positions.to(torch.float64)[:, None] * inv[None, :]
    return torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)


def rope_text(s_txt: int, head_dim: int, theta: float = 10000.0):
    """Text tokens: 1-D positions 0..S-1 over the whole head."""
    return rope_1d(torch.arange(s_txt), head_dim, theta)


def rope_image(grid_h: int, grid_w: int, head_dim: int, theta: float = 10000.0):
    """Image tokens on an h x w grid (row-major): pairs of the first half of the
    head rotate by the row index, pairs of the second half by the column."""
    j = torch.arange(grid_h * grid_w)
    ch, sh = rope_1d(j // grid_w, head_dim // 2, theta)
    cw, sw = rope_1d(j % grid_w, head_dim // 2, theta)
    return torch.cat([ch, cw], dim=1).contiguous(), torch.cat([sh, sw], dim=1).contiguous()


def qkv_epilogue_case(seed: int = 3, device="cpu", batch: int = 2, s_txt: int = 256,
                      grid_h: int = 64, grid_w: int = 64, heads: int = 24,
                      head_dim: int = 128, row_pad: int = 0) -> dict:
    """GEMM outputs txt [B, S_txt, 3*H*hd] and img [B, h*w, 3*H*hd] ~N(0,1) read
    through (optionally padded) row views; four norm weights [hd] = 1+N(0,0.05);
    per-token RoPE tables, theta = 10000."""
    g = _gen(seed, device)
    width = 3 * heads * head_dim
    s_img = grid_h * grid_w

    def act(S):
        buf = torch.full((batch * S, width + row_pad), float("nan"), dtype=BF16, device=device)
        buf[:, :width] = _normal(g, (batch * S, width), device=device)
        return buf[:, :width]

    txt = act(s_txt)
    img = act(s_img)
    ws = [_normal(g, (head_dim,), 0.05, 1.0, device=device) for _ in range(4)]
    cos_t, sin_t = rope_text(s_txt, head_dim)
    cos_i, sin_i = rope_image(grid_h, grid_w, head_dim)
    return dict(txt=txt, img=img, batch=batch, heads=heads, head_dim=head_dim,
                wq_txt=ws[0], wk_txt=ws[1], wq_img=ws[2], wk_img=ws[3],
                cos_txt=cos_t.to(device), sin_txt=sin_t.to(device),
                cos_img=cos_i.to(device), sin_img=sin_i.to(device), eps=1e-6)


def video_dit_block(seed: int = 4, device="cpu", seq: int = 32760, hidden: int = 5120) -> dict:
    """x [1,32760,5120] ~N(0,1); per-token scale/shift ~N(0,0.1); g, r ~N(0,1);
    rmsnorm weight [5120] = 1+N(0,0.05)."""
    g = _gen(seed, device)
    x = _normal(g, (1, seq, hidden), device=device)
    scale = _normal(g, (1, seq, hidden), 0.1, device=device)
    shift = _normal(g, (1, seq, hidden), 0.1, device=device)
    gate = _normal(g, (1, seq, hidden), device=device)
    residual = _normal(g, (1, seq, hidden), device=device)
    weight = _normal(g, (hidden,), 0.05, 1.0, device=device)
    return dict(x=x, scale=scale, shift=shift, gate=gate, residual=residual, weight=weight,
                eps=1e-6)


def padded(t: torch.Tensor, pad: int = PAD) -> torch.Tensor:
    """The same values as the 2-D tensor t, viewed from a buffer whose rows are
    `pad` elements longer; the pad holds NaN sentinels."""
    rows, D = t.shape
    buf = torch.full((rows, D + pad), float("nan"), dtype=t.dtype, device=t.device)
    buf[:, :D] = t
    return buf[:, :D]


def sweep_case(D: int, T: int, seed: int = 5, device="cpu", mod_rows: int = 1) -> dict:
    """One cell of the shape/stride sweep: x [T, D] ~N(0,1) with 0.1 % constant
    rows and one zero row, gate/residual/y [T, D] ~N(0,1), per-sample
    scale/shift/gate [mod_rows, D] ~N(0,0.1), weight [D]; every [T, D] input is
    a padded-row view (stride D + 64, NaN in the pad)."""
    g = _gen(seed * 1_000_003 + D * 131 + T, device)
    x = torch.randn((T, D), generator=g, dtype=torch.float32, device=device)
    const_rows = torch.rand((T,), generator=g, device=device) < 0.001
    const_val = torch.randn((T,), generator=g, dtype=torch.float32, device=device)
    x = torch.where(const_rows[:, None], const_val[:, None].expand(T, D), x)
    if T > 1:
        x[T // 2].zero_()
    x = x.to(BF16)
    other = _normal(g, (T, D), device=device)
    residual = _normal(g, (T, D), device=device)
    scale = _normal(g, (mod_rows, D), 0.1, device=device)
    shift = _normal(g, (mod_rows, D), 0.1, device=device)
    gate = _normal(g, (mod_rows, D), 0.1, device=device)
    weight = _normal(g, (D,), 0.05, 1.0, device=device)
    return dict(x=padded(x), y=padded(other), gate_tok=padded(other), residual=padded(residual),
                scale=padded(scale), shift=padded(shift), gate=padded(gate), weight=weight,
                eps=1e-6)


def grid_for(tokens: int) -> tuple[int, int]:
    """A square-ish image grid with exactly `tokens` cells (h <= w)."""
    h = int(math.isqrt(tokens))
    while tokens % h:
        h -= 1
    return h, tokens // h
