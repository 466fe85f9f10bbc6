"""Parity of the per-token modulation table (the (6, rows, D) layout of the
eager ``(table.unsqueeze(0) + temb.float()).chunk(6, dim=2)``) with the oracle:
every binary32 output bit equal.  Shapes: a Wan2.2-TI2V-like token count at
D = 3072 (sampled rows), both dtypes of each input, padded rows, ragged D and
misaligned views (the scalar path), a single token.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def mbx():
    import modulation_bit_exact_gb300 as m
    m.lib()
    return m


def _host(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _case(rows, D, tab_dt, emb_dt, seed=0, device="cpu"):
    g = torch.Generator(device=device).manual_seed(seed * 1009 + rows * 7 + D)
    table = (torch.randn(6, D, generator=g, device=device) / D ** 0.5).to(tab_dt)
    temb = torch.randn(rows, 6, D, generator=g, device=device).to(emb_dt)
    return table, temb


def _check(got, table, temb, rows_sel=None):
    T = _host(table)
    E = _host(temb.reshape(temb.shape[0], -1))
    if rows_sel is not None:
        E = E[rows_sel]
    want = oracle.modulation_table_add(T, E)
    g = got.detach().cpu().reshape(6, -1, table.shape[-1])
    if rows_sel is not None:
        g = g[:, torch.from_numpy(rows_sel)]
    g = g.contiguous().numpy()
    bad = g.view(np.uint32) != want.view(np.uint32)
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} differ; first at {tuple(np.argwhere(bad)[0])}"


@pytest.mark.parametrize("tab_dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("emb_dt", [torch.bfloat16, torch.float32])
def test_small_all_dtypes(mbx, tab_dt, emb_dt):
    table, temb = _case(333, 1024, tab_dt, emb_dt)
    out = mbx.modulation_table_add(table.to(DEV), temb.to(DEV))
    assert out.shape == (6, 333, 1024) and out.dtype == torch.float32
    _check(out, table, temb)


def test_wan_ti2v_shape_sampled(mbx):
    """B = 1, S = 31 x 44 x 80 = 109 120 latent tokens (704p, 121 frames),
    D = 3072: 4 GB of bf16 temb in, 8 GB of binary32 out."""
    rows, D = 31 * 44 * 80, 3072
    table, temb = _case(rows, D, torch.float32, torch.bfloat16, device=DEV)
    out = mbx.modulation_table_add(table, temb.view(1, rows, 6, D))
    assert out.shape == (6, 1, rows, D)
    rng = np.random.default_rng(3)
    sel = np.unique(np.r_[0, 1, rows // 2, rows - 1, rng.integers(0, rows, 200)])
    idx = torch.from_numpy(sel).to(DEV)
    got = out.view(6, rows, D).index_select(1, idx)
    _check(got, table, temb.index_select(0, idx))


def test_padded_rows_and_out_view(mbx):
    rows, D = 200, 512
    table, temb = _case(rows, D, torch.bfloat16, torch.bfloat16, seed=1)
    tbuf = torch.full((rows, 6 * D + 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    tbuf[:, :6 * D] = temb.reshape(rows, -1).to(DEV)
    obuf = torch.full((6 * rows, D + 32), 7.0, dtype=torch.float32, device=DEV)
    out = obuf[:, :D]
    mbx.modulation_table_add(table.to(DEV), tbuf[:, :6 * D], out=out)
    _check(out, table, temb)
    assert torch.all(obuf[:, D:] == 7.0)  # the pad is never written


@pytest.mark.parametrize("D", [1, 7, 100, 1000])
def test_ragged_d(mbx, D):
    table, temb = _case(41, D, torch.bfloat16, torch.float32, seed=2)
    _check(mbx.modulation_table_add(table.to(DEV), temb.to(DEV)), table, temb)


def test_misaligned_views(mbx):
    rows, D = 64, 256
    table, temb = _case(rows, D, torch.bfloat16, torch.bfloat16, seed=3)
    buf = torch.empty(rows * 6 * D + 8, dtype=torch.bfloat16, device=DEV)
    e = buf[1:1 + rows * 6 * D].view(rows, 6 * D)
    e.copy_(temb.reshape(rows, -1).to(DEV))
    _check(mbx.modulation_table_add(table.to(DEV), e), table, temb)


def test_single_token_and_non_finite(mbx):
    table, temb = _case(1, 64, torch.float32, torch.float32, seed=4)
    temb[0, 0, :3] = torch.tensor([float("inf"), -float("inf"), 3e38])
    table[0, 2] = 3e38
    out = mbx.modulation_table_add(table.to(DEV), temb.to(DEV)).cpu()
    assert out[0, 0, 0] == float("inf") and out[0, 0, 1] == -float("inf")
    assert out[0, 0, 2] == float("inf")  # 3e38 + 3e38 overflows
    _check(out, table, temb)
