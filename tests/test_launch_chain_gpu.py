"""Back-to-back dependent calls on one stream, with no synchronisation between
them.

Every kernel is launched with programmatic stream serialisation: it may start
while the previous kernel drains, and it must not read that kernel's output
before its grid-dependency wait returns.  Here each call consumes the output of
the call before it (two of them in place), at the image-DiT size, so a read
ahead of the wait would show as a mismatch.  Every intermediate result is
compared bit for bit with the same chain run by the oracle from the host inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import assert_bits_equal, u16

pytestmark = pytest.mark.gpu

DEV = "cuda"
BF16 = torch.bfloat16


@pytest.fixture(scope="module")
def mbx():
    import modulation_bit_exact_gb300 as m
    m.lib()
    return m


def _rand(g, shape, std=1.0, mean=0.0):
    return (torch.randn(shape, generator=g) * std + mean).to(BF16)


@pytest.mark.parametrize("B,S,D", [(2, 4352, 3072), (3, 700, 1024)])
def test_dependent_chain(mbx, B, S, D):
    g = torch.Generator().manual_seed(B * 1000 + D)
    rows = B * S
    host = dict(x=_rand(g, (rows, D)), y=_rand(g, (rows, D)), sc=_rand(g, (B, D), 0.1),
                sh=_rand(g, (B, D), 0.1), gt=_rand(g, (B, D), 0.1), sc2=_rand(g, (B, D), 0.1, 1.0),
                gt2=_rand(g, (B, D), 0.5), w=_rand(g, (D,), 0.05, 1.0), bias=_rand(g, (1, D), 0.5))
    d = {k: v.to(DEV) for k, v in host.items()}
    torch.cuda.synchronize()

    # the chain, launched back to back on the current stream
    a = mbx.ln_modulate(d["x"], d["sc"], d["sh"])
    b = mbx.residual_gate_add(a, d["gt"], d["y"])
    c = mbx.rmsnorm_scale(b, d["w"], d["sc2"])
    e = mbx.rmsnorm_tanh_residual(c, d["gt2"], b, d["w"])
    r, f = mbx.gated_residual_ln_modulate(e, d["gt"], c, d["sc"], d["sh"], bias=d["bias"])
    mbx.residual_gate_add(f, d["gt"], a, out=f)  # in place over the previous output
    h = mbx.ln_modulate(f, d["sc"], d["sh"])
    mbx.residual_gate_add(r, d["gt2"], h, out=r)  # in place over the fused op's residual
    # (the fused op's r' and output are overwritten in place; their checks go
    # through the two in-place steps that consume them)
    got = {k: u16(v) for k, v in (("ln", a), ("rga", b), ("rms", c), ("tanh", e), ("rga in place", f),
                                  ("ln of in-place", h), ("rga in place 2", r))}

    X, Y, SC, SH, GT = (u16(host[k]) for k in ("x", "y", "sc", "sh", "gt"))
    SC2, GT2, W, BI = (u16(host[k]) for k in ("sc2", "gt2", "w", "bias"))
    # the same chain run by the oracle alone, from the host inputs
    A = oracle.ln_modulate(X, SC, SH, 1e-6)
    Bv = oracle.residual_gate_add(A, GT, Y)
    C = oracle.rmsnorm_scale(Bv, W, SC2, 1e-6)
    E = oracle.rmsnorm_tanh_residual(C, GT2, Bv, W, 1e-6)
    R, F = oracle.gated_residual_ln_modulate(E, GT, C, BI, SC, SH, 1e-6)
    F2 = oracle.residual_gate_add(F, GT, A)
    H = oracle.ln_modulate(F2, SC, SH, 1e-6)
    R2 = oracle.residual_gate_add(R, GT2, H)
    for name, want in (("ln", A), ("rga", Bv), ("rms", C), ("tanh", E), ("rga in place", F2),
                       ("ln of in-place", H), ("rga in place 2", R2)):
        assert_bits_equal(got[name], want, name)


def test_cross_stream_event_order(mbx):
    """A call on a second stream, ordered after the first stream's call by an
    event, reads the finished output (the launch attribute relaxes only the
    order between neighbours in one stream)."""
    g = torch.Generator().manual_seed(5)
    B, S, D = 2, 4352, 3072
    x, y = _rand(g, (B * S, D)), _rand(g, (B * S, D))
    sc, sh, gt = _rand(g, (B, D), 0.1), _rand(g, (B, D), 0.1), _rand(g, (B, D), 0.1)
    d = [t.to(DEV) for t in (x, y, sc, sh, gt)]
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()
    with torch.cuda.stream(s1):
        a = mbx.ln_modulate(d[0], d[2], d[3])
        ev.record(s1)
    with torch.cuda.stream(s2):
        s2.wait_event(ev)
        b = mbx.residual_gate_add(a, d[4], d[1])
    torch.cuda.synchronize()
    A = oracle.ln_modulate(u16(x), u16(sc), u16(sh), 1e-6)
    assert_bits_equal(u16(a), A, "ln on stream 1")
    assert_bits_equal(u16(b), oracle.residual_gate_add(A, u16(gt), u16(y)), "rga on stream 2")
