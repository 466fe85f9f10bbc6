"""Pins of the CPU oracle against things other than itself.

Witnesses used: PyTorch CPU eager bfloat16/float32 ops (a library), mpmath at
50 digits, binary64 brute force, closed forms and invariants.  Nothing here
touches a GPU or the CUDA library.  Each pin is chosen so that a plausible
mistake in the oracle (a dropped term, a wrong sign or index, a missed or
extra rounding point) fails it.
"""
import math

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |v| (2^(e-7)), floored at the subnormal step."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.maximum(np.exp2(e - 7), 2.0 ** -133)


# ---------------------------------------------------------------- rounding


def _torch_bf16_bits(f32_bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(f32_bits.view(np.float32).copy())
    return u16(t.to(torch.bfloat16))


def _check_rounding(orc, bits):
    bits = np.ascontiguousarray(bits, dtype=np.uint32)
    got = orc.f32_to_bf16(bits.view(np.float32))
    ref = _torch_bf16_bits(bits)
    nan = (bits & 0x7FFFFFFF) > 0x7F800000
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(got[nan] == 0x7FFF)
    assert np.all((ref[nan] & 0x7FFF) > 0x7F80)  # torch also gives a NaN


def test_bf16_rounding_every_high_half(orc):
    """All 65536 kept halves x the discarded halves that decide nearest-even."""
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xBFFF, 0xFFFF], np.uint32)
    hi = np.arange(65536, dtype=np.uint32)
    _check_rounding(orc, ((hi[:, None] << 16) | lows[None, :]).reshape(-1))


def test_bf16_rounding_every_low_half(orc):
    """All 65536 discarded halves under kept halves of both parities, both signs,
    the subnormal range, the largest finite value and infinity."""
    his = np.array([0x0000, 0x0001, 0x007F, 0x0080, 0x3F80, 0x3F81, 0x4049, 0x7F7E, 0x7F7F,
                    0x7F80, 0x8000, 0x8001, 0xBF80, 0xBF81, 0xFF7F, 0xFF80], np.uint32)
    lo = np.arange(65536, dtype=np.uint32)
    _check_rounding(orc, ((his[:, None] << 16) | lo[None, :]).reshape(-1))


def test_bf16_rounding_random(orc):
    rng = np.random.default_rng(1)
    _check_rounding(orc, rng.integers(0, 2**32, size=1 << 22, dtype=np.uint64).astype(np.uint32))


def test_no_fused_multiply_add(orc):
    """(1+2^-12)^2 - (1+2^-11) is 2^-24 exactly; two roundings give 0."""
    a = 1.0 + 2.0 ** -12
    assert orc.probe_mul_add(a, a, -(1.0 + 2.0 ** -11)) == 0.0


# ---------------------------------------------------------------- tanh


def _nearest_bf16_mp(x_bits: int, mp) -> int:
    """The bfloat16 nearest to tanh(x) for a finite bfloat16 x, ties to even,
    searched among the neighbours of a binary64 estimate, compared at 50 digits."""
    x = float(np.array([x_bits << 16], np.uint32).view(np.float32)[0])
    t = mp.tanh(mp.mpf(x))
    est = np.array([float(t)], np.float32).view(np.uint32)[0] >> 16
    cands = set()
    for d in (-2, -1, 0, 1, 2):
        c = (int(est) + d) & 0xFFFF
        if (c & 0x7FFF) <= 0x7F80:
            cands.add(c)
    # also try the sign-flipped encodings near zero
    if abs(x) < 1e-30:
        cands.update({0x0000, 0x8000})
    best = None
    for c in sorted(cands):
        v = float(np.array([c << 16], np.uint32).view(np.float32)[0])
        err = abs(mp.mpf(v) - t)
        key = (err, c & 1)  # on a tie, the even encoding wins
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_tanh_table_exhaustive_against_mpmath(orc):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    table = orc.tanh_table()
    bad = []
    for g in range(65536):
        a = g & 0x7FFF
        if a > 0x7F80:
            if table[g] != 0x7FFF:
                bad.append(g)
            continue
        if a == 0x7F80:
            want = (g & 0x8000) | 0x3F80
        elif a == 0:
            want = g  # tanh(+-0) = +-0
        else:
            want = _nearest_bf16_mp(g, mp)
        if table[g] != want:
            bad.append(g)
    assert not bad, [hex(b) for b in bad[:10]]


def test_tanh_table_odd_and_saturating(orc):
    t = orc.tanh_table()
    g = np.arange(0x7F80)
    assert np.array_equal(t[g | 0x8000], t[g] | 0x8000)
    assert t[0x4080] == 0x3F80  # tanh(4) rounds to 1
    assert t[0x0000] == 0x0000 and t[0x8000] == 0x8000


# ---------------------------------------------------------------- Welford-128


def _welford_textbook(xs: np.ndarray):
    """Welford (1962) running mean and M2 in binary32, one element at a time
    (Knuth, TAOCP vol. 2, 4.2.2) -- the special case of a single active lane."""
    f = np.float32
    n = f(0); mean = f(0); m2 = f(0)
    for v in xs.astype(np.float32):
        n = f(n + f(1))
        d = f(v - mean)
        mean = f(mean + f(d / n))
        m2 = f(m2 + f(d * f(v - mean)))
    return mean, m2, n


def _chan(a, b):
    """Chan, Golub & LeVeque pairwise update, with r = nB/n (binary32)."""
    f = np.float32
    (ma, qa, na), (mb, qb, nb) = a, b
    n = f(na + nb)
    d = f(mb - ma)
    r = f(nb / n)
    return f(ma + f(d * r)), f(f(qa + qb) + f(f(d * d) * f(na * r))), n


@pytest.mark.parametrize("D", [1, 2, 3, 5, 7, 8])
def test_welford_single_lane_is_textbook(orc, D):
    rng = np.random.default_rng(D)
    for _ in range(50):
        x = orc.f32_to_bf16(rng.standard_normal(D).astype(np.float32) * 3 + 1)
        got = orc.welford128(x)
        want = _welford_textbook(orc.bf16_to_f32(x))
        assert got == tuple(float(v) for v in want)


def test_welford_two_lanes_is_one_chan_combine(orc):
    rng = np.random.default_rng(7)
    for D in (9, 12, 16):
        for _ in range(50):
            x = orc.f32_to_bf16(rng.standard_normal(D).astype(np.float32))
            xf = orc.bf16_to_f32(x)
            want = _chan(_welford_textbook(xf[:8]), _welford_textbook(xf[8:]))
            assert orc.welford128(x) == tuple(float(v) for v in want)


# The lane ownership and the halving tree beyond two lanes.  The fixed order
# (chunk c = e // 8 on lane c mod 128, lanes visiting their chunks in ascending
# order; then for s = 64, 32, ..., 1 every lane l < s takes combine(L[l],
# L[l+s])) is the 128-thread Welford with a fixed shuffle tree that the tahou.com
# SGLang diffusion article (section 扩散Kernel对数值精度的敏感性) names without
# spelling out.  Each expected value below is that tree unrolled by hand for the
# case at hand and evaluated with the textbook helpers above; the docstrings give
# the unrolling.  Each test also shows that the plausible wrong orders (adjacent
# pairing, swapped operands, another chunk-to-lane map) give other bits on the
# same rows, so a mistake of that kind in the oracle cannot pass.


def _Z(n):
    """Welford state of n zero elements: mean 0, M2 0 (every step is exact)."""
    f = np.float32
    return f(0), f(0), f(n)


def _W(xf):
    return _welford_textbook(np.asarray(xf, np.float32))


def _stats(t):
    return tuple(float(v) for v in t)


def _rows_lanes(rng, D, rows=60):
    """Random bf16 rows of length D (binary32 values and bit patterns)."""
    out = []
    for _ in range(rows):
        xf = (rng.standard_normal(D) * rng.choice([0.5, 3.0, 40.0]) + rng.choice([0.0, 2.0, -7.0]))
        out.append(xf.astype(np.float32))
    return out


def test_welford_three_to_eight_lanes_follow_the_halving_tree(orc):
    """Unrolled by hand (lanes with no element are skipped, being empty):
      3 lanes (D 24, and ragged D 21):  s = 2: L0 = C(L0, L2);  s = 1: C(L0, L1)
                                        -> C(C(W0, W2), W1)
      4 lanes (D 32):  C(C(W0, W2), C(W1, W3))
      5 lanes (D 40):  s = 4: L0 = C(W0, W4); s = 2: L0 = C(L0, W2), L1 = C(W1, W3)
                       -> C(C(C(W0, W4), W2), C(W1, W3))
      8 lanes (D 64):  C(C(C(W0, W4), C(W2, W6)), C(C(W1, W5), C(W3, W7)))
    with W_l the textbook Welford of lane l's chunk (elements 8l .. 8l+7) and C
    the Chan combine, its first operand the lower lane."""
    C = _chan
    rng = np.random.default_rng(31)
    cases = {
        21: lambda W: C(C(W[0], W[2]), W[1]),
        24: lambda W: C(C(W[0], W[2]), W[1]),
        32: lambda W: C(C(W[0], W[2]), C(W[1], W[3])),
        40: lambda W: C(C(C(W[0], W[4]), W[2]), C(W[1], W[3])),
        64: lambda W: C(C(C(W[0], W[4]), C(W[2], W[6])), C(C(W[1], W[5]), C(W[3], W[7]))),
    }
    # the same lanes combined in other orders: adjacent pairs first, or the
    # higher lane as the first operand
    wrong = {
        21: [lambda W: C(C(W[0], W[1]), W[2]), lambda W: C(W[1], C(W[2], W[0]))],
        24: [lambda W: C(C(W[0], W[1]), W[2]), lambda W: C(W[1], C(W[2], W[0]))],
        32: [lambda W: C(C(W[0], W[1]), C(W[2], W[3])), lambda W: C(C(W[1], W[3]), C(W[0], W[2]))],
        40: [lambda W: C(C(C(W[0], W[1]), C(W[2], W[3])), W[4]),
             lambda W: C(C(W[0], W[2]), C(C(W[1], W[3]), W[4]))],
        64: [lambda W: C(C(C(W[0], W[1]), C(W[2], W[3])), C(C(W[4], W[5]), C(W[6], W[7]))),
             lambda W: C(C(C(W[4], W[0]), C(W[6], W[2])), C(C(W[5], W[1]), C(W[7], W[3])))],
    }
    for D, tree in cases.items():
        differs = [0] * len(wrong[D])
        for xf in _rows_lanes(rng, D):
            x = orc.f32_to_bf16(xf)
            xb = orc.bf16_to_f32(x)
            W = [_W(xb[8 * l:8 * l + 8]) for l in range((D + 7) // 8)]
            got = orc.welford128(x)
            assert got == _stats(tree(W)), D
            for i, w in enumerate(wrong[D]):
                differs[i] += got != _stats(w(W))
        assert all(differs), (D, differs)


def test_welford_128_lanes_sparse_rows(orc):
    """Full rows with a few non-zero lanes, every other lane all zeros (state
    Z_n = (0, 0, n), and C(Z_n, Z_n) = Z_2n exactly), unrolled by hand:

    D = 1024, non-zero lanes 0, 1, 64, 96 (one chunk each, n = 8):
      s = 64: L0 = C(W0, W64), L1 = C(W1, Z8), L32 = C(Z8, W96), others Z16
      s = 32: L0 = C(L0, L32), L1 = C(L1, Z16), others Z32
      s = 16 .. 2: L0 = C(L0, Z_k), L1 = C(L1, Z_k) for k = 32, 64, 128, 256
      s = 1: C(L0, L1)
    D = 2048 (lane l owns chunks l and l+128, n = 16), non-zero chunks 0 and 128
    (both lane 0), 192 (lane 64) and 1 (lane 1):
      s = 64: L0 = C(W0, W64), L1 = C(W1, Z16), others Z32
      s = 32 .. 2: L0 = C(L0, Z_k), L1 = C(L1, Z_k) for k = 32 .. 512;  s = 1: C(L0, L1)
    D = 1030 (lane 0 owns chunk 0 and the 6-element chunk 128), non-zero chunks
    0, 128 and 64:
      s = 64: L0 = C(W0, W64) (n 14 + 8), others Z16
      s = 32 .. 1: L0 = C(L0, Z_k) for k = 16, 32, 64, 128, 256, 512."""
    C = _chan
    rng = np.random.default_rng(32)

    def chain(s, ks):
        for k in ks:
            s = C(s, _Z(k))
        return s

    def row(D, chunks):
        xf = np.zeros(D, np.float32)
        for c in chunks:
            n = min(8, D - 8 * c)
            xf[8 * c:8 * c + n] = rng.standard_normal(n) * rng.choice([0.3, 5.0]) + rng.choice([0.0, 3.0])
        return xf

    for _ in range(40):
        x = orc.f32_to_bf16(row(1024, [0, 1, 64, 96]))
        xb = orc.bf16_to_f32(x)
        W = lambda l: _W(xb[8 * l:8 * l + 8])
        left = chain(C(C(W(0), W(64)), C(_Z(8), W(96))), [32, 64, 128, 256])
        right = chain(C(C(W(1), _Z(8)), _Z(16)), [32, 64, 128, 256])
        assert orc.welford128(x) == _stats(C(left, right))

        x = orc.f32_to_bf16(row(2048, [0, 128, 192, 1]))
        xb = orc.bf16_to_f32(x)
        lane = lambda l: _W(np.concatenate([xb[8 * l:8 * l + 8], xb[1024 + 8 * l:1024 + 8 * l + 8]]))
        left = chain(C(lane(0), lane(64)), [32, 64, 128, 256, 512])
        right = chain(C(lane(1), _Z(16)), [32, 64, 128, 256, 512])
        assert orc.welford128(x) == _stats(C(left, right))

        x = orc.f32_to_bf16(row(1030, [0, 128, 64]))
        xb = orc.bf16_to_f32(x)
        w0 = _W(np.concatenate([xb[0:8], xb[1024:1030]]))
        want = chain(C(w0, _W(xb[512:520])), [16, 32, 64, 128, 256, 512])
        assert orc.welford128(x) == _stats(want)


def test_welford_128_lanes_crafted_row(orc):
    """D = 1024; lane 0 holds eight 2^24, lanes 64 and 96 eight 1.0 each, every
    other element is 0.  Each lane is constant, so its state is (c, 0, 8).
    Derived by hand in binary32, nearest-even:
      s = 64  L0 = C((2^24,0,8), (1,0,8)): d = 1 - 2^24 (exact), r = 1/2,
              mean = 2^24 - (2^23 - 1/2) = 2^23 + 1/2 -> tie -> 2^23;
              d*d = 2^48 - 2^25 + 1 -> 2^48 - 2^25; times nA*r = 4: M2 = 2^50 - 2^27
              L32 = C(Z8, (1,0,8)) = (1/2, 4, 16)
      s = 32  d = 1/2 - 2^23 (exact), mean = 2^23 - (2^22 - 1/4) = 2^22 + 1/4 -> tie -> 2^22;
              M2A + M2B = 2^50 - 2^27 + 4 -> 2^50 - 2^27;  d*d -> 2^46 - 2^23, times 8;
              M2 = 3*2^49 - 3*2^26 -> tie -> 3*2^49 - 2^28 (even significand)
      s = 16 .. 1, each C(L0, Z_n) with n = 32 .. 512: mean halves (exact) and
              M2 gains 2^48, 2^47, 2^46, 2^45, 2^44 (all exact at ulp 2^27)
    Result: mean 2^17, M2 127*2^44 - 2^28, n 1024 (the exact mean is
    2^17 + 2^-6).  Pairing lanes 64 and 96 before lane 0 keeps the 2^-6."""
    x = np.zeros(1024, np.uint16)
    x[0:8] = 0x4B80        # 2^24
    x[512:520] = 0x3F80    # 1.0, chunk 64
    x[768:776] = 0x3F80    # 1.0, chunk 96
    assert orc.welford128(x) == (2.0 ** 17, float(127 * 2 ** 44 - 2 ** 28), 1024.0)


@pytest.mark.parametrize("D", [1, 7, 8, 100, 512, 1000, 1024, 3072, 5120, 8192])
def test_welford_against_float64(orc, D):
    rng = np.random.default_rng(D)
    for scale_, offset in ((1.0, 0.0), (20.0, 3.0), (1e-3, 100.0)):
        x = orc.f32_to_bf16((rng.standard_normal(D) * scale_ + offset).astype(np.float32))
        xf = orc.bf16_to_f32(x).astype(np.float64)
        mean, m2, n = orc.welford128(x)
        assert n == D
        amax = np.abs(xf).max()
        assert abs(mean - xf.mean()) <= D * 2.0 ** -23 * amax
        var64 = ((xf - xf.mean()) ** 2).sum()
        assert abs(m2 - var64) <= 2.0 ** -12 * var64 + D * 2.0 ** -40 * amax * amax


def test_welford_constant_row_is_exact(orc):
    for D in (1, 9, 512, 3072, 8192):
        for c in (0x3F80, 0xC2C8, 0x0001, 0x7F00):
            mean, m2, n = orc.welford128(np.full(D, c, np.uint16))
            assert np.float32(mean).view(np.uint32) == np.uint32(c << 16)
            assert m2 == 0.0 and n == D


# ---------------------------------------------------------------- Sum-128


def test_sum128_integer_rows_are_exact(orc):
    """Small integers: every square and partial sum is exact, so S = sum x^2."""
    rng = np.random.default_rng(3)
    for D in (1, 8, 129, 1000, 8192):
        xi = rng.integers(-16, 17, size=D)
        x = orc.f32_to_bf16(xi.astype(np.float32))
        assert orc.sum128_sq(x) == float((xi * xi).sum())


def test_sum128_against_float64(orc):
    rng = np.random.default_rng(4)
    for D in (100, 3072, 8192):
        x = orc.f32_to_bf16(rng.standard_normal(D).astype(np.float32))
        xf = orc.bf16_to_f32(x).astype(np.float64)
        sq = orc.bf16_to_f32(orc.f32_to_bf16((xf * xf).astype(np.float32))).astype(np.float64)
        S = orc.sum128_sq(x)
        # binary32 summation error bound over at most 64 + 7 additions per path
        assert abs(S - sq.sum()) <= 80 * 2.0 ** -24 * sq.sum()
        # and the rounding of the squares is really there (relative 2^-9 scale)
        assert abs(S - (xf * xf).sum()) <= 2.0 ** -8 * (xf * xf).sum()


def test_sum128_crafted_rows_fix_tree_and_ownership(orc):
    """Rows of 2^12 (square 2^24) and ones, every other element 0, where
    2^24 + 1 rounds back to 2^24 (a tie, to the even significand) but
    2^24 + 2 is exact; so the result tells whether the two ones met each other
    before they met 2^24.  Derived by hand:
      A  D 1024: 2^12 at element 0 (lane 0), 1 at 512 (lane 64) and 768 (lane 96).
         s = 64: L0 = 2^24 + 1 -> 2^24, L32 = 1;  s = 32: 2^24 + 1 -> 2^24.  S = 2^24.
         (Adjacent pairing adds lanes 64 and 96 first: 2^24 + 2.)
      B  D 2048: 2^12 at 0, 1 at 8 (chunk 1) and 1032 (chunk 129): both ones on
         lane 1, summed first to 2; s = 1: 2^24 + 2.  S = 2^24 + 2.
         (Lane l owning chunks 2l, 2l+1 puts chunk 1 on lane 0 after 2^24 and
         chunk 129 on lane 64: 2^24.)
      C  D 1024: 2^12 at 0, 1 at 1 and 3: all in chunk 0 on lane 0, in element
         order: 2^24 + 1 + 0 + 1 -> 2^24.  S = 2^24.
         (Element e on lane e mod 128 adds the ones on lanes 1 and 3 first: 2^24 + 2.)
      D  D 2048: 1 at 0 and 1, 2^12 at 1024 (chunk 128, lane 0's second chunk):
         ascending chunks: 1 + 1 = 2, then 2 + 2^24 exact.  S = 2^24 + 2.
         (Visiting chunk 128 first: 2^24.)"""
    def row(D, ones, big):
        x = np.zeros(D, np.uint16)
        x[list(ones)] = 0x3F80  # 1.0
        x[big] = 0x4580         # 2^12
        return x

    assert orc.sum128_sq(row(1024, (512, 768), 0)) == 2.0 ** 24
    assert orc.sum128_sq(row(2048, (8, 1032), 0)) == 2.0 ** 24 + 2
    assert orc.sum128_sq(row(1024, (1, 3), 0)) == 2.0 ** 24
    assert orc.sum128_sq(row(2048, (0, 1), 1024)) == 2.0 ** 24 + 2


def test_sum128_sparse_rows_unrolled(orc):
    """The tree unrolled by hand on rows with a few non-zero lanes (a zero lane
    adds exactly 0):
      D 1024, lanes 0, 1, 64, 96:  s = 64: L0 = S0 + S64, L32 = S96;
        s = 32: L0 = (S0 + S64) + S96;  s = 1: ((S0 + S64) + S96) + S1
      D 2048, chunks 0 and 128 (lane 0), 192 (lane 64), 1 (lane 1):
        (S_lane0 + S_lane64) + S_lane1
    with S_l lane l's binary32 sum, in element order, of bf16(x*x) (PyTorch CPU
    eager bf16 products)."""
    rng = np.random.default_rng(33)
    f = np.float32

    def seq(q):
        acc = f(0)
        for v in q:
            acc = f(acc + v)
        return acc

    def sq(x):
        t = bf(x)
        return (t * t).float().numpy()

    differs = 0
    for _ in range(60):
        xf = np.zeros(1024, np.float32)
        for c in (0, 1, 64, 96):
            xf[8 * c:8 * c + 8] = rng.standard_normal(8) * rng.choice([0.5, 4.0, 30.0])
        x = orc.f32_to_bf16(xf)
        q = sq(x)
        S = [seq(q[8 * l:8 * l + 8]) for l in range(128)]
        got = orc.sum128_sq(x)
        assert got == float(f(f(f(S[0] + S[64]) + S[96]) + S[1]))
        differs += got != float(f(f(S[0] + S[1]) + f(S[64] + S[96])))

        xf = np.zeros(2048, np.float32)
        for c in (0, 128, 192, 1):
            xf[8 * c:8 * c + 8] = rng.standard_normal(8) * rng.choice([0.5, 4.0, 30.0])
        x = orc.f32_to_bf16(xf)
        q = sq(x)
        lane = lambda l: seq(np.concatenate([q[8 * l:8 * l + 8], q[1024 + 8 * l:1024 + 8 * l + 8]]))
        assert orc.sum128_sq(x) == float(f(f(lane(0) + lane(64)) + lane(1)))
    assert differs  # the adjacent grouping is not the same sum on these rows


# ---------------------------------------------------------------- LN + modulate


def _ln_case(D, rows=4, seed=0, mrows=2):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    sc = (torch.randn(mrows, D, generator=g) * 0.1).to(torch.bfloat16)
    sh = (torch.randn(mrows, D, generator=g) * 0.1).to(torch.bfloat16)
    return x, sc, sh


@pytest.mark.parametrize("D", [2, 3, 8, 16, 64, 512, 3072])
def test_ln_output_within_one_ulp_of_float64_layer_norm(orc, D):
    """scale = shift = 0 leaves n = bf16(LN(x)); compare with torch.layer_norm
    in binary64 (biased variance, eps inside the root)."""
    x, _, _ = _ln_case(D, rows=64, seed=D)
    zeros = np.zeros((1, D), np.uint16)
    n = orc.bf16_to_f32(orc.ln_modulate(u16(x), zeros, zeros, 1e-6)).astype(np.float64)
    ref = torch.nn.functional.layer_norm(x.double(), (D,), eps=float(np.float32(1e-6))).numpy()
    assert np.all(np.abs(n - ref) <= bf16_ulp(ref))


def test_modulate_step_equals_torch_eager_bf16(orc):
    """Given n, out must equal PyTorch CPU eager (n * (1 + scale)) + shift."""
    D, rows = 3072, 32
    x, sc, sh = _ln_case(D, rows=rows, seed=11, mrows=2)
    zeros = np.zeros((1, D), np.uint16)
    n = bf(orc.ln_modulate(u16(x), zeros, zeros, 1e-6)).reshape(rows, D)
    got = orc.ln_modulate(u16(x), u16(sc), u16(sh), 1e-6)
    per = rows // 2
    sc_r = sc.repeat_interleave(per, dim=0)
    sh_r = sh.repeat_interleave(per, dim=0)
    want = u16((n * (1 + sc_r)) + sh_r)
    assert np.array_equal(got.reshape(-1), want.reshape(-1))


def test_constant_row_gives_shift(orc):
    D = 512
    _, sc, sh = _ln_case(D, rows=2, seed=5, mrows=1)
    for c in (0.0, 1.0, -3.5, 1e-20):
        x = torch.full((3, D), c).to(torch.bfloat16)
        got = orc.ln_modulate(u16(x), u16(sc), u16(sh), 1e-6)
        assert np.array_equal(got, np.broadcast_to(u16(sh), got.shape))


def test_modulation_row_mapping(orc):
    """Row r uses modulation row r // (rows // mod_rows)."""
    D, rows = 64, 12
    x, sc, sh = _ln_case(D, rows=rows, seed=9, mrows=3)
    got = orc.ln_modulate(u16(x), u16(sc), u16(sh), 1e-6)
    for r in range(rows):
        one = orc.ln_modulate(u16(x[r:r + 1]), u16(sc[r // 4:r // 4 + 1]), u16(sh[r // 4:r // 4 + 1]))
        assert np.array_equal(got[r], one[0])


def test_ln_f64_reference_matches_torch(orc):
    D = 300
    x, sc, sh = _ln_case(D, rows=8, seed=13, mrows=2)
    out, mag = orc.ln_modulate_f64(u16(x), u16(sc), u16(sh), 1e-6)
    ln = torch.nn.functional.layer_norm(x.double(), (D,), eps=float(np.float32(1e-6)))
    want = ln * (1 + sc.double().repeat_interleave(4, 0)) + sh.double().repeat_interleave(4, 0)
    assert np.allclose(out, want.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(mag >= np.abs(out))


def test_lossless_ln_modulate_near_exact(orc):
    """First-order error budget of the bit-exact chain, with u = 2^-8 the unit
    roundoff of bfloat16 and an error of k*u relative to a term T being at most
    k ulps of T: n = bf16(LN) (u), t = bf16(1+scale) (u), bf16(n*t) (u): 3u on
    the product, plus half an ulp for the final sum.  So <= 3.5 bf16 ulps of the
    largest term of the exact result."""
    for d, D in ((synth.tiny_ln_modulate(), 512), (synth.image_dit_block(seq=64), 3072)):
        x, sc, sh = u16(d["x"]).reshape(-1, D), u16(d["scale"]), u16(d["shift"])
        got = orc.bf16_to_f32(orc.ln_modulate(x, sc, sh, 1e-6)).astype(np.float64)
        ex, mag = orc.ln_modulate_f64(x, sc, sh, 1e-6)
        assert np.all(np.abs(got - ex) <= 3.5 * 1.01 * bf16_ulp(mag))


# ---------------------------------------------------------------- RMSNorm


def _rms_chain_torch(x: torch.Tensor, S: np.ndarray, w: torch.Tensor, sc: torch.Tensor, eps=1e-6):
    """Everything after the row sum, in PyTorch CPU eager ops, following the
    rounding points of the BF16-native rmsnorm_scale excerpt (PR #34085 digest,
    关键源码片段)."""
    D = x.shape[-1]
    Sf = torch.from_numpy(np.asarray(S, np.float32)).reshape(-1, 1)
    ms = (Sf / D).to(torch.bfloat16)
    inner = (ms.float() + np.float32(eps)).to(torch.bfloat16)
    rstd = (1.0 / torch.sqrt(inner.float())).to(torch.bfloat16)
    return ((x * rstd) * w) * sc


def test_rmsnorm_scale_chain_equals_torch_eager(orc):
    d = synth.tiny_ln_modulate()
    x = d["x"].reshape(-1, 512)
    S = np.array([orc.sum128_sq(u16(x[r])) for r in range(x.shape[0])])
    got = orc.rmsnorm_scale(u16(x), u16(d["weight"]), u16(d["scale"]), 1e-6)
    want = _rms_chain_torch(x, S, d["weight"], d["scale"].repeat_interleave(256, 0))
    assert np.array_equal(got, u16(want))


def test_rmsnorm_constant_row_closed_form(orc):
    """Constant row c: S = D*bf16(c^2) exactly, so ms = bf16(c^2)."""
    D = 4096
    ones = np.full((1, D), 0x3F80, np.uint16)
    for c in (0.5, 1.25, -3.0, 7.0):
        x = np.full((2, D), int(orc.f32_to_bf16(np.array([c], np.float32))[0]), np.uint16)
        cb = float(orc.bf16_to_f32(x[:1, :1])[0, 0])
        sq = float(orc.bf16_to_f32(orc.f32_to_bf16(np.array([cb * cb], np.float32)))[0])
        assert orc.sum128_sq(x[0]) == D * sq
        inner = np.float32(orc.bf16_to_f32(orc.f32_to_bf16(np.array([np.float32(sq) + np.float32(1e-6)], np.float32)))[0])
        rstd = orc.bf16_to_f32(orc.f32_to_bf16(np.array([np.float32(1) / np.sqrt(inner)], np.float32)))[0]
        want = orc.f32_to_bf16(np.array([np.float32(cb) * rstd], np.float32))[0]
        got = orc.rmsnorm_scale(x, ones[0], ones, 1e-6)
        assert np.all(got == want)


def test_rmsnorm_zero_row_and_unit_rms(orc):
    D = 3072
    rng = np.random.default_rng(2)
    x = orc.f32_to_bf16(rng.standard_normal((16, D)).astype(np.float32) * 5)
    x[3] = 0
    ones = np.full((1, D), 0x3F80, np.uint16)
    y = orc.bf16_to_f32(orc.rmsnorm_scale(x, ones[0], ones, 1e-6)).astype(np.float64)
    assert np.all(y[3] == 0)
    rms = np.sqrt((np.delete(y, 3, 0) ** 2).mean(axis=1))
    assert np.all(np.abs(rms - 1.0) < 2.0 ** -6)


def test_rmsnorm_f64_reference_matches_torch(orc):
    d = synth.tiny_ln_modulate()
    x = d["x"].reshape(-1, 512)
    out, _ = orc.rmsnorm_scale_f64(u16(x), u16(d["weight"]), u16(d["scale"]), 1e-6)
    xd = x.double()
    want = xd * torch.rsqrt((xd * xd).mean(-1, keepdim=True) + float(np.float32(1e-6)))
    want = want * d["weight"].double() * d["scale"].double().repeat_interleave(256, 0)
    assert np.allclose(out, want.numpy(), rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- tanh residual


def test_rmsnorm_tanh_residual_composition(orc):
    """out = bf16(r + bf16(tanh_bf16(g) * n)) with n the rmsnorm chain without
    scale (rmsnorm_scale with scale 1 gives n, since bf16(n*1) = n); the last two
    steps are checked against PyTorch CPU eager bf16 ops."""
    D, rows = 1000, 24
    g = torch.Generator().manual_seed(21)
    x = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    gate = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    res = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    w = (1 + 0.05 * torch.randn(D, generator=g)).to(torch.bfloat16)
    ones = np.full((1, D), 0x3F80, np.uint16)
    n = bf(orc.rmsnorm_scale(u16(x), u16(w), ones, 1e-6))
    tg = bf(orc.tanh_table()[u16(gate)])
    want = u16(res + tg * n)
    got = orc.rmsnorm_tanh_residual(u16(x), u16(gate), u16(res), u16(w), 1e-6)
    assert np.array_equal(got, want)


def test_rmsnorm_chains_near_exact(orc):
    """First-order budget (u = 2^-8, k*u relative = at most k ulps): the rounded
    squares, bf16(S/D) and bf16(ms+eps) give 3u under the root, halved by it,
    plus u for bf16(rstd): 2.5u; bf16(x*rstd) and bf16(.*w): 4.5u on n.
    rmsnorm_scale adds bf16(n*scale): <= 5.5 ulps.  The tanh residual adds the
    rounded tanh and bf16(tg*n): 6.5u on p, plus half an ulp for the sum: <= 7."""
    for D, T in ((1024, 77), (3072, 300), (8192, 40)):
        d = synth.sweep_case(D, T)
        x, g, r, w, sc = (u16(d[k].contiguous())
                          for k in ("x", "gate_tok", "residual", "weight", "scale"))
        got = orc.bf16_to_f32(orc.rmsnorm_tanh_residual(x, g, r, w, 1e-6)).astype(np.float64)
        ex, mag = orc.rmsnorm_tanh_residual_f64(x, g, r, w, 1e-6)
        assert np.all(np.abs(got - ex) <= 7 * 1.01 * bf16_ulp(mag))
        got = orc.bf16_to_f32(orc.rmsnorm_scale(x, w, sc, 1e-6)).astype(np.float64)
        ex, mag = orc.rmsnorm_scale_f64(x, w, sc, 1e-6)
        assert np.all(np.abs(got - ex) <= 5.5 * 1.01 * bf16_ulp(mag))


# ---------------------------------------------------------------- gated residual


def test_residual_gate_add_equals_torch_eager(orc):
    g = torch.Generator().manual_seed(31)
    rows, D = 64, 777
    x = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    y = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    gate = (torch.randn(4, D, generator=g)).to(torch.bfloat16)
    # extremes: overflow to inf, subnormal products, exact cancellation
    x[0, :4] = torch.tensor([3e38, -3e38, 1e-38, 0.0]).to(torch.bfloat16)
    y[0, :4] = torch.tensor([3e38, 3e38, 1e-38, 0.0]).to(torch.bfloat16)
    got = orc.residual_gate_add(u16(x), u16(gate), u16(y))
    want = x + gate.repeat_interleave(16, 0) * y
    assert np.array_equal(got, u16(want))


def test_residual_gate_add_zero_gate_is_identity(orc):
    g = torch.Generator().manual_seed(32)
    x = torch.randn(8, 96, generator=g).to(torch.bfloat16)
    y = torch.randn(8, 96, generator=g).to(torch.bfloat16)
    z = np.zeros((1, 96), np.uint16)
    assert np.array_equal(orc.residual_gate_add(u16(x), z, u16(y)), u16(x))


# ---------------------------------------------------------------- QKV epilogue


def _small_qkv(**kw):
    return synth.qkv_epilogue_case(batch=2, s_txt=5, grid_h=3, grid_w=4, heads=3, **kw)


def _run_qkv(orc, d, cos_txt=None, sin_txt=None, cos_img=None, sin_img=None):
    return orc.qkv_epilogue(u16(d["txt"].contiguous()), u16(d["img"].contiguous()), d["batch"],
                            d["heads"], d["head_dim"], u16(d["wq_txt"]), u16(d["wk_txt"]),
                            u16(d["wq_img"]), u16(d["wk_img"]),
                            (d["cos_txt"] if cos_txt is None else cos_txt).numpy(),
                            (d["sin_txt"] if sin_txt is None else sin_txt).numpy(),
                            (d["cos_img"] if cos_img is None else cos_img).numpy(),
                            (d["sin_img"] if sin_img is None else sin_img).numpy(), d["eps"])


def test_qkv_v_is_bit_copy_and_layout(orc):
    d = _small_qkv()
    B, H, hd = d["batch"], d["heads"], d["head_dim"]
    joint = _run_qkv(orc, d)
    txt = u16(d["txt"].contiguous()).reshape(B, 5, 3, H, hd)
    img = u16(d["img"].contiguous()).reshape(B, 12, 3, H, hd)
    assert joint.shape == (B, 3, H, 17, hd)
    # V: text first, then image
    assert np.array_equal(joint[:, 2, :, :5], txt[:, :, 2].transpose(0, 2, 1, 3))
    assert np.array_equal(joint[:, 2, :, 5:], img[:, :, 2].transpose(0, 2, 1, 3))


def test_qkv_identity_rotation_is_head_rmsnorm(orc):
    """cos = 1, sin = 0: each Q/K head equals the rmsnorm chain at D = hd with
    scale 1, using the branch's own weight."""
    d = _small_qkv()
    B, H, hd = d["batch"], d["heads"], d["head_dim"]
    one = lambda S: torch.ones(S, hd // 2)
    zero = lambda S: torch.zeros(S, hd // 2)
    joint = _run_qkv(orc, d, one(5), zero(5), one(12), zero(12))
    ones = np.full((1, hd), 0x3F80, np.uint16)
    for name, S, off, wq, wk in (("txt", 5, 0, "wq_txt", "wk_txt"), ("img", 12, 5, "wq_img", "wk_img")):
        src = u16(d[name].contiguous()).reshape(B, S, 3, H, hd)
        for part, w in ((0, wq), (1, wk)):
            heads = src[:, :, part].reshape(-1, hd)
            want = orc.rmsnorm_scale(heads, u16(d[w]), ones, 1e-6).reshape(B, S, H, hd)
            assert np.array_equal(joint[:, part, :, off:off + S], want.transpose(0, 2, 1, 3))


def test_qkv_rotation_equals_torch_eager_and_position_zero(orc):
    """o0 = bf16(n0*c - n1*s), o1 = bf16(n0*s + n1*c) in binary32 eager ops,
    applied to the identity-rotation output n; token 0 (c=1, s=0) is n."""
    d = _small_qkv()
    B, H, hd = d["batch"], d["heads"], d["head_dim"]
    one = lambda S: torch.ones(S, hd // 2)
    zero = lambda S: torch.zeros(S, hd // 2)
    n = _run_qkv(orc, d, one(5), zero(5), one(12), zero(12))
    joint = _run_qkv(orc, d)
    cos = torch.cat([d["cos_txt"], d["cos_img"]])  # [17, hd/2]
    sin = torch.cat([d["sin_txt"], d["sin_img"]])
    nt = bf(n[:, :2]).float().reshape(B, 2, H, 17, hd // 2, 2)
    n0, n1 = nt[..., 0], nt[..., 1]
    o0 = (n0 * cos - n1 * sin).to(torch.bfloat16)
    o1 = (n0 * sin + n1 * cos).to(torch.bfloat16)
    want = torch.stack([o0, o1], -1).reshape(B, 2, H, 17, hd)
    assert np.array_equal(joint[:, :2], u16(want))
    assert np.array_equal(joint[:, :2, :, 0], n[:, :2, :, 0])  # text position 0
    assert np.array_equal(joint[:, :2, :, 5], n[:, :2, :, 5])  # image cell (0, 0)


def test_qkv_rotation_preserves_pair_norm(orc):
    d = _small_qkv()
    B, H, hd = d["batch"], d["heads"], d["head_dim"]
    one = lambda S: torch.ones(S, hd // 2)
    zero = lambda S: torch.zeros(S, hd // 2)
    n = orc.bf16_to_f32(_run_qkv(orc, d, one(5), zero(5), one(12), zero(12))[:, :2]).astype(np.float64)
    o = orc.bf16_to_f32(_run_qkv(orc, d)[:, :2]).astype(np.float64)
    n2 = (n.reshape(-1, 2) ** 2).sum(1)
    o2 = (o.reshape(-1, 2) ** 2).sum(1)
    amax = np.abs(n.reshape(-1, 2)).max(1)
    assert np.all(np.abs(np.sqrt(o2) - np.sqrt(n2)) <= 2 * bf16_ulp(amax))


def test_qkv_rotation_composes(orc):
    """Rotating by p1 and then by p2 matches rotating by p1 + p2 (binary64 check
    on the oracle's rotation with the synthetic text tables)."""
    d = synth.qkv_epilogue_case(batch=1, s_txt=40, grid_h=1, grid_w=1, heads=1)
    hd = d["head_dim"]
    cos, sin = d["cos_txt"].double().numpy(), d["sin_txt"].double().numpy()
    p1, p2 = 7, 30
    c = cos[p1] * cos[p2] - sin[p1] * sin[p2]
    s = sin[p1] * cos[p2] + cos[p1] * sin[p2]
    assert np.allclose(c, cos[p1 + p2], atol=1e-6) and np.allclose(s, sin[p1 + p2], atol=1e-6)
    # the oracle applies exactly these tables: the rotation of token p1+p2 is
    # within rounding of rotating token p1's normalised pair by table p2
    one = torch.ones(40, hd // 2); zero = torch.zeros(40, hd // 2)
    dd = dict(d)
    row = d["txt"][p1].clone()
    dd["txt"] = torch.stack([row] * 40)
    n = orc.bf16_to_f32(_run_qkv(orc, dd, one, zero, d["cos_img"], d["sin_img"])[0, 0, 0, 0]).astype(np.float64)
    o = orc.bf16_to_f32(_run_qkv(orc, dd)[0, 0, 0]).astype(np.float64)  # [40, hd]
    n0, n1 = n[0::2], n[1::2]
    a0 = n0 * cos[p1] - n1 * sin[p1]
    a1 = n0 * sin[p1] + n1 * cos[p1]
    b0 = a0 * cos[p2] - a1 * sin[p2]
    b1 = a0 * sin[p2] + a1 * cos[p2]
    assert np.allclose(o[p1 + p2, 0::2], b0, atol=2 * 2.0 ** -7 * np.abs(n).max())
    assert np.allclose(o[p1 + p2, 1::2], b1, atol=2 * 2.0 ** -7 * np.abs(n).max())


def test_qk_head_f64_reference(orc):
    d = _small_qkv()
    hd = d["head_dim"]
    src = u16(d["txt"][3, :hd].contiguous())
    out, _ = orc.qk_head_f64(src, u16(d["wq_txt"]), d["cos_txt"][3].numpy(), d["sin_txt"][3].numpy())
    x = d["txt"][3, :hd].double()
    n = x * torch.rsqrt((x * x).mean() + float(np.float32(1e-6))) * d["wq_txt"].double()
    c, s = d["cos_txt"][3].double(), d["sin_txt"][3].double()
    want = torch.stack([n[0::2] * c - n[1::2] * s, n[0::2] * s + n[1::2] * c], -1).reshape(-1)
    assert np.allclose(out, want.numpy(), rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- gated residual + LN + modulate


def test_gated_residual_ln_modulate_is_the_composition(orc):
    """Without a bias the fused chain is residual_gate_add followed by
    ln_modulate on its result; with one, the bias add is the eager bf16
    `update + bias` (PyTorch CPU) feeding the same composition."""
    g = torch.Generator().manual_seed(41)
    rows, D = 48, 1000
    r = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    u = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    b = (0.1 * torch.randn(D, generator=g)).to(torch.bfloat16)
    gate = (0.1 * torch.randn(3, D, generator=g)).to(torch.bfloat16)
    sc = (0.1 * torch.randn(3, D, generator=g)).to(torch.bfloat16)
    sh = (0.1 * torch.randn(3, D, generator=g)).to(torch.bfloat16)
    R, U, G, SC, SH = u16(r), u16(u), u16(gate), u16(sc), u16(sh)
    for bias, a in ((None, U), (u16(b), u16(u + b))):
        res, out = orc.gated_residual_ln_modulate(R, G, U, bias, SC, SH, 1e-6)
        want_res = orc.residual_gate_add(R, G, a)
        assert np.array_equal(res, want_res)
        assert np.array_equal(out, orc.ln_modulate(want_res, SC, SH, 1e-6))
    # the residual stream itself against PyTorch CPU eager bf16 ops
    res, _ = orc.gated_residual_ln_modulate(R, G, U, u16(b), SC, SH, 1e-6)
    assert np.array_equal(res, u16(r + gate.repeat_interleave(16, 0) * (u + b)))


# ------------------------------------------------------------ modulation table


def _eager_table(table: torch.Tensor, temb: torch.Tensor) -> np.ndarray:
    """The pages' eager expression, on the CPU, with the model's shapes: the
    table parameter [1, 6, D], temb [B=1, S, 6, D];
    (table.unsqueeze(0) + temb.float()).chunk(6, dim=2), stacked into (6, S, D)."""
    param = table.reshape(1, 6, -1)
    e = temb.reshape(1, -1, 6, param.shape[-1])
    chunks = (param.unsqueeze(0) + e.float()).chunk(6, dim=2)
    return torch.stack([c.reshape(e.shape[1], -1) for c in chunks]).numpy()


def f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def _bits_or_f32(t: torch.Tensor) -> np.ndarray:
    return u16(t) if t.dtype == torch.bfloat16 else t.numpy()


@pytest.mark.parametrize("tab_dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("emb_dt", [torch.bfloat16, torch.float32])
def test_modulation_table_equals_the_eager_expression(orc, tab_dt, emb_dt):
    """Bit for bit against PyTorch CPU eager on the pages' own expression,
    including signed zeros and huge/tiny operands."""
    g = torch.Generator().manual_seed(71)
    rows, D = 37, 24
    table = (torch.randn(6, D, generator=g) / D ** 0.5).to(tab_dt)
    temb = torch.randn(rows, 6, D, generator=g)
    temb[0, :, :4] = torch.tensor([0.0, -0.0, 3e38, 1e-40])
    temb = temb.to(emb_dt)
    want = _eager_table(table, temb)
    got = orc.modulation_table_add(_bits_or_f32(table), _bits_or_f32(temb))
    assert got.shape == (6, rows, D)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_modulation_table_closed_forms(orc):
    """A zero operand is the identity; bf16 operands whose exponents differ by
    at most 16 add exactly in binary32, so the result equals the binary64 sum."""
    g = torch.Generator().manual_seed(72)
    rows, D = 19, 40
    table = torch.randn(6, D, generator=g).to(torch.bfloat16)
    temb = torch.randn(rows, 6 * D, generator=g).to(torch.bfloat16)
    T, E = u16(table), u16(temb)
    zero_t = np.zeros_like(T)
    out = orc.modulation_table_add(zero_t, E)
    assert np.array_equal(out, f32(E).reshape(rows, 6, D).transpose(1, 0, 2))
    out = orc.modulation_table_add(T, np.zeros_like(E))
    assert np.array_equal(out, np.broadcast_to(f32(T)[:, None, :], (6, rows, D)))
    # exact sums: both operands in [1, 2) as bf16 -> the sum needs at most 9 bits
    t1 = (1 + torch.rand(6, D, generator=g)).to(torch.bfloat16)
    e1 = (1 + torch.rand(rows, 6 * D, generator=g)).to(torch.bfloat16)
    out = orc.modulation_table_add(u16(t1), u16(e1))
    exact = (f32(u16(t1)).astype(np.float64)[:, None, :]
             + f32(u16(e1)).astype(np.float64).reshape(rows, 6, D).transpose(1, 0, 2))
    assert np.array_equal(out.astype(np.float64), exact)


def test_modulation_table_layout(orc):
    """Plane k, row r, column d comes from temb[r, k*D + d] and table[k, d]."""
    rows, D = 5, 3
    table = np.arange(6 * D, dtype=np.float32).reshape(6, D) * 1000
    temb = np.arange(rows * 6 * D, dtype=np.float32).reshape(rows, 6 * D)
    out = orc.modulation_table_add(table, temb)
    for k in range(6):
        for r in range(rows):
            for d in range(D):
                assert out[k, r, d] == table[k, d] + temb[r, k * D + d]


# ------------------------------------------------------------ FP8 E4M3


def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_matches_torch_in_range(orc):
    """Every bfloat16 value below 448 in magnitude, random binary32 values, and
    every midpoint between neighbouring E4M3 values (ties to even), against
    PyTorch's CPU float8_e4m3fn conversion."""
    b = np.arange(65536, dtype=np.uint32)
    v = (b << 16).view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) < 448)]
    rng = np.random.default_rng(5)
    r = (rng.standard_normal(1 << 20) * np.exp2(rng.integers(-12, 9, 1 << 20))).astype(np.float32)
    r = r[np.abs(r) < 448]
    codes = np.arange(0x7f, dtype=np.uint8)  # all finite non-negative codes
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(np.float32)
    for x in (v, r, mids, -mids):
        assert np.array_equal(orc.f32_to_e4m3(x), _torch_e4m3(x))


def test_e4m3_closed_forms(orc):
    f = orc.f32_to_e4m3
    cases = [(448.0, 0x7E), (-448.0, 0xFE), (464.0, 0x7E), (500.0, 0x7E), (1e30, 0x7E),
             (float("inf"), 0x7E), (-float("inf"), 0xFE), (0.0, 0x00), (-0.0, 0x80), (2.0 ** -9, 0x01),
             (2.0 ** -10, 0x00), (3 * 2.0 ** -11, 0x01), (3 * 2.0 ** -10, 0x02), (5 * 2.0 ** -10, 0x02), (2.0 ** -6, 0x08), (1.0, 0x38), (1.0625, 0x38),
             (1.1875, 0x3A), (240.0, 0x77), (float("nan"), 0x7F), (-float("nan"), 0x7F)]
    for x, want in cases:
        assert int(f(np.array([x], np.float32))[0]) == want, (x, hex(want))
    # every code round-trips through its own value
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(f(vals), codes)


def test_quant_e4m3_of_a_bf16_output(orc):
    """The static quantiser multiplies by the correctly rounded 1/scale once."""
    g = torch.Generator().manual_seed(81)
    y = (torch.randn(20, 96, generator=g) * 3).to(torch.bfloat16)
    for scale in (1.0, 0.0173, 3.3e-3, 0.5, 7.0):
        inv = np.float32(1.0) / np.float32(scale)
        prod = y.float().numpy() * inv
        got = orc.quant_e4m3(u16(y), scale)
        inr = np.abs(prod) < 448
        assert np.array_equal(got[inr], _torch_e4m3(prod[inr]))
        assert np.all(got[~inr] == np.where(prod[~inr] > 0, 0x7E, 0xFE))  # saturated


# ------------------------------------------------------------ NVFP4

_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_brute(v: float) -> int:
    """Nearest of the 16 codes in binary64, ties to the code with mantissa 0."""
    if v != v:
        return 0x7
    a = min(abs(v), 6.0)
    best = min(range(8), key=lambda c: (abs(_E2M1[c] - a), c & 1))
    return (0x8 if math.copysign(1.0, v) < 0 else 0) | best


def test_e2m1_brute_force(orc):
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.uniform(-8, 8, 20000), rng.standard_normal(5000) * 0.3,
                        (_E2M1[:-1] + _E2M1[1:]) / 2, -(_E2M1[:-1] + _E2M1[1:]) / 2, _E2M1, -_E2M1,
                        [1e30, -1e30, np.inf, -np.inf, 6.0001, 1e-40]]).astype(np.float32)
    got = orc.f32_to_e2m1(v)
    want = np.array([_e2m1_brute(float(x)) for x in v], np.uint8)
    assert np.array_equal(got, want)
    assert orc.f32_to_e2m1(np.array([-0.0], np.float32))[0] == 0x8


def _swizzle_by_reshape(S: np.ndarray) -> np.ndarray:
    """The 128x4 tile layout by array reshaping (independent of the scalar
    index formula): rows -> (tile, band of 32, row in band), blocks -> (tile,
    column), ordered (row tile, column tile, row in band, band, column)."""
    mp, kp = S.shape
    return S.reshape(mp // 128, 4, 32, kp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)


def _unswizzle_by_reshape(sf: np.ndarray, mp: int, kp: int) -> np.ndarray:
    return sf.reshape(mp // 128, kp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(mp, kp)


def _nvfp4_reference_scales(y: np.ndarray, gs: float, orc) -> np.ndarray:
    f = (y.astype(np.uint32) << 16).view(np.float32)
    rows, D = f.shape
    amax = np.abs(f.reshape(rows, D // 16, 16)).max(axis=2)
    sf = ((amax.astype(np.float32) * np.float32(gs)).astype(np.float32) / np.float32(6)).astype(np.float32)
    return orc.f32_to_e4m3(sf)


def test_nvfp4_scales_and_swizzle(orc):
    g = torch.Generator().manual_seed(91)
    for rows, D in ((130, 256), (5, 64), (256, 1024)):
        y = u16((torch.randn(rows, D, generator=g) * 2).to(torch.bfloat16))
        gs = 448.0 * 6.0 / 9.0
        q, sf = orc.quant_nvfp4(y, gs, sf_fill=0xAB)
        mp, kp = orc.nvfp4_sf_shape(rows, D)
        S = np.full((mp, kp), 0xAB, np.uint8)
        S[:rows, :D // 16] = _nvfp4_reference_scales(y, gs, orc)
        assert np.array_equal(sf, _swizzle_by_reshape(S))


def test_nvfp4_elements_decode_close_and_block_max_is_six(orc):
    g = torch.Generator().manual_seed(92)
    rows, D = 64, 512
    y = u16((torch.randn(rows, D, generator=g) * 3).to(torch.bfloat16))
    gs = 448.0 * 6.0 / 12.0
    q, sf = orc.quant_nvfp4(y, gs)
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(rows, D)
    mag = _E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    Sm = _unswizzle_by_reshape(sf, *orc.nvfp4_sf_shape(rows, D))[:rows, :D // 16]
    sval = torch.from_numpy(Sm.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    scale = np.repeat(sval, 16, axis=1) / gs
    f = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    deq = mag * scale
    step = np.repeat(sval, 16, axis=1) / gs  # 1 E2M1 unit at the top binade is 2 * scale
    assert np.all(np.abs(deq - f) <= 1.0 * step + 1e-30)
    fb = np.abs(f).reshape(rows, D // 16, 16)
    cb = (codes & 7).reshape(rows, D // 16, 16)
    top = cb[np.arange(rows)[:, None], np.arange(D // 16)[None, :], fb.argmax(axis=2)]
    assert np.all(top == 7)  # the block's largest magnitude maps to +-6


def test_nvfp4_zero_block_and_exact_values(orc):
    rows, D = 2, 32
    vals = np.array([6, 4, 3, 2, 1.5, 1, 0.5, 0, -6, -4, -3, -2, -1.5, -1, -0.5, -0.0], np.float32)
    y = np.zeros((rows, D), np.float32)
    y[0, :16] = vals * 2.0  # block amax 12: scale 12 * gs / 6 = 2 * gs; gs = 0.5 -> s = 1.0 exactly
    y[1, 16:] = vals
    yb = orc.f32_to_bf16(y)
    q, sf = orc.quant_nvfp4(yb, 0.5)
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(rows, D)
    want = orc.f32_to_e2m1(vals)
    assert np.array_equal(codes[0, :16], want)
    assert np.all(codes[0, 16:] == 0) and np.all(codes[1, :16] == 0)  # zero blocks
    S = _unswizzle_by_reshape(sf, *orc.nvfp4_sf_shape(rows, D))
    assert S[0, 0] == 0x38 and S[0, 1] == 0 and S[1, 0] == 0  # 1.0 in E4M3; zero blocks: scale 0
