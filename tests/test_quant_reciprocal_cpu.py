"""The NVFP4 quantiser's divide-free arithmetic, checked on the CPU.

The NVFP4 conversion rule divides every element of a 16-element block by the
block's quantised e4m3 scale sf, correctly rounded, and rounds the quotient
to e2m1 (MegaMoE kernel-drop workflow page, sec. 三,
nvfp4_quantize_per_block_16; the oracle divides).  The kernels' quantiser
(quant_nvfp4_16 in csrc/quant.cuh, used for the GEMM1 input and for the
GEMM2 input after SwiGLU) instead takes r = RN(1/sf) once and, per element,
q = RN(x r) refined by one Newton step on the residual,
RN(q + RN(x - q sf) r), with both steps fused (one rounding each), and the
sign of x.  These tests emulate the fused steps exactly in float64 and check
that the refined value is the correctly rounded quotient:
- for every fp32 significand against every e4m3 significand (exponents only
  scale the steps while the residual stays normal, |x| >= 2^-99);
- for random fp32 values of every exponent against every e4m3 scale;
- and, for the layer's bf16 input, that every bf16 value under every scale a
  block can produce gets the divide's e2m1 code, the tiny quotients included.
CPU only.
"""
import numpy as np

import oracle


def _f32(a):
    return np.asarray(a, np.float64).astype(np.float32)


def _fma_sum_f32(a, b):
    """RN_f32(a + b) of float64 a, b whose exact sum may need more than 53 bits:
    TwoSum gives hi + lo = a + b exactly; hi rounds to float32 the same way as
    the exact sum unless hi lies halfway between two float32 numbers, where
    lo's sign decides."""
    hi = a + b
    bb = hi - a
    lo = (a - (hi - bb)) + (b - bb)
    h32 = hi.astype(np.float32)
    h64 = h32.astype(np.float64)
    up = np.nextafter(h32, np.float32(np.inf))
    dn = np.nextafter(h32, np.float32(-np.inf))
    out = h32.copy()
    sel = (hi == (h64 + up.astype(np.float64)) / 2) & (lo > 0)
    out[sel] = up[sel]
    sel = (hi == (h64 + dn.astype(np.float64)) / 2) & (lo < 0)
    out[sel] = dn[sel]
    return out


def _refined_quotient(x, s):
    """The kernel's steps for float32 x, scale s (float32 scalar)."""
    r = np.float32(1.0) / s                                   # RN(1/s)
    q = x * r                                                 # RN(x r)
    # fma(-q, s, x): q s has <= 28 significant bits and lies within a few ulp
    # of x, so x - q s is exact in float64 and rounds once to float32
    rho = _f32(x.astype(np.float64) - q.astype(np.float64) * np.float64(s))
    # fma(rho, r, q): rho r is exact in float64 (48 bits); the sum is not
    q2 = _fma_sum_f32(rho.astype(np.float64) * np.float64(r), q.astype(np.float64))
    return np.copysign(q2, x), q


def _all_pairs():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)              # +0 .. largest finite
    x = (bits << 16).view(np.float32)
    x = np.concatenate([x, -x])
    scales = oracle.decode("e4m3", np.arange(1, 0x7F, dtype=np.uint8))
    for s in scales:
        s = np.float32(s)
        yield s, x[(np.abs(x) <= 8 * s) | (s == np.float32(448.0))]


def test_refined_quotient_is_correctly_rounded_for_every_significand_pair():
    np.seterr(all="ignore")
    a = np.arange(0x3F800000, 0x40000000, dtype=np.uint32).view(np.float32)   # [1, 2)
    naive_bad = 0
    for m in range(8, 16):                                    # e4m3 significands 1.000 .. 1.111
        s = np.float32(m / 8.0)
        q2, q = _refined_quotient(a, s)
        assert np.array_equal(q2, a / s), m
        naive_bad += int((q != a / s).sum())
    # the plain product is wrong for most of them: the step is what makes it exact
    assert naive_bad > 10_000_000


def test_refined_quotient_is_correctly_rounded_at_every_exponent():
    np.seterr(all="ignore")
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 0x7F800000, 400_000, dtype=np.uint32)
    x = bits.view(np.float32)
    x = np.where(rng.random(x.size) < 0.5, -x, x)
    x = x[np.abs(x) >= np.float32(2.0 ** -99)]
    for s in oracle.decode("e4m3", np.arange(1, 0x7F, dtype=np.uint8)):
        s = np.float32(s)
        xs = x[(np.abs(x) <= 8 * s) | (s == np.float32(448.0))]
        q2, _ = _refined_quotient(xs, s)
        assert np.array_equal(q2, xs / s), float(s)


def test_refined_quotient_gives_the_divides_codes_for_every_bf16_pair():
    np.seterr(all="ignore")
    n = naive_bad = 0
    for s, x in _all_pairs():
        exact = x / s                                         # correctly rounded
        q2, q = _refined_quotient(x, s)
        want = oracle.encode("e2m1", exact)
        assert np.array_equal(oracle.encode("e2m1", q2), want), float(s)
        # the quotients themselves agree except far below the first e2m1 step
        diff = q2 != exact
        assert not diff.any() or np.abs(exact[diff]).max() < 1e-35, float(s)
        assert np.array_equal(np.signbit(q2), np.signbit(exact))
        naive_bad += int((oracle.encode("e2m1", q) != want).sum())
        n += x.size
    assert n > 4_000_000
    # without the Newton step, exact e2m1 midpoints under scales such as
    # 15 * 2^k land one ulp off and round the other way
    assert naive_bad > 0


def test_fused_sum_emulation_rounds_halfway_cases_by_the_low_part():
    # 1 + 2^-24 is halfway between float32 neighbours 1 and 1 + 2^-23
    a = np.array([1.0 + 2.0 ** -24, 1.0 + 2.0 ** -24, 1.0 + 2.0 ** -24])
    b = np.array([2.0 ** -80, -(2.0 ** -80), 0.0])
    got = _fma_sum_f32(a, b)
    assert got[0] == np.float32(1.0 + 2.0 ** -23)
    assert got[1] == np.float32(1.0)
    assert got[2] == np.float32(1.0)                          # tie to even
