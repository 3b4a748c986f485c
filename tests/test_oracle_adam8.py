"""Pins of the oracle's 8-bit Adam (the optimizer of state multiplier K = 6,
"DeepSpeed ZeRO Stages" sec. 1.2; block-wise quantization after Dettmers et
al., "8-bit Optimizers via Block-wise Quantization").  CPU only.

What fixes the oracle here, apart from itself:
  - the structure of the dynamic map: monotone, one decade per exponent run,
    2^f equally spaced values per decade, exact end points 1, 1e-6 and 1e-7;
  - nearest-code decisions checked by brute force, ties by exact midpoints;
  - a hand-traced first step (codes worked out by hand from the map);
  - reduction to the pinned fp32 Adam: the first step from a zero state, and
    every step of blocks whose states have one magnitude (x = +-1 is exact);
  - the decomposition dequantize -> fp32 Adam -> block absmax -> nearest code
    of m' / absmax, checked against the pinned fp32 Adam and a brute-force
    nearest search;
  - the normalization is the quotient m' / absmax rounded once: two blocks
    worked out in exact rational arithmetic where m' * fp32(1 / absmax) lands
    on the other side of a code threshold (a reciprocal-multiply reading
    fails them);
  - block isolation: a spike in one block of 2048 leaves the others alone.
"""
from fractions import Fraction

import numpy as np
import pytest

B = 2048
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _decode(oracle, m_codes, v_codes, m_scale, v_scale):
    """Dequantized m and v in float32, one multiply each (the oracle's own
    order: signed magnitude, then the block scale)."""
    mag7, mag8 = oracle.adam8_maps()
    blk = np.arange(m_codes.size) // B
    mag = mag7[m_codes & 0x7F]
    m = np.where(m_codes & 0x80, -mag, mag).astype(np.float32) * m_scale[blk]
    v = mag8[v_codes] * v_scale[blk]
    return m.astype(np.float32), v.astype(np.float32)


def _state(n):
    return (np.zeros(n, np.uint8), np.zeros(n, np.uint8), np.zeros((n + B - 1) // B, np.float32),
            np.zeros((n + B - 1) // B, np.float32))


@pytest.mark.parametrize("bits,name", [(7, "mag7"), (8, "mag8")])
def test_map_structure(oracle, bits, name):
    table = dict(zip(("mag7", "mag8"), oracle.adam8_maps()))[name].astype(np.float64)
    assert table.size == 1 << bits
    assert table[0] == 0.0 and table[-1] == 1.0
    assert table[1] == float(np.float32(10.0 ** -(bits - 1)))        # 1e-6 (signed) / 1e-7 (unsigned)
    assert np.all(np.diff(table) > 0)
    for e in range(bits):                                              # decade 10^-e: codes of bit length bits - e
        lo_code, hi_code = 1 << (bits - e - 1), 1 << (bits - e)
        vals = table[lo_code:hi_code]
        assert vals.size == 1 << (bits - e - 1)
        top = 10.0 ** -e
        assert np.all(vals > 0.1 * top * (1 + 1e-7)) and np.all(vals <= top * (1 + 1e-7))
        assert abs(vals[-1] - top) <= top * 1e-7                       # the decade's top value is its power of ten
        step = 0.9 * top / vals.size                                   # equal steps of [0.1, 1] * 10^-e
        np.testing.assert_allclose(np.diff(np.concatenate([[0.1 * top], vals])), step, rtol=0,
                                   atol=top * 2.0 ** -22)                      # two float roundings


def test_nearest_codes_brute_force(oracle):
    mag7, mag8 = (t.astype(np.float64) for t in oracle.adam8_maps())
    rng = np.random.Generator(np.random.PCG64(3))
    xs = np.concatenate([rng.uniform(-1, 1, 600), rng.standard_normal(200) * 1e-3,
                         np.sign(rng.standard_normal(200)) * 10.0 ** rng.uniform(-9, 0, 200),
                         mag7[rng.integers(0, 128, 50)], [0.0, -0.0, 1.0, -1.0, 4e-7, -6e-7]]).astype(np.float32)
    for x in xs:
        c = oracle.adam8_code_signed(float(x))
        k = c & 0x7F
        assert c & 0x80 == (0x80 if (x < 0 and k > 0) else 0)
        d = np.abs(abs(float(x)) - mag7)
        assert d[k] == d.min() and k == int(np.flatnonzero(d == d.min())[0]), (x, c)
    for x in np.abs(xs):
        k = oracle.adam8_code_unsigned(float(x))
        d = np.abs(float(x) - mag8)
        assert k == int(np.flatnonzero(d == d.min())[0]), (x, k)


def test_ties_go_to_the_smaller_magnitude(oracle):
    mag7, mag8 = (t.astype(np.float64) for t in oracle.adam8_maps())
    seen = 0
    for table, code in ((mag7, oracle.adam8_code_signed), (mag8, oracle.adam8_code_unsigned)):
        for k in range(table.size - 1):
            mid = (table[k] + table[k + 1]) / 2
            if float(np.float32(mid)) != mid:
                continue                                               # midpoint not a float: no tie possible
            seen += 1
            assert code(float(mid)) == k
            if code is oracle.adam8_code_signed and k > 0:
                assert code(-float(mid)) == 0x80 | k
    assert seen > 50


def test_hand_traced_first_step(oracle):
    # beta1 = 0.5, beta2 = 0.75, g = [1, -0.5, 0] from a zero state:
    #   m' = 0.5 g = [0.5, -0.25, 0],  v' = 0.25 g^2 = [0.25, 0.0625, 0]
    #   scales: max|m'| = 0.5, max v' = 0.25;  m'/0.5 = [1, -0.5, 0],  v'/0.25 = [1, 0.25, 0]
    #   signed map near 0.5: decade 1 values 0.1 + 0.9 (j+1)/64: j = 27 -> 0.49375 (off 0.00625),
    #     j = 28 -> 0.5078125 (off 0.0078125): code 64 + 27 = 91, with the sign bit 0x80 | 91 = 219
    #   unsigned map near 0.25: 0.1 + 0.9 (j+1)/128: j = 20 -> 0.24765625 (off 0.00234375),
    #     j = 21 -> 0.2546875 (off 0.0046875): code 128 + 20 = 148
    #   1 -> the top codes 127 / 255, 0 -> 0
    g = np.array([1.0, -0.5, 0.0], np.float32)
    master = np.array([1.0, 1.0, 1.0], np.float32)
    mc, vc, ms, vs = _state(3)
    oracle.adam8_apply(g, master, mc, vc, ms, vs, None, lr=0.5, beta1=0.5, beta2=0.75, eps=2.0 ** -10,
                       weight_decay=0.0, step=1)
    assert mc.tolist() == [127, 219, 0] and vc.tolist() == [255, 148, 0]
    assert ms.tolist() == [0.5] and vs.tolist() == [0.25]


def test_first_step_is_fp32_adam(oracle):
    n = 3 * B + 777
    rng = np.random.Generator(np.random.PCG64(8))
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    th0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    master, params = th0.copy(), np.zeros(n, np.uint16)
    mc, vc, ms, vs = _state(n)
    oracle.adam8_apply(g, master, mc, vc, ms, vs, params, step=1, **HP)
    ref, m, v, pref = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    oracle.adam_apply(g, ref, m, v, pref, step=1, **HP)
    assert np.array_equal(master.view(np.uint32), ref.view(np.uint32)) and np.array_equal(params, pref)
    for b in range(ms.size):
        sl = slice(b * B, min(n, (b + 1) * B))
        assert ms[b] == np.abs(m[sl]).max() and vs[b] == v[sl].max()


@pytest.mark.parametrize("n", [2 * B + 37, 5 * B])
def test_one_magnitude_blocks_stay_exact(oracle, n):
    """|g| constant inside each block (its own value per block and step) with
    one sign pattern for every step: within a block every |m'| and every v'
    is the same, so x = +-1 is stored exactly and 8-bit Adam equals fp32 Adam
    bit for bit at every step.  A wrong block size mixes scales and fails."""
    rng = np.random.Generator(np.random.PCG64(9))
    nb = (n + B - 1) // B
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0).astype(np.float32)
    blk = np.arange(n) // B
    th0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    master, params = th0.copy(), np.zeros(n, np.uint16)
    mc, vc, ms, vs = _state(n)
    ref, m, v, pref = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    for step in range(1, 6):
        mags = (10.0 ** rng.uniform(-4, -2, nb)).astype(np.float32)
        g = sign * mags[blk]
        oracle.adam8_apply(g, master, mc, vc, ms, vs, params, step=step, **HP)
        oracle.adam_apply(g, ref, m, v, pref, step=step, **HP)
        assert np.array_equal(master.view(np.uint32), ref.view(np.uint32)), step
        assert np.array_equal(params, pref)
        assert set(np.unique(mc)) <= {127, 255} and set(np.unique(vc)) == {255}
        dm, dv = _decode(oracle, mc, vc, ms, vs)
        assert np.array_equal(dm.view(np.uint32), m.view(np.uint32)) and np.array_equal(dv, v)


def test_step_is_dequantize_adam_quantize(oracle):
    """From a random quantized state: master and params equal fp32 Adam on
    the dequantized state, each scale is its block's max |m'| (max v'), and
    every new code is the nearest one to m' / scale (v' / scale)."""
    n = 2 * B + 500
    rng = np.random.Generator(np.random.PCG64(10))
    mag7, mag8 = (t.astype(np.float64) for t in oracle.adam8_maps())
    mc = rng.integers(0, 256, n).astype(np.uint8)
    vc = rng.integers(0, 256, n).astype(np.uint8)
    ms = rng.uniform(1e-5, 1e-3, (n + B - 1) // B).astype(np.float32)
    vs = rng.uniform(1e-9, 1e-7, (n + B - 1) // B).astype(np.float32)
    g = (rng.standard_normal(n) * 3e-4).astype(np.float32)
    th0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m_old, v_old = _decode(oracle, mc, vc, ms, vs)
    master, params = th0.copy(), np.zeros(n, np.uint16)
    oracle.adam8_apply(g, master, mc, vc, ms, vs, params, step=7, **HP)
    ref, m, v, pref = th0.copy(), m_old.copy(), v_old.copy(), np.zeros(n, np.uint16)
    oracle.adam_apply(g, ref, m, v, pref, step=7, **HP)
    assert np.array_equal(master.view(np.uint32), ref.view(np.uint32)) and np.array_equal(params, pref)
    blk = np.arange(n) // B
    for b in range(ms.size):
        sl = blk == b
        assert ms[b] == np.abs(m[sl]).max() and vs[b] == v[sl].max()
    xm = (m / ms[blk]).astype(np.float32).astype(np.float64)          # one IEEE fp32 division each
    xv = (v / vs[blk]).astype(np.float32).astype(np.float64)
    dm = np.abs(np.abs(xm)[:, None] - mag7[None, :])
    dv = np.abs(xv[:, None] - mag8[None, :])
    km = np.argmin(dm, axis=1)                                         # first minimum: the smaller magnitude
    assert np.array_equal(mc & 0x7F, km)
    assert np.array_equal(mc >> 7, ((xm < 0) & (km > 0)).astype(np.uint8))
    assert np.array_equal(vc, np.argmin(dv, axis=1))


def test_blocks_are_independent(oracle):
    n = 3 * B
    rng = np.random.Generator(np.random.PCG64(11))
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    th0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    out = []
    for spike in (False, True):
        gg = g.copy()
        if spike:
            gg[B + 5] = 1.0
        master = th0.copy()
        mc, vc, ms, vs = _state(n)
        for step in (1, 2):
            oracle.adam8_apply(gg, master, mc, vc, ms, vs, None, step=step, **HP)
        out.append((mc, vc, ms, vs))
    (a_mc, a_vc, a_ms, a_vs), (b_mc, b_vc, b_ms, b_vs) = out
    for sl in (slice(0, B), slice(2 * B, 3 * B)):
        assert np.array_equal(a_mc[sl], b_mc[sl]) and np.array_equal(a_vc[sl], b_vc[sl])
    assert a_ms[0] == b_ms[0] and a_ms[2] == b_ms[2] and a_ms[1] != b_ms[1]
    assert not np.array_equal(a_mc[B:2 * B], b_mc[B:2 * B])


def _rn32(q: Fraction) -> np.float32:
    """The float32 nearest to the rational q (ties to the even significand),
    found among the neighbours of a first guess by exact distances."""
    f = np.float32(float(q))
    cands = [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
    def key(c):
        return (abs(Fraction(float(c)) - q), int(np.array(c).view(np.uint32)) & 1)
    return min(cands, key=key)


def _nearest(a: np.float32, table) -> int:
    """Index of the table value nearest to a, by exact distances; ties to the smaller."""
    d = [abs(Fraction(float(a)) - Fraction(float(t))) for t in table]
    return d.index(min(d))


def test_normalization_is_the_ieee_quotient(oracle):
    """Two blocks, worked out by hand and checked here in exact rational
    arithmetic, where normalizing by a rounded reciprocal crosses a code
    threshold that the quotient itself does not.  First step from a zero
    state with beta1 = beta2 = 0.5, so m' = g / 2 and v' = fp32(g^2) / 2 are
    known exactly.

    Block 0 (the signed map, m): g = [2 s, 2 x], s = 0x3c0185d6
    (0.0079054441), x = 0x3bd9272f (0.0066269855).  m' = [s, x], scale s.
    The exact x / s = 0.838281239140 lies below 0.838281244040, the midpoint
    of mag7[115] = 0.831250012 and mag7[116] = 0.845312476; rounded once it
    is 0x3f569999 = 0.838281214237, still below: code 115.  fp32(1 / s) =
    0x42fcfd7f = 126.495109558 is 2.1e-8 (relative) above 1 / s, and
    x * fp32(1 / s) rounds to 0x3f56999a = 0.838281273842, above the
    midpoint: a reciprocal-multiply normalization would store code 116.

    Block 1 (the unsigned map, v): g = [ga, gb], ga = 0x3af8485f
    (0.0018942467), gb = 0x3ae79282 (0.0017667564).  v' = fp32(g^2) / 2,
    scale v'[0].  The exact quotient 0.869921888688 lies below
    0.869921892881, the midpoint of mag8[236] and mag8[237]; rounded once it
    is 0x3f5eb333 = 0.869921863079: code 236.  The reciprocal product is
    0x3f5eb334 = 0.869921922684: code 237.
    """
    mag7, mag8 = oracle.adam8_maps()
    f32 = lambda bits: np.array([bits], np.uint32).view(np.float32)[0]
    s, x = f32(0x3C0185D6), f32(0x3BD9272F)
    ga, gb = f32(0x3AF8485F), f32(0x3AE79282)
    n = 2 * B
    g = np.zeros(n, np.float32)
    g[0], g[1] = 2 * s, 2 * x                                          # exact doublings
    g[B], g[B + 1] = ga, gb
    master = np.zeros(n, np.float32)
    mc, vc, ms, vs = _state(n)
    oracle.adam8_apply(g, master, mc, vc, ms, vs, None, lr=1e-3, beta1=0.5, beta2=0.5, eps=1e-8,
                       weight_decay=0.0, step=1)

    # block 0, m: the scale and the code of x / s, all in exact arithmetic
    assert ms[0] == s
    q = Fraction(float(x)) / Fraction(float(s))
    k = _nearest(_rn32(q), mag7)
    mid = (Fraction(float(mag7[115])) + Fraction(float(mag7[116]))) / 2
    assert k == 115 and q < mid and Fraction(float(_rn32(q))) <= mid
    rcp = _rn32(Fraction(1) / Fraction(float(s)))
    assert _nearest(_rn32(Fraction(float(x)) * Fraction(float(rcp))), mag7) == 116   # the pin discriminates
    assert mc[0] == 127 and mc[1] == 115

    # block 1, v: v' = fp32(g^2) / 2 (the halving is exact)
    va = _rn32(Fraction(float(ga)) ** 2) / np.float32(2)
    vb = _rn32(Fraction(float(gb)) ** 2) / np.float32(2)
    assert vs[1] == va
    q = Fraction(float(vb)) / Fraction(float(va))
    mid = (Fraction(float(mag8[236])) + Fraction(float(mag8[237]))) / 2
    assert _nearest(_rn32(q), mag8) == 236 and q < mid
    rcp = _rn32(Fraction(1) / Fraction(float(va)))
    assert _nearest(_rn32(Fraction(float(vb)) * Fraction(float(rcp))), mag8) == 237
    assert vc[B] == 255 and vc[B + 1] == 236


def test_subnormal_scales(oracle):
    """A block whose moments decayed below 2^-126: the quotient m' / scale is
    still formed (a subnormal divided by a subnormal), so the block maximum
    keeps the top code and every other element the code nearest to its exact
    quotient rounded once -- checked in rational arithmetic; the stored
    scale is the block max."""
    mag7, mag8 = oracle.adam8_maps()
    rng = np.random.Generator(np.random.PCG64(12))
    n = B
    mc = rng.integers(0, 256, n).astype(np.uint8)
    vc = rng.integers(0, 256, n).astype(np.uint8)
    mc[:10] = 0                                                       # zero moments stay zero
    vc[:10] = 0
    mc[10], vc[10] = 0x7F, 0xFF                                       # one element at the block max
    ms = np.array([1e-39], np.float32)                                # subnormal scales
    vs = np.array([1e-39], np.float32)
    m_old, v_old = _decode(oracle, mc, vc, ms, vs)
    g = np.zeros(n, np.float32)
    master = np.full(n, 0.5, np.float32)
    oracle.adam8_apply(g, master, mc, vc, ms, vs, None, step=3, **HP)
    m_new = np.float32(HP["beta1"]) * m_old                           # g = 0: m' = b1 m, v' = b2 v
    v_new = np.float32(HP["beta2"]) * v_old
    assert ms[0] == np.abs(m_new).max() and vs[0] == v_new.max()
    assert mc[10] == 0x7F and vc[10] == 0xFF
    sm, sv = Fraction(float(ms[0])), Fraction(float(vs[0]))
    for j in range(0, n, 7):
        km = _nearest(_rn32(Fraction(float(abs(m_new[j]))) / sm), mag7)
        want_m = (0x80 | km) if (m_new[j] < 0 and km > 0) else km
        assert mc[j] == want_m, j
        assert vc[j] == _nearest(_rn32(Fraction(float(v_new[j])) / sv), mag8), j
