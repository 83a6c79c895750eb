"""Pins for oracle.quantize: closed forms, special cases, an explicit Hadamard
matrix, statistics of stochastic rounding, and transpose consistency."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import quantize as Q

rng = np.random.default_rng(42)


def test_amax_exact_and_order_free():
    x = rng.standard_normal((37, 53)).astype(np.float32)
    x[5, 7] = -9.25
    assert Q.amax(x) == np.float32(9.25)
    assert Q.amax(x[::-1, ::-1]) == Q.amax(x)
    assert Q.amax(np.array([-0.0, 0.0], np.float32)) == 0.0
    assert Q.amax(np.zeros((0, 4), np.float32)) == 0.0
    assert float(Q.amax(x)) == max(abs(float(v)) for v in x.ravel())


def test_fp8_row_col_copies_are_transposes():
    x = rng.standard_normal((64, 48)).astype(np.float32)
    q_row, q_col, a, si = Q.fp8_quantize(x, np.float32(30.0), "e5m2")
    np.testing.assert_array_equal(q_col, q_row.T)
    assert si == np.float32(1) / np.float32(30)
    # dequantization error bounded by half an E5M2 ulp (relative 2**-3) for normal values
    deq = Q.fp8_dequant(q_row, si, "e5m2")
    big = np.abs(x) > 2.0 ** -10
    assert np.all(np.abs(deq[big] - x[big]) <= np.abs(x[big]) * 2.0 ** -3 + 1e-12)


# ---- MXFP8 ----------------------------------------------------------------------

def test_mx_power_of_two_block():
    for k in (-20, 0, 3, 100):
        z = np.full((1, 32), 2.0 ** k, np.float32)
        q, s = Q.mxfp8_quantize(z)
        assert int(s[0, 0]) == k - 8 + 127
        assert np.all(q == 0x78)            # 2**8 in E4M3


def test_mx_spike_hits_448_and_saturation():
    z = np.zeros((1, 32), np.float32)
    z[0, 3] = 1.75 * 2.0 ** 5
    z[0, 9] = -1.0
    q, s = Q.mxfp8_quantize(z)
    assert int(s[0, 0]) == 5 - 8 + 127
    assert q[0, 3] == 0x7E
    z[0, 3] = 1.99 * 2.0 ** 5                # 1.99 * 2**8 after scaling -> saturates to 448
    q, _ = Q.mxfp8_quantize(z)
    assert q[0, 3] == 0x7E


def test_mx_zero_block_and_clamp():
    q, s = Q.mxfp8_quantize(np.zeros((2, 64), np.float32))
    assert np.all(s == 0) and np.all(q == 0)
    tiny = np.full((1, 32), 2.0 ** -140, np.float32)   # floor(log2) - 8 = -148 -> clamp -127
    q, s = Q.mxfp8_quantize(tiny)
    assert int(s[0, 0]) == 0
    # x * 2**127 = 2**-13 is below E4M3's smallest subnormal (2**-9): quantizes to zero
    assert np.all(q == 0)


def test_mx_dequant_reproduces_representable_values():
    # blocks whose elements are E4M3 values times 2**E, with the block max in [256, 448]
    R, C = 8, 64
    codes = rng.integers(0, 0x7F, size=(R, C))
    codes[:, ::32] = rng.integers(0x78, 0x7F, size=(R, C // 32))   # exponent field 15 -> [256, 448]
    signs = rng.integers(0, 2, size=(R, C)) << 7
    E = rng.integers(-100, 100, size=(R, C // 32))
    vals = F.decode(codes | signs, "e4m3") * np.exp2(np.repeat(E, 32, axis=1))
    z = vals.astype(np.float32)
    assert np.all(z.astype(np.float64) == vals)
    q, s = Q.mxfp8_quantize(z)
    np.testing.assert_array_equal(s.astype(np.int64) - 127, E)
    np.testing.assert_array_equal(Q.mxfp8_dequant(q, s), vals)


# ---- RHT ---------------------------------------------------------------------------

def _hadamard16():
    i = np.arange(16)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


def test_rht_matches_explicit_matrix():
    signs = 0b1010_0110_0011_1001
    H = _hadamard16()
    D = np.diag([-1.0 if (signs >> j) & 1 else 1.0 for j in range(16)])
    z = rng.standard_normal((5, 64)).astype(np.float32)
    y = Q.rht16(z, signs)
    ref = (z.astype(np.float64).reshape(-1, 16) @ (0.25 * H @ D).T).reshape(5, 64)
    # four fp32 rounding stages of sums of up to 16 terms
    assert np.max(np.abs(y - ref)) <= 1e-5 * np.max(np.abs(ref))
    # small integers: every butterfly is exact, so the result is exact
    zi = rng.integers(-50, 50, size=(3, 32)).astype(np.float32)
    yi = Q.rht16(zi, signs)
    refi = (zi.astype(np.float64).reshape(-1, 16) @ (0.25 * H @ D).T).reshape(3, 32)
    np.testing.assert_array_equal(yi, refi)


def test_rht_one_hot_inverse_and_dot_products():
    for j in range(16):
        e = np.zeros((1, 16), np.float32)
        e[0, j] = 1.0
        y = Q.rht16(e, 0)
        assert np.all(np.abs(y) == 0.25)
    signs = 0x5A3C
    x = rng.standard_normal((4, 48)).astype(np.float32)
    y = Q.rht16(x, signs)
    back = Q.rht16(y, 0) * 4.0                       # 1/4 H (1/4 H D x) * 4 = D x / ... = D x
    dvec = np.array([-1.0 if (signs >> j) & 1 else 1.0 for j in range(16)], np.float32)
    rec = (back.reshape(-1, 16) * dvec).reshape(x.shape) / 4.0
    np.testing.assert_allclose(rec, x, rtol=0, atol=1e-6 * np.abs(x).max())
    a = rng.standard_normal((1, 4096)).astype(np.float32)
    b = rng.standard_normal((1, 4096)).astype(np.float32)
    lhs = np.dot(Q.rht16(a, signs)[0].astype(np.float64), Q.rht16(b, signs)[0].astype(np.float64))
    rhs = np.dot(a[0].astype(np.float64), b[0].astype(np.float64))
    assert abs(lhs - rhs) <= 1e-4 * np.sqrt(4096)


# ---- NVFP4 ----------------------------------------------------------------------------

def test_nvfp4_global_scales():
    s, d = Q.nvfp4_global(np.float32(2688.0))
    assert s == 1.0 and d == 1.0
    s, d = Q.nvfp4_global(np.float32(0.0))
    assert s == 1.0 and d == 1.0
    s, d = Q.nvfp4_global(np.float32(1e-45))
    assert s == 1.0
    s, d = Q.nvfp4_global(np.float32(6.0))
    assert s == 448.0 and d == np.float32(1) / np.float32(448)


def test_nvfp4_block_at_tensor_amax_scales_to_448_and_6():
    z = rng.standard_normal((4, 64)).astype(np.float32)
    A = Q.amax(z)
    q, s, sd = Q.nvfp4_quantize(z, A)
    r, c = np.unravel_index(np.argmax(np.abs(z)), z.shape)
    assert s[r, c // 16] == 0x7E                  # 448
    assert q[r, c] & 0x7 == 0x7                   # |6|
    assert (q[r, c] >> 3) == (1 if z[r, c] < 0 else 0)


def test_nvfp4_uniform_block_all_six():
    for c in (0.3, 1.0, 7.7, 123.0):
        z = np.full((1, 16), c, np.float32)
        z = np.concatenate([z, np.full((1, 16), 1000.0, np.float32)], axis=1)  # tensor amax elsewhere
        q, s, _ = Q.nvfp4_quantize(z, Q.amax(z))
        assert F.decode_ue4m3(s[:, :1])[0, 0] >= 2.0 ** -6        # normal UE4M3
        assert np.all(q[0, :16] == 0x7)


def test_nvfp4_zero_tensor_and_zero_scale_block():
    q, s, sd = Q.nvfp4_quantize(np.zeros((2, 32), np.float32), 0.0)
    assert np.all(q == 0) and np.all(s == 0) and sd == 1.0
    z = np.zeros((1, 32), np.float32)
    z[0, 0] = 1.0
    z[0, 20] = -1e-9                               # block scale rounds to 0 -> r = 0 -> signed zero
    q, s, _ = Q.nvfp4_quantize(z, Q.amax(z))
    assert s[0, 1] == 0 and q[0, 20] == 0x8 and q[0, 21] == 0x0


def test_nvfp4_2d_transpose_consistency():
    w = (rng.standard_normal((48, 64)) * 0.02).astype(np.float32)
    A = Q.amax(w)
    q_r, s_r, _ = Q.nvfp4_quantize(w, A, block2d=True)
    q_c, s_c, _ = Q.nvfp4_quantize(np.ascontiguousarray(w.T), A, block2d=True)
    np.testing.assert_array_equal(q_c, q_r.T)
    # each 16x16 tile has one scale, replicated along both copies
    tile_r = s_r.reshape(3, 16, 4)
    assert np.all(tile_r == tile_r[:, :1, :])
    np.testing.assert_array_equal(s_c.reshape(4, 16, 3)[:, 0, :], tile_r[:, 0, :].T)


def test_nvfp4_dequant_error_bound():
    z = rng.standard_normal((32, 256)).astype(np.float32)
    A = Q.amax(z)
    q, s, sd = Q.nvfp4_quantize(z, A)
    deq = Q.nvfp4_dequant(q, s, sd)
    # element error <= half the E2M1 spacing at the block's scale (spacing <= 2 * unit), plus scale rounding
    unit = F.decode_ue4m3(s) * float(sd)
    bound = np.repeat(unit, 16, axis=1) * 1.0 + 1e-12
    assert np.all(np.abs(deq - z) <= bound)
    assert Q.amax(deq) <= A * (1 + 2.0 ** -3)


def test_pack_unpack_nibble_order():
    c = np.array([[1, 2, 3, 15, 0, 8]], np.uint8)
    p = Q.pack_e2m1(c)
    assert list(p[0]) == [0x21, 0xF3, 0x80]
    np.testing.assert_array_equal(Q.unpack_e2m1(p), c)


# ---- stochastic rounding ----------------------------------------------------------------

def test_sr_exact_values_never_move_and_neighbours_only():
    grid = np.concatenate([Q.E2M1_GRID, -Q.E2M1_GRID]).astype(np.float32)
    words = rng.integers(0, 1 << 16, size=grid.size, dtype=np.uint64).astype(np.uint32)
    np.testing.assert_array_equal(Q.e2m1_round_stochastic(grid, words), F.encode(grid, "e2m1"))
    v = rng.uniform(-7, 7, size=4096).astype(np.float32)
    words = rng.integers(0, 1 << 16, size=v.size, dtype=np.uint64).astype(np.uint32)
    got = F.decode(Q.e2m1_round_stochastic(v, words), "e2m1")
    a = np.minimum(np.abs(v), 6.0)
    lo = Q.E2M1_GRID[np.clip(np.searchsorted(Q.E2M1_GRID, a, side="right") - 1, 0, 7)]
    hi = Q.E2M1_GRID[np.clip(np.searchsorted(Q.E2M1_GRID, a, side="left"), 0, 7)]
    assert np.all((np.abs(got) == lo) | (np.abs(got) == hi))
    assert np.all(np.sign(got)[got != 0] == np.sign(v)[got != 0])


def test_sr_threshold_rule():
    # frac = 0.25 at v = 2.25 (between 2 and 3): up iff R + 16384 >= 65536, i.e. R >= 49152
    v = np.full(4, 2.25, np.float32)
    w = np.array([0, 49151, 49152, 0xFFFF], np.uint32)
    got = F.decode(Q.e2m1_round_stochastic(v, w), "e2m1")
    assert list(got) == [2.0, 2.0, 3.0, 3.0]
    # fractions below 2**-16 never round up; frac = 2**-16 exactly only with R = 0xFFFF
    v = np.full(2, 4.0 + 2.0 ** -20, np.float32)
    got = F.decode(Q.e2m1_round_stochastic(v, np.array([0, 0xFFFF], np.uint32)), "e2m1")
    assert list(got) == [4.0, 4.0]
    v = np.full(2, 4.0 + 2.0 ** -15, np.float32)
    got = F.decode(Q.e2m1_round_stochastic(v, np.array([0xFFFE, 0xFFFF], np.uint32)), "e2m1")
    assert list(got) == [4.0, 6.0]
    # negative values keep their sign, also when they round to zero
    got = Q.e2m1_round_stochastic(np.array([-0.1, -0.1], np.float32), np.array([0, 0xFFFF], np.uint32))
    assert list(got) == [0x8, 0x9]


@pytest.mark.parametrize("v", [0.0123, 0.3, 0.77, 1.1, 2.9, 3.01, 4.4, 5.999])
def test_sr_probability_over_all_random_values(v):
    # over every 16-bit R the round-up count is frac * 2**16 truncated: unbiased to 2**-16
    v32 = np.float32(v)
    got = F.decode(Q.e2m1_round_stochastic(np.full(1 << 16, v32), np.arange(1 << 16, dtype=np.uint32)), "e2m1")
    lo = Q.E2M1_GRID[np.searchsorted(Q.E2M1_GRID, v32, side="right") - 1]
    hi = Q.E2M1_GRID[np.searchsorted(Q.E2M1_GRID, v32, side="right")]
    frac = (float(v32) - lo) / (hi - lo)
    ups = int(np.sum(got == hi))
    assert np.all((got == hi) | (got == lo))
    assert 0 <= frac * 65536 - ups < 1


def test_sr_rand16_split_of_a_word():
    # P = (w[23:16] << 8) | w[7:0], Q = (w[31:24] << 8) | w[15:8]; positions take P, rev(P), Q, rev(Q)
    w = np.array([0x12345678] * 4 + [0x000000FF] * 4 + [0x80000000] * 4, np.uint32)
    pos = np.tile(np.arange(4), 3)
    got = list(Q.sr_rand16(w, pos))
    assert got == [0x3478, 0x1E2C, 0x1256, 0x6A48,
                   0x00FF, 0xFF00, 0x0000, 0x0000,
                   0x0000, 0x0000, 0x8000, 0x0001]


@pytest.mark.parametrize("v", [0.1, 0.8, 1.3, 2.6, 3.3, 4.9, 5.99])
def test_sr_unbiased(v):
    n = 1 << 18
    from oracle.philox import element_words
    words = element_words(n, 0, seed=977, copy_id=0, offset=int(v * 100))
    r16 = Q.sr_rand16(words, np.arange(n) & 3)
    got = F.decode(Q.e2m1_round_stochastic(np.full(n, v, np.float32), r16), "e2m1")
    lo = Q.E2M1_GRID[np.searchsorted(Q.E2M1_GRID, v) - 1]
    hi = Q.E2M1_GRID[np.searchsorted(Q.E2M1_GRID, v)]
    p = (v - lo) / (hi - lo)
    sigma = (hi - lo) * np.sqrt(p * (1 - p) / n)
    assert abs(got.mean() - np.float32(v)) < 4 * sigma + (hi - lo) * 2.0 ** -16
    for k in range(4):          # every position of a group is unbiased on its own
        sub = got[k::4]
        assert abs(sub.mean() - np.float32(v)) < 4 * sigma * 2 + (hi - lo) * 2.0 ** -16


# ---- stochastic rounding: fairness of the reading of a group's random word ----------------
#
# The rule reads one 32-bit word per group of four elements and gives each position a 16-bit
# value R.  What makes that a fair stochastic rounding is pinned here on the mathematics, with
# sr_rand16 as a black box: (1) the word's bits split into two disjoint 16-bit sets, positions
# 0 / 1 reading one and 2 / 3 the other (so the two halves of a group are independent); (2)
# over every setting of its 16 bits each position draws every 16-bit value exactly once
# (uniform R, hence the unbiased rounding probability floor(frac * 2**16) / 2**16); (3) the two
# positions that read the same bits round up nearly independently; (4) a stochastically rounded
# dot product has the variance of independent rounding.


def _rand16_dependencies():
    """For each group position, the set of word bits whose flip changes its R (black-box probe)."""
    base = rng.integers(0, 1 << 32, size=64, dtype=np.uint64).astype(np.uint32)
    deps = [set() for _ in range(4)]
    for pos in range(4):
        r0 = Q.sr_rand16(base, np.full(base.size, pos))
        for b in range(32):
            r1 = Q.sr_rand16(base ^ np.uint32(1 << b), np.full(base.size, pos))
            if np.any(r1 != r0):
                deps[pos].add(b)
    return deps


def test_sr_group_word_splits_into_two_disjoint_halves():
    deps = _rand16_dependencies()
    assert deps[0] == deps[1] and deps[2] == deps[3]
    assert len(deps[0]) == 16 and len(deps[2]) == 16
    assert deps[0].isdisjoint(deps[2]) and deps[0] | deps[2] == set(range(32))


def _words_over_bits(bits, fixed):
    """All 2**16 words that take every setting of ``bits`` (16 positions) with the rest from ``fixed``."""
    bits = sorted(bits)
    v = np.arange(1 << 16, dtype=np.uint64)
    w = np.full(v.size, fixed, dtype=np.uint64)
    for i, b in enumerate(bits):
        w &= ~np.uint64(1 << b)
        w |= ((v >> np.uint64(i)) & np.uint64(1)) << np.uint64(b)
    return w.astype(np.uint32)


def test_sr_each_position_draws_every_16_bit_value_once():
    # exhaustive over the 16 bits a half reads (the other half fixed at several random values):
    # positions reading those bits see each R in [0, 2**16) exactly once, the others do not move
    deps = _rand16_dependencies()
    for fixed in rng.integers(0, 1 << 32, size=3, dtype=np.uint64):
        for half, (mine, other) in enumerate(((0, 2), (2, 0))):
            w = _words_over_bits(deps[mine], int(fixed))
            for pos in (mine, mine + 1):
                r = Q.sr_rand16(w, np.full(w.size, pos))
                np.testing.assert_array_equal(np.sort(r), np.arange(1 << 16, dtype=np.uint32))
            for pos in (other, other + 1):
                r = Q.sr_rand16(w, np.full(w.size, pos))
                assert np.all(r == r[0])


def _up(r16, frac):
    """Round-up event of the rule at fraction ``frac`` for random values r16."""
    return (r16.astype(np.float64) + np.floor(frac * 65536.0)) >= 65536.0


@pytest.mark.parametrize("half", [0, 2])
def test_sr_positions_sharing_bits_round_up_nearly_independently(half):
    # exact over all 2**16 settings of the shared bits: |corr(up_a, up_b)| <= 1e-3 for every
    # pair of fractions 0.1 .. 0.9 (measured worst 5.7e-4; dyadic fractions give exactly 0)
    deps = _rand16_dependencies()
    w = _words_over_bits(deps[half], 0x5A5A5A5A)
    ra = Q.sr_rand16(w, np.full(w.size, half))
    rb = Q.sr_rand16(w, np.full(w.size, half + 1))
    fracs = [i / 10 for i in range(1, 10)]
    for fa in fracs:
        for fb in fracs:
            ua, ub = _up(ra, fa), _up(rb, fb)
            pa, pb, pab = ua.mean(), ub.mean(), (ua & ub).mean()
            corr = (pab - pa * pb) / np.sqrt(pa * (1 - pa) * pb * (1 - pb))
            assert abs(corr) <= 1e-3, (fa, fb, corr)
    for f in (0.25, 0.5, 0.75):           # dyadic fractions: exactly independent
        ua, ub = _up(ra, f), _up(rb, f)
        assert (ua & ub).mean() == ua.mean() * ub.mean()


def test_sr_dot_product_has_the_variance_of_independent_rounding():
    # sum over M = 2048 elements whose group positions pair equal values ([a, a, b, b]), so a
    # correlation between the positions that share bits would show in the variance; T trials
    # draw fresh words through the counter (offset); bar: 4 standard errors of a variance
    from oracle.philox import element_words
    M, T = 2048, 3000
    ab = rng.uniform(0.05, 5.95, size=M // 2).astype(np.float32)
    v = np.repeat(ab, 2)
    lo = Q.E2M1_GRID[np.searchsorted(Q.E2M1_GRID, v, side="right") - 1].astype(np.float64)
    hi = Q.E2M1_GRID[np.searchsorted(Q.E2M1_GRID, v, side="right")].astype(np.float64)
    frac = (v.astype(np.float64) - lo) / (hi - lo)
    p = np.floor(frac * 65536.0) / 65536.0
    var_indep = float(np.sum((hi - lo) ** 2 * p * (1 - p)))
    mean_exact = float(np.sum(lo + (hi - lo) * p))
    pos = np.arange(M) & 3
    sums = np.empty(T)
    for t in range(T):
        r16 = Q.sr_rand16(element_words(M, 0, seed=31337, copy_id=0, offset=t), pos)
        sums[t] = F.decode(Q.e2m1_round_stochastic(v, r16), "e2m1").sum()
    var = sums.var(ddof=1)
    assert abs(var / var_indep - 1.0) <= 4.0 * np.sqrt(2.0 / (T - 1)), (var, var_indep)
    assert abs(sums.mean() - mean_exact) <= 4.0 * np.sqrt(var_indep / T)


def test_nvfp4_sr_uses_copy_indexed_words():
    z = rng.standard_normal((32, 64)).astype(np.float32)
    A = Q.amax(z)
    sr = dict(seed=11, copy_id=1, offset=5, row0=0, cols=64)
    q_full, _, _ = Q.nvfp4_quantize(z, A, sr=sr)
    sr2 = dict(sr, row0=8)
    q_part, _, _ = Q.nvfp4_quantize(z[8:16], A, sr=sr2)
    np.testing.assert_array_equal(q_full[8:16], q_part)
    q_rn, _, _ = Q.nvfp4_quantize(z, A)
    assert np.mean(q_rn != q_full) > 0.05       # SR really differs from RN on random data


def test_dbias_closed_forms_and_loops():
    # ones -> number of rows; column j of value j * (row index) -> j * R (R - 1) / 2
    R, C = 37, 5
    np.testing.assert_array_equal(Q.dbias(np.ones((R, C), np.float32)), np.full(C, float(R)))
    t = np.arange(R)[:, None] * np.arange(C)[None, :]
    np.testing.assert_array_equal(Q.dbias(t), np.arange(C) * R * (R - 1) / 2)
    x = rng.standard_normal((9, 4)).astype(np.float32)
    brute = [sum(float(x[r, c]) for r in range(9)) for c in range(4)]
    np.testing.assert_allclose(Q.dbias(x), brute, rtol=0, atol=1e-12)
