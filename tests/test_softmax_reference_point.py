"""The attention kernel's online softmax keeps a reference point m per row
that only guards against overflow: a unit of 128 keys is weighted by
2^(s * scale - m) with m taken on the row's first unit with a finite score and
moved afterwards only by more than 2^8 on such a first unit, or when a unit's
sum of weights passes 2^64 (or is not finite), in which case that unit is
redone with the unit's maximum.  P is rounded to bf16 for the
P.V product, the row sum and O accumulate in fp32, and O / l and
m + log2(l) come out at the end.

The exactness rests on the identity sum_j 2^(x_j - m) v_j / sum_j 2^(x_j - m) =
the softmax-weighted mean of v for every finite m (FlashAttention's blockwise
rescaling, the online-softmax step behind the sglang article's prefill path),
and on fp32 / bf16 having the exponent range for weights up to 2^64 and sums
of them.  This file restates the scheme's arithmetic in numpy (a model of the
kernel's per-row steps, not the oracle) and checks it against float64
softmax on score sequences that stress the reference point: scores rising
slowly (56 in all, under the redo threshold) and fast (90 per unit, a redo
per unit), one spike far above the rest, falling scores, equal scores, and
fully masked leading units.
"""
import numpy as np
import pytest

UNIT = 128
RESCALE_LOG2 = 8.0
REDO_ABOVE = np.float32(2.0 ** 64)


def bf16(x):
    """Round float32 to bfloat16 (nearest even) and back."""
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(x), x, out)


def kernel_row(s, v, scale):
    """One query row through the kernel's steps: s (keys,) float32 scores
    with -inf for masked keys, v (keys, d) values."""
    m = np.float32(-np.inf)
    l = np.float32(0.0)
    o = np.zeros(v.shape[1], dtype=np.float32)
    redos = 0
    for u0 in range(0, len(s), UNIT):
        su = s[u0:u0 + UNIT].astype(np.float32)
        vu = v[u0:u0 + UNIT].astype(np.float32)
        m_prev = m
        for rnd in range(2):
            if rnd == 1 or m == -np.inf:
                mt = np.float32(np.max(su)) * np.float32(scale)
                m_new = np.float32(max(m, mt))
                if rnd == 1 or m == -np.inf or m_new > m + RESCALE_LOG2:
                    m = m_new
            nbase = np.float32(0.0) if m == -np.inf else -m
            with np.errstate(over="ignore", invalid="ignore"):
                x = su * np.float32(scale) + nbase
                p = np.exp2(x).astype(np.float32)
                ls = np.float32(p.sum(dtype=np.float32))
            if ls <= REDO_ABOVE:
                break
            redos += 1
        if m == m_prev:
            alpha = np.float32(1.0)
        elif m_prev == -np.inf:
            alpha = np.float32(0.0)
        else:
            alpha = np.float32(np.exp2(m_prev - m))
        l = np.float32(l * alpha + ls)
        o = (o * alpha + bf16(p) @ vu).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse2 = m + np.log2(l)
        return o / l, lse2, redos


def exact_row(s, v, scale):
    x = s.astype(np.float64) * scale
    mx = np.max(x)
    w = np.exp2(x - mx)
    return (w @ v.astype(np.float64)) / w.sum(), mx + np.log2(w.sum())


def scores(kind, n, rng):
    base = rng.standard_normal(n).astype(np.float32)
    u = np.arange(n) // UNIT
    if kind == "rising_under":   # each unit 7 log2 units above the last: 56 in all
        return base + 7.0 * u
    if kind == "rising_over":    # each unit 90 above the last: a redo per unit
        return base + 90.0 * u
    if kind == "spike":
        s = base.copy()
        s[n // 2 + 7] = 300.0
        return s
    if kind == "falling":
        return base - 50.0 * u
    if kind == "equal":
        return np.full(n, 3.0, dtype=np.float32)
    if kind == "masked_first":
        s = base.copy()
        s[:2 * UNIT] = -np.inf
        return s
    raise ValueError(kind)


KINDS = ["rising_under", "rising_over", "spike", "falling", "equal", "masked_first"]


@pytest.mark.parametrize("kind", KINDS)
def test_reference_point_keeps_softmax_exact(kind):
    rng = np.random.default_rng(11 + KINDS.index(kind))
    n, d = 8 * UNIT + 37, 64
    s = scores(kind, n, rng)
    v = bf16(rng.standard_normal((n, d)).astype(np.float32))
    o, lse2, redos = kernel_row(s, v, 1.0)
    want, want_lse2 = exact_row(s, v, 1.0)
    assert np.isfinite(o).all() and np.isfinite(lse2)
    # P in bf16: the weights carry about 2^-9 relative error each
    assert np.abs(o - want).max() <= 2e-2
    assert abs(lse2 - want_lse2) <= 1e-3 * max(1.0, abs(want_lse2))
    if kind == "rising_over":
        assert redos >= 7      # the scheme did take its second pass
    if kind in ("rising_under", "falling", "equal"):
        assert redos == 0      # and did not where no unit's sum passes 2^64


def test_weights_near_the_threshold_stay_finite():
    """Every unit's scores sit 56 above the first unit's maximum for 200
    units: weights near 2^56, unit sums near 2^63 (under the redo threshold),
    l near 2^71 and O of the same order stay finite in fp32 without a second
    pass."""
    rng = np.random.default_rng(3)
    n, d = 200 * UNIT, 16
    s = np.full(n, 56.0, dtype=np.float32)
    s[:UNIT] = 0.0
    v = bf16(rng.standard_normal((n, d)).astype(np.float32))
    o, lse2, redos = kernel_row(s, v, 1.0)
    want, want_lse2 = exact_row(s, v, 1.0)
    assert redos == 0
    assert np.isfinite(o).all()
    assert np.abs(o - want).max() <= 2e-2
    assert abs(lse2 - want_lse2) <= 1e-3 * abs(want_lse2)


def test_the_model_catches_a_missing_second_pass():
    """The same steps without the second pass overflow on the spike: the
    checks above would fail for a scheme that never redoes a unit."""
    rng = np.random.default_rng(7)
    n, d = 4 * UNIT, 8
    s = scores("spike", n, rng)
    v = bf16(rng.standard_normal((n, d)).astype(np.float32))
    global REDO_ABOVE
    saved = REDO_ABOVE
    try:
        REDO_ABOVE = np.float32(np.inf)  # never redo
        o, lse2, redos = kernel_row(s, v, 1.0)
    finally:
        REDO_ABOVE = saved
    assert redos == 0
    assert not (np.isfinite(o).all() and np.isfinite(lse2))
