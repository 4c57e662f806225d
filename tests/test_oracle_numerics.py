"""Pins of the oracle's number handling, imatrix statistic, importance weights and anchor.

Each test ties the oracle to something other than itself: numpy's IEEE conversions and float32
arithmetic (a library routine), exact histograms, closed forms, or a higher-precision sum.
"""
from fractions import Fraction

import numpy as np
import pytest

from ggml_iq_codebook_accumulate_b300 import synth


# --- fp16 conversion: IEEE binary16 round-to-nearest-even, pinned by numpy's conversion -----------

def test_half_from_float_matches_numpy(orc):
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001,
                  2.0 ** -26, 6.1035156e-05, 6.0975552e-05, np.inf, -np.inf], np.float32),
    ]).astype(np.float32)
    # exact ties between neighbouring halves (round half to even)
    h = np.arange(0x0001, 0x7BFF, 7, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float32)
    hi = (h + 1).view(np.float16).astype(np.float32)
    vals = np.concatenate([vals, (lo + hi) / 2, -(lo + hi) / 2]).astype(np.float32)
    ours = orc.half_from_float(vals)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_float_from_half_all_patterns(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.float_from_half(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


# --- imatrix accumulation ----------------------------------------------------------------------

def _set_hist(ids, E):
    c = np.zeros(E, np.int64)
    for row in ids:
        for e in set(int(v) for v in row if 0 <= v < E):
            c[e] += 1
    return c


def test_imatrix_counts_are_the_routed_histogram(orc):
    ids = synth.router(3000, 16, 4, idle=3, seed=5)
    x = synth.activations(3000, 256, seed=6)
    _, counts, st = orc.imatrix_accumulate(x, ids, 16, rows_per_chunk=1024)
    assert st == 0
    assert np.array_equal(counts, _set_hist(ids, 16))
    assert counts[-3:].sum() == 0 or (counts == 0).sum() >= 3


def test_imatrix_all_ones_gives_counts(orc):
    ids = synth.router(2500, 12, 3, idle=2, seed=7)
    x = np.ones((2500, 256), np.float32)
    s2, counts, _ = orc.imatrix_accumulate(x, ids, 12, rows_per_chunk=1024)
    assert np.array_equal(s2, np.repeat(counts.astype(np.float32)[:, None], 256, axis=1))


def f32_nearest(q: Fraction) -> np.float32:
    """The float32 nearest to the rational q, ties to even, found by exact comparison of the
    neighbours of a first guess (float() of a Fraction is correctly rounded to fp64; the fp64 ->
    fp32 step can be off by one ulp, which the neighbour check corrects)."""
    c = np.float32(float(q))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    return min(cands, key=lambda v: (abs(Fraction(float(v)) - q), int(np.float32(v).view(np.uint32)) & 1))


def running_sum_exact(col):
    """partial = fl(partial + fl(x*x)) for each x in order, with exact rational arithmetic: the
    square is correctly rounded to fp32 once, and the addition once more (two roundings a step)."""
    acc = np.float32(0.0)
    for x in col:
        sq = f32_nearest(Fraction(float(x)) ** 2)
        acc = f32_nearest(Fraction(float(acc)) + Fraction(float(sq)))
    return acc


def fused_running_sum_exact(col):
    """The other reading, partial = fl(partial + x*x) with the exact square and one rounding a step
    (a fused multiply-add), for telling the two apart."""
    acc = np.float32(0.0)
    for x in col:
        acc = f32_nearest(Fraction(float(acc)) + Fraction(float(x)) ** 2)
    return acc


def bounded_bf16_acts(tokens, cols, seed):
    """bf16-valued activations with 2^-4 <= |x| < 2^4.  A square then has at most 16 significant
    bits and lies in [2^-8, 2^8), so fl(x*x) = x*x exactly; a running sum of up to 1,024 of them
    stays below 2^18 with its lowest bit at or above 2^-31, so every step partial + x*x is exact in
    fp64 (at most 50 significant bits) and one fp64 -> fp32 rounding is the single correct rounding
    of the addition."""
    x = synth.activations(tokens, cols, seed=seed)
    mag = np.clip(np.abs(x), 2.0 ** -4, 2.0 ** 4 * (1 - 2.0 ** -9))
    x = np.where(x < 0, -mag, mag).astype(np.float32)
    return synth.as_dtype(x, "bf16")[1]


def running_sum_f64(rows):
    """Vectorised running sum over axis 0, one fp32 rounding per step from an exact fp64 step
    (valid for the bounded inputs above, whose squares are exact in fp32)."""
    acc = np.zeros(rows.shape[1], np.float32)
    for r in rows:
        acc = (acc.astype(np.float64) + r.astype(np.float64) ** 2).astype(np.float32)
    return acc


def test_imatrix_square_then_add_exact_small(orc):
    """Values spanning 1e-22 .. 1e4, fp32-valued, some squares subnormal: each step of the running
    sum rounds the square to fp32, then rounds the addition (exact rational reference)."""
    rng = np.random.default_rng(19)
    x = (rng.standard_normal((48, 40)) * 10.0 ** rng.integers(-22, 4, (48, 40))).astype(np.float32)
    x[5, 0] = np.float32(3e-20)            # square 9e-40: subnormal in fp32
    x[:3, 4] = np.float32(1e-23)           # squares far below the fp32 range, then larger terms
    s2, counts, _ = orc.imatrix_accumulate(x, np.zeros((48, 1), np.int32), 1, rows_per_chunk=1024)
    assert counts[0] == 48
    ref = np.array([running_sum_exact(x[:, j]) for j in range(40)], np.float32)
    assert np.array_equal(s2[0].view(np.uint32), ref.view(np.uint32))
    # the single-rounding reading (fused multiply-add) differs in some columns, so this pin tells
    # the two readings apart
    fused = np.array([fused_running_sum_exact(x[:, j]) for j in range(40)], np.float32)
    assert not np.array_equal(s2[0].view(np.uint32), fused.view(np.uint32))


def test_imatrix_single_expert_is_sequential_column_sum(orc):
    """One expert, top-1, one chunk: the sum is the running sum of x*x down each column, one rounding
    per addition (exact fp64 steps on bounded bf16 inputs, whose squares are exact)."""
    x = bounded_bf16_acts(700, 512, seed=8)
    ids = np.zeros((700, 1), np.int32)
    s2, counts, _ = orc.imatrix_accumulate(x, ids, 1, rows_per_chunk=1024)
    assert counts[0] == 700
    assert np.array_equal(s2[0], running_sum_f64(x))


def test_imatrix_chunks_add_partial_sums(orc):
    """Chunked: each chunk's per-expert partial (running sum over its routed tokens)
    is added to the running total (one fp32 add) in chunk order."""
    T, C, E, K, R = 530, 256, 6, 2, 128
    x = bounded_bf16_acts(T, C, seed=9)
    ids = synth.router(T, E, K, idle=1, seed=10)
    s2, _, _ = orc.imatrix_accumulate(x, ids, E, rows_per_chunk=R)
    ref = np.zeros((E, C), np.float32)
    for t0 in range(0, T, R):
        sl = slice(t0, min(T, t0 + R))
        for e in range(E):
            rows = [t for t in range(sl.start, sl.stop) if e in ids[t]]
            if rows:
                ref[e] = ref[e] + running_sum_f64(x[rows])
    assert np.array_equal(s2, ref)


def test_imatrix_close_to_fp64_sum(orc):
    T, C, E = 2048, 256, 8
    x = synth.activations(T, C, seed=11)
    ids = synth.router(T, E, 2, idle=1, seed=12)
    s2, _, _ = orc.imatrix_accumulate(x, ids, E)
    ref = np.zeros((E, C))
    for t in range(T):
        for e in set(ids[t].tolist()):
            ref[e] += x[t].astype(np.float64) ** 2
    rel = np.abs(s2 - ref) / np.maximum(ref, 1e-30)
    assert rel.max() < 2048 * 2.0 ** -24


def test_imatrix_split_on_chunk_boundary_accumulates(orc):
    """Accumulating two chunk-aligned halves in two calls equals one call (the statistic merges by
    adding, as the GGUF in_sum2/counts files do)."""
    T, C, E = 2048, 256, 8
    x = synth.activations(T, C, seed=13)
    ids = synth.router(T, E, 3, idle=1, seed=14)
    a, ca, _ = orc.imatrix_accumulate(x, ids, E)
    b, cb, _ = orc.imatrix_accumulate(x[:1024], ids[:1024], E)
    b, cb, _ = orc.imatrix_accumulate(x[1024:], ids[1024:], E, in_sum2=b, counts=cb)
    assert np.array_equal(a, b) and np.array_equal(ca, cb)


def test_imatrix_status_bits(orc):
    x = synth.activations(64, 256, seed=15)
    ids = np.tile(np.array([[0, 1]], np.int32), (64, 1))
    ids[3] = [0, 9]      # out of range: ignored, reported
    ids[5] = [1, 1]      # repeated: counted once, reported
    s2, counts, st = orc.imatrix_accumulate(x, ids, 4)
    assert st & orc.ST_BAD_EXPERT_ID and st & orc.ST_DUP_EXPERT_ID
    assert counts.tolist() == [63, 63, 0, 0]   # token 3 lacks expert 1, token 5 lacks expert 0
    # non-finite sums are reported only for experts this call touched
    s2 = np.zeros((4, 256), np.float32)
    s2[3, 7] = np.inf
    _, _, st = orc.imatrix_accumulate(x, np.zeros((64, 1), np.int32), 4, in_sum2=s2)
    assert not (st & orc.ST_NONFINITE_SUM2)
    xn = x.copy(); xn[2, 5] = np.nan
    _, _, st = orc.imatrix_accumulate(xn, np.zeros((64, 1), np.int32), 4)
    assert st & orc.ST_NONFINITE_SUM2


# --- importance weights ------------------------------------------------------------------------

def test_weights_sqrt_of_mean_and_idle_experts(orc):
    rng = np.random.default_rng(16)
    s2 = (rng.random((5, 256)) * 100).astype(np.float32)
    counts = np.array([3, 0, 1, 4096, 0], np.int64)
    w = orc.imatrix_weights(s2, counts)
    for e in range(5):
        if counts[e] == 0:
            assert np.all(w[e] == 1.0)
        else:
            ref = np.sqrt(s2[e] / np.float32(counts[e]))      # numpy: IEEE float32 div and sqrt
            assert np.array_equal(w[e], ref.astype(np.float32))
    wf = orc.imatrix_weights(s2, counts, floor=20.0)
    m = s2[0] / np.float32(3)
    assert np.array_equal(wf[0], np.sqrt(np.maximum(m, np.float32(20.0))))


# --- anchor ------------------------------------------------------------------------------------

def _half(x):
    return np.float32(x).astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("fmt,ratio,K", [("IQ2_XXS", 1.0, 166.625), ("IQ2_XS", 1.0, 166.625),
                                          ("IQ2_S", 1.0, 166.625), ("IQ1_S", 0.61, 15.0)])
def test_anchor_flat_ratio(orc, fmt, ratio, K):
    W = synth.weight_t4(4, 1024, seed=17)
    d16, st = orc.anchor_scales(fmt, W)
    assert st == 0
    amax = np.abs(W.reshape(-1, 256)).max(axis=1)
    ref = ((np.float32(ratio) * amax) / np.float32(K)).astype(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(d16, ref)
    # within half an fp16 ulp of the real-number formula
    exact = ratio * amax.astype(np.float64) / K
    got = d16.view(np.float16).astype(np.float64)
    assert np.all(np.abs(got - exact) <= np.spacing(got.astype(np.float16)).astype(np.float64) * 0.5 + 1e-12)


def test_anchor_iq1_m_peak_to_rms(orc):
    """clamp(0.58 + 0.035 * peak/rms, 0.65, 0.95): blocks with a known peak-to-RMS."""
    a = np.float32(0.5)
    W = np.zeros((1, 256 * 4), np.float32)
    W[0, 0:256] = a                       # p2r = 1  -> 0.615 -> clamped to 0.65
    W[0, 256] = a                         # one spike: p2r = 16 -> 1.14 -> clamped to 0.95
    W[0, 512:516] = a                     # 4 spikes: p2r = 8 -> 0.86
    W[0, 768:768 + 16] = -a               # 16 spikes: p2r = 4 -> 0.72
    d16, _ = orc.anchor_scales("IQ1_M", W)
    for b, ratio in enumerate([0.65, 0.95, 0.58 + 0.035 * 8, 0.58 + 0.035 * 4]):
        got = float(d16[b:b + 1].view(np.float16)[0])
        exact = ratio * 0.5 / 15.0
        assert abs(got - exact) <= float(np.spacing(np.float16(exact))), (b, got, exact)
    zero, _ = orc.anchor_scales("IQ1_M", np.zeros((1, 256), np.float32))
    assert zero[0] == 0


def test_anchor_iq1_m_sums_squares_in_the_fixed_tree(orc):
    """The IQ1_M anchor's sum of squares takes 32 sequential sums of 8 consecutive squares, then
    pairs them (l, l+16), (l, l+8), ..., (l, l+1).  Block A: eight even values whose squares sum to
    S0 = 33,624,288 (in [2^25, 2^26), where fp32 holds multiples of 4), then 248 ones.  In the tree
    the first 8-sum is S0 exactly, the other 31 are 8 each, and every pairing adds a multiple of 4
    below 2^26, so the tree gives the exact S0 + 248.  A sequential sum over the 256 squares rounds
    each S0 + 1 back to S0 and gives S0.  Block B (the same eight values, then 14, 6 and 4, whose
    squares add 248) and block C (the eight values alone) have only multiples of 4 below 2^26 in
    every partial sum, so they give S0 + 248 and S0 in any order.  A must anchor as B, not as C
    (the two differ in the last fp16 bit at this amax)."""
    big = np.array([2080, 2080, 2054, 2062, 2054, 2016, 2020, 2034], np.float32)
    assert int((big.astype(np.int64) ** 2).sum()) == 33624288
    A = np.ones(256, np.float32); A[:8] = big
    B = np.zeros(256, np.float32); B[:8] = big; B[8:11] = [14, 6, 4]
    C = np.zeros(256, np.float32); C[:8] = big
    d16, st = orc.anchor_scales("IQ1_M", np.concatenate([A, B, C])[None, :])
    assert st == 0
    assert d16[1] != d16[2]
    assert d16[0] == d16[1]


def test_anchor_reports_non_finite(orc):
    W = synth.weight_t4(1, 512, seed=18)
    W[0, 300] = np.nan
    d16, st = orc.anchor_scales("IQ2_S", W)
    assert st & orc.ST_BAD_INPUT and d16[1] == 0 and d16[0] != 0
