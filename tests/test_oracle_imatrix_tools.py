"""Pins of the imatrix merge / neutral-entry / coverage oracle (oracle/imatrix_tools.py) against
the C oracle's imatrix and closed forms."""
import numpy as np

import oracle
from oracle import imatrix_tools as it
from ggml_iq_codebook_accumulate_b300 import synth


def test_merging_statistics_of_disjoint_experts_equals_one_call():
    """Tokens of part A reach only experts 0..7 and those of part B only 8..15; with the split on a
    chunk boundary, merging the two statistics is bit for bit the statistic of one call over all
    the tokens (each expert's sum comes from one part, the other adds exactly +0)."""
    T, C, E, K, R = 512, 64, 16, 3, 128
    _, xv = synth.as_dtype(synth.activations(T, C, seed=31), "bf16")
    rng = np.random.default_rng(31)
    ids = np.stack([rng.choice(8, K, replace=False) + (0 if t < 256 else 8) for t in range(T)]).astype(np.int32)
    sa, ca, _ = oracle.imatrix_accumulate(xv[:256], ids[:256], E, rows_per_chunk=R)
    sb, cb, _ = oracle.imatrix_accumulate(xv[256:], ids[256:], E, rows_per_chunk=R)
    s, c, _ = oracle.imatrix_accumulate(xv, ids, E, rows_per_chunk=R)
    ms, mc = it.merge(sa, ca, sb, cb)
    assert np.array_equal(ms.view(np.uint32), s.view(np.uint32)) and np.array_equal(mc, c)


def test_merge_identity_and_order():
    rng = np.random.default_rng(32)
    s = (rng.standard_normal((5, 48)) ** 2).astype(np.float32)
    t = (rng.standard_normal((5, 48)) ** 2 * 1e3).astype(np.float32)
    c, d = rng.integers(0, 100, 5), rng.integers(0, 100, 5)
    z, zc = np.zeros_like(s), np.zeros_like(c)
    a, ac = it.merge(s, c, z, zc)
    assert np.array_equal(a.view(np.uint32), s.view(np.uint32)) and np.array_equal(ac, c)
    x, xc = it.merge(s, c, t, d)
    y, yc = it.merge(t, d, s, c)
    assert np.array_equal(x.view(np.uint32), y.view(np.uint32)) and np.array_equal(xc, yc)


def test_neutral_entries_have_weight_one_and_the_rest_is_unchanged():
    T, C, E, K = 300, 32, 12, 2
    _, xv = synth.as_dtype(synth.activations(T, C, seed=33), "bf16")
    ids = synth.router(T, E, K, idle=3, seed=33)
    s, c, _ = oracle.imatrix_accumulate(xv, ids, E)
    ns, nc = it.neutral_entries(s, c)
    idle = c == 0
    assert idle.sum() >= 3 and np.all(nc[idle] == 1) and np.all(ns[idle] == 1.0)
    assert np.array_equal(ns[~idle].view(np.uint32), s[~idle].view(np.uint32)) and np.array_equal(nc[~idle], c[~idle])
    w0, w1 = oracle.imatrix_weights(s, c), oracle.imatrix_weights(ns, nc)
    assert np.array_equal(w0.view(np.uint32), w1.view(np.uint32))   # count 0 and the neutral entry weigh 1


def test_coverage_closed_forms():
    T, C, E, K, idle = 1000, 16, 40, 4, 5
    _, xv = synth.as_dtype(synth.activations(T, C, seed=34), "bf16")
    ids = synth.router(T, E, K, idle=idle, seed=34)
    _, c, _ = oracle.imatrix_accumulate(xv, ids, E)
    touched, total, lo, hi = it.coverage(c)
    assert total == T * K                                   # every token reaches K distinct experts
    assert touched == E - idle and lo == 0                 # the idle experts have no tokens
    assert hi == max(int((ids == e).sum()) for e in range(E))
