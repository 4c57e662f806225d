"""Pins of the oracle's decoder, packer and codebook search.

* Decoder: hand-assembled payloads (tests/golden/decode_fixtures.txt, written by an independent bit
  writer) decode to the values their fields define.
* Search: exhaustive brute force over every assignment of a whole choice group with tiny codebooks;
  the one-entry closed form; the round trip (reported error = error of the decoded payload);
  projection; fixed choices reproduce the search (PR #3157 "[1/5]", Testing); the every-choice
  table's minimum is the searched choice (PR #3159); idle experts equal the unweighted search
  (PR #2735); all-zero blocks give all-zero payloads (PR #3157 review); error falls across the five
  formats (IQ1_M CUDA-encoder commit, Testing).
"""
import itertools
import os

import numpy as np
import pytest

from ggml_iq_codebook_accumulate_b300 import synth

FORMATS = ("IQ2_XXS", "IQ2_XS", "IQ2_S", "IQ1_S", "IQ1_M")
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "decode_fixtures.txt")


def _parity7(s):
    return bin(s & 0x7F).count("1") & 1


def semantic_values(fmt, fields, grid):
    """Decoded values from the fields, by the formats' value rule:
    IQ2: d * (2s+1)/8 * g, negated where the sign bit is set (bit 7 = parity of bits 0..6 for
    IQ2_XXS/XS); IQ1: d * (2s+1) * (g + delta), delta = +1/8 for delta bit 0, -1/8 for 1."""
    d = np.float32(np.uint16(fields["d16"]).view(np.float16))
    out = np.zeros(256, np.float32)
    for g in range(32):
        if fmt == "IQ2_XXS":
            s = fields["scale"][g // 4]
        elif fmt in ("IQ2_XS", "IQ2_S", "IQ1_M"):
            s = fields["scale"][g // 2]
        else:
            s = fields["scale"][g // 4]
        e = fields["idx"][g]
        for i in range(8):
            gv = np.float32(grid[e, i])
            if fmt.startswith("IQ2"):
                if fmt == "IQ2_S":
                    sg = (fields["sign8"][g] >> i) & 1
                else:
                    s7 = fields["sign7"][g]
                    sg = ((s7 | (_parity7(s7) << 7)) >> i) & 1
                v = np.float32(np.float32(d * np.float32(2 * s + 1)) * np.float32(0.125)) * gv
                out[8 * g + i] = -v if sg else v
            else:
                db = fields["dbit"][g // 4] if fmt == "IQ1_S" else fields["dbit"][g]
                delta = np.float32(-0.125 if db else 0.125)
                out[8 * g + i] = np.float32(d * np.float32(2 * s + 1)) * np.float32(gv + delta)
    return out


def load_fixtures():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        fmt, fields, hexs = line.strip().split("|")
        f = {}
        for kv in fields.split(";"):
            k, v = kv.split("=")
            vals = [int(t) for t in v.split(",")]
            f[k] = vals[0] if k == "d16" else vals
        rows.append((fmt, f, np.frombuffer(bytes.fromhex(hexs), np.uint8)))
    return rows


@pytest.mark.parametrize("k", range(15))
def test_decode_hand_assembled(orc, k):
    fmt, fields, payload = load_fixtures()[k]
    grid = synth.grid(fmt)
    ref = semantic_values(fmt, fields, grid)
    got = orc.decode(fmt, payload[None, :], 1, 256, grid)[0]
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_decode_mutated_scale_nibble_changes_values(orc):
    """A mis-set scale nibble must change the decoded values of exactly its own groups."""
    for fmt, fields, payload in load_fixtures():
        if fmt != "IQ1_M":
            continue
        grid = synth.grid(fmt)
        base = orc.decode(fmt, payload[None, :], 1, 256, grid)[0]
        mut = payload.copy()
        mut[48] ^= 0x07              # scale of choice group 0 (groups 0 and 1)
        got = orc.decode(fmt, mut[None, :], 1, 256, grid)[0]
        changed = np.nonzero(got != base)[0]
        assert changed.size and changed.min() >= 0 and changed.max() < 16


# --- search ------------------------------------------------------------------------------------

def _q(fmt, d, c, e, grid, sgn8=0, dbit=0):
    """Decoded 8 values of one vector under (choice, entry[, delta bit]) — the value rule above."""
    g = grid[e].astype(np.float32)
    if fmt.startswith("IQ2"):
        dl = np.float32(np.float32(d * np.float32(2 * c + 1)) * np.float32(0.125))
        v = dl * g
        return np.where([(sgn8 >> i) & 1 for i in range(8)], -v, v).astype(np.float32)
    s = c & 7 if fmt == "IQ1_S" else c
    db = (c >> 3) if fmt == "IQ1_S" else dbit
    delta = np.float32(-0.125 if db else 0.125)
    return (np.float32(d * np.float32(2 * s + 1)) * (g + delta)).astype(np.float32)


def _err(x, w, q):
    return float(np.sum(w.astype(np.float64) * (x.astype(np.float64) - q.astype(np.float64)) ** 2))


def _signs(fmt, x, w):
    m = sum(1 << i for i in range(8) if x[i] < 0)
    if fmt in ("IQ2_XXS", "IQ2_XS") and bin(m).count("1") % 2:
        k = np.float32(w) * (np.float32(x) * np.float32(x))
        m ^= 1 << int(np.argmin(k))
    return m


WIDE_IQ2_VALUES = (8.0, 25.0, 43.0, 47.0, 101.0, 127.0)   # squares up to 14 significant bits


@pytest.mark.parametrize("fmt,values", [(f, None) for f in FORMATS] +
                         [(f, WIDE_IQ2_VALUES) for f in ("IQ2_XXS", "IQ2_XS", "IQ2_S")])
def test_search_brute_force_whole_groups(orc, fmt, values):
    """Tiny codebooks (first 3 entries): enumerate every (choice, entry per vector[, delta per
    vector]) assignment of a choice group, score each by decode + fp64 error, and check that the
    oracle's group error is the minimum and its payload decodes to a minimising assignment.  The
    IQ2 formats also run on a grid over a wider value set (up to 127, the largest the formats'
    integer codebooks accept)."""
    info = orc.format_info(fmt)
    n_e = 3
    grid = synth.grid(fmt, values=values, seed=None if values is None else 77)
    rng = np.random.default_rng(FORMATS.index(fmt))
    W = synth.weight_t4(2, 256, seed=30 + FORMATS.index(fmt))
    imp = np.exp(rng.standard_normal(256)).astype(np.float32)
    payload, st, det = orc.encode(fmt, W, grid, importance=imp, details=True, entries=n_e)
    assert st == 0
    d16, _ = orc.anchor_scales(fmt, W)
    vpg, G, C = info["vectors_per_group"], info["groups"], info["num_choices"]
    n_checked = 0
    for b in range(2):
        d = np.float32(d16[b:b + 1].view(np.float16)[0])
        x = W[b].reshape(32, 8)
        w = imp.reshape(32, 8)
        dec = orc.decode(fmt, payload[b:b + 1], 1, 256, grid)[0].reshape(32, 8)
        for g in range(G):
            vs = range(g * vpg, (g + 1) * vpg)
            cands = [(e, db) for db in ((0, 1) if fmt == "IQ1_M" else (0,)) for e in range(n_e)]
            best = np.inf
            errs = {}
            for c in range(C):
                per_v = [[_err(x[v], w[v], _q(fmt, d, c, e, grid, _signs(fmt, x[v], w[v]), db)) for (e, db) in cands]
                         for v in vs]
                for combo in itertools.product(range(len(cands)), repeat=vpg):
                    tot = 0.0
                    for j, v in enumerate(vs):
                        tot = tot + per_v[j][combo[j]]
                    errs[(c, combo)] = tot
                    best = min(best, tot)
            assert det["gbest"][b, g] == pytest.approx(best, rel=1e-12, abs=1e-300)
            got = sum(_err(x[v], w[v], dec[v]) for v in vs)
            assert got == pytest.approx(best, rel=1e-12, abs=1e-300)
            n_checked += 1
    assert n_checked == 2 * G


@pytest.mark.parametrize("fmt", ["IQ2_XXS", "IQ2_S", "IQ1_S"])
def test_one_entry_codebook_picks_nearest_scale(orc, fmt):
    """With one codebook entry the group error is a parabola in the local scale alpha:
    E(alpha) = C - 2 alpha A + alpha^2 B (sums over the group), so the chosen choice is the alpha_c
    nearest to A/B (IQ1_S: per delta sign, the better of the two)."""
    info = orc.format_info(fmt)
    grid = synth.grid(fmt)
    W = synth.weight_t4(4, 256, seed=40)
    imp = np.exp(np.random.default_rng(41).standard_normal(256)).astype(np.float32)
    payload, _, det = orc.encode(fmt, W, grid, importance=imp, details=True, entries=1)
    d16, _ = orc.anchor_scales(fmt, W)
    vpg = info["vectors_per_group"]
    for b in range(4):
        d = float(d16[b:b + 1].view(np.float16)[0])
        x = W[b].astype(np.float64).reshape(32, 8)
        w = imp.astype(np.float64).reshape(32, 8)
        for g in range(info["groups"]):
            best_c, best_E = None, np.inf
            for c in range(info["num_choices"]):
                A = B = Cc = 0.0
                for v in range(g * vpg, (g + 1) * vpg):
                    if fmt.startswith("IQ2"):
                        sg = _signs(fmt, W[b].reshape(32, 8)[v], imp.reshape(32, 8)[v])
                        u = grid[0].astype(np.float64) * np.array([-1.0 if (sg >> i) & 1 else 1.0 for i in range(8)])
                        alpha = d * (2 * c + 1) / 8
                    else:
                        u = grid[0].astype(np.float64) + (-0.125 if c >> 3 else 0.125)
                        alpha = d * (2 * (c & 7) + 1)
                    A += np.sum(w[v] * x[v] * u); B += np.sum(w[v] * u * u); Cc += np.sum(w[v] * x[v] ** 2)
                E = Cc - 2 * alpha * A + alpha * alpha * B
                if best_c is None or E < best_E - 1e-12 * abs(best_E):
                    best_c, best_E = c, E
            assert det["chosen"][b, g] == best_c


@pytest.mark.parametrize("fmt", FORMATS)
def test_round_trip_error_and_fixed_choices(orc, fmt):
    """(a) the error the search reports is the error of its decoded payload; (b) fixing every
    group's choice to the searched one reproduces the payload byte for byte; (c) fixing one choice
    everywhere reproduces the searched fields at every group where that choice won; (d) the every-choice
    table's minimum is the searched choice's error."""
    info = orc.format_info(fmt)
    grid = synth.grid(fmt)
    W = synth.weight_t4(3, 512, seed=50)
    imp = np.exp(np.random.default_rng(51).standard_normal(512)).astype(np.float32)
    payload, st, det = orc.encode(fmt, W, grid, importance=imp, details=True)
    assert st == 0
    gerr, verr = orc.payload_errors(fmt, W, grid, payload, importance=imp)
    assert np.allclose(gerr, det["gbest"], rtol=1e-12, atol=0)
    assert np.allclose(verr, det["vbest"], rtol=1e-12, atol=0)
    p2, _ = orc.encode(fmt, W, grid, importance=imp, choices=det["chosen"])
    assert np.array_equal(p2, payload)
    common = int(np.bincount(det["chosen"].ravel()).argmax())
    seven = np.full_like(det["chosen"], common)
    p7, _, det7 = orc.encode(fmt, W, grid, importance=imp, choices=seven, details=True)
    dec = orc.decode(fmt, payload, 3, 512, grid).reshape(-1, 32, 8)
    dec7 = orc.decode(fmt, p7, 3, 512, grid).reshape(-1, 32, 8)
    vpg = info["vectors_per_group"]
    won = det["chosen"] == common
    for b, g in zip(*np.nonzero(won)):
        assert np.array_equal(dec[b, g * vpg:(g + 1) * vpg], dec7[b, g * vpg:(g + 1) * vpg])
    tbl = det["table"]
    assert np.array_equal(np.argmin(tbl, axis=2), det["chosen"])
    assert np.array_equal(tbl.min(axis=2), det["gbest"])


@pytest.mark.parametrize("fmt", FORMATS)
def test_projection_and_zero_block(orc, fmt):
    """Re-encoding decoded values under the same scale and positive weights reproduces them
    exactly; an all-zero block encodes to an all-zero payload."""
    grid = synth.grid(fmt)
    W = synth.weight_t4(2, 512, seed=60)
    W[1, 256:] = 0.0
    payload, _ = orc.encode(fmt, W, grid)
    assert not payload[3].any() and payload[0].any()
    dec = orc.decode(fmt, payload, 2, 512, grid)
    d16, _ = orc.anchor_scales(fmt, W)
    p2, _ = orc.encode(fmt, dec, grid, d16=d16)
    assert np.array_equal(orc.decode(fmt, p2, 2, 512, grid), dec)


def test_sign_rule_even_parity_flips_weakest(orc):
    """IQ2_XXS/XS store 7 sign bits; the 8th is implied by even parity, so an odd count of negative
    inputs flips the sign of argmin w*x^2 (the weakest element)."""
    grid = synth.grid("IQ2_XXS")
    rng = np.random.default_rng(70)
    W = (rng.standard_normal((1, 256)) * 0.02).astype(np.float32)
    imp = np.exp(rng.standard_normal(256)).astype(np.float32)
    payload, _ = orc.encode("IQ2_XXS", W, grid, importance=imp)
    dec = orc.decode("IQ2_XXS", payload, 1, 256, grid)[0].reshape(32, 8)
    x = W[0].reshape(32, 8); w = imp.reshape(32, 8)
    for v in range(32):
        neg = x[v] < 0
        dneg = dec[v] < 0
        assert dneg.sum() % 2 == 0
        if neg.sum() % 2 == 0:
            assert np.array_equal(neg, dneg)
        else:
            flipped = np.nonzero(neg != dneg)[0]
            assert flipped.tolist() == [int(np.argmin(w[v] * (x[v] * x[v])))]


def test_iq2_s_keeps_input_signs(orc):
    grid = synth.grid("IQ2_S")
    W = synth.weight_t4(1, 256, seed=71)
    payload, _ = orc.encode("IQ2_S", W, grid)
    dec = orc.decode("IQ2_S", payload, 1, 256, grid)[0]
    assert np.array_equal(dec < 0, W[0] < 0)


@pytest.mark.parametrize("fmt", ["IQ2_XXS", "IQ1_M"])
def test_idle_expert_equals_unweighted_search(orc, fmt):
    """An expert no token reached gets weight 1 on every channel (count 0), which is the plain
    search: same bytes as encoding without importance."""
    grid = synth.grid(fmt)
    E, rpe, C = 3, 2, 256
    W = synth.weight_t4(E * rpe, C, seed=80)
    x = synth.activations(64, C, seed=81)
    ids = np.tile(np.array([[0, 2]], np.int32), (64, 1))       # expert 1 is idle
    s2, counts, _ = orc.imatrix_accumulate(x, ids, E)
    w = orc.imatrix_weights(s2, counts)
    assert counts[1] == 0 and np.all(w[1] == 1.0)
    p_w, _ = orc.encode(fmt, W, grid, importance=w, rows_per_expert=rpe)
    p_plain, _ = orc.encode(fmt, W, grid)
    bpr = C // 256
    assert np.array_equal(p_w[1 * rpe * bpr:2 * rpe * bpr], p_plain[1 * rpe * bpr:2 * rpe * bpr])
    assert not np.array_equal(p_w[:rpe * bpr], p_plain[:rpe * bpr])


def test_reconstruction_error_falls_across_formats(orc):
    """Relative weighted reconstruction error: IQ1_S > IQ1_M > IQ2_XXS > IQ2_XS > IQ2_S (a sanity
    check with synthetic codebooks; the pages state it for the real ones)."""
    W = synth.as_dtype(synth.weight_t4(16, 512, seed=90), "bf16")[1]
    imp = np.exp(np.random.default_rng(91).standard_normal(512)).astype(np.float32)
    rel = {}
    for fmt in ("IQ1_S", "IQ1_M", "IQ2_XXS", "IQ2_XS", "IQ2_S"):
        grid = synth.grid(fmt)
        p, _ = orc.encode(fmt, W, grid, importance=imp)
        gerr, _ = orc.payload_errors(fmt, W, grid, p, importance=imp)
        rel[fmt] = gerr.sum() / np.sum(imp.astype(np.float64) * W.astype(np.float64) ** 2)
    seq = [rel[f] for f in ("IQ1_S", "IQ1_M", "IQ2_XXS", "IQ2_XS", "IQ2_S")]
    assert all(a > b for a, b in zip(seq, seq[1:])), rel


def test_bad_units_are_zeroed_and_reported(orc):
    fmt = "IQ2_XS"
    grid = synth.grid(fmt)
    W = synth.weight_t4(1, 1024, seed=95)
    W[0, 5] = np.inf
    imp = np.ones(1024, np.float32); imp[600] = -1.0
    ch = np.zeros((4, 16), np.uint8); ch[3, 2] = 16
    p, st = orc.encode(fmt, W, grid, importance=imp, choices=ch)
    assert st & orc.ST_BAD_INPUT and st & orc.ST_BAD_IMPORTANCE and st & orc.ST_BAD_CHOICE
    assert not p[0].any() and p[1].any() and not p[2].any() and not p[3].any()
    bad_grid = grid.copy(); bad_grid[3, 1] = 7.5
    p, st = orc.encode(fmt, W[:, 256:], bad_grid)
    assert st & orc.ST_BAD_GRID and not p.any()
