"""Pins of the local-Hessian choice search oracle (oracle/local_hessian.py) against facts that do
not come from its own code: the encoder's searched choices (plain C oracle), the separable case,
damping and scaling limits, monotone revisits, and the pages' claim that the search lowers the
layer-output error on correlated inputs (PR #3158, Testing)."""
import numpy as np
import pytest

import oracle
from oracle import local_hessian as lh
from ggml_iq_codebook_accumulate_b300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
FORMATS = synth.FORMATS


def weight(R, C, seed):
    _, wv = synth.as_dtype(synth.weight_t4(R, C, seed=seed), "bf16")
    return wv


def correlated_hessian(C, n, seed, rho=0.85):
    """H = X^T X / n for inputs whose neighbouring columns are correlated (AR(1) along the columns,
    coefficient rho) with log-normal column scales: a dense SPD matrix with strong coupling inside
    and across groups."""
    rng = np.random.default_rng(seed)
    Z = rng.standard_normal((n, C))
    X = np.empty_like(Z)
    X[:, 0] = Z[:, 0]
    for j in range(1, C):
        X[:, j] = rho * X[:, j - 1] + np.sqrt(1 - rho * rho) * Z[:, j]
    X *= np.exp(0.5 * rng.standard_normal(C))[None, :]
    return X, X.T @ X / n


def blocks_of(H, C):
    return np.stack([H[256 * j:256 * (j + 1), 256 * j:256 * (j + 1)] for j in range(C // 256)])


def searched_choices(fmt, W, grid, importance):
    _, _, det = oracle.encode(fmt, W, grid, importance=importance, details=True)
    return det["chosen"]


@pytest.mark.parametrize("fmt", FORMATS)
def test_identity_hessian_with_unit_importance_keeps_the_encoders_choices(fmt):
    """PR #3158 Testing: under H = I the search reproduces the encoder's own picks."""
    R, C = 4, 512
    W = weight(R, C, 11)
    grid = synth.grid(fmt)
    ones = np.ones(C, np.float32)
    pay = lh.every_choice_payloads(fmt, W, grid, importance=ones)
    H = np.stack([np.eye(256)] * (C // 256))
    got = lh.local_hessian_choices(fmt, W, grid, pay, H, perc_damp=0.3)
    assert np.array_equal(got, searched_choices(fmt, W, grid, ones))


@pytest.mark.parametrize("fmt", FORMATS)
def test_diagonal_hessian_equals_the_importance_weighted_search(fmt):
    """With H = diag(importance) and no damping, dw H dw^T is the encoder's weighted squared error,
    so every group's pick is the encoder's searched choice and the revisits move nothing."""
    R, C = 4, 512
    W = weight(R, C, 12)
    grid = synth.grid(fmt)
    rng = np.random.default_rng(3)
    imp = np.exp(rng.standard_normal(C)).astype(np.float32)
    pay = lh.every_choice_payloads(fmt, W, grid, importance=imp)
    H = np.stack([np.diag(imp[256 * j:256 * (j + 1)].astype(np.float64)) for j in range(C // 256)])
    got, traces = lh.local_hessian_choices(fmt, W, grid, pay, H, perc_damp=0.0, trace=True)
    assert np.array_equal(got, searched_choices(fmt, W, grid, imp))
    G = oracle.format_info(fmt)["groups"]
    for tr in traces:
        own = [t[3] for t in tr[:G]]
        assert [t[3] for t in tr[G:2 * G]] == own and [t[3] for t in tr[2 * G:]] == own


@pytest.mark.parametrize("fmt", ["IQ2_XXS", "IQ2_S", "IQ1_S"])
def test_block_diagonal_hessian_revisits_change_nothing(fmt):
    """No coupling between groups: the block error is a sum of per-group terms, so the revisits keep
    step 2's picks, which are each group's own minimum."""
    R, C = 3, 512
    W = weight(R, C, 13)
    grid = synth.grid(fmt)
    gs = 256 // oracle.format_info(fmt)["groups"]
    pay = lh.every_choice_payloads(fmt, W, grid)
    rng = np.random.default_rng(5)
    Hb = []
    for _ in range(C // 256):
        M = np.zeros((256, 256))
        for g in range(256 // gs):
            A = rng.standard_normal((gs, gs))
            M[g * gs:(g + 1) * gs, g * gs:(g + 1) * gs] = A @ A.T + gs * np.eye(gs)
        Hb.append(M)
    got, traces = lh.local_hessian_choices(fmt, W, grid, pay, np.stack(Hb), perc_damp=0.3, trace=True)
    dw = lh.block_dw(fmt, W, grid, pay)
    Hd = lh.damped_blocks(np.stack(Hb), 0.3)
    nb = C // 256
    for b, tr in enumerate(traces):
        r, j = divmod(b, nb)
        G = 256 // gs
        for g in range(G):
            s = slice(g * gs, (g + 1) * gs)
            d = dw[:, r, 256 * j:256 * (j + 1)][:, s]
            own = [float(d[c] @ Hd[j][s, s] @ d[c]) for c in range(d.shape[0])]
            assert got[b, g] == int(np.argmin(own))


@pytest.mark.parametrize("fmt", ["IQ2_XS", "IQ1_M"])
def test_heavy_damping_tends_to_the_unweighted_picks(fmt):
    """PR #3158 Testing: H = I is the limit heavy damping tends to."""
    R, C = 4, 512
    W = weight(R, C, 14)
    grid = synth.grid(fmt)
    ones = np.ones(C, np.float32)
    pay = lh.every_choice_payloads(fmt, W, grid, importance=ones)
    _, H = correlated_hessian(C, 2048, seed=6)
    got = lh.local_hessian_choices(fmt, W, grid, pay, blocks_of(H, C), perc_damp=1e9)
    assert np.array_equal(got, searched_choices(fmt, W, grid, ones))


def test_scaling_the_hessian_changes_nothing():
    fmt, R, C = "IQ2_S", 4, 512
    W = weight(R, C, 15)
    grid = synth.grid(fmt)
    _, H = correlated_hessian(C, 2048, seed=7)
    imp = np.sqrt(np.diag(H)).astype(np.float32)
    pay = lh.every_choice_payloads(fmt, W, grid, importance=imp)
    a = lh.local_hessian_choices(fmt, W, grid, pay, blocks_of(H, C), perc_damp=0.3)
    b = lh.local_hessian_choices(fmt, W, grid, pay, 8.0 * blocks_of(H, C), perc_damp=0.3)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("fmt", FORMATS)
def test_revisits_never_raise_the_block_error_and_do_move(fmt):
    """Each revisit keeps or lowers the block error; on correlated inputs some of them move."""
    R, C = 4, 512
    W = weight(R, C, 16)
    grid = synth.grid(fmt)
    _, H = correlated_hessian(C, 2048, seed=8)
    imp = np.sqrt(np.diag(H)).astype(np.float32)
    pay = lh.every_choice_payloads(fmt, W, grid, importance=imp)
    _, traces = lh.local_hessian_choices(fmt, W, grid, pay, blocks_of(H, C), perc_damp=0.3, trace=True)
    G = oracle.format_info(fmt)["groups"]
    moved = 0
    for tr in traces:
        prev = [t[3] for t in tr[:G]]
        for k, (kind, g, errs, pick) in enumerate(tr[G:]):
            assert kind == "revisit"
            assert errs[pick] <= errs[prev[g]]
            moved += pick != prev[g]
            prev[g] = pick
    assert moved > 0


@pytest.mark.parametrize("fmt", ["IQ2_XXS", "IQ2_XS", "IQ1_S"])
def test_search_lowers_the_output_error_of_correlated_inputs(fmt):
    """PR #3158 Testing: on correlated inputs the local-Hessian picks give a lower layer-output
    error ||X (W - Q)^T||^2 than the importance-weighted picks (importance = sqrt(diag H))."""
    R, C = 16, 512
    W = weight(R, C, 17)
    grid = synth.grid(fmt)
    X, H = correlated_hessian(C, 4096, seed=9)
    imp = np.sqrt(np.diag(H)).astype(np.float32)
    pay = lh.every_choice_payloads(fmt, W, grid, importance=imp)
    ch = lh.local_hessian_choices(fmt, W, grid, pay, blocks_of(H, C), perc_damp=0.3)
    p_lh, _ = oracle.encode(fmt, W, grid, importance=imp, choices=ch)
    p_im, _ = oracle.encode(fmt, W, grid, importance=imp)

    def out_err(p):
        dW = W.astype(np.float64) - oracle.decode(fmt, p, R, C, grid).astype(np.float64)
        return float(np.sum((X @ dW.T) ** 2))

    assert out_err(p_lh) < out_err(p_im)


@pytest.mark.parametrize("fmt", ["IQ2_S", "IQ1_M"])
def test_searched_payload_is_made_of_the_every_choice_payloads(fmt):
    """Each group of the payload encoded under the searched choices decodes to the same values as
    that group in the every-choice payload of its choice (a group's entries depend only on its
    own choice)."""
    R, C = 4, 512
    W = weight(R, C, 18)
    grid = synth.grid(fmt)
    _, H = correlated_hessian(C, 2048, seed=10)
    imp = np.sqrt(np.diag(H)).astype(np.float32)
    pay = lh.every_choice_payloads(fmt, W, grid, importance=imp)
    ch = lh.local_hessian_choices(fmt, W, grid, pay, blocks_of(H, C), perc_damp=0.3)
    p, _ = oracle.encode(fmt, W, grid, importance=imp, choices=ch)
    q = oracle.decode(fmt, p, R, C, grid).reshape(-1, 256)
    G = oracle.format_info(fmt)["groups"]
    gs = 256 // G
    qc = [oracle.decode(fmt, pay[c], R, C, grid).reshape(-1, 256) for c in range(len(pay))]
    for b in range(q.shape[0]):
        for g in range(G):
            s = slice(g * gs, (g + 1) * gs)
            assert np.array_equal(q[b, s], qc[ch[b, g]][b, s])


def test_revisits_on_a_hand_computed_block():
    """The revisit step (PR #3158: two passes, each group against the others' current choices,
    moving only to a strictly lower block error) on a block worked out by hand.

    Four groups of 64 columns and three choices; only column 64 g of group g is nonzero, with
    dw = a[g][c] under choice c (group 3 is all zero), so dw H dw^T is the quadratic form of the
    3 x 3 matrix M of H's entries at columns 0, 64, 128:
        a = [[-3, 0, 1], [-3, 2, 3], [-2, -3, 2]],   M = [[5, -2, 2], [-2, 4, -2], [2, -2, 2]]
        E(v) = 5 v0^2 + 4 v1^2 + 2 v2^2 - 4 v0 v1 + 4 v0 v2 - 4 v1 v2.
    Own blocks (a^2 M_gg): group 0 (45, 0, 5) -> 1; group 1 (36, 16, 36) -> 1; group 2 (8, 18, 8)
    -> 0 (lowest choice of two equal); group 3 all 0 -> 0.
    Revisit 1, start (1, 1, 0):
      group 0 with v1 = 2, v2 = -2: E = 5 v0^2 - 16 v0 + 40 = (133, 40, 29) -> moves to 2;
      group 1 with v0 = 1 (group 0's NEW choice), v2 = -2: E = 4 v1^2 + 4 v1 + 5 = (29, 29, 53):
        choice 0 only ties the current choice 1, so group 1 stays at 1 (with the stale v0 = 0 it
        would read (20, 40, 68) and move to 0);
      group 2 with v0 = 1, v1 = 2: E = 2 v2^2 - 4 v2 + 13 = (29, 43, 13) -> moves to 2.
    Revisit 2, start (2, 1, 2):
      group 0 with v1 = 2, v2 = 2: E = 5 v0^2 + 8 = (53, 8, 13) -> moves to 1 (only a second pass
        makes this move);
      group 1 with v0 = 0, v2 = 2: E = 4 v1^2 - 8 v1 + 8 = (68, 8, 20) -> stays at 1;
      group 2 with v0 = 0, v1 = 2: E = 2 v2^2 - 8 v2 + 16 = (40, 58, 8) -> stays at 2.
    Result (1, 1, 2, 0).  One pass would leave (2, 1, 2, 0); moving on equal errors would give
    group 1 choice 0; revisiting against the step-2 choices would also move group 1."""
    a = np.array([[-3, 0, 1], [-3, 2, 3], [-2, -3, 2]], np.float64)
    M = np.array([[5, -2, 2], [-2, 4, -2], [2, -2, 2]], np.float64)
    cols = [0, 64, 128]
    dw = np.zeros((3, 256))
    for g in range(3):
        dw[:, cols[g]] = a[g]
    H = np.eye(256)
    for i in range(3):
        for j in range(3):
            H[cols[i], cols[j]] = M[i, j]
    got, tr = lh.search_block(dw, H, 64, trace=True)
    assert got.tolist() == [1, 1, 2, 0]
    own = [t[3] for t in tr if t[0] == "own"]
    assert own == [1, 1, 0, 0]
    rev = [t for t in tr if t[0] == "revisit"]
    assert len(rev) == 8                                  # two passes over four groups
    assert [t[3] for t in rev] == [2, 1, 2, 0, 1, 1, 2, 0]
    assert rev[0][2].tolist() == [133, 40, 29]
    assert rev[1][2].tolist() == [29, 29, 53]
    assert rev[2][2].tolist() == [29, 43, 13]
    assert rev[4][2].tolist() == [53, 8, 13]
    assert rev[5][2].tolist() == [68, 8, 20]
    assert rev[6][2].tolist() == [40, 58, 8]
