"""Oracle of the local-Hessian choice search and of the every-choice payloads (fp64, numpy).

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU legs may call it; the library never
does.  It is built on this package's forced encode and decode (``encode``, ``decode``), and it
does its own arithmetic in fp64 with numpy.

Sources:
- PR #3159 "one-pass every-choice encode", *What does this PR do?* and *Usage*: for every choice
  c, the payload of the forced encode with every group at choice c.
- PR #3158 "local_hessian for GGML IQ", *What does this PR do?*: each group's local scale (and
  IQ1_S delta sign) is picked by the layer-output error dw H dw^T over the 256-column diagonal
  block of the input Hessian, the blocks damped by perc_damp as GPTQ damps (default 0.3).  The
  search: (1) encode each block under every choice; (2) give each group its best choice under its
  own H_gg block; (3) revisit the groups twice, each taking the choice that most lowers the
  block's error with the others held.

Readings (the pages leave these open):
- Damping: H' = H_bb + perc_damp * mean(diag(H_bb)) * I for each 256-column diagonal block H_bb.
- dw = x - q, with q the decoded values of a payload (the weight the block packs to), in fp64.
- Step 2 ties: the lowest choice.
- Step 3: groups are visited in ascending order, each against the other groups' current choices.
  A group moves only to a choice whose block error is strictly lower than with its current
  choice; among choices with the same lowest error, the lowest.
- The payload under the searched choices is the forced encode with those choices per group.

Parity status: pinned by tests/test_oracle_local_hessian.py: H = I with unit importance gives the
encoder's own searched choices (the pages' test); a block-diagonal H leaves step 2's picks
unchanged by the revisits and equals a per-group brute force; heavy damping tends to the
unweighted picks; scaling H changes nothing; the revisits never raise the block error; the
every-choice payloads equal the forced encodes.
"""
from __future__ import annotations

import numpy as np

from . import decode, encode, format_info


def every_choice_payloads(fmt, W, grid, importance=None, rows_per_expert=0, d16=None, threads=0):
    """[num_choices, B, block_bytes] uint8: payload c is the forced encode with every group at c."""
    info = format_info(fmt)
    W = np.asarray(W, np.float32)
    R, C = W.shape
    B = R * (C // 256)
    G, NC = info["groups"], info["num_choices"]
    out = np.empty((NC, B, info["block_bytes"]), np.uint8)
    for c in range(NC):
        out[c], _ = encode(fmt, W, grid, importance=importance, rows_per_expert=rows_per_expert, d16=d16,
                           choices=np.full((B, G), c, np.uint8), threads=threads)
    return out


def damped_blocks(H_blocks, perc_damp):
    """H' = H_bb + perc_damp * mean(diag(H_bb)) * I for each [256, 256] block, in fp64."""
    Hb = np.asarray(H_blocks, np.float64)
    lam = perc_damp * np.einsum("bii->b", Hb) / 256.0
    return Hb + lam[:, None, None] * np.eye(256)


def block_dw(fmt, W, grid, payloads):
    """dw[c, r, col] = x - q_c in fp64 for every choice's payload."""
    W = np.asarray(W, np.float32)
    R, C = W.shape
    X = W.astype(np.float64)
    return np.stack([X - decode(fmt, payloads[c], R, C, grid).astype(np.float64) for c in range(len(payloads))])


def local_hessian_choices(fmt, W, grid, payloads, H_blocks, perc_damp=0.3, trace=False):
    """Searched choices [B, G] uint8 for ``W`` [R, C] given the every-choice payloads and the
    256 x 256 diagonal blocks of the input Hessian ([C / 256, 256, 256]).

    With ``trace`` it also returns, per block, the list of decisions taken: for step 2 one
    (group, errors over the choices) per group, for each revisit one (group, block errors over
    the choices) per group, each with the choice taken.  Tests replay a device search against it.
    """
    info = format_info(fmt)
    R, C = np.asarray(W).shape
    G, NC = info["groups"], info["num_choices"]
    gs = 256 // G
    nb = C // 256
    Hd = damped_blocks(H_blocks, perc_damp)
    dw_all = block_dw(fmt, W, grid, payloads)  # [NC, R, C]
    choices = np.empty((R * nb, G), np.uint8)
    traces = []
    for r in range(R):
        for j in range(nb):
            cur, tr = search_block(dw_all[:, r, 256 * j:256 * (j + 1)], Hd[j], gs, trace=trace)
            choices[r * nb + j] = cur
            traces.append(tr)
    return (choices, traces) if trace else choices


def block_error(dw_cur, H):
    """dw H dw^T of one block (fp64)."""
    return float(dw_cur @ H @ dw_cur)


def search_block(dw, H, gs, trace=False):
    """The search on one block: dw [NC, 256] (every choice), H [256, 256] damped."""
    NC = dw.shape[0]
    G = 256 // gs
    cur = np.empty(G, np.int64)
    tr = []
    # step 2: each group's best choice under its own diagonal block
    for g in range(G):
        s = slice(g * gs, (g + 1) * gs)
        e = np.einsum("ci,ij,cj->c", dw[:, s], H[s, s], dw[:, s])
        cur[g] = int(np.argmin(e))                      # first minimum: the lowest choice
        if trace:
            tr.append(("own", g, e, int(cur[g])))
    # step 3: two revisits, each group against the others' current choices
    for _ in range(2):
        for g in range(G):
            s = slice(g * gs, (g + 1) * gs)
            base = np.concatenate([dw[cur[h], h * gs:(h + 1) * gs] for h in range(G)])
            D = np.repeat(base[None, :], NC, axis=0)
            D[:, s] = dw[:, s]
            errs = np.einsum("ci,ij,cj->c", D, H, D)
            pick = int(np.argmin(errs))
            if errs[pick] < errs[cur[g]]:
                cur[g] = pick
            if trace:
                tr.append(("revisit", g, errs, int(cur[g])))
    return cur.astype(np.uint8), tr
