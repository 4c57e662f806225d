"""Helpers shared by the GPU parity tests: the near-tie acceptance rule for encoded payloads.

Rule: payload bytes must equal the oracle's, except inside a choice group where the oracle's two
best choices (or, under the chosen choice, some vector's two best candidates) differ by less than
1e-6 of the best error; there the library's group is accepted if its own weighted error is within
1e-6 (relative) of the oracle's minimum.  Scale and sign fields are never exempt.
"""
import numpy as np

import oracle

REL = 1e-6


def group_values_differ(fmt, p_gpu, p_orc, rows, cols, grid):
    info = oracle.format_info(fmt)
    dg = oracle.decode(fmt, p_gpu, rows, cols, grid).reshape(-1, 32, 8)
    do = oracle.decode(fmt, p_orc, rows, cols, grid).reshape(-1, 32, 8)
    vpg = info["vectors_per_group"]
    diff_v = (dg != do).any(axis=2)                                   # [B, 32]
    return diff_v.reshape(-1, info["groups"], vpg).any(axis=2), diff_v  # [B, G], [B, 32]


def check_payload(fmt, W, grid, p_gpu, p_orc, det, importance=None, rows_per_expert=0, max_allowed=None):
    """Returns the number of accepted near-tie groups; raises AssertionError on a violation."""
    p_gpu = np.asarray(p_gpu, np.uint8)
    p_orc = np.asarray(p_orc, np.uint8)
    if np.array_equal(p_gpu, p_orc):
        return 0
    rows, cols = W.shape
    info = oracle.format_info(fmt)
    bad_blocks = np.nonzero((p_gpu != p_orc).any(axis=1))[0]
    gdiff, _ = group_values_differ(fmt, p_gpu, p_orc, rows, cols, grid)
    # bytes differ but decoded values agree: only possible through a field outside the values
    assert gdiff[bad_blocks].any(axis=1).all(), "payload bytes differ without a value difference"
    gerr, verr = oracle.payload_errors(fmt, W, grid, p_gpu, importance=importance, rows_per_expert=rows_per_expert)
    vpg = info["vectors_per_group"]
    accepted = 0
    for b, g in zip(*np.nonzero(gdiff)):
        best = det["gbest"][b, g]
        near_choice = (det["gsecond"][b, g] - best) < REL * best
        vs = slice(g * vpg, (g + 1) * vpg)
        near_vec = ((det["vsecond"][b, vs] - det["vbest"][b, vs]) < REL * det["vbest"][b, vs]).any()
        assert near_choice or near_vec, f"block {b} group {g}: differs with a clear oracle optimum"
        assert gerr[b, g] <= best * (1 + REL) + 1e-30, f"block {b} group {g}: error {gerr[b, g]} > {best}"
        accepted += 1
    if max_allowed is not None:
        assert accepted <= max_allowed
    return accepted
