"""GPU parity on IQ2 codebooks whose squares do not fit tf32.

The boundary accepts IQ2 codebook values that are integers in [1, 127].  Squares of values such as
47, 101 and 127 need up to 14 significant bits, more than the 11 of tf32, so the encoder feeds
h = g^2 to the tensor cores as two exact tf32 parts.  These grids hold 47, 101 and 127 next to
8, 25 and 43.  Every block of a small case, and sampled rows of the 5632 x 2048 encode-speed
weight, must be byte-identical to the oracle (searched, with importance; fixed choices too).
"""
import numpy as np
import pytest
import torch

import oracle
from ggml_iq_codebook_accumulate_b300 import api, synth
from parity import check_payload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
WIDE = (8.0, 25.0, 43.0, 47.0, 101.0, 127.0)


def dev_bf16(store):
    return torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(DEV)


def wide_grid(fmt):
    g = synth.grid(fmt, values=WIDE, seed=77)
    assert {47.0, 101.0, 127.0} <= set(np.unique(g).tolist())
    return g


def importance(cols, seed):
    x = synth.activations(512, cols, seed=seed)
    s2, cn, _ = oracle.imatrix_accumulate(x, np.zeros((512, 1), np.int32), 1)
    return oracle.imatrix_weights(s2, cn)[0]


@pytest.mark.parametrize("fmt", ["IQ2_XXS", "IQ2_XS", "IQ2_S"])
def test_wide_grid_every_block_small_case(fmt):
    R, C = 77, 1024                                # 308 blocks: several CTAs and a ragged last quad
    store, wv = synth.as_dtype(synth.weight_t4(R, C, seed=41), "bf16")
    grid = wide_grid(fmt)
    imp = importance(C, 42)
    g = torch.from_numpy(grid).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    p = api.encode(fmt, dev_bf16(store), g, importance=torch.from_numpy(imp).to(DEV), status=st)
    p_orc, st_orc, det = oracle.encode(fmt, wv, grid, importance=imp, details=True)
    assert int(st.item()) == st_orc == 0
    assert check_payload(fmt, wv, grid, p.cpu().numpy(), p_orc, det, importance=imp) == 0, "not byte-identical"
    # fixed choices (random per group) on the same grid
    info = oracle.format_info(fmt)
    ch = np.random.default_rng(43).integers(0, info["num_choices"], (R * C // 256, info["groups"])).astype(np.uint8)
    pf = api.encode(fmt, dev_bf16(store), g, importance=torch.from_numpy(imp).to(DEV),
                    choices=torch.from_numpy(ch).to(DEV))
    pf_orc, _ = oracle.encode(fmt, wv, grid, importance=imp, choices=ch)
    assert np.array_equal(pf.cpu().numpy(), pf_orc)


@pytest.mark.parametrize("fmt", ["IQ2_XS", "IQ2_S"])
def test_wide_grid_sampled_rows_full_size(fmt):
    R, C = 5632, 2048
    store, wv = synth.as_dtype(synth.weight_t4(R, C, seed=1), "bf16")
    grid = wide_grid(fmt)
    imp = importance(C, 44)
    p = api.encode(fmt, dev_bf16(store), torch.from_numpy(grid).to(DEV), importance=torch.from_numpy(imp).to(DEV))
    bpr = C // 256
    rows = np.linspace(0, R - 1, 12).astype(np.int64)
    sel = (rows[:, None] * bpr + np.arange(bpr)[None, :]).ravel()
    p_orc, _, det = oracle.encode(fmt, wv[rows], grid, importance=imp, details=True)
    assert check_payload(fmt, wv[rows], grid, p.cpu().numpy()[sel], p_orc, det, importance=imp) == 0
