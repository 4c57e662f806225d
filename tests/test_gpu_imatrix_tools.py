"""GPU parity of imatrix merging, neutral entries, coverage and the encode-and-write-back call
against the oracle, through the C ABI (bit-exact: every result has a single rounding or none)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import imatrix_tools as it
from ggml_iq_codebook_accumulate_b300 import api, synth
from parity import check_payload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def stats(T, C, E, K, idle, seed):
    xs, xv = synth.as_dtype(synth.activations(T, C, seed=seed), "bf16")
    ids = synth.router(T, E, K, idle=idle, seed=seed)
    x = torch.from_numpy(np.ascontiguousarray(xs).view(np.int16)).view(torch.bfloat16).to(DEV)
    s2, cn = api.imatrix_accumulate(x, torch.from_numpy(ids).to(DEV), E)
    return s2, cn


def test_merge_bit_exact_and_status():
    s2a, cna = stats(700, 1024, 24, 4, 3, 41)
    s2b, cnb = stats(900, 1024, 24, 4, 6, 42)
    ref_s, ref_c = it.merge(s2a.cpu().numpy(), cna.cpu().numpy(), s2b.cpu().numpy(), cnb.cpu().numpy())
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.imatrix_merge(s2a, cna, s2b, cnb, status=st)
    assert np.array_equal(s2a.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(cna.cpu().numpy(), ref_c) and int(st.item()) == 0
    # a sum that overflows is reported
    big = torch.full((2, 256), 3e38, dtype=torch.float32, device=DEV)
    api.imatrix_merge(big, torch.ones(2, dtype=torch.int64, device=DEV), big.clone(),
                      torch.ones(2, dtype=torch.int64, device=DEV), status=st)
    assert int(st.item()) & api.STATUS_BITS["NONFINITE_SUM2"]


def test_neutral_entries_and_coverage():
    s2, cn = stats(1500, 512, 40, 4, 7, 43)
    ref_cov = it.coverage(cn.cpu().numpy())
    assert tuple(api.imatrix_coverage(cn).cpu().tolist()) == ref_cov
    assert ref_cov[0] == 33 and ref_cov[1] == 1500 * 4
    ref_s, ref_c = it.neutral_entries(s2.cpu().numpy(), cn.cpu().numpy())
    api.imatrix_neutral_entries(s2, cn)
    assert np.array_equal(s2.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(cn.cpu().numpy(), ref_c)
    assert tuple(api.imatrix_coverage(cn).cpu().tolist()) == (40, 1500 * 4 + 7, 1, ref_cov[3])


@pytest.mark.parametrize("fmt", synth.FORMATS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_encode_write_back(fmt, dtype):
    """The fused write-back: the payload is the oracle's encode of the original W (byte-identical),
    and W is overwritten with its decode (exact in fp32, rounded to nearest even in bf16), for
    searched and for fixed choices; a zero block and a block with a non-finite value decode to
    zeros."""
    R, C = 24, 768
    x = synth.weight_t4(R, C, seed=44)
    x[3, 256:512] = 0.0                                     # zero-scale block
    x[5, 7] = np.nan                                        # rejected block (non-finite value)
    store, wv = synth.as_dtype(x, dtype)
    grid = synth.grid(fmt)
    g = torch.from_numpy(grid).to(DEV)
    imp_np = (np.random.default_rng(45).random(C) + 0.5).astype(np.float32)
    imp = torch.from_numpy(imp_np).to(DEV)
    info = oracle.format_info(fmt)
    ch = np.random.default_rng(46).integers(0, info["num_choices"], (R * C // 256, info["groups"])).astype(np.uint8)
    for choices in (None, ch):
        if dtype == "bf16":
            W = torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(DEV)
        else:
            W = torch.from_numpy(np.ascontiguousarray(store)).to(DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        pay = api.encode_write_back(fmt, W, g, importance=imp, status=st,
                                    choices=None if choices is None else torch.from_numpy(choices).to(DEV))
        p_orc, st_orc, det = oracle.encode(fmt, wv, grid, importance=imp_np, choices=choices, details=True)
        assert int(st.item()) == st_orc == oracle.ST_BAD_INPUT
        ph = pay.cpu().numpy()
        if choices is None:
            assert check_payload(fmt, wv, grid, ph, p_orc, det, importance=imp_np) == 0
        else:
            assert np.array_equal(ph, p_orc)
        q = oracle.decode(fmt, ph, R, C, grid)
        assert not q[3, 256:512].any() and not q[5, :256].any()
        if dtype == "f32":
            assert np.array_equal(W.cpu().numpy().view(np.uint32), q.view(np.uint32))
        else:
            ref = torch.from_numpy(q).to(torch.bfloat16)           # round to nearest even (CPU conversion)
            assert torch.equal(W.cpu().view(torch.int16), ref.view(torch.int16))
