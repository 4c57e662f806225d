"""GPU parity: every library call (through the C ABI) against the oracle on the same seeded inputs.

Bars: decode, anchor, imatrix sums/counts and weights bit-exact; encoded payloads bit-exact except
under the near-tie rule (tests/parity.py); every-choice error tables within the bound stated in
include/iq.h.  Sizes span several CTAs and a ragged tail; the full-size cases run the benchmark's
launch configuration and compare sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from ggml_iq_codebook_accumulate_b300 import api, synth
from parity import check_payload

pytestmark = pytest.mark.gpu
FORMATS = synth.FORMATS
DEV = "cuda:0"


def dev_tensor(store, dtype):
    """numpy storage (fp32 values or bf16 bit patterns) -> CUDA tensor"""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(DEV)
    return torch.from_numpy(np.ascontiguousarray(store)).to(DEV)


def host(t):
    return t.detach().cpu().numpy()


def importance_from_acts(cols, seed, tokens=512):
    x = synth.activations(tokens, cols, seed=seed)
    s2, cn, _ = oracle.imatrix_accumulate(x, np.zeros((tokens, 1), np.int32), 1)
    return oracle.imatrix_weights(s2, cn)[0]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    api.lib()
    yield


# ---- decode ---------------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_random_payloads(fmt, out_dtype):
    info = oracle.format_info(fmt)
    rng = np.random.default_rng(FORMATS.index(fmt))
    rows, cols = 37, 768                       # 111 blocks: several CTAs, ragged tail
    B = rows * cols // 256
    p = rng.integers(0, 256, (B, info["block_bytes"]), dtype=np.uint8)
    # keep the fp16 scale finite and positive
    d16 = rng.integers(0x0400, 0x3c00, B).astype(np.uint16)
    if fmt == "IQ1_M":
        for k in range(4):
            w = p[:, 48 + 2 * k].astype(np.uint16) | (p[:, 49 + 2 * k].astype(np.uint16) << 8)
            w = (w & 0x0FFF) | (((d16 >> (4 * k)) & 0xF) << 12)
            p[:, 48 + 2 * k] = w & 0xFF; p[:, 49 + 2 * k] = w >> 8
    else:
        p[:, 0] = d16 & 0xFF; p[:, 1] = d16 >> 8
    grid = synth.grid(fmt)
    ref = oracle.decode(fmt, p, rows, cols, grid)
    out = api.decode(fmt, torch.from_numpy(p).to(DEV), rows, cols, torch.from_numpy(grid).to(DEV), dtype=out_dtype)
    got = host(out.float())
    if out_dtype == torch.float32:
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    else:
        assert np.array_equal(got, torch.from_numpy(ref).to(torch.bfloat16).float().numpy())


def test_decode_hand_assembled_fixtures():
    from test_oracle_codec import load_fixtures, semantic_values
    for fmt, fields, payload in load_fixtures():
        grid = synth.grid(fmt)
        out = api.decode(fmt, torch.from_numpy(payload.copy()[None, :]).to(DEV), 1, 256, torch.from_numpy(grid).to(DEV))
        assert np.array_equal(host(out)[0], semantic_values(fmt, fields, grid))


# ---- imatrix --------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,C,E,K,R", [(2500, 192, 16, 4, 1024), (777, 64, 5, 2, 300), (4096, 128, 128, 8, 1024),
                                       (300, 256, 200, 3, 64), (600, 14336, 16, 2, 256), (301, 7168, 9, 3, 128),
                                       (130, 14400, 1, 1, 1024), (1500, 14336, 16, 3, 256),
                                       (3000, 320, 1, 1, 256), (4096, 2048, 1, 1, 1024)])
def test_imatrix_bit_exact(dtype, T, C, E, K, R):
    """Both launch layouts: few column tiles (chunks in parallel, partials combined in chunk order)
    and many tiles (one CTA walks a tile's chunks in order); ragged chunks and column tiles; many
    chunks of two stages each, where consumer warps drift a whole chunk apart (each expert's sums
    must keep one owner warp so their chunk-order additions stay ordered); the one-expert (dense)
    layout, with a ragged tile and with the bench's 4096 x 2048 pass."""
    x32 = synth.activations(T, C, seed=T + C)
    store, xv = synth.as_dtype(x32, dtype)
    ids = synth.router(T, E, K, idle=max(1, E // 16) if E > 1 else 0, seed=E + K)
    s0 = (np.random.default_rng(3).random((E, C)) * 5).astype(np.float32)   # accumulate into existing sums
    c0 = np.random.default_rng(4).integers(0, 50, E).astype(np.int64)
    ref_s, ref_c, ref_st = oracle.imatrix_accumulate(xv, ids, E, rows_per_chunk=R, in_sum2=s0, counts=c0)
    s2 = torch.from_numpy(s0.copy()).to(DEV)
    cn = torch.from_numpy(c0.copy()).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.imatrix_accumulate(dev_tensor(store, dtype), torch.from_numpy(ids).to(DEV), E, R, s2, cn, status=st)
    assert np.array_equal(host(s2).view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(host(cn), ref_c)
    assert int(st.item()) == ref_st


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_imatrix_tiny_values_round_the_square_first(dtype):
    """Activations near 2^-70, whose squares fall below fp32's normal range and round there: the
    sums must take the square's rounding before the addition's, as the definition does (a fused
    multiply-add rounds once and differs on such inputs)."""
    rng = np.random.default_rng(11)
    T, C, E = 300, 192, 3
    mant = rng.integers(128, 256, (T, C)).astype(np.float64) / 128.0
    x32 = (mant * np.exp2(rng.integers(-76, -64, (T, C))) * rng.choice([-1.0, 1.0], (T, C))).astype(np.float32)
    store, xv = synth.as_dtype(x32, dtype)
    ids = np.stack([rng.permutation(E)[:2] for _ in range(T)]).astype(np.int32)
    ref_s, ref_c, _ = oracle.imatrix_accumulate(xv, ids, E, rows_per_chunk=128)
    # what one rounding per row would give: the values have 8 significant bits, so x^2 and every
    # partial + x^2 below 2^-100 are exact in fp64 and the cast to fp32 is the single rounding
    fused = np.zeros_like(ref_s)
    for k0 in range(0, T, 128):
        part = np.zeros_like(ref_s)
        for t in range(k0, min(T, k0 + 128)):
            for e in ids[t]:
                part[e] = (part[e].astype(np.float64) + xv[t].astype(np.float64) ** 2).astype(np.float32)
        fused = fused + part
    assert not np.array_equal(fused, ref_s)              # the case does tell the two apart
    s2, cn = api.imatrix_accumulate(dev_tensor(store, dtype), torch.from_numpy(ids).to(DEV), E, 128)
    assert np.array_equal(host(s2).view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(host(cn), ref_c)


def test_imatrix_status_and_sets():
    x = synth.activations(64, 128, seed=5)
    ids = np.tile(np.array([[0, 1]], np.int32), (64, 1))
    ids[3] = [0, 9]
    ids[5] = [1, 1]
    ids[6] = [-1, 2]
    ref_s, ref_c, ref_st = oracle.imatrix_accumulate(x, ids, 4)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    s2, cn = api.imatrix_accumulate(torch.from_numpy(x).to(DEV), torch.from_numpy(ids).to(DEV), 4, status=st)
    assert np.array_equal(host(s2), ref_s) and np.array_equal(host(cn), ref_c)
    assert int(st.item()) == ref_st == (oracle.ST_BAD_EXPERT_ID | oracle.ST_DUP_EXPERT_ID)
    xn = x.copy(); xn[7, 3] = np.inf
    st.zero_()
    api.imatrix_accumulate(torch.from_numpy(xn).to(DEV), torch.zeros(64, 1, dtype=torch.int32, device=DEV), 4, status=st)
    assert int(st.item()) & api.STATUS_BITS["NONFINITE_SUM2"]
    # one expert (the dense layout): ids other than 0 are skipped and reported, a non-finite value
    # reaches the sums and is reported
    x1 = synth.activations(700, 128, seed=6)
    ids1 = np.zeros((700, 1), np.int32)
    ids1[[5, 300, 650]] = [[1], [-1], [7]]
    ref_s, ref_c, ref_st = oracle.imatrix_accumulate(x1, ids1, 1, rows_per_chunk=256)
    st.zero_()
    s2, cn = api.imatrix_accumulate(torch.from_numpy(x1).to(DEV), torch.from_numpy(ids1).to(DEV), 1, 256, status=st)
    assert np.array_equal(host(s2).view(np.uint32), ref_s.view(np.uint32)) and np.array_equal(host(cn), ref_c)
    assert int(st.item()) == ref_st == oracle.ST_BAD_EXPERT_ID
    x1[10, 7] = np.nan
    st.zero_()
    api.imatrix_accumulate(torch.from_numpy(x1).to(DEV), torch.from_numpy(ids1).to(DEV), 1, 256, status=st)
    assert int(st.item()) & api.STATUS_BITS["NONFINITE_SUM2"]


def test_weights_bit_exact():
    rng = np.random.default_rng(6)
    s2 = (rng.random((7, 320)) * 50).astype(np.float32)
    cn = np.array([0, 1, 3, 1000, 0, 7, 4096], np.int64)
    for floor in (0.0, 10.0):
        ref = oracle.imatrix_weights(s2, cn, floor)
        got = api.imatrix_weights(torch.from_numpy(s2).to(DEV), torch.from_numpy(cn).to(DEV), floor)
        assert np.array_equal(host(got).view(np.uint32), ref.view(np.uint32))


def test_imatrix_full_size_routed_moe():
    """4096 tokens x 17408-wide bf16 activations, 128 experts, Zipf(1.2) top-8 with 8 idle experts,
    1024-row chunks: sums and counts bit-exact over the whole [128, 17408] statistic."""
    T, C, E = 4096, 17408, 128
    store, xv = synth.as_dtype(synth.activations(T, C, seed=2), "bf16")
    ids = synth.router(T, E, 8, seed=2)
    ref_s, ref_c, _ = oracle.imatrix_accumulate(xv, ids, E)
    s2, cn = api.imatrix_accumulate(dev_tensor(store, "bf16"), torch.from_numpy(ids).to(DEV), E)
    assert np.array_equal(host(cn), ref_c)
    assert (ref_c == 0).sum() >= 8
    assert np.array_equal(host(s2).view(np.uint32), ref_s.view(np.uint32))


# ---- anchor ---------------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_anchor_bit_exact(fmt, dtype):
    store, wv = synth.as_dtype(synth.weight_t4(29, 1024, seed=7), dtype)
    wv = wv.copy(); store = store.copy()
    store.reshape(-1)[256 * 5: 256 * 6] = 0                  # an all-zero block
    wv.reshape(-1)[256 * 5: 256 * 6] = 0
    ref, _ = oracle.anchor_scales(fmt, wv)
    got = api.anchor_scales(fmt, dev_tensor(store, dtype))
    assert np.array_equal(host(got).view(np.uint16), ref)


# ---- encode ---------------------------------------------------------------------------------

def _encode_case(fmt, dtype, rows, cols, seed, rpe=0, experts=1, choices=None, every=False, d16=False):
    store, wv = synth.as_dtype(synth.weight_t4(rows, cols, seed=seed), dtype)
    if rpe:
        imp = np.stack([importance_from_acts(cols, seed + 100 + e) for e in range(experts)])
    else:
        imp = importance_from_acts(cols, seed + 100)
    grid = synth.grid(fmt)
    d16v = oracle.anchor_scales(fmt, wv)[0] if d16 else None
    p_orc, st_orc, det = oracle.encode(fmt, wv, grid, importance=imp, rows_per_expert=rpe, d16=d16v, choices=choices,
                                       details=True)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(importance=torch.from_numpy(imp).to(DEV), rows_per_expert=rpe, status=st,
              d16=None if d16v is None else torch.from_numpy(d16v.view(np.int16)).to(DEV),
              choices=None if choices is None else torch.from_numpy(choices).to(DEV), every_choice=every)
    out = api.encode(fmt, dev_tensor(store, dtype), torch.from_numpy(grid).to(DEV), **kw)
    torch.cuda.synchronize()
    return wv, imp, grid, out, p_orc, st_orc, det, int(st.item())


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_encode_searched_matches_oracle(fmt, dtype):
    wv, imp, grid, p, p_orc, st_orc, det, st = _encode_case(fmt, dtype, 75, 512, seed=11)   # 150 blocks
    assert st == st_orc == 0
    check_payload(fmt, wv, grid, host(p), p_orc, det, importance=imp)


@pytest.mark.parametrize("fmt", FORMATS)
def test_encode_given_scales_and_fixed_choices(fmt):
    info = oracle.format_info(fmt)
    rows, cols = 41, 512
    B = rows * cols // 256
    ch7 = np.full((B, info["groups"]), 7, np.uint8)
    wv, imp, grid, p, p_orc, _, det, st = _encode_case(fmt, "bf16", rows, cols, seed=12, choices=ch7, d16=True)
    assert st == 0
    check_payload(fmt, wv, grid, host(p), p_orc, det, importance=imp)
    rnd = np.random.default_rng(13).integers(0, info["num_choices"], (B, info["groups"])).astype(np.uint8)
    wv, imp, grid, p, p_orc, _, det, st = _encode_case(fmt, "bf16", rows, cols, seed=12, choices=rnd)
    check_payload(fmt, wv, grid, host(p), p_orc, det, importance=imp)


@pytest.mark.parametrize("fmt", FORMATS)
def test_every_choice_table_and_payload(fmt):
    wv, imp, grid, (p, tbl), p_orc, _, det, st = _encode_case(fmt, "bf16", 33, 768, seed=14, every=True)
    check_payload(fmt, wv, grid, host(p), p_orc, det, importance=imp)
    t = host(tbl).astype(np.float64)
    ref = det["table"]
    info = oracle.format_info(fmt)
    vpg = info["vectors_per_group"]
    cs = (imp.reshape(1, -1, 8).astype(np.float64) * wv.reshape(wv.shape[0], -1, 8).astype(np.float64) ** 2).sum(-1)
    Cg = cs.reshape(-1, info["groups"], vpg).sum(-1)[:, :, None]
    bound = 2.0 ** -17 * (4 * Cg + 2 * ref)
    assert np.all(np.abs(t - ref) <= bound)
    # the table-only call gives the same table
    tbl2 = api.group_errors(fmt, dev_tensor(synth.as_dtype(wv, "bf16")[0], "bf16"), torch.from_numpy(grid).to(DEV),
                            importance=torch.from_numpy(imp).to(DEV))
    assert torch.equal(tbl2, tbl)


@pytest.mark.parametrize("fmt", ["IQ2_XXS", "IQ1_M"])
def test_moe_experts_and_idle_expert(fmt):
    """Per-expert importance rows (row r uses expert r / rows_per_expert); an idle expert's weight 1
    gives the same bytes as encoding without importance."""
    E, rpe, cols = 4, 6, 512
    store, wv = synth.as_dtype(synth.weight_t4(E * rpe, cols, seed=15), "bf16")
    x = synth.activations(256, cols, seed=16)
    ids = np.tile(np.array([[0, 2, 3]], np.int32), (256, 1))
    s2, cn = api.imatrix_accumulate(torch.from_numpy(x).to(DEV), torch.from_numpy(ids).to(DEV), E)
    w = api.imatrix_weights(s2, cn)
    grid = synth.grid(fmt)
    g = torch.from_numpy(grid).to(DEV)
    p = host(api.encode(fmt, dev_tensor(store, "bf16"), g, importance=w, rows_per_expert=rpe))
    p_plain = host(api.encode(fmt, dev_tensor(store, "bf16"), g))
    bpr = cols // 256
    assert np.array_equal(p[rpe * bpr:2 * rpe * bpr], p_plain[rpe * bpr:2 * rpe * bpr])
    p_orc, _, det = oracle.encode(fmt, wv, grid, importance=host(w), rows_per_expert=rpe, details=True)
    check_payload(fmt, wv, grid, p, p_orc, det, importance=host(w), rows_per_expert=rpe)


def test_bad_units_zeroed_and_reported():
    fmt = "IQ2_XS"
    store, wv = synth.as_dtype(synth.weight_t4(1, 1024, seed=17), "f32")
    wv = wv.copy(); wv[0, 5] = np.inf
    imp = np.ones(1024, np.float32); imp[600] = -1.0
    ch = np.zeros((4, 16), np.uint8); ch[3, 2] = 16
    grid = synth.grid(fmt)
    p_orc, st_orc = oracle.encode(fmt, wv, grid, importance=imp, choices=ch)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    p = api.encode(fmt, torch.from_numpy(wv).to(DEV), torch.from_numpy(grid).to(DEV), importance=torch.from_numpy(imp).to(DEV),
                   choices=torch.from_numpy(ch).to(DEV), status=st)
    assert int(st.item()) == st_orc
    assert np.array_equal(host(p), p_orc)
    bad_grid = grid.copy(); bad_grid[3, 1] = 7.5
    st.zero_()
    p = api.encode(fmt, torch.from_numpy(wv[:, 256:].copy()).to(DEV), torch.from_numpy(bad_grid).to(DEV), status=st)
    assert int(st.item()) & api.STATUS_BITS["BAD_GRID"] and not host(p).any()


def test_zero_blocks_and_empty():
    fmt = "IQ1_S"
    store, wv = synth.as_dtype(synth.weight_t4(3, 512, seed=18), "bf16")
    store = store.copy(); store[1, :256] = 0
    grid = torch.from_numpy(synth.grid(fmt)).to(DEV)
    p = host(api.encode(fmt, dev_tensor(store, "bf16"), grid))
    assert not p[2].any() and p[0].any()
    e = api.encode(fmt, torch.empty(0, 512, dtype=torch.bfloat16, device=DEV), grid)
    assert e.shape == (0, 50)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("mode", ["searched", "fixed"])
def test_zero_importance_vectors_tie_exactly(fmt, mode):
    # importance 0 over whole 8-column vectors (one vector, a whole choice group, scattered
    # columns): every codebook entry then has error exactly 0 for such a vector, so the exact
    # rescoring sees more candidates within its bound than it lists at once and takes its
    # per-unit path; the lowest key (and, for a tied group, the lowest choice) must win as in the
    # oracle, bit for bit
    info = oracle.format_info(fmt)
    store, wv = synth.as_dtype(synth.weight_t4(6, 1024, seed=21), "bf16")
    imp = importance_from_acts(1024, seed=22).copy()
    imp[0:8] = 0; imp[256:288] = 0; imp[520:528] = 0; imp[768:1024:3] = 0
    grid = synth.grid(fmt)
    ch = None
    if mode == "fixed":
        rng = np.random.default_rng(23)
        ch = rng.integers(0, info["num_choices"], (6 * 4, info["groups"])).astype(np.uint8)
    p_orc, st_orc = oracle.encode(fmt, wv, grid, importance=imp, choices=ch)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    p = api.encode(fmt, dev_tensor(store, "bf16"), torch.from_numpy(grid).to(DEV), importance=torch.from_numpy(imp).to(DEV),
                   choices=None if ch is None else torch.from_numpy(ch).to(DEV), status=st)
    assert int(st.item()) == st_orc == 0
    assert np.array_equal(host(p), p_orc)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("mode", ["searched", "fixed"])
def test_zero_importance_vectors_many_flagged_blocks(fmt, mode):
    # every row's first vector has importance 0, so all 3072 rows' first blocks are flagged: more
    # items than resident warps, so each warp re-decides its own items; the tied vectors overflow
    # its candidate list, the other flagged groups fit it
    info = oracle.format_info(fmt)
    store, wv = synth.as_dtype(synth.weight_t4(3072, 512, seed=24), "bf16")
    imp = (np.abs(np.random.default_rng(25).standard_normal(512)) + 0.1).astype(np.float32)
    imp[0:8] = 0; imp[300:304] = 0
    grid = synth.grid(fmt)
    ch = None
    if mode == "fixed":
        ch = np.random.default_rng(26).integers(0, info["num_choices"], (3072 * 2, info["groups"])).astype(np.uint8)
    p_orc, st_orc = oracle.encode(fmt, wv, grid, importance=imp, choices=ch)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    p = api.encode(fmt, dev_tensor(store, "bf16"), torch.from_numpy(grid).to(DEV), importance=torch.from_numpy(imp).to(DEV),
                   choices=None if ch is None else torch.from_numpy(ch).to(DEV), status=st)
    assert int(st.item()) == st_orc == 0
    assert np.array_equal(host(p), p_orc)


def test_argument_errors_change_nothing():
    with pytest.raises(api.IQError):
        api.encode("IQ2_XXS", torch.zeros(2, 300, device=DEV), torch.from_numpy(synth.grid("IQ2_XXS")).to(DEV))


# ---- full-size, benchmark launch configuration, sampled rows ---------------------------------

@pytest.mark.parametrize("fmt", FORMATS)
def test_full_size_5632x2048_sampled(fmt):
    R, C = 5632, 2048
    store, wv = synth.as_dtype(synth.weight_t4(R, C, seed=1), "bf16")
    xs, xv = synth.as_dtype(synth.activations(4096, C, seed=1), "bf16")
    s2, cn = api.imatrix_accumulate(dev_tensor(xs, "bf16"), torch.zeros(4096, 1, dtype=torch.int32, device=DEV), 1)
    w = api.imatrix_weights(s2, cn)
    grid = synth.grid(fmt)
    p = host(api.encode(fmt, dev_tensor(store, "bf16"), torch.from_numpy(grid).to(DEV), importance=w[0]))
    rows = np.arange(0, R, 97)                                   # 59 sampled rows, 472 blocks
    bpr = C // 256
    sel = (rows[:, None] * bpr + np.arange(bpr)[None, :]).ravel()
    p_orc, _, det = oracle.encode(fmt, wv[rows], grid, importance=host(w[0]), details=True)
    check_payload(fmt, wv[rows], grid, p[sel], p_orc, det, importance=host(w[0]))
