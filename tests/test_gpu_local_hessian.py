"""GPU parity of the every-choice payloads and the local-Hessian choice search (PR #3159, PR #3158)
against the oracle, through the C ABI.

The every-choice payloads follow the encoder's rule (bytes equal to the oracle's forced encodes,
near ties accepted as in tests/parity.py).  The search runs in fp32 against an fp64 oracle: its
picks must equal the oracle's, except in blocks where some decision of the oracle had two choices
within fp32 rounding of each other; there the block error of the device's picks must be within
1e-4 (relative) of the oracle's.  The tolerance comes from the fp32 evaluation of dw H' dw^T over a
256-value block (sums of at most 256 products of values that are each rounded once).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import local_hessian as lh
from ggml_iq_codebook_accumulate_b300 import api, synth
from parity import check_payload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
NEAR = 1e-4


def dev_bf16(store):
    return torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(DEV)


def correlated_hessian(C, n, seed, rho=0.85):
    rng = np.random.default_rng(seed)
    Z = rng.standard_normal((n, C))
    X = np.empty_like(Z)
    X[:, 0] = Z[:, 0]
    for j in range(1, C):
        X[:, j] = rho * X[:, j - 1] + np.sqrt(1 - rho * rho) * Z[:, j]
    X *= np.exp(0.5 * rng.standard_normal(C))[None, :]
    return X.T @ X / n


def blocks_of(H, C):
    return np.ascontiguousarray(np.stack([H[256 * j:256 * (j + 1), 256 * j:256 * (j + 1)] for j in range(C // 256)]),
                                dtype=np.float32)


def check_choices(fmt, Wv, grid, pay_orc, Hb, perc_damp, got):
    """Device picks against the oracle's: equal, or a block with a near tie in the oracle's own
    decisions whose device block error is within NEAR of the oracle's."""
    ref, traces = lh.local_hessian_choices(fmt, Wv, grid, pay_orc, Hb.astype(np.float64), perc_damp, trace=True)
    same = np.all(got == ref, axis=1)
    if same.all():
        return 0
    R, C = Wv.shape
    nb = C // 256
    G = oracle.format_info(fmt)["groups"]
    gs = 256 // G
    dw = lh.block_dw(fmt, Wv, grid, pay_orc)
    Hd = lh.damped_blocks(Hb.astype(np.float64), perc_damp)
    for b in np.nonzero(~same)[0]:
        r, j = divmod(int(b), nb)
        near = False
        for kind, g, errs, pick in traces[b]:
            srt = np.sort(errs)
            near |= (srt[1] - srt[0]) <= NEAR * (abs(srt[0]) + abs(srt[1]))
        assert near, f"block {b}: picks differ from the oracle's with no near tie ({got[b]} vs {ref[b]})"
        d = dw[:, r, 256 * j:256 * (j + 1)]
        e_dev = lh.block_error(np.concatenate([d[got[b, g], g * gs:(g + 1) * gs] for g in range(G)]), Hd[j])
        e_ref = lh.block_error(np.concatenate([d[ref[b, g], g * gs:(g + 1) * gs] for g in range(G)]), Hd[j])
        assert e_dev <= e_ref * (1 + NEAR) + 1e-30, f"block {b}: device error {e_dev} above {e_ref}"
    return int((~same).sum())


@pytest.mark.parametrize("fmt", synth.FORMATS)
def test_every_choice_payloads_are_the_forced_encodes(fmt):
    R, C = 24, 512
    store, wv = synth.as_dtype(synth.weight_t4(R, C, seed=21), "bf16")
    H = correlated_hessian(C, 2048, seed=21)
    imp = np.sqrt(np.diag(H)).astype(np.float32)
    grid = synth.grid(fmt)
    g = torch.from_numpy(grid).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pay = api.encode_every_choice(fmt, dev_bf16(store), g, importance=torch.from_numpy(imp).to(DEV), status=st)
    assert int(st.item()) == 0
    info = oracle.format_info(fmt)
    B = R * C // 256
    for c in range(info["num_choices"]):
        ch = np.full((B, info["groups"]), c, np.uint8)
        p_orc, _, det = oracle.encode(fmt, wv, grid, importance=imp, choices=ch, details=True)
        check_payload(fmt, wv, grid, pay[c].cpu().numpy(), p_orc, det, importance=imp)


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_decode_of_an_unaligned_payload(offset):
    """A payload slice at any byte offset decodes like the same bytes at an aligned address."""
    fmt, R, C = "IQ2_XS", 5, 768
    rng = np.random.default_rng(offset)
    info = oracle.format_info(fmt)
    B = R * C // 256
    raw = rng.integers(0, 256, size=(B, info["block_bytes"]), dtype=np.uint8)
    raw[:, 0:2] = np.frombuffer(np.float16(0.01).tobytes(), np.uint8)  # finite scales
    grid = synth.grid(fmt)
    g = torch.from_numpy(grid).to(DEV)
    buf = torch.zeros(raw.size + 8, dtype=torch.uint8, device=DEV)
    buf[offset:offset + raw.size] = torch.from_numpy(raw.ravel()).to(DEV)
    out = torch.empty(R, C, dtype=torch.float32, device=DEV)
    api._check(api.lib().iq_decode(api.FMT_ID[fmt], buf.data_ptr() + offset, R, C, g.data_ptr(), out.data_ptr(),
                                   api.IQ_F32, api._stream(out.device)), "iq_decode")
    assert np.array_equal(out.cpu().numpy(), oracle.decode(fmt, raw, R, C, grid))


@pytest.mark.parametrize("fmt", synth.FORMATS)
def test_local_hessian_search_matches_the_oracle(fmt):
    R, C = 40, 768                      # 3 column blocks, a ragged last row tile
    store, wv = synth.as_dtype(synth.weight_t4(R, C, seed=22), "bf16")
    H = correlated_hessian(C, 4096, seed=22)
    Hb = blocks_of(H, C)
    imp = np.sqrt(np.diag(H)).astype(np.float32)
    grid = synth.grid(fmt)
    g = torch.from_numpy(grid).to(DEV)
    W = dev_bf16(store)
    pay = api.encode_every_choice(fmt, W, g, importance=torch.from_numpy(imp).to(DEV))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = api.local_hessian_choices(fmt, W, g, pay, torch.from_numpy(Hb).to(DEV), 0.3, status=st).cpu().numpy()
    assert int(st.item()) == 0
    # the search is compared on the device's own every-choice payloads (checked against the forced
    # encodes above)
    assert check_choices(fmt, wv, grid, pay.cpu().numpy(), Hb, 0.3, got) <= 2


@pytest.mark.parametrize("fmt", ["IQ2_XXS", "IQ1_M"])
def test_identity_hessian_keeps_the_encoders_choices_on_device(fmt):
    """PR #3158 Testing, on the device: H = I with unit importance gives the searched choices."""
    R, C = 32, 512
    store, wv = synth.as_dtype(synth.weight_t4(R, C, seed=23), "bf16")
    grid = synth.grid(fmt)
    g = torch.from_numpy(grid).to(DEV)
    W = dev_bf16(store)
    pay = api.encode_every_choice(fmt, W, g)
    Hb = torch.from_numpy(np.stack([np.eye(256, dtype=np.float32)] * (C // 256))).to(DEV)
    got = api.local_hessian_choices(fmt, W, g, pay, Hb, 0.3).cpu().numpy()
    _, _, det = oracle.encode(fmt, wv, grid, details=True)
    assert np.array_equal(got, det["chosen"])


def test_local_hessian_full_size_sampled_rows():
    """The 5632 x 2048 bf16 weight in IQ2_S: device search over the whole weight, oracle on 24 rows
    spread over it (a row's picks depend only on that row and the Hessian)."""
    fmt, R, C = "IQ2_S", 5632, 2048
    store, wv = synth.as_dtype(synth.weight_t4(R, C, seed=24), "bf16")
    H = correlated_hessian(C, 4096, seed=24)
    Hb = blocks_of(H, C)
    imp = np.sqrt(np.diag(H)).astype(np.float32)
    grid = synth.grid(fmt)
    g = torch.from_numpy(grid).to(DEV)
    W = dev_bf16(store)
    pay = api.encode_every_choice(fmt, W, g, importance=torch.from_numpy(imp).to(DEV))
    got = api.local_hessian_choices(fmt, W, g, pay, torch.from_numpy(Hb).to(DEV), 0.3).cpu().numpy()
    rows = np.linspace(0, R - 1, 24).astype(np.int64)
    nb = C // 256
    sel = (rows[:, None] * nb + np.arange(nb)[None, :]).ravel()
    pay_dev = np.ascontiguousarray(pay.cpu().numpy()[:, sel])
    info = oracle.format_info(fmt)
    for c in (0, 7, 15):                     # the payloads of three choices against the forced encode
        ch = np.full((len(sel), info["groups"]), c, np.uint8)
        p_orc, _, det = oracle.encode(fmt, wv[rows], grid, importance=imp, choices=ch, details=True)
        check_payload(fmt, wv[rows], grid, pay_dev[c], p_orc, det, importance=imp)
    assert check_choices(fmt, wv[rows], grid, pay_dev, Hb, 0.3, got[sel]) <= 3


@pytest.mark.parametrize("fmt", ["IQ1_S", "IQ2_XS"])
def test_every_choice_payloads_full_size_sampled_rows(fmt):
    """The one-pass every-choice payloads of the 5632 x 2048 weight (importance from the 4096-row
    imatrix recipe) against the oracle's forced encodes on 16 rows spread over the weight, for
    every choice."""
    R, C = 5632, 2048
    store, wv = synth.as_dtype(synth.weight_t4(R, C, seed=25), "bf16")
    xs, xv = synth.as_dtype(synth.activations(4096, C, seed=25), "bf16")
    x = torch.from_numpy(np.ascontiguousarray(xs).view(np.int16)).view(torch.bfloat16).to(DEV)
    s2, cn = api.imatrix_accumulate(x, torch.zeros(4096, 1, dtype=torch.int32, device=DEV), 1)
    w = api.imatrix_weights(s2, cn)[0]
    grid = synth.grid(fmt)
    g = torch.from_numpy(grid).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pay = api.encode_every_choice(fmt, dev_bf16(store), g, importance=w, status=st)
    assert int(st.item()) == 0
    rows = np.linspace(0, R - 1, 16).astype(np.int64)
    nb = C // 256
    sel = (rows[:, None] * nb + np.arange(nb)[None, :]).ravel()
    pay_dev = pay.cpu().numpy()[:, sel]
    wh = w.cpu().numpy()
    info = oracle.format_info(fmt)
    for c in range(info["num_choices"]):
        ch = np.full((len(sel), info["groups"]), c, np.uint8)
        p_orc, _, det = oracle.encode(fmt, wv[rows], grid, importance=wh, choices=ch, details=True)
        check_payload(fmt, wv[rows], grid, pay_dev[c], p_orc, det, importance=wh)
