"""GPU parity at the full sizes of the workloads the library is measured on, in the launch
configuration the benchmark uses, checked on sampled outputs the oracle computes one by one (the
small 256 x 1024 case in full).

* MoE expert encode: 128 experts x a fused gate/up weight [1536, 2048] bf16 (Student-t nu=4 x 0.02)
  in IQ2_XXS and IQ1_M, each expert weighted by its own imatrix (4096 routed tokens, top-8 from a
  Zipf(1.2) router with 8 idle experts, so idle experts get weight 1 on every channel).
* Large layers: [17408, 5120] and [5120, 17408] bf16 in all five formats, searched with the
  every-choice error table.
* The imatrix at its largest supported shape: 1024 experts, top-64, 4096-row chunks.
* The small case: a 256 x 1024 fp32 weight ~ N(0, 0.02) in IQ2_XXS, importance from 512 x 1024
  fp32 activations, every block against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from ggml_iq_codebook_accumulate_b300 import api, synth
from parity import check_payload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def dev_bf16(store):
    return torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(DEV)


def sample_blocks(rows, bpr, row_ids):
    return (np.asarray(row_ids)[:, None] * bpr + np.arange(bpr)[None, :]).ravel()


@pytest.fixture(scope="module")
def moe_importance():
    """Per-expert importance [128, 2048] from 4096 routed bf16 activations (GPU imatrix, checked
    bit for bit against the oracle here)."""
    T, C, E = 4096, 2048, 128
    xs, xv = synth.as_dtype(synth.activations(T, C, seed=3), "bf16")
    ids = synth.router(T, E, 8, seed=3)
    s2, cn = api.imatrix_accumulate(dev_bf16(xs), torch.from_numpy(ids).to(DEV), E)
    w = api.imatrix_weights(s2, cn)
    ref_s, ref_c, _ = oracle.imatrix_accumulate(xv, ids, E)
    ref_w = oracle.imatrix_weights(ref_s, ref_c)
    assert np.array_equal(cn.cpu().numpy(), ref_c)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref_w.view(np.uint32))
    idle = np.nonzero(ref_c == 0)[0]
    assert len(idle) >= 8
    return w, ref_w, idle


@pytest.mark.parametrize("fmt", ["IQ2_XXS", "IQ1_M"])
def test_moe_expert_encode_full_size(fmt, moe_importance):
    w, ref_w, idle = moe_importance
    E, R1, C = 128, 1536, 2048
    store, wv = synth.as_dtype(synth.weight_t4(E * R1, C, seed=3), "bf16")
    grid = synth.grid(fmt)
    g = torch.from_numpy(grid).to(DEV)
    W = dev_bf16(store)
    p = api.encode(fmt, W, g, importance=w, rows_per_expert=R1)
    # idle experts: weight 1 everywhere gives exactly the bytes of the unweighted search
    bpr = C // 256
    for e in idle[:3]:
        rs = slice(int(e) * R1, (int(e) + 1) * R1)
        plain = api.encode(fmt, W[rs], g)
        assert torch.equal(p[rs.start * bpr:rs.stop * bpr], plain)
    # sampled rows: the first and the last row of every expert
    rows = np.concatenate([np.arange(E) * R1, np.arange(E) * R1 + R1 - 1])
    rows.sort()
    sel = sample_blocks(E * R1, bpr, rows)
    ph = p.cpu().numpy()[sel]
    rpe_rows = rows // R1                       # expert of each sampled row
    imp_rows = ref_w[rpe_rows]                  # [n, C]: the sampled rows' importance, one row each
    p_orc, _, det = oracle.encode(fmt, wv[rows], grid, importance=imp_rows, rows_per_expert=1, details=True)
    check_payload(fmt, wv[rows], grid, ph, p_orc, det, importance=imp_rows, rows_per_expert=1)


@pytest.mark.parametrize("shape", [(17408, 5120), (5120, 17408)])
@pytest.mark.parametrize("fmt", synth.FORMATS)
def test_large_layers_every_choice_full_size(fmt, shape):
    R, C = shape
    store, wv = synth.as_dtype(synth.weight_t4(R, C, seed=4), "bf16")
    xs, xv = synth.as_dtype(synth.activations(4096, C, seed=4), "bf16")
    s2, cn = api.imatrix_accumulate(dev_bf16(xs), torch.zeros(4096, 1, dtype=torch.int32, device=DEV), 1)
    w = api.imatrix_weights(s2, cn)[0]
    grid = synth.grid(fmt)
    p, tbl = api.encode(fmt, dev_bf16(store), torch.from_numpy(grid).to(DEV), importance=w, every_choice=True)
    bpr = C // 256
    rows = np.linspace(0, R - 1, 9).astype(np.int64)      # 9 rows spread over the layer
    sel = sample_blocks(R, bpr, rows)
    wh = w.cpu().numpy()
    p_orc, _, det = oracle.encode(fmt, wv[rows], grid, importance=wh, details=True)
    check_payload(fmt, wv[rows], grid, p.cpu().numpy()[sel], p_orc, det, importance=wh)
    info = oracle.format_info(fmt)
    t = tbl.cpu().numpy()[sel].astype(np.float64)
    ref = det["table"]
    cs = (wh.reshape(1, -1, 8).astype(np.float64) * wv[rows].reshape(len(rows), -1, 8).astype(np.float64) ** 2).sum(-1)
    Cg = cs.reshape(-1, info["groups"], info["vectors_per_group"]).sum(-1)[:, :, None]
    assert np.all(np.abs(t - ref) <= 2.0 ** -17 * (4 * Cg + 2 * ref))


def test_imatrix_largest_supported_shape():
    """1024 experts, top-64 distinct ids per token, 4096-row chunks (the header's limits)."""
    T, C, E, K, R = 4096, 256, 1024, 64, 4096
    store, xv = synth.as_dtype(synth.activations(T, C, seed=5), "bf16")
    ids = synth.router(T, E, K, idle=64, seed=5)
    ref_s, ref_c, ref_st = oracle.imatrix_accumulate(xv, ids, E, rows_per_chunk=R)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    s2, cn = api.imatrix_accumulate(dev_bf16(store), torch.from_numpy(ids).to(DEV), E, R, status=st)
    assert np.array_equal(cn.cpu().numpy(), ref_c)
    assert np.array_equal(s2.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert int(st.item()) == ref_st == 0


def test_small_case_256x1024_whole_payload():
    """IQ2_XXS of a 256 x 1024 fp32 weight ~ N(0, 0.02) (seed 0); importance sqrt(in_sum2 / count)
    per column from 512 x 1024 fp32 activations (N(0, 1) x log-normal column scales, one expert
    every token reaches), through the GPU imatrix; the whole payload and its decode against the
    oracle."""
    R, C, T = 256, 1024, 512
    W = synth.weight_normal(R, C, seed=0)
    xs, xv = synth.as_dtype(synth.activations(T, C, seed=0), "f32")
    ids = np.zeros((T, 1), np.int32)
    s2, cn = api.imatrix_accumulate(torch.from_numpy(xs).to(DEV), torch.from_numpy(ids).to(DEV), 1)
    w = api.imatrix_weights(s2, cn)
    ref_s, ref_c, _ = oracle.imatrix_accumulate(xv, ids, 1)
    ref_w = oracle.imatrix_weights(ref_s, ref_c)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref_w.view(np.uint32))
    grid = synth.grid("IQ2_XXS")
    g = torch.from_numpy(grid).to(DEV)
    p = api.encode("IQ2_XXS", torch.from_numpy(W).to(DEV), g, importance=w[0])
    p_orc, _, det = oracle.encode("IQ2_XXS", W, grid, importance=ref_w[0], details=True)
    check_payload("IQ2_XXS", W, grid, p.cpu().numpy(), p_orc, det, importance=ref_w[0])
    q = api.decode("IQ2_XXS", p, R, C, g)
    assert np.array_equal(q.cpu().numpy(), oracle.decode("IQ2_XXS", p.cpu().numpy(), R, C, grid))
