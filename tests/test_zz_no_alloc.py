"""The encoder entry point that allocates nothing (iq_encode_static_scratch).

It serves callers that may not allocate device memory: code running under CUDA-graph stream capture
in the global mode (cudaMalloc is refused there), plug-ins inside a framework that owns all device
memory through its own pool, and serving loops that may not block on an allocation.  Its scratch is
the library's fixed 1 MiB device array instead of a caller workspace; everything else matches
iq_encode.  These tests call it through the C ABI and compare it with iq_encode (which takes a
workspace) on two calls in a row, so a second call that read the first call's leftover scratch
would show up.  This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from ggml_iq_codebook_accumulate_b300 import api, synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bf16(store):
    return torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(DEV)


@pytest.mark.parametrize("fmt", ["IQ2_XXS", "IQ1_M"])
def test_static_scratch_matches_workspace_encode_twice(fmt):
    grid = torch.from_numpy(synth.grid(fmt)).to(DEV)
    for call, seed in enumerate((31, 32)):           # two calls in a row, different weights
        rows = 96 + 37 * call
        store, _ = synth.as_dtype(synth.weight_t4(rows, 1024, seed=seed), "bf16")
        W = _bf16(store)
        imp = torch.from_numpy(np.exp(np.random.default_rng(seed).standard_normal(1024)).astype(np.float32)).to(DEV)
        st_a = torch.zeros(1, dtype=torch.int32, device=DEV)
        st_b = torch.zeros(1, dtype=torch.int32, device=DEV)
        p_ref, t_ref = api.encode(fmt, W, grid, importance=imp, every_choice=True, status=st_a)
        p_new, t_new = api.encode_static_scratch(fmt, W, grid, importance=imp, every_choice=True, status=st_b)
        torch.cuda.synchronize()
        assert torch.equal(p_new, p_ref), f"payload differs on call {call}"
        assert torch.equal(t_new, t_ref), f"every-choice table differs on call {call}"
        assert int(st_a.item()) == int(st_b.item()) == 0
        # fixed choices through the same entry point
        B = rows * 4
        info = api.format_info(fmt)
        ch = torch.from_numpy(np.random.default_rng(seed).integers(0, info["num_choices"], (B, info["choice_groups"]))
                              .astype(np.uint8)).to(DEV)
        assert torch.equal(api.encode_static_scratch(fmt, W, grid, importance=imp, choices=ch),
                           api.encode(fmt, W, grid, importance=imp, choices=ch))


def test_static_scratch_rejects_too_large():
    fmt = "IQ1_S"
    cap = api.encode_static_scratch_capacity(fmt)
    assert cap == 114656
    grid = torch.from_numpy(synth.grid(fmt)).to(DEV)
    W = torch.zeros(cap + 1, 256, dtype=torch.bfloat16, device=DEV)
    payload = torch.full((cap + 1, 50), 7, dtype=torch.uint8, device=DEV)
    with pytest.raises(api.IQError, match="-4"):
        api.encode_static_scratch(fmt, W, grid, payload=payload)
    torch.cuda.synchronize()
    assert bool((payload == 7).all()), "a refused call must not write"
    ok = api.encode_static_scratch(fmt, W[:cap], grid)       # exactly at the limit is accepted
    torch.cuda.synchronize()
    assert not ok.any()                                       # all-zero weight -> all-zero payload
