"""CPU checks of the boundary: the shared library loads and exports every call include/iq.h declares,
and format constants agree with the oracle's (independently written) table."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_calls():
    src = open(os.path.join(ROOT, "include", "iq.h")).read()
    return sorted(set(re.findall(r"^IQ_API int (iq_\w+)\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    calls = declared_calls()
    for name in ("iq_imatrix_accumulate", "iq_encode", "iq_decode", "iq_group_errors", "iq_imatrix_weights",
                 "iq_anchor_scales", "iq_format_info"):
        assert name in calls


def test_library_loads_and_exports_every_declared_call():
    from ggml_iq_codebook_accumulate_b300 import api, build
    build.build()
    L = ctypes.CDLL(api.LIB_PATH)
    for name in declared_calls():
        assert hasattr(L, name), name
    assert set(declared_calls()) <= set(api.EXPORTS)


def test_format_info_matches_oracle(orc):
    from ggml_iq_codebook_accumulate_b300 import api
    for fmt in api.FORMATS:
        a = api.format_info(fmt)        # host-only call, no GPU needed
        o = orc.format_info(fmt)
        assert (a["block_bytes"], a["choice_groups"], a["num_choices"], a["grid_entries"], a["vectors_per_group"]) == \
            (o["block_bytes"], o["groups"], o["num_choices"], o["entries"], o["vectors_per_group"])
        assert a["block_bytes"] * 8 / 256 == {"IQ2_XXS": 2.0625, "IQ2_XS": 2.3125, "IQ2_S": 2.5625,
                                              "IQ1_S": 1.5625, "IQ1_M": 1.75}[fmt]


def test_host_only_size_queries_and_argument_checks():
    """Workspace and capacity queries run on the host alone; bad arguments are refused with
    IQ_ERR_ARG (-1) before any device work."""
    from ggml_iq_codebook_accumulate_b300 import api
    L = api.lib()
    n = ctypes.c_size_t()
    assert L.iq_imatrix_workspace_size(4096, 17408, api.IQ_BF16, 128, 8, 1024, ctypes.byref(n)) == 0 and n.value > 0
    assert L.iq_imatrix_workspace_size(4096, 17408, api.IQ_BF16, 128, 65, 1024, ctypes.byref(n)) == -1  # top_k > 64
    assert L.iq_imatrix_workspace_size(4096, 17408, api.IQ_BF16, 1025, 8, 1024, ctypes.byref(n)) == -1  # > 1024 experts
    assert L.iq_imatrix_workspace_size(4096, 17408, api.IQ_BF16, 128, 8, 4097, ctypes.byref(n)) == -1  # chunk too big
    assert L.iq_encode_workspace_size(0, 5632, 2048, ctypes.byref(n)) == 0 and n.value >= 256 + 256 * 64
    assert L.iq_encode_workspace_size(0, 5632, 2000, ctypes.byref(n)) == -1                           # cols % 256
    assert L.iq_encode_workspace_size(7, 1, 256, ctypes.byref(n)) == -1                               # no such format
    caps = {f: api.encode_static_scratch_capacity(f) for f in api.FORMATS}
    assert caps["IQ1_S"] == caps["IQ1_M"] == 114656 and caps["IQ2_XXS"] == 128992
    # the capacity is exactly what fits in the 1 MiB array
    for f in api.FORMATS:
        assert L.iq_encode_workspace_size(api.FMT_ID[f], caps[f], 256, ctypes.byref(n)) == 0 and n.value <= 1 << 20
        assert L.iq_encode_workspace_size(api.FMT_ID[f], caps[f] + 1, 256, ctypes.byref(n)) == 0 and n.value > 1 << 20


def test_local_hessian_host_checks():
    """The local-Hessian search needs no workspace (it decodes the payloads itself); bad arguments
    are refused on the host (no device pointer is touched: the checks fail first)."""
    from ggml_iq_codebook_accumulate_b300 import api
    L = api.lib()
    n = ctypes.c_size_t(7)
    assert L.iq_local_hessian_workspace_size(0, 5632, 2048, ctypes.byref(n)) == 0 and n.value == 0
    assert L.iq_local_hessian_workspace_size(4, 10, 512, ctypes.byref(n)) == 0 and n.value == 0
    assert L.iq_local_hessian_workspace_size(0, 10, 500, ctypes.byref(n)) == -1
    fake = 1 << 20                                   # never dereferenced: every call below is refused
    args = dict(f=0, W=fake, dt=api.IQ_BF16, rows=4, cols=512, grid=fake, pay=fake, H=fake, damp=0.3,
                ch=fake, st=None, ws=fake, wsb=1 << 30, stream=None)

    def call(**kw):
        a = {**args, **kw}
        return L.iq_local_hessian_choices(a["f"], a["W"], a["dt"], a["rows"], a["cols"], a["grid"], a["pay"], a["H"],
                                          a["damp"], a["ch"], a["st"], a["ws"], a["wsb"], a["stream"])

    assert call(damp=-0.1) == -1                     # negative damping
    assert call(damp=float("nan")) == -1
    assert call(cols=500) == -1                      # cols % 256
    assert call(f=9) == -1                           # no such format
    assert call(H=None) == -1 and call(pay=None) == -1 and call(ch=None) == -1
    assert call(H=fake + 4) == -1                    # Hessian not 16-byte aligned
    assert call(pay=fake + 1) == -1                  # payloads read as 16-bit words
    assert L.iq_encode_every_choice(0, fake, api.IQ_BF16, 4, 500, None, 0, fake, None, fake, None, fake, 1 << 30,
                                    None) == -1      # cols % 256


def test_imatrix_tools_and_write_back_host_checks():
    """Refused on the host: bad sizes, missing or aliasing pointers (never dereferenced)."""
    from ggml_iq_codebook_accumulate_b300 import api
    L = api.lib()
    a, b = 1 << 20, 1 << 21
    assert L.iq_imatrix_merge(a, a + 64, b, b + 64, 0, 256, None, None) == -1          # no experts
    assert L.iq_imatrix_merge(a, a + 64, a, b + 64, 4, 256, None, None) == -1          # source aliases destination
    assert L.iq_imatrix_merge(None, a + 64, b, b + 64, 4, 256, None, None) == -1
    assert L.iq_imatrix_neutral_entries(a, a + 64, 4, 0, None) == -1                   # no columns
    assert L.iq_imatrix_coverage(a, 0, b, None) == -1 and L.iq_imatrix_coverage(None, 4, b, None) == -1
    assert L.iq_encode_write_back(0, a, api.IQ_BF16, 4, 500, None, 0, b, None, None, a, None, b, 1 << 30,
                                  None) == -1                                          # cols % 256
