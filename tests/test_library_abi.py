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
