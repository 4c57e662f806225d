"""Plain CPU oracle for the IQ codebook encoder, decoder and imatrix statistic.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may load it; the library never does.  The arithmetic lives in ``iq_oracle.c`` (plain C, fp64
direct-form errors), compiled by :func:`build` with ``-ffp-contract=off`` so that every fp32
multiply and add is rounded separately, as written.  This module only marshals numpy arrays.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against brute force,
closed forms, library routines or hand-assembled fixtures; see each test's docstring.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "iq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

FORMATS = ("IQ2_XXS", "IQ2_XS", "IQ2_S", "IQ1_S", "IQ1_M")
FMT_ID = {n: i for i, n in enumerate(FORMATS)}

ST_BAD_CHOICE = 1
ST_BAD_EXPERT_ID = 2
ST_NONFINITE_SUM2 = 4
ST_DUP_EXPERT_ID = 8
ST_BAD_INPUT = 16
ST_BAD_IMPORTANCE = 32
ST_BAD_SCALE = 64
ST_BAD_GRID = 128


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", _LIB_PATH + ".tmp", _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


_lib = None


def _L():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        _lib.or_format_info.argtypes = [i32] + [ctypes.POINTER(ctypes.c_int)] * 5
        _lib.or_half_from_float_n.argtypes = [p, p, i64]
        _lib.or_float_from_half_n.argtypes = [p, p, i64]
        _lib.or_imatrix_accumulate.argtypes = [p, i64, i64, p, i32, i32, i64, p, p, p]
        _lib.or_imatrix_weights.argtypes = [p, p, i32, i64, ctypes.c_float, p]
        _lib.or_anchor_scales.argtypes = [i32, p, i64, i64, p, p]
        _lib.or_encode.argtypes = [i32, p, i64, i64, p, i64, p, p, p, p, p, p, p, p, p, p, p, i32, i32]
        _lib.or_decode.argtypes = [i32, p, i64, i64, p, p]
        _lib.or_payload_errors.argtypes = [i32, p, i64, i64, p, i64, p, p, p, p]
        for fn in ("or_format_info", "or_imatrix_accumulate", "or_imatrix_weights", "or_anchor_scales",
                   "or_encode", "or_decode", "or_payload_errors"):
            getattr(_lib, fn).restype = ctypes.c_int
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def format_info(fmt: str) -> dict:
    vals = [ctypes.c_int() for _ in range(5)]
    rc = _L().or_format_info(FMT_ID[fmt], *[ctypes.byref(v) for v in vals])
    assert rc == 0
    bb, g, c, n, vpg = (v.value for v in vals)
    return dict(block_bytes=bb, groups=g, num_choices=c, entries=n, vectors_per_group=vpg)


def half_from_float(x: np.ndarray) -> np.ndarray:
    x = _f32(x).ravel()
    out = np.empty(x.size, np.uint16)
    _L().or_half_from_float_n(_ptr(x), _ptr(out), x.size)
    return out


def float_from_half(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.empty(h.size, np.float32)
    _L().or_float_from_half_n(_ptr(h), _ptr(out), h.size)
    return out


def imatrix_accumulate(x, ids, num_experts, rows_per_chunk=1024, in_sum2=None, counts=None):
    """Returns (in_sum2 [E, cols] f32, counts [E] i64, status); accumulates into copies of the
    given buffers.  ``x`` holds the activations as fp32 (bf16 inputs converted exactly)."""
    x = _f32(x)
    T, C = x.shape
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    top_k = ids.shape[1]
    s2 = np.zeros((num_experts, C), np.float32) if in_sum2 is None else np.array(in_sum2, np.float32)
    cn = np.zeros(num_experts, np.int64) if counts is None else np.array(counts, np.int64)
    st = np.zeros(1, np.int32)
    rc = _L().or_imatrix_accumulate(_ptr(x), T, C, _ptr(ids), top_k, num_experts, rows_per_chunk,
                                    _ptr(s2), _ptr(cn), _ptr(st))
    assert rc == 0, rc
    return s2, cn, int(st[0])


def imatrix_weights(in_sum2, counts, floor=0.0):
    s2 = _f32(in_sum2)
    cn = np.ascontiguousarray(counts, dtype=np.int64)
    E, C = s2.shape
    w = np.empty_like(s2)
    assert _L().or_imatrix_weights(_ptr(s2), _ptr(cn), E, C, float(floor), _ptr(w)) == 0
    return w


def anchor_scales(fmt, W):
    W = _f32(W)
    R, C = W.shape
    d16 = np.empty(R * (C // 256), np.uint16)
    st = np.zeros(1, np.int32)
    assert _L().or_anchor_scales(FMT_ID[fmt], _ptr(W), R, C, _ptr(d16), _ptr(st)) == 0
    return d16, int(st[0])


def encode(fmt, W, grid, importance=None, rows_per_expert=0, d16=None, choices=None, threads=0,
           details=False, entries=0):
    """Encode ``W`` [rows, cols] (fp32 values).  Returns payload [B, block_bytes] uint8 and the
    status word; with ``details`` also a dict of the fp64 error tables (see iq_oracle.c)."""
    info = format_info(fmt)
    W = _f32(W)
    R, C = W.shape
    B = R * (C // 256)
    G, NC = info["groups"], info["num_choices"]
    grid = _f32(grid)
    imp = _f32(importance)
    d16a = None if d16 is None else np.ascontiguousarray(d16, dtype=np.uint16)
    ch = None if choices is None else np.ascontiguousarray(choices, dtype=np.uint8).reshape(B, G)
    payload = np.zeros((B, info["block_bytes"]), np.uint8)
    st = np.zeros(1, np.int32)
    if details:
        table = np.empty((B, G, NC)); gbest = np.empty((B, G)); gsec = np.empty((B, G))
        vbest = np.empty((B, 32)); vsec = np.empty((B, 32)); chosen = np.empty((B, G), np.uint8)
    else:
        table = gbest = gsec = vbest = vsec = chosen = None
    rc = _L().or_encode(FMT_ID[fmt], _ptr(W), R, C, _ptr(imp), int(rows_per_expert), _ptr(grid), _ptr(d16a),
                        _ptr(ch), _ptr(payload), _ptr(table), _ptr(gbest), _ptr(gsec), _ptr(vbest),
                        _ptr(vsec), _ptr(chosen), _ptr(st), int(threads), int(entries))
    assert rc == 0, rc
    if details:
        return payload, int(st[0]), dict(table=table, gbest=gbest, gsecond=gsec, vbest=vbest,
                                         vsecond=vsec, chosen=chosen)
    return payload, int(st[0])


def decode(fmt, payload, rows, cols, grid):
    payload = np.ascontiguousarray(payload, dtype=np.uint8)
    out = np.empty((rows, cols), np.float32)
    assert _L().or_decode(FMT_ID[fmt], _ptr(payload), rows, cols, _ptr(_f32(grid)), _ptr(out)) == 0
    return out


def payload_errors(fmt, W, grid, payload, importance=None, rows_per_expert=0):
    """fp64 weighted squared error of ``payload`` per choice group [B, G] and per vector [B, 32]."""
    info = format_info(fmt)
    W = _f32(W)
    R, C = W.shape
    B = R * (C // 256)
    gerr = np.empty((B, info["groups"])); verr = np.empty((B, 32))
    payload = np.ascontiguousarray(payload, dtype=np.uint8)
    assert _L().or_payload_errors(FMT_ID[fmt], _ptr(W), R, C, _ptr(_f32(importance)), int(rows_per_expert),
                                  _ptr(_f32(grid)), _ptr(payload), _ptr(gerr), _ptr(verr)) == 0
    return gerr, verr
