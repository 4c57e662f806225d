"""Thin Python binding of ``libiq_b300.so`` (the C ABI in include/iq.h).

Argument marshalling only: every step runs in the library's CUDA kernels.  PyTorch provides device
memory (outputs and workspace are allocated here with torch) and the current CUDA stream.  There is
no CPU fallback: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libiq_b300.so")

FORMATS = ("IQ2_XXS", "IQ2_XS", "IQ2_S", "IQ1_S", "IQ1_M")
FMT_ID = {n: i for i, n in enumerate(FORMATS)}
IQ_F32, IQ_BF16 = 0, 1
EXPORTS = ("iq_format_info", "iq_imatrix_workspace_size", "iq_imatrix_accumulate", "iq_imatrix_weights",
           "iq_anchor_scales", "iq_encode_workspace_size", "iq_encode", "iq_group_errors", "iq_decode",
           "iq_encode_static_scratch_capacity", "iq_encode_static_scratch",
           "iq_encode_every_choice", "iq_local_hessian_workspace_size", "iq_local_hessian_choices",
           "iq_imatrix_merge", "iq_imatrix_neutral_entries", "iq_imatrix_coverage", "iq_encode_write_back")

STATUS_BITS = {
    "BAD_CHOICE": 1, "BAD_EXPERT_ID": 2, "NONFINITE_SUM2": 4, "DUP_EXPERT_ID": 8, "BAD_INPUT": 16,
    "BAD_IMPORTANCE": 32, "BAD_SCALE": 64, "BAD_GRID": 128, "TIMEOUT": 256,
}


class IQError(RuntimeError):
    pass


class _Info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("block_bytes", "choice_groups", "num_choices", "grid_entries",
                                            "vectors_per_group", "index_bits")]


_lib = None


def lib():
    """Loads the library (raises IQError if it is missing or incomplete)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise IQError(f"{LIB_PATH} is missing: build it with python -m ggml_iq_codebook_accumulate_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, p, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        L.iq_format_info.argtypes = [i32, ctypes.POINTER(_Info)]
        L.iq_imatrix_workspace_size.argtypes = [i64, i64, i32, i32, i32, i64, ctypes.POINTER(sz)]
        L.iq_imatrix_accumulate.argtypes = [p, i32, i64, i64, p, i32, i32, i64, p, p, p, p, sz, p]
        L.iq_imatrix_weights.argtypes = [p, p, i32, i64, ctypes.c_float, p, p]
        L.iq_anchor_scales.argtypes = [i32, p, i32, i64, i64, p, p, p]
        L.iq_encode_workspace_size.argtypes = [i32, i64, i64, ctypes.POINTER(sz)]
        L.iq_encode.argtypes = [i32, p, i32, i64, i64, p, i64, p, p, p, p, p, p, p, sz, p]
        L.iq_group_errors.argtypes = [i32, p, i32, i64, i64, p, i64, p, p, p, p, p, sz, p]
        L.iq_decode.argtypes = [i32, p, i64, i64, p, p, i32, p]
        L.iq_encode_static_scratch_capacity.argtypes = [i32, ctypes.POINTER(i64)]
        L.iq_encode_static_scratch.argtypes = [i32, p, i32, i64, i64, p, i64, p, p, p, p, p, p, p]
        L.iq_encode_every_choice.argtypes = [i32, p, i32, i64, i64, p, i64, p, p, p, p, p, sz, p]
        L.iq_local_hessian_workspace_size.argtypes = [i32, i64, i64, ctypes.POINTER(sz)]
        L.iq_local_hessian_choices.argtypes = [i32, p, i32, i64, i64, p, p, p, ctypes.c_float, p, p, p, sz, p]
        L.iq_imatrix_merge.argtypes = [p, p, p, p, i32, i64, p, p]
        L.iq_imatrix_neutral_entries.argtypes = [p, p, i32, i64, p]
        L.iq_imatrix_coverage.argtypes = [p, i32, p, p]
        L.iq_encode_write_back.argtypes = [i32, p, i32, i64, i64, p, i64, p, p, p, p, p, p, sz, p]
        for n in EXPORTS:
            getattr(L, n).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(rc, what):
    if rc != 0:
        raise IQError(f"{what} failed with code {rc}")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dt(t):
    if t.dtype == torch.float32:
        return IQ_F32
    if t.dtype == torch.bfloat16:
        return IQ_BF16
    raise IQError(f"unsupported dtype {t.dtype}")


def _cuda(t, name):
    if t is not None and (not t.is_cuda or not t.is_contiguous()):
        raise IQError(f"{name} must be a contiguous CUDA tensor")
    return t


def format_info(fmt: str) -> dict:
    info = _Info()
    _check(lib().iq_format_info(FMT_ID[fmt], ctypes.byref(info)), "iq_format_info")
    return {n: getattr(info, n) for n, _ in _Info._fields_}


def _workspace(nbytes, device):
    # 256-byte alignment: torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def imatrix_workspace(tokens, cols, dtype, num_experts, top_k, rows_per_chunk, device):
    nb = ctypes.c_size_t()
    dt = IQ_BF16 if dtype == torch.bfloat16 else IQ_F32
    _check(lib().iq_imatrix_workspace_size(tokens, cols, dt, num_experts, top_k, rows_per_chunk, ctypes.byref(nb)),
           "workspace size")
    return _workspace(nb.value, device)


def imatrix_accumulate(x, expert_ids, num_experts, rows_per_chunk=1024, in_sum2=None, counts=None, status=None,
                       workspace=None):
    """Accumulates the routed sum of squares into ``in_sum2`` [E, cols] fp32 and token counts into
    ``counts`` [E] int64 (both created as zeros when None).  Returns (in_sum2, counts)."""
    _cuda(x, "x"); _cuda(expert_ids, "expert_ids")
    T, C = x.shape
    dev = x.device
    if in_sum2 is None:
        in_sum2 = torch.zeros(num_experts, C, dtype=torch.float32, device=dev)
    if counts is None:
        counts = torch.zeros(num_experts, dtype=torch.int64, device=dev)
    ws = workspace if workspace is not None else imatrix_workspace(T, C, x.dtype, num_experts, expert_ids.shape[1],
                                                                    rows_per_chunk, dev)
    _check(lib().iq_imatrix_accumulate(_p(x), _dt(x), T, C, _p(expert_ids.to(torch.int32)), expert_ids.shape[1],
                                       num_experts, rows_per_chunk, _p(in_sum2), _p(counts), _p(status), _p(ws),
                                       ws.numel(), _stream(dev)), "iq_imatrix_accumulate")
    return in_sum2, counts


def imatrix_weights(in_sum2, counts, floor=0.0):
    _cuda(in_sum2, "in_sum2"); _cuda(counts, "counts")
    E, C = in_sum2.shape
    w = torch.empty_like(in_sum2)
    _check(lib().iq_imatrix_weights(_p(in_sum2), _p(counts), E, C, float(floor), _p(w), _stream(w.device)),
           "iq_imatrix_weights")
    return w


def anchor_scales(fmt, W, status=None):
    _cuda(W, "W")
    R, C = W.shape
    d16 = torch.empty(R * (C // 256), dtype=torch.int16, device=W.device)
    _check(lib().iq_anchor_scales(FMT_ID[fmt], _p(W), _dt(W), R, C, _p(d16), _p(status), _stream(W.device)),
           "iq_anchor_scales")
    return d16


def encode_workspace(fmt, rows, cols, device):
    nb = ctypes.c_size_t()
    _check(lib().iq_encode_workspace_size(FMT_ID[fmt], rows, cols, ctypes.byref(nb)), "workspace size")
    return _workspace(nb.value, device)


def encode(fmt, W, grid, importance=None, rows_per_expert=0, d16=None, choices=None, every_choice=False,
           status=None, payload=None, table=None, workspace=None):
    """Encodes W [rows, cols] (fp32 or bf16).  Returns the payload [B, block_bytes] uint8, or
    (payload, group_errors [B, groups, choices] fp32) with ``every_choice``."""
    for t, n in ((W, "W"), (grid, "grid"), (importance, "importance"), (d16, "d16"), (choices, "choices")):
        _cuda(t, n)
    info = format_info(fmt)
    R, C = W.shape
    B = R * (C // 256)
    dev = W.device
    if payload is None:
        payload = torch.empty(B, info["block_bytes"], dtype=torch.uint8, device=dev)
    if every_choice and table is None:
        table = torch.empty(B, info["choice_groups"], info["num_choices"], dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = encode_workspace(fmt, R, C, dev)
    _check(lib().iq_encode(FMT_ID[fmt], _p(W), _dt(W), R, C, _p(importance), int(rows_per_expert), _p(grid),
                           _p(d16), _p(choices), _p(payload), _p(table if every_choice else None), _p(status),
                           _p(workspace), workspace.numel(), _stream(dev)), "iq_encode")
    return (payload, table) if every_choice else payload


def group_errors(fmt, W, grid, importance=None, rows_per_expert=0, d16=None, status=None, table=None,
                 workspace=None):
    info = format_info(fmt)
    R, C = W.shape
    B = R * (C // 256)
    dev = W.device
    if table is None:
        table = torch.empty(B, info["choice_groups"], info["num_choices"], dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = encode_workspace(fmt, R, C, dev)
    _check(lib().iq_group_errors(FMT_ID[fmt], _p(W), _dt(W), R, C, _p(importance), int(rows_per_expert), _p(grid),
                                 _p(d16), _p(table), _p(status), _p(workspace), workspace.numel(), _stream(dev)),
           "iq_group_errors")
    return table


def encode_every_choice(fmt, W, grid, importance=None, rows_per_expert=0, d16=None, status=None, payloads=None,
                        workspace=None):
    """Payloads [num_choices, B, block_bytes] uint8: payloads[c] is the forced encode with every
    group at choice c."""
    for t, n in ((W, "W"), (grid, "grid"), (importance, "importance"), (d16, "d16")):
        _cuda(t, n)
    info = format_info(fmt)
    R, C = W.shape
    B = R * (C // 256)
    dev = W.device
    if payloads is None:
        payloads = torch.empty(info["num_choices"], B, info["block_bytes"], dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = encode_workspace(fmt, R * info["num_choices"], C, dev)
    _check(lib().iq_encode_every_choice(FMT_ID[fmt], _p(W), _dt(W), R, C, _p(importance), int(rows_per_expert),
                                        _p(grid), _p(d16), _p(payloads), _p(status), _p(workspace),
                                        workspace.numel(), _stream(dev)), "iq_encode_every_choice")
    return payloads


def local_hessian_workspace(fmt, rows, cols, device):
    n = ctypes.c_size_t()
    _check(lib().iq_local_hessian_workspace_size(FMT_ID[fmt], rows, cols, ctypes.byref(n)),
           "iq_local_hessian_workspace_size")
    return _workspace(n.value, device)


def local_hessian_choices(fmt, W, grid, payloads, hessian_blocks, perc_damp=0.3, status=None, choices=None,
                          workspace=None):
    """Searched choices [B, groups] uint8 from the every-choice payloads and the [cols / 256, 256,
    256] fp32 diagonal blocks of the input Hessian."""
    for t, n in ((W, "W"), (grid, "grid"), (payloads, "payloads"), (hessian_blocks, "hessian_blocks")):
        _cuda(t, n)
    info = format_info(fmt)
    R, C = W.shape
    B = R * (C // 256)
    dev = W.device
    if choices is None:
        choices = torch.empty(B, info["choice_groups"], dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = local_hessian_workspace(fmt, R, C, dev)
    _check(lib().iq_local_hessian_choices(FMT_ID[fmt], _p(W), _dt(W), R, C, _p(grid), _p(payloads),
                                          _p(hessian_blocks), float(perc_damp), _p(choices), _p(status),
                                          _p(workspace), workspace.numel(), _stream(dev)), "iq_local_hessian_choices")
    return choices


def imatrix_merge(in_sum2, counts, src_in_sum2, src_counts, status=None):
    """in_sum2 += src_in_sum2 and counts += src_counts, in place."""
    for t, n in ((in_sum2, "in_sum2"), (counts, "counts"), (src_in_sum2, "src_in_sum2"), (src_counts, "src_counts")):
        _cuda(t, n)
    E, C = in_sum2.shape
    _check(lib().iq_imatrix_merge(_p(in_sum2), _p(counts), _p(src_in_sum2), _p(src_counts), E, C, _p(status),
                                  _stream(in_sum2.device)), "iq_imatrix_merge")
    return in_sum2, counts


def imatrix_neutral_entries(in_sum2, counts):
    """Zero-count experts get in_sum2 = 1 and count 1, in place."""
    E, C = in_sum2.shape
    _check(lib().iq_imatrix_neutral_entries(_p(in_sum2), _p(counts), E, C, _stream(in_sum2.device)),
           "iq_imatrix_neutral_entries")
    return in_sum2, counts


def imatrix_coverage(counts):
    """Device int64 [4]: experts with tokens, total tokens, least and largest count."""
    out = torch.empty(4, dtype=torch.int64, device=counts.device)
    _check(lib().iq_imatrix_coverage(_p(counts), counts.numel(), _p(out), _stream(counts.device)), "iq_imatrix_coverage")
    return out


def encode_write_back(fmt, W, grid, importance=None, rows_per_expert=0, d16=None, choices=None, status=None,
                      payload=None, workspace=None):
    """Encodes W and overwrites it with the decoded payload (its own dtype).  Returns the payload."""
    for t, n in ((W, "W"), (grid, "grid"), (importance, "importance"), (d16, "d16"), (choices, "choices")):
        _cuda(t, n)
    info = format_info(fmt)
    R, C = W.shape
    B = R * (C // 256)
    dev = W.device
    if payload is None:
        payload = torch.empty(B, info["block_bytes"], dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = encode_workspace(fmt, R, C, dev)
    _check(lib().iq_encode_write_back(FMT_ID[fmt], _p(W), _dt(W), R, C, _p(importance), int(rows_per_expert),
                                      _p(grid), _p(d16), _p(choices), _p(payload), _p(status), _p(workspace),
                                      workspace.numel(), _stream(dev)), "iq_encode_write_back")
    return payload


def decode(fmt, payload, rows, cols, grid, dtype=torch.float32, out=None):
    _cuda(payload, "payload"); _cuda(grid, "grid")
    if out is None:
        out = torch.empty(rows, cols, dtype=dtype, device=payload.device)
    _check(lib().iq_decode(FMT_ID[fmt], _p(payload), rows, cols, _p(grid), _p(out), _dt(out),
                           _stream(payload.device)), "iq_decode")
    return out


def encode_static_scratch_capacity(fmt: str) -> int:
    """Largest number of 256-value blocks iq_encode_static_scratch accepts for ``fmt``."""
    n = ctypes.c_int64()
    _check(lib().iq_encode_static_scratch_capacity(FMT_ID[fmt], ctypes.byref(n)), "iq_encode_static_scratch_capacity")
    return n.value


def encode_static_scratch(fmt, W, grid, importance=None, rows_per_expert=0, d16=None, choices=None,
                          every_choice=False, status=None, payload=None, table=None):
    """iq_encode for callers that cannot allocate device scratch: the library's own fixed 1 MiB
    device array replaces the workspace (outputs are still the caller's).  Raises IQError with code
    -4 when the weight needs more scratch than that array holds."""
    for t, n in ((W, "W"), (grid, "grid"), (importance, "importance"), (d16, "d16"), (choices, "choices")):
        _cuda(t, n)
    info = format_info(fmt)
    R, C = W.shape
    B = R * (C // 256)
    dev = W.device
    if payload is None:
        payload = torch.empty(B, info["block_bytes"], dtype=torch.uint8, device=dev)
    if every_choice and table is None:
        table = torch.empty(B, info["choice_groups"], info["num_choices"], dtype=torch.float32, device=dev)
    _check(lib().iq_encode_static_scratch(FMT_ID[fmt], _p(W), _dt(W), R, C, _p(importance), int(rows_per_expert),
                                          _p(grid), _p(d16), _p(choices), _p(payload),
                                          _p(table if every_choice else None), _p(status), _stream(dev)),
           "iq_encode_static_scratch")
    return (payload, table) if every_choice else payload
