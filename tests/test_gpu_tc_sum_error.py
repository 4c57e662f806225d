"""The accumulation error of the encoder's tensor-core sums, measured against fp64.

The near-tie margin of the encoder, kMargin = 128 u (2 Cs + E1 + E2), was derived for fp32 FMA
chains of 8 terms, which err by about 8 u * sum |terms| (u = 2^-24), with a factor of two to spare:
it holds while every per-entry sum errs by at most 16 u * sum |terms|.  The tensor cores' internal
accumulation order and rounding are not documented, so this part of the exactness argument rests
on measurement.  tests/tc_sum_error.cu forms the sums as the encoder does (tf32 hi/lo split of the
fp32 per-vector operand, the parts' MMAs accumulated into one tensor-memory column) for the plain
sums (a . b with the four codebook operand kinds), the deferred-shift sums (w . h +- (w/4) . g,
four MMAs into one column) and the split sums of IQ2 grids whose squares need more bits than tf32
(a . (h hi + h lo), four MMAs), and the plain sums again with the encoder's own per-vector
operands (w and -2 w t for blocks drawn like the bench weight and its imatrix importance), and
prints the worst error over 160 random trials each.
"""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu
ALLOWANCE_U = 16.0


def test_tensor_core_sums_stay_within_the_margins_allowance(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tc_sum_error.cu")
    exe = str(tmp_path / "tc_sum_error")
    subprocess.run([nvcc, "-O2", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-o", exe, src],
                   check=True, capture_output=True, timeout=900)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    worst = {}
    for line in r.stdout.splitlines():
        *name, value = line.split()
        worst[" ".join(name)] = float(value)
    assert set(worst) == {"plain g2", "plain g", "plain ternary", "plain absternary", "deferred plus",
                          "deferred minus", "split g2wide", "plain encoder-operands"}, r.stdout
    for name, u in worst.items():
        assert u <= ALLOWANCE_U, f"{name}: {u:.2f} u above the margin's {ALLOWANCE_U} u"
