"""Oracle of merging imatrix statistics, neutral entries and the coverage figures (numpy).

TEST INFRASTRUCTURE ONLY: the tests may call it; the library never does.

Source: "MoE expert coverage in imatrix calibration", Facts: the GGUF imatrix format stores
in_sum2 and counts per tensor so that files can be merged; the legacy writer stores a zero-count
expert with value 1 and count 1 (a neutral entry, matching the weight 1 the reader gives it);
saving logs the share of experts with data ("partial data") and "no data" when no expert has any.

Readings: a merge adds the two statistics channel by channel in fp32 (one rounding per value)
and adds the counts; the coverage figures are the number of experts with at least one token, the
tokens over all experts, and the least and largest count.

Parity status: pinned by tests/test_oracle_imatrix_tools.py (merging statistics of disjoint
experts reproduces one call of the C oracle over all the tokens; zero statistics and argument
order leave a merge unchanged; neutral entries get weight 1 from the C oracle; the token total is
tokens x top_k).
"""
from __future__ import annotations

import numpy as np


def merge(in_sum2, counts, src_in_sum2, src_counts):
    """(in_sum2 + src_in_sum2 in fp32, counts + src_counts)."""
    a = np.asarray(in_sum2, np.float32)
    b = np.asarray(src_in_sum2, np.float32)
    return (a + b).astype(np.float32), np.asarray(counts, np.int64) + np.asarray(src_counts, np.int64)


def neutral_entries(in_sum2, counts):
    """Zero-count experts: in_sum2 = 1 on every channel and count 1."""
    s = np.array(in_sum2, np.float32, copy=True)
    c = np.array(counts, np.int64, copy=True)
    z = c == 0
    s[z] = 1.0
    c[z] = 1
    return s, c


def coverage(counts):
    """(experts with at least one token, tokens over all experts, least count, largest count)."""
    c = np.asarray(counts, np.int64)
    return int(np.count_nonzero(c)), int(c.sum()), int(c.min()), int(c.max())
