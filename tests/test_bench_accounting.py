"""The benchmark's accounting on CPU: the algorithmic flops (over permitted pairs only: 4 d_h
per pair forward, 8 d_h backward) and the accounted all-to-all bytes of each workload, against
the figures the workload table states (three or four significant digits)."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402

# workload: (forward flops, backward flops, accounted all-to-all bytes per rank, forward)
TABLE = {
    "tiny": (67.4e6, 134.7e6, 0.262e6),
    "gpt1.2b": (0.275e12, 0.0, 16.8e6),
    "gpt7b": (8.80e12, 17.59e12, 134e6),
    "long": (140.7e12, 281.5e12, 134e6),
    "block_sparse": (10.85e12, 21.70e12, 537e6),
}


@pytest.mark.parametrize("name", sorted(TABLE))
def test_flops_and_accounted_bytes(name):
    w = workloads.WORKLOADS[name]
    f_fwd, f_bwd = bench.flops(w)
    e_fwd, e_bwd, e_comm = TABLE[name]
    assert f_fwd == pytest.approx(e_fwd, rel=5e-3)
    assert f_bwd == pytest.approx(e_bwd, rel=5e-3)
    assert bench.accounted_alltoall_bytes(w) == pytest.approx(e_comm, rel=5e-3)


def test_permitted_pairs_closed_forms():
    w = workloads.WORKLOADS["gpt7b"]
    assert bench.permitted_pairs(w) == w.L * (w.L + 1) // 2
    # the block-sparse pattern: 20,211 active 128 x 128 tiles at L = 65536
    bs = workloads.WORKLOADS["block_sparse"]
    assert bench.permitted_pairs(bs) == 20211 * 128 * 128


def test_grouped_heads_exchange_fewer_bytes():
    """H = 32 query heads, H_kv = 8 key/value heads, P = 8 groups: each group receives one
    key/value head, so Q and O move 32 heads' worth and K and V only 8."""
    w = workloads.WORKLOADS["gpt7b_gqa"]
    assert bench.accounted_alltoall_bytes(w) == (2 * 32 + 2 * 8) * w.B * w.L * w.d * 2 // w.P
    assert bench.accounted_alltoall_bytes(w) < bench.accounted_alltoall_bytes(workloads.WORKLOADS["gpt7b"])
