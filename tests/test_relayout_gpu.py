"""GPU parity of the standalone relayouts against the oracle's index loops: bit-exact,
including NaN and denormal bf16 patterns, at small shapes (vector and fallback paths) and
at every workload's full size. Guard bytes around the output must stay untouched."""

import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_gb300 as U
import workloads
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements of canary before and after each output


def run_relayout(x_bits: np.ndarray, P: int, to_head: bool):
    """x_bits: uint16 source in its layout. Returns (output bits, guards intact)."""
    src = torch.from_numpy(x_bits.view(np.int16).copy()).cuda()
    if to_head:
        P_, B, Lp, H, d = x_bits.shape
        out_shape = (P, B, Lp * P, H // P, d)
        shape = U.Shape(B, Lp * P, H, d, P)
    else:
        P_, B, L, Hp, d = x_bits.shape
        out_shape = (P, B, L // P, Hp * P, d)
        shape = U.Shape(B, L, Hp * P, d, P)
    n = int(np.prod(out_shape))
    buf = torch.full((n + 2 * GUARD,), 0x5A5A, dtype=torch.int16, device="cuda")
    out = buf[GUARD:GUARD + n]
    fn = U.ulysses_seq_to_head if to_head else U.ulysses_head_to_seq
    U.check(fn(shape, src.data_ptr(), out.data_ptr(), torch.cuda.current_stream().cuda_stream), "relayout")
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    guards_ok = bool(np.all(host[:GUARD] == 0x5A5A) and np.all(host[GUARD + n:] == 0x5A5A))
    return host[GUARD:GUARD + n].view(np.uint16).reshape(out_shape), guards_ok


SMALL = [
    (4, 2, 16, 8, 64),    # 16-byte vector path
    (3, 1, 9, 6, 8),      # odd P
    (8, 1, 64, 8, 128),   # Hp = 1
    (2, 3, 6, 4, 3),      # runs not a whole vector: element path
    (1, 2, 8, 4, 16),     # P = 1: identity
    (4, 1, 4096, 32, 128),  # long rows (one warp per 8 KB row)
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("P,B,L,H,d", SMALL)
def test_relayout_small_bit_exact(P, B, L, H, d):
    rng = np.random.default_rng(P * 1000 + L)
    x = rng.integers(0, 1 << 16, size=(P, B, L // P, H, d), dtype=np.uint16)
    x.flat[: 8] = [0x7FC1, 0xFFFF, 0x7F81, 0x0001, 0x8001, 0x8000, 0x7F80, 0xFF80][: min(8, x.size)]
    y, ok = run_relayout(x, P, True)
    assert ok, "seq_to_head wrote outside its output"
    assert np.array_equal(y, oracle.seq_to_head(x, P))
    z, ok = run_relayout(y, P, False)
    assert ok, "head_to_seq wrote outside its output"
    assert np.array_equal(z, x)


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_relayout_workload_sizes_bit_exact(name):
    w = workloads.WORKLOADS[name]
    rng = np.random.default_rng(w.seed)
    x = rng.integers(0, 1 << 16, size=(w.P, w.B, w.Lp, w.H, w.d), dtype=np.uint16)
    y, ok = run_relayout(x, w.P, True)
    assert ok
    assert np.array_equal(y, oracle.seq_to_head(x, w.P))
    z, ok = run_relayout(y, w.P, False)
    assert ok
    assert np.array_equal(z, x)


def test_relayout_empty_is_a_no_op():
    s = U.Shape(0, 128, 8, 64, 4)
    assert U.ulysses_seq_to_head(s, 0, 0, 0) == U.OK
    torch.cuda.synchronize()
