"""The backward entry point that allocates nothing, checked against the regular one.

ulysses_attn_bwd_noalloc serves callers that cannot allocate device memory (their device
memory is owned by a host framework's pool, or their run-time memory plan forbids
cudaMalloc); it keeps the backward workspace in a fixed device array inside the library.
These tests call it through the C ABI, twice in a row, and compare every output with what
ulysses_attn_bwd produces from a caller-allocated workspace, and on the tiny workload with
the fp64 oracle. The file is named so that pytest collects it last; it also passes on its
own in a fresh process.
"""

import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_gb300 as U
import workloads
from gpu_util import MAX_ABS, REL_L2, need_gpu

pytestmark = pytest.mark.gpu


def _close(got: torch.Tensor, ref: torch.Tensor, name: str):
    g = got.float().cpu().double().numpy()
    r = ref.float().cpu().double().numpy()
    assert np.all(np.isfinite(g)), name
    max_abs = float(np.abs(g - r).max())
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    assert max_abs <= MAX_ABS and rel <= REL_L2, (name, max_abs, rel)


@pytest.mark.parametrize("B,L,H,d,P", [(1, 1024, 8, 128, 4), (2, 640, 4, 64, 2)])
def test_noalloc_backward_matches_workspace_backward(B, L, H, d, P):
    need_gpu()
    shape = U.Shape(B, L, H, d, P)
    assert U.ulysses_attn_bwd_workspace_size(shape) <= U.BWD_NOALLOC_SCRATCH_BYTES
    t = {n: x.cuda() for n, x in workloads.draw(B, L, H, d, P, seed=21).items()}
    mask = U.Mask.causal()
    o, lse = U.attn_fwd(t["q"], t["k"], t["v"], P, mask)
    ref = U.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], P, mask)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = (torch.full_like(t["q"], float("nan")) for _ in range(3))
        rc = U.ulysses_attn_bwd_noalloc(shape, mask.struct, 0.0, U.LAYOUT_TOKEN_SHARDED, t["q"].data_ptr(),
                                        t["k"].data_ptr(), t["v"].data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        t["do"].data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), stream)
        assert rc == U.OK, U.ulysses_status_string(rc)
        torch.cuda.synchronize()
        st, word = U.device_status()
        assert st == U.OK, hex(word)
        for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            _close(got, want, f"{name} (call {call + 1})")
        # dK and dV do not depend on the order of additions: they must match bit for bit
        assert torch.equal(dk.view(torch.int16), ref[1].view(torch.int16))
        assert torch.equal(dv.view(torch.int16), ref[2].view(torch.int16))


def test_noalloc_backward_refuses_shapes_beyond_its_array():
    need_gpu()
    big = U.Shape(1, 32768, 32, 128, 8)
    assert U.ulysses_attn_bwd_workspace_size(big) > U.BWD_NOALLOC_SCRATCH_BYTES
    m = U.MaskStruct(U.MASK_CAUSAL, 128, None, None, None, None, 0)
    p = [256 * (i + 1) for i in range(9)]  # never dereferenced: the size check comes first
    assert U.ulysses_attn_bwd_noalloc(big, m, 0.0, U.LAYOUT_TOKEN_SHARDED, *p, 0) == U.ERR_UNSUPPORTED


def test_noalloc_backward_matches_oracle():
    """The tiny workload (B=1, L=256, H=8, d_h=64, P=4, causal): dQ, dK, dV of two calls in a
    row against the oracle's analytic gradient, within the acceptance bound."""
    need_gpu()
    w = workloads.WORKLOADS["tiny"]
    t = workloads.draw_workload(w)
    bits = {n: workloads.to_bf16_bits(x) for n, x in t.items()}
    ref = oracle.attention_full(bits["q"], bits["k"], bits["v"], w.P, oracle.mask_for(w), do_tok=bits["do"])
    dev = {n: x.cuda() for n, x in t.items()}
    shape = U.Shape(w.B, w.L, w.H, w.d, w.P)
    mask = U.Mask.causal()
    o, lse = U.attn_fwd(dev["q"], dev["k"], dev["v"], w.P, mask)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = (torch.full_like(dev["q"], float("nan")) for _ in range(3))
        rc = U.ulysses_attn_bwd_noalloc(shape, mask.struct, 0.0, U.LAYOUT_TOKEN_SHARDED, dev["q"].data_ptr(),
                                        dev["k"].data_ptr(), dev["v"].data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        dev["do"].data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), stream)
        assert rc == U.OK, U.ulysses_status_string(rc)
        torch.cuda.synchronize()
        assert U.device_status()[0] == U.OK
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            g = got.float().cpu().double().numpy()
            r = ref[name]
            max_abs = float(np.abs(g - r).max())
            rel = float(np.linalg.norm(g - r) / np.linalg.norm(r))
            assert max_abs <= MAX_ABS and rel <= REL_L2, (name, call + 1, max_abs, rel)
