"""Failure detection on the GPU without a fault: a wait that nothing will ever satisfy runs
out after its bound, the kernel records the timeout and returns, the host reads the status,
and the context stays usable for real work afterwards."""

import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_gb300 as U
import workloads
from gpu_util import MAX_ABS, REL_L2, need_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    need_gpu()
    stream = torch.cuda.current_stream().cuda_stream
    st, _ = U.ulysses_get_device_status(stream)   # start from a clear error word
    assert st == U.OK
    assert U.ulysses_selftest_timeout(stream) == U.OK
    st, word = U.ulysses_get_device_status(stream)
    assert st == U.ERR_DEVICE_TIMEOUT
    assert word >> 24 == 3 and (word >> 16) & 0xff == 6 and (word & 0xffff) in (1, 2), hex(word)
    st, word = U.ulysses_get_device_status(stream)  # reading cleared it
    assert st == U.OK and word == 0

    # the context still runs the attention block correctly
    w = workloads.WORKLOADS["tiny"]
    t = workloads.draw_workload(w)
    dev = {n: x.cuda() for n, x in t.items()}
    o, lse = U.attn_fwd(dev["q"], dev["k"], dev["v"], w.P, U.Mask.causal())
    torch.cuda.synchronize()
    assert U.device_status()[0] == U.OK
    bits = {n: workloads.to_bf16_bits(x) for n, x in t.items()}
    ref = oracle.attention_full(bits["q"], bits["k"], bits["v"], w.P, oracle.mask_for(w))
    g = o.float().cpu().double().numpy()
    assert np.abs(g - ref["o"]).max() <= MAX_ABS
    assert np.linalg.norm(g - ref["o"]) / np.linalg.norm(ref["o"]) <= REL_L2
