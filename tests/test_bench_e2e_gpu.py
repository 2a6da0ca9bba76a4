"""The benchmark's end-to-end loop: copies in, kernels and copies out on three streams over two
device buffer sets. Every step must deliver the results of its own inputs. Five steps read
three different input sets in turn, and each step's host outputs must equal those of the same
calls run one at a time, so that a copy ordered wrongly against a kernel (an input overwritten
before it was read, an output read before it was written or after the next step overwrote it)
shows up as another input's results."""

import dataclasses

import pytest
import torch

import bench
import workloads

pytestmark = pytest.mark.gpu

STEPS = 5
N_INPUTS = 3


def _case(backward):
    import ulysses_sequence_gb300 as U
    w = dataclasses.replace(workloads.WORKLOADS["tiny"], name="e2e-check", L=1024, H=4, P=2, backward=backward)
    mask = U.Mask.causal()
    ins = []
    for seed in range(N_INPUTS):
        t = workloads.draw(w.B, w.L, w.H, w.d, w.P, 100 + seed)
        ins.append({n: x.pin_memory() for n, x in t.items()})
    # each input set run alone, synchronously
    refs = []
    for h in ins:
        x = {n: v.cuda() for n, v in h.items()}
        o, lse = U.attn_fwd(x["q"], x["k"], x["v"], w.P, mask)
        r = {"o": o, "lse": lse}
        if backward:
            r["dq"], r["dk"], r["dv"] = U.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], w.P, mask)
        torch.cuda.synchronize()
        refs.append({n: v.cpu() for n, v in r.items()})
    x0 = {n: v.cuda() for n, v in ins[0].items()}
    sets = []
    for _ in range(2):
        sets.append({"x": {n: torch.empty_like(v) for n, v in x0.items()}, "o": torch.empty_like(x0["q"]),
                     "lse": torch.empty(refs[0]["lse"].shape, dtype=torch.float32, device="cuda"),
                     "dq": torch.empty_like(x0["q"]), "dk": torch.empty_like(x0["k"]),
                     "dv": torch.empty_like(x0["v"]), "ws": U.bwd_workspace(x0["q"], w.P)})
    host_out = [{n: torch.full(v.shape, float("nan"), dtype=v.dtype).pin_memory() for n, v in refs[0].items()}
                for _ in range(STEPS)]
    elapsed, kernel_ms = bench.e2e_pipeline(U, w, mask, ins, sets, host_out, STEPS, torch.cuda.current_stream())
    st, word = U.device_status()
    assert st == U.OK, hex(word)
    assert elapsed > 0 and kernel_ms > 0
    return refs, host_out


@pytest.mark.parametrize("backward", [True, False], ids=["fwd+bwd", "fwd"])
def test_every_pipelined_step_gets_its_own_results(backward):
    refs, host_out = _case(backward)
    for i in range(STEPS):
        ref, got = refs[i % N_INPUTS], host_out[i]
        assert set(got) == set(ref)
        for n in ("o", "lse", "dk", "dv"):
            if n in ref:
                # deterministic kernels: the same bits as the lone call
                assert torch.equal(got[n], ref[n]), (i, n)
        if "dq" in ref:
            # dQ is summed by fp32 reductions whose order varies from run to run
            err = (got["dq"].float() - ref["dq"].float()).abs().max().item()
            assert err <= 1e-2 * ref["dq"].float().abs().max().item() + 1e-6, (i, err)
