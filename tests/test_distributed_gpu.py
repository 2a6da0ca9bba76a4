"""GPU parity of the multi-process Ulysses path's local pieces, through the C ABI.

- ulysses_a2a_pack / ulysses_a2a_unpack (one rank's side of the all-to-alls) are checked bit
  for bit against the oracle's whole-tensor relayout: chunk g of rank r's packed shard must be
  rank r's token block of head group g in oracle.seq_to_head, and unpacking the chunks a rank
  receives (each head group's block of its tokens) must give back its token shard.
- UlyssesAttention (ulysses_sequence_gb300.distributed) over NCCL with one process: the
  collective, the packing kernels and the local attention run as in a multi-GPU job, checked
  against the oracle's whole-sequence attention. The exchange across several ranks is covered
  on CPU with gloo in test_multirank_cpu.py.
"""

import os
import socket

import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_gb300 as U
import workloads
from gpu_util import ErrStats, LSE_MAX_ABS, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("B,L,H,d,P", [(1, 256, 8, 64, 4), (2, 384, 6, 128, 3), (1, 64, 4, 8, 2), (2, 96, 4, 6, 4)])
def test_pack_unpack_match_the_oracle_relayout(B, L, H, d, P):
    """Vector path (runs of whole 16-byte units) and element path (d = 6 makes odd runs)."""
    rng = np.random.default_rng(B * 1000 + L + H + d + P)
    bits = rng.integers(0, 1 << 16, size=(P, B, L // P, H, d), dtype=np.uint16)
    heads = oracle.seq_to_head(bits, P)  # [P][B][L][Hp][d]
    Lp, Hp = L // P, H // P
    dev = torch.from_numpy(bits.view(np.int16)).cuda()
    for r in range(P):
        packed = U.a2a_pack(dev[r].view(torch.bfloat16), P)
        want = heads[:, :, r * Lp:(r + 1) * Lp]  # [P][B][Lp][Hp][d]
        assert np.array_equal(_bits(packed), want)
        back = U.a2a_unpack(torch.from_numpy(np.ascontiguousarray(want).view(np.int16)).cuda().view(torch.bfloat16), P)
        assert np.array_equal(_bits(back), bits[r])


def test_pack_rejects_bad_shapes():
    x = torch.zeros((1, 64, 6, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(U.UlyssesError):
        U.a2a_pack(x, 4)  # 6 heads over 4 ranks
    assert U.ulysses_a2a_pack(U.Shape(1, 256, 8, 64, 3), 16, 32, 0) == U.ERR_INVALID_ARG  # L % P
    assert U.ulysses_a2a_unpack(U.Shape(1, 256, 8, 64, 4), 16, 16, 0) == U.ERR_INVALID_ARG  # in == out


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("B,L,H,Hkv,d", [(2, 512, 4, 4, 128), (1, 640, 8, 2, 64)])
def test_ulysses_attention_over_nccl_one_rank(B, L, H, Hkv, d):
    import torch.distributed as dist
    from ulysses_sequence_gb300.distributed import UlyssesAttention
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        t = workloads.draw(B, L, H, d, 1, seed=41, H_kv=Hkv)
        x = {n: v[0].cuda() for n, v in t.items()}  # the one rank's token shard: every token
        ua = UlyssesAttention(mask=U.Mask.causal())
        o, ctx = ua.forward(x["q"], x["k"], x["v"])
        dq, dk, dv = ua.backward(ctx, x["do"])
        torch.cuda.synchronize()
        st, word = U.device_status()
        assert st == U.OK, hex(word)
    finally:
        dist.destroy_process_group()
    bits = {n: workloads.to_bf16_bits(v) for n, v in t.items()}
    ref = oracle.attention_full(bits["q"], bits["k"], bits["v"], 1, oracle.Mask("causal"), do_tok=bits["do"])
    G = H // Hkv
    for n, got in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        s = ErrStats(n)
        g = oracle.bf16_to_f64(_bits(got))
        s.add(g, ref[n][0])
        if G > 1 and n in ("dk", "dv"):
            # grouped dK, dV sum G query heads' gradients: one bf16 rounding of the larger sum
            s.check(max_abs=None)
            assert np.all(np.abs(g - ref[n][0]) <= 2e-2 + 2.0 ** -8 * np.abs(ref[n][0])), n
        else:
            s.check()
    lse = ctx[4][0].cpu().double().numpy()  # [B][H][L]: with one rank, every head
    fin = np.isfinite(ref["lse"][0])
    assert np.abs(lse[fin] - ref["lse"][0][fin]).max() <= LSE_MAX_ABS
