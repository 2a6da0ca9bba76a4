"""GPU parity of the projections on either side of the attention block (QKV projection into
the token-sharded layout, output projection of the token-sharded O) through the C ABI
against the fp64 oracle: every element at small sizes (ragged row, column and K tails,
grouped key/value heads, B > 1), sampled token rows at the GPT-7B-like layer's size, and
the whole block X -> QKV -> attention -> output projection against the oracle's chain."""

import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_gb300 as U
import workloads
from gpu_util import ErrStats, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _f64(t):
    return t.float().cpu().double().numpy()


def _bits(t):
    return workloads.to_bf16_bits(t.cpu())


# P, B, L, H, H_kv, d, hidden: whole tiles; ragged rows (M = 400), ragged K (hidden 96) and
# columns (N = 6 heads of 64 = 384 = 1.5 tiles); grouped heads with d = 128
# hidden sizes: whole 128-wide K slices (256, 1024), an odd number of 64-wide chunks (320: the last
# slice's second chunk reads zeros) and a ragged K (96: 2-D boxes with zero fill past column 96)
CASES = [(2, 1, 256, 4, 4, 64, 256), (4, 2, 200, 4, 1, 64, 96), (4, 1, 512, 8, 2, 128, 1024),
         (2, 1, 256, 4, 2, 64, 320)]


@pytest.mark.parametrize("P,B,L,H,Hkv,d,hidden", CASES)
def test_qkv_and_out_projection_every_element(P, B, L, H, Hkv, d, hidden):
    x = workloads.draw_hidden(B, L, hidden, P, seed=P + H)
    w = workloads.draw_weight((H + 2 * Hkv) * d, hidden, seed=1 + H)
    wo = workloads.draw_weight(hidden, H * d, seed=2 + H)
    q, k, v = U.qkv_proj(x.cuda(), w.cuda(), P, H, Hkv, d)
    y = U.out_proj(q, wo.cuda(), P)
    torch.cuda.synchronize()
    st, word = U.device_status()
    assert st == U.OK, hex(word)
    ref = oracle.qkv_projection(_bits(x), _bits(w), H, Hkv, d)
    for name, got in (("q", q), ("k", k), ("v", v)):
        s = ErrStats(name)
        s.add(_f64(got), ref[name])
        s.check()
    # the output projection is checked on the GPU's own bf16 Q (its input here)
    s = ErrStats("y")
    s.add(_f64(y), oracle.out_projection(_bits(q), _bits(wo)))
    s.check()


def test_projection_at_the_gpt7b_layer_sampled_rows():
    """X [32768 tokens][4096] -> Q, K, V with 32 heads of 128: 512 seeded token rows checked."""
    w_ = workloads.WORKLOADS["gpt7b"]
    P, B, L, H, d = w_.P, w_.B, w_.L, w_.H, w_.d
    hidden = H * d
    x = workloads.draw_hidden(B, L, hidden, P, seed=11)
    w = workloads.draw_weight(3 * H * d, hidden, seed=12)
    q, k, v = U.qkv_proj(x.cuda(), w.cuda(), P, H, H, d)
    torch.cuda.synchronize()
    assert U.device_status()[0] == U.OK
    rows = np.sort(np.random.default_rng(13).choice(P * B * (L // P), size=512, replace=False))
    x_rows = _bits(x).reshape(-1, hidden)[rows][:, None, None, :]  # each sampled row as its own shard
    ref = oracle.qkv_projection(x_rows, _bits(w), H, H, d)
    for name, got in (("q", q), ("k", k), ("v", v)):
        s = ErrStats(name)
        s.add(_f64(got).reshape(P * B * (L // P), -1)[rows], ref[name].reshape(len(rows), -1))
        s.check()


def test_whole_block_matches_the_oracle_chain():
    """X -> QKV projection -> Ulysses attention (relayouts fused) -> output projection, against
    the oracle's chain on the GPU's bf16 intermediates (each stage checked on its own inputs)."""
    P, B, L, H, Hkv, d, hidden = 4, 1, 256, 8, 4, 64, 512
    x = workloads.draw_hidden(B, L, hidden, P, seed=21)
    w = workloads.draw_weight((H + 2 * Hkv) * d, hidden, seed=22)
    wo = workloads.draw_weight(hidden, H * d, seed=23)
    q, k, v = U.qkv_proj(x.cuda(), w.cuda(), P, H, Hkv, d)
    o, lse = U.attn_fwd(q, k, v, P, U.Mask.causal())
    y = U.out_proj(o, wo.cuda(), P)
    torch.cuda.synchronize()
    assert U.device_status()[0] == U.OK
    ref_o = oracle.attention_full(_bits(q), _bits(k), _bits(v), P, oracle.Mask("causal"))["o"]
    s = ErrStats("o")
    s.add(_f64(o), ref_o)
    s.check()
    s = ErrStats("y")
    s.add(_f64(y), oracle.out_projection(_bits(o), _bits(wo)))
    s.check()
