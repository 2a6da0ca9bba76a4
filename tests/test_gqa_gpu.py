"""GPU parity of grouped key/value heads (GQA/MQA) through the C ABI against the fp64 oracle.

Query head h attends with key/value head h // (H/H_kv). The key/value relayout gives head
group g its H_kv/P whole heads, or one copy of head g // (P/H_kv) when P > H_kv; its adjoint
sums the copies. Checked here: the K/V relayouts bit-exact (and the adjoint against the
oracle's fp64 sum within bf16 rounding), and forward + backward on every row at small
sizes for both layouts, all mask kinds, replicated and unreplicated heads, MQA, and a
ragged tail; plus GQA = multi-head attention on repeated key/value heads.
"""

import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_gb300 as U
import workloads
from gpu_util import ErrStats, LSE_MAX_ABS, gpu_mask, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _dev(bits: np.ndarray, dtype=torch.bfloat16) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(dtype).cuda()


# P, B, L, H_kv, d: whole heads per group (H_kv % P == 0), copies (P % H_kv == 0), MQA, a
# head width whose rows are not whole 16-byte vectors (element path)
KV_SHAPES = [(4, 2, 256, 8, 128), (4, 1, 128, 2, 64), (8, 1, 256, 1, 128), (4, 1, 96, 2, 20)]


@pytest.mark.parametrize("P,B,L,Hkv,d", KV_SHAPES)
def test_kv_seq_to_head_bit_exact(P, B, L, Hkv, d):
    rng = np.random.default_rng(P * 100 + Hkv)
    x = rng.integers(0, 1 << 16, size=(P, B, L // P, Hkv, d), dtype=np.uint16)
    y = U.kv_seq_to_head(_dev(x, torch.int16), P)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), oracle.kv_seq_to_head(x, P))


@pytest.mark.parametrize("P,B,L,Hkv,d", KV_SHAPES)
def test_kv_head_to_seq_sum_matches_oracle(P, B, L, Hkv, d):
    Hkvp = U.kv_heads_per_group(Hkv, P)
    g = torch.Generator().manual_seed(P + Hkv + d)
    y = torch.randn((P, B, L, Hkvp, d), generator=g).to(torch.bfloat16)
    z = U.kv_head_to_seq_sum(y.cuda(), P, Hkv)
    torch.cuda.synchronize()
    got = z.cpu().double().numpy()
    exact = oracle.kv_head_to_seq_sum(y.double().numpy(), P, Hkv)
    if Hkvp * P == Hkv:
        # one copy per head: the exact inverse permutation
        assert np.array_equal(_bits(z), oracle.head_to_seq(_bits(y), P))
    # an fp32 sum of a few bf16 values, rounded to nearest-even bf16: within half a bf16 unit
    assert np.all(np.abs(got - exact) <= np.abs(exact) * 2.0 ** -8 + 1e-30)


@pytest.mark.parametrize("P,B,L,Hkv,d", KV_SHAPES[:3])
def test_kv_round_trip_sums_the_copies(P, B, L, Hkv, d):
    """head_to_seq_sum(seq_to_head(x)) = (P / H_kv, or 1) * x, exact for powers of two."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn((P, B, L // P, Hkv, d), generator=g).to(torch.bfloat16).cuda()
    rep = 1 if Hkv % P == 0 else P // Hkv
    z = U.kv_head_to_seq_sum(U.kv_seq_to_head(x, P), P, Hkv)
    torch.cuda.synchronize()
    assert torch.equal(z.float(), x.float() * rep)


def _run(B, L, H, Hkv, d, P, kind, layout, seed, tiles=None):
    t = workloads.draw(B, L, H, d, P, seed, H_kv=Hkv)
    bits = {n: workloads.to_bf16_bits(x) for n, x in t.items()}
    omask = oracle.Mask(kind) if kind in ("causal", "none") else oracle.Mask("tiles", 128, tiles)
    ref = oracle.attention_full(bits["q"], bits["k"], bits["v"], P, omask, do_tok=bits["do"])
    mask = gpu_mask(kind, L, tiles)
    if layout == U.LAYOUT_HEAD_SHARDED:
        dev = {"q": _dev(oracle.seq_to_head(bits["q"], P)), "do": _dev(oracle.seq_to_head(bits["do"], P)),
               "k": _dev(oracle.kv_seq_to_head(bits["k"], P)), "v": _dev(oracle.kv_seq_to_head(bits["v"], P))}
    else:
        dev = {n: x.cuda() for n, x in t.items()}
    o, lse = U.attn_fwd(dev["q"], dev["k"], dev["v"], P, mask, layout, kv_heads=Hkv)
    dq, dk, dv = U.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], P, mask, layout, kv_heads=Hkv)
    if layout == U.LAYOUT_HEAD_SHARDED:
        o, dq = U.head_to_seq(o, P), U.head_to_seq(dq, P)
        dk, dv = U.kv_head_to_seq_sum(dk, P, Hkv), U.kv_head_to_seq_sum(dv, P, Hkv)
    torch.cuda.synchronize()
    st, word = U.device_status()
    assert st == U.OK, hex(word)
    got = {n: oracle.bf16_to_f64(_bits(x)) for n, x in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv))}
    got["lse"] = lse.cpu().double().numpy()
    return got, ref, dev


def _check(got, ref):
    for n in ("o", "dq", "dk", "dv"):
        s = ErrStats(n)
        s.add(got[n], ref[n])
        s.check(max_abs=None if n in ("dk", "dv") else 2e-2)
    # dK, dV sum the gradients of the G query heads of each key/value head, so they grow with G:
    # the bound adds the one bf16 rounding of the result (half a unit, 2^-9 relative) to the
    # absolute tolerance of the other outputs
    for n in ("dk", "dv"):
        err = np.abs(got[n] - ref[n])
        assert np.all(err <= 2e-2 + 2.0 ** -8 * np.abs(ref[n])), (n, float(err.max()))
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(np.isneginf(got["lse"]), np.isneginf(ref["lse"]))
    assert np.abs(got["lse"][fin] - ref["lse"][fin]).max() <= LSE_MAX_ABS


CASES = [
    # name, B, L, H, H_kv, d, P, mask, layout
    ("gqa_whole_heads", 1, 384, 8, 4, 128, 2, "causal", U.LAYOUT_TOKEN_SHARDED),
    ("mqa_b2_d64", 2, 256, 8, 1, 64, 4, "causal", U.LAYOUT_TOKEN_SHARDED),
    ("gqa_copies_dense_ragged", 1, 320, 8, 2, 128, 4, "none", U.LAYOUT_TOKEN_SHARDED),
    ("gqa_head_layout_whole", 2, 256, 8, 4, 128, 2, "causal", U.LAYOUT_HEAD_SHARDED),
    ("gqa_head_layout_copies", 1, 256, 8, 2, 64, 4, "causal", U.LAYOUT_HEAD_SHARDED),
]


@pytest.mark.parametrize("name,B,L,H,Hkv,d,P,kind,layout", CASES, ids=[c[0] for c in CASES])
def test_gqa_attention_every_row(name, B, L, H, Hkv, d, P, kind, layout):
    got, ref, _ = _run(B, L, H, Hkv, d, P, kind, layout, seed=sum(map(ord, name)))
    _check(got, ref)


def test_gqa_block_sparse_every_row():
    L = 1024
    tiles = oracle.window_global_tiles(L // 128, 1, 1, 4)
    got, ref, _ = _run(1, L, 8, 2, 128, 4, "tiles", U.LAYOUT_TOKEN_SHARDED, seed=41, tiles=tiles)
    _check(got, ref)


def test_gqa_equals_multi_head_on_repeated_kv():
    """The same attention through H_kv heads and through H heads that repeat them: O and lse
    bit for bit; dK, dV equal to the group sums of the repeated-head gradients."""
    B, L, H, Hkv, d, P = 1, 512, 8, 2, 128, 4
    G = H // Hkv
    t = {n: x.cuda() for n, x in workloads.draw(B, L, H, d, P, 17, H_kv=Hkv).items()}
    mask = U.Mask.causal()
    o1, lse1 = U.attn_fwd(t["q"], t["k"], t["v"], P, mask)
    dq1, dk1, dv1 = U.attn_bwd(t["q"], t["k"], t["v"], o1, lse1, t["do"], P, mask)
    kr, vr = (x.repeat_interleave(G, dim=3).contiguous() for x in (t["k"], t["v"]))
    o2, lse2 = U.attn_fwd(t["q"], kr, vr, P, mask)
    dq2, dk2, dv2 = U.attn_bwd(t["q"], kr, vr, o2, lse2, t["do"], P, mask)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    assert (dq1.float() - dq2.float()).abs().max().item() <= 2e-2
    for a, b in ((dk1, dk2), (dv1, dv2)):
        # G bf16 terms (each rounded once) against their fp32 sum rounded once
        summed = b.float().reshape(P, B, L // P, Hkv, G, d).sum(dim=4)
        bound = 1e-2 + 2.0 ** -8 * b.float().abs().reshape(P, B, L // P, Hkv, G, d).sum(dim=4)
        assert bool(((a.float() - summed).abs() <= bound).all())

