"""GPU parity of the attention forward and backward (through the C ABI) against the fp64
oracle: every row at small sizes (several tiles, ragged tails, B > 1, both layouts, all
mask kinds, an empty query tile), every row of the GPT-1.2B-like forward, and sampled rows
of the three large workloads; plus properties that hold at any size (results do not depend
on the shard count P or on fusing the relayouts, dK/dV are deterministic)."""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_gb300 as U
import workloads
from gpu_util import (ErrStats, LSE_MAX_ABS, env_rows, f64, gpu_mask, logical, lse_logical, need_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def oracle_mask(kind, L, tiles=None, w=None):
    if kind in ("causal", "none"):
        return oracle.Mask(kind)
    if w is not None:
        return oracle.mask_for(w)
    return oracle.Mask("tiles", 128, tiles)


def run_case(B, L, H, d, P, kind, layout, seed, tiles=None, backward=True):
    t = workloads.draw(B, L, H, d, P, seed)
    bits = {n: workloads.to_bf16_bits(x) for n, x in t.items()}
    ref = oracle.attention_full(bits["q"], bits["k"], bits["v"], P, oracle_mask(kind, L, tiles),
                                do_tok=bits["do"] if backward else None)
    if layout == U.LAYOUT_HEAD_SHARDED:
        dev = {n: torch.from_numpy(oracle.seq_to_head(b, P).view(np.int16)).view(torch.bfloat16).cuda()
               for n, b in bits.items()}
    else:
        dev = {n: x.cuda() for n, x in t.items()}
    mask = gpu_mask(kind, L, tiles)
    o, lse = U.attn_fwd(dev["q"], dev["k"], dev["v"], P, mask, layout)
    outs = {"o": o}
    if backward:
        dq, dk, dv = U.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], P, mask, layout)
        outs.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    st, word = U.device_status()
    assert st == U.OK, hex(word)
    got = {}
    for n, x in outs.items():
        bits_out = x.cpu().view(torch.int16).numpy().view(np.uint16)
        if layout == U.LAYOUT_HEAD_SHARDED:
            bits_out = oracle.head_to_seq(bits_out, P)
        got[n] = oracle.bf16_to_f64(bits_out)
    got["lse"] = lse.cpu().double().numpy()
    return got, ref


def check_all(got, ref, backward=True):
    for n in (["o", "dq", "dk", "dv"] if backward else ["o"]):
        s = ErrStats(n)
        s.add(got[n], ref[n])
        s.check()
    lg, lr = got["lse"], ref["lse"]
    assert np.array_equal(np.isneginf(lg), np.isneginf(lr))
    fin = np.isfinite(lr)
    assert np.abs(lg[fin] - lr[fin]).max() <= LSE_MAX_ABS


CASES = [
    # name, B, L, H, d, P, mask, layout
    ("tiny", 1, 256, 8, 64, 4, "causal", U.LAYOUT_TOKEN_SHARDED),
    ("b2_d128_causal", 2, 384, 4, 128, 2, "causal", U.LAYOUT_TOKEN_SHARDED),
    ("ragged_token", 1, 320, 4, 128, 4, "causal", U.LAYOUT_TOKEN_SHARDED),
    ("ragged_head_dense", 1, 300, 6, 64, 3, "none", U.LAYOUT_HEAD_SHARDED),
    ("dense_p1", 1, 512, 2, 128, 1, "none", U.LAYOUT_TOKEN_SHARDED),
    ("head_layout_causal", 2, 256, 4, 128, 4, "causal", U.LAYOUT_HEAD_SHARDED),
]


@pytest.mark.parametrize("name,B,L,H,d,P,kind,layout", CASES, ids=[c[0] for c in CASES])
def test_attention_small_full(name, B, L, H, d, P, kind, layout):
    got, ref = run_case(B, L, H, d, P, kind, layout, seed=sum(map(ord, name)))
    check_all(got, ref)


@pytest.mark.parametrize("layout", [U.LAYOUT_TOKEN_SHARDED, U.LAYOUT_HEAD_SHARDED])
def test_attention_block_sparse_small(layout):
    L = 1024
    tiles = oracle.window_global_tiles(L // 128, 1, 1, 4)
    got, ref = run_case(2, L, 4, 128, 4, "tiles", layout, seed=11, tiles=tiles)
    check_all(got, ref)


def test_attention_block_sparse_empty_query_tile():
    """A query tile with no key tile: O = 0, lse = -inf, dQ = 0 there, finite elsewhere."""
    L = 640
    tiles = oracle.window_global_tiles(L // 128, 1, 0, 3).copy()
    tiles[2, :] = False
    got, ref = run_case(1, L, 4, 128, 2, "tiles", U.LAYOUT_TOKEN_SHARDED, seed=12, tiles=tiles)
    check_all(got, ref)
    assert np.all(logical(got["o"])[:, 256:384] == 0)
    assert np.all(logical(got["dq"])[:, 256:384] == 0)


def test_tiny_workload():
    w = workloads.WORKLOADS["tiny"]
    t = workloads.draw_workload(w)
    bits = {n: workloads.to_bf16_bits(x) for n, x in t.items()}
    ref = oracle.attention_full(bits["q"], bits["k"], bits["v"], w.P, oracle.mask_for(w), do_tok=bits["do"])
    dev = {n: x.cuda() for n, x in t.items()}
    o, lse = U.attn_fwd(dev["q"], dev["k"], dev["v"], w.P, U.Mask.causal())
    dq, dk, dv = U.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], w.P, U.Mask.causal())
    got = {"o": f64(o), "dq": f64(dq), "dk": f64(dk), "dv": f64(dv), "lse": lse.cpu().double().numpy()}
    check_all(got, ref)


def test_shard_count_and_fusion_do_not_change_results():
    """Per-head attention does not depend on P, nor on reading through the token layout
    instead of relayouting first: forward outputs and dK, dV must be bit-identical."""
    B, L, H, d = 1, 512, 8, 128
    g = torch.Generator().manual_seed(7)
    x = {n: torch.randn((B, L, H, d), generator=g).to(torch.bfloat16) for n in ("q", "k", "v", "do")}
    base = None
    for P in (1, 2, 4, 8):
        tok = {n: workloads.shard_tokens(t, P).cuda() for n, t in x.items()}
        for layout in (U.LAYOUT_TOKEN_SHARDED, U.LAYOUT_HEAD_SHARDED):
            ins = tok if layout == U.LAYOUT_TOKEN_SHARDED else {n: U.seq_to_head(t, P) for n, t in tok.items()}
            o, lse = U.attn_fwd(ins["q"], ins["k"], ins["v"], P, U.Mask.causal(), layout)
            dq, dk, dv = U.attn_bwd(ins["q"], ins["k"], ins["v"], o, lse, ins["do"], P, U.Mask.causal(), layout)
            if layout == U.LAYOUT_HEAD_SHARDED:
                o, dq, dk, dv = (U.head_to_seq(t, P) for t in (o, dq, dk, dv))
            res = {n: t.cpu().permute(1, 0, 2, 3, 4).reshape(B, L, H, d) for n, t in
                   (("o", o), ("dq", dq), ("dk", dk), ("dv", dv))}
            res["lse"] = lse.cpu().permute(1, 0, 2, 3).reshape(B, H, L)
            if base is None:
                base = res
                continue
            for n in ("o", "lse", "dk", "dv"):
                assert torch.equal(res[n].view(torch.int16) if res[n].dtype == torch.bfloat16 else res[n],
                                   base[n].view(torch.int16) if base[n].dtype == torch.bfloat16 else base[n]), (P, layout, n)
            err = (res["dq"].float() - base["dq"].float()).abs().max().item()
            assert err <= 2e-2, (P, layout, err)


def test_forward_head_groups_with_a_partial_last_group():
    """The causal forward deals its CTAs out in groups of G heads (G from the K/V bytes per
    head: 2 at L = 32768, d_h = 128). With 3 heads the last group is partial and its spare CTAs
    leave at once. Every head's O and lse must equal, bit for bit, the same head run alone
    (one head: one group, the plain order)."""
    B, L, H, d, P = 1, 32768, 3, 128, 1
    g = torch.Generator().manual_seed(21)
    x = {n: torch.randn((P, B, L, H, d), generator=g).mul_(0.5).to(torch.bfloat16).cuda() for n in ("q", "k", "v")}
    o, lse = U.attn_fwd(x["q"], x["k"], x["v"], P, U.Mask.causal())
    for h in range(H):
        one = {n: t[:, :, :, h:h + 1, :].contiguous() for n, t in x.items()}
        o1, lse1 = U.attn_fwd(one["q"], one["k"], one["v"], P, U.Mask.causal())
        assert torch.equal(o[:, :, :, h:h + 1, :].view(torch.int16), o1.view(torch.int16)), h
        assert torch.equal(lse[:, :, h:h + 1, :], lse1), h
    st, word = U.device_status()
    assert st == U.OK, hex(word)


def test_backward_unit_groups_with_a_partial_last_group():
    """Short causal sequences run the backward's grouped order (G units per grid row: 2 at
    L = 16384, d_h = 128). With 3 heads the last group is partial and its spare CTAs leave at
    once. Each head's dK and dV must equal, bit for bit, the same head run alone (one unit: the
    plain kernel), and its dQ must agree up to the order of the fp32 additions."""
    B, L, H, d, P = 1, 16384, 3, 128, 1
    g = torch.Generator().manual_seed(22)
    x = {n: torch.randn((P, B, L, H, d), generator=g).mul_(0.5).to(torch.bfloat16).cuda()
         for n in ("q", "k", "v", "do")}
    mask = U.Mask.causal()
    o, lse = U.attn_fwd(x["q"], x["k"], x["v"], P, mask)
    dq, dk, dv = U.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], P, mask)
    for h in range(H):
        one = {n: t[:, :, :, h:h + 1, :].contiguous() for n, t in x.items()}
        o1, lse1 = U.attn_fwd(one["q"], one["k"], one["v"], P, mask)
        dq1, dk1, dv1 = U.attn_bwd(one["q"], one["k"], one["v"], o1, lse1, one["do"], P, mask)
        assert torch.equal(dk[:, :, :, h:h + 1, :].view(torch.int16), dk1.view(torch.int16)), h
        assert torch.equal(dv[:, :, :, h:h + 1, :].view(torch.int16), dv1.view(torch.int16)), h
        err = (dq[:, :, :, h:h + 1, :].float() - dq1.float()).abs().max().item()
        assert err <= 2e-2, (h, err)
    st, word = U.device_status()
    assert st == U.OK, hex(word)


def test_repeat_runs_are_deterministic_except_dq():
    w = workloads.Workload("rep", 1, 1024, 4, 128, 4, "causal", True, 5)
    t = {n: x.cuda() for n, x in workloads.draw_workload(w).items()}
    runs = []
    for _ in range(3):
        o, lse = U.attn_fwd(t["q"], t["k"], t["v"], w.P, U.Mask.causal())
        dq, dk, dv = U.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], w.P, U.Mask.causal())
        runs.append([x.clone() for x in (o, lse, dk, dv)])
    for r in runs[1:]:
        for a, b in zip(r, runs[0]):
            assert torch.equal(a, b)


def test_gpt1p2b_forward_every_row():
    w = workloads.WORKLOADS["gpt1.2b"]
    t = workloads.draw_workload(w, names=("q", "k", "v"))
    bits = {n: workloads.to_bf16_bits(x) for n, x in t.items()}
    dev = {n: x.cuda() for n, x in t.items()}
    o, lse = U.attn_fwd(dev["q"], dev["k"], dev["v"], w.P, U.Mask.causal())
    torch.cuda.synchronize()
    ref = oracle.attention_full(bits["q"], bits["k"], bits["v"], w.P, oracle.mask_for(w))
    check_all({"o": f64(o), "lse": lse.cpu().double().numpy()}, ref, backward=False)


# gpt7b and block_sparse check all 4096 rows on every head. Long and the grouped-query layer
# check every head too, each on its own quarter of the rows (query head h takes the sampled
# rows whose index is h mod 4, plus the first and last row of the sequence): at P=32 each head
# of Long is its own head group, so all 32 groups' fused relayouts are compared, and the fp64
# oracle does the work of 8 whole heads; every key/value head of the grouped layer sees all
# 4096 rows through its 4 query heads.
SAMPLED = [("gpt7b", False), ("long", True), ("block_sparse", False), ("gpt7b_gqa", True)]


def _head_rows(rows: np.ndarray, L: int, H: int, split: bool):
    """[(heads, rows)] groups for the oracle: every head with every row, or heads h = r mod 4
    with the rows of index r mod 4 (plus the sequence's first and last rows)."""
    if not split:
        return [(tuple(range(H)), rows)]
    edge = rows[(rows[:, 0] == 0) & ((rows[:, 1] == 0) | (rows[:, 1] == L - 1))]
    out = []
    for r in range(4):
        sub = np.unique(np.concatenate([edge, rows[r::4]]), axis=0)
        out.append((tuple(range(r, H, 4)), sub))
    return out


@pytest.mark.parametrize("name,split", SAMPLED, ids=[s[0] for s in SAMPLED])
def test_large_workload_sampled_rows(name, split):
    """4096 seeded query rows: O, lse and dQ of those rows from a pass with the full dO
    (run A), and dK, dV over every key from a pass whose dO is zero outside the checked
    (row, head) pairs (run B), which then hold exactly their gradient contributions. With
    grouped key/value heads, dK and dV are compared with the sum of the contributions of the
    query heads of each key/value head."""
    w = workloads.WORKLOADS[name]
    t = workloads.draw_workload(w)
    P, B, L, H, d = w.P, w.B, w.L, w.H, w.d
    rows = workloads.sample_rows(B, L, env_rows(w.sampled_rows), seed=w.seed)
    groups = _head_rows(rows, L, H, split)
    keep = torch.zeros((B, L, H), dtype=torch.bool)
    for hs, rr in groups:
        sel = keep[torch.from_numpy(rr[:, 0]), torch.from_numpy(rr[:, 1])]
        sel[:, list(hs)] = True
        keep[torch.from_numpy(rr[:, 0]), torch.from_numpy(rr[:, 1])] = sel
    keep_tok = keep.reshape(B, P, L // P, H).permute(1, 0, 2, 3)[..., None]
    dev = {n: x.cuda() for n, x in t.items()}
    mask = gpu_mask(w.mask, L, w=w) if w.mask == "block_sparse" else gpu_mask(w.mask, L)
    o, lse = U.attn_fwd(dev["q"], dev["k"], dev["v"], P, mask)
    dqA, _, _ = U.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], P, mask)
    do_b = dev["do"] * keep_tok.cuda().to(torch.bfloat16)
    dqB, dkB, dvB = U.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, do_b, P, mask)
    torch.cuda.synchronize()
    st, word = U.device_status()
    assert st == U.OK, hex(word)

    def logical_t(x):
        return x.cpu().permute(1, 0, 2, 3, 4).reshape(B, L, x.shape[3], d)

    O, dQA, dQB, dKB, dVB = (logical_t(x) for x in (o, dqA, dqB, dkB, dvB))
    LSE = lse.cpu().permute(1, 0, 2, 3).reshape(B, H, L)
    # (row, head) pairs outside the checked set get no dQ in run B
    assert torch.count_nonzero(dQB.float()[~keep]) == 0
    del dev, o, dqA, dqB, dkB, dvB, do_b
    torch.cuda.empty_cache()

    stats = {n: ErrStats(n) for n in ("o", "dq", "dk", "dv")}
    G = H // w.Hkv
    kv_ref = {}  # (b, key/value head) -> [summed dK, summed dV, query heads seen]
    lse_err = 0.0
    bits = {n: workloads.to_bf16_bits(x) for n, x in t.items()}
    workers = min(8, os.cpu_count() or 1)
    seen = set()
    for hs, rr in groups:
        for res in oracle.attention_sampled(bits["q"], bits["k"], bits["v"], bits["do"], P, oracle.mask_for(w), rr,
                                            heads=hs, workers=workers):
            b, h, r = res["b"], res["h"], torch.from_numpy(res["rows"])
            seen.add(h)
            stats["o"].add(O[b, r, h].double().numpy(), res["o"])
            stats["dq"].add(dQA[b, r, h].double().numpy(), res["dq"])
            acc = kv_ref.setdefault((b, res["kvh"]), [0.0, 0.0, 0])
            acc[0] = acc[0] + res["dk"]
            acc[1] = acc[1] + res["dv"]
            acc[2] += 1
            lse_err = max(lse_err, float(np.abs(LSE[b, h, r].double().numpy() - res["lse"]).max()))
    assert seen == set(range(H))
    excess = 0.0  # grouped heads: largest error beyond the bf16 rounding of the summed gradient
    for (b, kvh), (rdk, rdv, n) in kv_ref.items():
        assert n == G
        for name, got, ref in (("dk", dKB[b, :, kvh], rdk), ("dv", dVB[b, :, kvh], rdv)):
            g64 = got.double().numpy()
            stats[name].add(g64, ref)
            excess = max(excess, float((np.abs(g64 - ref) - 2.0 ** -8 * np.abs(ref)).max()))
    for n, s in stats.items():
        # with grouped key/value heads dK, dV sum G query heads' gradients and grow with G: their
        # bound adds the one bf16 rounding of the result (see test_gqa_gpu.py)
        s.check(max_abs=None if (G > 1 and n in ("dk", "dv")) else 2e-2)
    if G > 1:
        assert excess <= 2e-2, excess
    assert lse_err <= LSE_MAX_ABS, lse_err


GUARD = 4096


def _guarded(shape, dtype):
    """A tensor of `shape` in the middle of a buffer whose both ends hold a canary pattern."""
    n = int(np.prod(shape))
    elem = torch.int16 if dtype == torch.bfloat16 else torch.int32
    buf = torch.full((n + 2 * GUARD,), 0x5A5A, dtype=elem, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(dtype).view(shape)


def _guards_intact(buf):
    h = buf.cpu()
    return bool((h[:GUARD] == 0x5A5A).all() and (h[-GUARD:] == 0x5A5A).all())


@pytest.mark.parametrize("B,L,H,d,P,kind,layout", [(1, 320, 4, 128, 4, "causal", U.LAYOUT_TOKEN_SHARDED),
                                                    (1, 300, 6, 64, 3, "none", U.LAYOUT_HEAD_SHARDED),
                                                    (2, 640, 4, 128, 2, "tiles", U.LAYOUT_TOKEN_SHARDED)])
def test_attention_writes_stay_inside_outputs(B, L, H, d, P, kind, layout):
    """Ragged tails, both layouts and block-sparse lists: every output and the workspace are
    surrounded by canaries, which must be untouched after forward and backward."""
    t = workloads.draw(B, L, H, d, P, seed=31)
    if layout == U.LAYOUT_HEAD_SHARDED:
        dev = {n: U.seq_to_head(x.cuda(), P) for n, x in t.items()}
    else:
        dev = {n: x.cuda() for n, x in t.items()}
    tiles = oracle.window_global_tiles(-(-L // 128), 1, 0, 3) if kind == "tiles" else None
    mask = gpu_mask(kind, L, tiles)
    shape = dev["q"].shape
    bufs = {}
    bufs["o"], o = _guarded(shape, torch.bfloat16)
    bufs["lse"], lse = _guarded((P, B, H // P, L), torch.float32)
    bufs["dq"], dq = _guarded(shape, torch.bfloat16)
    bufs["dk"], dk = _guarded(shape, torch.bfloat16)
    bufs["dv"], dv = _guarded(shape, torch.bfloat16)
    ws_bytes = U.ulysses_attn_bwd_workspace_size(U.token_shape(t["q"], P))
    ws_buf = torch.full((ws_bytes + 2 * GUARD * 64,), 0x5A, dtype=torch.uint8, device="cuda")
    ws = ws_buf[GUARD * 64:GUARD * 64 + ws_bytes]
    U.attn_fwd(dev["q"], dev["k"], dev["v"], P, mask, layout, o=o, lse=lse)
    U.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], P, mask, layout, dq=dq, dk=dk, dv=dv, workspace=ws)
    torch.cuda.synchronize()
    assert U.device_status()[0] == U.OK
    for name, buf in bufs.items():
        assert _guards_intact(buf), name
    wh = ws_buf.cpu()
    assert bool((wh[:GUARD * 64] == 0x5A).all() and (wh[-GUARD * 64:] == 0x5A).all()), "workspace"
    for x in (o, dq, dk, dv):
        assert torch.isfinite(x.float()).all()
