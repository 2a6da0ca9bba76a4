"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

None of these re-types the oracle's own formulas. The pins are:
* relayouts: the receiver rule written as a closed-form cell code, an independent numpy
  reshape/transpose expression, round trip, bijection, P = 1 identity;
* forward: closed forms (Q = 0 gives the mean of the permitted values; V = 1 gives 1;
  causal row 0 gives V_0), invariances (joint key/value permutation, a constant shift of
  every key), and torch's fp64 scaled_dot_product_attention as an independent library;
* backward: central finite differences in fp64, torch fp64 autograd, and the exact
  column sums  sum_j dK_j = 0  and  sum_j dV_j = sum_i dO_i.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import Mask
import workloads

RNG = np.random.default_rng(1234)


def rand_bits(shape):
    return RNG.integers(0, 1 << 16, size=shape, dtype=np.uint16)


# ----------------------------------------------------------------------------- relayouts

SHAPES = [(4, 2, 16, 8, 3), (3, 1, 9, 6, 5), (1, 2, 8, 4, 2), (8, 1, 64, 8, 4), (2, 3, 6, 2, 1)]


@pytest.mark.parametrize("P,B,L,H,d", SHAPES)
def test_relayout_matches_numpy_transpose(P, B, L, H, d):
    Lp, Hp = L // P, H // P
    x = rand_bits((P, B, Lp, H, d))
    y = oracle.seq_to_head(x, P)
    # independent expression: split heads into (group, head-in-group), move group first,
    # then merge (sender rank, local token) into the global token index
    expect = x.reshape(P, B, Lp, P, Hp, d).transpose(3, 1, 0, 2, 4, 5).reshape(P, B, L, Hp, d)
    assert np.array_equal(y, expect)
    z = oracle.head_to_seq(y, P)
    assert np.array_equal(z, x)


@pytest.mark.parametrize("P,B,L,H,d", SHAPES)
def test_relayout_receiver_rule(P, B, L, H, d):
    """Each receiver holds one contiguous head group from every sender, token blocks in
    sender order: cell (r, b, t, h) carries a code; receiver g row s head j must carry the
    code of sender s // Lp, token s % Lp, head g*Hp + j."""
    Lp, Hp = L // P, H // P
    r, b, t, h, e = np.meshgrid(np.arange(P), np.arange(B), np.arange(Lp), np.arange(H), np.arange(d),
                                indexing="ij")
    code = ((((r * B + b) * Lp + t) * H + h) * d + e).astype(np.int64)
    y = oracle.seq_to_head(code, P)
    g, b2, s, j, e2 = np.meshgrid(np.arange(P), np.arange(B), np.arange(L), np.arange(Hp), np.arange(d),
                                  indexing="ij")
    want = (((((s // Lp) * B + b2) * Lp + s % Lp) * H + g * Hp + j) * d + e2)
    assert np.array_equal(y, want)


def test_relayout_bijection_and_identity():
    x = rand_bits((4, 2, 8, 8, 4))
    y = oracle.seq_to_head(x, 4)
    assert np.array_equal(np.sort(x.ravel()), np.sort(y.ravel()))
    x1 = rand_bits((1, 2, 16, 4, 8))
    assert np.array_equal(oracle.seq_to_head(x1, 1), x1)
    assert np.array_equal(oracle.head_to_seq(x1, 1), x1)


def test_relayout_keeps_nan_and_denormal_bits():
    specials = np.array([0x7FC1, 0xFFFF, 0x7F81, 0x0001, 0x8001, 0x8000, 0x7F80, 0xFF80], dtype=np.uint16)
    x = np.resize(specials, (2, 1, 4, 4, 8)).astype(np.uint16)
    y = oracle.seq_to_head(x, 2)
    assert np.array_equal(oracle.head_to_seq(y, 2), x)


def test_relayout_fp64_elements_and_bad_shapes():
    x = RNG.standard_normal((2, 1, 3, 4, 5))
    assert np.array_equal(oracle.head_to_seq(oracle.seq_to_head(x, 2), 2), x)
    with pytest.raises(AssertionError):
        oracle.seq_to_head(rand_bits((3, 1, 4, 4, 2)), 3)   # H % P != 0


def test_bf16_widening_matches_torch_for_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ----------------------------------------------------------------------------- forward

def rand_tok(P, B, L, H, d, scale=1.0):
    return RNG.standard_normal((P, B, L // P, H, d)) * scale


def logical(x_tok):
    """Token-sharded [P][B][Lp][H][d] -> logical [B][L][H][d] (the sequence re-joined)."""
    P, B, Lp, H, d = x_tok.shape
    return np.ascontiguousarray(x_tok.transpose(1, 0, 2, 3, 4).reshape(B, P * Lp, H, d))


def lse_logical(lse, P):
    """[P][B][Hp][L] -> [B][H][L]."""
    _, B, Hp, L = lse.shape
    return lse.transpose(1, 0, 2, 3).reshape(B, P * Hp, L)


def tiles_mask(L, tile, seed=0, empty_tile=None):
    n = L // tile
    t = oracle.window_global_tiles(n, 1, 0, 3)
    if empty_tile is not None:
        t = t.copy()
        t[empty_tile, :] = False
    return Mask("tiles", tile, t)


def dense_bool(mask, L):
    return mask.rows(np.arange(L), L)


MASKS = ["causal", "none", "tiles"]


def make_mask(kind, L):
    return tiles_mask(L, 4) if kind == "tiles" else Mask(kind)


@pytest.mark.parametrize("kind", MASKS)
def test_forward_zero_query_gives_mean_of_permitted_values(kind):
    P, B, L, H, d = 2, 2, 16, 4, 8
    mask = make_mask(kind, L)
    q = np.zeros((P, B, L // P, H, d))
    k, v = rand_tok(P, B, L, H, d), rand_tok(P, B, L, H, d)
    out = oracle.attention_full(q, k, v, P, mask)
    allow = dense_bool(mask, L).astype(np.float64)
    cnt = allow.sum(1)
    V = logical(v)
    O = logical(out["o"])
    want = np.einsum("ij,bjhd->bihd", allow, V) / cnt[None, :, None, None]
    np.testing.assert_allclose(O, want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_logical(out["lse"], P), np.broadcast_to(np.log(cnt), (B, H, L)),
                               rtol=0, atol=1e-12)


@pytest.mark.parametrize("kind", MASKS)
def test_forward_unit_values_give_unit_output(kind):
    """Softmax weights of every row sum to one, so V = 1 gives O = 1."""
    P, B, L, H, d = 2, 1, 16, 2, 4
    out = oracle.attention_full(rand_tok(P, B, L, H, d), rand_tok(P, B, L, H, d),
                                np.ones((P, B, L // P, H, d)), P, make_mask(kind, L))
    np.testing.assert_allclose(out["o"], 1.0, rtol=0, atol=1e-12)


def test_forward_causal_row_zero():
    P, B, L, H, d = 4, 1, 16, 4, 8
    q, k, v = (rand_tok(P, B, L, H, d) for _ in range(3))
    out = oracle.attention_full(q, k, v, P, Mask("causal"))
    O, V, Q, K = logical(out["o"]), logical(v), logical(q), logical(k)
    np.testing.assert_allclose(O[:, 0], V[:, 0], rtol=0, atol=1e-15)
    s00 = np.einsum("bhd,bhd->bh", Q[:, 0], K[:, 0]) / math.sqrt(d)
    np.testing.assert_allclose(lse_logical(out["lse"], P)[:, :, 0], s00, rtol=0, atol=1e-13)


@pytest.mark.parametrize("kind", MASKS)
@pytest.mark.parametrize("P", [1, 2, 4])
def test_forward_matches_torch_sdpa(kind, P):
    B, L, H, d = 2, 32, 4, 16
    mask = tiles_mask(L, 8) if kind == "tiles" else Mask(kind)
    q, k, v = (rand_tok(P, B, L, H, d) for _ in range(3))
    out = oracle.attention_full(q, k, v, P, mask)
    tq, tk, tv = (torch.from_numpy(logical(x)).permute(0, 2, 1, 3) for x in (q, k, v))
    am = torch.from_numpy(dense_bool(mask, L))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=am)
    np.testing.assert_allclose(logical(out["o"]), ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    s = torch.einsum("bhid,bhjd->bhij", tq, tk) / math.sqrt(d)
    s = s.masked_fill(~am, -math.inf)
    np.testing.assert_allclose(lse_logical(out["lse"], P), torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def test_forward_is_independent_of_shard_count():
    B, L, H, d = 1, 32, 8, 8
    x = [RNG.standard_normal((B, L, H, d)) for _ in range(3)]
    outs = []
    for P in (1, 2, 4, 8):
        tok = [np.ascontiguousarray(t.reshape(B, P, L // P, H, d).transpose(1, 0, 2, 3, 4)) for t in x]
        outs.append(logical(oracle.attention_full(*tok, P, Mask("causal"))["o"]))
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=1e-14)


def test_forward_dense_invariances():
    """Bidirectional: permuting keys and values together changes nothing, and adding one
    vector c to every key adds scale*Q_i.c to the whole row i of S, so O is unchanged."""
    P, B, L, H, d = 2, 1, 16, 2, 8
    q, k, v = (rand_tok(P, B, L, H, d) for _ in range(3))
    base = oracle.attention_full(q, k, v, P, Mask("none"))
    perm = RNG.permutation(L)
    K, V = logical(k), logical(v)
    def tok(xl):
        return np.ascontiguousarray(xl.reshape(B, P, L // P, H, d).transpose(1, 0, 2, 3, 4))
    out = oracle.attention_full(q, tok(K[:, perm]), tok(V[:, perm]), P, Mask("none"))
    np.testing.assert_allclose(out["o"], base["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out["lse"], base["lse"], rtol=0, atol=1e-12)
    c = RNG.standard_normal(d)
    out = oracle.attention_full(q, tok(K + c), v, P, Mask("none"))
    np.testing.assert_allclose(out["o"], base["o"], rtol=0, atol=1e-12)


def test_fully_masked_row_reading():
    """A query tile with no permitted key: O = 0, LSE = -inf, zero gradients, no NaN."""
    P, B, L, H, d = 2, 1, 16, 2, 4
    mask = tiles_mask(L, 4, empty_tile=2)
    q, k, v, do = (rand_tok(P, B, L, H, d) for _ in range(4))
    out = oracle.attention_full(q, k, v, P, mask, do_tok=do)
    for key in ("o", "dq", "dk", "dv"):
        assert np.all(np.isfinite(out[key]))
    O, dQ = logical(out["o"]), logical(out["dq"])
    assert np.all(O[:, 8:12] == 0) and np.all(dQ[:, 8:12] == 0)
    assert np.all(np.isneginf(lse_logical(out["lse"], P)[:, :, 8:12]))
    assert np.all(np.isfinite(lse_logical(out["lse"], P)[:, :, :8]))


# ----------------------------------------------------------------------------- backward

def loss(q, k, v, do, P, mask):
    return float(np.sum(do * oracle.attention_full(q, k, v, P, mask)["o"]))


@pytest.mark.parametrize("kind", ["causal", "tiles"])
def test_backward_central_finite_differences(kind):
    P, B, L, H, d = 2, 1, 16, 4, 8
    mask = make_mask(kind, L)
    q, k, v, do = (rand_tok(P, B, L, H, d) for _ in range(4))
    g = oracle.attention_full(q, k, v, P, mask, do_tok=do)
    eps = 1e-6
    for name, grad in (("q", g["dq"]), ("k", g["dk"]), ("v", g["dv"])):
        fd = np.zeros_like(grad)
        base = {"q": q, "k": k, "v": v}
        for idx in np.ndindex(grad.shape):
            plus = {n: a.copy() for n, a in base.items()}
            minus = {n: a.copy() for n, a in base.items()}
            plus[name][idx] += eps
            minus[name][idx] -= eps
            fd[idx] = (loss(plus["q"], plus["k"], plus["v"], do, P, mask)
                       - loss(minus["q"], minus["k"], minus["v"], do, P, mask)) / (2 * eps)
        err = np.linalg.norm(fd - grad) / np.linalg.norm(grad)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("kind", MASKS)
def test_backward_matches_torch_autograd(kind):
    P, B, L, H, d = 4, 2, 32, 8, 16
    mask = tiles_mask(L, 8) if kind == "tiles" else Mask(kind)
    q, k, v, do = (rand_tok(P, B, L, H, d) for _ in range(4))
    g = oracle.attention_full(q, k, v, P, mask, do_tok=do)
    tq, tk, tv = (torch.from_numpy(logical(x)).permute(0, 2, 1, 3).requires_grad_(True) for x in (q, k, v))
    am = torch.from_numpy(dense_bool(mask, L))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=am)
    o.backward(torch.from_numpy(logical(do)).permute(0, 2, 1, 3))
    for name, t in (("dq", tq), ("dk", tk), ("dv", tv)):
        np.testing.assert_allclose(logical(g[name]), t.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("kind", MASKS)
def test_backward_column_sums(kind):
    """sum_j dS_ij = 0 for every row, hence sum_j dK_j = 0; and sum_j dV_j = sum_i dO_i
    over rows that have a permitted key (their softmax weights sum to one)."""
    P, B, L, H, d = 2, 2, 16, 4, 8
    mask = make_mask(kind, L)
    q, k, v, do = (rand_tok(P, B, L, H, d) for _ in range(4))
    g = oracle.attention_full(q, k, v, P, mask, do_tok=do)
    dK, dV, dO = logical(g["dk"]), logical(g["dv"]), logical(do)
    np.testing.assert_allclose(dK.sum(axis=1), 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dV.sum(axis=1), dO.sum(axis=1), rtol=0, atol=1e-12)


def test_sampled_mode_matches_full_mode():
    P, B, L, H, d = 2, 2, 32, 4, 8
    mask = tiles_mask(L, 8)
    q, k, v, do = (rand_tok(P, B, L, H, d) for _ in range(4))
    rows = workloads.sample_rows(B, L, 11, seed=5)
    full = oracle.attention_full(q, k, v, P, mask, do_tok=do)
    # a pass whose dO is zero outside the sampled rows has exactly their contributions
    keep = np.zeros((B, L), dtype=bool)
    keep[rows[:, 0], rows[:, 1]] = True
    dol = logical(do) * keep[:, :, None, None]
    do_masked = np.ascontiguousarray(dol.reshape(B, P, L // P, H, d).transpose(1, 0, 2, 3, 4))
    part = oracle.attention_full(q, k, v, P, mask, do_tok=do_masked)
    O, LSE, dQ = logical(full["o"]), lse_logical(full["lse"], P), logical(full["dq"])
    dK, dV = logical(part["dk"]), logical(part["dv"])
    seen = 0
    for res in oracle.attention_sampled(q, k, v, do, P, mask, rows):
        b, h, r = res["b"], res["h"], res["rows"]
        np.testing.assert_allclose(res["o"], O[b, r, h], rtol=0, atol=1e-13)
        np.testing.assert_allclose(res["lse"], LSE[b, h, r], rtol=0, atol=1e-13)
        np.testing.assert_allclose(res["dq"], dQ[b, r, h], rtol=0, atol=1e-13)
        np.testing.assert_allclose(res["dk"], dK[b, :, h], rtol=0, atol=1e-13)
        np.testing.assert_allclose(res["dv"], dV[b, :, h], rtol=0, atol=1e-13)
        seen += 1
    assert seen == B * H


def test_sample_rows_recipe():
    rows = workloads.sample_rows(2, 1000, 64, seed=3)
    assert len(rows) == 64 and len({tuple(r) for r in rows}) == 64
    assert (0, 0) in {tuple(r) for r in rows} and (0, 999) in {tuple(r) for r in rows}
    assert np.array_equal(rows, workloads.sample_rows(2, 1000, 64, seed=3))


def test_golden_block_sparse_tile_counts():
    """Tile counts of the workloads' window-plus-global pattern (tests/golden)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "block_sparse_tiles.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    for L, tile, wb, wa, gs, active, total in ((int(x) for x in r) for r in rows):
        t = oracle.window_global_tiles(L // tile, wb, wa, gs)
        assert int(t.sum()) == active and t.size == total


# ----------------------------------------------------------------------------- grouped K/V heads

GQA = [(2, 8, 2), (4, 8, 2), (4, 8, 1), (8, 8, 4), (2, 4, 4)]  # (P, H, Hkv): both regimes, MQA, MHA


@pytest.mark.parametrize("P,H,Hkv", GQA)
def test_kv_relayout_receiver_rule(P, H, Hkv):
    B, L, d = 2, 16, 3
    Lp = L // P
    r, b, t, h, e = np.meshgrid(np.arange(P), np.arange(B), np.arange(Lp), np.arange(Hkv), np.arange(d), indexing="ij")
    code = ((((r * B + b) * Lp + t) * Hkv + h) * d + e).astype(np.int64)
    y = oracle.kv_seq_to_head(code, P)
    Hkvp = Hkv // P if Hkv % P == 0 else 1
    assert y.shape == (P, B, L, Hkvp, d)
    g, b2, s, j, e2 = np.meshgrid(np.arange(P), np.arange(B), np.arange(L), np.arange(Hkvp), np.arange(d), indexing="ij")
    # receiver g holds K/V heads [g*Hkv/P, ...) or, replicated, head floor(g*Hkv/P)
    src_head = g * Hkvp + j if Hkv % P == 0 else (g * Hkv) // P
    want = (((s // Lp) * B + b2) * Lp + s % Lp) * Hkv * d + src_head * d + e2
    assert np.array_equal(y, want)
    if Hkv % P == 0:
        assert np.array_equal(y, oracle.seq_to_head(code, P))


@pytest.mark.parametrize("P,H,Hkv", GQA)
def test_kv_relayout_adjoint_identity(P, H, Hkv):
    """<y, R x> == <R^T y, x> for the relayout R and its summing adjoint R^T."""
    B, L, d = 2, 8, 4
    x = RNG.standard_normal((P, B, L // P, Hkv, d))
    Hkvp = Hkv // P if Hkv % P == 0 else 1
    y = RNG.standard_normal((P, B, L, Hkvp, d))
    lhs = np.sum(y * oracle.kv_seq_to_head(x, P))
    rhs = np.sum(oracle.kv_head_to_seq_sum(y, P, Hkv) * x)
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def repeat_kv(x_tok, G):
    """[P][B][Lp][Hkv][d] -> [P][B][Lp][Hkv*G][d], each K/V head repeated for its G query heads."""
    return np.repeat(x_tok, G, axis=3)


@pytest.mark.parametrize("P,H,Hkv", GQA)
@pytest.mark.parametrize("kind", ["causal", "none"])
def test_gqa_equals_mha_on_repeated_heads(P, H, Hkv, kind):
    B, L, d = 1, 16, 8
    G = H // Hkv
    q, do = rand_tok(P, B, L, H, d), rand_tok(P, B, L, H, d)
    k, v = rand_tok(P, B, L, Hkv, d), rand_tok(P, B, L, Hkv, d)
    gqa = oracle.attention_full(q, k, v, P, Mask(kind), do_tok=do)
    mha = oracle.attention_full(q, repeat_kv(k, G), repeat_kv(v, G), P, Mask(kind), do_tok=do)
    for n in ("o", "lse", "dq"):
        np.testing.assert_allclose(gqa[n], mha[n], rtol=0, atol=1e-13)
    for n in ("dk", "dv"):
        summed = mha[n].reshape(P, B, L // P, Hkv, G, d).sum(axis=4)
        np.testing.assert_allclose(gqa[n], summed, rtol=0, atol=1e-12)


@pytest.mark.skipif(
    "enable_gqa" not in torch.nn.functional.scaled_dot_product_attention.__doc__, reason="torch without enable_gqa")
@pytest.mark.parametrize("P,H,Hkv", [(2, 8, 2), (4, 8, 1)])
def test_gqa_matches_torch_sdpa(P, H, Hkv):
    B, L, d = 2, 16, 8
    q, do = rand_tok(P, B, L, H, d), rand_tok(P, B, L, H, d)
    k, v = rand_tok(P, B, L, Hkv, d), rand_tok(P, B, L, Hkv, d)
    g = oracle.attention_full(q, k, v, P, Mask("causal"), do_tok=do)
    tq, tk, tv = (torch.from_numpy(logical(x)).permute(0, 2, 1, 3).requires_grad_(True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, enable_gqa=True)
    o.backward(torch.from_numpy(logical(do)).permute(0, 2, 1, 3))
    np.testing.assert_allclose(logical(g["o"]), o.detach().permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    for name, t in (("dq", tq), ("dk", tk), ("dv", tv)):
        np.testing.assert_allclose(logical(g[name]), t.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)


# --------------------------------------------------------------------------- projections

def _perm_weight(n_out, n_in, seed):
    """A 0/1 matrix whose row i selects input feature perm[i] (so y[:, i] = x[:, perm[i]])."""
    perm = np.random.default_rng(seed).integers(0, n_in, size=n_out)
    w = np.zeros((n_out, n_in))
    w[np.arange(n_out), perm] = 1.0
    return w, perm


@pytest.mark.parametrize("P,H,Hkv,d", [(2, 4, 4, 8), (4, 8, 2, 16), (2, 4, 1, 8)])
def test_qkv_projection_with_selection_weights(P, H, Hkv, d):
    """One-hot weight rows copy chosen input features: catches a transposed weight, a wrong
    Q/K/V block order and a wrong head split exactly."""
    B, L, hidden = 2, 16, 24
    x = RNG.standard_normal((P, B, L // P, hidden))
    w, perm = _perm_weight((H + 2 * Hkv) * d, hidden, seed=H + Hkv)
    out = oracle.qkv_projection(x, w, H, Hkv, d)
    flat = x[..., perm]  # [P][B][Lp][(H + 2 Hkv) d]
    np.testing.assert_array_equal(out["q"].reshape(P, B, L // P, -1), flat[..., :H * d])
    np.testing.assert_array_equal(out["k"].reshape(P, B, L // P, -1), flat[..., H * d:(H + Hkv) * d])
    np.testing.assert_array_equal(out["v"].reshape(P, B, L // P, -1), flat[..., (H + Hkv) * d:])


def test_projections_match_torch_linear():
    P, B, L, H, Hkv, d, hidden = 4, 2, 32, 4, 2, 8, 40
    x = RNG.standard_normal((P, B, L // P, hidden))
    w = RNG.standard_normal(((H + 2 * Hkv) * d, hidden))
    wo = RNG.standard_normal((hidden, H * d))
    out = oracle.qkv_projection(x, w, H, Hkv, d)
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(w)).numpy()
    got = np.concatenate([out[n].reshape(P, B, L // P, -1) for n in ("q", "k", "v")], axis=-1)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    o = RNG.standard_normal((P, B, L // P, H, d))
    y = oracle.out_projection(o, wo)
    ref = torch.nn.functional.linear(torch.from_numpy(o.reshape(P, B, L // P, H * d)), torch.from_numpy(wo)).numpy()
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


def test_projection_of_shards_equals_projection_of_the_sequence():
    """Each rank projects its own tokens: sharding the sequence first or after gives the same rows."""
    B, L, hidden, H, d = 2, 24, 16, 4, 8
    x = RNG.standard_normal((B, L, hidden))
    w = RNG.standard_normal((3 * H * d, hidden))
    ref = oracle.qkv_projection(x[None], w, H, H, d)  # one shard holding the whole sequence
    for P in (2, 3, 4):
        x_tok = x.reshape(B, P, L // P, hidden).transpose(1, 0, 2, 3)
        out = oracle.qkv_projection(x_tok, w, H, H, d)
        for n in ("q", "k", "v"):
            merged = out[n].transpose(1, 0, 2, 3, 4).reshape(B, L, H, d)
            np.testing.assert_allclose(merged, ref[n][0], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- ring merge

@pytest.mark.parametrize("n_parts", [1, 2, 3])
def test_merge_of_key_subsets_equals_attention_over_their_union(n_parts):
    """Attention over a key set, split into disjoint subsets, equals the merge of the
    attention results over each subset (lse and O) -- the identity ring attention relies on."""
    L, d = 24, 8
    q, k, v = RNG.standard_normal((L, d)), RNG.standard_normal((L, d)), RNG.standard_normal((L, d))
    rows = np.arange(L)
    full_o, full_lse = oracle.head_forward(q, k, v, rows, Mask("none"), 1.0 / math.sqrt(d))
    cuts = np.array_split(np.random.default_rng(n_parts).permutation(L), n_parts)
    parts = []
    for keys in cuts:
        o_j, l_j = oracle.head_forward(q, k[keys], v[keys], rows, Mask("none"), 1.0 / math.sqrt(d))
        parts.append((o_j, l_j))
    o, lse = oracle.merge_partials([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o, full_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, full_lse, rtol=0, atol=1e-12)


def test_merge_with_an_empty_part_and_an_empty_row():
    o1, l1 = np.ones((2, 3)), np.array([0.5, -np.inf])
    o2, l2 = np.zeros((2, 3)), np.array([-np.inf, -np.inf])
    o, lse = oracle.merge_partials([o1, o2], [l1, l2])
    np.testing.assert_array_equal(o, [[1, 1, 1], [0, 0, 0]])
    assert lse[0] == 0.5 and np.isneginf(lse[1])
