"""CPU checks of the C-ABI library: it loads, exports every function include/ulysses.h
declares, rejects bad arguments before touching the GPU, and its host-side block-sparse
tile-list builder agrees with the oracle's pattern. No compute call is made here."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import ulysses_sequence_gb300 as U

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from ulysses_sequence_gb300 import build
    build.build()
    return U.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ulysses.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ulysses_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("ulysses_seq_to_head", "ulysses_head_to_seq", "ulysses_attn_fwd", "ulysses_attn_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(U.EXPORTS) <= set(declared_functions())


def test_shutdown_with_no_thread_state_is_ok(lib):
    # a thread that made no side stream releases only its host-side map cache: no CUDA call,
    # so this holds without a GPU
    assert U.ulysses_shutdown() == U.OK
    U.shutdown()


def test_status_strings(lib):
    assert U.ulysses_status_string(U.OK) == "ULYSSES_OK"
    assert U.ulysses_status_string(U.ERR_DEVICE_TIMEOUT) == "ULYSSES_ERR_DEVICE_TIMEOUT"
    assert U.ulysses_status_string(99) == "ULYSSES_ERR_UNKNOWN"


@pytest.mark.parametrize("shape", [(1, 256, 8, 64, 3), (1, 250, 8, 64, 4), (0, 256, 0, 64, 4), (1, 256, 8, 64, 0),
                                   (-1, 256, 8, 64, 4)])
def test_relayout_rejects_bad_shapes(lib, shape):
    s = U.Shape(*shape)
    assert U.ulysses_seq_to_head(s, 16, 32, 0) == U.ERR_INVALID_ARG
    assert U.ulysses_head_to_seq(s, 16, 32, 0) == U.ERR_INVALID_ARG


def test_relayout_argument_checks(lib):
    s = U.Shape(1, 256, 8, 64, 4)
    assert U.ulysses_seq_to_head(s, 0, 64, 0) == U.ERR_INVALID_ARG        # null input
    assert U.ulysses_seq_to_head(s, 64, 64, 0) == U.ERR_INVALID_ARG       # in place
    assert U.ulysses_seq_to_head(s, 65, 128, 0) == U.ERR_MISALIGNED       # odd address
    assert U.ulysses_seq_to_head(U.Shape(0, 256, 8, 64, 4), 0, 0, 0) == U.OK   # empty: nothing to do
    assert U.ulysses_seq_to_head(U.Shape(2, 0, 8, 64, 4), 0, 0, 0) == U.OK


def fwd(shape, mask=None, layout=U.LAYOUT_TOKEN_SHARDED, ptrs=(256, 512, 768, 1024, 1280)):
    m = mask if mask is not None else U.MaskStruct(U.MASK_CAUSAL, 128, None, None, None, None, 0)
    return U.ulysses_attn_fwd(U.Shape(*shape), m, 0.0, layout, *ptrs, 0)


def test_attn_fwd_argument_checks(lib):
    assert fwd((1, 256, 8, 96, 4)) == U.ERR_UNSUPPORTED                   # d_h not 64/128
    assert fwd((1, 256, 6, 64, 4)) == U.ERR_INVALID_ARG                   # H % P
    assert fwd((1, 260, 8, 64, 4)) == U.ERR_UNSUPPORTED                   # token layout needs Lp % 8 == 0
    assert fwd((1, 256, 8, 64, 4), layout=7) == U.ERR_INVALID_ARG
    assert fwd((1, 256, 8, 64, 4), ptrs=(256, 512, 768, 1032, 1280)) == U.ERR_MISALIGNED
    assert fwd((1, 256, 8, 64, 4), ptrs=(256, 512, 768, 256, 1280)) == U.ERR_INVALID_ARG   # o aliases q
    assert fwd((1, 256, 8, 64, 4), ptrs=(256, 0, 768, 1024, 1280)) == U.ERR_INVALID_ARG
    bad = U.MaskStruct(U.MASK_BLOCK_SPARSE, 64, 16, 16, 16, 16, 1)
    assert fwd((1, 256, 8, 64, 4), mask=bad) == U.ERR_UNSUPPORTED        # tile must be 128
    bad = U.MaskStruct(U.MASK_BLOCK_SPARSE, 128, None, 16, 16, 16, 1)
    assert fwd((1, 256, 8, 64, 4), mask=bad) == U.ERR_INVALID_ARG
    bad = U.MaskStruct(9, 128, None, None, None, None, 0)
    assert fwd((1, 256, 8, 64, 4), mask=bad) == U.ERR_INVALID_ARG
    assert fwd((0, 256, 8, 64, 4), ptrs=(0, 0, 0, 0, 0)) == U.OK          # empty batch
    assert U.ulysses_attn_fwd(U.Shape(1, 256, 8, 64, 4), None, 0.0, 0, 256, 512, 768, 1024, 1280, 0) \
        == U.ERR_INVALID_ARG


def test_attn_bwd_argument_checks(lib):
    s = U.Shape(1, 256, 8, 64, 4)
    m = U.MaskStruct(U.MASK_CAUSAL, 128, None, None, None, None, 0)
    need = U.ulysses_attn_bwd_workspace_size(s)
    # fp32 dQ accumulator + Delta + the block-sparse schedule (four ints per key tile, 256-aligned)
    assert need == 256 * 8 * 64 * 4 + 256 * 8 * 4 + 256
    p = [256 * (i + 1) for i in range(9)]
    ws = 1 << 20
    assert U.ulysses_attn_bwd(s, m, 0.0, 0, *p, ws, need - 1, 0) == U.ERR_INVALID_ARG      # workspace too small
    assert U.ulysses_attn_bwd(s, m, 0.0, 0, *p[:6], p[0], p[7], p[8], ws, need, 0) == U.ERR_INVALID_ARG  # dq aliases q
    assert U.ulysses_attn_bwd(s, m, 0.0, 0, *p, ws + 16, need, 0) == U.ERR_MISALIGNED      # workspace 256-aligned
    assert U.ulysses_attn_bwd(U.Shape(1, 256, 8, 32, 4), m, 0.0, 0, *p, ws, need, 0) == U.ERR_UNSUPPORTED
    assert U.ulysses_attn_bwd_workspace_size(U.Shape(1, 256, 6, 64, 4)) == 0


@pytest.mark.parametrize("L,wb,wa,gs", [(65536, 4, 3, 16), (2048, 4, 3, 16), (1000, 1, 0, 3), (896, 2, 2, 5)])
def test_block_sparse_lists_match_oracle_pattern(lib, L, wb, wa, gs):
    rp, kc, cp, qr = U.ulysses_bsmask_build_window_global(L, 128, wb, wa, gs)
    n = -(-L // 128)
    want = oracle.window_global_tiles(n, wb, wa, gs)
    got = np.zeros((n, n), dtype=bool)
    for qt in range(n):
        cols = kc[rp[qt]:rp[qt + 1]]
        assert cols == sorted(cols)
        got[qt, cols] = True
    assert np.array_equal(got, want)
    got_c = np.zeros((n, n), dtype=bool)
    for kt in range(n):
        rows = qr[cp[kt]:cp[kt + 1]]
        assert rows == sorted(rows)
        got_c[rows, kt] = True
    assert np.array_equal(got_c, want)


def test_block_sparse_builder_capacity(lib):
    n = ctypes.c_int(3)
    rp = (ctypes.c_int32 * 17)()
    cp = (ctypes.c_int32 * 17)()
    kc = (ctypes.c_int32 * 3)()
    qr = (ctypes.c_int32 * 3)()
    rc = lib.ulysses_bsmask_build_window_global(2048, 128, 4, 3, 16, rp, kc, cp, qr, ctypes.byref(n))
    assert rc == U.ERR_INVALID_ARG and n.value == 123


def test_grouped_kv_head_counts_are_validated(lib):
    """H_kv must divide H, and either H_kv % P == 0 or P % H_kv == 0; rejected before any launch."""
    m = U.MaskStruct(U.MASK_CAUSAL, 128, None, None, None, None, 0)
    p = [256 * (i + 1) for i in range(5)]
    bad_group = U.Shape(1, 256, 8, 64, 4, 3)    # H % H_kv != 0
    bad_cut = U.Shape(1, 256, 12, 64, 4, 6)     # neither H_kv % P nor P % H_kv is 0
    for s in (bad_group, bad_cut):
        assert U.ulysses_attn_bwd_workspace_size(s) == 0
        assert U.ulysses_attn_fwd(s, m, 0.0, 0, *p, 0) == U.ERR_INVALID_ARG
        assert U.ulysses_kv_seq_to_head(s, 256, 512, 0) == U.ERR_INVALID_ARG
        assert U.ulysses_kv_head_to_seq_sum(s, 256, 512, 0) == U.ERR_INVALID_ARG
    # accepted: whole key/value heads per group, and copies
    for hkv in (8, 4, 2, 1):
        assert U.ulysses_attn_bwd_workspace_size(U.Shape(1, 256, 8, 64, 4, hkv)) > 0
    assert U.ulysses_kv_seq_to_head(U.Shape(0, 256, 8, 64, 4, 2), 0, 0, 0) == U.OK   # empty batch


def test_projection_argument_checks(lib):
    """The projections validate sizes, pointers and alignment on the host, before any launch."""
    s = U.Shape(1, 256, 8, 64, 4)
    p = [256 * (i + 1) for i in range(5)]
    assert U.ulysses_qkv_proj(s, 0, *p, 0) == U.ERR_INVALID_ARG                      # hidden 0
    assert U.ulysses_qkv_proj(s, 48, *p, 0) == U.ERR_UNSUPPORTED                     # hidden % 32
    assert U.ulysses_qkv_proj(U.Shape(1, 256, 6, 64, 4), 512, *p, 0) == U.ERR_INVALID_ARG  # H % P
    assert U.ulysses_qkv_proj(s, 512, 0, *p[1:], 0) == U.ERR_INVALID_ARG             # null x
    assert U.ulysses_qkv_proj(s, 512, p[0], p[1], p[0], p[3], p[4], 0) == U.ERR_INVALID_ARG  # q aliases x
    assert U.ulysses_qkv_proj(s, 512, p[0], p[1], p[2], p[2], p[4], 0) == U.ERR_INVALID_ARG  # q == k
    assert U.ulysses_qkv_proj(s, 512, p[0] + 8, *p[1:], 0) == U.ERR_MISALIGNED       # x not 16-aligned
    assert U.ulysses_qkv_proj(U.Shape(0, 256, 8, 64, 4), 512, 0, 0, 0, 0, 0, 0) == U.OK  # empty batch
    assert U.ulysses_out_proj(s, 512, p[0], p[1], p[0], 0) == U.ERR_INVALID_ARG      # y aliases o
    assert U.ulysses_out_proj(s, 512, p[0], p[1], p[2] + 2, 0) == U.ERR_MISALIGNED
    assert U.ulysses_out_proj(s, 40, *p[:3], 0) == U.ERR_UNSUPPORTED


def test_usp_argument_checks(lib):
    """The Ulysses-ring hybrid validates the split P = P_u * P_ring on the host: P_ring must
    divide P, each ring block must be a valid token-sharded attention shape (P_u | H, Lp % 8),
    block-sparse masks are not supported, the workspace is sized and 256-byte aligned."""
    m = U.MaskStruct(U.MASK_CAUSAL, 128, None, None, None, None, 0)
    s = U.Shape(1, 512, 4, 128, 8)                 # P = 8 > H = 4: only valid with P_ring >= 2
    need = U.ulysses_usp_workspace_size(s, 2)
    assert need > 0 and need % 256 == 0
    assert U.ulysses_usp_workspace_size(s, 1) == 0                               # P_u = 8 does not divide H
    assert U.ulysses_usp_workspace_size(s, 3) == 0                               # 3 does not divide 8
    assert U.ulysses_usp_workspace_size(s, 0) == 0
    assert U.ulysses_usp_workspace_size(s, 16) == 0                              # P_ring > P
    assert U.ulysses_usp_workspace_size(s, 65) == 0                              # beyond the ring limit
    assert U.ulysses_usp_workspace_size(U.Shape(1, 512, 4, 96, 8), 2) == 0       # d_h 96
    p = [256 * (i + 1) for i in range(10)]
    ws = 1 << 20
    assert U.ulysses_usp_attn_fwd(s, 2, m, 0.0, *p[:5], ws, need - 256, 0) == U.ERR_INVALID_ARG
    assert U.ulysses_usp_attn_fwd(s, 2, m, 0.0, *p[:5], ws + 64, need, 0) == U.ERR_MISALIGNED
    assert U.ulysses_usp_attn_fwd(s, 2, m, 0.0, p[0], p[1], p[2], p[0], p[4], ws, need, 0) == U.ERR_INVALID_ARG
    assert U.ulysses_usp_attn_fwd(s, 2, m, 0.0, p[0] + 8, *p[1:5], ws, need, 0) == U.ERR_MISALIGNED
    assert U.ulysses_usp_attn_fwd(s, 1, m, 0.0, *p[:5], ws, need, 0) == U.ERR_INVALID_ARG
    sparse = U.MaskStruct(U.MASK_BLOCK_SPARSE, 128, 16, 16, 16, 16, 1)
    assert U.ulysses_usp_attn_fwd(s, 2, sparse, 0.0, *p[:5], ws, need, 0) == U.ERR_UNSUPPORTED
    assert U.ulysses_usp_attn_fwd(U.Shape(0, 512, 4, 128, 8), 2, m, 0.0, 0, 0, 0, 0, 0, 0, 0, 0) == U.OK
    assert U.ulysses_usp_attn_bwd(s, 2, m, 0.0, *p[:9], ws, need - 256, 0) == U.ERR_INVALID_ARG
    assert U.ulysses_usp_attn_bwd(s, 2, m, 0.0, *p[:6], p[0], p[7], p[8], ws, need, 0) == U.ERR_INVALID_ARG  # dq aliases q
    assert U.ulysses_usp_attn_bwd(s, 2, m, 0.0, *p[:8], p[7], ws, need, 0) == U.ERR_INVALID_ARG   # dk == dv
