"""GB300 (sm_103a) DeepSpeed-Ulysses attention block: Python binding of libulysses.so.

The functions named ``ulysses_*`` are the C ABI of ``include/ulysses.h`` one for one
(ctypes, plain integers for pointers and streams). The snake-case helpers below them take
torch CUDA tensors and only marshal pointers, shapes and the current stream into those
calls; every step of the computation runs in the library's CUDA kernels. PyTorch provides
device memory and streams only.

There is no fallback: if libulysses.so has not been built (``python -m
ulysses_sequence_gb300.build`` or ``__graft_entry__.build()``), loading raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libulysses.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_CUDA, ERR_DEVICE_TIMEOUT = range(6)
LAYOUT_TOKEN_SHARDED, LAYOUT_HEAD_SHARDED = 0, 1
MASK_NONE, MASK_CAUSAL, MASK_BLOCK_SPARSE = 0, 1, 2


class Shape(ctypes.Structure):
    """ulysses_shape_t; H_kv = 0 (the default) means H key/value heads."""
    _fields_ = [("B", ctypes.c_int), ("L", ctypes.c_int), ("H", ctypes.c_int), ("d_h", ctypes.c_int),
                ("P", ctypes.c_int), ("H_kv", ctypes.c_int)]


class MaskStruct(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("tile", ctypes.c_int), ("q_rowptr", ctypes.c_void_p),
                ("q_kcols", ctypes.c_void_p), ("k_colptr", ctypes.c_void_p), ("k_qrows", ctypes.c_void_p),
                ("nnz", ctypes.c_int)]


EXPORTS = ("ulysses_seq_to_head", "ulysses_head_to_seq", "ulysses_kv_seq_to_head", "ulysses_kv_head_to_seq_sum",
           "ulysses_a2a_pack", "ulysses_a2a_unpack",
           "ulysses_qkv_proj", "ulysses_out_proj", "ulysses_usp_workspace_size", "ulysses_usp_attn_fwd",
           "ulysses_usp_attn_bwd", "ulysses_attn_fwd", "ulysses_attn_bwd_workspace_size",
           "ulysses_attn_bwd", "ulysses_attn_bwd_noalloc", "ulysses_bsmask_build_window_global",
           "ulysses_get_device_status", "ulysses_selftest_timeout", "ulysses_status_string", "ulysses_shutdown")
BWD_NOALLOC_SCRATCH_BYTES = 96 * 1024 * 1024  # ULYSSES_BWD_NOALLOC_SCRATCH_BYTES

_lib = None


def load() -> ctypes.CDLL:
    """Load libulysses.so from this package directory (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m ulysses_sequence_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.ulysses_seq_to_head.argtypes = [Shape, vp, vp, vp]
    lib.ulysses_head_to_seq.argtypes = [Shape, vp, vp, vp]
    lib.ulysses_kv_seq_to_head.argtypes = [Shape, vp, vp, vp]
    lib.ulysses_a2a_pack.argtypes = [Shape, vp, vp, vp]
    lib.ulysses_a2a_unpack.argtypes = [Shape, vp, vp, vp]
    lib.ulysses_qkv_proj.argtypes = [Shape, i, vp, vp, vp, vp, vp, vp]
    lib.ulysses_usp_workspace_size.argtypes = [Shape, i]
    lib.ulysses_usp_workspace_size.restype = sz
    lib.ulysses_usp_attn_fwd.argtypes = [Shape, i, ctypes.POINTER(MaskStruct), f, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ulysses_usp_attn_bwd.argtypes = [Shape, i, ctypes.POINTER(MaskStruct), f, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                         vp, sz, vp]
    lib.ulysses_out_proj.argtypes = [Shape, i, vp, vp, vp, vp]
    lib.ulysses_kv_head_to_seq_sum.argtypes = [Shape, vp, vp, vp]
    lib.ulysses_attn_fwd.argtypes = [Shape, ctypes.POINTER(MaskStruct), f, i, vp, vp, vp, vp, vp, vp]
    lib.ulysses_attn_bwd_workspace_size.argtypes = [Shape]
    lib.ulysses_attn_bwd_workspace_size.restype = sz
    lib.ulysses_attn_bwd.argtypes = [Shape, ctypes.POINTER(MaskStruct), f, i, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     vp, sz, vp]
    lib.ulysses_attn_bwd_noalloc.argtypes = [Shape, ctypes.POINTER(MaskStruct), f, i, vp, vp, vp, vp, vp, vp, vp, vp,
                                             vp, vp]
    ip = ctypes.POINTER(ctypes.c_int32)
    lib.ulysses_bsmask_build_window_global.argtypes = [i, i, i, i, i, ip, ip, ip, ip, ctypes.POINTER(ctypes.c_int)]
    lib.ulysses_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.ulysses_selftest_timeout.argtypes = [vp]
    lib.ulysses_status_string.argtypes = [i]
    lib.ulysses_shutdown.argtypes = []
    lib.ulysses_status_string.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("ulysses_attn_bwd_workspace_size", "ulysses_usp_workspace_size", "ulysses_status_string"):
            getattr(lib, name).restype = i
    _lib = lib
    return lib


# ----------------------------------------------------------------------------- raw C ABI

def _mref(mask):
    return None if mask is None else ctypes.byref(mask)


def ulysses_seq_to_head(shape: Shape, inp: int, out: int, stream: int) -> int:
    return load().ulysses_seq_to_head(shape, inp, out, stream)


def ulysses_head_to_seq(shape: Shape, inp: int, out: int, stream: int) -> int:
    return load().ulysses_head_to_seq(shape, inp, out, stream)


def ulysses_kv_seq_to_head(shape: Shape, inp: int, out: int, stream: int) -> int:
    return load().ulysses_kv_seq_to_head(shape, inp, out, stream)


def ulysses_kv_head_to_seq_sum(shape: Shape, inp: int, out: int, stream: int) -> int:
    return load().ulysses_kv_head_to_seq_sum(shape, inp, out, stream)


def ulysses_a2a_pack(shape: Shape, inp: int, out: int, stream: int) -> int:
    return load().ulysses_a2a_pack(shape, inp, out, stream)


def ulysses_a2a_unpack(shape: Shape, inp: int, out: int, stream: int) -> int:
    return load().ulysses_a2a_unpack(shape, inp, out, stream)


def ulysses_qkv_proj(shape: Shape, hidden: int, x: int, w_qkv: int, q: int, k: int, v: int, stream: int) -> int:
    return load().ulysses_qkv_proj(shape, hidden, x, w_qkv, q, k, v, stream)


def ulysses_out_proj(shape: Shape, hidden: int, o: int, w_o: int, y: int, stream: int) -> int:
    return load().ulysses_out_proj(shape, hidden, o, w_o, y, stream)


def ulysses_usp_workspace_size(shape: Shape, P_ring: int) -> int:
    return load().ulysses_usp_workspace_size(shape, P_ring)


def ulysses_usp_attn_fwd(shape: Shape, P_ring: int, mask: MaskStruct, softmax_scale: float, q: int, k: int, v: int,
                         o: int, lse: int, workspace: int, workspace_bytes: int, stream: int) -> int:
    return load().ulysses_usp_attn_fwd(shape, P_ring, _mref(mask), softmax_scale, q, k, v, o, lse, workspace,
                                       workspace_bytes, stream)


def ulysses_usp_attn_bwd(shape: Shape, P_ring: int, mask: MaskStruct, softmax_scale: float, q: int, k: int, v: int,
                         o: int, lse: int, dO: int, dq: int, dk: int, dv: int, workspace: int, workspace_bytes: int,
                         stream: int) -> int:
    return load().ulysses_usp_attn_bwd(shape, P_ring, _mref(mask), softmax_scale, q, k, v, o, lse, dO, dq, dk, dv,
                                       workspace, workspace_bytes, stream)


def ulysses_attn_fwd(shape: Shape, mask: MaskStruct, softmax_scale: float, io_layout: int, q: int, k: int, v: int,
                     o: int, lse: int, stream: int) -> int:
    return load().ulysses_attn_fwd(shape, _mref(mask), softmax_scale, io_layout, q, k, v, o, lse, stream)


def ulysses_attn_bwd_workspace_size(shape: Shape) -> int:
    return load().ulysses_attn_bwd_workspace_size(shape)


def ulysses_attn_bwd(shape: Shape, mask: MaskStruct, softmax_scale: float, io_layout: int, q: int, k: int, v: int,
                     o: int, lse: int, dO: int, dq: int, dk: int, dv: int, workspace: int, workspace_bytes: int,
                     stream: int) -> int:
    return load().ulysses_attn_bwd(shape, _mref(mask), softmax_scale, io_layout, q, k, v, o, lse, dO, dq, dk,
                                   dv, workspace, workspace_bytes, stream)


def ulysses_attn_bwd_noalloc(shape: Shape, mask: MaskStruct, softmax_scale: float, io_layout: int, q: int, k: int,
                             v: int, o: int, lse: int, dO: int, dq: int, dk: int, dv: int, stream: int) -> int:
    """ulysses_attn_bwd with the workspace in the library's fixed device array (for callers
    that cannot allocate device memory; see include/ulysses.h)."""
    return load().ulysses_attn_bwd_noalloc(shape, _mref(mask), softmax_scale, io_layout, q, k, v, o, lse, dO, dq, dk,
                                           dv, stream)


def ulysses_bsmask_build_window_global(L: int, tile: int, window_before: int, window_after: int,
                                       global_stride: int):
    """Returns host lists (rowptr, kcols, colptr, qrows) built by the library."""
    lib = load()
    n = (L + tile - 1) // tile
    nnz = ctypes.c_int(0)
    rp = (ctypes.c_int32 * (n + 1))()
    cp = (ctypes.c_int32 * (n + 1))()
    lib.ulysses_bsmask_build_window_global(L, tile, window_before, window_after, global_stride, rp, None, cp, None,
                                           ctypes.byref(nnz))
    cap = nnz.value
    kc = (ctypes.c_int32 * max(cap, 1))()
    qr = (ctypes.c_int32 * max(cap, 1))()
    nnz = ctypes.c_int(cap)
    rc = lib.ulysses_bsmask_build_window_global(L, tile, window_before, window_after, global_stride, rp, kc, cp, qr,
                                                ctypes.byref(nnz))
    check(rc, "ulysses_bsmask_build_window_global")
    return list(rp), list(kc)[:cap], list(cp), list(qr)[:cap]


def ulysses_get_device_status(stream: int) -> Tuple[int, int]:
    detail = ctypes.c_uint32(0)
    rc = load().ulysses_get_device_status(stream, ctypes.byref(detail))
    return rc, detail.value


def ulysses_selftest_timeout(stream: int) -> int:
    return load().ulysses_selftest_timeout(stream)


def ulysses_status_string(status: int) -> str:
    return load().ulysses_status_string(status).decode()


def ulysses_shutdown() -> int:
    return load().ulysses_shutdown()


class UlyssesError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {ulysses_status_string(status)}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != OK:
        raise UlyssesError(status, where)


# ----------------------------------------------------------------------------- torch helpers

def _stream(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def token_shape(x, P: int) -> Shape:
    """Shape of a token-sharded tensor [P][B][Lp][H][d]."""
    P_, B, Lp, H, d = x.shape
    assert P_ == P, "leading dimension must be the shard count P"
    return Shape(B, Lp * P, H, d, P)


def head_shape(y, P: int) -> Shape:
    """Shape of a head-sharded tensor [P][B][L][Hp][d]."""
    P_, B, L, Hp, d = y.shape
    assert P_ == P, "leading dimension must be the shard count P"
    return Shape(B, L, Hp * P, d, P)


class Mask:
    """An attention mask for the C ABI; for block-sparse masks it owns the device tile lists."""

    def __init__(self, kind: int, tile: int = 128, lists=None):
        self.kind, self.tile, self.lists = kind, tile, lists
        self.struct = MaskStruct(kind, tile, None, None, None, None, 0)
        if lists is not None:
            rp, kc, cp, qr = lists
            self.struct = MaskStruct(kind, tile, rp.data_ptr(), kc.data_ptr(), cp.data_ptr(), qr.data_ptr(),
                                     int(kc.numel()))

    @staticmethod
    def causal() -> "Mask":
        return Mask(MASK_CAUSAL)

    @staticmethod
    def none() -> "Mask":
        return Mask(MASK_NONE)

    @staticmethod
    def window_global(L: int, tile: int = 128, window_before: int = 4, window_after: int = 3,
                      global_stride: int = 16, device="cuda") -> "Mask":
        import torch
        rp, kc, cp, qr = ulysses_bsmask_build_window_global(L, tile, window_before, window_after, global_stride)
        t = [torch.tensor(x if x else [0], dtype=torch.int32, device=device) for x in (rp, kc, cp, qr)]
        return Mask(MASK_BLOCK_SPARSE, tile, t)

    @staticmethod
    def from_tile_lists(rowptr, kcols, colptr, qrows, tile: int = 128, device="cuda") -> "Mask":
        import torch
        t = [torch.as_tensor(x, dtype=torch.int32).to(device) for x in (rowptr, kcols, colptr, qrows)]
        return Mask(MASK_BLOCK_SPARSE, tile, t)


def seq_to_head(x, P: int, out=None, stream=None):
    """[P][B][Lp][H][d] -> [P][B][L][Hp][d] on the GPU (16-bit elements)."""
    import torch
    Pn, B, Lp, H, d = x.shape
    if out is None:
        out = torch.empty((P, B, Lp * P, H // P, d), dtype=x.dtype, device=x.device)
    check(ulysses_seq_to_head(token_shape(x, P), x.data_ptr(), out.data_ptr(), _stream(stream)), "seq_to_head")
    return out


def head_to_seq(y, P: int, out=None, stream=None):
    """[P][B][L][Hp][d] -> [P][B][Lp][H][d] on the GPU (16-bit elements)."""
    import torch
    Pn, B, L, Hp, d = y.shape
    if out is None:
        out = torch.empty((P, B, L // P, Hp * P, d), dtype=y.dtype, device=y.device)
    check(ulysses_head_to_seq(head_shape(y, P), y.data_ptr(), out.data_ptr(), _stream(stream)), "head_to_seq")
    return out


def a2a_pack(x, P: int, out=None, stream=None):
    """One rank's token shard [B][Lp][H][d] -> [P][B][Lp][H/P][d]: chunk g holds head group g,
    ready for an all-to-all whose rank g owns that group."""
    import torch
    B, Lp, H, d = x.shape
    if out is None:
        out = torch.empty((P, B, Lp, H // P, d), dtype=x.dtype, device=x.device)
    check(ulysses_a2a_pack(Shape(B, Lp * P, H, d, P), x.data_ptr(), out.data_ptr(), _stream(stream)), "a2a_pack")
    return out


def a2a_unpack(y, P: int, out=None, stream=None):
    """Inverse of a2a_pack: [P][B][Lp][H/P][d] (chunk g from head group g) -> [B][Lp][H][d]."""
    import torch
    Pn, B, Lp, Hg, d = y.shape
    if out is None:
        out = torch.empty((B, Lp, Hg * P, d), dtype=y.dtype, device=y.device)
    check(ulysses_a2a_unpack(Shape(B, Lp * P, Hg * P, d, P), y.data_ptr(), out.data_ptr(), _stream(stream)),
          "a2a_unpack")
    return out


def kv_heads_per_group(H_kv: int, P: int) -> int:
    """Key/value heads each head group holds: H_kv / P, or 1 when P > H_kv (a copy)."""
    return H_kv // P if H_kv % P == 0 else 1


def kv_seq_to_head(x, P: int, out=None, stream=None):
    """K/V [P][B][Lp][H_kv][d] -> [P][B][L][Hkvp][d] (heads replicated when P > H_kv)."""
    import torch
    Pn, B, Lp, Hkv, d = x.shape
    if out is None:
        out = torch.empty((P, B, Lp * P, kv_heads_per_group(Hkv, P), d), dtype=x.dtype, device=x.device)
    shape = Shape(B, Lp * P, Hkv, d, P, Hkv)
    check(ulysses_kv_seq_to_head(shape, x.data_ptr(), out.data_ptr(), _stream(stream)), "kv_seq_to_head")
    return out


def kv_head_to_seq_sum(y, P: int, H_kv: int, out=None, stream=None):
    """Adjoint of kv_seq_to_head on bf16 gradients: [P][B][L][Hkvp][d] -> [P][B][Lp][H_kv][d],
    the copies of each key/value head summed in fp32."""
    import torch
    Pn, B, L, Hkvp, d = y.shape
    if out is None:
        out = torch.empty((P, B, L // P, H_kv, d), dtype=y.dtype, device=y.device)
    shape = Shape(B, L, H_kv, d, P, H_kv)
    check(ulysses_kv_head_to_seq_sum(shape, y.data_ptr(), out.data_ptr(), _stream(stream)), "kv_head_to_seq_sum")
    return out


def _shape_of(x, P: int, layout: int, k=None, kv_heads: int = 0) -> Shape:
    """Shape of query-side tensor x; H_kv from kv_heads, else from k's head dimension (in the
    head layout k's Hkvp * P, which needs kv_heads when key/value heads are replicated)."""
    s = token_shape(x, P) if layout == LAYOUT_TOKEN_SHARDED else head_shape(x, P)
    if kv_heads:
        s.H_kv = kv_heads
    elif k is not None:
        s.H_kv = k.shape[3] if layout == LAYOUT_TOKEN_SHARDED else k.shape[3] * P
    return s


def qkv_proj(x, w_qkv, P: int, H: int, H_kv: int, d: int, q=None, k=None, v=None, stream=None):
    """QKV projection of token-sharded hidden states x [P][B][Lp][hidden] with w_qkv
    [(H + 2 H_kv) d][hidden]; returns q [P][B][Lp][H][d], k, v [P][B][Lp][H_kv][d]."""
    import torch
    Pn, B, Lp, hidden = x.shape
    shape = Shape(B, Lp * P, H, d, P, H_kv)
    q = torch.empty((P, B, Lp, H, d), dtype=x.dtype, device=x.device) if q is None else q
    k = torch.empty((P, B, Lp, H_kv, d), dtype=x.dtype, device=x.device) if k is None else k
    v = torch.empty((P, B, Lp, H_kv, d), dtype=x.dtype, device=x.device) if v is None else v
    check(ulysses_qkv_proj(shape, hidden, x.data_ptr(), w_qkv.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                           _stream(stream)), "qkv_proj")
    return q, k, v


def out_proj(o, w_o, P: int, y=None, stream=None):
    """Output projection of token-sharded o [P][B][Lp][H][d] with w_o [hidden][H d]."""
    import torch
    Pn, B, Lp, H, d = o.shape
    hidden = w_o.shape[0]
    y = torch.empty((P, B, Lp, hidden), dtype=o.dtype, device=o.device) if y is None else y
    check(ulysses_out_proj(Shape(B, Lp * P, H, d, P), hidden, o.data_ptr(), w_o.data_ptr(), y.data_ptr(),
                           _stream(stream)), "out_proj")
    return y


def usp_workspace(q, P: int, P_ring: int, kv_heads: int = 0):
    import torch
    n = ulysses_usp_workspace_size(_shape_of(q, P, LAYOUT_TOKEN_SHARDED, kv_heads=kv_heads), P_ring)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def usp_attn_fwd(q, k, v, P: int, P_ring: int, mask: Mask, scale: float = 0.0, o=None, lse=None, workspace=None,
                 stream=None):
    """Ulysses-ring hybrid forward on token-sharded q [P][B][Lp][H][d] (k, v with H_kv heads).
    Returns (o, lse[P_ring][P/P_ring][B][H/(P/P_ring)][L/P_ring] fp32)."""
    import torch
    shape = _shape_of(q, P, LAYOUT_TOKEN_SHARDED, k)
    o = torch.empty_like(q) if o is None else o
    if lse is None:
        # sized for a valid split; the library itself rejects an invalid one
        valid = P_ring > 0 and P % P_ring == 0 and shape.H % (P // P_ring) == 0
        Pu = P // P_ring if valid else 1
        lse = torch.empty((P_ring, Pu, shape.B, shape.H // Pu, shape.L // P_ring) if valid else (1,),
                          dtype=torch.float32, device=q.device)
    ws = usp_workspace(q, P, P_ring, shape.H_kv) if workspace is None else workspace
    check(ulysses_usp_attn_fwd(shape, P_ring, mask.struct, scale, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                               o.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)), "usp_attn_fwd")
    return o, lse


def usp_attn_bwd(q, k, v, o, lse, do, P: int, P_ring: int, mask: Mask, scale: float = 0.0, dq=None, dk=None, dv=None,
                 workspace=None, stream=None):
    """Ulysses-ring hybrid backward. Returns (dq, dk, dv)."""
    import torch
    shape = _shape_of(q, P, LAYOUT_TOKEN_SHARDED, k)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = usp_workspace(q, P, P_ring, shape.H_kv) if workspace is None else workspace
    check(ulysses_usp_attn_bwd(shape, P_ring, mask.struct, scale, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                               o.data_ptr(), lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                               ws.data_ptr(), ws.numel(), _stream(stream)), "usp_attn_bwd")
    return dq, dk, dv


def attn_fwd(q, k, v, P: int, mask: Mask, layout: int = LAYOUT_TOKEN_SHARDED, scale: float = 0.0, o=None,
             lse=None, stream=None, kv_heads: int = 0):
    """Attention forward through ulysses_attn_fwd. Returns (o, lse[P][B][Hp][L] fp32).
    k, v may have fewer heads than q (grouped key/value heads; kv_heads names H_kv when the
    head layout replicates them)."""
    import torch
    shape = _shape_of(q, P, layout, k, kv_heads)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((P, shape.B, shape.H // P, shape.L), dtype=torch.float32, device=q.device)
    check(ulysses_attn_fwd(shape, mask.struct, scale, layout, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), _stream(stream)), "attn_fwd")
    return o, lse


def bwd_workspace(q, P: int, layout: int = LAYOUT_TOKEN_SHARDED):
    import torch
    n = ulysses_attn_bwd_workspace_size(_shape_of(q, P, layout))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def attn_bwd(q, k, v, o, lse, do, P: int, mask: Mask, layout: int = LAYOUT_TOKEN_SHARDED, scale: float = 0.0,
             dq=None, dk=None, dv=None, workspace=None, stream=None, kv_heads: int = 0):
    """Attention backward through ulysses_attn_bwd. Returns (dq, dk, dv); dk, dv are shaped
    like k, v (with replicated key/value heads in the head layout: one part per copy)."""
    import torch
    shape = _shape_of(q, P, layout, k, kv_heads)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = bwd_workspace(q, P, layout) if workspace is None else workspace
    check(ulysses_attn_bwd(shape, mask.struct, scale, layout, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                           ws.numel(), _stream(stream)), "attn_bwd")
    return dq, dk, dv


def shutdown() -> None:
    """Releases the calling thread's side streams and cached tensor maps (made again on demand)."""
    check(ulysses_shutdown(), "shutdown")


def device_status(stream=None) -> Tuple[int, int]:
    """Synchronises the stream and reads/clears the device error word: (status, raw word)."""
    return ulysses_get_device_status(_stream(stream))
