"""CPU oracle for the DeepSpeed-Ulysses attention block -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package. It shares no code with the CUDA path (``ulysses_sequence_gb300``)
and never imports it.

What it computes, and where the pages define it:

* ``seq_to_head`` / ``head_to_seq`` -- the two all-to-alls as explicit index loops in C
  (``ulysses_oracle.c``): paper summary section 3.4.1 and the pinyu.ai page "Use the
  other independent axis" (contiguous head groups, token blocks joined in sender order).
* ``attention_fwd`` / ``attention_bwd`` -- exact attention per head over the full
  sequence, O_h = softmax(Q_h K_h^T / sqrt(d_h) + mask) V_h (paper summary section
  3.4.1, "The challenge at the attention boundary"; pinyu.ai page, "The layout that saves
  memory breaks at attention"), in fp64 on the exact bf16 input values, plus its analytic
  gradient. The pages never write the backward pass; the gradient used here is the
  textbook derivative of softmax attention:
      P_ij = exp(S_ij - LSE_i) on permitted (i, j), 0 elsewhere
      Delta_i = sum_e dO_ie O_ie
      dV_j = sum_i P_ij dO_i,   dP_ij = dO_i . V_j,   dS_ij = P_ij (dP_ij - Delta_i)
      dQ_i = scale sum_j dS_ij K_j,   dK_j = scale sum_i dS_ij Q_i
  Matrix products use numpy's fp64 matmul as a library step; rows are independent, so
  the sampled mode evaluates the same formulas on a subset of rows.

* ``qkv_projection`` / ``out_projection`` -- the steps on either side of the path: each
  rank projects its own token shard to Q, K, V before the first all-to-all, and projects
  the returned O after the second (paper summary section 3.2, "Big-Picture Architecture",
  and section 3.4.1, "Before attention"; pinyu.ai page, "One attention block, end to
  end"). Row r of a token shard is projected alone, so the projections are row-wise
  products with the weight matrices (y = x W^T, numpy's fp64 matmul as a library step)
  and keep the token-sharded layout.

Readings where the pages are silent (the plainest one the rest of the pages supports):
masked positions are excluded (-inf), a row with no permitted key has O = 0, LSE = -inf and
zero gradients; the log-sum-exp is natural-log of the scaled scores, stored [P][B][H/P][L].
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Iterator, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ulysses_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C part of the oracle with gcc (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64 = ctypes.c_int64
            for fn in ("oracle_seq_to_head", "oracle_head_to_seq"):
                f = getattr(lib, fn)
                f.restype = ctypes.c_int
                f.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_kv_seq_to_head.restype = ctypes.c_int
            lib.oracle_kv_seq_to_head.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_kv_head_to_seq_sum.restype = ctypes.c_int
            lib.oracle_kv_head_to_seq_sum.argtypes = [i64, i64, i64, i64, i64, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_bf16_to_f64.restype = None
            lib.oracle_bf16_to_f64.argtypes = [i64, ctypes.c_void_p, ctypes.c_void_p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# --------------------------------------------------------------------------- relayouts

def seq_to_head(x: np.ndarray, P: int) -> np.ndarray:
    """Token-sharded [P][B][Lp][H][d] -> head-sharded [P][B][L][Hp][d] (any element type)."""
    x = np.ascontiguousarray(x)
    P_, B, Lp, H, d = x.shape
    assert P_ == P and H % P == 0
    L = Lp * P
    y = np.empty((P, B, L, H // P, d), dtype=x.dtype)
    rc = _load().oracle_seq_to_head(P, B, L, H, d, x.itemsize, _ptr(x), _ptr(y))
    if rc != 0:
        raise ValueError("oracle_seq_to_head rejected the shape")
    return y


def head_to_seq(y: np.ndarray, P: int) -> np.ndarray:
    """Head-sharded [P][B][L][Hp][d] -> token-sharded [P][B][Lp][H][d] (any element type)."""
    y = np.ascontiguousarray(y)
    P_, B, L, Hp, d = y.shape
    assert P_ == P and L % P == 0
    H = Hp * P
    z = np.empty((P, B, L // P, H, d), dtype=y.dtype)
    rc = _load().oracle_head_to_seq(P, B, L, H, d, y.itemsize, _ptr(y), _ptr(z))
    if rc != 0:
        raise ValueError("oracle_head_to_seq rejected the shape")
    return z


def kv_heads_per_rank(Hkv: int, P: int) -> int:
    """K/V heads each head group holds: Hkv/P, or 1 when P > Hkv (heads replicated)."""
    if Hkv % P == 0:
        return Hkv // P
    if P % Hkv == 0:
        return 1
    raise ValueError("need Hkv % P == 0 or P % Hkv == 0")


def kv_seq_to_head(x: np.ndarray, P: int) -> np.ndarray:
    """Token-sharded K/V [P][B][Lp][Hkv][d] -> head-sharded [P][B][L][Hkvp][d] (C loops)."""
    x = np.ascontiguousarray(x)
    P_, B, Lp, Hkv, d = x.shape
    assert P_ == P
    Hkvp = kv_heads_per_rank(Hkv, P)
    y = np.empty((P, B, Lp * P, Hkvp, d), dtype=x.dtype)
    if _load().oracle_kv_seq_to_head(P, B, Lp * P, Hkv, d, x.itemsize, _ptr(x), _ptr(y)) != 0:
        raise ValueError("oracle_kv_seq_to_head rejected the shape")
    return y


def kv_head_to_seq_sum(y: np.ndarray, P: int, Hkv: int) -> np.ndarray:
    """Adjoint of kv_seq_to_head on fp64 gradients: sums the replicas of each K/V head."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    P_, B, L, Hkvp, d = y.shape
    assert P_ == P and Hkvp == kv_heads_per_rank(Hkv, P)
    z = np.empty((P, B, L // P, Hkv, d))
    if _load().oracle_kv_head_to_seq_sum(P, B, L, Hkv, d, _ptr(y), _ptr(z)) != 0:
        raise ValueError("oracle_kv_head_to_seq_sum rejected the shape")
    return z


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_bf16_to_f64(bits.size, _ptr(bits), _ptr(out))
    return out


# --------------------------------------------------------------------------- masks

class Mask:
    """Which (query i, key j) pairs are permitted, with global token indices.

    kind "none": every pair.  kind "causal": j <= i (a token sees itself and the past).
    kind "tiles": whole tile x tile blocks, permitted iff tiles[i // tile, j // tile].
    """

    def __init__(self, kind: str, tile: int = 0, tiles: Optional[np.ndarray] = None):
        assert kind in ("none", "causal", "tiles")
        self.kind, self.tile, self.tiles = kind, tile, tiles

    def rows(self, rows: np.ndarray, L: int) -> np.ndarray:
        """Bool [len(rows), L] of permitted keys for the given query rows."""
        j = np.arange(L)[None, :]
        i = np.asarray(rows)[:, None]
        if self.kind == "none":
            return np.ones((len(rows), L), dtype=bool)
        if self.kind == "causal":
            return j <= i
        return self.tiles[i // self.tile, j // self.tile]


def window_global_tiles(n_tiles: int, window_before: int, window_after: int,
                        global_stride: int) -> np.ndarray:
    """The block-sparse pattern of the workloads, as a tile bitmap.

    Query tile qt sees key tiles qt - window_before .. qt + window_after (clipped at the
    ends, no wrap) and every key tile kt with kt % global_stride == 0. The pages name a
    blocked sparse pattern without giving it; this window-plus-global reading is the one
    the workload table fixes.
    """
    qt = np.arange(n_tiles)[:, None]
    kt = np.arange(n_tiles)[None, :]
    return ((kt >= qt - window_before) & (kt <= qt + window_after)) | (kt % global_stride == 0)


def mask_for(workload) -> Mask:
    if workload.mask == "causal":
        return Mask("causal")
    if workload.mask == "none":
        return Mask("none")
    n = -(-workload.L // workload.tile)
    return Mask("tiles", workload.tile, window_global_tiles(
        n, workload.window_before, workload.window_after, workload.global_stride))


# --------------------------------------------------------------------------- attention

def _chunk_rows(L: int) -> int:
    return max(1, min(4096, (1 << 22) // max(L, 1)))


def head_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows: np.ndarray, mask: Mask,
                 scale: float):
    """Exact attention for one (batch, head) on the given query rows.

    q, k, v: fp64 [L, d] for the full sequence. Returns (O [n, d], LSE [n]).
    S_ij = scale * Q_i . K_j on permitted pairs; m_i = max_j S_ij;
    O_i = sum_j exp(S_ij - m_i) V_j / sum_j exp(S_ij - m_i); LSE_i = m_i + ln sum_j exp(S_ij - m_i).
    """
    L, d = k.shape
    n = len(rows)
    O = np.zeros((n, d))
    LSE = np.full(n, -np.inf)
    step = _chunk_rows(L)
    for c0 in range(0, n, step):
        r = rows[c0:c0 + step]
        allow = mask.rows(r, L)
        S = np.where(allow, (q[r] @ k.T) * scale, -np.inf)
        m = S.max(axis=1)
        has = np.isfinite(m)
        E = np.where(allow & has[:, None], np.exp(S - np.where(has, m, 0.0)[:, None]), 0.0)
        ell = E.sum(axis=1)
        safe = np.where(has, ell, 1.0)
        O[c0:c0 + step] = np.where(has[:, None], (E @ v) / safe[:, None], 0.0)
        LSE[c0:c0 + step] = np.where(has, m + np.log(safe), -np.inf)
    return O, LSE


def head_backward(q, k, v, dO_rows, O_rows, LSE_rows, rows, mask: Mask, scale: float):
    """Analytic gradient for one (batch, head), restricted to the given query rows.

    Returns (dQ [n, d] for those rows, dK [L, d], dV [L, d]) where dK and dV are the
    contributions of those rows only -- the full gradient when rows covers every row.
    """
    L, d = k.shape
    n = len(rows)
    dQ = np.zeros((n, d))
    dK = np.zeros((L, d))
    dV = np.zeros((L, d))
    step = _chunk_rows(L)
    for c0 in range(0, n, step):
        r = rows[c0:c0 + step]
        allow = mask.rows(r, L)
        lse = LSE_rows[c0:c0 + step]
        has = np.isfinite(lse)
        S = (q[r] @ k.T) * scale
        Pm = np.where(allow & has[:, None], np.exp(S - np.where(has, lse, 0.0)[:, None]), 0.0)
        dOr = dO_rows[c0:c0 + step]
        delta = np.sum(dOr * O_rows[c0:c0 + step], axis=1)
        dV += Pm.T @ dOr
        dP = dOr @ v.T
        dS = Pm * (dP - delta[:, None])
        dQ[c0:c0 + step] = scale * (dS @ k)
        dK += scale * (dS.T @ q[r])
    return dQ, dK, dV


def _head_view(y: np.ndarray, g: int, b: int, j: int) -> np.ndarray:
    return y[g, b, :, j, :]


def attention_full(q_tok: np.ndarray, k_tok: np.ndarray, v_tok: np.ndarray, P: int, mask: Mask,
                   do_tok: Optional[np.ndarray] = None, scale: Optional[float] = None) -> Dict[str, np.ndarray]:
    """The whole attention block on token-sharded inputs, every row.

    Inputs are bf16 bit patterns (uint16) or fp64 arrays: Q (and dO) [P][B][Lp][H][d], K and V
    [P][B][Lp][Hkv][d] with H % Hkv == 0 (Hkv == H is plain multi-head attention).
    Steps: seq->head relayout of Q (and dO) and of K, V (kv_seq_to_head); per head group and
    query head h, exact attention over the full sequence against K/V head h // (H/Hkv) (and its
    gradient); head->seq relayout of O, dQ, and the summing adjoint for dK, dV. Returns fp64
    "o" (and "dq", "dk", "dv") in the token layout and "lse" [P][B][Hp][L].
    """
    head = {"q": seq_to_head(q_tok, P), "k": kv_seq_to_head(k_tok, P), "v": kv_seq_to_head(v_tok, P)}
    if do_tok is not None:
        head["do"] = seq_to_head(do_tok, P)
    head = {n: bf16_to_f64(y) if y.dtype == np.uint16 else y.astype(np.float64) for n, y in head.items()}
    _, B, L, Hp, d = head["q"].shape
    Hkv = k_tok.shape[3]
    H = Hp * P
    G = H // Hkv
    Hkvp = head["k"].shape[3]
    sc = 1.0 / np.sqrt(d) if scale is None else scale
    o = np.zeros((P, B, L, Hp, d))
    lse = np.zeros((P, B, Hp, L))
    grads = {}
    if do_tok is not None:
        grads = {"dq": np.zeros((P, B, L, Hp, d)), "dk": np.zeros((P, B, L, Hkvp, d)),
                 "dv": np.zeros((P, B, L, Hkvp, d))}
    rows = np.arange(L)
    for g in range(P):
        for b in range(B):
            for j in range(Hp):
                h = g * Hp + j
                jk = h // G - g * Hkvp if Hkv >= P else 0
                qh = head["q"][g, b, :, j, :]
                kh, vh = head["k"][g, b, :, jk, :], head["v"][g, b, :, jk, :]
                O, LSE = head_forward(qh, kh, vh, rows, mask, sc)
                o[g, b, :, j, :] = O
                lse[g, b, j, :] = LSE
                if do_tok is not None:
                    dQ, dK, dV = head_backward(qh, kh, vh, head["do"][g, b, :, j, :], O, LSE, rows, mask, sc)
                    grads["dq"][g, b, :, j, :] = dQ
                    grads["dk"][g, b, :, jk, :] += dK
                    grads["dv"][g, b, :, jk, :] += dV
    out = {"o": head_to_seq(o, P), "lse": lse}
    if grads:
        out["dq"] = head_to_seq(grads["dq"], P)
        out["dk"] = kv_head_to_seq_sum(grads["dk"], P, Hkv)
        out["dv"] = kv_head_to_seq_sum(grads["dv"], P, Hkv)
    return out


# --------------------------------------------------------------------------- ring merge

def merge_partials(o_parts, lse_parts):
    """Combine attention results over disjoint key sets into the result over their union (the
    online-softmax rule that ring attention streams K/V blocks with; pages' Ring Attention /
    USP hybrid): with m = max_j lse_j, w_j = exp(lse_j - m),
        lse = m + ln sum_j w_j,   O = sum_j w_j O_j / sum_j w_j.
    o_parts: list of [..., n, d] arrays, lse_parts: list of matching [..., n] arrays (same
    leading shape). A row with lse = -inf in every part gets O = 0 and lse = -inf."""
    lse = np.stack([np.asarray(x, dtype=np.float64) for x in lse_parts])      # [J, ..., n]
    o = np.stack([np.asarray(x, dtype=np.float64) for x in o_parts])          # [J, ..., n, d]
    m = lse.max(axis=0)
    finite = np.isfinite(m)
    w = np.where(finite, np.exp(lse - np.where(finite, m, 0.0)), 0.0)
    tot = w.sum(axis=0)
    out_lse = np.where(finite, m + np.log(np.where(finite, tot, 1.0)), -np.inf)
    out_o = np.where(finite[..., None], (w[..., None] * o).sum(axis=0) / np.where(finite, tot, 1.0)[..., None], 0.0)
    return out_o, out_lse


# --------------------------------------------------------------------------- projections

def _as_f64(x: np.ndarray) -> np.ndarray:
    return bf16_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def qkv_projection(x_tok: np.ndarray, w_qkv: np.ndarray, H: int, Hkv: int, d: int) -> Dict[str, np.ndarray]:
    """Local QKV projection of token-sharded hidden states.

    x_tok [P][B][Lp][hidden] (bf16 bits or floats); w_qkv [(H + 2 Hkv) d][hidden], rows
    ordered Q heads, then K heads, then V heads (y = x W^T). Returns fp64 "q"
    [P][B][Lp][H][d], "k" and "v" [P][B][Lp][Hkv][d]: every token row of every shard is
    projected on its own, so the outputs keep the token-sharded layout.
    """
    x = _as_f64(x_tok)
    w = _as_f64(w_qkv)
    P, B, Lp, hidden = x.shape
    assert w.shape == ((H + 2 * Hkv) * d, hidden)
    y = (x.reshape(-1, hidden) @ w.T).reshape(P, B, Lp, H + 2 * Hkv, d)
    return {"q": y[:, :, :, :H], "k": y[:, :, :, H:H + Hkv], "v": y[:, :, :, H + Hkv:]}


def out_projection(o_tok: np.ndarray, w_o: np.ndarray) -> np.ndarray:
    """Output projection of the token-sharded attention output: o_tok [P][B][Lp][H][d],
    w_o [hidden][H d]; returns fp64 [P][B][Lp][hidden] (y = o W_o^T per token row)."""
    o = _as_f64(o_tok)
    w = _as_f64(w_o)
    P, B, Lp, H, d = o.shape
    return (o.reshape(-1, H * d) @ w.T).reshape(P, B, Lp, w.shape[0])


def _sampled_task(task):
    """One (batch, head) of the sampled mode; runs in the caller or in a pool worker."""
    b, h, kvh, rows, heads, mask, sc = task
    conv = {nme: bf16_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64) for nme, x in heads.items()}
    O, LSE = head_forward(conv["q"], conv["k"], conv["v"], rows, mask, sc)
    res = {"b": b, "h": h, "kvh": kvh, "rows": rows, "o": O, "lse": LSE}
    if "do" in conv:
        dQ, dK, dV = head_backward(conv["q"], conv["k"], conv["v"], conv["do"][rows], O, LSE, rows, mask, sc)
        res.update(dq=dQ, dk=dK, dv=dV)
    return res


_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def attention_sampled(q_tok, k_tok, v_tok, do_tok, P: int, mask: Mask, rows_bi: np.ndarray,
                      scale: Optional[float] = None, heads=None, workers: int = 0) -> Iterator[dict]:
    """Per-(batch, query head) results on sampled query rows, for workloads too large to do whole.

    rows_bi: int [n, 2] of (b, i). For each (b, h) yields a dict with "b", "h", "kvh" (the K/V
      head it attends with, h // (H/Hkv)), "rows" (sequence indices i), "o" [n_b, d], "lse"
      [n_b], and, when do_tok is given, "dq" [n_b, d] and "dk", "dv" [L, d]: this query head's
      sampled rows' gradient contributions to K/V head kvh (summing them over the query heads
      of a group gives what a pass whose dO is zero on every other row produces).
    (batch, head) pairs are independent; with workers > 1 they are spread over a process
    pool started with "spawn" (results arrive in the same order).
    """
    head = {"q": seq_to_head(q_tok, P), "k": kv_seq_to_head(k_tok, P), "v": kv_seq_to_head(v_tok, P)}
    if do_tok is not None:
        head["do"] = seq_to_head(do_tok, P)
    _, B, L, Hp, d = head["q"].shape
    H = Hp * P
    Hkv = k_tok.shape[3]
    G = H // Hkv
    Hkvp = head["k"].shape[3]
    sc = 1.0 / np.sqrt(d) if scale is None else scale

    def tasks():
        for b in range(B):
            rows = rows_bi[rows_bi[:, 0] == b, 1]
            if len(rows) == 0:
                continue
            for h in (range(H) if heads is None else heads):
                g, j = divmod(h, Hp)
                jk = h // G - g * Hkvp if Hkv >= P else 0
                views = {"q": head["q"][g, b, :, j, :], "k": head["k"][g, b, :, jk, :], "v": head["v"][g, b, :, jk, :]}
                if "do" in head:
                    views["do"] = head["do"][g, b, :, j, :]
                yield (b, h, h // G, rows, {n: np.ascontiguousarray(x) for n, x in views.items()}, mask, sc)

    if workers <= 1:
        for task in tasks():
            yield _sampled_task(task)
        return
    import concurrent.futures
    import multiprocessing
    ctx = multiprocessing.get_context("spawn")
    # one BLAS thread per worker (the pool supplies the parallelism): the variables must be
    # in the environment when a worker starts, before it loads numpy
    saved = {v: os.environ.get(v) for v in _BLAS_VARS}
    os.environ.update({v: "1" for v in _BLAS_VARS})
    try:
        with concurrent.futures.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as ex:
            pending = []
            for task in tasks():
                pending.append(ex.submit(_sampled_task, task))
                if len(pending) >= 2 * workers:
                    yield pending.pop(0).result()
            for f in pending:
                yield f.result()
    finally:
        for v, val in saved.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val
