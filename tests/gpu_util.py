"""Helpers shared by the GPU parity tests (test infrastructure only)."""

import os

import numpy as np
import pytest
import torch

import oracle
import ulysses_sequence_gb300 as U
import workloads

# Acceptance for bf16 outputs against the fp64 oracle, and for the fp32 log-sum-exp.
MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_MAX_ABS = 1e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ulysses_sequence_gb300 import build
    build.build()
    U.load()


class ErrStats:
    """Accumulates max-abs and relative-L2 error of many pieces of one tensor."""

    def __init__(self, name):
        self.name, self.max_abs, self.num, self.den, self.n = name, 0.0, 0.0, 0.0, 0

    def add(self, got, ref):
        got = np.asarray(got, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        assert got.shape == ref.shape, (self.name, got.shape, ref.shape)
        assert np.all(np.isfinite(got)), f"{self.name}: non-finite values"
        d = got - ref
        if d.size:
            self.max_abs = max(self.max_abs, float(np.abs(d).max()))
        self.num += float(np.sum(d * d))
        self.den += float(np.sum(ref * ref))
        self.n += d.size

    @property
    def rel_l2(self):
        return (self.num ** 0.5) / max(self.den ** 0.5, 1e-300)

    def check(self, max_abs=MAX_ABS, rel_l2=REL_L2):
        assert self.n > 0, self.name
        if max_abs is not None:
            assert self.max_abs <= max_abs, f"{self.name}: max-abs {self.max_abs:.3e} > {max_abs}"
        if rel_l2 is not None:
            assert self.rel_l2 <= rel_l2, f"{self.name}: rel-L2 {self.rel_l2:.3e} > {rel_l2}"
        return self


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def logical(x_tok: np.ndarray) -> np.ndarray:
    """[P][B][Lp][H][d] -> [B][L][H][d]."""
    P, B, Lp, H, d = x_tok.shape
    return x_tok.transpose(1, 0, 2, 3, 4).reshape(B, P * Lp, H, d)


def lse_logical(lse: np.ndarray) -> np.ndarray:
    """[P][B][Hp][L] -> [B][H][L]."""
    P, B, Hp, L = lse.shape
    return lse.transpose(1, 0, 2, 3).reshape(B, P * Hp, L)


def gpu_mask(kind: str, L: int, tiles: np.ndarray = None, w: "workloads.Workload" = None):
    """The library-side mask: causal / none, or block-sparse tile lists on the device."""
    if kind == "causal":
        return U.Mask.causal()
    if kind == "none":
        return U.Mask.none()
    if w is not None:
        return U.Mask.window_global(L, 128, w.window_before, w.window_after, w.global_stride)
    n = tiles.shape[0]
    rp, kc = [0], []
    for qt in range(n):
        kc += [int(k) for k in np.nonzero(tiles[qt])[0]]
        rp.append(len(kc))
    cp, qr = [0], []
    for kt in range(n):
        qr += [int(q) for q in np.nonzero(tiles[:, kt])[0]]
        cp.append(len(qr))
    return U.Mask.from_tile_lists(rp, kc if kc else [0], cp, qr if qr else [0])


def env_rows(default: int) -> int:
    return int(os.environ.get("ULYSSES_SAMPLED_ROWS", default))
