"""Seeded synthetic workloads for the Ulysses attention block.

This module holds the workload table and the random-input generators shared by the
tests, the benchmark and the smoke check. It contains none of the method's arithmetic:
it draws N(0, 1) values of the logical global shape [B, L, H, d_h], optionally scales
the queries, rounds to bf16 and cuts the sequence into P contiguous token shards. That
cut is the input partition of DeepSpeed-Ulysses (paper summary, section 3.2 "Big-Picture
Architecture", item 1, and section 3.4.1: rank i holds positions [i*N/P, (i+1)*N/P)),
so the returned tensors are in the token-sharded layout [P][B][L/P][H][d_h].

The paper trains on synthesized data and names no public dataset, so every input here
is synthetic by construction.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, Iterable, List, Optional, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention-block configuration.

    mask: "causal", "none" (bidirectional dense) or "block_sparse".
    For "block_sparse" the pattern is whole `tile` x `tile` blocks: query tile qt sees
    key tiles kt with qt - window_before <= kt <= qt + window_after (clipped at the
    sequence ends) plus every key tile with kt % global_stride == 0.
    """

    name: str
    B: int
    L: int
    H: int
    d: int
    P: int
    mask: str
    backward: bool
    seed: int
    q_scale: float = 1.0
    tile: int = 128
    window_before: int = 4
    window_after: int = 3
    global_stride: int = 16
    sampled_rows: int = 0  # 0: the oracle checks every row
    H_kv: int = 0          # key/value heads (grouped-query attention); 0: H

    @property
    def Lp(self) -> int:
        return self.L // self.P

    @property
    def Hp(self) -> int:
        return self.H // self.P

    @property
    def Hkv(self) -> int:
        return self.H_kv or self.H


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        # B=1, L=256, H=8, d_h=64, P=4; causal forward + backward; seed 0.
        Workload("tiny", 1, 256, 8, 64, 4, "causal", True, 0),
        # GPT-1.2B-like layer: B=1, L=8192, hidden 2048 = 16 heads x 128; P=8; forward only.
        Workload("gpt1.2b", 1, 8192, 16, 128, 8, "causal", False, 1),
        # GPT-7B-like layer: B=1, L=32768, H=32, d_h=128, P=8; Q scaled by 1/sqrt(d_h).
        Workload("gpt7b", 1, 32768, 32, 128, 8, "causal", True, 2,
                 q_scale=1.0 / math.sqrt(128.0), sampled_rows=4096),
        # Long sequence: B=1, L=131072, H=32, d_h=128, P=32 (one head per group).
        Workload("long", 1, 131072, 32, 128, 32, "causal", True, 3, sampled_rows=4096),
        # Block-sparse, bidirectional: B=2, L=65536, H=32, d_h=128, P=8, 128x128 tiles,
        # an 8-tile sliding window plus every 16th key tile as global.
        Workload("block_sparse", 2, 65536, 32, 128, 8, "block_sparse", True, 4,
                 sampled_rows=4096),
        # Grouped-query variant of the GPT-7B-like layer: 32 query heads share 8 key/value
        # heads (groups of 4); each of the P=8 head groups receives one whole key/value head.
        Workload("gpt7b_gqa", 1, 32768, 32, 128, 8, "causal", True, 5,
                 q_scale=1.0 / math.sqrt(128.0), sampled_rows=4096, H_kv=8),
    ]
}


def to_bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a bf16 tensor as a numpy uint16 array (no copy of values)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def shard_tokens(x: torch.Tensor, P: int) -> torch.Tensor:
    """[B, L, H, d] -> [P, B, L/P, H, d]: shard r holds global tokens [r*L/P, (r+1)*L/P)."""
    B, L, H, d = x.shape
    assert L % P == 0
    return x.reshape(B, P, L // P, H, d).permute(1, 0, 2, 3, 4).contiguous()


def draw(B: int, L: int, H: int, d: int, P: int, seed: int, names: Iterable[str] = ("q", "k", "v", "do"),
         q_scale: float = 1.0, H_kv: int = 0) -> Dict[str, torch.Tensor]:
    """Draw bf16 tensors in the token-sharded layout [P][B][L/P][H][d] from one CPU generator.

    Tensors are drawn in the order given (q, k, v, do by default) as fp32 N(0, 1) of the
    logical shape [B, L, H, d] (k and v with H_kv heads when H_kv is given); q is
    multiplied by q_scale in fp32 before the round-to-nearest-even conversion to bf16.
    """
    g = torch.Generator().manual_seed(seed)
    out = {}
    for n in names:
        heads = H_kv if (H_kv and n in ("k", "v")) else H
        x = torch.randn((B, L, heads, d), generator=g, dtype=torch.float32)
        if n == "q" and q_scale != 1.0:
            x.mul_(q_scale)
        out[n] = shard_tokens(x.to(torch.bfloat16), P)
        del x
    return out


def draw_weight(n_out: int, n_in: int, seed: int) -> torch.Tensor:
    """A bf16 projection weight [n_out][n_in] (the y = x W^T convention): fp32 N(0, 1) / sqrt(n_in)
    from its own CPU generator, rounded to nearest-even. The scale keeps projected values near
    unit size, as a trained layer's initialisation would."""
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((n_out, n_in), generator=g, dtype=torch.float32) / math.sqrt(n_in)).to(torch.bfloat16)


def draw_hidden(B: int, L: int, hidden: int, P: int, seed: int) -> torch.Tensor:
    """Token-sharded bf16 hidden states [P][B][L/P][hidden], fp32 N(0, 1) rounded to nearest-even."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((B, L, hidden), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return x.reshape(B, P, L // P, hidden).permute(1, 0, 2, 3).contiguous()


def draw_workload(w: Workload, names: Iterable[str] = ("q", "k", "v", "do")) -> Dict[str, torch.Tensor]:
    return draw(w.B, w.L, w.H, w.d, w.P, w.seed, names, q_scale=w.q_scale, H_kv=w.H_kv)


def sample_rows(B: int, L: int, n: int, seed: int) -> np.ndarray:
    """n distinct (b, i) query rows, uniform over the batch and sequence, always with
    (0, 0) and (0, L-1). Returns int64 [n, 2] sorted by (b, i)."""
    total = B * L
    n = min(n, total)
    rng = np.random.default_rng(seed)
    flat = set([0, L - 1])
    picked = rng.choice(total, size=n, replace=False)
    for f in picked:
        if len(flat) >= n:
            break
        flat.add(int(f))
    flat = np.array(sorted(flat), dtype=np.int64)
    return np.stack([flat // L, flat % L], axis=1)

