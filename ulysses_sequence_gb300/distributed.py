"""DeepSpeed-Ulysses across processes: one token shard per rank, an all-to-all on each side of
per-head-group attention (paper summary section 3.4.2 "The All-to-All Communication
Primitive"; aifetchly guide, "Explanation of the Implementation", item 2).

Each of the P processes of a torch.distributed group holds its own token shard
[B][L/P][H][d_h] on its own GPU. The forward pass:

1. packs Q, K and V into P contiguous per-destination chunks (``a2a_pack``: chunk g holds head
   group g, heads [g H/P, (g+1) H/P));
2. exchanges them with ``all_to_all_single``, so that rank g receives every rank's tokens of
   head group g in sender order: the head-sharded [B][L][H/P][d_h] of its group, the whole
   sequence;
3. runs the library's attention on that group alone (one shard, P = 1, every token local);
4. sends O back the same way (the second all-to-all) and unpacks it (``a2a_unpack``) into
   its token shard [B][L/P][H][d_h].

The backward pass mirrors it: dO travels like Q, the local backward runs on the rank's head
group, and dQ, dK, dV travel like O. lse stays with its head group, where the backward needs
it. The library kernels only ever touch this process's device memory; moving data between
processes is the collective's job (NCCL on GPUs). Key/value tensors may have H_kv < H heads
as long as H_kv % P == 0 (each rank keeps the key/value heads of its query heads).

The local steps are an object (``LibraryOps`` by default: the CUDA library on this process's
GPU) so that the same exchange code can be driven with other local compute.
"""

from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

import ulysses_sequence_gb300 as U


class LibraryOps:
    """The local steps of one rank, on its GPU, through libulysses: packing, unpacking and
    attention over one head group (P = 1)."""

    def __init__(self, mask: "U.Mask", scale: float = 0.0):
        self.mask, self.scale = mask, scale
        self._ws = None

    def empty(self, shape, like: torch.Tensor) -> torch.Tensor:
        return torch.empty(shape, dtype=like.dtype, device=like.device)

    def pack(self, x: torch.Tensor, P: int) -> torch.Tensor:
        return U.a2a_pack(x, P)

    def unpack(self, y: torch.Tensor, P: int, out: torch.Tensor) -> torch.Tensor:
        return U.a2a_unpack(y, P, out=out)

    def attn_fwd(self, q, k, v):
        """q [B][L][Hg][d], k, v [B][L][Hkvg][d] -> (o [B][L][Hg][d], lse [1][B][Hg][L] fp32)."""
        o, lse = U.attn_fwd(q[None], k[None], v[None], 1, self.mask, scale=self.scale)
        return o[0], lse

    def attn_bwd(self, q, k, v, o, lse, do):
        """The analytic gradient of attn_fwd on the same head group: (dq, dk, dv)."""
        n = U.ulysses_attn_bwd_workspace_size(U._shape_of(q[None], 1, U.LAYOUT_TOKEN_SHARDED, k[None]))
        if self._ws is None or self._ws.numel() < n or self._ws.device != q.device:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
        dq, dk, dv = U.attn_bwd(q[None], k[None], v[None], o[None], lse, do[None], 1, self.mask, scale=self.scale,
                                workspace=self._ws)
        return dq[0], dk[0], dv[0]


class UlyssesAttention:
    """Ulysses sequence-parallel attention over the processes of ``group``.

    forward(q, k, v) takes this rank's token shards (q [B][L/P][H][d_h], k and v with H_kv
    heads) and returns (o [B][L/P][H][d_h], ctx); backward(ctx, do) returns (dq, dk, dv) in
    the same token-sharded layout."""

    def __init__(self, group: Optional["dist.ProcessGroup"] = None, ops=None, mask: Optional["U.Mask"] = None,
                 scale: float = 0.0):
        self.group = group
        self.P = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.ops = ops if ops is not None else LibraryOps(mask if mask is not None else U.Mask.causal(), scale)

    # ------------------------------------------------------------------ the two exchanges
    def to_heads(self, x: torch.Tensor) -> torch.Tensor:
        """The first all-to-all: this rank's tokens [B][L/P][H][d] -> its head group over the
        whole sequence [B][L][H/P][d] (token order = sender order = global position)."""
        P = self.P
        B, Lp, H, d = x.shape
        if H % P != 0:
            raise ValueError(f"{H} heads do not split over {P} ranks")
        Hg = H // P
        out = self.ops.empty((B, Lp * P, Hg, d), x)
        for b in range(B):  # one exchange per batch row keeps each receive buffer contiguous
            send = self.ops.pack(x[b:b + 1], P)  # [P][1][Lp][Hg][d]
            dist.all_to_all_single(out[b].view(P, Lp, Hg, d), send.view(P, Lp, Hg, d), group=self.group)
        return out

    def to_tokens(self, y: torch.Tensor) -> torch.Tensor:
        """The second all-to-all: this rank's head group [B][L][Hg][d] -> its tokens with every
        head [B][L/P][P Hg][d]."""
        P = self.P
        B, L, Hg, d = y.shape
        Lp = L // P
        out = self.ops.empty((B, Lp, Hg * P, d), y)
        for b in range(B):
            recv = self.ops.empty((P, 1, Lp, Hg, d), y)
            dist.all_to_all_single(recv.view(P, Lp, Hg, d), y[b].view(P, Lp, Hg, d), group=self.group)
            self.ops.unpack(recv, P, out[b:b + 1])
        return out

    # ------------------------------------------------------------------ passes
    def forward(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
        if k.shape[2] % self.P != 0:
            raise ValueError(f"{k.shape[2]} key/value heads do not split over {self.P} ranks")
        qh, kh, vh = self.to_heads(q), self.to_heads(k), self.to_heads(v)
        oh, lse = self.ops.attn_fwd(qh, kh, vh)
        return self.to_tokens(oh), (qh, kh, vh, oh, lse)

    def backward(self, ctx, do: torch.Tensor):
        qh, kh, vh, oh, lse = ctx
        dqh, dkh, dvh = self.ops.attn_bwd(qh, kh, vh, oh, lse, self.to_heads(do))
        return self.to_tokens(dqh), self.to_tokens(dkh), self.to_tokens(dvh)
