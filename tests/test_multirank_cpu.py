"""Multi-rank paths on CPU with the gloo backend (world size 2).

- bench.py's plumbing: the barrier, the max-over-ranks timing reduction, and a torchrun launch
  of the reference arm in which only rank 0 works and prints exactly one JSON line.
- The method's exchanges with one shard per process: the package's Ulysses layer
  (ulysses_sequence_gb300.distributed: pack, all_to_all_single, per-head-group attention,
  all_to_all_single, unpack) driven over gloo with the oracle as each rank's local attention,
  and the USP ring, in which key/value
  blocks (and, backward, their dK/dV accumulators) travel from rank to rank and the partial
  results merge by the online-softmax rule. Each rank computes with the fp64 oracle; the
  assembled O, lse, dQ, dK, dV must equal whole-sequence attention.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + rank, w)
    out[rank] = m
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert dict(out) == {0: 11.0, 1: 11.0}


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3", "--ref-rows", "8",
           "--ref-heads", "1", "--gpus", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


# --------------------------------------------------------------------------------------------
# The method's exchanges across real process boundaries (gloo, CPU). One GPU per run here means
# the library keeps all P shards in one HBM; these tests run the same decomposition with one
# shard per process, exchanged by point-to-point messages, and the fp64 oracle as each rank's
# compute, against whole-sequence attention.

def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _exchange(send_parts, recv_shapes):
    """Send send_parts[g] to rank g and receive an array of recv_shapes[s] from each rank s
    (one's own part is kept): an all-to-all from point-to-point messages."""
    import numpy as np
    me, world = dist.get_rank(), dist.get_world_size()
    reqs = [dist.isend(torch.from_numpy(np.ascontiguousarray(send_parts[g])), dst=g)
            for g in range(world) if g != me]
    got = {}
    for s in range(world):
        if s == me:
            got[s] = np.ascontiguousarray(send_parts[me])
        else:
            buf = torch.empty(recv_shapes[s], dtype=torch.float64)
            dist.recv(buf, src=s)
            got[s] = buf.numpy()
    for r in reqs:
        r.wait()
    return [got[s] for s in range(world)]


def _inputs(B, L, H, d, P, seed):
    import oracle
    import workloads
    t = workloads.draw(B, L, H, d, P, seed)
    return {n: oracle.bf16_to_f64(workloads.to_bf16_bits(x)) for n, x in t.items()}


class _OracleOps:
    """Local steps on the CPU for the package's exchange code (UlyssesAttention): packing and
    unpacking written here with torch views, attention by the fp64 oracle per (batch, head)."""

    def __init__(self):
        import oracle
        self.oracle = oracle
        self.mask = oracle.Mask("causal")

    def empty(self, shape, like):
        return torch.empty(shape, dtype=torch.float64)

    def pack(self, x, P):
        B, Lp, H, d = x.shape
        return x.reshape(B, Lp, P, H // P, d).permute(2, 0, 1, 3, 4).contiguous()

    def unpack(self, y, P, out):
        Pn, B, Lp, Hg, d = y.shape
        out.copy_(y.permute(1, 2, 0, 3, 4).reshape(B, Lp, P * Hg, d))
        return out

    def _kv(self, j, Hg, Hkvg):
        return j // (Hg // Hkvg)

    def attn_fwd(self, q, k, v):
        import numpy as np
        B, L, Hg, d = q.shape
        rows = np.arange(L)
        sc = 1.0 / np.sqrt(d)
        o = np.zeros((B, L, Hg, d))
        lse = np.zeros((1, B, Hg, L))
        for b in range(B):
            for j in range(Hg):
                kj = self._kv(j, Hg, k.shape[2])
                o[b, :, j], lse[0, b, j] = self.oracle.head_forward(q[b, :, j].numpy(), k[b, :, kj].numpy(),
                                                                    v[b, :, kj].numpy(), rows, self.mask, sc)
        return torch.from_numpy(o), torch.from_numpy(lse)

    def attn_bwd(self, q, k, v, o, lse, do):
        import numpy as np
        B, L, Hg, d = q.shape
        rows = np.arange(L)
        sc = 1.0 / np.sqrt(d)
        dq = np.zeros((B, L, Hg, d))
        dk, dv = np.zeros(tuple(k.shape)), np.zeros(tuple(v.shape))
        for b in range(B):
            for j in range(Hg):
                kj = self._kv(j, Hg, k.shape[2])
                g = self.oracle.head_backward(q[b, :, j].numpy(), k[b, :, kj].numpy(), v[b, :, kj].numpy(),
                                              do[b, :, j].numpy(), o[b, :, j].numpy(), lse[0, b, j].numpy(), rows,
                                              self.mask, sc)
                dq[b, :, j] = g[0]
                dk[b, :, kj] += g[1]
                dv[b, :, kj] += g[2]
        return torch.from_numpy(dq), torch.from_numpy(dk), torch.from_numpy(dv)


ULY_CASES = {"mha": (2, 256, 4, 4, 32), "gqa": (1, 256, 8, 4, 32)}  # B, L, H, H_kv, d


def _ulysses_worker(rank, world, port, out, case):
    """The package's two all-to-alls (UlyssesAttention over gloo), one token shard per rank, the
    fp64 oracle as each rank's local attention, forward and backward."""
    _init(rank, world, port)
    import workloads
    from ulysses_sequence_gb300.distributed import UlyssesAttention
    import oracle
    B, L, H, Hkv, d = ULY_CASES[case]
    t = workloads.draw(B, L, H, d, world, seed=11, H_kv=Hkv)
    x = {n: torch.from_numpy(oracle.bf16_to_f64(workloads.to_bf16_bits(a))[rank]) for n, a in t.items()}
    ua = UlyssesAttention(ops=_OracleOps())
    o, ctx = ua.forward(x["q"], x["k"], x["v"])
    dq, dk, dv = ua.backward(ctx, x["do"])
    out[rank] = {"o": o.numpy(), "dq": dq.numpy(), "dk": dk.numpy(), "dv": dv.numpy(), "lse": ctx[4][0].numpy()}
    dist.destroy_process_group()


def _ring_worker(rank, world, port, out):
    """The USP ring with P_ring = world and P_u = 1: rank r holds ring block r (all heads). The
    key/value blocks travel around the ring; each rank attends its query block to every block
    that reaches it (causal: its own block causally, earlier blocks densely, later ones not at
    all) and merges the partial results by the online-softmax rule. In the backward pass the
    key/value blocks travel with their dK, dV accumulators and return to their owners."""
    _init(rank, world, port)
    import numpy as np
    import oracle
    B, L, H, d, P = 1, 256, 2, 32, world
    Lb = L // P
    x = {n: a[rank] for n, a in _inputs(B, L, H, d, P, seed=12).items()}  # ring block [B][Lb][H][d]
    sc = 1.0 / np.sqrt(d)
    rows = np.arange(Lb)
    nxt, prv = (rank + 1) % P, (rank - 1) % P

    def pass_on(arrays):
        """Send to the next rank, receive the same shapes from the previous one."""
        reqs = [dist.isend(torch.from_numpy(np.ascontiguousarray(a)), dst=nxt) for a in arrays]
        got = []
        for a in arrays:
            buf = torch.empty(a.shape, dtype=torch.float64)
            dist.recv(buf, src=prv)
            got.append(buf.numpy())
        for r in reqs:
            r.wait()
        return got

    def pair_mask(j):
        return oracle.Mask("causal") if j == rank else (oracle.Mask("none") if j < rank else None)

    # forward: partial (O, lse) per block that reaches this rank, then the merge
    k, v, j = x["k"], x["v"], rank
    o_parts, lse_parts = [], []
    for step in range(P):
        m = pair_mask(j)
        if m is not None:
            o_j = np.zeros((B, H, Lb, d))
            l_j = np.zeros((B, H, Lb))
            for b in range(B):
                for h in range(H):
                    o_j[b, h], l_j[b, h] = oracle.head_forward(x["q"][b, :, h], k[b, :, h], v[b, :, h], rows, m, sc)
            o_parts.append(o_j)
            lse_parts.append(l_j)
        k, v = pass_on([k, v])
        j = (j - 1) % P
    o, lse = oracle.merge_partials(o_parts, lse_parts)  # [B][H][Lb][d], [B][H][Lb]
    # backward: every block pair's gradient with the merged O and lse
    k, v, j = x["k"], x["v"], rank
    dk_acc, dv_acc = np.zeros_like(k), np.zeros_like(v)
    dq = np.zeros_like(x["q"])
    for step in range(P):
        m = pair_mask(j)
        if m is not None:
            for b in range(B):
                for h in range(H):
                    g_q, g_k, g_v = oracle.head_backward(x["q"][b, :, h], k[b, :, h], v[b, :, h], x["do"][b, :, h],
                                                         o[b, h], lse[b, h], rows, m, sc)
                    dq[b, :, h] += g_q
                    dk_acc[b, :, h] += g_k
                    dv_acc[b, :, h] += g_v
        k, v, dk_acc, dv_acc = pass_on([k, v, dk_acc, dv_acc])
        j = (j - 1) % P
    assert j == rank  # after a full circle each rank holds its own block and its gradients again
    out[rank] = {"o": o.transpose(0, 2, 1, 3), "lse": lse, "dq": dq, "dk": dk_acc, "dv": dv_acc}
    dist.destroy_process_group()


def _whole_sequence(B, L, H, d, P, seed):
    import oracle
    x = _inputs(B, L, H, d, P, seed)
    one = {n: a.transpose(1, 0, 2, 3, 4).reshape(1, B, L, H, d) for n, a in x.items()}
    ref = oracle.attention_full(one["q"], one["k"], one["v"], 1, oracle.Mask("causal"), do_tok=one["do"])
    return {n: ref[n][0] for n in ("o", "dq", "dk", "dv")}, ref["lse"][0]  # [B][L][H][d], [B][H][L]


def _run_ranks(worker, world):
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(worker, args=(world, port, out), nprocs=world, join=True)
    return dict(out)


@pytest.mark.parametrize("world,case", [(2, "mha"), (4, "gqa")])
def test_ulysses_all_to_all_across_ranks_equals_whole_sequence(world, case):
    """ulysses_sequence_gb300.distributed on gloo: every rank's O, dQ, dK, dV (its tokens) and
    lse (its head group) equal attention over the whole sequence."""
    import numpy as np
    import oracle
    import workloads
    port = _free_port()
    res = mp.get_context("spawn").Manager().dict()
    mp.spawn(_ulysses_worker, args=(world, port, res, case), nprocs=world, join=True)
    got = dict(res)
    B, L, H, Hkv, d = ULY_CASES[case]
    t = workloads.draw(B, L, H, d, world, seed=11, H_kv=Hkv)
    x = {n: oracle.bf16_to_f64(workloads.to_bf16_bits(a)) for n, a in t.items()}
    one = {n: a.transpose(1, 0, 2, 3, 4).reshape(1, B, L, a.shape[3], d) for n, a in x.items()}
    ref = oracle.attention_full(one["q"], one["k"], one["v"], 1, oracle.Mask("causal"), do_tok=one["do"])
    Lp, Hp = L // world, H // world
    for r in range(world):
        for n in ("o", "dq", "dk", "dv"):
            assert np.allclose(got[r][n], ref[n][0][:, r * Lp:(r + 1) * Lp], rtol=1e-10, atol=1e-12), (r, n)
        assert np.allclose(got[r]["lse"], ref["lse"][0][:, r * Hp:(r + 1) * Hp], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("world", [2])
def test_usp_ring_across_ranks_equals_whole_sequence(world):
    import numpy as np
    got = _run_ranks(_ring_worker, world)
    ref, ref_lse = _whole_sequence(1, 256, 2, 32, world, seed=12)
    Lb = 256 // world
    for r in range(world):
        for n in ("o", "dq", "dk", "dv"):
            assert np.allclose(got[r][n], ref[n][:, r * Lb:(r + 1) * Lb], rtol=1e-10, atol=1e-12), (r, n)
        assert np.allclose(got[r]["lse"], ref_lse[:, :, r * Lb:(r + 1) * Lb], rtol=1e-12, atol=1e-12)
