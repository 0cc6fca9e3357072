"""Multi-rank path on CPU: world size 2 over gloo.  Each rank decodes its own
request shard with the oracle; gathered, the shards equal the whole batch, and
max_over_ranks reduces timings across ranks."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from paged_latent_attention_mla_gb300.sharding import max_over_ranks, rank_seed, shard_rows


def test_shard_rows_partition():
    for B in (1, 2, 7, 64, 129):
        for world in (1, 2, 3, 8):
            spans = [shard_rows(B, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            sizes = [e - s for s, e in spans]
            assert max(sizes) - min(sizes) <= 1
    assert len({rank_seed(5, r) for r in range(8)}) == 8


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import oracle
    from paged_latent_attention_mla_gb300 import workloads as wl

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        prob = wl.make_problem("tiny", H=2, seq_lens=[100, 257, 64, 1, 300], B=5)
        p = prob.host_inputs()
        s, e = shard_rows(prob.B, world, rank)
        shard = dict(p, q_latent=p["q_latent"][s:e], q_rope=p["q_rope"][s:e], page_table=p["page_table"][s:e],
                     seq_lens=p["seq_lens"][s:e])
        O, L = oracle.decode(shard, threads=1)
        t = torch.from_numpy(np.concatenate([O.reshape(-1), L.reshape(-1)]))
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, torch.tensor([t.numel()], dtype=torch.int64))
        m = max(int(x) for x in sizes)
        buf = torch.zeros(m, dtype=torch.float64)
        buf[: t.numel()] = t
        outs = [torch.zeros(m, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(outs, buf)
        slow = max_over_ranks(float(rank + 1))
        if rank == 0:
            O_all, L_all = [], []
            for r in range(world):
                s2, e2 = shard_rows(prob.B, world, r)
                rows = (e2 - s2) * prob.Sq * prob.H
                v = outs[r][: rows * 513].numpy()
                O_all.append(v[: rows * 512].reshape(rows, 512))
                L_all.append(v[rows * 512:])
            Of, Lf = oracle.decode(p, threads=1)
            q.put((np.array_equal(np.concatenate(O_all), Of), np.array_equal(np.concatenate(L_all), Lf), slow))
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_equal_whole_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=240)
    assert all(pr.exitcode == 0 for pr in procs)
    same_o, same_l, slow = q.get(timeout=5)
    assert same_o and same_l
    assert slow == 2.0


# Decode context parallelism, exercised on CPU ranks: each rank holds its share of every
# request's keys (workloads.dcp_shard: runs of cp_interleave positions dealt in turn),
# decodes its share under the whole sequence's bounds, and the product's exchange
# (sharding.dcp_exchange, an all-gather) brings the ranks' (O, LSE) shares together in the
# layout mla_merge takes.  The shares come from the oracle here (no GPU) and are combined
# with the oracle's merge; the GPU tests run the CUDA decode and the CUDA merge.

def _dcp_worker(rank, world, interleave, port, q):
    import torch.distributed as dist

    import oracle
    from paged_latent_attention_mla_gb300 import workloads as wl
    from paged_latent_attention_mla_gb300.sharding import dcp_exchange

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # causal query blocks with a window, and requests too short for some ranks to hold a key
        prob = wl.make_problem("tiny", H=3, Sq=3, causal=True, window_left=70, seq_lens=[100, 257, 64, 1, 300, 129],
                               B=6)
        sh = wl.dcp_shard(prob, world, rank, interleave)
        O, L = oracle.decode_ex(sh.host_inputs(), cp_world=world, cp_rank=rank, cp_interleave=interleave,
                                global_seq_lens=sh.extra["global_seq_lens"], threads=1)
        B, Sq, H = prob.B, prob.Sq, prob.H
        out = torch.from_numpy(O).reshape(B, Sq, H, 512)
        lse = torch.from_numpy(L).reshape(B, Sq, H)
        o_parts, lse_parts = dcp_exchange(out, lse)
        ok = tuple(o_parts.shape) == (world, B, Sq, H, 512) and tuple(lse_parts.shape) == (world, B, Sq, H)
        ok = ok and torch.equal(o_parts[rank], out) and torch.equal(lse_parts[rank], lse)
        if rank == 0:
            n = B * Sq * H
            Om, Lm = oracle.merge([o.reshape(n, 512).numpy() for o in o_parts.unbind(0)],
                                  [x.reshape(n).numpy() for x in lse_parts.unbind(0)])
            Of, Lf = oracle.decode(prob.host_inputs(), threads=1)
            fin = np.isfinite(Lf)
            ok = ok and (np.array_equal(np.isfinite(Lm), fin) and np.all(Om[~fin] == 0)
                         and np.abs(Lm[fin] - Lf[fin]).max() <= 1e-12
                         and np.abs(Om - Of).max() <= 1e-12 * max(np.abs(Of).max(), 1e-300))
        q.put((rank, bool(ok)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,interleave", [(2, 1), (3, 4)])
def test_dcp_exchange_over_cpu_ranks_merges_to_whole_decode(world, interleave):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dcp_worker, args=(r, world, interleave, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=240)
    assert all(pr.exitcode == 0 for pr in procs)
    results = dict(q.get(timeout=5) for _ in range(world))
    assert all(results[r] for r in range(world))
