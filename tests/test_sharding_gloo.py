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


# Decode context parallelism, exercised on CPU ranks: every request's pages are dealt to
# the ranks in turn (logical page j to rank j % world), each rank decodes its own keys, the
# ranks exchange (O, LSE) and the pieces merge with the split-KV combine, in natural log:
# lse = m + ln(sum_r e^(lse_r - m)) and O = sum_r e^(lse_r - lse) O_r.  With Sq = 1 and no
# causal mask a row's softmax does not depend on the order of its keys, so a rank's piece
# is the decode of its keys as a request of their own.

def _dcp_local(p, world, rank):
    from paged_latent_attention_mla_gb300.workloads import PAD_PAGE

    pt, sl = p["page_table"], p["seq_lens"]
    P = p["ckv"].shape[1]
    B = pt.shape[0]
    width = max(1, (pt.shape[1] + world - 1) // world)
    lpt = torch.full((B, width), PAD_PAGE, dtype=torch.int32)
    lsl = torch.zeros(B, dtype=torch.int32)
    for b in range(B):
        K = int(sl[b])
        mine = [j for j in range((K + P - 1) // P) if j % world == rank]
        for i, j in enumerate(mine):
            lpt[b, i] = pt[b, j]
        lsl[b] = sum(min(P, K - j * P) for j in mine)  # a partial page is the request's last
    return dict(p, page_table=lpt, seq_lens=lsl)


def _merge(O_parts, L_parts):
    L = np.stack(L_parts)  # [world, rows]
    m = np.max(L, axis=0)
    m0 = np.where(np.isfinite(m), m, 0.0)
    s = np.sum(np.exp(L - m0), axis=0)
    lse = np.where(s > 0, m0 + np.log(np.where(s > 0, s, 1.0)), -np.inf)
    w = np.where(np.isfinite(L), np.exp(L - np.where(np.isfinite(lse), lse, 0.0)), 0.0)
    return np.einsum("rn,rnd->nd", w, np.stack(O_parts)), lse


def _dcp_worker(rank, world, port, q):
    import torch.distributed as dist

    import oracle
    from paged_latent_attention_mla_gb300 import workloads as wl

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # lengths with a request on one page only, so some ranks hold no key of it
        prob = wl.make_problem("tiny", H=3, seq_lens=[100, 257, 64, 1, 300, 129], B=6)
        p = prob.host_inputs()
        O, L = oracle.decode(_dcp_local(p, world, rank), threads=1)
        mine = torch.from_numpy(np.concatenate([O.reshape(-1), L.reshape(-1)]))
        outs = [torch.zeros_like(mine) for _ in range(world)]
        dist.all_gather(outs, mine)
        if rank == 0:
            n = O.shape[0]
            parts = [o.numpy() for o in outs]
            Om, Lm = _merge([v[: n * 512].reshape(n, 512) for v in parts], [v[n * 512:] for v in parts])
            Of, Lf = oracle.decode(p, threads=1)
            fin = np.isfinite(Lf)
            ok = (np.array_equal(np.isfinite(Lm), fin) and np.all(Om[~fin] == 0)
                  and np.abs(Lm[fin] - Lf[fin]).max() <= 1e-12
                  and np.abs(Om - Of).max() <= 1e-12 * max(np.abs(Of).max(), 1e-300))
            q.put(bool(ok))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_dcp_merge_over_cpu_ranks_equals_whole_decode(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dcp_worker, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=240)
    assert all(pr.exitcode == 0 for pr in procs)
    assert q.get(timeout=5)
