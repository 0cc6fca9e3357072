"""Seeded synthetic decode workloads (inputs only, none of the method's arithmetic).

Both the CUDA path's tests and the oracle draw their inputs from here, so the two
sides see identical bits.  Everything is drawn on the CPU from a
``torch.Generator`` seeded per workload, then (for the GPU) scattered into a
device page pool.

The five workloads are the decode shapes this library is measured on:

  tiny     B=2,   H=16,  Sq=1, K=[100, 257],        bf16, fp32 output
  uniform  B=64,  H=128, Sq=1, K=4096,              bf16
  varlen   B=128, H=128, Sq=1, K log-uniform [1, 32768] over a 2^18-page pool
  fp8spec  B=32,  H=128, Sq=2 causal, K=16384,      float8 e4m3: one scale for q, one for the key cache
  window   B=8,   H=128, Sq=4 causal, window_left=4096, K=131072, bf16

Cache layout (vLLM paged MLA): ckv [num_pages, page_size, 512], kpe
[num_pages, page_size, 64]; page_table [B, pages_per_request] int32; seq_lens [B]
int32 counts every cached key including the Sq new tokens.  Poison: cache
slots past a request's length, pages no request owns and page-table entries
past ceil(K / page_size) hold NaN / INT32_MAX, so any read of them shows.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D_LATENT = 512
D_ROPE = 64
PAGE_SIZE = 64
PAD_PAGE = 2**31 - 1  # page-table padding: never a valid page id


@dataclass
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    seq_lens: list | None  # fixed lengths, or None for log-uniform draws
    dtype: str = "bf16"  # "bf16" or "e4m3"
    out_dtype: str = "bf16"  # "f32" or "bf16"
    causal: bool = False
    window_left: int = -1
    pool_pages: int | None = None  # physical pool size (None = exactly the pages used)
    table_width: int | None = None  # page-table columns (None = ceil(max K / P))
    max_len: int = 32768  # log-uniform upper bound
    seed: int = 0
    page_size: int = PAGE_SIZE

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(D_LATENT + D_ROPE)


WORKLOADS = {
    "tiny": Workload("tiny", B=2, H=16, Sq=1, seq_lens=[100, 257], out_dtype="f32", pool_pages=16,
                     table_width=8, seed=20261),
    "uniform": Workload("uniform", B=64, H=128, Sq=1, seq_lens=[4096] * 64, seed=20262),
    "varlen": Workload("varlen", B=128, H=128, Sq=1, seq_lens=None, pool_pages=2**18, table_width=512,
                       seed=20263),
    "fp8spec": Workload("fp8spec", B=32, H=128, Sq=2, seq_lens=[16384] * 32, dtype="e4m3", causal=True,
                        seed=20264),
    "window": Workload("window", B=8, H=128, Sq=4, seq_lens=[131072] * 8, causal=True, window_left=4096,
                       seed=20265),
}


@dataclass
class Problem:
    """One decode batch: compact CPU tensors plus where each page sits in the device pool."""

    w: Workload
    q_latent: torch.Tensor  # [B, Sq, H, 512]
    q_rope: torch.Tensor  # [B, Sq, H, 64]
    ckv: torch.Tensor  # [n_used, P, 512] compact pool (page i = physical page phys_ids[i])
    kpe: torch.Tensor  # [n_used, P, 64]
    page_table: torch.Tensor  # [B, width] int32, compact ids, PAD_PAGE past ceil(K/P)
    seq_lens: torch.Tensor  # [B] int32
    phys_ids: torch.Tensor  # [n_used] int64, distinct ids in [0, pool_pages)
    pool_pages: int
    q_descale: float = 1.0
    ckv_descale: float = 1.0
    kpe_descale: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.w.B

    @property
    def H(self):
        return self.w.H

    @property
    def Sq(self):
        return self.w.Sq

    def common(self) -> dict:
        return dict(scale=self.w.scale, causal=self.w.causal, window_left=self.w.window_left,
                    q_descale=self.q_descale, ckv_descale=self.ckv_descale, kpe_descale=self.kpe_descale)

    def host_inputs(self) -> dict:
        """Compact CPU inputs: the page table indexes the compact pool directly."""
        d = dict(q_latent=self.q_latent, q_rope=self.q_rope, ckv=self.ckv, kpe=self.kpe,
                 page_table=self.page_table, seq_lens=self.seq_lens)
        d.update(self.common())
        return d

    def physical_page_table(self) -> torch.Tensor:
        pt = self.page_table.to(torch.int64)
        valid = pt != PAD_PAGE
        phys = torch.full_like(pt, PAD_PAGE)
        phys[valid] = self.phys_ids[pt[valid]]
        return phys.to(torch.int32)

    def device_inputs(self, device) -> dict:
        """Inputs in device memory: the full physical pool, NaN in every page no request owns."""
        dt = self.ckv.dtype
        P = self.w.page_size
        ckv = _poison_pool((self.pool_pages, P, D_LATENT), dt, device)
        kpe = _poison_pool((self.pool_pages, P, D_ROPE), dt, device)
        idx = self.phys_ids.to(device)
        chunk = 4096
        for s in range(0, idx.numel(), chunk):
            ckv[idx[s:s + chunk]] = self.ckv[s:s + chunk].to(device)
            kpe[idx[s:s + chunk]] = self.kpe[s:s + chunk].to(device)
        d = dict(q_latent=self.q_latent.to(device), q_rope=self.q_rope.to(device), ckv=ckv, kpe=kpe,
                 page_table=self.physical_page_table().to(device), seq_lens=self.seq_lens.to(device))
        d.update(self.common())
        return d


def _nan_bits(dtype):
    return {torch.bfloat16: 0x7FC0, torch.float8_e4m3fn: 0x7F}[dtype]


def _poison_pool(shape, dtype, device):
    if dtype == torch.bfloat16:
        return torch.full(shape, _nan_bits(dtype), dtype=torch.int16, device=device).view(torch.bfloat16)
    return torch.full(shape, _nan_bits(dtype), dtype=torch.uint8, device=device).view(torch.float8_e4m3fn)


def draw_seq_lens(w: Workload, g: torch.Generator) -> list:
    """Fixed lengths, or K = clamp(round(exp(u)), 1, max_len) with u ~ U[0, ln max_len]."""
    if w.seq_lens is not None:
        return list(w.seq_lens)
    u = torch.rand(w.B, generator=g, dtype=torch.float64) * math.log(w.max_len)
    return [int(min(max(round(math.exp(x)), 1), w.max_len)) for x in u.tolist()]


def _normal(shape, g, chunk_rows=2048):
    """N(0,1) float32, drawn in row chunks to bound peak memory."""
    out = torch.empty(shape, dtype=torch.float32)
    flat = out.view(shape[0], -1)
    for s in range(0, shape[0], chunk_rows):
        e = min(s + chunk_rows, shape[0])
        flat[s:e] = torch.randn((e - s, flat.shape[1]), generator=g, dtype=torch.float32)
    return out


def _quantize_e4m3(x: torch.Tensor):
    """Per-tensor scale: descale = amax / 448, stored value = e4m3(x / descale) (round to nearest even)."""
    amax = float(x.abs().max())
    descale = amax / 448.0 if amax > 0 else 1.0
    return (x / descale).to(torch.float8_e4m3fn), descale


def make_problem(w: Workload | str, *, seq_lens=None, seed=None, H=None, B=None, Sq=None, causal=None,
                 window_left=None, dtype=None, out_dtype=None, pool_pages=None, table_width=None,
                 page_size=None) -> Problem:
    """Draw one seeded decode batch.  Keyword overrides build smaller variants for tests."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    over = {k: v for k, v in dict(seq_lens=seq_lens, seed=seed, H=H, B=B, Sq=Sq, causal=causal,
                                   window_left=window_left, dtype=dtype, out_dtype=out_dtype,
                                   pool_pages=pool_pages, table_width=table_width,
                                   page_size=page_size).items() if v is not None}
    if over:
        d = dict(w.__dict__)
        d.update(over)
        if "seq_lens" in over:
            # new lengths: size the table and the pool for them unless told otherwise
            d["B"] = len(over["seq_lens"])
            d["table_width"] = over.get("table_width")
            d["pool_pages"] = over.get("pool_pages")
        w = Workload(**d)
    g = torch.Generator().manual_seed(w.seed)
    P = w.page_size
    lens = draw_seq_lens(w, g)
    assert len(lens) == w.B
    n_pages = [(k + P - 1) // P for k in lens]
    n_used = sum(n_pages)
    width = w.table_width or max(1, max(n_pages))
    assert width >= max(n_pages), "table too narrow for the longest request"
    pool = w.pool_pages or max(n_used, 1)
    assert pool >= n_used

    ql = _normal((w.B, w.Sq, w.H, D_LATENT), g)
    qr = _normal((w.B, w.Sq, w.H, D_ROPE), g)
    ckv = _normal((max(n_used, 1), P, D_LATENT), g)
    kpe = _normal((max(n_used, 1), P, D_ROPE), g)
    # one global shuffle of compact page ids, then physical placement in the pool
    order = torch.randperm(max(n_used, 1), generator=g)
    phys = torch.randperm(pool, generator=g)[: max(n_used, 1)].to(torch.int64)

    descales = dict(q_descale=1.0, ckv_descale=1.0, kpe_descale=1.0)
    if w.dtype == "e4m3":
        q_all = torch.cat([ql.reshape(-1), qr.reshape(-1)])
        _, qd = _quantize_e4m3(q_all)
        ql8, qr8 = (ql / qd).to(torch.float8_e4m3fn), (qr / qd).to(torch.float8_e4m3fn)
        # one scale for the key cache: latent and rope parts of a key share it
        kv_amax = max(float(ckv.abs().max()), float(kpe.abs().max()))
        kd = kv_amax / 448.0 if kv_amax > 0 else 1.0
        ckv8, kpe8 = (ckv / kd).to(torch.float8_e4m3fn), (kpe / kd).to(torch.float8_e4m3fn)
        ql, qr, ckv, kpe = ql8, qr8, ckv8, kpe8
        descales = dict(q_descale=qd, ckv_descale=kd, kpe_descale=kd)
    else:
        ql, qr, ckv, kpe = (t.to(torch.bfloat16) for t in (ql, qr, ckv, kpe))

    table = torch.full((w.B, width), PAD_PAGE, dtype=torch.int32)
    cursor = 0
    for b, np_b in enumerate(n_pages):
        table[b, :np_b] = order[cursor:cursor + np_b].to(torch.int32)
        cursor += np_b
    # NaN in the cache slots past each request's length (the tail of its last page)
    nan = _nan_bits(ckv.dtype)
    ckv_bits = ckv.view(torch.int16 if ckv.dtype == torch.bfloat16 else torch.uint8)
    kpe_bits = kpe.view(torch.int16 if kpe.dtype == torch.bfloat16 else torch.uint8)
    for b, k in enumerate(lens):
        if k % P and k > 0:
            last = int(table[b, (k - 1) // P])
            ckv_bits[last, k % P:] = nan
            kpe_bits[last, k % P:] = nan
    if n_used == 0:
        ckv_bits.fill_(nan)
        kpe_bits.fill_(nan)
    return Problem(w=w, q_latent=ql, q_rope=qr, ckv=ckv, kpe=kpe, page_table=table,
                   seq_lens=torch.tensor(lens, dtype=torch.int32), phys_ids=phys, pool_pages=pool, **descales)


def sample_rows(prob: Problem, n: int, seed: int = 7) -> list:
    """Flat row ids (b*Sq + t)*H + h for sampled checks: both ends plus seeded picks."""
    B, Sq, H = prob.B, prob.Sq, prob.H
    total = B * Sq * H
    g = torch.Generator().manual_seed(seed)
    lens = prob.seq_lens.tolist()
    picks = {0, total - 1}
    bmax, bmin = max(range(B), key=lambda b: lens[b]), min(range(B), key=lambda b: lens[b])
    for b in (bmax, bmin):
        for t in (0, Sq - 1):
            picks.add((b * Sq + t) * H + (H - 1))
            picks.add((b * Sq + t) * H)
    extra = torch.randint(0, total, (max(0, n - len(picks)),), generator=g).tolist()
    picks.update(extra)
    return sorted(picks)


def dcp_owner(j: int, world: int, interleave: int) -> int:
    """Rank holding key position j when positions are dealt in runs of `interleave` to the ranks in turn."""
    return (j // interleave) % world


def dcp_shard(prob: Problem, world: int, rank: int, interleave: int = 1, seed: int = 0) -> Problem:
    """One rank's share of a batch under decode context parallelism (inputs only).

    The rank holds the keys whose positions it owns (dcp_owner), in position order,
    packed into its own pages behind its own page table; seq_lens counts them and
    extra["global_seq_lens"] keeps the whole sequences' lengths.  Queries are the
    same on every rank.  Cache slots past each local length are NaN poison.
    """
    P = prob.w.page_size
    nan = _nan_bits(prob.ckv.dtype)
    ibits = torch.int16 if prob.ckv.dtype == torch.bfloat16 else torch.uint8
    src_c, src_k = prob.ckv.view(ibits).reshape(-1, D_LATENT), prob.kpe.view(ibits).reshape(-1, D_ROPE)
    lens = prob.seq_lens.tolist()
    local_rows, local_lens = [], []
    for b, K in enumerate(lens):
        mine = [j for j in range(K) if dcp_owner(j, world, interleave) == rank]
        rows = [int(prob.page_table[b, j // P]) * P + j % P for j in mine]
        local_rows.append(rows)
        local_lens.append(len(rows))
    n_pages = [(k + P - 1) // P for k in local_lens]
    n_used = max(1, sum(n_pages))
    width = max(1, max(n_pages))
    ckv = torch.full((n_used * P, D_LATENT), nan, dtype=ibits)
    kpe = torch.full((n_used * P, D_ROPE), nan, dtype=ibits)
    table = torch.full((prob.B, width), PAD_PAGE, dtype=torch.int32)
    cursor = 0
    for b, rows in enumerate(local_rows):
        if rows:
            idx = torch.tensor(rows, dtype=torch.int64)
            ckv[cursor * P: cursor * P + len(rows)] = src_c[idx]
            kpe[cursor * P: cursor * P + len(rows)] = src_k[idx]
        table[b, :n_pages[b]] = torch.arange(cursor, cursor + n_pages[b], dtype=torch.int32)
        cursor += n_pages[b]
    dt = prob.ckv.dtype
    ckv = ckv.view(dt).reshape(n_used, P, D_LATENT)
    kpe = kpe.view(dt).reshape(n_used, P, D_ROPE)
    g = torch.Generator().manual_seed(seed * 7919 + rank)
    phys = torch.randperm(n_used, generator=g).to(torch.int64)
    return Problem(w=prob.w, q_latent=prob.q_latent, q_rope=prob.q_rope, ckv=ckv, kpe=kpe, page_table=table,
                   seq_lens=torch.tensor(local_lens, dtype=torch.int32), phys_ids=phys, pool_pages=n_used,
                   q_descale=prob.q_descale, ckv_descale=prob.ckv_descale, kpe_descale=prob.kpe_descale,
                   extra={"global_seq_lens": prob.seq_lens.clone(), "cp": (world, rank, interleave)})
