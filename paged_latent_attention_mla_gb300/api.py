"""User-facing wrapper: plan once, keep the workspace, decode many times.

    dec = PagedMlaDecoder(H=128, seq_len_q=1, num_pages=..., page_table_stride=...,
                          qkv_dtype=torch.bfloat16)
    dec.plan(seq_lens_host)                  # sizes (and allocates) the workspace
    out, lse = dec(q_latent, q_rope, ckv, kpe, page_table, seq_lens_dev, scale)

Planning and decoding are the C-ABI calls mla_plan / mla_decode; torch only
provides the device memory.
"""

from __future__ import annotations

import torch

from . import _native

PAGE_SIZE = 64


class PagedMlaDecoder:
    """Plan once, keep the workspace, decode many times.

    Context parallelism: give cp_world / cp_rank / cp_interleave here and each call's
    global_seq_lens; combine the ranks' outputs with merge_ranks (sharding.py holds the
    exchange).  local_visible_lens, when given to a call, bounds each query token's keys.
    Rows cut into several pieces are combined by the reduction kernel; combine_in_kernel=True
    has the split-KV kernel combine them instead (the last piece of a row to finish does it).
    """

    def __init__(self, *, H: int, seq_len_q: int, num_pages: int, page_table_stride: int, qkv_dtype,
                 out_dtype=torch.bfloat16, causal: bool = False, window_left: int = -1, q_descale: float = 1.0,
                 kv_descale: float = 1.0, num_clusters: int = 0, page_size: int = PAGE_SIZE, cp_world: int = 1,
                 cp_rank: int = 0, cp_interleave: int = 1, partial_fp16=None, reducer_d_tiles: int = 0,
                 use_pdl: bool = True, combine_in_kernel: bool = False, device="cuda"):
        # fp16 partials (scaled per row and half of the dims, so any value fits) unless the
        # output is fp32, whose precision the fp32 partials keep
        if partial_fp16 is None:
            partial_fp16 = out_dtype != torch.float32
        self.H, self.Sq = H, seq_len_q
        self.window_left = window_left
        self.out_dtype = out_dtype
        self.page_size = page_size
        self.device = torch.device(device)
        self.cfg = _native.make_config(seq_len_q=seq_len_q, num_pages=num_pages, page_table_stride=page_table_stride,
                                       qkv_dtype=qkv_dtype, out_dtype=out_dtype, causal=causal, q_descale=q_descale,
                                       ckv_descale=kv_descale, kpe_descale=kv_descale, num_clusters=num_clusters,
                                       cp_world=cp_world, cp_rank=cp_rank, cp_interleave=cp_interleave,
                                       partial_fp16=partial_fp16, reducer_d_tiles=reducer_d_tiles, use_pdl=use_pdl,
                                       combine_in_kernel=combine_in_kernel)
        self.workspace = None
        self.split_kv = None

    def plan(self, seq_lens_host):
        sl = torch.as_tensor(seq_lens_host, dtype=torch.int32).cpu()
        self.split_kv, ws_bytes = _native.mla_plan(sl, sl.numel(), self.H, self.page_size, self.window_left, self.cfg)
        if self.workspace is None or self.workspace.numel() < ws_bytes:
            # zeroed once: the rows' arrival counters start at zero (later calls need no clearing)
            self.workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=self.device)
        return self.split_kv, ws_bytes

    def __call__(self, q_latent, q_rope, ckv, kpe, page_table, seq_lens, scale: float, out=None, lse=None,
                 stream=None, want_lse: bool = True, global_seq_lens=None, local_visible_lens=None):
        if self.workspace is None:
            raise RuntimeError("call plan(seq_lens) before decoding")
        B = q_latent.shape[0]
        if out is None:
            out = torch.empty((B, self.Sq, self.H, 512), dtype=self.out_dtype, device=q_latent.device)
        if lse is None and want_lse:
            lse = torch.empty((B, self.Sq, self.H), dtype=torch.float32, device=q_latent.device)
        _native.set_call_inputs(self.cfg, global_seq_lens, local_visible_lens)
        try:
            _native.mla_decode(q_latent, q_rope, ckv, kpe, page_table, seq_lens, scale, self.window_left, out, lse,
                               self.workspace, self.cfg, stream)
        finally:
            _native.set_call_inputs(self.cfg)
        return out, lse

    def launches_per_call(self) -> int:
        """Kernels one decode call launches: the split-KV kernel, and the reduction kernel
        unless the split-KV kernel combines the rows itself (combine_in_kernel)."""
        return 1 if self.cfg.combine_in_kernel else 2

    def status(self, stream=None) -> int:
        return _native.mla_workspace_status(self.workspace, stream)


def merge_ranks(o_parts, lse_parts, out=None, lse=None, stream=None):
    """The context-parallel merge (mla_merge) of gathered shares: o_parts [world, B, Sq, H, 512],
    lse_parts [world, B, Sq, H]; returns (out [B, Sq, H, 512], lse [B, Sq, H])."""
    if out is None:
        out = torch.empty(o_parts.shape[1:], dtype=o_parts.dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    _native.mla_merge(o_parts.contiguous(), lse_parts.contiguous(), out, lse, stream)
    return out, lse


def decoder_for(prob, device="cuda", num_clusters: int = 0, out_dtype=None, **options) -> PagedMlaDecoder:
    """A planned decoder for a workloads.Problem (its physical pool and page table); a
    context-parallel shard (workloads.dcp_shard) gets its rank's settings."""
    w = prob.w
    dt = torch.float8_e4m3fn if w.dtype == "e4m3" else torch.bfloat16
    od = out_dtype or (torch.float32 if w.out_dtype == "f32" else torch.bfloat16)
    if "cp" in prob.extra:
        world, rank, inter = prob.extra["cp"]
        options = dict(cp_world=world, cp_rank=rank, cp_interleave=inter, **options)
    dec = PagedMlaDecoder(H=w.H, seq_len_q=w.Sq, num_pages=prob.pool_pages,
                          page_table_stride=prob.page_table.shape[1], qkv_dtype=dt, out_dtype=od, causal=w.causal,
                          window_left=w.window_left, q_descale=prob.q_descale, kv_descale=prob.ckv_descale,
                          num_clusters=num_clusters, page_size=w.page_size, device=device, **options)
    dec.plan(prob.seq_lens)
    return dec
