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
    def __init__(self, *, H: int, seq_len_q: int, num_pages: int, page_table_stride: int, qkv_dtype,
                 out_dtype=torch.bfloat16, causal: bool = False, window_left: int = -1, q_descale: float = 1.0,
                 kv_descale: float = 1.0, num_clusters: int = 0, device="cuda"):
        self.H, self.Sq = H, seq_len_q
        self.window_left = window_left
        self.out_dtype = out_dtype
        self.device = torch.device(device)
        self.cfg = _native.make_config(seq_len_q=seq_len_q, num_pages=num_pages, page_table_stride=page_table_stride,
                                       qkv_dtype=qkv_dtype, out_dtype=out_dtype, causal=causal, q_descale=q_descale,
                                       ckv_descale=kv_descale, kpe_descale=kv_descale, num_clusters=num_clusters)
        self.workspace = None
        self.split_kv = None

    def plan(self, seq_lens_host):
        sl = torch.as_tensor(seq_lens_host, dtype=torch.int32).cpu()
        self.split_kv, ws_bytes = _native.mla_plan(sl, sl.numel(), self.H, PAGE_SIZE, self.window_left, self.cfg)
        if self.workspace is None or self.workspace.numel() < ws_bytes:
            self.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device)
        return self.split_kv, ws_bytes

    def __call__(self, q_latent, q_rope, ckv, kpe, page_table, seq_lens, scale: float, out=None, lse=None,
                 stream=None, want_lse: bool = True):
        if self.workspace is None:
            raise RuntimeError("call plan(seq_lens) before decoding")
        B = q_latent.shape[0]
        if out is None:
            out = torch.empty((B, self.Sq, self.H, 512), dtype=self.out_dtype, device=q_latent.device)
        if lse is None and want_lse:
            lse = torch.empty((B, self.Sq, self.H), dtype=torch.float32, device=q_latent.device)
        _native.mla_decode(q_latent, q_rope, ckv, kpe, page_table, seq_lens, scale, self.window_left, out, lse,
                           self.workspace, self.cfg, stream)
        return out, lse

    def launches_per_call(self) -> int:
        """Kernels one decode call launches: the split-KV kernel and the reduction."""
        return 2

    def status(self, stream=None) -> int:
        return _native.mla_workspace_status(self.workspace, stream)


def decoder_for(prob, device="cuda", num_clusters: int = 0) -> PagedMlaDecoder:
    """A planned decoder for a workloads.Problem (its physical pool and page table)."""
    w = prob.w
    dt = torch.float8_e4m3fn if w.dtype == "e4m3" else torch.bfloat16
    od = torch.float32 if w.out_dtype == "f32" else torch.bfloat16
    dec = PagedMlaDecoder(H=w.H, seq_len_q=w.Sq, num_pages=prob.pool_pages,
                          page_table_stride=prob.page_table.shape[1], qkv_dtype=dt, out_dtype=od, causal=w.causal,
                          window_left=w.window_left, q_descale=prob.q_descale, kv_descale=prob.ckv_descale,
                          num_clusters=num_clusters, device=device)
    dec.plan(prob.seq_lens)
    return dec
