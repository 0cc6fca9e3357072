"""C-ABI library checks that need no GPU: it loads, exports every symbol the
header declares, plans on the host, and rejects bad arguments before launching."""

import ctypes
import os
import re

import pytest
import torch

from paged_latent_attention_mla_gb300 import _native as n
from paged_latent_attention_mla_gb300 import build as nbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    nbuild.build()
    return n.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]*?\b(mla_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_symbols() == sorted(n.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    names = ["MLA_OK", "MLA_ERR_INVALID_ARG", "MLA_ERR_UNSUPPORTED", "MLA_ERR_WORKSPACE_TOO_SMALL", "MLA_ERR_CUDA",
             "MLA_ERR_TIMEOUT"]
    for code, name in enumerate(names):
        assert n.status_string(code) == name


def cfg(**kw):
    base = dict(seq_len_q=1, num_pages=64, page_table_stride=8, qkv_dtype=torch.bfloat16, num_clusters=76)
    base.update(kw)
    return n.make_config(**base)


def host_plan(lens, Sq, causal, window, G, tile=256, piece_cost=1):
    """Independent restatement of the batch deal: each row with visible keys costs piece_cost virtual
    tiles followed by its real tiles; the rows' virtual tiles end to end are dealt in equal contiguous
    shares to min(G, T) clusters; a row's pieces are the clusters whose share meets its real tiles."""
    rows = []
    for K in lens:
        for t in range(Sq):
            hi = K - (Sq - 1 - t) if causal else K
            lo = K - Sq - window + t if window >= 0 else 0
            hi, lo = min(max(hi, 0), K), min(max(lo, 0), K)
            lo = min(lo, hi)
            rows.append(0 if hi <= lo else (hi + tile - 1) // tile - lo // tile)
    cost = [nt + piece_cost if nt else 0 for nt in rows]
    T = sum(cost)
    Ge = max(1, min(G, T))
    shares = [(c * T // Ge, (c + 1) * T // Ge) for c in range(Ge)]
    assert all(e > b for b, e in shares) or T == 0
    parts, start = [], 0
    for nt, ct in zip(rows, cost):
        lo, hi = start + piece_cost, start + piece_cost + nt
        parts.append(sum(1 for b, e in shares if b < hi and lo < e) if nt else 0)
        start += ct
    return len(rows), max([1] + parts)


@pytest.mark.parametrize("lens,Sq,causal,window,G", [
    ([4096] * 64, 1, False, -1, 76),
    ([100, 257], 1, False, -1, 76),
    ([16384] * 32, 2, True, -1, 76),
    ([131072] * 8, 4, True, 4096, 76),
    ([1, 2, 3, 5000, 0, 77], 3, True, 100, 5),
    ([300] * 7, 1, False, -1, 1),
])
def test_plan_matches_independent_schedule(lib, lens, Sq, causal, window, G):
    stride = max(1, (max(lens) + 63) // 64)
    c = cfg(seq_len_q=Sq, causal=causal, page_table_stride=stride, num_clusters=G)
    split, ws = n.mla_plan(lens, len(lens), 128, 64, window, c)
    R, want_split = host_plan(lens, Sq, causal, window, G)
    assert split == want_split
    slots = R + G
    # the workspace holds at least the fp32 partials and their LSEs for every slot
    assert ws >= slots * 128 * (512 + 1) * 4
    assert ws % 256 == 0


@pytest.mark.parametrize("kw,status", [
    (dict(H=0), n.MLA_ERR_INVALID_ARG),
    (dict(H=129), n.MLA_ERR_UNSUPPORTED),
    (dict(page_size=32), n.MLA_ERR_UNSUPPORTED),
    (dict(window_left=-2), n.MLA_ERR_INVALID_ARG),
    (dict(cfg=dict(q_descale=0.5)), n.MLA_ERR_INVALID_ARG),  # bf16 inputs take no scales
    (dict(cfg=dict(qkv_dtype=torch.float8_e4m3fn, ckv_descale=0.5, kpe_descale=0.25)), n.MLA_ERR_UNSUPPORTED),
    (dict(cfg=dict(qkv_dtype=torch.float8_e4m3fn, ckv_descale=float("nan"), kpe_descale=float("nan"))),
     n.MLA_ERR_INVALID_ARG),
    (dict(cfg=dict(seq_len_q=0)), n.MLA_ERR_INVALID_ARG),
    (dict(cfg=dict(seq_len_q=65)), n.MLA_ERR_UNSUPPORTED),
    (dict(cfg=dict(out_dtype=torch.float8_e4m3fn)), n.MLA_ERR_INVALID_ARG),
    (dict(lens=[100, 513]), n.MLA_ERR_INVALID_ARG),  # longer than page_table_stride * page_size
    (dict(lens=[-1, 5]), n.MLA_ERR_INVALID_ARG),
])
def test_plan_rejects_bad_arguments(lib, kw, status):
    args = dict(lens=[100, 257], H=16, page_size=64, window_left=-1, cfg={})
    args.update(kw)
    c = cfg(**args["cfg"])
    with pytest.raises(n.MlaError) as e:
        n.mla_plan(args["lens"], len(args["lens"]), args["H"], args["page_size"], args["window_left"], c)
    assert e.value.status == status


class FakeTensor:
    """Only what the binding reads: a device address and a size; never dereferenced on these paths."""

    def __init__(self, addr, shape=(1,), nbytes=16):
        self.addr, self.shape, self._n = addr, shape, nbytes

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self._n

    def element_size(self):
        return 1


def decode_status(**over):
    B, Sq, H = 2, 1, 16
    a = dict(q_latent=FakeTensor(0x10000, (B, Sq, H, 512)), q_rope=FakeTensor(0x20000),
             ckv=FakeTensor(0x30000, (64, 64, 512)), kpe=FakeTensor(0x40000), pt=FakeTensor(0x50000),
             sl=FakeTensor(0x60000), out=FakeTensor(0x70000), lse=FakeTensor(0x80000),
             ws=FakeTensor(0x100000, nbytes=1 << 30), cfg={})
    a.update(over)
    c = cfg(**a["cfg"])
    try:
        n.mla_decode(a["q_latent"], a["q_rope"], a["ckv"], a["kpe"], a["pt"], a["sl"], 1 / 24, -1, a["out"], a["lse"],
                     a["ws"], c, stream=0)
    except n.MlaError as e:
        return e.status
    return n.MLA_OK


def test_decode_rejects_before_launch(lib):
    assert decode_status(q_latent=FakeTensor(0, (2, 1, 16, 512))) == n.MLA_ERR_INVALID_ARG
    assert decode_status(out=FakeTensor(0x70008)) == n.MLA_ERR_INVALID_ARG  # misaligned
    assert decode_status(ws=FakeTensor(0x100080, nbytes=1 << 30)) == n.MLA_ERR_INVALID_ARG  # workspace not 256-aligned
    assert decode_status(ws=FakeTensor(0x100000, nbytes=1024)) == n.MLA_ERR_WORKSPACE_TOO_SMALL
    assert decode_status(cfg=dict(seq_len_q=0)) == n.MLA_ERR_INVALID_ARG
    assert decode_status(ckv=FakeTensor(0x30000, (64, 32, 512))) == n.MLA_ERR_UNSUPPORTED  # page size 32
