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


def host_plan(lens, Sq, H, causal, window, G, e4m3=False, tile=256):
    """Independent restatement of the batch deal.

    A request's Sq*H (token, head) rows, token-major, form work rows of 128.  A group of
    wb = min(work rows per request, G) clusters takes a request's work rows side by side.
    Work is counted in quarter tiles: each sub-band (wb consecutive work rows of a request)
    costs a piece charge (4 units) plus 4 units per tile of the union of its
    rows' visible keys.  The sub-bands' units end to end are dealt in equal contiguous
    shares to min(G // wb, T // 4) groups; a tile goes to the group whose share holds its
    first unit, and a work row's pieces are the groups owning its tiles.
    Returns (slots, most pieces)."""
    piece = 4

    def keys(K, t):
        hi = K - (Sq - 1 - t) if causal else K
        lo = K - Sq - window + t if window >= 0 else 0
        hi, lo = min(max(hi, 0), K), min(max(lo, 0), K)
        return min(lo, hi), hi

    def span(K, tokens):
        rng = [keys(K, t) for t in tokens]
        rng = [(lo, hi) for lo, hi in rng if hi > lo]
        if not rng:
            return 0, 0
        lo, hi = min(r[0] for r in rng), max(r[1] for r in rng)
        return lo // tile, -(-hi // tile) - lo // tile

    rows_q = Sq * H
    Qb = -(-rows_q // 128)
    wb = min(Qb, G)
    nsub = -(-Qb // wb)
    Gg = max(1, G // wb)

    def tokens_of(i0, i1):
        return range(128 * i0 // H, (min(rows_q, 128 * (i1 + 1)) - 1) // H + 1)

    subs = []  # (b, k, ulo, U)
    for b, K in enumerate(lens):
        for k in range(nsub):
            ulo, U = span(K, tokens_of(k * wb, min(Qb, k * wb + wb) - 1))
            subs.append((b, k, ulo, U))
    starts, T = [], 0
    for _, _, _, U in subs:
        starts.append(T)
        T += piece + 4 * U if U else 0
    Gd = max(1, min(Gg, T // 4))
    bounds = [g * T // Gd for g in range(Gd + 1)]

    def owner(x):  # group whose share [bounds[g], bounds[g+1]) holds unit x
        return max(g for g in range(Gd) if bounds[g] <= x)

    most = 1
    for s, (b, k, ulo, U) in enumerate(subs):
        for i in range(k * wb, min(Qb, k * wb + wb)):
            tlo, n = span(lens[b], tokens_of(i, i))
            if not n:
                continue
            groups = {owner(starts[s] + piece + 4 * (tlo - ulo + t)) for t in range(n)}
            assert groups == set(range(min(groups), max(groups) + 1))  # consecutive groups
            most = max(most, len(groups))
    return (len(subs) + Gg) * wb, most


@pytest.mark.parametrize("lens,Sq,H,causal,window,G", [
    ([4096] * 64, 1, 128, False, -1, 76),
    ([100, 257], 1, 16, False, -1, 76),
    ([16384] * 32, 2, 128, True, -1, 76),
    ([131072] * 8, 4, 128, True, 4096, 76),
    ([1, 2, 3, 5000, 0, 77], 3, 128, True, 100, 5),
    ([300] * 7, 1, 128, False, -1, 1),
    ([900, 40, 3000], 8, 16, True, -1, 76),
    ([700, 5, 1500], 5, 48, True, 200, 76),
    ([2000, 64], 64, 16, True, -1, 3),
])
def test_plan_matches_independent_schedule(lib, lens, Sq, H, causal, window, G):
    stride = max(1, (max(lens) + 63) // 64)
    c = cfg(seq_len_q=Sq, causal=causal, page_table_stride=stride, num_clusters=G)
    split, ws = n.mla_plan(lens, len(lens), H, 64, window, c)
    slots, want_split = host_plan(lens, Sq, H, causal, window, G)
    assert split == want_split
    c8 = cfg(seq_len_q=Sq, causal=causal, page_table_stride=stride, num_clusters=G, qkv_dtype=torch.float8_e4m3fn,
             q_descale=0.5, ckv_descale=0.25, kpe_descale=0.25)
    split8, _ = n.mla_plan(lens, len(lens), H, 64, window, c8)
    assert split8 == host_plan(lens, Sq, H, causal, window, G, e4m3=True)[1]
    assert split == want_split
    # the workspace holds at least the fp32 partials and their LSEs for every slot
    assert ws >= slots * 128 * (512 + 1) * 4
    assert ws % 256 == 0
    c16 = cfg(seq_len_q=Sq, causal=causal, page_table_stride=stride, num_clusters=G, partial_fp16=True)
    _, ws16 = n.mla_plan(lens, len(lens), H, 64, window, c16)
    # fp16: the partials, their LSEs and one power-of-two exponent per row and half of the dims
    assert slots * 128 * (256 + 1 + 2) * 4 <= ws16 < ws


@pytest.mark.parametrize("kw,status", [
    (dict(H=0), n.MLA_ERR_INVALID_ARG),
    (dict(H=129), n.MLA_ERR_UNSUPPORTED),
    (dict(page_size=48), n.MLA_ERR_UNSUPPORTED),  # not a power of two
    (dict(page_size=4), n.MLA_ERR_UNSUPPORTED),  # below one 8-row swizzle group
    (dict(page_size=2048), n.MLA_ERR_UNSUPPORTED),
    (dict(cfg=dict(cp_world=2, cp_rank=2)), n.MLA_ERR_INVALID_ARG),
    (dict(cfg=dict(reducer_d_tiles=3)), n.MLA_ERR_INVALID_ARG),
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
    assert decode_status(ckv=FakeTensor(0x30000, (64, 48, 512))) == n.MLA_ERR_UNSUPPORTED  # page size 48
    # context parallelism needs the whole sequences' lengths
    assert decode_status(cfg=dict(cp_world=2, cp_rank=1)) == n.MLA_ERR_INVALID_ARG
