"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each test ties the oracle to something independent of its own code: a library
routine on densified inputs, a closed form, an invariant of softmax attention,
or an exhaustive table.  A plausible slip in the oracle (a dropped rope term, a
wrong page index, a transposed operand, an off-by-one in the causal or window
edge, a wrong log base) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_latent_attention_mla_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALE = 1.0 / 24.0  # 1/sqrt(512 + 64)


def contiguous_problem(lens, H, Sq, seed, dtype=torch.bfloat16, page_size=64, causal=False, window_left=-1,
                       descales=(1.0, 1.0, 1.0)):
    """Requests whose pages are consecutive in the pool: the dense view is a plain reshape."""
    g = torch.Generator().manual_seed(seed)
    n_pages = [max(1, (k + page_size - 1) // page_size) for k in lens]
    total = sum(n_pages)
    ckv = torch.randn((total, page_size, 512), generator=g)
    kpe = torch.randn((total, page_size, 64), generator=g)
    ql = torch.randn((len(lens), Sq, H, 512), generator=g)
    qr = torch.randn((len(lens), Sq, H, 64), generator=g)
    if dtype == torch.float8_e4m3fn:
        ckv, kpe, ql, qr = ((t * 8).clamp(-448, 448).to(dtype) for t in (ckv, kpe, ql, qr))
    else:
        ckv, kpe, ql, qr = (t.to(dtype) for t in (ckv, kpe, ql, qr))
    width = max(n_pages)
    table = torch.full((len(lens), width), wl.PAD_PAGE, dtype=torch.int32)
    starts, s = [], 0
    for b, n in enumerate(n_pages):
        table[b, :n] = torch.arange(s, s + n, dtype=torch.int32)
        starts.append(s)
        s += n
    p = dict(q_latent=ql, q_rope=qr, ckv=ckv, kpe=kpe, page_table=table,
             seq_lens=torch.tensor(lens, dtype=torch.int32), scale=SCALE, causal=causal,
             window_left=window_left, q_descale=descales[0], ckv_descale=descales[1], kpe_descale=descales[2])
    return p, starts


def dense_reference(p, starts, page_size=64):
    """Library SDPA (fp64, CPU) on the contiguous pool, with the textbook position mask.

    Query token t of a request with K keys sits at absolute position i = K - Sq + t.
    causal: it sees keys j <= i.  window W >= 0: it sees keys j >= i - W.
    """
    qd, cd, kd = p.get("q_descale", 1.0), p.get("ckv_descale", 1.0), p.get("kpe_descale", 1.0)
    ql, qr = p["q_latent"].double() * qd, p["q_rope"].double() * qd
    B, Sq, H, _ = ql.shape
    ckv = p["ckv"].double().reshape(-1, 512) * cd
    kpe = p["kpe"].double().reshape(-1, 64) * kd
    outs, lses = [], []
    for b in range(B):
        K = int(p["seq_lens"][b])
        base = starts[b] * page_size
        c, k = ckv[base:base + K], kpe[base:base + K]
        q = torch.cat([ql[b], qr[b]], dim=-1)  # [Sq, H, 576]
        keys = torch.cat([c, k], dim=-1)  # [K, 576]
        pos = torch.arange(Sq).unsqueeze(1) + (K - Sq)  # [Sq, 1]
        j = torch.arange(K).unsqueeze(0)  # [1, K]
        mask = torch.ones((Sq, K), dtype=torch.bool)
        if p["causal"]:
            mask &= j <= pos
        if p["window_left"] >= 0:
            mask &= j >= pos - p["window_left"]
        qh = q.permute(1, 0, 2)  # [H, Sq, 576]
        o = torch.nn.functional.scaled_dot_product_attention(
            qh.unsqueeze(0), keys.unsqueeze(0).unsqueeze(0), c.unsqueeze(0).unsqueeze(0),
            attn_mask=mask.unsqueeze(0).unsqueeze(0), scale=p["scale"])[0]  # [H, Sq, 512]
        s = (qh @ keys.T) * p["scale"]
        lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)  # [H, Sq]
        empty = ~mask.any(dim=-1)  # [Sq]
        o[:, empty] = 0.0
        outs.append(o.permute(1, 0, 2))
        lses.append(lse.T)
    return torch.stack(outs).reshape(-1, 512).numpy(), torch.stack(lses).reshape(-1).numpy()


CASES = [
    dict(lens=[100, 257], H=4, Sq=1),
    dict(lens=[1, 64, 65, 130], H=2, Sq=1),
    dict(lens=[70, 200], H=3, Sq=3, causal=True),
    dict(lens=[300, 9], H=2, Sq=4, causal=True, window_left=37),
    dict(lens=[150], H=2, Sq=2, causal=False, window_left=20),
    dict(lens=[129, 5], H=2, Sq=1, dtype=torch.float8_e4m3fn),
    dict(lens=[129, 70], H=2, Sq=2, causal=True, dtype=torch.float8_e4m3fn, descales=(0.03125, 0.0625, 0.5)),
    dict(lens=[40, 65], H=2, Sq=1, descales=(0.5, 2.0, 4.0)),
    dict(lens=[100, 257, 16], H=2, Sq=2, causal=True, page_size=16),
    dict(lens=[300, 129], H=2, Sq=3, causal=True, window_left=50, page_size=128),
    dict(lens=[70, 9], H=2, Sq=1, page_size=8),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items() if k != "dtype"))
def test_matches_dense_sdpa(case):
    case = dict(case)
    p, starts = contiguous_problem(seed=11, **case)
    O, L = oracle.decode(p)
    Oref, Lref = dense_reference(p, starts, page_size=case.get("page_size", 64))
    fin = np.isfinite(Lref)
    assert np.abs(O - Oref).max() <= 1e-12 * max(1.0, np.abs(Oref).max())
    assert np.all(np.abs(L[fin] - Lref[fin]) <= 1e-12 * np.maximum(1.0, np.abs(Lref[fin])))
    assert np.all(L[~fin] == -np.inf)


def test_page_permutation_is_bit_identical():
    """A consistent relabelling of physical pages (pool and table together) changes nothing."""
    p, _ = contiguous_problem([100, 257, 33], H=2, Sq=2, seed=5, causal=True)
    n = p["ckv"].shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n)
    q = dict(p)
    q["ckv"], q["kpe"] = p["ckv"][perm], p["kpe"][perm]  # new page i holds old page perm[i]
    pt = p["page_table"].clone()
    valid = pt != wl.PAD_PAGE
    pt[valid] = inv[pt[valid].long()].to(torch.int32)
    q["page_table"] = pt
    O1, L1 = oracle.decode(p)
    O2, L2 = oracle.decode(q)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_single_visible_key_returns_its_value_row():
    """window_left = 0 with causal Sq = 1: the row sees only its own key, so O = c_{K-1}, LSE = s."""
    p, starts = contiguous_problem([77, 128, 1], H=3, Sq=1, seed=9, causal=True, window_left=0)
    O, L = oracle.decode(p)
    ckv = p["ckv"].double().reshape(-1, 512)
    kpe = p["kpe"].double().reshape(-1, 64)
    for b, K in enumerate([77, 128, 1]):
        row = starts[b] * 64 + K - 1
        for h in range(3):
            r = b * 3 + h
            assert np.array_equal(O[r], ckv[row].numpy())
            s = SCALE * (float(p["q_latent"][b, 0, h].double() @ ckv[row]) + float(p["q_rope"][b, 0, h].double() @ kpe[row]))
            assert abs(L[r] - s) <= 1e-12 * max(1.0, abs(s))


def test_equal_scores_give_mean_of_values():
    """q_latent = 0 and identical kpe rows: every score equals s, so O = mean(c), LSE = s + ln n."""
    lens = [50, 200]
    p, starts = contiguous_problem(lens, H=2, Sq=1, seed=21)
    p["q_latent"] = torch.zeros_like(p["q_latent"])
    kpe = p["kpe"].clone()
    kpe[:] = kpe[0, 0]
    p["kpe"] = kpe
    O, L = oracle.decode(p)
    ckv = p["ckv"].double().reshape(-1, 512).numpy()
    k0 = p["kpe"][0, 0].double()
    for b, K in enumerate(lens):
        mean = ckv[starts[b] * 64: starts[b] * 64 + K].mean(axis=0)
        for h in range(2):
            s = SCALE * float(p["q_rope"][b, 0, h].double() @ k0)
            assert np.allclose(O[b * 2 + h], mean, rtol=0, atol=1e-12)
            assert abs(L[b * 2 + h] - (s + math.log(K))) <= 1e-12 * max(1.0, abs(s))
    # and with q = 0 entirely: LSE = ln(#visible)
    p["q_rope"] = torch.zeros_like(p["q_rope"])
    _, L0 = oracle.decode(p)
    assert np.allclose(L0, np.repeat(np.log(lens), 2), rtol=0, atol=1e-12)


@pytest.mark.parametrize("tile_n", [64, 128])
def test_split_recombination_equals_unsplit(tile_n):
    prob = wl.make_problem("tiny", H=2, seq_lens=[100, 257, 1000, 0], B=4)
    p = prob.host_inputs()
    O, L = oracle.decode(p)
    for split in range(1, 33):
        Os, Ls = oracle.decode_split(p, split, tile_n)
        fin = np.isfinite(L)
        assert np.abs(Os - O).max() <= 1e-12 * np.abs(O).max(), split
        assert np.abs(Ls[fin] - L[fin]).max() <= 1e-12 * np.abs(L[fin]).max(), split
        assert np.array_equal(np.isfinite(Ls), fin)


def test_split_recombination_with_window_and_causal():
    prob = wl.make_problem("window", B=2, Sq=3, H=2, seq_lens=[900, 333], window_left=150)
    p = prob.host_inputs()
    O, L = oracle.decode(p)
    for split in (1, 2, 3, 7, 16, 32):
        Os, Ls = oracle.decode_split(p, split, 128)
        assert np.abs(Os - O).max() <= 1e-12 * np.abs(O).max()
        assert np.abs(Ls - L).max() <= 1e-12 * np.abs(L).max()


def test_window_covering_everything_equals_no_window():
    prob = wl.make_problem("window", B=2, Sq=2, H=2, seq_lens=[300, 70], window_left=5000)
    p = prob.host_inputs()
    q = dict(p, window_left=-1)
    O1, L1 = oracle.decode(p)
    O2, L2 = oracle.decode(q)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_single_query_causal_equals_noncausal():
    prob = wl.make_problem("tiny", H=3)
    p = prob.host_inputs()
    O1, L1 = oracle.decode(dict(p, causal=True))
    O2, L2 = oracle.decode(dict(p, causal=False))
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_constant_score_shift_moves_lse_only():
    """Adding a constant to every score (one rope dim with constant kpe) shifts LSE by it, O unchanged."""
    p, _ = contiguous_problem([90, 260], H=2, Sq=1, seed=4)
    kpe = p["kpe"].clone()
    kpe[..., 0] = 2.0
    qr0 = p["q_rope"].clone()
    qr0[..., 0] = 0.0
    qr1 = qr0.clone()
    qr1[..., 0] = 3.0
    O0, L0 = oracle.decode(dict(p, kpe=kpe, q_rope=qr0))
    O1, L1 = oracle.decode(dict(p, kpe=kpe, q_rope=qr1))
    assert np.allclose(O1, O0, rtol=0, atol=1e-12 * np.abs(O0).max())
    assert np.allclose(L1 - L0, SCALE * 6.0, rtol=0, atol=1e-12)


def test_empty_rows():
    """No visible key (K = 0, or a causal row before the first key): O = 0 and LSE = -inf."""
    p, _ = contiguous_problem([0, 2, 40], H=2, Sq=4, seed=8, causal=True)
    O, L = oracle.decode(p)
    L = L.reshape(3, 4, 2)
    O = O.reshape(3, 4, 2, 512)
    assert np.all(L[0] == -np.inf) and np.all(O[0] == 0)
    # K = 2, Sq = 4: token t sits at position t - 2, so t = 0, 1 see nothing
    assert np.all(L[1, :2] == -np.inf) and np.all(O[1, :2] == 0)
    assert np.all(np.isfinite(L[1, 2:])) and np.all(np.isfinite(L[2]))


def test_visible_range_is_the_position_rule():
    """Exhaustive: [lo, hi) equals {j : j <= i (causal), j >= i - W (window)} with i = K - Sq + t."""
    for K in range(0, 40):
        for Sq in (1, 2, 3, 5):
            for causal in (False, True):
                for W in (-1, 0, 1, 3, 10, 50):
                    for t in range(Sq):
                        lo, hi = oracle.visible_range(K, Sq, t, causal, W)
                        i = K - Sq + t
                        want = [j for j in range(K) if (not causal or j <= i) and (W < 0 or j >= i - W)]
                        got = list(range(lo, hi))
                        assert got == want, (K, Sq, t, causal, W)


def test_visibility_bits_match_position_rule():
    lens = [0, 31, 32, 33, 100]
    bits = oracle.visibility_bits(lens, 3, True, 7, 128)
    for b, K in enumerate(lens):
        for t in range(3):
            i = K - 3 + t
            for j in range(128):
                want = j < K and j <= i and j >= i - 7
                assert bool((int(bits[b, t, j // 32]) >> (j % 32)) & 1) == want


def test_e4m3_decode_all_256_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    for c in range(256):
        v = oracle.e4m3_to_f64(c)
        if math.isnan(ref[c]):
            assert math.isnan(v)
        else:
            assert v == ref[c], c


def test_bf16_decode_codes():
    codes = list(range(0, 65536, 97)) + [0x0000, 0x8000, 0x3F80, 0x0001, 0x7F7F, 0xFF7F]
    ref = torch.tensor(codes, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).to(torch.float64).tolist()
    for c, r in zip(codes, ref):
        v = oracle.bf16_to_f64(c)
        assert (math.isnan(v) and math.isnan(r)) or v == r, hex(c)


def test_gather_matches_contiguous_view():
    p, starts = contiguous_problem([100, 257, 3], H=1, Sq=1, seed=2)
    dense = oracle.gather(p, 300)
    c = p["ckv"].view(torch.int16).reshape(-1, 512).numpy().view(np.uint16)
    k = p["kpe"].view(torch.int16).reshape(-1, 64).numpy().view(np.uint16)
    for b, K in enumerate([100, 257, 3]):
        base = starts[b] * 64
        assert np.array_equal(dense[b, :K, :512], c[base:base + K])
        assert np.array_equal(dense[b, :K, 512:], k[base:base + K])
        assert not dense[b, K:].any()


def test_golden_two_key_example():
    """Hand-worked closed form (tests/golden/two_keys.json): scores 1 and 0 give weights e/(e+1), 1/(e+1)."""
    with open(os.path.join(GOLDEN, "two_keys.json")) as f:
        g = json.load(f)
    ql = torch.zeros((1, 1, 1, 512))
    ql[0, 0, 0, 0] = g["q_latent_0"]
    ckv = torch.zeros((1, 64, 512))
    for j, row in enumerate(g["c_rows"]):
        for d, v in row.items():
            ckv[0, j, int(d)] = v
    p = dict(q_latent=ql.bfloat16(), q_rope=torch.zeros((1, 1, 1, 64)).bfloat16(), ckv=ckv.bfloat16(),
             kpe=torch.zeros((1, 64, 64)).bfloat16(), page_table=torch.zeros((1, 1), dtype=torch.int32),
             seq_lens=torch.tensor([2], dtype=torch.int32), scale=g["scale"], causal=False, window_left=-1)
    O, L = oracle.decode(p)
    e = math.e
    assert abs(L[0] - g["lse"]) <= 1e-15 and abs(g["lse"] - math.log(e + 1)) <= 1e-15
    for d, v in g["o"].items():
        assert abs(O[0, int(d)] - v) <= 1e-15
    assert O[0, 0] == pytest.approx(e / (e + 1), abs=1e-15)
    assert O[0, 1] == pytest.approx((2 * e - 4) / (e + 1), abs=1e-15)


# ---------------------------------------------------------------- context parallelism and local bounds
# Decode context parallelism splits every sequence's keys over ranks (runs of
# cp_interleave_size positions dealt in turn, the kv_balanced_mla kernel page's
# __init__ parameters); each rank attends to its own keys under the bounds of the
# whole sequence (causal_seqs of __call__), and the ranks' (O, LSE) pieces combine
# exactly.  The pin: the merged pieces equal the whole decode, so a wrong global
# position, a wrong bound or a wrong combine fails.

DCP_CASES = [
    dict(world=2, interleave=1, lens=[100, 257, 1, 0, 64], Sq=1, causal=False, window=-1),
    dict(world=2, interleave=1, lens=[300, 70, 5], Sq=3, causal=True, window=-1),
    dict(world=3, interleave=2, lens=[300, 129, 2], Sq=4, causal=True, window=37),
    dict(world=2, interleave=64, lens=[700, 64, 65], Sq=2, causal=True, window=-1),
    dict(world=4, interleave=5, lens=[333, 17], Sq=2, causal=False, window=60),
]


@pytest.mark.parametrize("case", DCP_CASES, ids=lambda c: f"w{c['world']}i{c['interleave']}sq{c['Sq']}")
def test_context_parallel_shares_merge_to_the_whole_decode(case):
    prob = wl.make_problem("tiny", H=3, B=len(case["lens"]), seq_lens=case["lens"], Sq=case["Sq"],
                           causal=case["causal"], window_left=case["window"], seed=17)
    whole_O, whole_L = oracle.decode(prob.host_inputs())
    Os, Ls = [], []
    for r in range(case["world"]):
        sh = wl.dcp_shard(prob, case["world"], r, case["interleave"])
        O, L = oracle.decode_ex(sh.host_inputs(), cp_world=case["world"], cp_rank=r, cp_interleave=case["interleave"],
                                global_seq_lens=sh.extra["global_seq_lens"])
        Os.append(O)
        Ls.append(L)
    Om, Lm = oracle.merge(Os, Ls)
    fin = np.isfinite(whole_L)
    assert np.array_equal(np.isfinite(Lm), fin)
    assert np.all(Om[~fin] == 0)
    assert np.abs(Om - whole_O).max() <= 1e-12 * max(1.0, np.abs(whole_O).max())
    assert np.abs(Lm[fin] - whole_L[fin]).max() <= 1e-12 * max(1.0, np.abs(whole_L[fin]).max())


def test_one_rank_context_parallel_is_the_plain_decode():
    prob = wl.make_problem("tiny", H=2, B=3, seq_lens=[90, 300, 3], Sq=3, causal=True, window_left=40, seed=3)
    p = prob.host_inputs()
    O1, L1 = oracle.decode(p)
    O2, L2 = oracle.decode_ex(p, cp_world=1)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_merge_of_one_piece_and_an_empty_piece():
    g = np.random.default_rng(1)
    O = g.standard_normal((5, 512))
    L = g.standard_normal(5)
    Om, Lm = oracle.merge([O, np.zeros((5, 512))], [L, np.full(5, -np.inf)])
    assert np.array_equal(Lm, L) and np.abs(Om - O).max() <= 1e-15
    Om, Lm = oracle.merge([np.zeros((2, 512))] * 3, [np.full(2, -np.inf)] * 3)
    assert np.all(Lm == -np.inf) and not Om.any()


def dense_prefix_reference(p, starts, lvl, page_size=64):
    """Library SDPA (fp64) with an explicit per-token prefix mask j < lvl[b, t] (and the window)."""
    ql, qr = p["q_latent"].double(), p["q_rope"].double()
    B, Sq, H, _ = ql.shape
    ckv = p["ckv"].double().reshape(-1, 512)
    kpe = p["kpe"].double().reshape(-1, 64)
    outs, lses = [], []
    for b in range(B):
        K = int(p["seq_lens"][b])
        base = starts[b] * page_size
        c, k = ckv[base:base + K], kpe[base:base + K]
        q = torch.cat([ql[b], qr[b]], dim=-1).permute(1, 0, 2)  # [H, Sq, 576]
        keys = torch.cat([c, k], dim=-1)
        j = torch.arange(K).unsqueeze(0)
        mask = j < torch.as_tensor(lvl[b]).reshape(Sq, 1)
        if p["window_left"] >= 0:
            pos = torch.arange(Sq).unsqueeze(1) + (K - Sq)
            mask &= j >= pos - p["window_left"]
        s = (q @ keys.T) * p["scale"]
        sm = s.masked_fill(~mask, -math.inf)
        lse = torch.logsumexp(sm, dim=-1)
        w = torch.where(mask, torch.exp(sm - torch.where(torch.isfinite(lse), lse, 0.0).unsqueeze(-1)), 0.0)
        outs.append((w @ c).permute(1, 0, 2))
        lses.append(lse.T)
    return torch.stack(outs).reshape(-1, 512).numpy(), torch.stack(lses).reshape(-1).numpy()


@pytest.mark.parametrize("window", [-1, 25])
def test_local_visible_lens_match_dense_prefix_mask(window):
    lens = [120, 260, 7]
    p, starts = contiguous_problem(lens, H=2, Sq=3, seed=13, window_left=window)
    lvl = [[0, 50, 120], [260, 3, 200], [7, 7, 1]]
    O, L = oracle.decode_ex(p, local_visible_lens=lvl)
    Oref, Lref = dense_prefix_reference(p, starts, lvl)
    fin = np.isfinite(Lref)
    assert np.array_equal(np.isfinite(L), fin)
    assert np.all(O[~fin] == 0)
    assert np.abs(O - Oref).max() <= 1e-12 * max(1.0, np.abs(Oref).max())
    assert np.abs(L[fin] - Lref[fin]).max() <= 1e-12 * max(1.0, np.abs(Lref[fin]).max())


def test_local_visible_lens_at_the_causal_bound_equal_causal():
    lens = [90, 300, 3]
    prob = wl.make_problem("tiny", H=2, B=3, seq_lens=lens, Sq=3, causal=True, seed=6)
    p = prob.host_inputs()
    lvl = [[K - (3 - 1 - t) for t in range(3)] for K in lens]
    O1, L1 = oracle.decode(p)
    O2, L2 = oracle.decode_ex(dict(p, causal=False), local_visible_lens=lvl)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_visibility_bits_ex_plain_equals_position_rule():
    lens = [0, 31, 32, 33, 100]
    for Sq, causal, W in ((1, False, -1), (3, True, 7), (2, False, 5)):
        assert np.array_equal(oracle.visibility_bits_ex(lens, Sq, causal, W, 128),
                              oracle.visibility_bits(lens, Sq, causal, W, 128))


@pytest.mark.parametrize("world,inter", [(2, 1), (3, 4), (4, 64)])
def test_visibility_bits_ex_ranks_partition_the_global_bits(world, inter):
    """Each rank's local bits, mapped to the positions it owns, are disjoint and together
    equal the whole sequence's position-rule bits."""
    glens = [0, 5, 130, 333]
    Sq, causal, W, max_k = 3, True, 40, 400
    whole = oracle.visibility_bits(glens, Sq, causal, W, max_k)
    got = np.zeros_like(whole)
    for r in range(world):
        owned = [[j for j in range(K) if wl.dcp_owner(j, world, inter) == r] for K in glens]
        bits = oracle.visibility_bits_ex([len(o) for o in owned], Sq, causal, W, max_k, cp_world=world, cp_rank=r,
                                         cp_interleave=inter, global_seq_lens=glens)
        for b, o in enumerate(owned):
            for t in range(Sq):
                for l, g in enumerate(o):
                    if (int(bits[b, t, l // 32]) >> (l % 32)) & 1:
                        assert not (int(got[b, t, g // 32]) >> (g % 32)) & 1
                        got[b, t, g // 32] |= np.uint32(1 << (g % 32))
    assert np.array_equal(got, whole)
