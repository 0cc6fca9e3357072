"""GPU parity of the decode's wider features through the C ABI, every row against the oracle.

  packed rows      H < 128: consecutive tokens' heads share one M tile (the page's pack_q)
  page sizes       8 ... 1024 keys per page (the page's page_size; TMA boxes per page)
  local bounds     per-token local_visible_lens (the page's __call__)
  context parallel each rank's share of every row (cp_world, cp_rank, cp_interleave_size,
                   causal_seqs), merged on the GPU with mla_merge
  combining        rows cut into pieces combined by the reduction kernel, or in the split-KV
                   kernel by their last piece (combine_in_kernel): fp16 or fp32 partials
                   (partial_fp16), reducer D bands (reducer_d_tiles), programmatic dependent launch

Tolerances as in test_gpu_parity: bf16 max|O - O*| <= 1e-2 max|O*|, |LSE - LSE*| <= 1e-3;
e4m3 5e-2 and 2e-2.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_latent_attention_mla_gb300 import _native as n
from paged_latent_attention_mla_gb300 import build as nbuild
from paged_latent_attention_mla_gb300 import decoder_for, merge_ranks
from paged_latent_attention_mla_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-3), "e4m3": (5e-2, 2e-2)}


@pytest.fixture(scope="module", autouse=True)
def built():
    nbuild.build()
    n.load()


def run(prob, d=None, out_dtype=None, global_seq_lens=None, local_visible_lens=None, **options):
    d = d or prob.device_inputs("cuda")
    dec = decoder_for(prob, out_dtype=out_dtype, **options)
    out, lse = dec(d["q_latent"], d["q_rope"], d["ckv"], d["kpe"], d["page_table"], d["seq_lens"], d["scale"],
                   global_seq_lens=global_seq_lens, local_visible_lens=local_visible_lens)
    torch.cuda.synchronize()
    assert dec.status() == n.MLA_OK
    return out, lse


def host(out, lse):
    return out.float().cpu().reshape(-1, 512).numpy(), lse.cpu().reshape(-1).numpy().astype(np.float64)


def compare(dtype, O, L, Or, Lr):
    tol_o, tol_l = TOL[dtype]
    assert np.isfinite(O).all(), "non-finite output"
    fin = np.isfinite(Lr)
    assert np.array_equal(np.isfinite(L), fin), "LSE finiteness differs (empty rows must give -inf)"
    assert np.all(L[~fin] == -np.inf)
    assert np.all(O[~fin] == 0), "empty rows must be zero"
    scale = max(np.abs(Or).max(), 1e-30)
    err_o = np.abs(O - Or).max()
    err_l = np.abs(L[fin] - Lr[fin]).max() if fin.any() else 0.0
    assert err_o <= tol_o * scale, f"O error {err_o:.3e} > {tol_o} * {scale:.3e}"
    assert err_l <= tol_l, f"LSE error {err_l:.3e} > {tol_l}"


# ---------------------------------------------------------------- packed rows (H < 128)
PACKED = {
    "h16_sq8_causal": dict(H=16, Sq=8, causal=True, seq_lens=[900, 40, 3000, 7]),
    "h48_sq5_window": dict(H=48, Sq=5, causal=True, window_left=200, seq_lens=[700, 5, 1500]),
    "h64_sq4_e4m3": dict(H=64, Sq=4, causal=True, dtype="e4m3", seq_lens=[2000, 300, 9]),
    "h32_sq2_noncausal": dict(H=32, Sq=2, causal=False, seq_lens=[513, 64, 1]),
    "h1_sq64_causal": dict(H=1, Sq=64, causal=True, seq_lens=[100, 63, 64, 3000]),
    "h16_sq64_many_tiles": dict(H=16, Sq=64, causal=True, seq_lens=[5000, 64]),
}


@pytest.mark.parametrize("name", list(PACKED))
def test_packed_rows_all_rows(name):
    prob = wl.make_problem("uniform", seed=101, **PACKED[name])
    O, L = host(*run(prob))
    compare(prob.w.dtype, O, L, *oracle.decode(prob.host_inputs()))


# ---------------------------------------------------------------- page sizes
@pytest.mark.parametrize("P,dtype", [(8, "bf16"), (16, "e4m3"), (32, "bf16"), (128, "bf16"), (256, "e4m3"),
                                     (1024, "bf16")])
def test_page_sizes_all_rows(P, dtype):
    prob = wl.make_problem("uniform", seed=202, H=128, Sq=2, causal=True, dtype=dtype, page_size=P,
                           seq_lens=[1000, 77, 2600, 257, 3])
    O, L = host(*run(prob))
    compare(dtype, O, L, *oracle.decode(prob.host_inputs()))


@pytest.mark.parametrize("P,dtype,clusters", [(8, "bf16", 1), (16, "e4m3", 3), (32, "bf16", 3), (64, "e4m3", 2),
                                              (128, "bf16", 5)])
def test_many_pieces_per_cluster_all_rows(P, dtype, clusters):
    """Few clusters over many short and long rows: every cluster walks many pieces, so the
    load and MMA pipeline crosses piece boundaries (the next piece's K ahead of the last
    piece's V, the page boxes of both pieces held at once) and rows are cut at the shares'
    ends."""
    lens = [1 + (53 * i) % 700 for i in range(24)] + [2300, 0, 64, 65]
    prob = wl.make_problem("uniform", seed=909, H=64, Sq=3, causal=True, dtype=dtype, page_size=P, seq_lens=lens)
    O, L = host(*run(prob, num_clusters=clusters))
    compare(dtype, O, L, *oracle.decode(prob.host_inputs()))


@pytest.mark.parametrize("P,dtype", [(64, "bf16"), (16, "e4m3")])
def test_segment_lists_past_shared_memory_all_rows(P, dtype):
    """600 short rows on 2 clusters: about 300 pieces per cluster, more than the 192 segments
    kept in shared memory (the rest are read from the workspace), one pipeline across all."""
    lens = [1 + (97 * i) % 300 for i in range(600)]
    prob = wl.make_problem("uniform", seed=919, H=128, Sq=1, dtype=dtype, page_size=P, seq_lens=lens)
    O, L = host(*run(prob, num_clusters=2))
    compare(dtype, O, L, *oracle.decode(prob.host_inputs()))


@pytest.mark.parametrize("P,dtype", [(8, "bf16"), (32, "e4m3"), (256, "bf16")])
def test_debug_gather_page_sizes_byte_exact(P, dtype):
    prob = wl.make_problem("uniform", seed=3, H=1, dtype=dtype, page_size=P, seq_lens=[100, 257, 64, 1, 0, 130])
    d = prob.device_inputs("cuda")
    max_k = P * prob.page_table.shape[1] + 5
    es = 2 if dtype == "bf16" else 1
    dense = torch.empty((prob.B, max_k, 576 * es), dtype=torch.uint8, device="cuda")
    cfg = n.make_config(seq_len_q=1, num_pages=prob.pool_pages, page_table_stride=prob.page_table.shape[1],
                        qkv_dtype=d["ckv"].dtype, ckv_descale=prob.ckv_descale, kpe_descale=prob.kpe_descale,
                        q_descale=prob.q_descale)
    n.mla_debug_gather(d["ckv"], d["kpe"], d["page_table"], d["seq_lens"], max_k, dense, cfg)
    torch.cuda.synchronize()
    want = oracle.gather(prob.host_inputs(), max_k)
    got = dense.cpu().numpy().view(want.dtype).reshape(want.shape)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- local bounds
@pytest.mark.parametrize("H,window,dtype", [(128, -1, "bf16"), (16, -1, "bf16"), (128, 300, "e4m3")])
def test_local_visible_lens_all_rows(H, window, dtype):
    lens = [1500, 90, 700, 2]
    Sq = 3
    prob = wl.make_problem("uniform", seed=303, H=H, Sq=Sq, causal=False, window_left=window, dtype=dtype,
                           seq_lens=lens)
    g = torch.Generator().manual_seed(5)
    lvl = torch.stack([torch.randint(0, K + 40, (Sq,), generator=g) for K in lens]).to(torch.int32)
    lvl[1, 0] = 0  # an empty row
    O, L = host(*run(prob, local_visible_lens=lvl.cuda()))
    compare(dtype, O, L, *oracle.decode_ex(prob.host_inputs(), local_visible_lens=lvl))


@pytest.mark.parametrize("dtype,P,clusters,window", [("bf16", 64, 2, -1), ("e4m3", 32, 3, 200), ("bf16", 16, 1, 500)])
def test_local_visible_lens_few_clusters_all_rows(dtype, P, clusters, window):
    """Per-token local bounds with many pieces per cluster (the loop-over-tokens spans)."""
    lens = [1 + (71 * i) % 900 for i in range(16)] + [3000]
    Sq = 4
    prob = wl.make_problem("uniform", seed=313, H=32, Sq=Sq, causal=False, window_left=window, dtype=dtype,
                           page_size=P, seq_lens=lens)
    g = torch.Generator().manual_seed(6)
    lvl = torch.stack([torch.randint(0, K + 40, (Sq,), generator=g) for K in lens]).to(torch.int32)
    O, L = host(*run(prob, num_clusters=clusters, local_visible_lens=lvl.cuda()))
    compare(dtype, O, L, *oracle.decode_ex(prob.host_inputs(), local_visible_lens=lvl))


@pytest.mark.parametrize("dtype,H,Sq,clusters", [("bf16", 128, 4, 3), ("e4m3", 64, 3, 2), ("bf16", 16, 8, 1)])
def test_in_kernel_combine_few_clusters_all_rows(dtype, H, Sq, clusters):
    """The in-kernel combine with many pieces per cluster, bands of clusters (Sq x H > 128)
    and packed rows."""
    lens = [1 + (89 * i) % 1200 for i in range(12)] + [4100, 0]
    prob = wl.make_problem("uniform", seed=323, H=H, Sq=Sq, causal=True, window_left=700, dtype=dtype, seq_lens=lens)
    O, L = host(*run(prob, num_clusters=clusters, combine_in_kernel=True))
    compare(dtype, O, L, *oracle.decode(prob.host_inputs()))


def test_debug_mask_local_visible_lens_bit_exact():
    lens = [0, 1, 31, 33, 257]
    Sq, max_k = 3, 300
    lvl = torch.tensor([[0, 0, 0], [1, 0, 1], [10, 31, 40], [33, 2, 17], [256, 100, 300]], dtype=torch.int32)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    bits = torch.empty((len(lens), Sq, (max_k + 31) // 32), dtype=torch.int32, device="cuda")
    cfg = n.make_config(seq_len_q=Sq, num_pages=1, page_table_stride=8, qkv_dtype=torch.bfloat16)
    lvl_d = lvl.cuda()
    n.set_call_inputs(cfg, local_visible_lens=lvl_d)
    n.mla_debug_mask(sl, 20, max_k, bits, cfg)
    torch.cuda.synchronize()
    want = oracle.visibility_bits_ex(lens, Sq, False, 20, max_k, local_visible_lens=lvl)
    assert np.array_equal(bits.cpu().numpy().view(np.uint32), want)


# ---------------------------------------------------------------- context parallelism
DCP = {
    "w2_i1_sq1": dict(world=2, inter=1, H=128, Sq=1, causal=False, window=-1, lens=[3000, 77, 1, 0, 640]),
    "w2_i64_sq2_causal": dict(world=2, inter=64, H=128, Sq=2, causal=True, window=-1, lens=[2600, 65, 129]),
    "w3_i5_sq4_window": dict(world=3, inter=5, H=128, Sq=4, causal=True, window=300, lens=[4000, 9, 700]),
    "w4_i1_h16_sq3": dict(world=4, inter=1, H=16, Sq=3, causal=True, window=-1, lens=[1000, 4, 2]),
}


@pytest.mark.parametrize("name,clusters,out_dtype",
                         [(k, 0, torch.float32) for k in DCP] +
                         [("w3_i5_sq4_window", 2, torch.float32), ("w2_i64_sq2_causal", 1, torch.float32),
                          ("w2_i64_sq2_causal", 3, torch.bfloat16), ("w4_i1_h16_sq3", 2, torch.bfloat16)])
def test_context_parallel_ranks_and_gpu_merge(name, clusters, out_dtype):
    """Every rank's share against the oracle's share, then the GPU merge against the whole
    decode; fp32 shares (fp32 partials), and bf16 shares (fp16 partials, merged in bf16)."""
    c = DCP[name]
    prob = wl.make_problem("uniform", seed=404, H=c["H"], Sq=c["Sq"], causal=c["causal"], window_left=c["window"],
                           seq_lens=c["lens"])
    outs, lses = [], []
    for r in range(c["world"]):
        sh = wl.dcp_shard(prob, c["world"], r, c["inter"], seed=1)
        gsl = sh.extra["global_seq_lens"]
        out, lse = run(sh, out_dtype=out_dtype, global_seq_lens=gsl.cuda(), num_clusters=clusters)
        # this rank's share against the oracle's share
        O, L = host(out, lse)
        compare("bf16", O, L, *oracle.decode_ex(sh.host_inputs(), cp_world=c["world"], cp_rank=r,
                                                cp_interleave=c["inter"], global_seq_lens=gsl))
        outs.append(out)
        lses.append(lse)
    out, lse = merge_ranks(torch.stack(outs), torch.stack(lses))
    torch.cuda.synchronize()
    O, L = host(out, lse)
    compare("bf16", O, L, *oracle.decode(prob.host_inputs()))


def test_debug_mask_context_parallel_bit_exact():
    glens = [0, 5, 130, 333]
    Sq, max_k, world, inter = 3, 200, 3, 4
    for r in range(world):
        local = [sum(1 for j in range(K) if wl.dcp_owner(j, world, inter) == r) for K in glens]
        sl = torch.tensor(local, dtype=torch.int32, device="cuda")
        bits = torch.empty((len(glens), Sq, (max_k + 31) // 32), dtype=torch.int32, device="cuda")
        cfg = n.make_config(seq_len_q=Sq, num_pages=1, page_table_stride=8, qkv_dtype=torch.bfloat16, causal=True,
                            cp_world=world, cp_rank=r, cp_interleave=inter)
        gd = torch.tensor(glens, dtype=torch.int32, device="cuda")
        n.set_call_inputs(cfg, global_seq_lens=gd)
        n.mla_debug_mask(sl, 40, max_k, bits, cfg)
        torch.cuda.synchronize()
        want = oracle.visibility_bits_ex(local, Sq, True, 40, max_k, cp_world=world, cp_rank=r, cp_interleave=inter,
                                         global_seq_lens=glens)
        assert np.array_equal(bits.cpu().numpy().view(np.uint32), want)


def test_merge_of_empty_and_single_pieces():
    rows = 300
    g = torch.Generator(device="cuda").manual_seed(2)
    o = torch.randn((2, rows, 512), generator=g, device="cuda")
    l = torch.randn((2, rows), generator=g, device="cuda")
    l[1] = -float("inf")  # rank 1 saw nothing: the merge is rank 0's piece
    l[0, :7] = -float("inf")  # rows no rank saw
    out, lse = merge_ranks(o, l)
    torch.cuda.synchronize()
    assert torch.all(lse[:7] == -float("inf")) and torch.all(out[:7] == 0)
    assert torch.allclose(out[7:], o[0, 7:], rtol=1e-6, atol=1e-6)
    assert torch.allclose(lse[7:], l[0, 7:], rtol=0, atol=1e-6)


# ---------------------------------------------------------------- fp16 partials, reducer bands, PDL
@pytest.mark.parametrize("opts", [dict(combine_in_kernel=True, partial_fp16=True),
                                  dict(combine_in_kernel=True, partial_fp16=False),
                                  dict(partial_fp16=True), dict(partial_fp16=True, reducer_d_tiles=1),
                                  dict(reducer_d_tiles=2), dict(reducer_d_tiles=4, use_pdl=True),
                                  dict(partial_fp16=True, use_pdl=True)])
def test_partial_formats_and_reducer_bands(opts):
    prob = wl.make_problem("uniform", seed=505, H=128, Sq=2, causal=True, seq_lens=[5000, 300, 2048, 9, 0])
    O, L = host(*run(prob, num_clusters=40, **opts))
    compare("bf16", O, L, *oracle.decode(prob.host_inputs()))


def test_combine_in_kernel_reuses_one_workspace_across_calls_and_shapes():
    """Rows cut into many pieces, combined by their last piece: one workspace, zeroed once,
    serves repeated calls and plans of other shapes (the arrival counters carry each call's
    tag), and agrees with the separate reduction kernel."""
    p1 = wl.make_problem("uniform", seed=71, H=128, Sq=2, causal=True, seq_lens=[5000, 300, 2048, 9, 0])
    p2 = wl.make_problem("uniform", seed=72, H=64, Sq=3, causal=True, seq_lens=[7000, 1, 4000, 640])
    d1 = decoder_for(p1, num_clusters=40, combine_in_kernel=True)
    d2 = decoder_for(p2, num_clusters=24, combine_in_kernel=True)
    shared = torch.zeros(max(d1.workspace.numel(), d2.workspace.numel()), dtype=torch.uint8, device="cuda")
    d1.workspace = d2.workspace = shared
    ref1, ref2 = oracle.decode(p1.host_inputs()), oracle.decode(p2.host_inputs())
    i1, i2 = p1.device_inputs("cuda"), p2.device_inputs("cuda")
    for prob, dec, d, ref in [(p1, d1, i1, ref1), (p2, d2, i2, ref2), (p1, d1, i1, ref1), (p2, d2, i2, ref2),
                              (p2, d2, i2, ref2)]:
        out, lse = dec(d["q_latent"], d["q_rope"], d["ckv"], d["kpe"], d["page_table"], d["seq_lens"], d["scale"])
        torch.cuda.synchronize()
        assert dec.status() == n.MLA_OK
        compare("bf16", *host(out, lse), *ref)
    o_red, l_red = run(p1, d=i1, num_clusters=40)
    o_fused, l_fused = run(p1, d=i1, num_clusters=40, combine_in_kernel=True)
    assert torch.allclose(o_fused.float(), o_red.float(), rtol=2e-2, atol=2e-3 * o_red.float().abs().max().item())
    fin = torch.isfinite(l_red)
    assert torch.equal(fin, torch.isfinite(l_fused))
    assert torch.allclose(l_fused[fin], l_red[fin], rtol=0, atol=1e-4)


@pytest.mark.parametrize("shift", [20, -30])
def test_fp16_partials_hold_any_value_range(shift):
    """The default fp16 partials with values far outside fp16's range (|O| ~ 2^20, beyond
    65504) and far below it (~2^-30, fp16 subnormal): the per-(row, half) power-of-two scale
    keeps them; rows cut into several pieces.  Scaling the latent cache by 2^shift and the
    latent queries by 2^-shift (both exact in bf16) leaves the scores unchanged."""
    prob = wl.make_problem("uniform", seed=515, H=128, Sq=1, seq_lens=[3000, 900, 17, 2048])
    prob.ckv = prob.ckv * 2.0 ** shift
    prob.q_latent = prob.q_latent * 2.0 ** -shift
    O, L = host(*run(prob, num_clusters=12))
    compare("bf16", O, L, *oracle.decode(prob.host_inputs()))


def test_fp16_partials_e4m3_full_size():
    prob = wl.make_problem("fp8spec")
    O, L = host(*run(prob, partial_fp16=True))
    compare("e4m3", O, L, *oracle.decode(prob.host_inputs()))
