"""mla_decode_noalloc: the decode for callers that cannot allocate device memory.

Callers hosted by a runtime that owns all device memory, or on paths that cannot
take an allocation's implicit synchronization, use this entry point: it keeps its
scratch in a fixed array inside the library.  These tests call it through the C
ABI twice in a row (with different batches, so the second call runs over the
first call's leftovers) and compare each result with mla_decode on a workspace of
its own, at the parity tolerances the other GPU tests use.  A batch too big for
the array is refused before anything launches.

This file is collected last and needs nothing from the other test files, so it
passes alone in a fresh process and after the rest of the suite.
"""

import numpy as np
import pytest
import torch

from paged_latent_attention_mla_gb300 import _native as n
from paged_latent_attention_mla_gb300 import build as nbuild
from paged_latent_attention_mla_gb300 import decoder_for
from paged_latent_attention_mla_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-3), "e4m3": (5e-2, 2e-2)}


@pytest.fixture(scope="module", autouse=True)
def built():
    nbuild.build()
    n.load()


def with_workspace(prob, d):
    dec = decoder_for(prob)
    out, lse = dec(d["q_latent"], d["q_rope"], d["ckv"], d["kpe"], d["page_table"], d["seq_lens"], d["scale"])
    return out, lse, dec.cfg


def without_allocation(prob, d, cfg):
    out = torch.empty((prob.B, prob.Sq, prob.H, 512), dtype=torch.float32 if prob.w.out_dtype == "f32" else torch.bfloat16,
                      device="cuda")
    lse = torch.empty((prob.B, prob.Sq, prob.H), dtype=torch.float32, device="cuda")
    n.mla_decode_noalloc(d["q_latent"], d["q_rope"], d["ckv"], d["kpe"], d["page_table"], d["seq_lens"], d["scale"],
                         prob.w.window_left, out, lse, cfg)
    return out, lse


def assert_close(prob, a, b):
    tol_o, tol_l = TOL[prob.w.dtype]
    (oa, la), (ob, lb) = a, b
    oa, ob = oa.float().cpu().numpy(), ob.float().cpu().numpy()
    la, lb = la.cpu().numpy(), lb.cpu().numpy()
    assert np.isfinite(ob).all()
    assert np.abs(oa - ob).max() <= tol_o * max(np.abs(oa).max(), 1e-30)
    fin = np.isfinite(la)
    assert np.array_equal(fin, np.isfinite(lb))
    if fin.any():
        assert np.abs(la[fin] - lb[fin]).max() <= tol_l


def test_two_calls_in_a_row_match_the_workspace_decode():
    first = wl.make_problem("uniform", seed=31, H=128, Sq=2, causal=True, seq_lens=[2600, 77, 1000, 300])
    second = wl.make_problem("uniform", seed=32, H=64, Sq=1, dtype="e4m3", seq_lens=[5000, 64, 129])
    for prob in (first, second):
        d = prob.device_inputs("cuda")
        out_ws, lse_ws, cfg = with_workspace(prob, d)
        out_na, lse_na = without_allocation(prob, d, cfg)
        torch.cuda.synchronize()
        assert n.mla_noalloc_status() == n.MLA_OK
        assert_close(prob, (out_ws, lse_ws), (out_na, lse_na))


def test_device_side_errors_are_readable():
    """A visible page id outside the pool is read as zeros and flagged on the device; the
    flag is read back from the library's array, and a clean call clears it."""
    prob = wl.make_problem("uniform", seed=34, H=128, seq_lens=[700, 300])
    d = prob.device_inputs("cuda")
    dec = decoder_for(prob)
    d["page_table"][0, 3] = prob.pool_pages + 11
    without_allocation(prob, d, dec.cfg)
    assert n.mla_noalloc_status() == n.MLA_ERR_INVALID_ARG
    d["page_table"][0, 3] = int(prob.physical_page_table()[0, 3])
    without_allocation(prob, d, dec.cfg)
    assert n.mla_noalloc_status() == n.MLA_OK


def test_batch_beyond_the_array_is_refused():
    # 1024 rows need ~290 MB of partials: more than the 64 MiB array holds
    prob = wl.make_problem("uniform", seed=33, H=128, seq_lens=[64] * 1024)
    d = prob.device_inputs("cuda")
    cfg = n.make_config(seq_len_q=1, num_pages=prob.pool_pages, page_table_stride=prob.page_table.shape[1],
                        qkv_dtype=torch.bfloat16)
    out = torch.zeros((prob.B, 1, prob.H, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(n.MlaError) as e:
        n.mla_decode_noalloc(d["q_latent"], d["q_rope"], d["ckv"], d["kpe"], d["page_table"], d["seq_lens"],
                             d["scale"], -1, out, None, cfg)
    assert e.value.status == n.MLA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert not out.float().abs().sum().item()  # nothing was launched
