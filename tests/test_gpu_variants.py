"""Selection options on the GPU (sv_quest_select_ex / sv_sparse_decode_ex)
against the CPU oracle: per-query-head selection, forced sink / window
pages, and dense layers.  Same bars as the base method: page sets exact
except near-ties (1e-4 relative of the K-th ranked score), bf16 outputs
max-abs 2e-2, lse 1e-3."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_quest_gb300 import binding, resident, synth

from helpers import check_selection
from test_gpu_parity import _with_lengths, check_attention, n_pages_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from query_aware_sparse_quest_gb300 import build
    build.build()
    binding.sv_get_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(reset=True) == 0


def run_variant(dw, K, opts):
    B, Hq, D = dw.q.shape
    Hkv = dw.cache.num_kv_heads
    R = Hq if opts.per_q_head else Hkv
    max_pages = dw.page_table.shape[1]
    sel_idx, sel_cnt = resident.select_buffers(B, R, K)
    scores = torch.full((B, R, max_pages), float("nan"), dtype=torch.float32, device="cuda")
    binding.sv_quest_select_ex(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, opts, sel_idx, sel_cnt,
                               scores_out=scores)
    ws = resident.workspace(binding.sv_quest_select_ex_workspace_size(B, Hq, Hkv, max_pages, opts))
    s2, c2 = resident.select_buffers(B, R, K)
    binding.sv_quest_select_ex(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, opts, s2, c2, workspace=ws)
    assert torch.equal(s2, sel_idx) and torch.equal(c2, sel_cnt)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    wsd = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, Hkv, K))
    binding.sv_sparse_decode_ex(dw.cache, dw.q, dw.page_table, dw.seq_lens, sel_idx, sel_cnt, opts, out, lse, wsd)
    return (sel_idx.cpu().numpy(), sel_cnt.cpu().numpy(), scores.cpu().numpy(), out.float().cpu().numpy(),
            lse.cpu().numpy())


def check_variant(host, wl, K, opts, res):
    sel, cnt, scores, out, lse = res
    ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, K,
                                                 per_q_head=bool(opts.per_q_head), sink_pages=opts.sink_pages,
                                                 window_pages=opts.window_pages)
    n = n_pages_of(wl)
    ranked = ref_scores.copy()   # forced pages rank first: +inf, as the GPU reports them
    for b in range(wl.spec.batch):
        nb = int(n[b])
        forced = np.zeros(nb, bool)
        forced[: min(nb, opts.sink_pages)] = True
        if opts.window_pages:
            forced[max(0, nb - opts.window_pages):] = True
        ranked[b, :, :nb][:, forced] = np.inf
        gpu = scores[b, :, :nb]
        assert np.all(np.isinf(gpu[:, forced]) & (gpu[:, forced] > 0))
        r = ref_scores[b, :, :nb][:, ~forced].astype(np.float64)
        if r.size:
            np.testing.assert_allclose(gpu[:, ~forced], r, rtol=1e-5, atol=1e-5 * np.abs(r).max())
    check_selection(sel, cnt, ref_sel, ref_cnt, ranked, n)
    check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, sel, cnt,
                                             per_q_head=bool(opts.per_q_head)))


@pytest.fixture(scope="module")
def cfg1():
    spec = synth.SPECS[1].scaled(batch=3, ctx=16 * 300 + 7, budget_pages=24)
    wl = synth.make_workload(spec)
    return wl, resident.upload(wl), oracle.build_cache(wl, synth.UNFILLED_BITS)


@pytest.mark.parametrize("per_q_head,sink,window", [(True, 0, 0), (False, 1, 0), (False, 0, 4), (False, 2, 3),
                                                    (True, 1, 2)])
def test_variant_parity(cfg1, per_q_head, sink, window):
    wl, dw, host = cfg1
    opts = binding.quest_opts(per_q_head=per_q_head, sink_pages=sink, window_pages=window)
    check_variant(host, wl, wl.spec.budget_pages, opts, run_variant(dw, wl.spec.budget_pages, opts))


def test_variant_config0_per_head_and_window():
    wl = synth.make_workload(synth.SPECS[0])
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    for opts in (binding.quest_opts(per_q_head=True), binding.quest_opts(sink_pages=1, window_pages=1)):
        check_variant(host, wl, wl.spec.budget_pages, opts, run_variant(dw, wl.spec.budget_pages, opts))


@pytest.mark.parametrize("hq,hkv", [(4, 1), (8, 2), (6, 2), (16, 8)])
def test_variant_head_geometries(hq, hkv):
    spec = synth.Spec("geom", batch=3, num_q_heads=hq, num_kv_heads=hkv, ctx=0, ragged=(1, 900),
                      budget_pages=7, seed=hq * 10 + hkv + 5, outlier_channels=True, shuffle_pool=True)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    for opts in (binding.quest_opts(per_q_head=True), binding.quest_opts(per_q_head=True, sink_pages=1,
                                                                         window_pages=2)):
        check_variant(host, wl, 7, opts, run_variant(dw, 7, opts))


def test_forced_pages_fill_a_small_budget():
    """More forced pages than the budget: the lowest-indexed forced pages win."""
    lens = np.array([1, 17, 16 * 40 + 1, 16 * 90], np.int32)
    spec = synth.Spec("short", batch=len(lens), num_q_heads=32, num_kv_heads=4, ctx=0, ragged=(1, 2),
                      budget_pages=3, seed=79, shuffle_pool=True)
    wl = _with_lengths(spec, lens)
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    for K in (1, 2, 3, 5):
        opts = binding.quest_opts(sink_pages=2, window_pages=2)
        check_variant(host, wl, K, opts, run_variant(dw, K, opts))


def test_dense_layers_skip_selection():
    """Below dense_layers: select_ex writes nothing, decode_ex reads every page
    (equal to the oracle's dense attention)."""
    spec = synth.SPECS[1].scaled(batch=2, ctx=16 * 120 + 5, budget_pages=9)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    B, Hq, D = dw.q.shape
    opts = binding.quest_opts(layer=0, dense_layers=3)
    sel_idx, sel_cnt = resident.select_buffers(B, 4, 9)
    sel_idx.fill_(-5)
    sel_cnt.fill_(-5)
    binding.sv_quest_select_ex(dw.cache, dw.q, dw.page_table, dw.seq_lens, 9, opts, sel_idx, sel_cnt,
                               workspace=resident.workspace(1))
    torch.cuda.synchronize()
    assert bool((sel_idx == -5).all()) and bool((sel_cnt == -5).all())
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ws = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, 4, dw.page_table.shape[1]))
    binding.sv_sparse_decode_ex(dw.cache, dw.q, dw.page_table, dw.seq_lens, sel_idx, sel_cnt, opts, out, lse, ws)
    check_attention(out.float().cpu().numpy(), lse.cpu().numpy(),
                    *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens))
    # The layer after the dense ones selects normally.
    opts2 = binding.quest_opts(layer=3, dense_layers=3)
    check_variant(host, wl, 9, opts2, run_variant(dw, 9, opts2))


@pytest.mark.parametrize("per_q_head,sink,window", [(True, 0, 0), (False, 1, 4)])
def test_variant_parity_at_full_size_sampled(per_q_head, sink, window):
    """The options on the 128k batch-8 workload (8000 pages per request, 256-page
    budget, shuffled pool), as the benchmark runs them; sampled requests are
    checked against the oracle one by one."""
    from test_gpu_parity import pair
    pr = pair(2)
    wl, host, K = pr.wl, pr.host, pr.wl.spec.budget_pages
    opts = binding.quest_opts(per_q_head=per_q_head, sink_pages=sink, window_pages=window)
    sel, cnt, scores, out, lse = run_variant(pr.dw, K, opts)
    n_all = n_pages_of(wl)
    for b in (0, 5):
        sl = slice(b, b + 1)
        nb = int(n_all[b])
        ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q[sl], wl.page_table[sl], wl.seq_lens[sl], K,
                                                     per_q_head=per_q_head, sink_pages=sink, window_pages=window)
        forced = np.zeros(nb, bool)
        forced[: min(nb, sink)] = True
        if window:
            forced[max(0, nb - window):] = True
        ranked = ref_scores.copy()
        ranked[0, :, :nb][:, forced] = np.inf
        gpu = scores[b, :, :nb]
        assert np.all(np.isinf(gpu[:, forced]) & (gpu[:, forced] > 0))
        r = ref_scores[0, :, :nb][:, ~forced].astype(np.float64)
        np.testing.assert_allclose(gpu[:, ~forced], r, rtol=1e-5, atol=1e-5 * np.abs(r).max())
        check_selection(sel[sl], cnt[sl], ref_sel, ref_cnt, ranked, n_all[sl])
        check_attention(out[sl], lse[sl], *oracle.decode(host, wl.q[sl], wl.page_table[sl], wl.seq_lens[sl],
                                                         sel[sl], cnt[sl], per_q_head=per_q_head))
