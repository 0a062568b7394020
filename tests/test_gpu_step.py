"""The one-call step (sv_quest_decode_step: page scores, top-K and sparse
attention) against the CPU oracle on the same seeded inputs.

Same bars as the separate calls: selected page sets exact except near-ties
(fp32 scores within 1e-4 relative of the K-th score); bf16 outputs within
max-abs 2e-2 of the oracle's fp32 attention over the selection the step made;
lse within 1e-3.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_quest_gb300 import binding, resident, synth

from helpers import check_selection
from test_gpu_parity import _with_lengths, check_attention, n_pages_of, pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from query_aware_sparse_quest_gb300 import build
    build.build()
    binding.sv_get_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(reset=True) == 0


def gpu_step(dw, budget_pages, page_table=None, q=None, ws=None):
    q = dw.q if q is None else q
    pt = dw.page_table if page_table is None else page_table
    B, Hq, D = q.shape
    Hkv = dw.cache.num_kv_heads
    sel_idx, sel_cnt = resident.select_buffers(B, Hkv, budget_pages)
    sel_idx.fill_(-7)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = binding.sv_quest_decode_step_workspace_size(B, Hq, Hkv, pt.shape[1], budget_pages)
    if ws is None:
        # Garbage in the workspace: the call must not rely on it starting at zero.
        ws = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    binding.sv_quest_decode_step(dw.cache, q, pt, dw.seq_lens, budget_pages, sel_idx, sel_cnt, out, lse, ws)
    return (sel_idx.cpu().numpy(), sel_cnt.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy())


def check_step(host, wl, result, K, q=None, seq_lens=None, page_table=None):
    q = wl.q if q is None else q
    seq = wl.seq_lens if seq_lens is None else seq_lens
    pt = wl.page_table if page_table is None else page_table
    sel, cnt, out, lse = result
    ref_sel, ref_cnt, ref_scores = oracle.select(host, q, pt, seq, K)
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, -(-seq // 16))
    check_attention(out, lse, *oracle.decode(host, q, pt, seq, sel, cnt))


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_step_parity(cfg):
    pr = pair(cfg)
    K = pr.wl.spec.budget_pages
    check_step(pr.host, pr.wl, gpu_step(pr.dw, K), K)


def test_step_repeatable_and_matches_separate_calls():
    """Three calls give bitwise equal results, the last two on one workspace
    that starts filled with garbage and is reused, and they
    agree with sv_quest_select + sv_sparse_decode: the same selection bit for
    bit (the same scores, the same exact top-K), attention within the bars."""
    pr = pair(2)
    K = pr.wl.spec.budget_pages
    dw = pr.dw
    B, Hq, D = dw.q.shape
    ws = torch.full((binding.sv_quest_decode_step_workspace_size(B, Hq, dw.cache.num_kv_heads,
                                                                 dw.page_table.shape[1], K),),
                    0x5A, dtype=torch.uint8, device="cuda")
    r1 = gpu_step(pr.dw, K)
    for _ in range(2):
        r2 = gpu_step(pr.dw, K, ws=ws)
        for a, b in zip(r1, r2):
            assert np.array_equal(a, b, equal_nan=True)
    dw = pr.dw
    B, Hq, D = dw.q.shape
    Hkv = dw.cache.num_kv_heads
    s2, c2 = resident.select_buffers(B, Hkv, K)
    ws = resident.workspace(binding.sv_quest_select_workspace_size(B, Hkv, dw.page_table.shape[1]))
    binding.sv_quest_select(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, s2, c2, workspace=ws)
    assert np.array_equal(c2.cpu().numpy(), r1[1])
    assert np.array_equal(s2.cpu().numpy(), r1[0])
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    wsd = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, Hkv, K))
    si = torch.as_tensor(r1[0], device="cuda")
    sc = torch.as_tensor(r1[1], device="cuda")
    binding.sv_sparse_decode(dw.cache, dw.q, dw.page_table, dw.seq_lens, si, sc, out, lse, wsd)
    check_attention(r1[2], r1[3], out.float().cpu().numpy(), lse.cpu().numpy())


@pytest.mark.parametrize("hq,hkv", [(4, 1), (8, 1), (8, 2), (6, 2), (32, 4), (8, 8), (16, 8)])
def test_step_head_geometries(hq, hkv):
    spec = synth.Spec("geom", batch=3, num_q_heads=hq, num_kv_heads=hkv, ctx=0, ragged=(1, 900),
                      budget_pages=7, seed=hq * 10 + hkv + 1, outlier_channels=True, shuffle_pool=True)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    for K in (7, 64):
        check_step(host, wl, gpu_step(dw, K), K)


def test_step_short_and_ragged_requests():
    """Single-token requests, exactly full pages, one-token last pages, n <= K
    (every page selected) and n > K, at budgets from 1 page up."""
    lens = np.array([1, 15, 16, 17, 31, 33, 16 * 40 + 1, 16 * 90], np.int32)
    spec = synth.Spec("short", batch=len(lens), num_q_heads=32, num_kv_heads=4, ctx=0,
                      ragged=(1, 2), budget_pages=3, seed=78, shuffle_pool=True)
    wl = _with_lengths(spec, lens)
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    for K in (1, 2, 3, 17, 64, 200):
        check_step(host, wl, gpu_step(dw, K), K)


def test_step_full_row_of_8192_pages():
    """A request of exactly 8192 pages and a one-page request in the same
    batch."""
    lens = np.array([8192 * 16, 16 * 3 + 5], np.int32)
    spec = synth.Spec("row8192", batch=2, num_q_heads=8, num_kv_heads=1, ctx=0, ragged=(1, 2),
                      budget_pages=100, seed=91, shuffle_pool=True)
    wl = _with_lengths(spec, lens)
    dw = resident.upload(wl)
    assert dw.page_table.shape[1] == 8192
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    check_step(host, wl, gpu_step(dw, 100), 100)


def test_step_wide_page_table():
    """max_pages of 8300 (rows wider than the scores of any request)."""
    spec = synth.SPECS[1].scaled(batch=3, ctx=16 * 700 + 9, budget_pages=40)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    B, width = wl.page_table.shape
    wide = np.full((B, 8300), -1, np.int32)
    wide[:, :width] = wl.page_table
    wide_t = torch.from_numpy(wide).cuda()
    r_wide = gpu_step(dw, 40, page_table=wide_t)
    check_step(host, wl, r_wide, 40, page_table=wide)


def test_step_exact_ties_go_to_lower_pages():
    spec = synth.Spec("ties", batch=2, num_q_heads=32, num_kv_heads=4, ctx=16 * 300, budget_pages=37,
                      seed=6, shuffle_pool=True)
    wl = synth.make_workload(spec)
    k = wl.k_tok.reshape(2, 300, 16, 4, 128)
    k[:] = wl.k_tok[:16].copy()[None, None]
    dw = resident.upload(wl)
    sel, cnt, out, lse = gpu_step(dw, 37)
    for b in range(2):
        for g in range(4):
            assert sel[b, g].tolist() == list(range(37))
            assert cnt[b, g] == 37
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, sel, cnt))


def test_step_nan_in_unfilled_slots_is_masked():
    spec = synth.SPECS[1].scaled(batch=3, ctx=16 * 50 + 3, budget_pages=9)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl, fill_bits=0x7FC0)
    host = oracle.build_cache(wl, 0x7FC0)
    res = gpu_step(dw, 9)
    assert np.isfinite(res[2]).all() and np.isfinite(res[3]).all()
    check_step(host, wl, res, 9)


def test_step_budget_sweep_after_append():
    """The full decode step of the budget-sweep workload: append one token per
    request, then the fused step at every budget of the sweep."""
    spec = synth.SPECS[4].scaled(batch=4, ctx=16 * 300 - 1)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    binding.sv_quest_update_meta(dw.cache, resident.bf16_tensor(wl.step_k[0], "cuda"),
                                 resident.bf16_tensor(wl.step_v[0], "cuda"),
                                 torch.from_numpy(wl.step_slots[0]).cuda())
    oracle.update_meta(host, wl.step_k[0], wl.step_v[0], wl.step_slots[0])
    seq = wl.seq_lens_after(1)
    dw.seq_lens.copy_(torch.from_numpy(seq))
    q = resident.bf16_tensor(wl.step_q[0], "cuda")
    for K in wl.spec.budget_sweep:
        check_step(host, wl, gpu_step(dw, K, q=q), K, q=wl.step_q[0], seq_lens=seq)


# ---------------------------------------------------------------- a reused workspace

def _flipped_q(wl):
    """The query with every sign flipped: other scores, another selection."""
    q_host = wl.q ^ np.uint16(0x8000)
    return q_host, resident.bf16_tensor(q_host, "cuda")


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_one_call_step_on_a_reused_workspace(cfg):
    """Nothing in the workspace needs to start at zero or survives a call:
    three calls on one workspace that starts filled with garbage, the second
    with every sign of q flipped (other scores, another selection), each
    match the oracle, and the first and third are bitwise equal."""
    pr = pair(cfg)
    wl, dw = pr.wl, pr.dw
    K = wl.spec.budget_pages
    B, Hq, D = dw.q.shape
    nbytes = binding.sv_quest_decode_step_workspace_size(B, Hq, dw.cache.num_kv_heads, dw.page_table.shape[1], K)
    ws = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    first = gpu_step(dw, K, ws=ws)
    check_step(pr.host, wl, first, K)
    q2_host, q2 = _flipped_q(wl)
    second = gpu_step(dw, K, q=q2, ws=ws)
    check_step(pr.host, wl, second, K, q=q2_host)
    third = gpu_step(dw, K, ws=ws)
    for a, b in zip(first, third):
        assert np.array_equal(a, b, equal_nan=True)


def test_one_call_step_workspace_shared_by_two_geometries():
    """One workspace alternating between two batch geometries (each call
    finds the other's scores and partials in it): every result matches the
    oracle."""
    a = synth.SPECS[2].scaled(batch=4, ctx=16 * 500 + 3, needles_per_request=4, budget_pages=40)
    b = synth.SPECS[1].scaled(batch=6, ctx=16 * 300 + 9, budget_pages=24)
    pairs = []
    for spec in (a, b):
        wl = synth.make_workload(spec)
        pairs.append((wl, resident.upload(wl), oracle.build_cache(wl, synth.UNFILLED_BITS)))
    nbytes = max(binding.sv_quest_decode_step_workspace_size(wl.spec.batch, wl.spec.num_q_heads,
                                                             wl.spec.num_kv_heads, wl.max_pages, wl.spec.budget_pages)
                 for wl, _, _ in pairs)
    ws = torch.full((nbytes,), 0x3C, dtype=torch.uint8, device="cuda")
    for wl, dw, host in pairs + pairs + pairs[:1] + pairs[:1]:
        K = wl.spec.budget_pages
        check_step(host, wl, gpu_step(dw, K, ws=ws), K)


def test_step_with_pinned_host_inputs_and_results():
    """q, page table and lengths in page-locked host memory, out and lse
    written straight into page-locked host memory: the kernels cross the host
    link themselves.  The results equal the device-memory call bit for bit."""
    pr = pair(1)
    wl, dw = pr.wl, pr.dw
    K = wl.spec.budget_pages
    B, Hq, D = dw.q.shape
    Hkv = dw.cache.num_kv_heads
    ref = gpu_step(dw, K)
    q_h, pt_h, sl_h = (t.cpu().pin_memory() for t in (dw.q, dw.page_table, dw.seq_lens))
    out_h = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.full((B, Hq), float("nan"), dtype=torch.float32).pin_memory()
    sel_idx, sel_cnt = resident.select_buffers(B, Hkv, K)
    ws = resident.workspace(binding.sv_quest_decode_step_workspace_size(B, Hq, Hkv, pt_h.shape[1], K))
    binding.sv_quest_decode_step(dw.cache, q_h, pt_h, sl_h, K, sel_idx, sel_cnt, out_h, lse_h, ws)
    torch.cuda.synchronize()
    assert np.array_equal(sel_idx.cpu().numpy(), ref[0]) and np.array_equal(sel_cnt.cpu().numpy(), ref[1])
    assert np.array_equal(out_h.float().numpy(), ref[2], equal_nan=True)
    assert np.array_equal(lse_h.numpy(), ref[3], equal_nan=True)
    check_step(pr.host, wl, (sel_idx.cpu().numpy(), sel_cnt.cpu().numpy(), out_h.float().numpy(), lse_h.numpy()), K)
    # The same call captured in a CUDA graph (as a serving loop would) and replayed.
    out_h.fill_(float("nan"))
    lse_h.fill_(float("nan"))

    def call():
        binding.sv_quest_decode_step(dw.cache, q_h, pt_h, sl_h, K, sel_idx, sel_cnt, out_h, lse_h, ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    out_h.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out_h.float().numpy(), ref[2], equal_nan=True)
    assert np.array_equal(lse_h.numpy(), ref[3], equal_nan=True)
