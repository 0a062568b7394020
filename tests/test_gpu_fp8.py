"""FP8 (e4m3) K/V pools on the GPU against the CPU oracle's fp8 pool.

Codes, scales and metadata bit-exact after appends; attention over the
decoded rows within the base bars (bf16 out max-abs 2e-2, lse 1e-3);
selection identical to the bf16 pool's (same metadata).  Unfilled slots hold
NaN codes and NaN scales, so a missing mask is loud."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_quest_gb300 import binding, resident, synth

from helpers import check_selection
from test_gpu_parity import check_attention, n_pages_of

pytestmark = pytest.mark.gpu

NAN_CODE = 0x7F


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from query_aware_sparse_quest_gb300 import build
    build.build()
    binding.sv_get_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(reset=True) == 0


def _pair(spec):
    wl = synth.make_workload(spec)
    dw = resident.upload(wl, fp8=True, fill_code=NAN_CODE, fill_scale=float("nan"))
    host = oracle.build_cache(wl, synth.UNFILLED_BITS, fp8=True, fill_code=NAN_CODE, fill_scale=float("nan"))
    return wl, dw, host


def _decode(dw, sel_idx=None, sel_cnt=None, opts=None):
    B, Hq, D = dw.q.shape
    Hkv = dw.cache.num_kv_heads
    pages = dw.page_table.shape[1] if sel_idx is None else sel_idx.shape[2]
    ws = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, Hkv, pages))
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    si = None if sel_idx is None else torch.as_tensor(sel_idx, device="cuda")
    sc = None if sel_cnt is None else torch.as_tensor(sel_cnt, device="cuda")
    binding.sv_sparse_decode_ex(dw.cache, dw.q, dw.page_table, dw.seq_lens, si, sc, opts, out, lse, ws)
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("chunk,lo,hi", [(1, 20, 700), (3, 20, 700), (16, 20, 700), (37, 20, 700),
                                         (4096, 20, 700), (4096, 700, 3000), (2048, 700, 3000)])
def test_fp8_append_bitexact(chunk, lo, hi):
    """Chunks under 2048 tokens take one-token windows; the longer requests in
    4096- and 2048-token chunks take 16-token windows (runs starting mid-window,
    runs cut by a chunk boundary, short last pages)."""
    spec = synth.SPECS[3].scaled(batch=3 if hi <= 700 else 6, ragged=(lo, hi), seed=60 + chunk + hi)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl, prefill=False, fp8=True)
    host = oracle.Cache(wl.num_phys_pages, spec.num_kv_heads, fp8=True, fill_code=NAN_CODE, fill_scale=float("nan"))
    T = wl.k_tok.shape[0]
    for a in range(0, T, chunk):
        e = min(T, a + chunk)
        binding.sv_quest_update_meta(dw.cache, resident.bf16_tensor(wl.k_tok[a:e], "cuda"),
                                     resident.bf16_tensor(wl.v_tok[a:e], "cuda"),
                                     torch.from_numpy(wl.slot_mapping[a:e]).cuda())
        oracle.update_meta(host, wl.k_tok[a:e], wl.v_tok[a:e], wl.slot_mapping[a:e])
    slots = wl.slot_mapping
    P = spec.page_size
    pg, off = slots // P, slots % P
    for gpu, ref in ((dw.cache.k_pool, host.k8), (dw.cache.v_pool, host.v8)):
        g = gpu.cpu().numpy()
        np.testing.assert_array_equal(g[pg, :, off], ref[pg, :, off])
    for gpu, ref in ((dw.cache.k_scale, host.ks), (dw.cache.v_scale, host.vs)):
        g = gpu.cpu().numpy()
        np.testing.assert_array_equal(g[pg, :, off].view(np.uint32), ref[pg, :, off].view(np.uint32))
    m = dw.cache.meta.view(torch.int16).cpu().numpy().view(np.uint16)
    touched = np.zeros(wl.num_phys_pages, bool)
    touched[pg] = True
    np.testing.assert_array_equal(m[touched], host.meta[touched])


@pytest.mark.parametrize("cfg", [0, 1])
def test_fp8_decode_parity(cfg):
    spec = synth.SPECS[cfg] if cfg == 0 else synth.SPECS[1].scaled(batch=3, ctx=16 * 400 + 5)
    wl, dw, host = _pair(spec)
    K = spec.budget_pages
    # Selection on an fp8 pool equals the bf16 method's (same metadata).
    B, Hq, _ = dw.q.shape
    sel_idx, sel_cnt = resident.select_buffers(B, spec.num_kv_heads, K)
    ws = resident.workspace(binding.sv_quest_select_workspace_size(B, spec.num_kv_heads, dw.page_table.shape[1]))
    binding.sv_quest_select(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, sel_idx, sel_cnt, workspace=ws)
    sel, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
    ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, K)
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n_pages_of(wl))
    out, lse = _decode(dw, sel, cnt)
    check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, sel, cnt))
    out, lse = _decode(dw)
    check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens))


def test_fp8_short_ragged_and_per_head():
    lens = np.array([1, 15, 16, 17, 33, 16 * 40 + 1, 16 * 90], np.int32)
    from test_gpu_parity import _with_lengths
    spec = synth.Spec("short", batch=len(lens), num_q_heads=32, num_kv_heads=4, ctx=0, ragged=(1, 2),
                      budget_pages=3, seed=81, shuffle_pool=True, outlier_channels=True)
    wl = _with_lengths(spec, lens)
    dw = resident.upload(wl, fp8=True, fill_code=NAN_CODE, fill_scale=float("nan"))
    host = oracle.build_cache(wl, synth.UNFILLED_BITS, fp8=True, fill_code=NAN_CODE, fill_scale=float("nan"))
    for K in (1, 3, 64):
        sel, cnt, _ = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, K)
        out, lse = _decode(dw, sel, cnt)
        assert np.isfinite(out).all()
        check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, sel, cnt))
    opts = binding.quest_opts(per_q_head=True)
    sel, cnt, _ = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, 5, per_q_head=True)
    out, lse = _decode(dw, sel, cnt, opts)
    check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, sel, cnt, per_q_head=True))


@pytest.mark.parametrize("hq,hkv", [(4, 1), (8, 2), (16, 8)])
def test_fp8_head_geometries(hq, hkv):
    spec = synth.Spec("geom", batch=3, num_q_heads=hq, num_kv_heads=hkv, ctx=0, ragged=(1, 900),
                      budget_pages=7, seed=hq * 10 + hkv + 9, outlier_channels=True, shuffle_pool=True)
    wl, dw, host = _pair(spec)
    sel, cnt, _ = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, 7)
    check_attention(*_decode(dw, sel, cnt), *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, sel, cnt))
    check_attention(*_decode(dw), *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens))


def test_fp8_decode_step_and_error_vs_bf16():
    """sv_quest_decode_step on an fp8 pool matches the oracle;
    the fp8 outputs stay close to the bf16 pool's (a statistic of the codec)."""
    spec = synth.SPECS[1].scaled(batch=2, ctx=16 * 300 + 3, budget_pages=40)
    wl, dw, host = _pair(spec)
    B, Hq, D = dw.q.shape
    K = spec.budget_pages
    sel_idx, sel_cnt = resident.select_buffers(B, spec.num_kv_heads, K)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ws = resident.workspace(binding.sv_quest_decode_step_workspace_size(B, Hq, spec.num_kv_heads,
                                                                        dw.page_table.shape[1], K))
    binding.sv_quest_decode_step(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, sel_idx, sel_cnt, out, lse, ws)
    sel, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
    o8, l8 = out.float().cpu().numpy(), lse.cpu().numpy()
    check_attention(o8, l8, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, sel, cnt))
    h16 = oracle.build_cache(wl, synth.UNFILLED_BITS)
    o16, _ = oracle.decode(h16, wl.q, wl.page_table, wl.seq_lens, sel, cnt)
    diff = np.abs(o8 - o16)
    print(f"fp8 vs bf16 pool: output difference max {diff.max():.4f}, mean {diff.mean():.5f}")
    # A statistic of the codec (per-row scales meet outlier key channels), not a
    # parity bar; the bound only catches a gross error such as a lost scale.
    assert diff.max() < 1.0


def test_fp8_step_full_size_128k():
    """The benchmark's workload (8 requests of 128000 tokens, budget 256
    pages, shuffled 64000-page pool) on an fp8 pool through
    sv_quest_decode_step, twice on one workspace: every selection against the
    oracle, attention of two sampled requests against the oracle's fp8
    decode over those selections, and the two calls bitwise equal."""
    wl, dw, host = _pair(synth.SPECS[2])
    spec = wl.spec
    K = spec.budget_pages
    B, Hq, D = dw.q.shape
    ws = resident.workspace(binding.sv_quest_decode_step_workspace_size(B, Hq, spec.num_kv_heads, wl.max_pages, K))
    runs = []
    for _ in range(2):
        sel_idx, sel_cnt = resident.select_buffers(B, spec.num_kv_heads, K)
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        binding.sv_quest_decode_step(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, sel_idx, sel_cnt, out, lse, ws)
        runs.append((sel_idx.cpu().numpy(), sel_cnt.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()))
    for a, b in zip(*runs):
        assert np.array_equal(a, b, equal_nan=True)
    sel, cnt, out, lse = runs[1]
    ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, K)
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n_pages_of(wl))
    for b in (0, 5):
        rows = slice(b, b + 1)
        ref_out, ref_lse = oracle.decode(host, wl.q[rows], wl.page_table[rows], wl.seq_lens[rows], sel[rows],
                                         cnt[rows])
        check_attention(out[rows], lse[rows], ref_out, ref_lse)


def test_fp8_step_full_size_512_page_budget():
    """The workload where selected K/V dominate (16 requests of 65536 tokens
    plus one appended slot, 512-page budget, shuffled pool) on an fp8 pool
    through sv_quest_decode_step: every selection against the oracle, attention
    of sampled requests against the oracle's fp8 decode over those selections."""
    wl, dw, host = _pair(synth.SPECS[4].scaled(budget_pages=512))
    spec = wl.spec
    K = 512
    B, Hq, D = dw.q.shape
    ws = resident.workspace(binding.sv_quest_decode_step_workspace_size(B, Hq, spec.num_kv_heads, wl.max_pages, K))
    sel_idx, sel_cnt = resident.select_buffers(B, spec.num_kv_heads, K)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    binding.sv_quest_decode_step(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, sel_idx, sel_cnt, out, lse, ws)
    sel, cnt = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, K)
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n_pages_of(wl))
    for b in (0, 9, 15):
        rows = slice(b, b + 1)
        ref_out, ref_lse = oracle.decode(host, wl.q[rows], wl.page_table[rows], wl.seq_lens[rows], sel[rows],
                                         cnt[rows])
        check_attention(out[rows], lse[rows], ref_out, ref_lse)
