"""GPU path (libsvquest.so through its C ABI) against the CPU oracle on the
same seeded inputs.

Bars: metadata and pool contents bit-exact; selected page sets exact except
near-ties (fp32 scores within 1e-4 relative of the K-th score); bf16 outputs
within max-abs 2e-2 of the oracle's fp32 outputs; fp32 lse within 1e-3.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_quest_gb300 import binding, resident, synth
from query_aware_sparse_quest_gb300.synth import bf16_bits_to_f32

from helpers import check_selection

pytestmark = pytest.mark.gpu

OUT_ATOL = 2e-2
LSE_ATOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from query_aware_sparse_quest_gb300 import build
    build.build()
    binding.sv_get_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(reset=True) == 0


# ---------------------------------------------------------------- helpers

def gpu_select(dw, budget_pages, use_workspace=True):
    B, Hkv = dw.batch, dw.cache.num_kv_heads
    max_pages = dw.page_table.shape[1]
    sel_idx, sel_cnt = resident.select_buffers(B, Hkv, budget_pages)
    scores = torch.full((B, Hkv, max_pages), float("nan"), dtype=torch.float32, device="cuda")
    binding.sv_quest_select(dw.cache, dw.q, dw.page_table, dw.seq_lens, budget_pages, sel_idx, sel_cnt,
                            scores_out=scores)
    if use_workspace:   # the workspace route must give the same selection
        ws = resident.workspace(binding.sv_quest_select_workspace_size(B, Hkv, max_pages))
        s2, c2 = resident.select_buffers(B, Hkv, budget_pages)
        binding.sv_quest_select(dw.cache, dw.q, dw.page_table, dw.seq_lens, budget_pages, s2, c2, workspace=ws)
        assert torch.equal(s2, sel_idx) and torch.equal(c2, sel_cnt)
    return sel_idx.cpu().numpy(), sel_cnt.cpu().numpy(), scores.cpu().numpy()


def gpu_decode(dw, sel_idx=None, sel_cnt=None, q=None):
    q = dw.q if q is None else q
    B, Hq, D = q.shape
    Hkv = dw.cache.num_kv_heads
    pages = dw.page_table.shape[1] if sel_idx is None else sel_idx.shape[2]
    ws = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, Hkv, pages))
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    si = None if sel_idx is None else torch.as_tensor(sel_idx, device="cuda")
    sc = None if sel_cnt is None else torch.as_tensor(sel_cnt, device="cuda")
    binding.sv_sparse_decode(dw.cache, q, dw.page_table, dw.seq_lens, si, sc, out, lse, ws)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check_scores(gpu, ref, n_pages):
    for b in range(ref.shape[0]):
        n = int(n_pages[b])
        r = ref[b, :, :n].astype(np.float64)
        gsc = gpu[b, :, :n].astype(np.float64)
        scale = np.abs(r).max()
        np.testing.assert_allclose(gsc, r, rtol=1e-5, atol=1e-5 * scale)


def check_attention(out, lse, ref_out, ref_lse):
    err = np.abs(out - ref_out).max()
    assert err <= OUT_ATOL, f"max abs output error {err}"
    finite = np.isfinite(ref_lse)
    assert np.array_equal(finite, np.isfinite(lse))
    lerr = np.abs(lse[finite] - ref_lse[finite]).max() if finite.any() else 0.0
    assert lerr <= LSE_ATOL, f"max abs lse error {lerr}"


def n_pages_of(wl, steps=0):
    return -(-(wl.seq_lens + steps) // wl.spec.page_size)


class Pair:
    """A workload resident on the GPU (pool built by sv_quest_update_meta) and on
    the host (pool built by the oracle) from the same token stream."""

    def __init__(self, spec, fill_bits=synth.UNFILLED_BITS):
        self.wl = synth.make_workload(spec)
        self.dw = resident.upload(self.wl, fill_bits=fill_bits)
        self.host = oracle.build_cache(self.wl, fill_bits)


_PAIRS = {}


def pair(cfg):
    if cfg not in _PAIRS:
        _PAIRS.clear()
        torch.cuda.empty_cache()
        _PAIRS[cfg] = Pair(synth.SPECS[cfg])
    return _PAIRS[cfg]


# ---------------------------------------------------------------- update_meta

# Chunks under 2048 tokens take one-token windows; 4096- and 2048-token chunks
# of the longer requests take 16-token windows, with runs that start in the
# middle of a window (request lengths are not multiples of 16), runs cut by a
# chunk boundary (folded into the stored min / max), whole pages written by
# one bulk store, and short last pages.
APPEND_CASES = [(1, 20, 700), (3, 20, 700), (16, 20, 700), (37, 20, 700), (4096, 20, 700),
                (4096, 700, 3000), (2048, 700, 3000)]


@pytest.mark.parametrize("chunk,lo,hi", APPEND_CASES)
def test_update_meta_bitexact(chunk, lo, hi):
    spec = synth.SPECS[3].scaled(batch=3 if hi <= 700 else 6, ragged=(lo, hi), seed=30 + chunk + hi)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl, prefill=False)
    host = oracle.Cache(wl.num_phys_pages, spec.num_kv_heads, fill_bits=synth.UNFILLED_BITS)
    T = wl.k_tok.shape[0]
    for a in range(0, T, chunk):
        e = min(T, a + chunk)
        binding.sv_quest_update_meta(dw.cache, resident.bf16_tensor(wl.k_tok[a:e], "cuda"),
                                     resident.bf16_tensor(wl.v_tok[a:e], "cuda"),
                                     torch.from_numpy(wl.slot_mapping[a:e]).cuda())
        oracle.update_meta(host, wl.k_tok[a:e], wl.v_tok[a:e], wl.slot_mapping[a:e])
    k = dw.cache.k_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    v = dw.cache.v_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    m = dw.cache.meta.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(k, host.k) and np.array_equal(v, host.v)
    touched = np.zeros(wl.num_phys_pages, bool)
    touched[wl.slot_mapping // 16] = True
    assert np.array_equal(bf16_bits_to_f32(m[touched]), bf16_bits_to_f32(host.meta[touched]))


def test_update_meta_decode_append_steps():
    """Config-4 style: one appended token per request per step, some starting a new page."""
    spec = synth.SPECS[4].scaled(batch=5, ctx=16 * 9 - 2, append_steps=4)
    wl = synth.make_workload(spec)
    p = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    for s in range(spec.append_steps):
        binding.sv_quest_update_meta(p.cache, resident.bf16_tensor(wl.step_k[s], "cuda"),
                                     resident.bf16_tensor(wl.step_v[s], "cuda"),
                                     torch.from_numpy(wl.step_slots[s]).cuda())
        oracle.update_meta(host, wl.step_k[s], wl.step_v[s], wl.step_slots[s])
    m = p.cache.meta.view(torch.int16).cpu().numpy().view(np.uint16)
    k = p.cache.k_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(k, host.k)
    assert np.array_equal(bf16_bits_to_f32(m), bf16_bits_to_f32(host.meta))


# ---------------------------------------------------------------- select + decode, all configs

@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_select_parity(cfg):
    pr = pair(cfg)
    wl = pr.wl
    K = wl.spec.budget_pages
    sel, cnt, scores = gpu_select(pr.dw, K)
    ref_sel, ref_cnt, ref_scores = oracle.select(pr.host, wl.q, wl.page_table, wl.seq_lens, K)
    n = n_pages_of(wl)
    check_scores(scores, ref_scores, n)
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n)


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_sparse_decode_parity(cfg):
    """Decode over the oracle's selection, then the full GPU select -> decode chain
    against the oracle's attention over the GPU's (tie-rule-checked) selection."""
    pr = pair(cfg)
    wl = pr.wl
    K = wl.spec.budget_pages
    ref_sel, ref_cnt, ref_scores = oracle.select(pr.host, wl.q, wl.page_table, wl.seq_lens, K)
    out, lse = gpu_decode(pr.dw, ref_sel, ref_cnt)
    ref_out, ref_lse = oracle.decode(pr.host, wl.q, wl.page_table, wl.seq_lens, ref_sel, ref_cnt)
    check_attention(out, lse, ref_out, ref_lse)
    sel, cnt, _ = gpu_select(pr.dw, K, use_workspace=False)
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n_pages_of(wl))
    out2, lse2 = gpu_decode(pr.dw, sel, cnt)
    ref_out2, ref_lse2 = oracle.decode(pr.host, wl.q, wl.page_table, wl.seq_lens, sel, cnt)
    check_attention(out2, lse2, ref_out2, ref_lse2)


@pytest.mark.parametrize("cfg,sample", [(0, None), (1, None), (2, [0, 5]), (3, [1, 17]), (4, [3])])
def test_dense_decode_parity(cfg, sample):
    pr = pair(cfg)
    wl = pr.wl
    out, lse = gpu_decode(pr.dw)
    rows = range(wl.spec.batch) if sample is None else sample
    for b in rows:
        sl = slice(b, b + 1)
        ref_out, ref_lse = oracle.decode(pr.host, wl.q[sl], wl.page_table[sl], wl.seq_lens[sl])
        check_attention(out[sl], lse[sl], ref_out, ref_lse)


def test_budget_sweep_step():
    """Config 4's step: append one token per request, then select + attend at each
    budget of the sweep and dense, against the oracle."""
    pr = pair(4)
    wl = pr.wl
    s = 0
    binding.sv_quest_update_meta(pr.dw.cache, resident.bf16_tensor(wl.step_k[s], "cuda"),
                                 resident.bf16_tensor(wl.step_v[s], "cuda"),
                                 torch.from_numpy(wl.step_slots[s]).cuda())
    oracle.update_meta(pr.host, wl.step_k[s], wl.step_v[s], wl.step_slots[s])
    seq = wl.seq_lens_after(s + 1)
    pr.dw.seq_lens.copy_(torch.from_numpy(seq))
    q = resident.bf16_tensor(wl.step_q[s], "cuda")
    dw = resident.DeviceWorkload(wl=wl, cache=pr.dw.cache, q=q, page_table=pr.dw.page_table, seq_lens=pr.dw.seq_lens)
    n = -(-seq // 16)
    for K in wl.spec.budget_sweep:
        sel, cnt, scores = gpu_select(dw, K, use_workspace=False)
        ref_sel, ref_cnt, ref_scores = oracle.select(pr.host, wl.step_q[s], wl.page_table, seq, K)
        check_scores(scores, ref_scores, n)
        check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n)
        out, lse = gpu_decode(dw, sel, cnt, q=q)
        ref_out, ref_lse = oracle.decode(pr.host, wl.step_q[s], wl.page_table, seq, sel, cnt)
        check_attention(out, lse, ref_out, ref_lse)
    out, lse = gpu_decode(dw, q=q)
    ref_out, ref_lse = oracle.decode(pr.host, wl.step_q[s][:2], wl.page_table[:2], seq[:2])
    check_attention(out[:2], lse[:2], ref_out, ref_lse)
    _PAIRS.clear()   # the resident pool changed


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("hq,hkv", [(4, 1), (8, 1), (8, 2), (6, 2), (32, 4), (8, 8), (16, 8)])
def test_head_geometries(hq, hkv):
    spec = synth.Spec("geom", batch=3, num_q_heads=hq, num_kv_heads=hkv, ctx=0, ragged=(1, 900),
                      budget_pages=7, seed=hq * 10 + hkv, outlier_channels=True, shuffle_pool=True)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    sel, cnt, scores = gpu_select(dw, 7)
    ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, 7)
    n = n_pages_of(wl)
    check_scores(scores, ref_scores, n)
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n)
    out, lse = gpu_decode(dw, ref_sel, ref_cnt)
    check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, ref_sel, ref_cnt))
    out, lse = gpu_decode(dw)
    check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens))


def test_short_and_ragged_requests():
    """Lengths 1, 15, 16, 17, 31, 33 and longer: single-token requests, exactly full
    pages, one-token last pages, n <= K (everything selected) and n > K."""
    lens = np.array([1, 15, 16, 17, 31, 33, 16 * 40 + 1, 16 * 90], np.int32)
    spec = synth.Spec("short", batch=len(lens), num_q_heads=32, num_kv_heads=4, ctx=0,
                      ragged=(1, 2), budget_pages=3, seed=77, shuffle_pool=True)
    wl = _with_lengths(spec, lens)
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    for K in (1, 2, 3, 64, 200):
        sel, cnt, scores = gpu_select(dw, K)
        ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, K)
        check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n_pages_of(wl))
        out, lse = gpu_decode(dw, sel, cnt)
        check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, sel, cnt))
    out, lse = gpu_decode(dw)
    check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens))


def _with_lengths(spec, lens):
    """A workload of `spec` whose requests have exactly the lengths `lens`."""
    lo = int(lens.min())
    base = synth.make_workload(spec.scaled(batch=len(lens), ragged=(int(lens.max()), int(lens.max()))))
    # Truncate each request of the max-length stream to its own length.
    P = spec.page_size
    keep = []
    off = 0
    for b, L in enumerate(lens):
        keep.append(np.arange(off, off + int(L)))
        off += int(base.seq_lens[b])
    keep = np.concatenate(keep)
    assert lo >= 1
    return dataclasses.replace(base, k_tok=base.k_tok[keep], v_tok=base.v_tok[keep],
                               slot_mapping=base.slot_mapping[keep], tok_request=base.tok_request[keep],
                               seq_lens=lens.astype(np.int32))


def test_exact_ties_go_to_lower_pages():
    """Every page holds the same keys, so every score is bitwise equal: the
    selection must be exactly pages 0..K-1 (not a near-tie case)."""
    spec = synth.Spec("ties", batch=2, num_q_heads=32, num_kv_heads=4, ctx=16 * 300, budget_pages=37,
                      seed=5, shuffle_pool=True)
    wl = synth.make_workload(spec)
    first_page = wl.k_tok[:16].copy()
    k = wl.k_tok.reshape(2, 300, 16, 4, 128)
    k[:] = first_page[None, None]
    dw = resident.upload(wl)
    sel, cnt, scores = gpu_select(dw, 37)
    for b in range(2):
        for g in range(4):
            assert np.all(scores[b, g, :300] == scores[b, g, 0])
            assert sel[b, g].tolist() == list(range(37))
            assert cnt[b, g] == 37


def test_nan_in_unfilled_slots_is_masked():
    """Unfilled pool slots holding NaN never reach the outputs."""
    spec = synth.SPECS[1].scaled(batch=3, ctx=16 * 50 + 3, budget_pages=9)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl, fill_bits=0x7FC0)
    host = oracle.build_cache(wl, 0x7FC0)
    sel, cnt, _ = gpu_select(dw, 9)
    ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, 9)
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n_pages_of(wl))
    for s_, c_ in ((sel, cnt), (None, None)):
        out, lse = gpu_decode(dw, s_, c_)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
        check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, s_, c_))


@pytest.mark.parametrize("slope", [3.0, 12.0])
def test_logits_rising_across_pages(slope):
    """Keys move along the query group's direction page after page, so the
    logits of the group's heads rise by about `slope` log2 units per page up to
    the last page (which keeps its own keys): at 12 the split kernel's running
    softmax base moves on every page, at 3 every few pages, with weights up to
    the 2^8 that the lazily moved base allows in between."""
    spec = synth.SPECS[1].scaled(batch=2, ctx=16 * 60 + 7, budget_pages=24)
    wl = synth.make_workload(spec)
    Hkv, Hq, P = spec.num_kv_heads, spec.num_q_heads, spec.page_size
    G = Hq // Hkv
    q = bf16_bits_to_f32(wl.q).astype(np.float64)
    k = bf16_bits_to_f32(wl.k_tok).astype(np.float64)
    scale_log2 = np.log2(np.e) / np.sqrt(spec.head_dim)
    off = 0
    for b, L in enumerate(wl.seq_lens):
        page = np.arange(int(L)) // P
        for g in range(Hkv):
            u = q[b, g * G:(g + 1) * G].sum(axis=0)
            step = slope / (scale_log2 * (u @ u) / G)   # u.(step u) / G heads ~ slope log2 units per head
            k[off:off + int(L), g] += np.outer(page - page[-1], step * u)
        off += int(L)
    wl = dataclasses.replace(wl, k_tok=synth.to_bf16_bits(k.astype(np.float32)))
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    sel, cnt, _ = gpu_select(dw, spec.budget_pages, use_workspace=False)
    ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, spec.budget_pages)
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n_pages_of(wl))
    for s_, c_ in ((sel, cnt), (None, None)):
        out, lse = gpu_decode(dw, s_, c_)
        check_attention(out, lse, *oracle.decode(host, wl.q, wl.page_table, wl.seq_lens, s_, c_))


def test_needle_recall_reported():
    """Needle pages of config 0 and 2 that the selection keeps (a statistic)."""
    for cfg in (0, 2):
        pr = pair(cfg)
        sel, cnt, _ = gpu_select(pr.dw, pr.wl.spec.budget_pages, use_workspace=False)
        hits = total = 0
        for b, p, _o in pr.wl.needles:
            for g in range(pr.wl.spec.num_kv_heads):
                hits += int(p in set(sel[b, g, : cnt[b, g]].tolist()))
                total += 1
        print(f"config {cfg}: needle pages selected {hits}/{total}")
        assert hits > total // 2
