"""Failure detection on the device without a fault: corrupt device-resident
indices (a page-table entry, a selected page, a slot, a length) are caught by
the kernels' own bounds checks, which skip the access and set a bit of the
device error word (sv_get_device_error), while every other request's results
still match the CPU oracle.

Every bad index is made on the host.  The pools carry a guard tail of extra
pages past the page count the library is told about, and each bad index
points exactly at the first guard page, so even a missing check would stay
inside the allocation; the tests check that the guard is left untouched.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_quest_gb300 import binding, resident, synth
from query_aware_sparse_quest_gb300.synth import bf16_bits_to_f32

from helpers import check_selection

pytestmark = pytest.mark.gpu

SV_DEVERR_PAGE_TABLE, SV_DEVERR_SEL_IDX, SV_DEVERR_SLOT, SV_DEVERR_SEQ_LEN = 0x1, 0x2, 0x4, 0x8
OUT_ATOL, LSE_ATOL = 2e-2, 1e-3
GUARD_PAGES = 4
GUARD_BITS = 0x7F7F          # bf16 pattern written to every guard page


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from query_aware_sparse_quest_gb300 import build
    build.build()
    binding.sv_get_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    binding.sv_get_device_error(reset=True)


class Guarded:
    """A prefilled device workload whose pools hold GUARD_PAGES extra pages past
    the num_phys_pages the library is given, plus the oracle's host copy."""

    def __init__(self, spec):
        self.wl = wl = synth.make_workload(spec)
        dw = resident.upload(wl)
        n = wl.num_phys_pages
        self.n_phys = n

        def grow(t):
            g = torch.empty((n + GUARD_PAGES, *t.shape[1:]), dtype=t.dtype, device=t.device)
            g[:n].copy_(t)
            g[n:].view(torch.int16).fill_(np.int16(np.uint16(GUARD_BITS)))
            return g

        self.k, self.v, self.meta = grow(dw.cache.k_pool), grow(dw.cache.v_pool), grow(dw.cache.meta)
        self.cache = binding.Cache(self.k, self.v, self.meta)
        self.cache.c.num_phys_pages = n            # the guard is outside the pool the library sees
        self.q, self.page_table, self.seq_lens = dw.q, dw.page_table, dw.seq_lens
        self.host = oracle.build_cache(wl, synth.UNFILLED_BITS)
        self.guard0 = [t[n:].clone() for t in (self.k, self.v, self.meta)]

    def guard_intact(self) -> bool:
        n = self.n_phys
        return all(torch.equal(t[n:], g) for t, g in zip((self.k, self.v, self.meta), self.guard0))


def _spec():
    return synth.SPECS[2].scaled(batch=4, ctx=16 * 300 + 7, budget_pages=24, needles_per_request=4)


def _step(gw, page_table, seq_lens, K):
    B, Hq, D = gw.q.shape
    Hkv, mp = gw.cache.num_kv_heads, page_table.shape[1]
    sel, cnt = resident.select_buffers(B, Hkv, K)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = resident.workspace(binding.sv_quest_decode_step_workspace_size(B, Hq, Hkv, mp, K))
    binding.sv_quest_decode_step(gw.cache, gw.q, page_table, seq_lens, K, sel, cnt, out, lse, ws)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), cnt.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()


def _oracle_rows(gw, rows, K, sel=None, cnt=None):
    """Oracle selection and attention of the requests `rows` alone."""
    wl = gw.wl
    q, pt, sl = wl.q[rows], wl.page_table[rows], wl.seq_lens[rows]
    ref_sel, ref_cnt, ref_sc = oracle.select(gw.host, q, pt, sl, K)
    if sel is None:
        sel, cnt = ref_sel, ref_cnt
    ref_out, ref_lse = oracle.decode(gw.host, q, pt, sl, sel, cnt)
    return ref_sel, ref_cnt, ref_sc, ref_out, ref_lse


def _check_attention(out, lse, ref_out, ref_lse):
    assert float(np.abs(out - ref_out).max()) <= OUT_ATOL
    assert float(np.abs(lse - ref_lse).max()) <= LSE_ATOL


def test_page_table_entry_past_the_pool_is_flagged_and_skipped():
    gw = Guarded(_spec())
    wl, K = gw.wl, gw.wl.spec.budget_pages
    bad_b, bad_p = 1, 37
    pt = gw.page_table.clone()
    pt[bad_b, bad_p] = gw.n_phys                  # first guard page
    binding.sv_get_device_error(reset=True)
    sel, cnt, out, lse = _step(gw, pt, gw.seq_lens, K)
    flags = binding.sv_get_device_error(reset=True)
    assert flags == SV_DEVERR_PAGE_TABLE, hex(flags)
    assert gw.guard_intact()
    good = np.array([b for b in range(wl.spec.batch) if b != bad_b])
    ref_sel, ref_cnt, ref_sc, ref_out, ref_lse = _oracle_rows(gw, good, K)
    n = -(-wl.seq_lens[good] // 16)
    check_selection(sel[good], cnt[good], ref_sel, ref_cnt, ref_sc, n)
    _, _, _, ref_out2, ref_lse2 = _oracle_rows(gw, good, K, sel[good], cnt[good])
    _check_attention(out[good], lse[good], ref_out2, ref_lse2)
    # The bad request still gets a full selection and finite outputs (its bad
    # page scores 0 and, if selected, contributes no token).
    assert np.all(cnt[bad_b] == K) and np.all(np.isfinite(out[bad_b])) and np.all(np.isfinite(lse[bad_b]))


def test_selected_page_past_the_request_is_flagged_and_skipped():
    gw = Guarded(_spec())
    wl, K = gw.wl, gw.wl.spec.budget_pages
    B, Hq, D = gw.q.shape
    Hkv = gw.cache.num_kv_heads
    ref_sel, ref_cnt, _ = oracle.select(gw.host, wl.q, wl.page_table, wl.seq_lens, K)
    bad_b, bad_g, bad_j = 2, 3, 5
    n_bad = int(-(-wl.seq_lens[bad_b] // 16))
    sel = ref_sel.copy()
    sel[bad_b, bad_g, bad_j] = n_bad              # one past the request's last page
    ws = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, Hkv, K))
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    binding.sv_get_device_error(reset=True)
    binding.sv_sparse_decode(gw.cache, gw.q, gw.page_table, gw.seq_lens, torch.as_tensor(sel, device="cuda"),
                             torch.as_tensor(ref_cnt, device="cuda"), out, lse, ws)
    torch.cuda.synchronize()
    flags = binding.sv_get_device_error(reset=True)
    assert flags == SV_DEVERR_SEL_IDX, hex(flags)
    assert gw.guard_intact()
    # Every head attends exactly the oracle's pages, except the bad row's,
    # which attend the row's other pages: the bad entry is skipped.
    expect_sel, expect_cnt = ref_sel.copy(), ref_cnt.copy()
    row = [p for j, p in enumerate(ref_sel[bad_b, bad_g, :ref_cnt[bad_b, bad_g]]) if j != bad_j]
    expect_sel[bad_b, bad_g] = -1
    expect_sel[bad_b, bad_g, :len(row)] = row
    expect_cnt[bad_b, bad_g] = len(row)
    ref_out, ref_lse = oracle.decode(gw.host, wl.q, wl.page_table, wl.seq_lens, expect_sel, expect_cnt)
    _check_attention(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse)


def test_slot_past_the_pool_is_flagged_and_skipped():
    spec = synth.SPECS[4].scaled(batch=5, ctx=16 * 40 - 3, budget_pages=8, append_steps=1)
    gw = Guarded(spec)
    wl = gw.wl
    slots = wl.step_slots[0].copy()
    bad_b = 3
    slots[bad_b] = gw.n_phys * 16                  # first slot of the first guard page
    binding.sv_get_device_error(reset=True)
    binding.sv_quest_update_meta(gw.cache, resident.bf16_tensor(wl.step_k[0], "cuda"),
                                 resident.bf16_tensor(wl.step_v[0], "cuda"), torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    flags = binding.sv_get_device_error(reset=True)
    assert flags == SV_DEVERR_SLOT, hex(flags)
    assert gw.guard_intact()
    keep = np.array([b for b in range(spec.batch) if b != bad_b])
    oracle.update_meta(gw.host, wl.step_k[0][keep], wl.step_v[0][keep], wl.step_slots[0][keep])
    n = gw.n_phys
    k = gw.k[:n].view(torch.int16).cpu().numpy().view(np.uint16)
    v = gw.v[:n].view(torch.int16).cpu().numpy().view(np.uint16)
    m = gw.meta[:n].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(k, gw.host.k) and np.array_equal(v, gw.host.v)
    assert np.array_equal(bf16_bits_to_f32(m), bf16_bits_to_f32(gw.host.meta))


@pytest.mark.parametrize("bad_len", [0, 16 * 400])
def test_bad_sequence_length_is_flagged(bad_len):
    """A length of 0, or one that needs more pages than the page table holds."""
    gw = Guarded(_spec())
    wl, K = gw.wl, gw.wl.spec.budget_pages
    bad_b = 0
    sl = gw.seq_lens.clone()
    sl[bad_b] = bad_len
    binding.sv_get_device_error(reset=True)
    sel, cnt, out, lse = _step(gw, gw.page_table, sl, K)
    flags = binding.sv_get_device_error(reset=True)
    assert flags == SV_DEVERR_SEQ_LEN, hex(flags)
    assert gw.guard_intact()
    good = np.array([b for b in range(wl.spec.batch) if b != bad_b])
    ref_sel, ref_cnt, ref_sc, _, _ = _oracle_rows(gw, good, K)
    check_selection(sel[good], cnt[good], ref_sel, ref_cnt, ref_sc, -(-wl.seq_lens[good] // 16))
    _, _, _, ref_out, ref_lse = _oracle_rows(gw, good, K, sel[good], cnt[good])
    _check_attention(out[good], lse[good], ref_out, ref_lse)
    if bad_len == 0:
        # No pages: an empty selection, out = 0 and lse = -inf for every head.
        assert np.all(cnt[bad_b] == 0) and np.all(sel[bad_b] == -1)
        assert np.all(out[bad_b] == 0) and np.all(np.isneginf(lse[bad_b]))
    else:
        # Clamped to the page table's row: every page counts as full.
        assert np.all(cnt[bad_b] == K) and np.all(np.isfinite(lse[bad_b]))
