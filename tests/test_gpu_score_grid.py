"""Page scores and selections for batch shapes that reach every way the
scoring kernel divides a batch over its CTAs: requests split by length over a
one-dimensional grid (all rows full: the even split taken directly; unequal
rows: the split computed from the lengths, including requests of one token
and rows shorter than a CTA's share), and one CTA per request when there are
more requests than the grid takes (a two-dimensional grid in waves).  Same
bars as the other parity tests: fp32 scores within 1e-5 relative of the
oracle's, selections exact except near-ties.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_quest_gb300 import binding, resident, synth

from helpers import check_selection
from test_gpu_parity import _with_lengths, check_scores, gpu_select, n_pages_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from query_aware_sparse_quest_gb300 import build
    build.build()
    binding.sv_get_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(reset=True) == 0


def run(lens, hq, hkv, K, seed):
    spec = synth.Spec("grid", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, ctx=0, ragged=(1, 2),
                      budget_pages=K, seed=seed, outlier_channels=True, shuffle_pool=True)
    wl = _with_lengths(spec, np.asarray(lens, np.int32))
    dw = resident.upload(wl)
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    sel, cnt, scores = gpu_select(dw, K)
    ref_sel, ref_cnt, ref_scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, K)
    check_scores(scores, ref_scores, n_pages_of(wl))
    check_selection(sel, cnt, ref_sel, ref_cnt, ref_scores, n_pages_of(wl))


def test_all_rows_full():
    """Every request fills the table's row: the even split, taken without the
    length computation."""
    run([16 * 700] * 6, 32, 4, 40, seed=501)


def test_one_short_request_among_full_ones():
    run([16 * 700] * 5 + [16 * 123 + 5], 32, 4, 40, seed=502)


@pytest.mark.parametrize("hq,hkv", [(32, 4), (8, 8), (4, 1)])
def test_mixed_lengths_with_single_token_requests(hq, hkv):
    rng = np.random.default_rng(503 + hkv)
    lens = rng.integers(1, 16 * 300, size=40)
    lens[[0, 7, 19]] = 1
    lens[3] = 16 * 300
    run(lens.tolist(), hq, hkv, 17, seed=504 + hkv)


def test_as_many_requests_as_a_wave_holds():
    """152 requests (the GB300's SM count): one CTA each when all are full."""
    run([16 * 40] * 152, 8, 2, 9, seed=505)


@pytest.mark.parametrize("batch", [200, 300])
def test_more_requests_than_the_wave(batch):
    """More requests than SMs (and than the split by length serves): one CTA
    per request, in waves."""
    rng = np.random.default_rng(batch)
    run(rng.integers(1, 16 * 60, size=batch).tolist(), 8, 2, 12, seed=506 + batch)
