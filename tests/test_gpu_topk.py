"""sv_quest_topk on given score rows against the oracle's selection step
(oracle.topk), bit-exact: both rank the same fp32 values by (score desc, page
asc).  The rows are shaped to reach every path of the kernel: few candidates
in the threshold's histogram bin (ranked inside each warp), 33 to 256 of them
(ranked by one thread each), a crowded bin (exact radix select), exact ties at
the threshold, infinities, rows with n <= K, and each register width (rows of
up to 8192, 16384 and 32768 pages).  Entries past a row's last page hold NaN
and must be ignored.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_quest_gb300 import binding, resident

pytestmark = pytest.mark.gpu

PAGE = 16


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from query_aware_sparse_quest_gb300 import build
    build.build()
    binding.sv_get_device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(reset=True) == 0


def rows_of(kind: str, rng, shape):
    if kind == "normal":
        return rng.standard_normal(shape)
    if kind == "dense_band":
        # one outlier stretches the histogram range, so the threshold's bin
        # holds more than a warp of candidates
        x = rng.uniform(0.0, 0.02, shape)
        x[..., 5] = 1.0
        return x
    if kind == "few_values":
        return rng.integers(0, 10, shape).astype(np.float64)
    if kind == "all_equal":
        return np.full(shape, 2.5)
    if kind == "with_inf":
        x = rng.standard_normal(shape)
        x[rng.random(shape) < 0.01] = np.inf
        x[rng.random(shape) < 0.05] = -np.inf
        return x
    if kind == "negative":
        return rng.standard_normal(shape) - 100.0
    if kind == "heavy_tail":
        return rng.lognormal(0.0, 3.0, shape)
    raise ValueError(kind)


def check(scores: np.ndarray, seq_lens: np.ndarray, K: int):
    B, R, mp = scores.shape
    n = -(-seq_lens // PAGE)
    padded = scores.astype(np.float32).copy()
    for b in range(B):
        padded[b, :, n[b]:] = np.nan
    sel, cnt = resident.select_buffers(B, R, K)
    sel.fill_(-7)
    binding.sv_quest_topk(torch.from_numpy(padded).cuda(), torch.from_numpy(seq_lens.astype(np.int32)).cuda(), K,
                          sel, cnt)
    ref_sel, ref_cnt = oracle.topk(np.nan_to_num(padded.reshape(B * R, mp), nan=0.0),
                                   np.repeat(n, R).astype(np.int32), K)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt.reshape(B, R))
    got = sel.cpu().numpy()
    want = ref_sel.reshape(B, R, K)
    bad = np.argwhere((got != want).any(axis=2))
    assert len(bad) == 0, f"rows differ: {bad[:5].tolist()}"


KINDS = ["normal", "dense_band", "few_values", "all_equal", "with_inf", "negative", "heavy_tail"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("K", [1, 37, 256])
def test_topk_rows_of_8000_pages(kind, K):
    rng = np.random.default_rng(1000 * KINDS.index(kind) + K)
    B, R, mp = 3, 4, 8000
    seq_lens = np.array([mp * PAGE, mp * PAGE - 7, 5000 * PAGE + 1])
    check(rows_of(kind, rng, (B, R, mp)), seq_lens, K)


@pytest.mark.parametrize("mp", [8192, 8193, 16384, 16385, 32768])
@pytest.mark.parametrize("kind", ["normal", "dense_band", "few_values"])
def test_topk_each_register_width(mp, kind):
    rng = np.random.default_rng(mp + KINDS.index(kind))
    B, R = 2, 2
    seq_lens = np.array([mp * PAGE, (mp // 3) * PAGE + 9])
    check(rows_of(kind, rng, (B, R, mp)), seq_lens, 300)


def test_topk_short_rows_and_large_budgets():
    """n <= K keeps every page; n = 1; K far above n; K = n exactly."""
    rng = np.random.default_rng(7)
    seq_lens = np.array([1, 16, 17, 16 * 100, 16 * 256, 16 * 257, 16 * 3000 + 3])
    scores = rng.standard_normal((len(seq_lens), 2, 3001))
    for K in (1, 100, 256, 257, 4096):
        check(scores, seq_lens, K)


@pytest.mark.parametrize("K", [1, 3, 5, 37, 256])
def test_topk_forced_pages_at_both_ends(K):
    """Forced pages (the first page and the last four of each row) score +inf,
    as the scoring kernel writes them: they rank above every scored page, among
    themselves by lower page index, and the histogram still spans the scored
    pages.  Budgets below, at and above the five forced pages."""
    rng = np.random.default_rng(500 + K)
    B, R, mp = 3, 4, 8000
    seq_lens = np.array([mp * PAGE, mp * PAGE - 7, 5000 * PAGE + 1])
    scores = rng.standard_normal((B, R, mp))
    n = -(-seq_lens // PAGE)
    for b in range(B):
        scores[b, :, 0] = np.inf
        scores[b, :, n[b] - 4:n[b]] = np.inf
    check(scores, seq_lens, K)
