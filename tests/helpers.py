"""Test helpers: fp64 reference pieces built from textbook definitions or
library routines, independent of the oracle's code, plus the selection
comparison rule."""
from __future__ import annotations

import itertools

import numpy as np

from query_aware_sparse_quest_gb300.synth import bf16_bits_to_f32, to_bf16_bits


def bf(x) -> np.ndarray:
    """Exact bf16 bits of small values (asserts they are representable)."""
    x = np.asarray(x, dtype=np.float64)
    b = to_bf16_bits(x)
    assert np.array_equal(bf16_bits_to_f32(b).astype(np.float64), x), "value not exact in bf16"
    return b


def page_tokens(wl, b: int, p: int, steps: int = 0) -> np.ndarray:
    """Indices into the prefill stream of request b's logical page p (valid tokens only)."""
    P = wl.spec.page_size
    base = int(np.concatenate([[0], np.cumsum(wl.seq_lens.astype(np.int64))])[b])
    L = int(wl.seq_lens[b])
    lo, hi = p * P, min(L, (p + 1) * P)
    return np.arange(base + lo, base + hi)


def request_keys(wl, b: int) -> tuple[np.ndarray, np.ndarray]:
    """fp64 keys/values [L][Hkv][D] of request b, taken from the token stream."""
    base = int(np.concatenate([[0], np.cumsum(wl.seq_lens.astype(np.int64))])[b])
    L = int(wl.seq_lens[b])
    k = bf16_bits_to_f32(wl.k_tok[base : base + L]).astype(np.float64)
    v = bf16_bits_to_f32(wl.v_tok[base : base + L]).astype(np.float64)
    return k, v


def box_bound_bruteforce(q_heads: np.ndarray, keys: np.ndarray) -> float:
    """max over every corner x of the per-channel box [min keys, max keys] of q_h . x,
    summed over heads -- the tightest bound of a linear form over that box (fp64)."""
    lo, hi = keys.min(axis=0), keys.max(axis=0)
    D = keys.shape[1]
    total = 0.0
    for qh in q_heads:
        best = -np.inf
        for corner in itertools.product((0, 1), repeat=D):
            x = np.where(np.asarray(corner, dtype=bool), hi, lo)
            best = max(best, float(qh @ x))
        total += best
    return total


def check_selection(sel_idx, sel_cnt, ref_idx, ref_cnt, ref_scores, n_pages, rel=1e-4):
    """Selected page sets must agree exactly except on near-ties.

    Per (request, kv head): both sets have min(K, n) pages; a page is ambiguous
    when its fp32 oracle score is within `rel` (relative) of the oracle's K-th
    best score; every non-ambiguous page is in both sets or in neither.
    Returns the number of (request, head) rows that needed the near-tie rule."""
    B, H, K = ref_idx.shape
    tie_rows = 0
    for b in range(B):
        n = int(n_pages[b])
        m = min(K, n)
        for g in range(H):
            assert int(sel_cnt[b, g]) == m, (b, g, int(sel_cnt[b, g]), m)
            assert int(ref_cnt[b, g]) == m
            got = np.asarray(sel_idx[b, g, :m])
            ref = np.asarray(ref_idx[b, g, :m])
            assert np.all(np.asarray(sel_idx[b, g, m:]) == -1)
            assert np.all(np.diff(got) > 0), "selected pages must be strictly ascending"
            if np.array_equal(got, ref):
                continue
            s = ref_scores[b, g, :n].astype(np.float64)
            kth = np.sort(s)[::-1][m - 1]
            amb = np.abs(s - kth) < rel * np.maximum(np.abs(s), abs(kth))
            gs, rs = set(got.tolist()), set(ref.tolist())
            assert all(0 <= p < n for p in gs)
            diff = gs ^ rs
            bad = [p for p in diff if not amb[p]]
            assert not bad, (b, g, sorted(bad)[:10])
            tie_rows += 1
    return tie_rows
