"""Pins of the CPU oracle against what the method and the mathematics fix
(no GPU).  Each test checks the oracle against something other than its own
code: hand-worked values, the box-corner definition of the bound, closed
forms, an invariant, brute-force subset search and torch's scaled-dot-product
attention in fp64."""
from __future__ import annotations

import itertools
import os

import numpy as np
import pytest
import torch

import oracle
from query_aware_sparse_quest_gb300 import synth
from query_aware_sparse_quest_gb300.synth import bf16_bits_to_f32, to_bf16_bits

from helpers import bf, box_bound_bruteforce, page_tokens, request_keys

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, *v = line.split()
        vals[k] = [float(x) for x in v]
    return vals


def _explicit_cache(pages, P, D, Hkv=1):
    """Cache holding `pages` (list of [P][Hkv][D] key arrays) contiguously."""
    n = len(pages)
    cache = oracle.Cache(n, Hkv, P, D, fill_bits=0)
    k = np.concatenate([bf(np.asarray(pg, dtype=np.float64).reshape(P, Hkv, D)) for pg in pages])
    v = np.zeros_like(k)
    oracle.update_meta(cache, k, v, np.arange(n * P, dtype=np.int32))
    return cache


# ---------------------------------------------------------------- worked example

def test_worked_example_scores_and_ties():
    g = _golden()
    pages = [[[1, 3], [-1, 0]], [[2, 0], [0, 1]], [[1, -1], [0, -1]], [[2, 0], [0, 0]]]
    cache = _explicit_cache(pages, P=2, D=2)
    q = bf([[[1, -2]]])
    pt = np.arange(4, dtype=np.int32)[None]
    sl = np.array([8], dtype=np.int32)
    idx2, cnt2, s = oracle.select(cache, q, pt, sl, 2)
    assert s[0, 0].tolist() == g["caseA_scores"]
    assert idx2[0, 0].tolist() == [int(x) for x in g["caseA_top2"]] and cnt2[0, 0] == 2
    idx3, _, _ = oracle.select(cache, q, pt, sl, 3)
    assert idx3[0, 0].tolist() == [int(x) for x in g["caseA_top3"]]
    # metadata layout: [0] = kmin, [1] = kmax
    meta0 = bf16_bits_to_f32(cache.meta[0, 0])
    assert meta0[0].tolist() == [-1, 0] and meta0[1].tolist() == [1, 3]


def test_worked_example_gqa_group_sum():
    g = _golden()
    cache = _explicit_cache([[[1, 3], [-1, 0]]], P=2, D=2)
    q = bf([[[1, -2], [-0.5, 0.25]]])           # two query heads, one kv group
    _, _, s = oracle.select(cache, q, np.zeros((1, 1), np.int32), np.array([2], np.int32), 1)
    assert s[0, 0, 0] == g["caseB_score"][0]


def test_worked_example_attention():
    g = _golden()
    cache = oracle.Cache(1, 1, 2, 2, fill_bits=0)
    oracle.update_meta(cache, bf([[[1, 3]], [[-1, 0]]]), bf([[[2, 0]], [[0, 4]]]),
                       np.array([0, 1], np.int32))
    out, lse = oracle.decode(cache, bf([[[1, -2]]]), np.zeros((1, 1), np.int32),
                             np.array([2], np.int32), scale=1.0)
    np.testing.assert_allclose(out[0, 0], g["caseC_out"], rtol=1e-6)
    np.testing.assert_allclose(lse[0, 0], g["caseC_lse"][0], rtol=1e-6)


# ---------------------------------------------------------------- bound definition

def _tiny_spec(**kw):
    base = dict(name="tiny", batch=2, num_q_heads=4, num_kv_heads=2, ctx=45, budget_pages=3,
                seed=11, head_dim=4, page_size=4, shuffle_pool=True)
    base.update(kw)
    return synth.Spec(**base)


@pytest.mark.parametrize("D,P,Hq,Hkv,ctx,outlier", [
    (1, 3, 1, 1, 10, False),
    (3, 4, 4, 2, 45, True),
    (5, 2, 3, 1, 9, False),
    (6, 5, 6, 3, 23, True),
])
def test_bound_equals_box_corner_maximum(D, P, Hq, Hkv, ctx, outlier):
    """The score of a page equals, per query head, the maximum of q.x over all
    2^D corners of the page's per-channel key box, summed over the group."""
    wl = synth.make_workload(_tiny_spec(head_dim=D, page_size=P, num_q_heads=Hq, num_kv_heads=Hkv,
                                        ctx=ctx, outlier_channels=outlier, seed=D * 7 + P))
    cache = oracle.build_cache(wl, synth.UNFILLED_BITS)
    _, _, scores = oracle.select(cache, wl.q, wl.page_table, wl.seq_lens, 2)
    G = Hq // Hkv
    qf = bf16_bits_to_f32(wl.q).astype(np.float64)
    for b in range(wl.spec.batch):
        k, _ = request_keys(wl, b)
        n = -(-int(wl.seq_lens[b]) // P)
        for p in range(n):
            toks = slice(p * P, min(int(wl.seq_lens[b]), (p + 1) * P))
            for g in range(Hkv):
                want = box_bound_bruteforce(qf[b, g * G : (g + 1) * G], k[toks, g])
                np.testing.assert_allclose(scores[b, g, p], want, rtol=2e-6, atol=1e-6)


@pytest.mark.parametrize("cfg", [0, 1])
def test_bound_dominates_true_max(cfg):
    """Invariant: for every page and kv group, the bound is at least the sum
    over the group's heads of each head's largest q.k on that page (fp64)."""
    spec = synth.SPECS[cfg]
    if cfg == 1:
        spec = spec.scaled(batch=2, ctx=1000)
    wl = synth.make_workload(spec)
    cache = oracle.build_cache(wl, synth.UNFILLED_BITS)
    _, _, scores = oracle.select(cache, wl.q, wl.page_table, wl.seq_lens, spec.budget_pages)
    P, Hkv = spec.page_size, spec.num_kv_heads
    G = spec.num_q_heads // Hkv
    qf = bf16_bits_to_f32(wl.q).astype(np.float64)
    for b in range(spec.batch):
        k, _ = request_keys(wl, b)
        L = int(wl.seq_lens[b])
        n = -(-L // P)
        for g in range(Hkv):
            logits = np.einsum("hd,td->ht", qf[b, g * G : (g + 1) * G], k[:, g])   # [G][L]
            pad = n * P - L
            lp = np.pad(logits, ((0, 0), (0, pad)), constant_values=-np.inf).reshape(G, n, P)
            true_max_group = lp.max(axis=2).sum(axis=0)                              # [n]
            s = scores[b, g, :n].astype(np.float64)
            assert np.all(s >= true_max_group - 1e-5 * np.abs(s) - 1e-4)


def test_bound_closed_forms():
    """One-token page: bound = sum_h q_h.k.  Identical keys: bound = sum_h q_h.k.
    All q >= 0: bound = sum_h q_h.kmax.  All q <= 0: bound = sum_h q_h.kmin."""
    rng = np.random.default_rng(5)
    D, P = 8, 4
    keys = to_bf16_bits(rng.standard_normal((3, P, 1, D)).astype(np.float32))
    keys[1] = keys[1][0:1]                 # page 1: four identical keys
    kf = bf16_bits_to_f32(keys).astype(np.float64)
    cache = oracle.Cache(3, 1, P, D, fill_bits=0)
    T = 2 * P + 1                          # page 2 holds a single token
    oracle.update_meta(cache, keys.reshape(-1, 1, D)[:T], keys.reshape(-1, 1, D)[:T],
                       np.arange(T, dtype=np.int32))
    pt = np.arange(3, dtype=np.int32)[None]
    sl = np.array([T], np.int32)
    qmix = to_bf16_bits(rng.standard_normal((1, 2, D)).astype(np.float32))
    qpos = to_bf16_bits(np.abs(rng.standard_normal((1, 2, D))).astype(np.float32))
    qneg = to_bf16_bits(-np.abs(rng.standard_normal((1, 2, D))).astype(np.float32))
    for q in (qmix, qpos, qneg):
        qf = bf16_bits_to_f32(q).astype(np.float64)[0]
        _, _, s = oracle.select(cache, q, pt, sl, 1)
        np.testing.assert_allclose(s[0, 0, 2], (qf @ kf[2, 0, 0]).sum(), rtol=1e-6)
        np.testing.assert_allclose(s[0, 0, 1], (qf @ kf[1, 0, 0]).sum(), rtol=1e-6)
    kmax, kmin = kf[0, :, 0].max(axis=0), kf[0, :, 0].min(axis=0)
    _, _, s = oracle.select(cache, qpos, pt, sl, 1)
    np.testing.assert_allclose(s[0, 0, 0], (bf16_bits_to_f32(qpos)[0] @ kmax).sum(), rtol=1e-6)
    _, _, s = oracle.select(cache, qneg, pt, sl, 1)
    np.testing.assert_allclose(s[0, 0, 0], (bf16_bits_to_f32(qneg)[0] @ kmin).sum(), rtol=1e-6)


# ---------------------------------------------------------------- ranking

@pytest.mark.parametrize("seed", range(12))
def test_ranking_matches_bruteforce_subsets(seed):
    """Tiny integer-valued inputs (exact scores, many exact ties): the selected
    set maximises the sum of page scores over all K-subsets, and among the
    maximisers it is the lexicographically smallest index set."""
    rng = np.random.default_rng(100 + seed)
    D, P = int(rng.integers(1, 5)), int(rng.integers(1, 4))
    Hkv, G = 1, int(rng.integers(1, 3))
    n = int(rng.integers(1, 11))
    L = (n - 1) * P + int(rng.integers(1, P + 1))
    K = int(rng.integers(1, n + 2))
    k = bf(rng.integers(-3, 4, size=(L, Hkv, D)).astype(np.float64))
    q = bf(rng.integers(-2, 3, size=(1, G * Hkv, D)).astype(np.float64))
    phys = rng.permutation(n).astype(np.int32)
    cache = oracle.Cache(n, Hkv, P, D, fill_bits=0)
    pos = np.arange(L)
    oracle.update_meta(cache, k, k, (phys[pos // P] * P + pos % P).astype(np.int32))
    sel, cnt, _ = oracle.select(cache, q, phys[None], np.array([L], np.int32), K)
    kf = bf16_bits_to_f32(k).astype(np.float64)
    qf = bf16_bits_to_f32(q).astype(np.float64)[0]
    s = [box_bound_bruteforce(qf, kf[p * P : min(L, (p + 1) * P), 0]) for p in range(n)]
    m = min(K, n)
    best = max(itertools.combinations(range(n), m),
               key=lambda c: (sum(s[i] for i in c), [-i for i in c]))
    assert cnt[0, 0] == m
    assert sel[0, 0, :m].tolist() == list(best)
    assert sel[0, 0, m:].tolist() == [-1] * (K - m)


@pytest.mark.parametrize("seed", range(12))
def test_topk_alone_matches_bruteforce_subsets(seed):
    """The selection step on given scores (oracle.topk): tiny rows drawn from a
    few values (many exact ties, also +-inf): the selected set maximises the
    score sum over all K-subsets and is the lexicographically smallest such
    index set; indices ascend and the row is padded with -1."""
    rng = np.random.default_rng(300 + seed)
    rows, width = 5, 9
    K = int(rng.integers(1, width + 2))
    vals = np.array([-np.inf, -2.0, -0.5, 0.0, 0.5, 3.0, np.inf], np.float32)
    scores = vals[rng.integers(0, len(vals), size=(rows, width))]
    n = rng.integers(0, width + 1, size=rows).astype(np.int32)
    sel, cnt = oracle.topk(scores, n, K)
    for r in range(rows):
        m = min(K, int(n[r]))
        # the sum with infinities, compared exactly: more +inf first, then fewer -inf, then the finite sum
        def key(c):
            x = scores[r, list(c)]
            return (int(np.sum(x == np.inf)), -int(np.sum(x == -np.inf)), float(np.sum(x[np.isfinite(x)])),
                    [-i for i in c])
        best = max(itertools.combinations(range(int(n[r])), m), key=key)
        assert cnt[r] == m
        assert sel[r, :m].tolist() == list(best)
        assert sel[r, m:].tolist() == [-1] * (K - m)


def test_topk_alone_agrees_with_select():
    """oracle.topk on the scores oracle.select reports reproduces its selection."""
    wl = synth.make_workload(synth.SPECS[1].scaled(batch=3, ctx=16 * 37 + 5, budget_pages=9))
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    sel, cnt, scores = oracle.select(host, wl.q, wl.page_table, wl.seq_lens, 9)
    B, R, mp = scores.shape
    n = np.repeat(-(-wl.seq_lens // 16), R).astype(np.int32)
    sel2, cnt2 = oracle.topk(np.nan_to_num(scores.reshape(B * R, mp), nan=0.0), n, 9)
    assert np.array_equal(sel2.reshape(B, R, 9), sel)
    assert np.array_equal(cnt2.reshape(B, R), cnt)


# ---------------------------------------------------------------- attention

def _sdpa_fp64(q_heads, k, v, scale):
    """torch's scaled_dot_product_attention (fp64, CPU) of heads [H][D] over tokens [T][D]."""
    qt = torch.from_numpy(q_heads)[None, :, None, :]           # [1][H][1][D]
    kt = torch.from_numpy(k)[None, None].expand(1, q_heads.shape[0], -1, -1)
    vt = torch.from_numpy(v)[None, None].expand(1, q_heads.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    z = (torch.from_numpy(q_heads) @ torch.from_numpy(k).T) * scale
    return o[0, :, 0].numpy(), torch.logsumexp(z, dim=1).numpy()


@pytest.mark.parametrize("cfg,ctx,batch", [(0, 4096, 1), (0, 1000, 1), (1, 777, 2), (3, 0, 3)])
def test_dense_and_full_budget_match_sdpa(cfg, ctx, batch):
    """(a) With K >= n every page is selected and sparse attention equals dense
    attention; both equal fp64 softmax attention (torch SDPA) over the request's
    valid tokens, and lse equals the log-sum-exp of the scaled logits."""
    spec = synth.SPECS[cfg]
    if cfg == 3:
        spec = spec.scaled(batch=batch, ragged=(50, 600))
    else:
        spec = spec.scaled(batch=batch, ctx=ctx)
    wl = synth.make_workload(spec)
    cache = oracle.build_cache(wl, synth.UNFILLED_BITS)
    n_pages = -(-wl.seq_lens // spec.page_size)
    K = int(n_pages.max()) + 3
    sel, cnt, _ = oracle.select(cache, wl.q, wl.page_table, wl.seq_lens, K)
    for b in range(spec.batch):
        assert cnt[b].tolist() == [n_pages[b]] * spec.num_kv_heads
        assert sel[b, :, : n_pages[b]].tolist() == [list(range(n_pages[b]))] * spec.num_kv_heads
    out_s, lse_s = oracle.decode(cache, wl.q, wl.page_table, wl.seq_lens, sel, cnt)
    out_d, lse_d = oracle.decode(cache, wl.q, wl.page_table, wl.seq_lens)
    assert np.array_equal(out_s, out_d) and np.array_equal(lse_s, lse_d)
    scale = 1.0 / np.sqrt(spec.head_dim)
    G = spec.num_q_heads // spec.num_kv_heads
    qf = bf16_bits_to_f32(wl.q).astype(np.float64)
    for b in range(spec.batch):
        k, v = request_keys(wl, b)
        for g in range(spec.num_kv_heads):
            o_ref, l_ref = _sdpa_fp64(qf[b, g * G : (g + 1) * G], k[:, g], v[:, g], scale)
            np.testing.assert_allclose(out_d[b, g * G : (g + 1) * G], o_ref, atol=2e-5, rtol=1e-4)
            np.testing.assert_allclose(lse_d[b, g * G : (g + 1) * G], l_ref, atol=1e-5, rtol=1e-6)


def test_sparse_attention_over_page_subset_matches_sdpa():
    """Sparse attention equals fp64 softmax attention over exactly the tokens of
    the listed pages, including a partial last page (its unfilled slots hold
    large values that must not leak in)."""
    spec = synth.SPECS[1].scaled(batch=2, ctx=16 * 37 + 5, budget_pages=9)
    wl = synth.make_workload(spec)
    cache = oracle.build_cache(wl, synth.UNFILLED_BITS)
    rng = np.random.default_rng(3)
    n = 38
    Hkv, G, P = spec.num_kv_heads, spec.num_q_heads // spec.num_kv_heads, spec.page_size
    sel = np.full((2, Hkv, 9), -1, np.int32)
    cnt = np.zeros((2, Hkv), np.int32)
    for b in range(2):
        for g in range(Hkv):
            m = int(rng.integers(1, 10))
            pages = np.sort(rng.choice(n, size=m, replace=False))
            if g == 0:
                pages = np.unique(np.append(pages[: m - 1], n - 1))   # include the partial page
            sel[b, g, : len(pages)] = pages
            cnt[b, g] = len(pages)
    out, lse = oracle.decode(cache, wl.q, wl.page_table, wl.seq_lens, sel, cnt)
    qf = bf16_bits_to_f32(wl.q).astype(np.float64)
    for b in range(2):
        k, v = request_keys(wl, b)
        for g in range(Hkv):
            toks = np.concatenate([np.arange(p * P, min(int(wl.seq_lens[b]), (p + 1) * P))
                                   for p in sel[b, g, : cnt[b, g]]])
            o_ref, l_ref = _sdpa_fp64(qf[b, g * G : (g + 1) * G], k[toks, g], v[toks, g],
                                      1.0 / np.sqrt(spec.head_dim))
            np.testing.assert_allclose(out[b, g * G : (g + 1) * G], o_ref, atol=2e-5, rtol=1e-4)
            np.testing.assert_allclose(lse[b, g * G : (g + 1) * G], l_ref, atol=1e-5)


# ---------------------------------------------------------------- metadata

@pytest.mark.parametrize("chunk", [1, 3, 16, 37])
def test_update_meta_matches_page_min_max(chunk):
    """After appends of `chunk` tokens per call, every page's metadata equals the
    channel-wise min and max of the tokens appended to it (numpy reductions over
    the token stream), the pool holds each token at its slot, and unfilled
    slots are untouched."""
    spec = synth.SPECS[3].scaled(batch=3, ragged=(20, 150), head_dim=8, seed=20 + chunk)
    wl = synth.make_workload(spec)
    P, Hkv = spec.page_size, spec.num_kv_heads
    cache = oracle.Cache(wl.num_phys_pages, Hkv, P, spec.head_dim, fill_bits=synth.UNFILLED_BITS)
    T = wl.k_tok.shape[0]
    for a in range(0, T, chunk):
        e = min(T, a + chunk)
        oracle.update_meta(cache, wl.k_tok[a:e], wl.v_tok[a:e], wl.slot_mapping[a:e])
    for b in range(spec.batch):
        L = int(wl.seq_lens[b])
        for p in range(-(-L // P)):
            toks = page_tokens(wl, b, p)
            phys = wl.page_table[b, p]
            kf = bf16_bits_to_f32(wl.k_tok[toks]).astype(np.float64)      # [t][Hkv][D]
            mf = bf16_bits_to_f32(cache.meta[phys]).astype(np.float64)    # [Hkv][2][D]
            assert np.array_equal(mf[:, 0], kf.min(axis=0))
            assert np.array_equal(mf[:, 1], kf.max(axis=0))
            nv = len(toks)
            assert np.array_equal(cache.k[phys, :, :nv].transpose(1, 0, 2), wl.k_tok[toks])
            assert np.array_equal(cache.v[phys, :, :nv].transpose(1, 0, 2), wl.v_tok[toks])
            assert np.all(cache.k[phys, :, nv:] == synth.UNFILLED_BITS)


def test_needle_pages_rank_high():
    """Sanity of the generator + bound (a statistic, not a parity claim): the
    planted +8 sigma needle pages rank, on average, well inside the top quarter
    of pages.  A single needle token does not always put its page in the top-K;
    the bound sees only the part of the needle that leaves the page's key box."""
    spec = synth.SPECS[2].scaled(batch=2, ctx=16000, needles_per_request=64)
    wl = synth.make_workload(spec)
    cache = oracle.build_cache(wl, synth.UNFILLED_BITS)
    _, _, scores = oracle.select(cache, wl.q, wl.page_table, wl.seq_lens, spec.budget_pages)
    pct = []
    for b, p, _ in wl.needles:
        for g in range(spec.num_kv_heads):
            s = scores[b, g, :1000]
            pct.append(float((s > s[p]).mean()))
    assert np.mean(pct) < 0.25, np.mean(pct)


# ---------------------------------------------------------------- selection options

def _tiny_integer_case(rng, G, Hkv=1):
    D, P = int(rng.integers(1, 5)), int(rng.integers(1, 4))
    n = int(rng.integers(1, 11))
    L = (n - 1) * P + int(rng.integers(1, P + 1))
    k = bf(rng.integers(-3, 4, size=(L, Hkv, D)).astype(np.float64))
    q = bf(rng.integers(-2, 3, size=(1, G * Hkv, D)).astype(np.float64))
    phys = rng.permutation(n).astype(np.int32)
    cache = oracle.Cache(n, Hkv, P, D, fill_bits=0)
    pos = np.arange(L)
    oracle.update_meta(cache, k, k, (phys[pos // P] * P + pos % P).astype(np.int32))
    return cache, q, phys, L, n, P, bf16_bits_to_f32(k).astype(np.float64), bf16_bits_to_f32(q).astype(np.float64)[0]


def _best_subset(scores, m, candidates):
    """Lexicographically smallest m-subset of `candidates` with the largest score sum."""
    return max(itertools.combinations(candidates, m), key=lambda c: (sum(scores[i] for i in c), [-i for i in c]))


@pytest.mark.parametrize("seed", range(10))
def test_per_q_head_selection_matches_bruteforce(seed):
    """Per-query-head selection: each head's scores are its own box bound and
    its page set is the best K-subset under that head's scores alone."""
    rng = np.random.default_rng(300 + seed)
    G = int(rng.integers(1, 4))
    cache, q, phys, L, n, P, kf, qf = _tiny_integer_case(rng, G)
    K = int(rng.integers(1, n + 2))
    sel, cnt, sc = oracle.select(cache, q, phys[None], np.array([L], np.int32), K, per_q_head=True)
    assert sel.shape == (1, G, K)
    m = min(K, n)
    for h in range(G):
        s = [box_bound_bruteforce(qf[h : h + 1], kf[p * P : min(L, (p + 1) * P), 0]) for p in range(n)]
        np.testing.assert_allclose(sc[0, h, :n], s, rtol=0, atol=0)
        assert cnt[0, h] == m
        assert sel[0, h, :m].tolist() == list(_best_subset(s, m, range(n)))


def test_per_q_head_with_one_head_per_group_equals_group_selection():
    wl = synth.make_workload(_tiny_spec(num_q_heads=2, num_kv_heads=2, ctx=60, seed=21))
    cache = oracle.build_cache(wl, synth.UNFILLED_BITS)
    a = oracle.select(cache, wl.q, wl.page_table, wl.seq_lens, 4)
    b = oracle.select(cache, wl.q, wl.page_table, wl.seq_lens, 4, per_q_head=True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("seed", range(12))
def test_sink_and_window_pages_always_kept(seed):
    """Forced pages: the first S and last W pages rank first (lower index first
    among them); the rest of the budget is the best subset of the other pages."""
    rng = np.random.default_rng(400 + seed)
    cache, q, phys, L, n, P, kf, qf = _tiny_integer_case(rng, G=2)
    K = int(rng.integers(1, n + 2))
    S, W = int(rng.integers(0, 3)), int(rng.integers(0, 3))
    sel, cnt, sc = oracle.select(cache, q, phys[None], np.array([L], np.int32), K, sink_pages=S, window_pages=W)
    s = [box_bound_bruteforce(qf, kf[p * P : min(L, (p + 1) * P), 0]) for p in range(n)]
    np.testing.assert_allclose(sc[0, 0, :n], s, rtol=0, atol=0)   # scores stay the bound
    forced = [p for p in range(n) if p < S or p >= n - W]
    others = [p for p in range(n) if p not in forced]
    m = min(K, n)
    keep = forced[:m]
    keep += list(_best_subset(s, m - len(keep), others)) if m > len(keep) else []
    assert cnt[0, 0] == m
    assert sel[0, 0, :m].tolist() == sorted(keep)
    assert sel[0, 0, m:].tolist() == [-1] * (K - m)


def test_per_q_head_decode_matches_sdpa_per_head():
    """Attention with one page list per query head equals, head by head, fp64
    scaled-dot-product attention over that head's pages; with every head of a
    group given the group's list it equals group-row attention."""
    wl = synth.make_workload(_tiny_spec(num_q_heads=4, num_kv_heads=2, ctx=70, seed=31, head_dim=8))
    cache = oracle.build_cache(wl, synth.UNFILLED_BITS)
    sel, cnt, _ = oracle.select(cache, wl.q, wl.page_table, wl.seq_lens, 3, per_q_head=True)
    scale = 0.3
    out, lse = oracle.decode(cache, wl.q, wl.page_table, wl.seq_lens, sel, cnt, scale=scale, per_q_head=True)
    P, G = wl.spec.page_size, 2
    qf = bf16_bits_to_f32(wl.q).astype(np.float64)
    for b in range(wl.spec.batch):
        k, v = request_keys(wl, b)
        for h in range(4):
            toks = np.concatenate([np.arange(p * P, min(int(wl.seq_lens[b]), (p + 1) * P))
                                   for p in sel[b, h, : cnt[b, h]]])
            o_ref, l_ref = _sdpa_fp64(qf[b, h : h + 1], k[toks, h // G], v[toks, h // G], scale)
            np.testing.assert_allclose(out[b, h], o_ref[0], rtol=2e-5, atol=2e-6)
            np.testing.assert_allclose(lse[b, h], l_ref[0], rtol=2e-6, atol=2e-6)
    gsel, gcnt, _ = oracle.select(cache, wl.q, wl.page_table, wl.seq_lens, 3)
    rep_sel, rep_cnt = np.repeat(gsel, G, axis=1), np.repeat(gcnt, G, axis=1)
    o1, l1 = oracle.decode(cache, wl.q, wl.page_table, wl.seq_lens, rep_sel, rep_cnt, scale=scale, per_q_head=True)
    o2, l2 = oracle.decode(cache, wl.q, wl.page_table, wl.seq_lens, gsel, gcnt, scale=scale)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ---------------------------------------------------------------- FP8 (e4m3) pages

def test_e4m3_codec_matches_torch_and_the_format():
    """Encoding agrees with torch's float8_e4m3fn cast (round to nearest even)
    on in-range values; decoding follows the format's definition; every
    finite code round-trips; out-of-range values saturate to +-448."""
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.uniform(-448, 448, 4000), rng.standard_normal(4000) * 0.01,
                         rng.standard_normal(2000) * 2.0 ** -8, [0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10,
                                                                   1.0625, 1.1875, 3 * 2.0 ** -10, 440.0, 447.9]])
    xs = xs.astype(np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(x) for x in xs], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)
    # decoding from the definition: sign, exponent bias 7, 3 mantissa bits, subnormals m * 2^-9
    assert oracle.e4m3_value(0x38) == 1.0 and oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9 and oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0xC5) == -3.25 and np.isnan(oracle.e4m3_value(0x7F))
    finite = [c for c in range(256) if c & 0x7F != 0x7F]
    vals = torch.tensor(finite, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c, v in zip(finite, vals):
        assert oracle.e4m3_value(c) == v
        assert oracle.e4m3_encode(v) == c
    for big in (448.5, 464.0, 500.0, 1e30):
        assert oracle.e4m3_encode(big) == 0x7E and oracle.e4m3_encode(-big) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_fp8_rows_and_attention():
    """Row scales are amax / 448 and the row's largest element codes to +-448;
    every decoded element is within half an e4m3 spacing (x scale) of the
    appended value; attention over an fp8 pool equals fp64 scaled-dot-product
    attention over the decoded rows; the metadata is the bf16 pool's."""
    spec = _tiny_spec(num_q_heads=4, num_kv_heads=2, ctx=70, seed=41, head_dim=8)
    wl = synth.make_workload(spec)
    c8 = oracle.build_cache(wl, synth.UNFILLED_BITS, fp8=True)
    c16 = oracle.build_cache(wl, synth.UNFILLED_BITS)
    np.testing.assert_array_equal(c8.meta, c16.meta)
    P = spec.page_size
    dec = lambda codes: torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    for t in range(wl.k_tok.shape[0]):
        slot = int(wl.slot_mapping[t])
        for h in range(spec.num_kv_heads):
            for raw, codes, scales in ((wl.k_tok, c8.k8, c8.ks), (wl.v_tok, c8.v8, c8.vs)):
                x = bf16_bits_to_f32(raw[t, h]).astype(np.float64)
                s = float(scales[slot // P, h, slot % P])
                amax = np.abs(x).max()
                assert s == np.float32(np.float32(amax) / np.float32(448.0))
                y = dec(codes[slot // P, h, slot % P]) * s
                if amax > 0:
                    assert np.abs(dec(codes[slot // P, h, slot % P])).max() == 448.0
                spacing = 2.0 ** (np.maximum(np.floor(np.log2(np.maximum(np.abs(x) / s, 2.0 ** -6))), -6) - 3)
                assert np.all(np.abs(y - x) <= 0.5 * spacing * s * (1 + 1e-6) + 1e-30)
    sel, cnt, _ = oracle.select(c8, wl.q, wl.page_table, wl.seq_lens, 3)
    out, lse = oracle.decode(c8, wl.q, wl.page_table, wl.seq_lens, sel, cnt, scale=0.3)
    G = 2
    qf = bf16_bits_to_f32(wl.q).astype(np.float64)
    kd = dec(c8.k8) * c8.ks[..., None].astype(np.float64)
    vd = dec(c8.v8) * c8.vs[..., None].astype(np.float64)
    for b in range(spec.batch):
        L = int(wl.seq_lens[b])
        for h in range(4):
            g = h // G
            rows = [(int(wl.page_table[b, p]), o) for p in sel[b, g, : cnt[b, g]]
                    for o in range(min(P, L - p * P))]
            k = np.stack([kd[ph, g, o] for ph, o in rows])
            v = np.stack([vd[ph, g, o] for ph, o in rows])
            o_ref, l_ref = _sdpa_fp64(qf[b, h : h + 1], k, v, 0.3)
            np.testing.assert_allclose(out[b, h], o_ref[0], rtol=2e-5, atol=2e-6)
            np.testing.assert_allclose(lse[b, h], l_ref[0], rtol=2e-6, atol=2e-6)


def test_openmp_build_matches_the_plain_build_bit_for_bit():
    """The OpenMP build only hands independent rows (request, head) to the
    host's threads: selections, scores, outputs and lse equal the plain
    build's bit for bit, on a ragged batch with partial last pages, dense and
    sparse, group and per-query-head rows."""
    wl = synth.make_workload(synth.SPECS[3].scaled(batch=5, ragged=(16 * 30 + 3, 16 * 90 + 11),
                                                   budget_pages=12))
    host = oracle.build_cache(wl, synth.UNFILLED_BITS)
    args = (host, wl.q, wl.page_table, wl.seq_lens)

    def run():
        res = []
        for per_head in (False, True):
            sel, cnt, sc = oracle.select(*args, wl.spec.budget_pages, per_q_head=per_head)
            res += [sel, cnt, sc, *oracle.decode(*args, sel, cnt, per_q_head=per_head)]
        res += list(oracle.decode(*args))
        return res

    plain = run()
    with oracle.parallel() as threads:
        assert threads >= 1
        par = run()
    assert oracle.num_threads() == 1
    for a, b in zip(plain, par):
        assert a.dtype == b.dtype and a.shape == b.shape
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
