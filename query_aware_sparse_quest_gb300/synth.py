"""Seeded synthetic decode workloads for query-aware (Quest-style) sparse decode.

This module only draws inputs: bf16 bit patterns for queries, keys and values,
the order in which tokens are appended to the paged pool, page tables and
sequence lengths.  It holds none of the method's arithmetic (no page bounds, no
selection, no attention) so that the CUDA path and the CPU oracle can both be
fed from it without sharing any computation.

Workload shapes follow the long-context decode geometry the pages describe:
Qwen3-30B-A3B attention (32 query heads, 4 kv heads, head_dim 128), pages of
16 tokens, contexts up to 128k tokens at batch 8 (the benchmark command in the
"add-sparse-method" skill, section "Validation": --lengths 128000
--batch_sizes 8).  No dataset is used: the pages measure on LongBench and on
their own bench script, and these seeded draws stand in for them.

Recipe (all values drawn in fp32, rounded to bf16 round-to-nearest-even):
  * q ~ N(0, 1) per element.
  * K ~ N(0, 1), optionally times a per-(kv head, channel) scale
    c = exp(N(0, 1)) shared by every token and request (outlier channels).
  * V ~ N(0, 1).
  * needles: a chosen token of a chosen page gets, for every kv head g, its key
    moved so that u.k = 8 sigma_u, where u is the sum of the group's query
    heads and sigma_u = sqrt(sum_i u_i^2 c_i^2) is the std of u.k under the
    key distribution.  The key's component orthogonal to u is kept.
  * physical pages are either contiguous per request or a random permutation
    of one shared pool.
  * pool slots past a request's last token hold a fixed large value so that a
    missing mask shows up as a large error.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Tuple

import numpy as np
import torch

PAGE_SIZE = 16
HEAD_DIM = 128
# bf16 bit pattern of 100.0, written to pool slots that hold no token.
UNFILLED_BITS = 0x42C8

# Sub-stream roles; each draws from its own SeedSequence child so that the
# order in which arrays are generated never changes their contents.
_ROLE_Q, _ROLE_K, _ROLE_V, _ROLE_SCALE, _ROLE_NEEDLE, _ROLE_LENS, _ROLE_PERM, _ROLE_STEP = range(8)
_CHUNK_TOKENS = 8192


@dataclasses.dataclass(frozen=True)
class Spec:
    """Shape and structure of one decode workload."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    ctx: int                          # context length (ignored when ragged is set)
    budget_pages: int                 # top-K pages kept per (request, kv head)
    seed: int
    ragged: Optional[Tuple[int, int]] = None   # inclusive uniform range of lengths
    needles_per_request: int = 0      # needle tokens, each in a distinct page
    outlier_channels: bool = False    # K scaled by exp(N(0,1)) per channel
    shuffle_pool: bool = False        # random physical page permutation
    append_steps: int = 0             # decode steps appending one token/request
    budget_sweep: Tuple[int, ...] = ()  # extra budgets (pages) swept per step
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE

    def scaled(self, **kw) -> "Spec":
        return dataclasses.replace(self, **kw)


# The five decode workloads (tiny parity case, Qwen3-30B-A3B geometry at 32k,
# the 128k batch-8 benchmark, a ragged serving batch, and an append + budget
# sweep step).  Budgets are in pages of 16 tokens.
SPECS = {
    0: Spec("tiny_b1_ctx4096_gqa4", batch=1, num_q_heads=4, num_kv_heads=1, ctx=4096,
            budget_pages=64, seed=0, needles_per_request=3),
    1: Spec("qwen3_b8_ctx32768_budget2048", batch=8, num_q_heads=32, num_kv_heads=4, ctx=32768,
            budget_pages=2048 // 16, seed=1, outlier_channels=True),
    2: Spec("qwen3_b8_ctx128000_budget4096", batch=8, num_q_heads=32, num_kv_heads=4, ctx=128000,
            budget_pages=4096 // 16, seed=2, outlier_channels=True, needles_per_request=64,
            shuffle_pool=True),
    3: Spec("ragged_b32_ctx8k-128k_budget2048", batch=32, num_q_heads=32, num_kv_heads=4, ctx=0,
            ragged=(8192, 131072), budget_pages=2048 // 16, seed=3, outlier_channels=True,
            shuffle_pool=True),
    4: Spec("append_b16_ctx65536_sweep", batch=16, num_q_heads=32, num_kv_heads=4, ctx=65536,
            budget_pages=2048 // 16, seed=4, outlier_channels=True, shuffle_pool=True,
            append_steps=1, budget_sweep=(512 // 16, 1024 // 16, 2048 // 16, 4096 // 16, 8192 // 16)),
}


@dataclasses.dataclass
class Workload:
    """Host arrays of one workload (bf16 data as uint16 bit patterns)."""

    spec: Spec
    q: np.ndarray               # uint16 [B][Hq][D]   decode query after the prefill
    k_tok: np.ndarray           # uint16 [T][Hkv][D]  prefill keys in append order
    v_tok: np.ndarray           # uint16 [T][Hkv][D]
    slot_mapping: np.ndarray    # int32 [T]  physical slot = page * P + offset
    tok_request: np.ndarray     # int32 [T]  request of each appended token
    page_table: np.ndarray      # int32 [B][max_pages] logical -> physical page
    seq_lens: np.ndarray        # int32 [B]  tokens after the prefill
    num_phys_pages: int
    k_scale: np.ndarray         # float32 [Hkv][D] per-channel key scale (ones if none)
    needles: np.ndarray         # int32 [N][3] (request, logical page, offset)
    # Decode steps that append one token per request (empty when append_steps == 0).
    step_q: np.ndarray          # uint16 [S][B][Hq][D]
    step_k: np.ndarray          # uint16 [S][B][Hkv][D]
    step_v: np.ndarray          # uint16 [S][B][Hkv][D]
    step_slots: np.ndarray      # int32 [S][B]

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    def prefill_chunks(self, chunk_tokens: int = 4096):
        """Yield (start, end) token ranges of a chunked prefill.

        Chunks never split a page across two calls out of order: tokens stay in
        append order, so pages fill without holes."""
        T = self.k_tok.shape[0]
        for s in range(0, T, chunk_tokens):
            yield s, min(T, s + chunk_tokens)

    def seq_lens_after(self, steps: int) -> np.ndarray:
        return (self.seq_lens + steps).astype(np.int32)


def _child(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(entropy=seed, spawn_key=tuple(key)))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32/fp64 -> bf16 bit patterns, round to nearest even (torch's conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(seed: int, role: int, n_tok: int, width: int, scale: Optional[np.ndarray]) -> np.ndarray:
    """n_tok rows of `width` N(0,1) values (times `scale` per column), as bf16 bits.

    Drawn in fixed chunks of tokens, each from its own seed child, in parallel."""
    out = np.empty((n_tok, width), dtype=np.uint16)
    n_chunks = (n_tok + _CHUNK_TOKENS - 1) // _CHUNK_TOKENS

    def work(c: int) -> None:
        s, e = c * _CHUNK_TOKENS, min(n_tok, (c + 1) * _CHUNK_TOKENS)
        x = _child(seed, role, c).standard_normal((e - s, width), dtype=np.float32)
        if scale is not None:
            x *= scale
        out[s:e] = to_bf16_bits(x)

    workers = max(1, min(16, os.cpu_count() or 1))
    if n_chunks <= 1:
        for c in range(n_chunks):
            work(c)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(work, range(n_chunks)))
    return out


def make_workload(spec: Spec) -> Workload:
    B, Hq, Hkv, D, P = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.page_size
    assert Hq % Hkv == 0
    G = Hq // Hkv
    S = spec.append_steps

    # Sequence lengths.
    if spec.ragged is not None:
        lo, hi = spec.ragged
        seq_lens = _child(spec.seed, _ROLE_LENS).integers(lo, hi, size=B, endpoint=True).astype(np.int32)
    else:
        seq_lens = np.full(B, spec.ctx, dtype=np.int32)
    if np.any(seq_lens < 1):
        raise ValueError("every request needs at least one token")

    # Logical pages per request, including room for the appended tokens.
    pages_final = (seq_lens.astype(np.int64) + S + P - 1) // P
    max_pages = int(pages_final.max())
    n_phys = int(pages_final.sum())
    page_base = np.concatenate([[0], np.cumsum(pages_final)[:-1]]).astype(np.int64)
    if spec.shuffle_pool:
        perm = _child(spec.seed, _ROLE_PERM).permutation(n_phys).astype(np.int32)
    else:
        perm = np.arange(n_phys, dtype=np.int32)
    # Unused tail entries point at a valid page (0) so that a stray read stays in bounds.
    page_table = np.zeros((B, max_pages), dtype=np.int32)
    for b in range(B):
        page_table[b, : pages_final[b]] = perm[page_base[b] : page_base[b] + pages_final[b]]

    # Key channel scale.
    if spec.outlier_channels:
        k_scale = np.exp(_child(spec.seed, _ROLE_SCALE).standard_normal((Hkv, D))).astype(np.float32)
    else:
        k_scale = np.ones((Hkv, D), dtype=np.float32)

    # Decode query.
    q = _normal_bf16(spec.seed, _ROLE_Q, B, Hq * D, None).reshape(B, Hq, D)

    # Prefill token stream: request-major, logical order.
    T = int(seq_lens.sum())
    k_tok = _normal_bf16(spec.seed, _ROLE_K, T, Hkv * D,
                         k_scale.reshape(-1) if spec.outlier_channels else None).reshape(T, Hkv, D)
    v_tok = _normal_bf16(spec.seed, _ROLE_V, T, Hkv * D, None).reshape(T, Hkv, D)
    tok_base = np.concatenate([[0], np.cumsum(seq_lens.astype(np.int64))[:-1]])
    slot_mapping = np.empty(T, dtype=np.int32)
    tok_request = np.empty(T, dtype=np.int32)
    for b in range(B):
        L = int(seq_lens[b])
        pos = np.arange(L, dtype=np.int64)
        slot_mapping[tok_base[b] : tok_base[b] + L] = page_table[b, pos // P].astype(np.int64) * P + pos % P
        tok_request[tok_base[b] : tok_base[b] + L] = b

    # Needles: one token in each of `needles_per_request` distinct pages.
    needles = np.zeros((0, 3), dtype=np.int32)
    if spec.needles_per_request:
        rng = _child(spec.seed, _ROLE_NEEDLE)
        rows = []
        qf = bf16_bits_to_f32(q).astype(np.float64)
        for b in range(B):
            L = int(seq_lens[b])
            n_pages = (L + P - 1) // P
            pages = np.sort(rng.choice(n_pages, size=spec.needles_per_request, replace=False))
            for p in pages:
                valid = min(P, L - int(p) * P)
                off = int(rng.integers(0, valid))
                rows.append((b, int(p), off))
                t = int(tok_base[b]) + int(p) * P + off
                for g in range(Hkv):
                    u = qf[b, g * G : (g + 1) * G].sum(axis=0)
                    k = bf16_bits_to_f32(k_tok[t, g]).astype(np.float64)
                    sigma_u = float(np.sqrt(np.sum((u * k_scale[g]) ** 2)))
                    uu = float(u @ u)
                    k_new = k - (u @ k) / uu * u + 8.0 * sigma_u * u / uu
                    k_tok[t, g] = to_bf16_bits(k_new)
        needles = np.asarray(rows, dtype=np.int32).reshape(-1, 3)

    # Appended decode steps.
    if S:
        step_q = _normal_bf16(spec.seed, _ROLE_STEP, S * B, Hq * D, None).reshape(S, B, Hq, D)
        step_k = _normal_bf16(spec.seed, _ROLE_STEP + 1, S * B, Hkv * D,
                              k_scale.reshape(-1) if spec.outlier_channels else None).reshape(S, B, Hkv, D)
        step_v = _normal_bf16(spec.seed, _ROLE_STEP + 2, S * B, Hkv * D, None).reshape(S, B, Hkv, D)
        step_slots = np.empty((S, B), dtype=np.int32)
        for s in range(S):
            pos = seq_lens.astype(np.int64) + s
            step_slots[s] = page_table[np.arange(B), pos // P].astype(np.int64) * P + pos % P
    else:
        step_q = np.zeros((0, B, Hq, D), dtype=np.uint16)
        step_k = np.zeros((0, B, Hkv, D), dtype=np.uint16)
        step_v = np.zeros((0, B, Hkv, D), dtype=np.uint16)
        step_slots = np.zeros((0, B), dtype=np.int32)

    return Workload(spec=spec, q=q, k_tok=k_tok, v_tok=v_tok, slot_mapping=slot_mapping,
                    tok_request=tok_request, page_table=page_table, seq_lens=seq_lens,
                    num_phys_pages=n_phys, k_scale=k_scale, needles=needles,
                    step_q=step_q, step_k=step_k, step_v=step_v, step_slots=step_slots)
