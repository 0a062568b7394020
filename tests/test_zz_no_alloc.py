"""sv_sparse_decode_static_scratch: the decode entry point for callers that
cannot allocate device memory (a host framework that owns every allocation,
or a serving loop that reserved HBM up front).  Its scratch is an array
compiled into the library, so these tests check, through the C ABI, that it
gives the same outputs as sv_sparse_decode with a caller workspace on two
calls in a row (sparse, then dense over the same shared array), and that it
refuses problems whose partials would not fit the array."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from query_aware_sparse_quest_gb300 import binding, build, resident, synth

pytestmark = pytest.mark.gpu

OUT_ATOL = 2e-2
LSE_ATOL = 1e-3


def _decode_with_workspace(dw, sel_idx, sel_cnt):
    B, Hq, D = dw.q.shape
    pages = dw.page_table.shape[1] if sel_idx is None else sel_idx.shape[2]
    ws = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, dw.cache.num_kv_heads, pages))
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    binding.sv_sparse_decode(dw.cache, dw.q, dw.page_table, dw.seq_lens, sel_idx, sel_cnt, out, lse, ws)
    return out, lse


def _decode_static(dw, sel_idx, sel_cnt):
    B, Hq, D = dw.q.shape
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    binding.sv_sparse_decode_static_scratch(dw.cache, dw.q, dw.page_table, dw.seq_lens, sel_idx, sel_cnt, out, lse)
    return out, lse


def _close(a, b):
    (out_a, lse_a), (out_b, lse_b) = a, b
    assert float((out_a.float() - out_b.float()).abs().max()) <= OUT_ATOL
    assert float((lse_a - lse_b).abs().max()) <= LSE_ATOL


def test_static_scratch_matches_workspace_decode(cuda_ok):
    build.build()
    spec = synth.SPECS[2].scaled(batch=8, ctx=16 * 700 + 9, needles_per_request=8)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl)
    K = spec.budget_pages
    sel_idx, sel_cnt = resident.select_buffers(spec.batch, spec.num_kv_heads, K)
    ws = resident.workspace(binding.sv_quest_select_workspace_size(spec.batch, spec.num_kv_heads, wl.max_pages))
    binding.sv_quest_select(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, sel_idx, sel_cnt, workspace=ws)

    # Call 1: sparse.  Call 2: dense, reusing the array the first call filled.
    ref_sparse = _decode_with_workspace(dw, sel_idx, sel_cnt)
    ref_dense = _decode_with_workspace(dw, None, None)
    got_sparse = _decode_static(dw, sel_idx, sel_cnt)
    got_dense = _decode_static(dw, None, None)
    torch.cuda.synchronize()
    _close(got_sparse, ref_sparse)
    _close(got_dense, ref_dense)
    # And once more in the first order, after the dense call left its partials behind.
    _close(_decode_static(dw, sel_idx, sel_cnt), ref_sparse)
    torch.cuda.synchronize()
    assert binding.sv_get_device_error(reset=True) == 0


def test_static_scratch_rejects_oversized_problems(cuda_ok):
    build.build()
    lib = binding.raw_library()
    # batch 32 x 32 query heads over 8192 pages needs 64 splits of partials: 34 MB > 16 MiB.
    need = binding.sv_sparse_decode_workspace_size(32, 32, 4, 8192)
    assert need > 16 << 20
    # Null pools and buffers: the size check comes first and returns
    # SV_ERR_WORKSPACE; were it ever skipped, the decode's own argument checks
    # would return SV_ERR_INVALID_ARG (1) on the nulls, so nothing can launch.
    cache = binding.sv_cache(None, None, None, 1000, 4, 16, 128)
    st = lib.sv_sparse_decode_static_scratch(ctypes.byref(cache), None, 32, None, None, 32, 8192, None, None, 0,
                                             0.088, None, None, None)
    assert st == 3    # SV_ERR_WORKSPACE, nothing launched
    # The largest batch-32 sparse problem that fits (248 pages) is accepted by the size check.
    assert binding.sv_sparse_decode_workspace_size(32, 32, 4, 248) <= 16 << 20
    assert binding.sv_sparse_decode_workspace_size(32, 32, 4, 256) > 16 << 20
