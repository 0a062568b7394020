"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks reject bad calls before any launch (no GPU needed)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch  # noqa: F401  (loads the CUDA runtime the library links against)

from query_aware_sparse_quest_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "svquest.h")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_WORKSPACE = 0, 1, 2, 3


# The argument-check tests below pass made-up device addresses: the checks
# under test reject them before any launch, but if a check regressed on a
# machine with a GPU the library would launch kernels on those addresses.
# They therefore run only where no GPU is visible (the CPU suite), where a
# launch cannot reach a device.
host_only = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="fake device addresses; host-only checks run without a GPU")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.raw_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_\w+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("sv_quest_update_meta", "sv_quest_select", "sv_sparse_decode"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert binding.sv_status_string(0) == "SV_OK"
    for st in (1, 2, 3, 4):
        assert binding.sv_status_string(st).startswith("SV_ERR")
    assert binding.sv_version() >= 100


def test_workspace_sizes(lib):
    # scores: B * Hkv * max_pages fp32, rounded up to 256 bytes
    assert binding.sv_quest_select_workspace_size(8, 4, 8000) == 8 * 4 * 8000 * 4
    assert binding.sv_quest_select_workspace_size(1, 1, 3) == 256
    assert binding.sv_quest_select_workspace_size(0, 4, 10) == 0
    # decode partials: at most 64 splits, at least 8 pages per split
    ws = binding.sv_sparse_decode_workspace_size(8, 32, 4, 256)
    assert ws >= 8 * 32 * 32 * (128 * 4 + 8)
    assert binding.sv_sparse_decode_workspace_size(8, 32, 4, 8000) >= 8 * 32 * 64 * 128 * 4
    assert binding.sv_sparse_decode_workspace_size(1, 4, 1, 1) >= 4 * (128 * 4 + 8)


def _fake_cache(page_size=16, head_dim=128, hkv=4, pages=10, null=False):
    # Host-side checks only read the struct; these addresses are never dereferenced.
    addr = 0 if null else 0x10000
    return binding.sv_cache(addr, addr, addr, pages, hkv, page_size, head_dim)


FAKE = ctypes.c_void_p(0x20000)


@host_only
@pytest.mark.parametrize("cache,hq,expect", [
    (_fake_cache(null=True), 32, SV_ERR_INVALID_ARG),
    (_fake_cache(page_size=32), 32, SV_ERR_UNSUPPORTED),
    (_fake_cache(head_dim=64), 32, SV_ERR_UNSUPPORTED),
    (_fake_cache(hkv=4), 30, SV_ERR_INVALID_ARG),       # Hq not a multiple of Hkv
    (_fake_cache(hkv=1), 16, SV_ERR_UNSUPPORTED),       # 16 query heads per kv head
    (_fake_cache(pages=0), 32, SV_ERR_INVALID_ARG),
])
def test_select_rejects_bad_geometry(lib, cache, hq, expect):
    st = lib.sv_quest_select(ctypes.byref(cache), FAKE, hq, FAKE, FAKE, 8, 100, 16, FAKE, FAKE, None,
                             FAKE, 1 << 20, None)
    assert st == expect


@host_only
def test_select_rejects_bad_sizes(lib):
    c = ctypes.byref(_fake_cache())
    assert lib.sv_quest_select(c, None, 32, FAKE, FAKE, 8, 100, 16, FAKE, FAKE, None, FAKE, 1 << 20, None) == SV_ERR_INVALID_ARG
    assert lib.sv_quest_select(c, FAKE, 32, FAKE, FAKE, 0, 100, 16, FAKE, FAKE, None, FAKE, 1 << 20, None) == SV_ERR_INVALID_ARG
    assert lib.sv_quest_select(c, FAKE, 32, FAKE, FAKE, 8, 100, 0, FAKE, FAKE, None, FAKE, 1 << 20, None) == SV_ERR_INVALID_ARG
    assert lib.sv_quest_select(c, FAKE, 32, FAKE, FAKE, 8, 40000, 16, FAKE, FAKE, None, FAKE, 1 << 30, None) == SV_ERR_UNSUPPORTED
    # scores need 8*4*100*4 bytes of workspace when scores_out is NULL
    assert lib.sv_quest_select(c, FAKE, 32, FAKE, FAKE, 8, 100, 16, FAKE, FAKE, None, FAKE, 100, None) == SV_ERR_WORKSPACE
    assert lib.sv_quest_select(c, FAKE, 32, FAKE, FAKE, 8, 100, 16, FAKE, FAKE, None, None, 1 << 20, None) == SV_ERR_WORKSPACE
    # misaligned q
    assert lib.sv_quest_select(c, ctypes.c_void_p(0x20002), 32, FAKE, FAKE, 8, 100, 16, FAKE, FAKE, None, FAKE,
                               1 << 20, None) == SV_ERR_INVALID_ARG


@host_only
def test_topk_rejects_bad_args(lib):
    assert lib.sv_quest_topk(None, FAKE, 8, 4, 100, 16, FAKE, FAKE, None) == SV_ERR_INVALID_ARG
    assert lib.sv_quest_topk(FAKE, FAKE, 8, 4, 100, 0, FAKE, FAKE, None) == SV_ERR_INVALID_ARG
    assert lib.sv_quest_topk(FAKE, FAKE, 8, 4, 32769, 16, FAKE, FAKE, None) == SV_ERR_UNSUPPORTED


@host_only
def test_decode_rejects_bad_args(lib):
    c = ctypes.byref(_fake_cache())
    ok = dict(q=FAKE, pt=FAKE, sl=FAKE, out=FAKE, lse=FAKE, ws=FAKE)

    def call(scale=0.088, sel=None, cnt=None, K=0, ws=FAKE, out=FAKE, hq=32, batch=8):
        return lib.sv_sparse_decode(c, ok["q"], hq, ok["pt"], ok["sl"], batch, 100, sel, cnt, K, scale, out,
                                    ok["lse"], ws, 1 << 20, None)
    assert call(out=None) == SV_ERR_INVALID_ARG
    assert call(scale=0.0) == SV_ERR_INVALID_ARG
    assert call(scale=float("nan")) == SV_ERR_INVALID_ARG
    assert call(sel=FAKE, cnt=None, K=16) == SV_ERR_INVALID_ARG
    assert call(sel=FAKE, cnt=FAKE, K=0) == SV_ERR_INVALID_ARG
    assert call(ws=None) == SV_ERR_WORKSPACE
    assert call(hq=33) == SV_ERR_INVALID_ARG
    # out and the workspace are moved 16 bytes at a time
    assert call(out=ctypes.c_void_p(0x20008)) == SV_ERR_INVALID_ARG
    assert call(ws=ctypes.c_void_p(0x20004)) == SV_ERR_INVALID_ARG


@host_only
def test_update_meta_rejects_bad_args(lib):
    c = ctypes.byref(_fake_cache())
    assert lib.sv_quest_update_meta(c, FAKE, FAKE, FAKE, -1, None) == SV_ERR_INVALID_ARG
    assert lib.sv_quest_update_meta(c, FAKE, FAKE, FAKE, 0, None) == SV_OK       # no-op, nothing launched
    assert lib.sv_quest_update_meta(c, None, FAKE, FAKE, 4, None) == SV_ERR_INVALID_ARG
    bad = ctypes.byref(_fake_cache(page_size=8))
    assert lib.sv_quest_update_meta(bad, FAKE, FAKE, FAKE, 4, None) == SV_ERR_UNSUPPORTED


def test_decode_step_workspace_size(lib):
    f = binding.sv_quest_decode_step_workspace_size
    # select scores + sparse-decode partials
    for args in ((8, 32, 4, 8000, 256), (2, 8, 1, 9000, 64), (32, 32, 4, 8192, 128)):
        B, Hq, Hkv, mp, K = args
        assert f(*args) >= (binding.sv_quest_select_workspace_size(B, Hkv, mp)
                            + binding.sv_sparse_decode_workspace_size(B, Hq, Hkv, K))
    assert f(8, 32, 4, 8000, 256) < f(8, 32, 4, 8000, 512)
    assert f(0, 32, 4, 100, 16) == 0
    assert f(8, 32, 4, 100, 0) == 0


@host_only
def test_decode_step_rejects_bad_args(lib):
    c = ctypes.byref(_fake_cache())

    def call(q=FAKE, hq=32, batch=8, max_pages=100, K=16, scale=0.088, sel=FAKE, cnt=FAKE, out=FAKE,
             lse=FAKE, ws=FAKE, ws_bytes=1 << 30, cache=c):
        return lib.sv_quest_decode_step(cache, q, hq, FAKE, FAKE, batch, max_pages, K, scale, sel, cnt, out, lse,
                                        ws, ws_bytes, None)
    assert call(q=None) == SV_ERR_INVALID_ARG
    assert call(sel=None) == SV_ERR_INVALID_ARG
    assert call(cnt=None) == SV_ERR_INVALID_ARG
    assert call(out=None) == SV_ERR_INVALID_ARG
    assert call(lse=None) == SV_ERR_INVALID_ARG
    assert call(K=0) == SV_ERR_INVALID_ARG
    assert call(batch=0) == SV_ERR_INVALID_ARG
    assert call(scale=0.0) == SV_ERR_INVALID_ARG
    assert call(scale=float("inf")) == SV_ERR_INVALID_ARG
    assert call(hq=30) == SV_ERR_INVALID_ARG
    assert call(max_pages=40000) == SV_ERR_UNSUPPORTED
    assert call(cache=ctypes.byref(_fake_cache(page_size=32))) == SV_ERR_UNSUPPORTED
    assert call(ws=None) == SV_ERR_WORKSPACE
    need = binding.sv_quest_decode_step_workspace_size(8, 32, 4, 100, 16)
    assert call(ws_bytes=need - 1) == SV_ERR_WORKSPACE
    assert call(q=ctypes.c_void_p(0x20002)) == SV_ERR_INVALID_ARG
    assert call(out=ctypes.c_void_p(0x20008)) == SV_ERR_INVALID_ARG
    assert call(ws=ctypes.c_void_p(0x20004)) == SV_ERR_INVALID_ARG


@host_only
def test_select_ex_and_decode_ex_option_checks(lib):
    c = ctypes.byref(_fake_cache())

    def sel(opts, ws_bytes=1 << 30):
        return lib.sv_quest_select_ex(c, FAKE, 32, FAKE, FAKE, 8, 100, 16, ctypes.byref(opts), FAKE, FAKE, None,
                                      FAKE, ws_bytes, None)

    def dec(opts, batch=8, sel=FAKE):
        return lib.sv_sparse_decode_ex(c, FAKE, 32, FAKE, FAKE, batch, 100, sel, FAKE, 16, ctypes.byref(opts),
                                       0.088, FAKE, FAKE, FAKE, 1 << 30, None)
    for bad in (binding.quest_opts(sink_pages=-1), binding.quest_opts(window_pages=-2),
                binding.quest_opts(layer=-1), binding.quest_opts(dense_layers=-1)):
        assert sel(bad) == SV_ERR_INVALID_ARG
        assert dec(bad) == SV_ERR_INVALID_ARG
    two = binding.quest_opts()
    two.per_q_head = 2
    assert sel(two) == SV_ERR_INVALID_ARG
    # A dense layer selects nothing: returns SV_OK before any launch.
    assert sel(binding.quest_opts(layer=1, dense_layers=2)) == SV_OK
    # Per-query-head rows: 2100 requests x 32 query heads exceed the 65535 grid rows.
    assert dec(binding.quest_opts(per_q_head=True), batch=2100) == SV_ERR_UNSUPPORTED
    # per-head scores need Hq rows of workspace
    need = binding.sv_quest_select_ex_workspace_size(8, 32, 4, 100, binding.quest_opts(per_q_head=True))
    assert need == 8 * 32 * 100 * 4
    assert sel(binding.quest_opts(per_q_head=True), ws_bytes=need - 1) == SV_ERR_WORKSPACE
    assert binding.sv_quest_select_ex_workspace_size(8, 32, 4, 100, None) == 8 * 4 * 100 * 4


@host_only
def test_fp8_cache_checks(lib):
    def cache(fmt, ks=0x10000, vs=0x10000):
        c = _fake_cache()
        c.kv_format, c.k_scale, c.v_scale = fmt, ks, vs
        return ctypes.byref(c)

    def sel(c):
        return lib.sv_quest_select(c, FAKE, 32, FAKE, FAKE, 8, 100, 16, FAKE, FAKE, None, FAKE, 1 << 30, None)
    assert sel(cache(binding.SV_KV_FP8_E4M3, ks=0)) == SV_ERR_INVALID_ARG      # scales required
    assert sel(cache(binding.SV_KV_FP8_E4M3, vs=0x10004)) == SV_ERR_INVALID_ARG  # 16-byte aligned
    assert sel(cache(7)) == SV_ERR_UNSUPPORTED
    assert ctypes.sizeof(binding.sv_cache) == 64


def test_binding_rejects_tensors_the_kernels_cannot_take():
    """Argument marshalling: a tensor reaches the C ABI only if it is
    contiguous, of the dtype the kernels read, and in device memory (or, for
    the one-call step's per-step buffers, page-locked host memory)."""
    import pytest
    import torch
    t = torch.zeros(4, 8, dtype=torch.int32)
    assert binding._p(None) is None
    with pytest.raises(ValueError, match="contiguous"):
        binding._p(t.t(), torch.int32, "page_table")
    with pytest.raises(TypeError, match="seq_lens"):
        binding._p(t.long(), torch.int32, "seq_lens")
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding._p(t, torch.int32, "page_table")
    with pytest.raises(ValueError, match="page-locked"):
        binding._p(t, torch.int32, "page_table", host_ok=True)
    pool = torch.zeros(2, 1, 16, 128, dtype=torch.bfloat16)
    meta = torch.zeros(2, 1, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="k_pool"):
        binding.Cache(pool, pool, meta)
