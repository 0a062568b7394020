"""Thin ctypes binding of libsvquest.so (include/svquest.h).

Argument marshalling only: every function takes torch tensors that already
live on the GPU, passes their data pointers, sizes and the current CUDA
stream to the C ABI function of the same name, and raises SvError on a
nonzero status.  There is no CPU fallback: if the library is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB_PATH

_lib = None


class SvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = _load().sv_status_string(status).decode()
        super().__init__(f"{fn} failed: {msg}")
        self.status = status


class sv_quest_opts(ctypes.Structure):
    _fields_ = [("per_q_head", ctypes.c_int32), ("sink_pages", ctypes.c_int32), ("window_pages", ctypes.c_int32),
                ("layer", ctypes.c_int32), ("dense_layers", ctypes.c_int32)]


SV_KV_BF16, SV_KV_FP8_E4M3 = 0, 1


class sv_cache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("meta", ctypes.c_void_p),
                ("num_phys_pages", ctypes.c_int64), ("num_kv_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("kv_format", ctypes.c_int32),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


def library_path() -> str:
    return LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libsvquest.so not built ({LIB_PATH}); run "
                           "`python -m query_aware_sparse_quest_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    cp = ctypes.POINTER(sv_cache)
    op = ctypes.POINTER(sv_quest_opts)
    sig = {
        "sv_quest_update_meta": [cp, vp, vp, vp, i64, vp],
        "sv_quest_score": [cp, vp, i32, vp, vp, i32, i32, vp, vp],
        "sv_quest_topk": [vp, vp, i32, i32, i32, i32, vp, vp, vp],
        "sv_quest_select": [cp, vp, i32, vp, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp],
        "sv_sparse_decode": [cp, vp, i32, vp, vp, i32, i32, vp, vp, i32, f32, vp, vp, vp, sz, vp],
        "sv_sparse_decode_static_scratch": [cp, vp, i32, vp, vp, i32, i32, vp, vp, i32, f32, vp, vp, vp],
        "sv_quest_decode_step": [cp, vp, i32, vp, vp, i32, i32, i32, f32, vp, vp, vp, vp, vp, sz, vp],
        "sv_quest_select_ex": [cp, vp, i32, vp, vp, i32, i32, i32, op, vp, vp, vp, vp, sz, vp],
        "sv_sparse_decode_ex": [cp, vp, i32, vp, vp, i32, i32, vp, vp, i32, op, f32, vp, vp, vp, sz, vp],
        "sv_get_device_error": [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.sv_quest_select_workspace_size.argtypes = [i32, i32, i32]
    lib.sv_quest_select_workspace_size.restype = sz
    lib.sv_sparse_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.sv_sparse_decode_workspace_size.restype = sz
    lib.sv_quest_decode_step_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.sv_quest_decode_step_workspace_size.restype = sz
    lib.sv_quest_select_ex_workspace_size.argtypes = [i32, i32, i32, i32, op]
    lib.sv_quest_select_ex_workspace_size.restype = sz
    lib.sv_status_string.argtypes = [ctypes.c_int]
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.sv_version.argtypes = []
    lib.sv_version.restype = ctypes.c_int
    _lib = lib
    return lib


_BF16, _I32, _F32 = torch.bfloat16, torch.int32, torch.float32


def _p(t: Optional[torch.Tensor], dtype: Optional[torch.dtype] = None, name: str = "tensor",
       host_ok: bool = False):
    """The tensor's address for the C ABI, after checking what the kernels
    assume of it: contiguous, of the given dtype, in device memory (or, where
    host_ok, in page-locked host memory)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or page-locked host memory" if host_ok else ""))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise SvError(fn, status)


class Cache:
    """A paged pool on the device: k/v [pages][Hkv][16][128] (bf16, or uint8 e4m3 codes with fp32 row
    scales k_scale / v_scale [pages][Hkv][16]), meta bf16 [pages][Hkv][2][128]."""

    def __init__(self, k_pool: torch.Tensor, v_pool: torch.Tensor, meta: torch.Tensor,
                 k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None):
        self.k_pool, self.v_pool, self.meta = k_pool, v_pool, meta
        self.k_scale, self.v_scale = k_scale, v_scale
        n, hkv, p, d = k_pool.shape
        fp8 = k_pool.dtype == torch.uint8
        pool_t = torch.uint8 if fp8 else _BF16
        _p(k_pool, pool_t, "k_pool")
        _p(v_pool, pool_t, "v_pool")
        _p(meta, _BF16, "meta")
        if fp8:
            if k_scale is None or v_scale is None:
                raise ValueError("an e4m3 pool needs k_scale and v_scale")
            _p(k_scale, _F32, "k_scale")
            _p(v_scale, _F32, "v_scale")
        self.c = sv_cache(k_pool.data_ptr(), v_pool.data_ptr(), meta.data_ptr(), n, hkv, p, d,
                          SV_KV_FP8_E4M3 if fp8 else SV_KV_BF16,
                          k_scale.data_ptr() if fp8 else None, v_scale.data_ptr() if fp8 else None)

    @classmethod
    def empty(cls, num_phys_pages: int, num_kv_heads: int, device="cuda", page_size: int = 16,
              head_dim: int = 128) -> "Cache":
        shape = (num_phys_pages, num_kv_heads, page_size, head_dim)
        k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        m = torch.zeros((num_phys_pages, num_kv_heads, 2, head_dim), dtype=torch.bfloat16, device=device)
        return cls(k, v, m)

    @property
    def num_kv_heads(self) -> int:
        return int(self.c.num_kv_heads)

    def ref(self):
        return ctypes.byref(self.c)


def sv_quest_update_meta(cache: Cache, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                         stream=None) -> None:
    _check("sv_quest_update_meta", _load().sv_quest_update_meta(
        cache.ref(), _p(k_new, _BF16, "k_new"), _p(v_new, _BF16, "v_new"), _p(slot_mapping, _I32, "slot_mapping"),
        int(slot_mapping.numel()), _stream(stream)))


def sv_quest_score(cache: Cache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                   scores: torch.Tensor, stream=None) -> None:
    B, Hq, _ = q.shape
    _check("sv_quest_score", _load().sv_quest_score(
        cache.ref(), _p(q, _BF16, "q"), Hq, _p(page_table, _I32, "page_table"), _p(seq_lens, _I32, "seq_lens"), B,
        int(page_table.shape[1]), _p(scores, _F32, "scores"), _stream(stream)))


def sv_quest_topk(scores: torch.Tensor, seq_lens: torch.Tensor, budget_pages: int, sel_idx: torch.Tensor,
                  sel_cnt: torch.Tensor, stream=None) -> None:
    B, Hkv, max_pages = scores.shape
    _check("sv_quest_topk", _load().sv_quest_topk(
        _p(scores, _F32, "scores"), _p(seq_lens, _I32, "seq_lens"), B, Hkv, max_pages, int(budget_pages),
        _p(sel_idx, _I32, "sel_idx"), _p(sel_cnt, _I32, "sel_cnt"), _stream(stream)))


def sv_quest_select_workspace_size(batch: int, num_kv_heads: int, max_pages: int) -> int:
    return int(_load().sv_quest_select_workspace_size(batch, num_kv_heads, max_pages))


def sv_quest_select(cache: Cache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                    budget_pages: int, sel_idx: torch.Tensor, sel_cnt: torch.Tensor,
                    scores_out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None) -> None:
    B, Hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("sv_quest_select", _load().sv_quest_select(
        cache.ref(), _p(q, _BF16, "q"), Hq, _p(page_table, _I32, "page_table"), _p(seq_lens, _I32, "seq_lens"), B,
        int(page_table.shape[1]), int(budget_pages),
        _p(sel_idx, _I32, "sel_idx"), _p(sel_cnt, _I32, "sel_cnt"), _p(scores_out, _F32, "scores_out"),
        _p(workspace, None, "workspace"), ws_bytes, _stream(stream)))


def sv_sparse_decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, pages: int) -> int:
    return int(_load().sv_sparse_decode_workspace_size(batch, num_q_heads, num_kv_heads, pages))


def sv_sparse_decode(cache: Cache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                     sel_idx: Optional[torch.Tensor], sel_cnt: Optional[torch.Tensor], out: torch.Tensor,
                     lse: torch.Tensor, workspace: torch.Tensor, softmax_scale: Optional[float] = None,
                     stream=None) -> None:
    B, Hq, D = q.shape
    K = 0 if sel_idx is None else int(sel_idx.shape[2])
    scale = float(D) ** -0.5 if softmax_scale is None else float(softmax_scale)
    _check("sv_sparse_decode", _load().sv_sparse_decode(
        cache.ref(), _p(q, _BF16, "q"), Hq, _p(page_table, _I32, "page_table"), _p(seq_lens, _I32, "seq_lens"), B,
        int(page_table.shape[1]), _p(sel_idx, _I32, "sel_idx"),
        _p(sel_cnt, _I32, "sel_cnt"), K, scale, _p(out, _BF16, "out"), _p(lse, _F32, "lse"),
        _p(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def sv_sparse_decode_static_scratch(cache: Cache, q: torch.Tensor, page_table: torch.Tensor,
                                    seq_lens: torch.Tensor, sel_idx: Optional[torch.Tensor],
                                    sel_cnt: Optional[torch.Tensor], out: torch.Tensor, lse: torch.Tensor,
                                    softmax_scale: Optional[float] = None, stream=None) -> None:
    """sv_sparse_decode with the library's fixed scratch array instead of a workspace."""
    B, Hq, D = q.shape
    K = 0 if sel_idx is None else int(sel_idx.shape[2])
    scale = float(D) ** -0.5 if softmax_scale is None else float(softmax_scale)
    _check("sv_sparse_decode_static_scratch", _load().sv_sparse_decode_static_scratch(
        cache.ref(), _p(q, _BF16, "q"), Hq, _p(page_table, _I32, "page_table"), _p(seq_lens, _I32, "seq_lens"), B,
        int(page_table.shape[1]), _p(sel_idx, _I32, "sel_idx"),
        _p(sel_cnt, _I32, "sel_cnt"), K, scale, _p(out, _BF16, "out"), _p(lse, _F32, "lse"), _stream(stream)))


def sv_quest_decode_step_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, max_pages: int,
                                        budget_pages: int) -> int:
    return int(_load().sv_quest_decode_step_workspace_size(batch, num_q_heads, num_kv_heads, max_pages,
                                                           budget_pages))


def _step(name: str, cache: Cache, q, page_table, seq_lens, budget_pages, sel_idx, sel_cnt, out, lse, workspace,
          softmax_scale, stream) -> None:
    B, Hq, D = q.shape
    scale = float(D) ** -0.5 if softmax_scale is None else float(softmax_scale)
    _check(name, getattr(_load(), name)(
        cache.ref(), _p(q, _BF16, "q", True), Hq, _p(page_table, _I32, "page_table", True),
        _p(seq_lens, _I32, "seq_lens", True), B, int(page_table.shape[1]), int(budget_pages), scale,
        _p(sel_idx, _I32, "sel_idx"), _p(sel_cnt, _I32, "sel_cnt"), _p(out, _BF16, "out", True),
        _p(lse, _F32, "lse", True), _p(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def sv_quest_decode_step(cache: Cache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                         budget_pages: int, sel_idx: torch.Tensor, sel_cnt: torch.Tensor, out: torch.Tensor,
                         lse: torch.Tensor, workspace: torch.Tensor, softmax_scale: Optional[float] = None,
                         stream=None) -> None:
    _step("sv_quest_decode_step", cache, q, page_table, seq_lens, budget_pages, sel_idx, sel_cnt, out, lse,
          workspace, softmax_scale, stream)


def quest_opts(per_q_head: bool = False, sink_pages: int = 0, window_pages: int = 0, layer: int = 0,
               dense_layers: int = 0) -> sv_quest_opts:
    return sv_quest_opts(int(bool(per_q_head)), int(sink_pages), int(window_pages), int(layer), int(dense_layers))


def sv_quest_select_ex_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, max_pages: int,
                                      opts: Optional[sv_quest_opts] = None) -> int:
    return int(_load().sv_quest_select_ex_workspace_size(batch, num_q_heads, num_kv_heads, max_pages,
                                                         None if opts is None else ctypes.byref(opts)))


def sv_quest_select_ex(cache: Cache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                       budget_pages: int, opts: Optional[sv_quest_opts], sel_idx: torch.Tensor,
                       sel_cnt: torch.Tensor, scores_out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    B, Hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("sv_quest_select_ex", _load().sv_quest_select_ex(
        cache.ref(), _p(q, _BF16, "q"), Hq, _p(page_table, _I32, "page_table"), _p(seq_lens, _I32, "seq_lens"), B,
        int(page_table.shape[1]), int(budget_pages),
        None if opts is None else ctypes.byref(opts), _p(sel_idx, _I32, "sel_idx"), _p(sel_cnt, _I32, "sel_cnt"), _p(scores_out, _F32, "scores_out"),
        _p(workspace, None, "workspace"),
        ws_bytes, _stream(stream)))


def sv_sparse_decode_ex(cache: Cache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                        sel_idx: Optional[torch.Tensor], sel_cnt: Optional[torch.Tensor],
                        opts: Optional[sv_quest_opts], out: torch.Tensor, lse: torch.Tensor,
                        workspace: torch.Tensor, softmax_scale: Optional[float] = None, stream=None) -> None:
    B, Hq, D = q.shape
    K = 0 if sel_idx is None else int(sel_idx.shape[2])
    scale = float(D) ** -0.5 if softmax_scale is None else float(softmax_scale)
    _check("sv_sparse_decode_ex", _load().sv_sparse_decode_ex(
        cache.ref(), _p(q, _BF16, "q"), Hq, _p(page_table, _I32, "page_table"), _p(seq_lens, _I32, "seq_lens"), B,
        int(page_table.shape[1]), _p(sel_idx, _I32, "sel_idx"),
        _p(sel_cnt, _I32, "sel_cnt"), K, None if opts is None else ctypes.byref(opts), scale,
        _p(out, _BF16, "out"), _p(lse, _F32, "lse"), _p(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def sv_get_device_error(reset: bool = True) -> int:
    flags = ctypes.c_uint32(0)
    _check("sv_get_device_error", _load().sv_get_device_error(ctypes.byref(flags), int(reset)))
    return int(flags.value)


def sv_status_string(status: int) -> str:
    return _load().sv_status_string(status).decode()


def sv_version() -> int:
    return int(_load().sv_version())


def raw_library():
    """The loaded ctypes library, for calls made with raw pointers."""
    return _load()
