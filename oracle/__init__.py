"""CPU oracle for query-aware sparse decode: ctypes wrapper over quest_oracle.c.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers; the product path (the CUDA library and
its Python binding) never imports this package.

Functions take numpy arrays (bf16 data as uint16 bit patterns) and return
numpy arrays.  See quest_oracle.c for what each one computes and which
passage it follows.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "quest_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libquest_oracle.so")
_OMP_LIB_PATH = os.path.join(_HERE, "_build", "libquest_oracle_omp.so")
_libs = {}
_openmp = False


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction).  With
    openmp, a second library of the same source whose row loops run on the
    host's threads (-fopenmp); the arithmetic of each row is unchanged."""
    path = _OMP_LIB_PATH if openmp else _LIB_PATH
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    os.makedirs(os.path.dirname(path), exist_ok=True)
    tmp = path + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                    *(["-fopenmp"] if openmp else []), "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, path)
    return path


@contextlib.contextmanager
def parallel():
    """Inside the block, select and decode run on the OpenMP build: their
    independent rows (request, head) are spread over the host's threads."""
    global _openmp
    prev, _openmp = _openmp, True
    try:
        yield num_threads()
    finally:
        _openmp = prev


def num_threads() -> int:
    """Threads the current build's row loops use (1 for the plain build)."""
    return int(_load().oracle_num_threads())


def _load():
    variant = _openmp
    lib = _libs.get(variant)
    if lib is None:
        lib = ctypes.CDLL(build(openmp=variant))
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.oracle_update_meta.argtypes = [P, P, P, i64, i32, i32, i32, P, P, P, i64]
        lib.oracle_select.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i64, P, P, P]
        lib.oracle_decode.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, P, P, i32, f32, P, P]
        lib.oracle_select_ex.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i64, i32, i32, i32,
                                         P, P, P]
        lib.oracle_decode_ex.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, P, P, i32, i32, f32,
                                         P, P]
        lib.oracle_quantize_rows.argtypes = [P, P, P, P, i64, i32, i32, i32, P, P, P, i64]
        lib.oracle_decode_fp8.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, P, P, i32, i32,
                                          f32, P, P]
        lib.oracle_topk.argtypes = [P, P, i32, i32, i32, P, P]
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = f32
        lib.oracle_e4m3_encode.argtypes = [f32]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_num_threads.argtypes = []
        for f in (lib.oracle_update_meta, lib.oracle_select, lib.oracle_decode, lib.oracle_select_ex,
                  lib.oracle_decode_ex, lib.oracle_quantize_rows, lib.oracle_decode_fp8, lib.oracle_topk,
                  lib.oracle_num_threads):
            f.restype = ctypes.c_int
        _libs[variant] = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


class Cache:
    """Host copy of a paged pool: k/v [n_phys][Hkv][P][D] and meta [n_phys][Hkv][2][D].

    With fp8, the pool also holds e4m3 codes k8/v8 [n_phys][Hkv][P][D] and fp32
    row scales ks/vs [n_phys][Hkv][P] (k/v then keep the appended bf16 rows,
    from which the metadata is computed)."""

    def __init__(self, n_phys: int, num_kv_heads: int, page_size: int = 16, head_dim: int = 128,
                 fill_bits: int = 0, fp8: bool = False, fill_code: int = 0, fill_scale: float = 0.0):
        shape = (n_phys, num_kv_heads, page_size, head_dim)
        self.k = np.full(shape, fill_bits, dtype=np.uint16)
        self.v = np.full(shape, fill_bits, dtype=np.uint16)
        self.meta = np.zeros((n_phys, num_kv_heads, 2, head_dim), dtype=np.uint16)
        self.n_phys, self.Hkv, self.P, self.D = n_phys, num_kv_heads, page_size, head_dim
        self.fp8 = fp8
        if fp8:
            self.k8 = np.full(shape, fill_code, dtype=np.uint8)
            self.v8 = np.full(shape, fill_code, dtype=np.uint8)
            self.ks = np.full(shape[:3], fill_scale, dtype=np.float32)
            self.vs = np.full(shape[:3], fill_scale, dtype=np.float32)


def update_meta(cache: Cache, k_new: np.ndarray, v_new: np.ndarray, slot_mapping: np.ndarray) -> None:
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    slot_mapping = _c(slot_mapping, np.int32)
    T = slot_mapping.shape[0]
    assert k_new.shape == (T, cache.Hkv, cache.D) and v_new.shape == k_new.shape
    rc = _load().oracle_update_meta(_ptr(cache.k), _ptr(cache.v), _ptr(cache.meta), cache.n_phys,
                                    cache.Hkv, cache.P, cache.D, _ptr(k_new), _ptr(v_new),
                                    _ptr(slot_mapping), T)
    if rc != 0:
        raise ValueError(f"oracle_update_meta failed ({rc})")
    if cache.fp8:
        rc = _load().oracle_quantize_rows(_ptr(cache.k8), _ptr(cache.v8), _ptr(cache.ks), _ptr(cache.vs),
                                          cache.n_phys, cache.Hkv, cache.P, cache.D, _ptr(k_new), _ptr(v_new),
                                          _ptr(slot_mapping), T)
        if rc != 0:
            raise ValueError(f"oracle_quantize_rows failed ({rc})")


def e4m3_value(code: int) -> float:
    return float(_load().oracle_e4m3_value(int(code)))


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def select(cache: Cache, q: np.ndarray, page_table: np.ndarray, seq_lens: np.ndarray,
           budget_pages: int, per_q_head: bool = False, sink_pages: int = 0,
           window_pages: int = 0) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Returns (sel_idx [B][R][K] int32, sel_cnt [B][R] int32, scores [B][R][max_pages] fp32),
    R = num_q_heads when per_q_head, else num_kv_heads.

    Score entries past a request's last page are NaN; forced (sink / window)
    pages keep their bound as the score."""
    q = _c(q, np.uint16)
    page_table = _c(page_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    R = Hq if per_q_head else cache.Hkv
    max_pages = page_table.shape[1]
    K = int(budget_pages)
    sel_idx = np.empty((B, R, K), dtype=np.int32)
    sel_cnt = np.empty((B, R), dtype=np.int32)
    scores = np.full((B, R, max_pages), np.nan, dtype=np.float32)
    rc = _load().oracle_select_ex(_ptr(q), _ptr(cache.meta), _ptr(page_table), _ptr(seq_lens), B, Hq,
                                  cache.Hkv, D, cache.P, max_pages, K, cache.n_phys, int(bool(per_q_head)),
                                  int(sink_pages), int(window_pages), _ptr(sel_idx), _ptr(sel_cnt), _ptr(scores))
    if rc != 0:
        raise ValueError(f"oracle_select failed ({rc})")
    return sel_idx, sel_cnt, scores


def topk(scores: np.ndarray, n_pages: np.ndarray, budget_pages: int) -> Tuple[np.ndarray, np.ndarray]:
    """The selection step on given scores [rows][max_pages] with n_pages[row] valid entries:
    returns (sel_idx [rows][K] ascending, -1 padded; sel_cnt [rows] = min(K, n))."""
    scores = _c(scores, np.float32)
    n_pages = _c(n_pages, np.int32)
    rows, max_pages = scores.shape
    K = int(budget_pages)
    sel_idx = np.empty((rows, K), dtype=np.int32)
    sel_cnt = np.empty((rows,), dtype=np.int32)
    rc = _load().oracle_topk(_ptr(scores), _ptr(n_pages), rows, max_pages, K, _ptr(sel_idx), _ptr(sel_cnt))
    if rc != 0:
        raise ValueError(f"oracle_topk failed ({rc})")
    return sel_idx, sel_cnt


def decode(cache: Cache, q: np.ndarray, page_table: np.ndarray, seq_lens: np.ndarray,
           sel_idx: Optional[np.ndarray] = None, sel_cnt: Optional[np.ndarray] = None,
           scale: Optional[float] = None, per_q_head: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Returns (out fp32 [B][Hq][D], lse fp32 [B][Hq]); dense when sel_idx is None.
    With per_q_head, sel_idx has one row per query head.  An fp8 cache attends
    over its decoded e4m3 rows."""
    q = _c(q, np.uint16)
    page_table = _c(page_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    max_pages = page_table.shape[1]
    if scale is None:
        scale = 1.0 / float(np.sqrt(D))
    K = 0
    if sel_idx is not None:
        sel_idx = _c(sel_idx, np.int32)
        sel_cnt = _c(sel_cnt, np.int32)
        K = sel_idx.shape[2]
    out = np.empty((B, Hq, D), dtype=np.float32)
    lse = np.empty((B, Hq), dtype=np.float32)
    if cache.fp8:
        rc = _load().oracle_decode_fp8(_ptr(q), _ptr(cache.k8), _ptr(cache.v8), _ptr(cache.ks), _ptr(cache.vs),
                                       _ptr(page_table), _ptr(seq_lens), B, Hq, cache.Hkv, D, cache.P, max_pages,
                                       cache.n_phys, _ptr(sel_idx), _ptr(sel_cnt), K, int(bool(per_q_head)),
                                       float(scale), _ptr(out), _ptr(lse))
        if rc != 0:
            raise ValueError(f"oracle_decode_fp8 failed ({rc})")
        return out, lse
    rc = _load().oracle_decode_ex(_ptr(q), _ptr(cache.k), _ptr(cache.v), _ptr(page_table), _ptr(seq_lens),
                                  B, Hq, cache.Hkv, D, cache.P, max_pages, cache.n_phys, _ptr(sel_idx),
                                  _ptr(sel_cnt), K, int(bool(per_q_head)), float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode failed ({rc})")
    return out, lse


def build_cache(wl, fill_bits: int, fp8: bool = False, fill_code: int = 0, fill_scale: float = 0.0) -> Cache:
    """Pool + metadata after a workload's whole prefill, appended in 4096-token chunks.

    `wl` is a synthetic workload (token stream, slot mapping, pool size);
    `fill_bits` is the bf16 pattern of pool slots that never receive a token
    (`fill_code` / `fill_scale` for the e4m3 codes and scales of an fp8 pool)."""
    s = wl.spec
    cache = Cache(wl.num_phys_pages, s.num_kv_heads, s.page_size, s.head_dim, fill_bits, fp8, fill_code, fill_scale)
    for a, b in wl.prefill_chunks():
        update_meta(cache, wl.k_tok[a:b], wl.v_tok[a:b], wl.slot_mapping[a:b])
    return cache
