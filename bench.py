"""Benchmark: Quest sparse decode steps/s and achieved HBM bandwidth on one GB300.

Workload: Qwen3-30B-A3B attention geometry (32 query / 4 kv heads, head_dim
128), batch 8, 128000-token contexts in pages of 16 tokens (8000 pages per
request), budget 4096 tokens (256 pages), 64 planted needle pages per request,
physical pages shuffled over one pool; bf16 K/V/q, seeded synthetic data.

A step is one attention layer's decode for the whole batch: page scoring,
top-K selection and split-K attention over the selected pages, through the
public one-call step sv_quest_decode_step (four kernels: scores, top-K, split
decode, log-sum-exp combine, chained by programmatic dependent launch),
captured once as a CUDA graph and replayed.  Inputs are resident in HBM.  The
K timed steps run back to back, one replay per step, between one pair of CUDA
events on the launching stream; L2 is not flushed between them because each
step reads 198.6 MB, more than L2 holds (per_step_ms gives the same step timed
alone with and without a flush).  Per-kernel durations come from a second
pass that times the separate calls (sv_quest_score, sv_quest_topk,
sv_sparse_decode) alone after an L2 flush.  The end-to-end figure runs the
same call with q, page table and lengths in page-locked host memory and
out / lse written into page-locked host memory by the kernels.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas; weak scaling, no collective on the data path); rank 0 prints one
JSON line with the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from query_aware_sparse_quest_gb300 import binding, build, resident, synth  # noqa: E402

METRIC = "sparse-decode steps/s and achieved HBM GB/s vs ~8 TB/s at 128k ctx, batch 8"
UNIT = "steps/s"
BENCH_CONFIG = 2
PROFILE_SUMMARIES = {"score_pages_kernel": "profiles/score_pages_qwen3_b8_ctx128000.txt",
                     "flash_decode_split_kernel": "profiles/flash_decode_qwen3_b8_ctx128000.txt"}
KERNEL_SOURCES = {"score_pages_kernel": "query_aware_sparse_quest_gb300/csrc/svq_select.cu",
                  "flash_decode_split_kernel": "query_aware_sparse_quest_gb300/csrc/svq_decode.cu"}


# ---------------------------------------------------------------- helpers

def dist_info():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, device=None) -> float:
    """The largest of every rank's x (all-reduce MAX); x itself on one rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world: int, ms_per_step: float) -> float:
    """Steps/s of the whole job: every rank runs one full-batch step per step,
    and the job's step time is the slowest rank's."""
    return world * 1e3 / ms_per_step


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(device_index), "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


class Sections:
    """NVTX ranges around the benchmark's sections (host-side markers, so that
    an ncu capture can be limited to one with --nvtx --nvtx-include <name>/);
    a no-op where NVTX is unavailable."""

    def __init__(self):
        self.open = False
        try:
            self.nvtx = torch.cuda.nvtx
            self.nvtx.range_push("probe")
            self.nvtx.range_pop()
        except Exception:
            self.nvtx = None

    def __call__(self, name: str):
        self.close()
        if self.nvtx is not None:
            self.nvtx.range_push(name)
            self.open = True

    def close(self):
        if self.open:
            self.nvtx.range_pop()
            self.open = False


def kernel_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, PROFILE_SUMMARIES[kernel])
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    src = os.path.join(ROOT, KERNEL_SOURCES[kernel])
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if vals.get(f"{kernel}.source_sha256_16") != digest:
        return None
    try:
        return float(vals[f"{kernel}.dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


def algorithmic_bytes(wl):
    """Per-step bytes the method must move (metadata + selected K/V + page tables + q/out),
    and per-kernel figures for the roofline."""
    s = wl.spec
    P, Hkv, Hq, D = s.page_size, s.num_kv_heads, s.num_q_heads, s.head_dim
    n = (wl.seq_lens.astype(np.int64) + P - 1) // P
    sel = np.minimum(n, s.budget_pages)
    meta = int(n.sum()) * Hkv * 2 * D * 2
    pt = int(n.sum()) * 4
    q = s.batch * Hq * D * 2
    scores_w = int(n.sum()) * Hkv * 4
    kv = int(sel.sum()) * Hkv * P * D * 2 * 2
    sel_rd = int(sel.sum()) * Hkv * 4 * 2          # sel_idx + page-table entry per selected page
    out = s.batch * Hq * D * 2 + s.batch * Hq * 4
    dense_kv = int(n.sum()) * Hkv * P * D * 2 * 2
    kv8 = int(sel.sum()) * Hkv * P * (D + 4) * 2      # e4m3 rows + fp32 row scales, K and V
    return {
        "fp8_step": meta + kv8 + pt + q + out,
        "fp8_decode": kv8 + sel_rd + q,
        "step": meta + kv + pt + q + out,
        "score_pages_kernel": meta + pt + q + scores_w,
        "flash_decode_split_kernel": kv + sel_rd + q,
        "dense_step": dense_kv + pt + q + out,
    }


# Kernels each public call launches (include/svquest.h): sv_quest_score and
# sv_quest_topk one each, sv_sparse_decode two (split-K flash decode, then the
# log-sum-exp combine), sv_quest_decode_step four (scores, top-K, split-K
# decode, combine), sv_quest_update_meta one.
KERNELS_PER_CALL = {"sv_quest_score": 1, "sv_quest_topk": 1, "sv_sparse_decode": 2, "sv_quest_decode_step": 4,
                    "sv_quest_update_meta": 1}
STEP_CALLS = ("sv_quest_decode_step",)


# ---------------------------------------------------------------- GPU arm

def run_gpu(args):
    rank, world, local_rank = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    build.build()

    spec = synth.SPECS[BENCH_CONFIG]
    wl = synth.make_workload(spec)
    dw = resident.upload(wl, device=dev)
    B, Hq, D = dw.q.shape
    Hkv = spec.num_kv_heads
    K = spec.budget_pages
    max_pages = wl.max_pages
    stream = torch.cuda.current_stream(dev)

    scores = torch.empty((B, Hkv, max_pages), dtype=torch.float32, device=dev)
    sel_idx, sel_cnt = resident.select_buffers(B, Hkv, K, dev)
    ws = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, Hkv, K), dev)
    ws_dense = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, Hkv, max_pages), dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    class _Flush:
        """Evicts L2 before a timed step: writes a buffer of twice the L2 size,
        then reads another one of that size, so that the step starts on a cold
        L2 holding no dirty lines of ours (their write-back is not charged to
        the step)."""

        @staticmethod
        def zero_():
            flush_w.zero_()
            flush_r.sum()

    flush = _Flush()

    def score(q=None, pt=None, sl=None):
        binding.sv_quest_score(dw.cache, dw.q if q is None else q, dw.page_table if pt is None else pt,
                               dw.seq_lens if sl is None else sl, scores)

    def topk(sl=None):
        binding.sv_quest_topk(scores, dw.seq_lens if sl is None else sl, K, sel_idx, sel_cnt)

    def decode(q=None, pt=None, sl=None):
        binding.sv_sparse_decode(dw.cache, dw.q if q is None else q, dw.page_table if pt is None else pt,
                                 dw.seq_lens if sl is None else sl, sel_idx, sel_cnt, out, lse, ws)

    ws_step = resident.workspace(binding.sv_quest_decode_step_workspace_size(B, Hq, Hkv, max_pages, K), dev)

    def step():
        binding.sv_quest_decode_step(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, sel_idx, sel_cnt, out, lse,
                                     ws_step)

    def dense():
        binding.sv_sparse_decode(dw.cache, dw.q, dw.page_table, dw.seq_lens, None, None, out, lse, ws_dense)

    def capture(fn):
        """One step as a CUDA graph: the kernels run back to back (programmatic
        dependent launch between them) and the host stays ahead of the GPU."""
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(2):
                fn()
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        torch.cuda.synchronize(dev)
        return graph

    def timed(run, n, warm=3, flush_l2=True):
        """n runs, each after an L2 flush (unless flush_l2 is False),
        bracketed by events on this stream; everything is enqueued before the
        single synchronisation."""
        for _ in range(warm):
            if flush_l2:
                flush.zero_()
            run()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize(dev)
        for e0, e1 in evs:
            if flush_l2:
                flush.zero_()
            e0.record(stream)
            run()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    def back_to_back(run, n, warm=3):
        """n runs back to back between one pair of events on this stream (no
        L2 flush); milliseconds per run."""
        for _ in range(warm):
            run()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n):
            run()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    launches_per_step = sum(KERNELS_PER_CALL[c] for c in STEP_CALLS)
    g_step = capture(step)
    g_dense = capture(dense)
    # Clock sampling starts before the warm-up, so that the timed steps
    # follow busy GPU work directly (no idle gap in which clocks could drop).
    sampler = ClockSampler(local_rank)
    time.sleep(0.25)
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()

    # ---- timed region: K steps back to back (one graph replay per step)
    # between one pair of events.  L2 is not flushed between steps: each
    # step reads 198.6 MB of metadata and K/V, more than the 126 MB L2, so
    # none of it survives to the next step (the per-step times below, taken
    # with and without a flush, differ only by the small structures the
    # kernels reuse: page table, scores, selection lists).
    mark = Sections()
    mark("headline_steps")
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(args.steps):
        g_step.replay()
    e_end.record(stream)
    mark.close()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(float(e_start.elapsed_time(e_end)), dev)
    ms_per_step = total_ms / args.steps
    # The same step timed alone: events around each replay, L2 flushed
    # before each one (so every step also pays its own launch and events).
    mark("step_alone")
    flushed_ms = float(np.mean(timed(g_step.replay, max(3, min(args.steps, 200)))))
    noflush_ms = float(np.mean(timed(g_step.replay, max(3, min(args.steps, 200)), flush_l2=False)))
    # Ten steps captured in one graph, as an engine that captures a whole
    # forward pass would run them: each step's scoring kernel then also
    # follows the previous step's combine by programmatic dependent launch.
    def ten_steps():
        for _ in range(10):
            step()

    g_ten = capture(ten_steps)
    chained_ms = back_to_back(g_ten.replay, max(3, min(args.steps, 200) // 10)) / 10
    del g_ten

    # ---- per-kernel durations (each call timed alone, same flush discipline)
    mark("per_kernel")
    n_k = max(3, min(args.steps, 200))
    t_score = float(np.mean(timed(score, n_k)))
    # The scoring kernel's average launch duration: launches back to back
    # between one pair of events (each reads 131 MB of metadata, more than L2
    # holds, so none of it carries over), without the per-call event floor.
    g_score = capture(score)
    t_score_b2b = back_to_back(g_score.replay, n_k)
    del g_score
    t_topk = float(np.mean(timed(topk, n_k)))
    t_dec = float(np.mean(timed(decode, n_k)))

    # ---- dense (all pages) comparator
    mark("dense")
    dense_ms = float(np.mean(timed(g_dense.replay, max(3, min(args.steps, 50)))))

    step()   # the step again (the dense comparator overwrote out / lse)
    torch.cuda.synchronize(dev)

    # ---- bulk prefill append: one 4096-token chunk through sv_quest_update_meta
    mark("prefill_append")
    # (request 0's first 4096 tokens rewritten into their own slots: same pool)
    T = min(4096, int(wl.seq_lens[0]))
    k_new = resident.bf16_tensor(wl.k_tok[:T], dev)
    v_new = resident.bf16_tensor(wl.v_tok[:T], dev)
    slots = torch.from_numpy(wl.slot_mapping[:T]).to(dev)

    def append():
        binding.sv_quest_update_meta(dw.cache, k_new, v_new, slots)

    append_ms = float(np.mean(timed(append, max(3, min(args.steps, 200)))))

    # A whole chunked prefill: request 0's tokens appended 4096 at a time (the
    # pages' chunk_prefill_size), all chunks captured as one graph, so that
    # back-to-back appends are timed as a prefill issues them.
    L0 = int(wl.seq_lens[0])
    k_all = resident.bf16_tensor(wl.k_tok[:L0], dev)
    v_all = resident.bf16_tensor(wl.v_tok[:L0], dev)
    slots_all = torch.from_numpy(wl.slot_mapping[:L0]).to(dev)
    chunks = [(c0, min(L0, c0 + 4096)) for c0 in range(0, L0, 4096)]

    def prefill():
        for c0, c1 in chunks:
            binding.sv_quest_update_meta(dw.cache, k_all[c0:c1], v_all[c0:c1], slots_all[c0:c1])

    prefill()
    g_prefill = capture(prefill)
    prefill_ms = float(np.mean(timed(g_prefill.replay, max(3, min(args.steps // 10, 20)))))
    del k_all, v_all, slots_all, g_prefill

    # ---- the same step over an fp8 (e4m3) pool of the same tokens
    mark("fp8_step")
    dw8 = resident.upload(wl, device=dev, fp8=True)
    sel8, cnt8 = resident.select_buffers(B, Hkv, K, dev)
    out8, lse8 = torch.empty_like(out), torch.empty_like(lse)

    def step8():
        binding.sv_quest_decode_step(dw8.cache, dw8.q, dw8.page_table, dw8.seq_lens, K, sel8, cnt8, out8, lse8,
                                     ws_step)

    for _ in range(3):
        step8()
    g_step8 = capture(step8)
    fp8_ms = back_to_back(g_step8.replay, max(3, min(args.steps, 200)))
    fp8_dec_ms = float(np.mean(timed(
        lambda: binding.sv_sparse_decode(dw8.cache, dw8.q, dw8.page_table, dw8.seq_lens, sel8, cnt8, out8, lse8, ws),
        max(3, min(args.steps, 200)))))
    fp8_same_sel = bool(torch.equal(cnt8, sel_cnt))
    del dw8, g_step8

    mark("quest_variants")
    # ---- the selection options on the same workload: sv_quest_select_ex +
    # sv_sparse_decode_ex as one CUDA graph, timed back to back like the
    # headline.  Forced pages (the first page and the last four, counted in the
    # budget) and one page set per query head (each of the 32 query heads reads
    # its own 256 pages of its kv head).
    n_pages = (wl.seq_lens.astype(np.int64) + spec.page_size - 1) // spec.page_size
    variants = {"note": "select_ex + decode_ex as one graph, back to back; bytes = metadata + the K/V of every "
                        "selection row + page table + q / out / lse"}
    for vname, vopts, rows in (("sink1_window4", binding.quest_opts(sink_pages=1, window_pages=4), Hkv),
                               ("per_q_head", binding.quest_opts(per_q_head=True), Hq)):
        sv, cv = resident.select_buffers(B, rows, K, dev)
        wsv = resident.workspace(binding.sv_quest_select_ex_workspace_size(B, Hq, Hkv, max_pages, vopts), dev)

        def var_step(vopts=vopts, sv=sv, cv=cv, wsv=wsv):
            binding.sv_quest_select_ex(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, vopts, sv, cv, workspace=wsv)
            binding.sv_sparse_decode_ex(dw.cache, dw.q, dw.page_table, dw.seq_lens, sv, cv, vopts, out, lse, ws)

        for _ in range(3):
            var_step()
        gv = capture(var_step)
        tv = back_to_back(gv.replay, max(3, min(args.steps, 200)))
        vbytes = (int(n_pages.sum()) * Hkv * 2 * D * 2                                 # metadata
                  + int(np.minimum(n_pages, K).sum()) * rows * spec.page_size * D * 2 * 2   # K/V per row
                  + int(n_pages.sum()) * 4 + B * Hq * (D * 2 + D * 2 + 4))           # page table, q, out, lse
        variants[vname] = {"ms_per_step": round(tv, 5), "steps_per_s": round(1e3 / tv, 2), "bytes": vbytes,
                           "gbs": round(vbytes / (tv * 1e-3) / 1e9, 1), "selection_rows_per_request": rows}
        del gv, sv, cv, wsv
    torch.cuda.synchronize(dev)

    mark("kv_heavy_budget512")
    # ---- where selected K/V bytes dominate: 16 requests of 65536 tokens at a
    # 512-page budget, the step over a bf16 and over an fp8 pool (each a CUDA
    # graph, timed back to back), and each sparse decode alone (L2 flushed).
    spec512 = synth.SPECS[4].scaled(budget_pages=512)
    wl512 = synth.make_workload(spec512)
    kv_heavy = {"workload": f"b{spec512.batch}_ctx{spec512.ctx}_budget{512 * spec512.page_size}"}
    ab512 = algorithmic_bytes(wl512)
    for fp8 in (False, True):
        d5 = resident.upload(wl512, device=dev, fp8=fp8)
        B5, Hq5, _ = d5.q.shape
        Hkv5, K5, mp5 = spec512.num_kv_heads, 512, wl512.max_pages
        s5, c5 = resident.select_buffers(B5, Hkv5, K5, dev)
        o5 = torch.empty((B5, Hq5, D), dtype=torch.bfloat16, device=dev)
        l5 = torch.empty((B5, Hq5), dtype=torch.float32, device=dev)
        w5 = resident.workspace(binding.sv_quest_decode_step_workspace_size(B5, Hq5, Hkv5, mp5, K5), dev)
        wd5 = resident.workspace(binding.sv_sparse_decode_workspace_size(B5, Hq5, Hkv5, K5), dev)

        def step5():
            binding.sv_quest_decode_step(d5.cache, d5.q, d5.page_table, d5.seq_lens, K5, s5, c5, o5, l5, w5)

        def dec5():
            binding.sv_sparse_decode(d5.cache, d5.q, d5.page_table, d5.seq_lens, s5, c5, o5, l5, wd5)

        for _ in range(3):
            step5()
        g5 = capture(step5)
        t5 = back_to_back(g5.replay, max(3, min(args.steps, 200)))
        td5 = float(np.mean(timed(dec5, max(3, min(args.steps, 200)))))
        # The sparse decode alone as graph replays back to back: each call
        # reads 139 MB (fp8) or 269 MB (bf16) of selected K/V through
        # evict-first copies, more than L2 holds, so nothing carries over.
        gd5 = capture(dec5)
        tdb5 = back_to_back(gd5.replay, max(3, min(args.steps, 200)))
        b_step = ab512["fp8_step" if fp8 else "step"]
        b_dec = ab512["fp8_decode" if fp8 else "flash_decode_split_kernel"]
        kv_heavy["fp8" if fp8 else "bf16"] = {
            "ms_per_step": round(t5, 5), "bytes": b_step, "gbs": round(b_step / (t5 * 1e-3) / 1e9, 1),
            "sparse_decode_ms": round(td5, 5), "decode_bytes": b_dec,
            "decode_gbs": round(b_dec / (td5 * 1e-3) / 1e9, 1),
            "sparse_decode_back_to_back_ms": round(tdb5, 5),
            "decode_back_to_back_gbs": round(b_dec / (tdb5 * 1e-3) / 1e9, 1)}
        del d5, g5, gd5, w5, wd5
        torch.cuda.synchronize(dev)
    kv_heavy["fp8_vs_bf16_step_time"] = round(kv_heavy["fp8"]["ms_per_step"] / kv_heavy["bf16"]["ms_per_step"], 4)
    def append_bytes_of(T):
        return (2 * T * Hkv * D * 2                      # k_new, v_new read
                + 2 * T * Hkv * D * 2                    # pool rows written
                + T * 4                                  # slot mapping
                + -(-T // spec.page_size) * Hkv * 2 * D * 2)   # metadata written

    append_bytes = append_bytes_of(T)
    prefill_bytes = sum(append_bytes_of(c1 - c0) for c0, c1 in chunks)

    mark("e2e")
    # ---- end to end through the public API: pinned host inputs in, results out
    # (a) The step's inputs (q, page table, lengths) and results (out, lse)
    # live in page-locked host memory and are passed to sv_quest_decode_step
    # as they are: its kernels read the inputs and write the results across
    # the host link, so every step moves them host->device and device->host.
    q_h, pt_h, sl_h = (t.cpu().pin_memory() for t in (dw.q, dw.page_table, dw.seq_lens))
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    def e2e_step():
        binding.sv_quest_decode_step(dw.cache, q_h, pt_h, sl_h, K, sel_idx, sel_cnt, out_h, lse_h, ws_step)

    # (b) The same with copy-engine transfers: inputs in one pinned host block
    # copied to one device block, results in one device block copied back.
    def packed(parts, device, pin):
        offs, total = [], 0
        for t in parts:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(total, dtype=torch.uint8, device=device)
        if pin:
            buf = buf.pin_memory()
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, parts)]
        return buf, views

    in_h, (q_hv, pt_hv, sl_hv) = packed([dw.q, dw.page_table, dw.seq_lens], "cpu", True)
    q_hv.copy_(dw.q.cpu())
    pt_hv.copy_(dw.page_table.cpu())
    sl_hv.copy_(dw.seq_lens.cpu())
    in_d, (q_d, pt_d, sl_d) = packed([dw.q, dw.page_table, dw.seq_lens], dev, False)
    res_d, (out_e, lse_e) = packed([out, lse], dev, False)
    res_h = torch.empty(res_d.numel(), dtype=torch.uint8).pin_memory()

    def e2e_copy_step():
        in_d.copy_(in_h, non_blocking=True)
        binding.sv_quest_decode_step(dw.cache, q_d, pt_d, sl_d, K, sel_idx, sel_cnt, out_e, lse_e, ws_step)
        res_h.copy_(res_d, non_blocking=True)

    # Each end-to-end step is captured once as a CUDA graph, as a serving loop
    # would, and replayed; the transfers run inside every replay.
    e2e_step()
    e2e_copy_step()
    torch.cuda.synchronize(dev)
    e2e_how = ("CUDA graph of sv_quest_decode_step with q / page table / lengths in page-locked host memory "
               "(q staged into the workspace by one copy kernel) and out / lse written into page-locked host "
               "memory by its kernels")
    e2e_eager_ms = float(np.mean(timed(e2e_step, max(3, min(args.steps, 200)))))
    g_e2e = capture(e2e_step)
    e2e_ms = max_over_ranks(back_to_back(g_e2e.replay, max(3, min(args.steps, 200))), dev)
    e2e_flushed_ms = float(np.mean(timed(g_e2e.replay, max(3, min(args.steps, 200)))))
    g_copy = capture(e2e_copy_step)
    e2e_copy_ms = back_to_back(g_copy.replay, max(3, min(args.steps, 200)))
    torch.cuda.synchronize(dev)
    e2e_ok = bool(torch.equal(out_h.to(dev), out) and torch.equal(lse_h.to(dev), lse)
                  and torch.equal(res_h[:out.numel() * 2].view(torch.bfloat16).view(out.shape).to(dev), out))
    h2d = sum(t.numel() * t.element_size() for t in (q_h, pt_h, sl_h))
    d2h = sum(t.numel() * t.element_size() for t in (out_h, lse_h))
    mark.close()

    torch.cuda.synchronize(dev)
    flags = binding.sv_get_device_error(reset=True)
    if flags:
        raise SystemExit(f"device error word {flags:#x}")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return None

    ab = algorithmic_bytes(wl)
    peak, peak_kind = measured_peaks()
    per_kernel = {"score_pages_kernel": t_score, "flash_decode_split_kernel": t_dec}
    dominant = max(per_kernel, key=per_kernel.get)
    dom_ms = per_kernel[dominant]
    if dominant == "flash_decode_split_kernel":
        dom_note = "sv_sparse_decode time includes the small lse_combine kernel"
        dom_timing = "each call alone between its own events after an L2 flush"
    else:
        dom_ms = t_score_b2b
        dom_note = "sv_quest_score: one launch of score_pages_kernel"
        dom_timing = ("average launch duration: launches back to back between one pair of events (each reads "
                      "131 MB of metadata, more than L2); timed alone after an L2 flush, with its own events: "
                      f"{t_score * 1e3:.2f} us")
    achieved = ab[dominant] / (dom_ms * 1e-3) / 1e9
    step_gbs = ab["step"] / (ms_per_step * 1e-3) / 1e9
    value = whole_job_value(world, ms_per_step)

    res = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": spec.name, "batch": B, "ctx_tokens": int(wl.seq_lens[0]), "page_size": spec.page_size,
                   "budget_tokens": K * spec.page_size, "num_q_heads": Hq, "num_kv_heads": Hkv, "head_dim": D,
                   "needle_pages_per_request": spec.needles_per_request, "pool": "shuffled",
                   "l2": "not flushed: the K timed steps run back to back and each reads 198.6 MB of metadata "
                         "and K/V, more than the 126 MB L2 (per-step times with and without a flush agree, "
                         "see per_step_ms)",
                   "parallelism": f"replicas x{world}"},
        "step_bytes": ab["step"],
        "chained_10_steps_ms_per_step": round(chained_ms, 5),
        "per_step_ms": {"flushed": round(flushed_ms, 5), "not_flushed": round(noflush_ms, 5),
                        "how": "the same graph replay timed alone between its own pair of events, min(K, 200) "
                               "times, with and without an L2 flush (write one 2xL2 buffer, read another) before "
                               "each; each number also pays one launch and one event pair"},
        "step_gbs": round(step_gbs, 1),
        "step_roofline_frac": round(step_gbs / peak, 4),
        "per_kernel_ms": {"score_pages": round(t_score, 5), "score_pages_back_to_back": round(t_score_b2b, 5),
                          "topk_pages": round(t_topk, 5),
                          "sparse_decode(split+combine)": round(t_dec, 5),
                          "note": "each call timed alone after an L2 flush; the step runs them back to back"},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "algorithmic_bytes": ab[dominant],
                     "traffic": kernel_traffic(dominant), "duration_ms": round(dom_ms, 5), "timing": dom_timing,
                     "note": dom_note},
        "dense": {"steps_per_s": round(1e3 / dense_ms, 2), "ms_per_step": round(dense_ms, 5),
                  "gbs": round(ab["dense_step"] / (dense_ms * 1e-3) / 1e9, 1), "bytes": ab["dense_step"]},
        "e2e": {"value": round(whole_job_value(world, e2e_ms), 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                "how": e2e_how,
                "eager_ms_per_step": round(e2e_eager_ms, 5), "result_copied_back": e2e_ok,
                "timing": "min(K, 200) graph replays back to back between one pair of events",
                "flushed_per_step_ms": round(e2e_flushed_ms, 5),
                "copy_engine_ms_per_step": round(e2e_copy_ms, 5),
                "copy_engine_how": "CUDA graph of: one pinned host->device copy of the inputs, "
                                   "sv_quest_decode_step, one device->pinned host copy of the results"},
        "fp8_step": {"ms_per_step": round(fp8_ms, 5), "steps_per_s": round(1e3 / fp8_ms, 2),
                     "bytes": ab["fp8_step"], "gbs": round(ab["fp8_step"] / (fp8_ms * 1e-3) / 1e9, 1),
                     "sparse_decode_ms": round(fp8_dec_ms, 5),
                     "decode_gbs": round(ab["fp8_decode"] / (fp8_dec_ms * 1e-3) / 1e9, 1),
                     "same_selection_counts": fp8_same_sel,
                     "note": "same step over an e4m3 K/V pool with per-row fp32 scales (bf16 metadata), timed "
                             "back to back like the headline; sparse_decode_ms alone after an L2 flush"},
        "prefill_append": {"tokens": T, "ms": round(append_ms, 5), "bytes": append_bytes,
                           "gbs": round(append_bytes / (append_ms * 1e-3) / 1e9, 1),
                           "note": "one 4096-token chunk, one eager call between events",
                           "chunked_prefill": {
                               "tokens": L0, "chunks": len(chunks), "ms": round(prefill_ms, 5),
                               "ms_per_chunk": round(prefill_ms / len(chunks), 5), "bytes": prefill_bytes,
                               "gbs": round(prefill_bytes / (prefill_ms * 1e-3) / 1e9, 1),
                               "how": "request 0's tokens in 4096-token chunks, one sv_quest_update_meta per "
                                      "chunk, all chunks one CUDA graph"}},
        "kv_heavy_budget512": kv_heavy,
        "quest_variants": variants,
        "gpu_launches": launches_per_step * args.steps,
        "launches_per_step": launches_per_step,
        "gpu_launches_source": "kernels per call (sv_quest_decode_step: score 1 + top-K 1 + split decode 1 + combine 1), "
                               "counted by construction: the timed region replays a graph of exactly this call",
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        res["cpu_baseline"] = cpu_baseline(wl, max_seconds=args.cpu_seconds)
    return res


# ---------------------------------------------------------------- every workload (--all-configs)

def step_bytes(wl, budget_pages, appended=0):
    """Algorithmic bytes of one step at a budget: metadata + selected K/V + page
    table + q / out / lse (+ the appended tokens' K/V, pool rows and metadata)."""
    s = wl.spec
    P, Hkv, Hq, D = s.page_size, s.num_kv_heads, s.num_q_heads, s.head_dim
    n = (wl.seq_lens.astype(np.int64) + appended + P - 1) // P
    sel = np.minimum(n, budget_pages)
    b = (int(n.sum()) * Hkv * 2 * D * 2 + int(sel.sum()) * Hkv * P * D * 2 * 2 + int(n.sum()) * 4
         + s.batch * Hq * D * 2 + s.batch * Hq * (D * 2 + 4))
    if appended:
        b += appended * s.batch * Hkv * D * 2 * (2 + 2) + appended * s.batch * Hkv * 2 * D * 2
    return b


def run_only(args):
    """One call type alone on the benchmark workload, for profiling with a
    small device footprint (one bf16 or fp8 pool): --only step (the one-call
    decode step, as a CUDA graph), append (one 4096-token sv_quest_update_meta),
    fp8_step (the step over an fp8 pool) or fp8_step_budget512 (the fp8 step of
    16 requests of 65536 tokens at a 512-page budget).  W untimed and K timed calls, each
    after an L2 flush; prints one JSON line with the mean time per call."""
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    spec = synth.SPECS[BENCH_CONFIG]
    if args.only == "fp8_step_budget512":       # 16 requests of 65536 tokens, K/V-dominated
        spec = synth.SPECS[4].scaled(budget_pages=512)
    wl = synth.make_workload(spec)
    dw = resident.upload(wl, device=dev, fp8=args.only.startswith("fp8_step"))
    B, Hq, D = dw.q.shape
    Hkv, K = spec.num_kv_heads, spec.budget_pages
    sel_idx, sel_cnt = resident.select_buffers(B, Hkv, K, dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = resident.workspace(binding.sv_quest_decode_step_workspace_size(B, Hq, Hkv, wl.max_pages, K), dev)
    if args.only == "append":
        T = min(4096, int(wl.seq_lens[0]))
        k_new = resident.bf16_tensor(wl.k_tok[:T], dev)
        v_new = resident.bf16_tensor(wl.v_tok[:T], dev)
        slots = torch.from_numpy(wl.slot_mapping[:T]).to(dev)

        def call():
            binding.sv_quest_update_meta(dw.cache, k_new, v_new, slots)
    else:
        def step():
            binding.sv_quest_decode_step(dw.cache, dw.q, dw.page_table, dw.seq_lens, K, sel_idx, sel_cnt, out, lse,
                                         ws)

        step()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        call = graph.replay
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        flush_w.zero_()
        flush_r.sum()
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for e0, e1 in evs:
        flush_w.zero_()
        flush_r.sum()
        e0.record()
        call()
        e1.record()
    torch.cuda.synchronize(dev)
    ms = float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs]))
    flags = binding.sv_get_device_error(reset=True)
    if flags:
        raise SystemExit(f"device error word {flags:#x}")
    print(json.dumps({"only": args.only, "workload": spec.name, "calls": args.steps, "warmup": args.warmup,
                      "ms_per_call": round(ms, 5)}), flush=True)


def run_all_configs(args):
    """One JSON line per workload: the step (sv_quest_decode_step, CUDA graph,
    L2 flushed before each replay, median of the timed replays) and the dense
    all-pages decode, with algorithmic GB/s.  The append + sweep workload appends
    one token per request (sv_quest_update_meta) before the step, at each budget
    of the sweep."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    peak, _ = measured_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    def timed(fn, n, warm):
        for _ in range(warm):
            flush_w.zero_(); flush_r.sum(); fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize(dev)
        for e0, e1 in evs:
            flush_w.zero_(); flush_r.sum()
            e0.record(); fn(); e1.record()
        torch.cuda.synchronize(dev)
        return float(np.median([e0.elapsed_time(e1) for e0, e1 in evs]))

    def graph_of(fn):
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            fn(); fn()
        torch.cuda.current_stream(dev).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize(dev)
        return g

    n_timed, n_warm = max(20, min(args.steps, 200)), max(3, min(args.warmup, 20))
    for cfg, spec in synth.SPECS.items():
        wl = synth.make_workload(spec)
        dw = resident.upload(wl, device=dev)
        B, Hq, D = dw.q.shape
        Hkv = spec.num_kv_heads
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        line = {"config": spec.name, "batch": B, "max_pages": wl.max_pages, "pool": "shuffled" if spec.shuffle_pool
                else "contiguous"}
        appended = 0
        q = dw.q
        pre = None
        if spec.append_steps:
            appended = 1
            k1 = resident.bf16_tensor(wl.step_k[0], dev)
            v1 = resident.bf16_tensor(wl.step_v[0], dev)
            s1 = torch.from_numpy(wl.step_slots[0]).to(dev)
            dw.seq_lens.copy_(torch.from_numpy(wl.seq_lens_after(1)))
            q = resident.bf16_tensor(wl.step_q[0], dev)

            def pre():
                binding.sv_quest_update_meta(dw.cache, k1, v1, s1)
        budgets = spec.budget_sweep or (spec.budget_pages,)
        steps = []
        for K in budgets:
            sel, cnt = resident.select_buffers(B, Hkv, K, dev)
            ws = resident.workspace(binding.sv_quest_decode_step_workspace_size(B, Hq, Hkv, wl.max_pages, K), dev)

            def step(K=K, sel=sel, cnt=cnt, ws=ws):
                if pre is not None:
                    pre()
                binding.sv_quest_decode_step(dw.cache, q, dw.page_table, dw.seq_lens, K, sel, cnt, out, lse, ws)

            ms = timed(graph_of(step).replay, n_timed, n_warm)
            nb = step_bytes(wl, K, appended)
            entry = {"budget_pages": K, "us": round(ms * 1e3, 2), "steps_per_s": round(1e3 / ms, 1),
                     "bytes": nb, "gbs": round(nb / (ms * 1e-3) / 1e9, 1),
                     "frac_of_measured": round(nb / (ms * 1e-3) / 1e9 / peak, 4)}
            steps.append(entry)
            del sel, cnt, ws
        wsd = resident.workspace(binding.sv_sparse_decode_workspace_size(B, Hq, Hkv, wl.max_pages), dev)
        dense = lambda: binding.sv_sparse_decode(dw.cache, q, dw.page_table, dw.seq_lens, None, None, out, lse, wsd)
        ms = timed(graph_of(dense).replay, max(5, n_timed // 4), n_warm)
        n_all = int(((wl.seq_lens.astype(np.int64) + appended + spec.page_size - 1) // spec.page_size).sum())
        nd = n_all * Hkv * spec.page_size * D * 2 * 2 + n_all * 4 + B * Hq * (D * 2 + D * 2 + 4)
        line["step"] = steps if len(steps) > 1 else steps[0]
        line["dense"] = {"us": round(ms * 1e3, 2), "bytes": nd, "gbs": round(nd / (ms * 1e-3) / 1e9, 1)}
        line["flags"] = binding.sv_get_device_error(reset=True)
        print(json.dumps(line), flush=True)
        del dw, out, lse, wsd
        torch.cuda.empty_cache()


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

def _oracle_host(wl):
    import oracle
    oracle.build()
    oracle.build(openmp=True)
    return oracle, oracle.build_cache(wl, synth.UNFILLED_BITS)


def _oracle_step(oracle, host, wl, reqs):
    """select + sparse decode of the requests `reqs` (a slice of the batch)."""
    sel, cnt, _ = oracle.select(host, wl.q[reqs], wl.page_table[reqs], wl.seq_lens[reqs], wl.spec.budget_pages)
    oracle.decode(host, wl.q[reqs], wl.page_table[reqs], wl.seq_lens[reqs], sel, cnt)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(wl, max_seconds=10.0):
    """The oracle as it stands, timed on this host's cores on the benchmark
    workload: whole batch steps (select + sparse decode of all requests) on
    the OpenMP build, whose rows (request, head) run on every host core; the
    plain single-threaded build over whole requests; and the dense all-pages
    decode of one request on the OpenMP build, scaled to the batch."""
    oracle, host = _oracle_host(wl)
    B = wl.spec.batch
    # single thread: whole requests for about a third of the budget
    t0 = time.perf_counter()
    done = 0
    while done < B and (done < 1 or time.perf_counter() - t0 < max_seconds / 3):
        _oracle_step(oracle, host, wl, slice(done, done + 1))
        done += 1
    dt1 = time.perf_counter() - t0
    single = {"value": round(1.0 / (dt1 / done * B), 4), "unit": UNIT, "cores": 1,
              "sample": f"{done} of the {B} requests, {dt1:.2f} s; steps/s = 1 / (time per request x {B})"}
    with oracle.parallel() as threads:
        _oracle_step(oracle, host, wl, slice(0, B))            # untimed warm-up
        t0 = time.perf_counter()
        steps = 0
        while steps < 1 or time.perf_counter() - t0 < max_seconds / 3:
            _oracle_step(oracle, host, wl, slice(0, B))
            steps += 1
        dtp = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.decode(host, wl.q[:1], wl.page_table[:1], wl.seq_lens[:1])
        dtd = time.perf_counter() - t0
    return {"value": round(steps / dtp, 4), "unit": UNIT, "cores": threads, "host_cores": host_cores(),
            "kind": "oracle",
            "sample": f"{steps} whole batch-{B} steps (select + sparse decode of every request) in {dtp:.2f} s, "
                      f"OpenMP build, rows (request, head) spread over {threads} threads",
            "single_thread": single,
            "dense": {"steps_per_s": round(1.0 / (dtd * B), 4), "cores": threads,
                      "sample": f"dense all-pages decode of 1 of the {B} requests ({dtd:.2f} s, OpenMP build); "
                                f"steps/s = 1 / (that time x {B})"}}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return None
    spec = synth.SPECS[BENCH_CONFIG]
    wl = synth.make_workload(spec)
    oracle, host = _oracle_host(wl)
    B = spec.batch
    with oracle.parallel() as threads:
        for _ in range(args.warmup):
            _oracle_step(oracle, host, wl, slice(0, B))
        t0 = time.perf_counter()
        for _ in range(args.steps):
            _oracle_step(oracle, host, wl, slice(0, B))
        dt = time.perf_counter() - t0
    per_step = dt / args.steps
    value = 1.0 / per_step
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": spec.name, "batch": B, "ctx_tokens": int(wl.seq_lens[0]), "page_size": spec.page_size,
                   "budget_tokens": spec.budget_pages * spec.page_size, "num_q_heads": spec.num_q_heads,
                   "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "host_cores": host_cores(),
                         "kind": "oracle",
                         "sample": f"every step = one whole batch-{B} step (select + sparse decode of every request) "
                                   f"on the OpenMP build of the oracle, rows (request, head) over {threads} threads; "
                                   f"ms_per_step is the wall time of one such step"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--all-configs", action="store_true",
                    help="instead of the benchmark line, one line per workload (step and dense timings)")
    ap.add_argument("--only", choices=["step", "append", "fp8_step", "fp8_step_budget512"],
                    help="time one call type alone on the benchmark workload (for profiling), no benchmark line")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)     # at least three untimed warm-up steps
    if args.only:
        run_only(args)
        return
    if args.all_configs:
        run_all_configs(args)
        return
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
