"""The benchmark's host logic: its byte accounting (the roofline numerator),
checked against counts written out by hand from the layouts (per (page, kv
head) 512 bytes of metadata and 2 x 16 x 128 bf16 of K/V, 4 bytes of page
table per page, q read once and out / lse written once); the rule that drops
a profile's ncu traffic once its kernel source changes; the NVTX sections."""
from __future__ import annotations

import numpy as np

import bench
from query_aware_sparse_quest_gb300 import synth


def test_step_bytes_of_the_128k_benchmark_by_hand():
    B, n, K, Hkv, Hq, D = 8, 8000, 256, 4, 32, 128
    meta = B * n * Hkv * 512
    kv = B * K * Hkv * 16 * D * 2 * 2
    pt = B * n * 4
    q_out = B * Hq * D * 2 + B * Hq * (D * 2 + 4)
    assert meta == 131_072_000 and kv == 67_108_864
    assert meta + kv + pt + q_out == 198_568_960


def _small(spec_index, **kw):
    return synth.make_workload(synth.SPECS[spec_index].scaled(**kw))


def test_algorithmic_bytes_and_step_bytes_agree_with_hand_counts():
    wl = _small(2, batch=3, ctx=16 * 40 + 5, budget_pages=7, needles_per_request=2)
    s = wl.spec
    n = int(-(-wl.seq_lens[0] // 16))
    assert n == 41
    hand = (s.batch * n * s.num_kv_heads * 512 + s.batch * 7 * s.num_kv_heads * 8192 + s.batch * n * 4
            + s.batch * s.num_q_heads * (128 * 2 + 128 * 2 + 4))
    ab = bench.algorithmic_bytes(wl)
    assert ab["step"] == hand
    assert bench.step_bytes(wl, 7) == hand
    # the parts the roofline charges to each kernel
    assert ab["score_pages_kernel"] == (s.batch * n * s.num_kv_heads * 512 + s.batch * n * 4
                                        + s.batch * s.num_q_heads * 256 + s.batch * n * s.num_kv_heads * 4)
    assert ab["flash_decode_split_kernel"] == (s.batch * 7 * s.num_kv_heads * 8192 + s.batch * 7 * s.num_kv_heads * 8
                                               + s.batch * s.num_q_heads * 256)
    # a budget past the row keeps every page: the K/V part equals the dense one
    assert bench.step_bytes(wl, 10_000) - bench.step_bytes(wl, 7) == s.batch * (n - 7) * s.num_kv_heads * 8192


def test_step_bytes_count_the_appended_token():
    wl = _small(4, batch=2, ctx=16 * 30)
    s = wl.spec
    base = bench.step_bytes(wl, 5)
    with_append = bench.step_bytes(wl, 5, appended=1)
    # one more page per request (31 instead of 30) adds its metadata and table entry,
    # and the appended token's K/V are read, written to the pool and its page's min/max rebuilt
    extra_pages = s.batch * 1
    expect = (extra_pages * s.num_kv_heads * 512 + extra_pages * 4
              + s.batch * s.num_kv_heads * 128 * 2 * 4 + s.batch * s.num_kv_heads * 2 * 128 * 2)
    assert with_append - base == expect
    assert np.all(wl.seq_lens == 16 * 30)


def test_kernel_traffic_is_dropped_once_the_source_changes(tmp_path, monkeypatch):
    """The ncu traffic of a committed profile is reported only while the
    kernel's source still hashes to the value stored beside it."""
    import hashlib
    src = tmp_path / "kernel.cu"
    src.write_text("__global__ void k() {}\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    prof = tmp_path / "k.txt"
    prof.write_text("# summary\nk.source_sha256_16=%s\nk.dram_bytes_per_launch_full_size=123456\n" % digest)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.PROFILE_SUMMARIES, "k", "k.txt")
    monkeypatch.setitem(bench.KERNEL_SOURCES, "k", "kernel.cu")
    assert bench.kernel_traffic("k") == 123456.0
    src.write_text("__global__ void k() { }\n")   # any edit of the source
    assert bench.kernel_traffic("k") is None


def test_sections_open_and_close_nvtx_ranges_in_pairs(monkeypatch):
    calls = []

    class FakeNvtx:
        @staticmethod
        def range_push(name):
            calls.append(("push", name))

        @staticmethod
        def range_pop():
            calls.append(("pop",))

    monkeypatch.setattr(bench.torch.cuda, "nvtx", FakeNvtx)
    mark = bench.Sections()
    calls.clear()
    mark("a")
    mark("b")
    mark.close()
    mark.close()
    assert calls == [("push", "a"), ("pop",), ("push", "b"), ("pop",)]
