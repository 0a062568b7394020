"""Device-resident copy of a synthetic workload, prefilled through the library.

Allocation (torch) and host->device copies only; the pool and its metadata
are written by sv_quest_update_meta, chunk by chunk, like a chunked prefill.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import binding
from .synth import UNFILLED_BITS, Workload


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device, non_blocking=False)


@dataclasses.dataclass
class DeviceWorkload:
    wl: Workload
    cache: binding.Cache
    q: torch.Tensor            # bf16 [B][Hq][D]
    page_table: torch.Tensor   # int32 [B][max_pages]
    seq_lens: torch.Tensor     # int32 [B]

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])


def upload(wl: Workload, device="cuda", prefill: bool = True, chunk_tokens: int = 4096,
           fill_bits: int = UNFILLED_BITS, fp8: bool = False, fill_code: int = 0x7F,
           fill_scale: float = float("nan")) -> DeviceWorkload:
    """Allocates the pool (unfilled slots hold the bf16 pattern `fill_bits`;
    for an fp8 pool the e4m3 code `fill_code` and the scale `fill_scale`),
    copies q / page table / lengths, and appends the prefill stream."""
    s = wl.spec
    shape = (wl.num_phys_pages, s.num_kv_heads, s.page_size, s.head_dim)
    meta = torch.zeros((wl.num_phys_pages, s.num_kv_heads, 2, s.head_dim), dtype=torch.bfloat16, device=device)
    if fp8:
        k = torch.full(shape, int(fill_code), dtype=torch.uint8, device=device)
        v = k.clone()
        ks = torch.full(shape[:3], float(fill_scale), dtype=torch.float32, device=device)
        vs = ks.clone()
        cache = binding.Cache(k, v, meta, ks, vs)
    else:
        k = torch.full(shape, int(np.int16(np.uint16(fill_bits))), dtype=torch.int16, device=device).view(torch.bfloat16)
        v = k.clone()
        cache = binding.Cache(k, v, meta)
    dw = DeviceWorkload(wl=wl, cache=cache, q=bf16_tensor(wl.q, device),
                        page_table=torch.from_numpy(wl.page_table).to(device),
                        seq_lens=torch.from_numpy(wl.seq_lens).to(device))
    if prefill:
        for a, b in wl.prefill_chunks(chunk_tokens):
            kt = bf16_tensor(wl.k_tok[a:b], device)
            vt = bf16_tensor(wl.v_tok[a:b], device)
            sm = torch.from_numpy(wl.slot_mapping[a:b]).to(device)
            binding.sv_quest_update_meta(cache, kt, vt, sm)
    return dw


def select_buffers(batch: int, num_kv_heads: int, budget_pages: int, device="cuda"):
    sel_idx = torch.empty((batch, num_kv_heads, budget_pages), dtype=torch.int32, device=device)
    sel_cnt = torch.empty((batch, num_kv_heads), dtype=torch.int32, device=device)
    return sel_idx, sel_cnt


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(1, int(nbytes)), dtype=torch.uint8, device=device)
