"""Sets up a seeded workload on the GPU through the library's public API.

Shared by the GPU tests, the benchmark and the smoke check.  It builds the
striped cache for a `dcp_workloads.Workload`: the C++ allocator hands out
virtual pages in a seeded order, every request's earlier tokens are written
with the library's slot-map + KV-append calls, and a `DecodeStep` holds the
step's inputs (the queries and the Tq new tokens per request).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import torch

import dcp_workloads as W
from decode_context_mla_gb300 import binding as B
from decode_context_mla_gb300.runner import DecodeStep, StripedKVCache


def kv_code(w: W.Workload) -> int:
    return B.KV_BF16 if w.kv_dtype == "bf16" else B.KV_E4M3


def base_code(w: W.Workload) -> int:
    return B.LSE_2 if w.lse_base == "2" else B.LSE_E


@dataclass
class DeviceWorkload:
    w: W.Workload
    cache: StripedKVCache
    step: DecodeStep
    lens: List[int]
    order: torch.Tensor


def build(w: W.Workload, device="cuda", chunk_tokens: int = 1 << 18,
          fill_byte: Optional[int] = None, append: bool = True, fused: bool = False) -> DeviceWorkload:
    lens = w.seq_lens()
    pages = w.pages_per_request()
    num_pages = sum(pages)
    order = W.free_list_order(w.seed, num_pages)
    cache = StripedKVCache(w.c, w.P, num_pages, kv_code(w), max_requests=w.B,
                           max_pages_per_request=max(pages), initial_order=order, device=device,
                           fill_byte=fill_byte, interleave=w.interleave)
    for b, L in enumerate(lens):
        cache.extend(b, L)
    step = DecodeStep(cache, range(w.B), w.Tq, w.H, w.sm_scale, base_code(w), append=append, fused=fused)

    # Earlier tokens (positions 0 .. L-Tq-1) go in through the same append path.
    n_pre = 0
    for b, L in enumerate(lens):
        upto = L - w.Tq if append else L
        for p0 in range(0, upto, chunk_tokens):
            p1 = min(upto, p0 + chunk_tokens)
            write_rows(w, cache, step.page_table, b, p0, p1, device)
            n_pre += p1 - p0
    step.q.copy_(W.q_tensor(w, device))
    if append:
        fill_new_rows(w, step, lens, device)
    torch.cuda.synchronize()
    err = cache.check_errors()
    if err:
        raise RuntimeError(f"device error bits {err} while building {w.name}")
    return DeviceWorkload(w, cache, step, lens, order)


def write_rows(w: W.Workload, cache: StripedKVCache, page_table_d: torch.Tensor, b: int, p0: int,
               p1: int, device) -> None:
    rows, scales = W.kv_rows(w, b, p0, p1, device)
    n = p1 - p0
    req = torch.full((n,), b, dtype=torch.int32, device=device)
    pos = torch.arange(p0, p1, dtype=torch.int64, device=device)
    owner = torch.empty(n, dtype=torch.int32, device=device)
    phys = torch.empty(n, dtype=torch.int64, device=device)
    cache.append(page_table_d, req, pos, rows[:, :W.D_LATENT], rows[:, W.D_LATENT:], scales,
                 owner, phys)


def new_rows_host(w: W.Workload, lens: List[int]):
    """The step's new tokens (the last Tq positions of each request), as host tensors."""
    rows, scales = [], []
    for b, L in enumerate(lens):
        r, s = W.kv_rows(w, b, L - w.Tq, L, "cpu")
        rows.append(r)
        if s is not None:
            scales.append(s)
    rows = torch.cat(rows)
    return rows, (torch.cat(scales) if scales else None)


def fill_new_rows(w: W.Workload, step: DecodeStep, lens: List[int], device) -> None:
    for b, L in enumerate(lens):
        r, s = W.kv_rows(w, b, L - w.Tq, L, device)
        sl = slice(b * w.Tq, (b + 1) * w.Tq)
        step.new_ckv[sl].copy_(r[:, :W.D_LATENT])
        step.new_krope[sl].copy_(r[:, W.D_LATENT:])
        if s is not None:
            step.new_scales[sl].copy_(s)
