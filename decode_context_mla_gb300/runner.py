"""Striped KV cache and a fixed-shape decode step built from the libdcpmla calls.

A decode step for a batch of requests is: map the new tokens' positions to
(owner shard, physical slot), write their rows into the owners' pools,
run the shard-local decode over the c shards, then merge the partials
(SGLang "Decode Context Parallelism" docs: Virtual KV layout, MLA decode
dataflow).  Each stage is one libdcpmla call on the caller's stream, so a
step can be captured in a CUDA graph.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from . import binding as B


class StripedKVCache:
    """c shard pools resident on one GPU, with the shared allocator and request map (host, C++)."""

    def __init__(self, c: int, P: int, num_pages: int, kv_dtype: int, max_requests: int,
                 max_pages_per_request: int, initial_order: Optional[torch.Tensor] = None,
                 device="cuda", fill_byte: Optional[int] = None, interleave: int = 1):
        self.c, self.P, self.num_pages, self.kv_dtype = c, P, num_pages, kv_dtype
        self.interleave = interleave
        self.max_pages = max_pages_per_request
        self.alloc = B.dcpmla_alloc_create(c, num_pages * P, P, initial_order)
        self.reqmap = B.dcpmla_reqmap_create(self.alloc, max_requests, max_pages_per_request)
        dt = torch.bfloat16 if kv_dtype == B.KV_BF16 else torch.uint8
        rows = num_pages * P
        self.pools: List[torch.Tensor] = [torch.empty((rows, B.D_K), dtype=dt, device=device)
                                          for _ in range(c)]
        if fill_byte is not None:
            for p in self.pools:
                p.view(torch.uint8).fill_(fill_byte)
        self.scales: Optional[List[torch.Tensor]] = None
        if kv_dtype == B.KV_E4M3:
            self.scales = [torch.zeros(rows, dtype=torch.float32, device=device) for _ in range(c)]
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.device = device

    @property
    def pool_rows(self) -> int:
        return self.num_pages * self.P

    def effective_page_size(self) -> int:
        return B.dcpmla_effective_page_size(self.alloc)

    def extend(self, req: int, n_new: int) -> int:
        return B.dcpmla_reqmap_extend(self.reqmap, req, n_new)

    def release(self, req: int) -> None:
        B.dcpmla_reqmap_release(self.reqmap, req)

    def tables(self, reqs: Sequence[int], max_pages: Optional[int] = None):
        """Host page table [len(reqs), max_pages] (pad -1) and lengths for `reqs`."""
        return B.dcpmla_reqmap_page_table(self.reqmap, reqs, max_pages or self.max_pages)

    def append(self, page_table_d: torch.Tensor, req_d: torch.Tensor, pos_d: torch.Tensor,
               ckv: torch.Tensor, krope: torch.Tensor, row_scales: Optional[torch.Tensor],
               owner_d: torch.Tensor, phys_d: torch.Tensor, vslot_d: Optional[torch.Tensor] = None,
               stream=None) -> None:
        """Slot map then compacting write of len(pos_d) new rows (device tensors)."""
        B.dcpmla_slot_map(page_table_d, self.num_pages, self.c, self.P, req_d, pos_d, vslot_d,
                          owner_d, phys_d, self.err, stream, interleave=self.interleave)
        B.dcpmla_kv_append(self.pools, self.scales, self.kv_dtype, owner_d, phys_d, ckv, krope,
                           row_scales, self.err, stream)

    def check_errors(self) -> int:
        return int(self.err.item())

    def close(self) -> None:
        if getattr(self, "reqmap", None):
            B.dcpmla_reqmap_destroy(self.reqmap)
            self.reqmap = None
        if getattr(self, "alloc", None):
            B.dcpmla_alloc_destroy(self.alloc)
            self.alloc = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DecodeStep:
    """Preallocated buffers for one batch shape: append Tq new tokens per request, decode, merge."""

    def __init__(self, cache: StripedKVCache, reqs: Sequence[int], Tq: int, H: int,
                 sm_scale: float, lse_base: int, append: bool = True, fused: bool = False):
        self.cache = cache
        self.reqs = list(reqs)
        self.Bn = len(self.reqs)
        self.Tq, self.H = Tq, H
        self.R = Tq * H
        self.sm_scale, self.lse_base = sm_scale, lse_base
        self.do_append = append
        self.fused = fused            # decode + merge in one call (no per-shard partials)
        dev = cache.device
        c = cache.c
        pt, lens = cache.tables(self.reqs)
        self.page_table = pt.to(dev)
        self.seq_lens = lens.to(dev)
        self.seq_lens_host = lens.clone()
        self.q = torch.empty((self.Bn, Tq, H, B.D_K), dtype=torch.bfloat16, device=dev)
        n_new = self.Bn * Tq
        dt = torch.bfloat16 if cache.kv_dtype == B.KV_BF16 else torch.uint8
        self.new_ckv = torch.empty((n_new, B.D_LATENT), dtype=dt, device=dev)
        self.new_krope = torch.empty((n_new, B.D_ROPE), dtype=dt, device=dev)
        self.new_scales = (torch.empty(n_new, dtype=torch.float32, device=dev)
                           if cache.kv_dtype == B.KV_E4M3 else None)
        # request index (row of the page table) and position of each new token
        self.new_req = torch.arange(self.Bn, dtype=torch.int32).repeat_interleave(Tq).to(dev)
        pos = torch.cat([torch.arange(int(L) - Tq, int(L), dtype=torch.int64) for L in lens])
        self.new_pos = pos.to(dev)
        self.owner = torch.empty(n_new, dtype=torch.int32, device=dev)
        self.phys = torch.empty(n_new, dtype=torch.int64, device=dev)
        self.o_part = torch.empty((c, self.Bn, Tq, H, B.D_LATENT), dtype=torch.float32, device=dev)
        self.lse_part = torch.empty((c, self.Bn, Tq, H), dtype=torch.float32, device=dev)
        self.o = torch.empty((self.Bn, Tq, H, B.D_LATENT), dtype=torch.float32, device=dev)
        self.lse = torch.empty((self.Bn, Tq, H), dtype=torch.float32, device=dev)
        ws = B.dcpmla_decode_workspace_size(self.Bn, Tq, H, cache.P, c, c, cache.kv_dtype,
                                            self.page_table.shape[1])
        if fused:
            ws = B.dcpmla_decode_merged_workspace_size(self.Bn, Tq, H, cache.P, c, cache.kv_dtype,
                                                       self.page_table.shape[1])
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)

    def run(self, stream=None) -> None:
        """Enqueue one step on the current (or given) stream."""
        self.run_append(stream)
        self.run_decode(stream)
        self.run_merge(stream)

    def run_append(self, stream=None) -> None:
        """Slot map + KV append of the step's new tokens (nothing when append is off)."""
        c = self.cache
        if self.do_append:
            c.append(self.page_table, self.new_req, self.new_pos, self.new_ckv, self.new_krope,
                     self.new_scales, self.owner, self.phys, None, stream)

    def run_decode(self, stream=None) -> None:
        """Shard-local decode of all c shards: o_part, lse_part (fused: merged o, lse)."""
        c = self.cache
        if self.fused:
            B.dcpmla_decode_merged(self.q, c.pools, c.scales, c.kv_dtype, self.page_table, self.seq_lens,
                                   c.P, c.c, self.sm_scale, self.lse_base, self.o, self.lse,
                                   self.workspace, c.err, stream, interleave=c.interleave)
            return
        B.dcpmla_decode(self.q, c.pools, c.scales, c.kv_dtype, self.page_table, self.seq_lens, c.P,
                        c.c, 0, c.c, self.sm_scale, self.lse_base, self.o_part, self.lse_part,
                        self.workspace, c.err, stream, interleave=c.interleave)

    def run_merge(self, stream=None) -> None:
        """Exact LSE merge of the c partials into o, lse (nothing to do when fused)."""
        if self.fused:
            return
        c = self.cache
        B.dcpmla_lse_merge(self.o_part, self.lse_part, c.c, self.Bn * self.R, self.lse_base,
                           self.o, self.lse, c.err, stream)

    def run_host(self, q_host: torch.Tensor, ckv_host: torch.Tensor, krope_host: torch.Tensor,
                 scales_host: Optional[torch.Tensor], o_host: torch.Tensor,
                 lse_host: torch.Tensor, stream=None) -> None:
        """End-to-end step from (pinned) host buffers: H2D inputs, run, D2H outputs."""
        self.q.copy_(q_host, non_blocking=True)
        if self.do_append:
            self.new_ckv.copy_(ckv_host, non_blocking=True)
            self.new_krope.copy_(krope_host, non_blocking=True)
            if scales_host is not None:
                self.new_scales.copy_(scales_host, non_blocking=True)
        self.run(stream)
        o_host.copy_(self.o, non_blocking=True)
        lse_host.copy_(self.lse, non_blocking=True)

    def h2d_bytes(self) -> int:
        n = self.q.numel() * 2
        if self.do_append:
            n += self.new_ckv.numel() * self.new_ckv.element_size()
            n += self.new_krope.numel() * self.new_krope.element_size()
            if self.new_scales is not None:
                n += self.new_scales.numel() * 4
        return n

    def d2h_bytes(self) -> int:
        return self.o.numel() * 4 + self.lse.numel() * 4
