"""Oracle results for a seeded workload, built on the CPU from the shared input generators.

Inputs come only from dcp_workloads (the same counter-based generator the GPU
side uses); expected values come only from the oracle.
"""
from __future__ import annotations

from typing import Dict, Iterable

import numpy as np
import torch

import dcp_workloads as W
import oracle as O


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(t.dtype)


class OracleWorkload:
    """The oracle's allocator replay and request map for a workload, plus lazily built pools."""

    def __init__(self, w: W.Workload):
        self.w = w
        self.lens = w.seq_lens()
        pages = w.pages_per_request()
        order = W.free_list_order(w.seed, sum(pages))
        self.alloc = O.SharedVirtualAllocator(w.c, sum(pages) * w.P, w.P, order.tolist())
        self.rmap = O.RequestTokenMap(self.alloc)
        for b, L in enumerate(self.lens):
            self.rmap.extend(b, L)
        self.pools = O.ShardPools(w.c, w.P, w.kv_dtype)
        self.loaded = set()

    def page_table(self) -> np.ndarray:
        return self.rmap.page_table(range(self.w.B), max(self.w.pages_per_request()))

    def load(self, b: int, gen_device="cpu", chunk: int = 1 << 18) -> None:
        if b in self.loaded:
            return
        L = self.lens[b]
        for p0 in range(0, L, chunk):
            p1 = min(L, p0 + chunk)
            rows, scales = W.kv_rows(self.w, b, p0, p1, gen_device)
            sc = None if scales is None else scales.cpu().numpy()
            O.append_tokens(self.pools, self.rmap, b, np.arange(p0, p1), bits(rows), sc,
                            I=self.w.interleave)
        self.loaded.add(b)

    def q(self, b: int, gen_device="cpu") -> np.ndarray:
        return O.bf16_to_f64(bits(W.q_tensor(self.w, gen_device, requests=[b])[0]))

    def decode(self, b: int, gen_device="cpu"):
        """(o_parts (c,R,512), lse_parts (c,R), o (R,512), lse (R,)) for request b."""
        self.load(b, gen_device)
        return O.decode_request_striped(self.q(b, gen_device), self.pools, self.rmap, b,
                                        self.lens[b], self.w.sm_scale, self.w.lse_base,
                                        I=self.w.interleave)

    def decode_many(self, reqs: Iterable[int], gen_device="cpu") -> Dict[int, tuple]:
        return {b: self.decode(b, gen_device) for b in reqs}


def row_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of ||got - ref||_inf / ||ref||_inf (absolute where the reference row is 0)."""
    got = np.asarray(got, dtype=np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    num = np.abs(got - ref).max(axis=1)
    den = np.abs(ref).max(axis=1)
    den = np.where(den > 0, den, 1.0)
    return float((num / den).max()) if len(num) else 0.0


def lse_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / max(|ref|, 1); -inf must meet -inf exactly (else returns inf)."""
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    ninf_g, ninf_r = np.isneginf(got), np.isneginf(ref)
    if not np.array_equal(ninf_g, ninf_r):
        return float("inf")
    live = ~ninf_r
    if not np.any(live):
        return 0.0
    return float((np.abs(got[live] - ref[live]) / np.maximum(np.abs(ref[live]), 1.0)).max())


TOL = {"bf16": 2e-3, "e4m3": 1e-2}
