"""Seeded synthetic workloads for striped absorbed-MLA decode.

This module is shared by the fp64 oracle tests, the GPU parity tests and the
benchmark.  It holds the five workload definitions and counter-based input
generators, and nothing of the method's arithmetic: no striping, no
allocation, no attention and no merge.  Every value is a pure function of
(seed, stream, counter), computed with 64-bit integer operations plus one
IEEE float32 multiply and one round-to-nearest-even conversion, so the CPU
and the GPU produce bit-identical inputs.  That lets the oracle regenerate
any request's keys on the host without copying the device cache back.

Workload shapes follow the pages' deployments: absorbed MLA with a 512-d
latent and a 64-d rope key, scores taken over all 576 dims and values over
the 512-d latent (vLLM GLM-5.3 serving post, footnote arithmetic section);
striping size c and physical page
P as in the SGLang DCP docs (section "Virtual KV layout"); the bimodal
context mix of agentic traffic (vLLM DCP explainer, section "Why focus on
decode": about 53% of requests at 64K tokens or more, the rest below 64K).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import List, Optional

import torch

D_LATENT = 512
D_ROPE = 64
D_K = D_LATENT + D_ROPE

M32 = 0xFFFFFFFF
_HASH_MUL = 0x45D9F3B          # < 2**27, so products of 32-bit values stay < 2**63
_IH4_STD = math.sqrt(4 * (256 * 256 - 1) / 12.0)   # std of a sum of four uniform bytes
_IH4_MEAN = 510                                      # mean of that sum (4 * 255 / 2)

# Sub-stream ids.
STREAM_Q = 1
STREAM_KV = 2
STREAM_LENGTHS = 3
STREAM_ALLOC = 4


# --------------------------------------------------------------------------
# Counter-based generator (32-bit integer finaliser, applied to int64 tensors)
# --------------------------------------------------------------------------
def hash32(x: torch.Tensor) -> torch.Tensor:
    """Integer avalanche finaliser on values in [0, 2**32); returns the same range."""
    x = ((x >> 16) ^ x) * _HASH_MUL & M32
    x = ((x >> 16) ^ x) * _HASH_MUL & M32
    return (x >> 16) ^ x


def _hash32_int(v: int) -> int:
    return int(hash32(torch.tensor([v & M32], dtype=torch.int64))[0])


def stream_key(seed: int, stream: int) -> int:
    return _hash32_int((seed & M32) ^ _hash32_int(stream * 0x9E37 + 0x7F4A))


def counter_bits(seed: int, stream: int, hi, lo: torch.Tensor) -> torch.Tensor:
    """32 random bits per element for counter (hi, lo); hi is an int or an int64 tensor."""
    key = stream_key(seed, stream)
    if isinstance(hi, int):
        h_hi = _hash32_int((hi + key) & M32)
    else:
        h_hi = hash32((hi + key) & M32)
    return hash32((lo & M32) ^ h_hi)


def normal_f32(bits: torch.Tensor) -> torch.Tensor:
    """Approximately N(0,1): centred sum of the four bytes of `bits`, unit variance."""
    s = (bits & 255) + ((bits >> 8) & 255) + ((bits >> 16) & 255) + (bits >> 24)
    inv = torch.tensor(1.0 / _IH4_STD, dtype=torch.float32, device=bits.device)
    return (s - _IH4_MEAN).to(torch.float32) * inv


def uniform_int(bits: torch.Tensor, lo: int, hi_inclusive: int) -> torch.Tensor:
    return lo + bits % (hi_inclusive - lo + 1)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    B: int                    # requests
    H: int                    # query heads (TP-local)
    Tq: int                   # query tokens per request (1 + draft tokens)
    c: int                    # DCP size: number of shard pools
    P: int                    # physical page size (tokens)
    kv_dtype: str             # "bf16" or "e4m3"
    lse_base: str             # "e" or "2"
    seed: int
    L: Optional[int] = None   # fixed context length (tokens attended, after append)
    lengths_mix: Optional[tuple] = None   # (n_long, long_lo, long_hi, short_lo, short_hi)
    sm_scale: float = 1.0 / math.sqrt(192.0)
    description: str = ""
    interleave: int = 1       # tokens go to shards in runs of this many positions

    @property
    def rows_per_request(self) -> int:
        return self.Tq * self.H

    @property
    def virtual_page(self) -> int:
        return self.P * self.c

    def seq_lens(self) -> List[int]:
        if self.lengths_mix is None:
            return [int(self.L)] * self.B
        n_long, llo, lhi, slo, shi = self.lengths_mix
        idx = torch.arange(self.B, dtype=torch.int64)
        bits = counter_bits(self.seed, STREAM_LENGTHS, 0, idx)
        long_l = uniform_int(bits, llo, lhi)
        bits2 = counter_bits(self.seed, STREAM_LENGTHS, 1, idx)
        short_l = uniform_int(bits2, slo, shi)
        lens = torch.where(idx < n_long, long_l, short_l)
        # seeded shuffle: order requests by a hash key (stable on ties)
        key = counter_bits(self.seed, STREAM_LENGTHS, 2, idx)
        order = torch.sort(key, stable=True).indices
        return [int(v) for v in lens[order]]

    def pages_per_request(self) -> List[int]:
        vp = self.virtual_page
        return [(L + vp - 1) // vp for L in self.seq_lens()]

    def num_pages(self) -> int:
        return sum(self.pages_per_request())

    def kv_bytes_per_token(self) -> int:
        return D_K * 2 if self.kv_dtype == "bf16" else D_K + 4


def free_list_order(seed: int, num_pages: int) -> torch.Tensor:
    """Seeded permutation of page ids 0..num_pages-1 (the allocator's initial free list)."""
    idx = torch.arange(num_pages, dtype=torch.int64)
    key = counter_bits(seed, STREAM_ALLOC, 0, idx)
    return torch.sort(key, stable=True).indices.to(torch.int32)


_BIMODAL_MIX = (round(0.53 * 256), 65536, 262144, 1024, 65535)

WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=16, Tq=1, c=4, P=16, kv_dtype="bf16", lse_base="e",
                     seed=1, L=1024,
                     description="batch 1, 16 heads, context 1024, c=4, P=16, base-e LSE"),
    "dsv3": Workload("dsv3", B=32, H=128, Tq=1, c=8, P=64, kv_dtype="bf16", lse_base="2",
                     seed=2, L=32768,
                     description="DeepSeek-V3-shaped decode: batch 32, 128 heads, context 32768, "
                                 "c=8, P=64, base-2 LSE"),
    "long": Workload("long", B=4, H=16, Tq=1, c=8, P=64, kv_dtype="bf16", lse_base="e",
                     seed=3, L=1048576,
                     description="long context: batch 4, 16 heads, context 1048576, c=8, P=64, "
                                 "one appended token per request per step"),
    "bimodal": Workload("bimodal", B=256, H=16, Tq=1, c=2, P=16, kv_dtype="bf16", lse_base="e",
                        seed=4, lengths_mix=_BIMODAL_MIX,
                        description="256 requests, 16 heads, 136 contexts U[65536,262144] + "
                                    "120 U[1024,65535], c=2, P=16, random page tables"),
    "fp8": Workload("fp8", B=64, H=128, Tq=4, c=8, P=64, kv_dtype="e4m3", lse_base="2",
                    seed=5, L=65536,
                    description="e4m3 KV with per-token fp32 scale + target verification: batch 64, "
                                "128 heads, 4 causal query tokens, context 65536, c=8, P=64"),
}


def scaled(w: Workload, **kw) -> Workload:
    """Same structure, smaller sizes (for oracle-checkable parity cases)."""
    return replace(w, **kw)


# --------------------------------------------------------------------------
# Input tensors
# --------------------------------------------------------------------------
def q_tensor(w: Workload, device="cpu", requests=None) -> torch.Tensor:
    """Q as bf16 [B, Tq, H, 576]: absorbed latent query (512) then rope query (64)."""
    reqs = list(range(w.B)) if requests is None else list(requests)
    lo = torch.arange(w.Tq * w.H * D_K, dtype=torch.int64, device=device)
    out = torch.empty((len(reqs), w.Tq, w.H, D_K), dtype=torch.bfloat16, device=device)
    for i, b in enumerate(reqs):
        bits = counter_bits(w.seed, STREAM_Q, b, lo)
        out[i] = normal_f32(bits).to(torch.bfloat16).view(w.Tq, w.H, D_K)
    return out


def kv_f32(w: Workload, b: int, p0: int, p1: int, device="cpu") -> torch.Tensor:
    """Unrounded float32 key rows [p1-p0, 576] of request b, positions p0..p1-1."""
    lo = (torch.arange(p0, p1, dtype=torch.int64, device=device)[:, None] * D_K
          + torch.arange(D_K, dtype=torch.int64, device=device)[None, :])
    return normal_f32(counter_bits(w.seed, STREAM_KV, b, lo))


def kv_rows(w: Workload, b: int, p0: int, p1: int, device="cpu"):
    """Stored key rows of request b at positions p0..p1-1, in the cache's storage format.

    bf16: returns (rows bf16 [n, 576], None).
    e4m3: returns (codes uint8 [n, 576], scale float32 [n]); the value of element d
    of row i is float(e4m3 code) * scale[i] (OCP E4M3FN, one scale per token).
    """
    x = kv_f32(w, b, p0, p1, device)
    if w.kv_dtype == "bf16":
        return x.to(torch.bfloat16), None
    amax = x.abs().amax(dim=1)
    fmax = torch.tensor(448.0, dtype=torch.float32, device=x.device)
    tiny = torch.tensor(1e-30, dtype=torch.float32, device=x.device)
    scale = torch.maximum(amax, tiny) / fmax
    y = torch.clamp(x / scale[:, None], -448.0, 448.0)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """uint16 bit patterns of a bf16 tensor, as int32 (for hashing / exact comparison)."""
    return t.view(torch.int16).to(torch.int32) & 0xFFFF
