"""fp64 CPU oracle for striped absorbed-MLA decode with an exact LSE merge.

TEST INFRASTRUCTURE ONLY.  This module is what the CUDA path is checked
against.  Only the tests, the smoke check and the benchmark's CPU-baseline
leg may import it; the library and its Python binding never do.  It shares no
code with the CUDA path: it takes plain numpy arrays and imports nothing from
the package.

Sources, by page and section:
  [SG-VKV]   SGLang "Decode Context Parallelism" docs, Architecture > Virtual KV
             layout: virtual capacity C*c, virtual page P*c, owner(v) = v mod c,
             physical(v) = floor(v/c); one shared request->token map; a rank keeps
             the positions it owns and compacts them into its physical pool.
  [SG-WHY]   same page, "Why decode context parallelism?": figure with c = 4 and
             tokens 0..7, rank r holding tokens r and r+4.
  [SG-FLOW]  same page, "MLA decode dataflow": shard r returns a locally
             normalised o_r and lse_r; lse = logsumexp_r(lse_r),
             o = sum_r exp(lse_r - lse) * o_r, exact up to reduction order, in the
             attention backend's LSE base (e or 2).
  [SG-SPEC]  same page, "DCP x speculative decoding": target verification runs on
             the shard with cp_world, cp_rank and the global KV length, so the
             causal mask sees global positions.
  [VL-DCP]   vLLM "Context Parallel Deployment", Decode Context Parallel: the
             effective block size is the physical block times the DCP size.
  [GLM-FN]   vLLM GLM-5.3 serving post, footnote arithmetic: absorbed MLA scores
             use the 576-d key (512 latent + 64 rope), values the 512-d latent.
  [SG-PD]    SGLang DCP docs, "DCP x PD disaggregation": dense prefill pages are not
             copied straight into striped decode storage; a DCP-1 prefill feeds DCP
             decode through a token relayout whose plan carries the exact token
             count, so a partial final page leaks no stale rows; physical page size
             and KV dtype match on both sides.
  [SG-EXT]   same page, "Communication backends", closing paragraph: extend gathers
             the cached prefix shards and restores token order (work that grows
             with the prefix).
  [GLM-AG]   vLLM GLM-5.3 serving post, "DCP: split the KV cache too": the prefill
             engine gathers the shards into a temporary full-context copy.
  [SG-HIC]   SGLang DCP docs, "DCP x HiCache L2": the controller addresses P*c slots
             per widened page while each buffer stores its P local rows; before a
             transfer both index lists keep the positions this rank owns and map
             i to floor(i / c).
  [VW-ILV]   vLLM DCP study page (llm-wiki), configuration example: the DCP KV
             interleave size (default 1 token) hands out tokens to ranks in runs of
             that many; larger runs trade balance for less sorting.

Readings where the pages are silent (each listed in the design notes):
  * the query of draft token t (of Tq) sits at global position L - Tq + t and sees
    keys at positions <= its own; Tq = 1 gives position L - 1;
  * a shard with no visible key returns lse = -inf and o = 0;
  * base-2 LSE is the natural LSE divided by ln 2;
  * e4m3 is OCP E4M3FN with one float scale per token over all 576 values.

Everything is computed in float64 from the stored bf16 / e4m3 bit patterns.
Matrix products use numpy's matmul as a library primitive; there is no
blocking, no online softmax and no reordering beyond the definitions above.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

D_LATENT = 512
D_ROPE = 64
D_K = D_LATENT + D_ROPE
LN2 = math.log(2.0)


# ---------------------------------------------------------------------------
# Virtual KV layout  [SG-VKV], [VL-DCP]
# ---------------------------------------------------------------------------
def virtual_capacity(C: int, c: int) -> int:
    """Tokens addressable through the shared allocator: per-rank capacity C times c."""
    return C * c


def virtual_page_size(P: int, c: int) -> int:
    """A virtual page spans P tokens on each of the c ranks."""
    return P * c


def effective_page_size(P: int, c: int) -> int:
    """Attention block size the engine reports with DCP on ([VL-DCP])."""
    return P * c


def owner(v, c: int):
    """Rank that stores virtual slot v."""
    return v % c


def physical(v, c: int):
    """Slot of virtual slot v inside its owner's compacted physical pool."""
    return v // c


class AllocatorExhausted(RuntimeError):
    pass


class SharedVirtualAllocator:
    """The one allocator every rank shares ([SG-VKV]).

    A page id g names virtual page g (virtual slots g*P*c .. g*P*c + P*c - 1),
    which is physical page g (physical slots g*P .. g*P + P - 1) on every rank.
    Pages are handed out from the front of the free list and returned to its
    back; `order` fixes the initial free list (default: ascending ids).
    """

    def __init__(self, c: int, phys_capacity_tokens: int, P: int,
                 order: Optional[Sequence[int]] = None):
        if c < 1 or P < 1 or phys_capacity_tokens < 0 or phys_capacity_tokens % P:
            raise ValueError("bad allocator geometry")
        self.c = c
        self.P = P
        self.C = phys_capacity_tokens
        self.num_pages = phys_capacity_tokens // P
        if order is None:
            free = list(range(self.num_pages))
        else:
            free = [int(x) for x in order]
            if sorted(free) != list(range(self.num_pages)):
                raise ValueError("order must be a permutation of the page ids")
        self.free = free
        self.in_use = set()

    @property
    def virtual_capacity(self) -> int:
        return virtual_capacity(self.C, self.c)

    @property
    def virtual_page(self) -> int:
        return virtual_page_size(self.P, self.c)

    def alloc(self, n: int) -> List[int]:
        if n < 0:
            raise ValueError("negative page count")
        if n > len(self.free):
            raise AllocatorExhausted(f"need {n} pages, {len(self.free)} free")
        out = self.free[:n]
        del self.free[:n]
        self.in_use.update(out)
        return out

    def release(self, ids: Sequence[int]) -> None:
        ids = [int(x) for x in ids]
        for g in ids:
            if g not in self.in_use:
                raise ValueError(f"page {g} is not allocated")
        for g in ids:
            self.in_use.remove(g)
            self.free.append(g)


class RequestTokenMap:
    """The request -> virtual-token map that all ranks share ([SG-VKV]).

    Request b's positions 0..len-1 are laid out in order over its list of
    virtual pages: position p is virtual slot pages[p // (P*c)] * (P*c) + p % (P*c).
    """

    def __init__(self, alloc: SharedVirtualAllocator):
        self.alloc = alloc
        self.pages: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}

    def extend(self, b: int, n_new: int) -> np.ndarray:
        """Grow request b by n_new tokens; allocate virtual pages as needed; return the new positions."""
        cur = self.lens.get(b, 0)
        new_len = cur + n_new
        vp = self.alloc.virtual_page
        need = -(-new_len // vp) - len(self.pages.get(b, []))
        if need > 0:
            self.pages.setdefault(b, []).extend(self.alloc.alloc(need))
        else:
            self.pages.setdefault(b, [])
        self.lens[b] = new_len
        return np.arange(cur, new_len, dtype=np.int64)

    def release(self, b: int) -> None:
        self.alloc.release(self.pages.pop(b, []))
        self.lens.pop(b, None)

    def vslot(self, b: int, p) -> np.ndarray:
        p = np.asarray(p, dtype=np.int64)
        if np.any(p < 0) or np.any(p >= self.lens.get(b, 0)):
            raise IndexError("position outside the request")
        vp = self.alloc.virtual_page
        pages = np.asarray(self.pages[b], dtype=np.int64)
        return pages[p // vp] * vp + p % vp

    def page_table(self, requests: Sequence[int], max_pages: int, pad: int = -1) -> np.ndarray:
        out = np.full((len(requests), max_pages), pad, dtype=np.int32)
        for i, b in enumerate(requests):
            pg = self.pages.get(b, [])
            if len(pg) > max_pages:
                raise ValueError("max_pages too small")
            out[i, :len(pg)] = pg
        return out


def map_positions(rmap: RequestTokenMap, b: int, positions,
                  I: int = 1) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Position -> (virtual slot, owner rank, physical slot) for request b ([SG-VKV]);
    with an interleave size I > 1 the owner and slot follow owner_i / physical_i ([VW-ILV])."""
    v = rmap.vslot(b, positions)
    c = rmap.alloc.c
    if I == 1:
        return v, owner(v, c), physical(v, c)
    return v, owner_i(v, c, I), physical_i(v, c, I)


# ---------------------------------------------------------------------------
# Shard pools and the compacting write  [SG-VKV]
# ---------------------------------------------------------------------------
class ShardPools:
    """c physical pools of stored rows, kept sparse by physical page.

    pools[r][g] is a (P, 576) array of stored bit patterns (uint16 for bf16,
    uint8 for e4m3); scales[r][g] is a (P,) float32 array (e4m3 only).
    `written[r]` records every physical slot a write touched.
    """

    def __init__(self, c: int, P: int, kv_dtype: str):
        if kv_dtype not in ("bf16", "e4m3"):
            raise ValueError(kv_dtype)
        self.c, self.P, self.kv_dtype = c, P, kv_dtype
        self.dt = np.uint16 if kv_dtype == "bf16" else np.uint8
        self.pools: List[Dict[int, np.ndarray]] = [dict() for _ in range(c)]
        self.scales: List[Dict[int, np.ndarray]] = [dict() for _ in range(c)]
        self.written: List[set] = [set() for _ in range(c)]

    def _page(self, r: int, g: int):
        if g not in self.pools[r]:
            self.pools[r][g] = np.zeros((self.P, D_K), dtype=self.dt)
            self.scales[r][g] = np.zeros((self.P,), dtype=np.float32)
        return self.pools[r][g], self.scales[r][g]

    def write(self, r: int, slot: int, row: np.ndarray, scale: Optional[float] = None) -> None:
        g, off = divmod(int(slot), self.P)
        page, sc = self._page(r, g)
        page[off] = row
        if scale is not None:
            sc[off] = scale
        self.written[r].add(int(slot))

    def read(self, r: int, slots: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        slots = np.asarray(slots, dtype=np.int64)
        if len(slots) == 0:
            return np.zeros((0, D_K), dtype=self.dt), np.zeros((0,), dtype=np.float32)
        g, off = slots // self.P, slots % self.P
        pages, inv = np.unique(g, return_inverse=True)
        rows = np.stack([self.pools[r][int(x)] for x in pages])[inv, off]
        scales = np.stack([self.scales[r][int(x)] for x in pages])[inv, off]
        return rows, scales


def append_tokens(pools: ShardPools, rmap: RequestTokenMap, b: int, positions,
                  rows: np.ndarray, row_scales: Optional[np.ndarray] = None, I: int = 1) -> None:
    """Compacting write: each new token goes only to the rank that owns its slot, at physical(v).

    Rows are written page by page (a page of one rank at a time); within the
    call, a later row for the same slot overwrites an earlier one.
    """
    positions = np.asarray(positions, dtype=np.int64)
    rows = np.asarray(rows)
    v, r, s = map_positions(rmap, b, positions, I)
    P = pools.P
    for rank in np.unique(r):
        idx = np.nonzero(r == rank)[0]
        idx = idx[np.argsort(s[idx] // P, kind="stable")]     # group by physical page
        pages = s[idx] // P
        ids, starts = np.unique(pages, return_index=True)
        bounds = list(starts[1:]) + [len(idx)]
        for g, lo, hi in zip(ids, starts, bounds):
            sel = idx[lo:hi]
            page, sc = pools._page(int(rank), int(g))
            page[s[sel] % P] = rows[sel]
            if row_scales is not None:
                sc[s[sel] % P] = np.asarray(row_scales)[sel]
            pools.written[int(rank)].update(s[sel].tolist())


def shard_view(rmap: RequestTokenMap, b: int, L: int, r: int,
               I: int = 1) -> Tuple[np.ndarray, np.ndarray]:
    """Rank r's part of request b's first L positions: (global positions, physical slots), in position order."""
    p = np.arange(L, dtype=np.int64)
    v = rmap.vslot(b, p) if L > 0 else np.zeros(0, dtype=np.int64)
    c = rmap.alloc.c
    keep = (owner(v, c) if I == 1 else owner_i(v, c, I)) == r
    return p[keep], (physical(v[keep], c) if I == 1 else physical_i(v[keep], c, I))


# ---------------------------------------------------------------------------
# Stored formats -> float64
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (a bf16 value is the top half of a float32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3FN codes -> float64: 1 sign, 4 exponent (bias 7), 3 mantissa bits.

    Exponent field 0 is subnormal (m/8 * 2**-6); S.1111.111 is NaN; there are no
    infinities, so exponent field 15 with mantissa < 7 is an ordinary value.
    """
    u = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(u & 0x80, -1.0, 1.0)
    e = (u >> 3) & 0xF
    m = (u & 0x7).astype(np.float64)
    val = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 0xF) & (m == 7), np.nan, val)
    return sign * val


def dequant(rows: np.ndarray, scales: np.ndarray, kv_dtype: str) -> np.ndarray:
    if kv_dtype == "bf16":
        return bf16_to_f64(rows)
    return e4m3_to_f64(rows) * scales.astype(np.float64)[:, None]


# ---------------------------------------------------------------------------
# Attention over one key set, and the merge  [GLM-FN], [SG-FLOW], [SG-SPEC]
# ---------------------------------------------------------------------------
def attend(q: np.ndarray, k: np.ndarray, kpos: np.ndarray, qpos: np.ndarray,
           sm_scale: float, base: str = "e") -> Tuple[np.ndarray, np.ndarray]:
    """Softmax attention of R query rows over n keys, normalised over those keys only.

    q: (R, 576) float64, absorbed latent query then rope query.
    k: (n, 576) float64, latent c_kv then rope key; the value of key j is k[j, :512].
    Key j is visible to row i iff kpos[j] <= qpos[i].
    Returns o (R, 512) and lse (R,) in the requested base; rows with no
    visible key get o = 0 and lse = -inf.
    """
    R = q.shape[0]
    n = k.shape[0]
    o = np.zeros((R, D_LATENT), dtype=np.float64)
    lse = np.full((R,), -np.inf, dtype=np.float64)
    if n == 0 or R == 0:
        return o, lse
    s = sm_scale * (q @ k.T)                                    # (R, n)
    visible = np.asarray(kpos)[None, :] <= np.asarray(qpos)[:, None]
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1)
    live = np.isfinite(m)
    if np.any(live):
        sl = s[live]
        ml = m[live]
        lse_e = ml + np.log(np.exp(sl - ml[:, None]).sum(axis=1))
        w = np.exp(sl - lse_e[:, None])                         # softmax weights
        o[live] = w @ k[:, :D_LATENT]
        lse[live] = lse_e if base == "e" else lse_e / LN2
    return o, lse


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray, base: str = "e") -> Tuple[np.ndarray, np.ndarray]:
    """Exact merge of per-shard partials ([SG-FLOW]).

    o_parts: (c, R, 512), lse_parts: (c, R).  In base b (e or 2):
    lse = log_b sum_r b**lse_r and o = sum_r b**(lse_r - lse) * o_r.
    The maximum is taken out of the sum so the powers cannot overflow; an
    all -inf row gives lse = -inf and o = 0.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    pw = np.exp if base == "e" else np.exp2
    lg = np.log if base == "e" else np.log2
    m = lse_parts.max(axis=0)
    live = np.isfinite(m)
    lse = np.full(m.shape, -np.inf)
    o = np.zeros(o_parts.shape[1:], dtype=np.float64)
    if np.any(live):
        ml = m[live]
        lse[live] = ml + lg(pw(lse_parts[:, live] - ml[None, :]).sum(axis=0))
        w = pw(lse_parts[:, live] - lse[live][None, :])          # (c, R_live)
        o[live] = (w[:, :, None] * o_parts[:, live, :]).sum(axis=0)
    return o, lse


def query_positions(L: int, Tq: int, H: int) -> np.ndarray:
    """Global position of each query row (row = t*H + h): draft token t sits at L - Tq + t."""
    return np.repeat(np.arange(L - Tq, L, dtype=np.int64), H)


# ---------------------------------------------------------------------------
# Striped decode of one request, and the unstriped brute force
# ---------------------------------------------------------------------------
def decode_request_striped(q_b: np.ndarray, pools: ShardPools, rmap: RequestTokenMap, b: int,
                           L: int, sm_scale: float, base: str,
                           shards: Optional[Sequence[int]] = None, I: int = 1):
    """Per-shard partials and their merge for request b.

    q_b: (Tq, H, 576) float64.  For each rank r, attention runs over the
    tokens rank r owns (read back from its pool through the shared map) with
    global positions for the causal test; then the partials are merged.
    Returns (o_parts (c, R, 512), lse_parts (c, R), o (R, 512), lse (R,)).
    """
    Tq, H, _ = q_b.shape
    R = Tq * H
    qrows = q_b.reshape(R, D_K)
    qpos = query_positions(L, Tq, H)
    c = pools.c
    shards = list(range(c)) if shards is None else list(shards)
    o_parts = np.zeros((len(shards), R, D_LATENT))
    lse_parts = np.full((len(shards), R), -np.inf)
    for i, r in enumerate(shards):
        pos, slots = shard_view(rmap, b, L, r, I)
        rows, scs = pools.read(r, slots)
        k = dequant(rows, scs, pools.kv_dtype)
        o_parts[i], lse_parts[i] = attend(qrows, k, pos, qpos, sm_scale, base)
    o, lse = lse_merge(o_parts, lse_parts, base)
    return o_parts, lse_parts, o, lse


def decode_request_dense(q_b: np.ndarray, k_dense: np.ndarray, L: int, sm_scale: float, base: str):
    """Brute force over the unstriped keys of one request (positions 0..L-1)."""
    Tq, H, _ = q_b.shape
    return attend(q_b.reshape(Tq * H, D_K), k_dense[:L], np.arange(L), query_positions(L, Tq, H),
                  sm_scale, base)


# ---------------------------------------------------------------------------
# Interleaved striping, relayout, un-stripe gather, HiCache index filter,
# per-token E4M3 quantisation
# ---------------------------------------------------------------------------
def owner_i(v, c: int, I: int = 1):
    """Rank that stores virtual slot v when tokens go to ranks in runs of I ([VW-ILV]).

    I = 1 is owner(v) = v mod c ([SG-VKV]).  Runs of I consecutive slots share a
    rank and the runs go round-robin over the c ranks.
    """
    return (np.asarray(v) // I) % c


def physical_i(v, c: int, I: int = 1):
    """Compacted slot of virtual slot v in its owner's pool with runs of I.

    Each round of I*c slots gives every rank I consecutive local slots, so the
    local slot is (round) * I + (offset inside the run); I = 1 is floor(v / c).
    """
    v = np.asarray(v)
    return (v // (I * c)) * I + v % I


def striped_slots(vpt_row: np.ndarray, positions, c: int, P: int, I: int = 1):
    """(owner, physical slot) of global positions of one request, from its virtual
    page table row (virtual page = P*c positions; I must divide P so that a virtual
    page is whole rounds and its rank-local part is one physical page)."""
    if P % I:
        raise ValueError("the interleave size must divide the physical page size")
    p = np.asarray(positions, dtype=np.int64)
    vp = P * c
    v = np.asarray(vpt_row, dtype=np.int64)[p // vp] * vp + p % vp
    return owner_i(v, c, I), physical_i(v, c, I)


def shard_positions(L: int, r: int, c: int, I: int = 1) -> np.ndarray:
    """Global positions < L that rank r owns, in order (shard-local token j is the
    j-th of them).  I = 1 gives r, r + c, r + 2c, ..."""
    p = np.arange(L, dtype=np.int64)
    return p[(p // I) % c == r]


def dense_slots(dense_pt_row: np.ndarray, positions, P: int) -> np.ndarray:
    """Slot of each position in a DCP-1 (unstriped) paged cache: page p // P, offset p % P."""
    p = np.asarray(positions, dtype=np.int64)
    return np.asarray(dense_pt_row, dtype=np.int64)[p // P] * P + p % P


def relayout_dense_to_striped(dense_rows: np.ndarray, dense_scales: Optional[np.ndarray],
                              dense_pt: np.ndarray, lens: Sequence[int], vpt: np.ndarray,
                              pools: List[np.ndarray], scale_pools: Optional[List[np.ndarray]],
                              c: int, P: int, I: int = 1) -> None:
    """DCP-1 prefill cache -> striped decode pools, token by token ([SG-PD]).

    For request b and every position p < lens[b] (the exact token count: rows past
    it in a partial final dense page are not copied), the stored row at the dense
    slot of p is copied bit for bit to pools[owner(p)][physical(p)]; per-token
    scales travel with their rows.  pools / scale_pools are updated in place.
    """
    for b, L in enumerate(lens):
        if L <= 0:
            continue
        p = np.arange(L, dtype=np.int64)
        src = dense_slots(dense_pt[b], p, P)
        own, dst = striped_slots(vpt[b], p, c, P, I)
        for r in range(c):
            sel = own == r
            pools[r][dst[sel]] = dense_rows[src[sel]]
            if scale_pools is not None:
                scale_pools[r][dst[sel]] = dense_scales[src[sel]]


def gather_unstriped(pools: List[np.ndarray], scale_pools: Optional[List[np.ndarray]],
                     vpt: np.ndarray, lens: Sequence[int], out: np.ndarray,
                     out_scales: Optional[np.ndarray], c: int, P: int, I: int = 1) -> None:
    """Striped pools -> one contiguous full-context copy per request, in token order
    ([SG-EXT], [GLM-AG]): out[b, p] = pools[owner(p)][physical(p)] for p < lens[b];
    rows at p >= lens[b] are left as they are."""
    for b, L in enumerate(lens):
        if L <= 0:
            continue
        p = np.arange(L, dtype=np.int64)
        own, src = striped_slots(vpt[b], p, c, P, I)
        for r in range(c):
            sel = own == r
            out[b, p[sel]] = pools[r][src[sel]]
            if out_scales is not None:
                out_scales[b, p[sel]] = scale_pools[r][src[sel]]


def hicache_filter(idx, c: int, rank: int, I: int = 1) -> np.ndarray:
    """Widened-page slot indices -> this rank's local slots ([SG-HIC]).

    Keeps the indices the rank owns, in their order, and maps each to its local
    slot (floor(i / c) for I = 1).
    """
    idx = np.asarray(idx, dtype=np.int64)
    keep = owner_i(idx, c, I) == rank
    return physical_i(idx[keep], c, I)


def _e4m3_magnitudes() -> np.ndarray:
    """Every finite non-negative E4M3FN value, by code 0x00..0x7E (increasing)."""
    return e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))


def round_to_e4m3(y: np.ndarray) -> np.ndarray:
    """Codes of the E4M3FN values nearest to y (|y| <= 448), ties to the even code.

    Written from the definition: among the 127 finite magnitudes pick the closest;
    at an exact midpoint take the code whose lowest mantissa bit is 0.  The sign
    bit is y's, so a negative value that rounds to zero is stored as -0 (0x80), as
    IEEE rounding gives it.
    """
    y = np.asarray(y, dtype=np.float64)
    mags = _e4m3_magnitudes()
    a = np.abs(y)
    if np.any(a > 448.0):
        raise ValueError("value outside the E4M3 range")
    hi = np.clip(np.searchsorted(mags, a, side="left"), 0, 126)   # first magnitude >= a
    lo = np.clip(hi - 1, 0, 126)
    dlo, dhi = a - mags[lo], mags[hi] - a
    pick = np.where(dhi < dlo, hi, lo)
    tie = (dhi == dlo) & (hi != lo)
    pick = np.where(tie, np.where(hi % 2 == 0, hi, lo), pick)
    sign = np.where(np.signbit(y), 0x80, 0x00)
    return (pick | sign).astype(np.uint8)


def quantize_e4m3_rows(rows_bf16_bits: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-token E4M3 quantisation of new KV rows (576 bf16 values each).

    In float32, as both sides compute it: amax = max |x| over the row,
    scale = amax / 448, codes = E4M3(clamp(x / scale, -448, 448)) rounded to
    nearest-even; a row of zeros gets scale 0 and all-zero codes.  (The pages fix
    an FP8 KV cache with a per-token scale; this recipe is the reading used.)
    """
    x = (np.asarray(rows_bf16_bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    amax = np.abs(x).max(axis=1).astype(np.float32)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    codes = np.zeros(x.shape, dtype=np.uint8)
    live = scale > 0
    if np.any(live):
        y = (x[live] / scale[live, None]).astype(np.float32)
        y = np.clip(y, np.float32(-448.0), np.float32(448.0))
        codes[live] = round_to_e4m3(y)
    return codes, scale
