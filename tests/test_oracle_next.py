"""Pins for the oracle's relayout, un-stripe gather, interleaved striping, HiCache
index filter and per-token E4M3 quantisation (CPU only).

Each function is checked against something other than itself: the pages' worked
striping example (tests/golden), the already-pinned compacting write and position
map, exhaustive search, a library cast, or invariants the definitions imply.
"""
import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden_lines


# --------------------------------------------------------------------- helpers
def _rows(n, seed, dtype=np.uint16):
    g = np.random.default_rng(seed)
    return g.integers(0, np.iinfo(dtype).max, size=(n, O.D_K), dtype=dtype)


def _pools(c, rows_per_pool, fill, dtype=np.uint16):
    return [np.full((rows_per_pool, O.D_K), fill, dtype=dtype) for _ in range(c)]


def _worked_example():
    lines = golden_lines("sglang_dcp4_tokens0_7.txt")
    c = int(lines[0].split()[1])
    n = int(lines[1].split()[1])
    held = {}
    for ln in lines[2:]:
        head, toks = ln.split(":")
        held[int(head.split()[1])] = [int(t) for t in toks.split()]
    return c, n, held


# ------------------------------------------------------- interleaved striping
@pytest.mark.parametrize("c", [1, 2, 3, 4, 8])
def test_interleave_one_is_the_plain_striping(c):
    v = np.arange(0, 5000, 7)
    assert np.array_equal(O.owner_i(v, c, 1), O.owner(v, c))
    assert np.array_equal(O.physical_i(v, c, 1), O.physical(v, c))


@pytest.mark.parametrize("c,I,L", [(2, 16, 1000), (4, 8, 777), (8, 16, 12345), (3, 4, 50), (8, 1, 99)])
def test_interleaved_shards_balance_within_one_run(c, I, L):
    counts = [len(O.shard_positions(L, r, c, I)) for r in range(c)]
    assert sum(counts) == L
    assert max(counts) - min(counts) <= I
    # a shard's tokens come in whole runs of I consecutive positions, round-robin
    for r in range(c):
        pos = O.shard_positions(L, r, c, I)
        assert np.all((pos // I) % c == r)


@pytest.mark.parametrize("c,P,I", [(4, 16, 4), (2, 64, 16), (8, 16, 16), (3, 8, 2), (4, 16, 1)])
def test_interleaved_widened_page_is_one_physical_page_per_rank(c, P, I):
    """Every widened page of P*c slots puts exactly P slots on each rank, on that rank's
    physical page with the same id, and no two slots collide."""
    for g in (0, 3, 11):
        v = g * P * c + np.arange(P * c)
        own, phys = O.owner_i(v, c, I), O.physical_i(v, c, I)
        for r in range(c):
            local = np.sort(phys[own == r])
            assert np.array_equal(local, g * P + np.arange(P))


def test_interleave_one_matches_the_pages_worked_example():
    c, n, held = _worked_example()
    for r in range(c):
        assert O.shard_positions(n, r, c, 1).tolist() == held[r]


# -------------------------------------------------------------------- relayout
def _dense_cache(L_list, P, seed, dtype=np.uint16):
    """A DCP-1 paged cache: pages shuffled, rows random, plus a row source per (b, p)."""
    g = np.random.default_rng(seed)
    pages = [(L + P - 1) // P for L in L_list]
    total = sum(pages) + 3
    ids = g.permutation(total)
    dense_pt = np.full((len(L_list), max(pages)), -1, dtype=np.int64)
    k = 0
    for b, n in enumerate(pages):
        dense_pt[b, :n] = ids[k:k + n]
        k += n
    rows = _rows(total * P, seed + 1, dtype)
    return rows, dense_pt


def test_relayout_equals_the_compacting_append_of_every_token():
    """Relayout of a dense cache = appending each of the L tokens through the shared
    map (the pinned a2/a3 oracle), for an allocator-built virtual page table."""
    c, P = 4, 16
    lens = [1000, 37, 64]
    dense, dense_pt = _dense_cache(lens, P, 5)
    alloc = O.SharedVirtualAllocator(c, 4096, P, order=np.random.default_rng(9).permutation(4096 // P))
    rmap = O.RequestTokenMap(alloc)
    for b, L in enumerate(lens):
        rmap.extend(b, L)
    vpt = rmap.page_table(range(len(lens)), max_pages=70)
    pool_rows = 4096
    pools = _pools(c, pool_rows, 0xA5A5)
    O.relayout_dense_to_striped(dense, None, dense_pt, lens, vpt, pools, None, c, P)
    ref = O.ShardPools(c, P, "bf16")
    for b, L in enumerate(lens):
        p = np.arange(L)
        O.append_tokens(ref, rmap, b, p, dense[O.dense_slots(dense_pt[b], p, P)])
    for r in range(c):
        written = sorted(ref.written[r])
        got, _ = ref.read(r, np.array(written))
        assert np.array_equal(pools[r][written], got)
        untouched = np.ones(pool_rows, bool)
        untouched[written] = False
        assert np.all(pools[r][untouched] == 0xA5A5)


def test_relayout_of_the_worked_example_puts_tokens_r_and_r_plus_c_on_rank_r():
    c, n, held = _worked_example()
    P = 2                                          # widened page of 8 = the example's 8 tokens
    dense, dense_pt = _dense_cache([n], P, 1)
    vpt = np.array([[3]])
    pools = _pools(c, 16, 0)
    O.relayout_dense_to_striped(dense, None, dense_pt, [n], vpt, pools, None, c, P)
    for r in range(c):
        want = dense[O.dense_slots(dense_pt[0], np.array(held[r]), P)]
        assert np.array_equal(pools[r][3 * P:3 * P + len(held[r])], want)


@pytest.mark.parametrize("L", [1, 15, 17, 31, 33])
def test_relayout_copies_the_exact_token_count(L):
    """Rows of a partial final dense page past L are not copied (no stale rows leak)."""
    c, P = 2, 16
    dense, dense_pt = _dense_cache([L], P, 7)
    vpt = np.array([[0, 1]])
    pools = _pools(c, 64, 0xA5A5)
    O.relayout_dense_to_striped(dense, None, dense_pt, [L], vpt, pools, None, c, P)
    written = sum(int(np.sum(np.any(pools[r] != 0xA5A5, axis=1))) for r in range(c))
    assert written == L


def test_relayout_moves_scales_with_their_rows():
    c, P = 4, 8
    lens = [50]
    dense, dense_pt = _dense_cache(lens, P, 3, np.uint8)
    dscales = np.random.default_rng(4).random(len(dense)).astype(np.float32)
    vpt = np.array([[2, 0]])
    pools = _pools(c, 32, 0, np.uint8)
    spools = [np.zeros(32, np.float32) for _ in range(c)]
    O.relayout_dense_to_striped(dense, dscales, dense_pt, lens, vpt, pools, spools, c, P)
    p = np.arange(50)
    own, dst = O.striped_slots(vpt[0], p, c, P)
    src = O.dense_slots(dense_pt[0], p, P)
    for r in range(c):
        assert np.array_equal(spools[r][dst[own == r]], dscales[src[own == r]])


# --------------------------------------------------------------------- gather
def test_gather_restores_token_order_of_the_worked_example():
    c, n, held = _worked_example()
    P = 2
    pools = _pools(c, 16, 0)
    for r in range(c):
        for j, tok in enumerate(held[r]):
            pools[r][3 * P + j] = tok + 1                   # row content = token id + 1
    out = np.zeros((1, n, O.D_K), np.uint16)
    O.gather_unstriped(pools, None, np.array([[3]]), [n], out, None, c, P)
    assert np.array_equal(out[0, :, 0], np.arange(n) + 1)


@pytest.mark.parametrize("c,P,I", [(1, 16, 1), (3, 16, 1), (8, 64, 1), (4, 16, 4), (2, 64, 16)])
def test_gather_inverts_relayout(c, P, I):
    lens = [700, 5, 130]
    dense, dense_pt = _dense_cache(lens, P, 11)
    vp = (max(lens) + P * c - 1) // (P * c)
    vpt = np.arange(len(lens) * vp).reshape(len(lens), vp)[:, ::-1].copy()
    pools = _pools(c, len(lens) * vp * P, 0)
    O.relayout_dense_to_striped(dense, None, dense_pt, lens, vpt, pools, None, c, P, I)
    out = np.full((len(lens), max(lens) + 3, O.D_K), 0x7777, np.uint16)
    O.gather_unstriped(pools, None, vpt, lens, out, None, c, P, I)
    for b, L in enumerate(lens):
        assert np.array_equal(out[b, :L], dense[O.dense_slots(dense_pt[b], np.arange(L), P)])
        assert np.all(out[b, L:] == 0x7777)


# ------------------------------------------------------------ HiCache filter
def test_hicache_filter_keeps_owned_slots_and_maps_to_floor_i_over_c():
    c = 4
    for rank in range(c):
        got = O.hicache_filter(np.arange(16), c, rank)
        assert got.tolist() == [0, 1, 2, 3]                  # i = rank + 4k -> k
        assert np.array_equal(O.hicache_filter(np.arange(16), c, rank), np.arange(rank, 16, c) // c)


@pytest.mark.parametrize("c,I", [(2, 1), (4, 1), (8, 1), (4, 4), (2, 16)])
def test_hicache_filter_partitions_the_list_and_keeps_order(c, I):
    g = np.random.default_rng(c * 10 + I)
    idx = g.permutation(4096)[:1000]
    total = 0
    for rank in range(c):
        loc = O.hicache_filter(idx, c, rank, I)
        mine = idx[O.owner_i(idx, c, I) == rank]
        total += len(loc)
        # local slot -> widened slot: run round, rank's run, offset
        back = (loc // I) * I * c + rank * I + loc % I
        assert np.array_equal(back, mine)                    # order kept, inverse exact
    assert total == len(idx)


# ------------------------------------------------------- E4M3 quantisation
def _e4m3_brute(y):
    vals = O.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    out = np.zeros(len(y), np.uint8)
    for i, t in enumerate(y):
        d = np.abs(vals - t)
        d[np.isnan(d)] = np.inf
        best = np.flatnonzero(d == d.min())
        best = [int(b) for b in best]
        if len(best) > 1:   # +0 and -0 (the sign of t decides), or an exact midpoint
            same_sign = [b for b in best if (b >= 0x80) == bool(np.signbit(t))]
            best = same_sign or best
            best = [b for b in best if b % 2 == 0] or best
        out[i] = best[0]
    return out


def test_round_to_e4m3_matches_exhaustive_search_including_ties():
    vals = O.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    g = np.random.default_rng(0)
    y = np.concatenate([mids, -mids, g.uniform(-448, 448, 300), g.uniform(-1e-2, 1e-2, 100),
                        [0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 3 * 2.0 ** -10, -2.0 ** -11]])
    assert np.array_equal(O.round_to_e4m3(y), _e4m3_brute(y))


def test_round_to_e4m3_agrees_with_the_library_cast():
    g = np.random.default_rng(1)
    y = np.concatenate([g.standard_normal(4000) * 50, g.standard_normal(1000) * 0.01]).astype(np.float32)
    y = np.clip(y, -448, 448)
    lib = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.round_to_e4m3(y), lib)


def test_quantize_rows_scale_codes_and_error_bound():
    g = np.random.default_rng(2)
    x = (g.standard_normal((64, O.D_K)) * np.exp(g.uniform(-5, 5, (64, 1)))).astype(np.float32)
    x[3] = 0.0                                               # an all-zero row
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)       # bf16 by truncation: any bf16 rows do
    xb = (bits.astype(np.uint32) << 16).view(np.float32)
    codes, scale = O.quantize_e4m3_rows(bits)
    assert scale[3] == 0 and np.all(codes[3] == 0)
    live = np.arange(64) != 3
    amax = np.abs(xb[live]).max(axis=1)
    assert np.array_equal(scale[live], (amax / np.float32(448)).astype(np.float32))
    # the element of largest magnitude lands on +-448 (code 0x7E / 0xFE)
    arg = np.abs(xb[live]).argmax(axis=1)
    top = codes[live][np.arange(live.sum()), arg]
    assert np.all((top & 0x7F) == 0x7E)
    # dequantised values are within half an E4M3 step of x (relative 2^-4 for normals)
    deq = O.e4m3_to_f64(codes[live]) * scale[live, None].astype(np.float64)
    err = np.abs(deq - xb[live])
    bound = np.maximum(np.abs(xb[live]) * 2.0 ** -4, scale[live, None] * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(err <= bound)
