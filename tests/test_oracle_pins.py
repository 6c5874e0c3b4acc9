"""Pins for the fp64 oracle: values and identities the pages or the mathematics fix.

Each test ties one oracle function to something other than itself: the pages'
worked examples (golden files), library routines (torch's scaled-dot-product
attention and float8/bfloat16 conversions), closed forms, invariants the pages
state, and brute force over the unstriped keys.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden_lines


def _rank_lines(lines):
    out = {}
    for ln in lines:
        if ln.startswith("rank"):
            head, rest = ln.split(":", 1)
            r = int(head.split()[1])
            toks = rest.split("|")[0].split()
            out[r] = [int(t) for t in toks]
    return out


def _kv(lines, key):
    for ln in lines:
        parts = ln.split()
        if parts[0] == key:
            return int(parts[1])
    raise KeyError(key)


def _striped_request(c, P, L, order_seed=None, extra_pages=0):
    pages = -(-L // (P * c)) + extra_pages
    order = None
    if order_seed is not None:
        order = np.random.default_rng(order_seed).permutation(max(pages, 1)).tolist()
        pages = max(pages, 1)
    alloc = O.SharedVirtualAllocator(c, max(pages, 1) * P, P, order)
    rmap = O.RequestTokenMap(alloc)
    rmap.extend(0, L)
    return alloc, rmap


# ---------------------------------------------------------------------------
# Striping: worked examples (golden), invariants the pages state
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("P", [1, 2, 3, 16])
@pytest.mark.parametrize("order_seed", [None, 7])
def test_sglang_worked_example_c4_tokens0_7(P, order_seed):
    g = golden_lines("sglang_dcp4_tokens0_7.txt")
    c, L = _kv(g, "c"), _kv(g, "tokens")
    want = _rank_lines(g)
    _, rmap = _striped_request(c, P, L, order_seed)
    for r in range(c):
        pos, _ = O.shard_view(rmap, 0, L, r)
        assert pos.tolist() == want[r]


@pytest.mark.parametrize("P", [1, 16, 64])
def test_vllm_explainer_example_4096_tokens(P):
    g = golden_lines("vllm_explainer_dcp4_4096.txt")
    c, L = _kv(g, "c"), _kv(g, "tokens")
    want = _rank_lines(g)
    _, rmap = _striped_request(c, P, L, order_seed=3)
    for r in range(c):
        pos, _ = O.shard_view(rmap, 0, L, r)
        assert pos[:3].tolist() == want[r]
        assert len(pos) * c == L          # a 1/4 share
        assert np.all(np.diff(pos) == c)  # every 4th token


def test_vllm_effective_block_size():
    (ln,) = golden_lines("vllm_cp_effective_block.txt")
    f = ln.split()
    c, P, eff = int(f[1]), int(f[3]), int(f[5])
    assert O.effective_page_size(P, c) == eff
    alloc = O.SharedVirtualAllocator(c, 10 * P, P)
    assert alloc.virtual_page == eff
    assert alloc.P == P                    # physical size keeps its meaning
    assert alloc.virtual_capacity == 10 * P * c


@pytest.mark.parametrize("c", list(range(1, 17)))
def test_balance_within_one_token_every_prefix(c):
    """SGLang docs, Virtual KV layout: the layout stays balanced to one token as the sequence grows."""
    Lmax = 512
    for P in (1, 2, 3, 5, 8):
        _, rmap = _striped_request(c, P, Lmax, order_seed=c * 31 + P)
        p = np.arange(Lmax)
        _, own, _ = O.map_positions(rmap, 0, p)
        counts = np.zeros((Lmax + 1, c), dtype=np.int64)
        counts[1:] = np.cumsum(own[:, None] == np.arange(c)[None, :], axis=0)
        spread = counts.max(axis=1) - counts.min(axis=1)
        assert spread.max() <= 1, (c, P)
        # and the owner never needs more than ceil(L/c) slots
        Ls = np.arange(Lmax + 1)
        assert np.all(counts.max(axis=1) == -(-Ls // c))


@pytest.mark.parametrize("c,P", [(1, 4), (2, 16), (3, 5), (4, 16), (8, 64), (16, 2)])
def test_widened_page_maps_to_one_physical_page_per_rank(c, P):
    """SGLang docs, Virtual KV layout: one virtual page of P*c tokens is one physical page of P per rank."""
    L = 7 * P * c + 3
    alloc, rmap = _striped_request(c, P, L, order_seed=11, extra_pages=2)
    p = np.arange(L)
    v, own, phys = O.map_positions(rmap, 0, p)
    page_of_pos = np.asarray(rmap.pages[0])[p // (P * c)]
    assert np.all(phys // P == page_of_pos)
    # compaction: distinct slots per rank, and a full virtual page fills the physical page
    for r in range(c):
        s = phys[own == r]
        assert len(np.unique(s)) == len(s)
        full = (p // (P * c)) < (L // (P * c))
        sf = phys[(own == r) & full]
        assert sorted((sf % P).tolist()) == sorted(list(range(P)) * (L // (P * c)))


def test_allocator_exhaustion_release_and_order():
    alloc = O.SharedVirtualAllocator(2, 4 * 8, 8, order=[3, 1, 0, 2])
    assert alloc.alloc(2) == [3, 1]
    with pytest.raises(O.AllocatorExhausted):
        alloc.alloc(3)
    alloc.release([3])
    assert alloc.alloc(2) == [0, 2]
    assert alloc.alloc(1) == [3]
    with pytest.raises(ValueError):
        alloc.release([5])
    with pytest.raises(ValueError):
        O.SharedVirtualAllocator(2, 10, 4)     # capacity not a whole number of pages
    with pytest.raises(ValueError):
        O.SharedVirtualAllocator(0, 8, 4)


def test_request_map_grows_across_pages_and_releases():
    alloc = O.SharedVirtualAllocator(4, 16 * 4, 4)
    rmap = O.RequestTokenMap(alloc)
    rmap.extend(0, 15)
    rmap.extend(1, 16)
    rmap.extend(0, 2)            # crosses into a second virtual page of 16 tokens
    assert len(rmap.pages[0]) == 2 and len(rmap.pages[1]) == 1
    pt = rmap.page_table([0, 1], 3)
    assert pt.tolist() == [[0, 2, -1], [1, -1, -1]]
    with pytest.raises(IndexError):
        rmap.vslot(1, 16)
    rmap.release(0)
    assert alloc.free[-2:] == [0, 2] and 1 not in alloc.free and len(alloc.free) == 15


# ---------------------------------------------------------------------------
# Stored formats: library conversions
# ---------------------------------------------------------------------------
def test_e4m3_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.all((ours == ref) | both_nan)
    assert np.nanmax(ours) == 448.0


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    bits = bits[~np.isnan(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy())]
    ours = O.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------------------
# Attention: library routine, closed forms
# ---------------------------------------------------------------------------
def _sdpa(q, k, v, scale, Tq=None, L=None):
    """torch scaled-dot-product attention in float64; bottom-right causal when Tq is given."""
    qt = torch.from_numpy(q)[None, None]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    if Tq is None:
        out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    else:
        from torch.nn.attention.bias import causal_lower_right
        out = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=causal_lower_right(q.shape[0], k.shape[0]), scale=scale)
    return out[0, 0].numpy()


@pytest.mark.parametrize("n", [1, 7, 64, 300])
def test_attend_equals_library_sdpa(n):
    rng = np.random.default_rng(n)
    R = 5
    q = rng.standard_normal((R, O.D_K))
    k = rng.standard_normal((n, O.D_K))
    scale = 1 / math.sqrt(192)
    o, lse = O.attend(q, k, np.arange(n), np.full(R, n - 1), scale, "e")
    ref = _sdpa(q, k, k[:, :O.D_LATENT], scale)
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("Tq,L", [(4, 4), (4, 37), (2, 300)])
def test_attend_causal_equals_library_lower_right_mask(Tq, L):
    """Draft token t at global position L-Tq+t sees keys at positions <= its own."""
    rng = np.random.default_rng(L)
    q = rng.standard_normal((Tq, O.D_K))
    k = rng.standard_normal((L, O.D_K))
    scale = 0.3
    o, _ = O.attend(q, k, np.arange(L), O.query_positions(L, Tq, 1), scale, "e")
    ref = _sdpa(q, k, k[:, :O.D_LATENT], scale, Tq=Tq, L=L)
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_attend_rope_part_counts_in_scores_not_values():
    """Scores use all 576 dims; values are only the 512-d latent."""
    q = np.zeros((1, O.D_K))
    q[0, O.D_LATENT] = 1.0                       # a rope-only query
    k = np.zeros((2, O.D_K))
    k[1, O.D_LATENT] = 5.0                       # key 1 differs only in its rope part
    k[0, 0], k[1, 0] = 1.0, -1.0                 # distinguishable values
    o, lse = O.attend(q, k, np.arange(2), np.array([1]), 1.0, "e")
    w1 = math.exp(5) / (1 + math.exp(5))
    assert o.shape == (1, 512)
    assert math.isclose(o[0, 0], (1 - w1) * 1.0 + w1 * -1.0, rel_tol=1e-13)
    assert math.isclose(lse[0], math.log(1 + math.exp(5)), rel_tol=1e-13)


@pytest.mark.parametrize("n", [1, 8, 1000])
def test_lse_closed_form_equal_scores(n):
    """Zero query: all scores 0, so lse = ln n (base e) or log2 n (base 2) and o = mean of values."""
    rng = np.random.default_rng(n)
    k = rng.standard_normal((n, O.D_K))
    q = np.zeros((3, O.D_K))
    o, lse = O.attend(q, k, np.arange(n), np.full(3, n), 0.5, "e")
    assert np.allclose(lse, math.log(n), rtol=0, atol=1e-13)
    assert np.allclose(o, k[:, :512].mean(axis=0)[None], rtol=1e-12, atol=1e-13)
    _, lse2 = O.attend(q, k, np.arange(n), np.full(3, n), 0.5, "2")
    assert np.allclose(lse2, math.log2(n), rtol=0, atol=1e-13)


def test_lse_closed_form_two_keys_and_large_scores():
    q = np.zeros((1, O.D_K))
    q[0, 3] = 1.0
    for a in (-30.0, -1.0, 0.0, 2.5, 40.0, 700.0):
        k = np.zeros((2, O.D_K))
        k[1, 3] = a
        _, lse = O.attend(q, k, np.arange(2), np.array([5]), 1.0, "e")
        want = max(0.0, a) + math.log1p(math.exp(-abs(a)))
        assert math.isclose(lse[0], want, rel_tol=1e-14, abs_tol=1e-14)


def test_attend_empty_and_fully_masked_rows():
    q = np.ones((2, O.D_K))
    o, lse = O.attend(q, np.zeros((0, O.D_K)), np.zeros(0, dtype=int), np.array([0, 1]), 1.0, "2")
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    k = np.ones((3, O.D_K))
    o, lse = O.attend(q, k, np.array([4, 5, 6]), np.array([3, 4]), 1.0, "e")
    assert np.all(o[0] == 0) and np.isneginf(lse[0])        # row 0 sees nothing
    assert np.allclose(o[1], 1.0) and math.isclose(lse[1], 576.0)


# ---------------------------------------------------------------------------
# Merge: exactness against brute force, c = 1 identity, base equivalence
# ---------------------------------------------------------------------------
def _random_case(c, P, L, Tq, H, seed, kv_dtype="bf16", I=1):
    rng = np.random.default_rng(seed)
    pages = -(-L // (P * c)) + 1
    alloc = O.SharedVirtualAllocator(c, pages * P, P, rng.permutation(pages).tolist())
    rmap = O.RequestTokenMap(alloc)
    pools = O.ShardPools(c, P, kv_dtype)
    pos = rmap.extend(0, L)
    x = rng.standard_normal((L, O.D_K)).astype(np.float32)
    if kv_dtype == "bf16":
        rows = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        scales = None
        k_dense = O.bf16_to_f64(rows)
    else:
        scales = np.abs(x).max(axis=1) / 448.0
        rows = torch.from_numpy(x / scales[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        k_dense = O.e4m3_to_f64(rows) * scales.astype(np.float64)[:, None]
    O.append_tokens(pools, rmap, 0, pos, rows, scales, I=I)
    q = O.bf16_to_f64(torch.from_numpy(rng.standard_normal((Tq, H, O.D_K)).astype(np.float32))
                      .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    return q, pools, rmap, k_dense


@pytest.mark.parametrize("c", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("L,Tq", [(1, 1), (3, 1), (16, 1), (37, 1), (64, 4), (130, 4), (257, 1)])
@pytest.mark.parametrize("base", ["e", "2"])
def test_striped_merge_equals_brute_force(c, L, Tq, base):
    """SGLang docs, MLA decode dataflow: the merged shard results are the full attention result."""
    if L < Tq:
        pytest.skip("context shorter than the query block")
    P = 4
    q, pools, rmap, k_dense = _random_case(c, P, L, Tq, 3, seed=c * 1000 + L)
    _, lse_parts, o, lse = O.decode_request_striped(q, pools, rmap, 0, L, 0.125, base)
    o_ref, lse_ref = O.decode_request_dense(q, k_dense, L, 0.125, base)
    assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)
    if L < c:   # some ranks hold nothing: their lse is -inf
        assert np.all(np.isneginf(lse_parts[L:]))


@pytest.mark.parametrize("c,I,P", [(2, 16, 16), (4, 4, 8), (8, 2, 4), (3, 8, 16), (8, 16, 64)])
@pytest.mark.parametrize("L,Tq", [(1, 1), (37, 1), (130, 4), (700, 2)])
def test_interleaved_striped_merge_equals_brute_force(c, I, P, L, Tq):
    """vLLM DCP study page, interleave size: handing tokens to ranks in runs of I changes
    which rank holds a token, not the merged result (full attention, any c and I)."""
    if L < Tq:
        pytest.skip("context shorter than the query block")
    q, pools, rmap, k_dense = _random_case(c, P, L, Tq, 3, seed=c * 100 + I * 7 + L, I=I)
    _, lse_parts, o, lse = O.decode_request_striped(q, pools, rmap, 0, L, 0.125, "2", I=I)
    o_ref, lse_ref = O.decode_request_dense(q, k_dense, L, 0.125, "2")
    assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)
    # a rank's tokens are the positions owned under runs of I
    for r in range(c):
        pos, _ = O.shard_view(rmap, 0, L, r, I)
        assert np.array_equal(pos, O.shard_positions(L, r, c, I))


def test_fp8_striped_equals_brute_force_on_dequantised_values():
    q, pools, rmap, k_dense = _random_case(8, 4, 200, 4, 2, seed=5, kv_dtype="e4m3")
    _, _, o, lse = O.decode_request_striped(q, pools, rmap, 0, 200, 0.1, "2")
    o_ref, lse_ref = O.decode_request_dense(q, k_dense, 200, 0.1, "2")
    assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_dcp1_is_unchanged():
    """SGLang docs: dcp_size = 1 keeps the non-DCP behaviour; the merge of one part is the identity."""
    q, pools, rmap, k_dense = _random_case(1, 8, 100, 1, 4, seed=9)
    o_parts, lse_parts, o, lse = O.decode_request_striped(q, pools, rmap, 0, 100, 0.2, "e")
    assert np.array_equal(o, o_parts[0]) and np.array_equal(lse, lse_parts[0])
    v, own, phys = O.map_positions(rmap, 0, np.arange(100))
    assert np.all(own == 0) and np.array_equal(phys, v)    # the plain paged cache


def test_merge_base2_equals_base_e():
    rng = np.random.default_rng(1)
    o_parts = rng.standard_normal((5, 7, 512))
    lse_e = rng.standard_normal((5, 7)) * 10
    lse_e[2, 3] = -np.inf
    o_e, l_e = O.lse_merge(o_parts, lse_e, "e")
    o_2, l_2 = O.lse_merge(o_parts, lse_e / O.LN2, "2")
    assert np.allclose(o_e, o_2, rtol=1e-13, atol=1e-13)
    assert np.allclose(l_e, l_2 * O.LN2, rtol=1e-13, atol=1e-13)


def test_merge_closed_forms():
    o_parts = np.stack([np.full((1, 512), 1.0), np.full((1, 512), 3.0)])
    o, lse = O.lse_merge(o_parts, np.array([[0.0], [0.0]]), "e")      # equal weights
    assert np.allclose(o, 2.0) and math.isclose(lse[0], math.log(2))
    o, lse = O.lse_merge(o_parts, np.array([[1.0], [3.0]]), "2")       # weights 2 : 8
    assert np.allclose(o, (2 * 1 + 8 * 3) / 10) and math.isclose(lse[0], math.log2(10))
    o, lse = O.lse_merge(o_parts, np.array([[-np.inf], [5.0]]), "e")   # one empty part
    assert np.array_equal(o, o_parts[1]) and lse[0] == 5.0
    o, lse = O.lse_merge(o_parts, np.array([[-np.inf], [-np.inf]]), "e")
    assert np.all(o == 0) and np.isneginf(lse[0])
    o, lse = O.lse_merge(o_parts, np.array([[1000.0], [1000.0]]), "e")  # no overflow
    assert np.allclose(o, 2.0) and math.isclose(lse[0], 1000 + math.log(2))
