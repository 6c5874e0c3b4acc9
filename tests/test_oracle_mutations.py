"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each one."""
import numpy as np
import pytest

import oracle as O
import oracle.dcp_oracle as OD
import test_oracle_pins as pins


def _plant(monkeypatch, name, fn):
    """Replace an oracle function both in its module and in the package namespace."""
    monkeypatch.setattr(OD, name, fn)
    monkeypatch.setattr(O, name, fn)


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def test_wrong_owner_formula_is_caught(monkeypatch):
    _plant(monkeypatch, "owner", lambda v, c: (v // c) % c)
    assert _fails(pins.test_sglang_worked_example_c4_tokens0_7, 1, None)


def test_wrong_physical_formula_is_caught(monkeypatch):
    _plant(monkeypatch, "physical", lambda v, c: v % c + (v // c) * 0)
    assert _fails(pins.test_widened_page_maps_to_one_physical_page_per_rank, 4, 16)


def test_dropped_rope_term_is_caught(monkeypatch):
    real = OD.attend

    def no_rope(q, k, kpos, qpos, sm_scale, base="e"):
        k2 = k.copy()
        k2[:, O.D_LATENT:] = 0
        o, lse = real(q, k2, kpos, qpos, sm_scale, base)
        return o, lse
    _plant(monkeypatch, "attend", no_rope)
    assert _fails(pins.test_attend_equals_library_sdpa, 64)


def test_causal_off_by_one_is_caught(monkeypatch):
    _plant(monkeypatch, "query_positions",
                        lambda L, Tq, H: np.repeat(np.arange(L - Tq, L) - 1, H))
    assert _fails(pins.test_attend_causal_equals_library_lower_right_mask, 4, 37)


def test_unnormalised_merge_is_caught(monkeypatch):
    real_merge = OD.lse_merge

    def bad_merge(o_parts, lse_parts, base="e"):
        o, lse = real_merge(o_parts, lse_parts, base)
        return o_parts.sum(axis=0) / max(len(o_parts), 1), lse   # plain average, no LSE weights
    _plant(monkeypatch, "lse_merge", bad_merge)
    assert _fails(pins.test_striped_merge_equals_brute_force, 4, 257, 1, "e")


def test_wrong_lse_base_is_caught(monkeypatch):
    real = OD.attend

    def base_e_always(q, k, kpos, qpos, sm_scale, base="e"):
        return real(q, k, kpos, qpos, sm_scale, "e")
    _plant(monkeypatch, "attend", base_e_always)
    assert _fails(pins.test_lse_closed_form_equal_scores, 8)


def test_e4m3_without_subnormals_is_caught(monkeypatch):
    real = OD.e4m3_to_f64

    def no_sub(codes):
        v = real(codes)
        u = np.asarray(codes, dtype=np.uint8)
        return np.where(((u >> 3) & 0xF) == 0, 0.0, v)
    _plant(monkeypatch, "e4m3_to_f64", no_sub)
    assert _fails(pins.test_e4m3_decode_matches_torch_for_all_codes)


# ---- relayout, gather, interleave, HiCache filter, E4M3 quantisation ----
import test_oracle_next as nxt  # noqa: E402


def test_interleave_ignored_in_physical_slot_is_caught(monkeypatch):
    _plant(monkeypatch, "physical_i", lambda v, c, I=1: np.asarray(v) // c)
    assert _fails(nxt.test_interleaved_widened_page_is_one_physical_page_per_rank, 2, 64, 16)


def test_relayout_of_whole_pages_is_caught(monkeypatch):
    real = OD.relayout_dense_to_striped

    def whole_pages(dense_rows, dense_scales, dense_pt, lens, vpt, pools, scale_pools, c, P, I=1):
        lens = [-(-L // P) * P for L in lens]                # stale rows of the last page leak
        return real(dense_rows, dense_scales, dense_pt, lens, vpt, pools, scale_pools, c, P, I)
    _plant(monkeypatch, "relayout_dense_to_striped", whole_pages)
    assert _fails(nxt.test_relayout_copies_the_exact_token_count, 17)


def test_gather_in_shard_order_is_caught(monkeypatch):
    def shard_major(pools, scale_pools, vpt, lens, out, out_scales, c, P, I=1):
        for b, L in enumerate(lens):
            own, src = OD.striped_slots(vpt[b], np.arange(L), c, P, I)
            order = np.argsort(own, kind="stable")               # shard 0's tokens first
            for k, i in enumerate(order):
                out[b, k] = pools[own[i]][src[i]]
    _plant(monkeypatch, "gather_unstriped", shard_major)
    assert _fails(nxt.test_gather_restores_token_order_of_the_worked_example)


def test_hicache_filter_with_remainder_instead_of_floor_is_caught(monkeypatch):
    def rem(idx, c, rank, I=1):
        idx = np.asarray(idx, dtype=np.int64)
        return idx[OD.owner_i(idx, c, I) == rank] % c
    _plant(monkeypatch, "hicache_filter", rem)
    assert _fails(nxt.test_hicache_filter_keeps_owned_slots_and_maps_to_floor_i_over_c)


def test_e4m3_ties_away_from_zero_is_caught(monkeypatch):
    def away(y):
        y = np.asarray(y, dtype=np.float64)
        mags = OD._e4m3_magnitudes()
        a = np.abs(y)
        hi = np.clip(np.searchsorted(mags, a, side="left"), 0, 126)
        lo = np.clip(hi - 1, 0, 126)
        pick = np.where(mags[hi] - a <= a - mags[lo], hi, lo)   # ties go up
        return (pick | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)
    _plant(monkeypatch, "round_to_e4m3", away)
    assert _fails(nxt.test_round_to_e4m3_matches_exhaustive_search_including_ties)
