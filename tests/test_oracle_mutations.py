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
