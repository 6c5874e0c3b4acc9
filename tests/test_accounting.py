"""The benchmark's byte / FLOP accounting reproduces the pages' footnote arithmetic."""
import math

import bench
import dcp_workloads as W
from conftest import golden_lines


def _golden():
    g = {}
    heads = {}
    for ln in golden_lines("glm_footnote_arithmetic.txt"):
        f = ln.split()
        if f[0] == "heads":
            heads[int(f[1])] = dict(zip(f[2::2], map(float, f[3::2])))
        else:
            g.update(dict(zip(f[0::2], map(float, f[1::2]))))
    return g, heads


def test_flops_per_row_head_and_query_output_bytes():
    g, _ = _golden()
    assert bench.flops_per_key_head() == g["flop_per_row_head"]
    assert bench.q_o_bytes_per_head() == g["per_head_bytes"]        # bf16 query + bf16 output


def test_sparse_mla_intensity_8_and_64_heads():
    g, heads = _golden()
    rows_bytes = g["rows"] * g["row_bytes"]
    for h, want in heads.items():
        flops = h * g["rows"] * bench.flops_per_key_head()
        nbytes = rows_bytes + h * bench.q_o_bytes_per_head()
        assert round(flops / 1e6, 1 if h == 8 else 0) == want["mflop"]
        assert round(nbytes / 1e6, 2) == want["mbytes"]
        assert round(flops / nbytes) == want["flop_per_byte"]
    assert round(g["h200_tflops"] / g["h200_tbps"]) == g["ridge"]


def test_kv_per_token_and_million_token_footprint():
    g, _ = _golden()
    per_tok = 78 * 656 + 21 * 132 + 788
    assert per_tok == g["kv_bytes_per_token"]
    assert round(per_tok * g["tokens"] / 2**30, 1) == g["gib"]


def test_workload_accounting_matches_definitions():
    w = W.WORKLOADS["dsv3"]
    lens = w.seq_lens()
    a = bench.accounting(w, lens, max(w.pages_per_request()))
    assert a["kv_bytes"] == 32 * 32768 * 1152 == 1_207_959_552
    assert a["q_bytes"] == 32 * 128 * 576 * 2
    assert a["flops"] == 32 * 128 * 32768 * 2176
    f = W.WORKLOADS["fp8"]
    af = bench.accounting(f, f.seq_lens(), max(f.pages_per_request()))
    assert af["kv_bytes"] == 64 * 65536 * 580
    # causal verification: query t of 4 sees L - 3 + t keys
    assert af["flops"] == 64 * 128 * sum(65536 - 3 + t for t in range(4)) * 2176
    assert math.isclose(af["flops"] / 1e12, 4.673, rel_tol=1e-3)
