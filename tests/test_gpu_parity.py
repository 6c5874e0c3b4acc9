"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Integers (page tables, slot maps, the appended cache) must match bit for bit;
the fp32 outputs within the stated tolerance: max row-relative error 2e-3 for
bf16 KV and 1e-2 for e4m3 KV (against the oracle on the dequantised values).
"""
import math

import numpy as np
import pytest
import torch

import dcp_harness as Hn
import dcp_workloads as W
import oracle as O
from decode_context_mla_gb300 import binding as B
from oracle_ref import TOL, OracleWorkload, bits, lse_err, row_rel_err

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from decode_context_mla_gb300.build import build
    build()


# Scaled-down workloads with the structure of the five configurations, plus
# edge cases: c = 1, odd c and page size, lengths below c and at page edges.
SMALL = {
    "tiny": W.WORKLOADS["tiny"],
    "dsv3_s": W.scaled(W.WORKLOADS["dsv3"], B=3, L=2000),
    "long_s": W.scaled(W.WORKLOADS["long"], B=2, L=40000),
    "bimodal_s": W.scaled(W.WORKLOADS["bimodal"], B=12, lengths_mix=(6, 3000, 9000, 1, 40)),
    "fp8_s": W.scaled(W.WORKLOADS["fp8"], B=2, L=3000),
    "c1": W.Workload("c1", B=2, H=16, Tq=1, c=1, P=16, kv_dtype="bf16", lse_base="e", seed=11,
                     L=1500),
    "c3_p5_tq2": W.Workload("c3", B=3, H=8, Tq=2, c=3, P=5, kv_dtype="bf16", lse_base="2",
                            seed=12, L=777),
    "c16_short": W.Workload("c16", B=9, H=16, Tq=1, c=16, P=4, kv_dtype="bf16", lse_base="e",
                            seed=13, lengths_mix=(3, 64, 200, 1, 15)),
    "fp8_h16_tq4": W.Workload("f8", B=2, H=16, Tq=4, c=4, P=16, kv_dtype="e4m3", lse_base="e",
                              seed=14, L=517),
    # tensor-core path: split-KV combine, 16-token pages, two causal query tokens per tile
    "dsv3_split": W.scaled(W.WORKLOADS["dsv3"], B=1, L=40000),
    "h64_tq2_p16": W.Workload("h64", B=2, H=64, Tq=2, c=4, P=16, kv_dtype="bf16", lse_base="2",
                              seed=15, L=1500),
    "h128_c1_short": W.Workload("h128c1", B=3, H=128, Tq=1, c=1, P=64, kv_dtype="bf16",
                                lse_base="e", seed=16, lengths_mix=(1, 100, 200, 1, 70)),
    # token-major tensor-core path (<= 16 query rows): causal query pairs with odd c,
    # padding rows (R = 8), empty shards with 8-token pages, 128-token pages, and
    # (request, shard) ranges cut into multi-tile units that are merged in the kernel
    "fh_tq2_c3": W.Workload("fhq", B=3, H=8, Tq=2, c=3, P=16, kv_dtype="bf16", lse_base="2",
                            seed=17, L=1000),
    "fh_r8_p64": W.Workload("fhr", B=2, H=4, Tq=2, c=2, P=64, kv_dtype="bf16", lse_base="e",
                            seed=18, L=900),
    "fh_short_p8": W.Workload("fhs", B=6, H=16, Tq=1, c=8, P=8, kv_dtype="bf16", lse_base="e",
                              seed=19, lengths_mix=(2, 1, 7, 9, 300)),
    "fh_p128": W.Workload("fhp", B=2, H=16, Tq=1, c=2, P=128, kv_dtype="bf16", lse_base="2",
                          seed=20, L=3001),
    "fh_chunked": W.scaled(W.WORKLOADS["long"], B=2, L=300000),
    # a few tiles per CTA of the persistent grid: most (request, shard) items are cut by share
    # boundaries, many units hold one 64-token tile, 8-token pages (eight page boxes a tile)
    "fh_many_cuts": W.Workload("fhm", B=24, H=16, Tq=1, c=2, P=8, kv_dtype="bf16", lse_base="e",
                               seed=37, lengths_mix=(8, 2000, 6000, 1, 300)),
    # page sizes above the 64-token tile and between the tested ones: the token-major kernel
    # copies a page box of gcd(P, 16) rows (whole 8-token groups) for all nine chunks at once,
    # so a box never crosses a page or a tile (P = 24 and P = 40: eight boxes a tile)
    "fh_p256": W.Workload("fh256", B=2, H=16, Tq=1, c=2, P=256, kv_dtype="bf16", lse_base="e",
                          seed=23, L=2333),
    "fh_p32_tq4": W.Workload("fh32", B=3, H=4, Tq=4, c=4, P=32, kv_dtype="bf16", lse_base="2",
                             seed=24, lengths_mix=(1, 4000, 6000, 5, 200)),
    "fh_p24_c3": W.Workload("fh24", B=3, H=16, Tq=1, c=3, P=24, kv_dtype="bf16", lse_base="e",
                            seed=35, lengths_mix=(2, 500, 3000, 1, 70)),
    "fh_p40_tq2": W.Workload("fh40", B=2, H=8, Tq=2, c=2, P=40, kv_dtype="bf16", lse_base="2",
                             seed=36, L=4321),
    # interleave size I > 1 (tokens to shards in runs of I) on each decode kernel
    "ilv16_long": W.scaled(W.WORKLOADS["long"], B=2, L=40000, interleave=16),
    "ilv2_c3_tq2": W.Workload("il2", B=3, H=8, Tq=2, c=3, P=16, kv_dtype="bf16", lse_base="2",
                              seed=22, L=777, interleave=2),
    "ilv4_dsv3": W.scaled(W.WORKLOADS["dsv3"], B=2, L=3000, interleave=4),
    "ilv8_fp8": W.scaled(W.WORKLOADS["fp8"], B=1, L=2000, interleave=8),
    "ilv2_c16": W.Workload("il16", B=4, H=16, Tq=1, c=16, P=4, kv_dtype="bf16", lse_base="e",
                           seed=23, lengths_mix=(2, 100, 300, 1, 40), interleave=2),
    # 128-row tensor-core path: 8-token pages (eight page boxes per tile) with odd c, 32-token
    # pages with causal query pairs, pages longer than a tile with four row tiles per request,
    # and the E4M3 kernel with 8-token pages; every length leaves a ragged last tile
    "tc_p8_c3": W.Workload("tcp8", B=2, H=128, Tq=1, c=3, P=8, kv_dtype="bf16", lse_base="e",
                           seed=25, L=1234),
    "tc_p32_tq2": W.Workload("tcp32", B=2, H=64, Tq=2, c=2, P=32, kv_dtype="bf16", lse_base="2",
                             seed=26, L=2101),
    "tc_p256_tq4": W.Workload("tcp256", B=2, H=128, Tq=4, c=4, P=256, kv_dtype="bf16",
                              lse_base="2", seed=27, L=3001),
    "tc_e4m3_p8": W.Workload("tce8", B=2, H=128, Tq=1, c=2, P=8, kv_dtype="e4m3", lse_base="e",
                             seed=28, L=999),
    # E4M3 on the CUDA cores: more shards than the tensor-core kernels take in one launch
    # (causal four-token verify, split-KV with last-arriver merge, contexts shorter than c),
    # and page sizes the TMA kernels reject (P = 5, P = 12)
    "fma_e4m3_c16_tq4": W.Workload("fe16", B=3, H=16, Tq=4, c=16, P=4, kv_dtype="e4m3",
                                   lse_base="2", seed=29, lengths_mix=(1, 2000, 3000, 4, 15)),
    "fma_e4m3_c3_p5": W.Workload("fe3", B=4, H=8, Tq=1, c=3, P=5, kv_dtype="e4m3", lse_base="e",
                                 seed=30, lengths_mix=(2, 700, 1500, 1, 2)),
    "fma_e4m3_h128_c12": W.Workload("fe12", B=2, H=128, Tq=2, c=12, P=16, kv_dtype="e4m3",
                                    lse_base="2", seed=31, L=2500),
    "fma_e4m3_p12_tq3": W.Workload("fe12p", B=2, H=32, Tq=3, c=2, P=12, kv_dtype="e4m3",
                                   lse_base="e", seed=32, L=4100),
    # 128-row persistent grid: 96 real rows in the tile (rows past R pad it), and one request
    # whose two shard items are each cut into dozens of cluster shares
    "tc_r96_c3": W.Workload("tcr96", B=3, H=32, Tq=3, c=3, P=64, kv_dtype="bf16", lse_base="e",
                            seed=33, L=5000),
    "tc_c2_cut": W.Workload("tccut", B=1, H=128, Tq=1, c=2, P=64, kv_dtype="bf16", lse_base="2",
                            seed=34, L=60000),
    # persistent grid with items that have no tiles (contexts shorter than c: empty shards)
    # beside items cut by share boundaries
    "tc_empty_c8": W.Workload("tcempty", B=4, H=128, Tq=1, c=8, P=64, kv_dtype="bf16", lse_base="2",
                              seed=37, lengths_mix=(2, 9000, 20000, 1, 6)),
}

# cases that must run on the CUDA-core decode (asserted by test_decode_path_per_workload)
FMA_CASES = ["c16_short", "c3_p5_tq2", "fma_e4m3_c16_tq4", "fma_e4m3_c3_p5", "fma_e4m3_h128_c12",
             "fma_e4m3_p12_tq3"]

SENTINEL = 0xA5


def _compare_pools(dw, ow: OracleWorkload):
    w = dw.w
    for b in range(w.B):
        ow.load(b)
    for r in range(w.c):
        dev = dw.cache.pools[r].view(torch.uint8).cpu().numpy().reshape(dw.cache.pool_rows, -1)
        written = sorted(ow.pools.written[r])
        if written:
            rows, scs = ow.pools.read(r, np.array(written))
            want = rows.view(np.uint8).reshape(len(written), -1)
            assert np.array_equal(dev[written], want), f"shard {r} rows differ"
            if w.kv_dtype == "e4m3":
                got_s = dw.cache.scales[r].cpu().numpy()[written]
                assert np.array_equal(got_s.view(np.uint32), scs.view(np.uint32))
        untouched = np.ones(dw.cache.pool_rows, dtype=bool)
        untouched[written] = False
        assert np.all(dev[untouched] == SENTINEL), f"shard {r}: a row outside the owner set was written"


@needs_cuda
@pytest.mark.parametrize("name", list(SMALL))
def test_step_parity_small(name):
    _check_step(SMALL[name], name)


def _fewhead_sweep(n=10, seed=2024):
    """Seeded random shapes inside the token-major kernel's limits (at most 16 query rows, at
    least 16 in the batch, P a multiple of 8, at most 8 shards), mixed long and short lengths."""
    rng = np.random.default_rng(seed)
    cases = []
    for k in range(n):
        Tq = int(rng.choice([1, 2, 3, 4]))
        H = int(rng.choice([h for h in (1, 2, 4, 5, 8, 16) if h * Tq <= 16]))
        Bn = max(int(rng.integers(1, 7)), -(-16 // (H * Tq)))
        cases.append(W.Workload(f"fhsw{k}", B=Bn, H=H, Tq=Tq, c=int(rng.choice([1, 2, 3, 4, 5, 8])),
                                P=int(rng.choice([8, 16, 24, 32, 48, 64, 96, 128])), kv_dtype="bf16",
                                lse_base=str(rng.choice(["e", "2"])), seed=100 + k,
                                lengths_mix=(int(rng.integers(0, Bn + 1)), 1000, 9000, Tq, 400)))
    return cases


FEWHEAD_SWEEP = _fewhead_sweep()


@needs_cuda
@pytest.mark.parametrize("w", FEWHEAD_SWEEP, ids=[w.name for w in FEWHEAD_SWEEP])
def test_fewhead_random_shapes(w):
    """The token-major kernel on seeded random shapes: path check, then the full step parity."""
    got = B.dcpmla_decode_path(w.B, w.Tq, w.H, w.P, w.c, w.c, B.KV_BF16, max(w.pages_per_request()))
    assert got == (B.PATH_TC_FEWHEAD, 2), (w, got)
    _check_step(w, w.name)


def _check_step(w, name):
    dw = Hn.build(w, fill_byte=SENTINEL)
    dw.step.run()
    torch.cuda.synchronize()
    assert dw.cache.check_errors() == 0
    ow = OracleWorkload(w)
    # page table bit-exact
    assert np.array_equal(dw.step.page_table.cpu().numpy(), ow.page_table())
    # appended cache bit-exact (including the step's own appends)
    _compare_pools(dw, ow)
    tol = TOL[w.kv_dtype]
    o_part = dw.step.o_part.cpu().numpy()
    lse_part = dw.step.lse_part.cpu().numpy()
    o = dw.step.o.cpu().numpy()
    lse = dw.step.lse.cpu().numpy()
    for b in range(w.B):
        op, lp, o_ref, l_ref = ow.decode(b)
        R = w.Tq * w.H
        assert row_rel_err(o_part[:, b].reshape(w.c, R, 512), op) < tol, (name, b, "o_part")
        assert lse_err(lse_part[:, b].reshape(w.c, R), lp) < tol, (name, b, "lse_part")
        assert row_rel_err(o[b].reshape(R, 512), o_ref) < tol, (name, b, "o")
        assert lse_err(lse[b].reshape(R), l_ref) < tol, (name, b, "lse")


@needs_cuda
def test_dcp1_merge_is_bit_identical():
    """dcp_size = 1: the merge returns the shard's (o, lse) unchanged, in both bases."""
    for base in ("e", "2"):
        w = W.Workload("c1b", B=2, H=16, Tq=1, c=1, P=16, kv_dtype="bf16", lse_base=base,
                       seed=21, L=700)
        dw = Hn.build(w)
        dw.step.run()
        torch.cuda.synchronize()
        assert torch.equal(dw.step.o.view(-1), dw.step.o_part.view(-1))
        assert torch.equal(dw.step.lse.view(-1), dw.step.lse_part.view(-1))


@needs_cuda
@pytest.mark.parametrize("base", [B.LSE_E, B.LSE_2])
@pytest.mark.parametrize("c", [1, 2, 3, 8, 16])
def test_lse_merge_parity(base, c):
    g = torch.Generator().manual_seed(c * 7 + base)
    rows = 257
    o_part = torch.randn((c, rows, 512), generator=g, dtype=torch.float32)
    lse_part = torch.randn((c, rows), generator=g, dtype=torch.float32) * 8
    lse_part[:, 5] = -math.inf                        # an all-empty row (o = 0 by convention)
    o_part[:, 5] = 0.0
    if c > 1:
        lse_part[0, 7] = -math.inf                    # one empty shard
        lse_part[1, 9] = 80.0                         # a dominant shard
    o = torch.empty((rows, 512), device="cuda")
    lse = torch.empty(rows, device="cuda")
    B.dcpmla_lse_merge(o_part.cuda(), lse_part.cuda(), c, rows, base, o, lse)
    torch.cuda.synchronize()
    bname = "2" if base == B.LSE_2 else "e"
    o_ref, l_ref = O.lse_merge(o_part.double().numpy(), lse_part.double().numpy(), bname)
    assert row_rel_err(o.cpu().numpy(), o_ref) < 1e-5
    assert lse_err(lse.cpu().numpy(), l_ref) < 1e-6
    if c == 1:
        assert torch.equal(o.cpu(), o_part[0]) and torch.equal(lse.cpu(), lse_part[0])


@needs_cuda
def test_slot_map_bit_exact_and_error_bits():
    w = SMALL["c3_p5_tq2"]
    ow = OracleWorkload(w)
    pt = torch.from_numpy(ow.page_table()).cuda()
    lens = ow.lens
    req = torch.cat([torch.full((L,), b, dtype=torch.int32) for b, L in enumerate(lens)])
    pos = torch.cat([torch.arange(L, dtype=torch.int64) for L in lens])
    n = pos.numel()
    v = torch.empty(n, dtype=torch.int64, device="cuda")
    own = torch.empty(n, dtype=torch.int32, device="cuda")
    ph = torch.empty(n, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dcpmla_slot_map(pt, ow.alloc.num_pages, w.c, w.P, req.cuda(), pos.cuda(), v, own, ph, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    for b in range(w.B):
        sel = (req == b).numpy()
        wv, wo, wp = O.map_positions(ow.rmap, b, pos.numpy()[sel])
        assert np.array_equal(v.cpu().numpy()[sel], wv)
        assert np.array_equal(own.cpu().numpy()[sel], wo)
        assert np.array_equal(ph.cpu().numpy()[sel], wp)
    # bad inputs: request out of range, position past the table, page id out of range
    pt_bad = pt.clone()
    pt_bad[0, 0] = ow.alloc.num_pages + 5
    req_b = torch.tensor([0, 1, 7, 2], dtype=torch.int32, device="cuda")
    pos_b = torch.tensor([0, 10**6, 0, 3], dtype=torch.int64, device="cuda")
    v4 = torch.zeros(4, dtype=torch.int64, device="cuda")
    o4 = torch.zeros(4, dtype=torch.int32, device="cuda")
    p4 = torch.zeros(4, dtype=torch.int64, device="cuda")
    err.zero_()
    B.dcpmla_slot_map(pt_bad, ow.alloc.num_pages, w.c, w.P, req_b, pos_b, v4, o4, p4, err)
    torch.cuda.synchronize()
    assert err.item() == (B.DERR_PAGE | B.DERR_POSITION)
    assert o4.tolist()[:3] == [-1, -1, -1] and o4.tolist()[3] >= 0


BAD_INPUT_CASES = {
    "dsv3_s": SMALL["dsv3_s"],                                       # 128-row tiles
    "long_split": W.scaled(W.WORKLOADS["long"], B=3, L=40000),      # token-major, merged units
    "fh_tq2_c3": SMALL["fh_tq2_c3"],                                 # token-major, one unit each
}


@needs_cuda
@pytest.mark.parametrize("name", list(BAD_INPUT_CASES))
def test_decode_flags_bad_page_and_short_length_without_faulting(name):
    """A page id outside the pools and a length below Tq are flagged; their work is empty."""
    w = BAD_INPUT_CASES[name]
    dw = Hn.build(w)
    st = dw.step
    st.run()                                         # append the step's new tokens first
    torch.cuda.synchronize()
    pt_good = st.page_table.clone()
    st.page_table[1, 0] = 10**8                      # request 1 points outside the pools
    st.seq_lens[2] = 0                               # request 2 shorter than its query block
    dw.cache.err.zero_()
    B.dcpmla_decode(st.q, dw.cache.pools, None, B.KV_BF16, st.page_table, st.seq_lens, w.P, w.c, 0,
                    w.c, w.sm_scale, st.lse_base, st.o_part, st.lse_part, st.workspace, dw.cache.err)
    torch.cuda.synchronize()
    e = dw.cache.check_errors()
    assert e & B.DERR_PAGE and e & B.DERR_LENGTH
    # the bad requests' shards that needed the bad page / length are empty, request 0 is fine
    assert torch.all(torch.isneginf(st.lse_part[:, 2]))
    assert torch.all(st.o_part[:, 2] == 0)
    assert torch.all(torch.isneginf(st.lse_part[:, 1])) and torch.all(st.o_part[:, 1] == 0)
    ow = OracleWorkload(w)
    op, lp, _, _ = ow.decode(0)
    assert row_rel_err(st.o_part[:, 0].cpu().numpy().reshape(w.c, -1, 512), op) < TOL["bf16"]
    st.page_table.copy_(pt_good)


@needs_cuda
@pytest.mark.parametrize("name", ["tiny", "dsv3", "long", "bimodal", "fp8"])
def test_input_generator_is_device_independent(name):
    """The counter-based generator gives the same bits on the GPU and the CPU."""
    w = W.WORKLOADS[name]
    L = w.seq_lens()[-1]
    for (p0, p1) in ((0, 300), (max(0, L - 300), L)):
        rc, sc = W.kv_rows(w, w.B - 1, p0, p1, "cpu")
        rg, sg = W.kv_rows(w, w.B - 1, p0, p1, "cuda")
        assert np.array_equal(bits(rc), bits(rg))
        if sc is not None:
            assert torch.equal(sc, sg.cpu())
    qc = W.q_tensor(w, "cpu", requests=[0, w.B - 1])
    qg = W.q_tensor(w, "cuda", requests=[0, w.B - 1])
    assert np.array_equal(bits(qc), bits(qg))


@needs_cuda
def test_decode_path_per_workload():
    """Few-row bf16 shapes take the token-major tensor-core kernel (decode + split merge),
    128-head shapes the 128-row tensor-core kernel, 16 shards per launch the CUDA cores."""
    want = {"tiny": B.PATH_TC_FEWHEAD, "long": B.PATH_TC_FEWHEAD, "bimodal": B.PATH_TC_FEWHEAD,
            "dsv3": B.PATH_TC_ROWS, "fp8": B.PATH_TC_ROWS}
    for name, path in want.items():
        w = W.WORKLOADS[name]
        kv = B.KV_BF16 if w.kv_dtype == "bf16" else B.KV_E4M3
        got = B.dcpmla_decode_path(w.B, w.Tq, w.H, w.P, w.c, w.c, kv, max(w.pages_per_request()))
        # few-head: decode + unit merge; 128-row bf16: tile prefix, persistent decode, unit
        # merge; 128-row E4M3: one launch
        launches = {B.PATH_TC_FEWHEAD: 2, B.PATH_TC_ROWS: 3 if kv == B.KV_BF16 else 1}[path]
        assert got == (path, launches), name
    for name in FMA_CASES:
        w = SMALL[name]
        kv = B.KV_BF16 if w.kv_dtype == "bf16" else B.KV_E4M3
        got = B.dcpmla_decode_path(w.B, w.Tq, w.H, w.P, w.c, w.c, kv, max(w.pages_per_request()))
        assert got == (B.PATH_CUDA_CORE, 1), name
    # page sizes that are multiples of 8 but neither divide nor are divided by the tile stay on
    # the token-major kernel (page boxes of gcd(P, 16) rows)
    for name in ("fh_p24_c3", "fh_p40_tq2", "fh_p256", "fh_short_p8", "fh_many_cuts"):
        w = SMALL[name]
        got = B.dcpmla_decode_path(w.B, w.Tq, w.H, w.P, w.c, w.c, B.KV_BF16, max(w.pages_per_request()))
        assert got == (B.PATH_TC_FEWHEAD, 2), name



FUSED_CASES = ["tiny", "dsv3_s", "long_s", "bimodal_s", "fp8_s", "c1", "c3_p5_tq2", "c16_short",
               "fma_e4m3_c16_tq4", "fma_e4m3_c3_p5", "tc_r96_c3", "tc_c2_cut",
               "dsv3_split", "h64_tq2_p16", "fh_tq2_c3", "fh_short_p8", "fh_chunked", "ilv4_dsv3",
               "ilv2_c16", "tc_p8_c3", "tc_p256_tq4", "tc_e4m3_p8", "ilv8_fp8", "fp8_h16_tq4", "fh_p24_c3",
               "fh_many_cuts"]


@needs_cuda
@pytest.mark.parametrize("name", FUSED_CASES)
def test_fused_decode_merge_parity(name):
    """dcpmla_decode_merged: the merged (o, lse) straight from the decode, on every kernel path."""
    w = SMALL[name]
    dw = Hn.build(w, fused=True)
    dw.step.run()
    torch.cuda.synchronize()
    assert dw.cache.check_errors() == 0
    ow = OracleWorkload(w)
    tol = TOL[w.kv_dtype]
    o = dw.step.o.cpu().numpy()
    lse = dw.step.lse.cpu().numpy()
    R = w.Tq * w.H
    for b in range(w.B):
        _, _, o_ref, l_ref = ow.decode(b)
        assert row_rel_err(o[b].reshape(R, 512), o_ref) < tol, (name, b, "o")
        assert lse_err(lse[b].reshape(R), l_ref) < tol, (name, b, "lse")


@needs_cuda
@pytest.mark.parametrize("name", ["dsv3_s", "fh_tq2_c3"])
def test_fused_decode_merge_leaves_out_a_bad_request(name):
    w = BAD_INPUT_CASES[name]
    dw = Hn.build(w, fused=True)
    st = dw.step
    st.run()
    torch.cuda.synchronize()
    st.page_table[1, 0] = 10**8
    dw.cache.err.zero_()
    st.run_decode()
    torch.cuda.synchronize()
    assert dw.cache.check_errors() & B.DERR_PAGE
    assert torch.all(torch.isneginf(st.lse[1])) and torch.all(st.o[1] == 0)
    ow = OracleWorkload(w)
    _, _, o_ref, _ = ow.decode(0)
    assert row_rel_err(st.o[0].cpu().numpy().reshape(-1, 512), o_ref) < TOL["bf16"]
