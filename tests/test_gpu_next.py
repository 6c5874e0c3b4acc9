"""GPU parity for the relayout, un-stripe gather, E4M3 quantising append and HiCache
index filter, through the C ABI, against the oracle (bit-exact: all four move or
encode bytes)."""
import numpy as np
import pytest
import torch

import dcp_workloads as W
import oracle as O
from decode_context_mla_gb300 import binding as B
from oracle_ref import bits

pytestmark = pytest.mark.gpu
needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
SENT = 0xA5


def _sent(dtype):
    """The sentinel byte pattern as an element of a host mirror of that dtype."""
    return 0xA5A5 if dtype == np.uint16 else SENT


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from decode_context_mla_gb300.build import build
    build()


def _case(B_, c, P, I, lens, kv, seed):
    """Dense DCP-1 cache on the GPU (shuffled pages), striped pools (sentinel) and a
    shuffled virtual page table; returns host copies for the oracle too."""
    g = np.random.default_rng(seed)
    dpages = [(L + P - 1) // P for L in lens]
    dtotal = sum(dpages) + 2
    dperm = g.permutation(dtotal)
    dpt = np.full((B_, max(dpages)), -1, np.int32)
    k = 0
    for b, n in enumerate(dpages):
        dpt[b, :n] = dperm[k:k + n]
        k += n
    vpages = [(L + P * c - 1) // (P * c) for L in lens]
    vtotal = sum(vpages) + 1
    vperm = g.permutation(vtotal)
    vpt = np.full((B_, max(vpages)), -1, np.int32)
    k = 0
    for b, n in enumerate(vpages):
        vpt[b, :n] = vperm[k:k + n]
        k += n
    dt = torch.bfloat16 if kv == "bf16" else torch.uint8
    dense = torch.randint(0, 255, (dtotal * P, O.D_K * (2 if kv == "bf16" else 1)), dtype=torch.uint8,
                          generator=torch.Generator().manual_seed(seed)).view(dt)
    dscales = (torch.rand(dtotal * P, generator=torch.Generator().manual_seed(seed + 1))
               if kv == "e4m3" else None)
    pools = [torch.full((vtotal * P, O.D_K), 0, dtype=dt, device="cuda") for _ in range(c)]
    for p in pools:
        p.view(torch.uint8).fill_(SENT)
    spools = [torch.full((vtotal * P,), -1.0, device="cuda") for _ in range(c)] if kv == "e4m3" else None
    return dict(dense=dense, dscales=dscales, dpt=dpt, vpt=vpt, pools=pools, spools=spools,
                lens=np.array(lens, np.int32), kv=B.KV_BF16 if kv == "bf16" else B.KV_E4M3,
                rows=vtotal * P)


def _np_rows(t):
    return t.cpu().view(torch.uint8).numpy() if t.dtype != torch.bfloat16 else bits(t.cpu())


CASES = [  # B, c, P, I, lens, kv
    (3, 4, 16, 1, [1000, 37, 64], "bf16"),
    (2, 8, 64, 16, [5000, 129], "bf16"),
    (4, 3, 16, 4, [333, 1, 16, 17], "bf16"),
    (2, 1, 16, 1, [700, 31], "bf16"),
    (3, 8, 64, 1, [3000, 65, 511], "e4m3"),
    (2, 2, 16, 8, [999, 48], "e4m3"),
]


@needs_cuda
@pytest.mark.parametrize("B_,c,P,I,lens,kv", CASES)
def test_relayout_then_gather_bit_exact(B_, c, P, I, lens, kv):
    x = _case(B_, c, P, I, lens, kv, seed=B_ * 7 + c + P + I)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dense_d = x["dense"].cuda()
    dsc_d = None if x["dscales"] is None else x["dscales"].cuda()
    B.dcpmla_relayout_dense_to_striped(dense_d, dsc_d, torch.from_numpy(x["dpt"]).cuda(), x["pools"],
                                       x["spools"], x["kv"], torch.from_numpy(x["vpt"]).cuda(),
                                       torch.from_numpy(x["lens"]).cuda(), P, c, err, interleave=I)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # oracle on host copies of the same bytes
    dense_h = _np_rows(x["dense"])
    dsc_h = None if x["dscales"] is None else x["dscales"].numpy()
    pools_h = [np.full_like(_np_rows(p), _sent(_np_rows(p).dtype)) for p in x["pools"]]
    spools_h = None if x["spools"] is None else [np.full(x["rows"], -1.0, np.float32) for _ in range(c)]
    O.relayout_dense_to_striped(dense_h, dsc_h, x["dpt"], x["lens"].tolist(), x["vpt"], pools_h, spools_h,
                                c, P, I)
    for r in range(c):
        assert np.array_equal(_np_rows(x["pools"][r]), pools_h[r]), f"pool {r}"
        if spools_h is not None:
            assert np.array_equal(x["spools"][r].cpu().numpy().view(np.uint32), spools_h[r].view(np.uint32))
    # gather back into token order (rows past each length keep the sentinel)
    cap = max(lens) + 5
    dt = x["pools"][0].dtype
    out = torch.empty((B_, cap, O.D_K), dtype=dt, device="cuda")
    out.view(torch.uint8).fill_(SENT)
    osc = torch.full((B_, cap), -2.0, device="cuda") if kv == "e4m3" else None
    B.dcpmla_gather_unstriped(x["pools"], x["spools"], x["kv"], torch.from_numpy(x["vpt"]).cuda(),
                              torch.from_numpy(x["lens"]).cuda(), P, c, out, osc, err, interleave=I)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    out_h = np.full((B_, cap) + pools_h[0].shape[1:], _sent(pools_h[0].dtype), pools_h[0].dtype)
    osc_h = None if osc is None else np.full((B_, cap), -2.0, np.float32)
    O.gather_unstriped(pools_h, spools_h, x["vpt"], x["lens"].tolist(), out_h, osc_h, c, P, I)
    got = out.cpu().view(torch.uint8).numpy() if dt != torch.bfloat16 else bits(out.cpu())
    assert np.array_equal(got, out_h)
    if osc is not None:
        assert np.array_equal(osc.cpu().numpy().view(np.uint32), osc_h.view(np.uint32))
    for b, L in enumerate(lens):          # the round trip restores the dense rows
        assert np.array_equal(got[b, :L], dense_h[O.dense_slots(x["dpt"][b], np.arange(L), P)])


@needs_cuda
def test_relayout_flags_bad_pages_and_lengths():
    x = _case(2, 4, 16, 1, [200, 100], "bf16", seed=3)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    vpt = torch.from_numpy(x["vpt"]).cuda()
    vpt[0, 0] = 10 ** 6
    lens = torch.tensor([200, 10 ** 7], dtype=torch.int32, device="cuda")
    B.dcpmla_relayout_dense_to_striped(x["dense"].cuda(), None, torch.from_numpy(x["dpt"]).cuda(), x["pools"],
                                       None, x["kv"], vpt, lens, 16, 4, err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & B.DERR_PAGE and e & B.DERR_LENGTH


@needs_cuda
def test_e4m3_quantising_append_many_rows_bit_exact():
    """16384 rows over a wide range of magnitudes: every code and scale matches the oracle's
    IEEE division (the kernel divides by Markstein's correction of a reciprocal product)."""
    c, P, n = 2, 64, 16384
    g = torch.Generator().manual_seed(9)
    x = torch.randn(n, O.D_K, generator=g) * torch.exp(torch.randn(n, 1, generator=g) * 8)
    rows = x.to(torch.bfloat16)
    pages = n // (P * c) * 2
    pools = [torch.full((pages * P, O.D_K), SENT, dtype=torch.uint8, device="cuda") for _ in range(c)]
    spools = [torch.full((pages * P,), -1.0, device="cuda") for _ in range(c)]
    pt = torch.arange(pages, dtype=torch.int32).view(1, -1)
    pos = torch.arange(n, dtype=torch.int64)
    req = torch.zeros(n, dtype=torch.int32)
    owner = torch.empty(n, dtype=torch.int32, device="cuda")
    phys = torch.empty(n, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dcpmla_slot_map(pt.cuda(), pages, c, P, req.cuda(), pos.cuda(), None, owner, phys, err)
    rows_d = rows.cuda()
    B.dcpmla_kv_append_e4m3(pools, spools, owner, phys, rows_d[:, :512], rows_d[:, 512:], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    codes, scales = O.quantize_e4m3_rows(bits(rows))
    own, ph = O.striped_slots(pt.numpy()[0], pos.numpy(), c, P, 1)
    for r in range(c):
        sel = own == r
        assert np.array_equal(pools[r].cpu().numpy()[ph[sel]], codes[sel])
        assert np.array_equal(spools[r].cpu().numpy()[ph[sel]].view(np.uint32), scales[sel].view(np.uint32))


@needs_cuda
@pytest.mark.parametrize("I", [1, 4])
def test_e4m3_quantising_append_bit_exact(I):
    c, P, n = 4, 16, 333
    g = torch.Generator().manual_seed(5)
    x = torch.randn(n, O.D_K, generator=g) * torch.exp(torch.randn(n, 1, generator=g) * 3)
    x[7] = 0.0                                             # an all-zero row
    x[8] = -0.0
    x[9, :] = 1e-30                                        # tiny values
    x[10, 5] = -3.0e4
    # rows whose quotients land exactly on E4M3 rounding midpoints (scale = 1 and 2): the
    # kernel's fast reciprocal path must hand these to the correctly rounded division
    mids = torch.tensor([1.0625, -1.1875, 2.125, 0.28125, -0.0068359375, 13.0, 104.0, 432.0])
    x[11, :] = mids.repeat(O.D_K // len(mids))
    x[11, 0] = 448.0
    x[12, :] = 2.0 * mids.repeat(O.D_K // len(mids))
    x[12, 1] = -896.0
    x[13, :] = 1e-37                                       # a subnormal scale (no finite reciprocal)
    x[13, 3] = -2e-37
    x[14, :] = 1e-40                                       # bf16 subnormals
    rows = x.to(torch.bfloat16)
    pages = 40
    pools = [torch.full((pages * P, O.D_K), SENT, dtype=torch.uint8, device="cuda") for _ in range(c)]
    spools = [torch.full((pages * P,), -1.0, device="cuda") for _ in range(c)]
    pt = torch.arange(pages, dtype=torch.int32).roll(3).view(1, -1)
    pos = torch.randperm(pages * P * c // 2, generator=g)[:n].to(torch.int64)
    req = torch.zeros(n, dtype=torch.int32)
    owner = torch.empty(n, dtype=torch.int32, device="cuda")
    phys = torch.empty(n, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dcpmla_slot_map(pt.cuda(), pages, c, P, req.cuda(), pos.cuda(), None, owner, phys, err, interleave=I)
    rows_d = rows.cuda()
    B.dcpmla_kv_append_e4m3(pools, spools, owner, phys, rows_d[:, :512], rows_d[:, 512:], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    codes, scales = O.quantize_e4m3_rows(bits(rows))
    alloc_pt = pt.numpy()
    own, ph = O.striped_slots(alloc_pt[0], pos.numpy(), c, P, I)
    for r in range(c):
        sel = own == r
        assert np.array_equal(pools[r].cpu().numpy()[ph[sel]], codes[sel])
        assert np.array_equal(spools[r].cpu().numpy()[ph[sel]].view(np.uint32), scales[sel].view(np.uint32))
        untouched = np.ones(pages * P, bool)
        untouched[ph[sel]] = False
        assert np.all(pools[r].cpu().numpy()[untouched] == SENT)


@needs_cuda
@pytest.mark.parametrize("n,c,I,rank", [(1, 4, 1, 0), (1000, 4, 1, 2), (100003, 8, 1, 7), (50000, 2, 16, 1),
                                        (4096, 3, 4, 0), (300000, 8, 2, 5)])
def test_hicache_filter_matches_oracle(n, c, I, rank):
    g = torch.Generator().manual_seed(n + c)
    hi = 1 << (40 if n % 2 else 31)                      # 64-bit and 32-bit index paths
    idx = torch.randint(0, hi, (n,), generator=g, dtype=torch.int64)
    ws = torch.empty(max(B.dcpmla_hicache_filter_workspace_size(n), 16), dtype=torch.uint8, device="cuda")
    out = torch.full((n,), -7, dtype=torch.int64, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dcpmla_hicache_filter(idx.cuda(), c, rank, out, cnt, ws, err, interleave=I)
    torch.cuda.synchronize()
    want = O.hicache_filter(idx.numpy(), c, rank, I)
    k = int(cnt.item())
    assert k == len(want) and int(err.item()) == 0
    assert np.array_equal(out.cpu().numpy()[:k], want)
    assert np.all(out.cpu().numpy()[k:] == -7)


@needs_cuda
def test_hicache_filter_flags_negative_slots():
    idx = torch.tensor([0, 5, -3, 9, 4], dtype=torch.int64, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = torch.empty(5, dtype=torch.int64, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dcpmla_hicache_filter(idx, 4, 0, out, cnt, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.DERR_POSITION
    assert int(cnt.item()) == 2 and out[:2].cpu().tolist() == [0, 1]
