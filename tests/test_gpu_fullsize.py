"""Parity at the five full workload sizes, in the launch configuration the benchmark times.

The whole step (slot map, append, decode over all c shards, merge) runs at
full size; the oracle then recomputes sampled requests one by one from the
same seeded generator (every shard's partial and the merged result; every
request of dsv3), and the sampled requests' rows in the shard pools are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import dcp_harness as Hn
import dcp_workloads as W
from oracle_ref import TOL, OracleWorkload, lse_err, row_rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from decode_context_mla_gb300.build import build
    build()


def _samples(w, lens):
    """Requests the oracle recomputes at full size.

    dsv3: all 32 (the persistent 128-row grid cuts items at its clusters' share
    boundaries, which fall inside different requests' shards).  fp8: eight requests
    spread over the batch, each covering all four 128-row tiles and the split merge of
    every shard (the oracle takes a few seconds per request there).  bimodal: the
    shortest, the median and the longest context.  Otherwise the first and last."""
    order = sorted(range(w.B), key=lambda b: lens[b])
    if w.name == "dsv3":
        return list(range(w.B))
    if w.name == "fp8":
        return sorted({round(i * (w.B - 1) / 7) for i in range(8)})
    if w.name == "bimodal":
        return [order[0], order[len(order) // 2], order[-1]]
    if w.B > 1:
        return [0, w.B - 1]
    return [0]


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
@pytest.mark.parametrize("name", ["tiny", "dsv3", "long", "bimodal", "fp8"])
def test_full_size_sampled(name):
    w = W.WORKLOADS[name]
    dw = Hn.build(w)
    dw.step.run()
    torch.cuda.synchronize()
    assert dw.cache.check_errors() == 0
    ow = OracleWorkload(w)
    assert np.array_equal(dw.step.page_table.cpu().numpy(), ow.page_table())
    R = w.Tq * w.H
    tol = TOL[w.kv_dtype]
    for b in _samples(w, dw.lens):
        op, lp, o_ref, l_ref = ow.decode(b, gen_device="cuda")
        assert row_rel_err(dw.step.o_part[:, b].cpu().numpy().reshape(w.c, R, 512), op) < tol
        assert lse_err(dw.step.lse_part[:, b].cpu().numpy().reshape(w.c, R), lp) < tol
        assert row_rel_err(dw.step.o[b].cpu().numpy().reshape(R, 512), o_ref) < tol
        assert lse_err(dw.step.lse[b].cpu().numpy().reshape(R), l_ref) < tol
        # this request's stored rows, bit for bit, in every shard
        for r in range(w.c):
            import oracle as O
            pos, slots = O.shard_view(ow.rmap, b, dw.lens[b], r)
            if len(slots) == 0:
                continue
            idx = torch.from_numpy(slots).cuda()
            got = dw.cache.pools[r].index_select(0, idx).view(torch.uint8).cpu().numpy()
            want, scs = ow.pools.read(r, slots)
            assert np.array_equal(got.reshape(len(slots), -1), want.view(np.uint8).reshape(len(slots), -1))
            if w.kv_dtype == "e4m3":
                gs = dw.cache.scales[r].index_select(0, idx).cpu().numpy()
                assert np.array_equal(gs.view(np.uint32), scs.view(np.uint32))
    del dw
    torch.cuda.empty_cache()
