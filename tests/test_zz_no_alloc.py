"""The allocation-free decode entry point, called through the C ABI.

dcpmla_decode_noalloc serves callers that cannot give the decode a device
workspace (a plugin whose host framework owns all device memory, a process
whose memory is fully reserved by a caching allocator, a latency-critical
loop where cudaMalloc would synchronise the device).  Its scratch is a static
device array inside the library.  These checks compare it with the regular
dcpmla_decode on the same inputs, two calls in a row, within the parity
tolerance, and check that oversized shapes are refused before any launch.

This file is collected last on purpose; it also passes when run alone.
"""
import pytest
import torch

import dcp_harness as Hn
import dcp_workloads as W
from decode_context_mla_gb300 import binding as B
from oracle_ref import TOL, lse_err, row_rel_err

pytestmark = pytest.mark.gpu
needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")

CASES = {
    "tiny": W.WORKLOADS["tiny"],
    "long_split": W.scaled(W.WORKLOADS["long"], B=2, L=40000),
    "fp8_verify": W.scaled(W.WORKLOADS["fp8"], B=2, L=3000),
    "bimodal_mix": W.scaled(W.WORKLOADS["bimodal"], B=10, lengths_mix=(5, 3000, 9000, 1, 40)),
}


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from decode_context_mla_gb300.build import build
    build()


def _args(dw):
    st, c = dw.step, dw.cache
    return (st.q, c.pools, c.scales, c.kv_dtype, st.page_table, st.seq_lens, c.P, c.c, 0, c.c,
            st.sm_scale, st.lse_base)


@needs_cuda
@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_regular_decode_two_calls(name):
    w = CASES[name]
    dw = Hn.build(w)
    dw.step.run()                                   # append the step's new tokens
    torch.cuda.synchronize()
    st = dw.step
    ref_o = torch.empty_like(st.o_part)
    ref_l = torch.empty_like(st.lse_part)
    B.dcpmla_decode(*_args(dw), ref_o, ref_l, st.workspace, dw.cache.err)
    torch.cuda.synchronize()
    tol = TOL[w.kv_dtype]
    free_after_first = None
    o = torch.empty_like(st.o_part)
    lse = torch.empty_like(st.lse_part)
    for call in range(2):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        B.dcpmla_decode_noalloc(*_args(dw), o, lse, dw.cache.err)
        torch.cuda.synchronize()
        assert dw.cache.check_errors() == 0
        assert row_rel_err(o.cpu().numpy(), ref_o.cpu().numpy()) < tol, (name, call)
        assert lse_err(lse.cpu().numpy(), ref_l.cpu().numpy()) < tol, (name, call)
        free_now = torch.cuda.mem_get_info()[0]
        if call == 0:
            free_after_first = free_now
        else:
            assert free_now == free_after_first      # the second call took no device memory


@needs_cuda
def test_noalloc_refuses_shapes_beyond_its_scratch():
    """Full bimodal batch: the CUDA-core decode's split-KV scratch for it exceeds the static
    array, so the call is refused before any launch."""
    w = W.WORKLOADS["bimodal"]
    pages = w.pages_per_request()
    dev = "cuda"
    q = torch.zeros((w.B, w.Tq, w.H, W.D_K), dtype=torch.bfloat16, device=dev)
    pools = [torch.zeros((w.P, W.D_K), dtype=torch.bfloat16, device=dev) for _ in range(w.c)]
    pt = torch.zeros((w.B, max(pages)), dtype=torch.int32, device=dev)
    lens = torch.ones(w.B, dtype=torch.int32, device=dev)
    o = torch.zeros((w.c, w.B, w.Tq, w.H, 512), dtype=torch.float32, device=dev)
    lse = torch.zeros((w.c, w.B, w.Tq, w.H), dtype=torch.float32, device=dev)
    with pytest.raises(B.DcpmlaError) as e:
        B.dcpmla_decode_noalloc(q, pools, None, B.KV_BF16, pt, lens, w.P, w.c, 0, w.c,
                                w.sm_scale, B.LSE_E, o, lse, None)
    assert e.value.status == B.ERR_CAPACITY
    torch.cuda.synchronize()
    assert torch.all(o == 0)                        # nothing was launched
