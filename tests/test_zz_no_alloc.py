"""The allocation-free decode entry point, called through the C ABI.

dcpmla_decode_noalloc serves callers that cannot give the decode a device
workspace (a plugin whose host framework owns all device memory, a process
whose memory is fully reserved by a caching allocator, a latency-critical
loop where cudaMalloc would synchronise the device).  Its scratch is a static
device array inside the library.  These checks compare it, two calls in a row,
with the fp64 oracle on the same seeded inputs (every shard's partial output and
LSE, within the parity tolerance: 2e-3 for bf16 KV, 1e-2 for E4M3 KV against the
dequantised oracle) and with the regular dcpmla_decode, and check that oversized
shapes are refused before any launch.

This file is collected last on purpose; it also passes when run alone.
"""
import pytest
import torch

import dcp_harness as Hn
import dcp_workloads as W
from decode_context_mla_gb300 import binding as B
from oracle_ref import TOL, OracleWorkload, lse_err, row_rel_err

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
def test_noalloc_matches_oracle_and_regular_decode_two_calls(name):
    w = CASES[name]
    dw = Hn.build(w)
    dw.step.run()                                   # append the step's new tokens
    torch.cuda.synchronize()
    st = dw.step
    R = w.Tq * w.H
    tol = TOL[w.kv_dtype]
    ow = OracleWorkload(w)
    want = {b: ow.decode(b)[:2] for b in range(w.B)}   # (o_parts (c,R,512), lse_parts (c,R))
    ref_o = torch.empty_like(st.o_part)
    ref_l = torch.empty_like(st.lse_part)
    B.dcpmla_decode(*_args(dw), ref_o, ref_l, st.workspace, dw.cache.err)
    torch.cuda.synchronize()
    ref_o, ref_l = ref_o.cpu().numpy(), ref_l.cpu().numpy()
    free_after_first = None
    o = torch.empty_like(st.o_part)
    lse = torch.empty_like(st.lse_part)
    for call in range(2):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        B.dcpmla_decode_noalloc(*_args(dw), o, lse, dw.cache.err)
        torch.cuda.synchronize()
        assert dw.cache.check_errors() == 0
        go, gl = o.cpu().numpy(), lse.cpu().numpy()
        for b in range(w.B):
            op, lp = want[b]
            assert row_rel_err(go[:, b].reshape(w.c, R, 512), op) < tol, (name, call, b, "o")
            assert lse_err(gl[:, b].reshape(w.c, R), lp) < tol, (name, call, b, "lse")
        assert row_rel_err(go, ref_o) < tol, (name, call)
        assert lse_err(gl, ref_l) < tol, (name, call)
        # A weak check that the call allocates nothing: device-wide free memory must not
        # drop by a cudaMalloc granule (2 MiB) between the first and the second call.  The
        # first call may load the library's module, which maps the static scratch array.
        free_now = torch.cuda.mem_get_info()[0]
        if call == 0:
            free_after_first = free_now
        else:
            assert free_after_first - free_now < (2 << 20)


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
