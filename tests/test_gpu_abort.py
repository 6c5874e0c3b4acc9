"""A pipeline wait that runs out, on the GPU: the error is reported and the context survives.

Every wait inside the tensor-core decode kernels gives up after a limit (about
one second by default).  Here the limit is lowered to one clock64 cycle
through the test-only dcpmla_testing_set_wait_limit, so the first wait of each
CTA that is not already satisfied gives up: the CTA aborts, every role leaves
its loop, the copies and MMAs already issued are waited for, TMEM is freed and
the kernel returns.  The call must come back (no hang), set
DCPMLA_DERR_TIMEOUT in the error word, and leave the context usable: the next
call at the default limit runs clean and matches the fp64 oracle.

Each case reaches one kernel: the token-major few-head kernel (tiny), the
persistent 128-row bf16 kernel (dsv3-shaped), the non-persistent 128-row bf16
kernel (the fused decode + merge) and the 128-row E4M3 kernel (fp8-shaped).
The barrier protocol of the abort path is modelled on the CPU in
test_tc_pipeline_protocol.py.
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
    "tiny": (W.WORKLOADS["tiny"], False, B.PATH_TC_FEWHEAD),
    "dsv3_persistent": (W.scaled(W.WORKLOADS["dsv3"], B=3, L=2000), False, B.PATH_TC_ROWS),
    "dsv3_fused": (W.scaled(W.WORKLOADS["dsv3"], B=2, L=3000), True, B.PATH_TC_ROWS),
    "fp8_verify": (W.scaled(W.WORKLOADS["fp8"], B=2, L=3000), False, B.PATH_TC_ROWS),
}


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from decode_context_mla_gb300.build import build
    build()


@needs_cuda
@pytest.mark.parametrize("name", list(CASES))
def test_wait_limit_runs_out_then_the_next_call_is_correct(name):
    w, fused, path = CASES[name]
    kv = B.KV_BF16 if w.kv_dtype == "bf16" else B.KV_E4M3
    assert B.dcpmla_decode_path(w.B, w.Tq, w.H, w.P, w.c, w.c, kv, max(w.pages_per_request()))[0] == path
    dw = Hn.build(w, fused=fused)
    st = dw.step
    st.run()                                          # the step's appends, at the default limit
    torch.cuda.synchronize()
    assert dw.cache.check_errors() == 0
    try:
        B.dcpmla_testing_set_wait_limit(1)
        dw.cache.err.zero_()
        st.run_decode()
        torch.cuda.synchronize()                      # the aborted launch returns
        assert dw.cache.check_errors() & B.DERR_TIMEOUT
    finally:
        B.dcpmla_testing_set_wait_limit(0)
    # the context survived: the same call at the default limit is clean and correct
    dw.cache.err.zero_()
    st.o.fill_(float("nan"))
    st.lse.fill_(float("nan"))
    st.run_decode()
    st.run_merge()
    torch.cuda.synchronize()
    assert dw.cache.check_errors() == 0
    ow = OracleWorkload(w)
    R = w.Tq * w.H
    tol = TOL[w.kv_dtype]
    o, lse = st.o.cpu().numpy(), st.lse.cpu().numpy()
    for b in range(w.B):
        _, _, o_ref, l_ref = ow.decode(b)
        assert row_rel_err(o[b].reshape(R, 512), o_ref) < tol, (name, b)
        assert lse_err(lse[b].reshape(R), l_ref) < tol, (name, b)


@needs_cuda
@pytest.mark.parametrize("name", list(CASES))
def test_waits_running_out_at_any_point_end_cleanly(name):
    """Limits from one cycle to ~0.1 ms make the waits run out at different points of the
    pipeline (or not at all): every call returns, and it either reports DCPMLA_DERR_TIMEOUT or
    its output matches the oracle; a call at the default limit afterwards is correct."""
    w, fused, _ = CASES[name]
    dw = Hn.build(w, fused=fused)
    st = dw.step
    st.run()
    torch.cuda.synchronize()
    assert dw.cache.check_errors() == 0
    ow = OracleWorkload(w)
    want = {b: ow.decode(b)[2:] for b in range(w.B)}
    R = w.Tq * w.H
    tol = TOL[w.kv_dtype]

    def matches():
        o, lse = st.o.cpu().numpy(), st.lse.cpu().numpy()
        return all(row_rel_err(o[b].reshape(R, 512), want[b][0]) < tol and
                   lse_err(lse[b].reshape(R), want[b][1]) < tol for b in range(w.B))

    timed_out = 0
    try:
        for limit in (1, 1 << 12, 1 << 15, 1 << 18):
            for _ in range(3):
                B.dcpmla_testing_set_wait_limit(limit)
                dw.cache.err.zero_()
                st.o.fill_(float("nan"))
                st.run_decode()
                st.run_merge()
                torch.cuda.synchronize()
                e = dw.cache.check_errors()
                assert e & ~B.DERR_TIMEOUT == 0, (name, limit, e)
                if e & B.DERR_TIMEOUT:
                    timed_out += 1
                else:
                    assert matches(), (name, limit)
    finally:
        B.dcpmla_testing_set_wait_limit(0)
    assert timed_out > 0
    dw.cache.err.zero_()
    st.run_decode()
    st.run_merge()
    torch.cuda.synchronize()
    assert dw.cache.check_errors() == 0
    assert matches()
