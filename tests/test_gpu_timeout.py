"""The GEMM kernels' wait limit, driven through unmodified kernels.

Every wait inside a GEMM kernel (a pipeline stage waiting for another) has a time
limit; one that runs past it raises the CTA's abort flag, the other roles give up,
each producer issues no further copy and waits for the copies or MMAs it already
started, and the kernel ends with QW_ERR_TIMEOUT in the device error word.  The QW_OPT_WAIT_LIMIT_US option
lowers the limit for the calls that follow: at 0 every wait that is not already
satisfied at its first (non-blocking) check gives up, so each kernel below takes the
abort path from its first pending wait on (no kernel is modified, nothing is left
waiting).  Each shape is chosen so that some wait is bound to pend.
Afterwards, with the default limit back and the workspace zero-filled again, the
same call gives the bits it gave before and matches the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = 5e-3
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    import int8_weight_quantized_int4_gb300 as q
    return q


def _nerr(y, ref):
    y = y.float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref).astype(np.float64)
    assert np.isfinite(y).all()
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-30))


# (mode, M, N, K): which kernel and roles each case drives
CASES = [
    ("w4a16", 1, 256, 256),        # decode kernel, one 8-token tile, stream-K split
    ("w4a16", 16, 256, 512),       # decode kernel, 16 tokens
    ("w4a8", 16, 256, 512),        # decode kernel widening int8 codes
    ("w4a8_fused", 2, 4096, 6144), # row-block kernel quantizing the fp16 rows itself
    ("w4a8_fused", 16, 5120, 2048), # the quantizer, then the row-block kernel on its codes
    ("w4a16", 64, 256, 512),       # tcgen05 GEMM, 64-token tile, two MMA issuers
    ("w4a8", 64, 384, 512),        # tcgen05 GEMM, int8 widened in the kernel
    ("w8a16", 16, 256, 512),       # tcgen05 GEMM, int8 weights, four issuers
    ("w4a16", 512, 512, 1024),     # tcgen05 GEMM, 256-token tiles
    ("w4a16", 1, 2048, 8192),      # decode kernel, several chunks per CTA (ring laps)
    ("w4a16", 64, 1024, 8192),     # tcgen05 GEMM, several chunks per CTA
]


def _setup(q, mode, M, N, K):
    bits = 8 if mode == "w8a16" else 4
    p = synth.make_problem(M, N, K, seed=900 + M + N + K, bits=bits,
                           **({"code_range": (-128, 127)} if bits == 8 else {}))
    x = p.x.to(DEV)
    if bits == 8:
        packed = q.qpack_w8(p.codes.to(DEV), p.scales.to(DEV))
        ref = oracle.w8a16(p.x, p.codes, p.scales)
        return (lambda ws: q.qgemm_w8a16(x, packed, N, K, ws=ws)), ref
    packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    if mode == "w4a16":
        return (lambda ws: q.qgemm_w4a16(x, packed, N, K, ws=ws)), oracle.w4a16(p.x, p.codes, p.scales)
    oq, os_ = oracle.quant_act_int8(p.x)
    ref = oracle.w4a8(oq, os_, p.codes, p.scales)
    if mode == "w4a8_fused":
        return (lambda ws: q.qgemm_w4a8_fused(x, packed, N, K, ws=ws)), ref
    xq, xs = q.quant_act_int8(x)
    return (lambda ws: q.qgemm_w4a8(xq, xs, packed, N, K, ws=ws)), ref


@pytest.mark.parametrize("mode,M,N,K", CASES)
def test_wait_limit_ends_kernel_with_timeout_then_recovers(q, mode, M, N, K):
    run, ref = _setup(q, mode, M, N, K)
    ws = q.Workspace(DEV)
    y0 = run(ws)
    assert q.device_error() == q.QW_OK
    assert _nerr(y0, ref) <= TOL
    launches = q.num_kernel_launches()
    q.set_wait_limit_us(0)
    errs = []
    try:
        for _ in range(3):                         # the abort path races copies in flight
            run(ws)                                # enqueues; the error is read below
            errs.append(q.device_error())
            ws.zero()
    finally:
        q.set_wait_limit_us(None)
    assert q.num_kernel_launches() > launches
    assert errs == [q.QW_ERR_TIMEOUT] * 3, errs
    assert q.lib().qw_get_option(q.QW_OPT_WAIT_LIMIT_US) == q.DEFAULT_WAIT_LIMIT_US
    ws.zero()
    y1 = run(ws)
    assert q.device_error() == q.QW_OK
    assert torch.equal(y1.view(torch.int16), y0.view(torch.int16))
    assert _nerr(y1, ref) <= TOL


def test_default_limit_gives_no_timeout(q):
    """A short but nonzero limit (a second) is far above any wait of a healthy kernel."""
    run, ref = _setup(q, "w4a16", 16, 256, 512)
    ws = q.Workspace(DEV)
    q.set_wait_limit_us(1_000_000)
    try:
        y = run(ws)
        err = q.device_error()
    finally:
        q.set_wait_limit_us(None)
    assert err == q.QW_OK
    assert _nerr(y, ref) <= TOL
