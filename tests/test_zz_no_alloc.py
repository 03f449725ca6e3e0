"""qgemm_w4a16_noalloc: the W4A16 GEMM for callers that cannot allocate device
memory -- a plugin inside a host runtime that owns every device allocation, or a
decode loop where a cudaMalloc (which may synchronize the device) is not allowed.
Its scratch is a fixed array inside the library.

Called through the C ABI and compared with qgemm_w4a16, which takes a
caller-provided workspace: the same kernel, schedule and reduction order, so the
two must agree bit for bit, on two calls in a row (the second call reuses the
scratch the first one left).  Both are also checked against the oracle.  The
first call of a process sets the scratch up; one case makes that first call on a
non-blocking stream in a fresh process.  This file is collected last on purpose.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = 5e-3
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nerr(y, ref):
    y = y.float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref).astype(np.float64)
    assert np.isfinite(y).all()
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-30))


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    import int8_weight_quantized_int4_gb300 as q
    return q


def _call(q, x, packed, M, N, K, y, stream):
    L = q.lib()
    return L.qgemm_w4a16_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(packed.data_ptr()), M, N, K,
                                 ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("M", [1, 16])
def test_noalloc_matches_workspace_entry_point(q, M):
    dev = torch.device("cuda:0")
    p = synth.projection(M)                         # K = N = 5120, a split-K (stream-K) shape
    packed = q.qpack_w4(p.codes.to(dev), p.scales.to(dev))
    x = p.x.to(dev)
    ref = q.qgemm_w4a16(x, packed, p.N, p.K)       # the entry point with a workspace
    torch.cuda.synchronize()
    exp = oracle.w4a16(p.x, p.codes, p.scales)
    assert _nerr(ref, exp) <= TOL
    stream = torch.cuda.current_stream(dev)
    for call in range(2):
        y = torch.full((M, p.N), float("nan"), dtype=torch.float16, device=dev)
        rc = _call(q, x, packed, M, p.N, p.K, y, stream)
        assert rc == q.QW_OK, q.lib().qw_last_error_string()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), call
        assert _nerr(y, exp) <= TOL, (call, _nerr(y, exp))
    assert q.device_error() == 0


_FRESH = r"""
import ctypes, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import int8_weight_quantized_int4_gb300 as q, synth
dev = torch.device("cuda:0"); torch.cuda.set_device(dev)
p = synth.projection(16)
packed = q.qpack_w4(p.codes.to(dev), p.scales.to(dev)); x = p.x.to(dev)
torch.cuda.synchronize()
s = torch.cuda.Stream(dev)                       # non-blocking with respect to the legacy stream
L = q.lib()
same = []
with torch.cuda.stream(s):
    ref = q.qgemm_w4a16(x, packed, p.N, p.K)
    for call in range(2):
        y = torch.full((16, p.N), float("nan"), dtype=torch.float16, device=dev)
        rc = L.qgemm_w4a16_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(packed.data_ptr()), 16,
                                   p.N, p.K, ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(s.cuda_stream))
        assert rc == 0, L.qw_last_error_string()
        s.synchronize()
        same.append(bool(torch.equal(y.view(torch.int16), ref.view(torch.int16))))
print("RESULT", same, q.device_error(s))
"""


def test_noalloc_first_call_on_a_nonblocking_stream(q):
    """A fresh process whose first qgemm_w4a16_noalloc call (the one that sets the scratch
    up) is on a non-blocking stream gets the same bits as qgemm_w4a16, twice."""
    r = subprocess.run([sys.executable, "-c", _FRESH, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT")][-1]
    assert line == "RESULT [True, True] 0", line


def test_noalloc_rejects_shapes_beyond_its_scratch(q):
    dev = torch.device("cuda:0")
    M, N, K = 64, 5120, 5120                         # needs ~10 MB of partial sums
    x = torch.zeros((M, K), dtype=torch.float16, device=dev)
    packed = torch.zeros(q.qpack_w4_bytes(N, K), dtype=torch.uint8, device=dev)
    y = torch.zeros((M, N), dtype=torch.float16, device=dev)
    rc = _call(q, x, packed, M, N, K, y, torch.cuda.current_stream(dev))
    assert rc == q.QW_ERR_WORKSPACE
    assert b"built-in scratch" in q.lib().qw_last_error_string()
