"""qgemm_w4a16_noalloc: the W4A16 GEMM for callers that cannot allocate device
memory (its scratch is a fixed array inside the library).  Called through the C
ABI and compared with qgemm_w4a16, which takes a caller-provided workspace, on
two calls in a row (the second call reuses the scratch the first one left).
This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

TOL = 5e-3


def _nerr(y, ref):
    y = y.float().cpu().numpy().astype(np.float64)
    ref = ref.float().cpu().numpy().astype(np.float64)
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


@pytest.mark.parametrize("M", [1, 16])
def test_noalloc_matches_workspace_entry_point(q, M):
    dev = torch.device("cuda:0")
    p = synth.projection(M)                         # K = N = 5120, a split-K (stream-K) shape
    packed = q.qpack_w4(p.codes.to(dev), p.scales.to(dev))
    x = p.x.to(dev)
    ref = q.qgemm_w4a16(x, packed, p.N, p.K)       # the entry point with a workspace
    L = q.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    for call in range(2):
        y = torch.full((M, p.N), float("nan"), dtype=torch.float16, device=dev)
        rc = L.qgemm_w4a16_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(packed.data_ptr()),
                                   M, p.N, p.K, ctypes.c_void_p(y.data_ptr()), stream)
        assert rc == q.QW_OK, L.qw_last_error_string()
        torch.cuda.synchronize()
        assert _nerr(y, ref) <= TOL, (call, _nerr(y, ref))
    assert q.device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(q):
    dev = torch.device("cuda:0")
    M, N, K = 64, 5120, 5120                         # needs ~10 MB of partial sums
    x = torch.zeros((M, K), dtype=torch.float16, device=dev)
    packed = torch.zeros(q.qpack_w4_bytes(N, K), dtype=torch.uint8, device=dev)
    y = torch.zeros((M, N), dtype=torch.float16, device=dev)
    L = q.lib()
    rc = L.qgemm_w4a16_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(packed.data_ptr()),
                               M, N, K, ctypes.c_void_p(y.data_ptr()), None)
    assert rc == q.QW_ERR_WORKSPACE
    assert b"built-in scratch" in L.qw_last_error_string()
