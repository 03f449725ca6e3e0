"""The measurement tools behind the design choices, through the C ABI.

* Route C for W4A8 on tcgen05 kind::f8f6f4: int4 weight codes are exact in e4m3, an
  int8 activation code q = 16 h + l (h = q >> 4 in [-8, 7], l = q & 15) is the sum of
  two e4m3-exact terms, so sum_k w_k q_k = sum_k w_k (16 h_k) + w_k l_k.  The test feeds
  those terms through one 128 x 16 x K MMA chain and compares with the integer dot
  product (int64 numpy matmul of the codes, the definition of the W4A8 inner sum).
* The warp-level MMA rate microbenchmark runs and reports a positive rate.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    import int8_weight_quantized_int4_gb300 as q
    return q


def _e4m3(v):
    import bench
    return bench.e4m3_of_int(v)


@pytest.mark.parametrize("K", [128, 512])
@pytest.mark.parametrize("a_tmem", [False, True])
def test_f8f6f4_int4_times_split_int8_is_exact(q, K, a_tmem):
    gen = synth.generator(700 + K)
    w = synth.codes_int4(128, K // 2, gen).numpy().astype(np.int64)
    a = synth.codes_int8(16, K // 2, gen).numpy().astype(np.int64)
    a[0, :] = -127                      # extreme magnitudes in the first token row
    w[0, :] = -8
    A = np.repeat(w, 2, axis=1)                                   # each weight code twice
    B = np.stack([16 * (a >> 4), a & 15], axis=2).reshape(16, K)  # 16 h, l interleaved
    ref = w @ a.T
    d = q.diag_f8f6f4_gemm(torch.from_numpy(_e4m3(A)).cuda(), torch.from_numpy(_e4m3(B)).cuda(), a_tmem)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    assert np.array_equal(d.cpu().numpy().astype(np.float64), ref.astype(np.float64))


def test_e4m3_encoder_against_torch():
    """The test's e4m3 encoder agrees with torch's float8_e4m3fn conversion."""
    v = np.arange(-16, 17)
    v = np.concatenate([v, 16 * np.arange(-8, 8)])
    ours = _e4m3(v)
    theirs = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_mma_rate_microbenchmark_runs(q):
    ops, sink = q.diag_mma_peak("s8", 8, 100, 8)
    torch.cuda.synchronize()
    assert ops == 2.0 * 16 * 8 * 32 * 8 * 8 * 100 * 8
    assert q.device_error() == 0
