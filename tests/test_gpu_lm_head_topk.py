"""The lm_head with the sampler's top-k fused in (qgemm_lm_head_topk).

Bars: the logits y are bit-identical to the plain GEMM on the same inputs (same kernel,
plan and reduction order) and within the GEMM tolerance of the oracle on sampled
columns; (vals, idx) equal the oracle's top-k of those logits exactly (largest first,
ties to the smaller index, -0 equal to +0).  Shapes: the 248,320-row head in both
weight formats at M in {1, 16, 64}, and small tie-heavy cases that make many 128-row
tiles share their maximum (more candidate tiles than one selection batch holds).
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


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy()


def _check_topk(y, vals, idx, k):
    ov, oi = oracle.topk(y.cpu().numpy(), k)
    assert np.array_equal(idx.cpu().numpy().astype(np.int64), oi)
    assert np.array_equal(bits(vals), ov.view(np.int16))


def _plain(q, mode, x, packed, N, K):
    return q.qgemm_w4a16(x, packed, N, K) if mode == q.MODE_W4A16 else q.qgemm_w8a16(x, packed, N, K)


_HEADS = {}


def _head(q, mode):
    if mode not in _HEADS:
        p = synth.lm_head_int4(64) if mode == q.MODE_W4A16 else synth.lm_head(64)
        pack = q.qpack_w4 if mode == q.MODE_W4A16 else q.qpack_w8
        _HEADS[mode] = (p, pack(p.codes.to(DEV), p.scales.to(DEV)))
    return _HEADS[mode]


@pytest.mark.parametrize("fmt", ["w4a16", "w8a16"])
@pytest.mark.parametrize("M", [1, 16, 64])
def test_lm_head_topk_full_vocabulary(q, fmt, M):
    mode = q.MODE_W4A16 if fmt == "w4a16" else q.MODE_W8A16
    p, packed = _head(q, mode)
    x = p.x[:M].contiguous().to(DEV)
    k = 64
    y, vals, idx = q.qgemm_lm_head_topk(mode, x, packed, p.N, p.K, k)
    ref_y = _plain(q, mode, x, packed, p.N, p.K)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    assert torch.equal(y.view(torch.int16), ref_y.view(torch.int16))
    cols = np.concatenate([np.arange(0, p.N, 1999), [p.N - 1]])
    ref = (oracle.w4a16 if mode == q.MODE_W4A16 else oracle.w8a16)(p.x[:M], p.codes[cols], p.scales[cols])
    got = y.cpu().numpy()[:, cols].astype(np.float64)
    assert np.abs(got - ref).max() / np.abs(ref).max() <= TOL
    _check_topk(y, vals, idx, k)
    # the winners' logits are the largest of their rows
    assert (vals.float().min(dim=1).values >= y.float().topk(k, dim=1).values[:, -1]).all()


def _tie_problem(M, N, K, seed):
    """Integer logits in a narrow range: codes in {-1, 0, 1}, scales 1, x in {0, 1}, so
    most 128-row tiles share their maximum."""
    gen = synth.generator(seed)
    codes = torch.randint(-1, 2, (N, K), generator=gen, dtype=torch.int8)
    scales = torch.ones((N, K // 128), dtype=torch.float16)
    x = torch.randint(0, 2, (M, K), generator=gen).to(torch.float16)
    return codes, scales, x


@pytest.mark.parametrize("M,N,K,k", [(1, 16384, 256, 64), (5, 16384, 256, 1), (16, 32768, 128, 64),
                                     (64, 8192, 256, 33), (3, 1024, 256, 64), (2, 256, 128, 7),
                                     # row-block kernel with two 8-token tiles, 2 and 3 row blocks a CTA
                                     (12, 4096, 512, 64), (16, 7168, 1024, 40)])
def test_lm_head_topk_ties(q, M, N, K, k):
    codes, scales, x = _tie_problem(M, N, K, seed=M * 131 + N + k)
    packed = q.qpack_w4(codes.to(DEV), scales.to(DEV))
    xd = x.to(DEV)
    ws = q.Workspace(DEV)
    for rep in range(2):                       # the tile maxima are cleared for the next call
        y, vals, idx = q.qgemm_lm_head_topk(q.MODE_W4A16, xd, packed, N, K, k, ws=ws)
        torch.cuda.synchronize()
        assert q.device_error() == 0
        assert torch.equal(y.view(torch.int16), q.qgemm_w4a16(xd, packed, N, K).view(torch.int16))
        _check_topk(y, vals, idx, k)
        zero = int(q.lib().qgemm_lm_head_topk_workspace_zero_bytes(q.MODE_W4A16, M, N, K, k))
        assert zero > 0 and int(ws.buf[:zero].count_nonzero()) == 0


def test_lm_head_topk_zero_rows(q):
    """x = 0: every logit is +0 or -0, all equal: the first k indices, the logits' own bits."""
    M, N, K, k = 3, 4096, 256, 64
    codes, scales, _ = _tie_problem(M, N, K, seed=7)
    scales[::3] = -1.0
    packed = q.qpack_w4(codes.to(DEV), scales.to(DEV))
    x = torch.zeros((M, K), dtype=torch.float16, device=DEV)
    y, vals, idx = q.qgemm_lm_head_topk(q.MODE_W4A16, x, packed, N, K, k)
    torch.cuda.synchronize()
    assert (idx.cpu() == torch.arange(k, dtype=torch.int32)).all()
    assert np.array_equal(bits(vals), bits(y[:, :k]))
    _check_topk(y, vals, idx, k)
