"""int8-QK causal prefill attention on the GPU against the oracle.

Bars: the query and key codes and their scales are bit-exact (the key side after the
per-channel mean smoothing); V^T is V transposed bit for bit; the output is within
max|o - o_ref| / max|o_ref| <= 5e-3 of the oracle (P . V runs with P in fp16) and its
cosine similarity to the oracle's binary64 result is above 0.99999 (the page's accuracy
statement).  Shapes: a full prefill (T = S), a chunk at the end of a 4k context, grouped
heads, a single block, and rows of zeros.
"""
import numpy as np
import pytest
import torch

import oracle.attention as attn
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


CASES = [(1024, 1024, 8, 2), (512, 4096, 4, 1), (128, 128, 2, 2), (256, 1024, 6, 3)]


@pytest.mark.parametrize("T,S,Hq,Hkv", CASES)
def test_attention_matches_oracle(q, T, S, Hq, Hkv):
    qq, kk, vv = synth.attention(T, S, Hq, Hkv, seed=T + S + Hq)
    if T >= 256:
        qq[5, 1] = 0.0                                   # a zero query row: scale 0, codes 0
    ws = q.Workspace(DEV)
    out = q.attn_int8qk_prefill(qq.to(DEV), kk.to(DEV), vv.to(DEV), ws=ws)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    qc, qs, kc, ks, vt = q.attn_int8qk_intermediates(ws, T, S, Hq, Hkv)
    oq, oqs = attn.quant_rows_f32(qq.numpy().astype(np.float32))        # [T, Hq, d], [T, Hq]
    ok_, oks = attn.quant_rows_f32(attn.smooth_k(kk.numpy()))           # [S, Hkv, d], [S, Hkv]
    assert np.array_equal(qc.cpu().float().numpy().astype(np.int64), oq.transpose(1, 0, 2).astype(np.int64))
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), oqs.T.copy().view(np.uint32))
    assert np.array_equal(kc.cpu().float().numpy().astype(np.int64), ok_.transpose(1, 0, 2).astype(np.int64))
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.T.copy().view(np.uint32))
    assert torch.equal(vt.cpu(), vv.permute(1, 2, 0).contiguous())
    ref64 = attn.attn_int8qk(qq.numpy(), kk.numpy(), vv.numpy(), out_f64=True)
    got = out.cpu().float().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    err = np.abs(got - ref64.astype(np.float16).astype(np.float64)).max() / np.abs(ref64).max()
    assert err <= TOL, err
    cos = float((got * ref64).sum() / np.sqrt((got * got).sum() * (ref64 * ref64).sum()))
    assert cos > 0.99999, cos


def test_attention_long_context_repeats_bitwise(q):
    """A 2k chunk at the end of a 16k context (128 key blocks a query block, several
    waves of CTAs), run 30 times: every run gives the same bits (the pipeline's waits
    leave no window for a read before its producer)."""
    T, S, Hq, Hkv = 2048, 16384, 24, 4
    qq, kk, vv = synth.attention(T, S, Hq, Hkv, seed=11)
    qd, kd, vd = qq.to(DEV), kk.to(DEV), vv.to(DEV)
    ws = q.Workspace(DEV)
    base = q.attn_int8qk_prefill(qd, kd, vd, ws=ws).clone()
    out = torch.empty_like(base)
    for _ in range(30):
        q.attn_int8qk_prefill(qd, kd, vd, out=out, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), base.view(torch.int16))
    assert q.device_error() == 0


def test_attention_repeat_is_bitwise_stable(q):
    T, S, Hq, Hkv = 256, 512, 4, 2
    qq, kk, vv = synth.attention(T, S, Hq, Hkv, seed=3)
    a = q.attn_int8qk_prefill(qq.to(DEV), kk.to(DEV), vv.to(DEV))
    b = q.attn_int8qk_prefill(qq.to(DEV), kk.to(DEV), vv.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
