"""Pins for the CPU oracle: exact brute force, closed forms, library routines and
the invariants the method implies.  CPU only.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, a wrong group index, a rounding mode) fails
at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    if isinstance(t, torch.Tensor):
        t = t.numpy()
    return np.ascontiguousarray(t).view(np.uint16)


# ---------------------------------------------------------------- binary16 ---

def test_half_to_double_exhaustive_vs_numpy():
    """Every finite binary16 pattern decodes to numpy's value (library routine)."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in allbits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_double_to_half_rne_vs_numpy():
    """binary64 -> binary16 is round-to-nearest-even, incl. ties, subnormals, overflow."""
    rng = np.random.default_rng(123)
    vals = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-9, 6, 3000))
    # exact ties between adjacent halves, in the normal and subnormal range
    h = np.arange(0, 0x7BFF, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    h2 = (np.arange(0, 0x7BFF, 37, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    vals += list((h + h2) / 2) + list(-(h + h2) / 2)
    vals += [65504.0, 65519.99, 65520.0, 70000.0, -65520.0, 2.0 ** -25, 2.0 ** -24 * 1.5,
             2.0 ** -14 - 2.0 ** -26, 0.0, -0.0, 1e-30]
    got = np.array([oracle.double_to_half(v) for v in vals], dtype=np.uint16)
    with np.errstate(over="ignore"):                  # 65520 and beyond round to inf, as intended
        ref = np.array(vals, dtype=np.float64).astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------- act quantizer ---

def _act_cases():
    gen = synth.generator(7)
    x = synth.activations(5, 256, gen, outlier_frac=0.02)
    x[1] = 0                                   # all-zero row -> s = 0, codes 0
    x[2] = 0
    x[2, 17] = -3.5                            # single non-zero element
    x[3, :] = (torch.arange(256, dtype=torch.float32) - 128).to(torch.float16) * 2 ** -20  # subnormals
    return x


def test_quant_act_bruteforce():
    x = _act_cases()
    q, s = oracle.quant_act_int8(x)
    bq, bs = _brute.quant_act_int8(_bits(x))
    assert np.array_equal(q.astype(np.int64), bq)
    assert np.array_equal(s.astype(np.float64), bs)
    assert s[1] == 0 and not q[1].any()
    assert q[2, 17] == -127 and np.count_nonzero(q[2]) == 1


def test_quant_act_rounding_ties_to_even():
    """Values on exact .5 boundaries of x/s round to the even code."""
    # amax = 127 -> s = 1 exactly; x = k + 0.5 must round to even integers
    row = np.array([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5] + [0.0] * 120, dtype=np.float16)
    q, s = oracle.quant_act_int8(row[None, :])
    assert s[0] == 1.0
    assert list(q[0, :8]) == [127, 0, 2, 2, 0, -2, -2, 4]


def test_quant_act_properties():
    gen = synth.generator(11)
    x = synth.activations(16, 1024, gen, outlier_frac=0.01)
    q, s = oracle.quant_act_int8(x)
    xf = x.float().numpy().astype(np.float64)
    # reconstruction within half a step (+ the binary32 rounding of x/s)
    err = np.abs(xf - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert np.all(err <= s[:, None] * (0.5 + 1e-6))
    # the absmax element maps to +-127
    idx = np.abs(xf).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(16), idx]) == 127)
    assert np.all(np.abs(q) <= 127)
    # scaling a row by 2**j scales s by 2**j and leaves the codes unchanged
    q2, s2 = oracle.quant_act_int8((x.float() * 0.25).to(torch.float16))
    assert np.array_equal(q2, q) and np.array_equal(s2, s * np.float32(0.25))


# ------------------------------------------------------------------ GEMMs ---

@pytest.mark.parametrize("M,N,K,seed", [(1, 3, 128, 21), (3, 5, 256, 22), (2, 7, 384, 23)])
def test_w4a16_bruteforce_small(M, N, K, seed):
    p = synth.make_problem(M, N, K, seed=seed, outlier_frac=0.02)
    y = oracle.w4a16(p.x, p.codes, p.scales)
    ref = _brute.gemm_wxa16(_bits(p.x), p.codes.numpy(), _bits(p.scales))
    assert np.array_equal(_bits(y), ref)


def test_w4a16_bruteforce_tiny_config():
    """The M=4, K=256, N=512 W4A16 check, all outputs, exact."""
    p = synth.tiny_w4a16()
    assert (p.scales < 0).float().mean().item() == pytest.approx(0.5, abs=0.05)
    y = oracle.w4a16(p.x, p.codes, p.scales)
    ref = _brute.gemm_wxa16(_bits(p.x), p.codes.numpy(), _bits(p.scales))
    assert np.array_equal(_bits(y), ref)


def test_w8a16_bruteforce_small():
    p = synth.make_problem(3, 6, 256, seed=31, bits=8, scale_lo=0.001, scale_hi=0.01)
    y = oracle.w8a16(p.x, p.codes, p.scales)
    ref = _brute.gemm_wxa16(_bits(p.x), p.codes.numpy(), _bits(p.scales))
    assert np.array_equal(_bits(y), ref)


def test_w4a8_bruteforce_small():
    p = synth.make_problem(3, 6, 384, seed=41, outlier_frac=0.02)
    qa, sx = oracle.quant_act_int8(p.x)
    y = oracle.w4a8(qa, sx, p.codes, p.scales)
    ref = _brute.gemm_w4a8(qa, sx, p.codes.numpy(), _bits(p.scales))
    assert np.array_equal(_bits(y), ref)


def test_integer_special_case_is_int_matmul():
    """All scales 1 and integer activations: W4A16 is an exact integer matmul."""
    gen = synth.generator(51)
    M, N, K = 4, 9, 256
    codes = synth.codes_int4(N, K, gen)
    xi = torch.randint(-3, 4, (M, K), generator=gen)
    scales = torch.ones((N, K // 128), dtype=torch.float16)
    y = oracle.w4a16(xi.to(torch.float16), codes, scales)
    ref = (xi.numpy().astype(np.int64) @ codes.numpy().astype(np.int64).T)
    assert np.array_equal(y.astype(np.float64), ref.astype(np.float64))


def test_group_index_and_scale_sign():
    """Closed form: one non-zero group scale picks exactly the K-range of that group,
    with its sign (the unsigned-scale failure mode would flip the result)."""
    M, N, K = 2, 3, 512
    x = torch.ones((M, K), dtype=torch.float16)
    x[1] = 2.0
    codes = torch.zeros((N, K), dtype=torch.int8)
    codes[:, 256:384] = 3            # group 2 only
    codes[1, 0:128] = 7              # group 0, whose scale is zero below
    scales = torch.zeros((N, K // 128), dtype=torch.float16)
    scales[:, 2] = torch.tensor([-0.5, 0.25, -1.0], dtype=torch.float16)
    y = oracle.w4a16(x, codes, scales).astype(np.float64)
    expect = np.array([[-0.5, 0.25, -1.0]]) * 3 * 128 * np.array([[1.0], [2.0]])
    assert np.array_equal(y, expect)
    # the same computation in W4A8 with unit token scale
    qa = x.to(torch.int8).numpy()
    y8 = oracle.w4a8(qa, np.ones(M, np.float32), codes, scales).astype(np.float64)
    assert np.array_equal(y8, expect)


def test_invariant_a_sign_fold():
    """Folding each negative scale's sign into its codes leaves the result unchanged
    (bit-identical): q' = -q, s' = -s on every group with s < 0."""
    p = synth.make_problem(5, 64, 512, seed=61, outlier_frac=0.01)
    G = p.K // 128
    neg = (p.scales < 0)
    assert 0.3 < neg.float().mean().item() < 0.7
    negk = neg.repeat_interleave(128, dim=1)
    folded_codes = torch.where(negk, -p.codes.to(torch.int16), p.codes.to(torch.int16)).to(torch.int8)
    folded_scales = torch.where(neg, -p.scales, p.scales)
    assert (folded_scales >= 0).all() and folded_codes.max() <= 8
    y = oracle.w4a16(p.x, p.codes, p.scales)
    yf = oracle.w8a16(p.x, folded_codes, folded_scales)   # codes may now be +8
    assert np.array_equal(_bits(y), _bits(yf))
    qa, sx = oracle.quant_act_int8(p.x)
    assert G == 4


def test_invariant_b_w4a8_equals_w4a16_on_int8_exact_activations():
    gen = synth.generator(71)
    M, N, K = 6, 48, 640
    x = synth.int8_exact_activations(M, K, gen)
    codes = synth.codes_int4(N, K, gen)
    scales = synth.signed_scales(N, K // 128, gen, 0.002, 0.02)
    qa, sx = oracle.quant_act_int8(x)
    # the quantizer reproduces c and 2**-e exactly
    xf = x.float().numpy().astype(np.float64)
    assert np.array_equal(qa.astype(np.float64) * sx[:, None].astype(np.float64), xf)
    assert np.all(np.log2(sx) == np.round(np.log2(sx)))
    y16 = oracle.w4a16(x, codes, scales)
    y8 = oracle.w4a8(qa, sx, codes, scales)
    assert np.array_equal(_bits(y16), _bits(y8))


def test_invariant_c_int8_g128_roundtrip_near_pages_figure():
    with open(os.path.join(GOLDEN, "roundtrip_int8_g128.json")) as fh:
        g = json.load(fh)
    gen = synth.generator(81)
    w = torch.randn((512, 5120), generator=gen, dtype=torch.float32)
    codes, scales, err = oracle.roundtrip_int8_g128(w)
    lo, hi = g["accept_percent"]
    assert lo <= 100 * err <= hi, 100 * err
    # codes are symmetric int8 and each group's absmax maps to +-127
    assert codes.min() >= -127 and codes.max() <= 127
    gmax = np.abs(codes.reshape(512, 40, 128)).max(axis=2)
    assert (gmax == 127).mean() > 0.95


def test_invariant_d_w8a16_equals_w4a16_on_int4_codes():
    p = synth.make_problem(3, 32, 384, seed=91)
    y4 = oracle.w4a16(p.x, p.codes, p.scales)
    y8 = oracle.w8a16(p.x, p.codes, p.scales)
    assert np.array_equal(_bits(y4), _bits(y8))


def test_oracle_rejects_out_of_range_int4_codes():
    p = synth.make_problem(1, 2, 128, seed=3)
    bad = p.codes.clone()
    bad[0, 0] = 8
    with pytest.raises(ValueError):
        oracle.w4a16(p.x, bad, p.scales)


def test_w4a16_linear_in_activations():
    """Doubling x doubles y exactly (power-of-two scaling commutes with every rounding)."""
    p = synth.make_problem(4, 40, 256, seed=101)
    y = oracle.w4a16(p.x, p.codes, p.scales).astype(np.float64)
    y2 = oracle.w4a16((p.x.float() * 2).to(torch.float16), p.codes, p.scales).astype(np.float64)
    assert np.array_equal(2 * y, y2)


def test_quant_act_divide_not_reciprocal_bruteforce():
    """Many rows, with absmax values picked where a reciprocal multiply would round
    differently from the IEEE divide, and element values where x*(1/s) != x/s;
    expected codes and scales from exact rational brute force."""
    gen = synth.generator(13)
    cand = (torch.rand(20000, generator=gen) * 40 + 0.01).to(torch.float16).float().numpy()
    recip = cand * np.float32(1.0 / 127.0)
    div = cand / np.float32(127.0)
    amaxes = cand[recip != div][:40]
    assert len(amaxes) == 40
    x = synth.activations(40, 128, gen).float()
    x = x / x.abs().amax(dim=1, keepdim=True) * torch.from_numpy(amaxes)[:, None] * 0.999
    x[:, 0] = torch.from_numpy(amaxes)
    x = x.to(torch.float16)
    q, s = oracle.quant_act_int8(x)
    bq, bs = _brute.quant_act_int8(_bits(x))
    assert np.array_equal(s.astype(np.float64), bs)
    assert np.array_equal(q.astype(np.int64), bq)


# ------------------------------------------------ embedding gather and top-k --

def test_embed_w8_matches_exact_brute_force():
    """Dequant-on-gather ("In full" items 1-2): exact rational product, rounded once."""
    rng = np.random.default_rng(21)
    V, D = 7, 256
    codes = rng.integers(-128, 128, (V, D)).astype(np.int8)
    scales = rng.uniform(-0.02, 0.02, (V, D // 128)).astype(np.float16)
    scales[2, 1] = np.float16(2.0 ** -20)                  # subnormal scale
    scales[4, 0] = np.float16(-0.0)
    ids = np.array([0, 6, 2, 2, 4, 3])
    got = oracle.embed_w8(ids, codes, scales).view(np.uint16)
    want = _brute.embed_w8(ids, codes, scales.view(np.uint16))
    assert np.array_equal(got, want)


def test_embed_w8_equals_w8a16_on_unit_vectors():
    """Row v of the gather is the int8 layer applied to unit vectors: W8A16 with
    x = e_k gives y[k, v] = fp16(scale[v, k/128] * code[v, k]) (one nonzero term)."""
    rng = np.random.default_rng(22)
    V, D = 9, 384
    codes = rng.integers(-127, 128, (V, D)).astype(np.int8)
    scales = rng.uniform(-0.05, 0.05, (V, D // 128)).astype(np.float16)
    eye = np.eye(D, dtype=np.float16)
    y = oracle.w8a16(eye, codes, scales)                    # [D, V]
    ids = np.arange(V)
    emb = oracle.embed_w8(ids, codes, scales)               # [V, D]
    # equal as numbers (exactly; the GEMM's sum turns a -0 product into +0)
    assert np.array_equal(emb.astype(np.float64), y.T.astype(np.float64))


def test_embed_w8_group_boundary_and_bad_id():
    """Feature 127 takes group 0's scale and 128 group 1's; an id outside [0, V) is rejected."""
    codes = np.ones((2, 256), np.int8)
    scales = np.array([[0.5, 0.25], [1.0, 2.0]], np.float16)
    out = oracle.embed_w8(np.array([1, 0]), codes, scales)
    assert out[0, 127] == 1.0 and out[0, 128] == 2.0 and out[1, 127] == 0.5 and out[1, 128] == 0.25
    with pytest.raises(ValueError):
        oracle.embed_w8(np.array([2]), codes, scales)


def test_topk_matches_brute_force_with_ties():
    """The sampler's top-k ("In full" item 6): largest first, ties to the smaller index;
    values drawn from a small set so ties are everywhere, +0 and -0 compare equal."""
    rng = np.random.default_rng(23)
    M, N, k = 5, 400, 37
    pool = np.array([-3.5, -0.0, 0.0, 0.125, 1.0, 1.0009765625, 7.0, 65504.0, -65504.0], np.float16)
    logits = pool[rng.integers(0, len(pool), (M, N))]
    vals, idx = oracle.topk(logits, k)
    for m in range(M):
        want = _brute.topk(logits[m], k)
        assert list(idx[m]) == want
        assert np.array_equal(vals[m].view(np.uint16), logits[m][want].view(np.uint16))


def test_topk_closed_forms():
    """k = N is a full stable sort; an all-equal row gives indices 0..k-1."""
    x = np.array([[2.0, -1.0, 2.0, 0.5]], np.float16)
    _, idx = oracle.topk(x, 4)
    assert list(idx[0]) == [0, 2, 3, 1]
    _, idx = oracle.topk(np.full((2, 50), 3.0, np.float16), 8)
    assert (idx == np.arange(8)).all()


# ---- int8-QK prefill attention (the page's paragraph "int8-QK prefill attention") ----

def test_attn_row_quantizer_is_the_activation_quantizer():
    """Q and smoothed K are quantized with the activation quantizer's arithmetic: on fp16
    rows (including a zero row and exact ties) the attention oracle's row quantizer and the
    C quantizer agree bit for bit."""
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((9, 96)) * 3).astype(np.float16)
    x[3] = 0
    x[4, :] = 0
    x[4, 0], x[4, 1], x[4, 2] = 127.0, 0.5, -1.5          # s = 1: halves round to even
    q1, s1 = oracle.quant_rows_f32(x.astype(np.float32))
    q2, s2 = oracle.quant_act_int8(x)
    assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    assert q1[4, 1] == 0 and q1[4, 2] == -2


def test_attn_row_quantizer_divides():
    """Rows built where a reciprocal multiply would give another code than the IEEE divide
    (elements x with rne(x * (1/s)) != rne(x / s) for their row's scale): the attention
    oracle's row quantizer matches the C quantizer bit for bit on them."""
    allv = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    pos = np.sort(allv[np.isfinite(allv) & (allv > 0)].astype(np.float32))
    rows = []
    for a in pos[(pos > 0.05) & (pos < 60)][::7]:
        xs = pos[pos <= a]
        s = np.float32(a / np.float32(127.0))
        odd = xs[np.rint(xs / s) != np.rint(xs * (np.float32(1.0) / s))]
        if len(odd):
            row = np.zeros(32, np.float32)
            row[0] = a
            row[1:1 + min(31, len(odd))] = odd[:31]
            rows.append(row)
        if len(rows) == 12:
            break
    x = np.array(rows, np.float32).astype(np.float16)
    q1, s1 = oracle.quant_rows_f32(x.astype(np.float32))
    q2, s2 = oracle.quant_act_int8(x)
    assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


def test_attn_two_keys_closed_form():
    """Two keys, d = 4: codes and scales come out exact (amax = 127 * 2^-6), so the score
    gap is 2 * 127^2 * 2^-6 * 2^-6 / sqrt(4) and the second query's output is the logistic
    mix of the two values; the first query sees only the first key (causal)."""
    a = 127.0 / 64.0                                       # exact in fp16
    k = np.zeros((2, 1, 4), np.float16)
    k[0, 0, 0], k[1, 0, 0] = -a, a                         # channel mean 0: smoothing is a no-op
    q = np.zeros((2, 1, 4), np.float16)
    q[0, 0, 1] = 1.0
    q[1, 0, 0] = a
    v = np.array([[[1.0, -2.0, 0.5, 3.0]], [[-1.0, 4.0, 0.25, 0.0]]], np.float16)
    o = oracle.attn_int8qk(q, k, v, out_f64=True)
    gap = 2 * 127 * 127 * 2.0 ** -12 / 2.0
    p1 = 1.0 / (1.0 + np.exp(-gap))
    want = (1 - p1) * v[0, 0].astype(np.float64) + p1 * v[1, 0].astype(np.float64)
    assert np.array_equal(o[0, 0], v[0, 0].astype(np.float64))
    assert np.allclose(o[1, 0], want, rtol=1e-13, atol=1e-15)


def test_attn_channel_offsets_are_invisible():
    """Smoothing removes any per-channel offset of K: with integer keys, integer offsets and
    S a power of two every step is exact, so the outputs are bit-identical (an oracle that
    skipped the smoothing, or averaged over channels, would differ)."""
    rng = np.random.default_rng(42)
    S, T, Hq, Hkv, d = 16, 8, 4, 2, 32
    k = rng.integers(-8, 9, (S, Hkv, d)).astype(np.float16)
    off = rng.integers(-100, 101, (1, Hkv, d)).astype(np.float16)
    q = rng.standard_normal((T, Hq, d)).astype(np.float16)
    v = rng.standard_normal((S, Hkv, d)).astype(np.float16)
    o1 = oracle.attn_int8qk(q, k, v)
    o2 = oracle.attn_int8qk(q, (k + off).astype(np.float16), v)
    assert np.array_equal(o1.view(np.uint16), o2.view(np.uint16))
    o3 = oracle.attn_int8qk(q, (k * 3).astype(np.float16), v)   # not an offset: must differ
    assert not np.array_equal(o1.view(np.uint16), o3.view(np.uint16))


def test_attn_causal_mask_and_grouped_heads():
    """One-hot value rows tagged with their KV head: query 0 returns value 0 exactly, query 1
    carries no weight on key 2 however large its score, query 2 puts most of it there; query
    head h reads KV head h // 2 (the tag comes back exactly)."""
    S, T, Hq, Hkv, d = 3, 3, 4, 2, 8
    k = np.zeros((S, Hkv, d), np.float16)
    k[2, :, 0] = 60.0
    q = np.zeros((T, Hq, d), np.float16)
    q[:, :, 0] = 2.0
    v = np.zeros((S, Hkv, d), np.float16)
    for j in range(S):
        v[j, :, j] = 1.0
    for g in range(Hkv):
        v[:, g, 7] = g + 1
    o = oracle.attn_int8qk(q, k, v, out_f64=True)
    for h in range(Hq):
        assert np.array_equal(o[0, h], v[0, h // 2].astype(np.float64))
        assert o[1, h, 2] == 0.0 and abs(o[1, h, 0] + o[1, h, 1] - 1.0) < 1e-15
        assert o[2, h, 2] > 0.99
        assert np.allclose(o[:, h, 7], h // 2 + 1, rtol=0, atol=1e-12)


def test_attn_uniform_when_keys_equal():
    """Equal keys smooth to zero (scale 0, codes 0): every visible key gets the same
    weight, so query i returns the mean of values 0 .. S - T + i."""
    rng = np.random.default_rng(43)
    S, T, H, d = 12, 5, 2, 16
    k = np.repeat(rng.standard_normal((1, H, d)).astype(np.float16), S, axis=0)
    q = rng.standard_normal((T, H, d)).astype(np.float16)
    v = rng.standard_normal((S, H, d)).astype(np.float16)
    o = oracle.attn_int8qk(q, k, v, out_f64=True)
    for i in range(T):
        n = S - T + i + 1
        assert np.allclose(o[i], v[:n].astype(np.float64).mean(axis=0), rtol=0, atol=1e-13)
