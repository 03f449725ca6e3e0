"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs.

Bars: activation codes and scales bit-exact; packed bytes bit-exact against the
layout the header documents; GEMM outputs within
max|y - y_ref| / max|y_ref| <= 5e-3 (fp16 outputs); repeated calls bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = 5e-3


@pytest.fixture(scope="module")
def q():
    import __graft_entry__
    __graft_entry__.build()
    import int8_weight_quantized_int4_gb300 as q
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return q


DEV = torch.device("cuda:0")


def nerr(y, ref):
    y = (y.float().cpu().numpy() if isinstance(y, torch.Tensor) else y).astype(np.float64)
    ref = np.asarray(ref).astype(np.float64)
    assert np.isfinite(y).all()
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-30))


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy() if isinstance(t, torch.Tensor) else t.view(np.int16)


# --------------------------------------------------------------- quantizer --

def _special_rows(x):
    x = x.clone()
    K = x.shape[1]
    if x.shape[0] >= 4:
        x[0] = 0
        x[1] = 0
        x[1, K // 3] = -7.25
        x[2] = ((torch.arange(K) % 17) - 8).to(torch.float16) * 2 ** -20     # subnormals
        x[3, :8] = torch.tensor([127, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5], dtype=torch.float16)
        x[3, 8:] = 0
    return x


@pytest.mark.parametrize("M,K", [(1, 5120), (4, 5120), (16, 5120), (64, 5120), (64, 17408),
                                 (7, 136), (5, 8), (33, 24576 + 64),
                                 # the narrow form (up to 8 tokens, from 256) on rows it re-reads
                                 (3, 17408), (256, 9216)])
def test_quant_act_bitexact(q, M, K):
    x = synth.activations(M, K, synth.generator(100 + M + K), outlier_frac=0.01)
    x = _special_rows(x)
    xq, xs = q.quant_act_int8(x.to(DEV))
    oq, os_ = oracle.quant_act_int8(x)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), oq)


@pytest.mark.parametrize("codes16", [False, True])
def test_quant_act_near_ties(q, codes16):
    """Every quotient x / s within a few 2^-12 of a half-integer, on 64 rows of 5120 with
    scales that are not powers of two: the quantizer's reciprocal product leaves most of
    these to its IEEE-divide branch (a group of eight holding one near-tie is redone).
    Codes and scales bit-exact against the oracle; the fp16-code output (W4A8 from fp16,
    read through identity weights) carries the same codes."""
    M, K = 64, 5120
    rng = np.random.default_rng(11)
    x = np.zeros((M, K), np.float16)
    for m in range(M):
        amax = float(np.float16(rng.uniform(0.01, 200.0)))
        s = np.float64(amax) / 127.0
        n = rng.integers(-127, 127, K)
        delta = rng.integers(-3, 4, K) * 2.0 ** -12
        x[m] = ((n + 0.5 + delta) * s).astype(np.float16)
        x[m, rng.integers(0, K)] = np.float16(amax)
    oq, os_ = oracle.quant_act_int8(x)
    xd = torch.from_numpy(x).to(DEV)
    if not codes16:
        xq, xs = q.quant_act_int8(xd)
        assert np.array_equal(xs.cpu().numpy().view(np.uint32), os_.view(np.uint32))
        assert np.array_equal(xq.cpu().numpy(), oq)
        return
    # through the fused entry at 64 tokens (quantizer with fp16 codes, then the GEMM): with
    # identity weights y[m, n] = fp16(s_m * q[m, n]) for n < N
    N = 1280
    codes = torch.zeros((N, K), dtype=torch.int8)
    codes[torch.arange(N), torch.arange(N)] = 1
    scales = torch.ones((N, K // 128), dtype=torch.float16)
    packed = q.qpack_w4(codes.to(DEV), scales.to(DEV))
    y = q.qgemm_w4a8_fused(xd, packed, N, K)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    expect = (oq[:, :N].astype(np.float32) * os_[:, None].astype(np.float32)).astype(np.float16)
    assert np.array_equal(bits(y), expect.view(np.int16))


def test_quant_act_prefill_size(q):
    x = synth.activations(8192, 5120, synth.generator(4))
    xq, xs = q.quant_act_int8(x.to(DEV))
    oq, os_ = oracle.quant_act_int8(x)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), oq)


# ----------------------------------------------------------------- packing --

def np_pack_w4(codes, scales):
    """The documented W4 layout, written independently in numpy: vector (b, h, c, i) of
    chunk (t, g) at position ((b*2 + h)*4 + c)*8 + (i ^ 2c); word w holds rows R = 16b + i
    and R + 8 at k0 = 16(4h + w) + 2c and k0 + 1, k0 + 8, k0 + 9 (nibble order below)."""
    u = ((codes.numpy().astype(np.int64) + 8) & 15).astype(np.uint32)
    N, K = u.shape
    T, G = N // 128, K // 128
    # u6[t, b, up, i, g, h, w, kk]: row 128t + 16b + 8up + i, k = 128g + 64h + 16w + kk
    u6 = u.reshape(T, 8, 2, 8, G, 2, 4, 16)
    words = np.zeros((T, G, 8, 2, 4, 8, 4), np.uint32)                # t g b h c i w
    for c in range(4):
        k0 = 2 * c
        # (up, k offset) of nibble p = 0..7
        sel = [(0, k0), (0, k0 + 8), (1, k0), (1, k0 + 8), (0, k0 + 1), (0, k0 + 9), (1, k0 + 1), (1, k0 + 9)]
        acc = np.zeros((T, 8, 8, G, 2, 4), np.uint32)                # t b i g h w
        for p, (up, kk) in enumerate(sel):
            acc |= u6[:, :, up, :, :, :, :, kk] << np.uint32(4 * p)
        perm = np.arange(8) ^ (2 * c)                                  # position of row i
        words[:, :, :, :, c, perm, :] = acc.transpose(0, 3, 1, 4, 2, 5)   # t g b h i w
    out = np.zeros((T, G, 8448), np.uint8)
    out[:, :, :8192] = words.reshape(T, G, -1).view(np.uint8).reshape(T, G, 8192)
    sc = scales.numpy().view(np.uint16).reshape(T, 8, 2, 8, G)         # t b up i g
    pairs = sc.transpose(0, 4, 1, 3, 2)                               # t g b i up
    out[:, :, 8192:] = np.ascontiguousarray(pairs).view(np.uint8).reshape(T, G, 256)
    return out.reshape(-1)


def np_pack_w8(codes, scales):
    c = codes.numpy().view(np.uint8) ^ 0x80
    N, K = c.shape
    T, G = N // 128, K // 128
    b = c.reshape(T, 128, G, 8, 16).transpose(0, 2, 3, 1, 4)          # t g j r b
    out = np.zeros((T, G, 16640), np.uint8)
    out[:, :, :16384] = b.reshape(T, G, 16384)
    s = scales.numpy().view(np.uint16).reshape(T, 128, G).transpose(0, 2, 1)
    out[:, :, 16384:] = np.ascontiguousarray(s).view(np.uint8).reshape(T, G, 256)
    return out.reshape(-1)


def test_pack_w4_layout_bitexact(q):
    p = synth.make_problem(1, 384, 640, seed=201)
    pk = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    assert pk.numel() == q.qpack_w4_bytes(384, 640)
    assert np.array_equal(pk.cpu().numpy(), np_pack_w4(p.codes, p.scales))
    assert q.device_error() == 0


def test_pack_w8_layout_bitexact(q):
    p = synth.make_problem(1, 256, 384, seed=202, bits=8, code_range=(-128, 127))
    pk = q.qpack_w8(p.codes.to(DEV), p.scales.to(DEV))
    assert np.array_equal(pk.cpu().numpy(), np_pack_w8(p.codes, p.scales))


def test_pack_w4_flags_out_of_range_codes(q):
    p = synth.make_problem(1, 128, 128, seed=203)
    bad = p.codes.clone()
    bad[5, 7] = 9
    q.qpack_w4(bad.to(DEV), p.scales.to(DEV))
    assert q.device_error() == q.QW_ERR_BAD_CODES
    assert q.device_error() == 0


# ------------------------------------------------------------------- GEMMs --

def run_modes(q, p, modes=("w4a16", "w4a8"), cols=None, rows=None):
    """Run the GPU path for each mode and compare with the oracle (optionally on a
    sample of output columns / token rows).  Returns {mode: normalized error}."""
    out = {}
    xd = p.x.to(DEV)
    cd, sd = p.codes.to(DEV), p.scales.to(DEV)
    cs = p.codes if cols is None else p.codes[cols]
    ss = p.scales if cols is None else p.scales[cols]
    rsel = slice(None) if rows is None else rows.numpy()
    if p.bits == 4:
        packed = q.qpack_w4(cd, sd)
    else:
        packed = q.qpack_w8(cd, sd)
    for mode in modes:
        if mode == "w4a16":
            y = q.qgemm_w4a16(xd, packed, p.N, p.K)
            ref = oracle.w4a16(p.x.numpy()[rsel], cs, ss)
        elif mode == "w8a16":
            y = q.qgemm_w8a16(xd, packed, p.N, p.K)
            ref = oracle.w8a16(p.x.numpy()[rsel], cs, ss)
        else:
            xq, xs = q.quant_act_int8(xd)
            oq, os_ = oracle.quant_act_int8(p.x.numpy()[rsel])
            assert np.array_equal(xq.cpu().numpy()[rsel], oq)
            y = q.qgemm_w4a8(xq, xs, packed, p.N, p.K)
            ref = oracle.w4a8(oq, os_, cs, ss)
        yc = y.cpu().numpy()[rsel]
        if cols is not None:
            yc = yc[:, cols.numpy()]
        out[mode] = nerr(yc, ref)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    return out


def test_tiny_config_all_modes(q):
    p = synth.tiny_w4a16()
    e = run_modes(q, p, ("w4a16", "w4a8"))
    p8 = synth.make_problem(4, 512, 256, seed=0, bits=8, scale_lo=0.001, scale_hi=0.01)
    e.update(run_modes(q, p8, ("w8a16",)))
    assert max(e.values()) <= TOL, e


def test_residue_sweep_all_M(q):
    """Every M from 1 to 130 (all residues of the 16/32/64/128 token tiles)."""
    base = synth.make_problem(130, 256, 384, seed=301, outlier_frac=0.02)
    packed = q.qpack_w4(base.codes.to(DEV), base.scales.to(DEV))
    ref_all = oracle.w4a16(base.x, base.codes, base.scales)
    xd = base.x.to(DEV)
    worst = 0.0
    for M in range(1, 131):
        y = q.qgemm_w4a16(xd[:M].contiguous(), packed, 256, 384)
        worst = max(worst, nerr(y, ref_all[:M]))
    assert worst <= TOL, worst
    assert q.device_error() == 0


@pytest.mark.parametrize("M", [1, 3, 17, 64, 100, 129, 300])
def test_w4a8_and_w8a16_ragged(q, M):
    p = synth.make_problem(M, 384, 512, seed=400 + M, outlier_frac=0.01)
    e = run_modes(q, p, ("w4a16", "w4a8"))
    p8 = synth.make_problem(M, 256, 384, seed=500 + M, bits=8, scale_lo=0.001, scale_hi=0.01)
    e.update(run_modes(q, p8, ("w8a16",)))
    assert max(e.values()) <= TOL, e


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_projection_5120(q, M):
    """Decode/verify projection K=N=5120 with 1% outlier channels, both modes, all outputs."""
    e = run_modes(q, synth.projection(M))
    assert max(e.values()) <= TOL, e


def test_projection_512_tokens(q):
    p = synth.projection(512)
    cols = torch.randperm(5120, generator=synth.generator(9))[:512].sort().values
    e = run_modes(q, p, cols=cols)
    assert max(e.values()) <= TOL, e


def test_ffn_pair_m64_w4a8(q):
    cols = torch.randperm(34816, generator=synth.generator(10))[:768].sort().values
    e_up = run_modes(q, synth.ffn_up(64), ("w4a8", "w4a16"), cols=cols)
    e_dn = run_modes(q, synth.ffn_down(64), ("w4a8", "w4a16"))
    assert max(e_up.values()) <= TOL and max(e_dn.values()) <= TOL, (e_up, e_dn)


@pytest.mark.parametrize("M,N,K", [(1, 5120, 5120), (3, 7296, 1152), (8, 2048, 640), (9, 5120, 2944),
                                   (16, 256, 128), (16, 4864, 17408), (5, 384, 8192), (2, 4096, 3072)])
def test_row_block_kernel(q, M, N, K):
    """Decode batches on layers of at most 3 x SMs 16-row blocks run on the row-block
    kernel: row blocks straddling 128-row tiles, K not a multiple of the 8-group stage
    (ragged last stage), fewer row blocks than SMs, one and two tiles of 8 tokens.  Every
    output (or a column sample of the widest) against the oracle in both modes, W4A8 from
    fp16 bit-identical to the two-step path, repeated calls bit-identical."""
    p = synth.make_problem(M, N, K, seed=5100 + M + N // 128 + K // 128, outlier_frac=0.01)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    pl = q.plan(q.MODE_W4A16, M, N, K, sms)
    if N // 16 > 3 * sms:
        pytest.skip("more row blocks than this device's row-block plans take")
    assert pl.decode_row_blocks > 0 and pl.stream_k == 0, (pl.decode_row_blocks, pl.decode_teams)
    cols = None if N * K <= 5120 * 5120 else torch.arange(0, N, 3)
    e = run_modes(q, p, ("w4a16", "w4a8"), cols=cols)
    assert max(e.values()) <= TOL, e
    xd = p.x.to(DEV)
    packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    y1 = q.qgemm_w4a16(xd, packed, N, K)
    y2 = q.qgemm_w4a16(xd, packed, N, K)
    xq, xs = q.quant_act_int8(xd)
    z1 = q.qgemm_w4a8(xq, xs, packed, N, K)
    z2 = q.qgemm_w4a8_fused(xd, packed, N, K)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    assert np.array_equal(bits(y1), bits(y2)) and np.array_equal(bits(z1), bits(z2))


@pytest.mark.parametrize("M", [1, 5, 16])
def test_decode_long_launch_two_ctas_per_sm(q, M):
    """A decode-sized batch over enough chunks that the schedule runs two CTAs per SM
    (more than 256 CTAs): every output against the oracle."""
    p = synth.make_problem(M, 16384, 5120, seed=470 + M, outlier_frac=0.01)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    pl = q.plan(q.MODE_W4A16, M, p.N, p.K, sms)
    assert pl.decode_teams > 0 and pl.grid > sms, (pl.grid, pl.decode_teams)
    e = run_modes(q, p, ("w4a16", "w4a8"))
    assert max(e.values()) <= TOL, e


@pytest.mark.slow
def test_prefill_8192_sampled(q):
    p = synth.prefill(8192)
    cols = torch.randperm(34816, generator=synth.generator(11))[:384].sort().values
    rows = torch.randperm(8192, generator=synth.generator(12))[:192].sort().values
    e = run_modes(q, p, ("w4a16", "w4a8"), cols=cols, rows=rows)
    assert max(e.values()) <= TOL, e


@pytest.mark.slow
@pytest.mark.parametrize("M", [1, 8, 16, 64])
def test_lm_head_w8a16(q, M):
    p = _lm_head(M)
    cols = torch.randperm(248320, generator=synth.generator(13))[:1024].sort().values
    # include the first and last row tiles
    cols = torch.cat([torch.arange(0, 64), cols, torch.arange(248320 - 64, 248320)]).unique()
    e = run_modes(q, p, ("w8a16",), cols=cols)
    assert e["w8a16"] <= TOL, e


_LM = {}


def _lm_head(M):
    if "p" not in _LM:
        _LM["p"] = synth.lm_head(64)
    p = _LM["p"]
    return synth.Problem(M, p.N, p.K, p.codes, p.scales, p.x[:M].contiguous(), 8)


# ----------------------------------------------------- determinism, invariants --

def test_repeated_calls_bit_identical(q):
    p = synth.projection(16)                   # a stream-K shape
    packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    xd = p.x.to(DEV)
    ys = [q.qgemm_w4a16(xd, packed, p.N, p.K).cpu() for _ in range(10)]
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


def test_invariant_b_w4a8_matches_w4a16_on_int8_exact_activations(q):
    gen = synth.generator(601)
    M, N, K = 24, 1024, 1280
    x = synth.int8_exact_activations(M, K, gen)
    codes = synth.codes_int4(N, K, gen)
    scales = synth.signed_scales(N, K // 128, gen, 0.002, 0.02)
    packed = q.qpack_w4(codes.to(DEV), scales.to(DEV))
    xd = x.to(DEV)
    y16 = q.qgemm_w4a16(xd, packed, N, K)
    xq, xs = q.quant_act_int8(xd)
    y8 = q.qgemm_w4a8(xq, xs, packed, N, K)
    ref = oracle.w4a16(x, codes, scales)
    assert nerr(y16, ref) <= TOL and nerr(y8, ref) <= TOL
    # power-of-two token scales commute with every rounding: identical bits
    assert torch.equal(y16.cpu().view(torch.int16), y8.cpu().view(torch.int16))


def test_signed_scales_sign_fold_equivalence(q):
    """(q, s) and (-q, -s) give bit-identical results (codes in [-7, 7]); all-negative
    scales match the oracle -- the unsigned-scale failure mode would break both."""
    p = synth.make_problem(16, 512, 768, seed=701, code_range=(-7, 7))
    neg = synth.make_problem(16, 512, 768, seed=701, code_range=(-7, 7))
    neg.scales = -neg.scales.abs()
    e = run_modes(q, neg, ("w4a16", "w4a8"))
    assert max(e.values()) <= TOL, e
    pa = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    pb = q.qpack_w4((-p.codes).to(DEV), (-p.scales).to(DEV))
    xd = p.x.to(DEV)
    ya = q.qgemm_w4a16(xd, pa, p.N, p.K)
    yb = q.qgemm_w4a16(xd, pb, p.N, p.K)
    assert torch.equal(ya.cpu().view(torch.int16), yb.cpu().view(torch.int16))


# ------------------------------------------------ W4A8 with the fused quantizer --

@pytest.mark.parametrize("M,N,K", [(1, 5120, 5120), (2, 640, 5120), (3, 384, 1280), (4, 5120, 5120),
                                   (7, 256, 3072), (16, 640, 640), (5, 640, 5120), (16, 5120, 5120),
                                   (17, 640, 640), (64, 640, 1024), (8, 27648, 5120), (48, 1280, 2048),
                                   (200, 1280, 2048)])
def test_w4a8_fused_bit_identical_to_two_step(q, M, N, K):
    """qgemm_w4a8_fused(x) equals qgemm_w4a8(quant_act_int8(x)) bit for bit -- in one
    row-block kernel that quantizes per token itself (M*K*2 <= 48 KB on a layer of few
    rows), or through the quantizer's fp16 codes where qgemm_w4a8 widens int8 ones
    (decode kernels at 1..16 tokens, a long two-CTAs-per-SM decode launch, tensor-core
    tiles of 32, 64 and 256) -- and meets the tolerance against the oracle."""
    p = synth.make_problem(M, N, K, seed=11 + M, outlier_frac=0.01)
    x = _special_rows(p.x) if M >= 4 else p.x
    xd = x.to(DEV)
    packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    xq, xs = q.quant_act_int8(xd)
    y2 = q.qgemm_w4a8(xq, xs, packed, N, K)
    y1 = q.qgemm_w4a8_fused(xd, packed, N, K)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    pl = q.plan(q.MODE_W4A8_FUSED, M, N, K, torch.cuda.get_device_properties(DEV).multi_processor_count)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    rb = M <= 16 and N // 16 <= 3 * sms and (M > 8 or (N // 128) * (K // 128) < 32 * sms)
    assert pl.fused == (1 if (rb and M <= 2 and M * K * 2 <= 48 * 1024) else 0)
    assert np.array_equal(bits(y1), bits(y2))
    oq, os_ = oracle.quant_act_int8(x.numpy())
    assert nerr(y1, oracle.w4a8(oq, os_, p.codes, p.scales)) <= TOL


@pytest.mark.parametrize("amaxes", [(100.0, 3.3), (0.0173, 55.5), (100.0, 3.3, 0.0173, 55.5)])
def test_w4a8_fused_quantizer_near_ties(q, amaxes):
    """Quotients x / s a few 2^-12 from half-integers, with scales that are not powers of
    two: through identity weights (y[m,n] = s_m * q[m,n]) every code shows in y, which must
    equal the two-step path bit for bit -- the codes of the row-block kernel's in-kernel
    quantizer (2 tokens: reciprocal product, IEEE quotient near ties) and of the standalone
    quantizer (4 tokens)."""
    M, N, K = len(amaxes), 1280, 1280
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert q.plan(q.MODE_W4A8_FUSED, M, N, K, sms).fused == (1 if M <= 2 else 0)
    rng = np.random.default_rng(5 + M)
    x = np.zeros((M, K), np.float16)
    for m, amax in enumerate(amaxes):
        s = np.float64(np.float16(amax)) / 127.0
        n = rng.integers(-127, 127, K)
        delta = rng.integers(-3, 4, K) * 2.0 ** -12
        x[m] = ((n + 0.5 + delta) * s).astype(np.float16)
        x[m, 0] = np.float16(amax)
    codes = torch.zeros((N, K), dtype=torch.int8)
    codes[torch.arange(N), torch.arange(N)] = 1
    scales = torch.ones((N, K // 128), dtype=torch.float16)
    packed = q.qpack_w4(codes.to(DEV), scales.to(DEV))
    xd = torch.from_numpy(x).to(DEV)
    xq, xs = q.quant_act_int8(xd)
    y2 = q.qgemm_w4a8(xq, xs, packed, N, K)
    y1 = q.qgemm_w4a8_fused(xd, packed, N, K)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    assert np.array_equal(bits(y1), bits(y2))
    oq, os_ = oracle.quant_act_int8(x)
    assert np.array_equal(xq.cpu().numpy(), oq)
    expect = (oq.astype(np.float64) * os_.astype(np.float64)[:, None]).astype(np.float16)
    assert nerr(y1, expect) <= 1e-3


def test_w4a8_fused_workspace_and_empty(q):
    """The fused entry leaves the workspace's zero region zero and accepts M = 0."""
    p = synth.projection(4)
    packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    zero = int(q.lib().qgemm_workspace_zero_bytes(q.MODE_W4A8_FUSED, 4, 5120, 5120))
    ws = q.Workspace(DEV)
    for _ in range(3):
        q.qgemm_w4a8_fused(p.x.to(DEV), packed, p.N, p.K, ws=ws)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    assert int(ws.buf[:zero].count_nonzero()) == 0
    y = q.qgemm_w4a8_fused(torch.empty((0, 5120), dtype=torch.float16, device=DEV), packed, p.N, p.K)
    assert tuple(y.shape) == (0, 5120)


@pytest.mark.slow
@pytest.mark.parametrize("M", [1, 16])
def test_lm_head_w4a16_sampled(q, M):
    """The int4 lm_head (W4A16 at N = 248,320) against the oracle on sampled columns."""
    p = synth.lm_head_int4(M)
    packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    y = q.qgemm_w4a16(p.x.to(DEV), packed, p.N, p.K)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    cols = np.concatenate([np.arange(0, p.N, 499), [p.N - 1]])
    ref = oracle.w4a16(p.x.numpy(), p.codes[cols], p.scales[cols])
    assert nerr(y.cpu().numpy()[:, cols], ref) <= TOL


# ------------------------------------------- embedding gather and top-k (next rows) --

@pytest.mark.parametrize("V,D,T", [(1024, 640, 300), (256, 5120, 64), (128, 128, 1)])
def test_embed_gather_w8_bitexact(q, V, D, T):
    """Dequant-on-gather from the qpack_w8 table equals the oracle bit for bit."""
    p = synth.make_problem(1, V, D, seed=31 + T, bits=8, scale_lo=0.001, scale_hi=0.01)
    packed = q.qpack_w8(p.codes.to(DEV), p.scales.to(DEV))
    ids = synth.token_ids(T, V, seed=32 + T)
    out = q.embed_gather_w8(ids.to(DEV), packed, V, D)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    ref = oracle.embed_w8(ids.numpy(), p.codes, p.scales)
    assert np.array_equal(bits(out), ref.view(np.int16))


def test_embed_gather_w8_bad_id(q):
    """An id outside [0, V) gives a zero row and QW_ERR_BAD_INDEX in the error word; the
    other rows are unaffected."""
    p = synth.make_problem(1, 256, 256, seed=33, bits=8)
    packed = q.qpack_w8(p.codes.to(DEV), p.scales.to(DEV))
    ids = torch.tensor([5, -1, 256, 7], dtype=torch.int32)
    out = q.embed_gather_w8(ids.to(DEV), packed, 256, 256)
    torch.cuda.synchronize()
    assert q.device_error() == q.QW_ERR_BAD_INDEX
    assert q.device_error() == 0
    o = out.cpu()
    assert int(o[1].abs().sum()) == 0 and int(o[2].abs().sum()) == 0
    ref = oracle.embed_w8(np.array([5, 7]), p.codes, p.scales)
    assert np.array_equal(bits(o[[0, 3]]), ref.view(np.int16))


@pytest.mark.parametrize("M,N,k", [(1, 248320, 64), (4, 248320, 8), (64, 32768, 64), (3, 4096, 1),
                                   (2, 2056, 17), (5, 8, 8), (7, 262144, 50)])
def test_topk_logits_match_oracle(q, M, N, k):
    """Top-k over logits: indices and values equal the oracle's (largest first, ties to
    the smaller index, -0 equal to +0) on tie-heavy synthetic logits."""
    x = synth.logits(M, N, seed=M * 7 + k)
    vals, idx = q.topk_logits(x.to(DEV), k)
    torch.cuda.synchronize()
    assert q.device_error() == 0
    ov, oi = oracle.topk(x.numpy(), k)
    assert np.array_equal(idx.cpu().numpy().astype(np.int64), oi)
    assert np.array_equal(bits(vals), ov.view(np.int16))


def test_topk_logits_constant_rows_and_repeat(q):
    """All-equal rows give indices 0..k-1; a second call on the same workspace agrees."""
    x = torch.full((3, 1024), 2.5, dtype=torch.float16)
    x[1] = -0.0
    for _ in range(2):
        vals, idx = q.topk_logits(x.to(DEV), 16)
        torch.cuda.synchronize()
        assert (idx.cpu() == torch.arange(16, dtype=torch.int32)).all()
        assert np.array_equal(bits(vals), x[:, :16].numpy().view(np.int16))


def test_workspace_contract(q):
    p = synth.projection(4)
    packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    need = q.workspace_bytes(q.MODE_W4A16, 4, 5120, 5120)
    zero = int(q.lib().qgemm_workspace_zero_bytes(q.MODE_W4A16, 4, 5120, 5120))
    assert need > 0 and 0 < zero <= need
    ws = q.Workspace(DEV)
    y = q.qgemm_w4a16(p.x.to(DEV), packed, p.N, p.K, ws=ws)
    torch.cuda.synchronize()
    assert int(ws.buf[:zero].count_nonzero()) == 0
    small = torch.zeros(need // 2 // 256 * 256, dtype=torch.uint8, device=DEV)
    import ctypes
    rc = q.lib().qgemm_w4a16(ctypes.c_void_p(p.x.to(DEV).data_ptr()), ctypes.c_void_p(packed.data_ptr()),
                             4, 5120, 5120, ctypes.c_void_p(y.data_ptr()),
                             ctypes.c_void_p(small.data_ptr()), small.numel(), None)
    assert rc == q.QW_ERR_WORKSPACE


def test_one_workspace_across_shapes(q):
    """A workspace zeroed once serves a sequence of calls of different shapes and modes
    (partials of one call must never land where another call keeps its counters)."""
    ws = q.Workspace(DEV)
    shapes = [(300, 1280, 1152), (64, 8192, 1024), (16, 256, 4096), (300, 1280, 1152), (64, 8192, 1024)]
    for i, (M, N, K) in enumerate(shapes):
        p = synth.make_problem(M, N, K, seed=900 + i, outlier_frac=0.01)
        packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
        xd = p.x.to(DEV)
        cols = np.arange(0, N, 7)
        y = q.qgemm_w4a16(xd, packed, N, K, ws=ws)
        assert nerr(y.cpu().numpy()[:, cols], oracle.w4a16(p.x, p.codes[cols], p.scales[cols])) <= TOL
        xq, xs = q.quant_act_int8(xd)
        y8 = q.qgemm_w4a8(xq, xs, packed, N, K, ws=ws)
        oq, os_ = oracle.quant_act_int8(p.x)
        assert nerr(y8.cpu().numpy()[:, cols], oracle.w4a8(oq, os_, p.codes[cols], p.scales[cols])) <= TOL
    zero = int(q.lib().qgemm_workspace_zero_bytes(q.MODE_W4A16, 4, 5120, 5120))
    torch.cuda.synchronize()
    assert int(ws.buf[:zero].count_nonzero()) == 0
    assert q.device_error() == 0


def test_empty_and_single_tile(q):
    p = synth.make_problem(1, 128, 128, seed=801)
    e = run_modes(q, p, ("w4a16", "w4a8"))
    assert max(e.values()) <= TOL
    packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    y = q.qgemm_w4a16(torch.empty((0, 128), dtype=torch.float16, device=DEV), packed, 128, 128)
    assert y.shape == (0, 128)
    assert q.device_error() == 0


def test_weights_immutable_option_back_to_back(q):
    """With QW_OPT_WEIGHTS_IMMUTABLE each GEMM streams its weights before the previous
    kernel on the stream has finished; results of a chain of back-to-back layers
    (with the int8 quantizer in between) must still match the oracle."""
    q.set_weights_immutable(True)
    try:
        layers = [synth.make_problem(16, 1024, 1280, seed=950 + i, outlier_frac=0.01) for i in range(4)]
        packed = [q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV)) for p in layers]
        torch.cuda.synchronize()                     # packing done before the option matters
        ys, ys8 = [], []
        for p, pk in zip(layers, packed):
            xd = p.x.to(DEV)
            ys.append(q.qgemm_w4a16(xd, pk, p.N, p.K))
            xq, xs = q.quant_act_int8(xd)
            ys8.append(q.qgemm_w4a8(xq, xs, pk, p.N, p.K))
        torch.cuda.synchronize()
        for p, y, y8 in zip(layers, ys, ys8):
            assert nerr(y, oracle.w4a16(p.x, p.codes, p.scales)) <= TOL
            oq, os_ = oracle.quant_act_int8(p.x)
            assert nerr(y8, oracle.w4a8(oq, os_, p.codes, p.scales)) <= TOL
        assert q.device_error() == 0
    finally:
        q.set_weights_immutable(False)


@pytest.mark.gpu
def test_binding_rejects_short_or_misshapen_buffers(q):
    """The binding checks every caller-supplied buffer against the shapes before anything
    is launched: a packed table smaller than N x K needs, outputs of the wrong shape."""
    p = synth.make_problem(2, 256, 256, seed=77)
    packed = q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV))
    x = p.x.to(DEV)
    with pytest.raises(ValueError):
        q.qgemm_w4a16(x, packed, 512, 256)                  # N = 512 needs twice the bytes
    with pytest.raises(ValueError):
        q.qgemm_w8a16(x, packed, 256, 256)                  # an int8 table needs more
    with pytest.raises(ValueError):
        q.qgemm_w4a16(x, packed[:100], 256, 256)
    with pytest.raises(ValueError):
        q.quant_act_int8(x, xq=torch.empty((2, 128), dtype=torch.int8, device=DEV))
    with pytest.raises(ValueError):
        q.qpack_w4(p.codes.to(DEV), p.scales.to(DEV), out=torch.empty(64, dtype=torch.uint8, device=DEV))
    ids = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError):
        q.embed_gather_w8(ids, packed, 256, 256)            # a W4 buffer is too small for W8
    torch.cuda.synchronize()
    assert q.device_error() == 0
    y = q.qgemm_w4a16(x, packed, 256, 256)                  # the right sizes still run
    assert y.shape == (2, 256)


@pytest.mark.parametrize("imm", [False, True])
@pytest.mark.parametrize("M,N,K", [(64, 5120, 5120), (64, 34816, 5120), (256, 34816, 5120), (128, 5120, 17408)])
def test_tc_warp_issue_repeat_bitwise(q, imm, M, N, K):
    """The tcgen05 GEMM on token tiles of 64 and more issues from whole warps (warp-voted
    waits, one elected lane issuing every MMA, commit and copy): repeated launches, with and
    without the weights-immutable overlap, give bit-identical results and no device error,
    and the first matches the oracle."""
    gen = synth.generator(900 + M + N // 128)
    codes = torch.randint(-8, 8, (N, K), generator=gen, dtype=torch.int8)
    scales = ((torch.rand((N, K // 128), generator=gen) - 0.3) * 0.02).to(torch.float16)
    x = (torch.randn((M, K), generator=gen) * 0.5).to(torch.float16)
    packed = q.qpack_w4(codes.to(DEV), scales.to(DEV))
    xd = x.to(DEV)
    ws = q.Workspace(DEV)
    y = torch.empty((M, N), dtype=torch.float16, device=DEV)
    q.set_weights_immutable(imm)
    try:
        q.qgemm_w4a16(xd, packed, N, K, y=y, ws=ws)
        ref = y.clone()
        for _ in range(30):
            q.qgemm_w4a16(xd, packed, N, K, y=y, ws=ws)
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        torch.cuda.synchronize()
        assert q.device_error() == 0
    finally:
        q.set_weights_immutable(False)
    cols = np.arange(0, N, 97)
    expect = oracle.w4a16(x, codes.numpy()[cols], scales.numpy()[cols])
    assert nerr(ref.cpu()[:, cols], expect) <= TOL
