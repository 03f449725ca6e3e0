"""CPU tests of the C-ABI library: it loads, exports every declared symbol, checks
its arguments before touching a device, and its schedule (shared host/device
code) covers every chunk exactly once.  No compute call reaches a GPU here."""
import ctypes
import json
import os
import re

import pytest
import torch

import int8_weight_quantized_int4_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemm.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    from int8_weight_quantized_int4_gb300 import build
    build.build()


def declared_functions():
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 15, names
    L = ctypes.CDLL(q.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(q.SIGNATURES), set(names) ^ set(q.SIGNATURES)


def test_packed_sizes():
    assert q.qpack_w4_bytes(5120, 5120) == 13_516_800
    assert q.qpack_w4_bytes(34816, 5120) == 91_914_240
    assert q.qpack_w4_bytes(5120, 17408) == 45_957_120
    assert q.qpack_w8_bytes(248320, 5120) == 1_291_264_000
    assert q.qpack_w4_bytes(100, 128) == 0 and q.qpack_w8_bytes(128, 100) == 0
    assert q.qpack_w4_bytes(-128, 128) == 0


def test_lm_head_size_matches_pages():
    with open(os.path.join(ROOT, "tests", "golden", "lm_head_bytes.json")) as fh:
        g = json.load(fh)
    gb = q.qpack_w8_bytes(g["rows"], g["K"]) / 1e9
    lo, hi = g["accept_GB"]
    assert lo <= gb <= hi


FAKE = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced on this path
MIS = ctypes.c_void_p((1 << 20) + 2)     # misaligned


def test_argument_errors_before_device():
    L = q.lib()
    n = ctypes.c_void_p(0)
    assert L.qgemm_w4a16(FAKE, FAKE, 4, 512, 100, FAKE, n, 0, n) == q.QW_ERR_UNSUPPORTED_SHAPE
    assert L.qgemm_w4a16(FAKE, FAKE, 4, 500, 256, FAKE, n, 0, n) == q.QW_ERR_UNSUPPORTED_SHAPE
    assert L.qgemm_w4a16(FAKE, FAKE, -1, 512, 256, FAKE, n, 0, n) == q.QW_ERR_INVALID_ARG
    assert L.qgemm_w4a16(n, FAKE, 4, 512, 256, FAKE, n, 0, n) == q.QW_ERR_INVALID_ARG
    assert L.qgemm_w4a8(FAKE, n, FAKE, 4, 512, 256, FAKE, n, 0, n) == q.QW_ERR_INVALID_ARG
    assert L.qgemm_w8a16(MIS, FAKE, 4, 512, 256, FAKE, n, 0, n) == q.QW_ERR_ALIGNMENT
    assert L.qgemm_w4a16(FAKE, FAKE, 4, 512, 256, FAKE, MIS, 1 << 20, n) == q.QW_ERR_ALIGNMENT
    assert b"multiple of 128" in L.qw_last_error_string() or L.qw_last_error_string()
    # empty problems succeed without touching anything
    assert L.qgemm_w4a16(n, n, 0, 512, 256, n, n, 0, n) == q.QW_OK
    assert L.qgemm_w4a16(n, n, 4, 0, 256, n, n, 0, n) == q.QW_OK
    assert L.quant_act_int8(n, 0, 256, n, n, n) == q.QW_OK
    assert L.quant_act_int8(FAKE, 2, 12, FAKE, FAKE, n) == q.QW_ERR_UNSUPPORTED_SHAPE
    assert L.quant_act_int8(n, 2, 16, FAKE, FAKE, n) == q.QW_ERR_INVALID_ARG
    assert L.qpack_w4(n, FAKE, 128, 128, FAKE, n) == q.QW_ERR_INVALID_ARG
    assert L.qpack_w8(FAKE, FAKE, 128, 130, FAKE, n) == q.QW_ERR_UNSUPPORTED_SHAPE


def test_alignment_rules_match_header():
    """Each alignment the header states is checked on the host before any device access:
    one pointer at a time is moved off its boundary by the smallest step that breaks it."""
    L = q.lib()
    n = ctypes.c_void_p(0)
    B = 1 << 20

    def at(off):
        return ctypes.c_void_p(B + off)

    A = q.QW_ERR_ALIGNMENT
    # GEMMs: activations and packed weights 16 B, workspace 256 B, y 2 B, xs 4 B
    assert L.qgemm_w4a16(at(8), at(0), 4, 512, 256, at(0), at(0), B, n) == A
    assert L.qgemm_w4a16(at(0), at(8), 4, 512, 256, at(0), at(0), B, n) == A
    assert L.qgemm_w4a16(at(0), at(0), 4, 512, 256, at(1), at(0), B, n) == A
    assert L.qgemm_w4a16(at(0), at(0), 4, 512, 256, at(0), at(128), B, n) == A
    assert L.qgemm_w4a8(at(0), at(2), at(0), 4, 512, 256, at(0), at(0), B, n) == A
    assert L.qgemm_w4a8_fused(at(8), at(0), 4, 512, 256, at(0), at(0), B, n) == A
    # y at 2 bytes and xs at 4 bytes are accepted (past the checks: no device here)
    ok = (q.QW_OK, q.QW_ERR_ARCH, q.QW_ERR_WORKSPACE)
    assert L.qgemm_w4a8(at(0), at(4), at(0), 4, 512, 256, at(2), at(0), B, n) in ok
    # packing: codes and packed 16 B, scales 2 B
    assert L.qpack_w4(at(8), at(0), 128, 128, at(0), n) == A
    assert L.qpack_w4(at(0), at(1), 128, 128, at(0), n) == A
    assert L.qpack_w8(at(0), at(0), 128, 128, at(8), n) == A
    # quantizer: x 16 B, xq 8 B, xs 4 B
    assert L.quant_act_int8(at(8), 2, 16, at(0), at(0), n) == A
    assert L.quant_act_int8(at(0), 2, 16, at(4), at(0), n) == A
    assert L.quant_act_int8(at(0), 2, 16, at(0), at(2), n) == A
    # gather: ids 4 B, table and output 16 B; top-k: logits 16 B, vals 2 B, idx 4 B, ws 256 B
    assert L.embed_gather_w8(at(2), 4, at(0), 256, 256, at(0), n) == A
    assert L.embed_gather_w8(at(0), 4, at(0), 256, 256, at(8), n) == A
    assert L.topk_logits(at(0), 2, 256, 4, at(1), at(0), at(0), B, n) == A
    assert L.topk_logits(at(0), 2, 256, 4, at(0), at(2), at(0), B, n) == A
    assert L.topk_logits(at(0), 2, 256, 4, at(0), at(0), at(128), B, n) == A


def test_options_host_only():
    L = q.lib()
    assert L.qw_get_option(q.QW_OPT_WEIGHTS_IMMUTABLE) == 0
    assert L.qw_set_option(q.QW_OPT_WEIGHTS_IMMUTABLE, 1) == q.QW_OK
    assert L.qw_get_option(q.QW_OPT_WEIGHTS_IMMUTABLE) == 1
    assert L.qw_set_option(q.QW_OPT_WEIGHTS_IMMUTABLE, 0) == q.QW_OK
    assert L.qw_set_option(7, 1) == q.QW_ERR_INVALID_ARG
    assert L.qw_set_option(q.QW_OPT_WEIGHTS_IMMUTABLE, 2) == q.QW_ERR_INVALID_ARG
    assert L.qw_get_option(7) == q.QW_ERR_INVALID_ARG
    # the wait-limit test hook: microseconds, 0 .. the 4 s default
    assert L.qw_get_option(q.QW_OPT_WAIT_LIMIT_US) == q.DEFAULT_WAIT_LIMIT_US == 4_000_000
    assert L.qw_set_option(q.QW_OPT_WAIT_LIMIT_US, 0) == q.QW_OK
    assert L.qw_get_option(q.QW_OPT_WAIT_LIMIT_US) == 0
    assert L.qw_set_option(q.QW_OPT_WAIT_LIMIT_US, -1) == q.QW_ERR_INVALID_ARG
    assert L.qw_set_option(q.QW_OPT_WAIT_LIMIT_US, 4_000_001) == q.QW_ERR_INVALID_ARG
    q.set_wait_limit_us(None)
    assert L.qw_get_option(q.QW_OPT_WAIT_LIMIT_US) == 4_000_000


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_no_device_reports_arch():
    L = q.lib()
    n = ctypes.c_void_p(0)
    assert L.qgemm_w4a16(FAKE, FAKE, 4, 512, 256, FAKE, n, 0, n) == q.QW_ERR_ARCH
    assert L.quant_act_int8(FAKE, 2, 16, FAKE, FAKE, n) == q.QW_ERR_ARCH
    assert L.qgemm_workspace_bytes(0, 4, 512, 256) == 0


def test_lm_head_topk_argument_checks():
    """Host-side rules of qgemm_lm_head_topk, checked before any device work."""
    L = q.lib()
    n = ctypes.c_void_p(0)
    B = ctypes.c_size_t(1 << 30)

    def call(mode, M, N, K, k, vals=FAKE, idx=FAKE):
        return L.qgemm_lm_head_topk(mode, FAKE, FAKE, M, N, K, k, FAKE, vals, idx, FAKE, B, n)
    assert call(q.MODE_W4A8, 4, 1024, 256, 8) == q.QW_ERR_INVALID_ARG       # modes W4A16, W8A16 only
    assert call(q.MODE_W4A8_FUSED, 4, 1024, 256, 8) == q.QW_ERR_INVALID_ARG
    assert call(q.MODE_W4A16, 4, 1024, 256, 0) == q.QW_ERR_INVALID_ARG
    assert call(q.MODE_W4A16, 4, 1024, 256, 65) == q.QW_ERR_INVALID_ARG      # k <= 64
    assert call(q.MODE_W4A16, 4, 262144 + 128, 256, 8) == q.QW_ERR_UNSUPPORTED_SHAPE
    assert call(q.MODE_W4A16, 4, 1000, 256, 8) == q.QW_ERR_UNSUPPORTED_SHAPE  # N % 128
    assert call(q.MODE_W4A16, 0, 1024, 256, 8) == q.QW_OK                      # empty
    assert call(q.MODE_W4A16, 4, 1024, 256, 8, vals=n) == q.QW_ERR_INVALID_ARG
    assert call(q.MODE_W4A16, 4, 1024, 256, 8, idx=ctypes.c_void_p((1 << 20) + 2)) == q.QW_ERR_ALIGNMENT
    assert L.qgemm_lm_head_topk_workspace_bytes(q.MODE_W4A8, 4, 1024, 256, 8) == 0
    assert L.qgemm_lm_head_topk_workspace_bytes(q.MODE_W4A16, 4, 1024, 256, 65) == 0


SHAPES = [
    (0, 4, 512, 256, 152), (1, 1, 5120, 5120, 152), (0, 64, 5120, 5120, 152),
    (1, 64, 34816, 5120, 152), (1, 64, 5120, 17408, 152), (0, 8192, 34816, 5120, 152),
    (2, 64, 248320, 5120, 152), (2, 1, 248320, 5120, 148), (0, 130, 384, 640, 152),
    (0, 512, 5120, 5120, 152), (0, 3, 128, 128, 152), (1, 300, 1280, 1152, 7),
]


def _check_row_blocks(p, M, N, sms):
    """Row-block plan: the N / 16 row blocks split into consecutive ranges of 1..rb_max
    (balanced within one) over min(N / 16, sms) CTAs, no stream-K, no segments."""
    RB = N // 16
    assert M <= 16 and RB <= 3 * sms and p.stream_k == 0 and p.decode_teams == 0
    assert p.grid == min(RB, sms) and 1 <= p.decode_row_blocks <= 3
    assert p.decode_row_blocks == -(-RB // p.grid)
    # one ring of stages of 8 K groups (activations and weights), 2 to 6 deep, one CTA per SM
    assert p.act_block == 8 and p.act_stages == p.stages and 2 <= p.stages <= 6
    assert p.smem_bytes <= 232448
    nxt, sizes = 0, []
    for cta in range(p.grid):
        assert q.plan_segments(p, cta) == []
        b, e = q.plan_row_blocks(p, cta)
        assert b == nxt and e > b
        nxt = e
        sizes.append(e - b)
    assert nxt == RB and max(sizes) - min(sizes) <= 1 and max(sizes) == p.decode_row_blocks


@pytest.mark.parametrize("mode,M,N,K,sms", SHAPES)
def test_schedule_covers_every_chunk_once(mode, M, N, K, sms):
    p = q.plan(mode, M, N, K, sms)
    assert p.bn in (16, 32, 64, 128, 256) and p.bn >= min(M, 256)
    assert p.token_tiles == -(-M // p.bn) and p.row_tiles == N // 128 and p.groups == K // 128
    assert 1 <= p.grid <= sms and p.stages >= 2 and p.smem_bytes <= 232448
    if p.decode_row_blocks:
        _check_row_blocks(p, M, N, sms)
        return
    seen = {}
    slots = set()
    pieces = {}
    for cta in range(p.grid):
        segs = q.plan_segments(p, cta)
        assert segs, "every CTA gets work"
        for tile, g0, g1, slot in segs:
            assert 0 <= tile < p.tiles and 0 <= g0 < g1 <= p.groups
            for g in range(g0, g1):
                assert (tile, g) not in seen
                seen[(tile, g)] = cta
            whole = (g0 == 0 and g1 == p.groups)
            assert (slot < 0) == whole
            if slot >= 0:
                assert p.stream_k and slot not in slots and slot // 2 == cta
                slots.add(slot)
                pieces.setdefault(tile, []).append((g0, cta, slot))
    assert len(seen) == p.chunks
    # a cut tile's pieces come from consecutive CTAs, in K order
    for tile, ps in pieces.items():
        ps.sort()
        ctas = [c for _, c, _ in ps]
        assert ctas == list(range(ctas[0], ctas[0] + len(ctas)))
        assert len(ps) >= 2
    if p.stream_k:
        assert p.ws_bytes >= p.ws_zero_bytes >= p.tiles * 4
    load = {}
    for (tile, g), cta in seen.items():
        load[cta] = load.get(cta, 0) + 1
    aligned = p.stream_k and 3 * p.tiles <= p.grid and p.chunks <= 16 * p.grid
    if p.stream_k and not aligned:
        assert max(load.values()) - min(load.values()) <= 1
    if aligned:                                   # one piece per CTA: G/b or G/(b+1) groups
        b = p.grid // p.tiles
        assert max(load.values()) <= -(-p.groups // b) and min(load.values()) >= p.groups // (b + 1)


def test_schedule_row_blocks_for_decode_projections():
    """Decode batches (M <= 16, int4 weights) on a 5120-row layer: the row-block kernel,
    320 row blocks over 152 CTAs (2 or 3 each); a layer of more than 3 x 152 row blocks,
    or up to 8 tokens over at least 32 chunks per SM, keeps the tile-based decode kernel."""
    for mode in (0, 1, 3):
        for M in (1, 4, 8, 9, 16):
            for K in (5120, 17408):
                p = q.plan(mode, M, 5120, K, 152)
                if K == 17408 and M <= 8:              # 5440 chunks: 35.8 per SM
                    assert p.decode_row_blocks == 0 and p.decode_teams > 0 and p.grid == 304
                    continue
                assert p.decode_row_blocks == 3 and p.grid == 152
                _check_row_blocks(p, M, 5120, 152)
    assert q.plan(0, 1, 7296, 5120, 152).decode_row_blocks == 3
    p = q.plan(0, 1, 7424, 5120, 152)
    assert p.decode_row_blocks == 0 and p.decode_teams > 0
    assert q.plan(0, 1, 248320, 5120, 152).decode_row_blocks == 0
    assert q.plan(0, 17, 5120, 5120, 152).decode_row_blocks == 0        # the tcgen05 GEMM
    assert q.plan(2, 16, 5120, 5120, 152).decode_row_blocks == 0        # int8 weights
    p = q.plan(0, 2, 256, 1024, 152)                                      # fewer row blocks than SMs
    assert p.grid == 16 and p.decode_row_blocks == 1
    _check_row_blocks(p, 2, 256, 152)


def test_schedule_tile_aligned_split_for_short_launches():
    """Projection-sized stream-K launches (>= 3 CTAs per tile, <= 16 chunks per CTA) cut
    every tile into b or b+1 equal pieces, one piece per CTA, larger pieces first."""
    for mode, M in ((0, 32), (1, 64), (0, 64)):
        p = q.plan(mode, M, 5120, 5120, 152)
        assert p.stream_k == 1 and p.tiles == 40 and p.grid == 152
        pieces = {}
        for cta in range(p.grid):
            segs = q.plan_segments(p, cta)
            assert len(segs) == 1, "one segment per CTA"
            tile, g0, g1, slot = segs[0]
            pieces.setdefault(tile, []).append((cta, g1 - g0))
        counts = [len(pieces[t]) for t in range(p.tiles)]
        assert sorted(set(counts)) == [3, 4] and sum(counts) == p.grid
        assert counts == sorted(counts), "tiles with larger pieces come first"
        for t, ps in pieces.items():
            sizes = [n for _, n in ps]
            assert sum(sizes) == p.groups and max(sizes) - min(sizes) <= 1
            ctas = [c for c, _ in ps]
            assert ctas == list(range(ctas[0], ctas[0] + len(ctas))), "contributors are consecutive"


def test_schedule_long_launches_stay_balanced():
    """Longer stream-K launches keep the chunk-balanced split (within one chunk)."""
    p = q.plan(1, 64, 5120, 17408, 152)          # FFN down: 35.8 chunks per CTA
    sizes = [sum(g1 - g0 for _, g0, g1, _ in q.plan_segments(p, c)) for c in range(p.grid)]
    assert max(sizes) - min(sizes) <= 1


def test_schedule_whole_tiles_for_prefill():
    p = q.plan(0, 8192, 34816, 5120, 152)
    assert p.stream_k == 0 and p.bn == 256 and p.tiles == 32 * 272
    assert p.ws_bytes == p.ws_zero_bytes          # only the counter region


def test_counter_region_is_shared_by_every_plan():
    """Every plan puts its tile counters in the same leading region and nothing else
    there, so one workspace zeroed once serves calls of any shape."""
    zs = set()
    for mode, M, N, K, sms in SHAPES:
        p = q.plan(mode, M, N, K, sms if sms == 152 else 152)
        zs.add(p.ws_zero_bytes)
        if p.stream_k:
            assert p.tiles * 4 <= p.ws_zero_bytes
    assert len(zs) == 1


def test_w4a8_workspace_holds_widened_codes():
    p = q.plan(1, 8192, 34816, 5120, 152)
    assert p.ws_bytes >= 8192 * 5120 * 2


def _topk_expected_ws(M, N, k):
    """The slice plan restated: slices of 2048 or 4096 positions, at most 64, covering N;
    workspace = M counters (256-byte aligned) + M x slices x k 8-byte candidates."""
    slices = min(64, max(1, -(-N // 2048)))
    per = -(-N // slices)
    slice_len = -(-per // 2048) * 2048
    slices = -(-N // slice_len)
    assert slice_len <= 4096 and slices <= 64 and slices * slice_len >= N
    counters = -(-(M * 4) // 256) * 256
    return counters, counters + M * slices * k * 8


@pytest.mark.parametrize("M,N,k", [(1, 248320, 64), (64, 248320, 64), (3, 4096, 1), (2, 2056, 17),
                                   (5, 8, 8), (7, 262144, 50), (1, 131080, 64)])
def test_topk_workspace_sizes(M, N, k):
    L = q.lib()
    zero, total = _topk_expected_ws(M, N, k)
    assert L.topk_workspace_zero_bytes(M, N, k) == zero
    assert L.topk_workspace_bytes(M, N, k) == total


def test_topk_and_gather_argument_errors_before_device():
    L = q.lib()
    n = ctypes.c_void_p(0)
    # unsupported top-k shapes: k out of [1, 64], k > N, N not a multiple of 8, N too large
    for M, N, k in [(1, 256, 0), (1, 256, 65), (1, 16, 17), (1, 260, 4), (1, 262144 + 8, 4)]:
        assert L.topk_workspace_bytes(M, N, k) == 0
        assert L.topk_logits(FAKE, M, N, k, FAKE, FAKE, FAKE, 1 << 20, n) == q.QW_ERR_UNSUPPORTED_SHAPE
    assert L.topk_logits(FAKE, -1, 256, 4, FAKE, FAKE, FAKE, 1 << 20, n) == q.QW_ERR_INVALID_ARG
    assert L.topk_logits(n, 0, 256, 4, n, n, n, 0, n) == q.QW_OK             # no rows: nothing to do
    assert L.topk_logits(n, 2, 256, 4, FAKE, FAKE, FAKE, 1 << 20, n) == q.QW_ERR_INVALID_ARG
    assert L.topk_logits(MIS, 2, 256, 4, FAKE, FAKE, FAKE, 1 << 20, n) == q.QW_ERR_ALIGNMENT
    need = L.topk_workspace_bytes(2, 256, 4)
    assert L.topk_logits(FAKE, 2, 256, 4, FAKE, FAKE, FAKE, need - 1, n) == q.QW_ERR_WORKSPACE
    assert L.topk_logits(FAKE, 2, 256, 4, FAKE, FAKE, n, 0, n) == q.QW_ERR_WORKSPACE
    # gather: shapes, pointers, alignment
    assert L.embed_gather_w8(FAKE, -1, FAKE, 256, 256, FAKE, n) == q.QW_ERR_INVALID_ARG
    assert L.embed_gather_w8(FAKE, 4, FAKE, 200, 256, FAKE, n) == q.QW_ERR_UNSUPPORTED_SHAPE
    assert L.embed_gather_w8(FAKE, 4, FAKE, 256, 0, FAKE, n) == q.QW_ERR_UNSUPPORTED_SHAPE
    assert L.embed_gather_w8(n, 0, n, 256, 256, n, n) == q.QW_OK                # no tokens
    assert L.embed_gather_w8(n, 4, FAKE, 256, 256, FAKE, n) == q.QW_ERR_INVALID_ARG
    assert L.embed_gather_w8(FAKE, 4, MIS, 256, 256, FAKE, n) == q.QW_ERR_ALIGNMENT
    # the fused W4A8 entry point shares the GEMM checks
    assert L.qgemm_w4a8_fused(FAKE, FAKE, 4, 512, 100, FAKE, n, 0, n) == q.QW_ERR_UNSUPPORTED_SHAPE
    assert L.qgemm_w4a8_fused(n, FAKE, 4, 512, 256, FAKE, n, 0, n) == q.QW_ERR_INVALID_ARG
    assert L.qgemm_w4a8_fused(n, n, 0, 512, 256, n, n, 0, n) == q.QW_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_next_rows_report_arch_without_device():
    L = q.lib()
    n = ctypes.c_void_p(0)
    need = L.topk_workspace_bytes(2, 256, 4)
    assert L.topk_logits(FAKE, 2, 256, 4, FAKE, FAKE, FAKE, need, n) == q.QW_ERR_ARCH
    assert L.embed_gather_w8(FAKE, 4, FAKE, 256, 256, FAKE, n) == q.QW_ERR_ARCH


def _check_partition(p):
    """Every (tile, group) chunk belongs to exactly one segment of one CTA; a segment that
    cuts a tile has a partial slot of its own CTA (2p or 2p + 1); a cut tile's pieces come
    from consecutive CTAs in K order and cover its groups without gaps."""
    owner = {}
    slots = set()
    pieces = {}
    for cta in range(p.grid):
        for tile, g0, g1, slot in q.plan_segments(p, cta):
            assert 0 <= tile < p.tiles and 0 <= g0 < g1 <= p.groups
            for g in range(g0, g1):
                assert (tile, g) not in owner
                owner[(tile, g)] = cta
            if g0 == 0 and g1 == p.groups:
                assert slot == -1
            else:
                assert p.stream_k and slot in (2 * cta, 2 * cta + 1) and slot not in slots
                slots.add(slot)
                pieces.setdefault(tile, []).append((g0, g1, cta))
    assert len(owner) == p.chunks
    for tile, ps in pieces.items():
        ps.sort()
        assert ps[0][0] == 0 and ps[-1][1] == p.groups
        for (a0, a1, ca), (b0, b1, cb) in zip(ps, ps[1:]):
            assert a1 == b0 and cb == ca + 1


def test_schedule_partition_random_shapes():
    """Seeded random shapes across all four modes, token counts 1..9000, widths up to
    2^18 rows, depths up to 2^15 and SM counts 1..152: the chunk partition invariants hold
    and the plan fits the device limits."""
    import random
    rng = random.Random(20261202)
    for _ in range(120):
        mode = rng.randrange(4)
        M = rng.choice([1, 2, 3, 4, 5, 8, 15, 16, 17, 31, 33, 64, 65, 100, 128, 129, 255, 300, 512,
                        1000, 2048, 4097, 9000])
        N = 128 * rng.choice([1, 2, 3, 5, 7, 40, 41, 96, 272, 1024, 1940])
        K = 128 * rng.choice([1, 2, 3, 5, 8, 40, 41, 136])
        sms = rng.choice([1, 2, 7, 64, 100, 148, 152])
        p = q.plan(mode, M, N, K, sms)
        if p.chunks > 200_000:                    # keep the CPU check quick
            continue
        # one CTA per SM; the decode-batch kernel (half an SM each) runs two for long launches
        assert 1 <= p.grid <= (2 * sms if p.decode_teams else sms) and p.smem_bytes <= 232448 and p.stages >= 2
        if p.decode_row_blocks:
            _check_row_blocks(p, M, N, sms)
            continue
        if p.decode_teams:
            assert p.smem_bytes <= 113 * 1024 and M <= 16 and mode in (0, 1, 3)
        assert p.bn >= min(M, 256) and p.token_tiles == -(-M // p.bn)
        # the weight ring is split into one half per chunk parity, each slot with a single
        # producer filling it in order: an odd depth would let a parity wait alias (ABA)
        assert p.stages % 2 == 0 and 4 <= p.stages <= 16, p.stages
        assert 2 <= p.act_stages <= 4 and p.act_block in (1, 2, 4)
        _check_partition(p)


def test_profile_link_hash_ignores_comments_only():
    """The hash that ties a profile summary to its kernel sources covers the code with
    comments and blank lines removed: a comment edit keeps it, any change the compiler
    sees breaks it."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    src = b"// header\nint f(int x) {  // trailing\n  /* block\n     comment */return x + 1;\n}\n\n"
    same = b"// another header\n\nint f(int x) {\n  return x + 1;   // reworded\n}\n"
    other = b"int f(int x) {\n  return x + 2;\n}\n"
    assert bench.code_only(src) == bench.code_only(same)
    assert bench.code_only(src) != bench.code_only(other)
    h = bench.sources_sha256(bench.KERNEL_SOURCES)
    assert len(h) == 64 and h == bench.sources_sha256(bench.KERNEL_SOURCES)
