// schedule.h -- work decomposition of the quantized GEMM over persistent CTAs.
// Host and device share this code, so the host-side tests check exactly what
// the kernels execute.  All device-side arithmetic is 32-bit, and the per-CTA
// chunk ranges are a table computed once on the host (no integer division by
// runtime values inside the pipeline loops).
//
// Work unit ("chunk"): 128 weight rows x one 128-wide K group of one token tile.
// A tile is (token tile u, row tile t); tile index tau orders tiles so that CTAs
// running at the same time share weights and activations in L2.
//
// Two assignments:
//  * whole tiles, round-robin (tile p, p+grid, ...): used when there are many
//    more tiles than CTAs; no partial sums, no workspace traffic.
//  * stream-K: CTA p takes the contiguous chunk range [begin[p], begin[p+1]) with
//    begin[p] = floor(p*C/grid); a tile cut between CTAs is summed from binary32
//    partials by the last CTA to finish it, in CTA order, so the result does not
//    depend on which CTA finishes last (deterministic).
#pragma once
#include <stdint.h>
#include <stddef.h>

#ifdef __CUDACC__
#define QW_HD __host__ __device__ __forceinline__
#else
#define QW_HD inline
#endif

namespace qw {

constexpr int kRows = 128;         // weight rows per tile (the MMA M, one per TMEM lane)
constexpr int kGroup = 128;        // K per group / per chunk
constexpr int kChunkW4 = 8192 + 256;
constexpr int kChunkW8 = 16384 + 256;
constexpr int kTokenSuperTiles = 16;   // token tiles kept hot in L2 together
constexpr int kMaxGrid = 320;          // persistent CTAs at most (one per SM, two for the decode kernel)

struct Plan {
  int mode, M, N, K;
  int bn, U, T, G;
  int tiles, chunks;
  int grid, stream_k;
  int stages;                    // weight ring depth (packed chunks)
  int xstages;                   // activation ring depth (blocks of xblock chunks)
  int xblock;                    // chunks per activation block (one tensor copy)
  int smem_bytes;
  int fused;                     // W4A8 with the per-token quantizer inside the GEMM (row-block plans)
  int ms_teams;                  // > 0: the warp-level MMA kernel for decode batches (M <= 16),
                                 // with this many teams of warps (one chunk per team at a time)
  int ms_red_bytes;              // its shared-memory buffer for the teams' partial sums
  int rb_max;                    // > 0: the row-block decode kernel, at most this many 16-row
                                 // blocks per CTA (begin[p]: first row block of CTA p)
  float grid_per_chunk;          // grid / chunks, to estimate a chunk's owner
  size_t ws_counters, ws_partials, ws_act, ws_quant, ws_bytes, ws_zero;
  int begin[kMaxGrid + 1];       // stream-K: first chunk of each CTA (begin[grid] = chunks)
  // stream-K: for CTA p's first ([p][0]) and last ([p][1]) segment, when that segment
  // is a cut tile, its contributors packed by cut_pack (p_first, p_last and the partial
  // slot of p_first; the others use 2 p'), else 0.  Lets a kernel find the partials of a
  // cut tile without searching the begin table.
  int cut[kMaxGrid][2];
};

// cut-tile contributors: p_first and p_last in 10 bits each (kMaxGrid <= 1024), the
// partial slot of p_first (< 2 kMaxGrid) in the upper 12 bits
static_assert(kMaxGrid <= 1024, "cut packing");
QW_HD int cut_pack(int pf, int pl, int slot) { return pf | (pl << 10) | (slot << 20); }
QW_HD int cut_first(int c) { return c & 0x3ff; }
QW_HD int cut_last(int c) { return (c >> 10) & 0x3ff; }
QW_HD int cut_slot(int c) { return (int)((unsigned)c >> 20); }

struct Seg {
  int tile;
  int g0, g1;       // groups [g0, g1) of the tile
  int slot;         // partial-sum slot, or -1 when the segment covers the whole tile
};

QW_HD int pick_bn(int M) {
  return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
}

// tile index -> (token tile u, row tile t).  Token tiles are taken in supergroups
// of kTokenSuperTiles; inside one, the token tile varies fastest.
QW_HD void tile_coords(const Plan &P, int tau, int &u, int &t) {
  if (P.U == 1) { u = 0; t = tau; return; }
  const int Z = P.U < kTokenSuperTiles ? P.U : kTokenSuperTiles;
  const int full = P.U / Z;                  // full supergroups
  const int per = P.T * Z;
  const int zg = tau / per;
  if (zg < full) {
    const int r = tau - zg * per;
    t = r / Z;
    u = zg * Z + r % Z;
  } else {
    const int Zl = P.U - full * Z;           // last, partial supergroup
    const int r = tau - full * per;
    t = r / Zl;
    u = full * Z + r % Zl;
  }
}

// CTA owning chunk c (stream-K): the largest p with begin[p] <= c.
QW_HD int sk_owner(const Plan &P, int c) {
  int p = (int)((float)c * P.grid_per_chunk);
  if (p > P.grid - 1) p = P.grid - 1;
  if (p < 0) p = 0;
  while (p + 1 < P.grid && P.begin[p + 1] <= c) ++p;
  while (p > 0 && P.begin[p] > c) --p;
  return p;
}

// i-th segment of CTA p; false when there is none.
QW_HD bool segment(const Plan &P, int p, int i, Seg &s) {
  if (!P.stream_k) {
    const int tau = p + i * P.grid;
    if (tau >= P.tiles) return false;
    s.tile = tau; s.g0 = 0; s.g1 = P.G; s.slot = -1;
    return true;
  }
  const int c0 = P.begin[p], c1 = P.begin[p + 1];
  // segment 0 starts at c0, later ones at tile starts
  const int first_tile = c0 / P.G;
  const int c = i == 0 ? c0 : (first_tile + i) * P.G;
  if (c >= c1) return false;
  s.tile = first_tile + i;
  s.g0 = c - s.tile * P.G;
  const int tile_end = (s.tile + 1) * P.G;
  s.g1 = (tile_end < c1 ? tile_end : c1) - s.tile * P.G;
  const bool whole = (s.g0 == 0 && s.g1 == P.G);
  s.slot = whole ? -1 : (i == 0 ? 2 * p : 2 * p + 1);
  return true;
}

// For a tile cut between CTAs: the CTAs that hold its partials, in K order.
QW_HD void tile_contributors(const Plan &P, int tile, int &p_first, int &p_last) {
  p_first = sk_owner(P, tile * P.G);
  p_last = sk_owner(P, tile * P.G + P.G - 1);
}

// Slot in which CTA p stored its partial of `tile` (its first or its last segment).
QW_HD int partial_slot(const Plan &P, int p, int tile) {
  const int b = P.begin[p];
  return (b >= tile * P.G && b < (tile + 1) * P.G) ? 2 * p : 2 * p + 1;
}

QW_HD size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int kSmemLimit = 232448;        // 227 KB opt-in dynamic shared memory per CTA
constexpr int kSmemReserve = 2048;        // barriers and bookkeeping
constexpr int kMaxWStages = 16;           // weight ring
constexpr int kMaxXStages = 4;            // activation ring
constexpr int kStreamKMaxTilesPerSm = 32;  // stream-K only below this many tiles per SM

QW_HD int chunk_bytes(int mode) { return mode == 2 ? kChunkW8 : kChunkW4; }

// Modes (as in the C ABI): 0 W4A16, 1 W4A8, 2 W8A16, 3 W4A8 from fp16 activations
// (quantized per token by the library).
// Mode 3 runs the standalone quantizer, which writes the codes into the workspace as
// fp16 values, with the token scales; the GEMM runs on them as plan mode kModeCodes16:
// int4 weights, fp16 activation tiles as in W4A16, token scales in the epilogue as in
// W4A8 (the products and sums are those of the int8 path: the codes are exact in fp16).
// On the row-block kernel, up to kFusedMaxTokens tokens whose fp16 rows take at most
// kFusedRowsMax bytes, the kernel quantizes instead (plan.fused, mode 3): every CTA reads
// the whole rows anyway, and quantizes all of them (each CTA needs every code), so the
// quantizer's arithmetic is paid once per CTA -- worth it only for a few tokens.
constexpr int kModeCodes16 = 4;
constexpr int kFusedRowsMax = 48 * 1024;
// Measured on the 5120 x 5120 layer (weights-immutable option): 8.1 / 9.1 us at 1 / 2
// tokens against ~9.8 / 10.4 for quantizer + GEMM; at 4 and 8 tokens 10.6 / 13.9 against
// 10.4 / 10.7 -- there the per-stage quantization in every CTA, not the scale pass (one
// round trip for all tokens), costs.
constexpr int kFusedMaxTokens = 2;

// W4A8 widens int8 activation codes to fp16 inside the GEMM (through a staging
// slot) for token tiles up to this size; larger tiles use a separate widening pass.
constexpr int kAct8InKernelMaxBn = 64;
QW_HD bool act8_in_kernel(int mode, int bn) { return mode == 1 && bn <= kAct8InKernelMaxBn; }

// Chunks per activation block: one tensor copy brings the activations of this many
// consecutive K groups of a token tile, so that small token tiles (4 KB per group
// at 16 tokens) do not pay one copy instruction per group.
QW_HD constexpr int act_block(int bn) { return bn <= 32 ? 4 : bn <= 64 ? 2 : 1; }

// Weight slot: one packed chunk (a multiple of 128 B; bulk copies need 16).
QW_HD int wstage_bytes(int mode) { return (int)align_up((size_t)chunk_bytes(mode), 128); }

// Activation slot: act_block(bn) fp16 tiles of bn x 128 (+ as many bn x 128 int8
// staging tiles when W4A8 widens in the kernel).
QW_HD int xstage_bytes(int mode, int bn) {
  return act_block(bn) * (bn * kGroup * 2 + (act8_in_kernel(mode, bn) ? bn * kGroup : 0));
}

// Decode batches (M <= kMsMaxTokens, int4 weights, fp16 or int8 activations) run on the
// warp-level MMA kernel: kMsTeams teams of warps, each team computing whole 128 x 128
// chunks, the dequantized weights going from registers straight into the MMA.  Its CTA
// takes at most half an SM (shared memory, registers), so that the next layer's CTAs
// can start on an SM while this layer's finish there.
constexpr int kMsMaxTokens = 16;
constexpr int kMsComputeWarps = 8;
constexpr int kMsRedStride = 132;        // floats per token row of a team's sum buffer
constexpr int kMsSmemLimit = 113 * 1024; // two CTAs per SM
// Launches of at least this many chunks per SM run two decode CTAs per SM (more warps
// streaming at once); shorter ones one, leaving the SM's other half to the next layer.
constexpr int kMsLongChunksPerSm = 32;
// With the weights declared immutable, the weight-copy thread pulls at most this many
// chunks past its ring into L2 before the preceding kernel ends (304 CTAs x 16 x 8.4 KB
// = 41 MB, well inside the 129 MB L2).
constexpr int kMsL2AheadChunks = 16;
QW_HD bool ms_kernel(int mode, int M) {
  return (mode == 0 || mode == 1 || mode == 3 || mode == kModeCodes16) && M >= 1 && M <= kMsMaxTokens;
}
// token rows of its activation tiles: 8 (one tile of eight tokens) or 16
QW_HD int ms_rows(int M) { return M <= 8 ? 8 : 16; }
// 16-row blocks of a chunk per warp: 4 for long launches of up to 8 tokens from fp16
// activations (more independent MMA chains per warp), else 2 (W4A8 always: the fp16-code
// plan sums in the order of the int8 one, which makes the two paths bit-identical).  A
// team computes one chunk at a time with 8 / (row blocks per warp) warps, so there are as
// many teams as row blocks per warp.
QW_HD int ms_row_blocks(int mode, int M, bool long_launch) { return long_launch && mode == 0 && M <= 8 ? 4 : 2; }
// the teams other than the first leave their sums here at the end of a tile segment
QW_HD int ms_red_bytes(int M, int teams) { return (teams - 1) * ms_rows(M) * kMsRedStride * 4; }
// activation slot: act_block(16) = 4 K groups of ms_rows(M) x 128 fp16 (+ int8 staging)
QW_HD int ms_xstage_bytes(int mode, int M) {
  return 4 * ms_rows(M) * kGroup * (mode == 1 ? 3 : 2);
}
// ring depths: three activation blocks when that leaves eight weight slots, else two;
// the weight slots (at most kMaxWStages) split evenly between the teams
QW_HD bool ms_ring_depths(int mode, int M, int teams, int &xst, int &wst) {
  const int xb = ms_xstage_bytes(mode, M), wb = (int)align_up((size_t)kChunkW4, 128);
  for (int x = 3; x >= 2; --x) {
    int w = (kMsSmemLimit - kSmemReserve - ms_red_bytes(M, teams) - x * xb) / wb;
    if (w > kMaxWStages) w = kMaxWStages;
    w -= w % teams;
    if (w >= 8 || (x == 2 && w >= 2 * teams)) { xst = x; wst = w; return true; }
  }
  return false;
}

// Decode batches on layers of few rows: the row-block kernel.  When the layer's 16-row
// blocks (N / 16) number at most kRbMax per SM, every CTA takes a contiguous range of 1 to
// kRbMax row blocks over the whole K and its compute warps split the K groups, adding their
// sums in shared memory at the end: no tile is cut between CTAs, so there are no partial
// sums, no tile counters and no last-arriver reduction.  Up to 8 tokens a launch long
// enough for two tile-kernel CTAs per SM (kMsLongChunksPerSm) stays on the tile kernel,
// which measured faster there (a 5120 x 17408 layer: 15.1 against 17.6 us at one token).
constexpr int kRbMax = 3;                 // row blocks per CTA at most
constexpr int kRbReserve = 4096;          // barriers, the in-kernel quantizer's amax and scales
constexpr int kRbXBlock = 8;              // K groups per ring stage: one per compute warp
constexpr int kRbMaxStages = 6;
QW_HD bool rb_kernel(int mode, int M, int N, int K, int num_sms) {
  if (!ms_kernel(mode, M) || (long long)(N / 16) > (long long)kRbMax * num_sms) return false;
  return ms_rows(M) > 8 || (long long)(N / kRows) * (K / kGroup) < (long long)kMsLongChunksPerSm * num_sms;
}
// one ring stage holds the data of kRbXBlock consecutive K groups: the activation tiles
// (8 groups of ms_rows(M) x 128 fp16, + the int8 staging tiles for W4A8 from int8 codes),
// then per row block the 8 groups' codes (8 x 1 KB) and scales (8 x 32 B); a multiple of
// 1 KB (the activation tiles' 128-byte swizzle)
QW_HD int rb_x_bytes(int mode, int M) { return kRbXBlock * ms_rows(M) * kGroup * (mode == 1 ? 3 : 2); }
constexpr int kRbWBytes = kRbMax * kRbXBlock * 1024;     // codes of a stage
constexpr int kRbSBytes = kRbMax * kRbXBlock * 32;       // scales of a stage
QW_HD int rb_stage_bytes(int mode, int M) {
  return (int)align_up((size_t)(rb_x_bytes(mode, M) + kRbWBytes + kRbSBytes), 1024);
}
// one CTA per SM, as many stages as fit (at most kRbMaxStages, at least 2)
QW_HD bool rb_ring_depths(int mode, int M, int &st) {
  st = (kSmemLimit - kRbReserve) / rb_stage_bytes(mode, M);
  if (st > kRbMaxStages) st = kRbMaxStages;
  return st >= 2;
}

// Ring depths: the deepest activation ring (at most kMaxXStages, or 3 for token
// tiles up to 64 whose blocks already span several groups, at least 2) that still
// leaves four weight slots; the weight ring takes the rest (at most kMaxWStages),
// rounded down to an even count (half per dequant group).  Returns false when
// even 2 + 4 slots do not fit.
QW_HD bool ring_depths(int mode, int bn, int &xst, int &wst, int split = 2) {
  const int xb = xstage_bytes(mode, bn), wb = wstage_bytes(mode);
  for (int x = bn <= 64 ? 3 : kMaxXStages; x >= 2; --x) {
    int w = (kSmemLimit - kSmemReserve - x * xb) / wb;
    if (w > kMaxWStages) w = kMaxWStages;
    w -= w % split;                      // the same number of slots per consumer
    if (w >= 2 * split) { xst = x; wst = w; return true; }
  }
  return false;
}

// Tile-aligned split for short stream-K launches: at least 3 CTAs per tile and at
// most this many chunks per CTA.
constexpr int kAlignedMaxChunksPerCta = 16;

QW_HD bool aligned_split(const Plan &P) {
  return P.stream_k && P.tiles > 0 && 3LL * P.tiles <= P.grid &&
         (long long)P.chunks <= (long long)kAlignedMaxChunksPerCta * P.grid;
}

// Fill the stream-K chunk table and the cut-tile contributors from grid and chunks (host).
//
// Two splits.  Long launches: CTA p takes chunks [floor(p C / grid), floor((p+1) C / grid)),
// balanced to one chunk.  Short launches (aligned_split): every tile is cut into b or
// b + 1 equal pieces (b = grid / tiles, the pieces summing to grid) and each CTA takes
// exactly one piece, tiles with the larger pieces first.  A CTA then holds a single
// segment, all contributors of a tile finish together, and the CTAs with the highest
// index -- the last to become resident when a launch follows another (they wait for the
// preceding kernel's slowest CTAs to leave their SM) -- get the smaller pieces.
inline void fill_begin(Plan &P) {
  if (aligned_split(P)) {
    const int b = P.grid / P.tiles, big = P.tiles - P.grid % P.tiles;   // tiles cut into b pieces
    int p = 0;
    for (int t = 0; t < P.tiles; ++t) {
      const int k = t < big ? b : b + 1;
      for (int j = 0; j < k; ++j) P.begin[p++] = t * P.G + (j * P.G) / k;
    }
    for (; p <= kMaxGrid; ++p) P.begin[p] = P.chunks;
  } else {
    for (int p = 0; p <= kMaxGrid; ++p)
      P.begin[p] = (P.grid && p <= P.grid) ? (int)((long long)p * P.chunks / P.grid) : P.chunks;
  }
  P.grid_per_chunk = P.chunks ? (float)P.grid / (float)P.chunks : 0.0f;
  for (int p = 0; p < kMaxGrid; ++p) P.cut[p][0] = P.cut[p][1] = 0;
  if (!P.stream_k) return;
  for (int p = 0; p < P.grid; ++p) {
    Seg s;
    int last = -1;
    for (int i = 0; segment(P, p, i, s); ++i) last = i;
    for (int e = 0; e < 2 && last >= 0; ++e) {
      segment(P, p, e == 0 ? 0 : last, s);
      if (s.slot < 0) continue;
      int pf, pl;
      tile_contributors(P, s.tile, pf, pl);
      P.cut[p][e] = cut_pack(pf, pl, partial_slot(P, pf, s.tile));
    }
  }
}

// Fill in a plan (host); returns 0, -2 (unsupported shape) or -1 (bad argument).
inline int make_plan(int mode, int M, int N, int K, int num_sms, Plan &P) {
  if (mode < 0 || mode > 3 || M < 0 || N < 0 || K < 0 || num_sms < 1) return -1;
  if (N % kRows || K % kGroup) return -2;
  if (num_sms > kMaxGrid / 2) num_sms = kMaxGrid / 2;
  P.fused = (mode == 3 && M <= kFusedMaxTokens && (long long)M * K * 2 <= kFusedRowsMax &&
             rb_kernel(kModeCodes16, M, N, K, num_sms)) ? 1 : 0;
  // mode 3 outside that is the quantizer (fp16 codes) followed by a kModeCodes16 plan
  const bool quant_first = mode == 3 && !P.fused;
  if (quant_first) mode = kModeCodes16;
  P.mode = mode; P.M = M; P.N = N; P.K = K;
  P.bn = pick_bn(M);
  P.U = (M + P.bn - 1) / P.bn;
  P.T = N / kRows;
  P.G = K / kGroup;
  const long long tiles = (long long)P.U * P.T;
  const long long chunks = tiles * P.G;
  if (chunks >= (1LL << 30)) return -2;      // 32-bit chunk indices with headroom
  P.tiles = (int)tiles;
  P.chunks = (int)chunks;
  // persistent CTAs: one per SM, two for long decode-kernel launches (at most kMaxGrid)
  int ctas = num_sms;
  if (ms_kernel(mode, M) && (long long)P.chunks >= (long long)kMsLongChunksPerSm * num_sms) ctas = 2 * num_sms;
  if (ctas > kMaxGrid) ctas = kMaxGrid;
  const bool many = P.tiles >= kStreamKMaxTilesPerSm * num_sms || (P.tiles % ctas) == 0;
  P.stream_k = (P.chunks > 0 && !many) ? 1 : 0;
  if (P.chunks == 0) P.grid = 0;
  else if (P.stream_k) P.grid = P.chunks < ctas ? P.chunks : ctas;
  else P.grid = P.tiles < ctas ? P.tiles : ctas;
  fill_begin(P);
  P.xblock = act_block(P.bn);
  P.ms_teams = ms_kernel(mode, M) ? ms_row_blocks(mode, M, ctas > num_sms) : 0;
  P.rb_max = 0;
  if (P.chunks > 0 && rb_kernel(mode, M, N, K, num_sms)) {
    // the row-block kernel: CTA p takes row blocks [begin[p], begin[p + 1])
    const int RB = N / 16;
    P.ms_teams = 0;
    P.stream_k = 0;
    P.grid = RB < num_sms ? RB : num_sms;
    for (int p = 0; p <= kMaxGrid; ++p)
      P.begin[p] = p <= P.grid ? (int)((long long)p * RB / P.grid) : RB;
    P.rb_max = (RB + P.grid - 1) / P.grid;
    for (int p = 0; p < kMaxGrid; ++p) P.cut[p][0] = P.cut[p][1] = 0;
    P.xblock = kRbXBlock;
    P.ms_red_bytes = 0;
    if (!rb_ring_depths(mode, M, P.stages)) return -2;
    P.xstages = P.stages;
    P.smem_bytes = P.stages * rb_stage_bytes(mode, M) + kRbReserve;
  } else if (P.ms_teams) {
    P.ms_red_bytes = ms_red_bytes(M, P.ms_teams);
    if (!ms_ring_depths(mode, M, P.ms_teams, P.xstages, P.stages)) return -2;
    P.smem_bytes = P.xstages * ms_xstage_bytes(mode, M) + P.stages * wstage_bytes(mode) + P.ms_red_bytes +
                   kSmemReserve;
  } else {
    P.ms_red_bytes = 0;
    if (!ring_depths(mode, P.bn, P.xstages, P.stages)) return -2;
    P.smem_bytes = P.xstages * xstage_bytes(mode, P.bn) + P.stages * wstage_bytes(mode) + kSmemReserve;
  }
  // Tile counters live in a fixed region at the start of every workspace, sized for
  // the largest stream-K plan (fewer than kStreamKMaxTilesPerSm tiles per SM), so
  // that no plan's partials or widened activations ever overlap another plan's
  // counters: a workspace zeroed once stays valid for calls of any shape.
  P.ws_counters = align_up((size_t)kStreamKMaxTilesPerSm * num_sms * 4, 256);
  P.ws_partials = P.stream_k ? (size_t)2 * P.grid * P.bn * kRows * 4 : 0;   // (row-block plans: 0)
  P.ws_act = (mode == 1 && !act8_in_kernel(mode, P.bn)) ? align_up((size_t)M * K * 2, 256) : 0;
  // quantizer output (fp16 codes, then binary32 token scales) when it runs first
  P.ws_quant = quant_first ? align_up((size_t)M * K * 2, 256) + align_up((size_t)M * 4, 256) : 0;
  P.ws_zero = P.ws_counters;
  P.ws_bytes = P.ws_counters + P.ws_partials + P.ws_act + P.ws_quant;
  return 0;
}

}  // namespace qw
