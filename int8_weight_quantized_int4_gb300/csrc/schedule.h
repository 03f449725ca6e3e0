// schedule.h -- work decomposition of the quantized GEMM over persistent CTAs.
// Host and device share this code, so the host-side tests check exactly what
// the kernels execute.
//
// Work unit ("chunk"): 128 weight rows x one 128-wide K group of one token tile.
// A tile is (token tile u, row tile t); tile index tau orders tiles so that CTAs
// running at the same time share weights and activations in L2.
//
// Two assignments:
//  * whole tiles, round-robin (tile p, p+grid, ...): used when there are many
//    more tiles than CTAs; no partial sums, no workspace traffic.
//  * stream-K: CTA p takes the contiguous chunk range
//    [floor(p*C/grid), floor((p+1)*C/grid)); a tile cut between CTAs is summed
//    from binary32 partials by the last CTA to finish it, in CTA order, so the
//    result does not depend on which CTA finishes last (deterministic).
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

struct Plan {
  int mode, M, N, K;
  int bn, U, T, G;
  long long tiles, chunks;
  int grid, stream_k, stages, smem_bytes;
  size_t ws_counters, ws_partials, ws_act, ws_bytes, ws_zero;
};

struct Seg {
  long long tile;
  int g0, g1;       // groups [g0, g1) of the tile
  int slot;         // partial-sum slot, or -1 when the segment covers the whole tile
};

QW_HD int pick_bn(int M) {
  return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
}

// tile index -> (token tile u, row tile t).  Token tiles are taken in supergroups
// of kTokenSuperTiles; inside one, the token tile varies fastest.
QW_HD void tile_coords(const Plan &P, long long tau, int &u, int &t) {
  const long long Z = P.U < kTokenSuperTiles ? P.U : kTokenSuperTiles;
  const long long full = P.U / Z;                  // full supergroups
  const long long per = (long long)P.T * Z;
  const long long zg = tau / per;
  if (zg < full) {
    const long long r = tau - zg * per;
    t = (int)(r / Z);
    u = (int)(zg * Z + r % Z);
  } else {
    const long long Zl = P.U - full * Z;           // last, partial supergroup
    const long long r = tau - full * per;
    t = (int)(r / Zl);
    u = (int)(full * Z + r % Zl);
  }
}

// first chunk of CTA p (stream-K)
QW_HD long long sk_begin(const Plan &P, int p) {
  return (long long)p * P.chunks / P.grid;
}

// CTA owning chunk c (stream-K): the largest p with sk_begin(p) <= c
QW_HD int sk_owner(const Plan &P, long long c) {
  return (int)(((c + 1) * (long long)P.grid - 1) / P.chunks);
}

// i-th segment of CTA p; false when there is none.
QW_HD bool segment(const Plan &P, int p, int i, Seg &s) {
  if (!P.stream_k) {
    const long long tau = (long long)p + (long long)i * P.grid;
    if (tau >= P.tiles) return false;
    s.tile = tau; s.g0 = 0; s.g1 = P.G; s.slot = -1;
    return true;
  }
  const long long c0 = sk_begin(P, p), c1 = sk_begin(P, p + 1);
  // walk segment boundaries: segment 0 starts at c0, later ones at tile starts
  long long c = c0;
  if (i > 0) {
    const long long first_tile = c0 / P.G;
    c = (first_tile + i) * (long long)P.G;
  }
  if (c >= c1) return false;
  s.tile = c / P.G;
  s.g0 = (int)(c - s.tile * P.G);
  const long long end = (s.tile + 1) * (long long)P.G < c1 ? (s.tile + 1) * (long long)P.G : c1;
  s.g1 = (int)(end - s.tile * P.G);
  const bool whole = (s.g0 == 0 && s.g1 == P.G);
  s.slot = whole ? -1 : (i == 0 ? 2 * p : 2 * p + 1);
  return true;
}

// For a tile cut between CTAs: the CTAs that hold its partials, in K order.
QW_HD void tile_contributors(const Plan &P, long long tile, int &p_first, int &p_last) {
  p_first = sk_owner(P, tile * P.G);
  p_last = sk_owner(P, tile * P.G + P.G - 1);
}

// Slot in which CTA p stored its partial of `tile`.
QW_HD int partial_slot(const Plan &P, int p, long long tile) {
  return (sk_begin(P, p) / P.G == tile) ? 2 * p : 2 * p + 1;
}

QW_HD size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int kSmemLimit = 232448;        // 227 KB opt-in dynamic shared memory per CTA
constexpr int kSmemReserve = 2048;        // barriers and bookkeeping
constexpr int kMaxStages = 12;
constexpr int kStreamKMaxTilesPerSm = 32;  // stream-K only below this many tiles per SM

QW_HD int chunk_bytes(int mode) { return mode == 2 ? kChunkW8 : kChunkW4; }

// W4A8 widens int8 activation codes to fp16 inside the GEMM (through a staging
// slot) for token tiles up to this size; larger tiles use a separate widening pass.
constexpr int kAct8InKernelMaxBn = 64;
QW_HD bool act8_in_kernel(int mode, int bn) { return mode == 1 && bn <= kAct8InKernelMaxBn; }

// Stage = one weight chunk (aligned to 1024 B) + the bn x 128 fp16 activation tile
// (+ a bn x 128 int8 staging slot when W4A8 widens in the kernel).
QW_HD int stage_bytes(int mode, int bn) {
  return (int)align_up((size_t)chunk_bytes(mode), 1024) + bn * kGroup * 2 +
         (act8_in_kernel(mode, bn) ? bn * kGroup : 0);
}

// Fill in a plan; returns 0 or -2 (unsupported shape) / -1 (bad argument).
QW_HD int make_plan(int mode, int M, int N, int K, int num_sms, Plan &P) {
  if (mode < 0 || mode > 2 || M < 0 || N < 0 || K < 0 || num_sms < 1) return -1;
  if (N % kRows || K % kGroup) return -2;
  P.mode = mode; P.M = M; P.N = N; P.K = K;
  P.bn = pick_bn(M);
  P.U = (M + P.bn - 1) / P.bn;
  P.T = N / kRows;
  P.G = K / kGroup;
  P.tiles = (long long)P.U * P.T;
  P.chunks = P.tiles * P.G;
  const bool many = P.tiles >= (long long)kStreamKMaxTilesPerSm * num_sms || (P.tiles % num_sms) == 0;
  P.stream_k = (P.chunks > 0 && !many) ? 1 : 0;
  if (P.chunks == 0) P.grid = 0;
  else if (P.stream_k) P.grid = (int)(P.chunks < num_sms ? P.chunks : num_sms);
  else P.grid = (int)(P.tiles < num_sms ? P.tiles : num_sms);
  const int sb = stage_bytes(mode, P.bn);
  int st = (kSmemLimit - kSmemReserve) / sb;
  if (st > kMaxStages) st = kMaxStages;
  P.stages = st;
  P.smem_bytes = st * sb + kSmemReserve;
  // Tile counters live in a fixed region at the start of every workspace, sized for
  // the largest stream-K plan (fewer than kStreamKMaxTilesPerSm tiles per SM), so
  // that no plan's partials or widened activations ever overlap another plan's
  // counters: a workspace zeroed once stays valid for calls of any shape.
  P.ws_counters = align_up((size_t)kStreamKMaxTilesPerSm * num_sms * 4, 256);
  P.ws_partials = P.stream_k ? (size_t)2 * P.grid * P.bn * kRows * 4 : 0;
  P.ws_act = (mode == 1 && !act8_in_kernel(mode, P.bn)) ? align_up((size_t)M * K * 2, 256) : 0;
  P.ws_zero = P.ws_counters;
  P.ws_bytes = P.ws_counters + P.ws_partials + P.ws_act;
  return 0;
}

}  // namespace qw
