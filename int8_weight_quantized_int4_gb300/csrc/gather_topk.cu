// gather_topk.cu -- the two ends of the quantized model around the GEMMs:
//   embed_gather_kernel : dequant-on-gather from an int8 group-128 table packed by
//                         qpack_w8 ("In full" items 1-2 of "What this repo does that
//                         stock vLLM doesn't": embeddings requantized to int8 g128 and
//                         read through a dequant-on-gather kernel)
//   topk_kernel         : per row the k largest logits, largest first, ties to the
//                         smaller index ("In full" item 6: with top-k known on the host
//                         the sampler's mask is one small top-k)
#include <stdint.h>
#include <cuda_fp16.h>
#include "ptx.cuh"
#include "schedule.h"
#include "launch.h"

namespace qw {

// ---------------------------------------------------------------- gather --
// One CTA per token, kGatherPer 16-feature pieces per thread with all their loads issued
// before any is used.  Feature k of table row v sits in chunk (v / 128, k / 128) of the
// packed table, slice (k % 128) / 16, at byte (v % 128) * 16 + k % 16, stored as
// code XOR 0x80; the row's fp16 scale follows the slices.  out = fp16(code * scale),
// one rounding (__hmul_rn of two exact fp16 operands).
constexpr int kGatherPer = 2;

__global__ void __launch_bounds__(256) embed_gather_kernel(const int32_t *__restrict__ ids,
                                                           const uint8_t *__restrict__ packed, int V,
                                                           int D, uint16_t *__restrict__ out,
                                                           int *err) {
  griddep_wait();
  griddep_launch_dependents();
  const int t = blockIdx.x;
  const int v = ids[t];
  const int G = D / kGroup;
  uint4 *orow = reinterpret_cast<uint4 *>(out + (size_t)t * D);
  if (v < 0 || v >= V) {
    for (int p = threadIdx.x; p < D / 8; p += blockDim.x) orow[p] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) atomicCAS(err, 0, -9);
    return;
  }
  const int r = v % kRows;
  const uint8_t *tile = packed + (size_t)(v / kRows) * G * kChunkW8;
  for (int p0 = threadIdx.x; p0 < G * 8; p0 += kGatherPer * blockDim.x) {
    uint4 c[kGatherPer];
    __half s[kGatherPer];
#pragma unroll
    for (int u = 0; u < kGatherPer; ++u) {
      const int p = p0 + u * blockDim.x;              // 16 features per piece
      if (p >= G * 8) break;
      const uint8_t *chunk = tile + (size_t)(p >> 3) * kChunkW8;
      c[u] = __ldg(reinterpret_cast<const uint4 *>(chunk + (p & 7) * 2048 + r * 16));
      s[u] = __ushort_as_half(__ldg(reinterpret_cast<const unsigned short *>(chunk + 16384 + r * 2)));
    }
#pragma unroll
    for (int u = 0; u < kGatherPer; ++u) {
      const int p = p0 + u * blockDim.x;
      if (p >= G * 8) break;
      const uint32_t w[4] = {c[u].x ^ 0x80808080u, c[u].y ^ 0x80808080u, c[u].z ^ 0x80808080u,
                             c[u].w ^ 0x80808080u};
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q0 = (int)(int8_t)((w[i] >> (16 * h)) & 0xffu);
          const int q1 = (int)(int8_t)((w[i] >> (16 * h + 8)) & 0xffu);
          const __half a = __hmul_rn(__int2half_rn(q0), s[u]), b = __hmul_rn(__int2half_rn(q1), s[u]);
          o[2 * i + h] = (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
        }
      }
      uint4 *dst = orow + (size_t)((p >> 3) * kGroup + (p & 7) * 16) / 8;
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

cudaError_t launch_embed_gather(const int32_t *ids, int T, const void *packed, int V, int D,
                                uint16_t *out, int *err, cudaStream_t st) {
  // kGatherPer pieces of 16 features per thread: D / 32 threads, in whole warps, 32..256
  int threads = (D / 16 + kGatherPer - 1) / kGatherPer;
  threads = (threads + 31) / 32 * 32;
  if (threads > 256) threads = 256;
  if (threads < 32) threads = 32;
  cudaError_t e = launch_pdl(reinterpret_cast<const void *>(embed_gather_kernel), dim3(T), dim3(threads), 0,
                             st, ids, static_cast<const uint8_t *>(packed), V, D, out, err);
  count_launch();
  return e;
}

// ------------------------------------------------------------------ top-k --
// Order: larger value first, equal values by smaller index.  key16 maps fp16 to an
// order-preserving 16-bit integer (-0 taken as +0, so the two tie); positions past N get
// key 0, which no finite fp16 value maps to.  Within a slice of at most 4096 positions an
// element is the 32-bit composite  key16 << 16 | (0xffff - local position), unique and in
// exactly that order.  A slice finds its k largest by radix selection: a first 8-bit pass
// over the top byte of the keys (computed two at a time from the packed fp16 words), then
// only the elements above the boundary bin (all taken) and in it (listed in shared memory
// for the next 8-bit passes) become composites.  It lists its winners in order in the
// workspace as 40-bit global composites  key16 << 24 | (2^24 - 1 - index).  The last slice
// CTA of a row selects again, the same way, over the row's S k candidates as
// key16 << 16 | (0xffff - slot): slices cover ascending index ranges and list their
// candidates in order, so among equal keys the smaller slot is the smaller index.
constexpr int kTopkThreads = 256;
constexpr int kTopkMaxK = 64;
constexpr int kTopkMaxSlices = 64;
constexpr int kTopkMaxVec = 2;                 // 16-byte vectors per thread per slice
constexpr int kTopkMerge = kTopkMaxSlices * kTopkMaxK / kTopkThreads;   // candidates per thread
static_assert(kTopkMaxSlices * kTopkMaxK <= kTopkMaxVec * 8 * kTopkThreads, "one list serves both selections");

__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t index) {
  return ((uint64_t)key << 24) | (uint64_t)(0xffffffu - index);
}

// Warp 0: the bin (of 256, scanning from the top) holding the remaining-th largest
// counted element -> bc[0] = bin, bc[1] = how many of it are still wanted, bc[2] = its
// count.  Lane l owns bins 255 - 8l .. 248 - 8l; a prefix sum over lanes finds the lane.
__device__ __forceinline__ void find_bin(const int *hist, int remaining, int *bc) {
  const int lane = threadIdx.x;
  int cnt[8], local = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    cnt[i] = hist[255 - 8 * lane - i];
    local += cnt[i];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining);
  if (lane == __ffs(hit) - 1) {
    int cum = incl - local;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (cum + cnt[i] >= remaining) {
        bc[0] = 255 - 8 * lane - i;
        bc[1] = remaining - cum;
        bc[2] = cnt[i];
        break;
      }
      cum += cnt[i];
    }
  }
}

// The shared state of one selection: hist 2 x 256 ints (one per pass in turn, the next
// cleared while the current one fills), bc 3 ints, the boundary-bin list (room for every
// element of the selection) and the winners.
template <int CAP>
struct TopkSmemT {
  int hist[2 * 256];
  int bc[3];
  int nlist, nsel;
  uint32_t list[CAP];
  uint32_t sel[kTopkMaxK];
};
using TopkSmem = TopkSmemT<kTopkMaxVec * 8 * kTopkThreads>;   // >= kTopkMaxSlices * kTopkMaxK

// Called by the whole CTA after the first pass (over the top byte) found the boundary bin
// b0 with r0 of its elements still wanted, every element of the CTA above b0 already in
// sel and every element in b0 in the list (T of them, all distinct composites with top
// byte b0), hist[256..511] zero.  Unless the bin is taken whole, the next 8-bit passes run
// over the list; its elements at or above the resulting threshold join sel, which then
// holds exactly k composites.
template <class SM>
__device__ void finish_select(SM &sm, uint32_t b0, int r0, bool whole) {
  const int T = sm.nlist;
  if (whole) {
    for (int j = threadIdx.x; j < T; j += kTopkThreads) sm.sel[atomicAdd(&sm.nsel, 1)] = sm.list[j];
    __syncthreads();
    return;
  }
  uint32_t prefix = b0 << 24;
  int remaining = r0;
#pragma unroll 1
  for (int pass = 1; pass < 4; ++pass) {
    int *h = sm.hist + 256 * (pass & 1);
    int *hn = sm.hist + 256 * ((pass + 1) & 1);
    const int shift = 24 - 8 * pass;
    const uint32_t above = 0xffffffffu << (shift + 8);   // bits already fixed
    for (int j = threadIdx.x; j < T; j += kTopkThreads) {
      const uint32_t v = sm.list[j];
      if (((v ^ prefix) & above) == 0u) atomicAdd(&h[(v >> shift) & 0xffu], 1);
    }
    for (int b = threadIdx.x; b < 256; b += kTopkThreads) hn[b] = 0;
    __syncthreads();
    if (threadIdx.x < 32) find_bin(h, remaining, sm.bc);
    __syncthreads();
    prefix |= (uint32_t)sm.bc[0] << shift;
    remaining = sm.bc[1];
    if (sm.bc[2] == remaining) break;                 // the bin is taken whole: done
  }
  for (int j = threadIdx.x; j < T; j += kTopkThreads)
    if (sm.list[j] >= prefix) sm.sel[atomicAdd(&sm.nsel, 1)] = sm.list[j];
  __syncthreads();
}

// First pass over register composites c[0..n) (at least k of them in the CTA): histogram
// of the top byte, boundary bin, then the split into winners and list; returns with sel
// holding the k largest.
template <int NMAX, class SM>
__device__ void select_regs(const uint32_t (&c)[NMAX], int n, int k, SM &sm) {
  for (int b = threadIdx.x; b < 512; b += kTopkThreads) sm.hist[b] = 0;
  if (threadIdx.x == 0) sm.nlist = sm.nsel = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NMAX; ++i)
    if (i < n) atomicAdd(&sm.hist[c[i] >> 24], 1);
  __syncthreads();
  if (threadIdx.x < 32) find_bin(sm.hist, k, sm.bc);
  __syncthreads();
  const uint32_t b0 = (uint32_t)sm.bc[0];
  const int r0 = sm.bc[1];
  const bool whole = sm.bc[2] == r0;
#pragma unroll
  for (int i = 0; i < NMAX; ++i) {
    if (i >= n) continue;
    const uint32_t tb = c[i] >> 24;
    if (tb > b0) sm.sel[atomicAdd(&sm.nsel, 1)] = c[i];
    else if (tb == b0) sm.list[atomicAdd(&sm.nlist, 1)] = c[i];
  }
  __syncthreads();
  finish_select(sm, b0, r0, whole);
}

// sel's k distinct composites in decreasing order: the rank of each among them.
__device__ __forceinline__ int rank_of(const uint32_t *sel, int k, int a) {
  int rank = 0;
  for (int b = 0; b < k; ++b) rank += sel[b] > sel[a];
  return rank;
}

// grid (slices, rows).  ws: [M] int counters (zero between calls), then candidates
// [M][slices][k] (40-bit global composites, each slice's in order).
// At most 48 registers a thread (five CTAs an SM); the kernel runs many CTAs per row.
__global__ void __launch_bounds__(kTopkThreads, 5) topk_kernel(const uint16_t *__restrict__ logits, int N,
                                                                int k, int slice_len, uint16_t *vals,
                                                                int32_t *idx, int *counters,
                                                                uint64_t *cand) {
  __shared__ TopkSmem sm;
  __shared__ int last;
  griddep_wait();
  griddep_launch_dependents();
  const int m = blockIdx.y, sl = blockIdx.x, S = gridDim.x;
  const uint16_t *row = logits + (size_t)m * N;
  uint64_t *rowcand = cand + (size_t)m * S * k;

  // ---- this slice: its k best (padding past N included when the slice is short)
  {
    uint32_t kw[kTopkMaxVec * 4];                     // order keys, two per word
    const int base = sl * slice_len;
    const int nvec = slice_len / (8 * kTopkThreads);
#pragma unroll
    for (int e = 0; e < kTopkMaxVec; ++e) {
      const int lp = 8 * (threadIdx.x + kTopkThreads * e);
      const bool in = e < nvec && base + lp < N;    // N % 8 == 0: a vector is all in or all out
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (in) v = __ldg(reinterpret_cast<const uint4 *>(row + base + lp));
      kw[4 * e + 0] = in ? order_keys2(v.x) : 0u;
      kw[4 * e + 1] = in ? order_keys2(v.y) : 0u;
      kw[4 * e + 2] = in ? order_keys2(v.z) : 0u;
      kw[4 * e + 3] = in ? order_keys2(v.w) : 0u;
    }
    for (int b = threadIdx.x; b < 512; b += kTopkThreads) sm.hist[b] = 0;
    if (threadIdx.x == 0) sm.nlist = sm.nsel = 0;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kTopkMaxVec * 4; ++w)
      if (w < 4 * nvec) {
        atomicAdd(&sm.hist[(kw[w] >> 8) & 0xffu], 1);
        atomicAdd(&sm.hist[kw[w] >> 24], 1);
      }
    __syncthreads();
    if (threadIdx.x < 32) find_bin(sm.hist, k, sm.bc);
    __syncthreads();
    const uint32_t b0 = (uint32_t)sm.bc[0];
    const int r0 = sm.bc[1];
    const bool whole = sm.bc[2] == r0;
#pragma unroll
    for (int w = 0; w < kTopkMaxVec * 4; ++w) {
      if (w >= 4 * nvec) continue;
      const uint32_t pos = (uint32_t)(8 * (threadIdx.x + kTopkThreads * (w >> 2)) + 2 * (w & 3));
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const uint32_t key = hf ? kw[w] >> 16 : kw[w] & 0xffffu;
        const uint32_t tb = key >> 8;
        if (tb < b0) continue;
        const uint32_t c = (key << 16) | (0xffffu - (pos + hf));
        if (tb > b0) sm.sel[atomicAdd(&sm.nsel, 1)] = c;
        else sm.list[atomicAdd(&sm.nlist, 1)] = c;
      }
    }
    __syncthreads();
    finish_select(sm, b0, r0, whole);
    for (int a = threadIdx.x; a < k; a += kTopkThreads)     // listed in order
      rowcand[(size_t)sl * k + rank_of(sm.sel, k, a)] =
          composite(sm.sel[a] >> 16, (uint32_t)base + (0xffffu - (sm.sel[a] & 0xffffu)));
  }

  // ---- publish; the last slice CTA of the row merges
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(counters + m, 1);
    last = (old == S - 1);
    if (last) counters[m] = 0;                      // leave the workspace zeroed
  }
  __syncthreads();
  if (!last) return;
  __threadfence();

  uint32_t c[kTopkMerge];
  const int total = S * k;
  const unsigned long long *rc = reinterpret_cast<const unsigned long long *>(rowcand);
#pragma unroll
  for (int i = 0; i < kTopkMerge; ++i) {
    const int q = threadIdx.x + kTopkThreads * i;
    c[i] = q < total ? ((uint32_t)(__ldcg(rc + q) >> 24) << 16) | (0xffffu - (uint32_t)q) : 0u;
  }
  const int nmine = total > threadIdx.x ? (total - 1 - (int)threadIdx.x) / kTopkThreads + 1 : 0;
  select_regs(c, nmine, k, sm);
  // rank sort of the k winners (all distinct), largest first
  for (int a = threadIdx.x; a < k; a += kTopkThreads) {
    const uint64_t g = __ldcg(rc + (0xffffu - (sm.sel[a] & 0xffffu)));
    const int n = 0xffffff - (int)(g & 0xffffffu);
    const int rank = rank_of(sm.sel, k, a);
    idx[(size_t)m * k + rank] = n;
    vals[(size_t)m * k + rank] = row[n];
  }
}

// ------------------------------------------------ top-k from tile maxima --
// The lm_head with top-k.  The GEMM's epilogue leaves, per token m and 128-row tile t of
// the logits, the largest order key among the tile's outputs (tile_max[m][t]).  With
// t_k the k-th largest of those maxima, at least k logits are >= t_k (one per tile of
// the k best), so every logit of the top k lies in a tile whose maximum is >= t_k: the
// candidate tiles, exactly k of them unless maxima tie.  kTopkSlices CTAs per token:
//   1. every CTA finds t_k, the k-th largest 16-bit key among the tile maxima (every
//      tile is a candidate when there are at most k), and lists the candidate tiles in
//      ascending order (one block-wide scan);
//   2. CTA s takes its share of the candidate tiles: the k largest of their logits
//      (T, the k-th largest key, and r, how many keys equal to T are among the k; every
//      logit above T and the first r equal to it, by warp ballots over consecutive
//      positions), written to the workspace as (key, index) pairs;
//   3. the last CTA of the token ranks the slices' pairs by (key descending, index
//      ascending), writes the first k, and clears the tile maxima and its counter (zero
//      again for the next call).
// A k-th largest key is built two bits at a time from the top: the largest prefix with
// at least k keys at or above it, by block-wide counts over keys held in registers two
// to a word (SIMD compares; no atomics, which crowd onto a few addresses when the keys
// of a row are close together).  A share with more logits than the registers hold (many
// tied tile maxima) is read from global memory instead, in the same order.
constexpr int kTileThreads = 256;
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kMaxTiles = kTopkMaxN / kRows;                   // 2048
constexpr int kTileWords = kMaxTiles / 2 / kTileThreads;       // 4: tile-maximum key pairs a thread
constexpr int kStageWords = 8;                                 // logit key pairs a thread, registers
constexpr int kStageKeys = 2 * kStageWords * kTileThreads;     // 4096 logits (32 tiles) a share
constexpr int kMergeMax = kTopkSlices * kTopkMaxK;             // pairs the last CTA ranks

struct TileTopkSmem {
  alignas(16) int cnt[2][4][kTileWarps];
  int wsum[2][kTileWarps];
  alignas(16) uint16_t tkey[kMaxTiles];
  uint16_t cand[kMaxTiles];
  alignas(16) uint16_t lkey[kStageKeys];
  unsigned long long mc[kMergeMax];               // merge: key << 32 | (2^32 - 1 - index)
  int last;
};

// Block-wide exclusive scan of a pair of counts; the totals in tot.  Two barriers.
__device__ __forceinline__ int2 block_scan2(int a, int b, int (&wsum)[2][kTileWarps], int2 &tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ta = __shfl_up_sync(0xffffffffu, ia, o), tb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += ta;
      ib += tb;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = ia;
    wsum[1][warp] = ib;
  }
  __syncthreads();
  int pa = 0, pb = 0;
  tot = make_int2(0, 0);
#pragma unroll
  for (int w = 0; w < kTileWarps; ++w) {
    if (w < warp) {
      pa += wsum[0][w];
      pb += wsum[1][w];
    }
    tot.x += wsum[0][w];
    tot.y += wsum[1][w];
  }
  __syncthreads();                                    // wsum free for the next scan
  return make_int2(pa + ia - a, pb + ib - b);
}

// Block-wide sums of four per-thread counts (one barrier; buffer `buf` of two).
__device__ __forceinline__ int4 block_sum4(int a, int b, int c, int d, TileTopkSmem &sm, int buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = __reduce_add_sync(0xffffffffu, a);
  b = __reduce_add_sync(0xffffffffu, b);
  c = __reduce_add_sync(0xffffffffu, c);
  d = __reduce_add_sync(0xffffffffu, d);
  if (lane == 0) {
    sm.cnt[buf][0][warp] = a;
    sm.cnt[buf][1][warp] = b;
    sm.cnt[buf][2][warp] = c;
    sm.cnt[buf][3][warp] = d;
  }
  __syncthreads();
  int4 t = make_int4(0, 0, 0, 0);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int4 u = reinterpret_cast<const int4 *>(sm.cnt[buf][q])[0];
    const int4 v = reinterpret_cast<const int4 *>(sm.cnt[buf][q])[1];
    const int sum = u.x + u.y + u.z + u.w + v.x + v.y + v.z + v.w;
    if (q == 0) t.x = sum;
    else if (q == 1) t.y = sum;
    else if (q == 2) t.z = sum;
    else t.w = sum;
  }
  return t;
}

// How many of the two 16-bit keys of word x are >= c (1 <= c <= 0xffff).
__device__ __forceinline__ int count_ge2(uint32_t x, uint32_t c) { return __popc(__vcmpgeu2(x, c | (c << 16))) >> 4; }

// The k-th largest of the CTA's keys (k <= their number; padding keys are 0) and, in
// *ties, how many keys equal to it are among the k largest.  each(f) calls f(word) for
// every word of two keys this thread holds.  Nine barriers and one at the end.
template <class Each>
__device__ uint32_t kth_key16(Each each, int k, TileTopkSmem &sm, int *ties) {
  uint32_t prefix = 0;
  int round = 0;
#pragma unroll 1
  for (int b = 14; b >= 0; b -= 2, ++round) {
    const uint32_t c1 = prefix | (1u << b), c2 = prefix | (2u << b), c3 = prefix | (3u << b);
    int n1 = 0, n2 = 0, n3 = 0;
    each([&](uint32_t x) {
      n1 += count_ge2(x, c1);
      n2 += count_ge2(x, c2);
      n3 += count_ge2(x, c3);
    });
    const int4 t = block_sum4(n1, n2, n3, 0, sm, round & 1);
    prefix = t.z >= k ? c3 : t.y >= k ? c2 : t.x >= k ? c1 : prefix;
  }
  int ngt = 0;
  if (prefix < 0xffffu) each([&](uint32_t x) { ngt += count_ge2(x, prefix + 1); });
  *ties = k - block_sum4(ngt, 0, 0, 0, sm, round & 1).x;
  __syncthreads();                                    // cnt free for the next use
  return prefix;
}

__global__ void __launch_bounds__(kTileThreads) topk_tiles_kernel(const uint16_t *__restrict__ y, int N, int k,
                                                                  uint32_t *tile_max, int *counters,
                                                                  unsigned long long *pairs, uint16_t *vals,
                                                                  int32_t *idx) {
  __shared__ TileTopkSmem sm;
  griddep_wait();
  griddep_launch_dependents();
  const int sl = blockIdx.x, S = gridDim.x, m = blockIdx.y, T = N / kRows, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const uint16_t *row = y + (size_t)m * N;
  uint32_t *tmx = tile_max + (size_t)m * T;

  // ---- 1. the tile maxima (tiles 2 (tid + 256 i) and the next one in word i; loads from
  // clamped addresses, issued together), t_k, the candidate tiles
  uint32_t tw[kTileWords];
  {
    uint32_t v[2 * kTileWords];
#pragma unroll
    for (int i = 0; i < kTileWords; ++i) {
      const int t = 2 * (tid + kTileThreads * i);
      v[2 * i] = __ldcg(tmx + min(t, T - 1));
      v[2 * i + 1] = __ldcg(tmx + min(t + 1, T - 1));
    }
#pragma unroll
    for (int i = 0; i < kTileWords; ++i) {
      const int t = 2 * (tid + kTileThreads * i);
      const uint32_t lo = t < T ? v[2 * i] : 0u, hi = t + 1 < T ? v[2 * i + 1] : 0u;
      tw[i] = lo | (hi << 16);
      if (t < T) reinterpret_cast<uint32_t *>(sm.tkey)[t >> 1] = tw[i];
    }
  }
  __syncthreads();
  int unused;
  const uint32_t thr = T > k ? kth_key16([&](auto f) {
#pragma unroll
    for (int i = 0; i < kTileWords; ++i) f(tw[i]);
  }, k, sm, &unused) : 1u;
  const int tp = (T + kTileThreads - 1) / kTileThreads;
  int nmine = 0;
  for (int t = tp * tid; t < tp * tid + tp && t < T; ++t) nmine += sm.tkey[t] >= thr;
  int2 tot;
  int pos = block_scan2(nmine, 0, sm.wsum, tot).x;
  for (int t = tp * tid; t < tp * tid + tp && t < T; ++t)
    if (sm.tkey[t] >= thr) sm.cand[pos++] = (uint16_t)t;
  const int ncand = tot.x;
  __syncthreads();

  // ---- 2. this slice's candidate tiles [c0, c1): position j = 128 (c - c0) + row
  const int c0 = (int)((long long)ncand * sl / S), c1 = (int)((long long)ncand * (sl + 1) / S);
  const int n = (c1 - c0) * kRows;                     // 0 or >= 128 > k
  unsigned long long *out = pairs + ((size_t)m * S + sl) * kTopkMaxK;
  if (n > 0) {
    const bool staged = n <= kStageKeys;               // uniform
    auto raw_at = [&](int j) { return row[(int)sm.cand[c0 + (j >> 7)] * kRows + (j & (kRows - 1))]; };
    auto key_at = [&](int j) -> uint32_t { return order_key16(__ushort_as_half(raw_at(j))); };
    uint32_t lw[kStageWords];                          // word i: positions 2 (tid + 256 i), + 1
    if (staged) {
      unsigned short v[2 * kStageWords];
#pragma unroll
      for (int i = 0; i < kStageWords; ++i) {
        const int j = 2 * (tid + kTileThreads * i);
        v[2 * i] = raw_at(min(j, n - 1));
        v[2 * i + 1] = raw_at(min(j + 1, n - 1));
      }
#pragma unroll
      for (int i = 0; i < kStageWords; ++i) {
        const int j = 2 * (tid + kTileThreads * i);
        lw[i] = (j < n ? order_key16(__ushort_as_half(v[2 * i])) : 0u) |
                ((j + 1 < n ? order_key16(__ushort_as_half(v[2 * i + 1])) : 0u) << 16);
        if (j < n) reinterpret_cast<uint32_t *>(sm.lkey)[j >> 1] = lw[i];
      }
    }
    // the classification below reads the staged keys by position (each barrier of the
    // selection orders these stores before it)
    int r;
    uint32_t tkey;
    if (staged) {
      tkey = kth_key16([&](auto f) {
#pragma unroll
        for (int i = 0; i < kStageWords; ++i) f(lw[i]);
      }, k, sm, &r);
    } else {
      tkey = kth_key16([&](auto f) {
        for (int j = 2 * tid; j < n; j += 2 * kTileThreads) f(key_at(j) | (j + 1 < n ? key_at(j + 1) << 16 : 0u));
      }, k, sm, &r);
    }
    // the k best: every key above T and the first r equal to it; warp w takes positions
    // [wc w, wc w + wc), lanes consecutive, so (warp, step, lane) is index order
    auto skey = [&](int j) -> uint32_t { return staged ? (uint32_t)sm.lkey[j] : key_at(j); };
    const int wc = ((n + kTileWarps - 1) / kTileWarps + 31) / 32 * 32;
    const int jb = wc * warp, je = min(jb + wc, n);
    const unsigned lt = (1u << lane) - 1u;
    int cg = 0, ce = 0;
    for (int j = jb + lane; j - lane < je; j += 32) {
      const uint32_t x = j < je ? skey(j) : 0u;
      cg += __popc(__ballot_sync(0xffffffffu, x > tkey));
      ce += __popc(__ballot_sync(0xffffffffu, j < je && x == tkey));
    }
    if (lane == 0) {
      sm.wsum[0][warp] = cg;
      sm.wsum[1][warp] = ce;
    }
    __syncthreads();
    int sg = 0, se = 0;
#pragma unroll
    for (int w = 0; w < kTileWarps; ++w)
      if (w < warp) {
        sg += sm.wsum[0][w];
        se += sm.wsum[1][w];
      }
    for (int j = jb + lane; j - lane < je; j += 32) {
      const uint32_t x = j < je ? skey(j) : 0u;
      const unsigned bg = __ballot_sync(0xffffffffu, x > tkey);
      const unsigned be = __ballot_sync(0xffffffffu, j < je && x == tkey);
      int slot = -1;
      if (x > tkey) slot = sg + __popc(bg & lt);
      else if (j < je && x == tkey && se + __popc(be & lt) < r) slot = (k - r) + se + __popc(be & lt);
      if (slot >= 0)
        out[slot] = ((unsigned long long)x << 32) |
                    (uint32_t)((int)sm.cand[c0 + (j >> 7)] * kRows + (j & (kRows - 1)));
      sg += __popc(bg);
      se += __popc(be);
    }
  } else {
    for (int e = tid; e < k; e += kTileThreads) out[e] = 0ull;   // key 0: below every logit
  }

  // ---- 3. publish; the last slice CTA of the token ranks the pairs and clears up
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int old = atomicAdd(counters + m, 1);
    sm.last = old == S - 1;
    if (sm.last) counters[m] = 0;
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  const int total = S * k;
  const unsigned long long *all = pairs + (size_t)m * S * kTopkMaxK;
  for (int e = tid; e < total; e += kTileThreads) {
    const unsigned long long p = __ldcg(all + (size_t)(e / k) * kTopkMaxK + e % k);
    sm.mc[e] = (p & 0xffffffff00000000ull) | (0xffffffffull - (p & 0xffffffffull));
  }
  for (int t = tid; t < T; t += kTileThreads) tmx[t] = 0u;
  __syncthreads();
  // a pair's rank: how many pairs come before it (distinct composites; padding keys 0)
  for (int e = tid; e < total; e += kTileThreads) {
    const unsigned long long ce = sm.mc[e];
    int rank = 0;
#pragma unroll 16
    for (int b = 0; b < total; ++b) rank += sm.mc[b] > ce;
    if ((ce >> 32) != 0ull && rank < k) {
      const int ie = (int)(0xffffffffull - (ce & 0xffffffffull));
      vals[(size_t)m * k + rank] = row[ie];
      idx[(size_t)m * k + rank] = ie;
    }
  }
  __syncthreads();
}

size_t topk_tiles_pair_bytes(int M) { return (size_t)M * kTopkSlices * kTopkMaxK * 8; }

cudaError_t launch_topk_tiles(const uint16_t *y, int M, int N, int k, uint32_t *tile_max, int *counters,
                              unsigned long long *pairs, uint16_t *vals, int32_t *idx, cudaStream_t st) {
  // an ordinary launch: started early (programmatic dependent launch), the CTAs would be
  // placed wherever the GEMM leaves room and share a few SMs after it ends
  topk_tiles_kernel<<<dim3(kTopkSlices, M), kTileThreads, 0, st>>>(y, N, k, tile_max, counters, pairs, vals, idx);
  cudaError_t e = cudaGetLastError();
  count_launch();
  return e;
}

TopkPlan topk_plan(int M, int N, int k) {
  TopkPlan tp{};
  // slices of 2048 or 4096 elements (one or two vectors per thread), at most 64
  tp.slices = (N + 2047) / 2048;
  if (tp.slices > kTopkMaxSlices) tp.slices = kTopkMaxSlices;
  if (tp.slices < 1) tp.slices = 1;
  const int per = (N + tp.slices - 1) / tp.slices;
  tp.slice_len = (per + 2047) / 2048 * 2048;
  tp.slices = (N + tp.slice_len - 1) / tp.slice_len;
  tp.ws_counters = align_up((size_t)M * 4, 256);
  tp.ws_bytes = tp.ws_counters + (size_t)M * tp.slices * k * 8;
  return tp;
}

cudaError_t launch_topk(const uint16_t *logits, int M, int N, int k, uint16_t *vals, int32_t *idx,
                        void *ws, cudaStream_t st) {
  const TopkPlan tp = topk_plan(M, N, k);
  uint8_t *w = static_cast<uint8_t *>(ws);
  cudaError_t e = launch_pdl(reinterpret_cast<const void *>(topk_kernel), dim3(tp.slices, M),
                             dim3(kTopkThreads), 0, st, logits, N, k, tp.slice_len, vals, idx,
                             reinterpret_cast<int *>(w), reinterpret_cast<uint64_t *>(w + tp.ws_counters));
  count_launch();
  return e;
}

}  // namespace qw
