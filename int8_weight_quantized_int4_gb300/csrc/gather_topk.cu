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
// candidate tiles, exactly k of them unless maxima tie.  One CTA per token:
//   1. the k largest tile maxima (radix selection over composites key << 16 | 0xffff - t)
//      give t_k; with at most k tiles every tile is a candidate;
//   2. the candidate tiles are listed in ascending order (per-warp ballots);
//   3. the k largest logits of the candidate tiles are selected kTileBatch tiles at a
//      time, the winners so far (all at smaller indices than the batch) listed first in
//      index order, so that list positions follow the indices and the composites
//      key << 16 | 0xffff - position order ties by the smaller index;
//   4. the winners are written largest first.
// The tile maxima are cleared on the way (zero again for the next call).
constexpr int kTileBatch = 64;
constexpr int kTileSel = (kTileBatch * kRows + kTopkMaxK + kTopkThreads - 1) / kTopkThreads;   // per thread
constexpr int kMaxTiles = kTopkMaxN / kRows;
constexpr int kTilesPer = kMaxTiles / kTopkThreads;                                           // 8
static_assert(kTileSel * kTopkThreads <= 65536 && kMaxTiles <= 65536, "16-bit list positions");

struct TileTopkSmem {
  TopkSmemT<kTileSel * kTopkThreads> s;
  uint16_t cand[kMaxTiles];
  int wcount[kTopkThreads / 32];
  uint32_t thr;
  uint32_t run_key[kTopkMaxK], nxt_key[kTopkMaxK];   // winners so far, in index order
  uint16_t run_val[kTopkMaxK], nxt_val[kTopkMaxK];
  int run_idx[kTopkMaxK], nxt_idx[kTopkMaxK];
};

__global__ void __launch_bounds__(kTopkThreads) topk_tiles_kernel(const uint16_t *__restrict__ y, int N, int k,
                                                                  uint32_t *tile_max, uint16_t *vals,
                                                                  int32_t *idx) {
  __shared__ TileTopkSmem sm;
  griddep_wait();
  griddep_launch_dependents();
  const int m = blockIdx.x, T = N / kRows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint16_t *row = y + (size_t)m * N;
  uint32_t *tmx = tile_max + (size_t)m * T;

  // ---- 1. the tile maxima (tile tid + 256 i in tk[i]), cleared for the next call
  uint32_t tk[kTilesPer];
#pragma unroll
  for (int i = 0; i < kTilesPer; ++i) {
    const int t = tid + kTopkThreads * i;
    tk[i] = t < T ? __ldcg(tmx + t) : 0u;
  }
#pragma unroll
  for (int i = 0; i < kTilesPer; ++i) {
    const int t = tid + kTopkThreads * i;
    if (t < T) tmx[t] = 0u;
  }
  if (tid == 0) sm.thr = T > k ? 0xffffffffu : 0u;
  if (T > k) {
    uint32_t c[kTilesPer];
#pragma unroll
    for (int i = 0; i < kTilesPer; ++i) c[i] = (tk[i] << 16) | (0xffffu - (uint32_t)(tid + kTopkThreads * i));
    select_regs(c, T > tid ? (T - 1 - tid) / kTopkThreads + 1 : 0, k, sm.s);
    if (tid < k) atomicMin(&sm.thr, sm.s.sel[tid] >> 16);
  }
  __syncthreads();
  const uint32_t thr = sm.thr;

  // ---- 2. candidate tiles, ascending
  int ncand = 0;
#pragma unroll
  for (int i = 0; i < kTilesPer; ++i) {
    if (kTopkThreads * i >= T) break;                // uniform
    const int t = tid + kTopkThreads * i;
    const bool flag = t < T && tk[i] >= thr;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    if (lane == 0) sm.wcount[warp] = __popc(bal);
    __syncthreads();
    int off = ncand, tot = 0;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
      off += w < warp ? sm.wcount[w] : 0;
      tot += sm.wcount[w];
    }
    if (flag) sm.cand[off + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)t;
    ncand += tot;
    __syncthreads();
  }

  // ---- 3. the k best logits of the candidate tiles, a batch of tiles at a time
  int nrun = 0;
  for (int b0 = 0; b0 < ncand; b0 += kTileBatch) {
    const int nb = ncand - b0 < kTileBatch ? ncand - b0 : kTileBatch;
    const int total = nrun + nb * kRows;             // >= 128 > k
    uint32_t c[kTileSel];
#pragma unroll
    for (int e = 0; e < kTileSel; ++e) {
      const int j = tid + kTopkThreads * e;
      uint32_t key = 0u;
      if (j < nrun) {
        key = sm.run_key[j];
      } else if (j < total) {
        const int q = j - nrun;
        key = order_key16(__ushort_as_half(row[(int)sm.cand[b0 + (q >> 7)] * kRows + (q & (kRows - 1))]));
      }
      c[e] = (key << 16) | (0xffffu - (uint32_t)j);
    }
    select_regs(c, total > tid ? (total - 1 - tid) / kTopkThreads + 1 : 0, k, sm.s);
    if (tid < k) {
      const uint32_t comp = sm.s.sel[tid];
      const int j = 0xffff - (int)(comp & 0xffffu);
      uint16_t v;
      int g;
      if (j < nrun) {
        v = sm.run_val[j];
        g = sm.run_idx[j];
      } else {
        const int q = j - nrun;
        g = (int)sm.cand[b0 + (q >> 7)] * kRows + (q & (kRows - 1));
        v = row[g];
      }
      int r = 0;                                     // rank by list position = by index
      for (int b = 0; b < k; ++b) r += (0xffff - (int)(sm.s.sel[b] & 0xffffu)) < j;
      sm.nxt_key[r] = comp >> 16;
      sm.nxt_val[r] = v;
      sm.nxt_idx[r] = g;
    }
    __syncthreads();
    if (tid < k) {
      sm.run_key[tid] = sm.nxt_key[tid];
      sm.run_val[tid] = sm.nxt_val[tid];
      sm.run_idx[tid] = sm.nxt_idx[tid];
    }
    nrun = k;
    __syncthreads();
  }

  // ---- 4. largest first (winners in index order: position breaks ties)
  if (tid < k) sm.s.sel[tid] = (sm.run_key[tid] << 16) | (0xffffu - (uint32_t)tid);
  __syncthreads();
  if (tid < k) {
    const int r = rank_of(sm.s.sel, k, tid);
    vals[(size_t)m * k + r] = sm.run_val[tid];
    idx[(size_t)m * k + r] = sm.run_idx[tid];
  }
}

cudaError_t launch_topk_tiles(const uint16_t *y, int M, int N, int k, uint32_t *tile_max, uint16_t *vals,
                              int32_t *idx, cudaStream_t st) {
  cudaError_t e = launch_pdl(reinterpret_cast<const void *>(topk_tiles_kernel), dim3(M), dim3(kTopkThreads), 0,
                             st, y, N, k, tile_max, vals, idx);
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
