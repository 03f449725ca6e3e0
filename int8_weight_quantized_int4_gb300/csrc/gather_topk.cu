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
// One CTA per token.  Feature k of table row v sits in chunk (v / 128, k / 128) of the
// packed table, slice (k % 128) / 16, at byte (v % 128) * 16 + k % 16, stored as
// code XOR 0x80; the row's fp16 scale follows the slices.  out = fp16(code * scale),
// one rounding (__hmul_rn of two exact fp16 operands).
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
  for (int p = threadIdx.x; p < G * 8; p += blockDim.x) {       // 16 features per piece
    const int g = p >> 3, j = p & 7;
    const uint8_t *chunk = tile + (size_t)g * kChunkW8;
    const uint4 c = __ldg(reinterpret_cast<const uint4 *>(chunk + j * 2048 + r * 16));
    const __half s = __ushort_as_half(__ldg(reinterpret_cast<const unsigned short *>(chunk + 16384 + r * 2)));
    const uint32_t w[4] = {c.x ^ 0x80808080u, c.y ^ 0x80808080u, c.z ^ 0x80808080u, c.w ^ 0x80808080u};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q0 = (int)(int8_t)((w[i] >> (16 * h)) & 0xffu);
        const int q1 = (int)(int8_t)((w[i] >> (16 * h + 8)) & 0xffu);
        const __half a = __hmul_rn(__int2half_rn(q0), s), b = __hmul_rn(__int2half_rn(q1), s);
        o[2 * i + h] = (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
      }
    }
    uint4 *dst = orow + (size_t)(g * kGroup + j * 16) / 8;
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

cudaError_t launch_embed_gather(const int32_t *ids, int T, const void *packed, int V, int D,
                                uint16_t *out, int *err, cudaStream_t st) {
  cudaError_t e = launch_pdl(reinterpret_cast<const void *>(embed_gather_kernel), dim3(T), dim3(256), 0,
                             st, ids, static_cast<const uint8_t *>(packed), V, D, out, err);
  count_launch();
  return e;
}

// ------------------------------------------------------------------ top-k --
// Order: larger value first, equal values by smaller index.  key16 maps fp16 to an
// order-preserving 16-bit integer (-0 taken as +0, so the two tie); positions past N get
// key 0, which no finite fp16 value maps to.  Within a slice of at most 4096 positions an
// element is the 32-bit composite  key16 << 16 | (0xffff - local position), unique and in
// exactly that order.  The slice's k largest are found by radix selection (8-bit passes,
// histograms in shared memory) and listed in order in the workspace as 40-bit global
// composites  key16 << 24 | (2^24 - 1 - index).  The last slice CTA of a row selects
// again over the row's S k candidates as  key16 << 16 | (0xffff - slot): slices cover
// ascending index ranges and list their candidates in order, so among equal keys the
// smaller slot is the smaller index.
constexpr int kTopkThreads = 256;
constexpr int kTopkMaxK = 64;
constexpr int kTopkMaxSlices = 64;
constexpr int kTopkMaxVec = 2;                 // 16-byte vectors per thread per slice
constexpr int kTopkMerge = kTopkMaxSlices * kTopkMaxK / kTopkThreads;   // candidates per thread
static_assert(kTopkMaxSlices * kTopkMaxK <= kTopkMaxVec * 8 * kTopkThreads, "one list serves both selections");

__device__ __forceinline__ uint32_t order_key(uint16_t h) {
  if (h == 0x8000u) h = 0;                      // -0 ties with +0
  return (h & 0x8000u) ? (uint32_t)(~h & 0xffffu) : (uint32_t)(h | 0x8000u);
}

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

// Radix selection over the CTA: every thread holds n distinct 32-bit composites in c[];
// returns a threshold th such that exactly k of them are >= th: the k-th largest, or a
// prefix of it as soon as the bin holding it holds exactly the elements still wanted
// (without ties at the boundary, after the two key bytes).  The first 8-bit pass runs over
// the registers; the elements of its boundary bin (usually a small fraction) are then
// listed in shared memory and the later passes run over that list.  hist: 2 x 256 ints
// (one per pass in turn, the next one cleared while the current one fills), bc: 3 ints,
// list: room for every element of the CTA, nlist: 1 int, all shared memory.
template <int NMAX>
__device__ uint32_t select_kth(const uint32_t (&c)[NMAX], int n, int k, int *hist, int *bc,
                               uint32_t *list, int *nlist) {
  for (int b = threadIdx.x; b < 256; b += kTopkThreads) hist[b] = 0;
  if (threadIdx.x == 0) *nlist = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NMAX; ++i)
    if (i < n) atomicAdd(&hist[c[i] >> 24], 1);
  for (int b = threadIdx.x; b < 256; b += kTopkThreads) hist[256 + b] = 0;
  __syncthreads();
  if (threadIdx.x < 32) find_bin(hist, k, bc);
  __syncthreads();
  uint32_t prefix = (uint32_t)bc[0] << 24;
  int remaining = bc[1];
  if (bc[2] == remaining) return prefix;            // the bin is taken whole: done
#pragma unroll
  for (int i = 0; i < NMAX; ++i)
    if (i < n && (c[i] >> 24) == (prefix >> 24)) list[atomicAdd(nlist, 1)] = c[i];
  __syncthreads();
  const int T = *nlist;
#pragma unroll 1
  for (int pass = 1; pass < 4; ++pass) {
    int *h = hist + 256 * (pass & 1);
    int *hn = hist + 256 * ((pass + 1) & 1);
    const int shift = 24 - 8 * pass;
    const uint32_t above = 0xffffffffu << (shift + 8);   // bits already fixed
    for (int j = threadIdx.x; j < T; j += kTopkThreads) {
      const uint32_t v = list[j];
      if (((v ^ prefix) & above) == 0u) atomicAdd(&h[(v >> shift) & 0xffu], 1);
    }
    for (int b = threadIdx.x; b < 256; b += kTopkThreads) hn[b] = 0;
    __syncthreads();
    if (threadIdx.x < 32) find_bin(h, remaining, bc);
    __syncthreads();
    prefix |= (uint32_t)bc[0] << shift;
    remaining = bc[1];
    if (bc[2] == remaining) break;                   // the bin is taken whole: done
  }
  return prefix;
}

// grid (slices, rows).  ws: [M] int counters (zero between calls), then candidates
// [M][slices][k] (40-bit global composites, each slice's in order).
// At most 48 registers a thread (five CTAs an SM); the kernel runs many CTAs per row.
__global__ void __launch_bounds__(kTopkThreads, 5) topk_kernel(const uint16_t *__restrict__ logits, int N,
                                                                int k, int slice_len, uint16_t *vals,
                                                                int32_t *idx, int *counters,
                                                                uint64_t *cand) {
  __shared__ int hist[2 * 256];
  __shared__ int bc[3];
  __shared__ int nsel;
  __shared__ int nlist;
  __shared__ uint32_t list[kTopkMaxVec * 8 * kTopkThreads];   // >= kTopkMaxSlices * kTopkMaxK
  __shared__ int last;
  __shared__ uint32_t sel[kTopkMaxK];
  griddep_wait();
  griddep_launch_dependents();
  const int m = blockIdx.y, sl = blockIdx.x, S = gridDim.x;
  const uint16_t *row = logits + (size_t)m * N;
  uint64_t *rowcand = cand + (size_t)m * S * k;

  // ---- this slice: its k best (padding past N included when the slice is short)
  {
    uint32_t c[kTopkMaxVec * 8];
    const int base = sl * slice_len;
    const int nvec = slice_len / (8 * kTopkThreads);
#pragma unroll
    for (int e = 0; e < kTopkMaxVec; ++e) {
      const int lp = 8 * (threadIdx.x + kTopkThreads * e);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      const bool in = e < nvec && base + lp < N;    // N % 8 == 0: a vector is all in or all out
      if (in) v = __ldg(reinterpret_cast<const uint4 *>(row + base + lp));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t key = in ? order_key((uint16_t)(w[j >> 1] >> (16 * (j & 1)))) : 0u;
        c[8 * e + j] = (key << 16) | (0xffffu - (uint32_t)(lp + j));
      }
    }
    const uint32_t th = select_kth(c, 8 * nvec, k, hist, bc, list, &nlist);
    if (threadIdx.x == 0) nsel = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTopkMaxVec * 8; ++i)
      if (i < 8 * nvec && c[i] >= th) sel[atomicAdd(&nsel, 1)] = c[i];
    __syncthreads();
    for (int a = threadIdx.x; a < k; a += kTopkThreads) {     // listed in order
      int rank = 0;
      for (int b = 0; b < k; ++b) rank += sel[b] > sel[a];
      rowcand[(size_t)sl * k + rank] = composite(sel[a] >> 16, (uint32_t)base + (0xffffu - (sel[a] & 0xffffu)));
    }
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
  const uint32_t th = select_kth(c, nmine, k, hist, bc, list, &nlist);
  if (threadIdx.x == 0) nsel = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kTopkMerge; ++i)
    if (i < nmine && c[i] >= th) sel[atomicAdd(&nsel, 1)] = c[i];
  __syncthreads();
  // rank sort of the k winners (all distinct), largest first
  for (int a = threadIdx.x; a < k; a += kTopkThreads) {
    int rank = 0;
    for (int b = 0; b < k; ++b) rank += sel[b] > sel[a];
    const uint64_t g = __ldcg(rc + (0xffffu - (sel[a] & 0xffffu)));
    const int n = 0xffffff - (int)(g & 0xffffffu);
    idx[(size_t)m * k + rank] = n;
    vals[(size_t)m * k + rank] = row[n];
  }
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
