// attention.cu -- int8-QK causal prefill attention ("What this repo does that stock
// vLLM doesn't", paragraph "int8-QK prefill attention"): attention scores from int8
// codes of the queries and of the keys smoothed by their per-head channel mean (the
// mean shifts every score of a query row by the same amount, which the softmax
// ignores), per-row scales, softmax, and P.V in 16-bit floating point.
//
// Three launches, chained by programmatic dependent launch:
//   attn_ksum_kernel : per KV head, channel and slice of 128 keys, the sum of K in
//                      2^-24 fixed point (exact: fp16 values are multiples of 2^-24
//                      below 2^16)
//   attn_prep_kernel : the channel means (binary64 sum / S rounded to binary32); per row
//                      of K - mean and per row of Q the int8 codes and scale (amax, s =
//                      amax / 127 with an IEEE divide, code = rne(x / s)), the codes kept
//                      as fp16 (exact) for the tensor cores; V transposed to [Hkv][d][S]
//   attn_fwd_kernel  : per (128-query block, query head), over the visible 128-key
//                      blocks: S = Qc . Kc^T on tcgen05 (kind::f16; the integer dot
//                      products are exact in fp32, |sum| < 2^24), the online softmax in
//                      two groups of four warps (a query row per thread, TMEM lane =
//                      row, each group half the keys of a block and half of O), P as
//                      fp16 written into TMEM over S, O += P . V on tcgen05 with P from
//                      TMEM, O / l at the end.
#include <stdint.h>
#include <cuda_fp16.h>
#include "ptx.cuh"
#include "schedule.h"
#include "launch.h"

namespace qw {

// ------------------------------------------------------------ K channel sums --
// grid (S / 128, Hkv), kAttnD threads: thread c sums channel c of keys 128 b .. 128 b + 127.
__global__ void __launch_bounds__(kAttnD) attn_ksum_kernel(const uint16_t *__restrict__ k, int S, int Hkv,
                                                           long long *__restrict__ part) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x, g = blockIdx.y, c = threadIdx.x;
  const uint16_t *src = k + ((size_t)b * kAttnBlk * Hkv + g) * kAttnD + c;
  long long acc = 0;
#pragma unroll 8
  for (int s = 0; s < kAttnBlk; ++s) {
    // value * 2^24 is an integer below 2^40, exact in binary32 and in the conversion
    const float v = __half2float(__ushort_as_half(__ldg(src + (size_t)s * Hkv * kAttnD)));
    acc += __float2ll_rn(v * 16777216.0f);
  }
  part[((size_t)b * Hkv + g) * kAttnD + c] = acc;
}

// ------------------------------------------------------------- quantize rows --
// One warp per row of kAttnD values, eight consecutive channels per lane: amax, scale,
// codes (fp16) -- the arithmetic of the activation quantizer (s = 0 and codes 0 for a
// zero row).  x holds the row in binary32.
__device__ __forceinline__ void quant_row_warp(const float (&x)[8], uint16_t *codes, float *scale, int lane) {
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.0f);
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float q0 = s == 0.0f ? 0.0f : rintf(__fdiv_rn(x[2 * e], s));
    const float q1 = s == 0.0f ? 0.0f : rintf(__fdiv_rn(x[2 * e + 1], s));
    w[e] = h2_as_u32(__floats2half2_rn(q0, q1));    // |q| <= 127: exact
  }
  *reinterpret_cast<uint4 *>(codes + lane * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  if (lane == 0) *scale = s;
}

// Block roles (256 threads), by blockIdx.x:
//   [0, nk)            K rows: 128 rows (keys) of one KV head, 16 per warp
//   [nk, nk + nq)      Q rows: 128 rows (queries) of one query head, 16 per warp
//   [nk + nq, ...)     V transpose: a 64-key x 64-channel tile of one KV head
constexpr int kPrepThreads = 256;
constexpr int kPrepRows = 128;
static_assert(kPrepThreads == kAttnD, "one thread per channel for the means");

__global__ void __launch_bounds__(kPrepThreads) attn_prep_kernel(const uint16_t *__restrict__ q,
                                                                 const uint16_t *__restrict__ k,
                                                                 const uint16_t *__restrict__ v, int T, int S,
                                                                 int Hq, int Hkv, const long long *__restrict__ part,
                                                                 uint16_t *qc, float *qs, uint16_t *kc, float *ks,
                                                                 uint16_t *vt) {
  __shared__ float mean[kAttnD];
  __shared__ __align__(16) uint16_t tile[64][64 + 8];
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = Hkv * (S / kPrepRows), nq = Hq * (T / kPrepRows);
  int blk = blockIdx.x;
  if (blk < nk) {
    const int g = blk / (S / kPrepRows), r0 = (blk % (S / kPrepRows)) * kPrepRows;
    {
      // the mean of channel c: the exact sum (|sum| < 2^53 for S <= 8192) in binary64,
      // divided by S in binary64, rounded to binary32
      const int c = threadIdx.x;
      long long acc = 0;
      for (int b = 0; b < S / kAttnBlk; ++b) acc += __ldg(part + ((size_t)b * Hkv + g) * kAttnD + c);
      mean[c] = __double2float_rn(__ddiv_rn((double)acc * (1.0 / 16777216.0), (double)S));
    }
    __syncthreads();
    float mu[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mu[e] = mean[lane * 8 + e];
    for (int r = r0 + warp; r < r0 + kPrepRows; r += kPrepThreads / 32) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(k + ((size_t)r * Hkv + g) * kAttnD) + lane);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      float x[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(u32_as_h2(w[e]));
        x[2 * e] = __fsub_rn(f.x, mu[2 * e]);
        x[2 * e + 1] = __fsub_rn(f.y, mu[2 * e + 1]);
      }
      quant_row_warp(x, kc + ((size_t)g * S + r) * kAttnD, ks + (size_t)g * S + r, lane);
    }
    return;
  }
  blk -= nk;
  if (blk < nq) {
    const int h = blk / (T / kPrepRows), r0 = (blk % (T / kPrepRows)) * kPrepRows;
    for (int r = r0 + warp; r < r0 + kPrepRows; r += kPrepThreads / 32) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(q + ((size_t)r * Hq + h) * kAttnD) + lane);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      float x[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(u32_as_h2(w[e]));
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
      }
      quant_row_warp(x, qc + ((size_t)h * T + r) * kAttnD, qs + (size_t)h * T + r, lane);
    }
    return;
  }
  blk -= nq;
  // V transpose: tiles of 64 keys x 64 channels, (g, key tile, channel tile)
  const int ct = blk % (kAttnD / 64), kt = (blk / (kAttnD / 64)) % (S / 64), g = blk / ((kAttnD / 64) * (S / 64));
  for (int u = threadIdx.x; u < 64 * 8; u += kPrepThreads) {      // 64 keys x 8 pieces of 8 channels
    const int s = u >> 3, p = u & 7;
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(v + ((size_t)(kt * 64 + s) * Hkv + g) * kAttnD + ct * 64) + p);
    const uint16_t *e = reinterpret_cast<const uint16_t *>(&raw);
#pragma unroll
    for (int i = 0; i < 8; ++i) tile[p * 8 + i][s] = e[i];
  }
  __syncthreads();
  for (int u = threadIdx.x; u < 64 * 8; u += kPrepThreads) {      // 64 channels x 8 pieces of 8 keys
    const int c = u >> 3, p = u & 7;
    const uint4 val = *reinterpret_cast<const uint4 *>(&tile[c][p * 8]);
    *reinterpret_cast<uint4 *>(vt + ((size_t)g * kAttnD + ct * 64 + c) * S + kt * 64 + p * 8) = val;
  }
}

// ----------------------------------------------------------------- forward --
// Warps: 0 Q and K copies, 1 MMA issue, 2 V copies, 3 idle, 4-11 softmax in two groups
// (warp w reads TMEM lanes 32 (w % 4) ..; group g = (w - 4) / 4 takes keys 64 g .. 64 g + 63
// of every block and O columns 128 g ..).
// Shared memory (1024-byte aligned): Q tile, K tile, V^T tile (each 64 KB: 128-byte rows,
// 128-byte swizzle, the K dimension split into 64-element halves), then the key scales
// of two blocks, the groups' row maxima of two blocks and their row sums, the barriers.  TMEM: O [0, 256),
// S/P buffers [256, 384) and [384, 512).
constexpr int kFwdThreads = 384;
constexpr int kSmGroups = 2;
constexpr uint32_t kTileBytes = 65536;
constexpr int kSoftmaxWarp0 = 4;
constexpr uint32_t kOCol = 0, kSCol = 256;

// 2^x (ex2.approx.ftz: relative error about 2^-22, 2^-inf = 0), for the softmax weights,
// which are rounded to fp16 right after
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct AttnArgs {
  CUtensorMap tq, tk, tv;     // Qc [Hq*T][256], Kc [Hkv*S][256] (64 x 128 x 4 boxes), V^T [Hkv*256][S] (64 x 256 x 2)
  const float *qs, *ks;       // [Hq][T], [Hkv][S]
  uint16_t *out;              // [T][Hq][256]
  int T, S, Hq, Hkv;
  int *err;
  unsigned long long wait_ns;
};

__global__ void __launch_bounds__(kFwdThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (sbase - raw);
  const uint32_t q_s = sbase, k_s = sbase + kTileBytes, v_s = sbase + 2 * kTileBytes;
  float *ksm = reinterpret_cast<float *>(gbase + 3 * kTileBytes);             // [2][128]
  float *xm = ksm + 2 * kAttnBlk;                                             // [2][2][128]
  float *lx = xm + 4 * kAttnBlk;                                              // [2][128]
  const uint32_t bars = sbase + 3 * kTileBytes + 4096;
  uint8_t *gbars = gbase + 3 * kTileBytes + 4096;
  // barriers: q_full, k_full, k_empty, v_full, v_empty, s_full[2], p_full[2], s_free[2], o_step
  // (every P.V), drain, o_done (the last P.V; the output must not wait on o_step by parity,
  // which may be two phases behind then)
  const uint32_t q_full = bars, k_full = bars + 8, k_empty = bars + 16, v_full = bars + 24, v_empty = bars + 32;
  auto s_full = [&](int b) { return bars + 40u + 8u * b; };
  auto p_full = [&](int b) { return bars + 56u + 8u * b; };
  auto s_free = [&](int b) { return bars + 72u + 8u * b; };
  const uint32_t o_step = bars + 88, drain = bars + 96, o_done = bars + 104;
  volatile WaitBlock *wctl = reinterpret_cast<volatile WaitBlock *>(gbars + 112);
  volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gbars + 112 + sizeof(WaitBlock));
  auto pwait = [&](uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity, wctl, a.wait_ns == 0); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = a.T / kAttnBlk;
  const int qb = nqb - 1 - (int)(blockIdx.x / a.Hq);     // the longest rows first
  const int h = (int)(blockIdx.x % a.Hq);
  const int g = h / (a.Hq / a.Hkv);
  const int nblk = (a.S - a.T) / kAttnBlk + qb + 1;      // key blocks up to the diagonal

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_full(b), 4 * kSmGroups);
      mbar_init(s_free(b), 1);
    }
    mbar_init(o_step, 1);
    mbar_init(drain, 1);
    mbar_init(o_done, 1);
    wait_block_init(wctl, a.wait_ns, a.err);
    fence_mbar_init();
  }
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&a.tq);
      prefetch_tensormap(&a.tk);
      prefetch_tensormap(&a.tv);
    }
    tmem_alloc(smem_u32(const_cast<uint32_t *>(tslot)), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------- Q and K copies --
    // (K and V have their own copy threads, so that K of the next block is requested as
    // soon as the scores of the current one are done, whatever P . V is doing)
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_3d(q_s, &a.tq, 0, h * a.T + qb * kAttnBlk, 0, q_full);
      int nk = 0;
      for (int j = 0; j < nblk; ++j) {
        if (j > 0 && !pwait(k_empty, (uint32_t)((j - 1) & 1))) break;
        mbar_arrive_expect_tx(k_full, kTileBytes);
        tma_load_3d(k_s, &a.tk, 0, g * a.S + j * kAttnBlk, 0, k_full);
        ++nk;
      }
      // every copy has landed before the CTA may exit
      mbar_drain(q_full, 0u, wctl);
      if (nk > 0) mbar_drain(k_full, (uint32_t)((nk - 1) & 1), wctl);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------- V copies --
    if (lane == 0) {
      int nv = 0;
      for (int j = 0; j < nblk; ++j) {
        if (j > 0 && !pwait(v_empty, (uint32_t)((j - 1) & 1))) break;
        mbar_arrive_expect_tx(v_full, kTileBytes);
        tma_load_3d(v_s, &a.tv, 0, g * kAttnD, 2 * j, v_full);
        ++nv;
      }
      if (nv > 0) mbar_drain(v_full, (uint32_t)((nv - 1) & 1), wctl);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA --
    // The whole warp runs the loop (waits are warp votes) and the leader lane issues:
    // see mma_f16_ts_w.
    const uint32_t leader = elect_leader();
    auto wwait = [&](uint32_t bar, uint32_t parity) { return __all_sync(0xffffffffu, pwait(bar, parity)); };
    constexpr uint32_t kIdS = idesc_f16_f32(128, kAttnBlk), kIdO = idesc_f16_f32(128, kAttnD);
    bool ok = wwait(q_full, 0u);
    for (int j = 0; ok && j <= nblk; ++j) {
      if (j < nblk) {
        const int b = j & 1;
        if (j >= 2 && !wwait(s_free(b), (uint32_t)(((j >> 1) - 1) & 1))) { ok = false; break; }
        if (!wwait(k_full, (uint32_t)(j & 1))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kAttnD / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * (kAttnBlk * 128) + (kk & 3) * 32);
          mma_f16_ss_w(leader, tmem + kSCol + (uint32_t)(b * kAttnBlk), smem_desc_sw128(q_s + off),
                       smem_desc_sw128(k_s + off), kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(leader, s_full(b));
        mma_commit_w(leader, k_empty);
      }
      if (j >= 1) {
        const int jp = j - 1, bp = jp & 1;
        if (!wwait(p_full(bp), (uint32_t)((jp >> 1) & 1))) { ok = false; break; }
        if (!wwait(v_full, (uint32_t)(jp & 1))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kAttnBlk / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * (kAttnD * 128) + (kk & 3) * 32);
          mma_f16_ts_w(leader, tmem + kOCol, tmem + kSCol + (uint32_t)(bp * kAttnBlk + 8 * kk),
                       smem_desc_sw128(v_s + off), kIdO, (jp > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit_w(leader, s_free(bp));
        mma_commit_w(leader, v_empty);
        mma_commit_w(leader, o_step);
        if (jp == nblk - 1) mma_commit_w(leader, o_done);
      }
    }
    // every MMA the leader issued has completed before the CTA may exit
    mma_commit_w(leader, drain);
    mbar_drain(drain, 0u, wctl);
  } else if (warp >= kSoftmaxWarp0) {
    // ----------------------------------------------------------- softmax --
    const int grp = (warp - kSoftmaxWarp0) >> 2;               // 0, 1: keys 64 grp .. of a block
    const int row = ((warp - kSoftmaxWarp0) & 3) * 32 + lane;  // query row of the block (TMEM lane)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int qi = qb * kAttnBlk + row;                         // query index in the chunk
    const int pos = a.S - a.T + qi;                             // its position in the context
    const int c0 = 64 * grp;                                    // the group's first key of a block
    constexpr int kSmThreads = 4 * kSmGroups * 32;
    // score in base 2: dot * ks * qs / sqrt(d) * log2(e)
    const float arow = __ldg(a.qs + (size_t)h * a.T + qi) * (1.4426950408889634f / 16.0f);
    float m_ref = -INFINITY, l = 0.0f;
    bool aborted = false;
    // key scales of a block: thread row < 64 of group grp stages key 64 grp + row; block j + 1
    // is staged during block j (visible after that block's barrier)
    if (row < 64) ksm[c0 + row] = __ldg(a.ks + (size_t)g * a.S + c0 + row);
    named_bar_sync(1, kSmThreads);
    for (int j = 0; j < nblk; ++j) {
      const int b = j & 1;
      if (row < 64 && j + 1 < nblk)
        ksm[((j + 1) & 1) * kAttnBlk + c0 + row] = __ldg(a.ks + (size_t)g * a.S + (j + 1) * kAttnBlk + c0 + row);
      const bool got = pwait(s_full(b), (uint32_t)((j >> 1) & 1));
      tc_fence_after();
      const uint32_t sadr = tmem + lane_base + kSCol + (uint32_t)(b * kAttnBlk);
      const bool masked = j * kAttnBlk + kAttnBlk - 1 > a.S - a.T + qb * kAttnBlk;   // block meets the diagonal
      // the group's 64 scores of the row, in registers
      float x[64];
      {
        uint32_t v[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          tmem_ld32(sadr + (uint32_t)(c0 + 32 * hh), v);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) x[32 * hh + c] = __uint_as_float(v[c]);
        }
      }
      const float *kss = ksm + b * kAttnBlk + c0;
      float mloc = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float t = x[c] * kss[c] * arow;
        if (masked && j * kAttnBlk + c0 + c > pos) t = -INFINITY;
        x[c] = t;
        mloc = fmaxf(mloc, t);
      }
      xm[(b * kSmGroups + grp) * kAttnBlk + row] = mloc;
      // both groups decide together; the row maxima and the next key scales are in place,
      // and both groups' reads of S precede the P stores over it
      tc_fence_before();
      if (named_bar_or(1, kSmThreads, aborted || !got || wctl->abort)) { aborted = true; break; }
      tc_fence_after();
      const float mblk = fmaxf(mloc, xm[(b * kSmGroups + (grp ^ 1)) * kAttnBlk + row]);
      // the reference maximum moves only when the new one is 2^8 above it (P stays below
      // 256 in fp16); then O and l are rescaled, once the previous P.V is done (both
      // groups take the same decision for a row)
      float factor = 1.0f;
      bool resc = false;
      if (mblk > m_ref + 8.0f) {
        if (m_ref != -INFINITY) {
          factor = ex2_approx(m_ref - mblk);
          resc = true;
        }
        m_ref = mblk;
      }
      if (__any_sync(0xffffffffu, resc) && j > 0) {
        const bool done = __all_sync(0xffffffffu, pwait(o_step, (uint32_t)((j - 1) & 1)));
        if (!done) {
          aborted = true;
        } else {
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < kAttnD / kSmGroups; cc += 32) {
            uint32_t v[32];
            const uint32_t oadr = tmem + lane_base + kOCol + (uint32_t)(grp * (kAttnD / kSmGroups) + cc);
            tmem_ld32(oadr, v);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * factor);
            tmem_st32(oadr, v);
          }
          tmem_wait_st();
        }
      }
      l *= factor;
      if (!aborted) {
        // P = 2^(x - m_ref) as fp16 pairs, over S columns already read by both groups
        uint32_t p[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const __half2 ph = __floats2half2_rn(ex2_approx(x[c] - m_ref), ex2_approx(x[c + 1] - m_ref));
          const float2 pf = __half22float2(ph);
          l += pf.x + pf.y;
          p[c / 2] = h2_as_u32(ph);
        }
        tmem_st32(sadr + (uint32_t)(c0 / 2), p);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !aborted) mbar_arrive(p_full(b));
    }
    // ---- O / l into the output row (group grp writes columns 128 grp ..)
    const bool got = !aborted && pwait(o_done, 0u);
    lx[grp * kAttnBlk + row] = l;
    if (!named_bar_or(1, kSmThreads, !got || wctl->abort)) {
      tc_fence_after();
      const float inv = 1.0f / (l + lx[(grp ^ 1) * kAttnBlk + row]);
      uint16_t *orow = a.out + ((size_t)qi * a.Hq + h) * kAttnD + grp * (kAttnD / kSmGroups);
#pragma unroll 1
      for (int cc = 0; cc < kAttnD / kSmGroups; cc += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kOCol + (uint32_t)(grp * (kAttnD / kSmGroups) + cc), v);
        tmem_wait_ld();
        uint32_t o[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          o[c] = h2_as_u32(__floats2half2_rn(__uint_as_float(v[2 * c]) * inv, __uint_as_float(v[2 * c + 1]) * inv));
#pragma unroll
        for (int u = 0; u < 4; ++u)
          reinterpret_cast<uint4 *>(orow + cc)[u] = make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
      }
    }
  }

  // --------------------------------------------------------------- teardown --
  // the copy and MMA threads drained what they started
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t attn_fwd_smem_bytes() { return 1024 + 3 * (size_t)kTileBytes + 4096 + 256; }

cudaError_t launch_attn(const AttnLaunch &L, cudaStream_t st) {
  cudaError_t e = launch_pdl(reinterpret_cast<const void *>(attn_ksum_kernel), dim3(L.S / kAttnBlk, L.Hkv),
                             dim3(kAttnD), 0, st, L.k, L.S, L.Hkv, L.part);
  count_launch();
  if (e != cudaSuccess) return e;
  const int nk = L.Hkv * (L.S / kPrepRows), nq = L.Hq * (L.T / kPrepRows), nv = L.Hkv * (L.S / 64) * (kAttnD / 64);
  e = launch_pdl(reinterpret_cast<const void *>(attn_prep_kernel), dim3(nk + nq + nv), dim3(kPrepThreads), 0, st,
                 L.q, L.k, L.v, L.T, L.S, L.Hq, L.Hkv, static_cast<const long long *>(L.part), L.qc, L.qs, L.kc,
                 L.ks, L.vt);
  count_launch();
  if (e != cudaSuccess) return e;
  AttnArgs a{};
  a.tq = L.tq;
  a.tk = L.tk;
  a.tv = L.tv;
  a.qs = L.qs;
  a.ks = L.ks;
  a.out = L.out;
  a.T = L.T;
  a.S = L.S;
  a.Hq = L.Hq;
  a.Hkv = L.Hkv;
  a.err = L.err;
  a.wait_ns = L.wait_ns;
  const size_t smem = attn_fwd_smem_bytes();
  e = ensure_smem_attr(reinterpret_cast<const void *>(attn_fwd_kernel), (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(reinterpret_cast<const void *>(attn_fwd_kernel), dim3((L.T / kAttnBlk) * L.Hq),
                 dim3(kFwdThreads), smem, st, a);
  count_launch();
  return e;
}

}  // namespace qw
