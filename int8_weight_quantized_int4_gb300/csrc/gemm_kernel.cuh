// gemm_kernel.cuh -- the quantized linear layer on 5th-generation tensor cores.
//
// y[m,n] = sum_g s[n,g] * sum_{k in g} a[m,k] * q[n,k]   ("In full" item 4 of
// "What this repo does that stock vLLM doesn't": int4 weights, signed group-128
// scales; W8 variant for the int8 group-128 lm_head, items 1 and 5).
//
// Orientation: the weights are the MMA's A operand (M = 128 weight rows, one per
// TMEM lane) and the tokens are its N (16..256), so a decode batch of 1..64
// tokens still fills the 128-row MMA.  Per 128 x 128 weight chunk:
//   copy warps     : one issues the 1-D bulk copy of each packed chunk (codes +
//                    signed scales), another the TMA tensor copy of the matching
//                    activation tile (128-byte swizzle, zero fill past M); both
//                    complete on the stage's mbarrier
//   widen warps    : W4A8 at decode sizes only -- int8 codes -> fp16 (exact) into
//                    the swizzled tile
//   dequant warps  : int4/int8 codes -> fp16 (q * s) in registers, with the
//                    scale's sign, stored into TMEM as the A operand
//   MMA warps      : 8 x tcgen05.mma kind::f16 (K = 16 each) per chunk, fp32
//                    accumulator in TMEM; tcgen05.commit frees the stage.  For
//                    token tiles of up to 64 two warps issue alternate chunks into
//                    two accumulators (an MMA with N <= 64 costs about as much issue
//                    time as a full one, so one issuing thread cannot keep up with
//                    HBM); the epilogue adds the two in a fixed order
//   epilogue warps : tcgen05.ld the accumulator, scale by the token scale (W4A8),
//                    write fp16 y, or a binary32 partial for a tile cut by the
//                    stream-K split; the last CTA of a cut tile sums the partials
//                    in CTA order (deterministic, no waiting) once its own work
//                    is done, pulling all of them into the idle stage buffers
//                    with bulk copies in a single round trip.
#pragma once
#include <stdint.h>
#include <cuda_fp16.h>
#include "ptx.cuh"
#include "schedule.h"
#include "launch.h"

namespace qw {

constexpr int kDeqWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kWidenWarps = 4;
constexpr int kWarpEpi0 = kDeqWarps;                 // 8
constexpr int kWarpWiden0 = kWarpEpi0 + kEpiWarps;   // 12
constexpr int kWarpTma = kWarpWiden0 + kWidenWarps;  // 16
constexpr int kWarpMma = kWarpTma + 1;               // 17
constexpr int kWarpAct = kWarpMma + 1;               // 18: activation tile copies
constexpr int kWarpMma2 = kWarpAct + 1;              // 19: second MMA issuer (token tiles <= 64)
constexpr int kThreads = (kWarpMma2 + 1) * 32;       // 640
constexpr int kMaxAStages = 8;                       // TMEM A-operand ring (64 columns per stage)
constexpr int kDeqGroups = 2;                        // dequant warp groups, alternate chunks
constexpr int kDeqGroupWarps = kDeqWarps / kDeqGroups;
constexpr int kTmemCols = 512;

// offsets inside the barrier block that follows the stages
constexpr int kBarFull = 0;
constexpr int kBarEmpty = kBarFull + 8 * kMaxStages;
constexpr int kBarBFull = kBarEmpty + 8 * kMaxStages;
constexpr int kBarAFull = kBarBFull + 8 * kMaxStages;
constexpr int kBarAEmpty = kBarAFull + 8 * kMaxAStages;
constexpr int kBarAccFull = kBarAEmpty + 8 * kMaxAStages;
constexpr int kBarAccEmpty = kBarAccFull + 8 * 2;
constexpr int kBarRed = kBarAccEmpty + 8 * 2;        // stream-K reduction loads
constexpr int kTmemSlot = kBarRed + 8;
constexpr int kAbortSlot = kTmemSlot + 4;
constexpr int kBcastSlot = kAbortSlot + 4;
static_assert(kBcastSlot + 4 <= kSmemReserve - 1024, "barrier block too large");

// ---- dequantization: packed codes -> 32 half2 (64 fp16 values q*s) per thread ----

// W4: two 16-byte slices (64 codes) of one row; nibble (q + 8) at bit 4p of each
// word holds element e = 2*(p % 4) + p / 4, so the masks below yield (k, k+1) pairs.
__device__ __forceinline__ void dequant_w4(const uint4 (&v)[2], __half2 s2, uint32_t (&o)[32]) {
  const __half2 k1032 = __float2half2_rn(1032.0f);
  const __half2 k16th = __float2half2_rn(0.0625f);
  const __half2 km72 = __float2half2_rn(-72.0f);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = w[i], hi = w[i] >> 8;
      // (1024 + u) - 1032 = q  and  (1024 + 16u)/16 - 72 = q, both exact in fp16
      const __half2 q0 = __hsub2(u32_as_h2(lop3_and_or(lo, 0x000f000fu, 0x64006400u)), k1032);
      const __half2 q1 = __hfma2(u32_as_h2(lop3_and_or(lo, 0x00f000f0u, 0x64006400u)), k16th, km72);
      const __half2 q2 = __hsub2(u32_as_h2(lop3_and_or(hi, 0x000f000fu, 0x64006400u)), k1032);
      const __half2 q3 = __hfma2(u32_as_h2(lop3_and_or(hi, 0x00f000f0u, 0x64006400u)), k16th, km72);
      o[16 * j + 4 * i + 0] = h2_as_u32(__hmul2_rn(q0, s2));
      o[16 * j + 4 * i + 1] = h2_as_u32(__hmul2_rn(q1, s2));
      o[16 * j + 4 * i + 2] = h2_as_u32(__hmul2_rn(q2, s2));
      o[16 * j + 4 * i + 3] = h2_as_u32(__hmul2_rn(q3, s2));
    }
  }
}

// W8: four 16-byte slices (64 codes) of one row, bytes (q XOR 0x80) in K order.
__device__ __forceinline__ void dequant_w8(const uint4 (&v)[4], __half2 s2, uint32_t (&o)[32]) {
  const __half2 k1152 = __float2half2_rn(1152.0f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 q0 = __hsub2(u32_as_h2(__byte_perm(w[i], 0x64646464u, 0x4140)), k1152);
      const __half2 q1 = __hsub2(u32_as_h2(__byte_perm(w[i], 0x64646464u, 0x4342)), k1152);
      o[8 * j + 2 * i + 0] = h2_as_u32(__hmul2_rn(q0, s2));
      o[8 * j + 2 * i + 1] = h2_as_u32(__hmul2_rn(q1, s2));
    }
  }
}

// W4A8 at decode sizes: widen the int8 staging tile (rows of 128 codes, unswizzled,
// right after the bn x 128 fp16 tile) into the 128-byte-swizzled fp16 tile.
// (1024 + (q XOR 0x80)) - 1152 = q, exact in fp16.
template <int BN>
__device__ __forceinline__ void widen_stage(uint8_t *btile, int t, int rows) {
  const uint8_t *stg = btile + BN * kGroup * 2;
  const __half2 k1152 = __float2half2_rn(1152.0f);
#pragma unroll 2
  for (int pc = t; pc < rows * 8; pc += kWidenWarps * 32) {
    const int r = pc >> 3, c8 = pc & 7;
    const uint4 v = *reinterpret_cast<const uint4 *>(stg + pc * 16);
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u,
                           v.w ^ 0x80808080u};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w[i], 0x64646464u, 0x4140)), k1152));
      o[2 * i + 1] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w[i], 0x64646464u, 0x4342)), k1152));
    }
    // 16 codes = fp16 pieces 2*c8 and 2*c8+1 (8 values each) of row r
    const int kc = c8 >> 2;
    const int cc0 = (2 * c8) & 7;
    uint8_t *row = btile + kc * BN * 128 + r * 128;
    *reinterpret_cast<uint4 *>(row + ((cc0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4 *>(row + (((cc0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

template <int BN, int WBITS, bool TOKSCALE>
__global__ void __launch_bounds__(kThreads, 1) qgemm_tc_kernel(const __grid_constant__ GemmArgs a) {
  constexpr uint32_t kChunk = WBITS == 8 ? kChunkW8 : kChunkW4;
  constexpr uint32_t kWAligned = (kChunk + 1023) / 1024 * 1024;
  constexpr bool kAct8 = TOKSCALE && BN <= kAct8InKernelMaxBn;
  constexpr uint32_t kStage = kWAligned + BN * kGroup * 2 + (kAct8 ? BN * kGroup : 0);
  constexpr uint32_t kActBytes = kAct8 ? BN * kGroup : BN * kGroup * 2;
  constexpr int kNAcc = BN <= 128 ? 2 : 1;
  constexpr bool kDual = BN <= 64;                     // two MMA issuers, two accumulators
  constexpr int kIssuers = kDual ? 2 : 1;
  // A-operand ring depth: whatever TMEM the accumulators leave free (6 stages for
  // token tiles up to 32, 4 otherwise); accumulators start after the ring
  constexpr int kAStages = BN <= 32 ? 6 : 4;
  constexpr int kAccCol0 = kAStages * 64;
  static_assert(kAccCol0 + (kDual ? 4 : kNAcc) * BN <= kTmemCols, "TMEM budget");
  static_assert(kAStages <= kMaxAStages, "A ring");
  constexpr uint32_t kIdesc = idesc_f16_f32(128, BN);

  extern __shared__ uint8_t smem_raw[];
  const Plan &P = a.P;
  const int S = P.stages;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + (uint32_t)S * kStage;
  uint8_t *gbars = gbase + (size_t)S * kStage;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(gbars + kAbortSlot);
  volatile int *bcast = reinterpret_cast<volatile int *>(gbars + kBcastSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  auto full_bar = [&](int s) { return bars + kBarFull + 8 * s; };
  auto empty_bar = [&](int s) { return bars + kBarEmpty + 8 * s; };
  auto bfull_bar = [&](int s) { return bars + kBarBFull + 8 * s; };
  auto afull_bar = [&](int i) { return bars + kBarAFull + 8 * i; };
  auto aempty_bar = [&](int i) { return bars + kBarAEmpty + 8 * i; };
  auto accfull_bar = [&](int i) { return bars + kBarAccFull + 8 * i; };
  auto accempty_bar = [&](int i) { return bars + kBarAccEmpty + 8 * i; };
  auto w_smem = [&](int s) { return sbase + (uint32_t)s * kStage; };
  auto b_smem = [&](int s) { return sbase + (uint32_t)s * kStage + kWAligned; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 2);
      mbar_init(empty_bar(s), 1);
      mbar_init(bfull_bar(s), kWidenWarps);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(afull_bar(i), kDeqGroupWarps);
      mbar_init(aempty_bar(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(accfull_bar(i), kIssuers);
      mbar_init(accempty_bar(i), kEpiWarps);
    }
    mbar_init(bars + kBarRed, 1);
    *abort_flag = 0;
    *bcast = 0;
    fence_mbar_init();
  }
  if (warp == kWarpAct && lane == 0) prefetch_tensormap(&a.tmap);
  if (warp == 0) {
    tmem_alloc(bars + kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbars + kTmemSlot);

  Seg sg;
  // Everything above overlaps the tail of the preceding kernel (programmatic
  // dependent launch).  By default every thread waits for that kernel here, before
  // touching global memory.  When the caller has declared the packed weights
  // immutable (QW_OPT_WEIGHTS_IMMUTABLE), the weight-copy and dequant warps go
  // ahead: they read only the weights and write only shared memory and TMEM, so the
  // next layer's weights stream in while the previous kernel finishes.  The roles
  // that read activations or write global memory (activation copies, epilogue)
  // still wait first; the MMA and widen warps only consume what those produce.
  const bool early = a.early_weights != 0;
  if (!early) griddep_wait();
  griddep_launch_dependents();

  if (warp == kWarpTma) {
    // ------------------------------------------------------ weight copies --
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
        int u, t;
        tile_coords(P, sg.tile, u, t);
        const uint8_t *src = a.wpack + ((size_t)t * P.G + sg.g0) * kChunk;
        for (int g = sg.g0; g < sg.g1; ++g, src += kChunk) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, a.err)) { ok = false; break; }
          mbar_arrive_expect_tx(full_bar(s), kChunk);
          bulk_g2s(w_smem(s), src, kChunk, full_bar(s), pol);
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp == kWarpAct) {
    // -------------------------------------------------- activation copies --
    if (lane == 0) {
      if (early) griddep_wait();
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
        int u, t;
        tile_coords(P, sg.tile, u, t);
        for (int g = sg.g0; g < sg.g1; ++g) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, a.err)) { ok = false; break; }
          mbar_arrive_expect_tx(full_bar(s), kActBytes);
          if constexpr (kAct8) {
            // int8 codes: one 128 x BN box into the staging slot (unswizzled)
            tma_load_2d(b_smem(s) + BN * kGroup * 2, &a.tmap, g * kGroup, u * BN, full_bar(s));
          } else {
            // fp16: one 64 x BN x 2 box (both 64-wide halves of the group), 128-byte swizzle
            tma_load_3d(b_smem(s), &a.tmap, 0, u * BN, 2 * g, full_bar(s));
          }
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp >= kWarpWiden0 && warp < kWarpWiden0 + kWidenWarps) {
    // ------------------------------------------ W4A8 int8 -> fp16 widening --
    if constexpr (kAct8) {
      const int wt = threadIdx.x - kWarpWiden0 * 32;   // 0..127
      const int rows = P.M < BN ? P.M : BN;            // a single token tile when widening here
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
        for (int g = sg.g0; g < sg.g1; ++g) {
          if (!mbar_wait(full_bar(s), ph, abort_flag, a.err)) { ok = false; break; }
          widen_stage<BN>(gbase + (size_t)s * kStage + kWAligned, wt, rows);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bfull_bar(s));
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp < kDeqWarps) {
    // ------------------------------------------------------- dequantize --
    // Two groups of four warps take alternate chunks (CTA-wide chunk parity), so
    // two chunks are being dequantized at once; within a group each warp covers 32
    // rows (its TMEM lane quarter) over the whole 128-wide group, in two halves.
    const int quad = warp & 3, grp = warp / kDeqGroupWarps;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int s = 0, ai = 0, cidx = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
      for (int g = sg.g0; g < sg.g1; ++g, ++cidx) {
        if ((cidx & 1) == grp) {
          if (!mbar_wait(full_bar(s), ph, abort_flag, a.err)) { ok = false; break; }
          if (!mbar_wait(aempty_bar(ai), aph ^ 1u, abort_flag, a.err)) { ok = false; break; }
          const uint8_t *wc = gbase + (size_t)s * kStage;
          const uint32_t tcol = tmem + lane_base + (uint32_t)(ai * 64);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t o[32];
            if constexpr (WBITS == 4) {
              uint4 v[2];
              v[0] = *reinterpret_cast<const uint4 *>(wc + (2 * h) * 2048 + row * 16);
              v[1] = *reinterpret_cast<const uint4 *>(wc + (2 * h + 1) * 2048 + row * 16);
              const __half sc = *reinterpret_cast<const __half *>(wc + 8192 + row * 2);
              dequant_w4(v, __half2half2(sc), o);
            } else {
              uint4 v[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                v[j] = *reinterpret_cast<const uint4 *>(wc + (4 * h + j) * 2048 + row * 16);
              const __half sc = *reinterpret_cast<const __half *>(wc + 16384 + row * 2);
              dequant_w8(v, __half2half2(sc), o);
            }
            tmem_st32(tcol + (uint32_t)(h * 32), o);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(afull_bar(ai));
        }
        if (++s == S) { s = 0; ph ^= 1u; }
        if (++ai == kAStages) { ai = 0; aph ^= 1u; }
      }
    }
  } else if (warp == kWarpMma || (kDual && warp == kWarpMma2)) {
    // ------------------------------------------------------------- MMA --
    if (lane == 0) {
      const int q = warp == kWarpMma ? 0 : 1;          // issuer: chunks of CTA-wide parity q
      int s = 0, ai = 0, cidx = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
        const int b = i % kNAcc;
        if (!mbar_wait(accempty_bar(b), ((i / kNAcc) & 1) ^ 1, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(kAccCol0 + (kDual ? 2 * b + q : b) * BN);
        bool first = true;
        for (int g = sg.g0; g < sg.g1; ++g, ++cidx) {
          if (kDual && (cidx & 1) != q) {
            if (++s == S) { s = 0; ph ^= 1u; }
            if (++ai == kAStages) { ai = 0; aph ^= 1u; }
            continue;
          }
          if (!mbar_wait(afull_bar(ai), aph, abort_flag, a.err)) { ok = false; break; }
          if (!mbar_wait(kAct8 ? bfull_bar(s) : full_bar(s), ph, abort_flag, a.err)) { ok = false; break; }
          tc_fence_after();
          // descriptor start addresses advance by (offset >> 4); no carry out of the
          // 14-bit field since shared-memory addresses stay below 256 KB
          const uint64_t bdesc0 = smem_desc_sw128(b_smem(s));
          const uint32_t a0 = tmem + (uint32_t)(ai * 64);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_f16_ts(d, a0 + (uint32_t)(k * 8),
                       bdesc0 + (uint64_t)(((k >> 2) * BN * 128 + (k & 3) * 32) >> 4), kIdesc,
                       (!first || k > 0) ? 1u : 0u);
          first = false;
          mma_commit(empty_bar(s));
          mma_commit(aempty_bar(ai));
          if (++s == S) { s = 0; ph ^= 1u; }
          if (++ai == kAStages) { ai = 0; aph ^= 1u; }
        }
        if (ok) mma_commit(accfull_bar(b));
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kEpiWarps) {
    // -------------------------------------------------------- epilogue --
    if (early) griddep_wait();
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int ept = threadIdx.x - kWarpEpi0 * 32;   // 0..127
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int cidx = 0;                                   // CTA-wide index of the segment's first chunk
    int npend = 0, pend_tile[2] = {0, 0};           // cut tiles this CTA must reduce (<= 2)
    bool aborted = false;
    for (int i = 0; segment(P, cta, i, sg); ++i) {
      const int b = i % kNAcc;
      const int nch = sg.g1 - sg.g0;
      // with two issuers, accumulator q holds the segment's chunks of parity q (if any)
      const bool valid0 = !kDual || nch >= 2 || (cidx & 1) == 0;
      const bool valid1 = kDual && (nch >= 2 || (cidx & 1) == 1);
      cidx += nch;
      mbar_wait(accfull_bar(b), (i / kNAcc) & 1, abort_flag, a.err);
      named_bar_sync(1, kEpiWarps * 32);           // all four warps decide together
      if (*abort_flag) { aborted = true; break; }
      tc_fence_after();
      int u, t;
      tile_coords(P, sg.tile, u, t);
      const int n = t * kRows + row;
      const int m0 = u * BN;
      const int mv = P.M - m0 < BN ? P.M - m0 : BN;   // valid tokens of this tile
      const uint32_t tacc = tmem + lane_base + (uint32_t)(kAccCol0 + (kDual ? 2 * b : b) * BN);
      float *part = sg.slot >= 0 ? a.partials + (size_t)sg.slot * (BN * kRows) : nullptr;
      constexpr int W = kDual ? 16 : 32;              // columns per TMEM load
#pragma unroll 1
      for (int cc = 0; cc < BN; cc += W) {
        uint32_t v[32], v1[32];
        if constexpr (kDual) {
          tmem_ld16(tacc + (uint32_t)cc, v);
          tmem_ld16(tacc + (uint32_t)(BN + cc), v1);
        } else {
          tmem_ld32(tacc + (uint32_t)cc, v);
        }
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < W; ++j) {
          float acc = valid0 ? __uint_as_float(v[j]) : 0.0f;
          if (kDual && valid1) acc += __uint_as_float(v1[j]);
          if (cc + j < mv) {
            if (part) {
              part[(cc + j) * kRows + row] = acc;
            } else {
              const int m = m0 + cc + j;
              const float val = TOKSCALE ? acc * a.xs[m] : acc;
              a.y[(size_t)m * P.N + n] = __half_as_ushort(__float2half_rn(val));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accempty_bar(b));
      if (part) {
        // publish this partial: the barrier orders every thread's partial stores
        // before one thread's device-scope acquire-release add, which also makes the
        // other contributors' partials visible to the last one, who reduces the tile
        named_bar_sync(1, kEpiWarps * 32);
        int pf, pl;
        tile_contributors(P, sg.tile, pf, pl);
        if (ept == 0) {
          const int old = atom_add_acq_rel_gpu(a.counters + sg.tile, 1);
          const int last = (old == pl - pf) ? 1 : 0;
          if (last) a.counters[sg.tile] = 0;    // leave the workspace zeroed for the next call
          *bcast = last;
        }
        named_bar_sync(1, kEpiWarps * 32);
        if (*bcast) pend_tile[npend++] = sg.tile;    // reduced once this CTA's own work is done
      }
    }
    // ---- stream-K reductions: all MMAs of this CTA have completed (its last
    // accumulator was read), so every stage buffer is idle.  Pull the contributors'
    // partials of each cut tile this CTA finished last into shared memory with
    // bulk copies (all in flight at once), then sum them in CTA order.
    uint32_t red_phase = 0;
    const uint32_t avail = (uint32_t)S * kStage;
    for (int r = 0; r < npend && !aborted; ++r) {
      const int tile = pend_tile[r];
      int pf, pl, u, t;
      tile_contributors(P, tile, pf, pl);
      tile_coords(P, tile, u, t);
      const int n = t * kRows + row;
      const int m0 = u * BN;
      const int mv = P.M - m0 < BN ? P.M - m0 : BN;
      const int nseg = pl - pf + 1;
      int jt = (int)(avail / ((uint32_t)nseg * kRows * 4));   // tokens per pass
      if (jt > mv) jt = mv;
      for (int j0 = 0; j0 < mv; j0 += jt) {
        const int jn = mv - j0 < jt ? mv - j0 : jt;
        const uint32_t bytes = (uint32_t)jn * kRows * 4;
        if (ept == 0) {
          fence_proxy_async_all();
          mbar_arrive_expect_tx(bars + kBarRed, bytes * nseg);
          for (int p = pf; p <= pl; ++p)
            bulk_g2s_nohint(sbase + (uint32_t)(p - pf) * bytes,
                            a.partials + (size_t)partial_slot(P, p, tile) * (BN * kRows) + (size_t)j0 * kRows,
                            bytes, bars + kBarRed);
        }
        if (!mbar_wait(bars + kBarRed, red_phase, abort_flag, a.err)) { aborted = true; break; }
        red_phase ^= 1u;
        const float *buf = reinterpret_cast<const float *>(gbase);
        for (int j = 0; j < jn; ++j) {
          float acc = 0.0f;
          for (int p = 0; p < nseg; ++p) acc += buf[(size_t)p * jn * kRows + (size_t)j * kRows + row];
          const int m = m0 + j0 + j;
          const float val = TOKSCALE ? acc * a.xs[m] : acc;
          a.y[(size_t)m * P.N + n] = __half_as_ushort(__float2half_rn(val));
        }
        named_bar_sync(1, kEpiWarps * 32);          // buffer free before the next pass
      }
    }
  }

  // --------------------------------------------------------------- teardown --
  __syncthreads();
  if (*abort_flag) {
    // let bulk copies and MMAs already issued land before the memory goes away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace qw
