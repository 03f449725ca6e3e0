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
//                    signed scales) into the weight ring, another one TMA tensor
//                    copy per block of up to four groups of activations (128-byte
//                    swizzle, zero fill past M) into the activation ring
//   widen warps    : W4A8 at decode sizes only -- int8 codes -> fp16 (exact) into
//                    the swizzled tile
//   dequant warps  : int4/int8 codes -> fp16 (q * s) in registers, with the
//                    scale's sign, stored into TMEM as the A operand
//   MMA warps      : 8 x tcgen05.mma kind::f16 (K = 16 each) per chunk, fp32
//                    accumulator in TMEM; tcgen05.commit frees the operands.  An
//                    MMA holds a lone issuing lane ~34 ns whatever its N (a converged
//                    warp ~9 ns: the form used on tiles of 64 tokens and more), so
//                    one issuer cannot keep up with HBM on small token tiles: up to
//                    four warps issue chunks round-robin into their own accumulators
//                    (4 for token tiles <= 32, 2 for 64, as TMEM allows), and the
//                    epilogue adds them in a fixed order
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
constexpr int kWidenWarps = 2;
constexpr int kMaxIssuers = 4;
constexpr int kWarpEpi0 = kDeqWarps;                 // 8
constexpr int kWarpWiden0 = kWarpEpi0 + kEpiWarps;   // 12
constexpr int kWarpTma = kWarpWiden0 + kWidenWarps;  // 14: weight chunk copies
constexpr int kWarpAct = kWarpTma + 1;               // 15: activation block copies
constexpr int kWarpMma0 = kWarpAct + 1;              // 16..19: MMA issuers
constexpr int kThreads = (kWarpMma0 + kMaxIssuers) * 32;   // 640
constexpr int kMaxAStages = 8;                       // TMEM A-operand ring (64 columns per stage)
constexpr int kDeqGroups = 2;                        // dequant warp groups, alternate chunks
constexpr int kDeqGroupWarps = kDeqWarps / kDeqGroups;
constexpr int kTmemCols = 512;

// offsets inside the barrier block that follows the rings
constexpr int kBarWFull = 0;                                  // weight ring
constexpr int kBarWEmpty = kBarWFull + 8 * kMaxWStages;
constexpr int kBarXFull = kBarWEmpty + 8 * kMaxWStages;       // activation ring
constexpr int kBarXEmpty = kBarXFull + 8 * kMaxXStages;
constexpr int kBarBFull = kBarXEmpty + 8 * kMaxXStages;       // W4A8: block widened
constexpr int kBarAFull = kBarBFull + 8 * kMaxXStages;        // TMEM A ring
constexpr int kBarAEmpty = kBarAFull + 8 * kMaxAStages;
constexpr int kBarAccFull = kBarAEmpty + 8 * kMaxAStages;
constexpr int kBarAccEmpty = kBarAccFull + 8 * 2;
constexpr int kBarRed = kBarAccEmpty + 8 * 2;        // stream-K reduction loads
constexpr int kBarDrain = kBarRed + 8;               // the issuers' last MMAs completed
constexpr int kWaitSlot = kBarDrain + 8;             // WaitBlock (abort flag, limit, error word)
constexpr int kTmemSlot = kWaitSlot + (int)sizeof(WaitBlock);
constexpr int kBcastSlot = kTmemSlot + 4;
static_assert(kWaitSlot % 8 == 0 && kBcastSlot + 4 <= kSmemReserve - 1024, "barrier block too large");

// ---- dequantization: packed codes -> 32 half2 (64 fp16 values q*s) per thread ----

// W4: the four 16-byte vectors (lane quarters c = 0..3) of one K half of row R (see
// the packer): word w of vector c holds the codes at k0 = 16 w + 2 c (+ 64 h), k0 + 1
// (nibbles 0 and 4) and k0 + 8, k0 + 9 (nibbles 1 and 5) of the row block's lower row;
// the upper row (R % 16 >= 8) reads the same word shifted right by 8.  TMEM column
// (k0 - 64 h) / 2 = 8 w + c holds the pair (k0, k0 + 1), column 8 w + c + 4 the pair
// (k0 + 8, k0 + 9).
__device__ __forceinline__ void dequant_w4(const uint4 (&v)[4], int sh, __half2 s2, uint32_t (&o)[32]) {
  const __half2 k1032 = __float2half2_rn(1032.0f);
  const __half2 k16th = __float2half2_rn(0.0625f);
  const __half2 km72 = __float2half2_rn(-72.0f);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w[4] = {v[c].x >> sh, v[c].y >> sh, v[c].z >> sh, v[c].w >> sh};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // (1024 + u) - 1032 = q  and  (1024 + 16u)/16 - 72 = q, both exact in fp16
      const __half2 q0 = __hsub2(u32_as_h2(lop3_and_or(w[i], 0x000f000fu, 0x64006400u)), k1032);
      const __half2 q1 = __hfma2(u32_as_h2(lop3_and_or(w[i], 0x00f000f0u, 0x64006400u)), k16th, km72);
      o[8 * i + c] = h2_as_u32(__hmul2_rn(q0, s2));
      o[8 * i + c + 4] = h2_as_u32(__hmul2_rn(q1, s2));
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

// W4A8 at decode sizes: widen one int8 staging tile (rows of 128 codes, unswizzled)
// into the 128-byte-swizzled fp16 tile of the same chunk.
// (1024 + (q XOR 0x80)) - 1152 = q, exact in fp16.
template <int BN, int NT>
__device__ __forceinline__ void widen_chunk(uint8_t *btile, const uint8_t *stg, int t, int rows) {
  const __half2 k1152 = __float2half2_rn(1152.0f);
#pragma unroll 2
  for (int pc = t; pc < rows * 8; pc += NT) {
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

// TOKSCALE: W4A8, the epilogue multiplies by the token scales.  ACT8: the activations
// are int8 codes, widened to fp16 in the kernel; otherwise fp16 tiles (fp16 x, or W4A8
// codes already in fp16).  TMAX: the epilogue also raises the per-tile maxima of the
// lm_head's fused top-k.
template <int BN, int WBITS, bool TOKSCALE, bool TMAX, bool ACT8>
__global__ void __launch_bounds__(kThreads, 1) qgemm_tc_kernel(const __grid_constant__ GemmArgs a) {
  static_assert(!TMAX || !TOKSCALE, "the lm_head's fused top-k is W4A16 or W8A16");
  static_assert(!ACT8 || (TOKSCALE && BN <= kAct8InKernelMaxBn), "int8 codes are widened for small tiles");
  constexpr uint32_t kChunk = WBITS == 8 ? kChunkW8 : kChunkW4;
  constexpr uint32_t kWStage = (kChunk + 127) / 128 * 128;
  static_assert(kChunk % 128 == 0, "weight slots stay 128-byte aligned");
  constexpr bool kAct8 = ACT8;
  constexpr int kXBlock = act_block(BN);                 // chunks per activation copy
  constexpr uint32_t kXChunk = BN * kGroup * 2;          // one fp16 tile (two swizzled halves)
  constexpr uint32_t kXStage = kXBlock * (kXChunk + (kAct8 ? BN * kGroup : 0));
  constexpr uint32_t kXBytes = kXBlock * (kAct8 ? BN * kGroup : kXChunk);   // per copy
  // MMA issuers, one accumulator each: a chunk's 8 MMAs hold a lone issuing lane
  // ~0.3 us (a converged warp ~0.1 us) and complete ~0.1 us after their commit --
  // several issuers keep the weight stream going (one measured 17 % slower at 64 tokens
  // even in the warp form); TMEM holds issuers x accumulator sets x BN columns plus the
  // A ring.
  constexpr int kNAcc = BN <= 128 ? 2 : 1;             // accumulator sets (double buffer)
  constexpr int kIssuers = BN <= 32 ? 4 : BN <= 64 ? 2 : 1;
  static_assert(kIssuers <= kMaxIssuers && (kIssuers & (kIssuers - 1)) == 0, "issuers");
  // The single-thread roles (copies, MMA issue) run as whole warps, the leader lane
  // issuing (see mma_f16_ts_w), on token tiles of 64 and more: a tcgen05.mma issued
  // that way costs a third of one issued by a lone lane.  On narrower tiles (four
  // issuers, the weight stream the limit) lane 0 runs them alone: every lane of six
  // warps polling the barriers measured 3 % slower there.
  constexpr bool kWarpIssue = kIssuers <= 2;
  // W4A8 widening: the two widen warps, plus the two issuer warps left idle when a
  // token tile needs at most two issuers
  constexpr int kWidenW = kIssuers <= 2 ? kWidenWarps + 2 : kWidenWarps;
  // A-operand ring: whatever TMEM the accumulators leave free (64 columns a stage),
  // in two halves, one per chunk parity (see the ring note below)
  constexpr int kAccCols = kNAcc * kIssuers * BN;
  constexpr int kAStagesFit = (kTmemCols - kAccCols) / 64;
  constexpr int kAStages = (kAStagesFit < kMaxAStages ? kAStagesFit : kMaxAStages) & ~1;
  constexpr int kAHalf = kAStages / 2;
  constexpr int kAccCol0 = kAStages * 64;
  static_assert(kAHalf >= 1 && kAccCol0 + kAccCols <= kTmemCols, "TMEM budget");
  constexpr uint32_t kIdesc = idesc_f16_f32(128, BN);

  extern __shared__ uint8_t smem_raw[];
  const Plan &P = a.P;
  const int SW = P.stages, SX = P.xstages;
  // Ring note.  A waiter on a slot's barrier by phase parity must not be able to
  // wait for fill n+1 while fill n is still pending.  Chunks alternate between the
  // two dequant groups by parity, so the weight ring and the TMEM A ring are split
  // into one half per parity: every slot has one producer that fills it in order.
  // The weight half has one consumer (its group).  An A slot is read by the issuers
  // of chunks c, c + 2 kAHalf, ... in turn; an issuer reaching chunk c has already
  // seen chunk c - 2 of the same half complete, which the group filled after chunk
  // c - 2 kAHalf, so the previous fill of the slot is complete too.  Every issuer
  // and the widen warps wait on every activation block, whether or not they use it.
  const int SWH = SW >> 1;                                   // weight slots per parity
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (sbase - raw);
  // activation ring first (1024-byte aligned slots for the swizzle), then weights
  const uint32_t wbase = sbase + (uint32_t)SX * kXStage;
  const uint32_t ring_bytes = (uint32_t)SX * kXStage + (uint32_t)SW * kWStage;
  const uint32_t bars = sbase + ring_bytes;
  uint8_t *gbars = gbase + ring_bytes;
  volatile WaitBlock *wctl = reinterpret_cast<volatile WaitBlock *>(gbars + kWaitSlot);
  volatile int *bcast = reinterpret_cast<volatile int *>(gbars + kBcastSlot);
  // a pipeline wait: bounded by the launch's limit, gives up once the CTA aborts
  auto pwait = [&](uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity, wctl, a.wait_ns == 0); };
  // the same in a single-thread role: run as a whole warp, every lane waits and the warp
  // goes on only if all saw the phase (their waits may end differently after an abort)
  auto vwait = [&](uint32_t bar, uint32_t parity) {
    const bool got = pwait(bar, parity);
    if constexpr (kWarpIssue) return __all_sync(0xffffffffu, got) != 0;
    else return got;
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  auto wfull_bar = [&](int s) { return bars + kBarWFull + 8 * s; };
  auto wempty_bar = [&](int s) { return bars + kBarWEmpty + 8 * s; };
  auto xfull_bar = [&](int s) { return bars + kBarXFull + 8 * s; };
  auto xempty_bar = [&](int s) { return bars + kBarXEmpty + 8 * s; };
  auto bfull_bar = [&](int s) { return bars + kBarBFull + 8 * s; };
  auto afull_bar = [&](int i) { return bars + kBarAFull + 8 * i; };
  auto aempty_bar = [&](int i) { return bars + kBarAEmpty + 8 * i; };
  auto accfull_bar = [&](int i) { return bars + kBarAccFull + 8 * i; };
  auto accempty_bar = [&](int i) { return bars + kBarAccEmpty + 8 * i; };
  auto w_smem = [&](int s) { return wbase + (uint32_t)s * kWStage; };
  auto x_smem = [&](int s) { return sbase + (uint32_t)s * kXStage; };

  // Warm the constant cache with this CTA's schedule entries (read by every role's
  // first segment() call), so that the miss overlaps the set-up below.
  if (threadIdx.x == 64) {
    const int warm = P.begin[cta] + P.begin[cta + 1] + P.cut[cta][0] + P.cut[cta][1];
    asm volatile("" ::"r"(warm));
  }
  // Barrier set-up spread over two warps (lane l initializes the l-th barrier of
  // each ring), each initializing thread fencing its own inits.
  if (threadIdx.x >= 32 && threadIdx.x < 64) {
    const int l = threadIdx.x - 32;
    if (l < SW) {
      mbar_init(wfull_bar(l), 1);
      mbar_init(wempty_bar(l), kDeqGroupWarps);
    }
    if (l < SX) {
      mbar_init(xfull_bar(l), 1);
      mbar_init(xempty_bar(l), kIssuers);
      mbar_init(bfull_bar(l), kWidenW);
    }
    fence_mbar_init();
  } else if (threadIdx.x >= 96 && threadIdx.x < 128) {
    const int l = threadIdx.x - 96;
    if (l < kAStages) {
      mbar_init(afull_bar(l), kDeqGroupWarps);
      mbar_init(aempty_bar(l), 1);
    }
    if (l < 2) {
      mbar_init(accfull_bar(l), kIssuers);
      mbar_init(accempty_bar(l), kEpiWarps);
    }
    if (l == 2) mbar_init(bars + kBarRed, 1);
    if (l == 3) mbar_init(bars + kBarDrain, kIssuers);
    if (l == 5) {
      wait_block_init(wctl, a.wait_ns, a.err);
      *bcast = 0;
    }
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
  // next layer's weights stream in and are dequantized while the previous kernel
  // finishes.  The roles that read activations or write global memory (activation
  // copies, epilogue) still wait first; the MMA and widen warps only consume what
  // those produce.
  const bool early = a.early_weights != 0;
  if (!early) griddep_wait();
  griddep_launch_dependents();

  if (warp == kWarpTma) {
    // ------------------------------------------------------ weight copies --
    if (kWarpIssue || lane == 0) {
      const uint32_t leader = kWarpIssue ? elect_leader() : 1u;
      // a chunk read by one token tile streams through L2 (evict first); with several
      // token tiles the CTAs of a supergroup read it within a short time, so it stays
      const uint64_t pol = P.U > 1 ? policy_evict_normal() : policy_evict_first();
      int s[2] = {0, 0}, nfill[2] = {0, 0}, cidx = 0;
      uint32_t ph[2] = {0, 0};
      bool ok = true;
      for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
        int u, t;
        tile_coords(P, sg.tile, u, t);
        const uint8_t *src = a.wpack + ((size_t)t * P.G + sg.g0) * kChunk;
        for (int g = sg.g0; g < sg.g1; ++g, ++cidx, src += kChunk) {
          const int p = cidx & 1, slot = p * SWH + s[p];
          if (!vwait(wempty_bar(slot), ph[p] ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx_w(leader, wfull_bar(slot), kChunk);
          bulk_g2s_w(leader, w_smem(slot), src, kChunk, wfull_bar(slot), pol);
          ++nfill[p];
          if (++s[p] == SWH) { s[p] = 0; ph[p] ^= 1u; }
        }
      }
      // the last fill of every slot has landed before the CTA may exit
      for (int p = 0; p < 2; ++p)
        for (int j = 0; j < SWH && j < nfill[p]; ++j)
          mbar_drain(wfull_bar(p * SWH + j), j < s[p] ? ph[p] : ph[p] ^ 1u, wctl);
    }
  } else if (warp == kWarpAct) {
    // -------------------------------------------------- activation copies --
    // one tensor copy per block of up to kXBlock consecutive groups of a segment;
    // a block that runs past the segment (or past K) brings data nobody reads
    if (kWarpIssue || lane == 0) {
      const uint32_t leader = kWarpIssue ? elect_leader() : 1u;
      if (early) griddep_wait();
      int s = 0, nfill = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
        int u, t;
        tile_coords(P, sg.tile, u, t);
        for (int g = sg.g0; g < sg.g1; g += kXBlock) {
          if (!vwait(xempty_bar(s), ph ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx_w(leader, xfull_bar(s), kXBytes);
          ++nfill;
          if constexpr (kAct8) {
            // int8 codes: a 128 x BN x kXBlock box into the staging tiles (unswizzled)
            tma_load_3d_w(leader, x_smem(s) + kXBlock * kXChunk, &a.tmap, 0, u * BN, g, xfull_bar(s));
          } else {
            // fp16: a 64 x BN x (2 kXBlock) box, both 64-wide halves of every group,
            // 128-byte swizzle
            tma_load_3d_w(leader, x_smem(s), &a.tmap, 0, u * BN, 2 * g, xfull_bar(s));
          }
          if (++s == SX) { s = 0; ph ^= 1u; }
        }
      }
      for (int j = 0; j < SX && j < nfill; ++j) mbar_drain(xfull_bar(j), j < s ? ph : ph ^ 1u, wctl);
    }
  } else if ((warp >= kWarpWiden0 && warp < kWarpWiden0 + kWidenWarps) ||
             (kWidenW > kWidenWarps && warp >= kWarpMma0 + 2)) {
    // ------------------------------------------ W4A8 int8 -> fp16 widening --
    if constexpr (kAct8) {
      const int wt = warp < kWarpTma ? threadIdx.x - kWarpWiden0 * 32                 // 0..63
                                     : kWidenWarps * 32 + threadIdx.x - (kWarpMma0 + 2) * 32;
      const int rows = P.M < BN ? P.M : BN;            // a single token tile when widening here
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
        for (int g = sg.g0; g < sg.g1; g += kXBlock) {
          // the lanes leave together (their waits may end differently after an abort)
          if (!__all_sync(0xffffffffu, pwait(xfull_bar(s), ph))) { ok = false; break; }
          const int nb = sg.g1 - g < kXBlock ? sg.g1 - g : kXBlock;
          uint8_t *xs = gbase + (size_t)s * kXStage;
          for (int j = 0; j < nb; ++j)
            widen_chunk<BN, kWidenW * 32>(xs + j * kXChunk, xs + kXBlock * kXChunk + j * (BN * kGroup), wt, rows);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bfull_bar(s));
          if (++s == SX) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp < kDeqWarps) {
    // ------------------------------------------------------- dequantize --
    // Two groups of four warps take alternate chunks (CTA-wide chunk parity), so
    // two chunks are being dequantized at once; within a group each warp covers 32
    // rows (its TMEM lane quarter) over the whole 128-wide group, in two halves.
    // The weight slot is handed back as soon as it has been read.
    const int quad = warp & 3, grp = warp / kDeqGroupWarps;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int s = 0, ai = 0, cidx = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
      for (int g = sg.g0; g < sg.g1; ++g, ++cidx) {
        if ((cidx & 1) == grp) {
          const int slot = grp * SWH + s, aslot = grp * kAHalf + ai;
          // the lanes leave together: the TMEM stores below are warp-collective
          bool got = pwait(aempty_bar(aslot), aph ^ 1u);
          got = got && pwait(wfull_bar(slot), ph);
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
          const uint8_t *wc = gbase + (size_t)SX * kXStage + (size_t)slot * kWStage;
          const uint32_t tcol = tmem + lane_base + (uint32_t)(aslot * 64);
          uint32_t o[2][32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if constexpr (WBITS == 4) {
              // row = 16 b + i (+ 8 for the upper eight rows of block b)
              const int rb = row >> 4, ri = row & 7, up = (row >> 3) & 1;
              uint4 v[4];
#pragma unroll
              for (int c = 0; c < 4; ++c)
                v[c] = *reinterpret_cast<const uint4 *>(wc + (((rb * 2 + h) * 4 + c) * 8 + (ri ^ (2 * c))) * 16);
              const __half sc = *reinterpret_cast<const __half *>(wc + 8192 + (rb * 8 + ri) * 4 + up * 2);
              dequant_w4(v, up * 8, __half2half2(sc), o[h]);
            } else {
              uint4 v[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                v[j] = *reinterpret_cast<const uint4 *>(wc + (4 * h + j) * 2048 + row * 16);
              const __half sc = *reinterpret_cast<const __half *>(wc + 16384 + row * 2);
              dequant_w8(v, __half2half2(sc), o[h]);
            }
            if (h == 1) {
              // every lane's reads of the slot are done (their results are in registers)
              __syncwarp();
              if (lane == 0) mbar_arrive(wempty_bar(slot));
            }
            tmem_st32(tcol + (uint32_t)(h * 32), o[h]);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(afull_bar(aslot));
          if (++s == SWH) { s = 0; ph ^= 1u; }
          if (++ai == kAHalf) { ai = 0; aph ^= 1u; }
        }
      }
    }
  } else if (warp >= kWarpMma0 && warp < kWarpMma0 + kIssuers) {
    // ------------------------------------------------------------- MMA --
    // Issuer q takes the chunks with CTA-wide index = q (mod kIssuers).  Each issuer
    // waits for every activation block and hands it back exactly once: by a commit
    // (completes when its MMAs on the block are done) if it used the block, else by
    // a plain arrive.
    if (kWarpIssue || lane == 0) {
      const uint32_t leader = kWarpIssue ? elect_leader() : 1u;
      const int q = warp - kWarpMma0;
      int xs = 0, cidx = 0;
      uint32_t xph = 0;
      bool ok = true;
      for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
        const int b = i % kNAcc;
        if (!vwait(accempty_bar(b), ((i / kNAcc) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(kAccCol0 + (b * kIssuers + q) * BN);
        bool first = true, xready = false, used = false;
        int j = 0;                                     // chunk within the activation block
        for (int g = sg.g0; g < sg.g1; ++g, ++cidx) {
          if (!xready) {
            if (!vwait(kAct8 ? bfull_bar(xs) : xfull_bar(xs), xph)) { ok = false; break; }
            xready = true;
          }
          if ((cidx & (kIssuers - 1)) == q) {
            const int h = cidx >> 1;                   // position in the parity's half
            const int aslot = (cidx & 1) * kAHalf + h % kAHalf;
            if (!vwait(afull_bar(aslot), (uint32_t)(h / kAHalf) & 1u)) { ok = false; break; }
            tc_fence_after();
            // descriptor start addresses advance by (offset >> 4); no carry out of the
            // 14-bit field since shared-memory addresses stay below 256 KB
            const uint64_t bdesc0 = smem_desc_sw128(x_smem(xs) + (uint32_t)j * kXChunk);
            const uint32_t a0 = tmem + (uint32_t)(aslot * 64);
  #pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_f16_ts_w(leader, d, a0 + (uint32_t)(k * 8),
                           bdesc0 + (uint64_t)(((k >> 2) * BN * 128 + (k & 3) * 32) >> 4), kIdesc,
                           (!first || k > 0) ? 1u : 0u);
            first = false;
            used = true;
            mma_commit_w(leader, aempty_bar(aslot));
          }
          if (++j == kXBlock || g + 1 == sg.g1) {
            if (used) mma_commit_w(leader, xempty_bar(xs));
            else mbar_arrive_w(leader, xempty_bar(xs));
            if (++xs == SX) { xs = 0; xph ^= 1u; }
            j = 0;
            xready = used = false;
          }
        }
        if (ok) mma_commit_w(leader, accfull_bar(b));
      }
      // every MMA the leader issued has completed before the CTA may exit
      mma_commit_w(leader, bars + kBarDrain);
      mbar_drain(bars + kBarDrain, 0, wctl);
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
    int pend_cut[2] = {0, 0};
    // contributors of this CTA's first and last segment (read now, while the
    // preceding kernel may still run, so the lookup is off the critical path)
    const int cut_first = P.cut[cta][0], cut_last = P.cut[cta][1];
    bool aborted = false;
    for (int i = 0; segment(P, cta, i, sg); ++i) {
      const int b = i % kNAcc;
      const int nch = sg.g1 - sg.g0;
      // accumulator q holds the segment's chunks with index = q (mod kIssuers), if any
      bool valid[kIssuers];
#pragma unroll
      for (int q = 0; q < kIssuers; ++q) valid[q] = nch >= kIssuers || ((q - cidx) & (kIssuers - 1)) < nch;
      cidx += nch;
      if constexpr (TOKSCALE) {
        // token scales of this tile into L1 while the accumulator is being produced
        int u_, t_;
        tile_coords(P, sg.tile, u_, t_);
        for (int m = u_ * BN + row; m < P.M && m < (u_ + 1) * BN; m += kRows) prefetch_l1(a.xs + m);
      }
      const bool got = pwait(accfull_bar(b), (i / kNAcc) & 1);
      // all four warps decide together, on the OR of their views
      if (named_bar_or(1, kEpiWarps * 32, !got || wctl->abort)) { aborted = true; break; }
      tc_fence_after();
      int u, t;
      tile_coords(P, sg.tile, u, t);
      const int n = t * kRows + row;
      const int m0 = u * BN;
      const int mv = P.M - m0 < BN ? P.M - m0 : BN;   // valid tokens of this tile
      const uint32_t tacc = tmem + lane_base + (uint32_t)(kAccCol0 + b * kIssuers * BN);
      float *part = sg.slot >= 0 ? a.partials + (size_t)sg.slot * (BN * kRows) : nullptr;
      constexpr int W = 32 / kIssuers;                // columns per TMEM load
#pragma unroll 1
      for (int cc = 0; cc < BN; cc += W) {
        uint32_t v[kIssuers][W];
#pragma unroll
        for (int q = 0; q < kIssuers; ++q) {
          if constexpr (W == 32) tmem_ld32(tacc + (uint32_t)(q * BN + cc), v[q]);
          else if constexpr (W == 16) tmem_ld16(tacc + (uint32_t)(q * BN + cc), v[q]);
          else tmem_ld8(tacc + (uint32_t)(q * BN + cc), v[q]);
        }
        // Wide tiles (one issuer, 32 columns per TMEM load; the epilogue holds up the
        // next tile's MMAs there) load the 32 columns' token scales before using any,
        // one per lane, and pass column j's along from lane j; narrow tiles read them
        // as they go (measured faster for those).
        constexpr bool kBatchScales = TOKSCALE && BN >= 128;
        static_assert(!kBatchScales || W == 32, "one token scale per lane");
        float tsc = 1.0f;
        if constexpr (kBatchScales)
          if (!part && cc + lane < mv) tsc = __ldg(a.xs + m0 + cc + lane);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < W; ++j) {
          float acc = 0.0f;                            // fixed order: issuer 0, 1, ...
#pragma unroll
          for (int q = 0; q < kIssuers; ++q)
            if (valid[q]) acc += __uint_as_float(v[q][j]);
          const float sj = kBatchScales ? __shfl_sync(0xffffffffu, tsc, j & 31) : 1.0f;
          if (cc + j < mv) {
            if (part) {
              part[(cc + j) * kRows + row] = acc;
            } else {
              const int m = m0 + cc + j;
              const float val = kBatchScales ? acc * sj : TOKSCALE ? acc * __ldg(a.xs + m) : acc;
              const __half hv = __float2half_rn(val);
              a.y[(size_t)m * P.N + n] = __half_as_ushort(hv);
              // the warp holds 32 rows of column m of tile t
              if constexpr (TMAX) tile_max_warp(a.tile_max + (size_t)m * P.T + t, order_key16(hv));
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
        // a cut segment is this CTA's first or its last
        const int cut = i == 0 ? cut_first : cut_last;
        const int pf = qw::cut_first(cut), pl = qw::cut_last(cut);
        if (ept == 0) {
          const int old = atom_add_acq_rel_gpu(a.counters + sg.tile, 1);
          const int last = (old == pl - pf) ? 1 : 0;
          if (last) a.counters[sg.tile] = 0;    // leave the workspace zeroed for the next call
          *bcast = last;
        }
        named_bar_sync(1, kEpiWarps * 32);
        if (*bcast) {                                // reduced once this CTA's own work is done
          pend_tile[npend] = sg.tile;
          pend_cut[npend++] = cut;
        }
      }
    }
    // ---- stream-K reductions: all MMAs of this CTA have completed (its last
    // accumulator was read), so every ring buffer is idle.  Sum the contributors'
    // partials of each cut tile this CTA finished last, in CTA order.  Up to 4
    // tokens each thread reads its row straight from L2; larger tiles pull all
    // partials into shared memory with bulk copies (all in flight at once).
    uint32_t red_phase = 0;
    const uint32_t avail = ring_bytes;
    for (int r = 0; r < npend && !aborted; ++r) {
      const int tile = pend_tile[r];
      const int pf = qw::cut_first(pend_cut[r]), pl = qw::cut_last(pend_cut[r]), pf_slot = qw::cut_slot(pend_cut[r]);
      int u, t;
      tile_coords(P, tile, u, t);
      const int n = t * kRows + row;
      const int m0 = u * BN;
      const int mv = P.M - m0 < BN ? P.M - m0 : BN;
      const int nseg = pl - pf + 1;
      auto put = [&](int m, float acc) {
        const float val = TOKSCALE ? acc * __ldg(a.xs + m) : acc;
        const __half hv = __float2half_rn(val);
        a.y[(size_t)m * P.N + n] = __half_as_ushort(hv);
        if constexpr (TMAX) tile_max_warp(a.tile_max + (size_t)m * P.T + t, order_key16(hv));   // whole warps call
      };
      if constexpr (TOKSCALE)  // warm L1 with this tile's token scales
        for (int m = m0 + row; m < m0 + mv; m += kRows) prefetch_l1(a.xs + m);
      if (mv <= 4) {
        // the atomic's acquire (thread 0) and the named barrier order these reads
        // after every contributor's release; .cg reads bypass L1.  Eight
        // contributors' loads are in flight at once, then summed in CTA order.
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int p0 = pf; p0 <= pl; p0 += 8) {
          float v[8][4];
#pragma unroll
          for (int pp = 0; pp < 8; ++pp) {
            const int p = p0 + pp;
            const float *src = a.partials + (size_t)(p == pf ? pf_slot : 2 * p) * (BN * kRows) + row;
#pragma unroll
            for (int j = 0; j < 4; ++j) v[pp][j] = (p <= pl && j < mv) ? __ldcg(src + j * kRows) : 0.0f;
          }
#pragma unroll
          for (int pp = 0; pp < 8; ++pp)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (p0 + pp <= pl) acc[j] += v[pp][j];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < mv) put(m0 + j, acc[j]);
        continue;
      }
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
                            a.partials + (size_t)(p == pf ? pf_slot : 2 * p) * (BN * kRows) + (size_t)j0 * kRows,
                            bytes, bars + kBarRed);
        }
        const bool got = pwait(bars + kBarRed, red_phase);
        if (named_bar_or(1, kEpiWarps * 32, !got)) {
          if (ept == 0) mbar_drain(bars + kBarRed, red_phase, wctl);   // its copies still land
          aborted = true;
          break;
        }
        red_phase ^= 1u;
        // eight tokens at a time so that the shared-memory loads overlap; each
        // token's sum still runs over the contributors in CTA order
        const float *buf = reinterpret_cast<const float *>(gbase) + row;
        const int pstride = jn * kRows;
        int j = 0;
        for (; j + 8 <= jn; j += 8) {
          float acc[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) acc[jj] = 0.0f;
          for (int p = 0; p < nseg; ++p) {
            const float *bp = buf + p * pstride + j * kRows;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) acc[jj] += bp[jj * kRows];
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) put(m0 + j0 + j + jj, acc[jj]);
        }
        for (; j < jn; ++j) {
          float acc = 0.0f;
          for (int p = 0; p < nseg; ++p) acc += buf[p * pstride + j * kRows];
          put(m0 + j0 + j, acc);
        }
        named_bar_sync(1, kEpiWarps * 32);          // buffer free before the next pass
      }
    }
  }

  // --------------------------------------------------------------- teardown --
  // Every producer has drained what it started (weight and activation copies, the
  // issuers' MMAs, the reduction copies), so nothing is still writing shared memory
  // or TMEM, aborted or not.
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace qw
