// gemm_rb.cuh -- the quantized linear layer for decode-sized batches (M <= 16 tokens) on
// layers of few rows: each CTA owns 1..kRbMax whole 16-row blocks of the weight matrix
// over the whole K, so no tile is split between CTAs.
//
// y[m,n] = sum_g s[n,g] * sum_{k in g} a[m,k] * q[n,k]   ("In full" item 4 of "What this
// repo does that stock vLLM doesn't": int4 weights with signed group-128 scales, fp16 or
// per-token int8 activations).
//
// Why a second decode kernel: a 5120-row projection has 40 tiles of 128 rows for 152 SMs,
// so the tile-based kernel (gemm_ms.cuh) cuts every tile's K range between 3 or 4 CTAs,
// and each cut costs a binary32 partial in global memory, an acq_rel ticket on the tile
// counter and a reduction by the last CTA to arrive -- round trips to L2 under the full
// weight stream, at the end of every CTA.  Here the 320 row blocks go 2 or 3 to a CTA, the
// CTA's eight compute warps split the 40 K groups (group g to warp g mod 8), and the eight
// sums meet in shared memory.
//
// Roles (persistent CTAs, one per SM; a ring of stages of 8 consecutive K groups each):
//   warp 0, lane 0 : per stage and row block of the CTA two TMA tensor copies over the 8
//                    groups: the row block's codes (1 KB a group, in the packer's fragment
//                    order) and its scales (32 B a group), through tensor maps that see the
//                    packed matrix as [row tiles][groups][1056 x 8 B] -- a few large copies
//                    instead of one small one per group and row block.
//   warp 1, lane 0 : per stage one TMA tensor copy of the 8 groups' activations (8 or 16
//                    token rows, 128-byte swizzle, zero fill past M and K).
//   compute warps  : sixteen; warp w takes K steps 4 (w / 8) .. 4 (w / 8) + 3 of group
//                    w mod 8 of every stage (two warps a group: four warps on every SM
//                    sub-partition keep its MMA pipe busier than two with twice the chain);
//                    the weights become MMA fragments (mma.sync m16n8k16, weights as the A
//                    operand in registers) and accumulate into a per-group fp32 sum per row
//                    block, scaled by the signed group scale into the running sum.  int8
//                    activations are first widened to fp16 in the tile, and fp16 ones to
//                    be quantized in the kernel turned into codes, each warp its own half.
//                    At the end the sixteen sums of every output are added in warp order in
//                    shared memory (deterministic) and written as fp16 y.
#pragma once
#include <stdint.h>
#include <cuda_fp16.h>
#include "gemm_ms.cuh"   // mma_16816, ldsm_x4, lds128, lds32, frag_w4, frag_w4_zp, ms_threads
#include "quant_code.cuh"

namespace qw {

// ldmatrix offsets of lane `lane` for the four pairs of K steps of a 128-wide group in an
// activation tile of bnx token rows: lane l addresses row l % 8 (token 8 jt + l % 8) of
// matrix l / 8 of the pair: K step 2 sp + (l / 8) / 2, eight K values (l / 8) % 2, in the
// 128-byte-swizzled tile (16-byte piece p of row r at (p ^ r % 8) * 16, two 64-wide halves
// of bnx rows).
constexpr int kRbCompute = 16;                        // compute warps
__host__ __device__ constexpr int rb_threads() { return (kMsWarpC0 + kRbCompute) * 32; }

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void rb_x_offsets(int lane, int bnx, uint32_t (&xoff)[4]) {
  const int mi = lane >> 3, lrow = lane & 7;
#pragma unroll
  for (int sp = 0; sp < 4; ++sp) {
    const int ks = 2 * sp + (mi >> 1), jch = 2 * (ks & 3) + (mi & 1);
    xoff[sp] = (uint32_t)((ks >> 2) * (bnx * 128) + lrow * 128 + ((jch ^ lrow) << 4));
  }
}

template <int NT8, int AMODE, bool TMAX>
__global__ void __launch_bounds__(rb_threads(), 1) qgemm_rb_kernel(const __grid_constant__ GemmArgs a) {
  constexpr bool ACT8 = AMODE == kActI8;
  constexpr bool QIN = AMODE == kActQuant;                 // fp16 x quantized per token here
  constexpr bool TOKS = ACT8 || QIN || AMODE == kActCodes16;   // token scales in the epilogue
  static_assert(!TMAX || AMODE == kActF16, "the lm_head's fused top-k is W4A16");
  static_assert(!QIN || NT8 == 1, "the in-kernel quantizer serves up to 8 tokens");
  static_assert(NT8 == 1 || NT8 == 2, "one or two tiles of 8 tokens");
  constexpr int kCompute = kRbCompute;
  constexpr int kCThreads = kCompute * 32;
  constexpr int BNX = 8 * NT8;                          // token rows of an activation tile
  constexpr int kXB = kRbXBlock;                        // K groups per stage
  static_assert(2 * kXB == kCompute, "two compute warps per group of a stage");
  constexpr uint32_t kXChunk = BNX * kGroup * 2;        // one fp16 tile: two 64-wide halves
  constexpr uint32_t kXTiles = kXB * (kXChunk + (ACT8 ? BNX * kGroup : 0));   // stage: activations
  constexpr uint32_t kXBytes = kXB * (ACT8 ? BNX * kGroup : kXChunk);          // per copy
  constexpr uint32_t kStage = (kXTiles + kRbWBytes + kRbSBytes + 1023) / 1024 * 1024;
  constexpr uint32_t kWOff = kXTiles;                   // codes: [row block][group][1 KB]
  constexpr uint32_t kSOff = kXTiles + kRbWBytes;       // scales: [row block][group][32 B]
  static_assert(kXTiles % 1024 == 0, "weight boxes 1 KB aligned");
  // Zero-point form for one tile of eight tokens (see gemm_ms.cuh): the MMAs take the raw
  // magic values and one more MMA per K step adds the zero point; for two tiles the
  // fragments hold the plain codes.
  constexpr bool kZP = NT8 == 1;
  constexpr int RBM = kRbMax;

  extern __shared__ uint8_t smem_raw[];
  const Plan &P = a.P;
  const int SS = P.stages;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + (uint32_t)SS * kStage;
  uint8_t *gbars = gbase + (bars - sbase);
  auto wfull_bar = [&](int s) { return bars + 8u * s; };     // the stage's weights landed
  auto xfull_bar = [&](int s) { return bars + 64u + 8u * s; };   // its activations landed
  auto empty_bar = [&](int s) { return bars + 128u + 8u * s; };  // the compute warps are done
  // the compute warps' common view of the abort flag, taken by one thread before a
  // named barrier, so that all of them pass the same barriers
  volatile int *decide = reinterpret_cast<volatile int *>(gbars + 192);
  volatile WaitBlock *wctl = reinterpret_cast<volatile WaitBlock *>(gbars + 200);
  // in-kernel quantizer: per-warp row maxima [16 warps][16 tokens], token scales s and 1/s
  float *qamax = reinterpret_cast<float *>(gbars + 256);
  float *qsc = qamax + kRbCompute * 16, *qrc = qsc + 16;
  static_assert(256 + (kRbCompute * 16 + 32) * 4 <= kRbReserve - 1024, "quantizer data in the reserve");
  // the compute warps' sums at the end: [warp][row block][token][16 rows, padded to kRS]
  // binary32 (the padding spreads a warp's stores over the banks), over the ring (every
  // copy into it has been waited for by then)
  constexpr int kRS = 17;
  float *red = reinterpret_cast<float *>(gbase);
  auto pwait = [&](uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity, wctl, a.wait_ns == 0); };
  auto stage = [&](int s) { return sbase + (uint32_t)s * kStage; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int rb0 = P.begin[cta], nrb = P.begin[cta + 1] - rb0;   // 1 .. kRbMax row blocks
  const int G = P.G;
  const int nst = (G + kXB - 1) / kXB;                          // stages of the CTA

  if (threadIdx.x == 32) {
    for (int s = 0; s < SS; ++s) {
      mbar_init(wfull_bar(s), 1);
      mbar_init(xfull_bar(s), 1);
      mbar_init(empty_bar(s), kCompute);
    }
    wait_block_init(wctl, a.wait_ns, a.err);
    *decide = 0;
    fence_mbar_init();
  }
  if (lane == 0 && warp == kMsWarpX) prefetch_tensormap(&a.tmap);
  if (lane == 0 && warp == kMsWarpW) {
    prefetch_tensormap(&a.wmap);
    prefetch_tensormap(&a.smap);
  }
  __syncthreads();

  // The weight copies may run ahead of the preceding kernel when the caller declared
  // the packed weights immutable; everything else waits for it first.
  const bool early = a.early_weights != 0;
  if (!(early && warp == kMsWarpW)) griddep_wait();
  griddep_launch_dependents();

  if (warp == kMsWarpW) {
    // ------------------------------------------------------ weight copies --
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      if (early) {
        // ahead of the preceding kernel: the stages that will not fit the ring now are
        // pulled into L2 (at most two ring's worth)
        for (int i = SS; i < nst && i < 3 * SS; ++i)
          for (int r = 0; r < nrb; ++r) {
            const int rb = rb0 + r;
            tma_prefetch_3d(&a.wmap, (rb & 7) * 128, i * kXB, rb >> 3);
          }
      }
      int s = 0, nfill = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nst; ++i) {
        if (!pwait(empty_bar(s), ph ^ 1u)) break;
        mbar_arrive_expect_tx(wfull_bar(s), (uint32_t)nrb * (kXB * (1024u + 32u)));
        for (int r = 0; r < nrb; ++r) {
          const int rb = rb0 + r;
          tma_load_3d_hint(stage(s) + kWOff + (uint32_t)r * (kXB * 1024), &a.wmap, (rb & 7) * 128, i * kXB,
                           rb >> 3, wfull_bar(s), pol);
          tma_load_3d_hint(stage(s) + kSOff + (uint32_t)r * (kXB * 32), &a.smap, 1024 + (rb & 7) * 4, i * kXB,
                           rb >> 3, wfull_bar(s), pol);
        }
        ++nfill;
        if (++s == SS) { s = 0; ph ^= 1u; }
      }
      // the last fill of every slot has landed before the CTA may exit
      for (int k = 0; k < SS && k < nfill; ++k) mbar_drain(wfull_bar(k), k < s ? ph : ph ^ 1u, wctl);
    }
  } else if (warp == kMsWarpX) {
    // -------------------------------------------------- activation copies --
    if (lane == 0) {
      int s = 0, nfill = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nst; ++i) {
        if (!pwait(empty_bar(s), ph ^ 1u)) break;
        mbar_arrive_expect_tx(xfull_bar(s), kXBytes);
        ++nfill;
        if constexpr (ACT8) tma_load_3d(stage(s) + kXB * kXChunk, &a.tmap, 0, 0, i * kXB, xfull_bar(s));
        else tma_load_3d(stage(s), &a.tmap, 0, 0, 2 * i * kXB, xfull_bar(s));
        if (++s == SS) { s = 0; ph ^= 1u; }
      }
      for (int k = 0; k < SS && k < nfill; ++k) mbar_drain(xfull_bar(k), k < s ? ph : ph ^ 1u, wctl);
    }
  } else if (warp >= kMsWarpC0) {
    // ------------------------------------------------------------ compute --
    const int cw = warp - kMsWarpC0;
    const int gj = cw & (kXB - 1), hh = cw / kXB;    // group of the stage, half of its K steps
    const int g8 = lane >> 2, c4 = lane & 3;
    const int ct = threadIdx.x - kMsWarpC0 * 32;     // 0 .. kCThreads - 1
    const int mv = P.M < BNX ? P.M : BNX;
    if constexpr (QIN) {
      // token scales, as the standalone quantizer: amax = max |x| over the whole row
      // (binary32, exact in any order), s = amax / 127 (IEEE divide); the rows come from
      // L2 while the first weights are in flight.  One token: the whole CTA on its row;
      // several: warps cw = m, m + mv, ... take token m, so that every row is requested
      // at once (four 16-byte loads a lane in flight: two rows of K <= 8192 in one trip)
      const int nv = G * 16;                        // 16-byte vectors of a row
      auto row_amax = [&](const uint4 *xr, int t0, int step) {
        float am = 0.0f;
        for (int v0 = t0; v0 < nv; v0 += 4 * step) {
          uint4 w[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int v = v0 + b * step;
            w[b] = v < nv ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const __half2 *hv = reinterpret_cast<const __half2 *>(&w[b]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __half22float2(hv[e]);
              am = fmaxf(am, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        return am;
      };
      float amax;
      if (mv == 1) {
        amax = row_amax(reinterpret_cast<const uint4 *>(a.xf16), ct, kCThreads);
      } else {
        const int m = cw % mv, nw = (kCompute - 1 - m) / mv + 1;   // token, its warps
        amax = row_amax(reinterpret_cast<const uint4 *>(a.xf16 + (size_t)m * P.K), (cw / mv) * 32 + lane,
                        nw * 32);
      }
      if (lane == 0) qamax[cw] = amax;
      named_bar_sync(2, kCThreads);
      if (ct < mv) {
        float am = 0.0f;
#pragma unroll
        for (int r = 0; r < kCompute; ++r) {        // the warps of token ct, loads independent
          const int w = ct + r * mv;
          if (w < kCompute) am = fmaxf(am, qamax[w]);
        }
        const float sc = am == 0.0f ? 0.0f : __fdiv_rn(am, 127.0f);
        qsc[ct] = sc;
        qrc[ct] = sc == 0.0f ? 0.0f : __frcp_rn(sc);
      }
      named_bar_sync(2, kCThreads);
    }
    uint32_t xoff[4];
    rb_x_offsets(lane, BNX, xoff);
    // the two pairs of K steps of this warp's half
    const uint32_t xoh[2] = {hh ? xoff[2] : xoff[0], hh ? xoff[3] : xoff[1]};
    // weights: within a row block's 1 KB of a group, the vector at ((h * 4 + c) * 8 + (i ^ 2 c))
    // for K steps 4 h .. 4 h + 3; its scale pair i at 4 i of the group's 32 B
    const uint32_t woff = (uint32_t)((c4 * 8 + (g8 ^ (2 * c4))) * 16);
    const __half2 k16th = __float2half2_rn(0.0625f);
    const uint32_t zp[4] = {h2_as_u32(__float2half2_rn(-1032.0f)), h2_as_u32(__float2half2_rn(-1032.0f)),
                            h2_as_u32(__float2half2_rn(-1152.0f)), h2_as_u32(__float2half2_rn(-1152.0f))};
    float acc[RBM][NT8][4];
#pragma unroll
    for (int r = 0; r < RBM; ++r)
#pragma unroll
      for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][jt][e] = 0.0f;
    int s = 0;
    uint32_t ph = 0;
    // a warp that saw a wait give up releases no stage again: a copy it gave up on may
    // still be landing, and a producer released now would arm that stage's phase twice
    bool live = true;
    for (int i = 0; i < nst; ++i) {
      // every compute warp waits for every stage and returns it once; after an abort every
      // wait gives up at once and the loop runs out quickly
      live = pwait(xfull_bar(s), ph) && live;
      live = pwait(wfull_bar(s), ph) && live;
      if (i * kXB + gj < G) {
        const uint32_t xt = stage(s) + (uint32_t)gj * kXChunk;
        if constexpr (QIN) {
          // this warp's 64-wide half of the group's tile becomes codes, in place (the other
          // half is the other warp's): rows below M, one pair of K values per lane and step
          // (pair j of row r: 8-value piece j / 4 of the half, swizzled by r % 8)
          const uint32_t half = xt + (uint32_t)hh * (BNX * 128);
          for (int pr = lane; pr < mv * 32; pr += 32) {
            const int r = pr >> 5, j = pr & 31;
            const uint32_t addr = half + (uint32_t)(r * 128 + (((j >> 2) ^ (r & 7)) << 4) + (j & 3) * 4);
            const float sc = qsc[r], rs = qrc[r];
            const float2 f = __half22float2(u32_as_h2(lds32(addr)));
            const int q0 = quant_code(f.x, sc, rs), q1 = quant_code(f.y, sc, rs);
            sts32(addr, h2_as_u32(__halves2half2(__int2half_rn(q0), __int2half_rn(q1))));
          }
          __syncwarp();
        }
        if constexpr (ACT8) {
          // this warp's half of the group's int8 codes (unswizzled staging rows) widened to
          // fp16 in its half of the tile: rows below M, 16 codes per lane and step
          const uint8_t *stg = gbase + (size_t)s * kStage + kXB * kXChunk + gj * (BNX * kGroup) + hh * 64;
          uint8_t *row0 = gbase + (size_t)s * kStage + gj * kXChunk + hh * (BNX * 128);
          const __half2 k1152 = __float2half2_rn(1152.0f);
          for (int pc = lane; pc < mv * 4; pc += 32) {
            const int r = pc >> 2, c = pc & 3;                // 16 codes: pieces 2c, 2c + 1
            const uint4 v = *reinterpret_cast<const uint4 *>(stg + r * kGroup + c * 16);
            const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u,
                                   v.w ^ 0x80808080u};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o[2 * i] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w[i], 0x64646464u, 0x4140)), k1152));
              o[2 * i + 1] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(w[i], 0x64646464u, 0x4342)), k1152));
            }
            uint8_t *row = row0 + r * 128;
            *reinterpret_cast<uint4 *>(row + (((2 * c) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(row + (((2 * c + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
          __syncwarp();
        }
        const uint32_t wc = stage(s) + kWOff + (uint32_t)gj * 1024u;
        const uint32_t sc = stage(s) + kSOff + (uint32_t)gj * 32u + (uint32_t)g8 * 4u;
        uint32_t sc2[RBM];
#pragma unroll
        for (int r = 0; r < RBM; ++r) sc2[r] = r < nrb ? lds32(sc + (uint32_t)r * (kXB * 32)) : 0u;
        float ga[RBM][NT8][4], gz[NT8][4];
#pragma unroll
        for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            gz[jt][e] = 0.0f;
#pragma unroll
            for (int r = 0; r < RBM; ++r) ga[r][jt][e] = 0.0f;
          }
        {
          const int h = hh;                              // K steps 4 h .. 4 h + 3
          uint4 v[RBM];
#pragma unroll
          for (int r = 0; r < RBM; ++r)
            v[r] = r < nrb ? lds128(wc + woff + (uint32_t)(r * (kXB * 1024) + h * 512)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int sp2 = 0; sp2 < 2; ++sp2) {
            uint32_t bf[2][NT8][2];
#pragma unroll
            for (int jt = 0; jt < NT8; ++jt) {
              ldsm_x4(xt + xoh[sp2] + (uint32_t)(jt * 1024), bf[0][jt][0], bf[0][jt][1], bf[1][jt][0],
                      bf[1][jt][1]);
              if constexpr (kZP) {
                bf[0][jt][1] = h2_as_u32(__hmul2(u32_as_h2(bf[0][jt][1]), k16th));
                bf[1][jt][1] = h2_as_u32(__hmul2(u32_as_h2(bf[1][jt][1]), k16th));
              }
            }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const int wd = (2 * sp2 + kk);           // word of the vector = K step % 4
              if constexpr (kZP) {
#pragma unroll
                for (int jt = 0; jt < NT8; ++jt) mma_16816(gz[jt], zp, bf[kk][jt][0], bf[kk][jt][1]);
              }
#pragma unroll
              for (int r = 0; r < RBM; ++r) {
                if (r < nrb) {
                  const uint32_t w = wd == 0 ? v[r].x : wd == 1 ? v[r].y : wd == 2 ? v[r].z : v[r].w;
                  uint32_t af[4];
                  if constexpr (kZP) frag_w4_zp(w, af);
                  else frag_w4(w, af);
#pragma unroll
                  for (int jt = 0; jt < NT8; ++jt) mma_16816(ga[r][jt], af, bf[kk][jt][0], bf[kk][jt][1]);
                }
              }
            }
          }
        }
#pragma unroll
        for (int r = 0; r < RBM; ++r) {
          const float2 sf = __half22float2(u32_as_h2(sc2[r]));   // (row R, row R + 8)
#pragma unroll
          for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float gs = kZP ? ga[r][jt][e] + gz[jt][e] : ga[r][jt][e];
              acc[r][jt][e] = fmaf(e < 2 ? sf.x : sf.y, gs, acc[r][jt][e]);
            }
        }
      }
      __syncwarp();
      if (lane == 0 && live) mbar_arrive(empty_bar(s));
      if (++s == SS) { s = 0; ph ^= 1u; }
    }
    // ---- the warps' sums meet in shared memory (over the ring: every copy into it has
    // been waited for by every compute warp), added in warp order.  The abort flag is read
    // once every compute warp has left its loop (no wait of theirs can fail after that):
    // after an abort a copy may still be landing in the ring, so nothing is written.
    named_bar_sync(1, kCThreads);
    if (ct == 0) *decide = wctl->abort;
    named_bar_sync(1, kCThreads);
    if (!*decide) {
#pragma unroll
      for (int r = 0; r < RBM; ++r)
#pragma unroll
        for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = 8 * jt + 2 * c4 + (e & 1), row = g8 + 8 * (e >> 1);
            red[((cw * RBM + r) * BNX + m) * kRS + row] = acc[r][jt][e];
          }
    }
    named_bar_sync(1, kCThreads);
    if (!*decide) {
      for (int idx = ct; idx < nrb * mv * 16; idx += kCThreads) {
        const int r = idx / (mv * 16), m = (idx >> 4) % mv, row = idx & 15;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kCompute; ++w) v += red[((w * RBM + r) * BNX + m) * kRS + row];
        const __half hv = __float2half_rn(QIN ? v * qsc[m] : TOKS ? v * __ldg(a.xs + m) : v);
        const int n = (rb0 + r) * 16 + row;
        a.y[(size_t)m * P.N + n] = __half_as_ushort(hv);
        if constexpr (TMAX) atomicMax(a.tile_max + (size_t)m * P.T + (n >> 7), order_key16(hv));
      }
    }
  }

  // --------------------------------------------------------------- teardown --
  // both copy threads have drained their copies: nothing still writes shared memory
  __syncthreads();
}

}  // namespace qw
