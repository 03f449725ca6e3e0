// gemm_ms.cuh -- the quantized linear layer for decode-sized batches (M <= 16 tokens)
// on the warp-level tensor-core MMA (mma.sync m16n8k16), the int4 weights dequantized
// in registers and fed straight into it.
//
// y[m,n] = sum_g s[n,g] * sum_{k in g} a[m,k] * q[n,k]   ("In full" item 4 of "What this
// repo does that stock vLLM doesn't": int4 weights with signed group-128 scales, fp16 or
// per-token int8 activations).
//
// At these batch sizes the layer is bound by streaming the packed weights from HBM: a
// 128 x 128 chunk (8,448 bytes) must be consumed every ~0.19 us per SM.  A 5th-generation
// MMA pipeline needs every chunk dequantized into TMEM before its eight tcgen05.mma
// (K = 16 each, ~34 ns apiece from a lone issuing lane, ~9 ns from a converged warp) and
// frees it ~0.1 us after their commit: a dequant -> TMEM -> MMA -> commit chain per chunk.
// Here the weights are the MMA's A operand (16 weight rows x 16 K per instruction, in
// registers), the tokens its B operand (8 per instruction: one n8 tile for M <= 8, two
// for M <= 16): 64 or 128 MMAs of 2k MACs per chunk, issued like any other instruction,
// with no asynchronous chain.
//
// Roles (persistent CTAs, the stream-K schedule of schedule.h; a CTA takes at most half
// an SM, so the next layer's CTAs start while this layer's finish):
//   warp 0, lane 0 : one bulk copy per packed chunk into the weight ring; the ring is
//                    split into one part per team and a team's chunks fill its part
//                    in order.  When the weights may be read ahead of the preceding
//                    kernel, the next chunks beyond the ring (kMsL2AheadChunks) are first
//                    prefetched into L2.
//   warp 1, lane 0 : one TMA tensor copy per block of four K groups of the
//                    activations (8 or 16 token rows, 128-byte swizzle, zero fill past M)
//   compute warps  : eight, in teams; team j takes the chunks with CTA-wide index = j
//                    (mod teams), visiting the activation blocks and, in each, only its
//                    own chunks.  A warp covers RBW 16-row blocks of a chunk: two (two
//                    teams of four warps), or four for long launches of up to 8 tokens
//                    (four teams of two: more independent MMA chains per warp).
//                    K step by K step the weights become MMA fragments and accumulate
//                    into a per-group fp32 sum, which is then scaled by the signed group
//                    scale (binary32) into the running sum.  At the end of a tile
//                    segment the other teams leave their sums in shared memory; the
//                    first team adds them in team order and writes fp16 y -- or a
//                    binary32 partial when the stream-K split cuts the tile, summed in
//                    CTA order by the last CTA to finish it (deterministic, no waiting).
//   int8 activations: when a block arrives, the compute warps together widen its int8
//                    codes to fp16 (exact) in the swizzled tile the MMA fragments are
//                    loaded from; fp16 activations quantized in the kernel: they first
//                    find the token scales (amax over whole rows, read from L2), then
//                    write each block's codes, rne(x / s) as the standalone quantizer
//                    computes them, over its fp16 tile (exact in fp16).
#pragma once
#include <stdint.h>
#include <cuda_fp16.h>
#include "ptx.cuh"
#include "schedule.h"
#include "launch.h"
#include "gemm_kernel.cuh"   // widen_chunk

namespace qw {

constexpr int kMsWarpW = 0;       // weight copies
constexpr int kMsWarpX = 1;       // activation copies
constexpr int kMsWarpC0 = 2;      // first compute warp

// activation modes: fp16 x (W4A16), int8 codes + token scales (W4A8), fp16 codes + token
// scales (W4A8 from fp16 after the standalone quantizer: the W4A16 data path, the W4A8
// epilogue), fp16 x quantized per token inside the kernel (W4A8 from fp16; row-block
// kernel only)
enum { kActF16 = 0, kActI8 = 1, kActCodes16 = 2, kActQuant = 3 };

__host__ __device__ constexpr int ms_threads() { return (kMsWarpC0 + kMsComputeWarps) * 32; }

// D (16 x 8, fp32) += A (16 x 16, fp16 rows) * B (16 x 8, fp16 columns)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8 x 8 fp16 matrices from shared memory; lane l gives the address of row l % 8 of
// matrix l / 8, and receives from each matrix its row l / 4, elements 2 (l % 4) and + 1.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// One packed word (see the packer) -> the A fragment of one 16 x 16 K step, rows R
// (nibbles 0/4 and 1/5) and R + 8 (nibbles 2/6 and 3/7).
//   frag_w4    : the codes q, exact in fp16: (1024 + u) - 1032 and (1024 + 16 u)/16 - 72.
//   frag_w4_zp : the raw values 1024 + u (positions k0, k0 + 1) and 1024 + 16 u (k0 + 8,
//                k0 + 9); the caller divides the activations at k0 + 8, k0 + 9 by 16 and
//                adds the per-token correction that one more MMA computes (see below).
__device__ __forceinline__ void frag_w4(uint32_t w, uint32_t (&a)[4]) {
  const __half2 k1032 = __float2half2_rn(1032.0f);
  const __half2 k16th = __float2half2_rn(0.0625f);
  const __half2 km72 = __float2half2_rn(-72.0f);
  const uint32_t x = w >> 8;
  a[0] = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w, 0x000f000fu, 0x64006400u)), k1032));         // R, k0..
  a[1] = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(x, 0x000f000fu, 0x64006400u)), k1032));         // R+8, k0..
  a[2] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w, 0x00f000f0u, 0x64006400u)), k16th, km72));   // R, k0+8..
  a[3] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(x, 0x00f000f0u, 0x64006400u)), k16th, km72));   // R+8, k0+8..
}
__device__ __forceinline__ void frag_w4_zp(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t x = w >> 8;
  a[0] = lop3_and_or(w, 0x000f000fu, 0x64006400u);
  a[1] = lop3_and_or(x, 0x000f000fu, 0x64006400u);
  a[2] = lop3_and_or(w, 0x00f000f0u, 0x64006400u);
  a[3] = lop3_and_or(x, 0x00f000f0u, 0x64006400u);
}

// TMAX: the epilogue also raises the per-tile maxima of the lm_head's fused top-k
template <int NT8, int AMODE, int RBW, bool TMAX>
__global__ void __launch_bounds__(ms_threads(), 2) qgemm_ms_kernel(const __grid_constant__ GemmArgs a) {
  constexpr bool ACT8 = AMODE == kActI8;
  constexpr bool TOKS = ACT8 || AMODE == kActCodes16;   // token scales in the epilogue
  constexpr bool kTileMax = TMAX;
  static_assert(!TMAX || AMODE == kActF16, "the lm_head's fused top-k is W4A16");
  static_assert(RBW == 2 || RBW == 4, "16-row blocks per warp in a chunk");
  constexpr int KS = 1;                                 // accumulator sets per row block
  constexpr int TW = 8 / RBW;                           // warps per team (a chunk has 8 row blocks)
  constexpr int TEAMS = kMsComputeWarps / TW;
  constexpr int kCompute = kMsComputeWarps;
  constexpr int kCThreads = kCompute * 32;
  constexpr int BNX = 8 * NT8;                          // token rows of an activation tile
  constexpr int kXBlock = act_block(kMsMaxTokens);      // K groups per activation copy (4)
  constexpr uint32_t kXChunk = BNX * kGroup * 2;        // one fp16 tile: two 64-wide halves
  constexpr uint32_t kXStage = kXBlock * (kXChunk + (ACT8 ? BNX * kGroup : 0));
  constexpr uint32_t kXBytes = kXBlock * (ACT8 ? BNX * kGroup : kXChunk);   // per copy
  constexpr uint32_t kWStage = kChunkW4;
  constexpr int PB = kMsMaxTokens * kRows;              // floats per partial slot
  // Zero-point form for one tile of eight tokens: the MMA multiplies the raw magic
  // values, and per K step one more MMA with a constant A operand (-1032 at the
  // positions k0, k0 + 1, -1152 at k0 + 8, k0 + 9, whose activations are divided by 16)
  // adds sum_k x_k * (-8 - the magic offset) to every row: exactly the zero point.  For
  // sixteen tokens that MMA would cost more tensor time than the subtraction it saves.
  constexpr bool kZP = NT8 == 1;
  static_assert(kWStage % 128 == 0, "weight slots stay 128-byte aligned");
  static_assert(NT8 == 1 || NT8 == 2, "one or two tiles of 8 tokens");
  static_assert(kXBlock == 4 && kXBlock % TEAMS == 0, "blocks of four chunks, at most one per team");
  constexpr int S = kMsRedStride;

  extern __shared__ uint8_t smem_raw[];
  const Plan &P = a.P;
  const int SW = P.stages, SX = P.xstages, SWT = SW / TEAMS;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (sbase - raw);
  const uint32_t wbase = sbase + (uint32_t)SX * kXStage;
  const uint32_t rbase = wbase + (uint32_t)SW * kWStage;
  float *red = reinterpret_cast<float *>(gbase + (rbase - sbase));
  const uint32_t bars = rbase + (uint32_t)P.ms_red_bytes;
  uint8_t *gbars = gbase + (bars - sbase);
  auto wfull_bar = [&](int s) { return bars + 8u * s; };
  auto wempty_bar = [&](int s) { return bars + 128u + 8u * s; };
  auto xfull_bar = [&](int s) { return bars + 256u + 8u * s; };
  auto xempty_bar = [&](int s) { return bars + 288u + 8u * s; };
  volatile int *bcast = reinterpret_cast<volatile int *>(gbars + 356);
  // the compute warps' common view of the abort flag, taken by one thread before a
  // named barrier, so that all of them pass the same barriers
  volatile int *decide = reinterpret_cast<volatile int *>(gbars + 360);
  volatile WaitBlock *wctl = reinterpret_cast<volatile WaitBlock *>(gbars + 368);
  // a pipeline wait: bounded by the launch's limit, gives up once the CTA aborts
  auto pwait = [&](uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity, wctl, a.wait_ns == 0); };
  auto w_smem = [&](int s) { return wbase + (uint32_t)s * kWStage; };
  auto x_smem = [&](int s) { return sbase + (uint32_t)s * kXStage; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  if (threadIdx.x == 32) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(wfull_bar(s), 1);
      mbar_init(wempty_bar(s), TW);
    }
    for (int s = 0; s < SX; ++s) {
      mbar_init(xfull_bar(s), 1);
      mbar_init(xempty_bar(s), kCompute);
    }
    wait_block_init(wctl, a.wait_ns, a.err);
    *bcast = 0;
    *decide = 0;
    fence_mbar_init();
  }
  if (warp == kMsWarpX && lane == 0) prefetch_tensormap(&a.tmap);
  __syncthreads();

  // The weight copies may run ahead of the preceding kernel when the caller declared
  // the packed weights immutable; everything else waits for it first.
  const bool early = a.early_weights != 0;
  if (!(early && warp == kMsWarpW)) griddep_wait();
  griddep_launch_dependents();

  Seg sg;
  if (warp == kMsWarpW) {
    // ------------------------------------------------------ weight copies --
    // (the whole warp runs the producer loops, waits are warp votes and the leader lane
    // issues: a copy issued by a lone lane in a divergent branch costs several times more)
    const uint32_t leader = elect_leader();
    const uint64_t pol = policy_evict_first();
    if (early) {
      // ahead of the preceding kernel: the next kMsL2AheadChunks chunks that will not
      // fit the ring now are pulled into L2, so that their copies after the wait come
      // from L2, not HBM (a bounded number: a long launch pulling all of its chunks
      // would push its own earlier ones out of L2 before they are copied)
      int c = 0;
      for (int i = 0; c < SW + kMsL2AheadChunks && segment(P, cta, i, sg); ++i) {
        int u, t;
        tile_coords(P, sg.tile, u, t);
        const uint8_t *src = a.wpack + ((size_t)t * P.G + sg.g0) * kChunkW4;
        for (int g = sg.g0; g < sg.g1 && c < SW + kMsL2AheadChunks; ++g, ++c, src += kChunkW4)
          if (c >= SW) prefetch_l2_w(leader, src, kChunkW4);
      }
    }
    int s[TEAMS], nfill[TEAMS], cidx = 0;
    uint32_t ph[TEAMS];
#pragma unroll
    for (int j = 0; j < TEAMS; ++j) s[j] = 0, nfill[j] = 0, ph[j] = 0;
    bool ok = true;
    for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
      int u, t;
      tile_coords(P, sg.tile, u, t);
      const uint8_t *src = a.wpack + ((size_t)t * P.G + sg.g0) * kChunkW4;
      for (int g = sg.g0; g < sg.g1; ++g, ++cidx, src += kChunkW4) {
        const int tm = cidx & (TEAMS - 1);
        int slot = 0;
        uint32_t par = 0;
#pragma unroll
        for (int j = 0; j < TEAMS; ++j)
          if (j == tm) { slot = j * SWT + s[j]; par = ph[j]; }
        if (!__all_sync(0xffffffffu, pwait(wempty_bar(slot), par ^ 1u))) { ok = false; break; }
        mbar_arrive_expect_tx_w(leader, wfull_bar(slot), kChunkW4);
        bulk_g2s_w(leader, w_smem(slot), src, kChunkW4, wfull_bar(slot), pol);
#pragma unroll
        for (int j = 0; j < TEAMS; ++j)
          if (j == tm) {
            ++nfill[j];
            if (++s[j] == SWT) { s[j] = 0; ph[j] ^= 1u; }
          }
      }
    }
    // the last fill of every slot has landed before the CTA may exit
#pragma unroll
    for (int j = 0; j < TEAMS; ++j)
      for (int k = 0; k < SWT && k < nfill[j]; ++k)
        mbar_drain(wfull_bar(j * SWT + k), k < s[j] ? ph[j] : ph[j] ^ 1u, wctl);
  } else if (warp == kMsWarpX) {
    // -------------------------------------------------- activation copies --
    const uint32_t leader = elect_leader();
    int s = 0, nfill = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int i = 0; ok && segment(P, cta, i, sg); ++i) {
      for (int g = sg.g0; g < sg.g1; g += kXBlock) {
        if (!__all_sync(0xffffffffu, pwait(xempty_bar(s), ph ^ 1u))) { ok = false; break; }
        mbar_arrive_expect_tx_w(leader, xfull_bar(s), kXBytes);
        ++nfill;
        if constexpr (ACT8) tma_load_3d_w(leader, x_smem(s) + kXBlock * kXChunk, &a.tmap, 0, 0, g, xfull_bar(s));
        else tma_load_3d_w(leader, x_smem(s), &a.tmap, 0, 0, 2 * g, xfull_bar(s));
        if (++s == SX) { s = 0; ph ^= 1u; }
      }
    }
    for (int k = 0; k < SX && k < nfill; ++k) mbar_drain(xfull_bar(k), k < s ? ph : ph ^ 1u, wctl);
  } else if (warp >= kMsWarpC0) {
    // ------------------------------------------------------------ compute --
    const int cw = warp - kMsWarpC0, tm = cw / TW, wi = cw % TW;
    const int g8 = lane >> 2, c4 = lane & 3;
    const int ct = threadIdx.x - kMsWarpC0 * 32;     // 0 .. kCThreads - 1
    // Lane-constant offsets.  ldmatrix: lane l addresses row l % 8 (token 8 jt + l % 8)
    // of matrix l / 8 of a pair of K steps: K step 2 sp + (l / 8) / 2, eight K values
    // (l / 8) % 2, in the 128-byte-swizzled tile (16-byte piece p of row r at
    // (p ^ r % 8) * 16, two 64-wide halves of BNX rows).
    uint32_t xoff[4];
    {
      const int mi = lane >> 3, lrow = lane & 7;
#pragma unroll
      for (int sp = 0; sp < 4; ++sp) {
        const int ks = 2 * sp + (mi >> 1), jch = 2 * (ks & 3) + (mi & 1);
        xoff[sp] = (uint32_t)((ks >> 2) * (BNX * 128) + lrow * 128 + ((jch ^ lrow) << 4));
      }
    }
    // weights: the vector at position ((b * 2 + h) * 4 + c) * 8 + (i ^ 2 c) of the chunk
    // for row block b = RBW wi + r, and the scale pair b * 8 + i
    const uint32_t woff = (uint32_t)(((2 * RBW * wi) * 32 + c4 * 8 + (g8 ^ (2 * c4))) * 16);
    const uint32_t soff = 8192u + (uint32_t)((RBW * wi * 8 + g8) * 4);
    const __half2 k16th = __float2half2_rn(0.0625f);
    const uint32_t zp[4] = {h2_as_u32(__float2half2_rn(-1032.0f)), h2_as_u32(__float2half2_rn(-1032.0f)),
                            h2_as_u32(__float2half2_rn(-1152.0f)), h2_as_u32(__float2half2_rn(-1152.0f))};
    int s = 0, xs = 0, cidx = 0;
    uint32_t ph = 0, xph = 0;
    int npend = 0, pend_tile[2] = {0, 0}, pend_cut[2] = {0, 0};
    const int cut_first = P.cut[cta][0], cut_last = P.cut[cta][1];
    bool aborted = false;
    // a warp that saw a wait give up releases no slot again: the copy it gave up on may
    // still be landing, and a producer released now would arm that slot's phase twice
    bool live = true;
    for (int i = 0; segment(P, cta, i, sg); ++i) {
      float acc[RBW][NT8][4];
#pragma unroll
      for (int r = 0; r < RBW; ++r)
#pragma unroll
        for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[r][jt][e] = 0.0f;
      for (int gb = sg.g0; gb < sg.g1; gb += kXBlock) {
        const int nb = sg.g1 - gb < kXBlock ? sg.g1 - gb : kXBlock;
        // every compute warp waits for every activation block and returns it once;
        // after an abort every wait gives up at once and the loops run out quickly
        live = pwait(xfull_bar(xs), xph) && live;
        if constexpr (ACT8) {
          // the compute warps together widen the block's int8 codes, then all wait
          uint8_t *xb = gbase + (size_t)xs * kXStage;
          for (int j = 0; j < nb; ++j)
            widen_chunk<BNX, kCThreads>(xb + j * kXChunk, xb + kXBlock * kXChunk + j * (BNX * kGroup), ct,
                                        P.M < BNX ? P.M : BNX);
          named_bar_sync(3, kCThreads);
        }
        for (int j = (tm - cidx) & (TEAMS - 1); j < nb; j += TEAMS) {
          const int slot = tm * SWT + s;
          live = pwait(wfull_bar(slot), ph) && live;
          const uint32_t xt = x_smem(xs) + (uint32_t)j * kXChunk;
          const uint32_t wc = w_smem(slot);
          uint32_t sc2[RBW];
#pragma unroll
          for (int r = 0; r < RBW; ++r) sc2[r] = lds32(wc + soff + (uint32_t)(r * 32));
          // KS accumulator sets (K step % KS): MMAs on one accumulator form a dependent
          // chain, and more sets shorten it
          float ga[KS][RBW][NT8][4], gz[KS][NT8][4];
#pragma unroll
          for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                gz[ks][jt][e] = 0.0f;
#pragma unroll
                for (int r = 0; r < RBW; ++r) ga[ks][r][jt][e] = 0.0f;
              }
#pragma unroll
          for (int h = 0; h < 2; ++h) {                  // K steps 4 h .. 4 h + 3
            uint4 v[RBW];
#pragma unroll
            for (int r = 0; r < RBW; ++r) v[r] = lds128(wc + woff + (uint32_t)(r * 1024 + h * 512));
#pragma unroll
            for (int sp2 = 0; sp2 < 2; ++sp2) {
              const int sp = 2 * h + sp2;
              uint32_t bf[2][NT8][2];
#pragma unroll
              for (int jt = 0; jt < NT8; ++jt) {
                ldsm_x4(xt + xoff[sp] + (uint32_t)(jt * 1024), bf[0][jt][0], bf[0][jt][1], bf[1][jt][0],
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
                  for (int jt = 0; jt < NT8; ++jt) mma_16816(gz[kk % KS][jt], zp, bf[kk][jt][0], bf[kk][jt][1]);
                }
#pragma unroll
                for (int r = 0; r < RBW; ++r) {
                  const uint32_t w = wd == 0 ? v[r].x : wd == 1 ? v[r].y : wd == 2 ? v[r].z : v[r].w;
                  uint32_t af[4];
                  if constexpr (kZP) frag_w4_zp(w, af);
                  else frag_w4(w, af);
#pragma unroll
                  for (int jt = 0; jt < NT8; ++jt) mma_16816(ga[kk % KS][r][jt], af, bf[kk][jt][0], bf[kk][jt][1]);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0 && live) mbar_arrive(wempty_bar(slot));
          if (++s == SWT) { s = 0; ph ^= 1u; }
#pragma unroll
          for (int r = 0; r < RBW; ++r) {
            const float2 sf = __half22float2(u32_as_h2(sc2[r]));   // (row R, row R + 8)
#pragma unroll
            for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float gs = 0.0f;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) gs += kZP ? ga[ks][r][jt][e] + gz[ks][jt][e] : ga[ks][r][jt][e];
                acc[r][jt][e] = fmaf(e < 2 ? sf.x : sf.y, gs, acc[r][jt][e]);
              }
          }
        }
        __syncwarp();
        if (lane == 0 && live) mbar_arrive(xempty_bar(xs));
        if (++xs == SX) { xs = 0; xph ^= 1u; }
        cidx += nb;
      }
      // ---- end of the tile segment: the other teams leave their sums in shared
      // memory, the first adds them (team order) and writes the result
      if (tm > 0) {
        float *rt = red + (tm - 1) * (BNX * S);
#pragma unroll
        for (int r = 0; r < RBW; ++r) {
          const int R = 16 * (RBW * wi + r) + g8;
#pragma unroll
          for (int jt = 0; jt < NT8; ++jt) {
            const int t0 = 8 * jt + 2 * c4;
            rt[t0 * S + R] = acc[r][jt][0];
            rt[(t0 + 1) * S + R] = acc[r][jt][1];
            rt[t0 * S + R + 8] = acc[r][jt][2];
            rt[(t0 + 1) * S + R + 8] = acc[r][jt][3];
          }
        }
      }
      if (ct == 0) *decide = wctl->abort;
      named_bar_sync(1, kCThreads);
      if (*decide) aborted = true;
      int u, t;
      tile_coords(P, sg.tile, u, t);
      float *part = sg.slot >= 0 ? a.partials + (size_t)sg.slot * PB : nullptr;
      if (tm == 0 && !aborted) {
        uint32_t tk[NT8][2];                        // lm_head top-k: largest key per token
#pragma unroll
        for (int jt = 0; jt < NT8; ++jt) tk[jt][0] = tk[jt][1] = 0u;
#pragma unroll
        for (int r = 0; r < RBW; ++r) {
          const int R = 16 * (RBW * wi + r) + g8;
#pragma unroll
          for (int jt = 0; jt < NT8; ++jt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int m = 8 * jt + 2 * c4 + (e & 1), row = R + 8 * (e >> 1);
              if (m < P.M) {
                float v = acc[r][jt][e];
#pragma unroll
                for (int q = 0; q < TEAMS - 1; ++q) v += red[q * (BNX * S) + m * S + row];
                if (part) {
                  part[m * kRows + row] = v;
                } else {
                  const __half hv = __float2half_rn(TOKS ? v * __ldg(a.xs + m) : v);
                  a.y[(size_t)m * P.N + t * kRows + row] = __half_as_ushort(hv);
                  if constexpr (kTileMax) tk[jt][e & 1] = max(tk[jt][e & 1], order_key16(hv));
                }
              }
            }
          }
        }
        if (kTileMax && !part) {
          // the eight lanes of a column (g8) hold the warp's rows of the same tokens
#pragma unroll
          for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t k = tk[jt][h];
              k = max(k, __shfl_xor_sync(0xffffffffu, k, 4));
              k = max(k, __shfl_xor_sync(0xffffffffu, k, 8));
              k = max(k, __shfl_xor_sync(0xffffffffu, k, 16));
              const int m = 8 * jt + 2 * c4 + h;
              if (g8 == 0 && m < P.M) atomicMax(a.tile_max + (size_t)m * P.T + t, k);
            }
        }
      }
      // the buffer is free again, and every partial store precedes the publish below
      named_bar_sync(1, kCThreads);
      if (part && !aborted) {
        const int cut = i == 0 ? cut_first : cut_last;
        const int pf = qw::cut_first(cut), pl = qw::cut_last(cut);
        if (ct == 0) {
          const int old = atom_add_acq_rel_gpu(a.counters + sg.tile, 1);
          const int last = (old == pl - pf) ? 1 : 0;
          if (last) a.counters[sg.tile] = 0;     // leave the workspace zeroed for the next call
          *bcast = last;
        }
        named_bar_sync(1, kCThreads);
        if (*bcast) {
          pend_tile[npend] = sg.tile;
          pend_cut[npend++] = cut;
        }
        named_bar_sync(1, kCThreads);             // bcast read by all before it is rewritten
      }
    }
    // ---- stream-K reductions of the cut tiles this CTA finished last: the
    // contributors' partials (the acquire of the ticket and the named barrier order
    // these reads after their release), summed in CTA order
    for (int r = 0; r < npend && !aborted; ++r) {
      const int tile = pend_tile[r];
      const int pf = qw::cut_first(pend_cut[r]), pl = qw::cut_last(pend_cut[r]), pf_slot = qw::cut_slot(pend_cut[r]);
      int u, t;
      tile_coords(P, tile, u, t);
      const int mv = P.M < kMsMaxTokens ? P.M : kMsMaxTokens;
      for (int idx = ct; idx < mv * kRows; idx += kCThreads) {
        const int m = idx >> 7, row = idx & (kRows - 1);
        float v = 0.0f;
        for (int p0 = pf; p0 <= pl; p0 += 4) {
          float x[4];
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            const int p = p0 + pp;
            x[pp] = p <= pl ? __ldcg(a.partials + (size_t)(p == pf ? pf_slot : 2 * p) * PB + idx) : 0.0f;
          }
#pragma unroll
          for (int pp = 0; pp < 4; ++pp)
            if (p0 + pp <= pl) v += x[pp];
        }
        const __half hv = __float2half_rn(TOKS ? v * __ldg(a.xs + m) : v);
        a.y[(size_t)m * P.N + t * kRows + row] = __half_as_ushort(hv);
        // a warp's 32 consecutive idx are 32 rows of one token (kCThreads and kRows are
        // multiples of 32), and whole warps run this loop
        if constexpr (kTileMax) tile_max_warp(a.tile_max + (size_t)m * P.T + t, order_key16(hv));
      }
    }
  }

  // --------------------------------------------------------------- teardown --
  // both copy threads have drained their copies: nothing still writes shared memory
  __syncthreads();
}

}  // namespace qw
