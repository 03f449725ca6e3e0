// diag.cu -- measurement and verification tools beside the GEMM (not on its path):
//
//   qw_diag_mma_peak     dense rate of the warp-level tensor-core MMA (mma.sync) for
//                        f16, s8, e4m3 and s4 operands.  On sm_103a this is the only
//                        int8 tensor-core instruction (tcgen05 has no kind::i8 for this
//                        target), so its s8 rate is the "dense int8 tensor peak" the W4A8
//                        mode is reported against ("In full" item 4 of "What this repo
//                        does that stock vLLM doesn't": int8 tensor cores for W4A8).
//   qw_diag_tc_probe     issue time, completion latency and dense rate of tcgen05.mma
//                        (kind::f16 and kind::f8f6f4, A from TMEM or shared memory) at the
//                        shapes the GEMM issues: one CTA per SM, each issuing thread
//                        streaming "chunks" of 128 x n x 128 products into its own
//                        accumulator.
//   qw_diag_f8f6f4_gemm  one 128 x 16 x K product on tcgen05 kind::f8f6f4 with e4m3
//                        operands (A from TMEM or shared memory), fp32 result: checks
//                        whether int4 x int8 products split into e4m3 terms are exact.
//
// Every wait is bounded; a wait that runs out records QW_ERR_TIMEOUT in the device error
// word and the kernel drains and returns.
#include <stdint.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include "qgemm.h"
#include "launch.h"
#include "ptx.cuh"

namespace qw {
namespace {

constexpr uint64_t kDiagWaitNs = 200000000ull;   // 0.2 s

__device__ bool diag_wait(uint32_t bar, uint32_t parity, int *err) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kDiagWaitNs) {
      atomicCAS(err, 0, QW_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------ mma.sync rate --
// kind 0: m16n8k16 f16 x f16 -> f32;  1: m16n8k32 s8 x s8 -> s32;
//      2: m16n8k32 e4m3 x e4m3 -> f32; 3: m16n8k64 s4 x s4 -> s32.
template <int KIND>
__device__ __forceinline__ void mma_sync_op(uint32_t (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  if constexpr (KIND == 0) {
    float *f = reinterpret_cast<float *>(d);
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(f[0]), "+f"(f[1]), "+f"(f[2]), "+f"(f[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  } else if constexpr (KIND == 1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  } else if constexpr (KIND == 2) {
    float *f = reinterpret_cast<float *>(d);
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(f[0]), "+f"(f[1]), "+f"(f[2]), "+f"(f[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k64.row.col.s32.s4.s4.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
}

constexpr int kPeakThreads = 256;

// CHAINS independent accumulators per thread: 8 saturate the pipe (rate), 1 exposes the
// latency of one MMA that depends on the previous one
template <int KIND, int CHAINS>
__global__ void __launch_bounds__(kPeakThreads) mma_peak_kernel(int iters, float *sink) {
  constexpr int kPeakChains = CHAINS;
  const uint32_t t = blockIdx.x * kPeakThreads + threadIdx.x;
  uint32_t a[4], b[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t r = (t * 2654435761u) ^ (0x9e3779b9u * (i + 1));
    // finite operands: fp16 in [1, 2), e4m3 in [1, 2); any bits for the integer kinds
    a[i] = KIND == 0 ? (0x3c003c00u | (r & 0x03ff03ffu)) : KIND == 2 ? (0x38383838u | (r & 0x07070707u)) : r;
    if (i < 2) b[i] = KIND == 0 ? (0x3c003c00u | ((r >> 7) & 0x03ff03ffu))
                                : KIND == 2 ? (0x38383838u | ((r >> 5) & 0x07070707u)) : (r >> 3) * 2654435761u;
  }
  uint32_t d[kPeakChains][4];
#pragma unroll
  for (int j = 0; j < kPeakChains; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) d[j][e] = 0u;
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < kPeakChains; ++j) mma_sync_op<KIND>(d[j], a, b);
  }
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < kPeakChains; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      s += (KIND == 0 || KIND == 2) ? __uint_as_float(d[j][e]) : (float)(int)d[j][e];
  sink[t] = s;
}

// -------------------------------------------------------- tcgen05 probe ----
struct TcProbe {
  int kind;       // 0: kind::f16 (8 MMAs of K = 16 per chunk), 1: kind::f8f6f4 e4m3 (4 of K = 32)
  int warp_form;  // 0: lane 0 issues inside a divergent branch; 1: the whole warp runs the
                  // loop and an elected lane issues (the form of the library's kernels)
  int a_tmem;     // 1: A from TMEM (a ring of 4 slots), 0: A from shared memory
  int n;          // MMA N
  int issuers;    // issuing warps 0..issuers-1, one accumulator each
  int chunks;     // chunks per issuer
  int window;     // 0: one commit at the end; w >= 1: a commit per chunk into a ring of w
                  // barriers, chunk c waiting for chunk c - w's commit first
  unsigned long long *out;   // [grid][4 issuers][4]: issue ns, wait ns, total ns, chunks done
  int *err;
};

constexpr int kProbeThreads = 128;

// warp-collective kind::f8f6f4 issue (as mma_f16_ts_w / mma_f16_ss_w)
__device__ __forceinline__ void mma_f8_ts_w(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 e, %5, 0;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mma_f8_ss_w(uint32_t leader, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 e, %5, 0;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
constexpr int kProbeMaxWindow = 8;

// F8: kind::f8f6f4 (else kind::f16); A_TMEM: A from TMEM (else shared memory); WARP: the
// warp-collective issue (else lane 0 alone).  The K loop of a chunk is unrolled with no
// branch inside, as in the GEMM.
template <bool F8, bool A_TMEM, bool WARP>
__global__ void __launch_bounds__(kProbeThreads, 1) tc_probe_kernel(const TcProbe p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  constexpr bool f8 = F8;
  const uint32_t row_bytes = f8 ? 128u : 256u;            // one 128-wide K group
  const uint32_t btile = base;                             // n rows
  const uint32_t atile = base + (uint32_t)p.n * row_bytes; // 128 rows (shared-memory A)
  const uint32_t bars = atile + 128u * row_bytes;
  uint8_t *gbars = gbase + (bars - base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // zero both tiles
  for (uint32_t i = threadIdx.x * 16u; i < bars - base; i += kProbeThreads * 16u)
    *reinterpret_cast<uint4 *>(gbase + i) = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x < 4 * kProbeMaxWindow) mbar_init(bars + 8u * threadIdx.x, 1);
  fence_mbar_init();
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(bars + 8u * 4 * kProbeMaxWindow, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbars + 8 * 4 * kProbeMaxWindow);
  // zero the four A slots (columns 256..511)
  {
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0u;
    const uint32_t lb = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
    for (int c = 256; c < 512; c += 32) tmem_st32(tmem + lb + (uint32_t)c, z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int q = warp;
  if (q < p.issuers && (WARP || lane == 0)) {
    const uint32_t leader = WARP ? elect_leader() : 1u;
    const uint32_t idesc = idesc_f16_f32(128, p.n);
    const uint32_t d = tmem + (uint32_t)(q * p.n);
    constexpr int nk = f8 ? 4 : 8;
    const uint64_t bdesc0 = smem_desc_sw128(btile), adesc0 = smem_desc_sw128(atile);
    uint64_t t_issue = 0, t_wait = 0;
    uint32_t phase = 0;   // bit w: parity of ring barrier w
    int done = 0;
    bool ok = true;
    const uint64_t T0 = globaltimer_ns();
    for (int c = 0; c < p.chunks && ok; ++c) {
      const int w = p.window > 0 ? c % p.window : 0;
      const uint32_t bar = bars + 8u * (uint32_t)(q * kProbeMaxWindow + w);
      const uint64_t t0 = globaltimer_ns();
      if (p.window > 0 && c >= p.window) {
        ok = diag_wait(bar, (phase >> w) & 1u, p.err);
        if (WARP) ok = __all_sync(0xffffffffu, ok);
        phase ^= 1u << w;
      }
      const uint64_t t1 = globaltimer_ns();
      const uint32_t a0 = tmem + 256u + (uint32_t)((c & 3) * 64);
#pragma unroll
      for (int k = 0; k < nk; ++k) {
        // K step k: f16 -> 64-wide half k / 4, 32 bytes (16 values) into it; f8 -> 32 bytes
        const uint32_t boff = f8 ? (uint32_t)k * 32u : (uint32_t)((k >> 2) * p.n * 128 + (k & 3) * 32);
        const uint32_t aoff = f8 ? (uint32_t)k * 32u : (uint32_t)((k >> 2) * 128 * 128 + (k & 3) * 32);
        const uint64_t bd = bdesc0 + (uint64_t)(boff >> 4);
        const uint32_t acc = (c > 0 || k > 0) ? 1u : 0u;
        if constexpr (WARP && F8 && A_TMEM) mma_f8_ts_w(leader, d, a0 + (uint32_t)(k * 8), bd, idesc, acc);
        else if constexpr (WARP && F8) mma_f8_ss_w(leader, d, adesc0 + (uint64_t)(aoff >> 4), bd, idesc, acc);
        else if constexpr (WARP && A_TMEM) mma_f16_ts_w(leader, d, a0 + (uint32_t)(k * 8), bd, idesc, acc);
        else if constexpr (WARP) mma_f16_ss_w(leader, d, adesc0 + (uint64_t)(aoff >> 4), bd, idesc, acc);
        else if constexpr (F8 && A_TMEM) mma_f8_ts(d, a0 + (uint32_t)(k * 8), bd, idesc, acc);
        else if constexpr (F8) mma_f8_ss(d, adesc0 + (uint64_t)(aoff >> 4), bd, idesc, acc);
        else if constexpr (A_TMEM) mma_f16_ts(d, a0 + (uint32_t)(k * 8), bd, idesc, acc);
        else mma_f16_ss(d, adesc0 + (uint64_t)(aoff >> 4), bd, idesc, acc);
      }
      if (p.window > 0) {
        if constexpr (WARP) mma_commit_w(leader, bar);
        else mma_commit(bar);
      }
      const uint64_t t2 = globaltimer_ns();
      t_wait += t1 - t0;
      t_issue += t2 - t1;
      ++done;
    }
    // drain: wait for every outstanding commit (or one final commit)
    if (ok) {
      const uint64_t t0 = globaltimer_ns();
      if (p.window == 0) {
        const uint32_t bar = bars + 8u * (uint32_t)(q * kProbeMaxWindow);
        if constexpr (WARP) mma_commit_w(leader, bar);
        else mma_commit(bar);
        ok = diag_wait(bar, 0u, p.err);
        if (WARP) ok = __all_sync(0xffffffffu, ok);
      } else {
        const int pend = p.chunks < p.window ? p.chunks : p.window;
        for (int j = 0; j < pend && ok; ++j) {
          const int c = p.chunks - pend + j;
          const int w = c % p.window;
          ok = diag_wait(bars + 8u * (uint32_t)(q * kProbeMaxWindow + w), (phase >> w) & 1u, p.err);
          if (WARP) ok = __all_sync(0xffffffffu, ok);
          phase ^= 1u << w;
        }
      }
      t_wait += globaltimer_ns() - t0;
    }
    const uint64_t total = globaltimer_ns() - T0;
    if (lane == 0) {
      unsigned long long *o = p.out + ((size_t)blockIdx.x * 4 + q) * 4;
      o[0] = t_issue;
      o[1] = t_wait;
      o[2] = total;
      o[3] = (unsigned long long)done;
    }
    if (!ok) {
      // let anything still in flight finish before the TMEM goes away
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 1000000ull) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------- f8f6f4 exactness check ---
// d[r][j] = sum_k a[r][k] * b[j][k] for r < 128, j < 16, K a multiple of 128 (<= 512),
// a and b given as e4m3 bytes, row-major.  Shared-memory tiles: per 128-wide K block,
// 128-byte rows in the 128-byte swizzle (16-byte piece i of row r at (i ^ (r % 8)) * 16).
constexpr int kF8MaxK = 512;

__global__ void __launch_bounds__(128, 1) f8f6f4_gemm_kernel(const uint8_t *__restrict__ a,
                                                           const uint8_t *__restrict__ b, int K, int a_tmem,
                                                           float *__restrict__ d, int *err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const int KB = K / 128;
  const uint32_t atile = base, btile = base + (uint32_t)KB * 128u * 128u;
  const uint32_t bars = btile + (uint32_t)KB * 16u * 128u;
  uint8_t *gbars = gbase + (bars - base);
  const int warp = threadIdx.x >> 5;
  const int r = threadIdx.x;

  for (int kb = 0; kb < KB; ++kb)
    for (int i = 0; i < 8; ++i) {
      const uint4 v = *reinterpret_cast<const uint4 *>(a + (size_t)r * K + kb * 128 + i * 16);
      *reinterpret_cast<uint4 *>(gbase + (size_t)kb * 16384 + r * 128 + ((i ^ (r & 7)) << 4)) = v;
    }
  for (int u = threadIdx.x; u < KB * 16 * 8; u += 128) {
    const int kb = u / 128, j = (u / 8) % 16, i = u % 8;
    const uint4 v = *reinterpret_cast<const uint4 *>(b + (size_t)j * K + kb * 128 + i * 16);
    *reinterpret_cast<uint4 *>(gbase + (btile - base) + (size_t)kb * 2048 + j * 128 + ((i ^ (j & 7)) << 4)) = v;
  }
  if (threadIdx.x == 0) mbar_init(bars, 1);
  fence_mbar_init();
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(bars + 8, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(gbars + 8);
  const uint32_t lb = (uint32_t)(warp * 32) << 16;
  if (a_tmem) {
    // row r -> TMEM lane r; column 64 + 32 kb + c holds a[r][128 kb + 4c .. 4c + 3]
    for (int kb = 0; kb < KB; ++kb) {
      uint32_t v[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) v[c] = *reinterpret_cast<const uint32_t *>(a + (size_t)r * K + kb * 128 + 4 * c);
      tmem_st32(tmem + lb + 64u + (uint32_t)(32 * kb), v);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_f16_f32(128, 16);
    for (int kb = 0; kb < KB; ++kb)
      for (int k = 0; k < 4; ++k) {
        const uint64_t bd = smem_desc_sw128(btile + (uint32_t)kb * 2048u + (uint32_t)k * 32u);
        const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
        if (a_tmem) mma_f8_ts(tmem, tmem + 64u + (uint32_t)(32 * kb + 8 * k), bd, idesc, acc);
        else mma_f8_ss(tmem, smem_desc_sw128(atile + (uint32_t)kb * 16384u + (uint32_t)k * 32u), bd, idesc, acc);
      }
    mma_commit(bars);
  }
  __syncwarp();
  const bool ok = diag_wait(bars, 0u, err);
  tc_fence_after();
  if (ok) {
    uint32_t v[16];
    tmem_ld16(tmem + lb, v);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) d[r * 16 + j] = __uint_as_float(v[j]);
  } else {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int KIND>
cudaError_t run_peak(int ctas, int iters, int chains, float *sink, cudaStream_t st) {
  if (chains == 1) mma_peak_kernel<KIND, 1><<<ctas, kPeakThreads, 0, st>>>(iters, sink);
  else if (chains == 2) mma_peak_kernel<KIND, 2><<<ctas, kPeakThreads, 0, st>>>(iters, sink);
  else if (chains == 4) mma_peak_kernel<KIND, 4><<<ctas, kPeakThreads, 0, st>>>(iters, sink);
  else mma_peak_kernel<KIND, 8><<<ctas, kPeakThreads, 0, st>>>(iters, sink);
  count_launch();
  return cudaGetLastError();
}

}  // namespace
}  // namespace qw

extern "C" {

int qw_diag_mma_peak(int kind, int ctas, int iters, int chains, float *sink, double *ops, qw_stream_t stream) {
  if (kind < 0 || kind > 3 || ctas < 1 || ctas > (1 << 20) || iters < 1 || !sink || !ops ||
      (chains != 1 && chains != 2 && chains != 4 && chains != 8))
    return qw::set_last_error(QW_ERR_INVALID_ARG, "qw_diag_mma_peak: bad kind, size, chains or pointer");
  int rc = qw::device_info(nullptr, nullptr);
  if (rc) return rc;
  // flops (or integer ops) of one MMA: 2 m n k
  static const double per_mma[4] = {2.0 * 16 * 8 * 16, 2.0 * 16 * 8 * 32, 2.0 * 16 * 8 * 32, 2.0 * 16 * 8 * 64};
  *ops = per_mma[kind] * (double)ctas * (qw::kPeakThreads / 32) * (double)iters * chains;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (kind) {
    case 0: e = qw::run_peak<0>(ctas, iters, chains, sink, st); break;
    case 1: e = qw::run_peak<1>(ctas, iters, chains, sink, st); break;
    case 2: e = qw::run_peak<2>(ctas, iters, chains, sink, st); break;
    default: e = qw::run_peak<3>(ctas, iters, chains, sink, st); break;
  }
  if (e != cudaSuccess) return qw::set_last_error(QW_ERR_CUDA, cudaGetErrorString(e));
  return QW_OK;
}

int qw_diag_tc_probe(int kind, int a_tmem, int n, int issuers, int chunks, int window,
                     unsigned long long *out, int grid, qw_stream_t stream) {
  if (kind < 0 || kind > 3 || n < 16 || n > 256 || n % 16 || issuers < 1 || issuers > 4 ||
      n * issuers > 256 || chunks < 1 || window < 0 || window > qw::kProbeMaxWindow || !out || grid < 1)
    return qw::set_last_error(QW_ERR_INVALID_ARG, "qw_diag_tc_probe: bad argument");
  int sms = 0, *err = nullptr;
  int rc = qw::device_info(&sms, &err);
  if (rc) return rc;
  if (grid > sms) return qw::set_last_error(QW_ERR_INVALID_ARG, "qw_diag_tc_probe: at most one CTA per SM");
  const int row_bytes = (kind & 1) ? 128 : 256;
  // tiles + barriers; at least 120 KB so that one CTA holds an SM (one TMEM allocation each)
  int smem = 1024 + (n + 128) * row_bytes + 1024;
  if (smem < 120 * 1024) smem = 120 * 1024;
  qw::TcProbe p{kind & 1, kind >> 1, a_tmem ? 1 : 0, n, issuers, chunks, window, out, err};
  void (*const kernels[8])(const qw::TcProbe) = {
      qw::tc_probe_kernel<false, false, false>, qw::tc_probe_kernel<false, true, false>,
      qw::tc_probe_kernel<true, false, false>,  qw::tc_probe_kernel<true, true, false>,
      qw::tc_probe_kernel<false, false, true>,  qw::tc_probe_kernel<false, true, true>,
      qw::tc_probe_kernel<true, false, true>,   qw::tc_probe_kernel<true, true, true>};
  const auto kern = kernels[(kind >> 1) * 4 + (kind & 1) * 2 + (a_tmem ? 1 : 0)];
  cudaError_t e = qw::ensure_smem_attr(reinterpret_cast<const void *>(kern), smem);
  if (e == cudaSuccess) {
    kern<<<grid, qw::kProbeThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    qw::count_launch();
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return qw::set_last_error(QW_ERR_CUDA, cudaGetErrorString(e));
  return QW_OK;
}

int qw_diag_f8f6f4_gemm(const uint8_t *a, const uint8_t *b, int K, int a_tmem, float *d, qw_stream_t stream) {
  if (!a || !b || !d || K < 128 || K > qw::kF8MaxK || K % 128)
    return qw::set_last_error(QW_ERR_INVALID_ARG, "qw_diag_f8f6f4_gemm: K must be 128..512, a multiple of 128");
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) % 16 || reinterpret_cast<uintptr_t>(d) % 4)
    return qw::set_last_error(QW_ERR_ALIGNMENT, "qw_diag_f8f6f4_gemm: a and b must be 16-byte aligned");
  int *err = nullptr;
  int rc = qw::device_info(nullptr, &err);
  if (rc) return rc;
  const int smem = 1024 + (K / 128) * (128 + 16) * 128 + 64;
  cudaError_t e = qw::ensure_smem_attr(reinterpret_cast<const void *>(qw::f8f6f4_gemm_kernel), smem);
  if (e == cudaSuccess) {
    qw::f8f6f4_gemm_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(a, b, K, a_tmem ? 1 : 0, d, err);
    qw::count_launch();
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return qw::set_last_error(QW_ERR_CUDA, cudaGetErrorString(e));
  return QW_OK;
}

}  // extern "C"
