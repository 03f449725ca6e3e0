// aux_kernels.cu -- the memory-bound kernels around the GEMM: per-token int8
// activation quantizer, weight packers, and the int8 -> fp16 code widening
// used by the W4A8 GEMM.
#include <stdint.h>
#include <type_traits>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include "launch.h"
#include "ptx.cuh"
#include "schedule.h"
#include "quant_code.cuh"

namespace qw {

// --------------------------------------------------------------------------
// Per-token int8 quantization ("In full" item 4 of "What this repo does that
// stock vLLM doesn't": activations quantized to int8 per token).
// One CTA per row.  amax over the row (warp shuffles, then shared memory),
// s = amax / 127 with the IEEE divide, q = rne(x / s) clamped to [-127, 127] -- the IEEE
// quotient's code, found from the reciprocal product except within 2^-14 of a tie
// (quant_code.cuh).
// The row is kept in registers (up to quant_regs(WIDE) 16-byte vectors per thread);
// longer rows are re-read (from L2) for the second pass.
// CODES16: the codes are written as fp16 values (exact: |q| <= 127) for a GEMM that
// reads them as fp16 tiles and applies the token scales in its epilogue, so that no
// widening of int8 codes is needed there; otherwise as int8.
// Two forms, by how the CTAs should share SMs (measured on the 5120 x 5120 W4A8 layer and
// the W4A8 prefill, same box):
//   narrow (WIDE false): 4 vectors a thread, ~48 registers.  Up to 8 tokens its CTAs fit
//     beside the row-block GEMM CTAs still on the SMs and start at once (4 tokens 9.26 ->
//     8.64 us a layer); from 256 tokens several share an SM and the stream runs faster
//     (2048-token prefill projection 136.0 -> 127.8 us).
//   wide (WIDE true): 12 vectors a thread, one CTA per SM stated in the launch bounds
//     (~100 registers; at the default register target this form spilled).  For 16-255
//     tokens, whose CTAs cannot fit beside the GEMM's: the narrow form's CTAs then crowd
//     onto the first SMs to free up (16 tokens 11.44 -> 12.01 us).
constexpr int kQuantThreads = 256;
constexpr int kQuantNarrowMaxTokens = 8, kQuantNarrowMinTokens = 256;
__host__ __device__ constexpr int quant_regs(bool wide) { return wide ? 12 : 4; }

template <bool CODES16, bool WIDE>
__global__ void __launch_bounds__(kQuantThreads, WIDE ? 1 : 0) quant_act_kernel(const uint16_t *__restrict__ x, int K,
                                                                  void *__restrict__ q,
                                                                  float *__restrict__ s) {
  using Out = typename std::conditional<CODES16, uint4, uint2>::type;   // 8 codes
  constexpr int kQuantRegs = quant_regs(WIDE);
  __shared__ float red[kQuantThreads / 32];
  griddep_wait();
  griddep_launch_dependents();
  const size_t row = blockIdx.x;
  const uint4 *xr = reinterpret_cast<const uint4 *>(x + row * (size_t)K);
  const int nv = K / 8;
  uint4 keep[kQuantRegs];
  float amax = 0.0f;
#pragma unroll
  for (int r = 0; r < kQuantRegs; ++r) {
    const int i = threadIdx.x + r * kQuantThreads;
    if (i < nv) {
      keep[r] = __ldg(xr + i);
      const __half2 *h = reinterpret_cast<const __half2 *>(&keep[r]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h[e]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
  }
  for (int i = threadIdx.x + kQuantRegs * kQuantThreads; i < nv; i += kQuantThreads) {
    uint4 v = __ldg(xr + i);
    const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(h[e]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, red[w]);

  const float sc = __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) s[row] = (amax == 0.0f) ? 0.0f : sc;
  Out *qr = reinterpret_cast<Out *>(q) + row * (size_t)(K / 8);

  const float rs = amax == 0.0f ? 0.0f : __frcp_rn(sc);
  auto quant8 = [&](const uint4 &v) -> Out {
    const __half2 *h = reinterpret_cast<const __half2 *>(&v);
    uint32_t out[4] = {0u, 0u, 0u, 0u};
    if (amax != 0.0f) {
      // the eight codes from the reciprocal product; near a tie all eight again from the
      // divide (a rare branch, kept out of the common path's registers)
      int qc[8];
      bool near_tie = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h[e]);
        bool t0, t1;
        qc[2 * e] = quant_code_fast(f.x, rs, t0);
        qc[2 * e + 1] = quant_code_fast(f.y, rs, t1);
        near_tie = near_tie || t0 || t1;
      }
      if (near_tie) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h[e]);
          qc[2 * e] = quant_code_div(f.x, sc);
          qc[2 * e + 1] = quant_code_div(f.y, sc);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int q0 = qc[2 * e], q1 = qc[2 * e + 1];
        if constexpr (CODES16) {
          out[e] = h2_as_u32(__halves2half2(__int2half_rn(q0), __int2half_rn(q1)));
        } else {
          const uint32_t pair = ((uint32_t)(q0 & 0xff)) | ((uint32_t)(q1 & 0xff) << 8);
          out[e >> 1] |= pair << (16 * (e & 1));
        }
      }
    }
    if constexpr (CODES16) return make_uint4(out[0], out[1], out[2], out[3]);
    else return make_uint2(out[0], out[1]);
  };
#pragma unroll
  for (int r = 0; r < kQuantRegs; ++r) {
    const int i = threadIdx.x + r * kQuantThreads;
    if (i < nv) qr[i] = quant8(keep[r]);
  }
  for (int i = threadIdx.x + kQuantRegs * kQuantThreads; i < nv; i += kQuantThreads)
    qr[i] = quant8(__ldg(xr + i));
}

// --------------------------------------------------------------------------
// int8 codes -> fp16 values (exact), for the fp16 tensor-core W4A8 path.
__global__ void widen_i8_kernel(const int8_t *__restrict__ src, uint16_t *__restrict__ dst, size_t n16) {
  griddep_wait();
  griddep_launch_dependents();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint4 o[2];
    uint32_t *op = reinterpret_cast<uint32_t *>(o);
    const __half2 k1152 = __float2half2_rn(1152.0f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t u = w[j] ^ 0x80808080u;       // two's complement -> offset binary (q + 128)
      // (1024 + u) - 1152 = q, exact in fp16
      op[2 * j] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4140)), k1152));
      op[2 * j + 1] = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4342)), k1152));
    }
    uint4 *d = reinterpret_cast<uint4 *>(dst) + 2 * i;
    d[0] = o[0];
    d[1] = o[1];
  }
}

// --------------------------------------------------------------------------
// Packers; see qgemm.h for the layouts.
//
// W4: one thread per 16-byte vector of a chunk: the vector at position
// ((b * 2 + h) * 4 + c) * 8 + (i ^ 2 c) (row block b of 16 rows, K half h, lane quarter
// c, row i of the block's upper-or-lower eight; the XOR keeps both the row-per-thread and
// the fragment-per-lane reads free of shared-memory bank conflicts) holds, in word w, the
// codes of rows R = 16 b + i and R + 8 at the four K offsets k0, k0 + 1, k0 + 8, k0 + 9
// with k0 = 16 (4 h + w) + 2 c.  Nibble p of a word:
//   p = 0, 4: (R, k0), (R, k0 + 1)        p = 1, 5: (R, k0 + 8), (R, k0 + 9)
//   p = 2, 6: (R + 8, k0), (R + 8, k0 + 1) p = 3, 7: (R + 8, k0 + 8), (R + 8, k0 + 9)
// stored as code + 8.  The scales follow as (R, R + 8) pairs, pair b * 8 + i.
__global__ void pack_w4_kernel(const int8_t *__restrict__ codes, const uint16_t *__restrict__ scales,
                               int N, int K, uint8_t *__restrict__ packed, int *err) {
  griddep_wait();
  griddep_launch_dependents();
  const int G = K / kGroup;
  const size_t total = (size_t)N * K / 32;   // 16-byte vectors
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const size_t chunk = idx / 512;
    const int v = (int)(idx % 512);                 // position in the chunk
    const int c = (v >> 3) & 3, i = (v & 7) ^ (2 * c), h = (v >> 5) & 1, b = v >> 6;
    const size_t t = chunk / G;
    const int g = (int)(chunk % G);
    const size_t R = t * kRows + 16 * b + i;
    const int8_t *lo = codes + R * K + (size_t)g * kGroup;
    const int8_t *hi = lo + (size_t)8 * K;
    uint32_t wds[4];
    bool bad = false;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int k0 = 16 * (4 * h + w) + 2 * c;
      const int q[8] = {lo[k0], lo[k0 + 8], hi[k0], hi[k0 + 8], lo[k0 + 1], lo[k0 + 9], hi[k0 + 1], hi[k0 + 9]};
      uint32_t wd = 0;
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        bad |= (q[p] < -8 || q[p] > 7);
        wd |= ((uint32_t)(q[p] + 8) & 15u) << (4 * p);
      }
      wds[w] = wd;
    }
    if (bad) atomicCAS(err, 0, -8);
    uint8_t *dst = packed + chunk * kChunkW4;
    *reinterpret_cast<uint4 *>(dst + v * 16) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
    if (h == 0 && c == 0) {
      const uint32_t pair = (uint32_t)scales[R * G + g] | ((uint32_t)scales[(R + 8) * G + g] << 16);
      *reinterpret_cast<uint32_t *>(dst + 8192 + (b * 8 + i) * 4) = pair;
    }
  }
}

__global__ void pack_w8_kernel(const int8_t *__restrict__ codes, const uint16_t *__restrict__ scales,
                               int N, int K, uint8_t *__restrict__ packed) {
  griddep_wait();
  griddep_launch_dependents();
  const int G = K / kGroup;
  const size_t total = (size_t)N * K / 16;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const size_t chunk = idx / 1024;
    const int j = (int)((idx / 128) % 8);
    const int r = (int)(idx % 128);
    const size_t t = chunk / G;
    const int g = (int)(chunk % G);
    const size_t n = t * kRows + r;
    uint4 v = __ldg(reinterpret_cast<const uint4 *>(codes + n * K + (size_t)g * kGroup + 16 * j));
    v.x ^= 0x80808080u; v.y ^= 0x80808080u; v.z ^= 0x80808080u; v.w ^= 0x80808080u;
    uint8_t *dst = packed + chunk * kChunkW8;
    *reinterpret_cast<uint4 *>(dst + j * 2048 + r * 16) = v;
    if (j == 0) *reinterpret_cast<uint16_t *>(dst + 16384 + r * 2) = scales[n * G + g];
  }
}

// ------------------------------------------------------------- launchers --
static int grid_for(size_t items, int threads, int sms) {
  size_t b = (items + threads - 1) / threads;
  const size_t cap = (size_t)sms * 8;
  if (b > cap) b = cap;
  return (int)(b < 1 ? 1 : b);
}

cudaError_t launch_quant_act(const uint16_t *x, int M, int K, void *q, bool codes16, float *s,
                             cudaStream_t st) {
  const bool wide = M > kQuantNarrowMaxTokens && M < kQuantNarrowMinTokens;
  const void *k = codes16 ? (wide ? reinterpret_cast<const void *>(quant_act_kernel<true, true>)
                                  : reinterpret_cast<const void *>(quant_act_kernel<true, false>))
                          : (wide ? reinterpret_cast<const void *>(quant_act_kernel<false, true>)
                                  : reinterpret_cast<const void *>(quant_act_kernel<false, false>));
  cudaError_t e = launch_pdl(k, dim3(M), dim3(kQuantThreads), 0, st, x, K, q, s);
  count_launch();
  return e;
}

cudaError_t launch_widen_i8(const int8_t *src, uint16_t *dst, size_t n, int sms, cudaStream_t st) {
  const size_t n16 = n / 16;
  cudaError_t e = launch_pdl(reinterpret_cast<const void *>(widen_i8_kernel),
                             dim3(grid_for(n16, 256, sms)), dim3(256), 0, st, src, dst, n16);
  count_launch();
  return e;
}

cudaError_t launch_pack_w4(const int8_t *codes, const uint16_t *scales, int N, int K, void *packed,
                           int *err, int sms, cudaStream_t st) {
  const size_t total = (size_t)N * K / 32;
  uint8_t *out = static_cast<uint8_t *>(packed);
  cudaError_t e = launch_pdl(reinterpret_cast<const void *>(pack_w4_kernel),
                             dim3(grid_for(total, 256, sms)), dim3(256), 0, st, codes, scales, N, K,
                             out, err);
  count_launch();
  return e;
}

cudaError_t launch_pack_w8(const int8_t *codes, const uint16_t *scales, int N, int K, void *packed,
                           int sms, cudaStream_t st) {
  const size_t total = (size_t)N * K / 16;
  uint8_t *out = static_cast<uint8_t *>(packed);
  cudaError_t e = launch_pdl(reinterpret_cast<const void *>(pack_w8_kernel),
                             dim3(grid_for(total, 256, sms)), dim3(256), 0, st, codes, scales, N, K,
                             out);
  count_launch();
  return e;
}

}  // namespace qw
