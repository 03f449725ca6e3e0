// launch.h -- internal interface between the C ABI (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once
#include <stdint.h>
#include <stddef.h>
#include <cuda.h>            // CUtensorMap (type only; the driver is reached through the runtime)
#include <cuda_runtime.h>
#include "schedule.h"

namespace qw {

struct GemmArgs {
  CUtensorMap tmap;         // activations: fp16 [M,K] (64 x bn boxes, 128-byte swizzle) or
                            // int8 [M,K] (128 x bn boxes) for W4A8 at decode sizes
  CUtensorMap wmap, smap;   // row-block decode kernel: the packed int4 weights seen as
                            // [row tiles][groups][1056 x 8 B]: boxes of one row block's codes
                            // (1 KB) and scales (32 B) over 8 consecutive groups
  Plan P;
  const float *xs;          // token scales [M] (W4A8) or nullptr
  const uint16_t *xf16;     // W4A8 quantized in the kernel: the fp16 activations [M,K]
  const uint8_t *wpack;     // packed weights
  uint16_t *y;              // fp16 [M,N]
  int *counters;            // [tiles] arrival counters (stream-K)
  float *partials;          // [2*grid][bn][128] binary32 partial sums (stream-K)
  int *err;                 // device error word
  int early_weights;        // weights may be streamed before the preceding kernel ends
  unsigned long long wait_ns;   // time limit of a pipeline wait (QW_OPT_WAIT_LIMIT_US)
  uint32_t *tile_max;       // lm_head with top-k: [M][N/128] the largest order key of each
                            // token's outputs in each 128-row tile (raised with atomicMax),
                            // or nullptr
};

void count_launch();
// Record a host-side error for qw_last_error_string(); returns `code`.
int set_last_error(int code, const char *msg);
// Check the current device (sm_103) and return its SM count and the address of its
// device error word; QW_OK or a QW_ERR_* code (recorded for qw_last_error_string()).
int device_info(int *sms, int **err);

// Launch `func` with programmatic stream serialization: it may start while the
// preceding kernel on the stream finishes; every kernel of this library executes
// griddepcontrol.wait before its first global-memory access (the GEMM only
// prefetches weights into L2 before it).
template <typename... Args>
cudaError_t launch_pdl(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       const Args &...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *argv[] = {const_cast<void *>(static_cast<const void *>(&args))...};
  return cudaLaunchKernelExC(&cfg, func, argv);
}
// Raise the dynamic shared-memory limit of `func` on the current device (once).
cudaError_t ensure_smem_attr(const void *func, int bytes);

// per-token quantizer: codes to q (int8 [M,K], or fp16 [M,K] when codes16), scales to s [M]
cudaError_t launch_quant_act(const uint16_t *x, int M, int K, void *q, bool codes16, float *s,
                             cudaStream_t st);
cudaError_t launch_widen_i8(const int8_t *src, uint16_t *dst, size_t n, int sms, cudaStream_t st);
cudaError_t launch_pack_w4(const int8_t *codes, const uint16_t *scales, int N, int K, void *packed,
                           int *err, int sms, cudaStream_t st);
cudaError_t launch_pack_w8(const int8_t *codes, const uint16_t *scales, int N, int K, void *packed,
                           int sms, cudaStream_t st);

// embedding gather and top-k (gather_topk.cu)
struct TopkPlan {
  int slices, slice_len;
  size_t ws_counters, ws_bytes;
};
constexpr int kTopkMaxN = 64 * 4096;
TopkPlan topk_plan(int M, int N, int k);
cudaError_t launch_embed_gather(const int32_t *ids, int T, const void *packed, int V, int D,
                                uint16_t *out, int *err, cudaStream_t st);
cudaError_t launch_topk(const uint16_t *logits, int M, int N, int k, uint16_t *vals, int32_t *idx,
                        void *ws, cudaStream_t st);
// lm_head with top-k: the k best of each row of y [M, N] from the GEMM's tile maxima
// (tile_max [M][N/128] and counters [M], zero, left zero), kTopkSlices CTAs a row whose
// (key, index) pairs go through `pairs` (topk_tiles_pair_bytes(M) bytes)
constexpr int kTopkSlices = 4;
size_t topk_tiles_pair_bytes(int M);
cudaError_t launch_topk_tiles(const uint16_t *y, int M, int N, int k, uint32_t *tile_max, int *counters,
                              unsigned long long *pairs, uint16_t *vals, int32_t *idx, cudaStream_t st);

// int8-QK causal prefill attention (attention.cu): head dimension and block sizes
constexpr int kAttnD = 256;       // head_dim
constexpr int kAttnBlk = 128;     // queries per block and keys per block
struct AttnLaunch {
  const uint16_t *q, *k, *v;      // [T][Hq][d], [S][Hkv][d], [S][Hkv][d] fp16
  uint16_t *out;                  // [T][Hq][d] fp16
  int T, S, Hq, Hkv;
  long long *part;                // [S/128][Hkv][d] channel partial sums (workspace)
  uint16_t *qc, *kc, *vt;         // [Hq][T][d], [Hkv][S][d] fp16 codes; [Hkv][d][S] fp16 V^T
  float *qs, *ks;                 // [Hq][T], [Hkv][S] row scales
  CUtensorMap tq, tk, tv;         // tensor maps of qc, kc, vt
  int *err;
  unsigned long long wait_ns;
};
size_t attn_fwd_smem_bytes();
cudaError_t launch_attn(const AttnLaunch &L, cudaStream_t st);

cudaError_t launch_gemm_w4a16(const GemmArgs &a, cudaStream_t st);
// W4A8 (token scales in the epilogue): act8, int8 codes widened in the kernel (token
// tiles up to kAct8InKernelMaxBn); otherwise fp16 codes read as fp16 tiles
cudaError_t launch_gemm_w4a8(const GemmArgs &a, bool act8, cudaStream_t st);
cudaError_t launch_gemm_w8a16(const GemmArgs &a, cudaStream_t st);
// decode batches (plan.ms_teams > 0); act: 0 fp16 activations (W4A16), 1 int8 codes and
// token scales (W4A8), 2 fp16 codes and token scales (W4A8 after the quantizer)
cudaError_t launch_gemm_ms(const GemmArgs &a, int act, cudaStream_t st);
// decode batches on layers of few rows (plan.rb_max > 0): the row-block kernel, act as above
// or 3: fp16 activations quantized per token in the kernel (plan.fused)
cudaError_t launch_gemm_rb(const GemmArgs &a, int act, cudaStream_t st);

}  // namespace qw
