// gemm_ms.cu -- instantiations of the decode-batch kernel (warp-level MMA): W4A16, W4A8
// from int8 codes (widened in shared memory) and W4A8 from fp16 codes (written by the
// standalone quantizer); one or two tiles of 8 tokens.
#include "gemm_ms.cuh"

namespace qw {

template <int NT8, int AMODE, int RBW = 2, bool TMAX = false>
static cudaError_t run_ms(const GemmArgs &a, cudaStream_t st) {
  auto *k = qgemm_ms_kernel<NT8, AMODE, RBW, TMAX>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(k), a.P.smem_bytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(reinterpret_cast<const void *>(k), dim3(a.P.grid), dim3(ms_threads()),
                 (size_t)a.P.smem_bytes, st, a);
  count_launch();
  return e;
}

cudaError_t launch_gemm_ms(const GemmArgs &a, int act, cudaStream_t st) {
  // teams = 16-row blocks per warp (plan); four only for eight tokens from fp16
  if ((a.P.ms_teams != 2 && a.P.ms_teams != 4) || a.P.bn != kMsMaxTokens) return cudaErrorInvalidValue;
  const bool one = a.P.M <= 8, four = a.P.ms_teams == 4;
  if (four && !(one && act == kActF16)) return cudaErrorInvalidValue;
  if (act == kActI8) return one ? run_ms<1, kActI8>(a, st) : run_ms<2, kActI8>(a, st);
  if (act == kActCodes16) return one ? run_ms<1, kActCodes16>(a, st) : run_ms<2, kActCodes16>(a, st);
  // the lm_head with top-k: the variant whose epilogue records the tile maxima
  if (a.tile_max) {
    if (four) return run_ms<1, kActF16, 4, true>(a, st);
    return one ? run_ms<1, kActF16, 2, true>(a, st) : run_ms<2, kActF16, 2, true>(a, st);
  }
  if (four) return run_ms<1, kActF16, 4>(a, st);
  return one ? run_ms<1, kActF16>(a, st) : run_ms<2, kActF16>(a, st);
}

}  // namespace qw
