// gemm_rb.cu -- instantiations of the row-block decode kernel: W4A16 (with and without
// the lm_head's tile maxima), W4A8 from int8 codes, from fp16 codes, and from fp16
// activations quantized in the kernel; one or two tiles of 8 tokens.
#include "gemm_rb.cuh"

namespace qw {

template <int NT8, int AMODE, bool TMAX = false>
static cudaError_t run_rb(const GemmArgs &a, cudaStream_t st) {
  auto *k = qgemm_rb_kernel<NT8, AMODE, TMAX>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(k), a.P.smem_bytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(reinterpret_cast<const void *>(k), dim3(a.P.grid), dim3(rb_threads()),
                 (size_t)a.P.smem_bytes, st, a);
  count_launch();
  return e;
}

cudaError_t launch_gemm_rb(const GemmArgs &a, int act, cudaStream_t st) {
  if (a.P.rb_max < 1 || a.P.rb_max > kRbMax || a.P.M < 1 || a.P.M > kMsMaxTokens) return cudaErrorInvalidValue;
  const bool one = a.P.M <= 8;
  if (act == kActI8) return one ? run_rb<1, kActI8>(a, st) : run_rb<2, kActI8>(a, st);
  if (act == kActCodes16) return one ? run_rb<1, kActCodes16>(a, st) : run_rb<2, kActCodes16>(a, st);
  if (act == kActQuant) return one ? run_rb<1, kActQuant>(a, st) : cudaErrorInvalidValue;
  if (a.tile_max) return one ? run_rb<1, kActF16, true>(a, st) : run_rb<2, kActF16, true>(a, st);
  return one ? run_rb<1, kActF16>(a, st) : run_rb<2, kActF16>(a, st);
}

}  // namespace qw
