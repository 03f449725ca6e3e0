// gemm_w4a16.cu -- instantiations of the tensor-core GEMM for W4A16 (one per token tile size).
#include "gemm_kernel.cuh"

namespace qw {

template <int BN, bool TMAX = false>
static cudaError_t run_w4a16(const GemmArgs &a, cudaStream_t st) {
  auto *k = qgemm_tc_kernel<BN, 4, false, TMAX, false>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(k), a.P.smem_bytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(reinterpret_cast<const void *>(k), dim3(a.P.grid), dim3(kThreads),
                 (size_t)a.P.smem_bytes, st, a);
  count_launch();
  return e;
}

cudaError_t launch_gemm_w4a16(const GemmArgs &a, cudaStream_t st) {
  if (a.tile_max) {
    // the lm_head with top-k (token tiles up to 64; larger batches take the plain GEMM
    // and the standalone top-k)
    switch (a.P.bn) {
      case 16: return run_w4a16<16, true>(a, st);
      case 32: return run_w4a16<32, true>(a, st);
      case 64: return run_w4a16<64, true>(a, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.P.bn) {
    case 16: return run_w4a16<16>(a, st);
    case 32: return run_w4a16<32>(a, st);
    case 64: return run_w4a16<64>(a, st);
    case 128: return run_w4a16<128>(a, st);
    case 256: return run_w4a16<256>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qw
