// gemm_w4a8.cu -- instantiations of the tensor-core GEMM for W4A8 (one per token tile size).
#include "gemm_kernel.cuh"

namespace qw {

template <int BN>
static cudaError_t run_w4a8(const GemmArgs &a, cudaStream_t st) {
  auto *k = qgemm_tc_kernel<BN, 4, true, false>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(k), a.P.smem_bytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(reinterpret_cast<const void *>(k), dim3(a.P.grid), dim3(kThreads),
                 (size_t)a.P.smem_bytes, st, a);
  count_launch();
  return e;
}

cudaError_t launch_gemm_w4a8(const GemmArgs &a, cudaStream_t st) {
  switch (a.P.bn) {
    case 16: return run_w4a8<16>(a, st);
    case 32: return run_w4a8<32>(a, st);
    case 64: return run_w4a8<64>(a, st);
    case 128: return run_w4a8<128>(a, st);
    case 256: return run_w4a8<256>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qw
