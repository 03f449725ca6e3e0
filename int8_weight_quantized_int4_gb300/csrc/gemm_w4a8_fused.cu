// gemm_w4a8_fused.cu -- W4A8 GEMM with the per-token activation quantizer inside the
// kernel (fp16 rows copied to shared memory, token tiles of 16).
#include "gemm_kernel.cuh"

namespace qw {

cudaError_t launch_gemm_w4a8_fused(const GemmArgs &a, cudaStream_t st) {
  if (a.P.bn != 16 || !a.P.fused) return cudaErrorInvalidValue;
  auto *k = qgemm_tc_kernel<16, 4, true, true>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(k), a.P.smem_bytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(reinterpret_cast<const void *>(k), dim3(a.P.grid), dim3(kThreads),
                 (size_t)a.P.smem_bytes, st, a);
  count_launch();
  return e;
}

}  // namespace qw
