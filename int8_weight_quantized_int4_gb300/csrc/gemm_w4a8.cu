// gemm_w4a8.cu -- instantiations of the tensor-core GEMM for W4A8 (one per token tile
// size): int8 codes widened in the kernel (tiles up to 64 tokens) or fp16 codes read as
// fp16 tiles (the widening pass's output, or the quantizer's fp16 codes).
#include "gemm_kernel.cuh"

namespace qw {

template <int BN, bool ACT8>
static cudaError_t run_w4a8(const GemmArgs &a, cudaStream_t st) {
  auto *k = qgemm_tc_kernel<BN, 4, true, false, ACT8>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(k), a.P.smem_bytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(reinterpret_cast<const void *>(k), dim3(a.P.grid), dim3(kThreads),
                 (size_t)a.P.smem_bytes, st, a);
  count_launch();
  return e;
}

// (token tiles of 16 run on the decode-batch kernel)
cudaError_t launch_gemm_w4a8(const GemmArgs &a, bool act8, cudaStream_t st) {
  if (act8) {
    switch (a.P.bn) {
      case 32: return run_w4a8<32, true>(a, st);
      case 64: return run_w4a8<64, true>(a, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.P.bn) {
    case 32: return run_w4a8<32, false>(a, st);
    case 64: return run_w4a8<64, false>(a, st);
    case 128: return run_w4a8<128, false>(a, st);
    case 256: return run_w4a8<256, false>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qw
