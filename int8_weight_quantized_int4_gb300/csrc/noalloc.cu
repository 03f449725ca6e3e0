// noalloc.cu -- qgemm_w4a16_noalloc: the W4A16 GEMM for callers that cannot
// allocate device memory.
//
// Some callers of this library have no way to hand it scratch memory: a plugin
// running inside a host inference runtime that owns every device allocation and
// passes its kernels only input and output buffers, or a latency-critical
// decode loop in which a cudaMalloc (which may synchronize the whole device and
// stall other streams) is not allowed.  For them this entry point keeps its
// scratch in a fixed array that is part of the library image on every GPU that
// loads it, so a call needs nothing beyond its inputs and outputs.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  The part that must start at zero (the stream-K tile counters) is
// cleared at set-up and left at zero by every successful call.  Calls that may
// run at the same time on the GPU (different streams, or different host
// threads on one device) race on the array and must be serialized by the
// caller.
#include <stdio.h>
#include <mutex>
#include <cuda_runtime.h>
#include "qgemm.h"
#include "launch.h"
#include "schedule.h"

namespace {

// The largest stream-K plan of a token tile of 16 (M <= 16): binary32 partial sums of
// two 16 x 128 tiles per CTA for up to kMaxGrid CTAs, after the fixed tile-counter
// region of every workspace.  Plans that assign whole tiles use only the counters.
constexpr size_t kCounterBytes = (size_t)qw::kStreamKMaxTilesPerSm * qw::kMaxGrid * 4;
constexpr size_t kScratchBytes =
    (kCounterBytes + 255) / 256 * 256 + (size_t)2 * qw::kMaxGrid * 16 * qw::kRows * 4;   // 5 MiB + 40 KiB
static_assert(kScratchBytes == ((size_t)5 << 20) + ((size_t)40 << 10), "scratch size");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDevices];   // device address of the array, per device (null until set up)

// With the device current: look up the array's device address (the host-side symbol
// is only a stand-in and must never reach a kernel).  The lookup allocates nothing
// and runs on every call, so that a module reloaded after a device reset is seen: a
// new address is set up again.  Set-up clears the array and waits for the clear
// (cudaMemset runs on the legacy default stream, which does not order work on
// non-blocking streams), so no kernel of the first call can see it half-done.
int scratch_for_current_device(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return qw::set_last_error(QW_ERR_ARCH, "qgemm_w4a16_noalloc: no usable CUDA device");
  }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    cudaGetLastError();
    return qw::set_last_error(QW_ERR_CUDA, "qgemm_w4a16_noalloc: cudaGetSymbolAddress failed");
  }
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scratch_ptr[dev] != p) {
    e = cudaMemset(p, 0, kScratchBytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      cudaGetLastError();
      return qw::set_last_error(QW_ERR_CUDA, "qgemm_w4a16_noalloc: clearing the scratch failed");
    }
    g_scratch_ptr[dev] = p;
  }
  *out = p;
  return QW_OK;
}

}  // namespace

extern "C" int qgemm_w4a16_noalloc(const uint16_t *x, const void *packed_w4, int M, int N, int K,
                                   uint16_t *y, qw_stream_t stream) {
  if (M < 0 || N < 0 || K < 0)
    return qw::set_last_error(QW_ERR_INVALID_ARG, "qgemm_w4a16_noalloc: negative size");
  if (M == 0 || N == 0 || K == 0 || K % 128 || N % 128)   // rejected or empty: no scratch involved
    return qgemm_w4a16(x, packed_w4, M, N, K, y, nullptr, 0, stream);
  // the size check comes before any device work
  const size_t need = qgemm_workspace_bytes(QW_MODE_W4A16, M, N, K);
  if (need == 0) return qgemm_w4a16(x, packed_w4, M, N, K, y, nullptr, 0, stream);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "qgemm_w4a16_noalloc: M=%d N=%d K=%d needs %zu bytes of scratch, the built-in scratch "
             "holds %zu; use qgemm_w4a16 with a caller-provided workspace",
             M, N, K, need, kScratchBytes);
    return qw::set_last_error(QW_ERR_WORKSPACE, msg);
  }
  void *scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  return qgemm_w4a16(x, packed_w4, M, N, K, y, scratch, kScratchBytes, stream);
}
