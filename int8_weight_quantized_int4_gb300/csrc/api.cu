// api.cu -- the C ABI declared in include/qgemm.h: argument checks, device
// checks, planning and launches.  No allocation, no synchronization on the
// compute calls, no CPU fallback.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <atomic>
#include <mutex>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include "qgemm.h"
#include "launch.h"
#include "ptx.cuh"
#include "schedule.h"

// Per-device error word written by the kernels (pipeline timeouts, bad codes).
__device__ int g_qw_err;

namespace {

thread_local char tl_err[512];
std::atomic<long long> g_launches{0};
std::atomic<int> g_opt_weights_immutable{0};
// QW_OPT_WAIT_LIMIT_US: the kernels' default limit unless a test lowers it
constexpr int kDefaultWaitLimitUs = 4000000;
static_assert(1000ull * kDefaultWaitLimitUs == qw::kWaitLimitNs, "default wait limit");
std::atomic<int> g_opt_wait_limit_us{kDefaultWaitLimitUs};

int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(tl_err, sizeof tl_err, fmt, ap);
  va_end(ap);
  return code;
}

int fail_cuda(cudaError_t e, const char *what) {
  return fail(QW_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DevInfo {
  bool ready = false;
  int status = QW_OK;
  int sms = 0;
  int smem_optin = 0;
  int *err = nullptr;
};

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

// Current device, checked to be an sm_103 part; caches SM count and the address
// of the error word.
int current_device(DevInfo *&out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(QW_ERR_ARCH, "no usable CUDA device (%s)", cudaGetErrorString(e));
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (major != 10 || minor != 3) {
      d.status = fail(QW_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                      major, minor);
    } else {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_qw_err);
      if (e != cudaSuccess) d.status = fail_cuda(e, "cudaGetSymbolAddress(error word)");
      d.err = static_cast<int *>(p);
    }
    d.ready = true;
  }
  if (d.status != QW_OK) return fail(d.status, "device %d is not usable by this library", dev);
  out = &d;
  return QW_OK;
}

// cuTensorMapEncodeTiled, fetched once through the runtime's driver entry point
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
bool load_encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
  });
  return g_encode != nullptr;
}

int encode_act_map(CUtensorMap *map, const void *ptr, int M, int K, int bn, int block, bool int8) {
  if (!load_encoder()) return fail(QW_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint32_t estride[3] = {1, 1, 1};
  CUresult r;
  if (int8) {
    // int8 codes [M,K] seen as [K/128][M][128]: one 128 x bn x block box brings the
    // codes of `block` consecutive groups, unswizzled (widened in the kernel)
    const cuuint64_t gdim[3] = {128, (cuuint64_t)M, (cuuint64_t)K / 128};
    const cuuint64_t gstride[2] = {(cuuint64_t)K, 128};
    const cuuint32_t box[3] = {128u, (cuuint32_t)bn, (cuuint32_t)block};
    r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), gdim, gstride, box,
                 estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // fp16 [M,K] seen as [K/64][M][64]: one 64 x bn x (2 block) box lands as the two
    // K-major 64-column halves of `block` consecutive groups, with the 128-byte
    // swizzle the MMA descriptor expects
    const cuuint64_t gdim[3] = {64, (cuuint64_t)M, (cuuint64_t)K / 64};
    const cuuint64_t gstride[2] = {(cuuint64_t)K * 2, 128};
    const cuuint32_t box[3] = {64u, (cuuint32_t)bn, (cuuint32_t)(2 * block)};
    r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), gdim, gstride, box,
                 estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return fail(QW_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return QW_OK;
}

// The packed int4 weights [N/128 row tiles][K/128 groups][8448 B] seen as 8-byte words
// [T][G][1056] for the row-block decode kernel: `codes` boxes are one row block's 1 KB of
// codes (128 words from word 128 b) over kRbXBlock groups; scale boxes its 32 B of scales
// (4 words from word 1024 + 4 b).  Unswizzled, zero fill past the last group.
int encode_weight_maps(CUtensorMap *codes, CUtensorMap *scales, const void *packed, int N, int K) {
  if (!load_encoder()) return fail(QW_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint32_t estride[3] = {1, 1, 1};
  const cuuint64_t gdim[3] = {qw::kChunkW4 / 8, (cuuint64_t)K / 128, (cuuint64_t)N / 128};
  const cuuint64_t gstride[2] = {(cuuint64_t)qw::kChunkW4, (cuuint64_t)qw::kChunkW4 * (K / 128)};
  const cuuint32_t cbox[3] = {128u, (cuuint32_t)qw::kRbXBlock, 1u};
  const cuuint32_t sbox[3] = {4u, (cuuint32_t)qw::kRbXBlock, 1u};
  CUresult r = g_encode(codes, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void *>(packed), gdim, gstride,
                        cbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS)
    r = g_encode(scales, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void *>(packed), gdim, gstride, sbox,
                 estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(QW_ERR_CUDA, "cuTensorMapEncodeTiled (weights) failed (%d)", (int)r);
  return QW_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kMaxN = 1 << 26;
constexpr int kMaxK = 1 << 20;

int check_shape(int M, int N, int K) {
  if (M < 0 || N < 0 || K < 0) return fail(QW_ERR_INVALID_ARG, "negative size (M=%d N=%d K=%d)", M, N, K);
  if (K == 0 || K % 128 || N % 128 || N > kMaxN || K > kMaxK)
    return fail(QW_ERR_UNSUPPORTED_SHAPE,
                "K and N must be positive multiples of 128 (K<=%d, N<=%d); got N=%d K=%d", kMaxK,
                kMaxN, N, K);
  return QW_OK;
}

int gemm_common(int mode, const void *act, const float *xs, const void *packed, int M, int N, int K,
                uint16_t *y, void *ws, size_t ws_bytes, qw_stream_t stream, uint32_t *tile_max = nullptr) {
  int rc = check_shape(M, N, K);
  if (rc) return rc;
  if (M == 0 || N == 0) return QW_OK;
  if (!act || !packed || !y || (mode == QW_MODE_W4A8 && !xs))
    return fail(QW_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(act, 16) || !aligned(packed, 16) || !aligned(y, 2) || (xs && !aligned(xs, 4)) ||
      (ws && !aligned(ws, 256)))
    return fail(QW_ERR_ALIGNMENT, "activations and packed weights must be 16-byte aligned, "
                                  "the workspace 256-byte aligned");
  DevInfo *d = nullptr;
  if ((rc = current_device(d))) return rc;
  qw::Plan P;
  if (qw::make_plan(mode, M, N, K, d->sms, P)) return fail(QW_ERR_UNSUPPORTED_SHAPE, "no plan");
  if (P.stages < 2 || P.smem_bytes > d->smem_optin)
    return fail(QW_ERR_UNSUPPORTED_SHAPE, "pipeline needs %d B of shared memory, device has %d",
                P.smem_bytes, d->smem_optin);
  if (P.ws_bytes > 0 && (!ws || ws_bytes < P.ws_bytes))
    return fail(QW_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", P.ws_bytes,
                ws ? ws_bytes : (size_t)0);
  uint8_t *w = static_cast<uint8_t *>(ws);
  qw::GemmArgs a{};
  a.P = P;
  a.xs = xs;
  a.wpack = static_cast<const uint8_t *>(packed);
  a.y = y;
  a.counters = P.ws_counters ? reinterpret_cast<int *>(w) : nullptr;
  a.partials = P.ws_partials ? reinterpret_cast<float *>(w + P.ws_counters) : nullptr;
  a.err = d->err;
  a.early_weights = g_opt_weights_immutable.load(std::memory_order_relaxed);
  a.wait_ns = 1000ull * (unsigned long long)g_opt_wait_limit_us.load(std::memory_order_relaxed);
  a.tile_max = tile_max;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  // the decode-batch kernels' activation tiles hold 8 or 16 token rows
  const bool decode = P.ms_teams > 0 || P.rb_max > 0;
  const int box_rows = decode ? qw::ms_rows(M) : P.bn;
  if (P.rb_max && (rc = encode_weight_maps(&a.wmap, &a.smap, packed, N, K))) return rc;
  auto launch_decode = [&](int act) {
    return P.rb_max ? qw::launch_gemm_rb(a, act, st) : qw::launch_gemm_ms(a, act, st);
  };
  if (mode == QW_MODE_W4A8_FUSED && P.fused) {
    // the row-block kernel quantizes per token itself: fp16 tiles, as W4A16
    a.xf16 = static_cast<const uint16_t *>(act);
    if ((rc = encode_act_map(&a.tmap, act, M, K, box_rows, P.xblock, false))) return rc;
    e = launch_decode(3);
  } else if (mode == QW_MODE_W4A8_FUSED) {
    // the standalone quantizer writes fp16 codes and token scales into the workspace;
    // the W4A8 GEMM reads the codes as fp16 tiles (plan mode kModeCodes16)
    uint16_t *q = reinterpret_cast<uint16_t *>(w + P.ws_counters + P.ws_partials + P.ws_act);
    float *s = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(q) + qw::align_up((size_t)M * K * 2, 256));
    e = qw::launch_quant_act(static_cast<const uint16_t *>(act), M, K, q, true, s, st);
    if (e != cudaSuccess) return fail_cuda(e, "quant kernel launch");
    a.xs = s;
    if ((rc = encode_act_map(&a.tmap, q, M, K, box_rows, P.xblock, false))) return rc;
    e = decode ? launch_decode(2) : qw::launch_gemm_w4a8(a, false, st);
  } else if (mode == QW_MODE_W4A8 && qw::act8_in_kernel(mode, P.bn)) {
    if ((rc = encode_act_map(&a.tmap, act, M, K, box_rows, P.xblock, true))) return rc;
    e = decode ? launch_decode(1) : qw::launch_gemm_w4a8(a, true, st);
  } else if (mode == QW_MODE_W4A8) {
    uint16_t *wide = reinterpret_cast<uint16_t *>(w + P.ws_counters + P.ws_partials);
    if ((rc = encode_act_map(&a.tmap, wide, M, K, P.bn, P.xblock, false))) return rc;
    e = qw::launch_widen_i8(static_cast<const int8_t *>(act), wide, (size_t)M * K, d->sms, st);
    if (e != cudaSuccess) return fail_cuda(e, "widen kernel launch");
    e = qw::launch_gemm_w4a8(a, false, st);
  } else {
    if ((rc = encode_act_map(&a.tmap, act, M, K, box_rows, P.xblock, false))) return rc;
    e = mode == QW_MODE_W8A16 ? qw::launch_gemm_w8a16(a, st)
        : decode              ? launch_decode(0)
                              : qw::launch_gemm_w4a16(a, st);
  }
  if (e != cudaSuccess) return fail_cuda(e, "GEMM kernel launch");
  return QW_OK;
}

size_t pack_bytes(int N, int K, int bytes_per_code_x2) {
  if (N < 0 || K <= 0 || N % 128 || K % 128 || N > kMaxN || K > kMaxK) return 0;
  return (size_t)N * K * bytes_per_code_x2 / 2 + (size_t)2 * N * (K / 128);
}

int pack_common(int bits, const int8_t *codes, const uint16_t *scales, int N, int K, void *packed,
                qw_stream_t stream) {
  int rc = check_shape(0, N, K);
  if (rc) return rc;
  if (N == 0) return QW_OK;
  if (!codes || !scales || !packed) return fail(QW_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(codes, 16) || !aligned(packed, 16) || !aligned(scales, 2))
    return fail(QW_ERR_ALIGNMENT, "codes and packed buffer must be 16-byte aligned");
  DevInfo *d = nullptr;
  if ((rc = current_device(d))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = bits == 4 ? qw::launch_pack_w4(codes, scales, N, K, packed, d->err, d->sms, st)
                            : qw::launch_pack_w8(codes, scales, N, K, packed, d->sms, st);
  if (e != cudaSuccess) return fail_cuda(e, "pack kernel launch");
  return QW_OK;
}

}  // namespace

namespace qw {

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int set_last_error(int code, const char *msg) { return fail(code, "%s", msg); }

int device_info(int *sms, int **err) {
  DevInfo *d = nullptr;
  const int rc = current_device(d);
  if (rc) return rc;
  if (sms) *sms = d->sms;
  if (err) *err = d->err;
  return QW_OK;
}

cudaError_t ensure_smem_attr(const void *func, int bytes) {
  struct Entry { const void *f; int dev; int bytes; };
  static Entry done[256];
  static int ndone = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < ndone; ++i)
    if (done[i].f == func && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < ndone; ++i)
    if (done[i].f == func && done[i].dev == dev) { done[i].bytes = bytes; return cudaSuccess; }
  if (ndone < 256) done[ndone++] = Entry{func, dev, bytes};
  return cudaSuccess;
}

}  // namespace qw

extern "C" {

size_t qpack_w4_bytes(int N, int K) { return pack_bytes(N, K, 1); }
size_t qpack_w8_bytes(int N, int K) { return pack_bytes(N, K, 2); }

int qpack_w4(const int8_t *codes, const uint16_t *scales, int N, int K, void *packed,
             qw_stream_t stream) {
  return pack_common(4, codes, scales, N, K, packed, stream);
}

int qpack_w8(const int8_t *codes, const uint16_t *scales, int N, int K, void *packed,
             qw_stream_t stream) {
  return pack_common(8, codes, scales, N, K, packed, stream);
}

int quant_act_int8(const uint16_t *x, int M, int K, int8_t *xq, float *xs, qw_stream_t stream) {
  if (M < 0 || K < 0) return fail(QW_ERR_INVALID_ARG, "negative size (M=%d K=%d)", M, K);
  if (K == 0 || K % 8 || K > (1 << 28))
    return fail(QW_ERR_UNSUPPORTED_SHAPE, "K must be a positive multiple of 8; got %d", K);
  if (M == 0) return QW_OK;
  if (!x || !xq || !xs) return fail(QW_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(x, 16) || !aligned(xq, 8) || !aligned(xs, 4))
    return fail(QW_ERR_ALIGNMENT, "x must be 16-byte aligned, xq 8-byte aligned");
  DevInfo *d = nullptr;
  int rc = current_device(d);
  if (rc) return rc;
  cudaError_t e = qw::launch_quant_act(x, M, K, xq, false, xs, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "quant kernel launch");
  return QW_OK;
}

size_t qgemm_workspace_bytes(int mode, int M, int N, int K) {
  DevInfo *d = nullptr;
  if (current_device(d)) return 0;
  qw::Plan P;
  if (qw::make_plan(mode, M, N, K, d->sms, P)) return 0;
  return P.ws_bytes;
}

size_t qgemm_workspace_zero_bytes(int mode, int M, int N, int K) {
  DevInfo *d = nullptr;
  if (current_device(d)) return 0;
  qw::Plan P;
  if (qw::make_plan(mode, M, N, K, d->sms, P)) return 0;
  return P.ws_zero;
}

int qgemm_w4a16(const uint16_t *x, const void *packed_w4, int M, int N, int K, uint16_t *y, void *ws,
                size_t ws_bytes, qw_stream_t stream) {
  return gemm_common(QW_MODE_W4A16, x, nullptr, packed_w4, M, N, K, y, ws, ws_bytes, stream);
}

int qgemm_w4a8(const int8_t *xq, const float *xs, const void *packed_w4, int M, int N, int K,
               uint16_t *y, void *ws, size_t ws_bytes, qw_stream_t stream) {
  return gemm_common(QW_MODE_W4A8, xq, xs, packed_w4, M, N, K, y, ws, ws_bytes, stream);
}

int embed_gather_w8(const int32_t *ids, int T, const void *packed_w8, int V, int D, uint16_t *out,
                    qw_stream_t stream) {
  if (T < 0 || V < 0 || D < 0) return fail(QW_ERR_INVALID_ARG, "negative size");
  if (V % 128 || D % 128 || D == 0 || D > kMaxK || V > kMaxN)
    return fail(QW_ERR_UNSUPPORTED_SHAPE, "V and D must be multiples of 128 (D > 0)");
  if (T == 0) return QW_OK;
  if (!ids || !packed_w8 || !out) return fail(QW_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(packed_w8, 16) || !aligned(out, 16) || !aligned(ids, 4))
    return fail(QW_ERR_ALIGNMENT, "packed table and output must be 16-byte aligned");
  DevInfo *d = nullptr;
  int rc = current_device(d);
  if (rc) return rc;
  cudaError_t e = qw::launch_embed_gather(ids, T, packed_w8, V, D, out, d->err,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "gather kernel launch");
  return QW_OK;
}

static int topk_shape(int M, int N, int k) {
  if (M < 0 || N < 0 || k < 0) return fail(QW_ERR_INVALID_ARG, "negative size");
  if (k < 1 || k > 64 || k > N || N > qw::kTopkMaxN || N % 8)
    return fail(QW_ERR_UNSUPPORTED_SHAPE, "need 1 <= k <= 64, k <= N <= %d, N a multiple of 8",
                qw::kTopkMaxN);
  return QW_OK;
}

size_t topk_workspace_bytes(int M, int N, int k) {
  if (topk_shape(M, N, k)) return 0;
  return qw::topk_plan(M, N, k).ws_bytes;
}

size_t topk_workspace_zero_bytes(int M, int N, int k) {
  if (topk_shape(M, N, k)) return 0;
  return qw::topk_plan(M, N, k).ws_counters;
}

int topk_logits(const uint16_t *logits, int M, int N, int k, uint16_t *vals, int32_t *idx, void *ws,
                size_t ws_bytes, qw_stream_t stream) {
  int rc = topk_shape(M, N, k);
  if (rc) return rc;
  if (M == 0) return QW_OK;
  if (!logits || !vals || !idx) return fail(QW_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(logits, 16) || !aligned(vals, 2) || !aligned(idx, 4) || (ws && !aligned(ws, 256)))
    return fail(QW_ERR_ALIGNMENT, "logits must be 16-byte aligned, the workspace 256-byte aligned");
  const qw::TopkPlan tp = qw::topk_plan(M, N, k);
  if (!ws || ws_bytes < tp.ws_bytes)
    return fail(QW_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", tp.ws_bytes,
                ws ? ws_bytes : (size_t)0);
  DevInfo *d = nullptr;
  if ((rc = current_device(d))) return rc;
  cudaError_t e = qw::launch_topk(logits, M, N, k, vals, idx, ws, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "top-k kernel launch");
  return QW_OK;
}

int qgemm_w4a8_fused(const uint16_t *x, const void *packed_w4, int M, int N, int K, uint16_t *y,
                     void *ws, size_t ws_bytes, qw_stream_t stream) {
  return gemm_common(QW_MODE_W4A8_FUSED, x, nullptr, packed_w4, M, N, K, y, ws, ws_bytes, stream);
}

int qgemm_w8a16(const uint16_t *x, const void *packed_w8, int M, int N, int K, uint16_t *y, void *ws,
                size_t ws_bytes, qw_stream_t stream) {
  return gemm_common(QW_MODE_W8A16, x, nullptr, packed_w8, M, N, K, y, ws, ws_bytes, stream);
}

// ---- lm_head with top-k: workspace = [tile maxima M x N/128 uint32 | row counters M]
// (zero) [GEMM workspace] [selection pairs]
static int lm_head_topk_shape(int mode, int M, int N, int K, int k) {
  if (mode != QW_MODE_W4A16 && mode != QW_MODE_W8A16)
    return fail(QW_ERR_INVALID_ARG, "mode %d: the lm_head with top-k takes QW_MODE_W4A16 or QW_MODE_W8A16", mode);
  int rc = check_shape(M, N, K);
  if (rc) return rc;
  if (N > qw::kTopkMaxN) return fail(QW_ERR_UNSUPPORTED_SHAPE, "N=%d above %d", N, qw::kTopkMaxN);
  if (k < 1 || k > 64 || k > N) return fail(QW_ERR_INVALID_ARG, "k=%d outside 1..min(64, N)", k);
  return QW_OK;
}
static size_t lm_head_tile_bytes(int M, int N) {
  return qw::align_up((size_t)M * (N / 128) * 4, 256) + qw::align_up((size_t)M * 4, 256);
}

// the GEMM runs on slices of at most 64 tokens (token tiles the tile-maxima epilogue has)
constexpr int kLmHeadSlice = 64;

size_t qgemm_lm_head_topk_workspace_bytes(int mode, int M, int N, int K, int k) {
  if (lm_head_topk_shape(mode, M, N, K, k)) return 0;
  return lm_head_tile_bytes(M, N) +
         qw::align_up(qgemm_workspace_bytes(mode, M < kLmHeadSlice ? M : kLmHeadSlice, N, K), 256) +
         qw::topk_tiles_pair_bytes(M);
}

size_t qgemm_lm_head_topk_workspace_zero_bytes(int mode, int M, int N, int K, int k) {
  if (lm_head_topk_shape(mode, M, N, K, k)) return 0;
  return lm_head_tile_bytes(M, N) + qgemm_workspace_zero_bytes(mode, M < kLmHeadSlice ? M : kLmHeadSlice, N, K);
}

int qgemm_lm_head_topk(int mode, const uint16_t *x, const void *packed, int M, int N, int K, int k, uint16_t *y,
                       uint16_t *vals, int32_t *idx, void *ws, size_t ws_bytes, qw_stream_t stream) {
  int rc = lm_head_topk_shape(mode, M, N, K, k);
  if (rc) return rc;
  if (M == 0) return QW_OK;
  if (!vals || !idx) return fail(QW_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(vals, 2) || !aligned(idx, 4) || (ws && !aligned(ws, 256)))
    return fail(QW_ERR_ALIGNMENT, "vals 2-byte, idx 4-byte and the workspace 256-byte aligned");
  const size_t tb = lm_head_tile_bytes(M, N);
  const size_t gb = qw::align_up(qgemm_workspace_bytes(mode, M < kLmHeadSlice ? M : kLmHeadSlice, N, K), 256);
  const size_t need = tb + gb + qw::topk_tiles_pair_bytes(M);
  if (!ws || ws_bytes < need)
    return fail(QW_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws ? ws_bytes : (size_t)0);
  uint8_t *w = static_cast<uint8_t *>(ws);
  uint32_t *tile_max = reinterpret_cast<uint32_t *>(w);
  int *counters = reinterpret_cast<int *>(w + qw::align_up((size_t)M * (N / 128) * 4, 256));
  for (int m0 = 0; m0 < M; m0 += kLmHeadSlice) {
    const int ms = M - m0 < kLmHeadSlice ? M - m0 : kLmHeadSlice;
    rc = gemm_common(mode, x + (size_t)m0 * K, nullptr, packed, ms, N, K, y + (size_t)m0 * N, w + tb, gb, stream,
                     tile_max + (size_t)m0 * (N / 128));
    if (rc) return rc;
  }
  cudaError_t e = qw::launch_topk_tiles(y, M, N, k, tile_max, counters,
                                        reinterpret_cast<unsigned long long *>(w + tb + gb), vals, idx,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "top-k kernel launch");
  return QW_OK;
}

// ---- int8-QK causal prefill attention
struct AttnWs {
  size_t part, qc, qs, kc, ks, vt, total;
};
static AttnWs attn_ws(int T, int S, int Hq, int Hkv) {
  AttnWs w{};
  size_t o = 0;
  auto take = [&](size_t n) {
    const size_t r = o;
    o += qw::align_up(n, 256);
    return r;
  };
  const size_t d = qw::kAttnD;
  w.part = take((size_t)(S / qw::kAttnBlk) * Hkv * d * 8);
  w.qc = take((size_t)Hq * T * d * 2);
  w.qs = take((size_t)Hq * T * 4);
  w.kc = take((size_t)Hkv * S * d * 2);
  w.ks = take((size_t)Hkv * S * 4);
  w.vt = take((size_t)Hkv * d * S * 2);
  w.total = o;
  return w;
}
static int attn_shape(int T, int S, int Hq, int Hkv, int d) {
  if (T < 0 || S < 0 || Hq < 1 || Hkv < 1) return fail(QW_ERR_INVALID_ARG, "bad size (T=%d S=%d Hq=%d Hkv=%d)", T, S, Hq, Hkv);
  if (d != qw::kAttnD) return fail(QW_ERR_UNSUPPORTED_SHAPE, "head_dim %d: only %d", d, qw::kAttnD);
  if (T % qw::kAttnBlk || S % qw::kAttnBlk || T > S || S > 65536 || Hq % Hkv || Hq > 1024)
    return fail(QW_ERR_UNSUPPORTED_SHAPE,
                "T and S must be multiples of %d with T <= S <= 65536, Hkv must divide Hq <= 1024 "
                "(T=%d S=%d Hq=%d Hkv=%d)", qw::kAttnBlk, T, S, Hq, Hkv);
  return QW_OK;
}

size_t attn_int8qk_workspace_bytes(int T, int S, int Hq, int Hkv, int d) {
  if (attn_shape(T, S, Hq, Hkv, d) || T == 0) return 0;
  return attn_ws(T, S, Hq, Hkv).total;
}

int attn_int8qk_workspace_layout(int T, int S, int Hq, int Hkv, int d, size_t *offsets) {
  int rc = attn_shape(T, S, Hq, Hkv, d);
  if (rc) return rc;
  if (!offsets) return fail(QW_ERR_INVALID_ARG, "null output");
  const AttnWs w = attn_ws(T, S, Hq, Hkv);
  offsets[0] = w.qc;
  offsets[1] = w.qs;
  offsets[2] = w.kc;
  offsets[3] = w.ks;
  offsets[4] = w.vt;
  offsets[5] = w.total;
  return QW_OK;
}

int attn_int8qk_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, int T, int S, int Hq, int Hkv,
                        int d, uint16_t *out, void *ws, size_t ws_bytes, qw_stream_t stream) {
  int rc = attn_shape(T, S, Hq, Hkv, d);
  if (rc) return rc;
  if (T == 0) return QW_OK;
  if (!q || !k || !v || !out) return fail(QW_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || (ws && !aligned(ws, 256)))
    return fail(QW_ERR_ALIGNMENT, "q, k, v and out must be 16-byte aligned, the workspace 256-byte aligned");
  const AttnWs w = attn_ws(T, S, Hq, Hkv);
  if (!ws || ws_bytes < w.total)
    return fail(QW_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", w.total, ws ? ws_bytes : (size_t)0);
  DevInfo *dv = nullptr;
  if ((rc = current_device(dv))) return rc;
  if ((int)qw::attn_fwd_smem_bytes() > dv->smem_optin)
    return fail(QW_ERR_UNSUPPORTED_SHAPE, "attention needs %zu B of shared memory, device has %d",
                qw::attn_fwd_smem_bytes(), dv->smem_optin);
  uint8_t *b = static_cast<uint8_t *>(ws);
  qw::AttnLaunch L{};
  L.q = q;
  L.k = k;
  L.v = v;
  L.out = out;
  L.T = T;
  L.S = S;
  L.Hq = Hq;
  L.Hkv = Hkv;
  L.part = reinterpret_cast<long long *>(b + w.part);
  L.qc = reinterpret_cast<uint16_t *>(b + w.qc);
  L.qs = reinterpret_cast<float *>(b + w.qs);
  L.kc = reinterpret_cast<uint16_t *>(b + w.kc);
  L.ks = reinterpret_cast<float *>(b + w.ks);
  L.vt = reinterpret_cast<uint16_t *>(b + w.vt);
  // 128-byte-swizzled boxes: Qc and Kc rows of 256 as four 64-wide slabs of 128 rows;
  // V^T rows of S keys as two 64-key slabs of 256 rows
  if ((rc = encode_act_map(&L.tq, L.qc, Hq * T, qw::kAttnD, qw::kAttnBlk, 2, false))) return rc;
  if ((rc = encode_act_map(&L.tk, L.kc, Hkv * S, qw::kAttnD, qw::kAttnBlk, 2, false))) return rc;
  if ((rc = encode_act_map(&L.tv, L.vt, Hkv * qw::kAttnD, S, qw::kAttnD, 1, false))) return rc;
  L.err = dv->err;
  L.wait_ns = 1000ull * (unsigned long long)g_opt_wait_limit_us.load(std::memory_order_relaxed);
  cudaError_t e = qw::launch_attn(L, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "attention kernel launch");
  return QW_OK;
}

const char *qw_last_error_string(void) { return tl_err; }

int qw_device_error(qw_stream_t stream) {
  DevInfo *d = nullptr;
  int rc = current_device(d);
  if (rc) return rc;
  // stream-ordered: the read sees every kernel enqueued on `stream` before it (and
  // whatever else has completed on the device by then), then the word is cleared
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_qw_err, sizeof v, 0, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail_cuda(e, "read error word");
  static const int zero = 0;
  e = cudaMemcpyToSymbolAsync(g_qw_err, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail_cuda(e, "clear error word");
  return v;
}

long long qw_num_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int qw_set_option(int option, int value) {
  if (option == QW_OPT_WEIGHTS_IMMUTABLE && (value == 0 || value == 1)) {
    g_opt_weights_immutable.store(value, std::memory_order_relaxed);
    return QW_OK;
  }
  if (option == QW_OPT_WAIT_LIMIT_US && value >= 0 && value <= kDefaultWaitLimitUs) {
    g_opt_wait_limit_us.store(value, std::memory_order_relaxed);
    return QW_OK;
  }
  return fail(QW_ERR_INVALID_ARG, "unknown option %d or value %d", option, value);
}

int qw_get_option(int option) {
  if (option == QW_OPT_WEIGHTS_IMMUTABLE) return g_opt_weights_immutable.load(std::memory_order_relaxed);
  if (option == QW_OPT_WAIT_LIMIT_US) return g_opt_wait_limit_us.load(std::memory_order_relaxed);
  return fail(QW_ERR_INVALID_ARG, "unknown option %d", option);
}

int qw_plan(int mode, int M, int N, int K, int num_sms, qw_plan_t *out) {
  if (!out) return fail(QW_ERR_INVALID_ARG, "null output");
  qw::Plan P;
  const int rc = qw::make_plan(mode, M, N, K, num_sms, P);
  if (rc == -1) return fail(QW_ERR_INVALID_ARG, "bad mode or size");
  if (rc) return fail(QW_ERR_UNSUPPORTED_SHAPE, "K and N must be multiples of 128");
  out->bn = P.bn;
  out->token_tiles = P.U;
  out->row_tiles = P.T;
  out->groups = P.G;
  out->tiles = P.tiles;
  out->chunks = P.chunks;
  out->grid = P.grid;
  out->stream_k = P.stream_k;
  out->stages = P.stages;
  out->smem_bytes = P.smem_bytes;
  out->ws_bytes = P.ws_bytes;
  out->ws_zero_bytes = P.ws_zero;
  out->act_stages = P.xstages;
  out->act_block = P.xblock;
  out->fused = P.fused;
  out->decode_teams = P.ms_teams;
  out->decode_row_blocks = P.rb_max;
  return QW_OK;
}

int qw_plan_row_blocks(const qw_plan_t *plan, int cta, int *rb_begin, int *rb_end) {
  if (!plan || plan->decode_row_blocks < 1 || cta < 0 || cta >= plan->grid || !rb_begin || !rb_end)
    return fail(QW_ERR_INVALID_ARG, "bad query");
  // the planner's balanced split of the N / 16 row blocks over the grid
  const long long RB = (long long)plan->row_tiles * 8;
  *rb_begin = (int)(cta * RB / plan->grid);
  *rb_end = (int)((cta + 1) * RB / plan->grid);
  return QW_OK;
}

int qw_plan_segments(const qw_plan_t *plan, int cta, int cap, long long *tile, int *g0, int *g1,
                     int *slot) {
  if (!plan || cta < 0 || cta >= plan->grid || cap < 0) return fail(QW_ERR_INVALID_ARG, "bad query");
  if (plan->decode_row_blocks > 0) return 0;
  qw::Plan P{};
  P.bn = plan->bn;
  P.U = plan->token_tiles;
  P.T = plan->row_tiles;
  P.G = plan->groups;
  P.tiles = (int)plan->tiles;
  P.chunks = (int)plan->chunks;
  P.grid = plan->grid;
  P.stream_k = plan->stream_k;
  qw::fill_begin(P);
  int n = 0;
  qw::Seg s;
  for (int i = 0; qw::segment(P, cta, i, s); ++i, ++n) {
    if (n < cap) {
      if (tile) tile[n] = s.tile;
      if (g0) g0[n] = s.g0;
      if (g1) g1[n] = s.g1;
      if (slot) slot[n] = s.slot;
    }
  }
  return n;
}

}  // extern "C"
