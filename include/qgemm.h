/*
 * qgemm.h -- C ABI of the GB300 (sm_103a) weight-quantized linear layer.
 *
 * The method: "What this repo does that stock vLLM doesn't"
 * (qwen38-27b-rtx3090 docs/optimizations.md), section "In full":
 *   item 4  int4 weights with symmetric group-128 fp16 scales (about half of them
 *           negative), activations either fp16 (W4A16) or quantized to int8 per
 *           token (W4A8); the bug the page reports came from reading the group
 *           scales as unsigned, and its fix keeps each scale's sign;
 *   item 1  lm_head / embed_tokens requantized to int8 group-128 (~0.6 % error);
 *   item 5  the 248k-row int8 lm_head run for every draft token (W8A16).
 *
 * The linear layer is  y[M,N] = x[M,K] . W^T  with the logical weight
 * W[n,k] = code[n,k] * scale[n, k/128]  (groups of 128 along K).
 *
 * Conventions for every function below:
 *   - All tensors are dense, row-major, and live in device memory owned by the
 *     caller.  The library never allocates device memory and never synchronizes
 *     on the calls marked "async"; they are enqueued on `stream`.
 *   - fp16 means IEEE binary16, passed as its bit pattern (uint16_t).
 *   - Return value: QW_OK (0) or a negative QW_ERR_* code.  Argument checks
 *     happen on the host before anything is enqueued; on an error nothing is
 *     enqueued and qw_last_error_string() describes it.  No C++ exception
 *     crosses this boundary.
 *   - Errors found on the device (a pipeline wait that exceeded its time limit,
 *     int4 codes out of range in qpack_w4) are recorded in a per-device error
 *     word; qw_device_error() reads and clears it.
 *   - Shapes: K and N must be positive multiples of 128.  M = 0 or N = 0 is
 *     an empty problem and returns QW_OK without enqueuing work.
 *   - Alignment, checked on every call (QW_ERR_ALIGNMENT otherwise): GEMM
 *     activations (x, xq), packed weights, weight codes, quantizer input x and
 *     logits 16 bytes; workspaces 256 bytes; quant_act_int8's xq 8 bytes;
 *     embed_gather_w8's output 16 bytes; every other fp16 array (outputs y and
 *     vals, weight scales) 2 bytes, binary32 token scales and int32 ids/indices
 *     4 bytes (their element sizes).
 *   - The device must be compute capability 10.3 (GB300); otherwise QW_ERR_ARCH.
 *   - There is no CPU fallback: every computing call runs hand-written CUDA
 *     kernels on the current device.
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st *qw_stream_t;

enum {
    QW_OK = 0,
    QW_ERR_INVALID_ARG = -1,        /* null pointer, negative size */
    QW_ERR_UNSUPPORTED_SHAPE = -2,  /* K or N not a multiple of 128, or too large */
    QW_ERR_ALIGNMENT = -3,          /* a pointer is below its required alignment */
    QW_ERR_WORKSPACE = -4,          /* workspace missing or smaller than required */
    QW_ERR_ARCH = -5,               /* no device, or the device is not sm_103 */
    QW_ERR_CUDA = -6,               /* a CUDA runtime call failed */
    QW_ERR_TIMEOUT = -7,            /* (device) a pipeline wait exceeded its limit */
    QW_ERR_BAD_CODES = -8,          /* (device) qpack_w4 saw a code outside [-8, 7] */
    QW_ERR_BAD_INDEX = -9           /* (device) embed_gather_w8 saw a row id outside [0, V) */
};

enum { QW_MODE_W4A16 = 0, QW_MODE_W4A8 = 1, QW_MODE_W8A16 = 2, QW_MODE_W4A8_FUSED = 3 };

/* ------------------------------------------------------------------------
 * Weight packing (load time, not on the hot path).
 *
 * Repacks logical weights into the tile-major layout the GEMM kernels stream
 * with one bulk copy per (128 rows x 128 K) chunk.  The sign of every group
 * scale is kept as it is: no folding into the codes, no unsigned
 * reinterpretation ("In full" item 4 describes the failure that unsigned
 * scales caused).
 *
 *   codes   [N, K] int8, device.  qpack_w4: each code in [-8, 7]; a code out of
 *           that range is packed as (code & 15) and sets QW_ERR_BAD_CODES in
 *           the device error word.  qpack_w8: any int8.
 *   scales  [N, K/128] fp16, device, signed.
 *   packed  device buffer of qpack_w4_bytes(N, K) / qpack_w8_bytes(N, K) bytes,
 *           written completely.  Its layout, chunk (t, g) for row tile
 *           t = n/128 and group g = k/128 at byte offset (t*(K/128)+g)*CHUNK:
 *             W4: CHUNK = 8448, in the fragment order of a warp-level
 *                 16 x 16 tensor-core tile (rows R and R + 8 of a 16-row block
 *                 share a word).  Bytes [0, 8192): 512 vectors of 16 bytes;
 *                 vector (b, h, c, i) (row block b = 0..7, K half h = 0..1,
 *                 c = 0..3, i = 0..7) at byte 16*(((b*2 + h)*4 + c)*8 + (i XOR 2c)).
 *                 With R = 128t +
 *                 16b + i and k0 = 128g + 16*(4h + w) + 2c, word w = 0..3 of the
 *                 vector holds 8 nibbles (code + 8); nibble p at bit 4p:
 *                   p = 0, 4: row R,     k0 and k0 + 1
 *                   p = 1, 5: row R,     k0 + 8 and k0 + 9
 *                   p = 2, 6: row R + 8, k0 and k0 + 1
 *                   p = 3, 7: row R + 8, k0 + 8 and k0 + 9.
 *                 Bytes [8192, 8448): scale pairs, pair b*8 + i = (scale of row
 *                 R, scale of row R + 8), fp16.
 *             W8: CHUNK = 16640.  Bytes [0, 16384): for slice j in 0..7 and row
 *                 r, 16 bytes at j*2048 + r*16 hold codes k = 128g + 16j + b
 *                 (b = 0..15, byte b) stored as (code XOR 0x80).  Bytes
 *                 [16384, 16640): the 128 scales, fp16.
 *   Async.  Returns QW_OK, QW_ERR_INVALID_ARG, QW_ERR_UNSUPPORTED_SHAPE,
 *   QW_ERR_ALIGNMENT, QW_ERR_ARCH or QW_ERR_CUDA.
 * ------------------------------------------------------------------------ */
size_t qpack_w4_bytes(int N, int K);   /* N*K/2 + 2*N*(K/128); 0 if the shape is invalid */
size_t qpack_w8_bytes(int N, int K);   /* N*K   + 2*N*(K/128); 0 if the shape is invalid */
int qpack_w4(const int8_t *codes, const uint16_t *scales, int N, int K, void *packed,
             qw_stream_t stream);
int qpack_w8(const int8_t *codes, const uint16_t *scales, int N, int K, void *packed,
             qw_stream_t stream);

/* ------------------------------------------------------------------------
 * Per-token int8 activation quantization ("In full" item 4: activations are
 * quantized to int8 per token).  For each row m:
 *   amax = max_k |x[m,k]|  (binary32),  xs[m] = amax / 127  (IEEE binary32
 *   divide, round to nearest even),  xq[m,k] = clamp(rne(x[m,k] / xs[m]),
 *   -127, 127)  (IEEE divide, then round half to even);  a row of zeros gives
 *   xs[m] = 0 and xq[m,:] = 0.  Codes and scales are bit-exact against that
 *   definition.
 *   x  [M, K] fp16, device.   xq [M, K] int8, device.   xs [M] binary32, device.
 *   K must be a positive multiple of 8.  Async.
 * ------------------------------------------------------------------------ */
int quant_act_int8(const uint16_t *x, int M, int K, int8_t *xq, float *xs, qw_stream_t stream);

/* ------------------------------------------------------------------------
 * Workspace.  qgemm_workspace_bytes() returns the bytes of scratch device
 * memory a qgemm_* call of this mode and shape needs on the current device
 * (0 when it needs none).  The caller allocates it and zero-fills it ONCE
 * before its first use; every call that returns QW_OK leaves its first
 * qgemm_workspace_zero_bytes() bytes zero again, so it can be reused by later
 * calls of any shape whose requirement fits.  A workspace must not be shared by
 * calls that may run concurrently (different streams).  After QW_ERR_TIMEOUT
 * zero-fill it again.
 * ------------------------------------------------------------------------ */
size_t qgemm_workspace_bytes(int mode, int M, int N, int K);
size_t qgemm_workspace_zero_bytes(int mode, int M, int N, int K);

/* ------------------------------------------------------------------------
 * The quantized GEMMs.  y[m,n] = fp16( sum_g scale[n,g] * sum_{k in g}
 * a[m,k] * code[n,k] ), accumulated in binary32 on tensor cores:
 *   qgemm_w4a16  a = x (fp16 [M,K]), int4 weights packed by qpack_w4
 *                ("In full" item 4; the W4A16 body of the model).
 *   qgemm_w4a8   a = xq (int8 [M,K]) and the result is multiplied by xs[m]
 *                (binary32 [M]) -- the output of quant_act_int8 ("In full"
 *                item 4, W4A8).  The int8 products are exact on the fp16
 *                tensor path used here (sm_103a has no int8 tcgen05 MMA).
 *   qgemm_w8a16  a = x (fp16), int8 weights packed by qpack_w8 (the int8
 *                group-128 lm_head, "In full" items 1 and 5).
 *   y [M, N] fp16, device, fully written.  ws / ws_bytes: the workspace above
 *   (may be NULL when qgemm_workspace_bytes() is 0).
 *   Accuracy: max|y - y_ref| / max|y_ref| <= 5e-3 against the binary64
 *   definition; results are bit-identical between repeated calls.
 *   Async.  Returns QW_OK, QW_ERR_INVALID_ARG, QW_ERR_UNSUPPORTED_SHAPE,
 *   QW_ERR_ALIGNMENT, QW_ERR_WORKSPACE, QW_ERR_ARCH or QW_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int qgemm_w4a16(const uint16_t *x, const void *packed_w4, int M, int N, int K, uint16_t *y,
                void *ws, size_t ws_bytes, qw_stream_t stream);
int qgemm_w4a8(const int8_t *xq, const float *xs, const void *packed_w4, int M, int N, int K,
               uint16_t *y, void *ws, size_t ws_bytes, qw_stream_t stream);
int qgemm_w8a16(const uint16_t *x, const void *packed_w8, int M, int N, int K, uint16_t *y,
                void *ws, size_t ws_bytes, qw_stream_t stream);

/* ------------------------------------------------------------------------
 * embed_gather_w8 -- dequant-on-gather embedding from an int8 group-128 table
 * ("In full" items 1 and 2: both embedding matrices requantized to int8
 * group-128 and read through a dequant-on-gather kernel):
 *   out[t, k] = fp16_rne( code[ids[t], k] * scale[ids[t], k / 128] )
 *   ids     [T] int32, device.
 *   packed  the table [V, D] packed by qpack_w8 (the same format as the int8
 *           lm_head); V and D multiples of 128.
 *   out     [T, D] fp16, device, 16-byte aligned, fully written.
 * An id outside [0, V) gives a row of zeros and sets QW_ERR_BAD_INDEX in the
 * device error word.  Async.  Returns QW_OK, QW_ERR_INVALID_ARG,
 * QW_ERR_UNSUPPORTED_SHAPE, QW_ERR_ALIGNMENT, QW_ERR_ARCH or QW_ERR_CUDA.
 * ------------------------------------------------------------------------ */
int embed_gather_w8(const int32_t *ids, int T, const void *packed_w8, int V, int D, uint16_t *out,
                    qw_stream_t stream);

/* ------------------------------------------------------------------------
 * topk_logits -- per row of an [M, N] fp16 logit matrix (for instance the
 * lm_head's output) the k largest values, largest first; equal values are
 * ordered by the smaller column index, and -0 equals +0 ("In full" item 6: the
 * sampler's mask with top-k known on the host is one small top-k).
 *   logits [M, N] fp16, device, 16-byte aligned; N a multiple of 8,
 *          k <= N <= 262144; NaN is out of contract.  1 <= k <= 64.
 *   vals [M, k] fp16 (the logits' own bit patterns), idx [M, k] int32, device.
 *   ws: topk_workspace_bytes(M, N, k) bytes, zero-filled once (the first
 *   topk_workspace_zero_bytes stay zero after every call that returns QW_OK).
 * One launch: each slice of a row keeps its k best by radix selection, and the
 * last slice of the row to finish merges.  Async.  Returns as embed_gather_w8,
 * or QW_ERR_WORKSPACE.
 * ------------------------------------------------------------------------ */
size_t topk_workspace_bytes(int M, int N, int k);
size_t topk_workspace_zero_bytes(int M, int N, int k);
int topk_logits(const uint16_t *logits, int M, int N, int k, uint16_t *vals, int32_t *idx, void *ws,
                size_t ws_bytes, qw_stream_t stream);

/* ------------------------------------------------------------------------
 * qgemm_lm_head_topk -- the lm_head with the sampler's top-k fused in: the
 * logits y = x . W^T of qgemm_w4a16 (mode QW_MODE_W4A16, the GPTQ-int4 head of
 * the serving README's step table) or qgemm_w8a16 (QW_MODE_W8A16, the int8
 * group-128 head, "In full" item 1), bit-identical to those calls, and per row
 * of y its k largest values as topk_logits gives them ("In full" item 6).
 * The GEMM's epilogue records each token's largest logit in every 128-row
 * tile; one small kernel then selects among the tiles that can hold the top k
 * (those whose maximum is at least the k-th largest tile maximum).
 *   x [M, K] fp16 and packed (qpack_w4 or qpack_w8 bytes) as the GEMM;
 *   y [M, N] fp16 logits, written;  vals [M, k] fp16, idx [M, k] int32.
 *   1 <= k <= min(64, N), N <= 262144 (and the GEMM's shape rules).  NaN
 *   logits are out of contract.
 *   ws: qgemm_lm_head_topk_workspace_bytes(mode, M, N, K, k) bytes, 256-byte
 *   aligned, zero-filled once; the first ..._workspace_zero_bytes stay zero
 *   after every call that returns QW_OK (zero-fill again after QW_ERR_TIMEOUT).
 * The GEMM runs on slices of at most 64 tokens (one launch each, the weights
 * read once per slice), then the selection: async.  Returns as qgemm_w4a16, or
 * QW_ERR_INVALID_ARG for another mode or k.
 * ------------------------------------------------------------------------ */
size_t qgemm_lm_head_topk_workspace_bytes(int mode, int M, int N, int K, int k);
size_t qgemm_lm_head_topk_workspace_zero_bytes(int mode, int M, int N, int K, int k);
int qgemm_lm_head_topk(int mode, const uint16_t *x, const void *packed, int M, int N, int K, int k,
                       uint16_t *y, uint16_t *vals, int32_t *idx, void *ws, size_t ws_bytes,
                       qw_stream_t stream);

/* ------------------------------------------------------------------------
 * attn_int8qk_prefill -- causal prefill attention with the scores computed from
 * int8 codes ("What this repo does that stock vLLM doesn't", paragraph "int8-QK
 * prefill attention"):
 *   1. K is smoothed by its per-head channel mean over the S keys (exact
 *      binary64 sum / S, rounded to binary32; K' = fp32(k - mean));
 *   2. every row of K' (one key of one KV head) and of Q (one query of one
 *      head) becomes int8 codes and a binary32 scale: s = amax / 127 (IEEE
 *      divide), code = round-half-to-even(x / s), s = 0 and codes 0 for a zero
 *      row -- the activation quantizer's arithmetic;
 *   3. score[i][j] = (sum_c qcode[i][c] kcode[j][c]) * sq[i] * sk[j] / sqrt(d),
 *      the integer dot products exact on the tensor cores;
 *   4. causal: the T queries are the last T positions of the S-token context
 *      (query i at position S - T + i sees keys 0 .. S - T + i);
 *   5. softmax, then P . V with P in fp16 and fp32 accumulation; out fp16.
 * Query head h reads KV head h / (Hq / Hkv).
 *   q [T][Hq][d], k and v [S][Hkv][d], out [T][Hq][d]: fp16, device, 16-byte
 *   aligned.  d = 256 (the head dimension of the pages' model); T and S
 *   multiples of 128 with T <= S <= 65536; Hkv divides Hq (<= 1024).  The
 *   channel means are bit-exact for S <= 8192.
 *   ws: attn_int8qk_workspace_bytes(...) bytes, 256-byte aligned, no zeroing
 *   needed.  attn_int8qk_workspace_layout fills offsets[0..5] with the byte
 *   offsets in ws of the query codes ([Hq][T][d] fp16 holding the int8 codes),
 *   query scales ([Hq][T] binary32), key codes ([Hkv][S][d] fp16), key scales
 *   ([Hkv][S] binary32), V^T ([Hkv][d][S] fp16) and the total size; they hold
 *   the call's intermediate results afterwards.
 * Three launches, async.  Returns QW_OK, QW_ERR_INVALID_ARG,
 * QW_ERR_UNSUPPORTED_SHAPE, QW_ERR_ALIGNMENT, QW_ERR_WORKSPACE, QW_ERR_ARCH or
 * QW_ERR_CUDA.
 * ------------------------------------------------------------------------ */
size_t attn_int8qk_workspace_bytes(int T, int S, int Hq, int Hkv, int d);
int attn_int8qk_workspace_layout(int T, int S, int Hq, int Hkv, int d, size_t *offsets);
int attn_int8qk_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, int T, int S, int Hq,
                        int Hkv, int d, uint16_t *out, void *ws, size_t ws_bytes, qw_stream_t stream);

/* ------------------------------------------------------------------------
 * qgemm_w4a8_fused -- the W4A8 layer from fp16 activations: y is bit-identical
 * to quant_act_int8(x) followed by qgemm_w4a8 on the same weights ("In full"
 * item 4: activations quantized to int8 per token, int4 weights).
 *   x [M, K] fp16, device, 16-byte aligned.  Other arguments as qgemm_w4a16;
 *   the workspace is qgemm_workspace_bytes(QW_MODE_W4A8_FUSED, M, N, K).
 * When the layer runs on the row-block decode kernel (N / 16 <= 3 x SMs), M <= 2
 * and the M fp16 rows take at most 48 KB (M*K*2 bytes), one launch: every CTA finds
 * the token scales (amax over the whole rows, from L2, while its first weights load)
 * and turns each activation tile into codes in shared memory with the quantizer's
 * exact arithmetic.  Otherwise two launches: the quantizer writes its codes, as fp16
 * values (exact, |q| <= 127), and the token scales into the workspace; the W4A8 GEMM
 * reads the codes as fp16 tiles (no widening of int8 codes) in the same order of
 * summation as qgemm_w4a8, and multiplies by the token scales in its epilogue.  Async.
 * Returns as qgemm_w4a8.
 * ------------------------------------------------------------------------ */
int qgemm_w4a8_fused(const uint16_t *x, const void *packed_w4, int M, int N, int K, uint16_t *y,
                     void *ws, size_t ws_bytes, qw_stream_t stream);

/* ------------------------------------------------------------------------
 * qgemm_w4a16_noalloc -- qgemm_w4a16 for callers that cannot allocate device
 * memory (for instance a plugin inside a host runtime that owns every device
 * allocation and gives its kernels only input and output buffers, or a decode
 * loop in which a cudaMalloc, which may synchronize the device, is not
 * allowed).  The source pages have no counterpart to this entry point.
 *
 * Same arguments and result as qgemm_w4a16 minus the workspace: the scratch
 * memory is a fixed array of 5 MiB + 40 KiB inside the library on every GPU that
 * loads it (held until the process exits).  That covers M <= 16 at any N and K on
 * any device of up to 160 SMs, and shapes whose schedule assigns whole tiles (at
 * least 32 x (number of SMs) output tiles); a shape that needs more returns
 * QW_ERR_WORKSPACE, with the sizes in qw_last_error_string(), before any device
 * work.  The call allocates nothing.  Every call looks up the array's device
 * address (cudaGetSymbolAddress, no allocation); the first call on a device, and
 * the first call after a device reset reloaded the library's module, sets the
 * scratch up: it clears it and waits for the device (cudaDeviceSynchronize), so
 * make that first call outside any stream capture.  Every call on a device shares
 * the same scratch: calls that may overlap on the GPU race and must be serialized
 * by the caller.  After QW_ERR_TIMEOUT the scratch may hold stale counters and
 * the process should stop using this entry point.
 * ------------------------------------------------------------------------ */
int qgemm_w4a16_noalloc(const uint16_t *x, const void *packed_w4, int M, int N, int K, uint16_t *y,
                        qw_stream_t stream);

/* ------------------------------------------------------------------------
 * Options (process-wide, read when a qgemm_* call is made; a CUDA graph keeps
 * the value in force when the call was captured).
 *
 *   QW_OPT_WEIGHTS_IMMUTABLE (default 0).  Every kernel of this library may
 *   start while the preceding kernel on its stream is still finishing
 *   (programmatic dependent launch); by default it touches no global memory
 *   until that kernel has completed.  Setting this option to 1 declares that the
 *   packed weights passed to qgemm_* are never written by the kernel that
 *   immediately precedes the call on its stream (true when the weights were
 *   packed once at load time and the stream was synchronized since).  The GEMM
 *   then streams and dequantizes its weights before that kernel completes, so
 *   consecutive layers overlap.  Leave it 0 when a weight-writing kernel (e.g.
 *   qpack_*) may directly precede a GEMM on the same stream.
 *
 *   QW_OPT_WAIT_LIMIT_US (default 4000000, i.e. 4 s; 0 .. 4000000).  The time
 *   limit, in microseconds, of every wait inside a GEMM kernel (a pipeline stage
 *   waiting for another).  A wait that runs past it ends the kernel early with
 *   QW_ERR_TIMEOUT in the device error word (qw_device_error) and an undefined
 *   y; the workspace must then be zero-filled again.  A test hook: lowering it
 *   (0 makes every wait that is not already satisfied when first checked give
 *   up) drives an unmodified kernel through that path.  Leave it at the default
 *   otherwise.
 *   qw_set_option returns QW_OK or QW_ERR_INVALID_ARG; qw_get_option returns the
 *   value or QW_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------ */
enum { QW_OPT_WEIGHTS_IMMUTABLE = 1, QW_OPT_WAIT_LIMIT_US = 2 };
int qw_set_option(int option, int value);
int qw_get_option(int option);

/* ------------------------------------------------------------------------
 * Diagnostics.
 *   qw_last_error_string  text of the last host-side error of the calling
 *                         thread ("" if none).  Never NULL.
 *   qw_device_error       waits for the work enqueued on `stream` (stream-ordered
 *                         read), returns the device error word of the current
 *                         device (QW_OK, QW_ERR_TIMEOUT, QW_ERR_BAD_CODES or
 *                         QW_ERR_BAD_INDEX) and clears it.  The word is one per
 *                         device: it also holds errors of kernels on other streams
 *                         that completed before the read.  QW_ERR_CUDA if the read
 *                         itself fails.
 *   qw_num_kernel_launches  number of kernels this library has enqueued in
 *                         this process (all devices, all threads).
 * ------------------------------------------------------------------------ */
const char *qw_last_error_string(void);
int qw_device_error(qw_stream_t stream);
long long qw_num_kernel_launches(void);

/* ------------------------------------------------------------------------
 * Measurement and verification tools (not on the GEMM's path).
 *
 *   qw_diag_mma_peak  dense rate of the warp-level tensor-core MMA (mma.sync):
 *       kind 0 f16 x f16 -> f32 (m16n8k16), 1 s8 x s8 -> s32 (m16n8k32),
 *       2 e4m3 x e4m3 -> f32 (m16n8k32), 3 s4 x s4 -> s32 (m16n8k64).  sm_103a has
 *       no int8 tcgen05 MMA, so kind 1 measures the int8 tensor-core rate that the
 *       W4A8 mode ("In full" item 4: int8 tensor cores) is reported against.
 *       Launches `ctas` CTAs of 256 threads; every thread keeps `chains` (1, 2, 4
 *       or 8) independent accumulators and its warp issues iters x chains MMAs on
 *       register operands (8 chains measure the rate, 1 the latency of dependent
 *       MMAs).  sink: ctas*256 binary32, device (written so the work is kept).
 *       *ops (host) = 2*m*n*k per MMA x the MMAs of the launch; the caller times
 *       the launch.  Async.
 *   qw_diag_tc_probe  tcgen05.mma timing at the GEMM's shapes: `grid` CTAs (<= SMs,
 *       one per SM); warps 0..issuers-1 each stream `chunks` chunks of a
 *       128 x n x 128 product (kind 0: kind::f16, 8 MMAs of K = 16; kind 1:
 *       kind::f8f6f4 with e4m3 operands, 4 MMAs of K = 32) into their own
 *       accumulator, A from TMEM (a_tmem = 1) or shared memory.  kind + 2 selects
 *       the warp-collective issue (the whole warp runs the loop, an elected lane
 *       issues: the form of the library's kernels) instead of lane 0 issuing alone
 *       inside a divergent branch.  window 0: one
 *       commit at the end; w >= 1: a commit per chunk, chunk c first waiting for
 *       chunk c - w's commit (a ring of w operand slots).  n*issuers <= 256,
 *       window <= 8.  out: device, grid*4*4 uint64; per (CTA, issuer): issue ns,
 *       wait ns, total ns, chunks done.  Async.
 *   qw_diag_f8f6f4_gemm  d[r][j] = sum_k a[r][k] * b[j][k] (r < 128, j < 16) on
 *       tcgen05 kind::f8f6f4, e4m3 operands given as bytes (a [128][K], b [16][K],
 *       row-major, device, 16-byte aligned), A from TMEM (a_tmem = 1) or shared
 *       memory, fp32 d [128][16] (device).  K = 128..512, a multiple of 128.  Checks
 *       whether int4 x int8 products (int4 codes and the two 4-bit halves of the
 *       int8 codes are exact in e4m3) accumulate exactly.  Async.
 * Return QW_OK, QW_ERR_INVALID_ARG, QW_ERR_ALIGNMENT, QW_ERR_ARCH or QW_ERR_CUDA;
 * a bounded wait that runs out records QW_ERR_TIMEOUT (read by qw_device_error).
 * ------------------------------------------------------------------------ */
int qw_diag_mma_peak(int kind, int ctas, int iters, int chains, float *sink, double *ops,
                     qw_stream_t stream);
int qw_diag_tc_probe(int kind, int a_tmem, int n, int issuers, int chunks, int window,
                     unsigned long long *out, int grid, qw_stream_t stream);
int qw_diag_f8f6f4_gemm(const uint8_t *a, const uint8_t *b, int K, int a_tmem, float *d,
                        qw_stream_t stream);

/* ------------------------------------------------------------------------
 * Schedule query (host only, no device access): how a qgemm call of this shape
 * is split over `num_sms` persistent CTAs.  For tests and tooling.
 * ------------------------------------------------------------------------ */
typedef struct {
    int bn;                 /* tokens per tile (the MMA N): 16, 32, 64, 128 or 256 */
    int token_tiles;        /* ceil(M / bn) */
    int row_tiles;          /* N / 128 */
    int groups;             /* K / 128 */
    long long tiles;        /* token_tiles * row_tiles */
    long long chunks;       /* tiles * groups: one chunk = 128 rows x 128 K */
    int grid;               /* persistent CTAs launched */
    int stream_k;           /* 1: contiguous chunk ranges with a reduction; 0: whole tiles */
    int stages;             /* weight ring depth in shared memory (packed chunks) */
    int smem_bytes;         /* dynamic shared memory per CTA */
    size_t ws_bytes;        /* workspace bytes (see qgemm_workspace_bytes) */
    size_t ws_zero_bytes;   /* leading workspace bytes that must be zero */
    int act_stages;         /* activation ring depth in shared memory (blocks) */
    int act_block;          /* K groups per activation block (one tensor copy) */
    int fused;              /* QW_MODE_W4A8_FUSED: 1 when the quantizer runs inside the GEMM */
    int decode_teams;       /* > 0: int4 weights and M <= 16 run on the decode-batch kernel
                               (warp-level MMA), with this many teams of four warps */
    int decode_row_blocks;  /* > 0: int4 weights and M <= 16 on a layer of at most 3 x
                               num_sms 16-row blocks run on the row-block decode kernel:
                               every CTA owns at most this many whole row blocks (all of K),
                               no stream-K split (stream_k = 0, no segments) */
} qw_plan_t;

int qw_plan(int mode, int M, int N, int K, int num_sms, qw_plan_t *out);

/* The segments (tile, first group, end group, partial slot or -1) CTA `cta`
 * processes under `plan`, in order; returns how many, writing at most `cap`
 * (0 under a row-block plan: see qw_plan_row_blocks). */
int qw_plan_segments(const qw_plan_t *plan, int cta, int cap, long long *tile, int *g0,
                     int *g1, int *slot);

/* Under a row-block plan (decode_row_blocks > 0): the 16-row blocks [*rb_begin, *rb_end)
 * CTA `cta` computes over all of K (rows 16 * rb_begin .. 16 * rb_end - 1 of y).  Returns
 * QW_OK, or QW_ERR_INVALID_ARG for another plan or a CTA outside the grid. */
int qw_plan_row_blocks(const qw_plan_t *plan, int cta, int *rb_begin, int *rb_end);

#ifdef __cplusplus
}
#endif
#endif /* QGEMM_H */
