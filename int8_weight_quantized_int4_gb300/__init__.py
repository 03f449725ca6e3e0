"""Python binding of libqgemm (include/qgemm.h): the GB300 weight-quantized
linear layer.  Argument marshalling only -- every computing step runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback.  PyTorch supplies
device memory and the current CUDA stream.

Entry points (same names as the C ABI):
    qpack_w4(codes, scales) -> packed        qpack_w8(codes, scales) -> packed
    quant_act_int8(x) -> (xq, xs)
    qgemm_w4a16(x, packed, N, K) -> y        qgemm_w4a8(xq, xs, packed, N, K) -> y
    qgemm_w4a8_fused(x, packed, N, K) -> y
    qgemm_w8a16(x, packed, N, K) -> y
    embed_gather_w8(ids, packed, V, D) -> out        topk_logits(logits, k) -> (vals, idx)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqgemm.so")

QW_OK = 0
QW_ERR_INVALID_ARG = -1
QW_ERR_UNSUPPORTED_SHAPE = -2
QW_ERR_ALIGNMENT = -3
QW_ERR_WORKSPACE = -4
QW_ERR_ARCH = -5
QW_ERR_CUDA = -6
QW_ERR_TIMEOUT = -7
QW_ERR_BAD_CODES = -8
QW_ERR_BAD_INDEX = -9
MODE_W4A16, MODE_W4A8, MODE_W8A16, MODE_W4A8_FUSED = 0, 1, 2, 3

# every function the header declares: name -> (restype, argtypes)
_p, _i, _sz, _ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong


class Plan(ctypes.Structure):
    _fields_ = [("bn", _i), ("token_tiles", _i), ("row_tiles", _i), ("groups", _i),
                ("tiles", _ll), ("chunks", _ll), ("grid", _i), ("stream_k", _i), ("stages", _i),
                ("smem_bytes", _i), ("ws_bytes", _sz), ("ws_zero_bytes", _sz),
                ("act_stages", _i), ("act_block", _i), ("fused", _i), ("decode_teams", _i),
                ("decode_row_blocks", _i)]


SIGNATURES = {
    "qpack_w4_bytes": (_sz, [_i, _i]),
    "qpack_w8_bytes": (_sz, [_i, _i]),
    "qpack_w4": (_i, [_p, _p, _i, _i, _p, _p]),
    "qpack_w8": (_i, [_p, _p, _i, _i, _p, _p]),
    "quant_act_int8": (_i, [_p, _i, _i, _p, _p, _p]),
    "qgemm_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "qgemm_workspace_zero_bytes": (_sz, [_i, _i, _i, _i]),
    "qgemm_w4a16": (_i, [_p, _p, _i, _i, _i, _p, _p, _sz, _p]),
    "qgemm_w4a8": (_i, [_p, _p, _p, _i, _i, _i, _p, _p, _sz, _p]),
    "qgemm_w4a8_fused": (_i, [_p, _p, _i, _i, _i, _p, _p, _sz, _p]),
    "embed_gather_w8": (_i, [_p, _i, _p, _i, _i, _p, _p]),
    "topk_workspace_bytes": (_sz, [_i, _i, _i]),
    "topk_workspace_zero_bytes": (_sz, [_i, _i, _i]),
    "topk_logits": (_i, [_p, _i, _i, _i, _p, _p, _p, _sz, _p]),
    "qgemm_w8a16": (_i, [_p, _p, _i, _i, _i, _p, _p, _sz, _p]),
    "qgemm_w4a16_noalloc": (_i, [_p, _p, _i, _i, _i, _p, _p]),
    "qgemm_lm_head_topk_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "qgemm_lm_head_topk_workspace_zero_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "qgemm_lm_head_topk": (_i, [_i, _p, _p, _i, _i, _i, _i, _p, _p, _p, _p, _sz, _p]),
    "attn_int8qk_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "attn_int8qk_workspace_layout": (_i, [_i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_size_t)]),
    "attn_int8qk_prefill": (_i, [_p, _p, _p, _i, _i, _i, _i, _i, _p, _p, _sz, _p]),
    "qw_last_error_string": (ctypes.c_char_p, []),
    "qw_device_error": (_i, [_p]),
    "qw_num_kernel_launches": (_ll, []),
    "qw_set_option": (_i, [_i, _i]),
    "qw_get_option": (_i, [_i]),
    "qw_diag_mma_peak": (_i, [_i, _i, _i, _i, _p, ctypes.POINTER(ctypes.c_double), _p]),
    "qw_diag_tc_probe": (_i, [_i, _i, _i, _i, _i, _i, _p, _i, _p]),
    "qw_diag_f8f6f4_gemm": (_i, [_p, _p, _i, _i, _p, _p]),
    "qw_plan": (_i, [_i, _i, _i, _i, _i, ctypes.POINTER(Plan)]),
    "qw_plan_segments": (_i, [ctypes.POINTER(Plan), _i, _i, _p, _p, _p, _p]),
    "qw_plan_row_blocks": (_i, [ctypes.POINTER(Plan), _i, _p, _p]),
}

_lib = None
_lock = threading.Lock()


class QgemmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"qgemm error {code}: {msg}")
        self.code = code


def lib():
    """Load libqgemm.so (built by build.py / __graft_entry__.build()); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with "
                                  "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _check(rc: int):
    if rc != QW_OK:
        raise QgemmError(rc, lib().qw_last_error_string().decode())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def _need_shape(t, shape, name):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _need_packed(packed, nbytes, like, name="packed"):
    """A packed weight buffer: a contiguous uint8 CUDA tensor on `like`'s device holding at
    least the nbytes the layout needs for the given shape (the kernels read all of them)."""
    _need(packed, torch.uint8, name)
    if packed.device != like.device:
        raise ValueError(f"{name} is on {packed.device}, the activations on {like.device}")
    if nbytes <= 0:
        return                          # an unsupported shape: the library rejects it
    if packed.numel() < nbytes:
        raise ValueError(f"{name} holds {packed.numel()} bytes, the layout needs {nbytes}")


# ------------------------------------------------------------------ packing --
def qpack_w4_bytes(N: int, K: int) -> int:
    return int(lib().qpack_w4_bytes(N, K))


def qpack_w8_bytes(N: int, K: int) -> int:
    return int(lib().qpack_w8_bytes(N, K))


def _pack(bits, codes, scales, out=None):
    _need(codes, torch.int8, "codes", 2)
    _need(scales, torch.float16, "scales", 2)
    N, K = codes.shape
    nbytes = (qpack_w4_bytes if bits == 4 else qpack_w8_bytes)(N, K)
    _need_shape(scales, (N, K // 128), "scales")
    if out is None:
        out = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=codes.device)
    elif nbytes > 0:
        _need_packed(out, nbytes, codes, "out")
    fn = lib().qpack_w4 if bits == 4 else lib().qpack_w8
    with torch.cuda.device(codes.device):
        _check(fn(_ptr(codes), _ptr(scales), N, K, _ptr(out), _stream(codes)))
    return out


def qpack_w4(codes: torch.Tensor, scales: torch.Tensor, out: torch.Tensor | None = None):
    """int4 codes int8 [N,K] in [-8,7] + signed fp16 scales [N,K/128] -> packed uint8 buffer."""
    return _pack(4, codes, scales, out)


def qpack_w8(codes: torch.Tensor, scales: torch.Tensor, out: torch.Tensor | None = None):
    """int8 codes [N,K] + signed fp16 scales [N,K/128] -> packed uint8 buffer."""
    return _pack(8, codes, scales, out)


# ------------------------------------------------------- activation quant --
def quant_act_int8(x: torch.Tensor, xq: torch.Tensor | None = None, xs: torch.Tensor | None = None):
    """fp16 [M,K] -> (int8 codes [M,K], binary32 per-token scales [M])."""
    _need(x, torch.float16, "x", 2)
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    _need(xq, torch.int8, "xq", 2)
    _need_shape(xq, (M, K), "xq")
    if xs is None:
        xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(xs, torch.float32, "xs", 1)
    _need_shape(xs, (M,), "xs")
    with torch.cuda.device(x.device):
        _check(lib().quant_act_int8(_ptr(x), M, K, _ptr(xq), _ptr(xs), _stream(x)))
    return xq, xs


# -------------------------------------------------------------- workspace --
def workspace_bytes(mode: int, M: int, N: int, K: int) -> int:
    return int(lib().qgemm_workspace_bytes(mode, M, N, K))


class Workspace:
    """A zero-initialised device workspace that grows on demand (one per stream)."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, mode: int, M: int, N: int, K: int):
        with torch.cuda.device(self.device):
            need = workspace_bytes(mode, M, N, K)
        if need == 0:
            return None, 0
        if self.buf is None or self.buf.numel() < need:
            self.buf = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self.buf, self.buf.numel()

    def get_bytes(self, need: int):
        """The buffer, grown to at least `need` bytes (zero-filled when grown)."""
        if need == 0:
            return None, 0
        if self.buf is None or self.buf.numel() < need:
            self.buf = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self.buf, self.buf.numel()

    def zero(self):
        """Zero-fill the buffer again (needed after a call that ended in QW_ERR_TIMEOUT)."""
        if self.buf is not None:
            self.buf.zero_()


_default_ws = {}


def _ws_for(t, mode, M, N, K, ws):
    if ws is None:
        key = (t.device, torch.cuda.current_stream(t.device).cuda_stream)
        ws = _default_ws.setdefault(key, Workspace(t.device))
    return ws.get(mode, M, N, K)


# ------------------------------------------------------------------ GEMMs --
def _out(y, M, N, dev):
    if y is None:
        return torch.empty((M, N), dtype=torch.float16, device=dev)
    _need(y, torch.float16, "y", 2)
    if tuple(y.shape) != (M, N):
        raise ValueError("y has the wrong shape")
    return y


def qgemm_w4a16(x, packed, N: int, K: int, y=None, ws: Workspace | None = None):
    """y[M,N] = x[M,K] . W^T with W int4 group-128 (packed by qpack_w4), fp16 out."""
    _need(x, torch.float16, "x", 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    y = _out(y, M, N, x.device)
    if M and N:
        _need_packed(packed, qpack_w4_bytes(N, K), x)
    wbuf, wbytes = _ws_for(x, MODE_W4A16, M, N, K, ws)
    with torch.cuda.device(x.device):
        _check(lib().qgemm_w4a16(_ptr(x), _ptr(packed), M, N, K, _ptr(y), _ptr(wbuf), wbytes,
                                 _stream(x)))
    return y


def qgemm_w4a8(xq, xs, packed, N: int, K: int, y=None, ws: Workspace | None = None):
    """y[M,N] = xs[m] * (xq[M,K] . W^T) with int8 per-token activations, int4 weights."""
    _need(xq, torch.int8, "xq", 2)
    _need(xs, torch.float32, "xs", 1)
    M = xq.shape[0]
    if xq.shape[1] != K or xs.shape[0] != M:
        raise ValueError("shape mismatch")
    y = _out(y, M, N, xq.device)
    if M and N:
        _need_packed(packed, qpack_w4_bytes(N, K), xq)
    wbuf, wbytes = _ws_for(xq, MODE_W4A8, M, N, K, ws)
    with torch.cuda.device(xq.device):
        _check(lib().qgemm_w4a8(_ptr(xq), _ptr(xs), _ptr(packed), M, N, K, _ptr(y), _ptr(wbuf),
                                wbytes, _stream(xq)))
    return y


def qgemm_w4a8_fused(x, packed, N: int, K: int, y=None, ws: Workspace | None = None):
    """The W4A8 layer from fp16 activations: bit-identical to qgemm_w4a8 applied to
    quant_act_int8(x).  Small decode batches quantize inside the row-block GEMM; otherwise
    the quantizer writes fp16 codes that the GEMM reads as fp16 tiles."""
    _need(x, torch.float16, "x", 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    y = _out(y, M, N, x.device)
    if M and N:
        _need_packed(packed, qpack_w4_bytes(N, K), x)
    wbuf, wbytes = _ws_for(x, MODE_W4A8_FUSED, M, N, K, ws)
    with torch.cuda.device(x.device):
        _check(lib().qgemm_w4a8_fused(_ptr(x), _ptr(packed), M, N, K, _ptr(y), _ptr(wbuf), wbytes,
                                      _stream(x)))
    return y


def qgemm_w8a16(x, packed, N: int, K: int, y=None, ws: Workspace | None = None):
    """y[M,N] = x[M,K] . W^T with W int8 group-128 (packed by qpack_w8), fp16 out."""
    _need(x, torch.float16, "x", 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    y = _out(y, M, N, x.device)
    if M and N:
        _need_packed(packed, qpack_w8_bytes(N, K), x)
    wbuf, wbytes = _ws_for(x, MODE_W8A16, M, N, K, ws)
    with torch.cuda.device(x.device):
        _check(lib().qgemm_w8a16(_ptr(x), _ptr(packed), M, N, K, _ptr(y), _ptr(wbuf), wbytes,
                                 _stream(x)))
    return y


def embed_gather_w8(ids, packed, V: int, D: int, out=None):
    """out[t] = the dequantized row ids[t] of an int8 group-128 table [V, D] packed by
    qpack_w8: fp16(code * scale).  ids int32 [T] on the device."""
    _need(ids, torch.int32, "ids", 1)
    T = ids.shape[0]
    if out is None:
        out = torch.empty((T, D), dtype=torch.float16, device=ids.device)
    _need(out, torch.float16, "out", 2)
    _need_shape(out, (T, D), "out")
    if T:
        _need_packed(packed, qpack_w8_bytes(V, D), ids)
    with torch.cuda.device(ids.device):
        _check(lib().embed_gather_w8(_ptr(ids), T, _ptr(packed), V, D, _ptr(out), _stream(ids)))
    return out


def attn_int8qk_prefill(q, k, v, out=None, ws: Workspace | None = None):
    """int8-QK causal prefill attention: q [T,Hq,d], k and v [S,Hkv,d] fp16 on the device
    (the T queries are the context's last T positions) -> out [T,Hq,d] fp16."""
    _need(q, torch.float16, "q", 3)
    _need(k, torch.float16, "k", 3)
    _need(v, torch.float16, "v", 3)
    T, Hq, d = q.shape
    S, Hkv, dk = k.shape
    if dk != d or tuple(v.shape) != (S, Hkv, d):
        raise ValueError("k and v must be [S, Hkv, d] with q's d")
    if out is None:
        out = torch.empty((T, Hq, d), dtype=torch.float16, device=q.device)
    _need(out, torch.float16, "out", 3)
    _need_shape(out, (T, Hq, d), "out")
    if ws is None:
        key = (q.device, torch.cuda.current_stream(q.device).cuda_stream, "attn")
        ws = _default_ws.setdefault(key, Workspace(q.device))
    with torch.cuda.device(q.device):
        wbuf, wbytes = ws.get_bytes(int(lib().attn_int8qk_workspace_bytes(T, S, Hq, Hkv, d)))
        _check(lib().attn_int8qk_prefill(_ptr(q), _ptr(k), _ptr(v), T, S, Hq, Hkv, d, _ptr(out), _ptr(wbuf),
                                         wbytes, _stream(q)))
    return out


def attn_int8qk_intermediates(ws: Workspace, T: int, S: int, Hq: int, Hkv: int, d: int = 256):
    """Views into the workspace of the last attn_int8qk_prefill call with these sizes:
    (query codes [Hq,T,d], query scales [Hq,T], key codes [Hkv,S,d], key scales [Hkv,S],
    V^T [Hkv,d,S]); codes as fp16 tensors holding the int8 values."""
    off = (ctypes.c_size_t * 6)()
    _check(lib().attn_int8qk_workspace_layout(T, S, Hq, Hkv, d, off))
    b = ws.buf

    def view(o, n, dt, shape):
        return b[o:o + n * torch.tensor([], dtype=dt).element_size()].view(dt).view(shape)
    return (view(off[0], Hq * T * d, torch.float16, (Hq, T, d)), view(off[1], Hq * T, torch.float32, (Hq, T)),
            view(off[2], Hkv * S * d, torch.float16, (Hkv, S, d)), view(off[3], Hkv * S, torch.float32, (Hkv, S)),
            view(off[4], Hkv * d * S, torch.float16, (Hkv, d, S)))


_topk_ws = {}


def qgemm_lm_head_topk(mode: int, x, packed, N: int, K: int, k: int, y=None, vals=None, idx=None,
                       ws: Workspace | None = None):
    """The lm_head (MODE_W4A16 on qpack_w4 bytes or MODE_W8A16 on qpack_w8 bytes) with the
    top-k of each row fused in: returns (y [M,N] fp16 logits, vals [M,k] fp16, idx [M,k] int32),
    y bit-identical to the plain GEMM and (vals, idx) equal to topk_logits(y, k)."""
    _need(x, torch.float16, "x", 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    y = _out(y, M, N, x.device)
    if vals is None:
        vals = torch.empty((M, k), dtype=torch.float16, device=x.device)
    if idx is None:
        idx = torch.empty((M, k), dtype=torch.int32, device=x.device)
    _need(vals, torch.float16, "vals", 2)
    _need(idx, torch.int32, "idx", 2)
    _need_shape(vals, (M, k), "vals")
    _need_shape(idx, (M, k), "idx")
    if M and N:
        _need_packed(packed, (qpack_w8_bytes if mode == MODE_W8A16 else qpack_w4_bytes)(N, K), x)
    if ws is None:
        key = (x.device, torch.cuda.current_stream(x.device).cuda_stream, "lm_head_topk")
        ws = _default_ws.setdefault(key, Workspace(x.device))
    with torch.cuda.device(x.device):
        need = int(lib().qgemm_lm_head_topk_workspace_bytes(mode, M, N, K, k))
        wbuf, wbytes = ws.get_bytes(need)
        _check(lib().qgemm_lm_head_topk(mode, _ptr(x), _ptr(packed), M, N, K, k, _ptr(y), _ptr(vals),
                                        _ptr(idx), _ptr(wbuf), wbytes, _stream(x)))
    return y, vals, idx


def topk_logits(logits, k: int):
    """Per row the k largest logits (largest first, ties to the smaller index):
    returns (values fp16 [M,k], indices int32 [M,k])."""
    _need(logits, torch.float16, "logits", 2)
    M, N = logits.shape
    vals = torch.empty((M, k), dtype=torch.float16, device=logits.device)
    idx = torch.empty((M, k), dtype=torch.int32, device=logits.device)
    need = int(lib().topk_workspace_bytes(M, N, k))
    key = (logits.device, torch.cuda.current_stream(logits.device).cuda_stream)
    buf = _topk_ws.get(key)
    if buf is None or buf.numel() < need:
        buf = torch.zeros(max(need, 256), dtype=torch.uint8, device=logits.device)
        _topk_ws[key] = buf
    with torch.cuda.device(logits.device):
        _check(lib().topk_logits(_ptr(logits), M, N, k, _ptr(vals), _ptr(idx), _ptr(buf), buf.numel(),
                                 _stream(logits)))
    return vals, idx


def qgemm_w4a16_noalloc(x, packed, N: int, K: int, y=None):
    """qgemm_w4a16 with the library's built-in scratch instead of a workspace (for
    callers that cannot allocate device memory; see include/qgemm.h)."""
    _need(x, torch.float16, "x", 2)
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError("x.shape[1] != K")
    y = _out(y, M, N, x.device)
    if M and N:
        _need_packed(packed, qpack_w4_bytes(N, K), x)
    with torch.cuda.device(x.device):
        _check(lib().qgemm_w4a16_noalloc(_ptr(x), _ptr(packed), M, N, K, _ptr(y), _stream(x)))
    return y


# -------------------------------------------------------------- diagnostics --
def device_error(stream=None) -> int:
    """Wait for the work enqueued on `stream` (default: the current stream of the current
    device), then return and clear the device error word of the current device."""
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(lib().qw_device_error(ctypes.c_void_p(stream.cuda_stream)))


QW_OPT_WEIGHTS_IMMUTABLE = 1


def set_weights_immutable(flag: bool = True):
    """Declare that packed weights are never written by the kernel that directly
    precedes a GEMM on its stream, letting each GEMM stream its weights while the
    preceding kernel finishes (see include/qgemm.h)."""
    _check(lib().qw_set_option(QW_OPT_WEIGHTS_IMMUTABLE, 1 if flag else 0))


QW_OPT_WAIT_LIMIT_US = 2
DEFAULT_WAIT_LIMIT_US = 4_000_000


def set_wait_limit_us(us: int | None = None):
    """Test hook: the time limit of every wait inside the GEMM kernels launched from now
    on, in microseconds (None restores the 4 s default).  A kernel whose wait runs past
    it ends early with QW_ERR_TIMEOUT in the device error word."""
    _check(lib().qw_set_option(QW_OPT_WAIT_LIMIT_US, DEFAULT_WAIT_LIMIT_US if us is None else int(us)))


def num_kernel_launches() -> int:
    return int(lib().qw_num_kernel_launches())


# ----------------------------------------------------- measurement tools --
MMA_KINDS = {"f16": 0, "s8": 1, "e4m3": 2, "s4": 3}


def diag_mma_peak(kind: str, ctas: int, iters: int, chains: int = 8, device=None):
    """Launch the mma.sync rate (chains=8) or latency (chains=1) microbenchmark on the
    current stream; returns (ops of the launch, sink tensor).  The caller times it."""
    dev = torch.device(device or "cuda")
    sink = torch.empty(ctas * 256, dtype=torch.float32, device=dev)
    ops = ctypes.c_double(0.0)
    with torch.cuda.device(dev):
        _check(lib().qw_diag_mma_peak(MMA_KINDS[kind], ctas, iters, chains, _ptr(sink), ctypes.byref(ops),
                                      _stream(sink)))
    return ops.value, sink


def diag_tc_probe(kind: int, a_tmem: bool, n: int, issuers: int, chunks: int, window: int, grid: int,
                  device=None):
    """tcgen05.mma timing probe; returns the device tensor [grid, 4, 4] (issue ns, wait ns,
    total ns, chunks) -- read it after synchronizing."""
    dev = torch.device(device or "cuda")
    out = torch.zeros((grid, 4, 4), dtype=torch.int64, device=dev)
    with torch.cuda.device(dev):
        _check(lib().qw_diag_tc_probe(kind, 1 if a_tmem else 0, n, issuers, chunks, window, _ptr(out), grid,
                                      _stream(out)))
    return out


def diag_f8f6f4_gemm(a_e4m3, b_e4m3, a_tmem: bool):
    """d [128, 16] fp32 = a [128, K] . b [16, K]^T on tcgen05 kind::f8f6f4 (e4m3 bytes as uint8)."""
    _need(a_e4m3, torch.uint8, "a", 2)
    _need(b_e4m3, torch.uint8, "b", 2)
    K = a_e4m3.shape[1]
    if tuple(a_e4m3.shape) != (128, K) or tuple(b_e4m3.shape) != (16, K):
        raise ValueError("a must be [128, K] and b [16, K]")
    d = torch.empty((128, 16), dtype=torch.float32, device=a_e4m3.device)
    with torch.cuda.device(a_e4m3.device):
        _check(lib().qw_diag_f8f6f4_gemm(_ptr(a_e4m3), _ptr(b_e4m3), K, 1 if a_tmem else 0, _ptr(d),
                                         _stream(a_e4m3)))
    return d


def plan(mode: int, M: int, N: int, K: int, num_sms: int) -> Plan:
    p = Plan()
    _check(lib().qw_plan(mode, M, N, K, num_sms, ctypes.byref(p)))
    return p


def plan_segments(p: Plan, cta: int):
    n = lib().qw_plan_segments(ctypes.byref(p), cta, 0, None, None, None, None)
    if n < 0:
        _check(n)
    tile = (ctypes.c_longlong * max(n, 1))()
    g0 = (ctypes.c_int * max(n, 1))()
    g1 = (ctypes.c_int * max(n, 1))()
    slot = (ctypes.c_int * max(n, 1))()
    lib().qw_plan_segments(ctypes.byref(p), cta, n, tile, g0, g1, slot)
    return [(tile[i], g0[i], g1[i], slot[i]) for i in range(n)]


def plan_row_blocks(p: Plan, cta: int):
    """Under a row-block plan: the 16-row blocks (begin, end) CTA `cta` computes."""
    b, e = ctypes.c_int(), ctypes.c_int()
    _check(lib().qw_plan_row_blocks(ctypes.byref(p), cta, ctypes.byref(b), ctypes.byref(e)))
    return b.value, e.value
