"""CPU oracle for the weight-quantized linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it; the two meet only on the seeded inputs from ``synth``.

What it computes (plain definitions, binary64 accumulation), following
"What this repo does that stock vLLM doesn't" (qwen38-27b-rtx3090
docs/optimizations.md), "In full" item 4 (int4 weights with signed group-128
scales, int8 per-token activations), item 1 (int8 group-128 requantization,
~0.6 % round trip) and item 5 (the 248k-row int8 lm_head):

* ``quant_act_int8(x)``   -- per-token symmetric int8 quantizer (binary32,
  IEEE divide, round-half-to-even, all-zero row -> scale 0, codes 0).
* ``w4a16(x, codes, scales)`` / ``w8a16(...)`` -- y = fp16(sum_g s*sum_k x*q).
* ``w4a8(qa, sx, codes, scales)`` -- y = fp16(sx * sum_g s * int64 sum_k qa*q).
* ``roundtrip_int8_g128(w)`` -- int8 group-128 requantizer and its relative
  Frobenius error.
* ``half_to_double`` / ``double_to_half`` -- binary16 conversions written from
  the format definition.
* ``attn_int8qk(q, k, v)`` (``oracle/attention.py``, numpy) -- int8-QK causal
  prefill attention, from the page's paragraph "int8-QK prefill attention": K
  smoothed by its per-head channel mean, per-row int8 Q and K, binary64 softmax
  and P.V.

Every function is pinned by ``tests/test_oracle_*.py`` against brute force in
exact rational arithmetic, closed forms and the invariants the pages imply.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .attention import attn_int8qk, quant_rows_f32, smooth_k  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_double_to_half.argtypes = [ctypes.c_double]
        lib.oracle_double_to_half.restype = ctypes.c_uint16
        lib.oracle_quant_act_int8.argtypes = [p, i64, i64, p, p]
        for name in ("oracle_w4a16", "oracle_w8a16"):
            getattr(lib, name).argtypes = [p, p, p, i64, i64, i64, p]
        lib.oracle_w4a8.argtypes = [p, p, p, p, i64, i64, i64, p]
        lib.oracle_roundtrip_int8_g128.argtypes = [p, i64, i64, p, p, ctypes.POINTER(ctypes.c_double)]
        lib.oracle_embed_w8.argtypes = [p, i64, p, p, i64, i64, p]
        lib.oracle_topk.argtypes = [p, i64, i64, i64, p, p]
        for name in ("oracle_quant_act_int8", "oracle_w4a16", "oracle_w8a16", "oracle_w4a8",
                     "oracle_roundtrip_int8_g128", "oracle_embed_w8", "oracle_topk"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _as(a, dtype) -> np.ndarray:
    """Contiguous numpy view/copy of ``a`` (numpy array or CPU torch tensor)."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().contiguous().numpy()
    return np.ascontiguousarray(a, dtype=dtype) if a.dtype != dtype else np.ascontiguousarray(a)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its input (code {rc})")


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits) & 0xFFFF)


def double_to_half(v: float) -> int:
    return int(_load().oracle_double_to_half(float(v)))


def _half_bits(x) -> np.ndarray:
    """binary16 bit patterns (uint16) from a float16 numpy array / torch tensor."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.float16:
            x = x.view(torch.int16)
        x = x.numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    return np.ascontiguousarray(x.astype(np.uint16, copy=False))


def quant_act_int8(x):
    """x: [M,K] float16 -> (q int8 [M,K], s float32 [M])."""
    xb = _half_bits(x)
    M, K = xb.shape
    q = np.zeros((M, K), np.int8)
    s = np.zeros((M,), np.float32)
    _check(_load().oracle_quant_act_int8(_ptr(xb), M, K, _ptr(q), _ptr(s)), "quant_act_int8")
    return q, s


def _gemm16(name, x, codes, scales):
    xb = _half_bits(x)
    c = _as(codes, np.int8)
    sb = _half_bits(scales)
    M, K = xb.shape
    N = c.shape[0]
    assert c.shape == (N, K) and sb.shape == (N, K // 128), (c.shape, sb.shape)
    y = np.zeros((M, N), np.uint16)
    _check(getattr(_load(), name)(_ptr(xb), _ptr(c), _ptr(sb), M, N, K, _ptr(y)), name)
    return y.view(np.float16)


def w4a16(x, codes, scales) -> np.ndarray:
    """y[M,N] float16 for x [M,K] f16, codes [N,K] in [-8,7], scales [N,K/128] f16."""
    return _gemm16("oracle_w4a16", x, codes, scales)


def w8a16(x, codes, scales) -> np.ndarray:
    """y[M,N] float16 for x [M,K] f16, codes [N,K] int8, scales [N,K/128] f16."""
    return _gemm16("oracle_w8a16", x, codes, scales)


def w4a8(qa, sx, codes, scales) -> np.ndarray:
    """y[M,N] float16 for qa [M,K] int8, sx [M] f32, codes [N,K] in [-8,7], scales f16."""
    a = _as(qa, np.int8)
    s = _as(sx, np.float32)
    c = _as(codes, np.int8)
    sb = _half_bits(scales)
    M, K = a.shape
    N = c.shape[0]
    assert s.shape == (M,) and c.shape == (N, K) and sb.shape == (N, K // 128)
    y = np.zeros((M, N), np.uint16)
    _check(_load().oracle_w4a8(_ptr(a), _ptr(s), _ptr(c), _ptr(sb), M, N, K, _ptr(y)), "w4a8")
    return y.view(np.float16)


def roundtrip_int8_g128(w):
    """w [N,K] float32 -> (codes int8 [N,K], scales f16 [N,K/128], relative Frobenius error)."""
    ww = _as(w, np.float32)
    N, K = ww.shape
    codes = np.zeros((N, K), np.int8)
    scales = np.zeros((N, K // 128), np.uint16)
    err = ctypes.c_double(0.0)
    _check(_load().oracle_roundtrip_int8_g128(_ptr(ww), N, K, _ptr(codes), _ptr(scales),
                                              ctypes.byref(err)), "roundtrip_int8_g128")
    return codes, scales.view(np.float16), float(err.value)


def embed_w8(ids, codes, scales):
    """Dequant-on-gather: out[t,k] = fp16(codes[ids[t],k] * scales[ids[t],k/128]).
    ids [T] integers in [0, V), codes [V,D] int8, scales [V,D/128] f16 -> out [T,D] f16."""
    i = _as(ids, np.int64)
    c = _as(codes, np.int8)
    sb = _half_bits(scales)
    V, D = c.shape
    assert sb.shape == (V, D // 128)
    out = np.zeros((i.shape[0], D), np.uint16)
    _check(_load().oracle_embed_w8(_ptr(i), i.shape[0], _ptr(c), _ptr(sb), V, D, _ptr(out)), "embed_w8")
    return out.view(np.float16)


def topk(logits, k: int):
    """Per row the k largest logits, largest first, ties to the smaller index.
    logits [M,N] f16 -> (values [M,k] f16, indices [M,k] int64)."""
    lb = _half_bits(logits)
    M, N = lb.shape
    vals = np.zeros((M, k), np.uint16)
    idx = np.zeros((M, k), np.int64)
    _check(_load().oracle_topk(_ptr(lb), M, N, k, _ptr(vals), _ptr(idx)), "topk")
    return vals.view(np.float16), idx
