"""CPU oracle for int8-QK prefill attention -- TEST INFRASTRUCTURE ONLY (plain numpy).

Follows "What this repo does that stock vLLM doesn't" (qwen38-27b-rtx3090
docs/optimizations.md), paragraph "int8-QK prefill attention": QK^T runs on int8
codes, SageAttention-style -- K is smoothed by its per-head channel mean (which
leaves the softmax unchanged, so the result is exact up to the int8 rounding), K
is quantized once per layer chunk, Q rows carry per-row scales, and P.V stays in
16-bit floating point.  The page states the accuracy as cos > 0.99999 against an
fp32 attention at 4k-51k context.

The steps, in the page's order, with the readings the page leaves open:

1. Smoothing.  For every KV head and channel, the mean of K over the S keys of the
   context: the sum of the fp16 values is exact in binary64 (they are multiples of
   2^-24 below 2^16, so any S < 2^13 sums exactly), divided by S in binary64 and
   rounded to binary32.  K' = fp32(k - mean), one rounding.
2. Quantization.  Per row (one key of one head for K', one query of one head for
   Q): s = fp32(amax / 127) with an IEEE divide, code = round-half-to-even of
   fp32(x / s), an all-zero row giving s = 0 and zero codes -- the arithmetic of
   the library's activation quantizer, applied to K' and to Q.
3. Scores.  S_ij = (sum_c qcode_ic * kcode_jc) * s_q_i * s_k_j / sqrt(d), binary64;
   the integer dot product is exact in binary64 (|terms| <= 127^2, d <= 2^12).
4. Causal prefill.  The T queries are the last T positions of the S-token context:
   query i sits at position S - T + i and sees keys 0 .. S - T + i.
5. Softmax and P.V in binary64 (V exact), one final rounding to fp16.

Grouped heads: query head h reads KV head h // (Hq / Hkv).
"""
from __future__ import annotations

import numpy as np


def quant_rows_f32(x):
    """Per-row symmetric int8 quantization of a binary32 array [..., d]:
    (codes int8 [..., d], scales float32 [...]) as in step 2."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    q = np.rint((x / safe[..., None]).astype(np.float32))
    q = np.where(s[..., None] == 0, 0.0, q)
    return q.astype(np.int8), s


def smooth_k(k):
    """Step 1: k [S, Hkv, d] fp16 -> K' [S, Hkv, d] float32 (k minus its channel mean)."""
    k = np.asarray(k, dtype=np.float16)
    S = k.shape[0]
    total = k.astype(np.float64).sum(axis=0)          # exact (see step 1)
    mean = (total / np.float64(S)).astype(np.float32)
    return (k.astype(np.float32) - mean[None]).astype(np.float32)


def attn_int8qk(q, k, v, out_f64: bool = False):
    """int8-QK causal prefill attention.

    q [T, Hq, d] fp16 -- the chunk's queries (positions S - T .. S - 1)
    k, v [S, Hkv, d] fp16 -- keys and values of positions 0 .. S - 1
    returns o [T, Hq, d]: fp16, or binary64 before the final rounding when out_f64.
    """
    q = np.asarray(q, dtype=np.float16)
    k = np.asarray(k, dtype=np.float16)
    v = np.asarray(v, dtype=np.float16)
    T, Hq, d = q.shape
    S, Hkv, dk = k.shape
    if dk != d or v.shape != k.shape or T > S or T < 1 or Hkv < 1 or Hq % Hkv:
        raise ValueError("shapes: q [T,Hq,d], k and v [S,Hkv,d], 1 <= T <= S, Hkv | Hq")
    kq, ks = quant_rows_f32(smooth_k(k))                 # [S, Hkv, d], [S, Hkv]
    qq, qs = quant_rows_f32(q.astype(np.float32))      # [T, Hq, d], [T, Hq]
    group = Hq // Hkv
    pos = np.arange(T)[:, None] + (S - T)               # absolute query positions
    visible = np.arange(S)[None, :] <= pos              # [T, S]
    out = np.zeros((T, Hq, d), np.float64)
    inv_sqrt_d = 1.0 / np.sqrt(np.float64(d))
    for h in range(Hq):
        g = h // group
        dots = qq[:, h, :].astype(np.float64) @ kq[:, g, :].astype(np.float64).T   # exact
        scores = dots * qs[:, h].astype(np.float64)[:, None] * ks[:, g].astype(np.float64)[None, :]
        scores = scores * inv_sqrt_d
        scores = np.where(visible, scores, -np.inf)
        scores = scores - scores.max(axis=1, keepdims=True)
        p = np.exp(scores)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :].astype(np.float64)
    return out if out_f64 else out.astype(np.float16)
