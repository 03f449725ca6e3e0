"""Seeded synthetic inputs for the weight-quantized linear layer.

This module only draws random numbers: it holds none of the method's arithmetic
(no quantization, no packing, no products).  Both the CPU oracle and the CUDA
path consume the tensors it returns, so that parity compares like with like.

The distributions follow the five workloads of the layer (int4 codes uniform in
[-8, 7], group-128 fp16 scales with |s| ~ U(lo, hi) and a random sign so that
about half are negative -- "What this repo does that stock vLLM doesn't",
"In full" item 4 -- fp16 activations ~ N(0, 1), optionally with 1 % outlier
channels scaled by 20, and int8 codes in [-127, 127] for the int8 group-128
lm_head, "In full" items 1 and 5).  Everything is generated on the CPU with a
seeded ``torch.Generator``.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

GROUP = 128


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def codes_int4(N: int, K: int, gen: torch.Generator, lo: int = -8, hi: int = 7) -> torch.Tensor:
    """Signed int4 codes, uniform in [lo, hi], as int8 [N, K]."""
    return torch.randint(lo, hi + 1, (N, K), generator=gen, dtype=torch.int8)


def codes_int8(N: int, K: int, gen: torch.Generator, lo: int = -127, hi: int = 127) -> torch.Tensor:
    """int8 codes, uniform in [lo, hi], as int8 [N, K]."""
    return torch.randint(lo, hi + 1, (N, K), generator=gen, dtype=torch.int8)


def signed_scales(N: int, G: int, gen: torch.Generator, lo: float, hi: float,
                  p_negative: float = 0.5) -> torch.Tensor:
    """fp16 [N, G] group scales: |s| ~ U(lo, hi), negative with probability p_negative."""
    mag = lo + (hi - lo) * torch.rand((N, G), generator=gen, dtype=torch.float32)
    neg = torch.rand((N, G), generator=gen, dtype=torch.float32) < p_negative
    return torch.where(neg, -mag, mag).to(torch.float16)


def activations(M: int, K: int, gen: torch.Generator, outlier_frac: float = 0.0,
                outlier_mult: float = 20.0) -> torch.Tensor:
    """fp16 [M, K] ~ N(0, 1); a fraction of channels (columns) scaled by outlier_mult."""
    x = torch.randn((M, K), generator=gen, dtype=torch.float32)
    n_out = int(round(outlier_frac * K))
    if n_out > 0:
        cols = torch.randperm(K, generator=gen)[:n_out]
        x[:, cols] *= outlier_mult
    return x.to(torch.float16)


def int8_exact_activations(M: int, K: int, gen: torch.Generator, exp_lo: int = 2,
                           exp_hi: int = 9) -> torch.Tensor:
    """fp16 [M, K] of the form c * 2**-e_m with integer c in [-127, 127] and one |c| == 127
    per row (so a symmetric per-token int8 quantizer reproduces c and 2**-e_m exactly)."""
    c = torch.randint(-127, 128, (M, K), generator=gen, dtype=torch.int32)
    pos = torch.randint(0, K, (M,), generator=gen)
    sign = torch.where(torch.rand((M,), generator=gen) < 0.5, -1, 1).to(torch.int32)
    c[torch.arange(M), pos] = 127 * sign
    e = torch.randint(exp_lo, exp_hi + 1, (M, 1), generator=gen).to(torch.float32)
    return (c.to(torch.float32) * torch.exp2(-e)).to(torch.float16)


@dataclass
class Problem:
    """One seeded problem: logical weights (codes, scales) and activations."""
    M: int
    N: int
    K: int
    codes: torch.Tensor      # int8 [N, K]
    scales: torch.Tensor     # fp16 [N, K/128]
    x: torch.Tensor          # fp16 [M, K]
    bits: int                # 4 or 8


def make_problem(M: int, N: int, K: int, seed: int, bits: int = 4, scale_lo: float = 0.002,
                 scale_hi: float = 0.02, outlier_frac: float = 0.0,
                 code_range: tuple | None = None) -> Problem:
    gen = generator(seed)
    G = K // GROUP
    if bits == 4:
        lo, hi = code_range or (-8, 7)
        codes = codes_int4(N, K, gen, lo, hi)
    else:
        lo, hi = code_range or (-127, 127)
        codes = codes_int8(N, K, gen, lo, hi)
    scales = signed_scales(N, G, gen, scale_lo, scale_hi)
    x = activations(M, K, gen, outlier_frac)
    return Problem(M, N, K, codes, scales, x, bits)


# The five workloads (shapes, value distributions and seeds).
def tiny_w4a16() -> Problem:
    """M=4, K=256, N=512 W4A16 oracle check, seed 0."""
    return make_problem(4, 512, 256, seed=0)


def projection(M: int, seed: int = 1) -> Problem:
    """Decode/verify projection K=N=5120, 1 % outlier channels x20, seed 1."""
    return make_problem(M, 5120, 5120, seed=seed, outlier_frac=0.01)


def ffn_up(M: int = 64) -> Problem:
    """Fused gate+up projection K=5120 -> N=34816, seed 2."""
    return make_problem(M, 34816, 5120, seed=2)


def ffn_down(M: int = 64) -> Problem:
    """Down projection K=17408 -> N=5120, seed 3."""
    return make_problem(M, 5120, 17408, seed=3)


def prefill(M: int = 8192) -> Problem:
    """Compute-bound prefill M=8192, K=5120, N=34816, seed 4."""
    return make_problem(M, 34816, 5120, seed=4)


def lm_head(M: int, N: int = 248320) -> Problem:
    """int8 group-128 lm_head N=248320, K=5120, |s| ~ U(0.001, 0.01) signed, seed 5."""
    return make_problem(M, N, 5120, seed=5, bits=8, scale_lo=0.001, scale_hi=0.01)


def lm_head_int4(M: int, N: int = 248320) -> Problem:
    """int4 group-128 lm_head (a symmetric GPTQ export's codes minus 8) N=248320, K=5120, seed 6."""
    return make_problem(M, N, 5120, seed=6, bits=4)


def logits(M: int, N: int, seed: int, step: float = 0.125) -> torch.Tensor:
    """fp16 [M, N] logits ~ 4 N(0, 1) on a grid of `step` (so equal values are common),
    with a few exact +0 / -0 entries per row."""
    gen = generator(seed)
    z = torch.round(4.0 * torch.randn((M, N), generator=gen) / step) * step
    pos = torch.randint(0, N, (M, 4), generator=gen)
    z.scatter_(1, pos[:, :2], 0.0)
    z.scatter_(1, pos[:, 2:], -0.0)
    return z.to(torch.float16)


def token_ids(T: int, V: int, seed: int) -> torch.Tensor:
    """int32 [T] row ids in [0, V), with the first and last rows and repeats present."""
    gen = generator(seed)
    ids = torch.randint(0, V, (T,), generator=gen, dtype=torch.int32)
    if T >= 3:
        ids[0], ids[1], ids[2] = 0, V - 1, ids[T - 1]
    return ids


def attention(T: int, S: int, Hq: int, Hkv: int, d: int = 256, seed: int = 60,
              k_offset_std: float = 4.0):
    """Prefill attention inputs: q [T, Hq, d], k and v [S, Hkv, d] fp16.  q, v ~ N(0, 1);
    k ~ N(0, 1) plus a per-(head, channel) offset ~ N(0, k_offset_std) shared by all keys
    (the channel bias that mean-smoothing removes, "int8-QK prefill attention")."""
    gen = generator(seed)
    q = torch.randn((T, Hq, d), generator=gen, dtype=torch.float32)
    off = k_offset_std * torch.randn((1, Hkv, d), generator=gen, dtype=torch.float32)
    k = torch.randn((S, Hkv, d), generator=gen, dtype=torch.float32) + off
    v = torch.randn((S, Hkv, d), generator=gen, dtype=torch.float32)
    return q.to(torch.float16), k.to(torch.float16), v.to(torch.float16)
