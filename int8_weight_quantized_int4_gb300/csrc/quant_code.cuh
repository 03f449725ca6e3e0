// quant_code.cuh -- the int8 code of one activation value under a per-token scale
// ("In full" item 4 of "What this repo does that stock vLLM doesn't": activations
// quantized to int8 per token), shared by the standalone quantizer and the row-block
// kernel's in-kernel one so that both give the same codes.
#pragma once
#include <cuda_runtime.h>

namespace qw {

// q = clamp(rne(x / s), -127, 127) with x / s the IEEE binary32 quotient (the definition of
// the per-token code, s = amax / 127), without a divide per value: t = x * (1/s) (correctly rounded
// reciprocal and product) is within 3 * 2^-24 * |x/s| <= 2.3e-5 of the quotient, since
// |x/s| <= 127 (1 + 2^-24).  So rne(t) = rne(x / s) unless t lies within 2^-14 of a
// half-integer, i.e. unless |t - rne(t)| >= 0.5 - 2^-14 (t - rne(t) is exact); only those
// values take the IEEE divide, out of line so that it is skipped rather than computed and
// discarded.  s = 0 (an all-zero row) has 1/s = 0, so t = 0 and q = 0.
__device__ __forceinline__ int quant_code_div(float x, float s) {
  return max(-127, min(127, __float2int_rn(__fdiv_rn(x, s))));
}
static __device__ __noinline__ int quant_code_exact(float x, float s) { return quant_code_div(x, s); }
// the reciprocal code, and whether t came within 2^-14 of a half-integer (then the code
// must come from the divide)
__device__ __forceinline__ int quant_code_fast(float x, float rs, bool &near_tie) {
  const float t = __fmul_rn(x, rs);
  const int q = __float2int_rn(t);
  near_tie = fabsf(t - (float)q) >= 0.5f - 6.103515625e-05f;
  return max(-127, min(127, q));
}
__device__ __forceinline__ int quant_code(float x, float s, float rs) {
  bool near_tie;
  const int q = quant_code_fast(x, rs, near_tie);
  return near_tie ? quant_code_exact(x, s) : q;
}

}  // namespace qw
