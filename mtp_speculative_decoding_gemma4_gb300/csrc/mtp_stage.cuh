// The staged operand of the tensor-core GEMMs: every fp32 activation value as three bf16
// terms whose sum is the value exactly, in a buffer [3][bp][K] (term, sequence, column).
#pragma once

#include <cuda_bf16.h>
#include <stddef.h>

namespace mtp {

// Writes v as its three bf16 terms (hi + mid + lo = v exactly) at (b, k).
__device__ __forceinline__ void stage_terms(__nv_bfloat16* xs, int bp, int K, int b, int k, float v) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  const size_t row = static_cast<size_t>(b) * K + k, term = static_cast<size_t>(bp) * K;
  xs[row] = hi;
  xs[term + row] = mid;
  xs[2 * term + row] = lo;
}

}  // namespace mtp
