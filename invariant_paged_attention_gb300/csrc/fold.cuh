// The fixed-order log-sum-exp fold of attention states, shared by every merge
// kernel so that all merge routes produce the same bits.
#pragma once

#include "ptx.cuh"

namespace bia {

// Folds state (lse_s, v) into the running state (L, o), left to right.
// A state with lse_s == -inf is skipped; the first finite state is taken as
// is.  Otherwise: M = max(L, lse_s), a = 2^((L-M)log2e), b = 2^((lse_s-M)log2e),
// the weights wa = a/(a+b) and wb = b/(a+b) (two divisions per state, not one
// per element), o = wa*o + wb*v, L = M + ln(a+b).  Explicit _rn intrinsics keep
// the compiler from contracting differently in different kernels.
template <int V>
__device__ __forceinline__ void fold_state(float &L, float (&o)[V], float lse_s,
                                           const float (&v)[V]) {
  if (lse_s == -INFINITY) return;
  if (L == -INFINITY) {
    L = lse_s;
#pragma unroll
    for (int i = 0; i < V; ++i) o[i] = v[i];
    return;
  }
  const float M = fmaxf(L, lse_s);
  const float a = ex2(__fmul_rn(__fsub_rn(L, M), kLog2e));
  const float b = ex2(__fmul_rn(__fsub_rn(lse_s, M), kLog2e));
  const float sum = __fadd_rn(a, b);
  const float wa = __fdiv_rn(a, sum), wb = __fdiv_rn(b, sum);
#pragma unroll
  for (int i = 0; i < V; ++i) o[i] = __fadd_rn(__fmul_rn(wa, o[i]), __fmul_rn(wb, v[i]));
  L = __fadd_rn(M, __fmul_rn(lg2(sum), kLn2));
}

} // namespace bia
