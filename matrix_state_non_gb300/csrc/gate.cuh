// The forget gate of one (b, t, n): either the caller's f, or computed from
// its pre-activation a with the per-head parameters of section 2.2 of the
// reading notes on "M2RNN: Non-Linear RNNs with Matrix-Valued States for
// Scalable Language Modeling" (the paper's Eq. 13 and 17):
//     f = (1 + exp(a + beta))^(-alpha) = exp(-alpha * softplus(a + beta)).
#pragma once

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace m2rnn {

struct GateSrc {
  const void* f;       // [B,T,N] in the input dtype (used when a == null)
  const void* a;       // gate pre-activation [B,T,N] in the input dtype, or null
  const float* alpha;  // [N], >= 0
  const float* beta;   // [N]
  bool bf16;
};

__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }

// idx = (b * T + t) * N + n.
__device__ __forceinline__ float gate_value(const GateSrc& s, int64_t idx, int n) {
  if (s.a != nullptr) {
    const float x = (s.bf16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(s.a)[idx])
                            : static_cast<const float*>(s.a)[idx]) + s.beta[n];
    return expf(-s.alpha[n] * softplus_f(x));
  }
  return s.bf16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(s.f)[idx]) : static_cast<const float*>(s.f)[idx];
}

}  // namespace m2rnn
