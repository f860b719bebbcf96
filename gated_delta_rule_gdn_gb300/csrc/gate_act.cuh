// In-kernel activation of the gate and of beta from raw logits ("Gated Delta Network (GDN)", §3.1 eq. 5: the
// Mamba2-style parameterisation log alpha = -exp(A_log) softplus(x + dt_bias); beta = sigmoid(x); §4 and §6 describe
// fusing both into the chunk kernel so no separate activation pass runs).
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace gdn {

// softplus(x) = log(1 + e^x), without overflow for large x
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }

// log alpha of head h from the raw gate logit (identity when no activation is requested)
__device__ __forceinline__ float act_gate(const GateAct& a, float raw, int h) {
    if (!a.A_log) return raw;
    const float dt = a.dt_bias ? a.dt_bias[h] : 0.f;
    return -expf(a.A_log[h]) * softplus_f(raw + dt);
}

__device__ __forceinline__ float act_beta(const GateAct& a, float raw) {
    return a.beta_sigmoid ? 1.f / (1.f + expf(-raw)) : raw;
}

}  // namespace gdn
