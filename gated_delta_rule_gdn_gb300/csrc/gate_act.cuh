// In-kernel activation of the gate and of beta from raw logits ("Gated Delta Network (GDN)", §3.1 eq. 5: the
// Mamba2-style parameterisation log alpha = -exp(A_log) softplus(x + dt_bias); beta = sigmoid(x), or 2 sigmoid(x) with negative eigenvalues allowed; §4 and §6 describe
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

// beta from its logit: sigmoid, or 2 sigmoid (beta in (0, 2), so the transition I - beta k k^T of a unit key can
// have the eigenvalue 1 - beta < 0; "Gated Delta Network (GDN)", §5 implementation notes)
__device__ __forceinline__ float act_beta(const GateAct& a, float raw) {
    return a.beta_sigmoid ? (float)a.beta_sigmoid / (1.f + expf(-raw)) : raw;
}

}  // namespace gdn
