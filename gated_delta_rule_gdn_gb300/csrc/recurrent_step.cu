// Decode step of the gated delta rule: one token for each of N independent sequences.
//
// "Gated Delta Network (GDN)", eq. 12 and §4.4: decode runs the recurrent form, one token at a
// time.  The fused recurrent kernel on "You Could Have Come Up With Kimi Delta Attention" gives
// the order of the steps: decay, predict, residual, rank-1 write, read, with the retention a
// per-key-channel vector for KDA.  In the transposed state h = S^T (d_k x d_v), with a_c = exp(g_c)
// (one value for every row c under the scalar gate):
//     p = h^T (a * k),   z = h^T (a * q),   r = beta (v - p),
//     o = scale (z + r (k . q)),   h <- diag(a) h + k r^T.
// This is the same update: h' = diag(a) h + k r^T, and o = scale h'^T q expands to the line above.
// So one read of h gives both reductions, and one write stores h'.  The step moves
// 2 * d_k * d_v * 4 bytes of state per (sequence, head), so it is bound by HBM bandwidth.
//
// Fast path (d_k = d_v = 128): one CTA of 256 threads per (sequence, head).  Warp w owns state
// rows [16w, 16w + 16); lane l owns columns [4l, 4l + 4).  Each thread keeps its 16 x 4 fp32
// slice in registers between the read and the write, so every access is a coalesced 16-byte
// vector.  Generic path: one thread per column; the state is read twice and written once.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "gate_act.cuh"

namespace gdn {
namespace {

template <typename T> __device__ __forceinline__ float ld_f32(const T* p);
template <> __device__ __forceinline__ float ld_f32<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void st_f32(T* p, float x);
template <> __device__ __forceinline__ void st_f32<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void st_f32<__nv_bfloat16>(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
}

constexpr int kD = 128;
constexpr int kRowsPerWarp = 16;

template <typename Tin, typename Tout, bool PERCH>
__global__ void __launch_bounds__(256, 2)
step_d128_kernel(const StepArgs a) {
    __shared__ float ks[kD], qs[kD], vs[kD], rs[kD], as[kD];
    __shared__ float red[2][8][kD];
    __shared__ float kq_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t nh = blockIdx.x;
    const int Hk = a.Hk > 0 ? a.Hk : a.H;   // grouped values: key head h / (H / Hk) serves value head h
    const size_t nk = (nh / a.H) * Hk + (nh % a.H) / (a.H / Hk);
    const Tin* q = static_cast<const Tin*>(a.q) + nk * kD;
    const Tin* k = static_cast<const Tin*>(a.k) + nk * kD;
    const Tin* v = static_cast<const Tin*>(a.v) + nh * kD;
    float* __restrict__ h = a.state + nh * (size_t)kD * kD;

    // issue the state loads first: they are the long pole
    float4 hr[kRowsPerWarp];
    const int row0 = warp * kRowsPerWarp;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
        hr[r] = __ldcs(reinterpret_cast<const float4*>(h + (size_t)(row0 + r) * kD) + lane);

    if (tid < kD) {
        ks[tid] = ld_f32<Tin>(k + tid);
        qs[tid] = ld_f32<Tin>(q + tid);
        vs[tid] = ld_f32<Tin>(v + tid);
        as[tid] = expf(PERCH ? a.g[nh * kD + tid] : act_gate(a.act, a.g[nh], (int)(nh % a.H)));
    }
    const float beta = act_beta(a.act, a.beta[nh]);
    __syncthreads();
    if (warp == 0) {
        float s = 0.f;
        for (int i = lane; i < kD; i += 32) s = fmaf(ks[i], qs[i], s);
        for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
        if (lane == 0) kq_s = s;
    }
    float4 p = make_float4(0.f, 0.f, 0.f, 0.f), z = p;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const float ar = as[row0 + r], kr = ar * ks[row0 + r], qr = ar * qs[row0 + r];
        p.x = fmaf(hr[r].x, kr, p.x); p.y = fmaf(hr[r].y, kr, p.y);
        p.z = fmaf(hr[r].z, kr, p.z); p.w = fmaf(hr[r].w, kr, p.w);
        z.x = fmaf(hr[r].x, qr, z.x); z.y = fmaf(hr[r].y, qr, z.y);
        z.z = fmaf(hr[r].z, qr, z.z); z.w = fmaf(hr[r].w, qr, z.w);
    }
    reinterpret_cast<float4*>(red[0][warp])[lane] = p;
    reinterpret_cast<float4*>(red[1][warp])[lane] = z;
    __syncthreads();
    if (tid < kD) {
        float P = 0.f, Z = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) { P += red[0][w][tid]; Z += red[1][w][tid]; }
        const float r = beta * (vs[tid] - P);
        rs[tid] = r;
        st_f32<Tout>(static_cast<Tout*>(a.o) + nh * kD + tid, a.scale * fmaf(r, kq_s, Z));
    }
    __syncthreads();
    const float4 r4 = reinterpret_cast<const float4*>(rs)[lane];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const float kr = ks[row0 + r], alpha = as[row0 + r];
        float4 x;
        x.x = fmaf(alpha, hr[r].x, kr * r4.x);
        x.y = fmaf(alpha, hr[r].y, kr * r4.y);
        x.z = fmaf(alpha, hr[r].z, kr * r4.z);
        x.w = fmaf(alpha, hr[r].w, kr * r4.w);
        __stcs(reinterpret_cast<float4*>(h + (size_t)(row0 + r) * kD) + lane, x);
    }
}

template <typename Tin, typename Tout, bool PERCH>
__global__ void __launch_bounds__(128)
step_generic_kernel(const StepArgs a) {
    extern __shared__ float sh[];
    float* ks = sh;
    float* qs = ks + a.dk;
    float* as = qs + a.dk;
    __shared__ float kq_s;
    const int tid = threadIdx.x;
    const size_t nh = blockIdx.x;
    const int dk = a.dk, dv = a.dv;
    const int Hk = a.Hk > 0 ? a.Hk : a.H;
    const size_t nk = (nh / a.H) * Hk + (nh % a.H) / (a.H / Hk);
    const Tin* q = static_cast<const Tin*>(a.q) + nk * dk;
    const Tin* k = static_cast<const Tin*>(a.k) + nk * dk;
    const Tin* v = static_cast<const Tin*>(a.v) + nh * dv;
    float* h = a.state + nh * (size_t)dk * dv;
    for (int i = tid; i < dk; i += blockDim.x) {
        ks[i] = ld_f32<Tin>(k + i);
        qs[i] = ld_f32<Tin>(q + i);
        as[i] = expf(PERCH ? a.g[nh * dk + i] : act_gate(a.act, a.g[nh], (int)(nh % a.H)));
    }
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int i = 0; i < dk; ++i) s = fmaf(ks[i], qs[i], s);
        kq_s = s;
    }
    __syncthreads();
    const float beta = act_beta(a.act, a.beta[nh]);
    for (int j = tid; j < dv; j += blockDim.x) {
        float P = 0.f, Z = 0.f;
        for (int i = 0; i < dk; ++i) {
            const float x = as[i] * h[(size_t)i * dv + j];
            P = fmaf(x, ks[i], P);
            Z = fmaf(x, qs[i], Z);
        }
        const float r = beta * (ld_f32<Tin>(v + j) - P);
        st_f32<Tout>(static_cast<Tout*>(a.o) + nh * dv + j, a.scale * fmaf(r, kq_s, Z));
        for (int i = 0; i < dk; ++i) {
            float* p = h + (size_t)i * dv + j;
            *p = fmaf(as[i], *p, ks[i] * r);
        }
    }
}

template <typename Tin, typename Tout>
void launch_typed(const StepArgs& a, cudaStream_t s, unsigned blocks, bool fast) {
    const size_t sh = 3 * (size_t)a.dk * sizeof(float);
    if (a.per_channel) {
        if (fast) step_d128_kernel<Tin, Tout, true><<<blocks, 256, 0, s>>>(a);
        else step_generic_kernel<Tin, Tout, true><<<blocks, 128, sh, s>>>(a);
    } else {
        if (fast) step_d128_kernel<Tin, Tout, false><<<blocks, 256, 0, s>>>(a);
        else step_generic_kernel<Tin, Tout, false><<<blocks, 128, sh, s>>>(a);
    }
}

}  // namespace

cudaError_t launch_recurrent_step(const StepArgs& a, cudaStream_t s) {
    const long blocks = (long)a.N * a.H;
    if (blocks == 0) return cudaSuccess;
    const bool fast = a.dk == kD && a.dv == kD && (reinterpret_cast<uintptr_t>(a.state) % 16 == 0);
    if (a.bf16) {
        if (a.o_f32) launch_typed<__nv_bfloat16, float>(a, s, (unsigned)blocks, fast);
        else launch_typed<__nv_bfloat16, __nv_bfloat16>(a, s, (unsigned)blocks, fast);
    } else {
        if (a.o_f32) launch_typed<float, float>(a, s, (unsigned)blocks, fast);
        else launch_typed<float, __nv_bfloat16>(a, s, (unsigned)blocks, fast);
    }
    return cudaGetLastError();
}

}  // namespace gdn
