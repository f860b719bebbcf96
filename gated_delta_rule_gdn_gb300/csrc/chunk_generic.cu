// Generic fp32 SIMT chunk kernel: gated delta rule (scalar gate) and KDA (per-key-channel gate).
//
// This is the plain chunkwise algorithm of "TileLang 实战：KDA 从零到一 -- Gated DeltaNet",
// §2.3 (paper eqs 11-12), extended to per-channel decays as on "You Could Have Come Up With Kimi
// Delta Attention" (chunkwise form).  Everything is fp32 in shared memory.  It serves:
//   * fp32 inputs (tensor-core TF32 cannot reach the 1e-4 tolerance fp32 inputs are held to);
//   * any 1 <= d_k, d_v <= 256 and chunk 16/32/64, within the shared memory of one CTA (fp32 tiles: d_k = 256
//     takes chunk 64 with the scalar gate, chunk 32 or less with the per-channel gate);
//   * the KDA path.
// It is the correctness-first shape of the fused kernel.
//
// One CTA owns one (sequence, head, d_v tile of BV = 32 columns) and walks the sequence's chunks in
// order, carrying its d_k x BV slice of the state S^T in shared memory.  Per chunk, with G the
// within-chunk cumulative log gate (per channel for KDA) and L the number of valid rows:
//   A[i][j] = beta_i sum_c k_ic k_jc exp(G_ic - G_jc)        j <  i   (strictly lower)
//   P[i][j] = scale sum_c q_ic k_jc exp(G_ic - G_jc)         j <= i   (read matrix)
//   R       = diag(beta) (V - (K * exp(G)) h)                          right-hand side
//   Delta   = (I + A)^{-1} R, by forward substitution on rows          (no T materialised)
//   O       = scale (Q * exp(G)) h + P Delta
//   h      <- diag(exp(G_L)) h + (K * exp(G_L - G))^T Delta
// For the scalar gate, exp(G_ic - G_jc) is one number per (i, j).  Exponents are differences,
// formed only where j <= i, so no factor exceeds 1 (TileLang page §4.1: mask before exp).
// Rows past a sequence's end are zero (beta = 0, g = 0), which leaves the state unchanged.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kBV = 32;  // d_v columns per CTA

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Shared-memory footprint in floats for (C, dk), per gate mode.
__host__ __device__ inline size_t generic_smem_floats(int C, int dk, bool per_channel) {
    const size_t gcols = per_channel ? (size_t)dk : 1;
    return (size_t)C * dk * 2          // Q, K
         + (size_t)C * kBV             // V tile
         + (size_t)C * gcols * 2       // G (later exp(G_L - G)), exp(G)
         + (size_t)C                   // beta
         + (size_t)C * (C + 1) * 2     // A, P (row stride C + 1)
         + (size_t)dk * kBV            // state tile
         + (size_t)C * kBV;            // R, then Delta
}

template <typename Tin, typename Tout, bool PERCH>
__global__ void __launch_bounds__(kThreads)
chunk_generic_kernel(const ChunkArgs a, int n_tiles) {
    extern __shared__ float smem[];
    const int C = a.C, dk = a.dk, dv = a.dv, H = a.H;
    const int gc = PERCH ? dk : 1;
    float* Qs = smem;
    float* Ks = Qs + C * dk;
    float* Vs = Ks + C * dk;
    float* Gs = Vs + C * kBV;        // cumulative log gate; later exp(G_L - G)
    float* Es = Gs + C * gc;         // exp(G)
    float* Bs = Es + C * gc;
    float* Am = Bs + C;
    float* Pm = Am + C * (C + 1);
    float* Hs = Pm + C * (C + 1);
    float* Ds = Hs + dk * kBV;

    const int tid = threadIdx.x;
    const long chain = blockIdx.x / n_tiles;
    const int tile = blockIdx.x % n_tiles;
    const long n = chain / H;
    const int hh = (int)(chain % H);
    long b, bos, len;
    if (a.cu) {
        long s0 = a.cu[n], s1 = a.cu[n + 1];
        s0 = s0 < 0 ? 0 : (s0 > a.T ? a.T : s0);
        s1 = s1 < s0 ? s0 : (s1 > a.T ? a.T : s1);
        b = 0; bos = s0; len = s1 - s0;
    } else {
        b = n; bos = 0; len = a.T;
    }
    const int j0 = tile * kBV;
    const int bw = min(kBV, dv - j0);

    const Tin* __restrict__ q = static_cast<const Tin*>(a.q);
    const Tin* __restrict__ k = static_cast<const Tin*>(a.k);
    const Tin* __restrict__ v = static_cast<const Tin*>(a.v);
    Tout* __restrict__ o = static_cast<Tout*>(a.o);
    const size_t sbase = ((size_t)n * H + hh) * (size_t)dk * dv;

    for (int idx = tid; idx < dk * kBV; idx += kThreads) {
        const int c = idx / kBV, j = idx % kBV;
        Hs[idx] = (a.h0 && j < bw) ? a.h0[sbase + (size_t)c * dv + j0 + j] : 0.f;
    }

    for (long cs = 0; cs < len; cs += C) {
        const int L = (int)min((long)C, len - cs);
        __syncthreads();  // previous chunk done with every buffer
        for (int idx = tid; idx < C * dk; idx += kThreads) {
            const int r = idx / dk, c = idx % dk;
            float qv = 0.f, kv = 0.f;
            if (r < L) {
                const size_t off = (((size_t)b * a.T + bos + cs + r) * H + hh) * dk + c;
                qv = to_f32<Tin>(q[off]);
                kv = to_f32<Tin>(k[off]);
            }
            Qs[idx] = qv;
            Ks[idx] = kv;
        }
        for (int idx = tid; idx < C * kBV; idx += kThreads) {
            const int r = idx / kBV, j = idx % kBV;
            float vv = 0.f;
            if (r < L && j < bw) vv = to_f32<Tin>(v[(((size_t)b * a.T + bos + cs + r) * H + hh) * dv + j0 + j]);
            Vs[idx] = vv;
        }
        for (int idx = tid; idx < C * gc; idx += kThreads) {
            const int r = idx / gc, c = idx % gc;
            const size_t tok = ((size_t)b * a.T + bos + cs + r) * H + hh;
            Gs[idx] = (r < L) ? a.g[PERCH ? tok * dk + c : tok] : 0.f;
        }
        for (int r = tid; r < C; r += kThreads) {
            Bs[r] = (r < L) ? a.beta[((size_t)b * a.T + bos + cs + r) * H + hh] : 0.f;
        }
        __syncthreads();
        // within-chunk prefix sum of the log gate, one column (channel) per thread
        for (int c = tid; c < gc; c += kThreads) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) { acc += Gs[r * gc + c]; Gs[r * gc + c] = acc; }
        }
        __syncthreads();
        // A (strictly lower, beta-scaled) and P (lower incl. diagonal, scaled)
        for (int idx = tid; idx < C * C; idx += kThreads) {
            const int i = idx / C, j = idx % C;
            float av = 0.f, pv = 0.f;
            if (j <= i) {
                float kk = 0.f, qk = 0.f;
                for (int c = 0; c < dk; ++c) {
                    const float kj = Ks[j * dk + c];
                    float e = 1.f;
                    if (PERCH) e = expf(Gs[i * gc + c] - Gs[j * gc + c]);
                    kk = fmaf(Ks[i * dk + c] * e, kj, kk);
                    qk = fmaf(Qs[i * dk + c] * e, kj, qk);
                }
                if (!PERCH) {
                    const float e = expf(Gs[i] - Gs[j]);
                    kk *= e;
                    qk *= e;
                }
                if (j < i) av = Bs[i] * kk;
                pv = a.scale * qk;
            }
            Am[i * (C + 1) + j] = av;
            Pm[i * (C + 1) + j] = pv;
        }
        __syncthreads();
        // decay factors: exp(G) and, in place of G, exp(G_L - G) (G_L = last valid row)
        for (int c = tid; c < gc; c += kThreads) {
            const float gl = Gs[(L - 1) * gc + c];
            for (int r = 0; r < C; ++r) {
                const float gr = Gs[r * gc + c];
                Es[r * gc + c] = expf(gr);
                Gs[r * gc + c] = expf(gl - gr);
            }
        }
        __syncthreads();
        // R = beta (V - (K * exp(G)) h)
        for (int idx = tid; idx < C * kBV; idx += kThreads) {
            const int i = idx / kBV, j = idx % kBV;
            float s = 0.f;
            for (int c = 0; c < dk; ++c) s = fmaf(Ks[i * dk + c] * Es[i * gc + (PERCH ? c : 0)], Hs[c * kBV + j], s);
            Ds[idx] = Bs[i] * (Vs[idx] - s);
        }
        __syncthreads();
        // forward substitution Delta[r] = R[r] - sum_{j<r} A[r][j] Delta[j]:
        // 8 lanes per column, 4 columns per warp, 8 warps cover the 32 columns
        {
            const int warp = tid >> 5, lane = tid & 31;
            const int col = warp * 4 + (lane >> 3), sub = lane & 7;
            for (int r = 1; r < L; ++r) {
                float acc = 0.f;
                for (int j = sub; j < r; j += 8) acc = fmaf(Am[r * (C + 1) + j], Ds[j * kBV + col], acc);
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                if (sub == 0) Ds[r * kBV + col] -= acc;
                __syncwarp();
            }
        }
        __syncthreads();
        // O = scale (Q * exp(G)) h + P Delta
        for (int idx = tid; idx < C * kBV; idx += kThreads) {
            const int i = idx / kBV, j = idx % kBV;
            if (i >= L || j >= bw) continue;
            float s = 0.f;
            for (int c = 0; c < dk; ++c) s = fmaf(Qs[i * dk + c] * Es[i * gc + (PERCH ? c : 0)], Hs[c * kBV + j], s);
            s *= a.scale;
            for (int m = 0; m <= i; ++m) s = fmaf(Pm[i * (C + 1) + m], Ds[m * kBV + j], s);
            o[(((size_t)b * a.T + bos + cs + i) * H + hh) * dv + j0 + j] = from_f32<Tout>(s);
        }
        __syncthreads();
        // h <- diag(exp(G_L)) h + (K * exp(G_L - G))^T Delta
        for (int idx = tid; idx < dk * kBV; idx += kThreads) {
            const int c = idx / kBV, j = idx % kBV;
            const int cc = PERCH ? c : 0;
            float s = Es[(L - 1) * gc + cc] * Hs[idx];
            for (int m = 0; m < L; ++m) s = fmaf(Ks[m * dk + c] * Gs[m * gc + cc], Ds[m * kBV + j], s);
            Hs[idx] = s;
        }
    }
    __syncthreads();
    if (a.hT) {
        for (int idx = tid; idx < dk * kBV; idx += kThreads) {
            const int c = idx / kBV, j = idx % kBV;
            if (j < bw) a.hT[sbase + (size_t)c * dv + j0 + j] = Hs[idx];
        }
    }
}

template <typename Tin, typename Tout, bool PERCH>
cudaError_t launch_typed(const ChunkArgs& a, cudaStream_t s) {
    const size_t bytes = generic_smem_floats(a.C, a.dk, PERCH) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(chunk_generic_kernel<Tin, Tout, PERCH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    const int n_tiles = (a.dv + kBV - 1) / kBV;
    const long blocks = (long)a.N() * a.H * n_tiles;
    if (blocks == 0) return cudaSuccess;
    chunk_generic_kernel<Tin, Tout, PERCH><<<(unsigned)blocks, kThreads, bytes, s>>>(a, n_tiles);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_gate(const ChunkArgs& a, cudaStream_t s) {
    return a.per_channel ? launch_typed<Tin, Tout, true>(a, s) : launch_typed<Tin, Tout, false>(a, s);
}

}  // namespace

size_t generic_smem_bytes(const ChunkArgs& a) {
    return generic_smem_floats(a.C, a.dk, a.per_channel != 0) * sizeof(float);
}

cudaError_t launch_chunk_generic(const ChunkArgs& a, cudaStream_t s) {
    if (a.bf16) return a.o_f32 ? launch_gate<__nv_bfloat16, float>(a, s) : launch_gate<__nv_bfloat16, __nv_bfloat16>(a, s);
    return a.o_f32 ? launch_gate<float, float>(a, s) : launch_gate<float, __nv_bfloat16>(a, s);
}

}  // namespace gdn
