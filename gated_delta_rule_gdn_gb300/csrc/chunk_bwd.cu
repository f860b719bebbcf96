// Chunkwise backward of the gated delta rule (scalar gate) and of KDA (per-key-channel gate), fp32 SIMT.
//
// The pages print the chunkwise backward of the ungated delta rule ("阅读笔记：DeltaNet 在 FLA 中的代码实现",
// 二、反向传播, steps 1-6: recompute U, W and the chunk states, then walk the chunks backwards carrying the
// state gradient).  This file takes the same route for the gated forms, in the algebra of the generic
// forward kernel (the state is carried transposed, h = S^T, [d_k, d_v]).  Per chunk, with G the
// within-chunk cumulative log gate (per channel for KDA), L the valid rows, E = exp(G), F = exp(G_L - G):
//   KK[r][s] = sum_c k_rc k_sc exp(G_rc - G_sc)   s < r      A = diag(beta) KK
//   P[r][s]  = scale sum_c q_rc k_sc exp(G_rc - G_sc)   s <= r
//   Z = V - (K*E) h,   R = diag(beta) Z,   Delta = (I + A)^{-1} R
//   O = scale (Q*E) h + P Delta,          h_out = diag(E_L) h + (K*F)^T Delta
// With dh the gradient of h_out (the state gradient carried from the later chunk) the adjoint is
//   dDelta = P^T dO + (K*F) dh,   Y = (I + A)^{-T} dDelta   (= dR: one back substitution, no inverse)
//   dV = diag(beta) Y,   dA = -Y Delta^T (strictly lower),   dP = dO Delta^T (lower)
//   dh_in = diag(E_L) dh + scale (Q*E)^T dO - (K*E)^T diag(beta) Y
// and dQ, dK, dbeta and the gradient of G collect the terms of every product above (the kernel below
// lists them where it forms them).  The gate gradient is that of the cumulative G, turned into dg by a
// reverse prefix sum over the chunk's rows.
//
// Two kernels:
//   * bwd_checkpoint_kernel: the forward over each (chain, 32-column d_v tile) that writes the state
//     entering every chunk (and the final state) to the workspace;
//   * bwd_chunk_kernel: one thread-block cluster per chain, one CTA per d_v tile, walking the chunks
//     from the last to the first.  The state recurrence is separable in d_v columns, so dV, the state
//     gradient and Y are complete per tile; dQ, dK, dbeta and dg sum over all d_v columns, and the CTAs
//     of the cluster add their tile parts through distributed shared memory, in rank order (the result
//     does not depend on scheduling).

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace cg = cooperative_groups;

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kBV = 32;        // d_v columns per CTA
constexpr int kTS = kBV + 1;   // padded row stride of every [rows][kBV] tile

template <typename T> __device__ __forceinline__ float ld_f32(const T* p, size_t i);
template <> __device__ __forceinline__ float ld_f32<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}

struct Geo {
    long b, bos, len;
    long slot0;  // checkpoint slot of the state entering the chain's first chunk
};

// Checkpoint slots: a batch row b takes ceil(T / C) + 1 slots from b (ceil(T / C) + 1); packed sequence n takes
// ceil(len_n / C) + 1 slots from floor(cu[n] / C) + 2 n.  Since ceil((y - x) / C) <= floor(y / C) - floor(x / C) + 1,
// the packed ranges never overlap and end at or before floor(T / C) + 2 n_seqs, for any cu_seqlens once clamped
// to [0, T].
__device__ __forceinline__ Geo chain_geo(const BwdArgs& a, long n) {
    Geo r;
    if (a.cu) {
        long s0 = a.cu[n], s1 = a.cu[n + 1];
        s0 = s0 < 0 ? 0 : (s0 > a.T ? a.T : s0);
        s1 = s1 < s0 ? s0 : (s1 > a.T ? a.T : s1);
        r.b = 0; r.bos = s0; r.len = s1 - s0;
        r.slot0 = s0 / a.C + 2 * n;
    } else {
        r.b = n; r.bos = 0; r.len = a.T;
        r.slot0 = n * ((a.T + a.C - 1) / a.C + 1);
    }
    return r;
}

__host__ __device__ inline long checkpoint_slots(int B, int T, int C, int n_seqs, bool varlen) {
    return varlen ? (long)(T / C) + 2L * n_seqs : (long)B * ((T + C - 1) / C + 1);
}

// Shared-memory carve-up, in floats.  Q and K rows (and the per-channel gate rows) are padded to d_k + 1 floats, so
// that lanes reading one column of consecutive rows hit distinct banks.  The backward kernel uses all of it; the checkpoint kernel the K, V, gate,
// beta, KK, state and Delta parts.
struct Lay {
    int Q, K, V, dO, G, E, F, Bt, KK, P, Ex, dP, dA, H, dH, Z, D, Y, pq, pk, pb, pw, pbeta, us, red, total;
};

__host__ __device__ inline Lay make_lay(int C, int dk, bool per_channel) {
    const int lg = per_channel ? dk + 1 : 1, cc = C * (C + 1), ct = C * kTS, ht = dk * kTS;
    Lay l;
    int o = 0;
    l.Q = o; o += C * (dk + 1);
    l.K = o; o += C * (dk + 1);
    l.V = o; o += ct;
    l.dO = o; o += ct;
    l.G = o; o += C * lg;
    l.E = o; o += C * lg;
    l.F = o; o += C * lg;
    l.Bt = o; o += C;
    l.KK = o; o += cc;
    l.P = o; o += cc;
    l.Ex = o; o += per_channel ? 0 : cc;   // exp(G_r - G_s), scalar gate only
    l.dP = o; o += cc;
    l.dA = o; o += cc;
    l.H = o; o += ht;
    l.dH = o; o += ht;
    l.Z = o; o += ct;
    l.D = o; o += ct;
    l.Y = o; o += ct;
    l.pq = o; o += C * dk;
    l.pk = o; o += C * dk;
    l.pb = o; o += C * dk;
    l.pw = o; o += C * dk;
    l.pbeta = o; o += C;
    l.us = o; o += dk;
    l.red = o; o += 2 * C + 1;
    l.total = o;
    return l;
}

__host__ __device__ inline int ck_floats(int C, int dk, bool per_channel) {
    const int lg = per_channel ? dk + 1 : 1;
    return C * (dk + 1) + C * kTS + 3 * C * lg + C + C * (C + 1) + dk * kTS + C * kTS;
}

// ---- steps shared by both kernels -------------------------------------------------------------------

// Load K (and Q), the V tile (and the dO tile), the gate and beta of one chunk; rows >= L are zero, which leaves
// the state unchanged (beta = 0, g = 0).
template <typename Tin, typename Tdo, bool PERCH, bool WITH_Q>
__device__ __forceinline__ void load_chunk(const BwdArgs& a, const Geo& geo, int hh, long cs, int L, int j0, int bw,
                                           float* Qs, float* Ks, float* Vs, float* Os, float* Gs, float* Bs) {
    const int C = a.C, dk = a.dk, dv = a.dv, H = a.H, gc = PERCH ? dk : 1, ld = dk + 1, lg = PERCH ? dk + 1 : 1;
    const Tin* q = static_cast<const Tin*>(a.q);
    const Tin* k = static_cast<const Tin*>(a.k);
    const Tin* v = static_cast<const Tin*>(a.v);
    const Tdo* dO = static_cast<const Tdo*>(a.dO);
    const size_t tok0 = ((size_t)geo.b * a.T + geo.bos + cs) * H + hh;
    for (int idx = threadIdx.x; idx < C * dk; idx += kThreads) {
        const int r = idx / dk, c = idx % dk;
        float kv = 0.f, qv = 0.f;
        if (r < L) {
            const size_t off = (tok0 + (size_t)r * H) * dk + c;
            kv = ld_f32<Tin>(k, off);
            if (WITH_Q) qv = ld_f32<Tin>(q, off);
        }
        Ks[r * ld + c] = kv;
        if (WITH_Q) Qs[r * ld + c] = qv;
    }
    for (int idx = threadIdx.x; idx < C * kBV; idx += kThreads) {
        const int r = idx / kBV, j = idx % kBV;
        float vv = 0.f, ov = 0.f;
        if (r < L && j < bw) {
            const size_t off = (tok0 + (size_t)r * H) * dv + j0 + j;
            vv = ld_f32<Tin>(v, off);
            if (WITH_Q) ov = ld_f32<Tdo>(dO, off);
        }
        Vs[r * kTS + j] = vv;
        if (WITH_Q) Os[r * kTS + j] = ov;
    }
    for (int idx = threadIdx.x; idx < C * gc; idx += kThreads) {
        const int r = idx / gc, c = idx % gc;
        const size_t tok = tok0 + (size_t)r * H;
        Gs[r * lg + c] = (r < L) ? a.g[PERCH ? tok * dk + c : tok] : 0.f;
    }
    for (int r = threadIdx.x; r < C; r += kThreads) Bs[r] = (r < L) ? a.beta[tok0 + (size_t)r * H] : 0.f;
}

// Load a [dk][kBV] state tile (columns >= bw zero) from a [dk][dv] state, or zeros.
__device__ __forceinline__ void load_state(float* Hs, const float* src, int dk, int dv, int j0, int bw) {
    for (int idx = threadIdx.x; idx < dk * kBV; idx += kThreads) {
        const int c = idx / kBV, j = idx % kBV;
        Hs[c * kTS + j] = (src && j < bw) ? src[(size_t)c * dv + j0 + j] : 0.f;
    }
}

__device__ __forceinline__ void store_state(float* dst, const float* Hs, int dk, int dv, int j0, int bw) {
    for (int idx = threadIdx.x; idx < dk * kBV; idx += kThreads) {
        const int c = idx / kBV, j = idx % kBV;
        if (j < bw) dst[(size_t)c * dv + j0 + j] = Hs[c * kTS + j];
    }
}

// Within-chunk prefix sum of the log gate, one channel per thread.
__device__ __forceinline__ void gate_prefix(float* Gs, int C, int gc, int lg) {
    for (int c = threadIdx.x; c < gc; c += kThreads) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) { acc += Gs[r * lg + c]; Gs[r * lg + c] = acc; }
    }
}

// E = exp(G), F = exp(G_L - G) (G_L: the last valid row).
__device__ __forceinline__ void gate_factors(const float* Gs, float* Es, float* Fs, int C, int gc, int lg, int L) {
    for (int c = threadIdx.x; c < gc; c += kThreads) {
        const float gl = Gs[(L - 1) * lg + c];
        for (int r = 0; r < C; ++r) {
            const float gr = Gs[r * lg + c];
            Es[r * lg + c] = expf(gr);
            Fs[r * lg + c] = expf(gl - gr);
        }
    }
}

// KK (strictly lower), and with WITH_P the read matrix P (lower incl. the diagonal, scaled) and, for the scalar
// gate, Ex[r][s] = exp(G_r - G_s) (s <= r).  Exponents are formed only for s <= r, so no factor exceeds 1.
template <bool PERCH, bool WITH_P>
__device__ __forceinline__ void pair_products(const float* Qs, const float* Ks, const float* Gs, float* KK, float* Pm,
                                              float* Ex, int C, int dk, float scale) {
    const int ld = dk + 1, lg = PERCH ? dk + 1 : 1;
    for (int idx = threadIdx.x; idx < C * C; idx += kThreads) {
        const int r = idx / C, s = idx % C;
        float kk = 0.f, qk = 0.f, e0 = 0.f;
        if (s <= r) {
            for (int c = 0; c < dk; ++c) {
                const float ks = Ks[s * ld + c];
                float e = 1.f;
                if (PERCH) e = expf(Gs[r * lg + c] - Gs[s * lg + c]);
                kk = fmaf(Ks[r * ld + c] * e, ks, kk);
                if (WITH_P) qk = fmaf(Qs[r * ld + c] * e, ks, qk);
            }
            if (!PERCH) {
                e0 = expf(Gs[r] - Gs[s]);
                kk *= e0;
                qk *= e0;
            }
        }
        KK[r * (C + 1) + s] = (s < r) ? kk : 0.f;
        if (WITH_P) {
            Pm[r * (C + 1) + s] = scale * qk;
            if (!PERCH) Ex[r * (C + 1) + s] = e0;
        }
    }
}

// Z = V - (K * E) h and R = diag(beta) Z (Z only if Zs is non-null).
template <bool PERCH>
__device__ __forceinline__ void residual(const float* Ks, const float* Es, const float* Vs, const float* Hs,
                                         const float* Bs, float* Zs, float* Ds, int C, int dk) {
    const int ld = dk + 1, lg = PERCH ? dk + 1 : 1;
    for (int idx = threadIdx.x; idx < C * kBV; idx += kThreads) {
        const int i = idx / kBV, j = idx % kBV;
        float s = 0.f;
        for (int c = 0; c < dk; ++c) s = fmaf(Ks[i * ld + c] * Es[i * lg + (PERCH ? c : 0)], Hs[c * kTS + j], s);
        const float z = Vs[i * kTS + j] - s;
        if (Zs) Zs[i * kTS + j] = z;
        Ds[i * kTS + j] = Bs[i] * z;
    }
}

// (I + A) X = X0 in place, A = diag(beta) KK strictly lower: rows in order.  8 lanes per column, 4 columns per
// warp, 8 warps: the 32 columns of the tile.
__device__ __forceinline__ void solve_lower(const float* KK, const float* Bs, float* X, int C, int L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = warp * 4 + (lane >> 3), sub = lane & 7;
    for (int r = 1; r < L; ++r) {
        float acc = 0.f;
        for (int j = sub; j < r; j += 8) acc = fmaf(KK[r * (C + 1) + j], X[j * kTS + col], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (sub == 0) X[r * kTS + col] -= Bs[r] * acc;
        __syncwarp();
    }
}

// (I + A)^T X = X0 in place: rows from the last valid one down.
__device__ __forceinline__ void solve_upper_t(const float* KK, const float* Bs, float* X, int C, int L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = warp * 4 + (lane >> 3), sub = lane & 7;
    for (int s = L - 2; s >= 0; --s) {
        float acc = 0.f;
        for (int r = s + 1 + sub; r < L; r += 8) acc = fmaf(Bs[r] * KK[r * (C + 1) + s], X[r * kTS + col], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (sub == 0) X[s * kTS + col] -= acc;
        __syncwarp();
    }
}

// ---- kernel 1: chunk-entry states ------------------------------------------------------------------------

template <typename Tin, bool PERCH>
__global__ void __launch_bounds__(kThreads) bwd_checkpoint_kernel(const BwdArgs a, int n_tiles) {
    extern __shared__ float smem[];
    const int C = a.C, dk = a.dk, dv = a.dv, H = a.H, gc = PERCH ? dk : 1, ld = dk + 1, lg = PERCH ? dk + 1 : 1;
    float* Ks = smem;
    float* Vs = Ks + C * ld;
    float* Gs = Vs + C * kTS;
    float* Es = Gs + C * lg;
    float* Fs = Es + C * lg;
    float* Bs = Fs + C * lg;
    float* KK = Bs + C;
    float* Hs = KK + C * (C + 1);
    float* Ds = Hs + dk * kTS;

    const long chain = blockIdx.x / n_tiles;
    const int tile = blockIdx.x % n_tiles;
    const long n = chain / H;
    const int hh = (int)(chain % H);
    const Geo geo = chain_geo(a, n);
    const int j0 = tile * kBV, bw = min(kBV, dv - j0);
    const size_t sstride = (size_t)H * dk * dv;
    float* ck = a.ck + (size_t)geo.slot0 * sstride + (size_t)hh * dk * dv;

    load_state(Hs, a.h0 ? a.h0 + ((size_t)n * H + hh) * dk * dv : nullptr, dk, dv, j0, bw);
    __syncthreads();
    store_state(ck, Hs, dk, dv, j0, bw);
    long ci = 0;
    for (long cs = 0; cs < geo.len; cs += C, ++ci) {
        const int L = (int)min((long)C, geo.len - cs);
        __syncthreads();
        load_chunk<Tin, Tin, PERCH, false>(a, geo, hh, cs, L, j0, bw, nullptr, Ks, Vs, nullptr, Gs, Bs);
        __syncthreads();
        gate_prefix(Gs, C, gc, lg);
        __syncthreads();
        gate_factors(Gs, Es, Fs, C, gc, lg, L);
        pair_products<PERCH, false>(nullptr, Ks, Gs, KK, nullptr, nullptr, C, dk, 0.f);
        __syncthreads();
        residual<PERCH>(Ks, Es, Vs, Hs, Bs, nullptr, Ds, C, dk);
        __syncthreads();
        solve_lower(KK, Bs, Ds, C, L);
        __syncthreads();
        // h <- diag(E_L) h + (K * F)^T Delta
        for (int idx = threadIdx.x; idx < dk * kBV; idx += kThreads) {
            const int c = idx / kBV, j = idx % kBV, cc = PERCH ? c : 0;
            float s = Es[(L - 1) * lg + cc] * Hs[c * kTS + j];
            for (int m = 0; m < L; ++m) s = fmaf(Ks[m * ld + c] * Fs[m * lg + cc], Ds[m * kTS + j], s);
            Hs[c * kTS + j] = s;
        }
        __syncthreads();
        store_state(ck + (size_t)(ci + 1) * sstride, Hs, dk, dv, j0, bw);
    }
}

// ---- kernel 2: the backward walk -------------------------------------------------------------------------

template <typename Tin, typename Tdo, bool PERCH>
__global__ void __launch_bounds__(kThreads) bwd_chunk_kernel(const BwdArgs a, int n_tiles) {
    extern __shared__ float smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int C = a.C, dk = a.dk, dv = a.dv, H = a.H, gc = PERCH ? dk : 1, ld = dk + 1, lg = PERCH ? dk + 1 : 1;
    const Lay ly = make_lay(C, dk, PERCH);
    float* Qs = smem + ly.Q;  float* Ks = smem + ly.K;  float* Vs = smem + ly.V;  float* Os = smem + ly.dO;
    float* Gs = smem + ly.G;  float* Es = smem + ly.E;  float* Fs = smem + ly.F;  float* Bs = smem + ly.Bt;
    float* KK = smem + ly.KK; float* Pm = smem + ly.P;  float* Ex = smem + ly.Ex;
    float* dPm = smem + ly.dP; float* dAm = smem + ly.dA;
    float* Hs = smem + ly.H;  float* dHs = smem + ly.dH;
    float* Zs = smem + ly.Z;  float* Ds = smem + ly.D;  float* Ys = smem + ly.Y;
    float* pq = smem + ly.pq; float* pk = smem + ly.pk; float* pb = smem + ly.pb; float* pw = smem + ly.pw;
    float* pbeta = smem + ly.pbeta; float* us = smem + ly.us; float* red = smem + ly.red;

    const int tid = threadIdx.x;
    const int rank = (int)cluster.block_rank();  // the d_v tile
    const long chain = blockIdx.x / n_tiles;
    const long n = chain / H;
    const int hh = (int)(chain % H);
    const Geo geo = chain_geo(a, n);
    const int j0 = rank * kBV, bw = min(kBV, dv - j0);
    const size_t sstride = (size_t)H * dk * dv;
    const float* ck = a.ck + (size_t)geo.slot0 * sstride + (size_t)hh * dk * dv;
    const long n_chunks = (geo.len + C - 1) / C;
    const float scale = a.scale;

    // state gradient at the end of the chain
    load_state(dHs, a.dhT ? a.dhT + ((size_t)n * H + hh) * dk * dv : nullptr, dk, dv, j0, bw);

    for (long ci = n_chunks - 1; ci >= 0; --ci) {
        const long cs = ci * C;
        const int L = (int)min((long)C, geo.len - cs);
        const size_t tok0 = ((size_t)geo.b * a.T + geo.bos + cs) * H + hh;
        __syncthreads();
        load_chunk<Tin, Tdo, PERCH, true>(a, geo, hh, cs, L, j0, bw, Qs, Ks, Vs, Os, Gs, Bs);
        load_state(Hs, ck + (size_t)ci * sstride, dk, dv, j0, bw);
        __syncthreads();
        gate_prefix(Gs, C, gc, lg);
        __syncthreads();
        gate_factors(Gs, Es, Fs, C, gc, lg, L);
        pair_products<PERCH, true>(Qs, Ks, Gs, KK, Pm, Ex, C, dk, scale);
        __syncthreads();
        // Z, R = beta Z (into Delta), and dDelta = P^T dO + (K * F) dh (into Y)
        residual<PERCH>(Ks, Es, Vs, Hs, Bs, Zs, Ds, C, dk);
        for (int idx = tid; idx < C * kBV; idx += kThreads) {
            const int i = idx / kBV, j = idx % kBV;
            float s = 0.f;
            for (int r = i; r < L; ++r) s = fmaf(Pm[r * (C + 1) + i], Os[r * kTS + j], s);
            for (int c = 0; c < dk; ++c)
                s = fmaf(Ks[i * ld + c] * Fs[i * lg + (PERCH ? c : 0)], dHs[c * kTS + j], s);
            Ys[i * kTS + j] = s;
        }
        __syncthreads();
        solve_lower(KK, Bs, Ds, C, L);      // Delta
        solve_upper_t(KK, Bs, Ys, C, L);    // Y = dR
        __syncthreads();
        // dV = diag(beta) Y (complete for this tile); dP = dO Delta^T (s <= r) and dA = -Y Delta^T (s < r)
        for (int idx = tid; idx < C * kBV; idx += kThreads) {
            const int i = idx / kBV, j = idx % kBV;
            if (i < L && j < bw) a.gv[(tok0 + (size_t)i * H) * dv + j0 + j] = Bs[i] * Ys[i * kTS + j];
        }
        for (int idx = tid; idx < C * C; idx += kThreads) {
            const int r = idx / C, s = idx % C;
            float dp = 0.f, da = 0.f;
            if (s <= r && r < L) {
                for (int j = 0; j < kBV; ++j) {
                    const float d = Ds[s * kTS + j];
                    dp = fmaf(Os[r * kTS + j], d, dp);
                    da = fmaf(Ys[r * kTS + j], d, da);
                }
            }
            dPm[r * (C + 1) + s] = dp;
            dAm[r * (C + 1) + s] = (s < r) ? -da : 0.f;
        }
        __syncthreads();
        // Tile parts of dQ, dK and the gradient of G, per (row r, channel c):
        //   xo = (h dO_r)_c, hy = (h Y_r)_c, dd = (dh Delta_r)_c
        //   SQ  = scale sum_{s<r} dP[r][s] k_sc e(r,s)         SAR = beta_r sum_{s<r} dA[r][s] k_sc e(r,s)
        //   SKP = scale sum_{u>r} dP[u][r] q_uc e(u,r)         SAC = sum_{u>r} dA[u][r] beta_u k_uc e(u,r)
        // with e(r,s) = exp(G_rc - G_sc), and the diagonal term D = scale dP[r][r];
        //   dQ = scale E xo + SQ + D k_rc
        //   dK = -beta E hy + F dd + SKP + D q_rc + SAR + SAC
        //   gradient of G_r: q SQ - k SKP + k SAR - k SAC + scale E q xo - beta E k hy   (pb)
        //                    and the write term F k dd, which reaches g_u for u > r only   (pw)
        // The diagonal of P carries exp(0) and drops out of the gate gradient; so does the last write of
        // the chunk, whose gate term and F term cancel.  Leaving both out in closed form (rather than
        // forming and cancelling them) keeps the gate gradient accurate under strong decay.
        for (int idx = tid; idx < C * dk; idx += kThreads) {
            const int r = idx / dk, c = idx % dk, cc = PERCH ? c : 0;
            if (r >= L) continue;
            float xo = 0.f, hy = 0.f, dd = 0.f;
            for (int j = 0; j < kBV; ++j) {
                const float hv = Hs[c * kTS + j];
                xo = fmaf(hv, Os[r * kTS + j], xo);
                hy = fmaf(hv, Ys[r * kTS + j], hy);
                dd = fmaf(dHs[c * kTS + j], Ds[r * kTS + j], dd);
            }
            float sq = 0.f, sar = 0.f, skp = 0.f, sac = 0.f;
            for (int s = 0; s < r; ++s) {
                const float e = PERCH ? expf(Gs[r * lg + c] - Gs[s * lg + c]) : Ex[r * (C + 1) + s];
                const float ke = Ks[s * ld + c] * e;
                sq = fmaf(dPm[r * (C + 1) + s], ke, sq);
                sar = fmaf(dAm[r * (C + 1) + s], ke, sar);
            }
            for (int u = r + 1; u < L; ++u) {
                const float e = PERCH ? expf(Gs[u * lg + c] - Gs[r * lg + c]) : Ex[u * (C + 1) + r];
                skp = fmaf(dPm[u * (C + 1) + r], Qs[u * ld + c] * e, skp);
                sac = fmaf(dAm[u * (C + 1) + r] * Bs[u], Ks[u * ld + c] * e, sac);
            }
            sq *= scale;
            skp *= scale;
            sar *= Bs[r];
            const float E = Es[r * lg + cc], F = Fs[r * lg + cc], br = Bs[r];
            const float qr = Qs[r * ld + c], kr = Ks[r * ld + c];
            const float dg0 = scale * dPm[r * (C + 1) + r];
            const float read = scale * E * xo;
            pq[idx] = read + sq + dg0 * kr;
            pk[idx] = -br * E * hy + F * dd + skp + dg0 * qr + sar + sac;
            pb[idx] = qr * (read + sq) - kr * (br * E * hy + skp - sar + sac);
            pw[idx] = F * kr * dd;
        }
        // us[c] = E_L sum_j dh[c][j] h[c][j]: the entry state's part of the gate term of h_out (tile part)
        for (int c = tid; c < dk; c += kThreads) {
            float s = 0.f;
            for (int j = 0; j < kBV; ++j) s = fmaf(dHs[c * kTS + j], Hs[c * kTS + j], s);
            us[c] = Es[(L - 1) * lg + (PERCH ? c : 0)] * s;
        }
        // tile part of dbeta: Y_r . Z_r + sum_{s<r} dA[r][s] KK[r][s]
        for (int r = tid; r < L; r += kThreads) {
            float s = 0.f;
            for (int j = 0; j < kBV; ++j) s = fmaf(Ys[r * kTS + j], Zs[r * kTS + j], s);
            for (int m = 0; m < r; ++m) s = fmaf(dAm[r * (C + 1) + m], KK[r * (C + 1) + m], s);
            pbeta[r] = s;
        }
        __syncthreads();
        // dh <- diag(E_L) dh + scale (Q * E)^T dO - (K * E)^T diag(beta) Y
        for (int idx = tid; idx < dk * kBV; idx += kThreads) {
            const int c = idx / kBV, j = idx % kBV, cc = PERCH ? c : 0;
            float s = Es[(L - 1) * lg + cc] * dHs[c * kTS + j];
            for (int r = 0; r < L; ++r) {
                const float e = Es[r * lg + cc];
                s = fmaf(scale * Qs[r * ld + c] * e, Os[r * kTS + j], s);
                s = fmaf(-Ks[r * ld + c] * e * Bs[r], Ys[r * kTS + j], s);
            }
            dHs[c * kTS + j] = s;
        }
        if (!PERCH) {
            // scalar gate: this tile's sums over the channels, per row (red[r], red[C + r]) and of us (red[2C])
            const int warp = tid >> 5, lane = tid & 31;
            for (int r = warp; r <= L; r += kThreads / 32) {
                float sb = 0.f, sw = 0.f;
                if (r < L) {
                    for (int c = lane; c < dk; c += 32) { sb += pb[r * dk + c]; sw += pw[r * dk + c]; }
                } else {
                    for (int c = lane; c < dk; c += 32) sb += us[c];
                }
                for (int o = 16; o > 0; o >>= 1) {
                    sb += __shfl_xor_sync(0xffffffffu, sb, o);
                    sw += __shfl_xor_sync(0xffffffffu, sw, o);
                }
                if (lane == 0) {
                    if (r < L) { red[r] = sb; red[C + r] = sw; } else { red[2 * C] = sb; }
                }
            }
        }
        cluster.sync();  // every tile part of this chunk is in shared memory
        {
            const int stride = n_tiles * kThreads;
            for (int idx = rank * kThreads + tid; idx < L * dk; idx += stride) {
                float sq = 0.f, sk = 0.f;
                for (int t = 0; t < n_tiles; ++t) {
                    sq += cluster.map_shared_rank(pq, t)[idx];
                    sk += cluster.map_shared_rank(pk, t)[idx];
                }
                const int r = idx / dk, c = idx % dk;
                const size_t off = (tok0 + (size_t)r * H) * dk + c;
                a.gq[off] = sq;
                a.gk[off] = sk;
            }
            for (int r = rank * kThreads + tid; r < L; r += stride) {
                float s = 0.f;
                for (int t = 0; t < n_tiles; ++t) s += cluster.map_shared_rank(pbeta, t)[r];
                a.gbeta[tok0 + (size_t)r * H] = s;
            }
            // dg[u] = sum_{r >= u} pb[r] + sum_{s < u} pw[s] + us, over the tiles (and the channels for the scalar
            // gate)
            if (PERCH) {
                // this CTA takes channels [c0, c0 + cw): first the tile sums of pb and pw for every (row, channel),
                // all loads independent, into the Q / K space (no other CTA reads it), then one thread per channel
                // runs the two prefix sums over the rows
                const int cw0 = (dk + n_tiles - 1) / n_tiles, c0 = rank * cw0, cw = max(0, min(dk - c0, cw0));
                float* sbuf = Qs;
                float* wbuf = Qs + C * cw0;
                for (int idx = tid; idx < L * cw; idx += kThreads) {
                    const int r = idx / cw, c = c0 + idx % cw;
                    float sb = 0.f, sw = 0.f;
                    for (int t = 0; t < n_tiles; ++t) {
                        sb += cluster.map_shared_rank(pb, t)[r * dk + c];
                        sw += cluster.map_shared_rank(pw, t)[r * dk + c];
                    }
                    sbuf[idx] = sb;
                    wbuf[idx] = sw;
                }
                __syncthreads();
                for (int cl = tid; cl < cw; cl += kThreads) {
                    const int c = c0 + cl;
                    float pre = 0.f;
                    for (int t = 0; t < n_tiles; ++t) pre += cluster.map_shared_rank(us, t)[c];
                    for (int u = 0; u < L; ++u) {
                        const float w = wbuf[u * cw + cl];
                        wbuf[u * cw + cl] = pre;
                        pre += w;
                    }
                    float acc = 0.f;
                    for (int r = L - 1; r >= 0; --r) {
                        acc += sbuf[r * cw + cl];
                        a.gg[(tok0 + (size_t)r * H) * dk + c] = acc + wbuf[r * cw + cl];
                    }
                }
            } else if (rank == 0 && tid < 32) {
                // one warp, lane r = row r (L <= 32): the tile sums of the per-row channel sums, then a reverse
                // inclusive scan of pb and a forward exclusive scan of pw across the lanes
                const int lane = tid;
                float sb = 0.f, sw = 0.f, ut = 0.f;
                for (int t = 0; t < n_tiles; ++t) {
                    const float* rr = cluster.map_shared_rank(red, t);
                    if (lane < L) { sb += rr[lane]; sw += rr[C + lane]; }
                    ut += rr[2 * C];
                }
                float rev = sb, fwd = sw;
                for (int o = 1; o < 32; o <<= 1) {
                    const float x = __shfl_down_sync(0xffffffffu, rev, o);
                    const float y = __shfl_up_sync(0xffffffffu, fwd, o);
                    if (lane + o < 32) rev += x;
                    if (lane >= o) fwd += y;
                }
                float ex = __shfl_up_sync(0xffffffffu, fwd, 1);   // exclusive: the inclusive sum of the lane before
                if (lane == 0) ex = 0.f;
                if (lane < L) a.gg[tok0 + (size_t)lane * H] = rev + ex + ut;
            }
        }
        cluster.sync();  // no CTA overwrites its tile parts while another still reads them
    }
    __syncthreads();
    if (a.gh0) store_state(a.gh0 + ((size_t)n * H + hh) * dk * dv, dHs, dk, dv, j0, bw);
}

template <typename Tin, typename Tdo, bool PERCH>
cudaError_t launch_typed(const BwdArgs& a, cudaStream_t s) {
    const int n_tiles = (a.dv + kBV - 1) / kBV;
    const long chains = (long)a.N() * a.H;
    if (chains == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)(chains * n_tiles);

    const size_t ck_bytes = (size_t)ck_floats(a.C, a.dk, PERCH) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(bwd_checkpoint_kernel<Tin, PERCH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ck_bytes);
    if (e != cudaSuccess) return e;
    bwd_checkpoint_kernel<Tin, PERCH><<<blocks, kThreads, ck_bytes, s>>>(a, n_tiles);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    const size_t bytes = bwd_smem_bytes(a.C, a.dk, PERCH);
    auto kern = bwd_chunk_kernel<Tin, Tdo, PERCH>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)n_tiles;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidClusterSize;
    return cudaLaunchKernelEx(&cfg, kern, a, n_tiles);
}

template <typename Tin>
cudaError_t launch_in(const BwdArgs& a, cudaStream_t s) {
    if (a.do_bf16)
        return a.per_channel ? launch_typed<Tin, __nv_bfloat16, true>(a, s) : launch_typed<Tin, __nv_bfloat16, false>(a, s);
    return a.per_channel ? launch_typed<Tin, float, true>(a, s) : launch_typed<Tin, float, false>(a, s);
}

}  // namespace

size_t bwd_smem_bytes(int C, int dk, bool per_channel) {
    return (size_t)make_lay(C, dk, per_channel).total * sizeof(float);
}

int bwd_auto_chunk(int dk, bool per_channel) {
    for (int C : {32, 16})
        if (bwd_smem_bytes(C, dk, per_channel) <= kMaxSmemPerBlock) return C;
    return 0;
}

size_t bwd_workspace_bytes(const BwdArgs& a) {
    return (size_t)checkpoint_slots(a.B, a.T, a.C, a.n_seqs, a.cu != nullptr) * a.H * a.dk * a.dv * sizeof(float);
}

cudaError_t launch_chunk_bwd(const BwdArgs& a, cudaStream_t s) {
    return a.bf16 ? launch_in<__nv_bfloat16>(a, s) : launch_in<float>(a, s);
}

}  // namespace gdn
