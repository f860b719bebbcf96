// Chunkwise backward of the gated delta rule (scalar gate) and of KDA (per-key-channel gate): fp32 arithmetic,
// FMAs and 3xTF32 warp MMAs (mma.sync m16n8k8, each operand split into a TF32 head and tail).
//
// The pages print the chunkwise backward of the ungated delta rule ("阅读笔记：DeltaNet 在 FLA 中的代码实现",
// 二、反向传播, steps 1-6): recompute the chunk states, walk the chunks backwards carrying the state gradient,
// then form the per-chunk gradients.  This file takes the same route for the gated forms, in the algebra of the
// generic forward kernel (the state is carried transposed, h = S^T, [d_k, d_v]).  Per chunk, with G the
// within-chunk cumulative log gate (per channel for KDA), L the valid rows, E = exp(G), F = exp(G_L - G):
//   KK[r][s] = sum_c k_rc k_sc exp(G_rc - G_sc)   s < r      A = diag(beta) KK
//   P[r][s]  = scale sum_c q_rc k_sc exp(G_rc - G_sc)   s <= r
//   Z = V - (K*E) h,   R = diag(beta) Z,   Delta = (I + A)^{-1} R
//   O = scale (Q*E) h + P Delta,          h_out = diag(E_L) h + (K*F)^T Delta
// With dh the gradient of h_out (the state gradient carried from the later chunk) the adjoint is
//   dDelta = P^T dO + (K*F) dh,   Y = (I + A)^{-T} dDelta   (= dR)
// The walks take both triangular systems as products by T = (I + A)^{-1}, which the prep kernel forms once per
// chunk by forward substitution (Delta = T R, Y = T^T dDelta).
//   dV = diag(beta) Y,   dA = -Y Delta^T (strictly lower),   dP = dO Delta^T (lower)
//   dh_in = diag(E_L) dh + scale (Q*E)^T dO - (K*E)^T diag(beta) Y
// and dQ, dK, dbeta and the gradient of G collect the terms of every product above (bwd_grad_kernel lists them
// where it forms them).  The gate gradient is that of the cumulative G, turned into dg by prefix sums over the
// chunk's rows.
//
// Four kernels, in three launches:
//   * bwd_prep_kernel, one CTA per (chunk, head): everything of a chunk that does not depend on the state -- the
//     cumulative gate, KK, P, scale Q*E, T = (I + A)^{-1}, K*E, K*F, exp(G_L) and beta -- into a per-chunk
//     record.
//   * bwd_walk_kernel, one CTA per (chain, 64-column d_v tile) and role.  The state recurrence is separable in
//     d_v columns, so each tile walks alone.  The forward role runs the chunks in order and stores, per chunk,
//     the entry state h, Delta and Z; the backward role runs them in reverse and stores, per chunk, the
//     gradient of h_out and Y.  Neither needs the other's results, so both roles share one launch.  Each
//     thread keeps its part of the state (or state gradient) in registers; the chunk records arrive by bulk
//     copies (cp.async.bulk, two stages), so a step waits only on its own dependent chain.
//   * bwd_grad_kernel, one CTA per (chunk, head), over all d_v tiles: every chunk is independent once the two
//     walks are done, so this runs over the whole GPU.  It writes dQ, dK, dV, dbeta and dg.
// Around them, when asked for: the gate / beta activations from raw logits before, and their chain rule after
// (bwd_act_*); with grouped value heads, the sum of the per-value-head dQ, dK parts per key head
// (bwd_group_sum_kernel).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "gate_act.cuh"
#include "tc_common.cuh"

namespace gdn {

__device__ unsigned g_bwd_status;   // bit 0: a walk gave up a bounded wait for its chunk records

namespace {

using namespace tc;
constexpr uint64_t kWaitNs = 2000000000ull;

constexpr int kThreads = 256;
constexpr int kBV = 32;        // d_v columns per tile of the gradient kernel
constexpr int kWB = 64;        // d_v columns per walk CTA
constexpr int kWS = 72;        // row stride of the walk's [rows][kWB] tiles: MMA fragment loads hit banks 8 t + g

template <typename T> __device__ __forceinline__ float ld_f32(const T* p, size_t i);
template <> __device__ __forceinline__ float ld_f32<float>(const float* p, size_t i) { return p[i]; }
template <> __device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}

__host__ __device__ inline int round4(int x) { return (x + 3) & ~3; }

// x = hi + lo with hi and lo TF32 (the high part rounded to nearest, the low part the rounded remainder)
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
    const float r = x - __uint_as_float(hi);
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// d (16 x 8) += A (16 x 8) B (8 x 8) to about fp32 accuracy from three TF32 warp products: A_hi B_hi + A_hi B_lo
// + A_lo B_hi (the dropped A_lo B_lo is below fp32 rounding).  Fragments as in the PTX m16n8k8 layout
// (lane = 4 g + t): A rows g, g + 8 and columns t, t + 4; B rows t, t + 4 and column g; d rows g, g + 8 and
// columns 2 t, 2 t + 1.
__device__ __forceinline__ void mma3_tf32(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                          const uint32_t (&bh)[2], const uint32_t (&bl)[2]) {
    mma_tf32(d, al, bh);
    mma_tf32(d, ah, bl);
    mma_tf32(d, ah, bh);
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned), in the calling thread's cp.async group
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most N of this thread's committed groups are still in flight
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// Channels of the state each walk thread keeps in registers (8 channel groups of kThreads / 32 warps).
__host__ __device__ inline int walk_cpt(int dk) { return dk <= 128 ? 16 : 32; }

struct Geo {
    long b, bos, len;
    long slot0;  // workspace slot of the chain's first chunk
};

// Workspace slots: a batch row b takes ceil(T / C) + 1 slots from b (ceil(T / C) + 1); packed sequence n takes
// ceil(len_n / C) + 1 slots from floor(cu[n] / C) + 2 n.  Since ceil((y - x) / C) <= floor(y / C) - floor(x / C) + 1,
// the packed ranges never overlap and end at or before floor(T / C) + 2 n_seqs, for any cu_seqlens once clamped
// to [0, T].  Slot slot0 + i holds chunk i; the last slot of a chain holds its final state.
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

__host__ __device__ inline long workspace_slots(int B, int T, int C, int n_seqs, bool varlen) {
    return varlen ? (long)(T / C) + 2L * n_seqs : (long)B * ((T + C - 1) / C + 1);
}

// The per-chunk record of the prep kernel (floats; every part starts on 16 bytes).  The walks copy its parts before
// G in one or two bulk copies, so the order matters: KK, P, QE, KE, KF, EL, B, then G.
//   KK [C][C+1]   sum_c k_rc k_sc exp(G_rc - G_sc), s < r      P [C][C+1]   the read matrix, s <= r
//   QE, KE, KF [C][ldk]   scale q exp(G), k exp(G), k exp(G_L - G), zero beyond d_k
//   EL [ldk or 4]   exp(G_L) per channel (scalar gate: repeated)      B [C]   beta
//   G  [C][lg]   the within-chunk cumulative log gate
struct Rec {
    int KK, P, QE, T, KE, KF, EL, B, G, total;
};

__host__ __device__ inline Rec rec_lay(int C, int dk, bool perch) {
    const int ldk = 8 * walk_cpt(dk) + 4, lg = perch ? ldk : 1, cc = C * (C + 1);
    Rec r;
    int o = 0;
    r.KK = o; o = round4(o + cc);
    r.P = o; o = round4(o + cc);
    r.QE = o; o = round4(o + C * ldk);
    r.T = o; o = round4(o + cc);
    r.KE = o; o = round4(o + C * ldk);
    r.KF = o; o = round4(o + C * ldk);
    r.EL = o; o = round4(o + (perch ? ldk : 4));
    r.B = o; o = round4(o + C);
    r.G = o; o = round4(o + C * lg);
    r.total = o;
    return r;
}

// Workspace: per slot and head, the entry state h and the gradient of h_out ([dk][dv] each); Delta, Y and Z
// ([C][dv] each); the chunk record.  Each region starts on 16 bytes.
struct Ws {
    float *h, *dh, *D, *Y, *Z, *rec;
};

__host__ __device__ inline size_t round4z(size_t x) { return (x + 3) & ~(size_t)3; }

__host__ __device__ inline size_t ws_floats(long slots, int H, int C, int dk, int dv, bool perch) {
    const size_t st = round4z((size_t)slots * H * dk * dv), ch = round4z((size_t)slots * H * C * dv);
    return 2 * st + 3 * ch + (size_t)slots * H * rec_lay(C, dk, perch).total;
}

__host__ __device__ inline Ws carve_ws(float* base, long slots, int H, int C, int dk, int dv) {
    const size_t st = round4z((size_t)slots * H * dk * dv), ch = round4z((size_t)slots * H * C * dv);
    Ws w;
    w.h = base;
    w.dh = w.h + st;
    w.D = w.dh + st;
    w.Y = w.D + ch;
    w.Z = w.Y + ch;
    w.rec = w.Z + ch;
    return w;
}

// ---- steps shared by the kernels --------------------------------------------------------------------

// Load the chunk's K (and Q) rows, zero beyond d_k up to `width`, and rows >= L zero (beta = 0, g = 0 there,
// which leaves the state unchanged); the gate rows (stride lg) and beta.
// q and k are read at the key head: qk0 is the (token, key head) index of row 0, rows Hk apart.
template <typename Tin, bool PERCH, bool WITH_Q>
__device__ __forceinline__ void load_qk(const BwdArgs& a, size_t tok0, size_t qk0, int L, int width, int ldk, int lg,
                                        float* Qs, float* Ks, float* Gs, float* Bs) {
    const int C = a.C, dk = a.dk, H = a.H, Hk = a.HK();
    const Tin* q = static_cast<const Tin*>(a.q);
    const Tin* k = static_cast<const Tin*>(a.k);
    for (int idx = threadIdx.x; idx < C * width; idx += kThreads) {
        const int r = idx / width, c = idx % width;
        float kv = 0.f, qv = 0.f, gv = 0.f;
        if (r < L && c < dk) {
            const size_t tok = tok0 + (size_t)r * H, qt = qk0 + (size_t)r * Hk;
            kv = ld_f32<Tin>(k, qt * dk + c);
            if (WITH_Q) qv = ld_f32<Tin>(q, qt * dk + c);
            if (PERCH) gv = a.g[tok * dk + c];
        }
        Ks[r * ldk + c] = kv;
        if (WITH_Q) Qs[r * ldk + c] = qv;
        if (PERCH) Gs[r * lg + c] = gv;
    }
    for (int r = threadIdx.x; r < C; r += kThreads) {
        const bool in = r < L;
        Bs[r] = in ? a.beta[tok0 + (size_t)r * H] : 0.f;
        if (!PERCH) Gs[r] = in ? a.g[tok0 + (size_t)r * H] : 0.f;
    }
}

// Within-chunk prefix sum of the log gate, one channel per thread.
__device__ __forceinline__ void gate_prefix(float* Gs, int C, int gc, int lg) {
    for (int c = threadIdx.x; c < gc; c += kThreads) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) { acc += Gs[r * lg + c]; Gs[r * lg + c] = acc; }
    }
}

// KK (strictly lower), and with WITH_P the read matrix P (lower incl. the diagonal, scaled) and, for the scalar
// gate, Ex[r][s] = exp(G_r - G_s) (s <= r).  Exponents are formed only for s <= r, so no factor exceeds 1.  Rows
// are read four channels at a time (rows 16-byte aligned, stride = 4 mod 32 banks: no conflicts).
template <bool PERCH, bool WITH_P>
__device__ __forceinline__ void pair_products(const float* Qs, const float* Ks, const float* Gs, float* KK, float* Pm,
                                              float* Ex, int C, int dkp, int ldk, int lg, float scale) {
    for (int idx = threadIdx.x; idx < C * C; idx += kThreads) {
        const int r = idx / C, s = idx % C;
        float kk = 0.f, qk = 0.f, e0 = 0.f;
        if (s <= r) {
            for (int c = 0; c < dkp; c += 4) {
                const float4 ks = *reinterpret_cast<const float4*>(Ks + s * ldk + c);
                float4 kr = *reinterpret_cast<const float4*>(Ks + r * ldk + c);
                float4 qr = make_float4(0.f, 0.f, 0.f, 0.f);
                if (WITH_P) qr = *reinterpret_cast<const float4*>(Qs + r * ldk + c);
                if (PERCH) {
                    const float4 gr = *reinterpret_cast<const float4*>(Gs + r * lg + c);
                    const float4 gs = *reinterpret_cast<const float4*>(Gs + s * lg + c);
                    const float ex = expf(gr.x - gs.x), ey = expf(gr.y - gs.y);
                    const float ez = expf(gr.z - gs.z), ew = expf(gr.w - gs.w);
                    kr.x *= ex; kr.y *= ey; kr.z *= ez; kr.w *= ew;
                    qr.x *= ex; qr.y *= ey; qr.z *= ez; qr.w *= ew;
                }
                kk = fmaf(kr.x, ks.x, fmaf(kr.y, ks.y, fmaf(kr.z, ks.z, fmaf(kr.w, ks.w, kk))));
                if (WITH_P) qk = fmaf(qr.x, ks.x, fmaf(qr.y, ks.y, fmaf(qr.z, ks.z, fmaf(qr.w, ks.w, qk))));
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
            if (!PERCH && Ex) Ex[r * (C + 1) + s] = e0;
        }
    }
}

// ---- the chunk records ---------------------------------------------------------------------------------------

// Find the chunk of workspace slot `slot`: returns false for slots that hold a final state (or none).
__device__ __forceinline__ bool slot_chunk(const BwdArgs& a, long slot, long* n_out, long* ci_out) {
    if (!a.cu) {
        const long per = (a.T + a.C - 1) / a.C + 1;
        *n_out = slot / per;
        *ci_out = slot % per;
        return *ci_out < per - 1;
    }
    // the last sequence whose first slot is <= slot (first slots increase with n for ordered cu_seqlens)
    long lo = 0, hi = a.n_seqs - 1;
    while (lo < hi) {
        const long mid = (lo + hi + 1) / 2;
        long s0 = a.cu[mid];
        s0 = s0 < 0 ? 0 : (s0 > a.T ? a.T : s0);
        if (s0 / a.C + 2 * mid <= slot) lo = mid; else hi = mid - 1;
    }
    const Geo geo = chain_geo(a, lo);
    *n_out = lo;
    *ci_out = slot - geo.slot0;
    return *ci_out >= 0 && *ci_out < (geo.len + a.C - 1) / a.C;
}


// One CTA per (workspace slot, head); slots that hold a final state (or none) return at once.
template <typename Tin, bool PERCH, int CC>
__global__ void __launch_bounds__(kThreads) bwd_prep_kernel(const BwdArgs a, Ws ws) {
    extern __shared__ __align__(16) float smem[];
    const int dk = a.dk, H = a.H, W = 8 * walk_cpt(dk), ldk = W + 4, lg = PERCH ? ldk : 1, dkp = round4(dk);
    const Rec rc = rec_lay(CC, dk, PERCH);
    float* Qs = smem;
    float* Ks = Qs + CC * ldk;
    float* R = Ks + CC * ldk;
    float* Gs = R + rc.G;
    const long slot = blockIdx.x / H;
    const int hh = (int)(blockIdx.x % H);
    long n, ci;
    if (!slot_chunk(a, slot, &n, &ci)) return;
    const Geo geo = chain_geo(a, n);
    const int L = (int)min((long)CC, geo.len - ci * CC);
    const size_t tok0 = ((size_t)geo.b * a.T + geo.bos + ci * CC) * H + hh;
    const float scale = a.scale;
    const size_t qk0 = ((size_t)geo.b * a.T + geo.bos + ci * CC) * a.HK() + hh / (H / a.HK());
    load_qk<Tin, PERCH, true>(a, tok0, qk0, L, W, ldk, lg, Qs, Ks, Gs, R + rc.B);
    __syncthreads();
    gate_prefix(Gs, CC, PERCH ? dk : 1, lg);
    __syncthreads();
    pair_products<PERCH, true>(Qs, Ks, Gs, R + rc.KK, R + rc.P, nullptr, CC, dkp, ldk, lg, scale);
    __syncthreads();   // KK complete
    if (threadIdx.x < 32) {
        // warp 0: T = (I + A)^{-1}, A = diag(beta) KK strictly lower: column c by forward substitution on the unit
        // vector (thread c, the column in registers; its entries above row c are exact zeros, so the sums may start
        // at row 0).  Rows past the chunk's end have beta = 0, so T is the identity there.
        if (threadIdx.x < CC) {
            const int c = threadIdx.x;
            const float* KK = R + rc.KK;
            const float* Bv = R + rc.B;
            float* Tm = R + rc.T;
            float tc[CC];
#pragma unroll
            for (int r = 0; r < CC; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int q = 0; q < r; ++q) acc = fmaf(KK[r * (CC + 1) + q], tc[q], acc);
                tc[r] = r == c ? 1.f : (r > c ? -Bv[r] * acc : 0.f);
                Tm[r * (CC + 1) + c] = tc[r];
            }
        }
    } else {
        // the other warps meanwhile: scale Q*E, K*E, K*F and exp(G_L)
        for (int idx = threadIdx.x - 32; idx < CC * W; idx += kThreads - 32) {
            const int r = idx / W, c = idx % W;
            const float g = PERCH ? Gs[r * lg + c] : Gs[r];
            const float gl = PERCH ? Gs[(L - 1) * lg + c] : Gs[L - 1];
            const float e = expf(g), k = Ks[r * ldk + c];
            R[rc.QE + r * ldk + c] = scale * Qs[r * ldk + c] * e;
            R[rc.KE + r * ldk + c] = k * e;
            R[rc.KF + r * ldk + c] = k * expf(gl - g);
        }
        for (int c = threadIdx.x - 32; c < (PERCH ? W : 4); c += kThreads - 32)
            R[rc.EL + c] = expf(PERCH ? Gs[(L - 1) * lg + c] : Gs[L - 1]);
    }
    __syncthreads();
    float4* dst = reinterpret_cast<float4*>(ws.rec + ((size_t)slot * H + hh) * rc.total);
    const float4* src = reinterpret_cast<const float4*>(R);
    for (int i = threadIdx.x; i < rc.total / 4; i += kThreads) dst[i] = src[i];
}

// ---- the two walks -----------------------------------------------------------------------------------------

// Shared memory of the walk kernel, in floats: two record stages (the record up to G), the state tile, the V / dO
// tile, the Delta / Y tile, two mbarriers.
struct WalkLay {
    int st0, st1, S, V, D, bar, total;
};

__host__ __device__ inline WalkLay walk_lay(int C, int dk, bool perch) {
    const Rec rc = rec_lay(C, dk, perch);
    WalkLay l;
    int o = 0;
    l.st0 = o; o = round4(o + rc.G);
    l.st1 = o; o = round4(o + rc.G);
    l.S = o; o = round4(o + 8 * walk_cpt(dk) * kWS);
    l.V = o; o = round4(o + C * kWS);
    l.D = o; o = round4(o + C * kWS);
    l.bar = o; o = round4(o + 4);
    l.total = o;
    return l;
}

// Rows of the next chunk's [C][kWB] tile that this thread loads ahead (thread: columns lane and lane + 32, rows
// warp + 8 k); element 2 k + u is column lane + 32 u of row warp + 8 k.
template <typename T, int NV>
__device__ __forceinline__ void prefetch_rows(float (&v)[NV], const T* src, size_t tok0, int H, int dv, int j0, int bw,
                                              int L) {
    const int j = threadIdx.x & 31, r0 = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < NV / 2; ++k) {
        const int r = r0 + 8 * k;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int jj = j + 32 * u;
            v[2 * k + u] = (r < L && jj < bw) ? ld_f32<T>(src, (tok0 + (size_t)r * H) * dv + j0 + jj) : 0.f;
        }
    }
}

// Operand fragments of m16n8k8 (lane = 4 g + t), split into TF32 heads and tails for mma3_tf32.
// A (16 x 8) at (row, col) = (r0 + g [+ 8], k0 + t [+ 4]) of a row-major matrix with row stride ld.
__device__ __forceinline__ void frag_a(const float* M, int ld, int r0, int k0, int g, int t, uint32_t (&h)[4],
                                       uint32_t (&l)[4]) {
    split_tf32(M[(r0 + g) * ld + k0 + t], h[0], l[0]);
    split_tf32(M[(r0 + g + 8) * ld + k0 + t], h[1], l[1]);
    split_tf32(M[(r0 + g) * ld + k0 + t + 4], h[2], l[2]);
    split_tf32(M[(r0 + g + 8) * ld + k0 + t + 4], h[3], l[3]);
}
// A (16 x 8) = the transpose of a row-major matrix N: A(row m, col k) = N[k][m].
__device__ __forceinline__ void frag_at(const float* N, int ld, int m0, int k0, int g, int t, uint32_t (&h)[4],
                                        uint32_t (&l)[4]) {
    split_tf32(N[(k0 + t) * ld + m0 + g], h[0], l[0]);
    split_tf32(N[(k0 + t) * ld + m0 + g + 8], h[1], l[1]);
    split_tf32(N[(k0 + t + 4) * ld + m0 + g], h[2], l[2]);
    split_tf32(N[(k0 + t + 4) * ld + m0 + g + 8], h[3], l[3]);
}
// B (8 x 8) at (row, col) = (k0 + t [+ 4], n0 + g) of a row-major matrix, each element times s.
__device__ __forceinline__ void frag_b(const float* M, int ld, int k0, int n0, int g, int t, float s0, float s1,
                                       uint32_t (&h)[2], uint32_t (&l)[2]) {
    split_tf32(s0 * M[(k0 + t) * ld + n0 + g], h[0], l[0]);
    split_tf32(s1 * M[(k0 + t + 4) * ld + n0 + g], h[1], l[1]);
}

// The state (or state gradient) fragments of a walk -- rows c, columns j and j + 1 of each m16n8 tile -- to shared
// memory and to the workspace rows at dst (row stride d_v): 8-byte pairs where every row starts on 8 bytes (d_v
// even), else element by element.
template <int MTW>
__device__ __forceinline__ void store_state(const float (&acc)[MTW][8][4], float* S, float* dst, int cw, int g, int t4,
                                            int dk, int dv, int bw) {
    const bool pairs = (dv & 1) == 0;
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int c = cw + 16 * mt + g + 8 * h2, j = 8 * nt + 2 * t4;
                const float x0 = acc[mt][nt][2 * h2], x1 = acc[mt][nt][2 * h2 + 1];
                *reinterpret_cast<float2*>(S + c * kWS + j) = make_float2(x0, x1);
                if (c < dk) {
                    float* p = dst + (size_t)c * dv + j;
                    if (pairs && j + 1 < bw) {
                        *reinterpret_cast<float2*>(p) = make_float2(x0, x1);
                    } else {
                        if (j < bw) p[0] = x0;
                        if (j + 1 < bw) p[1] = x1;
                    }
                }
            }
}

// The forward walk: per chunk, store the entry state, Z and Delta.  The state tile h [channels][64 columns] lives in
// m16n8 accumulator fragments: warp w owns channels [w CPT, w CPT + CPT) (CPT / 16 row blocks) and all eight
// 8-column blocks.  Per chunk, on 3xTF32 warp MMAs:
//   Z = V - (K*E) h       rows of the chunk x the warp's 8 columns, over the channels
//   h <- diag(E_L) h + (K*F)^T Delta       the warp's channels x 64 columns, over the chunk's rows
template <typename Tin, bool PERCH, int CC, int CPT>
__device__ __forceinline__ void walk_forward(const BwdArgs& a, const Ws& ws, float* smem, long chain, int tile) {
    constexpr int MTW = CPT / 16, MTC = CC / 16;
    const int dk = a.dk, dv = a.dv, H = a.H, ldk = 8 * CPT + 4, dk8 = (dk + 7) & ~7;
    const Rec rc = rec_lay(CC, dk, PERCH);
    const WalkLay ly = walk_lay(CC, dk, PERCH);
    float* Hs = smem + ly.S;  float* Ds = smem + ly.D;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ly.bar);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const long n = chain / H;
    const int hh = (int)(chain % H);
    const Geo geo = chain_geo(a, n);
    const int j0 = tile * kWB, bw = min(kWB, dv - j0);
    const size_t sstride = (size_t)H * dk * dv, cstride = (size_t)H * CC * dv, rstride = (size_t)H * rc.total;
    const size_t sbase = (size_t)geo.slot0 * sstride + (size_t)hh * dk * dv + j0;
    const size_t cbase = (size_t)geo.slot0 * cstride + (size_t)hh * CC * dv + j0;
    const float* recs = ws.rec + ((size_t)geo.slot0 * H + hh) * rc.total;
    const long n_chunks = (geo.len + CC - 1) / CC;
    const Tin* v = static_cast<const Tin*>(a.v);
    const int cw = warp * CPT;          // first channel of this warp
    const int jz = 8 * warp + 2 * t4;   // this thread's two columns of Z

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // thread 0: chunk c's T, KE .. B into stage c & 1
    auto issue = [&](long c) {
        float* st = smem + ((c & 1) ? ly.st1 : ly.st0);
        const float* src = recs + (size_t)c * rstride;
        const uint32_t b = (uint32_t)(rc.G - rc.T) * 4u;
        mbar_arrive_expect_tx(&bars[c & 1], b);
        if (a.test_skip_record && c == 0) return;   // test: these bytes never arrive, the wait for them runs out
        bulk_g2s(st + rc.T, src + rc.T, b, &bars[c & 1]);
    };
    long issued = 0, waited = 0;
    if (tid == 0) {
        for (; issued < 2 && issued < n_chunks; ++issued) issue(issued);
    }
    float hacc[MTW][8][4];
    {
        const float* src = a.h0 ? a.h0 + ((size_t)n * H + hh) * dk * dv + j0 : nullptr;
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = cw + 16 * mt + g + 8 * (i >> 1), j = 8 * nt + 2 * t4 + (i & 1);
                    hacc[mt][nt][i] = (src && c < dk && j < bw) ? src[(size_t)c * dv + j] : 0.f;
                }
    }
    // V at this thread's Z positions (rows 16 m + g [+ 8], columns jz, jz + 1), loaded one chunk ahead
    float vpre[MTC][4];
    auto prefetch_v = [&](long c) {
        const size_t tok0 = ((size_t)geo.b * a.T + geo.bos + c * CC) * H + hh;
        const int L = (int)min((long)CC, geo.len - c * CC);
#pragma unroll
        for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 16 * mc + g + 8 * (i >> 1), j = jz + (i & 1);
                vpre[mc][i] = (r < L && j < bw) ? ld_f32<Tin>(v, (tok0 + (size_t)r * H) * dv + j0 + j) : 0.f;
            }
    };
    if (n_chunks > 0) prefetch_v(0);
    bool ok = true;
    for (long ci = 0;; ++ci) {
        // the state entering chunk ci (ci = n_chunks: the final state), to shared memory and the workspace
        store_state<MTW>(hacc, Hs, ws.h + sbase + (size_t)ci * sstride, cw, g, t4, dk, dv, bw);
        if (ci == n_chunks) break;
        const int L = (int)min((long)CC, geo.len - ci * CC);
        float vcur[MTC][4];
#pragma unroll
        for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
            for (int i = 0; i < 4; ++i) vcur[mc][i] = vpre[mc][i];
        if (ci + 1 < n_chunks) prefetch_v(ci + 1);
        const float* st = smem + ((ci & 1) ? ly.st1 : ly.st0);
        if (ok) ok = mbar_wait(&bars[ci & 1], (uint32_t)((ci >> 1) & 1), kWaitNs);
        ok = !__syncthreads_or(!ok);
        if (!ok) {
            if (tid == 0) atomicOr(&g_bwd_status, 1u);
            break;
        }
        waited = ci + 1;
        const float* KE = st + rc.KE;
        const float* KF = st + rc.KF;
        const float* Tm = st + rc.T;
        const float* EL = st + rc.EL;
        const float* Bs = st + rc.B;
        // Z = V - (K*E) h, then R = beta Z into Ds
        {
            float z[MTC][4];
#pragma unroll
            for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
                for (int i = 0; i < 4; ++i) z[mc][i] = 0.f;
            for (int k0 = 0; k0 < dk8; k0 += 8) {
                uint32_t bh[2], bl[2];
                frag_b(Hs, kWS, k0, 8 * warp, g, t4, 1.f, 1.f, bh, bl);
#pragma unroll
                for (int mc = 0; mc < MTC; ++mc) {
                    uint32_t ah[4], al[4];
                    frag_a(KE, ldk, 16 * mc, k0, g, t4, ah, al);
                    mma3_tf32(z[mc], ah, al, bh, bl);
                }
            }
#pragma unroll
            for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 16 * mc + g + 8 * (i >> 1), j = jz + (i & 1);
                    const float zz = vcur[mc][i] - z[mc][i];
                    if (r < L && j < bw) ws.Z[cbase + (size_t)ci * cstride + (size_t)r * dv + j] = zz;
                    Ds[r * kWS + j] = Bs[r] * zz;
                }
        }
        __syncwarp();
        // Delta = T R, T = (I + A)^{-1} from the record: each warp on its own 8 columns
        {
            float dl[MTC][4];
#pragma unroll
            for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
                for (int i = 0; i < 4; ++i) dl[mc][i] = 0.f;
#pragma unroll
            for (int k0 = 0; k0 < CC; k0 += 8) {
                uint32_t bh[2], bl[2];
                frag_b(Ds, kWS, k0, 8 * warp, g, t4, 1.f, 1.f, bh, bl);
#pragma unroll
                for (int mc = 0; mc < MTC; ++mc) {
                    uint32_t ah[4], al[4];
                    frag_a(Tm, CC + 1, 16 * mc, k0, g, t4, ah, al);
                    mma3_tf32(dl[mc], ah, al, bh, bl);
                }
            }
            __syncwarp();   // every lane has read R
#pragma unroll
            for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
                for (int i = 0; i < 4; ++i) Ds[(16 * mc + g + 8 * (i >> 1)) * kWS + jz + (i & 1)] = dl[mc][i];
        }
        __syncthreads();
        // store Delta; h <- diag(E_L) h + (K*F)^T Delta
        for (int idx = tid; idx < L * kWB; idx += kThreads) {
            const int r = idx / kWB, j = idx % kWB;
            if (j < bw) ws.D[cbase + (size_t)ci * cstride + (size_t)r * dv + j] = Ds[r * kWS + j];
        }
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) {
            const float e0 = EL[PERCH ? cw + 16 * mt + g : 0], e1 = EL[PERCH ? cw + 16 * mt + g + 8 : 0];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                hacc[mt][nt][0] *= e0; hacc[mt][nt][1] *= e0;
                hacc[mt][nt][2] *= e1; hacc[mt][nt][3] *= e1;
            }
        }
#pragma unroll
        for (int k0 = 0; k0 < CC; k0 += 8) {
            uint32_t ah[MTW][4], al[MTW][4];
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt) frag_at(KF, ldk, cw + 16 * mt, k0, g, t4, ah[mt], al[mt]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                uint32_t bh[2], bl[2];
                frag_b(Ds, kWS, k0, 8 * nt, g, t4, 1.f, 1.f, bh, bl);
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) mma3_tf32(hacc[mt][nt], ah[mt], al[mt], bh, bl);
            }
        }
        __syncthreads();   // every thread is done with this stage and with Hs, Ds
        if (tid == 0 && ci + 2 < n_chunks) {
            issue(ci + 2);
            ++issued;
        }
    }
    // stages issued but never waited on (after a timeout) must land before the CTA exits
    if (tid == 0)
        for (long c = waited; c < issued; ++c) mbar_wait(&bars[c & 1], (uint32_t)((c >> 1) & 1), kWaitNs);
}

// The backward walk: per chunk (last to first), store the gradient of h_out and Y; finally the gradient of the
// initial state.  Layout as in the forward walk; per chunk:
//   dDelta = P^T dO + (K*F) dh        rows x the warp's 8 columns
//   dh <- diag(E_L) dh + scale (Q*E)^T dO - (K*E)^T diag(beta) Y        the warp's channels x 64 columns
template <typename Tin, typename Tdo, bool PERCH, int CC, int CPT>
__device__ __forceinline__ void walk_backward(const BwdArgs& a, const Ws& ws, float* smem, long chain, int tile) {
    constexpr int MTW = CPT / 16, MTC = CC / 16, NV = CC * kWB / kThreads;
    const int dk = a.dk, dv = a.dv, H = a.H, ldk = 8 * CPT + 4, dk8 = (dk + 7) & ~7;
    const Rec rc = rec_lay(CC, dk, PERCH);
    const WalkLay ly = walk_lay(CC, dk, PERCH);
    float* dHs = smem + ly.S; float* Os = smem + ly.V;  float* Ys = smem + ly.D;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ly.bar);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const long n = chain / H;
    const int hh = (int)(chain % H);
    const Geo geo = chain_geo(a, n);
    const int j0 = tile * kWB, bw = min(kWB, dv - j0);
    const size_t sstride = (size_t)H * dk * dv, cstride = (size_t)H * CC * dv, rstride = (size_t)H * rc.total;
    const size_t sbase = (size_t)geo.slot0 * sstride + (size_t)hh * dk * dv + j0;
    const size_t cbase = (size_t)geo.slot0 * cstride + (size_t)hh * CC * dv + j0;
    const size_t own = ((size_t)n * H + hh) * dk * dv + j0;
    const float* recs = ws.rec + ((size_t)geo.slot0 * H + hh) * rc.total;
    const long n_chunks = (geo.len + CC - 1) / CC;
    const Tdo* dO = static_cast<const Tdo*>(a.dO);
    const int cw = warp * CPT;
    const int jz = 8 * warp + 2 * t4;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // thread 0: the record of the k-th chunk walked (chunk n_chunks - 1 - k) into stage k & 1
    auto issue = [&](long k) {
        float* st = smem + ((k & 1) ? ly.st1 : ly.st0);
        const float* src = recs + (size_t)(n_chunks - 1 - k) * rstride;
        const uint32_t b = (uint32_t)(rc.G - rc.P) * 4u;
        mbar_arrive_expect_tx(&bars[k & 1], b);
        if (a.test_skip_record && k == 0) return;   // test: these bytes never arrive, the wait for them runs out
        bulk_g2s(st + rc.P, src + rc.P, b, &bars[k & 1]);
    };
    long issued = 0, waited = 0;
    if (tid == 0) {
        for (; issued < 2 && issued < n_chunks; ++issued) issue(issued);
    }
    float dacc[MTW][8][4];
#pragma unroll
    for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = cw + 16 * mt + g + 8 * (i >> 1), j = 8 * nt + 2 * t4 + (i & 1);
                dacc[mt][nt][i] = (a.dhT && c < dk && j < bw) ? a.dhT[own + (size_t)c * dv + j] : 0.f;
            }
    float opre[NV];
    if (n_chunks > 0) {
        const long cl = n_chunks - 1;
        prefetch_rows<Tdo, NV>(opre, dO, ((size_t)geo.b * a.T + geo.bos + cl * CC) * H + hh, H, dv, j0, bw,
                               (int)min((long)CC, geo.len - cl * CC));
    }
    bool ok = true;
    for (long k = 0; k < n_chunks; ++k) {
        const long ci = n_chunks - 1 - k;
        const int L = (int)min((long)CC, geo.len - ci * CC);
        // the gradient of this chunk's h_out, to shared memory and the workspace
        store_state<MTW>(dacc, dHs, ws.dh + sbase + (size_t)ci * sstride, cw, g, t4, dk, dv, bw);
        {
            const int jl = tid & 31, r0 = tid >> 5;
#pragma unroll
            for (int q = 0; q < NV / 2; ++q) {
                Os[(r0 + 8 * q) * kWS + jl] = opre[2 * q];
                Os[(r0 + 8 * q) * kWS + jl + 32] = opre[2 * q + 1];
            }
        }
        if (ci > 0)
            prefetch_rows<Tdo, NV>(opre, dO, ((size_t)geo.b * a.T + geo.bos + (ci - 1) * CC) * H + hh, H, dv, j0, bw,
                                   CC);
        const float* st = smem + ((k & 1) ? ly.st1 : ly.st0);
        if (ok) ok = mbar_wait(&bars[k & 1], (uint32_t)((k >> 1) & 1), kWaitNs);
        ok = !__syncthreads_or(!ok);
        if (!ok) {
            if (tid == 0) atomicOr(&g_bwd_status, 1u);
            break;
        }
        waited = k + 1;
        const float* Tm = st + rc.T;
        const float* Pm = st + rc.P;
        const float* QE = st + rc.QE;
        const float* KE = st + rc.KE;
        const float* KF = st + rc.KF;
        const float* EL = st + rc.EL;
        const float* Bs = st + rc.B;
        // dDelta = P^T dO + (K*F) dh into Ys
        {
            float z[MTC][4];
#pragma unroll
            for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
                for (int i = 0; i < 4; ++i) z[mc][i] = 0.f;
#pragma unroll
            for (int k0 = 0; k0 < CC; k0 += 8) {
                uint32_t bh[2], bl[2];
                frag_b(Os, kWS, k0, 8 * warp, g, t4, 1.f, 1.f, bh, bl);
#pragma unroll
                for (int mc = 0; mc < MTC; ++mc) {
                    uint32_t ah[4], al[4];
                    frag_at(Pm, CC + 1, 16 * mc, k0, g, t4, ah, al);
                    mma3_tf32(z[mc], ah, al, bh, bl);
                }
            }
            for (int k0 = 0; k0 < dk8; k0 += 8) {
                uint32_t bh[2], bl[2];
                frag_b(dHs, kWS, k0, 8 * warp, g, t4, 1.f, 1.f, bh, bl);
#pragma unroll
                for (int mc = 0; mc < MTC; ++mc) {
                    uint32_t ah[4], al[4];
                    frag_a(KF, ldk, 16 * mc, k0, g, t4, ah, al);
                    mma3_tf32(z[mc], ah, al, bh, bl);
                }
            }
#pragma unroll
            for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
                for (int i = 0; i < 4; ++i) Ys[(16 * mc + g + 8 * (i >> 1)) * kWS + jz + (i & 1)] = z[mc][i];
        }
        __syncwarp();
        // Y = T^T dDelta (the solution of (I + A)^T Y = dDelta): each warp on its own 8 columns
        {
            float yl[MTC][4];
#pragma unroll
            for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
                for (int i = 0; i < 4; ++i) yl[mc][i] = 0.f;
#pragma unroll
            for (int k0 = 0; k0 < CC; k0 += 8) {
                uint32_t bh[2], bl[2];
                frag_b(Ys, kWS, k0, 8 * warp, g, t4, 1.f, 1.f, bh, bl);
#pragma unroll
                for (int mc = 0; mc < MTC; ++mc) {
                    uint32_t ah[4], al[4];
                    frag_at(Tm, CC + 1, 16 * mc, k0, g, t4, ah, al);
                    mma3_tf32(yl[mc], ah, al, bh, bl);
                }
            }
            __syncwarp();   // every lane has read dDelta
#pragma unroll
            for (int mc = 0; mc < MTC; ++mc)
#pragma unroll
                for (int i = 0; i < 4; ++i) Ys[(16 * mc + g + 8 * (i >> 1)) * kWS + jz + (i & 1)] = yl[mc][i];
        }
        __syncthreads();
        for (int idx = tid; idx < L * kWB; idx += kThreads) {
            const int r = idx / kWB, j = idx % kWB;
            if (j < bw) ws.Y[cbase + (size_t)ci * cstride + (size_t)r * dv + j] = Ys[r * kWS + j];
        }
        // dh <- diag(E_L) dh + scale (Q*E)^T dO - (K*E)^T diag(beta) Y
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) {
            const float e0 = EL[PERCH ? cw + 16 * mt + g : 0], e1 = EL[PERCH ? cw + 16 * mt + g + 8 : 0];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                dacc[mt][nt][0] *= e0; dacc[mt][nt][1] *= e0;
                dacc[mt][nt][2] *= e1; dacc[mt][nt][3] *= e1;
            }
        }
#pragma unroll
        for (int k0 = 0; k0 < CC; k0 += 8) {
            uint32_t qh[MTW][4], ql[MTW][4], kh[MTW][4], kl[MTW][4];
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt) {
                frag_at(QE, ldk, cw + 16 * mt, k0, g, t4, qh[mt], ql[mt]);
                frag_at(KE, ldk, cw + 16 * mt, k0, g, t4, kh[mt], kl[mt]);
            }
            const float nb0 = -Bs[k0 + t4], nb1 = -Bs[k0 + t4 + 4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                uint32_t oh[2], ol[2], yh[2], yl[2];
                frag_b(Os, kWS, k0, 8 * nt, g, t4, 1.f, 1.f, oh, ol);
                frag_b(Ys, kWS, k0, 8 * nt, g, t4, nb0, nb1, yh, yl);
#pragma unroll
                for (int mt = 0; mt < MTW; ++mt) {
                    mma3_tf32(dacc[mt][nt], qh[mt], ql[mt], oh, ol);
                    mma3_tf32(dacc[mt][nt], kh[mt], kl[mt], yh, yl);
                }
            }
        }
        __syncthreads();   // every thread is done with this stage and with dHs, Os, Ys
        if (tid == 0 && k + 2 < n_chunks) {
            issue(k + 2);
            ++issued;
        }
    }
    if (tid == 0)
        for (long c = waited; c < issued; ++c) mbar_wait(&bars[c & 1], (uint32_t)((c >> 1) & 1), kWaitNs);
    if (a.gh0 && ok) {
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = cw + 16 * mt + g + 8 * (i >> 1), j = 8 * nt + 2 * t4 + (i & 1);
                    if (c < dk && j < bw) a.gh0[own + (size_t)c * dv + j] = dacc[mt][nt][i];
                }
    }
}

// Blocks [0, n_walk) run the forward walk of (chain, tile) = divmod(block, n_tiles); blocks [n_walk, 2 n_walk)
// the backward walk.
template <typename Tin, typename Tdo, bool PERCH, int CC, int CPT>
__global__ void __launch_bounds__(kThreads) bwd_walk_kernel(const BwdArgs a, Ws ws, int n_tiles, long n_walk) {
    extern __shared__ __align__(16) float smem[];
    const long blk = blockIdx.x;
    if (blk < n_walk)
        walk_forward<Tin, PERCH, CC, CPT>(a, ws, smem, blk / n_tiles, (int)(blk % n_tiles));
    else
        walk_backward<Tin, Tdo, PERCH, CC, CPT>(a, ws, smem, (blk - n_walk) / n_tiles, (int)((blk - n_walk) % n_tiles));
}

// ---- the per-chunk gradients ---------------------------------------------------------------------------------

struct GradLay {
    int G, B, KK, AB, Ex, dP, dA, HB, TB, pbeta, us, red, total;
    // scalar gate: Ex holds exp(G_r - G_s) until the pair factors are formed, then dA e; AB holds dA e beta_r
    // inside the scratch region HB .. (after the tile loop): raw Q and K rows, then xo, hy, dd
    int Q, K, XO, HY, DD;
};

// The d_v tiles are double-buffered: the entry state and the exit-state gradient ([8 walk_cpt(dk)][kHS] each) and the
// dO, Delta, Y and Z tiles ([C][kHS] each, row-major), two of each.  kHS = 36 keeps the warp-MMA fragment loads
// conflict-free (4 g + t banks).  After the tile loop the same space holds raw Q, K and the state products.
constexpr int kHS = 36;

__host__ __device__ inline GradLay grad_lay(int C, int dk, bool perch) {
    const int ldk = 8 * walk_cpt(dk) + 4, lg = perch ? ldk : 1, cc = C * (C + 1), hr = 8 * walk_cpt(dk);
    GradLay l;
    int o = 0;
    l.G = o; o += C * lg; o = round4(o);
    l.B = o; o += C; o = round4(o);
    l.KK = o; o += cc; o = round4(o);
    l.AB = o; o += cc; o = round4(o);
    l.Ex = o; o += perch ? 0 : cc; o = round4(o);
    l.dP = o; o += cc; o = round4(o);
    l.dA = o; o += cc; o = round4(o);
    const int tiles = 4 * hr * kHS + 8 * C * kHS;
    l.Q = 0; l.K = round4(C * ldk); l.XO = l.K + round4(C * ldk); l.HY = l.XO + C * dk; l.DD = l.HY + C * dk;
    const int after = l.DD + C * dk;
    l.HB = o; o += tiles > after ? tiles : after; o = round4(o);
    l.TB = l.HB + 4 * hr * kHS;
    l.pbeta = o; o += C; o = round4(o);
    l.us = o; o += 2 * dk; o = round4(o);
    l.red = o; o += 2 * C + 1; o = round4(o);
    l.total = o;
    return l;
}

// One CTA per (workspace slot, head).  Per tile of d_v it adds the tile's terms (thread-owned accumulators);
// then, per (row r, channel c):
//   xo = (h dO_r)_c, hy = (h Y_r)_c, dd = (dh Delta_r)_c          (summed over all d_v)
//   SQ  = scale sum_{s<r} dP[r][s] k_sc e(r,s)         SAR = beta_r sum_{s<r} dA[r][s] k_sc e(r,s)
//   SKP = scale sum_{u>r} dP[u][r] q_uc e(u,r)         SAC = sum_{u>r} dA[u][r] beta_u k_uc e(u,r)
// with e(r,s) = exp(G_rc - G_sc), and the diagonal term D = scale dP[r][r];
//   dQ = scale E xo + SQ + D k_rc
//   dK = -beta E hy + F dd + SKP + D q_rc + SAR + SAC
//   gradient of G_r: q SQ - k SKP + k SAR - k SAC + scale E q xo - beta E k hy   (pb)
//                    and the write term F k dd, which reaches g_u for u > r only   (pw)
// The diagonal of P carries exp(0) and drops out of the gate gradient; so does the last write of the chunk,
// whose gate term and F term cancel.  Leaving both out in closed form (rather than forming and cancelling them)
// keeps the gate gradient accurate under strong decay.  Then
//   dg[u] = sum_{r >= u} pb[r] + sum_{s < u} pw[s] + us,   us = E_L sum_j dh[c][j] h[c][j],
//   dbeta_r = Y_r . Z_r + sum_{s<r} dA[r][s] KK[r][s],   dV = diag(beta) Y.
template <typename Tin, typename Tdo, bool PERCH, int CC, int NTW>
__global__ void __launch_bounds__(kThreads) bwd_grad_kernel(const BwdArgs a, Ws ws, int n_tiles) {
    extern __shared__ __align__(16) float smem[];
    constexpr int MT = CC / 16;       // 16-row blocks of the chunk
    constexpr int NP = (CC * CC + kThreads - 1) / kThreads;
    constexpr int NO = CC * kBV / kThreads;   // dO elements per thread and tile
    const int dk = a.dk, dv = a.dv, H = a.H, ldk = 8 * walk_cpt(dk) + 4, lg = PERCH ? ldk : 1, dkp = round4(dk);
    const GradLay ly = grad_lay(CC, dk, PERCH);
    const Rec rc = rec_lay(CC, dk, PERCH);
    const int hrows = 8 * NTW * (kThreads / 32);
    float* Gs = smem + ly.G;  float* Bs = smem + ly.B;
    float* KK = smem + ly.KK; float* WAB = smem + ly.AB;  float* Ex = smem + ly.Ex;
    float* dPm = smem + ly.dP; float* dAm = smem + ly.dA;
    float* pbeta = smem + ly.pbeta; float* us = smem + ly.us; float* red = smem + ly.red;
    // tile buffers b = 0, 1: state, state gradient, then the dO, Delta, Y, Z tiles
    auto Hb = [&](int b) { return smem + ly.HB + b * hrows * kHS; };
    auto dHb = [&](int b) { return smem + ly.HB + (2 + b) * hrows * kHS; };
    auto Tb = [&](int which, int b) { return smem + ly.TB + (2 * which + b) * CC * kHS; };   // 0 dO, 1 D, 2 Y, 3 Z
    const int tid = threadIdx.x;
    const long slot = blockIdx.x / H;
    const int hh = (int)(blockIdx.x % H);
    long n, ci;
    if (!slot_chunk(a, slot, &n, &ci)) return;
    const Geo geo = chain_geo(a, n);
    const long cs = ci * CC;
    const int L = (int)min((long)CC, geo.len - cs);
    const size_t tok0 = ((size_t)geo.b * a.T + geo.bos + cs) * H + hh;
    const int Hk = a.HK();
    const size_t qk0 = ((size_t)geo.b * a.T + geo.bos + cs) * Hk + hh / (H / Hk);
    const float scale = a.scale;
    const size_t sbase = ((size_t)slot * H + hh) * dk * dv, cbase = ((size_t)slot * H + hh) * CC * dv;
    const bool vec = (dv & 3) == 0;   // 16-byte copies need every row start on 16 bytes
    const Tdo* dO = static_cast<const Tdo*>(a.dO);

    // the tile's state rows and D, Y, Z rows into buffer b, as one cp.async group (plain loads where a 16-byte
    // copy does not apply: the tile's ragged edge, or d_v not a multiple of 4)
    auto issue_tile = [&](int t, int b) {
        const int j0 = t * kBV, bw = min(kBV, dv - j0);
        float* h_ = Hb(b);
        float* dh_ = dHb(b);
        for (int idx = tid; idx < hrows * 8; idx += kThreads) {
            const int c = idx >> 3, j = 4 * (idx & 7);
            const size_t o = sbase + (size_t)c * dv + j0 + j;
            if (vec && c < dk && j + 4 <= bw) {
                cp_async16(h_ + c * kHS + j, ws.h + o);
                cp_async16(dh_ + c * kHS + j, ws.dh + o);
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const bool in = c < dk && j + u < bw;
                    h_[c * kHS + j + u] = in ? ws.h[o + u] : 0.f;
                    dh_[c * kHS + j + u] = in ? ws.dh[o + u] : 0.f;
                }
            }
        }
        float* D_ = Tb(1, b);
        float* Y_ = Tb(2, b);
        float* Z_ = Tb(3, b);
        for (int idx = tid; idx < CC * 8; idx += kThreads) {
            const int r = idx >> 3, j = 4 * (idx & 7);
            const size_t o = cbase + (size_t)r * dv + j0 + j;
            if (vec && r < L && j + 4 <= bw) {
                cp_async16(D_ + r * kHS + j, ws.D + o);
                cp_async16(Y_ + r * kHS + j, ws.Y + o);
                cp_async16(Z_ + r * kHS + j, ws.Z + o);
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const bool in = r < L && j + u < bw;
                    D_[r * kHS + j + u] = in ? ws.D[o + u] : 0.f;
                    Y_[r * kHS + j + u] = in ? ws.Y[o + u] : 0.f;
                    Z_[r * kHS + j + u] = in ? ws.Z[o + u] : 0.f;
                }
            }
        }
        cp_async_commit();
    };
    // dO of tile t into registers (element k: row (tid + 256 k) / 32, column lane)
    float opre[NO];
    auto load_do = [&](int t) {
        const int j0 = t * kBV, bw = min(kBV, dv - j0);
#pragma unroll
        for (int k = 0; k < NO; ++k) {
            const int idx = tid + k * kThreads, r = idx / kBV, j = idx % kBV;
            opre[k] = (r < L && j < bw) ? ld_f32<Tdo>(dO, (tok0 + (size_t)r * H) * dv + j0 + j) : 0.f;
        }
    };
    if (n_tiles > 0) {
        issue_tile(0, 0);
        load_do(0);
    }

    // KK, P, the cumulative gate and beta from the chunk record
    {
        const float* rec = ws.rec + ((size_t)slot * H + hh) * rc.total;
        for (int i = tid; i < CC * (CC + 1); i += kThreads) KK[i] = rec[rc.KK + i];
        for (int i = tid; i < CC * lg; i += kThreads) Gs[i] = rec[rc.G + i];
        for (int i = tid; i < CC; i += kThreads) Bs[i] = rec[rc.B + i];
    }
    for (int c = tid; c < 2 * dk; c += kThreads) us[c] = 0.f;
    if (!PERCH) {
        __syncthreads();
        for (int idx = tid; idx < CC * CC; idx += kThreads) {
            const int r = idx / CC, s2 = idx % CC;
            Ex[r * (CC + 1) + s2] = s2 <= r ? expf(Gs[r] - Gs[s2]) : 0.f;
        }
    }

    float dp[NP], da[NP], ubeta = 0.f;
#pragma unroll
    for (int k = 0; k < NP; ++k) { dp[k] = 0.f; da[k] = 0.f; }
    // the state products xo = dO h^T, hy = Y h^T, dd = Delta dh^T ([C][channel]) on warp MMAs: warp w owns
    // channel blocks (w NTW + n) * 8, all rows; the accumulators stay in registers across the d_v tiles
    const int warp = tid >> 5, lane = tid & 31, fg = lane >> 2, ft = lane & 3;
    float acc[3][MT][NTW][4];
#pragma unroll
    for (int p = 0; p < 3; ++p)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int nn = 0; nn < NTW; ++nn)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[p][m][nn][i] = 0.f;
    for (int t = 0; t < n_tiles; ++t) {
        const int bf = t & 1, j0 = t * kBV, bw = min(kBV, dv - j0);
        float* Hs = Hb(bf);
        float* dHs = dHb(bf);
        float* O_ = Tb(0, bf);
        float* D_ = Tb(1, bf);
        float* Y_ = Tb(2, bf);
        float* Z_ = Tb(3, bf);
#pragma unroll
        for (int k = 0; k < NO; ++k) {
            const int idx = tid + k * kThreads;
            O_[(idx / kBV) * kHS + idx % kBV] = opre[k];
        }
        if (t + 1 < n_tiles) {
            issue_tile(t + 1, bf ^ 1);
            load_do(t + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        // dV = diag(beta) Y
        for (int idx = tid; idx < CC * kBV; idx += kThreads) {
            const int r = idx / kBV, j = idx % kBV;
            if (r < L && j < bw) a.gv[(tok0 + (size_t)r * H) * dv + j0 + j] = Bs[r] * Y_[r * kHS + j];
        }
        // dP = dO Delta^T, dA = -Y Delta^T (pairs owned by threads across the tiles)
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const int idx = tid + k * kThreads;
            if (idx < CC * CC) {
                const int r = idx / CC, s = idx % CC;
                if (s <= r) {
                    float x = dp[k], y = da[k];
                    const float4* o4 = reinterpret_cast<const float4*>(O_ + r * kHS);
                    const float4* y4 = reinterpret_cast<const float4*>(Y_ + r * kHS);
                    const float4* d4 = reinterpret_cast<const float4*>(D_ + s * kHS);
#pragma unroll
                    for (int q = 0; q < kBV / 4; ++q) {   // columns in order, four per 16-byte load
                        const float4 d = d4[q], o = o4[q], yv = y4[q];
                        x = fmaf(o.x, d.x, x); x = fmaf(o.y, d.y, x); x = fmaf(o.z, d.z, x); x = fmaf(o.w, d.w, x);
                        y = fmaf(yv.x, d.x, y); y = fmaf(yv.y, d.y, y); y = fmaf(yv.z, d.z, y); y = fmaf(yv.w, d.w, y);
                    }
                    dp[k] = x;
                    da[k] = y;
                }
            }
        }
        if (tid < CC) {
            const float4* y4 = reinterpret_cast<const float4*>(Y_ + tid * kHS);
            const float4* z4 = reinterpret_cast<const float4*>(Z_ + tid * kHS);
#pragma unroll
            for (int q = 0; q < kBV / 4; ++q) {
                const float4 yv = y4[q], zv = z4[q];
                ubeta = fmaf(yv.x, zv.x, ubeta); ubeta = fmaf(yv.y, zv.y, ubeta);
                ubeta = fmaf(yv.z, zv.z, ubeta); ubeta = fmaf(yv.w, zv.w, ubeta);
            }
        }
        // us[half dk + c] += sum over the tile's columns 16 half .. 16 half + 15 of dh[c][j] h[c][j]: one thread per
        // (channel, half), 16-byte loads (each pair always meets the same thread, so the sums need no atomics; the
        // halves are added after the last tile)
        for (int e = tid; e < 2 * dk; e += kThreads) {
            const int hf = e / dk, c = e - hf * dk;
            const float4* a4 = reinterpret_cast<const float4*>(dHs + c * kHS + 16 * hf);
            const float4* b4 = reinterpret_cast<const float4*>(Hs + c * kHS + 16 * hf);
            float x = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 u = a4[q], v = b4[q];
                x = fmaf(u.x, v.x, x); x = fmaf(u.y, v.y, x); x = fmaf(u.z, v.z, x); x = fmaf(u.w, v.w, x);
            }
            us[e] += x;
        }
        // the state products, 8 columns of the tile per step
#pragma unroll
        for (int k0 = 0; k0 < kBV; k0 += 8) {
            uint32_t bhh[NTW][2], bhl[NTW][2], bdh[NTW][2], bdl[NTW][2];
#pragma unroll
            for (int nn = 0; nn < NTW; ++nn) {
                const int c = (warp * NTW + nn) * 8 + fg;
                split_tf32(Hs[c * kHS + k0 + ft], bhh[nn][0], bhl[nn][0]);
                split_tf32(Hs[c * kHS + k0 + ft + 4], bhh[nn][1], bhl[nn][1]);
                split_tf32(dHs[c * kHS + k0 + ft], bdh[nn][0], bdl[nn][0]);
                split_tf32(dHs[c * kHS + k0 + ft + 4], bdh[nn][1], bdl[nn][1]);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                uint32_t oh[4], ol[4], yh[4], yl[4], dh4[4], dl4[4];
                frag_a(O_, kHS, 16 * m, k0, fg, ft, oh, ol);
                frag_a(Y_, kHS, 16 * m, k0, fg, ft, yh, yl);
                frag_a(D_, kHS, 16 * m, k0, fg, ft, dh4, dl4);
#pragma unroll
                for (int nn = 0; nn < NTW; ++nn) {
                    mma3_tf32(acc[0][m][nn], oh, ol, bhh[nn], bhl[nn]);
                    mma3_tf32(acc[1][m][nn], yh, yl, bhh[nn], bhl[nn]);
                    mma3_tf32(acc[2][m][nn], dh4, dl4, bdh[nn], bdl[nn]);
                }
            }
        }
        __syncthreads();   // this tile's buffers are free for the tile after next
    }
    // the tile space now holds raw q, k rows and the state products [C][dk] (channels below d_k only)
    float* Qs = smem + ly.HB + ly.Q;
    float* Ks = smem + ly.HB + ly.K;
    float* XO = smem + ly.HB + ly.XO;
    float* HY = smem + ly.HB + ly.HY;
    float* DD = smem + ly.HB + ly.DD;
    {
        const Tin* q = static_cast<const Tin*>(a.q);
        const Tin* k = static_cast<const Tin*>(a.k);
        for (int idx = tid; idx < CC * dkp; idx += kThreads) {
            const int r = idx / dkp, c = idx % dkp;
            const bool in = r < L && c < dk;
            const size_t off = (qk0 + (size_t)r * Hk) * dk + c;
            Qs[r * ldk + c] = in ? ld_f32<Tin>(q, off) : 0.f;
            Ks[r * ldk + c] = in ? ld_f32<Tin>(k, off) : 0.f;
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int nn = 0; nn < NTW; ++nn) {
            const int c = (warp * NTW + nn) * 8 + 2 * ft, r = 16 * m + fg;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int rr = r + 8 * (i >> 1), cc2 = c + (i & 1);
                if (cc2 < dk) {
                    XO[rr * dk + cc2] = acc[0][m][nn][i];
                    HY[rr * dk + cc2] = acc[1][m][nn][i];
                    DD[rr * dk + cc2] = acc[2][m][nn][i];
                }
            }
        }
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        const int idx = tid + k * kThreads;
        if (idx < CC * CC) {
            const int r = idx / CC, s = idx % CC, o = r * (CC + 1) + s;
            dAm[o] = (s < r) ? -da[k] : 0.f;
            if (PERCH) {
                dPm[o] = (s <= r) ? dp[k] : 0.f;
            } else {
                // the scalar gate's factors folded in once per pair: dP e, dA e (in place of e) and dA e beta_r,
                // with e = exp(G_r - G_s) (1 on the diagonal)
                const float e = Ex[o];
                dPm[o] = (s <= r) ? dp[k] * e : 0.f;
                const float ae = (s < r) ? -da[k] * e : 0.f;
                Ex[o] = ae;
                WAB[o] = ae * Bs[r];
            }
        }
    }
    if (tid < CC) pbeta[tid] = ubeta;
    __syncthreads();
    if (tid < dk) us[tid] = (us[tid] + us[dk + tid]) * expf(PERCH ? Gs[(L - 1) * lg + tid] : Gs[L - 1]);
    __syncthreads();

    // per (row, channel): dQ, dK written; the gate terms pb, pw kept in place of xo, hy
    for (int idx = tid; idx < L * dk; idx += kThreads) {
        const int r = idx / dk, c = idx % dk;
        const float gr = PERCH ? Gs[r * lg + c] : Gs[r];
        float sq = 0.f, sar = 0.f, skp = 0.f, sac = 0.f;
        if (PERCH) {
            for (int s = 0; s < r; ++s) {
                const float e = expf(gr - Gs[s * lg + c]);
                const float ke = Ks[s * ldk + c] * e;
                sq = fmaf(dPm[r * (CC + 1) + s], ke, sq);
                sar = fmaf(dAm[r * (CC + 1) + s], ke, sar);
            }
            for (int u = r + 1; u < L; ++u) {
                const float e = expf(Gs[u * lg + c] - gr);
                skp = fmaf(dPm[u * (CC + 1) + r], Qs[u * ldk + c] * e, skp);
                sac = fmaf(dAm[u * (CC + 1) + r] * Bs[u], Ks[u * ldk + c] * e, sac);
            }
        } else {   // the pair factors carry the gate (and beta_u for sac)
            for (int s = 0; s < r; ++s) {
                const float kv = Ks[s * ldk + c];
                sq = fmaf(dPm[r * (CC + 1) + s], kv, sq);
                sar = fmaf(Ex[r * (CC + 1) + s], kv, sar);
            }
            for (int u = r + 1; u < L; ++u) {
                skp = fmaf(dPm[u * (CC + 1) + r], Qs[u * ldk + c], skp);
                sac = fmaf(WAB[u * (CC + 1) + r], Ks[u * ldk + c], sac);
            }
        }
        sq *= scale;
        skp *= scale;
        sar *= Bs[r];
        const float gl = PERCH ? Gs[(L - 1) * lg + c] : Gs[L - 1];
        const float E = expf(gr), F = expf(gl - gr), br = Bs[r];
        const float qr = Qs[r * ldk + c], kr = Ks[r * ldk + c];
        const float dg0 = scale * dPm[r * (CC + 1) + r];
        const float xo = XO[idx], hy = HY[idx], dd = DD[idx];
        const float read = scale * E * xo;
        // grouped value heads: this value head's part, summed per key head afterwards
        const size_t off = a.gq_part ? (tok0 + (size_t)r * H) * dk + c : (qk0 + (size_t)r * Hk) * dk + c;
        (a.gq_part ? a.gq_part : a.gq)[off] = read + sq + dg0 * kr;
        (a.gk_part ? a.gk_part : a.gk)[off] = -br * E * hy + F * dd + skp + dg0 * qr + sar + sac;
        XO[idx] = qr * (read + sq) - kr * (br * E * hy + skp - sar + sac);   // pb
        HY[idx] = F * kr * dd;                                              // pw
    }
    for (int r = tid; r < L; r += kThreads) {
        float s = pbeta[r];
        for (int m = 0; m < r; ++m) s = fmaf(dAm[r * (CC + 1) + m], KK[r * (CC + 1) + m], s);
        a.gbeta[tok0 + (size_t)r * H] = s;
    }
    __syncthreads();
    // dg[u] = sum_{r >= u} pb[r] + sum_{s < u} pw[s] + us
    if (PERCH) {
        for (int c = tid; c < dk; c += kThreads) {
            float pre = us[c];
            for (int u = 0; u < L; ++u) {
                const float w = HY[u * dk + c];
                HY[u * dk + c] = pre;
                pre += w;
            }
            float acc = 0.f;
            for (int r = L - 1; r >= 0; --r) {
                acc += XO[r * dk + c];
                a.gg[(tok0 + (size_t)r * H) * dk + c] = acc + HY[r * dk + c];
            }
        }
    } else {
        // per row, the sums over the channels (one warp per row), then the two prefix sums over rows
        const int warp = tid >> 5, lane = tid & 31;
        for (int r = warp; r <= L; r += kThreads / 32) {
            float sb = 0.f, sw = 0.f;
            if (r < L) {
                for (int c = lane; c < dk; c += 32) { sb += XO[r * dk + c]; sw += HY[r * dk + c]; }
            } else {
                for (int c = lane; c < dk; c += 32) sb += us[c];
            }
            for (int o = 16; o > 0; o >>= 1) {
                sb += __shfl_xor_sync(0xffffffffu, sb, o);
                sw += __shfl_xor_sync(0xffffffffu, sw, o);
            }
            if (lane == 0) {
                if (r < L) { red[r] = sb; red[CC + r] = sw; } else { red[2 * CC] = sb; }
            }
        }
        __syncthreads();
        if (tid < 32) {
            const float sb = tid < L ? red[tid] : 0.f, sw = tid < L ? red[CC + tid] : 0.f;
            float rev = sb, fwd = sw;
            for (int o = 1; o < 32; o <<= 1) {
                const float x = __shfl_down_sync(0xffffffffu, rev, o);
                const float y = __shfl_up_sync(0xffffffffu, fwd, o);
                if (tid + o < 32) rev += x;
                if (tid >= o) fwd += y;
            }
            float ex = __shfl_up_sync(0xffffffffu, fwd, 1);   // exclusive: the inclusive sum of the lane before
            if (tid == 0) ex = 0.f;
            if (tid < L) a.gg[tok0 + (size_t)tid * H] = rev + ex + red[2 * CC];
        }
    }
}

// ---- launch ------------------------------------------------------------------------------------------------

__host__ __device__ inline size_t prep_smem_bytes(int C, int dk, bool perch) {
    return ((size_t)2 * C * (8 * walk_cpt(dk) + 4) + rec_lay(C, dk, perch).total) * sizeof(float);
}

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename Tin, typename Tdo, bool PERCH, int CC>
cudaError_t launch_c(const BwdArgs& a, cudaStream_t s) {
    const int n_tiles = (a.dv + kBV - 1) / kBV, n_wtiles = (a.dv + kWB - 1) / kWB;
    const long chains = (long)a.N() * a.H;
    if (chains == 0) return cudaSuccess;
    const long slots = workspace_slots(a.B, a.T, a.C, a.n_seqs, a.cu != nullptr);
    const Ws ws = carve_ws(a.ck, slots, a.H, a.C, a.dk, a.dv);
    const long n_walk = chains * n_wtiles;
    const size_t wbytes = (size_t)walk_lay(CC, a.dk, PERCH).total * sizeof(float);
    cudaError_t e;
    if ((long)a.B * a.T > 0) {
        const size_t pbytes = prep_smem_bytes(CC, a.dk, PERCH);
        auto pk = bwd_prep_kernel<Tin, PERCH, CC>;
        if ((e = set_smem(pk, pbytes)) != cudaSuccess) return e;
        pk<<<(unsigned)(slots * a.H), kThreads, pbytes, s>>>(a, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (walk_cpt(a.dk) == 16) {
        auto k = bwd_walk_kernel<Tin, Tdo, PERCH, CC, 16>;
        if ((e = set_smem(k, wbytes)) != cudaSuccess) return e;
        k<<<(unsigned)(2 * n_walk), kThreads, wbytes, s>>>(a, ws, n_wtiles, n_walk);
    } else {
        auto k = bwd_walk_kernel<Tin, Tdo, PERCH, CC, 32>;
        if ((e = set_smem(k, wbytes)) != cudaSuccess) return e;
        k<<<(unsigned)(2 * n_walk), kThreads, wbytes, s>>>(a, ws, n_wtiles, n_walk);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((long)a.B * a.T == 0) return cudaSuccess;
    const size_t gbytes = (size_t)grad_lay(CC, a.dk, PERCH).total * sizeof(float);
    if (walk_cpt(a.dk) == 16) {
        auto g = bwd_grad_kernel<Tin, Tdo, PERCH, CC, 2>;
        if ((e = set_smem(g, gbytes)) != cudaSuccess) return e;
        g<<<(unsigned)(slots * a.H), kThreads, gbytes, s>>>(a, ws, n_tiles);
    } else {
        auto g = bwd_grad_kernel<Tin, Tdo, PERCH, CC, 4>;
        if ((e = set_smem(g, gbytes)) != cudaSuccess) return e;
        g<<<(unsigned)(slots * a.H), kThreads, gbytes, s>>>(a, ws, n_tiles);
    }
    return cudaGetLastError();
}

template <typename Tin, typename Tdo, bool PERCH>
cudaError_t launch_gate(const BwdArgs& a, cudaStream_t s) {
    return a.C == 16 ? launch_c<Tin, Tdo, PERCH, 16>(a, s) : launch_c<Tin, Tdo, PERCH, 32>(a, s);
}

template <typename Tin>
cudaError_t launch_in(const BwdArgs& a, cudaStream_t s) {
    if (a.do_bf16)
        return a.per_channel ? launch_gate<Tin, __nv_bfloat16, true>(a, s) : launch_gate<Tin, __nv_bfloat16, false>(a, s);
    return a.per_channel ? launch_gate<Tin, float, true>(a, s) : launch_gate<Tin, float, false>(a, s);
}

// ---- the gate and beta activations around the backward ------------------------------------------------------

// log alpha and beta of every token from their raw logits (the activation of the forward, gate_act.cuh)
__global__ void bwd_act_apply_kernel(const float* x, const float* b, const GateAct act, float* g_out, float* beta_out,
                                     long n, int H) {
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int h = (int)(i % H);
        if (act.A_log) g_out[i] = act_gate(act, x[i], h);
        if (act.beta_sigmoid) beta_out[i] = act_beta(act, b[i]);
    }
}

__device__ __forceinline__ float sigmoid_f(float y) { return 1.f / (1.f + expf(-y)); }

// Per head h: dA_log[h] = sum_t dg_t log alpha_t and ddt_bias[h] = sum_t dg_t (-exp(A_log) sigmoid(x_t + dt_bias)),
// over every token, in a fixed order (thread-strided sums, then a fixed tree): the result does not depend on
// scheduling.  One CTA per head.
__global__ void __launch_bounds__(kThreads) bwd_act_head_kernel(const float* x, const float* g_act, const float* dg,
                                                                const GateAct act, float* dA_log, float* ddt,
                                                                long rows, int H) {
    __shared__ float red[2][kThreads];
    const int h = blockIdx.x, tid = threadIdx.x;
    const float e = expf(act.A_log[h]), dtb = act.dt_bias ? act.dt_bias[h] : 0.f;
    float sa = 0.f, sd = 0.f;
    for (long r = tid; r < rows; r += kThreads) {
        const long i = r * H + h;
        sa = fmaf(dg[i], g_act[i], sa);
        sd = fmaf(dg[i], -e * sigmoid_f(x[i] + dtb), sd);
    }
    red[0][tid] = sa;
    red[1][tid] = sd;
    __syncthreads();
    for (int o = kThreads / 2; o > 0; o >>= 1) {
        if (tid < o) {
            red[0][tid] += red[0][tid + o];
            red[1][tid] += red[1][tid + o];
        }
        __syncthreads();
    }
    if (tid == 0) {
        dA_log[h] = red[0][0];
        if (ddt) ddt[h] = red[1][0];
    }
}

// In place: dg <- dg (-exp(A_log) sigmoid(x + dt_bias)) (gradient of the raw gate logit) and
// dbeta <- dbeta * m sigmoid(b) (1 - sigmoid(b)) (gradient of the raw beta logit, m = 1 or 2).
__global__ void bwd_act_chain_kernel(const float* x, const float* b, const GateAct act, float* dg, float* dbeta,
                                     long n, int H) {
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int h = (int)(i % H);
        if (act.A_log) {
            const float dtb = act.dt_bias ? act.dt_bias[h] : 0.f;
            dg[i] *= -expf(act.A_log[h]) * sigmoid_f(x[i] + dtb);
        }
        if (act.beta_sigmoid) {
            const float s = sigmoid_f(b[i]);
            dbeta[i] *= (float)act.beta_sigmoid * s * (1.f - s);
        }
    }
}

// Grouped value heads: dq, dk of key head hk = the sum of its value heads hk G .. hk G + G - 1, in that order.
__global__ void bwd_group_sum_kernel(const float* part, float* out, long n_out, int Hk, int G, int dk) {
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n_out; i += (long)gridDim.x * blockDim.x) {
        const long c = i % dk, th = i / dk, t = th / Hk;
        const int hk = (int)(th % Hk);
        const float* p = part + ((t * Hk * G) + (long)hk * G) * dk + c;
        float s = 0.f;
        for (int u = 0; u < G; ++u) s += p[(long)u * dk];
        out[i] = s;
    }
}

}  // namespace

cudaError_t launch_bwd_group_sum(const BwdArgs& a, cudaStream_t s) {
    const int Hk = a.HK(), G = a.H / Hk;
    const long n_out = (long)a.B * a.T * Hk * a.dk;
    if (n_out == 0 || !a.gq_part) return cudaSuccess;
    const unsigned blocks = (unsigned)min((n_out + kThreads - 1) / kThreads, 152L * 16);
    bwd_group_sum_kernel<<<blocks, kThreads, 0, s>>>(a.gq_part, a.gq, n_out, Hk, G, a.dk);
    bwd_group_sum_kernel<<<blocks, kThreads, 0, s>>>(a.gk_part, a.gk, n_out, Hk, G, a.dk);
    return cudaGetLastError();
}

cudaError_t launch_bwd_act_apply(const float* x, const float* b, const GateAct& act, float* g_out, float* beta_out,
                                 long n, int H, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)min((n + kThreads - 1) / kThreads, 152L * 16);
    bwd_act_apply_kernel<<<blocks, kThreads, 0, s>>>(x, b, act, g_out, beta_out, n, H);
    return cudaGetLastError();
}

cudaError_t launch_bwd_act_post(const float* x, const float* b, const float* g_act, const GateAct& act, float* dg,
                                float* dbeta, float* dA_log, float* ddt, long rows, int H, cudaStream_t s) {
    if (act.gate()) {
        bwd_act_head_kernel<<<(unsigned)H, kThreads, 0, s>>>(x, g_act, dg, act, dA_log, ddt, rows, H);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const long n = rows * H;
    if (n == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)min((n + kThreads - 1) / kThreads, 152L * 16);
    bwd_act_chain_kernel<<<blocks, kThreads, 0, s>>>(x, b, act, dg, dbeta, n, H);
    return cudaGetLastError();
}

size_t bwd_smem_bytes(int C, int dk, bool per_channel) {
    const size_t w = (size_t)walk_lay(C, dk, per_channel).total * sizeof(float);
    const size_t g = (size_t)grad_lay(C, dk, per_channel).total * sizeof(float);
    const size_t p = prep_smem_bytes(C, dk, per_channel);
    return w > g ? (w > p ? w : p) : (g > p ? g : p);
}

// Chunk 16: smaller per-chunk tiles and triangular products; it measured faster than 32 on every workload timed.
int bwd_auto_chunk(int dk, bool per_channel) {
    for (int C : {16, 32})
        if (bwd_smem_bytes(C, dk, per_channel) <= kMaxSmemPerBlock) return C;
    return 0;
}

size_t bwd_act_offset(const BwdArgs& a) {
    const long slots = workspace_slots(a.B, a.T, a.C, a.n_seqs, a.cu != nullptr);
    return (ws_floats(slots, a.H, a.C, a.dk, a.dv, a.per_channel != 0) * sizeof(float) + 255) & ~(size_t)255;
}

// byte offset of the per-value-head dq, dk parts (grouped value heads only)
size_t bwd_part_offset(const BwdArgs& a) {
    return (bwd_act_offset(a) + (size_t)2 * a.B * a.T * a.H * sizeof(float) + 255) & ~(size_t)255;
}

// the walks' workspace, then room for the activated log alpha and beta ([B, T, H] fp32 each) and, with grouped
// value heads, the per-value-head dq and dk ([B, T, H, dk] fp32 each)
size_t bwd_workspace_bytes(const BwdArgs& a) {
    const size_t parts = a.HK() < a.H ? (size_t)2 * a.B * a.T * a.H * a.dk * sizeof(float) : 0;
    return bwd_part_offset(a) + parts;
}

cudaError_t bwd_read_and_clear_status(unsigned* value, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_bwd_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned));
}

cudaError_t launch_chunk_bwd(const BwdArgs& a, cudaStream_t s) {
    return a.bf16 ? launch_in<__nv_bfloat16>(a, s) : launch_in<float>(a, s);
}

}  // namespace gdn
