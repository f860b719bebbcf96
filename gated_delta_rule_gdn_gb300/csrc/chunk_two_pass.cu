// Two-pass chunkwise forward of the per-key-channel gate (Kimi Delta Attention) on tcgen05 tensor cores (sm_103a):
// bf16 q/k/v, d_k = d_v = 128, chunk C = 64, fp32 state, o in fp32 or bf16.  (The scalar gate has its own pair of
// kernels in chunk_gdn_tmem.cu.)
//
// The chunk algebra is "You Could Have Come Up With Kimi Delta Attention" (the chunkwise form: decays per key channel
// between tokens, the strictly lower key-key system, the read matrix with its diagonal), in the WY/UT form of
// "TileLang 实战：KDA 从零到一 -- Gated DeltaNet", §2.3, split the way "Gated Delta Network (GDN)", §4(b3)-(d) splits
// the scalar-gate chunk: every state-independent product first, then the serial state pass.  Per chunk of L <= C
// rows, with G_ic the within-chunk cumulative log gate of channel c:
//   A_ij = beta_i sum_c k_ic k_jc 2^(G_ic - G_jc)  (j < i)     P_ij = scale sum_c q_ic k_jc 2^(G_ic - G_jc)  (j <= i)
//   T = (I + A)^{-1},  W = T diag(beta) (K * 2^G),  U = T diag(beta) V,
//   Q^ = scale (Q * 2^G),  Ktilde = K * 2^(G_last - G),  gamma_C = 2^(G_last) per channel.
//
// Pass 1, chunk_intra_kernel<true>: one item per (chunk slot, head), one persistent CTA per SM.  A and P come from
// TF32 warp products over the channels, with the decays factored through 16-row block references (an exact per-term
// fallback covers large spreads); the blocked inverse solves T in place; one N = 256 tcgen05 product
// [T; T] [beta V | beta (K * 2^G)] gives U and W.  The record per item is 74,240 bytes, all fp16, already in the
// operand layouts of pass 2: [Q^; W] (32 KB, 128 x 128 K-major), Ktilde (16 KB), U (two d_v halves, 16 KB), P (8 KB)
// and gamma_C (512 B).
//
// Pass 2, chunk_state_kernel: one CTA per (sequence, head, 64-column d_v half), 8 warps; the fp32 state h = S^T tile
// sits in registers (thread = d_k row, 32 columns).  Per chunk, its record arrives by bulk copy (two-stage ring):
//   D3 = [Q^; W] h~ (M = 128, N = 64, K = 128): rows 0-63 Q^ h~, rows 64-127 W h~;  Delta = U - W h~ (fp16)
//   D4 = Ktilde^T Delta;  D5 = P Delta;  h <- diag(gamma_C) h + D4;  O = Q^ h~ + P Delta (written one chunk later).
// Slot of sequence n's chunk t: floor(start_n / C) + n + t.
//
// Every mbarrier wait is bounded (2 s); a wait that gives up sets a bit in the status word read by
// gdn_device_status, and the CTA skips the rest of its work, drains its copies, frees TMEM and exits.  The state
// kernel checks every value it writes to o and the final state and sets the non-finite bit when one is not finite
// (an fp16 intermediate past 65,504, or a non-finite input).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "tc_common.cuh"
#include "chunk_common.cuh"
#include "gate_act.cuh"
#include "chunk_wy_common.cuh"

namespace gdn {

__device__ unsigned g_tp_status;

// Scratch of the no-allocation entry point (gdn_chunk_fwd_noalloc): the two-pass workspace of any request that needs
// at most this much.  Every call on a device shares it.
constexpr size_t kStaticWorkspaceBytes = 64ull << 20;
__device__ __align__(256) unsigned char g_static_ws[kStaticWorkspaceBytes];

namespace {

using namespace tc;

constexpr int DVT = 64;

// workspace, per item
constexpr uint32_t WS_WQ = 32768;   // [Q^; W] fp16 K-major 128 x 128 (rows 0-63 Q^ = scale gamma Q, rows 64-127 W), two
                                    // 64-column slabs, 128-byte swizzle
constexpr uint32_t WS_KT = 16384;   // Ktilde fp16 [j][c] 64 x 128, two 64-column slabs, 128-byte swizzle
constexpr uint32_t WS_U = 16384;    // U fp16, two d_v halves of 64 rows x 64 columns (rows 128 B, 16-byte chunks swizzled)
constexpr uint32_t WS_P = 8192;     // P fp16 K-major 64 x 64, 128-byte swizzle
constexpr uint32_t WS_GC = 512;     // gamma_C per d_k row (fp32)
constexpr size_t WS_ITEM = (size_t)WS_WQ + WS_KT + WS_U + WS_P + WS_GC;

struct Ws {
    uint8_t* wq;
    uint8_t* kt;
    uint8_t* u;
    uint8_t* pp;
    float* gc;
};

__device__ __forceinline__ void set_status(unsigned bit) { atomicOr(&g_tp_status, bit); }

// ==================================================================== pass 1: per-chunk products
struct IntraParams {
    Geo geo;
    const float* g;
    const float* beta;
    float scale;
    long n_slots;
    Ws ws;
    GateAct act;   // the gate activation for the scalar gate only; beta for both
    int group;     // value heads per key head: q and k of item head h come from key head h / group
};

// shared memory of pass 1 (bytes from a 1024-aligned base)
constexpr uint32_t I_KQ = 0;        // [K; Q] rows, two K-slabs of 16 KB (K rows 0-63, Q rows 64-127)
constexpr uint32_t I_B2 = 32768;    // X = [beta V | beta gamma K], fp16 MN-major 64 x 256 in four 8 KB slabs
constexpr uint32_t I_A1 = 65536;    // [-; P] (rows 64-127, copied to the workspace) then [T; T], fp16 K-major 128 x 64
constexpr uint32_t I_B1 = 81920;    // the solve's scratch
constexpr uint32_t I_AM = 90112;    // fp32 A, then T in place (row stride TS)
constexpr uint32_t I_RT = I_B1;
constexpr uint32_t I_END = I_AM + 64 * TS * 4;
static_assert(32 * RS * 4 <= 8192, "the solve scratch must fit in the T buffer");
// KDA only: V tile, and the per-element gate factors (row stride ES floats)
constexpr int ES = 132;
constexpr uint32_t I_VB = I_END;                      // V, two 64-column bf16 slabs (TMA)
constexpr uint32_t I_EF = I_VB + 16384;               // the [64][128] fp32 gate tile (TMA), then
                                                      // E = exp(G - R_block), fp32 [64][ES]
constexpr uint32_t I_FF = I_EF + 64 * ES * 4;         // F = k exp(R_block - G) (fallback: log2 of the cumulative gate)

struct ISmall {
    uint64_t full_kq;         // K, Q of the item landed (TMA transaction bytes)
    uint64_t full_v;          // V (and the KDA gate tile) of the item landed
    uint64_t m0, m2;
    uint32_t tmem_base;
    uint32_t pad;
    float gbuf[C];            // g of the item (0 past the end; scalar gate)
    float bbuf[C];            // beta of the item (0 past the end)
    float lg[C];              // log2 of the within-chunk cumulative retention (scalar gate)
    float gam[C];             // gamma_j
    float kdec[C];            // gamma_C / gamma_j
    float gC;
};
// KDA: per-channel vectors of the gate (log2 units; R_a = cumulative gate at the end of 16-row block a - 1)
struct KSmall {
    float er[4][128];         // 2^R_a
    float espl[4][128];       // 2^(G_last - R_a)
    float dab[6][128];        // 2^(R_a - R_b) for b < a, pair a (a - 1) / 2 + b
    float lg63[128];          // G_last
    float p47[128], p63[128]; // the second half's partial sums at rows 47 and 63 (exchange between the halves)
    float tot1[128];          // the first half's total (row 31)
    int fast;                 // every block's spread is small enough for the factored products
};
constexpr uint32_t I_SMALL_KDA = I_FF + 64 * ES * 4;
constexpr uint32_t I_KSMALL = I_SMALL_KDA + ((sizeof(ISmall) + 127) & ~127u);   // 16-byte vector loads need alignment
constexpr uint32_t I_SMEM_KDA = I_KSMALL + sizeof(KSmall) + 1024;
static_assert(I_SMEM_KDA <= 227 * 1024, "KDA intra kernel shared memory");
// D2 = [T; T] [beta V | beta gamma K] = [U | W; U | W] spans all 256 columns (D0 is read before MMA2 is issued)
constexpr uint32_t I_TM_D2 = 0, I_TM_COLS = 256;
constexpr int I_THREADS = 256;
// largest |cumulative gate - block reference| (log2 units) for the factored KDA products: 2^100 keeps every
// factor and a 128-term sum of their products inside fp32
constexpr float KDA_SPREAD_MAX = 100.f;

// TMA loads of an item: K and Q as 2 x 2 boxes of 64 tokens x 64 columns; V as two boxes (GDN: into X's V slabs,
// KDA: into its own tile, with the fp32 gate tile into X).
__device__ __forceinline__ void intra_issue_kq(uint8_t* smem, ISmall& S, const CUtensorMap* mq, const CUtensorMap* mk,
                                               const Item& x, int group) {
    const int row = (int)x.row, hk = x.h / group;
    mbar_arrive_expect_tx(&S.full_kq, 32768);
    uint8_t* kq = smem + I_KQ;
    tma_load_3d(kq, mk, &S.full_kq, 0, hk, row);
    tma_load_3d(kq + 8192, mq, &S.full_kq, 0, hk, row);
    tma_load_3d(kq + 16384, mk, &S.full_kq, 64, hk, row);
    tma_load_3d(kq + 16384 + 8192, mq, &S.full_kq, 64, hk, row);
}
template <bool KDA>
__device__ __forceinline__ void intra_issue_v(uint8_t* smem, ISmall& S, const CUtensorMap* mv, const CUtensorMap* mg,
                                              const Item& x) {
    const int row = (int)x.row;
    mbar_arrive_expect_tx(&S.full_v, KDA ? 16384 + 32768 : 16384);
    uint8_t* vb = smem + (KDA ? I_VB : I_B2);   // KDA: the gate tile goes to the E table's place
    tma_load_3d(vb, mv, &S.full_v, 0, x.h, row);
    tma_load_3d(vb + 8192, mv, &S.full_v, 64, x.h, row);
    if (KDA) tma_load_3d(smem + I_EF, mg, &S.full_v, 0, x.h, row);
}

// g (scalar gate only) and beta of an item (0 past its end): lane l holds tokens l and l + 32
template <bool KDA>
__device__ __forceinline__ void intra_load_gb(const IntraParams& p, const Item& x, int lane, float (&g)[2],
                                              float (&b)[2]) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int r = lane + 32 * k;
        const size_t tok = (size_t)(x.row + r) * p.geo.H + x.h;
        g[k] = (!KDA && r < x.L) ? act_gate(p.act, __ldg(p.g + tok), x.h) : 0.f;
        b[k] = r < x.L ? act_beta(p.act, __ldg(p.beta + tok)) : 0.f;
    }
}

__device__ __forceinline__ uint4 scale_chunk_h(const float (&f)[8], float s, uint32_t m) {
    return make_uint4(pack_h2(f[0] * s, f[1] * s) & m, pack_h2(f[2] * s, f[3] * s) & m, pack_h2(f[4] * s, f[5] * s) & m,
                      pack_h2(f[6] * s, f[7] * s) & m);
}
__device__ __forceinline__ uint4 scale_chunk_hv(const float (&f)[8], const float (&s)[8], uint32_t m) {
    return make_uint4(pack_h2(f[0] * s[0], f[1] * s[1]) & m, pack_h2(f[2] * s[2], f[3] * s[3]) & m,
                      pack_h2(f[4] * s[4], f[5] * s[5]) & m, pack_h2(f[6] * s[6], f[7] * s[7]) & m);
}
__device__ __forceinline__ void ld_f8(const float* p, float (&f)[8]) {
    const float4 a = ld4(p), b = ld4(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
// one bf16 element (row r, column c) of a [rows][128] tile stored as two 128-byte-swizzled 64-column slabs
__device__ __forceinline__ float ld_bf16_sw(const uint8_t* base, int r, int c) {
    const uint16_t u = *reinterpret_cast<const uint16_t*>(base + (c >> 6) * 16384 + sw128_off(r, c & 63));
    return __uint_as_float((uint32_t)u << 16);
}

// KDA: within-chunk cumulative gate per channel (thread c < 128 owns channel c), its 16-row block references
// and the factors of the factored K K^T / Q K^T products:
//   E[i][c] = 2^(G_ic - R_a),  F[i][c] = k_ic 2^(R_a - G_ic)   (i in block a; R_a = G at the end of block a - 1,
//   R_0 = 0; F carries the key itself, the column operand of the products and the decayed key of the record)
// The fast path needs every gate <= 0 (G non-increasing: E <= 1, F <= 2^(block spread)) and every block spread
// <= KDA_SPREAD_MAX.  Otherwise F keeps G itself and the products are formed exactly, one exponential per term.
// Also writes gamma_C.  The gate tile sits where E goes: every thread reads its 32 gates before any writes E.
__device__ void kda_gate_tables(uint8_t* smem, KSmall& K, int L, float* gc_out, int tid) {
    const float LOG2E = 1.4426950408889634f;
    // thread (half, c): channel c, rows 32 half .. 32 half + 31; the second half's sums start at row 32
    const int c = tid & 127, half = tid >> 7, i0 = 32 * half;
    const float* gt = reinterpret_cast<const float*>(smem + I_EF);
    float* E = reinterpret_cast<float*>(smem + I_EF);
    float* F = reinterpret_cast<float*>(smem + I_FF);
    bool fine = true;
    float part[32];
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float gi = i0 + i < L ? gt[(i0 + i) * 128 + c] : 0.f;
        fine = fine && gi <= 0.f;   // retention <= 1: every factor below stays <= 1 or <= the block spread
        acc += gi;
        part[i] = acc * LOG2E;
    }
    __syncthreads();   // the gate tile is read
    // block references relative to this half's start: R_{2 half} = 0, R_{2 half + 1} = part[15]
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
        const float R = bb == 0 ? 0.f : part[15];
        fine = fine && R - part[16 * bb + 15] <= KDA_SPREAD_MAX;
#pragma unroll
        for (int i = 16 * bb; i < 16 * bb + 16; ++i) {
            E[(i0 + i) * ES + c] = ex2(part[i] - R);
            F[(i0 + i) * ES + c] = ld_bf16_sw(smem + I_KQ, i0 + i, c) * ex2(R - part[i]);
        }
    }
    if (half == 0) K.tot1[c] = part[31];
    else {
        K.p47[c] = part[15];
        K.p63[c] = part[31];
    }
    const bool fast = __syncthreads_and(fine) != 0;
    const float t1 = K.tot1[c];
    if (!fast) {   // the exact path keeps the absolute cumulative gate (log2) in F
#pragma unroll
        for (int i = 0; i < 32; ++i) F[(i0 + i) * ES + c] = part[i] + (half ? t1 : 0.f);
    }
    if (half == 0) {
        const float R[4] = {0.f, part[15], t1, t1 + K.p47[c]};
        const float Gl = t1 + K.p63[c];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            K.er[a][c] = ex2(R[a]);
            K.espl[a][c] = ex2(Gl - R[a]);
#pragma unroll
            for (int b = 0; b < a; ++b) K.dab[a * (a - 1) / 2 + b][c] = ex2(R[a] - R[b]);
        }
        K.lg63[c] = Gl;
        __stcg(gc_out + c, ex2(Gl));
        if (c == 0) K.fast = fast ? 1 : 0;
    }
}

// The 32 channels a lane quad t reduces over: the 8-channel chunks t, t + 4, t + 8, t + 12 (interleaved so that the
// 16-byte loads of a quarter-warp fall in distinct bank groups).  Row r of a bf16 [rows][128] tile stored as two
// 128-byte-swizzled 64-column slabs, as fp32:
__device__ __forceinline__ void ld_bf16_chunks(const uint8_t* base, int r, int t, float (&f)[32]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int cidx = t + 4 * u;
        float x[8];
        bf16x8_to_f32(ld16(base + (cidx >> 3) * 16384 + r * 128 + (((cidx & 7) ^ (r & 7)) << 4)), x);
#pragma unroll
        for (int k = 0; k < 8; ++k) f[8 * u + k] = x[k];
    }
}
// the same channels of an fp32 row
__device__ __forceinline__ void ld_f32_chunks(const float* row, int t, float (&f)[32]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float4 v0 = ld4(row + 8 * (t + 4 * u)), v1 = ld4(row + 8 * (t + 4 * u) + 4);
        f[8 * u] = v0.x; f[8 * u + 1] = v0.y; f[8 * u + 2] = v0.z; f[8 * u + 3] = v0.w;
        f[8 * u + 4] = v1.x; f[8 * u + 5] = v1.y; f[8 * u + 6] = v1.z; f[8 * u + 7] = v1.w;
    }
}

// KDA, fast path: A = diag(beta)(K K^T with per-channel decays) strictly lower -> Am (fp32) and P = scale (Q K^T with
// decays) lower incl. the diagonal -> A1 rows 64-127.  TF32 warp MMAs over the 128
// channels, with the channel (reduction) order permuted so that lane quad t owns the 32 channels of ld_bf16_chunks:
// step ks reduces over its channels 2 ks and 2 ks + 1 (the same permutation on both operands leaves the sum alone),
// which makes every operand load a 16-byte vector.  For row block a against column block b <= a:
//   row operand x_ic 2^(G_ic - R_a) = x_ic E_ic;   column operand k_jc 2^(R_a - G_jc) =
//   F_jc (b = a),   F_jc 2^(R_a - R_b) (b < a; F_jc <= |k_jc| 2^(block spread), 2^(R_a - R_b) <= 1).
// Warp w: product op = w % 2 (K or Q rows), row blocks {0, 3} or {1, 2} ((w / 2) % 2), 8-column half nt = w / 4 of
// every column block: five 16 x 8 output tiles per warp.
__device__ void kda_products_fast(uint8_t* smem, const KSmall& K, const float* bb, float scale, int warp, int lane) {
    const int op = warp & 1, grp = (warp >> 1) & 1, nt = warp >> 2;
    const int g8 = lane >> 2, t4 = lane & 3;
    const float* E = reinterpret_cast<const float*>(smem + I_EF);
    const float* F = reinterpret_cast<const float*>(smem + I_FF);
    const uint8_t* xb = smem + I_KQ + op * 8192;     // K or Q rows
    float* Am = reinterpret_cast<float*>(smem + I_AM);
    uint8_t* a1 = smem + I_A1;
#pragma unroll 1
    for (int ai = 0; ai < 2; ++ai) {
        const int a = grp == 0 ? 3 * ai : 1 + ai;    // {0, 3} or {1, 2}: five column blocks either way
        const int r0 = 16 * a + g8, r1 = r0 + 8;
        uint32_t afr[16][4];
        {
            float x0[32], x1[32], e[32];
            ld_bf16_chunks(xb, r0, t4, x0);
            ld_bf16_chunks(xb, r1, t4, x1);
            ld_f32_chunks(E + r0 * ES, t4, e);
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                afr[ks][0] = to_tf32(x0[2 * ks] * e[2 * ks]);
                afr[ks][2] = to_tf32(x0[2 * ks + 1] * e[2 * ks + 1]);
            }
            ld_f32_chunks(E + r1 * ES, t4, e);
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                afr[ks][1] = to_tf32(x1[2 * ks] * e[2 * ks]);
                afr[ks][3] = to_tf32(x1[2 * ks + 1] * e[2 * ks + 1]);
            }
        }
        const float s0 = op == 0 ? bb[r0] : scale, s1 = op == 0 ? bb[r1] : scale;
#pragma unroll 1
        for (int b = 0; b <= a; ++b) {
            const int j = 16 * b + 8 * nt + g8;
            float f[32];
            ld_f32_chunks(F + j * ES, t4, f);
            if (b < a) {   // 2^(R_a - G_j) = F_j 2^(R_a - R_b); where the second factor underflows the product is < 2^-26
                float dd[32];
                ld_f32_chunks(K.dab[a * (a - 1) / 2 + b], t4, dd);
#pragma unroll
                for (int q = 0; q < 32; ++q) f[q] *= dd[q];
            }
            float d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};   // two independent chains
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                const uint32_t b0 = to_tf32(f[2 * ks]), b1 = to_tf32(f[2 * ks + 1]);
                float (&acc)[4] = (ks & 1) ? d2 : d;
                asm volatile(
                    "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                    "{%0, %1, %2, %3};"
                    : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3])
                    : "r"(afr[ks][0]), "r"(afr[ks][1]), "r"(afr[ks][2]), "r"(afr[ks][3]), "r"(b0), "r"(b1));
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) d[q] += d2[q];
            const int cc = 16 * b + 8 * nt + 2 * t4;
            if (op == 0) {
                // A = beta_i (K K^T)_ij for j < i
                *reinterpret_cast<float2*>(Am + r0 * TS + cc) =
                    make_float2(cc < r0 ? s0 * d[0] : 0.f, cc + 1 < r0 ? s0 * d[1] : 0.f);
                *reinterpret_cast<float2*>(Am + r1 * TS + cc) =
                    make_float2(cc < r1 ? s1 * d[2] : 0.f, cc + 1 < r1 ? s1 * d[3] : 0.f);
            } else {
                // P = scale (Q K^T)_ij for j <= i
                *reinterpret_cast<uint32_t*>(a1 + sw128_off(64 + r0, cc)) =
                    pack_h2(cc <= r0 ? s0 * d[0] : 0.f, cc + 1 <= r0 ? s0 * d[1] : 0.f);
                *reinterpret_cast<uint32_t*>(a1 + sw128_off(64 + r1, cc)) =
                    pack_h2(cc <= r1 ? s1 * d[2] : 0.f, cc + 1 <= r1 ? s1 * d[3] : 0.f);
            }
        }
        if (nt != 0) continue;
        // zeros above the diagonal blocks: A inside the 32 x 32 diagonal blocks (what the solve reads), P everywhere
        if (op == 0) {
            if ((a & 1) == 0) {
                const int zr = 16 * a + (lane >> 1), zc = 16 * (a + 1) + 8 * (lane & 1);
                *reinterpret_cast<float4*>(Am + zr * TS + zc) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4*>(Am + zr * TS + zc + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        } else {
            for (int e = lane; e < (3 - a) * 16 * 2; e += 32) {   // 16 rows x (3 - a) blocks x two 8-column chunks
                const int zr = 16 * a + (e & 15), zc = 16 * (a + 1) + 8 * (e >> 4);
                st16(a1 + sw128_off(64 + zr, zc), 0u, 0u, 0u, 0u);
            }
        }
    }
}

// KDA, fallback: the same A and P, every term with its own exponential of the gate difference
// (G in log2 units is in F).  Exact for any gate; used only when some block's spread is too large.
__device__ void kda_products_direct(uint8_t* smem, const float* bb, float scale, int tid) {
    const float* G = reinterpret_cast<const float*>(smem + I_FF);
    const uint8_t* kb = smem + I_KQ;
    const uint8_t* qb = smem + I_KQ + 8192;
    float* Am = reinterpret_cast<float*>(smem + I_AM);
    uint8_t* a1 = smem + I_A1;
    for (int e = tid; e < 64 * 64; e += I_THREADS) {
        const int i = e >> 6, j = e & 63;
        float ak = 0.f, aq = 0.f;
        if (j <= i) {
            for (int c = 0; c < 128; ++c) {
                const float w = ex2(G[i * ES + c] - G[j * ES + c]) * ld_bf16_sw(kb, j, c);
                ak = fmaf(ld_bf16_sw(kb, i, c), w, ak);
                aq = fmaf(ld_bf16_sw(qb, i, c), w, aq);
            }
        }
        Am[i * TS + j] = j < i ? bb[i] * ak : 0.f;
        *reinterpret_cast<__half*>(a1 + sw128_off(64 + i, j)) = __float2half_rn(j <= i ? scale * aq : 0.f);
    }
}

// Per item (per-channel gate): [A] its tiles have landed (K and Q; V; the fp32 gate tile, in the E table's place);
// [B] the gate tables (E, F, the 16-row block references); A and [I; P] from the factored warp products; X =
// [beta V | beta 2^G K] in shared memory, Ktilde and Q^ with their per-element decays straight to the workspace.
// [C] K, Q, V, E and F are dead: the next item's tiles are loaded, a whole solve ahead of their use; P to the
// workspace; the solve; [T; T] in fp16; MMA2 = [T; T] X = [U | W; U | W]; the epilogue writes U and W to the
// workspace.
template <bool KDA>
__global__ void __launch_bounds__(I_THREADS, KDA ? 1 : 2)
chunk_intra_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_g,
                   const IntraParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    ISmall& S = *reinterpret_cast<ISmall*>(smem + I_SMALL_KDA);
    KSmall& KS = *reinterpret_cast<KSmall*>(smem + I_KSMALL);   // KDA only
    float* Am = reinterpret_cast<float*>(smem + I_AM);
    float* Rt = reinterpret_cast<float*>(smem + I_RT);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3;                       // TMEM lane quarter of this warp
    const int pw = warp >> 2;                      // which of the two warps on this quarter (64-column half)
    const bool leader = (tid == 0);
    const bool loader = (tid == 64);
    const int H = p.geo.H;
    const float LOG2E = 1.4426950408889634f;
    (void)LOG2E;
    griddep_launch_dependents();   // the state kernel may take SMs as this grid's CTAs retire

    if (warp == 0) {
        tmem_alloc(&S.tmem_base, I_TM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(&S.full_kq, 1);
        mbar_init(&S.full_v, 1);
        mbar_init(&S.m0, 1);
        mbar_init(&S.m2, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);

    const int ds = (int)(gridDim.x / H), dh = (int)(gridDim.x % H);
    const long first = p.n_slots * H - 1 - (long)blockIdx.x;
    Cursor cur{first / H, (int)(first % H), p.geo.N() - 1};
    Item x;
    bool have = cursor_next_valid(p.geo, cur, ds, dh, x);
    float ng[2] = {0.f, 0.f}, nb[2] = {0.f, 0.f};   // g, beta of the next item (warp 1, in flight)
    uint32_t kq_issued = 0, kq_waited = 0, v_issued = 0, v_waited = 0;   // loader's count of load phases
    if (have) {
        if (loader) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            if (KDA) prefetch_tmap(&tmap_g);
            intra_issue_kq(smem, S, &tmap_q, &tmap_k, x, p.group);
            intra_issue_v<KDA>(smem, S, &tmap_v, &tmap_g, x);
            kq_issued = v_issued = 1;
        }
        if (warp == 1) {
            float gg[2], bb[2];
            intra_load_gb<KDA>(p, x, lane, gg, bb);
            S.gbuf[lane] = gg[0];
            S.gbuf[lane + 32] = gg[1];
            S.bbuf[lane] = bb[0];
            S.bbuf[lane + 32] = bb[1];
        }
    }
    bool ok = true;
    uint32_t ic = 0;   // items done by this CTA: the parity of every barrier phase
    const Ws& ws = p.ws;
    while (have) {
        const Item it = x;
        Cursor nc = cur;
        cursor_step(nc, ds, dh, H);
        Item nx;
        const bool have_next = cursor_next_valid(p.geo, nc, ds, dh, nx);
        const uint32_t par = ic & 1;
        const int L = it.L;
        __syncthreads();   // [A] g and beta of this item are in shared memory; the previous item is retired
        if (warp == 1) {
            if (have_next) intra_load_gb<KDA>(p, nx, lane, ng, nb);
        }
        if (ok) ok = mbar_wait(&S.full_kq, par, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && tid == 0) set_status(1u);
        if (ok && loader) kq_waited = ic + 1;
            if (ok) ok = mbar_wait(&S.full_v, par, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && tid == 0) set_status(2u);
            if (ok && loader) v_waited = ic + 1;
            if (lane == 0) bulk_wait_read();   // the previous item's staging rows (F, A1) have been read
            __syncthreads();                   // ... by every warp's copies, before any thread writes F
            // [B] the gate tables (contains the barrier that decides the fast path)
            kda_gate_tables(smem, KS, ok ? L : 0, ws.gc + (size_t)it.it * 128, tid);
            __syncthreads();
            const bool fast = KS.fast != 0;
            if (ok) {
                if (fast) kda_products_fast(smem, KS, S.bbuf, p.scale, warp, lane);
                else kda_products_direct(smem, S.bbuf, p.scale, tid);
            }
            // X = [beta V | beta 2^G K], Ktilde = 2^(G_last - G) K and Q^ = scale 2^G Q (coalesced, as in the scalar-gate
            // path)
            if (ok) {
                const float* E = reinterpret_cast<const float*>(smem + I_EF);
                const float* F = reinterpret_cast<const float*>(smem + I_FF);
                uint8_t* kt = ws.kt + (size_t)it.it * WS_KT;
                uint8_t* wq = ws.wq + (size_t)it.it * WS_WQ;
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    const int e = tid + 256 * cc, slab = e >> 9, r = (e >> 3) & 63, pos = e & 7;
                    const int c = slab * 64 + ((pos ^ (r & 7)) << 3), a = r >> 4;
                    const uint32_t off = (uint32_t)(r * 128 + pos * 16);
                    const uint32_t m = r < L ? 0xFFFFFFFFu : 0u;
                    float f[8], v[8], qv[8], eg[8], ek[8], eq[8];
                    uint4 kd;
                    bf16x8_to_f32(ld16(smem + I_VB + slab * 8192 + off), v);
                    const uint4 xv = scale_chunk_h(v, S.bbuf[r], m);
                    st16(smem + I_B2 + slab * 8192 + off, xv.x, xv.y, xv.z, xv.w);
                    bf16x8_to_f32(ld16(smem + I_KQ + slab * 16384 + off), f);
                    bf16x8_to_f32(ld16(smem + I_KQ + slab * 16384 + 8192 + off), qv);
                    if (fast) {
                        float e8[8], f8[8], er[8], el[8];
                        ld_f8(E + r * ES + c, e8);
                        ld_f8(F + r * ES + c, f8);
                        ld_f8(&KS.er[a][c], er);
                        ld_f8(&KS.espl[a][c], el);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float g2 = e8[q] * er[q];   // 2^(G - R_a) 2^(R_a)
                            eg[q] = S.bbuf[r] * g2;
                            eq[q] = p.scale * g2;
                            ek[q] = f8[q] * el[q];   // k 2^(R_a - G) 2^(G_last - R_a)
                        }
                        kd = scale_chunk_h(ek, 1.f, m);
                    } else {
                        float g8[8], l8[8];
                        ld_f8(F + r * ES + c, g8);
                        ld_f8(&KS.lg63[c], l8);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float g2 = ex2(g8[q]);
                            eg[q] = S.bbuf[r] * g2;
                            eq[q] = p.scale * g2;
                            ek[q] = ex2(l8[q] - g8[q]);
                        }
                        kd = scale_chunk_hv(f, ek, m);
                    }
                    const uint4 xk = scale_chunk_hv(f, eg, m), qh = scale_chunk_hv(qv, eq, m);
                    st16(smem + I_B2 + 16384 + slab * 8192 + off, xk.x, xk.y, xk.z, xk.w);
                    stg16(kt + slab * 8192 + off, kd.x, kd.y, kd.z, kd.w);
                    stg16(wq + slab * 16384 + off, qh.x, qh.y, qh.z, qh.w);
                }
            }
            fence_async_smem();
            tmem_st_wait();
            tc_fence_before();
            __syncthreads();   // [C] A, [I; P] and X are in shared memory; K, Q, V, E and F are dead
            tc_fence_after();
            // the next item's tiles: K and Q, V, and its gate tile into E's place, a whole solve ahead of their use
            if (ok && loader && have_next) {
                intra_issue_kq(smem, S, &tmap_q, &tmap_k, nx, p.group);
                intra_issue_v<KDA>(smem, S, &tmap_v, &tmap_g, nx);
                kq_issued = ic + 2;
                v_issued = ic + 2;
            }
        // P (rows 64-127 of A1, fp16 K-major) to the workspace, one bulk copy; its rows are overwritten with T below
        if (ok && tid == 96) {
            bulk_s2g(ws.pp + (size_t)it.it * WS_P, smem + I_A1 + 8192, WS_P);
            bulk_commit();
        }
        // UT transform, T = (I + A)^{-1} in place
        solve_unit_lower_inplace(Am, Rt, tid, ok);
        if (tid == 96) bulk_wait_read();
        __syncthreads();   // the copy of P has read A1
        // T to fp16 into both halves of A1: [T; T], K-major (operand A of MMA2)
        if (ok) {
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                const int e = tid + I_THREADS * k2, j = e >> 3, c8 = e & 7;
                const float4 x0 = ld4(Am + j * TS + c8 * 8), x1 = ld4(Am + j * TS + c8 * 8 + 4);
                const float f[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                float gq[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) gq[q] = (c8 * 8 + q <= j) ? f[q] : 0.f;
                st_h8(smem + I_A1 + sw128_off(j, c8 * 8), gq);
                st_h8(smem + I_A1 + sw128_off(64 + j, c8 * 8), gq);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // MMA2: D2 = [T; T] [beta V | beta gamma K] -> [U | W; U | W], one N = 256 product (both halves of the rows
        // alike, so that every warp's TMEM lane quarter holds a share of the epilogue)
        if (ok && leader) {
            tc_fence_after();
            const uint32_t id = idesc_f16(128, 256, false, false, true);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f16(tmem + I_TM_D2, sdesc(sbase + I_A1 + ks * 32, 16, 1024),
                        sdesc(sbase + I_B2 + ks * 2048, 8192, 1024), id, ks > 0);
            mma_commit(&S.m2);
        }
        if (ok) ok = mbar_wait(&S.m2, par, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && tid == 0) set_status(16u);
        tc_fence_after();
        // epilogue 2: U and W to the workspace, one 32-row x 64-column tile per warp.  D2's two row halves are alike,
        // so warp (q4, pw) takes token rows 32 (q4 % 2) .. + 31 of column quarter 2 (q4 / 2) + pw: U of d_v half 0 or
        // 1, W of d_k slab 0 or 1.  It stages the tile (4 KB, the workspace's swizzled row layout) in shared memory
        // nothing reads or loads into any more this item (A1 after MMA2; the F table, which the next item's gate tables
        // rewrite only after waiting for these copies), then writes it out as 512-byte runs.
        if (ok) {
            uint8_t* stg = smem + (pw == 0 ? I_A1 : I_FF) + q4 * 4096;
            const int rh = q4 & 1, cq = ((q4 >> 1) << 1) | pw;
            uint8_t* dst = cq < 2 ? ws.u + (size_t)it.it * WS_U + cq * 8192 + rh * 4096
                                  : ws.wq + (size_t)it.it * WS_WQ + (cq - 2) * 16384 + 8192 + rh * 4096;
#pragma unroll
            for (int cp = 0; cp < 2; ++cp) {
                uint32_t r[2][16];
                tmem_ld16(tl + I_TM_D2 + cq * 64 + cp * 32, r[0]);
                tmem_ld16(tl + I_TM_D2 + cq * 64 + cp * 32 + 16, r[1]);
                tmem_ld_wait();
#pragma unroll
                for (int h8 = 0; h8 < 4; ++h8) {
                    float f[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) f[q] = __uint_as_float(r[h8 >> 1][(h8 & 1) * 8 + q]);
                    st_h8(stg + sw128_off(lane, cp * 32 + h8 * 8), f);
                }
            }
            fence_async_smem();   // the staging rows are read by the bulk-copy engine
            __syncwarp();
            if (lane == 0) {
                bulk_s2g(dst, stg, 4096);
                bulk_commit();
            }
        }
        tc_fence_before();
        if (warp == 1 && have_next) {   // every read of this item's g and beta is behind a barrier already
            S.gbuf[lane] = ng[0];
            S.gbuf[lane + 32] = ng[1];
            S.bbuf[lane] = nb[0];
            S.bbuf[lane + 32] = nb[1];
        }
        x = nx;
        cur = nc;
        have = ok && have_next;
        if (ok) ++ic;
    }
    if (lane == 0) bulk_wait_all();       // the workspace writes are complete before the CTA exits
    // loads that were issued but never waited on (after a timeout) must land before the CTA exits
    if (loader) {
        for (uint32_t k = kq_waited; k < kq_issued; ++k) mbar_wait(&S.full_kq, k & 1, kWaitNs);
        for (uint32_t k = v_waited; k < v_issued; ++k) mbar_wait(&S.full_v, k & 1, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, I_TM_COLS);
}

// ==================================================================== pass 2: state pass
struct StateParams {
    Geo geo;
    const float* h0;
    float* hT;
    void* o;
    Ws ws;
    int test_skip;   // test of the bounded waits: the first chunk record is never copied
};

// Pass 2: one CTA per (sequence, head, 64-column d_v half), 8 warps; warp w reads TMEM lane quarter w % 4 and the 32
// columns w / 4 of the half (the fp32 state is 32 registers per thread).  Per chunk
// (its workspace slot streamed by bulk copies through a two-stage ring):
//   MMA3   D3 = [Q^; W] h~ : rows 0-63 Q^ h~ (for O), rows 64-127 W h~
//   Delta = U - W h~ (lane quarters 2-3), to fp16 in shared memory
//   MMA4   D4 = Ktilde^T Delta, and MMA5  D5 = P Delta (rows 0-63; an M = 128 product whose rows 64-127 read past P
//          into U and are never used)
//   h <- gamma_C h + D4 (all lanes: row d_k), fp16 copy h~ for the next MMA3
//   O = Q^ h~ + P Delta (lane quarters 0-1), written one chunk later, while the next MMA3 runs (D3 and D5 are
//   double-buffered by chunk parity)
struct SLayout {
    static constexpr uint32_t WQ = 0, KT = 32768, PP = 49152, U = 57344, GC = 65536;   // one workspace slot
    static constexpr uint32_t STAGE = 66560;
    static constexpr uint32_t H = 2 * STAGE;         // h~, fp16 MN-major [d][n] 128 x 64
    static constexpr uint32_t D = H + 16384;         // Delta, fp16 MN-major [j][n] 64 x 64
    static constexpr uint32_t SMALL = D + 8192;
    static constexpr int THREADS = 256;
    static constexpr uint32_t TM_D3 = 0, TM_D4 = 128, TM_D5 = 192, TM_COLS = 512;   // D3, D5: two each
};
struct SSmall {
    uint64_t full[2];
    uint64_t m3, m4;
    uint32_t tmem_base;
    uint32_t pad;
};
constexpr uint32_t s_smem_bytes() { return SLayout::SMALL + sizeof(SSmall) + 1024; }
static_assert(s_smem_bytes() <= 227 * 1024, "state kernel shared memory");

struct Chain {
    int n, h, half, len;
    long row0;
};

// CTA -> (sequence, head, d_v half); packed sequences longest first (their chains are the longest serial paths)
__device__ Chain resolve_chain(const Geo& g) {
    Chain c;
    const int per_seq = g.H * 2;
    const int seq_rank = blockIdx.x / per_seq;
    const int rem = blockIdx.x % per_seq;
    c.h = rem / 2;
    c.half = rem % 2;
    int n = seq_rank;
    if (g.cu && g.n_seqs <= 32) {
        const int lane = threadIdx.x & 31;
        int rank = -1;
        if (lane < g.n_seqs) {
            long s0;
            int lm;
            g.seq(lane, s0, lm);
            rank = 0;
            for (int m2 = 0; m2 < g.n_seqs; ++m2) {
                long s2;
                int l2;
                g.seq(m2, s2, l2);
                rank += (l2 > lm) || (l2 == lm && m2 < lane);
            }
        }
        const unsigned hit = __ballot_sync(0xffffffffu, rank == seq_rank);
        if (hit) n = __ffs(hit) - 1;
    }
    c.n = n;
    g.seq(n, c.row0, c.len);
    return c;
}

__device__ __forceinline__ void state_issue(uint8_t* smem, SSmall& S, const Ws& ws, long it, int half, int s) {
    using LY = SLayout;
    uint8_t* st = smem + s * LY::STAGE;
    mbar_arrive_expect_tx(&S.full[s], WS_WQ + WS_KT + WS_P + 8192 + WS_GC);
    bulk_g2s(st + LY::WQ, ws.wq + (size_t)it * WS_WQ, WS_WQ, &S.full[s]);
    bulk_g2s(st + LY::KT, ws.kt + (size_t)it * WS_KT, WS_KT, &S.full[s]);
    bulk_g2s(st + LY::PP, ws.pp + (size_t)it * WS_P, WS_P, &S.full[s]);
    bulk_g2s(st + LY::U, ws.u + (size_t)it * WS_U + half * 8192, 8192, &S.full[s]);
    bulk_g2s(st + LY::GC, ws.gc + (size_t)it * 128, WS_GC, &S.full[s]);
}

// O = Q^ h~ + P Delta of chunk t (token rows 0-63: lane quarters 0 and 1), columns cs .. cs + 31 of the half, from
// D3 and D5 of its parity
template <bool O_F32>
__device__ __forceinline__ bool state_output(const StateParams& p, const Chain& ch, uint32_t tl, int t, int row,
                                             int cs) {
    bool finite = true;
    using LY = SLayout;
    const int L = min(C, ch.len - t * C);
    const size_t orow = ((size_t)(ch.row0 + (long)t * C + row) * p.geo.H + ch.h) * DV + ch.half * DVT;
    {   // 32 columns: four loads, one wait
        const int h2 = cs >> 5;
        uint32_t a[2][16], b[2][16];
        tmem_ld16(tl + LY::TM_D3 + (t & 1) * 64 + h2 * 32, a[0]);
        tmem_ld16(tl + LY::TM_D3 + (t & 1) * 64 + h2 * 32 + 16, a[1]);
        tmem_ld16(tl + LY::TM_D5 + (t & 1) * 64 + h2 * 32, b[0]);
        tmem_ld16(tl + LY::TM_D5 + (t & 1) * 64 + h2 * 32 + 16, b[1]);
        tmem_ld_wait();
        if (row < L) {
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                float f[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    f[k] = __uint_as_float(a[hq][k]) + __uint_as_float(b[hq][k]);
                    finite = finite && isfinite(f[k]);
                }
                const size_t o0 = orow + h2 * 32 + hq * 16;
                if (O_F32) {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + o0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) dst[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + o0);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        uint32_t pk[4];
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(f[8 * q + 2 * m], f[8 * q + 2 * m + 1]);
                            pk[m] = *reinterpret_cast<uint32_t*>(&b2);
                        }
                        dst[q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
        }
    }
    return finite;
}

template <bool O_F32>
__global__ void __launch_bounds__(SLayout::THREADS, 1) chunk_state_kernel(const StateParams p) {
    using LY = SLayout;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    SSmall& S = *reinterpret_cast<SSmall*>(smem + LY::SMALL);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3;                    // TMEM lane quarter
    const int cs = 32 * (warp >> 2);            // this thread's first column within the half
    const Chain ch = resolve_chain(p.geo);
    const int n_chunks = (ch.len + C - 1) / C;
    const long slot0 = ch.row0 / C + ch.n;
    const int H = p.geo.H;
    const int row = 32 * q4 + lane;             // TMEM lane: token row of D3 and D5, d_k row of D4 and of h
    const bool leader = (tid == 64);            // issues the products (a Delta warp)
    const bool issuer = (tid == 32);            // issues the copies, off the leader's path
    const bool out_warp = q4 < 2;               // O (token rows 0-63); the others form Delta (rows 64-127)
    const int col0 = ch.half * DVT + cs;        // first d_v column of this thread in the head

    if (warp == 0) {
        tmem_alloc(&S.tmem_base, LY::TM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(&S.full[0], 1);
        mbar_init(&S.full[1], 1);
        mbar_init(&S.m3, 1);
        mbar_init(&S.m4, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);

    // the per-chunk kernel has completed and its workspace writes are visible (with a programmatic launch this
    // CTA may have started before that; everything above reads only inputs)
    griddep_wait();
    if (issuer) {
        for (int t = 0; t < 2 && t < n_chunks; ++t)
            if (!(p.test_skip && t == 0)) state_issue(smem, S, p.ws, (slot0 + t) * H + ch.h, ch.half, t);
    }
    int issued = n_chunks < 2 ? n_chunks : 2;

    const size_t sidx = ((size_t)ch.n * H + ch.h) * DK * DV + (size_t)row * DV + col0;
    float hreg[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 v = p.h0 ? reinterpret_cast<const float4*>(p.h0 + sidx)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        hreg[4 * q] = v.x;
        hreg[4 * q + 1] = v.y;
        hreg[4 * q + 2] = v.z;
        hreg[4 * q + 3] = v.w;
    }
    // h to fp16, MN-major [d][n] (operand B of MMA3)
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) st_h8(smem + LY::H + sw128_off(row, cs + c8 * 8), hreg + c8 * 8);
    fence_async_smem();
    __syncthreads();

    // Operand descriptors, built once; a k-step adds its byte offset >> 4 to the start-address field (the operands
    // lie below 256 KB, so the field never carries).
    const uint64_t dH = sdesc(sbase + LY::H, 16384, 1024), dD = sdesc(sbase + LY::D, 8192, 1024);
    const uint64_t dWQ = sdesc(sbase + LY::WQ, 16, 1024), dKT = sdesc(sbase + LY::KT, 8192, 1024);
    const uint64_t dP = sdesc(sbase + LY::PP, 16, 1024);
    const uint32_t id3 = idesc_f16(128, 64, false, false, true), id4 = idesc_f16(128, 64, false, true, true);
    bool ok = true;
    bool finite = true;   // every value this thread wrote to o and the final state is finite
    int waited = 0;   // chunks whose stage wait completed
    for (int t = 0; t < n_chunks; ++t) {
        const int s = t & 1;
        const uint8_t* st = smem + s * LY::STAGE;
        const uint64_t so = (uint64_t)((s * LY::STAGE) >> 4);
        if (ok) ok = mbar_wait(&S.full[s], (t >> 1) & 1, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && tid == 0) set_status(32u);
        if (ok) waited = t + 1;
        // MMA3: D3[t & 1] = [Q^; W] h~
        if (ok && leader) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_f16(tmem + LY::TM_D3 + s * 64, dWQ + so + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2),
                        dH + (uint64_t)(ks * 128), id3, ks > 0);
            mma_commit(&S.m3);
        }
        // meanwhile the output of the previous chunk (its D3 and D5 are the other parity)
        if (ok && out_warp && t > 0) finite = state_output<O_F32>(p, ch, tl, t - 1, row, cs) && finite;
        if (ok) ok = mbar_wait(&S.m3, t & 1, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && tid == 0) set_status(64u);
        tc_fence_after();
        if (!out_warp) {
            // Delta = U - W h~ (token row i = row - 64) to fp16 MN-major [j][n] (operand B of MMA4 and MMA5)
            const int i = row - 64;
            if (ok) {
                {
                    const int h2 = cs >> 5;
                    uint32_t a[2][16];
                    tmem_ld16(tl + LY::TM_D3 + s * 64 + h2 * 32, a[0]);
                    tmem_ld16(tl + LY::TM_D3 + s * 64 + h2 * 32 + 16, a[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int h8 = 0; h8 < 4; ++h8) {
                        float u[8], f[8];
                        h8_to_f32(ld16(st + LY::U + sw128_off(i, h2 * 32 + h8 * 8)), u);
#pragma unroll
                        for (int q = 0; q < 8; ++q) f[q] = u[q] - __uint_as_float(a[h8 >> 1][(h8 & 1) * 8 + q]);
                        st_h8(smem + LY::D + sw128_off(i, h2 * 32 + h8 * 8), f);
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            named_bar(1, 128);   // the Delta warps (lane quarters 2 and 3)
            // MMA4: D4 = Ktilde^T Delta; MMA5: D5[t & 1] = [P; -] Delta
            if (ok && leader) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(tmem + LY::TM_D4, dKT + so + (uint64_t)(ks * 128), dD + (uint64_t)(ks * 128), id4, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(tmem + LY::TM_D5 + s * 64, dP + so + (uint64_t)(ks * 2), dD + (uint64_t)(ks * 128), id3,
                            ks > 0);
                mma_commit(&S.m4);
            }
        }
        if (ok) ok = mbar_wait(&S.m4, t & 1, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && tid == 0) set_status(128u);
        tc_fence_after();
        // h <- gamma_C h + Ktilde^T Delta; fp16 copy for the next MMA3
        if (ok) {
            const float gC = reinterpret_cast<const float*>(st + LY::GC)[row];
            uint32_t r[2][16];
            tmem_ld16(tl + LY::TM_D4 + cs, r[0]);
            tmem_ld16(tl + LY::TM_D4 + cs + 16, r[1]);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) hreg[k] = fmaf(gC, hreg[k], __uint_as_float(r[k >> 4][k & 15]));
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) st_h8(smem + LY::H + sw128_off(row, cs + c8 * 8), hreg + c8 * 8);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();   // stage s, D4 and Delta are free; D3 and D5 of chunk t hold its output
        if (ok && issuer && t + 2 < n_chunks) {
            state_issue(smem, S, p.ws, (slot0 + t + 2) * H + ch.h, ch.half, s);
            issued = t + 3;
        }
    }
    if (ok && out_warp && n_chunks > 0) {
        tc_fence_after();
        finite = state_output<O_F32>(p, ch, tl, n_chunks - 1, row, cs) && finite;
    }
    // stages issued but never waited on (after a timeout) must land before the CTA exits
    if (issuer) {
        for (int t = waited; t < issued; ++t)
            if (!(p.test_skip && t == 0)) mbar_wait(&S.full[t & 1], (t >> 1) & 1, kWaitNs);
    }
    if (p.hT && ok) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(p.hT + sidx)[q] =
                make_float4(hreg[4 * q], hreg[4 * q + 1], hreg[4 * q + 2], hreg[4 * q + 3]);
#pragma unroll
        for (int k = 0; k < 32; ++k) finite = finite && isfinite(hreg[k]);
    }
    if (__any_sync(0xffffffffu, !finite) && lane == 0) set_status(kStatusNonfinite);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, LY::TM_COLS);
}

long n_slots(const ChunkArgs& a) { return (long)a.B * a.T / C + a.N() + 1; }

}  // namespace

const char* two_pass_unsupported_reason(const ChunkArgs& a) {
    if (a.per_channel && a.act.gate()) return "the gate activation applies to the scalar gate only";
    if (!a.bf16) return "q, k, v must be bf16";
    const bool d256 = !a.per_channel && a.dk == 256 && a.dv == 256;
    if ((a.dk != DK || a.dv != DV) && !d256)
        return a.per_channel ? "d_k and d_v must be 128" : "d_k and d_v must both be 128 or both be 256";
    if (a.C != C) return "chunk_size must be 64";
    auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) % 16) == 0; };
    if (!al16(a.q) || !al16(a.k) || !al16(a.v) || !al16(a.o) || (a.h0 && !al16(a.h0)) || (a.hT && !al16(a.hT)) ||
        (a.per_channel && !al16(a.g)))
        return "tensors must be 16-byte aligned";
    return nullptr;
}

size_t two_pass_workspace_bytes(const ChunkArgs& a) {
    if (!a.per_channel) return a.dk == 256 ? gdn_d256_workspace_bytes(a) : gdn_tmem_workspace_bytes(a);
    if ((long)a.B * a.T == 0) return 0;
    return (size_t)n_slots(a) * a.H * WS_ITEM;
}

cudaError_t launch_chunk_two_pass(const ChunkArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t s) {
    if (!a.per_channel)
        return a.dk == 256 ? launch_chunk_gdn_d256(a, workspace, workspace_bytes, s)
                           : launch_chunk_gdn_tmem(a, workspace, workspace_bytes, s);
    const long chains = (long)a.N() * a.H;
    if (chains == 0) return cudaSuccess;
    if (!device_is_sm100_family()) return cudaErrorNoKernelImageForDevice;
    const long rows = (long)a.B * a.T;
    if (rows == 0) {
        if (a.hT) {
            const size_t bytes = (size_t)a.N() * a.H * DK * DV * sizeof(float);
            return a.h0 ? cudaMemcpyAsync(a.hT, a.h0, bytes, cudaMemcpyDeviceToDevice, s)
                        : cudaMemsetAsync(a.hT, 0, bytes, s);
        }
        return cudaSuccess;
    }
    const size_t need = two_pass_workspace_bytes(a);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % 256) != 0)
        return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, rows, a.HK(), DK) || !make_map(&mk, a.k, rows, a.HK(), DK) ||
        !make_map(&mv, a.v, rows, a.H, DV))
        return cudaErrorInvalidValue;
    const long items = n_slots(a) * a.H;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    Ws ws;
    ws.wq = base;
    ws.kt = ws.wq + (size_t)items * WS_WQ;
    ws.u = ws.kt + (size_t)items * WS_KT;
    ws.pp = ws.u + (size_t)items * WS_U;
    ws.gc = reinterpret_cast<float*>(ws.pp + (size_t)items * WS_P);
    Geo geo{a.cu, a.n_seqs, a.B, a.T, a.H};

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    IntraParams ip{geo, a.g, a.beta, a.scale, n_slots(a), ws, a.act, a.H / a.HK()};
    CUtensorMap mg;
    if (!make_map_f32_rows(&mg, a.g, rows, a.H, DK)) return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(chunk_intra_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)I_SMEM_KDA);
    if (e != cudaSuccess) return e;
    const long grid1 = items < sms ? items : sms;
    chunk_intra_kernel<true><<<(unsigned)grid1, I_THREADS, I_SMEM_KDA, s>>>(mq, mk, mv, mg, ip);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    StateParams sp{geo, a.h0, a.hT, a.o, ws, a.test_fwd == 1 ? 1 : 0};
    const unsigned grid2 = (unsigned)(chains * 2);
    // Programmatic stream serialisation: the state kernel's CTAs may start on SMs the per-chunk kernel has left,
    // and wait (griddepcontrol.wait) for its completion before they read the workspace.
    auto launch2 = [&](auto kern) -> cudaError_t {
        cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_smem_bytes());
        if (e2 != cudaSuccess) return e2;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(grid2);
        cfg.blockDim = dim3(SLayout::THREADS);
        cfg.dynamicSmemBytes = s_smem_bytes();
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, sp);
    };
    e = a.o_f32 ? launch2(chunk_state_kernel<true>) : launch2(chunk_state_kernel<false>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

size_t static_workspace_capacity() { return kStaticWorkspaceBytes; }

cudaError_t static_workspace(void** ptr) {
    static std::mutex mu;
    static void* addr[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);   // with this device current
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

cudaError_t tp_read_and_clear_status(unsigned* value, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_tp_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    if (clear && *value) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_tp_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace gdn
