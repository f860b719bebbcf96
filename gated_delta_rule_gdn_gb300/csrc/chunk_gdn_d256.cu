// Scalar-gate (GDN) chunk forward at head size 256 (d_k = d_v = 256) in two passes on tcgen05 tensor cores
// (sm_103a): bf16 q/k/v, chunk C = 64, fp32 state, o in fp32 or bf16.
//
// The algebra is the chunkwise WY/UT form of "TileLang 实战：KDA 从零到一 -- Gated DeltaNet", §2.3, split as
// "Gated Delta Network (GDN)", §4(b3)-(d) splits it, and the same as the head-size-128 pair (chunk_gdn_tmem.cu); that
// page's §4.3 bounds the head sizes at 256.  Per chunk of L <= C rows, with G the within-chunk cumulative log gate
// (log2 units), gamma_i = 2^{G_i}, Gamma_ij = 2^{G_i - G_j} (j <= i):
//   A = diag(beta)(Gamma * K K^T) strictly lower,  P = scale (Gamma * Q K^T) lower including the diagonal,
//   T = (I + A)^{-1},  W = T diag(beta gamma) K,  U = T diag(beta) V,
//   Delta = U - W h,  O = scale diag(gamma) Q h + P Delta,  h <- gamma_C h + K~^T Delta,  K~ = diag(gamma_C / gamma) K.
//
// Pass 1, gdn_intra256_kernel: one item per (chunk slot, head), persistent CTAs, two per SM.  MMA0 = [K; Q] K^T over
// d_k = 256 (16 K steps) gives A and P; the blocked inverse T in place; MMA2 = [T diag(beta gamma); same] K (N = 256)
// gives W.  The item's record, 112 KB in the operand layouts of pass 2: [-W; Q~] (64 KB), K~ (32 KB), P^T and
// T diag(beta) (8 KB each), with Q~ = diag(scale gamma) Q and K~ = diag(gamma_C / gamma) K converted to fp16 here,
// from the tiles the per-chunk products already hold.  (Converted in the state kernel instead, the two tiles cost
// that kernel 128 KB of shared-memory traffic per chunk, about a quarter of all of it, and slowed every chain step.)
//
// Pass 2, gdn_state256_kernel: one CTA per (sequence, head, d_v half of 128 columns).  It works in the transposed
// orientation (tensor-memory lane = d_v row).  The half's state, 128 d_v rows x 256 d_k columns of fp32, is too large
// for registers: it lives in tensor memory, scaled ahead by the next chunk's gamma_C (H = gamma_C h), and the state
// update is a product accumulating onto it.  Per chunk:
//   MMA_U  D3[:, 0:64] = V^T (T diag beta)^T                   (V converted to fp16 in the kernel; off the chain)
//   MMA3   D3 += h~^T [-W; Q~]^T (A = h~^T, the state's fp16 copy in tensor memory, K = d_k = 256): columns 0-63
//          become Delta^T, 64-127 (Q~ h)^T
//   Delta epilogue: Delta^T to fp16 in place
//   MMA4   H += Delta^T K~ (N = 256): H becomes h of the chunk's end
//   MMA5   D3[:, 64:128] += Delta^T P^T: O^T
//   lane warps: h~ = fp16(H) for the next MMA3, H <- gamma_C' H for the next MMA4 (the final state unscaled)
//   output warps: O^T from tensor memory to a staging tile, out by tensor stores of 32 tokens (plain per-thread
//   stores of the same rows were several times slower)
// Tensor memory holds H (256 columns), h~ (128) and D3 (128): all 512.  Sixteen warps: eight lane warps (two per lane
// quarter, 128 d_k columns each) run the Delta epilogue and the state scaling; four output warps (one per lane
// quarter) write O; one warp issues the products, one the copies; two convert V (one of them first computes gamma_C).
//
// Operand precision is that of the head-size-128 pair: fp16 operands (h~, -W, P, T diag(beta), Delta, and q, k, v
// converted to fp16 with their gate factors applied first), fp32 accumulation, the state itself fp32.  fp16
// saturates at 65,504; the state kernel checks what it writes and reports a non-finite value through the device
// status (GDN_ERR_NONFINITE).
//
// Every mbarrier wait is bounded (2 s); a wait that gives up sets a status bit, the CTA drops its work, lands its copies
// in flight, frees its tensor memory and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc_common.cuh"
#include "chunk_common.cuh"
#include "gate_act.cuh"
#include "chunk_wy_common.cuh"
#include "chunk_gdn_common.cuh"

namespace gdn {

__device__ unsigned g_d256_status;

namespace {

constexpr int D2 = 256;      // d_k = d_v
constexpr int VT = 128;      // d_v columns of one state CTA

// workspace record of one (chunk slot, head) item, in the operand layouts of the state kernel (rows of 128 B,
// 128-byte swizzle)
constexpr uint32_t R_WQ = 0;        // [-W; Q~] fp16 [token][d_k]: per 64-column slab (four, 16 KB apart) 64 rows of -W,
                                    // then 64 rows of Q~ = diag(scale gamma) Q
constexpr uint32_t R_K = 65536;     // K~ = diag(gamma_C / gamma) K fp16 [token][d_k], four 64-column slabs of 64 rows
constexpr uint32_t R_P = 98304;     // P^T fp16 [j][i]
constexpr uint32_t R_TB = 106496;   // T diag(beta) fp16 [i][j]
constexpr uint32_t R_ITEM = 114688;

__device__ __forceinline__ void d_status(unsigned bit) { atomicOr(&g_d256_status, bit); }

// ==================================================================== pass 1: per-chunk products
struct IParams {
    Geo geo;
    const float* g;
    const float* beta;
    float scale;
    long n_slots;
    uint8_t* ws;
    GateAct act;
    int group;    // value heads per key head
};

// shared memory of pass 1 (byte offsets from a 1024-aligned base); about 98 KB, two CTAs per SM
constexpr uint32_t I_KQ = 0;          // [K; Q]: per 64-column slab (four), 64 K rows then 64 Q rows (16 KB)
constexpr uint32_t I_A1 = 65536;      // [T diag(beta gamma); same] bf16 K-major 128 x 64 (operand A of MMA2); the
                                      // solve's scratch before that
constexpr uint32_t I_PS = I_A1 + 8192;   // P fp16 staging for the bulk copy, in the second half of A1 (past the solve's
                                         // scratch; the T scalings overwrite it once the copy has read it)
constexpr uint32_t I_AM = 81920;      // fp32 A, then T in place (row stride TS)
constexpr uint32_t I_WST = I_A1;      // -W staging (32 KB, over A1 and A: both dead once MMA2 has completed)
constexpr uint32_t I_END = I_AM + 64 * TS * 4;
static_assert(32 * RS * 4 <= 8192, "the solve scratch must fit in the first half of A1");
static_assert(I_END - I_WST >= 32768, "-W staging must fit over A1 and A");

struct ISmall {
    uint64_t full_kq;
    uint64_t m0, m2;
    uint32_t tmem_base;
    uint32_t pad;
    float gbuf[C];       // g of the item (0 past the end)
    float bbuf[C];       // beta of the item (0 past the end)
    float lg[C];         // log2 cumulative gate
    float bg[C];         // beta_j gamma_j
};
constexpr uint32_t I_SMEM = I_END + sizeof(ISmall) + 1024;
constexpr int I_THREADS = 256;
constexpr int I_CTAS_PER_SM = 2;
constexpr uint32_t I_TM_COLS = 256;   // D0 (64 columns) and, after the solve, D2 (256 columns) at column 0

__global__ void __launch_bounds__(I_THREADS, I_CTAS_PER_SM)
gdn_intra256_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const IParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    ISmall& S = *reinterpret_cast<ISmall*>(smem + I_END);
    float* Am = reinterpret_cast<float*>(smem + I_AM);
    float* Rt = reinterpret_cast<float*>(smem + I_A1);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, pw = warp >> 2;
    const int row = 32 * q4 + lane;
    const bool leader = (tid == 0);
    const bool loader = (tid == 64);
    const int H = p.geo.H;
    griddep_launch_dependents();

    if (warp == 0) {
        tmem_alloc(&S.tmem_base, I_TM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(&S.full_kq, 1);
        mbar_init(&S.m0, 1);
        mbar_init(&S.m2, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);

    auto issue_kq = [&](const Item& x) {
        const int r = (int)x.row, hk = x.h / p.group;
        uint8_t* kq = smem + I_KQ;
        mbar_arrive_expect_tx(&S.full_kq, 65536);
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
            tma_load_3d(kq + sl * 16384, &tmap_k, &S.full_kq, 64 * sl, hk, r);
            tma_load_3d(kq + sl * 16384 + 8192, &tmap_q, &S.full_kq, 64 * sl, hk, r);
        }
    };
    auto load_gb = [&](const Item& x, float (&g)[2], float (&b)[2]) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = lane + 32 * k;
            const size_t tok = (size_t)(x.row + r) * H + x.h;
            g[k] = r < x.L ? act_gate(p.act, __ldg(p.g + tok), x.h) : 0.f;
            b[k] = r < x.L ? act_beta(p.act, __ldg(p.beta + tok)) : 0.f;
        }
    };

    const int ds = (int)(gridDim.x / H), dh = (int)(gridDim.x % H);
    const long first = p.n_slots * H - 1 - (long)blockIdx.x;
    Cursor cur{first / H, (int)(first % H), p.geo.N() - 1};
    Item x;
    bool have = cursor_next_valid(p.geo, cur, ds, dh, x);
    float ng[2] = {0.f, 0.f}, nb[2] = {0.f, 0.f};
    uint32_t issued = 0, waited = 0;   // loader's count of K/Q loads issued and waited
    if (have) {
        if (loader) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            issue_kq(x);
            issued = 1;
        }
        if (warp == 1) {
            float gg[2], bb[2];
            load_gb(x, gg, bb);
            S.gbuf[lane] = gg[0];
            S.gbuf[lane + 32] = gg[1];
            S.bbuf[lane] = bb[0];
            S.bbuf[lane + 32] = bb[1];
        }
    }
    bool ok = true;
    uint32_t ic = 0;
    while (have) {
        const Item it = x;
        Cursor nc = cur;
        cursor_step(nc, ds, dh, H);
        Item nx;
        const bool have_next = cursor_next_valid(p.geo, nc, ds, dh, nx);
        const uint32_t par = ic & 1;
        uint8_t* kq = smem + I_KQ;
        uint8_t* rec = p.ws + (size_t)it.it * R_ITEM;
        __syncthreads();   // [A] g, beta of this item in shared memory; the previous item is retired
        if (warp == 1) {
            float G0, G1, Gl;
            gate_prefix2(S.gbuf[2 * lane], S.gbuf[2 * lane + 1], lane, G0, G1, Gl);
            S.lg[2 * lane] = G0;
            S.lg[2 * lane + 1] = G1;
            S.bg[2 * lane] = S.bbuf[2 * lane] * ex2(G0);
            S.bg[2 * lane + 1] = S.bbuf[2 * lane + 1] * ex2(G1);
            if (have_next) load_gb(nx, ng, nb);
        }
        if (ok) ok = mbar_wait(&S.full_kq, par, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && tid == 0) d_status(1u);
        if (ok && loader) waited = ic + 1;
        // MMA0: D0 = [K; Q] K^T (M = 128, N = 64, K = 256)
        if (ok && leader) {
            tc_fence_after();
            const uint32_t id = idesc_f16(128, 64, true, false, false);
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                const uint32_t a = smem_u32(kq) + (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_f16(tmem, sdesc(a, 16, 1024), sdesc(a, 16, 1024), id, ks > 0);
            }
            mma_commit(&S.m0);
        }
        // the previous item's -W copy has read its staging (over A1 and A)
        if (lane == 0) bulk_wait_read();
        if (ok && leader) ok = mbar_wait(&S.m0, par, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && leader) d_status(2u);
        tc_fence_before();
        __syncthreads();   // [B] D0 ready; the staging buffers are free
        tc_fence_after();
        if (ok) epilogue_kkt<false>(tl, row, q4, pw, S.lg, S.bbuf, p.scale, Am, smem + I_PS - 8192);
        fence_async_smem();   // P staging is read by the bulk copy
        tc_fence_before();
        __syncthreads();   // [C] A and P are in shared memory
        if (ok && tid == 96) {
            bulk_s2g(rec + R_P, smem + I_PS, 8192);
            bulk_commit();
        }
        // UT transform, T = (I + A)^{-1} in place (the scratch is the first half of A1)
        solve_unit_lower_inplace(Am, Rt, tid, ok);
        if (tid == 96) bulk_wait_read();   // the copy of P has read its staging, which the scalings overwrite
        __syncthreads();
        // T diag(beta gamma) in bf16 into both row halves of A1 (operand A of MMA2), and T diag(beta) in fp16 straight
        // to the record.  Thread e: row i = e / 8, physical 16-byte chunk pc = e % 8 of the swizzled row.
        if (ok) {
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                const int e = tid + I_THREADS * k2, i = e >> 3, pc = e & 7, c0 = (pc ^ (i & 7)) << 3;
                const float4 x0 = ld4(Am + i * TS + c0), x1 = ld4(Am + i * TS + c0 + 4);
                const float t[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                float tb[8], tg[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const bool on = c0 + q <= i;
                    tb[q] = on ? t[q] * S.bbuf[c0 + q] : 0.f;
                    tg[q] = on ? t[q] * S.bg[c0 + q] : 0.f;
                }
                const uint32_t o = (uint32_t)(i * 128 + pc * 16);
                const uint32_t g0 = pack_bf2(tg[0], tg[1]), g1 = pack_bf2(tg[2], tg[3]), g2 = pack_bf2(tg[4], tg[5]),
                               g3 = pack_bf2(tg[6], tg[7]);
                st16(smem + I_A1 + o, g0, g1, g2, g3);
                st16(smem + I_A1 + 8192 + o, g0, g1, g2, g3);
                stg16(rec + R_TB + o, pack_h2(tb[0], tb[1]), pack_h2(tb[2], tb[3]), pack_h2(tb[4], tb[5]),
                      pack_h2(tb[6], tb[7]));
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();   // [D] A1 ready; every read of T is done
        // MMA2: D2 = A1 K (M = 128, N = 256 = d_k, K = 64 tokens; K is the MN-major view of the raw K tile, its four
        // 64-column slabs 16 KB apart)
        if (ok && leader) {
            tc_fence_after();
            const uint32_t id = idesc_f16(128, 256, true, false, true);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f16(tmem, sdesc(sbase + I_A1 + ks * 32, 16, 1024), sdesc(smem_u32(kq) + ks * 2048, 16384, 1024),
                        id, ks > 0);
            mma_commit(&S.m2);
        }
        // Q~ = diag(scale gamma) Q and K~ = diag(gamma_C / gamma) K in fp16 straight to the record, in the layout of
        // their tiles (rows past the end: zeros), while MMA2 runs (it reads only the K rows).  Piece c (16 bytes):
        // tile c / 2048 (Q, K), slab (c / 512) % 4, byte offset 16 (c % 512) of the slab's 64 rows.
        if (ok) {
            const float Gl = S.lg[C - 1];
#pragma unroll 4
            for (int k2 = 0; k2 < 16; ++k2) {
                const int c = tid + I_THREADS * k2;
                const int isk = c >> 11, sl = (c >> 9) & 3, off = (c & 511) * 16, r = off >> 7;
                float x[8];
                bf16x8_to_f32(ld16(kq + sl * 16384 + (isk ? 0 : 8192) + off), x);
                const float f = isk ? ex2(Gl - S.lg[r]) : p.scale * ex2(S.lg[r]);
                const uint32_t m = r < it.L ? 0xFFFFFFFFu : 0u;
                stg16(rec + (isk ? R_K + sl * 8192 : R_WQ + sl * 16384 + 8192) + off, pack_h2(f * x[0], f * x[1]) & m,
                      pack_h2(f * x[2], f * x[3]) & m, pack_h2(f * x[4], f * x[5]) & m, pack_h2(f * x[6], f * x[7]) & m);
            }
        }
        __syncthreads();   // [D'] every thread has read the K and Q tiles: the next item's may land over them
        if (ok) ok = mbar_wait(&S.m2, par, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && tid == 0) d_status(4u);
        // MMA2 has read K: the next item's K and Q can land
        if (ok && loader && have_next) {
            issue_kq(nx);
            issued = ic + 2;
        }
        tc_fence_after();
        // epilogue 2: -W in fp16 into the staging (A1 and A, now dead) as [token][d_k] in four swizzled 64-column
        // slabs.  D2's two row halves are alike, so warp (q4, pw) takes token rows 32 (q4 % 2) .. + 31 and the d_k
        // column blocks cq = 2 (q4 / 2) + pw and cq + 4 (32 columns each).
        if (ok) {
            const int tr = 32 * (q4 & 1) + lane;
#pragma unroll 1
            for (int rep = 0; rep < 2; ++rep) {
                const int cq = 4 * rep + 2 * (q4 >> 1) + pw;
                uint32_t r[2][16];
                tmem_ld16(tl + cq * 32, r[0]);
                tmem_ld16(tl + cq * 32 + 16, r[1]);
                tmem_ld_wait();
                uint8_t* wst = smem + I_WST + (cq >> 1) * 8192;
#pragma unroll
                for (int h8 = 0; h8 < 4; ++h8) {
                    uint32_t w4[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int k = h8 * 8 + 2 * m;
                        w4[m] = pack_h2(-__uint_as_float(r[k >> 4][k & 15]),
                                        -__uint_as_float(r[(k + 1) >> 4][(k + 1) & 15]));
                    }
                    st16(wst + sw128_off(tr, (cq & 1) * 32 + h8 * 8), w4[0], w4[1], w4[2], w4[3]);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();   // [E] -W staged
        if (ok && tid == 0) {
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) bulk_s2g(rec + R_WQ + sl * 16384, smem + I_WST + sl * 8192, 8192);
            bulk_commit();
        }
        if (warp == 1 && have_next) {
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
    if (lane == 0) bulk_wait_all();   // the record writes are complete before the CTA exits
    if (loader) {
        for (uint32_t k = waited; k < issued; ++k) mbar_wait(&S.full_kq, k & 1, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, I_TM_COLS);
}

// ==================================================================== pass 2: state pass
struct SParams {
    Geo geo;
    const float* g;
    float scale;
    const float* h0;
    float* hT;
    void* o;
    const uint8_t* ws;
    GateAct act;
    int group;
    int test;     // 1: leave out the first record copy (the waits for it run out); 2: a one-chunk-deep [-W; Q~] ring
};

// Shared memory of pass 2 (byte offsets from a 1024-aligned base; every operand base is 1024-aligned)
struct SL {
    static constexpr uint32_t QW = 0;          // two stages of [-W; Q~] fp16 K-major (record, one copy), four
                                               // 64-column slabs of 128 rows (16 KB each)
    static constexpr uint32_t QW_STAGE = 65536;
    static constexpr uint32_t KF = 131072;     // K~ fp16 (record), MN-major operand of MMA4, four 64-column slabs of
                                               // 64 rows
    static constexpr uint32_t PT = 163840;     // P^T fp16 (record), MN-major operand of MMA5
    static constexpr uint32_t OST = 172032;    // half of O of a chunk for the tensor store, [32 tokens][128] in o's
                                               // dtype
    static constexpr uint32_t VF = 188416;     // two stages of the V tile of the d_v half (TMA, bf16) -> fp16 in place;
                                               // MN-major operand of MMA_U (16 KB each)
    static constexpr uint32_t TB = 221184;     // T diag(beta) fp16 (record)
    static constexpr uint32_t VEC = 229376;    // 2 x SVec (gamma_C of the chunk)
    static constexpr int THREADS = 512;        // lane warps 0-7, output warps 8-11, issuer 12, copies 13, gate and
                                               // V warps 14 and 15
    static constexpr int LW = 256, OW = 128, CW = 64;
    // tensor memory columns
    static constexpr uint32_t TM_H = 0, TM_HF = 256, TM_D3 = 384, TM_COLS = 512;
};
struct SVec {
    float gC;
    float pad[3];
};
struct SSmall {
    uint64_t fullV[2], fullTB, fullQ[2], fullK, fullP;   // copies landed: V; T diag(beta); [-W; Q~]; K~; P^T
    uint64_t emptyV[2], emptyTB, emptyQ[2], emptyK;      // the products that read them have completed (MMA_U; MMA_U;
                                                         // MMA3; MMA4 + MMA5)
    uint64_t convU[2];                         // V written in fp16 (one arrival per converting warp)
    uint64_t m3, m4, m5;                       // product completions: Delta^T ready; H updated; O^T ready
    uint64_t ofree;                            // the output warps have read O of chunk t (phase t), one arrival each
    uint64_t staged, sfree;                    // O of chunk t is in the staging (one arrival per output warp); the
                                               // copies of chunk t have read it (output thread 0)
    uint64_t hready, dready;                   // h~ / Delta operands stored in tensor memory (one arrival per lane warp)
    uint64_t vready[2];                        // gamma_C of the ring slot written (one phase per two chunks)
    uint64_t vfree[2];                         // ... and read for the last time (one arrival per lane warp)
    uint32_t tmem_base;
    uint32_t pad;
    float gbuf[C];
};
constexpr uint32_t s_smem_bytes() { return SL::VEC + 2 * sizeof(SVec) + sizeof(SSmall) + 1024; }
static_assert(s_smem_bytes() <= 227 * 1024, "state kernel shared memory");

template <bool O_F32>
__global__ void __launch_bounds__(SL::THREADS, 1) gdn_state256_kernel(const __grid_constant__ CUtensorMap tmap_v,
                                                                      const __grid_constant__ CUtensorMap tmap_o,
                                                                      const SParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    SVec* vec = reinterpret_cast<SVec*>(smem + SL::VEC);
    SSmall& S = *reinterpret_cast<SSmall*>(smem + SL::VEC + 2 * sizeof(SVec));

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int vh = blockIdx.x & 1;                       // d_v half
    const GChain ch = g_resolve_chain(p.geo, blockIdx.x >> 1);
    const int n_chunks = (ch.len + C - 1) / C;
    const long slot0 = ch.row0 / C + ch.n;
    const int H = p.geo.H;

    if (warp == 12) {
        tmem_alloc(&S.tmem_base, SL::TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&S.fullTB, 1);
        mbar_init(&S.fullK, 1);
        mbar_init(&S.fullP, 1);
        mbar_init(&S.emptyTB, 1);
        mbar_init(&S.emptyK, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.fullV[s], 1);
            mbar_init(&S.emptyV[s], 1);
            mbar_init(&S.convU[s], SL::CW / 32);
            mbar_init(&S.fullQ[s], 1);
            mbar_init(&S.emptyQ[s], 1);
            mbar_init(&S.vready[s], 1);
            mbar_init(&S.vfree[s], SL::LW / 32);
        }
        mbar_init(&S.m3, 1);
        mbar_init(&S.m4, 1);
        mbar_init(&S.m5, 1);
        mbar_init(&S.ofree, SL::OW / 32);
        mbar_init(&S.staged, SL::OW / 32);
        mbar_init(&S.sfree, 1);
        mbar_init(&S.hready, SL::LW / 32);
        mbar_init(&S.dready, SL::LW / 32);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    // the per-chunk kernel has completed and its records are visible (with a programmatic launch this CTA may have
    // started before that; everything above reads only inputs)
    griddep_wait();

    bool ok = true;
    if (warp < 8) {
        // ---------------------------------------------------------------- lane warps: Delta and the state scaling
        const int q4 = warp & 3, hf = warp >> 2;
        const int dvr = 32 * q4 + lane;                  // d_v row of this thread within the half
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        // h[c][d_v] of this thread's row at sidx + c * D2
        const size_t sidx = ((size_t)ch.n * H + ch.h) * D2 * D2 + (size_t)vh * VT + dvr;
        bool finite = true;
        if (n_chunks == 0) {   // an empty sequence: the final state is the initial one
            if (p.hT)
                for (int c = 128 * hf; c < 128 * hf + 128; ++c)
                    p.hT[sidx + (size_t)c * D2] = p.h0 ? __ldg(p.h0 + sidx + (size_t)c * D2) : 0.f;
        } else {
            // h0: h~ = fp16(h0), H = gamma_C(0) h0
            ok = mbar_wait(&S.vready[0], 0, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            float gC = ok ? vec[0].gC : 0.f;
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.vfree[0]);
            if (ok) {
#pragma unroll 1
                for (int gq = 0; gq < 4; ++gq) {
                    const int c0 = 128 * hf + 32 * gq;
                    float x[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = p.h0 ? __ldg(p.h0 + sidx + (size_t)(c0 + j) * D2) : 0.f;
                    uint32_t pk[16], s0[16], s1[16];
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        pk[m] = pack_h2(x[2 * m], x[2 * m + 1]);
                        s0[m] = __float_as_uint(gC * x[m]);
                        s1[m] = __float_as_uint(gC * x[16 + m]);
                    }
                    tmem_st16(tl + SL::TM_HF + c0 / 2, pk);
                    tmem_st16(tl + SL::TM_H + c0, s0);
                    tmem_st16(tl + SL::TM_H + c0 + 16, s1);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.hready);
            }
            if (!ok && lane == 0) d_status(1u << 16);
            const uint32_t d3 = tl + SL::TM_D3;
            for (int t = 0; t < n_chunks && ok; ++t) {
                // Delta epilogue: Delta^T (columns 32 hf .. + 31 of D3) -> fp16 Delta^T in place, at columns 32 hf ..
                // + 15
                ok = mbar_wait(&S.m3, t & 1, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) d_status(16u);
                    break;
                }
                tc_fence_after();
                {
                    uint32_t r[2][16];
                    tmem_ld16(d3 + 32 * hf, r[0]);
                    tmem_ld16(d3 + 32 * hf + 16, r[1]);
                    tmem_ld_wait();
                    uint32_t da[16];
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const int k = 2 * m;
                        da[m] = pack_h2(__uint_as_float(r[k >> 4][k & 15]),
                                        __uint_as_float(r[(k + 1) >> 4][(k + 1) & 15]));
                    }
                    tmem_st16(d3 + 32 * hf, da);
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.dready);
                const bool last = t + 1 == n_chunks;
                if (!last) {   // gamma_C of the next chunk
                    const int u = t + 1;
                    ok = mbar_wait(&S.vready[u & 1], (u >> 1) & 1, kWaitNs);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) {
                        if (lane == 0) d_status(1u << 17);
                        break;
                    }
                    gC = vec[u & 1].gC;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.vfree[u & 1]);
                }
                // the state of the chunk's end: h~ = fp16(H) for MMA3 of the next chunk, 64 columns per tensor-memory
                // round trip (after the last chunk, the final state); then H <- gamma_C' H for its MMA4 while that MMA3
                // runs (MMA3 reads only h~; MMA4 is issued after this warp's next Delta epilogue)
                ok = mbar_wait(&S.m4, t & 1, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) d_status(32u);
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int hb = 0; hb < 2; ++hb) {
                    const int c0 = 128 * hf + 64 * hb;
                    uint32_t r[4][16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) tmem_ld16(tl + SL::TM_H + c0 + 16 * i, r[i]);
                    tmem_ld_wait();
                    if (last) {
                        if (p.hT) {
#pragma unroll
                            for (int j = 0; j < 64; ++j) {
                                const float hv = __uint_as_float(r[j >> 4][j & 15]);
                                finite = finite && isfinite(hv);
                                p.hT[sidx + (size_t)(c0 + j) * D2] = hv;
                            }
                        }
                    } else {
                        uint32_t pk[2][16];
#pragma unroll
                        for (int m = 0; m < 32; ++m) {
                            const int k = 2 * m;
                            pk[m >> 4][m & 15] = pack_h2(__uint_as_float(r[k >> 4][k & 15]),
                                                         __uint_as_float(r[(k + 1) >> 4][(k + 1) & 15]));
                        }
                        tmem_st16(tl + SL::TM_HF + c0 / 2, pk[0]);
                        tmem_st16(tl + SL::TM_HF + c0 / 2 + 16, pk[1]);
                    }
                }
                if (!last) {
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.hready);
#pragma unroll 1
                    for (int hb = 0; hb < 2; ++hb) {
                        const int c0 = 128 * hf + 64 * hb;
                        uint32_t r[4][16];
#pragma unroll
                        for (int i = 0; i < 4; ++i) tmem_ld16(tl + SL::TM_H + c0 + 16 * i, r[i]);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) r[i][j] = __float_as_uint(gC * __uint_as_float(r[i][j]));
                            tmem_st16(tl + SL::TM_H + c0 + 16 * i, r[i]);
                        }
                    }
                    tmem_st_wait();
                }
            }
        }
        if (__any_sync(0xffffffffu, !finite) && lane == 0) d_status(kStatusNonfinite);
    } else if (warp < 12) {
        // ---------------------------------------------------------------- output warps: O of each chunk
        const int q4 = warp & 3;
        const int dvr = 32 * q4 + lane;                  // d_v row of this thread within the half
        const int otid = tid - SL::LW;                   // 0 .. 127
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        bool finite = true;
        for (int t = 0; t < n_chunks && ok; ++t) {
            const int L = min(C, ch.len - t * C);
            // O^T = (Q~ h~)^T + Delta^T P^T: columns 64 .. 127 of D3, complete at m5
            ok = mbar_wait(&S.m5, t & 1, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) d_status(64u);
                break;
            }
            tc_fence_after();
            uint32_t a[4][16];
#pragma unroll
            for (int i0 = 0; i0 < 4; ++i0) tmem_ld16(tl + SL::TM_D3 + 64 + 16 * i0, a[i0]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.ofree);   // D3 may be overwritten from here
            // O^T to the staging as [token][d_v] rows in o's dtype, 32 tokens per round, each round out by one tensor
            // store (a partial half: its valid rows one by one) issued by output thread 0
            float nf = 0.f;    // stays 0 unless a written value is not finite (x * 0 is NaN for inf and NaN)
            const long orow0 = ch.row0 + (long)t * C;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                const int rnd = 2 * t + hb;
                if (ok && otid == 0 && rnd >= 1) {   // the previous round's copies have read the staging
                    bulk_wait_read();
                    mbar_arrive(&S.sfree);
                }
                if (ok && rnd >= 1) ok = mbar_wait(&S.sfree, (rnd - 1) & 1, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int tok = 32 * hb + i;
                    const float ov = __uint_as_float(a[tok >> 4][tok & 15]);
                    nf = tok < L ? fmaf(ov, 0.f, nf) : nf;
                    if (O_F32) sts32(sbase + SL::OST + 4 * (i * VT + dvr), __float_as_uint(ov));
                    else sts16(sbase + SL::OST + 2 * (i * VT + dvr), __bfloat16_as_ushort(__float2bfloat16_rn(ov)));
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.staged);
                if (otid == 0) {   // once all four warps' rows are staged
                    ok = mbar_wait(&S.staged, rnd & 1, kWaitNs);
                    const int nv = min(32, max(0, L - 32 * hb));   // valid rows of the round
                    if (ok && nv == 32) {
                        tma_store_3d(&tmap_o, smem + SL::OST, VT * vh, ch.h, (int)(orow0 + 32 * hb));
                    } else if (ok) {
                        constexpr uint32_t ES = O_F32 ? 4 : 2, RB = VT * ES;   // bytes of one staged row
                        for (int i = 0; i < nv; ++i)
                            bulk_s2g(static_cast<uint8_t*>(p.o) +
                                         (((size_t)(orow0 + 32 * hb + i) * H + ch.h) * D2 + (size_t)VT * vh) * ES,
                                     smem + SL::OST + i * RB, RB);
                    }
                    bulk_commit();
                }
                ok = __all_sync(0xffffffffu, ok);
            }
            finite = finite && nf == 0.f;
            if (!ok) {
                if (lane == 0) d_status(1u << 21);
                break;
            }
        }
        if (otid == 0) bulk_wait_all();                // the o rows are written before the CTA exits
        if (__any_sync(0xffffffffu, !finite) && lane == 0) d_status(kStatusNonfinite);
    } else if (warp == 12) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t id3 = idesc_f16(128, 128, false, false, false);  // h~^T (TMEM) x [-W; Q~]^T (K-major)
        const uint32_t id3h = idesc_f16(128, 64, false, false, false);  // the same, one half of [-W; Q~] (rows 0-63 or 64-127)
        const uint32_t idU = idesc_f16(128, 64, false, true, false);    // V^T (MN-major) x (T diag beta)^T
        const uint32_t id4 = idesc_f16(128, 256, false, false, true);   // Delta^T (TMEM) x K~ (MN-major)
        const uint32_t id5 = idesc_f16(128, 64, false, false, true);    // Delta^T (TMEM) x P^T (MN-major)
        if (lane == 0 && n_chunks > 0) {
            // shared-memory descriptors built once: a K step's offset goes into the start-address field (16-byte
            // units, no carry below 256 KB) by a plain add
            const uint64_t dQW0 = sdesc(sbase + SL::QW, 16, 1024), dQW1 = sdesc(sbase + SL::QW + SL::QW_STAGE, 16, 1024);
            const uint64_t dKF = sdesc(sbase + SL::KF, 8192, 1024), dPT = sdesc(sbase + SL::PT, 8192, 1024);
            const uint64_t dVF0 = sdesc(sbase + SL::VF, 8192, 1024), dVF1 = sdesc(sbase + SL::VF + 16384, 8192, 1024);
            const uint64_t dTB = sdesc(sbase + SL::TB, 16, 1024);
            const uint32_t d3 = tmem + SL::TM_D3;
            for (int t = 0; t < n_chunks && ok; ++t) {
                const int s = t & 1;
                const uint64_t dqw = s ? dQW1 : dQW0;
                // MMA_U: D3[:, 0:64] = V^T (T diag beta)^T, off the chain: it needs only D3 free (the output warps have
                // read O of chunk t - 1, which was complete with MMA4 and MMA5 of chunk t - 1, the readers of the Delta
                // half).  Each wait is a shared-memory access, slow under this kernel's traffic: the ones that have
                // normally completed come first, the one on the lane warps last.
                ok = (t == 0 || mbar_wait(&S.ofree, (t - 1) & 1, kWaitNs)) &&
                     mbar_wait(&S.convU[s], (t >> 1) & 1, kWaitNs) && mbar_wait(&S.fullTB, t & 1, kWaitNs);
                if (!ok) {
                    d_status(1024u);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(d3, (s ? dVF1 : dVF0) + ks * 128, dTB + ks * 2, idU, ks > 0 ? 1u : 0u);
                mma_commit(&S.emptyV[s]);
                mma_commit(&S.emptyTB);
                // MMA3: D3 += h~^T [-W; Q~]^T (N = 128, K = 256 = d_k): columns 0-63 become Delta^T; the first K step
                // starts columns 64-127 (the output's inter-chunk term) afresh
                ok = mbar_wait(&S.fullQ[s], (t >> 1) & 1, kWaitNs) && mbar_spin(&S.hready, t & 1, kWaitNs);
                if (!ok) {
                    d_status(1u << 14);
                    break;
                }
                tc_fence_after();
                mma_f16_ts(d3, tmem + SL::TM_HF, dqw, id3h, 1u);
                mma_f16_ts(d3 + 64, tmem + SL::TM_HF, dqw + 512, id3h, 0u);
#pragma unroll
                for (int ks = 1; ks < 16; ++ks)
                    mma_f16_ts(d3, tmem + SL::TM_HF + ks * 8, dqw + (ks >> 2) * 1024 + (ks & 3) * 2, id3, 1u);
                mma_commit(&S.emptyQ[s]);
                mma_commit(&S.m3);
                // MMA4: H += Delta^T K~ (N = 256, K = 64 tokens); A = the fp16 columns 32 hb .. + 15 of D3 (tokens
                // 32 hb .. + 31)
                ok = mbar_wait(&S.fullK, t & 1, kWaitNs) && mbar_wait(&S.fullP, t & 1, kWaitNs) &&
                     mbar_spin(&S.dready, t & 1, kWaitNs);
                if (!ok) {
                    d_status(512u);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16_ts(tmem + SL::TM_H, d3 + (ks >> 1) * 32 + (ks & 1) * 8, dKF + ks * 128, id4, 1u);
                mma_commit(&S.m4);
                // MMA5: D3[:, 64:128] += Delta^T P^T
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16_ts(d3 + 64, d3 + (ks >> 1) * 32 + (ks & 1) * 8, dPT + ks * 128, id5, 1u);
                mma_commit(&S.m5);
                mma_commit(&S.emptyK);
            }
        }
    } else if (warp == 13) {
        // ---------------------------------------------------------------- producer: TMA tiles and record copies
        if (lane == 0 && n_chunks > 0) {
            prefetch_tmap(&tmap_v);
            // Three streams, each refilled as soon as the products that read its buffers have completed: polled
            // without blocking, so that no stream waits behind another's buffer.  (-W, Q), two stages: MMA3 of chunk
            // t - 2 has read the stage (test 2: chunk t - 1's too).  V, two stages: MMA_U of chunk t - 2.  T diag(beta),
            // one stage: MMA_U of chunk t - 1.  (K~, P^T), one stage: MMA4 and MMA5 of chunk t - 1.
            int issQ = 0, issU = 0, issT = 0, issK = 0;   // chunks whose loads were issued, per stream
            uint64_t t_last = globaltimer_ns();            // the last progress
            while (issQ < n_chunks || issU < n_chunks || issT < n_chunks || issK < n_chunks) {
                bool progress = false;
                if (issQ < n_chunks) {
                    const int t = issQ, s = t & 1;
                    if ((t < 2 || mbar_test(&S.emptyQ[s], ((t >> 1) + 1) & 1)) &&
                        (p.test != 2 || t < 1 || mbar_test(&S.emptyQ[s ^ 1], ((t - 1) >> 1) & 1))) {
                        if (!(p.test == 1 && t == 0)) {   // test: the first chunk's -W and Q never arrive
                            const uint8_t* rec = p.ws + (size_t)((slot0 + t) * H + ch.h) * R_ITEM;
                            mbar_arrive_expect_tx(&S.fullQ[s], 65536);
                            bulk_g2s(smem + SL::QW + s * SL::QW_STAGE, rec + R_WQ, 65536, &S.fullQ[s]);
                        }
                        issQ = t + 1;
                        progress = true;
                    }
                }
                if (issU < n_chunks) {
                    const int t = issU, s = t & 1;
                    if (t < 2 || mbar_test(&S.emptyV[s], ((t >> 1) + 1) & 1)) {
                        const int r = (int)(ch.row0 + (long)t * C);
                        uint8_t* vf = smem + SL::VF + s * 16384;
                        mbar_arrive_expect_tx(&S.fullV[s], 16384);
                        tma_load_3d(vf, &tmap_v, &S.fullV[s], VT * vh, ch.h, r);
                        tma_load_3d(vf + 8192, &tmap_v, &S.fullV[s], VT * vh + 64, ch.h, r);
                        issU = t + 1;
                        progress = true;
                    }
                }
                if (issT < n_chunks) {
                    const int t = issT;
                    if (t < 1 || mbar_test(&S.emptyTB, (t - 1) & 1)) {
                        const uint8_t* rec = p.ws + (size_t)((slot0 + t) * H + ch.h) * R_ITEM;
                        mbar_arrive_expect_tx(&S.fullTB, 8192);
                        bulk_g2s(smem + SL::TB, rec + R_TB, 8192, &S.fullTB);
                        issT = t + 1;
                        progress = true;
                    }
                }
                if (issK < n_chunks) {
                    const int t = issK;
                    if (t < 1 || mbar_test(&S.emptyK, (t - 1) & 1)) {
                        const uint8_t* rec = p.ws + (size_t)((slot0 + t) * H + ch.h) * R_ITEM;
                        mbar_arrive_expect_tx(&S.fullK, 32768);
                        bulk_g2s(smem + SL::KF, rec + R_K, 32768, &S.fullK);
                        mbar_arrive_expect_tx(&S.fullP, 8192);
                        bulk_g2s(smem + SL::PT, rec + R_P, 8192, &S.fullP);
                        issK = t + 1;
                        progress = true;
                    }
                }
                if (progress) {
                    t_last = globaltimer_ns();
                } else {
                    if (globaltimer_ns() - t_last > kWaitNs) {
                        ok = false;
                        break;
                    }
                    __nanosleep(32);
                }
            }
            if (!ok) d_status(2048u);
            // copies issued whose barrier nobody waited on must land before the CTA exits: wait for every issued
            // phase (bounded)
            for (int t = (issU > 2 ? issU - 2 : 0); t < issU; ++t) mbar_wait(&S.fullV[t & 1], (t >> 1) & 1, kWaitNs);
            if (issT > 0) mbar_wait(&S.fullTB, (issT - 1) & 1, kWaitNs);
            if (issK > 0) mbar_wait(&S.fullK, (issK - 1) & 1, kWaitNs);
            if (issK > 0) mbar_wait(&S.fullP, (issK - 1) & 1, kWaitNs);
            for (int t = (issQ > 2 ? issQ - 2 : 0); t < issQ; ++t)
                if (!(p.test == 1 && t == 0)) mbar_wait(&S.fullQ[t & 1], (t >> 1) & 1, kWaitNs);
        }
    } else {
        // ---------------------------------------------------------------- warps 14 and 15: V in fp16, half of each
        // tile per warp (rows past the end: zeros); warp 15 first computes each chunk's gamma_C
        const int cidx = tid - (SL::THREADS - SL::CW);   // 0 .. 63
        float gn[2] = {0.f, 0.f};
        auto load_g = [&](int t, float (&gg)[2]) {
            const int Lt = min(C, ch.len - t * C);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int r = lane + 32 * k;
                gg[k] = r < Lt ? act_gate(p.act, __ldg(p.g + (size_t)(ch.row0 + (long)t * C + r) * H + ch.h), ch.h) : 0.f;
            }
        };
        if (warp == 15 && n_chunks > 0) load_g(0, gn);
        for (int u = 0; u < n_chunks && ok; ++u) {
            const int slot = u & 1;
            if (warp == 15) {
                // gamma_C of chunk u, into ring slot u % 2 once its readers have released it (chunk u - 2)
                if (u >= 2) ok = mbar_wait(&S.vfree[slot], ((u >> 1) + 1) & 1, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) d_status(8192u);
                    break;
                }
                S.gbuf[lane] = gn[0];
                S.gbuf[lane + 32] = gn[1];
                __syncwarp();
                float G0, G1, Gl;
                gate_prefix2(S.gbuf[2 * lane], S.gbuf[2 * lane + 1], lane, G0, G1, Gl);
                if (lane == 0) vec[slot].gC = ex2(Gl);
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.vready[slot]);
                if (u + 1 < n_chunks) load_g(u + 1, gn);
            }
            // V of chunk u, in place in its stage
            ok = mbar_wait(&S.fullV[u & 1], (u >> 1) & 1, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) d_status(4096u);
                break;
            }
            const uint32_t vf = sbase + SL::VF + (u & 1) * 16384;
            tile_to_f16<SL::CW, false>(vf, vf, 8192, min(C, ch.len - u * C), cidx, 0u);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.convU[u & 1]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 12) tmem_dealloc(tmem, SL::TM_COLS);
}

long n_slots256(const ChunkArgs& a) { return (long)a.B * a.T / C + a.N() + 1; }

}  // namespace

size_t gdn_d256_workspace_bytes(const ChunkArgs& a) {
    if ((long)a.B * a.T == 0) return 0;
    return (size_t)n_slots256(a) * a.H * R_ITEM;
}

cudaError_t launch_chunk_gdn_d256(const ChunkArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t s) {
    const long chains = (long)a.N() * a.H;
    if (chains == 0) return cudaSuccess;
    if (!device_is_sm100_family()) return cudaErrorNoKernelImageForDevice;
    const long rows = (long)a.B * a.T;
    if (rows == 0) {
        if (a.hT) {
            const size_t bytes = (size_t)a.N() * a.H * D2 * D2 * sizeof(float);
            return a.h0 ? cudaMemcpyAsync(a.hT, a.h0, bytes, cudaMemcpyDeviceToDevice, s)
                        : cudaMemsetAsync(a.hT, 0, bytes, s);
        }
        return cudaSuccess;
    }
    const size_t need = gdn_d256_workspace_bytes(a);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % 256) != 0)
        return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, rows, a.HK(), D2) || !make_map(&mk, a.k, rows, a.HK(), D2) ||
        !make_map(&mv, a.v, rows, a.H, D2))
        return cudaErrorInvalidValue;
    Geo geo{a.cu, a.n_seqs, a.B, a.T, a.H};
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long items = n_slots256(a) * a.H;
    IParams ip{geo, a.g, a.beta, a.scale, n_slots256(a), static_cast<uint8_t*>(workspace), a.act, a.H / a.HK()};
    e = cudaFuncSetAttribute(gdn_intra256_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)I_SMEM);
    if (e != cudaSuccess) return e;
    const long grid1 = items < (long)I_CTAS_PER_SM * sms ? items : (long)I_CTAS_PER_SM * sms;
    gdn_intra256_kernel<<<(unsigned)grid1, I_THREADS, I_SMEM, s>>>(mq, mk, ip);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    SParams sp{geo, a.g, a.scale, a.h0, a.hT, a.o, static_cast<const uint8_t*>(workspace), a.act, a.H / a.HK(),
               a.test_fwd};
    CUtensorMap mo;
    if (!make_map_rows(&mo, a.o, rows, a.H, D2, a.o_f32 != 0, VT, 32)) return cudaErrorInvalidValue;
    auto launch2 = [&](auto kern) -> cudaError_t {
        cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s_smem_bytes());
        if (e2 != cudaSuccess) return e2;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)(2 * chains));
        cfg.blockDim = dim3(SL::THREADS);
        cfg.dynamicSmemBytes = s_smem_bytes();
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, mv, mo, sp);
    };
    e = a.o_f32 ? launch2(gdn_state256_kernel<true>) : launch2(gdn_state256_kernel<false>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t d256_read_and_clear_status(unsigned* value, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_d256_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    if (clear && *value) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_d256_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace gdn
