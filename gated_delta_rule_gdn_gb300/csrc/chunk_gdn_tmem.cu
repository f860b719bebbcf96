// Scalar-gate (GDN) chunk forward in two passes on tcgen05 tensor cores (sm_103a): bf16 q/k/v, d_k = d_v = 128,
// chunk C = 64, fp32 state, o in fp32 or bf16.
//
// The algebra is the chunkwise WY/UT form of "TileLang 实战：KDA 从零到一 -- Gated DeltaNet", §2.3, split the way
// "Gated Delta Network (GDN)", §4(b3)-(d) splits it: the state-independent products of every chunk first, then the
// serial state pass.  Per chunk of L <= C rows, with G the within-chunk cumulative log gate (log2 units in the
// kernels), gamma_i = 2^{G_i}, Gamma_ij = 2^{G_i - G_j} (j <= i):
//   A = diag(beta)(Gamma * K K^T) strictly lower,  P = scale (Gamma * Q K^T) lower including the diagonal,
//   T = (I + A)^{-1},  W = T diag(beta gamma) K,  U = T diag(beta) V,
// and, with h = S^T [d_k, d_v] entering the chunk,
//   Delta = U - W h,  O = scale diag(gamma) Q h + P Delta,  h <- gamma_C h + K~^T Delta,  K~ = diag(gamma_C / gamma) K.
//
// Pass 1, gdn_intra_kernel: one item per (chunk slot, head); persistent CTAs, two per SM.  Per item: MMA0 = [K; Q] K^T
// (raw bf16 tiles) gives A (fp32, for the solve) and P; the blocked inverse T = (I + A)^{-1} in place; MMA2 =
// [T diag(beta gamma); same] K (the raw K tile again, as an MN-major operand) gives W.  The item's workspace record is
// -W, P and T diag(beta) (fp16), 32 KB, already in the operand layouts of pass 2.  q and k are the only
// tensors it reads.
//
// Pass 2, gdn_state_kernel: one CTA per (sequence, head) chain over the whole d_v.  It works in the transposed
// orientation (tensor-memory lane = d_v row), so that the operands that change along the chain stay in tensor memory:
//   MMA_U  D3[:, 0:64] = U^T = V^T (T diag beta)^T                 (V converted to fp16 in the kernel)
//   MMA3   D3 += h~^T [-W; Q~]^T,  Q~ = diag(scale gamma) Q         (A = h~^T, the state's fp16 copy, in tensor
//          memory; Q scaled and converted to fp16 in the kernel): columns 0-63 become Delta^T, 64-127 (Q~ h~)^T
//   Delta epilogue: Delta^T to fp16, in place in tensor memory
//   MMA45  D45 = Delta^T [K~ | P^T],  K~ = diag(gamma_C / gamma) K  (K scaled and converted to fp16 in the kernel):
//          columns 0-127 (K~^T Delta)^T, 128-191 (P Delta)^T
//   h <- gamma_C h + D45[:, 0:128] (registers, thread = d_v row; h~^T back to tensor memory);
//   O^T = D3[:, 64:128] + D45[:, 128:192].
// The serial chain is MMA3 -> Delta epilogue -> MMA45 -> state update, with no shared-memory round trip.  The tensor
// core instructions of a chunk are few and wide (8 + 4 + 4: a single issuing thread spends about as long on an
// instruction of N <= 128 as the tensor core spends on one of N = 256).  Sixteen warps share the work: eight lane
// warps (two per tensor-memory lane quarter) hold h in registers, write the Delta and h~ operands and convert Q and
// K; one issues the products, one the copies; two compute the gate vectors and convert V; four (one per lane quarter)
// copy O out of tensor memory and store it.  The lane warps run with 168 registers, the rest with 88.
//
// Operand precision: every operand of the state pass is fp16 (h~, -W, P, T diag(beta), Delta, and q, k, v converted
// from bf16 in the kernel, q and k with their gate factors applied first); the per-chunk kernel's products read the
// raw bf16 q and k, with T diag(beta gamma) rounded to bf16 for W (a rounding that changes the error measurably
// nowhere: W itself is stored in fp16).  A bf16 copy of the state for the output product Q h~ would break the 2e-2
// max-error bound.  fp16 saturates at 65,504: an intermediate beyond that becomes inf and the output or final state
// non-finite; the state kernel checks what it writes and sets the non-finite bit of the device status
// (gdn_device_status then reports GDN_ERR_NONFINITE).
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

__device__ unsigned g_gt_status;

namespace {

// workspace record of one (chunk slot, head) item
constexpr uint32_t GW_W = 0;         // -W fp16 [token][d_k], two 64-column slabs of 64 rows x 128 B, 128-byte swizzle
constexpr uint32_t GW_P = 16384;     // P^T fp16 [j][i], 64 rows x 128 B, 128-byte swizzle
constexpr uint32_t GW_TB = 24576;    // T diag(beta) fp16 [i][j], 64 rows x 128 B, 128-byte swizzle
constexpr uint32_t GW_ITEM = 32768;


__device__ __forceinline__ void gt_status(unsigned bit) { atomicOr(&g_gt_status, bit); }

// ==================================================================== pass 1: per-chunk products
struct GIntraParams {
    Geo geo;
    const float* g;
    const float* beta;
    float scale;
    long n_slots;
    uint8_t* ws;
    GateAct act;
    int group;    // value heads per key head
};

// shared memory of pass 1 (byte offsets from a 1024-aligned base); 65 KB, so that three CTAs fit on an SM
constexpr uint32_t GI_KQ = 0;         // [K; Q]: per 64-column slab 64 K rows then 64 Q rows (16 KB)
constexpr uint32_t GI_A1 = 32768;     // [T diag(beta gamma); same] bf16 K-major 128 x 64 (operand A of MMA2); the
                                      // solve's scratch before that
constexpr uint32_t GI_PS = 8192;      // P fp16 staging for the bulk copy, in the Q rows of the first slab (dead once
                                      // MMA0 has read them)
constexpr uint32_t GI_AM = 49152;     // fp32 A, then T in place (row stride TS); then -W staging (16 KB)
constexpr uint32_t GI_END = GI_AM + 64 * TS * 4;
static_assert(32 * RS * 4 <= 16384, "the solve scratch must fit in A1");
static_assert(64 * TS * 4 >= 16384, "-W staging must fit in the A buffer");

struct GISmall {
    uint64_t full_kq;
    uint64_t m0, m2;
    uint32_t tmem_base;
    uint32_t pad;
    float gbuf[C];       // g of the item (0 past the end)
    float bbuf[C];       // beta of the item (0 past the end)
    float lg[C];         // log2 cumulative gate
    float bg[C];         // beta_j gamma_j
};
constexpr uint32_t GI_SMEM = GI_END + sizeof(GISmall) + 1024;
constexpr int GI_THREADS = 256;
constexpr int GI_CTAS_PER_SM = 3;
constexpr uint32_t GI_TM_COLS = 128;   // D0 (64 columns) and, after the solve, D2 (128 columns) at column 0

__global__ void __launch_bounds__(GI_THREADS, GI_CTAS_PER_SM)
gdn_intra_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                 const GIntraParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    GISmall& S = *reinterpret_cast<GISmall*>(smem + GI_END);
    float* Am = reinterpret_cast<float*>(smem + GI_AM);
    float* Rt = reinterpret_cast<float*>(smem + GI_A1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, pw = warp >> 2;
    const int row = 32 * q4 + lane;
    const bool leader = (tid == 0);
    const bool loader = (tid == 64);
    const int H = p.geo.H;
    griddep_launch_dependents();

    if (warp == 0) {
        tmem_alloc(&S.tmem_base, GI_TM_COLS);
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
        uint8_t* kq = smem + GI_KQ;
        mbar_arrive_expect_tx(&S.full_kq, 32768);
        tma_load_3d(kq, &tmap_k, &S.full_kq, 0, hk, r);
        tma_load_3d(kq + 8192, &tmap_q, &S.full_kq, 0, hk, r);
        tma_load_3d(kq + 16384, &tmap_k, &S.full_kq, 64, hk, r);
        tma_load_3d(kq + 16384 + 8192, &tmap_q, &S.full_kq, 64, hk, r);
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
        uint8_t* kq = smem + GI_KQ;
        uint8_t* rec = p.ws + (size_t)it.it * GW_ITEM;
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
        if (!ok && tid == 0) gt_status(1u);
        if (ok && loader) waited = ic + 1;
        // MMA0: D0 = [K; Q] K^T (M = 128, N = 64, K = 128)
        if (ok && leader) {
            tc_fence_after();
            const uint32_t id = idesc_f16(128, 64, true, false, false);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t a = smem_u32(kq) + (ks >> 2) * 16384 + (ks & 3) * 32;
                mma_f16(tmem, sdesc(a, 16, 1024), sdesc(a, 16, 1024), id, ks > 0);
            }
            mma_commit(&S.m0);
        }
        // the previous item's -W copy has read its staging (the A buffer)
        if (lane == 0) bulk_wait_read();
        if (ok && leader) ok = mbar_wait(&S.m0, par, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && leader) gt_status(2u);
        tc_fence_before();
        __syncthreads();   // [B] D0 ready; the staging buffers are free
        tc_fence_after();
        if (ok) epilogue_kkt<false>(tl, row, q4, pw, S.lg, S.bbuf, p.scale, Am, smem + GI_PS - 8192);
        fence_async_smem();   // P staging is read by the bulk copy
        tc_fence_before();
        __syncthreads();   // [C] A and P are in shared memory
        if (ok && tid == 96) {
            bulk_s2g(rec + GW_P, smem + GI_PS, 8192);
            bulk_commit();
        }
        // UT transform, T = (I + A)^{-1} in place (the scratch is A1, dead until the scalings below)
        solve_unit_lower_inplace(Am, Rt, tid, ok);
        // T diag(beta gamma) in bf16 into both row halves of A1 (operand A of MMA2), and T diag(beta) in fp16 straight
        // to the record.  Thread e: row i = e / 8, physical 16-byte chunk pc = e % 8 of the swizzled row (logical
        // columns 8 (pc ^ (i % 8)) ..); consecutive lanes write consecutive 16 bytes of a record row.
        if (ok) {
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
                const int e = tid + GI_THREADS * k2, i = e >> 3, pc = e & 7, c0 = (pc ^ (i & 7)) << 3;
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
                st16(smem + GI_A1 + o, g0, g1, g2, g3);
                st16(smem + GI_A1 + 8192 + o, g0, g1, g2, g3);
                stg16(rec + GW_TB + o, pack_h2(tb[0], tb[1]), pack_h2(tb[2], tb[3]), pack_h2(tb[4], tb[5]),
                      pack_h2(tb[6], tb[7]));
            }
        }
        fence_async_smem();
        tc_fence_before();
        if (tid == 96) bulk_wait_read();   // the copy of P has read its staging in the [K; Q] buffer
        __syncthreads();   // [D] A1 ready; every read of T is done; P is out of the [K; Q] buffer
        // MMA2: D2 = A1 K (M = 128, N = 128 = d_k, K = 64 tokens; K is the MN-major view of the raw K tile)
        if (ok && leader) {
            tc_fence_after();
            const uint32_t id = idesc_f16(128, 128, true, false, true);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f16(tmem, sdesc(sbase + GI_A1 + ks * 32, 16, 1024), sdesc(smem_u32(kq) + ks * 2048, 16384, 1024),
                        id, ks > 0);
            mma_commit(&S.m2);
        }
        if (ok) ok = mbar_wait(&S.m2, par, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && tid == 0) gt_status(4u);
        // MMA2 has read K: the next item's K and Q can land (its loads overlap this item's epilogue and the next
        // item's gate prefix; the other CTAs on the SM cover the rest of their latency)
        if (ok && loader && have_next) {
            issue_kq(nx);
            issued = ic + 2;
        }
        tc_fence_after();
        // epilogue 2: -W in fp16 into the A buffer (now dead) as [token][d_k] in two swizzled 64-column slabs.  D2's
        // two row halves are alike, so warp (q4, pw) takes token rows 32 (q4 % 2) .. + 31 and d_k columns
        // 32 (2 (q4 / 2) + pw) .. + 31.
        if (ok) {
            const int tr = 32 * (q4 & 1) + lane, cq = 2 * (q4 >> 1) + pw;
            uint32_t r[2][16];
            tmem_ld16(tl + cq * 32, r[0]);
            tmem_ld16(tl + cq * 32 + 16, r[1]);
            tmem_ld_wait();
            uint8_t* wst = smem + GI_AM + (cq >> 1) * 8192;
#pragma unroll
            for (int h8 = 0; h8 < 4; ++h8) {
                uint32_t w4[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int k = h8 * 8 + 2 * m;
                    w4[m] = pack_h2(-__uint_as_float(r[k >> 4][k & 15]), -__uint_as_float(r[(k + 1) >> 4][(k + 1) & 15]));
                }
                st16(wst + sw128_off(tr, (cq & 1) * 32 + h8 * 8), w4[0], w4[1], w4[2], w4[3]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();   // [E] -W staged
        if (ok && tid == 0) {
            bulk_s2g(rec + GW_W, smem + GI_AM, 16384);
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
    if (warp == 0) tmem_dealloc(tmem, GI_TM_COLS);
}

// ==================================================================== pass 2: state pass
struct GStateParams {
    Geo geo;
    const float* g;
    float scale;
    const float* h0;
    float* hT;
    void* o;
    const uint8_t* ws;
    GateAct act;
    int group;
    int test;     // 1: leave out the first record copy (the waits for it run out); 2: a one-chunk-deep ring
};

// Shared memory of pass 2: two stages of a chunk's operands, then a four-deep ring of its gate vectors.
struct GL {
    static constexpr uint32_t QW = 0;          // [-W; Q~] fp16 K-major, two 64-column slabs of 128 rows (16 KB each):
                                               // rows 0-63 -W (record), rows 64-127 Q (TMA, bf16) -> Q~ in place
    static constexpr uint32_t KF = 32768;      // [K~ | P^T] MN-major operand of MMA45, three 64-column slabs of 64
                                               // rows: K (TMA, bf16) -> K~ fp16 in place, then P^T (record)
    static constexpr uint32_t VF = 57344;      // V tile (TMA, bf16) -> fp16 in place; MN-major operand of MMA_U
    static constexpr uint32_t TB = 73728;      // T diag(beta) fp16 (record)
    static constexpr uint32_t STAGE = 81920;
    static constexpr uint32_t OST = 2 * STAGE; // o of one chunk, [64 tokens][128] in o's dtype (32 KB for fp32)
    static constexpr uint32_t VEC = OST + 32768;   // 4 x GVec
    static constexpr int LW = 256;             // the lane warps: 8, two per tensor-memory lane quarter
    static constexpr int OW = 128;             // the output warps: 4, one per lane quarter
    static constexpr int THREADS = 512;        // + issuer, producer, 2 converter warps, then the output warps
    // registers per thread: 128 at launch; the lane warps raise theirs, the other two warpgroups lower theirs
    static constexpr uint32_t REG_LAUNCH = 128, REG_LANE = 168, REG_REST = 88;
    // tensor memory columns
    static constexpr uint32_t TM_HT = 0, TM_D3 = 64, TM_D45 = 320, TM_COLS = 512;
};
struct GVec {
    float qs[C];     // scale gamma_i (the rows of Q)
    float kd[C];     // gamma_C / gamma_i (the rows of K)
    float gC;
    float pad[3];
};
struct GSmall {
    uint64_t fullU[2], fullQ[2], fullK[2];     // TMA / bulk copies landed: V + T diag(beta); Q + -W; K + P^T
    uint64_t emptyU[2], emptyQ[2], emptyK[2];  // the products that read them have completed
    uint64_t convU[2], convQ[2], convK[2];     // V, Q and K converted to fp16 (one arrival per converter, output or
                                               // lane warp)
    uint64_t m3, m4;                           // product completions (MMA3; MMA45)
    uint64_t ofree;                            // the output warps have zeroed the output halves of D3 (phase 0), then
                                               // read D45 and the output half of chunk t (phase t + 1); one arrival
                                               // per output warp
    uint64_t hready, dready;                   // h~ / Delta operands stored in tensor memory (one arrival per lane warp)
    uint64_t vready[4];                        // gate vectors of the ring slot written (one phase per four chunks)
    uint64_t vfree[4];                         // ... and read for the last time (one arrival per lane warp)
    uint32_t tmem_base;
    uint32_t pad;
    float gbuf[C];
};
constexpr uint32_t gs_smem_bytes() { return GL::VEC + 4 * sizeof(GVec) + sizeof(GSmall) + 1024; }
static_assert(gs_smem_bytes() <= 227 * 1024, "state kernel shared memory");
static_assert(GL::LW * GL::REG_LANE + (GL::THREADS - GL::LW) * GL::REG_REST <= GL::THREADS * GL::REG_LAUNCH,
              "register split above the launch budget");

__device__ __forceinline__ void tmem_st_zero16(uint32_t taddr) {
    const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    tmem_st16(taddr, z);
}

template <bool O_F32>
__global__ void __launch_bounds__(GL::THREADS, 1) gdn_state_kernel(const __grid_constant__ CUtensorMap tmap_q,
                                                                   const __grid_constant__ CUtensorMap tmap_k,
                                                                   const __grid_constant__ CUtensorMap tmap_v,
                                                                   const __grid_constant__ CUtensorMap tmap_o,
                                                                   const GStateParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    GVec* vec = reinterpret_cast<GVec*>(smem + GL::VEC);
    GSmall& S = *reinterpret_cast<GSmall*>(smem + GL::VEC + 4 * sizeof(GVec));

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const GChain ch = g_resolve_chain(p.geo, blockIdx.x);
    const int n_chunks = (ch.len + C - 1) / C;
    const long slot0 = ch.row0 / C + ch.n;
    const int H = p.geo.H;
    const int hk = ch.h / p.group;

    if (warp == 8) {
        tmem_alloc(&S.tmem_base, GL::TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.fullU[s], 1);
            mbar_init(&S.fullQ[s], 1);
            mbar_init(&S.fullK[s], 1);
            mbar_init(&S.emptyU[s], 1);
            mbar_init(&S.emptyQ[s], 1);
            mbar_init(&S.emptyK[s], 1);
            mbar_init(&S.convU[s], 2);
            mbar_init(&S.convQ[s], GL::LW / 32);
            mbar_init(&S.convK[s], GL::LW / 32);
        }
        mbar_init(&S.m3, 1);
        mbar_init(&S.m4, 1);
        mbar_init(&S.ofree, GL::OW / 32);
        mbar_init(&S.hready, GL::LW / 32);
        mbar_init(&S.dready, GL::LW / 32);
        for (int v = 0; v < 4; ++v) {
            mbar_init(&S.vready[v], 1);
            mbar_init(&S.vfree[v], GL::LW / 32);
        }
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    // the per-chunk kernel has completed and its records are visible (with a programmatic launch this CTA may have
    // started before that; everything above reads only inputs)
    griddep_wait();

    if (warp < 8) setmaxnreg_inc<GL::REG_LANE>();
    else setmaxnreg_dec<GL::REG_REST>();

    bool ok = true;
    if (warp < 8) {
        // ---------------------------------------------------------------- lane warps: the state chain
        const int q4 = warp & 3, hf = warp >> 2;
        const int dvr = 32 * q4 + lane;                  // d_v row of this thread
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        const size_t sbase_idx = ((size_t)ch.n * H + ch.h) * DK * DV + dvr;   // h[c][dvr] at + c * DV
        float h[64];                                     // h[64 hf + c][dvr]
#pragma unroll
        for (int c = 0; c < 64; ++c) h[c] = p.h0 ? __ldg(p.h0 + sbase_idx + (size_t)(64 * hf + c) * DV) : 0.f;
        {   // h~^T to tensor memory (fp16 pairs along d_k)
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = pack_h2(h[2 * c], h[2 * c + 1]);
            tmem_st16(tl + GL::TM_HT + 32 * hf, *reinterpret_cast<uint32_t(*)[16]>(pk));
            tmem_st16(tl + GL::TM_HT + 32 * hf + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.hready);
        }
        // Q or K of chunk u to fp16 in place, row i of Q scaled by scale gamma_i, row j of K by gamma_C / gamma_j (rows
        // past the end: zeros), so that MMA3 gives the output's inter-chunk term and MMA45 the state's increment
        // directly.  K of chunk t + 1 is converted in the wait for MMA45 of chunk t, Q of chunk t + 2 in the wait for
        // MMA3 of chunk t + 1.
        auto convert = [&](bool is_q, int u) -> bool {
            const int su = u & 1;
            bool okc = mbar_wait(is_q ? &S.fullQ[su] : &S.fullK[su], (u >> 1) & 1, kWaitNs);
            if (okc) okc = mbar_wait(&S.vready[u & 3], (u >> 2) & 1, kWaitNs);
            okc = __all_sync(0xffffffffu, okc);
            if (!okc) return false;
            if (is_q)
                tile_to_f16<GL::LW, true>(sbase + su * GL::STAGE + GL::QW + 8192, sbase + su * GL::STAGE + GL::QW + 8192,
                                          16384, min(C, ch.len - u * C), tid, smem_u32(vec[u & 3].qs));
            else
                tile_to_f16<GL::LW, true>(sbase + su * GL::STAGE + GL::KF, sbase + su * GL::STAGE + GL::KF, 8192,
                                          min(C, ch.len - u * C), tid, smem_u32(vec[u & 3].kd));
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(is_q ? &S.convQ[su] : &S.convK[su]);
            return true;
        };
        for (int u = 0; u < min(n_chunks, 2) && ok; ++u) ok = convert(true, u);
        if (ok && n_chunks > 0) ok = convert(false, 0);
        if (!ok && lane == 0) gt_status(1u << 15);
        bool finite = true;
        for (int t = 0; t < n_chunks && ok; ++t) {
            const int s = t & 1;
            const GVec& V = vec[t & 3];
            const uint32_t d3 = tl + GL::TM_D3 + 128 * s;
            // Delta epilogue: Delta^T (columns 32 hf .. + 31 of D3) -> fp16 Delta^T in place, at columns 32 hf .. + 15
            if (ok) ok = mbar_wait(&S.m3, t & 1, kWaitNs);
            if (ok) ok = mbar_wait(&S.vready[t & 3], (t >> 2) & 1, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) gt_status(16u);
                break;
            }
            tc_fence_after();
            float gC;
            {
                uint32_t r[2][16];
                tmem_ld16(d3 + 32 * hf, r[0]);
                tmem_ld16(d3 + 32 * hf + 16, r[1]);
                tmem_ld_wait();
                gC = V.gC;   // the last read of this chunk's gate vectors
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.vfree[t & 3]);
                uint32_t da[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const int k = 2 * m;
                    da[m] = pack_h2(__uint_as_float(r[k >> 4][k & 15]), __uint_as_float(r[(k + 1) >> 4][(k + 1) & 15]));
                }
                tmem_st16(d3 + 32 * hf, da);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.dready);
            if (t + 1 < n_chunks && !convert(false, t + 1)) {   // while MMA45 runs
                ok = false;
                if (lane == 0) gt_status(1u << 15);
                break;
            }
            // state update: h <- gamma_C h + D4 (columns 64 hf .. + 63 of D45), h~^T back to tensor memory
            if (ok) ok = mbar_wait(&S.m4, t & 1, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) gt_status(32u);
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r[2][16];
                tmem_ld16(tl + GL::TM_D45 + 64 * hf + 32 * half, r[0]);
                tmem_ld16(tl + GL::TM_D45 + 64 * hf + 32 * half + 16, r[1]);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const int c = 32 * half + 2 * m;
                    h[c] = fmaf(gC, h[c], __uint_as_float(r[(2 * m) >> 4][(2 * m) & 15]));
                    h[c + 1] = fmaf(gC, h[c + 1], __uint_as_float(r[(2 * m + 1) >> 4][(2 * m + 1) & 15]));
                    pk[m] = pack_h2(h[c], h[c + 1]);
                }
                tmem_st16(tl + GL::TM_HT + 32 * hf + 16 * half, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.hready);
            if (t + 2 < n_chunks && !convert(true, t + 2)) {   // while MMA3 of chunk t + 1 runs
                ok = false;
                if (lane == 0) gt_status(1u << 15);
                break;
            }
        }
        if (ok && p.hT) {
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                finite = finite && isfinite(h[c]);
                p.hT[sbase_idx + (size_t)(64 * hf + c) * DV] = h[c];
            }
        }
        if (__any_sync(0xffffffffu, !finite) && lane == 0) gt_status(kStatusNonfinite);
    } else if (warp >= 12) {
        // ---------------------------------------------------------------- output warps: O of each chunk
        const int q4 = warp & 3;
        const int dvr = 32 * q4 + lane;                  // d_v row of this thread
        const int otid = tid - (GL::THREADS - GL::OW);   // 0 .. 127
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        // zeros in the output halves of both D3 buffers (MMA3 accumulates onto them), published to the issuer by a
        // first arrival on ofree
        for (int s = 0; s < 2; ++s)
            for (int c = 0; c < 64; c += 16) tmem_st_zero16(tl + GL::TM_D3 + 128 * s + 64 + c);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.ofree);
        bool finite = true;
        for (int t = 0; t < n_chunks && ok; ++t) {
            const int s = t & 1;
            const uint32_t d3 = tl + GL::TM_D3 + 128 * s;
            const int L = min(C, ch.len - t * C);
            // O^T = h~^T (diag(scale gamma) Q)^T (columns 64 .. 127 of D3, from MMA3) + Delta^T P^T (columns 128 ..
            // 191 of D45, from MMA45; both complete at m4), staged in shared memory as [token][d_v] rows and written
            // by one tensor store (a partial chunk: one bulk copy per valid token row)
            ok = mbar_wait(&S.m4, t & 1, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) gt_status(64u);
                break;
            }
            tc_fence_after();
            if (otid < C) bulk_wait_read();   // the previous chunk's copies have read the staging
            named_bar(2, GL::OW);
            float nf = 0.f;    // stays 0 unless a written value is not finite (x * 0 is NaN for inf and NaN)
#pragma unroll
            for (int i0 = 0; i0 < C; i0 += 16) {   // 16 tokens at a time
                uint32_t a[16], b[16];
                tmem_ld16(d3 + 64 + i0, a);
                tmem_ld16(tl + GL::TM_D45 + 128 + i0, b);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float ov = __uint_as_float(a[k]) + __uint_as_float(b[k]);
                    nf = i0 + k < L ? fmaf(ov, 0.f, nf) : nf;
                    if (O_F32) sts32(sbase + GL::OST + 4 * ((i0 + k) * DV + dvr), __float_as_uint(ov));
                    else sts16(sbase + GL::OST + 2 * ((i0 + k) * DV + dvr), __bfloat16_as_ushort(__float2bfloat16_rn(ov)));
                }
            }
            finite = finite && nf == 0.f;
            // the output half of D3 back to zero for MMA3 two chunks on; D45 may be overwritten from here
            for (int c = 0; c < 64; c += 16) tmem_st_zero16(d3 + 64 + c);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.ofree);
            fence_async_smem();
            named_bar(2, GL::OW);
            const long orow0 = ch.row0 + (long)t * C;
            if (L == C) {   // a full chunk: one tensor store of the [64][128] tile
                if (otid == 0) {
                    tma_store_3d(&tmap_o, smem + GL::OST, 0, ch.h, (int)orow0);
                    bulk_commit();
                }
            } else if (otid < L) {   // a sequence's last, partial chunk: its valid rows one by one
                constexpr uint32_t RB = DV * (O_F32 ? 4 : 2);   // bytes of one o row
                uint8_t* orow = static_cast<uint8_t*>(p.o) + ((size_t)(orow0 + otid) * H + ch.h) * RB;
                bulk_s2g(orow, smem + GL::OST + otid * RB, RB);
                bulk_commit();
            }
        }
        if (otid < C) bulk_wait_all();                 // the o rows are written before the CTA exits
        if (__any_sync(0xffffffffu, !finite) && lane == 0) gt_status(kStatusNonfinite);
    } else if (warp == 8) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t idU = idesc_f16(128, 64, false, true, false);    // V^T (MN-major) x (T diag beta)^T
        const uint32_t id3 = idesc_f16(128, 128, false, false, false);  // h~^T (TMEM) x [-W; Q~]^T (K-major)
        const uint32_t id45 = idesc_f16(128, 192, false, false, true);  // Delta^T (TMEM) x [K~ | P^T] (MN-major)
        if (lane == 0 && n_chunks > 0) {
            // the shared-memory descriptors of both stages, built once: a K step's offset goes into the start-address
            // field (16-byte units, no carry below 256 KB) by a plain add, so the issue loops stay short
            const uint64_t dQW0 = sdesc(sbase + GL::QW, 16, 1024), dQW1 = sdesc(sbase + GL::STAGE + GL::QW, 16, 1024);
            const uint64_t dKF0 = sdesc(sbase + GL::KF, 8192, 1024), dKF1 = sdesc(sbase + GL::STAGE + GL::KF, 8192, 1024);
            const uint64_t dVF0 = sdesc(sbase + GL::VF, 8192, 1024), dVF1 = sdesc(sbase + GL::STAGE + GL::VF, 8192, 1024);
            const uint64_t dTB0 = sdesc(sbase + GL::TB, 16, 1024), dTB1 = sdesc(sbase + GL::STAGE + GL::TB, 16, 1024);
            // MMA_U of chunk u, K steps k0 .. k1 - 1 of 4: D3[0:64] = V^T (T diag beta)^T
            auto mma_u = [&](int u, int k0, int k1) {
                const uint64_t dv = (u & 1) ? dVF1 : dVF0, dt = (u & 1) ? dTB1 : dTB0;
#pragma unroll
                for (int ks = k0; ks < k1; ++ks)
                    mma_f16(tmem + GL::TM_D3 + 128 * (u & 1), dv + ks * 128, dt + ks * 2, idU, ks > 0);
            };
            // V of chunk 0 converted, and the output halves of D3 zeroed (phase 0 of ofree)
            ok = mbar_wait(&S.convU[0], 0, kWaitNs) && mbar_wait(&S.ofree, 0, kWaitNs);
            if (ok) {
                tc_fence_after();
                mma_u(0, 0, 4);
                mma_commit(&S.emptyU[0]);
            } else {
                gt_status(128u);
            }
            for (int t = 0; t < n_chunks && ok; ++t) {
                const int s = t & 1;
                const uint64_t dqw = s ? dQW1 : dQW0, dkf = s ? dKF1 : dKF0;
                const uint32_t d3 = tmem + GL::TM_D3 + 128 * s;
                const bool next = t + 1 < n_chunks;
                ok = mbar_wait(&S.convQ[s], (t >> 1) & 1, kWaitNs) && mbar_spin(&S.hready, t & 1, kWaitNs);
                if (!ok) {
                    gt_status(1u << 14);
                    break;
                }
                tc_fence_after();
                // MMA3: D3 += h~^T [-W; Q~]^T (N = 128, K = 128 = d_k): columns 0-63 become Delta^T, columns 64-127
                // (zero before) the output's inter-chunk term
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_f16_ts(d3, tmem + GL::TM_HT + ks * 8, dqw + (ks >> 2) * 1024 + (ks & 3) * 2, id3, 1u);
                mma_commit(&S.m3);
                mma_commit(&S.emptyQ[s]);
                // the first half of the next chunk's U^T, into the other D3 buffer during the Delta epilogue.  Its
                // Delta operand was read by MMA45 of chunk t - 1; that phase of m4 is the last one committed, so the
                // wait is unambiguous.
                if (next) {
                    ok = mbar_wait(&S.convU[s ^ 1], ((t + 1) >> 1) & 1, kWaitNs) &&
                         (t == 0 || mbar_spin(&S.m4, (t - 1) & 1, kWaitNs));
                    if (!ok) {
                        gt_status(1024u);
                        break;
                    }
                    tc_fence_after();
                    mma_u(t + 1, 0, 2);
                }
                // (MMA45 overwrites D45, which the output warps read for chunk t - 1: phase t of ofree, after the
                // initial zeroing's phase 0)
                ok = mbar_wait(&S.convK[s], (t >> 1) & 1, kWaitNs) && mbar_wait(&S.ofree, t & 1, kWaitNs) &&
                     mbar_spin(&S.dready, t & 1, kWaitNs);
                if (!ok) {
                    gt_status(512u);
                    break;
                }
                tc_fence_after();
                // MMA45: D45 = Delta^T [K~ | P^T] (N = 192 = d_k + C, K = 64 tokens): columns 0-127 (K~^T Delta)^T for
                // the state update, 128-191 (P Delta)^T for the output.  A = the fp16 columns 32 hb .. + 15 of D3
                // (tokens 32 hb .. + 31).
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16_ts(tmem + GL::TM_D45, d3 + (ks >> 1) * 32 + (ks & 1) * 8, dkf + ks * 128, id45, ks > 0);
                mma_commit(&S.m4);
                mma_commit(&S.emptyK[s]);
                // the second half of the next chunk's U^T, during the state update
                if (next) {
                    mma_u(t + 1, 2, 4);
                    mma_commit(&S.emptyU[s ^ 1]);
                }
            }
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------------- producer: TMA tiles and record copies
        if (lane == 0 && n_chunks > 0) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            int issU = 0, issQ = 0, issK = 0;    // chunks whose loads were issued, per group
            for (int t = 0; t < n_chunks && ok; ++t) {
                const int s = t & 1;
                const int r = (int)(ch.row0 + (long)t * C);
                const uint8_t* rec = p.ws + (size_t)((slot0 + t) * H + ch.h) * GW_ITEM;
                uint8_t* st = smem + s * GL::STAGE;
                const uint32_t ph = ((t >> 1) + 1) & 1;   // phase of the empty barriers released by chunk t - 2
                // test: one chunk in flight per group (each group refilled once the products of chunk t - 1 that read
                // the same group have completed)
                const bool one = p.test == 2 && t >= 1;
                const uint32_t p1 = ((t - 1) >> 1) & 1;
                if (one) ok = mbar_wait(&S.emptyU[s ^ 1], p1, kWaitNs);
                if (ok && t >= 2) ok = mbar_wait(&S.emptyU[s], ph, kWaitNs);
                if (!ok) break;
                mbar_arrive_expect_tx(&S.fullU[s], 16384 + 8192);
                tma_load_3d(st + GL::VF, &tmap_v, &S.fullU[s], 0, ch.h, r);
                tma_load_3d(st + GL::VF + 8192, &tmap_v, &S.fullU[s], 64, ch.h, r);
                bulk_g2s(st + GL::TB, rec + GW_TB, 8192, &S.fullU[s]);
                issU = t + 1;
                if (one) ok = mbar_wait(&S.emptyQ[s ^ 1], p1, kWaitNs);
                if (ok && t >= 2) ok = mbar_wait(&S.emptyQ[s], ph, kWaitNs);
                if (!ok) break;
                if (!(p.test == 1 && t == 0)) {   // test: the first chunk's Q and -W never arrive
                    mbar_arrive_expect_tx(&S.fullQ[s], 32768);
                    bulk_g2s(st + GL::QW, rec + GW_W, 8192, &S.fullQ[s]);
                    bulk_g2s(st + GL::QW + 16384, rec + GW_W + 8192, 8192, &S.fullQ[s]);
                    tma_load_3d(st + GL::QW + 8192, &tmap_q, &S.fullQ[s], 0, hk, r);
                    tma_load_3d(st + GL::QW + 16384 + 8192, &tmap_q, &S.fullQ[s], 64, hk, r);
                }
                issQ = t + 1;
                if (one) ok = mbar_wait(&S.emptyK[s ^ 1], p1, kWaitNs);
                if (ok && t >= 2) ok = mbar_wait(&S.emptyK[s], ph, kWaitNs);
                if (!ok) break;
                mbar_arrive_expect_tx(&S.fullK[s], 16384 + 8192);
                tma_load_3d(st + GL::KF, &tmap_k, &S.fullK[s], 0, hk, r);
                tma_load_3d(st + GL::KF + 8192, &tmap_k, &S.fullK[s], 64, hk, r);
                bulk_g2s(st + GL::KF + 16384, rec + GW_P, 8192, &S.fullK[s]);
                issK = t + 1;
            }
            if (!ok) gt_status(2048u);
            // copies issued whose barrier nobody waited on must land before the CTA exits: wait for every issued
            // phase (bounded)
            for (int t = (issU > 2 ? issU - 2 : 0); t < issU; ++t) mbar_wait(&S.fullU[t & 1], (t >> 1) & 1, kWaitNs);
            for (int t = (issQ > 2 ? issQ - 2 : 0); t < issQ; ++t)
                if (!(p.test == 1 && t == 0)) mbar_wait(&S.fullQ[t & 1], (t >> 1) & 1, kWaitNs);
            for (int t = (issK > 2 ? issK - 2 : 0); t < issK; ++t) mbar_wait(&S.fullK[t & 1], (t >> 1) & 1, kWaitNs);
        }
    } else {
        // ---------------------------------------------------------------- warps 10 and 11: V to fp16, half of each
        // tile per warp (rows past the end: zeros); warp 10 first computes the gate vectors
        const int cidx = tid - 10 * 32;   // 0 .. 63
        float gn[2] = {0.f, 0.f};
        auto load_g = [&](int t, float (&gg)[2]) {
            const int Lt = min(C, ch.len - t * C);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int r = lane + 32 * k;
                gg[k] = r < Lt ? act_gate(p.act, __ldg(p.g + (size_t)(ch.row0 + (long)t * C + r) * H + ch.h), ch.h) : 0.f;
            }
        };
        if (warp == 10 && n_chunks > 0) load_g(0, gn);
        for (int t = 0; t < n_chunks; ++t) {
            const int s = t & 1;
            const int L = min(C, ch.len - t * C);
            if (warp == 10) {
                // the gate vectors of chunk t, into ring slot t % 4 once the lane warps have released it (chunk t - 4)
                if (t >= 4) ok = mbar_wait(&S.vfree[t & 3], ((t >> 2) + 1) & 1, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) gt_status(8192u);
                    break;
                }
                S.gbuf[lane] = gn[0];
                S.gbuf[lane + 32] = gn[1];
                __syncwarp();
                float G0, G1, Gl;
                gate_prefix2(S.gbuf[2 * lane], S.gbuf[2 * lane + 1], lane, G0, G1, Gl);
                GVec& V = vec[t & 3];
                V.qs[2 * lane] = p.scale * ex2(G0);
                V.qs[2 * lane + 1] = p.scale * ex2(G1);
                V.kd[2 * lane] = ex2(Gl - G0);
                V.kd[2 * lane + 1] = ex2(Gl - G1);
                if (lane == 0) V.gC = ex2(Gl);
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.vready[t & 3]);
                if (t + 1 < n_chunks) load_g(t + 1, gn);
            }
            if (ok) ok = mbar_wait(&S.fullU[s], (t >> 1) & 1, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) gt_status(4096u);
                break;
            }
            tile_to_f16<64, false>(sbase + s * GL::STAGE + GL::VF, sbase + s * GL::STAGE + GL::VF, 8192, L, cidx, 0u);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.convU[s]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 8) tmem_dealloc(tmem, GL::TM_COLS);
}

long g_n_slots(const ChunkArgs& a) { return (long)a.B * a.T / C + a.N() + 1; }

}  // namespace

size_t gdn_tmem_workspace_bytes(const ChunkArgs& a) {
    if ((long)a.B * a.T == 0) return 0;
    return (size_t)g_n_slots(a) * a.H * GW_ITEM;
}

cudaError_t launch_chunk_gdn_tmem(const ChunkArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t s) {
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
    const size_t need = gdn_tmem_workspace_bytes(a);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % 256) != 0)
        return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, rows, a.HK(), DK) || !make_map(&mk, a.k, rows, a.HK(), DK) ||
        !make_map(&mv, a.v, rows, a.H, DV))
        return cudaErrorInvalidValue;
    Geo geo{a.cu, a.n_seqs, a.B, a.T, a.H};
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long items = g_n_slots(a) * a.H;
    GIntraParams ip{geo, a.g, a.beta, a.scale, g_n_slots(a), static_cast<uint8_t*>(workspace), a.act, a.H / a.HK()};
    e = cudaFuncSetAttribute(gdn_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GI_SMEM);
    if (e != cudaSuccess) return e;
    const long grid1 = items < (long)GI_CTAS_PER_SM * sms ? items : (long)GI_CTAS_PER_SM * sms;
    gdn_intra_kernel<<<(unsigned)grid1, GI_THREADS, GI_SMEM, s>>>(mq, mk, ip);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    GStateParams sp{geo, a.g, a.scale, a.h0, a.hT, a.o, static_cast<const uint8_t*>(workspace), a.act, a.H / a.HK(),
                    a.test_fwd};
    CUtensorMap mo;
    if (!make_map_rows(&mo, a.o, rows, a.H, DV, a.o_f32 != 0)) return cudaErrorInvalidValue;
    auto launch2 = [&](auto kern) -> cudaError_t {
        // the warpgroups' register targets add up to the launch budget only at exactly REG_LAUNCH registers per
        // thread; with fewer, the lane warps' raise would wait forever
        cudaFuncAttributes fa{};
        cudaError_t e2 = cudaFuncGetAttributes(&fa, kern);
        if (e2 != cudaSuccess) return e2;
        if (fa.numRegs != (int)GL::REG_LAUNCH) return cudaErrorInvalidConfiguration;
        e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gs_smem_bytes());
        if (e2 != cudaSuccess) return e2;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)chains);
        cfg.blockDim = dim3(GL::THREADS);
        cfg.dynamicSmemBytes = gs_smem_bytes();
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, sp);
    };
    e = a.o_f32 ? launch2(gdn_state_kernel<true>) : launch2(gdn_state_kernel<false>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t gt_read_and_clear_status(unsigned* value, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_gt_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    if (clear && *value) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_gt_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace gdn
