// Fused chunkwise gated delta rule forward on tcgen05 tensor cores (sm_103a): scalar gate, bf16 q/k/v,
// d_k = d_v = 128, chunk C = 64, fp32 state, o in fp32 or bf16.
//
// The algorithm is the gated chunk form of "TileLang 实战：KDA 从零到一 -- Gated DeltaNet", §2.3
// (paper eqs 11-12), organised as in "Gated Delta Network (GDN)", §4(b3)-(d): the S-independent
// intra-chunk products, then the serial inter-chunk state pass.  Per chunk of C tokens, with G the
// within-chunk cumulative log gate, gamma = exp(G), Gamma_ij = exp(G_i - G_j) (j <= i), and L valid rows:
//   A    = diag(beta) (Gamma * K K^T), strictly lower        P = scale (Gamma * Q K^T), lower incl. diag
//   T    = (I + A)^{-1}                                      (UT transform, blocked triangular inverse)
//   W    = T diag(beta gamma) K      U  = T diag(beta) V     (WY pseudo-keys / pseudo-values)
//   Q'   = scale diag(gamma) Q - P W U' = P U                (read side folded through T, S-independent)
// and the serial pass over chunks, with h = S^T (d_k x d_v tile) kept in fp32 registers:
//   Delta = U - W h                     (solved corrections, "V_new")
//   O     = U' + Q' h                   (= scale gamma Q h + P Delta, the read of eq. 12)
//   h    <- gamma_C h + Ktilde^T Delta  Ktilde = diag(exp(G_C - G)) K   (eq. 11)
// The stacking [W; Q'] makes both S-dependent products one M = 128 MMA against h.
//
// One CTA owns one (sequence, head, d_v half of 64 columns) and walks the sequence's chunks in order.
// Warp roles (384 threads; 12 warps = 3 per SM sub-partition, so each thread can hold up to 168 registers):
//   warps 0-7   "prep" (two warpgroups, 256 threads): everything that does not depend on h, one chunk ahead of
//               the serial pass; the two warps that share a TMEM lane quarter split the columns of each row.
//               Warp 2 also loads the inputs: at the end of chunk t it issues the TMA loads of chunk t + 2 into
//               the stage chunk t has released (2-stage ring), and reads g and beta into registers.
//   warps 8-11  "serial" warpgroup: the state pass; each thread keeps one row of h in registers
// MMAs (tcgen05.mma kind::f16, fp32 accumulators in TMEM, one issuing thread per warpgroup):
//   MMA0  D0 = [K; Q] K^T          M=128 N=64  K=128  bf16 operands straight from the TMA tiles
//   MMA1  D1 = [I; P] T            M=128 N=64  K=64   -> [T; P T]
//   MMA2  D2 = [T; PT] [beta gamma K | beta V]   M=128 N=192 K=64  -> [W | U ; P W | P U]
//   MMA3  D3 = [W; Q'] h           M=128 N=64  K=128  (serial)
//   MMA4  D4 = Ktilde^T Delta      M=128 N=64  K=64   (serial)
// Internal operands are fp16 (11-bit significand): with bf16 operands the error of the state pass alone
// exceeds the 2e-2 max-error bound the output is held to; the inputs' bf16 values convert exactly.
// Decay exponents are differences masked before exp2, so no factor exceeds 1 (TileLang page §4.1).
// Rows past a sequence's end get beta = 0 and g = 0 and are zeroed where they would enter a product, so
// packed sequences give bit-identical results to separate runs.
//
// Every mbarrier wait is bounded (2 s of wall time).  A wait that gives up sets a status bit
// (read by gdn_device_status), and its warpgroup skips the rest of its work while still passing every
// named barrier, so the CTA drains, frees its TMEM and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "internal.h"
#include "tc_common.cuh"
#include "chunk_common.cuh"

namespace gdn {

__device__ unsigned g_tc_status;

namespace {

using namespace tc;

constexpr int C = 64;        // chunk
constexpr int DK = 128;
constexpr int DV = 128;
constexpr int DVT = 64;      // d_v columns per CTA
constexpr int NTHREADS = 384;
constexpr int NPREP = 256;
constexpr uint64_t kWaitNs = 2000000000ull;

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;                       // 2 stages x 32 KB: [K; Q] rows, 2 K-slabs of 16 KB
constexpr uint32_t STAGE_KQ = 32768;
constexpr uint32_t OFF_V = OFF_KQ + 2 * STAGE_KQ;    // 2 stages x 8 KB: V tile [64 tok][64 col]
constexpr uint32_t STAGE_V = 8192;
constexpr uint32_t OFF_A1 = OFF_V + 2 * STAGE_V;     // [I; P] then [T; PT], fp16 K-major 128 x 64
constexpr uint32_t OFF_B1 = OFF_A1 + 16384;          // T, fp16 MN-major [j][n] 64 x 64
constexpr uint32_t OFF_B2 = OFF_B1 + 8192;           // X = [beta gamma K | beta V], fp16 MN-major 64 x 192
constexpr uint32_t OFF_WQ = OFF_B2 + 24576;          // [W; Q'], fp16 K-major 128 x 128
constexpr uint32_t OFF_KT = OFF_WQ + 32768;          // Ktilde, fp16 MN-major [j][c] 64 x 128
constexpr uint32_t OFF_H = OFF_KT + 16384;           // h, fp16 MN-major [d][n] 128 x 64
constexpr uint32_t OFF_D = OFF_H + 16384;            // Delta, fp16 MN-major [j][n] 64 x 64
constexpr uint32_t OFF_T32 = OFF_D + 8192;           // T in fp32, row stride 68 floats
constexpr uint32_t OFF_SMALL = OFF_T32 + 64 * TS * 4;
// the fp32 A of the solve lives in the X buffer (X is built only after the solve)
constexpr uint32_t OFF_AM = OFF_B2;
constexpr uint32_t OFF_RT = OFF_B2 + 64 * TS * 4;   // 32 x 36 fp32 scratch of the solve
static_assert(64 * TS * 4 + 32 * 36 * 4 <= 24576, "A and the solve scratch must fit in the X buffer");

struct Small {
    uint64_t full[2];        // stage loaded (TMA transaction bytes)
    uint64_t m0, m1, m2;     // prep MMA commits
    uint64_t m3, m4;         // serial MMA commits
    uint64_t prep_done;      // prep -> serial: [W; Q'], Ktilde, D2 ready for the chunk
    uint64_t d2_free;        // serial -> prep: U, U' read out of TMEM
    uint32_t tmem_base;
    uint32_t pad;
    float gbuf[2][C];        // per stage: g (0 past the end)
    float bbuf[2][C];        // per stage: beta (0 past the end)
    float lg[2][C];          // per chunk parity: log2 of the within-chunk cumulative retention
    float gam[2][C];         // gamma_j
    float kdec[2][C];        // gamma_C / gamma_j
    float info_gC[4];        // per-chunk gamma_C for the serial pass (4 slots: written two chunks ahead)
    int info_L[4];           // per-chunk valid rows
};
constexpr uint32_t SMEM_BYTES = OFF_SMALL + sizeof(Small) + 1024;  // + alignment slack

// TMEM columns
// D0 is double-buffered (columns 0 and 64) so MMA0 of the next chunk can run ahead
constexpr uint32_t TM_D0 = 0, TM_D1 = 128, TM_D2 = 192, TM_D3 = 384, TM_D4 = 448, TM_COLS = 512;

struct TcParams {
    const float* g;
    const float* beta;
    float scale;
    const float* h0;
    float* hT;
    const int32_t* cu;
    int n_seqs;
    void* o;
    int B, T, H;
    int o_f32;
};

__device__ __forceinline__ void set_status(unsigned bit) { atomicOr(&g_tc_status, bit); }

// Resolve (sequence, head, half) for this CTA and the sequence's token range.
struct Work {
    int n, h, half;
    long row0;   // first token row in the [B*T] dimension
    int len;
};

__device__ Work resolve_work(const TcParams& p) {
    Work w;
    const int per_seq = p.H * 2;
    int seq_rank = blockIdx.x / per_seq;
    const int rem = blockIdx.x % per_seq;
    w.h = rem / 2;
    w.half = rem % 2;
    if (p.cu) {
        // longest sequences first (their chains are the longest serial paths); ties by index
        int n = seq_rank;
        if (p.n_seqs <= 32) {
            // lane m ranks sequence m; the lane whose rank equals this CTA's slot names the sequence
            const int lane = threadIdx.x & 31;
            int rank = -1;
            if (lane < p.n_seqs) {
                const int lm = p.cu[lane + 1] - p.cu[lane];
                rank = 0;
                for (int m2 = 0; m2 < p.n_seqs; ++m2) {
                    const int l2 = p.cu[m2 + 1] - p.cu[m2];
                    rank += (l2 > lm) || (l2 == lm && m2 < lane);
                }
            }
            const unsigned hit = __ballot_sync(0xffffffffu, rank == seq_rank);
            if (hit) n = __ffs(hit) - 1;
        }
        long s0 = p.cu[n], s1 = p.cu[n + 1];
        s0 = s0 < 0 ? 0 : (s0 > p.T ? p.T : s0);
        s1 = s1 < s0 ? s0 : (s1 > p.T ? p.T : s1);
        w.n = n;
        w.row0 = s0;
        w.len = (int)(s1 - s0);
    } else {
        w.n = seq_rank;
        w.row0 = (long)seq_rank * p.T;
        w.len = p.T;
    }
    return w;
}

// Blocked inverse of the unit lower-triangular (I + A), 64 x 64, by the 128 prep threads.
// A (strictly lower) is in Am (fp32, row stride TS); T is written to the lower triangle of T32 (fp32, row
// stride TS), whose upper triangle stays zero, so every product below can run over full tiles.
// Rt is a 32 x RS fp32 scratch tile for the intermediate products.
// Level 0: the four 16 x 16 diagonal blocks by right-looking forward substitution in fp32, one column per
// thread.  Levels 1 and 2: T_ab = -T_aa (A_ab T_bb), first for the 16-wide then for the 32-wide off-diagonal
// block (block rows of (I + A) T = I), as warp-level tensor-core products (mma.sync m16n8k8, TF32 inputs,
// fp32 accumulation): these tiles are far below the 64-row minimum of tcgen05.


// Loads of one chunk's inputs.  K and Q arrive as 2 x 2 boxes of 64 tokens x 64 columns into the rows 0-63 / 64-127
// of the two K-slabs of the stage; the V box is this CTA's 64 columns.  All transaction bytes count on full[s].
__device__ __forceinline__ void issue_stage(uint8_t* smem, Small& S, const CUtensorMap* mq, const CUtensorMap* mk,
                                            const CUtensorMap* mv, const Work& w, int t, int lane) {
    if (lane != 0) return;
    const int s = t & 1;
    const int row = (int)(w.row0 + (long)t * C);
    mbar_arrive_expect_tx(&S.full[s], STAGE_KQ + STAGE_V);
    uint8_t* kq = smem + OFF_KQ + s * STAGE_KQ;
    tma_load_3d(kq, mk, &S.full[s], 0, w.h, row);
    tma_load_3d(kq + 8192, mq, &S.full[s], 0, w.h, row);
    tma_load_3d(kq + 16384, mk, &S.full[s], 64, w.h, row);
    tma_load_3d(kq + 16384 + 8192, mq, &S.full[s], 64, w.h, row);
    tma_load_3d(smem + OFF_V + s * STAGE_V, mv, &S.full[s], w.half * DVT, w.h, row);
}
// g and beta of chunk t (0 past the sequence end): lane l holds tokens l and l + 32
__device__ __forceinline__ void load_gb(const TcParams& p, const Work& w, int t, int lane, float (&g)[2],
                                        float (&b)[2]) {
    const int L = min(C, w.len - t * C);
    const long row = w.row0 + (long)t * C;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int r = lane + 32 * k;
        const size_t tok = (size_t)(row + r) * p.H + w.h;
        g[k] = r < L ? __ldg(p.g + tok) : 0.f;
        b[k] = r < L ? __ldg(p.beta + tok) : 0.f;
    }
}
__device__ __forceinline__ void store_gb(Small& S, int t, int lane, const float (&g)[2], const float (&b)[2]) {
    const int s = t & 1;
    S.gbuf[s][lane] = g[0];
    S.gbuf[s][lane + 32] = g[1];
    S.bbuf[s][lane] = b[0];
    S.bbuf[s][lane + 32] = b[1];
}


// Gate prefix of chunk t (one warp): log2 cumulative retention lg, gamma = 2^lg, gamma_C / gamma, and gamma_C / L
// for the serial pass.  Rows past the sequence end have g = 0.
__device__ __forceinline__ void gate_prefix(Small& S, int t, int L, int lane) {
    const int s = t & 1;
    const float LOG2E = 1.4426950408889634f;
    const float g0 = S.gbuf[s][2 * lane], g1 = S.gbuf[s][2 * lane + 1];
    float x = g0 + g1;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, m);
        if (lane >= m) x += y;
    }
    const float G1 = x * LOG2E, G0 = (x - g1) * LOG2E;
    S.lg[s][2 * lane] = G0;
    S.lg[s][2 * lane + 1] = G1;
    const float Glast = __shfl_sync(0xffffffffu, G1, 31);
    S.gam[s][2 * lane] = ex2(G0);
    S.gam[s][2 * lane + 1] = ex2(G1);
    S.kdec[s][2 * lane] = ex2(Glast - G0);
    S.kdec[s][2 * lane + 1] = ex2(Glast - G1);
    if (lane == 31) {
        S.info_gC[t & 3] = ex2(Glast);
        S.info_L[t & 3] = L;
    }
}

// Every thread passes the same four named barriers whether or not it computes (work = false after an
// aborted wait), so the warpgroup can never fall out of step.
__device__ void solve_unit_lower(const float* Am, float* T32, float* Rt, int t, bool work) {
    const int w = t >> 5, lane = t & 31;   // 8 warps
    if (work && t < 64) {
        const int b = t >> 4, c = t & 15, o = 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
#pragma unroll
            for (int r = j + 1; r < 16; ++r) x[r] = fmaf(-Am[(o + r) * TS + o + j], x[j], x[r]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) T32[(o + r) * TS + o + c] = x[r];
    }
    named_bar(1, NPREP);
    if (work && w < 4) {   // level 1: warp w -> pair p (o = 32 p), columns 8 nt .. 8 nt + 7 of the 16-wide block
        const int pr = w >> 1, nt = w & 1, o = 32 * pr;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
            mma_tile_tf32(d, Am + (o + 16) * TS + o + 8 * ks, TS, T32 + (o + 8 * ks) * TS + o + 8 * nt, TS, lane);
        st_tile(Rt + (16 * pr) * RS + 8 * nt, RS, d, lane, 1.f);
        __syncwarp();
        float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
            mma_tile_tf32(e, T32 + (o + 16) * TS + o + 16 + 8 * ks, TS, Rt + (16 * pr + 8 * ks) * RS + 8 * nt, RS, lane);
        st_tile(T32 + (o + 16) * TS + o + 8 * nt, TS, e, lane, -1.f);
    }
    named_bar(1, NPREP);
    const int mt = w & 1, nq = w >> 1;   // 2 row tiles x 4 column tiles of 8
    if (work) {   // level 2, stage 1: R = A[32..63][0..31] T[0..31][0..31]; warp -> rows 16 mt, columns 8 nq .. + 7
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_tile_tf32(d, Am + (32 + 16 * mt) * TS + 8 * ks, TS, T32 + (8 * ks) * TS + 8 * nq, TS, lane);
        st_tile(Rt + (16 * mt) * RS + 8 * nq, RS, d, lane, 1.f);
    }
    named_bar(1, NPREP);
    if (work) {   // level 2, stage 2: T[32..63][0..31] = -T[32..63][32..63] R
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_tile_tf32(d, T32 + (32 + 16 * mt) * TS + 32 + 8 * ks, TS, Rt + (8 * ks) * RS + 8 * nq, RS, lane);
        st_tile(T32 + (32 + 16 * mt) * TS + 8 * nq, TS, d, lane, -1.f);
    }
    named_bar(1, NPREP);
}

// Epilogue of D2 columns 0-127: W rows (0-63) and Q' = scale gamma Q - P W rows (64-127) to fp16 into [W; Q']
// (K-major, two 64-column slabs).  Q comes from the stage's TMA tile, rows 64-127 of each slab.
__device__ __forceinline__ void epilogue_wq(uint32_t tl, int row, int slab, const Small& S, int s, float scale,
                                            const uint8_t* kqp, uint8_t* wq) {
    // this thread: row `row`, the 64 columns of slab `slab`
    const int i = row & 63;
    const float qs = scale * S.gam[s][i];
    uint32_t r[4][16];
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) tmem_ld16(tl + TM_D2 + slab * 64 + cb * 16, r[cb]);
    tmem_ld_wait();
    if (row < 64) {
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            float f[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = __uint_as_float(r[c8 >> 1][(c8 & 1) * 8 + q]);
            st_h8(wq + slab * 16384 + sw128_off(row, c8 * 8), f);
        }
    } else {
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            float qv[8], f[8];
            bf16x8_to_f32(ld16(kqp + slab * 16384 + sw128_off(row, c8 * 8)), qv);
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = fmaf(qs, qv[q], -__uint_as_float(r[c8 >> 1][(c8 & 1) * 8 + q]));
            st_h8(wq + slab * 16384 + sw128_off(row, c8 * 8), f);
        }
    }
}

template <bool O_F32>
__global__ void __launch_bounds__(NTHREADS, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    // align by offsetting the shared array itself, so the compiler keeps every access in the shared space
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    Small& S = *reinterpret_cast<Small*>(smem + OFF_SMALL);
    float* Am = reinterpret_cast<float*>(smem + OFF_AM);
    float* T32 = reinterpret_cast<float*>(smem + OFF_T32);
    float* Rt = reinterpret_cast<float*>(smem + OFF_RT);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const Work w = resolve_work(p);
    const int n_chunks = (w.len + C - 1) / C;

    if (warp == 0) {
        tmem_alloc(&S.tmem_base, TM_COLS);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(&S.full[0], 1);
        mbar_init(&S.full[1], 1);
        mbar_init(&S.m0, 1);
        mbar_init(&S.m1, 1);
        mbar_init(&S.m2, 1);
        mbar_init(&S.m3, 1);
        mbar_init(&S.m4, 1);
        mbar_init(&S.prep_done, 1);
        mbar_init(&S.d2_free, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;

    if (warp < 8) {
        // ------------------------------------------------------------ prep (two warpgroups)
        const int t256 = tid;                          // 0..255
        const int q4 = warp & 3;                       // TMEM lane quarter of this warp
        const int pw = warp >> 2;                      // which of the two warps on this quarter
        const int row = 32 * q4 + lane;                // TMEM lane this thread reads
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        const bool leader = (t256 == 0);               // warp 0 lane 0 issues the prep MMAs
        const bool loader = (warp == 2);
        float ldg[2] = {0.f, 0.f}, ldb[2] = {0.f, 0.f};   // g, beta of chunk t + 2 (loader warp, in flight)
        int issued = 0;                                // chunks whose TMA loads have been issued
        const int jrow = t256 & 63, part = t256 >> 6;  // (row, quarter of the columns) for the elementwise builds
        bool ok = true;
        for (int e = t256; e < 64 * TS; e += NPREP) T32[e] = 0.f;   // the upper triangle stays zero
        if (loader) {
            prefetch_tmap(&tmap_q);
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            for (int t = 0; t < 2 && t < n_chunks; ++t) {
                issue_stage(smem, S, &tmap_q, &tmap_k, &tmap_v, w, t, lane);
                float gg[2], bb[2];
                load_gb(p, w, t, lane, gg, bb);
                store_gb(S, t, lane, gg, bb);
                issued = t + 1;
            }
        }
        named_bar(1, NPREP);   // g and beta of chunks 0 and 1 are in shared memory
        if (warp == 1 && n_chunks > 0) gate_prefix(S, 0, min(C, w.len), lane);
        named_bar(1, NPREP);
        for (int t = 0; t < n_chunks; ++t) {
            const int s = t & 1;
            const int L = min(C, w.len - t * C);
            const uint32_t kq = sbase + OFF_KQ + s * STAGE_KQ;
            uint8_t* kqp = smem + OFF_KQ + s * STAGE_KQ;
            uint8_t* vsp = smem + OFF_V + s * STAGE_V;
            const uint32_t d0 = TM_D0 + 64u * (uint32_t)(t & 1);
            if (ok) ok = mbar_wait(&S.full[s], (t >> 1) & 1, kWaitNs);
            if (!ok && t256 == 0) set_status(4u);
            // MMA0: D0 = [K; Q] K^T (for t > 0 it was issued during the previous chunk)
            if (ok && leader && t == 0) {
                tc_fence_after();
                const uint32_t id = idesc_f16(128, 64, true, false, false);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t a = kq + (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_f16(tmem + d0, sdesc(a, 16, 1024), sdesc(a, 16, 1024), id, ks > 0);
                }
                mma_commit(&S.m0);
            }
            // MMA0 of chunk 0 is awaited here; for later chunks the leader awaited it during the previous chunk,
            // and the barriers since then carry its completion to every thread
            if (ok && leader && t == 0) ok = mbar_wait(&S.m0, 0, kWaitNs);
            if (!ok && leader) set_status(8u);
            named_bar(1, NPREP);
            // epilogue 0: A (rows 0-63) to fp32 for the solve, P (rows 64-127) and the identity rows to A1
            tc_fence_after();
            if (ok) epilogue_kkt<true>(tl + d0, row, q4, pw, S.lg[s], S.bbuf[s], p.scale, Am, smem + OFF_A1);
            tc_fence_before();
            named_bar(1, NPREP);
            // MMA0 of the next chunk runs ahead into the other D0 buffer while this chunk is solved
            if (ok && leader && t + 1 < n_chunks) {
                const int s1 = (t + 1) & 1;
                ok = mbar_wait(&S.full[s1], ((t + 1) >> 1) & 1, kWaitNs);
                if (!ok) set_status(2048u);
                if (ok) {
                    tc_fence_after();
                    const uint32_t kq1 = sbase + OFF_KQ + s1 * STAGE_KQ;
                    const uint32_t id = idesc_f16(128, 64, true, false, false);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t a = kq1 + (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_f16(tmem + TM_D0 + 64u * (uint32_t)((t + 1) & 1), sdesc(a, 16, 1024), sdesc(a, 16, 1024),
                                id, ks > 0);
                    }
                    mma_commit(&S.m0);
                    ok = mbar_wait(&S.m0, (t + 1) & 1, kWaitNs);
                    if (!ok) set_status(8u);
                }
            }
            // UT transform: T = (I + A)^{-1}
            solve_unit_lower(Am, T32, Rt, t256, ok);
            // g and beta of chunk t + 1 (loaded at the end of chunk t - 1) go to the slot chunk t - 1 used; the
            // gate prefix of chunk t + 1 reads them after the next barrier
            if (loader && t >= 1 && t + 1 < issued) store_gb(S, t + 1, lane, ldg, ldb);
            // T to fp16, MN-major [j][n] (operand B of MMA1)
            if (ok) {
#pragma unroll
                for (int it = 0; it < 2; ++it) {
                    const int e = t256 + NPREP * it, j = e >> 3, c8 = e & 7;
                    const float4 x0 = ld4(T32 + j * TS + c8 * 8), x1 = ld4(T32 + j * TS + c8 * 8 + 4);
                    const float f[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    float g[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) g[q] = (c8 * 8 + q <= j) ? f[q] : 0.f;
                    st_h8(smem + OFF_B1 + sw128_off(j, c8 * 8), g);
                }
            }
            fence_async_smem();
            named_bar(1, NPREP);
            // MMA1: D1 = [I; P] T
            if (ok && leader) {
                tc_fence_after();
                const uint32_t id = idesc_f16(128, 64, false, false, true);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16(tmem + TM_D1, sdesc(sbase + OFF_A1 + ks * 32, 16, 1024),
                            sdesc(sbase + OFF_B1 + ks * 2048, 8192, 1024), id, ks > 0);
                mma_commit(&S.m1);
            }
            // X = [beta gamma K | beta V] (operand B of MMA2), fp16 MN-major [j][n], 3 atoms of 64 columns.
            // Thread (jrow, part): chunk columns 6 part .. 6 part + 5 of row jrow (0-7 K slab 0, 8-15 K slab 1,
            // 16-23 V); part is warp-uniform.
            if (ok) {
                const bool zero = jrow >= L;
                const float sk = S.bbuf[s][jrow] * S.gam[s][jrow], sv = S.bbuf[s][jrow];
#pragma unroll
                for (int cc = 0; cc < 6; ++cc) {
                    const int c = 6 * part + cc;
                    if (c < 16) {
                        const uint32_t o8 = sw128_off(jrow, (c & 7) * 8);
                        copy_scaled_chunk(kqp + (c >> 3) * 16384 + o8, smem + OFF_B2 + (c >> 3) * 8192 + o8, sk, zero);
                    } else {
                        const uint32_t o8 = sw128_off(jrow, (c - 16) * 8);
                        copy_scaled_chunk(vsp + o8, smem + OFF_B2 + 2 * 8192 + o8, sv, zero);
                    }
                }
            }
            // gate prefix of the next chunk (its g and beta are already in shared memory), one chunk ahead
            if (warp == 1 && t + 1 < n_chunks) gate_prefix(S, t + 1, min(C, w.len - (t + 1) * C), lane);
            // epilogue 1: [T; PT] to fp16 into A1 (operand A of MMA2); columns [32 pw, 32 pw + 32)
            if (ok) ok = mbar_wait(&S.m1, t & 1, kWaitNs);
            if (!ok && t256 == 0) set_status(16u);
            tc_fence_after();
            if (ok) {
                uint32_t r[2][16];
                tmem_ld16(tl + TM_D1 + 32 * pw, r[0]);
                tmem_ld16(tl + TM_D1 + 32 * pw + 16, r[1]);
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float f[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) f[q] = __uint_as_float(r[cc >> 1][(cc & 1) * 8 + q]);
                    st_h8(smem + OFF_A1 + sw128_off(row, 32 * pw + cc * 8), f);
                }
            }
            fence_async_smem();
            tc_fence_before();
            named_bar(1, NPREP);
            // MMA2: D2 = [T; PT] X, once the serial pass has read U, U' of the previous chunk
            if (ok && leader) {
                if (t > 0) ok = mbar_wait(&S.d2_free, (t - 1) & 1, kWaitNs);
                if (!ok) set_status(32u);
                if (ok) {
                    tc_fence_after();
                    const uint32_t id = idesc_f16(128, 192, false, false, true);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tmem + TM_D2, sdesc(sbase + OFF_A1 + ks * 32, 16, 1024),
                                sdesc(sbase + OFF_B2 + ks * 2048, 8192, 1024), id, ks > 0);
                    mma_commit(&S.m2);
                }
            }
            // Ktilde = diag(gamma_C / gamma) K (operand A of MMA4), once MMA4 of the previous chunk is done.
            // Thread (jrow, part): chunks 4 (part & 1) .. + 3 of K slab part >> 1, row jrow.
            if (ok && t > 0) ok = mbar_wait(&S.m4, (t - 1) & 1, kWaitNs);
            if (!ok && t256 == 0) set_status(64u);
            if (ok) {
                const bool zero = jrow >= L;
                const float sd = S.kdec[s][jrow];
                const int slab = part >> 1;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const uint32_t o8 = sw128_off(jrow, (4 * (part & 1) + cc) * 8);
                    copy_scaled_chunk(kqp + slab * 16384 + o8, smem + OFF_KT + slab * 8192 + o8, sd, zero);
                }
            }
            // epilogue 2: W (rows 0-63) and Q' = scale gamma Q - P W (rows 64-127) into [W; Q'], once MMA3 of the
            // previous chunk has consumed the buffer; this thread does the 64 columns of slab pw
            named_bar(1, NPREP);   // the leader's MMA2 issue precedes every thread's wait on m2
            if (ok && t > 0) ok = mbar_wait(&S.m3, (t - 1) & 1, kWaitNs);
            if (ok) ok = mbar_wait(&S.m2, t & 1, kWaitNs);
            if (!ok && t256 == 0) set_status(128u);
            tc_fence_after();
            if (ok) epilogue_wq(tl, row, pw, S, s, p.scale, kqp, smem + OFF_WQ);
            fence_async_smem();
            tc_fence_before();
            named_bar(1, NPREP);
            if (t256 == 0) mbar_arrive(&S.prep_done);
            // the stage of chunk t is free: load chunk t + 2 into it
            if (loader && ok && t + 2 < n_chunks) {
                issue_stage(smem, S, &tmap_q, &tmap_k, &tmap_v, w, t + 2, lane);
                load_gb(p, w, t + 2, lane, ldg, ldb);
                issued = t + 3;
            }
        }
        // drain: a stage whose TMA was issued but never waited on (after an abort) must land before exit
        if (loader && issued > 0 && !ok) {
            const int t = issued - 1;
            mbar_wait(&S.full[t & 1], (t >> 1) & 1, kWaitNs);
        }
    } else {
        // ------------------------------------------------------------ serial warpgroup
        // Warps with TMEM lane quarters 0 and 1 own the Delta rows (tokens 0-63) of D3; the other two own the
        // output rows.  The Delta warps issue MMA4 as soon as Delta is in shared memory.
        const int t128 = tid - 256;
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;                // TMEM lane: token (D3 rows) and d_k row (D4 rows)
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        const bool leader = (t128 == 0);               // warp 8 lane 0 (quarter 0, a Delta warp)
        const bool delta_warp = q4 < 2;
        bool ok = true;
        const size_t sidx = ((size_t)w.n * p.H + w.h) * DK * DV + (size_t)row * DV + w.half * DVT;
        float hreg[DVT];
#pragma unroll
        for (int q = 0; q < DVT / 4; ++q) {
            float4 x = p.h0 ? reinterpret_cast<const float4*>(p.h0 + sidx)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            hreg[4 * q] = x.x; hreg[4 * q + 1] = x.y; hreg[4 * q + 2] = x.z; hreg[4 * q + 3] = x.w;
        }
        // h to fp16, MN-major [d][n] (operand B of MMA3)
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) st_h8(smem + OFF_H + sw128_off(row, c8 * 8), hreg + c8 * 8);
        fence_async_smem();
        named_bar(2, 128);
        for (int t = 0; t < n_chunks; ++t) {
            if (ok) ok = mbar_wait(&S.prep_done, t & 1, kWaitNs);
            if (!ok && t128 == 0) set_status(256u);
            const int L = S.info_L[t & 3];
            const float gC = S.info_gC[t & 3];
            // MMA3: D3 = [W; Q'] h
            if (ok && leader) {
                tc_fence_after();
                const uint32_t id = idesc_f16(128, 64, false, false, true);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_f16(tmem + TM_D3, sdesc(sbase + OFF_WQ + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                            sdesc(sbase + OFF_H + ks * 2048, 1024, 1024), id, ks > 0);
                mma_commit(&S.m3);
            }
            if (ok) ok = mbar_wait(&S.m3, t & 1, kWaitNs);
            if (!ok && t128 == 0) set_status(512u);
            tc_fence_after();
            const int i = row - 64;
            const bool store_o = !delta_warp && i < L;
            const size_t orow = ((size_t)(w.row0 + (long)t * C + (row & 63)) * p.H + w.h) * DV + w.half * DVT;
            // four passes of 16 columns keep the live TMEM tiles small (h stays in registers throughout)
#pragma unroll
            for (int hp = 0; hp < 4; ++hp) {
                uint32_t a[16], u[16];
                if (ok) {
                    tmem_ld16(tl + TM_D3 + hp * 16, a);
                    tmem_ld16(tl + TM_D2 + 128 + hp * 16, u);
                    tmem_ld_wait();
                }
                if (ok && delta_warp) {
                    // Delta = U - W h (token rows 0-63) to fp16 MN-major [j][n] (operand B of MMA4)
#pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        float f[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) f[q] = __uint_as_float(u[h8 * 8 + q]) - __uint_as_float(a[h8 * 8 + q]);
                        st_h8(smem + OFF_D + sw128_off(row, hp * 16 + h8 * 8), f);
                    }
                } else if (ok && store_o) {
                    // O = U' + Q' h (token rows 64-127) to HBM
                    float f[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k) f[k] = __uint_as_float(u[k]) + __uint_as_float(a[k]);
                    if (O_F32) {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow + hp * 16);
#pragma unroll
                        for (int q = 0; q < 4; ++q) dst[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow + hp * 16);
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
            if (delta_warp) {
                fence_async_smem();
                tc_fence_before();
                named_bar(3, 64);
                // MMA4: D4 = Ktilde^T Delta
                if (ok && leader) {
                    tc_fence_after();
                    const uint32_t id = idesc_f16(128, 64, false, true, true);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tmem + TM_D4, sdesc(sbase + OFF_KT + ks * 2048, 8192, 1024),
                                sdesc(sbase + OFF_D + ks * 2048, 1024, 1024), id, ks > 0);
                    mma_commit(&S.m4);
                }
            }
            tc_fence_before();
            named_bar(2, 128);
            if (ok && leader) mbar_arrive(&S.d2_free);    // U and U' have been read out of TMEM
            if (ok) ok = mbar_wait(&S.m4, t & 1, kWaitNs);
            if (!ok && t128 == 0) set_status(1024u);
            tc_fence_after();
            // epilogue 2: h <- gamma_C h + Ktilde^T Delta; fp16 copy for the next MMA3
            if (ok) {
                uint32_t r[4][16];
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) tmem_ld16(tl + TM_D4 + cb * 16, r[cb]);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 64; ++k) hreg[k] = fmaf(gC, hreg[k], __uint_as_float(r[k >> 4][k & 15]));
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) st_h8(smem + OFF_H + sw128_off(row, c8 * 8), hreg + c8 * 8);
            }
            fence_async_smem();
            tc_fence_before();
            named_bar(2, 128);
        }
        if (p.hT && ok) {
#pragma unroll
            for (int q = 0; q < DVT / 4; ++q)
                reinterpret_cast<float4*>(p.hT + sidx)[q] =
                    make_float4(hreg[4 * q], hreg[4 * q + 1], hreg[4 * q + 2], hreg[4 * q + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [rows][H][d] bf16 tensor, box = 64 d-elements x 1 head x 64 rows, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, long rows, int H, int d) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_f32_rows(CUtensorMap* m, const float* base, long rows, int H, int d) {
    auto enc = get_encode();
    if (!enc || d > 256) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4};
    cuuint32_t box[3] = {(cuuint32_t)d, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool device_is_sm100_family() {
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    return major == 10;
}


const char* tc_chunk_unsupported_reason(const ChunkArgs& a) {
    if (a.per_channel) return "per-channel (KDA) gates use another kernel";
    if (a.act.any()) return "the gate activation runs on the two-pass path";
    if (a.HK() != a.H) return "grouped values run on the two-pass path";
    if (!a.bf16) return "q, k, v must be bf16";
    if (a.dk != DK || a.dv != DV) return "d_k and d_v must be 128";
    if (a.C != C) return "chunk_size must be 64";
    auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) % 16) == 0; };
    if (!al16(a.q) || !al16(a.k) || !al16(a.v) || !al16(a.o) || (a.h0 && !al16(a.h0)) || (a.hT && !al16(a.hT)))
        return "tensors must be 16-byte aligned";
    return nullptr;
}

cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t s) {
    const long ctas = (long)a.N() * a.H * 2;
    if (ctas == 0) return cudaSuccess;
    if (!device_is_sm100_family()) return cudaErrorNoKernelImageForDevice;
    const long rows = (long)a.B * a.T;
    if (rows == 0) {
        // no tokens: the final state is the initial state
        if (a.hT) {
            const size_t bytes = (size_t)a.N() * a.H * DK * DV * sizeof(float);
            return a.h0 ? cudaMemcpyAsync(a.hT, a.h0, bytes, cudaMemcpyDeviceToDevice, s)
                        : cudaMemsetAsync(a.hT, 0, bytes, s);
        }
        return cudaSuccess;
    }
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, rows, a.H, DK) || !make_map(&mk, a.k, rows, a.H, DK) || !make_map(&mv, a.v, rows, a.H, DV))
        return cudaErrorInvalidValue;
    TcParams p{a.g, a.beta, a.scale, a.h0, a.hT, a.cu, a.n_seqs, a.o, a.B, a.T, a.H, a.o_f32};
    cudaError_t e;
    if (a.o_f32) {
        e = cudaFuncSetAttribute(chunk_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        chunk_tc_kernel<true><<<(unsigned)ctas, NTHREADS, SMEM_BYTES, s>>>(mq, mk, mv, p);
    } else {
        e = cudaFuncSetAttribute(chunk_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        chunk_tc_kernel<false><<<(unsigned)ctas, NTHREADS, SMEM_BYTES, s>>>(mq, mk, mv, p);
    }
    return cudaGetLastError();
}

cudaError_t tc_read_and_clear_status(unsigned* value, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_tc_status, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    if (clear && *value) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace gdn
