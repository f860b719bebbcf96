// Device pieces shared by the two-pass chunk kernels (chunk_two_pass.cu: the per-channel gate; chunk_gdn_tmem.cu:
// the scalar gate): the fixed tile sizes, the sequence geometry of a call (packed or batched), the walk of a
// persistent CTA over (chunk slot, head) items, and the blocked inverse of the unit lower-triangular chunk
// system T = (I + A)^{-1} ("TileLang 实战：KDA 从零到一 -- Gated DeltaNet", §2.2.4 and §4.2: forward
// substitution on the 16 x 16 diagonal blocks, then the off-diagonal blocks by products).
#pragma once

#include <cstdint>

#include "chunk_common.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int C = 64;
constexpr int DK = 128;
constexpr int DV = 128;
constexpr uint64_t kWaitNs = 2000000000ull;

// Sequence geometry: packed (cu_seqlens) or B rows of T tokens.
struct Geo {
    const int32_t* cu;
    int n_seqs;
    int B, T, H;
    __device__ int N() const { return cu ? n_seqs : B; }
    __device__ void seq(int n, long& s0, int& len) const {
        if (cu) {
            long a = cu[n], b = cu[n + 1];
            a = a < 0 ? 0 : (a > T ? T : a);
            b = b < a ? a : (b > T ? T : b);
            s0 = a;
            len = (int)(b - a);
        } else {
            s0 = (long)n * T;
            len = T;
        }
    }
    // first workspace slot of sequence n (strictly increasing in n for valid cu_seqlens)
    __device__ long slot0(int n) const {
        long s0;
        int len;
        seq(n, s0, len);
        return s0 / C + n;
    }
};

struct Item {
    int n, h, t, L;
    long row;     // first token row of the chunk
    long it;      // workspace item index (slot * H + head)
};

// A CTA visits the virtual items slot * H + head = last - blockIdx.x, last - blockIdx.x - gridDim.x, ... (the last
// slots first: the first chunks of every sequence are written last, and the state pass, which starts there, finds
// them still in L2); the cursor keeps (slot, head) and the sequence whose slots begin at or before the slot
// (non-increasing along the walk).
struct Cursor {
    long s;
    int h, n;
};

__device__ __forceinline__ void cursor_step(Cursor& c, int ds, int dh, int H) {
    c.h -= dh;
    c.s -= ds;
    if (c.h < 0) {
        c.h += H;
        --c.s;
    }
}

// The first valid item at or before the cursor (slots between sequences are unused); false below slot 0.
__device__ bool cursor_next_valid(const Geo& g, Cursor& c, int ds, int dh, Item& x) {
    for (; c.s >= 0; cursor_step(c, ds, dh, g.H)) {
        while (c.n > 0 && g.slot0(c.n) > c.s) --c.n;
        long s0;
        int len;
        g.seq(c.n, s0, len);
        const long t = c.s - (s0 / C + c.n);
        if (t < 0 || t * C >= len) continue;
        x.n = c.n;
        x.h = c.h;
        x.t = (int)t;
        x.row = s0 + t * C;
        x.L = min(C, len - (int)t * C);
        x.it = c.s * g.H + c.h;
        return true;
    }
    return false;
}

// Level 0 of the blocked inverse for the 16 x 16 diagonal block at offset o (one warp): the two 8 x 8 diagonal
// sub-blocks by forward substitution (lane 8 s + c owns column c of sub-block s; their 28 coefficients are loaded
// before the 8-step chain), then the block below them, T21 = -T22 (A21 T11), 8 x 8 products in fp32.  A is
// overwritten by T in place; Rw is this warp's 64-float scratch.
__device__ __forceinline__ void solve_block16(float* Am, float* Rw, int o, int lane) {
    if (lane < 16) {
        const int o8 = o + 8 * (lane >> 3), c = lane & 7;
        float a[28];
#pragma unroll
        for (int r = 1; r < 8; ++r)
#pragma unroll
            for (int j = 0; j < r; ++j) a[r * (r - 1) / 2 + j] = Am[(o8 + r) * TS + o8 + j];
        float x[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int r = j + 1; r < 8; ++r) x[r] = fmaf(-a[r * (r - 1) / 2 + j], x[j], x[r]);
        __syncwarp(0x0000FFFFu);   // the sub-block's coefficients are read before any column is overwritten
#pragma unroll
        for (int r = 0; r < 8; ++r) Am[(o8 + r) * TS + o8 + c] = x[r];
    }
    __syncwarp();
    const int i = lane >> 2, c2 = 2 * (lane & 3);   // row i, columns c2, c2 + 1 of the 8 x 8 products
    float r0 = 0.f, r1 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float aik = Am[(o + 8 + i) * TS + o + k];
        r0 = fmaf(aik, Am[(o + k) * TS + o + c2], r0);
        r1 = fmaf(aik, Am[(o + k) * TS + o + c2 + 1], r1);
    }
    Rw[i * 8 + c2] = r0;
    Rw[i * 8 + c2 + 1] = r1;
    __syncwarp();   // A21 is read and R written by every lane
    float t0 = 0.f, t1 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float tik = Am[(o + 8 + i) * TS + o + 8 + k];
        t0 = fmaf(tik, Rw[k * 8 + c2], t0);
        t1 = fmaf(tik, Rw[k * 8 + c2 + 1], t1);
    }
    Am[(o + 8 + i) * TS + o + c2] = -t0;
    Am[(o + 8 + i) * TS + o + c2 + 1] = -t1;
}

// Blocked inverse of the unit lower-triangular (I + A), 64 x 64, in place: A (strictly lower, fp32, row stride
// TS) is overwritten by T = (I + A)^{-1}.  Level 0: the four 16 x 16 diagonal blocks, one warp each.  Level 1:
// the 16 x 16 blocks below them in the two 32 x 32 diagonal blocks, T21 = -T22 (A21 T11).
// Level 2: the 32 x 32 block, T21 = -T22 (A21 T11) over 8 warps with a barrier between the two products.
// (Level 1 runs on two warps per block, column halves, with a pair barrier before T21 overwrites A21.)
// Levels 1 and 2 are TF32 warp-level tile products with fp32 accumulation.  The upper triangle of every
// 32 x 32 diagonal block must hold zeros on entry (the epilogue writes them); the block above the diagonal
// of the whole matrix is never read.  Every thread passes every barrier.
__device__ void solve_unit_lower_inplace(float* Am, float* Rt, int t, bool work) {
    const int w = t >> 5, lane = t & 31;
    if (work && w < 4) solve_block16(Am, Rt + 64 * w, 16 * w, lane);
    __syncthreads();
    if (work && w < 4) {   // level 1: block pair pr, column half nt; R = A21 T11, then T21 = -T22 R
        const int pr = w >> 1, nt = w & 1, o1 = 32 * pr;
        float* Rw = Rt + 16 * pr * RS;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
            mma_tile_tf32(d, Am + (o1 + 16) * TS + o1 + 8 * ks, TS, Am + (o1 + 8 * ks) * TS + o1 + 8 * nt, TS, lane);
        st_tile(Rw + 8 * nt, RS, d, lane, 1.f);
        if (pr == 0) named_bar(1, 64);   // both column halves have read A21 before T21 overwrites it
        else named_bar(2, 64);
        float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
            mma_tile_tf32(e, Am + (o1 + 16) * TS + o1 + 16 + 8 * ks, TS, Rw + (8 * ks) * RS + 8 * nt, RS, lane);
        st_tile(Am + (o1 + 16) * TS + o1 + 8 * nt, TS, e, lane, -1.f);
    }
    __syncthreads();
    const int mt = w & 1, nq = w >> 1;   // level 2: 2 row tiles x 4 column tiles of 8
    if (work) {   // R = A[32..63][0..31] T[0..31][0..31]
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_tile_tf32(d, Am + (32 + 16 * mt) * TS + 8 * ks, TS, Am + (8 * ks) * TS + 8 * nq, TS, lane);
        st_tile(Rt + (16 * mt) * RS + 8 * nq, RS, d, lane, 1.f);
    }
    __syncthreads();
    if (work) {   // T[32..63][0..31] = -T[32..63][32..63] R
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_tile_tf32(d, Am + (32 + 16 * mt) * TS + 32 + 8 * ks, TS, Rt + (8 * ks) * RS + 8 * nq, RS, lane);
        st_tile(Am + (32 + 16 * mt) * TS + 8 * nq, TS, d, lane, -1.f);
    }
    __syncthreads();
}

}  // namespace
}  // namespace gdn
