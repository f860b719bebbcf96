// Device pieces shared by the scalar-gate chunk pairs (chunk_gdn_tmem.cu at head size 128, chunk_gdn_d256.cu at
// head size 256): the within-chunk gate prefix, the chain a state CTA walks, and the bf16 -> fp16 conversion of the
// operand tiles the state kernels stage in shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "chunk_wy_common.cuh"

namespace gdn {
namespace {

// Within-chunk cumulative gate, log2 units: lane l holds tokens 2l and 2l + 1 (natural-log gates g0, g1; 0 past the
// sequence end).  Both passes of a pair use this one function, so their gate factors agree bitwise.
__device__ __forceinline__ void gate_prefix2(float g0, float g1, int lane, float& G0, float& G1, float& Glast) {
    const float LOG2E = 1.4426950408889634f;
    float x = g0 + g1;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, m);
        if (lane >= m) x += y;
    }
    G1 = x * LOG2E;
    G0 = (x - g1) * LOG2E;
    Glast = __shfl_sync(0xffffffffu, G1, 31);
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

struct GChain {
    int n, h, len;
    long row0;
};

// Chain index -> (sequence, head); packed sequences longest first (their chains are the longest serial paths)
__device__ GChain g_resolve_chain(const Geo& g, int idx) {
    GChain c;
    const int seq_rank = idx / g.H;
    c.h = idx % g.H;
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

// One 16 KB tile at shared address `src` (two 64-column bf16 slabs of 64 rows, 128-byte swizzled, the second at
// src + stride) to fp16 at `dst` (same layout; dst == src converts in place) by NTHR threads; rows past the end
// become zeros, and with SCALE row r is multiplied by the fp32 rs[r] (shared address rs) first.  The loads of a batch
// of 8 chunks are issued before their stores, so that their latencies overlap.
template <int NTHR, bool SCALE>
__device__ __forceinline__ void tile_to_f16(uint32_t src, uint32_t dst, uint32_t stride, int L, int idx, uint32_t rs) {
    constexpr int PER = 1024 / NTHR, BATCH = PER < 8 ? PER : 8;
#pragma unroll 1
    for (int u0 = 0; u0 < PER; u0 += BATCH) {
        uint4 v[BATCH];
        float f[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int e = idx + NTHR * (u0 + u);
            v[u] = lds128(src + (e >> 9) * stride + (e & 511) * 16);
            f[u] = SCALE ? lds32f(rs + 4 * ((e >> 3) & 63)) : 1.f;
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int e = idx + NTHR * (u0 + u);
            const bool zero = ((e >> 3) & 63) >= L;
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = zero ? 0u
                            : pack_h2(f[u] * __uint_as_float(w[i] << 16), f[u] * __uint_as_float(w[i] & 0xFFFF0000u));
            sts128(dst + (e >> 9) * stride + (e & 511) * 16, o[0], o[1], o[2], o[3]);
        }
    }
}

}  // namespace
}  // namespace gdn
