// Device helpers shared by the chunk kernels built on tcgen05 (chunk_tc.cu, chunk_two_pass.cu): named
// barriers, 16-byte shared/global accesses, fp16 packing, the hardware exp2, and the warp-level TF32 tile
// product of the triangular solve.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "tc_common.cuh"

namespace gdn {
namespace tc {

// Row strides (floats) of the fp32 64 x 64 matrices of the solve and of its 32-row scratch tile.
constexpr int TS = 68;
constexpr int RS = 36;

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 16-byte shared-memory accesses through pointers into the shared array (the compiler emits STS/LDS and
// schedules them freely; ordering against the async proxy comes from the explicit fences and barriers)
__device__ __forceinline__ void st16(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}
__device__ __forceinline__ uint4 ld16(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void bf16x8_to_f32(uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void h8_to_f32(uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// Scaled copy of a row chunk of 8 bf16 values into 8 fp16 values (scale 0 writes exact zeros).
__device__ __forceinline__ void copy_scaled_chunk(const uint8_t* src, uint8_t* dst, float s, bool zero) {
    float f[8];
    bf16x8_to_f32(ld16(src), f);
    const uint32_t m = zero ? 0u : 0xFFFFFFFFu;     // exact zeros for rows past the sequence end
    st16(dst, pack_h2(f[0] * s, f[1] * s) & m, pack_h2(f[2] * s, f[3] * s) & m, pack_h2(f[4] * s, f[5] * s) & m,
         pack_h2(f[6] * s, f[7] * s) & m);
}

// 2^x by the hardware's ex2.approx (flush-to-zero): |relative error| ~2^-22; large negative x gives +0
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// d (16 x 8, fp32) += A (16 x 8) B (8 x 8); A and B are fp32 row-major tiles in shared memory.
// Fragment ownership (lane = 4 g + t): A rows g, g + 8 and columns t, t + 4; B rows t, t + 4 and column g;
// d rows g, g + 8 and columns 2 t, 2 t + 1.
__device__ __forceinline__ void mma_tile_tf32(float (&d)[4], const float* A, int lda, const float* B, int ldb,
                                              int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t a0 = to_tf32(A[g * lda + t]), a1 = to_tf32(A[(g + 8) * lda + t]);
    const uint32_t a2 = to_tf32(A[g * lda + t + 4]), a3 = to_tf32(A[(g + 8) * lda + t + 4]);
    const uint32_t b0 = to_tf32(B[t * ldb + g]), b1 = to_tf32(B[(t + 4) * ldb + g]);
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void st_tile(float* D, int ldd, const float (&d)[4], int lane, float sgn) {
    const int g = lane >> 2, t = lane & 3;
    D[g * ldd + 2 * t] = sgn * d[0];
    D[g * ldd + 2 * t + 1] = sgn * d[1];
    D[(g + 8) * ldd + 2 * t] = sgn * d[2];
    D[(g + 8) * ldd + 2 * t + 1] = sgn * d[3];
}

// 8 fp32 values to fp16, one 16-byte shared store
__device__ __forceinline__ void st_h8(uint8_t* p, const float* f) {
    st16(p, pack_h2(f[0], f[1]), pack_h2(f[2], f[3]), pack_h2(f[4], f[5]), pack_h2(f[6], f[7]));
}

// 16 bytes to global memory, cached in L2 only (the data is read back by another kernel)
__device__ __forceinline__ void stg16(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    __stcg(reinterpret_cast<uint4*>(p), make_uint4(a, b, c, d));
}
__device__ __forceinline__ void stg_h8(uint8_t* p, const float* f) {
    stg16(p, pack_h2(f[0], f[1]), pack_h2(f[2], f[3]), pack_h2(f[4], f[5]), pack_h2(f[6], f[7]));
}

// Epilogue of D0 = [K; Q] K^T.  Rows 0-63 (token i): A[i][j] = beta_i 2^(lg_i - lg_j) (K K^T)_ij for j < i, in
// fp32 for the solve, plus (IDENTITY) row i of the identity in [I; P].  Rows 64-127 (token i = row - 64):
// P[i][j] = scale 2^(lg_i - lg_j) (Q K^T)_ij for j <= i, in fp16, stored transposed: element (j, i) at row 64 + j,
// column i of [I; P^T] (128-byte swizzled rows).  Column blocks wholly above the diagonal for every row of the warp
// are skipped (warp-uniform); the solve never reads A above the diagonal.
template <bool IDENTITY>
__device__ __forceinline__ void epilogue_kkt(uint32_t tl, int row, int q4, int pw, const float* lg, const float* bb, float scale,
                                             float* Am, uint8_t* a1) {
    // this thread: row `row`, columns [32 pw, 32 pw + 32)
    const int c0 = 32 * pw;
    uint32_t r[2][16];
    tmem_ld16(tl + c0, r[0]);
    tmem_ld16(tl + c0 + 16, r[1]);
    tmem_ld_wait();
    const int i = row & 63;
    const int imax = 32 * (q4 & 1) + 31;      // last row of this warp, within its 64-row half
    const bool live = c0 <= imax;             // warp-uniform: some column of the half can be on or below the diagonal
    const float li = lg[i];
    if (row < 64) {
        if (live) {
            const float bi = bb[i];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                float v[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int j = c0 + cb * 16 + q;
                    const float e = ex2(li - lg[j]);
                    v[q] = (j < i) ? bi * e * __uint_as_float(r[cb][q]) : 0.f;
                }
                float4* dst = reinterpret_cast<float4*>(Am + i * TS + c0 + cb * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
        const uint32_t one = (i & 1) ? 0x3C000000u : 0x00003C00u;     // fp16 1.0 in the low or high half
#pragma unroll
        for (int cc = 0; cc < (IDENTITY ? 4 : 0); ++cc) {
            const int c8 = 4 * pw + cc;
            const bool here = (i >> 3) == c8;
            const int qw = (i & 7) >> 1;
            st16(a1 + sw128_off(row, c8 * 8), here && qw == 0 ? one : 0u, here && qw == 1 ? one : 0u,
                 here && qw == 2 ? one : 0u, here && qw == 3 ? one : 0u);
        }
    } else {
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            float v[16];
            if (!live) {
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] = 0.f;
            } else {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int j = c0 + cb * 16 + q;
                    const float e = ex2(li - lg[j]);
                    v[q] = (j <= i) ? scale * e * __uint_as_float(r[cb][q]) : 0.f;
                }
            }
            // neighbouring lanes (rows i, i + 1 with i even) swap one value per column pair: the even lane stores
            // (P[i][j], P[i+1][j]) into row j of P^T, the odd lane (P[i][j+1], P[i+1][j+1]) into row j + 1
            const bool odd = row & 1;
#pragma unroll
            for (int q = 0; q < 16; q += 2) {
                const int j = c0 + cb * 16 + q;
                const float recv = __shfl_xor_sync(0xffffffffu, odd ? v[q] : v[q + 1], 1);
                const uint32_t w = odd ? pack_h2(recv, v[q + 1]) : pack_h2(v[q], recv);
                *reinterpret_cast<uint32_t*>(a1 + sw128_off(64 + j + odd, (i & ~1))) = w;
            }
        }
    }
}

}  // namespace tc
}  // namespace gdn
