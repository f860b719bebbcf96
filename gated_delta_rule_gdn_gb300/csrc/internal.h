// Host-side interface between the C ABI (api.cu) and the kernel translation units.
// Not installed; include/gdn.h is the public boundary.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace gdn {

// One chunk-forward request, already validated by api.cu.
struct ChunkArgs {
    const void* q;          // [B, T, H, dk]
    const void* k;          // [B, T, H, dk]
    const void* v;          // [B, T, H, dv]
    const float* g;         // [B, T, H] or [B, T, H, dk] (per_channel)
    const float* beta;      // [B, T, H]
    float scale;
    const float* h0;        // [N, H, dk, dv] or nullptr
    float* hT;              // [N, H, dk, dv] or nullptr
    const int32_t* cu;      // [n_seqs + 1] device or nullptr
    int n_seqs;
    void* o;                // [B, T, H, dv]
    int B, T, H, dk, dv, C;
    int bf16;               // 1: q, k, v are bf16; 0: fp32
    int per_channel;        // 1: KDA gate [.., dk]
    int o_f32;              // 1: o is fp32; 0: o is bf16
    int N() const { return cu ? n_seqs : B; }
};

struct StepArgs {
    const void* q;          // [N, H, dk]
    const void* k;          // [N, H, dk]
    const void* v;          // [N, H, dv]
    const float* g;         // [N, H]
    const float* beta;      // [N, H]
    float scale;
    float* state;           // [N, H, dk, dv] in place
    void* o;                // [N, H, dv]
    int N, H, dk, dv;
    int bf16;               // 1: q, k, v are bf16; 0: fp32
    int o_f32;              // 1: o is fp32; 0: o is bf16
};

// Generic fp32 SIMT chunk kernel (chunk_generic.cu).
cudaError_t launch_chunk_generic(const ChunkArgs& a, cudaStream_t s);

// Fused tcgen05/TMA chunk kernel for the scalar gate (chunk_tc.cu).
// Returns nullptr if the request fits the kernel, else a reason.
const char* tc_chunk_unsupported_reason(const ChunkArgs& a);
cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t s);

// Decode step (recurrent_step.cu).
cudaError_t launch_recurrent_step(const StepArgs& a, cudaStream_t s);

// Device-side status words of kernels with bounded waits.
cudaError_t tc_read_and_clear_status(unsigned* value, bool clear);

}  // namespace gdn
