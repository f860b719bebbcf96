// Host-side interface between the C ABI (api.cu) and the kernel translation units.
// Not installed; include/gdn.h is the public boundary.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace gdn {

// Optional in-kernel activation of the scalar gate and of beta (all null / zero: the inputs are already log alpha
// and beta).
struct GateAct {
    const float* A_log;     // [H] or nullptr: g holds log alpha itself
    const float* dt_bias;   // [H] or nullptr (zero)
    int beta_sigmoid;       // 1: beta = sigmoid(logit); 2: beta = 2 sigmoid(logit); 0: beta as given
    bool any() const { return A_log != nullptr || beta_sigmoid != 0; }
    bool gate() const { return A_log != nullptr; }
};

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
    GateAct act;            // gate / beta activation (two-pass path, scalar gate only)
    int Hk;                 // key heads of q and k (0: H); H (value heads) is a multiple of it
    int test_fwd;           // test of the two-pass state kernels: 1 their first record copy is left out (its bounded
                            // waits run out); 2 the scalar-gate ring runs one chunk deep (must not change the result)
    int N() const { return cu ? n_seqs : B; }
    int HK() const { return Hk > 0 ? Hk : H; }
};

struct StepArgs {
    const void* q;          // [N, H, dk]
    const void* k;          // [N, H, dk]
    const void* v;          // [N, H, dv]
    const float* g;         // [N, H] or [N, H, dk] (per_channel)
    const float* beta;      // [N, H]
    float scale;
    float* state;           // [N, H, dk, dv] in place
    void* o;                // [N, H, dv]
    int N, H, dk, dv;
    int bf16;               // 1: q, k, v are bf16; 0: fp32
    int o_f32;              // 1: o is fp32; 0: o is bf16
    int per_channel;        // 1: KDA gate [N, H, dk]
    GateAct act;            // gate / beta activation (scalar gate only)
    int Hk;                 // key heads of q and k (0: H); H (value heads) is a multiple of it
};

// Generic fp32 SIMT chunk kernel (chunk_generic.cu).
cudaError_t launch_chunk_generic(const ChunkArgs& a, cudaStream_t s);
// Dynamic shared memory the generic kernel needs for this request, and the most one CTA may have.
size_t generic_smem_bytes(const ChunkArgs& a);
constexpr size_t kMaxSmemPerBlock = 227 * 1024;

// Two-pass tcgen05 chunk path.  The per-channel gate (chunk_two_pass.cu): a per-chunk kernel over all SMs writes the
// state-independent products to a workspace, then a state kernel walks each (chain, d_v half).  The scalar gate
// (chunk_gdn_tmem.cu): a per-chunk kernel writes -W, P and T diag(beta), then a transposed state kernel walks each
// chain with its chain operands in tensor memory.  launch_chunk_two_pass and two_pass_workspace_bytes pick the pair.
const char* two_pass_unsupported_reason(const ChunkArgs& a);
size_t two_pass_workspace_bytes(const ChunkArgs& a);
cudaError_t launch_chunk_two_pass(const ChunkArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t s);
size_t gdn_tmem_workspace_bytes(const ChunkArgs& a);
cudaError_t launch_chunk_gdn_tmem(const ChunkArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t s);
// The scalar gate at d_k = d_v = 256 (chunk_gdn_d256.cu): the same two passes, the state kernel per (chain, d_v half)
// with the fp32 state in tensor memory.
size_t gdn_d256_workspace_bytes(const ChunkArgs& a);
cudaError_t launch_chunk_gdn_d256(const ChunkArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t s);
// The statically allocated two-pass workspace: its size, and its device address on the current device (looked up
// once per device with cudaGetSymbolAddress).
size_t static_workspace_capacity();
cudaError_t static_workspace(void** ptr);

// Host helpers of the tcgen05 paths (tensor_map.cu).
// TMA map of a [rows][H][d] bf16 tensor, box 64 elements x 1 head x 64 rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, long rows, int H, int d);
// TMA map of a [rows][H][d] fp32 tensor (d <= 256), box d x 1 head x 64 rows, no swizzle: a 64-row tile lands
// as a dense row-major [64][d] block.
bool make_map_f32_rows(CUtensorMap* m, const float* base, long rows, int H, int d);
// The same for fp32 or bf16 (f32 false), for loads and stores; box_d > 0 narrows the box to box_d elements of d, and
// box_rows sets its height.
bool make_map_rows(CUtensorMap* m, const void* base, long rows, int H, int d, bool f32, int box_d = 0,
                   int box_rows = 64);
bool device_is_sm100_family();

// Decode step (recurrent_step.cu).
cudaError_t launch_recurrent_step(const StepArgs& a, cudaStream_t s);

// Device-side status words of the kernels with bounded waits.  Bits 0-7 and 9-15: a wait that gave up; bit 8
// (kStatusNonfinite): a chunk-forward state kernel wrote a non-finite value to o or the final state.
constexpr unsigned kStatusNonfinite = 1u << 8;
cudaError_t tp_read_and_clear_status(unsigned* value, bool clear);
cudaError_t gt_read_and_clear_status(unsigned* value, bool clear);
cudaError_t d256_read_and_clear_status(unsigned* value, bool clear);

// One chunk-backward request, already validated by api.cu.  Gradients are of
// L = <dO, o> + <dhT, final state> with respect to every input of the forward.
struct BwdArgs {
    const void* q;          // [B, T, H, dk]
    const void* k;          // [B, T, H, dk]
    const void* v;          // [B, T, H, dv]
    const float* g;         // [B, T, H] or [B, T, H, dk] (per_channel)
    const float* beta;      // [B, T, H]
    float scale;
    const float* h0;        // [N, H, dk, dv] or nullptr
    const void* dO;         // [B, T, H, dv]
    const float* dhT;       // [N, H, dk, dv] or nullptr (zero)
    const int32_t* cu;      // [n_seqs + 1] device or nullptr
    int n_seqs;
    float* gq;              // [B, T, H, dk]
    float* gk;              // [B, T, H, dk]
    float* gv;              // [B, T, H, dv]
    float* gg;              // like g
    float* gbeta;           // [B, T, H]
    float* gh0;             // [N, H, dk, dv] or nullptr
    float* ck;              // chunk-entry state checkpoints (workspace)
    int B, T, H, dk, dv, C;
    int bf16;               // q, k, v dtype: 1 bf16, 0 fp32
    int do_bf16;            // dO dtype
    int per_channel;
    int test_skip_record;   // test of the bounded waits: the walks leave out the copy of their first chunk record
    int Hk;                 // key heads of q and k (0: H); value head h reads key head h / (H / Hk)
    float* gq_part;         // with Hk < H: per-value-head dq, dk ([B, T, H, dk]), summed per key head afterwards
    float* gk_part;
    int N() const { return cu ? n_seqs : B; }
    __host__ __device__ int HK() const { return Hk > 0 ? Hk : H; }
};

// One-shot test injection armed by gdn_test_inject (api.cu): true, and disarmed, if the armed injection is `what`.
bool take_test_injection(int what);

// Chunk backward (chunk_bwd.cu).
size_t bwd_smem_bytes(int C, int dk, bool per_channel);
// The chunk the backward takes when the caller leaves it open (0 if none fits one CTA's shared memory).
int bwd_auto_chunk(int dk, bool per_channel);
size_t bwd_workspace_bytes(const BwdArgs& a);
// byte offsets in the workspace of the activated log alpha and beta, and of the per-value-head dq, dk parts
size_t bwd_act_offset(const BwdArgs& a);
size_t bwd_part_offset(const BwdArgs& a);
// grouped value heads: dq, dk summed per key head from the parts
cudaError_t launch_bwd_group_sum(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_chunk_bwd(const BwdArgs& a, cudaStream_t s);
cudaError_t bwd_read_and_clear_status(unsigned* value, bool clear);
// The gate / beta activations around the backward: log alpha and beta from raw logits (into g_out, beta_out), and
// afterwards the chain rule (dg, dbeta in place; per-head dA_log, ddt from the gradient of log alpha).
cudaError_t launch_bwd_act_apply(const float* x, const float* b, const GateAct& act, float* g_out, float* beta_out,
                                 long n, int H, cudaStream_t s);
cudaError_t launch_bwd_act_post(const float* x, const float* b, const float* g_act, const GateAct& act, float* dg,
                                float* dbeta, float* dA_log, float* ddt, long rows, int H, cudaStream_t s);

}  // namespace gdn
